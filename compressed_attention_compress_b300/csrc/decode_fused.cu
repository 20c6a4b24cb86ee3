// One CSA decode step in one cooperative launch: indexer scores, exact top-k and
// the attention over the selected entries plus the window, for one query token
// per sequence, bf16, d = 128, H in {64, 128}.
//
// QbitAI article "DeepSeek V4报告太详尽了！", section 混合注意力机制: CSA step 2 (a light
// indexer scores the query against every compressed entry and keeps the top-k),
// CSA step 3 (MQA over the selected entries) and the sliding-window paragraph
// (the most recent raw tokens join the same softmax).  The result equals
// hsa_index_topk followed by hsa_attn_decode (same selection, bit-exact; the
// attention within the bf16 tolerance); only the order of the work differs.
//
// The CTAs of a row (one sequence) each own a contiguous chunk of its entries
// and meet at three row barriers (the launch is cooperative, so every CTA is
// resident; every wait is bounded and raises the device flag if it gives up):
//   P1  dp4a scores of the chunk, streamed through bulk-copy stages, kept in
//       shared memory as biased keys; a 2048-bin histogram of the high key bits
//       is added to the row's histogram.                         -- barrier 1
//   P2  every CTA reads the row histogram and finds the bin b1 holding the k-th
//       largest key; it counts its keys above b1 and appends its keys in b1
//       (key, index) to the row's b1 list.                        -- barrier 2
//   P3  every CTA reads the (short) b1 list and resolves the exact threshold key
//       T and how many keys equal to T are taken (the first in index order), so
//       it knows every chunk's number of winners and its own winners' places in
//       the ascending output, which it writes.  It then runs the attention over
//       its own winners and its share of the window on the tensor cores
//       -- S = Q K^T with M = 128 query heads (H = 64 pads Q with zero rows) and
//       N = 64 items, an online softmax, O += P V in TMEM -- and writes its
//       partial (O in bf16, maximum, sum).  The window tokens are dealt round
//       robin over the row's CTAs.                                 -- barrier 3
//   P4  every CTA combines a share of the heads over the row's partials with the
//       log-sum-exp rule and writes the output and the log-sum-exp.
// The histogram is cleared after barrier 2, the counters by the row's last CTA
// out, so the workspace is left zero for the next call.
#include <math.h>

#include "block_scan.cuh"
#include "internal.h"
#include "tc_common.cuh"

namespace hsa {

namespace {

constexpr int kThreads = 256;
constexpr int kNB1 = 2048;                     // level-1 histogram bins
constexpr int kStages = 3;                     // key-stream stages
constexpr int kStageBytes = 16384;
constexpr int kM = 128;                        // MMA M: query heads (padded)
constexpr int kD = 128;                        // head dim
constexpr int kNT = 64;                        // items per attention tile (MMA N of S)
constexpr int kQBlk = kM * 128;                // 16 KiB: one 64-column block of Q
constexpr int kQBytes = 2 * kQBlk;             // 32 KiB
constexpr int kTBlk = kNT * 128;               // 8 KiB: one 64-column block of a K or V tile
constexpr int kTile = 2 * kTBlk;               // 16 KiB
// P [128 heads][64 items] bf16 (16 KiB) takes the K tile's place once S is done
// (the V tile's when one buffer is both K and V)
constexpr int kAttnBytes = kQBytes + 2 * kTile;  // 64 KiB
constexpr int kWorkBytes = 16384 + kStages * kStageBytes;  // P1: histogram + stages (64 KiB)
static_assert(kWorkBytes <= kAttnBytes, "the key stages fit the attention tiles' space");
constexpr int kMaxChunks = 256;                // CTAs per row (one value per thread in the scans)
constexpr unsigned long long kWaitNs = 200ull * 1000 * 1000;  // any wait gives up after 200 ms
// device-flag bits of the wait that gave up (or the check that failed)
constexpr unsigned kGaveUpBarrier = 0x100u;  // << k for row barrier k = 0, 1, 2
constexpr unsigned kGaveUpStage = 0x800u;
constexpr unsigned kGaveUpS = 0x1000u;
constexpr unsigned kGaveUpPV = 0x2000u;
constexpr unsigned kBadCount = 0x4000u;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct StepArgs {
    const int8_t *qi;     // [B, DI] (row stride qi_sb)
    int64_t qi_sb;
    const int8_t *ki;     // [B, E_cap, DI], rows contiguous (stride DI)
    int64_t ki_sb, E_cap;
    int B, DI, m, topk, H, window, shared_kv;
    int32_t *idx_out, *cnt_out;  // [B, topk], [B]
    const __nv_bfloat16 *q;      // [B, H, d]
    const __nv_bfloat16 *kc, *vc, *k_raw, *v_raw;
    int64_t c_sb, c_se, r_sb, r_st, N_cap;
    const int64_t *ctx;          // [B]: the query sits at p = ctx - 1
    float scale_log2;
    __nv_bfloat16 *out;          // [B, H, d]
    float *lse;                  // [B, H] or null
};

struct Ws {
    unsigned *hist;     // [kNB1]
    unsigned *bar;      // [4]: barrier counter, b1 list length
    int *rec;           // [ctas_per_row]: keys above b1 per chunk
    uint2 *b1;          // [E_cap]: (key, index) of the keys in b1
    __nv_bfloat16 *po;  // [ctas_per_row][H][d]: partial O
    float *pml;         // [ctas_per_row][2][H]: maximum (log2 units), sum
};
__device__ __forceinline__ Ws carve(void *ws, const DecodeStepPlan &p, const StepArgs &a, int r) {
    char *b = static_cast<char *>(ws);
    Ws w;
    w.hist = reinterpret_cast<unsigned *>(b + p.off_hist) + (size_t)r * kNB1;
    w.bar = reinterpret_cast<unsigned *>(b + p.off_bar) + (size_t)r * 4;
    w.rec = reinterpret_cast<int *>(b + p.off_rec) + (size_t)r * p.ctas_per_row;
    w.b1 = reinterpret_cast<uint2 *>(b + p.off_b1) + (size_t)r * a.E_cap;
    w.po = reinterpret_cast<__nv_bfloat16 *>(b + p.off_po) + (size_t)r * p.ctas_per_row * a.H * kD;
    w.pml = reinterpret_cast<float *>(b + p.off_pml) + (size_t)r * p.ctas_per_row * 2 * a.H;
    return w;
}

__device__ __forceinline__ unsigned long long gtime() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Row barrier k (0, 1, 2) on a counter that only grows within a launch: every CTA
// adds one and waits for `target`.  false (and the device flag) if the wait gives
// up after kWaitNs.
__device__ __forceinline__ bool row_barrier(unsigned *ctr, unsigned target, int k, int *s_flag) {
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(ctr, 1u);
        const unsigned long long t0 = gtime();
        int ok = 1;
        while (ld_acquire(ctr) < target) {
            if (gtime() - t0 > kWaitNs) {
                raise_flag(FLAG_INDEX_RANGE | (kGaveUpBarrier << k));
                ok = 0;
                break;
            }
            __nanosleep(32);
        }
        *s_flag = ok;
    }
    __syncthreads();
    return *s_flag != 0;
}

__device__ __forceinline__ int dot16(const int4 &x, const int4 &y) {
    int s = __dp4a(x.x, y.x, 0);
    s = __dp4a(x.y, y.y, s);
    s = __dp4a(x.z, y.z, s);
    return __dp4a(x.w, y.w, s);
}

// Wait for an mbarrier phase; false after kWaitNs.
__device__ __forceinline__ bool wait_phase(uint64_t *bar, unsigned parity) {
    const unsigned long long t0 = gtime();
    for (unsigned i = 0;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 15) == 15 && gtime() - t0 > kWaitNs) return false;
    }
}

// 16-byte chunk c of row r of a 128-byte-swizzled K-major tile of 64-column blocks
__device__ __forceinline__ uint32_t sw_off(int r, int c, int blk_bytes) {
    return (uint32_t)((c >> 3) * blk_bytes + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// Largest bin t (from the top) of hist[0..nb) whose suffix count reaches `need`;
// s_out[0] = t, s_out[1] = keys in bins above t.  Every thread calls it.
__device__ __forceinline__ void find_threshold(const unsigned *hist, int nb, int need, int *s_scan, int *s_out) {
    const int per = nb / kThreads;
    const int top = nb - 1 - threadIdx.x * per;
    int local = 0;
    for (int q = 0; q < per; ++q) local += (int)hist[top - q];
    int tot;
    const int before = block_exclusive_sum(local, s_scan, tot);
    if (before < need && before + local >= need) {
        int cum = before;
        for (int q = 0; q < per; ++q) {
            const int hv = (int)hist[top - q];
            if (cum + hv >= need) {
                s_out[0] = top - q;
                s_out[1] = cum;
                break;
            }
            cum += hv;
        }
    }
    __syncthreads();
}

template <int LPE>
__global__ void __launch_bounds__(kThreads, 1) decode_step_kernel(StepArgs a, DecodeStepPlan p, void *ws) {
    extern __shared__ __align__(16) unsigned char smem_raw[];  // rounded up to 1024 at run time
    unsigned char *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    // [0, 80 KiB): P1 histogram (16 KiB) + key stages; P3 level-2 histogram; then
    // the attention tiles Q | K | V | P.  After it: the chunk's keys, its winners.
    unsigned char *s_work = smem;
    unsigned *s_h = reinterpret_cast<unsigned *>(s_work);
    unsigned char *s_stage = s_work + 16384;
    uint32_t *s_keys = reinterpret_cast<uint32_t *>(smem + kAttnBytes);
    int32_t *s_win = reinterpret_cast<int32_t *>(smem + kAttnBytes + (size_t)p.chunk * 4);
    // P takes the K tile's place once S is done (the V tile's when K and V are one buffer)
    unsigned char *sQ = s_work, *sK = s_work + kQBytes, *sV = sK + kTile, *sP = a.shared_kv ? sV : sK;
    __shared__ int s_scan[33];
    __shared__ int s_misc[16];
    __shared__ int s_gt[kMaxChunks], s_eq[kMaxChunks];
    __shared__ __align__(8) uint64_t s_bar[kStages];
    __shared__ __align__(8) uint64_t bar_s, bar_o, bar_f;
    __shared__ uint32_t s_tmem;

    const int row = blockIdx.y, c = blockIdx.x, tid = threadIdx.x, warp = tid >> 5;
    const int64_t pos = a.ctx[row] - 1;
    int64_t E = num_entries(pos, a.m);
    if (E > a.E_cap) {
        if (c == 0 && tid == 0) raise_flag(FLAG_INDEX_RANGE);
        E = a.E_cap;
    }
    const int kE = (int)(E < a.topk ? E : a.topk);
    const int nch = E > 0 ? (int)((E + p.chunk - 1) / p.chunk) : 1;
    if (c >= nch) return;
    const int64_t c0 = (int64_t)c * p.chunk;
    const int n = E > 0 ? (int)(E - c0 < p.chunk ? E - c0 : p.chunk) : 0;
    const Ws w = carve(ws, p, a, row);
    int32_t *idx_out = a.idx_out + (int64_t)row * a.topk;
    if (c == 0) {
        for (int i = kE + tid; i < a.topk; i += kThreads) idx_out[i] = -1;
        if (tid == 0) a.cnt_out[row] = kE;
    }
    if (tid == 0) {
        for (int st = 0; st < kStages; ++st) mbar_init(&s_bar[st], 1);
        mbar_init(&bar_s, 1);
        mbar_init(&bar_o, 1);
        mbar_init(&bar_f, 1);
        fence_mbar_init();
    }
    if (warp == 0) tc::tmem_alloc(&s_tmem, 256);  // S: columns [0, 64), O: [128, 256)
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = s_tmem, tS = tmem, tO = tmem + 128;
    bool ok = true;

    // ---------------------------------------------------------------- P1
    const int bias = a.DI * 16256;
    if (n > 0) {
        for (int i = tid; i < kNB1; i += kThreads) s_h[i] = 0;
        const int lane_e = tid % LPE, grp = tid / LPE;
        constexpr int kGroups = kThreads / LPE;
        const int4 qv = *reinterpret_cast<const int4 *>(a.qi + row * a.qi_sb + lane_e * 16);
        const int eps = kStageBytes / a.DI;  // entries per stage
        const int nst = (n + eps - 1) / eps;
        const char *src = reinterpret_cast<const char *>(a.ki + row * a.ki_sb + c0 * a.DI);
        __syncthreads();
        auto issue = [&](int it) {
            const int st = it % kStages;
            const int ne = min(eps, n - it * eps);
            const unsigned bytes = (unsigned)(ne * a.DI);
            mbar_expect_tx(&s_bar[st], bytes);
            bulk_g2s(s_stage + st * kStageBytes, src + (int64_t)it * kStageBytes, bytes, &s_bar[st]);
        };
        if (tid == 0)
            for (int it = 0; it < nst && it < kStages; ++it) issue(it);
        int it = 0;
        for (; it < nst; ++it) {
            const int st = it % kStages;
            if (!__syncthreads_and(wait_phase(&s_bar[st], (unsigned)((it / kStages) & 1)))) {
                ok = false;
                break;
            }
            const int ne = min(eps, n - it * eps);
            const unsigned char *base = s_stage + st * kStageBytes + lane_e * 16;
            for (int el0 = 0; el0 < ne; el0 += kGroups) {
                const int el = el0 + grp;
                const bool valid = el < ne;
                const int4 kv = valid ? *reinterpret_cast<const int4 *>(base + el * a.DI) : make_int4(0, 0, 0, 0);
                int s = dot16(qv, kv);
#pragma unroll
                for (int o = 1; o < LPE; o <<= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
                if (lane_e == 0 && valid) {
                    const uint32_t key = (uint32_t)(s + bias);
                    s_keys[it * eps + el] = key;
                    atomicAdd(&s_h[key >> p.shift1], 1u);
                }
            }
            __syncthreads();  // stage consumed by every thread
            if (tid == 0 && it + kStages < nst) issue(it + kStages);
        }
        if (!ok) {
            // a stage wait gave up: flag it and let the copies already issued land
            if (tid == 0) raise_flag(FLAG_INDEX_RANGE | kGaveUpStage);
            for (int j = it; j < nst && j < it + kStages; ++j) wait_phase(&s_bar[j % kStages], (unsigned)((j / kStages) & 1));
        }
        __syncthreads();
        for (int i = tid; i < kNB1; i += kThreads)
            if (s_h[i]) atomicAdd(&w.hist[i], s_h[i]);
    }
    ok = ok && row_barrier(&w.bar[0], (unsigned)nch, 0, &s_misc[15]);

    // ---------------------------------------------------------------- P2
    // b1 = the bin holding the k-th largest key; this chunk counts its keys above b1
    // and appends its keys in b1 to the row's list
    int b1 = 0, count_above = 0;
    if (ok && kE > 0) {
        constexpr int PB = kNB1 / kThreads;  // bins per thread, descending
        if (tid == 0) s_misc[0] = s_misc[1] = 0;
        const int top = kNB1 - 1 - tid * PB;
        int hv[PB];
        int local = 0;
#pragma unroll
        for (int q = 0; q < PB; ++q) {
            hv[q] = (int)__ldcg(&w.hist[top - q]);
            local += hv[q];
        }
        int tot;
        const int before = block_exclusive_sum(local, s_scan, tot);
        if (before < kE && before + local >= kE) {
            int cum = before;
#pragma unroll
            for (int q = 0; q < PB; ++q) {
                if (cum + hv[q] >= kE) {
                    s_misc[0] = top - q;  // b1
                    s_misc[1] = cum;      // keys in bins above b1
                    break;
                }
                cum += hv[q];
            }
        }
        __syncthreads();
        b1 = s_misc[0];
        count_above = s_misc[1];
        const int per = (p.chunk + kThreads - 1) / kThreads;
        const int my0 = tid * per;
        int n_above = 0, n_in = 0;
        for (int q = 0; q < per; ++q) {
            const int e = my0 + q;
            if (e < n) {
                const int bin = (int)(s_keys[e] >> p.shift1);
                n_above += bin > b1;
                n_in += bin == b1;
            }
        }
        int tot_above, tot_in;
        block_exclusive_sum(n_above, s_scan, tot_above);
        int o = block_exclusive_sum(n_in, s_scan, tot_in);
        if (tid == 0) {
            w.rec[c] = tot_above;
            s_misc[2] = tot_in ? (int)atomicAdd(&w.bar[1], (unsigned)tot_in) : 0;
        }
        __syncthreads();
        o += s_misc[2];
        for (int q = 0; q < per && n_in; ++q) {
            const int e = my0 + q;
            if (e < n) {
                const uint32_t u = s_keys[e];
                if ((int)(u >> p.shift1) == b1) {
                    w.b1[o++] = make_uint2(u, (uint32_t)(c0 + e));
                    --n_in;
                }
            }
        }
    }
    ok = ok && row_barrier(&w.bar[0], 2u * (unsigned)nch, 1, &s_misc[15]);

    // ---------------------------------------------------------------- P3
    int n_win = 0;  // this chunk's winners (ascending, in s_win)
    if (ok && kE > 0) {
        // the row histogram has been read by every CTA: clear this CTA's share
        for (int i = c * kNB1 / nch + tid; i < (c + 1) * kNB1 / nch; i += kThreads) w.hist[i] = 0;
        const int n_list = (int)__ldcg(&w.bar[1]);
        const int need = kE - count_above;  // >= 1: keys of b1 to take
        const uint32_t mask2 = (uint32_t)p.nb2 - 1u;
        // level-2 histogram of the low key bits over the b1 list
        for (int i = tid; i < p.nb2; i += kThreads) s_h[i] = 0;
        if (tid == 0) s_misc[4] = s_misc[5] = 0;
        __syncthreads();
        for (int i = tid; i < n_list; i += kThreads) atomicAdd(&s_h[__ldcg(&w.b1[i]).x & mask2], 1u);
        __syncthreads();
        find_threshold(s_h, p.nb2, need, s_scan, &s_misc[4]);
        const uint32_t T = ((uint32_t)b1 << p.shift1) | (uint32_t)s_misc[4];
        const int n_eq_need = need - s_misc[5];  // keys equal to T to take, the first in index order
        // per chunk: keys of b1 above T and keys equal to T
        for (int i = tid; i < nch; i += kThreads) s_gt[i] = s_eq[i] = 0;
        __syncthreads();
        for (int i = tid; i < n_list; i += kThreads) {
            const uint2 v = __ldcg(&w.b1[i]);
            const int ch = (int)(v.y / (uint32_t)p.chunk);
            if (v.x > T) atomicAdd(&s_gt[ch], 1);
            else if (v.x == T) atomicAdd(&s_eq[ch], 1);
        }
        __syncthreads();
        // winners of chunk t = keys above b1 + keys of b1 above T + the ties it takes;
        // the prefix over the chunks places this chunk's winners in the output
        const int t = tid;
        const int eq_t = t < nch ? s_eq[t] : 0;
        int tot;
        const int eq_before = block_exclusive_sum(eq_t, s_scan, tot);
        int take = n_eq_need - eq_before;
        take = take < 0 ? 0 : (take > eq_t ? eq_t : take);
        const int win_t = t < nch ? __ldcg(&w.rec[t]) + s_gt[t] + take : 0;
        const int off_t = block_exclusive_sum(win_t, s_scan, tot);
        if (t == c) {
            s_misc[6] = off_t;
            s_misc[7] = take;
            s_misc[8] = win_t;
        }
        if (tid == 0 && tot != kE) raise_flag(FLAG_INDEX_RANGE | kBadCount);
        __syncthreads();
        const int my_off = s_misc[6], my_take = s_misc[7], my_win = s_misc[8];
        // this chunk's winners in index order: keys above b1, keys of b1 above T, and
        // its first my_take keys equal to T
        const int per = (p.chunk + kThreads - 1) / kThreads;
        const int my0 = tid * per;
        int n_eq = 0;
        for (int q = 0; q < per; ++q) {
            const int e = my0 + q;
            if (e < n) n_eq += s_keys[e] == T;
        }
        int eq_rank = block_exclusive_sum(n_eq, s_scan, tot);
        int n_sel = 0;
        for (int q = 0, r = eq_rank; q < per; ++q) {
            const int e = my0 + q;
            if (e < n) {
                const uint32_t u = s_keys[e];
                const bool eq = u == T;
                n_sel += u > T || (eq && r < my_take);
                r += eq;
            }
        }
        int o = block_exclusive_sum(n_sel, s_scan, n_win);
        for (int q = 0, r = eq_rank; q < per && n_sel; ++q) {
            const int e = my0 + q;
            if (e < n) {
                const uint32_t u = s_keys[e];
                const bool eq = u == T;
                if (u > T || (eq && r < my_take)) {
                    s_win[o] = (int32_t)(c0 + e);
                    if (my_off + o < a.topk) idx_out[my_off + o] = (int32_t)(c0 + e);
                    ++o;
                    --n_sel;
                }
                r += eq;
            }
        }
        if (tid == 0 && n_win != my_win) raise_flag(FLAG_INDEX_RANGE | kBadCount);
        __syncthreads();
    }

    // attention over this chunk's winners and window tokens w_lo + c, w_lo + c + nch,
    // ...: 64-item tiles, one thread per head row of S and O (TMEM lane = head)
    int64_t w_lo = 0;
    int n_wnd = 0;
    if (a.window > 0 && pos >= 0) {
        w_lo = pos - a.window + 1 < 0 ? 0 : pos - a.window + 1;
        const int n_all = (int)(pos - w_lo + 1);
        n_wnd = c < n_all ? (n_all - c + nch - 1) / nch : 0;
        if (pos >= a.N_cap) {
            if (tid == 0 && c == 0) raise_flag(FLAG_ATTN_RANGE);
            n_wnd = 0;
        }
    }
    const int n_items = ok ? n_win + n_wnd : 0;
    float m_run = -INFINITY, l_run = 0.f;  // of head row tid (threads 0-127)
    const __nv_bfloat16 *qrow = a.q + (int64_t)row * a.H * kD;
    if (n_items > 0) {
        // Q: 128 head rows (rows >= H zero), 128-byte-swizzled K-major
        for (int i = tid; i < kM * 16; i += kThreads) {
            const int h = i >> 4, ch = i & 15;
            const bool v = h < a.H;
            cp_async_16(smem_u32(sQ + sw_off(h, ch, kQBlk)), v ? (const void *)(qrow + h * kD + ch * 8) : (const void *)a.q,
                        v ? 16 : 0);
        }
        cp_async_commit();
    }
    const int n_tiles = (n_items + kNT - 1) / kNT;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    for (int j = 0; j < n_tiles && ok; ++j) {
        // K and V rows of items [64j, 64j + 64): item i is winner s_win[i] or window token
        for (int i = tid; i < kNT * 16; i += kThreads) {
            const int r = i >> 4, ch = i & 15;
            const int item = j * kNT + r;
            const __nv_bfloat16 *ks = nullptr, *vs = nullptr;
            if (item < n_win) {
                const int64_t e = s_win[item];
                ks = a.kc + row * a.c_sb + e * a.c_se;
                vs = a.vc + row * a.c_sb + e * a.c_se;
            } else if (item < n_items) {
                const int64_t tk = w_lo + c + (int64_t)(item - n_win) * nch;
                ks = a.k_raw + row * a.r_sb + tk * a.r_st;
                vs = a.v_raw + row * a.r_sb + tk * a.r_st;
            }
            const uint32_t off = sw_off(r, ch, kTBlk);
            cp_async_16(smem_u32(sK + off), ks ? (const void *)(ks + ch * 8) : (const void *)a.q, ks ? 16 : 0);
            if (!a.shared_kv)
                cp_async_16(smem_u32(sV + off), vs ? (const void *)(vs + ch * 8) : (const void *)a.q, vs ? 16 : 0);
        }
        cp_async_commit();
        cp_async_wait<0>();
        tc::fence_proxy_async();
        tc::fence_before();
        __syncthreads();
        tc::fence_after();
        const unsigned char *tV = a.shared_kv ? sK : sV;
        if (tid == 0) {
            constexpr uint32_t idS = tc::idesc_bf16(kM, kNT, false, false);
            const uint32_t aQ = smem_u32(sQ), aK = smem_u32(sK);
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk) {
                const uint64_t da = tc::desc_sw128(aQ + (kk >> 2) * kQBlk + (kk & 3) * 32, 16, 1024);
                const uint64_t db = tc::desc_sw128(aK + (kk >> 2) * kTBlk + (kk & 3) * 32, 16, 1024);
                tc::mma_bf16(tS, da, db, idS, kk > 0 ? 1u : 0u);
            }
            tc::commit(&bar_s);
        }
        ok = __syncthreads_and(wait_phase(&bar_s, (unsigned)(j & 1))) != 0;
        if (!ok && tid == 0) raise_flag(FLAG_ATTN_RANGE | kGaveUpS);
        tc::fence_after();
        if (ok && warp < 4) {
            // softmax of head row tid over the tile, online across tiles
            const int valid = n_items - j * kNT < kNT ? n_items - j * kNT : kNT;
            uint32_t v[kNT];
            tc::tmem_ld32(tS + lane_off, v);
            tc::tmem_ld32(tS + lane_off + 32, v + 32);
            tc::tmem_wait_ld();
            float mx = -INFINITY;
#pragma unroll
            for (int cc = 0; cc < kNT; ++cc) {
                if (cc >= valid) v[cc] = __float_as_uint(-INFINITY);
                mx = fmaxf(mx, __uint_as_float(v[cc]));
            }
            const float m_new = fmaxf(m_run, mx == -INFINITY ? -INFINITY : mx * a.scale_log2);
            const float alpha = m_run == -INFINITY ? 0.f : tc::ex2(m_run - m_new);
            if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                // O holds the previous tiles (their PV has completed): scale it.  The
                // TMEM loads and stores are warp-collective, so the whole warp takes
                // this branch; each lane scales its own head row by its own alpha.
#pragma unroll
                for (int q = 0; q < kD / 32; ++q) {
                    uint32_t o[32];
                    tc::tmem_ld32(tO + lane_off + q * 32, o);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                    tc::tmem_st32(tO + lane_off + q * 32, o);
                }
                tc::tmem_wait_st();
            }
            const float nm = m_new == -INFINITY ? 0.f : -m_new;
            float sum = 0.f;
#pragma unroll
            for (int cc = 0; cc < kNT / 8; ++cc) {
                uint32_t pk[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float p0 = tc::ex2(fmaf(__uint_as_float(v[cc * 8 + 2 * e]), a.scale_log2, nm));
                    const float p1 = tc::ex2(fmaf(__uint_as_float(v[cc * 8 + 2 * e + 1]), a.scale_log2, nm));
                    sum += p0 + p1;
                    pk[e] = pack_bf16x2(p0, p1);
                }
                *reinterpret_cast<uint4 *>(sP + tid * 128 + ((cc ^ (tid & 7)) << 4)) =
                    make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
            l_run = l_run * alpha + sum;
            m_run = m_new;
        }
        tc::fence_proxy_async();
        tc::fence_before();
        __syncthreads();
        tc::fence_after();
        if (ok && tid == 0) {
            constexpr uint32_t idO = tc::idesc_bf16(kM, kD, false, true);
            const uint32_t aP = smem_u32(sP), aV = smem_u32(tV);
#pragma unroll
            for (int kk = 0; kk < kNT / 16; ++kk) {
                const uint64_t da = tc::desc_sw128(aP + kk * 32, 16, 1024);
                const uint64_t db = tc::desc_sw128(aV + kk * 16 * 128, kTBlk, 1024);
                tc::mma_bf16(tO, da, db, idO, (j > 0 || kk > 0) ? 1u : 0u);
            }
            tc::commit(&bar_o);
        }
        // the tiles' shared memory and O are reused by the next tile only after this PV
        const bool pv_ok = !ok || wait_phase(&bar_o, (unsigned)(j & 1));
        if (!pv_ok && tid == 0) raise_flag(FLAG_ATTN_RANGE | kGaveUpPV);
        ok = __syncthreads_and(ok && pv_ok) != 0;
        tc::fence_after();
    }
    // this chunk's partial: O (bf16, unnormalised), maximum and sum of each head
    if (warp < 4) {
        const int h = tid;
        if (ok && n_tiles > 0) {
#pragma unroll
            for (int q = 0; q < kD / 32; ++q) {
                uint32_t o[32];
                tc::tmem_ld32(tO + lane_off + q * 32, o);
                tc::tmem_wait_ld();
                if (h < a.H) {
                    __nv_bfloat16 *po = w.po + ((int64_t)c * a.H + h) * kD + q * 32;
#pragma unroll
                    for (int e = 0; e < 32; e += 8)
                        *reinterpret_cast<uint4 *>(po + e) = make_uint4(
                            pack_bf16x2(__uint_as_float(o[e]), __uint_as_float(o[e + 1])),
                            pack_bf16x2(__uint_as_float(o[e + 2]), __uint_as_float(o[e + 3])),
                            pack_bf16x2(__uint_as_float(o[e + 4]), __uint_as_float(o[e + 5])),
                            pack_bf16x2(__uint_as_float(o[e + 6]), __uint_as_float(o[e + 7])));
                }
            }
        }
        if (h < a.H) {
            float *pml = w.pml + (int64_t)c * 2 * a.H;
            pml[h] = (ok && n_tiles > 0) ? m_run : -INFINITY;  // -inf: nothing to merge from this chunk
            pml[a.H + h] = (ok && n_tiles > 0) ? l_run : 0.f;
        }
    }
    ok = ok && row_barrier(&w.bar[0], 3u * (unsigned)nch, 2, &s_misc[15]);

    // ---------------------------------------------------------------- P4
    // heads [c * hpc, (c + 1) * hpc) over the row's nch partials, one head at a time
    // by the whole CTA: warp g takes the partials g, g + 8, ... (all its loads in
    // flight at once), lane l the columns 4l..4l+3; the warps' sums are added in
    // warp order.
    if (ok) {
        const int hpc = (a.H + nch - 1) / nch;
        const int lane = tid & 31;
        float *s_red = reinterpret_cast<float *>(s_work);  // [8][132]
        for (int h = c * hpc; h < a.H && h < (c + 1) * hpc; ++h) {
            float mv = -INFINITY;
            for (int i = tid; i < nch; i += kThreads) mv = fmaxf(mv, __ldcg(w.pml + (int64_t)i * 2 * a.H + h));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mv = fmaxf(mv, __shfl_xor_sync(0xffffffffu, mv, o));
            if (lane == 0) s_red[warp * 132 + 128] = mv;
            __syncthreads();
            float M = -INFINITY;
#pragma unroll
            for (int g = 0; g < kThreads / 32; ++g) M = fmaxf(M, s_red[g * 132 + 128]);
            float L = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
            if (M != -INFINITY) {
                constexpr int U = 16;
                for (int i0 = warp; i0 < nch; i0 += U * (kThreads / 32)) {
                    float m_[U], l_[U];
                    uint2 ov[U];
#pragma unroll
                    for (int k = 0; k < U; ++k) {
                        const int i = i0 + k * (kThreads / 32);
                        m_[k] = -INFINITY;
                        if (i < nch) {
                            const float *pml = w.pml + (int64_t)i * 2 * a.H;
                            m_[k] = __ldcg(pml + h);
                            l_[k] = __ldcg(pml + a.H + h);
                            ov[k] = __ldcg(reinterpret_cast<const uint2 *>(w.po + ((int64_t)i * a.H + h) * kD) + lane);
                        }
                    }
#pragma unroll
                    for (int k = 0; k < U; ++k) {
                        if (m_[k] == -INFINITY) continue;  // nothing from that chunk (its O is not used)
                        const float wk = tc::ex2(m_[k] - M);
                        L = fmaf(wk, l_[k], L);
                        acc[0] = fmaf(wk, bf16_lo(ov[k].x), acc[0]);
                        acc[1] = fmaf(wk, bf16_hi(ov[k].x), acc[1]);
                        acc[2] = fmaf(wk, bf16_lo(ov[k].y), acc[2]);
                        acc[3] = fmaf(wk, bf16_hi(ov[k].y), acc[3]);
                    }
                }
            }
            __syncthreads();  // M read by every warp before the slots are reused
#pragma unroll
            for (int e = 0; e < 4; ++e) s_red[warp * 132 + 4 * lane + e] = acc[e];
            if (lane == 0) s_red[warp * 132 + 129] = L;
            __syncthreads();
            if (warp == 0) {
                float Lt = 0.f, o4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int g = 0; g < kThreads / 32; ++g) {
                    Lt += s_red[g * 132 + 129];
#pragma unroll
                    for (int e = 0; e < 4; ++e) o4[e] += s_red[g * 132 + 4 * lane + e];
                }
                const bool empty = !(Lt > 0.f);
                const float inv = empty ? 0.f : 1.f / Lt;
                uint2 pk;
                pk.x = pack_bf16x2(o4[0] * inv, o4[1] * inv);
                pk.y = pack_bf16x2(o4[2] * inv, o4[3] * inv);
                *reinterpret_cast<uint2 *>(a.out + ((int64_t)row * a.H + h) * kD + lane * 4) = pk;
                if (a.lse && lane == 0) a.lse[(int64_t)row * a.H + h] = empty ? -INFINITY : (M + log2f(Lt)) * kLn2;
            }
            __syncthreads();
        }
    }
    // the row's last CTA out returns its counters to zero for the next call
    __syncthreads();
    if (tid == 0 && ok) {
        __threadfence();
        if (atomicAdd(&w.bar[0], 1u) == 4u * (unsigned)nch - 1u) {
            w.bar[0] = 0;
            w.bar[1] = 0;
        }
    }
    // every MMA this CTA issued has completed before its TMEM is released
    if (tid == 0) {
        tc::commit(&bar_f);
        wait_phase(&bar_f, 0u);
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (warp == 0) tc::tmem_dealloc(tmem, 256);
}

int key_bits_for(int DI) {
    const long long maxkey = (long long)DI * 32640;
    int kb = 0;
    while ((1ll << kb) <= maxkey) ++kb;
    return kb;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

template <int LPE>
int occupancy(size_t smem) {
    static unsigned long long done = 0;
    if (smem_limit_once(decode_step_kernel<LPE>, 200 * 1024, done) != cudaSuccess) return 0;
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, decode_step_kernel<LPE>, kThreads, smem) != cudaSuccess)
        return 0;
    return occ;
}
int occupancy_for(int DI, size_t smem) {
    switch (DI) {
        case 16: return occupancy<1>(smem);
        case 32: return occupancy<2>(smem);
        case 64: return occupancy<4>(smem);
        case 128: return occupancy<8>(smem);
        default: return 0;
    }
}

}  // namespace

DecodeStepPlan plan_decode_step(int B, int H, int DI, int64_t E_cap, int num_sms) {
    DecodeStepPlan p{};
    p.ok = false;
    if (B <= 0 || E_cap <= 0 || (H != 64 && H != 128) || B > 65535) return p;
    if (DI != 16 && DI != 32 && DI != 64 && DI != 128) return p;
    p.rows = B;
    p.key_bits = key_bits_for(DI);
    p.shift1 = p.key_bits - 11;
    p.nb2 = 1 << p.shift1;
    if (p.nb2 * 4 > 16384) return p;
    // the smallest chunk (a multiple of 64 entries) whose launch is resident at once
    // (the occupancy query counts one CTA per SM for a kernel that allocates tensor
    // memory)
    for (int chunk = 256; chunk <= 16384; chunk += 64) {
        const int64_t C = (E_cap + chunk - 1) / chunk;
        if (C > kMaxChunks) continue;
        const size_t smem = 1024 + (size_t)kAttnBytes + 2 * (size_t)chunk * 4;
        if (smem > 200 * 1024) break;
        int occ = occupancy_for(DI, smem);
        if (occ <= 0) return p;
        if (occ > 2) occ = 2;
        if (C * B <= (int64_t)occ * num_sms) {
            p.chunk = chunk;
            p.ctas_per_row = (int)C;
            p.smem = smem;
            p.ok = true;
            break;
        }
    }
    if (!p.ok) return p;
    size_t off = 0;
    p.off_hist = off;
    off = align256(off + sizeof(unsigned) * kNB1 * (size_t)B);
    p.off_bar = off;
    off = align256(off + sizeof(unsigned) * 4 * (size_t)B);
    p.zero_bytes = off;
    p.off_rec = off;
    off = align256(off + sizeof(int) * (size_t)p.ctas_per_row * B);
    p.off_b1 = off;
    off = align256(off + sizeof(uint2) * (size_t)E_cap * B);
    p.off_po = off;
    off = align256(off + sizeof(__nv_bfloat16) * (size_t)p.ctas_per_row * H * kD * B);
    p.off_pml = off;
    off = align256(off + sizeof(float) * (size_t)p.ctas_per_row * 2 * H * B);
    p.total = off;
    return p;
}

template <int LPE>
static cudaError_t launch_lpe(const StepArgs &a, const DecodeStepPlan &p, void *ws, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.ctas_per_row, p.rows);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_step_kernel<LPE>, a, p, ws);
}

cudaError_t launch_decode_step(const DecodeStepCall &c, const DecodeStepPlan &p, void *ws, cudaStream_t s) {
    StepArgs a;
    a.qi = c.qi;
    a.qi_sb = c.qi_sb;
    a.ki = c.ki;
    a.ki_sb = c.ki_sb;
    a.E_cap = c.E_cap;
    a.B = c.B;
    a.DI = c.DI;
    a.m = c.m;
    a.topk = c.topk;
    a.H = c.H;
    a.window = c.window;
    a.idx_out = c.idx_out;
    a.cnt_out = c.cnt_out;
    a.q = static_cast<const __nv_bfloat16 *>(c.q);
    a.kc = static_cast<const __nv_bfloat16 *>(c.kc);
    a.vc = static_cast<const __nv_bfloat16 *>(c.vc);
    a.k_raw = static_cast<const __nv_bfloat16 *>(c.k_raw);
    a.v_raw = static_cast<const __nv_bfloat16 *>(c.v_raw);
    a.shared_kv = c.kc == c.vc && c.k_raw == c.v_raw;
    a.c_sb = c.c_sb;
    a.c_se = c.c_se;
    a.r_sb = c.r_sb;
    a.r_st = c.r_st;
    a.N_cap = c.N_cap;
    a.ctx = c.ctx;
    a.scale_log2 = c.scale * kLog2e;
    a.out = static_cast<__nv_bfloat16 *>(c.out);
    a.lse = c.lse;
    switch (c.DI) {
        case 16: return launch_lpe<1>(a, p, ws, s);
        case 32: return launch_lpe<2>(a, p, ws, s);
        case 64: return launch_lpe<4>(a, p, ws, s);
        case 128: return launch_lpe<8>(a, p, ws, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace hsa
