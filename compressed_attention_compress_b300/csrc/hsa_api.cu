// C-ABI layer: argument validation, workspace carving and launch sequencing.
// Every entry point enqueues on the caller's stream and never allocates,
// frees or synchronises (hsa_check excepted).
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <initializer_list>
#include <mutex>

#include "../../include/hsa.h"
#include "common.cuh"
#include "internal.h"

namespace hsa {
__device__ unsigned int g_device_flag = 0;
}

namespace {

thread_local char t_err[512] = "";

hsa_status_t fail(hsa_status_t st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_err, sizeof t_err, fmt, ap);
    va_end(ap);
    return st;
}

hsa_status_t ok() {
    t_err[0] = '\0';
    return HSA_OK;
}

struct DevInfo {
    int num_sms = 0;
    int major = 0, minor = 0;
};

hsa_status_t device_info(DevInfo &di) {
    static thread_local int cached_dev = -1;
    static thread_local DevInfo cached;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(HSA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev != cached_dev) {
        cudaDeviceProp pr;
        e = cudaGetDeviceProperties(&pr, dev);
        if (e != cudaSuccess) return fail(HSA_ERR_CUDA, "cudaGetDeviceProperties: %s", cudaGetErrorString(e));
        cached.num_sms = pr.multiProcessorCount;
        cached.major = pr.major;
        cached.minor = pr.minor;
        cached_dev = dev;
    }
    di = cached;
    if (di.major != 10) return fail(HSA_ERR_UNSUPPORTED, "device sm_%d%d: this library is built for sm_103a", di.major, di.minor);
    return HSA_OK;
}

hsa_status_t pending_error() {
    cudaError_t e = cudaPeekAtLastError();
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(HSA_ERR_CUDA, "pending CUDA error: %s", cudaGetErrorString(e));
    }
    return HSA_OK;
}

hsa_status_t launched(cudaError_t e, const char *what) {
    if (e != cudaSuccess) return fail(HSA_ERR_CUDA, "%s launch: %s", what, cudaGetErrorString(e));
    return ok();
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Every buffer must be memory the current device addresses directly: device
// memory of this device or managed memory.  Host memory (pageable or pinned) and
// another device's memory are refused on the host, before anything is enqueued,
// so that a wrong pointer never reaches a kernel.  Null pointers are skipped here
// (whether an argument may be null is checked by the caller).
hsa_status_t check_pointer(const void *p, const char *what) {
    if (!p) return HSA_OK;
    cudaPointerAttributes at;
    cudaError_t e = cudaPointerGetAttributes(&at, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(HSA_ERR_INVALID_ARG, "%s: not a CUDA-visible pointer (%s)", what, cudaGetErrorString(e));
    }
    if (at.type == cudaMemoryTypeManaged) return HSA_OK;
    if (at.type != cudaMemoryTypeDevice)
        return fail(HSA_ERR_INVALID_ARG, "%s: host memory (%s); pass device memory", what,
                    at.type == cudaMemoryTypeHost ? "pinned" : "pageable");
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(HSA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (at.device != dev)
        return fail(HSA_ERR_INVALID_ARG, "%s: memory of device %d, the current device is %d", what, at.device, dev);
    return HSA_OK;
}

struct NamedPtr {
    const void *p;
    const char *what;
};
hsa_status_t check_pointers(std::initializer_list<NamedPtr> ptrs) {
    for (const NamedPtr &x : ptrs) {
        hsa_status_t st = check_pointer(x.p, x.what);
        if (st != HSA_OK) return st;
    }
    return HSA_OK;
}

// Query rows (B * T) an indexer or attention call may take: the launch grids and
// per-row workspace offsets are sized in int for at most this many rows.
constexpr int64_t kMaxRows = 1ll << 24;
size_t esize(hsa_dtype_t dt) { return dt == HSA_BF16 ? 2 : 4; }
bool dtype_ok(hsa_dtype_t dt) { return dt == HSA_BF16 || dt == HSA_F32; }

// Rows of the indexer handled per launch group: bounded so that the stored keys
// stay under 1 GiB of workspace.
int index_group_rows(int rows, int64_t E_cap) {
    const int64_t per_row = (E_cap > 0 ? E_cap : 1) * 4 + 65536;
    int64_t g = (1ll << 30) / per_row;
    if (g < 1) g = 1;
    return (int)(g < rows ? g : rows);
}

// Decode attention split planning: the split size depends on the shape only, and
// the split count of a row on its own set size.
struct DecodePlan {
    int split, max_splits;
    size_t off_o, off_lse, total;
};
DecodePlan plan_decode(hsa_dtype_t dt, int B, int H, int d, int64_t E_cap, int m, int topk, int window,
                       bool dense, int num_sms) {
    DecodePlan p{};
    (void)m;
    if (dt == HSA_BF16 && !dense && hsa::decode_tc_shape(H, d, topk, window)) {
        // tcgen05 kernel: one cluster per (sequence, head group), partials in the workspace
        const hsa::DecodeTcWorkspace w = hsa::decode_tc_workspace(B, H, topk, window);
        p.split = -1;
        p.max_splits = 1;
        p.off_o = w.off_o;
        p.off_lse = w.off_ml;
        p.total = w.total;
        return p;
    }
    if (dt == HSA_BF16 && dense && hsa::decode_dense_tc_shape(B, H, d)) {
        // tcgen05 dense kernel: one partial per 128-item tile, merged in tile order
        const hsa::DecodeDenseWorkspace w = hsa::decode_dense_workspace(B, H, E_cap, window);
        p.split = -2;
        p.max_splits = 1;
        p.off_o = w.off_o;
        p.off_lse = w.off_ml;
        p.total = w.total;
        return p;
    }
    if (dt == HSA_BF16 && hsa::decode_cluster_supported(H, d)) {
        p.split = -1;  // cluster kernel: splits live in one cluster, no workspace
        p.max_splits = 1;
        p.total = 0;
        return p;
    }
    const int64_t max_items = (dense ? E_cap : (int64_t)topk) + window;
    p.split = hsa::attn_split_size(dt == HSA_BF16, dense, H, B, max_items, num_sms);
    if (p.split <= 0) {
        p.max_splits = 1;
        p.total = 0;
        return p;
    }
    p.max_splits = (int)((max_items + p.split - 1) / p.split);
    if (p.max_splits < 1) p.max_splits = 1;
    p.off_o = 0;
    p.off_lse = ((size_t)B * p.max_splits * H * d * sizeof(float) + 255) & ~(size_t)255;
    p.total = p.off_lse + (((size_t)B * p.max_splits * H * sizeof(float) + 255) & ~(size_t)255);
    return p;
}

hsa_status_t check_attn_common(const void *q, hsa_dtype_t dt, int B, int T, int H, int d, const void *kc,
                               const void *vc, int64_t c_sb, int64_t c_se, int64_t E_cap, int m,
                               const int32_t *idx, int topk, const void *k_raw, const void *v_raw, int64_t r_sb,
                               int64_t r_st, int64_t N_cap, int window, const int64_t *pos, const void *out) {
    if (!dtype_ok(dt)) return fail(HSA_ERR_UNSUPPORTED, "dtype %d", (int)dt);
    if (B < 0 || T < 0 || H <= 0 || d <= 0 || m <= 0 || window < 0 || E_cap < 0 || N_cap < 0)
        return fail(HSA_ERR_INVALID_ARG, "negative or zero size (B=%d T=%d H=%d d=%d m=%d window=%d)", B, T, H, d, m,
                    window);
    if (idx && topk <= 0) return fail(HSA_ERR_INVALID_ARG, "topk must be positive when idx is given");
    if (B * (int64_t)T == 0) return HSA_OK;
    if (!q || !out || !pos) return fail(HSA_ERR_INVALID_ARG, "null q/out/position pointer");
    if (window > 0 && (!k_raw || !v_raw)) return fail(HSA_ERR_INVALID_ARG, "null raw cache with window > 0");
    if (E_cap > 0 && (!kc || !vc)) return fail(HSA_ERR_INVALID_ARG, "null compressed cache");
    if (dt == HSA_BF16) {
        if (d != 64 && d != 128) return fail(HSA_ERR_UNSUPPORTED, "bf16 path supports d in {64,128}, got %d", d);
        if (H % 16 != 0 || H > 128) return fail(HSA_ERR_UNSUPPORTED, "bf16 path needs H a multiple of 16 up to 128, got %d", H);
    } else {
        if (d % 32 != 0 || d > 256) return fail(HSA_ERR_UNSUPPORTED, "fp32 path needs d a multiple of 32 up to 256, got %d", d);
    }
    const size_t es = esize(dt);
    const int64_t vec = 16 / (int64_t)es;
    if (!aligned16(q) || !aligned16(out) || (kc && !aligned16(kc)) || (vc && !aligned16(vc)) ||
        (k_raw && !aligned16(k_raw)) || (v_raw && !aligned16(v_raw)))
        return fail(HSA_ERR_UNSUPPORTED, "q, out and caches must be 16-byte aligned");
    if (c_sb % vec || c_se % vec || r_sb % vec || r_st % vec)
        return fail(HSA_ERR_UNSUPPORTED, "cache strides must be multiples of 16 bytes");
    if (c_se < d || r_st < d || c_sb < 0 || r_sb < 0) return fail(HSA_ERR_INVALID_ARG, "cache strides overlap rows");
    if (B * (int64_t)T > kMaxRows) return fail(HSA_ERR_UNSUPPORTED, "B*T above 2^24");
    return check_pointers({{q, "q"}, {kc, "kc"}, {vc, "vc"}, {idx, "idx"}, {k_raw, "k_raw"}, {v_raw, "v_raw"},
                           {pos, "positions"}, {out, "out"}});
}

}  // namespace

extern "C" {

const char *hsa_last_error(void) { return t_err; }

int hsa_version(void) { return 200; }

hsa_status_t hsa_check_pointer(const void *p) {
    if (!p) return fail(HSA_ERR_INVALID_ARG, "null pointer");
    hsa_status_t st = check_pointer(p, "pointer");
    return st == HSA_OK ? ok() : st;
}

hsa_status_t hsa_check(hsa_stream_t stream) {
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(HSA_ERR_CUDA, "stream: %s", cudaGetErrorString(e));
    unsigned flag = 0;
    e = cudaMemcpyFromSymbol(&flag, hsa::g_device_flag, sizeof flag);
    if (e != cudaSuccess) return fail(HSA_ERR_CUDA, "reading device flag: %s", cudaGetErrorString(e));
    if (flag) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(hsa::g_device_flag, &zero, sizeof zero);
        if (e != cudaSuccess) return fail(HSA_ERR_CUDA, "clearing device flag: %s", cudaGetErrorString(e));
        return fail(HSA_ERR_DEVICE_FLAG, "device range flag 0x%x (1=compress 2=index 4=attn range 8=attn index)", flag);
    }
    return ok();
}

hsa_status_t hsa_compress(const void *k, const void *v, hsa_dtype_t dt, int B, int d, int64_t in_sb, int64_t in_st,
                          int64_t N_cap, const int64_t *tok_begin, const int64_t *tok_end, int64_t max_blocks,
                          const float *w, int m, void *kc, void *vc, int64_t out_sb, int64_t out_se, int64_t E_cap,
                          hsa_stream_t stream) {
    if (!dtype_ok(dt)) return fail(HSA_ERR_UNSUPPORTED, "dtype %d", (int)dt);
    if (B < 0 || d <= 0 || m <= 0 || max_blocks < 0 || N_cap < 0 || E_cap < 0)
        return fail(HSA_ERR_INVALID_ARG, "bad size (B=%d d=%d m=%d max_blocks=%lld)", B, d, m, (long long)max_blocks);
    if (m > 4096) return fail(HSA_ERR_UNSUPPORTED, "m > 4096");
    if (B == 0 || max_blocks == 0) return ok();
    if (!k || !v || !kc || !vc || !tok_begin || !tok_end || !w) return fail(HSA_ERR_INVALID_ARG, "null pointer");
    const int64_t vec = 16 / (int64_t)esize(dt);
    if (d % vec || d > 512) return fail(HSA_ERR_UNSUPPORTED, "d must be a multiple of %lld and <= 512", (long long)vec);
    if (!aligned16(k) || !aligned16(v) || !aligned16(kc) || !aligned16(vc))
        return fail(HSA_ERR_UNSUPPORTED, "tensors must be 16-byte aligned");
    if (in_sb % vec || in_st % vec || out_sb % vec || out_se % vec)
        return fail(HSA_ERR_UNSUPPORTED, "strides must be multiples of 16 bytes");
    if (in_st < d || out_se < d) return fail(HSA_ERR_INVALID_ARG, "row strides overlap rows");
    DevInfo di;
    hsa_status_t st = device_info(di);
    if (st != HSA_OK) return st;
    if ((st = check_pointers({{k, "k"}, {v, "v"}, {tok_begin, "tok_begin"}, {tok_end, "tok_end"}, {w, "w"},
                              {kc, "kc"}, {vc, "vc"}})) != HSA_OK)
        return st;
    if ((st = pending_error()) != HSA_OK) return st;
    hsa::CompressArgs a{k, v, B, d, in_sb, in_st, N_cap, tok_begin, tok_end, max_blocks, w, m, kc, vc, out_sb, out_se, E_cap};
    return launched(hsa::launch_compress(a, dt == HSA_BF16, di.num_sms, reinterpret_cast<cudaStream_t>(stream)),
                    "compress");
}

hsa_status_t hsa_compress_v4(const void *k, hsa_dtype_t dt, int B, int d, int64_t in_sb, int64_t in_st,
                             int64_t N_cap, const int64_t *tok_begin, const int64_t *tok_end, int64_t max_blocks,
                             const float *w, int m, void *kc, int64_t out_sb, int64_t out_se, int64_t E_cap,
                             const float *gamma, float eps, int rope_dims, float theta, hsa_stream_t stream) {
    if (!dtype_ok(dt)) return fail(HSA_ERR_UNSUPPORTED, "dtype %d", (int)dt);
    if (B < 0 || d <= 0 || m <= 0 || max_blocks < 0 || N_cap < 0 || E_cap < 0)
        return fail(HSA_ERR_INVALID_ARG, "bad size (B=%d d=%d m=%d max_blocks=%lld)", B, d, m, (long long)max_blocks);
    if (m > 4096) return fail(HSA_ERR_UNSUPPORTED, "m > 4096");
    if (d % 64 || d > 512) return fail(HSA_ERR_UNSUPPORTED, "d must be a multiple of 64 up to 512, got %d", d);
    if (rope_dims < 0 || rope_dims % 2 || rope_dims > d || !(theta > 0.f) || !(eps >= 0.f))
        return fail(HSA_ERR_INVALID_ARG, "rope_dims must be even in [0, d]; theta > 0, eps >= 0");
    if (rope_dims > hsa::kMaxRopeDims) return fail(HSA_ERR_UNSUPPORTED, "rope_dims above %d", hsa::kMaxRopeDims);
    if (B > 65535) return fail(HSA_ERR_UNSUPPORTED, "B above 65535");
    if (B == 0 || max_blocks == 0) return ok();
    if (!k || !kc || !tok_begin || !tok_end || !w) return fail(HSA_ERR_INVALID_ARG, "null pointer");
    if (in_st < d || out_se < d) return fail(HSA_ERR_INVALID_ARG, "row strides overlap rows");
    DevInfo di;
    hsa_status_t st = device_info(di);
    if (st != HSA_OK) return st;
    if ((st = check_pointers({{k, "k"}, {tok_begin, "tok_begin"}, {tok_end, "tok_end"}, {w, "w"}, {kc, "kc"},
                              {gamma, "gamma"}})) != HSA_OK)
        return st;
    if ((st = pending_error()) != HSA_OK) return st;
    hsa::CompressArgs a{k, k, B, d, in_sb, in_st, N_cap, tok_begin, tok_end, max_blocks, w, m, kc, kc, out_sb, out_se, E_cap};
    hsa::CompressV4Args v{gamma, eps, rope_dims, {}};
    for (int i = 0; i < rope_dims / 2; ++i) v.inv_freq[i] = pow((double)theta, -2.0 * i / rope_dims);
    return launched(hsa::launch_compress_v4(a, v, dt == HSA_BF16, reinterpret_cast<cudaStream_t>(stream)),
                    "compress_v4");
}

hsa_status_t hsa_compress_learned(const void *k, const void *v, hsa_dtype_t dt, int B, int d, int64_t in_sb,
                                  int64_t in_st, int64_t N_cap, const int64_t *tok_begin, const int64_t *tok_end,
                                  int64_t max_blocks, const float *u, const float *bias, int m, int L, void *kc,
                                  void *vc, int64_t out_sb, int64_t out_se, int64_t E_cap, hsa_stream_t stream) {
    if (!dtype_ok(dt)) return fail(HSA_ERR_UNSUPPORTED, "dtype %d", (int)dt);
    if (B < 0 || d <= 0 || m <= 0 || L < 1 || max_blocks < 0 || N_cap < 0 || E_cap < 0)
        return fail(HSA_ERR_INVALID_ARG, "bad size (B=%d d=%d m=%d L=%d)", B, d, m, L);
    if (L > 1024 || m > 4096) return fail(HSA_ERR_UNSUPPORTED, "L above 1024 or m above 4096");
    if (d % 32 || d > 512) return fail(HSA_ERR_UNSUPPORTED, "d must be a multiple of 32 up to 512");
    if (B == 0 || max_blocks == 0) return ok();
    if (!k || !v || !kc || !vc || !tok_begin || !tok_end || !u || !bias) return fail(HSA_ERR_INVALID_ARG, "null pointer");
    if (in_st < d || out_se < d) return fail(HSA_ERR_INVALID_ARG, "row strides overlap rows");
    const int64_t vec = 16 / (int64_t)esize(dt);
    if (!aligned16(k) || !aligned16(v) || in_sb % vec || in_st % vec)
        return fail(HSA_ERR_UNSUPPORTED, "k, v and their strides must be 16-byte aligned");
    DevInfo di;
    hsa_status_t st = device_info(di);
    if (st != HSA_OK) return st;
    if ((st = check_pointers({{k, "k"}, {v, "v"}, {tok_begin, "tok_begin"}, {tok_end, "tok_end"}, {u, "u"},
                              {bias, "bias"}, {kc, "kc"}, {vc, "vc"}})) != HSA_OK)
        return st;
    if ((st = pending_error()) != HSA_OK) return st;
    hsa::CompressLearnedArgs a{k, v, B, d, in_sb, in_st, N_cap, tok_begin, tok_end, max_blocks, u, bias, m, L,
                               kc, vc, out_sb, out_se, E_cap};
    return launched(hsa::launch_compress_learned(a, dt == HSA_BF16, reinterpret_cast<cudaStream_t>(stream)),
                    "compress_learned");
}

hsa_status_t hsa_compress_append(const void *k_new, const void *v_new, hsa_dtype_t dt, int B, int T, int d,
                                 int64_t new_sb, int64_t new_st, const int64_t *pos0, const float *w, int m,
                                 float *state_k, float *state_v, int64_t state_sb, void *kc, void *vc, int64_t out_sb,
                                 int64_t out_se, int64_t E_cap, hsa_stream_t stream) {
    if (!dtype_ok(dt)) return fail(HSA_ERR_UNSUPPORTED, "dtype %d", (int)dt);
    if (B < 0 || T < 0 || d <= 0 || m <= 0 || E_cap < 0) return fail(HSA_ERR_INVALID_ARG, "bad size");
    if (m > 4096) return fail(HSA_ERR_UNSUPPORTED, "m > 4096");
    if (B == 0 || T == 0) return ok();
    if (!k_new || !v_new || !pos0 || !w || !state_k || !state_v || !kc || !vc)
        return fail(HSA_ERR_INVALID_ARG, "null pointer");
    const int64_t vec = 16 / (int64_t)esize(dt);
    if (d % vec || d > 512) return fail(HSA_ERR_UNSUPPORTED, "d must be a multiple of %lld and <= 512", (long long)vec);
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(kc) || !aligned16(vc) || !aligned16(state_k) ||
        !aligned16(state_v))
        return fail(HSA_ERR_UNSUPPORTED, "tensors must be 16-byte aligned");
    if (new_sb % vec || new_st % vec || out_sb % vec || out_se % vec || state_sb % 4)
        return fail(HSA_ERR_UNSUPPORTED, "strides must be multiples of 16 bytes");
    if (new_st < d || out_se < d || state_sb < d) return fail(HSA_ERR_INVALID_ARG, "row strides overlap rows");
    DevInfo di;
    hsa_status_t st = device_info(di);
    if (st != HSA_OK) return st;
    if ((st = check_pointers({{k_new, "k_new"}, {v_new, "v_new"}, {pos0, "pos0"}, {w, "w"}, {state_k, "state_k"},
                              {state_v, "state_v"}, {kc, "kc"}, {vc, "vc"}})) != HSA_OK)
        return st;
    if ((st = pending_error()) != HSA_OK) return st;
    hsa::CompressAppendArgs a{k_new, v_new, B, T, d, new_sb, new_st, pos0, w, m, state_k, state_v, state_sb,
                              kc, vc, out_sb, out_se, E_cap};
    return launched(hsa::launch_compress_append(a, dt == HSA_BF16, reinterpret_cast<cudaStream_t>(stream)),
                    "compress_append");
}

}  // extern "C"

namespace {
// Decode-shaped calls (all CTAs of the rows resident at once) take the fused
// cooperative kernel; larger row counts take the two-kernel path in groups.
struct IndexChoice {
    bool fused, prefill;
    hsa::FusedIndexPlan fp;
    hsa::PrefillIndexPlan pp;
    hsa::IndexPlan tp;
    int group;
    size_t bytes;
};
// Decode shapes take the fused cooperative kernel; many query rows per sequence
// take the tensor-core path; what remains takes the two-kernel dp4a path.
IndexChoice choose_index(int B, int T, int DI, int64_t E_cap, int topk, int num_sms) {
    IndexChoice c{};
    const int rows = B * T;
    c.fp = hsa::plan_index_fused(rows, DI, E_cap, num_sms);
    if (c.fp.ok) {
        c.fused = true;
        c.bytes = c.fp.total;
        return c;
    }
    c.pp = hsa::plan_index_prefill(B, T, DI, E_cap, topk, num_sms);
    if (c.pp.ok) {
        c.prefill = true;
        c.bytes = c.pp.total;
        return c;
    }
    c.group = index_group_rows(rows, E_cap);
    c.tp = hsa::plan_index(c.group, DI, E_cap, topk, num_sms);
    c.bytes = c.tp.total;
    return c;
}
}  // namespace

extern "C" {

hsa_status_t hsa_index_topk_workspace_size(int B, int T, int DI, int64_t E_cap, int topk, size_t *bytes) {
    if (!bytes) return fail(HSA_ERR_INVALID_ARG, "null bytes");
    if (B < 0 || T < 0 || E_cap < 0 || topk <= 0 || DI <= 0) return fail(HSA_ERR_INVALID_ARG, "bad size");
    if (DI != 16 && DI != 32 && DI != 64 && DI != 128)
        return fail(HSA_ERR_UNSUPPORTED, "indexer dim must be 16, 32, 64 or 128, got %d", DI);
    if (B * (int64_t)T > kMaxRows) return fail(HSA_ERR_UNSUPPORTED, "B*T above 2^24");
    if (E_cap > (int64_t)1 << 30) return fail(HSA_ERR_UNSUPPORTED, "E_cap above 2^30");
    DevInfo di;
    hsa_status_t st = device_info(di);
    if (st != HSA_OK) return st;
    const int rows = B * T;
    if (rows == 0 || E_cap == 0) {
        *bytes = 0;
        return ok();
    }
    *bytes = choose_index(B, T, DI, E_cap, topk, di.num_sms).bytes;
    return ok();
}

hsa_status_t hsa_index_topk(const int8_t *q_idx, int64_t q_sb, int64_t q_st, const int8_t *k_idx, int64_t k_sb,
                            int64_t k_se, int64_t E_cap, int B, int T, int DI, const int64_t *q_pos0, int m, int topk,
                            int32_t *idx_out, int32_t *cnt_out, void *ws, size_t ws_bytes, hsa_stream_t stream) {
    if (B < 0 || T < 0 || E_cap < 0 || m <= 0) return fail(HSA_ERR_INVALID_ARG, "bad size");
    if (topk <= 0 || topk > 4096) return fail(HSA_ERR_UNSUPPORTED, "topk must be in [1, 4096], got %d", topk);
    if (DI != 16 && DI != 32 && DI != 64 && DI != 128)
        return fail(HSA_ERR_UNSUPPORTED, "indexer dim must be 16, 32, 64 or 128, got %d", DI);
    if (B * (int64_t)T > kMaxRows) return fail(HSA_ERR_UNSUPPORTED, "B*T above 2^24");
    const int rows = B * T;
    if (rows == 0) return ok();
    if (!q_idx || !k_idx || !q_pos0 || !idx_out || !cnt_out) return fail(HSA_ERR_INVALID_ARG, "null pointer");
    if (E_cap > (int64_t)1 << 30) return fail(HSA_ERR_UNSUPPORTED, "E_cap above 2^30");
    if (!aligned16(q_idx) || !aligned16(k_idx) || q_sb % 16 || q_st % 16 || k_sb % 16 || k_se % 16)
        return fail(HSA_ERR_UNSUPPORTED, "indexer tensors and strides must be 16-byte aligned");
    if (k_se < DI || q_st < DI) return fail(HSA_ERR_INVALID_ARG, "indexer strides overlap rows");
    DevInfo di;
    hsa_status_t st = device_info(di);
    if (st != HSA_OK) return st;
    if ((st = check_pointers({{q_idx, "q_idx"}, {k_idx, "k_idx"}, {q_pos0, "q_pos0"}, {idx_out, "idx_out"},
                              {cnt_out, "cnt_out"}})) != HSA_OK)
        return st;
    hsa::IndexArgs a{q_idx, q_sb, q_st, k_idx, k_sb, k_se, E_cap, B, T, DI, q_pos0, m, topk, idx_out, cnt_out};
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (E_cap == 0) {
        // no entry can be visible: everything is padding
        if ((st = pending_error()) != HSA_OK) return st;
        cudaError_t e = cudaMemsetAsync(idx_out, 0xff, sizeof(int32_t) * (size_t)rows * topk, s);
        if (e == cudaSuccess) e = cudaMemsetAsync(cnt_out, 0, sizeof(int32_t) * (size_t)rows, s);
        return launched(e, "index (empty)");
    }
    const IndexChoice ch = choose_index(B, T, DI, E_cap, topk, di.num_sms);
    if (!ws || ws_bytes < ch.bytes)
        return fail(HSA_ERR_WORKSPACE, "index workspace needs %zu bytes, got %zu", ch.bytes, ws_bytes);
    if ((reinterpret_cast<uintptr_t>(ws) & 255) != 0) return fail(HSA_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    if ((st = check_pointer(ws, "workspace")) != HSA_OK) return st;
    if ((st = pending_error()) != HSA_OK) return st;
    if (ch.fused) return launched(hsa::launch_index_fused(a, ch.fp, ws, s), "index_topk (fused)");
    if (ch.prefill) return launched(hsa::launch_index_prefill(a, ch.pp, ws, di.num_sms, s), "index_topk (tensor cores)");
    for (int r0 = 0; r0 < rows; r0 += ch.group) {
        cudaError_t e = hsa::launch_index_topk(a, ch.tp, ws, r0, s);
        if (e != cudaSuccess) return launched(e, "index_topk");
    }
    return ok();
}

hsa_status_t hsa_attn_decode_workspace_size(hsa_dtype_t dt, int B, int H, int d, int64_t E_cap, int m, int topk,
                                            int window, size_t *bytes) {
    if (!bytes) return fail(HSA_ERR_INVALID_ARG, "null bytes");
    if (B < 0 || H <= 0 || d <= 0 || E_cap < 0 || window < 0) return fail(HSA_ERR_INVALID_ARG, "bad size");
    DevInfo di;
    hsa_status_t st = device_info(di);
    if (st != HSA_OK) return st;
    // topk <= 0 means dense (HCA)
    const DecodePlan p = plan_decode(dt, B, H, d, E_cap, m, topk, window, topk <= 0, di.num_sms);
    *bytes = p.total;
    return ok();
}

hsa_status_t hsa_attn_decode(const void *q, hsa_dtype_t dt, int B, int H, int d, const void *kc, const void *vc,
                             int64_t c_sb, int64_t c_se, int64_t E_cap, int m, const int32_t *idx, const int32_t *cnt,
                             int topk, const void *k_raw, const void *v_raw, int64_t r_sb, int64_t r_st,
                             int64_t N_cap, int window, const int64_t *ctx_len, float scale, void *out, float *lse,
                             void *ws, size_t ws_bytes, hsa_stream_t stream) {
    hsa_status_t st = check_attn_common(q, dt, B, 1, H, d, kc, vc, c_sb, c_se, E_cap, m, idx, topk, k_raw, v_raw,
                                        r_sb, r_st, N_cap, window, ctx_len, out);
    if (st != HSA_OK) return st;
    if (B == 0) return ok();
    DevInfo di;
    if ((st = device_info(di)) != HSA_OK) return st;
    const bool dense = idx == nullptr;
    const DecodePlan p = plan_decode(dt, B, H, d, E_cap, m, dense ? 0 : topk, window, dense, di.num_sms);
    if (p.total > 0 && (!ws || ws_bytes < p.total))
        return fail(HSA_ERR_WORKSPACE, "decode workspace needs %zu bytes, got %zu", p.total, ws_bytes);
    if (p.total > 0 && (reinterpret_cast<uintptr_t>(ws) & 255) != 0)
        return fail(HSA_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    if ((st = check_pointers({{cnt, "cnt"}, {lse, "lse"}, {p.total > 0 ? ws : nullptr, "workspace"}})) != HSA_OK)
        return st;
    if ((st = pending_error()) != HSA_OK) return st;
    hsa::AttnArgs a{};
    a.q = q; a.rows = B; a.T = 1; a.H = H; a.d = d;
    a.kc = kc; a.vc = vc; a.c_sb = c_sb; a.c_se = c_se; a.E_cap = E_cap; a.m = m;
    a.idx = idx; a.cnt = cnt; a.topk = dense ? 0 : topk;
    a.k_raw = k_raw; a.v_raw = v_raw; a.r_sb = r_sb; a.r_st = r_st; a.N_cap = N_cap; a.window = window;
    a.pos = ctx_len; a.pos_is_ctx = 1; a.scale = scale; a.out = out; a.lse = lse;
    a.shared_kv = kc == vc && k_raw == v_raw;
    a.split = p.split; a.max_splits = p.max_splits;
    a.part_o = p.total ? reinterpret_cast<float *>(static_cast<char *>(ws) + p.off_o) : nullptr;
    a.part_lse = p.total ? reinterpret_cast<float *>(static_cast<char *>(ws) + p.off_lse) : nullptr;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (p.split == -2) return launched(hsa::launch_attn_decode_dense_tc(a, di.num_sms, s), "attn_decode (tcgen05 dense)");
    if (p.split < 0) {
        if (hsa::decode_tc_supported(a)) return launched(hsa::launch_attn_decode_tc(a, s), "attn_decode (tcgen05)");
        return launched(hsa::launch_attn_decode_cluster(a, s), "attn_decode (cluster)");
    }
    cudaError_t e = dt == HSA_BF16 ? hsa::launch_attn_bf16(a, s) : hsa::launch_attn_f32(a, s);
    if (e != cudaSuccess) return launched(e, "attn_decode");
    return launched(hsa::launch_attn_merge(a, dt == HSA_BF16, s), "attn_merge");
}

hsa_status_t hsa_attn_decode_v4(const void *q, hsa_dtype_t dt, int B, int H, int d, const void *kc, const void *vc,
                                int64_t c_sb, int64_t c_se, int64_t E_cap, int m, const int32_t *idx,
                                const int32_t *cnt, int topk, const void *k_raw, const void *v_raw, int64_t r_sb,
                                int64_t r_st, int64_t N_cap, int window, const int64_t *ctx_len, float scale,
                                const float *gamma_q, float eps, int rope_dims, float theta, const float *sink,
                                void *out, float *lse, void *ws, size_t ws_bytes, hsa_stream_t stream) {
    hsa_status_t st = check_attn_common(q, dt, B, 1, H, d, kc, vc, c_sb, c_se, E_cap, m, idx, topk, k_raw, v_raw,
                                        r_sb, r_st, N_cap, window, ctx_len, out);
    if (st != HSA_OK) return st;
    if (rope_dims < 0 || rope_dims % 2 || rope_dims > d || !(theta > 0.f) || !(eps >= 0.f))
        return fail(HSA_ERR_INVALID_ARG, "rope_dims must be even in [0, d]; theta > 0, eps >= 0");
    if (B == 0) return ok();
    if (dt != HSA_BF16 || d != 128 || !idx || !hsa::decode_tc_shape(H, d, topk, window))
        return fail(HSA_ERR_UNSUPPORTED,
                    "hsa_attn_decode_v4 runs on the tensor-core CSA decode path: bf16, d = 128, H a multiple of 64, "
                    "selected entries (idx), topk + window <= 2048");
    DevInfo di;
    if ((st = device_info(di)) != HSA_OK) return st;
    const DecodePlan p = plan_decode(dt, B, H, d, E_cap, m, topk, window, false, di.num_sms);
    if (p.total > 0 && (!ws || ws_bytes < p.total))
        return fail(HSA_ERR_WORKSPACE, "decode workspace needs %zu bytes, got %zu", p.total, ws_bytes);
    if (p.total > 0 && (reinterpret_cast<uintptr_t>(ws) & 255) != 0)
        return fail(HSA_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    if ((st = check_pointers({{cnt, "cnt"}, {lse, "lse"}, {p.total > 0 ? ws : nullptr, "workspace"},
                              {gamma_q, "gamma_q"}, {sink, "sink"}})) != HSA_OK)
        return st;
    if ((st = pending_error()) != HSA_OK) return st;
    hsa::AttnArgs a{};
    a.q = q; a.rows = B; a.T = 1; a.H = H; a.d = d;
    a.kc = kc; a.vc = vc; a.c_sb = c_sb; a.c_se = c_se; a.E_cap = E_cap; a.m = m;
    a.idx = idx; a.cnt = cnt; a.topk = topk;
    a.k_raw = k_raw; a.v_raw = v_raw; a.r_sb = r_sb; a.r_st = r_st; a.N_cap = N_cap; a.window = window;
    a.pos = ctx_len; a.pos_is_ctx = 1; a.scale = scale; a.out = out; a.lse = lse;
    a.shared_kv = kc == vc && k_raw == v_raw;
    a.split = p.split; a.max_splits = p.max_splits;
    a.part_o = p.total ? reinterpret_cast<float *>(static_cast<char *>(ws) + p.off_o) : nullptr;
    a.part_lse = p.total ? reinterpret_cast<float *>(static_cast<char *>(ws) + p.off_lse) : nullptr;
    a.v4 = 1;
    a.gamma_q = gamma_q;
    a.sink = sink;
    a.eps = eps;
    a.rope_dims = rope_dims;
    for (int k = 0; k < rope_dims / 2; ++k) a.inv_freq[k] = pow((double)theta, -2.0 * k / rope_dims);
    if (p.split >= 0 || !hsa::decode_tc_supported(a))
        return fail(HSA_ERR_UNSUPPORTED, "hsa_attn_decode_v4: this shape does not take the tensor-core decode path");
    return launched(hsa::launch_attn_decode_tc(a, reinterpret_cast<cudaStream_t>(stream)), "attn_decode_v4");
}

hsa_status_t hsa_decode_csa_workspace_size(int B, int H, int d, int DI, int64_t E_cap, size_t *bytes) {
    if (!bytes) return fail(HSA_ERR_INVALID_ARG, "null bytes");
    if (B < 0 || H <= 0 || d <= 0 || DI <= 0 || E_cap < 0) return fail(HSA_ERR_INVALID_ARG, "bad size");
    if (B == 0) {
        *bytes = 0;
        return ok();
    }
    DevInfo di;
    hsa_status_t st = device_info(di);
    if (st != HSA_OK) return st;
    if (d != 128) return fail(HSA_ERR_UNSUPPORTED, "hsa_decode_csa needs d = 128, got %d", d);
    const hsa::DecodeStepPlan pl = hsa::plan_decode_step(B, H, DI, E_cap, di.num_sms);
    if (!pl.ok)
        return fail(HSA_ERR_UNSUPPORTED, "hsa_decode_csa: B=%d H=%d DI=%d E_cap=%lld does not fit one resident launch "
                    "(use hsa_index_topk and hsa_attn_decode)", B, H, DI, (long long)E_cap);
    *bytes = pl.total;
    return ok();
}

hsa_status_t hsa_decode_csa(const int8_t *q_idx, int64_t qi_sb, const int8_t *k_idx, int64_t k_sb, int64_t k_se,
                            int64_t E_cap, int DI, int m, int topk, int32_t *idx_out, int32_t *cnt_out, const void *q,
                            hsa_dtype_t dt, int B, int H, int d, const void *kc, const void *vc, int64_t c_sb,
                            int64_t c_se, const void *k_raw, const void *v_raw, int64_t r_sb, int64_t r_st,
                            int64_t N_cap, int window, const int64_t *ctx_len, float scale, void *out, float *lse,
                            void *ws, size_t ws_bytes, hsa_stream_t stream) {
    if (B < 0 || H <= 0 || d <= 0 || DI <= 0 || E_cap < 0 || m <= 0 || window < 0 || N_cap < 0)
        return fail(HSA_ERR_INVALID_ARG, "bad size");
    if (dt != HSA_BF16 || d != 128 || (H != 64 && H != 128))
        return fail(HSA_ERR_UNSUPPORTED, "hsa_decode_csa needs bf16, d = 128 and H in {64, 128}");
    if (topk <= 0 || topk > 4096) return fail(HSA_ERR_UNSUPPORTED, "topk must be in [1, 4096], got %d", topk);
    if (DI != 16 && DI != 32 && DI != 64 && DI != 128)
        return fail(HSA_ERR_UNSUPPORTED, "indexer dim must be 16, 32, 64 or 128, got %d", DI);
    if (B == 0) return ok();
    if (B > 65535) return fail(HSA_ERR_UNSUPPORTED, "more than 65535 sequences");
    if (E_cap == 0) return fail(HSA_ERR_UNSUPPORTED, "no compressed entries: use hsa_attn_decode");
    if (E_cap > (int64_t)1 << 30) return fail(HSA_ERR_UNSUPPORTED, "E_cap above 2^30");
    if (!q_idx || !k_idx || !idx_out || !cnt_out || !q || !kc || !vc || !ctx_len || !out)
        return fail(HSA_ERR_INVALID_ARG, "null pointer");
    if (window > 0 && (!k_raw || !v_raw)) return fail(HSA_ERR_INVALID_ARG, "null raw cache with window > 0");
    if (k_se != DI) return fail(HSA_ERR_UNSUPPORTED, "hsa_decode_csa needs contiguous indexer rows (k_se == DI)");
    if (!aligned16(q_idx) || !aligned16(k_idx) || qi_sb % 16 || k_sb % 16)
        return fail(HSA_ERR_UNSUPPORTED, "indexer tensors and strides must be 16-byte aligned");
    if (!aligned16(q) || !aligned16(out) || !aligned16(kc) || !aligned16(vc) || (k_raw && !aligned16(k_raw)) ||
        (v_raw && !aligned16(v_raw)))
        return fail(HSA_ERR_UNSUPPORTED, "q, out and caches must be 16-byte aligned");
    if (c_sb % 8 || c_se % 8 || r_sb % 8 || r_st % 8) return fail(HSA_ERR_UNSUPPORTED, "cache strides must be multiples of 16 bytes");
    if (c_se < d || r_st < d || c_sb < 0 || r_sb < 0) return fail(HSA_ERR_INVALID_ARG, "cache strides overlap rows");
    DevInfo di;
    hsa_status_t st = device_info(di);
    if (st != HSA_OK) return st;
    const hsa::DecodeStepPlan pl = hsa::plan_decode_step(B, H, DI, E_cap, di.num_sms);
    if (!pl.ok)
        return fail(HSA_ERR_UNSUPPORTED, "hsa_decode_csa: B=%d H=%d DI=%d E_cap=%lld does not fit one resident launch "
                    "(use hsa_index_topk and hsa_attn_decode)", B, H, DI, (long long)E_cap);
    if (!ws || ws_bytes < pl.total) return fail(HSA_ERR_WORKSPACE, "decode workspace needs %zu bytes, got %zu", pl.total, ws_bytes);
    if ((reinterpret_cast<uintptr_t>(ws) & 255) != 0) return fail(HSA_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    if ((st = check_pointers({{q_idx, "q_idx"}, {k_idx, "k_idx"}, {idx_out, "idx_out"}, {cnt_out, "cnt_out"}, {q, "q"},
                              {kc, "kc"}, {vc, "vc"}, {k_raw, "k_raw"}, {v_raw, "v_raw"}, {ctx_len, "ctx_len"},
                              {out, "out"}, {lse, "lse"}, {ws, "workspace"}})) != HSA_OK)
        return st;
    if ((st = pending_error()) != HSA_OK) return st;
    hsa::DecodeStepCall c{q_idx, qi_sb, k_idx, k_sb, E_cap, B, DI, m, topk, H, window, idx_out, cnt_out, q, kc, vc,
                          k_raw, v_raw, c_sb, c_se, r_sb, r_st, N_cap, ctx_len, scale, out, lse};
    return launched(hsa::launch_decode_step(c, pl, ws, reinterpret_cast<cudaStream_t>(stream)), "decode_csa");
}

hsa_status_t hsa_attn_prefill_workspace_size(hsa_dtype_t dt, int B, int T, int H, int d, int64_t E_cap, int m,
                                             int topk, int window, size_t *bytes) {
    (void)dt; (void)B; (void)T; (void)H; (void)d; (void)E_cap; (void)m; (void)topk; (void)window;
    if (!bytes) return fail(HSA_ERR_INVALID_ARG, "null bytes");
    *bytes = 0;
    return ok();
}

hsa_status_t hsa_attn_prefill(const void *q, hsa_dtype_t dt, int B, int T, int H, int d, const void *kc,
                              const void *vc, int64_t c_sb, int64_t c_se, int64_t E_cap, int m, const int32_t *idx,
                              const int32_t *cnt, int topk, const void *k_raw, const void *v_raw, int64_t r_sb,
                              int64_t r_st, int64_t N_cap, int window, const int64_t *q_pos0, float scale, void *out,
                              float *lse, void *ws, size_t ws_bytes, hsa_stream_t stream) {
    (void)ws; (void)ws_bytes;
    hsa_status_t st = check_attn_common(q, dt, B, T, H, d, kc, vc, c_sb, c_se, E_cap, m, idx, topk, k_raw, v_raw,
                                        r_sb, r_st, N_cap, window, q_pos0, out);
    if (st != HSA_OK) return st;
    if (B == 0 || T == 0) return ok();
    DevInfo di;
    if ((st = device_info(di)) != HSA_OK) return st;
    if ((st = check_pointers({{cnt, "cnt"}, {lse, "lse"}})) != HSA_OK) return st;
    if ((st = pending_error()) != HSA_OK) return st;
    const bool dense = idx == nullptr;
    hsa::AttnArgs a{};
    a.q = q; a.rows = B * T; a.T = T; a.H = H; a.d = d;
    a.kc = kc; a.vc = vc; a.c_sb = c_sb; a.c_se = c_se; a.E_cap = E_cap; a.m = m;
    a.idx = idx; a.cnt = cnt; a.topk = dense ? 0 : topk;
    a.k_raw = k_raw; a.v_raw = v_raw; a.r_sb = r_sb; a.r_st = r_st; a.N_cap = N_cap; a.window = window;
    a.pos = q_pos0; a.pos_is_ctx = 0; a.scale = scale; a.out = out; a.lse = lse;
    a.shared_kv = kc == vc && k_raw == v_raw;
    a.split = 0; a.max_splits = 1;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (dt == HSA_BF16 && hsa::prefill_tc_supported(a))
        return launched(hsa::launch_attn_prefill_tc(a, di.num_sms, s), "attn_prefill (tcgen05)");
    if (dt == HSA_BF16 && hsa::gather_tc_supported(a))
        return launched(hsa::launch_attn_gather_tc(a, di.num_sms, s), "attn_prefill (tcgen05 gather)");
    cudaError_t e = dt == HSA_BF16 ? hsa::launch_attn_bf16(a, s) : hsa::launch_attn_f32(a, s);
    return launched(e, "attn_prefill");
}

}  // extern "C"

// ------------------------------------------------------------------------
// Allocation-free indexer: the scratch lives in this file-scope device array.
// Host code never uses its name as an address; the device address is looked
// up once per device with cudaGetSymbolAddress and passed to the kernels.
namespace {
static __device__ __align__(256) unsigned char g_noalloc_scratch[HSA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void *g_noalloc_addr[kMaxDevices] = {};

hsa_status_t noalloc_scratch(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(HSA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail(HSA_ERR_UNSUPPORTED, "device ordinal %d above %d", dev, kMaxDevices);
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);  // with `dev` current
        if (e != cudaSuccess || !p)
            return fail(HSA_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
        g_noalloc_addr[dev] = p;
    }
    *out = g_noalloc_addr[dev];
    return HSA_OK;
}
}  // namespace

extern "C" hsa_status_t hsa_index_topk_noalloc(const int8_t *q_idx, int64_t q_sb, int64_t q_st, const int8_t *k_idx,
                                               int64_t k_sb, int64_t k_se, int64_t E_cap, int B, int T, int DI,
                                               const int64_t *q_pos0, int m, int topk, int32_t *idx_out,
                                               int32_t *cnt_out, hsa_stream_t stream) {
    if (B < 0 || T < 0 || E_cap < 0 || m <= 0) return fail(HSA_ERR_INVALID_ARG, "bad size");
    if (topk <= 0 || topk > 4096) return fail(HSA_ERR_UNSUPPORTED, "topk must be in [1, 4096], got %d", topk);
    if (DI != 16 && DI != 32 && DI != 64 && DI != 128)
        return fail(HSA_ERR_UNSUPPORTED, "indexer dim must be 16, 32, 64 or 128, got %d", DI);
    if (B * (int64_t)T > kMaxRows) return fail(HSA_ERR_UNSUPPORTED, "B*T above 2^24");
    const int rows = B * T;
    if (rows == 0) return ok();
    if (!q_idx || !k_idx || !q_pos0 || !idx_out || !cnt_out) return fail(HSA_ERR_INVALID_ARG, "null pointer");
    if (E_cap > (int64_t)1 << 30) return fail(HSA_ERR_UNSUPPORTED, "E_cap above 2^30");
    if (!aligned16(q_idx) || !aligned16(k_idx) || q_sb % 16 || q_st % 16 || k_sb % 16 || k_se % 16)
        return fail(HSA_ERR_UNSUPPORTED, "indexer tensors and strides must be 16-byte aligned");
    if (k_se < DI || q_st < DI) return fail(HSA_ERR_INVALID_ARG, "indexer strides overlap rows");
    DevInfo di;
    hsa_status_t st = device_info(di);
    if (st != HSA_OK) return st;
    if ((st = check_pointers({{q_idx, "q_idx"}, {k_idx, "k_idx"}, {q_pos0, "q_pos0"}, {idx_out, "idx_out"},
                              {cnt_out, "cnt_out"}})) != HSA_OK)
        return st;
    hsa::IndexArgs a{q_idx, q_sb, q_st, k_idx, k_sb, k_se, E_cap, B, T, DI, q_pos0, m, topk, idx_out, cnt_out};
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (E_cap == 0) {
        if ((st = pending_error()) != HSA_OK) return st;
        cudaError_t e = cudaMemsetAsync(idx_out, 0xff, sizeof(int32_t) * (size_t)rows * topk, s);
        if (e == cudaSuccess) e = cudaMemsetAsync(cnt_out, 0, sizeof(int32_t) * (size_t)rows, s);
        return launched(e, "index (empty)");
    }
    const IndexChoice ch = choose_index(B, T, DI, E_cap, topk, di.num_sms);
    if (ch.bytes > (size_t)HSA_NOALLOC_SCRATCH_BYTES)
        return fail(HSA_ERR_WORKSPACE,
                    "hsa_index_topk_noalloc: these sizes need %zu bytes of scratch, the built-in scratch holds %u; "
                    "call hsa_index_topk with a workspace instead",
                    ch.bytes, (unsigned)HSA_NOALLOC_SCRATCH_BYTES);
    void *ws = nullptr;
    if ((st = noalloc_scratch(&ws)) != HSA_OK) return st;
    if ((st = pending_error()) != HSA_OK) return st;
    // the array keeps the previous call's contents: zero what this call's kernels expect zeroed
    cudaError_t e = cudaMemsetAsync(ws, 0, ch.fused ? ch.fp.zero_bytes : ch.bytes, s);
    if (e != cudaSuccess) return launched(e, "index_topk_noalloc (clear scratch)");
    if (ch.fused) return launched(hsa::launch_index_fused(a, ch.fp, ws, s), "index_topk_noalloc (fused)");
    if (ch.prefill) return launched(hsa::launch_index_prefill(a, ch.pp, ws, di.num_sms, s), "index_topk_noalloc (tensor cores)");
    for (int r0 = 0; r0 < rows; r0 += ch.group) {
        e = hsa::launch_index_topk(a, ch.tp, ws, r0, s);
        if (e != cudaSuccess) return launched(e, "index_topk_noalloc");
    }
    return ok();
}

extern "C" {

hsa_status_t hsa_index_scores(const int8_t *q_idx, int64_t q_sb, int64_t q_st, const int8_t *k_idx, int64_t k_sb,
                              int64_t k_se, int64_t E_cap, int B, int T, int DI, const int32_t *idx, const int32_t *cnt,
                              int topk, int32_t *scores, hsa_stream_t stream) {
    if (B < 0 || T < 0 || E_cap < 0 || topk <= 0 || topk > 4096) return fail(HSA_ERR_INVALID_ARG, "bad size");
    if (DI != 16 && DI != 32 && DI != 64 && DI != 128)
        return fail(HSA_ERR_UNSUPPORTED, "indexer dim must be 16, 32, 64 or 128, got %d", DI);
    if (B * (int64_t)T == 0) return ok();
    if (!q_idx || !k_idx || !idx || !scores) return fail(HSA_ERR_INVALID_ARG, "null pointer");
    if (!aligned16(q_idx) || !aligned16(k_idx) || q_sb % 16 || q_st % 16 || k_sb % 16 || k_se % 16)
        return fail(HSA_ERR_UNSUPPORTED, "indexer tensors and strides must be 16-byte aligned");
    if (k_se < DI || q_st < DI) return fail(HSA_ERR_INVALID_ARG, "indexer strides overlap rows");
    if (B * (int64_t)T > 65535) return fail(HSA_ERR_UNSUPPORTED, "more than 65535 query rows");
    DevInfo di;
    hsa_status_t st = device_info(di);
    if (st != HSA_OK) return st;
    if ((st = pending_error()) != HSA_OK) return st;
    if ((st = check_pointers({{q_idx, "q_idx"}, {k_idx, "k_idx"}, {idx, "idx"}, {cnt, "cnt"}, {scores, "scores"}})) !=
        HSA_OK)
        return st;
    hsa::IndexScoreArgs a{q_idx, q_sb, q_st, k_idx, k_sb, k_se, E_cap, B, T, DI, idx, cnt, topk, scores};
    return launched(hsa::launch_index_scores(a, reinterpret_cast<cudaStream_t>(stream)), "index_scores");
}

hsa_status_t hsa_topk_merge(const int32_t *scores, const int32_t *idx, int rows, int n, int topk, int32_t *idx_out,
                            int32_t *cnt_out, hsa_stream_t stream) {
    if (rows < 0 || n <= 0 || n > (1 << 20) || topk <= 0 || topk > 4096)
        return fail(HSA_ERR_INVALID_ARG, "bad size (rows=%d n=%d topk=%d)", rows, n, topk);
    if (rows == 0) return ok();
    if (!scores || !idx || !idx_out || !cnt_out) return fail(HSA_ERR_INVALID_ARG, "null pointer");
    DevInfo di;
    hsa_status_t st = device_info(di);
    if (st != HSA_OK) return st;
    if ((st = pending_error()) != HSA_OK) return st;
    if ((st = check_pointers({{scores, "scores"}, {idx, "idx"}, {idx_out, "idx_out"}, {cnt_out, "cnt_out"}})) != HSA_OK)
        return st;
    hsa::TopkMergeArgs a{scores, idx, rows, n, topk, idx_out, cnt_out};
    return launched(hsa::launch_topk_merge(a, reinterpret_cast<cudaStream_t>(stream)), "topk_merge");
}

hsa_status_t hsa_lse_merge(const void *parts_o, const float *parts_lse, hsa_dtype_t dt, int S, int rows, int H, int d,
                           void *out, float *lse_out, hsa_stream_t stream) {
    if (!dtype_ok(dt)) return fail(HSA_ERR_UNSUPPORTED, "dtype %d", (int)dt);
    if (S <= 0 || rows < 0 || H <= 0 || d <= 0 || d > 1024) return fail(HSA_ERR_INVALID_ARG, "bad size");
    if (d % (dt == HSA_BF16 ? 8 : 4)) return fail(HSA_ERR_UNSUPPORTED, "d must be a multiple of 8 (bf16) or 4 (fp32)");
    if (rows == 0) return ok();
    if (rows > 65535) return fail(HSA_ERR_UNSUPPORTED, "more than 65535 rows");
    if (!parts_o || !parts_lse || !out) return fail(HSA_ERR_INVALID_ARG, "null pointer");
    if (!aligned16(parts_o) || !aligned16(out)) return fail(HSA_ERR_UNSUPPORTED, "parts_o and out must be 16-byte aligned");
    DevInfo di;
    hsa_status_t st = device_info(di);
    if (st != HSA_OK) return st;
    if ((st = pending_error()) != HSA_OK) return st;
    if ((st = check_pointers({{parts_o, "parts_o"}, {parts_lse, "parts_lse"}, {out, "out"}, {lse_out, "lse_out"}})) !=
        HSA_OK)
        return st;
    hsa::LseMergeArgs a{parts_o, parts_lse, S, rows, H, d, out, lse_out};
    return launched(hsa::launch_lse_merge(a, dt == HSA_BF16, reinterpret_cast<cudaStream_t>(stream)), "lse_merge");
}

hsa_status_t hsa_rmsnorm_rope(void *x, hsa_dtype_t dt, int B, int H, int d, int64_t x_sb, int64_t x_sn,
                              int64_t n_cap, const int64_t *n_begin, const int64_t *n_end, int64_t max_rows,
                              const int64_t *pos_base, int64_t pos_stride, int64_t pos_offset, const float *gamma,
                              float eps, int rope_dims, float theta, hsa_stream_t stream) {
    if (!dtype_ok(dt)) return fail(HSA_ERR_UNSUPPORTED, "dtype %d", (int)dt);
    if (B < 0 || H <= 0 || d <= 0 || n_cap < 0 || max_rows < 0 || !(eps >= 0.f) || rope_dims < 0 || !(theta > 0.f))
        return fail(HSA_ERR_INVALID_ARG, "bad size or parameter");
    if (d % 64 || d > 512) return fail(HSA_ERR_UNSUPPORTED, "d must be a multiple of 64 up to 512, got %d", d);
    if (rope_dims % 2 || rope_dims > d) return fail(HSA_ERR_INVALID_ARG, "rope_dims must be even and <= d");
    if (rope_dims > hsa::kMaxRopeDims) return fail(HSA_ERR_UNSUPPORTED, "rope_dims above %d", hsa::kMaxRopeDims);
    if (B == 0 || max_rows == 0) return ok();
    if (B > 65535) return fail(HSA_ERR_UNSUPPORTED, "more than 65535 sequences");
    if (!x || !n_begin || !n_end) return fail(HSA_ERR_INVALID_ARG, "null pointer");
    if (x_sn < (int64_t)H * d || x_sb < 0) return fail(HSA_ERR_INVALID_ARG, "row strides overlap rows");
    DevInfo di;
    hsa_status_t st = device_info(di);
    if (st != HSA_OK) return st;
    if ((st = pending_error()) != HSA_OK) return st;
    if ((st = check_pointers({{x, "x"}, {n_begin, "n_begin"}, {n_end, "n_end"}, {pos_base, "pos_base"},
                              {gamma, "gamma"}})) != HSA_OK)
        return st;
    hsa::NormRopeArgs a{x, B, H, d, x_sb, x_sn, n_cap, n_begin, n_end, max_rows, pos_base, pos_stride, pos_offset,
                        gamma, eps, rope_dims, {}};
    for (int k = 0; k < rope_dims / 2; ++k) a.inv_freq[k] = pow((double)theta, -2.0 * k / rope_dims);
    return launched(hsa::launch_rmsnorm_rope(a, dt == HSA_BF16, reinterpret_cast<cudaStream_t>(stream)),
                    "rmsnorm_rope");
}

hsa_status_t hsa_attn_finalize(void *out, float *lse, hsa_dtype_t dt, int B, int T, int H, int d,
                               const int64_t *q_pos0, const float *sink, int rope_dims, float theta,
                               hsa_stream_t stream) {
    if (!dtype_ok(dt)) return fail(HSA_ERR_UNSUPPORTED, "dtype %d", (int)dt);
    if (B < 0 || T < 0 || H <= 0 || d <= 0 || rope_dims < 0 || !(theta > 0.f))
        return fail(HSA_ERR_INVALID_ARG, "bad size or parameter");
    if (d % 64 || d > 512) return fail(HSA_ERR_UNSUPPORTED, "d must be a multiple of 64 up to 512, got %d", d);
    if (rope_dims % 2 || rope_dims > d) return fail(HSA_ERR_INVALID_ARG, "rope_dims must be even and <= d");
    if (rope_dims > hsa::kMaxRopeDims) return fail(HSA_ERR_UNSUPPORTED, "rope_dims above %d", hsa::kMaxRopeDims);
    if (B * (int64_t)T == 0) return ok();
    if (B * (int64_t)T > 65535) return fail(HSA_ERR_UNSUPPORTED, "more than 65535 query rows");
    if (!out || !q_pos0 || (sink && !lse)) return fail(HSA_ERR_INVALID_ARG, "null pointer (a sink needs lse)");
    DevInfo di;
    hsa_status_t st = device_info(di);
    if (st != HSA_OK) return st;
    if ((st = pending_error()) != HSA_OK) return st;
    if ((st = check_pointers({{out, "out"}, {lse, "lse"}, {q_pos0, "q_pos0"}, {sink, "sink"}})) != HSA_OK) return st;
    hsa::FinalizeArgs a{out, lse, B, T, H, d, q_pos0, sink, rope_dims, {}};
    for (int k = 0; k < rope_dims / 2; ++k) a.inv_freq[k] = pow((double)theta, -2.0 * k / rope_dims);
    return launched(hsa::launch_attn_finalize(a, dt == HSA_BF16, reinterpret_cast<cudaStream_t>(stream)),
                    "attn_finalize");
}

}  // extern "C"
