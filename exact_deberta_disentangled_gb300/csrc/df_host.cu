// df_host.cu -- the C ABI of libdfattn (declared in include/df_attn.h):
// argument validation, workspace carve-up and the launch sequence of the
// forward and backward passes.  Nothing here allocates device memory.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "df_internal.h"

namespace df {
namespace {

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Bounded-wait limits and the test-only stall injection
// (df_attn_debug_inject_stall), copied into every call's ProblemDev.
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;   // 2 s
constexpr uint32_t kDefaultWaitProbes = 1u << 20;
unsigned long long g_wait_ns = kDefaultWaitNs;
uint32_t g_wait_probes = kDefaultWaitProbes;
int g_fault_kernel = -1, g_fault_tile = -1;

// The relative index of the kernels (delta_of in df_common.cuh), in double
// precision on the host, for sizing the stored-bias table.
int host_delta(int r, int span, int nb, int mp) {
    int bkt = r;
    if (nb > 0 && mp > 0) {
        const int mid = nb / 2, a = r < 0 ? -r : r;
        if (a > mid) {
            const double x = std::log((double)a / mid) / std::log((double)(mp - 1) / mid) * (double)(mid - 1);
            const int m = mid + (int)std::ceil(x);
            bkt = r < 0 ? -m : m;
        }
    }
    const int d = bkt + span;
    return d < 0 ? 0 : (d > 2 * span - 1 ? 2 * span - 1 : d);
}

// Key blocks kept on each side of a query block in the stored-bias table:
// the largest |qt - kt| of a 128 x 128 band block (relative positions
// [128 k - 127, 128 k + 127] for k = qt - kt not all clamped to R-1, or to 0
// for k < 0), plus one block of margin, so that a last-bit difference
// between the host's and the device's logarithm cannot move a band block
// out of the table.  The relative index is monotone in r, so the first
// clamped position on each side is found by bisection.
int bias_reach(const ProblemDev& p) {
    const int nrb = (p.L + 127) / 128, last = p.L - 1;
    auto first_clamped = [&](int sign, int target) {
        if (host_delta(sign * last, p.span, p.nb, p.mp) != target) return last + 1;
        int lo = 0, hi = last;   // delta(sign * hi) == target
        while (lo < hi) {
            const int mid = (lo + hi) / 2;
            if (host_delta(sign * mid, p.span, p.nb, p.mp) == target) hi = mid; else lo = mid + 1;
        }
        return lo;
    };
    const int rpos = first_clamped(1, p.R - 1), rneg = first_clamped(-1, 0);
    int kb = 0;
    for (int k = 1; k < nrb; ++k)
        if (128 * k - 127 < rpos || 128 * k - 127 < rneg) kb = k;
    return kb + 1 < nrb ? kb + 1 : nrb - 1;
}

// Validated problem: fills `out` and returns DF_OK, or an error code.
df_status resolve(const df_attn_params* a, ProblemDev& out) {
    if (!a) return DF_ERR_INVALID_ARG;
    if (a->B < 1 || a->L < 1 || a->H < 1 || a->D < 1 || a->att_span < 1) return DF_ERR_INVALID_ARG;
    if (a->dtype != DF_BF16 && a->dtype != DF_FP16 && a->dtype != DF_FP32 && a->dtype != DF_FP32_FAST)
        return DF_ERR_INVALID_ARG;
    if (!(a->dropout_p >= 0.f && a->dropout_p < 1.f)) return DF_ERR_INVALID_ARG;
    if (!(a->softmax_scale >= 0.f) || !std::isfinite(a->softmax_scale)) return DF_ERR_INVALID_ARG;
    if (a->philox_offset >> 32) return DF_ERR_INVALID_ARG;
    if (a->D != 32 && a->D != 64 && a->D != 128) return DF_ERR_UNSUPPORTED;
    if (a->L > 8192) return DF_ERR_UNSUPPORTED;
    if (a->att_span > 512) return DF_ERR_UNSUPPORTED;
    const bool bucketing = a->position_buckets > 0 && a->max_relative_positions > 0;
    if (bucketing && (a->position_buckets < 2 || a->max_relative_positions - 1 <= a->position_buckets / 2))
        return DF_ERR_UNSUPPORTED;
    if (bucketing && a->dtype != DF_FP32) {
        // the tensor-core kernels size their band windows for a relative index
        // that moves by at most one per relative position: the log segment's
        // first step, from |r| = buckets / 2, is its largest
        const double mid = (double)(a->position_buckets / 2);
        if ((mid - 1.0) * std::log1p(1.0 / mid) > std::log((a->max_relative_positions - 1) / mid))
            return DF_ERR_UNSUPPORTED;
    }
    long long T;
    if (a->cu_seqlens) {
        if (a->query_mask || a->key_mask) return DF_ERR_UNSUPPORTED;  // masks are a padded-layout feature
        if (a->total_tokens < 1) return DF_ERR_INVALID_ARG;
        if ((long long)a->total_tokens > (long long)a->B * a->L) return DF_ERR_INVALID_ARG;
        T = a->total_tokens;
    } else {
        T = (long long)a->B * a->L;
    }
    if (T * a->H >= (1ll << 31) || (long long)a->B * a->L * a->H >= (1ll << 31)) return DF_ERR_UNSUPPORTED;
    std::memset(&out, 0, sizeof(out));
    out.B = a->B;
    out.L = a->L;
    out.H = a->H;
    out.D = a->D;
    out.span = a->att_span;
    out.R = 2 * a->att_span;
    out.nb = bucketing ? a->position_buckets : 0;
    out.mp = bucketing ? a->max_relative_positions : 0;
    out.T = (int)T;
    out.cu = a->cu_seqlens;
    out.qmask = a->query_mask;
    out.kmask = a->key_mask;
    out.scale = a->softmax_scale > 0.f ? a->softmax_scale : (float)(1.0 / std::sqrt(3.0 * a->D));
    const double p = (double)a->dropout_p;
    out.dropout = p > 0.0;
    out.keep_all = p > 0.0 ? 0 : 1;
    out.drop_scale = p > 0.0 ? (float)(1.0 / (1.0 - p)) : 1.f;
    if (p > 0.0) {
        const double t = std::floor((1.0 - p) * 4294967296.0);
        out.keep_thr = t >= 4294967295.0 ? 0xFFFFFFFFu : (uint32_t)t;
        if (t >= 4294967296.0) out.keep_all = 1;
    } else {
        out.keep_thr = 0xFFFFFFFFu;
    }
    out.seed_lo = (uint32_t)a->philox_seed;
    out.seed_hi = (uint32_t)(a->philox_seed >> 32);
    out.philox_offset = (uint32_t)a->philox_offset;
    out.wait_ns = g_wait_ns;
    out.wait_probes = g_wait_probes;
    out.fault_kernel = g_fault_kernel;
    out.fault_tile = g_fault_tile;
    out.bias_kb = bias_reach(out);
    out.bias_nslot = 2 * out.bias_kb + 1;
    out.saved_bias = nullptr;
    if (a->band_bias && a->dtype != DF_FP32) {
        if ((uintptr_t)a->band_bias & 15u) return DF_ERR_INVALID_ARG;
        out.saved_bias = (uint16_t*)a->band_bias;
    }
    return DF_OK;
}

int elem_bytes(df_dtype d) { return d == DF_FP32 || d == DF_FP32_FAST ? 4 : 2; }

int rel_chunks(const ProblemDev& p) {
    // Token chunks of the relative-gradient reduction: enough CTAs to fill
    // the GPU twice, each chunk at least 512 tokens.
    const int rb = (p.R + 127) / 128;
    int c = (2 * 152 + p.H * rb - 1) / (p.H * rb);
    const int maxc = (p.T + 511) / 512;
    if (c > maxc) c = maxc;
    return c < 1 ? 1 : c;
}

// Rows of the stored band bias ([rows][128] fp16): 128 x 128 blocks,
// bias_nslot per query block of each (sequence, head) pair (row index in
// df_tile.cuh, bias_block_row).
size_t bias_table_rows(const ProblemDev& p) {
    const size_t nrbg = (size_t)(p.T - 1) / 128 + (size_t)p.B + 1;
    return nrbg * (size_t)p.H * (size_t)p.bias_nslot * 128;
}

// The fast fp32 mode's fp16 copies of the inputs and outputs, placed after
// the fp16 workspace; with base == nullptr only the size is computed.
struct FastBufs {
    char *q, *k, *v, *qr, *kr, *out, *dout, *dq, *dk, *dv, *dqr, *dkr;
    size_t bytes;
};
FastBufs fast_bufs(const ProblemDev& p, bool backward, char* base) {
    FastBufs f;
    std::memset(&f, 0, sizeof(f));
    size_t off = 0;
    auto take = [&](size_t bytes) -> char* {
        char* r = base ? base + off : nullptr;
        off += align_up(bytes);
        return r;
    };
    const size_t tok = sizeof(uint16_t) * (size_t)p.T * p.H * p.D, rel = sizeof(uint16_t) * (size_t)p.H * p.R * p.D;
    f.q = take(tok);
    f.k = take(tok);
    f.v = take(tok);
    f.qr = take(rel);
    f.kr = take(rel);
    f.out = take(tok);
    if (backward) {
        f.dout = take(tok);
        f.dq = take(tok);
        f.dk = take(tok);
        f.dv = take(tok);
        f.dqr = take(rel);
        f.dkr = take(rel);
    }
    f.bytes = off;
    return f;
}

// Carve the workspace; with base == nullptr only the size is computed.  The
// fast fp32 mode is the fp16 workspace (error word first, as always) and then
// the fp16 copies.
Workspace carve(const ProblemDev& p, df_dtype dt, bool backward, void* base) {
    if (dt == DF_FP32_FAST) {
        Workspace w = carve(p, DF_FP16, backward, base);
        w.bytes += fast_bufs(p, backward, nullptr).bytes;
        return w;
    }
    Workspace w;
    std::memset(&w, 0, sizeof(w));
    size_t off = 0;
    auto take = [&](size_t bytes) -> char* {
        char* r = base ? (char*)base + off : nullptr;
        off += align_up(bytes);
        return r;
    };
    w.err = (int*)take(kAlign);
    w.dtab = (int32_t*)take(sizeof(int32_t) * (size_t)(2 * p.L - 1));
    if (dt != DF_FP32) w.relb = (float*)take(sizeof(float) * 4 * (size_t)p.T * p.H);
    w.Rp = dt == DF_FP32 ? p.R : (p.R + 63) / 64 * 64;
    if (backward) {
        w.rowterm = (float*)take(sizeof(float) * (size_t)p.H * (size_t)p.B * p.L);
        const size_t g = (size_t)elem_bytes(dt) * (size_t)p.T * p.H * w.Rp;
        w.G = take(g);
        w.Gp = take(g);
        if (dt != DF_FP32) {
            w.nchunk = rel_chunks(p);
            const size_t part = sizeof(float) * (size_t)w.nchunk * p.H * p.R * p.D;
            w.part_kr = (float*)take(part);
            w.part_qr = (float*)take(part);
            const size_t a = sizeof(float) * (size_t)p.T * p.H * p.D;
            w.acc32a = (float*)take(a);
            w.acc32b = (float*)take(a);
            // stored band bias: the caller's saved buffer, else part of the workspace
            w.bias_rows = bias_table_rows(p);
            w.bias = p.saved_bias ? p.saved_bias : (uint16_t*)take(sizeof(uint16_t) * w.bias_rows * 128);
        }
    }
    w.bytes = off;
    return w;
}

df_status cuda_status(int e) { return e == 0 ? DF_OK : DF_ERR_CUDA; }

cudaEvent_t g_prof[2 * kProfPhases];
int g_prof_on = 0;

}  // namespace

void prof_record(int phase, int end, cudaStream_t st) {
    if (g_prof_on && phase >= 0 && phase < kProfPhases) cudaEventRecord(g_prof[2 * phase + (end ? 1 : 0)], st);
}

// ------------------------------------------------------------- TMA encode

int encode_tmap(void* tmap, int dtype_code, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
                const uint32_t* box, int swizzle_bytes, const void* base) {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)ptr;
    });
    if (!fn) return 1;
    CUtensorMapDataType t = dtype_code == 0   ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                            : dtype_code == 1 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                              : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_NONE;
    if (swizzle_bytes == 128) sw = CU_TENSOR_MAP_SWIZZLE_128B;
    if (swizzle_bytes == 64) sw = CU_TENSOR_MAP_SWIZZLE_64B;
    if (swizzle_bytes == 32) sw = CU_TENSOR_MAP_SWIZZLE_32B;
    cuuint64_t d[5], s[4];
    cuuint32_t bx[5], es[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        bx[i] = box[i];
        es[i] = 1;
        if (i > 0) s[i - 1] = strides_bytes[i - 1];
    }
    CUresult r = fn((CUtensorMap*)tmap, t, (cuuint32_t)rank, const_cast<void*>(base), d, s, bx, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? 0 : 2;
}

}  // namespace df

using namespace df;

extern "C" {

const char* df_status_string(df_status s) {
    switch (s) {
        case DF_OK: return "DF_OK";
        case DF_ERR_INVALID_ARG: return "DF_ERR_INVALID_ARG: bad pointer, size, alignment or value";
        case DF_ERR_UNSUPPORTED: return "DF_ERR_UNSUPPORTED: configuration outside the supported contract";
        case DF_ERR_WORKSPACE: return "DF_ERR_WORKSPACE: workspace missing or too small";
        case DF_ERR_CUDA: return "DF_ERR_CUDA: CUDA runtime or launch error";
        case DF_ERR_TIMEOUT: return "DF_ERR_TIMEOUT: a bounded device wait gave up";
        case DF_ERR_DEVICE_ARG: return "DF_ERR_DEVICE_ARG: cu_seqlens inconsistent with B, L, total_tokens";
        case DF_ERR_DEVICE_CHECK: return "DF_ERR_DEVICE_CHECK: a checked build found an index outside its buffer";
    }
    return "unknown df_status";
}

const char* df_version(void) { return "0.1.0"; }

df_status df_attn_set_profile_events(void* const* events, int n) {
    if (!events || n == 0) {
        g_prof_on = 0;
        return DF_OK;
    }
    if (n != 2 * kProfPhases) return DF_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i) {
        if (!events[i]) return DF_ERR_INVALID_ARG;
        g_prof[i] = (cudaEvent_t)events[i];
    }
    g_prof_on = 1;
    return DF_OK;
}

df_status df_attn_debug_inject_stall(int kernel, int tile, uint64_t wait_limit_ns, uint32_t wait_min_probes) {
    if (kernel < 0) {
        g_fault_kernel = g_fault_tile = -1;
        g_wait_ns = kDefaultWaitNs;
        g_wait_probes = kDefaultWaitProbes;
        return DF_OK;
    }
    if (kernel > 2 || tile < 0 || wait_limit_ns == 0 || wait_limit_ns > kDefaultWaitNs) return DF_ERR_INVALID_ARG;
    g_fault_kernel = kernel;
    g_fault_tile = tile;
    g_wait_ns = wait_limit_ns;
    g_wait_probes = wait_min_probes;
    return DF_OK;
}

size_t df_attn_band_bias_size(const df_attn_params* a) {
    ProblemDev p;
    if (resolve(a, p) != DF_OK || a->dtype == DF_FP32) return 0;
    return sizeof(uint16_t) * bias_table_rows(p) * 128;
}

size_t df_attn_workspace_size(const df_attn_params* a, int backward) {
    ProblemDev p;
    if (resolve(a, p) != DF_OK) return 0;
    return carve(p, a->dtype, backward != 0, nullptr).bytes;
}

static df_status common_prologue(const df_attn_params* a, ProblemDev& p, Workspace& w, bool backward,
                                 void* workspace, size_t ws_bytes, cudaStream_t st) {
    df_status s = resolve(a, p);
    if (s != DF_OK) return s;
    if (!workspace || !aligned16(workspace)) return DF_ERR_WORKSPACE;
    const size_t need = carve(p, a->dtype, backward, nullptr).bytes;
    if (ws_bytes < need) return DF_ERR_WORKSPACE;
    w = carve(p, a->dtype, backward, workspace);
    p.err = w.err;
    if (launch_clear_error(w.err, st)) return DF_ERR_CUDA;
    if (launch_delta_table(p.L, p.span, p.nb, p.mp, w.dtab, st)) return DF_ERR_CUDA;
    if (p.cu && launch_check_cu(p, st)) return DF_ERR_CUDA;
    return DF_OK;
}

static df_status fast_fwd(const df_attn_params* a, const void* q, const void* k, const void* v, const void* qr,
                          const void* kr, void* out, float* lse, void* workspace, size_t ws_bytes,
                          df_stream_t stream);
static df_status fast_bwd(const df_attn_params* a, const void* q, const void* k, const void* v, const void* qr,
                          const void* kr, const void* out, const float* lse, const void* dout, void* dq, void* dk,
                          void* dv, void* dqr, void* dkr, void* workspace, size_t ws_bytes, df_stream_t stream);

// A forward in two parts (the host-buffer step): sequences [0, b_split),
// then, once `second_ready` has been recorded, sequences [b_split, B), whose
// tokens start at tok_split.
struct FwdParts {
    int b_split, tok_split;
    cudaEvent_t second_ready;
};

// The forward with or without the LSE store (lse == nullptr: inference).
static df_status fwd_common(const df_attn_params* a, const void* q, const void* k, const void* v, const void* qr,
                            const void* kr, void* out, float* lse, void* workspace, size_t ws_bytes,
                            df_stream_t stream, const FwdParts* parts = nullptr) {
    const void* ptrs[] = {q, k, v, qr, kr, out};
    for (const void* x : ptrs)
        if (!x || !aligned16(x)) return DF_ERR_INVALID_ARG;
    if (lse && !aligned16(lse)) return DF_ERR_INVALID_ARG;
    if (a && a->cu_seqlens && ((uintptr_t)a->cu_seqlens & 3u)) return DF_ERR_INVALID_ARG;
    if (a && a->dtype == DF_FP32_FAST) return fast_fwd(a, q, k, v, qr, kr, out, lse, workspace, ws_bytes, stream);
    ProblemDev p;
    Workspace w;
    cudaStream_t st = (cudaStream_t)stream;
    df_status s = common_prologue(a, p, w, false, workspace, ws_bytes, st);
    if (s != DF_OK) return s;
    if (a->dtype == DF_FP32)
        return cuda_status(launch_fwd_f32(p, w, (const float*)q, (const float*)k, (const float*)v, (const float*)qr,
                                          (const float*)kr, (float*)out, lse, st));
    if (parts && parts->b_split > 0 && parts->b_split < p.B) {
        ProblemDev p1 = p, p2 = p;
        p1.b_count = parts->b_split;
        p2.b_base = parts->b_split;
        p2.b_count = p.B - parts->b_split;
        if (launch_relbias(p, a->dtype, q, k, qr, kr, w.relb, st, 0, parts->tok_split) ||
            launch_fwd_tc(p1, w, a->dtype, q, k, v, qr, kr, out, lse, st) ||
            cudaStreamWaitEvent(st, parts->second_ready, 0) != cudaSuccess ||
            launch_relbias(p, a->dtype, q, k, qr, kr, w.relb, st, parts->tok_split, -1))
            return DF_ERR_CUDA;
        return cuda_status(launch_fwd_tc(p2, w, a->dtype, q, k, v, qr, kr, out, lse, st));
    }
    if (launch_relbias(p, a->dtype, q, k, qr, kr, w.relb, st)) return DF_ERR_CUDA;
    return cuda_status(launch_fwd_tc(p, w, a->dtype, q, k, v, qr, kr, out, lse, st));
}

df_status df_attn_fwd(const df_attn_params* a, const void* q, const void* k, const void* v, const void* qr,
                      const void* kr, void* out, float* lse, void* workspace, size_t ws_bytes, df_stream_t stream) {
    if (!lse) return DF_ERR_INVALID_ARG;
    return fwd_common(a, q, k, v, qr, kr, out, lse, workspace, ws_bytes, stream);
}

df_status df_attn_fwd_inference(const df_attn_params* a, const void* q, const void* k, const void* v,
                                const void* qr, const void* kr, void* out, void* workspace, size_t ws_bytes,
                                df_stream_t stream) {
    return fwd_common(a, q, k, v, qr, kr, out, nullptr, workspace, ws_bytes, stream);
}

// The backward, with the optional hook of the tensor-core path (the
// host-buffer step copies finished gradients down while later kernels run).
static df_status bwd_common(const df_attn_params* a, const void* q, const void* k, const void* v, const void* qr,
                            const void* kr, const void* out, const float* lse, const void* dout, void* dq, void* dk,
                            void* dv, void* dqr, void* dkr, void* workspace, size_t ws_bytes, df_stream_t stream,
                            const BwdHook* hook) {
    const void* ptrs[] = {q, k, v, qr, kr, out, lse, dout, dq, dk, dv, dqr, dkr};
    for (const void* x : ptrs)
        if (!x || !aligned16(x)) return DF_ERR_INVALID_ARG;
    if (a && a->cu_seqlens && ((uintptr_t)a->cu_seqlens & 3u)) return DF_ERR_INVALID_ARG;
    if (a && a->dtype == DF_FP32_FAST)
        return fast_bwd(a, q, k, v, qr, kr, out, lse, dout, dq, dk, dv, dqr, dkr, workspace, ws_bytes, stream);
    ProblemDev p;
    Workspace w;
    cudaStream_t st = (cudaStream_t)stream;
    df_status s = common_prologue(a, p, w, true, workspace, ws_bytes, st);
    if (s != DF_OK) return s;
    if (a->dtype == DF_FP32) {
        if (launch_rowterm(p, a->dtype, out, dout, w.rowterm, st)) return DF_ERR_CUDA;
        return cuda_status(launch_bwd_f32(p, w, (const float*)q, (const float*)k, (const float*)v,
                                          (const float*)qr, (const float*)kr, lse, (const float*)dout, (float*)dq,
                                          (float*)dk, (float*)dv, (float*)dqr, (float*)dkr, st));
    }
    return cuda_status(
        launch_bwd_tc(p, w, a->dtype, q, k, v, qr, kr, out, lse, dout, dq, dk, dv, dqr, dkr, st, hook));
}

// ------------------------------------------------------- fast fp32 mode
// ("DisentangledFlash", section "Status": the optional fast FP32/TF32 mode)
// fp32 in and out; the inputs are rounded to fp16 (TF32's 10-bit
// significand) into the workspace, the fp16 tensor-core path runs on them,
// and its fp16 results are widened to fp32.

namespace {
struct FastSetup {
    df_status s;
    size_t inner;   // bytes of the fp16 workspace at the start
    FastBufs f;
    long long tok, rel;   // elements of a token tensor / a relative tensor
};
FastSetup fast_setup(const df_attn_params* a, bool backward, void* workspace, size_t ws_bytes) {
    FastSetup r;
    std::memset(&r, 0, sizeof(r));
    ProblemDev p;
    r.s = resolve(a, p);
    if (r.s != DF_OK) return r;
    if (!workspace || !aligned16(workspace)) {
        r.s = DF_ERR_WORKSPACE;
        return r;
    }
    r.inner = carve(p, DF_FP16, backward, nullptr).bytes;
    r.f = fast_bufs(p, backward, (char*)workspace + r.inner);
    if (ws_bytes < r.inner + r.f.bytes) r.s = DF_ERR_WORKSPACE;
    r.tok = (long long)p.T * p.H * p.D;
    r.rel = (long long)p.H * p.R * p.D;
    return r;
}
void conv_add(ConvList& cl, const void* src, void* dst, long long n) {
    cl.src[cl.nseg] = src;
    cl.dst[cl.nseg] = dst;
    cl.n[cl.nseg] = n;
    ++cl.nseg;
}
}  // namespace

static df_status fast_fwd(const df_attn_params* a, const void* q, const void* k, const void* v, const void* qr,
                          const void* kr, void* out, float* lse, void* workspace, size_t ws_bytes,
                          df_stream_t stream) {
    const FastSetup fs = fast_setup(a, false, workspace, ws_bytes);
    if (fs.s != DF_OK) return fs.s;
    const FastBufs& f = fs.f;
    cudaStream_t st = (cudaStream_t)stream;
    ConvList in{};
    conv_add(in, q, f.q, fs.tok);
    conv_add(in, k, f.k, fs.tok);
    conv_add(in, v, f.v, fs.tok);
    conv_add(in, qr, f.qr, fs.rel);
    conv_add(in, kr, f.kr, fs.rel);
    if (launch_convert(in, true, st)) return DF_ERR_CUDA;
    df_attn_params a16 = *a;
    a16.dtype = DF_FP16;
    const df_status s = fwd_common(&a16, f.q, f.k, f.v, f.qr, f.kr, f.out, lse, workspace, fs.inner, stream);
    if (s != DF_OK) return s;
    ConvList o{};
    conv_add(o, f.out, out, fs.tok);
    return cuda_status(launch_convert(o, false, st));
}

static df_status fast_bwd(const df_attn_params* a, const void* q, const void* k, const void* v, const void* qr,
                          const void* kr, const void* out, const float* lse, const void* dout, void* dq, void* dk,
                          void* dv, void* dqr, void* dkr, void* workspace, size_t ws_bytes, df_stream_t stream) {
    const FastSetup fs = fast_setup(a, true, workspace, ws_bytes);
    if (fs.s != DF_OK) return fs.s;
    const FastBufs& f = fs.f;
    cudaStream_t st = (cudaStream_t)stream;
    ConvList in{};
    conv_add(in, q, f.q, fs.tok);
    conv_add(in, k, f.k, fs.tok);
    conv_add(in, v, f.v, fs.tok);
    conv_add(in, qr, f.qr, fs.rel);
    conv_add(in, kr, f.kr, fs.rel);
    conv_add(in, out, f.out, fs.tok);
    conv_add(in, dout, f.dout, fs.tok);
    if (launch_convert(in, true, st)) return DF_ERR_CUDA;
    df_attn_params a16 = *a;
    a16.dtype = DF_FP16;
    const df_status s = bwd_common(&a16, f.q, f.k, f.v, f.qr, f.kr, f.out, lse, f.dout, f.dq, f.dk, f.dv, f.dqr,
                                   f.dkr, workspace, fs.inner, stream, nullptr);
    if (s != DF_OK) return s;
    ConvList o{};
    conv_add(o, f.dq, dq, fs.tok);
    conv_add(o, f.dk, dk, fs.tok);
    conv_add(o, f.dv, dv, fs.tok);
    conv_add(o, f.dqr, dqr, fs.rel);
    conv_add(o, f.dkr, dkr, fs.rel);
    return cuda_status(launch_convert(o, false, st));
}

df_status df_attn_bwd(const df_attn_params* a, const void* q, const void* k, const void* v, const void* qr,
                      const void* kr, const void* out, const float* lse, const void* dout, void* dq, void* dk,
                      void* dv, void* dqr, void* dkr, void* workspace, size_t ws_bytes, df_stream_t stream) {
    return bwd_common(a, q, k, v, qr, kr, out, lse, dout, dq, dk, dv, dqr, dkr, workspace, ws_bytes, stream, nullptr);
}

// ------------------------------------------------------- host-buffer step

namespace {
struct Arena {
    size_t q, k, v, qr, kr, dout, out, lse, dq, dk, dv, dqr, dkr, cu, qm, km, bias, ws, bytes;
};
Arena arena_layout(const df_attn_params* a, const ProblemDev& p) {
    Arena r;
    size_t off = 0;
    auto take = [&](size_t b) {
        size_t o = off;
        off += align_up(b);
        return o;
    };
    const size_t e = (size_t)elem_bytes(a->dtype);
    const size_t tok = e * (size_t)p.T * p.H * p.D;
    const size_t rel = e * (size_t)p.H * p.R * p.D;
    const size_t lse = sizeof(float) * (size_t)p.H * (p.cu ? (size_t)p.T : (size_t)p.B * p.L);
    r.q = take(tok);
    r.k = take(tok);
    r.v = take(tok);
    r.qr = take(rel);
    r.kr = take(rel);
    r.dout = take(tok);
    r.out = take(tok);
    r.lse = take(lse);
    r.dq = take(tok);
    r.dk = take(tok);
    r.dv = take(tok);
    r.dqr = take(rel);
    r.dkr = take(rel);
    r.cu = take(sizeof(int32_t) * (size_t)(p.B + 1));
    r.qm = take((size_t)p.B * p.L);
    r.km = take((size_t)p.B * p.L);
    // the band bias, saved by the forward for the backward (bf16 / fp16): the
    // workspace then leaves it out
    const size_t bb = a->dtype == DF_FP32 ? 0 : sizeof(uint16_t) * bias_table_rows(p) * 128;
    r.bias = take(bb);
    ProblemDev ps = p;
    if (bb) ps.saved_bias = reinterpret_cast<uint16_t*>(kAlign);   // any non-null value: sizes only
    const size_t wf = carve(ps, a->dtype, false, nullptr).bytes, wb = carve(ps, a->dtype, true, nullptr).bytes;
    r.ws = take(wf > wb ? wf : wb);
    r.bytes = off;
    return r;
}
}  // namespace

namespace {
// A copy stream and its events per device for df_attn_step_host, created on
// first use with that device current: the second half of the sequences' Q /
// K / V and then dO go up while the forward runs, and the results come down
// while the backward runs.  The events are shared by
// every call on the device, so one call's enqueue sequence holds g_copy_mu.
constexpr int kMaxCopyDevices = 64;
std::mutex g_copy_mu;
bool g_copy_tried[kMaxCopyDevices];
cudaStream_t g_copy_st[kMaxCopyDevices];
cudaEvent_t g_copy_ev[kMaxCopyDevices][8];   // start, dout up, forward done, copies down done, dV / dQ / dK final,
                                              // second forward part's inputs up

bool copy_stream(int dev, cudaStream_t& cs, cudaEvent_t*& ev) {
    if (dev < 0 || dev >= kMaxCopyDevices) return false;
    if (!g_copy_tried[dev]) {
        g_copy_tried[dev] = true;
        bool ok = cudaStreamCreateWithFlags(&g_copy_st[dev], cudaStreamNonBlocking) == cudaSuccess;
        for (int i = 0; i < 8 && ok; ++i)
            ok = cudaEventCreateWithFlags(&g_copy_ev[dev][i], cudaEventDisableTiming) == cudaSuccess;
        if (!ok) {
            cudaGetLastError();
            g_copy_st[dev] = nullptr;
        }
    }
    if (!g_copy_st[dev]) return false;
    cs = g_copy_st[dev];
    ev = g_copy_ev[dev];
    return true;
}
}  // namespace

size_t df_attn_step_host_arena_size(const df_attn_params* a) {
    ProblemDev p;
    if (resolve(a, p) != DF_OK) return 0;
    return arena_layout(a, p).bytes;
}

df_status df_attn_step_host(const df_attn_params* a, const void* q, const void* k, const void* v, const void* qr,
                            const void* kr, const void* dout, void* out, float* lse, void* dq, void* dk, void* dv,
                            void* dqr, void* dkr, void* arena, size_t arena_bytes, df_stream_t stream) {
    const void* ptrs[] = {q, k, v, qr, kr, dout, out, lse, dq, dk, dv, dqr, dkr};
    for (const void* x : ptrs)
        if (!x) return DF_ERR_INVALID_ARG;
    ProblemDev p;
    df_status s = resolve(a, p);
    if (s != DF_OK) return s;
    if (!arena || !aligned16(arena)) return DF_ERR_WORKSPACE;
    const Arena L = arena_layout(a, p);
    if (arena_bytes < L.bytes) return DF_ERR_WORKSPACE;
    char* base = (char*)arena;
    cudaStream_t st = (cudaStream_t)stream;
    const size_t e = (size_t)elem_bytes(a->dtype);
    const size_t tok = e * (size_t)p.T * p.H * p.D;
    const size_t rel = e * (size_t)p.H * p.R * p.D;
    const size_t lseb = sizeof(float) * (size_t)p.H * (p.cu ? (size_t)p.T : (size_t)p.B * p.L);
    auto h2d = [&](size_t off, const void* src, size_t n) {
        return cudaMemcpyAsync(base + off, src, n, cudaMemcpyHostToDevice, st) == cudaSuccess;
    };
    auto d2h = [&](void* dst, size_t off, size_t n, cudaStream_t s2) {
        return cudaMemcpyAsync(dst, base + off, n, cudaMemcpyDeviceToHost, s2) == cudaSuccess;
    };
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return DF_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_copy_mu);
    cudaStream_t cs = nullptr;
    cudaEvent_t* ev = nullptr;
    const bool side = copy_stream(dev, cs, ev);
    df_attn_params dp = *a;
    if (a->dtype != DF_FP32) dp.band_bias = base + L.bias;
    // With two or more sequences the tensor-core forward runs in two parts:
    // the first half of the sequences' Q / K / V go up on the caller's
    // stream, the rest on the copy stream while the first part runs
    FwdParts parts{0, 0, side ? ev[7] : nullptr};
    if (side && (a->dtype == DF_BF16 || a->dtype == DF_FP16) && p.B >= 2) {
        parts.b_split = p.B / 2;
        parts.tok_split = a->cu_seqlens ? a->cu_seqlens[parts.b_split] : parts.b_split * p.L;
    }
    const size_t tok1 = e * (size_t)parts.tok_split * p.H * p.D;   // bytes of the first part's rows
    bool ok = h2d(L.qr, qr, rel) && h2d(L.kr, kr, rel) && h2d(L.q, q, tok1 ? tok1 : tok) &&
              h2d(L.k, k, tok1 ? tok1 : tok) && h2d(L.v, v, tok1 ? tok1 : tok);
    // dO is needed by the backward only: on the copy stream, during the forward
    if (side) {
        ok = ok && cudaEventRecord(ev[0], st) == cudaSuccess && cudaStreamWaitEvent(cs, ev[0], 0) == cudaSuccess;
        if (tok1) {
            auto up2 = [&](size_t off, const void* src) {
                return cudaMemcpyAsync(base + off + tok1, (const char*)src + tok1, tok - tok1, cudaMemcpyHostToDevice,
                                       cs) == cudaSuccess;
            };
            ok = ok && up2(L.q, q) && up2(L.k, k) && up2(L.v, v) && cudaEventRecord(ev[7], cs) == cudaSuccess;
        }
        ok = ok && cudaMemcpyAsync(base + L.dout, dout, tok, cudaMemcpyHostToDevice, cs) == cudaSuccess &&
             cudaEventRecord(ev[1], cs) == cudaSuccess;
    } else {
        ok = ok && h2d(L.dout, dout, tok);
    }
    if (ok && a->cu_seqlens) {
        ok = h2d(L.cu, a->cu_seqlens, sizeof(int32_t) * (size_t)(p.B + 1));
        dp.cu_seqlens = (const int32_t*)(base + L.cu);
    }
    if (ok && a->query_mask) {
        ok = h2d(L.qm, a->query_mask, (size_t)p.B * p.L);
        dp.query_mask = (const uint8_t*)(base + L.qm);
    }
    if (ok && a->key_mask) {
        ok = h2d(L.km, a->key_mask, (size_t)p.B * p.L);
        dp.key_mask = (const uint8_t*)(base + L.km);
    }
    if (!ok) return DF_ERR_CUDA;
    const size_t wsb = arena_bytes - L.ws;
    s = fwd_common(&dp, base + L.q, base + L.k, base + L.v, base + L.qr, base + L.kr, base + L.out,
                   (float*)(base + L.lse), base + L.ws, wsb, stream, tok1 ? &parts : nullptr);
    if (s != DF_OK) return s;
    // O and the LSE are final after the forward: down on the copy stream during the backward
    if (side) {
        ok = cudaEventRecord(ev[2], st) == cudaSuccess && cudaStreamWaitEvent(cs, ev[2], 0) == cudaSuccess &&
             d2h(out, L.out, tok, cs) && d2h(lse, L.lse, lseb, cs) && cudaStreamWaitEvent(st, ev[1], 0) == cudaSuccess;
        if (!ok) return DF_ERR_CUDA;
    }
    // dQ (after the dQ kernel and its relative-gradient half), dV and dK are
    // final before the backward's last kernels: the backward's hook sends each
    // down on the copy stream while the rest runs
    struct Down {
        cudaStream_t cs;
        cudaEvent_t* ev;
        const char* base;
        size_t off_dv, off_dq, off_dk, tok;
        void *dv, *dq, *dk;
        bool sent[3], ok;
    } down{cs, ev, base, L.dv, L.dq, L.dk, tok, dv, dq, dk, {false, false, false}, true};
    const BwdHook hook{[](void* ctx, int point, cudaStream_t s2) {
                           Down& d = *static_cast<Down*>(ctx);
                           cudaEvent_t e = d.ev[4 + point];
                           d.ok = d.ok && cudaEventRecord(e, s2) == cudaSuccess &&
                                  cudaStreamWaitEvent(d.cs, e, 0) == cudaSuccess;
                           auto down1 = [&](void* dst, size_t off) {
                               d.ok = d.ok && cudaMemcpyAsync(dst, d.base + off, d.tok, cudaMemcpyDeviceToHost,
                                                              d.cs) == cudaSuccess;
                           };
                           if (point == 0) down1(d.dv, d.off_dv);
                           else if (point == 1) down1(d.dq, d.off_dq);
                           else down1(d.dk, d.off_dk);
                           d.sent[point] = true;
                       },
                       &down};
    s = bwd_common(&dp, base + L.q, base + L.k, base + L.v, base + L.qr, base + L.kr, base + L.out,
                   (const float*)(base + L.lse), base + L.dout, base + L.dq, base + L.dk, base + L.dv, base + L.dqr,
                   base + L.dkr, base + L.ws, wsb, stream, side ? &hook : nullptr);
    if (s != DF_OK) return s;
    if (!down.ok) return DF_ERR_CUDA;
    ok = d2h(dqr, L.dqr, rel, st) && d2h(dkr, L.dkr, rel, st);
    if (!down.sent[0]) ok = ok && d2h(dv, L.dv, tok, st);
    if (!down.sent[1]) ok = ok && d2h(dq, L.dq, tok, st);
    if (!down.sent[2]) ok = ok && d2h(dk, L.dk, tok, st);
    if (!side) ok = ok && d2h(out, L.out, tok, st) && d2h(lse, L.lse, lseb, st);
    else ok = ok && cudaEventRecord(ev[3], cs) == cudaSuccess && cudaStreamWaitEvent(st, ev[3], 0) == cudaSuccess;
    if (!ok) return DF_ERR_CUDA;
    // one host round trip: the error word's read (into pageable memory, so the
    // copy returns only once it and every earlier copy and kernel of the
    // stream are done) and the stream synchronisation, which reports a
    // failure of any of them
    return df_get_device_error(base + L.ws, stream);
}

df_status df_rel_index_table(int32_t L, int32_t att_span, int32_t nb, int32_t mp, int32_t* out_dev,
                             df_stream_t stream) {
    if (L < 1 || L > 8192 || att_span < 1 || att_span > 512 || !out_dev) return DF_ERR_INVALID_ARG;
    const bool bucketing = nb > 0 && mp > 0;
    if (bucketing && (nb < 2 || mp - 1 <= nb / 2)) return DF_ERR_UNSUPPORTED;
    return cuda_status(
        launch_delta_table(L, att_span, bucketing ? nb : 0, bucketing ? mp : 0, out_dev, (cudaStream_t)stream));
}

df_status df_dropout_keep_mask(const df_attn_params* a, int32_t b, int32_t h, int32_t form, uint8_t* out_dev,
                               df_stream_t stream) {
    ProblemDev p;
    df_status s = resolve(a, p);
    if (s != DF_OK) return s;
    if (b < 0 || b >= p.B || h < 0 || h >= p.H || (form != 0 && form != 1) || !out_dev) return DF_ERR_INVALID_ARG;
    if (a->cu_seqlens && ((uintptr_t)a->cu_seqlens & 3u)) return DF_ERR_INVALID_ARG;
    return cuda_status(launch_keep_mask(p, b, h, form, out_dev, (cudaStream_t)stream));
}

df_status df_get_device_error(const void* workspace, df_stream_t stream) {
    if (!workspace) return DF_ERR_WORKSPACE;
    int word = 0;
    if (cudaMemcpyAsync(&word, workspace, sizeof(int), cudaMemcpyDeviceToHost, (cudaStream_t)stream) !=
        cudaSuccess)
        return DF_ERR_CUDA;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return DF_ERR_CUDA;
    return (df_status)word;
}

}  // extern "C"
