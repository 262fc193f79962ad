// df_internal.h -- structures shared by the host side of libdfattn and its
// kernels (not part of the public ABI).
#pragma once

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#include "../../include/df_attn.h"

namespace df {

// Everything a kernel needs to know about one attention call.
struct ProblemDev {
    int B, L, H, D, R, span, nb, mp;
    int T;                    // total tokens (B * L when padded)
    const int32_t* cu;        // device cu_seqlens or nullptr (padded)
    const uint8_t* qmask;     // padded only, [B * L] or nullptr
    const uint8_t* kmask;
    float scale;              // c
    float drop_scale;         // 1 / (1 - p)
    uint32_t keep_thr;        // keep iff philox word < keep_thr (unless keep_all)
    int keep_all;             // 1 when p == 0
    int dropout;              // p > 0
    uint32_t seed_lo, seed_hi, philox_offset;
    int* err;                 // device error word (workspace)
    // bounded waits: a wait gives up once wait_ns have passed AND wait_probes
    // probes have failed (defaults 2 s and 2^20; df_attn_debug_inject_stall
    // shortens them for its test)
    unsigned long long wait_ns;
    uint32_t wait_probes;
    // test-only stall injection (df_attn_debug_inject_stall): the MMA-issuing
    // warp of every CTA of kernel `fault_kernel` (0 forward, 1 dQ, 2 dK/dV)
    // stops before tile `fault_tile`; -1 = off
    int fault_kernel;
    int fault_tile;
    // stored band bias: key blocks kept on each side of a query block, slots
    // per query block (2 bias_kb + 1), and the caller's saved-bias buffer
    // (df_attn_params.band_bias; the forward writes it, the backward reads
    // it) or nullptr
    int bias_kb, bias_nslot;
    uint16_t* saved_bias;
    // the forward kernel's batch range: sequences b_base .. b_base + b_count
    // - 1 (b_count 0: all), so that a caller can run it in parts as inputs
    // arrive (the host-buffer step); the CTAs of sequences before b_base
    // exit at once
    int b_base, b_count;
};

// Workspace carve-up (device pointers, all 256-byte aligned).
struct Workspace {
    int* err;                 // error word
    int32_t* dtab;            // [2L - 1] delta(r) at r + L - 1
    float* relb;              // [H, 4, T]: c*log2e * (Q.Kr[0], Q.Kr[R-1], K.Qr[0], K.Qr[R-1])
    float* rowterm;           // [H, T] Dl_i (backward)
    void* G;                  // [T, H, R] diagonal sums of dZ by row (backward)
    void* Gp;                 // [T, H, R] diagonal sums of dZ by column (backward)
    float* part_kr;           // [nchunk, H, R, D] partial dKr (backward)
    float* part_qr;           // [nchunk, H, R, D] partial dQr (backward)
    float* acc32a;            // [T, H, D] fp32 dQ before the relative term (backward)
    float* acc32b;            // [T, H, D] fp32 dK before the relative term (backward)
    uint16_t* bias;           // stored band bias, [bias_rows, 128] fp16 (backward, tensor-core path)
    size_t bias_rows;
    int nchunk;
    int Rp;                   // row length of G / G' (R, or R rounded up to 64 on the tensor-core path)
    size_t bytes;
};

// Launch helpers implemented in the .cu files.  Each returns a cudaError_t
// as int (0 = success).
int launch_delta_table(int L, int span, int nb, int mp, int32_t* out, cudaStream_t st);
int launch_check_cu(const ProblemDev& p, cudaStream_t st);
int launch_clear_error(int* err, cudaStream_t st);
// (tokens tok0 .. tok1 - 1; tok1 < 0: through the last token)
int launch_relbias(const ProblemDev& p, df_dtype dt, const void* q, const void* k, const void* qr, const void* kr,
                   float* relb, cudaStream_t st, int tok0 = 0, int tok1 = -1);
int launch_rowterm(const ProblemDev& p, df_dtype dt, const void* out, const void* dout, float* rowterm,
                   cudaStream_t st);
int launch_keep_mask(const ProblemDev& p, int b, int h, int form, uint8_t* out, cudaStream_t st);
// Element-wise fp32 <-> fp16 (round to nearest even) of up to kConvSegs
// arrays in one launch (the fast fp32 mode); every count is a multiple of 4
// and every pointer 16-byte aligned.
constexpr int kConvSegs = 8;
struct ConvList {
    const void* src[kConvSegs];
    void* dst[kConvSegs];
    long long n[kConvSegs];   // elements
    int nseg;
};
int launch_convert(const ConvList& cl, bool to_half, cudaStream_t st);

// strict fp32 path
int launch_fwd_f32(const ProblemDev& p, const Workspace& ws, const float* q, const float* k, const float* v,
                   const float* qr, const float* kr, float* out, float* lse, cudaStream_t st);
int launch_bwd_f32(const ProblemDev& p, const Workspace& ws, const float* q, const float* k, const float* v,
                   const float* qr, const float* kr, const float* lse, const float* dout, float* dq, float* dk,
                   float* dv, float* dqr, float* dkr, cudaStream_t st);

// tensor-core path (bf16 / fp16)
int launch_fwd_tc(const ProblemDev& p, const Workspace& ws, df_dtype dt, const void* q, const void* k,
                  const void* v, const void* qr, const void* kr, void* out, float* lse, cudaStream_t st);
// Optional hook of the tensor-core backward: called with the launching stream
// right after the launches that finish dV (point 0), dQ (point 1, on the
// stream of the dQ kernel) and dK (point 2), so that a caller can start
// copying those gradients while the rest runs.
struct BwdHook {
    void (*fn)(void* ctx, int point, cudaStream_t st);
    void* ctx;
};
// The tensor-core backward from the forward's O and LSE: row terms, row /
// column biases, band bias (unless saved), both kernels and both halves of
// the relative-position gradients.
int launch_bwd_tc(const ProblemDev& p, const Workspace& ws, df_dtype dt, const void* q, const void* k,
                  const void* v, const void* qr, const void* kr, const void* out, const float* lse,
                  const void* dout, void* dq, void* dk, void* dv, void* dqr, void* dkr, cudaStream_t st,
                  const BwdHook* hook = nullptr);

// the two attention-backward kernels (df_bwd_dq.cu, df_bwd_dkv.cu): rows r1 / r2,
// columns c1 / c2; band tiles read the stored band bias (ws.bias)
int launch_bwd_dq(const ProblemDev& p, const Workspace& ws, df_dtype dt, const void* r1, const void* r2,
                  const void* c1, const void* c2, void* Gbuf, int Rp, float* acc1, void* acc2, const float* lse,
                  cudaStream_t st);
int launch_bwd_dkv(const ProblemDev& p, const Workspace& ws, df_dtype dt, const void* r1, const void* r2,
                   const void* c1, const void* c2, void* Gbuf, int Rp, float* acc1, void* acc2, const float* lse,
                   cudaStream_t st);
// the stored band bias of every band block (df_bias.cu)
int launch_band_bias(const ProblemDev& p, const Workspace& ws, df_dtype dt, const void* q, const void* k,
                     const void* qr, const void* kr, cudaStream_t st);
// One half of the relative-position gradients (df_rel.cu).  Half 0, from G
// (the dQ kernel's diagonal sums):  dQ = acc(dQ) + G Kr,  dKr = sum G^T Q.
// Half 1, from G' (the dK/dV kernel's):  dK = acc(dK) + G' Qr,  dQr = sum G'^T K.
// x / xr are Q / Kr (half 0) or K / Qr (half 1); out_tok is dQ / dK and
// out_rel dKr / dQr.  The hook is called at point 1 + half once out_tok is final.
int launch_rel_tc(const ProblemDev& p, const Workspace& ws, df_dtype dt, int Rp, int half, const void* x,
                  const void* xr, void* out_tok, void* out_rel, cudaStream_t st, const BwdHook* hook = nullptr);

// Optional benchmark timing hooks (df_attn_set_profile_events): record the
// begin / end event of a kernel phase on the launching stream.
enum ProfPhase { kProfFwd = 0, kProfDq = 1, kProfDkv = 2, kProfRel = 3, kProfPhases = 4 };
void prof_record(int phase, int end, cudaStream_t st);

// Encode a 2-D or 3-D tiled TMA descriptor (innermost dimension first);
// dtype_code 0 = bf16, 1 = fp16, 2 = fp32.  Returns 0 on success.
int encode_tmap(void* tmap, int dtype_code, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
                const uint32_t* box, int swizzle_bytes, const void* base);

}  // namespace df
