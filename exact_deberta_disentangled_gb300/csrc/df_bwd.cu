// df_bwd.cu -- the backward pass: clears the diagonal-sum buffers G / G',
// runs the dQ kernel and the dK/dV kernel (df_bwd_kernel.cuh) and then the
// relative-position gradients (df_rel.cu).
//
// "DisentangledFlash" (section "Hugging Face usage") splits the fused
// backward into a dQ kernel and a dK/dV kernel; section "Performance" counts
// the relative-position gradients.
#include "df_internal.h"

namespace df {

int launch_bwd_tc(const ProblemDev& p, const Workspace& ws, df_dtype dt, const void* q, const void* k,
                  const void* v, const void* qr, const void* kr, const float* lse, const void* dout, void* dq,
                  void* dk, void* dv, void* dqr, void* dkr, cudaStream_t st) {
    if (p.D != 32 && p.D != 64 && p.D != 128) return (int)cudaErrorInvalidValue;
    const int Rp = ws.Rp;
    const size_t gbytes = (size_t)p.T * p.H * Rp * 2;
    cudaError_t ce = cudaMemsetAsync(ws.G, 0, gbytes, st);
    if (ce == cudaSuccess) ce = cudaMemsetAsync(ws.Gp, 0, gbytes, st);
    if (ce != cudaSuccess) return (int)ce;
    // dQ kernel: rows = queries (Q, dO), columns = keys (K, V); own band Kr, cross Qr
    int e = launch_bwd_dq(p, ws, dt, q, dout, k, v, kr, qr, ws.G, Rp, ws.acc32a, nullptr, lse, st);
    if (e) return e;
    // dK/dV kernel: rows = keys (K, V), columns = queries (Q, dO); own band Qr, cross Kr
    e = launch_bwd_dkv(p, ws, dt, k, v, q, dout, qr, kr, ws.Gp, Rp, ws.acc32b, dv, lse, st);
    if (e) return e;
    return launch_rel_tc(p, ws, dt, Rp, q, k, qr, kr, dq, dk, dqr, dkr, st);
}

}  // namespace df
