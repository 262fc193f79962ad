// df_aux.cu -- small kernels around the attention kernels: the relative-
// position index table, the cu_seqlens consistency check, the per-token
// relative-position dot products used by tiles whose relative index is
// clamped (saturated tiles), and the backward row term Dl_i = dO_i . O_i.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "df_common.cuh"

namespace df {

// delta(r) for r = -(L-1) .. L-1 at out[r + L - 1].
__global__ void delta_table_kernel(int L, int span, int nb, int mp, int32_t* out) {
    const int n = 2 * L - 1;
    for (int x = blockIdx.x * blockDim.x + threadIdx.x; x < n; x += gridDim.x * blockDim.x)
        out[x] = delta_of(x - (L - 1), span, nb, mp);
}

int launch_delta_table(int L, int span, int nb, int mp, int32_t* out, cudaStream_t st) {
    const int n = 2 * L - 1;
    int blocks = (n + 255) / 256;
    if (blocks > 1024) blocks = 1024;
    delta_table_kernel<<<blocks, 256, 0, st>>>(L, span, nb, mp, out);
    return (int)cudaGetLastError();
}

// cu_seqlens must start at 0, grow by 1 .. L per sequence and end at T.
__global__ void check_cu_kernel(ProblemDev p) {
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    bool bad = p.cu[0] != 0 || p.cu[p.B] != p.T;
    for (int b = 0; b < p.B && !bad; ++b) {
        const int n = p.cu[b + 1] - p.cu[b];
        bad = n < 1 || n > p.L;
    }
    if (bad) raise_error(p.err, DF_ERR_DEVICE_ARG);
}

int launch_check_cu(const ProblemDev& p, cudaStream_t st) {
    check_cu_kernel<<<1, 32, 0, st>>>(p);
    return (int)cudaGetLastError();
}

int launch_clear_error(int* err, cudaStream_t st) { return (int)cudaMemsetAsync(err, 0, sizeof(int), st); }

template <typename T>
DF_DEV float to_f(T x);
template <>
DF_DEV float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }
template <>
DF_DEV float to_f<__half>(__half x) { return __half2float(x); }
template <>
DF_DEV float to_f<float>(float x) { return x; }

DF_DEV float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Per (token t, head h): the four dot products, stored [H, 4, T]: Q_t.Kr[0], Q_t.Kr[R-1],
// K_t.Qr[0], K_t.Qr[R-1], pre-multiplied by c*log2(e) (the kernels work in
// base-2 exponent units).  A masked key gets -inf in its two K terms, which
// is how the key mask enters saturated tiles.  One warp per (t, h).
template <typename T>
__global__ void relbias_kernel(ProblemDev p, const T* __restrict__ q, const T* __restrict__ k,
                               const T* __restrict__ qr, const T* __restrict__ kr, float* __restrict__ relb) {
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (warp >= p.T * p.H) return;
    const int t = warp / p.H, h = warp % p.H;
    const int D = p.D, R = p.R;
    const T* qt = q + ((size_t)t * p.H + h) * D;
    const T* kt = k + ((size_t)t * p.H + h) * D;
    const T* kr0 = kr + (size_t)h * R * D;
    const T* kr1 = kr0 + (size_t)(R - 1) * D;
    const T* qr0 = qr + (size_t)h * R * D;
    const T* qr1 = qr0 + (size_t)(R - 1) * D;
    float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
    for (int d = lane; d < D; d += 32) {
        const float qd = to_f(qt[d]), kd = to_f(kt[d]);
        a0 = fmaf(qd, to_f(kr0[d]), a0);
        a1 = fmaf(qd, to_f(kr1[d]), a1);
        b0 = fmaf(kd, to_f(qr0[d]), b0);
        b1 = fmaf(kd, to_f(qr1[d]), b1);
    }
    a0 = warp_sum(a0);
    a1 = warp_sum(a1);
    b0 = warp_sum(b0);
    b1 = warp_sum(b1);
    if (lane == 0) {
        const float sc = p.scale * 1.4426950408889634f;
        bool kvalid = true;
        if (p.kmask) kvalid = p.kmask[t] != 0;
        const size_t T = (size_t)p.T, base = (size_t)h * 4 * T + t;
        relb[base] = a0 * sc;
        relb[base + T] = a1 * sc;
        relb[base + 2 * T] = kvalid ? b0 * sc : -INFINITY;
        relb[base + 3 * T] = kvalid ? b1 * sc : -INFINITY;
    }
}

int launch_relbias(const ProblemDev& p, df_dtype dt, const void* q, const void* k, const void* qr, const void* kr,
                   float* relb, cudaStream_t st) {
    const long warps = (long)p.T * p.H;
    const int blocks = (int)((warps * 32 + 255) / 256);
    if (dt == DF_BF16)
        relbias_kernel<__nv_bfloat16><<<blocks, 256, 0, st>>>(p, (const __nv_bfloat16*)q, (const __nv_bfloat16*)k,
                                                              (const __nv_bfloat16*)qr, (const __nv_bfloat16*)kr,
                                                              relb);
    else if (dt == DF_FP16)
        relbias_kernel<__half><<<blocks, 256, 0, st>>>(p, (const __half*)q, (const __half*)k, (const __half*)qr,
                                                       (const __half*)kr, relb);
    else
        relbias_kernel<float><<<blocks, 256, 0, st>>>(p, (const float*)q, (const float*)k, (const float*)qr,
                                                      (const float*)kr, relb);
    return (int)cudaGetLastError();
}

// Dl_i = sum_d dO[i, d] * O[i, d] in fp32, stored at the LSE index of row i.
template <typename T>
__global__ void rowterm_kernel(ProblemDev p, const T* __restrict__ o, const T* __restrict__ dout,
                               float* __restrict__ rowterm) {
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (warp >= p.B * p.L * p.H) return;
    // (b, i, h) over the padded index space; packed sequences shorter than L
    // leave the tail of their range unused.
    const int h = warp % p.H;
    const int bi = warp / p.H;
    const int b = bi / p.L, i = bi % p.L;
    int t0, n;
    seq_range(p, b, t0, n);
    if (n < 0 || n > p.L || t0 < 0 || t0 + n > p.T || i >= n) return;
    const size_t base = ((size_t)(t0 + i) * p.H + h) * p.D;
    float acc = 0.f;
    for (int d = lane; d < p.D; d += 32) acc = fmaf(to_f(dout[base + d]), to_f(o[base + d]), acc);
    acc = warp_sum(acc);
    if (lane == 0) rowterm[lse_index(p, b, h, t0, i)] = acc;
}

int launch_rowterm(const ProblemDev& p, df_dtype dt, const void* out, const void* dout, float* rowterm,
                   cudaStream_t st) {
    const long warps = (long)p.B * p.L * p.H;
    const int blocks = (int)((warps * 32 + 255) / 256);
    if (dt == DF_BF16)
        rowterm_kernel<__nv_bfloat16><<<blocks, 256, 0, st>>>(p, (const __nv_bfloat16*)out,
                                                              (const __nv_bfloat16*)dout, rowterm);
    else if (dt == DF_FP16)
        rowterm_kernel<__half><<<blocks, 256, 0, st>>>(p, (const __half*)out, (const __half*)dout, rowterm);
    else
        rowterm_kernel<float><<<blocks, 256, 0, st>>>(p, (const float*)out, (const float*)dout, rowterm);
    return (int)cudaGetLastError();
}

}  // namespace df
