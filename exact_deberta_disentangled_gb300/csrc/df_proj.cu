// df_proj.cu -- the steps on either side of the attention: the fused QKV
// projection and the relative-position projections, forward and backward
// ("DisentangledFlash", section "Status": the fused QKV projection is always
// on; section "Hugging Face usage": the query / key / value and relative-
// position projections stay in the autograd graph).
//
// DeBERTa-v2/v3 (shared attention keys) projects the hidden states with one
// weight W = [W_q; W_k; W_v] ([3, H D, C]) and the layer-normalised relative
// embeddings with the same W_q and W_k:
//   [Q; K; V] = X W_j^T + b_j                X [T, C] -> [3, T, H D]
//   E = LayerNorm(rel) ([R, C], gamma, beta, eps)
//   Qr[h] = E W_q[h]^T + b_q[h],  Kr[h] = E W_k[h]^T + b_k[h]    -> [H, R, D]
// with W_q[h] the D rows of head h.  The products are plain GEMMs (cuBLASLt,
// fp32 accumulation, bias in the epilogue, no workspace); the layer norm, its
// backward and the bias / gamma / beta gradient sums are small kernels here,
// every sum in a fixed order.
#include <cublasLt.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>
#include <mutex>

#include "df_internal.h"

namespace df {
namespace {

std::mutex g_lt_mu;
cublasLtHandle_t g_lt = nullptr;
bool g_lt_tried = false;

cublasLtHandle_t lt_handle() {
    std::lock_guard<std::mutex> lock(g_lt_mu);
    if (!g_lt_tried) {
        g_lt_tried = true;
        if (cublasLtCreate(&g_lt) != CUBLAS_STATUS_SUCCESS) g_lt = nullptr;
    }
    return g_lt;
}

// Row-major C[M, N] (ldc) = op_a(A) op_b(B) (+ beta C) (+ bias[N] added to
// every row), `batch` independent products with element strides sA, sB, sC,
// sBias.  op_a(A) is [M, K]: A stored [M, K] (lda) or, ta, stored [K, M];
// op_b(B) is [K, N]: B stored [K, N] (ldb) or, tb, stored [N, K].  A and B
// are of type ab, C of type c.  A row-major product is the column-major
// product of the same memory with the operands swapped, which is what
// cuBLASLt is given.
int gemm(cudaDataType_t ab, cudaDataType_t ct, bool ta, bool tb, int M, int N, int K, const void* A, long lda,
         long sA, const void* B, long ldb, long sB, float beta, void* C, long ldc, long sC, const void* bias,
         long sBias, int batch, cudaStream_t st) {
    cublasLtHandle_t lt = lt_handle();
    if (!lt) return 1;
    cublasLtMatmulDesc_t op = nullptr;
    cublasLtMatrixLayout_t la = nullptr, lb = nullptr, lc = nullptr;
    cublasLtMatmulPreference_t pref = nullptr;
    int rc = 1;
    do {
        if (cublasLtMatmulDescCreate(&op, CUBLAS_COMPUTE_32F, CUDA_R_32F) != CUBLAS_STATUS_SUCCESS) break;
        // column-major operands: first = B's memory with op_b, second = A's memory with op_a
        const cublasOperation_t t1 = tb ? CUBLAS_OP_T : CUBLAS_OP_N, t2 = ta ? CUBLAS_OP_T : CUBLAS_OP_N;
        cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_TRANSA, &t1, sizeof(t1));
        cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_TRANSB, &t2, sizeof(t2));
        if (bias) {
            const cublasLtEpilogue_t ep = CUBLASLT_EPILOGUE_BIAS;
            cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_EPILOGUE, &ep, sizeof(ep));
            cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_BIAS_POINTER, &bias, sizeof(bias));
            if (batch > 1) {
                const int64_t s = sBias;
                cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_BIAS_BATCH_STRIDE, &s, sizeof(s));
            }
        }
        // column-major shapes: first operand [N, K] (stored [K, N] when tb), second [K, M] ([M, K] when ta)
        if (cublasLtMatrixLayoutCreate(&la, ab, tb ? K : N, tb ? N : K, ldb) != CUBLAS_STATUS_SUCCESS) break;
        if (cublasLtMatrixLayoutCreate(&lb, ab, ta ? M : K, ta ? K : M, lda) != CUBLAS_STATUS_SUCCESS) break;
        if (cublasLtMatrixLayoutCreate(&lc, ct, N, M, ldc) != CUBLAS_STATUS_SUCCESS) break;
        if (batch > 1) {
            const int32_t bc = batch;
            const int64_t s1 = sB, s2 = sA, s3 = sC;
            cublasLtMatrixLayoutSetAttribute(la, CUBLASLT_MATRIX_LAYOUT_BATCH_COUNT, &bc, sizeof(bc));
            cublasLtMatrixLayoutSetAttribute(la, CUBLASLT_MATRIX_LAYOUT_STRIDED_BATCH_OFFSET, &s1, sizeof(s1));
            cublasLtMatrixLayoutSetAttribute(lb, CUBLASLT_MATRIX_LAYOUT_BATCH_COUNT, &bc, sizeof(bc));
            cublasLtMatrixLayoutSetAttribute(lb, CUBLASLT_MATRIX_LAYOUT_STRIDED_BATCH_OFFSET, &s2, sizeof(s2));
            cublasLtMatrixLayoutSetAttribute(lc, CUBLASLT_MATRIX_LAYOUT_BATCH_COUNT, &bc, sizeof(bc));
            cublasLtMatrixLayoutSetAttribute(lc, CUBLASLT_MATRIX_LAYOUT_STRIDED_BATCH_OFFSET, &s3, sizeof(s3));
        }
        if (cublasLtMatmulPreferenceCreate(&pref) != CUBLAS_STATUS_SUCCESS) break;
        const size_t ws = 0;   // no scratch: nothing is allocated
        cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES, &ws, sizeof(ws));
        cublasLtMatmulHeuristicResult_t heur;
        int found = 0;
        if (cublasLtMatmulAlgoGetHeuristic(lt, op, la, lb, lc, lc, pref, 1, &heur, &found) != CUBLAS_STATUS_SUCCESS ||
            found < 1)
            break;
        const float alpha = 1.f;
        if (cublasLtMatmul(lt, op, &alpha, B, la, A, lb, &beta, C, lc, C, lc, &heur.algo, nullptr, 0, st) !=
            CUBLAS_STATUS_SUCCESS)
            break;
        rc = 0;
    } while (false);
    if (pref) cublasLtMatmulPreferenceDestroy(pref);
    if (lc) cublasLtMatrixLayoutDestroy(lc);
    if (lb) cublasLtMatrixLayoutDestroy(lb);
    if (la) cublasLtMatrixLayoutDestroy(la);
    if (op) cublasLtMatmulDescDestroy(op);
    return rc;
}

__device__ __forceinline__ float tof(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ float tof(__half v) { return __half2float(v); }
__device__ __forceinline__ float tof(float v) { return v; }
template <typename T>
__device__ __forceinline__ T fromf(float v);
template <>
__device__ __forceinline__ __nv_bfloat16 fromf<__nv_bfloat16>(float v) { return __float2bfloat16(v); }
template <>
__device__ __forceinline__ __half fromf<__half>(float v) { return __float2half(v); }

__device__ __forceinline__ float warp_sum(float x) {
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Layer norm of each row of x [R, C], one warp per row, fp32 statistics:
// y = (x - mean) rstd gamma + beta;  stats[r] = (mean, rstd).
template <typename T>
__global__ void layernorm_fwd_kernel(const T* __restrict__ x, const T* __restrict__ gamma, const T* __restrict__ beta,
                                     float eps, int R, int C, T* __restrict__ y, float* __restrict__ stats) {
    const int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (r >= R) return;
    const T* xr = x + (size_t)r * C;
    float s = 0.f;
    for (int c = lane; c < C; c += 32) s += tof(xr[c]);
    const float mean = warp_sum(s) / (float)C;
    float v = 0.f;
    for (int c = lane; c < C; c += 32) {
        const float d = tof(xr[c]) - mean;
        v += d * d;
    }
    const float rstd = rsqrtf(warp_sum(v) / (float)C + eps);
    for (int c = lane; c < C; c += 32)
        y[(size_t)r * C + c] = fromf<T>((tof(xr[c]) - mean) * rstd * tof(gamma[c]) + tof(beta[c]));
    if (lane == 0) {
        stats[2 * r] = mean;
        stats[2 * r + 1] = rstd;
    }
}

// Layer-norm backward of each row: with xh = (x - mean) rstd and g = dy gamma,
// dx = rstd (g - mean(g) - xh mean(g xh)).
template <typename T>
__global__ void layernorm_bwd_kernel(const T* __restrict__ x, const T* __restrict__ gamma,
                                     const float* __restrict__ stats, const float* __restrict__ dy, int R, int C,
                                     T* __restrict__ dx) {
    const int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (r >= R) return;
    const float mean = stats[2 * r], rstd = stats[2 * r + 1];
    const T* xr = x + (size_t)r * C;
    const float* dyr = dy + (size_t)r * C;
    float sg = 0.f, sgx = 0.f;
    for (int c = lane; c < C; c += 32) {
        const float g = dyr[c] * tof(gamma[c]);
        sg += g;
        sgx += g * (tof(xr[c]) - mean) * rstd;
    }
    sg = warp_sum(sg) / (float)C;
    sgx = warp_sum(sgx) / (float)C;
    for (int c = lane; c < C; c += 32) {
        const float xh = (tof(xr[c]) - mean) * rstd;
        dx[(size_t)r * C + c] = fromf<T>(rstd * (dyr[c] * tof(gamma[c]) - sg - xh * sgx));
    }
}

// Column sums in two passes, both in a fixed order (so the result is
// deterministic) and with enough threads to stream the matrix:
//   pass 1: part[k][0][col] = sum of rows in chunk k of column col, where
//           col = j * C + c addresses column c of matrix a[j] ([R, C] at
//           a + j * sa); with xs (the layer norm's input) also
//           part[k][1][col] = sum over the chunk of a[r, c] xh[r, c]
//   pass 2: out[col] (+)= sum over k of part[k][0][col] (k ascending), and
//           out2[c] (+)= sum over k of part[k][1][c]
constexpr int kColChunks = 64;

template <typename TA, typename T>
__global__ void colsum_part_kernel(const TA* __restrict__ a, long sa, int nmat, int R, int C, int rows_per,
                                   const T* __restrict__ xs, const float* __restrict__ stats,
                                   float* __restrict__ part) {
    const int col = blockIdx.x * blockDim.x + threadIdx.x, k = blockIdx.y;
    const int ncol = nmat * C;
    if (col >= ncol) return;
    const int j = col / C, c = col % C;
    const TA* aj = a + (size_t)j * sa;
    const int r0 = k * rows_per, r1 = min(R, r0 + rows_per);
    float s = 0.f, s2 = 0.f;
    for (int r = r0; r < r1; ++r) {
        const float v = tof(aj[(size_t)r * C + c]);
        s += v;
        if (xs) s2 += v * (tof(xs[(size_t)r * C + c]) - stats[2 * r]) * stats[2 * r + 1];
    }
    part[((size_t)k * 2) * ncol + col] = s;
    part[((size_t)k * 2 + 1) * ncol + col] = s2;
}

template <typename T>
__global__ void colsum_final_kernel(const float* __restrict__ part, int nchunk, int ncol, int accumulate,
                                    T* __restrict__ out, T* __restrict__ out2) {
    const int col = blockIdx.x * blockDim.x + threadIdx.x;
    if (col >= ncol) return;
    float s = 0.f, s2 = 0.f;
    for (int k = 0; k < nchunk; ++k) {
        s += part[((size_t)k * 2) * ncol + col];
        s2 += part[((size_t)k * 2 + 1) * ncol + col];
    }
    if (accumulate) s += tof(out[col]);
    out[col] = fromf<T>(s);
    if (out2) {
        if (accumulate) s2 += tof(out2[col]);
        out2[col] = fromf<T>(s2);
    }
}

size_t colsum_ws_bytes(int ncol) { return (size_t)kColChunks * 2 * (size_t)ncol * sizeof(float); }

template <typename TA, typename T>
void colsum(const TA* a, long sa, int nmat, int R, int C, int accumulate, T* out, const T* xs, const float* stats,
            T* out2, float* part, cudaStream_t st) {
    const int ncol = nmat * C;
    const int nchunk = R < kColChunks ? R : kColChunks;
    const int rows_per = (R + nchunk - 1) / nchunk;
    colsum_part_kernel<TA, T><<<dim3((ncol + 127) / 128, nchunk), 128, 0, st>>>(a, sa, nmat, R, C, rows_per, xs, stats,
                                                                               part);
    colsum_final_kernel<T><<<(ncol + 127) / 128, 128, 0, st>>>(part, nchunk, ncol, accumulate, out, out2);
}

// [H, R, D] -> [R, H D]
template <typename T>
__global__ void heads_to_rows_kernel(const T* __restrict__ in, int H, int R, int D, T* __restrict__ out) {
    const long n = (long)H * R * D;
    for (long x = (long)blockIdx.x * blockDim.x + threadIdx.x; x < n; x += (long)gridDim.x * blockDim.x) {
        const int d = (int)(x % D);
        const long hr = x / D;
        const int r = (int)(hr % R), h = (int)(hr / R);
        out[((size_t)r * H + h) * D + d] = in[x];
    }
}

int nblocks(long n, int per) {
    long b = (n + per - 1) / per;
    return (int)(b < 1 ? 1 : (b > 4096 ? 4096 : b));
}

cudaDataType_t cuda_type(df_dtype dt) { return dt == DF_BF16 ? CUDA_R_16BF : CUDA_R_16F; }

bool al16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

template <typename T>
df_status rel_bwd_impl(int R, int C, int H, int D, df_dtype dt, const void* rel, const void* gamma,
                       const void* rel_ln, const float* stats, const void* w, const void* dqr, const void* dkr,
                       void* drel, void* dgamma, void* dbeta, void* dw, void* dbias, int acc, char* ws,
                       cudaStream_t st) {
    const int HD = H * D;
    const cudaDataType_t ab = cuda_type(dt);
    T* dq_t = reinterpret_cast<T*>(ws);
    T* dk_t = dq_t + (size_t)R * HD;
    float* de = reinterpret_cast<float*>(ws + 2 * sizeof(T) * (size_t)R * HD);
    float* part = de + (size_t)R * C;
    const long n = (long)H * R * D;
    heads_to_rows_kernel<T><<<nblocks(n, 256), 256, 0, st>>>((const T*)dqr, H, R, D, dq_t);
    heads_to_rows_kernel<T><<<nblocks(n, 256), 256, 0, st>>>((const T*)dkr, H, R, D, dk_t);
    const T* W = (const T*)w;
    T* dW = (T*)dw;
    const float b0 = acc ? 1.f : 0.f;
    // dW_q (+)= dQr_t^T E, dW_k (+)= dKr_t^T E     ([HD, R] x [R, C])
    if (gemm(ab, ab, true, false, HD, C, R, dq_t, HD, 0, rel_ln, C, 0, b0, dW, C, 0, nullptr, 0, 1, st) ||
        gemm(ab, ab, true, false, HD, C, R, dk_t, HD, 0, rel_ln, C, 0, b0, dW + (size_t)HD * C, C, 0, nullptr, 0, 1,
             st))
        return DF_ERR_CUDA;
    if (dbias) {   // rows q and k of dbias: the two transposed gradients are adjacent ([2, R, HD])
        colsum<T, T>(dq_t, (long)R * HD, 2, R, HD, acc, (T*)dbias, (const T*)nullptr, nullptr, (T*)nullptr, part, st);
    }
    // dE = dQr_t W_q + dKr_t W_k    ([R, HD] x [HD, C], fp32)
    if (gemm(ab, CUDA_R_32F, false, false, R, C, HD, dq_t, HD, 0, W, C, 0, 0.f, de, C, 0, nullptr, 0, 1, st) ||
        gemm(ab, CUDA_R_32F, false, false, R, C, HD, dk_t, HD, 0, W + (size_t)HD * C, C, 0, 1.f, de, C, 0, nullptr,
             0, 1, st))
        return DF_ERR_CUDA;
    layernorm_bwd_kernel<T><<<nblocks(R, 8), 256, 0, st>>>((const T*)rel, (const T*)gamma, stats, de, R, C, (T*)drel);
    colsum<float, T>(de, 0, 1, R, C, acc, (T*)dbeta, (const T*)rel, stats, (T*)dgamma, part, st);
    return cudaGetLastError() == cudaSuccess ? DF_OK : DF_ERR_CUDA;
}

}  // namespace
}  // namespace df

using namespace df;

extern "C" {

df_status df_qkv_proj_fwd(int32_t T, int32_t C, int32_t HD, df_dtype dt, const void* x, const void* w,
                          const void* bias, void* qkv, df_stream_t stream) {
    if (T < 1 || C < 1 || HD < 1 || !x || !w || !qkv) return DF_ERR_INVALID_ARG;
    if (dt != DF_BF16 && dt != DF_FP16) return DF_ERR_UNSUPPORTED;
    if (!al16(x) || !al16(w) || !al16(qkv) || (bias && !al16(bias)) || C % 8 || HD % 8) return DF_ERR_INVALID_ARG;
    const cudaDataType_t ab = cuda_type(dt);
    // [Q; K; V][j] = X W_j^T + b_j: one batched product over j
    if (gemm(ab, ab, false, true, T, HD, C, x, C, 0, w, C, (long)HD * C, 0.f, qkv, HD, (long)T * HD, bias, HD, 3,
             (cudaStream_t)stream))
        return DF_ERR_CUDA;
    return DF_OK;
}

size_t df_qkv_proj_workspace_size(int32_t HD) { return HD < 1 ? 0 : colsum_ws_bytes(3 * HD); }

df_status df_qkv_proj_bwd(int32_t T, int32_t C, int32_t HD, df_dtype dt, const void* x, const void* w,
                          const void* dqkv, void* dx, void* dw, void* dbias, int32_t accumulate, void* workspace,
                          size_t workspace_bytes, df_stream_t stream) {
    if (T < 1 || C < 1 || HD < 1 || !x || !w || !dqkv || !dx || !dw) return DF_ERR_INVALID_ARG;
    if (dt != DF_BF16 && dt != DF_FP16) return DF_ERR_UNSUPPORTED;
    if (!al16(x) || !al16(w) || !al16(dqkv) || !al16(dx) || !al16(dw) || (dbias && !al16(dbias)) || C % 8 || HD % 8)
        return DF_ERR_INVALID_ARG;
    if (dbias && (!workspace || !al16(workspace) || workspace_bytes < df_qkv_proj_workspace_size(HD)))
        return DF_ERR_WORKSPACE;
    cudaStream_t st = (cudaStream_t)stream;
    const cudaDataType_t ab = cuda_type(dt);
    const size_t es = 2;
    const char* dy = (const char*)dqkv;
    const char* W = (const char*)w;
    // dX = sum_j dY_j W_j   ([T, HD] x [HD, C]), j in order
    for (int j = 0; j < 3; ++j)
        if (gemm(ab, ab, false, false, T, C, HD, dy + es * (size_t)j * T * HD, HD, 0, W + es * (size_t)j * HD * C, C,
                 0, j ? 1.f : 0.f, dx, C, 0, nullptr, 0, 1, st))
            return DF_ERR_CUDA;
    // dW_j (+)= dY_j^T X    ([HD, T] x [T, C]), batched over j
    if (gemm(ab, ab, true, false, HD, C, T, dqkv, HD, (long)T * HD, x, C, 0, accumulate ? 1.f : 0.f, dw, C,
             (long)HD * C, nullptr, 0, 3, st))
        return DF_ERR_CUDA;
    if (dbias) {
        float* part = (float*)workspace;
        if (dt == DF_BF16)
            colsum<__nv_bfloat16, __nv_bfloat16>((const __nv_bfloat16*)dqkv, (long)T * HD, 3, T, HD, accumulate,
                                                 (__nv_bfloat16*)dbias, (const __nv_bfloat16*)nullptr, nullptr,
                                                 (__nv_bfloat16*)nullptr, part, st);
        else
            colsum<__half, __half>((const __half*)dqkv, (long)T * HD, 3, T, HD, accumulate, (__half*)dbias,
                                   (const __half*)nullptr, nullptr, (__half*)nullptr, part, st);
    }
    return cudaGetLastError() == cudaSuccess ? DF_OK : DF_ERR_CUDA;
}

size_t df_rel_proj_workspace_size(int32_t R, int32_t C, int32_t H, int32_t D) {
    if (R < 1 || C < 1 || H < 1 || D < 1) return 0;
    const int ncol = 2 * H * D > C ? 2 * H * D : C;
    return 2 * 2 * (size_t)R * H * D + 4 * (size_t)R * C + colsum_ws_bytes(ncol);
}

df_status df_rel_proj_fwd(int32_t R, int32_t C, int32_t H, int32_t D, df_dtype dt, const void* rel, const void* gamma,
                          const void* beta, float eps, const void* w, const void* bias, void* rel_ln, float* ln_stats,
                          void* qr, void* kr, df_stream_t stream) {
    if (R < 1 || C < 1 || H < 1 || D < 1 || !rel || !gamma || !beta || !w || !rel_ln || !ln_stats || !qr || !kr)
        return DF_ERR_INVALID_ARG;
    if (dt != DF_BF16 && dt != DF_FP16) return DF_ERR_UNSUPPORTED;
    if (!(eps > 0.f) || !al16(w) || !al16(rel_ln) || !al16(qr) || !al16(kr) || (bias && !al16(bias)) || C % 8 ||
        D % 8)
        return DF_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    const int HD = H * D;
    if (dt == DF_BF16)
        layernorm_fwd_kernel<__nv_bfloat16><<<nblocks(R, 8), 256, 0, st>>>(
            (const __nv_bfloat16*)rel, (const __nv_bfloat16*)gamma, (const __nv_bfloat16*)beta, eps, R, C,
            (__nv_bfloat16*)rel_ln, ln_stats);
    else
        layernorm_fwd_kernel<__half><<<nblocks(R, 8), 256, 0, st>>>((const __half*)rel, (const __half*)gamma,
                                                                   (const __half*)beta, eps, R, C, (__half*)rel_ln,
                                                                   ln_stats);
    const cudaDataType_t ab = cuda_type(dt);
    const size_t es = 2;   // bytes per element
    const char* W = (const char*)w;
    const char* bz = (const char*)bias;
    // Qr[h] = E W_q[h]^T + b_q[h], Kr[h] = E W_k[h]^T + b_k[h]: batched over heads
    // (W_q[h] = D rows of W_q, W_k = rows [HD, 2 HD) of the fused weight; E shared)
    if (gemm(ab, ab, false, true, R, D, C, rel_ln, C, 0, W, C, (long)D * C, 0.f, qr, D, (long)R * D, bias, D, H, st) ||
        gemm(ab, ab, false, true, R, D, C, rel_ln, C, 0, W + es * (size_t)HD * C, C, (long)D * C, 0.f, kr, D,
             (long)R * D, bias ? bz + es * (size_t)HD : nullptr, D, H, st))
        return DF_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? DF_OK : DF_ERR_CUDA;
}

df_status df_rel_proj_bwd(int32_t R, int32_t C, int32_t H, int32_t D, df_dtype dt, const void* rel,
                          const void* gamma, const void* rel_ln, const float* ln_stats, const void* w, const void* dqr,
                          const void* dkr, void* drel, void* dgamma, void* dbeta, void* dw, void* dbias,
                          int32_t accumulate, void* workspace, size_t workspace_bytes, df_stream_t stream) {
    if (R < 1 || C < 1 || H < 1 || D < 1 || !rel || !gamma || !rel_ln || !ln_stats || !w || !dqr || !dkr || !drel ||
        !dgamma || !dbeta || !dw)
        return DF_ERR_INVALID_ARG;
    if (dt != DF_BF16 && dt != DF_FP16) return DF_ERR_UNSUPPORTED;
    if (!al16(w) || !al16(rel_ln) || !al16(dqr) || !al16(dkr) || !al16(dw) || C % 8 || D % 8) return DF_ERR_INVALID_ARG;
    if (!workspace || !al16(workspace) || workspace_bytes < df_rel_proj_workspace_size(R, C, H, D))
        return DF_ERR_WORKSPACE;
    // the relative path uses W_q (rows [0, HD)) and W_k (rows [HD, 2 HD)) of the fused weight; its
    // gradients go to the same rows of dw and of dbias
    char* ws = (char*)workspace;
    if (dt == DF_BF16)
        return rel_bwd_impl<__nv_bfloat16>(R, C, H, D, dt, rel, gamma, rel_ln, ln_stats, w, dqr, dkr, drel, dgamma,
                                           dbeta, dw, dbias, accumulate, ws, (cudaStream_t)stream);
    return rel_bwd_impl<__half>(R, C, H, D, dt, rel, gamma, rel_ln, ln_stats, w, dqr, dkr, drel, dgamma, dbeta, dw,
                                dbias, accumulate, ws, (cudaStream_t)stream);
}

}  // extern "C"
