// df_aux.cu -- small kernels around the attention kernels: the relative-
// position index table, the cu_seqlens consistency check, the per-token
// relative-position dot products used by tiles whose relative index is
// clamped (saturated tiles), the backward row term Dl_i = dO_i . O_i, and the
// fp32 <-> fp16 conversions of the fast fp32 mode.
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

// The dropout keep mask of sequence b, head h, as the attention kernels draw
// it: form 0 through the row generator (the forward and dQ kernels: one lane
// per query, 32 keys a call), form 1 through the column generator (the dK/dV
// kernel: one lane per key, 32 queries a call, lanes of a quad sharing their
// Philox outputs).  One warp per 32 x 32 block; out[i * n + j] = keep(i, j).
__global__ void keep_mask_kernel(ProblemDev p, int b, int h, int form, uint8_t* __restrict__ out) {
    int t0, n;
    if (!seq_ok(p, b, t0, n)) return;
    const int lane = threadIdx.x & 31;
    const long wg = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int nb32 = (n + 31) / 32;
    if (wg >= (long)nb32 * nb32) return;   // the whole warp leaves together
    const int bi = (int)(wg / nb32), bj = (int)(wg % nb32);
    if (form == 0) {
        const int i = 32 * bi + lane;
        const uint32_t k = keep_bits32_row(p, b, h, i, 32 * bj);
        if (i < n)
            for (int e = 0; e < 32 && 32 * bj + e < n; ++e) out[(size_t)i * n + 32 * bj + e] = (uint8_t)((k >> e) & 1u);
    } else {
        const int j = 32 * bj + lane;
        const uint32_t k = keep_bits32_col(p, b, h, 32 * bi, j);
        if (j < n)
            for (int q = 0; q < 32 && 32 * bi + q < n; ++q) out[(size_t)(32 * bi + q) * n + j] = (uint8_t)((k >> q) & 1u);
    }
}

int launch_keep_mask(const ProblemDev& p, int b, int h, int form, uint8_t* out, cudaStream_t st) {
    const long nb32 = (p.L + 31) / 32;
    const long warps = nb32 * nb32;
    keep_mask_kernel<<<(unsigned)((warps * 32 + 255) / 256), 256, 0, st>>>(p, b, h, form, out);
    return (int)cudaGetLastError();
}

// 16 bytes of T (8 bf16 / fp16 or 4 fp32 values) from a 16-byte aligned
// address, as floats.
template <typename T>
DF_DEV void load16(const T* src, float* f);
template <>
DF_DEV void load16<__nv_bfloat16>(const __nv_bfloat16* src, float* f) {
    const uint4 u = *reinterpret_cast<const uint4*>(src);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        f[2 * j] = __uint_as_float(w[j] << 16);
        f[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    }
}
template <>
DF_DEV void load16<__half>(const __half* src, float* f) {
    const uint4 u = *reinterpret_cast<const uint4*>(src);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float2 v = __half22float2(*reinterpret_cast<const __half2*>(&w[j]));
        f[2 * j] = v.x;
        f[2 * j + 1] = v.y;
    }
}
template <>
DF_DEV void load16<float>(const float* src, float* f) {
    const float4 v = *reinterpret_cast<const float4*>(src);
    f[0] = v.x;
    f[1] = v.y;
    f[2] = v.z;
    f[3] = v.w;
}

// Rows of D values are read 16 bytes per lane: LPR lanes per row, RPW rows
// per warp; a row's partial dot products meet by shuffles within its lanes.
template <typename T, int D>
struct RowSplit {
    static constexpr int VEC = 16 / (int)sizeof(T);
    static constexpr int LPR = D / VEC;
    static constexpr int RPW = 32 / LPR;
    static_assert(LPR >= 1 && LPR <= 32 && 32 % LPR == 0, "row split");
};

template <int LPR>
DF_DEV float group_sum(float x) {
#pragma unroll
    for (int o = LPR / 2; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

template <typename T, int VEC>
DF_DEV float dot16(const float* a, const T* b) {
    float f[VEC];
    load16<T>(b, f);
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < VEC; ++j) s = fmaf(a[j], f[j], s);
    return s;
}

// Per (token t, head h): the four dot products, stored [H, 4, T]: Q_t.Kr[0], Q_t.Kr[R-1],
// K_t.Qr[0], K_t.Qr[R-1], pre-multiplied by c*log2(e) (the kernels work in
// base-2 exponent units).  A masked key gets -inf in its two K terms, which
// is how the key mask enters saturated tiles.
template <typename T, int D>
__global__ void relbias_kernel(ProblemDev p, const T* __restrict__ q, const T* __restrict__ k,
                               const T* __restrict__ qr, const T* __restrict__ kr, float* __restrict__ relb,
                               long row0, long row1) {
    using RS = RowSplit<T, D>;
    const long gw = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31, part = lane % RS::LPR;
    const long row = row0 + gw * RS::RPW + lane / RS::LPR;   // t * H + h
    const bool ok = row < row1;
    const long rs = ok ? row : 0;                     // a row that is safe to load
    const int t = (int)(rs / p.H), h = (int)(rs % p.H);
    const int R = p.R, off = part * RS::VEC;
    float qv[RS::VEC], kv[RS::VEC];
    load16<T>(q + rs * D + off, qv);
    load16<T>(k + rs * D + off, kv);
    const T* kr0 = kr + (size_t)h * R * D + off;
    const T* qr0 = qr + (size_t)h * R * D + off;
    float a0 = dot16<T, RS::VEC>(qv, kr0), a1 = dot16<T, RS::VEC>(qv, kr0 + (size_t)(R - 1) * D);
    float b0 = dot16<T, RS::VEC>(kv, qr0), b1 = dot16<T, RS::VEC>(kv, qr0 + (size_t)(R - 1) * D);
    a0 = group_sum<RS::LPR>(a0);
    a1 = group_sum<RS::LPR>(a1);
    b0 = group_sum<RS::LPR>(b0);
    b1 = group_sum<RS::LPR>(b1);
    if (ok && part == 0) {
        const float sc = p.scale * 1.4426950408889634f;
        bool kvalid = true;
        if (p.kmask) kvalid = p.kmask[t] != 0;
        const size_t NT = (size_t)p.T, base = (size_t)h * 4 * NT + t;
        relb[base] = a0 * sc;
        relb[base + NT] = a1 * sc;
        relb[base + 2 * NT] = kvalid ? b0 * sc : -INFINITY;
        relb[base + 3 * NT] = kvalid ? b1 * sc : -INFINITY;
    }
}

template <typename T, int D>
int relbias_one(const ProblemDev& p, const void* q, const void* k, const void* qr, const void* kr, float* relb,
                cudaStream_t st, int tok0, int tok1) {
    using RS = RowSplit<T, D>;
    const long row0 = (long)tok0 * p.H, row1 = (long)tok1 * p.H;
    if (row1 <= row0) return 0;
    const long warps = (row1 - row0 + RS::RPW - 1) / RS::RPW;
    const int blocks = (int)((warps * 32 + 255) / 256);
    relbias_kernel<T, D><<<blocks, 256, 0, st>>>(p, (const T*)q, (const T*)k, (const T*)qr, (const T*)kr, relb, row0,
                                                row1);
    return (int)cudaGetLastError();
}

template <typename T>
int relbias_d(const ProblemDev& p, const void* q, const void* k, const void* qr, const void* kr, float* relb,
              cudaStream_t st, int tok0, int tok1) {
    switch (p.D) {
        case 32: return relbias_one<T, 32>(p, q, k, qr, kr, relb, st, tok0, tok1);
        case 64: return relbias_one<T, 64>(p, q, k, qr, kr, relb, st, tok0, tok1);
        case 128: return relbias_one<T, 128>(p, q, k, qr, kr, relb, st, tok0, tok1);
    }
    return (int)cudaErrorInvalidValue;
}

int launch_relbias(const ProblemDev& p, df_dtype dt, const void* q, const void* k, const void* qr, const void* kr,
                   float* relb, cudaStream_t st, int tok0, int tok1) {
    if (tok1 < 0) tok1 = p.T;
    if (dt == DF_BF16) return relbias_d<__nv_bfloat16>(p, q, k, qr, kr, relb, st, tok0, tok1);
    if (dt == DF_FP16) return relbias_d<__half>(p, q, k, qr, kr, relb, st, tok0, tok1);
    return relbias_d<float>(p, q, k, qr, kr, relb, st, tok0, tok1);
}

// Dl_i = sum_d dO[i, d] * O[i, d] in fp32, stored at the LSE index of row i.
// Rows run over the padded index space (b, i, h); packed sequences shorter
// than L leave the tail of their range unused.
template <typename T, int D>
__global__ void rowterm_kernel(ProblemDev p, const T* __restrict__ o, const T* __restrict__ dout,
                               float* __restrict__ rowterm) {
    using RS = RowSplit<T, D>;
    const long gw = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31, part = lane % RS::LPR;
    const long row = gw * RS::RPW + lane / RS::LPR;
    bool ok = row < (long)p.B * p.L * p.H;
    const long rs = ok ? row : 0;
    const int h = (int)(rs % p.H);
    const long bi = rs / p.H;
    const int b = (int)(bi / p.L), i = (int)(bi % p.L);
    int t0, n;
    seq_range(p, b, t0, n);
    ok = ok && !(n < 0 || n > p.L || t0 < 0 || t0 + n > p.T || i >= n);
    const size_t base = ok ? ((size_t)(t0 + i) * p.H + h) * D + part * RS::VEC : (size_t)part * RS::VEC;
    float ov[RS::VEC];
    load16<T>(o + base, ov);
    float acc = group_sum<RS::LPR>(dot16<T, RS::VEC>(ov, dout + base));
    if (ok && part == 0) rowterm[lse_index(p, b, h, t0, i)] = acc;
}

template <typename T, int D>
int rowterm_one(const ProblemDev& p, const void* out, const void* dout, float* rowterm, cudaStream_t st) {
    using RS = RowSplit<T, D>;
    const long warps = ((long)p.B * p.L * p.H + RS::RPW - 1) / RS::RPW;
    const int blocks = (int)((warps * 32 + 255) / 256);
    rowterm_kernel<T, D><<<blocks, 256, 0, st>>>(p, (const T*)out, (const T*)dout, rowterm);
    return (int)cudaGetLastError();
}

template <typename T>
int rowterm_d(const ProblemDev& p, const void* out, const void* dout, float* rowterm, cudaStream_t st) {
    switch (p.D) {
        case 32: return rowterm_one<T, 32>(p, out, dout, rowterm, st);
        case 64: return rowterm_one<T, 64>(p, out, dout, rowterm, st);
        case 128: return rowterm_one<T, 128>(p, out, dout, rowterm, st);
    }
    return (int)cudaErrorInvalidValue;
}

int launch_rowterm(const ProblemDev& p, df_dtype dt, const void* out, const void* dout, float* rowterm,
                   cudaStream_t st) {
    if (dt == DF_BF16) return rowterm_d<__nv_bfloat16>(p, out, dout, rowterm, st);
    if (dt == DF_FP16) return rowterm_d<__half>(p, out, dout, rowterm, st);
    return rowterm_d<float>(p, out, dout, rowterm, st);
}

// One segment per blockIdx.y, four elements per thread and step.
template <bool TO_HALF>
__global__ void convert_kernel(ConvList cl) {
    const int sgi = blockIdx.y;
    const long long n4 = cl.n[sgi] / 4;
    for (long long x = (long long)blockIdx.x * blockDim.x + threadIdx.x; x < n4; x += (long long)gridDim.x * blockDim.x) {
        if (TO_HALF) {
            const float4 v = reinterpret_cast<const float4*>(cl.src[sgi])[x];
            const __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
            uint2 w;
            w.x = *reinterpret_cast<const uint32_t*>(&a);
            w.y = *reinterpret_cast<const uint32_t*>(&b);
            reinterpret_cast<uint2*>(cl.dst[sgi])[x] = w;
        } else {
            const uint2 w = reinterpret_cast<const uint2*>(cl.src[sgi])[x];
            const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&w.x));
            const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&w.y));
            reinterpret_cast<float4*>(cl.dst[sgi])[x] = make_float4(a.x, a.y, b.x, b.y);
        }
    }
}

int launch_convert(const ConvList& cl, bool to_half, cudaStream_t st) {
    if (cl.nseg < 1 || cl.nseg > kConvSegs) return (int)cudaErrorInvalidValue;
    long long most = 0;
    for (int i = 0; i < cl.nseg; ++i) {
        if (cl.n[i] % 4 || ((uintptr_t)cl.src[i] | (uintptr_t)cl.dst[i]) & 15u) return (int)cudaErrorInvalidValue;
        most = cl.n[i] > most ? cl.n[i] : most;
    }
    // enough blocks to fill the GPU a few times over across the segments
    long long bx = (most / 4 + 255) / 256;
    const long long cap = (4 * 152 + cl.nseg - 1) / cl.nseg;
    bx = bx < 1 ? 1 : (bx > cap ? cap : bx);
    const dim3 grid((unsigned)bx, (unsigned)cl.nseg);
    if (to_half)
        convert_kernel<true><<<grid, 256, 0, st>>>(cl);
    else
        convert_kernel<false><<<grid, 256, 0, st>>>(cl);
    return (int)cudaGetLastError();
}

}  // namespace df
