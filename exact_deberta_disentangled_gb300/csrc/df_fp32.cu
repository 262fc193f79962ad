// df_fp32.cu -- strict-fp32 disentangled attention on the CUDA cores.
//
// "DisentangledFlash" (section "Status") lists strict FP32 next to FP16 and
// BF16.  Tensor-core TF32 cannot keep an fp32 result within a 1e-5 relative
// error, so this dtype runs every product as fp32 FMA: one warp per query row
// (forward, dQ) or per key row (dK / dV), lanes over 32 keys (or queries) at
// a time for the score dot products, lanes over the head dimension for the
// output accumulation.  Nothing is ever stored per (query, key) pair.
//
// Backward split (no atomics anywhere, every sum in a fixed order):
//   dq kernel   -- row owner: dQ_i and G[i, r] = sum_{j: delta(i-j)=r} dZ_ij
//   dkv kernel  -- key owner: dK_j, dV_j and G'[j, r] = sum_{i: delta=r} dZ_ij
//   rel kernel  -- dKr[r] = sum_t G[t, r] Q_t,  dQr[r] = sum_t G'[t, r] K_t
#include "df_common.cuh"

namespace df {

namespace {

constexpr int kRowsPerBlock = 8;   // one warp per row
constexpr int kMaxD = 128;
constexpr int kMaxR = 1024;

DF_DEV float wmax(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}
DF_DEV float wsum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// z = a.b + a.kr_d + b.qr_d over D terms (a = query row, b = key row)
DF_DEV float score_raw(const float* a, const float* b, const float* krd, const float* qrd, int D) {
    float z1 = 0.f, z2 = 0.f, z3 = 0.f;
    for (int d = 0; d < D; ++d) {
        const float ad = a[d], bd = b[d];
        z1 = fmaf(ad, bd, z1);
        z2 = fmaf(ad, krd[d], z2);
        z3 = fmaf(bd, qrd[d], z3);
    }
    return z1 + z2 + z3;
}

DF_DEV bool keep_at(const ProblemDev& p, int b, int h, int i, int j) {
    if (!p.dropout) return true;
    return (keep_bits4(p, b, h, i, j >> 2) >> (j & 3)) & 1u;
}

__global__ void __launch_bounds__(256) fwd_f32_kernel(ProblemDev p, const int32_t* __restrict__ dtab,
                                                      const float* __restrict__ q, const float* __restrict__ k,
                                                      const float* __restrict__ v, const float* __restrict__ qr,
                                                      const float* __restrict__ kr, float* __restrict__ out,
                                                      float* __restrict__ lse) {
    __shared__ float qs[kRowsPerBlock][kMaxD];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.z, h = blockIdx.y, i = blockIdx.x * kRowsPerBlock + warp;
    int t0, n;
    seq_ok(p, b, t0, n);
    if (i >= n) return;
    const int D = p.D, R = p.R;
    const size_t ts = (size_t)p.H * D;
    const float* qi = q + (size_t)(t0 + i) * ts + (size_t)h * D;
    for (int d = lane; d < D; d += 32) qs[warp][d] = qi[d];
    __syncwarp();
    const bool qvalid = !p.qmask || p.qmask[t0 + i];
    const float* krh = kr + (size_t)h * R * D;
    const float* qrh = qr + (size_t)h * R * D;
    float m = -INFINITY, l = 0.f;
    float acc[kMaxD / 32] = {0.f, 0.f, 0.f, 0.f};
    for (int j0 = 0; j0 < n && qvalid; j0 += 32) {
        const int j = j0 + lane;
        float s = -INFINITY;
        if (j < n && (!p.kmask || p.kmask[t0 + j])) {
            const int dl = dtab[i - j + p.L - 1];
            s = p.scale * score_raw(qs[warp], k + (size_t)(t0 + j) * ts + (size_t)h * D, krh + (size_t)dl * D,
                                    qrh + (size_t)dl * D, D);
        }
        const float mn = fmaxf(m, wmax(s));
        if (mn == -INFINITY) continue;
        const float pj = s == -INFINITY ? 0.f : expf(s - mn);
        const float alpha = m == -INFINITY ? 0.f : expf(m - mn);
        l = l * alpha + wsum(pj);
        m = mn;
        const float pd = (j < n && keep_at(p, b, h, i, j)) ? pj * p.drop_scale : 0.f;
#pragma unroll
        for (int c = 0; c < kMaxD / 32; ++c) acc[c] *= alpha;
        const int jn = min(32, n - j0);
        for (int jj = 0; jj < jn; ++jj) {
            const float w = __shfl_sync(0xffffffffu, pd, jj);
            if (w == 0.f) continue;
            const float* vj = v + (size_t)(t0 + j0 + jj) * ts + (size_t)h * D;
#pragma unroll
            for (int c = 0; c < kMaxD / 32; ++c)
                if (lane + 32 * c < D) acc[c] = fmaf(w, vj[lane + 32 * c], acc[c]);
        }
    }
    float* oi = out + (size_t)(t0 + i) * ts + (size_t)h * D;
    const bool any = l > 0.f;
    const float inv = any ? 1.f / l : 0.f;
#pragma unroll
    for (int c = 0; c < kMaxD / 32; ++c)
        if (lane + 32 * c < D) oi[lane + 32 * c] = any ? acc[c] * inv : 0.f;
    if (lane == 0 && lse) lse[lse_index(p, b, h, t0, i)] = any ? m + logf(l) : INFINITY;   // lse == NULL: inference
}

__global__ void __launch_bounds__(256) dq_f32_kernel(ProblemDev p, const int32_t* __restrict__ dtab,
                                                     const float* __restrict__ q, const float* __restrict__ k,
                                                     const float* __restrict__ v, const float* __restrict__ qr,
                                                     const float* __restrict__ kr, const float* __restrict__ lse,
                                                     const float* __restrict__ rowterm,
                                                     const float* __restrict__ dout, float* __restrict__ dq,
                                                     float* __restrict__ G) {
    __shared__ float qs[kRowsPerBlock][kMaxD];
    __shared__ float ds[kRowsPerBlock][kMaxD];
    __shared__ float gs[kRowsPerBlock][kMaxR];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.z, h = blockIdx.y, i = blockIdx.x * kRowsPerBlock + warp;
    int t0, n;
    seq_ok(p, b, t0, n);
    if (i >= n) return;
    const int D = p.D, R = p.R;
    const size_t ts = (size_t)p.H * D;
    const size_t rowoff = (size_t)(t0 + i) * ts + (size_t)h * D;
    for (int d = lane; d < D; d += 32) {
        qs[warp][d] = q[rowoff + d];
        ds[warp][d] = dout[rowoff + d];
    }
    for (int r = lane; r < R; r += 32) gs[warp][r] = 0.f;
    __syncwarp();
    const float Li = lse[lse_index(p, b, h, t0, i)];
    const float Dl = rowterm[lse_index(p, b, h, t0, i)];
    const bool live = (!p.qmask || p.qmask[t0 + i]) && Li != INFINITY;
    const float* krh = kr + (size_t)h * R * D;
    const float* qrh = qr + (size_t)h * R * D;
    float acc[kMaxD / 32] = {0.f, 0.f, 0.f, 0.f};
    for (int j0 = 0; j0 < n && live; j0 += 32) {
        const int j = j0 + lane;
        float dz = 0.f;
        int dl = 0;
        if (j < n && (!p.kmask || p.kmask[t0 + j])) {
            dl = dtab[i - j + p.L - 1];
            const float* kj = k + (size_t)(t0 + j) * ts + (size_t)h * D;
            const float* vj = v + (size_t)(t0 + j) * ts + (size_t)h * D;
            const float s = p.scale * score_raw(qs[warp], kj, krh + (size_t)dl * D, qrh + (size_t)dl * D, D);
            const float pr = expf(s - Li);
            float dpd = 0.f;
            for (int d = 0; d < D; ++d) dpd = fmaf(ds[warp][d], vj[d], dpd);
            const float kp = keep_at(p, b, h, i, j) ? p.drop_scale : 0.f;
            dz = p.scale * pr * (dpd * kp - Dl);
        }
        const int jn = min(32, n - j0);
        for (int jj = 0; jj < jn; ++jj) {
            const float g = __shfl_sync(0xffffffffu, dz, jj);
            const int r = __shfl_sync(0xffffffffu, dl, jj);
            if (g == 0.f) continue;
            const float* kj = k + (size_t)(t0 + j0 + jj) * ts + (size_t)h * D;
            const float* krd = krh + (size_t)r * D;
#pragma unroll
            for (int c = 0; c < kMaxD / 32; ++c) {
                const int d = lane + 32 * c;
                if (d < D) acc[c] = fmaf(g, kj[d] + krd[d], acc[c]);
            }
            if (lane == 0) gs[warp][r] += g;
            __syncwarp();
        }
    }
#pragma unroll
    for (int c = 0; c < kMaxD / 32; ++c)
        if (lane + 32 * c < D) dq[rowoff + lane + 32 * c] = acc[c];
    __syncwarp();
    float* grow = G + ((size_t)(t0 + i) * p.H + h) * R;
    for (int r = lane; r < R; r += 32) grow[r] = gs[warp][r];
}

__global__ void __launch_bounds__(256) dkv_f32_kernel(ProblemDev p, const int32_t* __restrict__ dtab,
                                                      const float* __restrict__ q, const float* __restrict__ k,
                                                      const float* __restrict__ v, const float* __restrict__ qr,
                                                      const float* __restrict__ kr, const float* __restrict__ lse,
                                                      const float* __restrict__ rowterm,
                                                      const float* __restrict__ dout, float* __restrict__ dk,
                                                      float* __restrict__ dv, float* __restrict__ Gp) {
    __shared__ float ks[kRowsPerBlock][kMaxD];
    __shared__ float vs[kRowsPerBlock][kMaxD];
    __shared__ float gs[kRowsPerBlock][kMaxR];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.z, h = blockIdx.y, j = blockIdx.x * kRowsPerBlock + warp;
    int t0, n;
    seq_ok(p, b, t0, n);
    if (j >= n) return;
    const int D = p.D, R = p.R;
    const size_t ts = (size_t)p.H * D;
    const size_t rowoff = (size_t)(t0 + j) * ts + (size_t)h * D;
    for (int d = lane; d < D; d += 32) {
        ks[warp][d] = k[rowoff + d];
        vs[warp][d] = v[rowoff + d];
    }
    for (int r = lane; r < R; r += 32) gs[warp][r] = 0.f;
    __syncwarp();
    const bool kvalid = !p.kmask || p.kmask[t0 + j];
    const float* krh = kr + (size_t)h * R * D;
    const float* qrh = qr + (size_t)h * R * D;
    float adk[kMaxD / 32] = {0.f, 0.f, 0.f, 0.f};
    float adv[kMaxD / 32] = {0.f, 0.f, 0.f, 0.f};
    for (int i0 = 0; i0 < n && kvalid; i0 += 32) {
        const int i = i0 + lane;
        float dz = 0.f, pd = 0.f;
        int dl = 0;
        if (i < n && (!p.qmask || p.qmask[t0 + i])) {
            const float Li = lse[lse_index(p, b, h, t0, i)];
            if (Li != INFINITY) {
                dl = dtab[i - j + p.L - 1];
                const float* qi = q + (size_t)(t0 + i) * ts + (size_t)h * D;
                const float* doi = dout + (size_t)(t0 + i) * ts + (size_t)h * D;
                const float s = p.scale * score_raw(qi, ks[warp], krh + (size_t)dl * D, qrh + (size_t)dl * D, D);
                const float pr = expf(s - Li);
                float dpd = 0.f;
                for (int d = 0; d < D; ++d) dpd = fmaf(doi[d], vs[warp][d], dpd);
                const float kp = keep_at(p, b, h, i, j) ? p.drop_scale : 0.f;
                pd = pr * kp;
                dz = p.scale * pr * (dpd * kp - rowterm[lse_index(p, b, h, t0, i)]);
            }
        }
        const int in = min(32, n - i0);
        for (int ii = 0; ii < in; ++ii) {
            const float w = __shfl_sync(0xffffffffu, pd, ii);
            const float g = __shfl_sync(0xffffffffu, dz, ii);
            const int r = __shfl_sync(0xffffffffu, dl, ii);
            const size_t off = (size_t)(t0 + i0 + ii) * ts + (size_t)h * D;
            if (w != 0.f) {
#pragma unroll
                for (int c = 0; c < kMaxD / 32; ++c) {
                    const int d = lane + 32 * c;
                    if (d < D) adv[c] = fmaf(w, dout[off + d], adv[c]);
                }
            }
            if (g != 0.f) {
                const float* qrd = qrh + (size_t)r * D;
#pragma unroll
                for (int c = 0; c < kMaxD / 32; ++c) {
                    const int d = lane + 32 * c;
                    if (d < D) adk[c] = fmaf(g, q[off + d] + qrd[d], adk[c]);
                }
                if (lane == 0) gs[warp][r] += g;
                __syncwarp();
            }
        }
    }
#pragma unroll
    for (int c = 0; c < kMaxD / 32; ++c)
        if (lane + 32 * c < D) {
            dk[rowoff + lane + 32 * c] = adk[c];
            dv[rowoff + lane + 32 * c] = adv[c];
        }
    __syncwarp();
    float* grow = Gp + ((size_t)(t0 + j) * p.H + h) * R;
    for (int r = lane; r < R; r += 32) grow[r] = gs[warp][r];
}

// out[h, r, :] = sum over tokens t (ascending) of G[t, h, r] * X[t, h, :].
// Tokens outside every sequence (the padded tail of a packed buffer cannot
// occur; padded rows hold zero G) contribute nothing.
__global__ void rel_f32_kernel(ProblemDev p, const float* __restrict__ G, const float* __restrict__ X,
                               float* __restrict__ out) {
    const int r = blockIdx.x, h = blockIdx.y, d = threadIdx.x;
    if (d >= p.D) return;
    const size_t gs = (size_t)p.H * p.R, xs = (size_t)p.H * p.D;
    const float* g = G + (size_t)h * p.R + r;
    const float* x = X + (size_t)h * p.D + d;
    float acc = 0.f;
    for (int t = 0; t < p.T; ++t) acc = fmaf(g[(size_t)t * gs], x[(size_t)t * xs], acc);
    out[((size_t)h * p.R + r) * p.D + d] = acc;
}

}  // namespace

int launch_fwd_f32(const ProblemDev& p, const Workspace& ws, const float* q, const float* k, const float* v,
                   const float* qr, const float* kr, float* out, float* lse, cudaStream_t st) {
    dim3 grid((p.L + kRowsPerBlock - 1) / kRowsPerBlock, p.H, p.B);
    fwd_f32_kernel<<<grid, 256, 0, st>>>(p, ws.dtab, q, k, v, qr, kr, out, lse);
    return (int)cudaGetLastError();
}

int launch_bwd_f32(const ProblemDev& p, const Workspace& ws, const float* q, const float* k, const float* v,
                   const float* qr, const float* kr, const float* lse, const float* dout, float* dq, float* dk,
                   float* dv, float* dqr, float* dkr, cudaStream_t st) {
    dim3 grid((p.L + kRowsPerBlock - 1) / kRowsPerBlock, p.H, p.B);
    float* G = (float*)ws.G;
    float* Gp = (float*)ws.Gp;
    // rows of G / G' that no kernel writes (query-masked rows are written as
    // zeros; every token of a sequence is visited) -- nothing to clear.
    dq_f32_kernel<<<grid, 256, 0, st>>>(p, ws.dtab, q, k, v, qr, kr, lse, ws.rowterm, dout, dq, G);
    int e = (int)cudaGetLastError();
    if (e) return e;
    dkv_f32_kernel<<<grid, 256, 0, st>>>(p, ws.dtab, q, k, v, qr, kr, lse, ws.rowterm, dout, dk, dv, Gp);
    e = (int)cudaGetLastError();
    if (e) return e;
    dim3 rg(p.R, p.H);
    const int thr = ((p.D + 31) / 32) * 32;
    rel_f32_kernel<<<rg, thr, 0, st>>>(p, G, q, dkr);
    rel_f32_kernel<<<rg, thr, 0, st>>>(p, Gp, k, dqr);
    return (int)cudaGetLastError();
}

}  // namespace df
