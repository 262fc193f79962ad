// df_rel.cu -- the relative-position gradient products of the backward, from
// the diagonal sums G / G' written by the attention backward kernels
// ("DisentangledFlash", section "Performance": the relative-position
// gradients counted in the backward's 12 L R D term):
//
//   dQ  = dQattn + G  Kr        dK  = dKattn + G' Qr      (row products)
//   dKr = sum_tokens G^T Q      dQr = sum_tokens G'^T K  (column products)
//
// Row products: one CTA per (128-token tile, head), K = Rp relative rows in
// chunks of 64.  Column products: one CTA per (128 relative rows, head,
// token chunk) writes an fp32 partial; a second kernel sums the partials in
// chunk order, so dKr / dQr are bitwise reproducible.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "df_tile.cuh"

namespace df {
namespace {

constexpr int kRelThreads = 128;
constexpr int kChunkTok = 64;   // tokens per k-step group of the column products

template <int D>
struct RowSmem {
    using G = Geo<D>;
    static constexpr int AB = 128 * 64 * 2;          // G tile [128 tok x 64 r]
    static constexpr int BB = 64 * D * 2;            // Xr chunk [64 r x D]
    static constexpr int STAGE = AB + BB;
    static constexpr int BYTES = 2 * STAGE + 256;
    static constexpr int ALLOC = BYTES + 1024;
};

struct RelBars {
    uint64_t full[2], empty[2], done;
    uint32_t tmem_base;
    int abort_flag;
};

// out[tok, h, :] = bf16/fp16(acc32[tok, h, :] + sum_r G[tok, h, r] Xr[h, r, :])
template <int D, bool BF16>
__global__ void __launch_bounds__(kRelThreads, 1)
    rel_row_kernel(const __grid_constant__ CUtensorMap tmG, const __grid_constant__ CUtensorMap tmX,
                   const ProblemDev p, int Rp, const float* __restrict__ acc32, void* __restrict__ out_) {
    using G = Geo<D>;
    using S = RowSmem<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_align1024(smem_raw);
    RelBars* bars = reinterpret_cast<RelBars*>(smem + 2 * S::STAGE);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tok0 = blockIdx.x * 128, h = blockIdx.y;
    const int nk = Rp / 64 + (Rp % 64 ? 1 : 0);
    if (threadIdx.x == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->empty[s], 1);
        }
        mbar_init(&bars->done, 1);
        bars->abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0) {
        tc_alloc(&bars->tmem_base, 128);
        tc_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    const WaitCtx wc = wait_ctx(p, &bars->abort_flag);
    bool ok = true;
    int nload[2] = {0, 0};   // copies issued per stage
    if (threadIdx.x == 0) {
        constexpr uint32_t id = idesc_f16(128, D, BF16, false, true);
        auto issue_load = [&](int c) {
            const int s = c & 1;
            uint8_t* st = smem + s * S::STAGE;
            ++nload[s];
            mbar_arrive_expect_tx(&bars->full[s], S::STAGE);
            tma_load_2d(st, &tmG, h * Rp + 64 * c, tok0, &bars->full[s]);
            for (int q = 0; q < G::NCH; ++q)
                tma_load_2d(st + S::AB + q * 64 * G::CW * 2, &tmX, q * G::CW, h * p.R + 64 * c, &bars->full[s]);
        };
        issue_load(0);
        if (nk > 1) issue_load(1);
        for (int c = 0; c < nk && ok; ++c) {
            const int s = c & 1;
            if (!(ok = mbar_wait(&bars->full[s], (c >> 1) & 1, wc))) break;
            tc_fence_after();
            const uint32_t sA = smem_u32(smem + s * S::STAGE), sB = sA + S::AB;
            for (int k = 0; k < 4; ++k)
                tc_mma_ss(tmem, sdesc(sA + 32 * k, 16, 1024, 2), desc_mn<G>(sB, 64, k), id, (c | k) != 0);
            tc_commit(&bars->empty[s]);
            if (c + 2 < nk) {
                if (!(ok = mbar_wait(&bars->empty[s], (c >> 1) & 1, wc))) break;
                issue_load(c + 2);
            }
        }
        tc_commit(&bars->done);
        // no copy is still landing in shared memory when the CTA exits
        for (int s = 0; s < 2; ++s)
            if (nload[s] > 0) mbar_drain(&bars->full[s], (nload[s] - 1) & 1, wc.limit_ns);
    }
    const int row = 32 * warp + lane, tok = tok0 + row;
    // this row's attention part of the output, loaded while the products run
    float4 accv[D / 4];
    {
        const float4* a4 = reinterpret_cast<const float4*>(acc32 + ((size_t)(tok < p.T ? tok : 0) * p.H + h) * D);
#pragma unroll
        for (int v = 0; v < D / 4; ++v) accv[v] = a4[v];
    }
    __syncthreads();
    ok = __all_sync(0xffffffffu, ok);
    if (ok) ok = mbar_wait_warp(&bars->done, 0, wc);
    if (!ok) mbar_drain(&bars->done, 0, wc.limit_ns);   // the MMAs, before the tensor memory is freed
    tc_fence_after();
    using T16 = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
    if (ok) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
            uint32_t r[32];
            tc_ld32(tmem + ((uint32_t)(32 * warp) << 16) + 32 * c, r);
            tc_wait_ld();
            if (tok < p.T) {
                T16* o = reinterpret_cast<T16*>(out_) + ((size_t)tok * p.H + h) * D + 32 * c;
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const float4 x0 = accv[8 * c + 2 * v];
                    const float4 x1 = accv[8 * c + 2 * v + 1];
                    uint4 w;
                    w.x = pack2<BF16>(x0.x + __uint_as_float(r[8 * v + 0]), x0.y + __uint_as_float(r[8 * v + 1]));
                    w.y = pack2<BF16>(x0.z + __uint_as_float(r[8 * v + 2]), x0.w + __uint_as_float(r[8 * v + 3]));
                    w.z = pack2<BF16>(x1.x + __uint_as_float(r[8 * v + 4]), x1.y + __uint_as_float(r[8 * v + 5]));
                    w.w = pack2<BF16>(x1.z + __uint_as_float(r[8 * v + 6]), x1.w + __uint_as_float(r[8 * v + 7]));
                    reinterpret_cast<uint4*>(o)[v] = w;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tc_dealloc(tmem, 128);
    }
}

template <int D>
struct ColSmem {
    using G = Geo<D>;
    static constexpr int AB = kChunkTok * 128 * 2;   // G^T tile: [64 tok x 128 r] as two [64 x 64] regions
    static constexpr int BB = kChunkTok * D * 2;     // X tile [64 tok x D]
    static constexpr int STAGE = AB + BB;
    static constexpr int BYTES = 2 * STAGE + 256;
    static constexpr int ALLOC = BYTES + 1024;
};

// part[c, h, r, :] = sum over tokens of chunk c of G[tok, h, r] X[tok, h, :]
// for r in [128 * blockIdx.x, +128).
template <int D, bool BF16>
__global__ void __launch_bounds__(kRelThreads, 1)
    rel_col_kernel(const __grid_constant__ CUtensorMap tmG, const __grid_constant__ CUtensorMap tmX,
                   const ProblemDev p, int Rp, int chunk_tokens, float* __restrict__ part) {
    using G = Geo<D>;
    using S = ColSmem<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_align1024(smem_raw);
    RelBars* bars = reinterpret_cast<RelBars*>(smem + 2 * S::STAGE);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rb = blockIdx.x, h = blockIdx.y, ch = blockIdx.z;
    const int tbeg = ch * chunk_tokens;
    const int tend = min(p.T, tbeg + chunk_tokens);
    const int nk = tend > tbeg ? (tend - tbeg + kChunkTok - 1) / kChunkTok : 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->empty[s], 1);
        }
        mbar_init(&bars->done, 1);
        bars->abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0) {
        tc_alloc(&bars->tmem_base, 128);
        tc_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    const WaitCtx wc = wait_ctx(p, &bars->abort_flag);
    bool ok = true;
    int nload[2] = {0, 0};   // copies issued per stage
    if (threadIdx.x == 0 && nk > 0) {
        constexpr uint32_t id = idesc_f16(128, D, BF16, true, true);
        auto issue_load = [&](int c) {
            const int s = c & 1;
            uint8_t* st = smem + s * S::STAGE;
            const int t = tbeg + c * kChunkTok;
            ++nload[s];
            mbar_arrive_expect_tx(&bars->full[s], S::STAGE);
            tma_load_2d(st, &tmG, h * Rp + 128 * rb, t, &bars->full[s]);
            tma_load_2d(st + kChunkTok * 64 * 2, &tmG, h * Rp + 128 * rb + 64, t, &bars->full[s]);
            for (int q = 0; q < G::NCH; ++q)
                tma_load_2d(st + S::AB + q * kChunkTok * G::CW * 2, &tmX, h * D + q * G::CW, t, &bars->full[s]);
        };
        issue_load(0);
        if (nk > 1) issue_load(1);
        for (int c = 0; c < nk && ok; ++c) {
            const int s = c & 1;
            if (!(ok = mbar_wait(&bars->full[s], (c >> 1) & 1, wc))) break;
            tc_fence_after();
            const uint32_t sA = smem_u32(smem + s * S::STAGE), sB = sA + S::AB;
            for (int k = 0; k < kChunkTok / 16; ++k) {
                // A = G^T: M = r (two 64-wide swizzle atoms 8 KB apart), K = tokens
                const uint64_t ad = sdesc(sA + k * 16 * 128, kChunkTok * 128, 1024, 2);
                tc_mma_ss(tmem, ad, desc_mn<G>(sB, kChunkTok, k), id, (c | k) != 0);
            }
            tc_commit(&bars->empty[s]);
            if (c + 2 < nk) {
                if (!(ok = mbar_wait(&bars->empty[s], (c >> 1) & 1, wc))) break;
                issue_load(c + 2);
            }
        }
        tc_commit(&bars->done);
        // no copy is still landing in shared memory when the CTA exits
        for (int s = 0; s < 2; ++s)
            if (nload[s] > 0) mbar_drain(&bars->full[s], (nload[s] - 1) & 1, wc.limit_ns);
    }
    __syncthreads();
    ok = __all_sync(0xffffffffu, ok);
    if (nk > 0 && ok) ok = mbar_wait_warp(&bars->done, 0, wc);
    if (nk > 0 && !ok) mbar_drain(&bars->done, 0, wc.limit_ns);   // the MMAs, before the tensor memory is freed
    tc_fence_after();
    const int r = 128 * rb + 32 * warp + lane;
    float* dst = part + (((size_t)ch * p.H + h) * p.R + r) * D;
    if (ok) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
            uint32_t v[32];
            if (nk > 0) {
                tc_ld32(tmem + ((uint32_t)(32 * warp) << 16) + 32 * c, v);
                tc_wait_ld();
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = 0u;
            }
            if (r < p.R) {
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    reinterpret_cast<float4*>(dst + 32 * c)[e] =
                        make_float4(__uint_as_float(v[4 * e]), __uint_as_float(v[4 * e + 1]),
                                    __uint_as_float(v[4 * e + 2]), __uint_as_float(v[4 * e + 3]));
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tc_dealloc(tmem, 128);
    }
}

// out[h, r, d] = sum over chunks (ascending) of part[c, h, r, d]
template <bool BF16>
__global__ void rel_reduce_kernel(const float* __restrict__ part, int nchunk, size_t per_chunk, void* __restrict__ out) {
    using T16 = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
    for (size_t x = (size_t)blockIdx.x * blockDim.x + threadIdx.x; x < per_chunk; x += (size_t)gridDim.x * blockDim.x) {
        float acc = 0.f;
        for (int c = 0; c < nchunk; ++c) acc += part[(size_t)c * per_chunk + x];
        if (BF16)
            reinterpret_cast<__nv_bfloat16*>(out)[x] = __float2bfloat16(acc);
        else
            reinterpret_cast<__half*>(out)[x] = __float2half(acc);
    }
}

template <int D, bool BF16>
int rel_impl(const ProblemDev& p, const Workspace& ws, int Rp, int half, const void* x, const void* xr,
             void* out_tok, void* out_rel, cudaStream_t st, const BwdHook* hook) {
    using G = Geo<D>;
    const int code = BF16 ? 0 : 1;
    void* gbuf = half ? ws.Gp : ws.G;
    const float* acc = half ? ws.acc32b : ws.acc32a;
    float* part = half ? ws.part_qr : ws.part_kr;
    CUtensorMap mG, mXr, mX, mGc;
    const uint64_t g_dims[2] = {(uint64_t)p.H * Rp, (uint64_t)p.T};
    const uint64_t g_str[1] = {(uint64_t)p.H * Rp * 2};
    const uint64_t rel_dims[2] = {(uint64_t)D, (uint64_t)p.H * p.R};
    const uint64_t rel_str[1] = {(uint64_t)D * 2};
    const uint64_t tok_dims[2] = {(uint64_t)p.H * D, (uint64_t)p.T};
    const uint64_t tok_str[1] = {(uint64_t)p.H * D * 2};
    const uint32_t box_ga[2] = {64, 128};
    const uint32_t box_gc[2] = {64, (uint32_t)kChunkTok};
    const uint32_t box_x[2] = {(uint32_t)G::CW, 64};
    if (encode_tmap(&mG, code, 2, g_dims, g_str, box_ga, 128, gbuf) ||
        encode_tmap(&mXr, code, 2, rel_dims, rel_str, box_x, G::SWZB, xr) ||
        encode_tmap(&mX, code, 2, tok_dims, tok_str, box_x, G::SWZB, x) ||
        encode_tmap(&mGc, code, 2, g_dims, g_str, box_gc, 128, gbuf))
        return (int)cudaErrorInvalidValue;
    // the benchmark's relative-gradient phase is the half on the caller's stream
    if (half) prof_record(kProfRel, 0, st);
    {
        auto kern = rel_row_kernel<D, BF16>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, RowSmem<D>::ALLOC);
        if (e != cudaSuccess) return (int)e;
        dim3 grid((p.T + 127) / 128, p.H);
        kern<<<grid, kRelThreads, RowSmem<D>::ALLOC, st>>>(mG, mXr, p, Rp, acc, out_tok);
        if ((e = cudaGetLastError()) != cudaSuccess) return (int)e;
        if (hook) hook->fn(hook->ctx, 1 + half, st);   // dQ (dK) is final
    }
    {
        auto kern = rel_col_kernel<D, BF16>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, ColSmem<D>::ALLOC);
        if (e != cudaSuccess) return (int)e;
        const int chunk_tokens = ((p.T + ws.nchunk - 1) / ws.nchunk + kChunkTok - 1) / kChunkTok * kChunkTok;
        dim3 grid((p.R + 127) / 128, p.H, ws.nchunk);
        kern<<<grid, kRelThreads, ColSmem<D>::ALLOC, st>>>(mGc, mX, p, Rp, chunk_tokens, part);
        if ((e = cudaGetLastError()) != cudaSuccess) return (int)e;
    }
    const size_t per = (size_t)p.H * p.R * D;
    const int blocks = (int)((per + 255) / 256 < 1024 ? (per + 255) / 256 : 1024);
    rel_reduce_kernel<BF16><<<blocks, 256, 0, st>>>(part, ws.nchunk, per, out_rel);
    if (half) prof_record(kProfRel, 1, st);
    return (int)cudaGetLastError();
}

}  // namespace

int launch_rel_tc(const ProblemDev& p, const Workspace& ws, df_dtype dt, int Rp, int half, const void* x,
                  const void* xr, void* out_tok, void* out_rel, cudaStream_t st, const BwdHook* hook) {
    const bool bf = dt == DF_BF16;
#define DF_REL(D_) (bf ? rel_impl<D_, true>(p, ws, Rp, half, x, xr, out_tok, out_rel, st, hook) \
                       : rel_impl<D_, false>(p, ws, Rp, half, x, xr, out_tok, out_rel, st, hook))
    switch (p.D) {
        case 32: return DF_REL(32);
        case 64: return DF_REL(64);
        case 128: return DF_REL(128);
    }
#undef DF_REL
    return (int)cudaErrorInvalidValue;
}

}  // namespace df
