// df_bias.cu -- the relative-position bias of the band blocks, computed once
// per backward for the dQ and dK/dV kernels.
//
// "DisentangledFlash" (section "Status") adds the DeBERTa-v2/v3 C2P and P2C
// terms to every score.  Far from the diagonal they collapse to one value per
// query and one per key (the clamped relative index), which the attention
// kernels take from the per-token table of df_aux.cu.  In a band block (a
// 128 x 128 block of (query, key) pairs whose relative index is not constant
// at 0 or R-1) every pair has its own value
//     B[i][j] = c log2(e) (Q_i . Kr[delta(i - j)] + K_j . Qr[delta(i - j)]).
// This kernel writes B of every band block to the stored-bias table (layout
// in df_tile.cuh), so that the two backward kernels read each band tile's
// bias with one tensor copy instead of recomputing two band products each.
//
// One CTA per 128-query block of a (sequence, head) pair walks the band
// blocks of its row:
//   warp 0      TMA producer: the query block once, then per band block its
//               128 keys and the Kr / Qr band rows (head-dim chunks);
//   warp 1      tcgen05 issuer: Town = Q . Kr[band]^T into tensor-memory
//               columns [0, 256) and Tcross = K . Qr[band]^T into [256, 512);
//   warps 2..17 copy both products to shared-memory windows (scaled to base-2
//               units and rounded to fp16, as the forward does), gather
//               Town[i][delta - dlo] + Tcross[j][delta - dlo] per pair, round
//               the sum to fp16 and store the block.
// The products of block m + 1 run while block m is gathered.  Sixteen
// gather warps (four per tensor-memory lane quarter, a 32-column quarter of
// the block each) keep the shared-memory pipe busy: the gathers are two
// 16-bit loads per pair, and the relative index of a pair comes from the
// first index of its 32 columns and a step mask (the index moves by at most
// one per column) instead of a load of its own.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "df_tile.cuh"

namespace df {
namespace {

constexpr int kBiasThreads = 576;   // producer, issuer, sixteen gather warps
constexpr int kGatherThreads = kBiasThreads - 64;
constexpr float kLog2eB = 1.4426950408889634f;

template <int D>
struct BiasSmem {
    using G = Geo<D>;
    static constexpr int BB = kBiasBB;
    static constexpr int NBAND = 2 * BB;                 // a block reaches 2 BB - 1 relative rows
    static constexpr int OWN_S = 178;                    // window strides (halves): 32 rows x 128 columns
    static constexpr int CROSS_S = 176;                  // reach at most 159 relative rows, from a 16-aligned start
    static constexpr int QB = BB * D * 2;                // a [128 x D] token block
    static constexpr int KST = D == 128 ? 1 : 2;         // key-block stages (D = 128: shared memory)
    static constexpr int BST = 2;                        // band-row chunk stages
    static constexpr int Q = 0;
    static constexpr int K0 = Q + QB;                    // [KST] stages
    static constexpr int BAND = K0 + KST * QB;           // [BST] stages
    static constexpr int BANDB = NBAND * G::CW * 2;
    static constexpr int OWN = BAND + BST * BANDB;
    static constexpr int OWNB = BB * OWN_S * 2;
    static constexpr int CROSS = (OWN + OWNB + 15) / 16 * 16;
    static constexpr int CROSSB = BB * CROSS_S * 2;
    static constexpr int DWIN = (CROSS + CROSSB + 15) / 16 * 16;
    static constexpr int kMaxBlocks = 8192 / BB;          // L <= 8192
    static constexpr int STEPW = DWIN + 2 * BB * 2;       // step bits of the index window (9 words)
    static constexpr int KINDS = STEPW + 64;              // packed TileKind of every key block
    static constexpr int BLIST = KINDS + kMaxBlocks * 4;  // the band key blocks, in order
    static constexpr int MISC = BLIST + kMaxBlocks * 4;
    static constexpr int BYTES = MISC + 256;
    static constexpr int ALLOC = BYTES + 1024;
    static_assert(ALLOC <= 232448, "shared memory");
    static_assert(K0 % 1024 == 0 && BAND % 1024 == 0, "swizzled operands");
};

struct BiasBars {
    uint64_t q_full;
    uint64_t k_full[2], k_empty[2];
    uint64_t band_full[2], band_empty[2];
    uint64_t t_full, t_empty;
    uint64_t drain;   // the issuer's last MMAs, before the tensor memory is freed
    uint32_t tmem_base;
    int abort_flag;
    int cross_base[4];
    int nblocks;
};

template <int D, bool BF16>
__global__ void __launch_bounds__(kBiasThreads, 1)
    bias_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmKr, const __grid_constant__ CUtensorMap tmQr,
                   const ProblemDev p, const int32_t* __restrict__ dtab, uint16_t* __restrict__ bias) {
    using G = Geo<D>;
    using S = BiasSmem<D>;
    constexpr int BB = kBiasBB;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_align1024(smem_raw);
    BiasBars* bars = reinterpret_cast<BiasBars*>(smem + S::MISC);
    int16_t* dwin = reinterpret_cast<int16_t*>(smem + S::DWIN);
    uint16_t* own = reinterpret_cast<uint16_t*>(smem + S::OWN);
    uint16_t* cross = reinterpret_cast<uint16_t*>(smem + S::CROSS);
    uint32_t* kinds = reinterpret_cast<uint32_t*>(smem + S::KINDS);
    uint32_t* stepw = reinterpret_cast<uint32_t*>(smem + S::STEPW);
    int* blist = reinterpret_cast<int*>(smem + S::BLIST);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.x, b = blockIdx.y, qt = blockIdx.z;
    int t0, n;
    seq_ok(p, b, t0, n);
    const int i0 = qt * BB;
    if (i0 >= n) return;
    const int nkb = (n + BB - 1) / BB;

    // the kind of every key block (two relative-index loads each), then the
    // list of band blocks
    for (int t = threadIdx.x; t < nkb; t += kBiasThreads) kinds[t] = pack_kind(classify<BB, BB, 1>(p, dtab, i0 - t * BB));
    __syncthreads();
    if (threadIdx.x == 0) {
        mbar_init(&bars->q_full, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars->k_full[s], 1);
            mbar_init(&bars->k_empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars->band_full[s], 1);
            mbar_init(&bars->band_empty[s], 1);
        }
        mbar_init(&bars->t_full, 1);
        mbar_init(&bars->t_empty, kGatherThreads / 32);
        mbar_init(&bars->drain, 1);
        bars->abort_flag = 0;
        int nbl = 0;
        for (int kt = 0; kt < nkb; ++kt) {
            if (unpack_kind(kinds[kt]).uniform) continue;
            // a band block outside the kept slots cannot happen (the host keeps
            // one block of margin beyond the band's reach)
            if (bias_block_row(p, b, h, t0, qt, kt) < 0) {
                raise_error(p.err, DF_ERR_DEVICE_ARG);
                continue;
            }
            blist[nbl++] = kt;
        }
        bars->nblocks = nbl;
        fence_barrier_init();
    }
    if (warp == 1) {
        tc_alloc(&bars->tmem_base, 512);
        tc_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    const int nbl = bars->nblocks;
    const WaitCtx wc = wait_ctx(p, &bars->abort_flag);

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        int band_loads = 0, k_cnt[2] = {0, 0};   // band chunks issued; copies issued per key stage
        if (lane == 0 && nbl > 0) {
            mbar_arrive_expect_tx(&bars->q_full, S::QB);
            for (int c = 0; c < G::NCH; ++c)
                tma_load_2d(smem + S::Q + c * BB * G::CW * 2, &tmQ, h * D + c * G::CW, t0 + i0, &bars->q_full);
        }
        for (int m = 0; m < nbl; ++m) {
            const int s = m % S::KST, use = m / S::KST;
            const int kt = blist[m];
            const TileKind tk = unpack_kind(kinds[kt]);
            // K of block m once the cross product of block m - KST has read its stage
            if (use > 0 && !mbar_wait_warp(&bars->k_empty[s], (use - 1) & 1, wc)) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(&bars->k_full[s], S::QB);
                for (int c = 0; c < G::NCH; ++c)
                    tma_load_2d(smem + S::K0 + s * S::QB + c * BB * G::CW * 2, &tmK, h * D + c * G::CW,
                                t0 + kt * BB, &bars->k_full[s]);
            }
            ++k_cnt[s];
            // the Kr band rows (own product), then the Qr band rows (cross), a
            // head-dim chunk at a time through the band ring: chunk n goes to
            // stage n % BST once the product of chunk n - BST has read it
            bool ok = true;
            for (int pass = 0; pass < 2 && ok; ++pass) {
                for (int c = 0; c < G::NCH; ++c) {
                    const int bs = band_loads % S::BST, buse = band_loads / S::BST;
                    if (buse > 0 && !mbar_wait_warp(&bars->band_empty[bs], (buse - 1) & 1, wc)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) {
                        mbar_arrive_expect_tx(&bars->band_full[bs], S::BANDB);
                        tma_load_2d(smem + S::BAND + bs * S::BANDB, pass == 0 ? &tmKr : &tmQr, c * G::CW,
                                    h * p.R + tk.dlo, &bars->band_full[bs]);
                    }
                    ++band_loads;
                }
            }
            if (!ok) break;
        }
        // no copy of this CTA is still landing in shared memory when it exits
        // (each barrier's last phase is its last copy)
        if (lane == 0) {
            if (nbl > 0) mbar_drain(&bars->q_full, 0, wc.limit_ns);
            for (int s = 0; s < S::KST; ++s)
                if (k_cnt[s] > 0) mbar_drain(&bars->k_full[s], (k_cnt[s] - 1) & 1, wc.limit_ns);
            for (int s = 0; s < S::BST; ++s) {
                const int cnt = band_loads / S::BST + (s < band_loads % S::BST ? 1 : 0);
                if (cnt > 0) mbar_drain(&bars->band_full[s], (cnt - 1) & 1, wc.limit_ns);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        const uint32_t sQ = smem_u32(smem + S::Q), sBand = smem_u32(smem + S::BAND);
        constexpr uint32_t idT = idesc_f16(128, S::NBAND, BF16, false, false);
        const uint64_t dQ = desc_k<G>(sQ, BB, 0), dBand = desc_k<G>(sBand, S::NBAND, 0);
        const uint64_t dK0 = desc_k<G>(smem_u32(smem + S::K0), BB, 0), dK1 = dadd(dK0, S::QB);
        bool ok = nbl == 0 || mbar_wait_warp(&bars->q_full, 0, wc);
        int band_used = 0;
        for (int m = 0; m < nbl && ok; ++m) {
            const int s = m % S::KST, use = m / S::KST;
            // both products reuse the tensor memory: block m - 1's windows are copied out
            if (m > 0 && !(ok = mbar_wait_warp(&bars->t_empty, (m - 1) & 1, wc))) break;
            for (int pass = 0; pass < 2 && ok; ++pass) {
                if (pass == 1 && !(ok = mbar_wait_warp(&bars->k_full[s], use & 1, wc))) break;
                const uint64_t dA = pass == 0 ? dQ : (s ? dK1 : dK0);
                const uint32_t dcol = tmem + (pass == 0 ? 0u : (uint32_t)S::NBAND);
                for (int c = 0; c < G::NCH; ++c) {
                    const int bs = band_used % S::BST, buse = band_used / S::BST;
                    if (!(ok = mbar_wait_warp(&bars->band_full[bs], buse & 1, wc))) break;
                    tc_fence_after();
                    const uint64_t dB = dadd(dBand, (uint32_t)(bs * S::BANDB));
                    for (int k = 0; k < G::CW / 16; ++k)
                        tc_mma_ss_w(dcol, dadd(dA, kofs<G>(BB, c * (G::CW / 16) + k)),
                                    dadd(dB, kofs<G>(S::NBAND, k)), idT, (c | k) != 0);
                    tc_commit_w(&bars->band_empty[bs]);
                    ++band_used;
                }
            }
            if (!ok) break;
            tc_commit_w(&bars->t_full);
            tc_commit_w(&bars->k_empty[s]);
        }
        // every MMA issued above has completed before the tensor memory is freed
        tc_commit_w(&bars->drain);
        mbar_drain(&bars->drain, 0, wc.limit_ns);
    } else {
        // ------------------------------------------------------------ gather warps
        // Warp w owns TMEM lanes 32 (w & 3) .. +31 (query rows of Town, key
        // rows of Tcross) and column quarter cq of every block row; the four
        // warps of a lane quarter split the window copies.
        const int w4 = warp & 3;
        const int cq = (warp - 2) >> 2;     // 0..3
        const int row = 32 * w4 + lane;
        const int tid = threadIdx.x - 64;   // 0..511
        const uint32_t lane_base = tmem + ((uint32_t)(32 * w4) << 16);
        const float kscale = p.scale * kLog2eB;
        uint16_t* own_row = own + row * S::OWN_S;
        bool ok = true;
        BandRaw bn = {0, 0, 0};
        if (nbl > 0) bn = band_fetch<BB, BB, 1, true>(p, dtab, i0 - blist[0] * BB, w4, tid, lane);
        // every warp walks every block and meets every named barrier, also
        // after a bounded wait gave up (the work is then skipped)
        for (int m = 0; m < nbl; ++m) {
            const int kt = blist[m];
            const TileKind tk = unpack_kind(kinds[kt]);
            named_bar_sync(1, kGatherThreads);   // block m - 1's windows and index window are no longer read
            BandRaw bc = bn;          // this block's indices (fetched during the previous block)
            if (m + 1 < nbl) bn = band_fetch<BB, BB, 1, true>(p, dtab, i0 - blist[m + 1] * BB, w4, tid, lane);
            pin(bc.dw);
            pin(bc.dwp);
            pin(bc.rng);
            if (tid < 2 * BB - 1) dwin[tid] = (int16_t)(bc.dw - tk.dlo);
            if (tid < 2 * BB) put_step_bits(stepw, bc, tid, lane, 2 * BB - 1);   // the first eight warps
            const int lo = __shfl_sync(0xffffffffu, bc.rng, 0) - tk.dlo;
            const int hi = __shfl_sync(0xffffffffu, bc.rng, 1) - tk.dlo;
            const int clo = __shfl_sync(0xffffffffu, bc.rng, 2) - tk.dlo;
            const int chi = __shfl_sync(0xffffffffu, bc.rng, 3) - tk.dlo;
            const int own_a = lo & ~15;
            ok = ok && mbar_wait_warp(&bars->t_full, m & 1, wc);
            if (ok) {
                tc_fence_after();
                copy_band_window(lane_base, lo, hi, own_row, kscale, cq, 4);
                const int ca = copy_band_window(lane_base + (uint32_t)S::NBAND, clo, chi,
                                                cross + row * S::CROSS_S, kscale, cq, 4);
                if (lane == 0 && cq == 0) bars->cross_base[w4] = ca;
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->t_empty);
            }
            named_bar_sync(1, kGatherThreads);   // windows, index window, step bits and window bases complete
            if (!ok) continue;
            // B[row][j] for this quarter's 32 key columns j = 32 cq + e, stored
            // as four 16-byte chunks.  Column j's entry of the index window is
            // x0 - e; the index drops by one after each step bit.
            uint4* dst4 = reinterpret_cast<uint4*>(bias + ((size_t)bias_block_row(p, b, h, t0, qt, kt) + row) * BB);
            const uint16_t* orow = own_row - own_a;
            const uint16_t* crow = cross + 32 * cq * S::CROSS_S - bars->cross_base[cq];
            const int x0 = row - 32 * cq + BB - 1;
            int mi = dwin[x0];
            uint32_t mk = step_bits(stepw, x0 - 31);   // bit 31 - e: step at x0 - e
            uint32_t pk[16];
            float vprev = 0.f;
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                int mo = mi, mc = mi;
                DF_CLAMP_CHECK(mo, own_a, own_a + S::OWN_S, p.err);
                DF_CLAMP_CHECK(mc, bars->cross_base[cq], bars->cross_base[cq] + S::CROSS_S, p.err);
                const float v = h2f(orow[mo]) + h2f(crow[e * S::CROSS_S + mc]);
                mi -= (int)(mk >> 31);
                mk <<= 1;
                if (e & 1) pk[e >> 1] = pack2<false>(vprev, v); else vprev = v;
            }
#pragma unroll
            for (int q = 0; q < 4; ++q)
                dst4[bias_chunk(row, 4 * cq + q)] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tc_dealloc(tmem, 512);
    }
}

template <int D, bool BF16>
int launch_bias_impl(const ProblemDev& p, const Workspace& ws, const void* q, const void* k, const void* qr,
                     const void* kr, cudaStream_t st) {
    using G = Geo<D>;
    using S = BiasSmem<D>;
    CUtensorMap mq, mk, mkr, mqr;
    const uint64_t tok_dims[2] = {(uint64_t)p.H * D, (uint64_t)p.T};
    const uint64_t tok_str[1] = {(uint64_t)p.H * D * 2};
    const uint64_t rel_dims[2] = {(uint64_t)D, (uint64_t)p.H * p.R};
    const uint64_t rel_str[1] = {(uint64_t)D * 2};
    const uint32_t boxt[2] = {(uint32_t)G::CW, (uint32_t)S::BB};
    const uint32_t boxr[2] = {(uint32_t)G::CW, (uint32_t)S::NBAND};
    const int code = BF16 ? 0 : 1;
    if (encode_tmap(&mq, code, 2, tok_dims, tok_str, boxt, G::SWZB, q) ||
        encode_tmap(&mk, code, 2, tok_dims, tok_str, boxt, G::SWZB, k) ||
        encode_tmap(&mkr, code, 2, rel_dims, rel_str, boxr, G::SWZB, kr) ||
        encode_tmap(&mqr, code, 2, rel_dims, rel_str, boxr, G::SWZB, qr))
        return (int)cudaErrorInvalidValue;
    auto kern = bias_tc_kernel<D, BF16>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::ALLOC);
    if (e != cudaSuccess) return (int)e;
    dim3 grid(p.H, p.B, (p.L + S::BB - 1) / S::BB);
    kern<<<grid, kBiasThreads, S::ALLOC, st>>>(mq, mk, mkr, mqr, p, ws.dtab, ws.bias);
    return (int)cudaGetLastError();
}

}  // namespace

int launch_band_bias(const ProblemDev& p, const Workspace& ws, df_dtype dt, const void* q, const void* k,
                     const void* qr, const void* kr, cudaStream_t st) {
    if (!ws.bias) return (int)cudaErrorInvalidValue;
#define DF_ONE(D_, BF_) launch_bias_impl<D_, BF_>(p, ws, q, k, qr, kr, st)
#define DF_DT(D_) (dt == DF_BF16 ? DF_ONE(D_, true) : DF_ONE(D_, false))
    switch (p.D) {
        case 32: return DF_DT(32);
        case 64: return DF_DT(64);
        case 128: return DF_DT(128);
    }
#undef DF_DT
#undef DF_ONE
    return (int)cudaErrorInvalidValue;
}

}  // namespace df
