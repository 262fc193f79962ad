// df_bwd_kernel.cuh -- tensor-core backward of exact disentangled attention:
// the kernel template, instantiated by df_bwd_dq.cu and df_bwd_dkv.cu.
//
// "DisentangledFlash" (section "Hugging Face usage") splits the fused
// backward into a dQ kernel and a dK/dV kernel; section "Performance" counts
// the relative-position gradients.  Here both attention kernels are one
// template, mirrored by SIGMA:
//
//   SIGMA = +1 (dQ kernel):   rows = 128 queries, columns = key tiles
//        S = Q K^T, dPd = dO V^T, dZ = c P (dP - Dl),  dQ += dZ K
//        G[i, r]  = sum_{j: delta(i-j) = r} dZ[i, j]
//   SIGMA = -1 (dK/dV kernel): rows = 128 keys, columns = query tiles
//        S^T = K Q^T, dPd^T = V dO^T,  dV += Pd^T dO,  dK += dZ^T Q
//        G'[j, r] = sum_{i: delta(i-j) = r} dZ[i, j]
//
// P is recomputed from the forward's LSE (never stored) and the dropout mask
// is regenerated from the same Philox stream.  Every output row has exactly
// one owner CTA and every sum runs in a fixed order, so the result is
// bitwise reproducible with no floating-point atomics.
//
// The relative-position part of a score is a per-row and a per-column
// scalar in uniform tiles (the per-token table of df_aux.cu) and, in band
// tiles, a value per pair read from the stored band bias (df_bias.cu writes
// it before these kernels run): one tensor copy of the tile's bias box into a
// double-buffered stage.
//
// G / G' ([T, H, Rp] in the input dtype) feed the relative-position
// gradients (df_rel.cu):  dQ += G Kr,  dK += G' Qr,  dKr = sum G^T Q,
// dQr = sum G'^T K.  A band tile adds its diagonal sums with TMA reduce-adds,
// one [32 rows x QW sums] box per quarter of its rows; every element receives
// at most two non-zero additions that way (neighbouring tiles share at most
// one relative row), so the order of the additions cannot change the result.  The two
// clamped rows (delta 0 and R-1), which collect the far field, are summed in
// registers and added once at the end.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "df_tile.cuh"

namespace df {
namespace {

constexpr int kThreads = 352;   // producer, S / dP issuer, eight softmax warps, product issuer
constexpr float kLog2e = 1.4426950408889634f;

// Tensor-memory columns (512 per CTA).  The fp32 S and dP of the tile being
// processed sit in [256, 256 + 2 BN).  The 16-bit dZ and P~ that feed the
// dK / dQ / dV products have their own columns, so the S / dP issuer can
// compute the next tile's S / dP as soon as the softmax warps have read this
// tile's into registers.
template <int D>
struct BwdTmem {
    using G = Geo<D>;
    static constexpr uint32_t ACC1 = 0, ACC2 = D;                       // fp32 accumulators
    // dQ kernel (one accumulator): its rows' Q and dO, 16-bit, as the A
    // operands of S / dP and of the own band product, in ACC2's columns
    static constexpr uint32_t A1 = D, A2 = D + D / 2;
    static constexpr uint32_t S = 256, P = 256 + G::BN;                 // fp32 S, dP
    static constexpr uint32_t Z = 2 * D + G::BN <= 256 ? 2 * D : 256 + 2 * G::BN;   // 16-bit dZ, then P~
    static_assert(P + G::BN <= 512 && Z + G::BN <= 512, "tensor memory");
    static_assert(Z >= 2 * D && (Z + G::BN <= 256 || Z >= P + G::BN), "overlap");
};

template <int D>
struct BwdSmem {
    using G = Geo<D>;
    static constexpr int kMaxTiles = 8192 / G::BN;          // L <= 8192
    // diagonal-sum staging, one box per quarter of 32 tile rows: 32 rows of
    // QW 16-bit sums covering relative rows [qa0, qa0 + QW), qa0 the
    // quarter's lowest relative row rounded down to a multiple of 8.  The
    // quarter's rows reach at most BN + 31 relative rows (the relative row
    // moves by at most one per column), starting at most 7 in: slots up to
    // BN + 37.
    static constexpr int QW = (G::BN + 38 + 7) / 8 * 8;
    static constexpr int QSB = 32 * QW * 2;                  // bytes of one quarter's box
    static constexpr int R1 = 0;
    static constexpr int RB = G::BM * D * 2;
    static constexpr int R2 = R1 + RB;
    static constexpr int CB = G::BN * D * 2;
    // Column tiles go through a three-stage ring: a stage is released when
    // the tile's dK / dV (dQ) products complete, at the end of its softmax
    // pass, and the copy of the tile three ahead then has a tile and a half to
    // land before its S / dP are due.
    static constexpr int CST = 3;
    static constexpr int C1 = R2 + RB;                       // [CST] stages
    static constexpr int C2 = C1 + CST * CB;                 // [CST] stages
    // a band tile's stored bias: rows x columns halves, one stage (a band
    // tile's copy lands while the previous band tile sums its diagonals)
    static constexpr int BST = 1;
    static constexpr int BIAS = C2 + CST * CB;
    static constexpr int BIASB = G::BM * G::BN * 2;
    static constexpr int GST = BIAS + BST * BIASB;           // the four diagonal-sum boxes
    static constexpr int DWIN = (GST + 4 * QSB + 15) / 16 * 16;
    static constexpr int COLV = (DWIN + (G::BM + G::BN) * 2 + 15) / 16 * 16;  // [4 tiles][colb | cdl][BN]
    static constexpr int XCH = COLV + 8 * G::BN * 4;       // [4][BM] floats: exchanges between the two halves
    static constexpr int KINDS = XCH + 4 * G::BM * 4;        // packed TileKind of every column tile
    static constexpr int MISC = KINDS + kMaxTiles * 4;
    static constexpr int BYTES = MISC + 256;
    static constexpr int ALLOC = BYTES + 1024;
    static_assert(ALLOC <= 232448, "shared memory");
    static_assert(BIAS % 1024 == 0 && GST % 128 == 0 && QSB % 128 == 0 && QW <= 256, "staging boxes");
};

struct BwdBars {
    uint64_t row_full, a_full;
    uint64_t c_full[3], c_empty[3];        // column-tile ring
    uint64_t bias_full[1], bias_empty[1];  // stored-bias stage of band tiles
    uint64_t s_full, sread, z_full, zread, mma3_done;
    uint64_t drain;   // both issuers' last MMAs, before the tensor memory is freed
    uint32_t tmem_base;
    int abort_flag;
    uint32_t stepw[9];
};
static_assert(sizeof(BwdBars) <= 256, "barrier block (the MISC region)");

DF_DEV void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

DF_DEV void tma_reduce_add_2d(const CUtensorMap* m, const void* smem_src, int x, int y) {
    asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     (uint64_t)m),
                 "r"(smem_u32(smem_src)), "r"(x), "r"(y)
                 : "memory");
}
DF_DEV void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
DF_DEV void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
DF_DEV void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

template <bool BF16>
DF_DEV uint16_t f2h16(float v) {
    return (uint16_t)(pack2<BF16>(v, 0.f) & 0xFFFFu);
}
template <bool BF16>
DF_DEV float h16f(uint16_t v) {
    return BF16 ? __uint_as_float((uint32_t)v << 16) : h2f(v);
}

template <int D, bool BF16, int SIGMA, bool DROP>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_tc_kernel(const __grid_constant__ CUtensorMap tmR1, const __grid_constant__ CUtensorMap tmR2,
                  const __grid_constant__ CUtensorMap tmC1, const __grid_constant__ CUtensorMap tmC2,
                  const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmG, const ProblemDev p, const int32_t* __restrict__ dtab,
                  const float* __restrict__ relb, const float* __restrict__ lse, const float* __restrict__ rowterm,
                  float* __restrict__ acc1_out, void* __restrict__ acc2_out, void* __restrict__ Gbuf, int Rp,
                  const void* __restrict__ r1_rows, const void* __restrict__ r2_rows) {
    using G = Geo<D>;
    using S = BwdSmem<D>;
    using TM = BwdTmem<D>;
    using T16 = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
    constexpr int BM = G::BM, BN = G::BN;
    constexpr bool ROWQ = SIGMA > 0;   // rows are queries
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_align1024(smem_raw);
    BwdBars* bars = reinterpret_cast<BwdBars*>(smem + S::MISC);
    int16_t* dwin = reinterpret_cast<int16_t*>(smem + S::DWIN);
    float* colv = reinterpret_cast<float*>(smem + S::COLV);
    float* xch = reinterpret_cast<float*>(smem + S::XCH);
    uint16_t* gstage = reinterpret_cast<uint16_t*>(smem + S::GST);
    uint32_t* kinds = reinterpret_cast<uint32_t*>(smem + S::KINDS);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // grid (H, B, row blocks): every (sequence, head) pair's most expensive
    // row blocks are launched before any pair's cheapest ones
    const int h = blockIdx.x, b = blockIdx.y;
    int t0, n;
    seq_ok(p, b, t0, n);
    const int r0 = row_block_of(p, blockIdx.z, gridDim.z, BM) * BM;   // first row token (query or key) of this CTA
    if (r0 >= n) return;
    const int ntiles = (n + BN - 1) / BN;
    auto tile_base = [&](int m) { return ROWQ ? r0 - m * BN : m * BN - r0; };

    if (threadIdx.x == 0) {
        mbar_init(&bars->row_full, 1);
        mbar_init(&bars->a_full, 8);
        for (int s = 0; s < S::CST; ++s) {
            mbar_init(&bars->c_full[s], 1);
            mbar_init(&bars->c_empty[s], 1);
        }
        for (int s = 0; s < S::BST; ++s) {
            mbar_init(&bars->bias_full[s], 1);
            mbar_init(&bars->bias_empty[s], 8);
        }
        mbar_init(&bars->s_full, 1 + 32);   // S / dP's commit and the producer's 32 lanes (column terms)
        mbar_init(&bars->sread, 8);
        mbar_init(&bars->z_full, 8);
        mbar_init(&bars->zread, 8);
        mbar_init(&bars->mma3_done, 1);
        mbar_init(&bars->drain, 2);   // both issuers' last MMAs
        bars->abort_flag = 0;
        fence_barrier_init();
    }
    // the kind of every column tile (two relative-index loads each), once
    for (int t = threadIdx.x; t < ntiles; t += kThreads)
        kinds[t] = pack_kind(classify<BM, BN, SIGMA>(p, dtab, tile_base(t)));
    if (warp == 1) {
        tc_alloc(&bars->tmem_base, 512);
        tc_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_base;
    const WaitCtx wc = wait_ctx(p, &bars->abort_flag);

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // The warp walks the tiles: lane 0 issues the tensor copies, and the
        // warp writes each tile's per-column terms to shared memory
        // (double-buffered) for the softmax warps:
        //   cv0 = column bias (P2C of keys / C2P of queries in uniform tiles,
        //         0 in band tiles, -inf for masked or missing columns), minus the
        //         column's LSE (base 2) when the columns are queries;
        //   cv1 = c * Dl of the column (dK/dV kernel only).
        // Slot m & 3 is free when tile m's columns are loaded: tile m - 3's
        // column stage was released, so its products -- issued after the
        // softmax warps finished reading tile m - 3's terms, and those of tile
        // m - 4 before them -- have completed.  The terms are announced on tile
        // m's S / dP barrier.
        const size_t T = (size_t)p.T;
        const float* relb_h = relb + (size_t)h * 4 * T;
        const uint8_t* cmask = ROWQ ? p.kmask : p.qmask;
        auto put_columns = [&](int m) -> bool {
            const TileKind k = unpack_kind(kinds[m]);
            float* cv = colv + (m & 3) * 2 * BN;
            constexpr int NJ = BN / 32;
            // every load of the tile first (one memory round trip), then the terms
            float cb[NJ], ls[NJ], rt[NJ];
            int mk[NJ];
#pragma unroll
            for (int q = 0; q < NJ; ++q) {
                const int ct = m * BN + 32 * q + lane;
                const int cs = ct < n ? ct : 0;   // an index that is safe to load
                cb[q] = k.uniform ? ld_early(relb_h + ((ROWQ ? 2 : 0) + k.which) * T + t0 + cs) : 0.f;
                mk[q] = cmask ? ld_early(cmask + t0 + cs) : 1;
                ls[q] = ROWQ ? 0.f : ld_early(lse + lse_index(p, b, h, t0, cs));
                rt[q] = ROWQ ? 0.f : ld_early(rowterm + lse_index(p, b, h, t0, cs));
            }
#pragma unroll
            for (int q = 0; q < NJ; ++q) {
                const int j = 32 * q + lane;
                const bool valid = m * BN + j < n && mk[q] != 0;
                cv[j] = valid ? (ROWQ ? cb[q] : cb[q] - ls[q] * kLog2e) : -INFINITY;
                cv[BN + j] = valid && !ROWQ ? p.scale * rt[q] : 0.f;
            }
            // the terms are announced with S / dP of tile m (the barrier counts
            // the producer's lanes too), once the barrier has completed tile
            // m - 1's phase: an arrival never counts toward an older tile
            if (m >= 1 && !mbar_wait_warp(&bars->s_full, (m - 1) & 1, wc)) return false;
            mbar_arrive(&bars->s_full);
            return true;
        };
        if (lane == 0 && !ROWQ) {   // the dQ kernel's row operands go to tensor memory instead
            mbar_arrive_expect_tx(&bars->row_full, 2 * S::RB);
            for (int c = 0; c < G::NCH; ++c) {
                tma_load_2d(smem + S::R1 + c * BM * G::CW * 2, &tmR1, h * D + c * G::CW, t0 + r0, &bars->row_full);
                tma_load_2d(smem + S::R2 + c * BM * G::CW * 2, &tmR2, h * D + c * G::CW, t0 + r0, &bars->row_full);
            }
        }
        int c_cnt[S::CST] = {}, b_cnt[S::BST] = {};   // copies issued per barrier
        int bias_loads = 0;                          // band tiles so far
        // the stored-bias box of a column tile: the 128 x 128 block of the
        // (query block, key block) pair, and the tile's part of it
        const int rblk = r0 / kBiasBB;
        for (int it = 0; it < ntiles; ++it) {
            const int s = it % S::CST, use = it / S::CST;
            const int c0 = it * BN;
            if (use > 0 && !mbar_wait_warp(&bars->c_empty[s], (use - 1) & 1, wc)) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(&bars->c_full[s], 2 * S::CB);
                for (int c = 0; c < G::NCH; ++c) {
                    tma_load_2d(smem + S::C1 + s * S::CB + c * BN * G::CW * 2, &tmC1, h * D + c * G::CW, t0 + c0,
                                &bars->c_full[s]);
                    tma_load_2d(smem + S::C2 + s * S::CB + c * BN * G::CW * 2, &tmC2, h * D + c * G::CW, t0 + c0,
                                &bars->c_full[s]);
                }
            }
            ++c_cnt[s];
            if (!put_columns(it)) break;
            const TileKind tk = unpack_kind(kinds[it]);
            if (tk.uniform) continue;
            // a band tile: its bias box into stage bias_loads % BST, once the
            // softmax warps are done with the band tile that used the stage before
            const int bs = bias_loads % S::BST, buse = bias_loads / S::BST;
            if (buse > 0 && !mbar_wait_warp(&bars->bias_empty[bs], (buse - 1) & 1, wc)) break;
            if (lane == 0) {
                const int cblk = c0 / kBiasBB, cin = c0 % kBiasBB;
                int brow = ROWQ ? bias_block_row(p, b, h, t0, rblk, cblk) : bias_block_row(p, b, h, t0, cblk, rblk);
                if (brow < 0) {   // cannot happen: the table keeps every band block
                    raise_error(p.err, DF_ERR_DEVICE_ARG);
                    brow = 0;
                }
                mbar_arrive_expect_tx(&bars->bias_full[bs], S::BIASB);
                // query rows x key columns: the dQ kernel's rows are the box rows,
                // the dK/dV kernel's columns are
                tma_load_2d(smem + S::BIAS + bs * S::BIASB, &tmB, ROWQ ? cin : 0, brow + (ROWQ ? 0 : cin),
                            &bars->bias_full[bs]);
            }
            ++b_cnt[bs];
            ++bias_loads;
        }
        // no copy of this CTA is still landing in shared memory when it exits
        // (each barrier's last phase is its last copy; the ones before it
        // completed before that copy was issued)
        if (lane == 0) {
            if (!ROWQ) mbar_drain(&bars->row_full, 0, wc.limit_ns);
            for (int s = 0; s < S::CST; ++s)
                if (c_cnt[s] > 0) mbar_drain(&bars->c_full[s], (c_cnt[s] - 1) & 1, wc.limit_ns);
            for (int s = 0; s < S::BST; ++s)
                if (b_cnt[s] > 0) mbar_drain(&bars->bias_full[s], (b_cnt[s] - 1) & 1, wc.limit_ns);
        }
    } else if (warp == 1 || warp == 10) {
        // ------------------------------------------------------------ MMA issuers
        // Warp 1 issues S / dP of tile m + 1 once the softmax warps have read
        // tile m's into registers; warp 10 the dK / dV (dQ) products of tile m
        // once its 16-bit dZ / P~ are written (sread comes before z_full in
        // every softmax warp, so S / dP of tile m + 1 normally go first; the
        // two touch different tensor memory and stages either way).  Band
        // tiles take the same order: their relative-position part comes from
        // the stored bias.  Each warp walks its issue loop (control flow
        // warp-uniform); the MMAs and commits are the elect.sync forms, issued
        // by one lane.  Operand descriptors are built once (per CTA or per ring
        // stage) and advanced per k-step by a constant.  The product issuer
        // reads a column stage only after z_full of its tile, which the softmax
        // warps arrive on after S / dP of that tile -- issued once the stage
        // had landed -- completed.
        {
            const uint32_t sR1 = smem_u32(smem + S::R1), sR2 = smem_u32(smem + S::R2);
            constexpr uint32_t idS = idesc_f16(128, BN, BF16, false, false);
            constexpr uint32_t idA = idesc_f16(128, D, BF16, false, true);
            const uint64_t dR1 = desc_k<G>(sR1, BM, 0), dR2 = desc_k<G>(sR2, BM, 0);
            // column operands, K-major and MN-major, of ring stages 0 and 1
            const uint32_t sC10 = smem_u32(smem + S::C1), sC20 = smem_u32(smem + S::C2);
            const uint64_t dC1k0 = desc_k<G>(sC10, BN, 0), dC2k0 = desc_k<G>(sC20, BN, 0);
            const uint64_t dC1m0 = desc_mn<G>(sC10, BN, 0), dC2m0 = desc_mn<G>(sC20, BN, 0);
            auto stage_ofs = [](int s) { return (uint32_t)(s * S::CB); };
            bool ok = true;
            if (warp == 1) {   // the A operands of S / dP: tensor memory (dQ) or shared memory rows
                ok = mbar_wait_warp(ROWQ ? &bars->a_full : &bars->row_full, 0, wc);
                if (ROWQ) tc_fence_after();
            }
            // tile m's column operands in shared memory
            auto wait_cols = [&](int m) -> bool {
                if (!mbar_wait_warp(&bars->c_full[m % S::CST], (m / S::CST) & 1, wc)) return false;
                tc_fence_after();
                return true;
            };
            // S / dP of tile m (its column operands waited for)
            auto issue_s = [&](int m) -> bool {
                const int s = m % S::CST;
                const uint64_t dS = dadd(dC1k0, stage_ofs(s)), dP = dadd(dC2k0, stage_ofs(s));
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    if (ROWQ) {
                        tc_mma_ts_w(tmem + TM::S, tmem + TM::A1 + 8 * k, dadd(dS, kofs<G>(BN, k)), idS, k != 0);
                        tc_mma_ts_w(tmem + TM::P, tmem + TM::A2 + 8 * k, dadd(dP, kofs<G>(BN, k)), idS, k != 0);
                    } else {
                        tc_mma_ss_w(tmem + TM::S, dadd(dR1, kofs<G>(BM, k)), dadd(dS, kofs<G>(BN, k)), idS, k != 0);
                        tc_mma_ss_w(tmem + TM::P, dadd(dR2, kofs<G>(BM, k)), dadd(dP, kofs<G>(BN, k)), idS, k != 0);
                    }
                }
                tc_commit_w(&bars->s_full);
                return true;
            };
            auto issue_acc = [&](int m) -> bool {
                const int s = m % S::CST;
                if (!mbar_wait_warp(&bars->z_full, m & 1, wc)) return false;
                tc_fence_after();
                const uint64_t d1 = dadd(dC1m0, stage_ofs(s)), d2 = dadd(dC2m0, stage_ofs(s));
#pragma unroll
                for (int k = 0; k < BN / 16; ++k) {
                    // acc1 += dZ . C1   (dQ += dZ K  |  dK += dZ^T Q)
                    tc_mma_ts_w(tmem + TM::ACC1, tmem + TM::Z + k * 8, dadd(d1, mnofs<G>(k)), idA, (m | k) != 0);
                    // dV += Pd^T dO
                    if (!ROWQ)
                        tc_mma_ts_w(tmem + TM::ACC2, tmem + TM::Z + BN / 2 + k * 8, dadd(d2, mnofs<G>(k)), idA,
                                    (m | k) != 0);
                }
                tc_commit_w(&bars->c_empty[s]);
                tc_commit_w(&bars->mma3_done);
                return true;
            };
            if (warp == 1) {
                // test-only stall injection: S / dP stop before this tile, so
                // that the other roles' bounded waits run out
                const int stall = p.fault_kernel == (ROWQ ? 1 : 2) ? p.fault_tile : -1;
                if (ok && stall != 0) ok = wait_cols(0) && issue_s(0);
                for (int it = 0; it + 1 < ntiles && ok; ++it) {
                    if (stall >= 0 && it + 1 >= stall) break;
                    // tile it + 1's columns, normally in place long before:
                    // their wait is off the chain from the softmax warps'
                    // read of tile it to the next S / dP
                    if (!(ok = wait_cols(it + 1))) break;
                    if (!(ok = mbar_wait_warp(&bars->sread, it & 1, wc))) break;
                    if (!(ok = issue_s(it + 1))) break;
                }
            } else {
                for (int it = 0; it < ntiles && ok; ++it) ok = issue_acc(it);
            }
            // every MMA this warp issued has completed (and, through the
            // barrier's count of 2, the other issuer's) before the tensor
            // memory is freed
            tc_commit_w(&bars->drain);
            mbar_drain(&bars->drain, 0, wc.limit_ns);
        }
    } else {   // warps 2 .. 9
        // ------------------------------------------------------------ softmax / gradient warps
        // Eight warps: warp w owns TMEM lanes 32 (w & 3) .. +31 (rows) and
        // column half hf = (w - 2) / 4 of every tile.  Band-window copies and
        // the diagonal sums of band tiles are split between the two halves;
        // every warp takes the same bounded waits.
        const int w4 = warp & 3;
        const int hf = (warp - 2) >> 2;
        const int row = 32 * w4 + lane;
        const int tid = threadIdx.x - 64;     // 0..255
        const int pair_bar = 2 + w4;
        const uint32_t lane_base = tmem + ((uint32_t)(32 * w4) << 16);
        constexpr int NCT = BN / 64;          // 32-column chunks per thread
        constexpr int HC = BN / 2;            // columns per half
        const int cbeg = hf * NCT;
        const int rt = r0 + row;              // row token position in the sequence
        const bool row_in = rt < n;
        const size_t T = (size_t)p.T;
        const float* relb_h = relb + (size_t)h * 4 * T;
        const float kscale = p.scale * kLog2e;
        // per-row constants
        float rb0 = -INFINITY, rb1 = -INFINITY, lse2 = INFINITY, dl = 0.f;
        if (row_in) {
            const bool rvalid = ROWQ ? (!p.qmask || p.qmask[t0 + rt]) : (!p.kmask || p.kmask[t0 + rt]);
            if (rvalid) {
                rb0 = relb_h[(ROWQ ? 0 : 2) * T + t0 + rt];
                rb1 = relb_h[(ROWQ ? 1 : 3) * T + t0 + rt];
            }
            if (ROWQ) {
                lse2 = lse[lse_index(p, b, h, t0, rt)] * kLog2e;
                dl = rowterm[lse_index(p, b, h, t0, rt)];
            }
        }
        const bool rvalid = rb0 != -INFINITY;
        const float dls_row = p.scale * dl;
        if constexpr (ROWQ) {
            // the A operands of S / dP: this row's Q (first column half) or dO
            // (second), 16-bit, two elements per column (zero past the sequence)
            constexpr int NW = D / 2;
            uint32_t a[NW];
            const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(hf ? r2_rows : r1_rows) +
                                                              ((size_t)(t0 + (row_in ? rt : 0)) * p.H + h) * D);
#pragma unroll
            for (int v = 0; v < NW / 4; ++v) {
                const uint4 w = row_in ? src[v] : make_uint4(0u, 0u, 0u, 0u);
                a[4 * v] = w.x;
                a[4 * v + 1] = w.y;
                a[4 * v + 2] = w.z;
                a[4 * v + 3] = w.w;
            }
            const uint32_t acol = lane_base + (hf ? TM::A2 : TM::A1);
#pragma unroll
            for (int q = 0; q < NW / 16; ++q) {
                uint32_t r16[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) r16[e] = a[16 * q + e];
                tc_st16(acol + 16 * q, r16);
            }
            tc_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->a_full);
        }
        float g_lo = 0.f, g_hi = 0.f;     // this thread's share of the diagonal sums at delta 0 and R-1
        int bias_uses = 0;                // band tiles so far (stored-bias stage bias_uses % BST)
        bool ok = true;
        auto kind_of = [&](int t) { return unpack_kind(kinds[t < ntiles ? t : ntiles - 1]); };
        BandRaw bn = band_fetch<BM, BN, SIGMA, true>(p, dtab, tile_base(0), w4, tid, lane);   // band indices, one tile ahead
        // Every warp walks every tile and meets every named barrier, also after
        // a bounded wait gave up (ok == false: the work is skipped, no wait is
        // taken): a warp that left the loop early would leave its siblings
        // parked in bar.sync for good.
        for (int it = 0; it < ntiles; ++it) {
            const int c0 = it * BN;
            const int base = tile_base(it);
            const TileKind tk = kind_of(it);
            const float* colb = colv + (it & 3) * 2 * BN;
            const float* cdl = colb + BN;
            // every tile starts with all eight warps: band tiles rewrite the index
            // window, and the per-warp arrivals on the tile's barriers (counts
            // of 8, or 4 per column half) must never meet a warp that is a whole
            // tile ahead -- its arrival would complete the previous tile's phase
            named_bar_sync(1, 256);
            BandRaw bc = bn;   // this tile's band indices (fetched during the previous tile)
            if (it + 1 < ntiles && !kind_of(it + 1).uniform)
                bn = band_fetch<BM, BN, SIGMA, true>(p, dtab, tile_base(it + 1), w4, tid, lane);
            if (!tk.uniform) {
                // the index window and its step bits, read by the diagonal sums
                // after the tile's middle barrier
                pin(bc.dw);
                pin(bc.dwp);
                if (tid < BM + BN - 1) dwin[tid] = (int16_t)(bc.dw - tk.dlo);
                put_step_bits(bars->stepw, bc, tid, lane, BM + BN - 1);
            }
            // S / dP of this tile and its column terms (the producer arrives on the same barrier)
            ok = ok && mbar_wait_warp(&bars->s_full, it & 1, wc);
            const bool band = !tk.uniform;
            const int bstage = bias_uses % S::BST;
            // and, for a band tile, its stored bias
            if (band) ok = ok && mbar_wait_warp(&bars->bias_full[bstage], (bias_uses / S::BST) & 1, wc);
            tc_fence_after();
            const float rb = tk.uniform ? (tk.which ? rb1 : rb0) : (rvalid ? 0.f : -INFINITY);
            const uint16_t* bbox = reinterpret_cast<const uint16_t*>(smem + S::BIAS + bstage * S::BIASB);
            // per-row constant of the exponent (base 2): row bias, minus the row LSE for query rows
            const float rowc = ROWQ ? rb - lse2 : rb;
            float rs[4] = {0.f, 0.f, 0.f, 0.f};
            // this thread's 32-column chunks: S, dP -> P, dZ (and Pd for the dK/dV kernel)
#pragma unroll 1
            for (int cc = 0; cc < NCT && ok; ++cc) {
                const int c = cbeg + cc;
                uint32_t sr[32], pr[32];
                tc_ld32(lane_base + TM::S + 32 * c, sr);
                tc_ld32(lane_base + TM::P + 32 * c, pr);
                tc_wait_ld();
                if (cc == NCT - 1) {
                    // all of this warp's S / dP columns are in registers
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars->sread);
                }
                const float4* cv0p = reinterpret_cast<const float4*>(colb + 32 * c);
                if (band) {
                    // the stored bias of these 32 columns (base-2 units, fp16)
                    if constexpr (ROWQ) {
                        // box row `row`: this tile's columns of the block row, as
                        // 16-byte chunks starting at block chunk xo
                        const int xo = (c0 % kBiasBB) / 8;
                        const uint4* brow4 = reinterpret_cast<const uint4*>(bbox + row * BN);
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            int ci = bias_chunk(row, xo + 4 * c + q) - xo;   // 16-byte chunk of the box row
                            DF_CLAMP_CHECK(ci, 0, BN / 8, p.err);
                            const uint4 w = brow4[ci];
                            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
                            const float4 ca = cv0p[2 * q], cb = cv0p[2 * q + 1];
                            const float cvs[8] = {ca.x, ca.y, ca.z, ca.w, cb.x, cb.y, cb.z, cb.w};
#pragma unroll
                            for (int t = 0; t < 8; ++t) {
                                const int e = 8 * q + t;
                                const uint16_t hv = (uint16_t)(ww[t >> 1] >> (16 * (t & 1)));
                                sr[e] = __float_as_uint(fmaf(__uint_as_float(sr[e]), kscale, cvs[t]) + rowc + h2f(hv));
                            }
                        }
                    } else {
                        // box column `row` (this thread's key), one half per query row
                        const uint16_t* bcol = bbox + ((row >> 3) & 8) * 8 + (row & 7);
                        const int r3 = (row >> 3) & 7;
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const float4 cv = cv0p[q];
                            const float cvs[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
                            for (int t = 0; t < 4; ++t) {
                                const int e = 4 * q + t;
                                const float bv = h2f(bcol[(32 * c + e) * kBiasBB + ((r3 ^ e) & 7) * 8]);
                                sr[e] = __float_as_uint(fmaf(__uint_as_float(sr[e]), kscale, cvs[t]) + rowc + bv);
                            }
                        }
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const float4 cv = cv0p[q];
                        float a0, a1, a2, a3;
                        ffma2(a0, a1, __uint_as_float(sr[4 * q + 0]), __uint_as_float(sr[4 * q + 1]), kscale, kscale,
                              cv.x, cv.y);
                        ffma2(a2, a3, __uint_as_float(sr[4 * q + 2]), __uint_as_float(sr[4 * q + 3]), kscale, kscale,
                              cv.z, cv.w);
                        fadd2(a0, a1, a0, a1, rowc, rowc);
                        fadd2(a2, a3, a2, a3, rowc, rowc);
                        sr[4 * q + 0] = __float_as_uint(a0);
                        sr[4 * q + 1] = __float_as_uint(a1);
                        sr[4 * q + 2] = __float_as_uint(a2);
                        sr[4 * q + 3] = __float_as_uint(a3);
                    }
                }
                uint32_t keep = 0xFFFFFFFFu;
                if constexpr (DROP)
                    keep = ROWQ ? keep_bits32_row(p, b, h, rt, c0 + 32 * c) : keep_bits32_col(p, b, h, c0 + 32 * c, rt);
                const float4* cv1p = reinterpret_cast<const float4*>(cdl + 32 * c);
                uint32_t zp[16], pp[16];   // packed as they are formed, so S / dP registers die early
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    float dlq[4] = {dls_row, dls_row, dls_row, dls_row};
                    if (!ROWQ) {
                        const float4 d4 = cv1p[q];
                        dlq[0] = d4.x;
                        dlq[1] = d4.y;
                        dlq[2] = d4.z;
                        dlq[3] = d4.w;
                    }
                    float z[4], pd[4];
                    if constexpr (DROP) {
#pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            const int e = 4 * q + t;
                            const float pr_ = ex2(__uint_as_float(sr[e]));
                            const float kp = ((keep >> e) & 1u) ? p.drop_scale : 0.f;
                            z[t] = pr_ * fmaf(__uint_as_float(pr[e]), p.scale * kp, -dlq[t]);
                            pd[t] = pr_ * kp;
                            rs[t] += z[t];
                        }
                    } else {
                        // the same arithmetic as above with keep = 1, two lanes per instruction
#pragma unroll
                        for (int t = 0; t < 4; ++t) pd[t] = ex2(__uint_as_float(sr[4 * q + t]));
                        float u0, u1, u2, u3;
                        ffma2(u0, u1, __uint_as_float(pr[4 * q + 0]), __uint_as_float(pr[4 * q + 1]), p.scale,
                              p.scale, -dlq[0], -dlq[1]);
                        ffma2(u2, u3, __uint_as_float(pr[4 * q + 2]), __uint_as_float(pr[4 * q + 3]), p.scale,
                              p.scale, -dlq[2], -dlq[3]);
                        fmul2(z[0], z[1], pd[0], pd[1], u0, u1);
                        fmul2(z[2], z[3], pd[2], pd[3], u2, u3);
                        fadd2(rs[0], rs[1], rs[0], rs[1], z[0], z[1]);
                        fadd2(rs[2], rs[3], rs[2], rs[3], z[2], z[3]);
                    }
                    zp[2 * q] = pack2<BF16>(z[0], z[1]);
                    zp[2 * q + 1] = pack2<BF16>(z[2], z[3]);
                    pp[2 * q] = pack2<BF16>(pd[0], pd[1]);
                    pp[2 * q + 1] = pack2<BF16>(pd[2], pd[3]);
                }
                if (cc == 0 && it > 0) {
                    // the previous tile's products must have read their 16-bit operands
                    if (!(ok = mbar_wait_warp(&bars->mma3_done, (it - 1) & 1, wc))) break;
                    tc_fence_after();
                }
                tc_st16(lane_base + TM::Z + 16 * c, zp);
                if (!ROWQ) tc_st16(lane_base + TM::Z + BN / 2 + 16 * c, pp);
            }
            if (band) {
                // the stored bias of this tile is no longer read
                if (ok) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars->bias_empty[bstage]);
                }
                ++bias_uses;
            }
            const float rowsum = (rs[0] + rs[1]) + (rs[2] + rs[3]);
            if (ok) {
                tc_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->z_full);
            }
            // ---- diagonal sums of dZ for this tile
            if (!band) {
                if (ok) {
                    if (tk.which) g_hi += rowsum; else g_lo += rowsum;
                    if (lane == 0) mbar_arrive(&bars->zread);
                }
            } else {
                // (after a give-up only the named barriers below are met)
                named_bar_sync(1, 256);   // every dZ is in tensor memory; the index window is complete
                tc_fence_after();
                // this quarter's relative rows: the index into dwin grows (or
                // falls) monotonically from one corner of the quarter to the other
                const int xa = ROWQ ? 32 * w4 : BM - 32 - 32 * w4;
                const int xb = xa + BN + 30;
                const int qa = dwin[xa], qb = dwin[xb];
                const int qmin = qa < qb ? qa : qb, qmax = qa < qb ? qb : qa;
                const int qa0 = (tk.dlo + qmin) & ~7;   // first relative row of the box (absolute)
                const int qoff = tk.dlo - qa0;          // slot of relative row dlo + m is m + qoff
                uint16_t* qstage = gstage + (size_t)w4 * 32 * S::QW;
                uint16_t* grow = qstage + lane * S::QW + qoff;
                const int mmax = S::QW - 1 - qoff;   // a clamp: grow[m] stays inside the row
                // every relative row of the quarter has its slot in the box
                // (qmin + qoff >= 0 by the choice of qa0); a tile breaking the
                // other end is flagged and its runs are not stored
                const bool bad = qmax + qoff > S::QW - 1;   // cannot happen for a valid tile
                // this box still holds the previous band tile's sums until their
                // reduce-add has read it: its issuer waits here, a whole chunk
                // loop after issuing it, and the pair barrier passes that on
                if (hf == 0 && lane == 0) bulk_wait_read0();
                named_bar_sync(pair_bar, 64);
                if (ok) {
                    // the quarter's two warps clear its box, lanes on consecutive
                    // 16-byte chunks (the box is one dense block)
                    constexpr int NCK = S::QSB / 16;
                    uint4* qz = reinterpret_cast<uint4*>(qstage);
#pragma unroll
                    for (int i = hf * 32 + lane; i < NCK; i += 64) qz[i] = make_uint4(0u, 0u, 0u, 0u);
                }
                named_bar_sync(pair_bar, 64);   // the box is cleared
                // Runs of equal relative index along the row (the index is
                // monotone in the column).  With prefix sums along the row, a run
                // ends where the next column's index differs and its sum is the
                // difference of the prefix sums at its two ends (so the chain per
                // element is one add).  Each half stores its runs; a run that
                // crosses from the first half into the second was stored by the
                // second half (its first run) and the first half adds its own part
                // to it afterwards -- the slot is zero otherwise, since the second
                // half's indices are all on the other side of the first half's.
                const int cst = hf * HC;
                // relative row of column cst + e of this row: the window entry at
                // x0 - e (query rows) or x0 + e; a run ends where a step bit is set
                const int x0 = ROWQ ? row - cst + BN - 1 : cst - row + BM - 1;
                float pre = 0.f, last = 0.f;
                int m_cur = dwin[x0];
                uint16_t* gp = grow + m_cur;   // the slot of the current run
                if (ok && !bad) {
                    // this half's dZ columns (16-bit, as the products use them), 32 at a time
#pragma unroll
                    for (int g = 0; g < HC / 32; ++g) {
                        uint32_t zr[16];
                        tc_ld16p(lane_base + TM::Z + hf * (HC / 2) + 16 * g, zr);
                        // bit 31 - e2 (query rows) or e2: step between columns 32 g + e2 and + 1
                        const uint32_t mk = step_bits(bars->stepw, ROWQ ? x0 - 32 * g - 31 : x0 + 32 * g + 1);
                        tc_wait_ld();
#pragma unroll
                        for (int e2 = 0; e2 < 32; ++e2) {
                            pre += h16f<BF16>((uint16_t)(zr[e2 >> 1] >> (16 * (e2 & 1))));
                            const bool step = ((ROWQ ? mk >> (31 - e2) : mk >> e2) & 1u) != 0;
                            if (32 * g + e2 + 1 < HC && step) {
                                *gp = f2h16<BF16>(pre - last);
                                last = pre;
                                gp += ROWQ ? -1 : 1;
                            }
                        }
                    }
                    m_cur = (int)(gp - grow);
                }
                const float tail = pre - last;   // the run that ends this half
                if (ok && hf) {
                    if (!bad) *gp = f2h16<BF16>(tail);
                    fence_proxy_async_smem();   // the box is read by the tensor-memory-access unit
                }
                tc_fence_before();
                named_bar_sync(pair_bar, 64);
                if (ok && lane == 0) mbar_arrive(&bars->zread);   // dZ no longer read by this warp
                if (ok && !hf) {
                    const int ms = m_cur < mmax ? m_cur : mmax;
                    grow[ms] = f2h16<BF16>(h16f<BF16>(grow[ms]) + tail);
                    // the clamped relative rows (far field) are summed in registers
                    if (tk.dlo == 0 && qoff >= 0) {
                        g_lo += h16f<BF16>(grow[0]);
                        grow[0] = 0;
                    }
                    if (tk.dhi == p.R - 1) {
                        const int m = p.R - 1 - tk.dlo;
                        if (m + qoff >= 0 && m <= mmax) {
                            g_hi += h16f<BF16>(grow[m]);
                            grow[m] = 0;
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_reduce_add_2d(&tmG, qstage, h * Rp + qa0, t0 + r0 + 32 * w4);
                        bulk_commit();
                    }
                }
                if (ok && bad) raise_error(p.err, DF_ERR_DEVICE_ARG);   // cannot happen for a valid tile
            }
        }
        if (hf == 0 && lane == 0) bulk_wait0();   // this quarter's boxes
        // ------------------------------------------------------------ epilogue
        ok = ok && mbar_wait_warp(&bars->mma3_done, (ntiles - 1) & 1, wc);
        tc_fence_after();
        if (ok) {
            // accumulator columns [hf D/2, (hf+1) D/2), 16 at a time
            float* a1 = acc1_out + ((size_t)(t0 + rt) * p.H + h) * D + hf * (D / 2);
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t r[16];
                tc_ld16(lane_base + TM::ACC1 + hf * (D / 2) + 16 * c, r);
                tc_wait_ld();
                if (row_in) {
                    float4* dst = reinterpret_cast<float4*>(a1 + 16 * c);
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        dst[v] = make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                             __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
                }
            }
            if (!ROWQ) {
                T16* a2 = reinterpret_cast<T16*>(acc2_out) + ((size_t)(t0 + rt) * p.H + h) * D + hf * (D / 2);
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t r[16];
                    tc_ld16(lane_base + TM::ACC2 + hf * (D / 2) + 16 * c, r);
                    tc_wait_ld();
                    if (row_in) {
                        uint4* dst = reinterpret_cast<uint4*>(a2 + 16 * c);
#pragma unroll
                        for (int v = 0; v < 2; ++v) {
                            uint4 w;
                            w.x = pack2<BF16>(__uint_as_float(r[8 * v + 0]), __uint_as_float(r[8 * v + 1]));
                            w.y = pack2<BF16>(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3]));
                            w.z = pack2<BF16>(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5]));
                            w.w = pack2<BF16>(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7]));
                            dst[v] = w;
                        }
                    }
                }
            }
        }
        // the far-field diagonal sums: the two halves' shares, added once;
        // concurrent box additions to these two entries only ever add zero
        xch[hf * BM + row] = g_lo;
        xch[2 * BM + hf * BM + row] = g_hi;
        named_bar_sync(pair_bar, 64);   // both warps of the pair, whatever their state
        if (ok) {
            if (row_in && hf == 0) {
                const float glo = xch[row] + xch[BM + row];
                const float ghi = xch[2 * BM + row] + xch[3 * BM + row];
                uint16_t* grow = reinterpret_cast<uint16_t*>(Gbuf) + ((size_t)(t0 + rt) * p.H + h) * Rp;
                if (glo != 0.f) grow[0] = f2h16<BF16>(h16f<BF16>(grow[0]) + glo);
                if (ghi != 0.f) grow[p.R - 1] = f2h16<BF16>(h16f<BF16>(grow[p.R - 1]) + ghi);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tc_dealloc(tmem, 512);
    }
}

template <int D, bool BF16, int SIGMA, bool DROP>
int launch_one(const ProblemDev& p, const Workspace& ws, const void* r1, const void* r2, const void* c1,
               const void* c2, void* Gbuf, int Rp, float* acc1, void* acc2, const float* lse, cudaStream_t st) {
    using G = Geo<D>;
    using S = BwdSmem<D>;
    CUtensorMap m1, m2, m3, m4, mb, mg;
    const uint64_t tok_dims[2] = {(uint64_t)p.H * D, (uint64_t)p.T};
    const uint64_t tok_str[1] = {(uint64_t)p.H * D * 2};
    // the stored band bias as [rows][128] halves; the box is the tile's part
    // of a block: 128 query rows x BN key columns (dQ kernel) or BN query
    // rows x 128 key columns (dK/dV kernel)
    const uint64_t b_dims[2] = {(uint64_t)kBiasBB, (uint64_t)ws.bias_rows};
    const uint64_t b_str[1] = {(uint64_t)kBiasBB * 2};
    // G viewed as [T][H Rp]: a box of 32 rows of QW sums (the box starts on a
    // multiple of 8 sums, 16 bytes)
    const uint64_t g_dims[2] = {(uint64_t)p.H * Rp, (uint64_t)p.T};
    const uint64_t g_str[1] = {(uint64_t)p.H * Rp * 2};
    const uint32_t boxr[2] = {(uint32_t)G::CW, (uint32_t)G::BM};
    const uint32_t boxc[2] = {(uint32_t)G::CW, (uint32_t)G::BN};
    const uint32_t boxb[2] = {(uint32_t)(SIGMA > 0 ? G::BN : kBiasBB), (uint32_t)(SIGMA > 0 ? kBiasBB : G::BN)};
    const uint32_t boxg[2] = {(uint32_t)S::QW, 32};
    const int code = BF16 ? 0 : 1;
    if (encode_tmap(&m1, code, 2, tok_dims, tok_str, boxr, G::SWZB, r1) ||
        encode_tmap(&m2, code, 2, tok_dims, tok_str, boxr, G::SWZB, r2) ||
        encode_tmap(&m3, code, 2, tok_dims, tok_str, boxc, G::SWZB, c1) ||
        encode_tmap(&m4, code, 2, tok_dims, tok_str, boxc, G::SWZB, c2) ||
        encode_tmap(&mb, 1, 2, b_dims, b_str, boxb, 0, ws.bias) ||
        encode_tmap(&mg, code, 2, g_dims, g_str, boxg, 0, Gbuf))
        return (int)cudaErrorInvalidValue;
    auto kern = bwd_tc_kernel<D, BF16, SIGMA, DROP>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::ALLOC);
    if (e != cudaSuccess) return (int)e;
    dim3 grid(p.H, p.B, (p.L + G::BM - 1) / G::BM);
    const int phase = SIGMA > 0 ? kProfDq : kProfDkv;
    prof_record(phase, 0, st);
    kern<<<grid, kThreads, S::ALLOC, st>>>(m1, m2, m3, m4, mb, mg, p, ws.dtab, ws.relb, lse, ws.rowterm, acc1,
                                           acc2, Gbuf, Rp, r1, r2);
    prof_record(phase, 1, st);
    return (int)cudaGetLastError();
}

}  // namespace
}  // namespace df
