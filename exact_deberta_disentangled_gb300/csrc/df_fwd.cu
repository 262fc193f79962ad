// df_fwd.cu -- tensor-core forward of exact disentangled attention (bf16 /
// fp16 storage, fp32 accumulation) for sm_103a.
//
// One CTA owns 128 query rows of one (sequence, head) and walks the key
// tiles of the sequence, keeping the running max / sum of an online softmax
// ("DisentangledFlash", section "Hugging Face usage": an LSE-producing
// forward; section "Status": the [B, H, L, L] matrix is never stored).
//
// Warp roles (352 threads):
//   warp 0      TMA producer: Q once, K/V tiles into a 2-stage ring, for
//               band tiles the Kr / Qr band rows; it also writes each key
//               tile's column term to shared memory.
//   warp 1      tcgen05 issuer of S and the band products (the whole warp
//               walks the loop, elect.sync picks the issuing lane) and TMEM
//               owner.
//   warps 2..9  softmax: a thread owns one query row (= TMEM lane) and one
//               half of the columns of every key tile.
//   warp 10     tcgen05 issuer of the P.V products.  S of tile n + 2 waits
//               for P.V of tile n (same S buffer); with one issuer for both,
//               P.V of tile n + 1 queued behind that wait.  A commit tracks
//               the MMAs of its own thread, so each issuer's barriers see
//               only its own products.
// The two column halves of a row run independent online softmaxes, each with
// its own running max and sum and its own output accumulator in tensor
// memory (O_h += P_h V_h, K = BN/2 per tile); they are merged once, in the
// epilogue, so no maxima are exchanged inside the key loop (every tile still
// starts with a barrier of the eight softmax warps).
// Tensor memory (512 columns): O_0 and O_1 [0, 2D), two S / P buffers and,
// in [384, 512), two buffers of band-product chunks.  Tile n uses S buffer
// n & 1: S of tile n + 1 is computed while the softmax works on tile n, band
// tile or not.  A band tile's two products (own, then cross)
// are computed 64 band positions at a time (only the chunks the tile's
// relative-index range reaches) into the chunk buffers alternately, so that
// the softmax warps copy one chunk to shared memory while the next one is
// computed; the first two chunks of a band tile are computed while the
// softmax still works on the tile before it.  P (16-bit) is written over the middle half of S, columns
// [BN/4, 3 BN/4), half h's part inside the S columns half h has already read
// (the first half walks its chunks backwards), and feeds the P.V products
// straight from tensor memory.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "df_tile.cuh"

namespace df {
namespace {

constexpr int kThreads = 352;   // producer, S issuer, eight softmax warps, P.V issuer
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleSlack = 8.f;   // keep a stale max while the new one exceeds it by <= 8 (2^8 headroom)
constexpr int kBandChunk = 64;         // band positions per band-product chunk

// chunks of one band product a tile needs: its relative rows dlo .. dhi
DF_DEV int band_chunks(const TileKind& k) { return (k.dhi - k.dlo) / kBandChunk + 1; }

template <int D>
struct FwdTmem {
    using G = Geo<D>;
    static constexpr uint32_t O0 = 0, O1 = D;                  // output accumulators of the column halves
    static constexpr uint32_t S0 = 2 * D > 128 ? 2 * D : 128;  // S / P of even tiles
    static constexpr uint32_t S1 = S0 + G::BN;                 // S / P of odd tiles
    static constexpr uint32_t TB = 384;                        // two band-product chunk buffers
    static constexpr uint32_t POFF = G::BN / 4;                // P starts a quarter into its S buffer
    static_assert(S1 + G::BN <= TB && TB + 2 * kBandChunk <= 512, "tensor memory");
};

template <int D>
struct FwdSmem {
    using G = Geo<D>;
    static constexpr int kStages = 2;
    static constexpr int Q = 0;
    static constexpr int QB = G::BM * D * 2;
    static constexpr int KVB = G::BN * D * 2;
    static constexpr int K0 = Q + QB;
    static constexpr int V0 = K0 + kStages * KVB;
    static constexpr int BAND = V0 + kStages * KVB;
    static constexpr int BSLOT = kBandChunk * D * 2;      // one chunk's band rows ([D / CW][64][CW])
    static constexpr int NBS = D == 128 ? 2 : 4;          // band-row ring slots
    static constexpr int BANDB = NBS * BSLOT;
    static constexpr int OWN = BAND + BANDB;
    static constexpr int OWNB = G::BM * G::OWN_S * 2;
    static constexpr int CROSS = (OWN + OWNB + 15) / 16 * 16;
    static constexpr int CROSSB = G::BN * G::CROSS_S * 2;
    static constexpr int DWIN = CROSS + CROSSB;
    static constexpr int COLB = (DWIN + (G::BM + G::BN) * 4 + 15) / 16 * 16;   // [4 tiles][BN]
    static constexpr int XCH = COLB + 4 * G::BN * 4;      // [4][BM] floats: the halves' maxima and sums
    static constexpr int kMaxTiles = 8192 / G::BN;        // L <= 8192
    static constexpr int KINDS = XCH + 4 * G::BM * 4;     // packed TileKind of every key tile
    static constexpr int MISC = KINDS + kMaxTiles * 4;
    static constexpr int BYTES = MISC + 512;
    static constexpr int ALLOC = BYTES + 1024;  // slack for 1024-byte alignment
    static_assert(ALLOC <= 232448, "shared memory");
};

struct FwdBars {
    uint64_t q_full;
    uint64_t k_full[2], k_empty[2], v_full[2], v_empty[2];   // K and V rings: K is released after S, V after P.V
    uint64_t band_full[4], band_empty[4];   // band-row ring (NBS slots)
    uint64_t tb_full[2], tb_empty[2];       // band-product chunk buffers in tensor memory
    uint64_t s_full[2], pv_done[2];
    uint64_t p_full[4];   // [column half][tile parity]: P of a half of a tile is in tensor memory
    uint64_t drain;   // both issuers' last MMAs, before the tensor memory is freed
    uint32_t tmem_base;
    int abort_flag;
    int cross_base[4];
};
static_assert(sizeof(FwdBars) <= 512, "barrier block");

template <int D, bool BF16, bool DROP>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmKr,
                  const __grid_constant__ CUtensorMap tmQr, const ProblemDev p, const int32_t* __restrict__ dtab,
                  const float* __restrict__ relb, void* __restrict__ out_, float* __restrict__ lse) {
    using G = Geo<D>;
    using S = FwdSmem<D>;
    using TM = FwdTmem<D>;
    constexpr int BM = G::BM, BN = G::BN;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_align1024(smem_raw);
    FwdBars* bars = reinterpret_cast<FwdBars*>(smem + S::MISC);
    uint32_t* dwin2 = reinterpret_cast<uint32_t*>(smem + S::DWIN);
    float* colv = reinterpret_cast<float*>(smem + S::COLB);
    float* xch = reinterpret_cast<float*>(smem + S::XCH);
    uint16_t* own = reinterpret_cast<uint16_t*>(smem + S::OWN);
    uint16_t* cross = reinterpret_cast<uint16_t*>(smem + S::CROSS);
    uint32_t* kinds = reinterpret_cast<uint32_t*>(smem + S::KINDS);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.y, b = blockIdx.z;
    int t0, n;
    seq_ok(p, b, t0, n);
    const int i0 = blockIdx.x * BM;
    if (i0 >= n || b < p.b_base) return;   // (sequences before b_base: an earlier part's)
    const int ntiles = (n + BN - 1) / BN;
    auto s_col = [](int it) -> uint32_t { return (it & 1) ? TM::S1 : TM::S0; };

    if (threadIdx.x == 0) {
        mbar_init(&bars->q_full, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars->k_full[s], 1);
            mbar_init(&bars->k_empty[s], 1);
            mbar_init(&bars->v_full[s], 1);
            mbar_init(&bars->v_empty[s], 1);
            mbar_init(&bars->s_full[s], 1 + 32);   // S's commit and the producer's 32 lanes (column terms)
            mbar_init(&bars->pv_done[s], 1);
            mbar_init(&bars->p_full[s], 4);
            mbar_init(&bars->p_full[2 + s], 4);
        }
        for (int r = 0; r < S::NBS; ++r) {
            mbar_init(&bars->band_full[r], 1);
            mbar_init(&bars->band_empty[r], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars->tb_full[s], 1);
            mbar_init(&bars->tb_empty[s], 8);
        }
        mbar_init(&bars->drain, 2);
        bars->abort_flag = 0;
        fence_barrier_init();
    }
    // the kind of every key tile (two relative-index loads each), once.  When
    // the band bias is saved, every tile of a 128 x 128 band block is a band
    // tile (the saved blocks are then complete; with BN = 128 tile = block).
    for (int t = threadIdx.x; t < ntiles; t += kThreads) {
        TileKind k = classify<BM, BN, 1>(p, dtab, i0 - t * BN);
        if (BN < kBiasBB && p.saved_bias && k.uniform) {
            const int j0b = t * BN / kBiasBB * kBiasBB;
            if (!classify<BM, kBiasBB, 1>(p, dtab, i0 - j0b).uniform) k.uniform = 0;
        }
        kinds[t] = pack_kind(k);
    }
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
        // The warp walks the key tiles: lane 0 issues the tensor copies, and
        // the warp writes each tile's per-key column term to shared memory
        // (P2C scalar of uniform tiles, with the key mask folded in; key mask
        // of band tiles; -inf past the sequence end), four tiles deep, and
        // announces it on tile m's S barrier.  Tile m's term goes to slot m & 3
        // once V of tile m - 1 is loaded: that load waited for P.V of tile
        // m - 3, so tile m - 4 is long done.  Per tile n: V(n), then K(n + 1),
        // the column terms of n + 1 (their global loads issued a tile ahead)
        // and the band rows of n + 1, so that K, which S waits for, is never
        // queued behind the column terms' loads.
        const size_t T = (size_t)p.T;
        const float* relb_h = relb + (size_t)h * 4 * T;
        constexpr int NJ = BN / 32;
        float cb[NJ];
        int mk[NJ];
        auto fetch_columns = [&](int m) {
            const TileKind k = unpack_kind(kinds[m]);
#pragma unroll
            for (int q = 0; q < NJ; ++q) {
                const int j = m * BN + 32 * q + lane;
                const int js = j < n ? j : 0;   // an index that is safe to load
                cb[q] = k.uniform ? ld_early(relb_h + (2 + k.which) * T + t0 + js) : 0.f;
                mk[q] = (!k.uniform && p.kmask) ? ld_early(p.kmask + t0 + js) : 1;
            }
        };
        auto put_columns = [&](int m) -> bool {
            float* cv = colv + (m & 3) * BN;
#pragma unroll
            for (int q = 0; q < NJ; ++q) {
                const int j = 32 * q + lane;
                cv[j] = (m * BN + j < n && mk[q] != 0) ? cb[q] : -INFINITY;
            }
            // the terms are announced with S of tile m (its S buffer's barrier
            // counts the producer's lanes too), once that barrier has completed
            // the phase of tile m - 2: an arrival never counts toward an older tile
            if (m >= 2 && !mbar_wait_warp(&bars->s_full[m & 1], ((m - 2) >> 1) & 1, wc)) return false;
            mbar_arrive(&bars->s_full[m & 1]);
            return true;
        };
        int band_loads = 0, k_cnt[2] = {0, 0}, v_cnt[2] = {0, 0};   // copies issued per barrier
        // K of tile m as soon as S (band tile: and the cross product) of tile
        // m - 2 has read its stage
        auto load_k = [&](int m) -> bool {
            const int s = m & 1, use = m >> 1;
            if (use > 0 && !mbar_wait_warp(&bars->k_empty[s], (use - 1) & 1, wc)) return false;
            if (lane == 0) {
                mbar_arrive_expect_tx(&bars->k_full[s], S::KVB);
                for (int c = 0; c < G::NCH; ++c)
                    tma_load_2d(smem + S::K0 + s * S::KVB + c * BN * G::CW * 2, &tmK, h * D + c * G::CW,
                                t0 + m * BN, &bars->k_full[s]);
            }
            ++k_cnt[s];
            return true;
        };
        // V of tile m once P.V of tile m - 2 has read its stage
        auto load_v = [&](int m) -> bool {
            const int s = m & 1, use = m >> 1;
            if (use > 0 && !mbar_wait_warp(&bars->v_empty[s], (use - 1) & 1, wc)) return false;
            if (lane == 0) {
                mbar_arrive_expect_tx(&bars->v_full[s], S::KVB);
                for (int c = 0; c < G::NCH; ++c)
                    tma_load_2d(smem + S::V0 + s * S::KVB + c * BN * G::CW * 2, &tmV, h * D + c * G::CW,
                                t0 + m * BN, &bars->v_full[s]);
            }
            ++v_cnt[s];
            return true;
        };
        // band rows of tile m's product chunks: Kr rows for the own product,
        // then Qr rows for the cross product, 64 per ring slot
        auto load_band = [&](int m) -> bool {
            const TileKind tk = unpack_kind(kinds[m]);
            const int nch = tk.uniform ? 0 : band_chunks(tk);
            for (int g = 0; g < 2 * nch; ++g) {
                const int r = band_loads % S::NBS, u = band_loads / S::NBS;
                if (u > 0 && !mbar_wait_warp(&bars->band_empty[r], (u - 1) & 1, wc)) return false;
                if (lane == 0) {
                    const int row0 = h * p.R + tk.dlo + kBandChunk * (g < nch ? g : g - nch);
                    mbar_arrive_expect_tx(&bars->band_full[r], S::BSLOT);
                    for (int c = 0; c < G::NCH; ++c)
                        tma_load_2d(smem + S::BAND + r * S::BSLOT + c * kBandChunk * G::CW * 2,
                                    g < nch ? &tmKr : &tmQr, c * G::CW, row0, &bars->band_full[r]);
                }
                ++band_loads;
            }
            return true;
        };
        if (lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            mbar_arrive_expect_tx(&bars->q_full, S::QB);
            for (int c = 0; c < G::NCH; ++c)
                tma_load_2d(smem + S::Q + c * BM * G::CW * 2, &tmQ, h * D + c * G::CW, t0 + i0, &bars->q_full);
        }
        fetch_columns(0);
        bool ok = load_k(0) && put_columns(0);
        if (ntiles > 1) fetch_columns(1);
        ok = ok && load_band(0);
        for (int it = 0; it < ntiles && ok; ++it) {
            if (!(ok = load_v(it)) || it + 1 == ntiles) break;
            ok = load_k(it + 1) && put_columns(it + 1);
            if (it + 2 < ntiles) fetch_columns(it + 2);
            ok = ok && load_band(it + 1);
        }
        // no copy of this CTA is still landing in shared memory when it exits
        // (each barrier's last phase is its last copy; the ones before it
        // completed before that copy was issued)
        if (lane == 0) {
            mbar_drain(&bars->q_full, 0, wc.limit_ns);
            for (int s = 0; s < 2; ++s) {
                if (k_cnt[s] > 0) mbar_drain(&bars->k_full[s], (k_cnt[s] - 1) & 1, wc.limit_ns);
                if (v_cnt[s] > 0) mbar_drain(&bars->v_full[s], (v_cnt[s] - 1) & 1, wc.limit_ns);
            }
            for (int r = 0; r < S::NBS && r < band_loads; ++r)
                mbar_drain(&bars->band_full[r], ((band_loads - 1 - r) / S::NBS) & 1, wc.limit_ns);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ S / band-product issuer
        // The whole warp walks the issue loop (its control flow warp-uniform);
        // the MMAs and commits are the elect.sync forms, issued by one lane.
        // Operand descriptors are built once (per CTA or per ring stage) and
        // advanced per k-step by a constant.
        {
            const uint32_t sQ = smem_u32(smem + S::Q), sBand = smem_u32(smem + S::BAND);
            constexpr uint32_t idS = idesc_f16(128, BN, BF16, false, false);
            constexpr uint32_t idT = idesc_f16(128, kBandChunk, BF16, false, false);
            const uint64_t dQ = desc_k<G>(sQ, BM, 0), dBand = desc_k<G>(sBand, kBandChunk, 0);
            const uint64_t dK0 = desc_k<G>(smem_u32(smem + S::K0), BN, 0), dK1 = dadd(dK0, S::KVB);
            bool ok = mbar_wait_warp(&bars->q_full, 0, wc);
            int bc = 0;   // band chunks issued: ring slot bc % NBS, chunk buffer bc & 1
            // S of tile m into buffer m & 1.  K's stage is released here for a
            // uniform tile, after the cross product for a band tile.
            auto issue_s = [&](int m, const TileKind& tk) -> bool {
                const int s = m & 1, use = m >> 1;
                const uint64_t dK = s ? dK1 : dK0;
                if (!mbar_wait_warp(&bars->k_full[s], use & 1, wc)) return false;
                // buffer s free: P.V of tile m - 2 has consumed its P
                if (m >= 2 && !mbar_wait_warp(&bars->pv_done[s], ((m - 2) >> 1) & 1, wc)) return false;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < D / 16; ++k)
                    tc_mma_ss_w(tmem + s_col(m), dadd(dQ, kofs<G>(BM, k)), dadd(dK, kofs<G>(BN, k)), idS, k != 0);
                tc_commit_w(&bars->s_full[s]);
                if (tk.uniform) tc_commit_w(&bars->k_empty[s]);
                return true;
            };
            // the chunks of band tile m's products: chunk g < nch is
            // Q . Kr[dlo + 64 g ..]^T (lanes = query rows), chunk nch + g is
            // K . Qr[dlo + 64 g ..]^T (lanes = key columns).  Each waits for its
            // chunk buffer's previous chunk to be copied out and its band rows.
            auto issue_band = [&](int m, const TileKind& tk) -> bool {
                const int nch = band_chunks(tk);
                const int s = m & 1, use = m >> 1;
                const uint64_t dK = s ? dK1 : dK0;
                for (int g = 0; g < 2 * nch; ++g) {
                    const int tb = bc & 1, r = bc % S::NBS;
                    // the chunk's band rows (normally landed long before; their
                    // copy needs only chunk bc - NBS's product, issued above)
                    if (!mbar_wait_warp(&bars->band_full[r], (bc / S::NBS) & 1, wc)) return false;
                    // K of tile m stays in its stage until the last cross chunk (S(m) has waited for it)
                    if (g == nch && !mbar_wait_warp(&bars->k_full[s], use & 1, wc)) return false;
                    // then the gate: the softmax warps have copied chunk bc - 2 out of this slot
                    if (bc >= 2 && !mbar_wait_warp(&bars->tb_empty[tb], ((bc >> 1) - 1) & 1, wc)) return false;
                    tc_fence_after();
                    const bool cross_pass = g >= nch;
                    const uint64_t dA = cross_pass ? dK : dQ;
                    const int arows = cross_pass ? BN : BM;
                    const uint64_t dB = dadd(dBand, (uint32_t)(r * S::BSLOT));
#pragma unroll
                    for (int k = 0; k < D / 16; ++k)
                        tc_mma_ss_w(tmem + TM::TB + tb * kBandChunk, dadd(dA, kofs<G>(arows, k)),
                                    dadd(dB, kofs<G>(kBandChunk, k)), idT, k != 0);
                    tc_commit_w(&bars->band_empty[r]);
                    tc_commit_w(&bars->tb_full[tb]);
                    if (g == 2 * nch - 1) tc_commit_w(&bars->k_empty[s]);
                    ++bc;
                }
                return true;
            };
            // test-only stall injection: this issuer stops before this tile, so
            // that the other roles' bounded waits run out
            const int stall = p.fault_kernel == 0 ? p.fault_tile : -1;
            // S of every tile, then its band chunks: the first two as soon as
            // the previous band tile's chunks are copied out (early in that
            // tile), the rest as the softmax warps copy this tile's own, so S
            // of the next tile follows this tile's copies, well before the
            // softmax warps need it
            for (int m = 0; m < ntiles && ok; ++m) {
                if (stall >= 0 && m >= stall) break;
                const TileKind tk = unpack_kind(kinds[m]);
                ok = issue_s(m, tk) && (tk.uniform || issue_band(m, tk));
            }
            // every MMA issued above has completed before the tensor memory is freed
            tc_commit_w(&bars->drain);
            mbar_drain(&bars->drain, 0, wc.limit_ns);
        }
    } else if (warp == 10) {
        // ------------------------------------------------------------ P.V issuer
        // O_h += P_h V_h for the two column halves of every tile, each as soon
        // as its P is ready; V's stage and the S buffer are released after.
        {
            constexpr uint32_t idO = idesc_f16(128, D, BF16, false, true);
            const uint64_t dV0 = desc_mn<G>(smem_u32(smem + S::V0), BN, 0), dV1 = dadd(dV0, S::KVB);
            bool ok = true;
            for (int it = 0; it < ntiles && ok; ++it) {
                const int s = it & 1;
                const uint64_t dV = s ? dV1 : dV0;
                if (!(ok = mbar_wait_warp(&bars->v_full[s], (it >> 1) & 1, wc))) break;
                for (int hf = 0; hf < 2 && ok; ++hf) {
                    if (!(ok = mbar_wait_warp(&bars->p_full[2 * hf + (it & 1)], (it >> 1) & 1, wc))) break;
                    tc_fence_after();
#pragma unroll
                    for (int k = 0; k < BN / 32; ++k)
                        tc_mma_ts_w(tmem + (hf ? TM::O1 : TM::O0), tmem + s_col(it) + TM::POFF + hf * (BN / 4) + k * 8,
                                    dadd(dV, mnofs<G>(hf * (BN / 32) + k)), idO, (it | k) != 0);
                }
                if (!ok) break;
                tc_commit_w(&bars->v_empty[s]);
                tc_commit_w(&bars->pv_done[it & 1]);
            }
            tc_commit_w(&bars->drain);
            mbar_drain(&bars->drain, 0, wc.limit_ns);
        }
    } else {
        // ------------------------------------------------------------ softmax
        // Eight warps: warp w owns TMEM lanes 32 (w & 3) .. +31 (query rows)
        // and column half hf = (w - 2) / 4 of every key tile, so two warps
        // share each SM sub-partition.
        const int w4 = warp & 3;
        const int hf = (warp - 2) >> 2;
        const int row = 32 * w4 + lane;           // query row in the tile == TMEM lane
        const int tid = threadIdx.x - 64;         // 0..255
        const int pair_bar = 2 + w4;              // named barrier of this row's two warps
        const uint32_t lane_base = tmem + ((uint32_t)(32 * w4) << 16);
        const uint32_t ocol = hf ? TM::O1 : TM::O0;
        constexpr int NCT = BN / 64;              // 32-column chunks per thread
        const int cbeg = hf * NCT;
        // chunk order: backwards in the first half, so that the 16-bit result of
        // chunk c (TMEM columns BN/4 + 16 c ..) only covers chunks already read
        auto chunk = [&](int cc) { return hf ? cbeg + cc : cbeg + NCT - 1 - cc; };
        const int i = i0 + row;
        const bool row_in = i < n;
        const bool row_valid = row_in && (!p.qmask || p.qmask[t0 + i]);
        const size_t T = (size_t)p.T;
        const float* relb_h = relb + (size_t)h * 4 * T;
        const float a0 = row_in ? relb_h[t0 + i] : 0.f;
        const float a1 = row_in ? relb_h[T + t0 + i] : 0.f;
        const float kscale = p.scale * kLog2e;
        float m_run = -INFINITY, l_part = 0.f;   // this half's running max (log2 units) and sum
        int gc = 0;   // band-product chunks copied out (chunk buffer gc & 1)
        bool ok = true;
        uint16_t* own_row = own + row * G::OWN_S;
        // this half's output accumulator, all D columns, 16 at a time
        auto rescale_o = [&](float alpha) {
#pragma unroll
            for (int c = 0; c < D / 16; ++c) {
                uint32_t r[16];
                tc_ld16(lane_base + ocol + 16 * c, r);
                tc_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
                tc_st16(lane_base + ocol + 16 * c, r);
            }
        };
        auto kind_of = [&](int t) { return unpack_kind(kinds[t < ntiles ? t : ntiles - 1]); };
        BandRaw bn = band_fetch<BM, BN, 1, true>(p, dtab, i0, w4, tid, lane);   // band indices, one tile ahead
        // Every warp walks every tile and meets every named barrier, also after
        // a bounded wait gave up (ok == false: the work is skipped, no wait is
        // taken): a warp that left the loop early would leave its siblings
        // parked in bar.sync for good.
        for (int it = 0; it < ntiles; ++it) {
            const int j0 = it * BN;
            const TileKind tk = kind_of(it);
            const float* colb = colv + (it & 3) * BN;
            // every tile starts with all eight warps: band tiles rewrite the index
            // window and the band windows, and the per-warp arrivals on the
            // tile's barriers (counts of 8, or 4 per column half) must never
            // meet a warp that is a whole tile ahead -- its arrival would
            // complete the previous tile's phase
            named_bar_sync(1, 256);
            BandRaw bc = bn;   // this tile's band indices (fetched during the previous tile)
            if (it + 1 < ntiles && !kind_of(it + 1).uniform)
                bn = band_fetch<BM, BN, 1, true>(p, dtab, i0 - j0 - BN, w4, tid, lane);
            int own_a = 0;
            if (!tk.uniform) {
                pin(bc.dw);
                pin(bc.dwp);
                pin(bc.rng);
                // index window entry x with entry x - 1 beside it: the band
                // coordinates of two neighbouring columns of a row in one load
                if (tid < BM + BN - 1)
                    dwin2[tid] = ((uint32_t)(bc.dw - tk.dlo) & 0xFFFFu) | ((uint32_t)(bc.dwp - tk.dlo) << 16);
                int lo = __shfl_sync(0xffffffffu, bc.rng, 0) - tk.dlo, hi = __shfl_sync(0xffffffffu, bc.rng, 1) - tk.dlo;
                const int clo = __shfl_sync(0xffffffffu, bc.rng, 2) - tk.dlo, chi = __shfl_sync(0xffffffffu, bc.rng, 3) - tk.dlo;
                own_a = lo & ~15;
                const int ca = clo & ~15;
                // the chunks of the own product, then of the cross product; the
                // two warps of a lane quarter copy half of each chunk's part of
                // the quarter's window
                const int nch = band_chunks(tk);
                for (int g = 0; g < 2 * nch; ++g, ++gc) {
                    const int tb = gc & 1;
                    ok = ok && mbar_wait_warp(&bars->tb_full[tb], (gc >> 1) & 1, wc);
                    if (!ok) continue;
                    tc_fence_after();
                    const uint32_t tcol = lane_base + TM::TB + tb * kBandChunk;
                    if (g < nch)
                        copy_band_chunk(tcol, kBandChunk * g, lo, hi, own_a, own_row, kscale, hf, G::OWN_S, p.err);
                    else if (32 * w4 < BN)
                        copy_band_chunk(tcol, kBandChunk * (g - nch), clo, chi, ca, cross + row * G::CROSS_S,
                                        kscale, hf, G::CROSS_S, p.err);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars->tb_empty[tb]);
                }
                if (lane == 0 && hf == 0) bars->cross_base[w4] = ca;
                named_bar_sync(1, 256);   // dwin, own / cross windows complete
            }
            // S of this tile and its column terms (the producer arrives on the same barrier)
            ok = ok && mbar_wait_warp(&bars->s_full[it & 1], (it >> 1) & 1, wc);
            if (!ok) continue;   // no named barrier below this point of the tile
            tc_fence_after();
            const uint32_t scol = s_col(it);
            float rb = tk.uniform ? (tk.which ? a1 : a0) : 0.f;
            if (!row_valid) rb = -INFINITY;
            const bool band = !tk.uniform;
            // a new running max for this half: rescale the sum now and the
            // accumulator after this tile's P is stored (fewer live registers),
            // once the previous tile's P.V has landed
            float alpha = 1.f;
            bool resc = false;
            auto raise_max = [&](float tmax) {
                const bool need = tmax > m_run + kRescaleSlack || (m_run == -INFINITY && tmax > -INFINITY);
                if (need) {
                    const float a = m_run == -INFINITY ? 0.f : ex2(m_run - tmax);
                    alpha *= a;
                    l_part *= a;
                    m_run = tmax;
                }
                resc |= need;
            };
            // Probabilities of this thread's chunks against the running max,
            // written as 16-bit P over the middle half of S, chunk by chunk in
            // chunk() order.  RAW: S holds Q.K^T (uniform tile: scale and column
            // term applied here); otherwise band pass 1 left the biased logits.
            auto p_pass = [&](auto raw_tag) -> float {
                constexpr bool RAW = decltype(raw_tag)::value;
                const float mm = (m_run == -INFINITY || rb == -INFINITY) ? INFINITY : m_run - rb;
                const float nmm = -mm;
                float sm0 = 0.f, sm1 = 0.f;
#pragma unroll 1
                for (int cc = 0; cc < NCT; ++cc) {
                    const int c = chunk(cc);
                    uint32_t r[32];
                    tc_ld32(lane_base + scol + 32 * c, r);
                    tc_wait_ld();
                    uint32_t keep = 0xFFFFFFFFu;
                    if constexpr (DROP) keep = keep_bits32_row(p, b, h, i, j0 + 32 * c);
                    const float2* cbp = reinterpret_cast<const float2*>(colb + 32 * c);
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        float x0 = __uint_as_float(r[2 * e]), x1 = __uint_as_float(r[2 * e + 1]);
                        if constexpr (RAW) {
                            const float2 cv = cbp[e];
                            ffma2(x0, x1, x0, x1, kscale, kscale, cv.x, cv.y);
                        }
                        fadd2(x0, x1, x0, x1, nmm, nmm);
                        const float p0 = ex2(x0);
                        const float p1 = ex2(x1);
                        fadd2(sm0, sm1, sm0, sm1, p0, p1);
                        float d0 = p0, d1 = p1;
                        if constexpr (DROP) {
                            d0 = ((keep >> (2 * e)) & 1u) ? p0 * p.drop_scale : 0.f;
                            d1 = ((keep >> (2 * e + 1)) & 1u) ? p1 * p.drop_scale : 0.f;
                        }
                        pk[e] = pack2<BF16>(d0, d1);
                    }
                    tc_st16(lane_base + scol + TM::POFF + 16 * c, pk);
                }
                return sm0 + sm1;
            };
            float sum = 0.f;
            if (!band) {
                // Uniform tile, one pass against the running max (+inf for a dead
                // row or before the first max: every probability 0), kept in
                // registers.  When the tile moves the running max by more than
                // kRescaleSlack (and on the first tile) the warp recomputes P
                // with p_pass instead.
                uint32_t pk[16 * NCT];
                const bool attempted = m_run != -INFINITY && rb != -INFINITY;
                const float mm = attempted ? m_run - rb : INFINITY;
                const float nmm = -mm;
                float tm01 = -INFINITY, tm23 = -INFINITY;
                float sm[4] = {0.f, 0.f, 0.f, 0.f};
                // all of this thread's S columns in one tensor-memory round trip
                uint32_t rr[32 * NCT];
#pragma unroll
                for (int cc = 0; cc < NCT; ++cc) tc_ld32p(lane_base + scol + 32 * (cbeg + cc), rr + 32 * cc);
                tc_wait_ld();
#pragma unroll
                for (int cc = 0; cc < NCT; ++cc) {
                    const int c = cbeg + cc;
                    const uint32_t* r = rr + 32 * cc;
                    uint32_t keep = 0xFFFFFFFFu;
                    if constexpr (DROP) keep = keep_bits32_row(p, b, h, i, j0 + 32 * c);
                    const float4* cb4 = reinterpret_cast<const float4*>(colb + 32 * c);
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const float4 cv = cb4[q];
                        float x0, x1, x2, x3;
                        ffma2(x0, x1, __uint_as_float(r[4 * q + 0]), __uint_as_float(r[4 * q + 1]), kscale, kscale,
                              cv.x, cv.y);
                        ffma2(x2, x3, __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]), kscale, kscale,
                              cv.z, cv.w);
                        tm01 = fmax3(tm01, x0, x1);
                        tm23 = fmax3(tm23, x2, x3);
                        float d0, d1, d2, d3;
                        fadd2(d0, d1, x0, x1, nmm, nmm);
                        fadd2(d2, d3, x2, x3, nmm, nmm);
                        float p0 = ex2(d0), p1 = ex2(d1);
                        float p2 = ex2(d2), p3 = ex2(d3);
                        fadd2(sm[0], sm[1], sm[0], sm[1], p0, p1);
                        fadd2(sm[2], sm[3], sm[2], sm[3], p2, p3);
                        if constexpr (DROP) {
                            const uint32_t kq = keep >> (4 * q);
                            p0 = (kq & 1u) ? p0 * p.drop_scale : 0.f;
                            p1 = (kq & 2u) ? p1 * p.drop_scale : 0.f;
                            p2 = (kq & 4u) ? p2 * p.drop_scale : 0.f;
                            p3 = (kq & 8u) ? p3 * p.drop_scale : 0.f;
                        }
                        pk[16 * cc + 2 * q] = pack2<BF16>(p0, p1);
                        pk[16 * cc + 2 * q + 1] = pack2<BF16>(p2, p3);
                    }
                }
                sum = (sm[0] + sm[1]) + (sm[2] + sm[3]);
                raise_max(fmaxf(tm01, tm23) + rb);
                const bool redo = resc || (!attempted && m_run != -INFINITY && rb != -INFINITY);
                if (__any_sync(0xffffffffu, redo)) {
                    sum = p_pass(std::true_type{});
                } else {
#pragma unroll
                    for (int cc = 0; cc < NCT; ++cc) {
                        uint32_t r16[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e) r16[e] = pk[16 * cc + e];
                        tc_st16(lane_base + scol + TM::POFF + 16 * (cbeg + cc), r16);
                    }
                }
            } else {
                // ---- band tile, pass 1: biased logits (written back over S) and
                // the tile max; pass 2 (p_pass): probabilities.  With a saved
                // band bias, pass 1 also stores this row's bias values.
                float tm = -INFINITY;
                uint4* bias_dst = nullptr;
                if (p.saved_bias) {
                    const int brow = bias_block_row(p, b, h, t0, i0 / kBiasBB, j0 / kBiasBB);
                    if (brow >= 0)
                        bias_dst = reinterpret_cast<uint4*>(p.saved_bias + ((size_t)brow + row) * kBiasBB);
                    else if (lane == 0)
                        raise_error(p.err, DF_ERR_DEVICE_ARG);   // cannot happen: the table keeps every band block
                }
#pragma unroll 1
                for (int cc = 0; cc < NCT; ++cc) {
                    const int c = cbeg + cc;
                    uint32_t r[32];
                    tc_ld32(lane_base + scol + 32 * c, r);
                    tc_wait_ld();
                    const float2* cb2 = reinterpret_cast<const float2*>(colb + 32 * c);
                    const uint16_t* crow = cross + 32 * c * G::CROSS_S - bars->cross_base[c];
                    const uint32_t* dw2 = dwin2 + row - 32 * c + BN - 1;
                    const uint16_t* orow = own_row - own_a;
                    uint32_t bpk[16];
                    // columns 2q, 2q + 1: band coordinates m0, m1 (entries x, x - 1)
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        const uint32_t mm = dw2[-2 * q];
                        int m0 = (int)(mm & 0xFFFFu), m1 = (int)(mm >> 16);
                        int c0 = m0, c1 = m1;   // the cross window's own range check
                        DF_CLAMP_CHECK(m0, own_a, own_a + G::OWN_S, p.err);
                        DF_CLAMP_CHECK(m1, own_a, own_a + G::OWN_S, p.err);
                        DF_CLAMP_CHECK(c0, bars->cross_base[c], bars->cross_base[c] + G::CROSS_S, p.err);
                        DF_CLAMP_CHECK(c1, bars->cross_base[c], bars->cross_base[c] + G::CROSS_S, p.err);
                        const uint32_t ov = __byte_perm(orow[m0], orow[m1], 0x5410);
                        const uint32_t cv =
                            __byte_perm(crow[2 * q * G::CROSS_S + c0], crow[(2 * q + 1) * G::CROSS_S + c1], 0x5410);
                        const uint32_t bb = band_bias2(ov, cv);
                        bpk[q] = bb;
                        float b0, b1;
                        h2x2f(bb, b0, b1);
                        const float2 cb = cb2[q];
                        float x0, x1;
                        ffma2(x0, x1, __uint_as_float(r[2 * q]), __uint_as_float(r[2 * q + 1]), kscale, kscale, cb.x,
                              cb.y);
                        fadd2(x0, x1, x0, x1, b0, b1);
                        tm = fmax3(tm, x0, x1);
                        r[2 * q] = __float_as_uint(x0);
                        r[2 * q + 1] = __float_as_uint(x1);
                    }
                    tc_st32(lane_base + scol + 32 * c, r);
                    if (bias_dst) {
                        const int lc0 = (j0 % kBiasBB + 32 * c) / 8;   // block chunk of column 32 c
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            bias_dst[bias_chunk(row, lc0 + q)] =
                                make_uint4(bpk[4 * q], bpk[4 * q + 1], bpk[4 * q + 2], bpk[4 * q + 3]);
                    }
                }
                tc_wait_st();
                raise_max(tm + rb);
                sum = p_pass(std::false_type{});
            }
            l_part += sum;
            // a new running max: O_h is rescaled once P.V of the previous tile
            // has landed in it
            if (__any_sync(0xffffffffu, resc) && it > 0) {
                if (!(ok = mbar_wait_warp(&bars->pv_done[(it - 1) & 1], ((it - 1) >> 1) & 1, wc))) continue;
                tc_fence_after();
                rescale_o(alpha);
            }
            tc_wait_st();
            tc_fence_before();
            __syncwarp();
            // P of this half is announced on the barrier of the tile's parity.
            // S of the next tile is computed before the P.V issuer waits for
            // this tile's P (and V), so the softmax warps can announce the next
            // tile's P before the P.V issuer takes this one; on a single
            // barrier the two phases would be indistinguishable to its parity
            // wait (a slow V copy made it wait for good).  The next phase of
            // this tile's barrier is two tiles on, whose S waits for P.V of
            // this tile, which the P.V issuer issues only after taking this P.
            if (lane == 0) mbar_arrive(&bars->p_full[2 * hf + (it & 1)]);
        }
        // ------------------------------------------------------------ epilogue
        // merge the two halves: m = max(m_0, m_1), l = sum_h l_h 2^(m_h - m),
        // O = sum_h O_h 2^(m_h - m) / l
        ok = ok && mbar_wait_warp(&bars->pv_done[(ntiles - 1) & 1], ((ntiles - 1) >> 1) & 1, wc);
        tc_fence_after();
        xch[hf * BM + row] = m_run;
        xch[2 * BM + hf * BM + row] = l_part;
        named_bar_sync(pair_bar, 64);   // both warps of the pair, whatever their state
        if (ok) {
            const float m0 = xch[row], m1 = xch[BM + row];
            const float mx = fmaxf(m0, m1);
            const float s0 = m0 == -INFINITY ? 0.f : ex2(m0 - mx);
            const float s1 = m1 == -INFINITY ? 0.f : ex2(m1 - mx);
            const float l_run = xch[2 * BM + row] * s0 + xch[3 * BM + row] * s1;
            const bool any = row_valid && l_run > 0.f;
            const float inv = any ? 1.f / l_run : 0.f;
            const float f0 = s0 * inv, f1 = s1 * inv;
            using OutT = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
            OutT* orow = reinterpret_cast<OutT*>(out_) + ((size_t)(t0 + i) * p.H + h) * D + hf * (D / 2);
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t r0[16], r1[16];
                tc_ld16(lane_base + TM::O0 + hf * (D / 2) + 16 * c, r0);
                tc_ld16(lane_base + TM::O1 + hf * (D / 2) + 16 * c, r1);
                tc_wait_ld();
                if (row_in) {
                    float o[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        o[e] = fmaf(__uint_as_float(r0[e]), f0, __uint_as_float(r1[e]) * f1);
                    uint4* dst = reinterpret_cast<uint4*>(orow + 16 * c);
#pragma unroll
                    for (int v = 0; v < 2; ++v) {
                        uint4 w;
                        w.x = pack2<BF16>(o[8 * v + 0], o[8 * v + 1]);
                        w.y = pack2<BF16>(o[8 * v + 2], o[8 * v + 3]);
                        w.z = pack2<BF16>(o[8 * v + 4], o[8 * v + 5]);
                        w.w = pack2<BF16>(o[8 * v + 6], o[8 * v + 7]);
                        dst[v] = w;
                    }
                }
            }
            // lse == nullptr: the inference forward, which keeps no LSE
            if (row_in && hf == 0 && lse) lse[lse_index(p, b, h, t0, i)] = any ? (mx + log2f(l_run)) * kLn2 : INFINITY;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tc_dealloc(tmem, 512);
    }
}

template <int D, bool BF16, bool DROP>
int launch_fwd_impl(const ProblemDev& p, const Workspace& ws, const void* q, const void* k, const void* v,
                    const void* qr, const void* kr, void* out, float* lse, cudaStream_t st) {
    using G = Geo<D>;
    using S = FwdSmem<D>;
    CUtensorMap mq, mk, mv, mkr, mqr;
    const uint64_t tok_dims[2] = {(uint64_t)p.H * D, (uint64_t)p.T};
    const uint64_t tok_str[1] = {(uint64_t)p.H * D * 2};
    const uint64_t rel_dims[2] = {(uint64_t)D, (uint64_t)p.H * p.R};
    const uint64_t rel_str[1] = {(uint64_t)D * 2};
    const uint32_t boxq[2] = {(uint32_t)G::CW, (uint32_t)G::BM};
    const uint32_t boxk[2] = {(uint32_t)G::CW, (uint32_t)G::BN};
    const uint32_t boxr[2] = {(uint32_t)G::CW, (uint32_t)kBandChunk};
    const int code = BF16 ? 0 : 1;
    if (encode_tmap(&mq, code, 2, tok_dims, tok_str, boxq, G::SWZB, q) ||
        encode_tmap(&mk, code, 2, tok_dims, tok_str, boxk, G::SWZB, k) ||
        encode_tmap(&mv, code, 2, tok_dims, tok_str, boxk, G::SWZB, v) ||
        encode_tmap(&mkr, code, 2, rel_dims, rel_str, boxr, G::SWZB, kr) ||
        encode_tmap(&mqr, code, 2, rel_dims, rel_str, boxr, G::SWZB, qr))
        return (int)cudaErrorInvalidValue;
    auto kern = fwd_tc_kernel<D, BF16, DROP>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::ALLOC);
    if (e != cudaSuccess) return (int)e;
    dim3 grid((p.L + G::BM - 1) / G::BM, p.H, p.b_count > 0 ? p.b_base + p.b_count : p.B);
    prof_record(kProfFwd, 0, st);
    kern<<<grid, kThreads, S::ALLOC, st>>>(mq, mk, mv, mkr, mqr, p, ws.dtab, ws.relb, out, lse);
    prof_record(kProfFwd, 1, st);
    return (int)cudaGetLastError();
}

}  // namespace

int launch_fwd_tc(const ProblemDev& p, const Workspace& ws, df_dtype dt, const void* q, const void* k,
                  const void* v, const void* qr, const void* kr, void* out, float* lse, cudaStream_t st) {
#define DF_ONE(D_, BF_, DR_) launch_fwd_impl<D_, BF_, DR_>(p, ws, q, k, v, qr, kr, out, lse, st)
#define DF_DT(D_, DR_) (dt == DF_BF16 ? DF_ONE(D_, true, DR_) : DF_ONE(D_, false, DR_))
#define DF_DROP(D_) (p.dropout ? DF_DT(D_, true) : DF_DT(D_, false))
    switch (p.D) {
        case 32: return DF_DROP(32);
        case 64: return DF_DROP(64);
        case 128: return DF_DROP(128);
    }
#undef DF_DROP
#undef DF_DT
#undef DF_ONE
    return (int)cudaErrorInvalidValue;
}

}  // namespace df
