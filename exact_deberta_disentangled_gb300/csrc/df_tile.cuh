// df_tile.cuh -- tile geometry and the relative-position machinery shared by
// the tensor-core forward and backward kernels.
//
// A tile pairs NR "row" tokens (the tokens a thread of the softmax warpgroup
// owns: queries in the forward and dQ kernels, keys in the dK/dV kernel)
// with NC "column" tokens.  Its relative positions are
//     r = base + SIGMA * (row - col),   base = i0 - j0,
// SIGMA = +1 when rows are queries and -1 when rows are keys.
//
// Uniform tiles: every r maps to delta = 0 or every r to delta = R - 1 (the
// clamped far field).  There C2P / P2C collapse to one value per query and
// one per key, taken from the per-token table of df_aux.cu.
//
// Band tiles: the tile reaches at most NR + NC - 1 consecutive relative rows
// [dlo, dlo + NBAND).  Two tensor-core products give every value the tile
// can need:  Town = Rows . Xr[band]^T   (lanes = rows)
//            Tcross = Cols . Yr[band]^T  (lanes = columns)
// (Xr = Kr, Yr = Qr when rows are queries; swapped when rows are keys).  Each
// is copied from tensor memory to shared memory, scaled by c*log2(e) and
// rounded to fp16, and the softmax gathers  Town[row][delta(r) - dlo] +
// Tcross[col][delta(r) - dlo]  per element.  The own window is private to its
// thread; the cross window is shared by the warpgroup.
#pragma once

#include "df_common.cuh"

namespace df {

template <int D_>
struct Geo {
    static constexpr int D = D_;
    static constexpr int BM = 128;                      // rows per tile (TMEM lanes)
    static constexpr int BN = D == 128 ? 64 : 128;      // columns per tile
    static constexpr int CW = D == 32 ? 32 : 64;        // elements per swizzled row chunk
    static constexpr int NCH = D / CW;                  // chunks per head-dim row
    static constexpr uint32_t SWZ = D == 32 ? 4u : 2u;  // descriptor swizzle code (64B / 128B)
    static constexpr int SWZB = CW * 2;                 // TMA swizzle span in bytes
    static constexpr int NBAND = BM + BN - 1 <= 192 ? 192 : 256;
    static constexpr int OWN_S = BN == 64 ? 114 : 178;  // own window stride (halves), >= 16*ceil((BN+46)/16)
    static constexpr int CROSS_S = 176;                                // cross window stride (halves)
};

// Launch order of a sequence's row blocks: the blocks whose key range
// reaches the band on both sides (the most band tiles, the most work) first,
// the w blocks at each end of the sequence last, so that a grid's final,
// partial wave holds the cheapest CTAs.  rank -> row block is a bijection of
// [0, nrb) for any w; w is the band's reach in row blocks (beyond it the
// relative index is clamped): max_relative_positions with log bucketing, else
// att_span.
DF_DEV int row_block_of(const ProblemDev& p, int rank, int nrb, int bm) {
    const int reach = p.nb > 0 ? p.mp : p.span;
    int w = (reach + bm - 1) / bm;
    const int mid = nrb - 2 * w;
    if (w <= 0 || mid <= 0) return rank;
    if (rank < mid) return w + rank;
    const int e = rank - mid;
    return e < w ? e : mid + e;
}

DF_DEV int dclamp(const ProblemDev& p, const int32_t* __restrict__ dtab, int r) {
    r = r > p.L - 1 ? p.L - 1 : r;
    r = r < -(p.L - 1) ? -(p.L - 1) : r;
    return __ldg(dtab + r + p.L - 1);
}

// dclamp for prefetches (the load is issued where the call stands)
DF_DEV int dclamp_early(const ProblemDev& p, const int32_t* __restrict__ dtab, int r) {
    r = r > p.L - 1 ? p.L - 1 : r;
    r = r < -(p.L - 1) ? -(p.L - 1) : r;
    return ld_early(dtab + r + p.L - 1);
}

// K-major operand: `rows` rows of a [rows x D] tile stored as D/CW regions of
// [rows x CW] (TMA swizzle), k-step of 16 elements.
template <class G>
DF_DEV uint64_t desc_k(uint32_t base, int rows, int kstep) {
    constexpr int per = G::CW / 16;
    const int region = kstep / per, within = kstep % per;
    return sdesc(base + (uint32_t)(region * rows * G::CW * 2 + within * 32), 16, 8 * G::CW * 2, G::SWZ);
}

// MN-major B operand: N = head dim (D/CW regions of [rows x CW]), K = rows,
// k-step of 16 rows.
template <class G>
DF_DEV uint64_t desc_mn(uint32_t base, int rows, int kstep) {
    return sdesc(base + (uint32_t)(kstep * 16 * G::CW * 2), (uint32_t)(rows * G::CW * 2), 8 * G::CW * 2, G::SWZ);
}

// Byte offset of k-step `kstep` within a K-major operand of `rows` rows (the
// term desc_k adds to the base address), and within an MN-major one
// (desc_mn).  A descriptor's start-address field holds address >> 4 in 14
// bits and shared-memory addresses stay below 2^18, so adding offset >> 4 to
// the descriptor of k-step 0 gives the descriptor of k-step kstep: the MMA
// issue loops build each operand's descriptor once.
template <class G>
__host__ __device__ constexpr uint32_t kofs(int rows, int kstep) {
    return (uint32_t)((kstep / (G::CW / 16)) * rows * G::CW * 2 + (kstep % (G::CW / 16)) * 32);
}
template <class G>
__host__ __device__ constexpr uint32_t mnofs(int kstep) {
    return (uint32_t)(kstep * 16 * G::CW * 2);
}
DF_DEV uint64_t dadd(uint64_t desc, uint32_t byte_ofs) { return desc + (uint64_t)(byte_ofs >> 4); }

struct TileKind {
    int dlo, dhi;
    int uniform;   // 1: every element has delta == dlo, and dlo is 0 or R-1
    int which;     // uniform tiles: 0 -> delta 0, 1 -> delta R-1
};

// A TileKind in one register (dlo, dhi < R <= 1024), so that the kind of a
// tile can be fetched a few tiles ahead: classify reads the relative-index
// table from global memory, and using its result at once stalls the thread.
DF_DEV uint32_t pack_kind(const TileKind& k) {
    return (uint32_t)k.dlo | ((uint32_t)k.dhi << 14) | ((uint32_t)k.uniform << 28) | ((uint32_t)k.which << 29);
}
DF_DEV TileKind unpack_kind(uint32_t v) {
    TileKind k;
    k.dlo = (int)(v & 0x3FFFu);
    k.dhi = (int)((v >> 14) & 0x3FFFu);
    k.uniform = (int)((v >> 28) & 1u);
    k.which = (int)((v >> 29) & 1u);
    return k;
}

// The two relative indices that decide a tile's kind, as loaded: kind_fetch
// only issues the loads, kind_finish (a tile later) uses them.
struct KindRaw {
    int dlo, dhi;
};

template <int NR, int NC, int SIGMA>
DF_DEV KindRaw kind_fetch(const ProblemDev& p, const int32_t* __restrict__ dtab, int base) {
    const int rlo = SIGMA > 0 ? base - (NC - 1) : base - (NR - 1);
    const int rhi = SIGMA > 0 ? base + (NR - 1) : base + (NC - 1);
    KindRaw r;
    r.dlo = dclamp(p, dtab, rlo);
    r.dhi = dclamp(p, dtab, rhi);
    return r;
}

DF_DEV TileKind kind_finish(const ProblemDev& p, const KindRaw& r) {
    TileKind k;
    k.dlo = r.dlo;
    k.dhi = r.dhi;
    k.uniform = k.dlo == k.dhi && (k.dlo == 0 || k.dlo == p.R - 1);
    k.which = k.dlo == 0 ? 0 : 1;
    return k;
}

template <int NR, int NC, int SIGMA>
DF_DEV TileKind classify(const ProblemDev& p, const int32_t* __restrict__ dtab, int base) {
    return kind_finish(p, kind_fetch<NR, NC, SIGMA>(p, dtab, base));
}

// dwin[x] = delta(r) - dlo for the tile, x = SIGMA*(row - col) + (SIGMA > 0 ? NC - 1 : NR - 1),
// i.e. r = base + x - (SIGMA > 0 ? NC - 1 : NR - 1); thread x fills entry x (band_fetch).

// The relative indices a band tile needs, as loaded from the table, for one
// softmax thread: its entry of the tile's index window (thread tid < NR + NC
// - 1) and, in lanes 0-3, one end each of the own and cross windows of its
// lane quarter (lane 0 own low, 1 own high, 2 cross low, 3 cross high; the
// warp reads them with shuffles).  The kernels fetch them one tile ahead and
// use them when the tile comes, so no band tile waits on the table.
struct BandRaw {
    int dw, dwp, rng;
};

// STEPS: also the index one position back (for the step bits)
template <int NR, int NC, int SIGMA, bool STEPS = false>
DF_DEV BandRaw band_fetch(const ProblemDev& p, const int32_t* __restrict__ dtab, int base, int w, int tid,
                          int lane) {
    BandRaw r;
    const int x = tid < NR + NC - 1 ? tid : 0;
    r.dw = dclamp_early(p, dtab, base + x - (SIGMA > 0 ? NC - 1 : NR - 1));
    r.dwp = STEPS ? dclamp_early(p, dtab, base + x - 1 - (SIGMA > 0 ? NC - 1 : NR - 1)) : 0;
    // own window of rows [32w, 32w + 32), cross window of columns [32w, 32w + 32)
    const int k = lane & 3;
    const int rel = SIGMA > 0 ? (k == 0   ? base + 32 * w - (NC - 1)
                                 : k == 1 ? base + 32 * w + 31
                                 : k == 2 ? base - (32 * w + 31)
                                          : base + (NR - 1) - 32 * w)
                              : (k == 0   ? base - (32 * w + 31)
                                 : k == 1 ? base - 32 * w + (NC - 1)
                                 : k == 2 ? base + 32 * w - (NR - 1)
                                          : base + 32 * w + 31);
    r.rng = dclamp_early(p, dtab, rel);
    return r;
}

// Step bits of a band tile's index window: bit x of `stepw` (9 words) is set
// where the window's relative index changes between positions x - 1 and x.
// The index moves by at most one per position (the host checks the bucketing
// for 16-bit inputs), so the indices along a row follow from the first one
// and these bits: one shared-memory load per 32 columns instead of 32.  All
// 256 softmax threads call this (thread x holds the index at x and x - 1).
DF_DEV void put_step_bits(uint32_t* stepw, const BandRaw& b, int tid, int lane, int nx) {
    const unsigned bits = __ballot_sync(0xffffffffu, tid > 0 && tid < nx && b.dw != b.dwp);
    if (lane == 0) stepw[tid >> 5] = bits;
    if (tid == 0) stepw[8] = 0u;
}

// 32 step bits from position xl on (bit k: step at position xl + k), 0 <= xl <= 224
DF_DEV uint32_t step_bits(const uint32_t* stepw, int xl) {
    return __funnelshift_r(stepw[xl >> 5], stepw[(xl >> 5) + 1], (uint32_t)(xl & 31));
}

// Copy the columns of a band product that a lane quarter needs (`lo` ..
// `hi`, band coordinates) from tensor memory to the thread's shared-memory
// row, scaled to base-2 exponent units and rounded to fp16.  The window is cut
// into 16-column chunks; the warp copies chunks part, part + nparts, ... (the
// two warps of a lane quarter share the work).  Returns the band coordinate
// of dst[0] (warp-uniform, a multiple of 16).
DF_DEV int copy_band_window(uint32_t t_lane_col0, int lo, int hi, uint16_t* dst, float scale, int part = 0,
                            int nparts = 1) {
    const int a = lo & ~15;
    const int nch = ((hi - a) >> 4) + 1;
    for (int c = part; c < nch; c += 2 * nparts) {
        // two chunks per tensor-memory round trip
        const bool two = c + nparts < nch;
        uint32_t r[32];
        tc_ld16p(t_lane_col0 + (uint32_t)(a + 16 * c), r);
        if (two) tc_ld16p(t_lane_col0 + (uint32_t)(a + 16 * (c + nparts)), r + 16);
        tc_wait_ld();
        uint32_t* d32 = reinterpret_cast<uint32_t*>(dst + 16 * c);
#pragma unroll
        for (int x = 0; x < 8; ++x)
            d32[x] = pack2<false>(__uint_as_float(r[2 * x]) * scale, __uint_as_float(r[2 * x + 1]) * scale);
        if (two) {
            uint32_t* e32 = reinterpret_cast<uint32_t*>(dst + 16 * (c + nparts));
#pragma unroll
            for (int x = 0; x < 8; ++x)
                e32[x] = pack2<false>(__uint_as_float(r[16 + 2 * x]) * scale,
                                      __uint_as_float(r[16 + 2 * x + 1]) * scale);
        }
    }
    return a;
}

// Band products computed in chunks of 64 band positions: copy the part of
// the chunk at band coordinates [kb, kb + 64) (tensor-memory columns t_chunk
// .. + 63 of the warp's lanes) that the lane quarter's window [lo, hi]
// covers, scaled and rounded as in copy_band_window, to dst[x - a] for band
// coordinate x (a = lo & ~15, so the 16-column parts land where
// copy_band_window puts them).  The chunk's four 16-column parts go to the
// quarter's two warps alternately (part 0 / 1): one tensor-memory round trip
// per warp.
// (stride: the destination row's length in halves, for a checked build's
// range check; err: the error word)
DF_DEV void copy_band_chunk(uint32_t t_chunk, int kb, int lo, int hi, int a, uint16_t* dst, float scale, int part,
                            int stride, int* err) {
    if (hi < kb || lo >= kb + 64) return;
    const int s = (lo > kb ? (lo - kb) >> 4 : 0) + part;
    const int s_hi = hi < kb + 63 ? (hi - kb) >> 4 : 3;
    if (s > s_hi) return;
    const bool two = s + 2 <= s_hi;
    uint32_t r[32];
    tc_ld16p(t_chunk + (uint32_t)(16 * s), r);
    if (two) tc_ld16p(t_chunk + (uint32_t)(16 * (s + 2)), r + 16);
    tc_wait_ld();
    int off = kb + 16 * s - a;   // the parts written: [off, off + 16) and, if two, [off + 32, off + 48)
    DF_CLAMP_CHECK(off, 0, stride - (two ? 47 : 15), err);
    uint32_t* d32 = reinterpret_cast<uint32_t*>(dst + off);
#pragma unroll
    for (int x = 0; x < 8; ++x)
        d32[x] = pack2<false>(__uint_as_float(r[2 * x]) * scale, __uint_as_float(r[2 * x + 1]) * scale);
    if (two) {
#pragma unroll
        for (int x = 0; x < 8; ++x)
            d32[16 + x] = pack2<false>(__uint_as_float(r[16 + 2 * x]) * scale,
                                       __uint_as_float(r[16 + 2 * x + 1]) * scale);
    }
}

// ---- stored band bias (written by df_bias.cu, read by the backward kernels)
//
// The bias of a band tile, c log2(e) (Q_i . Kr[delta] + K_j . Qr[delta]),
// kept per 128 x 128 block of (query, key) pairs of one sequence: query block
// qt, key block kt.  Only blocks near the diagonal can be band blocks; the
// table keeps 2 bias_kb + 1 key blocks per query block (slot = kt - qt +
// bias_kb), fp16, [block][128 query rows][128 key columns].
constexpr int kBiasBB = 128;

// floor(t0 / 128) + qt + b differs for every (sequence, query block) pair
// and stays below (T - 1) / 128 + B + 1: the table's query-block rows.
DF_DEV int bias_rbg(int t0, int qt, int b) { return t0 / kBiasBB + qt + b; }

// First row of block (qt, kt) of (b, h) in the table viewed as [rows x 128]
// halves, or -1 when kt is outside the kept band of key blocks.
DF_DEV int bias_block_row(const ProblemDev& p, int b, int h, int t0, int qt, int kt) {
    const int slot = kt - qt + p.bias_kb;
    if (slot < 0 || slot >= p.bias_nslot) return -1;
    return ((bias_rbg(t0, qt, b) * p.H + h) * p.bias_nslot + slot) * kBiasBB;
}

// 16-byte chunk c (eight halves) of block row r sits at chunk
// (c & 8) | ((c ^ r) & 7): a warp reading one logical chunk of 32
// consecutive rows touches every bank, and each 64-column half of a row stays
// in its own half.
DF_DEV int bias_chunk(int r, int c) { return (c & 8) | ((c ^ r) & 7); }

DF_DEV float h2f(uint16_t h) {
    float f;
    asm("{ .reg .f16 t; mov.b16 t, %1; cvt.f32.f16 %0, t; }" : "=f"(f) : "h"(h));
    return f;
}

// The band bias of a pair as every kernel uses it: the own and cross window
// values (fp16) summed and rounded to fp16 once more, so that the forward
// and the stored bias of the backward give the same logits.  band_bias2 does
// two pairs with one f16x2 addition: the sum of two fp16 values is exact in
// fp32 unless their exponents differ by more than 13, and then the smaller
// one is below a quarter of the larger one's fp16 spacing, so rounding the
// fp32 sum to fp16 and rounding the exact sum to fp16 (add.rn.f16x2) both
// give the larger value: the two forms agree bit for bit.
DF_DEV uint32_t band_bias2(uint32_t own_v2, uint32_t cross_v2) {
    uint32_t d;
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(own_v2), "r"(cross_v2));
    return d;
}

// both halves of an f16x2 word as fp32 (low half first)
DF_DEV void h2x2f(uint32_t h, float& lo, float& hi) {
    asm("{\n\t.reg .f16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(h));
}

}  // namespace df
