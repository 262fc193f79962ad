"""CPU model of the tensor-core kernels' band-tile index arithmetic
(csrc/df_tile.cuh: classify, band_fetch (the index window and the own /
cross window ends), copy_band_window, the step bits that give the gathers'
and the scatter's relative indices; csrc/df_bwd_kernel.cuh: the
per-quarter diagonal-sum staging boxes).  For every tile
of the workloads' shapes it checks that each gathered relative index lies in
the window the warp copied out of tensor memory, that the copied columns stay
inside the band product, and that each staged diagonal sum lands inside its
shared-memory box -- so no kernel can read or write outside its buffers."""
import numpy as np
import pytest

from oracle import oracle

BM = 128


def geo(D):
    BN = 64 if D == 128 else 128
    nband = 192 if BM + BN - 1 <= 192 else 256
    own_s = 114 if BN == 64 else 178
    cross_s = 176
    qw = (BN + 38 + 7) // 8 * 8           # staging box row width (16-bit sums)
    return BN, nband, own_s, cross_s, qw


def step_words(dwin):
    """The nine 32-bit words put_step_bits writes (256 threads, thread x = position x)."""
    nx = len(dwin)
    bits = np.zeros(9 * 32, dtype=np.uint64)
    for x in range(1, nx):
        bits[x] = 1 if dwin[x] != dwin[x - 1] else 0
    return [int(sum(int(bits[32 * w + k]) << k for k in range(32))) for w in range(9)]


def step_bits(words, xl):
    """step_bits: 32 bits from position xl on (funnel shift of two words)."""
    assert 0 <= xl <= 224
    v = words[xl >> 5] | (words[(xl >> 5) + 1] << 32)
    return (v >> (xl & 31)) & 0xFFFFFFFF


def check_step_bits(dwin, sigma, NR, NC):
    steps = np.diff(dwin)
    assert steps.min() >= 0 and steps.max() <= 1       # the host's bucketing check guarantees it
    words = step_words(dwin)
    # gathers: rows x 32-column chunks
    for row in range(NR):
        for c in range(NC // 32):
            x0 = row - 32 * c + NC - 1 if sigma > 0 else 32 * c - row + NR - 1
            mk = step_bits(words, x0 - 31 if sigma > 0 else x0 + 1)
            m = int(dwin[x0])
            for e in range(32):
                x = x0 - e if sigma > 0 else x0 + e
                assert m == dwin[x], (row, c, e)
                if sigma > 0:
                    m -= (mk >> (31 - e)) & 1
                else:
                    m += (mk >> e) & 1
    # scatter: each column half, 32-column groups; a run ends at a step bit
    HC = NC // 2
    for row in range(NR):
        for hf in range(2):
            cst = hf * HC
            x0 = row - cst + NC - 1 if sigma > 0 else cst - row + NR - 1
            for g in range(HC // 32):
                mk = step_bits(words, x0 - 32 * g - 31 if sigma > 0 else x0 + 32 * g + 1)
                for e2 in range(32):
                    e = 32 * g + e2
                    if e + 1 >= HC:
                        continue
                    xa = x0 - e if sigma > 0 else x0 + e
                    xb = x0 - e - 1 if sigma > 0 else x0 + e + 1
                    bit = (mk >> (31 - e2)) & 1 if sigma > 0 else (mk >> e2) & 1
                    assert bit == (1 if dwin[xa] != dwin[xb] else 0), (row, hf, e)


def check_kernel(L, span, nb, mp, D, sigma, n=None):
    """All (row tile, column tile) pairs of one sequence of length n <= L."""
    n = L if n is None else n
    BN, NBAND, OWN_S, CROSS_S, QW = geo(D)
    NR, NC = BM, BN
    R = 2 * span
    tab = oracle.delta_table(L, span, nb, mp)

    def dcl(r):
        r = np.clip(r, -(L - 1), L - 1)
        return tab[r + L - 1]

    OFF = NC - 1 if sigma > 0 else NR - 1
    rows = np.arange(NR)[:, None]
    cols = np.arange(NC)[None, :]
    xidx = sigma * (rows - cols) + OFF                       # dwin index of every element
    assert xidx.min() >= 0 and xidx.max() < NR + NC - 1
    nband_tiles = 0
    for r0 in range(0, n, BM):
        for c0 in range(0, n, BN):
            base = r0 - c0 if sigma > 0 else c0 - r0
            rlo = base - (NC - 1) if sigma > 0 else base - (NR - 1)
            rhi = base + (NR - 1) if sigma > 0 else base + (NC - 1)
            dlo, dhi = int(dcl(rlo)), int(dcl(rhi))
            if dlo == dhi and dlo in (0, R - 1):
                continue
            nband_tiles += 1
            assert 0 <= dhi - dlo < NBAND
            x = np.arange(NR + NC - 1)
            dwin = dcl(base + x - OFF) - dlo                 # band_fetch: index window
            assert dwin.min() >= 0 and dwin.max() < NBAND
            m = dwin[xidx]                                   # [NR, NC] gathered band index
            # exact relative index of each element equals the table's value
            assert np.array_equal(m + dlo, dcl(base + sigma * (rows - cols)))
            for w in range(4):
                rmin = base + 32 * w - (NC - 1) if sigma > 0 else base - (32 * w + 31)
                rmax = base + 32 * w + 31 if sigma > 0 else base - 32 * w + (NC - 1)
                lo, hi = int(dcl(rmin)) - dlo, int(dcl(rmax)) - dlo
                a = lo & ~15
                nch = ((hi - a) >> 4) + 1
                assert a >= 0 and a + 16 * nch <= NBAND and 16 * nch <= OWN_S
                mw = m[32 * w:32 * w + 32]
                assert mw.min() >= lo and mw.max() <= hi
            for u in range(4):
                if 32 * u >= NC:
                    continue
                rmin = base - (32 * u + 31) if sigma > 0 else base + 32 * u - (NR - 1)
                rmax = base + (NR - 1) - 32 * u if sigma > 0 else base + 32 * u + 31
                lo, hi = int(dcl(rmin)) - dlo, int(dcl(rmax)) - dlo
                a = lo & ~15
                nch = ((hi - a) >> 4) + 1
                assert a >= 0 and a + 16 * nch <= NBAND and 16 * nch <= CROSS_S
                mu = m[:, 32 * u:32 * u + 32]
                assert mu.min() >= lo and mu.max() <= hi
            # step bits (put_step_bits / step_bits): bit x set where the window
            # index changes between x - 1 and x; the gathers and the scatter
            # derive every index of a 32-column chunk from its first entry
            if nband_tiles <= 3:   # (pure-Python loops: a few tiles per case)
                check_step_bits(dwin, sigma, NR, NC)
            # backward: staged diagonal sums, one box per quarter of 32 rows
            # (32 rows of QW sums from the quarter's lowest relative row rounded
            # down to 8, which the kernel reads at two corners of the index
            # window), and the far-field entries
            assert QW % 8 == 0 and QW // 8 <= 256
            for w in range(4):
                xa = 32 * w if sigma > 0 else NR - 32 - 32 * w
                xb = xa + NC + 30
                mq = m[32 * w:32 * w + 32]
                qmin, qmax = min(dwin[xa], dwin[xb]), max(dwin[xa], dwin[xb])
                assert mq.min() == qmin and mq.max() == qmax
                qa0 = (dlo + qmin) & ~7
                qoff = dlo - qa0
                slots = mq + qoff
                assert slots.min() >= 0 and slots.max() < QW
                for far in (0, R - 1):
                    if dlo <= far <= dhi and mq.min() <= far - dlo <= mq.max():
                        assert 0 <= far - dlo + qoff < QW
    return nband_tiles


CASES = [
    # (L, span, nb, mp, D)
    (8192, 256, 256, 512, 64), (4096, 256, 256, 512, 64), (2048, 256, 256, 512, 64), (1024, 256, 256, 512, 64),
    (512, 256, 256, 512, 64), (128, 64, 64, 128, 64), (4096, 256, 256, 512, 128), (2048, 256, 256, 512, 32),
    (600, 256, 256, 512, 128), (520, 256, 256, 512, 32), (1536, 256, 256, 512, 64), (333, 17, 12, 100, 64),
    (2048, 256, 0, 0, 64), (1000, 8, 4, 8, 128),
    # shapes of the edge-case parity tests
    (1, 256, 256, 512, 64), (7, 256, 256, 512, 64), (130, 256, 256, 512, 64), (700, 256, 0, 0, 64),
    (600, 8, 4, 8, 64), (1500, 512, 512, 1024, 64), (2048, 512, 512, 1024, 128), (2048, 512, 512, 1024, 32),
]


@pytest.mark.parametrize("L,span,nb,mp,D", CASES)
@pytest.mark.parametrize("sigma", [1, -1])
def test_band_tile_indices_stay_in_their_buffers(L, span, nb, mp, D, sigma):
    nt = check_kernel(L, span, nb, mp, D, sigma)
    assert nt > 0
    # a shorter sequence of the same packed batch (table built for L)
    check_kernel(L, span, nb, mp, D, sigma, n=max(1, L // 3 + 17))


def test_model_catches_a_flipped_relative_index():
    """The model itself rejects the sign error it was written to catch."""
    import tests.test_tile_indexing_cpu as mod
    L, span, nb, mp, D = 1536, 256, 256, 512, 64
    BN = geo(D)[0]
    tab = oracle.delta_table(L, span, nb, mp)
    base, NR = 0 - 512, BM
    x = np.arange(NR + BN - 1)
    good = tab[np.clip(base + x - (NR - 1), -(L - 1), L - 1) + L - 1]
    bad = tab[np.clip(base - (x - (NR - 1)), -(L - 1), L - 1) + L - 1]
    assert not np.array_equal(good, bad)



def row_block_of(rank, nrb, bm, nb, mp, span):
    """Model of row_block_of (csrc/df_tile.cuh): the backward kernels' launch
    order of a sequence's row blocks."""
    reach = mp if nb > 0 else span
    w = (reach + bm - 1) // bm
    mid = nrb - 2 * w
    if w <= 0 or mid <= 0:
        return rank
    if rank < mid:
        return w + rank
    e = rank - mid
    return e if e < w else mid + e


@pytest.mark.parametrize("nb,mp,span", [(256, 512, 256), (0, 0, 256), (4, 8, 8), (512, 1024, 512), (12, 100, 17)])
def test_row_block_launch_order_is_a_permutation(nb, mp, span):
    """Every row block of every sequence length is launched exactly once, the
    blocks within the band's reach of either end last."""
    for nrb in range(1, 65):
        order = [row_block_of(r, nrb, BM, nb, mp, span) for r in range(nrb)]
        assert sorted(order) == list(range(nrb))
        w = ((mp if nb > 0 else span) + BM - 1) // BM
        if nrb > 2 * w:
            assert order[:nrb - 2 * w] == list(range(w, nrb - w))
