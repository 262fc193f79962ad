"""CPU model of the tensor-core kernels' band-tile index arithmetic
(csrc/df_tile.cuh: classify, band_fetch (the index window and the own /
cross window ends), copy_band_window; csrc/df_bwd_kernel.cuh: the
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

