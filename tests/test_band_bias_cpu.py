"""Host-side rules of the stored band bias (no GPU needed).

The backward reads the band bias from a table that keeps, for every
128-query block, the key blocks kt with |kt - qt| <= KB.  Every 128 x 128
block whose relative index is not constant at 0 or R-1 (a band block: its
pairs have their own relative-position values) must lie inside that reach,
or the kernels would flag DF_ERR_DEVICE_ARG.  KB is read back from
df_attn_band_bias_size and checked against the band blocks found by brute
force over the oracle's relative-index table (the definition of delta,
written out independently of the library), for the workloads' bucketing and
for no bucketing, a small span and the largest span.  The library keeps one
block of margin beyond the exact reach.

Also: the size is 0 for strict fp32, a backward given a saved buffer needs
exactly that much less workspace, and a misaligned buffer is rejected.  And
the rounding rule the forward relies on when it adds the own and cross
values of two pairs with one f16x2 addition: rounding the fp32 sum of two
fp16 values to fp16 equals rounding their exact sum to fp16.
"""
import numpy as np
import pytest
import torch

import __graft_entry__
from exact_deberta_disentangled_gb300 import binding as B
from oracle import oracle


@pytest.fixture(scope="module", autouse=True)
def _built():
    __graft_entry__.build()


class Fake:
    def __init__(self, addr):
        self.addr = addr

    def data_ptr(self):
        return self.addr


def geom(**kw):
    base = dict(B=2, L=8192, H=12, D=64, span=256, nb=256, mp=512)
    base.update(kw)
    return B.Geometry(**base)


def table_reach(g) -> int:
    """KB from the table size: (T - 1) // 128 + B + 1 query-block rows per
    head, 2 KB + 1 blocks of 128 x 128 halves each."""
    n = B.band_bias_size(g, torch.bfloat16)
    per_slot = ((g.T - 1) // 128 + g.B + 1) * g.H * 128 * 128 * 2
    assert n > 0 and n % per_slot == 0
    nslot = n // per_slot
    assert nslot % 2 == 1
    return (nslot - 1) // 2


def brute_reach(L, span, nb, mp) -> int:
    d = oracle.delta_table(L, span, nb, mp)   # index r + L - 1
    R, nrb = 2 * span, (L + 127) // 128
    reach = 0
    for k in range(-(nrb - 1), nrb):
        lo, hi = max(128 * k - 127, -(L - 1)), min(128 * k + 127, L - 1)
        v = d[lo + L - 1: hi + L]
        if not (v.min() == v.max() and v[0] in (0, R - 1)):
            reach = max(reach, abs(k))
    return reach


@pytest.mark.parametrize("L,span,nb,mp", [
    (8192, 256, 256, 512),     # the workloads (DeBERTa-v3 settings)
    (512, 256, 256, 512),
    (3000, 256, 256, 512),
    (2048, 64, 0, 0),          # no bucketing: clamped beyond the span
    (4096, 32, 64, 128),       # small span and buckets
    (8192, 512, 512, 1024),    # the largest span
    (1000, 512, 256, 512),     # span above the bucket range: never clamped on this length
])
def test_table_reach_covers_every_band_block(L, span, nb, mp):
    g = geom(L=L, span=span, nb=nb, mp=mp)
    kb, exact = table_reach(g), brute_reach(L, span, nb, mp)
    nrb = (L + 127) // 128
    assert exact <= kb <= min(exact + 1, nrb - 1)


def test_sizes_and_workspace():
    g = geom(L=1024)
    n = B.band_bias_size(g, torch.bfloat16)
    assert n == B.band_bias_size(g, torch.float16) > 0
    assert B.band_bias_size(g, torch.float32) == 0
    full = B.workspace_size(g, torch.bfloat16, True)
    g.band_bias = Fake(0x10000)
    assert B.workspace_size(g, torch.bfloat16, True) == full - n
    assert B.workspace_size(g, torch.bfloat16, False) == B.workspace_size(geom(L=1024), torch.bfloat16, False)
    # strict fp32 ignores the buffer
    assert B.workspace_size(g, torch.float32, True) == B.workspace_size(geom(L=1024), torch.float32, True)


def test_misaligned_buffer_is_invalid():
    g = geom(L=1024)
    g.band_bias = Fake(0x10008)
    assert B.workspace_size(g, torch.bfloat16, True) == 0
    assert B.band_bias_size(g, torch.bfloat16) == 0


def test_fp16_sum_rounding_through_fp32_is_exact_rounding():
    """rn16(rn32(a + b)) == rn16(a + b) for fp16 a, b: every finite pair whose
    exponents are within 13 of each other (the sum is exact in fp32), every
    pair 14 or more apart (the small one is below a quarter spacing), ties,
    subnormals and a dense random sample.  The exact sum is taken in fp64,
    where every sum of two fp16 values is exact."""
    # the fp64 -> fp16 conversion used as the reference rounds directly (a
    # value just above a tie rounds up; through fp32 it would round to even)
    assert np.float16(np.float64(1 + 2.0 ** -11 + 2.0 ** -40)) == np.float16(1 + 2.0 ** -10)
    rng = np.random.default_rng(7)
    allh = np.arange(0, 1 << 16, dtype=np.uint16).view(np.float16)
    finite = allh[np.isfinite(allh)]
    # every finite fp16 against a spread of partners: powers of two, values just
    # off them, subnormals, the largest values, and random ones
    partners = np.concatenate([
        np.float16(2.0) ** np.arange(-24, 16, dtype=np.float64),
        np.nextafter(np.float16(2.0) ** np.arange(-14, 16, dtype=np.float64), np.float16(0)).astype(np.float16),
        allh[1:64], -allh[1:64], np.array([65504.0, -65504.0, 0.5, -0.5, 1.0, -1.0]),
        rng.choice(finite, 400)]).astype(np.float16)
    a = np.repeat(finite, partners.size)
    b = np.tile(partners, finite.size)
    extra = rng.choice(finite, (2, 4_000_000))
    a = np.concatenate([a, extra[0]])
    b = np.concatenate([b, extra[1]])
    exact = (a.astype(np.float64) + b.astype(np.float64)).astype(np.float16)
    via32 = (a.astype(np.float32) + b.astype(np.float32)).astype(np.float16)
    same = (exact.view(np.uint16) == via32.view(np.uint16)) | (np.isnan(exact) & np.isnan(via32))
    assert same.all(), (a[~same][:5], b[~same][:5])
