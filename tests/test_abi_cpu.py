"""Host-side checks of the C ABI that need no GPU: the library builds and
exports every symbol its header declares, and argument validation returns
the documented status codes before anything is enqueued."""
import ctypes
import os
import re

import pytest

import __graft_entry__
from exact_deberta_disentangled_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "df_attn.h")


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    return B.load()


def header_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(df_[a-z_0-9]+)\s*\(", src)))


def test_header_symbols_are_exported(lib):
    names = header_functions()
    assert "df_attn_fwd" in names and "df_attn_bwd" in names
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) <= set(B.EXPORTS) | set(names)


def test_status_strings(lib):
    for code in range(7):
        s = B.status_string(code)
        assert s.startswith("DF_")
    assert lib.df_version().decode().count(".") == 2


def geom(**kw):
    base = dict(B=2, L=512, H=12, D=64, span=256, nb=256, mp=512)
    base.update(kw)
    return B.Geometry(**base)


def test_workspace_sizes(lib):
    import torch
    f = B.workspace_size(geom(), torch.bfloat16, False)
    b = B.workspace_size(geom(), torch.bfloat16, True)
    assert 0 < f < b
    assert B.workspace_size(geom(D=48), torch.bfloat16, False) == 0
    assert B.workspace_size(geom(L=8193), torch.bfloat16, False) == 0
    assert B.workspace_size(geom(span=0), torch.bfloat16, False) == 0
    # backward scratch holds the two [T, H, R] diagonal-sum buffers
    T, H, R = 2 * 512, 12, 512
    assert b - f >= 2 * 2 * T * H * R


def test_fast_fp32_workspace_and_rules(lib):
    """The fast fp32 mode (fp32 tensors through the fp16 tensor-core path):
    its workspace is the fp16 one plus fp16 copies of the inputs and outputs
    (forward: Q, K, V, O and Qr, Kr; backward also dO, dQ, dK, dV and dQr,
    dKr), its saved band bias is the fp16 one, and the 16-bit kernels'
    bucketing rule applies to it."""
    import torch
    al = lambda x: (x + 255) // 256 * 256
    for kw in ({}, dict(D=32, L=384, span=64, nb=64, mp=128), dict(D=128, B=3, L=700, span=512, nb=0, mp=0)):
        g, gf = geom(**kw), geom(fp32_fast=True, **kw)
        T, H, D, R = g.T, g.H, g.D, g.R
        tok, rel = al(2 * T * H * D), al(2 * H * R * D)
        for bwd, ntok, nrel in ((False, 4, 2), (True, 8, 4)):
            w16 = B.workspace_size(g, torch.float16, bwd)
            assert w16 > 0
            assert B.workspace_size(gf, torch.float32, bwd) == w16 + ntok * tok + nrel * rel
        assert B.band_bias_size(gf, torch.float32) == B.band_bias_size(g, torch.float16) > 0
        assert B.band_bias_size(g, torch.float32) == 0          # strict fp32 stores none
    # a bucketing configuration the 16-bit kernels reject (the index jumps by 2)
    bad = dict(nb=256, mp=300)
    assert B.workspace_size(geom(fp32_fast=True, **bad), torch.float32, True) == 0
    assert B.workspace_size(geom(**bad), torch.float32, True) > 0


class FakeTensor:
    """An aligned non-null address that is never dereferenced (validation
    fails before any device work)."""

    def __init__(self, addr=0x10000):
        self.addr = addr

    def data_ptr(self):
        return self.addr


def call_fwd(g, dtype_code=0, ws_bytes=1 << 30, ptr=0x10000, ws_ptr=0x20000):
    import torch
    lib = B.load()
    p = g.params(torch.bfloat16)
    p.dtype = dtype_code
    vp = [ctypes.c_void_p(ptr)] * 7
    return lib.df_attn_fwd(ctypes.byref(p), *vp, ctypes.c_void_p(ws_ptr), ws_bytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(D=48), B.DF_ERR_UNSUPPORTED),
    (dict(D=256), B.DF_ERR_UNSUPPORTED),
    (dict(L=8193), B.DF_ERR_UNSUPPORTED),
    (dict(span=600), B.DF_ERR_UNSUPPORTED),
    (dict(nb=256, mp=100), B.DF_ERR_UNSUPPORTED),
    (dict(nb=256, mp=300), B.DF_ERR_UNSUPPORTED),   # bucket steps of two (16-bit path)
    (dict(B=0), B.DF_ERR_INVALID_ARG),
    (dict(H=0), B.DF_ERR_INVALID_ARG),
    (dict(span=0), B.DF_ERR_INVALID_ARG),
    (dict(dropout_p=1.0), B.DF_ERR_INVALID_ARG),
    (dict(dropout_p=-0.1), B.DF_ERR_INVALID_ARG),
    (dict(offset=1 << 32), B.DF_ERR_INVALID_ARG),
    (dict(scale=-1.0), B.DF_ERR_INVALID_ARG),
])
def test_validation_codes(lib, kw, code):
    assert call_fwd(geom(**kw)) == code


def test_pointer_and_workspace_checks(lib):
    g = geom()
    assert call_fwd(g, ptr=0) == B.DF_ERR_INVALID_ARG           # null tensor
    assert call_fwd(g, ptr=0x10008) == B.DF_ERR_INVALID_ARG     # not 16-byte aligned
    assert call_fwd(g, ws_bytes=1024) == B.DF_ERR_WORKSPACE      # too small
    assert call_fwd(g, ws_ptr=0) == B.DF_ERR_WORKSPACE           # missing
    assert call_fwd(g, dtype_code=7) == B.DF_ERR_INVALID_ARG     # unknown dtype


def test_packed_layout_rules(lib):
    g = geom(cu_seqlens=FakeTensor(), total_tokens=600)
    g.query_mask = FakeTensor()
    assert call_fwd(g) == B.DF_ERR_UNSUPPORTED                  # masks only in the padded layout
    g = geom(cu_seqlens=FakeTensor(), total_tokens=0)
    assert call_fwd(g) == B.DF_ERR_INVALID_ARG
    g = geom(cu_seqlens=FakeTensor(), total_tokens=2 * 512 + 1)
    assert call_fwd(g) == B.DF_ERR_INVALID_ARG                  # more tokens than B*L


@pytest.mark.parametrize("nb", [4, 12, 64, 256, 512])
def test_bucket_step_rule_matches_the_relative_index_table(lib, nb):
    """The 16-bit kernels accept a bucketing configuration exactly when the
    oracle's relative-index table moves by at most one per relative position
    (the property their band windows are sized for); fp32 accepts all."""
    import numpy as np
    import torch

    from oracle import oracle
    span = max(nb, 8)
    for mp in range(nb // 2 + 2, 4 * nb + 2, max(1, nb // 16)):
        tab = oracle.delta_table(2048, span, nb, mp)
        unit = int(np.abs(np.diff(tab)).max()) <= 1
        g = geom(nb=nb, mp=mp, span=span, L=2048)
        assert (B.workspace_size(g, torch.bfloat16, True) > 0) == unit, (nb, mp)
        assert B.workspace_size(g, torch.float32, True) > 0


def test_packing_validation_codes(lib):
    """df_pack_info / df_pack_rows / df_unpack_rows check their arguments on
    the host and return a status before any device work."""
    vp = ctypes.c_void_p
    a, w = vp(0x10000), vp(0x20000)
    assert lib.df_pack_workspace_size(0) == 0 and lib.df_pack_workspace_size(5) >= 40
    assert lib.df_pack_info(a, 0, 8, a, a, a, w, 1 << 20, None) == B.DF_ERR_INVALID_ARG
    assert lib.df_pack_info(a, 2, 0, a, a, a, w, 1 << 20, None) == B.DF_ERR_INVALID_ARG
    assert lib.df_pack_info(None, 2, 8, a, a, a, w, 1 << 20, None) == B.DF_ERR_INVALID_ARG
    assert lib.df_pack_info(a, 2, 8, a, a, a, None, 0, None) == B.DF_ERR_WORKSPACE
    assert lib.df_pack_info(a, 2, 8, a, a, a, w, 4, None) == B.DF_ERR_WORKSPACE
    assert lib.df_pack_info(a, 1 << 16, 1 << 16, a, a, a, w, 1 << 30, None) == B.DF_ERR_UNSUPPORTED
    assert lib.df_pack_rows(a, 16, a, a, 16, 24, a, None) == B.DF_ERR_INVALID_ARG        # 24-byte rows
    assert lib.df_pack_rows(vp(0x10008), 16, a, a, 16, 32, a, None) == B.DF_ERR_INVALID_ARG   # unaligned
    assert lib.df_pack_rows(a, 16, a, a, 0, 32, a, None) == B.DF_ERR_INVALID_ARG
    assert lib.df_unpack_rows(a, a, a, 16, 32, 0, a, None) == B.DF_ERR_INVALID_ARG
    assert lib.df_unpack_rows(a, None, a, 16, 32, 16, a, None) == B.DF_ERR_INVALID_ARG
