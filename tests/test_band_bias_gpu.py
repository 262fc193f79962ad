"""The saved band bias on the GPU.

Near the diagonal every (query, key) pair has its own relative-position term
("DisentangledFlash", section "Status": C2P and P2C).  The backward reads it
from a table of 128 x 128 fp16 blocks that either the training forward saved
(df_attn_params.band_bias) or the backward's own bias kernel computed.  Both
compute each value the same way (the two band products, fp16 windows, the
sum rounded to fp16), so the backward must give bit-identical gradients
either way, for every head dim (D = 128 also covers the 64-wide forward
tiles, which save whole blocks), for padding masks, packed sequences and
dropout.  The saved path is also checked against the fp64 oracle at the
workload bars.
"""
import pytest
import torch

from exact_deberta_disentangled_gb300 import binding as B
from exact_deberta_disentangled_gb300 import synth
from tests.test_parity_tc_gpu import check_against_oracle, geometry

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


CASES = {
    "v3_base": dict(w="v3_base", B=3, L=640, H=2),
    "long": dict(w="sweep_L8192", B=1, L=1536, H=2),
    "hd128": dict(w="hd128_dropout", B=1, L=900, H=2),
    "hd32": dict(w="hd32_dropout", B=2, L=700, H=2),
    "varlen": dict(w="varlen", H=2, total_tokens=2500),
    "fp16": dict(w="mnli_fp16", B=3, L=512, H=3),
}


def inputs(name):
    kw = dict(CASES[name])
    w = synth.WORKLOADS[kw.pop("w")]
    return w, synth.make_inputs(w, **kw)


@pytest.mark.parametrize("name", list(CASES))
def test_saved_and_recomputed_bias_give_identical_gradients(name):
    w, x = inputs(name)
    H = x.q.shape[1]
    g = geometry(x, w, H, p_drop=w.dropout_p, seed=3, offset=8)
    t = [a.to("cuda") for a in (x.q, x.k, x.v, x.qr, x.kr, x.dout)]
    g.band_bias = B.alloc_band_bias(g, t[0].dtype)
    assert g.band_bias.numel() == B.band_bias_size(g, t[0].dtype)
    out, lse, wsf = B.attn_fwd(g, *t[:5])
    saved, wsb1 = B.attn_bwd(g, *t[:5], out, lse, t[5])
    bias = g.band_bias
    g.band_bias = None   # the backward computes the table itself
    recomputed, wsb2 = B.attn_bwd(g, *t[:5], out, lse, t[5])
    torch.cuda.synchronize()
    for ws in (wsf, wsb1, wsb2):
        assert B.device_error(ws) == B.DF_OK
    for nm, a, b in zip(("dq", "dk", "dv", "dqr", "dkr"), saved, recomputed):
        assert torch.equal(a, b), nm
    # the forward's outputs do not depend on saving (tiles of 128 keys: the
    # same code path; 64-key tiles of a band block take the band path then)
    g.band_bias = None
    out2, lse2, _ = B.attn_fwd(g, *t[:5])
    torch.cuda.synchronize()
    if w.D != 128:
        assert torch.equal(out, out2) and torch.equal(lse, lse2)
    else:
        assert (out.float() - out2.float()).abs().max().item() < 2e-2
    del bias


@pytest.mark.parametrize("name", ["v3_base", "long", "hd128", "varlen"])
def test_saved_bias_against_oracle(name):
    w, x = inputs(name)
    H = x.q.shape[1]
    check_against_oracle(x, w, H, p_drop=w.dropout_p, seed=5, offset=0, saved_bias=True)


def test_misaligned_band_bias_is_rejected():
    w, x = inputs("v3_base")
    g = geometry(x, w, 2)
    t = [a.to("cuda") for a in (x.q, x.k, x.v, x.qr, x.kr)]
    buf = B.alloc_band_bias(g, t[0].dtype)
    g.band_bias = buf[8:]
    with pytest.raises(B.DfError) as e:
        B.attn_fwd(g, *t)
    assert e.value.code == B.DF_ERR_INVALID_ARG
