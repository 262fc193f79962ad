"""GPU parity of the strict-fp32 path and the relative-index table, through
the C ABI, against the fp64 oracle on the same seeded inputs."""
import numpy as np
import pytest
import torch

from exact_deberta_disentangled_gb300 import binding as B
from exact_deberta_disentangled_gb300 import synth
from oracle import oracle
from tests.helpers import f64, lse_to_oracle_layout, max_abs, problem_of, rel_l2

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("L,span,nb,mp", [(8192, 256, 256, 512), (128, 64, 64, 128), (4096, 256, 256, 512),
                                          (2048, 256, 0, 0), (333, 17, 12, 100)])
def test_rel_index_table_bit_exact(L, span, nb, mp):
    got = B.rel_index_table(L, span, nb, mp).cpu().numpy()
    want = oracle.delta_table(L, span, nb if nb > 0 and mp > 0 else 0, mp if nb > 0 and mp > 0 else 0)
    assert np.array_equal(got, want)


def run_case(x, w, H, p_drop=0.0, seed=0, offset=0):
    dev = torch.device(DEV)
    g = B.Geometry(B=x.B, L=x.L, H=H, D=w.D, span=w.span, nb=w.nb, mp=w.mp, dropout_p=p_drop, seed=seed,
                   offset=offset)
    if x.packed:
        g.cu_seqlens = x.cu_seqlens.to(dev)
        g.total_tokens = int(x.cu_seqlens[-1])
    if x.qmask is not None:
        g.query_mask, g.key_mask = x.qmask.to(dev), x.kmask.to(dev)
    t = [a.to(dev) for a in (x.q, x.k, x.v, x.qr, x.kr, x.dout)]
    out, lse, ws = B.attn_fwd(g, *t[:5])
    grads, wsb = B.attn_bwd(g, *t[:5], out, lse, t[5])
    torch.cuda.synchronize()
    assert B.device_error(ws) == 0 and B.device_error(wsb) == 0
    prob = problem_of(x, w, H, p_drop, seed, offset)
    args = [f64(a) for a in (x.q, x.k, x.v, x.qr, x.kr)]
    o_ref, lse_ref = oracle.forward(prob, *args)
    g_ref = oracle.backward(prob, *args, f64(x.dout))
    lse_got = lse_to_oracle_layout(lse, x.packed, x.B, H, x.L)
    return out, lse_got, grads, o_ref, lse_ref, g_ref, (g, t, out, lse)


def check_fp32(out, lse_got, grads, o_ref, lse_ref, g_ref, tol=1e-5):
    assert rel_l2(out, o_ref) <= tol
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lse_got), fin)
    assert rel_l2(lse_got[fin], lse_ref[fin]) <= tol
    for name, a, b in zip(["dq", "dk", "dv", "dqr", "dkr"], grads, g_ref):
        assert rel_l2(a, b) <= tol, name


def test_fp32_tiny_workload():
    w = synth.WORKLOADS["tiny_fp32"]
    x = synth.make_inputs(w)
    out, lse_got, grads, o_ref, lse_ref, g_ref, _ = run_case(x, w, w.H)
    check_fp32(out, lse_got, grads, o_ref, lse_ref, g_ref)
    assert max_abs(out, o_ref) <= 1e-5


def test_fp32_masked_padded():
    w = synth.WORKLOADS["v3_base"]
    x = synth.make_inputs(w, B=3, L=160, H=2, dtype="fp32")
    check_fp32(*run_case(x, w, 2)[:6])


def test_fp32_packed_varlen():
    w = synth.WORKLOADS["varlen"]
    x = synth.make_inputs(w, H=2, total_tokens=700, dtype="fp32")
    check_fp32(*run_case(x, w, 2)[:6])


def test_fp32_dropout_regenerated_in_backward():
    w = synth.WORKLOADS["hd32_dropout"]
    x = synth.make_inputs(w, B=2, L=200, H=2, dtype="fp32")
    check_fp32(*run_case(x, w, 2, p_drop=0.1, seed=0xDEADBEEF12, offset=5)[:6])


def test_fp32_backward_is_bitwise_deterministic():
    w = synth.WORKLOADS["tiny_fp32"]
    x = synth.make_inputs(w)
    *_, (g, t, out, lse) = run_case(x, w, w.H)
    a, _ = B.attn_bwd(g, *t[:5], out, lse, t[5])
    b, _ = B.attn_bwd(g, *t[:5], out, lse, t[5])
    for u, v in zip(a, b):
        assert torch.equal(u, v)


def test_inconsistent_cu_seqlens_are_reported_not_faulted():
    w = synth.WORKLOADS["varlen"]
    x = synth.make_inputs(w, H=2, total_tokens=300, dtype="fp32")
    dev = torch.device(DEV)
    cu = torch.tensor([0, 205, 100, 300], dtype=torch.int32)   # non-monotone offsets
    g = B.Geometry(B=3, L=205, H=2, D=w.D, span=w.span, nb=w.nb, mp=w.mp, cu_seqlens=cu.to(dev),
                   total_tokens=300)
    t = [a.to(dev) for a in (x.q, x.k, x.v, x.qr, x.kr)]
    out, lse, ws = B.attn_fwd(g, *t)
    assert B.device_error(ws) == B.DF_ERR_DEVICE_ARG
    # the context stays usable
    assert torch.isfinite(torch.ones(4, device=dev).sum())
