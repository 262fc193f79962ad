"""The fast fp32 mode (DF_FP32_FAST) on the GPU.

fp32 tensors go through the fp16 tensor-core path: the inputs are rounded to
fp16 (TF32's 10-bit significand) in the workspace and the fp16 results are
widened back ("DisentangledFlash", section "Status": the optional fast
FP32/TF32 mode).  So every output must equal, bit for bit, the fp16 path run
on the inputs rounded by torch (round to nearest even) and widened by torch;
and against the fp64 oracle on the unrounded fp32 inputs the mode meets the
16-bit path's bars (output and LSE rel-L2 <= 5e-3, max-abs <= 2e-2, every
gradient rel-L2 <= 1e-2).  Cases: padding masks, packed sequences with
dropout, D = 32 / 128, the saved band bias and the host-buffer step.
"""
import numpy as np
import pytest
import torch

from exact_deberta_disentangled_gb300 import binding as B
from exact_deberta_disentangled_gb300 import synth
from oracle import oracle
from tests.helpers import f64, lse_to_oracle_layout, max_abs, problem_of, rel_l2
from tests.test_parity_tc_gpu import GRAD_TOL, OUT_MAX, OUT_TOL, geometry

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def run(x, w, H, fast, saved_bias=False, **kw):
    """fast: fp32 tensors in the fast mode; else the fp16 path on the inputs
    rounded by torch, results widened by torch."""
    g = geometry(x, w, H, **kw)
    g.fp32_fast = fast
    t = [a.to("cuda").float() for a in (x.q, x.k, x.v, x.qr, x.kr, x.dout)]
    if not fast:
        t = [a.half() for a in t]
    if saved_bias:
        g.band_bias = B.alloc_band_bias(g, t[0].dtype)
    out, lse, ws = B.attn_fwd(g, *t[:5])
    grads, wsb = B.attn_bwd(g, *t[:5], out, lse, t[5])
    torch.cuda.synchronize()
    assert B.device_error(ws) == 0 and B.device_error(wsb) == 0
    return out.float(), lse, [a.float() for a in grads]


CASES = {
    "masked": lambda: (synth.WORKLOADS["v3_base"], dict(B=3, L=384, H=2), {}),
    "packed_dropout": lambda: (synth.WORKLOADS["varlen"], dict(H=2, total_tokens=1500),
                               dict(p_drop=0.1, seed=7, offset=2)),
    "hd32": lambda: (synth.WORKLOADS["hd32_dropout"], dict(B=2, L=520, H=2), {}),
    "hd128_long": lambda: (synth.WORKLOADS["hd128_dropout"], dict(B=1, L=1100, H=2), {}),
}


@pytest.mark.parametrize("saved_bias", [False, True], ids=["bias_kernel", "bias_saved"])
@pytest.mark.parametrize("name", list(CASES))
def test_fast_equals_fp16_path_on_rounded_inputs(name, saved_bias):
    w, shape, kw = CASES[name]()
    x = synth.make_inputs(w, dtype="fp32", **shape)
    o1, l1, g1 = run(x, w, shape["H"], True, saved_bias, **kw)
    o2, l2, g2 = run(x, w, shape["H"], False, saved_bias, **kw)
    assert o1.dtype == torch.float32 and torch.equal(o1, o2)
    assert torch.equal(l1, l2)
    for n, a, b in zip(("dq", "dk", "dv", "dqr", "dkr"), g1, g2):
        assert a.dtype == torch.float32 and torch.equal(a, b), n


@pytest.mark.parametrize("name", ["masked", "packed_dropout", "hd128_long"])
def test_fast_against_oracle(name):
    w, shape, kw = CASES[name]()
    H = shape["H"]
    x = synth.make_inputs(w, dtype="fp32", **shape)
    out, lse, grads = run(x, w, H, True, **kw)
    prob = problem_of(x, w, H, kw.get("p_drop", 0.0), kw.get("seed", 0), kw.get("offset", 0))
    args = [f64(a) for a in (x.q, x.k, x.v, x.qr, x.kr)]
    o_ref, lse_ref = oracle.forward(prob, *args)
    assert rel_l2(out, o_ref) <= OUT_TOL and max_abs(out, o_ref) <= OUT_MAX
    lse_got = lse_to_oracle_layout(lse, x.packed, x.B, H, x.L)
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lse_got), fin)
    assert rel_l2(lse_got[fin], lse_ref[fin]) <= OUT_TOL and max_abs(lse_got[fin], lse_ref[fin]) <= OUT_MAX
    ref = oracle.backward(prob, *args, f64(x.dout))
    for n, a, b in zip(("dq", "dk", "dv", "dqr", "dkr"), grads, ref):
        assert rel_l2(a, b) <= GRAD_TOL, (n, rel_l2(a, b))


def test_fast_host_buffer_step():
    """df_attn_step_host in the fast mode equals the device calls bit for bit."""
    from tests.test_step_host_gpu import host_step
    w = synth.WORKLOADS["v3_base"]
    x = synth.make_inputs(w, B=2, L=320, H=2, dtype="fp32")
    g, pin, outs, arena, (hcu, hqm, hkm) = host_step(x, w, 2)
    g.fp32_fast = True
    arena = torch.empty(B.step_host_arena_size(g, torch.float32), dtype=torch.uint8, device="cuda")
    gd = geometry(x, w, 2)
    gd.fp32_fast = True
    t = [a.to("cuda") for a in (x.q, x.k, x.v, x.qr, x.kr, x.dout)]
    gd.band_bias = B.alloc_band_bias(gd, torch.float32)
    out, lse, _ = B.attn_fwd(gd, *t[:5])
    grads, _ = B.attn_bwd(gd, *t[:5], out, lse, t[5])
    torch.cuda.synchronize()
    for o in outs:
        o.fill_(float("nan"))
    B.step_host(g, *pin, outs, arena, host_cu=hcu, host_qmask=hqm, host_kmask=hkm)
    for name, got, ref in zip(("out", "lse", "dq", "dk", "dv", "dqr", "dkr"), outs, (out, lse) + tuple(grads)):
        assert torch.equal(got, ref.cpu()), name


def test_fast_inference_and_noalloc_forward():
    """The fast mode through the inference forward (no LSE) and through the
    no-workspace forward gives the training forward's O bit for bit."""
    w = synth.WORKLOADS["v3_base"]
    x = synth.make_inputs(w, B=2, L=256, H=2, dtype="fp32")
    g = geometry(x, w, 2)
    g.fp32_fast = True
    t = [a.to("cuda") for a in (x.q, x.k, x.v, x.qr, x.kr)]
    out, lse, _ = B.attn_fwd(g, *t)
    out_inf, _ = B.attn_fwd_inference(g, *t)
    out_na, lse_na = torch.empty_like(out), torch.empty_like(lse)
    B.attn_fwd_noalloc(g, *t, out_na, lse_na)
    torch.cuda.synchronize()
    assert torch.equal(out, out_inf)
    assert torch.equal(out, out_na) and torch.equal(lse, lse_na)


def test_fast_rejects_what_the_16_bit_path_rejects():
    """A bucketing configuration whose index jumps by two is unsupported for
    the tensor-core path, hence for the fast mode, and fine in strict fp32."""
    w = synth.WORKLOADS["v3_base"]
    x = synth.make_inputs(w, B=1, L=128, H=1, dtype="fp32")
    g = geometry(x, w, 1)
    g.nb, g.mp = 256, 300
    g.fp32_fast = True
    t = [a.to("cuda") for a in (x.q, x.k, x.v, x.qr, x.kr)]
    with pytest.raises(B.DfError) as e:
        B.attn_fwd(g, *t, workspace=torch.empty(1 << 20, dtype=torch.uint8, device="cuda"))
    assert e.value.code == B.DF_ERR_UNSUPPORTED
