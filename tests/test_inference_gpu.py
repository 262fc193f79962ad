"""The inference forward (df_attn_fwd_inference: no LSE) on the GPU.

"DisentangledFlash" (section "Status") keeps an inference path beside the
training path, and its Hugging Face integration presets run lengths from 64
up (section "Hugging Face usage").  At short lengths (64, 128, 384: a single
tile, one tile plus a tail, three tiles) and the v3-base head layout (H=12,
D=64, padding masks) the inference output must equal the training forward's
output bit for bit (same kernel, the LSE store skipped) and match the fp64
oracle within the forward bars (rel-L2 <= 5e-3, max-abs <= 2e-2).  The MNLI
stand-in shape (fp16, batch 8, length bucket 512, 24 heads) is checked the
same way.
"""
import pytest
import torch

from exact_deberta_disentangled_gb300 import binding as B
from exact_deberta_disentangled_gb300 import synth
from oracle import oracle
from tests.helpers import f64, max_abs, problem_of, rel_l2
from tests.test_parity_tc_gpu import OUT_MAX, OUT_TOL, check_against_oracle, geometry

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def inference_vs_training(x, w, H):
    g = geometry(x, w, H)
    t = [a.to("cuda") for a in (x.q, x.k, x.v, x.qr, x.kr)]
    out_tr, _, _ = B.attn_fwd(g, *t)
    out_inf, ws = B.attn_fwd_inference(g, *t)
    torch.cuda.synchronize()
    assert B.device_error(ws) == B.DF_OK
    assert torch.equal(out_tr, out_inf)
    o_ref, _ = oracle.forward(problem_of(x, w, H), *[f64(a) for a in (x.q, x.k, x.v, x.qr, x.kr)])
    assert rel_l2(out_inf, o_ref) <= OUT_TOL and max_abs(out_inf, o_ref) <= OUT_MAX


@pytest.mark.parametrize("L", [64, 128, 384])
def test_short_length_inference(L):
    w = synth.WORKLOADS["v3_base"]
    x = synth.make_inputs(w, B=8, L=L, H=12)
    inference_vs_training(x, w, 12)


def test_mnli_shape_fp16_inference_and_training():
    w = synth.WORKLOADS["mnli_fp16"]
    x = synth.make_inputs(w)
    assert x.q.dtype == torch.float16 and (x.B, x.L, x.q.shape[1]) == (8, 512, 24)
    inference_vs_training(x, w, 24)
    check_against_oracle(x, w, 24)


def test_inference_rejects_bad_pointers():
    w = synth.WORKLOADS["v3_base"]
    x = synth.make_inputs(w, B=1, L=64, H=2)
    g = geometry(x, w, 2)
    t = [a.to("cuda") for a in (x.q, x.k, x.v, x.qr, x.kr)]
    out = torch.empty_like(t[0])
    ws = B.alloc_workspace(g, t[0].dtype, False)
    p = g.params(t[0].dtype)
    import ctypes
    rc = B.load().df_attn_fwd_inference(ctypes.byref(p), None, B._ptr(t[1]), B._ptr(t[2]), B._ptr(t[3]),
                                        B._ptr(t[4]), B._ptr(out), B._ptr(ws), ws.numel(), B._stream())
    assert rc == B.DF_ERR_INVALID_ARG
