"""The checked build (DF_CHECKED) on the GPU.

Built with DF_CHECKED, the tensor-core kernels range-check the indices of
their shared-memory gathers -- the forward's own and cross band windows, the
band-bias kernel's windows, the dQ kernel's row of the stored-bias box --
and the destination range of the forward's band-window copies; a failed
check records DF_ERR_DEVICE_CHECK in the workspace error word and clamps the
access into its buffer (no trap, no fault).  Over the parity workloads --
bucketed and plain relative positions, the smallest and the largest span,
D = 32 / 64 / 128, bf16 and fp16, padding masks, packed sequences, dropout,
and the band bias saved by the forward or computed by the backward -- no
check may fire (run_gpu asserts both workspaces' error words are clear),
and the checks must not change a single output bit against the plain build.
"""
import dataclasses

import pytest
import torch

from exact_deberta_disentangled_gb300 import binding as B
from exact_deberta_disentangled_gb300 import build as build_mod
from exact_deberta_disentangled_gb300 import synth
from tests.test_parity_tc_gpu import run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def checked_lib():
    import __graft_entry__
    __graft_entry__.build()
    return build_mod.build(checked=True)


def _case(name):
    w = synth.WORKLOADS
    if name == "v3_masked":
        return w["v3_base"], synth.make_inputs(w["v3_base"], B=3, L=384, H=2), 2, {}
    if name == "long_band":
        return w["sweep_L8192"], synth.make_inputs(w["sweep_L8192"], B=1, L=1536, H=2), 2, {}
    if name == "packed":
        return w["varlen"], synth.make_inputs(w["varlen"], H=2, total_tokens=1500), 2, {}
    if name == "hd128_dropout":
        wd = w["hd128_dropout"]
        return wd, synth.make_inputs(wd, B=1, L=600, H=2), 2, dict(p_drop=wd.dropout_p, seed=1234, offset=3)
    if name == "hd32_dropout":
        wd = w["hd32_dropout"]
        return wd, synth.make_inputs(wd, B=2, L=520, H=2), 2, dict(p_drop=wd.dropout_p, seed=99)
    if name == "fp16":
        return w["v3_base"], synth.make_inputs(w["v3_base"], B=2, L=700, H=2, dtype="fp16"), 2, {}
    if name == "no_bucketing":
        wd = dataclasses.replace(w["sweep_L1024"], nb=0, mp=0)
        return wd, synth.make_inputs(wd, B=1, L=700, H=2), 2, {}
    if name == "small_span":
        wd = dataclasses.replace(w["sweep_L1024"], span=8, nb=4, mp=8)
        return wd, synth.make_inputs(wd, B=1, L=600, H=2), 2, {}
    if name == "largest_span":
        wd = dataclasses.replace(w["sweep_L2048"], span=512, nb=512, mp=1024)
        return wd, synth.make_inputs(wd, B=1, L=1500, H=2), 2, {}
    raise KeyError(name)


CASES = ["v3_masked", "long_band", "packed", "hd128_dropout", "hd32_dropout", "fp16", "no_bucketing",
         "small_span", "largest_span"]


@pytest.mark.parametrize("saved_bias", [True, False], ids=["bias_saved", "bias_kernel"])
@pytest.mark.parametrize("name", CASES)
def test_checked_build_no_check_fires_and_results_unchanged(checked_lib, name, saved_bias):
    w, x, H, kw = _case(name)
    _, _, out, lse, grads = run_gpu(x, w, H, saved_bias=saved_bias, **kw)
    with B.checked_library(checked_lib):
        _, _, out_c, lse_c, grads_c = run_gpu(x, w, H, saved_bias=saved_bias, **kw)
    assert torch.equal(out, out_c)
    assert torch.equal(lse, lse_c)
    for a, b in zip(grads, grads_c):
        assert torch.equal(a, b)
