"""The bounded-wait path of the three attention kernels on the GPU.

Every wait of a kernel on an mbarrier is bounded: when it runs out it records
DF_ERR_TIMEOUT in the call's device error word, sets a CTA-wide abort flag,
and every role of the CTA leaves its loop (the softmax warps still meet every
named barrier on the way out, and the copy and MMA roles wait for their own
work in flight).  Here the library's test hook makes the MMA-issuing warp of
one kernel stop at a chosen tile, so that the other roles wait for work that
never comes; no fault, trap or endless loop is involved.  Each case checks
that the call returns within a few seconds, that the error word says
DF_ERR_TIMEOUT, and that the next, normal call on the same context gives
outputs that match the oracle.
"""
import time

import pytest
import torch

from exact_deberta_disentangled_gb300 import binding as B
from exact_deberta_disentangled_gb300 import synth
from tests.test_parity_tc_gpu import check_against_oracle, geometry

pytestmark = pytest.mark.gpu
LIMIT_NS = 20_000_000   # 20 ms per wait
PROBES = 64


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    yield
    B.debug_inject_stall(-1)


def small_case():
    # 16 row blocks x 2 heads = 32 CTAs per kernel (one wave); tiles near the
    # diagonal are band tiles, the far ones uniform
    w = synth.WORKLOADS["sweep_L2048"]
    x = synth.make_inputs(w, B=1, L=2048, H=2)
    return w, x


@pytest.mark.parametrize("kernel,tile", [(0, 0), (0, 9), (1, 0), (1, 5), (2, 1), (2, 12)])
def test_stalled_kernel_gives_up_and_context_stays_usable(kernel, tile):
    w, x = small_case()
    g = geometry(x, w, 2)
    t = [a.to("cuda") for a in (x.q, x.k, x.v, x.qr, x.kr, x.dout)]
    out, lse, wsf = B.attn_fwd(g, *t[:5])
    torch.cuda.synchronize()
    assert B.device_error(wsf) == B.DF_OK
    B.debug_inject_stall(kernel, tile, LIMIT_NS, PROBES)
    try:
        t0 = time.perf_counter()
        if kernel == 0:
            B.attn_fwd(g, *t[:5], out=out, lse=lse, workspace=wsf)
            ws = wsf
        else:
            _, ws = B.attn_bwd(g, *t[:5], out, lse, t[5])
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
    finally:
        B.debug_inject_stall(-1)
    assert B.device_error(ws) == B.DF_ERR_TIMEOUT
    assert elapsed < 10.0, elapsed
    # the same context, the default limits again: a normal call is correct
    check_against_oracle(x, w, 2)
