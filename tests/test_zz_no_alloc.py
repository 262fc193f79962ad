"""The allocation-free forward (df_attn_fwd_noalloc) against the regular
forward (df_attn_fwd) through the C ABI.

Some callers cannot allocate device memory -- a plugin inside a framework
that owns the device arena, or a latency-critical loop that must not
synchronise on cudaMalloc -- so this entry point keeps its scratch in a
static device array of the library.  This file is collected last: it must
pass on its own in a fresh process and after every other test, and two calls
in a row must both agree with the workspace-based forward (the second call
reuses the array the first one left behind)."""
import numpy as np
import pytest
import torch

from exact_deberta_disentangled_gb300 import binding as B
from exact_deberta_disentangled_gb300 import synth
from tests.helpers import max_abs, rel_l2

pytestmark = pytest.mark.gpu
OUT_TOL, OUT_MAX = 5e-3, 2e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("name,kw", [("v3_base", dict(B=2, L=384, H=2)),
                                     ("tiny_fp32", dict())])
def test_noalloc_forward_matches_workspace_forward_twice(name, kw):
    w = synth.WORKLOADS[name]
    x = synth.make_inputs(w, **kw)
    dev = torch.device("cuda")
    g = B.Geometry(B=x.B, L=x.L, H=x.q.shape[1], D=w.D, span=w.span, nb=w.nb, mp=w.mp)
    if x.qmask is not None:
        g.query_mask, g.key_mask = x.qmask.to(dev), x.kmask.to(dev)
    t = [a.to(dev) for a in (x.q, x.k, x.v, x.qr, x.kr)]
    ref_out, ref_lse, _ = B.attn_fwd(g, *t)
    for _ in range(2):
        out = torch.full_like(t[0], float("nan"))
        lse = torch.full(g.lse_shape(), float("nan"), dtype=torch.float32, device=dev)
        B.attn_fwd_noalloc(g, *t, out, lse)
        torch.cuda.synchronize()
        assert B.noalloc_device_error() == B.DF_OK
        want = ref_out.double().cpu().numpy()
        assert rel_l2(out, want) <= OUT_TOL and max_abs(out, want) <= OUT_MAX
        lw = ref_lse.double().cpu().numpy()
        lg = lse.double().cpu().numpy()
        fin = np.isfinite(lw)
        assert np.array_equal(np.isfinite(lg), fin)
        assert rel_l2(lg[fin], lw[fin]) <= OUT_TOL


def test_noalloc_rejects_problems_beyond_its_scratch():
    g = B.Geometry(B=64, L=8192, H=16, D=64, span=256, nb=256, mp=512)   # 8.4M token-heads
    dev = torch.device("cuda")
    z = torch.zeros(16, dtype=torch.bfloat16, device=dev)
    lse = torch.zeros(16, dtype=torch.float32, device=dev)
    rc = B.attn_fwd_noalloc(g, z, z, z, z, z, z, lse, check=False)
    assert rc == B.DF_ERR_WORKSPACE
