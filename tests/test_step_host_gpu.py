"""The training step from host buffers (df_attn_step_host) on the GPU.

The step copies the inputs up, runs the forward and the backward and copies
the results down, with dO's upload and the O / LSE download on a copy stream
that overlaps the kernels.  Both kernels are deterministic (the backward
reduces the relative-position gradients in a fixed order), so every output
of the host-buffer step must equal, bit for bit, the same forward + backward
run on device tensors: for padding masks (query mask equal to and different
from the key mask), packed sequences and dropout, and for several calls in a
row through one arena (the copy stream's events are reused).  The step is
checked against the fp64 oracle once as well.
"""
import pytest
import torch

from exact_deberta_disentangled_gb300 import binding as B
from exact_deberta_disentangled_gb300 import synth
from oracle import oracle
from tests.helpers import f64, max_abs, problem_of, rel_l2
from tests.test_parity_tc_gpu import OUT_MAX, OUT_TOL, geometry, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def host_step(x, w, H, **kw):
    g = geometry(x, w, H, **kw)
    pin = [a.contiguous().pin_memory() for a in (x.q, x.k, x.v, x.qr, x.kr, x.dout)]
    outs = (torch.empty_like(pin[0]).pin_memory(), torch.empty(g.lse_shape(), dtype=torch.float32).pin_memory(),
            torch.empty_like(pin[0]).pin_memory(), torch.empty_like(pin[1]).pin_memory(),
            torch.empty_like(pin[2]).pin_memory(), torch.empty_like(pin[3]).pin_memory(),
            torch.empty_like(pin[4]).pin_memory())
    arena = torch.empty(B.step_host_arena_size(g, x.q.dtype), dtype=torch.uint8, device="cuda")
    host_cu = x.cu_seqlens.to(torch.int32).contiguous() if x.packed else None
    host_qm = x.qmask.contiguous() if x.qmask is not None else None
    host_km = x.kmask.contiguous() if x.kmask is not None else None
    return g, pin, outs, arena, (host_cu, host_qm, host_km)


def check_step_equals_device(x, w, H, calls=1, **kw):
    g, pin, outs, arena, (hcu, hqm, hkm) = host_step(x, w, H, **kw)
    _, _, out, lse, grads = run_gpu(x, w, H, **kw)
    for _ in range(calls):
        for o in outs:
            o.fill_(float("nan")) if o.is_floating_point() else o.zero_()
        B.step_host(g, *pin, outs, arena, host_cu=hcu, host_qmask=hqm, host_kmask=hkm)
        want = (out, lse) + tuple(grads)
        for name, got, ref in zip(("out", "lse", "dq", "dk", "dv", "dqr", "dkr"), outs, want):
            assert torch.equal(got, ref.cpu()), name
    return outs


def test_padded_masks_bit_exact():
    w = synth.WORKLOADS["v3_base"]
    x = synth.make_inputs(w, B=3, L=320, H=4)
    assert x.qmask is not None
    check_step_equals_device(x, w, 4, calls=3)


def test_independent_key_mask_bit_exact():
    w = synth.WORKLOADS["v3_base"]
    x = synth.make_inputs(w, B=2, L=256, H=3, key_mask="independent")
    assert not torch.equal(x.qmask, x.kmask)
    check_step_equals_device(x, w, 3)


def test_packed_and_dropout_bit_exact():
    w = synth.WORKLOADS["varlen"]
    x = synth.make_inputs(w, H=2, total_tokens=1500)
    assert x.packed
    check_step_equals_device(x, w, 2, p_drop=0.1, seed=11, offset=4)


def test_step_against_oracle():
    w = synth.WORKLOADS["v3_base"]
    x = synth.make_inputs(w, B=2, L=192, H=2)
    outs = check_step_equals_device(x, w, 2)
    o_ref, _ = oracle.forward(problem_of(x, w, 2), *[f64(a) for a in (x.q, x.k, x.v, x.qr, x.kr)])
    assert rel_l2(outs[0], o_ref) <= OUT_TOL and max_abs(outs[0], o_ref) <= OUT_MAX
