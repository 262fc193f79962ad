"""The steps on either side of the attention on the GPU, against the fp64
oracle: the fused QKV projection and the layer-normalised relative-position
projections with shared query / key weights, forward and backward
("DisentangledFlash", section "Status": the fused QKV projection; section
"Hugging Face usage": the projections stay in the autograd graph).

Shapes of a DeBERTa-v3-base layer (hidden 768 = 12 heads x 64, R = 512
relative rows) over 2,048 tokens, bf16 and fp16 storage with fp32
accumulation; bars: rel-L2 <= 1e-2 for every output and gradient (bf16
storage rounds at 2^-9).  Then the whole layer step: projections, attention
forward and backward, projection backward, with the gradients of the shared
weights accumulated in order, against the oracle's composition.
"""
import numpy as np
import pytest
import torch

from exact_deberta_disentangled_gb300 import binding as B
from oracle import oracle
from tests.helpers import rel_l2

pytestmark = pytest.mark.gpu
TOL = 1e-2
EPS = 1e-7


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def draw(gen, shape, scale=1.0, dtype=torch.bfloat16):
    return (torch.randn(shape, generator=gen) * scale).to(dtype)


def f64(t):
    return t.double().cpu().numpy()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_qkv_projection(dtype):
    g = torch.Generator().manual_seed(11)
    T, C, H, D = 2048, 768, 12, 64
    x, w, b = draw(g, (T, C), 1.0, dtype), draw(g, (3, H * D, C), C ** -0.5, dtype), draw(g, (3, H * D), 0.1, dtype)
    dy = draw(g, (3, T, H * D), 1.0, dtype)
    xd, wd, bd, dyd = (a.cuda() for a in (x, w, b, dy))
    qkv = B.qkv_proj_fwd(xd, wd, bd)
    dx, dw, db = B.qkv_proj_bwd(xd, wd, dyd)
    torch.cuda.synchronize()
    assert rel_l2(qkv, oracle.qkv_projection(f64(x), f64(w), f64(b))) <= TOL
    rdx, rdw, rdb = oracle.qkv_projection_backward(f64(x), f64(w), f64(dy))
    for got, want in ((dx, rdx), (dw, rdw), (db, rdb)):
        assert rel_l2(got, want) <= TOL
    # accumulate adds to what is there
    dw2, db2 = dw.clone(), db.clone()
    B.qkv_proj_bwd(xd, wd, dyd, dw=dw2, dbias=db2, accumulate=True)
    assert rel_l2(dw2, 2 * rdw) <= TOL and rel_l2(db2, 2 * rdb) <= TOL


def test_relative_projection():
    g = torch.Generator().manual_seed(12)
    R, C, H, D = 512, 768, 12, 64
    rel, gamma, beta = draw(g, (R, C)), 1 + draw(g, (C,), 0.1), draw(g, (C,), 0.1)
    w, b = draw(g, (3, H * D, C), C ** -0.5), draw(g, (3, H * D), 0.1)
    dqr, dkr = draw(g, (H, R, D)), draw(g, (H, R, D))
    dev = [a.cuda() for a in (rel, gamma, beta, w, b, dqr, dkr)]
    qr, kr, rel_ln, stats = B.rel_proj_fwd(dev[0], dev[1], dev[2], EPS, dev[3], dev[4], H, D)
    dw = torch.zeros_like(dev[3])
    dbias = torch.zeros_like(dev[4])
    drel, dgamma, dbeta = B.rel_proj_bwd(dev[0], dev[1], rel_ln, stats, dev[3], dev[5], dev[6], dw, dbias)
    torch.cuda.synchronize()
    E, Q, K = oracle.rel_projection(f64(rel), f64(gamma), f64(beta), EPS, f64(w), f64(b), H, D)
    assert rel_l2(rel_ln, E) <= TOL and rel_l2(qr, Q) <= TOL and rel_l2(kr, K) <= TOL
    r = oracle.rel_projection_backward(f64(rel), f64(gamma), f64(beta), EPS, f64(w), f64(dqr), f64(dkr), H, D)
    for got, want in ((drel, r[0]), (dgamma, r[1]), (dbeta, r[2]), (dw[:2], r[3]), (dbias[:2], r[4])):
        assert rel_l2(got, want) <= TOL
    assert not dw[2].any() and not dbias[2].any()   # W_v rows untouched


def test_layer_step_with_shared_weights():
    """Projections + attention + projection gradients of one DeBERTa layer
    (the v3-base head layout over 2 sequences of 512 tokens)."""
    from exact_deberta_disentangled_gb300 import synth
    gen = torch.Generator().manual_seed(13)
    Bn, L, H, D, C, span = 2, 512, 12, 64, 768, 256
    R, T = 2 * span, Bn * L
    x, rel = draw(gen, (T, C)), draw(gen, (R, C))
    gamma, beta = 1 + draw(gen, (C,), 0.1), draw(gen, (C,), 0.1)
    w, b = draw(gen, (3, H * D, C), C ** -0.5), draw(gen, (3, H * D), 0.1)
    dout = draw(gen, (T, H, D))
    xd, reld, gd, bed, wd, bd, dod = (a.cuda() for a in (x, rel, gamma, beta, w, b, dout))
    qkv = B.qkv_proj_fwd(xd, wd, bd)
    qr, kr, rel_ln, stats = B.rel_proj_fwd(reld, gd, bed, EPS, wd, bd, H, D)
    geo = B.Geometry(B=Bn, L=L, H=H, D=D, span=span, nb=256, mp=512)
    q, k, v = (qkv[j].reshape(T, H, D) for j in range(3))
    out, lse, _ = B.attn_fwd(geo, q, k, v, qr, kr)
    (dq, dk, dv, dqr, dkr), _ = B.attn_bwd(geo, q, k, v, qr, kr, out, lse, dod)
    dqkv = torch.stack([dq.reshape(T, H * D), dk.reshape(T, H * D), dv.reshape(T, H * D)])
    dx, dw, dbias = B.qkv_proj_bwd(xd, wd, dqkv)
    drel, dgamma, dbeta = B.rel_proj_bwd(reld, gd, rel_ln, stats, wd, dqr, dkr, dw, dbias, accumulate=True)
    torch.cuda.synchronize()

    # the oracle's composition, from the same rounded parameters
    yq = oracle.qkv_projection(f64(x), f64(w), f64(b))
    E, Qr, Kr = oracle.rel_projection(f64(rel), f64(gamma), f64(beta), EPS, f64(w), f64(b), H, D)
    prob = oracle.Problem(np.arange(Bn + 1) * L, H, D, span, 256, 512)
    args = [yq[j].reshape(T, H, D) for j in range(3)] + [Qr, Kr]
    o_ref, _ = oracle.forward(prob, *args)
    gq, gk, gv, gqr, gkr = oracle.backward(prob, *args, f64(dout))
    rdx, rdw, rdb = oracle.qkv_projection_backward(f64(x), f64(w),
                                                   np.stack([a.reshape(T, H * D) for a in (gq, gk, gv)]))
    rr = oracle.rel_projection_backward(f64(rel), f64(gamma), f64(beta), EPS, f64(w), gqr, gkr, H, D)
    rdw[:2] += rr[3]
    rdb[:2] += rr[4]
    assert rel_l2(out, o_ref) <= 5e-3 * 2   # the projected inputs are themselves rounded to bf16
    for got, want in ((dx, rdx), (dw, rdw), (dbias, rdb), (drel, rr[0]), (dgamma, rr[1]), (dbeta, rr[2])):
        assert rel_l2(got, want) <= 2 * TOL
