"""Pins of the oracle's projection functions (the steps on either side of the
attention: fused QKV projection, layer-normalised relative-position
projections with shared query / key weights), independent of the oracle's
own formulas:

- the forward against a second formulation in torch (float64, CPU): einsum
  for the projections and torch.nn.functional.layer_norm;
- every gradient against torch autograd of that formulation and against
  central finite differences on small shapes.
"""
import numpy as np
import pytest
import torch

from oracle import oracle

pytestmark = pytest.mark.filterwarnings("ignore")
RNG = np.random.default_rng(1234)
T, C, H, D, R, EPS = 6, 16, 2, 4, 7, 1e-7
HD = H * D


def draw(*shape):
    return RNG.standard_normal(shape)


def torch_rel(rel, g, b, w, bias):
    e = torch.nn.functional.layer_norm(rel, (C,), g, b, EPS)
    qr = (e @ w[0].T + bias[0]).reshape(R, H, D).permute(1, 0, 2)
    kr = (e @ w[1].T + bias[1]).reshape(R, H, D).permute(1, 0, 2)
    return e, qr, kr


def test_qkv_projection_against_torch_autograd_and_differences():
    x, w, b, dy = draw(T, C), draw(3, HD, C), draw(3, HD), draw(3, T, HD)
    xt, wt, bt = (torch.tensor(a, requires_grad=True) for a in (x, w, b))
    y = torch.einsum("tc,jnc->jtn", xt, wt) + bt[:, None, :]
    assert np.allclose(oracle.qkv_projection(x, w, b), y.detach().numpy(), atol=1e-12)
    y.backward(torch.tensor(dy))
    dx, dw, db = oracle.qkv_projection_backward(x, w, dy)
    for got, want in ((dx, xt.grad), (dw, wt.grad), (db, bt.grad)):
        assert np.allclose(got, want.numpy(), atol=1e-12)
    # central differences of L = <dy, y> in a few coordinates of x and w
    f = lambda xx, ww: float((oracle.qkv_projection(xx, ww, b) * dy).sum())
    h = 1e-6
    for (t, c) in ((0, 0), (3, 7), (5, 15)):
        e = np.zeros_like(x)
        e[t, c] = h
        assert abs((f(x + e, w) - f(x - e, w)) / (2 * h) - dx[t, c]) < 1e-6
    for (j, n, c) in ((0, 0, 0), (1, 5, 3), (2, 7, 15)):
        e = np.zeros_like(w)
        e[j, n, c] = h
        assert abs((f(x, w + e) - f(x, w - e)) / (2 * h) - dw[j, n, c]) < 1e-6


def test_layer_norm_against_torch():
    x, g, b = draw(R, C), draw(C), draw(C)
    y, mean, rstd = oracle.layer_norm(x, g, b, EPS)
    want = torch.nn.functional.layer_norm(torch.tensor(x), (C,), torch.tensor(g), torch.tensor(b), EPS)
    assert np.allclose(y, want.numpy(), atol=1e-12)
    assert np.allclose(mean, x.mean(1)) and np.allclose(rstd, 1 / np.sqrt(x.var(1) + EPS))


def test_rel_projection_against_torch_autograd_and_differences():
    rel, g, be, w, bias = draw(R, C), draw(C), draw(C), draw(3, HD, C), draw(3, HD)
    dq, dk = draw(H, R, D), draw(H, R, D)
    ts = [torch.tensor(a, requires_grad=True) for a in (rel, g, be, w, bias)]
    e, qr, kr = torch_rel(*ts)
    E, Q, K = oracle.rel_projection(rel, g, be, EPS, w, bias, H, D)
    assert np.allclose(E, e.detach().numpy(), atol=1e-12)
    assert np.allclose(Q, qr.detach().numpy(), atol=1e-12) and np.allclose(K, kr.detach().numpy(), atol=1e-12)
    ((qr * torch.tensor(dq)).sum() + (kr * torch.tensor(dk)).sum()).backward()
    drel, dg, dbe, dw, db = oracle.rel_projection_backward(rel, g, be, EPS, w, dq, dk, H, D)
    assert np.allclose(drel, ts[0].grad.numpy(), atol=1e-10)
    assert np.allclose(dg, ts[1].grad.numpy(), atol=1e-10) and np.allclose(dbe, ts[2].grad.numpy(), atol=1e-10)
    assert np.allclose(dw, ts[3].grad.numpy()[:2], atol=1e-10) and np.allclose(db, ts[4].grad.numpy()[:2], atol=1e-10)
    assert not ts[3].grad.numpy()[2].any()   # W_v takes no part in the relative projections

    def loss(rr, gg):
        _, q, k = oracle.rel_projection(rr, gg, be, EPS, w, bias, H, D)
        return float((q * dq).sum() + (k * dk).sum())
    h = 1e-6
    for (r, c) in ((0, 0), (4, 9), (6, 15)):
        e1 = np.zeros_like(rel)
        e1[r, c] = h
        assert abs((loss(rel + e1, g) - loss(rel - e1, g)) / (2 * h) - drel[r, c]) < 1e-5
    for c in (0, 8, 15):
        e2 = np.zeros_like(g)
        e2[c] = h
        assert abs((loss(rel, g + e2) - loss(rel, g - e2)) / (2 * h) - dg[c]) < 1e-5
