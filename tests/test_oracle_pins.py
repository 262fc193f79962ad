"""Pins for the fp64 CPU oracle: it is checked here against things other than
itself -- hand-worked index values, library attention, closed forms,
invariants, an autograd formulation and finite differences -- before any GPU
result is compared with it.  CPU only.
"""
import math
import os

import numpy as np
import pytest
import torch

from oracle import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "delta_points.txt")


def _rng(seed):
    return np.random.default_rng(seed)


def _problem_inputs(cu, H, D, span, seed, scale_kr=1.0):
    T = int(cu[-1])
    R = 2 * span
    g = _rng(seed)
    q, k, v, do = (g.standard_normal((T, H, D)) for _ in range(4))
    qr, kr = (g.standard_normal((H, R, D)) * scale_kr for _ in range(2))
    return q, k, v, qr, kr, do


# ------------------------------------------------------------------ delta

def test_delta_golden_points():
    rows = [l.split() for l in open(GOLDEN) if l.strip() and not l.startswith("#")]
    assert len(rows) >= 20
    for span, nb, mp, r, d in (map(int, x) for x in rows):
        assert O.delta(r, span, nb, mp) == d, (span, nb, mp, r)


@pytest.mark.parametrize("span,nb,mp,L", [(256, 256, 512, 8192), (64, 64, 128, 128), (4, 4, 8, 16),
                                          (256, 0, 512, 2048), (32, 64, 1024, 4096)])
def test_delta_table_properties(span, nb, mp, L):
    tab = O.delta_table(L, span, nb, mp)
    r = np.arange(-(L - 1), L)
    R = 2 * span
    assert tab.min() >= 0 and tab.max() <= R - 1
    # monotone non-decreasing in r
    assert np.all(np.diff(tab) >= 0)
    # bucket is odd: delta(-r) - span = -(delta(r) - span) wherever neither side is clamped
    b = tab - span
    unclamped = (tab > 0) & (tab < R - 1) & (tab[::-1] > 0) & (tab[::-1] < R - 1)
    assert np.all(b[unclamped] == -b[::-1][unclamped])
    # linear region keeps r
    mid = nb // 2 if nb > 0 else L
    lin = (np.abs(r) <= mid) & (r + span >= 0) & (r + span <= R - 1)
    assert np.all(tab[lin] == r[lin] + span)


def test_delta_fp32_log_gives_same_indices():
    """The pages leave the precision of the bucket logarithm open; the oracle
    uses fp64.  For the workloads' bucket settings fp32 arithmetic reaches the
    same integers, so the choice does not change any index."""
    for nb, mp, L, span in [(256, 512, 8192, 256), (64, 128, 128, 64)]:
        mid = nb // 2
        r = np.arange(mid + 1, L, dtype=np.int64)
        x32 = (np.log((r / mid).astype(np.float32)) / np.float32(np.log(np.float32((mp - 1) / mid)))
               * np.float32(mid - 1)).astype(np.float32)
        b32 = mid + np.ceil(x32).astype(np.int64)
        b64 = np.array([O.bucket(int(v), nb, mp) for v in r])
        assert np.array_equal(np.minimum(b32 + span, 2 * span - 1), np.minimum(b64 + span, 2 * span - 1))


# ---------------------------------------------------------- forward pins

def test_plain_attention_matches_library_sdpa():
    """Kr = Qr = 0 reduces the method to softmax attention with scale
    1/sqrt(3D): compare with torch's scaled_dot_product_attention (fp64)."""
    B, L, H, D = 2, 24, 3, 8
    cu = np.arange(B + 1) * L
    q, k, v, qr, kr, _ = _problem_inputs(cu, H, D, 8, 1)
    qr[:] = 0
    kr[:] = 0
    g = _rng(7)
    lens = [17, 24]
    km = np.concatenate([(np.arange(L) < n) for n in lens]).astype(np.uint8)
    prob = O.Problem(cu, H, D, 8, 8, 16, kmask=km)
    o, lse = O.forward(prob, q, k, v, qr, kr)
    t = lambda a: torch.from_numpy(a.reshape(B, L, H, D)).permute(0, 2, 1, 3)
    mask = torch.from_numpy(km.reshape(B, 1, 1, L).astype(bool))
    ref = torch.nn.functional.scaled_dot_product_attention(t(q), t(k), t(v), attn_mask=mask,
                                                           scale=1.0 / math.sqrt(3 * D))
    np.testing.assert_allclose(o.reshape(B, L, H, D), ref.permute(0, 2, 1, 3).numpy(), rtol=1e-12, atol=1e-12)
    # LSE against torch.logsumexp of the library's own masked scores
    s = (t(q) @ t(k).transpose(-1, -2)) / math.sqrt(3 * D)
    s = s.masked_fill(~mask, -math.inf)
    lse_ref = torch.logsumexp(s, -1)  # [B, H, L]
    np.testing.assert_allclose(lse.reshape(H, B, L).transpose(1, 0, 2), lse_ref.numpy(), rtol=1e-12)


def test_rows_sum_to_one_and_single_token():
    cu = np.array([0, 1, 9, 20])
    H, D = 2, 6
    q, k, v, qr, kr, _ = _problem_inputs(cu, H, D, 4, 2)
    prob = O.Problem(cu, H, D, 4, 4, 8)
    ones = np.ones_like(v)
    o, _ = O.forward(prob, q, k, ones, qr, kr)
    np.testing.assert_allclose(o, 1.0, rtol=1e-13)
    o, lse = O.forward(prob, q, k, v, qr, kr)
    # the length-1 sequence attends only to itself: O = V, LSE = S[0,0]
    np.testing.assert_allclose(o[0], v[0], rtol=1e-13)
    c = 1 / math.sqrt(3 * D)
    d0 = O.delta(0, 4, 4, 8)
    s00 = c * (q[0] @ k[0].T).diagonal() + c * np.einsum("hd,hd->h", q[0], kr[:, d0]) \
        + c * np.einsum("hd,hd->h", k[0], qr[:, d0])
    np.testing.assert_allclose(lse[:, 0], s00, rtol=1e-12)


def test_equal_keys_give_mean_of_values():
    cu = np.array([0, 13])
    H, D = 1, 5
    q, k, v, qr, kr, _ = _problem_inputs(cu, H, D, 4, 3)
    k[:] = k[0:1]
    qr[:] = 0
    kr[:] = 0
    o, _ = O.forward(O.Problem(cu, H, D, 4, 4, 8), q, k, v, qr, kr)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(0, keepdims=True), o.shape), rtol=1e-12)


@pytest.mark.parametrize("which", ["c2p", "p2c"])
def test_relative_terms_closed_form(which):
    """With the content terms switched off and a one-hot design, the scores
    are c*alpha*delta(i-j) exactly; with V = identity, O is the probability
    matrix, which must equal the softmax of those values.  C2P uses Q with Kr,
    P2C uses K with Qr, and both index delta(i - j) (not j - i)."""
    n, D, span, nb, mp = 12, 16, 6, 6, 12
    alpha = 0.37
    R = 2 * span
    cu = np.array([0, n])
    q = np.zeros((n, 1, D))
    k = np.zeros((n, 1, D))
    qr = np.zeros((1, R, D))
    kr = np.zeros((1, R, D))
    rel = alpha * np.arange(R)
    if which == "c2p":
        q[:, 0, 0] = 1.0
        kr[0, :, 0] = rel
    else:
        k[:, 0, 0] = 1.0
        qr[0, :, 0] = rel
    v = np.zeros((n, 1, D))
    v[np.arange(n), 0, np.arange(n)] = 1.0
    o, _ = O.forward(O.Problem(cu, 1, D, span, nb, mp), q, k, v, qr, kr)
    P = o[:, 0, :n]
    c = 1 / math.sqrt(3 * D)
    dtab = O.delta_table(n, span, nb, mp)
    idx = dtab[(np.arange(n)[:, None] - np.arange(n)[None, :]) + n - 1]
    e = np.exp(c * alpha * idx - (c * alpha * idx).max(1, keepdims=True))
    np.testing.assert_allclose(P, e / e.sum(1, keepdims=True), rtol=1e-12)
    # and the matrix is constant along diagonals (it depends on i - j only)
    # up to the per-row normaliser: check the unnormalised ratios
    ratio = P[:, :-1] / P[:, 1:]
    for d in range(-n + 2, n - 1):
        dv = np.diagonal(ratio, d)
        np.testing.assert_allclose(dv, dv[0], rtol=1e-12)


def test_masked_keys_have_exactly_zero_weight_and_masked_rows_are_zero():
    B, L, H, D = 2, 10, 2, 4
    cu = np.arange(B + 1) * L
    q, k, v, qr, kr, do = _problem_inputs(cu, H, D, 4, 5)
    m = np.concatenate([(np.arange(L) < 7), (np.arange(L) < 10)]).astype(np.uint8)
    prob = O.Problem(cu, H, D, 4, 4, 8, qmask=m, kmask=m)
    v1 = v.copy()
    v2 = v.copy()
    v1[m == 0] = 0.0
    v2[m == 0] = 1e300
    o1, lse1 = O.forward(prob, q, k, v1, qr, kr)
    o2, lse2 = O.forward(prob, q, k, v2, qr, kr)
    assert np.array_equal(o1, o2) and np.array_equal(lse1, lse2)
    assert np.all(o1[m == 0] == 0.0)
    assert np.all(np.isinf(lse1[:, m == 0])) and np.all(lse1[:, m == 0] > 0)
    dq, dk, dv, dqr, dkr = O.backward(prob, q, k, v, qr, kr, do)
    assert np.all(dq[m == 0] == 0) and np.all(dk[m == 0] == 0) and np.all(dv[m == 0] == 0)


def test_packed_equals_padded_with_masks():
    lens = [9, 4, 13]
    L, H, D, span = 13, 2, 6, 4
    g = _rng(11)
    Tp = len(lens) * L
    q, k, v, do = (g.standard_normal((Tp, H, D)) for _ in range(4))
    qr, kr = (g.standard_normal((H, 2 * span, D)) for _ in range(2))
    m = np.concatenate([(np.arange(L) < n) for n in lens]).astype(np.uint8)
    cu_pad = np.arange(len(lens) + 1) * L
    pad = O.Problem(cu_pad, H, D, span, 4, 8, qmask=m, kmask=m)
    o_p, lse_p = O.forward(pad, q, k, v, qr, kr)
    g_p = O.backward(pad, q, k, v, qr, kr, do)
    sel = m.astype(bool)
    cu_pk = np.concatenate([[0], np.cumsum(lens)])
    pk = O.Problem(cu_pk, H, D, span, 4, 8)
    o_k, lse_k = O.forward(pk, q[sel], k[sel], v[sel], qr, kr)
    g_k = O.backward(pk, q[sel], k[sel], v[sel], qr, kr, do[sel])
    np.testing.assert_allclose(o_p[sel], o_k, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(lse_p[:, sel], lse_k, rtol=1e-13)
    for a, b in zip(g_p[:3], g_k[:3]):
        np.testing.assert_allclose(a[sel], b, rtol=1e-11, atol=1e-13)
    for a, b in zip(g_p[3:], g_k[3:]):
        np.testing.assert_allclose(a, b, rtol=1e-11, atol=1e-13)


# ---------------------------------------------- independent formulation

def torch_reference(prob, q, k, v, qr, kr, dout, keep=None):
    """A second formulation: dense relative products gathered by the delta
    index matrix, masked softmax, autograd for the gradients.  fp64, CPU."""
    H, D, R = prob.H, prob.D, prob.R
    c = prob.scale if prob.scale > 0 else 1 / math.sqrt(3 * D)
    tq, tk, tv, tqr, tkr = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (q, k, v, qr, kr))
    outs, lses = [], []
    for s in range(prob.nseq):
        t0, t1 = int(prob.cu[s]), int(prob.cu[s + 1])
        n = t1 - t0
        dt = torch.from_numpy(O.delta_table(max(n, 1), prob.span, prob.nb, prob.mp).astype(np.int64))
        ii = torch.arange(n)
        idx = dt[(ii[:, None] - ii[None, :]) + n - 1]
        qs, ks, vs = tq[t0:t1].transpose(0, 1), tk[t0:t1].transpose(0, 1), tv[t0:t1].transpose(0, 1)  # [H,n,D]
        a = qs @ tkr.transpose(1, 2)   # [H, n, R]   Q . Kr
        b = ks @ tqr.transpose(1, 2)   # [H, n, R]   K . Qr
        c2p = torch.gather(a, 2, idx.expand(H, n, n))
        p2c = torch.gather(b, 2, idx.t().expand(H, n, n)).transpose(1, 2)
        S = c * (qs @ ks.transpose(1, 2) + c2p + p2c)
        valid = torch.ones(n, n, dtype=torch.bool)
        if prob.qmask is not None:
            valid &= torch.from_numpy(prob.qmask[t0:t1].astype(bool))[:, None]
        if prob.kmask is not None:
            valid &= torch.from_numpy(prob.kmask[t0:t1].astype(bool))[None, :]
        rowok = valid.any(1)
        S = S.masked_fill(~valid, -math.inf)
        S = torch.where(rowok[:, None], S, torch.zeros_like(S))
        lse = torch.logsumexp(S, -1)
        P = torch.exp(S - lse[..., None]) * rowok[:, None]
        if keep is not None:
            P = P * torch.from_numpy(np.stack([keep[(s, h)] for h in range(H)])).double() / (1 - prob.p_drop)
        outs.append((P @ vs).transpose(0, 1))
        lses.append(torch.where(rowok, lse, torch.full_like(lse, math.inf)))
    o = torch.cat(outs, 0)
    lse = torch.cat(lses, 1)
    (o * torch.from_numpy(dout)).sum().backward()
    return (o.detach().numpy(), lse.detach().numpy(), tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy(),
            tqr.grad.numpy(), tkr.grad.numpy())


@pytest.mark.parametrize("case", ["padded_masked", "packed", "dropout", "far_field"])
def test_oracle_matches_autograd_formulation(case):
    H, D = 2, 8
    if case == "padded_masked":
        L, B, span, nb, mp = 20, 2, 6, 8, 16
        cu = np.arange(B + 1) * L
        m = np.concatenate([(np.arange(L) < 14), (np.arange(L) < 20)]).astype(np.uint8)
        prob = O.Problem(cu, H, D, span, nb, mp, qmask=m, kmask=m)
    elif case == "packed":
        cu = np.array([0, 7, 23, 24, 40])
        prob = O.Problem(cu, H, D, 5, 6, 12)
    elif case == "dropout":
        cu = np.array([0, 18, 30])
        prob = O.Problem(cu, H, D, 6, 8, 16, p_drop=0.3, seed=0x1234_5678_9ABC, offset=7)
    else:  # sequence much longer than the relative window: clamped and log regions
        cu = np.array([0, 64])
        prob = O.Problem(cu, H, D, 4, 4, 8)
    q, k, v, qr, kr, do = _problem_inputs(prob.cu, H, D, prob.span, 21)
    keep = None
    if prob.p_drop > 0:
        keep = {(s, h): O.keep_mask(prob, s, h) for s in range(prob.nseq) for h in range(H)}
    ref = torch_reference(prob, q, k, v, qr, kr, do, keep)
    o, lse = O.forward(prob, q, k, v, qr, kr)
    grads = O.backward(prob, q, k, v, qr, kr, do)
    np.testing.assert_allclose(o, ref[0], rtol=1e-11, atol=1e-12)
    fin = np.isfinite(ref[1])
    assert np.array_equal(fin, np.isfinite(lse))
    np.testing.assert_allclose(lse[fin], ref[1][fin], rtol=1e-12)
    for name, a, b in zip(["dq", "dk", "dv", "dqr", "dkr"], grads, ref[2:]):
        np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-11, err_msg=name)


# ------------------------------------------------------ finite differences

def _loss(prob, w, q, k, v, qr, kr):
    o, _ = O.forward(prob, q, k, v, qr, kr)
    return float((o * w).sum())


@pytest.mark.parametrize("case", ["plain", "masked_dropout"])
def test_every_gradient_element_by_central_differences(case):
    H, D = 2, 3
    if case == "plain":
        cu = np.array([0, 6, 9])
        prob = O.Problem(cu, H, D, 4, 4, 8)
    else:
        cu = np.array([0, 7, 14])
        m = np.concatenate([(np.arange(7) < 5), (np.arange(7) < 7)]).astype(np.uint8)
        prob = O.Problem(cu, H, D, 4, 4, 8, qmask=m, kmask=m, p_drop=0.25, seed=99, offset=3)
    q, k, v, qr, kr, w = _problem_inputs(prob.cu, H, D, prob.span, 5)
    grads = O.backward(prob, q, k, v, qr, kr, w)
    names = ["q", "k", "v", "qr", "kr"]
    gmap = dict(zip(["q", "k", "v", "qr", "kr"], [grads[0], grads[1], grads[2], grads[3], grads[4]]))
    args = dict(q=q, k=k, v=v, qr=qr, kr=kr)
    eps = 1e-5
    for nm in names:
        a = args[nm]
        fd = np.zeros_like(a)
        for ix in np.ndindex(a.shape):
            old = a[ix]
            a[ix] = old + eps
            lp = _loss(prob, w, **args)
            a[ix] = old - eps
            lm = _loss(prob, w, **args)
            a[ix] = old
            fd[ix] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(gmap[nm], fd, rtol=1e-6, atol=1e-8, err_msg=nm)


def test_directional_derivatives_on_tiny_fp32_workload_shape():
    """Random directional derivatives on the B=1, H=2, L=128, D=64 shape."""
    cu = np.array([0, 128])
    H, D, span = 2, 64, 64
    prob = O.Problem(cu, H, D, span, 64, 128)
    q, k, v, qr, kr, w = _problem_inputs(cu, H, D, span, 8)
    grads = O.backward(prob, q, k, v, qr, kr, w)
    g = _rng(9)
    args = [q, k, v, qr, kr]
    gl = [grads[0], grads[1], grads[2], grads[3], grads[4]]
    dirs = [g.standard_normal(a.shape) for a in args]
    eps = 1e-5
    lp = _loss(prob, w, *[a + eps * d for a, d in zip(args, dirs)])
    lm = _loss(prob, w, *[a - eps * d for a, d in zip(args, dirs)])
    fd = (lp - lm) / (2 * eps)
    an = sum(float((gg * d).sum()) for gg, d in zip(gl, dirs))
    assert abs(fd - an) <= 1e-6 * max(1.0, abs(an))


# -------------------------------------------------------------- invariants

def test_gradient_invariants():
    cu = np.array([0, 40, 64])
    H, D, span = 2, 8, 8
    prob = O.Problem(cu, H, D, span, 8, 32)
    q, k, v, qr, kr, do = _problem_inputs(cu, H, D, span, 13)
    dq, dk, dv, dqr, dkr = O.backward(prob, q, k, v, qr, kr, do)
    # a constant shift of every Kr row moves each score row by a constant
    np.testing.assert_allclose(dkr.sum(1), 0.0, atol=1e-10)
    # probability rows sum to one: sum_j dV_j = sum_i dO_i per sequence
    for s in range(prob.nseq):
        t0, t1 = cu[s], cu[s + 1]
        np.testing.assert_allclose(dv[t0:t1].sum(0), do[t0:t1].sum(0), rtol=1e-11, atol=1e-11)
    # sum_j dZ_ij = 0 per row  <=>  shifting every K_j by a constant vector
    # leaves O unchanged  <=>  sum_j dK_j = sum_i (...)Qr-part only when Qr=0
    prob0 = O.Problem(cu, H, D, span, 8, 32)
    qr0 = np.zeros_like(qr)
    _, dk0, _, _, _ = O.backward(prob0, q, k, v, qr0, kr, do)
    for s in range(prob.nseq):
        t0, t1 = cu[s], cu[s + 1]
        np.testing.assert_allclose(dk0[t0:t1].sum(0), 0.0, atol=1e-10)
    # relative rows that no token pair reaches get exactly zero gradient
    # (span 64 with sequences of at most 40 tokens leaves both ends unused)
    span2 = 64
    prob2 = O.Problem(cu, H, D, span2, 64, 128)
    q2, k2, v2, qr2, kr2, do2 = _problem_inputs(cu, H, D, span2, 14)
    _, _, _, dqr2, dkr2 = O.backward(prob2, q2, k2, v2, qr2, kr2, do2)
    tab = O.delta_table(40, span2, 64, 128)
    reached = np.zeros(2 * span2, bool)
    reached[np.unique(tab)] = True
    assert reached.sum() < 2 * span2 and reached[np.unique(tab)].all()
    assert np.all(dkr2[:, ~reached] == 0) and np.all(dqr2[:, ~reached] == 0)
    assert np.all(np.abs(dkr2[:, reached]).sum(-1) > 0)


def test_plain_attention_gradients_match_library():
    B, L, H, D = 2, 16, 2, 8
    cu = np.arange(B + 1) * L
    q, k, v, qr, kr, do = _problem_inputs(cu, H, D, 4, 17)
    qr[:] = 0
    kr[:] = 0
    dq, dk, dv, _, _ = O.backward(O.Problem(cu, H, D, 4, 4, 8), q, k, v, qr, kr, do)
    t = lambda a: torch.tensor(a.reshape(B, L, H, D)).permute(0, 2, 1, 3).requires_grad_(True)
    tq, tk, tv = t(q), t(k), t(v)
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=1 / math.sqrt(3 * D))
    (o * torch.tensor(do.reshape(B, L, H, D)).permute(0, 2, 1, 3)).sum().backward()
    for a, b in [(dq, tq), (dk, tk), (dv, tv)]:
        np.testing.assert_allclose(a.reshape(B, L, H, D), b.grad.permute(0, 2, 1, 3).numpy(), rtol=1e-11,
                                   atol=1e-12)


# ----------------------------------------------------------------- dropout

def test_dropout_statistics_and_p0():
    cu = np.array([0, 256])
    prob = O.Problem(cu, 2, 4, 8, 8, 16, p_drop=0.1, seed=2024, offset=1)
    m = np.concatenate([O.keep_mask(prob, 0, h).ravel() for h in range(2)])
    n = m.size
    mean = m.mean()
    # binomial 6-sigma bound around 0.9
    assert abs(mean - 0.9) < 6 * math.sqrt(0.9 * 0.1 / n)
    # different heads / offsets give different masks
    prob2 = O.Problem(cu, 2, 4, 8, 8, 16, p_drop=0.1, seed=2024, offset=2)
    assert not np.array_equal(O.keep_mask(prob, 0, 0), O.keep_mask(prob2, 0, 0))
    assert not np.array_equal(O.keep_mask(prob, 0, 0), O.keep_mask(prob, 0, 1))
    # adjacent words of one Philox block are not correlated
    a = O.keep_mask(prob, 0, 0).astype(float)
    cc = np.corrcoef(a[:, 0::4].ravel(), a[:, 1::4].ravel())[0, 1]
    assert abs(cc) < 0.05
    # threshold is floor((1-p) 2^32); p = 0 keeps everything
    assert O.keep_threshold(0.1) == math.floor(0.9 * 2 ** 32)
    assert O.keep_threshold(0.0) == 2 ** 32
    q, k, v, qr, kr, _ = _problem_inputs(cu, 2, 4, 8, 3)
    p0 = O.Problem(cu, 2, 4, 8, 8, 16, p_drop=0.0, seed=5)
    pn = O.Problem(cu, 2, 4, 8, 8, 16)
    assert np.array_equal(O.forward(p0, q, k, v, qr, kr)[0], O.forward(pn, q, k, v, qr, kr)[0])


def test_philox_output_words_are_uniform_and_key_sensitive():
    words = np.array([O.philox4x32_10([i, 0, 0, 0], [1, 2]) for i in range(2000)], dtype=np.uint64)
    # uniform bits: every bit position set about half the time
    bits = ((words[..., None] >> np.arange(32, dtype=np.uint64)) & 1).reshape(-1, 32)
    assert np.all(np.abs(bits.mean(0) - 0.5) < 0.03)
    # one-bit change of the counter or the key flips about half the output bits
    base = O.philox4x32_10([5, 6, 7, 8], [9, 10])
    for ctr, key in [([4, 6, 7, 8], [9, 10]), ([5, 6, 7, 8], [9, 11])]:
        x = O.philox4x32_10(ctr, key) ^ base
        flips = sum(bin(int(w)).count("1") for w in x)
        assert 40 < flips < 88


def test_sampled_backward_matches_full_backward():
    """The sampled-row routine used for full-size checks agrees with the full
    oracle backward (masks and dropout included)."""
    cu = np.array([0, 40, 90])
    H, D, span = 2, 8, 6
    m = np.ones(90, np.uint8)
    m[33:40] = 0
    prob = O.Problem(cu, H, D, span, 8, 16, qmask=m, kmask=m, p_drop=0.2, seed=77, offset=2)
    q, k, v, qr, kr, do = _problem_inputs(cu, H, D, span, 31)
    dq, dk, dv, _, _ = O.backward(prob, q, k, v, qr, kr, do)
    rows = [0, 5, 33, 39]
    cols = [1, 20, 35, 49]
    for s in range(2):
        for h in range(H):
            t0 = cu[s]
            n = cu[s + 1] - t0
            rr = [r for r in rows if r < n]
            cc = [c for c in cols if c < n]
            sq, sk, sv = O.backward_sample(prob, s, h, rr, cc, q, k, v, qr, kr, do)
            np.testing.assert_allclose(sq, dq[t0 + np.array(rr), h], rtol=1e-10, atol=1e-12)
            np.testing.assert_allclose(sk, dk[t0 + np.array(cc), h], rtol=1e-10, atol=1e-12)
            np.testing.assert_allclose(sv, dv[t0 + np.array(cc), h], rtol=1e-10, atol=1e-12)
