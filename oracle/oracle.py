"""Python face of the fp64 CPU oracle (``df_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline leg use it.  Nothing on the product path imports this module.

Every function takes and returns numpy arrays in the oracle's layouts:
Q, K, V, dO, O, dQ, dK, dV ``[T, H, D]`` float64, Qr, Kr, dQr, dKr
``[H, R, D]`` float64, LSE ``[H, T]`` float64, masks ``[T]`` uint8, and
``cu`` the ``[nseq + 1]`` token offsets of the sequences.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "df_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile df_oracle.c into liboracle.so (gcc, OpenMP, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Cfg(ctypes.Structure):
    _fields_ = [
        ("nseq", ctypes.c_int),
        ("cu", ctypes.POINTER(ctypes.c_int)),
        ("T", ctypes.c_int),
        ("H", ctypes.c_int),
        ("D", ctypes.c_int),
        ("span", ctypes.c_int),
        ("nb", ctypes.c_int),
        ("mp", ctypes.c_int),
        ("qmask", ctypes.POINTER(ctypes.c_ubyte)),
        ("kmask", ctypes.POINTER(ctypes.c_ubyte)),
        ("scale", ctypes.c_double),
        ("p_drop", ctypes.c_double),
        ("seed", ctypes.c_uint64),
        ("offset", ctypes.c_uint32),
    ]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            dp = ctypes.POINTER(ctypes.c_double)
            cp = ctypes.POINTER(_Cfg)
            lib.orc_bucket.restype = ctypes.c_long
            lib.orc_bucket.argtypes = [ctypes.c_long, ctypes.c_int, ctypes.c_int]
            lib.orc_delta.restype = ctypes.c_long
            lib.orc_delta.argtypes = [ctypes.c_long, ctypes.c_int, ctypes.c_int, ctypes.c_int]
            lib.orc_delta_table.argtypes = [ctypes.c_int] * 4 + [ctypes.POINTER(ctypes.c_int32)]
            lib.orc_philox4x32_10.argtypes = [ctypes.POINTER(ctypes.c_uint32)] * 3
            lib.orc_philox4x32_10.restype = None
            lib.orc_keep_threshold.restype = ctypes.c_uint64
            lib.orc_keep_threshold.argtypes = [ctypes.c_double]
            lib.orc_keep_mask.argtypes = [cp, ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_ubyte)]
            lib.orc_forward_pair.argtypes = [cp, ctypes.c_int, ctypes.c_int] + [dp] * 7 + [
                ctypes.c_int, ctypes.POINTER(ctypes.c_int)]
            lib.orc_forward.argtypes = [cp] + [dp] * 7 + [ctypes.c_int]
            lib.orc_backward_pair.argtypes = [cp, ctypes.c_int, ctypes.c_int] + [dp] * 11
            lib.orc_backward.argtypes = [cp] + [dp] * 11 + [ctypes.c_int]
            lib.orc_backward_sample.argtypes = [cp, ctypes.c_int, ctypes.c_int] + [dp] * 6 + [
                ctypes.c_int, ctypes.POINTER(ctypes.c_int), ctypes.c_int, ctypes.POINTER(ctypes.c_int), dp, dp, dp]
            lib.orc_step_rows_sample.restype = ctypes.c_double
            lib.orc_step_rows_sample.argtypes = [cp, ctypes.c_int, ctypes.POINTER(ctypes.c_int), ctypes.c_int,
                                                 ctypes.c_int] + [dp] * 6 + [ctypes.c_int]
            lib.orc_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().orc_max_threads())


def _dp(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


class Problem:
    """Shapes and options of one attention call, in the oracle's terms."""

    def __init__(self, cu, H, D, span, nb, mp, qmask=None, kmask=None, scale=0.0,
                 p_drop=0.0, seed=0, offset=0):
        self.cu = np.ascontiguousarray(np.asarray(cu, dtype=np.int32))
        self.nseq = len(self.cu) - 1
        self.T = int(self.cu[-1])
        self.H, self.D = int(H), int(D)
        self.span, self.nb, self.mp = int(span), int(nb), int(mp)
        self.R = 2 * self.span
        self.qmask = None if qmask is None else np.ascontiguousarray(np.asarray(qmask, dtype=np.uint8))
        self.kmask = None if kmask is None else np.ascontiguousarray(np.asarray(kmask, dtype=np.uint8))
        self.scale = float(scale)
        self.p_drop = float(p_drop)
        self.seed = int(seed)
        self.offset = int(offset)

    def _cfg(self):
        c = _Cfg()
        c.nseq = self.nseq
        c.cu = self.cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int))
        c.T, c.H, c.D = self.T, self.H, self.D
        c.span, c.nb, c.mp = self.span, self.nb, self.mp
        ub = ctypes.POINTER(ctypes.c_ubyte)
        c.qmask = self.qmask.ctypes.data_as(ub) if self.qmask is not None else ub()
        c.kmask = self.kmask.ctypes.data_as(ub) if self.kmask is not None else ub()
        c.scale = self.scale
        c.p_drop = self.p_drop
        c.seed = self.seed & ((1 << 64) - 1)
        c.offset = self.offset & 0xFFFFFFFF
        return c


def bucket(r: int, nb: int, mp: int) -> int:
    return int(_load().orc_bucket(int(r), int(nb), int(mp)))


def delta(r: int, span: int, nb: int, mp: int) -> int:
    return int(_load().orc_delta(int(r), int(span), int(nb), int(mp)))


def delta_table(L: int, span: int, nb: int, mp: int) -> np.ndarray:
    """delta(r) for r = -(L-1) .. L-1 (index r + L - 1), int32."""
    out = np.zeros(2 * L - 1, dtype=np.int32)
    rc = _load().orc_delta_table(L, span, nb, mp, out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)))
    if rc != 0:
        raise ValueError("bad delta-table arguments")
    return out


def philox4x32_10(ctr, key) -> np.ndarray:
    c = np.ascontiguousarray(np.asarray(ctr, dtype=np.uint32))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint32))
    o = np.zeros(4, dtype=np.uint32)
    u32 = ctypes.POINTER(ctypes.c_uint32)
    _load().orc_philox4x32_10(c.ctypes.data_as(u32), k.ctypes.data_as(u32), o.ctypes.data_as(u32))
    return o


def keep_threshold(p: float) -> int:
    return int(_load().orc_keep_threshold(float(p)))


def keep_mask(prob: Problem, s: int, h: int) -> np.ndarray:
    n = int(prob.cu[s + 1] - prob.cu[s])
    out = np.zeros((n, n), dtype=np.uint8)
    c = prob._cfg()
    _load().orc_keep_mask(ctypes.byref(c), s, h, out.ctypes.data_as(ctypes.POINTER(ctypes.c_ubyte)))
    return out


def forward(prob: Problem, q, k, v, qr, kr, nthreads: int = 0):
    """Returns (O [T,H,D], LSE [H,T]) in float64."""
    q, k, v, qr, kr = map(_f64, (q, k, v, qr, kr))
    o = np.zeros((prob.T, prob.H, prob.D))
    lse = np.zeros((prob.H, prob.T))
    c = prob._cfg()
    rc = _load().orc_forward(ctypes.byref(c), _dp(q), _dp(k), _dp(v), _dp(qr), _dp(kr), _dp(o), _dp(lse),
                             int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle forward failed")
    return o, lse


def forward_rows(prob: Problem, s: int, h: int, rows, q, k, v, qr, kr):
    """O and LSE of selected rows (positions inside sequence s) of head h.
    Returns (O [len(rows), D], LSE [len(rows)])."""
    q, k, v, qr, kr = map(_f64, (q, k, v, qr, kr))
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
    o = np.zeros((prob.T, prob.H, prob.D))
    lse = np.zeros((prob.H, prob.T))
    c = prob._cfg()
    rc = _load().orc_forward_pair(ctypes.byref(c), int(s), int(h), _dp(q), _dp(k), _dp(v), _dp(qr), _dp(kr),
                                  _dp(o), _dp(lse), len(rows), rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int)))
    if rc != 0:
        raise RuntimeError("oracle forward_rows failed")
    t0 = int(prob.cu[s])
    return o[t0 + rows, h, :].copy(), lse[h, t0 + rows].copy()


def backward(prob: Problem, q, k, v, qr, kr, dout, nthreads: int = 0):
    """Returns (dQ, dK, dV [T,H,D], dQr, dKr [H,R,D]) in float64."""
    q, k, v, qr, kr, dout = map(_f64, (q, k, v, qr, kr, dout))
    dq = np.zeros((prob.T, prob.H, prob.D))
    dk = np.zeros_like(dq)
    dv = np.zeros_like(dq)
    dqr = np.zeros((prob.H, prob.R, prob.D))
    dkr = np.zeros_like(dqr)
    c = prob._cfg()
    rc = _load().orc_backward(ctypes.byref(c), _dp(q), _dp(k), _dp(v), _dp(qr), _dp(kr), _dp(dout), _dp(dq),
                              _dp(dk), _dp(dv), _dp(dqr), _dp(dkr), int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle backward failed")
    return dq, dk, dv, dqr, dkr


def backward_pair(prob: Problem, s: int, h: int, q, k, v, qr, kr, dout):
    """Backward of one (sequence, head) pair.  Returns (dQ, dK, dV) rows of
    that pair ([n, D] each) and the pair's contribution to dQr, dKr ([R, D])."""
    q, k, v, qr, kr, dout = map(_f64, (q, k, v, qr, kr, dout))
    dq = np.zeros((prob.T, prob.H, prob.D))
    dk = np.zeros_like(dq)
    dv = np.zeros_like(dq)
    pk = np.zeros((prob.R, prob.D))
    pq = np.zeros_like(pk)
    c = prob._cfg()
    rc = _load().orc_backward_pair(ctypes.byref(c), int(s), int(h), _dp(q), _dp(k), _dp(v), _dp(qr), _dp(kr),
                                   _dp(dout), _dp(dq), _dp(dk), _dp(dv), _dp(pk), _dp(pq))
    if rc != 0:
        raise RuntimeError("oracle backward_pair failed")
    t0, t1 = int(prob.cu[s]), int(prob.cu[s + 1])
    return dq[t0:t1, h].copy(), dk[t0:t1, h].copy(), dv[t0:t1, h].copy(), pq, pk


def backward_sample(prob: Problem, s: int, h: int, rows, cols, q, k, v, qr, kr, dout):
    """dQ of selected rows and dK, dV of selected keys of one (sequence,
    head) pair (positions inside the sequence)."""
    q, k, v, qr, kr, dout = map(_f64, (q, k, v, qr, kr, dout))
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
    cols = np.ascontiguousarray(np.asarray(cols, dtype=np.int32))
    dq = np.zeros((len(rows), prob.D))
    dk = np.zeros((len(cols), prob.D))
    dv = np.zeros((len(cols), prob.D))
    c = prob._cfg()
    ip = ctypes.POINTER(ctypes.c_int)
    rc = _load().orc_backward_sample(ctypes.byref(c), int(s), int(h), _dp(q), _dp(k), _dp(v), _dp(qr), _dp(kr),
                                     _dp(dout), len(rows), rows.ctypes.data_as(ip), len(cols),
                                     cols.ctypes.data_as(ip), _dp(dq), _dp(dk), _dp(dv))
    if rc != 0:
        raise RuntimeError("oracle backward_sample failed")
    return dq, dk, dv


def step_rows_sample(prob: Problem, pairs, r0: int, r1: int, q, k, v, qr, kr, dout, nthreads: int = 0) -> float:
    """Forward + backward work of query rows [r0, r1) of the listed (s, h)
    pairs, one pair per thread; returns a checksum."""
    q, k, v, qr, kr, dout = map(_f64, (q, k, v, qr, kr, dout))
    pr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1))
    c = prob._cfg()
    return float(_load().orc_step_rows_sample(ctypes.byref(c), len(pr) // 2, pr.ctypes.data_as(ctypes.POINTER(ctypes.c_int)),
                                              int(r0), int(r1), _dp(q), _dp(k), _dp(v), _dp(qr), _dp(kr), _dp(dout),
                                              int(nthreads)))


# --------------------------------------------------------------------------
# The steps on either side of the attention: the fused QKV projection and
# the relative-position projections (DeBERTa-v2/v3 with shared attention
# keys), written from their definitions in float64 numpy.  "DisentangledFlash",
# section "Status" (the fused QKV projection) and section "Hugging Face usage"
# (the query / key / value and relative-position projections in the autograd
# graph).  The backward functions are the plain calculus of the forward ones.

def qkv_projection(x, w, b=None):
    """[Q; K; V] = x W_j^T + b_j: x [T, C], w [3, HD, C], b [3, HD] -> [3, T, HD]."""
    x, w = _f64(x), _f64(w)
    y = np.einsum("tc,jnc->jtn", x, w)
    if b is not None:
        y = y + _f64(b)[:, None, :]
    return y


def qkv_projection_backward(x, w, dy):
    """Gradients of qkv_projection for dy [3, T, HD]: dx [T, C] = sum_j dy_j W_j,
    dw [3, HD, C] = dy_j^T x, db [3, HD] = sum_t dy_j[t]."""
    x, w, dy = _f64(x), _f64(w), _f64(dy)
    dx = np.einsum("jtn,jnc->tc", dy, w)
    dw = np.einsum("jtn,tc->jnc", dy, x)
    db = dy.sum(axis=1)
    return dx, dw, db


def layer_norm(x, gamma, beta, eps):
    """Row-wise layer norm of x [R, C]: (x - mean) / sqrt(var + eps) gamma + beta
    (biased variance); also returns mean and 1/std."""
    x = _f64(x)
    mean = x.mean(axis=1, keepdims=True)
    var = ((x - mean) ** 2).mean(axis=1, keepdims=True)
    rstd = 1.0 / np.sqrt(var + eps)
    return (x - mean) * rstd * _f64(gamma) + _f64(beta), mean[:, 0], rstd[:, 0]


def rel_projection(rel, gamma, beta, eps, w, b, H, D):
    """E = LayerNorm(rel); Qr[h] = E W_q[h]^T + b_q[h], Kr[h] = E W_k[h]^T + b_k[h]
    with W_q = w[0], W_k = w[1] ([HD, C], head h = rows h D .. h D + D).
    Returns (E [R, C], Qr [H, R, D], Kr [H, R, D])."""
    e, _, _ = layer_norm(rel, gamma, beta, eps)
    w = _f64(w)
    out = []
    for j in (0, 1):
        y = e @ w[j].T                                   # [R, HD]
        if b is not None:
            y = y + _f64(b)[j][None, :]
        out.append(y.reshape(e.shape[0], H, D).transpose(1, 0, 2))
    return e, out[0], out[1]


def rel_projection_backward(rel, gamma, beta, eps, w, dqr, dkr, H, D):
    """Gradients of rel_projection for dqr, dkr [H, R, D]: drel [R, C],
    dgamma [C], dbeta [C], dw_qk [2, HD, C], db_qk [2, HD]."""
    x = _f64(rel)
    e, mean, rstd = layer_norm(x, gamma, beta, eps)
    w = _f64(w)
    R, C = x.shape
    g_rows = [_f64(d).transpose(1, 0, 2).reshape(R, H * D) for d in (dqr, dkr)]   # [R, HD]
    dw = np.stack([g.T @ e for g in g_rows])
    db = np.stack([g.sum(axis=0) for g in g_rows])
    de = g_rows[0] @ w[0] + g_rows[1] @ w[1]              # dL/dE  [R, C]
    xh = (x - mean[:, None]) * rstd[:, None]
    dbeta = de.sum(axis=0)
    dgamma = (de * xh).sum(axis=0)
    g = de * _f64(gamma)
    drel = rstd[:, None] * (g - g.mean(axis=1, keepdims=True) - xh * (g * xh).mean(axis=1, keepdims=True))
    return drel, dgamma, dbeta, dw, db
