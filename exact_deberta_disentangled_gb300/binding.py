"""Thin Python binding of libdfattn's C ABI (include/df_attn.h).

Argument marshalling only: tensors are passed to the library as raw device
pointers and every step of the computation runs in the library's CUDA
kernels.  PyTorch is used for device memory and streams.  If the library has
not been built (``exact_deberta_disentangled_gb300.build.build()``), loading
it raises -- there is no other implementation to fall back on.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import threading
from dataclasses import dataclass
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdfattn.so")

DF_OK, DF_ERR_INVALID_ARG, DF_ERR_UNSUPPORTED, DF_ERR_WORKSPACE, DF_ERR_CUDA, DF_ERR_TIMEOUT, DF_ERR_DEVICE_ARG = range(7)
DTYPE_CODE = {torch.bfloat16: 0, torch.float16: 1, torch.float32: 2}
DF_FP32_FAST = 3   # fp32 tensors, inputs rounded to fp16 for the tensor-core path

EXPORTS = ["df_attn_workspace_size", "df_attn_fwd", "df_attn_bwd", "df_attn_step_host_arena_size",
           "df_attn_step_host", "df_rel_index_table", "df_get_device_error", "df_status_string", "df_version",
           "df_attn_set_profile_events", "df_attn_fwd_noalloc", "df_attn_debug_inject_stall",
           "df_dropout_keep_mask", "df_attn_fwd_inference", "df_attn_fwd_noalloc_device_error",
           "df_pack_workspace_size", "df_pack_info", "df_pack_rows", "df_unpack_rows",
           "df_qkv_proj_fwd", "df_qkv_proj_bwd", "df_qkv_proj_workspace_size", "df_rel_proj_workspace_size", "df_rel_proj_fwd",
           "df_rel_proj_bwd", "df_attn_band_bias_size"]


class DfError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)}")


class Params(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32), ("L", ctypes.c_int32), ("H", ctypes.c_int32), ("D", ctypes.c_int32),
        ("cu_seqlens", ctypes.c_void_p),
        ("total_tokens", ctypes.c_int32),
        ("att_span", ctypes.c_int32),
        ("position_buckets", ctypes.c_int32),
        ("max_relative_positions", ctypes.c_int32),
        ("query_mask", ctypes.c_void_p),
        ("key_mask", ctypes.c_void_p),
        ("dropout_p", ctypes.c_float),
        ("philox_seed", ctypes.c_uint64),
        ("philox_offset", ctypes.c_uint64),
        ("softmax_scale", ctypes.c_float),
        ("dtype", ctypes.c_int),
        ("band_bias", ctypes.c_void_p),
    ]


_lib = None
_lock = threading.Lock()


def load():
    """Load libdfattn.so (raises if it is missing)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with exact_deberta_disentangled_gb300.build.build()")
            _lib = _configure(ctypes.CDLL(LIB_PATH))
    return _lib


@contextlib.contextmanager
def checked_library(path: str):
    """Route every call of this module to the library at `path` (a build
    with DF_CHECKED, see build.build(checked=True)) inside the block."""
    global _lib
    lib = _configure(ctypes.CDLL(path))
    with _lock:
        prev, _lib = _lib, lib
    try:
        yield lib
    finally:
        with _lock:
            _lib = prev


def _configure(lib):
    """Declare the argument and result types of the library's entry points."""
    vp, sz = ctypes.c_void_p, ctypes.c_size_t
    P = ctypes.POINTER(Params)
    lib.df_attn_workspace_size.restype = sz
    lib.df_attn_workspace_size.argtypes = [P, ctypes.c_int]
    lib.df_attn_band_bias_size.restype = sz
    lib.df_attn_band_bias_size.argtypes = [P]
    lib.df_attn_fwd.restype = ctypes.c_int
    lib.df_attn_fwd.argtypes = [P] + [vp] * 7 + [vp, sz, vp]
    lib.df_attn_fwd_inference.restype = ctypes.c_int
    lib.df_attn_fwd_inference.argtypes = [P] + [vp] * 6 + [vp, sz, vp]
    lib.df_attn_bwd.restype = ctypes.c_int
    lib.df_attn_bwd.argtypes = [P] + [vp] * 13 + [vp, sz, vp]
    lib.df_attn_step_host_arena_size.restype = sz
    lib.df_attn_step_host_arena_size.argtypes = [P]
    lib.df_attn_step_host.restype = ctypes.c_int
    lib.df_attn_step_host.argtypes = [P] + [vp] * 13 + [vp, sz, vp]
    lib.df_rel_index_table.restype = ctypes.c_int
    lib.df_rel_index_table.argtypes = [ctypes.c_int32] * 4 + [vp, vp]
    lib.df_get_device_error.restype = ctypes.c_int
    lib.df_get_device_error.argtypes = [vp, vp]
    lib.df_status_string.restype = ctypes.c_char_p
    lib.df_status_string.argtypes = [ctypes.c_int]
    lib.df_version.restype = ctypes.c_char_p
    lib.df_attn_fwd_noalloc.restype = ctypes.c_int
    lib.df_attn_fwd_noalloc.argtypes = [P] + [vp] * 7 + [vp]
    lib.df_attn_fwd_noalloc_device_error.restype = ctypes.c_int
    lib.df_attn_fwd_noalloc_device_error.argtypes = [vp]
    lib.df_dropout_keep_mask.restype = ctypes.c_int
    lib.df_dropout_keep_mask.argtypes = [P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, vp, vp]
    lib.df_attn_debug_inject_stall.restype = ctypes.c_int
    lib.df_attn_debug_inject_stall.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_uint64, ctypes.c_uint32]
    lib.df_pack_workspace_size.restype = sz
    lib.df_pack_workspace_size.argtypes = [ctypes.c_int32]
    lib.df_pack_info.restype = ctypes.c_int
    lib.df_pack_info.argtypes = [vp, ctypes.c_int32, ctypes.c_int32, vp, vp, vp, vp, sz, vp]
    lib.df_pack_rows.restype = ctypes.c_int
    lib.df_pack_rows.argtypes = [vp, ctypes.c_int32, vp, vp, ctypes.c_int32, sz, vp, vp]
    lib.df_unpack_rows.restype = ctypes.c_int
    lib.df_unpack_rows.argtypes = [vp, vp, vp, ctypes.c_int32, sz, ctypes.c_int32, vp, vp]
    i32 = ctypes.c_int32
    lib.df_qkv_proj_fwd.restype = ctypes.c_int
    lib.df_qkv_proj_fwd.argtypes = [i32, i32, i32, ctypes.c_int, vp, vp, vp, vp, vp]
    lib.df_qkv_proj_bwd.restype = ctypes.c_int
    lib.df_qkv_proj_bwd.argtypes = [i32, i32, i32, ctypes.c_int, vp, vp, vp, vp, vp, vp, i32, vp, sz, vp]
    lib.df_qkv_proj_workspace_size.restype = sz
    lib.df_qkv_proj_workspace_size.argtypes = [i32]
    lib.df_rel_proj_workspace_size.restype = sz
    lib.df_rel_proj_workspace_size.argtypes = [i32] * 4
    lib.df_rel_proj_fwd.restype = ctypes.c_int
    lib.df_rel_proj_fwd.argtypes = [i32] * 4 + [ctypes.c_int, vp, vp, vp, ctypes.c_float, vp, vp, vp, vp,
                                                vp, vp, vp]
    lib.df_rel_proj_bwd.restype = ctypes.c_int
    lib.df_rel_proj_bwd.argtypes = [i32] * 4 + [ctypes.c_int] + [vp] * 12 + [i32, vp, sz, vp]
    lib.df_attn_set_profile_events.restype = ctypes.c_int
    lib.df_attn_set_profile_events.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_int]
    return lib


def status_string(code: int) -> str:
    return load().df_status_string(int(code)).decode()


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


@dataclass
class Geometry:
    """Attention call geometry: B sequences of (at most) L tokens."""
    B: int
    L: int
    H: int
    D: int
    span: int
    nb: int
    mp: int
    cu_seqlens: Optional[torch.Tensor] = None   # device int32 [B+1] (packed layout)
    total_tokens: int = 0
    query_mask: Optional[torch.Tensor] = None   # device uint8 [B*L] (padded layout)
    key_mask: Optional[torch.Tensor] = None
    dropout_p: float = 0.0
    seed: int = 0
    offset: int = 0
    scale: float = 0.0
    band_bias: Optional[torch.Tensor] = None    # saved band bias (device uint8, band_bias_size bytes)
    fp32_fast: bool = False   # fp32 tensors: the fast mode (DF_FP32_FAST) instead of strict fp32

    @property
    def R(self):
        return 2 * self.span

    @property
    def T(self):
        return self.total_tokens if self.cu_seqlens is not None else self.B * self.L

    def params(self, dtype: torch.dtype) -> Params:
        p = Params()
        p.B, p.L, p.H, p.D = self.B, self.L, self.H, self.D
        p.cu_seqlens = None if self.cu_seqlens is None else self.cu_seqlens.data_ptr()
        p.total_tokens = self.total_tokens
        p.att_span, p.position_buckets, p.max_relative_positions = self.span, self.nb, self.mp
        p.query_mask = None if self.query_mask is None else self.query_mask.data_ptr()
        p.key_mask = None if self.key_mask is None else self.key_mask.data_ptr()
        p.dropout_p = self.dropout_p
        p.philox_seed = self.seed & ((1 << 64) - 1)
        p.philox_offset = self.offset
        p.softmax_scale = self.scale
        p.dtype = DF_FP32_FAST if dtype == torch.float32 and self.fp32_fast else DTYPE_CODE[dtype]
        p.band_bias = None if self.band_bias is None else self.band_bias.data_ptr()
        return p

    def lse_shape(self):
        return (self.H, self.T) if self.cu_seqlens is not None else (self.B, self.H, self.L)


def workspace_size(g: Geometry, dtype: torch.dtype, backward: bool) -> int:
    p = g.params(dtype)
    return int(load().df_attn_workspace_size(ctypes.byref(p), 1 if backward else 0))


def band_bias_size(g: Geometry, dtype: torch.dtype) -> int:
    p = g.params(dtype)
    return int(load().df_attn_band_bias_size(ctypes.byref(p)))


def alloc_band_bias(g: Geometry, dtype: torch.dtype, device="cuda") -> torch.Tensor:
    """A saved-band-bias buffer for g (set g.band_bias to it before the forward)."""
    return torch.empty(max(band_bias_size(g, dtype), 16), dtype=torch.uint8, device=device)


def alloc_workspace(g: Geometry, dtype: torch.dtype, backward: bool, device="cuda") -> torch.Tensor:
    n = workspace_size(g, dtype, backward)
    if n == 0:
        raise DfError(DF_ERR_INVALID_ARG, "df_attn_workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=device)


def attn_fwd(g: Geometry, q, k, v, qr, kr, out=None, lse=None, workspace=None, stream=None, check=True):
    """Forward through df_attn_fwd; returns (out, lse, workspace)."""
    dt = q.dtype
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(g.lse_shape(), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = alloc_workspace(g, dt, False, q.device)
    p = g.params(dt)
    rc = load().df_attn_fwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(qr), _ptr(kr), _ptr(out), _ptr(lse),
                            _ptr(workspace), workspace.numel(), _stream(stream))
    if check and rc != DF_OK:
        raise DfError(rc, "df_attn_fwd")
    return out, lse, workspace


def attn_fwd_inference(g: Geometry, q, k, v, qr, kr, out=None, workspace=None, stream=None, check=True):
    """Inference forward (no LSE) through df_attn_fwd_inference; returns (out, workspace)."""
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = alloc_workspace(g, q.dtype, False, q.device)
    p = g.params(q.dtype)
    rc = load().df_attn_fwd_inference(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(qr), _ptr(kr), _ptr(out),
                                      _ptr(workspace), workspace.numel(), _stream(stream))
    if check and rc != DF_OK:
        raise DfError(rc, "df_attn_fwd_inference")
    return out, workspace


def attn_bwd(g: Geometry, q, k, v, qr, kr, out, lse, dout, grads=None, workspace=None, stream=None, check=True):
    """Backward through df_attn_bwd; returns ((dq, dk, dv, dqr, dkr), workspace)."""
    dt = q.dtype
    if grads is None:
        grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), torch.empty_like(qr),
                 torch.empty_like(kr))
    if workspace is None:
        workspace = alloc_workspace(g, dt, True, q.device)
    dq, dk, dv, dqr, dkr = grads
    p = g.params(dt)
    rc = load().df_attn_bwd(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(qr), _ptr(kr), _ptr(out), _ptr(lse),
                            _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dqr), _ptr(dkr), _ptr(workspace),
                            workspace.numel(), _stream(stream))
    if check and rc != DF_OK:
        raise DfError(rc, "df_attn_bwd")
    return grads, workspace


def step_host(g: Geometry, q, k, v, qr, kr, dout, outs, arena, stream=None, host_cu=None, host_qmask=None,
              host_kmask=None):
    """One fwd + bwd from pinned host tensors via df_attn_step_host.
    outs = (out, lse, dq, dk, dv, dqr, dkr) host tensors."""
    dt = q.dtype
    g2 = Geometry(**{**g.__dict__})
    g2.cu_seqlens, g2.query_mask, g2.key_mask = host_cu, host_qmask, host_kmask
    p = g2.params(dt)
    out, lse, dq, dk, dv, dqr, dkr = outs
    rc = load().df_attn_step_host(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(qr), _ptr(kr), _ptr(dout),
                                  _ptr(out), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dqr), _ptr(dkr),
                                  _ptr(arena), arena.numel(), _stream(stream))
    if rc != DF_OK:
        raise DfError(rc, "df_attn_step_host")


def step_host_arena_size(g: Geometry, dtype: torch.dtype) -> int:
    p = g.params(dtype)
    return int(load().df_attn_step_host_arena_size(ctypes.byref(p)))


def rel_index_table(L: int, span: int, nb: int, mp: int, device="cuda", stream=None) -> torch.Tensor:
    out = torch.empty(2 * L - 1, dtype=torch.int32, device=device)
    rc = load().df_rel_index_table(L, span, nb, mp, _ptr(out), _stream(stream))
    if rc != DF_OK:
        raise DfError(rc, "df_rel_index_table")
    return out


def device_error(workspace: torch.Tensor, stream=None) -> int:
    return int(load().df_get_device_error(_ptr(workspace), _stream(stream)))


PROFILE_PHASES = ("fwd", "dq", "dkv", "rel")


def set_profile_events(events):
    """Install (list of 8 torch.cuda.Event, begin/end per phase) or clear
    (None) the library's per-phase timing hooks."""
    lib = load()
    if events is None:
        rc = lib.df_attn_set_profile_events(None, 0)
    else:
        arr = (ctypes.c_void_p * len(events))(*[ctypes.c_void_p(e.cuda_event) for e in events])
        rc = lib.df_attn_set_profile_events(arr, len(events))
    if rc != DF_OK:
        raise DfError(rc, "df_attn_set_profile_events")


def attn_fwd_noalloc(g: Geometry, q, k, v, qr, kr, out, lse, stream=None, check=True):
    """Forward through df_attn_fwd_noalloc (no workspace: the library's
    static device scratch); the caller passes the outputs."""
    p = g.params(q.dtype)
    rc = load().df_attn_fwd_noalloc(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(qr), _ptr(kr), _ptr(out),
                                    _ptr(lse), _stream(stream))
    if check and rc != DF_OK:
        raise DfError(rc, "df_attn_fwd_noalloc")
    return rc


def debug_inject_stall(kernel: int, tile: int = 0, wait_limit_ns: int = 0, wait_min_probes: int = 0):
    """Test hook of the bounded-wait path (df_attn_debug_inject_stall): the
    MMA-issuing warp of `kernel` (0 forward, 1 dQ, 2 dK/dV) stops at `tile`
    and device waits give up after the given limits; kernel=-1 switches it off."""
    rc = load().df_attn_debug_inject_stall(int(kernel), int(tile), int(wait_limit_ns), int(wait_min_probes))
    if rc != DF_OK:
        raise DfError(rc, "df_attn_debug_inject_stall")


def dropout_keep_mask(g: Geometry, dtype: torch.dtype, b: int, h: int, form: int, n: int, device="cuda",
                      stream=None) -> torch.Tensor:
    """The [n, n] keep mask of sequence b, head h as the kernels draw it
    (form 0: row generator, 1: column generator), via df_dropout_keep_mask."""
    out = torch.full((n, n), 255, dtype=torch.uint8, device=device)
    p = g.params(dtype)
    rc = load().df_dropout_keep_mask(ctypes.byref(p), int(b), int(h), int(form), _ptr(out), _stream(stream))
    if rc != DF_OK:
        raise DfError(rc, "df_dropout_keep_mask")
    return out


def noalloc_device_error(stream=None) -> int:
    """Error word of df_attn_fwd_noalloc's static scratch on the current device."""
    return int(load().df_attn_fwd_noalloc_device_error(_stream(stream)))


@dataclass
class PackInfo:
    """What df_pack_info found for a padded batch (device tensors plus the
    three counts read back to the host)."""
    cu_seqlens: torch.Tensor   # device int32 [nseq + 1]
    index: torch.Tensor        # device int32 [total]: padded row b * L + l of each packed row
    total: int
    max_seqlen: int
    nseq: int
    B: int
    L: int


def pack_info(mask: torch.Tensor, stream=None) -> PackInfo:
    """Sequence offsets and row index of the packed layout of a padded batch
    (mask [B, L], device, nonzero = valid), via df_pack_info.  Reads the three
    counts back to the host (one synchronisation)."""
    B, L = mask.shape
    m = mask.to(torch.uint8).contiguous()
    dev = m.device
    cu = torch.empty(B + 1, dtype=torch.int32, device=dev)
    index = torch.empty(B * L, dtype=torch.int32, device=dev)
    info = torch.empty(4, dtype=torch.int32, device=dev)
    ws = torch.empty(max(int(load().df_pack_workspace_size(B)), 16), dtype=torch.uint8, device=dev)
    rc = load().df_pack_info(_ptr(m), B, L, _ptr(cu), _ptr(index), _ptr(info), _ptr(ws), ws.numel(),
                             _stream(stream))
    if rc != DF_OK:
        raise DfError(rc, "df_pack_info")
    total, longest, nseq = (int(v) for v in info[:3].cpu())
    return PackInfo(cu[:nseq + 1], index[:total], total, longest, nseq, B, L)


def _rows(x: torch.Tensor, lead: int):
    return x.numel() // lead * x.element_size()


def pack_rows(x: torch.Tensor, pi: PackInfo, stream=None) -> torch.Tensor:
    """[B, L, ...] -> [total, ...]: the valid rows, sequence after sequence."""
    x = x.contiguous()
    out = torch.empty((pi.total,) + tuple(x.shape[2:]), dtype=x.dtype, device=x.device)
    if pi.total == 0:
        return out
    info = torch.tensor([pi.total, pi.max_seqlen, pi.nseq, 0], dtype=torch.int32, device=x.device)
    rc = load().df_pack_rows(_ptr(x), pi.B * pi.L, _ptr(pi.index), _ptr(info), pi.total, _rows(x, pi.B * pi.L),
                             _ptr(out), _stream(stream))
    if rc != DF_OK:
        raise DfError(rc, "df_pack_rows")
    return out


def unpack_rows(packed: torch.Tensor, pi: PackInfo, stream=None) -> torch.Tensor:
    """[total, ...] -> [B, L, ...] with zero rows at the padding."""
    packed = packed.contiguous()
    out = torch.empty((pi.B, pi.L) + tuple(packed.shape[1:]), dtype=packed.dtype, device=packed.device)
    row_bytes = _rows(out, pi.B * pi.L)
    if pi.total == 0:
        return out.zero_()
    info = torch.tensor([pi.total, pi.max_seqlen, pi.nseq, 0], dtype=torch.int32, device=packed.device)
    rc = load().df_unpack_rows(_ptr(packed), _ptr(pi.index), _ptr(info), pi.total, row_bytes, pi.B * pi.L,
                               _ptr(out), _stream(stream))
    if rc != DF_OK:
        raise DfError(rc, "df_unpack_rows")
    return out


def pack_padded_with_info(x: torch.Tensor, mask: torch.Tensor, stream=None):
    """Pack a padded batch x [B, L, ...] by its mask [B, L]: (packed, PackInfo)."""
    pi = pack_info(mask, stream)
    return pack_rows(x, pi, stream), pi


def unpack_packed(packed: torch.Tensor, pi: PackInfo, stream=None) -> torch.Tensor:
    """Inverse of pack_padded_with_info: [total, ...] -> [B, L, ...], zero at the padding."""
    return unpack_rows(packed, pi, stream)


def qkv_proj_fwd(x, w, bias=None, stream=None):
    """Fused QKV projection (df_qkv_proj_fwd): x [T, C], w [3, H*D, C], bias
    [3, H*D] -> qkv [3, T, H*D] (Q, K, V back to back)."""
    T, C = x.shape
    HD = w.shape[1]
    qkv = torch.empty((3, T, HD), dtype=x.dtype, device=x.device)
    rc = load().df_qkv_proj_fwd(T, C, HD, DTYPE_CODE[x.dtype], _ptr(x), _ptr(w), _ptr(bias), _ptr(qkv),
                                _stream(stream))
    if rc != DF_OK:
        raise DfError(rc, "df_qkv_proj_fwd")
    return qkv


def qkv_proj_bwd(x, w, dqkv, with_bias=True, dw=None, dbias=None, accumulate=False, stream=None):
    """Backward of qkv_proj_fwd (df_qkv_proj_bwd): returns (dx, dw, dbias)."""
    T, C = x.shape
    HD = w.shape[1]
    dx = torch.empty_like(x)
    dw = torch.empty_like(w) if dw is None else dw
    if with_bias and dbias is None:
        dbias = torch.empty((3, HD), dtype=x.dtype, device=x.device)
    ws = torch.empty(int(load().df_qkv_proj_workspace_size(HD)), dtype=torch.uint8, device=x.device)
    rc = load().df_qkv_proj_bwd(T, C, HD, DTYPE_CODE[x.dtype], _ptr(x), _ptr(w), _ptr(dqkv), _ptr(dx), _ptr(dw),
                                _ptr(dbias if with_bias else None), 1 if accumulate else 0, _ptr(ws), ws.numel(),
                                _stream(stream))
    if rc != DF_OK:
        raise DfError(rc, "df_qkv_proj_bwd")
    return dx, dw, dbias


def rel_proj_fwd(rel, gamma, beta, eps, w, bias, H, D, stream=None):
    """Relative projections (df_rel_proj_fwd): returns (qr [H, R, D], kr, rel_ln, ln_stats)."""
    R, C = rel.shape
    dev = rel.device
    rel_ln = torch.empty_like(rel)
    stats = torch.empty((R, 2), dtype=torch.float32, device=dev)
    qr = torch.empty((H, R, D), dtype=rel.dtype, device=dev)
    kr = torch.empty_like(qr)
    rc = load().df_rel_proj_fwd(R, C, H, D, DTYPE_CODE[rel.dtype], _ptr(rel), _ptr(gamma), _ptr(beta), float(eps),
                                _ptr(w), _ptr(bias), _ptr(rel_ln), _ptr(stats), _ptr(qr), _ptr(kr), _stream(stream))
    if rc != DF_OK:
        raise DfError(rc, "df_rel_proj_fwd")
    return qr, kr, rel_ln, stats


def rel_proj_bwd(rel, gamma, rel_ln, stats, w, dqr, dkr, dw, dbias=None, dgamma=None, dbeta=None,
                 accumulate=False, stream=None):
    """Backward of rel_proj_fwd (df_rel_proj_bwd): returns (drel, dgamma, dbeta);
    dw / dbias rows q and k are written (or, accumulate, added to)."""
    R, C = rel.shape
    H, _, D = dqr.shape
    drel = torch.empty_like(rel)
    # with accumulate the library adds to dgamma / dbeta too: fresh buffers start at zero
    dgamma = torch.zeros_like(gamma) if dgamma is None else dgamma
    dbeta = torch.zeros_like(gamma) if dbeta is None else dbeta
    ws = torch.empty(int(load().df_rel_proj_workspace_size(R, C, H, D)), dtype=torch.uint8, device=rel.device)
    rc = load().df_rel_proj_bwd(R, C, H, D, DTYPE_CODE[rel.dtype], _ptr(rel), _ptr(gamma), _ptr(rel_ln),
                                _ptr(stats), _ptr(w), _ptr(dqr), _ptr(dkr), _ptr(drel), _ptr(dgamma), _ptr(dbeta),
                                _ptr(dw), _ptr(dbias), 1 if accumulate else 0, _ptr(ws), ws.numel(),
                                _stream(stream))
    if rc != DF_OK:
        raise DfError(rc, "df_rel_proj_bwd")
    return drel, dgamma, dbeta
