"""Dropout randomness on the GPU, bit for bit.

1. The oracle's Philox4x32-10 (written from the SC'11 description by Salmon,
   Moraes, Dror and Shaw) against cuRAND's header-defined device function
   curand_Philox4x32_10(counter, key), run on the GPU for a grid of counters
   and keys: an implementation that is not this project's, so a misread
   multiplier, Weyl constant, word order or key schedule in the oracle fails
   here.  The mapping is direct: counter words (c0, c1, c2, c3) and key words
   (k0, k1) are passed as cuRAND's uint4 / uint2 in that order.
2. The keep mask that the attention kernels draw ("DisentangledFlash",
   section "Status": the Philox mask is regenerated in the backward, never
   stored), through the library's df_dropout_keep_mask export, against the
   oracle's keep mask of the same (sequence, head): every bit, for the row
   generator of the forward / dQ kernels and the column generator of the
   dK/dV kernel, padded and packed, at several seeds and offsets.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

from exact_deberta_disentangled_gb300 import binding as B
from exact_deberta_disentangled_gb300 import synth
from oracle import oracle
from tests.helpers import problem_of
from tests.test_parity_tc_gpu import geometry

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.fixture(scope="module")
def curand_probe():
    src = os.path.join(ROOT, "tests", "curand_philox_probe.cu")
    out_dir = os.path.join(ROOT, "_build")
    os.makedirs(out_dir, exist_ok=True)
    so = os.path.join(out_dir, "curand_philox_probe.so")
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-shared", "-Xcompiler", "-fPIC",
                    "-o", so, src], check=True)
    lib = ctypes.CDLL(so)
    u32p = ctypes.POINTER(ctypes.c_uint32)
    lib.curand_philox4x32_10_batch.argtypes = [u32p, u32p, u32p, ctypes.c_int]
    lib.curand_philox4x32_10_batch.restype = ctypes.c_int
    return lib


def test_oracle_philox_matches_curand(curand_probe):
    rng = np.random.default_rng(20240611)
    n = 4096
    ctr = rng.integers(0, 2 ** 32, size=(n, 4), dtype=np.uint64).astype(np.uint32)
    key = rng.integers(0, 2 ** 32, size=(n, 2), dtype=np.uint64).astype(np.uint32)
    # structured counters as the kernels use them: (j >> 2, i, seq * H + h, offset)
    for t in range(256):
        ctr[t] = (t % 16, t // 16, 3, 7)
        key[t] = (0x12345678, 0x9ABCDEF0)
    ctr[256], key[256] = (0, 0, 0, 0), (0, 0)
    ctr[257], key[257] = (0xFFFFFFFF,) * 4, (0xFFFFFFFF,) * 2
    out = np.zeros((n, 4), dtype=np.uint32)
    u32p = ctypes.POINTER(ctypes.c_uint32)
    rc = curand_probe.curand_philox4x32_10_batch(np.ascontiguousarray(ctr).ctypes.data_as(u32p),
                                                 np.ascontiguousarray(key).ctypes.data_as(u32p),
                                                 out.ctypes.data_as(u32p), n)
    assert rc == 0
    want = np.stack([oracle.philox4x32_10(ctr[t], key[t]) for t in range(n)])
    assert np.array_equal(out, want)


CASES = [
    # (workload, make_inputs kwargs, seed, offset)
    ("hd128_dropout", dict(B=2, L=300, H=3), 1234, 0),
    ("hd32_dropout", dict(B=1, L=517, H=2), 2 ** 40 + 99, 5),
    ("v3_base", dict(B=2, L=129, H=2), 7, 2 ** 31 + 11),
]


@pytest.mark.parametrize("name,kw,seed,offset", CASES)
@pytest.mark.parametrize("form", [0, 1])
def test_kernel_keep_mask_matches_oracle_bitwise(name, kw, seed, offset, form):
    w = synth.WORKLOADS[name]
    x = synth.make_inputs(w, **kw)
    H = kw["H"]
    g = geometry(x, w, H, p_drop=0.1, seed=seed, offset=offset)
    prob = problem_of(x, w, H, 0.1, seed, offset)
    for s in range(x.B):
        n = int(x.cu_seqlens[s + 1] - x.cu_seqlens[s])
        for h in range(H):
            got = B.dropout_keep_mask(g, x.q.dtype, s, h, form, n).cpu().numpy()
            want = oracle.keep_mask(prob, s, h)
            assert np.array_equal(got, want), (s, h, int((got != want).sum()))
    rate = float(want.mean())
    assert 0.85 < rate < 0.95


@pytest.mark.parametrize("form", [0, 1])
def test_kernel_keep_mask_packed(form):
    w = synth.WORKLOADS["varlen"]
    x = synth.make_inputs(w, H=2, total_tokens=900)
    g = geometry(x, w, 2, p_drop=0.25, seed=42, offset=1)
    prob = problem_of(x, w, 2, 0.25, 42, 1)
    for s in range(x.B):
        n = int(x.cu_seqlens[s + 1] - x.cu_seqlens[s])
        got = B.dropout_keep_mask(g, x.q.dtype, s, 1, form, n).cpu().numpy()
        assert np.array_equal(got, oracle.keep_mask(prob, s, 1)), s
