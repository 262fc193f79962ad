"""Packing between the padded and the packed layout on the GPU
("DisentangledFlash", section "Packed unpadded inference and training":
pack_padded_with_info / unpack_packed).

- The packed rows, sequence offsets and counts equal a plain numpy
  restatement of the definition (valid positions of each sequence in order,
  empty sequences dropped), for right padding, masks with holes and empty
  sequences; unpacking restores the valid rows and zeroes the padding.
- With right padding, attention over the packed layout (pack Q, K, V, dO,
  run the packed forward and backward, unpack) equals the masked padded
  attention on the valid rows, and dQr / dKr agree, within the parity bars.
"""
import numpy as np
import pytest
import torch

from exact_deberta_disentangled_gb300 import binding as B
from exact_deberta_disentangled_gb300 import synth
from tests.helpers import rel_l2

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def reference_pack(mask):
    """numpy restatement: padded row index of every packed row, offsets, counts."""
    Bn, L = mask.shape
    index, cu = [], [0]
    for b in range(Bn):
        pos = np.nonzero(mask[b])[0]
        if len(pos) == 0:
            continue
        index.extend(b * L + pos)
        cu.append(cu[-1] + len(pos))
    lens = np.diff(cu)
    return np.array(index, dtype=np.int64), np.array(cu), int(lens.max()) if len(lens) else 0


@pytest.mark.parametrize("kind", ["right", "holes", "empty"])
def test_pack_matches_definition(kind):
    g = torch.Generator().manual_seed(7)
    Bn, L, C = 7, 1100, 48
    if kind == "right":
        lens = torch.randint(1, L + 1, (Bn,), generator=g)
        mask = (torch.arange(L)[None, :] < lens[:, None])
    else:
        mask = torch.rand(Bn, L, generator=g) < 0.6
        if kind == "empty":
            mask[2] = False
            mask[5] = False
    mask = mask.to(torch.uint8)
    x = torch.randn(Bn, L, C, generator=g).to(torch.bfloat16)
    packed, pi = B.pack_padded_with_info(x.to(DEV), mask.to(DEV))
    idx, cu, longest = reference_pack(mask.numpy())
    assert pi.total == len(idx) and pi.nseq == len(cu) - 1 and pi.max_seqlen == longest
    assert np.array_equal(pi.cu_seqlens.cpu().numpy(), cu)
    assert np.array_equal(pi.index.cpu().numpy(), idx)
    assert torch.equal(packed.cpu(), x.reshape(Bn * L, C)[torch.from_numpy(idx)])
    back = B.unpack_packed(packed, pi).cpu()
    want = torch.where(mask[:, :, None].bool(), x, torch.zeros_like(x))
    assert torch.equal(back, want)


def test_packed_attention_equals_masked_padded_attention():
    w = synth.WORKLOADS["v3_base"]
    x = synth.make_inputs(w, B=5, L=400, H=3)     # right padding, query mask == key mask
    H = 3
    dev = torch.device(DEV)
    g_pad = B.Geometry(B=x.B, L=x.L, H=H, D=w.D, span=w.span, nb=w.nb, mp=w.mp,
                       query_mask=x.qmask.to(dev), key_mask=x.kmask.to(dev))
    t = [a.to(dev) for a in (x.q, x.k, x.v, x.qr, x.kr, x.dout)]
    out_p, lse_p, _ = B.attn_fwd(g_pad, *t[:5])
    grads_p, _ = B.attn_bwd(g_pad, *t[:5], out_p, lse_p, t[5])

    mask2 = x.qmask.reshape(x.B, x.L).to(dev)
    pq = [B.pack_rows(a.reshape(x.B, x.L, H, w.D), B.pack_info(mask2)) for a in (t[0], t[1], t[2], t[5])]
    pi = B.pack_info(mask2)
    g_pk = B.Geometry(B=pi.nseq, L=pi.max_seqlen, H=H, D=w.D, span=w.span, nb=w.nb, mp=w.mp,
                      cu_seqlens=pi.cu_seqlens, total_tokens=pi.total)
    out_k, lse_k, _ = B.attn_fwd(g_pk, pq[0], pq[1], pq[2], t[3], t[4])
    grads_k, _ = B.attn_bwd(g_pk, pq[0], pq[1], pq[2], t[3], t[4], out_k, lse_k, pq[3])
    torch.cuda.synchronize()

    valid = x.qmask.bool().cpu()
    un = lambda a: B.unpack_packed(a, pi).reshape(x.B * x.L, H, w.D).cpu()
    assert rel_l2(un(out_k)[valid], out_p.cpu()[valid].double().numpy()) <= 5e-3
    for a, b in zip(grads_k[:3], grads_p[:3]):
        assert rel_l2(un(a)[valid], b.cpu()[valid].double().numpy()) <= 1e-2
    for a, b in zip(grads_k[3:], grads_p[3:]):
        assert rel_l2(a.cpu(), b.cpu().double().numpy()) <= 1e-2
    # LSE: packed [H, T] against the padded [B, H, L] at the valid positions
    lse_pad = lse_p.permute(1, 0, 2).reshape(H, x.B * x.L)[:, valid.to(lse_p.device)].cpu()
    assert rel_l2(lse_k.cpu(), lse_pad.double().numpy()) <= 5e-3


def test_pack_rejects_bad_arguments():
    m = torch.ones(2, 8, dtype=torch.uint8, device=DEV)
    cu = torch.empty(3, dtype=torch.int32, device=DEV)
    idx = torch.empty(16, dtype=torch.int32, device=DEV)
    info = torch.empty(4, dtype=torch.int32, device=DEV)
    lib = B.load()
    assert lib.df_pack_info(B._ptr(m), 2, 8, B._ptr(cu), B._ptr(idx), B._ptr(info), None, 0,
                            B._stream()) == B.DF_ERR_WORKSPACE
    assert lib.df_pack_info(B._ptr(m), 0, 8, B._ptr(cu), B._ptr(idx), B._ptr(info), None, 0,
                            B._stream()) == B.DF_ERR_INVALID_ARG
    x = torch.zeros(16, 3, dtype=torch.uint8, device=DEV)   # 3-byte rows: not a multiple of 16
    out = torch.zeros(16, 3, dtype=torch.uint8, device=DEV)
    assert lib.df_pack_rows(B._ptr(x), 16, B._ptr(idx), B._ptr(info), 16, 3, B._ptr(out),
                            B._stream()) == B.DF_ERR_INVALID_ARG
