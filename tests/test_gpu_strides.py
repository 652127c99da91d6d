"""Strided tensors through the C ABI: Q, K and V as views into one fused QKV
projection buffer [B][S][Hq + 2 Hkv][D] (head stride D, sequence stride
(Hq + 2 Hkv) D), the output written into a buffer with padding rows between
sequences, and the gradients written into views of a fused gradient buffer.
Results must equal the contiguous run (forward bit for bit; backward within
the tolerance its atomic dQ accumulation allows) and match the oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import block_select_ref
from synthetic import MaskSpec, qkv, qkv_block_structured

pytestmark = pytest.mark.gpu

lc = pytest.importorskip("long_context_masked_mask_gb300")


def relf(g, r):
    return float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30))


def fused_views(x, Hq, Hkv, pad=0):
    """q, k, v as slices of one [B, S, Hq + 2 Hkv, D] buffer (plus `pad` spare heads)."""
    B, S, _, D = x["q"].shape
    buf = torch.zeros(B, S, Hq + 2 * Hkv + pad, D, dtype=torch.bfloat16, device="cuda")
    buf[:, :, :Hq] = x["q"].cuda()
    buf[:, :, Hq:Hq + Hkv] = x["k"].cuda()
    buf[:, :, Hq + Hkv:Hq + 2 * Hkv] = x["v"].cuda()
    return buf, buf[:, :, :Hq], buf[:, :, Hq:Hq + Hkv], buf[:, :, Hq + Hkv:Hq + 2 * Hkv]


@pytest.mark.parametrize("D,B,N,Hq,Hkv,kind", [(128, 2, 520, 8, 2, "CAUSAL_DOCUMENT"),
                                                (64, 1, 700, 4, 4, "CAUSAL"),
                                                (128, 1, 1000, 4, 1, "UNIFORM_BLOCK")])
def test_fused_qkv_layout_forward_backward(D, B, N, Hq, Hkv, kind):
    if kind == "CAUSAL_DOCUMENT":
        spec = MaskSpec(kind, {"doc_lens": [200, 300, 20]})
    elif kind == "UNIFORM_BLOCK":
        from synthetic import block_keep
        spec = MaskSpec(kind, {"block": 64, "keep": block_keep(Hq, -(-N // 64), -(-N // 64), 0.5, 2)})
    else:
        spec = MaskSpec(kind)
    x = qkv(B, N, Hq, Hkv, D, seed=31)
    buf, q, k, v = fused_views(x, Hq, Hkv, pad=1)
    assert q.stride() == (N * (Hq + 2 * Hkv + 1) * D, (Hq + 2 * Hkv + 1) * D, D, 1)
    d_o = x["do"].cuda()
    # O and dO in a buffer with 3 padding rows after every sequence.
    obuf = torch.full((B, N + 3, Hq, D), 7.0, dtype=torch.bfloat16, device="cuda")
    o = obuf[:, :N]
    dobuf = torch.zeros_like(obuf)
    dobuf[:, :N] = d_o
    d_o_v = dobuf[:, :N]
    gbuf = torch.full_like(buf, 5.0)
    dq, dk, dv = gbuf[:, :, :Hq], gbuf[:, :, Hq:Hq + Hkv], gbuf[:, :, Hq + Hkv:Hq + 2 * Hkv]

    mask = lc.DeviceMask(spec, N, Hq, B, device="cuda")
    shape = lc.make_shape(q, k, v, o)
    meta = lc.lcattn_mask_compile(shape, mask)
    o, lse = lc.lcattn_fwd_ws(q, k, v, mask, meta, o=o)
    lc.lcattn_bwd(q, k, v, o, d_o_v, lse, mask, meta, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert lc.lcattn_read_status(meta) == 0
    # padding rows and spare heads untouched
    assert (obuf[:, N:] == 7.0).all() and (gbuf[:, :, Hq + 2 * Hkv:] == 5.0).all()

    ref = lc.attention(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), spec, d_o=d_o)
    torch.cuda.synchronize()
    assert torch.equal(o, ref["o"]), "forward differs from the contiguous run"
    assert torch.equal(lse, ref["lse"])
    for g, r in ((dq, ref["dq"]), (dk, ref["dk"]), (dv, ref["dv"])):
        assert relf(g.double().cpu().numpy(), r.double().cpu().numpy()) <= 1e-2

    f64 = {n: t.double().numpy() for n, t in x.items()}
    dQ, dK, dV, O, LSE = oracle.attention_bwd(f64["q"], f64["k"], f64["v"], f64["do"], spec,
                                              1.0 / math.sqrt(D))
    assert relf(o.double().cpu().numpy(), O) <= 1e-2
    for g, r in ((dq, dQ), (dk, dK), (dv, dV)):
        assert relf(g.double().cpu().numpy(), r) <= 3e-2


def test_fused_qkv_layout_decode_split_path():
    """Decode rows from a fused buffer through the split-KV forward."""
    B, Sq, Sk, Hq, Hkv, D = 2, 1, 3000, 16, 2, 128
    x = qkv(B, Sq, Hq, Hkv, D, seed=5, Sk=Sk, with_do=False)
    qbuf = torch.zeros(B, Sq, Hq + 8, D, dtype=torch.bfloat16, device="cuda")
    qbuf[:, :, 4:4 + Hq] = x["q"].cuda()
    q = qbuf[:, :, 4:4 + Hq]
    kvbuf = torch.zeros(B, Sk, 2 * Hkv, D, dtype=torch.bfloat16, device="cuda")
    kvbuf[:, :, :Hkv] = x["k"].cuda()
    kvbuf[:, :, Hkv:] = x["v"].cuda()
    k, v = kvbuf[:, :, :Hkv], kvbuf[:, :, Hkv:]
    mask = lc.DeviceMask(MaskSpec("CAUSAL"), Sq, Hq, B, device="cuda", Sk=Sk)
    shape = lc.make_shape(q, k, v)
    meta = lc.lcattn_mask_compile(shape, mask)
    assert lc.lcattn_fwd_workspace_size(shape, mask) > 0
    o, lse = lc.lcattn_fwd_ws(q, k, v, mask, meta)
    torch.cuda.synchronize()
    f64 = {n: t.double().numpy() for n, t in x.items()}
    O, LSE = oracle.attention_fwd(f64["q"], f64["k"], f64["v"], MaskSpec("CAUSAL"), 1.0 / math.sqrt(D))
    g = o.double().cpu().numpy()
    assert np.abs(g - O).max() <= 2e-2 and relf(g, O) <= 1e-2
    assert np.abs(lse.double().cpu().numpy() - LSE).max() <= 5e-3


def test_fused_qkv_layout_block_select():
    """Block selection reads Q and K through their strides."""
    B, N, Hq, Hkv = 1, 1024, 8, 2
    x = qkv_block_structured(B, N, Hq, Hkv, 128, strength=1.5, seed=8)
    buf, q, k, _ = fused_views(x, Hq, Hkv)
    offs = torch.arange(0, N + 1, 128, dtype=torch.int32, device="cuda")
    gmap, _ = lc.lcattn_block_select(q, k, offs, offs, "topk", top_k=3, causal=True)
    ref, _ = lc.lcattn_block_select(x["q"].cuda(), x["k"].cuda(), offs, offs, "topk", top_k=3, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(gmap, ref)
    want, _ = block_select_ref.block_select(x["q"].double().numpy(), x["k"].double().numpy(),
                                            offs.cpu().numpy(), offs.cpu().numpy(), "topk",
                                            1.0 / math.sqrt(128), top_k=3, causal=True)
    assert np.array_equal(gmap.cpu().numpy(), want)
