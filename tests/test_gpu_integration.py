"""Integration with PyTorch's execution models: CUDA-graph capture of a whole
step (every library call is asynchronous on the current stream and allocates
nothing), and the autograd binding inside a small training graph."""
import math

import numpy as np
import pytest
import torch

import oracle
from synthetic import MaskSpec, qkv, qkv_block_structured

pytestmark = pytest.mark.gpu

lc = pytest.importorskip("long_context_masked_mask_gb300")


def relf(g, r):
    return float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30))


def test_cuda_graph_capture_of_a_step():
    """Block selection -> mask compile -> forward -> backward captured once in a
    CUDA graph and replayed on new inputs: the replay equals eager calls on those
    inputs (forward bit for bit, backward within the atomic dQ tolerance)."""
    B, N, Hq, Hkv, D = 1, 1536, 8, 2, 128
    x = qkv_block_structured(B, N, Hq, Hkv, 128, strength=1.5, seed=1, device="cuda")
    q, k, v, d_o = (x[n].clone() for n in ("q", "k", "v", "do"))
    offs = torch.arange(0, N + 1, 128, dtype=torch.int32, device="cuda")
    nb = offs.numel() - 1
    bmap = torch.empty(B, Hq, nb, nb, dtype=torch.uint8, device="cuda")
    sel_ws = torch.empty(lc.lcattn_block_select_workspace_size(q, k, lc.select_desc("topk", offs, offs, top_k=4)),
                         dtype=torch.uint8, device="cuda")
    mask = lc.DeviceMask.from_block_map(bmap, offs, offs)
    shape = lc.make_shape(q, k, v)
    meta = torch.empty(lc._lib.lcattn_tile_meta_size(lc.ctypes.byref(shape), lc.ctypes.byref(mask.desc)),
                       dtype=torch.uint8, device="cuda")
    ws = torch.empty(lc.lcattn_bwd_workspace_size(shape), dtype=torch.uint8, device="cuda")
    o, lse = torch.empty_like(q), torch.empty(B, Hq, N, dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

    def step():
        lc.lcattn_block_select(q, k, offs, offs, "topk", top_k=4, causal=True, block_map=bmap, workspace=sel_ws)
        lc.lcattn_mask_compile(shape, mask, meta)
        lc.lcattn_fwd(q, k, v, mask, meta, o=o, lse=lse)
        lc.lcattn_bwd(q, k, v, o, d_o, lse, mask, meta, dq=dq, dk=dk, dv=dv, workspace=ws)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()  # warm up (kernel attributes are set outside the capture)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for seed in (2, 3):
        y = qkv_block_structured(B, N, Hq, Hkv, 128, strength=1.5, seed=seed, device="cuda")
        for n, t in (("q", q), ("k", k), ("v", v), ("do", d_o)):
            t.copy_(y[n])
        g.replay()
        torch.cuda.synchronize()
        assert lc.lcattn_read_status(meta) == 0
        got = [t.clone() for t in (bmap, o, lse, dq, dk, dv)]
        step()
        torch.cuda.synchronize()
        assert torch.equal(got[0], bmap) and torch.equal(got[1], o) and torch.equal(got[2], lse)
        for a_, b_ in zip(got[3:], (dq, dk, dv)):
            assert relf(a_.double().cpu().numpy(), b_.double().cpu().numpy()) <= 1e-2


def test_autograd_binding_in_a_training_graph():
    """q, k, v from a linear projection, attention through the autograd binding,
    a scalar loss: the weight gradient matches the one obtained with the fp64
    oracle's attention gradients pushed back through the same projection."""
    torch.manual_seed(0)
    B, N, Hq, Hkv, D, E = 1, 384, 4, 2, 128, 256
    spec = MaskSpec("CAUSAL_DOCUMENT", {"doc_lens": [100, 200, 84]})
    xin = torch.randn(B, N, E, device="cuda", dtype=torch.bfloat16)
    W = (torch.randn((Hq + 2 * Hkv) * D, E, device="cuda") / math.sqrt(E)).to(torch.bfloat16).requires_grad_()
    mask = lc.DeviceMask(spec, N, Hq, B, device="cuda")
    proj = (xin @ W.t()).view(B, N, Hq + 2 * Hkv, D)
    q, k, v = proj[:, :, :Hq], proj[:, :, Hq:Hq + Hkv], proj[:, :, Hq + Hkv:]
    shape = lc.make_shape(q, k, v)
    meta = lc.lcattn_mask_compile(shape, mask)
    o = lc.MaskedAttention.apply(q, k, v, mask, meta)
    g_out = torch.randn_like(o)
    (o.float() * g_out.float()).sum().backward()
    # Reference: the oracle's gradients for the same q, k, v, then back through the projection.
    f = lambda t: t.detach().double().cpu().numpy()
    dQ, dK, dV, O, _ = oracle.attention_bwd(f(q), f(k), f(v), f(g_out), spec, 1.0 / math.sqrt(D))
    assert relf(f(o), O) <= 1e-2
    dproj = np.concatenate([dQ, dK, dV], axis=2).reshape(B * N, -1)
    dW_ref = dproj.T @ f(xin).reshape(B * N, E)
    assert relf(f(W.grad), dW_ref) <= 3e-2
