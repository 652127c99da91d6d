"""lcattn_bwd_noalloc: the backward for callers that may not allocate device
memory (plugins inside runtimes that own every allocation, serving paths that
forbid cudaMalloc after start-up).  Its scratch is a fixed array inside the
library instead of a caller workspace.

Checked through the C ABI, on two calls in a row (the second call finds the
first call's contents in the shared array), against lcattn_bwd on the same
inputs and against the fp64 oracle, with the gradient tolerance of the parity
tests (relative Frobenius 3e-2), at head dims 64 and 128, on contiguous tensors
and on Q, K, V that are views of one fused QKV buffer; and a problem larger
than the array must be refused before any launch.  This file is collected last
on purpose.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
from synthetic import MaskSpec, qkv

pytestmark = pytest.mark.gpu

lc = pytest.importorskip("long_context_masked_mask_gb300")


def relf(g, r):
    g = g.double().cpu().numpy() if isinstance(g, torch.Tensor) else g
    r = r.double().cpu().numpy() if isinstance(r, torch.Tensor) else r
    return float(np.linalg.norm(g - r) / np.linalg.norm(r))


def _inputs(B, N, Hq, Hkv, D, seed, fused):
    x = qkv(B, N, Hq, Hkv, D, seed=seed)
    if not fused:
        return {k: t.cuda() for k, t in x.items()}, x
    # Q, K, V as views of one [B, N, Hq + 2 Hkv, D] projection output.
    buf = torch.cat([x["q"], x["k"], x["v"]], dim=2).cuda()
    dev = {"q": buf[:, :, :Hq], "k": buf[:, :, Hq:Hq + Hkv], "v": buf[:, :, Hq + Hkv:],
           "do": x["do"].cuda()}
    return dev, x


@pytest.mark.parametrize("D,fused", [(128, False), (64, False), (128, True)],
                         ids=["hd128", "hd64", "hd128-fused-qkv"])
def test_noalloc_matches_bwd_and_oracle_on_two_calls(D, fused):
    B, N, Hq, Hkv = 1, 1000, 4, 2
    spec = MaskSpec("GLOBAL_SLIDING", {"global_tokens": 64, "window": 200})
    x, host = _inputs(B, N, Hq, Hkv, D, 11, fused)
    mask = lc.DeviceMask(spec, N, Hq, B)
    shape = lc.make_shape(x["q"], x["k"], x["v"])
    meta = lc.lcattn_mask_compile(shape, mask)
    o, lse = lc.lcattn_fwd(x["q"], x["k"], x["v"], mask, meta)
    ref = lc.lcattn_bwd(x["q"], x["k"], x["v"], o, x["do"], lse, mask, meta)
    torch.cuda.synchronize()
    f64 = {k: t.double().numpy() for k, t in host.items()}
    want = oracle.attention_bwd(f64["q"], f64["k"], f64["v"], f64["do"], spec, 1.0 / math.sqrt(D))[:3]
    for call in range(2):
        # Outputs with the inputs' strides, filled with stale values that must vanish.
        outs = tuple(torch.empty_strided(t.shape, t.stride(), dtype=t.dtype, device=t.device).fill_(7 + call)
                     for t in (x["q"], x["k"], x["v"]))
        lc.lcattn_bwd_noalloc(x["q"], x["k"], x["v"], o, x["do"], lse, mask, meta,
                              dq=outs[0], dk=outs[1], dv=outs[2])
        torch.cuda.synchronize()
        assert lc.lcattn_read_status(meta) == 0
        for name, got, same, exact in zip(("dq", "dk", "dv"), outs, ref, want):
            assert torch.isfinite(got.float()).all(), name
            assert relf(got, same) <= 3e-2, (call, name, relf(got, same))
            assert relf(got, exact) <= 3e-2, (call, name, relf(got, exact))


def test_noalloc_refuses_problems_beyond_the_array():
    s = lc.lcattn_shape()
    s.B, s.Sq, s.Sk, s.Hq, s.Hkv, s.D = 1, 131072, 131072, 64, 8, 128
    s.q_stride[:] = s.o_stride[:] = (131072 * 64 * 128, 64 * 128, 128)
    s.k_stride[:] = s.v_stride[:] = (131072 * 8 * 128, 8 * 128, 128)
    assert lc.library().lcattn_bwd_workspace_size(ctypes.byref(s)) > lc.LCATTN_NOALLOC_SCRATCH_BYTES
    d = lc.lcattn_mask_desc()
    d.kind = lc.LCATTN_MASK_COLBOUNDS
    st = lc.library().lcattn_bwd_noalloc(ctypes.byref(s), None, None, None, None, None, None, None,
                                         ctypes.byref(d), 1.0 / math.sqrt(128), None, None, None, None)
    assert st == lc.LCATTN_ERR_SCRATCH_LIMIT
    assert "no-allocation" in lc.status_string(st)
