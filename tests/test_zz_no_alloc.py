"""lcattn_bwd_noalloc: the backward for callers that may not allocate device
memory (plugins inside runtimes that own every allocation, serving paths that
forbid cudaMalloc after start-up).  Its scratch is a fixed array inside the
library instead of a caller workspace.

Checked through the C ABI against lcattn_bwd on the same inputs, on two calls
in a row (the second call finds the first call's contents in the shared
array), with the gradient tolerance of the parity tests (relative Frobenius
3e-2); and a problem larger than the array must be refused before any launch.
This file is collected last on purpose.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

from synthetic import MaskSpec, qkv

pytestmark = pytest.mark.gpu

lc = pytest.importorskip("long_context_masked_mask_gb300")


def relf(g, r):
    g = g.double().cpu().numpy()
    r = r.double().cpu().numpy()
    return float(np.linalg.norm(g - r) / np.linalg.norm(r))


def test_noalloc_matches_bwd_on_two_calls():
    B, N, Hq, Hkv = 1, 1000, 4, 2
    spec = MaskSpec("GLOBAL_SLIDING", {"global_tokens": 64, "window": 200})
    x = {k: t.cuda() for k, t in qkv(B, N, Hq, Hkv, 128, seed=11).items()}
    mask = lc.DeviceMask(spec, N, Hq, B)
    shape = lc.make_shape(x["q"], x["k"], x["v"])
    meta = lc.lcattn_mask_compile(shape, mask)
    o, lse = lc.lcattn_fwd(x["q"], x["k"], x["v"], mask, meta)
    ref = lc.lcattn_bwd(x["q"], x["k"], x["v"], o, x["do"], lse, mask, meta)
    torch.cuda.synchronize()
    for call in range(2):
        outs = tuple(torch.full_like(t, float(7 + call)) for t in ref)  # stale values must vanish
        lc.lcattn_bwd_noalloc(x["q"], x["k"], x["v"], o, x["do"], lse, mask, meta,
                              dq=outs[0], dk=outs[1], dv=outs[2])
        torch.cuda.synchronize()
        assert lc.lcattn_read_status(meta) == 0
        for name, got, want in zip(("dq", "dk", "dv"), outs, ref):
            assert torch.isfinite(got.float()).all(), name
            assert relf(got, want) <= 3e-2, (call, name, relf(got, want))


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
