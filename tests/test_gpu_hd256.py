"""Head dim 256, forward only (its backward does not fit in tensor memory and
returns LCATTN_ERR_UNSUPPORTED): O and LSE through the C ABI against the fp64
oracle with the bars of the 128 case, on both descriptor kinds, MHA and GQA,
ragged lengths, and the split-KV forward for decode-style rows."""
import math

import numpy as np
import pytest
import torch

import oracle
from synthetic import MaskSpec, qkv
from test_gpu_parity import relf, spec_for

pytestmark = pytest.mark.gpu

lc = pytest.importorskip("long_context_masked_mask_gb300")

D = 256


def forward_and_check(spec, B, Sq, Sk, Hq, Hkv, seed, expect_split=None):
    x = qkv(B, Sq, Hq, Hkv, D, seed=seed, Sk=Sk, with_do=False)
    dev = {n: t.cuda() for n, t in x.items()}
    mask = lc.DeviceMask(spec, Sq, Hq, B, device="cuda", Sk=Sk)
    shape = lc.make_shape(dev["q"], dev["k"], dev["v"])
    meta = lc.lcattn_mask_compile(shape, mask)
    if expect_split is not None:
        assert (lc.lcattn_fwd_workspace_size(shape, mask) > 0) == expect_split
    o, lse = lc.lcattn_fwd_ws(dev["q"], dev["k"], dev["v"], mask, meta)
    o2, lse2 = lc.lcattn_fwd(dev["q"], dev["k"], dev["v"], mask, meta)
    torch.cuda.synchronize()
    assert lc.lcattn_read_status(meta) == 0
    f64 = {n: t.double().numpy() for n, t in x.items()}
    O, LSE = oracle.attention_fwd(f64["q"], f64["k"], f64["v"], spec, 1.0 / math.sqrt(D))
    fin = np.isfinite(LSE)
    for oo, ll in ((o, lse), (o2, lse2)):
        g = oo.double().cpu().numpy()
        assert np.abs(g - O).max() <= 2e-2 and relf(g, O) <= 1e-2
        gl = ll.double().cpu().numpy()
        np.testing.assert_array_equal(np.isfinite(gl), fin)
        if fin.any():
            assert np.abs(gl[fin] - LSE[fin]).max() <= 5e-3
    return dev, mask, meta, o, lse


@pytest.mark.parametrize("kind", ["FULL", "CAUSAL", "CAUSAL_DOCUMENT", "CAUSAL_SLIDING_WINDOW",
                                  "PREFIX_LM_CAUSAL", "UNIFORM_BLOCK", "VARIABLE_BLOCK"])
def test_hd256_forward_families(kind):
    N, Hq, Hkv = 392, 4, 2
    forward_and_check(spec_for(kind, N, Hq), 1, N, N, Hq, Hkv, seed=3)


@pytest.mark.parametrize("B,N,Hq,Hkv", [(2, 700, 2, 2), (1, 1100, 6, 1)])
def test_hd256_forward_mha_gqa(B, N, Hq, Hkv):
    forward_and_check(MaskSpec("CAUSAL"), B, N, N, Hq, Hkv, seed=5)


@pytest.mark.parametrize("B,Sq,Sk,Hq,Hkv", [(2, 1, 3000, 16, 2), (1, 40, 2500, 4, 4)])
def test_hd256_split_forward(B, Sq, Sk, Hq, Hkv):
    forward_and_check(MaskSpec("CAUSAL"), B, Sq, Sk, Hq, Hkv, seed=7, expect_split=True)


def test_hd256_backward_is_refused():
    dev, mask, meta, o, lse = forward_and_check(MaskSpec("FULL"), 1, 256, 256, 2, 1, seed=9)
    with pytest.raises(lc.LcattnError) as err:
        lc.lcattn_bwd(dev["q"], dev["k"], dev["v"], o, torch.ones_like(o), lse, mask, meta,
                      workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert err.value.status == lc.LCATTN_ERR_UNSUPPORTED


@pytest.mark.parametrize("kind", ["CAUSAL", "UNIFORM_BLOCK_EMPTY_ROWS"])
def test_hd256_many_items_per_cta(kind):
    """More work items than SMs (several per persistent CTA), of uneven length
    and some empty, so the K/V ring's order runs across item boundaries
    (an item's last V is produced after the next item's first K)."""
    B, N, Hq, Hkv = 1, 4096, 16, 4
    if kind == "CAUSAL":
        spec = MaskSpec("CAUSAL")
    else:
        from synthetic import block_keep
        nb = N // 128
        keep = block_keep(Hq, nb, nb, 0.3, 11, force_diagonal=False)
        keep[:, ::3, :] = False  # every third query block of every head has an empty list
        spec = MaskSpec("UNIFORM_BLOCK", {"block": 128, "keep": keep})
    x = qkv(B, N, Hq, Hkv, D, seed=13, with_do=False)
    dev = {n: t.cuda() for n, t in x.items()}
    mask = lc.DeviceMask(spec, N, Hq, B, device="cuda")
    shape = lc.make_shape(dev["q"], dev["k"], dev["v"])
    meta = lc.lcattn_mask_compile(shape, mask)
    o, lse = lc.lcattn_fwd(dev["q"], dev["k"], dev["v"], mask, meta)
    o_again, _ = lc.lcattn_fwd(dev["q"], dev["k"], dev["v"], mask, meta)
    torch.cuda.synchronize()
    assert lc.lcattn_read_status(meta) == 0
    assert torch.equal(o, o_again)
    f64 = {n: t.double().numpy() for n, t in x.items()}
    rng = np.random.default_rng(1)
    rows = np.array(sorted({0, 127, 128, 129, N - 1} | {int(r) for r in rng.integers(0, N, 40)}))
    scale = 1.0 / math.sqrt(D)
    for h in (0, 5, Hq - 1):
        ref_o, ref_l = oracle.attention_fwd_rows(f64["q"], f64["k"], f64["v"], spec, scale, 0, h, rows)
        g = o[0, rows, h].double().cpu().numpy()
        assert np.abs(g - ref_o).max() <= 2e-2 and relf(g, ref_o) <= 1e-2, h
        gl = lse[0, h, rows].double().cpu().numpy()
        fin = np.isfinite(ref_l)
        np.testing.assert_array_equal(np.isfinite(gl), fin)
        if fin.any():
            assert np.abs(gl[fin] - ref_l[fin]).max() <= 5e-3
