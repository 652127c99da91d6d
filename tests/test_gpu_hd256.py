"""Head dim 256: forward (O, LSE) and backward (dQ, dK, dV) through the C ABI
against the fp64 oracle with the bars of the 128 case, on both descriptor
kinds, MHA and GQA, ragged lengths, the split-KV forward for decode-style
rows, and the backward's dK/dV units that run as two CTAs (one per half of the
head dim) with split and unsplit head shares, the allocation-free and the
accumulate entry points; the deterministic backward refuses head dim 256."""
import math

import numpy as np
import pytest
import torch

import oracle
from synthetic import MaskSpec, qkv
from test_gpu_parity import relf, run_and_compare, spec_for

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


@pytest.mark.parametrize("kind", ["FULL", "CAUSAL", "CAUSAL_DOCUMENT", "CAUSAL_SLIDING_WINDOW",
                                  "PREFIX_LM_CAUSAL", "SHARED_QUESTION", "UNIFORM_BLOCK", "VARIABLE_BLOCK"])
def test_hd256_backward_families(kind):
    """GQA 4:2, N = 392 (a ragged last tile): split head shares (units are few)."""
    N, Hq, Hkv = 392, 4, 2
    run_and_compare(spec_for(kind, N, Hq), 1, N, Hq, Hkv, seed=21, D=D)


@pytest.mark.parametrize("B,N,Hq,Hkv,kind", [(2, 300, 3, 3, "CAUSAL"), (1, 1100, 6, 1, "FULL_DOCUMENT"),
                                             (1, 129, 2, 2, "GLOBAL_SLIDING")])
def test_hd256_backward_batch_mha_mqa(B, N, Hq, Hkv, kind):
    run_and_compare(spec_for(kind, N, Hq), B, N, Hq, Hkv, seed=22, D=D)


def test_hd256_backward_unsplit_long_lists():
    """2048 tokens, GQA 3:1 (a group that does not split evenly: no partials),
    16 query tiles per unit, so the half-tile ring wraps many times."""
    run_and_compare(spec_for("CAUSAL", 2048, 3), 1, 2048, 3, 1, seed=23, check_classes=False, D=D)


def test_hd256_noalloc_and_accumulate_match_oracle():
    """lcattn_bwd_noalloc and lcattn_bwd_accum (fp32 accumulators that start at
    zero) at head dim 256 against the oracle; the deterministic backward refuses."""
    B, N, Hq, Hkv = 1, 520, 4, 2
    spec = MaskSpec("CAUSAL")
    x = qkv(B, N, Hq, Hkv, D, seed=24)
    dev = {n: t.cuda() for n, t in x.items()}
    out = lc.attention(dev["q"], dev["k"], dev["v"], spec)
    mask, meta = out["mask"], out["tile_meta"]
    dq, dk, dv = lc.lcattn_bwd_noalloc(dev["q"], dev["k"], dev["v"], out["o"], dev["do"], out["lse"], mask, meta)
    acc = {n: torch.zeros(t.shape, dtype=torch.float32, device="cuda") for n, t in
           (("dq", dev["q"]), ("dk", dev["k"]), ("dv", dev["v"]))}
    lc.lcattn_bwd_accum(dev["q"], dev["k"], dev["v"], out["o"], dev["do"], out["lse"], mask, meta,
                        acc["dq"], acc["dk"], acc["dv"])
    torch.cuda.synchronize()
    assert lc.lcattn_read_status(meta) == 0
    f64 = {n: t.double().numpy() for n, t in x.items()}
    dQ, dK, dV, _, _ = oracle.attention_bwd(f64["q"], f64["k"], f64["v"], f64["do"], spec, 1.0 / math.sqrt(D))
    for got in ((dq, dk, dv), (acc["dq"], acc["dk"], acc["dv"])):
        for g, ref, name in zip(got, (dQ, dK, dV), ("dq", "dk", "dv")):
            assert relf(g.double().cpu().numpy(), ref) <= 3e-2, name
    with pytest.raises(lc.LcattnError) as err:
        lc.lcattn_bwd_deterministic(dev["q"], dev["k"], dev["v"], out["o"], dev["do"], out["lse"], mask, meta,
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


@pytest.mark.parametrize("Sq,Sk,Hq,Hkv,kind", [(300, 777, 4, 2, "CAUSAL"), (700, 129, 2, 1, "FULL"),
                                               (40, 2600, 4, 4, "CAUSAL_SLIDING_WINDOW")])
def test_hd256_rectangular_backward(Sq, Sk, Hq, Hkv, kind):
    """Sq != Sk at head dim 256 (bottom-right aligned), forward and backward
    against the oracle: ragged tiles on both axes, more queries than keys."""
    B = 1
    spec = MaskSpec(kind, {"window": Sk // 3} if "WINDOW" in kind else {})
    x = qkv(B, Sq, Hq, Hkv, D, seed=Sq + Sk, Sk=Sk)
    dev = {n: t.cuda() for n, t in x.items()}
    out = lc.attention(dev["q"], dev["k"], dev["v"], spec, d_o=dev["do"])
    torch.cuda.synchronize()
    assert lc.lcattn_read_status(out["tile_meta"]) == 0
    f64 = {n: t.double().numpy() for n, t in x.items()}
    dQ, dK, dV, O, LSE = oracle.attention_bwd(f64["q"], f64["k"], f64["v"], f64["do"], spec, 1.0 / math.sqrt(D))
    g = out["o"].double().cpu().numpy()
    assert np.abs(g - O).max() <= 2e-2 and relf(g, O) <= 1e-2
    lse = out["lse"].double().cpu().numpy()
    fin = np.isfinite(LSE)
    np.testing.assert_array_equal(np.isfinite(lse), fin)
    if fin.any():
        assert np.abs(lse[fin] - LSE[fin]).max() <= 5e-3
    for name, ref in (("dq", dQ), ("dk", dK), ("dv", dV)):
        assert relf(out[name].double().cpu().numpy(), ref) <= 3e-2, name
