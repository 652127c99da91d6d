"""GPU parity when query and key lengths differ (Sq != Sk), bottom-right
aligned: decode-style rows (Sq = 1, 3), chunks of queries against a longer key
sequence, more queries than keys (the first Sq - Sk rows of a causal mask allow
nothing), ragged tiles on both axes, MHA and GQA, column bounds and block maps.
Everything goes through the C ABI; the bars are the square case's: O max-abs
2e-2 and relative Frobenius 1e-2, dQ/dK/dV relative Frobenius 3e-2, LSE
max-abs 5e-3 with -inf exactly where the oracle has it, tile classes bit-exact."""
import math

import numpy as np
import pytest
import torch

import oracle
from synthetic import MaskSpec, block_keep, qkv

pytestmark = pytest.mark.gpu

lc = pytest.importorskip("long_context_masked_mask_gb300")


def relf(g, r):
    nr = np.linalg.norm(r)
    return float(np.linalg.norm(g - r) / nr) if nr > 0 else float(np.linalg.norm(g))


def spec_for(kind, Sq, Sk, Hq):
    if kind == "CAUSAL_SLIDING_WINDOW":
        return MaskSpec(kind, {"window": max(1, Sk // 3)})
    if kind == "FULL_SLIDING_WINDOW":
        return MaskSpec(kind, {"window": max(1, Sk // 4)})
    if kind == "UNIFORM_BLOCK":
        bs = 64
        return MaskSpec(kind, {"block": bs, "keep": block_keep(Hq, -(-Sq // bs), -(-Sk // bs), 0.5, 7,
                                                               force_diagonal=False)})
    return MaskSpec(kind)


SHAPES = [(1, 1000), (3, 777), (64, 1000), (129, 300), (300, 129), (500, 2000), (700, 1)]
KINDS = ["FULL", "CAUSAL", "CAUSAL_SLIDING_WINDOW", "FULL_SLIDING_WINDOW", "UNIFORM_BLOCK"]


@pytest.mark.parametrize("Sq,Sk", SHAPES, ids=[f"q{a}_k{b}" for a, b in SHAPES])
@pytest.mark.parametrize("kind", KINDS)
def test_rectangular_matches_oracle(Sq, Sk, kind):
    B, Hq, Hkv, D = (2, 4, 2, 128) if Sq * Sk <= 300000 else (1, 4, 2, 128)
    spec = spec_for(kind, Sq, Sk, Hq)
    x = qkv(B, Sq, Hq, Hkv, D, seed=Sq + 7 * Sk, Sk=Sk)
    dev = {n: t.cuda() for n, t in x.items()}
    out = lc.attention(dev["q"], dev["k"], dev["v"], spec, d_o=dev["do"])
    torch.cuda.synchronize()
    assert lc.lcattn_read_status(out["tile_meta"]) == 0
    scale = 1.0 / math.sqrt(D)
    f64 = {n: t.double().numpy() for n, t in x.items()}
    dQ, dK, dV, O, LSE = oracle.attention_bwd(f64["q"], f64["k"], f64["v"], f64["do"], spec, scale)
    o = out["o"].double().cpu().numpy()
    assert np.abs(o - O).max() <= 2e-2 and relf(o, O) <= 1e-2
    lse = out["lse"].double().cpu().numpy()
    fin = np.isfinite(LSE)
    np.testing.assert_array_equal(np.isfinite(lse), fin)
    if fin.any():
        assert np.abs(lse[fin] - LSE[fin]).max() <= 5e-3
    for name, ref in (("dq", dQ), ("dk", dK), ("dv", dV)):
        g = out[name].double().cpu().numpy()
        assert relf(g, ref) <= 3e-2, (name, relf(g, ref))
    # tile classes, bit-exact
    shape = lc.make_shape(dev["q"], dev["k"], dev["v"])
    cls = lc.tile_classes(out["tile_meta"], shape, out["mask"]).cpu().numpy()
    for h in ([0, Hq - 1] if spec.per_head else [0]):
        want = oracle.classify_tiles(spec, Sq, 128, 128, head=h, Sk=Sk)
        np.testing.assert_array_equal(cls[0, h if spec.per_head else 0], want)


def test_more_queries_than_keys_leaves_leading_rows_empty():
    """CAUSAL with Sq = 300 > Sk = 129: rows 0..170 allow nothing (O = 0,
    LSE = -inf, no gradient); the rest see every key up to their position."""
    B, Sq, Sk, Hq, Hkv, D = 1, 300, 129, 2, 1, 128
    x = qkv(B, Sq, Hq, Hkv, D, seed=3, Sk=Sk)
    dev = {n: t.cuda() for n, t in x.items()}
    out = lc.attention(dev["q"], dev["k"], dev["v"], MaskSpec("CAUSAL"), d_o=dev["do"])
    torch.cuda.synchronize()
    empty = Sq - Sk
    assert torch.isinf(out["lse"][:, :, :empty]).all() and (out["lse"][:, :, :empty] < 0).all()
    assert torch.isfinite(out["lse"][:, :, empty:]).all()
    assert (out["o"][:, :empty] == 0).all() and (out["dq"][:, :empty] == 0).all()


SPLIT_CASES = [
    # B, Sq, Sk, Hq, Hkv, kind
    (1, 1, 4096, 64, 8, "CAUSAL"),         # one decode row per sequence, GQA 8 packed per tile
    (3, 1, 2500, 16, 2, "FULL"),           # ragged key tail
    (2, 5, 3000, 8, 2, "CAUSAL_SLIDING_WINDOW"),
    (1, 40, 5000, 4, 4, "CAUSAL"),         # MHA: one head per tile, 128 positions
    (1, 200, 6000, 12, 4, "FULL_SLIDING_WINDOW"),  # G = 3: heads are not packed
    (1, 2200, 2048, 2, 1, "CAUSAL"),       # more queries than keys: leading rows empty
]


@pytest.mark.parametrize("B,Sq,Sk,Hq,Hkv,kind", SPLIT_CASES,
                         ids=[f"b{c[0]}_q{c[1]}_k{c[2]}_{c[3]}x{c[4]}_{c[5]}" for c in SPLIT_CASES])
def test_split_forward_matches_oracle(B, Sq, Sk, Hq, Hkv, kind):
    """lcattn_fwd_ws takes the split-KV path on these shapes (its workspace is
    non-empty); O and LSE must match the oracle, and the regular forward."""
    D = 128
    spec = spec_for(kind, Sq, Sk, Hq)
    x = qkv(B, Sq, Hq, Hkv, D, seed=11 * Sq + Sk, Sk=Sk, with_do=False)
    dev = {n: t.cuda() for n, t in x.items()}
    mask = lc.DeviceMask(spec, Sq, Hq, B, device="cuda", Sk=Sk)
    shape = lc.make_shape(dev["q"], dev["k"], dev["v"])
    meta = lc.lcattn_mask_compile(shape, mask)
    assert lc.lcattn_fwd_workspace_size(shape, mask) > 0, "expected the split path"
    o, lse = lc.lcattn_fwd_ws(dev["q"], dev["k"], dev["v"], mask, meta)
    o_reg, lse_reg = lc.lcattn_fwd(dev["q"], dev["k"], dev["v"], mask, meta)
    torch.cuda.synchronize()
    assert lc.lcattn_read_status(meta) == 0
    scale = 1.0 / math.sqrt(D)
    f64 = {n: t.double().numpy() for n, t in x.items()}
    O, LSE = oracle.attention_fwd(f64["q"], f64["k"], f64["v"], spec, scale)
    for oo, ll in ((o, lse), (o_reg, lse_reg)):
        g = oo.double().cpu().numpy()
        assert np.abs(g - O).max() <= 2e-2 and relf(g, O) <= 1e-2
        gl = ll.double().cpu().numpy()
        fin = np.isfinite(LSE)
        np.testing.assert_array_equal(np.isfinite(gl), fin)
        if fin.any():
            assert np.abs(gl[fin] - LSE[fin]).max() <= 5e-3
    # The split result agrees with the regular path to bf16 rounding.
    assert (o.float() - o_reg.float()).abs().max().item() <= 1e-2
