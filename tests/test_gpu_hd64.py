"""Head dim 64 (a variant next to the pages' 128): forward and backward through
the C ABI against the fp64 oracle, with the bars of the 128 case.  Covers the
mask families on both descriptor kinds, GQA and MHA, batch 2, ragged lengths,
query and key lengths that differ (regular and split-KV forwards), and a
larger problem whose dK/dV units are not split."""
import math

import numpy as np
import pytest
import torch

import oracle
from synthetic import MaskSpec, qkv
from test_gpu_parity import relf, run_and_compare, spec_for

pytestmark = pytest.mark.gpu

lc = pytest.importorskip("long_context_masked_mask_gb300")

KINDS_64 = ["FULL", "CAUSAL", "CAUSAL_DOCUMENT", "CAUSAL_SLIDING_WINDOW", "SHARED_QUESTION",
            "PREFIX_LM_DOCUMENT", "UNIFORM_BLOCK", "VARIABLE_BLOCK"]


@pytest.mark.parametrize("kind", KINDS_64)
def test_hd64_mask_family_gqa_ragged(kind):
    N, Hq, Hkv = 392, 4, 2
    run_and_compare(spec_for(kind, N, Hq), 1, N, Hq, Hkv, D=64)


@pytest.mark.parametrize("B,N,Hq,Hkv,kind", [(2, 300, 3, 3, "CAUSAL"), (1, 1000, 8, 1, "FULL_DOCUMENT"),
                                             (1, 129, 2, 2, "GLOBAL_SLIDING")])
def test_hd64_batch_mha_mqa(B, N, Hq, Hkv, kind):
    run_and_compare(spec_for(kind, N, Hq), B, N, Hq, Hkv, seed=4, D=64)


@pytest.mark.parametrize("Sq,Sk,Hq,Hkv,kind", [(1, 3000, 16, 2, "CAUSAL"), (40, 2600, 4, 4, "FULL"),
                                               (200, 129, 4, 2, "CAUSAL"), (700, 2500, 8, 2, "CAUSAL_SLIDING_WINDOW")])
def test_hd64_rectangular(Sq, Sk, Hq, Hkv, kind):
    """Sq != Sk, forward (attention() takes the split-KV path where it applies,
    and the persistent forward is checked too) and backward."""
    B, D = 1, 64
    spec = MaskSpec(kind, {"window": Sk // 3} if "WINDOW" in kind else {})
    x = qkv(B, Sq, Hq, Hkv, D, seed=Sq + Sk, Sk=Sk)
    dev = {n: t.cuda() for n, t in x.items()}
    out = lc.attention(dev["q"], dev["k"], dev["v"], spec, d_o=dev["do"])
    o2, _ = lc.lcattn_fwd(dev["q"], dev["k"], dev["v"], out["mask"], out["tile_meta"])
    torch.cuda.synchronize()
    assert lc.lcattn_read_status(out["tile_meta"]) == 0
    f64 = {n: t.double().numpy() for n, t in x.items()}
    dQ, dK, dV, O, LSE = oracle.attention_bwd(f64["q"], f64["k"], f64["v"], f64["do"], spec,
                                              1.0 / math.sqrt(D))
    for o in (out["o"], o2):
        g = o.double().cpu().numpy()
        assert np.abs(g - O).max() <= 2e-2 and relf(g, O) <= 1e-2
    lse = out["lse"].double().cpu().numpy()
    fin = np.isfinite(LSE)
    np.testing.assert_array_equal(np.isfinite(lse), fin)
    if fin.any():
        assert np.abs(lse[fin] - LSE[fin]).max() <= 5e-3
    for name, ref in (("dq", dQ), ("dk", dK), ("dv", dV)):
        assert relf(out[name].double().cpu().numpy(), ref) <= 3e-2, name


def test_hd64_unsplit_units():
    """2048 tokens, GQA 3:1: a group that does not split evenly, so dK/dV units
    are not split over head shares (no partials), with 16 query tiles per unit."""
    run_and_compare(spec_for("CAUSAL", 2048, 3), 1, 2048, 3, 1, seed=9, check_classes=False, D=64)
