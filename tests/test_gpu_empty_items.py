"""Work items with empty key lists in the persistent forward.  The mask
compiler's longest-first order puts them at the end, so one CTA can fetch a
non-empty item and then more empty ones than its item queue holds.  The
forward must close the non-empty item (issue its last PV) without waiting for
another non-empty item.  Covered for one-head items (a block map with empty
query blocks) and two-head items (bottom-right causal with far more queries
than keys), at head dims 128, 64 and 256, against the oracle on sampled rows."""
import math

import numpy as np
import pytest
import torch

import oracle
from synthetic import MaskSpec, block_keep, qkv

pytestmark = pytest.mark.gpu

lc = pytest.importorskip("long_context_masked_mask_gb300")


def relf(g, r):
    return float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30))


def run(spec, B, Sq, Sk, Hq, Hkv, D, seed=0):
    x = qkv(B, Sq, Hq, Hkv, D, seed=seed, Sk=Sk, with_do=False)
    dev = {n: t.cuda() for n, t in x.items()}
    mask = lc.DeviceMask(spec, Sq, Hq, B, device="cuda", Sk=Sk)
    shape = lc.make_shape(dev["q"], dev["k"], dev["v"])
    meta = lc.lcattn_mask_compile(shape, mask)
    o, lse = lc.lcattn_fwd(dev["q"], dev["k"], dev["v"], mask, meta)
    torch.cuda.synchronize()
    assert lc.lcattn_read_status(meta) == 0, "a bounded wait expired"
    f64 = {n: t.double().numpy() for n, t in x.items()}
    rng = np.random.default_rng(seed)
    rows = np.array(sorted({0, 127, 128, Sq - 1, Sq - 129} | {int(r) for r in rng.integers(0, Sq, 30)}))
    scale = 1.0 / math.sqrt(D)
    for h in (0, Hq // 2, Hq - 1):
        ref_o, ref_l = oracle.attention_fwd_rows(f64["q"], f64["k"], f64["v"], spec, scale, 0, h, rows)
        g = o[0, rows, h].double().cpu().numpy()
        assert np.abs(g - ref_o).max() <= 2e-2 and relf(g, ref_o) <= 1e-2
        gl = lse[0, h, rows].double().cpu().numpy()
        fin = np.isfinite(ref_l)
        np.testing.assert_array_equal(np.isfinite(gl), fin)
        if fin.any():
            assert np.abs(gl[fin] - ref_l[fin]).max() <= 5e-3


@pytest.mark.parametrize("D", [128, 64, 256])
def test_block_map_with_empty_query_blocks(D):
    N, Hq, Hkv = 4096, 16, 4
    nb = N // 128
    keep = block_keep(Hq, nb, nb, 0.3, 5, force_diagonal=False)
    keep[:, ::3, :] = False
    run(MaskSpec("UNIFORM_BLOCK", {"block": 128, "keep": keep}), 1, N, N, Hq, Hkv, D, seed=D)


@pytest.mark.parametrize("D", [128, 64])
def test_bottom_right_causal_with_empty_query_tiles(D):
    """Sq = 8192 queries against Sk = 1024 keys: the first 7168 rows (56 of 64
    query tiles) see no key; two heads per item (GQA 16:8)."""
    run(MaskSpec("CAUSAL"), 1, 8192, 1024, 16, 8, D, seed=D + 1)
