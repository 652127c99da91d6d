"""Block-map backward with chunked dK/dV units: lcattn_bwd splits the units
of a mask with per-head lists and at least 512 query tiles into ranges of 64
query tiles, launched chunk-major, with dK/dV reduce-added into an fp32
accumulator.  Checked through the C ABI at N = 65836 (9 chunks, the last of
one ragged tile), GQA 2:1, a uniform and a variable block map, and the uniform
map at head dim 256 (two CTAs per unit, one per head-dim half):

* dQ on sampled query rows (the ragged tail included) against the fp64 oracle,
  relF <= 3e-2, and O within the forward's bars;
* dK and dV against the unchunked accumulate-mode backward (lcattn_bwd_accum,
  itself checked against the oracle by the ring tests), relF <= 1e-2;
* the identities sum_j dK_j = 0 and sum_j dV_j = sum of dO over rows that
  allow a key, per KV head.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from synthetic import MaskSpec, block_keep, qkv, segment_lengths

pytestmark = pytest.mark.gpu

lc = pytest.importorskip("long_context_masked_mask_gb300")


def relf(g, r):
    return float(np.linalg.norm(g - r) / np.linalg.norm(r))


@pytest.mark.parametrize("kind,D", [("UNIFORM_BLOCK", 128), ("VARIABLE_BLOCK", 128), ("UNIFORM_BLOCK", 256)])
def test_chunked_block_map_backward(kind, D):
    B, N, Hq, Hkv = 1, 65836, 2, 1  # 515 query tiles: 9 chunks of 64 (the last has 3)
    if kind == "UNIFORM_BLOCK":
        nb = -(-N // 128)
        spec = MaskSpec("UNIFORM_BLOCK", {"block": 128, "keep": block_keep(Hq, nb, nb, 0.2, 1)})
    else:
        ql = segment_lengths(N, 200, 1500, 4)
        kl = segment_lengths(N, 200, 1500, 5)
        keep = block_keep(Hq, len(ql), len(kl), 0.2, 6, force_diagonal=False)
        keep[:, 3, :] = False  # a query block with no keys: fully masked rows
        spec = MaskSpec("VARIABLE_BLOCK", {"q_block_lens": ql, "k_block_lens": kl, "keep": keep})
    x = qkv(B, N, Hq, Hkv, D, seed=17)
    dev = {k: t.cuda() for k, t in x.items()}
    out = lc.attention(dev["q"], dev["k"], dev["v"], spec, d_o=dev["do"])
    m, meta = out["mask"], out["tile_meta"]
    acc = [torch.zeros(t.shape, dtype=torch.float32, device="cuda") for t in (dev["q"], dev["k"], dev["v"])]
    lc.lcattn_bwd_accum(dev["q"], dev["k"], dev["v"], out["o"], dev["do"], out["lse"], m, meta, *acc)
    torch.cuda.synchronize()
    assert lc.lcattn_read_status(meta) == 0
    f = {k: t.double().numpy() for k, t in x.items()}
    s = 1.0 / math.sqrt(D)
    rows = np.array([0, 1, 700, 5000, 33333, 65535, 65600, 65835])
    for h in range(Hq):
        o_ref, _ = oracle.attention_fwd_rows(f["q"], f["k"], f["v"], spec, s, 0, h, rows)
        o = out["o"][0, rows, h].double().cpu().numpy()
        assert np.abs(o - o_ref).max() <= 2e-2
    dq_ref, _, _ = oracle.attention_bwd_sampled(f["q"], f["k"], f["v"], f["do"], spec, s, 0, 0, rows, [])
    dq = out["dq"][0][rows].double().cpu().numpy().transpose(1, 0, 2)
    assert relf(dq, dq_ref) <= 3e-2, relf(dq, dq_ref)
    for name, got, ref in (("dk", out["dk"], acc[1]), ("dv", out["dv"], acc[2])):
        g, r = got.double().cpu().numpy(), ref.double().cpu().numpy()
        assert relf(g, r) <= 1e-2, (name, relf(g, r))
    # Identities (one KV head): residuals within 3e-2 of the gradient's norm.
    dk = out["dk"][0, :, 0].double().cpu().numpy()
    dv = out["dv"][0, :, 0].double().cpu().numpy()
    has = torch.isfinite(out["lse"][0]).cpu().numpy()          # [Hq, N]: rows that allow a key
    do_sum = sum((f["do"][0, :, h] * has[h][:, None]).sum(0) for h in range(Hq))
    assert np.linalg.norm(dk.sum(0)) <= 3e-2 * np.linalg.norm(dk)
    assert np.linalg.norm(dv.sum(0) - do_sum) <= 3e-2 * np.linalg.norm(dv)
