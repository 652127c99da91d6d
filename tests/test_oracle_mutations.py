"""The oracle's pins reject planted mistakes (CPU only).

Each case takes the oracle's own source, changes one token -- an off-by-one in
a mask predicate, a dropped softmax scale, a wrong GQA head mapping, a dropped
D term in dS, a transposed operand, an overwrite where a sum belongs -- runs the
mutant as a fresh module, and requires at least one pin that does not depend
on the oracle's arithmetic to fail:

* the hand-derived golden masks and tile classes under ``tests/golden``;
* torch's fp64 ``scaled_dot_product_attention`` with autograd, on a small GQA
  case that also has fully-masked query rows and several row chunks;
* for the block selection: the hand-derived maps of ``select_small.json``,
  brute force over subsets, the pooled-score identity and the causal rule
  checked position by position (``test_oracle_block_select``).

The mutants exist only in this test process; the oracle files are not touched.
"""
import inspect
import json
import math
import os
import types

import numpy as np
import pytest
import torch

import oracle.attention_ref as attention_ref
import oracle.masks_ref as masks_ref
from synthetic import MaskSpec

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
_pristine_allowed = masks_ref.allowed


def mutant(module, old, new, occurrence=0):
    """A fresh copy of ``module`` with the ``occurrence``-th ``old`` replaced by ``new``."""
    src = inspect.getsource(module)
    at = -1
    for _ in range(occurrence + 1):
        at = src.find(old, at + 1)
        assert at >= 0, f"mutation anchor not found: {old!r}"
    src = src[:at] + new + src[at + len(old):]
    mod = types.ModuleType(module.__name__ + "_mutant")
    mod.__package__ = "oracle"
    exec(compile(src, f"<mutant of {module.__name__}>", "exec"), mod.__dict__)
    return mod


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)["cases"]


def _params(case):
    params = dict(case["params"])
    if "keep" in params:
        params["keep"] = np.array(params["keep"], dtype=bool)
    return params


def golden_masks_hold(mr):
    for case in _golden("masks_small.json"):
        want = np.array([[c == "1" for c in row] for row in case["rows"]], dtype=bool)
        got = mr.allowed(MaskSpec(case["kind"], _params(case)), case["N"], Sk=case.get("Sk"))
        if got.shape != want.shape or not np.array_equal(got, want):
            return False
    return True


def golden_tiles_hold(ar):
    code = {"E": ar.EMPTY, "F": ar.FULL, "P": ar.PARTIAL}
    for case in _golden("tiles_small.json"):
        want = np.array([[code[c] for c in row] for row in case["classes"]], dtype=np.uint8)
        got = ar.classify_tiles(MaskSpec(case["kind"], _params(case)), case["N"], case["BM"], case["BN"])
        if got.shape != want.shape or not np.array_equal(got, want):
            return False
    return True


# Small GQA problem: 4 query heads over 2 KV heads, N = 13.  The block map
# leaves query rows 0..3 of head 1 with nothing allowed, so the fully-masked
# convention (O = 0, LSE = -inf, no gradient) is exercised too.
_B, _N, _HQ, _HKV, _D = 1, 13, 4, 2, 8
_KEEP = np.array([[[1, 0, 1, 1], [1, 1, 0, 0], [0, 1, 1, 0], [1, 1, 1, 1]],
                  [[0, 0, 0, 0], [1, 1, 0, 0], [0, 0, 1, 1], [1, 0, 0, 1]],
                  [[1, 1, 1, 1], [0, 1, 0, 1], [1, 0, 1, 0], [0, 0, 1, 1]],
                  [[1, 0, 0, 0], [1, 1, 0, 0], [1, 1, 1, 0], [1, 1, 1, 1]]], dtype=bool)
_SPECS = [MaskSpec("CAUSAL_SLIDING_WINDOW", {"window": 5}),
          MaskSpec("UNIFORM_BLOCK", {"block": 4, "keep": _KEEP})]


def _inputs():
    rng = np.random.default_rng(3)
    return [rng.standard_normal(s) for s in ((_B, _N, _HQ, _D), (_B, _N, _HKV, _D),
                                             (_B, _N, _HKV, _D), (_B, _N, _HQ, _D))]


def _torch_reference(q, k, v, do, spec, scale):
    G = _HQ // _HKV
    qt, kt, vt = (torch.tensor(x).permute(0, 2, 1, 3).requires_grad_(True) for x in (q, k, v))
    mask = torch.stack([torch.tensor(_pristine_allowed(spec, _N, head=h)) for h in range(_HQ)])[None]
    rows_any = mask.any(-1, keepdim=True)
    o = torch.nn.functional.scaled_dot_product_attention(
        qt, kt.repeat_interleave(G, 1), vt.repeat_interleave(G, 1),
        attn_mask=mask | ~rows_any, scale=scale)
    o = o * rows_any  # rows that allow nothing are zero by definition
    (o * torch.tensor(do).permute(0, 2, 1, 3)).sum().backward()
    back = lambda t: t.detach().permute(0, 2, 1, 3).numpy()
    return back(o), back(qt.grad), back(kt.grad), back(vt.grad), rows_any[0, :, :, 0].numpy()


def torch_pin_holds(ar):
    q, k, v, do = _inputs()
    scale = 1.0 / math.sqrt(_D)
    close = lambda a, b: a.shape == b.shape and np.allclose(a, b, rtol=0, atol=1e-10)
    for spec in _SPECS:
        O, dQ, dK, dV, has = _torch_reference(q, k, v, do, spec, scale)
        # chunk = 5 splits the rows into three chunks, so per-chunk sums are exercised
        gQ, gK, gV, gO, LSE = ar.attention_bwd(q, k, v, do, spec, scale, chunk=5)
        if not all(close(a, b) for a, b in ((gO, O), (gQ, dQ), (gK, dK), (gV, dV))):
            return False
        if not np.array_equal(np.isfinite(LSE[0]), has):
            return False
        # Row subsets: dQ and O rows as torch's, and the dK/dV terms of a
        # partition of every head's rows summing to torch's dK/dV.
        rK, rV = np.zeros_like(dK[0]), np.zeros_like(dV[0])
        for h in range(_HQ):
            for part in (np.arange(0, 6), np.arange(6, _N)):
                pQ, pK, pV, pO, _ = ar.attention_bwd_rows(q, k, v, do, spec, scale, 0, h, part)
                if not (close(pQ, dQ[0, part, h]) and close(pO, O[0, part, h])):
                    return False
                rK[:, h // 2] += pK
                rV[:, h // 2] += pV
        if not (close(rK, dK[0]) and close(rV, dV[0])):
            return False
        cols, rows = np.array([0, 4, 7, 12]), np.array([1, 5, 12])
        for g in range(_HKV):
            sQ, sK, sV = ar.attention_bwd_sampled(q, k, v, do, spec, scale, 0, g, rows, cols)
            heads = slice(g * 2, g * 2 + 2)
            if not (close(sQ, dQ[0][rows][:, heads].transpose(1, 0, 2))
                    and close(sK, dK[0, cols, g]) and close(sV, dV[0, cols, g])):
                return False
    return True


def test_pins_accept_the_oracle():
    assert golden_masks_hold(masks_ref)
    assert golden_tiles_hold(attention_ref)
    assert torch_pin_holds(attention_ref)


MASK_MUTANTS = [
    ("causal strict", "return j <= i\n", "return j < i\n"),
    ("causal window one wider", "(d < p[\"window\"])", "(d <= p[\"window\"])"),
    ("sliding window one wider", "np.abs(i - j) < p[\"window\"]", "np.abs(i - j) <= p[\"window\"]"),
    ("shared question drops the question", "(sj == 0) | (sj == si)", "(sj == si)"),
    ("global rows dropped", "(i < g) | (j < g)", "(j < g)"),
    ("blockwise last block not global", "(bi == bj) | (bi == last)", "(bi == bj)"),
    ("prefix one longer", "(j < p[\"prefix\"])", "(j <= p[\"prefix\"])"),
    ("prefix ignores documents", "(di == dj) & (in_prefix", "(in_prefix"),
    ("block causal strict", "(bj <= bi)", "(bj < bi)"),
    ("segment boundary side", "side=\"right\"", "side=\"left\""),
    ("uniform block transposed", "keep[i // bs, j // bs]", "keep[j // bs, i // bs]"),
    ("top-left alignment for Sq != Sk", "i = i + (Sk - N)", "i = i + 0"),
    ("alignment shift reversed", "i = i + (Sk - N)", "i = i + (N - Sk)"),
    ("variable block lens swapped", "keep[_segment_of(i, p[\"q_block_lens\"]), _segment_of(j, p[\"k_block_lens\"])]",
     "keep[_segment_of(i, p[\"k_block_lens\"]), _segment_of(j, p[\"q_block_lens\"])]"),
]


@pytest.mark.parametrize("name,old,new", MASK_MUTANTS, ids=[m[0] for m in MASK_MUTANTS])
def test_golden_masks_reject_mask_mutant(name, old, new):
    assert not golden_masks_hold(mutant(masks_ref, old, new))


ATTN_MUTANTS = [
    ("dropped scale in S", "S = scale * (qr @ k.T)", "S = (qr @ k.T)", 0),
    ("LSE without the max", "m_safe + np.log(", "np.log(", 0),
    ("P not normalised", "P = E / np.where(has, l, 1.0)[:, None]", "P = E", 0),
    ("GQA head map in the forward", "g = h // G", "g = h % Hkv", 0),
    ("GQA head map in the backward", "g = h // G", "g = h % Hkv", 1),
    ("dropped D term", "dS = P * (dP - Dr[:, None])", "dS = P * dP", 0),
    ("D from dO alone", "Dr = (dOr * O[b, rows, h]).sum(axis=1)", "Dr = (dOr * dOr).sum(axis=1)", 0),
    ("dV overwritten across heads", "dV[b, :, g] += P.T @ dOr", "dV[b, :, g] = P.T @ dOr", 0),
    ("dQ without scale", "dQ[b, rows, h] = scale * (dS @ kk)", "dQ[b, rows, h] = (dS @ kk)", 0),
    ("dK transposed operand", "scale * (dS.T @ q[b, rows, h])", "scale * (dS.T @ do[b, rows, h])", 0),
    ("dP transposed operand", "dP = dOr @ vv.T\n                Dr", "dP = dOr @ kk.T\n                Dr", 0),
    ("sampled path misses rows", "need = allowed(spec, N, rows, head=h, cols=k_cols, Sk=Sk).any(axis=1)",
     "need = allowed(spec, N, rows, head=h, cols=k_cols, Sk=Sk).all(axis=1)", 0),
    ("sampled dK without scale", "dK += scale * (dSc.T @ q[b, rr, h])", "dK += (dSc.T @ q[b, rr, h])", 0),
    ("row-subset dS drops D", "dS = P * (dP - Dr[:, None])", "dS = P * dP", 1),
    ("row-subset dK without scale", "dK = scale * (dS.T @ q[b, rows, h])", "dK = (dS.T @ q[b, rows, h])", 0),
    ("row-subset dV from Q", "dV = P.T @ dOr", "dV = P.T @ q[b, rows, h]", 0),
    ("row-subset GQA head map", "kk, vv = k[b, :, h // G], v[b, :, h // G]", "kk, vv = k[b, :, h % 2], v[b, :, h % 2]", 0),
    ("sampled dQ drops D", "dS = P * (dP - Dr[:, None])", "dS = P * dP", 2),
]


@pytest.mark.parametrize("name,old,new,occ", ATTN_MUTANTS, ids=[m[0] for m in ATTN_MUTANTS])
def test_torch_pin_rejects_attention_mutant(name, old, new, occ):
    assert not torch_pin_holds(mutant(attention_ref, old, new, occ))


TILE_MUTANTS = [
    ("ragged column tile one wider", "M[:, kt * BN:min(Sk, (kt + 1) * BN)]", "M[:, kt * BN:min(Sk, (kt + 1) * BN + 1)]"),
    ("ragged row tile cut short", "np.arange(qt * BM, min(N, (qt + 1) * BM))", "np.arange(qt * BM, min(N - 1, (qt + 1) * BM))"),
    ("FULL and PARTIAL swapped", "out[r, kt] = FULL\n", "out[r, kt] = PARTIAL\n"),
]


@pytest.mark.parametrize("name,old,new", TILE_MUTANTS, ids=[m[0] for m in TILE_MUTANTS])
def test_golden_tiles_reject_tile_mutant(name, old, new):
    assert not golden_tiles_hold(mutant(attention_ref, old, new))


# ---- block selection (TopK / TopP over pooled Q K^T) ------------------------
import oracle.block_select_ref as block_select_ref  # noqa: E402
from test_oracle_block_select import select_pins_hold  # noqa: E402


def test_select_pins_accept_the_oracle():
    assert select_pins_hold(block_select_ref)


SELECT_MUTANTS = [
    ("sum_pool", ".mean(axis=1)", ".sum(axis=1)", 0),
    ("first_row_pool", "x[:, lo:hi, :, :].astype(np.float64).mean(axis=1)",
     "x[:, lo, :, :].astype(np.float64)", 0),
    ("block_end_off_by_one", "offs[i + 1])", "offs[i + 1]) - 1", 0),
    ("gqa_modulo", "kb[:, h // G]", "kb[:, h % Hkv]", 0),
    ("scale_dropped", "scale * np.einsum", "np.einsum", 0),
    ("causal_le", "k_offs[:-1][None, :] < q_offs[1:][:, None]", "k_offs[:-1][None, :] <= q_offs[1:][:, None]", 0),
    ("causal_query_start", "k_offs[:-1][None, :] < q_offs[1:][:, None]", "k_offs[:-1][None, :] < q_offs[:-1][:, None]", 0),
    ("empty_key_block_kept", "c = q_nonempty[:, None] & k_nonempty[None, :]",
     "c = q_nonempty[:, None] & np.ones_like(k_nonempty)[None, :]", 0),
    ("rank_ascending", "np.lexsort((idx, -s))", "np.lexsort((idx, s))", 0),
    ("tie_larger_index", "np.lexsort((idx, -s))", "np.lexsort((-idx, -s))", 0),
    ("topk_off_by_one", "[:max(int(k), 0)]", "[:max(int(k) + 1, 0)]", 0),
    ("topp_le", "mass_before < p", "mass_before <= p", 0),
    ("topp_inclusive_mass", "np.concatenate([[0.0], np.cumsum(prob)[:-1]])", "np.cumsum(prob)", 0),
    ("topp_unnormalised", "prob = e / e.sum()", "prob = e", 0),
]


@pytest.mark.parametrize("name,old,new,occ", SELECT_MUTANTS, ids=[m[0] for m in SELECT_MUTANTS])
def test_select_pins_reject_mutant(name, old, new, occ):
    assert not select_pins_hold(mutant(block_select_ref, old, new, occ))
