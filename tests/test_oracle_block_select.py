"""Pins of the block-selection oracle (TopK / TopP over pooled Q K^T).

The pins come from outside the oracle: hand-derived maps (tests/golden/
select_small.json), brute force over every subset on tiny rows, the identity
that a pooled score is the average of the token-level logits of its block pair,
closed forms for the pooling, and the invariants the selection rules imply.
"""
import itertools
import json
import os

import numpy as np
import pytest

from oracle import block_select_ref as bs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "select_small.json")


def _one_hot_case(case):
    A = np.asarray(case["A"], dtype=np.float64)
    D, Hq = case["D"], case["Hq"]
    nb = A.shape[0]
    q = np.zeros((1, 2 * nb, Hq, D))
    k = np.zeros((1, 2 * nb, 1, D))
    for i in range(nb):
        for t, sgn in ((0, 1.0), (1, -1.0)):
            r = 2 * i + t
            q[0, r, 0, i] = 1.0
            q[0, r, 1, i] = -1.0
            q[0, r, :, 7] = sgn
    for j in range(nb):
        for t, sgn in ((0, 1.0), (1, -1.0)):
            r = 2 * j + t
            k[0, r, 0, :nb] = A[:, j]
            k[0, r, 0, 7] = sgn * (j + 1)
    return q, k


def _case_inputs(case):
    if "A" in case:
        return _one_hot_case(case)
    q = np.asarray(case["q"], dtype=np.float64)[None]
    k = np.asarray(case["k"], dtype=np.float64)[None]
    return q, k


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


def golden_maps_hold(mod, case):
    q, k = _case_inputs(case)
    for e in case["expect"]:
        keep, S = mod.block_select(q, k, case["q_offs"], case["k_offs"], e["rule"], case["scale"],
                                   top_k=e.get("k", 0), top_p=e.get("p", 0.0), causal=e["causal"])
        if keep[0].tolist() != e["map"]:
            return False
    if "A" in case:
        A = np.asarray(case["A"], dtype=np.float64)
        if not (np.array_equal(S[0, 0], A) and np.array_equal(S[0, 1], -A)):
            return False
    if "scores" in case and not np.array_equal(S[0, 0], np.asarray(case["scores"], dtype=np.float64)):
        return False
    return True


@pytest.mark.parametrize("case", _golden(), ids=lambda c: c["name"])
def test_golden_maps(case):
    assert golden_maps_hold(bs, case)


def token_mean_holds(mod):
    """<mean q, mean k> = mean over the block pair of <q_r, k_c> (bilinearity):
    the pooled score equals the average token-level logit of its pair."""
    rng = np.random.default_rng(3)
    q = rng.standard_normal((2, 23, 4, 16))
    k = rng.standard_normal((2, 23, 2, 16))
    q_offs = [0, 5, 5, 12, 23]
    k_offs = [0, 7, 8, 23]
    scale = 0.37
    S = mod.block_scores(q, k, q_offs, k_offs, scale)
    for b in range(2):
        for h in range(4):
            logits = scale * q[b, :, h] @ k[b, :, h // 2].T
            for i in range(4):
                for j in range(3):
                    a, c = q_offs[i], q_offs[i + 1]
                    d, e = k_offs[j], k_offs[j + 1]
                    if c == a:
                        if S[b, h, i, j] != 0.0:
                            return False
                    elif not np.isclose(S[b, h, i, j], logits[a:c, d:e].mean(), rtol=1e-12, atol=1e-14):
                        return False
    return True


def test_pooled_score_is_mean_of_token_logits():
    assert token_mean_holds(bs)


def select_pins_hold(mod):
    """Every module-level pin above, for a (possibly mutated) oracle module."""
    return (all(golden_maps_hold(mod, c) for c in _golden()) and token_mean_holds(mod)
            and gqa_mapping_holds(mod) and brute_force_holds(mod) and causal_rule_holds(mod))


def test_block_means_closed_forms():
    # rows x[r] = r: the mean of block [a, b) is (a + b - 1) / 2.
    N = 40
    x = np.broadcast_to(np.arange(N, dtype=np.float64)[None, :, None, None], (1, N, 3, 5)).copy()
    offs = [0, 1, 9, 9, 31, 40]
    m = bs.block_means(x, offs)
    for i in range(5):
        a, b = offs[i], offs[i + 1]
        want = 0.0 if b == a else (a + b - 1) / 2
        assert np.all(m[0, :, i, :] == want)
    # Permuting rows inside a block changes nothing.
    rng = np.random.default_rng(0)
    y = rng.standard_normal((1, N, 2, 4))
    z = y.copy()
    z[0, 9:31] = z[0, 9:31][rng.permutation(22)]
    assert np.allclose(bs.block_means(y, offs), bs.block_means(z, offs), rtol=1e-13, atol=1e-15)


def gqa_mapping_holds(mod):
    """Query head h reads KV head h // (Hq / Hkv)."""
    Hq, Hkv, N, D = 8, 2, 6, 4
    q = np.zeros((1, N, Hq, D))
    q[..., 0] = 1.0
    k = np.zeros((1, N, Hkv, D))
    for g in range(Hkv):
        k[0, :, g, 0] = g + 1.0
    S = mod.block_scores(q, k, [0, 3, 6], [0, 2, 6], 0.5)
    return all(np.all(S[0, h] == 0.5 * (h // (Hq // Hkv) + 1)) for h in range(Hq))


def test_gqa_head_to_group():
    assert gqa_mapping_holds(bs)


def _brute_topk(s, cand, k):
    idx = [j for j in range(len(s)) if cand[j]]
    kk = min(k, len(idx))
    best = max(itertools.combinations(idx, kk), key=lambda c: sum(s[j] for j in c))
    out = np.zeros(len(s), dtype=bool)
    out[list(best)] = True
    return out


def _brute_topp(s, cand, p):
    """Smallest candidate set whose softmax mass reaches p, the largest-mass one
    among those; every candidate when no set reaches p."""
    idx = [j for j in range(len(s)) if cand[j]]
    out = np.zeros(len(s), dtype=bool)
    if not idx:
        return out
    e = np.exp(np.asarray([s[j] for j in idx]) - max(s[j] for j in idx))
    pr = dict(zip(idx, e / e.sum()))
    for n in range(0, len(idx) + 1):
        sets = [c for c in itertools.combinations(idx, n) if sum(pr[j] for j in c) >= p]
        if sets:
            best = max(sets, key=lambda c: sum(pr[j] for j in c))
            out[list(best)] = True
            return out
    out[idx] = True
    return out


def brute_force_holds(mod):
    rng = np.random.default_rng(11)
    for trial in range(300):
        n = int(rng.integers(1, 8))
        s = rng.standard_normal(n) * rng.choice([0.3, 1.0, 4.0])
        cand = rng.random(n) < 0.8
        k = int(rng.integers(0, n + 2))
        p = float(rng.choice([0.0, 0.1, 0.5, 0.8, 0.95, 1.0, 1.2]))
        if not np.array_equal(mod.select_topk_row(s, cand, k), _brute_topk(s, cand, k)):
            return False
        if not np.array_equal(mod.select_topp_row(s, cand, p), _brute_topp(s, cand, p)):
            return False
    return True


def test_topk_topp_match_brute_force():
    assert brute_force_holds(bs)


def causal_rule_holds(mod):
    q_offs = [0, 128, 256, 300, 300, 512]
    k_offs = [0, 100, 256, 256, 257, 512]
    C = mod.candidates(q_offs, k_offs, causal=True)
    Cn = mod.candidates(q_offs, k_offs, causal=False)
    for i in range(5):
        for j in range(5):
            qa, qb = q_offs[i], q_offs[i + 1]
            ka, kb = k_offs[j], k_offs[j + 1]
            # brute force: some key position in block j at or before some query position in block i
            want = any(kk <= qq for qq in range(qa, qb) for kk in range(ka, kb))
            if C[i, j] != want or Cn[i, j] != (qb > qa and kb > ka):
                return False
    return True


def test_candidates_causal_rule():
    assert causal_rule_holds(bs)


def test_selection_invariants():
    rng = np.random.default_rng(5)
    q = rng.standard_normal((1, 96, 4, 8))
    k = rng.standard_normal((1, 96, 2, 8))
    offs = list(range(0, 97, 8))
    n = len(offs) - 1
    C = bs.candidates(offs, offs, True)
    prev = np.zeros((1, 4, n, n), dtype=np.uint8)
    for kk in range(0, n + 2):
        keep, S = bs.block_select(q, k, offs, offs, bs.TOPK, 0.3, top_k=kk, causal=True)
        assert np.all(keep <= C[None, None])                       # only candidates
        assert np.all(prev <= keep)                                # monotone in k
        assert np.array_equal(keep.sum(-1), np.minimum(kk, C.sum(-1))[None, None].repeat(4, 1))
        # a positive rescale of the scores changes no TopK map
        keep2, _ = bs.block_select(q, k, offs, offs, bs.TOPK, 7.0, top_k=kk, causal=True)
        assert np.array_equal(keep, keep2)
        prev = keep
    assert np.array_equal(prev[0, 0], C.astype(np.uint8))
    prev = np.zeros_like(prev)
    for p in (0.0, 0.2, 0.5, 0.9, 0.99, 1.0 + 1e-9):
        keep, S = bs.block_select(q, k, offs, offs, bs.TOPP, 0.3, top_p=p, causal=True)
        assert np.all(prev <= keep)                                # monotone in p
        if p > 0:
            best = np.where(C[None, None], S, -np.inf).argmax(-1)  # the best block is always kept
            assert np.all(np.take_along_axis(keep, best[..., None], -1) == 1)
        prev = keep
    assert np.array_equal(prev[0, 1], C.astype(np.uint8))
