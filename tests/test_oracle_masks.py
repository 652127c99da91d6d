"""Pins for the oracle's mask predicates and tile classifier (CPU only).

Each mask predicate is checked against hand-derived small masks
(tests/golden/masks_small.json) and against the relations between families that
follow from the mask names on the pages ("Long-Context Attention Benchmark",
xllm-io blog review, section 注意力掩码模式).  The tile classifier is checked
against hand-derived classes and against a per-element scan.
"""
import json
import os

import numpy as np
import pytest

from oracle import allowed, classify_tiles, EMPTY, FULL, PARTIAL
from synthetic import MaskSpec, block_keep, doc_lengths_lognormal, segment_lengths

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


@pytest.mark.parametrize("case", _golden("masks_small.json")["cases"], ids=lambda c: c["name"])
def test_mask_golden(case):
    spec = MaskSpec(case["kind"], dict(case["params"]))
    if "keep" in spec.params:
        spec.params["keep"] = np.array(spec.params["keep"], dtype=bool)
    want = np.array([[c == "1" for c in row] for row in case["rows"]], dtype=bool)
    got = allowed(spec, case["N"], Sk=case.get("Sk"))
    np.testing.assert_array_equal(got, want)


def _full(N):
    return allowed(MaskSpec("FULL"), N)


def _causal(N):
    return allowed(MaskSpec("CAUSAL"), N)


@pytest.mark.parametrize("N", [1, 7, 33])
def test_document_single_doc_is_full_or_causal(N):
    np.testing.assert_array_equal(allowed(MaskSpec("FULL_DOCUMENT", {"doc_lens": [N]}), N), _full(N))
    np.testing.assert_array_equal(allowed(MaskSpec("CAUSAL_DOCUMENT", {"doc_lens": [N]}), N), _causal(N))


@pytest.mark.parametrize("N,w", [(9, 9), (9, 20), (16, 16)])
def test_window_covering_sequence(N, w):
    np.testing.assert_array_equal(allowed(MaskSpec("FULL_SLIDING_WINDOW", {"window": w}), N), _full(N))
    np.testing.assert_array_equal(allowed(MaskSpec("CAUSAL_SLIDING_WINDOW", {"window": w}), N), _causal(N))


@pytest.mark.parametrize("N,w", [(13, 1), (13, 4), (40, 7)])
def test_csw_is_fsw_and_causal(N, w):
    fsw = allowed(MaskSpec("FULL_SLIDING_WINDOW", {"window": w}), N)
    csw = allowed(MaskSpec("CAUSAL_SLIDING_WINDOW", {"window": w}), N)
    np.testing.assert_array_equal(csw, fsw & _causal(N))
    # each row of CSW holds min(i+1, w) keys
    np.testing.assert_array_equal(csw.sum(1), np.minimum(np.arange(N) + 1, w))


def test_prefix_zero_is_causal_and_full_prefix_is_full():
    N = 17
    np.testing.assert_array_equal(allowed(MaskSpec("PREFIX_LM_CAUSAL", {"prefix": 0}), N), _causal(N))
    np.testing.assert_array_equal(allowed(MaskSpec("PREFIX_LM_CAUSAL", {"prefix": N}), N), _full(N))


def test_blockwise_single_block_is_causal():
    N = 19
    np.testing.assert_array_equal(allowed(MaskSpec("CAUSAL_BLOCKWISE", {"block": N}), N), _causal(N))
    np.testing.assert_array_equal(allowed(MaskSpec("CAUSAL_BLOCKWISE", {"block": 100}), N), _causal(N))


def test_shared_question_one_answer_is_causal():
    N = 21
    spec = MaskSpec("SHARED_QUESTION", {"question_len": 5, "answer_lens": [16]})
    np.testing.assert_array_equal(allowed(spec, N), _causal(N))


def test_shared_question_answers_do_not_see_each_other():
    spec = MaskSpec("SHARED_QUESTION", {"question_len": 4, "answer_lens": [3, 5, 2]})
    M = allowed(spec, 14)
    # answer 2 (rows 7..11) never sees answer 1 (keys 4..6)
    assert not M[7:12, 4:7].any()
    # every answer row sees the whole question
    assert M[4:, :4].all()


def test_global_sliding_zero_globals_is_fsw():
    N, w = 23, 3
    np.testing.assert_array_equal(
        allowed(MaskSpec("GLOBAL_SLIDING", {"global_tokens": 0, "window": w}), N),
        allowed(MaskSpec("FULL_SLIDING_WINDOW", {"window": w}), N))


def test_prefix_document_reductions():
    lens = [5, 9, 3]
    N = sum(lens)
    cd = allowed(MaskSpec("CAUSAL_DOCUMENT", {"doc_lens": lens}), N)
    fd = allowed(MaskSpec("FULL_DOCUMENT", {"doc_lens": lens}), N)
    np.testing.assert_array_equal(
        allowed(MaskSpec("PREFIX_LM_DOCUMENT", {"doc_lens": lens, "prefix_lens": [0, 0, 0]}), N), cd)
    np.testing.assert_array_equal(
        allowed(MaskSpec("PREFIX_LM_DOCUMENT", {"doc_lens": lens, "prefix_lens": lens}), N), fd)


def test_block_causal_document_reductions():
    lens = [6, 4, 7]
    N = sum(lens)
    # one token per block = causal document; one block per document = full document
    ones = [[1] * L for L in lens]
    np.testing.assert_array_equal(
        allowed(MaskSpec("BLOCK_CAUSAL_DOCUMENT", {"doc_lens": lens, "block_lens": ones}), N),
        allowed(MaskSpec("CAUSAL_DOCUMENT", {"doc_lens": lens}), N))
    whole = [[L] for L in lens]
    np.testing.assert_array_equal(
        allowed(MaskSpec("BLOCK_CAUSAL_DOCUMENT", {"doc_lens": lens, "block_lens": whole}), N),
        allowed(MaskSpec("FULL_DOCUMENT", {"doc_lens": lens}), N))


def test_block_maps_all_ones_is_full_and_uniform_equals_variable():
    N, bs = 21, 4
    nb = (N + bs - 1) // bs
    keep = block_keep(3, nb, nb, p=0.5, seed=3)
    ones = np.ones_like(keep)
    np.testing.assert_array_equal(allowed(MaskSpec("UNIFORM_BLOCK", {"block": bs, "keep": ones}), N, head=1), _full(N))
    lens = [bs] * (N // bs) + [N % bs]
    for h in range(3):
        np.testing.assert_array_equal(
            allowed(MaskSpec("UNIFORM_BLOCK", {"block": bs, "keep": keep}), N, head=h),
            allowed(MaskSpec("VARIABLE_BLOCK", {"q_block_lens": lens, "k_block_lens": lens, "keep": keep}), N, head=h))


def test_every_named_mask_allows_the_diagonal():
    """No family on the pages leaves a query with no key: the diagonal is always allowed."""
    N = 64
    docs = [10, 30, 24]
    specs = [
        MaskSpec("FULL"), MaskSpec("CAUSAL"),
        MaskSpec("FULL_DOCUMENT", {"doc_lens": docs}), MaskSpec("CAUSAL_DOCUMENT", {"doc_lens": docs}),
        MaskSpec("FULL_SLIDING_WINDOW", {"window": 5}), MaskSpec("CAUSAL_SLIDING_WINDOW", {"window": 5}),
        MaskSpec("SHARED_QUESTION", {"question_len": 16, "answer_lens": [16, 16, 16]}),
        MaskSpec("GLOBAL_SLIDING", {"global_tokens": 4, "window": 6}),
        MaskSpec("CAUSAL_BLOCKWISE", {"block": 16}),
        MaskSpec("PREFIX_LM_CAUSAL", {"prefix": 20}),
        MaskSpec("PREFIX_LM_DOCUMENT", {"doc_lens": docs, "prefix_lens": [5, 15, 12]}),
        MaskSpec("BLOCK_CAUSAL_DOCUMENT", {"doc_lens": docs, "block_lens": [[4, 6], [10, 20], [24]]}),
        MaskSpec("UNIFORM_BLOCK", {"block": 8, "keep": block_keep(2, 8, 8, 0.5, 1)}),
    ]
    for s in specs:
        assert np.diag(allowed(s, N)).all(), s.kind


def test_doc_lengths_recipe():
    lens = doc_lengths_lognormal(32768, seed=0)
    assert sum(lens) == 32768
    assert all(256 <= x <= 16384 for x in lens[:-1])
    segs = segment_lengths(1000, 32, 512, seed=5)
    assert sum(segs) == 1000 and all(1 <= x <= 512 for x in segs)


# ----------------------------------------------------------------------------
# Tile classifier
# ----------------------------------------------------------------------------

_CODE = {"E": EMPTY, "F": FULL, "P": PARTIAL}


@pytest.mark.parametrize("case", _golden("tiles_small.json")["cases"], ids=lambda c: c["kind"])
def test_classify_golden(case):
    spec = MaskSpec(case["kind"], dict(case["params"]))
    want = np.array([[_CODE[c] for c in row] for row in case["classes"]], dtype=np.uint8)
    got = classify_tiles(spec, case["N"], case["BM"], case["BN"])
    np.testing.assert_array_equal(got, want)


def _scan_classes(M, BM, BN):
    """Per-element scan: count allowed pairs in each tile and compare with its size."""
    N = M.shape[0]
    nq, nk = -(-N // BM), -(-N // BN)
    out = np.zeros((nq, nk), dtype=np.uint8)
    for a in range(nq):
        for c in range(nk):
            cnt = size = 0
            for i in range(a * BM, min(N, (a + 1) * BM)):
                for j in range(c * BN, min(N, (c + 1) * BN)):
                    size += 1
                    cnt += int(M[i, j])
            out[a, c] = EMPTY if cnt == 0 else (FULL if cnt == size else PARTIAL)
    return out


@pytest.mark.parametrize("spec", [
    MaskSpec("CAUSAL"),
    MaskSpec("CAUSAL_DOCUMENT", {"doc_lens": [9, 14, 20]}),
    MaskSpec("GLOBAL_SLIDING", {"global_tokens": 3, "window": 5}),
    MaskSpec("SHARED_QUESTION", {"question_len": 11, "answer_lens": [10, 11, 11]}),
], ids=lambda s: s.kind)
def test_classify_matches_scan(spec):
    N, BM, BN = 43, 8, 8
    M = allowed(spec, N)
    np.testing.assert_array_equal(classify_tiles(spec, N, BM, BN), _scan_classes(M, BM, BN))
