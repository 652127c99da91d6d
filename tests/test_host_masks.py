"""Host-side mask descriptors (product) against the oracle's predicates (CPU only).

The column-bounds, row-bounds and block-map builders of ``long_context_masked_mask_gb300.masks``
are expanded back to boolean masks here and compared element by element with
``oracle.allowed``, which evaluates each family's predicate directly.  The
allowed-pair counts used by the FLOP metric are checked the same way.
"""
import numpy as np
import pytest

from oracle import allowed, allowed_pairs
from synthetic import MaskSpec, block_keep, doc_lengths_lognormal, segment_lengths

masks = pytest.importorskip("long_context_masked_mask_gb300.masks")


def expand_bounds(cb, N):
    i = np.arange(N)[:, None]
    a0, b0, a1, b1 = (cb[:, k][None, :] for k in range(4))
    return ((a0 <= i) & (i < b0)) | ((a1 <= i) & (i < b1))


def expand_blocks(keep, q_offs, k_offs, h):
    ql = np.diff(q_offs)
    kl = np.diff(k_offs)
    return np.repeat(np.repeat(keep[h].astype(bool), ql, axis=0), kl, axis=1)


def static_specs(N, seed):
    rng = np.random.default_rng(seed)
    docs = segment_lengths(N, max(1, N // 8), max(2, N // 3), seed)
    blocks = [segment_lengths(L, 1, max(1, L // 2), seed + 7 + i) for i, L in enumerate(docs)]
    q = int(rng.integers(1, N // 2))
    rest = N - q
    answers = segment_lengths(rest, 1, max(1, rest // 2), seed + 3)
    return [
        MaskSpec("FULL"), MaskSpec("CAUSAL"),
        MaskSpec("FULL_DOCUMENT", {"doc_lens": docs}),
        MaskSpec("CAUSAL_DOCUMENT", {"doc_lens": docs}),
        MaskSpec("FULL_SLIDING_WINDOW", {"window": int(rng.integers(1, N + 3))}),
        MaskSpec("CAUSAL_SLIDING_WINDOW", {"window": int(rng.integers(1, N + 3))}),
        MaskSpec("SHARED_QUESTION", {"question_len": q, "answer_lens": answers}),
        MaskSpec("GLOBAL_SLIDING", {"global_tokens": int(rng.integers(0, N // 3)),
                                    "window": int(rng.integers(1, N // 2))}),
        MaskSpec("CAUSAL_BLOCKWISE", {"block": int(rng.integers(1, N + 2))}),
        MaskSpec("PREFIX_LM_CAUSAL", {"prefix": int(rng.integers(0, N + 1))}),
        MaskSpec("PREFIX_LM_DOCUMENT", {"doc_lens": docs,
                                        "prefix_lens": [int(rng.integers(0, L + 1)) for L in docs]}),
        MaskSpec("BLOCK_CAUSAL_DOCUMENT", {"doc_lens": docs, "block_lens": blocks}),
    ]


@pytest.mark.parametrize("N,seed", [(6, 0), (9, 1), (64, 2), (130, 3), (257, 4)])
def test_col_bounds_match_predicates(N, seed):
    for spec in static_specs(N, seed):
        cb = masks.col_bounds(spec, N)
        assert cb.dtype == np.int32 and cb.shape == (N, 4)
        np.testing.assert_array_equal(expand_bounds(cb, N), allowed(spec, N), err_msg=spec.kind)
        assert masks.allowed_pairs_from_bounds(cb, N) == allowed_pairs(spec, N), spec.kind


def expand_rows(rb, N):
    j = np.arange(N)[None, :]
    c0, d0, c1, d1 = (rb[:, k][:, None] for k in range(4))
    return ((c0 <= j) & (j < d0)) | ((c1 <= j) & (j < d1))


@pytest.mark.parametrize("N,seed", [(6, 0), (9, 1), (64, 2), (130, 3), (257, 4), (1000, 5)])
def test_row_bounds_match_predicates(N, seed):
    """The per-row form (key intervals of each query row) is the same mask."""
    for spec in static_specs(N, seed):
        rb = masks.row_bounds(spec, N)
        assert rb.dtype == np.int32 and rb.shape == (N, 4)
        np.testing.assert_array_equal(expand_rows(rb, N), allowed(spec, N), err_msg=spec.kind)


def test_single_token_sequence():
    for spec in (MaskSpec("FULL"), MaskSpec("CAUSAL"), MaskSpec("CAUSAL_SLIDING_WINDOW", {"window": 4})):
        cb = masks.col_bounds(spec, 1)
        np.testing.assert_array_equal(expand_bounds(cb, 1), allowed(spec, 1))


def test_config_masks_match_predicates():
    N = 16384
    specs = [
        MaskSpec("CAUSAL_SLIDING_WINDOW", {"window": 2048}),
        MaskSpec("GLOBAL_SLIDING", {"global_tokens": 256, "window": 1024}),
        MaskSpec("PREFIX_LM_CAUSAL", {"prefix": 4096}),
        MaskSpec("SHARED_QUESTION", {"question_len": 2048, "answer_lens": [3584] * 4}),
        MaskSpec("CAUSAL_BLOCKWISE", {"block": 1024}),
        MaskSpec("CAUSAL_DOCUMENT", {"doc_lens": doc_lengths_lognormal(N, seed=0)}),
    ]
    rows = np.r_[0:40, 2000:2100, 4090:4100, 16300:16384]
    for spec in specs:
        cb = masks.col_bounds(spec, N)
        i = rows[:, None]
        a0, b0, a1, b1 = (cb[:, k][None, :] for k in range(4))
        got = ((a0 <= i) & (i < b0)) | ((a1 <= i) & (i < b1))
        np.testing.assert_array_equal(got, allowed(spec, N, rows), err_msg=spec.kind)
        rb = masks.row_bounds(spec, N)[rows]
        np.testing.assert_array_equal(expand_rows(rb, N), allowed(spec, N, rows), err_msg=spec.kind)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_block_maps_match_predicates(seed):
    N, Hq = 203, 3
    bs = [16, 64, 128][seed]
    nb = -(-N // bs)
    spec = MaskSpec("UNIFORM_BLOCK", {"block": bs, "keep": block_keep(Hq, nb, nb, 0.5, seed)})
    keep, qo, ko = masks.block_map(spec, N, Hq)
    for h in range(Hq):
        np.testing.assert_array_equal(expand_blocks(keep, qo, ko, h), allowed(spec, N, head=h))
    assert masks.allowed_pairs_from_blocks(keep, qo, ko) == sum(allowed_pairs(spec, N, h) for h in range(Hq))
    ql = segment_lengths(N, 1, 70, seed + 10)
    kl = segment_lengths(N, 1, 90, seed + 20)
    spec = MaskSpec("VARIABLE_BLOCK", {"q_block_lens": ql, "k_block_lens": kl,
                                       "keep": block_keep(Hq, len(ql), len(kl), 0.4, seed)})
    keep, qo, ko = masks.block_map(spec, N, Hq)
    for h in range(Hq):
        np.testing.assert_array_equal(expand_blocks(keep, qo, ko, h), allowed(spec, N, head=h))


def test_builders_reject_bad_lengths():
    with pytest.raises(ValueError):
        masks.col_bounds(MaskSpec("FULL_DOCUMENT", {"doc_lens": [3, 4]}), 8)
    with pytest.raises(ValueError):
        masks.col_bounds(MaskSpec("UNIFORM_BLOCK", {"block": 4, "keep": np.ones((1, 2, 2))}), 8)


@pytest.mark.parametrize("Sq,Sk", [(1, 9), (5, 130), (130, 5), (3, 3), (64, 257), (200, 64)])
def test_rectangular_bounds_match_predicates(Sq, Sk):
    """Query and key lengths that differ (bottom-right alignment): column and
    row bounds of FULL, CAUSAL and the sliding windows against the oracle's
    predicates, and block maps with separate query and key blocks."""
    rng = np.random.default_rng(Sq * 1000 + Sk)
    specs = [MaskSpec("FULL"), MaskSpec("CAUSAL")]
    for w in (1, 2, int(rng.integers(1, Sk + 3)), Sk + Sq):
        specs += [MaskSpec("FULL_SLIDING_WINDOW", {"window": w}),
                  MaskSpec("CAUSAL_SLIDING_WINDOW", {"window": w})]
    for spec in specs:
        want = allowed(spec, Sq, Sk=Sk)
        cb = masks.col_bounds(spec, Sq, Sk)
        assert cb.shape == (Sk, 4)
        np.testing.assert_array_equal(expand_bounds(cb, Sq), want, err_msg=spec.label())
        assert masks.allowed_pairs_from_bounds(cb, Sq) == int(want.sum())
        rb = masks.row_bounds(spec, Sq, Sk)
        assert rb.shape == (Sq, 4)
        np.testing.assert_array_equal(expand_rows(rb, Sk), want, err_msg=spec.label())
    bs = 16
    keep = rng.random((2, -(-Sq // bs), -(-Sk // bs))) < 0.5
    spec = MaskSpec("UNIFORM_BLOCK", {"block": bs, "keep": keep})
    kp, qo, ko = masks.block_map(spec, Sq, 2, Sk)
    assert qo[-1] == Sq and ko[-1] == Sk
    for h in range(2):
        ql, kl = np.diff(qo), np.diff(ko)
        dense = np.repeat(np.repeat(kp[h].astype(bool), ql, 0), kl, 1)
        np.testing.assert_array_equal(dense, allowed(spec, Sq, head=h, Sk=Sk))


def test_rectangular_rejected_where_undefined():
    with pytest.raises(ValueError):
        masks.col_bounds(MaskSpec("PREFIX_LM_CAUSAL", {"prefix": 2}), 4, 6)
