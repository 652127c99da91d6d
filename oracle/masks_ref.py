"""Explicit boolean masks, straight from each mask family's predicate.

TEST INFRASTRUCTURE (see the package docstring): nothing in the product imports
this module.

The pages list the fourteen families with a one-line purpose each and no
formula (xllm-io blog, section "注意力掩码模式": regular masks FULL, CAUSAL,
FULL/CAUSAL DOCUMENT, FULL/CAUSAL SLIDING WINDOW; heterogeneous masks SHARED
QUESTION, GLOBAL SLIDING, CAUSAL BLOCKWISE, PREFIX LM CAUSAL, PREFIX LM
DOCUMENT, BLOCK CAUSAL DOCUMENT; dynamic masks Uniform Block "e.g. 64x64" and
Variable Block).  Each predicate below is the plainest reading of the name;
i is the query index and j the key index, both 0-based, and a pair is allowed
when the predicate is true:

    FULL                    true
    CAUSAL                  j <= i
    FULL_DOCUMENT           doc(i) == doc(j)
    CAUSAL_DOCUMENT         doc(i) == doc(j) and j <= i
    FULL_SLIDING_WINDOW     |i - j| < w           (w counts the token itself)
    CAUSAL_SLIDING_WINDOW   0 <= i - j < w
    SHARED_QUESTION         j <= i and (seg(j) is the question or seg(j) == seg(i))
    GLOBAL_SLIDING          i < g or j < g or |i - j| < w      (non-causal)
    CAUSAL_BLOCKWISE        j <= i and (blk(i) == blk(j) or blk(i) is the last block)
    PREFIX_LM_CAUSAL        j < p or j <= i
    PREFIX_LM_DOCUMENT      doc(i) == doc(j) and (j - start(doc(j)) < p_doc or j <= i)
    BLOCK_CAUSAL_DOCUMENT   doc(i) == doc(j) and blk(j) <= blk(i)
    UNIFORM_BLOCK           keep[h, i // bs, j // bs]
    VARIABLE_BLOCK          keep[h, qblk(i), kblk(j)]

Query and key lengths may differ (Sq queries, Sk keys) for FULL, CAUSAL and the
two sliding windows, the variants the pages' kernels take for decode-style and
chunked rows.  The reading is bottom-right alignment: query i stands at key
position i + (Sk - Sq), and the predicates above apply with that position in
place of i (so CAUSAL is j <= i + Sk - Sq; for Sq > Sk the first Sq - Sk rows
allow nothing).  With Sq = Sk the shift is 0.  Block maps index query and key
blocks on their own axes, with no shift.  The other families are defined for
Sq = Sk only.
"""
from __future__ import annotations

import numpy as np


def _segment_of(idx: np.ndarray, lens) -> np.ndarray:
    """Index of the segment (from consecutive lengths) that holds each position."""
    ends = np.cumsum(np.asarray(lens, dtype=np.int64))
    return np.searchsorted(ends, idx, side="right")


def _segment_start(seg: np.ndarray, lens) -> np.ndarray:
    starts = np.concatenate([[0], np.cumsum(np.asarray(lens, dtype=np.int64))[:-1]])
    return starts[seg]


RECTANGULAR = ("FULL", "CAUSAL", "FULL_SLIDING_WINDOW", "CAUSAL_SLIDING_WINDOW",
               "UNIFORM_BLOCK", "VARIABLE_BLOCK")


def allowed(spec, N: int, rows=None, head: int = 0, cols=None, Sk=None) -> np.ndarray:
    """Boolean mask rows: ``out[r, c]`` is True when query ``rows[r]`` may attend
    key ``cols[c]`` under ``spec`` for query head ``head``.  ``N`` is the number
    of queries and ``Sk`` of keys (default ``N``); ``cols`` defaults to every key."""
    Sk = N if Sk is None else int(Sk)
    if rows is None:
        rows = np.arange(N)
    i = np.asarray(rows, dtype=np.int64)[:, None]
    j = (np.arange(Sk, dtype=np.int64) if cols is None else np.asarray(cols, dtype=np.int64))[None, :]
    k = spec.kind
    p = spec.params
    if Sk != N and k not in RECTANGULAR:
        raise ValueError(f"{k} is defined for equal query and key lengths only")
    if k == "UNIFORM_BLOCK":
        bs = p["block"]
        keep = np.asarray(p["keep"], dtype=bool)[head]
        return keep[i // bs, j // bs]
    if k == "VARIABLE_BLOCK":
        keep = np.asarray(p["keep"], dtype=bool)[head]
        return keep[_segment_of(i, p["q_block_lens"]), _segment_of(j, p["k_block_lens"])]
    i = i + (Sk - N)  # the query's position on the key axis (bottom-right alignment)
    if k == "FULL":
        return np.ones((i.shape[0], j.shape[1]), dtype=bool)
    if k == "CAUSAL":
        return j <= i
    if k in ("FULL_DOCUMENT", "CAUSAL_DOCUMENT"):
        same = _segment_of(i, p["doc_lens"]) == _segment_of(j, p["doc_lens"])
        return same & (j <= i) if k == "CAUSAL_DOCUMENT" else same
    if k == "FULL_SLIDING_WINDOW":
        return np.abs(i - j) < p["window"]
    if k == "CAUSAL_SLIDING_WINDOW":
        d = i - j
        return (d >= 0) & (d < p["window"])
    if k == "SHARED_QUESTION":
        lens = [p["question_len"]] + list(p["answer_lens"])
        si, sj = _segment_of(i, lens), _segment_of(j, lens)
        return (j <= i) & ((sj == 0) | (sj == si))
    if k == "GLOBAL_SLIDING":
        g, w = p["global_tokens"], p["window"]
        return (i < g) | (j < g) | (np.abs(i - j) < w)
    if k == "CAUSAL_BLOCKWISE":
        bs = p["block"]
        last = (N - 1) // bs
        bi, bj = i // bs, j // bs
        return (j <= i) & ((bi == bj) | (bi == last))
    if k == "PREFIX_LM_CAUSAL":
        return (j < p["prefix"]) | (j <= i)
    if k == "PREFIX_LM_DOCUMENT":
        lens = p["doc_lens"]
        di, dj = _segment_of(i, lens), _segment_of(j, lens)
        pref = np.asarray(p["prefix_lens"], dtype=np.int64)[dj]
        in_prefix = (j - _segment_start(dj, lens)) < pref
        return (di == dj) & (in_prefix | (j <= i))
    if k == "BLOCK_CAUSAL_DOCUMENT":
        lens = p["doc_lens"]
        flat_blocks = [b for doc in p["block_lens"] for b in doc]
        di, dj = _segment_of(i, lens), _segment_of(j, lens)
        bi, bj = _segment_of(i, flat_blocks), _segment_of(j, flat_blocks)
        return (di == dj) & (bj <= bi)
    raise ValueError(k)


def allowed_pairs(spec, N: int, head: int = 0, chunk: int = 4096, Sk=None) -> int:
    """Number of allowed (i, j) pairs for one head, by explicit enumeration."""
    total = 0
    for r0 in range(0, N, chunk):
        total += int(allowed(spec, N, np.arange(r0, min(N, r0 + chunk)), head, Sk=Sk).sum())
    return total
