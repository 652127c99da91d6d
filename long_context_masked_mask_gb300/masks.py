"""Mask descriptors for the C ABI, built on the host from a mask spec.

Each of the twelve static mask families of the pages ("Long-Context Attention
Benchmark", xllm-io blog review, section "注意力掩码模式") is turned into the
column-bounds form: for key column j, the allowed query rows are
[a0, b0) U [a1, b1).  This is the column-wise representation the pages credit
to FlashMask (sections "掩码支持" and "关键洞察").  The two dynamic families
(Uniform Block, Variable Block) become a block map with block boundaries.

The builders follow the same readings of the mask names as the oracle but are
written independently of it (the oracle evaluates predicates element by
element; these derive interval end points per key).  All work here is O(N) per
mask; the per-tile and per-element work happens in the CUDA kernels.
"""
from __future__ import annotations

from typing import List, Sequence, Tuple

import numpy as np


def _starts_ends(lens: Sequence[int]) -> Tuple[np.ndarray, np.ndarray]:
    ends = np.cumsum(np.asarray(lens, dtype=np.int64))
    starts = ends - np.asarray(lens, dtype=np.int64)
    return starts, ends


def _per_key(lens: Sequence[int], N: int):
    """(segment index, segment start, segment end) for every key 0..N-1."""
    starts, ends = _starts_ends(lens)
    if ends[-1] != N:
        raise ValueError(f"segment lengths sum to {int(ends[-1])}, expected {N}")
    seg = np.repeat(np.arange(len(lens)), np.asarray(lens, dtype=np.int64))
    return seg, starts[seg], ends[seg]


# Families with a reading for query and key lengths that differ: query i
# stands at key position i + (Sk - Sq) (bottom-right alignment, the decode /
# chunked-prefill convention); the rest are defined for Sq = Sk only.
RECTANGULAR = ("FULL", "CAUSAL", "FULL_SLIDING_WINDOW", "CAUSAL_SLIDING_WINDOW")


def _lengths(spec, N: int, Sk):
    Sk = N if Sk is None else int(Sk)
    if Sk != N and spec.kind not in RECTANGULAR + ("UNIFORM_BLOCK", "VARIABLE_BLOCK"):
        raise ValueError(f"{spec.kind} needs equal query and key lengths")
    return Sk, Sk - N


def col_bounds(spec, N: int, Sk=None) -> np.ndarray:
    """int32 [Sk, 4] = (a0, b0, a1, b1) per key column for a static mask over N
    query rows and Sk keys (default N)."""
    k, p = spec.kind, spec.params
    Sk, off = _lengths(spec, N, Sk)
    j = np.arange(Sk, dtype=np.int64)
    a0 = np.zeros(Sk, np.int64)
    b0 = np.full(Sk, N, np.int64)
    a1 = np.zeros(Sk, np.int64)
    b1 = np.zeros(Sk, np.int64)  # second interval empty unless set
    if k == "FULL":
        pass
    elif k == "CAUSAL":
        a0 = np.maximum(0, j - off)
    elif k == "FULL_DOCUMENT":
        _, a0, b0 = _per_key(p["doc_lens"], N)
    elif k == "CAUSAL_DOCUMENT":
        _, _, b0 = _per_key(p["doc_lens"], N)
        a0 = j.copy()
    elif k == "FULL_SLIDING_WINDOW":
        w = int(p["window"])
        a0 = np.maximum(0, j - w + 1 - off)
        b0 = np.clip(j + w - off, 0, N)
    elif k == "CAUSAL_SLIDING_WINDOW":
        w = int(p["window"])
        a0 = np.maximum(0, j - off)
        b0 = np.clip(j + w - off, 0, N)
    elif k == "SHARED_QUESTION":
        lens = [int(p["question_len"])] + [int(x) for x in p["answer_lens"]]
        seg, _, end = _per_key(lens, N)
        a0 = j.copy()
        b0 = np.where(seg == 0, N, end)  # question keys: every later row of the sample
    elif k == "GLOBAL_SLIDING":
        g, w = int(p["global_tokens"]), int(p["window"])
        glob = j < g
        a0 = np.where(glob, 0, np.maximum(0, j - w + 1))
        b0 = np.where(glob, N, np.minimum(N, j + w))
        a1 = np.zeros(N, np.int64)
        b1 = np.where(glob, 0, min(g, N))  # global query rows see every key
    elif k == "CAUSAL_BLOCKWISE":
        bs = int(p["block"])
        last = (N - 1) // bs
        blk = j // bs
        a0 = j.copy()
        b0 = np.minimum(N, (blk + 1) * bs)
        in_last = blk == last
        b0 = np.where(in_last, N, b0)
        a1 = np.where(in_last, 0, last * bs)
        b1 = np.where(in_last, 0, N)  # the final block's rows see every earlier key
    elif k == "PREFIX_LM_CAUSAL":
        pre = int(p["prefix"])
        a0 = np.where(j < pre, 0, j)
    elif k == "PREFIX_LM_DOCUMENT":
        seg, start, end = _per_key(p["doc_lens"], N)
        pref = np.asarray(p["prefix_lens"], dtype=np.int64)[seg]
        a0 = np.where(j - start < pref, start, j)
        b0 = end
    elif k == "BLOCK_CAUSAL_DOCUMENT":
        _, _, dend = _per_key(p["doc_lens"], N)
        flat = [int(x) for doc in p["block_lens"] for x in doc]
        _, bstart, _ = _per_key(flat, N)
        a0 = bstart  # rows from the key's block start to the end of its document
        b0 = dend
    else:
        raise ValueError(f"{k} is not a column-bounds mask")
    out = np.stack([a0, b0, a1, b1], axis=1)
    return np.ascontiguousarray(out.astype(np.int32))


def row_bounds(spec, N: int, Sk=None) -> np.ndarray:
    """int32 [N, 4] = (c0, d0, c1, d1) per query row: row i may attend the keys
    [c0, d0) U [c1, d1).  The same mask as :func:`col_bounds`, transposed; every
    static family has at most two key intervals per row.  The forward kernel
    uses this form to build a partial tile's row masks cheaply."""
    k, p = spec.kind, spec.params
    Sk, off = _lengths(spec, N, Sk)
    i = np.arange(N, dtype=np.int64)
    c0 = np.zeros(N, np.int64)
    d0 = np.full(N, Sk, np.int64)
    c1 = np.zeros(N, np.int64)
    d1 = np.zeros(N, np.int64)  # second interval empty unless set
    if k == "FULL":
        pass
    elif k == "CAUSAL":
        d0 = np.clip(i + off + 1, 0, Sk)
    elif k == "FULL_DOCUMENT":
        _, c0, d0 = _per_key(p["doc_lens"], N)
    elif k == "CAUSAL_DOCUMENT":
        _, c0, _ = _per_key(p["doc_lens"], N)
        d0 = i + 1
    elif k == "FULL_SLIDING_WINDOW":
        w = int(p["window"])
        c0 = np.maximum(0, i + off - w + 1)
        d0 = np.clip(i + off + w, 0, Sk)
    elif k == "CAUSAL_SLIDING_WINDOW":
        w = int(p["window"])
        c0 = np.maximum(0, i + off - w + 1)
        d0 = np.clip(i + off + 1, 0, Sk)
    elif k == "SHARED_QUESTION":
        q = int(p["question_len"])
        lens = [q] + [int(x) for x in p["answer_lens"]]
        seg, start, _ = _per_key(lens, N)
        # the question's rows: causal over the question; an answer's rows: the
        # whole question, then causal inside their own answer
        c0 = np.where(seg == 0, 0, start)
        d0 = i + 1
        d1 = np.where(seg == 0, 0, min(q, N))
    elif k == "GLOBAL_SLIDING":
        g, w = int(p["global_tokens"]), int(p["window"])
        glob = i < g
        c0 = np.where(glob, 0, np.maximum(0, i - w + 1))
        d0 = np.where(glob, N, np.minimum(N, i + w))
        d1 = np.where(glob, 0, min(g, N))  # every row sees the global keys
    elif k == "CAUSAL_BLOCKWISE":
        bs = int(p["block"])
        last = (N - 1) // bs
        blk = i // bs
        c0 = np.where(blk == last, 0, blk * bs)  # the final block's rows see every earlier key
        d0 = i + 1
    elif k == "PREFIX_LM_CAUSAL":
        pre = min(int(p["prefix"]), N)
        d0 = np.maximum(pre, i + 1)
    elif k == "PREFIX_LM_DOCUMENT":
        seg, start, end = _per_key(p["doc_lens"], N)
        pref = np.minimum(np.asarray(p["prefix_lens"], dtype=np.int64)[seg], end - start)
        c0 = start
        d0 = np.maximum(start + pref, i + 1)
    elif k == "BLOCK_CAUSAL_DOCUMENT":
        _, dstart, _ = _per_key(p["doc_lens"], N)
        flat = [int(x) for doc in p["block_lens"] for x in doc]
        _, _, bend = _per_key(flat, N)
        c0 = dstart  # keys from the row's document start to the end of its block
        d0 = bend
    else:
        raise ValueError(f"{k} is not a column-bounds mask")
    out = np.stack([c0, d0, c1, d1], axis=1)
    return np.ascontiguousarray(out.astype(np.int32))


def block_map(spec, N: int, Hq: int, Sk=None):
    """(keep uint8 [Hq, nQb, nKb], q_offs int32 [nQb+1], k_offs int32 [nKb+1])
    for N query rows and Sk keys (default N)."""
    k, p = spec.kind, spec.params
    Sk = N if Sk is None else int(Sk)
    if k == "UNIFORM_BLOCK":
        bs = int(p["block"])
        nqb, nkb = (N + bs - 1) // bs, (Sk + bs - 1) // bs
        q_offs = np.minimum(np.arange(nqb + 1, dtype=np.int64) * bs, N)
        k_offs = np.minimum(np.arange(nkb + 1, dtype=np.int64) * bs, Sk)
    elif k == "VARIABLE_BLOCK":
        q_offs = np.concatenate([[0], np.cumsum(np.asarray(p["q_block_lens"], np.int64))])
        k_offs = np.concatenate([[0], np.cumsum(np.asarray(p["k_block_lens"], np.int64))])
    else:
        raise ValueError(f"{k} is not a block mask")
    keep = np.asarray(p["keep"], dtype=bool)
    if keep.shape != (Hq, len(q_offs) - 1, len(k_offs) - 1):
        raise ValueError(f"keep map shape {keep.shape} does not match ({Hq}, {len(q_offs)-1}, {len(k_offs)-1})")
    return (np.ascontiguousarray(keep.astype(np.uint8)), q_offs.astype(np.int32),
            k_offs.astype(np.int32))


def allowed_pairs_from_bounds(cb: np.ndarray, Sq: int) -> int:
    """Exact number of allowed (query, key) pairs: the size of the union of the
    two clipped intervals of every column, summed (the metric's unmasked pairs)."""
    cb = cb.astype(np.int64)
    clip = lambda a, b: np.maximum(0, np.minimum(b, Sq) - np.maximum(a, 0))
    a0, b0, a1, b1 = cb[:, 0], cb[:, 1], cb[:, 2], cb[:, 3]
    inter = clip(np.maximum(a0, a1), np.minimum(b0, b1))
    return int((clip(a0, b0) + clip(a1, b1) - inter).sum())


def allowed_pairs_from_blocks(keep: np.ndarray, q_offs: np.ndarray, k_offs: np.ndarray) -> int:
    """Allowed pairs summed over all heads of a block map."""
    ql = np.diff(q_offs.astype(np.int64))
    kl = np.diff(k_offs.astype(np.int64))
    return int(np.einsum("hqk,q,k->", keep.astype(np.int64), ql, kl))
