"""fp64 dynamic block selection: TopK / TopP over pooled Q K^T -> block keep map.

TEST INFRASTRUCTURE (see the package docstring): nothing in the product imports
this module.

What the pages say.  The dynamic masks are block maps, "Uniform Block" (fixed
blocks, e.g. 64x64) and "Variable Block" (xllm-io blog, section
"注意力掩码模式", dynamic masks).  The peer reviews on tomesphere's page for
the paper (section "Peer Reviews", weakness 2) name the step that produces
such a map in practice -- dynamic block-sparse attention whose blocks are chosen
by a TopK or TopP criterion -- and the sparse kernels the blog compares
(section "稀疏注意力内核": VSA, FA2 Sparse, ...) consume a map per head.  No
page writes the criterion out, so this module takes the plainest reading:

  1. pooling: the representative of a block is the mean of its rows, per head
     (q_bar[b, h, i] over query block i, k_bar[b, g, j] over key block j; the
     mean of an empty block is taken as 0);
  2. block score: s[b, h, i, j] = scale * <q_bar[b, h, i], k_bar[b, g(h), j]>,
     g(h) = h // (Hq / Hkv) (contiguous GQA groups, as in the attention);
  3. candidates: both blocks non-empty and, for a causal selection, key block j
     starts before query block i ends (k_offs[j] < q_offs[i + 1]: the pair
     holds at least one key at or before one of the queries);
  4. ranking: candidates by score, largest first; equal scores by smaller key
     block index first;
  5. TopK keeps the first min(k, #candidates) of the ranking;
     TopP turns the candidates' scores into probabilities (softmax over the
     candidates of the row) and keeps a block while the probability ranked
     before it sums to less than p -- the shortest prefix of the ranking whose
     mass reaches p (none for p <= 0, every candidate when p exceeds the mass).

All arithmetic is fp64 on the values given.  The rows of the map are per
(batch, query head, query block), matching the block map the attention
consumes ([B][Hq][nQb][nKb], nonzero = keep).
"""
from __future__ import annotations

import numpy as np

TOPK, TOPP = "topk", "topp"


def block_means(x: np.ndarray, offs) -> np.ndarray:
    """x [B, S, H, D] -> [B, H, nb, D]: mean of rows offs[i] .. offs[i+1]-1 of each
    head (reading 1); 0 for an empty block."""
    offs = np.asarray(offs, dtype=np.int64)
    B, S, H, D = x.shape
    nb = len(offs) - 1
    out = np.zeros((B, H, nb, D), dtype=np.float64)
    for i in range(nb):
        lo, hi = int(offs[i]), int(offs[i + 1])
        if hi > lo:
            out[:, :, i, :] = x[:, lo:hi, :, :].astype(np.float64).mean(axis=1)
    return out


def block_scores(q: np.ndarray, k: np.ndarray, q_offs, k_offs, scale: float) -> np.ndarray:
    """[B, Hq, nQb, nKb] pooled scores (reading 2) for q [B, Sq, Hq, D], k [B, Sk, Hkv, D]."""
    qb = block_means(q, q_offs)
    kb = block_means(k, k_offs)
    Hq, Hkv = q.shape[2], k.shape[2]
    G = Hq // Hkv
    out = np.empty((q.shape[0], Hq, qb.shape[2], kb.shape[2]), dtype=np.float64)
    for h in range(Hq):
        out[:, h] = scale * np.einsum("bid,bjd->bij", qb[:, h], kb[:, h // G])
    return out


def candidates(q_offs, k_offs, causal: bool) -> np.ndarray:
    """[nQb, nKb] bool (reading 3)."""
    q_offs = np.asarray(q_offs, dtype=np.int64)
    k_offs = np.asarray(k_offs, dtype=np.int64)
    q_nonempty = q_offs[1:] > q_offs[:-1]
    k_nonempty = k_offs[1:] > k_offs[:-1]
    c = q_nonempty[:, None] & k_nonempty[None, :]
    if causal:
        c &= k_offs[:-1][None, :] < q_offs[1:][:, None]
    return c


def ranking(scores_row: np.ndarray, cand_row: np.ndarray) -> np.ndarray:
    """Candidate key-block indices, best first (reading 4)."""
    idx = np.nonzero(cand_row)[0]
    s = scores_row[idx]
    # lexsort sorts by the last key first: score descending, then index ascending.
    return idx[np.lexsort((idx, -s))]


def select_topk_row(scores_row, cand_row, k: int) -> np.ndarray:
    keep = np.zeros(len(cand_row), dtype=bool)
    keep[ranking(scores_row, cand_row)[:max(int(k), 0)]] = True
    return keep


def select_topp_row(scores_row, cand_row, p: float) -> np.ndarray:
    keep = np.zeros(len(cand_row), dtype=bool)
    order = ranking(scores_row, cand_row)
    if len(order) == 0:
        return keep
    s = scores_row[order]
    e = np.exp(s - s.max())
    prob = e / e.sum()
    mass_before = np.concatenate([[0.0], np.cumsum(prob)[:-1]])
    keep[order[mass_before < p]] = True
    return keep


def block_select(q: np.ndarray, k: np.ndarray, q_offs, k_offs, rule: str, scale: float,
                 top_k: int = 0, top_p: float = 0.0, causal: bool = False):
    """Block keep map [B, Hq, nQb, nKb] (uint8, 1 = keep) and the pooled scores."""
    S = block_scores(q, k, q_offs, k_offs, scale)
    C = candidates(q_offs, k_offs, causal)
    B, Hq, nQb, nKb = S.shape
    keep = np.zeros(S.shape, dtype=np.uint8)
    for b in range(B):
        for h in range(Hq):
            for i in range(nQb):
                if rule == TOPK:
                    row = select_topk_row(S[b, h, i], C[i], top_k)
                elif rule == TOPP:
                    row = select_topp_row(S[b, h, i], C[i], top_p)
                else:
                    raise ValueError(rule)
                keep[b, h, i] = row
    return keep, S
