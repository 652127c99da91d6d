"""fp64 masked attention, forward and backward, and the tile classifier.

TEST INFRASTRUCTURE (see the package docstring): nothing in the product imports
this module.

Definition (the textbook operator that every kernel on the pages computes --
"Long-Context Attention Benchmark", xllm-io blog, sections "密集注意力内核" and
"稀疏注意力内核"; the pages give no formula).  For batch b and query head h with
KV head g = h // (Hq / Hkv) (contiguous GQA groups), with M the boolean mask
from ``masks_ref.allowed`` and s the softmax scale:

    S_ij   = s * <q_i, k_j>
    LSE_i  = log sum_j M_ij exp(S_ij)           (-inf when row i allows nothing)
    P_ij   = M_ij exp(S_ij - LSE_i)             (0 when row i allows nothing)
    O_i    = sum_j P_ij v_j

Backward of L = sum <O, dO>:

    dV_j   = sum_{h in group} sum_i P_ij dO_i
    dP_ij  = <dO_i, v_j>
    D_i    = <dO_i, O_i>
    dS_ij  = P_ij (dP_ij - D_i)
    dQ_i   = s * sum_j dS_ij k_j
    dK_j   = s * sum_{h in group} sum_i dS_ij q_i

All arithmetic is fp64 on the values given (bf16 inputs are upcast exactly by
the caller).  Rows are processed in chunks only to bound memory; nothing is
reordered beyond that.
"""
from __future__ import annotations

import numpy as np

from .masks_ref import allowed

EMPTY, FULL, PARTIAL = 0, 1, 2


def _rows_fwd(qr, k, v, M, scale):
    """Forward for a block of query rows of one head: qr [R, D], k/v [N, D], M [R, N]."""
    S = scale * (qr @ k.T)
    Sm = np.where(M, S, -np.inf)
    m = Sm.max(axis=1)
    has = np.isfinite(m)
    m_safe = np.where(has, m, 0.0)
    E = np.where(M, np.exp(Sm - m_safe[:, None]), 0.0)
    l = E.sum(axis=1)
    lse = np.where(has, m_safe + np.log(np.where(has, l, 1.0)), -np.inf)
    P = E / np.where(has, l, 1.0)[:, None]
    O = P @ v
    return O, lse, P


def attention_fwd(q, k, v, spec, scale, chunk: int = 1024):
    """O [B, N, Hq, D] and LSE [B, Hq, N] for fp64 arrays q [B,N,Hq,D], k/v [B,Sk,Hkv,D]."""
    B, N, Hq, D = q.shape
    Sk = k.shape[1]
    Hkv = k.shape[2]
    G = Hq // Hkv
    O = np.zeros((B, N, Hq, v.shape[3]), dtype=np.float64)
    LSE = np.zeros((B, Hq, N), dtype=np.float64)
    for b in range(B):
        for h in range(Hq):
            g = h // G
            for r0 in range(0, N, chunk):
                rows = np.arange(r0, min(N, r0 + chunk))
                M = allowed(spec, N, rows, head=h, Sk=Sk)
                o, lse, _ = _rows_fwd(q[b, rows, h], k[b, :, g], v[b, :, g], M, scale)
                O[b, rows, h] = o
                LSE[b, h, rows] = lse
    return O, LSE


def attention_fwd_rows(q, k, v, spec, scale, b: int, h: int, rows):
    """O [R, D] and LSE [R] for selected query rows of one (batch, head)."""
    N, Sk = q.shape[1], k.shape[1]
    G = q.shape[2] // k.shape[2]
    rows = np.asarray(rows, dtype=np.int64)
    M = allowed(spec, N, rows, head=h, Sk=Sk)
    o, lse, _ = _rows_fwd(q[b, rows, h], k[b, :, h // G], v[b, :, h // G], M, scale)
    return o, lse


def attention_bwd(q, k, v, do, spec, scale, chunk: int = 1024):
    """(dQ, dK, dV, O, LSE) for the whole problem, from the definition above."""
    B, N, Hq, D = q.shape
    Sk = k.shape[1]
    Hkv = k.shape[2]
    G = Hq // Hkv
    O, LSE = attention_fwd(q, k, v, spec, scale, chunk)
    dQ = np.zeros_like(q)
    dK = np.zeros_like(k)
    dV = np.zeros_like(v)
    for b in range(B):
        for h in range(Hq):
            g = h // G
            kk, vv = k[b, :, g], v[b, :, g]
            for r0 in range(0, N, chunk):
                rows = np.arange(r0, min(N, r0 + chunk))
                M = allowed(spec, N, rows, head=h, Sk=Sk)
                lse = LSE[b, h, rows]
                has = np.isfinite(lse)
                S = scale * (q[b, rows, h] @ kk.T)
                P = np.where(M & has[:, None], np.exp(S - np.where(has, lse, 0.0)[:, None]), 0.0)
                dOr = do[b, rows, h]
                dV[b, :, g] += P.T @ dOr
                dP = dOr @ vv.T
                Dr = (dOr * O[b, rows, h]).sum(axis=1)
                dS = P * (dP - Dr[:, None])
                dQ[b, rows, h] = scale * (dS @ kk)
                dK[b, :, g] += scale * (dS.T @ q[b, rows, h])
    return dQ, dK, dV, O, LSE


def attention_bwd_rows(q, k, v, do, spec, scale, b: int, h: int, rows):
    """The backward restricted to selected query rows of one (batch, query head h):

    * O [R, D], LSE [R] and dQ [R, D] of those rows;
    * dK, dV [Sk, D]: the terms of dK_j = s * sum_i dS_ij q_i and
      dV_j = sum_i P_ij dO_i that come from those rows (for head h only).

    The same formulas as :func:`attention_bwd`, applied to the rows given; over a
    partition of every head's rows the dK/dV terms add up to the full result.
    Used for bounded timing samples of long sequences.
    """
    N, Sk = q.shape[1], k.shape[1]
    G = q.shape[2] // k.shape[2]
    rows = np.asarray(rows, dtype=np.int64)
    kk, vv = k[b, :, h // G], v[b, :, h // G]
    M = allowed(spec, N, rows, head=h, Sk=Sk)
    o, lse, P = _rows_fwd(q[b, rows, h], kk, vv, M, scale)
    dOr = do[b, rows, h]
    dV = P.T @ dOr
    dP = dOr @ vv.T
    Dr = (dOr * o).sum(axis=1)
    dS = P * (dP - Dr[:, None])
    dQ = scale * (dS @ kk)
    dK = scale * (dS.T @ q[b, rows, h])
    return dQ, dK, dV, o, lse


def attention_bwd_sampled(q, k, v, do, spec, scale, b: int, g: int, q_rows, k_cols):
    """Gradients at sampled positions of one (batch, KV head g):

    * dQ [G, len(q_rows), D] for every query head of the group at ``q_rows``;
    * dK, dV [len(k_cols), D] at ``k_cols``.

    dK_j and dV_j need O_i and LSE_i for every query row i that attends key j;
    those rows are found from the mask and computed in full, so the cost is
    proportional to the number of such rows times N.
    """
    N, Sk = q.shape[1], k.shape[1]
    Hq, Hkv = q.shape[2], k.shape[2]
    G = Hq // Hkv
    kk, vv = k[b, :, g], v[b, :, g]
    q_rows = np.asarray(q_rows, dtype=np.int64)
    k_cols = np.asarray(k_cols, dtype=np.int64)
    dQ = np.zeros((G, len(q_rows), q.shape[3]))
    dK = np.zeros((len(k_cols), k.shape[3]))
    dV = np.zeros((len(k_cols), v.shape[3]))
    for hi in range(G):
        h = g * G + hi
        # dQ rows: each needs its own full row of P and dP.
        M = allowed(spec, N, q_rows, head=h, Sk=Sk)
        o, lse, P = _rows_fwd(q[b, q_rows, h], kk, vv, M, scale)
        dOr = do[b, q_rows, h]
        dP = dOr @ vv.T
        Dr = (dOr * o).sum(axis=1)
        dS = P * (dP - Dr[:, None])
        dQ[hi] = scale * (dS @ kk)
        # dK/dV columns: find every row that attends at least one sampled key.
        for r0 in range(0, N, 8192):
            rows = np.arange(r0, min(N, r0 + 8192))
            need = allowed(spec, N, rows, head=h, cols=k_cols, Sk=Sk).any(axis=1)
            if not need.any():
                continue
            rr = rows[need]
            Mr = allowed(spec, N, rr, head=h, Sk=Sk)
            o, lse, P = _rows_fwd(q[b, rr, h], kk, vv, Mr, scale)
            dOr = do[b, rr, h]
            Pc = P[:, k_cols]
            dPc = dOr @ vv[k_cols].T
            Dr = (dOr * o).sum(axis=1)
            dSc = Pc * (dPc - Dr[:, None])
            dV += Pc.T @ dOr
            dK += scale * (dSc.T @ q[b, rr, h])
    return dQ, dK, dV


def classify_tiles(spec, N: int, BM: int = 128, BN: int = 128, head: int = 0,
                   q_tiles=None, Sk=None) -> np.ndarray:
    """Class of every (query tile, key tile) pair: EMPTY when no in-range pair of
    the tile is allowed, FULL when all are, PARTIAL otherwise.  Rows past N and
    columns past Sk (default N; a ragged last tile) are not part of the tile.
    With ``q_tiles``, only those rows of tiles are classified (output row r =
    q_tiles[r])."""
    Sk = N if Sk is None else int(Sk)
    nQt = (N + BM - 1) // BM
    nKt = (Sk + BN - 1) // BN
    tiles = range(nQt) if q_tiles is None else list(q_tiles)
    out = np.zeros((len(tiles), nKt), dtype=np.uint8)
    for r, qt in enumerate(tiles):
        rows = np.arange(qt * BM, min(N, (qt + 1) * BM))
        M = allowed(spec, N, rows, head=head, Sk=Sk)
        for kt in range(nKt):
            blk = M[:, kt * BN:min(Sk, (kt + 1) * BN)]
            if not blk.any():
                out[r, kt] = EMPTY
            elif blk.all():
                out[r, kt] = FULL
            else:
                out[r, kt] = PARTIAL
    return out
