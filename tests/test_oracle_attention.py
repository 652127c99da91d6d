"""Pins for the oracle's fp64 attention (CPU only).

The oracle is checked against things other than itself:
* torch's own fp64 ``scaled_dot_product_attention`` with an explicit boolean mask
  (a library routine) and torch autograd through it, on tiny random problems;
* closed forms: one key (O = v_0, LSE = s q.k), identical keys (O = mean of the
  allowed values, LSE = s q.k + log count), rows of P summing to 1;
* central finite differences of L = <O, dO> for the backward;
* fully-masked rows (O = 0, LSE = -inf, no gradient) and GQA = MHA with
  replicated KV heads.
"""
import math

import numpy as np
import pytest
import torch

from oracle import (allowed, attention_bwd, attention_bwd_sampled, attention_fwd,
                    attention_fwd_rows)
from oracle.attention_ref import _rows_fwd
import oracle
from synthetic import MaskSpec, block_keep

SPECS = [
    MaskSpec("FULL"),
    MaskSpec("CAUSAL"),
    MaskSpec("FULL_DOCUMENT", {"doc_lens": [5, 11, 8]}),
    MaskSpec("CAUSAL_DOCUMENT", {"doc_lens": [5, 11, 8]}),
    MaskSpec("FULL_SLIDING_WINDOW", {"window": 4}),
    MaskSpec("CAUSAL_SLIDING_WINDOW", {"window": 4}),
    MaskSpec("SHARED_QUESTION", {"question_len": 6, "answer_lens": [6, 7, 5]}),
    MaskSpec("GLOBAL_SLIDING", {"global_tokens": 2, "window": 3}),
    MaskSpec("CAUSAL_BLOCKWISE", {"block": 5}),
    MaskSpec("PREFIX_LM_CAUSAL", {"prefix": 7}),
    MaskSpec("PREFIX_LM_DOCUMENT", {"doc_lens": [5, 11, 8], "prefix_lens": [2, 5, 0]}),
    MaskSpec("BLOCK_CAUSAL_DOCUMENT", {"doc_lens": [5, 11, 8], "block_lens": [[2, 3], [4, 4, 3], [8]]}),
    MaskSpec("UNIFORM_BLOCK", {"block": 4, "keep": block_keep(4, 6, 6, 0.5, 7)}),
    MaskSpec("VARIABLE_BLOCK", {"q_block_lens": [3, 9, 12], "k_block_lens": [7, 2, 15],
                                "keep": block_keep(4, 3, 3, 0.5, 9)}),
]


def _rand(B, N, Hq, Hkv, D, seed):
    g = np.random.default_rng(seed)
    return (g.standard_normal((B, N, Hq, D)), g.standard_normal((B, N, Hkv, D)),
            g.standard_normal((B, N, Hkv, D)), g.standard_normal((B, N, Hq, D)))


def _sdpa_torch(q, k, v, spec, scale):
    """torch fp64 SDPA per head with the explicit bool mask; KV heads repeated per group."""
    B, N, Hq, D = q.shape
    G = Hq // k.shape[2]
    qt = torch.tensor(q).permute(0, 2, 1, 3).requires_grad_(True)
    kt = torch.tensor(k).permute(0, 2, 1, 3).requires_grad_(True)
    vt = torch.tensor(v).permute(0, 2, 1, 3).requires_grad_(True)
    mask = torch.stack([torch.tensor(allowed(spec, N, head=h)) for h in range(Hq)])[None]
    ke = kt.repeat_interleave(G, dim=1)
    ve = vt.repeat_interleave(G, dim=1)
    o = torch.nn.functional.scaled_dot_product_attention(qt, ke, ve, attn_mask=mask, scale=scale)
    return o, (qt, kt, vt), mask


@pytest.mark.parametrize("spec", SPECS, ids=lambda s: s.kind)
def test_fwd_bwd_vs_torch_sdpa(spec):
    B, N, Hq, Hkv, D = 1, 24, 4, 2, 8
    q, k, v, do = _rand(B, N, Hq, Hkv, D, seed=11)
    scale = 1.0 / math.sqrt(D)
    O, LSE = attention_fwd(q, k, v, spec, scale, chunk=7)
    o_t, (qt, kt, vt), mask = _sdpa_torch(q, k, v, spec, scale)
    np.testing.assert_allclose(O, o_t.permute(0, 2, 1, 3).detach().numpy(), rtol=0, atol=1e-12)
    # LSE against torch.logsumexp of the masked scores
    ke = torch.tensor(k).permute(0, 2, 1, 3).repeat_interleave(Hq // Hkv, dim=1)
    s = scale * torch.tensor(q).permute(0, 2, 1, 3) @ ke.transpose(-1, -2)
    lse_t = torch.logsumexp(s.masked_fill(~mask, -math.inf), dim=-1)
    np.testing.assert_allclose(LSE, lse_t.numpy(), rtol=0, atol=1e-12)
    # backward against autograd
    (o_t * torch.tensor(do).permute(0, 2, 1, 3)).sum().backward()
    dQ, dK, dV, _, _ = attention_bwd(q, k, v, do, spec, scale, chunk=5)
    np.testing.assert_allclose(dQ, qt.grad.permute(0, 2, 1, 3).numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dK, kt.grad.permute(0, 2, 1, 3).numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dV, vt.grad.permute(0, 2, 1, 3).numpy(), rtol=0, atol=1e-11)


def test_single_key_closed_form():
    q, k, v, _ = _rand(2, 1, 3, 3, 5, seed=1)
    s = 0.37
    O, LSE = attention_fwd(q, k, v, MaskSpec("FULL"), s)
    np.testing.assert_allclose(O, v, atol=1e-15)
    np.testing.assert_allclose(LSE, s * np.einsum("bnhd,bnhd->bhn", q, k), atol=1e-14)


@pytest.mark.parametrize("spec", SPECS, ids=lambda s: s.kind)
def test_identical_keys_closed_form(spec):
    """With every key equal, softmax is uniform over the allowed keys of a row."""
    N, D = 24, 6
    q, k, v, _ = _rand(1, N, 4, 2, D, seed=4)
    k[:] = k[:, :1]
    s = 0.5
    O, LSE = attention_fwd(q, k, v, spec, s)
    for h in range(4):
        M = allowed(spec, N, head=h)
        cnt = M.sum(1)
        g = h // 2
        want_o = (M.astype(float) @ v[0, :, g]) / cnt[:, None]
        want_lse = s * q[0, :, h] @ k[0, 0, g] + np.log(cnt)
        np.testing.assert_allclose(O[0, :, h], want_o, atol=1e-12)
        np.testing.assert_allclose(LSE[0, h], want_lse, atol=1e-12)


def test_rows_of_p_sum_to_one():
    N, D = 40, 8
    q, k, v, _ = _rand(1, N, 1, 1, D, seed=5)
    spec = MaskSpec("GLOBAL_SLIDING", {"global_tokens": 3, "window": 4})
    M = allowed(spec, N)
    _, lse, P = _rows_fwd(q[0, :, 0], k[0, :, 0], v[0, :, 0], M, 0.3)
    np.testing.assert_allclose(P.sum(1), 1.0, atol=1e-12)
    assert (P[~M] == 0).all()
    # LSE is the log of the normaliser: P_ij = exp(S_ij - LSE_i) on allowed pairs
    S = 0.3 * q[0, :, 0] @ k[0, :, 0].T
    np.testing.assert_allclose(P[M], np.exp(S - lse[:, None])[M], rtol=1e-12)


def test_fully_masked_rows():
    """A row that allows no key gives O = 0, LSE = -inf and contributes no gradient."""
    N, D = 12, 4
    q, k, v, do = _rand(1, N, 2, 1, D, seed=6)
    keep = np.ones((2, 3, 3), dtype=bool)
    keep[:, 1, :] = False  # query block 1 (rows 4..7) sees nothing
    spec = MaskSpec("UNIFORM_BLOCK", {"block": 4, "keep": keep})
    O, LSE = attention_fwd(q, k, v, spec, 0.5)
    assert (O[0, 4:8] == 0).all()
    assert np.isneginf(LSE[0, :, 4:8]).all()
    assert np.isfinite(LSE[0, :, :4]).all() and np.isfinite(LSE[0, :, 8:]).all()
    dQ, dK, dV, _, _ = attention_bwd(q, k, v, do, spec, 0.5)
    assert (dQ[0, 4:8] == 0).all()
    # the masked rows' q and dO do not influence dK/dV
    q2, do2 = q.copy(), do.copy()
    q2[0, 4:8] += 3.0
    do2[0, 4:8] -= 2.0
    _, dK2, dV2, _, _ = attention_bwd(q2, k, v, do2, spec, 0.5)
    np.testing.assert_allclose(dK2, dK, atol=1e-13)
    np.testing.assert_allclose(dV2, dV, atol=1e-13)


def test_gqa_equals_mha_with_replicated_kv():
    N, D = 16, 4
    q, k, v, do = _rand(1, N, 4, 2, D, seed=8)
    spec = MaskSpec("CAUSAL_SLIDING_WINDOW", {"window": 5})
    O, LSE = attention_fwd(q, k, v, spec, 0.4)
    O2, LSE2 = attention_fwd(q, np.repeat(k, 2, axis=2), np.repeat(v, 2, axis=2), spec, 0.4)
    np.testing.assert_allclose(O, O2, atol=1e-14)
    np.testing.assert_allclose(LSE, LSE2, atol=1e-14)
    dQ, dK, dV, _, _ = attention_bwd(q, k, v, do, spec, 0.4)
    dQ2, dK2, dV2, _, _ = attention_bwd(q, np.repeat(k, 2, axis=2), np.repeat(v, 2, axis=2), do, spec, 0.4)
    np.testing.assert_allclose(dQ, dQ2, atol=1e-13)
    # the group's KV gradient is the sum over its query heads
    np.testing.assert_allclose(dK, dK2.reshape(1, N, 2, 2, D).sum(3), atol=1e-13)
    np.testing.assert_allclose(dV, dV2.reshape(1, N, 2, 2, D).sum(3), atol=1e-13)


@pytest.mark.parametrize("spec", [SPECS[1], SPECS[6], SPECS[7], SPECS[12]], ids=lambda s: s.kind)
def test_bwd_finite_differences(spec):
    """Central differences of L = <O, dO>, autograd-free, h = 1e-6."""
    B, N, Hq, Hkv, D = 1, 12, 4, 2, 4
    q, k, v, do = _rand(B, N, Hq, Hkv, D, seed=21)
    if spec.kind == "SHARED_QUESTION":
        spec = MaskSpec("SHARED_QUESTION", {"question_len": 3, "answer_lens": [4, 5]})
    if spec.kind == "UNIFORM_BLOCK":
        spec = MaskSpec("UNIFORM_BLOCK", {"block": 4, "keep": block_keep(4, 3, 3, 0.5, 2)})
    s = 0.45
    dQ, dK, dV, _, _ = attention_bwd(q, k, v, do, spec, s)

    def loss(qq, kk, vv):
        O, _ = attention_fwd(qq, kk, vv, spec, s)
        return float((O * do).sum())

    rng = np.random.default_rng(0)
    h = 1e-6
    for name, arr, grad in (("q", q, dQ), ("k", k, dK), ("v", v, dV)):
        for _ in range(6):
            idx = tuple(int(rng.integers(0, n)) for n in arr.shape)
            a_p = arr.copy(); a_p[idx] += h
            a_m = arr.copy(); a_m[idx] -= h
            p_args = {"q": q, "k": k, "v": v, name: a_p}
            m_args = {"q": q, "k": k, "v": v, name: a_m}
            fd = (loss(p_args["q"], p_args["k"], p_args["v"]) -
                  loss(m_args["q"], m_args["k"], m_args["v"])) / (2 * h)
            assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(grad[idx])), (name, idx, fd, grad[idx])


def test_sampled_paths_match_full():
    B, N, Hq, Hkv, D = 1, 40, 4, 2, 8
    q, k, v, do = _rand(B, N, Hq, Hkv, D, seed=31)
    spec = MaskSpec("PREFIX_LM_CAUSAL", {"prefix": 9})
    s = 0.3
    dQ, dK, dV, O, LSE = attention_bwd(q, k, v, do, spec, s)
    rows = np.array([0, 5, 17, 39])
    o, lse = attention_fwd_rows(q, k, v, spec, s, 0, 3, rows)
    np.testing.assert_allclose(o, O[0, rows, 3], atol=1e-13)
    np.testing.assert_allclose(lse, LSE[0, 3, rows], atol=1e-13)
    cols = np.array([0, 8, 9, 30, 39])
    sdq, sdk, sdv = attention_bwd_sampled(q, k, v, do, spec, s, 0, 1, rows, cols)
    np.testing.assert_allclose(sdq, dQ[0][rows][:, 2:4].transpose(1, 0, 2), atol=1e-12)
    np.testing.assert_allclose(sdk, dK[0, cols, 1], atol=1e-12)
    np.testing.assert_allclose(sdv, dV[0, cols, 1], atol=1e-12)


@pytest.mark.parametrize("spec", [MaskSpec("CAUSAL_DOCUMENT", {"doc_lens": [11, 20, 9]}),
                                  MaskSpec("UNIFORM_BLOCK", {"block": 8, "keep": block_keep(4, 5, 5, 0.5, 3)})],
                         ids=lambda s: s.kind)
def test_bwd_rows_vs_torch_with_do_zero_elsewhere(spec):
    """attention_bwd_rows for rows R of head h equals torch's fp64 SDPA autograd
    on a problem whose dO is zero outside (R, h): then only those rows reach the
    loss, so torch's dK/dV are exactly their terms and its dQ rows are theirs."""
    B, N, Hq, Hkv, D = 1, 40, 4, 2, 8
    q, k, v, do = _rand(B, N, Hq, Hkv, D, seed=53)
    s, h = 0.3, 3
    rows = np.array([2, 9, 10, 25, 39])
    do_sel = np.zeros_like(do)
    do_sel[0, rows, h] = do[0, rows, h]
    o, (qt, kt, vt), _ = _sdpa_torch(q, k, v, spec, s)
    (o * torch.tensor(do_sel).permute(0, 2, 1, 3)).sum().backward()
    dQ, dK, dV, O, LSE = oracle.attention_bwd_rows(q, k, v, do, spec, s, 0, h, rows)
    np.testing.assert_allclose(O, o.detach().permute(0, 2, 1, 3).numpy()[0, rows, h], atol=1e-12)
    np.testing.assert_allclose(dQ, qt.grad.permute(0, 2, 1, 3).numpy()[0, rows, h], atol=1e-12)
    np.testing.assert_allclose(dK, kt.grad.permute(0, 2, 1, 3).numpy()[0, :, h // 2], atol=1e-12)
    np.testing.assert_allclose(dV, vt.grad.permute(0, 2, 1, 3).numpy()[0, :, h // 2], atol=1e-12)
    # Over a partition of every head's rows the terms add up to the full backward.
    fdQ, fdK, fdV, _, fLSE = attention_bwd(q, k, v, do, spec, s)
    np.testing.assert_allclose(LSE, fLSE[0, h, rows], atol=1e-12)
    sk, sv = np.zeros_like(k[0]), np.zeros_like(v[0])
    for hh in range(Hq):
        for part in (np.arange(0, 17), np.arange(17, N)):
            _, dk_, dv_, _, _ = oracle.attention_bwd_rows(q, k, v, do, spec, s, 0, hh, part)
            sk[:, hh // 2] += dk_
            sv[:, hh // 2] += dv_
    np.testing.assert_allclose(sk, fdK[0], atol=1e-11)
    np.testing.assert_allclose(sv, fdV[0], atol=1e-11)


def test_gradient_sum_identities():
    """sum_j dK_j = 0 and sum_j dV_j = sum over non-empty rows of dO (per KV head).

    Both follow from sum_j P_ij = 1 and sum_j dS_ij = <dO_i, O_i> - D_i = 0; the
    GPU tests use them at sizes the oracle cannot reach."""
    N, D = 30, 6
    q, k, v, do = _rand(1, N, 4, 2, D, seed=41)
    spec = MaskSpec("CAUSAL_DOCUMENT", {"doc_lens": [10, 12, 8]})
    dQ, dK, dV, _, _ = attention_bwd(q, k, v, do, spec, 0.25)
    np.testing.assert_allclose(dK.sum(1), 0.0, atol=1e-12)
    np.testing.assert_allclose(dV.sum(1), do.reshape(1, N, 2, 2, D).sum(axis=(1, 3)), atol=1e-12)


# ---- query and key lengths that differ (bottom-right alignment) -------------

def _rect_inputs(B, Sq, Sk, Hq, Hkv, D, seed):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((B, Sq, Hq, D)), rng.standard_normal((B, Sk, Hkv, D)),
            rng.standard_normal((B, Sk, Hkv, D)), rng.standard_normal((B, Sq, Hq, D)))


# torch warns that its lower-right bias gives NaN rows when Sq > Sk; the test
# compares only the rows that allow a key.
@pytest.mark.filterwarnings("ignore:Lower right causal bias")
@pytest.mark.parametrize("Sq,Sk", [(5, 13), (1, 9), (9, 4), (7, 7)])
def test_causal_rectangular_matches_torch_lower_right(Sq, Sk):
    """CAUSAL with Sq != Sk against torch's own lower-right causal bias
    (torch.nn.attention.bias.causal_lower_right) and autograd, in fp64."""
    from torch.nn.attention.bias import causal_lower_right
    B, Hq, Hkv, D = 1, 4, 2, 8
    q, k, v, do = _rect_inputs(B, Sq, Sk, Hq, Hkv, D, 17)
    scale = 0.31
    spec = MaskSpec("CAUSAL")
    dQ, dK, dV, O, LSE = oracle.attention_bwd(q, k, v, do, spec, scale, chunk=3)
    G = Hq // Hkv
    qt, kt, vt = (torch.tensor(x).permute(0, 2, 1, 3).requires_grad_(True) for x in (q, k, v))
    bias = causal_lower_right(Sq, Sk)
    dense = bias._materialize(device=torch.device("cpu"))          # True = allowed, [Sq, Sk]
    has = dense.any(-1)
    o = torch.nn.functional.scaled_dot_product_attention(
        qt, kt.repeat_interleave(G, 1), vt.repeat_interleave(G, 1),
        attn_mask=dense | ~has[:, None], scale=scale)
    o = o * has[None, None, :, None]
    (o * torch.tensor(do).permute(0, 2, 1, 3)).sum().backward()
    back = lambda t: t.detach().permute(0, 2, 1, 3).numpy()
    for got, want in ((O, back(o)), (dQ, back(qt.grad)), (dK, back(kt.grad)), (dV, back(vt.grad))):
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-10)
    np.testing.assert_array_equal(np.isfinite(LSE[0, 0]), has.numpy())
    assert int(has.sum()) == min(Sq, Sk) if Sq > Sk else int(has.sum()) == Sq


@pytest.mark.parametrize("kind,params", [("CAUSAL", {}), ("CAUSAL_SLIDING_WINDOW", {"window": 4}),
                                         ("FULL_SLIDING_WINDOW", {"window": 3}), ("FULL", {})])
@pytest.mark.parametrize("Sq", [1, 4, 11])
def test_rectangular_is_the_suffix_of_the_square_problem(kind, params, Sq):
    """Bottom-right alignment: the Sq queries behave exactly like the last Sq
    rows of the square problem over the same Sk keys.  With dO = 0 on the other
    rows, dK and dV agree too."""
    B, Sk, Hq, Hkv, D = 1, 12, 2, 1, 8
    q, k, v, do = _rect_inputs(B, Sq, Sk, Hq, Hkv, D, 5)
    spec = MaskSpec(kind, params)
    scale = 0.4
    rng = np.random.default_rng(6)
    qs = np.concatenate([rng.standard_normal((B, Sk - Sq, Hq, D)), q], axis=1)
    dos = np.concatenate([np.zeros((B, Sk - Sq, Hq, D)), do], axis=1)
    r = oracle.attention_bwd(q, k, v, do, spec, scale)
    s = oracle.attention_bwd(qs, k, v, dos, spec, scale)
    np.testing.assert_allclose(r[3], s[3][:, Sk - Sq:], rtol=0, atol=1e-12)        # O
    np.testing.assert_allclose(r[4], s[4][:, :, Sk - Sq:], rtol=0, atol=1e-12)     # LSE
    np.testing.assert_allclose(r[0], s[0][:, Sk - Sq:], rtol=0, atol=1e-12)        # dQ
    np.testing.assert_allclose(r[1], s[1], rtol=0, atol=1e-12)                     # dK
    np.testing.assert_allclose(r[2], s[2], rtol=0, atol=1e-12)                     # dV


def test_rectangular_only_where_defined():
    with pytest.raises(ValueError):
        oracle.allowed(MaskSpec("CAUSAL_DOCUMENT", {"doc_lens": [3, 2]}), 5, Sk=7)
