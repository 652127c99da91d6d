"""GPU parity of dynamic block selection (TopK / TopP over pooled Q K^T), all
through the C ABI.

The kernel scores in fp32 and the oracle in fp64, and a selection is an integer
decided by those floats, so the comparison is split the way the arithmetic
allows:

* scores: |s_gpu - s_oracle| <= eps, a worst-case fp32 bound derived per
  (query block, key block) from the oracle's own block means (summation of n
  rows: n u sum|x|; a 128-term dot product: 130 u sum|q_bar||k_bar|);
* maps: every decision the oracle takes with a margin larger than the score
  bound must match exactly; the rest (near-ties) must still be a valid TopK /
  TopP set under scores perturbed within eps -- kept blocks never rank below
  dropped ones by more than the bound, TopK keeps exactly min(k, #candidates),
  TopP's kept mass reaches p and is the shortest such prefix, within the fp32
  mass bound;
* the map must also be exactly the selection of the kernel's own fp32 scores
  for TopK (ranking is exact on given floats, equal scores by smaller index).

On the block-structured inputs used here the near-tie set is empty in practice,
so the maps are compared bit for bit; the tests report how many decisions
needed the tolerance path.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import block_select_ref as bs
from synthetic import MaskSpec, qkv_block_structured, segment_lengths

pytestmark = pytest.mark.gpu

lc = pytest.importorskip("long_context_masked_mask_gb300")

U = 2.0 ** -24


def offs_uniform(N, block):
    return np.array(list(range(0, N, block)) + [N], dtype=np.int32)


def offs_from_lens(lens):
    return np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)


def _np(t):
    return t.float().cpu().numpy().astype(np.float64)


def score_bound(q, k, q_offs, k_offs, scale, G):
    """Worst-case |fp32 score - exact score| per (b, h, i, j)."""
    qb = bs.block_means(q, q_offs)
    kb = bs.block_means(k, k_offs)
    qa = bs.block_means(np.abs(q), q_offs)      # mean |x| per block and column
    ka = bs.block_means(np.abs(k), k_offs)
    nq = np.diff(np.asarray(q_offs, dtype=np.int64)).astype(np.float64)
    nk = np.diff(np.asarray(k_offs, dtype=np.int64)).astype(np.float64)
    B, Hq = q.shape[0], q.shape[2]
    out = np.empty((B, Hq, len(nq), len(nk)))
    for h in range(Hq):
        g = h // G
        A = np.einsum("bic,bjc->bij", np.abs(qb[:, h]), np.abs(kb[:, g]))
        Bq = np.einsum("bic,bjc->bij", qa[:, h], np.abs(kb[:, g]))
        Bk = np.einsum("bic,bjc->bij", np.abs(qb[:, h]), ka[:, g])
        s = np.abs(np.einsum("bic,bjc->bij", qb[:, h], kb[:, g]))
        out[:, h] = scale * (130 * U * A + (nq[None, :, None] + 2) * U * Bq
                             + (nk[None, None, :] + 2) * U * Bk + 2 * U * s) * 1.01 + 1e-30
    return out


def check_selection(gmap, S, eps, C, rule, top_k=0, top_p=0.0):
    """Validity of the GPU map against the oracle's fp64 scores S, bound eps and
    candidates C; returns (decisions that needed the tolerance path, rows)."""
    B, Hq, nQb, nKb = S.shape
    loose = 0
    for b in range(B):
        for h in range(Hq):
            for i in range(nQb):
                keep = gmap[b, h, i].astype(bool)
                c = C[i]
                assert not (keep & ~c).any(), "kept a non-candidate"
                idx = np.nonzero(c)[0]
                if len(idx) == 0:
                    continue
                s, e = S[b, h, i], eps[b, h, i]
                kept, dropped = np.nonzero(keep)[0], np.nonzero(c & ~keep)[0]
                if len(kept) and len(dropped):
                    assert (s[kept] + e[kept]).min() >= (s[dropped] - e[dropped]).max(), \
                        f"row {(b, h, i)}: a dropped block outranks a kept one beyond the fp32 bound"
                if rule == bs.TOPK:
                    assert len(kept) == min(top_k, len(idx)), (b, h, i)
                    want = bs.select_topk_row(s, c, top_k)
                else:
                    z = s[idx] - s[idx].max()
                    pr = np.zeros(nKb)
                    pr[idx] = np.exp(z) / np.exp(z).sum()
                    em = float(e[idx].max())
                    delta = 4 * em + (len(idx) + 8) * 2 * U
                    mass = pr[kept].sum()
                    if len(kept) < len(idx):
                        assert mass >= top_p - delta, f"row {(b, h, i)}: kept mass below p"
                    if len(kept):
                        low = kept[s[kept] <= s[kept].min() + 2 * em]
                        assert mass - pr[low].max() < top_p + delta, f"row {(b, h, i)}: not the shortest prefix"
                    want = bs.select_topp_row(s, c, top_p)
                loose += int((want != keep).sum())
    return loose


def run_select(q, k, q_offs, k_offs, rule, top_k=0, top_p=0.0, causal=False, scale=None):
    qo = torch.from_numpy(q_offs).cuda()
    ko = torch.from_numpy(k_offs).cuda()
    m, sc = lc.lcattn_block_select(q.cuda(), k.cuda(), qo, ko, rule, top_k=top_k, top_p=top_p,
                                   causal=causal, scale=scale, want_scores=True)
    torch.cuda.synchronize()
    return m.cpu().numpy(), sc.cpu().numpy().astype(np.float64)


CASES = [
    # name, B, N, Hq, Hkv, q_offs, k_offs
    ("uniform128_ragged_gqa", 2, 1000, 8, 2, offs_uniform(1000, 128), offs_uniform(1000, 128)),
    ("uniform64_mha", 1, 2048, 4, 4, offs_uniform(2048, 64), offs_uniform(2048, 64)),
    ("variable_with_empty", 1, 1500, 4, 2,
     offs_from_lens([100, 0, 37, 300] + segment_lengths(1063, 40, 250, 7)),
     offs_from_lens(segment_lengths(700, 20, 160, 8) + [0, 0] + segment_lengths(800, 50, 300, 9))),
    ("many_key_blocks", 1, 4100, 2, 1, offs_uniform(4100, 256), offs_uniform(4100, 16)),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("rule,param,causal", [
    ("topk", 3, False), ("topk", 5, True), ("topp", 0.5, False), ("topp", 0.9, True)])
def test_block_select_matches_oracle(case, rule, param, causal):
    name, B, N, Hq, Hkv, q_offs, k_offs = case
    x = qkv_block_structured(B, N, Hq, Hkv, 128, strength=1.5, seed=11)
    q64, k64 = _np(x["q"]), _np(x["k"])
    scale = 1.0 / math.sqrt(128)
    top_k = param if rule == "topk" else 0
    top_p = param if rule == "topp" else 0.0
    gmap, gs = run_select(x["q"], x["k"], q_offs, k_offs, rule, top_k, top_p, causal)
    want, S = bs.block_select(q64, k64, q_offs, k_offs, rule, scale, top_k=top_k, top_p=top_p,
                              causal=causal)
    eps = score_bound(q64, k64, q_offs, k_offs, scale, Hq // Hkv)
    err = np.abs(gs - S)
    assert (err <= eps).all(), f"score error {err.max():.3e} above bound (max bound {eps.max():.3e})"
    C = bs.candidates(q_offs, k_offs, causal)
    loose = check_selection(gmap, S, eps, C, rule, top_k, top_p)
    assert loose <= max(2, gmap.size // 5000), f"{loose} decisions differ from the oracle"
    if rule == "topk":
        # exact on the kernel's own fp32 scores: rank by (score desc, index asc)
        for b in range(B):
            for h in range(Hq):
                for i in range(len(q_offs) - 1):
                    idx = np.nonzero(C[i])[0]
                    s32 = gs[b, h, i, idx].astype(np.float32)
                    order = idx[np.lexsort((idx, -s32))]
                    row = np.zeros(len(k_offs) - 1, dtype=np.uint8)
                    row[order[:top_k]] = 1
                    assert np.array_equal(gmap[b, h, i], row), (b, h, i)


@pytest.mark.parametrize("rule,param,expect", [
    ("topk", 0, "none"), ("topk", 10 ** 6, "all"), ("topp", 0.0, "none"), ("topp", -1.0, "none"),
    ("topp", 1.5, "all")])
@pytest.mark.parametrize("causal", [False, True])
def test_block_select_degenerate_parameters(rule, param, expect, causal):
    B, N, Hq, Hkv = 1, 777, 4, 2
    x = qkv_block_structured(B, N, Hq, Hkv, 128, seed=3)
    q_offs = offs_from_lens([50, 0, 300, 427])
    k_offs = offs_uniform(N, 100)
    gmap, _ = run_select(x["q"], x["k"], q_offs, k_offs, rule,
                         top_k=param if rule == "topk" else 0, top_p=param if rule == "topp" else 0.0,
                         causal=causal)
    C = bs.candidates(q_offs, k_offs, causal).astype(np.uint8)
    want = np.zeros_like(gmap) if expect == "none" else np.broadcast_to(C, gmap.shape)
    assert np.array_equal(gmap, want)


def test_block_select_single_block_and_determinism():
    x = qkv_block_structured(1, 300, 2, 1, 128, seed=5)
    one = np.array([0, 300], dtype=np.int32)
    gmap, gs = run_select(x["q"], x["k"], one, one, "topk", top_k=1)
    assert gmap.shape == (1, 2, 1, 1) and gmap.all()
    x = qkv_block_structured(2, 3000, 8, 2, 128, seed=6)
    offs = offs_uniform(3000, 64)
    a = run_select(x["q"], x["k"], offs, offs, "topp", top_p=0.7, causal=True)
    b = run_select(x["q"], x["k"], offs, offs, "topp", top_p=0.7, causal=True)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("nKb", [8192, 16384])
def test_block_select_widest_rows(nKb):
    """The widest sorts (one query block per CTA): 8192 and 16384 key blocks."""
    N = 32768
    x = qkv_block_structured(1, N, 1, 1, 128, strength=1.5, seed=9)
    q_offs = offs_uniform(N, 2048)
    k_offs = offs_uniform(N, N // nKb)
    q64, k64 = _np(x["q"]), _np(x["k"])
    scale = 1.0 / math.sqrt(128)
    for rule, kw in (("topk", {"top_k": 100}), ("topp", {"top_p": 0.8})):
        gmap, gs = run_select(x["q"], x["k"], q_offs, k_offs, rule, causal=True, **kw)
        want, S = bs.block_select(q64, k64, q_offs, k_offs, rule, scale, causal=True, **kw)
        eps = score_bound(q64, k64, q_offs, k_offs, scale, 1)
        assert (np.abs(gs - S) <= eps).all()
        C = bs.candidates(q_offs, k_offs, True)
        loose = check_selection(gmap, S, eps, C, rule, kw.get("top_k", 0), kw.get("top_p", 0.0))
        assert loose <= 4


def _spec_from_map(keep, q_offs, k_offs):
    return MaskSpec("VARIABLE_BLOCK", {"q_block_lens": np.diff(q_offs).tolist(),
                                       "k_block_lens": np.diff(k_offs).tolist(),
                                       "keep": keep.astype(bool)})


@pytest.mark.parametrize("rule,kw", [("topk", {"top_k": 4, "causal": False}),
                                     ("topp", {"top_p": 0.85, "causal": True})])
def test_selected_map_drives_attention(rule, kw):
    """select -> mask compile -> forward + backward on the selected map, against
    the oracle's attention on the oracle's own selection (maps must agree)."""
    B, N, Hq, Hkv = 1, 1100, 4, 2
    x = qkv_block_structured(B, N, Hq, Hkv, 128, strength=1.5, seed=21)
    offs = offs_uniform(N, 128)
    scale = 1.0 / math.sqrt(128)
    q64, k64 = _np(x["q"]), _np(x["k"])
    want, _ = bs.block_select(q64, k64, offs, offs, rule, scale, **kw)
    dev = {n: t.cuda() for n, t in x.items()}
    qo, ko = torch.from_numpy(offs).cuda(), torch.from_numpy(offs).cuda()
    gmap, _ = lc.lcattn_block_select(dev["q"], dev["k"], qo, ko, rule, **kw)
    assert np.array_equal(gmap.cpu().numpy(), want), "maps differ on a seed with no near-ties"
    mask = lc.DeviceMask.from_block_map(gmap, qo, ko)
    shape = lc.make_shape(dev["q"], dev["k"], dev["v"])
    meta = lc.lcattn_mask_compile(shape, mask)
    o, lse = lc.lcattn_fwd(dev["q"], dev["k"], dev["v"], mask, meta)
    dq, dk, dv = lc.lcattn_bwd(dev["q"], dev["k"], dev["v"], o, dev["do"], lse, mask, meta)
    assert lc.lcattn_read_status(meta) == 0
    spec = _spec_from_map(want[0], offs, offs)
    O, LSE = oracle.attention_fwd(q64, k64, _np(x["v"]), spec, scale)
    dQ, dK, dV = oracle.attention_bwd(q64, k64, _np(x["v"]), _np(x["do"]), spec, scale)[:3]

    def relf(g, r):
        return float(np.linalg.norm(g - r) / np.linalg.norm(r))

    go = _np(o)
    assert np.abs(go - O).max() <= 2e-2 and relf(go, O) <= 1e-2
    fin = np.isfinite(LSE)
    gl = lse.cpu().numpy()
    assert np.array_equal(np.isfinite(gl), fin) and np.abs(gl[fin] - LSE[fin]).max() <= 5e-3
    for g, r in ((dq, dQ), (dk, dK), (dv, dV)):
        assert relf(_np(g), r) <= 3e-2
    assert mask.allowed_pairs == int(sum(
        want[0, h, i, j] * (offs[i + 1] - offs[i]) * (offs[j + 1] - offs[j])
        for h in range(Hq) for i in range(len(offs) - 1) for j in range(len(offs) - 1)))


@pytest.mark.parametrize("si", [0, 1])
def test_dynamic_32k_full_size(si):
    """The dynamic workload at its full size (B=1, N=32768, GQA 64:8), in the
    launch configuration the benchmark times: select -> compile -> forward ->
    backward.  The oracle selects for two KV groups (16 query heads) whole and
    checks the attention at sampled rows and key columns of one group."""
    from synthetic import workload
    wl = workload("dynamic_32k")
    sel = wl.selects[si]
    B, N, Hq, Hkv, D = wl.B, wl.N, wl.Hq, wl.Hkv, wl.D
    G = Hq // Hkv
    x = qkv_block_structured(B, N, Hq, Hkv, sel.block, strength=wl.structure, seed=0, device="cuda")
    offs = offs_uniform(N, sel.block)
    qo = torch.from_numpy(offs).cuda()
    kw = {"top_k": sel.top_k} if sel.rule == "topk" else {"top_p": sel.top_p}
    gmap, gs = lc.lcattn_block_select(x["q"], x["k"], qo, qo, sel.rule, causal=sel.causal,
                                      want_scores=True, **kw)
    mask = lc.DeviceMask.from_block_map(gmap, qo, qo)
    shape = lc.make_shape(x["q"], x["k"], x["v"])
    meta = lc.lcattn_mask_compile(shape, mask)
    o, lse = lc.lcattn_fwd(x["q"], x["k"], x["v"], mask, meta)
    dq, dk, dv = lc.lcattn_bwd(x["q"], x["k"], x["v"], o, x["do"], lse, mask, meta)
    torch.cuda.synchronize()
    assert lc.lcattn_read_status(meta) == 0
    scale = 1.0 / math.sqrt(D)
    gmap_h, gs_h = gmap.cpu().numpy(), gs.cpu().numpy().astype(np.float64)
    C = bs.candidates(offs, offs, sel.causal)
    for g in (0, Hkv - 1):
        heads = slice(g * G, (g + 1) * G)
        q64 = x["q"][:, :, heads].double().cpu().numpy()
        k64 = x["k"][:, :, g:g + 1].double().cpu().numpy()
        want, S = bs.block_select(q64, k64, offs, offs, sel.rule, scale, causal=sel.causal, **kw)
        eps = score_bound(q64, k64, offs, offs, scale, G)
        assert (np.abs(gs_h[:, heads] - S) <= eps).all()
        loose = check_selection(gmap_h[:, heads], S, eps, C, sel.rule, kw.get("top_k", 0),
                                kw.get("top_p", 0.0))
        assert loose <= 4
    # attention on the selected map, group 0, against the oracle on that same map
    # (the map was just shown to be the oracle's selection up to near-ties)
    heads = list(range(G))
    spec = _spec_from_map(gmap_h[0, heads], offs, offs)
    f64 = lambda t, sl: t[:, :, sl].double().cpu().numpy()
    q, do = f64(x["q"], slice(0, G)), f64(x["do"], slice(0, G))
    k, v = f64(x["k"], slice(0, 1)), f64(x["v"], slice(0, 1))
    rng = np.random.default_rng(2)
    rows = np.array(sorted({0, 1, N - 1, N // 2} | {int(r) for r in rng.integers(0, N, 20)}))
    ref = [oracle.attention_fwd_rows(q, k, v, spec, scale, 0, hi, rows) for hi in range(G)]
    O_ref = np.stack([r[0] for r in ref], 1)
    L_ref = np.stack([r[1] for r in ref], 0)
    o_gpu = o[0][:, heads][rows].double().cpu().numpy()
    l_gpu = lse[0][heads][:, rows].double().cpu().numpy()
    assert np.abs(o_gpu - O_ref).max() <= 2e-2
    assert np.linalg.norm(o_gpu - O_ref) <= 1e-2 * np.linalg.norm(O_ref)
    fin = np.isfinite(L_ref)
    assert np.array_equal(np.isfinite(l_gpu), fin) and np.abs(l_gpu[fin] - L_ref[fin]).max() <= 5e-3
    cols = np.array([N // 3, N - 1])
    dQ_ref, dK_ref, dV_ref = oracle.attention_bwd_sampled(q, k, v, do, spec, scale, 0, 0, rows, cols)
    dq_gpu = dq[0][:, heads][rows].double().cpu().numpy().transpose(1, 0, 2)
    assert np.linalg.norm(dq_gpu - dQ_ref) <= 3e-2 * np.linalg.norm(dQ_ref)
    for gg, r in ((dk[0, cols, 0], dK_ref), (dv[0, cols, 0], dV_ref)):
        gg = gg.double().cpu().numpy()
        assert np.linalg.norm(gg - r) <= 3e-2 * max(np.linalg.norm(r), 1e-30)
