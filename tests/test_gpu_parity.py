"""GPU parity at sizes the oracle finishes in seconds (spanning several tiles and
a ragged tail): every mask family, MHA and GQA, both descriptor kinds.  All
calls go through the C ABI.  Bars: O max-abs <= 2e-2 and relative Frobenius
<= 1e-2; dQ/dK/dV relative Frobenius <= 3e-2; LSE max-abs <= 5e-3 with -inf
at exactly the oracle's -inf rows; tile classes bit-exact."""
import math

import numpy as np
import pytest
import torch

import oracle
from synthetic import MaskSpec, block_keep, qkv, segment_lengths

pytestmark = pytest.mark.gpu

lc = pytest.importorskip("long_context_masked_mask_gb300")

O_MAXABS, O_RELF, G_RELF, LSE_MAXABS = 2e-2, 1e-2, 3e-2, 5e-3


def relf(g, r):
    nr = np.linalg.norm(r)
    return float(np.linalg.norm(g - r) / nr) if nr > 0 else float(np.linalg.norm(g))


def spec_for(kind, N, Hq, seed=0):
    docs = segment_lengths(N, max(1, N // 6), max(2, N // 2), seed)
    if kind == "FULL":
        return MaskSpec("FULL")
    if kind == "CAUSAL":
        return MaskSpec("CAUSAL")
    if kind == "FULL_DOCUMENT":
        return MaskSpec("FULL_DOCUMENT", {"doc_lens": docs})
    if kind == "CAUSAL_DOCUMENT":
        return MaskSpec("CAUSAL_DOCUMENT", {"doc_lens": docs})
    if kind == "FULL_SLIDING_WINDOW":
        return MaskSpec("FULL_SLIDING_WINDOW", {"window": max(1, N // 5)})
    if kind == "CAUSAL_SLIDING_WINDOW":
        return MaskSpec("CAUSAL_SLIDING_WINDOW", {"window": max(1, N // 4)})
    if kind == "SHARED_QUESTION":
        q = N // 4
        return MaskSpec("SHARED_QUESTION", {"question_len": q,
                                            "answer_lens": segment_lengths(N - q, 20, N // 3, seed + 1)})
    if kind == "GLOBAL_SLIDING":
        return MaskSpec("GLOBAL_SLIDING", {"global_tokens": max(1, N // 16), "window": max(1, N // 8)})
    if kind == "CAUSAL_BLOCKWISE":
        return MaskSpec("CAUSAL_BLOCKWISE", {"block": max(1, N // 5)})
    if kind == "PREFIX_LM_CAUSAL":
        return MaskSpec("PREFIX_LM_CAUSAL", {"prefix": N // 3})
    if kind == "PREFIX_LM_DOCUMENT":
        return MaskSpec("PREFIX_LM_DOCUMENT", {"doc_lens": docs, "prefix_lens": [L // 2 for L in docs]})
    if kind == "BLOCK_CAUSAL_DOCUMENT":
        blocks = [segment_lengths(L, 16, 96, seed + 5 + i) for i, L in enumerate(docs)]
        return MaskSpec("BLOCK_CAUSAL_DOCUMENT", {"doc_lens": docs, "block_lens": blocks})
    if kind == "UNIFORM_BLOCK":
        bs = 64
        nb = -(-N // bs)
        return MaskSpec("UNIFORM_BLOCK", {"block": bs, "keep": block_keep(Hq, nb, nb, 0.5, seed)})
    if kind == "UNIFORM_BLOCK_128":
        nb = -(-N // 128)
        return MaskSpec("UNIFORM_BLOCK", {"block": 128, "keep": block_keep(Hq, nb, nb, 0.5, seed)})
    if kind == "VARIABLE_BLOCK":
        ql = segment_lengths(N, 32, 200, seed + 2)
        kl = segment_lengths(N, 32, 200, seed + 3)
        return MaskSpec("VARIABLE_BLOCK", {"q_block_lens": ql, "k_block_lens": kl,
                                           "keep": block_keep(Hq, len(ql), len(kl), 0.5, seed, force_diagonal=False)})
    raise KeyError(kind)


KINDS = ["FULL", "CAUSAL", "FULL_DOCUMENT", "CAUSAL_DOCUMENT", "FULL_SLIDING_WINDOW",
         "CAUSAL_SLIDING_WINDOW", "SHARED_QUESTION", "GLOBAL_SLIDING", "CAUSAL_BLOCKWISE",
         "PREFIX_LM_CAUSAL", "PREFIX_LM_DOCUMENT", "BLOCK_CAUSAL_DOCUMENT", "UNIFORM_BLOCK",
         "UNIFORM_BLOCK_128", "VARIABLE_BLOCK"]


def run_and_compare(spec, B, N, Hq, Hkv, seed=0, check_classes=True, D=128):
    x = qkv(B, N, Hq, Hkv, D, seed=seed)
    dev = {k: t.cuda() for k, t in x.items()}
    out = lc.attention(dev["q"], dev["k"], dev["v"], spec, d_o=dev["do"])
    torch.cuda.synchronize()
    assert lc.lcattn_read_status(out["tile_meta"]) == 0
    f64 = {k: t.double().numpy() for k, t in x.items()}
    scale = 1.0 / math.sqrt(D)
    dQ, dK, dV, O, LSE = oracle.attention_bwd(f64["q"], f64["k"], f64["v"], f64["do"], spec, scale)
    o = out["o"].double().cpu().numpy()
    lse = out["lse"].double().cpu().numpy()
    assert np.abs(o - O).max() <= O_MAXABS, np.abs(o - O).max()
    assert relf(o, O) <= O_RELF, relf(o, O)
    inf_ref = np.isneginf(LSE)
    np.testing.assert_array_equal(np.isneginf(lse), inf_ref)
    if (~inf_ref).any():
        assert np.abs(lse[~inf_ref] - LSE[~inf_ref]).max() <= LSE_MAXABS
    for name, ref in (("dq", dQ), ("dk", dK), ("dv", dV)):
        g = out[name].double().cpu().numpy()
        assert np.isfinite(g).all(), name
        assert relf(g, ref) <= G_RELF, (name, relf(g, ref))
    # attention() runs lcattn_fwd_ws, which takes the split-KV path on small
    # problems with column bounds; the regular persistent forward must match too.
    o2, lse2 = lc.lcattn_fwd(dev["q"], dev["k"], dev["v"], out["mask"], out["tile_meta"])
    o2 = o2.double().cpu().numpy()
    lse2 = lse2.double().cpu().numpy()
    assert np.abs(o2 - O).max() <= O_MAXABS and relf(o2, O) <= O_RELF
    np.testing.assert_array_equal(np.isneginf(lse2), inf_ref)
    if (~inf_ref).any():
        assert np.abs(lse2[~inf_ref] - LSE[~inf_ref]).max() <= LSE_MAXABS
    if check_classes:
        shape = lc.make_shape(dev["q"], dev["k"], dev["v"])
        cls = lc.tile_classes(out["tile_meta"], shape, out["mask"]).cpu().numpy()
        heads = range(Hq) if spec.per_head else [0]
        for b in range(B):
            for hi, h in enumerate(heads):
                np.testing.assert_array_equal(cls[b, hi], oracle.classify_tiles(spec, N, 128, 128, head=h))
    return out, (dQ, dK, dV, O, LSE)


@pytest.mark.parametrize("kind", KINDS)
def test_mask_family_gqa_ragged(kind):
    N, Hq, Hkv = 392, 4, 2
    run_and_compare(spec_for(kind, N, Hq), 1, N, Hq, Hkv)


COLUMN_KINDS = [k for k in KINDS if not k.startswith(("UNIFORM", "VARIABLE"))]


@pytest.mark.parametrize("kind", COLUMN_KINDS)
def test_forward_column_path_matches_row_path(kind):
    """A column-bounds descriptor without the per-row form makes the forward
    build partial-tile masks from the 128 column bounds (staged in shared
    memory) instead of the row intervals: the oracle and the row path agree."""
    N, Hq, Hkv = 392, 4, 2
    spec = spec_for(kind, N, Hq)
    x = qkv(1, N, Hq, Hkv, 128, seed=6, with_do=False)
    dev = {k: t.cuda() for k, t in x.items()}
    shape = lc.make_shape(dev["q"], dev["k"], dev["v"])
    outs = []
    for rows in (True, False):
        mask = lc.DeviceMask(spec, N, Hq, row_bounds=rows)
        meta = lc.lcattn_mask_compile(shape, mask)
        o, lse = lc.lcattn_fwd(dev["q"], dev["k"], dev["v"], mask, meta)
        assert lc.lcattn_read_status(meta) == 0
        outs.append((o.clone(), lse.clone()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    f64 = {k: t.double().numpy() for k, t in x.items()}
    O, LSE = oracle.attention_fwd(f64["q"], f64["k"], f64["v"], spec, 1.0 / math.sqrt(128))
    o = outs[1][0].double().cpu().numpy()
    assert np.abs(o - O).max() <= O_MAXABS and relf(o, O) <= O_RELF


@pytest.mark.parametrize("kind", ["CAUSAL", "GLOBAL_SLIDING", "SHARED_QUESTION", "UNIFORM_BLOCK"])
def test_mha_and_batch(kind):
    N, Hq = 512, 2
    run_and_compare(spec_for(kind, N, Hq, seed=3), 2, N, Hq, Hq, seed=1)


@pytest.mark.parametrize("Hq,Hkv", [(6, 2), (8, 1)])
def test_odd_and_wide_groups(Hq, Hkv):
    run_and_compare(spec_for("CAUSAL_DOCUMENT", 300, Hq), 1, 300, Hq, Hkv, seed=2)


@pytest.mark.parametrize("N", [1, 2, 127, 128, 129])
def test_tiny_and_boundary_lengths(N):
    run_and_compare(MaskSpec("CAUSAL"), 1, N, 2, 1, seed=4)
    run_and_compare(MaskSpec("FULL"), 1, N, 2, 2, seed=5)


def test_fully_masked_rows():
    """Query blocks whose keep row is all zero: O = 0, LSE = -inf, dQ = 0."""
    N, Hq, bs = 384, 2, 64
    nb = N // bs
    keep = np.ones((Hq, nb, nb), dtype=bool)
    keep[:, 2, :] = False      # rows 128..191: nothing allowed (inside a partial tile row)
    keep[0, 4:6, :] = False    # head 0, rows 256..383: an entire query tile with no key
    spec = MaskSpec("UNIFORM_BLOCK", {"block": bs, "keep": keep})
    out, (dQ, dK, dV, O, LSE) = run_and_compare(spec, 1, N, Hq, 1, seed=6)
    o = out["o"].float().cpu().numpy()
    dq = out["dq"].float().cpu().numpy()
    assert (o[0, 128:192] == 0).all() and (dq[0, 128:192] == 0).all()
    assert (o[0, 256:, 0] == 0).all() and (dq[0, 256:, 0] == 0).all()
    assert np.isneginf(out["lse"].cpu().numpy()[0, 0, 256:]).all()


def test_key_tile_seen_by_no_query():
    """A key tile no query attends gets dK = dV = 0 (written, not left stale)."""
    N, Hq = 384, 2
    nb = 3
    keep = np.ones((Hq, nb, nb), dtype=bool)
    keep[:, :, 1] = False
    spec = MaskSpec("UNIFORM_BLOCK", {"block": 128, "keep": keep})
    x = qkv(1, N, Hq, 1, 128, seed=8)
    dev = {k: t.cuda() for k, t in x.items()}
    mask = lc.DeviceMask(spec, N, Hq)
    shape = lc.make_shape(dev["q"], dev["k"], dev["v"])
    meta = lc.lcattn_mask_compile(shape, mask)
    o, lse = lc.lcattn_fwd(dev["q"], dev["k"], dev["v"], mask, meta)
    dk = torch.full_like(dev["k"], 7.0)
    dv = torch.full_like(dev["v"], 7.0)
    lc.lcattn_bwd(dev["q"], dev["k"], dev["v"], o, dev["do"], lse, mask, meta, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert (dk[0, 128:256] == 0).all() and (dv[0, 128:256] == 0).all()


def test_tile_lists_consistent_with_classes():
    N, Hq = 1000, 2
    spec = spec_for("GLOBAL_SLIDING", N, Hq)
    x = qkv(1, N, Hq, 1, 128, seed=0, with_do=False)
    dev = {k: t.cuda() for k, t in x.items()}
    mask = lc.DeviceMask(spec, N, Hq)
    shape = lc.make_shape(dev["q"], dev["k"], dev["v"])
    meta = lc.lcattn_mask_compile(shape, mask)
    cls = lc.tile_classes(meta, shape, mask).cpu().numpy()[0, 0]
    fc, fl, fo, bc, bl, bo = (t.cpu().numpy() for t in lc.tile_lists(meta, shape, mask))
    nq, nk = cls.shape
    for qt in range(nq):
        want = [(kt << 1) | int(cls[qt, kt] == 2) for kt in range(nk) if cls[qt, kt] != 0]
        assert fc[0, qt] == len(want) and list(fl[0, qt, :len(want)]) == want
    for kt in range(nk):
        want = [(qt << 1) | int(cls[qt, kt] == 2) for qt in range(nq) if cls[qt, kt] != 0]
        assert bc[0, kt] == len(want) and list(bl[0, kt, :len(want)]) == want
    assert sorted(fo[0]) == list(range(nq)) and sorted(bo[0]) == list(range(nk))
    assert all(fc[0, fo[0, i]] >= fc[0, fo[0, i + 1]] for i in range(nq - 1))
    assert all(bc[0, bo[0, i]] >= bc[0, bo[0, i + 1]] for i in range(nk - 1))


def test_bad_block_offsets_reported_on_device():
    N, Hq = 256, 1
    spec = MaskSpec("VARIABLE_BLOCK", {"q_block_lens": [100, 156], "k_block_lens": [128, 128],
                                       "keep": np.ones((1, 2, 2), bool)})
    mask = lc.DeviceMask(spec, N, Hq)
    mask.q_offs.copy_(torch.tensor([0, 200, 100], dtype=torch.int32))  # not nondecreasing, wrong end
    q = torch.zeros(1, N, Hq, 128, dtype=torch.bfloat16, device="cuda")
    shape = lc.make_shape(q, q, q)
    meta = lc.lcattn_mask_compile(shape, mask)
    assert lc.lcattn_read_status(meta) == lc.LCATTN_ERR_DEVICE_MASK
    lc.lcattn_clear_status(meta)
    assert lc.lcattn_read_status(meta) == 0


def _sched_words(meta):
    torch.cuda.synchronize()
    return meta[16:32].view(torch.int64).cpu().tolist()


def test_persistent_forward_repeats_exactly():
    """The forward's CTAs take work items from a counter in the tile-meta
    scheduler words, and the last CTA to run out of work resets it.  Repeated
    calls on one compiled mask give identical bits and leave the words at zero;
    with more items than CTAs (256 here: 8 query tiles x 32 head pairs) every
    query tile is still covered, which the sampled oracle rows check."""
    N, Hq, Hkv = 1000, 64, 8
    spec = spec_for("CAUSAL_DOCUMENT", N, Hq, seed=3)
    x = qkv(1, N, Hq, Hkv, 128, seed=11, with_do=False)
    dev = {k: t.cuda() for k, t in x.items()}
    mask = lc.DeviceMask(spec, N, Hq)
    shape = lc.make_shape(dev["q"], dev["k"], dev["v"])
    meta = lc.lcattn_mask_compile(shape, mask)
    assert _sched_words(meta) == [0, 0]
    outs = []
    for _ in range(3):
        o, lse = lc.lcattn_fwd(dev["q"], dev["k"], dev["v"], mask, meta)
        assert _sched_words(meta) == [0, 0]
        outs.append((o.clone(), lse.clone()))
    assert lc.lcattn_read_status(meta) == 0
    for o, lse in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(lse, outs[0][1])
    q, k, v = (x[n].double().numpy() for n in ("q", "k", "v"))
    scale = 1.0 / math.sqrt(128)
    rows = np.array([0, 127, 128, 500, 871, 999])
    o, lse = outs[0]
    for h in (0, 1, 37, 63):
        ro, rl = oracle.attention_fwd_rows(q, k, v, spec, scale, 0, h, rows)
        got = o[0, rows, h].double().cpu().numpy()
        assert np.abs(got - ro).max() <= O_MAXABS
        assert np.abs(lse[0, h, rows].double().cpu().numpy() - rl).max() <= LSE_MAXABS


@pytest.mark.parametrize("case", ["mha_window", "block_sparse_empty_units", "gqa_hd64"])
def test_backward_many_units(case):
    """More dK/dV units than SMs (several waves of CTAs), at 2048 rows: every
    gradient matches the oracle, and repeated calls give identical dK and dV
    bits (each comes out of one unit, or a fixed-order sum of head shares).
    The block-sparse case has key tiles that no query tile of a head reaches
    (empty units, whose dK and dV rows are written as zeros); the head-dim-64
    case splits units over head shares."""
    D = 128
    if case == "mha_window":
        N, Hq, Hkv = 2048, 20, 20
        spec = MaskSpec("CAUSAL_SLIDING_WINDOW", {"window": 700})
    elif case == "block_sparse_empty_units":
        N, Hq, Hkv = 2048, 16, 16
        nb = N // 128
        keep = block_keep(Hq, nb, nb, 0.08, seed=4, force_diagonal=False)
        assert (~keep.any(axis=1)).any()  # some (head, key block) sees no query block
        spec = MaskSpec("UNIFORM_BLOCK", {"block": 128, "keep": keep})
    else:
        N, Hq, Hkv, D = 2048, 32, 16, 64
        spec = MaskSpec("CAUSAL")
    assert (N // 128) * Hkv > 152  # more units than SMs, before any head-share split
    x = qkv(1, N, Hq, Hkv, D, seed=21)
    dev = {k: t.cuda() for k, t in x.items()}
    out = lc.attention(dev["q"], dev["k"], dev["v"], spec, d_o=dev["do"])
    meta = out["tile_meta"]
    assert lc.lcattn_read_status(meta) == 0
    f64 = {k: t.double().numpy() for k, t in x.items()}
    dQ, dK, dV, O, LSE = oracle.attention_bwd(f64["q"], f64["k"], f64["v"], f64["do"], spec, 1.0 / math.sqrt(D))
    for name, ref in (("dq", dQ), ("dk", dK), ("dv", dV)):
        g = out[name].double().cpu().numpy()
        assert np.isfinite(g).all(), name
        assert relf(g, ref) <= G_RELF, (name, relf(g, ref))
    first = (out["dk"].clone(), out["dv"].clone())
    for _ in range(3):
        dq, dk, dv = lc.lcattn_bwd(dev["q"], dev["k"], dev["v"], out["o"], dev["do"], out["lse"],
                                   out["mask"], meta)
        assert lc.lcattn_read_status(meta) == 0
        assert torch.equal(dk, first[0]) and torch.equal(dv, first[1])
        assert relf(dq.double().cpu().numpy(), dQ) <= G_RELF


@pytest.mark.parametrize("case", ["block_sparse_gqa", "mha_many_items"])
def test_forward_one_head_items_repeat(case):
    """Work items that carry one query head run S one tile ahead of PV with S
    double-buffered.  A synchronisation slip there shows as intermittent wrong
    O rows, so the forward is repeated and every run checked against the
    oracle: a 392-row block-sparse GQA case (whose item's first tile leaves some
    rows empty), and an MHA case with more items than CTAs (item boundaries)."""
    if case == "block_sparse_gqa":
        N, Hq, Hkv = 392, 4, 2
        spec = spec_for("UNIFORM_BLOCK", N, Hq)
    else:
        N, Hq, Hkv = 2048, 20, 20
        spec = MaskSpec("CAUSAL_SLIDING_WINDOW", {"window": 700})
    x = qkv(1, N, Hq, Hkv, 128, seed=9, with_do=False)
    dev = {k: t.cuda() for k, t in x.items()}
    f64 = {k: t.double().numpy() for k, t in x.items()}
    O, LSE = oracle.attention_fwd(f64["q"], f64["k"], f64["v"], spec, 1.0 / math.sqrt(128))
    mask = lc.DeviceMask(spec, N, Hq)
    shape = lc.make_shape(dev["q"], dev["k"], dev["v"])
    meta = lc.lcattn_mask_compile(shape, mask)
    for rep in range(8):
        o, lse = lc.lcattn_fwd(dev["q"], dev["k"], dev["v"], mask, meta)
        assert lc.lcattn_read_status(meta) == 0
        err = np.abs(o.double().cpu().numpy() - O)
        assert err.max() <= O_MAXABS, (rep, err.max(), np.argwhere(err > O_MAXABS)[:4])
        fin = np.isfinite(LSE)
        assert np.abs(lse.double().cpu().numpy()[fin] - LSE[fin]).max() <= LSE_MAXABS
