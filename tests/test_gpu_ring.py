"""Ring P2P building blocks on one GPU, through the C ABI: the shard descriptor
(lcattn_mask_shard), the LSE merge (lcattn_lse_merge), the shard backward in
accumulate mode (lcattn_bwd_accum) and the fp32 -> bf16 conversion, composed
by ``ring.emulate`` into the whole ring over ``world`` emulated devices, and
checked against the fp64 oracle of the unsplit problem at the parity
tolerances (O max-abs 2e-2 / relF 1e-2, LSE 5e-3 with -inf exact, gradients
relF 3e-2).  Shards are ragged (N not a multiple of the shard count or of 128),
and CAUSAL leaves whole shard pairs without an allowed key (their partial LSE
is -inf and the merge must ignore them)."""
import math

import numpy as np
import pytest
import torch

import oracle
from synthetic import MaskSpec, block_keep, qkv, segment_lengths

pytestmark = pytest.mark.gpu

lc = pytest.importorskip("long_context_masked_mask_gb300")
from long_context_masked_mask_gb300 import ring  # noqa: E402

O_MAXABS, O_RELF, G_RELF, LSE_MAXABS = 2e-2, 1e-2, 3e-2, 5e-3


def relf(g, r):
    return float(np.linalg.norm(g - r) / np.linalg.norm(r))


def _spec(kind, N, Hq, seed=0):
    docs = segment_lengths(N, N // 6, N // 2, seed)
    return {
        "FULL": lambda: MaskSpec("FULL"),
        "CAUSAL": lambda: MaskSpec("CAUSAL"),
        "FULL_DOCUMENT": lambda: MaskSpec("FULL_DOCUMENT", {"doc_lens": docs}),
        "CAUSAL_DOCUMENT": lambda: MaskSpec("CAUSAL_DOCUMENT", {"doc_lens": docs}),
        "GLOBAL_SLIDING": lambda: MaskSpec("GLOBAL_SLIDING", {"global_tokens": 40, "window": 90}),
        "UNIFORM_BLOCK": lambda: MaskSpec("UNIFORM_BLOCK", {"block": 64, "keep": block_keep(Hq, -(-N // 64),
                                                                                            -(-N // 64), 0.5, seed)}),
    }[kind]()


def _check(out, x, spec, D, with_grad=True):
    f = {k: t.double().numpy() for k, t in x.items()}
    s = 1.0 / math.sqrt(D)
    dQ, dK, dV, O, LSE = oracle.attention_bwd(f["q"], f["k"], f["v"], f["do"], spec, s)
    o = out["o"].double().cpu().numpy()
    assert np.abs(o - O).max() <= O_MAXABS and relf(o, O) <= O_RELF
    lse = out["lse"].double().cpu().numpy()
    assert np.array_equal(np.isneginf(lse), np.isneginf(LSE))
    fin = np.isfinite(LSE)
    assert np.abs(lse[fin] - LSE[fin]).max() <= LSE_MAXABS
    if with_grad:
        for name, ref in (("dq", dQ), ("dk", dK), ("dv", dV)):
            got = out[name].double().cpu().numpy()
            assert relf(got, ref) <= G_RELF, (name, relf(got, ref))


@pytest.mark.parametrize("kind", ["CAUSAL", "FULL_DOCUMENT", "CAUSAL_DOCUMENT", "FULL", "GLOBAL_SLIDING",
                                  "UNIFORM_BLOCK"])
@pytest.mark.parametrize("world", [2, 3, 4])
def test_ring_emulation_matches_oracle(kind, world):
    B, N, Hq, Hkv, D = 1, 700, 4, 2, 128
    spec = _spec(kind, N, Hq)
    x = qkv(B, N, Hq, Hkv, D, seed=21 + world)
    dev = {k: t.cuda() for k, t in x.items()}
    mask = lc.DeviceMask(spec, N, Hq, B)
    out = ring.emulate(dev["q"], dev["k"], dev["v"], mask, world, d_o=dev["do"])
    torch.cuda.synchronize()
    _check(out, x, spec, D)


def test_ring_emulation_head_dim_64_and_batch_2():
    B, N, Hq, Hkv, D = 2, 520, 8, 2, 64
    spec = _spec("CAUSAL_DOCUMENT", N, Hq, seed=3)
    x = qkv(B, N, Hq, Hkv, D, seed=5)
    dev = {k: t.cuda() for k, t in x.items()}
    mask = lc.DeviceMask(spec, N, Hq, B)
    out = ring.emulate(dev["q"], dev["k"], dev["v"], mask, 3, d_o=dev["do"])
    torch.cuda.synchronize()
    _check(out, x, spec, D)


def test_ring_forward_equals_single_device_forward():
    """The merged ring O matches the one-device forward to bf16 rounding."""
    B, N, Hq, Hkv, D = 1, 1024, 8, 8, 128
    spec = MaskSpec("CAUSAL")
    x = {k: t.cuda() for k, t in qkv(B, N, Hq, Hkv, D, seed=9).items()}
    mask = lc.DeviceMask(spec, N, Hq, B)
    out = ring.emulate(x["q"], x["k"], x["v"], mask, 4)
    ref = lc.attention(x["q"], x["k"], x["v"], spec)
    torch.cuda.synchronize()
    d = (out["o"].float() - ref["o"].float()).abs().max().item()
    assert d <= 1.6e-2, d
    fin = torch.isfinite(ref["lse"])
    assert torch.equal(fin, torch.isfinite(out["lse"]))
    assert (out["lse"][fin] - ref["lse"][fin]).abs().max().item() <= 1e-4


def test_lse_merge_of_two_key_halves():
    """Two forwards over disjoint key halves, merged, give the forward over all keys;
    rows that one half leaves empty take the other half's result unchanged."""
    B, N, Hq, Hkv, D = 1, 384, 4, 4, 128
    x = {k: t.cuda() for k, t in qkv(B, N, Hq, Hkv, D, seed=13).items()}
    spec = MaskSpec("CAUSAL")
    full = lc.attention(x["q"], x["k"], x["v"], spec)
    o_acc = torch.empty(B, N, Hq, D, dtype=torch.float32, device="cuda")
    lse_acc = torch.empty(B, Hq, N, dtype=torch.float32, device="cuda")
    o_out = torch.empty_like(x["q"])
    gmask = lc.DeviceMask(spec, N, Hq, B)
    for i, (k0, k1) in enumerate(((0, 200), (200, N))):
        sm = lc.lcattn_mask_shard(gmask, B, N, N, 0, N, k0, k1 - k0)
        kk, vv = x["k"][:, k0:k1], x["v"][:, k0:k1]
        meta = lc.lcattn_mask_compile(lc.make_shape(x["q"], kk, vv), sm)
        o_p, lse_p = lc.lcattn_fwd(x["q"], kk, vv, sm, meta)
        lc.lcattn_lse_merge(o_acc, lse_acc, o_p, lse_p, o_out=o_out if i == 1 else None, first=(i == 0))
    torch.cuda.synchronize()
    assert (o_out.float() - full["o"].float()).abs().max().item() <= 1.6e-2
    assert (lse_acc - full["lse"]).abs().max().item() <= 1e-4
    # rows 0..199 see only the first half: the second half's partial is -inf there
    assert torch.equal(o_out[:, :200], full["o"][:, :200]) or \
        (o_out[:, :200].float() - full["o"][:, :200].float()).abs().max().item() <= 8e-3


def test_shard_descriptor_bits():
    """lcattn_mask_shard on column and row bounds: the shard's bounds are the
    global ones shifted and clamped, checked element by element."""
    B, N, Hq = 2, 300, 2
    spec = _spec("CAUSAL_DOCUMENT", N, Hq, seed=7)
    m = lc.DeviceMask(spec, N, Hq, B)
    q0, sq, k0, sk = 70, 110, 150, 90
    sm = lc.lcattn_mask_shard(m, B, N, N, q0, sq, k0, sk)
    torch.cuda.synchronize()
    cb = m.col_bounds.cpu().numpy().astype(np.int64)
    rb = m.row_bounds.cpu().numpy().astype(np.int64)
    assert np.array_equal(sm.col_bounds.cpu().numpy(), np.clip(cb[:, k0:k0 + sk] - q0, 0, sq))
    assert np.array_equal(sm.row_bounds.cpu().numpy(), np.clip(rb[:, q0:q0 + sq] - k0, 0, sk))
    # block-map offsets
    spec = _spec("UNIFORM_BLOCK", N, Hq)
    m = lc.DeviceMask(spec, N, Hq, B)
    sm = lc.lcattn_mask_shard(m, B, N, N, q0, sq, k0, sk)
    torch.cuda.synchronize()
    qo = m.q_offs.cpu().numpy().astype(np.int64)
    assert np.array_equal(sm.q_offs.cpu().numpy(), np.clip(qo - q0, 0, sq))
    assert np.array_equal(sm.k_offs.cpu().numpy(), np.clip(qo - k0, 0, sk))


@pytest.mark.parametrize("kind", ["CAUSAL", "CAUSAL_DOCUMENT", "UNIFORM_BLOCK"])
@pytest.mark.parametrize("world", [2, 3, 8])
def test_ring_zigzag_layout_matches_oracle(kind, world):
    """Zigzag shards (an early and a late chunk per device): every device
    computes two query chunks against the two K/V chunks it holds per round."""
    B, N, Hq, Hkv, D = 1, 700, 4, 2, 128
    spec = _spec(kind, N, Hq, seed=2)
    x = qkv(B, N, Hq, Hkv, D, seed=31 + world)
    dev = {k: t.cuda() for k, t in x.items()}
    mask = lc.DeviceMask(spec, N, Hq, B)
    out = ring.emulate(dev["q"], dev["k"], dev["v"], mask, world, d_o=dev["do"], layout="zigzag")
    torch.cuda.synchronize()
    _check(out, x, spec, D)


@pytest.mark.parametrize("kind", ["FULL", "CAUSAL_DOCUMENT"])
def test_ring_eight_devices_merge_error_stays_in_bounds(kind):
    """Eight emulated devices: every query row merges eight partial results by
    LSE (fp32 running O and LSE), and the merged O, LSE and gradients stay
    within the single-device parity bars (the pages note that Ring P2P's
    numeric error can accumulate over rounds)."""
    B, N, Hq, Hkv, D = 1, 1000, 4, 2, 128
    spec = _spec(kind, N, Hq, seed=4)
    x = qkv(B, N, Hq, Hkv, D, seed=41)
    dev = {k: t.cuda() for k, t in x.items()}
    mask = lc.DeviceMask(spec, N, Hq, B)
    out = ring.emulate(dev["q"], dev["k"], dev["v"], mask, 8, d_o=dev["do"])
    torch.cuda.synchronize()
    _check(out, x, spec, D)
