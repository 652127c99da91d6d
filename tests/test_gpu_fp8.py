"""The FP8 forward (lcattn_fwd_fp8) through the C ABI against the fp64 oracle
on the decoded E4M3 inputs (oracle.fp8_ref).

Tolerance, from the arithmetic: the logits and the row sum are exact fp32
functions of the fp8 inputs, but P enters the P V product as e4m3(16 P), with
P <= 16 (the running max moves when a row max grows by more than 4 in log2
units), which rounds each P to 3 mantissa bits, a relative error of at most
2^-4, and flushes P < 2^-14 to zero.  So:
O relative Frobenius error <= 5e-2 (the rounding errors of many P partly
cancel: a CPU model of exactly this arithmetic gave 1.7e-2 to 2.6e-2 on these
shapes), O max-abs <= 2^-4 * max|O| + 1e-2 (bf16 output rounding), LSE
max-abs <= 5e-3 with -inf exactly where the oracle has it (P's rounding does
not enter the LSE)."""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import fp8_ref
from synthetic import MaskSpec, block_keep, qkv_fp8, segment_lengths

pytestmark = pytest.mark.gpu

lc = pytest.importorskip("long_context_masked_mask_gb300")


def _spec(kind, N, Hq):
    if kind == "CAUSAL_DOCUMENT":
        return MaskSpec("CAUSAL_DOCUMENT", {"doc_lens": segment_lengths(N, N // 6, N // 2, 1)})
    if kind == "UNIFORM_BLOCK":
        nb = -(-N // 64)
        return MaskSpec("UNIFORM_BLOCK", {"block": 64, "keep": block_keep(Hq, nb, nb, 0.5, 2)})
    if kind == "VARIABLE_BLOCK":
        ql, kl = segment_lengths(N, 32, 200, 3), segment_lengths(N, 32, 200, 4)
        keep = block_keep(Hq, len(ql), len(kl), 0.5, 5, force_diagonal=False)
        keep[:, 1, :] = False  # fully masked rows
        return MaskSpec("VARIABLE_BLOCK", {"q_block_lens": ql, "k_block_lens": kl, "keep": keep})
    if kind == "GLOBAL_SLIDING":
        return MaskSpec("GLOBAL_SLIDING", {"global_tokens": 40, "window": 100})
    return MaskSpec(kind)


def _check(o, lse, O, L):
    o = o.double().cpu().numpy()
    lse = lse.double().cpu().numpy()
    relf = float(np.linalg.norm(o - O) / max(np.linalg.norm(O), 1e-30))
    assert relf <= 5e-2, relf
    assert np.abs(o - O).max() <= 2.0 ** -4 * max(1.0, np.abs(O).max()) + 1e-2
    assert np.array_equal(np.isneginf(lse), np.isneginf(L))
    fin = np.isfinite(L)
    if fin.any():
        assert np.abs(lse[fin] - L[fin]).max() <= 5e-3


@pytest.mark.parametrize("kind,B,N,Hq,Hkv", [
    ("CAUSAL", 1, 392, 4, 2), ("FULL", 1, 700, 8, 2), ("CAUSAL_DOCUMENT", 2, 520, 4, 4),
    ("GLOBAL_SLIDING", 1, 600, 4, 1), ("UNIFORM_BLOCK", 1, 400, 4, 2), ("VARIABLE_BLOCK", 1, 600, 2, 2),
    ("CAUSAL", 1, 1, 2, 1), ("FULL", 1, 129, 2, 2),
])
def test_fp8_forward_matches_oracle(kind, B, N, Hq, Hkv):
    spec = _spec(kind, N, Hq)
    x = qkv_fp8(B, N, Hq, Hkv, 128, seed=11)
    dev = {k: (t.cuda() if torch.is_tensor(t) else t) for k, t in x.items()}
    mask = lc.DeviceMask(spec, N, Hq, B)
    shape = lc.make_shape(dev["q8"], dev["k8"], dev["v8"])
    meta = lc.lcattn_mask_compile(shape, mask)
    o, lse = lc.lcattn_fwd_fp8(dev["q8"], dev["k8"], dev["v8"], x["q_scale"], x["k_scale"], x["v_scale"], mask, meta)
    torch.cuda.synchronize()
    assert lc.lcattn_read_status(meta) == 0
    O, L = fp8_ref.attention_fwd_fp8(x["q8"].numpy(), x["k8"].numpy(), x["v8"].numpy(), x["q_scale"],
                                     x["k_scale"], x["v_scale"], spec, 1.0 / math.sqrt(128))
    _check(o, lse, O, L)


def test_fp8_rectangular_and_column_bounds_only():
    """Sq != Sk (bottom-right causal, a ragged key tail) and the column-bounds path
    without row bounds, which must give the same bits as with them."""
    Sq, Sk, Hq, Hkv = 300, 777, 4, 2
    x = qkv_fp8(1, Sq, Hq, Hkv, 128, seed=13, Sk=Sk)
    dev = {k: (t.cuda() if torch.is_tensor(t) else t) for k, t in x.items()}
    spec = MaskSpec("CAUSAL")
    outs = []
    for rows in (True, False):
        mask = lc.DeviceMask(spec, Sq, Hq, 1, Sk=Sk, row_bounds=rows)
        meta = lc.lcattn_mask_compile(lc.make_shape(dev["q8"], dev["k8"], dev["v8"]), mask)
        outs.append(lc.lcattn_fwd_fp8(dev["q8"], dev["k8"], dev["v8"], x["q_scale"], x["k_scale"], x["v_scale"],
                                      mask, meta))
    torch.cuda.synchronize()
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    O, L = fp8_ref.attention_fwd_fp8(x["q8"].numpy(), x["k8"].numpy(), x["v8"].numpy(), x["q_scale"],
                                     x["k_scale"], x["v_scale"], spec, 1.0 / math.sqrt(128))
    _check(outs[0][0], outs[0][1], O, L)


def test_fp8_refuses_other_head_dims_and_strides():
    x = torch.zeros(1, 64, 2, 64, dtype=torch.uint8, device="cuda")
    m = lc.DeviceMask(MaskSpec("FULL"), 64, 2, 1)
    meta = lc.lcattn_mask_compile(lc.make_shape(x, x, x), m)
    with pytest.raises(lc.LcattnError):
        lc.lcattn_fwd_fp8(x, x, x, 1.0, 1.0, 1.0, m, meta)


@pytest.mark.parametrize("kind", ["FULL", "CAUSAL"])
def test_fp8_forward_full_size_sampled_rows(kind):
    """The dense 8K workload (B=1, N=8192, GQA 64:8) in the launch the bench
    times: sampled rows of three query heads against the oracle's rows."""
    N, Hq, Hkv = 8192, 64, 8
    x = qkv_fp8(1, N, Hq, Hkv, 128, seed=17)
    dev = {k: (t.cuda() if torch.is_tensor(t) else t) for k, t in x.items()}
    spec = MaskSpec(kind)
    mask = lc.DeviceMask(spec, N, Hq, 1)
    meta = lc.lcattn_mask_compile(lc.make_shape(dev["q8"], dev["k8"], dev["v8"]), mask)
    o, lse = lc.lcattn_fwd_fp8(dev["q8"], dev["k8"], dev["v8"], x["q_scale"], x["k_scale"], x["v_scale"], mask, meta)
    torch.cuda.synchronize()
    assert lc.lcattn_read_status(meta) == 0
    q = fp8_ref.e4m3_decode(x["q8"].numpy()) * x["q_scale"]
    k = fp8_ref.e4m3_decode(x["k8"].numpy()) * x["k_scale"]
    v = fp8_ref.e4m3_decode(x["v8"].numpy()) * x["v_scale"]
    rng = np.random.default_rng(3)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, N - 129, N - 1], rng.integers(0, N, 42)]))
    ri = torch.as_tensor(rows, device=o.device)
    for h in (0, 9, 63):
        O, L = oracle.attention_fwd_rows(q, k, v, spec, 1.0 / math.sqrt(128), 0, h, rows)
        _check(o[0, ri, h], lse[0, h, ri], O, L)


def test_fp8_views_of_a_fused_qkv_buffer():
    """Q, K and V as views of one fused [B, S, Hq + 2 Hkv, 128] e4m3 buffer (row
    strides of (Hq + 2 Hkv) x 128 bytes) give the same bits as contiguous copies."""
    B, N, Hq, Hkv = 2, 333, 4, 2
    x = qkv_fp8(B, N, Hq, Hkv, 128, seed=19)
    fused = torch.cat([x["q8"], x["k8"], x["v8"]], dim=2).cuda()
    q, k, v = fused[:, :, :Hq], fused[:, :, Hq:Hq + Hkv], fused[:, :, Hq + Hkv:]
    assert q.stride(1) == (Hq + 2 * Hkv) * 128
    spec = MaskSpec("CAUSAL")
    mask = lc.DeviceMask(spec, N, Hq, B)
    meta = lc.lcattn_mask_compile(lc.make_shape(q, k, v), mask)
    o_view, lse_view = lc.lcattn_fwd_fp8(q, k, v, x["q_scale"], x["k_scale"], x["v_scale"], mask, meta)
    qc, kc, vc = q.contiguous(), k.contiguous(), v.contiguous()
    meta_c = lc.lcattn_mask_compile(lc.make_shape(qc, kc, vc), mask)
    o_c, lse_c = lc.lcattn_fwd_fp8(qc, kc, vc, x["q_scale"], x["k_scale"], x["v_scale"], mask, meta_c)
    torch.cuda.synchronize()
    assert lc.lcattn_read_status(meta) == 0 and lc.lcattn_read_status(meta_c) == 0
    assert torch.equal(o_view, o_c) and torch.equal(lse_view, lse_c)
    O, L = fp8_ref.attention_fwd_fp8(x["q8"].numpy(), x["k8"].numpy(), x["v8"].numpy(), x["q_scale"],
                                     x["k_scale"], x["v_scale"], spec, 1.0 / math.sqrt(128))
    _check(o_view, lse_view, O, L)


@pytest.mark.parametrize("B,Sq,Sk,Hq,Hkv,kind", [(2, 1, 3000, 16, 2, "CAUSAL"), (1, 40, 2500, 4, 4, "FULL"),
                                                 (3, 16, 1100, 8, 1, "CAUSAL_SLIDING_WINDOW")])
def test_fp8_split_kv_decode_rows(B, Sq, Sk, Hq, Hkv, kind):
    """Short query sides take the e4m3 split-KV path (checked: its workspace is
    non-zero): lcattn_fwd_fp8 and lcattn_fwd_fp8_vt on a V^T made once by
    lcattn_fp8_transpose_v give the same bits, and match the oracle."""
    spec = MaskSpec(kind, {"window": Sk // 3} if "WINDOW" in kind else {})
    x = qkv_fp8(B, Sq, Hq, Hkv, 128, seed=23, Sk=Sk)
    dev = {k: (t.cuda() if torch.is_tensor(t) else t) for k, t in x.items()}
    mask = lc.DeviceMask(spec, Sq, Hq, B, Sk=Sk)
    shape = lc.make_shape(dev["q8"], dev["k8"], dev["v8"])
    assert lc.library().lcattn_fwd_fp8_vt_workspace_size(lc.ctypes.byref(shape), lc.ctypes.byref(mask.desc)) > 0
    meta = lc.lcattn_mask_compile(shape, mask)
    o1, l1 = lc.lcattn_fwd_fp8(dev["q8"], dev["k8"], dev["v8"], x["q_scale"], x["k_scale"], x["v_scale"], mask, meta)
    vt = lc.lcattn_fp8_transpose_v(dev["v8"], dev["k8"], dev["q8"])
    o2, l2 = lc.lcattn_fwd_fp8_vt(dev["q8"], dev["k8"], vt, dev["v8"], x["q_scale"], x["k_scale"], x["v_scale"],
                                  mask, meta)
    torch.cuda.synchronize()
    assert lc.lcattn_read_status(meta) == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    O, L = fp8_ref.attention_fwd_fp8(x["q8"].numpy(), x["k8"].numpy(), x["v8"].numpy(), x["q_scale"],
                                     x["k_scale"], x["v_scale"], spec, 1.0 / math.sqrt(128))
    _check(o1, l1, O, L)


def test_fp8_vt_entry_regular_path_without_workspace():
    """A square problem takes the persistent kernel: lcattn_fwd_fp8_vt needs no
    workspace there, and its V^T input gives the bits of lcattn_fwd_fp8."""
    B, N, Hq, Hkv = 1, 520, 4, 2
    x = qkv_fp8(B, N, Hq, Hkv, 128, seed=29)
    dev = {k: (t.cuda() if torch.is_tensor(t) else t) for k, t in x.items()}
    spec = MaskSpec("CAUSAL_DOCUMENT", {"doc_lens": segment_lengths(N, 60, 300, 2)})
    mask = lc.DeviceMask(spec, N, Hq, B)
    shape = lc.make_shape(dev["q8"], dev["k8"], dev["v8"])
    assert lc.library().lcattn_fwd_fp8_vt_workspace_size(lc.ctypes.byref(shape), lc.ctypes.byref(mask.desc)) == 0
    meta = lc.lcattn_mask_compile(shape, mask)
    o1, l1 = lc.lcattn_fwd_fp8(dev["q8"], dev["k8"], dev["v8"], x["q_scale"], x["k_scale"], x["v_scale"], mask, meta)
    vt = lc.lcattn_fp8_transpose_v(dev["v8"], dev["k8"], dev["q8"])
    o2, l2 = lc.lcattn_fwd_fp8_vt(dev["q8"], dev["k8"], vt, dev["v8"], x["q_scale"], x["k_scale"], x["v_scale"],
                                  mask, meta)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    # V^T itself: key-contiguous rows, zero padding up to a multiple of 16 keys.
    v = dev["v8"]
    assert torch.equal(vt[:, :, :, :N], v.permute(0, 2, 3, 1))
    assert (vt[:, :, :, N:] == 0).all()
