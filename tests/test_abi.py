"""The C-ABI library loads, exports every declared entry point, and validates
arguments on the host before launching anything (CPU only: no call here
reaches the GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
lc = pytest.importorskip("long_context_masked_mask_gb300")


def declared_functions():
    text = open(os.path.join(ROOT, "include", "lcattn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lcattn_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported():
    names = declared_functions()
    assert "lcattn_fwd" in names and "lcattn_bwd" in names and "lcattn_mask_compile" in names
    lib = ctypes.CDLL(lc._LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(lc.EXPORTED)


def _shape(B=1, S=256, Hq=4, Hkv=2, D=128):
    s = lc.lcattn_shape()
    s.B, s.Sq, s.Sk, s.Hq, s.Hkv, s.D = B, S, S, Hq, Hkv, D
    for name, H in (("q_stride", Hq), ("k_stride", Hkv), ("v_stride", Hkv), ("o_stride", Hq)):
        getattr(s, name)[:] = (S * H * 128, H * 128, 128)
    return s


def _colbounds_desc(ptr=0x1000):
    d = lc.lcattn_mask_desc()
    d.kind = lc.LCATTN_MASK_COLBOUNDS
    d.col_bounds = ptr
    return d


def _layout(shape, desc):
    L = lc.lcattn_tile_meta_layout()
    st = lc.library().lcattn_tile_meta_layout_of(ctypes.byref(shape), ctypes.byref(desc), ctypes.byref(L))
    return st, L


def test_layout_sizes_and_alignment():
    st, L = _layout(_shape(S=300), _colbounds_desc())
    assert st == 0
    assert (L.nQt, L.nKt, L.nH, L.B) == (3, 3, 1, 1)
    offs = [L.off_status, L.off_class, L.off_fwd_cnt, L.off_fwd_lst, L.off_fwd_ord,
            L.off_bwd_cnt, L.off_bwd_lst, L.off_bwd_ord, L.total_bytes]
    assert all(o % 256 == 0 for o in offs) and offs == sorted(offs)
    # the scheduler words sit right behind the four status words, which
    # lcattn_clear_status (given only the base pointer) relies on
    assert L.off_status == 0 and L.off_sched == 16 and L.off_sched + 16 <= L.off_class
    assert L.off_fwd_lst - L.off_fwd_cnt >= 4 * 3
    assert L.off_fwd_ord - L.off_fwd_lst >= 4 * 9
    # block maps carry one list per query head
    d = lc.lcattn_mask_desc()
    d.kind, d.block_map, d.q_block_offs, d.k_block_offs, d.nQb, d.nKb = 2, 0x1000, 0x2000, 0x3000, 3, 3
    st, L = _layout(_shape(S=300, Hq=4), d)
    assert st == 0 and L.nH == 4


@pytest.mark.parametrize("field,value,status", [
    ("D", 96, lc.LCATTN_ERR_UNSUPPORTED),
    ("D", 512, lc.LCATTN_ERR_UNSUPPORTED),
    ("Hkv", 3, lc.LCATTN_ERR_UNSUPPORTED),
    ("Sq", 0, lc.LCATTN_ERR_INVALID_ARG),
    ("B", 0, lc.LCATTN_ERR_INVALID_ARG),
])
def test_shape_validation(field, value, status):
    s = _shape()
    setattr(s, field, value)
    st, _ = _layout(s, _colbounds_desc())
    assert st == status
    assert lc.library().lcattn_tile_meta_size(ctypes.byref(s), ctypes.byref(_colbounds_desc())) == 0


@pytest.mark.parametrize("name", ["q_stride", "k_stride", "v_stride", "o_stride"])
def test_zero_batch_stride_refused_for_several_batch_entries(name):
    """A broadcast view (batch stride 0, what tensor.expand gives) cannot serve
    B > 1: outputs would overlap and the TMA and plain-load paths would read
    different rows.  With B = 1 the batch stride is never applied."""
    s = _shape(B=2)
    getattr(s, name)[0] = 0
    st, _ = _layout(s, _colbounds_desc())
    assert st == lc.LCATTN_ERR_UNSUPPORTED
    s = _shape(B=1)
    getattr(s, name)[0] = 0
    st, _ = _layout(s, _colbounds_desc())
    assert st == lc.LCATTN_OK


def test_backward_wrappers_check_gradient_layouts():
    """Both backward wrappers (workspace and no-allocation) refuse a dO whose
    strides differ from O's and gradients whose strides differ from their
    inputs', before any call into the library (CPU tensors suffice)."""
    import torch
    fused = torch.zeros(1, 64, 3 * 4, 128, dtype=torch.bfloat16)
    q, k, v = fused[:, :, 0:4], fused[:, :, 4:8], fused[:, :, 8:12]
    o = torch.zeros(1, 64, 4, 128, dtype=torch.bfloat16)
    d_o = torch.zeros(1, 64, 4, 128, dtype=torch.bfloat16)
    for fn in (lc.lcattn_bwd, lc.lcattn_bwd_noalloc):
        with pytest.raises(ValueError):
            fn(q, k, v, o, d_o.transpose(1, 2).contiguous().transpose(1, 2), None, None, None)
        with pytest.raises(ValueError):  # a dense dq for a strided q
            fn(q, k, v, o, d_o, None, None, None, dq=torch.empty(1, 64, 4, 128, dtype=torch.bfloat16))
    # Missing gradients take their inputs' strides.
    dq, dk, dv = lc._grad_buffers(q, k, v, o, d_o, None, None, None)
    assert dq.stride() == q.stride() and dk.stride() == k.stride() and dv.stride() == v.stride()


def test_stride_and_descriptor_validation():
    s = _shape()
    s.q_stride[2] = 130  # not a multiple of 8 elements
    assert _layout(s, _colbounds_desc())[0] == lc.LCATTN_ERR_UNSUPPORTED
    assert _layout(_shape(), _colbounds_desc(ptr=0))[0] == lc.LCATTN_ERR_INVALID_ARG
    d = lc.lcattn_mask_desc()
    d.kind = 7
    assert _layout(_shape(), d)[0] == lc.LCATTN_ERR_INVALID_ARG
    d.kind = lc.LCATTN_MASK_BLOCKMAP  # null block map
    assert _layout(_shape(), d)[0] == lc.LCATTN_ERR_INVALID_ARG


def test_calls_reject_bad_pointers_before_launch():
    lib = lc.library()
    s, d = _shape(), _colbounds_desc()
    st = lib.lcattn_fwd(ctypes.byref(s), None, 0x1000, 0x1000, 0x1000, ctypes.byref(d), 0.1, 0x1000, 0x1000, None)
    assert st == lc.LCATTN_ERR_INVALID_ARG
    st = lib.lcattn_fwd(ctypes.byref(s), 0x1008, 0x1000, 0x1000, 0x1000, ctypes.byref(d), 0.1, 0x1000, 0x1000, None)
    assert st == lc.LCATTN_ERR_UNSUPPORTED  # misaligned q
    st = lib.lcattn_fwd(ctypes.byref(s), 0x1000, 0x1000, 0x1000, 0x1000, ctypes.byref(d), -1.0, 0x1000, 0x1000, None)
    assert st == lc.LCATTN_ERR_INVALID_ARG  # bad scale
    st = lib.lcattn_mask_compile(ctypes.byref(s), ctypes.byref(d), 0x1000, 16, None)
    assert st == lc.LCATTN_ERR_WORKSPACE
    ws = lib.lcattn_bwd_workspace_size(ctypes.byref(s))
    # D [B][Hq][Sq] + the dQ accumulator [B][Hq][Sq][128], fp32; this shape has
    # 2 key tiles x 2 KV heads = 4 dK/dV units with GQA groups of 2, so the
    # units are split over two head shares and the fp32 dK/dV partials
    # [2][2][B][Sk][Hkv][128] follow.
    assert (s.B, s.Sq, s.Sk, s.Hq, s.Hkv) == (1, 256, 256, 4, 2)
    assert ws == 4 * 4 * 256 + 4 * 256 * 4 * 128 + 2 * 2 * 4 * 256 * 2 * 128
    st = lib.lcattn_bwd(ctypes.byref(s), *([0x1000] * 7), ctypes.byref(d), 0.1, 0x1000, 0x1000, 0x1000,
                        0x1000, ws - 1, None)
    assert st == lc.LCATTN_ERR_WORKSPACE


def test_status_strings():
    for code in range(-7, 1):
        assert lc.status_string(code) not in ("", "unknown status")
    assert lc.status_string(-99) == "unknown status"
    assert lc.library().lcattn_version() >= 100


def _select_desc(rule=1, top_k=4, top_p=0.9, causal=0, nQb=2, nKb=2, ptr=0x1000):
    d = lc.lcattn_select_desc()
    d.rule, d.top_k, d.top_p, d.causal = rule, top_k, top_p, causal
    d.q_block_offs = ptr
    d.k_block_offs = ptr
    d.nQb, d.nKb = nQb, nKb
    return d


def test_block_select_workspace_and_validation():
    lib = lc.library()
    s = _shape(B=2, S=256, Hq=4, Hkv=2)
    ws = lib.lcattn_block_select_workspace_size(ctypes.byref(s), ctypes.byref(_select_desc(nQb=3, nKb=5)))
    # fp32 block means: q_bar [2][4][3][128], k_bar [2][2][5][128], each 256-aligned
    assert ws == 4 * 128 * 2 * 4 * 3 + 4 * 128 * 2 * 2 * 5
    bad = [
        (_select_desc(rule=3), lc.LCATTN_ERR_INVALID_ARG),
        (_select_desc(top_k=-1), lc.LCATTN_ERR_INVALID_ARG),
        (_select_desc(rule=2, top_p=float("nan")), lc.LCATTN_ERR_INVALID_ARG),
        (_select_desc(rule=2, top_p=float("inf")), lc.LCATTN_ERR_INVALID_ARG),
        (_select_desc(causal=2), lc.LCATTN_ERR_INVALID_ARG),
        (_select_desc(nQb=0), lc.LCATTN_ERR_INVALID_ARG),
        (_select_desc(nKb=257), lc.LCATTN_ERR_INVALID_ARG),
        (_select_desc(ptr=0), lc.LCATTN_ERR_INVALID_ARG),
    ]
    for d, status in bad:
        assert lib.lcattn_block_select_workspace_size(ctypes.byref(s), ctypes.byref(d)) == 0
        st = lib.lcattn_block_select(ctypes.byref(s), 0x1000, 0x1000, ctypes.byref(d), 0.1, 0x1000,
                                     None, 0x1000, 1 << 30, None)
        assert st == status, (d.rule, d.top_k, d.top_p, d.causal, d.nQb, d.nKb)
    big = _shape(S=1 << 20, Hq=1, Hkv=1)
    assert lib.lcattn_block_select(ctypes.byref(big), 0x1000, 0x1000,
                                   ctypes.byref(_select_desc(nKb=lc.LCATTN_SELECT_MAX_KB + 1)), 0.1,
                                   0x1000, None, 0x1000, 1 << 40, None) == lc.LCATTN_ERR_UNSUPPORTED
    good = _select_desc()
    assert lib.lcattn_block_select(ctypes.byref(s), 0x1001, 0x1000, ctypes.byref(good), 0.1, 0x1000,
                                   None, 0x1000, 1 << 30, None) == lc.LCATTN_ERR_UNSUPPORTED
    assert lib.lcattn_block_select(ctypes.byref(s), 0x1000, 0x1000, ctypes.byref(good), 0.1, 0x1000,
                                   0x1002, 0x1000, 1 << 30, None) == lc.LCATTN_ERR_UNSUPPORTED
    assert lib.lcattn_block_select(ctypes.byref(s), 0x1000, 0x1000, ctypes.byref(good), 0.0, 0x1000,
                                   None, 0x1000, 1 << 30, None) == lc.LCATTN_ERR_INVALID_ARG
    assert lib.lcattn_block_select(ctypes.byref(s), 0x1000, 0x1000, ctypes.byref(good), 0.1, 0x1000,
                                   None, 0x1000, 16, None) == lc.LCATTN_ERR_WORKSPACE
    for stage in (0, 3):
        assert lib.lcattn_block_select_stage(stage, ctypes.byref(s), 0x1000, 0x1000, ctypes.byref(good),
                                             0.1, 0x1000, None, 0x1000, 1 << 30, None) == \
            lc.LCATTN_ERR_INVALID_ARG


def test_head_dim_64_is_accepted():
    """Head dim 64 is a supported variant (its strides must still separate rows);
    block selection takes head dim 128 only."""
    s = _shape(D=64)
    for name, H in (("q_stride", 4), ("k_stride", 2), ("v_stride", 2), ("o_stride", 4)):
        getattr(s, name)[:] = (256 * H * 64, H * 64, 64)
    st, L = _layout(s, _colbounds_desc())
    assert st == 0
    assert lc.library().lcattn_bwd_workspace_size(ctypes.byref(s)) == \
        4 * 4 * 256 + 4 * 256 * 4 * 64 + 2 * 2 * 4 * 256 * 2 * 64
    s.q_stride[2] = 32  # head stride below the head dim
    assert _layout(s, _colbounds_desc())[0] == lc.LCATTN_ERR_INVALID_ARG
    s.q_stride[2] = 64
    sel = _select_desc()
    assert lc.library().lcattn_block_select_workspace_size(ctypes.byref(s), ctypes.byref(sel)) == 0
    assert lc.library().lcattn_block_select(ctypes.byref(s), 0x1000, 0x1000, ctypes.byref(sel), 0.1, 0x1000,
                                            None, 0x1000, 1 << 30, None) == lc.LCATTN_ERR_UNSUPPORTED


def test_head_dim_256_backward_sizes_and_refusals():
    """Head dim 256: the backward's workspace counts the units twice (one CTA
    per head-dim half) when choosing head-share splits; the deterministic
    backward refuses it before touching the device."""
    s = _shape(D=256)
    for name, H in (("q_stride", 4), ("k_stride", 2), ("v_stride", 2), ("o_stride", 4)):
        getattr(s, name)[:] = (256 * H * 256, H * 256, 256)
    d = _colbounds_desc()
    st, L = _layout(s, d)
    assert st == 0
    lib = lc.library()
    # D [1][4][256] fp32 + dQ accumulator [1][4][256][256] fp32 + 2 head shares of
    # fp32 dK/dV partials [2][1][256][2][256] (2 key tiles x 2 KV heads x 2 halves = 8 units).
    assert lib.lcattn_bwd_workspace_size(ctypes.byref(s)) == 4 * 4 * 256 + 4 * 256 * 4 * 256 + 2 * 2 * 4 * 256 * 2 * 256
    assert lib.lcattn_bwd_deterministic_workspace_size(ctypes.byref(s)) == 0
    P = 0x1000
    args = (ctypes.byref(s), P, P, P, P, P, P, P, ctypes.byref(d), 0.1, P, P, P)
    assert lib.lcattn_bwd_deterministic(*args, P, 1 << 30, None) == lc.LCATTN_ERR_UNSUPPORTED
    s.D = 512
    assert _layout(s, d)[0] == lc.LCATTN_ERR_UNSUPPORTED


@pytest.mark.parametrize("B,Sq,Sk,Hq,Hkv,kind", [
    (1, 1, 1, 1, 1, "cb"), (1, 127, 4097, 4, 2, "cb"), (3, 129, 128, 6, 3, "cb"),
    (2, 1000, 300, 8, 1, "bm"), (1, 4097, 129, 4, 4, "bm"), (2, 128, 128, 2, 2, "bm"),
])
def test_layout_regions_hold_their_contents(B, Sq, Sk, Hq, Hkv, kind):
    """Every tile-metadata region is 256-byte aligned, follows the previous one,
    and has room for what it holds: a class byte per (batch, list head, query
    tile, key tile), per-list counts and orders, and full-length lists in both
    directions (a list head is one query head for block maps, else all heads)."""
    s = _shape(B=B, S=Sq, Hq=Hq, Hkv=Hkv)
    s.Sk = Sk
    for name, H in (("k_stride", Hkv), ("v_stride", Hkv)):
        getattr(s, name)[:] = (Sk * H * 128, H * 128, 128)
    if kind == "cb":
        d = _colbounds_desc()
    else:
        d = lc.lcattn_mask_desc()
        d.kind, d.block_map, d.q_block_offs, d.k_block_offs = lc.LCATTN_MASK_BLOCKMAP, 0x1000, 0x2000, 0x3000
        d.nQb, d.nKb = 1, 1
    st, L = _layout(s, d)
    assert st == 0
    nQt, nKt = -(-Sq // 128), -(-Sk // 128)
    nH = Hq if kind == "bm" else 1
    assert (L.nQt, L.nKt, L.nH, L.B) == (nQt, nKt, nH, B)
    lists = B * nH
    regions = [(L.off_status, 32), (L.off_class, lists * nQt * nKt), (L.off_fwd_cnt, 4 * lists * nQt),
               (L.off_fwd_lst, 4 * lists * nQt * nKt), (L.off_fwd_ord, 4 * lists * nQt),
               (L.off_bwd_cnt, 4 * lists * nKt), (L.off_bwd_lst, 4 * lists * nKt * nQt),
               (L.off_bwd_ord, 4 * lists * nKt)]
    for (o, n), (o_next, _) in zip(regions, regions[1:] + [(L.total_bytes, 0)]):
        assert o % 256 == 0 and o + n <= o_next
    size = lc.library().lcattn_tile_meta_size(ctypes.byref(s), ctypes.byref(d))
    assert size == L.total_bytes


def test_ring_building_blocks_validate_before_launch():
    lib = lc.library()
    d = _colbounds_desc()
    # shard outside the global problem
    st = lib.lcattn_mask_shard(ctypes.byref(d), 1, 256, 256, 200, 100, 0, 256, 0x1000, None, None, None, None)
    assert st == lc.LCATTN_ERR_INVALID_ARG
    st = lib.lcattn_mask_shard(ctypes.byref(d), 1, 256, 256, 0, 128, -1, 10, 0x1000, None, None, None, None)
    assert st == lc.LCATTN_ERR_INVALID_ARG
    st = lib.lcattn_mask_shard(ctypes.byref(d), 1, 256, 256, 0, 128, 0, 128, None, None, None, None, None)
    assert st == lc.LCATTN_ERR_INVALID_ARG  # no output buffer
    st = lib.lcattn_mask_shard(ctypes.byref(d), 1, 256, 256, 0, 128, 0, 128, 0x1000, 0x2000, None, None, None)
    assert st == lc.LCATTN_ERR_INVALID_ARG  # row bounds asked for, none given
    s = _shape()
    st = lib.lcattn_lse_merge(ctypes.byref(s), 0x1000, 0x1000, 0x1000, 0x1000, None, None, 2, None)
    assert st == lc.LCATTN_ERR_INVALID_ARG
    st = lib.lcattn_lse_merge(ctypes.byref(s), 0x1008, 0x1000, 0x1000, 0x1000, None, None, 0, None)
    assert st == lc.LCATTN_ERR_UNSUPPORTED  # misaligned accumulator
    # accumulate-mode backward: D only, and all three accumulators required
    assert lib.lcattn_bwd_accum_workspace_size(ctypes.byref(s)) == 4 * 4 * 256
    st = lib.lcattn_bwd_accum(ctypes.byref(s), *([0x1000] * 7), ctypes.byref(d), 0.1, 0x1000, None, 0x1000,
                              0x1000, 4096, None)
    assert st == lc.LCATTN_ERR_INVALID_ARG
    st = lib.lcattn_bwd_accum(ctypes.byref(s), *([0x1000] * 7), ctypes.byref(d), 0.1, 0x1000, 0x1000, 0x1000,
                              0x1000, 4 * 4 * 256 - 1, None)
    assert st == lc.LCATTN_ERR_WORKSPACE
    st3 = (ctypes.c_int64 * 3)(256 * 4 * 128, 4 * 128, 128)
    assert lib.lcattn_f32_to_bf16(0x1000, 0x1000, 1, 256, 4, 96, st3, None) == lc.LCATTN_ERR_UNSUPPORTED
    bad = (ctypes.c_int64 * 3)(256 * 4 * 128, 4 * 128, 100)
    assert lib.lcattn_f32_to_bf16(0x1000, 0x1000, 1, 256, 4, 128, bad, None) == lc.LCATTN_ERR_UNSUPPORTED
