"""GB300-native fused masked attention (forward and backward), bf16, head dim 128 or 64.

Python binding of the C-ABI library ``liblcattn.so`` (declared in
``include/lcattn.h``).  This module only marshals arguments: every step of the
attention path (mask compilation, forward, backward) runs in the library's CUDA
kernels.  PyTorch provides device memory and the current stream.

The functions carry the C names:

* :func:`lcattn_mask_compile` -- descriptor -> tile classes and tile lists
* :func:`lcattn_fwd` -- O and LSE
* :func:`lcattn_fwd_ws` -- the same, split over the key side for short query sides
* :func:`lcattn_bwd` -- dQ, dK, dV
* :func:`lcattn_read_status` -- device status words (bounded-wait expiry etc.)
* :func:`lcattn_block_select` -- TopK / TopP block map from pooled Q K^T

plus :class:`DeviceMask`, which uploads a host-built mask descriptor
(see :mod:`.masks`).

There is no fallback: importing this module fails when the library is missing,
and every call fails when there is no CUDA device.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Tuple

import numpy as np
import torch

from . import masks

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "liblcattn.so")

LCATTN_OK = 0
LCATTN_ERR_INVALID_ARG = -1
LCATTN_ERR_UNSUPPORTED = -2
LCATTN_ERR_WORKSPACE = -3
LCATTN_ERR_CUDA = -4
LCATTN_ERR_DEVICE_TIMEOUT = -5
LCATTN_ERR_DEVICE_MASK = -6
LCATTN_ERR_SCRATCH_LIMIT = -7
LCATTN_NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024
LCATTN_MASK_COLBOUNDS = 1
LCATTN_MASK_BLOCKMAP = 2
LCATTN_TILE_EMPTY, LCATTN_TILE_FULL, LCATTN_TILE_PARTIAL = 0, 1, 2
LCATTN_SELECT_TOPK, LCATTN_SELECT_TOPP = 1, 2
LCATTN_SELECT_MAX_KB = 16384
BLOCK_M = BLOCK_N = 128

# Every entry point include/lcattn.h declares.
EXPORTED = (
    "lcattn_tile_meta_layout_of", "lcattn_tile_meta_size", "lcattn_mask_compile", "lcattn_fwd",
    "lcattn_bwd_workspace_size", "lcattn_bwd", "lcattn_bwd_stage", "lcattn_read_status", "lcattn_clear_status",
    "lcattn_status_string", "lcattn_version", "lcattn_bwd_noalloc", "lcattn_selftest_wait_timeout",
    "lcattn_block_select_workspace_size", "lcattn_block_select", "lcattn_block_select_stage",
    "lcattn_fwd_workspace_size", "lcattn_fwd_ws",
    "lcattn_mask_shard", "lcattn_lse_merge", "lcattn_bwd_accum_workspace_size", "lcattn_bwd_accum",
    "lcattn_f32_to_bf16", "lcattn_bwd_deterministic_workspace_size", "lcattn_bwd_deterministic",
    "lcattn_fwd_fp8_workspace_size", "lcattn_fwd_fp8", "lcattn_fp8_vt_size", "lcattn_fp8_transpose_v",
    "lcattn_fwd_fp8_vt_workspace_size", "lcattn_fwd_fp8_vt",
)


class lcattn_shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("Sq", ctypes.c_int64), ("Sk", ctypes.c_int64),
                ("Hq", ctypes.c_int64), ("Hkv", ctypes.c_int64), ("D", ctypes.c_int64),
                ("q_stride", ctypes.c_int64 * 3), ("k_stride", ctypes.c_int64 * 3),
                ("v_stride", ctypes.c_int64 * 3), ("o_stride", ctypes.c_int64 * 3)]


class lcattn_mask_desc(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("col_bounds", ctypes.c_void_p),
                ("block_map", ctypes.c_void_p), ("q_block_offs", ctypes.c_void_p),
                ("k_block_offs", ctypes.c_void_p), ("nQb", ctypes.c_int32), ("nKb", ctypes.c_int32),
                ("row_bounds", ctypes.c_void_p)]


class lcattn_select_desc(ctypes.Structure):
    _fields_ = [("rule", ctypes.c_int32), ("top_k", ctypes.c_int32), ("top_p", ctypes.c_float),
                ("causal", ctypes.c_int32), ("q_block_offs", ctypes.c_void_p),
                ("k_block_offs", ctypes.c_void_p), ("nQb", ctypes.c_int32), ("nKb", ctypes.c_int32)]


class lcattn_tile_meta_layout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in (
        "nQt", "nKt", "nH", "B", "off_status", "off_sched", "off_class", "off_fwd_cnt", "off_fwd_lst",
        "off_fwd_ord", "off_bwd_cnt", "off_bwd_lst", "off_bwd_ord", "total_bytes")]


class LcattnError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} ({status})")
        self.status = status


def _load():
    if not os.path.exists(_LIB_PATH):
        raise ImportError(
            f"{_LIB_PATH} is missing; build it with "
            "`python long_context_masked_mask_gb300/build.py` (needs nvcc for sm_103a)")
    lib = ctypes.CDLL(_LIB_PATH)
    P = ctypes.c_void_p
    S = ctypes.POINTER(lcattn_shape)
    M = ctypes.POINTER(lcattn_mask_desc)
    SD = ctypes.POINTER(lcattn_select_desc)
    sig = {
        "lcattn_tile_meta_layout_of": (ctypes.c_int, [S, M, ctypes.POINTER(lcattn_tile_meta_layout)]),
        "lcattn_tile_meta_size": (ctypes.c_size_t, [S, M]),
        "lcattn_mask_compile": (ctypes.c_int, [S, M, P, ctypes.c_size_t, P]),
        "lcattn_fwd": (ctypes.c_int, [S, P, P, P, P, M, ctypes.c_float, P, P, P]),
        "lcattn_bwd_workspace_size": (ctypes.c_size_t, [S]),
        "lcattn_bwd": (ctypes.c_int, [S, P, P, P, P, P, P, P, M, ctypes.c_float, P, P, P, P,
                                      ctypes.c_size_t, P]),
        "lcattn_bwd_stage": (ctypes.c_int, [ctypes.c_int, S, P, P, P, P, P, P, P, M, ctypes.c_float,
                                            P, P, P, P, ctypes.c_size_t, P]),
        "lcattn_bwd_noalloc": (ctypes.c_int, [S, P, P, P, P, P, P, P, M, ctypes.c_float, P, P, P, P]),
        "lcattn_bwd_deterministic_workspace_size": (ctypes.c_size_t, [S]),
        "lcattn_fwd_fp8_workspace_size": (ctypes.c_size_t, [S]),
        "lcattn_fwd_fp8": (ctypes.c_int, [S, P, P, P, ctypes.c_float, ctypes.c_float, ctypes.c_float, P, M,
                                          ctypes.c_float, P, P, P, ctypes.c_size_t, P]),
        "lcattn_fp8_vt_size": (ctypes.c_size_t, [S]),
        "lcattn_fp8_transpose_v": (ctypes.c_int, [S, P, P, P]),
        "lcattn_fwd_fp8_vt_workspace_size": (ctypes.c_size_t, [S, M]),
        "lcattn_fwd_fp8_vt": (ctypes.c_int, [S, P, P, P, ctypes.c_float, ctypes.c_float, ctypes.c_float, P, M,
                                             ctypes.c_float, P, P, P, ctypes.c_size_t, P]),
        "lcattn_bwd_deterministic": (ctypes.c_int, [S, P, P, P, P, P, P, P, M, ctypes.c_float, P, P, P, P,
                                                    ctypes.c_size_t, P]),
        "lcattn_read_status": (ctypes.c_int, [P, P]),
        "lcattn_clear_status": (ctypes.c_int, [P, P]),
        "lcattn_selftest_wait_timeout": (ctypes.c_int, [P, P]),
        "lcattn_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "lcattn_version": (ctypes.c_int, []),
        "lcattn_fwd_workspace_size": (ctypes.c_size_t, [S, M]),
        "lcattn_fwd_ws": (ctypes.c_int, [S, P, P, P, P, M, ctypes.c_float, P, P, P, ctypes.c_size_t, P]),
        "lcattn_block_select_workspace_size": (ctypes.c_size_t, [S, SD]),
        "lcattn_block_select": (ctypes.c_int, [S, P, P, SD, ctypes.c_float, P, P, P, ctypes.c_size_t, P]),
        "lcattn_block_select_stage": (ctypes.c_int, [ctypes.c_int, S, P, P, SD, ctypes.c_float, P, P, P,
                                                     ctypes.c_size_t, P]),
        "lcattn_mask_shard": (ctypes.c_int, [M] + [ctypes.c_int64] * 7 + [P, P, P, P, P]),
        "lcattn_lse_merge": (ctypes.c_int, [S, P, P, P, P, P, ctypes.POINTER(ctypes.c_int64), ctypes.c_int, P]),
        "lcattn_bwd_accum_workspace_size": (ctypes.c_size_t, [S]),
        "lcattn_bwd_accum": (ctypes.c_int, [S, P, P, P, P, P, P, P, M, ctypes.c_float, P, P, P, P,
                                            ctypes.c_size_t, P]),
        "lcattn_f32_to_bf16": (ctypes.c_int, [P, P] + [ctypes.c_int64] * 4 + [ctypes.POINTER(ctypes.c_int64), P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()


def library():
    """The loaded ctypes library."""
    return _lib


def status_string(status: int) -> str:
    return _lib.lcattn_status_string(int(status)).decode()


def _check(status: int, what: str):
    if status != LCATTN_OK:
        raise LcattnError(status, what)


def _stream_ptr(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _bshd_strides(t: torch.Tensor):
    if t.dim() != 4 or t.stride(3) != 1:
        raise ValueError("expected a [B, S, H, 128] tensor with a contiguous last dim")
    return (t.stride(0), t.stride(1), t.stride(2))


def make_shape(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
               o: Optional[torch.Tensor] = None) -> lcattn_shape:
    """lcattn_shape from [B, S, H, D] tensors (o defaults to q's layout)."""
    B, Sq, Hq, D = q.shape
    s = lcattn_shape()
    s.B, s.Sq, s.Sk, s.Hq, s.Hkv, s.D = B, Sq, k.shape[1], Hq, k.shape[2], D
    s.q_stride[:] = _bshd_strides(q)
    s.k_stride[:] = _bshd_strides(k)
    s.v_stride[:] = _bshd_strides(v)
    s.o_stride[:] = _bshd_strides(o if o is not None else q)
    return s


class DeviceMask:
    """A mask descriptor uploaded to the device, plus the host-side facts the
    benchmark needs (allowed pair count).  Built from a mask spec with the
    host builders of :mod:`.masks`; the same descriptor serves every batch
    entry (it is replicated ``B`` times)."""

    def __init__(self, spec, N: int, Hq: int, B: int = 1, device: str = "cuda",
                 row_bounds: bool = True, Sk: Optional[int] = None):
        self.spec = spec
        self.N, self.Hq, self.B = N, Hq, B
        self.Sk = N if Sk is None else int(Sk)
        self.desc = lcattn_mask_desc()
        if spec.kind in ("UNIFORM_BLOCK", "VARIABLE_BLOCK"):
            keep, q_offs, k_offs = masks.block_map(spec, N, Hq, self.Sk)
            self.pairs_per_batch = masks.allowed_pairs_from_blocks(keep, q_offs, k_offs)
            self.block_map = torch.from_numpy(np.broadcast_to(keep, (B,) + keep.shape).copy()).to(device)
            self.q_offs = torch.from_numpy(q_offs).to(device)
            self.k_offs = torch.from_numpy(k_offs).to(device)
            self.desc.kind = LCATTN_MASK_BLOCKMAP
            self.desc.block_map = self.block_map.data_ptr()
            self.desc.q_block_offs = self.q_offs.data_ptr()
            self.desc.k_block_offs = self.k_offs.data_ptr()
            self.desc.nQb = keep.shape[1]
            self.desc.nKb = keep.shape[2]
        else:
            cb = masks.col_bounds(spec, N, self.Sk)
            self.pairs_per_batch = Hq * masks.allowed_pairs_from_bounds(cb, N)
            self.col_bounds = torch.from_numpy(np.broadcast_to(cb, (B,) + cb.shape).copy()).to(device)
            self.desc.kind = LCATTN_MASK_COLBOUNDS
            self.desc.col_bounds = self.col_bounds.data_ptr()
            if row_bounds:  # the same mask per query row, for the forward's partial tiles
                rb = masks.row_bounds(spec, N, self.Sk)
                self.row_bounds = torch.from_numpy(np.broadcast_to(rb, (B,) + rb.shape).copy()).to(device)
                self.desc.row_bounds = self.row_bounds.data_ptr()

    @classmethod
    def from_block_map(cls, block_map: torch.Tensor, q_offs: torch.Tensor, k_offs: torch.Tensor):
        """Block-map descriptor over device tensors the caller keeps alive: a uint8
        map [B, Hq, nQb, nKb] (for example from :func:`lcattn_block_select`) and
        int32 block offsets [nQb + 1], [nKb + 1]."""
        if block_map.dtype != torch.uint8 or block_map.dim() != 4 or not block_map.is_contiguous():
            raise ValueError("block_map must be a contiguous uint8 [B, Hq, nQb, nKb] tensor")
        if q_offs.dtype != torch.int32 or k_offs.dtype != torch.int32:
            raise ValueError("block offsets must be int32")
        self = cls.__new__(cls)
        self.spec = None
        self.B, self.Hq = block_map.shape[0], block_map.shape[1]
        self.N = None
        self.block_map, self.q_offs, self.k_offs = block_map, q_offs, k_offs
        self.desc = lcattn_mask_desc()
        self.desc.kind = LCATTN_MASK_BLOCKMAP
        self.desc.block_map = block_map.data_ptr()
        self.desc.q_block_offs = q_offs.data_ptr()
        self.desc.k_block_offs = k_offs.data_ptr()
        self.desc.nQb = block_map.shape[2]
        self.desc.nKb = block_map.shape[3]
        self.pairs_per_batch = None
        return self

    @property
    def allowed_pairs(self) -> int:
        """Allowed (query, key) pairs summed over batch and query heads."""
        if self.pairs_per_batch is None:  # a device map: count its blocks' areas
            qs = (self.q_offs[1:] - self.q_offs[:-1]).to(torch.float64)
            ks = (self.k_offs[1:] - self.k_offs[:-1]).to(torch.float64)
            area = (self.block_map.to(torch.float64) * qs[:, None] * ks[None, :]).sum()
            return int(round(float(area)))
        return self.B * self.pairs_per_batch


def tile_meta_layout(shape: lcattn_shape, mask: DeviceMask) -> lcattn_tile_meta_layout:
    L = lcattn_tile_meta_layout()
    _check(_lib.lcattn_tile_meta_layout_of(ctypes.byref(shape), ctypes.byref(mask.desc),
                                           ctypes.byref(L)), "lcattn_tile_meta_layout_of")
    return L


def lcattn_mask_compile(shape: lcattn_shape, mask: DeviceMask, tile_meta: Optional[torch.Tensor] = None,
                        stream=None, device="cuda") -> torch.Tensor:
    """Runs the mask compiler; returns the (uint8) tile-meta buffer."""
    nbytes = _lib.lcattn_tile_meta_size(ctypes.byref(shape), ctypes.byref(mask.desc))
    if nbytes == 0:
        tile_meta_layout(shape, mask)  # raises with the reason
    if tile_meta is None:
        tile_meta = torch.empty(nbytes, dtype=torch.uint8, device=device)
    _check(_lib.lcattn_mask_compile(ctypes.byref(shape), ctypes.byref(mask.desc), tile_meta.data_ptr(),
                                    tile_meta.numel(), _stream_ptr(stream)), "lcattn_mask_compile")
    return tile_meta


def lcattn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, mask: DeviceMask,
               tile_meta: torch.Tensor, scale: Optional[float] = None,
               o: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
               stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Forward: returns (O [B,Sq,Hq,128] bf16, LSE [B,Hq,Sq] fp32)."""
    B, Sq, Hq, D = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(B, Hq, Sq, dtype=torch.float32, device=q.device)
    for t in (q, k, v, o):
        if t.dtype != torch.bfloat16:
            raise TypeError("q, k, v and o must be bf16")
    shape = make_shape(q, k, v, o)
    _check(_lib.lcattn_fwd(ctypes.byref(shape), q.data_ptr(), k.data_ptr(), v.data_ptr(),
                           tile_meta.data_ptr(), ctypes.byref(mask.desc), float(scale), o.data_ptr(),
                           lse.data_ptr(), _stream_ptr(stream)), "lcattn_fwd")
    return o, lse


def lcattn_fwd_fp8(q8: torch.Tensor, k8: torch.Tensor, v8: torch.Tensor, q_scale: float, k_scale: float,
                   v_scale: float, mask: DeviceMask, tile_meta: torch.Tensor, scale: Optional[float] = None,
                   o: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                   workspace: Optional[torch.Tensor] = None, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """FP8 forward (lcattn_fwd_fp8): q8, k8, v8 are uint8 tensors of e4m3 codes,
    [B, S, H, 128], with per-tensor descale factors.  Returns (O bf16, LSE fp32)."""
    for t in (q8, k8, v8):
        if t.dtype != torch.uint8:
            raise TypeError("q8, k8 and v8 must hold e4m3 codes as uint8")
    B, Sq, Hq, D = q8.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if o is None:
        o = torch.empty(B, Sq, Hq, D, dtype=torch.bfloat16, device=q8.device)
    if lse is None:
        lse = torch.empty(B, Hq, Sq, dtype=torch.float32, device=q8.device)
    shape = make_shape(q8, k8, v8, o)
    nbytes = int(_lib.lcattn_fwd_fp8_workspace_size(ctypes.byref(shape)))
    if nbytes == 0:
        raise LcattnError(LCATTN_ERR_UNSUPPORTED, "lcattn_fwd_fp8_workspace_size")
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q8.device)
    _check(_lib.lcattn_fwd_fp8(ctypes.byref(shape), q8.data_ptr(), k8.data_ptr(), v8.data_ptr(), float(q_scale),
                               float(k_scale), float(v_scale), tile_meta.data_ptr(), ctypes.byref(mask.desc),
                               float(scale), o.data_ptr(), lse.data_ptr(), workspace.data_ptr(), workspace.numel(),
                               _stream_ptr(stream)), "lcattn_fwd_fp8")
    return o, lse


def lcattn_fp8_transpose_v(v8: torch.Tensor, k8: torch.Tensor, q8: torch.Tensor, vt: Optional[torch.Tensor] = None,
                           stream=None) -> torch.Tensor:
    """V^T of the e4m3 codes v8 [B, Sk, Hkv, 128] (lcattn_fp8_transpose_v): a
    uint8 tensor [B, Hkv, 128, Skp], Skp = Sk rounded up to 16.  q8 and k8 give
    the problem's shape (they are not read)."""
    shape = make_shape(q8, k8, v8)
    nbytes = int(_lib.lcattn_fp8_vt_size(ctypes.byref(shape)))
    if nbytes == 0:
        raise LcattnError(LCATTN_ERR_UNSUPPORTED, "lcattn_fp8_vt_size")
    B, Sk, Hkv, _ = v8.shape
    skp = -(-Sk // 16) * 16
    if vt is None:
        vt = torch.empty(B, Hkv, 128, skp, dtype=torch.uint8, device=v8.device)
    if vt.numel() < B * Hkv * 128 * skp or not vt.is_contiguous():
        raise ValueError("vt must be a contiguous uint8 tensor of B * Hkv * 128 * Skp elements")
    _check(_lib.lcattn_fp8_transpose_v(ctypes.byref(shape), v8.data_ptr(), vt.data_ptr(), _stream_ptr(stream)),
           "lcattn_fp8_transpose_v")
    return vt


def lcattn_fwd_fp8_vt(q8: torch.Tensor, k8: torch.Tensor, vt: torch.Tensor, v_shape_like: torch.Tensor,
                      q_scale: float, k_scale: float, v_scale: float, mask: DeviceMask, tile_meta: torch.Tensor,
                      scale: Optional[float] = None, o: Optional[torch.Tensor] = None,
                      lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                      stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """FP8 forward on V^T from :func:`lcattn_fp8_transpose_v` (lcattn_fwd_fp8_vt).
    ``v_shape_like`` is V (or any tensor of V's shape and strides): it gives the
    problem's shape and is not read."""
    for t in (q8, k8, vt):
        if t.dtype != torch.uint8:
            raise TypeError("q8, k8 and vt must hold e4m3 codes as uint8")
    B, Sq, Hq, D = q8.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if o is None:
        o = torch.empty(B, Sq, Hq, D, dtype=torch.bfloat16, device=q8.device)
    if lse is None:
        lse = torch.empty(B, Hq, Sq, dtype=torch.float32, device=q8.device)
    shape = make_shape(q8, k8, v_shape_like, o)
    nbytes = int(_lib.lcattn_fwd_fp8_vt_workspace_size(ctypes.byref(shape), ctypes.byref(mask.desc)))
    if workspace is None and nbytes > 0:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q8.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_len = workspace.numel() if workspace is not None else 0
    _check(_lib.lcattn_fwd_fp8_vt(ctypes.byref(shape), q8.data_ptr(), k8.data_ptr(), vt.data_ptr(), float(q_scale),
                                  float(k_scale), float(v_scale), tile_meta.data_ptr(), ctypes.byref(mask.desc),
                                  float(scale), o.data_ptr(), lse.data_ptr(), ws_ptr, ws_len, _stream_ptr(stream)),
           "lcattn_fwd_fp8_vt")
    return o, lse


def lcattn_fwd_workspace_size(shape: lcattn_shape, mask: DeviceMask) -> int:
    return int(_lib.lcattn_fwd_workspace_size(ctypes.byref(shape), ctypes.byref(mask.desc)))


def lcattn_fwd_ws(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, mask: DeviceMask,
                  tile_meta: torch.Tensor, scale: Optional[float] = None,
                  o: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                  workspace: Optional[torch.Tensor] = None, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Forward through lcattn_fwd_ws: splits the key side over SMs when the query
    side is too short to fill the GPU (decode-style rows), else lcattn_fwd."""
    B, Sq, Hq, D = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(B, Hq, Sq, dtype=torch.float32, device=q.device)
    for t in (q, k, v, o):
        if t.dtype != torch.bfloat16:
            raise TypeError("q, k, v and o must be bf16")
    shape = make_shape(q, k, v, o)
    nbytes = lcattn_fwd_workspace_size(shape, mask)
    if workspace is None and nbytes > 0:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_len = workspace.numel() if workspace is not None else 0
    _check(_lib.lcattn_fwd_ws(ctypes.byref(shape), q.data_ptr(), k.data_ptr(), v.data_ptr(),
                              tile_meta.data_ptr(), ctypes.byref(mask.desc), float(scale), o.data_ptr(),
                              lse.data_ptr(), ws_ptr, ws_len, _stream_ptr(stream)), "lcattn_fwd_ws")
    return o, lse


def _grad_buffers(q, k, v, o, d_o, dq, dk, dv):
    """The gradient outputs of a backward call.  The library reads dO through
    O's strides and writes dQ, dK, dV through Q's, K's and V's, so those
    layouts must agree; missing gradients are allocated with their inputs'
    strides (a view such as a slice of a fused QKV buffer included)."""
    if d_o.shape != o.shape or d_o.stride() != o.stride():
        raise ValueError("dO must have O's shape and strides")
    dq = torch.empty_strided(q.shape, q.stride(), dtype=q.dtype, device=q.device) if dq is None else dq
    dk = torch.empty_strided(k.shape, k.stride(), dtype=k.dtype, device=k.device) if dk is None else dk
    dv = torch.empty_strided(v.shape, v.stride(), dtype=v.dtype, device=v.device) if dv is None else dv
    for g, x in ((dq, q), (dk, k), (dv, v)):
        if g.shape != x.shape or g.stride() != x.stride():
            raise ValueError("gradients must have their inputs' shapes and strides")
        if g.dtype != torch.bfloat16:
            raise TypeError("gradients must be bf16")
    return dq, dk, dv


def lcattn_bwd_workspace_size(shape: lcattn_shape) -> int:
    return int(_lib.lcattn_bwd_workspace_size(ctypes.byref(shape)))


def lcattn_bwd(q, k, v, o, d_o, lse, mask: DeviceMask, tile_meta, scale: Optional[float] = None,
               dq=None, dk=None, dv=None, workspace=None, stream=None, stage: Optional[int] = None):
    """Backward: returns (dQ, dK, dV), bf16, laid out like q, k, v.  With
    ``stage`` in (1, 2, 3), runs only that stage (lcattn_bwd_stage)."""
    D = q.shape[3]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dq, dk, dv = _grad_buffers(q, k, v, o, d_o, dq, dk, dv)
    shape = make_shape(q, k, v, o)
    ws_bytes = lcattn_bwd_workspace_size(shape)
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    args = (ctypes.byref(shape), q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
            d_o.data_ptr(), lse.data_ptr(), tile_meta.data_ptr(), ctypes.byref(mask.desc),
            float(scale), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
            workspace.data_ptr(), workspace.numel(), _stream_ptr(stream))
    if stage is None:
        _check(_lib.lcattn_bwd(*args), "lcattn_bwd")
    else:
        _check(_lib.lcattn_bwd_stage(int(stage), *args), f"lcattn_bwd_stage({stage})")
    return dq, dk, dv


def lcattn_bwd_deterministic_workspace_size(shape: lcattn_shape) -> int:
    return int(_lib.lcattn_bwd_deterministic_workspace_size(ctypes.byref(shape)))


def lcattn_bwd_deterministic(q, k, v, o, d_o, lse, mask: DeviceMask, tile_meta, scale: Optional[float] = None,
                            dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Backward through lcattn_bwd_deterministic: the same gradients as
    :func:`lcattn_bwd` with no atomics, so repeated calls give identical bits."""
    D = q.shape[3]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dq, dk, dv = _grad_buffers(q, k, v, o, d_o, dq, dk, dv)
    shape = make_shape(q, k, v, o)
    ws_bytes = lcattn_bwd_deterministic_workspace_size(shape)
    if workspace is None:
        workspace = torch.empty(max(16, ws_bytes), dtype=torch.uint8, device=q.device)
    _check(_lib.lcattn_bwd_deterministic(ctypes.byref(shape), q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                         o.data_ptr(), d_o.data_ptr(), lse.data_ptr(), tile_meta.data_ptr(),
                                         ctypes.byref(mask.desc), float(scale), dq.data_ptr(), dk.data_ptr(),
                                         dv.data_ptr(), workspace.data_ptr(), workspace.numel(),
                                         _stream_ptr(stream)), "lcattn_bwd_deterministic")
    return dq, dk, dv


def lcattn_bwd_noalloc(q, k, v, o, d_o, lse, mask: DeviceMask, tile_meta, scale: Optional[float] = None,
                       dq=None, dk=None, dv=None, stream=None):
    """Backward through lcattn_bwd_noalloc: the library takes its scratch from a
    fixed 32 MiB device array instead of a caller workspace.  Meant for callers
    that may not allocate device memory; outputs given here are written in
    place (this wrapper allocates them only when they are omitted)."""
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[3])
    dq, dk, dv = _grad_buffers(q, k, v, o, d_o, dq, dk, dv)
    shape = make_shape(q, k, v, o)
    _check(_lib.lcattn_bwd_noalloc(ctypes.byref(shape), q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                   o.data_ptr(), d_o.data_ptr(), lse.data_ptr(), tile_meta.data_ptr(),
                                   ctypes.byref(mask.desc), float(scale), dq.data_ptr(), dk.data_ptr(),
                                   dv.data_ptr(), _stream_ptr(stream)), "lcattn_bwd_noalloc")
    return dq, dk, dv


def lcattn_mask_shard(mask: "DeviceMask", B: int, Sq: int, Sk: int, q0: int, Sq_s: int, k0: int,
                      Sk_s: int, stream=None) -> "DeviceMask":
    """Descriptor of query rows [q0, q0+Sq_s) against keys [k0, k0+Sk_s) of the
    global mask ``mask`` (lcattn_mask_shard): a :class:`DeviceMask` of the
    Sq_s x Sk_s problem, holding its own device buffers (a block map's map
    array is shared with ``mask``)."""
    dev = (mask.col_bounds if mask.desc.kind == LCATTN_MASK_COLBOUNDS else mask.block_map).device
    out = DeviceMask.__new__(DeviceMask)
    out.spec, out.N, out.Sk, out.Hq, out.B = None, Sq_s, Sk_s, mask.Hq, B
    out.pairs_per_batch = None
    out.desc = lcattn_mask_desc()
    out.desc.kind = mask.desc.kind
    col = row = qo = ko = None
    if mask.desc.kind == LCATTN_MASK_COLBOUNDS:
        out.col_bounds = col = torch.empty(B, Sk_s, 4, dtype=torch.int32, device=dev)
        out.desc.col_bounds = col.data_ptr()
        if mask.desc.row_bounds:
            out.row_bounds = row = torch.empty(B, Sq_s, 4, dtype=torch.int32, device=dev)
            out.desc.row_bounds = row.data_ptr()
    else:
        out.block_map = mask.block_map
        out.q_offs = qo = torch.empty(mask.desc.nQb + 1, dtype=torch.int32, device=dev)
        out.k_offs = ko = torch.empty(mask.desc.nKb + 1, dtype=torch.int32, device=dev)
        out.desc.block_map = mask.desc.block_map
        out.desc.q_block_offs, out.desc.k_block_offs = qo.data_ptr(), ko.data_ptr()
        out.desc.nQb, out.desc.nKb = mask.desc.nQb, mask.desc.nKb
    ptr = lambda t: t.data_ptr() if t is not None else None
    _check(_lib.lcattn_mask_shard(ctypes.byref(mask.desc), B, Sq, Sk, q0, Sq_s, k0, Sk_s, ptr(col), ptr(row),
                                  ptr(qo), ptr(ko), _stream_ptr(stream)), "lcattn_mask_shard")
    return out


def lcattn_lse_merge(o_acc: torch.Tensor, lse_acc: torch.Tensor, o_part: torch.Tensor, lse_part: torch.Tensor,
                     o_out: Optional[torch.Tensor] = None, first: bool = False, stream=None) -> None:
    """Merges a shard pair's (O, LSE) into the running fp32 (o_acc, lse_acc) of a
    query shard by log-sum-exp (lcattn_lse_merge); writes bf16 ``o_out`` too
    when given.  o_acc [B, Sq, Hq, D] fp32 contiguous, lse [B, Hq, Sq] fp32."""
    if o_acc.dtype != torch.float32 or not o_acc.is_contiguous():
        raise ValueError("o_acc must be a contiguous fp32 [B, Sq, Hq, D] tensor")
    if o_out is not None and (o_out.shape != o_part.shape or o_out.dtype != torch.bfloat16):
        raise ValueError("o_out must be bf16 with o_part's shape")
    for t in (lse_acc, lse_part):
        if t.dtype != torch.float32 or not t.is_contiguous() or t.shape != (o_acc.shape[0], o_acc.shape[2], o_acc.shape[1]):
            raise ValueError("LSE tensors must be contiguous fp32 [B, Hq, Sq]")
    shape = make_shape(o_part, o_part, o_part, o_part)
    out_st = (ctypes.c_int64 * 3)(*_bshd_strides(o_out)) if o_out is not None else None
    _check(_lib.lcattn_lse_merge(ctypes.byref(shape), o_acc.data_ptr(), lse_acc.data_ptr(), o_part.data_ptr(),
                                 lse_part.data_ptr(), o_out.data_ptr() if o_out is not None else None, out_st,
                                 1 if first else 0, _stream_ptr(stream)), "lcattn_lse_merge")


def lcattn_bwd_accum(q, k, v, o, d_o, lse, mask: "DeviceMask", tile_meta, dq_acc, dk_acc, dv_acc,
                     scale: Optional[float] = None, workspace=None, stream=None) -> None:
    """Shard backward (lcattn_bwd_accum): adds this shard pair's dQ terms into
    ``dq_acc`` [B, Sq, Hq, D] and its dK / dV terms into ``dk_acc`` / ``dv_acc``
    [B, Sk, Hkv, D] (fp32, contiguous).  ``o`` and ``lse`` are the query
    shard's final (merged) output and LSE."""
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[3])
    if d_o.shape != o.shape or d_o.stride() != o.stride():
        raise ValueError("dO must have O's shape and strides")
    for acc, x in ((dq_acc, q), (dk_acc, k), (dv_acc, v)):
        if acc.dtype != torch.float32 or not acc.is_contiguous() or acc.shape != x.shape:
            raise ValueError("accumulators must be contiguous fp32 tensors shaped like q, k, v")
    shape = make_shape(q, k, v, o)
    nbytes = int(_lib.lcattn_bwd_accum_workspace_size(ctypes.byref(shape)))
    if workspace is None:
        workspace = torch.empty(max(16, nbytes), dtype=torch.uint8, device=q.device)
    _check(_lib.lcattn_bwd_accum(ctypes.byref(shape), q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                 d_o.data_ptr(), lse.data_ptr(), tile_meta.data_ptr(), ctypes.byref(mask.desc),
                                 float(scale), dq_acc.data_ptr(), dk_acc.data_ptr(), dv_acc.data_ptr(),
                                 workspace.data_ptr(), workspace.numel(), _stream_ptr(stream)), "lcattn_bwd_accum")


def lcattn_f32_to_bf16(src: torch.Tensor, dst: torch.Tensor, stream=None) -> torch.Tensor:
    """Contiguous fp32 [B, S, H, D] -> bf16 ``dst`` of the same shape (any BSHD strides)."""
    if src.dtype != torch.float32 or not src.is_contiguous() or dst.dtype != torch.bfloat16 or src.shape != dst.shape:
        raise ValueError("src must be contiguous fp32 and dst bf16 of the same shape")
    B, S, H, D = src.shape
    st = (ctypes.c_int64 * 3)(*_bshd_strides(dst))
    _check(_lib.lcattn_f32_to_bf16(src.data_ptr(), dst.data_ptr(), B, S, H, D, st, _stream_ptr(stream)),
           "lcattn_f32_to_bf16")
    return dst


def select_desc(rule: str, q_offs: torch.Tensor, k_offs: torch.Tensor, top_k: int = 0,
                top_p: float = 0.0, causal: bool = False) -> lcattn_select_desc:
    """lcattn_select_desc for ``rule`` in ("topk", "topp") over int32 device offsets."""
    d = lcattn_select_desc()
    d.rule = {"topk": LCATTN_SELECT_TOPK, "topp": LCATTN_SELECT_TOPP}[rule]
    d.top_k = int(top_k)
    d.top_p = float(top_p)
    d.causal = 1 if causal else 0
    if q_offs.dtype != torch.int32 or k_offs.dtype != torch.int32:
        raise ValueError("block offsets must be int32")
    d.q_block_offs = q_offs.data_ptr()
    d.k_block_offs = k_offs.data_ptr()
    d.nQb = q_offs.numel() - 1
    d.nKb = k_offs.numel() - 1
    return d


def lcattn_block_select_workspace_size(q: torch.Tensor, k: torch.Tensor, sel: lcattn_select_desc) -> int:
    shape = make_shape(q, k, k, q)
    return int(_lib.lcattn_block_select_workspace_size(ctypes.byref(shape), ctypes.byref(sel)))


def lcattn_block_select(q: torch.Tensor, k: torch.Tensor, q_offs: torch.Tensor, k_offs: torch.Tensor,
                        rule: str, top_k: int = 0, top_p: float = 0.0, causal: bool = False,
                        scale: Optional[float] = None, block_map: Optional[torch.Tensor] = None,
                        scores: Optional[torch.Tensor] = None, want_scores: bool = False,
                        workspace: Optional[torch.Tensor] = None, stream=None,
                        stage: Optional[int] = None):
    """Dynamic block selection (lcattn_block_select): returns (block_map uint8
    [B, Hq, nQb, nKb], scores fp32 of the same shape or None).  With ``stage``
    in (1, 2), runs only that stage (lcattn_block_select_stage)."""
    for t in (q, k):
        if t.dtype != torch.bfloat16:
            raise TypeError("q and k must be bf16")
    B, _, Hq, D = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    sel = select_desc(rule, q_offs, k_offs, top_k, top_p, causal)
    shape = make_shape(q, k, k, q)
    if block_map is None:
        block_map = torch.empty(B, Hq, sel.nQb, sel.nKb, dtype=torch.uint8, device=q.device)
    if scores is None and want_scores:
        scores = torch.empty(B, Hq, sel.nQb, sel.nKb, dtype=torch.float32, device=q.device)
    ws_bytes = int(_lib.lcattn_block_select_workspace_size(ctypes.byref(shape), ctypes.byref(sel)))
    if ws_bytes == 0:
        raise LcattnError(LCATTN_ERR_INVALID_ARG, "lcattn_block_select_workspace_size")
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    args = (ctypes.byref(shape), q.data_ptr(), k.data_ptr(), ctypes.byref(sel), float(scale),
            block_map.data_ptr(), scores.data_ptr() if scores is not None else None,
            workspace.data_ptr(), workspace.numel(), _stream_ptr(stream))
    if stage is None:
        _check(_lib.lcattn_block_select(*args), "lcattn_block_select")
    else:
        _check(_lib.lcattn_block_select_stage(int(stage), *args), f"lcattn_block_select_stage({stage})")
    return block_map, scores


def lcattn_read_status(tile_meta: torch.Tensor, stream=None) -> int:
    """Synchronises the stream and returns the first nonzero device status word."""
    return int(_lib.lcattn_read_status(tile_meta.data_ptr(), _stream_ptr(stream)))


def lcattn_selftest_wait_timeout(tile_meta: torch.Tensor, stream=None) -> None:
    """Launches the diagnostic kernel whose bounded wait expires (~2 s) and
    records LCATTN_ERR_DEVICE_TIMEOUT in `tile_meta`'s status words."""
    _check(_lib.lcattn_selftest_wait_timeout(tile_meta.data_ptr(), _stream_ptr(stream)),
           "lcattn_selftest_wait_timeout")


def lcattn_clear_status(tile_meta: torch.Tensor, stream=None) -> None:
    _check(_lib.lcattn_clear_status(tile_meta.data_ptr(), _stream_ptr(stream)), "lcattn_clear_status")


def tile_classes(tile_meta: torch.Tensor, shape: lcattn_shape, mask: DeviceMask) -> torch.Tensor:
    """View of the class bytes [B, nH, nQt, nKt] inside a compiled tile-meta buffer."""
    L = tile_meta_layout(shape, mask)
    n = L.B * L.nH * L.nQt * L.nKt
    return tile_meta[L.off_class:L.off_class + n].view(L.B, L.nH, L.nQt, L.nKt)


def tile_lists(tile_meta: torch.Tensor, shape: lcattn_shape, mask: DeviceMask):
    """Views (fwd_cnt, fwd_lst, fwd_ord, bwd_cnt, bwd_lst, bwd_ord) of a tile-meta buffer."""
    L = tile_meta_layout(shape, mask)
    bh = L.B * L.nH

    def view(off, *dims):
        n = int(np.prod(dims)) * 4
        return tile_meta[off:off + n].view(torch.int32).view(*dims)

    return (view(L.off_fwd_cnt, bh, L.nQt), view(L.off_fwd_lst, bh, L.nQt, L.nKt),
            view(L.off_fwd_ord, bh, L.nQt), view(L.off_bwd_cnt, bh, L.nKt),
            view(L.off_bwd_lst, bh, L.nKt, L.nQt), view(L.off_bwd_ord, bh, L.nKt))


def attention(q, k, v, spec, scale=None, d_o=None, stream=None):
    """Convenience composition of the C calls: compile the mask, run the
    forward, and (when ``d_o`` is given) the backward.  Returns a dict."""
    B, N, Hq, _ = q.shape
    mask = DeviceMask(spec, N, Hq, B, device=q.device, Sk=k.shape[1])
    shape = make_shape(q, k, v)
    meta = lcattn_mask_compile(shape, mask, stream=stream, device=q.device)
    o, lse = lcattn_fwd_ws(q, k, v, mask, meta, scale, stream=stream)
    out = {"o": o, "lse": lse, "mask": mask, "tile_meta": meta}
    if d_o is not None:
        out["dq"], out["dk"], out["dv"] = lcattn_bwd(q, k, v, o, d_o, lse, mask, meta, scale, stream=stream)
    return out


class MaskedAttention(torch.autograd.Function):
    """Autograd binding of the C calls, for use inside a PyTorch training graph:
    ``MaskedAttention.apply(q, k, v, mask, tile_meta, scale)`` runs lcattn_fwd_ws
    and, on backward, lcattn_bwd.  ``mask`` is a :class:`DeviceMask` and
    ``tile_meta`` its compiled buffer (:func:`lcattn_mask_compile`), built once
    and reused across steps.  Inputs are [B, S, H, D] bf16 tensors with a
    contiguous last dim; gradients come back in the inputs' layouts."""

    @staticmethod
    def forward(ctx, q, k, v, mask, tile_meta, scale=None):
        o, lse = lcattn_fwd_ws(q, k, v, mask, tile_meta, scale)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.mask, ctx.tile_meta, ctx.scale = mask, tile_meta, scale
        return o

    @staticmethod
    def backward(ctx, d_o):
        q, k, v, o, lse = ctx.saved_tensors
        if d_o.stride() != o.stride():
            d_o = d_o.contiguous() if o.is_contiguous() else torch.empty_like(o).copy_(d_o)
        dq = torch.empty_strided(q.shape, q.stride(), dtype=q.dtype, device=q.device)
        dk = torch.empty_strided(k.shape, k.stride(), dtype=k.dtype, device=k.device)
        dv = torch.empty_strided(v.shape, v.stride(), dtype=v.dtype, device=v.device)
        lcattn_bwd(q, k, v, o, d_o, lse, ctx.mask, ctx.tile_meta, ctx.scale, dq=dq, dk=dk, dv=dv)
        return dq, dk, dv, None, None, None
