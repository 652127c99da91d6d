"""Context parallelism by Ring P2P over the library's per-device building blocks.

The pages' distributed half ("Long-Context Attention Benchmark", xllm-io blog
review, section "分布式注意力机制": Ring P2P exchanges K/V in several
point-to-point rounds and overlaps them with the computation; section
"分布式性能": it does best on FULL masks and fluctuates on DOCUMENT masks)
splits the sequence over ``world`` devices.  Device ``r`` holds query shard
``r`` and K/V shard ``r``.  In round ``t`` it holds K/V shard
``(r - t) mod world``: it computes its query shard against it
(:func:`forward_round`), merges the partial result into its running one by
log-sum-exp, and hands the K/V shard on to device ``r + 1`` (:func:`hop`).
The backward walks the same ring (:func:`backward_round`): dQ terms add up
locally, and each K/V shard's dK/dV accumulators travel with it and arrive
back at the owner after ``world`` hops.

Every computation runs in the library's CUDA kernels through the C ABI
(lcattn_mask_shard, lcattn_mask_compile, lcattn_fwd, lcattn_lse_merge,
lcattn_bwd_accum, lcattn_f32_to_bf16).  :func:`hop` moves tensors with
``torch.distributed`` point-to-point calls and is independent of the compute.
:func:`emulate` runs every device's rounds in order on one GPU, with the
hops replaced by handing the same tensors over, which is how the building
blocks are checked against the single-device attention.
"""
from __future__ import annotations

import math
from typing import Dict, List, Optional, Sequence

import torch

from . import (DeviceMask, lcattn_bwd_accum, lcattn_f32_to_bf16, lcattn_fwd, lcattn_lse_merge,
               lcattn_mask_compile, lcattn_mask_shard, make_shape)


def shard_starts(N: int, world: int) -> List[int]:
    """Boundaries of ``world`` contiguous shards of a length-N sequence
    (shard r is [starts[r], starts[r+1]))."""
    if world < 1 or world > N:
        raise ValueError("need 1 <= world <= N")
    return [r * N // world for r in range(world + 1)]


def kv_shard_at(rank: int, step: int, world: int) -> int:
    """The K/V shard device ``rank`` holds in round ``step``."""
    return (rank - step) % world


def schedule(rank: int, world: int) -> List[int]:
    """K/V shards device ``rank`` computes against, in round order."""
    return [kv_shard_at(rank, t, world) for t in range(world)]


def hop(tensors: Sequence[torch.Tensor], rank: int, world: int, group=None) -> List[torch.Tensor]:
    """One ring hop: sends ``tensors`` to device ``rank + 1`` and returns the
    tensors received from device ``rank - 1`` (same shapes and dtypes), with
    ``torch.distributed`` point-to-point operations issued as one batch."""
    import torch.distributed as dist
    if world == 1:
        return list(tensors)
    nxt, prv = (rank + 1) % world, (rank - 1) % world
    recv = [torch.empty_like(t) for t in tensors]
    ops = [dist.P2POp(dist.isend, t, nxt, group) for t in tensors]
    ops += [dist.P2POp(dist.irecv, t, prv, group) for t in recv]
    for req in dist.batch_isend_irecv(ops):
        req.wait()
    return recv


def forward_round(q_r: torch.Tensor, k_s: torch.Tensor, v_s: torch.Tensor, shard_mask: DeviceMask,
                  o_acc: torch.Tensor, lse_acc: torch.Tensor, first: bool,
                  o_out: Optional[torch.Tensor] = None, scale: Optional[float] = None, stream=None):
    """One forward round on one device: the query shard against the K/V shard
    it holds, merged into the running (o_acc fp32, lse_acc).  Pass ``o_out`` in
    the last round to receive the merged bf16 O.  Returns the round's tile
    metadata (the backward reuses it)."""
    meta = lcattn_mask_compile(make_shape(q_r, k_s, v_s), shard_mask, stream=stream, device=q_r.device)
    o_p, lse_p = lcattn_fwd(q_r, k_s, v_s, shard_mask, meta, scale, stream=stream)
    lcattn_lse_merge(o_acc, lse_acc, o_p, lse_p, o_out=o_out, first=first, stream=stream)
    return meta


def backward_round(q_r, k_s, v_s, o_r, do_r, lse_r, shard_mask: DeviceMask, meta, dq_acc, dk_acc_s, dv_acc_s,
                   scale: Optional[float] = None, workspace=None, stream=None) -> None:
    """One backward round on one device: adds the pair's dQ terms into the
    query shard's ``dq_acc`` and its dK / dV terms into the travelling
    accumulators of the K/V shard.  ``o_r`` and ``lse_r`` are the query shard's
    final output and LSE."""
    lcattn_bwd_accum(q_r, k_s, v_s, o_r, do_r, lse_r, shard_mask, meta, dq_acc, dk_acc_s, dv_acc_s,
                     scale=scale, workspace=workspace, stream=stream)


def emulate(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, mask: DeviceMask, world: int,
            d_o: Optional[torch.Tensor] = None, scale: Optional[float] = None) -> Dict[str, torch.Tensor]:
    """Ring P2P over ``world`` emulated devices on one GPU.

    q [B, N, Hq, D], k/v [B, N, Hkv, D] bf16 and the global ``mask`` of the
    N x N problem.  Each emulated device r runs its rounds in schedule order
    (rounds of all devices interleaved as the ring would run them); a hop is
    the hand-over of the same tensors.  Returns O and LSE (and dQ, dK, dV when
    ``d_o`` is given) assembled over the shards."""
    B, N, Hq, D = q.shape
    Hkv = k.shape[2]
    if k.shape[1] != N:
        raise ValueError("the ring splits one sequence: Sq must equal Sk")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    st = shard_starts(N, world)
    qs = [q[:, st[r]:st[r + 1]] for r in range(world)]
    ks = [k[:, st[r]:st[r + 1]] for r in range(world)]
    vs = [v[:, st[r]:st[r + 1]] for r in range(world)]
    dev = q.device
    o_acc = [torch.empty(B, st[r + 1] - st[r], Hq, D, dtype=torch.float32, device=dev) for r in range(world)]
    lse = [torch.empty(B, Hq, st[r + 1] - st[r], dtype=torch.float32, device=dev) for r in range(world)]
    o = torch.empty_like(q)
    metas, masks = {}, {}
    for t in range(world):
        for r in range(world):
            s = kv_shard_at(r, t, world)
            m = lcattn_mask_shard(mask, B, N, N, st[r], st[r + 1] - st[r], st[s], st[s + 1] - st[s])
            masks[r, s] = m
            metas[r, s] = forward_round(qs[r], ks[s], vs[s], m, o_acc[r], lse[r], first=(t == 0),
                                        o_out=o[:, st[r]:st[r + 1]] if t == world - 1 else None, scale=scale)
    out = {"o": o, "lse": torch.cat(lse, dim=2)}
    if d_o is None:
        return out
    # Each device's dQ accumulator for its query shard, and each K/V shard's
    # travelling dK / dV accumulators (as a device would hold them).
    n = [st[r + 1] - st[r] for r in range(world)]
    dq_acc = [torch.zeros(B, n[r], Hq, D, dtype=torch.float32, device=dev) for r in range(world)]
    dk_acc = [torch.zeros(B, n[s], Hkv, D, dtype=torch.float32, device=dev) for s in range(world)]
    dv_acc = [torch.zeros(B, n[s], Hkv, D, dtype=torch.float32, device=dev) for s in range(world)]
    for t in range(world):
        for r in range(world):
            s = kv_shard_at(r, t, world)
            sq = slice(st[r], st[r + 1])
            backward_round(qs[r], ks[s], vs[s], o[:, sq], d_o[:, sq], lse[r], masks[r, s], metas[r, s],
                           dq_acc[r], dk_acc[s], dv_acc[s], scale=scale)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    for r in range(world):
        sl = slice(st[r], st[r + 1])
        lcattn_f32_to_bf16(dq_acc[r], dq[:, sl])
        lcattn_f32_to_bf16(dk_acc[r], dk[:, sl])
        lcattn_f32_to_bf16(dv_acc[r], dv[:, sl])
    out["dq"], out["dk"], out["dv"] = dq, dk, dv
    return out
