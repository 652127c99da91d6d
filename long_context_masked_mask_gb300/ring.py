"""Context parallelism by Ring P2P over the library's per-device building blocks.

The pages' distributed half ("Long-Context Attention Benchmark", xllm-io blog
review, section "分布式注意力机制": Ring P2P exchanges K/V in several
point-to-point rounds and overlaps them with the computation; section
"分布式性能": it does best on FULL masks and fluctuates on DOCUMENT masks)
splits the sequence over ``world`` devices.  Device ``r`` holds query shard
``r`` and K/V shard ``r`` (one contiguous chunk, or an early and a late chunk
in the zigzag layout that balances causal masks: :func:`shard_chunks`).  In round ``t`` it holds K/V shard
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
from typing import Dict, List, Optional, Sequence, Tuple

import torch

from . import (DeviceMask, lcattn_bwd_accum, lcattn_f32_to_bf16, lcattn_fwd, lcattn_lse_merge,
               lcattn_mask_compile, lcattn_mask_shard, make_shape)


def shard_starts(N: int, world: int) -> List[int]:
    """Boundaries of ``world`` contiguous shards of a length-N sequence
    (shard r is [starts[r], starts[r+1]))."""
    if world < 1 or world > N:
        raise ValueError("need 1 <= world <= N")
    return [r * N // world for r in range(world + 1)]


def shard_chunks(N: int, world: int, layout: str = "contiguous") -> List[List[Tuple[int, int]]]:
    """The (start, length) chunks of the sequence that shard r holds.

    ``contiguous``: one chunk, [starts[r], starts[r+1]).  ``zigzag``: the
    sequence cut into 2 * world chunks, shard r holding chunks r and
    2 * world - 1 - r, so that under a causal mask every shard has one early
    and one late chunk and the devices do equal work in every round (with
    contiguous shards the last device does about 2 * world - 1 times the work
    of the first).  The pages note that Ring P2P's rate fluctuates with the
    mask (blog section "分布式性能"); this layout is the usual remedy for the
    causal case."""
    if layout == "contiguous":
        st = shard_starts(N, world)
        return [[(st[r], st[r + 1] - st[r])] for r in range(world)]
    if layout == "zigzag":
        if 2 * world > N:
            raise ValueError("zigzag needs N >= 2 * world")
        c = [j * N // (2 * world) for j in range(2 * world + 1)]
        return [[(c[r], c[r + 1] - c[r]), (c[2 * world - 1 - r], c[2 * world - r] - c[2 * world - 1 - r])]
                for r in range(world)]
    raise ValueError(f"unknown shard layout {layout!r}")


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
            d_o: Optional[torch.Tensor] = None, scale: Optional[float] = None,
            layout: str = "contiguous") -> Dict[str, torch.Tensor]:
    """Ring P2P over ``world`` emulated devices on one GPU.

    q [B, N, Hq, D], k/v [B, N, Hkv, D] bf16 and the global ``mask`` of the
    N x N problem.  Device r holds the query and K/V chunks of shard r
    (:func:`shard_chunks`, ``layout`` contiguous or zigzag).  Each emulated
    device runs its rounds in schedule order (rounds of all devices
    interleaved as the ring would run them); in a round it computes each of
    its query chunks against each K/V chunk it holds.  A hop is the hand-over
    of the same tensors.  Returns O and LSE (and dQ, dK, dV when ``d_o`` is
    given) assembled over the chunks."""
    B, N, Hq, D = q.shape
    Hkv = k.shape[2]
    if k.shape[1] != N:
        raise ValueError("the ring splits one sequence: Sq must equal Sk")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    shards = shard_chunks(N, world, layout)
    chunks = sorted({c for sh in shards for c in sh})   # every (start, length) once
    dev = q.device
    sl = {c: slice(c[0], c[0] + c[1]) for c in chunks}
    o_acc = {c: torch.empty(B, c[1], Hq, D, dtype=torch.float32, device=dev) for c in chunks}
    lse = {c: torch.empty(B, Hq, c[1], dtype=torch.float32, device=dev) for c in chunks}
    o = torch.empty_like(q)
    metas, masks = {}, {}
    seen = {c: 0 for c in chunks}          # K/V chunks merged so far, per query chunk
    n_kv = sum(len(sh) for sh in shards)   # K/V chunks each query chunk meets over the ring
    for t in range(world):
        for r in range(world):
            s = kv_shard_at(r, t, world)
            for a in shards[r]:
                for c in shards[s]:
                    m = lcattn_mask_shard(mask, B, N, N, a[0], a[1], c[0], c[1])
                    masks[a, c] = m
                    last = seen[a] == n_kv - 1
                    metas[a, c] = forward_round(q[:, sl[a]], k[:, sl[c]], v[:, sl[c]], m, o_acc[a], lse[a],
                                                first=seen[a] == 0, o_out=o[:, sl[a]] if last else None,
                                                scale=scale)
                    seen[a] += 1
    out = {"o": o, "lse": torch.cat([lse[c] for c in chunks], dim=2)}
    if d_o is None:
        return out
    # Each device's dQ accumulators for its query chunks, and each K/V chunk's
    # travelling dK / dV accumulators (as a device would hold them).
    dq_acc = {c: torch.zeros(B, c[1], Hq, D, dtype=torch.float32, device=dev) for c in chunks}
    dk_acc = {c: torch.zeros(B, c[1], Hkv, D, dtype=torch.float32, device=dev) for c in chunks}
    dv_acc = {c: torch.zeros(B, c[1], Hkv, D, dtype=torch.float32, device=dev) for c in chunks}
    for t in range(world):
        for r in range(world):
            s = kv_shard_at(r, t, world)
            for a in shards[r]:
                for c in shards[s]:
                    backward_round(q[:, sl[a]], k[:, sl[c]], v[:, sl[c]], o[:, sl[a]], d_o[:, sl[a]], lse[a],
                                   masks[a, c], metas[a, c], dq_acc[a], dk_acc[c], dv_acc[c], scale=scale)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    for c in chunks:
        lcattn_f32_to_bf16(dq_acc[c], dq[:, sl[c]])
        lcattn_f32_to_bf16(dk_acc[c], dk[:, sl[c]])
        lcattn_f32_to_bf16(dv_acc[c], dv[:, sl[c]])
    out["dq"], out["dk"], out["dv"] = dq, dk, dv
    return out
