#!/usr/bin/env python
"""Benchmark: effective attention TFLOP/s (forward + backward, unmasked FLOPs).

One step is the whole hot path over one synthetic batch, for every mask of the
workload: mask compile -> forward -> backward (D pre-pass, dK/dV, dQ).  The
default workload, the one the JSON line's ``value`` is measured on, is the
long-context configuration: B=1, N=131072, GQA 64:8, head dim 128, bf16, the
CAUSAL mask and a uniform 128x128 block-sparse mask (each block kept with
probability 0.5 per query head, diagonal kept).  The same run then times the
dense 8K (FULL, CAUSAL), packed-document 32K (FULL/CAUSAL DOCUMENT) and
heterogeneous 16K MHA workloads and reports them under ``per_workload``.

Effective FLOPs count only allowed (query, key) pairs: forward 4*D per pair
and query head, backward 2.5x the forward (five GEMMs against two).

Fractions of peak: a kernel timed alone (the per-mask and roofline figures)
is divided by the measured burst bf16 GEMM rate; the whole step, timed over
many back-to-back steps, is also given against the sustained rate.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the fp64 CPU oracle, same metric

Under torchrun every rank runs its own copy of the workload on its own GPU
(weak scaling, no collective on the data path); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "effective attention TFLOP/s fwd/bwd (unmasked FLOPs) and % of GB300 bf16 peak"
UNIT = "TFLOP/s"
L2_FLUSH_BYTES = 512 << 20  # > 129 MB of L2, written before every timed step
DEFAULT_WORKLOAD = "long_128k"
DEFAULT_PER_WORKLOAD = "dense_8k,docs_32k,hetero_16k"
# Pairs of one head the oracle sample covers per mask (about a second of
# fp64 work on 16 cores per mask for the forward and backward together).
ORACLE_SAMPLE_PAIRS = 1 << 25


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="lcattn", choices=["lcattn", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--per-workload", default=DEFAULT_PER_WORKLOAD,
                    help="comma-separated workloads also timed in this run ('' for none)")
    ap.add_argument("--per-workload-steps", type=int, default=10)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--breakdown-reps", type=int, default=3)
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--out", default=None, help="also write the JSON line to this file")
    return ap.parse_args(argv)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"burst": float(p["bf16_tflops"]), "sustained": float(p["bf16_tflops_sustained"]),
                "hbm_gbs": float(p["hbm_gbs"]), "source": "measured"}
    return {"burst": 1900.0, "sustained": 1700.0, "hbm_gbs": 6800.0, "source": "fallback"}


def mask_labels(wl):
    return "+".join([s.label() for s in wl.masks] + [s.label() for s in wl.selects])


def workload_desc(wl):
    desc = (f"{wl.name}: B={wl.B}, N={wl.N}, Hq:Hkv={wl.Hq}:{wl.Hkv}, hd={wl.D}, "
            f"{'e4m3 inputs (per-tensor factors), bf16 O' if wl.fp8 else 'bf16'}, masks "
            + mask_labels(wl))
    if wl.selects:
        desc += (f" (dynamic masks selected every step from block-structured Q/K, strength "
                 f"{wl.structure:g}; the selection runs inside the step)")
    if wl.Sq is not None:
        desc += f", Sq={wl.Sq} queries per sequence against the N keys (bottom-right aligned)"
    if wl.forward_only:
        desc += (", forward only; FLOPs of the forward" if wl.fp8 and wl.Sq is None else
                 ", forward only (decode-style rows); FLOPs and bytes of the forward")
    if wl.vt_cache:
        desc += "; V held transposed as an e4m3 K/V cache would hold it (V^T made once, outside the step)"
    return desc


def offsets_uniform(N, block):
    import numpy as np
    return np.array(list(range(0, N, block)) + [N], dtype=np.int32)


def select_kw(sel):
    return {"top_k": sel.top_k} if sel.rule == "topk" else {"top_p": sel.top_p}


# ----------------------------------------------------------------------------
# oracle timing (CPU): the bounded sample shared by cpu_baseline and --impl reference
# ----------------------------------------------------------------------------

def oracle_sample_rows(wl):
    """Query rows of the oracle sample: the last R rows of the sequence, R a
    multiple of 128 chosen so that R x N stays near ORACLE_SAMPLE_PAIRS (all
    rows for short query sides)."""
    import numpy as np
    Sq = wl.q_len
    R = max(128, (ORACLE_SAMPLE_PAIRS // max(1, wl.N)) // 128 * 128)
    return np.arange(max(0, Sq - R), Sq)


def oracle_sample(wl, seed):
    """Inputs for the oracle sample: query head 0 with its KV head over the full
    key sequence (the query rows are chosen by oracle_sample_rows)."""
    from synthetic import qkv, qkv_block_structured, qkv_fp8
    if wl.fp8:
        from oracle import fp8_ref
        x = qkv_fp8(1, wl.q_len, 1, 1, wl.D, seed=seed, Sk=wl.N)
        out = {n: fp8_ref.e4m3_decode(x[n + "8"].numpy()) * x[n + "_scale"] for n in ("q", "k", "v")}
        out["rows"] = oracle_sample_rows(wl)
        return out
    if wl.structure > 0:
        x = qkv_block_structured(1, wl.N, 1, 1, wl.selects[0].block, strength=wl.structure, seed=seed)
    else:
        x = qkv(1, wl.q_len, 1, 1, wl.D, seed=seed, Sk=wl.N)
    out = {k: t.double().numpy() for k, t in x.items()}
    out["rows"] = oracle_sample_rows(wl)
    return out


def sample_desc(wl, sample):
    rows = sample["rows"]
    what = "fwd" if wl.forward_only else "fwd+bwd"
    return (f"fp64 NumPy oracle {what} of query head 0 / KV head 0 of {wl.name}: query rows "
            f"{int(rows[0])}..{int(rows[-1])} ({len(rows)} of {wl.q_len}) against all N={wl.N} keys, "
            f"masks {mask_labels(wl)}; effective FLOPs of those rows")


def oracle_step(wl, sample):
    """One oracle pass over the sample; returns the sample's effective FLOPs."""
    import numpy as np
    import oracle
    from oracle import block_select_ref
    from synthetic import MaskSpec
    flops = 0.0
    scale = 1.0 / math.sqrt(wl.D)
    rows = sample["rows"]
    specs = list(wl.masks)
    for sel in wl.selects:  # the selection is part of the step, as on the GPU
        offs = offsets_uniform(wl.N, sel.block)
        keep, _ = block_select_ref.block_select(sample["q"], sample["k"], offs, offs, sel.rule, scale,
                                                causal=sel.causal, **select_kw(sel))
        specs.append(MaskSpec("VARIABLE_BLOCK", {"q_block_lens": np.diff(offs).tolist(),
                                                 "k_block_lens": np.diff(offs).tolist(),
                                                 "keep": keep[0].astype(bool)}))
    for spec in specs:
        pairs = int(oracle.allowed(spec, wl.q_len, rows, head=0, Sk=wl.N).sum())
        if wl.forward_only:
            oracle.attention_fwd_rows(sample["q"], sample["k"], sample["v"], spec, scale, 0, 0, rows)
            flops += 4.0 * wl.D * pairs
        else:
            oracle.attention_bwd_rows(sample["q"], sample["k"], sample["v"], sample["do"], spec, scale,
                                      0, 0, rows)
            flops += 4.0 * wl.D * pairs * 3.5
    return flops


def cpu_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n and n[0]:
            return int(n[0])
    except Exception:
        pass
    return os.cpu_count()


def cpu_baseline(wl, seed):
    sample = oracle_sample(wl, seed)
    oracle_step(wl, sample)  # first touch of the inputs and the BLAS threads
    t0 = time.perf_counter()
    reps, flops = 0, 0.0
    while reps < 1 or (time.perf_counter() - t0 < 10.0 and reps < 8):
        flops += oracle_step(wl, sample)
        reps += 1
    dt = time.perf_counter() - t0
    return {"value": flops / dt / 1e12, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
            "seconds": round(dt, 3), "passes": reps, "sample": sample_desc(wl, sample)}


def run_reference(args, rank, world):
    from synthetic import workload
    wl = workload(args.workload, args.seed)
    if rank != 0:
        return
    sample = oracle_sample(wl, args.seed)
    for _ in range(args.warmup):
        oracle_step(wl, sample)
    times, flops = [], 0.0
    for _ in range(args.steps):
        t0 = time.perf_counter()
        flops = oracle_step(wl, sample)
        times.append(time.perf_counter() - t0)
    ms = 1e3 * statistics.mean(times)
    value = flops / (ms / 1e3) / 1e12
    desc = sample_desc(wl, sample)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_desc(wl), "sample": desc},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    emit(line, args)


def emit(line, args):
    text = json.dumps(line)
    print(text, flush=True)
    if args.out:
        with open(args.out, "w") as f:
            f.write(text + "\n")


# ----------------------------------------------------------------------------
# clocks
# ----------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.path = tempfile.mktemp(prefix="clocks_", suffix=".csv")
        self.proc = None
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(gpu_index)], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    rows.append({"sm": float(parts[1]), "max": float(parts[2]), "util": float(parts[4]),
                                 "hw": parts[6], "hw_th": parts[7], "sw_th": parts[8], "pcap": parts[9]})
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return None
        load = [r for r in rows if r["util"] >= 50] or rows
        reasons = set()
        for r in load:
            for key, name in (("hw", "hw_slowdown"), ("hw_th", "hw_thermal_slowdown"),
                              ("sw_th", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in load), "sm_max_mhz": max(r["max"] for r in rows),
                "reasons": sorted(reasons), "samples": len(load)}


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------

def max_over_ranks(x, dist, device=None):
    """The largest of the ranks' values of `x` (each rank passes its own), or `x`
    itself without a process group: the whole job is as slow as its slowest rank."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world, flops_per_rank_step, ms):
    """TFLOP/s of the whole job: every rank does `flops_per_rank_step` per step
    (independent replicas, weak scaling) and a step takes `ms` (max over ranks)."""
    return world * flops_per_rank_step / (ms / 1e3) / 1e12


def traffic_lookup(kernel, workload):
    """DRAM bytes per launch recorded from an ncu capture of this kernel on this
    workload, if the kernel's source has not changed since (profiles/traffic.json:
    per kernel, one record or a list of records, one per workload)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        recs = json.load(f).get(kernel)
    if isinstance(recs, dict):
        recs = [recs]
    rec = next((r for r in recs or [] if r.get("workload") == workload), None)
    if rec is None:
        return None
    src = os.path.join(ROOT, "long_context_masked_mask_gb300", "csrc", rec["source"])
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
    if sha != rec["source_sha256"]:
        return None
    out = {"bytes": rec["dram_bytes_per_launch"], "launch": rec["launch"]}
    if "scaled_from" in rec:
        out["scaled_from"] = rec["scaled_from"]
    return out


class Leg:
    """One workload on one GPU: inputs, compiled masks and buffers, and the
    timings of its step (all through the C ABI of the library)."""

    def __init__(self, name, seed, rank, dev):
        import torch
        import long_context_masked_mask_gb300 as lc
        from synthetic import qkv, qkv_block_structured, qkv_device, qkv_fp8, workload
        self.torch, self.lc, self.dev = torch, lc, dev
        self.wl = wl = workload(name, seed)
        B, N, Hq, Hkv, D = wl.B, wl.N, wl.Hq, wl.Hkv, wl.D
        s = seed + 1000 * rank
        self.fp8 = wl.fp8
        self.peak_mult = 2.0 if wl.fp8 else 1.0
        if wl.fp8:  # e4m3 codes (uint8) with per-tensor factors; forward only
            x = qkv_fp8(B, wl.q_len, Hq, Hkv, D, seed=s, Sk=N, device=str(dev))
            self.scales = (x["q_scale"], x["k_scale"], x["v_scale"])
            x = {"q": x["q8"], "k": x["k8"], "v": x["v8"], "do": None}
        elif wl.structure > 0:
            x = qkv_block_structured(B, N, Hq, Hkv, wl.selects[0].block, strength=wl.structure, seed=s,
                                     device=str(dev))
        elif wl.device_inputs:
            x = qkv_device(B, N, Hq, Hkv, D, seed=s, device=str(dev))
        else:
            x = {k: t.to(dev) for k, t in qkv(B, wl.q_len, Hq, Hkv, D, seed=s, Sk=N).items()}
        self.q, self.k, self.v, self.d_o = x["q"], x["k"], x["v"], x["do"]
        q = self.q
        self.Sq = Sq = q.shape[1]
        self.fwd_only = wl.forward_only
        self.shape = shape = lc.make_shape(self.q, self.k, self.v)
        # An e4m3 K/V cache keeps V transposed: the step's V input is then V^T,
        # made once here (self.v_src keeps V's shape for the calls).
        self.vt_cache = wl.vt_cache
        if self.vt_cache:
            self.v_src = self.v
            self.v = lc.lcattn_fp8_transpose_v(self.v_src, self.k, self.q)
            torch.cuda.synchronize()
        self.ws = torch.empty(max(16, 0 if self.fwd_only else lc.lcattn_bwd_workspace_size(shape)),
                              dtype=torch.uint8, device=dev)
        runs = []
        for spec in wl.masks:
            m = lc.DeviceMask(spec, Sq, Hq, B, device=dev, Sk=N)
            meta = lc.lcattn_mask_compile(shape, m, device=dev)
            fwd_flops = 4.0 * D * m.allowed_pairs
            runs.append({"spec": spec, "mask": m, "meta": meta,
                         "fwd_flops": fwd_flops, "bwd_flops": 0.0 if self.fwd_only else 2.5 * fwd_flops,
                         "launches": (6 if spec.per_head else 5) + (0 if self.fwd_only else 3)})
        for sel in wl.selects:
            offs = torch.from_numpy(offsets_uniform(N, sel.block)).to(dev)
            bmap = torch.empty(B, Hq, offs.numel() - 1, offs.numel() - 1, dtype=torch.uint8, device=dev)
            sws = torch.empty(lc.lcattn_block_select_workspace_size(q, self.k, lc.select_desc(
                sel.rule, offs, offs, causal=sel.causal, **select_kw(sel))), dtype=torch.uint8, device=dev)
            lc.lcattn_block_select(q, self.k, offs, offs, sel.rule, causal=sel.causal, block_map=bmap,
                                   workspace=sws, **select_kw(sel))
            m = lc.DeviceMask.from_block_map(bmap, offs, offs)
            meta = lc.lcattn_mask_compile(shape, m, device=dev)
            # The inputs are fixed, so every step selects this same map (the
            # selection is deterministic): its allowed pairs give the step's FLOPs.
            fwd_flops = 4.0 * D * m.allowed_pairs
            runs.append({"spec": sel, "sel": sel, "offs": offs, "sws": sws, "mask": m, "meta": meta,
                         "fwd_flops": fwd_flops, "bwd_flops": 2.5 * fwd_flops, "launches": 2 + 6 + 3})
        for r in runs:
            r["o"] = torch.empty(B, Sq, Hq, D, dtype=torch.bfloat16, device=dev)
            r["lse"] = torch.empty(B, Hq, Sq, dtype=torch.float32, device=dev)
            if not self.fwd_only:
                r["dq"], r["dk"], r["dv"] = torch.empty_like(q), torch.empty_like(self.k), torch.empty_like(self.v)
            if self.fp8:
                # V^T pre-pass (unless V is held transposed) and the forward, through
                # the split-KV path (slices + merge) for short query sides.
                split_ws = int(lc.library().lcattn_fwd_fp8_vt_workspace_size(lc.ctypes.byref(shape),
                                                                               lc.ctypes.byref(r["mask"].desc)))
                fws = split_ws if self.vt_cache else \
                    int(lc.library().lcattn_fwd_fp8_workspace_size(lc.ctypes.byref(shape)))
                r["fws"] = torch.empty(max(16, fws), dtype=torch.uint8, device=dev)
                r["split"] = split_ws > 0
                r["launches"] += (0 if self.vt_cache else 1) + (2 if split_ws > 0 else 1)
                continue
            # The forward's split-KV workspace (empty unless the query side is short).
            fws = lc.lcattn_fwd_workspace_size(shape, r["mask"])
            r["fws"] = torch.empty(max(16, fws), dtype=torch.uint8, device=dev)
            r["split"] = fws > 0
            r["launches"] += 2 if fws > 0 else 1  # split-KV forward: slices + merge
        self.runs = runs
        self.step_flops = sum(r["fwd_flops"] + r["bwd_flops"] for r in runs)
        self.launches_per_step = sum(r["launches"] for r in runs)

    def fwd(self, r, qq, kk, vv):
        if self.fp8 and self.vt_cache:  # vv is V^T
            self.lc.lcattn_fwd_fp8_vt(qq, kk, vv, self.v_src, *self.scales, r["mask"], r["meta"], o=r["o"],
                                      lse=r["lse"], workspace=r["fws"])
        elif self.fp8:
            self.lc.lcattn_fwd_fp8(qq, kk, vv, *self.scales, r["mask"], r["meta"], o=r["o"], lse=r["lse"],
                                   workspace=r["fws"])
        else:
            self.lc.lcattn_fwd_ws(qq, kk, vv, r["mask"], r["meta"], o=r["o"], lse=r["lse"], workspace=r["fws"])

    def select(self, r, qq, kk, stage=None):
        sel = r["sel"]
        self.lc.lcattn_block_select(qq, kk, r["offs"], r["offs"], sel.rule, causal=sel.causal,
                                    block_map=r["mask"].block_map, workspace=r["sws"], stage=stage,
                                    **select_kw(sel))

    def step(self, qq=None, kk=None, vv=None, dd=None):
        lc = self.lc
        qq = self.q if qq is None else qq
        kk = self.k if kk is None else kk
        vv = self.v if vv is None else vv
        dd = self.d_o if dd is None else dd
        for r in self.runs:
            if "sel" in r:
                self.select(r, qq, kk)
            lc.lcattn_mask_compile(self.shape, r["mask"], r["meta"])
            self.fwd(r, qq, kk, vv)
            if not self.fwd_only:
                lc.lcattn_bwd(qq, kk, vv, r["o"], dd, r["lse"], r["mask"], r["meta"],
                              dq=r["dq"], dk=r["dk"], dv=r["dv"], workspace=self.ws)

    def check_status(self):
        for r in self.runs:
            st = self.lc.lcattn_read_status(r["meta"])
            if st != 0:
                raise RuntimeError(f"{self.wl.name}: device status {st}: {self.lc.status_string(st)}")

    def time_steps(self, steps, warmup, flush, stream, barrier=lambda: None):
        """Device time (ms) of each of `steps` steps after `warmup` untimed ones;
        L2 is flushed before every step."""
        torch = self.torch
        for _ in range(warmup):
            flush.zero_()
            self.step()
        torch.cuda.synchronize()
        self.check_status()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        barrier()
        torch.cuda.synchronize()
        for e0, e1 in evs:
            flush.zero_()
            e0.record(stream)
            self.step()
            e1.record(stream)
        torch.cuda.synchronize()
        barrier()
        return [e0.elapsed_time(e1) for e0, e1 in evs]

    def breakdown(self, reps, flush, stream, pk):
        """Each kernel alone (CUDA events on the launching stream, L2 flushed
        before each launch): per-mask forward / backward rates and the total
        time per kernel name."""
        torch, lc = self.torch, self.lc
        wl, q, k, v, d_o = self.wl, self.q, self.k, self.v, self.d_o
        B, N, Hq, Hkv, D = wl.B, wl.N, wl.Hq, wl.Hkv, wl.D
        kernels = {"mask_compile": [0.0, 0.0, 0], "fwd_kernel": [0.0, 0.0, 0],
                   "bwd_prepass": [0.0, 0.0, 0], "dkdv_kernel": [0.0, 0.0, 0], "dq_convert": [0.0, 0.0, 0]}
        if wl.selects:
            kernels["pool_kernel"] = [0.0, 0.0, 0]
            kernels["select_kernel"] = [0.0, 0.0, 0]
        self.select_roof = None

        def timed(fn):
            tot = 0.0
            for _ in range(reps):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                torch.cuda.synchronize()
                tot += e0.elapsed_time(e1)
            return tot / reps

        def graph_timed(fn, n=8):
            """Average device time of fn's launches, replayed from a CUDA graph of n
            back-to-back calls (no host launch overhead between them).  Used for the
            sub-millisecond selection kernels; the pool kernel's inputs (Q and K) are
            larger than L2, so consecutive launches still stream them from HBM."""
            fn()
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for _ in range(n):
                    fn()
            tot = 0.0
            for _ in range(reps):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                g.replay()
                e1.record(stream)
                torch.cuda.synchronize()
                tot += e0.elapsed_time(e1)
            return tot / reps / n

        per_mask = []
        for r in self.runs:
            m, meta = r["mask"], r["meta"]
            t_sel = None
            if "sel" in r:
                t_pool = graph_timed(lambda: self.select(r, q, k, stage=1))
                t_pick = graph_timed(lambda: self.select(r, q, k, stage=2))
                t_sel = (t_pool, t_pick)
                kernels["pool_kernel"][0] += t_pool
                kernels["pool_kernel"][2] += 1
                kernels["select_kernel"][0] += t_pick
                kernels["select_kernel"][2] += 1
                nb = r["offs"].numel() - 1
                pool_bytes = (B * N * (Hq + Hkv) * D * q.element_size()       # Q and K read once
                              + B * (Hq + Hkv) * nb * D * 4)                 # fp32 block means written
                gbs = pool_bytes / (t_pool / 1e3) / 1e9
                self.select_roof = {"kernel": "pool_kernel", "bound": "hbm", "achieved": round(gbs, 1),
                                    "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": round(gbs / pk["hbm_gbs"], 4),
                                    "algorithmic_bytes": pool_bytes,
                                    "peak_kind": f"{pk['source']} copy bandwidth",
                                    "traffic": (traffic_lookup("pool_kernel", wl.name) or {}).get("bytes")}
            t_c = timed(lambda: lc.lcattn_mask_compile(self.shape, m, meta))
            t_f = timed(lambda: self.fwd(r, q, k, v))
            tb = [0.0, 0.0, 0.0]
            if not self.fwd_only:
                tb = [timed(lambda: lc.lcattn_bwd(q, k, v, r["o"], d_o, r["lse"], m, meta, dq=r["dq"],
                                                  dk=r["dk"], dv=r["dv"], workspace=self.ws, stage=stage))
                      for stage in (1, 2, 3)]
            for name, t, fl in (("mask_compile", t_c, 0.0), ("fwd_kernel", t_f, r["fwd_flops"]),
                                ("bwd_prepass", tb[0], 0.0), ("dkdv_kernel", tb[1], r["bwd_flops"]),
                                ("dq_convert", tb[2], 0.0)):
                kernels[name][0] += t
                kernels[name][1] += fl
                kernels[name][2] += 1
            fwd_tf = r["fwd_flops"] / (t_f / 1e3) / 1e12
            bwd_tf = r["bwd_flops"] / (sum(tb) / 1e3) / 1e12 if not self.fwd_only else 0.0
            per_mask.append({"mask": r["spec"].label(), "allowed_pairs": r["mask"].allowed_pairs,
                             "density": r["mask"].allowed_pairs / (B * Hq * self.Sq * N),
                             "forward_path": "split-KV (heads packed)" if r["split"] else "persistent",
                             "fwd_ms": round(t_f, 4), "bwd_ms": round(sum(tb), 4),
                             "bwd_stage_ms": [round(t, 4) for t in tb], "mask_compile_ms": round(t_c, 4),
                             "fwd_tflops": round(fwd_tf, 1), "bwd_tflops": round(bwd_tf, 1),
                             "fwd_frac_of_peak": round(fwd_tf / (pk["burst"] * self.peak_mult), 4),
                             "bwd_frac_of_peak": round(bwd_tf / pk["burst"], 4)})
            if t_sel is not None:
                per_mask[-1]["select_ms"] = [round(t_sel[0], 4), round(t_sel[1], 4)]
        self.kernels = kernels
        return per_mask, kernels

    def roofline(self, pk):
        """The dominant kernel (most event time in the breakdown) against its roof."""
        kernels, wl, q = self.kernels, self.wl, self.q
        B, Hq = wl.B, wl.Hq
        dom = max(kernels, key=lambda n: kernels[n][0])
        t_dom, fl_dom, n_dom = kernels[dom]
        # Q, K and V (or V^T) read, O (bf16) and LSE (fp32) written.
        fwd_bytes = (q.numel() * q.element_size() + self.k.numel() * self.k.element_size() +
                     self.v.numel() * self.v.element_size() + q.numel() * 2 + B * Hq * self.Sq * 4)
        # A forward-only step is HBM-bound when its arithmetic intensity (FLOPs per
        # algorithmic byte) is below the ridge point of the two measured peaks.
        hbm_bound = self.fwd_only and (self.step_flops / len(self.runs)) / fwd_bytes < \
            pk["burst"] * 1e12 / (pk["hbm_gbs"] * 1e9)
        if hbm_bound:
            # Decode-style rows read every K/V byte once per step and do little
            # arithmetic per byte.  Algorithmic bytes: Q, K, V read, O and LSE
            # written, per mask.
            gbs = fwd_bytes * n_dom / (t_dom / 1e3) / 1e9
            roof = {"kernel": ("split_kernel + combine_kernel" if self.runs[0]["split"] else "fwd_kernel") +
                              (" (e4m3)" if self.fp8 else ""),
                    "bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                    "frac": round(gbs / pk["hbm_gbs"], 4), "algorithmic_bytes": fwd_bytes,
                    "peak_kind": f"{pk['source']} copy bandwidth"}
        elif fl_dom > 0:
            achieved = fl_dom / (t_dom / 1e3) / 1e12
            peak = pk["burst"] * self.peak_mult
            roof = {"kernel": "vt8_kernel + fwd_kernel (e4m3)" if self.fp8 else dom, "bound": "tensor", "achieved": round(achieved, 1),
                    "peak": peak, "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                    "frac_of_sustained": round(achieved / (pk["sustained"] * self.peak_mult), 4),
                    "algorithmic_flops_per_launch": fl_dom / max(1, n_dom),
                    "launches": n_dom, "ms_per_launch": round(t_dom / max(1, n_dom), 4),
                    "peak_kind": (f"e4m3 dense: 2x the {pk['source']} bf16 burst (the nominal fp8/bf16 ratio)"
                                  if self.fp8 else f"bf16 dense, {pk['source']} burst (each kernel timed alone)")}
        else:  # a memory-bound kernel dominating would be reported against HBM
            roof = {"kernel": dom, "bound": "hbm", "achieved": None, "peak": pk["hbm_gbs"], "unit": "GB/s",
                    "frac": None, "peak_kind": f"{pk['source']} copy bandwidth"}
        tr = traffic_lookup("split_kernel" if hbm_bound and self.runs[0]["split"] else dom, wl.name)
        roof["traffic"] = tr["bytes"] if tr else None
        if tr:
            roof["traffic_launch"] = tr["launch"]
            if "scaled_from" in tr:
                roof["traffic_scaled_from"] = tr["scaled_from"]
        return roof

    def e2e(self, warmup, steps, flush, stream):
        """The same step end to end through the C ABI with host buffers: pinned
        host inputs copied up and every result copied down inside the timed region."""
        torch, lc = self.torch, self.lc
        q, k, v, d_o = self.q, self.k, self.v, self.d_o
        ins = (("q", q), ("k", k), ("v", v)) + ((("do", d_o),) if not self.fwd_only else ())
        host = {n: t.cpu().pin_memory() for n, t in ins}
        q_, k_, v_ = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        do_ = torch.empty_like(d_o) if d_o is not None else None
        out_names = ("o", "lse") if self.fwd_only else ("o", "lse", "dq", "dk", "dv")
        outs = [{n: torch.empty(r[n].shape, dtype=r[n].dtype, pin_memory=True) for n in out_names}
                for r in self.runs]
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = sum(t.numel() * t.element_size() for o in outs for t in o.values())
        # Copies overlap compute the way a training loop would: dO goes up on a
        # copy stream while the first forward runs, each mask's O and LSE go down
        # on it while its backward runs, and its gradients while the next mask
        # computes.  Every byte still moves inside the timed region: e1 is
        # recorded after the copy stream has been joined.
        copy_stream = torch.cuda.Stream(device=self.dev)
        ms = []
        for i in range(warmup + steps):
            flush.zero_()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            copy_stream.wait_stream(stream)
            with torch.cuda.stream(copy_stream):
                if not self.fwd_only:
                    do_.copy_(host["do"], non_blocking=True)
            do_ready = torch.cuda.Event()
            do_ready.record(copy_stream)
            q_.copy_(host["q"], non_blocking=True)
            k_.copy_(host["k"], non_blocking=True)
            v_.copy_(host["v"], non_blocking=True)
            for j, (r, o) in enumerate(zip(self.runs, outs)):
                if "sel" in r:
                    self.select(r, q_, k_)
                lc.lcattn_mask_compile(self.shape, r["mask"], r["meta"])
                self.fwd(r, q_, k_, v_)
                copy_stream.wait_stream(stream)
                with torch.cuda.stream(copy_stream):
                    for n in ("o", "lse"):
                        o[n].copy_(r[n], non_blocking=True)
                if j == 0:
                    stream.wait_event(do_ready)
                if not self.fwd_only:
                    lc.lcattn_bwd(q_, k_, v_, r["o"], do_, r["lse"], r["mask"], r["meta"],
                                  dq=r["dq"], dk=r["dk"], dv=r["dv"], workspace=self.ws)
                    copy_stream.wait_stream(stream)
                    with torch.cuda.stream(copy_stream):
                        for n in ("dq", "dk", "dv"):
                            o[n].copy_(r[n], non_blocking=True)
            stream.wait_stream(copy_stream)
            e1.record(stream)
            torch.cuda.synchronize()
            if i >= warmup:
                ms.append(e0.elapsed_time(e1))
        return ms, h2d, d2h

    def summary(self, steps, ms, world, per_mask, kernels, roof):
        return {"workload": workload_desc(self.wl), "steps": steps, "ms_per_step": round(ms, 4),
                "value": round(whole_job_rate(world, self.step_flops, ms), 2), "unit": UNIT,
                "per_mask": per_mask, "kernel_ms": {n: round(v[0], 4) for n, v in kernels.items()},
                "roofline": roof}


def run_gpu(args, rank, world, dist):
    import torch

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    pk = peaks()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def barrier():
        if dist is not None:
            dist.barrier()

    # ---- headline workload -------------------------------------------------
    leg = Leg(args.workload, args.seed, rank, dev)
    wl = leg.wl
    try:
        gpu_sel = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_sel = str(local)
    # Warm-up first, then the clock sampler: it must see the timed region.
    for _ in range(args.warmup):
        flush.zero_()
        leg.step()
    torch.cuda.synchronize()
    sampler = ClockSampler(gpu_sel)
    time.sleep(0.3)
    ms_steps = leg.time_steps(args.steps, 0, flush, stream, barrier)
    clocks = sampler.stop()
    ms = max_over_ranks(statistics.mean(ms_steps), dist, dev)
    value = whole_job_rate(world, leg.step_flops, ms)
    # The end-to-end leg follows the timed steps directly, so that both see the
    # GPU in the same state; the per-kernel breakdown (diagnostics) comes last.
    # Clocks are sampled through the end-to-end leg as well: its steps can meet a
    # GPU that has been power-capped for longer than the timed steps did.
    e2e_sampler = ClockSampler(gpu_sel)
    time.sleep(0.3)
    e2e_ms, h2d, d2h = leg.e2e(min(args.warmup, 3), args.e2e_steps, flush, stream)
    e2e_clocks = e2e_sampler.stop()
    per_mask, kernels = leg.breakdown(args.breakdown_reps, flush, stream, pk)
    roof = leg.roofline(pk)
    e2e_t = max_over_ranks(statistics.mean(e2e_ms), dist, dev)
    e2e = {"value": whole_job_rate(world, leg.step_flops, e2e_t), "unit": UNIT, "ms_per_step": e2e_t,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "copies": "pinned host buffers; dO and each mask's results move on a copy stream that "
                     "overlaps compute; all copies inside the timed region",
           "ms_steps": [round(t, 3) for t in e2e_ms], "clocks": e2e_clocks}
    leg.check_status()
    select_roof = getattr(leg, "select_roof", None)
    launches = leg.launches_per_step * args.steps
    headline = {"B": wl.B, "N": wl.N, "Hq": wl.Hq, "Hkv": wl.Hkv, "D": wl.D}
    del leg
    torch.cuda.empty_cache()

    # ---- the other configurations, timed in the same run ----------------------
    per_workload = []
    names = [n for n in (args.per_workload or "").split(",") if n and n != args.workload]
    for name in names:
        other = Leg(name, args.seed, rank, dev)
        ms_o = other.time_steps(args.per_workload_steps, max(3, min(args.warmup, 5)), flush, stream, barrier)
        ms_o = max_over_ranks(statistics.mean(ms_o), dist, dev)
        pm, kn = other.breakdown(args.breakdown_reps, flush, stream, pk)
        summary = other.summary(args.per_workload_steps, ms_o, world, pm, kn, other.roofline(pk))
        other.check_status()
        per_workload.append(summary)
        del other
        torch.cuda.empty_cache()

    if rank != 0:
        return
    line = {"metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3" if wl.fp8 else "bf16",
            "data": "synthetic",
            "config": {"workload": workload_desc(wl), "seq_len": headline["N"],
                       "global_batch": headline["B"] * world,
                       "heads": f"{headline['Hq']}:{headline['Hkv']}", "head_dim": headline["D"],
                       "parallelism": f"replicas x{world} (independent batches, no collective)",
                       "l2": f"flushed by a {L2_FLUSH_BYTES >> 20} MiB write before every timed step"},
            "frac_of_peak": round(value / pk["burst"], 4),
            "frac_of_sustained_peak": round(value / pk["sustained"], 4),
            "peak_tflops": {"burst": pk["burst"], "sustained": pk["sustained"], "source": pk["source"],
                            "per_mask_and_roofline": "burst (each kernel timed alone)"},
            "per_mask": per_mask,
            "kernel_ms": {n: round(v[0], 4) for n, v in kernels.items()},
            "roofline": roof, "e2e": e2e, "gpu_launches": launches,
            "clocks": clocks, "per_workload": per_workload}
    if select_roof is not None:
        line["roofline_select"] = select_roof
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, args.seed)
    emit(line, args)


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist_mod
        dist = dist_mod
        if args.impl == "reference":
            run_reference(args, rank, world)
            return
        import torch
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl")
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    try:
        run_gpu(args, rank, world, dist)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
