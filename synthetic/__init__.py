"""Seeded synthetic inputs and workload shapes.

This module is shared by both sides of every parity check: the fp64 oracle
(``oracle/``) and the CUDA path (``long_context_masked_mask_gb300``).  It holds
random draws and the plain description of each workload only -- no attention
arithmetic and no mask predicate.  Each side interprets a :class:`MaskSpec` on
its own.

The pages this project follows ("Long-Context Attention Benchmark: From Kernel
Efficiency to Distributed Context Parallelism", the xllm-io blog review, section
"四、实验结果 / 实验设置") run bf16 attention with head dim 128, GQA 64:8 and MHA
64:64, at sequence lengths from 1K to 512K, on packed data from Pile, ProLong and
SlimPajama.  Those datasets are not available here; the generators below stand
in for them with i.i.d. normal activations and lognormal document lengths.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Any, Dict, List, Optional, Sequence

import numpy as np
import torch

# Mask families named by the pages (xllm-io blog, section "注意力掩码模式":
# six regular masks, six heterogeneous masks, two dynamic block masks).
MASK_KINDS = (
    "FULL",
    "CAUSAL",
    "FULL_DOCUMENT",
    "CAUSAL_DOCUMENT",
    "FULL_SLIDING_WINDOW",
    "CAUSAL_SLIDING_WINDOW",
    "SHARED_QUESTION",
    "GLOBAL_SLIDING",
    "CAUSAL_BLOCKWISE",
    "PREFIX_LM_CAUSAL",
    "PREFIX_LM_DOCUMENT",
    "BLOCK_CAUSAL_DOCUMENT",
    "UNIFORM_BLOCK",
    "VARIABLE_BLOCK",
)


@dataclasses.dataclass
class MaskSpec:
    """A mask family plus its parameters, as plain data.

    ``params`` keys by kind (all lengths in tokens):

    * FULL_DOCUMENT / CAUSAL_DOCUMENT: ``doc_lens`` (list, sums to N)
    * FULL_SLIDING_WINDOW / CAUSAL_SLIDING_WINDOW: ``window``
    * SHARED_QUESTION: ``question_len``, ``answer_lens`` (question + answers = N)
    * GLOBAL_SLIDING: ``global_tokens``, ``window``
    * CAUSAL_BLOCKWISE: ``block``
    * PREFIX_LM_CAUSAL: ``prefix``
    * PREFIX_LM_DOCUMENT: ``doc_lens``, ``prefix_lens`` (one per document)
    * BLOCK_CAUSAL_DOCUMENT: ``doc_lens``, ``block_lens`` (one list per document,
      each summing to that document's length)
    * UNIFORM_BLOCK: ``block`` and ``keep`` (bool array [Hq, ceil(N/block), ceil(N/block)])
    * VARIABLE_BLOCK: ``q_block_lens``, ``k_block_lens`` and ``keep`` (bool array
      [Hq, len(q_block_lens), len(k_block_lens)])
    """

    kind: str
    params: Dict[str, Any] = dataclasses.field(default_factory=dict)

    def __post_init__(self):
        if self.kind not in MASK_KINDS:
            raise ValueError(f"unknown mask kind {self.kind!r}")

    @property
    def per_head(self) -> bool:
        return self.kind in ("UNIFORM_BLOCK", "VARIABLE_BLOCK")

    def label(self) -> str:
        p = self.params
        extra = {
            "FULL_SLIDING_WINDOW": lambda: f"w{p['window']}",
            "CAUSAL_SLIDING_WINDOW": lambda: f"w{p['window']}",
            "GLOBAL_SLIDING": lambda: f"g{p['global_tokens']}w{p['window']}",
            "CAUSAL_BLOCKWISE": lambda: f"b{p['block']}",
            "PREFIX_LM_CAUSAL": lambda: f"p{p['prefix']}",
            "UNIFORM_BLOCK": lambda: f"b{p['block']}",
        }.get(self.kind)
        return self.kind + ("_" + extra() if extra else "")


# --------------------------------------------------------------------------
# Activations
# --------------------------------------------------------------------------

def qkv(B: int, N: int, Hq: int, Hkv: int, D: int = 128, seed: int = 0,
        with_do: bool = True, Sk: Optional[int] = None) -> Dict[str, torch.Tensor]:
    """Q, K, V (and dO) as CPU bf16 tensors in [B, S, H, D] layout.

    Values are i.i.d. N(0,1) drawn in fp32 by ``torch.Generator`` seeded with
    ``seed`` in the order Q, K, V, dO, then rounded to bf16.
    """
    Sk = N if Sk is None else Sk
    g = torch.Generator().manual_seed(seed)
    out = {
        "q": torch.randn(B, N, Hq, D, generator=g, dtype=torch.float32).to(torch.bfloat16),
        "k": torch.randn(B, Sk, Hkv, D, generator=g, dtype=torch.float32).to(torch.bfloat16),
        "v": torch.randn(B, Sk, Hkv, D, generator=g, dtype=torch.float32).to(torch.bfloat16),
    }
    if with_do:
        out["do"] = torch.randn(B, N, Hq, D, generator=g, dtype=torch.float32).to(torch.bfloat16)
    return out


def qkv_fp8(B: int, N: int, Hq: int, Hkv: int, D: int = 128, seed: int = 0,
            Sk: Optional[int] = None, device: str = "cpu") -> Dict[str, Any]:
    """Q, K, V as OCP FP8 E4M3 codes (uint8 tensors, [B, S, H, D]) with per-tensor
    descale factors: each tensor is drawn i.i.d. N(0,1) in fp32 as in
    :func:`qkv` (order Q, K, V, one ``torch.Generator`` seeded with ``seed`` on
    ``device``), divided by its factor amax / 448 and rounded to E4M3 by torch's
    float8_e4m3fn conversion, so its largest magnitude maps to E4M3's largest
    finite value.  The real inputs are code value x factor."""
    Sk = N if Sk is None else Sk
    g = torch.Generator(device=device).manual_seed(seed)
    out: Dict[str, Any] = {}
    for name, S, H in (("q", N, Hq), ("k", Sk, Hkv), ("v", Sk, Hkv)):
        x = torch.randn(B, S, H, D, generator=g, device=device, dtype=torch.float32)
        f = float(x.abs().max()) / 448.0
        out[name + "8"] = (x / f).to(torch.float8_e4m3fn).view(torch.uint8)
        out[name + "_scale"] = f
    return out


def qkv_device(B: int, N: int, Hq: int, Hkv: int, D: int = 128, seed: int = 0,
               device: str = "cuda") -> Dict[str, torch.Tensor]:
    """Same distribution as :func:`qkv`, drawn directly on ``device``.

    Used for the largest workloads, where drawing gigabytes on the host would
    dominate the run; the values differ from :func:`qkv` for the same seed.
    """
    g = torch.Generator(device=device).manual_seed(seed)
    mk = lambda S, H: torch.randn(B, S, H, D, generator=g, device=device,
                                  dtype=torch.float32).to(torch.bfloat16)
    return {"q": mk(N, Hq), "k": mk(N, Hkv), "v": mk(N, Hkv), "do": mk(N, Hq)}


def qkv_block_structured(B: int, N: int, Hq: int, Hkv: int, block: int, strength: float = 1.0,
                         D: int = 128, seed: int = 0, device: str = "cpu") -> Dict[str, torch.Tensor]:
    """Q, K, V, dO in [B, S, H, D] bf16 whose Q and K rows share a direction per
    block of ``block`` positions.

    Row r of query head h is N(0, I) noise plus ``strength`` * u[b, r // block, h],
    and row r of KV head g is noise plus ``strength`` * w[b, r // block, g], with u
    and w drawn N(0, I) once per block; V and dO are i.i.d. N(0, 1).  Draw order:
    noise Q, K, V, dO, then u, w, all from one ``torch.Generator`` seeded with
    ``seed`` on ``device``.  The dynamic sparse masks of the pages are chosen from
    real activations, whose block averages differ from block to block; with
    i.i.d. rows every pooled score would be close to zero and the selection close
    to arbitrary, so the shared per-block direction stands in for that structure.
    """
    g = torch.Generator(device=device).manual_seed(seed)
    mk = lambda *shape: torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    q, k, v, do = mk(B, N, Hq, D), mk(B, N, Hkv, D), mk(B, N, Hkv, D), mk(B, N, Hq, D)
    nb = (N + block - 1) // block
    u, w = mk(B, nb, Hq, D), mk(B, nb, Hkv, D)
    rows = torch.arange(N, device=device) // block
    q += strength * u[:, rows]
    k += strength * w[:, rows]
    return {"q": q.to(torch.bfloat16), "k": k.to(torch.bfloat16), "v": v.to(torch.bfloat16),
            "do": do.to(torch.bfloat16)}


# --------------------------------------------------------------------------
# Random structure for the masks
# --------------------------------------------------------------------------

def doc_lengths_lognormal(total: int, median: float = 2048.0, sigma: float = 1.0,
                          lo: int = 256, hi: int = 16384, seed: int = 0) -> List[int]:
    """Packed-document lengths: lognormal(ln median, sigma) rounded and clipped
    to [lo, hi], appended until they reach ``total``; the last one is cut so
    that the lengths sum to exactly ``total``."""
    rng = np.random.default_rng(seed)
    lens: List[int] = []
    acc = 0
    while acc < total:
        x = int(round(float(rng.lognormal(mean=math.log(median), sigma=sigma))))
        x = max(lo, min(hi, x))
        x = min(x, total - acc)
        lens.append(x)
        acc += x
    return lens


def segment_lengths(total: int, lo: int, hi: int, seed: int) -> List[int]:
    """Uniform random integer lengths in [lo, hi] that sum to ``total`` (last one cut)."""
    rng = np.random.default_rng(seed)
    lens: List[int] = []
    acc = 0
    while acc < total:
        x = int(rng.integers(lo, hi + 1))
        x = min(x, total - acc)
        lens.append(x)
        acc += x
    return lens


def block_keep(Hq: int, nqb: int, nkb: int, p: float = 0.5, seed: int = 0,
               force_diagonal: bool = True) -> np.ndarray:
    """Bernoulli(p) keep map per query head, [Hq, nqb, nkb] bool; the diagonal
    blocks are forced on when ``force_diagonal``."""
    rng = np.random.default_rng(seed)
    keep = rng.random((Hq, nqb, nkb)) < p
    if force_diagonal:
        d = np.arange(min(nqb, nkb))
        keep[:, d, d] = True
    return keep


# --------------------------------------------------------------------------
# Workloads (the five benchmark configurations)
# --------------------------------------------------------------------------

@dataclasses.dataclass
class SelectSpec:
    """A dynamic block mask chosen from the activations: TopK or TopP over pooled
    Q K^T, with uniform blocks of ``block`` tokens (plain data; each side
    interprets it on its own)."""

    rule: str            # "topk" or "topp"
    block: int = 128
    top_k: int = 0
    top_p: float = 0.0
    causal: bool = False

    def label(self) -> str:
        crit = f"k{self.top_k}" if self.rule == "topk" else f"p{self.top_p:g}"
        return f"{self.rule.upper()}_{crit}_b{self.block}{'_causal' if self.causal else ''}"


@dataclasses.dataclass
class Workload:
    name: str
    B: int
    N: int
    Hq: int
    Hkv: int
    D: int
    masks: List[MaskSpec]
    device_inputs: bool = False  # draw activations on the GPU (largest sizes only)
    selects: List[SelectSpec] = dataclasses.field(default_factory=list)
    structure: float = 0.0       # > 0: block-structured Q/K (qkv_block_structured strength)
    Sq: Optional[int] = None     # query length when it differs from the key length N
    forward_only: bool = False   # decode-style rows: the step is the forward alone
    fp8: bool = False            # e4m3 Q, K, V with per-tensor factors (forward only)
    vt_cache: bool = False       # e4m3 V kept transposed, as a K/V cache would hold it: the step reads V^T

    @property
    def q_len(self) -> int:
        return self.N if self.Sq is None else self.Sq


def workload(name: str, seed: int = 0) -> Workload:
    """The benchmark configurations, by name.

    * ``causal_1k``: B=1, N=1024, 8:8 heads, CAUSAL.
    * ``dense_8k``: B=1, N=8192, GQA 64:8, FULL and CAUSAL.
    * ``docs_32k``: B=1, N=32768, GQA 64:8, FULL_DOCUMENT and CAUSAL_DOCUMENT over
      lognormal documents (median 2048, clipped to [256, 16384]).
    * ``hetero_16k``: B=1, N=16384, MHA 64:64, the five heterogeneous masks.
    * ``long_128k``: B=1, N=131072, GQA 64:8, CAUSAL and a 128x128 uniform block
      mask kept with probability 0.5 per head (diagonal forced).
    * ``long_128k_8to1``: the same with GQA 8:1 (one KV group), for profiler
      captures of the 128K kernels at a size a multi-pass capture can hold.
    * ``dense_8k_fp8``: as ``dense_8k`` with e4m3 Q, K, V (per-tensor factors,
      :func:`qkv_fp8`), forward only.
    * ``decode_32k_fp8``: as ``decode_32k`` with e4m3 Q, K, V, and V kept
      transposed (an e4m3 K/V cache): the step is the forward on Q, K and V^T.
    * ``dense_8k_hd64``: as ``dense_8k`` with head dim 64 (the variant next to the
      pages' 128).
    * ``dense_8k_hd256``: B=1, N=8192, GQA 32:8, head dim 256, FULL and CAUSAL.
    * ``dense_8k_hd256_fwd``: the same, forward only.
    * ``decode_32k``: B=8 sequences of one query row each against N=32768 keys,
      GQA 64:8, CAUSAL (bottom-right aligned: the row sees every key), forward only.
    * ``dynamic_32k``: B=1, N=32768, GQA 64:8, block-structured Q/K (strength 1.5),
      and two dynamic block masks chosen from them with 128-token blocks: TopK
      with k = 32 of 256 key blocks, and causal TopP with p = 0.9.
    """
    if name == "causal_1k":
        return Workload(name, 1, 1024, 8, 8, 128, [MaskSpec("CAUSAL")])
    if name == "dense_8k":
        return Workload(name, 1, 8192, 64, 8, 128, [MaskSpec("FULL"), MaskSpec("CAUSAL")])
    if name == "docs_32k":
        docs = doc_lengths_lognormal(32768, seed=seed)
        return Workload(name, 1, 32768, 64, 8, 128,
                        [MaskSpec("FULL_DOCUMENT", {"doc_lens": docs}),
                         MaskSpec("CAUSAL_DOCUMENT", {"doc_lens": docs})])
    if name == "hetero_16k":
        N = 16384
        return Workload(name, 1, N, 64, 64, 128, [
            MaskSpec("CAUSAL_SLIDING_WINDOW", {"window": 2048}),
            MaskSpec("GLOBAL_SLIDING", {"global_tokens": 256, "window": 1024}),
            MaskSpec("PREFIX_LM_CAUSAL", {"prefix": 4096}),
            MaskSpec("SHARED_QUESTION", {"question_len": 2048, "answer_lens": [3584] * 4}),
            MaskSpec("CAUSAL_BLOCKWISE", {"block": 1024}),
        ])
    if name == "long_128k":
        N, bs, Hq = 131072, 128, 64
        nb = N // bs
        return Workload(name, 1, N, Hq, 8, 128, [
            MaskSpec("CAUSAL"),
            MaskSpec("UNIFORM_BLOCK", {"block": bs, "keep": block_keep(Hq, nb, nb, 0.5, seed)}),
        ], device_inputs=True)
    if name == "long_128k_8to1":
        # The 128K workload with one KV group (8 query heads): the same masks,
        # lists and per-unit work, 1/8 of the units; small enough (about 1.8 GB
        # on the device) for multi-pass profiler captures.
        N, bs, Hq = 131072, 128, 8
        nb = N // bs
        return Workload(name, 1, N, Hq, 1, 128, [
            MaskSpec("CAUSAL"),
            MaskSpec("UNIFORM_BLOCK", {"block": bs, "keep": block_keep(Hq, nb, nb, 0.5, seed)}),
        ], device_inputs=True)
    if name == "dense_8k_fp8":
        return Workload(name, 1, 8192, 64, 8, 128, [MaskSpec("FULL"), MaskSpec("CAUSAL")], forward_only=True,
                        fp8=True)
    if name == "decode_32k_fp8":
        return Workload(name, 8, 32768, 64, 8, 128, [MaskSpec("CAUSAL")], Sq=1, forward_only=True, fp8=True,
                        vt_cache=True)
    if name == "dense_8k_hd64":
        return Workload(name, 1, 8192, 64, 8, 64, [MaskSpec("FULL"), MaskSpec("CAUSAL")])
    if name == "dense_8k_hd256":
        return Workload(name, 1, 8192, 32, 8, 256, [MaskSpec("FULL"), MaskSpec("CAUSAL")])
    if name == "dense_8k_hd256_fwd":
        return Workload(name, 1, 8192, 32, 8, 256, [MaskSpec("FULL"), MaskSpec("CAUSAL")], forward_only=True)
    if name == "decode_32k":
        return Workload(name, 8, 32768, 64, 8, 128, [MaskSpec("CAUSAL")], Sq=1, forward_only=True)
    if name == "dynamic_32k":
        return Workload(name, 1, 32768, 64, 8, 128, [],
                        selects=[SelectSpec("topk", 128, top_k=32),
                                 SelectSpec("topp", 128, top_p=0.9, causal=True)],
                        structure=1.5)
    raise KeyError(name)


WORKLOADS = ("causal_1k", "dense_8k", "docs_32k", "hetero_16k", "long_128k", "long_128k_8to1", "dynamic_32k",
             "decode_32k", "dense_8k_fp8", "decode_32k_fp8",
             "dense_8k_hd64", "dense_8k_hd256", "dense_8k_hd256_fwd")
