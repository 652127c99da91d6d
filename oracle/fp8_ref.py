"""FP8 (E4M3) inputs for the oracle: decoding of the codes and the forward on
the decoded values.

TEST INFRASTRUCTURE (see the package docstring): nothing in the product imports
this module.

The pages benchmark bf16 attention and fix no fp8 semantics; the reading the
FP8 forward is checked against is: the inputs are OCP FP8 E4M3 codes times a
per-tensor factor, and the result is the attention of those real values.  The
decoding follows the format's definition: bit 7 sign, bits 6..3 exponent
(bias 7), bits 2..0 mantissa; exponent 0 is subnormal, (m / 8) * 2^-6;
otherwise (1 + m / 8) * 2^(e - 7); exponent 15 with mantissa 7 is NaN; there
are no infinities (largest finite 448).
"""
from __future__ import annotations

import numpy as np

from .attention_ref import attention_fwd


def e4m3_decode(codes) -> np.ndarray:
    """fp64 values of uint8 E4M3 codes (NaN for the NaN codes)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    sub = (m / 8.0) * 2.0 ** -6
    norm = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    val = sign * np.where(e == 0, sub, norm)
    return np.where((e == 15) & (m == 7), np.nan, val)


def attention_fwd_fp8(q8, k8, v8, q_scale, k_scale, v_scale, spec, scale, chunk: int = 1024):
    """O and LSE of the attention of the decoded inputs (code value x factor),
    in fp64: attention_fwd applied to them."""
    return attention_fwd(e4m3_decode(q8) * q_scale, e4m3_decode(k8) * k_scale, e4m3_decode(v8) * v_scale,
                         spec, scale, chunk)
