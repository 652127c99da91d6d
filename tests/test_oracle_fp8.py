"""Pins of the oracle's FP8 part (CPU): the E4M3 decoder against torch's own
float8_e4m3fn conversion on all 256 codes and against hand-derived values
from the format's definition; mutants of the decoder (wrong bias, wrong
subnormal scale, wrong mantissa weight, no NaN) are rejected; the fp8 forward
equals torch's fp64 SDPA on the decoded inputs."""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import fp8_ref
from synthetic import MaskSpec, qkv_fp8

from test_oracle_mutations import mutant

HAND = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0, 0x3C: 1.5,
        0x40: 2.0, 0x7E: 448.0, 0x80: -0.0, 0xB8: -1.0, 0xFE: -448.0}


def _torch_decode(codes):
    return torch.tensor(codes, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _decoder_holds(mod):
    codes = np.arange(256, dtype=np.uint8)
    got, want = mod.e4m3_decode(codes), _torch_decode(codes)
    if not np.array_equal(np.isnan(got), np.isnan(want)):
        return False
    if not np.array_equal(got[~np.isnan(got)], want[~np.isnan(want)]):
        return False
    return all(mod.e4m3_decode(np.array([c], dtype=np.uint8))[0] == v for c, v in HAND.items())


def test_decoder_matches_torch_and_hand_values():
    assert _decoder_holds(fp8_ref)
    assert np.isnan(fp8_ref.e4m3_decode(np.array([0x7F, 0xFF], dtype=np.uint8))).all()


@pytest.mark.parametrize("old,new", [
    ("np.exp2(e.astype(np.float64) - 7.0)", "np.exp2(e.astype(np.float64) - 8.0)"),
    ("(m / 8.0) * 2.0 ** -6", "(m / 8.0) * 2.0 ** -7"),
    ("(1.0 + m / 8.0)", "(1.0 + m / 16.0)"),
    ("(e == 15) & (m == 7)", "(e == 16) & (m == 7)"),
])
def test_decoder_mutants_rejected(old, new):
    assert not _decoder_holds(mutant(fp8_ref, old, new))


def test_fp8_forward_is_sdpa_of_decoded_inputs():
    x = qkv_fp8(1, 40, 4, 2, 16, seed=5)
    spec = MaskSpec("CAUSAL")
    s = 0.3
    O, L = fp8_ref.attention_fwd_fp8(x["q8"].numpy(), x["k8"].numpy(), x["v8"].numpy(), x["q_scale"],
                                     x["k_scale"], x["v_scale"], spec, s)
    dec = lambda t, f: torch.tensor(fp8_ref.e4m3_decode(t.numpy()) * f).permute(0, 2, 1, 3)
    q, k, v = dec(x["q8"], x["q_scale"]), dec(x["k8"], x["k_scale"]), dec(x["v8"], x["v_scale"])
    k, v = k.repeat_interleave(2, 1), v.repeat_interleave(2, 1)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True, scale=s)
    np.testing.assert_allclose(O, ref.permute(0, 2, 1, 3).numpy(), atol=1e-12)
    # the inputs use the whole E4M3 range: each tensor's largest magnitude is 448
    for n in ("q8", "k8", "v8"):
        assert np.nanmax(np.abs(fp8_ref.e4m3_decode(x[n].numpy()))) == 448.0
