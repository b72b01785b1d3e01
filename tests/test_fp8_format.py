"""The FP8 inputs are OCP FP8 E4M3 (1 sign bit, 4 exponent bits with bias 7, 3 mantissa
bits, subnormals at exponent 0, no infinities, NaN only at S.1111.111): every one of the
256 codes, decoded by the cast the input recipe uses, equals the value the definition
gives, and the recipe's scales map each tensor's largest magnitude to 448. CPU only."""
import math

import numpy as np
import torch

from swin_window_attention_gb300 import inputs


def _e4m3_by_definition(code: int) -> float:
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return math.nan
    if e == 0:
        return s * (m / 8.0) * 2.0 ** (1 - 7)
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def test_every_e4m3_code_decodes_as_defined():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    got = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    want = np.array([_e4m3_by_definition(c) for c in range(256)])
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert want[0x7E] == 448.0 and want[0x01] == 2.0 ** -9


def test_recipe_scales_and_decoding():
    wl = inputs.Workload("fp8", 9, 5, 2, 14, 14, 64, 2, 7, 3, "bf16")
    q8, scales = inputs.make_qkv_fp8(wl)
    assert q8.dtype == torch.float8_e4m3fn and q8.shape == (2, 14, 14, 192)
    x = inputs.normal((2, 14, 14, 192), wl.seed).double().numpy()
    d = inputs.fp8_decoded_f64(q8, scales, 64)
    for t in range(3):
        sl = slice(64 * t, 64 * (t + 1))
        assert abs(float(q8[..., sl].to(torch.float64).abs().max()) - 448.0) < 1e-9
        # each value within half an E4M3 step (2^-4 relative) of the fp32 draw, or within
        # half the subnormal step near zero
        err = np.abs(d[..., sl] - x[..., sl])
        assert np.all(err <= np.maximum(2.0 ** -4 * np.abs(x[..., sl]), scales[t] * 2.0 ** -10) * (1 + 1e-12))
