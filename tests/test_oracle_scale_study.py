"""Pins of the facts the global-scale study counts ("Accelerating Long-Context and Agentic
Inference with NVFP4 KV Cache", LMSYS: "Limitations" runs with a global scale of 1.0 and names
calibration as open; the calibrated choice here is g = amax / (448 * 6)). Each pin follows
from the E4M3 / E2M1 definitions alone: the calibrated g never saturates a block scale, g = 1
saturates (and clips) a block whose maximum exceeds 6 * 448, and rounds a block's scale to 0
(every value to 0) below half the smallest subnormal step."""
import numpy as np
import pytest

import oracle


def _bf16(x):
    return (np.asarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _bf16_vals(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_calibrated_global_scale_never_saturates_a_block():
    """g = fp32(amax / 2688): every block amax a has fp32(a / fp32(6 g)) <= 448 up to fp32
    rounding (so below 464, the midpoint to the next E4M3 step: no scale saturates), and
    decoding never clips: the largest decoded magnitude of a block is within the encoder's
    error bound of its amax."""
    rng = np.random.default_rng(31)
    x = rng.standard_normal((4, 2, 16, 64)).astype(np.float32)
    x.reshape(-1, 16)[rng.permutation(x.size // 16)[:6]] *= 1e3
    bits = _bf16(x)
    g = oracle.global_scale(bits, oracle.BF16, 2, 64, 16)
    d, s = oracle.quantize_pages(bits, oracle.BF16, 2, 64, 16, g)
    xs = _bf16_vals(bits).reshape(-1, 16)
    amax = np.abs(xs).max(1)
    q = np.float32(6.0 * np.float32(g))
    assert np.all((amax / q).astype(np.float32) <= np.float32(448.0) * (1 + 2 ** -22))
    y = _bf16_vals(oracle.dequantize_pages(d, s, 2, 64, 16, g)).reshape(-1, 16)
    # the block maximum comes back within a quarter of a scale step (no clipping at 2688 g)
    sv = np.vectorize(oracle.e4m3_value)(s.reshape(-1).astype(int)) * g
    assert np.all(np.abs(np.abs(y).max(1) - amax) <= 1.0 * sv + 1e-30)


def test_unit_global_scale_saturates_and_clips_large_blocks():
    """g = 1 and a block whose maximum is 5000 > 6 * 448: the scale saturates at 448 (byte
    0x7E) and that value decodes to the clipped 2688."""
    x = np.zeros((1, 1, 1, 16), np.float32)
    x[0, 0, 0, :4] = [5000.0, -3000.0, 100.0, 1.0]
    bits = _bf16(x)
    d, s = oracle.quantize_pages(bits, oracle.BF16, 1, 16, 1, 1.0)
    assert s.reshape(-1)[0] == 0x7E
    y = _bf16_vals(oracle.dequantize_pages(d, s, 1, 16, 1, 1.0)).reshape(-1)
    assert y[0] == 2688.0 and y[1] == -2688.0


@pytest.mark.parametrize("amax,zero,subnormal", [(0.004, True, False), (0.03, False, True),
                                                 (0.1, False, False)])
def test_unit_global_scale_underflow_and_subnormal_scales(amax, zero, subnormal):
    """g = 1: amax / 6 below half the smallest subnormal E4M3 step (2^-10) rounds the scale to
    0 and the whole block to 0; between that and 2^-6 the scale is subnormal (exponent bits 0);
    above, normal."""
    x = np.zeros((1, 1, 1, 16), np.float32)
    x[0, 0, 0, 0] = amax
    x[0, 0, 0, 1] = -amax / 3
    bits = _bf16(x)
    d, s = oracle.quantize_pages(bits, oracle.BF16, 1, 16, 1, 1.0)
    sb = int(s.reshape(-1)[0])
    assert (sb == 0) == zero
    assert (sb != 0 and (sb & 0x78) == 0) == subnormal
    y = _bf16_vals(oracle.dequantize_pages(d, s, 1, 16, 1, 1.0)).reshape(-1)
    if zero:
        assert not np.any(y)
