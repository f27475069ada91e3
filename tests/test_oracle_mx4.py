"""Pins of the oracle's FP4 (E2M1) weight codec and of the FP8 x FP4 layer (no GPU needed).

The E2M1 values are derived here from the bit fields (sign, two exponent bits with bias
1, one mantissa bit), and rounding is checked by brute force over all sixteen codes, so
neither check reuses the oracle's value table or its search.
"""
import numpy as np
import pytest

from oracle import moe_oracle as om
from oracle import mx


def _field_value(code):
    s, e, m = (code >> 3) & 1, (code >> 1) & 3, code & 1
    mag = m * 0.5 if e == 0 else (1.0 + 0.5 * m) * 2.0 ** (e - 1)
    return -mag if s else mag


def _brute_encode(v):
    """Nearest of the sixteen code values; ties to the code with mantissa bit 0; beyond
    6 in magnitude the largest code of that sign (saturation)."""
    out = []
    for x in np.ravel(v):
        sign = 8 if np.signbit(x) else 0
        a = min(abs(x), 6.0)
        best = None
        for c in range(8):
            dist = abs(_field_value(c) - a)
            if best is None or dist < best[0] or (dist == best[0] and (c & 1) == 0 and (best[1] & 1)):
                best = (dist, c)
        out.append(sign | best[1])
    return np.array(out, np.uint8).reshape(np.shape(v))


def test_e2m1_decode_follows_the_bit_fields():
    codes = np.arange(16, dtype=np.uint8)
    assert np.array_equal(mx.e2m1_decode(codes), np.array([_field_value(c) for c in range(16)]))
    assert mx.e2m1_decode(np.array([7], np.uint8))[0] == 6.0
    assert mx.e2m1_decode(np.array([1], np.uint8))[0] == 0.5    # the one subnormal step


def test_e2m1_encode_round_trips_every_code():
    codes = np.arange(16, dtype=np.uint8)
    vals = np.array([_field_value(c) for c in range(16)])
    vals[8] = -0.0
    assert np.array_equal(mx.e2m1_encode(vals), codes)


def test_e2m1_encode_matches_brute_force_including_ties_and_saturation():
    grid = np.arange(-8.0, 8.0 + 1e-9, 0.0625)          # every midpoint between codes is on it
    extra = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.5, 7.0, 1e6, -5.0, -0.25, 1e-30])
    v = np.concatenate([grid, extra])
    assert np.array_equal(mx.e2m1_encode(v), _brute_encode(v))
    # the ties by hand: 0.25 -> 0, 0.75 -> 1, 1.25 -> 1, 1.75 -> 2, 2.5 -> 2, 3.5 -> 4, 5 -> 4
    ties = mx.e2m1_decode(mx.e2m1_encode(np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])))
    assert list(ties) == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0]


def test_e2m1_scale_rule_closed_forms():
    amax = np.array([6.0, 4.0, 7.99, 1.0, 0.75, 2.0 ** 20, 0.0, 2.0 ** -140, 2.0 ** 140])
    e = mx.scale_exponent_e2m1(amax)
    assert list(e) == [0, 0, 0, -2, -3, 18, -127, -127, 127]
    assert np.array_equal(e, np.clip(np.where(amax > 0, np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - 2,
                                              -127), -127, 127))
    codes, sc = mx.mx4_quantize(np.zeros((1, 32)))
    assert np.all(codes == 0) and sc[0, 0] == 0
    x = np.full((1, 32), 7.0)                            # scaled 7 > 6: saturates
    codes, sc = mx.mx4_quantize(x)
    assert sc[0, 0] == 127 and np.all(codes == 7)


def test_qdq4_is_blockwise_nearest_on_the_scaled_grid():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((16, 96)) * np.exp2(rng.integers(-30, 30, (16, 1)))
    x[3, 32:64] = 0.0                                     # an all-zero block
    q = mx.qdq4(x)
    blocks = x.reshape(16, 3, 32)
    amax = np.abs(blocks).max(-1)
    e = np.where(amax > 0, np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - 2, -127)
    scale = np.exp2(e)[..., None]
    ref = np.vectorize(_field_value)(_brute_encode(blocks / scale)) * scale
    assert np.array_equal(q, ref.reshape(16, 96))
    # padding: a 40-wide row quantises as its zero-padded 64-wide form
    y = rng.standard_normal((2, 40))
    assert np.array_equal(mx.qdq4(y), mx.qdq4(np.concatenate([y, np.zeros((2, 24))], 1))[:, :40])
    # mx4_quantize / mx4_dequantize give the same values
    assert np.array_equal(mx.mx4_dequantize(*mx.mx4_quantize(x)), q)


def _layer_inputs(seed, T=24, d=64, f=64, E=3):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, d))
    logits = rng.standard_normal((T, E))
    w_gu = rng.standard_normal((E, 2 * f, d)) * 0.2
    w_d = rng.standard_normal((E, d, f)) * 0.2
    dy = rng.standard_normal((T, d))
    return x, logits, w_gu, w_d, dy


def _exactly_fp4_representable(shape, rng):
    """Weights whose every 32-block (along either axis) is E2M1 values times one power of
    two with 6 at that power present, so both E2M1 and E4M3 block quantisation keep them."""
    v = rng.choice(np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]), size=shape) * rng.choice([-1.0, 1.0], size=shape)
    v[..., ::32] = 6.0                 # row blocks along the last axis
    v[..., ::32, :] = 6.0              # and column blocks along the other one
    return v * 2.0 ** -4


def test_fp8_fp4_layer_equals_fp8_layer_when_the_weights_are_fp4_values():
    """E2M1-representable weights (with the scale fixed by a 6 in every block) pass both
    quantisers unchanged, so the FP8 x FP4 layer must give the FP8 layer's exact values; a
    weight product routed through the wrong quantiser, or an activation quantised as FP4,
    changes them."""
    rng = np.random.default_rng(11)
    x, logits, _, _, dy = _layer_inputs(7)
    w_gu = _exactly_fp4_representable((3, 128, 64), rng)
    w_d = _exactly_fp4_representable((3, 64, 64), rng)
    assert np.array_equal(mx.qdq4(w_gu), w_gu) and np.array_equal(mx.qdq(w_gu), w_gu)
    assert np.array_equal(mx.qdq4(np.swapaxes(w_d, 1, 2)), np.swapaxes(w_d, 1, 2))
    f8 = mx.moe_forward_mx(x, logits, w_gu, w_d, 2)
    f4 = mx.moe_forward_mx(x, logits, w_gu, w_d, 2, wmatmul=mx.mx_matmul_w4)
    assert np.array_equal(f4["Y"], f8["Y"])
    b8 = mx.moe_backward_mx(x, logits, w_gu, w_d, dy, f8, 2)
    b4 = mx.moe_backward_mx(x, logits, w_gu, w_d, dy, f4, 2, wmatmul=mx.mx_matmul_w4)
    for key in ("dX", "dW_gu", "dW_d", "d_logits"):
        assert np.array_equal(b4[key], b8[key]), key


def test_fp4_quantiser_sees_only_weight_operands():
    """Every product handed to wmatmul has a weight matrix (or its transpose) as its second
    operand, and every weight product goes through it."""
    x, logits, w_gu, w_d, dy = _layer_inputs(8)
    mats = [w_gu[e] for e in range(3)] + [w_d[e] for e in range(3)]
    seen = []

    def spy(a, b, dtype=np.float64):
        assert any(np.array_equal(b, m) or np.array_equal(b, m.T) for m in mats)
        seen.append(b.shape)
        return mx.mx_matmul_w4(a, b, dtype)

    fwd = mx.moe_forward_mx(x, logits, w_gu, w_d, 2, wmatmul=spy)
    n_fwd = len(seen)
    mx.moe_backward_mx(x, logits, w_gu, w_d, dy, fwd, 2, wmatmul=spy)
    experts_used = len(np.unique(fwd["idx"]))
    assert n_fwd == 2 * experts_used and len(seen) == 4 * experts_used


def test_fp8_fp4_layer_error_is_that_of_fp4_weights():
    """Against the plain layer, the FP8 x FP4 forward is further off than the FP8 one but
    within a few times E2M1's relative step (1/4 at worst per weight, about 1/12 rms)."""
    x, logits, w_gu, w_d, _ = _layer_inputs(9, T=64, d=128, f=128, E=2)
    ref = om.moe_forward(x, logits, w_gu, w_d, 2)["Y"]
    e8 = np.abs(mx.moe_forward_mx(x, logits, w_gu, w_d, 2)["Y"] - ref).max() / np.abs(ref).max()
    e4 = np.abs(mx.moe_forward_mx(x, logits, w_gu, w_d, 2, wmatmul=mx.mx_matmul_w4)["Y"] - ref).max() / np.abs(ref).max()
    assert e8 < e4 < 0.25
