"""Pins of the oracle's MXFP8 codec, block-scale rule and MX layer (no GPU needed)."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as om
from oracle import mx
from dropless_mixture_experts_warp_gb300 import synth


def _all_bf16_finite():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = synth.bf16_to_f32(bits)
    return v[np.isfinite(v)].astype(np.float64)


def test_e4m3_encode_matches_torch_on_every_bf16_value():
    """In range, encoding equals torch's float8_e4m3fn cast (RNE); beyond +-448 it saturates."""
    v = _all_bf16_finite()
    inside = np.abs(v) <= 448
    ref = torch.from_numpy(v[inside]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(mx.e4m3_encode(v[inside]), ref)
    out = mx.e4m3_encode(v[~inside])
    assert np.all((out & 0x7F) == 0x7E)
    assert np.array_equal(out >> 7, np.signbit(v[~inside]).astype(np.uint8))


def test_e4m3_round_trip_of_every_code():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    vals = mx.e4m3_decode(codes)
    assert np.array_equal(mx.e4m3_encode(vals), codes)
    assert vals.max() == 448 and np.min(np.abs(vals[vals != 0])) == 2.0 ** -9
    assert mx.e4m3_encode(np.array([-0.0]))[0] == 0x80


def test_e4m3_ties_go_to_even_code():
    # 1 + 1/16 lies halfway between 1 (0x38) and 1.125 (0x39): even code wins
    assert mx.e4m3_encode(np.array([1.0625]))[0] == 0x38
    assert mx.e4m3_encode(np.array([1.1875]))[0] == 0x3A      # between 0x39 and 0x3A
    assert mx.e4m3_encode(np.array([2.0 ** -10]))[0] == 0x00  # half the smallest subnormal


def test_scale_rule_closed_forms():
    e = mx.scale_exponent(np.array([448.0, 256.0, 511.99, 1.0, 2.0 ** 20, 0.0, 2.0 ** -140, 3.0 * 2 ** 130]))
    assert list(e) == [0, 0, 0, -8, 12, -127, -127, 123]
    x = np.zeros((1, 32))
    codes, sc = mx.mx_quantize(x)
    assert np.all(codes == 0) and sc[0, 0] == 0
    x = np.full((1, 32), 448.0)
    codes, sc = mx.mx_quantize(x)
    assert sc[0, 0] == 127 and np.all(codes == 0x7E)


def test_qdq_error_bound_and_exact_values():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((64, 256)) * np.exp2(rng.integers(-20, 20, (64, 1)))
    q = mx.qdq(x)
    blocks = np.abs(x).reshape(64, 8, 32).max(-1)
    e = mx.scale_exponent(blocks)
    scale = np.repeat(np.exp2(e.astype(float)), 32, axis=1)
    err = np.abs(q - x)
    # half an E4M3 quantum: 2^-4 relative for normals, 2^-10 * scale below 2^-6 * scale;
    # scaled values in (448, 512) saturate to 448
    bound = np.maximum.reduce([np.abs(x) * 2.0 ** -4, scale * 2.0 ** -10, np.abs(x) - 448 * scale])
    assert np.all(err <= bound * (1 + 1e-12))
    # values already on the grid (E4M3 code x block scale) pass through unchanged
    codes = rng.integers(0, 0x7E, (4, 64)).astype(np.uint8)
    codes[:, ::32] = 0x7E                           # each block reaches 448 -> scale 2^0 * s
    sc = rng.integers(100, 140, (4, 2)).astype(np.uint8)
    grid = mx.mx_dequantize(codes, sc)
    assert np.array_equal(mx.qdq(grid), grid)


def test_mx_matmul_quantises_along_the_shared_axis():
    rng = np.random.default_rng(4)
    a = rng.standard_normal((16, 64))
    a[:, 5] *= 1000.0                               # one outlier column
    eye = np.eye(64)
    assert np.array_equal(mx.mx_matmul(a, eye), mx.qdq(a))     # identity rows are exact on the grid
    # quantising along M instead of K would give another result: the outlier column
    # then only shares its scale with itself
    wrong = mx.qdq(a.T).T
    assert np.abs(wrong - mx.qdq(a)).max() > 1e-3


def _small(seed=5, T=40, d=64, f=32, E=4, k=2, shared=False):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, d))
    w_gu = rng.standard_normal((E, 2 * f, d)) / np.sqrt(d)
    w_d = rng.standard_normal((E, d, f)) / np.sqrt(f)
    dy = rng.standard_normal((T, d))
    logits = rng.standard_normal((T, E))
    s = None
    if shared:
        s = (rng.standard_normal((64, d)) / np.sqrt(d), rng.standard_normal((d, 32)) / np.sqrt(32))
    return x, logits, w_gu, w_d, dy, s


@pytest.mark.parametrize("shared", [False, True])
def test_mx_layer_with_plain_matmul_is_the_bf16_oracle(shared):
    """The MX forward/backward differ from the plain oracle only in the GEMM used."""
    x, logits, w_gu, w_d, dy, s = _small(shared=shared)
    kw = {} if s is None else {"w_gu_s": s[0], "w_d_s": s[1]}
    plain = lambda a, b, dtype=np.float64: (a @ b.T).astype(dtype)  # noqa: E731
    f1 = mx.moe_forward_mx(x, logits, w_gu, w_d, 2, "sigmoid", matmul=plain, **kw)
    b1 = mx.moe_backward_mx(x, logits, w_gu, w_d, dy, f1, 2, "sigmoid", matmul=plain, **kw)
    f0 = om.moe_forward(x, logits, w_gu, w_d, 2, "sigmoid", **kw)
    b0 = om.moe_backward(x, logits, w_gu, w_d, dy, f0, 2, "sigmoid", **kw)
    np.testing.assert_allclose(f1["Y"], f0["Y"], rtol=1e-12, atol=1e-12)
    for key in b0:
        np.testing.assert_allclose(b1[key], b0[key], rtol=1e-10, atol=1e-12, err_msg=key)


def test_mx_layer_close_to_plain_layer():
    x, logits, w_gu, w_d, dy, _ = _small(seed=6)
    f1 = mx.moe_forward_mx(x, logits, w_gu, w_d, 2)
    b1 = mx.moe_backward_mx(x, logits, w_gu, w_d, dy, f1, 2)
    f0 = om.moe_forward(x, logits, w_gu, w_d, 2)
    b0 = om.moe_backward(x, logits, w_gu, w_d, dy, f0, 2)

    def rel(a, b):
        return np.abs(a - b).max() / np.abs(b).max()
    # quantisation is active; E4M3 keeps 3 mantissa bits, so a few percent RMS per GEMM
    assert 1e-3 < rel(f1["Y"], f0["Y"]) < 0.25
    for key in ("dX", "dW_gu", "dW_d", "d_logits"):
        assert rel(b1[key], b0[key]) < 0.25, key


def test_weight_gradient_row_blocks_start_at_the_segment():
    """Quantising dW operands along rows: each expert's first row starts a 32-row block."""
    x, logits, w_gu, w_d, dy, _ = _small(seed=7, T=70, E=3, k=1)
    f1 = mx.moe_forward_mx(x, logits, w_gu, w_d, 1)
    b1 = mx.moe_backward_mx(x, logits, w_gu, w_d, dy, f1, 1)
    idx = f1["idx"][:, 0]
    for e in range(3):
        t = np.nonzero(idx == e)[0]
        g, u = f1["g"][t, 0], f1["u"][t, 0]
        h = f1["w"][t, 0][:, None] * g * (1 / (1 + np.exp(-g))) * u
        ref = mx.qdq(dy[t].T) @ mx.qdq(h.T).T
        np.testing.assert_allclose(b1["dW_d"][e], ref, rtol=1e-12, atol=1e-12)


def test_sampled_mx_wgrad_entries_match_full_mx_backward():
    x, logits, w_gu, w_d, dy, _ = _small(seed=8, T=90, E=3, k=2)
    f1 = mx.moe_forward_mx(x, logits, w_gu, w_d, 2)
    b1 = mx.moe_backward_mx(x, logits, w_gu, w_d, dy, f1, 2)
    rows = np.array([0, 7, 31, 32, 50, 63])
    cols = np.array([1, 17, 30])
    for e in range(3):
        s = mx.expert_wgrad_sampled_mx(x, logits, dy, w_gu[e], w_d[e], e, 2, rows, cols)
        np.testing.assert_allclose(s["dW_gu_rows"], b1["dW_gu"][e][rows], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(s["dW_d_cols"], b1["dW_d"][e][:, cols], rtol=1e-10, atol=1e-12)


def test_sampled_fp4_weight_wgrad_entries_match_full_backward():
    """The same restriction with E2M1 weights: the entries equal the FP8 x FP4 layer's."""
    x, logits, w_gu, w_d, dy, _ = _small(seed=11, T=90, E=3, k=2)
    f1 = mx.moe_forward_mx(x, logits, w_gu, w_d, 2, wmatmul=mx.mx_matmul_w4)
    b1 = mx.moe_backward_mx(x, logits, w_gu, w_d, dy, f1, 2, wmatmul=mx.mx_matmul_w4)
    b8 = mx.moe_backward_mx(x, logits, w_gu, w_d, dy, mx.moe_forward_mx(x, logits, w_gu, w_d, 2), 2)
    rows = np.array([0, 7, 31, 32, 50, 63])
    cols = np.array([1, 17, 30])
    for e in range(3):
        s = mx.expert_wgrad_sampled_mx(x, logits, dy, w_gu[e], w_d[e], e, 2, rows, cols, wq=mx.qdq4)
        np.testing.assert_allclose(s["dW_gu_rows"], b1["dW_gu"][e][rows], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(s["dW_d_cols"], b1["dW_d"][e][:, cols], rtol=1e-10, atol=1e-12)
        assert not np.allclose(s["dW_gu_rows"], b8["dW_gu"][e][rows], rtol=1e-6)   # FP4 weights do change it


def test_fast_qdq4_equals_code_table_path():
    """The arithmetic E2M1 path gives the code-table path's values bit for bit: every bf16
    value in blocks of every scale, the E2M1 ties, saturation, zeros of both signs."""
    rng = np.random.default_rng(10)
    v = _all_bf16_finite()
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, 6.5, 7.0, 100.0])
    x = np.concatenate([v, rng.standard_normal(4096) * 1e-3, np.zeros(64), -np.zeros(32), ties, -ties])
    x = np.concatenate([x, np.zeros((-x.size) % 32)]).reshape(-1, 32)
    ref = mx.mx4_dequantize(*mx.mx4_quantize(x))
    got = mx.qdq4(x)
    assert np.array_equal(got, ref)
    assert np.array_equal(np.signbit(got), np.signbit(ref))
    y = rng.standard_normal((50, 96)) * np.exp2(rng.integers(-30, 30, (50, 1)))
    assert np.array_equal(mx.qdq4(y), mx.mx4_dequantize(*mx.mx4_quantize(y)))
    # blocks whose scale puts the ties exactly on grid midpoints (amax 6: scale 2^0)
    t = np.concatenate([ties[:8], -ties[:8], np.full(16, 0.1)])[None, :]
    t[0, 0] = 6.0
    assert np.array_equal(mx.qdq4(t), mx.mx4_dequantize(*mx.mx4_quantize(t)))


def test_fast_qdq_equals_code_table_path():
    rng = np.random.default_rng(9)
    v = _all_bf16_finite()
    x = np.concatenate([v, rng.standard_normal(4096) * 1e-3, np.zeros(64), -np.zeros(32)])
    x = np.concatenate([x, np.zeros((-x.size) % 32)]).reshape(-1, 32)
    ref = mx.mx_dequantize(*mx.mx_quantize(x))
    got = mx.qdq(x)
    assert np.array_equal(got, ref)
    assert np.array_equal(np.signbit(got), np.signbit(ref))
    y = rng.standard_normal((50, 96)) * np.exp2(rng.integers(-30, 30, (50, 1)))
    assert np.array_equal(mx.qdq(y), mx.mx_dequantize(*mx.mx_quantize(y)))
    # the fp32 path gives the same values as the fp64 one
    x32 = x.astype(np.float32)
    assert np.array_equal(mx.qdq(x32).astype(np.float64), mx.qdq(x32.astype(np.float64)))
    y32 = y.astype(np.float32)
    assert np.array_equal(mx.qdq(y32).astype(np.float64), mx.qdq(y32.astype(np.float64)))


def test_mx_expert_rows_assemble_the_mx_layer():
    """The per-expert MXFP8 form gives exactly the MXFP8 layer oracle's results (the same
    quantised products on the same operands), and per-row results do not depend on the
    other rows present."""
    x, logits, w_gu, w_d, dy, _ = _small(seed=8, T=64, E=4, k=2)
    fwd = mx.moe_forward_mx(x, logits, w_gu, w_d, 2)
    bwd = mx.moe_backward_mx(x, logits, w_gu, w_d, dy, fwd, 2)
    idx, w = fwd["idx"], fwd["w"]
    y_slot, dx_slot, dw = np.zeros((64, 2, 64)), np.zeros((64, 2, 64)), np.zeros((64, 2))
    for e in range(4):
        t_sel, j_sel = np.nonzero(idx == e)
        r = mx.expert_rows_mx(x[t_sel], w[t_sel, j_sel], dy[t_sel], w_gu[e], w_d[e])
        y_slot[t_sel, j_sel], dx_slot[t_sel, j_sel], dw[t_sel, j_sel] = r["y"], r["dx"], r["dw"]
        np.testing.assert_array_equal(r["dW_gu"], bwd["dW_gu"][e])
        np.testing.assert_array_equal(r["dW_d"], bwd["dW_d"][e])
        sub = np.array([0, len(t_sel) // 2, len(t_sel) - 1])
        part = mx.expert_rows_mx(x[t_sel[sub]], w[t_sel[sub], j_sel[sub]], dy[t_sel[sub]], w_gu[e], w_d[e],
                                 full=False)
        for key in ("y", "dx", "dw", "dGU"):
            np.testing.assert_array_equal(part[key], r[key][sub], err_msg=key)
    np.testing.assert_array_equal(y_slot[:, 0] + y_slot[:, 1], fwd["Y"])
    np.testing.assert_array_equal(dx_slot[:, 0] + dx_slot[:, 1], bwd["dX"])
    np.testing.assert_array_equal(dw, bwd["dw"])
