"""FP8 x FP4 experts (MXFP8 activations, MXFP4 weights) on the GPU against the oracle.

The E2M1 codes and E8M0 scales of the weight quantiser are compared bit for bit with the
oracle's mx4_quantize, in both orientations; the block-scaled GEMM with an E2M1 B operand
against a dequantised matmul; the whole layer (prec mxfp8-w4) against the MXFP8 oracle with
its weight products through mx_matmul_w4, within the MXFP8 tolerance: both sides quantise
the weights to the same codes, so what remains differs as in the MXFP8 layer (accumulation
order, and h and dG|dU quantised from fp32 on one side and fp64 on the other).
"""
import numpy as np
import pytest
import torch

from gpu_util import bf16_dev, f32_dev, host, need_gpu, rel_err
from oracle import mx
from test_gpu_mx import _bf16_matrix_with_every_value, scales_from_tiles, sf_tiles
from dropless_mixture_experts_warp_gb300 import synth

pytestmark = pytest.mark.gpu

TOL_MXFP8 = 6e-2


def unpack4(packed: np.ndarray) -> np.ndarray:
    """[..., n/2] bytes -> [..., n] four-bit codes, the lower element from the lower four bits."""
    packed = np.asarray(packed, np.uint8)
    return np.stack([packed & 0x0F, packed >> 4], axis=-1).reshape(*packed.shape[:-1], packed.shape[-1] * 2)


def pack4(codes: np.ndarray) -> np.ndarray:
    codes = np.asarray(codes, np.uint8)
    return (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)


def _hand_blocks(m):
    """Blocks whose scale is 2^0 (amax 6) holding every rounding tie of E2M1, both signs,
    negative values that round to zero, saturation and an all-zero block."""
    ties = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0]          # -> 0, 1, 1, 2, 2, 4, 4, 6
    near = [0.2, 0.3, 0.7, 0.8, 1.1, 1.4, 1.6, 1.9]
    row = np.array(ties + [-t for t in ties] + near + [-0.1, -0.0, 0.0, 0.1, 2.9, 3.1, 4.9, 5.1], np.float32)
    m[2, :32] = synth.bf16_bits(row)
    m[2, 32:64] = synth.bf16_bits(np.array([7.0, 7.9, -7.9] + [1.0] * 29, np.float32))   # amax < 8: scale 2^0, saturation at 6
    m[2, 64:96] = 0
    m[2, 96:128] = synth.bf16_bits(np.full(32, -0.0, np.float32))
    return m


def test_mx4_quantize_both_orientations_bit_exact():
    need_gpu()
    from dropless_mixture_experts_warp_gb300 import binding as B
    batch, rows, C = 2, 256, 384
    m = _hand_blocks(_bf16_matrix_with_every_value(batch * rows, C, 5)).reshape(batch, rows, C)
    codes_t = torch.zeros(batch, C, rows // 2, dtype=torch.uint8, device="cuda")
    sc_t = torch.zeros(batch * C * rows // 32, dtype=torch.uint8, device="cuda")
    codes = torch.zeros(batch * rows, C // 2, dtype=torch.uint8, device="cuda")
    sc = torch.zeros(batch * rows * C // 32, dtype=torch.uint8, device="cuda")
    B.moe_mx4_quantize_cols(bf16_dev(m), batch, rows, C, codes_t, sc_t, codes, sc)
    torch.cuda.synchronize()
    f64 = synth.bf16_to_f32(m).astype(np.float64)
    got_t, sct = unpack4(host(codes_t)), host(sc_t).reshape(batch, -1)
    for b in range(batch):                      # blocks of 32 rows down each column
        ref_c, ref_s = mx.mx4_quantize(f64[b].T)
        assert np.array_equal(got_t[b], ref_c), np.argwhere(got_t[b] != ref_c)[:5]
        assert np.array_equal(scales_from_tiles(sct[b], C, rows), ref_s)
    ref_c, ref_s = mx.mx4_quantize(f64.reshape(batch * rows, C))    # blocks along each row
    got = unpack4(host(codes))
    assert np.array_equal(got, ref_c), np.argwhere(got != ref_c)[:5]
    assert np.array_equal(scales_from_tiles(host(sc), batch * rows, C), ref_s)


@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (256, 256, 512), (384, 128, 256), (128, 256, 1024),
                                   (512, 512, 2048)])
def test_mxf8f4_gemm_matches_dequantised_matmul(M, N, K):
    need_gpu()
    from dropless_mixture_experts_warp_gb300 import binding as B
    rng = np.random.default_rng(M + N + K + 1)
    a = rng.standard_normal((M, K)) * np.exp2(rng.integers(-6, 6, (M, 1)))
    b = rng.standard_normal((N, K)) * np.exp2(rng.integers(-6, 6, (1, K)))
    ac, asc = mx.mx_quantize(a)
    bc, bsc = mx.mx4_quantize(b)
    ref = mx.mx_dequantize(ac, asc) @ mx.mx4_dequantize(bc, bsc).T
    C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()  # noqa: E731
    B.moe_gemm_mxf8f4(dev(ac), dev(sf_tiles(asc)), dev(pack4(bc)), dev(sf_tiles(bsc)), C, M, N, K, status)
    assert B.moe_check_status(status) == 0
    err = rel_err(host(C), ref)
    print(f"M={M} N={N} K={K}: rel err {err:.2e}")
    assert err < 5e-3


CASES = {
    "w4-ragged": synth.small_config("w4-ragged", T=1000, d=256, f=128, E=8, k=2, bias_param=0.7, seed=51),
    "w4-zipf": synth.small_config("w4-zipf", T=777, d=384, f=256, E=16, k=4, score=synth.SIGMOID, bias="zipf",
                                  bias_param=1.0, forced_empty=2, seed=52),
    "w4-shared": synth.small_config("w4-shared", T=384, d=256, f=128, E=16, k=4, score=synth.SIGMOID,
                                    bias="zipf", bias_param=1.0, forced_empty=2, f_shared=128, seed=53),
}


def _run(cfg):
    from dropless_mixture_experts_warp_gb300 import layer
    inp = synth.token_inputs(cfg)
    w_gu_b, w_d_b = synth.all_expert_weights(cfg)
    dims = layer.dims_of(cfg.T, cfg.d, cfg.f, cfg.E, cfg.k, cfg.f_shared, cfg.score, "mxfp8-w4")
    b = layer.allocate(dims)
    w_gu, w_d = bf16_dev(w_gu_b), bf16_dev(w_d_b)
    logits = f32_dev(inp["logits"])
    sh = {}
    if cfg.f_shared:
        s_gu, s_d = synth.shared_weights(cfg)
        sh = {"w_gu_s": bf16_dev(s_gu), "w_d_s": bf16_dev(s_d)}
    x = bf16_dev(inp["x"])
    layer.forward(b, x, logits, w_gu, w_d, **sh)
    layer.backward(b, bf16_dev(inp["dy"]), logits, w_gu, w_d, x=x, **sh)
    layer.check(b)
    return b, inp, w_gu_b, w_d_b


def _a256(x):
    return (x + 255) // 256 * 256


def test_mx4_layer_weight_codes_bit_exact():
    """The layer's weight quantisation: W_gu along d and along 2f, W_d along f and along d,
    as packed E2M1 codes with their SF tiles, bit for bit."""
    need_gpu()
    cfg = CASES["w4-ragged"]
    b, inp, w_gu_b, w_d_b = _run(cfg)
    wq = host(b.wq)
    E, f, d = cfg.E, cfg.f, cfg.d
    n, m = E * 2 * f * d, E * f * d
    assert wq.size >= 2 * (_a256(n // 2) + _a256(n // 32)) + 2 * (_a256(m // 2) + _a256(m // 32))
    regions, off = [], 0
    for elems in (n, n, m, m):
        regions.append((wq[off:off + elems // 2], wq[off + _a256(elems // 2):off + _a256(elems // 2) + elems // 32]))
        off += _a256(elems // 2) + _a256(elems // 32)
    w_gu = synth.bf16_to_f32(w_gu_b).astype(np.float64)
    w_d = synth.bf16_to_f32(w_d_b).astype(np.float64)
    for (codes, scales), mat in zip(regions, (w_gu.reshape(E * 2 * f, d),
                                              np.swapaxes(w_gu, 1, 2).reshape(E * d, 2 * f),
                                              w_d.reshape(E * d, f),
                                              np.swapaxes(w_d, 1, 2).reshape(E * f, d))):
        c, s = mx.mx4_quantize(mat)
        assert np.array_equal(unpack4(codes.reshape(mat.shape[0], -1)), c)
        assert np.array_equal(scales_from_tiles(scales, *mat.shape), s)


@pytest.mark.parametrize("name", list(CASES))
def test_mx4_layer_matches_oracle(name):
    need_gpu()
    cfg = CASES[name]
    b, inp, w_gu_b, w_d_b = _run(cfg)
    f64 = lambda a: synth.bf16_to_f32(a).astype(np.float64)  # noqa: E731
    kw = {"wmatmul": mx.mx_matmul_w4}
    if cfg.f_shared:
        s_gu, s_d = synth.shared_weights(cfg)
        kw.update(w_gu_s=f64(s_gu), w_d_s=f64(s_d))
    fwd = mx.moe_forward_mx(f64(inp["x"]), inp["logits"], f64(w_gu_b), f64(w_d_b), cfg.k, cfg.score, **kw)
    bwd = mx.moe_backward_mx(f64(inp["x"]), inp["logits"], f64(w_gu_b), f64(w_d_b), f64(inp["dy"]), fwd,
                             cfg.k, cfg.score, **kw)
    errs = {"Y": rel_err(host(b.y), fwd["Y"]), "dX": rel_err(host(b.dx), bwd["dX"]),
            "dW_gu": rel_err(host(b.dw_gu), bwd["dW_gu"]), "dW_d": rel_err(host(b.dw_d), bwd["dW_d"]),
            "d_logits": rel_err(host(b.d_logits), bwd["d_logits"])}
    if cfg.f_shared:
        errs["dW_gu_s"] = rel_err(host(b.dw_gu_s), bwd["dW_gu_s"])
        errs["dW_d_s"] = rel_err(host(b.dw_d_s), bwd["dW_d_s"])
    print(f"{name}: " + ", ".join(f"{k} {v:.2e}" for k, v in errs.items()))
    assert all(v <= TOL_MXFP8 for v in errs.values()), errs
    # FP4 weights move the result further from the plain layer than FP8 ones do
    fwd8 = mx.moe_forward_mx(f64(inp["x"]), inp["logits"], f64(w_gu_b), f64(w_d_b), cfg.k, cfg.score,
                             **{k: v for k, v in kw.items() if k != "wmatmul"})
    assert rel_err(host(b.y), fwd8["Y"]) > errs["Y"]
