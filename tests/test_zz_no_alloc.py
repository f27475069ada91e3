"""moe_gemm_down_dgrad_noalloc against moe_gemm_down_dgrad and the oracle, through the C ABI.

The no-allocation variant serves callers that cannot call cudaMalloc (a host
program that owns all device memory and gives plugins no allocator, or a loop where
allocations are not allowed); it keeps the per-tile dw partials in the library's
static device array instead of a caller workspace.  It launches the same kernels as
the workspace version, so it must give the same bits, call after call, although
every call reuses (and leaves behind) the same array; and both must match the
oracle's dG|dU and dw.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

from gpu_util import bf16_dev, f32_dev, host, need_gpu, rel_err
from oracle import moe_oracle as om
from dropless_mixture_experts_warp_gb300 import synth

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2


def _prepare(cfg, dy_seed=None):
    """Forward pass and dY rows through the existing entry points; dy_seed redraws dY."""
    from dropless_mixture_experts_warp_gb300 import binding as B, layer
    inp = synth.token_inputs(cfg)
    if dy_seed is not None:
        rng = np.random.default_rng(dy_seed)
        inp["dy"] = synth.bf16_bits(rng.standard_normal((cfg.T, cfg.d)).astype(np.float32))
    w_gu_b, w_d_b = synth.all_expert_weights(cfg)
    dims = layer.dims_of(cfg.T, cfg.d, cfg.f, cfg.E, cfg.k, 0, cfg.score)
    b = layer.allocate(dims)
    w_gu, w_d = bf16_dev(w_gu_b), bf16_dev(w_d_b)
    layer.forward(b, bf16_dev(inp["x"]), f32_dev(inp["logits"]), w_gu, w_d)
    B.moe_combine_bwd(dims, bf16_dev(inp["dy"]), b.token_to_row, b.split_sizes, b.row_offsets, b.dy_rows)
    layer.check(b)
    return dims, b, w_d, (inp, w_gu_b, w_d_b)


def _oracle(cfg, inp, w_gu_b, w_d_b):
    f64 = lambda a: synth.bf16_to_f32(a).astype(np.float64)  # noqa: E731
    x, wg, wd = f64(inp["x"]), f64(w_gu_b), f64(w_d_b)
    fwd = om.moe_forward(x, inp["logits"], wg, wd, cfg.k, cfg.score)
    return om.moe_backward(x, inp["logits"], wg, wd, f64(inp["dy"]), fwd, cfg.k, cfg.score)


def _both(dims, b, w_d):
    from dropless_mixture_experts_warp_gb300 import binding as B
    dgu_ref, dw_ref = torch.zeros_like(b.dgu), torch.zeros_like(b.dw_rows)
    B.moe_gemm_down_dgrad(dims, b.dy_rows, b.row_offsets, b.w_rows, w_d, b.gu, dgu_ref, dw_ref, b.workspace,
                          b.status)
    dgu, dw = torch.full_like(b.dgu, float("nan")), torch.full_like(b.dw_rows, float("nan"))
    B.moe_gemm_down_dgrad_noalloc(dims, b.dy_rows, b.row_offsets, b.w_rows, w_d, b.gu, dgu, dw, b.status)
    assert B.moe_check_status(b.status) == 0
    return dgu, dw, dgu_ref, dw_ref


def _check_against_oracle(cfg, b, dgu, dw, inputs):
    bwd = _oracle(cfg, *inputs)
    t2r = host(b.token_to_row).astype(np.int64)          # [T, k] rows of every (token, slot)
    gpu_dgu = host(dgu)[t2r]                               # [T, k, 2f]
    gpu_dw = host(dw)[t2r]                                 # [T, k]
    e_dgu = rel_err(gpu_dgu, bwd["dGU"])
    e_dw = rel_err(gpu_dw, bwd["dw"])
    print(f"{cfg.name}: dGU rel err {e_dgu:.2e}, dw rel err {e_dw:.2e} (limit {TOL_BF16})")
    assert e_dgu <= TOL_BF16 and e_dw <= TOL_BF16


def test_noalloc_dgrad_bitwise_equal_to_workspace_version_and_to_oracle():
    """Three calls in a row: a larger case that fills more of the shared array, then two
    smaller ones on the same shape with different dY, so the later calls find stale
    partials of earlier calls in the array.  Each is bit for bit the workspace call's
    result (same kernels) and within the bf16 tolerance of the oracle."""
    need_gpu()
    cases = [(synth.small_config("noalloc-a", T=1000, d=256, f=192, E=8, k=2, seed=31), None),   # BN 64: single CTA
             (synth.small_config("noalloc-b", T=300, d=128, f=256, E=4, k=2, seed=32), None),    # BN 256: CTA pair
             (synth.small_config("noalloc-b", T=300, d=128, f=256, E=4, k=2, seed=32), 77)]      # same, new dY
    prev_dw = None
    for cfg, dy_seed in cases:
        dims, b, w_d, inputs = _prepare(cfg, dy_seed)
        n = int(host(b.row_offsets)[-1])                 # rows past n are never written
        real = torch.zeros_like(b.row_to_token, dtype=torch.bool)
        real[:n] = b.row_to_token[:n] >= 0               # rows that hold a token (not padding)
        dgu, dw, dgu_ref, dw_ref = _both(dims, b, w_d)
        assert torch.equal(dgu[real], dgu_ref[real])
        assert torch.equal(dw[real], dw_ref[real])
        _check_against_oracle(cfg, b, dgu, dw, inputs)
        if dy_seed is not None:
            assert not torch.equal(dw[real], prev_dw[real])    # the new dY reached the result
        prev_dw = dw


def test_noalloc_rejects_problems_beyond_its_scratch():
    need_gpu()
    from dropless_mixture_experts_warp_gb300 import binding as B
    assert B.moe_noalloc_scratch_bytes() == 8 << 20
    # rows x (f / 64) partials: 2^21 floats fit, this needs about 3.1e6
    dims = B.make_dims(16384, 128, 1536 + 64, 8, 8)
    with pytest.raises(B.MoeError) as e:
        B.moe_gemm_down_dgrad_noalloc(dims, 16, 16, 16, 16, 16, 16, 16, 16, stream=0)
    assert e.value.status == 8
