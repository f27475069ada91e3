"""moe_gemm_down_dgrad_noalloc against moe_gemm_down_dgrad, through the C ABI.

The no-allocation variant serves callers that cannot call cudaMalloc (a host
program that owns all device memory and gives plugins no allocator, or a loop where
allocations are not allowed); it keeps the per-tile dw partials in the library's
static device array instead of a caller workspace.  It must give the same dgu and
dw_rows as the workspace version, call after call, although every call reuses (and
leaves behind) the same array.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

from gpu_util import bf16_dev, f32_dev, host, need_gpu, rel_err
from dropless_mixture_experts_warp_gb300 import synth

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2


def _prepare(cfg):
    """Forward pass and dY rows through the existing entry points."""
    from dropless_mixture_experts_warp_gb300 import binding as B, layer
    inp = synth.token_inputs(cfg)
    w_gu_b, w_d_b = synth.all_expert_weights(cfg)
    dims = layer.dims_of(cfg.T, cfg.d, cfg.f, cfg.E, cfg.k, 0, cfg.score)
    b = layer.allocate(dims)
    w_gu, w_d = bf16_dev(w_gu_b), bf16_dev(w_d_b)
    layer.forward(b, bf16_dev(inp["x"]), f32_dev(inp["logits"]), w_gu, w_d)
    B.moe_combine_bwd(dims, bf16_dev(inp["dy"]), b.token_to_row, b.split_sizes, b.row_offsets, b.dy_rows)
    layer.check(b)
    return dims, b, w_d


def test_noalloc_dgrad_matches_workspace_version_two_calls_in_a_row():
    need_gpu()
    from dropless_mixture_experts_warp_gb300 import binding as B
    cases = [synth.small_config("noalloc-a", T=1000, d=256, f=192, E=8, k=2, seed=31),
             synth.small_config("noalloc-b", T=300, d=128, f=256, E=4, k=2, seed=32)]
    for cfg in cases:                      # the second call finds the first call's partials
        dims, b, w_d = _prepare(cfg)
        n = int(host(b.row_offsets)[-1])
        dgu_ref = torch.zeros_like(b.dgu)
        dw_ref = torch.zeros_like(b.dw_rows)
        B.moe_gemm_down_dgrad(dims, b.dy_rows, b.row_offsets, b.w_rows, w_d, b.gu, dgu_ref, dw_ref,
                              b.workspace, b.status)
        dgu = torch.zeros_like(b.dgu)
        dw = torch.zeros_like(b.dw_rows)
        B.moe_gemm_down_dgrad_noalloc(dims, b.dy_rows, b.row_offsets, b.w_rows, w_d, b.gu, dgu, dw, b.status)
        assert B.moe_check_status(b.status) == 0
        assert rel_err(host(dgu[:n]), host(dgu_ref[:n]).astype(np.float64)) <= TOL_BF16
        assert rel_err(host(dw[:n]), host(dw_ref[:n]).astype(np.float64)) <= TOL_BF16


def test_noalloc_rejects_problems_beyond_its_scratch():
    need_gpu()
    from dropless_mixture_experts_warp_gb300 import binding as B
    assert B.moe_noalloc_scratch_bytes() == 8 << 20
    # rows x (f / 64) partials: 2^21 floats fit, this needs about 3.1e6
    dims = B.make_dims(16384, 128, 1536 + 64, 8, 8)
    with pytest.raises(B.MoeError) as e:
        B.moe_gemm_down_dgrad_noalloc(dims, 16, 16, 16, 16, 16, 16, 16, 16, stream=0)
    assert e.value.status == 8
