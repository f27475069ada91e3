"""Group-limited sigmoid routing (a DeepSeek-V3 router variant) on the GPU against the
oracle.  Selection is decided in fp32 on both sides, but the two sigmoids may round
differently in the last bit, so indices are compared bit for bit on every token whose
group and expert decisions clear a margin of a few fp32 ulps (at least 98 % of the
tokens); every other token's choice must be one that lies within that margin of both
cuts (route_util.assert_valid_near_ties)."""
import numpy as np
import pytest
import torch

from gpu_util import bf16_dev, f32_dev, host, need_gpu, rel_err
from route_util import assert_valid_near_ties, decision_margins
from oracle import moe_oracle as om
from dropless_mixture_experts_warp_gb300 import synth

pytestmark = pytest.mark.gpu
MARGIN = 2e-6
TOL_BF16 = 2e-2


def _route_gpu(T, E, k, logits, bias, n_group, topk_group, scale):
    from dropless_mixture_experts_warp_gb300 import binding as B, layer
    dims = layer.dims_of(T, 128, 128, E, k, 0, synth.SIGMOID)
    b = layer.allocate(dims)
    B.moe_route_topk_grouped(dims, f32_dev(logits), f32_dev(bias), n_group, topk_group, scale, b.topk_idx,
                             b.topk_w, b.split_sizes, b.offsets, b.row_offsets, b.workspace, b.status)
    layer.check(b)
    return host(b.topk_idx), host(b.topk_w), host(b.split_sizes)


@pytest.mark.parametrize("T,E,k,n_group,topk_group", [(3000, 256, 8, 8, 4), (1000, 64, 6, 4, 2),
                                                      (777, 32, 4, 16, 3), (500, 128, 8, 32, 8),
                                                      (640, 16, 2, 1, 1)])
def test_grouped_route_matches_oracle(T, E, k, n_group, topk_group):
    need_gpu()
    rng = np.random.default_rng(T + E)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    bias = (rng.standard_normal(E) * 0.2).astype(np.float32)
    idx, w, split = _route_gpu(T, E, k, logits, bias, n_group, topk_group, 2.5)
    ref_idx, ref_w = om.route_grouped(logits, k, n_group, topk_group, bias, 2.5)
    decided = decision_margins(logits, k, n_group, topk_group, bias) > MARGIN
    print(f"T={T} E={E}: {int((~decided).sum())} tokens within {MARGIN} of a cut")
    assert decided.mean() > 0.98
    assert np.array_equal(idx[decided], ref_idx[decided])
    assert np.abs(w[decided] - ref_w[decided]).max() <= 1e-5 * np.abs(ref_w).max()
    # the other tokens: a choice an exact router could make, within the margin of both cuts
    assert_valid_near_ties(idx, logits, k, n_group, topk_group, bias, MARGIN, np.nonzero(~decided)[0])
    assert np.array_equal(split, np.bincount(idx.ravel(), minlength=E))
    np.testing.assert_allclose(w.sum(axis=1), 2.5, rtol=1e-5)


def test_grouped_layer_fwd_bwd_matches_oracle():
    """The whole bf16 layer with the grouped router, a selection bias and a routed scale."""
    need_gpu()
    from dropless_mixture_experts_warp_gb300 import layer
    cfg = synth.small_config("grouped", T=600, d=256, f=128, E=16, k=4, score=synth.SIGMOID, seed=61)
    inp = synth.token_inputs(cfg)
    rng = np.random.default_rng(62)
    bias = (rng.standard_normal(cfg.E) * 0.1).astype(np.float32)
    n_group, topk_group, scale = 4, 2, 2.5
    assert (decision_margins(inp["logits"], cfg.k, n_group, topk_group, bias) > MARGIN).all()
    w_gu_b, w_d_b = synth.all_expert_weights(cfg)
    dims = layer.dims_of(cfg.T, cfg.d, cfg.f, cfg.E, cfg.k, 0, cfg.score)
    b = layer.allocate(dims)
    x, dy, logits = bf16_dev(inp["x"]), bf16_dev(inp["dy"]), f32_dev(inp["logits"])
    w_gu, w_d = bf16_dev(w_gu_b), bf16_dev(w_d_b)
    gr = {"n_group": n_group, "topk_group": topk_group, "bias": f32_dev(bias), "routed_scale": scale}
    layer.forward(b, x, logits, w_gu, w_d, grouped=gr)
    layer.backward(b, dy, logits, w_gu, w_d, x=x, grouped=gr)
    layer.check(b)
    f64 = lambda a: synth.bf16_to_f32(a).astype(np.float64)  # noqa: E731
    og = {"n_group": n_group, "topk_group": topk_group, "bias": bias, "routed_scale": scale}
    fwd = om.moe_forward(f64(inp["x"]), inp["logits"], f64(w_gu_b), f64(w_d_b), cfg.k, cfg.score, grouped=og)
    bwd = om.moe_backward(f64(inp["x"]), inp["logits"], f64(w_gu_b), f64(w_d_b), f64(inp["dy"]), fwd, cfg.k,
                          cfg.score, grouped=og)
    assert np.array_equal(host(b.topk_idx), fwd["idx"])
    errs = {"Y": rel_err(host(b.y), fwd["Y"]), "dX": rel_err(host(b.dx), bwd["dX"]),
            "dW_gu": rel_err(host(b.dw_gu), bwd["dW_gu"]), "dW_d": rel_err(host(b.dw_d), bwd["dW_d"]),
            "d_logits": rel_err(host(b.d_logits), bwd["d_logits"])}
    assert all(v <= TOL_BF16 for v in errs.values()), errs


def test_grouped_route_rejects_bad_options():
    need_gpu()
    from dropless_mixture_experts_warp_gb300 import binding as B, layer
    dims = layer.dims_of(64, 128, 128, 16, 4, 0, synth.SIGMOID)
    b = layer.allocate(dims)
    lg = torch.zeros(64, 16, device="cuda")
    for n_group, topk_group, scale in ((3, 1, 1.0), (4, 0, 1.0), (4, 5, 1.0), (16, 2, 1.0), (4, 1, 0.0),
                                       (64, 1, 1.0)):
        with pytest.raises(B.MoeError):
            B.moe_route_topk_grouped(dims, lg, None, n_group, topk_group, scale, b.topk_idx, b.topk_w,
                                     b.split_sizes, b.offsets, b.row_offsets, b.workspace, b.status)
