"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Routing outputs, counts and the permutation are compared bit for bit; floating
point outputs by max|gpu - oracle| / max|oracle| <= 2e-2 (bf16 path).
"""
import numpy as np
import pytest
import torch

from gpu_util import bf16_dev, f32_dev, host, need_gpu, rel_err
from oracle import moe_oracle as om
from dropless_mixture_experts_warp_gb300 import synth

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2

CASES = {
    "tiny": synth.CONFIGS["tiny"],
    # several M/N/K tiles per expert, ragged tails, N tiles of 64 and 128 columns
    "ragged": synth.small_config("ragged", T=1000, d=256, f=192, E=8, k=2, bias_param=0.7, seed=11),
    "sigmoid": synth.small_config("sigmoid", T=777, d=384, f=256, E=16, k=4, score=synth.SIGMOID,
                                  bias="zipf", bias_param=1.0, forced_empty=2, seed=12),
    "many": synth.small_config("many", T=512, d=128, f=128, E=64, k=8, bias="zipf", bias_param=1.1,
                               forced_empty=3, seed=13),
    # DeepSeek-V3-like: sigmoid scores, Zipf load, forced-empty experts, shared expert
    # the declared limits: E = 1024 experts, k = 32 (about 16 rows per expert, many empty)
    "limits": synth.small_config("limits", T=512, d=128, f=64, E=1024, k=32, bias_param=1.0, seed=14),
    "shared": synth.small_config("shared", T=300, d=256, f=128, E=16, k=4, score=synth.SIGMOID,
                                 bias="zipf", bias_param=1.0, forced_empty=2, f_shared=192, seed=14),
}


def run_layer(cfg, inp=None, weights=None, repeat=1):
    from dropless_mixture_experts_warp_gb300 import layer
    inp = inp or synth.token_inputs(cfg)
    w_gu_b, w_d_b = weights or synth.all_expert_weights(cfg)
    dims = layer.dims_of(cfg.T, cfg.d, cfg.f, cfg.E, cfg.k, cfg.f_shared, cfg.score)
    bufs = layer.allocate(dims)
    x, dy, logits = bf16_dev(inp["x"]), bf16_dev(inp["dy"]), f32_dev(inp["logits"])
    w_gu, w_d = bf16_dev(w_gu_b), bf16_dev(w_d_b)
    sh = {}
    if cfg.f_shared:
        s_gu, s_d = synth.shared_weights(cfg)
        sh = {"w_gu_s": bf16_dev(s_gu), "w_d_s": bf16_dev(s_d)}
    keys = ["y", "dx", "dw_gu", "dw_d", "d_logits", "topk_idx", "topk_w", "split_sizes", "offsets",
            "row_offsets", "token_to_row", "row_to_token", "w_rows", "xp", "dw_rows"]
    if cfg.f_shared:
        keys += ["dw_gu_s", "dw_d_s"]
    outs = []
    for _ in range(repeat):
        layer.forward(bufs, x, logits, w_gu, w_d, **sh)
        layer.backward(bufs, dy, logits, w_gu, w_d, x=x, **sh)
        layer.check(bufs)
        outs.append({k: getattr(bufs, k).clone() for k in keys})
    return bufs, outs, (inp, w_gu_b, w_d_b)


def oracle_layer(cfg, inp, w_gu_b, w_d_b):
    x = synth.bf16_to_f32(inp["x"]).astype(np.float64)
    dy = synth.bf16_to_f32(inp["dy"]).astype(np.float64)
    w_gu = synth.bf16_to_f32(w_gu_b).astype(np.float64)
    w_d = synth.bf16_to_f32(w_d_b).astype(np.float64)
    kw = {}
    if cfg.f_shared:
        s_gu, s_d = synth.shared_weights(cfg)
        kw = {"w_gu_s": synth.bf16_to_f32(s_gu).astype(np.float64),
              "w_d_s": synth.bf16_to_f32(s_d).astype(np.float64)}
    fwd = om.moe_forward(x, inp["logits"], w_gu, w_d, cfg.k, cfg.score, **kw)
    bwd = om.moe_backward(x, inp["logits"], w_gu, w_d, dy, fwd, cfg.k, cfg.score, **kw)
    return fwd, bwd


@pytest.mark.parametrize("name", list(CASES))
def test_routing_and_permutation_bit_exact(name):
    need_gpu()
    cfg = CASES[name]
    bufs, outs, (inp, _, _) = run_layer(cfg)
    o = outs[0]
    idx, w = om.route(inp["logits"], cfg.k, cfg.score)
    split, offsets, t2r, r2t = om.dispatch(idx, cfg.E)
    assert np.array_equal(host(o["topk_idx"]), idx)
    assert np.array_equal(host(o["split_sizes"]), split)
    assert np.array_equal(host(o["offsets"]), offsets)
    ro = host(o["row_offsets"]).astype(np.int64)
    assert np.array_equal(ro, np.concatenate([[0], np.cumsum((split + 127) // 128 * 128)]))
    # same rank of every (token, slot) inside its expert segment
    g_t2r = host(o["token_to_row"]).astype(np.int64)
    e_of = idx
    assert np.array_equal(g_t2r - ro[e_of], t2r - offsets[e_of])
    assert np.abs(host(o["topk_w"]) - w).max() < 2e-6
    # permuted rows are exact copies; padding rows are zero and marked
    x = synth.bf16_to_f32(inp["x"])
    xp = host(o["xp"])
    r2t_g = host(o["row_to_token"])
    w_rows = host(o["w_rows"])
    for e in range(cfg.E):
        a, n, b = ro[e], split[e], ro[e + 1]
        toks = r2t[offsets[e]:offsets[e] + n]
        assert np.array_equal(r2t_g[a:a + n], toks)
        assert np.array_equal(xp[a:a + n], x[toks])
        assert np.all(r2t_g[a + n:b] == -1)
        assert np.all(xp[a + n:b] == 0)
        assert np.all(w_rows[a + n:b] == 0)


def test_identity_round_trip_bit_exact():
    """combine(permute(x)) == k * x exactly (unweighted combine of the copies)."""
    need_gpu()
    from dropless_mixture_experts_warp_gb300 import binding as B
    cfg = CASES["many"]
    bufs, outs, (inp, _, _) = run_layer(cfg)
    out = torch.empty_like(bufs.y)
    B.moe_combine_fwd(bufs.dims, bufs.xp, bufs.token_to_row, None, out)
    torch.cuda.synchronize()
    x = synth.bf16_to_f32(inp["x"])
    assert np.array_equal(host(out), np.float32(cfg.k) * x)


@pytest.mark.parametrize("name", list(CASES))
def test_layer_fwd_bwd_matches_oracle(name):
    need_gpu()
    cfg = CASES[name]
    _, outs, (inp, w_gu_b, w_d_b) = run_layer(cfg)
    o = outs[0]
    fwd, bwd = oracle_layer(cfg, inp, w_gu_b, w_d_b)
    errs = {
        "Y": rel_err(host(o["y"]), fwd["Y"]),
        "dX": rel_err(host(o["dx"]), bwd["dX"]),
        "dW_gu": rel_err(host(o["dw_gu"]), bwd["dW_gu"]),
        "dW_d": rel_err(host(o["dw_d"]), bwd["dW_d"]),
        "d_logits": rel_err(host(o["d_logits"]), bwd["d_logits"]),
    }
    if cfg.f_shared:
        errs["dW_gu_s"] = rel_err(host(o["dw_gu_s"]), bwd["dW_gu_s"])
        errs["dW_d_s"] = rel_err(host(o["dw_d_s"]), bwd["dW_d_s"])
    assert all(v <= TOL_BF16 for v in errs.values()), errs
    # experts with no token get an exactly zero weight gradient
    split = host(o["split_sizes"])
    for e in np.nonzero(split == 0)[0]:
        assert np.all(host(o["dw_gu"][e]) == 0) and np.all(host(o["dw_d"][e]) == 0)


def test_deterministic_bitwise():
    need_gpu()
    _, outs, _ = run_layer(CASES["ragged"], repeat=2)
    for key in ("y", "dx", "dw_gu", "dw_d", "d_logits", "dw_rows"):
        assert torch.equal(outs[0][key], outs[1][key]), key


def test_all_tokens_on_one_expert():
    need_gpu()
    cfg = synth.small_config("one", T=300, d=128, f=64, E=4, k=1, seed=21)
    inp = synth.token_inputs(cfg)
    inp["logits"] = inp["logits"].copy()
    inp["logits"][:, 2] += 1e4          # every token picks expert 2
    _, outs, (inp, w_gu_b, w_d_b) = run_layer(cfg, inp=inp)
    o = outs[0]
    assert list(host(o["split_sizes"])) == [0, 0, 300, 0]
    fwd, bwd = oracle_layer(cfg, inp, w_gu_b, w_d_b)
    assert rel_err(host(o["y"]), fwd["Y"]) <= TOL_BF16
    assert rel_err(host(o["dw_gu"]), bwd["dW_gu"]) <= TOL_BF16
    assert np.all(host(o["dw_d"][0]) == 0)


def test_zero_tokens():
    need_gpu()
    cfg = synth.small_config("empty", T=0, d=128, f=64, E=4, k=2, seed=22)
    from dropless_mixture_experts_warp_gb300 import layer
    dims = layer.dims_of(0, cfg.d, cfg.f, cfg.E, cfg.k)
    bufs = layer.allocate(dims)
    bufs.dw_gu.fill_(1.0)
    bufs.dw_d.fill_(1.0)
    z = torch.empty(0, cfg.d, dtype=torch.bfloat16, device="cuda")
    lz = torch.empty(0, cfg.E, dtype=torch.float32, device="cuda")
    w_gu = torch.randn(cfg.E, 2 * cfg.f, cfg.d, device="cuda").to(torch.bfloat16)
    w_d = torch.randn(cfg.E, cfg.d, cfg.f, device="cuda").to(torch.bfloat16)
    layer.forward(bufs, z, lz, w_gu, w_d)
    layer.backward(bufs, z, lz, w_gu, w_d)
    layer.check(bufs)
    assert host(bufs.split_sizes).sum() == 0 and host(bufs.row_offsets)[-1] == 0
    assert torch.count_nonzero(bufs.dw_gu) == 0 and torch.count_nonzero(bufs.dw_d) == 0


def test_single_expert_single_token():
    need_gpu()
    cfg = synth.small_config("single", T=1, d=128, f=64, E=1, k=1, seed=23)
    _, outs, (inp, w_gu_b, w_d_b) = run_layer(cfg)
    fwd, bwd = oracle_layer(cfg, inp, w_gu_b, w_d_b)
    o = outs[0]
    assert rel_err(host(o["y"]), fwd["Y"]) <= TOL_BF16
    assert rel_err(host(o["dx"]), bwd["dX"]) <= TOL_BF16
    assert rel_err(host(o["dw_gu"]), bwd["dW_gu"]) <= TOL_BF16
    assert rel_err(host(o["dw_d"]), bwd["dW_d"]) <= TOL_BF16


def test_shared_expert_zero_tokens_gives_zero_gradients():
    need_gpu()
    from dropless_mixture_experts_warp_gb300 import layer
    dims = layer.dims_of(0, 128, 64, 4, 2, 64, "sigmoid")
    bufs = layer.allocate(dims)
    bufs.dw_gu_s.fill_(1.0)
    bufs.dw_d_s.fill_(1.0)
    z = torch.empty(0, 128, dtype=torch.bfloat16, device="cuda")
    lz = torch.empty(0, 4, dtype=torch.float32, device="cuda")
    w_gu = torch.randn(4, 128, 128, device="cuda").to(torch.bfloat16)
    w_d = torch.randn(4, 128, 64, device="cuda").to(torch.bfloat16)
    s_gu = torch.randn(128, 128, device="cuda").to(torch.bfloat16)
    s_d = torch.randn(128, 64, device="cuda").to(torch.bfloat16)
    layer.forward(bufs, z, lz, w_gu, w_d, w_gu_s=s_gu, w_d_s=s_d)
    layer.backward(bufs, z, lz, w_gu, w_d, x=z, w_gu_s=s_gu, w_d_s=s_d)
    layer.check(bufs)
    assert torch.count_nonzero(bufs.dw_gu_s) == 0 and torch.count_nonzero(bufs.dw_d_s) == 0


def test_bounded_wait_times_out_and_context_survives():
    """A device wait on a barrier nothing arrives on gives up and reports MOE_ERR_TIMEOUT."""
    need_gpu()
    from dropless_mixture_experts_warp_gb300 import binding as B
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.moe_test_wait_timeout(status, 1 << 24)       # about 8 ms at 2 GHz
    assert B.moe_check_status(status) == 6         # MOE_ERR_TIMEOUT
    # the context is still usable: a GEMM after the timeout runs and is right
    A = torch.randn(128, 64, device="cuda").to(torch.bfloat16)
    Bm = torch.randn(64, 64, device="cuda").to(torch.bfloat16)
    C = torch.empty(128, 64, dtype=torch.bfloat16, device="cuda")
    ok = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.moe_gemm_bf16(A, Bm, C, 128, 64, 64, 0, 0, ok)
    assert B.moe_check_status(ok) == 0
    ref = A.float() @ Bm.float().T
    assert rel_err(host(C), host(ref).astype(np.float64)) < 1e-2
