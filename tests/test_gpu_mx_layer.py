"""The MXFP8 layer path through the C ABI against the MXFP8 oracle.

Codes and scales of what both sides quantise from the same bits (the weights, the
routed x rows, dY's routed rows, in both orientations) are compared bit for bit;
layer outputs and gradients by max|gpu - oracle| / max|oracle| <= 6e-2.  h and dG|dU
are quantised from fp32 on the GPU and from fp64 in the oracle after different
accumulation orders, so their codes may differ by one step; the tolerance covers that.
"""
import numpy as np
import pytest
import torch

from gpu_util import bf16_dev, f32_dev, host, need_gpu, rel_err
from oracle import mx
from dropless_mixture_experts_warp_gb300 import synth

pytestmark = pytest.mark.gpu

TOL_MXFP8 = 6e-2

CASES = {
    "mx-ragged": synth.small_config("mx-ragged", T=1000, d=256, f=128, E=8, k=2, bias_param=0.7, seed=41),
    "mx-zipf": synth.small_config("mx-zipf", T=777, d=384, f=256, E=16, k=4, score=synth.SIGMOID, bias="zipf",
                                  bias_param=1.0, forced_empty=2, seed=42),
    # the declared limits: E = 1024 experts, k = 32
    "mx-limits": synth.small_config("mx-limits", T=512, d=128, f=128, E=1024, k=32, bias_param=1.0, seed=44),
    # DeepSeek-V3-like with the shared expert (T a multiple of 128 for its row blocks)
    "mx-shared": synth.small_config("mx-shared", T=384, d=256, f=128, E=16, k=4, score=synth.SIGMOID,
                                    bias="zipf", bias_param=1.0, forced_empty=2, f_shared=128, seed=43),
}


def _run(cfg, inp=None):
    from dropless_mixture_experts_warp_gb300 import layer
    inp = inp or synth.token_inputs(cfg)
    w_gu_b, w_d_b = synth.all_expert_weights(cfg)
    dims = layer.dims_of(cfg.T, cfg.d, cfg.f, cfg.E, cfg.k, cfg.f_shared, cfg.score, "mxfp8")
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


@pytest.mark.parametrize("name", list(CASES))
def test_mx_layer_matches_mx_oracle(name):
    need_gpu()
    cfg = CASES[name]
    b, inp, w_gu_b, w_d_b = _run(cfg)
    f64 = lambda a: synth.bf16_to_f32(a).astype(np.float64)  # noqa: E731
    kw = {}
    if cfg.f_shared:
        s_gu, s_d = synth.shared_weights(cfg)
        kw = {"w_gu_s": f64(s_gu), "w_d_s": f64(s_d)}
    fwd = mx.moe_forward_mx(f64(inp["x"]), inp["logits"], f64(w_gu_b), f64(w_d_b), cfg.k, cfg.score, **kw)
    bwd = mx.moe_backward_mx(f64(inp["x"]), inp["logits"], f64(w_gu_b), f64(w_d_b), f64(inp["dy"]), fwd,
                             cfg.k, cfg.score, **kw)
    errs = {"Y": rel_err(host(b.y), fwd["Y"]), "dX": rel_err(host(b.dx), bwd["dX"]),
            "dW_gu": rel_err(host(b.dw_gu), bwd["dW_gu"]), "dW_d": rel_err(host(b.dw_d), bwd["dW_d"]),
            "d_logits": rel_err(host(b.d_logits), bwd["d_logits"])}
    if cfg.f_shared:
        errs["dW_gu_s"] = rel_err(host(b.dw_gu_s), bwd["dW_gu_s"])
        errs["dW_d_s"] = rel_err(host(b.dw_d_s), bwd["dW_d_s"])
    assert all(v <= TOL_MXFP8 for v in errs.values()), errs
    split = host(b.split_sizes)
    for e in np.nonzero(split == 0)[0]:
        assert torch.count_nonzero(b.dw_gu[int(e)]) == 0 and torch.count_nonzero(b.dw_d[int(e)]) == 0


def _a256(x):
    return (x + 255) // 256 * 256


def test_mx_weight_codes_and_scales_bit_exact():
    need_gpu()
    from test_gpu_mx import scales_from_tiles
    cfg = CASES["mx-ragged"]
    b, inp, w_gu_b, w_d_b = _run(cfg)
    wq = host(b.wq)
    E, f, d = cfg.E, cfg.f, cfg.d
    n, m = E * 2 * f * d, E * f * d
    regions = []
    off = 0
    for elems in (n, n, m, m):
        regions.append((wq[off:off + elems], wq[off + _a256(elems):off + _a256(elems) + elems // 32]))
        off += _a256(elems) + _a256(elems // 32)
    w_gu = synth.bf16_to_f32(w_gu_b).astype(np.float64)
    w_d = synth.bf16_to_f32(w_d_b).astype(np.float64)
    # W_gu along d, rows [E*2f]
    c, s = mx.mx_quantize(w_gu.reshape(E * 2 * f, d))
    assert np.array_equal(regions[0][0].reshape(E * 2 * f, d), c)
    assert np.array_equal(scales_from_tiles(regions[0][1], E * 2 * f, d), s)
    # W_gu along 2f, stored [E][d][2f]
    c, s = mx.mx_quantize(np.swapaxes(w_gu, 1, 2).reshape(E * d, 2 * f))
    assert np.array_equal(regions[1][0].reshape(E * d, 2 * f), c)
    assert np.array_equal(scales_from_tiles(regions[1][1], E * d, 2 * f), s)
    # W_d along f, rows [E*d]
    c, s = mx.mx_quantize(w_d.reshape(E * d, f))
    assert np.array_equal(regions[2][0].reshape(E * d, f), c)
    assert np.array_equal(scales_from_tiles(regions[2][1], E * d, f), s)
    # W_d along d, stored [E][f][d]
    c, s = mx.mx_quantize(np.swapaxes(w_d, 1, 2).reshape(E * f, d))
    assert np.array_equal(regions[3][0].reshape(E * f, d), c)
    assert np.array_equal(scales_from_tiles(regions[3][1], E * f, d), s)


def _mx_ws_regions(b, R_cap, d, f):
    """(codes, scales) of the step's quantised activations, in the library's order."""
    ws = host(b.mx_ws)
    rd, rf = R_cap * d, R_cap * f
    out, off = {}, 0
    for name, elems in (("xp_rows", rd), ("xp_cols", rd), ("h_rows", rf), ("h_cols", rf), ("dy_rows", rd),
                        ("dy_cols", rd), ("dgu_rows", 2 * rf), ("dgu_cols", 2 * rf)):
        out[name] = (ws[off:off + elems], ws[off + _a256(elems):off + _a256(elems) + elems // 32])
        off += _a256(elems) + _a256(elems // 32)
    return out


@pytest.mark.parametrize("name", ["mx-ragged", "mx-zipf"])
def test_mx_activation_codes_bit_exact(name):
    """Routed x rows and dY rows: row-wise codes (blocks along d) and column-wise codes
    (blocks of 32 rows of the 128-aligned expert segments), padding rows all zero."""
    need_gpu()
    from test_gpu_mx import scales_from_tiles
    cfg = CASES[name]
    b, inp, _, _ = _run(cfg)
    d, f = cfg.d, cfg.f
    r2t = host(b.row_to_token)
    R_cap = r2t.size
    ro = host(b.row_offsets)
    used = int(ro[-1])
    reg = _mx_ws_regions(b, R_cap, d, f)
    for src, rows_key, cols_key in ((inp["x"], "xp_rows", "xp_cols"), (inp["dy"], "dy_rows", "dy_cols")):
        vals = synth.bf16_to_f32(src).astype(np.float64)
        p = np.zeros((used, d))
        live = r2t[:used] >= 0
        p[live] = vals[r2t[:used][live]]
        c, sc = mx.mx_quantize(p)
        codes, sf = reg[rows_key]
        assert np.array_equal(codes.reshape(R_cap, d)[:used], c), rows_key
        assert np.array_equal(scales_from_tiles(sf, R_cap, d)[:used], sc), rows_key
        c, sc = mx.mx_quantize(p.T)
        codes, sf = reg[cols_key]
        assert np.array_equal(codes.reshape(d, R_cap)[:, :used], c), cols_key
        assert np.array_equal(scales_from_tiles(sf, d, R_cap)[:, :used // 32], sc), cols_key


def _mx_oracle(cfg, inp, w_gu_b, w_d_b):
    f64 = lambda a: synth.bf16_to_f32(a).astype(np.float64)  # noqa: E731
    fwd = mx.moe_forward_mx(f64(inp["x"]), inp["logits"], f64(w_gu_b), f64(w_d_b), cfg.k, cfg.score)
    bwd = mx.moe_backward_mx(f64(inp["x"]), inp["logits"], f64(w_gu_b), f64(w_d_b), f64(inp["dy"]), fwd,
                             cfg.k, cfg.score)
    return fwd, bwd


def test_mx_all_tokens_on_one_expert():
    """One expert takes every row (many 128-row tiles), the others are empty."""
    need_gpu()
    cfg = synth.small_config("mx-one", T=300, d=128, f=128, E=4, k=1, seed=44)
    inp = synth.token_inputs(cfg)
    inp["logits"] = inp["logits"].copy()
    inp["logits"][:, 2] += 1e4
    b, inp, w_gu_b, w_d_b = _run(cfg, inp)
    assert list(host(b.split_sizes)) == [0, 0, 300, 0]
    fwd, bwd = _mx_oracle(cfg, inp, w_gu_b, w_d_b)
    for key, got in (("Y", b.y), ("dX", b.dx), ("dW_gu", b.dw_gu), ("dW_d", b.dw_d)):
        assert rel_err(host(got), fwd[key] if key == "Y" else bwd[key]) <= TOL_MXFP8, key
    for e in (0, 1, 3):
        assert torch.count_nonzero(b.dw_gu[e]) == 0 and torch.count_nonzero(b.dw_d[e]) == 0


def test_mx_single_token():
    need_gpu()
    cfg = synth.small_config("mx-single", T=1, d=128, f=128, E=1, k=1, seed=45)
    b, inp, w_gu_b, w_d_b = _run(cfg)
    fwd, bwd = _mx_oracle(cfg, inp, w_gu_b, w_d_b)
    for key, got in (("Y", b.y), ("dX", b.dx), ("dW_gu", b.dw_gu), ("dW_d", b.dw_d)):
        assert rel_err(host(got), fwd[key] if key == "Y" else bwd[key]) <= TOL_MXFP8, key


def test_mx_zero_tokens():
    need_gpu()
    from dropless_mixture_experts_warp_gb300 import layer
    d, f, E, k = 128, 128, 4, 2
    dims = layer.dims_of(0, d, f, E, k, 0, synth.SOFTMAX, "mxfp8")
    b = layer.allocate(dims)
    b.dw_gu.fill_(1.0)
    b.dw_d.fill_(1.0)
    z = torch.empty(0, d, dtype=torch.bfloat16, device="cuda")
    lz = torch.empty(0, E, dtype=torch.float32, device="cuda")
    w_gu = torch.randn(E, 2 * f, d, device="cuda").to(torch.bfloat16)
    w_d = torch.randn(E, d, f, device="cuda").to(torch.bfloat16)
    layer.forward(b, z, lz, w_gu, w_d)
    layer.backward(b, z, lz, w_gu, w_d, x=z)
    layer.check(b)
    assert host(b.split_sizes).sum() == 0 and host(b.row_offsets)[-1] == 0
    assert torch.count_nonzero(b.dw_gu) == 0 and torch.count_nonzero(b.dw_d) == 0


@pytest.mark.parametrize("name", ["mx-ragged", "mx-shared"])
def test_mx_weights_cached_across_micro_batches(name):
    """Weights quantised once per optimiser step and reused by two micro-batches give the same
    bits as quantising them in every forward(), and the cached codes are left untouched."""
    need_gpu()
    import dataclasses
    from dropless_mixture_experts_warp_gb300 import layer
    cfg = CASES[name]
    w_gu_b, w_d_b = synth.all_expert_weights(cfg)
    w_gu, w_d = bf16_dev(w_gu_b), bf16_dev(w_d_b)
    sh = {}
    if cfg.f_shared:
        s_gu, s_d = synth.shared_weights(cfg)
        sh = {"w_gu_s": bf16_dev(s_gu), "w_d_s": bf16_dev(s_d)}
    micro = [synth.token_inputs(cfg), synth.token_inputs(dataclasses.replace(cfg, seed=cfg.seed + 100))]
    dims = layer.dims_of(cfg.T, cfg.d, cfg.f, cfg.E, cfg.k, cfg.f_shared, cfg.score, "mxfp8")
    cached = layer.allocate(dims)
    layer.quantize_weights(cached, w_gu, w_d, **sh)
    wq0 = cached.wq.clone()
    outs = ("y", "dx", "d_logits", "dw_gu", "dw_d")
    for inp in micro:
        x, logits, dy = bf16_dev(inp["x"]), f32_dev(inp["logits"]), bf16_dev(inp["dy"])
        layer.forward(cached, x, logits, w_gu, w_d, weights_cached=True, **sh)
        layer.backward(cached, dy, logits, w_gu, w_d, x=x, **sh)
        layer.check(cached)
        ref, _, _, _ = _run(cfg, inp)
        for key in outs:
            assert torch.equal(getattr(cached, key), getattr(ref, key)), key
        if cfg.f_shared:
            assert torch.equal(cached.dw_gu_s, ref.dw_gu_s) and torch.equal(cached.dw_d_s, ref.dw_d_s)
    assert torch.equal(cached.wq, wq0)
    assert not torch.equal(getattr(_run(cfg, micro[1])[0], "y"), getattr(_run(cfg, micro[0])[0], "y"))


def test_mx_composites_equal_the_per_gemm_calls():
    """moe_grouped_mlp_fwd_mx / moe_grouped_mlp_bwd_mx (used by layer.forward/backward, which the
    tests above compare with the oracle) give the same bits as the six per-GEMM calls in order."""
    need_gpu()
    from dropless_mixture_experts_warp_gb300 import binding as B
    cfg = CASES["mx-zipf"]
    b, inp, w_gu_b, w_d_b = _run(cfg)
    dm = b.dims
    got = {k: getattr(b, k).clone() for k in ("gu", "y_rows", "dxp", "dw_gu", "dw_d", "dw_rows")}
    # repeat the MLP steps through the per-GEMM calls on the same quantised operands
    for name in ("gu", "y_rows", "dxp", "dw_gu", "dw_d", "dw_rows"):
        getattr(b, name).zero_()
    B.moe_gemm_gate_up_mx(dm, b.row_offsets, b.w_rows, b.wq, b.mx_ws, b.gu, b.status)
    B.moe_gemm_down_mx(dm, b.row_offsets, b.wq, b.mx_ws, b.y_rows, b.status)
    B.moe_combine_bwd_mx(dm, bf16_dev(inp["dy"]), b.row_to_token, b.split_sizes, b.row_offsets, b.mx_ws)
    B.moe_gemm_down_dgrad_mx(dm, b.row_offsets, b.w_rows, b.wq, b.mx_ws, b.gu, b.dw_rows, b.workspace, b.status)
    B.moe_gemm_down_wgrad_mx(dm, b.row_offsets, b.mx_ws, b.dw_d, b.status)
    B.moe_gemm_gate_up_dgrad_mx(dm, b.row_offsets, b.wq, b.mx_ws, b.dxp, b.status)
    B.moe_gemm_gate_up_wgrad_mx(dm, b.row_offsets, b.mx_ws, b.dw_gu, b.status)
    assert B.moe_check_status(b.status) == 0
    n = int(host(b.row_offsets)[-1])
    real = torch.zeros(b.rows, dtype=torch.bool, device=b.row_to_token.device)
    real[:n] = b.row_to_token[:n] >= 0              # rows holding a token (padding rows aside)
    for name, ref in got.items():
        cur = getattr(b, name)
        if cur.shape[0] == b.rows:
            assert torch.equal(cur[real], ref[real]), name
        else:
            assert torch.equal(cur, ref), name
    with pytest.raises(B.MoeError):       # an argument error comes back before anything runs
        B.moe_grouped_mlp_bwd_mx(dm, b.row_offsets, b.w_rows, b.wq, b.mx_ws, b.gu, None, b.dw_gu, b.dw_d,
                                 b.dw_rows, b.workspace, b.status)
