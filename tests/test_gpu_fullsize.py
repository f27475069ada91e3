"""Parity at the pages' full workload sizes, sampled where the oracle cannot do it all.

Inputs come from the seeded device generator (the layers are tens of GB); the oracle
receives the same bf16 bits.  Routing, counts and the permutation are compared in
full and bit for bit; Y, dX and d_logits on a random token sample; the weight
gradients on sampled rows/columns of the hottest, the coldest non-empty and two
random experts (fp32 oracle), and in full (exact zeros) for empty experts.
"""
import numpy as np
import pytest
import torch

from gpu_util import LazyExperts, host, need_gpu, rel_err
from oracle import moe_oracle as om
from dropless_mixture_experts_warp_gb300 import synth

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2
TOL_MXFP8 = 6e-2
CASES = [("mixtral", "bf16"), ("qwen30b", "bf16"), ("qwen235b", "bf16"), ("qwen235b-zipf", "bf16"),
         ("dsv3", "bf16"), ("qwen30b", "mxfp8"), ("qwen235b", "mxfp8"), ("qwen235b-zipf", "mxfp8"),
         ("dsv3", "mxfp8")]
N_TOKENS = 96
N_ENTRIES = 12


@pytest.mark.parametrize("name,prec", CASES)
def test_full_size_layer(name, prec):
    need_gpu()
    from dropless_mixture_experts_warp_gb300 import layer
    from oracle import mx
    cfg = synth.CONFIGS[name]
    mx8 = prec == "mxfp8"
    tol = TOL_MXFP8 if mx8 else TOL_BF16
    fwd_fn, bwd_fn = (mx.moe_forward_mx, mx.moe_backward_mx) if mx8 else (om.moe_forward, om.moe_backward)
    wg_fn = mx.expert_wgrad_sampled_mx if mx8 else om.expert_wgrad_sampled
    inp = synth.torch_inputs(cfg, torch.device("cuda"))
    dims = layer.dims_of(cfg.T, cfg.d, cfg.f, cfg.E, cfg.k, cfg.f_shared, cfg.score, prec)
    bufs = layer.allocate(dims)
    sh = {"w_gu_s": inp["w_gu_s"], "w_d_s": inp["w_d_s"]} if cfg.f_shared else {}
    layer.forward(bufs, inp["x"], inp["logits"], inp["w_gu"], inp["w_d"], **sh)
    layer.backward(bufs, inp["dy"], inp["logits"], inp["w_gu"], inp["w_d"], x=inp["x"], **sh)
    layer.check(bufs)

    # ---- routing and permutation, in full, bit for bit
    logits = host(inp["logits"])
    idx, w = om.route(logits, cfg.k, cfg.score, np.float64)
    split, offsets, t2r, _ = om.dispatch(idx, cfg.E)
    assert np.array_equal(host(bufs.topk_idx), idx)
    assert np.array_equal(host(bufs.split_sizes), split)
    assert np.array_equal(host(bufs.offsets), offsets)
    ro = host(bufs.row_offsets).astype(np.int64)
    assert np.array_equal(ro, np.concatenate([[0], np.cumsum((split + 127) // 128 * 128)]))
    assert np.array_equal(host(bufs.token_to_row) - ro[idx], t2r - offsets[idx])
    assert np.abs(host(bufs.topk_w) - w).max() < 2e-6

    # ---- sampled tokens: Y, dX, d_logits
    rng = np.random.default_rng(cfg.seed)
    # each sampled token pulls its k experts to the host (and, for MXFP8, through four
    # weight quantisations each)
    n_tok = 8 if mx8 else (N_TOKENS if cfg.E <= 128 else 32)
    sub = np.sort(rng.choice(cfg.T, size=n_tok, replace=False))
    sub_t = torch.from_numpy(sub).cuda()
    xs = host(inp["x"][sub_t])
    dys = host(inp["dy"][sub_t])
    w_gu = LazyExperts(inp["w_gu"])
    w_d = LazyExperts(inp["w_d"])
    skw = {}
    if cfg.f_shared:
        skw = {"w_gu_s": host(inp["w_gu_s"]), "w_d_s": host(inp["w_d_s"])}
    fwd = fwd_fn(xs, logits[sub], w_gu, w_d, cfg.k, cfg.score, dtype=np.float32, **skw)
    bwd = bwd_fn(xs, logits[sub], w_gu, w_d, dys, fwd, cfg.k, cfg.score, dtype=np.float32, **skw)
    errs = {"Y": rel_err(host(bufs.y[sub_t]), fwd["Y"]),
            "dX": rel_err(host(bufs.dx[sub_t]), bwd["dX"]),
            "d_logits": rel_err(host(bufs.d_logits[sub_t]), bwd["d_logits"])}

    # ---- sampled weight-gradient entries
    x_all, dy_all = inp["x"], inp["dy"]
    order = np.argsort(split, kind="stable")
    nonempty = order[split[order] > 0]
    experts = {int(nonempty[-1]), int(nonempty[0])} | {int(e) for e in rng.choice(nonempty, 2, replace=False)}
    for e in sorted(experts):
        toks = torch.from_numpy(np.nonzero((idx == e).any(axis=1))[0]).cuda()
        rows = rng.choice(2 * cfg.f, size=N_ENTRIES, replace=False)
        cols = rng.choice(cfg.f, size=N_ENTRIES, replace=False)
        tok_np = toks.cpu().numpy()
        s = wg_fn(host(x_all[toks]), logits[tok_np], host(dy_all[toks]), w_gu[e], w_d[e],
                  e, cfg.k, rows, cols, cfg.score, dtype=np.float32)
        errs[f"dW_gu[{e}]"] = rel_err(host(bufs.dw_gu[e][torch.from_numpy(rows).cuda()]), s["dW_gu_rows"])
        errs[f"dW_d[{e}]"] = rel_err(host(bufs.dw_d[e][:, torch.from_numpy(cols).cuda()]), s["dW_d_cols"])
    if cfg.f_shared:
        # the shared expert is one dense group of all T tokens with weight 1: the
        # oracle's sampled single-expert formula with a one-expert router gives it
        fs = cfg.f_shared
        rows = rng.choice(2 * fs, size=N_ENTRIES, replace=False)
        cols = rng.choice(fs, size=N_ENTRIES, replace=False)
        s = wg_fn(host(x_all), np.zeros((cfg.T, 1), np.float32), host(dy_all),
                  skw["w_gu_s"], skw["w_d_s"], 0, 1, rows, cols, om.SOFTMAX, dtype=np.float32)
        errs["dW_gu_s"] = rel_err(host(bufs.dw_gu_s[torch.from_numpy(rows).cuda()]), s["dW_gu_rows"])
        errs["dW_d_s"] = rel_err(host(bufs.dw_d_s[:, torch.from_numpy(cols).cuda()]), s["dW_d_cols"])
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, errs
    for e in np.nonzero(split == 0)[0]:
        assert torch.count_nonzero(bufs.dw_gu[int(e)]) == 0 and torch.count_nonzero(bufs.dw_d[int(e)]) == 0
