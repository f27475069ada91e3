"""Parity at the pages' full workload sizes, sampled where the oracle cannot do it all.

Inputs come from the seeded device generator (the layers are tens of GB); the oracle
receives the same bf16 bits.  Routing, counts and the permutation are compared in full and
bit for bit (the group-limited router: bit for bit on tokens clear of a near-tie, checked for
validity on the rest).  Y, dX and d_logits are compared on 256 random tokens; the weight
gradients in full for the hottest, the coldest non-empty and one random expert, and in full
(exact zeros) for empty experts.  FP8 x FP4 experts (mxfp8-w4) are checked the same way
against the MXFP8 oracle with E2M1 weight operands.  The shared expert's weight gradients are compared on
sampled rows and columns.

The oracle goes through the experts one at a time (oracle.expert_rows / expert_rows_mx, the
loop bodies of the layer oracle), spread over host threads: in MXFP8 each expert's weights
are quantised in four orientations (seconds per DeepSeek-V3 expert), so this is what makes
a few hundred tokens affordable.  The errors of every case are printed (pytest -s).
"""
import concurrent.futures as cf
import os

import numpy as np
import pytest
import torch

from gpu_util import host, need_gpu, rel_err
from oracle import moe_oracle as om
from route_util import assert_valid_near_ties, decision_margins
from dropless_mixture_experts_warp_gb300 import synth

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2
TOL_MXFP8 = 6e-2
MARGIN = 2e-6
CASES = [("mixtral", "bf16"), ("qwen30b", "bf16"), ("qwen235b", "bf16"), ("qwen235b-zipf", "bf16"),
         ("dsv3", "bf16"), ("dsv3-grouped", "bf16"), ("qwen30b", "mxfp8"), ("qwen235b", "mxfp8"),
         ("qwen235b-zipf", "mxfp8"), ("dsv3", "mxfp8"), ("qwen235b", "mxfp8-w4"), ("dsv3", "mxfp8-w4")]
N_TOKENS = 256
N_ENTRIES = 12
THREADS = max(1, min(8, os.cpu_count() or 1))   # each holds about 1 GB of one expert's arrays


def _routing(cfg, logits, bufs):
    """Oracle routing, compared with the GPU's; returns (idx, w, tokens whose choice differs)."""
    gr = synth.grouped_options(cfg)
    if gr is None:
        idx, w = om.route(logits, cfg.k, cfg.score, np.float64)
    else:
        idx, w = om.route_grouped(logits, cfg.k, gr["n_group"], gr["topk_group"], gr["bias"], gr["routed_scale"],
                                  np.float64)
    g_idx = host(bufs.topk_idx)
    differ = np.nonzero((g_idx != idx).any(axis=1))[0]
    if gr is None:
        assert differ.size == 0
    else:
        decided = decision_margins(logits, cfg.k, gr["n_group"], gr["topk_group"], gr["bias"]) > MARGIN
        assert decided.mean() > 0.98 and not np.isin(differ, np.nonzero(decided)[0]).any()
        assert_valid_near_ties(g_idx, logits, cfg.k, gr["n_group"], gr["topk_group"], gr["bias"], MARGIN, differ)
        print(f"{cfg.name}: {int((~decided).sum())} tokens near a routing cut, {differ.size} chosen differently")
    split, offsets, t2r, _ = om.dispatch(idx, cfg.E)
    if differ.size == 0:
        assert np.array_equal(host(bufs.split_sizes), split)
        assert np.array_equal(host(bufs.offsets), offsets)
        ro = host(bufs.row_offsets).astype(np.int64)
        assert np.array_equal(ro, np.concatenate([[0], np.cumsum((split + 127) // 128 * 128)]))
        assert np.array_equal(host(bufs.token_to_row) - ro[idx], t2r - offsets[idx])
    keep = np.setdiff1d(np.arange(cfg.T), differ)
    assert np.abs(host(bufs.topk_w)[keep] - w[keep]).max() < 2e-6 * max(1.0, float(np.abs(w).max()))
    # experts whose rows differ between the two sides: reached by a differing choice on either
    touched = set(np.unique(idx[differ]).tolist()) | set(np.unique(g_idx[differ]).tolist())
    return idx, w, differ, touched


def _expert_job(e, rows_t, rows_j, full, ctx):
    """Oracle rows of expert e (forward and backward) on the given (token, slot) pairs."""
    from oracle import mx
    inp, w, mx8, w4 = ctx["inp"], ctx["w"], ctx["mx8"], ctx["w4"]
    toks = torch.from_numpy(rows_t).to(inp["x"].device)
    x = host(inp["x"][toks])
    dy = host(inp["dy"][toks])
    w_gu = inp["w_gu"][e].float().cpu().numpy()
    w_d = inp["w_d"][e].float().cpu().numpy()
    if mx8:   # FP8 x FP4 experts: the products with a weight operand take E2M1 weights
        return mx.expert_rows_mx(x, w[rows_t, rows_j], dy, w_gu, w_d, dtype=np.float32, full=full,
                                 wmatmul=mx.mx_matmul_w4 if w4 else None)
    return om.expert_rows(x, w[rows_t, rows_j], dy, w_gu, w_d, dtype=np.float32, full=full)


@pytest.mark.parametrize("name,prec", CASES)
def test_full_size_layer(name, prec):
    need_gpu()
    from dropless_mixture_experts_warp_gb300 import layer
    from oracle import mx
    cfg = synth.CONFIGS[name]
    mx8 = prec in ("mxfp8", "mxfp8-w4")
    w4 = prec == "mxfp8-w4"
    tol = TOL_MXFP8 if mx8 else TOL_BF16
    inp = synth.torch_inputs(cfg, torch.device("cuda"))
    dims = layer.dims_of(cfg.T, cfg.d, cfg.f, cfg.E, cfg.k, cfg.f_shared, cfg.score, prec)
    bufs = layer.allocate(dims)
    sh = {"w_gu_s": inp["w_gu_s"], "w_d_s": inp["w_d_s"]} if cfg.f_shared else {}
    gr = synth.grouped_options(cfg)
    grouped = None if gr is None else dict(gr, bias=torch.from_numpy(gr["bias"]).cuda())
    layer.forward(bufs, inp["x"], inp["logits"], inp["w_gu"], inp["w_d"], grouped=grouped, **sh)
    layer.backward(bufs, inp["dy"], inp["logits"], inp["w_gu"], inp["w_d"], x=inp["x"], grouped=grouped, **sh)
    layer.check(bufs)

    # ---- routing and permutation, in full
    logits = host(inp["logits"])
    idx, w, differ, touched = _routing(cfg, logits, bufs)
    split = np.bincount(idx.ravel(), minlength=cfg.E)

    # ---- what the oracle computes: sampled tokens (all k slots) and three whole experts
    rng = np.random.default_rng(cfg.seed)
    sub = np.sort(rng.choice(np.setdiff1d(np.arange(cfg.T), differ), size=N_TOKENS, replace=False))
    order = np.argsort(split, kind="stable")
    nonempty = order[split[order] > 0]
    candidates = [int(e) for e in nonempty if int(e) not in touched]
    full_experts = {candidates[-1], candidates[0], int(rng.choice(candidates[1:-1]))}
    jobs = {}
    for e in range(cfg.E):
        if e in full_experts:
            t_sel, j_sel = np.nonzero(idx == e)
        else:
            t_sub, j_sel = np.nonzero(idx[sub] == e)
            t_sel = sub[t_sub]
        if t_sel.size:
            jobs[e] = (t_sel, j_sel, e in full_experts)
    ctx = {"inp": inp, "w": w.astype(np.float32), "mx8": mx8, "w4": w4}
    with cf.ThreadPoolExecutor(THREADS) as pool:
        futs = {e: pool.submit(_expert_job, e, t, j, full, ctx) for e, (t, j, full) in jobs.items()}
        res = {e: f.result() for e, f in futs.items()}

    pos = {int(t): i for i, t in enumerate(sub)}
    y_slot = np.zeros((N_TOKENS, cfg.k, cfg.d))
    dx_slot = np.zeros((N_TOKENS, cfg.k, cfg.d))
    dw = np.zeros((N_TOKENS, cfg.k))
    for e, (t_sel, j_sel, _) in jobs.items():
        r = res[e]
        for n, (t, j) in enumerate(zip(t_sel, j_sel)):
            i = pos.get(int(t))
            if i is not None:
                y_slot[i, j], dx_slot[i, j], dw[i, j] = r["y"][n], r["dx"][n], r["dw"][n]
    y_ref, dx_ref = y_slot.sum(axis=1), dx_slot.sum(axis=1)
    sub_t = torch.from_numpy(sub).cuda()
    skw = {}
    if cfg.f_shared:                     # the shared expert: one dense expert with weight 1
        skw = {"w_gu_s": host(inp["w_gu_s"]), "w_d_s": host(inp["w_d_s"])}
        rs_kw = {"wmatmul": mx.mx_matmul_w4} if w4 else {}
        fn = mx.expert_rows_mx if mx8 else om.expert_rows
        rs = fn(host(inp["x"][sub_t]), np.ones(N_TOKENS, np.float32), host(inp["dy"][sub_t]), skw["w_gu_s"],
                skw["w_d_s"], dtype=np.float32, full=False, **rs_kw)
        y_ref, dx_ref = y_ref + rs["y"], dx_ref + rs["dx"]
    scale = 1.0 if gr is None else gr["routed_scale"]
    dl_ref = om.route_backward(logits[sub], idx[sub], w[sub], dw, om.SIGMOID if gr else cfg.score, np.float64,
                               scale)
    errs = {"Y": rel_err(host(bufs.y[sub_t]), y_ref), "dX": rel_err(host(bufs.dx[sub_t]), dx_ref),
            "d_logits": rel_err(host(bufs.d_logits[sub_t]), dl_ref)}
    for e in sorted(full_experts):
        errs[f"dW_gu[{e}] ({split[e]} rows)"] = rel_err(host(bufs.dw_gu[e]), res[e]["dW_gu"])
        errs[f"dW_d[{e}] ({split[e]} rows)"] = rel_err(host(bufs.dw_d[e]), res[e]["dW_d"])
    if cfg.f_shared:
        # sampled entries of the shared expert's weight gradients over all T tokens
        wg_fn = mx.expert_wgrad_sampled_mx if mx8 else om.expert_wgrad_sampled
        fs = cfg.f_shared
        rows = rng.choice(2 * fs, size=N_ENTRIES, replace=False)
        cols = rng.choice(fs, size=N_ENTRIES, replace=False)
        wq_kw = {"wq": mx.qdq4} if w4 else {}
        s = wg_fn(host(inp["x"]), np.zeros((cfg.T, 1), np.float32), host(inp["dy"]), skw["w_gu_s"], skw["w_d_s"],
                  0, 1, rows, cols, om.SOFTMAX, dtype=np.float32, **wq_kw)
        errs["dW_gu_s"] = rel_err(host(bufs.dw_gu_s[torch.from_numpy(rows).cuda()]), s["dW_gu_rows"])
        errs["dW_d_s"] = rel_err(host(bufs.dw_d_s[:, torch.from_numpy(cols).cuda()]), s["dW_d_cols"])
    print(f"{name} {prec}: " + ", ".join(f"{k} {v:.2e}" for k, v in errs.items()) + f" (limit {tol})")
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, errs
    for e in np.nonzero(split == 0)[0]:
        assert torch.count_nonzero(bufs.dw_gu[int(e)]) == 0 and torch.count_nonzero(bufs.dw_d[int(e)]) == 0
