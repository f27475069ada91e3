"""Pins of the CPU oracle against facts other than itself (no GPU needed).

Each test pins one part of the oracle to something independent: brute force on
tiny inputs, a library routine, an independent dense formulation, a textbook
special case, finite differences, or an exact identity.
"""
import itertools

import numpy as np
import pytest
import scipy.special

import oracle
from oracle import moe_oracle as om
from dropless_mixture_experts_warp_gb300 import synth


# ---------------------------------------------------------------- routing

def _rank_bruteforce(lrow):
    """rank(e) = #experts strictly better: larger logit, or equal logit and lower index."""
    E = len(lrow)
    return [sum(1 for e2 in range(E) if lrow[e2] > lrow[e] or (lrow[e2] == lrow[e] and e2 < e))
            for e in range(E)]


def test_topk_matches_bruteforce_with_ties():
    rng = np.random.default_rng(0)
    logits = rng.integers(-2, 3, size=(64, 6)).astype(np.float32)    # many exact ties
    logits[0] = 0.0
    logits[1, :] = [-0.0, 0.0, -0.0, 1.0, 1.0, -1.0]                  # signed zeros tie
    for k in (1, 2, 3, 6):
        idx = om.select_topk(logits, k)
        for t in range(logits.shape[0]):
            rank = _rank_bruteforce(list(logits[t]))
            expect = [rank.index(j) for j in range(k)]
            assert list(idx[t]) == expect


def test_topk_all_subsets_tiny():
    """The selected set maximises the logit sum and, among ties, is lexicographically smallest."""
    rng = np.random.default_rng(1)
    logits = rng.integers(0, 4, size=(40, 5)).astype(np.float64)
    k = 2
    idx = om.select_topk(logits, k)
    for t in range(40):
        best = max(itertools.combinations(range(5), k),
                   key=lambda s: (sum(logits[t, list(s)]), [-e for e in s]))
        assert sorted(idx[t]) == sorted(best)


def test_softmax_weights_are_softmax_over_selected():
    rng = np.random.default_rng(2)
    logits = rng.standard_normal((32, 16)).astype(np.float32) * 3
    idx, w = om.route(logits, 4, om.SOFTMAX)
    for t in range(32):
        ref = scipy.special.softmax(logits[t, idx[t]].astype(np.float64))
        np.testing.assert_allclose(w[t], ref, rtol=1e-12, atol=0)
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=1e-14)
    assert np.all(np.diff(w, axis=1) <= 0)        # slot order follows the score order


def test_sigmoid_weights_closed_form():
    rng = np.random.default_rng(3)
    logits = rng.standard_normal((32, 16)).astype(np.float32) * 2
    idx, w = om.route(logits, 4, om.SIGMOID)
    for t in range(32):
        s = scipy.special.expit(logits[t, idx[t]].astype(np.float64))
        np.testing.assert_allclose(w[t], s / s.sum(), rtol=1e-12, atol=0)


def test_dispatch_invariants_tiny_config():
    cfg = synth.CONFIGS["tiny"]
    inp = synth.token_inputs(cfg)
    idx, _ = om.route(inp["logits"], cfg.k, cfg.score)
    split, offsets, t2r, r2t = om.dispatch(idx, cfg.E)
    R = cfg.T * cfg.k
    assert split.sum() == R
    assert offsets[0] == 0 and offsets[-1] == R
    assert np.array_equal(np.diff(offsets), split)
    assert split[3] == 0                                     # forced-empty expert
    assert np.array_equal(np.sort(t2r.ravel()), np.arange(R))  # bijection onto [0, R)
    for t in range(cfg.T):
        for j in range(cfg.k):
            r = t2r[t, j]
            assert r2t[r] == t
            e = idx[t, j]
            assert offsets[e] <= r < offsets[e + 1]
    for e in range(cfg.E):                                   # stable: token order inside a segment
        toks = r2t[offsets[e]:offsets[e + 1]]
        assert np.all(np.diff(toks) > 0)


def test_identity_round_trip_is_exact():
    """combine(permute(x)) = k * x bit for bit (k a power of two, x bf16-representable)."""
    cfg = synth.CONFIGS["tiny"]
    inp = synth.token_inputs(cfg)
    x = synth.bf16_to_f32(inp["x"])
    idx, _ = om.route(inp["logits"], cfg.k, cfg.score)
    _, _, t2r, r2t = om.dispatch(idx, cfg.E)
    rows = om.permute_rows(x, r2t)
    back = om.combine_rows(rows, t2r, dtype=np.float32)
    assert np.array_equal(back, np.float32(cfg.k) * x)


# ---------------------------------------------------------------- forward

def _small_problem(seed, T=24, d=20, f=12, E=5, k=2, shared=False, margin=True):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, d))
    w_gu = rng.standard_normal((E, 2 * f, d)) / np.sqrt(d)
    w_d = rng.standard_normal((E, d, f)) / np.sqrt(f)
    dy = rng.standard_normal((T, d))
    if margin:
        # distinct logits with gaps >= 0.05 so a finite-difference step never flips top-k
        base = np.arange(E, dtype=np.float64) * 0.3
        logits = np.stack([rng.permutation(base) for _ in range(T)]) + rng.uniform(-0.1, 0.1, (T, 1))
    else:
        logits = rng.standard_normal((T, E))
    s = None
    if shared:
        fs = 8
        s = (rng.standard_normal((2 * fs, d)) / np.sqrt(d), rng.standard_normal((d, fs)) / np.sqrt(fs))
    return x, logits, w_gu, w_d, dy, s


@pytest.mark.parametrize("score", [om.SOFTMAX, om.SIGMOID])
def test_forward_equals_dense_compute_all_then_mask(score):
    x, logits, w_gu, w_d, dy, _ = _small_problem(11, margin=False)
    k = 2
    out = om.moe_forward(x, logits, w_gu, w_d, k, score)
    E, f = w_gu.shape[0], w_d.shape[2]
    # Dense form: run every expert on every token, then mask with a [T,E] gate matrix
    # built from an independent brute-force selection.
    T = x.shape[0]
    gate = np.zeros((T, E))
    for t in range(T):
        rank = _rank_bruteforce(list(logits[t]))
        sel = [e for e in range(E) if rank[e] < k]
        if score == om.SOFTMAX:
            sc = scipy.special.softmax(logits[t])
        else:
            sc = scipy.special.expit(logits[t])
        for e in sel:
            gate[t, e] = sc[e] / sum(sc[s] for s in sel)
    G = np.einsum("td,efd->tef", x, w_gu[:, :f])
    U = np.einsum("td,efd->tef", x, w_gu[:, f:])
    A = G * scipy.special.expit(G) * U
    Yall = np.einsum("tef,edf->ted", A, w_d)
    Ydense = np.einsum("te,ted->td", gate, Yall)
    np.testing.assert_allclose(out["Y"], Ydense, rtol=1e-12, atol=1e-12)


def test_single_expert_reduces_to_swiglu_mlp():
    rng = np.random.default_rng(5)
    T, d, f = 16, 12, 10
    x = rng.standard_normal((T, d))
    wg = rng.standard_normal((f, d))
    wu = rng.standard_normal((f, d))
    wd = rng.standard_normal((d, f))
    logits = rng.standard_normal((T, 1))
    out = om.moe_forward(x, logits, np.concatenate([wg, wu])[None], wd[None], 1, om.SOFTMAX)
    gate = x @ wg.T
    ref = ((gate / (1 + np.exp(-gate))) * (x @ wu.T)) @ wd.T
    np.testing.assert_allclose(out["Y"], ref, rtol=1e-13, atol=1e-13)
    assert np.all(out["w"] == 1.0)


def test_shared_expert_adds_dense_mlp():
    x, logits, w_gu, w_d, dy, s = _small_problem(12, shared=True)
    routed = om.moe_forward(x, logits, w_gu, w_d, 2, om.SIGMOID)
    both = om.moe_forward(x, logits, w_gu, w_d, 2, om.SIGMOID, w_gu_s=s[0], w_d_s=s[1])
    fs = s[1].shape[1]
    g = x @ s[0][:fs].T
    ref = (g * scipy.special.expit(g) * (x @ s[0][fs:].T)) @ s[1].T
    np.testing.assert_allclose(both["Y"] - routed["Y"], ref, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- backward

def _loss(x, logits, w_gu, w_d, dy, k, score, s):
    kw = {} if s is None else {"w_gu_s": s[0], "w_d_s": s[1]}
    return float((om.moe_forward(x, logits, w_gu, w_d, k, score, **kw)["Y"] * dy).sum())


def _fd(fun, arr, eps=1e-6):
    grad = np.zeros_like(arr)
    it = np.nditer(arr, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        old = arr[i]
        arr[i] = old + eps
        lp = fun()
        arr[i] = old - eps
        lm = fun()
        arr[i] = old
        grad[i] = (lp - lm) / (2 * eps)
    return grad


@pytest.mark.parametrize("score,shared", [(om.SOFTMAX, False), (om.SIGMOID, False), (om.SIGMOID, True)])
def test_backward_matches_finite_differences(score, shared):
    x, logits, w_gu, w_d, dy, s = _small_problem(21, T=8, d=16, f=8, E=4, k=2, shared=shared)
    k = 2
    kw = {} if s is None else {"w_gu_s": s[0], "w_d_s": s[1]}
    fwd = om.moe_forward(x, logits, w_gu, w_d, k, score, **kw)
    bwd = om.moe_backward(x, logits, w_gu, w_d, dy, fwd, k, score, **kw)
    fun = lambda: _loss(x, logits, w_gu, w_d, dy, k, score, s)  # noqa: E731

    def rel(a, b):
        return np.abs(a - b).max() / np.abs(b).max()

    assert rel(bwd["dX"], _fd(fun, x)) < 1e-6
    assert rel(bwd["d_logits"], _fd(fun, logits)) < 1e-6
    assert rel(bwd["dW_d"], _fd(fun, w_d)) < 1e-6
    assert rel(bwd["dW_gu"], _fd(fun, w_gu)) < 1e-6
    if shared:
        assert rel(bwd["dW_gu_s"], _fd(fun, s[0])) < 1e-6
        assert rel(bwd["dW_d_s"], _fd(fun, s[1])) < 1e-6


def test_router_gradient_zero_off_selection_and_sums_to_zero_for_softmax():
    x, logits, w_gu, w_d, dy, _ = _small_problem(31)
    fwd = om.moe_forward(x, logits, w_gu, w_d, 2, om.SOFTMAX)
    bwd = om.moe_backward(x, logits, w_gu, w_d, dy, fwd, 2, om.SOFTMAX)
    dl = bwd["d_logits"]
    mask = np.zeros_like(dl, bool)
    np.put_along_axis(mask, fwd["idx"], True, axis=1)
    assert np.abs(dl[~mask]).max() <= 1e-14 * np.abs(dl).max()   # zero up to rounding
    # w is invariant to adding a constant to all logits -> the gradient sums to zero
    np.testing.assert_allclose(dl.sum(axis=1), 0, atol=1e-13)


def test_expert_wgrad_matches_full_backward():
    x, logits, w_gu, w_d, dy, _ = _small_problem(41, E=6, k=3)
    fwd = om.moe_forward(x, logits, w_gu, w_d, 3, om.SOFTMAX)
    bwd = om.moe_backward(x, logits, w_gu, w_d, dy, fwd, 3, om.SOFTMAX)
    for e in range(6):
        r = om.expert_wgrad(x, logits, dy, w_gu[e], w_d[e], e, 3, om.SOFTMAX)
        np.testing.assert_allclose(r["dW_gu"], bwd["dW_gu"][e], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(r["dW_d"], bwd["dW_d"][e], rtol=1e-12, atol=1e-12)


def test_sampled_wgrad_entries_match_full_wgrad():
    x, logits, w_gu, w_d, dy, _ = _small_problem(42, E=6, k=3, d=20, f=12)
    rows = np.array([0, 5, 11, 12, 17, 23])          # gate and up rows
    cols = np.array([0, 3, 11])
    for e in range(6):
        full = om.expert_wgrad(x, logits, dy, w_gu[e], w_d[e], e, 3, om.SOFTMAX)
        s = om.expert_wgrad_sampled(x, logits, dy, w_gu[e], w_d[e], e, 3, rows, cols, om.SOFTMAX,
                                    dtype=np.float64)
        np.testing.assert_allclose(s["dW_gu_rows"], full["dW_gu"][rows], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(s["dW_d_cols"], full["dW_d"][:, cols], rtol=1e-12, atol=1e-12)


def test_token_subset_equals_full_batch():
    """Rows of Y, dX and d_logits depend on their own token only (used by sampled checks)."""
    x, logits, w_gu, w_d, dy, _ = _small_problem(51)
    full_f = om.moe_forward(x, logits, w_gu, w_d, 2, om.SOFTMAX)
    full_b = om.moe_backward(x, logits, w_gu, w_d, dy, full_f, 2, om.SOFTMAX)
    sub = np.array([3, 0, 17, 9])
    f = om.moe_forward(x[sub], logits[sub], w_gu, w_d, 2, om.SOFTMAX)
    b = om.moe_backward(x[sub], logits[sub], w_gu, w_d, dy[sub], f, 2, om.SOFTMAX)
    np.testing.assert_allclose(f["Y"], full_f["Y"][sub], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(b["dX"], full_b["dX"][sub], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(b["d_logits"], full_b["d_logits"][sub], rtol=1e-13, atol=1e-13)


def _assemble_expert_rows(fn, x, logits, w_gu, w_d, dy, k, score, full=True):
    """Y, dX, dw, dGU, d_logits and the weight gradients put together from per-expert calls."""
    idx, w = om.route(logits, k, score)
    T, d = x.shape
    E, f2 = w_gu.shape[0], w_gu.shape[1]
    y_slot, dx_slot = np.zeros((T, k, d)), np.zeros((T, k, d))
    dgu, dw = np.zeros((T, k, f2)), np.zeros((T, k))
    dW_gu, dW_d = np.zeros_like(w_gu), np.zeros_like(w_d)
    for e in range(E):
        t_sel, j_sel = np.nonzero(idx == e)
        if t_sel.size == 0:
            continue
        r = fn(x[t_sel], w[t_sel, j_sel], dy[t_sel], w_gu[e], w_d[e], full=full)
        y_slot[t_sel, j_sel], dx_slot[t_sel, j_sel] = r["y"], r["dx"]
        dgu[t_sel, j_sel], dw[t_sel, j_sel] = r["dGU"], r["dw"]
        if full:
            dW_gu[e], dW_d[e] = r["dW_gu"], r["dW_d"]
    return {"Y": y_slot.sum(axis=1), "dX": dx_slot.sum(axis=1), "dw": dw, "dGU": dgu, "dW_gu": dW_gu,
            "dW_d": dW_d, "d_logits": om.route_backward(logits, idx, w, dw, score)}


@pytest.mark.parametrize("score", [om.SOFTMAX, om.SIGMOID])
def test_expert_rows_assemble_the_layer(score):
    """The per-expert form (used to spread full-size checks over threads) gives the layer
    oracle's forward and backward, and the layer's dGU reassembles its dW_gu and dX."""
    x, logits, w_gu, w_d, dy, _ = _small_problem(43, E=6, k=3)
    fwd = om.moe_forward(x, logits, w_gu, w_d, 3, score)
    bwd = om.moe_backward(x, logits, w_gu, w_d, dy, fwd, 3, score)
    got = _assemble_expert_rows(om.expert_rows, x, logits, w_gu, w_d, dy, 3, score)
    for key, ref in (("Y", fwd["Y"]), ("dX", bwd["dX"]), ("dw", bwd["dw"]), ("dGU", bwd["dGU"]),
                     ("dW_gu", bwd["dW_gu"]), ("dW_d", bwd["dW_d"]), ("d_logits", bwd["d_logits"])):
        np.testing.assert_allclose(got[key], ref, rtol=1e-12, atol=1e-12, err_msg=key)
    idx = fwd["idx"]
    for e in range(6):                              # dW_gu[e] = dGU_e^T X_e, dX = sum_j dGU W_gu
        t_sel, j_sel = np.nonzero(idx == e)
        np.testing.assert_allclose(bwd["dGU"][t_sel, j_sel].T @ x[t_sel], bwd["dW_gu"][e], rtol=1e-12, atol=1e-12)
    dx = sum(np.einsum("tf,tfd->td", bwd["dGU"][:, j], w_gu[idx[:, j]]) for j in range(3))
    np.testing.assert_allclose(dx, bwd["dX"], rtol=1e-12, atol=1e-12)


def test_expert_rows_of_a_row_subset_equal_those_of_all_rows():
    """Per-row results depend on their own row only (sampled full-size checks rely on it)."""
    x, logits, w_gu, w_d, dy, _ = _small_problem(44, E=3, k=2)
    idx, w = om.route(logits, 2, om.SOFTMAX)
    t_sel, j_sel = np.nonzero(idx == 1)
    full = om.expert_rows(x[t_sel], w[t_sel, j_sel], dy[t_sel], w_gu[1], w_d[1])
    sub = np.array([0, 2, len(t_sel) - 1])
    part = om.expert_rows(x[t_sel[sub]], w[t_sel[sub], j_sel[sub]], dy[t_sel[sub]], w_gu[1], w_d[1], full=False)
    for key in ("y", "dx", "dw", "dGU"):
        np.testing.assert_allclose(part[key], full[key][sub], rtol=1e-13, atol=1e-13, err_msg=key)


# ---------------------------------------------------------------- planted mistakes

def _dense_forward_error(score=om.SOFTMAX):
    x, logits, w_gu, w_d, dy, _ = _small_problem(61, margin=False)
    out = om.moe_forward(x, logits, w_gu, w_d, 2, score)
    f = w_d.shape[2]
    T, E = logits.shape
    gate = np.zeros((T, E))
    for t in range(T):
        rank = _rank_bruteforce(list(logits[t]))
        sel = [e for e in range(E) if rank[e] < 2]
        sc = scipy.special.softmax(logits[t])
        for e in sel:
            gate[t, e] = sc[e] / sum(sc[s] for s in sel)
    G = np.einsum("td,efd->tef", x, w_gu[:, :f])
    U = np.einsum("td,efd->tef", x, w_gu[:, f:])
    Y = np.einsum("te,ted->td", gate, np.einsum("tef,edf->ted", G * scipy.special.expit(G) * U, w_d))
    return np.abs(out["Y"] - Y).max() / np.abs(Y).max()


def _fd_router_error():
    x, logits, w_gu, w_d, dy, _ = _small_problem(62, T=6, d=8, f=4, E=3, k=2)
    fwd = om.moe_forward(x, logits, w_gu, w_d, 2, om.SOFTMAX)
    bwd = om.moe_backward(x, logits, w_gu, w_d, dy, fwd, 2, om.SOFTMAX)
    fd = _fd(lambda: _loss(x, logits, w_gu, w_d, dy, 2, om.SOFTMAX, None), logits)
    return np.abs(bwd["d_logits"] - fd).max() / np.abs(fd).max()


def _topk_mismatches():
    rng = np.random.default_rng(64)
    logits = rng.integers(-2, 3, size=(32, 6)).astype(np.float32)
    idx = om.select_topk(logits, 3)
    bad = 0
    for t in range(32):
        rank = _rank_bruteforce(list(logits[t]))
        bad += list(idx[t]) != [rank.index(j) for j in range(3)]
    return bad


def test_planted_mistakes_are_caught(monkeypatch):
    """Mutants planted in the oracle (on the CPU) must fail the pins above."""
    assert _dense_forward_error() < 1e-12 and _fd_router_error() < 1e-6 and _topk_mismatches() == 0
    with monkeypatch.context() as m:             # sign error inside the activation
        m.setattr(om, "_silu", lambda v: v / (1.0 + np.exp(v)))
        assert _dense_forward_error() > 1e-3
    with monkeypatch.context() as m:             # sign error in the router gradient
        real = om.route_backward
        m.setattr(om, "route_backward", lambda *a, **kw: -real(*a, **kw))
        assert _fd_router_error() > 1e-3
    with monkeypatch.context() as m:             # ties broken towards the higher index
        def topk_high(lg, k):
            ids = np.broadcast_to(np.arange(lg.shape[1]), lg.shape)
            return np.lexsort((-ids, -lg.astype(np.float64)), axis=-1)[:, :k]
        m.setattr(om, "select_topk", topk_high)
        assert _topk_mismatches() > 0
    # a transposed down projection cannot be applied when d != f
    x, logits, w_gu, w_d, dy, _ = _small_problem(63)
    with pytest.raises(ValueError):
        om.moe_forward(x, logits, w_gu, np.swapaxes(w_d, 1, 2), 2, om.SOFTMAX)


# ---------------------------------------------------------------- group-limited routing

def _sig32(l):
    one = np.float32(1.0)
    return one / (one + np.exp(-np.asarray(l, np.float32)))


def _grouped_by_loops(logits, k, n_group, topk_group, bias):
    """The group-limited selection written as per-token loops with explicit sort keys."""
    T, E = logits.shape
    gs = E // n_group
    out = np.zeros((T, k), np.int64)
    for t in range(T):
        c = [np.float32(_sig32(logits[t, e]) + np.float32(bias[e])) for e in range(E)]
        gsc = []
        for g in range(n_group):
            vals = sorted((c[e] for e in range(g * gs, (g + 1) * gs)), reverse=True)
            gsc.append(np.float32(vals[0] + vals[1]))
        groups = sorted(range(n_group), key=lambda g: (-float(gsc[g]), g))[:topk_group]
        cand = [e for e in range(E) if e // gs in groups]
        out[t] = sorted(cand, key=lambda e: (-float(c[e]), e))[:k]
    return out


@pytest.mark.parametrize("E,n_group,topk_group,k", [(16, 4, 2, 4), (24, 3, 1, 2), (32, 8, 4, 8), (12, 6, 6, 3)])
def test_grouped_routing_matches_loop_definition(E, n_group, topk_group, k):
    rng = np.random.default_rng(E + n_group)
    logits = rng.standard_normal((40, E)).astype(np.float32)
    bias = rng.standard_normal(E).astype(np.float32) * 0.3
    idx, w = om.route_grouped(logits, k, n_group, topk_group, bias, 2.5)
    assert np.array_equal(idx, _grouped_by_loops(logits, k, n_group, topk_group, bias))
    s = scipy.special.expit(np.take_along_axis(logits.astype(np.float64), idx, axis=1))
    np.testing.assert_allclose(w, 2.5 * s / s.sum(axis=1, keepdims=True), rtol=1e-12)


def test_grouped_routing_with_one_group_is_plain_sigmoid_topk():
    rng = np.random.default_rng(5)
    logits = rng.standard_normal((64, 16)).astype(np.float32)
    idx, w = om.route_grouped(logits, 4, 1, 1)
    idx0, w0 = om.route(logits, 4, om.SIGMOID)
    assert np.array_equal(idx, idx0)
    np.testing.assert_allclose(w, w0, rtol=1e-12)


def test_grouped_routing_bias_steers_selection_only():
    rng = np.random.default_rng(6)
    logits = rng.standard_normal((32, 16)).astype(np.float32)
    bias = np.zeros(16, np.float32)
    bias[11] = 10.0                      # expert 11 (group 2 of 4) is always chosen
    idx, w = om.route_grouped(logits, 3, 4, 2, bias)
    assert np.all((idx == 11).any(axis=1))
    s = scipy.special.expit(np.take_along_axis(logits.astype(np.float64), idx, axis=1))
    np.testing.assert_allclose(w, s / s.sum(axis=1, keepdims=True), rtol=1e-12)   # no bias in w


def test_grouped_routing_only_picks_from_the_best_groups():
    rng = np.random.default_rng(7)
    E, n_group, topk_group, k = 32, 8, 2, 4
    logits = rng.standard_normal((50, E)).astype(np.float32)
    idx, _ = om.route_grouped(logits, k, n_group, topk_group)
    c = _sig32(logits).reshape(50, n_group, E // n_group)
    gsc = np.sort(c, axis=2)[:, :, -2:].sum(axis=2)
    for t in range(50):
        best = set(np.argsort(-gsc[t], kind="stable")[:topk_group])
        assert set(idx[t] // (E // n_group)) <= best


def test_grouped_router_backward_matches_finite_differences():
    x, logits, w_gu, w_d, dy, _ = _small_problem(51, T=8, d=16, f=8, E=8, k=2)
    bias = np.linspace(-0.2, 0.2, 8)
    grouped = {"n_group": 4, "topk_group": 2, "bias": bias, "routed_scale": 2.5}
    fwd = om.moe_forward(x, logits, w_gu, w_d, 2, om.SIGMOID, grouped=grouped)
    bwd = om.moe_backward(x, logits, w_gu, w_d, dy, fwd, 2, om.SIGMOID, grouped=grouped)

    def fun():
        return float((om.moe_forward(x, logits, w_gu, w_d, 2, om.SIGMOID, grouped=grouped)["Y"] * dy).sum())
    fd = _fd(fun, logits)
    assert np.abs(bwd["d_logits"] - fd).max() / np.abs(fd).max() < 1e-6
    assert np.abs(bwd["dX"] - _fd(fun, x)).max() / np.abs(bwd["dX"]).max() < 1e-6
