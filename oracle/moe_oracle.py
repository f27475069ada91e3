"""Plain CPU oracle of the dropless mixture-of-experts layer, forward and backward.

TEST INFRASTRUCTURE ONLY (see the package docstring): never imported by the
product path, and sharing no code with it.

What the layer computes, and where each step is stated:

* A learned router scores every expert for every token and only the top-K experts
  run for that token -- NVIDIA dropless-MoE page, "Az NVIDIA szerint tízszer
  gyorsabb lett a dropless MoE tanítása JAX-ban", section "A dropless MoE minden
  tokent feldolgoz".  Scores are a softmax over the experts (or a sigmoid for the
  DeepSeek-V3 shape); the K selected weights are renormalised to sum to one.
* Dropless: every token reaches every expert it selected, whatever the load; no
  capacity and no token is dropped (same section).
* Tokens are grouped per expert into ragged groups, the per-expert counts being the
  ``split_sizes`` argument of a grouped linear -- NVIDIA biology-MoE page
  ("NVIDIA מציגה דרך יעילה לאמן מודלי MoE בביולוגיה"), section "מומחים מקובצים
  במקום לולאת Python"; ragged per-expert tensors: NVIDIA dropless-MoE page,
  section "Az egyenetlen terhelés lassítja a tanítást".
* Each expert is GroupedLinear -> ScaledSwiGLU -> GroupedLinear, i.e. a SwiGLU MLP
  whose activation is scaled by the token's routing weight -- biology-MoE page,
  section "צמצום הזיכרון ותקורות הכימות" (and the routing-weight scaling inside the
  grouped MLP, section "מומחים מקובצים במקום לולאת Python").
* Combine returns every token's expert outputs to token order and sums them --
  DeepGEMM Mega MoE page (itsolotime.com, section "Mega MoE คืออะไร?": dispatch,
  two linear layers, SwiGLU, combine).

The form below is the plain per-expert loop the biology-MoE page names as the
baseline (one expert after another), with a library matmul as the only primitive.
The backward is the exact derivative of that forward (checked by finite
differences in the tests).

Readings where the pages are silent:
  R1  top-k ranks the raw logits (softmax and sigmoid are strictly increasing),
      ties go to the lower expert index; slot j holds the j-th best expert.
  R2  rows of one expert are ordered by token index (stable counting sort).
  R3  the routing weight multiplies the SwiGLU output before the down projection;
      combine is then an unweighted sum over the k slots in slot order.
  R4  nn.Linear layout [out, in]: W_gu[e] = [W_gate; W_up] is [2f, d] (gate rows
      first), W_d[e] is [d, f].
  R5  the shared expert (DeepSeek-V3 shape only) is a dense SwiGLU MLP on every
      token with weight 1, added after the k routed terms; it does not touch the
      router gradient.
  R6  group-limited routing (a DeepSeek-V3 router variant, from neither page): the
      E experts form n_group equal groups; a group's score is the sum of its two
      largest selection scores c = sigmoid(l) + b (b a per-expert bias that steers
      selection only); the topk_group best groups (ties to the lower group) are
      eligible and the top-k of c among their experts are chosen (ties to the lower
      index); weights are routed_scale * s_j / sum_S s.  Selection is decided in
      fp32, the precision the kernel decides in.
"""
from __future__ import annotations

from typing import Dict, Optional

import numpy as np

SOFTMAX = "softmax"
SIGMOID = "sigmoid"


# ----------------------------------------------------------------------------------
# Routing
# ----------------------------------------------------------------------------------

def select_topk(logits: np.ndarray, k: int) -> np.ndarray:
    """Indices [T, k] of the k largest logits per token, ties to the lower index (R1).

    Sort key per token: (-logit, expert index), taken by a stable lexicographic sort.
    """
    T, E = logits.shape
    if not (1 <= k <= E):
        raise ValueError("need 1 <= k <= E")
    expert_ids = np.broadcast_to(np.arange(E), (T, E))
    order = np.lexsort((expert_ids, -logits.astype(np.float64)), axis=-1)
    return order[:, :k].astype(np.int64)


def route(logits: np.ndarray, k: int, score: str = SOFTMAX, dtype=np.float64):
    """Top-k routing with renormalised weights.

    softmax: p = softmax(l) over all E experts, S = top-k, w_j = p_j / sum_S p.
    sigmoid: s = sigmoid(l), S = top-k, w_j = s_j / sum_S s.
    Returns (idx [T,k] int64, w [T,k] dtype).
    """
    l = logits.astype(dtype)
    idx = select_topk(logits, k)
    if score == SOFTMAX:
        z = np.exp(l - l.max(axis=1, keepdims=True))
        p = z / z.sum(axis=1, keepdims=True)
    elif score == SIGMOID:
        with np.errstate(over="ignore"):      # exp(-l) = inf for very negative l gives s = 0
            p = 1.0 / (1.0 + np.exp(-l))
    else:
        raise ValueError(score)
    ps = np.take_along_axis(p, idx, axis=1)
    w = ps / ps.sum(axis=1, keepdims=True)
    return idx, w


def route_grouped(logits: np.ndarray, k: int, n_group: int, topk_group: int, bias=None,
                  routed_scale: float = 1.0, dtype=np.float64):
    """Group-limited top-k with sigmoid scores (R6).  Returns (idx [T,k], w [T,k]).

    The selection scores c = fp32(sigmoid(l)) + fp32(b) and the group scores (sum of a
    group's two largest c) are fp32, as in the kernel; the weights use dtype.
    """
    T, E = logits.shape
    if E % n_group or E // n_group < 2 or not (1 <= topk_group <= n_group):
        raise ValueError("need E % n_group == 0, at least 2 experts per group, 1 <= topk_group <= n_group")
    gs = E // n_group
    if not (1 <= k <= topk_group * gs):
        raise ValueError("need 1 <= k <= topk_group * E / n_group")
    l32 = np.asarray(logits, np.float32)
    one = np.float32(1.0)
    with np.errstate(over="ignore"):
        s32 = one / (one + np.exp(-l32))
    b32 = np.zeros(E, np.float32) if bias is None else np.asarray(bias, np.float32)
    c = s32 + b32[None, :]
    top2 = -np.sort(-c.reshape(T, n_group, gs), axis=2)[:, :, :2]
    gscore = top2[:, :, 0] + top2[:, :, 1]                       # fp32 sum
    gorder = np.lexsort((np.broadcast_to(np.arange(n_group), (T, n_group)), -gscore.astype(np.float64)), axis=-1)
    eligible = np.zeros((T, n_group), bool)
    np.put_along_axis(eligible, gorder[:, :topk_group], True, axis=1)
    masked = np.where(np.repeat(eligible, gs, axis=1), c.astype(np.float64), -np.inf)
    idx = select_topk(masked, k)
    l = np.asarray(logits, dtype)
    with np.errstate(over="ignore"):
        sp = 1.0 / (1.0 + np.exp(-np.take_along_axis(l, idx, axis=1)))
    w = routed_scale * sp / sp.sum(axis=1, keepdims=True)
    return idx, w


def dispatch(idx: np.ndarray, E: int):
    """Stable counting sort of the (token, slot) pairs by expert (R2).

    Returns split_sizes [E], offsets [E+1] (exclusive prefix sum, offsets[E] = T*k),
    token_to_row [T,k] and row_to_token [T*k] (row = offsets[e] + number of earlier
    tokens that also chose expert e).
    """
    T, k = idx.shape
    split_sizes = np.zeros(E, np.int64)
    for e in idx.ravel():
        split_sizes[e] += 1
    offsets = np.zeros(E + 1, np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + split_sizes[e]
    fill = offsets[:-1].copy()
    token_to_row = np.empty((T, k), np.int64)
    row_to_token = np.empty(T * k, np.int64)
    for t in range(T):
        for j in range(k):
            e = idx[t, j]
            token_to_row[t, j] = fill[e]
            row_to_token[fill[e]] = t
            fill[e] += 1
    return split_sizes, offsets, token_to_row, row_to_token


def permute_rows(x: np.ndarray, row_to_token: np.ndarray) -> np.ndarray:
    """Expert-contiguous copy of the token rows: rows[r] = x[row_to_token[r]]."""
    return x[row_to_token]


def combine_rows(rows: np.ndarray, token_to_row: np.ndarray, dtype=np.float64) -> np.ndarray:
    """Token-order sum over the k slots, slot 0 first: out[t] = sum_j rows[token_to_row[t, j]]."""
    T, k = token_to_row.shape
    out = np.zeros((T, rows.shape[1]), dtype)
    for j in range(k):
        out += rows[token_to_row[:, j]].astype(dtype)
    return out


# ----------------------------------------------------------------------------------
# Expert MLP
# ----------------------------------------------------------------------------------

def _sigmoid(v):
    with np.errstate(over="ignore"):          # exp(-v) = inf for very negative v gives 0
        return 1.0 / (1.0 + np.exp(-v))


def _silu(v):
    return v * _sigmoid(v)


def swiglu_expert_forward(x_rows: np.ndarray, w_gu: np.ndarray, w_d: np.ndarray,
                          w_rows: Optional[np.ndarray] = None) -> Dict[str, np.ndarray]:
    """One expert on its rows: G = X W_gate^T, U = X W_up^T, A = silu(G)*U, H = w*A, Y = H W_d^T."""
    f = w_d.shape[1]
    g = x_rows @ w_gu[:f].T
    u = x_rows @ w_gu[f:].T
    a = _silu(g) * u
    h = a if w_rows is None else a * w_rows[:, None]
    y = h @ w_d.T
    return {"g": g, "u": u, "a": a, "h": h, "y": y}


def expert_rows(x_rows, w_rows, dy_rows, w_gu_e, w_d_e, dtype=np.float64, full: bool = True):
    """One expert's share of the layer, forward and backward, on rows routed to it.

    The loop bodies of moe_forward and moe_backward for a single expert e, for callers
    that go through the experts themselves (one at a time, or several side by side):
      x_rows [n,d], dy_rows [n,d]: X and dY of the tokens routed to e (token order);
      w_rows [n]: their routing weights for e.
    Returns per row: y (the term combine adds for this slot), g, u, dw (dL/d routing
    weight), dGU = [dG | dU], dx (the term the un-permute adds); with full=True (the rows
    are all of e's rows) also dW_gu [2f,d] and dW_d [d,f].
    """
    x = np.asarray(x_rows, dtype)
    dy = np.asarray(dy_rows, dtype)
    wg = np.asarray(w_gu_e, dtype)
    wd = np.asarray(w_d_e, dtype)
    f = wd.shape[1]
    we = np.asarray(w_rows, dtype)[:, None]
    r = swiglu_expert_forward(x, wg, wd, np.asarray(w_rows, dtype))
    g, u, a = r["g"], r["u"], r["a"]
    sg = _sigmoid(g)
    dh = dy @ wd
    da = we * dh
    dg = da * u * sg * (1.0 + g * (1.0 - sg))
    du = da * g * sg
    out = {"y": r["y"], "g": g, "u": u, "dw": (a * dh).sum(axis=1), "dGU": np.concatenate([dg, du], axis=1),
           "dx": dg @ wg[:f] + du @ wg[f:]}
    if full:
        out["dW_d"] = dy.T @ (we * a)
        out["dW_gu"] = np.concatenate([dg.T @ x, du.T @ x], axis=0)
    return out


def moe_forward(x, logits, w_gu, w_d, k: int, score: str = SOFTMAX,
                w_gu_s=None, w_d_s=None, dtype=np.float64, grouped: Optional[dict] = None) -> Dict[str, np.ndarray]:
    """Forward of the layer on token-major inputs.

    x [T,d], logits [T,E], w_gu [E,2f,d], w_d [E,d,f] (any float type; widened to
    ``dtype``).  Returns Y [T,d] plus the routing and per-(token, slot) values the
    backward needs.  grouped: {"n_group", "topk_group", "bias", "routed_scale"} selects
    the group-limited sigmoid router (R6) instead of route().
    """
    x = np.asarray(x, dtype)
    T, d = x.shape
    E = w_gu.shape[0]
    f = w_d.shape[2]
    if grouped is not None:
        idx, w = route_grouped(logits, k, grouped["n_group"], grouped["topk_group"], grouped.get("bias"),
                               grouped.get("routed_scale", 1.0), dtype)
    else:
        idx, w = route(logits, k, score, dtype)
    y_slot = np.zeros((T, k, d), dtype)
    g_slot = np.zeros((T, k, f), dtype)
    u_slot = np.zeros((T, k, f), dtype)
    for e in range(E):                                   # one expert after another
        t_sel, j_sel = np.nonzero(idx == e)              # token order
        if t_sel.size == 0:
            continue
        r = swiglu_expert_forward(x[t_sel], np.asarray(w_gu[e], dtype), np.asarray(w_d[e], dtype),
                                  w[t_sel, j_sel])
        y_slot[t_sel, j_sel] = r["y"]
        g_slot[t_sel, j_sel] = r["g"]
        u_slot[t_sel, j_sel] = r["u"]
    y = np.zeros((T, d), dtype)
    for j in range(k):                                   # combine, slot order
        y += y_slot[:, j]
    out = {"Y": y, "idx": idx, "w": w, "g": g_slot, "u": u_slot}
    if w_gu_s is not None:
        rs = swiglu_expert_forward(x, np.asarray(w_gu_s, dtype), np.asarray(w_d_s, dtype))
        out["Y"] = y + rs["y"]
        out["g_s"], out["u_s"] = rs["g"], rs["u"]
    return out


def route_backward(logits, idx, w, dw, score: str = SOFTMAX, dtype=np.float64,
                   routed_scale: float = 1.0) -> np.ndarray:
    """Gradient of the router logits from dL/dw [T,k], by the chain rule through route()
    (and through route_grouped(): w = routed_scale * s_j / Z_S, the bias steering the
    selection only).

    softmax: w_j = p_j / Z_S with Z_S = sum_S p and p = softmax(l):
        dL/dp_i = (dw_i - sum_S w dw) / Z_S for i in S, 0 otherwise;
        dL/dl_m = p_m (dL/dp_m - sum_i p_i dL/dp_i).
    sigmoid: w_j = a s_j / Z_S with s = sigmoid(l) (a = routed_scale, 1 for route()):
        dL/ds_i = (a dw_i - sum_S w dw) / Z_S for i in S; dL/dl = dL/ds * s (1 - s).
    """
    l = np.asarray(logits, dtype)
    T, E = l.shape
    if score == SOFTMAX:
        z = np.exp(l - l.max(axis=1, keepdims=True))
        p = z / z.sum(axis=1, keepdims=True)
    else:
        p = _sigmoid(l)
    ps = np.take_along_axis(p, idx, axis=1)
    zs = ps.sum(axis=1, keepdims=True)
    c = (w * dw).sum(axis=1, keepdims=True)
    dp = np.zeros((T, E), dtype)
    np.put_along_axis(dp, idx, (routed_scale * dw - c) / zs, axis=1)
    if score == SOFTMAX:
        return p * (dp - (p * dp).sum(axis=1, keepdims=True))
    return dp * p * (1.0 - p)


def moe_backward(x, logits, w_gu, w_d, dy, fwd: Dict[str, np.ndarray], k: int,
                 score: str = SOFTMAX, w_gu_s=None, w_d_s=None,
                 dtype=np.float64, grouped: Optional[dict] = None) -> Dict[str, np.ndarray]:
    """Backward of moe_forward for the loss L = sum(Y * dY).

    Per expert e and each of its rows (token t, slot j):
      dH = dY[t] W_d[e]          dw[t,j] = sum_f A * dH
      dA = w dH                  dG = dA * U * silu'(G),   dU = dA * silu(G)
      dX[t] += dG W_gate[e] + dU W_up[e]       (dGU[t,j] = [dG | dU] is returned too)
      dW_d[e] += dY[t]^T H,  dW_gate[e] += dG^T X[t],  dW_up[e] += dU^T X[t]
    with silu'(g) = sigmoid(g) (1 + g (1 - sigmoid(g))).
    """
    x = np.asarray(x, dtype)
    dy = np.asarray(dy, dtype)
    T, d = x.shape
    E = w_gu.shape[0]
    f = w_d.shape[2]
    idx, w = fwd["idx"], fwd["w"]
    dx_slot = np.zeros((T, k, d), dtype)
    dgu_slot = np.zeros((T, k, 2 * f), dtype)
    dw = np.zeros((T, k), dtype)
    dw_gu = np.zeros((E, 2 * f, d), dtype)
    dw_d = np.zeros((E, d, f), dtype)
    for e in range(E):
        t_sel, j_sel = np.nonzero(idx == e)
        if t_sel.size == 0:
            continue
        wg = np.asarray(w_gu[e], dtype)
        wd = np.asarray(w_d[e], dtype)
        g = fwd["g"][t_sel, j_sel]
        u = fwd["u"][t_sel, j_sel]
        sg = _sigmoid(g)
        a = g * sg * u
        we = w[t_sel, j_sel][:, None]
        dh = dy[t_sel] @ wd
        dw[t_sel, j_sel] = (a * dh).sum(axis=1)
        da = we * dh
        dg = da * u * sg * (1.0 + g * (1.0 - sg))
        du = da * g * sg
        dgu_slot[t_sel, j_sel, :f] = dg
        dgu_slot[t_sel, j_sel, f:] = du
        dx_slot[t_sel, j_sel] = dg @ wg[:f] + du @ wg[f:]
        dw_d[e] = dy[t_sel].T @ (we * a)
        dw_gu[e, :f] = dg.T @ x[t_sel]
        dw_gu[e, f:] = du.T @ x[t_sel]
    dx = np.zeros((T, d), dtype)
    for j in range(k):
        dx += dx_slot[:, j]
    out = {"dX": dx, "dW_gu": dw_gu, "dW_d": dw_d, "dw": dw, "dGU": dgu_slot,
           "d_logits": route_backward(logits, idx, w, dw, SIGMOID if grouped is not None else score, dtype,
                                      1.0 if grouped is None else grouped.get("routed_scale", 1.0))}
    if w_gu_s is not None:
        fs = w_d_s.shape[1]
        wg = np.asarray(w_gu_s, dtype)
        wd = np.asarray(w_d_s, dtype)
        g, u = fwd["g_s"], fwd["u_s"]
        sg = _sigmoid(g)
        dh = dy @ wd
        dg = dh * u * sg * (1.0 + g * (1.0 - sg))
        du = dh * g * sg
        out["dX"] = dx + dg @ wg[:fs] + du @ wg[fs:]
        out["dW_d_s"] = dy.T @ (g * sg * u)
        out["dW_gu_s"] = np.concatenate([dg.T @ x, du.T @ x], axis=0)
    return out


def expert_wgrad(x, logits, dy, w_gu_e, w_d_e, e: int, k: int, score: str = SOFTMAX,
                 dtype=np.float64) -> Dict[str, np.ndarray]:
    """dW_gu[e] and dW_d[e] alone (for sampled checks on large layers).

    Uses only the rows routed to expert e: the same per-row formulas as
    moe_backward, summed over every token that selected e.
    """
    idx, w = route(logits, k, score, dtype)
    t_sel, j_sel = np.nonzero(idx == e)
    f = w_d_e.shape[1]
    d = w_d_e.shape[0]
    if t_sel.size == 0:
        return {"dW_gu": np.zeros((2 * f, d), dtype), "dW_d": np.zeros((d, f), dtype), "n": 0}
    xe = np.asarray(x[t_sel], dtype)
    dye = np.asarray(dy[t_sel], dtype)
    wg = np.asarray(w_gu_e, dtype)
    wd = np.asarray(w_d_e, dtype)
    we = w[t_sel, j_sel][:, None]
    g = xe @ wg[:f].T
    u = xe @ wg[f:].T
    sg = _sigmoid(g)
    a = g * sg * u
    dh = dye @ wd
    da = we * dh
    dg = da * u * sg * (1.0 + g * (1.0 - sg))
    du = da * g * sg
    return {"dW_gu": np.concatenate([dg.T @ xe, du.T @ xe], axis=0),
            "dW_d": dye.T @ (we * a), "n": int(t_sel.size)}


def expert_wgrad_sampled(x, logits, dy, w_gu_e, w_d_e, e: int, k: int, gu_rows, d_cols,
                         score: str = SOFTMAX, dtype=np.float32) -> Dict[str, np.ndarray]:
    """Selected entries of expert e's weight gradients, for sampled checks on large layers.

    Returns dW_gu[e][gu_rows, :] (full rows; row j < f is a gate row, j >= f an up row)
    and dW_d[e][:, d_cols] (full columns).  Same per-row formulas as moe_backward,
    evaluated only for the intermediate columns those entries depend on.
    """
    idx, w = route(logits, k, score, dtype)
    t_sel, j_sel = np.nonzero(idx == e)
    f = w_d_e.shape[1]
    d = w_d_e.shape[0]
    gu_rows = np.asarray(gu_rows)
    d_cols = np.asarray(d_cols)
    if t_sel.size == 0:
        return {"dW_gu_rows": np.zeros((gu_rows.size, d), dtype),
                "dW_d_cols": np.zeros((d, d_cols.size), dtype), "n": 0}
    xe = np.asarray(x[t_sel], dtype)
    dye = np.asarray(dy[t_sel], dtype)
    wg = np.asarray(w_gu_e, dtype)
    wd = np.asarray(w_d_e, dtype)
    we = w[t_sel, j_sel][:, None]
    # rows of dW_gu: need columns c = j mod f of G, U and dH
    cols = gu_rows % f
    g = xe @ wg[cols].T
    u = xe @ wg[f + cols].T
    sg = _sigmoid(g)
    dh = dye @ wd[:, cols]
    da = we * dh
    dg = da * u * sg * (1.0 + g * (1.0 - sg))
    du = da * g * sg
    sel = np.where((gu_rows < f)[None, :], dg, du)          # [n_e, len(gu_rows)]
    dw_gu_rows = sel.T @ xe
    # columns of dW_d: need columns c of H = w * silu(G) * U
    g2 = xe @ wg[d_cols].T
    u2 = xe @ wg[f + d_cols].T
    h2 = we * g2 * _sigmoid(g2) * u2
    return {"dW_gu_rows": dw_gu_rows, "dW_d_cols": dye.T @ h2, "n": int(t_sel.size)}
