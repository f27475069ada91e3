"""MXFP8 (E4M3 elements, one E8M0 scale per 32 consecutive elements) for the oracle,
and FP4 weights (E2M1 elements, same scales) for FP8 x FP4 experts (end of the file).

TEST INFRASTRUCTURE ONLY (see the package docstring).

The biology-MoE page ("NVIDIA מציגה דרך יעילה לאמן מודלי MoE בביולוגיה", section
"צמצום הזיכרון ותקורות הכימות") states the format: 8-bit values with one scale
factor per block of 32 consecutive values, run on Blackwell's block-scaled tensor
cores; the dropless-MoE page ("Az NVIDIA szerint tízszer gyorsabb lett a dropless
MoE tanítása JAX-ban", section "Csoportosított mátrixszorzás és összevont
adatmozgatás") applies it to the expert GEMMs with group-aware quantisation.  The
pages do not give the rounding or scale rule; the readings taken here:

  * element format E4M3 (bias 7, 3 mantissa bits, no infinities, largest finite
    448); encoding rounds to the nearest representable value, ties to the even
    code, and saturates to +-448 (never produces NaN);
  * scale = 2^(floor(log2(amax)) - 8), 8 being the largest exponent of E4M3, with
    the exponent clamped to [-127, 127] and stored as the biased byte e + 127
    (E8M0); an all-zero block gets scale byte 0 and zero codes;
  * every GEMM operand is quantised along its own contraction axis; blocks of rows
    start at the first row of each expert's segment (rows past its end count as 0).
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
EMAX_E4M3 = 8
BLOCK = 32


def _e4m3_table() -> np.ndarray:
    """Values of the 128 non-negative codes (0x7F is NaN and excluded by callers)."""
    vals = np.empty(128, np.float64)
    for code in range(128):
        e = code >> 3
        m = code & 7
        vals[code] = (m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
    vals[0x7F] = np.nan
    return vals


E4M3_VALUES = _e4m3_table()
_FINITE = E4M3_VALUES[:0x7F]          # codes 0x00..0x7E, increasing


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    codes = np.asarray(codes, np.uint8)
    mag = E4M3_VALUES[codes & 0x7F]
    return np.where(codes & 0x80, -mag, mag)


def e4m3_encode(v: np.ndarray) -> np.ndarray:
    """Round to the nearest E4M3 value, ties to the even code, saturating at 448."""
    v = np.asarray(v, np.float64)
    if not np.all(np.isfinite(v)):
        raise ValueError("e4m3_encode: non-finite input")
    a = np.minimum(np.abs(v), E4M3_MAX)
    hi = np.searchsorted(_FINITE, a, side="left")          # first code with value >= a
    hi = np.minimum(hi, 0x7E)
    lo = np.maximum(hi - 1, 0)
    d_lo = a - _FINITE[lo]
    d_hi = _FINITE[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(_FINITE[hi] == a, hi, np.where(pick_hi, hi, lo)).astype(np.uint8)
    return (code | (np.signbit(v).astype(np.uint8) << 7)).astype(np.uint8)   # sign kept, -0 = 0x80


def scale_exponent(amax: np.ndarray) -> np.ndarray:
    """floor(log2(amax)) - 8, clamped to [-127, 127]; -127 for amax = 0."""
    amax = np.asarray(amax, np.float64)
    _, ex = np.frexp(amax)                       # amax = m 2^ex, m in [0.5, 1)
    e = ex.astype(np.int64) - 1 - EMAX_E4M3
    e = np.where(amax > 0, e, -127)
    return np.clip(e, -127, 127)


def mx_quantize(x: np.ndarray):
    """Quantise along the last axis (length a multiple of 32).

    Returns (codes uint8 like x, scale bytes uint8 [..., K/32]).
    """
    x = np.asarray(x, np.float64)
    K = x.shape[-1]
    if K % BLOCK:
        raise ValueError("last axis must be a multiple of 32")
    blocks = x.reshape(*x.shape[:-1], K // BLOCK, BLOCK)
    e = scale_exponent(np.abs(blocks).max(axis=-1))
    codes = e4m3_encode(blocks * np.exp2(-e)[..., None])     # exact power-of-two scaling
    return codes.reshape(x.shape), (e + 127).astype(np.uint8)


def mx_dequantize(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    codes = np.asarray(codes, np.uint8)
    K = codes.shape[-1]
    v = e4m3_decode(codes).reshape(*codes.shape[:-1], K // BLOCK, BLOCK)
    return (v * np.exp2(scales.astype(np.float64) - 127)[..., None]).reshape(codes.shape)


def e4m3_round(a: np.ndarray) -> np.ndarray:
    """Value of e4m3_encode, computed arithmetically: |a| rounded to the E4M3 grid.

    For |a| >= 2^-6 the grid step is 2^(floor(log2|a|) - 3), below it 2^-9; np.rint
    rounds half to even, which is the even code; the result saturates at 448.
    """
    a = np.asarray(a)
    if a.dtype not in (np.float32, np.float64):
        a = a.astype(np.float64)
    mag = np.minimum(np.abs(a), a.dtype.type(E4M3_MAX))
    _, ex = np.frexp(mag)                         # mag = m 2^ex, m in [0.5, 1)
    step = np.ldexp(a.dtype.type(1), np.maximum(ex - 1, -6) - 3)
    r = np.minimum(np.rint(mag / step) * step, a.dtype.type(E4M3_MAX))
    return np.copysign(r, a)


def qdq(x: np.ndarray) -> np.ndarray:
    """Quantise then dequantise along the last axis, zero-padding it to a multiple of 32.

    Equal to mx_dequantize(*mx_quantize(x)) (checked in the tests), computed without
    the code table so large operands stay cheap.
    """
    x = np.asarray(x)
    if x.dtype != np.float32:        # fp32 stays fp32: every E4M3 code times 2^[-127,119] is an fp32
        x = x.astype(np.float64)
    K = x.shape[-1]
    pad = (-K) % BLOCK
    if pad:
        x = np.concatenate([x, np.zeros((*x.shape[:-1], pad), x.dtype)], axis=-1)
    blocks = x.reshape(*x.shape[:-1], x.shape[-1] // BLOCK, BLOCK)
    e = scale_exponent(np.abs(blocks).max(axis=-1).astype(np.float64))
    scale = np.ldexp(x.dtype.type(1), e)[..., None]
    return (e4m3_round(blocks / scale) * scale).reshape(x.shape)[..., :K]


def mx_matmul(a: np.ndarray, b: np.ndarray, dtype=np.float64) -> np.ndarray:
    """a [M,K] x b [N,K]^T with both operands MXFP8-quantised along K (the shared axis)."""
    return qdq(a).astype(dtype) @ qdq(b).astype(dtype).T


# ----------------------------------------------------------------------------------
# The layer with MXFP8 GEMM operands
# ----------------------------------------------------------------------------------

def moe_forward_mx(x, logits, w_gu, w_d, k, score="softmax", w_gu_s=None, w_d_s=None,
                   dtype=np.float64, matmul=mx_matmul, grouped=None, wmatmul=None):
    """Forward of the layer with every GEMM operand quantised along its contraction axis.

    Same steps as moe_oracle.moe_forward; the two GEMMs of each expert become
    G|U = mx(X_e, W_gu[e]) (both along d) and Y = mx(H_e, W_d[e]) (both along f).
    ``matmul`` is the GEMM used (identity quantisation gives back the plain forward);
    ``wmatmul`` (default: ``matmul``) is the one for these products, whose second
    operand is a weight (mx_matmul_w4 for FP8 x FP4 experts); ``grouped`` selects the
    group-limited router as in moe_oracle.moe_forward.
    """
    wmatmul = matmul if wmatmul is None else wmatmul
    from . import moe_oracle as om
    x = np.asarray(x, dtype)
    T, d = x.shape
    E = w_gu.shape[0]
    f = w_d.shape[2]
    if grouped is not None:
        idx, w = om.route_grouped(logits, k, grouped["n_group"], grouped["topk_group"], grouped.get("bias"),
                                  grouped.get("routed_scale", 1.0), dtype)
    else:
        idx, w = om.route(logits, k, score, dtype)
    y_slot = np.zeros((T, k, d), dtype)
    g_slot = np.zeros((T, k, f), dtype)
    u_slot = np.zeros((T, k, f), dtype)
    for e in range(E):
        t_sel, j_sel = np.nonzero(idx == e)
        if t_sel.size == 0:
            continue
        wg = np.asarray(w_gu[e], dtype)
        wd = np.asarray(w_d[e], dtype)
        gu = wmatmul(x[t_sel], wg, dtype)
        g, u = gu[:, :f], gu[:, f:]
        h = w[t_sel, j_sel][:, None] * (g * om._sigmoid(g) * u)
        y_slot[t_sel, j_sel] = wmatmul(h, wd, dtype)
        g_slot[t_sel, j_sel] = g
        u_slot[t_sel, j_sel] = u
    y = np.zeros((T, d), dtype)
    for j in range(k):
        y += y_slot[:, j]
    out = {"Y": y, "idx": idx, "w": w, "g": g_slot, "u": u_slot}
    if w_gu_s is not None:
        fs = w_d_s.shape[1]
        gu = wmatmul(x, np.asarray(w_gu_s, dtype), dtype)
        g, u = gu[:, :fs], gu[:, fs:]
        out["Y"] = y + wmatmul(g * om._sigmoid(g) * u, np.asarray(w_d_s, dtype), dtype)
        out["g_s"], out["u_s"] = g, u
    return out


def moe_backward_mx(x, logits, w_gu, w_d, dy, fwd, k, score="softmax", w_gu_s=None, w_d_s=None,
                    dtype=np.float64, matmul=mx_matmul, grouped=None, wmatmul=None):
    """Backward with MXFP8 GEMM operands (quantisation treated as identity in the chain rule).

    Per expert e, rows in token order (its segment):
      dH = mx(dY_e, W_d[e]^T)         both along d           (wmatmul: weight operand)
      dX_e = mx(dGU_e, W_gu[e]^T)     both along 2f          (wmatmul: weight operand)
      dW_d[e] = mx(dY_e^T, H_e^T)     both along the rows of e
      dW_gu[e] = mx(dGU_e^T, X_e^T)   both along the rows of e
    The SwiGLU' step, dw and the router gradient are as in moe_oracle.moe_backward.
    """
    wmatmul = matmul if wmatmul is None else wmatmul
    from . import moe_oracle as om
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
        sg = om._sigmoid(g)
        a = g * sg * u
        we = w[t_sel, j_sel][:, None]
        dye = dy[t_sel]
        dh = wmatmul(dye, wd.T, dtype)
        dw[t_sel, j_sel] = (a * dh).sum(axis=1)
        da = we * dh
        dgu = np.concatenate([da * u * sg * (1.0 + g * (1.0 - sg)), da * g * sg], axis=1)
        dgu_slot[t_sel, j_sel] = dgu
        dx_slot[t_sel, j_sel] = wmatmul(dgu, wg.T, dtype)
        dw_d[e] = matmul(dye.T, (we * a).T, dtype)
        dw_gu[e] = matmul(dgu.T, x[t_sel].T, dtype)
    dx = np.zeros((T, d), dtype)
    for j in range(k):
        dx += dx_slot[:, j]
    out = {"dX": dx, "dW_gu": dw_gu, "dW_d": dw_d, "dw": dw, "dGU": dgu_slot,
           "d_logits": om.route_backward(logits, idx, w, dw, om.SIGMOID if grouped is not None else score, dtype,
                                         1.0 if grouped is None else grouped.get("routed_scale", 1.0))}
    if w_gu_s is not None:
        fs = w_d_s.shape[1]
        wg = np.asarray(w_gu_s, dtype)
        wd = np.asarray(w_d_s, dtype)
        g, u = fwd["g_s"], fwd["u_s"]
        sg = om._sigmoid(g)
        dh = wmatmul(dy, wd.T, dtype)
        dgu = np.concatenate([dh * u * sg * (1.0 + g * (1.0 - sg)), dh * g * sg], axis=1)
        out["dX"] = dx + wmatmul(dgu, wg.T, dtype)
        out["dW_d_s"] = matmul(dy.T, (g * sg * u).T, dtype)
        out["dW_gu_s"] = matmul(dgu.T, x.T, dtype)
    return out


def expert_rows_mx(x_rows, w_rows, dy_rows, w_gu_e, w_d_e, dtype=np.float64, full=True, matmul=mx_matmul,
                   wmatmul=None):
    """One expert's share of the MXFP8 layer, forward and backward, on rows routed to it.

    The loop bodies of moe_forward_mx and moe_backward_mx for a single expert (arguments
    and results as moe_oracle.expert_rows): every GEMM operand quantised along that
    GEMM's contraction; with full=True the rows are all of the expert's rows, in token
    order, so the weight gradients' row blocks start at the segment's first row.
    ``wmatmul`` (default ``matmul``) is the product whose second operand is a weight.
    """
    from . import moe_oracle as om
    wmatmul = matmul if wmatmul is None else wmatmul
    x = np.asarray(x_rows, dtype)
    dy = np.asarray(dy_rows, dtype)
    wg = np.asarray(w_gu_e, dtype)
    wd = np.asarray(w_d_e, dtype)
    f = wd.shape[1]
    we = np.asarray(w_rows, dtype)[:, None]
    gu = wmatmul(x, wg, dtype)
    g, u = gu[:, :f], gu[:, f:]
    sg = om._sigmoid(g)
    a = g * sg * u
    h = we * a
    dh = wmatmul(dy, wd.T, dtype)
    da = we * dh
    dgu = np.concatenate([da * u * sg * (1.0 + g * (1.0 - sg)), da * g * sg], axis=1)
    out = {"y": wmatmul(h, wd, dtype), "g": g, "u": u, "dw": (a * dh).sum(axis=1), "dGU": dgu,
           "dx": wmatmul(dgu, wg.T, dtype)}
    if full:
        out["dW_d"] = matmul(dy.T, h.T, dtype)
        out["dW_gu"] = matmul(dgu.T, x.T, dtype)
    return out


def expert_wgrad_sampled_mx(x, logits, dy, w_gu_e, w_d_e, e, k, gu_rows, d_cols, score="softmax",
                            dtype=np.float64, wq=None):
    """Selected entries of expert e's weight gradients in the MXFP8 layer.

    dW_gu[e][gu_rows, :] and dW_d[e][:, d_cols], by the formulas of moe_backward_mx
    restricted to the intermediate columns those entries need (each quantisation
    block lies inside one row or one column, so the restriction is exact).  ``wq`` is the
    quantise-dequantise of the weight operands (default qdq, E4M3; qdq4 for FP8 x FP4
    experts, the layer of moe_backward_mx with wmatmul=mx_matmul_w4).
    """
    from . import moe_oracle as om
    idx, w = om.route(logits, k, score, dtype)
    t_sel, j_sel = np.nonzero(idx == e)
    f = w_d_e.shape[1]
    d = w_d_e.shape[0]
    gu_rows = np.asarray(gu_rows)
    d_cols = np.asarray(d_cols)
    if t_sel.size == 0:
        return {"dW_gu_rows": np.zeros((gu_rows.size, d), dtype), "dW_d_cols": np.zeros((d, d_cols.size), dtype)}
    xe = np.asarray(x[t_sel], dtype)
    dye = np.asarray(dy[t_sel], dtype)
    wg = np.asarray(w_gu_e, dtype)
    wd = np.asarray(w_d_e, dtype)
    we = w[t_sel, j_sel][:, None]
    qx = qdq(xe)                      # X_e along d (forward)
    qdy = qdq(dye)                    # dY_e along d (dgrad)

    wq = qdq if wq is None else wq

    def gu_cols(cols):                # columns of G and U = mx(X_e, W_gu[e])
        return qx @ wq(wg[cols]).T, qx @ wq(wg[f + cols]).T

    # dW_d[:, c] = mx(dY_e^T, H_e^T): both along the rows of e
    g2, u2 = gu_cols(d_cols)
    h2 = we * g2 * om._sigmoid(g2) * u2
    dw_d_cols = qdq(dye.T) @ qdq(h2.T).T
    # dW_gu[j, :] = mx(dGU_e^T, X_e^T)
    cols = gu_rows % f
    g, u = gu_cols(cols)
    sg = om._sigmoid(g)
    dh = qdy @ wq(wd.T[cols]).T        # dH = mx(dY_e, W_d[e]^T), columns `cols`
    da = we * dh
    dg = da * u * sg * (1.0 + g * (1.0 - sg))
    du = da * g * sg
    sel = np.where((gu_rows < f)[None, :], dg, du)
    dw_gu_rows = qdq(sel.T) @ qdq(xe.T).T
    return {"dW_gu_rows": dw_gu_rows.astype(dtype), "dW_d_cols": dw_d_cols.astype(dtype)}


# ----------------------------------------------------------------------------------
# FP4 weights for FP8 x FP4 expert GEMMs (E2M1 elements, one E8M0 scale per 32)
# ----------------------------------------------------------------------------------
# The DeepGEMM Mega MoE page (itsolotime.com, Thai; section "ทิศทางการปรับปรุงใน
# ระดับลึกยิ่งขึ้น") names FP8 x FP4 mixed-precision computation as a direction and
# gives no recipe.  Readings taken here:
#   * the weights (the operand shared by every token of an expert) are E2M1: a sign,
#     two exponent bits with bias 1 and one mantissa bit, magnitudes 0, 0.5, 1, 1.5,
#     2, 3, 4, 6, no infinities or NaN; a code is the 4-bit pattern sign<<3 | exp<<1 |
#     mantissa, held in a uint8 here;
#   * one E8M0 scale per 32 consecutive elements along the contraction axis, the
#     MXFP8 block, with the same rule: 2^(floor(log2(amax)) - 2), 2 being E2M1's
#     largest exponent, clamped to [-127, 127]; an all-zero block gets byte 0;
#   * elements round to the nearest value, ties to the even code, saturating at +-6;
#   * activations and gradients stay MXFP8, so the products with a weight operand
#     (gate/up and down forward, their input gradients) are FP8 x FP4 and the weight
#     gradients (activation x gradient) stay FP8 x FP8.

E2M1_MAX = 6.0
EMAX_E2M1 = 2
E2M1_VALUES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])   # codes 0..7


def e2m1_decode(codes: np.ndarray) -> np.ndarray:
    codes = np.asarray(codes, np.uint8)
    mag = E2M1_VALUES[codes & 7]
    return np.where(codes & 8, -mag, mag)


def e2m1_encode(v: np.ndarray) -> np.ndarray:
    """Nearest E2M1 value (ties to the even code, saturating at 6) as a 4-bit code."""
    v = np.asarray(v, np.float64)
    if not np.all(np.isfinite(v)):
        raise ValueError("e2m1_encode: non-finite input")
    a = np.minimum(np.abs(v), E2M1_MAX)
    hi = np.minimum(np.searchsorted(E2M1_VALUES, a, side="left"), 7)   # first value >= a
    lo = np.maximum(hi - 1, 0)
    d_lo = a - E2M1_VALUES[lo]
    d_hi = E2M1_VALUES[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(E2M1_VALUES[hi] == a, hi, np.where(pick_hi, hi, lo)).astype(np.uint8)
    return (code | (np.signbit(v).astype(np.uint8) << 3)).astype(np.uint8)


def scale_exponent_e2m1(amax: np.ndarray) -> np.ndarray:
    """floor(log2(amax)) - 2, clamped to [-127, 127]; -127 for amax = 0."""
    amax = np.asarray(amax, np.float64)
    _, ex = np.frexp(amax)                       # amax = m 2^ex, m in [0.5, 1)
    e = ex.astype(np.int64) - 1 - EMAX_E2M1
    e = np.where(amax > 0, e, -127)
    return np.clip(e, -127, 127)


def mx4_quantize(x: np.ndarray):
    """Quantise along the last axis (a multiple of 32) to E2M1 codes and E8M0 scale bytes."""
    x = np.asarray(x, np.float64)
    K = x.shape[-1]
    if K % BLOCK:
        raise ValueError("last axis must be a multiple of 32")
    blocks = x.reshape(*x.shape[:-1], K // BLOCK, BLOCK)
    e = scale_exponent_e2m1(np.abs(blocks).max(axis=-1))
    codes = e2m1_encode(blocks * np.exp2(-e)[..., None])     # exact power-of-two scaling
    return codes.reshape(x.shape), (e + 127).astype(np.uint8)


def mx4_dequantize(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    codes = np.asarray(codes, np.uint8)
    K = codes.shape[-1]
    v = e2m1_decode(codes).reshape(*codes.shape[:-1], K // BLOCK, BLOCK)
    return (v * np.exp2(scales.astype(np.float64) - 127)[..., None]).reshape(codes.shape)


def e2m1_round(a: np.ndarray) -> np.ndarray:
    """Value of e2m1_encode, computed arithmetically: |a| rounded to the E2M1 grid.

    For |a| >= 1 the grid step is 2^(floor(log2|a|) - 1), below it 0.5 (the subnormal
    0.5); np.rint rounds half to even, which is the even code; the result saturates at 6.
    """
    a = np.asarray(a, np.float64)
    mag = np.minimum(np.abs(a), E2M1_MAX)
    _, ex = np.frexp(mag)                         # mag = m 2^ex, m in [0.5, 1)
    step = np.ldexp(1.0, np.maximum(ex - 1, 0) - 1)
    r = np.minimum(np.rint(mag / step) * step, E2M1_MAX)
    return np.copysign(r, a)


def qdq4(x: np.ndarray) -> np.ndarray:
    """E2M1 quantise-dequantise along the last axis, zero-padding it to a multiple of 32.

    Equal to mx4_dequantize(*mx4_quantize(x)) (checked in the tests), computed without
    the code table so whole expert weights stay cheap.
    """
    x = np.asarray(x, np.float64)
    K = x.shape[-1]
    pad = (-K) % BLOCK
    if pad:
        x = np.concatenate([x, np.zeros((*x.shape[:-1], pad))], axis=-1)
    blocks = x.reshape(*x.shape[:-1], x.shape[-1] // BLOCK, BLOCK)
    e = scale_exponent_e2m1(np.abs(blocks).max(axis=-1))
    scale = np.ldexp(1.0, e)[..., None]
    return (e2m1_round(blocks / scale) * scale).reshape(x.shape)[..., :K]


def mx_matmul_w4(a: np.ndarray, b: np.ndarray, dtype=np.float64) -> np.ndarray:
    """a [M,K] (activations, MXFP8) x b [N,K]^T (weights, E2M1), both blocked along K."""
    return qdq(a).astype(dtype) @ qdq4(b).astype(dtype).T
