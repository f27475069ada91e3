"""One dropless MoE layer step through the C ABI: buffers and the call sequence.

PyTorch only allocates device memory and provides the stream; every step runs in
libmoe.so's kernels.  Forward: route -> permute -> grouped MLP -> combine.
Backward: combine_bwd -> grouped MLP backward -> un-permute (combine of dXp) ->
route backward.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import binding as B


@dataclass
class Buffers:
    dims: B.moe_dims
    rows: int
    topk_idx: torch.Tensor
    topk_w: torch.Tensor
    split_sizes: torch.Tensor
    offsets: torch.Tensor
    row_offsets: torch.Tensor
    xp: torch.Tensor
    row_to_token: torch.Tensor
    token_to_row: torch.Tensor
    w_rows: torch.Tensor
    gu: torch.Tensor
    h: torch.Tensor
    y_rows: torch.Tensor
    y: torch.Tensor
    dy_rows: torch.Tensor
    dgu: torch.Tensor
    dxp: torch.Tensor
    dw_gu: torch.Tensor
    dw_d: torch.Tensor
    dw_rows: torch.Tensor
    dx: torch.Tensor
    d_logits: torch.Tensor
    workspace: torch.Tensor
    status: torch.Tensor
    # shared expert (dims.f_shared > 0), else None
    gu_s: torch.Tensor = None
    h_s: torch.Tensor = None
    y_s: torch.Tensor = None
    dgu_s: torch.Tensor = None
    dx_s: torch.Tensor = None
    dw_gu_s: torch.Tensor = None
    dw_d_s: torch.Tensor = None
    # MXFP8 path (dims.prec == mxfp8): quantised weights and activation scratch
    wq: torch.Tensor = None
    mx_ws: torch.Tensor = None
    wq_s: torch.Tensor = None
    mx_ws_s: torch.Tensor = None


def dims_of(T, d, f, E, k, f_shared=0, score="softmax", prec="bf16") -> B.moe_dims:
    dims = B.make_dims(T, d, f, E, k, f_shared, score, prec)
    st = B.moe_check_dims(dims)
    if st != B.MOE_OK:
        raise B.MoeError("moe_check_dims", st)
    return dims


def allocate(dims: B.moe_dims, device="cuda") -> Buffers:
    T, d, f, E, k = dims.T, dims.d, dims.f, dims.E, dims.k
    rows = B.moe_row_capacity(dims)
    i32, f32, bf = torch.int32, torch.float32, torch.bfloat16
    e = lambda *s, dt=bf: torch.empty(*s, dtype=dt, device=device)  # noqa: E731
    shared = {}
    if dims.f_shared:
        fs = dims.f_shared
        shared = dict(gu_s=e(T, 2 * fs), h_s=e(T, fs), y_s=e(T, d), dgu_s=e(T, 2 * fs), dx_s=e(T, d),
                      dw_gu_s=e(2 * fs, d), dw_d_s=e(d, fs))
    if dims.prec in (1, 2):
        shared["wq"] = torch.empty(B.moe_mx_weights_size(dims), dtype=torch.uint8, device=device)
        shared["mx_ws"] = torch.empty(B.moe_mx_workspace_size(dims), dtype=torch.uint8, device=device)
        if dims.f_shared:
            shared["wq_s"] = torch.empty(B.moe_mx_shared_weights_size(dims), dtype=torch.uint8, device=device)
            shared["mx_ws_s"] = torch.empty(max(1, B.moe_mx_shared_workspace_size(dims)), dtype=torch.uint8,
                                            device=device)
    return Buffers(**shared,
        dims=dims, rows=rows,
        topk_idx=e(T, k, dt=i32), topk_w=e(T, k, dt=f32), split_sizes=e(E, dt=i32),
        offsets=e(E + 1, dt=i32), row_offsets=e(E + 1, dt=i32),
        xp=e(rows, d), row_to_token=e(rows, dt=i32), token_to_row=e(T, k, dt=i32), w_rows=e(rows, dt=f32),
        gu=e(rows, 2 * f), h=e(rows, f), y_rows=e(rows, d), y=e(T, d),
        dy_rows=e(rows, d), dgu=e(rows, 2 * f), dxp=e(rows, d),
        dw_gu=e(E, 2 * f, d), dw_d=e(E, d, f), dw_rows=e(rows, dt=f32), dx=e(T, d), d_logits=e(T, E, dt=f32),
        workspace=torch.empty(max(1, B.moe_workspace_size(dims)), dtype=torch.uint8, device=device),
        status=torch.zeros(1, dtype=i32, device=device),
    )


def quantize_weights(b: Buffers, w_gu, w_d, stream=None, w_gu_s=None, w_d_s=None):
    """MXFP8: the 16-bit master weights -> b.wq (and b.wq_s for the shared expert), codes and
    scales in both contraction orientations.  The weights change once per optimiser step, so a
    step of several micro-batches quantises them once and passes weights_cached=True to every
    forward() of the step."""
    dm = b.dims
    if dm.prec not in (1, 2):
        raise ValueError("quantize_weights: the layer is not MXFP8")
    B.moe_mx_quantize_weights(dm, w_gu, w_d, b.wq, stream)
    if dm.f_shared:
        B.moe_mx_quantize_shared_weights(dm, w_gu_s, w_d_s, b.wq_s, stream)


def forward(b: Buffers, x, logits, w_gu, w_d, stream=None, w_gu_s=None, w_d_s=None, grouped=None,
            weights_cached=False):
    """grouped: {"n_group", "topk_group", "bias" (device [E] fp32 or None), "routed_scale"} selects the
    group-limited sigmoid router instead of the plain top-k.  weights_cached (MXFP8): b.wq (and
    b.wq_s) already hold this step's quantised weights (quantize_weights()), so they are not
    quantised again."""
    dm = b.dims
    mx8 = dm.prec in (1, 2)   # MXFP8, or FP8 x FP4 (MXFP4 weights)
    if mx8 and not weights_cached:
        quantize_weights(b, w_gu, w_d, stream, w_gu_s, w_d_s)
    shared_out = None
    if dm.f_shared and mx8:
        B.moe_shared_mlp_fwd_mx(dm, x, b.wq_s, b.mx_ws_s, b.gu_s, b.y_s, b.status, stream)
        shared_out = b.y_s
    elif dm.f_shared:
        B.moe_shared_mlp_fwd(dm, x, w_gu_s, w_d_s, b.gu_s, b.h_s, b.y_s, b.status, stream)
        shared_out = b.y_s
    if grouped is not None:
        B.moe_route_topk_grouped(dm, logits, grouped.get("bias"), grouped["n_group"], grouped["topk_group"],
                                 grouped.get("routed_scale", 1.0), b.topk_idx, b.topk_w, b.split_sizes,
                                 b.offsets, b.row_offsets, b.workspace, b.status, stream)
    else:
        B.moe_route_topk(dm, logits, b.topk_idx, b.topk_w, b.split_sizes, b.offsets, b.row_offsets,
                         b.workspace, b.status, stream)
    if mx8:
        B.moe_permute_mx(dm, x, b.topk_idx, b.topk_w, b.split_sizes, b.row_offsets, b.workspace, b.mx_ws,
                         b.row_to_token, b.token_to_row, b.w_rows, b.status, stream)
        B.moe_grouped_mlp_fwd_mx(dm, b.row_offsets, b.w_rows, b.wq, b.mx_ws, b.gu, b.y_rows, b.status, stream)
    else:
        B.moe_permute(dm, x, b.topk_idx, b.topk_w, b.split_sizes, b.row_offsets, b.workspace, b.xp,
                      b.row_to_token, b.token_to_row, b.w_rows, b.status, stream)
        B.moe_grouped_mlp_fwd(dm, b.xp, b.row_offsets, b.w_rows, w_gu, w_d, b.gu, b.h, b.y_rows, b.status,
                              stream)
    B.moe_combine_fwd(dm, b.y_rows, b.token_to_row, shared_out, b.y, stream)
    return b.y


def backward(b: Buffers, dy, logits, w_gu, w_d, stream=None, x=None, w_gu_s=None, w_d_s=None, grouped=None):
    """x (the forward's input) is needed by the shared expert and by the MXFP8 path; grouped as in
    forward()."""
    dm = b.dims
    mx8 = dm.prec in (1, 2)   # MXFP8, or FP8 x FP4 (MXFP4 weights)
    shared_dx = None
    if dm.f_shared and mx8:
        B.moe_shared_mlp_bwd_mx(dm, b.wq_s, b.mx_ws_s, b.gu_s, dy, b.dx_s, b.dw_gu_s, b.dw_d_s, b.status,
                                stream)
        shared_dx = b.dx_s
    elif dm.f_shared:
        B.moe_shared_mlp_bwd(dm, x, w_gu_s, w_d_s, b.gu_s, b.h_s, dy, b.dgu_s, b.dx_s, b.dw_gu_s, b.dw_d_s,
                             b.status, stream)
        shared_dx = b.dx_s
    if mx8:
        B.moe_combine_bwd_mx(dm, dy, b.row_to_token, b.split_sizes, b.row_offsets, b.mx_ws, stream)
        B.moe_grouped_mlp_bwd_mx(dm, b.row_offsets, b.w_rows, b.wq, b.mx_ws, b.gu, b.dxp, b.dw_gu, b.dw_d,
                                 b.dw_rows, b.workspace, b.status, stream)
    else:
        B.moe_combine_bwd(dm, dy, b.token_to_row, b.split_sizes, b.row_offsets, b.dy_rows, stream)
        B.moe_grouped_mlp_bwd(dm, b.xp, b.row_offsets, b.w_rows, w_gu, w_d, b.gu, b.h, b.dy_rows, b.dgu,
                              b.dxp, b.dw_gu, b.dw_d, b.dw_rows, b.workspace, b.status, stream)
    B.moe_combine_fwd(dm, b.dxp, b.token_to_row, shared_dx, b.dx, stream)
    if grouped is not None:
        B.moe_route_topk_bwd_scaled(dm, logits, b.topk_idx, b.topk_w, grouped.get("routed_scale", 1.0), b.dw_rows,
                                    b.token_to_row, b.d_logits, stream)
    else:
        B.moe_route_topk_bwd(dm, logits, b.topk_idx, b.topk_w, b.dw_rows, b.token_to_row, b.d_logits, stream)
    return b.dx


def check(b: Buffers, stream=None):
    st = B.moe_check_status(b.status, stream)
    if st != B.MOE_OK:
        raise B.MoeError("device status", st)
