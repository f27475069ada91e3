"""ctypes binding of libmoe.so: the C entry points under the same names.

Argument marshalling only: torch tensors (or raw integers) become device
pointers, ``dims`` becomes a ``moe_dims`` struct, ``stream`` a cudaStream_t
handle.  Every computation runs in the library's CUDA kernels; if the library is
missing this module raises instead of falling back to anything else.
Non-zero statuses raise :class:`MoeError`.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

MOE_OK = 0
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_ALIGNMENT",
                4: "MOE_ERR_WORKSPACE", 5: "MOE_ERR_CUDA", 6: "MOE_ERR_TIMEOUT", 7: "MOE_ERR_INVARIANT",
                8: "MOE_ERR_SCRATCH_LIMIT"}
SCORE = {"softmax": 0, "sigmoid": 1}
PREC = {"bf16": 0, "mxfp8": 1, "mxfp8-w4": 2}


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} returned {STATUS_NAMES.get(status, status)}")
        self.status = status


class moe_dims(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d", ctypes.c_int32), ("f", ctypes.c_int32),
                ("E", ctypes.c_int32), ("k", ctypes.c_int32), ("f_shared", ctypes.c_int32),
                ("score", ctypes.c_int32), ("prec", ctypes.c_int32)]


def make_dims(T, d, f, E, k, f_shared=0, score="softmax", prec="bf16") -> moe_dims:
    return moe_dims(T, d, f, E, k, f_shared, SCORE[score] if isinstance(score, str) else score,
                    PREC[prec] if isinstance(prec, str) else prec)


_P = ctypes.c_void_p
_I = ctypes.c_int32
_D = ctypes.POINTER(moe_dims)

# name -> (restype, argtypes)
SIGNATURES = {
    "moe_abi_version": (ctypes.c_int32, []),
    "moe_status_string": (ctypes.c_char_p, [_I]),
    "moe_check_dims": (ctypes.c_int32, [_D]),
    "moe_row_capacity": (ctypes.c_int64, [_D]),
    "moe_workspace_size": (ctypes.c_size_t, [_D]),
    "moe_launch_count": (ctypes.c_uint64, []),
    "moe_route_topk": (ctypes.c_int32, [_D, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_permute": (ctypes.c_int32, [_D, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_grouped_mlp_fwd": (ctypes.c_int32, [_D, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_combine_fwd": (ctypes.c_int32, [_D, _P, _P, _P, _P, _P]),
    "moe_combine_bwd": (ctypes.c_int32, [_D, _P, _P, _P, _P, _P, _P]),
    "moe_grouped_mlp_bwd": (ctypes.c_int32, [_D] + [_P] * 16),
    "moe_route_topk_bwd": (ctypes.c_int32, [_D, _P, _P, _P, _P, _P, _P, _P]),
    "moe_route_topk_grouped": (ctypes.c_int32, [_D, _P, _P, _I, _I, ctypes.c_float] + [_P] * 8),
    "moe_route_topk_bwd_scaled": (ctypes.c_int32, [_D, _P, _P, _P, ctypes.c_float, _P, _P, _P, _P]),
    "moe_check_status": (ctypes.c_int32, [_P, _P]),
    "moe_gemm_bf16": (ctypes.c_int32, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P]),
    "moe_gemm_gate_up": (ctypes.c_int32, [_D, _P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_gemm_down": (ctypes.c_int32, [_D, _P, _P, _P, _P, _P, _P]),
    "moe_gemm_down_dgrad": (ctypes.c_int32, [_D, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_gemm_down_wgrad": (ctypes.c_int32, [_D, _P, _P, _P, _P, _P, _P]),
    "moe_gemm_gate_up_dgrad": (ctypes.c_int32, [_D, _P, _P, _P, _P, _P, _P]),
    "moe_gemm_gate_up_wgrad": (ctypes.c_int32, [_D, _P, _P, _P, _P, _P, _P]),
    "moe_gemm_down_dgrad_noalloc": (ctypes.c_int32, [_D, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_noalloc_scratch_bytes": (ctypes.c_size_t, []),
    "moe_shared_mlp_fwd": (ctypes.c_int32, [_D, _P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_shared_mlp_bwd": (ctypes.c_int32, [_D] + [_P] * 12),
    "moe_test_wait_timeout": (ctypes.c_int32, [_P, ctypes.c_int64, _P]),
    "moe_gemm_bf16_pair": (ctypes.c_int32, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P]),
    "moe_mx_shared_weights_size": (ctypes.c_size_t, [_D]),
    "moe_mx_shared_workspace_size": (ctypes.c_size_t, [_D]),
    "moe_mx_quantize_shared_weights": (ctypes.c_int32, [_D, _P, _P, _P, _P]),
    "moe_shared_mlp_fwd_mx": (ctypes.c_int32, [_D] + [_P] * 7),
    "moe_shared_mlp_bwd_mx": (ctypes.c_int32, [_D] + [_P] * 9),
    "moe_mx_quantize_rows": (ctypes.c_int32, [_P, ctypes.c_int64, _I, ctypes.c_int64, _P, _P, _P, _P]),
    "moe_mx_quantize_cols": (ctypes.c_int32, [_P, _I, ctypes.c_int64, _I, _P, _P, _P, _P]),
    "moe_gemm_mxfp8": (ctypes.c_int32, [_P, _P, _P, _P, _P, _I, _I, _I, _P, _P]),
    "moe_mx_weights_size": (ctypes.c_size_t, [_D]),
    "moe_mx_workspace_size": (ctypes.c_size_t, [_D]),
    "moe_mx_quantize_weights": (ctypes.c_int32, [_D, _P, _P, _P, _P]),
    "moe_permute_mx": (ctypes.c_int32, [_D] + [_P] * 12),
    "moe_combine_bwd_mx": (ctypes.c_int32, [_D] + [_P] * 6),
    "moe_gemm_gate_up_mx": (ctypes.c_int32, [_D] + [_P] * 7),
    "moe_gemm_down_mx": (ctypes.c_int32, [_D] + [_P] * 6),
    "moe_gemm_down_dgrad_mx": (ctypes.c_int32, [_D] + [_P] * 9),
    "moe_gemm_down_wgrad_mx": (ctypes.c_int32, [_D] + [_P] * 5),
    "moe_gemm_gate_up_dgrad_mx": (ctypes.c_int32, [_D] + [_P] * 6),
    "moe_gemm_gate_up_wgrad_mx": (ctypes.c_int32, [_D] + [_P] * 5),
    "moe_gemm_mxf8f4": (ctypes.c_int32, [_P, _P, _P, _P, _P, _I, _I, _I, _P, _P]),
    "moe_mx4_quantize_cols": (ctypes.c_int32, [_P, _I, ctypes.c_int64, _I, _P, _P, _P, _P, _P]),
    "moe_grouped_mlp_fwd_mx": (ctypes.c_int32, [_D] + [_P] * 7),
    "moe_grouped_mlp_bwd_mx": (ctypes.c_int32, [_D] + [_P] * 11),
}

_lib: Optional[ctypes.CDLL] = None


def lib() -> ctypes.CDLL:
    """Load libmoe.so (built in-tree by __graft_entry__.build()); raise if absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _call(name: str, *args):
    st = getattr(lib(), name)(*args)
    if st != MOE_OK:
        raise MoeError(name, st)
    return st


def _d(dims: moe_dims):
    return ctypes.byref(dims)


# ------------------------------------------------------------------ entry points

def moe_abi_version() -> int:
    return lib().moe_abi_version()


def moe_status_string(status: int) -> str:
    return lib().moe_status_string(status).decode()


def moe_check_dims(dims: moe_dims) -> int:
    return lib().moe_check_dims(_d(dims))


def moe_row_capacity(dims: moe_dims) -> int:
    return lib().moe_row_capacity(_d(dims))


def moe_workspace_size(dims: moe_dims) -> int:
    return lib().moe_workspace_size(_d(dims))


def moe_launch_count() -> int:
    return lib().moe_launch_count()


def moe_route_topk(dims, logits, topk_idx, topk_w, split_sizes, offsets, row_offsets, workspace,
                   dev_status, stream=None):
    return _call("moe_route_topk", _d(dims), _ptr(logits), _ptr(topk_idx), _ptr(topk_w), _ptr(split_sizes),
                 _ptr(offsets), _ptr(row_offsets), _ptr(workspace), _ptr(dev_status), _stream(stream))


def moe_permute(dims, x, topk_idx, topk_w, split_sizes, row_offsets, workspace, xp, row_to_token,
                token_to_row, w_rows, dev_status, stream=None):
    return _call("moe_permute", _d(dims), _ptr(x), _ptr(topk_idx), _ptr(topk_w), _ptr(split_sizes),
                 _ptr(row_offsets), _ptr(workspace), _ptr(xp), _ptr(row_to_token), _ptr(token_to_row),
                 _ptr(w_rows), _ptr(dev_status), _stream(stream))


def moe_grouped_mlp_fwd(dims, xp, row_offsets, w_rows, w_gu, w_d, gu, h, y_rows, dev_status, stream=None):
    return _call("moe_grouped_mlp_fwd", _d(dims), _ptr(xp), _ptr(row_offsets), _ptr(w_rows), _ptr(w_gu),
                 _ptr(w_d), _ptr(gu), _ptr(h), _ptr(y_rows), _ptr(dev_status), _stream(stream))


def moe_combine_fwd(dims, rows, token_to_row, shared, out, stream=None):
    return _call("moe_combine_fwd", _d(dims), _ptr(rows), _ptr(token_to_row), _ptr(shared), _ptr(out),
                 _stream(stream))


def moe_combine_bwd(dims, dy, token_to_row, split_sizes, row_offsets, dy_rows, stream=None):
    return _call("moe_combine_bwd", _d(dims), _ptr(dy), _ptr(token_to_row), _ptr(split_sizes),
                 _ptr(row_offsets), _ptr(dy_rows), _stream(stream))


def moe_grouped_mlp_bwd(dims, xp, row_offsets, w_rows, w_gu, w_d, gu, h, dy_rows, dgu, dxp, dw_gu, dw_d,
                        dw_rows, workspace, dev_status, stream=None):
    return _call("moe_grouped_mlp_bwd", _d(dims), _ptr(xp), _ptr(row_offsets), _ptr(w_rows), _ptr(w_gu),
                 _ptr(w_d), _ptr(gu), _ptr(h), _ptr(dy_rows), _ptr(dgu), _ptr(dxp), _ptr(dw_gu), _ptr(dw_d),
                 _ptr(dw_rows), _ptr(workspace), _ptr(dev_status), _stream(stream))


def moe_route_topk_grouped(dims, logits, bias, n_group, topk_group, routed_scale, topk_idx, topk_w, split_sizes,
                           offsets, row_offsets, workspace, dev_status, stream=None):
    return _call("moe_route_topk_grouped", _d(dims), _ptr(logits), _ptr(bias), int(n_group), int(topk_group),
                 float(routed_scale), _ptr(topk_idx), _ptr(topk_w), _ptr(split_sizes), _ptr(offsets),
                 _ptr(row_offsets), _ptr(workspace), _ptr(dev_status), _stream(stream))


def moe_route_topk_bwd_scaled(dims, logits, topk_idx, topk_w, routed_scale, dw_rows, token_to_row, d_logits,
                              stream=None):
    return _call("moe_route_topk_bwd_scaled", _d(dims), _ptr(logits), _ptr(topk_idx), _ptr(topk_w),
                 float(routed_scale), _ptr(dw_rows), _ptr(token_to_row), _ptr(d_logits), _stream(stream))


def moe_route_topk_bwd(dims, logits, topk_idx, topk_w, dw_rows, token_to_row, d_logits, stream=None):
    return _call("moe_route_topk_bwd", _d(dims), _ptr(logits), _ptr(topk_idx), _ptr(topk_w), _ptr(dw_rows),
                 _ptr(token_to_row), _ptr(d_logits), _stream(stream))


def moe_check_status(dev_status, stream=None) -> int:
    """Synchronise the stream and return the device status word (0 = ok)."""
    return lib().moe_check_status(_ptr(dev_status), _stream(stream))


def moe_gemm_bf16(A, B, C, M, N, K, a_layout, b_layout, dev_status, stream=None):
    return _call("moe_gemm_bf16", _ptr(A), _ptr(B), _ptr(C), M, N, K, a_layout, b_layout,
                 _ptr(dev_status), _stream(stream))


def moe_gemm_gate_up(dims, xp, row_offsets, w_rows, w_gu, gu, h, dev_status, stream=None):
    return _call("moe_gemm_gate_up", _d(dims), _ptr(xp), _ptr(row_offsets), _ptr(w_rows), _ptr(w_gu),
                 _ptr(gu), _ptr(h), _ptr(dev_status), _stream(stream))


def moe_gemm_down(dims, h, row_offsets, w_d, y_rows, dev_status, stream=None):
    return _call("moe_gemm_down", _d(dims), _ptr(h), _ptr(row_offsets), _ptr(w_d), _ptr(y_rows),
                 _ptr(dev_status), _stream(stream))


def moe_gemm_down_dgrad(dims, dy_rows, row_offsets, w_rows, w_d, gu, dgu, dw_rows, workspace, dev_status,
                        stream=None):
    return _call("moe_gemm_down_dgrad", _d(dims), _ptr(dy_rows), _ptr(row_offsets), _ptr(w_rows), _ptr(w_d),
                 _ptr(gu), _ptr(dgu), _ptr(dw_rows), _ptr(workspace), _ptr(dev_status), _stream(stream))


def moe_gemm_down_wgrad(dims, dy_rows, h, row_offsets, dw_d, dev_status, stream=None):
    return _call("moe_gemm_down_wgrad", _d(dims), _ptr(dy_rows), _ptr(h), _ptr(row_offsets), _ptr(dw_d),
                 _ptr(dev_status), _stream(stream))


def moe_gemm_gate_up_dgrad(dims, dgu, row_offsets, w_gu, dxp, dev_status, stream=None):
    return _call("moe_gemm_gate_up_dgrad", _d(dims), _ptr(dgu), _ptr(row_offsets), _ptr(w_gu), _ptr(dxp),
                 _ptr(dev_status), _stream(stream))


def moe_gemm_gate_up_wgrad(dims, dgu, xp, row_offsets, dw_gu, dev_status, stream=None):
    return _call("moe_gemm_gate_up_wgrad", _d(dims), _ptr(dgu), _ptr(xp), _ptr(row_offsets), _ptr(dw_gu),
                 _ptr(dev_status), _stream(stream))


def moe_gemm_down_dgrad_noalloc(dims, dy_rows, row_offsets, w_rows, w_d, gu, dgu, dw_rows, dev_status,
                                stream=None):
    """moe_gemm_down_dgrad without a workspace: the dw partials live in the library's static array."""
    return _call("moe_gemm_down_dgrad_noalloc", _d(dims), _ptr(dy_rows), _ptr(row_offsets), _ptr(w_rows),
                 _ptr(w_d), _ptr(gu), _ptr(dgu), _ptr(dw_rows), _ptr(dev_status), _stream(stream))


def moe_noalloc_scratch_bytes() -> int:
    return lib().moe_noalloc_scratch_bytes()


def moe_shared_mlp_fwd(dims, x, w_gu_s, w_d_s, gu_s, h_s, y_s, dev_status, stream=None):
    return _call("moe_shared_mlp_fwd", _d(dims), _ptr(x), _ptr(w_gu_s), _ptr(w_d_s), _ptr(gu_s), _ptr(h_s),
                 _ptr(y_s), _ptr(dev_status), _stream(stream))


def moe_shared_mlp_bwd(dims, x, w_gu_s, w_d_s, gu_s, h_s, dy, dgu_s, dx_s, dw_gu_s, dw_d_s, dev_status,
                       stream=None):
    return _call("moe_shared_mlp_bwd", _d(dims), _ptr(x), _ptr(w_gu_s), _ptr(w_d_s), _ptr(gu_s), _ptr(h_s),
                 _ptr(dy), _ptr(dgu_s), _ptr(dx_s), _ptr(dw_gu_s), _ptr(dw_d_s), _ptr(dev_status),
                 _stream(stream))


def moe_test_wait_timeout(dev_status, limit_cycles, stream=None):
    return _call("moe_test_wait_timeout", _ptr(dev_status), limit_cycles, _stream(stream))


def moe_mx_quantize_rows(src, rows, C, ld, nrows_dev, codes, scales, stream=None):
    return _call("moe_mx_quantize_rows", _ptr(src), rows, C, ld, _ptr(nrows_dev), _ptr(codes), _ptr(scales),
                 _stream(stream))


def moe_mx_quantize_cols(src, batch, rows, C, nrows_dev, codes_t, scales, stream=None):
    return _call("moe_mx_quantize_cols", _ptr(src), batch, rows, C, _ptr(nrows_dev), _ptr(codes_t),
                 _ptr(scales), _stream(stream))


def moe_gemm_mxfp8(a, a_sf, b, b_sf, c, M, N, K, dev_status, stream=None):
    return _call("moe_gemm_mxfp8", _ptr(a), _ptr(a_sf), _ptr(b), _ptr(b_sf), _ptr(c), M, N, K,
                 _ptr(dev_status), _stream(stream))


def moe_mx_weights_size(dims) -> int:
    return lib().moe_mx_weights_size(_d(dims))


def moe_mx_workspace_size(dims) -> int:
    return lib().moe_mx_workspace_size(_d(dims))


def moe_mx_quantize_weights(dims, w_gu, w_d, wq, stream=None):
    return _call("moe_mx_quantize_weights", _d(dims), _ptr(w_gu), _ptr(w_d), _ptr(wq), _stream(stream))


def moe_permute_mx(dims, x, topk_idx, topk_w, split_sizes, row_offsets, workspace, mx_ws, row_to_token,
                   token_to_row, w_rows, dev_status, stream=None):
    return _call("moe_permute_mx", _d(dims), _ptr(x), _ptr(topk_idx), _ptr(topk_w), _ptr(split_sizes),
                 _ptr(row_offsets), _ptr(workspace), _ptr(mx_ws), _ptr(row_to_token), _ptr(token_to_row),
                 _ptr(w_rows), _ptr(dev_status), _stream(stream))


def moe_combine_bwd_mx(dims, dy, row_to_token, split_sizes, row_offsets, mx_ws, stream=None):
    return _call("moe_combine_bwd_mx", _d(dims), _ptr(dy), _ptr(row_to_token), _ptr(split_sizes),
                 _ptr(row_offsets), _ptr(mx_ws), _stream(stream))


def moe_gemm_gate_up_mx(dims, row_offsets, w_rows, wq, mx_ws, gu, dev_status, stream=None):
    return _call("moe_gemm_gate_up_mx", _d(dims), _ptr(row_offsets), _ptr(w_rows), _ptr(wq), _ptr(mx_ws),
                 _ptr(gu), _ptr(dev_status), _stream(stream))


def moe_gemm_down_mx(dims, row_offsets, wq, mx_ws, y_rows, dev_status, stream=None):
    return _call("moe_gemm_down_mx", _d(dims), _ptr(row_offsets), _ptr(wq), _ptr(mx_ws), _ptr(y_rows),
                 _ptr(dev_status), _stream(stream))


def moe_gemm_down_dgrad_mx(dims, row_offsets, w_rows, wq, mx_ws, gu, dw_rows, workspace, dev_status,
                           stream=None):
    return _call("moe_gemm_down_dgrad_mx", _d(dims), _ptr(row_offsets), _ptr(w_rows), _ptr(wq), _ptr(mx_ws),
                 _ptr(gu), _ptr(dw_rows), _ptr(workspace), _ptr(dev_status), _stream(stream))


def moe_gemm_down_wgrad_mx(dims, row_offsets, mx_ws, dw_d, dev_status, stream=None):
    return _call("moe_gemm_down_wgrad_mx", _d(dims), _ptr(row_offsets), _ptr(mx_ws), _ptr(dw_d),
                 _ptr(dev_status), _stream(stream))


def moe_gemm_gate_up_dgrad_mx(dims, row_offsets, wq, mx_ws, dxp, dev_status, stream=None):
    return _call("moe_gemm_gate_up_dgrad_mx", _d(dims), _ptr(row_offsets), _ptr(wq), _ptr(mx_ws), _ptr(dxp),
                 _ptr(dev_status), _stream(stream))


def moe_gemm_gate_up_wgrad_mx(dims, row_offsets, mx_ws, dw_gu, dev_status, stream=None):
    return _call("moe_gemm_gate_up_wgrad_mx", _d(dims), _ptr(row_offsets), _ptr(mx_ws), _ptr(dw_gu),
                 _ptr(dev_status), _stream(stream))


def moe_gemm_mxf8f4(a, a_sf, b4, b_sf, c, M, N, K, dev_status, stream=None):
    return _call("moe_gemm_mxf8f4", _ptr(a), _ptr(a_sf), _ptr(b4), _ptr(b_sf), _ptr(c), M, N, K, _ptr(dev_status),
                 _stream(stream))


def moe_mx4_quantize_cols(src, batch, rows, C, codes_t, scales_t, codes, scales, stream=None):
    return _call("moe_mx4_quantize_cols", _ptr(src), batch, rows, C, _ptr(codes_t), _ptr(scales_t), _ptr(codes),
                 _ptr(scales), _stream(stream))


def moe_grouped_mlp_fwd_mx(dims, row_offsets, w_rows, wq, mx_ws, gu, y_rows, dev_status, stream=None):
    return _call("moe_grouped_mlp_fwd_mx", _d(dims), _ptr(row_offsets), _ptr(w_rows), _ptr(wq), _ptr(mx_ws),
                 _ptr(gu), _ptr(y_rows), _ptr(dev_status), _stream(stream))


def moe_grouped_mlp_bwd_mx(dims, row_offsets, w_rows, wq, mx_ws, gu, dxp, dw_gu, dw_d, dw_rows, workspace,
                           dev_status, stream=None):
    return _call("moe_grouped_mlp_bwd_mx", _d(dims), _ptr(row_offsets), _ptr(w_rows), _ptr(wq), _ptr(mx_ws),
                 _ptr(gu), _ptr(dxp), _ptr(dw_gu), _ptr(dw_d), _ptr(dw_rows), _ptr(workspace), _ptr(dev_status),
                 _stream(stream))


def moe_mx_shared_weights_size(dims) -> int:
    return lib().moe_mx_shared_weights_size(_d(dims))


def moe_mx_shared_workspace_size(dims) -> int:
    return lib().moe_mx_shared_workspace_size(_d(dims))


def moe_mx_quantize_shared_weights(dims, w_gu_s, w_d_s, wq_s, stream=None):
    return _call("moe_mx_quantize_shared_weights", _d(dims), _ptr(w_gu_s), _ptr(w_d_s), _ptr(wq_s),
                 _stream(stream))


def moe_shared_mlp_fwd_mx(dims, x, wq_s, mx_ws_s, gu_s, y_s, dev_status, stream=None):
    return _call("moe_shared_mlp_fwd_mx", _d(dims), _ptr(x), _ptr(wq_s), _ptr(mx_ws_s), _ptr(gu_s), _ptr(y_s),
                 _ptr(dev_status), _stream(stream))


def moe_shared_mlp_bwd_mx(dims, wq_s, mx_ws_s, gu_s, dy, dx_s, dw_gu_s, dw_d_s, dev_status, stream=None):
    return _call("moe_shared_mlp_bwd_mx", _d(dims), _ptr(wq_s), _ptr(mx_ws_s), _ptr(gu_s), _ptr(dy),
                 _ptr(dx_s), _ptr(dw_gu_s), _ptr(dw_d_s), _ptr(dev_status), _stream(stream))


def moe_gemm_bf16_pair(A, B, C, M, N, K, a_layout, b_layout, dev_status, stream=None):
    return _call("moe_gemm_bf16_pair", _ptr(A), _ptr(B), _ptr(C), M, N, K, a_layout, b_layout,
                 _ptr(dev_status), _stream(stream))
