"""The C-ABI library builds, loads and exports every symbol include/moe.h declares.

Host-only: no call here reaches a GPU (argument errors are found on the host).
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from dropless_mixture_experts_warp_gb300 import build, binding
    build.build()
    return binding.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("moe_route_topk", "moe_permute", "moe_grouped_mlp_fwd", "moe_grouped_mlp_bwd",
                     "moe_combine_fwd", "moe_combine_bwd", "moe_route_topk_bwd", "moe_check_status"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    from dropless_mixture_experts_warp_gb300 import binding
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in binding.SIGNATURES, name
        assert callable(getattr(binding, name)), name


def test_host_queries(lib):
    from dropless_mixture_experts_warp_gb300 import binding as B
    assert B.moe_abi_version() == 1
    assert B.moe_status_string(0) == "ok"
    dims = B.make_dims(256, 128, 64, 8, 2)
    assert B.moe_check_dims(dims) == 0
    assert B.moe_row_capacity(dims) == 512 + 128 * 8
    assert B.moe_workspace_size(dims) > 0
    bad = [B.make_dims(256, 128, 64, 8, 9),     # k > E
           B.make_dims(256, 128, 64, 8, 0),     # k = 0
           B.make_dims(-1, 128, 64, 8, 2),      # T < 0
           B.make_dims(256, 128, 64, 8, 2, score=5)]
    for dm in bad:
        assert B.moe_check_dims(dm) == 1
    assert B.moe_check_dims(B.make_dims(256, 96, 64, 8, 2)) == 2      # d % 128
    assert B.moe_check_dims(B.make_dims(256, 128, 48, 8, 2)) == 2     # f % 64
    assert B.moe_check_dims(B.make_dims(256, 128, 64, 2048, 2)) == 2  # E > 1024
    assert B.moe_row_capacity(B.make_dims(256, 128, 64, 8, 9)) == -1


def test_argument_errors_are_returned_without_launching(lib):
    from dropless_mixture_experts_warp_gb300 import binding as B
    dims = B.make_dims(256, 128, 64, 8, 2)
    before = B.moe_launch_count()
    with pytest.raises(B.MoeError) as e:
        B.moe_route_topk(dims, None, None, None, None, None, None, None, None, stream=0)
    assert e.value.status == 1
    with pytest.raises(B.MoeError) as e:   # workspace missing
        B.moe_route_topk(dims, 16, 16, 16, 16, 16, 16, None, 16, stream=0)
    assert e.value.status == 4
    with pytest.raises(B.MoeError) as e:   # misaligned activation pointer
        B.moe_permute(dims, 18, 16, 16, 16, 16, 16, 16, 16, 16, 16, 16, stream=0)
    assert e.value.status == 3
    with pytest.raises(B.MoeError) as e:
        B.moe_gemm_bf16(16, 16, 16, 128, 100, 64, 0, 0, 16, stream=0)   # N % 64
    assert e.value.status == 2
    assert B.moe_launch_count() == before


def test_grouped_routing_and_mxfp8_argument_checks(lib):
    from dropless_mixture_experts_warp_gb300 import binding as B
    before = B.moe_launch_count()
    sig = B.make_dims(256, 128, 64, 16, 4, score="sigmoid")
    p = 16                                      # any aligned non-null pointer: nothing is launched

    def grouped(dims, n_group, topk_group, scale):
        with pytest.raises(B.MoeError) as e:
            B.moe_route_topk_grouped(dims, p, None, n_group, topk_group, scale, p, p, p, p, p, p, p, stream=0)
        return e.value.status

    assert grouped(sig, 3, 2, 1.0) == 1         # 16 experts do not split into 3 groups
    assert grouped(sig, 4, 5, 1.0) == 1         # more eligible groups than groups
    assert grouped(sig, 8, 1, 1.0) == 1         # k = 4 > 1 group of 2 experts
    assert grouped(sig, 4, 2, 0.0) == 1         # routed scale must be positive
    assert grouped(sig, 16, 4, 1.0) == 1        # groups of one expert
    soft = B.make_dims(256, 128, 64, 16, 4)
    assert grouped(soft, 4, 2, 1.0) == 1        # group-limited routing is sigmoid-only
    mx = B.make_dims(256, 128, 64, 8, 2, prec="mxfp8")
    assert B.moe_check_dims(mx) == 2            # MXFP8 needs f % 128
    assert B.moe_mx_weights_size(mx) == 0 and B.moe_mx_workspace_size(mx) == 0
    ok = B.make_dims(256, 128, 128, 8, 2, prec="mxfp8")
    assert B.moe_check_dims(ok) == 0
    # codes (1 byte) and scales (1/32) of both weights in both orientations
    assert B.moe_mx_weights_size(ok) >= 2 * 3 * 8 * 128 * 128 * (1 + 1 / 32)
    assert B.moe_launch_count() == before
