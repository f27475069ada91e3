"""MXFP8 building blocks on the GPU against the oracle: quantisers bit for bit, the
block-scaled tcgen05 GEMM against a dequantised matmul."""
import numpy as np
import pytest
import torch

from gpu_util import bf16_dev, host, need_gpu, rel_err
from oracle import mx
from dropless_mixture_experts_warp_gb300 import synth

pytestmark = pytest.mark.gpu


def sf_tiles(scales: np.ndarray) -> np.ndarray:
    """Scale bytes [R][K/32] (R % 128 == 0, K % 128 == 0) in the library's SF-tile layout."""
    R, G = scales.shape
    kt = G // 4
    out = np.zeros(R * G, np.uint8)
    r = np.arange(R)[:, None]
    g = np.arange(G)[None, :]
    off = ((r // 128) * kt + g // 4) * 512 + ((r % 32) * 4 + (r % 128) // 32) * 4 + g % 4
    out[off.ravel()] = scales.ravel()
    return out


def scales_from_tiles(buf: np.ndarray, R: int, K: int) -> np.ndarray:
    G = K // 32
    r = np.arange(R)[:, None]
    g = np.arange(G)[None, :]
    off = ((r // 128) * (G // 4) + g // 4) * 512 + ((r % 32) * 4 + (r % 128) // 32) * 4 + g % 4
    return buf[off]


def _bf16_matrix_with_every_value(rows, cols, seed):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = synth.bf16_to_f32(bits)
    bits = bits[np.isfinite(v)]
    rng = np.random.default_rng(seed)
    out = bits[rng.integers(0, bits.size, rows * cols)]
    out[: bits.size] = rng.permutation(bits)[: min(bits.size, rows * cols)]
    m = out.reshape(rows, cols)
    m[0, :32] = 0                                   # all-zero block
    m[0, 32:64] = synth.bf16_bits(np.full(32, 448.0, np.float32))
    m[0, 64:96] = synth.bf16_bits(np.full(32, 449.0, np.float32))
    m[0, 96:128] = 0x8000                           # -0
    m[1, :32] = 0x0001                              # smallest subnormal
    return m


def test_quantize_rows_bit_exact_including_every_bf16_value():
    need_gpu()
    from dropless_mixture_experts_warp_gb300 import binding as B
    rows, C = 256, 512
    m = _bf16_matrix_with_every_value(rows, C, 1)
    codes = torch.zeros(rows, C, dtype=torch.uint8, device="cuda")
    sf = torch.zeros(rows * C // 32, dtype=torch.uint8, device="cuda")
    B.moe_mx_quantize_rows(bf16_dev(m), rows, C, C, None, codes, sf)
    torch.cuda.synchronize()
    ref_codes, ref_sc = mx.mx_quantize(synth.bf16_to_f32(m).astype(np.float64))
    got = host(codes)
    assert np.array_equal(got, ref_codes), np.argwhere(got != ref_codes)[:5]
    assert np.array_equal(scales_from_tiles(host(sf), rows, C), ref_sc)


def test_quantize_rows_respects_row_count_and_stride():
    need_gpu()
    from dropless_mixture_experts_warp_gb300 import binding as B
    rows, C, ld = 256, 256, 384
    rng = np.random.default_rng(2)
    m = synth.bf16_bits(rng.standard_normal((rows, ld)).astype(np.float32))
    codes = torch.full((rows, C), 0xAB, dtype=torch.uint8, device="cuda")
    sf = torch.zeros(rows * C // 32, dtype=torch.uint8, device="cuda")
    n = torch.tensor([200], dtype=torch.int32, device="cuda")
    B.moe_mx_quantize_rows(bf16_dev(m), rows, C, ld, n, codes, sf)
    torch.cuda.synchronize()
    ref_codes, ref_sc = mx.mx_quantize(synth.bf16_to_f32(m[:, :C]).astype(np.float64))
    got = host(codes)
    assert np.array_equal(got[:200], ref_codes[:200]) and np.all(got[200:] == 0xAB)
    assert np.array_equal(scales_from_tiles(host(sf), rows, C)[:200], ref_sc[:200])


def test_quantize_cols_bit_exact():
    need_gpu()
    from dropless_mixture_experts_warp_gb300 import binding as B
    batch, rows, C = 2, 256, 384
    m = _bf16_matrix_with_every_value(batch * rows, C, 3).reshape(batch, rows, C)
    codes = torch.zeros(batch, C, rows, dtype=torch.uint8, device="cuda")
    sf = torch.zeros(batch * C * rows // 32, dtype=torch.uint8, device="cuda")
    B.moe_mx_quantize_cols(bf16_dev(m), batch, rows, C, None, codes, sf)
    torch.cuda.synchronize()
    got = host(codes)
    sfh = host(sf).reshape(batch, -1)
    for b in range(batch):
        ref_codes, ref_sc = mx.mx_quantize(synth.bf16_to_f32(m[b]).astype(np.float64).T)
        assert np.array_equal(got[b], ref_codes)
        assert np.array_equal(scales_from_tiles(sfh[b], C, rows), ref_sc)


@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (256, 256, 512), (384, 128, 256), (128, 256, 1024),
                                   (512, 512, 2048)])
def test_mxfp8_gemm_matches_dequantised_matmul(M, N, K):
    need_gpu()
    from dropless_mixture_experts_warp_gb300 import binding as B
    rng = np.random.default_rng(M + N + K)
    a = rng.standard_normal((M, K)) * np.exp2(rng.integers(-6, 6, (M, 1)))
    b = rng.standard_normal((N, K)) * np.exp2(rng.integers(-6, 6, (1, K)))
    ac, asc = mx.mx_quantize(a)
    bc, bsc = mx.mx_quantize(b)
    ref = mx.mx_dequantize(ac, asc) @ mx.mx_dequantize(bc, bsc).T
    C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()  # noqa: E731
    B.moe_gemm_mxfp8(dev(ac), dev(sf_tiles(asc)), dev(bc), dev(sf_tiles(bsc)), C, M, N, K, status)
    assert B.moe_check_status(status) == 0
    assert rel_err(host(C), ref) < 5e-3
