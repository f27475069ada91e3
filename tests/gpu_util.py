"""Helpers shared by the GPU parity tests (device transfer of synthetic inputs)."""
import numpy as np
import pytest
import torch


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dropless_mixture_experts_warp_gb300 import build
    build.build()


def bf16_dev(bits: np.ndarray) -> torch.Tensor:
    """uint16 bf16 bit patterns -> bf16 tensor on cuda:0."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def f32_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.float().numpy()
    return t.numpy()


def rel_err(gpu: np.ndarray, ref: np.ndarray) -> float:
    """max|gpu - ref| / max|ref| (0 when both are all zero)."""
    den = float(np.abs(ref).max()) if ref.size else 0.0
    num = float(np.abs(np.asarray(gpu, np.float64) - ref).max()) if ref.size else 0.0
    return num / den if den > 0 else num


class LazyExperts:
    """Expert weights left on the device; ``[e]`` returns expert e as a float32 host array.

    Lets the oracle's per-expert loop touch only the experts a sampled check needs,
    one at a time, instead of copying tens of GB to the host.
    """

    def __init__(self, dev_tensor: torch.Tensor):
        self.t = dev_tensor
        self.shape = tuple(dev_tensor.shape)

    def __getitem__(self, e):
        return self.t[e].float().cpu().numpy()

    def __len__(self):
        return self.shape[0]
