"""Seeded synthetic inputs for the dropless MoE layer.

This module is the only code shared by the CUDA path's harness (tests, bench,
smoke) and the CPU oracle's callers.  It draws random numbers and rounds them
to bf16; it holds none of the layer's arithmetic.  The router projection
``logits = x @ W_r + b`` is computed here because it sits outside the layer's
boundary (the layer starts at the router logits); both sides receive the same
fp32 logit bits.

Workload shapes follow the models the pages measure (Mixtral-8x7B, Qwen3-30B-A3B,
Qwen3-235B-A22B, DeepSeek-V3): NVIDIA dropless-MoE page ("Az NVIDIA szerint
tízszer gyorsabb lett a dropless MoE tanítása JAX-ban", section "A dropless MoE
minden tokent feldolgoz") and the Prime Intellect page ("Prime Mega MoE: tanításra
is jó a DeepSeek MoE kernele", section "Mit csinált a Prime Intellect?").  The
trained weights and data those pages use are not available, so every tensor is
drawn from the distributions listed per config below.

Two generators:
  * ``numpy``: PCG64 ``default_rng``; every expert's weights come from their own
    stream so a single expert can be regenerated alone (used by tests, the
    oracle-side sampling and smoke).
  * ``torch``: torch's device RNG, used by the bench to create multi-GB weight
    tensors quickly.  Seeded, deterministic, different values from ``numpy``.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional, Tuple

import numpy as np

SOFTMAX = "softmax"
SIGMOID = "sigmoid"


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int          # tokens
    d: int          # hidden size
    f: int          # expert intermediate size
    E: int          # routed experts
    k: int          # experts per token
    score: str      # "softmax" or "sigmoid"
    bias: str       # "normal", "zipf" or "zero"
    bias_param: float = 0.0      # std for "normal", exponent s for "zipf"
    forced_empty: int = 0        # experts pinned to a -1e4 bias (coldest first for zipf)
    forced_empty_ids: Tuple[int, ...] = ()
    f_shared: int = 0            # always-on shared expert width (0 = none)
    router_std: float = 0.02
    seed: int = 1000
    # group-limited sigmoid routing (0 = plain top-k): groups, eligible groups, the
    # routed scaling factor and the std of a per-expert selection bias
    n_group: int = 0
    topk_group: int = 0
    routed_scale: float = 1.0
    sel_bias_std: float = 0.0

    @property
    def R(self) -> int:
        return self.T * self.k

    def flops_fwd_bwd(self) -> float:
        """Algorithmic FLOPs of one forward+backward: 18*R*d*f (+18*T*d*f_shared)."""
        return 18.0 * self.R * self.d * self.f + 18.0 * self.T * self.d * self.f_shared


CONFIGS: Dict[str, MoEConfig] = {
    "tiny": MoEConfig("tiny", T=256, d=128, f=64, E=8, k=2, score=SOFTMAX,
                      bias="normal", bias_param=1.0, forced_empty_ids=(3,), seed=1000),
    "mixtral": MoEConfig("mixtral", T=8192, d=4096, f=14336, E=8, k=2, score=SOFTMAX,
                         bias="normal", bias_param=0.5, seed=1001),
    "qwen30b": MoEConfig("qwen30b", T=16384, d=2048, f=768, E=128, k=8, score=SOFTMAX,
                         bias="zipf", bias_param=1.1, forced_empty=2, seed=1002),
    "qwen235b": MoEConfig("qwen235b", T=16384, d=4096, f=1536, E=128, k=8, score=SOFTMAX,
                          bias="zero", seed=1003),
    "qwen235b-zipf": MoEConfig("qwen235b-zipf", T=16384, d=4096, f=1536, E=128, k=8,
                               score=SOFTMAX, bias="zipf", bias_param=1.2, seed=1004),
    # profiling case: the Mixtral per-expert GEMM shapes (about 2048 rows per expert)
    # with two experts, so an ncu capture stays near 2 GB of device memory
    "mixtral-e2": MoEConfig("mixtral-e2", T=4096, d=4096, f=14336, E=2, k=1, score=SOFTMAX,
                            bias="normal", bias_param=0.1, seed=1006),
    # profiling case: the Qwen3-235B-A22B per-expert shapes (about 1024 rows per expert)
    # with 16 experts, near 2 GB of device memory
    "qwen235b-e16": MoEConfig("qwen235b-e16", T=2048, d=4096, f=1536, E=16, k=8, score=SOFTMAX,
                              bias="zero", seed=1007),
    # profiling case for the memory-bound kernels: token rows far larger than L2
    # (x 256 MB, routed rows 512 MB) with small experts
    "hbm-probe": MoEConfig("hbm-probe", T=32768, d=4096, f=128, E=8, k=2, score=SOFTMAX,
                           bias="normal", bias_param=0.5, seed=1008),
    # profiling case for the ragged-K weight gradients: DeepSeek-V3's expert width
    # (f = 2048) and routing (sigmoid, Zipf(1.0) load, top-8) at about 256 rows per expert
    # and 64 experts, near 3.5 GB of device memory
    "dsv3-proxy": MoEConfig("dsv3-proxy", T=2048, d=2048, f=2048, E=64, k=8, score=SIGMOID,
                            bias="zipf", bias_param=1.0, forced_empty=1, seed=1010),
    # DeepSeek-V3 shape with its group-limited router: 8 groups of 32, 4 eligible,
    # routed scale 2.5, a small per-expert selection bias
    "dsv3-grouped": MoEConfig("dsv3-grouped", T=16384, d=7168, f=2048, E=256, k=8, score=SIGMOID,
                              bias="zipf", bias_param=1.0, forced_empty=4, f_shared=2048, seed=1009,
                              n_group=8, topk_group=4, routed_scale=2.5, sel_bias_std=0.05),
    "dsv3": MoEConfig("dsv3", T=16384, d=7168, f=2048, E=256, k=8, score=SIGMOID,
                      bias="zipf", bias_param=1.0, forced_empty=4, f_shared=2048, seed=1005),
}


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (round to nearest, ties to even); returns the uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    rounding = ((u >> 16) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + rounding) >> 16).astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 exactly."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _expert_rng(cfg: MoEConfig, tag: int, e: int) -> np.random.Generator:
    return np.random.default_rng([cfg.seed, tag, e])


def expert_weights(cfg: MoEConfig, e: int) -> Tuple[np.ndarray, np.ndarray]:
    """bf16 bits of one routed expert: W_gu[e] (2f x d, gate rows then up rows), W_d[e] (d x f).

    nn.Linear convention [out, in]; entries N(0, 1/sqrt(fan_in)) with fan_in = d for
    the gate/up projection and f for the down projection.
    """
    rng = _expert_rng(cfg, 1, e)
    w_gu = rng.standard_normal((2 * cfg.f, cfg.d), dtype=np.float32) * np.float32(1.0 / math.sqrt(cfg.d))
    w_d = rng.standard_normal((cfg.d, cfg.f), dtype=np.float32) * np.float32(1.0 / math.sqrt(cfg.f))
    return bf16_bits(w_gu), bf16_bits(w_d)


def shared_weights(cfg: MoEConfig) -> Tuple[np.ndarray, np.ndarray]:
    """bf16 bits of the always-on shared expert: W_gu_s (2 f_s x d), W_d_s (d x f_s)."""
    assert cfg.f_shared > 0
    rng = _expert_rng(cfg, 2, 0)
    fs = cfg.f_shared
    w_gu = rng.standard_normal((2 * fs, cfg.d), dtype=np.float32) * np.float32(1.0 / math.sqrt(cfg.d))
    w_d = rng.standard_normal((cfg.d, fs), dtype=np.float32) * np.float32(1.0 / math.sqrt(fs))
    return bf16_bits(w_gu), bf16_bits(w_d)


def router_bias(cfg: MoEConfig) -> np.ndarray:
    """Per-expert logit bias that skews the load (fp32, length E)."""
    rng = _expert_rng(cfg, 3, 0)
    E = cfg.E
    if cfg.bias == "normal":
        b = rng.standard_normal(E, dtype=np.float32) * np.float32(cfg.bias_param)
    elif cfg.bias == "zero":
        b = np.zeros(E, np.float32)
    elif cfg.bias == "zipf":
        # Expert perm[r] gets popularity rank r+1; bias = ln(pmf) with pmf ~ rank^-s.
        perm = rng.permutation(E)
        ranks = np.arange(1, E + 1, dtype=np.float64)
        pmf = ranks ** (-cfg.bias_param)
        pmf /= pmf.sum()
        b = np.empty(E, np.float32)
        b[perm] = np.log(pmf).astype(np.float32)
        for r in range(cfg.forced_empty):          # coldest ranks
            b[perm[E - 1 - r]] = np.float32(-1e4)
    else:
        raise ValueError(cfg.bias)
    for e in cfg.forced_empty_ids:
        b[e] = np.float32(-1e4)
    return b


def selection_bias(cfg: MoEConfig) -> np.ndarray:
    """Per-expert selection bias [E] fp32 of the group-limited router (zeros if unused)."""
    if not cfg.n_group or cfg.sel_bias_std == 0.0:
        return np.zeros(cfg.E, np.float32)
    return (np.random.default_rng(cfg.seed + 31).standard_normal(cfg.E) * cfg.sel_bias_std).astype(np.float32)


def grouped_options(cfg: MoEConfig):
    """The group-limited routing options of a config as plain values (None if plain top-k)."""
    if not cfg.n_group:
        return None
    return {"n_group": cfg.n_group, "topk_group": cfg.topk_group, "routed_scale": cfg.routed_scale,
            "bias": selection_bias(cfg)}


def token_inputs(cfg: MoEConfig, T: Optional[int] = None) -> Dict[str, np.ndarray]:
    """Activations of the step: x (bf16 bits [T,d]), logits (fp32 [T,E]), dY (bf16 bits [T,d]).

    logits = fp32(x) @ W_r + b with W_r ~ N(0, router_std); this router projection
    lies outside the layer and is done once here so both sides see the same bits.
    """
    T = cfg.T if T is None else T
    rng = _expert_rng(cfg, 0, 0)
    x = bf16_bits(rng.standard_normal((T, cfg.d), dtype=np.float32))
    w_r = rng.standard_normal((cfg.d, cfg.E), dtype=np.float32) * np.float32(cfg.router_std)
    dy = bf16_bits(rng.standard_normal((T, cfg.d), dtype=np.float32))
    logits = (bf16_to_f32(x) @ w_r + router_bias(cfg)[None, :]).astype(np.float32)
    return {"x": x, "logits": np.ascontiguousarray(logits), "dy": dy}


def all_expert_weights(cfg: MoEConfig) -> Tuple[np.ndarray, np.ndarray]:
    """Stacked bf16 bits W_gu [E,2f,d] and W_d [E,d,f] (numpy generator, expert by expert)."""
    w_gu = np.empty((cfg.E, 2 * cfg.f, cfg.d), np.uint16)
    w_d = np.empty((cfg.E, cfg.d, cfg.f), np.uint16)
    for e in range(cfg.E):
        w_gu[e], w_d[e] = expert_weights(cfg, e)
    return w_gu, w_d


def small_config(name: str = "small", *, T: int, d: int, f: int, E: int, k: int,
                 score: str = SOFTMAX, bias: str = "normal", bias_param: float = 1.0,
                 forced_empty_ids: Tuple[int, ...] = (), f_shared: int = 0,
                 seed: int = 7, router_std: float = 0.02, forced_empty: int = 0) -> MoEConfig:
    """An ad-hoc configuration for parity and edge-case tests."""
    return MoEConfig(name, T=T, d=d, f=f, E=E, k=k, score=score, bias=bias,
                     bias_param=bias_param, forced_empty=forced_empty,
                     forced_empty_ids=forced_empty_ids, f_shared=f_shared,
                     router_std=router_std, seed=seed)


def torch_inputs(cfg: MoEConfig, device, seed: Optional[int] = None):
    """Device-resident inputs drawn with torch's RNG (fast path for large configs).

    Returns a dict of torch tensors: x, dy (bf16), logits (fp32), w_gu, w_d (bf16),
    and w_gu_s, w_d_s when the config has a shared expert.  Same distributions as
    the numpy generator, different values.
    """
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(cfg.seed if seed is None else seed)
    T, d, f, E = cfg.T, cfg.d, cfg.f, cfg.E

    def randn(*shape, scale=1.0):
        out = torch.empty(shape, dtype=torch.bfloat16, device=device)
        # draw in chunks so the fp32 temporary stays small
        flat = out.view(-1)
        step = 1 << 28
        for s in range(0, flat.numel(), step):
            n = min(step, flat.numel() - s)
            flat[s:s + n] = (torch.randn(n, generator=g, device=device) * scale).to(torch.bfloat16)
        return out

    out = {}
    out["x"] = randn(T, d)
    w_r = torch.randn(d, E, generator=g, device=device) * cfg.router_std
    b = torch.from_numpy(router_bias(cfg)).to(device)
    out["logits"] = (out["x"].float() @ w_r + b[None, :]).contiguous()
    out["dy"] = randn(T, d)
    out["w_gu"] = randn(E, 2 * f, d, scale=1.0 / math.sqrt(d))
    out["w_d"] = randn(E, d, f, scale=1.0 / math.sqrt(f))
    if cfg.f_shared:
        fs = cfg.f_shared
        out["w_gu_s"] = randn(2 * fs, d, scale=1.0 / math.sqrt(d))
        out["w_d_s"] = randn(d, fs, scale=1.0 / math.sqrt(fs))
    return out
