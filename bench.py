#!/usr/bin/env python
"""Throughput of one dropless MoE layer step (forward + backward) on GB300.

A step is the whole hot path on one batch: route -> permute -> grouped GEMM
gate/up (+SwiGLU*w) -> grouped GEMM down -> combine -> combine backward ->
grouped-GEMM backward (4 GEMMs) -> un-permute -> route backward (plus, for the
DeepSeek-V3 shape, the always-on shared expert; for MXFP8, the per-step
quantisation of the 16-bit master weights).

Default workload: the DeepSeek-V3-shaped routed-expert layer (T=16384 tokens,
d=7168, f=2048, E=256, top-8, sigmoid scores with a Zipf(1.0) per-expert bias,
plus one shared expert of width 2048), the largest single-GPU configuration:
the headline is its bf16 step (bf16 operands, fp32 accumulation), and the same
line carries its MXFP8 step (E4M3 values, one E8M0 scale per 32 along each
GEMM's contraction) under "mxfp8".  Inputs are synthetic (seeded) and resident in
HBM; the 22.5 GB of expert weights exceed the 129 MB L2, so no flush is needed
between steps.

  python bench.py [--gpus N --steps K --warmup W] [--config NAME] [--prec P]
                  [--second-prec mxfp8|none] [--impl reference]

--impl reference times the CPU oracle (the plain NumPy implementation the tests
compare against) on the host cores, on a bounded token sample of the same
workload per step.  Under torchrun, rank 0 alone runs it.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE layer fwd+bwd TFLOPS & tokens/s on 1 GB300; % of bf16/MXFP8 tensor peak"
UNIT = "TFLOP/s"
MX_PRECS = ("mxfp8", "mxfp8-w4")   # block-scaled precisions: the MXFP8 layer calls
GEMMS = ["gate_up", "down", "down_dgrad", "down_wgrad", "gate_up_dgrad", "gate_up_wgrad"]
GEMM_FLOP_FACTOR = {"gate_up": 4, "down": 2, "down_dgrad": 2, "down_wgrad": 2, "gate_up_dgrad": 4,
                    "gate_up_wgrad": 4}   # x R*d*f
GEMM_KERNEL_MX = {"gate_up": "grouped_gemm_mx_kernel<0,3>", "down": "grouped_gemm_mx_kernel<0,0>",
                  "down_dgrad": "grouped_gemm_mx_kernel<0,4> + dw_reduce_kernel",
                  "down_wgrad": "grouped_gemm_mx_pair_kernel<1>", "gate_up_dgrad": "grouped_gemm_mx_kernel<0,0>",
                  "gate_up_wgrad": "grouped_gemm_mx_pair_kernel<1>"}
GEMM_KERNEL = {"gate_up": "grouped_gemm_pair_kernel<0,1,0,0>", "down": "grouped_gemm_pair_kernel<0,0,0,0>",
               "down_dgrad": "grouped_gemm_pair_kernel<0,2,0,1> + dw_reduce_kernel",
               "down_wgrad": "grouped_gemm_pair_kernel<1,0,1,1>", "gate_up_dgrad": "grouped_gemm_pair_kernel<0,0,0,1>",
               "gate_up_wgrad": "grouped_gemm_pair_kernel<1,0,1,1>"}


def workload_name(cfg) -> str:
    names = {"tiny": "tiny MoE layer", "mixtral": "Mixtral-8x7B-shaped MoE layer",
             "qwen30b": "Qwen3-30B-A3B-shaped MoE layer", "qwen235b": "Qwen3-235B-A22B-shaped MoE layer",
             "qwen235b-zipf": "Qwen3-235B-A22B-shaped MoE layer (Zipf routing)",
             "dsv3": "DeepSeek-V3-shaped routed-expert layer",
             "dsv3-grouped": "DeepSeek-V3-shaped routed-expert layer with group-limited routing",
             "mixtral-e2": "Mixtral-8x7B-shaped experts (2 of them) MoE layer",
             "dsv3-proxy": "DeepSeek-V3-width experts (64 of them, d=2048) MoE layer"}
    return names.get(cfg.name, cfg.name) + " fwd+bwd"


def l2_note(cfg) -> str:
    weights = 3 * cfg.E * cfg.d * cfg.f * 2
    if weights > 129e6:
        return f"inputs larger than L2 (expert weights alone {weights / 1e9:.2f} GB > 129 MB)"
    return "inputs smaller than L2 (a small case: not a bandwidth measurement)"


def config_json(cfg, prec="bf16", weights_cached=False):
    bias = {"normal": f"N(0,{cfg.bias_param})", "zipf": f"Zipf(s={cfg.bias_param})", "zero": "0"}[cfg.bias]
    return {"workload": workload_name(cfg), "T": cfg.T, "d": cfg.d, "f": cfg.f, "E": cfg.E, "k": cfg.k,
            "f_shared": cfg.f_shared, "routing": f"{cfg.score} top-{cfg.k}, router bias {bias}" +
            (f", group-limited ({cfg.topk_group} of {cfg.n_group} groups), routed scale {cfg.routed_scale}, "
             f"selection bias N(0,{cfg.sel_bias_std})" if cfg.n_group else ""),
            "precision": prec, "l2": l2_note(cfg),
            "parallelism": "replicas"} | ({"weights": "MXFP8 weights quantised once per optimiser step, "
                                                   "before the timed micro-batches"} if weights_cached else {})


# The files that define each precision's dominant GEMM kernel and its launch (tile
# shape, schedule, tensor maps): recorded DRAM traffic stays valid while they are
# unchanged.
KERNEL_SOURCES = {
    "bf16": ("common.cuh", "gemm.cuh", "gemm2.cuh", "gemm_pair.cu", "kernels.h", "api.cu"),
    "mxfp8": ("common.cuh", "gemm.cuh", "gemm2.cuh", "gemm_mx.cuh", "gemm_mx.cu", "gemm_mx2.cuh",
              "gemm_mx_pair.cu", "kernels.h", "api_mx.cu"),
    "mxfp8-w4": ("common.cuh", "gemm.cuh", "gemm2.cuh", "gemm_mx.cuh", "gemm_mx.cu", "gemm_mx2.cuh",
                 "gemm_mx_pair.cu", "kernels.h", "api_mx.cu", "api.cu"),
}


def source_hash(prec: str) -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "dropless_mixture_experts_warp_gb300", "csrc")
    for name in KERNEL_SOURCES[prec]:
        h.update(name.encode())
        h.update(open(os.path.join(csrc, name), "rb").read())
    return h.hexdigest()[:16]


def read_traffic(kernel_key: str):
    """DRAM bytes per launch recorded from an ncu capture, if the kernel's sources have not
    changed since.  kernel_key is "<precision>:<config>:<gemm>"."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    cur = source_hash(kernel_key.split(":")[0])
    for line in open(path):
        parts = line.split()
        if len(parts) >= 3 and not line.startswith("#") and parts[0] == kernel_key and parts[2] == cur:
            return float(parts[1])
    return None


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        return json.load(open(path)), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ---------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of this GPU's clocks and throttle reasons every 25 ms; stop()
    keeps the samples whose timestamps fall inside the timed window [t0, t1] (host
    wall-clock seconds) and reports their median SM clock and every reason seen (the
    power column, an average over a longer window, is not reported)."""
    FIELDS = ("timestamp,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, uuid: str):
        self.uuid = uuid.lower().replace("gpu-", "")
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "25"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self, t0=None, t1=None):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        return self.summarise(out, self.uuid, t0, t1)

    @classmethod
    def summarise(cls, out: str, uuid: str, t0=None, t1=None):
        import datetime
        rows = [[f.strip() for f in r.split(",")] for r in out.strip().splitlines() if r.count(",") >= 8]
        mine = [r for r in rows if uuid and uuid in r[1].lower()] or rows

        def when(r):
            try:
                return datetime.datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                return None
        inside = [r for r in mine if t0 is not None and when(r) is not None and t0 <= when(r) <= t1]
        use = inside or mine
        if not use:
            return None
        num = lambda v: float(v) if v.replace(".", "", 1).isdigit() else None  # noqa: E731
        sm = [num(r[2]) for r in use if num(r[2]) is not None]
        smax = [num(r[3]) for r in use if num(r[3]) is not None]
        reasons = sorted({cls.REASONS[i] for r in use for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(use), "in_timed_window": bool(inside)}


# ---------------------------------------------------------------------------- CPU oracle timing

ORACLE_POOL = 8   # distinct expert weight sets the CPU legs hold (timing only; see ExpertPool)


class ExpertPool:
    """Expert weights for the CPU oracle legs, fp32, ``[e]`` -> expert e's matrix.

    The timed CPU oracle runs on a bounded token sample, and its cost per expert does not
    depend on the weights' values; holding all E experts on the host (45 GB in fp32 for
    the DeepSeek-V3 shape, minutes to draw) would only slow the measurement.  So ORACLE_POOL
    experts are materialised once, before any timing, and expert e reads pool entry
    e % ORACLE_POOL.  The results are discarded: these legs measure time, not values."""

    def __init__(self, make, E: int, shape):
        self.pool = [make(p) for p in range(min(E, ORACLE_POOL))]
        self.shape = (E,) + tuple(shape)

    def __getitem__(self, e):
        return self.pool[int(e) % len(self.pool)]

    def __len__(self):
        return self.shape[0]


def weight_cached_wmatmul(fp4=False):
    """The MXFP8 oracle's weight product (mx.mx_matmul) with each weight operand's
    quantisation done once and kept: the layer quantises its weights once per step, not
    once per token chunk, so the timed chunks must not pay it again and again.  Keyed by
    the operand's memory and strides (a weight and its transpose are blocked along
    different axes)."""
    import numpy as np
    from oracle import mx
    cache = {}

    def wmatmul(a, b, dtype=np.float64):
        key = (b.__array_interface__["data"][0], b.strides, b.shape, np.dtype(dtype).str)
        q = cache.get(key)
        if q is None:
            q = cache[key] = (mx.qdq4(b) if fp4 else mx.qdq(b)).astype(dtype)
        return mx.qdq(a).astype(dtype) @ q.T
    return wmatmul


def weight_quant_seconds(w_gu, w_d, w_gu_s=None, w_d_s=None, fp4=False) -> float:
    """Host time of one full step's MXFP8 weight quantisation by the oracle's qdq: every
    routed expert's W_gu and W_d in both of their contraction orientations (timed on one
    pool expert, times E) plus the shared expert's."""
    from oracle import mx
    qdq = mx.qdq4 if fp4 else mx.qdq
    t0 = time.perf_counter()
    for m in (w_gu[0], w_d[0]):
        qdq(m)
        qdq(m.T)
    t = (time.perf_counter() - t0) * len(w_gu)
    if w_gu_s is not None:
        t0 = time.perf_counter()
        for m in (w_gu_s, w_d_s):
            qdq(m)
            qdq(m.T)
        t += time.perf_counter() - t0
    return t


def sample_flops(cfg, tokens: int) -> float:
    """Algorithmic FLOPs of the layer step restricted to `tokens` tokens (shared expert included)."""
    return 18.0 * tokens * (cfg.k * cfg.d * cfg.f + cfg.d * cfg.f_shared)


def prequantise_pool(cfg, w_gu, w_d, shared, wmatmul):
    """Fill weight_cached_wmatmul's cache for every pool expert (and the shared expert), in
    all four weight orientations, by one single-expert layer pass each; untimed."""
    import numpy as np
    from oracle import mx
    kw = {"wmatmul": wmatmul}
    if shared is not None:
        kw.update(w_gu_s=shared[0], w_d_s=shared[1])
    x = np.ones((1, cfg.d), np.float32)
    for e in range(min(len(w_gu), ORACLE_POOL)):
        lg = np.full((1, len(w_gu)), -1e4, np.float32)
        lg[0, e] = 1.0
        fwd = mx.moe_forward_mx(x, lg, w_gu, w_d, 1, cfg.score, dtype=np.float32, **kw)
        mx.moe_backward_mx(x, lg, w_gu, w_d, x, fwd, 1, cfg.score, dtype=np.float32, **kw)


def oracle_sample_rate(cfg, x_bits, logits, dy_bits, w_gu, w_d, seconds: float, chunk: int, seed=0,
                       prec="bf16", shared=None, wmatmul=None, wq_seconds=0.0):
    """Run the CPU oracle (fp32) on random token chunks for about `seconds` (at least one
    chunk); returns (FLOP/s, tokens, seconds).  MXFP8: `wmatmul` holds the weights
    quantised once (weight_cached_wmatmul, filled by prequantise_pool) and each chunk is
    charged its token share of one full step's weight quantisation, `wq_seconds`."""
    import numpy as np
    from oracle import moe_oracle as om
    from oracle import mx
    from dropless_mixture_experts_warp_gb300 import synth
    mx8 = prec in MX_PRECS
    fwd_fn, bwd_fn = (mx.moe_forward_mx, mx.moe_backward_mx) if mx8 else (om.moe_forward, om.moe_backward)
    kw = {"wmatmul": wmatmul} if mx8 and wmatmul is not None else {}
    if shared is not None:
        kw.update(w_gu_s=shared[0], w_d_s=shared[1])
    gr = synth.grouped_options(cfg)
    rng = np.random.default_rng(seed)
    done_tok, t_total = 0, 0.0
    while t_total < seconds or done_tok == 0:
        sub = np.sort(rng.choice(x_bits.shape[0], size=chunk, replace=False))
        x = synth.bf16_to_f32(x_bits[sub])
        dy = synth.bf16_to_f32(dy_bits[sub])
        lg = logits[sub]
        t0 = time.perf_counter()
        fwd = fwd_fn(x, lg, w_gu, w_d, cfg.k, cfg.score, dtype=np.float32, grouped=gr, **kw)
        bwd_fn(x, lg, w_gu, w_d, dy, fwd, cfg.k, cfg.score, dtype=np.float32, grouped=gr, **kw)
        t_total += time.perf_counter() - t0 + wq_seconds * chunk / cfg.T
        done_tok += chunk
    return sample_flops(cfg, done_tok) / t_total, done_tok, t_total


def oracle_setup(cfg, prec, w_gu, w_d, shared):
    """(wmatmul, wq_seconds) for oracle_sample_rate: MXFP8 weights quantised once, untimed,
    and the host time of one full step's weight quantisation; (None, 0) for bf16."""
    if prec not in MX_PRECS:
        return None, 0.0
    wq_s = weight_quant_seconds(w_gu, w_d, *(shared or ()), fp4=prec == "mxfp8-w4")
    wm = weight_cached_wmatmul(fp4=prec == "mxfp8-w4")
    prequantise_pool(cfg, w_gu, w_d, shared, wm)
    return wm, wq_s


def oracle_chunk(args) -> int:
    """Tokens per oracle sample: the MXFP8 oracle quantises every activation operand of a
    sample in fp64-exact NumPy, several times the bf16 oracle's cost per token."""
    return max(1, args.ref_tokens if args.prec == "bf16" else args.ref_tokens // 8)


def sample_note(cfg, prec, ntok, secs, wq_seconds) -> str:
    note = (f"{ntok} random tokens of the {cfg.T}-token batch, fp32 NumPy, {secs:.1f} s; expert weights: "
            f"{min(cfg.E, ORACLE_POOL)} distinct sets reused cyclically over the {cfg.E} experts (timing only)")
    if cfg.f_shared:
        note += "; the shared expert runs and is counted"
    if prec in MX_PRECS:
        note += (f"; weights quantised once, each sample charged its token share of one full step's weight "
                 f"quantisation ({wq_seconds:.1f} s on the host)")
    return note


def run_reference(args, cfg):
    """--impl reference: the CPU oracle, timed per step on a bounded token sample."""
    from dropless_mixture_experts_warp_gb300 import synth
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    inp = synth.token_inputs(cfg)
    f32 = lambda bits: synth.bf16_to_f32(bits).reshape(bits.shape)  # noqa: E731
    w_gu = ExpertPool(lambda e: f32(synth.expert_weights(cfg, e)[0]), cfg.E, (2 * cfg.f, cfg.d))
    w_d = ExpertPool(lambda e: f32(synth.expert_weights(cfg, e)[1]), cfg.E, (cfg.d, cfg.f))
    shared = tuple(f32(w) for w in synth.shared_weights(cfg)) if cfg.f_shared else None
    wm, wq_s = oracle_setup(cfg, args.prec, w_gu, w_d, shared)
    chunk = oracle_chunk(args)
    run = lambda seed: oracle_sample_rate(cfg, inp["x"], inp["logits"], inp["dy"], w_gu, w_d, 0.0, chunk,  # noqa
                                          seed=seed, prec=args.prec, shared=shared, wmatmul=wm, wq_seconds=wq_s)
    for i in range(args.warmup):
        run(1000 + i)
    times, tok = [], 0
    for s in range(args.steps):
        _, n, t = run(s + 1)
        times.append(t)
        tok += n
    total = sum(times)
    value = sample_flops(cfg, tok) / total / 1e12
    ms = total / args.steps * 1e3
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": config_json(cfg, f"{args.prec} (fp32 oracle)"),
            "tokens_per_s": tok / total,
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                             "sample": sample_note(cfg, args.prec, chunk, total / args.steps, wq_s) +
                             f"; {chunk} tokens per step",
                             "extrapolated_full_step_s": cfg.flops_fwd_bwd() / (value * 1e12)},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------- replicas

def reduce_max(values, dist, device):
    """Elementwise maximum of per-rank values over all ranks: with N replicas the
    slowest one sets the job's time.  Identity without a process group."""
    if dist is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_rate(world, flops_per_replica, ms):
    """Whole-job throughput in TFLOP/s: every replica's FLOPs over the slowest step time."""
    return world * flops_per_replica / (ms * 1e-3) / 1e12


def _mlp_bytes(N, d, w, G, mx8, quantise_weights, w4=False):
    """Algorithmic bytes of the six GEMMs of N rows through G experts of width w (each
    kernel reads its operands once and writes its results once); w4: MXFP4 weights."""
    q = 1.0 + 1.0 / 32                  # an MXFP8 element with its share of a block scale
    a = q if mx8 else 2.0               # a GEMM operand element (activation)
    qw = (0.5 + 1.0 / 32) if w4 else a  # a weight element as the GEMMs read it
    wgu, wd = 2.0 * w * d * G, 1.0 * d * w * G
    h_out = 2.0 * N * w * q if mx8 else N * w * 2.0        # h: both code orientations in MXFP8
    dgu_out = 2.0 * N * 2 * w * q if mx8 else N * 2 * w * 2.0
    b = 0.0
    if mx8 and quantise_weights:        # both weights, read once, both orientations written
        b += (wgu + wd) * 2.0 + 2.0 * (wgu + wd) * qw
    b += N * d * a + wgu * qw + N * 2 * w * 2.0 + h_out     # gate/up + SwiGLU: G|U saved in bf16
    b += N * w * a + wd * qw + N * d * 2.0                  # down
    b += N * d * a + wd * qw + N * 2 * w * 2.0 + dgu_out    # down dgrad + SwiGLU'
    b += N * d * a + N * w * a + wd * 2.0                   # down wgrad
    b += N * 2 * w * a + wgu * qw + N * d * 2.0             # gate/up dgrad
    b += N * 2 * w * a + N * d * a + wgu * 2.0              # gate/up wgrad
    return b


def step_bytes(cfg, prec="bf16", weights_cached=False) -> float:
    """Algorithmic HBM bytes of one layer step (forward and backward): every kernel reads
    its inputs once and writes its outputs once; x and dY count once although a token's
    k routed rows are gathered from them.  Index maps, routing weights and dw partials
    (well under 1 %) are left out."""
    T, d, f, E, k, fs = cfg.T, cfg.d, cfg.f, cfg.E, cfg.k, cfg.f_shared
    R = T * k
    mx8 = prec in MX_PRECS
    w4 = prec == "mxfp8-w4"
    q = 1.0 + 1.0 / 32
    b = T * E * 4.0 + T * k * 8.0                           # route
    b += T * d * 2.0 + (2.0 * R * d * q if mx8 else R * d * 2.0)   # dispatch of x
    b += _mlp_bytes(R, d, f, E, mx8, not weights_cached, w4)
    b += R * d * 2.0 + T * d * 2.0                          # combine
    b += T * d * 2.0 + (2.0 * R * d * q if mx8 else R * d * 2.0)   # combine backward (dY rows)
    b += R * d * 2.0 + T * d * 2.0                          # un-permute (dX)
    b += T * E * 4.0 * 2 + T * k * 12.0                     # router backward
    if fs:
        if mx8:                                             # x and dY quantised for the shared GEMMs
            b += 2 * (T * d * 2.0 + 2.0 * T * d * q)
        b += _mlp_bytes(T, d, fs, 1, mx8, not weights_cached, w4)
        b += 2 * T * d * 2.0                                # its output read by combine, its dX by un-permute
    return b


def step_bound(cfg, prec, weights_cached, ms, peak_tflops, hbm_gbs):
    """The step's combined roofline: max(FLOPs / tensor peak, bytes / HBM bandwidth)."""
    flop_ms = cfg.flops_fwd_bwd() / (peak_tflops * 1e12) * 1e3
    nbytes = step_bytes(cfg, prec, weights_cached)
    byte_ms = nbytes / (hbm_gbs * 1e9) * 1e3
    bound_ms = max(flop_ms, byte_ms)
    return {"bound": "tensor" if flop_ms >= byte_ms else "hbm", "flop_ms": flop_ms, "byte_ms": byte_ms,
            "bytes": nbytes, "bound_ms": bound_ms, "frac": bound_ms / ms}


# ---------------------------------------------------------------------------- native

# event windows of a step: mark 0 after permute, 1 after gate_up, 2 after down, 3 after
# combine_bwd, 4..7 after each backward GEMM call
GEMM_WINDOWS = {"gate_up": (0, 1), "down": (1, 2), "down_dgrad": (3, 4), "down_wgrad": (4, 5),
                "gate_up_dgrad": (5, 6), "gate_up_wgrad": (6, 7)}


class Ctx:
    """What every measured step shares: the device, the stream, the inputs, the replicas."""

    def __init__(self, cfg, dev, stream, inp, world, dist):
        self.cfg, self.dev, self.stream, self.inp, self.world, self.dist = cfg, dev, stream, inp, world, dist


def make_step(ctx, bufs, dims, prec, weights_cached):
    """The library calls of one layer step on ctx.stream; step(ev, io) records the GEMM
    event marks in ev (if given) and runs on the io tensors (x, logits, dy, y, dx, d_logits;
    default: the base inputs and bufs' outputs)."""
    import torch
    from dropless_mixture_experts_warp_gb300 import binding as B, synth
    cfg, stream, inp = ctx.cfg, ctx.stream, ctx.inp
    mx8 = prec in MX_PRECS
    w_gu, w_d = inp["w_gu"], inp["w_d"]
    grouped = synth.grouped_options(cfg)
    sel_bias = torch.from_numpy(grouped["bias"]).to(ctx.dev) if grouped is not None else None
    base_io = (inp["x"], inp["logits"], inp["dy"], bufs.y, bufs.dx, bufs.d_logits)

    def step(ev=None, io=None):
        b, dm = bufs, dims
        x, logits, dy, y_out, dx_out, dl_out = io if io is not None else base_io

        def mark(i):
            if ev is not None:
                ev[i].record(stream)
        if grouped is not None:
            B.moe_route_topk_grouped(dm, logits, sel_bias, grouped["n_group"], grouped["topk_group"],
                                     grouped["routed_scale"], b.topk_idx, b.topk_w, b.split_sizes, b.offsets,
                                     b.row_offsets, b.workspace, b.status, stream)
        else:
            B.moe_route_topk(dm, logits, b.topk_idx, b.topk_w, b.split_sizes, b.offsets, b.row_offsets,
                             b.workspace, b.status, stream)
        if mx8:
            # the 16-bit master weights are quantised every step (unless they are cached for
            # the optimiser step's micro-batches); x is quantised in the dispatch
            if not weights_cached:
                B.moe_mx_quantize_weights(dm, w_gu, w_d, b.wq, stream)
            B.moe_permute_mx(dm, x, b.topk_idx, b.topk_w, b.split_sizes, b.row_offsets, b.workspace, b.mx_ws,
                             b.row_to_token, b.token_to_row, b.w_rows, b.status, stream)
        else:
            B.moe_permute(dm, x, b.topk_idx, b.topk_w, b.split_sizes, b.row_offsets, b.workspace, b.xp,
                          b.row_to_token, b.token_to_row, b.w_rows, b.status, stream)
        mark(0)
        if mx8:
            B.moe_gemm_gate_up_mx(dm, b.row_offsets, b.w_rows, b.wq, b.mx_ws, b.gu, b.status, stream)
        else:
            B.moe_gemm_gate_up(dm, b.xp, b.row_offsets, b.w_rows, w_gu, b.gu, b.h, b.status, stream)
        mark(1)
        if mx8:
            B.moe_gemm_down_mx(dm, b.row_offsets, b.wq, b.mx_ws, b.y_rows, b.status, stream)
        else:
            B.moe_gemm_down(dm, b.h, b.row_offsets, w_d, b.y_rows, b.status, stream)
        mark(2)
        if cfg.f_shared and mx8:
            if not weights_cached:
                B.moe_mx_quantize_shared_weights(dm, inp["w_gu_s"], inp["w_d_s"], b.wq_s, stream)
            B.moe_shared_mlp_fwd_mx(dm, x, b.wq_s, b.mx_ws_s, b.gu_s, b.y_s, b.status, stream)
        elif cfg.f_shared:
            B.moe_shared_mlp_fwd(dm, x, inp["w_gu_s"], inp["w_d_s"], b.gu_s, b.h_s, b.y_s, b.status, stream)
        B.moe_combine_fwd(dm, b.y_rows, b.token_to_row, b.y_s, y_out, stream)
        if mx8:
            B.moe_combine_bwd_mx(dm, dy, b.row_to_token, b.split_sizes, b.row_offsets, b.mx_ws, stream)
        else:
            B.moe_combine_bwd(dm, dy, b.token_to_row, b.split_sizes, b.row_offsets, b.dy_rows, stream)
        mark(3)
        if mx8:
            B.moe_gemm_down_dgrad_mx(dm, b.row_offsets, b.w_rows, b.wq, b.mx_ws, b.gu, b.dw_rows, b.workspace,
                                     b.status, stream)
            mark(4)
            B.moe_gemm_down_wgrad_mx(dm, b.row_offsets, b.mx_ws, b.dw_d, b.status, stream)
            mark(5)
            B.moe_gemm_gate_up_dgrad_mx(dm, b.row_offsets, b.wq, b.mx_ws, b.dxp, b.status, stream)
            mark(6)
            B.moe_gemm_gate_up_wgrad_mx(dm, b.row_offsets, b.mx_ws, b.dw_gu, b.status, stream)
        else:
            B.moe_gemm_down_dgrad(dm, b.dy_rows, b.row_offsets, b.w_rows, w_d, b.gu, b.dgu, b.dw_rows,
                                  b.workspace, b.status, stream)
            mark(4)
            B.moe_gemm_down_wgrad(dm, b.dy_rows, b.h, b.row_offsets, b.dw_d, b.status, stream)
            mark(5)
            B.moe_gemm_gate_up_dgrad(dm, b.dgu, b.row_offsets, w_gu, b.dxp, b.status, stream)
            mark(6)
            B.moe_gemm_gate_up_wgrad(dm, b.dgu, b.xp, b.row_offsets, b.dw_gu, b.status, stream)
        mark(7)
        if cfg.f_shared and mx8:
            B.moe_shared_mlp_bwd_mx(dm, b.wq_s, b.mx_ws_s, b.gu_s, dy, b.dx_s, b.dw_gu_s, b.dw_d_s, b.status,
                                    stream)
        elif cfg.f_shared:
            B.moe_shared_mlp_bwd(dm, x, inp["w_gu_s"], inp["w_d_s"], b.gu_s, b.h_s, dy, b.dgu_s, b.dx_s,
                                 b.dw_gu_s, b.dw_d_s, b.status, stream)
        B.moe_combine_fwd(dm, b.dxp, b.token_to_row, b.dx_s, dx_out, stream)
        if grouped is not None:
            B.moe_route_topk_bwd_scaled(dm, logits, b.topk_idx, b.topk_w, grouped["routed_scale"], b.dw_rows,
                                        b.token_to_row, dl_out, stream)
        else:
            B.moe_route_topk_bwd(dm, logits, b.topk_idx, b.topk_w, b.dw_rows, b.token_to_row, dl_out, stream)

    return step, base_io


def time_e2e(ctx, step, bufs, base_io, steps):
    """End to end through the same calls with host buffers: every step's inputs (x, logits,
    dY) come from pinned host memory and its results (Y, dX, d_logits) go back to pinned
    host memory inside the timed region.  As an input pipeline does, a copy stream moves
    step s + 1's inputs in and step s's results out while the compute stream runs the
    neighbouring step; the step's device inputs and results are double-buffered.  Times
    the same number of steps as the device-timed region.  Returns (ms per step, h2d bytes,
    d2h bytes)."""
    import torch
    dev, stream, dist = ctx.dev, ctx.stream, ctx.dist
    x, logits, dy = base_io[:3]
    x_h = torch.empty(x.shape, dtype=x.dtype, pin_memory=True).copy_(x)
    lg_h = torch.empty(logits.shape, dtype=logits.dtype, pin_memory=True).copy_(logits)
    dy_h = torch.empty(dy.shape, dtype=dy.dtype, pin_memory=True).copy_(dy)
    outs = (bufs.y, bufs.dx, bufs.d_logits)
    host_out = [tuple(torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs) for _ in range(2)]
    dev_io = [base_io, tuple(torch.empty_like(t) for t in base_io)]
    h2d = x_h.nbytes + lg_h.nbytes + dy_h.nbytes
    d2h = sum(t.nbytes for t in host_out[0])
    e2e_steps = max(2, steps)
    copy = torch.cuda.Stream(dev)
    in_ready = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    out_free = [torch.cuda.Event() for _ in range(2)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def to_device(i):
        with torch.cuda.stream(copy):
            for d, h in zip(dev_io[i][:3], (x_h, lg_h, dy_h)):
                d.copy_(h, non_blocking=True)
            in_ready[i].record(copy)

    def to_host(i):
        with torch.cuda.stream(copy):
            copy.wait_event(done[i])
            for h, d in zip(host_out[i], dev_io[i][3:]):
                h.copy_(d, non_blocking=True)
            out_free[i].record(copy)

    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    start.record(stream)
    copy.wait_stream(stream)
    to_device(0)
    for s in range(e2e_steps):
        i = s % 2
        if s + 1 < e2e_steps:
            if s >= 1:
                copy.wait_event(done[1 - i])  # step s - 1 has finished with buffer 1 - i
            to_device(1 - i)
        stream.wait_event(in_ready[i])
        if s >= 2:
            stream.wait_event(out_free[i])  # step s - 2's results have left buffer i
        with torch.cuda.stream(stream):
            step(io=dev_io[i])
        done[i].record(stream)
        to_host(i)
    stream.wait_event(out_free[0])
    stream.wait_event(out_free[1])
    end.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = reduce_max([start.elapsed_time(end) / e2e_steps], dist, dev)[0]
    for h, d in zip(host_out[(e2e_steps - 1) % 2], outs):  # the last step's results reached the host
        if not torch.equal(h.to(dev), d):
            raise RuntimeError("end-to-end results differ from the device-timed step's")
    return e2e_ms, h2d, d2h


def measure(ctx, args, prec, weights_cached):
    """Warm-up, K device-timed steps (CUDA events on the launching stream, barrier and
    synchronize on both sides, max over ranks, clocks sampled meanwhile), then K end-to-end
    steps.  Returns the part of the JSON line that belongs to this precision."""
    import torch
    from dropless_mixture_experts_warp_gb300 import binding as B, layer
    cfg, dev, stream, dist, world = ctx.cfg, ctx.dev, ctx.stream, ctx.dist, ctx.world
    mx8 = prec in MX_PRECS
    dims = layer.dims_of(cfg.T, cfg.d, cfg.f, cfg.E, cfg.k, cfg.f_shared, cfg.score, prec)
    bufs = layer.allocate(dims, dev)
    torch.cuda.synchronize(dev)
    step, base_io = make_step(ctx, bufs, dims, prec, weights_cached)
    if weights_cached:
        # once per optimiser step, outside the timed micro-batches
        with torch.cuda.stream(stream):
            layer.quantize_weights(bufs, ctx.inp["w_gu"], ctx.inp["w_d"], stream, ctx.inp.get("w_gu_s"),
                                   ctx.inp.get("w_d_s"))
    for _ in range(args.warmup):
        step()
    layer.check(bufs, stream)

    uuid = ""
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(8)] for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    launches0 = B.moe_launch_count()
    sampler.start()
    time.sleep(0.3)
    t0 = time.time()
    start.record(stream)
    for s in range(args.steps):
        step(evs[s])
    end.record(stream)
    torch.cuda.synchronize(dev)
    t1 = time.time()
    clocks = sampler.stop(t0, t1)
    launches = B.moe_launch_count() - launches0
    if dist:
        dist.barrier()
    layer.check(bufs, stream)
    ms = reduce_max([start.elapsed_time(end) / args.steps], dist, dev)[0]
    gemm_ms = {g: statistics.mean(evs[s][a].elapsed_time(evs[s][b]) for s in range(args.steps))
               for g, (a, b) in GEMM_WINDOWS.items()}

    e2e_ms, h2d, d2h = time_e2e(ctx, step, bufs, base_io, args.steps)
    layer.check(bufs, stream)
    del bufs, step, base_io
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()

    peaks, peak_src = measured_peaks()
    flops = cfg.flops_fwd_bwd()
    unit = cfg.T * cfg.k * cfg.d * cfg.f
    value = job_rate(world, flops, ms)
    dom = max(GEMMS, key=lambda g: gemm_ms[g])
    dom_flops = GEMM_FLOP_FACTOR[dom] * unit
    achieved = dom_flops / (gemm_ms[dom] * 1e-3) / 1e12
    # the burst figure: the timed region is well under the seconds-long loop behind the
    # sustained one.  MXFP8 has no measured peak: bf16's measured burst figure times the
    # nominal 2x ratio of the dense MXFP8 and bf16 tensor rates
    peak = peaks["bf16_tflops"] * (2.0 if mx8 else 1.0)
    src = (f"{peak_src} bf16_tflops (burst) x 2, the nominal MXFP8/bf16 ratio (FP8 x FP4 runs the same "
           f"MMA kind at the same rate)" if prec == "mxfp8-w4" else
           f"{peak_src} bf16_tflops (burst) x 2, the nominal MXFP8/bf16 ratio" if mx8 else
           f"{peak_src} bf16_tflops (burst: the timed region lasts {args.steps * ms / 1e3:.2f} s)")
    return {
        "value": value, "ms_per_step": ms, "tokens_per_s": world * cfg.T / (ms * 1e-3),
        "dtype": ("e4m3 x e2m1, e8m0 scales (MXFP8 x MXFP4), fp32 acc" if prec == "mxfp8-w4" else
                  "e4m3+e8m0 (MXFP8), fp32 acc" if mx8 else "bf16"),
        "precision": prec,
        "frac_of_peak": value / world / peak,
        "roofline": {"bound": "tensor", "kernel": f"{dom} ({(GEMM_KERNEL_MX if mx8 else GEMM_KERNEL)[dom]})",
                     "achieved": achieved, "peak": peak, "unit": UNIT, "frac": achieved / peak,
                     "traffic": read_traffic(f"{prec}:{cfg.name}:{dom}"), "peak_source": src,
                     "flops_per_launch": dom_flops, "ms_per_launch": gemm_ms[dom]},
        "gemm_ms": {g: round(v, 4) for g, v in gemm_ms.items()},
        "gemm_tflops": {g: GEMM_FLOP_FACTOR[g] * unit / (gemm_ms[g] * 1e-3) / 1e12 for g in GEMMS},
        "e2e": {"value": job_rate(world, flops, e2e_ms), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "steps": max(2, args.steps)},
        "gpu_launches": launches,
        "clocks": clocks,
        "step_bound": step_bound(cfg, prec, weights_cached, ms, peak, peaks["hbm_gbs"]),
        "weights_cached": weights_cached,
    }


def run_native(args, cfg):
    import numpy as np
    import torch
    from dropless_mixture_experts_warp_gb300 import binding as B, build, synth

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    if rank == 0 or world == 1:
        build.build()
    if dist:
        dist.barrier()
    B.lib()

    dev = torch.device("cuda", local)
    inp = synth.torch_inputs(cfg, dev, seed=cfg.seed + 7919 * rank)
    # one explicit stream carries every library call, copy and timing event
    ctx = Ctx(cfg, dev, torch.cuda.Stream(dev), inp, world, dist)
    head = measure(ctx, args, args.prec, args.weights_cached)
    second, second_skip = None, None
    if args.second_prec != "none" and args.second_prec != args.prec:
        dims2 = B.make_dims(cfg.T, cfg.d, cfg.f, cfg.E, cfg.k, cfg.f_shared, cfg.score, args.second_prec)
        st = B.moe_check_dims(dims2)
        if st == B.MOE_OK:
            second = measure(ctx, args, args.second_prec, False)
        else:
            second_skip = f"not measured: this shape is outside the {args.second_prec} path's limits " \
                          f"({B.STATUS_NAMES.get(st, st)})"

    line = {"metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": head["dtype"], "data": "synthetic",
            "config": config_json(cfg, args.prec, args.weights_cached)}
    line.update({k: v for k, v in head.items() if k not in ("value", "ms_per_step", "dtype", "precision",
                                                            "weights_cached")})
    if second is not None:
        line[second["precision"]] = {k: v for k, v in second.items() if k != "precision"} | {
            "config": config_json(cfg, second["precision"], False)}
    elif second_skip:
        line[args.second_prec] = {"skipped": second_skip}

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # the oracle as it stands, on this host's cores, on a bounded random token sample
        ex = {"x": inp["x"].view(torch.int16).cpu().numpy().view(np.uint16),
              "dy": inp["dy"].view(torch.int16).cpu().numpy().view(np.uint16), "logits": inp["logits"].cpu().numpy()}
        w_gu = ExpertPool(lambda e: inp["w_gu"][e].float().cpu().numpy(), cfg.E, (2 * cfg.f, cfg.d))
        w_d = ExpertPool(lambda e: inp["w_d"][e].float().cpu().numpy(), cfg.E, (cfg.d, cfg.f))
        shared = (inp["w_gu_s"].float().cpu().numpy(), inp["w_d_s"].float().cpu().numpy()) if cfg.f_shared else None
        wm, wq_s = oracle_setup(cfg, args.prec, w_gu, w_d, shared)
        rate, ntok, secs = oracle_sample_rate(cfg, ex["x"], ex["logits"], ex["dy"], w_gu, w_d, args.cpu_seconds,
                                              oracle_chunk(args), prec=args.prec, shared=shared, wmatmul=wm,
                                              wq_seconds=wq_s)
        line["cpu_baseline"] = {"value": rate / 1e12, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                                "precision": args.prec,
                                "sample": sample_note(cfg, args.prec, ntok, secs, wq_s),
                                "extrapolated_full_step_s": cfg.flops_fwd_bwd() / rate}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--config", default="dsv3")
    ap.add_argument("--prec", default="bf16", choices=["bf16", "mxfp8", "mxfp8-w4"],
                    help="mxfp8-w4: FP8 x FP4 experts (MXFP8 activations, MXFP4 weights)")
    ap.add_argument("--second-prec", default="mxfp8", choices=["bf16", "mxfp8", "mxfp8-w4", "none"],
                    help="also measure the same workload in this precision and report it in the same line "
                         "under its name (per-step weight quantisation); 'none' or the headline's own "
                         "precision skips it")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-tokens", type=int, default=32)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--weights-cached", action="store_true",
                    help="MXFP8: quantise the weights once before timing (one optimiser step shared by "
                         "micro-batches) instead of in every timed step")
    args = ap.parse_args()
    if args.weights_cached and args.prec not in MX_PRECS:
        ap.error("--weights-cached applies to --prec mxfp8")
    from dropless_mixture_experts_warp_gb300 import synth
    cfg = synth.CONFIGS[args.config]
    if args.impl == "reference":
        return run_reference(args, cfg)
    return run_native(args, cfg)


if __name__ == "__main__":
    sys.exit(main())
