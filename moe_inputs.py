"""Seeded synthetic inputs for the MoE layer workloads.

This module only draws random numbers and casts them to the storage type of a
workload: it holds none of the layer's arithmetic.  Both the CUDA path (via
the tests and the benchmark) and the CPU oracle consume exactly what it
returns, so neither side derives its inputs from the other.

Every tensor has its own generator stream, seeded from ``(seed, stream id)``,
so a tensor can be re-drawn alone.  Draws are made in fp32 with
``torch.randn`` on the requested device and rounded to bf16 with
round-to-nearest-even (``Tensor.to``) where the workload is bf16.  Draws on
different devices give different (but individually reproducible) values; a
test always hands the oracle host copies of the very tensors the GPU sees.

Workloads (shapes and distributions of the layer; names say what they are):

=====================  ======  ====  ====  ===  =  =========================
name                   T       D     H     E    k  router / notes
=====================  ======  ====  ====  ===  =  =========================
tiny-fp32              256     128   256   8    2  softmax, no renorm, fp32;
                                                   also tp=2 H-shards
fine-grained-bf16      4096    2048  1408  64   6  softmax renormalised over k
deepseek-v3-shaped     8192    7168  2048  256  8  sigmoid renormalised, w std
                                                   0.006 (22.5 GB of experts)
zipf-skewed            16384   4096  1536  64   8  softmax renormalised; per-
                                                   expert router bias so loads
                                                   follow Zipf(1.2); 4 experts
                                                   forced empty
decode-masked          128     7168  2048  256  8  sigmoid renormalised, masked
                                                   per-expert layout; also 8
                                                   expert ranges x 4 H-shards
=====================  ======  ====  ====  ===  =  =========================

x ~ N(0, 1); W_g, w1, w3, w2 ~ N(0, std) with std 0.02 unless stated.
"""
from __future__ import annotations

from dataclasses import dataclass, replace
from typing import Optional

import numpy as np
import torch

STREAM_X, STREAM_WG, STREAM_BIAS, STREAM_W1, STREAM_W3, STREAM_W2, STREAM_AUX = range(7)


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    D: int
    H: int
    E: int
    k: int
    dtype: str            # "f32" or "bf16"
    score: str            # "softmax" or "sigmoid"
    renorm: bool
    wstd: float = 0.02
    layout: str = "contiguous"   # or "masked"
    zipf_s: Optional[float] = None
    zipf_c: float = 2.0          # bias scale: b_e = c * ln(p_e)
    zipf_empty: int = 4          # lowest-ranked experts pushed to zero load
    tp: int = 1                  # H-shards used by the shard-equivalence check
    ep: int = 1                  # expert ranges used by the shard check
    n_group: int = 0             # > 1: group-limited routing over n_group groups
    topk_group: int = 0          # groups a token may use

    def scaled(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    "tiny-fp32": Workload("tiny-fp32", 256, 128, 256, 8, 2, "f32", "softmax", False, tp=2),
    "fine-grained-bf16": Workload("fine-grained-bf16", 4096, 2048, 1408, 64, 6, "bf16",
                                  "softmax", True),
    "deepseek-v3-shaped": Workload("deepseek-v3-shaped", 8192, 7168, 2048, 256, 8, "bf16",
                                   "sigmoid", True, wstd=0.006),
    "zipf-skewed": Workload("zipf-skewed", 16384, 4096, 1536, 64, 8, "bf16", "softmax", True,
                            zipf_s=1.2),
    "decode-masked": Workload("decode-masked", 128, 7168, 2048, 256, 8, "bf16", "sigmoid", True,
                              wstd=0.006, layout="masked", ep=8, tp=4),
}
# order in which the workloads are listed by the benchmark specification
WORKLOAD_ORDER = ["tiny-fp32", "fine-grained-bf16", "deepseek-v3-shaped", "zipf-skewed",
                  "decode-masked"]


def torch_dtype(w: Workload) -> torch.dtype:
    return torch.float32 if w.dtype == "f32" else torch.bfloat16


def _gen(device, seed: int, stream: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1_000_003 + stream)
    return g


def _normal(shape, std, g, device, dtype) -> torch.Tensor:
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


@dataclass
class Inputs:
    w: Workload
    x: torch.Tensor                # [T, D]
    wg: torch.Tensor               # [E, D]
    bias: Optional[torch.Tensor]   # [E] fp32 or None
    w1: Optional[torch.Tensor]     # [E, H, D]
    w3: Optional[torch.Tensor]     # [E, H, D]
    w2: Optional[torch.Tensor]     # [E, D, H]


def zipf_bias(w: Workload, device, seed: int) -> torch.Tensor:
    """Router bias giving expert loads roughly Zipf(s): b_e = c ln p_e.

    p_e is proportional to r_e^-s for a seeded permutation r of 1..E; the
    ``zipf_empty`` lowest-ranked experts get an extra -30 so they receive no
    tokens.  (A load exactly Zipf(1.2) is impossible with distinct top-k
    experts: one expert can take at most T of the T*k routed rows.)
    """
    g = _gen("cpu", seed, STREAM_BIAS)
    r = torch.randperm(w.E, generator=g).to(torch.float64) + 1.0
    p = r.pow(-w.zipf_s)
    p = p / p.sum()
    b = w.zipf_c * torch.log(p)
    b[r > w.E - w.zipf_empty] -= 30.0
    return b.to(torch.float32).to(device)


def expert_weights(w: Workload, e: int, device="cpu", seed: int = 0):
    """w1[e], w3[e], w2[e] drawn alone, with the workload's distribution.

    Each expert here has its own generator streams, so any subset of experts
    can be drawn without the others (used where only the experts a token
    sample reaches are needed).  The values are not those make_inputs()
    gives expert e; only the distribution is the same.
    """
    dt = torch_dtype(w)
    out = []
    for sid, shape in ((STREAM_W1, (w.H, w.D)), (STREAM_W3, (w.H, w.D)), (STREAM_W2, (w.D, w.H))):
        g = _gen(device, seed * 4099 + e + 1, 100 + sid)
        out.append(_normal(shape, w.wstd, g, device, dt))
    return tuple(out)


def make_inputs(w: Workload, device="cpu", seed: int = 0, weights: bool = True) -> Inputs:
    dt = torch_dtype(w)
    x = _normal((w.T, w.D), 1.0, _gen(device, seed, STREAM_X), device, dt)
    wg = _normal((w.E, w.D), w.wstd, _gen(device, seed, STREAM_WG), device, dt)
    bias = zipf_bias(w, device, seed) if w.zipf_s else None
    w1 = w3 = w2 = None
    if weights:
        w1 = torch.empty((w.E, w.H, w.D), dtype=dt, device=device)
        w3 = torch.empty((w.E, w.H, w.D), dtype=dt, device=device)
        w2 = torch.empty((w.E, w.D, w.H), dtype=dt, device=device)
        for dst, sid, shape in ((w1, STREAM_W1, (w.H, w.D)), (w3, STREAM_W3, (w.H, w.D)),
                                (w2, STREAM_W2, (w.D, w.H))):
            g = _gen(device, seed, sid)
            for e in range(w.E):   # one expert at a time bounds the fp32 temporary
                dst[e].copy_(_normal(shape, w.wstd, g, device, dt))
    return Inputs(w, x, wg, bias, w1, w3, w2)


def random_topk_idx(T: int, E: int, k: int, seed: int = 0, skew: float = 0.0) -> np.ndarray:
    """Seeded routing table [T,k] of distinct experts per token.

    With ``skew`` > 0 expert e is drawn with weight (e+1)^-skew, which leaves
    some experts empty and makes segment lengths ragged.
    """
    rng = np.random.default_rng(seed)
    p = (np.arange(E) + 1.0) ** (-skew)
    p /= p.sum()
    idx = np.empty((T, k), np.int32)
    for t in range(T):
        idx[t] = rng.choice(E, size=k, replace=False, p=p)
    return idx


def random_weights(T: int, k: int, seed: int = 0) -> np.ndarray:
    rng = np.random.default_rng(seed + 7)
    return rng.uniform(0.05, 1.0, size=(T, k)).astype(np.float32)


def exact_router_inputs(T: int, D: int, E: int, seed: int = 0):
    """x and W_g whose dot products are exact in fp32, whatever the order.

    x holds integers in [-2, 2] and W_g holds multiples of 1/8 in [-1, 1], so
    every logit is a multiple of 1/8 bounded by 2*D; for D <= 2^20 every
    partial sum is exact in fp32 and bf16 stores both inputs exactly.  Small
    integer ranges make many exact ties between experts.
    """
    rng = np.random.default_rng(seed)
    x = rng.integers(-2, 3, size=(T, D)).astype(np.float32)
    wg = (rng.integers(-8, 9, size=(E, D)) / 8.0).astype(np.float32)
    return x, wg


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Host numpy view of a bf16 tensor's bit patterns (uint16)."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def host_array(t: torch.Tensor) -> np.ndarray:
    """Host numpy array in the oracle's conventions (bf16 -> uint16 bits)."""
    if t.dtype == torch.bfloat16:
        return bf16_bits(t)
    return t.detach().cpu().contiguous().numpy()
