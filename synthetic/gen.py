"""Seeded generators for the five gpt-oss-shaped MoE layer workloads.

Every tensor is drawn from one ``numpy.random.Generator(PCG64(seed))`` in a fixed
order, so a (config, seed) pair names one set of inputs on any machine that runs
the same numpy.

Value distributions (gpt-oss-shaped synthetic data; no checkpoint is involved):

* activations ``x``      ~ N(0, 1), rounded to bf16 (round to nearest even);
* router weight ``W_r``  ~ N(0, 0.02^2), rounded to bf16;
* expert weights: MXFP4 -- every 4-bit E2M1 code uniform over 0..15, every E8M0
  scale byte uniform over an integer exponent range (tiny layer: 121..125, i.e.
  2^-6..2^-2; gpt-oss shapes: 120..124, i.e. 2^-7..2^-3);
* prefill workload: a per-expert router bias ``beta * ln p_r`` where ranks ``r``
  come from a seeded permutation and ``p_r`` is Zipf(s = 1.1) over the experts.

Storage layouts (row-major):

* ``x``          uint16 [T, H]        bf16 bit patterns
* ``w_router``   uint16 [E, H]        bf16 bit patterns
* ``router_bias`` float32 [E] or None
* ``gu_codes``   uint8 [E, 2I, H/2]   gate rows 0..I-1, up rows I..2I-1; two
  E2M1 codes per byte, the even K index in the low nibble
* ``gu_scales``  uint8 [E, 2I, H/32]  one E8M0 byte per 32 consecutive K values
* ``dn_codes``   uint8 [E, H, I/2]
* ``dn_scales``  uint8 [E, H, I/32]
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np


def bf16_bits_from_f32(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return the bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclass
class LayerInputs:
    name: str
    T: int
    H: int
    I: int
    E: int
    k: int
    x: np.ndarray
    w_router: np.ndarray
    gu_codes: np.ndarray
    gu_scales: np.ndarray
    dn_codes: np.ndarray
    dn_scales: np.ndarray
    router_bias: Optional[np.ndarray] = None
    meta: dict = field(default_factory=dict)


@dataclass(frozen=True)
class LayerConfig:
    name: str
    T: int
    H: int
    I: int
    E: int
    k: int
    scale_lo: int
    scale_hi: int
    zipf_s: Optional[float] = None
    zipf_beta: float = 1.0
    description: str = ""


CONFIGS = {
    "tiny": LayerConfig(
        "tiny", T=4, H=256, I=256, E=8, k=2, scale_lo=121, scale_hi=125,
        description="tiny MoE layer: T=4, H=I=256, 8 experts, top-2"),
    "gptoss20b_b1": LayerConfig(
        "gptoss20b_b1", T=1, H=2880, I=2880, E=32, k=4, scale_lo=120, scale_hi=124,
        description="gpt-oss-20b-shaped MoE layer, decode batch 1"),
    "gptoss20b_b64": LayerConfig(
        "gptoss20b_b64", T=64, H=2880, I=2880, E=32, k=4, scale_lo=120, scale_hi=124,
        description="gpt-oss-20b-shaped MoE layer, decode batch 64"),
    "gptoss120b_b64": LayerConfig(
        "gptoss120b_b64", T=64, H=2880, I=2880, E=128, k=4, scale_lo=120, scale_hi=124,
        description="gpt-oss-120b-shaped MoE layer, decode batch 64"),
    "gptoss120b_b1": LayerConfig(
        "gptoss120b_b1", T=1, H=2880, I=2880, E=128, k=4, scale_lo=120, scale_hi=124,
        description="gpt-oss-120b-shaped MoE layer, decode batch 1"),
    "gptoss120b_prefill4096": LayerConfig(
        "gptoss120b_prefill4096", T=4096, H=2880, I=2880, E=128, k=4, scale_lo=120,
        scale_hi=124, zipf_s=1.1, zipf_beta=1.0,
        description="gpt-oss-120b-shaped prefill, T=4096, Zipf(1.1) router bias"),
}


def zipf_router_bias(E: int, s: float, beta: float, rng: np.random.Generator) -> np.ndarray:
    """Per-expert log-prior bias: expert e gets rank r(e) from a seeded permutation and
    bias beta * ln p_r with p_r proportional to r^-s (normalised over the E experts)."""
    ranks = rng.permutation(E) + 1
    p = ranks.astype(np.float64) ** (-s)
    p /= p.sum()
    return (beta * np.log(p)).astype(np.float32)


def _draw_mxfp4(rng, rows_shape, K, lo, hi):
    codes = rng.integers(0, 256, size=tuple(rows_shape) + (K // 2,), dtype=np.uint8)
    scales = rng.integers(lo, hi + 1, size=tuple(rows_shape) + (K // 32,), dtype=np.uint8)
    return codes, scales


def make_layer(T, H, I, E, k, seed=0, scale_lo=120, scale_hi=124, zipf_s=None,
               zipf_beta=1.0, name="custom") -> LayerInputs:
    """Draw one layer's inputs (shapes and distributions as in the module docstring)."""
    if H % 32 or I % 32:
        raise ValueError("H and I must be multiples of 32 (one MX block)")
    rng = np.random.Generator(np.random.PCG64(seed))
    x = bf16_bits_from_f32(rng.standard_normal((T, H), dtype=np.float32))
    w_router = bf16_bits_from_f32(0.02 * rng.standard_normal((E, H), dtype=np.float32))
    gu_codes, gu_scales = _draw_mxfp4(rng, (E, 2 * I), H, scale_lo, scale_hi)
    dn_codes, dn_scales = _draw_mxfp4(rng, (E, H), I, scale_lo, scale_hi)
    bias = None
    if zipf_s is not None:
        bias = zipf_router_bias(E, zipf_s, zipf_beta, rng)
    return LayerInputs(name, T, H, I, E, k, x, w_router, gu_codes, gu_scales, dn_codes,
                       dn_scales, bias, meta={"seed": seed, "scale_range": (scale_lo, scale_hi),
                                              "zipf_s": zipf_s, "zipf_beta": zipf_beta})


def make_config(name: str, seed: int = 0, T: Optional[int] = None) -> LayerInputs:
    """Inputs of a named workload (``T`` may be overridden for smaller samples)."""
    c = CONFIGS[name]
    return make_layer(c.T if T is None else T, c.H, c.I, c.E, c.k, seed=seed,
                      scale_lo=c.scale_lo, scale_hi=c.scale_hi, zipf_s=c.zipf_s,
                      zipf_beta=c.zipf_beta, name=name)


def make_norm_inputs(T: int, H: int, seed: int = 0):
    """Inputs of the RMSNorm + residual step before the layer: the residual stream
    (bf16 [T, H], normal with standard deviation 2), the per-feature norm weight
    (bf16 [H], 1 + 0.25 * normal) and eps = 1e-5."""
    rng = np.random.Generator(np.random.PCG64(seed + 7919))
    residual = bf16_bits_from_f32(2.0 * rng.standard_normal((T, H), dtype=np.float32))
    gamma = bf16_bits_from_f32(1.0 + 0.25 * rng.standard_normal(H, dtype=np.float32))
    return residual, gamma, 1e-5


@dataclass
class DenseLayerInputs:
    """The layer with bf16 expert weights: w_gateup [E, 2I, H] (gate rows, then up
    rows), w_down [E, H, I], bf16 bit patterns."""
    name: str
    T: int
    H: int
    I: int
    E: int
    k: int
    x: np.ndarray
    w_router: np.ndarray
    w_gateup: np.ndarray
    w_down: np.ndarray
    router_bias: Optional[np.ndarray] = None
    meta: dict = field(default_factory=dict)


def make_dense_layer(T, H, I, E, k, seed=0, w_std=0.02, name="custom_dense") -> DenseLayerInputs:
    """x ~ N(0, 1); router weight ~ N(0, 0.02^2); expert weights ~ N(0, w_std^2), drawn
    one expert at a time; all rounded to bf16."""
    rng = np.random.Generator(np.random.PCG64(seed + 104729))
    x = bf16_bits_from_f32(rng.standard_normal((T, H), dtype=np.float32))
    w_router = bf16_bits_from_f32(0.02 * rng.standard_normal((E, H), dtype=np.float32))
    w_gateup = np.empty((E, 2 * I, H), np.uint16)
    w_down = np.empty((E, H, I), np.uint16)
    for e in range(E):
        w_gateup[e] = bf16_bits_from_f32(w_std * rng.standard_normal((2 * I, H), dtype=np.float32))
        w_down[e] = bf16_bits_from_f32(w_std * rng.standard_normal((H, I), dtype=np.float32))
    return DenseLayerInputs(name, T, H, I, E, k, x, w_router, w_gateup, w_down,
                            meta={"seed": seed, "w_std": w_std})


# bf16-weight workloads: Mixtral-8x7B expert shapes at the token counts of the
# fused-MoE dispatch table, and a small case for quick parity
DENSE_CONFIGS = {
    "dense_tiny": dict(T=8, H=256, I=384, E=4, k=2),
    "mixtral_t32": dict(T=32, H=4096, I=14336, E=8, k=2),
    "mixtral_t128": dict(T=128, H=4096, I=14336, E=8, k=2),
    "mixtral_t512": dict(T=512, H=4096, I=14336, E=8, k=2),
    "mixtral_t2048": dict(T=2048, H=4096, I=14336, E=8, k=2),
}


def make_dense_config(name: str, seed: int = 0, T: Optional[int] = None) -> DenseLayerInputs:
    c = dict(DENSE_CONFIGS[name])
    if T is not None:
        c["T"] = T
    return make_dense_layer(seed=seed, name=name, **c)


def random_logits(T: int, E: int, seed: int = 0, n_ties: int = 0) -> np.ndarray:
    """Router logits drawn N(0, 1) in float32.  ``n_ties`` tokens get an exact tie
    planted between two experts so tie-breaking is exercised."""
    rng = np.random.Generator(np.random.PCG64(seed))
    lg = rng.standard_normal((T, E), dtype=np.float32)
    for t in range(min(n_ties, T) if E >= 2 else 0):
        a, b = rng.choice(E, size=2, replace=False)
        lg[t, b] = lg[t, a]
    return lg


def random_topk_idx(T: int, E: int, k: int, seed: int = 0, skew: float = 0.0) -> np.ndarray:
    """k distinct expert indices per token (int32 [T, k]); ``skew`` > 0 draws experts
    with Zipf-like weights so some experts receive many tokens."""
    rng = np.random.Generator(np.random.PCG64(seed))
    p = None
    if skew > 0:
        p = (np.arange(1, E + 1, dtype=np.float64) ** -skew)
        p = p[rng.permutation(E)]
        p /= p.sum()
    out = np.empty((T, k), dtype=np.int32)
    for t in range(T):
        out[t] = rng.choice(E, size=k, replace=False, p=p)
    return out
