"""Plain CPU oracle of the MXFP4 mixture-of-experts layer.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the CPU-baseline leg of
the benchmark use it; the product path never does.

What it computes is the plain definition of a gpt-oss-style MoE layer, step by
step, in the order the sources state it:

* "A 297-line kernel file that decodes faster than vLLM" (cloudy.so), section
  "Where the time went", table rows "Router + top-k", "MoE gate/up + SwiGLU",
  "MoE down + combine": the three stages of the layer.
* same page, section "Optimizations", rows "MXFP4 MoE on tensor cores" and
  "Per-expert routing tile table"; section "Correctness" (a float32 reference is
  what every kernel is compared against, so float32 is the default precision).
* "triton-kernels" README (github bassrehab/triton-kernels), section "Quick Start",
  "Fused MoE Dispatch": router -> permute -> fused expert FFN -> unpermute, with
  softmax gating, returning output, expert indices and expert weights; section
  "Project Structure" names a loop-over-experts PyTorch ground truth, which is the
  pattern followed here.
* MXFP4 itself is the OCP Microscaling (MX) v1.0 format: blocks of 32 FP4 E2M1
  elements sharing one E8M0 scale, value = E2M1(code) * 2^(scale - 127).

Readings taken where the sources are silent (each is also listed in the design
notes): even K index in the low nibble; gate rows [0, I) then up rows [I, 2I);
no biases other than an optional per-expert router bias, no SwiGLU clamp; softmax
over the k selected logits only; top-k ties broken towards the lower expert index;
rows of one expert ordered by ascending t*k + j; output rounded once to bf16.

Every function works in ``dtype`` (float32 by default, float64 for self-checks);
library primitives (matmul, stable sort) are used as single steps, with no
blocking, fusion or reordering beyond the definition.
"""

from __future__ import annotations

import numpy as np

# OCP MX v1.0, FP4 E2M1: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0.
E2M1_VALUES = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
               -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 (bf16 is the top half of a float32)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def bf16_round(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); returned as float32.
    NaN is kept as a quiet NaN."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    out = r.astype(np.uint32).view(np.float32).copy()
    nan = np.isnan(a)
    out[nan] = np.float32("nan")
    return out


def decode_e8m0(scales: np.ndarray, dtype=np.float32) -> np.ndarray:
    """E8M0 scale byte s -> 2^(s - 127).  s = 255 is NaN in the MX format and is
    rejected: a layer whose weights carry it has no defined output."""
    s = np.asarray(scales)
    if np.any(s == 255):
        raise ValueError("E8M0 scale 255 (NaN) in MXFP4 weights")
    one = np.ones(s.shape, dtype=dtype)
    return np.ldexp(one, s.astype(np.int32) - 127).astype(dtype)


def decode_mxfp4(codes: np.ndarray, scales: np.ndarray, dtype=np.float32) -> np.ndarray:
    """MXFP4 rows -> real values.  ``codes`` [..., K/2] (even K index in the low
    nibble), ``scales`` [..., K/32]; returns [..., K] in ``dtype``.  Every value is
    E2M1[code] * 2^(s - 127), exact in float32."""
    codes = np.asarray(codes, dtype=np.uint8)
    K = codes.shape[-1] * 2
    # byte b holds two codes: (b & 15) at the even K index, (b >> 4) at the odd one
    pair = np.array([[E2M1_VALUES[b & 0x0F], E2M1_VALUES[b >> 4]] for b in range(256)], dtype=dtype)
    vals = pair[codes].reshape(codes.shape[:-1] + (K // 32, 32))
    sc = decode_e8m0(scales, dtype)
    if sc.shape[-1] * 32 != K:
        raise ValueError("scales must hold one byte per 32 codes")
    return (vals * sc[..., None]).reshape(codes.shape[:-1] + (K,))


def router_logits(x_bits: np.ndarray, w_router_bits: np.ndarray, bias=None,
                  dtype=np.float32) -> np.ndarray:
    """logits[t, e] = sum_h x[t, h] * W_r[e, h] (+ bias[e]); x, W_r given as bf16 bits."""
    x = bf16_to_f32(x_bits).astype(dtype)
    w = bf16_to_f32(w_router_bits).astype(dtype)
    lg = x @ w.T
    if bias is not None:
        lg = lg + np.asarray(bias, dtype=dtype)[None, :]
    return lg.astype(dtype)


def topk_softmax(logits: np.ndarray, k: int, dtype=np.float32):
    """Top-k experts per token by (logit descending, expert index ascending), listed
    in that order; weights = softmax over the k selected logits only.
    Returns (idx int32 [T, k], w [T, k])."""
    lg = np.asarray(logits)
    T, E = lg.shape
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    idx = np.empty((T, k), dtype=np.int32)
    for t in range(T):
        order = np.lexsort((np.arange(E), -lg[t].astype(np.float64)))
        idx[t] = order[:k]
    sel = np.take_along_axis(lg, idx, axis=1).astype(dtype)
    m = sel[:, :1]
    ex = np.exp(sel - m)
    w = ex / ex.sum(axis=1, keepdims=True)
    return idx, w.astype(dtype)


# Gating variants ("triton-kernels" README, section "Project Structure": the router
# does softmax or sigmoid gating + top-k; section "References": DeepSeek-V3, sigmoid
# gating).  The selection is the same in every variant (both maps are increasing):
GATING_SOFTMAX_TOPK = 0  # softmax over the k selected logits (the default)
GATING_SOFTMAX_ALL = 1   # softmax over all E logits; the selected experts' probabilities
GATING_SIGMOID = 2       # sigmoid of each selected logit, normalised to sum to 1


def topk_gating(logits: np.ndarray, k: int, gating: int = GATING_SOFTMAX_TOPK, dtype=np.float32):
    """Top-k experts per token by (logit descending, expert index ascending) and their
    weights under ``gating``.  Returns (idx int32 [T, k], w [T, k])."""
    if gating == GATING_SOFTMAX_TOPK:
        return topk_softmax(logits, k, dtype)
    idx, _ = topk_softmax(logits, k, dtype)
    lg = np.asarray(logits).astype(dtype)
    sel = np.take_along_axis(lg, idx, axis=1)
    if gating == GATING_SOFTMAX_ALL:
        m = lg.max(axis=1, keepdims=True)
        ex = np.exp(lg - m)
        w = np.take_along_axis(ex, idx, axis=1) / ex.sum(axis=1, keepdims=True)
    elif gating == GATING_SIGMOID:
        sg = 1.0 / (1.0 + np.exp(-sel))
        w = sg / sg.sum(axis=1, keepdims=True)
    else:
        raise ValueError("gating must be 0, 1 or 2")
    return idx, w.astype(dtype)


def topk_margin(logits: np.ndarray, k: int) -> np.ndarray:
    """Per token: (k-th largest logit) - ((k+1)-th largest); +inf when k == E.  A
    small margin marks a near-tie whose selection depends on rounding."""
    lg = np.sort(np.asarray(logits, dtype=np.float64), axis=1)[:, ::-1]
    if k >= lg.shape[1]:
        return np.full(lg.shape[0], np.inf)
    return lg[:, k - 1] - lg[:, k]


def tile_rows_policy(T: int, k: int, E: int) -> int:
    """Token rows per tile from the mean tokens per expert m = T*k/E: 16 for decode
    (m <= 16), 64 for m <= 64, else 128 ("token tile follows tokens per expert")."""
    m = T * k / E
    if m <= 16:
        return 16
    if m <= 64:
        return 64
    return 128


def max_tiles_bound(T: int, k: int, E: int, bm: int) -> int:
    """Upper bound on the number of tiles: sum_e ceil(c_e / bm) <= T*k//bm + min(E, T*k)."""
    return (T * k) // bm + min(E, T * k)


def tile_table(idx: np.ndarray, E: int, bm: int):
    """Per-expert tile table of a routing.

    counts[e]  = assignments (t, j) with idx[t, j] == e
    offsets    = exclusive prefix sum of counts, offsets[E] = T*k
    perm[s]    = the assignment a = t*k + j stored at sorted row s; rows are sorted
                 by expert, and within an expert by ascending a
    inv_perm[a] = s
    tiles[i]   = (expert, first sorted row, rows in tile, i*bm) for each expert in
                 ascending order, ceil(c_e / bm) tiles of bm consecutive rows, the
                 last one possibly partial
    """
    flat = np.asarray(idx, dtype=np.int64).reshape(-1)
    if flat.size and (flat.min() < 0 or flat.max() >= E):
        raise ValueError("expert index out of range")
    counts = np.bincount(flat, minlength=E).astype(np.int32)
    offsets = np.zeros(E + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    perm = np.argsort(flat, kind="stable").astype(np.int32)
    inv_perm = np.empty_like(perm)
    inv_perm[perm] = np.arange(flat.size, dtype=np.int32)
    tiles = []
    for e in range(E):
        c = int(counts[e])
        q = 0
        while q * bm < c:
            tiles.append((e, int(offsets[e]) + q * bm, min(bm, c - q * bm), len(tiles) * bm))
            q += 1
    tiles = np.asarray(tiles, dtype=np.int32).reshape(-1, 4)
    return {"counts": counts, "offsets": offsets, "perm": perm, "inv_perm": inv_perm,
            "tiles": tiles, "num_tiles": int(tiles.shape[0])}


def silu(g: np.ndarray) -> np.ndarray:
    """silu(g) = g * sigmoid(g) = g / (1 + exp(-g))."""
    with np.errstate(over="ignore"):
        return g / (1 + np.exp(-g))


def expert_hidden(x_rows: np.ndarray, gu_codes_e, gu_scales_e, I: int, dtype=np.float32):
    """Gate/up of one expert for rows of x: g = x W_gate^T, u = x W_up^T,
    h = silu(g) * u.  ``x_rows`` real [n, H]; returns h [n, I]."""
    w = decode_mxfp4(gu_codes_e, gu_scales_e, dtype)
    x_rows = np.asarray(x_rows, dtype=dtype)
    g = x_rows @ w[:I].T
    u = x_rows @ w[I:2 * I].T
    return (silu(g) * u).astype(dtype)


def expert_output(h_rows: np.ndarray, dn_codes_e, dn_scales_e, dtype=np.float32):
    """Down projection of one expert: y = h W_down^T; returns [n, H]."""
    w = decode_mxfp4(dn_codes_e, dn_scales_e, dtype)
    return (np.asarray(h_rows, dtype=dtype) @ w.T).astype(dtype)


def expert_hidden_dense(x_rows: np.ndarray, w_gateup_e_bits, I: int, dtype=np.float32):
    """Gate/up of one expert with bf16 weights (gate rows [0, I), up rows [I, 2I)):
    h = silu(x W_gate^T) * (x W_up^T); returns [n, I]."""
    w = bf16_to_f32(w_gateup_e_bits).astype(dtype)
    x_rows = np.asarray(x_rows, dtype=dtype)
    g = x_rows @ w[:I].T
    u = x_rows @ w[I:2 * I].T
    return (silu(g) * u).astype(dtype)


def expert_output_dense(h_rows: np.ndarray, w_down_e_bits, dtype=np.float32):
    """Down projection of one expert with bf16 weights: y = h W_down^T; [n, H]."""
    w = bf16_to_f32(w_down_e_bits).astype(dtype)
    return (np.asarray(h_rows, dtype=dtype) @ w.T).astype(dtype)


def moe_layer_dense(inp, dtype=np.float32, tokens=None, gating=None):
    """The same layer with bf16 expert weights (no MX scales): "triton-kernels"
    README, "Quick Start", "Fused MoE Dispatch (Mixtral / DeepSeek-V3 / Qwen2-MoE
    style)" (router -> permute -> fused expert FFN -> unpermute, gate/up/down weights
    [E, F, H] / [E, H, F], softmax gating over the top-k) and "MoE Dispatch
    Results" (Mixtral-8x7B: 8 experts, top-2, hidden 4096, ffn 14336).  Routing,
    gating and the combine are those of ``moe_layer``; ``inp`` carries ``w_gateup``
    (bf16 bits [E, 2I, H], gate rows then up rows) and ``w_down`` ([E, H, I])."""
    return moe_layer(inp, dtype=dtype, tokens=tokens,
                     gating=GATING_SOFTMAX_TOPK if gating is None else gating,
                     _experts=(lambda e, x: expert_hidden_dense(x, inp.w_gateup[e], inp.I, dtype),
                               lambda e, h: expert_output_dense(h, inp.w_down[e], dtype)))


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round to the nearest bf16 (ties to even) and return the bit patterns."""
    return (bf16_round(a).view(np.uint32) >> 16).astype(np.uint16)


def rmsnorm_residual(x_bits: np.ndarray, r_bits: np.ndarray, gamma_bits: np.ndarray, eps: float,
                     dtype=np.float32):
    """The step before the router on every decode layer: residual add, then RMSNorm.

    "triton-kernels" README (github bassrehab/triton-kernels), section "Kernels"
    (row ``rmsnorm_residual_fused``) and section "Quick Start", "Fused RMSNorm +
    Residual": the normalisation of x + residual with a per-feature weight and eps;
    "A 297-line kernel file that decodes faster than vLLM" (cloudy.so), section "Where
    the time went", row "RMSNorm + residual" (the step just before "Router + top-k").
    RMSNorm itself (Zhang & Sennrich, 2019): y = s / sqrt(mean(s^2) + eps) * gamma.

    Readings: the sum s = x + r is what the bf16 residual stream holds, so it is
    rounded to bf16 once (from its float32 value) and the norm is taken of that
    rounded s; y is rounded to bf16 (the layer's activations are bf16).
    Returns (s, y) as bf16 bit patterns, [T, H] each.
    """
    x = bf16_to_f32(x_bits)
    r = bf16_to_f32(r_bits)
    s = bf16_round((x + r).astype(np.float32))
    sd = s.astype(dtype)
    ms = np.mean(sd * sd, axis=-1, keepdims=True)
    y = sd / np.sqrt(ms + dtype(eps)) * bf16_to_f32(gamma_bits).astype(dtype)
    return bf16_bits(s), bf16_bits(y.astype(np.float32))


def moe_layer_norm(inp, residual_bits: np.ndarray, gamma_bits: np.ndarray, eps: float,
                   dtype=np.float32, **kw):
    """RMSNorm + residual (``rmsnorm_residual``), then the layer on the normalised
    rows: ``moe_layer`` with x replaced by y.  The result adds "residual_out" (s) and
    "x_norm" (y), bf16 bit patterns of all T rows."""
    import dataclasses
    s_bits, y_bits = rmsnorm_residual(inp.x, residual_bits, gamma_bits, eps, dtype)
    res = moe_layer(dataclasses.replace(inp, x=y_bits), dtype=dtype, **kw)
    res["residual_out"] = s_bits
    res["x_norm"] = y_bits
    return res


def moe_layer(inp, dtype=np.float32, tokens=None, logits=None, return_hidden=False,
              gating=GATING_SOFTMAX_TOPK, _experts=None):
    """The whole layer on the tokens ``tokens`` (default: all).

    Router -> top-k + gating weights -> per expert: gate/up + SwiGLU, down -> per token
    out[t] = sum_{j=0..k-1} w[t, j] * y[t, j] (j ascending), rounded once to bf16.
    ``logits`` may be supplied (float [T, E]) instead of being computed.

    Returns a dict with logits, idx, w, y [n, k, H], out (bf16 values as float32)
    and, when asked, h [n, k, I]; all restricted to ``tokens``.
    """
    T, H, I, E, k = inp.T, inp.H, inp.I, inp.E, inp.k
    tok = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    x_all = bf16_to_f32(inp.x[tok]).astype(dtype)
    if logits is None:
        lg = router_logits(inp.x[tok], inp.w_router, inp.router_bias, dtype)
    else:
        lg = np.asarray(logits, dtype=dtype)[tok]
    idx, w = topk_gating(lg, k, gating, dtype)
    n = tok.size
    y = np.zeros((n, k, H), dtype=dtype)
    h_all = np.zeros((n, k, I), dtype=dtype) if return_hidden else None
    if _experts is None:  # MXFP4 experts
        _experts = (lambda e, xr: expert_hidden(xr, inp.gu_codes[e], inp.gu_scales[e], I, dtype),
                    lambda e, hr: expert_output(hr, inp.dn_codes[e], inp.dn_scales[e], dtype))
    for e in np.unique(idx):
        rows, slots = np.nonzero(idx == e)
        h = _experts[0](e, x_all[rows])
        y[rows, slots] = _experts[1](e, h)
        if return_hidden:
            h_all[rows, slots] = h
    acc = np.zeros((n, H), dtype=dtype)
    for j in range(k):
        acc = acc + w[:, j:j + 1] * y[:, j]
    out = bf16_round(acc.astype(np.float32))
    res = {"tokens": tok, "logits": lg, "idx": idx, "w": w, "y": y, "out": out,
           "out_unrounded": acc}
    if return_hidden:
        res["h"] = h_all
    return res
