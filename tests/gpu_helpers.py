"""Helpers shared by the GPU parity tests: move seeded inputs to the device, run
the library through its C ABI, and measure errors against the oracle."""

from __future__ import annotations

import numpy as np

TOL_REL_FROB = 5e-3      # relative Frobenius error bound on the layer output
TOL_MAX_ABS = 2e-2       # max abs error bound, relative to max |ref|


def to_dev(a: np.ndarray, dev="cuda"):
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
    return torch.from_numpy(a).to(dev)


def bf16_to_np(t) -> np.ndarray:
    return t.contiguous().view(__import__("torch").int16).cpu().numpy().view(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def errors(got: np.ndarray, ref: np.ndarray):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    mx = np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30)
    return rel, mx


def build_layer(inp, dev="cuda"):
    import mxfp4_expert_layer_gb300 as pkg
    pkg.build()
    wr = to_dev(inp.w_router, dev)
    bias = None if inp.router_bias is None else to_dev(inp.router_bias, dev)
    layer = pkg.MoELayer.from_mxfp4(wr, to_dev(inp.gu_codes, dev), to_dev(inp.gu_scales, dev),
                                    to_dev(inp.dn_codes, dev), to_dev(inp.dn_scales, dev), k=inp.k,
                                    router_bias=bias)
    return layer


def logit_band(inp, x_bits=None, factor=4.0, floor=1e-6):
    """Near-tie exclusion band for layer-level comparisons, from the logit error
    actually measured on this input: `factor` times the largest |GPU - oracle| router
    logit (the GPU's router on the same bf16 rows), at least `floor` (the 1e-6
    margin the workload statement gives).  A token whose oracle top-k margin exceeds
    twice the largest logit error routes to the same experts on both sides; the
    factor leaves room on top of that.  Returns (band, measured error)."""
    import oracle
    import mxfp4_expert_layer_gb300 as pkg
    xb = inp.x if x_bits is None else x_bits
    bias = None if inp.router_bias is None else to_dev(inp.router_bias)
    lg, _, _ = pkg.route(to_dev(xb), to_dev(inp.w_router), inp.k, bias=bias)
    ref = oracle.router_logits(xb, inp.w_router, inp.router_bias)
    err = float(np.abs(lg.cpu().numpy().astype(np.float64) - ref.astype(np.float64)).max())
    return max(factor * err, floor), err


def tile_edge_tokens(idx: np.ndarray, E: int, bm: int) -> np.ndarray:
    """Tokens whose assignments sit at the first or the last row of some tile of the
    routing `idx` (every expert's tiles, partial last tiles included), so that a
    sampled comparison reaches every tile of the grouped GEMMs."""
    import oracle
    tab = oracle.tile_table(idx, E, bm)
    k = idx.shape[1]
    rows = []
    for e, s0, n, _ in tab["tiles"]:
        rows += [int(s0), int(s0) + int(n) - 1]
    return np.unique(tab["perm"][np.asarray(rows, dtype=np.int64)] // k)
