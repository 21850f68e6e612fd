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
