"""Torch-facing wrappers over the C ABI.  PyTorch supplies device memory and the
current CUDA stream; every step of the layer runs in the library's kernels.

    layer = MoELayer.from_mxfp4(w_router, gu_codes, gu_scales, dn_codes, dn_scales, k=4)
    out = layer(x)                      # x bf16 [T, H] on cuda -> bf16 [T, H]
"""

from __future__ import annotations

from typing import Optional

import torch

from . import _lib as L


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def _need_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


def prepare_weights(codes: torch.Tensor, scales: torch.Tensor, kind: int) -> torch.Tensor:
    """Raw MXFP4 [E, rows, K/2] codes + [E, rows, K/32] scales (uint8, cuda) ->
    prepared weight buffer (uint8, cuda)."""
    _need_cuda(codes, scales)
    E, rows, half_k = codes.shape
    K = half_k * 2
    nbytes = L.moe_prepared_weight_bytes(E, rows, K, kind)
    if nbytes == 0:
        raise ValueError(f"unsupported weight shape {tuple(codes.shape)}")
    dst = torch.empty(nbytes, dtype=torch.uint8, device=codes.device)
    L.check("moe_prepare_weights", L.moe_prepare_weights(codes.data_ptr(), scales.data_ptr(), E, rows, K, kind,
                                                          dst.data_ptr(), nbytes, _stream()))
    return dst


def prepare_weights_bf16(w: torch.Tensor, kind: int) -> torch.Tensor:
    """Raw bf16 expert weights [E, rows, K] (cuda) -> the prepared tile buffer
    (uint8, cuda) that moe_forward_bf16 streams."""
    _need_cuda(w)
    E, rows, K = w.shape
    nbytes = L.moe_prepared_weight_bytes_bf16(E, rows, K, kind)
    if nbytes == 0:
        raise ValueError(f"unsupported weight shape {tuple(w.shape)}")
    w = w.contiguous()
    dst = torch.empty(nbytes, dtype=torch.uint8, device=w.device)
    L.check("moe_prepare_weights_bf16", L.moe_prepare_weights_bf16(w.data_ptr(), E, rows, K, kind, dst.data_ptr(),
                                                                    nbytes, _stream()))
    return dst


def workspace(T: int, H: int, I: int, E: int, k: int, device="cuda") -> torch.Tensor:
    n = L.moe_workspace_bytes(T, H, I, E, k)
    if n == 0:
        raise ValueError("unsupported shape")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def tile_rows(T: int, k: int, E: int) -> int:
    return L.moe_tile_rows(T, k, E)


def max_tiles(T: int, k: int, E: int, bm: int) -> int:
    return L.moe_max_tiles(T, k, E, bm)


def route(x, w_router, k, bias=None, logits=None, from_logits=False, ws=None, gating=0):
    """Router logits (or given ones) -> (logits, topk_idx int32, topk_w float32).
    ``gating``: 0 (softmax over the k selected), MOE_ROUTE_GATING_SOFTMAX_ALL or
    MOE_ROUTE_GATING_SIGMOID."""
    if from_logits:
        T, E = logits.shape
        H = 32
    else:
        T, H = x.shape
        E = w_router.shape[0]
        _need_cuda(x, w_router, bias)
        if logits is None:
            logits = torch.empty(T, E, dtype=torch.float32, device=x.device)
    dev = logits.device
    idx = torch.empty(T, k, dtype=torch.int32, device=dev)
    w = torch.empty(T, k, dtype=torch.float32, device=dev)
    if ws is None:
        ws = workspace(T, 32, 32, E, k, dev)
    flags = (L.MOE_ROUTE_FROM_LOGITS if from_logits else 0) | gating
    L.check("moe_route", L.moe_route(_ptr(x), _ptr(w_router), _ptr(bias), T, H, E, k, logits.data_ptr(), flags,
                                     idx.data_ptr(), w.data_ptr(), ws.data_ptr(), ws.numel(), _stream()))
    return logits, idx, w


def build_tile_table(idx: torch.Tensor, E: int, bm: int = 0):
    _need_cuda(idx)
    T, k = idx.shape
    bm_eff = bm or L.moe_tile_rows(T, k, E)
    mt = L.moe_max_tiles(T, k, E, bm_eff)
    dev = idx.device
    out = {
        "counts": torch.empty(E, dtype=torch.int32, device=dev),
        "offsets": torch.empty(E + 1, dtype=torch.int32, device=dev),
        "perm": torch.empty(T * k, dtype=torch.int32, device=dev),
        "inv_perm": torch.empty(T * k, dtype=torch.int32, device=dev),
        "tiles": torch.zeros(max(mt, 1), 4, dtype=torch.int32, device=dev),
        "num_tiles": torch.empty(1, dtype=torch.int32, device=dev),
    }
    L.check("moe_build_tile_table",
            L.moe_build_tile_table(idx.data_ptr(), T, k, E, bm, out["counts"].data_ptr(),
                                   out["offsets"].data_ptr(), out["perm"].data_ptr(), out["inv_perm"].data_ptr(),
                                   out["tiles"].data_ptr(), out["num_tiles"].data_ptr(), _stream()))
    out["bm"] = bm_eff
    return out


class MoELayer:
    """One MXFP4 MoE layer: router weight, prepared expert weights and a workspace
    per token count."""

    def __init__(self, w_router: torch.Tensor, w_gateup: torch.Tensor, w_down: torch.Tensor, H: int, I: int,
                 E: int, k: int, router_bias: Optional[torch.Tensor] = None):
        self.w_router, self.w_gateup, self.w_down = w_router, w_gateup, w_down
        self.router_bias = router_bias
        self.H, self.I, self.E, self.k = H, I, E, k
        self._ws = {}

    @classmethod
    def from_mxfp4(cls, w_router, gu_codes, gu_scales, dn_codes, dn_scales, k, router_bias=None):
        E, two_i, half_h = gu_codes.shape
        H, I = half_h * 2, two_i // 2
        wgu = prepare_weights(gu_codes, gu_scales, L.MOE_WEIGHTS_GATEUP)
        wd = prepare_weights(dn_codes, dn_scales, L.MOE_WEIGHTS_DOWN)
        return cls(w_router, wgu, wd, H, I, E, k, router_bias)

    def workspace(self, T: int) -> torch.Tensor:
        ws = self._ws.get(T)
        if ws is None:
            ws = workspace(T, self.H, self.I, self.E, self.k, self.w_router.device)
            self._ws[T] = ws
        return ws

    def forward(self, x: torch.Tensor, out: Optional[torch.Tensor] = None, topk_idx=None, topk_w=None,
                ws: Optional[torch.Tensor] = None, gating: int = 0, residual: Optional[torch.Tensor] = None,
                norm_weight: Optional[torch.Tensor] = None, eps: float = 1e-5,
                residual_out: Optional[torch.Tensor] = None) -> torch.Tensor:
        """out = MoE(x); with ``residual`` and ``norm_weight``, out = MoE(RMSNorm(x +
        residual)) and, when given, ``residual_out`` receives bf16(x + residual)
        (moe_forward_norm)."""
        _need_cuda(x)
        T = x.shape[0]
        if out is None:
            out = torch.empty(T, self.H, dtype=torch.bfloat16, device=x.device)
        if ws is None:
            ws = self.workspace(T)
        if residual is not None or norm_weight is not None:
            if residual is None or norm_weight is None:
                raise ValueError("the norm step needs both residual and norm_weight")
            L.check("moe_forward_norm", L.moe_forward_norm(
                x.data_ptr(), residual.data_ptr(), norm_weight.data_ptr(), eps, self.w_router.data_ptr(),
                _ptr(self.router_bias), self.w_gateup.data_ptr(), self.w_down.data_ptr(), T, self.H, self.I,
                self.E, self.k, gating, ws.data_ptr(), ws.numel(), out.data_ptr(), _ptr(residual_out),
                _ptr(topk_idx), _ptr(topk_w), _stream()))
            return out
        if gating:
            L.check("moe_forward_gated", L.moe_forward_gated(
                x.data_ptr(), self.w_router.data_ptr(), _ptr(self.router_bias), self.w_gateup.data_ptr(),
                self.w_down.data_ptr(), T, self.H, self.I, self.E, self.k, gating, ws.data_ptr(), ws.numel(),
                out.data_ptr(), _ptr(topk_idx), _ptr(topk_w), _stream()))
            return out
        L.check("moe_forward", L.moe_forward(
            x.data_ptr(), self.w_router.data_ptr(), _ptr(self.router_bias), self.w_gateup.data_ptr(),
            self.w_down.data_ptr(), T, self.H, self.I, self.E, self.k, ws.data_ptr(), ws.numel(), out.data_ptr(),
            _ptr(topk_idx), _ptr(topk_w), _stream()))
        return out

    __call__ = forward

    def device_status(self, T: int) -> int:
        import ctypes
        ws = self.workspace(T)
        st = ctypes.c_int(0)
        L.moe_get_device_status(ws.data_ptr(), ws.numel(), ctypes.byref(st), _stream())
        return st.value


class MoELayerBF16:
    """The same layer with bf16 expert weights (moe_forward_bf16): w_gateup [E, 2I, H]
    (gate rows, then up rows) and w_down [E, H, I], prepared once into the tiles the
    kernels stream (moe_prepare_weights_bf16); the layer keeps only the prepared
    buffers."""

    def __init__(self, w_router: torch.Tensor, w_gateup: torch.Tensor, w_down: torch.Tensor, k: int,
                 router_bias: Optional[torch.Tensor] = None):
        E, two_i, H = w_gateup.shape
        self.w_router = w_router
        self.w_gateup = prepare_weights_bf16(w_gateup, L.MOE_WEIGHTS_GATEUP)
        self.w_down = prepare_weights_bf16(w_down, L.MOE_WEIGHTS_DOWN)
        self.router_bias = router_bias
        self.H, self.I, self.E, self.k = H, two_i // 2, E, k
        self._ws = {}

    def workspace(self, T: int) -> torch.Tensor:
        ws = self._ws.get(T)
        if ws is None:
            ws = workspace(T, self.H, self.I, self.E, self.k, self.w_router.device)
            self._ws[T] = ws
        return ws

    def forward(self, x: torch.Tensor, out: Optional[torch.Tensor] = None, topk_idx=None, topk_w=None,
                ws: Optional[torch.Tensor] = None) -> torch.Tensor:
        _need_cuda(x)
        T = x.shape[0]
        if out is None:
            out = torch.empty(T, self.H, dtype=torch.bfloat16, device=x.device)
        if ws is None:
            ws = self.workspace(T)
        L.check("moe_forward_bf16", L.moe_forward_bf16(
            x.data_ptr(), self.w_router.data_ptr(), _ptr(self.router_bias), self.w_gateup.data_ptr(),
            self.w_down.data_ptr(), T, self.H, self.I, self.E, self.k, ws.data_ptr(), ws.numel(), out.data_ptr(),
            _ptr(topk_idx), _ptr(topk_w), _stream()))
        return out

    __call__ = forward

    def device_status(self, T: int) -> int:
        import ctypes
        ws = self.workspace(T)
        st = ctypes.c_int(0)
        L.moe_get_device_status(ws.data_ptr(), ws.numel(), ctypes.byref(st), _stream())
        return st.value

