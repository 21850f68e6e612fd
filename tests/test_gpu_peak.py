"""The tensor-pipe rate probe that the compute-bound roofline is taken against:
both MMA forms run to completion and give rates in the range a GB300 can reach
(kind::mxf4 above kind::f16, both below the nominal dense peaks)."""

import ctypes

import pytest

pytestmark = pytest.mark.gpu


def test_tensor_peak_probe():
    import torch
    import mxfp4_expert_layer_gb300 as pkg
    from mxfp4_expert_layer_gb300 import _lib as L
    pkg.build()
    s = torch.cuda.current_stream().cuda_stream
    mx, bf = ctypes.c_double(0), ctypes.c_double(0)
    assert L.moe_tensor_peak(L.MOE_PEAK_MXF4, 4096, ctypes.byref(mx), s) == L.MOE_OK
    assert L.moe_tensor_peak(L.MOE_PEAK_BF16, 4096, ctypes.byref(bf), s) == L.MOE_OK
    assert 500.0 < bf.value < 2600.0, bf.value        # nominal dense bf16: 2.25 PFLOP/s
    assert 2.0 * bf.value < mx.value < 14000.0, (mx.value, bf.value)  # nominal dense fp4: 13.5 PFLOP/s
    assert L.moe_tensor_peak(7, 4096, ctypes.byref(mx), s) == L.MOE_ERR_INVALID_ARG
    assert L.moe_tensor_peak(L.MOE_PEAK_MXF4, 4, ctypes.byref(mx), s) == L.MOE_ERR_INVALID_ARG
