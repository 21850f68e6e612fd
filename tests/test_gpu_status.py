"""Failure detection on the GPU: the device status word and its read-back.

Every bounded device wait that gives up sets a bit in a status word instead of
trapping; moe_get_device_status reads and clears it.  The read-and-clear logic is
exercised here with a word planted from the host (no kernel is made to fail)."""

import ctypes

import pytest

pytestmark = pytest.mark.gpu


def test_status_word_is_read_and_cleared():
    import torch
    import mxfp4_expert_layer_gb300 as pkg
    from mxfp4_expert_layer_gb300 import _lib as L
    pkg.build()
    ws = pkg.workspace(4, 256, 256, 8, 2)
    s = torch.cuda.current_stream().cuda_stream
    v = ctypes.c_int(-1)
    assert L.moe_get_device_status(ws.data_ptr(), ws.numel(), ctypes.byref(v), s) == L.MOE_OK and v.value == 0
    ws[:4] = torch.tensor([5, 0, 0, 0], dtype=torch.uint8, device="cuda")  # bits 0 and 2
    ws[4:256] = 7  # the rest of the status block is cleared too
    assert L.moe_get_device_status(ws.data_ptr(), ws.numel(), ctypes.byref(v), s) == L.MOE_ERR_DEVICE_TIMEOUT
    assert v.value == 5
    assert int(ws[:256].sum()) == 0
    assert L.moe_get_device_status(ws.data_ptr(), ws.numel(), ctypes.byref(v), s) == L.MOE_OK and v.value == 0
    assert L.moe_get_device_status(ws.data_ptr(), 255, ctypes.byref(v), s) == L.MOE_ERR_INVALID_ARG
