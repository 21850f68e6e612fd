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


def test_gemm_waits_time_out_into_the_status_word():
    """A wait limit far below the pipeline's own latency makes the expert GEMMs' waits
    give up on an ordinary call.  Each kernel sets its status bit, drains the copies
    and tensor-core work it already issued, and exits.  Nothing traps and the context
    stays usable: the next call, with the default limit and a re-zeroed workspace,
    matches the oracle."""
    import numpy as np
    import torch
    import mxfp4_expert_layer_gb300 as pkg
    from mxfp4_expert_layer_gb300 import _lib as L
    import oracle
    from synthetic import make_config
    from tests.gpu_helpers import (TOL_MAX_ABS, TOL_REL_FROB, bf16_bits_to_f32, bf16_to_np, build_layer, errors,
                                   logit_band, to_dev)
    pkg.build()
    inp = make_config("gptoss20b_b1")
    layer = build_layer(inp)
    x = to_dev(inp.x)
    assert L.moe_set_wait_limit_ns(1) == L.MOE_OK
    try:
        layer(x)
        torch.cuda.synchronize()
        st = layer.device_status(inp.T)
    finally:
        assert L.moe_set_wait_limit_ns(0) == L.MOE_OK
    timeout_bits = 0b111  # main loop, epilogue, producer
    assert st != 0 and (st & ~timeout_bits) == 0, st
    assert L.moe_set_wait_limit_ns(11 * 10 ** 9) == L.MOE_ERR_INVALID_ARG
    # the context is healthy: a normal call on the re-zeroed workspace is correct
    layer.workspace(inp.T).zero_()
    out = layer(x)
    torch.cuda.synchronize()
    assert layer.device_status(inp.T) == 0
    ref = oracle.moe_layer(inp)
    keep = oracle.topk_margin(ref["logits"], inp.k) > logit_band(inp)[0]
    rel, mx = errors(bf16_bits_to_f32(bf16_to_np(out))[keep], ref["out"][keep])
    assert rel <= TOL_REL_FROB and mx <= TOL_MAX_ABS, (rel, mx)
