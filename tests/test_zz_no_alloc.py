"""The allocation-free routing entry point gives the same routing as moe_route.

moe_route_noalloc serves callers that cannot call cudaMalloc (a runtime that owns
a fixed memory pool, a plugin handed only its input and output buffers): its
scratch lives in a fixed array inside the library instead of a caller workspace.
The cases reach every routing kernel through it: the one-cluster router (T <= 64),
the many-token tensor-core router (T > 64, up to the array's 8192-token limit) and
the logits-given path, whose last-block hand-off uses the array's arrival
counters; each case runs twice in a row, so the second call finds the counters the
first one left.  This file is collected last so that a run stopping at the first
failure has run every other test first; it passes alone in a fresh process and
after the rest.
"""

import ctypes

import numpy as np
import pytest

import oracle
from synthetic import make_config, make_layer, random_logits
from tests.gpu_helpers import to_dev

pytestmark = pytest.mark.gpu


def _lib():
    import mxfp4_expert_layer_gb300 as pkg
    from mxfp4_expert_layer_gb300 import _lib as L
    pkg.build()
    return L


def _noalloc(L, x, wr, bias, T, H, E, k, flags, logits=None):
    import torch
    s = torch.cuda.current_stream().cuda_stream
    lg = logits if logits is not None else torch.full((T, E), float("nan"), dtype=torch.float32, device="cuda")
    idx = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
    w = torch.full((T, k), float("nan"), dtype=torch.float32, device="cuda")
    p = lambda t: None if t is None else t.data_ptr()
    st = L.moe_route_noalloc(p(x), p(wr), p(bias), T, H, E, k, lg.data_ptr(), flags, idx.data_ptr(), w.data_ptr(),
                             s)
    assert st == 0, L.moe_error_string(st)
    torch.cuda.synchronize()
    return lg.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy()


def _status(L):
    import torch
    v = ctypes.c_int(-1)
    rc = L.moe_route_noalloc_status(ctypes.byref(v), torch.cuda.current_stream().cuda_stream)
    return rc, v.value


CASES = [
    ("gptoss20b_b64", lambda: make_config("gptoss20b_b64")),                         # cluster router
    ("ragged_T37", lambda: make_layer(T=37, H=256, I=64, E=16, k=3, seed=4)),         # cluster router
    ("T300", lambda: make_layer(T=300, H=512, I=64, E=64, k=4, seed=5)),              # many-token router
    ("T8192_zipf_bias", lambda: make_layer(T=8192, H=2880, I=32, E=128, k=4, seed=6, zipf_s=1.1)),  # the limit
]


@pytest.mark.parametrize("name,make", CASES, ids=[c[0] for c in CASES])
def test_noalloc_route_matches_workspace_route_twice(name, make):
    import mxfp4_expert_layer_gb300 as pkg
    L = _lib()
    inp = make()
    T, H, E, k = inp.T, inp.H, inp.E, inp.k
    x, wr = to_dev(inp.x), to_dev(inp.w_router)
    bias = None if inp.router_bias is None else to_dev(inp.router_bias)
    ref_lg, ref_idx, ref_w = (t.cpu().numpy() for t in pkg.route(x, wr, k, bias=bias))
    for _ in range(2):
        lg, idx, w = _noalloc(L, x, wr, bias, T, H, E, k, 0)
        np.testing.assert_array_equal(lg, ref_lg)
        np.testing.assert_array_equal(idx, ref_idx)
        np.testing.assert_allclose(w, ref_w, rtol=2e-6, atol=1e-7)
    assert _status(L) == (0, 0)


@pytest.mark.parametrize("T,E,k", [(1000, 32, 4), (8192, 128, 4), (5, 8, 8)])
def test_noalloc_route_from_logits_matches_oracle_twice(T, E, k):
    """Given identical logits (ties planted), the indices are the oracle's bit for bit
    and the weights its softmax over the selected logits."""
    L = _lib()
    lg_np = random_logits(T, E, seed=T + E, n_ties=min(T, 64))
    ref_idx, ref_w = oracle.topk_softmax(lg_np, k)
    lg = to_dev(lg_np)
    for _ in range(2):
        _, idx, w = _noalloc(L, None, None, None, T, 32, E, k, L.MOE_ROUTE_FROM_LOGITS, logits=lg)
        np.testing.assert_array_equal(idx, ref_idx)
        np.testing.assert_allclose(w, ref_w, rtol=2e-6, atol=1e-7)
    assert _status(L) == (0, 0)


def test_noalloc_route_rejects_tokens_beyond_its_scratch():
    L = _lib()
    fake = 1 << 20
    st = L.moe_route_noalloc(fake, fake, None, 8193, 2880, 32, 4, fake, 0, fake, fake, None)
    assert st == L.MOE_ERR_UNSUPPORTED_SHAPE
    assert L.moe_route_noalloc_status(None, None) == L.MOE_ERR_INVALID_ARG
