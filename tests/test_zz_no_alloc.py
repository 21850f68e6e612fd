"""The allocation-free routing entry point gives the same routing as moe_route.

moe_route_noalloc serves callers that cannot call cudaMalloc (a runtime that owns
a fixed memory pool, a plugin handed only its input and output buffers): its
scratch lives in a fixed array inside the library instead of a caller workspace.
This file is collected last so that a run stopping at the first failure has run
every other test first; it passes alone in a fresh process and after the rest.
"""

import numpy as np
import pytest

from synthetic import make_config, make_layer
from tests.gpu_helpers import to_dev

pytestmark = pytest.mark.gpu


def _route_both(inp, calls=2):
    import torch
    import mxfp4_expert_layer_gb300 as pkg
    from mxfp4_expert_layer_gb300 import _lib as L
    pkg.build()
    T, H, E, k = inp.T, inp.H, inp.E, inp.k
    x, wr = to_dev(inp.x), to_dev(inp.w_router)
    bias = None if inp.router_bias is None else to_dev(inp.router_bias)
    ref_lg, ref_idx, ref_w = pkg.route(x, wr, k, bias=bias)
    s = torch.cuda.current_stream().cuda_stream
    results = []
    for _ in range(calls):
        lg = torch.full((T, E), float("nan"), dtype=torch.float32, device="cuda")
        idx = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
        w = torch.full((T, k), float("nan"), dtype=torch.float32, device="cuda")
        st = L.moe_route_noalloc(x.data_ptr(), wr.data_ptr(), None if bias is None else bias.data_ptr(), T, H, E,
                                 k, lg.data_ptr(), 0, idx.data_ptr(), w.data_ptr(), s)
        assert st == 0, L.moe_error_string(st)
        torch.cuda.synchronize()
        results.append((lg.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy()))
    return (ref_lg.cpu().numpy(), ref_idx.cpu().numpy(), ref_w.cpu().numpy()), results


@pytest.mark.parametrize("inp", [make_config("gptoss20b_b64"), make_layer(T=37, H=256, I=64, E=16, k=3, seed=4)],
                         ids=["gptoss20b_b64", "ragged_T37"])
def test_noalloc_route_matches_workspace_route_twice(inp):
    (ref_lg, ref_idx, ref_w), results = _route_both(inp, calls=2)
    for lg, idx, w in results:
        np.testing.assert_allclose(lg, ref_lg, rtol=0, atol=0)
        assert np.array_equal(idx, ref_idx)
        np.testing.assert_allclose(w, ref_w, rtol=2e-6, atol=1e-7)


def test_noalloc_route_rejects_tokens_beyond_its_scratch():
    import mxfp4_expert_layer_gb300 as pkg
    from mxfp4_expert_layer_gb300 import _lib as L
    pkg.build()
    fake = 1 << 20
    st = L.moe_route_noalloc(fake, fake, None, 8193, 2880, 32, 4, fake, 0, fake, fake, None)
    assert st == L.MOE_ERR_UNSUPPORTED_SHAPE
