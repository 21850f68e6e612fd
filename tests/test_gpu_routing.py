"""GPU parity of the routing stages against the oracle: top-k and softmax from
identical logits (bit-exact indices), router logits, and the tile table
(bit-exact counts, offsets, permutation and tiles)."""

import numpy as np
import pytest

import oracle
from synthetic import make_config, make_layer, random_logits, random_topk_idx
from tests.gpu_helpers import to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api():
    import mxfp4_expert_layer_gb300 as pkg
    pkg.build()
    from mxfp4_expert_layer_gb300 import api
    return api


@pytest.mark.parametrize("T,E,k,seed", [(4, 8, 2, 0), (1, 32, 4, 1), (64, 32, 4, 2), (64, 128, 4, 3),
                                        (4096, 128, 4, 4), (37, 256, 8, 5), (9, 5, 5, 6), (3, 1, 1, 7)])
def test_topk_softmax_from_identical_logits(api, T, E, k, seed):
    lg = random_logits(T, E, seed=seed, n_ties=T // 3)
    _, idx, w = api.route(None, None, k, logits=to_dev(lg), from_logits=True)
    ref_idx, ref_w = oracle.topk_softmax(lg, k)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    np.testing.assert_allclose(w.cpu().numpy(), ref_w, rtol=2e-6, atol=1e-7)


@pytest.mark.parametrize("T,E,k,seed", [(5, 8, 2, 0), (3, 32, 4, 1), (70, 128, 4, 2), (37, 256, 8, 3)])
@pytest.mark.parametrize("flag,gating", [(2, 1), (4, 2)])
def test_gating_variants_from_identical_logits(api, T, E, k, seed, flag, gating):
    """Softmax over all experts (flag 2) and normalised sigmoid (flag 4): the same
    selection as the default, weights by the oracle's variant."""
    lg = random_logits(T, E, seed=seed, n_ties=T // 3)
    _, idx, w = api.route(None, None, k, logits=to_dev(lg), from_logits=True, gating=flag)
    ref_idx, ref_w = oracle.topk_gating(lg, k, gating)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    np.testing.assert_allclose(w.cpu().numpy(), ref_w, rtol=2e-6, atol=1e-7)


@pytest.mark.parametrize("name,T,flag,gating", [("gptoss20b_b64", None, 4, 2), ("gptoss120b_b64", None, 2, 1),
                                                ("gptoss120b_prefill4096", 300, 4, 2)])
def test_router_gating_variants(api, name, T, flag, gating):
    """The variants through the decode cluster router and the many-token router."""
    inp = make_config(name, T=T)
    x, wr = to_dev(inp.x), to_dev(inp.w_router)
    bias = None if inp.router_bias is None else to_dev(inp.router_bias)
    lg, idx, w = api.route(x, wr, inp.k, bias=bias, gating=flag)
    # weights from the GPU's own logits: the selection is bit-exact and the weights
    # follow the variant's formula
    ref_idx, ref_w = oracle.topk_gating(lg.cpu().numpy(), inp.k, gating)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    np.testing.assert_allclose(w.cpu().numpy(), ref_w, rtol=2e-6, atol=1e-7)


@pytest.mark.parametrize("name,T", [("tiny", None), ("gptoss20b_b1", None), ("gptoss20b_b64", None),
                                    ("gptoss120b_b64", None), ("gptoss120b_prefill4096", None)])
def test_router_logits_and_selection(api, name, T):
    inp = make_config(name, T=T)
    x, wr = to_dev(inp.x), to_dev(inp.w_router)
    bias = None if inp.router_bias is None else to_dev(inp.router_bias)
    lg, idx, w = api.route(x, wr, inp.k, bias=bias)
    ref = oracle.router_logits(inp.x, inp.w_router, inp.router_bias)
    got = lg.cpu().numpy()
    # fp32 sums of H products in a different order: bound by H * eps * sum|x w|
    xa = np.abs(oracle.bf16_to_f32(inp.x)).astype(np.float64)
    wa = np.abs(oracle.bf16_to_f32(inp.w_router)).astype(np.float64)
    bound = inp.H * 2.0 ** -24 * (xa @ wa.T) + 1e-6
    assert np.all(np.abs(got - ref) <= bound)
    # selections agree wherever the top-k margin exceeds twice the largest logit error
    # (band: four times the error measured here, at least 1e-6)
    margin = oracle.topk_margin(ref, inp.k)
    ok = margin > max(4.0 * float(np.abs(got.astype(np.float64) - ref).max()), 1e-6)
    ref_idx, ref_w = oracle.topk_softmax(ref, inp.k)
    assert np.array_equal(idx.cpu().numpy()[ok], ref_idx[ok])
    np.testing.assert_allclose(w.cpu().numpy()[ok], ref_w[ok], rtol=1e-4, atol=1e-6)
    assert ok.mean() > 0.9


@pytest.mark.parametrize("T,H,E,k,zipf", [(100, 256, 256, 8, None), (300, 512, 32, 4, 1.1), (65, 2880, 128, 4, None)])
def test_router_many_tokens(api, T, H, E, k, zipf):
    """The many-token router (blocks of 32 tokens on the tensor cores): a partial last
    block, 256 experts (several column blocks per warp), 32 experts (idle warps), a bias."""
    inp = make_layer(T=T, H=H, I=64, E=E, k=k, seed=T + E, zipf_s=zipf)
    x, wr = to_dev(inp.x), to_dev(inp.w_router)
    bias = None if inp.router_bias is None else to_dev(inp.router_bias)
    lg, idx, w = api.route(x, wr, k, bias=bias)
    ref = oracle.router_logits(inp.x, inp.w_router, inp.router_bias)
    xa = np.abs(oracle.bf16_to_f32(inp.x)).astype(np.float64)
    wa = np.abs(oracle.bf16_to_f32(inp.w_router)).astype(np.float64)
    bound = inp.H * 2.0 ** -24 * (xa @ wa.T) + 1e-6
    assert np.all(np.abs(lg.cpu().numpy() - ref) <= bound)
    margin = oracle.topk_margin(ref, k)
    ok = margin > 1e-4
    ref_idx, _ = oracle.topk_softmax(ref, k)
    assert np.array_equal(idx.cpu().numpy()[ok], ref_idx[ok])
    assert ok.mean() > 0.8


CASES = [(4, 8, 2, 16, 0.0), (1, 32, 4, 16, 0.0), (64, 32, 4, 16, 0.0), (64, 128, 4, 16, 0.0),
         (4096, 128, 4, 128, 1.1), (4096, 128, 4, 64, 0.0), (777, 16, 2, 64, 1.5), (300, 1, 1, 128, 0.0),
         (50, 256, 8, 16, 0.7), (2048, 8, 8, 128, 0.0),
         # at most 32 assignments (the one-warp builder): at the limit, k = E, one expert, skewed
         (8, 256, 4, 16, 0.0), (32, 64, 1, 16, 1.5), (5, 3, 3, 16, 0.0), (3, 1, 1, 16, 0.0), (6, 200, 5, 64, 0.0),
         (33, 64, 1, 16, 0.0)]


@pytest.mark.parametrize("T,E,k,bm,skew", CASES)
def test_tile_table_bit_exact(api, T, E, k, bm, skew):
    idx = random_topk_idx(T, E, k, seed=T + E + k, skew=skew)
    got = api.build_tile_table(to_dev(idx), E, bm)
    ref = oracle.tile_table(idx, E, bm)
    for key in ("counts", "offsets", "perm", "inv_perm"):
        assert np.array_equal(got[key].cpu().numpy(), ref[key]), key
    n = int(got["num_tiles"].item())
    assert n == ref["num_tiles"]
    assert np.array_equal(got["tiles"].cpu().numpy()[:n], ref["tiles"])


def test_tile_table_policy_rows(api):
    for T, E, k in [(1, 32, 4), (64, 128, 4), (4096, 128, 4), (512, 32, 4)]:
        assert api.tile_rows(T, k, E) == oracle.tile_rows_policy(T, k, E)
        assert api.max_tiles(T, k, E, 16) == oracle.max_tiles_bound(T, k, E, 16)
