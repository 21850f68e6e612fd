"""GPU parity of the MXFP4 expert path: the one-time weight re-layout (byte
exact), the gate/up + SwiGLU output h, and the whole layer against the oracle on
the five gpt-oss-shaped workloads plus ragged and degenerate shapes."""

import math

import numpy as np
import pytest

import oracle
from synthetic import make_config, make_layer, make_norm_inputs
from tests.gpu_helpers import (TOL_MAX_ABS, TOL_REL_FROB, bf16_bits_to_f32, bf16_to_np, build_layer, errors,
                               logit_band, tile_edge_tokens, to_dev)

pytestmark = pytest.mark.gpu


def expected_prepared(codes: np.ndarray, scales: np.ndarray, groups: int) -> np.ndarray:
    """The documented prepared layout, restated: the codes unchanged (row major
    [E][G * rows per group][K/2]), then (256-aligned) scale atoms
    [E][G][MT][KG][32 l][4 c][4 b] = scale of row 32c + l of the M tile, MX block
    4*kg + b (127 outside the matrix), KG = K groups of 128 rounded up to even, then a
    256-byte status trailer."""
    E, R, half = codes.shape
    K = half * 2
    rpg = R // groups
    MT = math.ceil(rpg / 128)
    KG = math.ceil(K / 256) * 2
    cp = codes
    sc = np.full((E, groups, MT, KG, 32, 4, 4), 127, np.uint8)
    blocks = K // 32
    for mt in range(MT):
        for c in range(4):
            for l in range(32):
                row = mt * 128 + 32 * c + l
                if row >= rpg:
                    continue
                for g in range(groups):
                    src = scales[:, g * rpg + row, :]  # [E, blocks]
                    for kg in range(KG):
                        for b in range(4):
                            blk = kg * 4 + b
                            if blk < blocks:
                                sc[:, g, mt, kg, l, c, b] = src[:, blk]
    codes_bytes = cp.size
    scales_off = (codes_bytes + 255) // 256 * 256
    total = (scales_off + sc.size + 255) // 256 * 256 + 256
    out = np.zeros(total, np.uint8)
    out[:codes_bytes] = np.ascontiguousarray(cp).reshape(-1)
    out[scales_off:scales_off + sc.size] = sc.reshape(-1)
    return out, scales_off + sc.size


@pytest.mark.parametrize("E,I,H", [(8, 256, 256), (3, 96, 160), (2, 2880, 2880)])
def test_prepare_weights_byte_exact(E, I, H):
    import mxfp4_expert_layer_gb300 as pkg
    from mxfp4_expert_layer_gb300 import _lib as L
    pkg.build()
    inp = make_layer(T=1, H=H, I=I, E=E, k=1, seed=11)
    for codes, scales, kind, groups in ((inp.gu_codes, inp.gu_scales, L.MOE_WEIGHTS_GATEUP, 2),
                                        (inp.dn_codes, inp.dn_scales, L.MOE_WEIGHTS_DOWN, 1)):
        got = pkg.prepare_weights(to_dev(codes), to_dev(scales), kind).cpu().numpy()
        want, used = expected_prepared(codes, scales, groups)
        assert got.size == want.size
        assert np.array_equal(got[:used], want[:used])


def test_prepare_rejects_nan_scale():
    import mxfp4_expert_layer_gb300 as pkg
    from mxfp4_expert_layer_gb300 import _lib as L
    pkg.build()
    inp = make_layer(T=1, H=64, I=64, E=2, k=1, seed=1)
    sc = inp.gu_scales.copy()
    sc[1, 5, 1] = 255
    with pytest.raises(L.MoEError) as ei:
        pkg.prepare_weights(to_dev(inp.gu_codes), to_dev(sc), L.MOE_WEIGHTS_GATEUP)
    assert ei.value.status == L.MOE_ERR_NAN_SCALE


def run_layer(inp, tokens=None, gating=0):
    import torch
    layer = build_layer(inp)
    x = to_dev(inp.x)
    idx = torch.empty(inp.T, inp.k, dtype=torch.int32, device="cuda")
    w = torch.empty(inp.T, inp.k, dtype=torch.float32, device="cuda")
    out = layer(x, topk_idx=idx, topk_w=w, gating=gating)
    torch.cuda.synchronize()
    assert layer.device_status(inp.T) == 0
    return layer, bf16_bits_to_f32(bf16_to_np(out)), idx.cpu().numpy(), w.cpu().numpy()


GATING_OF_FLAG = {0: 0, 2: 1, 4: 2}  # MOE_ROUTE_GATING_* flag -> oracle gating variant


def check_layer(inp, tokens=None, gating=0, band=None, min_kept=0.9):
    """The layer's output and routing against the oracle on `tokens` (default all).
    Tokens whose oracle top-k margin lies inside the near-tie band are left out of
    the comparison; the band comes from the router logit error measured on this
    input (gpu_helpers.logit_band) unless one is given."""
    layer, out, idx, w = run_layer(inp, gating=gating)
    ref = oracle.moe_layer(inp, tokens=tokens, gating=GATING_OF_FLAG[gating])
    tok = ref["tokens"]
    if band is None:
        band, _ = logit_band(inp)
    keep = oracle.topk_margin(ref["logits"], inp.k) > band
    assert keep.mean() >= min_kept, (keep.mean(), band)
    assert np.array_equal(idx[tok][keep], ref["idx"][keep])
    rel, mx = errors(out[tok][keep], ref["out"][keep])
    assert rel <= TOL_REL_FROB and mx <= TOL_MAX_ABS, (rel, mx)
    return rel, mx, idx


def test_layer_tiny():
    check_layer(make_config("tiny"))


@pytest.mark.parametrize("name,gating", [("tiny", 2), ("tiny", 4), ("gptoss20b_b1", 4), ("gptoss20b_b64", 2)])
def test_layer_gating_variants(name, gating):
    """moe_forward_gated: softmax over all experts (flag 2) and normalised sigmoid (4)."""
    check_layer(make_config(name), gating=gating)


def test_layer_gptoss20b_b1():
    check_layer(make_config("gptoss20b_b1"))


def test_layer_gptoss20b_b64():
    check_layer(make_config("gptoss20b_b64"))


def test_layer_gptoss120b_b1():
    check_layer(make_config("gptoss120b_b1"))


def test_layer_gptoss120b_b64():
    check_layer(make_config("gptoss120b_b64"))


def test_layer_gptoss120b_prefill4096_every_tile():
    """4096 tokens with the Zipf router bias: the oracle checks the tokens at the
    first and the last row of every tile the GPU's routing produced (hot experts'
    full 128-row tiles and every partial last tile), plus a random sample."""
    inp = make_config("gptoss120b_prefill4096")
    layer, out, idx, w = run_layer(inp)
    bm = oracle.tile_rows_policy(inp.T, inp.k, inp.E)
    tab = oracle.tile_table(idx, inp.E, bm)
    assert tab["num_tiles"] > inp.E // 2 and np.max(tab["counts"]) > 4 * bm  # skewed: several hot experts
    tokens = np.union1d(tile_edge_tokens(idx, inp.E, bm), np.random.default_rng(0).choice(inp.T, 32, replace=False))
    ref = oracle.moe_layer(inp, tokens=tokens)
    band, _ = logit_band(inp)
    keep = oracle.topk_margin(ref["logits"], inp.k) > band
    assert keep.mean() >= 0.9, (keep.mean(), band)
    assert np.array_equal(idx[tokens][keep], ref["idx"][keep])
    # every tile keeps at least one compared token at one of its edges
    kept = set(tokens[keep].tolist())
    for e, s0, n, _ in tab["tiles"]:
        edge = {int(tab["perm"][s0]) // inp.k, int(tab["perm"][s0 + n - 1]) // inp.k}
        assert edge & kept, (e, s0, n)
    rel, mx = errors(out[tokens][keep], ref["out"][keep])
    assert rel <= TOL_REL_FROB and mx <= TOL_MAX_ABS, (rel, mx)


def with_outliers(inp, factors=(100.0, 1000.0), fixed_channels=False, seed=0):
    """x with a heavy tail: in every 32-value block of every row, one element scaled
    by each of `factors` -- at random positions, or (fixed_channels) at the same
    channels for every token, as massive activations sit in fixed channels."""
    import dataclasses
    from synthetic import bf16_bits_from_f32
    rng = np.random.default_rng(seed)
    x = oracle.bf16_to_f32(inp.x).copy()
    T, H = x.shape
    for b in range(H // 32):
        fixed = rng.choice(32, len(factors), replace=False)
        for t in range(T):
            pos = fixed if fixed_channels else rng.choice(32, len(factors), replace=False)
            for f, q in zip(factors, pos):
                x[t, b * 32 + q] *= f
    return dataclasses.replace(inp, x=bf16_bits_from_f32(x))


@pytest.mark.parametrize("name", ["tiny", "gptoss20b_b64"])
@pytest.mark.parametrize("fixed", [False, True], ids=["random_positions", "fixed_channels"])
def test_layer_heavy_tailed_activations(name, fixed):
    """One x100 and one x1000 element in every 32-value block.  Each E2M1 term of the
    activation encoding is scaled to its block's largest residual, so the other values
    of such a block keep less relative precision (about 1e-2 of their block's
    non-outlier maximum after four terms, against about 1e-4 without outliers); with
    the expert weights as drawn the outliers dominate every dot product and the layer
    stays within the tolerance."""
    rel, mx, _ = check_layer(with_outliers(make_config(name), fixed_channels=fixed))
    print(f"{name} heavy-tailed x ({'fixed channels' if fixed else 'random positions'}): rel {rel:.2e} max {mx:.2e}")


@pytest.mark.parametrize("T,H,I,E,k", [(200, 256, 256, 16, 2),    # 64-row tiles, ragged tails
                                       (1000, 256, 512, 8, 2),    # 128-row tiles
                                       (13, 160, 96, 3, 3),       # k = E, I < one M tile, K tails
                                       (5, 64, 64, 1, 1),         # one expert: dense FFN
                                       (33, 2880, 2880, 4, 1)])   # gpt-oss widths, K = 22.5 groups
def test_layer_ragged_and_degenerate(T, H, I, E, k):
    check_layer(make_layer(T, H, I, E, k, seed=T + E))


def test_hidden_matches_oracle():
    import torch
    from mxfp4_expert_layer_gb300 import _lib as L
    inp = make_config("gptoss20b_b64")
    layer = build_layer(inp)
    T, H, I, E, k = inp.T, inp.H, inp.I, inp.E, inp.k
    x = to_dev(inp.x)
    # identical routing on both sides: route on the oracle's logits
    ref_lg = oracle.router_logits(inp.x, inp.w_router)
    _, idx, w = __import__("mxfp4_expert_layer_gb300").route(None, None, k, logits=to_dev(ref_lg),
                                                               from_logits=True)
    tab = __import__("mxfp4_expert_layer_gb300").build_tile_table(idx, E)
    ws = layer.workspace(T)
    st = L.moe_mxfp4_gateup_swiglu(x.data_ptr(), tab["perm"].data_ptr(), tab["tiles"].data_ptr(),
                                   tab["num_tiles"].data_ptr(), 0, layer.w_gateup.data_ptr(), T, H, I, E, k,
                                   ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream)
    assert st == 0
    h = torch.zeros(T * k, I, dtype=torch.float32, device="cuda")
    st = L.moe_hidden_dequant(tab["perm"].data_ptr(), tab["tiles"].data_ptr(), tab["num_tiles"].data_ptr(), 0, T,
                              H, I, E, k, ws.data_ptr(), ws.numel(), h.data_ptr(),
                              torch.cuda.current_stream().cuda_stream)
    assert st == 0
    out = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    st = L.moe_mxfp4_down_combine(tab["perm"].data_ptr(), tab["tiles"].data_ptr(), tab["num_tiles"].data_ptr(), 0,
                                  w.data_ptr(), layer.w_down.data_ptr(), T, H, I, E, k, ws.data_ptr(), ws.numel(),
                                  out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    ref = oracle.moe_layer(inp, logits=ref_lg, return_hidden=True)
    assert np.array_equal(idx.cpu().numpy(), ref["idx"])
    rel_h, mx_h = errors(h.cpu().numpy().reshape(T, k, I), ref["h"])
    assert rel_h <= 3e-3, (rel_h, mx_h)
    rel, mx = errors(bf16_bits_to_f32(bf16_to_np(out)), ref["out"])
    assert rel <= TOL_REL_FROB and mx <= TOL_MAX_ABS, (rel, mx)


def test_layer_is_bit_reproducible():
    import torch
    inp = make_config("gptoss20b_b64")
    layer = build_layer(inp)
    x = to_dev(inp.x)
    a = layer(x).clone()
    b = layer(x).clone()
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("name", ["gptoss20b_b1", "gptoss20b_b64"])
def test_consecutive_calls_with_new_routing(name):
    """Calls back to back on one workspace with different tokens (so a different
    routing and tile table each time) each match the oracle: no launch may read a
    routing result, an encoded row or a counter left over from the call before."""
    import dataclasses
    import torch
    from synthetic.gen import bf16_bits_from_f32
    base = make_config(name)
    layer = build_layer(base)
    outs, inps = [], []
    for s in range(4):
        rng = np.random.default_rng(100 + s)
        x = bf16_bits_from_f32(rng.standard_normal((base.T, base.H), dtype=np.float32))
        inp = dataclasses.replace(base, x=x)
        inps.append(inp)
        outs.append(layer(to_dev(x)).clone())
    torch.cuda.synchronize()
    assert layer.device_status(base.T) == 0
    for inp, out in zip(inps, outs):
        ref = oracle.moe_layer(inp)
        keep = oracle.topk_margin(ref["logits"], inp.k) > logit_band(inp)[0]
        rel, mx = errors(bf16_bits_to_f32(bf16_to_np(out))[keep], ref["out"][keep])
        assert rel <= TOL_REL_FROB and mx <= TOL_MAX_ABS, (rel, mx)


@pytest.mark.parametrize("name,T", [("tiny", None), ("gptoss20b_b1", None), ("gptoss20b_b64", None),
                                    ("gptoss20b_b64", 200), ("gptoss20b_b64", 512)])
def test_layer_norm_residual(name, T):
    """RMSNorm + residual in front of the layer: the router (cluster kernel for T <= 64,
    many-token kernel above) and the encoder normalise the rows themselves; the
    combine kernel writes the residual stream."""
    import torch
    inp = make_config(name, T=T)
    r, g, eps = make_norm_inputs(inp.T, inp.H, seed=1)
    layer = build_layer(inp)
    x, rd, gd = to_dev(inp.x), to_dev(r), to_dev(g)
    idx = torch.empty(inp.T, inp.k, dtype=torch.int32, device="cuda")
    w = torch.empty(inp.T, inp.k, dtype=torch.float32, device="cuda")
    res_out = torch.empty_like(x)
    out = layer(x, topk_idx=idx, topk_w=w, residual=rd, norm_weight=gd, eps=eps, residual_out=res_out)
    torch.cuda.synchronize()
    assert layer.device_status(inp.T) == 0
    ref = oracle.moe_layer_norm(inp, r, g, eps)
    assert np.array_equal(bf16_to_np(res_out), ref["residual_out"])
    got = bf16_bits_to_f32(bf16_to_np(out))
    # the router's input is y: the band comes from the router error measured on the oracle's y
    keep = oracle.topk_margin(ref["logits"], inp.k) > logit_band(inp, x_bits=ref["x_norm"])[0]
    assert keep.mean() > 0.9
    assert np.array_equal(idx.cpu().numpy()[keep], ref["idx"][keep])
    rel, mx = errors(got[keep], ref["out"][keep])
    assert rel <= TOL_REL_FROB and mx <= TOL_MAX_ABS, (rel, mx)
    # in place: the residual stream written over the residual input, same results
    rd2 = rd.clone()
    out2 = layer(x, residual=rd2, norm_weight=gd, eps=eps, residual_out=rd2)
    torch.cuda.synchronize()
    assert torch.equal(out2, out) and torch.equal(rd2, res_out)
