"""Pins of the CPU oracle against things other than itself: the E2M1 format
definition and its printed table, exact rational brute force, brute-force sorting,
closed forms, invariants, and an independent library (torch CPU)."""

import numpy as np
import pytest

import oracle
from synthetic import make_layer, make_config, random_topk_idx
from tests import oracle_checks as oc


def test_e2m1_table_matches_format_definition_and_golden():
    gold = oc.golden_e2m1()
    assert sorted(gold) == list(range(16))
    for c in range(16):
        want = oc.e2m1_from_bitfields(c)
        assert float(gold[c]) == float(want)
        assert oracle.E2M1_VALUES[c] == float(want)
        if c == 8:
            assert gold[c].startswith("-") and str(oracle.E2M1_VALUES[c]) == "-0.0"


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_decode_all_codes_all_scales(dtype):
    oc.check_decode_enumeration(oracle.decode_mxfp4, dtype)


def test_e8m0_nan_scale_rejected():
    with pytest.raises(ValueError):
        oracle.decode_mxfp4(np.zeros((1, 16), np.uint8), np.full((1, 1), 255, np.uint8))


def test_nibble_order_reading():
    # byte 0x21: even K index = low nibble = code 1 (0.5), odd K index = code 2 (1.0)
    codes = np.zeros((1, 16), np.uint8)
    codes[0, 0] = 0x21
    v = oracle.decode_mxfp4(codes, np.full((1, 1), 127, np.uint8))
    assert v[0, 0] == 0.5 and v[0, 1] == 1.0 and np.all(v[0, 2:] == 0)


@pytest.mark.parametrize("dtype,rtol", [(np.float64, 1e-12), (np.float32, 2e-5)])
def test_brute_force_one_block(dtype, rtol):
    oc.check_brute_force(oracle.expert_hidden, oracle.expert_output, oracle.bf16_to_f32,
                         dtype, rtol)


def test_topk_against_full_sort_and_softmax_closed_form():
    oc.check_topk(oracle.topk_softmax)
    oc.check_topk(oracle.topk_softmax, T=17, E=128, k=4, seed=11)
    oc.check_topk(oracle.topk_softmax, T=5, E=8, k=8, seed=2)


def test_topk_single_expert_weight_is_one():
    lg = np.random.default_rng(0).standard_normal((9, 8)).astype(np.float32)
    idx, w = oracle.topk_softmax(lg, 1)
    assert np.all(idx[:, 0] == lg.argmax(1)) and np.all(w == 1)


def test_gating_variants_closed_forms():
    """Each gating variant against its closed form, evaluated one value at a time with
    the math module (not the oracle's vectorised expression), plus invariants."""
    import math
    rows = [[2.0, 1.0, 0.0, -1.0], [0.5, -0.25, 3.0, 3.0], [0.0, 0.0, 0.0, 0.0], [-4.0, 7.5, 1.25, -0.5]]
    lg = np.array(rows, np.float64)
    k = 2
    for gating in (oracle.GATING_SOFTMAX_TOPK, oracle.GATING_SOFTMAX_ALL, oracle.GATING_SIGMOID):
        idx, w = oracle.topk_gating(lg, k, gating, np.float64)
        for t, row in enumerate(rows):
            order = sorted(range(len(row)), key=lambda e: (-row[e], e))[:k]
            assert list(idx[t]) == order
            if gating == oracle.GATING_SOFTMAX_TOPK:
                z = sum(math.exp(row[e] - row[order[0]]) for e in order)
                want = [math.exp(row[e] - row[order[0]]) / z for e in order]
            elif gating == oracle.GATING_SOFTMAX_ALL:
                z = sum(math.exp(v - max(row)) for v in row)
                want = [math.exp(row[e] - max(row)) / z for e in order]
            else:
                sg = [1.0 / (1.0 + math.exp(-row[e])) for e in order]
                want = [v / sum(sg) for v in sg]
            np.testing.assert_allclose(w[t], want, rtol=1e-13)
    rng = np.random.default_rng(4)
    lg = rng.standard_normal((7, 6))
    # all experts selected: softmax over all = softmax over the selected
    i0, w0 = oracle.topk_gating(lg, 6, oracle.GATING_SOFTMAX_TOPK, np.float64)
    i1, w1 = oracle.topk_gating(lg, 6, oracle.GATING_SOFTMAX_ALL, np.float64)
    assert np.array_equal(i0, i1)
    np.testing.assert_allclose(w0, w1, rtol=1e-12)
    # the same selection in every variant; sigmoid weights sum to 1, softmax-over-all
    # weights of a strict subset to less than 1
    i2, w2 = oracle.topk_gating(lg, 3, oracle.GATING_SIGMOID, np.float64)
    i3, w3 = oracle.topk_gating(lg, 3, oracle.GATING_SOFTMAX_ALL, np.float64)
    assert np.array_equal(i2, oracle.topk_softmax(lg, 3, np.float64)[0]) and np.array_equal(i2, i3)
    np.testing.assert_allclose(w2.sum(1), 1.0, rtol=1e-12)
    assert np.all(w3.sum(1) < 1.0)
    # equal logits: sigmoid gating gives every selected expert 1/k
    _, w4 = oracle.topk_gating(np.zeros((2, 5)), 4, oracle.GATING_SIGMOID, np.float64)
    np.testing.assert_allclose(w4, 0.25, rtol=1e-15)


def test_topk_margin_against_full_sort():
    oc.check_topk_margin(oracle.topk_margin)
    oc.check_topk_margin(oracle.topk_margin, T=20, E=128, k=4, seed=9)
    oc.check_topk_margin(oracle.topk_margin, T=12, E=8, k=2, seed=10)


def test_router_logits_bias_closed_forms():
    from synthetic import bf16_bits_from_f32
    oc.check_router_logits(oracle.router_logits, bf16_bits_from_f32)


def test_tile_rows_policy_worked_values():
    oc.check_tile_rows_policy(oracle.tile_rows_policy)


def test_tile_table_brute_force_and_invariants():
    cases = []
    for (T, E, k, bm, skew, seed) in [(4, 8, 2, 16, 0, 0), (1, 32, 4, 16, 0, 1),
                                       (64, 32, 4, 16, 0, 2), (64, 128, 4, 16, 0, 3),
                                       (512, 128, 4, 64, 1.1, 4), (300, 16, 2, 128, 1.5, 5)]:
        cases.append((random_topk_idx(T, E, k, seed=seed, skew=skew), E, bm))
    # degenerate cases: one expert gets everything; an empty routing
    cases.append((np.zeros((40, 1), np.int32), 4, 16))
    cases.append((np.zeros((0, 2), np.int32), 4, 16))
    oc.check_tile_table(oracle.tile_table, cases)


def test_tile_bound_and_policy():
    for T, E, k in [(1, 32, 4), (64, 32, 4), (64, 128, 4), (4096, 128, 4), (4, 8, 2)]:
        bm = oracle.tile_rows_policy(T, k, E)
        assert bm in (16, 64, 128)
        for seed in range(3):
            idx = random_topk_idx(T, E, k, seed=seed, skew=1.1 if T > 1000 else 0)
            assert oracle.tile_table(idx, E, bm)["num_tiles"] <= oracle.max_tiles_bound(T, k, E, bm)
    assert oracle.tile_rows_policy(64, 4, 32) == 16
    assert oracle.tile_rows_policy(4096, 4, 128) == 128


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_identical_experts_make_output_independent_of_routing(dtype):
    inp = make_layer(T=6, H=64, I=96, E=5, k=3, seed=7)
    for arr in (inp.gu_codes, inp.gu_scales, inp.dn_codes, inp.dn_scales):
        arr[:] = arr[0:1]
    oc.check_identical_experts(oracle.moe_layer, oracle.expert_hidden, oracle.expert_output,
                               oracle.bf16_to_f32, inp, dtype)


def test_single_expert_layer_is_dense_ffn_by_loops():
    inp = make_layer(T=2, H=32, I=64, E=1, k=1, seed=9)
    ref = oc.dense_reference_loops(inp)
    res = oracle.moe_layer(inp, dtype=np.float64)
    assert np.allclose(res["out_unrounded"], ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    assert np.all(res["w"] == 1.0)


def test_weighted_combine_order_and_bf16_rounding():
    inp = make_config("tiny")
    res = oracle.moe_layer(inp, dtype=np.float64)
    acc = sum(res["w"][:, j:j + 1] * res["y"][:, j] for j in range(inp.k))
    assert np.allclose(res["out_unrounded"], acc, rtol=0, atol=1e-12 * np.abs(acc).max())
    # bf16 rounding: at most half an ulp of bf16 (2^-8 relative) and exact bf16 values
    r = oracle.bf16_round(acc.astype(np.float32))
    assert np.all((r.view(np.uint32) & 0xFFFF) == 0)
    assert np.all(np.abs(r - acc) <= np.abs(acc) * 2.0 ** -8 + 1e-30)


def test_bf16_round_ties_to_even():
    vals = np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8, 1.0 + 2 ** -8 + 2 ** -20],
                    dtype=np.float32)
    want = np.array([1.0, 1.0 + 2 ** -6, -1.0, 1.0 + 2 ** -7], dtype=np.float32)
    assert np.array_equal(oracle.bf16_round(vals), want)


def test_layer_matches_torch_cpu_library_path():
    torch = pytest.importorskip("torch")
    inp = make_config("tiny")
    res = oracle.moe_layer(inp, dtype=np.float32, return_hidden=True)
    x = torch.from_numpy(oracle.bf16_to_f32(inp.x))
    wr = torch.from_numpy(oracle.bf16_to_f32(inp.w_router))
    lg = x @ wr.T
    top = torch.topk(lg, inp.k, dim=1)
    w = torch.softmax(top.values, dim=1)
    out = torch.zeros(inp.T, inp.H)
    for t in range(inp.T):
        for j in range(inp.k):
            e = int(top.indices[t, j])
            wgu = torch.from_numpy(oracle.decode_mxfp4(inp.gu_codes[e], inp.gu_scales[e]))
            wd = torch.from_numpy(oracle.decode_mxfp4(inp.dn_codes[e], inp.dn_scales[e]))
            g = wgu[:inp.I] @ x[t]
            u = wgu[inp.I:] @ x[t]
            out[t] += w[t, j] * (wd @ (torch.nn.functional.silu(g) * u))
    assert np.array_equal(top.indices.numpy(), res["idx"])
    ref = out.numpy()
    assert np.abs(res["out_unrounded"] - ref).max() <= 1e-5 * np.abs(ref).max()


def _f(bits):
    return oracle.bf16_to_f32(bits)


def _b(vals):
    return oracle.bf16_bits(np.asarray(vals, dtype=np.float32))


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_rmsnorm_residual_closed_forms(dtype):
    # s = (1 + 2, 4 + 0) = (3, 4): mean square 12.5; y = (3, 4) / sqrt(12.5), rounded by
    # hand to bf16: 0.848528 -> 217 * 2^-8, 1.131371 -> 145 * 2^-7
    s, y = oracle.rmsnorm_residual(_b([[1, 4]]), _b([[2, 0]]), _b([1, 1]), 0.0, dtype)
    assert np.array_equal(_f(s), np.array([[3.0, 4.0]], np.float32))
    assert np.array_equal(_f(y), np.array([[217 * 2.0 ** -8, 145 * 2.0 ** -7]], np.float32))
    # eps inside the root: 12.5 + 3.5 = 16 -> (0.75, 1), and the weight multiplies
    _, y = oracle.rmsnorm_residual(_b([[3, 4]]), _b([[0, 0]]), _b([1, -2]), 3.5, dtype)
    assert np.array_equal(_f(y), np.array([[0.75, -2.0]], np.float32))
    # a row of +-c has rms c: y is the sign times the weight, whatever c (eps 0)
    g = _b(np.linspace(-1.5, 1.5, 64))
    for c in (3.0, 0.375, 96.0):
        row = np.where(np.arange(64) % 2 == 0, c, -c)
        _, y = oracle.rmsnorm_residual(_b(row[None]), _b(np.zeros((1, 64))), g, 0.0, dtype)
        assert np.array_equal(_f(y)[0], np.sign(row) * _f(g))
    # a zero row with eps > 0 normalises to zeros
    _, y = oracle.rmsnorm_residual(_b(np.zeros((1, 8))), _b(np.zeros((1, 8))), _b(np.ones(8)), 1e-5, dtype)
    assert np.array_equal(_f(y), np.zeros((1, 8), np.float32))


def test_rmsnorm_residual_rounds_the_stream_once():
    # 1 + 2^-9 is a quarter bf16 ulp above 1 (rounds down), 1 + 3 * 2^-9 three
    # quarters (rounds up to 1 + 2^-7): the sum is held in bf16 before the norm
    s, _ = oracle.rmsnorm_residual(_b([[1.0, 1.0]]), _b([[2.0 ** -9, 3 * 2.0 ** -9]]), _b([1, 1]), 0.0)
    assert np.array_equal(_f(s), np.array([[1.0, 1.0 + 2.0 ** -7]], np.float32))


def test_rmsnorm_residual_invariants():
    from synthetic import make_norm_inputs
    inp = make_layer(T=16, H=384, I=64, E=4, k=2, seed=5)
    r, g, _ = make_norm_inputs(16, 384, seed=5)
    s, y = oracle.rmsnorm_residual(inp.x, r, g, 0.0, np.float64)
    # unit weight: every row has mean square 1 up to bf16 rounding
    _, y1 = oracle.rmsnorm_residual(inp.x, r, _b(np.ones(384)), 0.0, np.float64)
    ms = np.mean(_f(y1).astype(np.float64) ** 2, axis=1)
    assert np.all(np.abs(ms - 1.0) < 4e-3)
    # scaling the stream by a power of two changes nothing (eps 0), and x and the
    # residual enter only through their sum
    s2, y2 = oracle.rmsnorm_residual(_b(_f(inp.x) * 8), _b(_f(r) * 8), g, 0.0, np.float64)
    assert np.array_equal(y2, y) and np.array_equal(_f(s2), _f(s) * 8)
    s3, y3 = oracle.rmsnorm_residual(r, inp.x, g, 0.0, np.float64)
    assert np.array_equal(s3, s) and np.array_equal(y3, y)


def test_layer_norm_is_scale_free_and_routes_on_the_normalised_rows():
    from synthetic import make_norm_inputs
    inp = make_config("tiny")
    r, g, _ = make_norm_inputs(inp.T, inp.H, seed=3)
    a = oracle.moe_layer_norm(inp, r, g, 0.0)
    import dataclasses
    b = oracle.moe_layer_norm(dataclasses.replace(inp, x=_b(_f(inp.x) * 4)), _b(_f(r) * 4), g, 0.0)
    assert np.array_equal(a["out"], b["out"]) and np.array_equal(a["idx"], b["idx"])
    assert np.array_equal(_f(b["residual_out"]), _f(a["residual_out"]) * 4)
    # the router sees y: its logits are y @ W_r^T
    lg = _f(a["x_norm"]).astype(np.float64) @ _f(inp.w_router).astype(np.float64).T
    assert np.allclose(a["logits"], lg, rtol=1e-5, atol=1e-5)


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_dense_layer_equals_mxfp4_layer_on_exactly_representable_weights(dtype):
    # E2M1 values times a power of two have at most two significant bits, so the
    # decoded MXFP4 weights are exact in bf16: the bf16-weight layer on those weights
    # must reproduce the (separately pinned) MXFP4 layer bit for bit
    from synthetic import DenseLayerInputs
    inp = make_config("tiny")
    wgu = np.stack([oracle.decode_mxfp4(inp.gu_codes[e], inp.gu_scales[e]) for e in range(inp.E)])
    wd = np.stack([oracle.decode_mxfp4(inp.dn_codes[e], inp.dn_scales[e]) for e in range(inp.E)])
    assert np.array_equal(oracle.bf16_round(wgu), wgu) and np.array_equal(oracle.bf16_round(wd), wd)
    dense = DenseLayerInputs("tiny_dense", inp.T, inp.H, inp.I, inp.E, inp.k, inp.x, inp.w_router,
                             oracle.bf16_bits(wgu), oracle.bf16_bits(wd))
    a = oracle.moe_layer(inp, dtype=dtype)
    b = oracle.moe_layer_dense(dense, dtype=dtype)
    for key in ("idx", "w", "y", "out"):
        assert np.array_equal(a[key], b[key]), key


def test_dense_layer_against_python_loops():
    from synthetic import make_dense_layer
    inp = make_dense_layer(T=3, H=8, I=8, E=2, k=1, seed=4, w_std=0.5)
    res = oracle.moe_layer_dense(inp, dtype=np.float64)
    x = oracle.bf16_to_f32(inp.x).astype(np.float64)
    wr = oracle.bf16_to_f32(inp.w_router).astype(np.float64)
    wgu = oracle.bf16_to_f32(inp.w_gateup).astype(np.float64)
    wd = oracle.bf16_to_f32(inp.w_down).astype(np.float64)
    for t in range(inp.T):
        logits = [sum(x[t, i] * wr[e, i] for i in range(inp.H)) for e in range(inp.E)]
        e = max(range(inp.E), key=lambda q: (logits[q], -q))
        h = []
        for f in range(inp.I):
            g = sum(x[t, i] * wgu[e, f, i] for i in range(inp.H))
            u = sum(x[t, i] * wgu[e, inp.I + f, i] for i in range(inp.H))
            h.append(g / (1.0 + np.exp(-g)) * u)
        y = [sum(h[f] * wd[e, o, f] for f in range(inp.I)) for o in range(inp.H)]
        assert res["idx"][t, 0] == e
        assert np.allclose(res["out_unrounded"][t], y, rtol=1e-12, atol=1e-12)


def test_rmsnorm_residual_against_high_precision():
    # y recomputed from the definition in 40-digit decimal arithmetic: the sum of two
    # bf16 values is exact in a double, rounded to bf16 (the stream), the mean square
    # is exact as a fraction, and the root and quotient are taken to 40 digits; y is then
    # rounded once to bf16.  The oracle must agree bit for bit.
    from decimal import Decimal, getcontext
    from fractions import Fraction
    getcontext().prec = 40
    rng = np.random.Generator(np.random.PCG64(21))
    T, H = 24, 16
    x = oracle.bf16_bits(rng.standard_normal((T, H)).astype(np.float32) * 3)
    r = oracle.bf16_bits((rng.standard_normal((T, H)) * np.exp2(rng.integers(-9, 2, (T, H)))).astype(np.float32))
    g = oracle.bf16_bits((1 + 0.3 * rng.standard_normal(H)).astype(np.float32))
    eps = 1e-5
    s_bits, y_bits = oracle.rmsnorm_residual(x, r, g, eps, np.float64)
    xf, rf, gf = _f(x).astype(np.float64), _f(r).astype(np.float64), _f(g).astype(np.float64)
    s = oracle.bf16_round((xf + rf).astype(np.float32))  # x + r is exact in a double
    assert np.array_equal(_f(s_bits), s)
    for t in range(T):
        ms = sum(Fraction(float(v)) ** 2 for v in s[t]) / H + Fraction(eps)
        root = (Decimal(ms.numerator) / Decimal(ms.denominator)).sqrt()
        want = [float(Decimal(float(s[t, i])) / root * Decimal(float(gf[i]))) for i in range(H)]
        assert np.array_equal(_f(y_bits[t]), oracle.bf16_round(np.array(want, np.float32))), t
