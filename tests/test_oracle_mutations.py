"""Deliberately broken oracles must fail the pins ("deliberately broken kernels fail
them", page "A 297-line kernel file that decodes faster than vLLM", section
"Correctness").  Every mistake is planted in a CPU copy of an oracle function."""

import numpy as np
import pytest

import oracle
from oracle import moe_oracle as mo
from synthetic import make_layer, random_topk_idx
from tests import oracle_checks as oc

_real_decode = mo.decode_mxfp4


def _decode_swapped_nibbles(codes, scales, dtype=np.float32):
    codes = np.asarray(codes, np.uint8)
    swapped = ((codes >> 4) | (codes << 4)).astype(np.uint8)
    return _real_decode(swapped, scales, dtype)


def _decode_no_scale(codes, scales, dtype=np.float32):
    return _real_decode(codes, np.full_like(np.asarray(scales), 127), dtype)


def _decode_scale_off_by_one(codes, scales, dtype=np.float32):
    return _real_decode(codes, np.asarray(scales) + 1, dtype) if np.max(scales) < 254 else \
        _real_decode(codes, np.minimum(np.asarray(scales), 253), dtype) * 2


def _topk_ties_to_high_index(logits, k, dtype=np.float32):
    lg = np.asarray(logits)
    T, E = lg.shape
    idx = np.empty((T, k), np.int32)
    for t in range(T):
        order = np.lexsort((-np.arange(E), -lg[t].astype(np.float64)))
        idx[t] = order[:k]
    sel = np.take_along_axis(lg, idx, 1).astype(dtype)
    ex = np.exp(sel - sel[:, :1])
    return idx, (ex / ex.sum(1, keepdims=True)).astype(dtype)


def _topk_softmax_over_all(logits, k, dtype=np.float32):
    idx, _ = mo.topk_softmax(logits, k, dtype)
    lg = np.asarray(logits, dtype)
    ex = np.exp(lg - lg.max(1, keepdims=True))
    p = ex / ex.sum(1, keepdims=True)
    return idx, np.take_along_axis(p, idx, 1).astype(dtype)


def _tile_table_unstable(idx, E, bm):
    res = mo.tile_table(idx, E, bm)
    perm = res["perm"].copy()
    for e in range(E):  # reverse order within each expert
        a, b = res["offsets"][e], res["offsets"][e + 1]
        perm[a:b] = perm[a:b][::-1]
    res["perm"] = perm
    res["inv_perm"][perm] = np.arange(perm.size, dtype=np.int32)
    return res


def _hidden_gate_up_swapped(x_rows, c, s, I, dtype=np.float32):
    w = mo.decode_mxfp4(c, s, dtype)
    g = np.asarray(x_rows, dtype) @ w[:I].T
    u = np.asarray(x_rows, dtype) @ w[I:2 * I].T
    return (mo.silu(u) * g).astype(dtype)


def _hidden_silu_sign(x_rows, c, s, I, dtype=np.float32):
    w = mo.decode_mxfp4(c, s, dtype)
    g = np.asarray(x_rows, dtype) @ w[:I].T
    u = np.asarray(x_rows, dtype) @ w[I:2 * I].T
    return (g / (1 + np.exp(g)) * u).astype(dtype)


def _output_transposed(h_rows, c, s, dtype=np.float32):
    w = mo.decode_mxfp4(c, s, dtype)
    return (np.asarray(h_rows, dtype) @ w).astype(dtype)


def test_broken_decoders_fail_enumeration():
    for bad in (_decode_swapped_nibbles, _decode_no_scale, _decode_scale_off_by_one):
        with pytest.raises(AssertionError):
            oc.check_decode_enumeration(bad, np.float32)


def test_broken_ffn_fails_brute_force():
    for hid, outp in ((_hidden_gate_up_swapped, mo.expert_output),
                      (_hidden_silu_sign, mo.expert_output),
                      (mo.expert_hidden, _output_transposed)):
        with pytest.raises(AssertionError):
            oc.check_brute_force(hid, outp, mo.bf16_to_f32, np.float64, 1e-12)


def test_broken_decoder_fails_brute_force(monkeypatch):
    monkeypatch.setattr(mo, "decode_mxfp4", _decode_swapped_nibbles)
    with pytest.raises(AssertionError):
        oc.check_brute_force(mo.expert_hidden, mo.expert_output, mo.bf16_to_f32, np.float64, 1e-12)


def test_broken_topk_fails():
    for bad in (_topk_ties_to_high_index, _topk_softmax_over_all):
        with pytest.raises(AssertionError):
            oc.check_topk(bad)


def test_unstable_tile_table_fails():
    idx = random_topk_idx(64, 32, 4, seed=2)
    with pytest.raises(AssertionError):
        oc.check_tile_table(_tile_table_unstable, [(idx, 32, 16)])


def test_skipped_slot_fails_identical_expert_invariant(monkeypatch):
    real = mo.topk_softmax

    def drop_last_slot(logits, k, dtype=np.float32):
        idx, w = real(logits, k, dtype)
        w = w.copy()
        w[:, -1] = 0
        return idx, w

    monkeypatch.setattr(mo, "topk_softmax", drop_last_slot)
    inp = make_layer(T=6, H=64, I=96, E=5, k=3, seed=7)
    for arr in (inp.gu_codes, inp.gu_scales, inp.dn_codes, inp.dn_scales):
        arr[:] = arr[0:1]
    with pytest.raises(AssertionError):
        oc.check_identical_experts(mo.moe_layer, mo.expert_hidden, mo.expert_output,
                                   mo.bf16_to_f32, inp, np.float64)


def test_truncating_bf16_fails_rounding_pin(monkeypatch):
    def trunc(a):
        return (np.ascontiguousarray(a, np.float32).view(np.uint32) & 0xFFFF0000).view(np.float32)

    vals = np.array([1.0 + 3 * 2 ** -8], dtype=np.float32)
    assert not np.array_equal(trunc(vals), oracle.bf16_round(vals))


# ---------------------------------------------------------------- RMSNorm + residual
def _norm_variant(kind):
    def f(x_bits, r_bits, gamma_bits, eps, dtype=np.float32):
        x = mo.bf16_to_f32(x_bits)
        r = mo.bf16_to_f32(r_bits)
        exact = (x + r).astype(np.float32)
        s = mo.bf16_round(exact)
        sn = (exact if kind == "unrounded_stream" else (x if kind == "dropped_residual" else s)).astype(dtype)
        gam = mo.bf16_to_f32(gamma_bits).astype(dtype)
        msq = np.sum(sn * sn, axis=-1, keepdims=True) if kind == "sum_not_mean" else \
            np.mean(sn * sn, axis=-1, keepdims=True)
        if kind == "eps_outside_root":
            y = sn / (np.sqrt(msq) + dtype(eps)) * gam
        elif kind == "no_weight":
            y = sn / np.sqrt(msq + dtype(eps))
        elif kind == "one_plus_weight":
            y = sn / np.sqrt(msq + dtype(eps)) * (1 + gam)
        else:
            y = sn / np.sqrt(msq + dtype(eps)) * gam
        return mo.bf16_bits(s), mo.bf16_bits(y.astype(np.float32))
    return f


@pytest.mark.parametrize("kind", ["dropped_residual", "sum_not_mean", "eps_outside_root", "no_weight",
                                  "one_plus_weight", "unrounded_stream"])
def test_broken_rmsnorm_fails_pins(monkeypatch, kind):
    from tests import test_oracle_pins as pins
    monkeypatch.setattr(oracle, "rmsnorm_residual", _norm_variant(kind))
    monkeypatch.setattr(mo, "rmsnorm_residual", _norm_variant(kind))
    failed = 0
    for pin in (lambda: pins.test_rmsnorm_residual_closed_forms(np.float64),
                pins.test_rmsnorm_residual_rounds_the_stream_once,
                pins.test_rmsnorm_residual_invariants,
                pins.test_rmsnorm_residual_against_high_precision):
        try:
            pin()
        except AssertionError:
            failed += 1
    assert failed > 0, kind


def test_unbroken_rmsnorm_variant_passes_pins(monkeypatch):
    # the harness itself: the faithful restatement passes every pin
    from tests import test_oracle_pins as pins
    monkeypatch.setattr(oracle, "rmsnorm_residual", _norm_variant("faithful"))
    pins.test_rmsnorm_residual_closed_forms(np.float64)
    pins.test_rmsnorm_residual_rounds_the_stream_once()
    pins.test_rmsnorm_residual_invariants()
    pins.test_rmsnorm_residual_against_high_precision()


# ---------------------------------------------------------------- bf16-weight experts
def _dense_hidden_swapped(x_rows, w_e, I, dtype=np.float32):
    w = mo.bf16_to_f32(w_e).astype(dtype)
    x_rows = np.asarray(x_rows, dtype)
    g, u = x_rows @ w[I:2 * I].T, x_rows @ w[:I].T
    return (mo.silu(g) * u).astype(dtype)


def _dense_hidden_no_silu(x_rows, w_e, I, dtype=np.float32):
    w = mo.bf16_to_f32(w_e).astype(dtype)
    x_rows = np.asarray(x_rows, dtype)
    return ((x_rows @ w[:I].T) * (x_rows @ w[I:2 * I].T)).astype(dtype)


def _dense_output_transposed(h_rows, w_e, dtype=np.float32):
    w = mo.bf16_to_f32(w_e).astype(dtype)
    return (np.asarray(h_rows, dtype) @ w).astype(dtype)


@pytest.mark.parametrize("name,fn", [("expert_hidden_dense", _dense_hidden_swapped),
                                     ("expert_hidden_dense", _dense_hidden_no_silu),
                                     ("expert_output_dense", _dense_output_transposed)])
def test_broken_dense_experts_fail_pins(monkeypatch, name, fn):
    from tests import test_oracle_pins as pins
    monkeypatch.setattr(mo, name, fn)
    failed = 0
    for pin in (lambda: pins.test_dense_layer_equals_mxfp4_layer_on_exactly_representable_weights(np.float32),
                pins.test_dense_layer_against_python_loops):
        try:
            pin()
        except AssertionError:
            failed += 1
    assert failed > 0, name


# ---------------------------------------------------------------- margin, router bias, tile policy
def _margin_off_by_one_low(logits, k):
    lg = np.sort(np.asarray(logits, np.float64), axis=1)[:, ::-1]
    if k >= lg.shape[1]:
        return np.full(lg.shape[0], np.inf)
    return lg[:, max(k - 2, 0)] - lg[:, k - 1]


def _margin_off_by_one_high(logits, k):
    lg = np.sort(np.asarray(logits, np.float64), axis=1)[:, ::-1]
    if k + 1 >= lg.shape[1]:
        return np.full(lg.shape[0], np.inf)
    return lg[:, k - 1] - lg[:, k + 1]


def _margin_no_inf(logits, k):
    lg = np.sort(np.asarray(logits, np.float64), axis=1)[:, ::-1]
    return lg[:, k - 1] - lg[:, min(k, lg.shape[1] - 1)]


@pytest.mark.parametrize("bad", [_margin_off_by_one_low, _margin_off_by_one_high, _margin_no_inf])
def test_broken_margin_fails_pin(bad):
    with pytest.raises(AssertionError):
        oc.check_topk_margin(bad)


def _logits_variant(kind):
    def f(x_bits, w_router_bits, bias=None, dtype=np.float32):
        x = mo.bf16_to_f32(x_bits).astype(dtype)
        w = mo.bf16_to_f32(w_router_bits).astype(dtype)
        lg = x @ w.T
        if bias is not None and kind != "dropped":
            b = np.asarray(bias, dtype)[None, :]
            lg = lg + (2 * b if kind == "twice" else (-b if kind == "negated" else b))
        if kind == "transposed_w":
            lg = (x @ w.reshape(w.shape[1], w.shape[0])).astype(dtype)
        return lg.astype(dtype)
    return f


@pytest.mark.parametrize("kind", ["dropped", "twice", "negated", "transposed_w"])
def test_broken_router_bias_fails_pin(kind):
    from synthetic import bf16_bits_from_f32
    with pytest.raises(AssertionError):
        oc.check_router_logits(_logits_variant(kind), bf16_bits_from_f32)


def test_faithful_router_variant_passes_pin():
    from synthetic import bf16_bits_from_f32
    oc.check_router_logits(_logits_variant("faithful"), bf16_bits_from_f32)


def _policy_strict(T, k, E):
    m = T * k / E
    return 16 if m < 16 else (64 if m < 64 else 128)


def _policy_no_middle(T, k, E):
    return 16 if T * k / E <= 16 else 128


@pytest.mark.parametrize("bad", [_policy_strict, _policy_no_middle])
def test_broken_tile_policy_fails_pin(bad):
    with pytest.raises(AssertionError):
        oc.check_tile_rows_policy(bad)
