"""Independent checks that pin the CPU oracle to the format definition, to brute
force and to closed forms.  Each check takes the oracle functions it tests as
arguments, so the mutation tests can hand it a deliberately broken variant and
confirm the check rejects it."""

from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------- format values
def e2m1_from_bitfields(code: int) -> Fraction:
    """E2M1 value from its bit fields (OCP MX v1.0, FP4 E2M1): sign bit 3, exponent
    bits 2..1 with bias 1, mantissa bit 0; exponent 0 is subnormal (0.m * 2^0)."""
    sign = -1 if (code >> 3) & 1 else 1
    e = (code >> 1) & 3
    m = code & 1
    if e == 0:
        mag = Fraction(m, 2)
    else:
        mag = (1 + Fraction(m, 2)) * Fraction(2) ** (e - 1)
    return sign * mag


def golden_e2m1():
    vals = {}
    with open(os.path.join(GOLDEN, "e2m1_ocp_mx_v1.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            c, v = line.split()
            vals[int(c)] = v
    return vals


def check_decode_enumeration(decode_mxfp4, dtype):
    """All 16 codes x every finite E8M0 scale (0..254) decode exactly to
    E2M1(code) * 2^(s-127), with the even K index taken from the low nibble."""
    codes = np.arange(16, dtype=np.uint8)
    # one row per scale: 32 elements = codes 0..15 then codes 15..0 so both nibbles
    # of a byte differ (even index low nibble, odd index high nibble)
    elems = np.concatenate([codes, codes[::-1]])
    packed = (elems[0::2] | (elems[1::2] << 4)).astype(np.uint8)
    scales = np.arange(255, dtype=np.uint8)
    rows_codes = np.tile(packed, (scales.size, 1))
    rows_scales = scales.reshape(-1, 1)
    got = decode_mxfp4(rows_codes, rows_scales, dtype)
    assert got.shape == (255, 32)
    for s in range(255):
        p2 = Fraction(2) ** (s - 127)
        for i, c in enumerate(elems):
            want = e2m1_from_bitfields(int(c)) * p2
            g = got[s, i]
            if abs(want) > Fraction(float(np.finfo(dtype).max)):
                # beyond the working precision's range (only scales >= 253 in float32)
                assert np.isinf(g) and (g > 0) == (want > 0), (s, i, g)
                continue
            assert Fraction(float(g)) == want, (s, i, int(c), g, want)
            if c == 8:
                assert math.copysign(1.0, float(g)) == -1.0, "code 8 is -0"


# ------------------------------------------------------------- brute force layer
def _exact_dot(a, b):
    return sum((Fraction(float(p)) * Fraction(float(q)) for p, q in zip(a, b)), Fraction(0))


def brute_force_single_token(seed=3, H=32, I=32):
    """1 token, 1 expert, k = 1, H = I = 32 (one MX block): g and u in exact
    rational arithmetic, silu in float64, y again exact given h."""
    rng = np.random.Generator(np.random.PCG64(seed))
    x_bits = (rng.standard_normal((1, H)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    gu_codes = rng.integers(0, 256, size=(1, 2 * I, H // 2), dtype=np.uint8)
    gu_scales = rng.integers(122, 127, size=(1, 2 * I, H // 32), dtype=np.uint8)
    dn_codes = rng.integers(0, 256, size=(1, H, I // 2), dtype=np.uint8)
    dn_scales = rng.integers(122, 127, size=(1, H, I // 32), dtype=np.uint8)

    def dec_row(codes_row, scales_row):
        out = []
        for kk in range(codes_row.size * 2):
            byte = int(codes_row[kk // 2])
            c = byte & 0xF if kk % 2 == 0 else byte >> 4
            out.append(e2m1_from_bitfields(c) * Fraction(2) ** (int(scales_row[kk // 32]) - 127))
        return out

    x = [Fraction(float(v)) for v in (x_bits[0].astype(np.uint32) << 16).view(np.float32)]
    h = []
    for i in range(I):
        wg = dec_row(gu_codes[0, i], gu_scales[0, i])
        wu = dec_row(gu_codes[0, I + i], gu_scales[0, I + i])
        g = sum((a * b for a, b in zip(x, wg)), Fraction(0))
        u = sum((a * b for a, b in zip(x, wu)), Fraction(0))
        gf = float(g)
        h.append(gf / (1.0 + math.exp(-gf)) * float(u))
    y = []
    for n in range(H):
        wd = dec_row(dn_codes[0, n], dn_scales[0, n])
        y.append(float(sum((Fraction(hv) * b for hv, b in zip(h, wd)), Fraction(0))))
    return {"x": x_bits, "gu_codes": gu_codes, "gu_scales": gu_scales, "dn_codes": dn_codes,
            "dn_scales": dn_scales, "h": np.array(h), "y": np.array(y)}


def check_brute_force(expert_hidden, expert_output, bf16_to_f32, dtype, rtol):
    bf = brute_force_single_token()
    I = bf["h"].size
    x = bf16_to_f32(bf["x"]).astype(dtype)
    h = expert_hidden(x, bf["gu_codes"][0], bf["gu_scales"][0], I, dtype)
    y = expert_output(h, bf["dn_codes"][0], bf["dn_scales"][0], dtype)
    scale_h = np.abs(bf["h"]).max()
    scale_y = np.abs(bf["y"]).max()
    assert np.abs(h[0] - bf["h"]).max() <= rtol * scale_h, np.abs(h[0] - bf["h"]).max() / scale_h
    assert np.abs(y[0] - bf["y"]).max() <= rtol * scale_y, np.abs(y[0] - bf["y"]).max() / scale_y


# ------------------------------------------------------------------- routing
def brute_topk(row, k):
    """Top-k by full sort of (value descending, index ascending) pairs."""
    pairs = sorted(((-float(v), e) for e, v in enumerate(row)))
    return [e for _, e in pairs[:k]]


def check_topk(topk_softmax, T=64, E=16, k=4, seed=5):
    rng = np.random.Generator(np.random.PCG64(seed))
    lg = rng.standard_normal((T, E)).astype(np.float32)
    # plant exact ties, including ties straddling the k-th position
    for t in range(0, T, 3):
        a, b = rng.choice(E, 2, replace=False)
        lg[t, b] = lg[t, a]
    for t in range(1, T if k < E else 0, 7):
        srt = np.argsort(-lg[t], kind="stable")
        lg[t, srt[k]] = lg[t, srt[k - 1]]
    idx, w = topk_softmax(lg, k)
    for t in range(T):
        assert list(idx[t]) == brute_topk(lg[t], k), (t, idx[t], brute_topk(lg[t], k))
    # softmax over the selected logits: weights sum to 1 and ratios are exp(l_i - l_j)
    sel = np.take_along_axis(lg.astype(np.float64), idx.astype(np.int64), axis=1)
    assert np.abs(w.astype(np.float64).sum(1) - 1).max() <= 1e-6
    ratio = w[:, 1:].astype(np.float64) / w[:, :1]
    assert np.allclose(ratio, np.exp(sel[:, 1:] - sel[:, :1]), rtol=1e-5, atol=0)
    assert np.all(np.diff(sel, axis=1) <= 0)


def brute_margin(row, k):
    """(k-th largest) - ((k+1)-th largest) of a row by a Python full sort of its values,
    in float64; +inf when the row has no (k+1)-th value (k = E)."""
    vals = sorted((float(v) for v in row), reverse=True)
    if k >= len(vals):
        return math.inf
    return vals[k - 1] - vals[k]


def check_topk_margin(topk_margin, T=48, E=16, k=4, seed=8):
    """The near-tie margin against a brute-force sort, on rows with exact ties planted
    at positions (k-1, k) (margin exactly 0), inside the selection (k-2, k-1) and just
    outside it (k, k+1); k = E gives +inf."""
    rng = np.random.Generator(np.random.PCG64(seed))
    lg = rng.standard_normal((T, E)).astype(np.float32)
    for t in range(T):
        srt = np.argsort(-lg[t].astype(np.float64), kind="stable")
        if t % 4 == 0:
            lg[t, srt[k]] = lg[t, srt[k - 1]]
        elif t % 4 == 1:
            lg[t, srt[k - 2]] = lg[t, srt[k - 1]]
        elif t % 4 == 2:
            lg[t, srt[k + 1]] = lg[t, srt[k]]
    got = np.asarray(topk_margin(lg, k), dtype=np.float64)
    assert got.shape == (T,)
    for t in range(T):
        assert got[t] == brute_margin(lg[t], k), (t, got[t], brute_margin(lg[t], k))
    assert np.all(got[0::4] == 0.0)
    assert np.all(got[1::4] > 0.0) and np.all(got[2::4] > 0.0)
    # a hand-written row: sorted values 5, 3, 2.5, 2.5, -1 -> margin(2) = 0.5, margin(3) = 0, margin(4) = 3.5
    row = np.array([[2.5, -1.0, 5.0, 2.5, 3.0]], np.float32)
    assert [float(topk_margin(row, kk)[0]) for kk in (1, 2, 3, 4)] == [2.0, 0.5, 0.0, 3.5]
    # k = E: every expert is selected, no competitor
    assert np.all(np.isinf(np.asarray(topk_margin(lg[:, :k], k))))


def check_router_logits(router_logits, bf16_bits_of, seed=12):
    """Router logits with a bias against closed forms: x = 0 gives the bias exactly;
    a one-hot x row (x[t, h] = 1) gives column h of W_r plus the bias, one float32
    rounding of an exact sum; and a small case against pure-Python float64 loops."""
    rng = np.random.Generator(np.random.PCG64(seed))
    E, H = 8, 64
    w_bits = bf16_bits_of((0.02 * rng.standard_normal((E, H))).astype(np.float32))
    w = (w_bits.astype(np.uint32) << 16).view(np.float32)
    bias = (rng.standard_normal(E) * 3).astype(np.float32)
    zero = np.zeros((3, H), np.uint16)
    lg = router_logits(zero, w_bits, bias)
    assert np.array_equal(lg, np.broadcast_to(bias, (3, E)))
    assert np.array_equal(router_logits(zero, w_bits, None), np.zeros((3, E), np.float32))
    hot = [0, 17, 63]
    x1 = np.zeros((3, H), np.uint16)
    for t, h in enumerate(hot):
        x1[t, h] = 0x3F80  # bf16 1.0
    lg = router_logits(x1, w_bits, bias)
    for t, h in enumerate(hot):
        for e in range(E):
            want = np.float32(float(w[e, h]) + float(bias[e]))  # exact sum of two floats, rounded once
            assert lg[t, e] == want, (t, e, lg[t, e], want)
    assert np.array_equal(router_logits(x1, w_bits, None), w[:, hot].T)
    # brute force: float64 loops over h, the bias added last
    x_bits = bf16_bits_of(rng.standard_normal((5, H)).astype(np.float32))
    x = (x_bits.astype(np.uint32) << 16).view(np.float32)
    lg = router_logits(x_bits, w_bits, bias, np.float64)
    for t in range(5):
        for e in range(E):
            want = sum(float(x[t, h]) * float(w[e, h]) for h in range(H)) + float(bias[e])
            assert abs(lg[t, e] - want) <= 1e-12 * (1 + abs(want)), (t, e)


# tokens-per-expert -> tile rows, worked by hand from the rule "16 if m <= 16, 64 if
# m <= 64, else 128" with m = T*k/E (both boundaries included in the smaller tile)
TILE_ROWS_CASES = [
    (1, 4, 32, 16),      # m = 0.125
    (128, 4, 32, 16),    # m = 16 exactly
    (129, 4, 32, 64),    # m = 16.125
    (200, 2, 16, 64),    # m = 25
    (512, 4, 32, 64),    # m = 64 exactly
    (513, 4, 32, 128),   # m = 64.125
    (64, 4, 128, 16),    # m = 2
    (4096, 4, 128, 128),  # m = 128
    (13, 3, 3, 16),      # m = 13
    (17, 1, 1, 64),      # m = 17
]


def check_tile_rows_policy(tile_rows_policy):
    for T, k, E, want in TILE_ROWS_CASES:
        assert tile_rows_policy(T, k, E) == want, (T, k, E, tile_rows_policy(T, k, E), want)


def brute_tile_table(idx, E, bm):
    """Counting sort by hand with Python lists."""
    flat = [int(v) for v in np.asarray(idx).reshape(-1)]
    buckets = [[] for _ in range(E)]
    for a, e in enumerate(flat):
        buckets[e].append(a)
    counts = [len(b) for b in buckets]
    offsets = [0]
    for c in counts:
        offsets.append(offsets[-1] + c)
    perm = [a for b in buckets for a in b]
    inv = [0] * len(flat)
    for s, a in enumerate(perm):
        inv[a] = s
    tiles = []
    for e in range(E):
        start = offsets[e]
        while start < offsets[e + 1]:
            n = min(bm, offsets[e + 1] - start)
            tiles.append((e, start, n, len(tiles) * bm))
            start += n
    return counts, offsets, perm, inv, tiles


def check_tile_table(tile_table, cases):
    for idx, E, bm in cases:
        got = tile_table(idx, E, bm)
        counts, offsets, perm, inv, tiles = brute_tile_table(idx, E, bm)
        assert list(got["counts"]) == counts
        assert list(got["offsets"]) == offsets
        assert list(got["perm"]) == perm
        assert list(got["inv_perm"]) == inv
        assert [tuple(int(v) for v in r) for r in got["tiles"]] == tiles
        assert got["num_tiles"] == len(tiles)
        # invariants: counts sum to T*k, every tile inside its expert, rows covered once
        Tk = np.asarray(idx).size
        assert sum(counts) == Tk
        covered = np.zeros(Tk, dtype=int)
        for e, s, n, _ in tiles:
            assert offsets[e] <= s and s + n <= offsets[e + 1] and 1 <= n <= bm
            covered[s:s + n] += 1
        assert np.all(covered == 1)
        # permute then unpermute is the identity
        X = np.random.default_rng(0).standard_normal((Tk, 3))
        P = X[got["perm"]]
        assert np.array_equal(P[got["inv_perm"]], X)


# ------------------------------------------------------------ layer invariants
def check_identical_experts(moe_layer, expert_hidden, expert_output, bf16_to_f32, inp, dtype):
    """With every expert equal and softmax weights summing to 1, the layer is the
    dense FFN of that expert whatever the routing."""
    res = moe_layer(inp, dtype=dtype)
    x = bf16_to_f32(inp.x).astype(dtype)
    dense = expert_output(expert_hidden(x, inp.gu_codes[0], inp.gu_scales[0], inp.I, dtype),
                          inp.dn_codes[0], inp.dn_scales[0], dtype)
    err = np.abs(res["out_unrounded"] - dense).max() / np.abs(dense).max()
    assert err <= (1e-5 if dtype == np.float32 else 1e-12), err


def dense_reference_loops(inp):
    """E = 1, k = 1 layer by explicit float64 Python-level decoding and sums
    (no table, no matmul), for small H, I."""
    I, H = inp.I, inp.H

    def dec(codes, scales, r, kk):
        byte = int(codes[r, kk // 2])
        c = byte & 0xF if kk % 2 == 0 else byte >> 4
        return float(e2m1_from_bitfields(c)) * 2.0 ** (int(scales[r, kk // 32]) - 127)

    out = np.zeros((inp.T, H))
    for t in range(inp.T):
        x = [float(np.uint32(int(v) << 16).view(np.float32)) for v in inp.x[t]]
        h = []
        for i in range(I):
            g = sum(x[kk] * dec(inp.gu_codes[0], inp.gu_scales[0], i, kk) for kk in range(H))
            u = sum(x[kk] * dec(inp.gu_codes[0], inp.gu_scales[0], I + i, kk) for kk in range(H))
            h.append(g / (1 + math.exp(-g)) * u)
        for n in range(H):
            out[t, n] = sum(h[i] * dec(inp.dn_codes[0], inp.dn_scales[0], n, i) for i in range(I))
    return out
