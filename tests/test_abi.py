"""CPU checks of the C ABI: the library builds, loads, exports every function the
header declares, and rejects bad arguments on the host before any launch."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import mxfp4_expert_layer_gb300 as pkg
    pkg.build()
    return pkg._lib.load()


def declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", fn)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names += re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", txt)
    return sorted(set(names))


def test_every_declared_symbol_is_exported_and_bound(lib):
    from mxfp4_expert_layer_gb300 import _lib as L
    names = declared_functions()
    assert len(names) >= 14
    for n in names:
        assert hasattr(lib, n), n
        assert n in L.SIGNATURES, n


def test_error_strings(lib):
    from mxfp4_expert_layer_gb300 import _lib as L
    for code in (0, -1, -2, -3, -4, -5, -6, -99):
        assert L.moe_error_string(code)


def test_library_tile_policy_matches_worked_values(lib):
    # the host-side policy of the C ABI against the values worked by hand for the
    # oracle's pin (no GPU involved: moe_tile_rows is host arithmetic)
    from mxfp4_expert_layer_gb300 import _lib as L
    from tests.oracle_checks import TILE_ROWS_CASES
    for T, k, E, want in TILE_ROWS_CASES:
        assert L.moe_tile_rows(T, k, E) == want, (T, k, E)


def test_sizes_and_policy(lib):
    from mxfp4_expert_layer_gb300 import _lib as L
    import oracle
    assert L.moe_workspace_bytes(64, 2880, 2880, 32, 4) > 0
    assert L.moe_workspace_bytes(64, 2880, 2880, 32, 33) == 0        # k > E
    assert L.moe_workspace_bytes(64, 2881, 2880, 32, 4) == 0         # H % 32
    assert L.moe_workspace_bytes(4, 256, 256, 300, 2) == 0           # E > 256
    for T, E, k in [(1, 32, 4), (64, 32, 4), (64, 128, 4), (4096, 128, 4), (4, 8, 2), (300, 8, 2)]:
        assert L.moe_tile_rows(T, k, E) == oracle.tile_rows_policy(T, k, E)
        for bm in (16, 64, 128):
            assert L.moe_max_tiles(T, k, E, bm) == oracle.max_tiles_bound(T, k, E, bm)
    # prepared bytes: the row-major codes, 512-byte scale atoms over an even number of
    # 128-value K groups (2880 -> 24), a trailer
    E, I, H = 32, 2880, 2880
    n = L.moe_prepared_weight_bytes(E, 2 * I, H, L.MOE_WEIGHTS_GATEUP)
    codes = E * 2 * I * H // 2
    atoms = E * 2 * 23 * 24 * 512
    assert n == ((codes + 255) // 256 * 256 + atoms + 255) // 256 * 256 + 256
    assert L.moe_prepared_weight_bytes(E, 2 * I + 1, H, L.MOE_WEIGHTS_GATEUP) == 0
    assert L.moe_forward_launches(64, 2880, 2880, 32, 4) == 5


def test_host_argument_checks_return_codes(lib):
    from mxfp4_expert_layer_gb300 import _lib as L
    T, H, I, E, k = 64, 2880, 2880, 32, 4
    ws = L.moe_workspace_bytes(T, H, I, E, k)
    fake = 1 << 20  # aligned, never dereferenced: every call below fails its checks first
    args = dict(x=fake, wr=fake, b=None, wgu=fake, wd=fake, ws=fake, out=fake)

    def fwd(**kw):
        a = dict(args, **kw)
        return L.moe_forward(a["x"], a["wr"], a["b"], a["wgu"], a["wd"], kw.get("T", T), H, I, E, k, a["ws"],
                             kw.get("ws_bytes", ws), a["out"], None, None, None)

    assert fwd(x=None) == L.MOE_ERR_INVALID_ARG
    assert fwd(out=None) == L.MOE_ERR_INVALID_ARG
    assert fwd(x=fake + 2) == L.MOE_ERR_INVALID_ARG          # misaligned
    assert fwd(ws=fake + 16) == L.MOE_ERR_INVALID_ARG        # workspace must be 256-aligned
    assert fwd(ws_bytes=ws - 1) == L.MOE_ERR_WORKSPACE_TOO_SMALL
    assert fwd(T=0) == L.MOE_ERR_UNSUPPORTED_SHAPE
    assert L.moe_route(fake, fake, None, T, H, E, k, fake, 7, fake, fake, fake, ws, None) == L.MOE_ERR_INVALID_ARG
    assert L.moe_route(None, None, None, T, H, E, k, None, 0, fake, fake, fake, ws, None) == L.MOE_ERR_INVALID_ARG
    # both gating variants at once, or an unknown flag bit
    assert L.moe_route(fake, fake, None, T, H, E, k, fake, 6, fake, fake, fake, ws, None) == L.MOE_ERR_INVALID_ARG
    assert L.moe_route(fake, fake, None, T, H, E, k, fake, 8, fake, fake, fake, ws, None) == L.MOE_ERR_INVALID_ARG
    assert L.moe_forward_gated(fake, fake, None, fake, fake, T, H, I, E, k, 3, fake, ws, fake, None, None,
                               None) == L.MOE_ERR_INVALID_ARG
    # the norm step: missing or misaligned residual / weight, bad eps, residual_out == out
    def fnorm(res=fake, gam=fake, eps=1e-5, gating=0, rout=None, out=fake):
        return L.moe_forward_norm(fake, res, gam, eps, fake, None, fake, fake, T, H, I, E, k, gating, fake, ws, out,
                                  rout, None, None, None)
    assert fnorm(res=None) == L.MOE_ERR_INVALID_ARG
    assert fnorm(gam=fake + 2) == L.MOE_ERR_INVALID_ARG
    assert fnorm(eps=-1.0) == L.MOE_ERR_INVALID_ARG
    assert fnorm(eps=float("nan")) == L.MOE_ERR_INVALID_ARG
    assert fnorm(eps=float("inf")) == L.MOE_ERR_INVALID_ARG
    assert fnorm(gating=3) == L.MOE_ERR_INVALID_ARG
    assert fnorm(rout=fake) == L.MOE_ERR_INVALID_ARG           # residual_out may not be out
    assert fnorm(rout=fake + 8) == L.MOE_ERR_INVALID_ARG       # misaligned residual_out
    # the bf16-weight layer: H and I must be multiples of 64
    def f16(H_=H, I_=I, x=fake, wgu=fake):
        return L.moe_forward_bf16(x, fake, None, wgu, fake, T, H_, I_, E, k, fake, ws, fake, None, None, None)
    assert f16(H_=2880 + 32) == L.MOE_ERR_UNSUPPORTED_SHAPE
    assert f16(I_=2880 + 32) == L.MOE_ERR_UNSUPPORTED_SHAPE
    assert f16(I_=16384 + 64) == L.MOE_ERR_UNSUPPORTED_SHAPE    # I above its limit
    assert f16(x=None) == L.MOE_ERR_INVALID_ARG
    assert f16(wgu=fake + 8) == L.MOE_ERR_INVALID_ARG
    assert L.moe_build_tile_table(fake, T, k, E, 32, fake, fake, fake, fake, fake, fake, None) == \
        L.MOE_ERR_UNSUPPORTED_SHAPE                            # tile rows must be 16, 64 or 128
    assert L.moe_prepare_weights(fake, fake, E, 2 * I, H, 5, fake, 1 << 40, None) == L.MOE_ERR_UNSUPPORTED_SHAPE
    assert L.moe_prepare_weights(fake, fake, E, 2 * I, H, 0, fake, 16, None) == L.MOE_ERR_WORKSPACE_TOO_SMALL
    # bf16 weight tiles: (tiles + one zero tile) x 16 KB; K a multiple of 64, rows of whole groups
    assert L.moe_prepared_weight_bytes_bf16(8, 2 * 14336, 4096, L.MOE_WEIGHTS_GATEUP) == (8 * 2 * 112 * 64 + 1) * 16384
    assert L.moe_prepared_weight_bytes_bf16(2, 2 * 192, 128, L.MOE_WEIGHTS_GATEUP) == (2 * 2 * 2 * 2 + 1) * 16384
    assert L.moe_prepared_weight_bytes_bf16(8, 4096, 14336 + 32, L.MOE_WEIGHTS_DOWN) == 0
    assert L.moe_prepared_weight_bytes_bf16(8, 4097, 4096, L.MOE_WEIGHTS_GATEUP) == 0
    assert L.moe_prepared_weight_bytes_bf16(8, 4096, 4096, 7) == 0
    assert L.moe_prepare_weights_bf16(fake, E, H, I, L.MOE_WEIGHTS_DOWN, fake + 16, 1 << 40, None) == \
        L.MOE_ERR_INVALID_ARG                                  # destination not 256-byte aligned
    assert L.moe_prepare_weights_bf16(fake, E, H, I, L.MOE_WEIGHTS_DOWN, fake, 16, None) == \
        L.MOE_ERR_WORKSPACE_TOO_SMALL
    st = ctypes.c_int(0)
    assert L.moe_get_device_status(None, 0, ctypes.byref(st), None) == L.MOE_ERR_INVALID_ARG


def test_product_path_does_not_import_oracle():
    pkg_dir = os.path.join(ROOT, "mxfp4_expert_layer_gb300")
    for dirpath, _, files in os.walk(pkg_dir):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                txt = open(os.path.join(dirpath, fn)).read()
                assert "import oracle" not in txt and "from oracle" not in txt, fn
                assert "synthetic" not in txt, fn
