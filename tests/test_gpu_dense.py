"""GPU parity of the bf16-weight layer (moe_forward_bf16: the same routing, then
grouped kind::f16 tcgen05 GEMMs) against the oracle's moe_layer_dense, on ragged
shapes covering the three tile sizes and on Mixtral-8x7B shapes (sampled tokens)."""

import numpy as np
import pytest

import oracle
from synthetic import make_dense_config, make_dense_layer
from tests.gpu_helpers import TOL_MAX_ABS, TOL_REL_FROB, bf16_bits_to_f32, bf16_to_np, errors, logit_band, to_dev

pytestmark = pytest.mark.gpu


def run_dense(inp):
    import torch
    import mxfp4_expert_layer_gb300 as pkg
    pkg.build()
    layer = pkg.MoELayerBF16(to_dev(inp.w_router), to_dev(inp.w_gateup), to_dev(inp.w_down), k=inp.k)
    idx = torch.empty(inp.T, inp.k, dtype=torch.int32, device="cuda")
    w = torch.empty(inp.T, inp.k, dtype=torch.float32, device="cuda")
    out = layer(to_dev(inp.x), topk_idx=idx, topk_w=w)
    torch.cuda.synchronize()
    assert layer.device_status(inp.T) == 0
    return layer, bf16_bits_to_f32(bf16_to_np(out)), idx.cpu().numpy(), w.cpu().numpy()


def check_dense(inp, tokens=None):
    import mxfp4_expert_layer_gb300 as pkg
    from mxfp4_expert_layer_gb300 import _lib as L
    pkg.build()
    _, out, idx, w = run_dense(inp)
    ref = oracle.moe_layer_dense(inp, tokens=tokens)
    tok = ref["tokens"]
    keep = oracle.topk_margin(ref["logits"], inp.k) > logit_band(inp)[0]
    assert keep.mean() > 0.9
    assert np.array_equal(idx[tok][keep], ref["idx"][keep])
    assert np.allclose(w[tok][keep], ref["w"][keep], rtol=1e-4, atol=1e-5)
    rel, mx = errors(out[tok][keep], ref["out"][keep])
    assert rel <= TOL_REL_FROB and mx <= TOL_MAX_ABS, (rel, mx, L.moe_tile_rows(inp.T, inp.k, inp.E))
    return rel, mx


@pytest.mark.parametrize("T,H,I,E,k,bm", [
    (8, 256, 384, 4, 2, 16),      # dense_tiny shape
    (37, 512, 448, 6, 2, 16),     # ragged tiles, I not a multiple of 128
    (150, 256, 320, 8, 2, 64),
    (400, 256, 256, 4, 2, 128),   # two epilogue groups
    (600, 256, 256, 4, 2, 256),   # 256-row tiles (N = 256 MMAs), a 44-row last tile
    (700, 256, 192, 2, 1, 256),   # 256-row tiles, an M tile of 64 real rows
    (1, 128, 192, 3, 3, 16),      # one token, every expert
])
def test_dense_layer_shapes(T, H, I, E, k, bm):
    """bm: the tile rows the bf16 layer uses -- the MXFP4 policy's, or 256 once the
    mean tokens per expert reach 256."""
    from mxfp4_expert_layer_gb300 import _lib as L
    import mxfp4_expert_layer_gb300 as pkg
    pkg.build()
    assert (256 if T * k >= 256 * E else L.moe_tile_rows(T, k, E)) == bm
    check_dense(make_dense_layer(T, H, I, E, k, seed=T + H))


def test_dense_mixtral_shapes_sampled():
    # Mixtral-8x7B experts (H 4096, F 14336, 8 experts, top-2) at 2048 tokens (256-row
    # tiles) and at its first 32 tokens (16-row tiles), sampled tokens against the oracle
    import dataclasses
    big = make_dense_config("mixtral_t2048")
    check_dense(big, tokens=np.arange(0, 2048, 97))
    small = dataclasses.replace(big, T=32, x=big.x[:32])
    check_dense(small, tokens=np.arange(0, 32, 3))


def test_dense_layer_is_bit_reproducible():
    inp = make_dense_layer(64, 256, 256, 8, 2, seed=9)
    _, a, ia, _ = run_dense(inp)
    _, b, ib, _ = run_dense(inp)
    assert np.array_equal(a, b) and np.array_equal(ia, ib)


def swizzled_tiles(w: np.ndarray, groups: int) -> np.ndarray:
    """The prepared bf16 layout restated in numpy (moe_prepare_weights_bf16): tiles of
    128 rows x 64 values per (expert, row group, 128-row M tile, 64-value K stage),
    rows past the group zero, 16-byte chunk c of row r stored at c ^ (r % 8), then one
    zero tile.  Returns the bytes."""
    E, rows, K = w.shape
    rpg = rows // groups
    mt, ks = -(-rpg // 128), K // 64
    tiles = np.zeros((E, groups, mt, ks, 128, 8, 8), dtype=np.uint16)  # [.., row, chunk, value]
    for e in range(E):
        for g in range(groups):
            for m in range(mt):
                block = w[e, g * rpg + m * 128: g * rpg + min(rpg, (m + 1) * 128)]
                for s in range(ks):
                    vals = block[:, s * 64:(s + 1) * 64].reshape(-1, 8, 8)
                    for r in range(vals.shape[0]):
                        tiles[e, g, m, s, r, np.arange(8) ^ (r % 8)] = vals[r]
    flat = tiles.reshape(-1, 128 * 64)
    return np.concatenate([flat, np.zeros((1, 128 * 64), np.uint16)]).view(np.uint8).reshape(-1)


@pytest.mark.parametrize("E,rows,K,kind", [(2, 2 * 192, 128, 0), (2, 128, 192, 1), (1, 2 * 64, 64, 0)])
def test_prepare_weights_bf16_byte_exact(E, rows, K, kind):
    """The prepared bf16 tiles, byte for byte: ragged M tiles (192 and 64 rows per
    group), several K stages, both families."""
    import torch
    import mxfp4_expert_layer_gb300 as pkg
    pkg.build()
    rng = np.random.default_rng(E * 1000 + rows + K)
    w = rng.integers(0, 1 << 16, size=(E, rows, K), dtype=np.uint16)
    got = pkg.prepare_weights_bf16(to_dev(w), kind)
    torch.cuda.synchronize()
    want = swizzled_tiles(w, 2 if kind == 0 else 1)
    assert got.numel() == want.size
    assert np.array_equal(got.cpu().numpy(), want)
