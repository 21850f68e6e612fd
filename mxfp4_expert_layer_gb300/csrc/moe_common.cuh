// Shared definitions of the MXFP4 MoE layer kernels: shapes, workspace layout,
// the four-term E2M1 activation encoding and device status reporting.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "moe_mxfp4.h"

namespace moe {

// ----------------------------------------------------------------- constants
constexpr int kMxBlock = 32;         // K values sharing one E8M0 scale
constexpr int kKGroup = 128;         // K values per pipeline stage (4 MX blocks)
constexpr int kMTile = 128;          // weight rows per MMA tile (MMA M)
constexpr int kSfAtomBytes = 512;    // scale-factor atom: 128 rows x 4 MX blocks
constexpr int kMaxExperts = 256;
// Gating variants of the top-k weights (the selection is the same in every one):
// softmax over the k selected logits, softmax over all E logits (the selected
// probabilities), or the selected logits' sigmoids normalised to sum to one.
constexpr int kGatingSoftmaxTopk = 0;
constexpr int kGatingSoftmaxAll = 1;
constexpr int kGatingSigmoid = 2;
constexpr int kMaxTopK = 32;
constexpr int kMaxCtas = 160;        // persistent GEMM CTAs (one per SM; GB300 has 152)
constexpr int kTerms = 4;            // E2M1 terms of the activation encoding

// Device status word bits (read back with moe_get_device_status).
constexpr uint32_t kStatusTimeoutMain = 1u << 0;
constexpr uint32_t kStatusTimeoutEpi = 1u << 1;
constexpr uint32_t kStatusTimeoutProducer = 1u << 2;
constexpr uint32_t kStatusBadIndex = 1u << 3;

__host__ __device__ inline int ceil_div(int a, int b) { return (a + b - 1) / b; }
__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// K rounded up to whole pipeline stages (the prepared weight rows carry this many
// 4-bit codes; codes past the real K are zero).
// K groups of 128 values (one scale atom each) over K, rounded up to an even count so
// that a 256-value pipeline stage always finds two atoms
__host__ __device__ inline int kgroups_even(int K) { return ceil_div(K, 2 * kKGroup) * 2; }

// Token rows per tile from the mean tokens per expert ("token tile follows tokens
// per expert"): 16 for decode-sized loads, 64 for medium, 128 for prefill.
__host__ __device__ inline int tile_rows_policy(int T, int k, int E) {
  long long tk = (long long)T * k;
  if (tk <= 16LL * E) return 16;
  if (tk <= 64LL * E) return 64;
  return 128;
}

// bf16-weight layer: 256-row tiles once the mean tokens per expert fill them (an
// N = 256 MMA carries twice the work of an N = 128 one for the same issued
// instruction); below that the policy above.
__host__ __device__ inline int tile_rows_policy_bf16(int T, int k, int E) {
  return (long long)T * k >= 256LL * E ? 256 : tile_rows_policy(T, k, E);
}

__host__ __device__ inline int max_tiles_bound(int T, int k, int E, int bm) {
  long long tk = (long long)T * k;
  long long b = tk / bm + (E < tk ? E : tk);
  return (int)b;
}

// ----------------------------------------------------------------- tiles
struct TileEntry {
  int32_t expert;     // expert of every row in the tile
  int32_t row_begin;  // first sorted row (index into perm)
  int32_t n_rows;     // valid rows, 1..bm
  int32_t pad_row;    // first row of the tile in the padded activation buffers (= tile * bm)
};

// One tile-table entry through L2 only (16-byte load): the table is produced by an
// earlier kernel of the same call.
__device__ __forceinline__ TileEntry load_tile(const TileEntry* t) {
  const int4 v = __ldcg(reinterpret_cast<const int4*>(t));
  TileEntry e;
  e.expert = v.x;
  e.row_begin = v.y;
  e.n_rows = v.z;
  e.pad_row = v.w;
  return e;
}

// ----------------------------------------------------------------- workspace
// Byte offsets of every region inside the caller-allocated workspace.
struct WsLayout {
  int T, H, I, E, k, bm, max_tiles, pad_rows;
  int kg_h, kg_i;        // K groups of 128 over H and over I, rounded up to even
  int mt_h, mt_i;        // M tiles (of 128) over H and over I
  size_t status;         // uint32 device status word (+ padding)
  size_t route_sync;     // uint32 [ceil(T/8) + 1] arrival counters of the routing kernel
  size_t logits;         // f32 [T, E]
  size_t idx;            // i32 [T, k]
  size_t w;              // f32 [T, k]
  size_t counts;         // i32 [E]
  size_t offsets;        // i32 [E + 1]
  size_t perm;           // i32 [T*k]
  size_t inv_perm;       // i32 [T*k]: each assignment's padded row (tile x bm + row in tile)
  size_t tiles;          // TileEntry [max_tiles]
  size_t num_tiles;      // i32
  size_t xt_q;           // x encoded per token: [kg_h][T][kTerms][64 bytes] packed E2M1
  size_t xt_sf;          // its E8M0 exponents: u32 [kg_h][T][kTerms] (4 MX blocks each)
  size_t x_q;            // x gathered into tile order (act_offset): kg_h * 128 values per row
  size_t x_sf;           // its scale atoms [max_tiles][kg_h][512 * act_sf_atoms(bm)]
  size_t h_q;            // h encoded, tile order (act_offset): kg_i * 128 values per row
  size_t h_sf;           // [max_tiles][kg_i][512 * act_sf_atoms(bm)]
  size_t slots;          // f32 [T*k, H]: weighted expert outputs awaiting the combine
  size_t total;
};

// Scale atoms (128 rows each) per tile and K group of an encoded activation: the
// tile's rows are the kTerms terms of its bm token rows, term-major.
__host__ __device__ inline int act_sf_atoms(int bm) { return (kTerms * bm + 127) / 128; }

inline WsLayout make_ws_layout(int T, int H, int I, int E, int k, int bm) {
  WsLayout L{};
  L.T = T; L.H = H; L.I = I; L.E = E; L.k = k; L.bm = bm;
  L.max_tiles = max_tiles_bound(T, k, E, bm);
  L.pad_rows = L.max_tiles * bm;
  L.kg_h = kgroups_even(H);
  L.kg_i = kgroups_even(I);
  L.mt_h = ceil_div(H, kMTile);
  L.mt_i = ceil_div(I, kMTile);
  const size_t A = 256;
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t r = o; o = align_up(o + bytes, A); return r; };
  const size_t tk = (size_t)T * k;
  const size_t sfa = (size_t)act_sf_atoms(bm) * kSfAtomBytes;
  L.status = take(256);
  L.route_sync = take(sizeof(uint32_t) * (size_t)(ceil_div(T, 8) + 1));
  L.logits = take(sizeof(float) * (size_t)T * E);
  L.idx = take(sizeof(int32_t) * tk);
  L.w = take(sizeof(float) * tk);
  L.counts = take(sizeof(int32_t) * (size_t)E);
  L.offsets = take(sizeof(int32_t) * (size_t)(E + 1));
  L.perm = take(sizeof(int32_t) * tk);
  L.inv_perm = take(sizeof(int32_t) * tk);
  L.tiles = take(sizeof(TileEntry) * (size_t)L.max_tiles);
  L.num_tiles = take(sizeof(int32_t));
  L.xt_q = take((size_t)L.kg_h * T * kTerms * 64);
  L.xt_sf = take((size_t)L.kg_h * T * kTerms * sizeof(uint32_t));
  L.x_q = take((size_t)L.kg_h * L.pad_rows * kTerms * 64);
  L.x_sf = take((size_t)L.max_tiles * L.kg_h * sfa);
  L.h_q = take((size_t)L.kg_i * L.pad_rows * kTerms * 64);
  L.h_sf = take((size_t)L.max_tiles * L.kg_i * sfa);
  L.slots = take(sizeof(float) * tk * H);
  L.total = o;
  return L;
}

template <typename P>
__host__ __device__ inline P* ws_ptr(void* ws, size_t off) {
  return reinterpret_cast<P*>(reinterpret_cast<uint8_t*>(ws) + off);
}

// ----------------------------------------------------------------- MXFP4 weights
// Prepared weight layout of one matrix family (gate/up or down) for E experts:
//   codes  [E][G][rows per group][K / 2]  the raw row-major codes, unchanged: a TMA box
//                         of 128 rows x 128 bytes (or 64) is one 256-code (128-code)
//                         K step of an M tile; the box past K reads zeros (TMA fill).
//                         G = 2 for gate/up (gate rows, up rows), 1 for down.
//   scales [E][G][MT][KG][512]  MT = ceil(rows per group / 128), KG = K groups of 128
//                         rounded up to even; each 512-byte atom holds the E8M0 scales
//                         of 128 rows x 4 MX blocks: byte (l*16 + c*4 + b) = scale of
//                         row 32c + l, block b (127 outside the matrix).
//   trailer (256 bytes): a status word the preparing kernel sets when it meets
//                         an E8M0 scale of 255 (NaN).
struct PreparedLayout {
  int E, R, K, groups, rows_per_group, mt, kg;
  size_t codes_bytes;   // E * R * K / 2
  size_t scales_off;    // aligned start of the scale atoms
  size_t flag_off;      // status trailer
  size_t total;
};

inline PreparedLayout make_prepared_layout(int E, int R, int K, int groups) {
  PreparedLayout P{};
  P.E = E; P.R = R; P.K = K; P.groups = groups;
  P.rows_per_group = R / groups;
  P.mt = ceil_div(P.rows_per_group, kMTile);
  P.kg = kgroups_even(K);
  P.codes_bytes = (size_t)E * R * (K / 2);
  P.scales_off = align_up(P.codes_bytes, 256);
  P.flag_off = align_up(P.scales_off + (size_t)E * groups * P.mt * P.kg * kSfAtomBytes, 256);
  P.total = P.flag_off + 256;
  return P;
}

// ----------------------------------------------------------------- activations
// Exponents are kept in [-126, 127] so 2^p and 2^-p are normal floats and the
// E8M0 byte p + 127 is never 255 (NaN).
__device__ __forceinline__ float pow2_int(int e) { return __int_as_float((e + 127) << 23); }

// E2M1 terms: p is the smallest exponent with amax <= 6 * 2^p (6 = largest E2M1).
__device__ __forceinline__ int mx_e2m1_exponent(float amax) {
  if (!(amax > 0.f)) return 0;
  // floor(log2(amax)) from the exponent field (subnormals clamp to the minimum below)
  int e = (int)((__float_as_uint(amax) >> 23) & 0xFFu) - 127 - 2;  // amax / 2^e in [4, 8)
  if (e < -126) e = -126;
  if (e > 127) e = 127;
  if (amax > 6.f * pow2_int(e) && e < 127) e += 1;
  return e;
}

// Nearest E2M1 codes of (lo, hi), ties to even, saturating at +-6, packed as one
// byte: lo in bits 0-3, hi in bits 4-7 (the hardware conversion instruction puts its
// first source operand in the upper half).
__device__ __forceinline__ uint32_t f32x2_to_e2m1x2(float lo, float hi) {
  uint16_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %2, %1;\n\tmov.b16 %0, {t, 0};\n\t}"
      : "=h"(r)
      : "f"(lo), "f"(hi));
  return static_cast<uint32_t>(r) & 0xFFu;
}

// Nearest E2M1 code of v as a 4-bit code.
__device__ __forceinline__ uint32_t f32_to_e2m1(float v) { return f32x2_to_e2m1x2(v, 0.f) & 0xFu; }

// Value of a 4-bit E2M1 code built from its bit fields with integer operations only
// (no conversion instruction; exact): sign bit 3; magnitude m = bits 0-2 is 0, 0.5
// (m = 1) or (1 + (m & 1) / 2) * 2^((m >> 1) - 1) for m >= 2, whose float32 exponent
// field is (m >> 1) + 126 and whose top mantissa bit is m & 1.
__device__ __forceinline__ float e2m1_to_f32(uint32_t code) {
  const uint32_t m = code & 7u;
  const uint32_t mag = m >= 2u ? ((((m >> 1) + 126u) << 23) | ((m & 1u) << 22)) : (m ? 0x3F000000u : 0u);
  return __uint_as_float(mag | ((code & 8u) << 28));
}

// Values of the two E2M1 codes of one byte (low nibble -> .x), through the hardware
// E2M1 -> f16 conversion (exact: every E2M1 value is an f16).  In the gate/up
// epilogue this measured faster than rebuilding the values with integer operations.
__device__ __forceinline__ float2 e2m1x2_to_f32x2(uint32_t byte) {
  uint32_t h2;
  const uint16_t b16 = static_cast<uint16_t>(byte & 0xFFu);
  asm("{\n\t.reg .b8 t, z;\n\tmov.b16 {t, z}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(h2) : "h"(b16));
  return __half22float2(*reinterpret_cast<const __half2*>(&h2));
}

// Row of (term t, token row r) inside an activation tile's B operand.  Tiles of at
// most 16 token rows (all terms in one MMA along N) are token major, so the rows of
// the tile's real tokens come first and one TMA box of 4 x (tokens rounded up to a
// power of two) rows covers them; larger tiles are term major (one MMA per term).
__host__ __device__ constexpr bool act_token_major(int bm) { return kTerms * bm <= 64; }
// K values per pipeline stage of the expert GEMMs: 256 for every tile size (128-byte
// operand rows, 128-byte swizzle).
__host__ __device__ constexpr int gemm_kstage(int) { return 256; }
__host__ __device__ inline int act_row(int t, int r, int bm) {
  return act_token_major(bm) ? r * kTerms + t : t * bm + r;
}
// Byte offset of the code byte holding values (k, k+1) (k even) of term t of row r
// of tile `tile` in an encoded activation buffer
// [K / 256][max_tiles][kTerms * bm rows][128 bytes].  One tile's rows of one stage
// form a contiguous image that is exactly the 128-byte-swizzled shared-memory tile
// the MMA reads (16-byte chunk c of image row i stored at chunk c ^ (i % 8)), so
// the GEMMs load it with a plain bulk copy; writers of more than one byte at a time
// stay within one 16-byte chunk.
__host__ __device__ inline size_t act_offset(int tile, int t, int r, int k, int max_tiles, int bm) {
  const int row = act_row(t, r, bm);
  const int byte = (k % 256) >> 1;
  return (((size_t)(k / 256) * max_tiles + tile) * (kTerms * bm) + row) * 128 +
         ((((byte >> 4) ^ (row & 7)) << 4) | (byte & 15));
}

// Scale atom byte offset of (row r within a tile, MX block b within a K group).
// bf16 activations (the bf16-weight GEMMs): one image per (64-value K stage, tile)
// of bm rows x 128 bytes, 128-byte swizzled (16-byte chunk c of row r stored at
// c ^ (r % 8)), so one bulk copy lands it in the layout the MMA reads:
// [K / 64][max_tiles][bm][128 B].
__host__ __device__ inline size_t act16_offset(int tile, int r, int k, int max_tiles, int bm) {
  const int byte = (k % 64) * 2;
  return (((size_t)(k / 64) * max_tiles + tile) * bm + r) * 128 + ((((byte >> 4) ^ (r & 7)) << 4) | (byte & 15));
}

__host__ __device__ inline int sf_atom_offset(int r, int b) {
  return (r >> 7) * kSfAtomBytes + (r & 31) * 16 + ((r >> 5) & 3) * 4 + b;
}

__device__ __forceinline__ void report_status(uint32_t* status, uint32_t bits) {
  if (status) atomicOr(status, bits);
}

}  // namespace moe
