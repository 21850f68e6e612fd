// Launch parameters and launchers of the MoE kernels (internal to the library).
#pragma once

#include <cuda.h>

#include "moe_common.cuh"

namespace moe {

struct RouteParams {
  const uint16_t* x;        // bf16 [T, H]
  const uint16_t* w_router; // bf16 [E, H]
  const float* bias;        // f32 [E] or null
  int T, H, E, k;
  int from_logits;          // logits are an input
  int experts_per_block;    // experts per block slice (multiple of 8)
  float* logits;            // f32 [T, E]
  int32_t* topk_idx;        // i32 [T, k]
  float* topk_w;            // f32 [T, k]
  uint32_t* sync;           // arrival counters [ceil(T/8) + 1], zero between calls
  int build_table;          // also build the tile table (last block)
  int bm;
  int32_t *counts, *offsets, *perm, *inv_perm, *num_tiles;
  TileEntry* tiles;
  uint32_t* status;
};

cudaError_t launch_route(const RouteParams& p, cudaStream_t stream);
cudaError_t launch_tile_table(const int32_t* idx, int Tk, int E, int bm, int32_t* counts, int32_t* offsets,
                              int32_t* perm, int32_t* inv_perm, TileEntry* tiles, int32_t* num_tiles,
                              cudaStream_t stream);

// Gather + two-term E4M3 encoding of the activation rows of every tile.
struct QuantXParams {
  const uint16_t* x;       // bf16 [T, H]
  const int32_t* perm;
  const TileEntry* tiles;
  const int32_t* num_tiles;
  int T, H, k, bm, max_tiles, kg;
  uint8_t *q_hi, *q_lo;    // [pad_rows, H]
  uint8_t *sf_hi, *sf_lo;  // [max_tiles][kg][512 * atoms]
  int32_t* zero_buf;       // combine counters to clear (or null)
  int zero_count;
};
cudaError_t launch_quant_x(const QuantXParams& p, cudaStream_t stream);

struct GemmParams {
  // operand tensor maps (TMA)
  CUtensorMap tm_w;        // weights: 4-bit codes [E][groups][rows][Kp] (16U4_ALIGN16B)
  CUtensorMap tm_act_hi;   // activations e4m3 [pad_rows][K]
  CUtensorMap tm_act_lo;
  const uint8_t* w_sf;     // weight scale atoms [E][groups][mt][kg][512]
  const uint8_t* act_sf_hi;// activation scale atoms [max_tiles][kg][512 * atoms]
  const uint8_t* act_sf_lo;
  const TileEntry* tiles;
  const int32_t* num_tiles;
  const int32_t* perm;
  int T, H, I, E, k, bm, max_tiles;
  int K;                   // contraction length (H for gate/up, I for down)
  int kg;                  // K groups of 128
  int mt;                  // M tiles of the output features
  int rows_out;            // output features (I for gate/up, H for down)
  int w_groups;            // 2 (gate, up) or 1 (down)
  int group_tiles;         // tiles per raster group
  // gate/up epilogue outputs (two-term e4m3 h)
  uint8_t *h_hi, *h_lo, *h_sf_hi, *h_sf_lo;
  int kg_out;              // K groups of h along I
  // down epilogue
  const float* topk_w;
  float* slots;            // f32 [T*k, H]
  int32_t* combine_cnt;    // [T, mt]
  uint16_t* out;           // bf16 [T, H]
  uint32_t* status;
};
cudaError_t launch_gateup(const GemmParams& p, cudaStream_t stream);
cudaError_t launch_down(const GemmParams& p, cudaStream_t stream);

struct PrepareParams {
  const uint8_t* codes;    // [E][R][K/2]
  const uint8_t* scales;   // [E][R][K/32]
  int E, R, K, Kp, groups, rows_per_group, mt, kg;
  uint8_t* dst_codes;
  uint8_t* dst_scales;
  uint32_t* flag;          // set to 1 when a scale byte is 255
};
cudaError_t launch_prepare(const PrepareParams& p, cudaStream_t stream);

struct HiddenDequantParams {
  const int32_t* perm;
  const TileEntry* tiles;
  const int32_t* num_tiles;
  int I, bm, max_tiles, kg;
  const uint8_t *h_hi, *h_lo, *sf_hi, *sf_lo;
  float* out;              // [T*k, I]
};
cudaError_t launch_hidden_dequant(const HiddenDequantParams& p, cudaStream_t stream);

}  // namespace moe
