// Launch parameters and launchers of the MoE kernels (internal to the library).
#pragma once

#include <cuda.h>

#include <atomic>
#include <mutex>

#include "moe_common.cuh"
#include "moe_norm.cuh"

namespace moe {

constexpr int kMaxDevices = 64;  // devices with a per-device host-side cache entry

// Raises a kernel's dynamic shared-memory limit on the current device to at least
// `bytes`.  The limit is a per-device function attribute, so it is set once per
// device and increase.  Host threads making their first calls at the same time are
// serialised by a lock; later calls read the published value without it.
class SmemOptIn {
 public:
  template <typename Kern>
  cudaError_t ensure(Kern kern, int bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (done_[dev].load(std::memory_order_acquire) >= bytes) return cudaSuccess;
    std::lock_guard<std::mutex> lock(mu_);
    if (done_[dev].load(std::memory_order_relaxed) >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done_[dev].store(bytes, std::memory_order_release);
    return e;
  }

 private:
  std::atomic<int> done_[kMaxDevices] = {};
  std::mutex mu_;
};

// Launches `kern` with programmatic stream serialization: it may begin while the
// previous kernel on the stream finishes; the kernel itself waits (pdl_wait) before
// it touches memory that kernel produced.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Synchronises `stream`, reads the device status word at `word` (a device address)
// into *status and, when it is non-zero, zero-fills `clear_bytes` bytes from `word`
// (the word itself and whatever the timed-out kernels may have left behind).
// Returns MOE_OK, MOE_ERR_DEVICE_TIMEOUT (a bit was set) or MOE_ERR_CUDA.
int read_and_clear_status(void* word, size_t clear_bytes, cudaStream_t stream, int* status);

// Route flags (the public MOE_ROUTE_* values) -> gating variant, or -1 for a bad set.
constexpr int kRouteFlagFromLogits = 1, kRouteFlagSoftmaxAll = 2, kRouteFlagSigmoid = 4;
inline int gating_from_flags(int flags) {
  if (flags & ~(kRouteFlagFromLogits | kRouteFlagSoftmaxAll | kRouteFlagSigmoid)) return -1;
  const bool all = (flags & kRouteFlagSoftmaxAll) != 0, sig = (flags & kRouteFlagSigmoid) != 0;
  if (all && sig) return -1;
  return all ? kGatingSoftmaxAll : sig ? kGatingSigmoid : kGatingSoftmaxTopk;
}

// Optional RMSNorm + residual in front of the layer (norm_w null: x is the input).
struct NormArgs {
  const uint16_t* residual;  // bf16 [T, H]
  const uint16_t* norm_w;    // bf16 [H]
  float eps;
};

struct RouteParams {
  const uint16_t* x;        // bf16 [T, H]
  const uint16_t* w_router; // bf16 [E, H]
  const float* bias;        // f32 [E] or null
  int T, H, E, k;
  int from_logits;          // logits are an input
  int gating;               // kGatingSoftmaxTopk / kGatingSoftmaxAll / kGatingSigmoid
  int experts_per_block;    // experts per block slice (multiple of 8)
  float* logits;            // f32 [T, E]
  int32_t* topk_idx;        // i32 [T, k]
  float* topk_w;            // f32 [T, k]
  uint32_t* sync;           // arrival counters [ceil(T/8) + 1], zero between calls
  int build_table;          // also build the tile table (last block)
  int bm;
  int32_t *counts, *offsets, *perm, *inv_perm, *num_tiles;
  int pad_inv;              // inv_perm holds padded rows (tile x bm + row in tile), not sorted rows
  TileEntry* tiles;
  uint32_t* status;
  NormArgs norm;            // the router sees y = RMSNorm(x + residual) (norm.norm_w set)
};

cudaError_t launch_route(const RouteParams& p, cudaStream_t stream);
cudaError_t launch_tile_table(const int32_t* idx, int Tk, int E, int bm, int32_t* counts, int32_t* offsets,
                              int32_t* perm, int32_t* inv_perm, TileEntry* tiles, int32_t* num_tiles,
                              cudaStream_t stream);

// Four-term E2M1 encoding of every token's activation row, token major.
struct EncodeXParams {
  const uint16_t* x;       // bf16 [T, H]
  int T, H;
  uint8_t* q;              // [kg][T][kTerms][64 bytes]: packed E2M1 codes (low nibble first)
  uint32_t* sf;            // [kg][T][kTerms]: E8M0 exponents of the 4 MX blocks of a K group
  int wait_at_end;         // dependency wait after the encoding (the launch before it already
                           // waited for earlier work), so this launch completes after that one
  // permute after the wait (needs wait_at_end): the encoded rows go straight to the
  // tile rows of the token's k assignments instead of q / sf
  int scatter;
  const int32_t* topk_idx;    // [T, k]
  const int32_t* pad_row;     // [T*k]: padded row of each assignment (tile x bm + row in tile)
  int E, k, bm, max_tiles, kg_tile;
  uint8_t* q_tile;            // GatherXParams::q layout
  uint8_t* sf_tile;           // GatherXParams::sf layout
  NormArgs norm;              // encode y = RMSNorm(x + residual) instead of x (norm.norm_w set)
};
cudaError_t launch_encode_x(const EncodeXParams& p, cudaStream_t stream);

// The permute step of the bf16-weight layer: after routing, every token's bf16 row
// goes to the tile rows of its k assignments (act16_offset layout).  Its x loads
// are issued before the dependency wait (routing waited for earlier work).
struct ScatterX16Params {
  const uint16_t* x;          // bf16 [T, H]
  int T, H, E, k, bm, max_tiles;
  const int32_t* topk_idx;    // [T, k]
  const int32_t* pad_row;     // [T*k]: padded row of each assignment (tile x bm + row in tile)
  uint8_t* q_tile;            // act16_offset layout
};
cudaError_t launch_scatter_x16(const ScatterX16Params& p, cudaStream_t stream);

// The permute step: encoded x rows copied from token order into the tile order of
// the gate/up GEMM's B operand.
struct GatherXParams {
  const uint8_t* xt_q;     // [kg][T][kTerms][64 bytes] (EncodeXParams::q)
  const uint32_t* xt_sf;   // [kg][T][kTerms]
  const int32_t* perm;
  const TileEntry* tiles;
  const int32_t* num_tiles;
  int T, k, bm, max_tiles, kg;
  uint8_t* q;              // [kg][max_tiles][kTerms][bm][64 bytes]
  uint8_t* sf;             // [max_tiles][kg][512 * act_sf_atoms(bm)]
};
cudaError_t launch_gather_x(const GatherXParams& p, cudaStream_t stream);

struct GemmParams {
  // operand tensor maps (TMA)
  CUtensorMap tm_w;        // weights: packed E2M1 codes, row major [E*groups][rows][K/2 B]
  // activations (x in tile order, or h): packed E2M1 terms, act_offset layout
  // [stages][max_tiles][kTerms*bm rows][128 B], each (stage, tile) image pre-swizzled
  const uint8_t* act_q;
  const uint8_t* w_sf;     // weight scale atoms [E][groups][mt][kg_sf][512]
  const uint8_t* act_sf;   // activation scale atoms [max_tiles][kg_sf][512 * act_sf_atoms]
  const TileEntry* tiles;
  const int32_t* num_tiles;
  const int32_t* perm;
  int T, H, I, E, k, bm, max_tiles;
  int K;                   // contraction length (H for gate/up, I for down)
  int kg;                  // pipeline stages along K (K / gemm_kstage(bm), rounded up)
  int kg_sf;               // K groups of 128 (scale atoms) along K, rounded up to even
  int mt;                  // M units of the output features (M tiles, or pairs of them)
  int rows_out;            // output features (I for gate/up, H for down)
  int w_groups;            // 2 (gate, up) or 1 (down)
  int w_mt;                // 128-row M tiles per group of the prepared weights
  int m_pair;              // down: a unit covers the M tiles 2 mt and 2 mt + 1
  int group_tiles;         // tiles per raster group
  // gate/up epilogue outputs (four-term E2M1 h)
  uint8_t *h_q, *h_sf;
  int kg_out;              // K groups of 128 of h along I, rounded up to even
  // down epilogue
  const float* topk_w;
  float* slots;            // f32 [T*k, H]: w_tj * y_tj per assignment
  int grid;                // persistent CTAs (<= kMaxCtas)
  uint32_t* status;
  int w16;                 // bf16 weights and activations (act16_offset layout, no scales)
  const uint8_t* w_tiles;  // bf16 weights prepared by moe_prepare_weights_bf16 (W16 kernels)
  uint64_t wait_ns;        // limit of each pipeline wait (ns); teardown drains wait up to 1 s
};

// Limit of the expert GEMMs' pipeline waits for launches made from now on (ns; the
// default is 1 s), set by moe_set_wait_limit_ns.
uint64_t gemm_wait_limit_ns();
cudaError_t launch_gateup(const GemmParams& p, cudaStream_t stream);
cudaError_t launch_down(const GemmParams& p, cudaStream_t stream);

// Weighted top-k combine + unpermute of the down GEMM's slots into bf16 rows.
struct CombineParams {
  const float* slots;      // f32 [T*k, H], slot t*k + j = w_tj * y_tj
  int T, H, k;
  uint16_t* out;           // bf16 [T, H]
  // optional residual stream output bf16(x + residual) (the norm step's sum); written
  // here, after every reader of x and residual has finished, so it may alias either
  const uint16_t* x;
  const uint16_t* residual;
  uint16_t* residual_out;
};
cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream);

struct PrepareParams {
  const uint8_t* codes;    // [E][R][K/2]
  const uint8_t* scales;   // [E][R][K/32]
  int E, R, K, groups, rows_per_group, mt, kg;
  uint8_t* dst_codes;
  uint8_t* dst_scales;
  uint32_t* flag;          // set to 1 when a scale byte is 255
};
cudaError_t launch_prepare(const PrepareParams& p, cudaStream_t stream);

// bf16 weights into swizzled 128-row x 64-value tiles (moe_prepare_weights_bf16).
constexpr int kW16TileBytes = kMTile * 128;  // one prepared tile: 128 rows x 128 bytes
struct PrepareBf16Params {
  const uint16_t* w;       // [E][groups * rows_per_group][K]
  int E, groups, rows_per_group, K;
  int mt, ks;              // tiles per group along rows (rounded up) and along K
  uint8_t* dst;            // [E * groups * mt * ks + 1][16 KB]
};
cudaError_t launch_prepare_bf16(const PrepareBf16Params& p, cudaStream_t stream);

struct HiddenDequantParams {
  const int32_t* perm;
  const TileEntry* tiles;
  const int32_t* num_tiles;
  int I, bm, max_tiles, kg;
  const uint8_t *h_q, *sf;
  float* out;              // [T*k, I]
};
cudaError_t launch_hidden_dequant(const HiddenDequantParams& p, cudaStream_t stream);

}  // namespace moe
