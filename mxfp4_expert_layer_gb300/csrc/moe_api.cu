// C ABI of the MXFP4 MoE layer: argument checks, workspace carving, TMA tensor
// maps and the launch sequence of the hot path.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>

#include "moe_common.cuh"
#include "moe_kernels.cuh"

using namespace moe;

namespace {

// ------------------------------------------------------------------ checks
bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

constexpr int kMaxDim = 8192;     // H (a routing row, an encoder block of the norm step)
constexpr int kMaxInter = 16384;  // I (Mixtral-8x7B's is 14336)

int check_shape(int T, int H, int I, int E, int k) {
  if (T < 1 || H < 32 || I < 32 || E < 1 || k < 1) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (H % 32 || I % 32 || H > kMaxDim || I > kMaxInter) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (E > kMaxExperts || k > E || k > kMaxTopK) return MOE_ERR_UNSUPPORTED_SHAPE;
  if ((long long)T * k > (1LL << 24)) return MOE_ERR_UNSUPPORTED_SHAPE;
  return MOE_OK;
}

int resolve_bm(int T, int k, int E, int tile_rows) {
  if (tile_rows == 0) return tile_rows_policy(T, k, E);
  if (tile_rows == 16 || tile_rows == 64 || tile_rows == 128) return tile_rows;
  return -1;
}

// ------------------------------------------------------------------ tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

struct MapKey {
  const void* ptr;
  int dtype, rank;
  cuuint64_t dims[4], strides[3];
  cuuint32_t box[4];
  bool operator==(const MapKey& o) const { return std::memcmp(this, &o, sizeof(MapKey)) == 0; }
};

struct MapCache {
  static constexpr int kSlots = 64;
  MapKey keys[kSlots];
  CUtensorMap maps[kSlots];
  bool used[kSlots] = {};
  int next = 0;
  std::mutex mu;
};

MapCache& map_cache() {
  static MapCache c;
  return c;
}

// Encodes (or fetches from a small cache) a tiled tensor map; false on failure.
bool make_map(CUtensorMap* out, const void* ptr, CUtensorMapDataType dtype, int rank, const cuuint64_t* dims,
              const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle swizzle) {
  MapKey key;
  std::memset(&key, 0, sizeof key);
  key.ptr = ptr;
  key.dtype = (int)dtype;
  key.rank = rank * 16 + (int)swizzle;
  for (int i = 0; i < rank; ++i) {
    key.dims[i] = dims[i];
    key.box[i] = box[i];
    if (i < rank - 1) key.strides[i] = strides[i];
  }
  MapCache& c = map_cache();
  std::lock_guard<std::mutex> lock(c.mu);
  for (int i = 0; i < MapCache::kSlots; ++i) {
    if (c.used[i] && c.keys[i] == key) {
      *out = c.maps[i];
      return true;
    }
  }
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = enc(out, dtype, rank, const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  const int slot = c.next;
  c.next = (c.next + 1) % MapCache::kSlots;
  c.keys[slot] = key;
  c.maps[slot] = *out;
  c.used[slot] = true;
  return true;
}

// MXFP4 codes of one prepared family, row major, as a 3-D byte map {K/2 bytes, rows
// per group, E * groups}: one box = 128 rows x (one pipeline stage of K: 128 bytes =
// 256 codes with the 128-byte swizzle, or 64 bytes with the 64-byte swizzle), kept
// packed in shared memory.  Parts of a box past K or past the group's rows are
// outside the map and read as zero without touching memory.
bool weight_map(CUtensorMap* out, const void* prepared, const PreparedLayout& P, int bm) {
  const cuuint64_t row_bytes = (cuuint64_t)P.K / 2;
  cuuint64_t dims[3] = {row_bytes, (cuuint64_t)P.rows_per_group, (cuuint64_t)P.E * P.groups};
  cuuint64_t strides[2] = {row_bytes, row_bytes * P.rows_per_group};
  const int kb = gemm_kstage(bm) / 2;
  cuuint32_t box[3] = {(cuuint32_t)kb, (cuuint32_t)kMTile, 1};
  return make_map(out, prepared, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, dims, strides, box,
                  kb == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// Records a caller event; while the stream is being captured the record is made an
// external event node so the event is recorded on every replay of the graph.
cudaError_t record_event(void* ev, cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(s, &cs);
  if (e != cudaSuccess) return e;
  if (cs == cudaStreamCaptureStatusActive)
    return cudaEventRecordWithFlags(reinterpret_cast<cudaEvent_t>(ev), s, cudaEventRecordExternal);
  return cudaEventRecord(reinterpret_cast<cudaEvent_t>(ev), s);
}

// One persistent GEMM CTA per SM of the current device (cached per device; every
// thread computes the same value, so publishing it needs no lock).
int persistent_ctas() {
  static std::atomic<int> cached[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return kMaxCtas;
  if (dev >= 0 && dev < kMaxDevices) {
    const int c = cached[dev].load(std::memory_order_relaxed);
    if (c) return c;
  }
  int sms = kMaxCtas;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) sms = kMaxCtas;
  if (sms > kMaxCtas) sms = kMaxCtas;
  if (sms < 1) sms = 1;
  if (dev >= 0 && dev < kMaxDevices) cached[dev].store(sms, std::memory_order_relaxed);
  return sms;
}

// ------------------------------------------------------------------ stage bodies
// Per-token activation encoding.
int run_encode_x(const uint16_t* x, int T, int H, void* ws, const WsLayout& L, cudaStream_t stream) {
  EncodeXParams q{};
  q.x = x;
  q.T = T; q.H = H;
  q.q = ws_ptr<uint8_t>(ws, L.xt_q);
  q.sf = ws_ptr<uint32_t>(ws, L.xt_sf);
  return cuda_status(launch_encode_x(q, stream));
}

// Per-token activation encoding that overlaps the routing launch before it, waits
// for it, and writes the encoded rows straight into tile order (the permute step).
int run_encode_permute_x(const uint16_t* x, const int32_t* idx, int T, int H, int E, int k, int bm, void* ws,
                         const WsLayout& L, cudaStream_t stream, const NormArgs& norm = NormArgs{}) {
  EncodeXParams q{};
  q.x = x;
  q.norm = norm;
  q.T = T; q.H = H;
  q.wait_at_end = 1;
  q.scatter = 1;
  q.topk_idx = idx;
  q.pad_row = ws_ptr<int32_t>(ws, L.inv_perm);  // the routing wrote padded rows there
  q.E = E; q.k = k; q.bm = bm; q.max_tiles = L.max_tiles; q.kg_tile = L.kg_h;
  q.q_tile = ws_ptr<uint8_t>(ws, L.x_q);
  q.sf_tile = ws_ptr<uint8_t>(ws, L.x_sf);
  return cuda_status(launch_encode_x(q, stream));
}

// The permute (gather of the token-order encoded rows into tile order).
int run_gather_x(const int32_t* perm, const TileEntry* tiles, const int32_t* num_tiles, int bm, int T, int H, int k,
                 void* ws, const WsLayout& L, cudaStream_t stream) {
  GatherXParams gx{};
  gx.xt_q = ws_ptr<uint8_t>(ws, L.xt_q);
  gx.xt_sf = ws_ptr<uint32_t>(ws, L.xt_sf);
  gx.perm = perm;
  gx.tiles = tiles;
  gx.num_tiles = num_tiles;
  gx.T = T; gx.k = k; gx.bm = bm; gx.max_tiles = L.max_tiles; gx.kg = L.kg_h;
  gx.q = ws_ptr<uint8_t>(ws, L.x_q);
  gx.sf = ws_ptr<uint8_t>(ws, L.x_sf);
  return cuda_status(launch_gather_x(gx, stream));
}

// The gate/up GEMM + SwiGLU over x in tile order (run_gather_x or run_encode_permute_x).
int run_gateup(const int32_t* perm, const TileEntry* tiles, const int32_t* num_tiles, int bm, const void* w_gateup,
               int T, int H, int I, int E, int k, void* ws, const WsLayout& L, cudaStream_t stream) {
  const PreparedLayout P = make_prepared_layout(E, 2 * I, H, 2);
  GemmParams g{};
  if (!weight_map(&g.tm_w, w_gateup, P, bm)) return MOE_ERR_CUDA;
  g.act_q = ws_ptr<uint8_t>(ws, L.x_q);
  g.w_sf = static_cast<const uint8_t*>(w_gateup) + P.scales_off;
  g.act_sf = ws_ptr<uint8_t>(ws, L.x_sf);
  g.tiles = tiles;
  g.num_tiles = num_tiles;
  g.perm = perm;
  g.T = T; g.H = H; g.I = I; g.E = E; g.k = k; g.bm = bm; g.max_tiles = L.max_tiles;
  g.K = H;
  g.kg = ceil_div(H, gemm_kstage(bm));
  g.kg_sf = P.kg;
  g.mt = L.mt_i;
  g.rows_out = I;
  g.w_groups = 2;
  g.w_mt = P.mt;
  g.group_tiles = bm >= 128 ? 32 : (bm >= 64 ? 16 : 1);
  g.h_q = ws_ptr<uint8_t>(ws, L.h_q);
  g.h_sf = ws_ptr<uint8_t>(ws, L.h_sf);
  g.kg_out = L.kg_i;
  g.grid = persistent_ctas();
  g.status = ws_ptr<uint32_t>(ws, L.status);
  g.wait_ns = gemm_wait_limit_ns();
  return cuda_status(launch_gateup(g, stream));
}

// The down GEMM (w * y into the slots), then the combine; `between` (may be null) is
// called after the GEMM's launch and before the combine's.
template <typename Between>
int run_down(const int32_t* perm, const TileEntry* tiles, const int32_t* num_tiles, int bm, const float* topk_w,
             const void* w_down, int T, int H, int I, int E, int k, void* ws, const WsLayout& L, uint16_t* out,
             cudaStream_t stream, Between between, const uint16_t* x = nullptr, const uint16_t* residual = nullptr,
             uint16_t* residual_out = nullptr) {
  const PreparedLayout P = make_prepared_layout(E, H, I, 1);
  GemmParams g{};
  if (!weight_map(&g.tm_w, w_down, P, bm)) return MOE_ERR_CUDA;
  g.act_q = ws_ptr<uint8_t>(ws, L.h_q);
  g.w_sf = static_cast<const uint8_t*>(w_down) + P.scales_off;
  g.act_sf = ws_ptr<uint8_t>(ws, L.h_sf);
  g.tiles = tiles;
  g.num_tiles = num_tiles;
  g.perm = perm;
  g.T = T; g.H = H; g.I = I; g.E = E; g.k = k; g.bm = bm; g.max_tiles = L.max_tiles;
  g.K = I;
  g.kg = ceil_div(I, gemm_kstage(bm));
  g.kg_sf = P.kg;
  // pairs of M tiles per unit when there are units enough to keep every SM busy
  g.m_pair = (long long)std::min(E, T * k) * ceil_div(L.mt_h, 2) >= 2LL * persistent_ctas() ? 1 : 0;
  g.mt = g.m_pair ? ceil_div(L.mt_h, 2) : L.mt_h;
  g.w_mt = P.mt;
  g.rows_out = H;
  g.w_groups = 1;
  g.group_tiles = bm >= 128 ? 32 : (bm >= 64 ? 16 : 1);
  g.topk_w = topk_w;
  g.slots = ws_ptr<float>(ws, L.slots);
  g.grid = persistent_ctas();
  g.status = ws_ptr<uint32_t>(ws, L.status);
  g.wait_ns = gemm_wait_limit_ns();
  int st = cuda_status(launch_down(g, stream));
  if (st != MOE_OK) return st;
  st = between();
  if (st != MOE_OK) return st;
  CombineParams c{};
  c.slots = g.slots;
  c.T = T; c.H = H; c.k = k;
  c.out = out;
  c.x = x;
  c.residual = residual;
  c.residual_out = residual_out;
  return cuda_status(launch_combine(c, stream));
}

}  // namespace

namespace {
constexpr uint64_t kDefaultWaitNs = 1000000000ull;  // 1 s
std::atomic<uint64_t> g_wait_limit_ns{kDefaultWaitNs};
}  // namespace

uint64_t moe::gemm_wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }

int moe::read_and_clear_status(void* word, size_t clear_bytes, cudaStream_t stream, int* status) {
  uint32_t h = 0;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemcpy(&h, word, sizeof h, cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (h && cudaMemset(word, 0, clear_bytes) != cudaSuccess) return MOE_ERR_CUDA;
  *status = (int)h;
  return h ? MOE_ERR_DEVICE_TIMEOUT : MOE_OK;
}

namespace {

static_assert(MOE_ROUTE_FROM_LOGITS == kRouteFlagFromLogits && MOE_ROUTE_GATING_SOFTMAX_ALL == kRouteFlagSoftmaxAll &&
                  MOE_ROUTE_GATING_SIGMOID == kRouteFlagSigmoid,
              "route flag values");

RouteParams route_params(const uint16_t* x, const uint16_t* w_router, const float* bias, int T, int H, int E, int k,
                         float* logits, int from_logits, int32_t* idx, float* w, void* ws, const WsLayout& L) {
  RouteParams r{};
  r.x = x;
  r.w_router = w_router;
  r.bias = bias;
  r.T = T; r.H = H; r.E = E; r.k = k;
  r.from_logits = from_logits;
  r.experts_per_block = T <= 64 ? 8 : 32;
  r.logits = logits;
  r.topk_idx = idx;
  r.topk_w = w;
  r.sync = ws_ptr<uint32_t>(ws, L.route_sync);
  r.status = ws_ptr<uint32_t>(ws, L.status);
  return r;
}

}  // namespace

extern "C" {

const char* moe_error_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument (null pointer, misalignment or bad flag)";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA launch or driver call failed";
    case MOE_ERR_DEVICE_TIMEOUT: return "a bounded device-side wait timed out";
    case MOE_ERR_NAN_SCALE: return "E8M0 scale 255 (NaN) in the weights";
    default: return "unknown status";
  }
}

size_t moe_prepared_weight_bytes(int E, int rows, int K, int kind) {
  if (E < 1 || rows < 1 || K < 32 || K % 32 || (kind != MOE_WEIGHTS_GATEUP && kind != MOE_WEIGHTS_DOWN)) return 0;
  const int groups = kind == MOE_WEIGHTS_GATEUP ? 2 : 1;
  if (rows % (groups * 32)) return 0;
  return make_prepared_layout(E, rows, K, groups).total;
}

int moe_prepare_weights(const uint8_t* codes, const uint8_t* scales, int E, int rows, int K, int kind, void* dst,
                        size_t dst_bytes, moe_stream_t stream) {
  const size_t need = moe_prepared_weight_bytes(E, rows, K, kind);
  if (need == 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!codes || !scales || !dst || !aligned(codes, 16) || !aligned(dst, 256)) return MOE_ERR_INVALID_ARG;
  if (dst_bytes < need) return MOE_ERR_WORKSPACE_TOO_SMALL;
  const int groups = kind == MOE_WEIGHTS_GATEUP ? 2 : 1;
  const PreparedLayout P = make_prepared_layout(E, rows, K, groups);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint32_t* flag = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(dst) + P.flag_off);
  if (cudaMemsetAsync(flag, 0, 256, s) != cudaSuccess) return MOE_ERR_CUDA;
  PrepareParams pp{};
  pp.codes = codes;
  pp.scales = scales;
  pp.E = E; pp.R = rows; pp.K = K; pp.groups = groups; pp.rows_per_group = P.rows_per_group;
  pp.mt = P.mt; pp.kg = P.kg;
  pp.dst_codes = static_cast<uint8_t*>(dst);
  pp.dst_scales = static_cast<uint8_t*>(dst) + P.scales_off;
  pp.flag = flag;
  if (launch_prepare(pp, s) != cudaSuccess) return MOE_ERR_CUDA;
  uint32_t h = 0;
  if (cudaMemcpyAsync(&h, flag, sizeof h, cudaMemcpyDeviceToHost, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  return h ? MOE_ERR_NAN_SCALE : MOE_OK;
}

size_t moe_prepared_weight_bytes_bf16(int E, int rows, int K, int kind) {
  if (E < 1 || rows < 1 || K < 64 || K % 64 || (kind != MOE_WEIGHTS_GATEUP && kind != MOE_WEIGHTS_DOWN)) return 0;
  const int groups = kind == MOE_WEIGHTS_GATEUP ? 2 : 1;
  if (rows % groups) return 0;
  const size_t tiles = (size_t)E * groups * ceil_div(rows / groups, kMTile) * (K / 64);
  return (tiles + 1) * kW16TileBytes;
}

int moe_prepare_weights_bf16(const uint16_t* w, int E, int rows, int K, int kind, void* dst, size_t dst_bytes,
                             moe_stream_t stream) {
  const size_t need = moe_prepared_weight_bytes_bf16(E, rows, K, kind);
  if (need == 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!w || !dst || !aligned(w, 16) || !aligned(dst, 256)) return MOE_ERR_INVALID_ARG;
  if (dst_bytes < need) return MOE_ERR_WORKSPACE_TOO_SMALL;
  PrepareBf16Params pp{};
  pp.w = w;
  pp.E = E;
  pp.groups = kind == MOE_WEIGHTS_GATEUP ? 2 : 1;
  pp.rows_per_group = rows / pp.groups;
  pp.K = K;
  pp.mt = ceil_div(pp.rows_per_group, kMTile);
  pp.ks = K / 64;
  pp.dst = static_cast<uint8_t*>(dst);
  return cuda_status(launch_prepare_bf16(pp, reinterpret_cast<cudaStream_t>(stream)));
}

int moe_tile_rows(int T, int k, int E) {
  if (T < 1 || k < 1 || E < 1) return 0;
  return tile_rows_policy(T, k, E);
}

int moe_max_tiles(int T, int k, int E, int tile_rows) {
  if (T < 1 || k < 1 || E < 1 || tile_rows < 1) return 0;
  return max_tiles_bound(T, k, E, tile_rows);
}

size_t moe_workspace_bytes(int T, int H, int I, int E, int k) {
  if (check_shape(T, H, I, E, k) != MOE_OK) return 0;
  // room for both layers' layouts (the bf16 layer may use 256-row tiles)
  const size_t a = make_ws_layout(T, H, I, E, k, tile_rows_policy(T, k, E)).total;
  const size_t b = make_ws_layout(T, H, I, E, k, tile_rows_policy_bf16(T, k, E)).total;
  return a > b ? a : b;
}

int moe_route(const uint16_t* x, const uint16_t* w_router, const float* router_bias, int T, int H, int E, int k,
              float* logits, int flags, int32_t* topk_idx, float* topk_w, void* workspace, size_t workspace_bytes,
              moe_stream_t stream) {
  const int gating = gating_from_flags(flags);
  if (gating < 0) return MOE_ERR_INVALID_ARG;
  const int from_logits = (flags & MOE_ROUTE_FROM_LOGITS) ? 1 : 0;
  const int Hs = from_logits ? 32 : H;
  int st = check_shape(T, Hs, 32, E, k);
  if (st != MOE_OK) return st;
  if (!logits || !topk_idx || !topk_w || !workspace || !aligned(workspace, 256)) return MOE_ERR_INVALID_ARG;
  if (!from_logits && (!x || !w_router || !aligned(x, 16) || !aligned(w_router, 16))) return MOE_ERR_INVALID_ARG;
  const WsLayout L = make_ws_layout(T, 32, 32, E, k, tile_rows_policy(T, k, E));
  if (workspace_bytes < L.route_sync + sizeof(uint32_t) * (size_t)(ceil_div(T, 8) + 1))
    return MOE_ERR_WORKSPACE_TOO_SMALL;
  RouteParams r = route_params(x, w_router, router_bias, T, Hs, E, k, logits, from_logits, topk_idx, topk_w,
                               workspace, L);
  r.build_table = 0;
  r.gating = gating;
  return cuda_status(launch_route(r, reinterpret_cast<cudaStream_t>(stream)));
}

int moe_build_tile_table(const int32_t* topk_idx, int T, int k, int E, int tile_rows, int32_t* counts,
                         int32_t* offsets, int32_t* perm, int32_t* inv_perm, int32_t* tiles, int32_t* num_tiles,
                         moe_stream_t stream) {
  if (T < 1 || k < 1 || E < 1 || E > kMaxExperts || k > E || (long long)T * k > (1LL << 24))
    return MOE_ERR_UNSUPPORTED_SHAPE;
  const int bm = resolve_bm(T, k, E, tile_rows);
  if (bm < 0) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!topk_idx || !counts || !offsets || !perm || !inv_perm || !tiles || !num_tiles || !aligned(tiles, 16))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_tile_table(topk_idx, T * k, E, bm, counts, offsets, perm, inv_perm,
                                       reinterpret_cast<TileEntry*>(tiles), num_tiles,
                                       reinterpret_cast<cudaStream_t>(stream)));
}

int moe_mxfp4_gateup_swiglu(const uint16_t* x, const int32_t* perm, const int32_t* tiles, const int32_t* num_tiles,
                            int tile_rows, const void* w_gateup, int T, int H, int I, int E, int k, void* workspace,
                            size_t workspace_bytes, moe_stream_t stream) {
  int st = check_shape(T, H, I, E, k);
  if (st != MOE_OK) return st;
  const int bm = resolve_bm(T, k, E, tile_rows);
  if (bm != tile_rows_policy(T, k, E)) return MOE_ERR_UNSUPPORTED_SHAPE;  // workspace is sized for the policy tile
  if (!x || !perm || !tiles || !num_tiles || !w_gateup || !workspace) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(tiles, 16) || !aligned(w_gateup, 256) || !aligned(workspace, 256))
    return MOE_ERR_INVALID_ARG;
  const WsLayout L = make_ws_layout(T, H, I, E, k, bm);
  if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  st = run_encode_x(x, T, H, workspace, L, s);
  if (st != MOE_OK) return st;
  st = run_gather_x(perm, reinterpret_cast<const TileEntry*>(tiles), num_tiles, bm, T, H, k, workspace, L, s);
  if (st != MOE_OK) return st;
  return run_gateup(perm, reinterpret_cast<const TileEntry*>(tiles), num_tiles, bm, w_gateup, T, H, I, E, k,
                    workspace, L, s);
}

int moe_mxfp4_down_combine(const int32_t* perm, const int32_t* tiles, const int32_t* num_tiles, int tile_rows,
                           const float* topk_w, const void* w_down, int T, int H, int I, int E, int k,
                           void* workspace, size_t workspace_bytes, uint16_t* out, moe_stream_t stream) {
  int st = check_shape(T, H, I, E, k);
  if (st != MOE_OK) return st;
  const int bm = resolve_bm(T, k, E, tile_rows);
  if (bm != tile_rows_policy(T, k, E)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!perm || !tiles || !num_tiles || !topk_w || !w_down || !workspace || !out) return MOE_ERR_INVALID_ARG;
  if (!aligned(tiles, 16) || !aligned(w_down, 256) || !aligned(workspace, 256) || !aligned(out, 16))
    return MOE_ERR_INVALID_ARG;
  const WsLayout L = make_ws_layout(T, H, I, E, k, bm);
  if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  return run_down(perm, reinterpret_cast<const TileEntry*>(tiles), num_tiles, bm, topk_w, w_down, T, H, I, E, k,
                  workspace, L, out, reinterpret_cast<cudaStream_t>(stream), [] { return MOE_OK; });
}

int moe_hidden_dequant(const int32_t* perm, const int32_t* tiles, const int32_t* num_tiles, int tile_rows, int T,
                       int H, int I, int E, int k, const void* workspace, size_t workspace_bytes, float* h_out,
                       moe_stream_t stream) {
  int st = check_shape(T, H, I, E, k);
  if (st != MOE_OK) return st;
  const int bm = resolve_bm(T, k, E, tile_rows);
  if (bm != tile_rows_policy(T, k, E)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!perm || !tiles || !num_tiles || !workspace || !h_out) return MOE_ERR_INVALID_ARG;
  const WsLayout L = make_ws_layout(T, H, I, E, k, bm);
  if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  void* ws = const_cast<void*>(workspace);
  HiddenDequantParams hp{};
  hp.perm = perm;
  hp.tiles = reinterpret_cast<const TileEntry*>(tiles);
  hp.num_tiles = num_tiles;
  hp.I = I; hp.bm = bm; hp.max_tiles = L.max_tiles; hp.kg = L.kg_i;
  hp.h_q = ws_ptr<uint8_t>(ws, L.h_q);
  hp.sf = ws_ptr<uint8_t>(ws, L.h_sf);
  hp.out = h_out;
  return cuda_status(launch_hidden_dequant(hp, reinterpret_cast<cudaStream_t>(stream)));
}

static int forward_impl(const uint16_t* x, const uint16_t* w_router, const float* router_bias,
                        const void* w_gateup, const void* w_down, int T, int H, int I, int E, int k,
                        void* workspace, size_t workspace_bytes, uint16_t* out, int32_t* topk_idx_out,
                        float* topk_w_out, void* const* events, moe_stream_t stream, int gating = kGatingSoftmaxTopk,
                        const NormArgs& norm = NormArgs{}, uint16_t* residual_out = nullptr) {
  int st = check_shape(T, H, I, E, k);
  if (st != MOE_OK) return st;
  if (!x || !w_router || !w_gateup || !w_down || !workspace || !out) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(w_router, 16) || !aligned(out, 16) || !aligned(w_gateup, 256) ||
      !aligned(w_down, 256) || !aligned(workspace, 256))
    return MOE_ERR_INVALID_ARG;
  const int bm = tile_rows_policy(T, k, E);
  const WsLayout L = make_ws_layout(T, H, I, E, k, bm);
  if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  void* ws = workspace;
  int32_t* idx = topk_idx_out ? topk_idx_out : ws_ptr<int32_t>(ws, L.idx);
  float* w = topk_w_out ? topk_w_out : ws_ptr<float>(ws, L.w);
  int32_t* perm = ws_ptr<int32_t>(ws, L.perm);
  TileEntry* tiles = ws_ptr<TileEntry>(ws, L.tiles);
  int32_t* num_tiles = ws_ptr<int32_t>(ws, L.num_tiles);

  RouteParams r = route_params(x, w_router, router_bias, T, H, E, k, ws_ptr<float>(ws, L.logits), 0, idx, w, ws, L);
  r.build_table = 1;
  r.gating = gating;
  r.bm = bm;
  r.counts = ws_ptr<int32_t>(ws, L.counts);
  r.offsets = ws_ptr<int32_t>(ws, L.offsets);
  r.perm = perm;
  r.inv_perm = ws_ptr<int32_t>(ws, L.inv_perm);
  r.tiles = tiles;
  r.num_tiles = num_tiles;
  r.pad_inv = 1;  // the permute step reads each assignment's padded row
  r.norm = norm;
  bool ev_ok = true;
  auto mark = [&](int i) {
    if (events && record_event(events[i], s) != cudaSuccess) ev_ok = false;
  };
  // stages: [0] route + top-k + tile table, [1] encode + permute x, [2] gate/up,
  // [3] down, [4] combine.  Routing goes first (it waits for the previous kernel);
  // the encoding overlaps it, waits for it at its end and writes the tile order.
  mark(0);
  if (!ev_ok) return MOE_ERR_INVALID_ARG;
  if (launch_route(r, s) != cudaSuccess) return MOE_ERR_CUDA;
  mark(1);
  st = run_encode_permute_x(x, idx, T, H, E, k, bm, ws, L, s, norm);
  if (st != MOE_OK) return st;
  mark(2);
  st = run_gateup(perm, tiles, num_tiles, bm, w_gateup, T, H, I, E, k, ws, L, s);
  if (st != MOE_OK) return st;
  mark(3);
  st = run_down(perm, tiles, num_tiles, bm, w, w_down, T, H, I, E, k, ws, L, out, s,
                [&] {
                  mark(4);
                  return ev_ok ? MOE_OK : MOE_ERR_INVALID_ARG;
                },
                x, norm.residual, residual_out);
  mark(5);
  return st;
}

int moe_forward(const uint16_t* x, const uint16_t* w_router, const float* router_bias, const void* w_gateup,
                const void* w_down, int T, int H, int I, int E, int k, void* workspace, size_t workspace_bytes,
                uint16_t* out, int32_t* topk_idx_out, float* topk_w_out, moe_stream_t stream) {
  return forward_impl(x, w_router, router_bias, w_gateup, w_down, T, H, I, E, k, workspace, workspace_bytes, out,
                      topk_idx_out, topk_w_out, nullptr, stream);
}

int moe_forward_gated(const uint16_t* x, const uint16_t* w_router, const float* router_bias, const void* w_gateup,
                      const void* w_down, int T, int H, int I, int E, int k, int gating, void* workspace,
                      size_t workspace_bytes, uint16_t* out, int32_t* topk_idx_out, float* topk_w_out,
                      moe_stream_t stream) {
  const int g = gating == 0 ? kGatingSoftmaxTopk : gating_from_flags(gating);
  if (g < 0 || (gating & MOE_ROUTE_FROM_LOGITS)) return MOE_ERR_INVALID_ARG;
  return forward_impl(x, w_router, router_bias, w_gateup, w_down, T, H, I, E, k, workspace, workspace_bytes, out,
                      topk_idx_out, topk_w_out, nullptr, stream, g);
}

int moe_forward_norm(const uint16_t* x, const uint16_t* residual, const uint16_t* norm_weight, float eps,
                     const uint16_t* w_router, const float* router_bias, const void* w_gateup, const void* w_down,
                     int T, int H, int I, int E, int k, int gating, void* workspace, size_t workspace_bytes,
                     uint16_t* out, uint16_t* residual_out, int32_t* topk_idx_out, float* topk_w_out,
                     moe_stream_t stream) {
  const int g = gating == 0 ? kGatingSoftmaxTopk : gating_from_flags(gating);
  if (g < 0 || (gating & MOE_ROUTE_FROM_LOGITS)) return MOE_ERR_INVALID_ARG;
  if (!residual || !norm_weight || !aligned(residual, 16) || !aligned(norm_weight, 16)) return MOE_ERR_INVALID_ARG;
  if (!(eps >= 0.f) || !(eps < 3.0e38f)) return MOE_ERR_INVALID_ARG;  // negative, NaN or infinite
  if (residual_out && (!aligned(residual_out, 16) || residual_out == out)) return MOE_ERR_INVALID_ARG;
  NormArgs norm;
  norm.residual = residual;
  norm.norm_w = norm_weight;
  norm.eps = eps;
  return forward_impl(x, w_router, router_bias, w_gateup, w_down, T, H, I, E, k, workspace, workspace_bytes, out,
                      topk_idx_out, topk_w_out, nullptr, stream, g, norm, residual_out);
}

int moe_forward_bf16(const uint16_t* x, const uint16_t* w_router, const float* router_bias, const uint16_t* w_gateup,
                     const uint16_t* w_down, int T, int H, int I, int E, int k, void* workspace,
                     size_t workspace_bytes, uint16_t* out, int32_t* topk_idx_out, float* topk_w_out,
                     moe_stream_t stream) {
  int st = check_shape(T, H, I, E, k);
  if (st != MOE_OK) return st;
  if (H % 64 || I % 64) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!x || !w_router || !w_gateup || !w_down || !workspace || !out) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(w_router, 16) || !aligned(out, 16) || !aligned(w_gateup, 16) ||
      !aligned(w_down, 16) || !aligned(workspace, 256))
    return MOE_ERR_INVALID_ARG;
  const int bm = tile_rows_policy_bf16(T, k, E);
  const WsLayout L = make_ws_layout(T, H, I, E, k, bm);
  if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  void* ws = workspace;
  int32_t* idx = topk_idx_out ? topk_idx_out : ws_ptr<int32_t>(ws, L.idx);
  float* w = topk_w_out ? topk_w_out : ws_ptr<float>(ws, L.w);
  int32_t* perm = ws_ptr<int32_t>(ws, L.perm);
  TileEntry* tiles = ws_ptr<TileEntry>(ws, L.tiles);
  int32_t* num_tiles = ws_ptr<int32_t>(ws, L.num_tiles);

  // route + top-k + table: the same launch as the MXFP4 layer
  RouteParams r = route_params(x, w_router, router_bias, T, H, E, k, ws_ptr<float>(ws, L.logits), 0, idx, w, ws, L);
  r.build_table = 1;
  r.bm = bm;
  r.counts = ws_ptr<int32_t>(ws, L.counts);
  r.offsets = ws_ptr<int32_t>(ws, L.offsets);
  r.perm = perm;
  r.inv_perm = ws_ptr<int32_t>(ws, L.inv_perm);
  r.tiles = tiles;
  r.num_tiles = num_tiles;
  r.pad_inv = 1;  // the permute step reads each assignment's padded row
  if (launch_route(r, s) != cudaSuccess) return MOE_ERR_CUDA;

  // permute: bf16 rows of x into tile order
  ScatterX16Params sx{};
  sx.x = x;
  sx.T = T; sx.H = H; sx.E = E; sx.k = k; sx.bm = bm; sx.max_tiles = L.max_tiles;
  sx.topk_idx = idx;
  sx.pad_row = r.inv_perm;
  sx.q_tile = ws_ptr<uint8_t>(ws, L.x_q);
  if (launch_scatter_x16(sx, s) != cudaSuccess) return MOE_ERR_CUDA;

  // gate/up + SwiGLU (h in bf16, tile order), then down into the slots
  GemmParams g{};
  g.w_tiles = reinterpret_cast<const uint8_t*>(w_gateup);
  g.w16 = 1;
  g.act_q = ws_ptr<uint8_t>(ws, L.x_q);
  g.tiles = tiles;
  g.num_tiles = num_tiles;
  g.perm = perm;
  g.T = T; g.H = H; g.I = I; g.E = E; g.k = k; g.bm = bm; g.max_tiles = L.max_tiles;
  g.K = H;
  g.kg = H / 64;
  g.mt = ceil_div(I, kMTile);
  g.rows_out = I;
  g.w_groups = 2;
  g.w_mt = g.mt;
  g.group_tiles = bm >= 128 ? 32 : (bm >= 64 ? 16 : 1);
  g.h_q = ws_ptr<uint8_t>(ws, L.h_q);
  g.grid = persistent_ctas();
  g.status = ws_ptr<uint32_t>(ws, L.status);
  g.wait_ns = gemm_wait_limit_ns();
  st = cuda_status(launch_gateup(g, s));
  if (st != MOE_OK) return st;

  GemmParams d{};
  d.w_tiles = reinterpret_cast<const uint8_t*>(w_down);
  d.w16 = 1;
  d.act_q = ws_ptr<uint8_t>(ws, L.h_q);
  d.tiles = tiles;
  d.num_tiles = num_tiles;
  d.perm = perm;
  d.T = T; d.H = H; d.I = I; d.E = E; d.k = k; d.bm = bm; d.max_tiles = L.max_tiles;
  d.K = I;
  d.kg = I / 64;
  // 64- and 128-row tiles: two M tiles per unit share each stage's activation tile
  // (BM x 128 bytes, a third or a half of an unpaired stage), when the paired units
  // still fill the GPU twice over (measured at Mixtral shapes: pairs 7% faster at
  // 2048 tokens, 32 tiles; 5% slower at 512 tokens, 8 tiles, where 128 paired units
  // leave SMs idle).  Tiles are estimated from the token count.
  d.w_mt = ceil_div(H, kMTile);
  {
    const long long est_tiles = std::max<long long>(std::min(E, T * k), (long long)T * k / bm);
    d.m_pair = (bm >= 64 && bm <= 128 && est_tiles * ceil_div(d.w_mt, 2) >= 2LL * persistent_ctas()) ? 1 : 0;
  }
  d.mt = d.m_pair ? ceil_div(d.w_mt, 2) : d.w_mt;
  d.rows_out = H;
  d.w_groups = 1;
  d.group_tiles = bm >= 128 ? 32 : (bm >= 64 ? 16 : 1);
  d.topk_w = w;
  d.slots = ws_ptr<float>(ws, L.slots);
  d.grid = persistent_ctas();
  d.status = ws_ptr<uint32_t>(ws, L.status);
  d.wait_ns = gemm_wait_limit_ns();
  st = cuda_status(launch_down(d, s));
  if (st != MOE_OK) return st;
  CombineParams c{};
  c.slots = d.slots;
  c.T = T; c.H = H; c.k = k;
  c.out = out;
  return cuda_status(launch_combine(c, s));
}

int moe_forward_timed(const uint16_t* x, const uint16_t* w_router, const float* router_bias, const void* w_gateup,
                      const void* w_down, int T, int H, int I, int E, int k, void* workspace,
                      size_t workspace_bytes, uint16_t* out, int32_t* topk_idx_out, float* topk_w_out,
                      void* const* events, moe_stream_t stream) {
  if (!events) return MOE_ERR_INVALID_ARG;
  return forward_impl(x, w_router, router_bias, w_gateup, w_down, T, H, I, E, k, workspace, workspace_bytes, out,
                      topk_idx_out, topk_w_out, events, stream);
}

int moe_forward_launches(int T, int H, int I, int E, int k) {
  if (check_shape(T, H, I, E, k) != MOE_OK) return 0;
  return 5;  // route + table, encode + permute x, gate/up, down, combine
}

int moe_set_wait_limit_ns(unsigned long long ns) {
  if (ns > 10ull * kDefaultWaitNs) return MOE_ERR_INVALID_ARG;
  g_wait_limit_ns.store(ns ? (uint64_t)ns : kDefaultWaitNs, std::memory_order_relaxed);
  return MOE_OK;
}

int moe_get_device_status(void* workspace, size_t workspace_bytes, int* status, moe_stream_t stream) {
  if (!workspace || !status || workspace_bytes < 256) return MOE_ERR_INVALID_ARG;
  return read_and_clear_status(workspace, 256, reinterpret_cast<cudaStream_t>(stream), status);
}

}  // extern "C"
