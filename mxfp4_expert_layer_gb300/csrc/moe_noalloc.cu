// Routing entry point for callers that cannot allocate device memory.
//
// Some callers have no way to call cudaMalloc: code running where the allocator is
// owned by someone else (a serving runtime with a fixed memory pool, a plugin
// handed only input and output buffers), or code that must not grow the device
// footprint at run time.  moe_route needs a little scratch memory besides its
// inputs and outputs -- the arrival counters of its last-block hand-off and a
// status word -- which moe_route takes from a caller-allocated workspace.
// moe_route_noalloc takes that scratch from a fixed array compiled into this
// library instead, so the caller passes only inputs and outputs.
//
// The array lives in every GPU that loads the library, for the life of the
// process: kNoAllocScratchBytes bytes, enough for T <= kNoAllocMaxTokens.  It is
// zero when the library is loaded; every routing call leaves its counters at zero
// again, and moe_route_noalloc_status clears the whole array after a reported
// timeout (a kernel that gave up may have left a counter behind).
#include <cuda_runtime.h>

#include <mutex>

#include "moe_common.cuh"
#include "moe_kernels.cuh"

namespace {

constexpr int kNoAllocMaxTokens = 8192;
// status word (256 bytes) + one arrival counter per group of 8 tokens + the table counter
constexpr size_t kNoAllocScratchBytes = 256 + sizeof(uint32_t) * (kNoAllocMaxTokens / 8 + 1);

static __device__ __align__(256) uint8_t g_route_scratch[kNoAllocScratchBytes];

// Device address of g_route_scratch per device, resolved once per device.  In host
// code the name g_route_scratch is only a host-side stand-in for the symbol; the
// kernel must be given the address cudaGetSymbolAddress returns for the current
// device.
void* g_scratch_addr[moe::kMaxDevices] = {};
std::mutex g_scratch_mu;

int scratch_for_current_device(uint8_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= moe::kMaxDevices) return MOE_ERR_UNSUPPORTED_SHAPE;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = static_cast<uint8_t*>(g_scratch_addr[dev]);
  return MOE_OK;
}

}  // namespace

extern "C" int moe_route_noalloc(const uint16_t* x, const uint16_t* w_router, const float* router_bias, int T,
                                 int H, int E, int k, float* logits, int flags, int32_t* topk_idx, float* topk_w,
                                 moe_stream_t stream) {
  using namespace moe;
  const int gating = gating_from_flags(flags);
  if (gating < 0) return MOE_ERR_INVALID_ARG;
  const int from_logits = (flags & MOE_ROUTE_FROM_LOGITS) ? 1 : 0;
  const int Hs = from_logits ? 32 : H;
  if (T < 1 || T > kNoAllocMaxTokens) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (Hs < 32 || Hs % 32 || Hs > 8192 || E < 1 || E > kMaxExperts || k < 1 || k > E || k > kMaxTopK)
    return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!logits || !topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
  if (!from_logits && (!x || !w_router || (reinterpret_cast<uintptr_t>(x) % 16) ||
                       (reinterpret_cast<uintptr_t>(w_router) % 16)))
    return MOE_ERR_INVALID_ARG;
  uint8_t* scratch = nullptr;
  int st = scratch_for_current_device(&scratch);
  if (st != MOE_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // The arrival counters are zero here: zero at load, and reset by the last arriver
  // of every call (after a timeout, moe_route_noalloc_status clears them).
  RouteParams r{};
  r.x = x;
  r.w_router = w_router;
  r.bias = router_bias;
  r.T = T; r.H = Hs; r.E = E; r.k = k;
  r.from_logits = from_logits;
  r.gating = gating;
  r.experts_per_block = T <= 64 ? 8 : 32;
  r.logits = logits;
  r.topk_idx = topk_idx;
  r.topk_w = topk_w;
  r.sync = reinterpret_cast<uint32_t*>(scratch + 256);
  r.status = reinterpret_cast<uint32_t*>(scratch);
  r.build_table = 0;
  return launch_route(r, s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

extern "C" int moe_route_noalloc_status(int* status, moe_stream_t stream) {
  if (!status) return MOE_ERR_INVALID_ARG;
  uint8_t* scratch = nullptr;
  const int st = scratch_for_current_device(&scratch);
  if (st != MOE_OK) return st;
  return moe::read_and_clear_status(scratch, kNoAllocScratchBytes, reinterpret_cast<cudaStream_t>(stream), status);
}
