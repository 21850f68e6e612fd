// Measured dense tensor-pipe rate of this GPU for the MMA forms the expert GEMMs
// issue: kind::mxf4 block-scaled (E2M1 x E2M1, E8M0 scales, the MXFP4 layer) and
// kind::f16 (bf16 x bf16, the bf16-weight layer), both cta_group::1 with M = 128
// and N = 256 (the widest single-CTA form).  The roofline of the compute-bound
// (4096-token prefill) workload is taken against this rate.
//
// One CTA per SM allocates the whole tensor memory, fills its operand tiles in
// shared memory with finite values, and one thread issues `mmas` MMAs back to back
// into one accumulator (the data is irrelevant: only the issue rate is timed), then
// waits -- bounded -- for their completion.
#include "moe_common.cuh"
#include "moe_kernels.cuh"
#include "sm100_ptx.cuh"

namespace moe {

using namespace ptx;

namespace {

constexpr int kPeakM = 128;
constexpr int kPeakN = 256;
constexpr int kPeakThreads = 128;
constexpr uint64_t kPeakWaitLimit = 2000000000ull;  // ns a bounded wait may take (2 s)
constexpr int kPeakABytes = kPeakM * 128;           // 128 rows x 128 bytes, 128-byte swizzle
constexpr int kPeakBBytes = kPeakN * 128;
constexpr int kPeakSfBytes = kSfAtomBytes;
// more shared memory than two CTAs can hold, so each SM runs exactly one of them
constexpr int kPeakSmem = 120 * 1024;

__device__ uint32_t g_peak_status;  // bit 0: the completion wait gave up

template <bool kMxf4>
__global__ void __launch_bounds__(kPeakThreads, 1) tensor_peak_kernel(int mmas) {
  extern __shared__ uint8_t peak_smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(peak_smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sa = base;
  uint8_t* sb = base + kPeakABytes;
  uint8_t* ssf = sb + kPeakBBytes;
  __shared__ uint64_t done_bar;
  __shared__ uint32_t tmem_slot;
  const int tid = threadIdx.x, warp = tid >> 5;
  // operands: E2M1 code 2 (1.0) in every nibble, or bf16 1.0; scale bytes 127 (2^0)
  const uint32_t fill = kMxf4 ? 0x22222222u : 0x3F803F80u;
  for (int i = tid; i < (kPeakABytes + kPeakBBytes) / 4; i += kPeakThreads) reinterpret_cast<uint32_t*>(sa)[i] = fill;
  for (int i = tid; i < kPeakSfBytes / 4; i += kPeakThreads) reinterpret_cast<uint32_t*>(ssf)[i] = 0x7F7F7F7Fu;
  if (warp == 0) {
    tmem_alloc(&tmem_slot, 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&done_bar, 1);
    fence_mbar_init();
  }
  fence_proxy_async_smem();  // the operand writes above are seen by the tensor core
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;  // accumulator: columns [0, 256); scales after it
  if (tid == 0) {
    const uint32_t sfa = tmem + kPeakN, sfb = sfa + 4;
    if constexpr (kMxf4) {
      // A scales (4 columns) and B scales (N = 256 rows read from 8 columns)
      const uint64_t d = smem_desc(smem_u32(ssf), 0, 128, 0);
      tmem_cp_32x128b_warpx4(sfa, d);
      tmem_cp_32x128b_warpx4(sfb, d);
      tmem_cp_32x128b_warpx4(sfb + 4, d);
    }
    const uint32_t idesc = kMxf4 ? idesc_mxf4(kPeakM, kPeakN, 0, 0) : idesc_bf16(kPeakM, kPeakN);
    for (int r = 0; r < mmas; ++r) {
      const int ks = r & 3;  // one 32-byte K step of the 128-byte rows
      const uint64_t ad = smem_desc_kmajor_sw128(smem_u32(sa) + 32 * ks);
      const uint64_t bd = smem_desc_kmajor_sw128(smem_u32(sb) + 32 * ks);
      if constexpr (kMxf4)
        mma_mxf4(tmem, ad, bd, idesc, sfa, sfb, r > 0 ? 1u : 0u);
      else
        mma_bf16(tmem, ad, bd, idesc, r > 0 ? 1u : 0u);
    }
    mma_commit(&done_bar);
  }
  __syncwarp();
  if (!mbar_wait_bounded(&done_bar, 0, kPeakWaitLimit) && (tid & 31) == 0) atomicOr(&g_peak_status, 1u);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

template <bool kMxf4>
int run_peak(int mmas, double* tflops, cudaStream_t s) {
  static SmemOptIn opt_in;
  if (opt_in.ensure(tensor_peak_kernel<kMxf4>, kPeakSmem) != cudaSuccess) return MOE_ERR_CUDA;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
    return MOE_ERR_CUDA;
  const uint32_t zero = 0;
  if (cudaMemcpyToSymbolAsync(g_peak_status, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) return MOE_ERR_CUDA;
  int st = MOE_OK;
  // one warm-up launch, then the timed one
  tensor_peak_kernel<kMxf4><<<sms, kPeakThreads, kPeakSmem, s>>>(mmas / 8 > 0 ? mmas / 8 : 1);
  cudaEventRecord(e0, s);
  tensor_peak_kernel<kMxf4><<<sms, kPeakThreads, kPeakSmem, s>>>(mmas);
  cudaEventRecord(e1, s);
  float ms = 0.f;
  uint32_t h = 0;
  if (cudaGetLastError() != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess ||
      cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess ||
      cudaMemcpyFromSymbol(&h, g_peak_status, sizeof h) != cudaSuccess)
    st = MOE_ERR_CUDA;
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (st != MOE_OK) return st;
  if (h) return MOE_ERR_DEVICE_TIMEOUT;
  const double k = kMxf4 ? 64.0 : 16.0;  // K per instruction
  *tflops = 2.0 * kPeakM * kPeakN * k * (double)mmas * sms / (ms * 1e-3) / 1e12;
  return MOE_OK;
}

}  // namespace

}  // namespace moe

extern "C" int moe_tensor_peak(int kind, int mmas_per_sm, double* tflops, moe_stream_t stream) {
  if (!tflops || mmas_per_sm < 8 || mmas_per_sm > (1 << 24)) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (kind == MOE_PEAK_MXF4) return moe::run_peak<true>(mmas_per_sm, tflops, s);
  if (kind == MOE_PEAK_BF16) return moe::run_peak<false>(mmas_per_sm, tflops, s);
  return MOE_ERR_INVALID_ARG;
}
