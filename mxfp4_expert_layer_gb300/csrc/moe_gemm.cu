// Grouped MXFP4 expert GEMMs on the 5th-generation tensor cores (tcgen05):
//   gate/up + SwiGLU   h = silu(x W_gate^T) * (x W_up^T)
//   down + combine     out[t] = sum_j w_tj * (h_tj W_down^T)
//
// Sources: "A 297-line kernel file that decodes faster than vLLM", section "Where
// the time went" (rows "MoE gate/up + SwiGLU" and "MoE down + combine") and
// section "Optimizations" (row "MXFP4 MoE on tensor cores": weights re-laid out
// once at load, one grouped kernel for any token count; row "MoE token tile
// follows tokens per expert").
//
// Design (swap-AB): the MMA's M dimension is 128 weight rows (output features), N
// is the tile's token rows (16/64/128), K runs over the contraction in groups of
// 128.  A = MXFP4 weights (E2M1, loaded by TMA in the 16-byte-aligned unpacked
// shared-memory form), B = activations as two E4M3 terms, each with its own E8M0
// block scales; both scale sets are copied into tensor memory with tcgen05.cp and
// consumed natively by the block-scaled MMA (kind::mxf8f6f4, one scale per 32 K).
// Accumulators live in tensor memory.  Warp roles: warp 0 issues TMA loads into a
// ring of shared-memory stages, warp 1 issues MMAs, warps 2-5 run the epilogue.
#include "moe_common.cuh"
#include "moe_kernels.cuh"
#include "sm100_ptx.cuh"

namespace moe {

using namespace ptx;

namespace {

constexpr int kGemmThreads = 192;
constexpr uint64_t kWaitLimit = 1000000000ull;  // ns a bounded mbarrier wait may take (1 s)

template <int BM, bool GATEUP>
struct GemmCfg {
  static constexpr int kA = GATEUP ? 2 : 1;                 // weight tiles per stage
  static constexpr int kNb = BM > 128 ? 2 : 1;              // scale atoms per activation term
  static constexpr int kATileBytes = kMTile * 128;          // smem bytes of one A tile
  static constexpr int kBTileBytes = BM * 128;              // smem bytes of one B tile
  static constexpr int kSfBytes = (kA + 2 * kNb) * kSfAtomBytes;
  static constexpr int kStageRaw = kA * kATileBytes + 2 * kBTileBytes + kSfBytes;
  static constexpr int kStageBytes = (kStageRaw + 1023) / 1024 * 1024;
  static constexpr int kSmemBudget = 220 * 1024;
  static constexpr int kStagesRaw = kSmemBudget / kStageBytes;
  static constexpr int kStages = kStagesRaw > 8 ? 8 : kStagesRaw;
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024 /*align*/ + 1024 /*barriers*/;
  // expected transaction bytes per stage: the FP4 tiles count their packed global bytes
  static constexpr uint32_t kTxBytes = kA * kMTile * 64 + 2 * BM * 128 + kSfBytes;
  // tensor memory columns: accumulators first, then one scale ring slot per stage
  static constexpr int kAccCols = kA * BM;
  static constexpr int kSfColsPerStage = 4 * kA + 2 * 4 * kNb;
  static constexpr int kTmemNeed = kAccCols + kStages * kSfColsPerStage;
  static constexpr int kTmemCols = kTmemNeed <= 32 ? 32 : kTmemNeed <= 64 ? 64 : kTmemNeed <= 128 ? 128
                                   : kTmemNeed <= 256 ? 256 : 512;
  static_assert(kTmemNeed <= 512, "tensor memory budget");
  static_assert(kStages >= 2, "pipeline depth");
};

struct WorkUnit {
  int tile, mt;
};

// Raster: units are grouped in blocks of `group` tiles; within a block, the M tile
// varies slowest, so co-resident CTAs share weight tiles (same expert) and
// activation tiles through L2.
__device__ __forceinline__ bool map_unit(int u, int num_tiles, int mt_count, int group, WorkUnit& w) {
  if (u >= num_tiles * mt_count) return false;
  const int g = u / (group * mt_count);
  const int first = g * group;
  const int gsize = min(group, num_tiles - first);
  const int within = u - first * mt_count;
  w.mt = within / gsize;
  w.tile = first + within % gsize;
  return true;
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.f + expf(-g)); }

// Warp-wide two-term E4M3 encoding of one value per lane (the 32 lanes form one
// MX block).  Returns the codes and the exponents of both terms.
__device__ __forceinline__ void encode_two_term(float v, uint8_t& q1, uint8_t& q2, int& p1, int& p2) {
  float a = fabsf(v);
  a = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(a)));
  p1 = mx_e4m3_exponent(a);
  q1 = f32_to_e4m3(v * pow2_int(-p1));
  const float r = v - e4m3_to_f32(q1) * pow2_int(p1);
  float ar = fabsf(r);
  ar = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(ar)));
  p2 = mx_e4m3_exponent(ar);
  q2 = f32_to_e4m3(r * pow2_int(-p2));
}

}  // namespace

template <int BM, bool GATEUP>
__global__ void __launch_bounds__(kGemmThreads, 1) moe_gemm_kernel(const __grid_constant__ GemmParams p) {
  using C = GemmCfg<BM, GATEUP>;
  extern __shared__ uint8_t gemm_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(gemm_smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStageBytes);
  uint64_t* empty_bar = full_bar + C::kStages;
  uint64_t* accum_bar = empty_bar + C::kStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accum_bar + 1);
  int* s_flags = reinterpret_cast<int*>(tmem_slot + 1);  // [0] error, [1..BM] combine finalisers

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int num_tiles = __ldg(p.num_tiles);
  WorkUnit wu;
  if (!map_unit(blockIdx.x, num_tiles, p.mt, p.group_tiles, wu)) return;
  const TileEntry te = p.tiles[wu.tile];

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(accum_bar, 1);
    s_flags[0] = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tm_w);
    tma_prefetch_desc(&p.tm_act_hi);
    tma_prefetch_desc(&p.tm_act_lo);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto stage_ptr = [&](int s) { return smem + s * C::kStageBytes; };
  // stage layout: [A tiles][B hi][B lo][SF A x kA][SF B hi x kNb][SF B lo x kNb]
  auto a_tile = [&](int s, int j) { return stage_ptr(s) + j * C::kATileBytes; };
  auto b_tile = [&](int s, int term) { return stage_ptr(s) + C::kA * C::kATileBytes + term * C::kBTileBytes; };
  auto sf_a = [&](int s, int j) {
    return stage_ptr(s) + C::kA * C::kATileBytes + 2 * C::kBTileBytes + j * kSfAtomBytes;
  };
  auto sf_b = [&](int s, int term) {
    return stage_ptr(s) + C::kA * C::kATileBytes + 2 * C::kBTileBytes + (C::kA + term * C::kNb) * kSfAtomBytes;
  };

  const int kblocks = p.K / kMxBlock;  // real MX blocks along K (padded blocks are skipped)
  const int kg = p.kg;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint8_t* wsf_base = p.w_sf + ((size_t)te.expert * p.w_groups * p.mt + wu.mt) * (size_t)kg * kSfAtomBytes;
      const size_t wsf_group_stride = (size_t)p.mt * kg * kSfAtomBytes;
      const size_t asf_tile = (size_t)wu.tile * kg * (kSfAtomBytes * C::kNb);
      int g = 0;
      for (; g < kg; ++g) {
        const int s = g % C::kStages;
        const uint32_t ph = (g / C::kStages) & 1;
        if (!mbar_wait_bounded(&empty_bar[s], ph ^ 1, kWaitLimit)) {
          report_status(p.status, kStatusTimeoutProducer);
          s_flags[0] = 1;
          break;
        }
        mbar_arrive_expect_tx(&full_bar[s], C::kTxBytes);
        const int kc = g * kKGroup;
        for (int j = 0; j < C::kA; ++j) {
          tma_load_4d(a_tile(s, j), &p.tm_w, &full_bar[s], kc, wu.mt * kMTile, j, te.expert);
          bulk_load(sf_a(s, j), wsf_base + j * wsf_group_stride + (size_t)g * kSfAtomBytes, kSfAtomBytes,
                    &full_bar[s]);
        }
        tma_load_2d(b_tile(s, 0), &p.tm_act_hi, &full_bar[s], kc, te.pad_row);
        tma_load_2d(b_tile(s, 1), &p.tm_act_lo, &full_bar[s], kc, te.pad_row);
        bulk_load(sf_b(s, 0), p.act_sf_hi + asf_tile + (size_t)g * kSfAtomBytes * C::kNb, kSfAtomBytes * C::kNb,
                  &full_bar[s]);
        bulk_load(sf_b(s, 1), p.act_sf_lo + asf_tile + (size_t)g * kSfAtomBytes * C::kNb, kSfAtomBytes * C::kNb,
                  &full_bar[s]);
      }
      // on an error, wait (bounded) for the copies already issued to land
      if (s_flags[0]) {
        for (int gg = max(0, g - C::kStages); gg < g; ++gg) {
          mbar_wait_bounded(&full_bar[gg % C::kStages], (gg / C::kStages) & 1, kWaitLimit);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t sf_col0 = C::kAccCols;
      for (int g = 0; g < kg; ++g) {
        const int s = g % C::kStages;
        const uint32_t ph = (g / C::kStages) & 1;
        if (!mbar_wait_bounded(&full_bar[s], ph, kWaitLimit)) {
          report_status(p.status, kStatusTimeoutMain);
          s_flags[0] = 1;
          break;
        }
        tc_fence_after();
        const uint32_t sfc = tmem + sf_col0 + s * C::kSfColsPerStage;
        // scale atoms -> tensor memory (32 rows x 16 bytes, replicated to 4 lane quarters)
        for (int j = 0; j < C::kA; ++j) tmem_cp_32x128b_warpx4(sfc + 4 * j, smem_desc(smem_u32(sf_a(s, j)), 0, 128, 0));
        for (int term = 0; term < 2; ++term)
          for (int q = 0; q < C::kNb; ++q)
            tmem_cp_32x128b_warpx4(sfc + 4 * C::kA + term * 4 * C::kNb + 4 * q,
                                   smem_desc(smem_u32(sf_b(s, term)) + q * kSfAtomBytes, 0, 128, 0));
        for (int kb = 0; kb < 4; ++kb) {
          if (g * 4 + kb >= kblocks) break;
          const uint32_t idesc = idesc_mx(kMTile, BM, kFmtE2M1, kFmtE4M3, kb, kb);
          for (int term = 0; term < 2; ++term) {
            const uint64_t bdesc = smem_desc_kmajor_sw128(smem_u32(b_tile(s, term)) + 32 * kb);
            const uint32_t sfb = sfc + 4 * C::kA + term * 4 * C::kNb;
            const uint32_t acc = (g | kb | term) != 0;
            for (int j = 0; j < C::kA; ++j) {
              const uint64_t adesc = smem_desc_kmajor_sw128(smem_u32(a_tile(s, j)) + 32 * kb);
              mma_mxf8f6f4(tmem + j * BM, adesc, bdesc, idesc, sfc + 4 * j, sfb, acc);
            }
          }
        }
        mma_commit(&empty_bar[s]);  // frees the stage once these MMAs have read it
      }
      mma_commit(accum_bar);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                // tensor-memory lane quarter of this warp
    const int m = q * 32 + lane;           // row of the 128-row tile
    const int feat = wu.mt * kMTile + m;   // output feature
    const bool ok = mbar_wait_bounded(accum_bar, 0, kWaitLimit);
    if (!ok) {
      report_status(p.status, kStatusTimeoutEpi);
      s_flags[0] = 1;
    }
    tc_fence_after();
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const int nrows = te.n_rows;
    if (ok) {
      if constexpr (GATEUP) {
        const bool fvalid = feat < p.I;
        uint8_t* sfh = p.h_sf_hi + ((size_t)wu.tile * p.kg_out + wu.mt) * (kSfAtomBytes * C::kNb);
        uint8_t* sfl = p.h_sf_lo + ((size_t)wu.tile * p.kg_out + wu.mt) * (kSfAtomBytes * C::kNb);
#pragma unroll 1
        for (int c0 = 0; c0 < BM; c0 += 16) {
          if (c0 >= nrows) break;
          uint32_t rg[16], ru[16];
          tmem_ld_32x32b_x16(lane_base + c0, rg);
          tmem_ld_32x32b_x16(lane_base + BM + c0, ru);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int r = c0 + j;
            const float g = __uint_as_float(rg[j]);
            const float u = __uint_as_float(ru[j]);
            const float h = fvalid ? silu_f(g) * u : 0.f;
            uint8_t q1, q2;
            int p1, p2;
            encode_two_term(h, q1, q2, p1, p2);
            if (r < nrows) {
              const size_t row = (size_t)(te.pad_row + r);
              if (fvalid) {
                p.h_hi[row * p.I + feat] = q1;
                p.h_lo[row * p.I + feat] = q2;
              }
              if (lane == 0) {
                const int off = sf_atom_offset(r, q);
                sfh[off] = static_cast<uint8_t>(p1 + 127);
                sfl[off] = static_cast<uint8_t>(p2 + 127);
              }
            }
          }
        }
      } else {
        const bool fvalid = feat < p.H;
#pragma unroll 1
        for (int c0 = 0; c0 < BM; c0 += 16) {
          if (c0 >= nrows) break;
          uint32_t rd[16];
          tmem_ld_32x32b_x16(lane_base + c0, rd);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int r = c0 + j;
            if (r < nrows && fvalid) {
              const int a = __ldg(p.perm + te.row_begin + r);
              const float wgt = __ldg(p.topk_w + a);
              p.slots[(size_t)a * p.H + feat] = wgt * __uint_as_float(rd[j]);
            }
          }
        }
      }
    }
    if constexpr (!GATEUP) {
      // deterministic combine: the last CTA to finish a (token, output tile) sums the
      // token's k weighted slots in ascending j and writes the bf16 output
      __threadfence();
      asm volatile("bar.sync 1, 128;" ::: "memory");
      const int et = threadIdx.x - 64;  // 0..127
      if (et < BM) {
        int fin = 0;
        if (et < nrows && ok) {
          const int a = __ldg(p.perm + te.row_begin + et);
          const int t = a / p.k;
          int* cnt = p.combine_cnt + (size_t)t * p.mt + wu.mt;
          const int old = atomicAdd(cnt, 1);
          if (old == p.k - 1) {
            fin = 1;
            *cnt = 0;  // ready for the next call
          }
        }
        s_flags[1 + et] = fin;
      }
      asm volatile("bar.sync 1, 128;" ::: "memory");
      __threadfence();
      if (ok && feat < p.H) {
        for (int r = 0; r < nrows; ++r) {
          if (!s_flags[1 + r]) continue;
          const int a = __ldg(p.perm + te.row_begin + r);
          const int t = a / p.k;
          float acc = 0.f;
          for (int j = 0; j < p.k; ++j) acc += __ldcg(p.slots + ((size_t)t * p.k + j) * p.H + feat);
          p.out[(size_t)t * p.H + feat] = __bfloat16_as_ushort(__float2bfloat16_rn(acc));
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::kTmemCols);
}

template <int BM, bool GATEUP>
static cudaError_t launch_gemm_t(const GemmParams& p, cudaStream_t stream) {
  using C = GemmCfg<BM, GATEUP>;
  auto kern = moe_gemm_kernel<BM, GATEUP>;
  // the shared-memory opt-in is a per-device function attribute: set it once per device
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev] = true;
  }
  const int units = p.max_tiles * p.mt;
  kern<<<units, kGemmThreads, C::kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

template <bool GATEUP>
static cudaError_t launch_gemm(const GemmParams& p, cudaStream_t stream) {
  switch (p.bm) {
    case 16: return launch_gemm_t<16, GATEUP>(p, stream);
    case 64: return launch_gemm_t<64, GATEUP>(p, stream);
    case 128: return launch_gemm_t<128, GATEUP>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_gateup(const GemmParams& p, cudaStream_t stream) { return launch_gemm<true>(p, stream); }
cudaError_t launch_down(const GemmParams& p, cudaStream_t stream) { return launch_gemm<false>(p, stream); }

}  // namespace moe
