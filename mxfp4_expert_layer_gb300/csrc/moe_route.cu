// Router GEMV/GEMM, warp-shuffle top-k with softmax over the selected logits, and
// the atomic-free per-expert tile table.
//
// Sources: "A 297-line kernel file that decodes faster than vLLM", section "Where
// the time went" (row "Router + top-k") and section "Optimizations" (row
// "Per-expert routing tile table": every expert writes its own tiles instead of a
// kernel searching a tiles x experts grid); "triton-kernels" README, section
// "Quick Start" (softmax gating + top-k, expert indices and weights returned).
//
// One launch does all three steps.
//  * Few tokens (decode): one thread-block cluster splits the hidden dimension,
//    exchanges partial logits through distributed shared memory and needs no
//    global atomics.
//  * Many tokens: blocks of 32 tokens x all experts compute logits on the tensor
//    cores, and the last block to finish (an integer arrival count, no spinning)
//    builds the tile table.
//  * Logits given: blocks of 8 tokens select the top-k.
// With the norm step in front of the layer, both logit kernels normalise the rows
// they stage (RMSNorm + residual, the range-sum order of moe_norm.cuh).  Every
// result is computed by one fixed thread or warp in a fixed order, so the outputs
// are bit-reproducible run to run.
#include "moe_common.cuh"
#include "moe_kernels.cuh"
#include "sm100_ptx.cuh"

#include <cooperative_groups.h>

namespace moe {

using namespace ptx;

namespace {

constexpr int kRouteThreads = 256;
constexpr int kRouteWarps = kRouteThreads / 32;
constexpr int kTokensPerGroup = 8;
constexpr int kStageVecs = 12;   // 16-byte activation loads in flight per thread

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// Unsigned key with the order of the float it encodes (larger float -> larger key).
__device__ __forceinline__ uint32_t sortable_key(float v) {
  if (v == 0.f) v = 0.f;  // -0 and +0 compare equal
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// (value, index) order used by top-k: larger value first, then smaller index.
__device__ __forceinline__ bool topk_better(float v1, int i1, float v2, int i2) {
  return v1 > v2 || (v1 == v2 && i1 < i2);
}

}  // namespace

// Deterministic counting sort of the assignments by expert, stable in t*k+j,
// executed by one block of 256 threads.  Each warp owns a contiguous chunk of
// assignments and a private histogram row; lanes with equal experts are grouped
// with __match_any_sync, so no atomics are used anywhere.  One warp turns the
// histograms into counts, row offsets, tile entries and per-warp bases (both
// scans over experts in one pass), so the whole build takes three block barriers.
// kSharedIdx: the top-k indices are in this block's shared memory (else global,
// read through L2).  pad_inv: inv_perm receives each assignment's padded row (its
// tile x bm + its row within the tile) instead of its sorted row, so that the
// permute step finds the tile row with one load.
template <bool kSharedIdx = false>
__device__ void build_tile_table_block(const int32_t* __restrict__ idx, int Tk, int E, int bm, int32_t* counts,
                                       int32_t* offsets, int32_t* perm, int32_t* inv_perm, TileEntry* tiles,
                                       int32_t* num_tiles, uint32_t* status, bool pad_inv = false) {
  __shared__ int hist[kRouteWarps][kMaxExperts];
  __shared__ int pad_delta[kMaxExperts];  // padded row minus sorted row, per expert
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid < E) {
#pragma unroll
    for (int w = 0; w < kRouteWarps; ++w) hist[w][tid] = 0;
  }
  __syncthreads();
  const int chunk = ceil_div(Tk, kRouteWarps);
  const int a_begin = warp * chunk;
  const int a_end = min(Tk, a_begin + chunk);
  const unsigned lt_mask = (1u << lane) - 1u;
  // phase 1: per-warp histograms
  for (int base = a_begin; base < a_end; base += 32) {
    const int a = base + lane;
    int e = -1;
    if (a < a_end) {
      e = kSharedIdx ? idx[a] : __ldcg(idx + a);
      if (e < 0 || e >= E) {
        report_status(status, kStatusBadIndex);
        e = -1;
      }
    }
    const unsigned grp = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && (grp & lt_mask) == 0) hist[warp][e] += __popc(grp);
  }
  __syncthreads();
  // phase 2 (warp 0): lane l owns experts [l*per, l*per + per); counts, then one
  // warp scan of (rows, tiles) gives each expert's first sorted row and first tile.
  // bm is a power of two; rows and tiles share one 32-bit scan when both fit in 16 bits.
  if (warp == 0) {
    const int lgbm = __ffs(bm) - 1;
    const int per = (E + 31) >> 5;
    const int e0 = lane * per;
    int cnt[kMaxExperts / 32];
    int rows = 0, ntl = 0;
#pragma unroll
    for (int i = 0; i < kMaxExperts / 32; ++i) {
      int c = 0;
      if (i < per && e0 + i < E) {
#pragma unroll
        for (int w = 0; w < kRouteWarps; ++w) c += hist[w][e0 + i];
      }
      cnt[i] = c;
      rows += c;
      ntl += (c + bm - 1) >> lgbm;
    }
    int rows_incl, ntl_incl;
    if (Tk < 65536) {
      int packed = rows | (ntl << 16);  // tiles <= Tk / bm + E < 65536 as well
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, packed, d);
        if (lane >= d) packed += o;
      }
      rows_incl = packed & 0xFFFF;
      ntl_incl = (int)((unsigned)packed >> 16);
    } else {
      rows_incl = rows;
      ntl_incl = ntl;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int ro = __shfl_up_sync(0xffffffffu, rows_incl, d);
        const int to = __shfl_up_sync(0xffffffffu, ntl_incl, d);
        if (lane >= d) {
          rows_incl += ro;
          ntl_incl += to;
        }
      }
    }
    int off = rows_incl - rows, t0 = ntl_incl - ntl;
#pragma unroll
    for (int i = 0; i < kMaxExperts / 32; ++i) {
      const int e = e0 + i;
      if (i >= per || e >= E) break;
      const int c = cnt[i];
      counts[e] = c;
      offsets[e] = off;
      pad_delta[e] = (t0 << lgbm) - off;
      int run = off;
#pragma unroll
      for (int w = 0; w < kRouteWarps; ++w) {
        const int h = hist[w][e];
        hist[w][e] = run;  // becomes the next free sorted row of (warp, expert)
        run += h;
      }
      const int nt = (c + bm - 1) >> lgbm;
      for (int q = 0; q < nt; ++q) {
        TileEntry te;
        te.expert = e;
        te.row_begin = off + (q << lgbm);
        te.n_rows = min(bm, c - (q << lgbm));
        te.pad_row = (t0 + q) << lgbm;
        tiles[t0 + q] = te;
      }
      off += c;
      t0 += nt;
    }
    if (lane == 31) {
      offsets[E] = rows_incl;
      *num_tiles = ntl_incl;
    }
  }
  __syncthreads();
  // phase 3: scatter assignments to their sorted rows (stable in a)
  for (int base = a_begin; base < a_end; base += 32) {
    const int a = base + lane;
    int e = -1;
    if (a < a_end) {
      e = kSharedIdx ? idx[a] : __ldcg(idx + a);
      if (e < 0 || e >= E) e = -1;
    }
    const unsigned grp = __match_any_sync(0xffffffffu, e);
    int pos = 0;
    if (e >= 0) pos = hist[warp][e] + __popc(grp & lt_mask);
    __syncwarp();
    if (e >= 0) {
      perm[pos] = a;
      inv_perm[a] = pad_inv ? pos + pad_delta[e] : pos;
      if ((grp & lt_mask) == 0) hist[warp][e] += __popc(grp);
    }
    __syncwarp();
  }
}

// The same table for at most 32 assignments, built by one warp with no block
// barrier (the decode shapes): lane a holds assignment a, lanes with equal experts
// count themselves into one shared histogram row (__match_any_sync, no atomics), and
// the scan, offsets, tiles and the stable scatter are those of the block version, so
// the bits are identical (pad_inv as there).
template <bool kSharedIdx = false>
__device__ void build_tile_table_warp(const int32_t* __restrict__ idx, int Tk, int E, int bm, int32_t* counts,
                                      int32_t* offsets, int32_t* perm, int32_t* inv_perm, TileEntry* tiles,
                                      int32_t* num_tiles, uint32_t* status, bool pad_inv = false) {
  __shared__ int whist[kMaxExperts];
  __shared__ int wpad_delta[kMaxExperts];  // padded row minus sorted row, per expert
  const int lane = threadIdx.x & 31;
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int e = lane; e < E; e += 32) whist[e] = 0;
  int ea = -1;
  if (lane < Tk) {
    ea = kSharedIdx ? idx[lane] : __ldcg(idx + lane);
    if (ea < 0 || ea >= E) {
      report_status(status, kStatusBadIndex);
      ea = -1;
    }
  }
  const unsigned grp = __match_any_sync(0xffffffffu, ea);
  __syncwarp();
  if (ea >= 0 && (grp & lt_mask) == 0) whist[ea] = __popc(grp);
  __syncwarp();
  // lane l owns experts [l*per, l*per + per): counts, then one warp scan of the packed
  // (rows, tiles) pairs gives each expert's first sorted row and first tile
  const int lgbm = __ffs(bm) - 1;
  const int per = (E + 31) >> 5;
  const int e0 = lane * per;
  int cnt[kMaxExperts / 32];
  int rows = 0, ntl = 0;
#pragma unroll
  for (int i = 0; i < kMaxExperts / 32; ++i) {
    const int c = (i < per && e0 + i < E) ? whist[e0 + i] : 0;
    cnt[i] = c;
    rows += c;
    ntl += (c + bm - 1) >> lgbm;
  }
  int packed = rows | (ntl << 16);  // at most 32 rows and 32 tiles
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, packed, d);
    if (lane >= d) packed += o;
  }
  const int rows_incl = packed & 0xFFFF, ntl_incl = (int)((unsigned)packed >> 16);
  int off = rows_incl - rows, t0 = ntl_incl - ntl;
  __syncwarp();  // every lane has read whist before it becomes the row offsets
#pragma unroll
  for (int i = 0; i < kMaxExperts / 32; ++i) {
    const int e = e0 + i;
    if (i >= per || e >= E) break;
    const int c = cnt[i];
    counts[e] = c;
    offsets[e] = off;
    wpad_delta[e] = (t0 << lgbm) - off;
    whist[e] = off;
    const int nt = (c + bm - 1) >> lgbm;
    for (int q = 0; q < nt; ++q) {
      TileEntry te;
      te.expert = e;
      te.row_begin = off + (q << lgbm);
      te.n_rows = min(bm, c - (q << lgbm));
      te.pad_row = (t0 + q) << lgbm;
      tiles[t0 + q] = te;
    }
    off += c;
    t0 += nt;
  }
  if (lane == 31) {
    offsets[E] = rows_incl;
    *num_tiles = ntl_incl;
  }
  __syncwarp();
  // stable scatter: an assignment's sorted row is its expert's first row plus the
  // number of lower lanes with the same expert
  if (ea >= 0) {
    const int pos = whist[ea] + __popc(grp & lt_mask);
    perm[pos] = lane;
    inv_perm[lane] = pad_inv ? pos + wpad_delta[ea] : pos;
  }
}

// Top-k of one token by one warp: each lane holds logits e = lane + 32*i; k rounds
// of a warp arg-max on (value desc, index asc).  Weights by `gating` (MoeGating):
// softmax over the k selected (exponentials relative to the largest, summed in
// selection order), softmax over all E (the selected exponentials over the sum of all,
// reduced by a fixed butterfly), or the selected sigmoids normalised to sum to one.
// kShared: the logits row is in shared memory (else global, read through L2).
// Returns the j-th selected expert in lane j < k.
template <bool kShared = false>
__device__ int topk_softmax_warp(const float* __restrict__ lg_row, int E, int k, int32_t* idx_out, float* w_out,
                                 int gating = kGatingSoftmaxTopk) {
  const int lane = threadIdx.x & 31;
  float my_v = -INFINITY;  // lane j keeps the j-th selection
  int my_i = 0;
  float all_part = 0.f;    // softmax over all: this lane's share of sum_e exp(l_e - max)
  if (E <= 32) {
    // one logit per lane: a round is one warp max of the order-preserving key, the
    // lowest lane holding it (= the lower expert index among equal values), and a
    // shuffle of its value; a selected lane's key drops to 0, below every logit's
    const float vl = lane < E ? (kShared ? lg_row[lane] : __ldcg(lg_row + lane)) : -INFINITY;
    uint32_t key = lane < E ? sortable_key(vl) : 0u;
    for (int j = 0; j < k; ++j) {
      const uint32_t kmax = __reduce_max_sync(0xffffffffu, key);
      const int win = __ffs(__ballot_sync(0xffffffffu, key == kmax)) - 1;
      const float bv = __shfl_sync(0xffffffffu, vl, win);
      if (lane == win) key = 0u;
      if (lane == j) {
        my_v = bv;
        my_i = win;
      }
    }
    if (gating == kGatingSoftmaxAll) {
      const float mx = __shfl_sync(0xffffffffu, my_v, 0);  // every lane takes part
      if (lane < E) all_part = expf(vl - mx);
    }
  } else {
    float v[kMaxExperts / 32];
#pragma unroll
    for (int i = 0; i < kMaxExperts / 32; ++i) {
      const int e = lane + 32 * i;
      v[i] = (e < E) ? (kShared ? lg_row[e] : __ldcg(lg_row + e)) : -INFINITY;
    }
    unsigned taken = 0;  // bit i: element e = lane + 32*i already selected
    for (int j = 0; j < k; ++j) {
      // this lane's best remaining element (larger value, then smaller index)
      float bv = -INFINITY;
      int bi = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < kMaxExperts / 32; ++i) {
        const int e = lane + 32 * i;
        if (e < E && !((taken >> i) & 1u) && topk_better(v[i], e, bv, bi)) {
          bv = v[i];
          bi = e;
        }
      }
      // warp arg-max in two reductions: the largest value (as an order-preserving
      // unsigned key), then the smallest index among the lanes holding it
      const uint32_t key = sortable_key(bv);
      const uint32_t kmax = __reduce_max_sync(0xffffffffu, key);
      bi = (int)__reduce_min_sync(0xffffffffu, key == kmax ? (uint32_t)bi : 0xffffffffu);
      bv = __shfl_sync(0xffffffffu, bv, bi & 31);
      if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
      if (lane == j) {
        my_v = bv;
        my_i = bi;
      }
    }
    if (gating == kGatingSoftmaxAll) {
      const float mx = __shfl_sync(0xffffffffu, my_v, 0);
#pragma unroll
      for (int i = 0; i < kMaxExperts / 32; ++i)
        if (lane + 32 * i < E) all_part += expf(v[i] - mx);
    }
  }
  const float m = __shfl_sync(0xffffffffu, my_v, 0);
  float num, den = 0.f;
  if (gating == kGatingSigmoid) {
    num = lane < k ? 1.f / (1.f + expf(-my_v)) : 0.f;
    for (int j = 0; j < k; ++j) den += __shfl_sync(0xffffffffu, num, j);
  } else {
    num = lane < k ? expf(my_v - m) : 0.f;
    if (gating == kGatingSoftmaxAll) {
      den = all_part;
#pragma unroll
      for (int d = 16; d > 0; d >>= 1) den += __shfl_xor_sync(0xffffffffu, den, d);
    } else {
      for (int j = 0; j < k; ++j) den += __shfl_sync(0xffffffffu, num, j);
    }
  }
  if (lane < k) {
    idx_out[lane] = my_i;
    w_out[lane] = num / den;
  }
  return my_i;
}

// grid = (token groups of 8, expert slices); block = 256 threads.  kRouterVecs:
// 16-byte router-weight loads in flight per lane (more for few tokens, where the
// loads' latency dominates; fewer for many, where registers bound the occupancy).
template <int kRouterVecs>
__global__ void __launch_bounds__(kRouteThreads) route_kernel(RouteParams p) {
  extern __shared__ __align__(16) uint8_t route_smem[];
  __shared__ int s_last;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // The previous kernel on the stream may still write x or read this call's outputs
  pdl_wait();
  pdl_launch_dependents();
  const int g = blockIdx.x;
  const int t0 = g * kTokensPerGroup;
  const int nt = min(kTokensPerGroup, p.T - t0);
  if (!p.from_logits) {
    const int vec_per_row = p.H / 8;
    const int e_begin = blockIdx.y * p.experts_per_block;
    const int e_end = min(p.E, e_begin + p.experts_per_block);
    // the first chunk of this warp's router weights is requested before the
    // activations are staged, so both latencies overlap
    const int e_first = e_begin + warp;
    uint4 wpre[kRouterVecs];
    if (e_first < e_end) {
      const uint4* wr = reinterpret_cast<const uint4*>(p.w_router + (size_t)e_first * p.H);
#pragma unroll
      for (int u = 0; u < kRouterVecs; ++u) {
        const int c = lane + 32 * u;
        wpre[u] = c < vec_per_row ? __ldg(wr + c) : make_uint4(0, 0, 0, 0);
      }
    }
    // stage the group's activations in shared memory (16-byte vectors); rows of one
    // group are contiguous in x
    uint4* xs = reinterpret_cast<uint4*>(route_smem);
    const uint4* xg = reinterpret_cast<const uint4*>(p.x + (size_t)t0 * p.H);
    const int nx = nt * vec_per_row;
    for (int i0 = tid; i0 < nx; i0 += kStageVecs * kRouteThreads) {
      uint4 v[kStageVecs];
#pragma unroll
      for (int u = 0; u < kStageVecs; ++u) {
        const int i = i0 + u * kRouteThreads;
        v[u] = i < nx ? __ldg(xg + i) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < kStageVecs; ++u) {
        const int i = i0 + u * kRouteThreads;
        if (i < nx) xs[i] = v[u];
      }
    }
    __syncthreads();
    for (int e = e_first; e < e_end; e += kRouteWarps) {
      float acc[kTokensPerGroup];
#pragma unroll
      for (int r = 0; r < kTokensPerGroup; ++r) acc[r] = 0.f;
      const uint4* wr = reinterpret_cast<const uint4*>(p.w_router + (size_t)e * p.H);
      // kRouterVecs router-weight loads in flight per lane, then their FMAs in a
      // fixed order (per lane: ascending vector index)
      for (int c0 = 0; c0 < vec_per_row; c0 += 32 * kRouterVecs) {
        uint4 wv4[kRouterVecs];
        if (e == e_first && c0 == 0) {
#pragma unroll
          for (int u = 0; u < kRouterVecs; ++u) wv4[u] = wpre[u];
        } else {
#pragma unroll
          for (int u = 0; u < kRouterVecs; ++u) {
            const int c = c0 + lane + 32 * u;
            wv4[u] = c < vec_per_row ? __ldg(wr + c) : make_uint4(0, 0, 0, 0);
          }
        }
#pragma unroll
        for (int u = 0; u < kRouterVecs; ++u) {
          const int c = c0 + lane + 32 * u;
          if (c >= vec_per_row) break;
          const uint4 wv = wv4[u];
          const float w0 = bf16_lo(wv.x), w1 = bf16_hi(wv.x), w2 = bf16_lo(wv.y), w3 = bf16_hi(wv.y);
          const float w4 = bf16_lo(wv.z), w5 = bf16_hi(wv.z), w6 = bf16_lo(wv.w), w7 = bf16_hi(wv.w);
#pragma unroll
          for (int r = 0; r < kTokensPerGroup; ++r) {
            if (r < nt) {
              const uint4 xv = xs[r * vec_per_row + c];
              float a = acc[r];
              a = fmaf(bf16_lo(xv.x), w0, a);
              a = fmaf(bf16_hi(xv.x), w1, a);
              a = fmaf(bf16_lo(xv.y), w2, a);
              a = fmaf(bf16_hi(xv.y), w3, a);
              a = fmaf(bf16_lo(xv.z), w4, a);
              a = fmaf(bf16_hi(xv.z), w5, a);
              a = fmaf(bf16_lo(xv.w), w6, a);
              a = fmaf(bf16_hi(xv.w), w7, a);
              acc[r] = a;
            }
          }
        }
      }
#pragma unroll
      for (int r = 0; r < kTokensPerGroup; ++r) {
        float a = acc[r];
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) a += __shfl_xor_sync(0xffffffffu, a, d);
        if (lane == 0 && r < nt) {
          if (p.bias) a += __ldg(p.bias + e);
          p.logits[(size_t)(t0 + r) * p.E + e] = a;
        }
      }
    }
    // arrival of this expert slice for the token group
    __threadfence();
    __syncthreads();
    if (tid == 0) {
      const unsigned old = atomicAdd(p.sync + g, 1u);
      s_last = (old == gridDim.y - 1) ? 1 : 0;
      if (s_last) p.sync[g] = 0;  // ready for the next call
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
  }
  // top-k of the group's tokens: one warp per token
  if (warp < nt) {
    const int t = t0 + warp;
    topk_softmax_warp(p.logits + (size_t)t * p.E, p.E, p.k, p.topk_idx + (size_t)t * p.k,
                      p.topk_w + (size_t)t * p.k, p.gating);
  }
  if (!p.build_table) return;
  __threadfence();
  __syncthreads();
  if (gridDim.x > 1) {
    // the last token group to finish builds the table
    if (tid == 0) {
      const unsigned old = atomicAdd(p.sync + gridDim.x, 1u);
      s_last = (old == gridDim.x - 1) ? 1 : 0;
      if (s_last) p.sync[gridDim.x] = 0;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
  }
  build_tile_table_block(p.topk_idx, p.T * p.k, p.E, p.bm, p.counts, p.offsets, p.perm, p.inv_perm, p.tiles,
                         p.num_tiles, p.status, p.pad_inv != 0);
}

// ------------------------------------------------------------------ decode routing
// Few tokens (T <= 64): one cluster of kClusterCtas CTAs does the whole routing with
// no global atomics and no full cluster barrier after the start.  CTA r computes
// the partial logits of every token and expert over its slice of the hidden
// dimension on the tensor cores (mma.sync bf16, fp32 accumulate) and pushes the
// partials of tokens 8q..8q+7 into CTA q's shared memory (st.async, counted on
// CTA q's mbarrier).  CTA q sums the kClusterCtas partials in rank order, selects
// the top-k of its tokens and pushes the indices to CTA 0, which builds the tile
// table.  A CTA's shared memory is written by its peers only before its own wait
// on the matching barrier returns, so every CTA may exit right after its last push.
constexpr int kClusterCtas = 8;
constexpr int kClusterMaxTokens = kClusterCtas * kTokensPerGroup;

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x2(uint32_t (&r)[2], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r[0]), "=r"(r[1]) : "r"(addr));
}
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

constexpr int kMmaIlp = 4;  // 8-expert column blocks per warp pass (one A fragment serves all)

// Shared-memory layout of the cluster routing kernel for (T, H, E, k).  A warp
// item is (16-token row block, kMmaIlp column blocks); when there are fewer items
// than warps, each item's K range is split over nsplit warps whose partial sums
// meet in the split area.
constexpr size_t kClusterSmemCap = 200 * 1024;  // dynamic shared memory of the cluster kernel

struct ClusterRouteSmem {
  int mrows, erows, pitch;        // staged x rows (multiple of 16), router rows (multiple of 8), row bytes
  int nitems, nsplit;
  int rs_staged;                  // norm step: residual slices staged beside x (else read from global)
  size_t x_off, w_off, rs_off, split_off, recv_off, lg_off, bias_off, idx_off, norm_off, bar_off, total;
};
static_assert(kClusterCtas == kNormSlices, "a cluster CTA sums one range of the norm's row cut");
__host__ __device__ inline ClusterRouteSmem cluster_route_smem(int T, int H, int E, int k, bool norm) {
  ClusterRouteSmem L;
  const int ksteps = H / 16;
  const int kmax = ((ksteps + kClusterCtas - 1) / kClusterCtas) * 16;  // largest slice, elements
  L.mrows = ((T + 15) / 16) * 16;
  L.erows = ((E + 7) / 8) * 8;
  L.pitch = kmax * 2 + 16;  // +16 bytes: rows fall in different banks for ldmatrix
  const int ngroups = (L.erows / 8 + kMmaIlp - 1) / kMmaIlp;
  L.nitems = (L.mrows / 16) * ngroups;
  L.nsplit = 1;
  while (L.nsplit * 2 * L.nitems <= kRouteWarps) L.nsplit *= 2;
  L.x_off = 0;
  L.w_off = L.x_off + (size_t)L.mrows * L.pitch;
  L.rs_off = L.w_off + (size_t)L.erows * L.pitch;  // norm step: residual slices, like x
  L.rs_staged = norm ? 1 : 0;
  L.split_off = L.rs_off + (L.rs_staged ? (size_t)L.mrows * L.pitch : 0);
  const size_t split_bytes = L.nsplit > 1 ? sizeof(float) * (size_t)L.nsplit * L.mrows * L.erows : 0;
  L.recv_off = L.split_off + split_bytes;  // [kClusterCtas][kTokensPerGroup][erows] partials
  L.lg_off = L.recv_off + sizeof(float) * (size_t)kClusterCtas * kTokensPerGroup * L.erows;
  L.bias_off = L.lg_off + sizeof(float) * (size_t)kTokensPerGroup * L.erows;
  L.idx_off = L.bias_off + sizeof(float) * (size_t)L.erows;
  L.norm_off = L.idx_off + ((sizeof(int32_t) * (size_t)T * k + 15) / 16) * 16;
  // norm step: [kClusterCtas][mrows] range sums received, [mrows] own sums, [mrows] 1 / rms
  const size_t norm_bytes = norm ? sizeof(float) * (size_t)(kClusterCtas + 2) * L.mrows : 0;
  L.bar_off = L.norm_off + norm_bytes;
  L.total = L.bar_off + 32;
  if (L.rs_staged && L.total > kClusterSmemCap) {
    // no room for the residual slices: the kernel reads them from global memory
    const size_t rs_bytes = (size_t)L.mrows * L.pitch;
    L.rs_staged = 0;
    L.split_off -= rs_bytes;
    L.recv_off -= rs_bytes;
    L.lg_off -= rs_bytes;
    L.bias_off -= rs_bytes;
    L.idx_off -= rs_bytes;
    L.norm_off -= rs_bytes;
    L.bar_off -= rs_bytes;
    L.total -= rs_bytes;
  }
  return L;
}

constexpr uint64_t kRouteWaitLimit = 1000000000ull;  // ns a bounded wait may take (1 s)

__global__ void __cluster_dims__(kClusterCtas, 1, 1) __launch_bounds__(kRouteThreads)
    route_cluster_kernel(RouteParams p) {
  extern __shared__ __align__(16) uint8_t rc_smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  namespace cg = cooperative_groups;
  const int rank = (int)cg::this_cluster().block_rank();
  const bool norm = p.norm.norm_w != nullptr;
  const ClusterRouteSmem L = cluster_route_smem(p.T, p.H, p.E, p.k, norm);
  uint8_t* xs = rc_smem + L.x_off;
  uint8_t* wsm = rc_smem + L.w_off;
  uint8_t* rs = rc_smem + L.rs_off;
  float* split = reinterpret_cast<float*>(rc_smem + L.split_off);  // [nsplit][mrows][erows]
  float* recv = reinterpret_cast<float*>(rc_smem + L.recv_off);    // [src rank][token - 8*rank][erows]
  float* lg = reinterpret_cast<float*>(rc_smem + L.lg_off);        // [8][erows]
  float* sbias = reinterpret_cast<float*>(rc_smem + L.bias_off);   // [erows]
  int32_t* sidx = reinterpret_cast<int32_t*>(rc_smem + L.idx_off); // [T*k], filled in CTA 0
  uint64_t* bar = reinterpret_cast<uint64_t*>(rc_smem + L.bar_off);
  uint64_t* bar_stage = bar;      // this CTA's operand slices have landed
  uint64_t* bar_part = bar + 1;   // every peer's partials of this CTA's tokens have landed
  uint64_t* bar_idx = bar + 2;    // (CTA 0) every token's top-k indices have landed
  uint64_t* bar_norm = bar + 3;   // (norm step) every CTA's range sums have landed
  float* norm_recv = reinterpret_cast<float*>(rc_smem + L.norm_off);  // [src rank][mrows]
  float* norm_own = norm_recv + kClusterCtas * L.mrows;               // [mrows]
  float* norm_rinv_s = norm_own + L.mrows;                            // [mrows]
  const int t_own = rank * kTokensPerGroup;
  const int n_own = max(0, min(kTokensPerGroup, p.T - t_own));
  const bool builds = rank == 0 && p.build_table;

  // this CTA's slice of the hidden dimension, in steps of 16
  const int ksteps = p.H / 16;
  const int ks0 = rank * ksteps / kClusterCtas, ks1 = (rank + 1) * ksteps / kClusterCtas;
  const uint32_t slice_bytes = (uint32_t)(ks1 - ks0) * 32;
  if (tid == 0) {
    mbar_init(bar_stage, 1);
    mbar_init(bar_part, 1);
    mbar_init(bar_idx, 1);
    mbar_init(bar_norm, 1);
    fence_mbar_init();
    if (norm) mbar_arrive_expect_tx(bar_norm, (uint32_t)(kClusterCtas * p.T * sizeof(float)));
    if (n_own > 0) mbar_arrive_expect_tx(bar_part, (uint32_t)(kClusterCtas * n_own * L.erows * sizeof(float)));
    if (builds) mbar_arrive_expect_tx(bar_idx, (uint32_t)(p.T * p.k * sizeof(int32_t)));
    if (slice_bytes > 0)
      mbar_arrive_expect_tx(bar_stage, slice_bytes * (uint32_t)(p.T + p.E + (L.rs_staged ? p.T : 0)));
  }
  __syncthreads();
  cluster_arrive_release();  // this CTA's barriers are initialised
  // Router rows and bias first: weights, never written by the launches before this
  // one.  Then the dependency wait, and only after it the activation rows (x may
  // come from the previous kernel) and every write.
  if (slice_bytes > 0) {
    for (int r = tid; r < p.E; r += kRouteThreads)
      bulk_load(wsm + (size_t)r * L.pitch, p.w_router + (size_t)r * p.H + ks0 * 16, slice_bytes, bar_stage);
  }
  if (p.bias && n_own > 0 && tid < p.E) sbias[tid] = __ldg(p.bias + tid);
  pdl_wait();
  pdl_launch_dependents();
  if (slice_bytes > 0) {
    for (int r = tid; r < p.T; r += kRouteThreads) {
      bulk_load(xs + (size_t)r * L.pitch, p.x + (size_t)r * p.H + ks0 * 16, slice_bytes, bar_stage);
      if (L.rs_staged)
        bulk_load(rs + (size_t)r * L.pitch, p.norm.residual + (size_t)r * p.H + ks0 * 16, slice_bytes, bar_stage);
    }
  }
  // rows the copies never touch: x rows past T, router rows past E
  for (int i = tid; i < (L.mrows - p.T) * (L.pitch / 16); i += kRouteThreads) {
    const int r = p.T + i / (L.pitch / 16), c = i % (L.pitch / 16);
    *reinterpret_cast<uint4*>(xs + (size_t)r * L.pitch + c * 16) = make_uint4(0, 0, 0, 0);
  }
  for (int i = tid; i < (L.erows - p.E) * (L.pitch / 16); i += kRouteThreads) {
    const int r = p.E + i / (L.pitch / 16), c = i % (L.pitch / 16);
    *reinterpret_cast<uint4*>(wsm + (size_t)r * L.pitch + c * 16) = make_uint4(0, 0, 0, 0);
  }
  if (slice_bytes > 0 && !mbar_wait_bounded(bar_stage, 0, kRouteWaitLimit)) report_status(p.status, kStatusTimeoutMain);
  // norm step: this CTA's slice of residual row t (shared or global memory)
  auto res_slice = [&](int t) -> const uint16_t* {
    return L.rs_staged ? reinterpret_cast<const uint16_t*>(rs + (size_t)t * L.pitch)
                       : p.norm.residual + (size_t)t * p.H + ks0 * 16;
  };
  if (norm) {
    // this CTA's range of every row (the range cut every kernel uses)
    for (int t = warp; t < p.T; t += kRouteWarps) {
      const float ssq = norm_range_ssq(reinterpret_cast<const uint16_t*>(xs + (size_t)t * L.pitch), res_slice(t), 0,
                                       2 * (ks1 - ks0));
      if (lane == 0) norm_own[t] = ssq;
    }
  }
  __syncthreads();  // zero rows, the bias and the range sums written by other threads
  cluster_wait_acquire();  // every peer's barriers are initialised: pushes may start
  if (norm) {
    // every CTA gets every range sum, adds them in range order (the same bits in
    // every CTA and in the encoder) and turns its x slice into y in place
    for (int i = tid; i < p.T * kClusterCtas; i += kRouteThreads) {
      const int t = i / kClusterCtas;
      const uint32_t dst = (uint32_t)(i - t * kClusterCtas);
      st_async_b32(mapa_shared(smem_u32(norm_recv + rank * L.mrows + t), dst), __float_as_uint(norm_own[t]),
                   mapa_shared(smem_u32(bar_norm), dst));
    }
    if (!mbar_wait_cluster_bounded(bar_norm, 0, kRouteWaitLimit)) report_status(p.status, kStatusTimeoutMain);
    for (int t = tid; t < p.T; t += kRouteThreads) {
      float part[kNormSlices];
#pragma unroll
      for (int q = 0; q < kNormSlices; ++q) part[q] = norm_recv[q * L.mrows + t];
      norm_rinv_s[t] = norm_rinv(part, p.H, p.norm.eps);
    }
    __syncthreads();
    const int nv = 2 * (ks1 - ks0);
    const uint4* gam = reinterpret_cast<const uint4*>(p.norm.norm_w) + 2 * ks0;
    for (int i = tid; i < p.T * nv; i += kRouteThreads) {
      const int t = i / nv, v = i - t * nv;
      uint4* xp = reinterpret_cast<uint4*>(xs + (size_t)t * L.pitch) + v;
      *xp = norm_apply8(*xp, reinterpret_cast<const uint4*>(res_slice(t))[v], __ldg(gam + v), norm_rinv_s[t]);
    }
    __syncthreads();
  }

  // shared::cluster addresses of every owner's receive area and barrier
  const uint32_t recv_u = smem_u32(recv), bar_part_u = smem_u32(bar_part);
  // partial logits: a warp takes one (row block, column group) item, or one K
  // share of it; each A fragment loaded from shared memory serves kMmaIlp MMAs
  {
    const int ntn = L.erows / 8;
    const int ngroups = (ntn + kMmaIlp - 1) / kMmaIlp;
    const int kn = ks1 - ks0;
    const uint32_t xs_u = smem_u32(xs), ws_u = smem_u32(wsm);
    for (int job = warp; job < L.nitems * L.nsplit; job += kRouteWarps) {
      const int item = job / L.nsplit, sp = job - item * L.nsplit;
      const int mi = item / ngroups, n0 = (item - mi * ngroups) * kMmaIlp;
      const int kk0 = sp * kn / L.nsplit, kk1 = (sp + 1) * kn / L.nsplit;
      float c[kMmaIlp][4];
      uint32_t b_addr[kMmaIlp];
      // ldmatrix row addresses: A rows mi*16 + lane%16, column half lane/16; B rows
      // ni*8 + lane%8, column half (lane/8)%2 (a column block past E repeats the last)
      const uint32_t a_addr = xs_u + (uint32_t)((mi * 16 + (lane & 15)) * L.pitch + (lane >> 4) * 16);
#pragma unroll
      for (int q = 0; q < kMmaIlp; ++q) {
        const int ni = min(n0 + q, ntn - 1);
        b_addr[q] = ws_u + (uint32_t)((ni * 8 + (lane & 7)) * L.pitch + ((lane >> 3) & 1) * 16);
        c[q][0] = c[q][1] = c[q][2] = c[q][3] = 0.f;
      }
      for (int kk = kk0; kk < kk1; ++kk) {
        uint32_t a[4];
        ldmatrix_x4(a, a_addr + kk * 32);
#pragma unroll
        for (int q = 0; q < kMmaIlp; ++q) {
          uint32_t b[2];
          ldmatrix_x2(b, b_addr[q] + kk * 32);
          mma_bf16_16816(c[q], a, b);
        }
      }
      // fragment rows r0 = mi*16 + lane/4 and r0 + 8, columns ni*8 + 2*(lane%4) + {0,1}
      const int r0 = mi * 16 + (lane >> 2);
#pragma unroll
      for (int q = 0; q < kMmaIlp; ++q) {
        const int ni = n0 + q;
        if (ni >= ntn) break;
        const int c0 = ni * 8 + (lane & 3) * 2;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int r = r0 + 8 * h;
          if (L.nsplit > 1) {
            *reinterpret_cast<float2*>(split + ((size_t)sp * L.mrows + r) * L.erows + c0) =
                make_float2(c[q][2 * h], c[q][2 * h + 1]);
          } else if (r < p.T) {
            const uint32_t owner = (uint32_t)(r / kTokensPerGroup);
            const uint32_t off = (uint32_t)(((rank * kTokensPerGroup + r % kTokensPerGroup) * L.erows + c0) * 4);
            st_async_v2_f32(mapa_shared(recv_u + off, owner), c[q][2 * h], c[q][2 * h + 1],
                            mapa_shared(bar_part_u, owner));
          }
        }
      }
    }
    if (L.nsplit > 1) {
      // the K shares of each partial, summed in share order, then pushed
      __syncthreads();
      const int c4n = L.erows / 4;
      for (int i = tid; i < p.T * c4n; i += kRouteThreads) {
        const int r = i / c4n, c4 = i - r * c4n;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int sp = 0; sp < L.nsplit; ++sp) {
          const float4 u = *reinterpret_cast<const float4*>(split + ((size_t)sp * L.mrows + r) * L.erows + 4 * c4);
          v.x += u.x;
          v.y += u.y;
          v.z += u.z;
          v.w += u.w;
        }
        const uint32_t owner = (uint32_t)(r / kTokensPerGroup);
        const uint32_t off = (uint32_t)(((rank * kTokensPerGroup + r % kTokensPerGroup) * L.erows + 4 * c4) * 4);
        st_async_v4_f32(mapa_shared(recv_u + off, owner), v, mapa_shared(bar_part_u, owner));
      }
    }
  }
  // logits of this CTA's tokens: partials summed in rank order, then the bias
  if (n_own > 0) {
    if (!mbar_wait_cluster_bounded(bar_part, 0, kRouteWaitLimit)) report_status(p.status, kStatusTimeoutMain);
    for (int i = tid; i < n_own * p.E; i += kRouteThreads) {
      const int r = i / p.E, e = i - r * p.E;
      float sum = 0.f;
#pragma unroll
      for (int b = 0; b < kClusterCtas; ++b) sum += recv[(b * kTokensPerGroup + r) * L.erows + e];
      if (p.bias) sum += sbias[e];
      lg[r * L.erows + e] = sum;
      p.logits[(size_t)(t_own + r) * p.E + e] = sum;
    }
    __syncthreads();
    // top-k of one token per warp; the indices also go to CTA 0
    if (warp < n_own) {
      const int t = t_own + warp;
      const int sel = topk_softmax_warp<true>(lg + warp * L.erows, p.E, p.k, p.topk_idx + (size_t)t * p.k,
                                              p.topk_w + (size_t)t * p.k, p.gating);
      if (p.build_table && lane < p.k)
        st_async_b32(mapa_shared(smem_u32(sidx + t * p.k + lane), 0), (uint32_t)sel, mapa_shared(smem_u32(bar_idx), 0));
    }
  }
  if (!builds) return;
  if (p.T * p.k <= 32) {
    // few assignments: one warp builds the table
    if (warp != 0) return;
    if (!mbar_wait_cluster_bounded(bar_idx, 0, kRouteWaitLimit)) report_status(p.status, kStatusTimeoutMain);
    build_tile_table_warp<true>(sidx, p.T * p.k, p.E, p.bm, p.counts, p.offsets, p.perm, p.inv_perm, p.tiles,
                                p.num_tiles, p.status, p.pad_inv != 0);
    return;
  }
  if (!mbar_wait_cluster_bounded(bar_idx, 0, kRouteWaitLimit)) report_status(p.status, kStatusTimeoutMain);
  build_tile_table_block<true>(sidx, p.T * p.k, p.E, p.bm, p.counts, p.offsets, p.perm, p.inv_perm, p.tiles,
                               p.num_tiles, p.status, p.pad_inv != 0);
}

// ------------------------------------------------------------------ many tokens
// T > 64: one block per 32 tokens computes the logits of all experts on the tensor
// cores (mma.sync bf16, fp32 accumulate), with x and router chunks of 128 values
// staged by cp.async into a double-buffered ring; then one warp per token selects
// its top-k, and the last block to finish (an integer arrival count, no spinning)
// builds the tile table.  Every block reads the router weights once (L2).
constexpr int kMmaTokens = 32;
constexpr int kMmaKChunk = 128;
constexpr int kMmaPitch = kMmaKChunk * 2 + 16;  // bytes per staged row: an odd multiple of 16
constexpr int kMmaMaxNtpw = kMaxExperts / 8 / kRouteWarps;  // 8-expert column blocks per warp

struct MmaRouteSmem {
  int erows;
  size_t stage, xo, wo, ro, go, lg_off, total;  // stage b of buffer "o" starts at b * stage + o
  __host__ __device__ size_t x_off(int b) const { return b * stage + xo; }
  __host__ __device__ size_t w_off(int b) const { return b * stage + wo; }
  __host__ __device__ size_t r_off(int b) const { return b * stage + ro; }
  __host__ __device__ size_t g_off(int b) const { return b * stage + go; }
};
// norm: two more buffers per stage, the residual chunk [32][pitch] and the weight chunk [128]
__host__ __device__ inline MmaRouteSmem mma_route_smem(int E, bool norm) {
  MmaRouteSmem L;
  L.erows = ((E + 7) / 8) * 8;
  const size_t xb = (size_t)kMmaTokens * kMmaPitch, wb = (size_t)L.erows * kMmaPitch;
  const size_t rb = norm ? xb : 0, gb = norm ? kMmaKChunk * 2 : 0;
  L.stage = xb + wb + rb + gb;
  L.xo = 0;
  L.wo = xb;
  L.ro = xb + wb;
  L.go = xb + wb + rb;
  L.lg_off = 2 * L.stage;
  L.total = L.lg_off + sizeof(float) * (size_t)kMmaTokens * L.erows;
  return L;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int kPending>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(kPending) : "memory");
}

__global__ void __launch_bounds__(kRouteThreads) route_mma_kernel(RouteParams p) {
  extern __shared__ __align__(16) uint8_t rm_smem[];
  __shared__ int s_last;
  __shared__ float s_rinv[kMmaTokens];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_wait();  // the previous kernel may still write x or read this call's outputs
  pdl_launch_dependents();
  const bool norm = p.norm.norm_w != nullptr;
  const MmaRouteSmem L = mma_route_smem(p.E, norm);
  const int t0 = blockIdx.x * kMmaTokens;
  const int nt = min(kMmaTokens, p.T - t0);
  const int nchunks = (p.H + kMmaKChunk - 1) / kMmaKChunk;
  const uint32_t smem0 = smem_u32(rm_smem);
  // chunk c of x rows t0.. and of every router row into buffer b; 16-byte segments
  // past H or past the last token / expert are zero-filled (H is a multiple of 32)
  auto stage = [&](int c, int b) {
    const int k0 = c * kMmaKChunk;
    for (int i = tid; i < kMmaTokens * (kMmaKChunk / 8); i += kRouteThreads) {
      const int r = i / (kMmaKChunk / 8), sg = i - r * (kMmaKChunk / 8), k = k0 + sg * 8;
      const bool ok = r < nt && k < p.H;
      cp_async16(smem0 + (uint32_t)(L.x_off(b) + r * kMmaPitch + sg * 16), ok ? p.x + (size_t)(t0 + r) * p.H + k : p.x,
                 ok ? 16u : 0u);
    }
    for (int i = tid; i < L.erows * (kMmaKChunk / 8); i += kRouteThreads) {
      const int r = i / (kMmaKChunk / 8), sg = i - r * (kMmaKChunk / 8), k = k0 + sg * 8;
      const bool ok = r < p.E && k < p.H;
      cp_async16(smem0 + (uint32_t)(L.w_off(b) + r * kMmaPitch + sg * 16),
                 ok ? p.w_router + (size_t)r * p.H + k : p.w_router, ok ? 16u : 0u);
    }
    if (norm) {
      for (int i = tid; i < kMmaTokens * (kMmaKChunk / 8); i += kRouteThreads) {
        const int r = i / (kMmaKChunk / 8), sg = i - r * (kMmaKChunk / 8), k = k0 + sg * 8;
        const bool ok = r < nt && k < p.H;
        cp_async16(smem0 + (uint32_t)(L.r_off(b) + r * kMmaPitch + sg * 16),
                   ok ? p.norm.residual + (size_t)(t0 + r) * p.H + k : p.norm.residual, ok ? 16u : 0u);
      }
      for (int sg = tid; sg < kMmaKChunk / 8; sg += kRouteThreads) {
        const bool ok = k0 + sg * 8 < p.H;
        cp_async16(smem0 + (uint32_t)(L.g_off(b) + sg * 16), ok ? p.norm.norm_w + k0 + sg * 8 : p.norm.norm_w,
                   ok ? 16u : 0u);
      }
    }
    cp_async_commit();
  };
  if (norm) {
    // 1 / rms of the block's rows (the same range cut and order as every other kernel)
    for (int r = warp; r < nt; r += kRouteWarps) {
      const float ri = norm_row_rinv(p.x + (size_t)(t0 + r) * p.H, p.norm.residual + (size_t)(t0 + r) * p.H, p.H,
                                     p.norm.eps);
      if (lane == 0) s_rinv[r] = ri;
    }
  }
  // warp w owns 8-expert column blocks [w ntpw, (w + 1) ntpw) and both 16-token row blocks
  const int ntiles = L.erows / 8;
  const int ntpw = (ntiles + kRouteWarps - 1) / kRouteWarps;
  const int nb0 = warp * ntpw;
  float acc[2][kMmaMaxNtpw][4];
#pragma unroll
  for (int mi = 0; mi < 2; ++mi)
#pragma unroll
    for (int q = 0; q < kMmaMaxNtpw; ++q) acc[mi][q][0] = acc[mi][q][1] = acc[mi][q][2] = acc[mi][q][3] = 0.f;
  stage(0, 0);
  for (int c = 0; c < nchunks; ++c) {
    const int b = c & 1;
    if (c + 1 < nchunks) {
      stage(c + 1, b ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    if (norm) {
      // x chunk -> y chunk in place
      const int k0 = c * kMmaKChunk;
      for (int i = tid; i < nt * (kMmaKChunk / 8); i += kRouteThreads) {
        const int r = i / (kMmaKChunk / 8), sg = i - r * (kMmaKChunk / 8);
        if (k0 + sg * 8 >= p.H) continue;
        uint4* xp = reinterpret_cast<uint4*>(rm_smem + L.x_off(b) + r * kMmaPitch + sg * 16);
        const uint4 rv = *reinterpret_cast<const uint4*>(rm_smem + L.r_off(b) + r * kMmaPitch + sg * 16);
        const uint4 gv = *reinterpret_cast<const uint4*>(rm_smem + L.g_off(b) + sg * 16);
        *xp = norm_apply8(*xp, rv, gv, s_rinv[r]);
      }
      __syncthreads();
    }
    const uint32_t xs = smem0 + (uint32_t)L.x_off(b), wsm = smem0 + (uint32_t)L.w_off(b);
#pragma unroll
    for (int ks = 0; ks < kMmaKChunk / 16; ++ks) {
      uint32_t a0[4], a1[4];
      ldmatrix_x4(a0, xs + (uint32_t)(((lane & 15)) * kMmaPitch + ks * 32 + (lane >> 4) * 16));
      ldmatrix_x4(a1, xs + (uint32_t)((16 + (lane & 15)) * kMmaPitch + ks * 32 + (lane >> 4) * 16));
#pragma unroll
      for (int q = 0; q < kMmaMaxNtpw; ++q) {
        const int ni = nb0 + q;
        if (q < ntpw && ni < ntiles) {
          uint32_t bf[2];
          ldmatrix_x2(bf, wsm + (uint32_t)((ni * 8 + (lane & 7)) * kMmaPitch + ks * 32 + ((lane >> 3) & 1) * 16));
          mma_bf16_16816(acc[0][q], a0, bf);
          mma_bf16_16816(acc[1][q], a1, bf);
        }
      }
    }
    __syncthreads();  // buffer b is staged again two chunks later
  }
  // logits (+ bias): fragment rows mi*16 + lane/4 (+8), columns ni*8 + 2*(lane%4) (+1)
  float* lg = reinterpret_cast<float*>(rm_smem + L.lg_off);  // [32][erows]
#pragma unroll
  for (int mi = 0; mi < 2; ++mi)
#pragma unroll
    for (int q = 0; q < kMmaMaxNtpw; ++q) {
      const int ni = nb0 + q;
      if (q >= ntpw || ni >= ntiles) continue;
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int r = mi * 16 + (lane >> 2) + 8 * h, e = ni * 8 + (lane & 3) * 2 + cc;
          float v = acc[mi][q][2 * h + cc];
          if (e < p.E) {
            if (p.bias) v += __ldg(p.bias + e);
            lg[r * L.erows + e] = v;
            if (r < nt) p.logits[(size_t)(t0 + r) * p.E + e] = v;
          }
        }
    }
  __syncthreads();
  // top-k of one token per warp
  for (int r = warp; r < nt; r += kRouteWarps) {
    const int t = t0 + r;
    topk_softmax_warp<true>(lg + r * L.erows, p.E, p.k, p.topk_idx + (size_t)t * p.k, p.topk_w + (size_t)t * p.k,
                            p.gating);
  }
  if (!p.build_table) return;
  // the last block to finish builds the table
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const unsigned old = atomicAdd(p.sync, 1u);
    s_last = (old == gridDim.x - 1) ? 1 : 0;
    if (s_last) p.sync[0] = 0;  // ready for the next call
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // every block's indices into this block's (now idle) shared memory first, with
  // wide loads all in flight, so the table's passes over them do not wait on L2
  const int Tk = p.T * p.k;
  if ((size_t)Tk * sizeof(int32_t) <= L.total) {
    int32_t* sidx = reinterpret_cast<int32_t*>(rm_smem);
    // wide loads only from a 16-byte aligned array (a caller's output buffer may not be)
    const int n4 = (reinterpret_cast<uintptr_t>(p.topk_idx) & 15) == 0 ? Tk / 4 : 0;
    const int4* src4 = reinterpret_cast<const int4*>(p.topk_idx);
    for (int i0 = tid; i0 < n4; i0 += 8 * kRouteThreads) {
      int4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + u * kRouteThreads;
        v[u] = i < n4 ? __ldcg(src4 + i) : make_int4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + u * kRouteThreads;
        if (i < n4) reinterpret_cast<int4*>(sidx)[i] = v[u];
      }
    }
    for (int i = n4 * 4 + tid; i < Tk; i += kRouteThreads) sidx[i] = __ldcg(p.topk_idx + i);
    __syncthreads();
    build_tile_table_block<true>(sidx, Tk, p.E, p.bm, p.counts, p.offsets, p.perm, p.inv_perm, p.tiles,
                                 p.num_tiles, p.status, p.pad_inv != 0);
  } else {
    build_tile_table_block(p.topk_idx, Tk, p.E, p.bm, p.counts, p.offsets, p.perm, p.inv_perm, p.tiles,
                           p.num_tiles, p.status, p.pad_inv != 0);
  }
}

__global__ void __launch_bounds__(kRouteThreads) tile_table_kernel(const int32_t* idx, int Tk, int E, int bm,
                                                                   int32_t* counts, int32_t* offsets, int32_t* perm,
                                                                   int32_t* inv_perm, TileEntry* tiles,
                                                                   int32_t* num_tiles) {
  if (Tk <= 32) {
    if (threadIdx.x < 32) build_tile_table_warp(idx, Tk, E, bm, counts, offsets, perm, inv_perm, tiles, num_tiles, nullptr);
    return;
  }
  build_tile_table_block(idx, Tk, E, bm, counts, offsets, perm, inv_perm, tiles, num_tiles, nullptr);
}

// The cluster kernel serves few tokens when its operands fit in shared memory and
// the device can place one cluster of kClusterCtas CTAs with that much memory.
static bool use_cluster_route(const RouteParams& p, size_t* smem_out) {
  if (p.from_logits || p.T > kClusterMaxTokens) return false;
  const ClusterRouteSmem L = cluster_route_smem(p.T, p.H, p.E, p.k, p.norm.norm_w != nullptr);
  if (L.total > kClusterSmemCap) return false;
  // per device: 0 not probed yet, 1 usable, -1 not.  The probe runs under a lock and
  // its result is published once, so concurrent first calls all see the same answer.
  static std::atomic<int> state[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  int st = state[dev].load(std::memory_order_acquire);
  if (st == 0) {
    std::lock_guard<std::mutex> lock(mu);
    st = state[dev].load(std::memory_order_relaxed);
    if (st == 0) {
      st = -1;
      if (cudaFuncSetAttribute(route_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)kClusterSmemCap) == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(kClusterCtas);
        cfg.blockDim = dim3(kRouteThreads);
        cfg.dynamicSmemBytes = kClusterSmemCap;
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, route_cluster_kernel, &cfg) == cudaSuccess && clusters > 0)
          st = 1;
      }
      cudaGetLastError();  // a refused query leaves no sticky error
      state[dev].store(st, std::memory_order_release);
    }
  }
  *smem_out = L.total;
  return st == 1;
}

cudaError_t launch_route(const RouteParams& p, cudaStream_t stream) {
  size_t csmem = 0;
  if (use_cluster_route(p, &csmem))
    return launch_pdl(route_cluster_kernel, dim3(kClusterCtas), dim3(kRouteThreads), csmem, stream, p);
  if (!p.from_logits) {
    // many tokens: tensor-core logits, 32 tokens per block
    const MmaRouteSmem L = mma_route_smem(p.E, p.norm.norm_w != nullptr);
    static SmemOptIn opt_in;
    const cudaError_t e = opt_in.ensure(route_mma_kernel, (int)L.total);
    if (e != cudaSuccess) return e;
    return launch_pdl(route_mma_kernel, dim3(ceil_div(p.T, kMmaTokens)), dim3(kRouteThreads), L.total, stream, p);
  }
  const int groups = ceil_div(p.T, kTokensPerGroup);
  dim3 grid(groups, p.from_logits ? 1 : ceil_div(p.E, p.experts_per_block));
  const size_t smem = p.from_logits ? 0 : (size_t)kTokensPerGroup * p.H * sizeof(uint16_t);
  // static (tile-table scratch) + dynamic (activation tile) shared memory may exceed
  // the 48 KB default window
  static SmemOptIn opt_in12, opt_in4;
  cudaError_t e = opt_in12.ensure(route_kernel<12>, (int)smem);
  if (e == cudaSuccess) e = opt_in4.ensure(route_kernel<4>, (int)smem);
  if (e != cudaSuccess) return e;
  if (p.T <= 64) return launch_pdl(route_kernel<12>, grid, dim3(kRouteThreads), smem, stream, p);
  return launch_pdl(route_kernel<4>, grid, dim3(kRouteThreads), smem, stream, p);
}

cudaError_t launch_tile_table(const int32_t* idx, int Tk, int E, int bm, int32_t* counts, int32_t* offsets,
                              int32_t* perm, int32_t* inv_perm, TileEntry* tiles, int32_t* num_tiles,
                              cudaStream_t stream) {
  tile_table_kernel<<<1, kRouteThreads, 0, stream>>>(idx, Tk, E, bm, counts, offsets, perm, inv_perm, tiles,
                                                      num_tiles);
  return cudaGetLastError();
}

}  // namespace moe
