// Data movement kernels around the expert GEMMs:
//  * encode_x: activation rows encoded once per token as four E2M1 terms with E8M0
//    block scales (the tensor-core B operand).  In the forward it overlaps routing,
//    then writes its rows straight into the tile order of the token's assignments
//    (the permute); with the norm step it encodes y = RMSNorm(x + residual);
//  * gather_x: the permute for the stage entry point (token order -> tile order);
//  * scatter_x16: the permute of the bf16-weight layer (bf16 rows into tile order);
//  * combine: weighted top-k sum of the down GEMM's slots, bf16 out, and the
//    residual stream of the norm step;
//  * prepare: one-time re-layout of the E8M0 scales of raw MXFP4 expert weights into
//    the tensor-memory atom order ("MXFP4 MoE on tensor cores": weights permuted once
//    at load; nothing is re-quantised; the codes stay row major);
//  * hidden_dequant: expands the encoded SwiGLU output for inspection.
#include "moe_common.cuh"
#include "moe_kernels.cuh"
#include "sm100_ptx.cuh"

namespace moe {

namespace {
constexpr int kAuxThreads = 256;

}  // namespace

// Max over the 4 lanes (aligned groups of 4) that hold one 32-value MX block.
__device__ __forceinline__ float quad_max(float v) {
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
  return v;
}

// Activation encoding, once per token: one warp per (token, 256-value chunk of x),
// so every load of a call is in flight at once.  Each lane owns 8 consecutive
// values (one 16-byte load); four lanes form one 32-value MX block, and the block
// is written as kTerms E2M1 terms x ~ sum_t q_t * 2^p_t, each term with its own
// E8M0 exponent chosen for the residual left by the terms before.  Values past H
// up to the next multiple of 64 are encoded as zeros so every 64-value MMA step
// reads finite data.  Each token is encoded once however many experts it is routed
// to.  Either the rows are written in token order and the gather below permutes
// them, or (scatter, in the layer's forward) the warp waits for routing and writes
// its encoded values straight to the tile rows of the token's k assignments -- the
// permute step without a launch of its own.
// kNorm: the rows are y = RMSNorm(x + residual).  That instance runs one block per
// token (a warp per 256-value chunk, at least kNormSlices warps): warp q < kNormSlices
// sums range q of the row, and every warp forms the row's 1 / rms from the eight
// sums (the same bits the router computes).
constexpr int kEncodeNormMaxThreads = 1024;
template <bool kNorm>
__global__ void __launch_bounds__(kNorm ? kEncodeNormMaxThreads : kAuxThreads) encode_x_kernel(EncodeXParams p) {
  // the previous kernel may still write x or read this call's buffers, unless the
  // launch before this one already waited for it.  Waiting at the end, this launch
  // also signals its dependents only after that wait: the GEMM after it reads the
  // tile table before its own wait.
  if (!p.wait_at_end) {
    ptx::pdl_wait();
    ptx::pdl_launch_dependents();
  }
  const int lane = threadIdx.x & 31;
  const int nvec_pad = ((p.H + 63) / 64) * 8;  // 8-value vectors per row, padded to 64 values
  const int nchunks = (nvec_pad + 31) / 32;
  int t, chunk;
  float rinv = 0.f;
  if constexpr (kNorm) {
    __shared__ float s_part[kNormSlices];
    t = blockIdx.x;
    chunk = threadIdx.x >> 5;
    if (chunk < kNormSlices) {
      const float ssq = norm_range_ssq(p.x + (size_t)t * p.H, p.norm.residual + (size_t)t * p.H,
                                       norm_slice_vec(p.H, chunk), norm_slice_vec(p.H, chunk + 1));
      if (lane == 0) s_part[chunk] = ssq;
    }
    __syncthreads();
    float part[kNormSlices];
#pragma unroll
    for (int q = 0; q < kNormSlices; ++q) part[q] = s_part[q];
    rinv = norm_rinv(part, p.H, p.norm.eps);
  } else {
    const long long gw = ((long long)blockIdx.x * kAuxThreads + threadIdx.x) >> 5;
    t = (int)(gw / nchunks);
    chunk = (int)(gw - (long long)t * nchunks);
  }
  if (t >= p.T || chunk >= nchunks) {
    if (p.wait_at_end) {
      ptx::pdl_wait();
      ptx::pdl_launch_dependents();
    }
    return;
  }
  const int v = chunk * 32 + lane;
  const int nvec = p.H / 8;
  float f[8];
  if (v < nvec) {
    uint4 raw = __ldg(reinterpret_cast<const uint4*>(p.x + (size_t)t * p.H) + v);
    if (kNorm)
      raw = norm_apply8(raw, __ldg(reinterpret_cast<const uint4*>(p.norm.residual + (size_t)t * p.H) + v),
                        __ldg(reinterpret_cast<const uint4*>(p.norm.norm_w) + v), rinv);
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) f[i] = 0.f;
  }
  const int kgroup = v >> 4;  // 16 vectors = 128 values per K group
  uint32_t words[kTerms], sfws[kTerms];
#pragma unroll
  for (int term = 0; term < kTerms; ++term) {
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
    amax = quad_max(amax);
    const int pe = mx_e2m1_exponent(amax);
    const float inv = pow2_int(-pe), sc = pow2_int(pe);
    uint32_t word = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t pair = f32x2_to_e2m1x2(f[2 * i] * inv, f[2 * i + 1] * inv);
      f[2 * i] -= e2m1_to_f32(pair & 15u) * sc;
      f[2 * i + 1] -= e2m1_to_f32(pair >> 4) * sc;
      word |= pair << (8 * i);
    }
    // exponents of 4 consecutive MX blocks sit in lanes 0, 4, 8, 12 (and 16..28)
    const uint32_t e8 = static_cast<uint32_t>(pe + 127);
    const int base = lane & ~15;
    const uint32_t sfw = __shfl_sync(0xffffffffu, e8, base) | (__shfl_sync(0xffffffffu, e8, base + 4) << 8) |
                         (__shfl_sync(0xffffffffu, e8, base + 8) << 16) |
                         (__shfl_sync(0xffffffffu, e8, base + 12) << 24);
    words[term] = word;
    sfws[term] = sfw;
    if (!p.scatter && v < nvec_pad) {
      const size_t row = ((size_t)kgroup * p.T + t) * kTerms + term;
      *reinterpret_cast<uint32_t*>(p.q + row * 64 + (v & 15) * 4) = word;
      if ((lane & 15) == 0) p.sf[row] = sfw;
    }
  }
  if (!p.wait_at_end) return;
  ptx::pdl_wait();  // routing has completed: its tile table is visible
  ptx::pdl_launch_dependents();
  if (!p.scatter) return;
  // the permute step: this token's rows go to the tile rows of its k assignments
  // (padded row v: tile v / bm, row v % bm; an invalid expert has no row)
  for (int j0 = 0; j0 < p.k; j0 += 32) {
    int tile_j = -1, r_j = 0;
    if (j0 + lane < p.k) {
      const int a = t * p.k + j0 + lane;
      const int e = __ldcg(p.topk_idx + a);
      const int prow = __ldcg(p.pad_row + a);
      if (e >= 0 && e < p.E && prow >= 0) {
        tile_j = prow / p.bm;
        r_j = prow % p.bm;
      }
    }
    const int nj = min(32, p.k - j0);
    for (int j = 0; j < nj; ++j) {
      const int tile = __shfl_sync(0xffffffffu, tile_j, j), r = __shfl_sync(0xffffffffu, r_j, j);
      if (tile < 0 || tile >= p.max_tiles || v >= nvec_pad) continue;
      uint8_t* sf = p.sf_tile + ((size_t)tile * p.kg_tile + kgroup) * (kSfAtomBytes * act_sf_atoms(p.bm));
#pragma unroll
      for (int term = 0; term < kTerms; ++term) {
        *reinterpret_cast<uint32_t*>(p.q_tile + act_offset(tile, term, r, v * 8, p.max_tiles, p.bm)) = words[term];
        if ((lane & 15) == 0) *reinterpret_cast<uint32_t*>(sf + sf_atom_offset(act_row(term, r, p.bm), 0)) = sfws[term];
      }
    }
  }
}

cudaError_t launch_encode_x(const EncodeXParams& p, cudaStream_t stream) {
  const int nvec_pad = ((p.H + 63) / 64) * 8;
  const long long warps = (long long)p.T * ((nvec_pad + 31) / 32);
  const int blocks = (int)((warps * 32 + kAuxThreads - 1) / kAuxThreads);
  if (p.norm.norm_w) {
    const int nw = (nvec_pad + 31) / 32 > kNormSlices ? (nvec_pad + 31) / 32 : kNormSlices;
    if (nw * 32 > kEncodeNormMaxThreads) return cudaErrorInvalidValue;
    return launch_pdl(encode_x_kernel<true>, dim3(p.T > 0 ? p.T : 1), dim3(nw * 32), 0, stream, p);
  }
  return launch_pdl(encode_x_kernel<false>, dim3(blocks > 0 ? blocks : 1), dim3(kAuxThreads), 0, stream, p);
}

__global__ void __launch_bounds__(kAuxThreads) scatter_x16_kernel(ScatterX16Params p) {
  const int nv = p.H / 8;
  const long long i = (long long)blockIdx.x * kAuxThreads + threadIdx.x;
  const bool live = i < (long long)p.T * nv;
  const int t = live ? (int)(i / nv) : 0, v = live ? (int)(i - (long long)t * nv) : 0;
  uint4 val = make_uint4(0, 0, 0, 0);
  if (live) val = __ldg(reinterpret_cast<const uint4*>(p.x + (size_t)t * p.H) + v);
  ptx::pdl_wait();  // routing has completed: its tile table is visible
  ptx::pdl_launch_dependents();
  if (!live) return;
  for (int j = 0; j < p.k; ++j) {
    const int a = t * p.k + j;
    const int e = __ldcg(p.topk_idx + a), prow = __ldcg(p.pad_row + a);
    if (e < 0 || e >= p.E || prow < 0) continue;
    const int tile = prow / p.bm, r = prow % p.bm;
    if (tile >= p.max_tiles) continue;
    *reinterpret_cast<uint4*>(p.q_tile + act16_offset(tile, r, 8 * v, p.max_tiles, p.bm)) = val;
  }
}

cudaError_t launch_scatter_x16(const ScatterX16Params& p, cudaStream_t stream) {
  const long long threads = (long long)p.T * (p.H / 8);
  const int blocks = (int)((threads + kAuxThreads - 1) / kAuxThreads);
  return launch_pdl(scatter_x16_kernel, dim3(blocks > 0 ? blocks : 1), dim3(kAuxThreads), 0, stream, p);
}

// The permute step: every (tile row, K group) copies its token's four encoded
// 64-byte code runs and their exponent words from token order into the tile order
// the gate/up GEMM loads by TMA.  Rows past a tile's last token are left as they
// are (finite: zero-filled once, or earlier encodings) and their products are never
// read.
__global__ void __launch_bounds__(kAuxThreads) gather_x_kernel(GatherXParams p) {
  ptx::pdl_wait();  // the routing launch (tile table) and the encoding before it
  ptx::pdl_launch_dependents();
  const long long i = (long long)blockIdx.x * kAuxThreads + threadIdx.x;
  const int kg = (int)(i % p.kg);
  const long long row = i / p.kg;
  const int tile = (int)(row / p.bm), r = (int)(row - (long long)tile * p.bm);
  if (tile >= p.max_tiles || tile >= __ldcg(p.num_tiles)) return;
  const TileEntry te = load_tile(p.tiles + tile);
  if (r >= te.n_rows) return;
  const int tok = __ldcg(p.perm + te.row_begin + r) / p.k;
  const size_t src_row = ((size_t)kg * p.T + tok) * kTerms;
  const uint4* src = reinterpret_cast<const uint4*>(p.xt_q + src_row * 64);
  uint4 v[kTerms * 4];
#pragma unroll
  for (int j = 0; j < kTerms * 4; ++j) v[j] = __ldcg(src + j);
  const uint4 e = __ldcg(reinterpret_cast<const uint4*>(p.xt_sf + src_row));
  const uint32_t ew[kTerms] = {e.x, e.y, e.z, e.w};
  uint8_t* sf = p.sf + ((size_t)tile * p.kg + kg) * (kSfAtomBytes * act_sf_atoms(p.bm));
#pragma unroll
  for (int t = 0; t < kTerms; ++t) {
    // 16-byte chunks (32 values each) land at their swizzled positions
#pragma unroll
    for (int j = 0; j < 4; ++j)
      *reinterpret_cast<uint4*>(p.q + act_offset(tile, t, r, kg * kKGroup + 32 * j, p.max_tiles, p.bm)) = v[t * 4 + j];
    *reinterpret_cast<uint32_t*>(sf + sf_atom_offset(act_row(t, r, p.bm), 0)) = ew[t];
  }
}

cudaError_t launch_gather_x(const GatherXParams& p, cudaStream_t stream) {
  const long long threads = (long long)p.max_tiles * p.bm * p.kg;
  const int blocks = (int)((threads + kAuxThreads - 1) / kAuxThreads);
  return launch_pdl(gather_x_kernel, dim3(blocks > 0 ? blocks : 1), dim3(kAuxThreads), 0, stream, p);
}

// Weighted top-k combine + unpermute ("Where the time went", row "MoE down +
// combine"): out[t, f] = sum_{j<k} slot[t*k + j, f], each slot already holding
// w_tj * y_tj, summed in fp32 in ascending j and rounded once to bf16 (RNE) -- the
// same order every call.  One thread per 4 features of one token.
__global__ void __launch_bounds__(kAuxThreads) combine_kernel(CombineParams p) {
  ptx::pdl_wait();
  ptx::pdl_launch_dependents();
  const int nq = p.H / 4;
  const long long i = (long long)blockIdx.x * kAuxThreads + threadIdx.x;
  if (i >= (long long)p.T * nq) return;
  const int t = (int)(i / nq), q = (int)(i - (long long)t * nq);
  const float4* s = reinterpret_cast<const float4*>(p.slots + (size_t)t * p.k * p.H) + q;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
  for (int j = 0; j < p.k; ++j) {
    const float4 v = __ldcg(s + (size_t)j * nq);
    acc.x += v.x;
    acc.y += v.y;
    acc.z += v.z;
    acc.w += v.w;
  }
  const uint32_t lo = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(acc.x)) |
                      ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(acc.y)) << 16);
  const uint32_t hi = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(acc.z)) |
                      ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(acc.w)) << 16);
  // the residual stream after the norm step's add, read before out is written and
  // written by the thread that read it: out and residual_out may each alias x or residual
  uint2 res = make_uint2(0, 0);
  if (p.residual_out) {
    const uint2 xv = reinterpret_cast<const uint2*>(p.x + (size_t)t * p.H)[q];
    const uint2 rv = reinterpret_cast<const uint2*>(p.residual + (size_t)t * p.H)[q];
    const uint32_t xw[2] = {xv.x, xv.y}, rw[2] = {rv.x, rv.y};
    uint32_t o[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float a = bf16_round_f32(__fadd_rn(__uint_as_float(xw[i] << 16), __uint_as_float(rw[i] << 16)));
      const float b = bf16_round_f32(__fadd_rn(__uint_as_float(xw[i] & 0xFFFF0000u), __uint_as_float(rw[i] & 0xFFFF0000u)));
      o[i] = (__float_as_uint(a) >> 16) | (__float_as_uint(b) & 0xFFFF0000u);
    }
    res = make_uint2(o[0], o[1]);
  }
  reinterpret_cast<uint2*>(p.out + (size_t)t * p.H)[q] = make_uint2(lo, hi);
  if (p.residual_out) reinterpret_cast<uint2*>(p.residual_out + (size_t)t * p.H)[q] = res;
}

cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream) {
  const long long threads = (long long)p.T * (p.H / 4);
  const int blocks = (int)((threads + kAuxThreads - 1) / kAuxThreads);
  return launch_pdl(combine_kernel, dim3(blocks > 0 ? blocks : 1), dim3(kAuxThreads), 0, stream, p);
}

// Scales: one thread per atom byte; rows past the group and blocks past K get 127.
__global__ void prepare_scales_kernel(PrepareParams p) {
  const long long atoms = (long long)p.E * p.groups * p.mt * p.kg;
  const long long total = atoms * kSfAtomBytes;
  const int kblocks = p.K / kMxBlock;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    long long atom = i / kSfAtomBytes;
    const int byte = (int)(i - atom * kSfAtomBytes);
    const int kgi = (int)(atom % p.kg);
    atom /= p.kg;
    const int mt = (int)(atom % p.mt);
    atom /= p.mt;
    const int grp = (int)(atom % p.groups);
    const int e = (int)(atom / p.groups);
    const int l = byte >> 4, c = (byte >> 2) & 3, b = byte & 3;
    const int row = mt * kMTile + c * 32 + l;
    const int blk = kgi * 4 + b;
    uint8_t val = 127;
    if (row < p.rows_per_group && blk < kblocks) {
      val = p.scales[((size_t)e * p.R + (size_t)grp * p.rows_per_group + row) * kblocks + blk];
      if (val == 255) atomicOr(p.flag, 1u);
    }
    p.dst_scales[i] = val;
  }
}

cudaError_t launch_prepare(const PrepareParams& p, cudaStream_t stream) {
  // the codes keep their row-major layout
  cudaError_t e = cudaMemcpyAsync(p.dst_codes, p.codes, (size_t)p.E * p.R * (p.K / 2), cudaMemcpyDeviceToDevice, stream);
  if (e != cudaSuccess) return e;
  prepare_scales_kernel<<<1184, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

// bf16 weight tiles: one thread per 16-byte chunk of the output.  Chunk position
// `pos` of row r holds the row's chunk pos ^ (r % 8) (the 128-byte swizzle), so the
// eight threads of one tile row read the 128 source bytes of that row together.
__global__ void prepare_bf16_kernel(PrepareBf16Params p) {
  const long long ntiles = (long long)p.E * p.groups * p.mt * p.ks;
  const long long total = (ntiles + 1) * 1024;  // 16-byte chunks, the zero tile included
  for (long long q = (long long)blockIdx.x * blockDim.x + threadIdx.x; q < total;
       q += (long long)gridDim.x * blockDim.x) {
    const long long tile = q >> 10;
    const int r = (int)(q & 1023) >> 3, c = ((int)q & 7) ^ (r & 7);
    uint4 v = make_uint4(0, 0, 0, 0);
    if (tile < ntiles) {
      long long t = tile;
      const int s = (int)(t % p.ks);
      t /= p.ks;
      const int m = (int)(t % p.mt);
      t /= p.mt;
      const int g = (int)(t % p.groups);
      const int e = (int)(t / p.groups);
      const int row = m * kMTile + r;
      if (row < p.rows_per_group)
        v = __ldg(reinterpret_cast<const uint4*>(p.w + (((size_t)e * p.groups + g) * p.rows_per_group + row) * p.K +
                                                 (size_t)s * 64) + c);
    }
    reinterpret_cast<uint4*>(p.dst)[q] = v;
  }
}

cudaError_t launch_prepare_bf16(const PrepareBf16Params& p, cudaStream_t stream) {
  const long long total = ((long long)p.E * p.groups * p.mt * p.ks + 1) * 1024;
  const long long want = (total + kAuxThreads - 1) / kAuxThreads;
  const int blocks = (int)(want < 4096 ? want : 4096);
  prepare_bf16_kernel<<<blocks, kAuxThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

// out[a][i] = sum_t e2m1(q_t) * 2^(s_t - 127) for every valid tile row.
__global__ void hidden_dequant_kernel(HiddenDequantParams p) {
  const int num_tiles = __ldcg(p.num_tiles);
  const long long total = (long long)num_tiles * p.bm * p.I;
  const int natoms = act_sf_atoms(p.bm);
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const long long row = i / p.I;
    const int f = (int)(i - row * p.I);
    const int tile = (int)(row / p.bm);
    const int r = (int)(row - (long long)tile * p.bm);
    const TileEntry te = load_tile(p.tiles + tile);
    if (r >= te.n_rows) continue;
    const int a = __ldcg(p.perm + te.row_begin + r);
    float v = 0.f;
    for (int t = 0; t < kTerms; ++t) {
      const uint8_t byte = p.h_q[act_offset(tile, t, r, f & ~1, p.max_tiles, p.bm)];
      const uint32_t code = (f & 1) ? (byte >> 4) : (byte & 15u);
      const size_t off = ((size_t)tile * p.kg + (f >> 7)) * (kSfAtomBytes * natoms) +
                         sf_atom_offset(act_row(t, r, p.bm), (f >> 5) & 3);
      v += e2m1_to_f32(code) * pow2_int((int)p.sf[off] - 127);
    }
    p.out[(size_t)a * p.I + f] = v;
  }
}

cudaError_t launch_hidden_dequant(const HiddenDequantParams& p, cudaStream_t stream) {
  hidden_dequant_kernel<<<1184, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace moe
