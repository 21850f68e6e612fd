// Data movement kernels around the expert GEMMs:
//  * quant_x: the permute step -- activation rows gathered into tile order and
//    encoded as two E4M3 terms with E8M0 block scales (the tensor-core B operand);
//  * prepare: one-time re-layout of raw MXFP4 expert weights ("MXFP4 MoE on tensor
//    cores": weights permuted once at load; nothing is re-quantised);
//  * hidden_dequant: expands the encoded SwiGLU output for inspection.
#include "moe_common.cuh"
#include "moe_kernels.cuh"

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

// One warp per padded tile row: gather x[token] and encode each 32-value block as
// two E4M3 terms.  Each lane owns 8 consecutive values (one 16-byte load), so four
// lanes form a block and a warp covers 256 values per step.
__global__ void __launch_bounds__(kAuxThreads) quant_x_kernel(QuantXParams p) {
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * kAuxThreads + threadIdx.x) >> 5;
  // clear the combine arrival counters of the down kernel (grid-stride)
  if (p.zero_buf) {
    for (int i = blockIdx.x * kAuxThreads + threadIdx.x; i < p.zero_count; i += gridDim.x * kAuxThreads)
      p.zero_buf[i] = 0;
  }
  const int num_tiles = __ldg(p.num_tiles);
  const int row = gw;
  const int tile = row / p.bm;
  if (tile >= num_tiles) return;
  const int r = row - tile * p.bm;
  const TileEntry te = p.tiles[tile];
  if (r >= te.n_rows) return;
  const int a = __ldg(p.perm + te.row_begin + r);
  const int t = a / p.k;
  const uint4* xr = reinterpret_cast<const uint4*>(p.x + (size_t)t * p.H);
  uint2* qh = reinterpret_cast<uint2*>(p.q_hi + (size_t)row * p.H);
  uint2* ql = reinterpret_cast<uint2*>(p.q_lo + (size_t)row * p.H);
  const int nb = sf_atoms_per_tile(p.bm);
  uint8_t* sfh = p.sf_hi + (size_t)tile * p.kg * (kSfAtomBytes * nb);
  uint8_t* sfl = p.sf_lo + (size_t)tile * p.kg * (kSfAtomBytes * nb);
  const int nvec = p.H / 8;
  for (int v0 = 0; v0 < nvec; v0 += 32) {
    const int v = v0 + lane;
    const bool valid = v < nvec;
    float f[8];
    if (valid) {
      const uint4 raw = __ldg(xr + v);
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
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
    amax = quad_max(amax);
    const int p1 = mx_e4m3_exponent(amax);
    const float inv1 = pow2_int(-p1), sc1 = pow2_int(p1);
    uint8_t q1[8];
    float res[8], amax2 = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      q1[i] = f32_to_e4m3(f[i] * inv1);
      res[i] = f[i] - e4m3_to_f32(q1[i]) * sc1;
      amax2 = fmaxf(amax2, fabsf(res[i]));
    }
    amax2 = quad_max(amax2);
    const int p2 = mx_e4m3_exponent(amax2);
    const float inv2 = pow2_int(-p2);
    uint8_t q2[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) q2[i] = f32_to_e4m3(res[i] * inv2);
    if (valid) {
      uint2 h, l;
      h.x = q1[0] | (q1[1] << 8) | (q1[2] << 16) | ((uint32_t)q1[3] << 24);
      h.y = q1[4] | (q1[5] << 8) | (q1[6] << 16) | ((uint32_t)q1[7] << 24);
      l.x = q2[0] | (q2[1] << 8) | (q2[2] << 16) | ((uint32_t)q2[3] << 24);
      l.y = q2[4] | (q2[5] << 8) | (q2[6] << 16) | ((uint32_t)q2[7] << 24);
      qh[v] = h;
      ql[v] = l;
      if ((lane & 3) == 0) {
        const int b = v >> 2;  // MX block index along H
        const size_t off = (size_t)(b >> 2) * (kSfAtomBytes * nb) + sf_atom_offset(r, b & 3);
        sfh[off] = static_cast<uint8_t>(p1 + 127);
        sfl[off] = static_cast<uint8_t>(p2 + 127);
      }
    }
  }
}

cudaError_t launch_quant_x(const QuantXParams& p, cudaStream_t stream) {
  const long long rows = (long long)p.max_tiles * p.bm;
  const int blocks = (int)((rows * 32 + kAuxThreads - 1) / kAuxThreads);
  quant_x_kernel<<<blocks, kAuxThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

// Codes: each row copied in 16-byte vectors, zero-padded from K/2 to Kp/2 bytes.
__global__ void prepare_codes_kernel(PrepareParams p) {
  const int src_vec = p.K / 32;   // 16-byte vectors per source row (K/2 bytes)
  const int dst_vec = p.Kp / 32;
  const long long total = (long long)p.E * p.R * dst_vec;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const long long row = i / dst_vec;
    const int v = (int)(i - row * dst_vec);
    uint4 val = make_uint4(0, 0, 0, 0);
    if (v < src_vec) val = __ldg(reinterpret_cast<const uint4*>(p.codes + row * (p.K / 2)) + v);
    reinterpret_cast<uint4*>(p.dst_codes + row * (p.Kp / 2))[v] = val;
  }
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
  prepare_codes_kernel<<<1184, 256, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  prepare_scales_kernel<<<1184, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

// out[a][i] = q_hi * 2^(s_hi - 127) + q_lo * 2^(s_lo - 127) for every tile row.
__global__ void hidden_dequant_kernel(HiddenDequantParams p) {
  const int num_tiles = __ldg(p.num_tiles);
  const long long total = (long long)num_tiles * p.bm * p.I;
  const int nb = sf_atoms_per_tile(p.bm);
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const long long row = i / p.I;
    const int f = (int)(i - row * p.I);
    const int tile = (int)(row / p.bm);
    const int r = (int)(row - (long long)tile * p.bm);
    const TileEntry te = p.tiles[tile];
    if (r >= te.n_rows) continue;
    const int a = p.perm[te.row_begin + r];
    const size_t off = ((size_t)tile * p.kg + (f >> 7)) * (kSfAtomBytes * nb) + sf_atom_offset(r, (f >> 5) & 3);
    const float v = e4m3_to_f32(p.h_hi[row * p.I + f]) * pow2_int((int)p.sf_hi[off] - 127) +
                    e4m3_to_f32(p.h_lo[row * p.I + f]) * pow2_int((int)p.sf_lo[off] - 127);
    p.out[(size_t)a * p.I + f] = v;
  }
}

cudaError_t launch_hidden_dequant(const HiddenDequantParams& p, cudaStream_t stream) {
  hidden_dequant_kernel<<<1184, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace moe
