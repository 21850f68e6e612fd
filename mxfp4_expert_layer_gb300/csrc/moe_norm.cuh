// RMSNorm + residual in front of the layer: the shared arithmetic of every kernel
// that normalises a row (internal to the library).
#pragma once

#include "moe_common.cuh"

namespace moe {

// The step before the router ("triton-kernels" README, "Kernels" row
// rmsnorm_residual_fused and "Quick Start", "Fused RMSNorm + Residual"): the residual
// stream s = bf16(x + r), then y = bf16(s / sqrt(mean(s^2) + eps) * gamma).  Several
// kernels normalise the same row (the router's and the encoder's), and the router
// and the experts must see the same y, so every kernel takes the sum of squares
// through the functions below: the row is cut into kNormSlices ranges of whole
// 16-value steps; within a range, lane l of a warp adds the squares of the 8-value
// vectors l, l + 32, ... in order (fused multiply-adds), the lanes combine by a
// butterfly, and the range sums are added in range order.  The rows may sit in
// global or shared memory (generic loads): the bits do not depend on where.

constexpr int kNormSlices = 8;

// First 8-value vector of range q of a row of H values (H a multiple of 16).
__host__ __device__ inline int norm_slice_vec(int H, int q) { return 2 * (q * (H / 16) / kNormSlices); }

__device__ __forceinline__ float bf16_round_f32(float v) {
  uint32_t u = __float_as_uint(v);
  u = (u + 0x7FFFu + ((u >> 16) & 1u)) & 0xFFFF0000u;  // nearest, ties to even (finite v)
  return __uint_as_float(u);
}

// s = bf16(x + r) of eight bf16 pairs.
__device__ __forceinline__ void residual_sum8(const uint4& xv, const uint4& rv, float (&s)[8]) {
  const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w}, rw[4] = {rv.x, rv.y, rv.z, rv.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    s[2 * i] = bf16_round_f32(__fadd_rn(__uint_as_float(xw[i] << 16), __uint_as_float(rw[i] << 16)));
    s[2 * i + 1] = bf16_round_f32(__fadd_rn(__uint_as_float(xw[i] & 0xFFFF0000u), __uint_as_float(rw[i] & 0xFFFF0000u)));
  }
}

__device__ __forceinline__ float ssq_accumulate(float acc, const uint4& xv, const uint4& rv) {
  float s[8];
  residual_sum8(xv, rv, s);
#pragma unroll
  for (int i = 0; i < 8; ++i) acc = __fmaf_rn(s[i], s[i], acc);
  return acc;
}

__device__ __forceinline__ float warp_sum_butterfly(float acc) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, o));
  return acc;
}

// Sum of s^2 over the vectors [v0, v1) of one row (one range), by one warp; every
// lane returns the same bits.
__device__ __forceinline__ float norm_range_ssq(const uint16_t* x_row, const uint16_t* r_row, int v0, int v1) {
  const int lane = threadIdx.x & 31;
  const uint4* xv = reinterpret_cast<const uint4*>(x_row);
  const uint4* rv = reinterpret_cast<const uint4*>(r_row);
  float acc = 0.f;
  for (int v = v0 + lane; v < v1; v += 32) acc = ssq_accumulate(acc, xv[v], rv[v]);
  return warp_sum_butterfly(acc);
}

// 1 / sqrt(mean + eps) from the range sums, added in range order.
__device__ __forceinline__ float norm_rinv(const float (&part)[kNormSlices], int H, float eps) {
  float tot = 0.f;
#pragma unroll
  for (int q = 0; q < kNormSlices; ++q) tot = __fadd_rn(tot, part[q]);
  return rsqrtf(__fadd_rn(__fdiv_rn(tot, (float)H), eps));
}

// The whole row's 1 / rms, by one warp: the kNormSlices ranges of norm_range_ssq
// advanced together (the loads of all ranges in flight at once), each range's lane
// sum in the same order as there.
__device__ __forceinline__ float norm_row_rinv(const uint16_t* x_row, const uint16_t* r_row, int H, float eps) {
  const int lane = threadIdx.x & 31;
  const uint4* xv = reinterpret_cast<const uint4*>(x_row);
  const uint4* rv = reinterpret_cast<const uint4*>(r_row);
  float acc[kNormSlices];
  int nmax = 0;
#pragma unroll
  for (int q = 0; q < kNormSlices; ++q) {
    acc[q] = 0.f;
    nmax = max(nmax, norm_slice_vec(H, q + 1) - norm_slice_vec(H, q));
  }
  for (int base = 0; base < nmax; base += 32) {
    uint4 xa[kNormSlices], ra[kNormSlices];
#pragma unroll
    for (int q = 0; q < kNormSlices; ++q) {
      const int v = norm_slice_vec(H, q) + base + lane;
      if (v < norm_slice_vec(H, q + 1)) {
        xa[q] = xv[v];
        ra[q] = rv[v];
      }
    }
#pragma unroll
    for (int q = 0; q < kNormSlices; ++q)
      if (norm_slice_vec(H, q) + base + lane < norm_slice_vec(H, q + 1)) acc[q] = ssq_accumulate(acc[q], xa[q], ra[q]);
  }
#pragma unroll
  for (int q = 0; q < kNormSlices; ++q) acc[q] = warp_sum_butterfly(acc[q]);
  return norm_rinv(acc, H, eps);
}

// y of eight values: bf16(s * rinv * gamma), packed as bf16 pairs.
__device__ __forceinline__ uint4 norm_apply8(const uint4& xv, const uint4& rv, const uint4& gv, float rinv) {
  float s[8];
  residual_sum8(xv, rv, s);
  const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float lo = bf16_round_f32(__fmul_rn(__fmul_rn(s[2 * i], rinv), __uint_as_float(gw[i] << 16)));
    const float hi = bf16_round_f32(__fmul_rn(__fmul_rn(s[2 * i + 1], rinv), __uint_as_float(gw[i] & 0xFFFF0000u)));
    o[i] = (__float_as_uint(lo) >> 16) | (__float_as_uint(hi) & 0xFFFF0000u);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

}  // namespace moe
