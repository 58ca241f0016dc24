// Row records shared by the tensor-core backward kernels.
//
// "ATMA: Length-Invariant Language Modeling via Polar Attention and
// Gated-Delta Compression Memory", §2.1 gives the forward; its gradient per
// query row i reduces to a handful of scalars (derivation in
// polar_backward.cu).  The forward kernel run in backward mode writes them,
// seven per row, already in the form the tile kernels consume:
//   p_ij            = exp2(S_ij * cl2 + nlse2)          S_ij = q_i . k_j
//   coef * ds_ij    = p_ij * (coef * dP_ij + cmdc + ec * p_ij)
//   dq_i           += qfloor * q_i                       (null-floor term)
//   dw[h]          += count * g_i
#pragma once

#include <cuda_runtime.h>

namespace polar {

enum GradRow {
  kGCl2 = 0,   // tau / sqrt(d) * log2(e)
  kGNLse2,     // -lse * log2(e)
  kGCoef,      // tau / sqrt(d)
  kGCmDc,      // coef * (C - D)
  kGEc,        // coef * E
  kGQFloor,    // -dlse * (sigma / |q|) * f(n) / |q|
  kGCount,     // count of the row
};

// Layout: per (b, h) the rows are padded to whole 128-row tiles (tpad) and
// stored in pairs: rows 2i and 2i + 1 share a block of kGPairFloats floats
// in which each field holds the two rows side by side, so a kernel that
// works on two consecutive rows at once loads ready packed pairs.  Blocks
// are 80 bytes (14 floats used): four consecutive blocks then start in four
// different shared-memory bank groups.
constexpr int kGPairFloats = 20;
__host__ __device__ __forceinline__ int grad_rows_tpad(int T) { return (T + 127) / 128 * 128; }
__host__ __device__ __forceinline__ size_t grad_row_index(size_t bh, int tpad, int row,
                                                          int field) {
  return (bh * (size_t)(tpad / 2) + (size_t)(row >> 1)) * kGPairFloats + 2 * field + (row & 1);
}
__host__ __device__ __forceinline__ size_t grad_rows_floats(size_t BH, int T) {
  return BH * (size_t)(grad_rows_tpad(T) / 2) * kGPairFloats;
}

// Expected-maximum factor f(n) of the null floor b = sigma f(n): leading
// order sqrt(2 ln n), or the second-order Gumbel form (0 at n = 1).
__device__ __forceinline__ float polar_floor_factor(float n, int order) {
  const float r = sqrtf(2.0f * logf(n));
  if (order != 2) return r;
  if (n < 2.0f) return 0.0f;
  constexpr float kLn4Pi = 2.5310242469692907f;
  constexpr float kEulerGamma = 0.5772156649015329f;
  return r - (logf(logf(n)) + kLn4Pi) / (2.0f * r) + kEulerGamma / r;
}

}  // namespace polar
