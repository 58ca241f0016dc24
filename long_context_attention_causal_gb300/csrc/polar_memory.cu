// In-place gated-delta memory step: the producer of the memory stream.
//
// "ATMA: Length-Invariant Language Modeling via Polar Attention and
// Gated-Delta Compression Memory", §2.1 item 3 (a gated-delta memory whose
// keys and queries are L2-normalised, which bounds the eigenvalues of the
// update) and §2.2 (an in-place step kernel).  Per head and token:
//   k^ = k / max(|k|, eps),  q^ = q / max(|q|, eps)
//   S <- alpha S (I - beta k^ k^T) + beta v k^T
//     = alpha S + (beta v - alpha beta (S k^)) k^T      (row form used here)
//   mem = S q^
// S is d x d fp32 (row i = value dimension i), updated in place in HBM: one
// read and one write of the state per call, whatever T.
//
// One CTA per (b, h), 8 warps; warp w keeps rows [w*d/8, (w+1)*d/8) of S in
// registers for all T tokens (lane c holds columns 4c..4c+3 at d = 128), so
// the row loads and stores are coalesced 512-byte rows.  Each row needs two
// dot products per token (S_i . k^ and S_new_i . q^), reduced with xor
// shuffles; the token's k^ and q^ are recomputed by every warp (cheap).
#include "polar_device.cuh"
#include "polar_internal.h"

namespace polar {

namespace {

constexpr int kMemWarps = 8;

template <typename T>
__device__ __forceinline__ float load_elem(const T* p);
template <>
__device__ __forceinline__ float load_elem<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float load_elem<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}
template <typename T>
__device__ __forceinline__ T store_cast(float x);
template <>
__device__ __forceinline__ float store_cast<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 store_cast<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Two CTAs per SM (registers capped at 128, no spills): one CTA's loads
// then overlap the other's update and stores; at one CTA per SM (162
// registers uncapped) the step ran at 4.3 TB/s instead of 6.2.
template <int D, typename T>
__global__ void __launch_bounds__(kMemWarps * 32, 2)
    polar_memory_step_kernel(float* __restrict__ state, const T* __restrict__ q,
                             const T* __restrict__ k, const T* __restrict__ v,
                             const float* __restrict__ alpha, const float* __restrict__ beta,
                             T* __restrict__ mem, int Tn, float eps) {
  constexpr int RPW = D / kMemWarps;  // rows per warp
  constexpr int CPL = D / 32;         // columns per lane
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t bh = blockIdx.x;
  float* S = state + bh * D * D;
  const int row0 = warp * RPW;

  float s[RPW][CPL];
#pragma unroll
  for (int r = 0; r < RPW; ++r) {
    const float* src = S + (size_t)(row0 + r) * D + lane * CPL;
    if (CPL == 4) {
      const float4 x = *reinterpret_cast<const float4*>(src);
      s[r][0] = x.x;
      s[r][1] = x.y;
      s[r][2 % CPL] = x.z;
      s[r][3 % CPL] = x.w;
    } else {
      const float2 x = *reinterpret_cast<const float2*>(src);
      s[r][0] = x.x;
      s[r][1 % CPL] = x.y;
    }
  }

  for (int t = 0; t < Tn; ++t) {
    const size_t tok = bh * Tn + t;
    const T* kt = k + tok * D + lane * CPL;
    const T* qt = q + tok * D + lane * CPL;
    float kh[CPL], qh[CPL];
    float kk = 0.f, qq = 0.f;
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      kh[c] = load_elem<T>(kt + c);
      qh[c] = load_elem<T>(qt + c);
      kk = fmaf(kh[c], kh[c], kk);
      qq = fmaf(qh[c], qh[c], qq);
    }
    const float kinv = 1.0f / fmaxf(sqrtf(warp_sum(kk)), eps);
    const float qinv = 1.0f / fmaxf(sqrtf(warp_sum(qq)), eps);
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      kh[c] *= kinv;
      qh[c] *= qinv;
    }
    const float a = alpha[tok], b = beta[tok];
    // v for this warp's rows, one row per lane, broadcast below
    const float vl = lane < RPW ? load_elem<T>(v + tok * D + row0 + lane) : 0.f;
    float my_out = 0.f;
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
      float u = 0.f;
#pragma unroll
      for (int c = 0; c < CPL; ++c) u = fmaf(s[r][c], kh[c], u);
      u = warp_sum(u);  // (S k^)_i
      const float vi = __shfl_sync(0xffffffffu, vl, r);
      const float coef = b * vi - a * b * u;
      float o = 0.f;
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        s[r][c] = fmaf(a, s[r][c], coef * kh[c]);
        o = fmaf(s[r][c], qh[c], o);
      }
      o = warp_sum(o);  // (S_new q^)_i
      if (lane == r) my_out = o;
    }
    if (lane < RPW) mem[tok * D + row0 + lane] = store_cast<T>(my_out);
  }

#pragma unroll
  for (int r = 0; r < RPW; ++r) {
    float* dst = S + (size_t)(row0 + r) * D + lane * CPL;
    if (CPL == 4) {
      *reinterpret_cast<float4*>(dst) = make_float4(s[r][0], s[r][1], s[r][2 % CPL], s[r][3 % CPL]);
    } else {
      *reinterpret_cast<float2*>(dst) = make_float2(s[r][0], s[r][1 % CPL]);
    }
  }
}

template <int D, typename T>
cudaError_t launch_d(const MemoryArgs& a, cudaStream_t s) {
  polar_memory_step_kernel<D, T><<<a.B * a.H, kMemWarps * 32, 0, s>>>(
      a.state, static_cast<const T*>(a.q), static_cast<const T*>(a.k),
      static_cast<const T*>(a.v), a.alpha, a.beta, static_cast<T*>(a.mem), a.T, a.eps);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_memory_step(const MemoryArgs& a, int dtype, cudaStream_t s) {
  if (dtype == POLAR_BF16)
    return a.d == 64 ? launch_d<64, __nv_bfloat16>(a, s) : launch_d<128, __nv_bfloat16>(a, s);
  return a.d == 64 ? launch_d<64, float>(a, s) : launch_d<128, float>(a, s);
}

}  // namespace polar
