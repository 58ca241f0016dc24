// Causal Polar Attention prefill, fp32, on the FP32 pipes.
//
// "ATMA: Length-Invariant Language Modeling via Polar Attention and
// Gated-Delta Compression Memory", §2.1 (three output channels) and §2.2
// (online participation ratio with streaming accumulators and squared
// correction factors).  fp32 inputs rule out the bf16 tensor-core path, so
// this kernel keeps everything in fp32 with accurate expf/logf:
//
//   * a CTA of 8 warps owns 8 consecutive query rows of one (b, h), one warp
//     per row; key/value tiles (64 keys at d = 64, 32 at d = 128) are staged
//     in shared memory (K rows padded to d+4 floats so lane-per-key float4
//     reads are conflict-free), the next tile read into registers while the
//     current one is used;
//   * lane j scores keys j, j + 32, ... of the tile (full dot products from
//     shared memory), warp-shuffle reductions give the tile max, l and Q2
//     updates; each lane owns d/32 output columns of the value accumulator;
//   * the epilogue reduces |acc|^2 with shuffles and writes coalesced rows.
#include "polar_device.cuh"
#include "polar_internal.h"

namespace polar {

namespace {

constexpr int kRows = 8;   // rows (warps) per CTA

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}
__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

template <int D>
__global__ void __launch_bounds__(kRows * 32)
    polar_fwd_f32_kernel(const float* __restrict__ q, const float* __restrict__ k,
                         const float* __restrict__ v, const float* __restrict__ mem,
                         const float* __restrict__ w_count, float* __restrict__ out,
                         float* __restrict__ n_eff, float* __restrict__ conf, int H,
                         int T, int row_blocks, polar_consts_t c) {
  // K rows padded to D + 4 floats: lane j reads its key's row as float4s,
  // and the eight lanes of each quarter-warp phase then hit 32 distinct
  // banks
  // keys per tile: 64 at d = 64 (two per lane), 32 at d = 128 (the
  // static shared-memory limit), so the barriers and reductions of a tile
  // are paid once per 64 keys where they fit
  constexpr int KPL = D == 64 ? 2 : 1;
  constexpr int kKT = 32 * KPL;
  __shared__ __align__(16) float ks[kKT][D + 4];
  __shared__ __align__(16) float vs[kKT][D];
  __shared__ __align__(16) float qs[kRows][D];
  __shared__ __align__(16) float ps[kRows][kKT];  // a warp's p of the tile

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // heaviest row blocks first
  const int rb = row_blocks - 1 - (int)(blockIdx.x % row_blocks);
  const int bh = (int)(blockIdx.x / row_blocks);
  const int h = bh % H;
  const int row0 = rb * kRows;
  const int row = row0 + warp;
  const bool valid = row < T;
  const size_t base = (size_t)bh * T * D;

  for (int x = lane; x < D; x += 32) qs[warp][x] = valid ? q[base + (size_t)row * D + x] : 0.f;

  const float n = (float)(row + 1);
  const float tau = polar_tau(n, c.log_t0);
  const float scale = tau * rsqrtf((float)D);
  float m = -INFINITY, l = 0.f, q2 = 0.f;
  float acc[D / 32];
#pragma unroll
  for (int x = 0; x < D / 32; ++x) acc[x] = 0.f;

  const int last_row = min(row0 + kRows, T) - 1;
  // The next key tile is read into registers while the current one is
  // used, so a tile's global-memory latency overlaps the previous tile's
  // arithmetic (one tile at a time left the kernel waiting on each load).
  constexpr int kPer = kKT * D / (kRows * 32);  // elements of K (and V) per thread per tile
  float kr[kPer], vr[kPer];
  auto fetch = [&](int j0) {
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int e = threadIdx.x + i * kRows * 32;
      const int key = j0 + e / D;
      const bool in = key < T;
      kr[i] = in ? k[base + (size_t)key * D + e % D] : 0.f;
      vr[i] = in ? v[base + (size_t)key * D + e % D] : 0.f;
    }
  };
  fetch(0);
  for (int j0 = 0; j0 <= last_row; j0 += kKT) {
    __syncthreads();  // the previous tile's reads of ks / vs are done
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int e = threadIdx.x + i * kRows * 32;
      ks[e / D][e % D] = kr[i];
      vs[e / D][e % D] = vr[i];
    }
    __syncthreads();
    if (j0 + kKT <= last_row) fetch(j0 + kKT);
    if (!valid || j0 > row) continue;
    // lane j scores keys j0 + j + 32 i (i < KPL): four partial dot
    // products each, both rows read as float4s (q broadcast to the warp)
    const float4* qq = reinterpret_cast<const float4*>(&qs[warp][0]);
    float sk[KPL];
#pragma unroll
    for (int i = 0; i < KPL; ++i) {
      float s4[4] = {0.f, 0.f, 0.f, 0.f};
      const float4* kq = reinterpret_cast<const float4*>(&ks[lane + 32 * i][0]);
#pragma unroll 8
      for (int x4 = 0; x4 < D / 4; ++x4) {
        const float4 kv = kq[x4], qv = qq[x4];
        s4[0] = fmaf(qv.x, kv.x, s4[0]);
        s4[1] = fmaf(qv.y, kv.y, s4[1]);
        s4[2] = fmaf(qv.z, kv.z, s4[2]);
        s4[3] = fmaf(qv.w, kv.w, s4[3]);
      }
      const float sv = (s4[0] + s4[1]) + (s4[2] + s4[3]);
      sk[i] = j0 + lane + 32 * i <= row ? sv * scale : -INFINITY;
    }
    float smax = sk[0];
#pragma unroll
    for (int i = 1; i < KPL; ++i) smax = fmaxf(smax, sk[i]);
    const float mt = warp_max(smax);
    const float mn = fmaxf(m, mt);
    const float alpha = expf(m - mn);  // 0 while m = -inf
    float pk[KPL], psum = 0.f, psq = 0.f;
#pragma unroll
    for (int i = 0; i < KPL; ++i) {
      pk[i] = j0 + lane + 32 * i <= row ? expf(sk[i] - mn) : 0.f;
      psum += pk[i];
      psq = fmaf(pk[i], pk[i], psq);
    }
    l = l * alpha + warp_sum(psum);
    q2 = q2 * alpha * alpha + warp_sum(psq);  // squared correction factor
#pragma unroll
    for (int x = 0; x < D / 32; ++x) acc[x] *= alpha;
    // every key of the tile (p = 0 past the row, and V rows past T are
    // zero): a fixed trip count the compiler can unroll and overlap; the
    // tile's p go through shared memory once and come back four at a time
    // (broadcast float4 reads instead of one shuffle per key)
#pragma unroll
    for (int i = 0; i < KPL; ++i) ps[warp][lane + 32 * i] = pk[i];
    __syncwarp();
    const float4* p4 = reinterpret_cast<const float4*>(&ps[warp][0]);
#pragma unroll 2
    for (int j4 = 0; j4 < kKT / 4; ++j4) {
      const float4 pv = p4[j4];
      const float pw[4] = {pv.x, pv.y, pv.z, pv.w};
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int x = 0; x < D / 32; ++x)
          acc[x] = fmaf(pw[u], vs[4 * j4 + u][lane + 32 * x], acc[x]);
    }
    __syncwarp();  // ps is rewritten by the next tile
    m = mn;
  }
  if (!valid) return;
  float asq = 0.f, qsq = 0.f;
#pragma unroll
  for (int x = 0; x < D / 32; ++x) {
    asq = fmaf(acc[x], acc[x], asq);
    const float qv = qs[warp][lane + 32 * x];
    qsq = fmaf(qv, qv, qsq);
  }
  asq = warp_sum(asq);
  qsq = warp_sum(qsq);
  const RowResult res = polar_finish(m, l, q2, asq, qsq, n, D, c);
  const size_t ro = base + (size_t)row * D;
#pragma unroll
  for (int x = 0; x < D / 32; ++x) {
    const int col = lane + 32 * x;
    out[ro + col] = fmaf(acc[x], res.scale_u, fmaf(res.count, w_count[h * D + col], mem[ro + col]));
  }
  if (lane == 0) {
    n_eff[(size_t)bh * T + row] = res.n_eff;
    if (conf) conf[(size_t)bh * T + row] = res.conf;
  }
}

template <int D>
cudaError_t launch_d(const FwdArgs& a, cudaStream_t s) {
  const int row_blocks = (a.T + kRows - 1) / kRows;
  const long long blocks = (long long)row_blocks * a.B * a.H;
  polar_fwd_f32_kernel<D><<<(unsigned)blocks, kRows * 32, 0, s>>>(
      static_cast<const float*>(a.q), static_cast<const float*>(a.k),
      static_cast<const float*>(a.v), static_cast<const float*>(a.mem), a.w_count,
      static_cast<float*>(a.out), a.n_eff, a.conf, a.H, a.T, row_blocks, a.c);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_f32(const FwdArgs& a, cudaStream_t s) {
  if (a.d == 64) return launch_d<64>(a, s);
  return launch_d<128>(a, s);
}

}  // namespace polar
