// Backward of causal Polar Attention, bf16, on the sm_103a tensor cores.
//
// "ATMA: Length-Invariant Language Modeling via Polar Attention and
// Gated-Delta Compression Memory" trains its model (§3), so the fused kernel
// of §2.2 needs gradients; they follow from the forward of §2.1 and reduce,
// per query row, to the record of polar_grad.cuh (written by the forward
// kernel in backward mode together with dA = dL/da in bf16).  What is left
// is attention-shaped:
//   p_ij  = exp(s_ij - lse_i),  dP_ij = dA_i . v_j,
//   dS'_ij = coef_i ds_ij = p_ij (coef_i dP_ij + cmdc_i + ec_i p_ij)
//   dV_j = sum_i p_ij dA_i,  dK_j = sum_i dS'_ij q_i,
//   dQ_i = sum_j dS'_ij k_j + qfloor_i q_i.
//
// Two kernels, one CTA per SM each (512 TMEM columns):
//   * dK/dV: a CTA owns a 128-key tile of one (b, h), keeps K and V in
//     shared memory and streams the 64-query halves at or after it (Q, dA
//     and the row records, TMA into a ring of half-tile stages, so a stage
//     is refilled as soon as its own MMAs are done).  Consecutive halves
//     alternate between two TMEM buffers:
//       S^T = K Q_h^T, dP^T = V dA_h^T      (SS, M = 128 keys, N = 64)
//       P^T, dS'^T (bf16) written over them by softmax warpgroup h
//       dV += P^T dA_h, dK += dS'^T Q_h       (TS: A from TMEM, K = 64)
//     so one warpgroup's elementwise work overlaps the other half's MMAs.
//   * dQ: a CTA owns a 128-query tile, keeps Q and dA, streams the causal
//     64-key halves (K and V ring):
//       S = Q K_h^T, dP = dA V_h^T;  dS' over dP;  dQ += dS' K_h.
// Roles (384 threads): warps 0-3 and 4-7 the two elementwise warpgroups
// (thread = TMEM lane = key or query row of the tile), warp 8 TMA, warp 9
// MMA issuer and TMEM owner.  Every wait is bounded (status 1 on timeout).
// TMEM columns: S buffers 0-63 / 64-127, dP buffers 128-191 / 192-255,
// accumulators from 256 (dV then dK, or dQ).
#include "polar_device.cuh"
#include "polar_grad.cuh"
#include "polar_internal.h"

namespace polar {

namespace {

constexpr int kTile = 128;  // keys or queries per resident tile
constexpr int kHalf = 64;   // keys or queries per streamed stage / MMA step
constexpr int kNSMax = 8;
constexpr int kThreads = 384;
constexpr int kWarpTMA = 8;
constexpr int kWarpMMA = 9;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColDP = 128, kColAcc = 256;

template <int D>
struct Layout {
  // resident tiles: 128 rows, two 64-column swizzle atoms of 16 KB at D = 128
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kAtom = kTile * 128;
  // streamed halves: 64 rows, atoms of 8 KB
  static constexpr int kHalfBytes = kHalf * D * 2;
  static constexpr int kHalfAtom = kHalf * 128;
  static constexpr int kRecBytes = kHalf * kGRowFloats * 4;
  static constexpr int kNS = D == 128 ? 4 : 8;  // ring stages
  static constexpr int kR0 = 0;
  static constexpr int kR1 = kR0 + kTileBytes;
  static constexpr int kRing = kR1 + kTileBytes;
  static constexpr int kStageBytes = 2 * kHalfBytes + kRecBytes;
  static constexpr int kBarOff = kRing + kNS * kStageBytes;
  // padded above half of the SM's shared memory: one CTA per SM, so the
  // 512 TMEM columns it allocates are never contended
  static constexpr int kNeed = kBarOff + 256 + 1024;
  static constexpr int kSmemBytes = kNeed > 232448 / 2 + 1024 ? kNeed : 232448 / 2 + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory");
  static_assert(kNS <= kNSMax, "ring");
};

struct Bars {
  uint64_t res_full;             // resident tiles landed
  uint64_t full[kNSMax], empty[kNSMax];
  uint64_t s_full[2], p_full[2];
  uint64_t acc_full;
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

struct BwdTcParams {
  const __nv_bfloat16* q;  // for the floor term of dQ
  const float* rows;       // [BH, tpad, kGRowFloats], pair-interleaved
  float *dq, *dk, *dv;     // [BH, T, D] fp32
  int* status;
  int T, BH, n_t, tpad;
};

// K-major descriptor offset of K step kk (16 elements) in a tile whose
// 64-column swizzle atoms are kAtomBytes apart.
template <int kAtomBytes>
__device__ __forceinline__ uint64_t kstep(int kk) {
  return (uint64_t)((kk >> 2) * (kAtomBytes >> 4) + (kk & 3) * 2);
}

__device__ __forceinline__ void setup_barriers(Bars* bars, int ns) {
  mbar_init(&bars->res_full, 1);
  for (int s = 0; s < ns; ++s) {
    mbar_init(&bars->full[s], 1);
    mbar_init(&bars->empty[s], 1);
  }
  for (int b = 0; b < 2; ++b) {
    mbar_init(&bars->s_full[b], 1);
    mbar_init(&bars->p_full[b], 128);
  }
  mbar_init(&bars->acc_full, 1);
  mbar_init(&bars->drain, 1);
  bars->abort_flag = 0;
  fence_barrier_init();
}

// Elementwise work on one 32-column chunk of a TMEM buffer, two columns at
// a time with packed fp32 pairs:
//   p = exp2(S cl2 + nlse2),  dS' = p (coef dP + cmdc + ec p)
// kMasked: entries outside the causal triangle or past T are selected to 0
// (p and dS'; the records of rows past T are not initialised).  The mask is
// a template parameter so that the unrolled loop has no branch: each chunk
// is one basic block, and its 16 independent pairs overlap.

// dK/dV kernel: columns are queries; their scalars come from the pair
// blocks of the row records in shared memory (rec points at column 0).
template <bool kMasked>
__device__ __forceinline__ void dkdv_chunk(const uint32_t (&sv)[32], const uint32_t (&dv)[32],
                                           const float* rec, int key, int q_first, int T,
                                           uint32_t (&pk)[16], uint32_t (&dsk)[16]) {
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    const float4 r0 = *reinterpret_cast<const float4*>(rec + 16 * e);      // cl2, nlse2
    const float4 r1 = *reinterpret_cast<const float4*>(rec + 16 * e + 4);  // coef, cmdc
    const float2 ec = *reinterpret_cast<const float2*>(rec + 16 * e + 8);
    const float2 x = ffma2(make_float2(__uint_as_float(sv[2 * e]), __uint_as_float(sv[2 * e + 1])),
                           make_float2(r0.x, r0.y), make_float2(r0.z, r0.w));
    float2 pp = make_float2(ex2_approx(x.x), ex2_approx(x.y));
    const float2 t = ffma2(make_float2(__uint_as_float(dv[2 * e]), __uint_as_float(dv[2 * e + 1])),
                           make_float2(r1.x, r1.y), make_float2(r1.z, r1.w));
    bool v0 = true, v1 = true;
    if (kMasked) {
      const int qa = q_first + 2 * e;
      v0 = key <= qa && qa < T;
      v1 = key <= qa + 1 && qa + 1 < T;
      pp.x = v0 ? pp.x : 0.f;
      pp.y = v1 ? pp.y : 0.f;
    }
    const float2 u = ffma2(ec, pp, t);
    float2 ds = ffma2(pp, u, make_float2(0.f, 0.f));
    if (kMasked) {
      ds.x = v0 ? ds.x : 0.f;
      ds.y = v1 ? ds.y : 0.f;
    }
    pk[e] = pack_bf16x2(pp.x, pp.y);
    dsk[e] = pack_bf16x2(ds.x, ds.y);
  }
}

// dQ kernel: the row's scalars are the same for every column (packed pairs
// in registers); masked chunks are those of the diagonal tile.
template <bool kMasked>
__device__ __forceinline__ void dq_chunk(const uint32_t (&sv)[32], const uint32_t (&dv)[32],
                                         float2 cl2, float2 nlse2, float2 coef, float2 cmdc,
                                         float2 ec, int row, int k_first,
                                         uint32_t (&dsk)[16]) {
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    const float2 x = ffma2(make_float2(__uint_as_float(sv[2 * e]), __uint_as_float(sv[2 * e + 1])),
                           cl2, nlse2);
    float2 pp = make_float2(ex2_approx(x.x), ex2_approx(x.y));
    const float2 t = ffma2(make_float2(__uint_as_float(dv[2 * e]), __uint_as_float(dv[2 * e + 1])),
                           coef, cmdc);
    if (kMasked) {
      const int ka = k_first + 2 * e;
      pp.x = ka <= row ? pp.x : 0.f;
      pp.y = ka + 1 <= row ? pp.y : 0.f;
    }
    const float2 u = ffma2(ec, pp, t);
    const float2 ds = ffma2(pp, u, make_float2(0.f, 0.f));
    dsk[e] = pack_bf16x2(ds.x, ds.y);
  }
}

// Maps: 128-row boxes for the resident tiles, 64-row boxes for the stream.
struct TileMaps {
  CUtensorMap q, k, v, da;          // box 64 x 128
  CUtensorMap q64, k64, v64, da64;  // box 64 x 64
};

// ============================================================ dK and dV ==
// Step j = one 64-query half (queries 128 kt + 64 j ...), ring stage j % NS,
// TMEM buffer / elementwise warpgroup j & 1.
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    polar_bwd_dkdv_kernel(const __grid_constant__ TileMaps m, const BwdTcParams p) {
  using L = Layout<D>;
  constexpr int kNS = L::kNS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + L::kBarOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // heaviest key tiles (most queries after them) first
  const int kt = (int)(blockIdx.x / p.BH);
  const int bh = (int)(blockIdx.x % p.BH);
  const int nsteps = (p.T + kHalf - 1) / kHalf - 2 * kt;  // halves with a query < T

  if (threadIdx.x == 0) setup_barriers(bars, kNS);
  if (warp == kWarpMMA) tmem_alloc(&bars->tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  volatile int* abort_flag = &bars->abort_flag;
  auto stage_q = [&](int s) { return smem + L::kRing + s * L::kStageBytes; };
  auto stage_da = [&](int s) { return stage_q(s) + L::kHalfBytes; };
  auto stage_rec = [&](int s) {
    return reinterpret_cast<const float*>(stage_q(s) + 2 * L::kHalfBytes);
  };

  if (warp == kWarpTMA) {
    if (lane == 0) {
      tma_prefetch_desc(&m.q64);
      tma_prefetch_desc(&m.da64);
      mbar_arrive_expect_tx(&bars->res_full, 2 * L::kTileBytes);
      for (int a = 0; a < D / 64; ++a) {
        tma_load_3d(smem + L::kR0 + a * L::kAtom, &m.k, &bars->res_full, 64 * a, kTile * kt, bh);
        tma_load_3d(smem + L::kR1 + a * L::kAtom, &m.v, &bars->res_full, 64 * a, kTile * kt, bh);
      }
      bool ok = true;
      int issued = 0;
      for (int j = 0; j < nsteps && ok; ++j) {
        const int s = j % kNS, q0 = kTile * kt + kHalf * j;
        if (j >= kNS) ok = mbar_wait(&bars->empty[s], (uint32_t)(j / kNS - 1) & 1, abort_flag, p.status);
        if (!ok) break;
        mbar_arrive_expect_tx(&bars->full[s], 2 * L::kHalfBytes + L::kRecBytes);
        for (int a = 0; a < D / 64; ++a) {
          tma_load_3d(stage_q(s) + a * L::kHalfAtom, &m.q64, &bars->full[s], 64 * a, q0, bh);
          tma_load_3d(stage_da(s) + a * L::kHalfAtom, &m.da64, &bars->full[s], 64 * a, q0, bh);
        }
        bulk_g2s(const_cast<float*>(stage_rec(s)),
                 p.rows + ((size_t)bh * p.tpad + (size_t)q0) * kGRowFloats,
                 (uint32_t)L::kRecBytes, &bars->full[s]);
        issued = j + 1;
      }
      if (!ok) {
        volatile int never = 0;
        const long long lim = kWaitLimitCycles / 4;
        for (int j = issued - 1; j >= 0 && j >= issued - kNS; --j)
          mbar_wait(&bars->full[j % kNS], (uint32_t)(j / kNS) & 1, &never, p.status, lim);
        mbar_wait(&bars->res_full, 0, &never, p.status, lim);
      }
    }
  } else if (warp == kWarpMMA) {
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16_f32(128, kHalf, 0, 0);
      constexpr uint32_t kIdAcc = idesc_bf16_f32(128, D, 0, 1);
      const uint64_t ak = smem_desc_sw128(smem_u32(smem + L::kR0), 16, 1024);
      const uint64_t av = smem_desc_sw128(smem_u32(smem + L::kR1), 16, 1024);
      const uint32_t lbo_mn = D == 128 ? L::kHalfAtom : 0;
      bool ok = mbar_wait(&bars->res_full, 0, abort_flag, p.status);
      bool any = false;
      auto issue_s = [&](int j) -> bool {
        const int s = j % kNS, b = j & 1;
        if (!mbar_wait(&bars->full[s], (uint32_t)(j / kNS) & 1, abort_flag, p.status)) return false;
        tc_fence_after();
        const uint64_t bq = smem_desc_sw128(smem_u32(stage_q(s)), 16, 1024);
        const uint64_t bd = smem_desc_sw128(smem_u32(stage_da(s)), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ss(tmem + kColS + kHalf * b, ak + kstep<L::kAtom>(kk), bq + kstep<L::kHalfAtom>(kk),
                  kIdS, kk > 0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ss(tmem + kColDP + kHalf * b, av + kstep<L::kAtom>(kk), bd + kstep<L::kHalfAtom>(kk),
                  kIdS, kk > 0);
        umma_commit(&bars->s_full[b]);
        any = true;
        return true;
      };
      if (ok) ok = issue_s(0);
      if (ok && nsteps > 1) ok = issue_s(1);
      for (int j = 0; j < nsteps && ok; ++j) {
        const int s = j % kNS, b = j & 1;
        ok = mbar_wait(&bars->p_full[b], (uint32_t)(j >> 1) & 1, abort_flag, p.status);
        if (!ok) break;
        tc_fence_after();
        const uint64_t bd = smem_desc_sw128(smem_u32(stage_da(s)), lbo_mn, 1024);
        const uint64_t bq = smem_desc_sw128(smem_u32(stage_q(s)), lbo_mn, 1024);
#pragma unroll
        for (int kk = 0; kk < kHalf / 16; ++kk)
          umma_ts(tmem + kColAcc, tmem + kColS + kHalf * b + 8 * kk,
                  bd + (uint64_t)(kk * (2048 >> 4)), kIdAcc, (j > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < kHalf / 16; ++kk)
          umma_ts(tmem + kColAcc + D, tmem + kColDP + kHalf * b + 8 * kk,
                  bq + (uint64_t)(kk * (2048 >> 4)), kIdAcc, (j > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&bars->empty[s]);
        if (j + 2 < nsteps) ok = issue_s(j + 2);
      }
      if (ok) umma_commit(&bars->acc_full);
      if (!ok && any) {
        volatile int never = 0;
        umma_commit(&bars->drain);
        mbar_wait(&bars->drain, 0, &never, p.status, kWaitLimitCycles / 4);
      }
    }
  } else if (warp < 8) {
    const int wg = warp >> 2;  // steps j with j & 1 == wg
    const int r = threadIdx.x & 127;
    const int key = kt * kTile + r;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t s_tm = tmem + lane_base + kColS + kHalf * wg;
    const uint32_t dp_tm = tmem + lane_base + kColDP + kHalf * wg;
    bool ok = true;
    for (int j = wg; j < nsteps && ok; j += 2) {
      const int s = j % kNS;
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->full[s], (uint32_t)(j / kNS) & 1, abort_flag, p.status));
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bars->s_full[wg], (uint32_t)(j >> 1) & 1, abort_flag, p.status));
      if (!ok) break;
      tc_fence_after();
      const float* rec = stage_rec(s);
      const int q0 = kt * kTile + kHalf * j;  // first query of this half
      const bool masked = (q0 < kt * kTile + kTile) || (q0 + kHalf > p.T);
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        uint32_t sv[32], dv[32];
        tmem_ld32(s_tm + 32 * c, sv);
        tmem_ld32(dp_tm + 32 * c, dv);
        tmem_ld_wait();
        reg_fence32(sv);
        reg_fence32(dv);
        uint32_t pk[16], dsk[16];
        if (masked)
          dkdv_chunk<true>(sv, dv, rec + 32 * c * kGRowFloats, key, q0 + 32 * c, p.T, pk, dsk);
        else
          dkdv_chunk<false>(sv, dv, rec + 32 * c * kGRowFloats, key, q0 + 32 * c, p.T, pk, dsk);
        tmem_st16(s_tm + 16 * c, pk);
        tmem_st16(dp_tm + 16 * c, dsk);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars->p_full[wg]);
    }
    // epilogue: warpgroup 0 writes dV, warpgroup 1 dK (fp32 rows)
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bars->acc_full, 0, abort_flag, p.status));
    if (ok) {
      tc_fence_after();
      const uint32_t acc_tm = tmem + lane_base + kColAcc + (uint32_t)(wg * D);
      float* dst = (wg == 0 ? p.dv : p.dk) + ((size_t)bh * p.T + (size_t)key) * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t ov[32];
        tmem_ld32(acc_tm + 32 * c, ov);
        tmem_ld_wait();
        reg_fence32(ov);
        if (key < p.T) {
          float4* o4 = reinterpret_cast<float4*>(dst + 32 * c);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            o4[e] = make_float4(__uint_as_float(ov[4 * e]), __uint_as_float(ov[4 * e + 1]),
                                __uint_as_float(ov[4 * e + 2]), __uint_as_float(ov[4 * e + 3]));
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMMA) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ================================================================== dQ ==
// Step j = one 64-key half (keys 64 j ...), ring stage j % NS, TMEM buffer /
// elementwise warpgroup j & 1.
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    polar_bwd_dq_kernel(const __grid_constant__ TileMaps m, const BwdTcParams p) {
  using L = Layout<D>;
  constexpr int kNS = L::kNS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + L::kBarOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // heaviest query tiles (most keys) first
  const int qt = p.n_t - 1 - (int)(blockIdx.x / p.BH);
  const int bh = (int)(blockIdx.x % p.BH);
  // causal halves 0 .. 2 qt + 1, without halves that start past the last row
  const int nsteps = min(2 * qt + 2, (p.T + kHalf - 1) / kHalf);

  if (threadIdx.x == 0) setup_barriers(bars, kNS);
  if (warp == kWarpMMA) tmem_alloc(&bars->tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  volatile int* abort_flag = &bars->abort_flag;
  auto stage_k = [&](int s) { return smem + L::kRing + s * L::kStageBytes; };
  auto stage_v = [&](int s) { return stage_k(s) + L::kHalfBytes; };

  if (warp == kWarpTMA) {
    if (lane == 0) {
      tma_prefetch_desc(&m.k64);
      tma_prefetch_desc(&m.v64);
      mbar_arrive_expect_tx(&bars->res_full, 2 * L::kTileBytes);
      for (int a = 0; a < D / 64; ++a) {
        tma_load_3d(smem + L::kR0 + a * L::kAtom, &m.q, &bars->res_full, 64 * a, kTile * qt, bh);
        tma_load_3d(smem + L::kR1 + a * L::kAtom, &m.da, &bars->res_full, 64 * a, kTile * qt, bh);
      }
      bool ok = true;
      int issued = 0;
      for (int j = 0; j < nsteps && ok; ++j) {
        const int s = j % kNS;
        if (j >= kNS) ok = mbar_wait(&bars->empty[s], (uint32_t)(j / kNS - 1) & 1, abort_flag, p.status);
        if (!ok) break;
        mbar_arrive_expect_tx(&bars->full[s], 2 * L::kHalfBytes);
        for (int a = 0; a < D / 64; ++a) {
          tma_load_3d(stage_k(s) + a * L::kHalfAtom, &m.k64, &bars->full[s], 64 * a, kHalf * j, bh);
          tma_load_3d(stage_v(s) + a * L::kHalfAtom, &m.v64, &bars->full[s], 64 * a, kHalf * j, bh);
        }
        issued = j + 1;
      }
      if (!ok) {
        volatile int never = 0;
        const long long lim = kWaitLimitCycles / 4;
        for (int j = issued - 1; j >= 0 && j >= issued - kNS; --j)
          mbar_wait(&bars->full[j % kNS], (uint32_t)(j / kNS) & 1, &never, p.status, lim);
        mbar_wait(&bars->res_full, 0, &never, p.status, lim);
      }
    }
  } else if (warp == kWarpMMA) {
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16_f32(128, kHalf, 0, 0);
      constexpr uint32_t kIdAcc = idesc_bf16_f32(128, D, 0, 1);
      const uint64_t aq = smem_desc_sw128(smem_u32(smem + L::kR0), 16, 1024);
      const uint64_t ad = smem_desc_sw128(smem_u32(smem + L::kR1), 16, 1024);
      const uint32_t lbo_mn = D == 128 ? L::kHalfAtom : 0;
      bool ok = mbar_wait(&bars->res_full, 0, abort_flag, p.status);
      bool any = false;
      auto issue_s = [&](int j) -> bool {
        const int s = j % kNS, b = j & 1;
        if (!mbar_wait(&bars->full[s], (uint32_t)(j / kNS) & 1, abort_flag, p.status)) return false;
        tc_fence_after();
        const uint64_t bk = smem_desc_sw128(smem_u32(stage_k(s)), 16, 1024);
        const uint64_t bv = smem_desc_sw128(smem_u32(stage_v(s)), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ss(tmem + kColS + kHalf * b, aq + kstep<L::kAtom>(kk), bk + kstep<L::kHalfAtom>(kk),
                  kIdS, kk > 0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ss(tmem + kColDP + kHalf * b, ad + kstep<L::kAtom>(kk), bv + kstep<L::kHalfAtom>(kk),
                  kIdS, kk > 0);
        umma_commit(&bars->s_full[b]);
        any = true;
        return true;
      };
      if (ok) ok = issue_s(0);
      if (ok && nsteps > 1) ok = issue_s(1);
      for (int j = 0; j < nsteps && ok; ++j) {
        const int s = j % kNS, b = j & 1;
        ok = mbar_wait(&bars->p_full[b], (uint32_t)(j >> 1) & 1, abort_flag, p.status);
        if (!ok) break;
        tc_fence_after();
        const uint64_t bk = smem_desc_sw128(smem_u32(stage_k(s)), lbo_mn, 1024);
#pragma unroll
        for (int kk = 0; kk < kHalf / 16; ++kk)
          umma_ts(tmem + kColAcc, tmem + kColDP + kHalf * b + 8 * kk,
                  bk + (uint64_t)(kk * (2048 >> 4)), kIdAcc, (j > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&bars->empty[s]);
        if (j + 2 < nsteps) ok = issue_s(j + 2);
      }
      if (ok) umma_commit(&bars->acc_full);
      if (!ok && any) {
        volatile int never = 0;
        umma_commit(&bars->drain);
        mbar_wait(&bars->drain, 0, &never, p.status, kWaitLimitCycles / 4);
      }
    }
  } else if (warp < 8) {
    const int wg = warp >> 2;  // steps j with j & 1 == wg
    const int r = threadIdx.x & 127;
    const int row = qt * kTile + r;
    const bool valid = row < p.T;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t s_tm = tmem + lane_base + kColS + kHalf * wg;
    const uint32_t dp_tm = tmem + lane_base + kColDP + kHalf * wg;
    // rows past T: p = 0 and dS' = 0 (cl2 = 0, nlse2 = -inf, the rest 0)
    float cl2 = 0.f, nlse2 = -INFINITY, coef = 0.f, cmdc = 0.f, ec = 0.f, qfloor = 0.f;
    if (valid) {
      auto ld = [&](int f) { return __ldg(p.rows + grad_row_index(bh, p.tpad, row, f)); };
      cl2 = ld(kGCl2);
      nlse2 = ld(kGNLse2);
      coef = ld(kGCoef);
      cmdc = ld(kGCmDc);
      ec = ld(kGEc);
      qfloor = ld(kGQFloor);
    }
    const float2 cl2p = make_float2(cl2, cl2), nlse2p = make_float2(nlse2, nlse2);
    const float2 coefp = make_float2(coef, coef), cmdcp = make_float2(cmdc, cmdc);
    const float2 ecp = make_float2(ec, ec);
    bool ok = true;
    for (int j = wg; j < nsteps && ok; j += 2) {
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->s_full[wg], (uint32_t)(j >> 1) & 1, abort_flag, p.status));
      if (!ok) break;
      tc_fence_after();
      const int k0 = kHalf * j;  // first key of this half
      const bool masked = k0 + kHalf > qt * kTile;  // halves of the diagonal tile
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        uint32_t sv[32], dv[32];
        tmem_ld32(s_tm + 32 * c, sv);
        tmem_ld32(dp_tm + 32 * c, dv);
        tmem_ld_wait();
        reg_fence32(sv);
        reg_fence32(dv);
        uint32_t dsk[16];
        if (masked)
          dq_chunk<true>(sv, dv, cl2p, nlse2p, coefp, cmdcp, ecp, row, k0 + 32 * c, dsk);
        else
          dq_chunk<false>(sv, dv, cl2p, nlse2p, coefp, cmdcp, ecp, row, k0 + 32 * c, dsk);
        tmem_st16(dp_tm + 16 * c, dsk);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars->p_full[wg]);
    }
    // epilogue: dq = acc + qfloor q; warpgroup w writes columns [w D/2, (w+1) D/2)
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bars->acc_full, 0, abort_flag, p.status));
    if (ok) {
      tc_fence_after();
      const size_t roff = ((size_t)bh * p.T + (size_t)(valid ? row : 0)) * D;
#pragma unroll 1
      for (int c = wg * (D / 64); c < (wg + 1) * (D / 64); ++c) {
        uint32_t ov[32];
        tmem_ld32(tmem + lane_base + kColAcc + 32 * c, ov);
        tmem_ld_wait();
        reg_fence32(ov);
        if (valid) {
          const uint4* qp = reinterpret_cast<const uint4*>(p.q + roff + 32 * c);
          float4* o4 = reinterpret_cast<float4*>(p.dq + roff + 32 * c);
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            const uint4 qu = __ldg(qp + g);
            const uint32_t qw[4] = {qu.x, qu.y, qu.z, qu.w};
            float y[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              y[2 * e] = fmaf(qfloor, __uint_as_float(qw[e] << 16), __uint_as_float(ov[8 * g + 2 * e]));
              y[2 * e + 1] = fmaf(qfloor, __uint_as_float(qw[e] & 0xFFFF0000u),
                                  __uint_as_float(ov[8 * g + 2 * e + 1]));
            }
            o4[2 * g] = make_float4(y[0], y[1], y[2], y[3]);
            o4[2 * g + 1] = make_float4(y[4], y[5], y[6], y[7]);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMMA) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ========================================================== dw reduce ==
// dw[h][x] = sum over b and 32-row blocks of the count * g partials.
template <int D>
__global__ void __launch_bounds__(256)
    polar_bwd_dw_reduce_kernel(const float* __restrict__ part, float* __restrict__ dw, int B, int H,
                               int nblk) {
  __shared__ float red[8][32];
  const int h = blockIdx.x, x = blockIdx.y * 32 + (threadIdx.x & 31), w = threadIdx.x >> 5;
  const int items = B * nblk;
  float s = 0.f;
#pragma unroll 4
  for (int it = w; it < items; it += 8) {
    const int b = it / nblk, blk = it - b * nblk;
    s += part[(((size_t)b * H + h) * nblk + blk) * D + x];
  }
  red[w][threadIdx.x & 31] = s;
  __syncthreads();
  if (w == 0) {
    float t = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) t += red[i][threadIdx.x & 31];
    dw[(size_t)h * D + x] = t;
  }
}

template <int D>
cudaError_t launch_tiles(const BwdArgs& a, const BwdTcLayout& w, const TileMaps& maps,
                         cudaStream_t s) {
  using L = Layout<D>;
  BwdTcParams p;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.rows = w.rows;
  p.dq = a.dq;
  p.dk = a.dk;
  p.dv = a.dv;
  p.status = a.status;
  p.T = a.T;
  p.BH = a.B * a.H;
  p.n_t = (a.T + kTile - 1) / kTile;
  p.tpad = grad_rows_tpad(a.T);
  const unsigned grid = (unsigned)((long long)p.n_t * p.BH);
  cudaError_t e = cudaFuncSetAttribute(polar_bwd_dkdv_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemBytes);
  if (e != cudaSuccess) return e;
  polar_bwd_dkdv_kernel<D><<<grid, kThreads, L::kSmemBytes, s>>>(maps, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  e = cudaFuncSetAttribute(polar_bwd_dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           L::kSmemBytes);
  if (e != cudaSuccess) return e;
  polar_bwd_dq_kernel<D><<<grid, kThreads, L::kSmemBytes, s>>>(maps, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int nblk = (a.T + 31) / 32;
  polar_bwd_dw_reduce_kernel<D><<<dim3(a.H, D / 32), 256, 0, s>>>(w.dw_part, a.dw, a.B, a.H, nblk);
  return cudaGetLastError();
}

}  // namespace

BwdTcLayout bwd_tc_layout(void* workspace, int B, int H, int T, int d) {
  const size_t rows = (size_t)B * H * T;
  const size_t rec_rows = (size_t)B * H * grad_rows_tpad(T);
  BwdTcLayout w;
  uint8_t* base = static_cast<uint8_t*>(workspace);
  w.da = base;
  w.rows = reinterpret_cast<float*>(base + rows * d * 2);
  w.dw_part = w.rows + rec_rows * kGRowFloats;
  w.bytes = rows * d * 2 + rec_rows * kGRowFloats * 4 + (size_t)B * H * ((T + 31) / 32) * d * 4;
  return w;
}

cudaError_t launch_bwd_tc(const BwdArgs& a, const BwdTcLayout& w, const CUtensorMap* maps,
                          cudaStream_t s) {
  TileMaps m;
  m.q = maps[0];
  m.k = maps[1];
  m.v = maps[2];
  m.da = maps[3];
  m.q64 = maps[4];
  m.k64 = maps[5];
  m.v64 = maps[6];
  m.da64 = maps[7];
  return a.d == 64 ? launch_tiles<64>(a, w, m, s) : launch_tiles<128>(a, w, m, s);
}

}  // namespace polar
