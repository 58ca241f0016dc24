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
//     shared memory and streams the query tiles at or after it (Q, dA and
//     the row records, TMA into a 2-stage ring).  Each 128-query tile is
//     processed as two 64-query halves h, one per TMEM buffer:
//       S^T = K Q_h^T, dP^T = V dA_h^T      (SS, M = 128 keys, N = 64)
//       P^T, dS'^T (bf16) written over them by softmax warpgroup h
//       dV += P^T dA_h, dK += dS'^T Q_h       (TS: A from TMEM, K = 64)
//     so one warpgroup's elementwise work overlaps the other half's MMAs.
//   * dQ: a CTA owns a 128-query tile, keeps Q and dA, streams the causal
//     key tiles (K and V ring), 64-key halves:
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

constexpr int kTile = 128;  // keys or queries per tile
constexpr int kHalf = 64;   // per MMA step (one TMEM buffer)
constexpr int kNS = 2;      // ring stages
constexpr int kThreads = 384;
constexpr int kWarpTMA = 8;
constexpr int kWarpMMA = 9;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColDP = 128, kColAcc = 256;

template <int D>
struct TileGeom {
  static constexpr int kTileBytes = kTile * D * 2;   // 128 rows x D bf16
  static constexpr int kAtomBytes = kTile * 128;     // one 64-column swizzle atom
  static constexpr int kHalfRowsBytes = kHalf * 128; // 64 rows inside an atom
  static constexpr int kRowRecBytes = kTile * kGRowFloats * 4;
};

// Both kernels hold two resident tiles (R0, R1) and a ring of kNS stages of
// two tiles (+ row records in the dK/dV kernel).
template <int D>
struct Layout {
  using G = TileGeom<D>;
  static constexpr int kR0 = 0;
  static constexpr int kR1 = kR0 + G::kTileBytes;
  static constexpr int kRing = kR1 + G::kTileBytes;
  static constexpr int kStageBytes = 2 * G::kTileBytes + G::kRowRecBytes;
  static constexpr int kBarOff = kRing + kNS * kStageBytes;
  // padded above half of the SM's shared memory: one CTA per SM, so the
  // 512 TMEM columns it allocates are never contended
  static constexpr int kNeed = kBarOff + 256 + 1024;
  static constexpr int kSmemBytes = kNeed > 232448 / 2 + 1024 ? kNeed : 232448 / 2 + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory");
};

struct Bars {
  uint64_t res_full;             // resident tiles landed
  uint64_t full[kNS], empty[kNS];
  uint64_t s_full[2], p_full[2];
  uint64_t acc_full;
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

struct BwdTcParams {
  const __nv_bfloat16* q;  // for the floor term of dQ
  const float* rows;       // [BH, T, kGRowFloats]
  float *dq, *dk, *dv;     // [BH, T, D] fp32
  int* status;
  int T, BH, n_t;
};

// K-major descriptor offset of K step kk (16 elements) in a tile of two
// 64-column swizzle atoms.
template <int D>
__device__ __forceinline__ uint64_t kstep(int kk) {
  return (uint64_t)((kk >> 2) * (TileGeom<D>::kAtomBytes >> 4) + (kk & 3) * 2);
}

__device__ __forceinline__ void setup_barriers(Bars* bars) {
  mbar_init(&bars->res_full, 1);
  for (int s = 0; s < kNS; ++s) {
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

// Elementwise step on one 64-column buffer for 32-column chunk c:
// p = exp2(S cl2 + nlse2), dS' = p (coef dP + cmdc + ec p), masked.
// Per-column scalars (dK/dV kernel) come from the row records in shared
// memory; per-row scalars (dQ kernel) are passed as a broadcast record.
struct Scal {
  float cl2, nlse2, coef, cmdc, ec;
};

__device__ __forceinline__ void grad_pair(float s0, float s1, float dp0, float dp1,
                                          const Scal& a, const Scal& b, bool v0, bool v1,
                                          uint32_t& pk, uint32_t& dsk) {
  const float2 x = ffma2(make_float2(s0, s1), make_float2(a.cl2, b.cl2),
                         make_float2(a.nlse2, b.nlse2));
  float p0 = ex2_approx(x.x), p1 = ex2_approx(x.y);
  p0 = v0 ? p0 : 0.f;
  p1 = v1 ? p1 : 0.f;
  const float2 t = ffma2(make_float2(dp0, dp1), make_float2(a.coef, b.coef),
                         make_float2(a.cmdc, b.cmdc));
  const float2 u = ffma2(make_float2(a.ec, b.ec), make_float2(p0, p1), t);
  pk = pack_bf16x2(p0, p1);
  // masked entries are selected to 0 (their records may be stale)
  dsk = pack_bf16x2(v0 ? p0 * u.x : 0.f, v1 ? p1 * u.y : 0.f);
}

// ============================================================ dK and dV ==
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    polar_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap map_q,
                          const __grid_constant__ CUtensorMap map_k,
                          const __grid_constant__ CUtensorMap map_v,
                          const __grid_constant__ CUtensorMap map_da, const BwdTcParams p) {
  using L = Layout<D>;
  using G = TileGeom<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + L::kBarOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // heaviest key tiles (most query tiles after them) first
  const int kt = (int)(blockIdx.x / p.BH);
  const int bh = (int)(blockIdx.x % p.BH);
  const int nq = p.n_t - kt;  // query tiles kt .. n_t - 1
  const int nsteps = 2 * nq;

  if (threadIdx.x == 0) setup_barriers(bars);
  if (warp == kWarpMMA) tmem_alloc(&bars->tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  volatile int* abort_flag = &bars->abort_flag;
  auto stage_q = [&](int s) { return smem + L::kRing + s * L::kStageBytes; };
  auto stage_da = [&](int s) { return stage_q(s) + G::kTileBytes; };
  auto stage_rec = [&](int s) {
    return reinterpret_cast<const float*>(stage_q(s) + 2 * G::kTileBytes);
  };

  if (warp == kWarpTMA) {
    if (lane == 0) {
      tma_prefetch_desc(&map_q);
      tma_prefetch_desc(&map_da);
      mbar_arrive_expect_tx(&bars->res_full, 2 * G::kTileBytes);
      for (int a = 0; a < D / 64; ++a) {
        tma_load_3d(smem + L::kR0 + a * G::kAtomBytes, &map_k, &bars->res_full, 64 * a,
                    kTile * kt, bh);
        tma_load_3d(smem + L::kR1 + a * G::kAtomBytes, &map_v, &bars->res_full, 64 * a,
                    kTile * kt, bh);
      }
      bool ok = true;
      int issued = 0;
      for (int i = 0; i < nq && ok; ++i) {
        const int s = i % kNS, qt = kt + i;
        if (i >= kNS) ok = mbar_wait(&bars->empty[s], (uint32_t)(i / kNS - 1) & 1, abort_flag, p.status);
        if (!ok) break;
        const int nvalid = min(kTile, p.T - qt * kTile);
        mbar_arrive_expect_tx(&bars->full[s], 2 * G::kTileBytes + nvalid * kGRowFloats * 4);
        for (int a = 0; a < D / 64; ++a) {
          tma_load_3d(stage_q(s) + a * G::kAtomBytes, &map_q, &bars->full[s], 64 * a,
                      kTile * qt, bh);
          tma_load_3d(stage_da(s) + a * G::kAtomBytes, &map_da, &bars->full[s], 64 * a,
                      kTile * qt, bh);
        }
        bulk_g2s(const_cast<float*>(stage_rec(s)),
                 p.rows + ((size_t)bh * p.T + (size_t)qt * kTile) * kGRowFloats,
                 (uint32_t)(nvalid * kGRowFloats * 4), &bars->full[s]);
        issued = i + 1;
      }
      if (!ok) {
        volatile int never = 0;
        const long long lim = kWaitLimitCycles / 4;
        for (int i = issued - 1; i >= 0 && i >= issued - kNS; --i)
          mbar_wait(&bars->full[i % kNS], (uint32_t)(i / kNS) & 1, &never, p.status, lim);
        mbar_wait(&bars->res_full, 0, &never, p.status, lim);
      }
    }
  } else if (warp == kWarpMMA) {
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16_f32(128, kHalf, 0, 0);
      constexpr uint32_t kIdAcc = idesc_bf16_f32(128, D, 0, 1);
      const uint64_t dk_ = smem_desc_sw128(smem_u32(smem + L::kR0), 16, 1024);
      const uint64_t dv_ = smem_desc_sw128(smem_u32(smem + L::kR1), 16, 1024);
      const uint32_t lbo_mn = D == 128 ? G::kAtomBytes : 0;
      bool ok = mbar_wait(&bars->res_full, 0, abort_flag, p.status);
      bool any = false;
      auto issue_s = [&](int j) -> bool {
        const int i = j >> 1, hh = j & 1, s = i % kNS;
        if (hh == 0) {
          if (!mbar_wait(&bars->full[s], (uint32_t)(i / kNS) & 1, abort_flag, p.status))
            return false;
          tc_fence_after();
        }
        const uint64_t bq = smem_desc_sw128(smem_u32(stage_q(s) + hh * G::kHalfRowsBytes), 16, 1024);
        const uint64_t bd = smem_desc_sw128(smem_u32(stage_da(s) + hh * G::kHalfRowsBytes), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ss(tmem + kColS + kHalf * hh, dk_ + kstep<D>(kk), bq + kstep<D>(kk), kIdS, kk > 0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ss(tmem + kColDP + kHalf * hh, dv_ + kstep<D>(kk), bd + kstep<D>(kk), kIdS, kk > 0);
        umma_commit(&bars->s_full[hh]);
        any = true;
        return true;
      };
      if (ok) ok = issue_s(0);
      if (ok) ok = issue_s(1);
      for (int j = 0; j < nsteps && ok; ++j) {
        const int i = j >> 1, hh = j & 1, s = i % kNS;
        ok = mbar_wait(&bars->p_full[hh], (uint32_t)i & 1, abort_flag, p.status);
        if (!ok) break;
        tc_fence_after();
        const uint64_t bd = smem_desc_sw128(smem_u32(stage_da(s) + hh * G::kHalfRowsBytes), lbo_mn, 1024);
        const uint64_t bq = smem_desc_sw128(smem_u32(stage_q(s) + hh * G::kHalfRowsBytes), lbo_mn, 1024);
#pragma unroll
        for (int kk = 0; kk < kHalf / 16; ++kk)
          umma_ts(tmem + kColAcc, tmem + kColS + kHalf * hh + 8 * kk,
                  bd + (uint64_t)(kk * (2048 >> 4)), kIdAcc, (j > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < kHalf / 16; ++kk)
          umma_ts(tmem + kColAcc + D, tmem + kColDP + kHalf * hh + 8 * kk,
                  bq + (uint64_t)(kk * (2048 >> 4)), kIdAcc, (j > 0 || kk > 0) ? 1u : 0u);
        if (hh == 1) umma_commit(&bars->empty[s]);
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
    const int wg = warp >> 2;  // 64-query half handled by this warpgroup
    const int r = threadIdx.x & 127;
    const int key = kt * kTile + r;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t s_tm = tmem + lane_base + kColS + kHalf * wg;
    const uint32_t dp_tm = tmem + lane_base + kColDP + kHalf * wg;
    bool ok = true;
    for (int i = 0; i < nq && ok; ++i) {
      const int s = i % kNS, qt = kt + i;
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->full[s], (uint32_t)(i / kNS) & 1, abort_flag, p.status));
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bars->s_full[wg], (uint32_t)i & 1, abort_flag, p.status));
      if (!ok) break;
      tc_fence_after();
      const float* rec = stage_rec(s) + (size_t)kHalf * wg * kGRowFloats;
      const int q0 = qt * kTile + kHalf * wg;  // first query of this half
      const bool masked = (qt == kt) || (q0 + kHalf > p.T);
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        uint32_t sv[32], dv[32];
        tmem_ld32(s_tm + 32 * c, sv);
        tmem_ld32(dp_tm + 32 * c, dv);
        tmem_ld_wait();
        reg_fence32(sv);
        reg_fence32(dv);
        uint32_t pk[16], dsk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int col = 32 * c + 2 * e;
          const float4 ra = *reinterpret_cast<const float4*>(rec + col * kGRowFloats);
          const float rae = rec[col * kGRowFloats + kGEc];
          const float4 rb = *reinterpret_cast<const float4*>(rec + (col + 1) * kGRowFloats);
          const float rbe = rec[(col + 1) * kGRowFloats + kGEc];
          const Scal sa{ra.x, ra.y, ra.z, ra.w, rae}, sb{rb.x, rb.y, rb.z, rb.w, rbe};
          bool v0 = true, v1 = true;
          if (masked) {
            const int qa = q0 + col;
            v0 = key <= qa && qa < p.T;
            v1 = key <= qa + 1 && qa + 1 < p.T;
          }
          grad_pair(__uint_as_float(sv[2 * e]), __uint_as_float(sv[2 * e + 1]),
                    __uint_as_float(dv[2 * e]), __uint_as_float(dv[2 * e + 1]), sa, sb, v0, v1,
                    pk[e], dsk[e]);
        }
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
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    polar_bwd_dq_kernel(const __grid_constant__ CUtensorMap map_q,
                        const __grid_constant__ CUtensorMap map_k,
                        const __grid_constant__ CUtensorMap map_v,
                        const __grid_constant__ CUtensorMap map_da, const BwdTcParams p) {
  using L = Layout<D>;
  using G = TileGeom<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + L::kBarOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // heaviest query tiles (most key tiles) first
  const int qt = p.n_t - 1 - (int)(blockIdx.x / p.BH);
  const int bh = (int)(blockIdx.x % p.BH);
  const int nk = qt + 1;  // key tiles 0 .. qt
  const int nsteps = 2 * nk;

  if (threadIdx.x == 0) setup_barriers(bars);
  if (warp == kWarpMMA) tmem_alloc(&bars->tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  volatile int* abort_flag = &bars->abort_flag;
  auto stage_k = [&](int s) { return smem + L::kRing + s * L::kStageBytes; };
  auto stage_v = [&](int s) { return stage_k(s) + G::kTileBytes; };

  if (warp == kWarpTMA) {
    if (lane == 0) {
      tma_prefetch_desc(&map_k);
      tma_prefetch_desc(&map_v);
      mbar_arrive_expect_tx(&bars->res_full, 2 * G::kTileBytes);
      for (int a = 0; a < D / 64; ++a) {
        tma_load_3d(smem + L::kR0 + a * G::kAtomBytes, &map_q, &bars->res_full, 64 * a,
                    kTile * qt, bh);
        tma_load_3d(smem + L::kR1 + a * G::kAtomBytes, &map_da, &bars->res_full, 64 * a,
                    kTile * qt, bh);
      }
      bool ok = true;
      int issued = 0;
      for (int i = 0; i < nk && ok; ++i) {
        const int s = i % kNS;
        if (i >= kNS) ok = mbar_wait(&bars->empty[s], (uint32_t)(i / kNS - 1) & 1, abort_flag, p.status);
        if (!ok) break;
        mbar_arrive_expect_tx(&bars->full[s], 2 * G::kTileBytes);
        for (int a = 0; a < D / 64; ++a) {
          tma_load_3d(stage_k(s) + a * G::kAtomBytes, &map_k, &bars->full[s], 64 * a, kTile * i, bh);
          tma_load_3d(stage_v(s) + a * G::kAtomBytes, &map_v, &bars->full[s], 64 * a, kTile * i, bh);
        }
        issued = i + 1;
      }
      if (!ok) {
        volatile int never = 0;
        const long long lim = kWaitLimitCycles / 4;
        for (int i = issued - 1; i >= 0 && i >= issued - kNS; --i)
          mbar_wait(&bars->full[i % kNS], (uint32_t)(i / kNS) & 1, &never, p.status, lim);
        mbar_wait(&bars->res_full, 0, &never, p.status, lim);
      }
    }
  } else if (warp == kWarpMMA) {
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16_f32(128, kHalf, 0, 0);
      constexpr uint32_t kIdAcc = idesc_bf16_f32(128, D, 0, 1);
      const uint64_t aq = smem_desc_sw128(smem_u32(smem + L::kR0), 16, 1024);
      const uint64_t ad = smem_desc_sw128(smem_u32(smem + L::kR1), 16, 1024);
      const uint32_t lbo_mn = D == 128 ? G::kAtomBytes : 0;
      bool ok = mbar_wait(&bars->res_full, 0, abort_flag, p.status);
      bool any = false;
      auto issue_s = [&](int j) -> bool {
        const int i = j >> 1, hh = j & 1, s = i % kNS;
        if (hh == 0) {
          if (!mbar_wait(&bars->full[s], (uint32_t)(i / kNS) & 1, abort_flag, p.status))
            return false;
          tc_fence_after();
        }
        const uint64_t bk = smem_desc_sw128(smem_u32(stage_k(s) + hh * G::kHalfRowsBytes), 16, 1024);
        const uint64_t bv = smem_desc_sw128(smem_u32(stage_v(s) + hh * G::kHalfRowsBytes), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ss(tmem + kColS + kHalf * hh, aq + kstep<D>(kk), bk + kstep<D>(kk), kIdS, kk > 0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ss(tmem + kColDP + kHalf * hh, ad + kstep<D>(kk), bv + kstep<D>(kk), kIdS, kk > 0);
        umma_commit(&bars->s_full[hh]);
        any = true;
        return true;
      };
      if (ok) ok = issue_s(0);
      if (ok) ok = issue_s(1);
      for (int j = 0; j < nsteps && ok; ++j) {
        const int i = j >> 1, hh = j & 1, s = i % kNS;
        ok = mbar_wait(&bars->p_full[hh], (uint32_t)i & 1, abort_flag, p.status);
        if (!ok) break;
        tc_fence_after();
        const uint64_t bk = smem_desc_sw128(smem_u32(stage_k(s) + hh * G::kHalfRowsBytes), lbo_mn, 1024);
#pragma unroll
        for (int kk = 0; kk < kHalf / 16; ++kk)
          umma_ts(tmem + kColAcc, tmem + kColDP + kHalf * hh + 8 * kk,
                  bk + (uint64_t)(kk * (2048 >> 4)), kIdAcc, (j > 0 || kk > 0) ? 1u : 0u);
        if (hh == 1) umma_commit(&bars->empty[s]);
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
    const int wg = warp >> 2;  // 64-key half handled by this warpgroup
    const int r = threadIdx.x & 127;
    const int row = qt * kTile + r;
    const bool valid = row < p.T;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t s_tm = tmem + lane_base + kColS + kHalf * wg;
    const uint32_t dp_tm = tmem + lane_base + kColDP + kHalf * wg;
    Scal sc{0.f, -INFINITY, 0.f, 0.f, 0.f};  // rows past T: p = 0, dS' = 0
    float qfloor = 0.f;
    if (valid) {
      const float4* rp = reinterpret_cast<const float4*>(p.rows + ((size_t)bh * p.T + row) * kGRowFloats);
      const float4 a = __ldg(rp), b = __ldg(rp + 1);
      sc = Scal{a.x, a.y, a.z, a.w, b.x};
      qfloor = b.y;
    }
    bool ok = true;
    for (int i = 0; i < nk && ok; ++i) {
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->s_full[wg], (uint32_t)i & 1, abort_flag, p.status));
      if (!ok) break;
      tc_fence_after();
      const int k0 = i * kTile + kHalf * wg;  // first key of this half
      const bool masked = i == qt;
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        uint32_t sv[32], dv[32];
        tmem_ld32(s_tm + 32 * c, sv);
        tmem_ld32(dp_tm + 32 * c, dv);
        tmem_ld_wait();
        reg_fence32(sv);
        reg_fence32(dv);
        uint32_t pk[16], dsk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          bool v0 = true, v1 = true;
          if (masked) {
            const int ka = k0 + 32 * c + 2 * e;
            v0 = ka <= row;
            v1 = ka + 1 <= row;
          }
          grad_pair(__uint_as_float(sv[2 * e]), __uint_as_float(sv[2 * e + 1]),
                    __uint_as_float(dv[2 * e]), __uint_as_float(dv[2 * e + 1]), sc, sc, v0, v1,
                    pk[e], dsk[e]);
        }
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
cudaError_t launch_tiles(const BwdArgs& a, const BwdTcLayout& w, const CUtensorMap& mq,
                         const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mda,
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
  const unsigned grid = (unsigned)((long long)p.n_t * p.BH);
  cudaError_t e = cudaFuncSetAttribute(polar_bwd_dkdv_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemBytes);
  if (e != cudaSuccess) return e;
  polar_bwd_dkdv_kernel<D><<<grid, kThreads, L::kSmemBytes, s>>>(mq, mk, mv, mda, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  e = cudaFuncSetAttribute(polar_bwd_dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           L::kSmemBytes);
  if (e != cudaSuccess) return e;
  polar_bwd_dq_kernel<D><<<grid, kThreads, L::kSmemBytes, s>>>(mq, mk, mv, mda, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int nblk = (a.T + 31) / 32;
  polar_bwd_dw_reduce_kernel<D><<<dim3(a.H, D / 32), 256, 0, s>>>(w.dw_part, a.dw, a.B, a.H, nblk);
  return cudaGetLastError();
}

}  // namespace

BwdTcLayout bwd_tc_layout(void* workspace, int B, int H, int T, int d) {
  const size_t rows = (size_t)B * H * T;
  BwdTcLayout w;
  uint8_t* base = static_cast<uint8_t*>(workspace);
  w.da = base;
  w.rows = reinterpret_cast<float*>(base + rows * d * 2);
  w.dw_part = w.rows + rows * kGRowFloats;
  w.bytes = rows * d * 2 + rows * kGRowFloats * 4 + (size_t)B * H * ((T + 31) / 32) * d * 4;
  return w;
}

cudaError_t launch_bwd_tc(const BwdArgs& a, const BwdTcLayout& w, const CUtensorMap& mq,
                          const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mda,
                          cudaStream_t s) {
  return a.d == 64 ? launch_tiles<64>(a, w, mq, mk, mv, mda, s)
                   : launch_tiles<128>(a, w, mq, mk, mv, mda, s);
}

}  // namespace polar
