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
// Two kernels, one CTA per SM each (512 TMEM columns), 128-row steps so
// that every MMA is M = 128, N = 128 (an N = 64 MMA with both operands in
// shared memory is bound by shared-memory bandwidth, not by the tensor core):
//   * dK/dV: a CTA owns a 128-key tile of one (b, h), keeps K and V in
//     shared memory and streams the query tiles at or after it (a ring of
//     Q + row records, freed after dK, and a ring of dA, freed after dV).
//     TMEM: S^T (cols 0-127), dP^T (128-255), dV, dK.  Per step:
//       S^T = K Q^T, dP^T = V dA^T;  phase A: P^T (bf16) over S^T;
//       dV += P^T dA;  S^T of the next step;  phase B: dS'^T over dP^T;
//       dK += dS'^T Q;  dP^T of the next step
//     so each elementwise phase overlaps two 128 x 128 x d products.
//   * dQ: a CTA owns a 128-query tile, keeps Q and dA and streams the
//     causal key tiles (a ring of K, freed after dQ, and a ring of V, freed
//     after dP).  TMEM: S (0-127), two dP buffers (128-383), dQ.  Per step:
//       S = Q K^T (one step ahead), dP = dA V^T (two steps ahead);
//       dS' over dP;  dQ += dS' K.
// Roles (384 threads): warps 0-3 and 4-7 are two elementwise warpgroups
// that split the 128 columns of a step (64 each; thread = TMEM lane = key
// or query row of the tile; each writes its bf16 results only over columns
// it has already read), warp 8 issues TMA, warp 9 issues the MMAs and owns
// TMEM.  Every wait is bounded (status 1 on timeout).
#include <mutex>

#include "polar_device.cuh"
#include "polar_grad.cuh"
#include "polar_internal.h"

namespace polar {

namespace {

constexpr int kTile = 128;  // keys or queries per step
constexpr int kNSMax = 3;
constexpr int kThreads = 384;
constexpr int kWarpTMA = 8;
constexpr int kWarpMMA = 9;
constexpr uint32_t kTmemCols = 512;

// Shared memory: two resident tiles (R0, R1) and two rings of streamed
// tiles (A: with the row records in the dK/dV kernel; B).
template <int D, bool kDkdv>
struct Layout {
  static constexpr int kTileBytes = kTile * D * 2;  // 128 rows x D bf16
  static constexpr int kAtom = kTile * 128;         // one 64-column swizzle atom
  static constexpr int kRecBytes = kDkdv ? (kTile / 2) * kGPairFloats * 4 : 0;
  static constexpr int kNSA = D == 128 ? (kDkdv ? 2 : 3) : 3;
  static constexpr int kNSB = D == 128 ? 2 : 3;
  static constexpr int kStageA = kTileBytes + kRecBytes;
  static constexpr int kStageB = kTileBytes;
  static constexpr int kR0 = 0;
  static constexpr int kR1 = kTileBytes;
  static constexpr int kRingA = 2 * kTileBytes;
  static constexpr int kRingB = kRingA + kNSA * kStageA;
  static constexpr int kBarOff = kRingB + kNSB * kStageB;
  // padded above half of the SM's shared memory: one CTA per SM, so the
  // 512 TMEM columns it allocates are never contended
  static constexpr int kNeed = kBarOff + 256 + 1024;
  static constexpr int kSmemBytes = kNeed > 232448 / 2 + 1024 ? kNeed : 232448 / 2 + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory");
  static_assert(kNSA <= kNSMax && kNSB <= kNSMax, "ring");
  static_assert(kStageA % 1024 == 0 && kStageB % 1024 == 0, "swizzle alignment");
};

struct Bars {
  uint64_t res_full;  // resident tiles landed
  uint64_t full_a[kNSMax], empty_a[kNSMax];
  uint64_t full_b[kNSMax], empty_b[kNSMax];
  uint64_t s_full[2];   // dK/dV: S^T, dP^T done;  dQ: S done ([0])
  uint64_t dp_full[2];  // dQ: dP buffer done
  uint64_t pa, pb;      // elementwise phases done (256 arrivals each)
  uint64_t acc_full;
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

struct BwdTcParams {
  const __nv_bfloat16* q;  // for the floor term of dQ
  const float* rows;       // pair blocks (polar_grad.cuh)
  float *dq, *dk, *dv;     // [BH, T, D] fp32
  int* status;
  int T, BH, n_t, tpad;
  int head_group;  // CTA order: heads per group (l2_head_group)
};

struct TileMaps {
  CUtensorMap q, k, v, da;  // box 64 x 128, 128-byte swizzle
};

// K-major descriptor offset of K step kk (16 elements) in a 128-row tile of
// two 64-column swizzle atoms.
__device__ __forceinline__ uint64_t kstep(int kk) {
  return (uint64_t)((kk >> 2) * ((kTile * 128) >> 4) + (kk & 3) * 2);
}

// TMEM column of the bf16 A operand for K step kk of a 128-column step:
// warpgroup 0 wrote columns 0-63 of the step packed into base + 0..31,
// warpgroup 1 columns 64-127 into base + 64..95.
__device__ __forceinline__ uint32_t a_col(int kk) {
  return kk < 4 ? 8u * kk : 64u + 8u * (kk - 4);
}

__device__ __forceinline__ void setup_barriers(Bars* bars, int nsa, int nsb) {
  mbar_init(&bars->res_full, 1);
  for (int s = 0; s < nsa; ++s) {
    mbar_init(&bars->full_a[s], 1);
    mbar_init(&bars->empty_a[s], 1);
  }
  for (int s = 0; s < nsb; ++s) {
    mbar_init(&bars->full_b[s], 1);
    mbar_init(&bars->empty_b[s], 1);
  }
  for (int b = 0; b < 2; ++b) {
    mbar_init(&bars->s_full[b], 1);
    mbar_init(&bars->dp_full[b], 1);
  }
  // one arrival per elementwise warp (lane 0, after the warp's stores):
  // 256 per-thread arrivals on one word serialise in shared memory
  mbar_init(&bars->pa, 8);
  mbar_init(&bars->pb, 8);
  mbar_init(&bars->acc_full, 1);
  mbar_init(&bars->drain, 1);
  bars->abort_flag = 0;
  fence_barrier_init();
}

// TMA producer of both kernels, run by a whole warp (one elected lane
// issues): the resident tiles, then the two rings in step order.  On abort
// it lets its copies in flight land.
template <int D, bool kDkdv>
__device__ __forceinline__ void produce(uint8_t* smem, Bars* bars, const CUtensorMap* r0,
                                        const CUtensorMap* r1, int r_row, const CUtensorMap* ma,
                                        const CUtensorMap* mb, int row0, int nsteps, int bh,
                                        const BwdTcParams& p, volatile int* abort_flag) {
  using L = Layout<D, kDkdv>;
  if ((threadIdx.x & 31) == 0) {
    tma_prefetch_desc(ma);
    tma_prefetch_desc(mb);
  }
  __syncwarp();
  mbar_arrive_expect_tx_warp(&bars->res_full, 2 * L::kTileBytes);
  for (int a = 0; a < D / 64; ++a) {
    tma_load_3d_warp(smem + L::kR0 + a * L::kAtom, r0, &bars->res_full, 64 * a, r_row, bh);
    tma_load_3d_warp(smem + L::kR1 + a * L::kAtom, r1, &bars->res_full, 64 * a, r_row, bh);
  }
  bool ok = true;
  int ia = 0, ib = 0;
  for (int j = 0; j < nsteps && ok; ++j) {
    const int row = row0 + kTile * j;
    const int sa = j % L::kNSA, sb = j % L::kNSB;
    if (j >= L::kNSA)
      ok = mbar_wait_warp(&bars->empty_a[sa], (uint32_t)(j / L::kNSA - 1) & 1, abort_flag,
                          p.status);
    if (!ok) break;
    uint8_t* da = smem + L::kRingA + sa * L::kStageA;
    mbar_arrive_expect_tx_warp(&bars->full_a[sa], L::kStageA);
    for (int a = 0; a < D / 64; ++a)
      tma_load_3d_warp(da + a * L::kAtom, ma, &bars->full_a[sa], 64 * a, row, bh);
    if (kDkdv)
      bulk_g2s_warp(da + L::kTileBytes, p.rows + grad_row_index(bh, p.tpad, row, 0),
               (uint32_t)L::kRecBytes, &bars->full_a[sa]);
    ia = j + 1;
    if (j >= L::kNSB)
      ok = mbar_wait_warp(&bars->empty_b[sb], (uint32_t)(j / L::kNSB - 1) & 1, abort_flag,
                          p.status);
    if (!ok) break;
    uint8_t* db = smem + L::kRingB + sb * L::kStageB;
    mbar_arrive_expect_tx_warp(&bars->full_b[sb], L::kStageB);
    for (int a = 0; a < D / 64; ++a)
      tma_load_3d_warp(db + a * L::kAtom, mb, &bars->full_b[sb], 64 * a, row, bh);
    ib = j + 1;
  }
  if (!ok) {
    volatile int never = 0;
    const long long lim = kWaitLimitCycles / 4;
    for (int j = ia - 1; j >= 0 && j >= ia - L::kNSA; --j)
      mbar_wait(&bars->full_a[j % L::kNSA], (uint32_t)(j / L::kNSA) & 1, &never, p.status, lim);
    for (int j = ib - 1; j >= 0 && j >= ib - L::kNSB; --j)
      mbar_wait(&bars->full_b[j % L::kNSB], (uint32_t)(j / L::kNSB) & 1, &never, p.status, lim);
    mbar_wait(&bars->res_full, 0, &never, p.status, lim);
    __syncwarp();
  }
}

// ----------------------------------------------------- elementwise chunks
// One 32-column chunk, two columns at a time with packed fp32 pairs:
//   p = exp2(S cl2 + nlse2),  dS' = p (coef dP + cmdc + ec p)
// kMasked: entries outside the causal triangle or past T are selected to 0
// (the records of rows past T are not initialised).  The mask is a template
// parameter so that the unrolled loop has no branch: each chunk is one
// basic block and its 16 independent pairs overlap.

// dK/dV kernel: TMEM is read with the 16-lane shape .16x256b (x8: 64
// columns of 16 lanes), so a thread holds two keys (lanes t/4 and t/4 + 8 of
// the 16) for 8 pairs of consecutive queries (columns 8m + 2 (t % 4) + 0/1):
// per step it needs the scalars of 16 queries instead of 64.  Register
// 4m + 0/1 holds key t/4, 4m + 2/3 key t/4 + 8.  The packed bf16 results
// go back with .16x128b.x8, whose thread layout puts register 2m (2m + 1) at
// lane t/4 (t/4 + 8), column 4m + t % 4: the packed column of the pair.
// The scalars of pair m come from the pair block 4m blocks after the
// thread's first one (ra / rb / re below), loaded once per step for both
// 16-lane halves.

// phase A: P^T
template <bool kMasked>
__device__ __forceinline__ void dkdv_p(const uint32_t (&sv)[32], const float4 (&ra)[8], int key0,
                                       int q0, int T, uint32_t (&pk)[16]) {
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    const float4 r0 = ra[m];  // cl2, nlse2
    const float2 c2 = make_float2(r0.x, r0.y), n2 = make_float2(r0.z, r0.w);
    const float2 x0 = ffma2(make_float2(__uint_as_float(sv[4 * m]), __uint_as_float(sv[4 * m + 1])), c2, n2);
    const float2 x1 = ffma2(make_float2(__uint_as_float(sv[4 * m + 2]), __uint_as_float(sv[4 * m + 3])), c2, n2);
    float2 p0 = make_float2(ex2_approx(x0.x), ex2_approx(x0.y));
    float2 p1 = make_float2(ex2_approx(x1.x), ex2_approx(x1.y));
    if (kMasked) {
      const int q = q0 + 8 * m;
      const bool qa = q < T, qb = q + 1 < T;
      p0.x = (key0 <= q && qa) ? p0.x : 0.f;
      p0.y = (key0 <= q + 1 && qb) ? p0.y : 0.f;
      p1.x = (key0 + 8 <= q && qa) ? p1.x : 0.f;
      p1.y = (key0 + 8 <= q + 1 && qb) ? p1.y : 0.f;
    }
    pk[2 * m] = pack_bf16x2(p0.x, p0.y);
    pk[2 * m + 1] = pack_bf16x2(p1.x, p1.y);
  }
}

// phase B: dS'^T from dP^T and the (bf16) p of phase A
template <bool kMasked>
__device__ __forceinline__ void dkdv_ds(const uint32_t (&dv)[32], const uint32_t (&pk)[16],
                                        const float4 (&rb)[8], const float2 (&re)[8], int key0,
                                        int q0, int T, uint32_t (&dsk)[16]) {
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    const float4 r1 = rb[m];  // coef, cmdc
    const float2 ec = re[m];
    const float2 cf = make_float2(r1.x, r1.y), cm = make_float2(r1.z, r1.w);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t pw = pk[2 * m + h];
      const float2 pp = make_float2(__uint_as_float(pw << 16), __uint_as_float(pw & 0xFFFF0000u));
      const float2 t = ffma2(make_float2(__uint_as_float(dv[4 * m + 2 * h]),
                                         __uint_as_float(dv[4 * m + 2 * h + 1])), cf, cm);
      const float2 u = ffma2(ec, pp, t);
      float2 ds = ffma2(pp, u, make_float2(0.f, 0.f));
      if (kMasked) {
        const int q = q0 + 8 * m, key = key0 + 8 * h;
        ds.x = (key <= q && q < T) ? ds.x : 0.f;
        ds.y = (key <= q + 1 && q + 1 < T) ? ds.y : 0.f;
      }
      dsk[2 * m + h] = pack_bf16x2(ds.x, ds.y);
    }
  }
}

__device__ __forceinline__ void tmem_ld_16x256b_x8(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x8.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
        "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
        "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]),
        "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
        "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_st_16x128b_x8(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x128b.x8.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

// dQ: the row's scalars are the same for every column (packed pairs in
// registers); masked chunks are those of the diagonal tile.
template <bool kMasked>
__device__ __forceinline__ void chunk_ds(const uint32_t (&sv)[32], const uint32_t (&dv)[32],
                                         float2 cl2, float2 nlse2, float2 coef, float2 cmdc,
                                         float2 ec, int row, int k_first, uint32_t (&dsk)[16]) {
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

// Epilogue store of 32 fp32 accumulator columns of one row.
__device__ __forceinline__ void store_row32(float* dst, const uint32_t (&ov)[32]) {
  float4* o4 = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int e = 0; e < 8; ++e)
    o4[e] = make_float4(__uint_as_float(ov[4 * e]), __uint_as_float(ov[4 * e + 1]),
                        __uint_as_float(ov[4 * e + 2]), __uint_as_float(ov[4 * e + 3]));
}

// ============================================================ dK and dV ==
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    polar_bwd_dkdv_kernel(const __grid_constant__ TileMaps m, const BwdTcParams p) {
  using L = Layout<D, true>;
  constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + L::kBarOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // heads in L2-sized groups (their streamed Q and dA stay in L2), heaviest
  // key tiles (most query tiles after them) first within a group
  const int full = p.n_t * p.head_group;
  const int grp = (int)(blockIdx.x / full);
  const int rem = (int)blockIdx.x - grp * full;
  const int hg = min(p.head_group, p.BH - grp * p.head_group);
  const int kt = rem / hg;
  const int bh = grp * p.head_group + rem % hg;
  const int nq = p.n_t - kt;  // query tiles kt .. n_t - 1

  if (threadIdx.x == 0) setup_barriers(bars, L::kNSA, L::kNSB);
  if (warp == kWarpMMA) tmem_alloc(&bars->tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  volatile int* abort_flag = &bars->abort_flag;
  auto stage_q = [&](int j) { return smem + L::kRingA + (j % L::kNSA) * L::kStageA; };
  auto stage_da = [&](int j) { return smem + L::kRingB + (j % L::kNSB) * L::kStageB; };

  if (warp == kWarpTMA) {
    // the whole warp; one elected lane issues the copies
    produce<D, true>(smem, bars, &m.k, &m.v, kTile * kt, &m.q, &m.da, kTile * kt, nq, bh, p,
                     abort_flag);
  } else if (warp == kWarpMMA) {
    // whole warp: uniform waits and descriptors, one elected lane issues
    {
      constexpr uint32_t kIdS = idesc_bf16_f32(128, kTile, 0, 0);
      constexpr uint32_t kIdAcc = idesc_bf16_f32(128, D, 0, 1);
      const uint64_t ak = smem_desc_sw128(smem_u32(smem + L::kR0), 16, 1024);
      const uint64_t av = smem_desc_sw128(smem_u32(smem + L::kR1), 16, 1024);
      const uint32_t lbo_mn = D == 128 ? L::kAtom : 0;
      bool ok = mbar_wait_warp(&bars->res_full, 0, abort_flag, p.status);
      bool any = false;
      auto issue_st = [&](int j) -> bool {  // S^T = K Q^T
        if (!mbar_wait_warp(&bars->full_a[j % L::kNSA], (uint32_t)(j / L::kNSA) & 1, abort_flag,
                            p.status))
          return false;
        tc_fence_after();
        const uint64_t bq = smem_desc_sw128(smem_u32(stage_q(j)), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ss_warp(tmem + kColS, ak + kstep(kk), bq + kstep(kk), kIdS, kk > 0);
        umma_commit_warp(&bars->s_full[0]);
        any = true;
        return true;
      };
      auto issue_dpt = [&](int j) -> bool {  // dP^T = V dA^T
        if (!mbar_wait_warp(&bars->full_b[j % L::kNSB], (uint32_t)(j / L::kNSB) & 1, abort_flag,
                            p.status))
          return false;
        tc_fence_after();
        const uint64_t bd = smem_desc_sw128(smem_u32(stage_da(j)), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ss_warp(tmem + kColDP, av + kstep(kk), bd + kstep(kk), kIdS, kk > 0);
        umma_commit_warp(&bars->s_full[1]);
        return true;
      };
      if (ok) ok = issue_st(0);
      if (ok) ok = issue_dpt(0);
      for (int j = 0; j < nq && ok; ++j) {
        // dV += P^T dA once phase A has written P^T
        ok = mbar_wait_warp(&bars->pa, (uint32_t)j & 1, abort_flag, p.status);
        if (!ok) break;
        tc_fence_after();
        const uint64_t bd = smem_desc_sw128(smem_u32(stage_da(j)), lbo_mn, 1024);
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          umma_ts_warp(tmem + kColDV, tmem + kColS + a_col(kk), bd + (uint64_t)(kk * (2048 >> 4)),
                       kIdAcc, (j > 0 || kk > 0) ? 1u : 0u);
        umma_commit_warp(&bars->empty_b[j % L::kNSB]);
        if (j + 1 < nq) ok = issue_st(j + 1);  // over P^T: ordered after the dV MMAs
        if (!ok) break;
        // dK += dS'^T Q once phase B has written dS'^T
        ok = mbar_wait_warp(&bars->pb, (uint32_t)j & 1, abort_flag, p.status);
        if (!ok) break;
        tc_fence_after();
        const uint64_t bq = smem_desc_sw128(smem_u32(stage_q(j)), lbo_mn, 1024);
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          umma_ts_warp(tmem + kColDK, tmem + kColDP + a_col(kk), bq + (uint64_t)(kk * (2048 >> 4)),
                       kIdAcc, (j > 0 || kk > 0) ? 1u : 0u);
        umma_commit_warp(&bars->empty_a[j % L::kNSA]);
        if (j + 1 < nq) ok = issue_dpt(j + 1);  // over dS'^T: ordered after the dK MMAs
      }
      if (ok) umma_commit_warp(&bars->acc_full);
      if (!ok && any) {
        volatile int never = 0;
        umma_commit_warp(&bars->drain);
        __syncwarp();
        mbar_wait(&bars->drain, 0, &never, p.status, kWaitLimitCycles / 4);
        __syncwarp();
      }
    }
  } else if (warp < 8) {
    const int wg = warp >> 2;  // query columns 64 wg .. 64 wg + 63 of each step
    const int sub = warp & 3;  // TMEM lanes 32 sub .. 32 sub + 31
    const int t4 = lane >> 2, tq = lane & 3;
    bool ok = true;
    for (int j = 0; j < nq && ok; ++j) {
      const int qt = kt + j;
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->full_a[j % L::kNSA], (uint32_t)(j / L::kNSA) & 1,
                                             abort_flag, p.status));
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bars->s_full[0], (uint32_t)j & 1, abort_flag, p.status));
      if (!ok) break;
      tc_fence_after();
      // this thread's first pair block: query pair 64 wg + 2 tq
      const float* rec = reinterpret_cast<const float*>(stage_q(j) + L::kTileBytes) +
                         (32 * wg + tq) * kGPairFloats;
      const int q0 = qt * kTile + 64 * wg + 2 * tq;
      const bool masked = j == 0 || qt * kTile + 64 * wg + 64 > p.T;
      // phase A: P^T, per 16-lane half h of the warp's 32 keys.  The row
      // records are loaded once for both halves (they depend on the query
      // columns only): shared-memory wavefronts were the busiest resource
      uint32_t pk[2][16];
      {
        float4 ra[8];
#pragma unroll
        for (int m = 0; m < 8; ++m)
          ra[m] = *reinterpret_cast<const float4*>(rec + 4 * m * kGPairFloats);  // cl2, nlse2
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t lanes = (uint32_t)(32 * sub + 16 * h) << 16;
          const int key0 = kt * kTile + 32 * sub + 16 * h + t4;
          uint32_t sv[32];
          tmem_ld_16x256b_x8(tmem + lanes + kColS + 64 * wg, sv);
          tmem_ld_wait();
          reg_fence32(sv);
          if (masked)
            dkdv_p<true>(sv, ra, key0, q0, p.T, pk[h]);
          else
            dkdv_p<false>(sv, ra, key0, q0, p.T, pk[h]);
          tmem_st_16x128b_x8(tmem + lanes + kColS + 64 * wg, pk[h]);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->pa);
      // phase B: dS'^T
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->s_full[1], (uint32_t)j & 1, abort_flag, p.status));
      if (!ok) break;
      tc_fence_after();
      float4 rb[8];
      float2 re[8];
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        rb[m] = *reinterpret_cast<const float4*>(rec + 4 * m * kGPairFloats + 4);  // coef, cmdc
        re[m] = *reinterpret_cast<const float2*>(rec + 4 * m * kGPairFloats + 8);  // ec
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t lanes = (uint32_t)(32 * sub + 16 * h) << 16;
        const int key0 = kt * kTile + 32 * sub + 16 * h + t4;
        uint32_t dv[32], dsk[16];
        tmem_ld_16x256b_x8(tmem + lanes + kColDP + 64 * wg, dv);
        tmem_ld_wait();
        reg_fence32(dv);
        if (masked)
          dkdv_ds<true>(dv, pk[h], rb, re, key0, q0, p.T, dsk);
        else
          dkdv_ds<false>(dv, pk[h], rb, re, key0, q0, p.T, dsk);
        tmem_st_16x128b_x8(tmem + lanes + kColDP + 64 * wg, dsk);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->pb);
    }
    // epilogue: warpgroup 0 writes dV, warpgroup 1 dK (fp32 rows)
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bars->acc_full, 0, abort_flag, p.status));
    if (ok) {
      tc_fence_after();
      const int key = kt * kTile + (threadIdx.x & 127);
      const uint32_t lane_base = (uint32_t)(32 * sub) << 16;
      const uint32_t acc_tm = tmem + lane_base + (wg == 0 ? kColDV : kColDK);
      float* dst = (wg == 0 ? p.dv : p.dk) + ((size_t)bh * p.T + (size_t)key) * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t ov[32];
        tmem_ld32(acc_tm + 32 * c, ov);
        tmem_ld_wait();
        reg_fence32(ov);
        if (key < p.T) store_row32(dst + 32 * c, ov);
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
    polar_bwd_dq_kernel(const __grid_constant__ TileMaps m, const BwdTcParams p) {
  using L = Layout<D, false>;
  constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 384;  // dP buffers at 128 and 256
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + L::kBarOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // heads in L2-sized groups (their streamed K and V stay in L2), heaviest
  // query tiles (most key tiles) first within a group
  const int full = p.n_t * p.head_group;
  const int grp = (int)(blockIdx.x / full);
  const int rem = (int)blockIdx.x - grp * full;
  const int hg = min(p.head_group, p.BH - grp * p.head_group);
  const int qt = p.n_t - 1 - rem / hg;
  const int bh = grp * p.head_group + rem % hg;
  const int nk = qt + 1;  // key tiles 0 .. qt

  if (threadIdx.x == 0) setup_barriers(bars, L::kNSA, L::kNSB);
  if (warp == kWarpMMA) tmem_alloc(&bars->tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  volatile int* abort_flag = &bars->abort_flag;
  auto stage_k = [&](int j) { return smem + L::kRingA + (j % L::kNSA) * L::kStageA; };
  auto stage_v = [&](int j) { return smem + L::kRingB + (j % L::kNSB) * L::kStageB; };

  if (warp == kWarpTMA) {
    // the whole warp; one elected lane issues the copies
    produce<D, false>(smem, bars, &m.q, &m.da, kTile * qt, &m.k, &m.v, 0, nk, bh, p, abort_flag);
  } else if (warp == kWarpMMA) {
    // whole warp: uniform waits and descriptors, one elected lane issues
    {
      constexpr uint32_t kIdS = idesc_bf16_f32(128, kTile, 0, 0);
      constexpr uint32_t kIdAcc = idesc_bf16_f32(128, D, 0, 1);
      const uint64_t aq = smem_desc_sw128(smem_u32(smem + L::kR0), 16, 1024);
      const uint64_t ad = smem_desc_sw128(smem_u32(smem + L::kR1), 16, 1024);
      const uint32_t lbo_mn = D == 128 ? L::kAtom : 0;
      bool ok = mbar_wait_warp(&bars->res_full, 0, abort_flag, p.status);
      bool any = false;
      auto issue_s = [&](int j) -> bool {  // S = Q K^T
        if (!mbar_wait_warp(&bars->full_a[j % L::kNSA], (uint32_t)(j / L::kNSA) & 1, abort_flag,
                            p.status))
          return false;
        tc_fence_after();
        const uint64_t bk = smem_desc_sw128(smem_u32(stage_k(j)), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ss_warp(tmem + kColS, aq + kstep(kk), bk + kstep(kk), kIdS, kk > 0);
        umma_commit_warp(&bars->s_full[0]);
        any = true;
        return true;
      };
      auto issue_dp = [&](int j) -> bool {  // dP = dA V^T into buffer j & 1
        if (!mbar_wait_warp(&bars->full_b[j % L::kNSB], (uint32_t)(j / L::kNSB) & 1, abort_flag,
                            p.status))
          return false;
        tc_fence_after();
        const uint64_t bv = smem_desc_sw128(smem_u32(stage_v(j)), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ss_warp(tmem + kColDP + 128 * (j & 1), ad + kstep(kk), bv + kstep(kk), kIdS, kk > 0);
        umma_commit_warp(&bars->dp_full[j & 1]);
        umma_commit_warp(&bars->empty_b[j % L::kNSB]);
        any = true;
        return true;
      };
      if (ok) ok = issue_s(0);
      if (ok) ok = issue_dp(0);
      if (ok && nk > 1) ok = issue_dp(1);
      for (int j = 0; j < nk && ok; ++j) {
        ok = mbar_wait_warp(&bars->pa, (uint32_t)j & 1, abort_flag, p.status);
        if (!ok) break;
        tc_fence_after();
        if (j + 1 < nk) ok = issue_s(j + 1);  // S was read by the elementwise step j
        if (!ok) break;
        // dQ += dS' K, dS' in the dP buffer of step j
        const uint64_t bk = smem_desc_sw128(smem_u32(stage_k(j)), lbo_mn, 1024);
        const uint32_t ds_col = kColDP + 128 * (j & 1);
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          umma_ts_warp(tmem + kColDQ, tmem + ds_col + a_col(kk), bk + (uint64_t)(kk * (2048 >> 4)),
                       kIdAcc, (j > 0 || kk > 0) ? 1u : 0u);
        umma_commit_warp(&bars->empty_a[j % L::kNSA]);
        if (j + 2 < nk) ok = issue_dp(j + 2);  // over dS' of step j: ordered after the dQ MMAs
      }
      if (ok) umma_commit_warp(&bars->acc_full);
      if (!ok && any) {
        volatile int never = 0;
        umma_commit_warp(&bars->drain);
        __syncwarp();
        mbar_wait(&bars->drain, 0, &never, p.status, kWaitLimitCycles / 4);
        __syncwarp();
      }
    }
  } else if (warp < 8) {
    const int wg = warp >> 2;  // key columns 64 wg .. 64 wg + 63 of each step
    const int r = threadIdx.x & 127;
    const int row = qt * kTile + r;
    const bool valid = row < p.T;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t s_tm = tmem + lane_base + kColS + 64 * wg;
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
    for (int j = 0; j < nk && ok; ++j) {
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->s_full[0], (uint32_t)j & 1, abort_flag, p.status));
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bars->dp_full[j & 1], (uint32_t)(j >> 1) & 1,
                                                    abort_flag, p.status));
      if (!ok) break;
      tc_fence_after();
      const uint32_t dp_tm = tmem + lane_base + kColDP + 128 * (j & 1) + 64 * wg;
      const int k_first = j * kTile + 64 * wg;
      const bool masked = j == qt;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t sv[32], dv[32], dsk[16];
        tmem_ld32(s_tm + 32 * c, sv);
        tmem_ld32(dp_tm + 32 * c, dv);
        tmem_ld_wait();
        reg_fence32(sv);
        reg_fence32(dv);
        if (masked)
          chunk_ds<true>(sv, dv, cl2p, nlse2p, coefp, cmdcp, ecp, row, k_first + 32 * c, dsk);
        else
          chunk_ds<false>(sv, dv, cl2p, nlse2p, coefp, cmdcp, ecp, row, k_first + 32 * c, dsk);
        tmem_st16(dp_tm + 16 * c, dsk);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->pa);
    }
    // epilogue: dq = acc + qfloor q; warpgroup w writes columns [w D/2, (w+1) D/2)
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bars->acc_full, 0, abort_flag, p.status));
    if (ok) {
      tc_fence_after();
      const size_t roff = ((size_t)bh * p.T + (size_t)(valid ? row : 0)) * D;
#pragma unroll 1
      for (int c = wg * (D / 64); c < (wg + 1) * (D / 64); ++c) {
        uint32_t ov[32];
        tmem_ld32(tmem + lane_base + kColDQ + 32 * c, ov);
        tmem_ld_wait();
        reg_fence32(ov);
        if (valid) {
          const uint4* qp = reinterpret_cast<const uint4*>(p.q + roff + 32 * c);
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            const uint4 qu = __ldg(qp + g);
            const uint32_t qw[4] = {qu.x, qu.y, qu.z, qu.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              ov[8 * g + 2 * e] = __float_as_uint(
                  fmaf(qfloor, __uint_as_float(qw[e] << 16), __uint_as_float(ov[8 * g + 2 * e])));
              ov[8 * g + 2 * e + 1] = __float_as_uint(fmaf(
                  qfloor, __uint_as_float(qw[e] & 0xFFFF0000u), __uint_as_float(ov[8 * g + 2 * e + 1])));
            }
          }
          store_row32(p.dq + roff + 32 * c, ov);
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

// ============================================== row pass from saved rows ==
// Alternative to the forward kernel's backward mode when the forward kept
// its outputs: per row the direction is recovered from them,
//   count = conf tanh(ln n_eff / kappa),  u = out - count w - mem,
//   a = max(|a|, eps) u   (|a| and logsumexp from the saved stats),
// and the row gradient is formed as in the backward mode (same records,
// dA in bf16, count * g partials).  One CTA of four warps per 32-row block,
// eight rows per warp (more rows in flight than one warp per block); lane
// owns D / 32 consecutive columns.  Memory-bound: ~5 d bf16 values per row.
template <int D>
__global__ void __launch_bounds__(128)
    polar_bwd_rows_saved_kernel(const __nv_bfloat16* __restrict__ q,
                                const __nv_bfloat16* __restrict__ out,
                                const __nv_bfloat16* __restrict__ mem,
                                const __nv_bfloat16* __restrict__ dout,
                                const float* __restrict__ w_count, const float* __restrict__ n_eff,
                                const float* __restrict__ conf, const float* __restrict__ stats,
                                __nv_bfloat16* __restrict__ da, float* __restrict__ rows,
                                float* __restrict__ dw_part, int BH, int H, int T, int nblk,
                                int tpad, polar_consts_t c) {
  constexpr int E = D / 32;
  __shared__ float red[4][D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = (int)(blockIdx.x / nblk), blk = (int)(blockIdx.x % nblk);
  const int h = bh % H;
  float wv[E], dw[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    wv[e] = __ldg(w_count + (size_t)h * D + lane * E + e);
    dw[e] = 0.f;
  }
  auto unpack = [](const __nv_bfloat16* p, float (&v)[E]) {
    if (E == 4) {
      const uint2 x = __ldg(reinterpret_cast<const uint2*>(p));
      v[0] = __uint_as_float(x.x << 16);
      v[1 % E] = __uint_as_float(x.x & 0xFFFF0000u);
      v[2 % E] = __uint_as_float(x.y << 16);
      v[3 % E] = __uint_as_float(x.y & 0xFFFF0000u);
    } else {
      const uint32_t x = __ldg(reinterpret_cast<const unsigned int*>(p));
      v[0] = __uint_as_float(x << 16);
      v[1 % E] = __uint_as_float(x & 0xFFFF0000u);
    }
  };
  auto wsum = [](float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
  };
  // warp w takes rows 8 w .. 8 w + 7 of the 32-row block
  const int r_end = min(8 * warp + 8, T - 32 * blk);
#pragma unroll 1
  for (int r = 8 * warp; r < r_end; ++r) {
    const int row = 32 * blk + r;
    const size_t ri = (size_t)bh * T + row;
    const size_t off = ri * D + lane * E;
    float ov[E], mv[E], gv[E], qv[E];
    unpack(out + off, ov);
    unpack(mem + off, mv);
    unpack(dout + off, gv);
    unpack(q + off, qv);
    const float ne = __ldg(n_eff + ri), cf = __ldg(conf + ri);
    const float2 st = __ldg(reinterpret_cast<const float2*>(stats) + ri);  // lse, |a|
    const float n = (float)(row + 1);
    const float coef = polar_tau(n, c.log_t0) * rsqrtf((float)D);
    const float tt = tanhf(logf(ne) / c.kappa);
    const float count = cf * tt;
    float u[E], ug = 0.f, gw = 0.f, qsq = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      u[e] = ov[e] - fmaf(count, wv[e], mv[e]);
      ug = fmaf(u[e], gv[e], ug);
      gw = fmaf(gv[e], wv[e], gw);
      qsq = fmaf(qv[e], qv[e], qsq);
      dw[e] = fmaf(count, gv[e], dw[e]);
    }
    ug = wsum(ug);
    gw = wsum(gw);
    qsq = wsum(qsq);
    const bool big = st.y > c.eps;
    const float den = big ? st.y : c.eps;  // a = den * u
    const float inv = 1.0f / den;
    float dd = 0.f;
    uint32_t dk[(E + 1) / 2];
#pragma unroll
    for (int e = 0; e < E; e += 2) {
      const float d0 = big ? (gv[e] - u[e] * ug) * inv : gv[e] * inv;
      const float d1 = big ? (gv[e + 1] - u[e + 1] * ug) * inv : gv[e + 1] * inv;
      dk[e / 2] = pack_bf16x2(d0, d1);
      dd = fmaf(den * u[e], __uint_as_float(dk[e / 2] << 16), dd);
      dd = fmaf(den * u[e + 1], __uint_as_float(dk[e / 2] & 0xFFFF0000u), dd);
    }
    dd = wsum(dd);
    if (E == 4)
      *reinterpret_cast<uint2*>(da + off) = make_uint2(dk[0], dk[1 % ((E + 1) / 2)]);
    else
      *reinterpret_cast<uint32_t*>(da + off) = dk[0];
    if (lane == 0) {
      const float q2n = 1.0f / ne;
      const float dq2 = -gw * cf * (1.0f - tt * tt) / (c.kappa * q2n);
      const float dlse = gw * tt * cf * (1.0f - cf);
      const float cc = dlse - 2.0f * dq2 * q2n, ee = 2.0f * dq2;
      const float qn = sqrtf(qsq);
      const float f = polar_floor_factor(n, c.floor_order);
      const float sig_per_q = coef * c.sigma_k;
      rows[grad_row_index(bh, tpad, row, kGCl2)] = coef * 1.4426950408889634f;
      rows[grad_row_index(bh, tpad, row, kGNLse2)] = -st.x * 1.4426950408889634f;
      rows[grad_row_index(bh, tpad, row, kGCoef)] = coef;
      rows[grad_row_index(bh, tpad, row, kGCmDc)] = coef * (cc - dd);
      rows[grad_row_index(bh, tpad, row, kGEc)] = coef * ee;
      rows[grad_row_index(bh, tpad, row, kGQFloor)] = qn > 0.f ? -dlse * sig_per_q * f / qn : 0.f;
      rows[grad_row_index(bh, tpad, row, kGCount)] = count;
    }
  }
  // the block's count * g partial: the four warps' sums, added in warp order
#pragma unroll
  for (int e = 0; e < E; ++e) red[warp][lane * E + e] = dw[e];
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int x = lane * E + e;
      dw_part[((size_t)bh * nblk + blk) * D + x] = ((red[0][x] + red[1][x]) + red[2][x]) + red[3][x];
    }
  }
}

template <int D>
cudaError_t launch_rows_saved(const BwdArgs& a, const SavedRows& sv, const BwdTcLayout& w,
                              cudaStream_t s) {
  const int BH = a.B * a.H, nblk = (a.T + 31) / 32;
  const long long blocks = (long long)BH * nblk;  // one CTA per 32-row block
  polar_bwd_rows_saved_kernel<D><<<(unsigned)blocks, 128, 0, s>>>(
      static_cast<const __nv_bfloat16*>(a.q), static_cast<const __nv_bfloat16*>(sv.out),
      static_cast<const __nv_bfloat16*>(sv.mem), static_cast<const __nv_bfloat16*>(a.dout),
      a.w_count, sv.n_eff, sv.conf, sv.stats, static_cast<__nv_bfloat16*>(w.da), w.rows,
      w.dw_part, BH, a.H, a.T, nblk, grad_rows_tpad(a.T), a.c);
  return cudaGetLastError();
}

// A second stream per device for the dQ kernel: the dK/dV and dQ kernels
// only read the workspace and write disjoint outputs, so running them side
// by side lets each fill the SMs the other's last wave leaves idle.
struct SideStream {
  bool ready = false;
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
std::mutex g_side_mutex;
SideStream g_side[64];

cudaError_t side_init(SideStream& ss) {
  if (ss.ready) return cudaSuccess;
  cudaError_t e = cudaStreamCreateWithFlags(&ss.s, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming);
  ss.ready = e == cudaSuccess;
  return e;
}

template <int D>
cudaError_t launch_tiles(const BwdArgs& a, const BwdTcLayout& w, const TileMaps& maps,
                         cudaStream_t s) {
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
  p.head_group = l2_head_group(p.BH, 4.0 * (double)a.T * D);  // two [T, D] bf16 streams
  const unsigned grid = (unsigned)((long long)p.n_t * p.BH);
  constexpr int smem_kv = Layout<D, true>::kSmemBytes, smem_q = Layout<D, false>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(polar_bwd_dkdv_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem_kv);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(polar_bwd_dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem_q);
  if (e != cudaSuccess) return e;
  int dev = 0;
  const bool have_dev = cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < 64;
  std::unique_lock<std::mutex> lock(g_side_mutex);
  SideStream* ss = have_dev && side_init(g_side[dev]) == cudaSuccess ? &g_side[dev] : nullptr;
  if (!ss) lock.unlock();
  cudaStream_t sq = s;
  if (ss) {
    // dQ on the side stream, after everything already on s
    if ((e = cudaEventRecord(ss->fork, s)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(ss->s, ss->fork, 0)) != cudaSuccess) return e;
    sq = ss->s;
  }
  polar_bwd_dkdv_kernel<D><<<grid, kThreads, smem_kv, s>>>(maps, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  polar_bwd_dq_kernel<D><<<grid, kThreads, smem_q, sq>>>(maps, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (ss) {
    // s continues only after dQ
    if ((e = cudaEventRecord(ss->join, ss->s)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(s, ss->join, 0)) != cudaSuccess) return e;
  }
  const int nblk = (a.T + 31) / 32;
  polar_bwd_dw_reduce_kernel<D><<<dim3(a.H, D / 32), 256, 0, s>>>(w.dw_part, a.dw, a.B, a.H, nblk);
  return cudaGetLastError();
}

}  // namespace

BwdTcLayout bwd_tc_layout(void* workspace, int B, int H, int T, int d) {
  const size_t rows = (size_t)B * H * T;
  const size_t rec_floats = grad_rows_floats((size_t)B * H, T);
  BwdTcLayout w;
  uint8_t* base = static_cast<uint8_t*>(workspace);
  w.da = base;
  w.rows = reinterpret_cast<float*>(base + rows * d * 2);
  w.dw_part = w.rows + rec_floats;
  w.bytes = rows * d * 2 + rec_floats * 4 + (size_t)B * H * ((T + 31) / 32) * d * 4;
  return w;
}

cudaError_t launch_bwd_rows_saved(const BwdArgs& a, const SavedRows& sv, const BwdTcLayout& w,
                                  cudaStream_t s) {
  return a.d == 64 ? launch_rows_saved<64>(a, sv, w, s) : launch_rows_saved<128>(a, sv, w, s);
}

cudaError_t launch_bwd_tc(const BwdArgs& a, const BwdTcLayout& w, const CUtensorMap* maps,
                          cudaStream_t s) {
  TileMaps m;
  m.q = maps[0];
  m.k = maps[1];
  m.v = maps[2];
  m.da = maps[3];
  return a.d == 64 ? launch_tiles<64>(a, w, m, s) : launch_tiles<128>(a, w, m, s);
}

}  // namespace polar
