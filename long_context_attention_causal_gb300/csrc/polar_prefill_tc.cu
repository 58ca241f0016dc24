// Causal Polar Attention prefill, bf16, on the sm_103a tensor cores.
//
// "ATMA: Length-Invariant Language Modeling via Polar Attention and
// Gated-Delta Compression Memory", §2.2 (fused Polar Attention kernel): the
// participation ratio is computed online with streaming accumulators and
// squared correction factors, in O(block) memory; §2.1 gives the three
// output channels.  This kernel is a new design for Blackwell:
//
//   * one CTA owns two 128-row query tiles of one (b, h) (rows 256p..256p+255)
//     and streams the causal key/value tiles 0..qt through a 2-stage shared
//     memory ring filled by TMA (128-byte swizzle, 3-D tensor maps so rows
//     past T read as zeros);
//   * one thread issues tcgen05.mma: S_t = Q_t K_j^T into TMEM (fp32), then,
//     once the softmax warpgroup has written P_t (bf16) over S_t in TMEM,
//     O_t += P_t V_j with A read from TMEM;
//   * a softmax warpgroup per query tile (thread r <-> row r <-> TMEM lane r)
//     applies the length temperature, the causal mask on the diagonal tile,
//     and carries the running reference max m, l = sum p and Q2 = sum p^2;
//     when the max grows by more than 2^8 it rescales l by a, Q2 by a^2 and
//     O (in TMEM) by a, a = 2^(m_old - m_new) (squared correction factor);
//   * the same warpgroup runs the epilogue: n_eff = l^2/Q2, null-floor gate,
//     tanh-log count, unit-sphere direction, + memory, bf16 stores.
//
// Warp roles (384 threads): warps 0-3 softmax of tile 0, warps 4-7 softmax
// of tile 1, warp 8 TMA producer, warp 9 MMA issuer and TMEM owner, warps
// 10-11 idle (the register file is granted per warpgroup).
// TMEM (512 columns): tile t uses S/P at columns 256t..256t+127 and O at
// 256t+128..256t+128+D-1.
//
// Backward mode (template flag): the same streaming pass, but the epilogue
// turns the row's final state and the upstream gradient g into the inputs
// of the backward tile kernels instead of the output: dA (bf16), the 8-float
// row record (polar_grad.cuh) and per-32-row partial sums of count * g.
#include "polar_device.cuh"
#include "polar_grad.cuh"
#include "polar_internal.h"

namespace polar {

namespace {

constexpr int kBM = 128;  // query rows per tile
constexpr int kBN = 128;  // keys per tile
constexpr int kNQ = 2;    // query tiles per CTA
constexpr int kNSMax = 4; // ring stages (K and V each), upper bound
constexpr int kThreads = 384;  // 3 warpgroups: registers are granted per 4 warps
constexpr int kWarpTMA = 8;
constexpr int kWarpMMA = 9;
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct Layout {
  // Ring depths.  d = 128: 2 K + 2 V stages (a third K stage fits in the
  // 227 KB but measured slower); d = 64: 4 + 4.  Shared memory stays above
  // half of the SM's, so one CTA per SM holds the 512 TMEM columns.
  static constexpr int kNSK = D == 128 ? 2 : 4;
  static constexpr int kNSV = kNSK;
  static constexpr int kTileBytes = kBM * D * 2;  // 128 x D bf16
  static constexpr int kHalfBytes = kBM * 128;    // one 64-column swizzle atom
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kNQ * kTileBytes;
  static constexpr int kVOff = kKOff + kNSK * kTileBytes;
  static constexpr int kBarOff = kVOff + kNSV * kTileBytes;
  static constexpr int kSmemBytes = kBarOff + 256 + 1024;  // + align slack
  static_assert(kSmemBytes <= 232448, "shared memory");
  static_assert(kSmemBytes > 232448 / 2, "one CTA per SM (512 TMEM columns)");
  static_assert(kNSK == kNSV, "K and V stages are released together");
};

// Step j of the key loop consumes V_j (for P V_j) and K_{j+1} (for the next
// S); both are released when the step's MMAs are done.  One barrier per
// ring stage therefore signals "inputs of step j landed" (kv_full) and one
// "step j done" (step_done): one probe and one commit per step.  K_0, used
// before the loop, has its own pair.
struct Bars {
  uint64_t q_full;
  uint64_t k0_full, k0_empty;
  uint64_t kv_full[kNSMax], step_done[kNSMax];
  uint64_t s_full[kNQ];  // per TMEM S region (not per tile; see s_region)
  uint64_t p_full[kNQ];  // per TMEM S region
  uint64_t o_final[kNQ];
  uint64_t pv_bar[kNQ];  // PV done, one phase per one-tile step (see s_region)
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

struct TcParams {
  const __nv_bfloat16* mem;
  const float* w_count;
  __nv_bfloat16* out;
  float* n_eff;
  float* conf;
  float* stats;  // optional [BH, T, 2]: logsumexp, |a| (for the backward)
  int* status;  // device status word (bounded-wait timeouts)
  int H, T, BH, n_pairs, n_qt;
  int head_group;  // multi-wave order: heads per group (see the CTA order below)
  polar_consts_t c;
  // backward mode only
  const __nv_bfloat16* dout;  // g, [BH, T, D]
  __nv_bfloat16* da;          // [BH, T, D]
  float* grad_rows;           // [BH, tpad, kGRowFloats], pair-interleaved
  float* dw_part;             // [BH, ceil(T / 32), D]
};

// The 128 threads of query tile t's softmax warpgroup meet at named barrier
// 1 + t; returns true iff `ok` holds in every one of them.  Every thread of
// the warpgroup reaches it, whatever its own `ok`, so an aborted warp cannot
// leave the others waiting.
__device__ __forceinline__ bool tile_bar_and(int t, bool ok) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %2, 0;\n\t"
      "bar.red.and.pred po, %1, 128, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"(1 + t), "r"((uint32_t)ok)
      : "memory");
  return r != 0;
}

// TMA tile store shared -> global (bulk-group completion); rows past the
// tensor's extent are not written.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* smem_src, int x,
                                             int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(smem_src)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// Commit this thread's TMA stores and wait until they have read their
// shared-memory source (the buffer may be released after this returns).
__device__ __forceinline__ void tma_store_commit_wait_read() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA) reads of them.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Sum of v[c] over the 32 lanes of the warp for every c: lane c receives the
// total of column c (five exchange rounds, 31 shuffles).
__device__ __forceinline__ float warp_reduce_scatter32(float (&v)[32], int lane) {
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
    const bool upper = (lane & w) != 0;
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const float send = upper ? v[i] : v[i + w];
      const float keep = upper ? v[i + w] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
    }
  }
  return v[0];
}

// Backward-mode epilogue of one row (thread = row = TMEM lane).  With
// a = acc / l, u = a / max(|a|, eps), g the upstream gradient and w the
// head's count direction:
//   da   = (g - u (u.g)) / |a|   (|a| > eps),  g / eps otherwise
//   D    = a . da (with da rounded to bf16, as the tile kernels read it)
//   dQ2  = -(g.w) conf (1 - T^2) / (kappa Q2),  dlse = (g.w) T conf (1 - conf)
//   C    = dlse - 2 dQ2 Q2,  E = 2 dQ2,  T = tanh(-ln Q2 / kappa)
template <int D>
__device__ __forceinline__ void bwd_row_epilogue(const TcParams& p, uint32_t o_tm, float m_log2,
                                                 float l, float q2, float acc_sq, float q_sq,
                                                 float n, int row, int bh, int h, int lane) {
  const bool valid = row < p.T;
  const float coef = polar_tau(n, p.c.log_t0) * rsqrtf((float)D);
  const float lse = m_log2 * kLn2 + logf(l);
  const float q2n = q2 / (l * l);
  const float an = sqrtf(acc_sq) / l;
  const float qn = sqrtf(q_sq);
  const float f = polar_floor_factor(n, p.c.floor_order);
  const float sig_per_q = coef * p.c.sigma_k;
  const float cf = 1.0f / (1.0f + expf(sig_per_q * qn * f - lse));
  const float tt = tanhf(-logf(q2n) / p.c.kappa);
  const float count = cf * tt;
  const bool big = an > p.c.eps;
  const float inv = 1.0f / (big ? an : p.c.eps);
  const float su = inv / l;  // u = acc * su
  const size_t roff = ((size_t)bh * p.T + (size_t)(valid ? row : 0)) * D;
  const uint4* gp = reinterpret_cast<const uint4*>(p.dout + roff);
  const float4* wp = reinterpret_cast<const float4*>(p.w_count + (size_t)h * D);
  // pass 1: acc . g and g . w
  float ag = 0.f, gw = 0.f;
#pragma unroll 1
  for (int c = 0; c < D / 32; ++c) {
    uint32_t ov[32];
    tmem_ld32(o_tm + 32 * c, ov);
    tmem_ld_wait();
    reg_fence32(ov);
    if (valid) {
#pragma unroll
      for (int g4 = 0; g4 < 4; ++g4) {
        const uint4 gu = __ldg(gp + 4 * c + g4);
        const float4 w0 = __ldg(wp + 8 * c + 2 * g4), w1 = __ldg(wp + 8 * c + 2 * g4 + 1);
        const float wf[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
        const uint32_t gw4[4] = {gu.x, gu.y, gu.z, gu.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float g0 = __uint_as_float(gw4[e] << 16);
          const float g1 = __uint_as_float(gw4[e] & 0xFFFF0000u);
          ag = fmaf(__uint_as_float(ov[8 * g4 + 2 * e]), g0, ag);
          ag = fmaf(__uint_as_float(ov[8 * g4 + 2 * e + 1]), g1, ag);
          gw = fmaf(g0, wf[2 * e], gw);
          gw = fmaf(g1, wf[2 * e + 1], gw);
        }
      }
    }
  }
  const float ug = ag * su;  // u . g
  // pass 2: da (bf16), D, and the warp's partial of count * g
  float dd = 0.f;
  const int blk = row >> 5;  // the same for the 32 rows of this warp
  const bool warp_live = (row - lane) < p.T;
  const int nblk = (p.T + 31) >> 5;
#pragma unroll 1
  for (int c = 0; c < D / 32; ++c) {
    uint32_t ov[32];
    tmem_ld32(o_tm + 32 * c, ov);
    tmem_ld_wait();
    reg_fence32(ov);
    float gv[32];
#pragma unroll
    for (int g4 = 0; g4 < 4; ++g4) {
      const uint4 gu = valid ? __ldg(gp + 4 * c + g4) : make_uint4(0u, 0u, 0u, 0u);
      const uint32_t gw4[4] = {gu.x, gu.y, gu.z, gu.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        gv[8 * g4 + 2 * e] = __uint_as_float(gw4[e] << 16);
        gv[8 * g4 + 2 * e + 1] = __uint_as_float(gw4[e] & 0xFFFF0000u);
      }
    }
    uint32_t dk[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const float a0 = __uint_as_float(ov[2 * e]), a1 = __uint_as_float(ov[2 * e + 1]);
      const float d0 = big ? (gv[2 * e] - a0 * su * ug) * inv : gv[2 * e] * inv;
      const float d1 = big ? (gv[2 * e + 1] - a1 * su * ug) * inv : gv[2 * e + 1] * inv;
      dk[e] = pack_bf16x2(d0, d1);
      dd = fmaf(a0, __uint_as_float(dk[e] << 16), dd);
      dd = fmaf(a1, __uint_as_float(dk[e] & 0xFFFF0000u), dd);
    }
    if (valid) {
      uint4* dp = reinterpret_cast<uint4*>(p.da + roff + 32 * c);
#pragma unroll
      for (int g4 = 0; g4 < 4; ++g4)
        dp[g4] = make_uint4(dk[4 * g4], dk[4 * g4 + 1], dk[4 * g4 + 2], dk[4 * g4 + 3]);
    }
#pragma unroll
    for (int e = 0; e < 32; ++e) gv[e] *= count;  // rows past T hold g = 0
    const float colsum = warp_reduce_scatter32(gv, lane);
    if (warp_live) p.dw_part[((size_t)bh * nblk + blk) * D + 32 * c + lane] = colsum;
  }
  if (!valid) return;
  dd /= l;  // a . da
  const float dq2 = -gw * cf * (1.0f - tt * tt) / (p.c.kappa * q2n);
  const float dlse = gw * tt * cf * (1.0f - cf);
  const float cc = dlse - 2.0f * dq2 * q2n;
  const float ee = 2.0f * dq2;
  const int tpad = grad_rows_tpad(p.T);
  float* rp = p.grad_rows;
  rp[grad_row_index(bh, tpad, row, kGCl2)] = coef * kLog2e;
  rp[grad_row_index(bh, tpad, row, kGNLse2)] = -lse * kLog2e;
  rp[grad_row_index(bh, tpad, row, kGCoef)] = coef;
  rp[grad_row_index(bh, tpad, row, kGCmDc)] = coef * (cc - dd);
  rp[grad_row_index(bh, tpad, row, kGEc)] = coef * ee;
  rp[grad_row_index(bh, tpad, row, kGQFloor)] = qn > 0.f ? -dlse * sig_per_q * f / qn : 0.f;
  rp[grad_row_index(bh, tpad, row, kGCount)] = count;
}

// kBal = false: CTA `pair` owns query tiles 2 pair and 2 pair + 1, heaviest
// pairs first.  kBal = true (all CTAs fit in one wave, where the heaviest
// CTA alone sets the time): tiles pair and n_qt - 1 - pair, so every CTA
// streams about the same keys, and the long tile's one-tile steps use the
// short tile's idle S region as a second S buffer.
template <int D, bool kBwd, bool kBal>
__global__ void __launch_bounds__(kThreads, 1)
    polar_fwd_tc_kernel(const __grid_constant__ CUtensorMap map_q,
                        const __grid_constant__ CUtensorMap map_k,
                        const __grid_constant__ CUtensorMap map_v,
                        const __grid_constant__ CUtensorMap map_o,
                        const TcParams p) {
  using L = Layout<D>;
  constexpr int kNSK = L::kNSK;
  constexpr int kNSV = L::kNSV;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + L::kBarOff);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // heaviest query-tile pairs first (causal work grows with the pair index)
  // CTA order.  One wave: heaviest pairs first over all heads.  Several
  // waves: the (b, h) slices are taken head_group at a time, heaviest pairs
  // first within a group, so that the K and V the running CTAs stream (one
  // group's) stay in L2: keyscale_16k read 2.19 GB of DRAM per launch in a
  // global heaviest-first order and 0.55 GB (its inputs once) in groups of
  // 4 heads.  The host picks the group (launch_d).
  int pair, bh;
  if (kBal) {
    pair = p.n_pairs - 1 - (int)(blockIdx.x / p.BH);
    bh = (int)(blockIdx.x % p.BH);
  } else {
    const int full = p.n_pairs * p.head_group;
    const int g = (int)(blockIdx.x / full);
    const int rem = (int)blockIdx.x - g * full;
    const int hg = min(p.head_group, p.BH - g * p.head_group);
    pair = p.n_pairs - 1 - rem / hg;
    bh = g * p.head_group + rem % hg;
  }
  const int h = bh % p.H;
  int qt[kNQ], nkv[kNQ];
  int nkmax = 0;
  static_assert(kNQ == 2, "tile pairing");
  if (kBal) {
    qt[0] = pair;
    qt[1] = p.n_qt - 1 - pair;  // == pair for the middle tile of an odd count
  } else {
    qt[0] = 2 * pair;
    qt[1] = 2 * pair + 1;
  }
#pragma unroll
  for (int t = 0; t < kNQ; ++t) {
    nkv[t] = qt[t] < p.n_qt ? qt[t] + 1 : 0;
    if (t == 1 && qt[1] == qt[0]) nkv[1] = 0;
    nkmax = nkv[t] > nkmax ? nkv[t] : nkmax;
  }
  // Steps j >= js run the long tile tl alone.  From step js + 1 on, its S
  // alternates between its own TMEM region and the other tile's, which is
  // idle: S(j + 1) is then issued before PV(j) and computes while the
  // softmax of step j runs.
  const int tl = nkv[1] >= nkv[0] ? 1 : 0;
  const int js = nkv[1 - tl];
  // s_full[r] and p_full[r] belong to region r, one phase per S written
  // there, so the next phase of a barrier always needs its waiter first (a
  // per-tile barrier could complete S(j) and the early S(j + 1) before the
  // softmax looked, and a parity wait would then miss).  s_phase: the phase
  // of step j's S on its region's barriers (the short tile wrote js).
  auto s_region = [tl, js](int t, int j) -> int {
    return (kBal && t == tl && j > js && ((j - js) & 1)) ? 1 - t : t;
  };
  auto s_phase = [tl, js](int t, int j) -> uint32_t {
    return (kBal && t == tl && j > js) ? (uint32_t)(js + ((j - js) >> 1)) : (uint32_t)j;
  };

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->k0_full, 1);
    mbar_init(&bars->k0_empty, 1);
    for (int s = 0; s < kNSK; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->step_done[s], 1);
    }
    for (int t = 0; t < kNQ; ++t) {
      mbar_init(&bars->s_full[t], 1);
      // one arrival per softmax warp (lane 0, after the warp's stores):
      // 128 per-thread arrivals on one word serialise in shared memory
      mbar_init(&bars->p_full[t], kBM / 32);
      mbar_init(&bars->o_final[t], 1);
      mbar_init(&bars->pv_bar[t], 1);
    }
    mbar_init(&bars->drain, 1);
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kWarpMMA) tmem_alloc(&bars->tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  volatile int* abort_flag = &bars->abort_flag;

  if (warp == kWarpTMA) {
    // ------------------------------------------------------ TMA producer --
    // whole warp, one elected lane issuing (as the MMA issuer)
    {
      if (lane == 0) {
        tma_prefetch_desc(&map_q);
        tma_prefetch_desc(&map_k);
        tma_prefetch_desc(&map_v);
      }
      __syncwarp();
      int nact = 0;
      for (int t = 0; t < kNQ; ++t) nact += nkv[t] > 0;
      mbar_arrive_expect_tx_warp(&bars->q_full, nact * L::kTileBytes);
      for (int t = 0; t < kNQ; ++t) {
        if (nkv[t] == 0) continue;
        for (int hh = 0; hh < D / 64; ++hh)
          tma_load_3d_warp(smem + L::kQOff + t * L::kTileBytes + hh * L::kHalfBytes,
                      &map_q, &bars->q_full, 64 * hh, kBM * qt[t], bh);
      }
      // K_0 into K stage 0
      mbar_arrive_expect_tx_warp(&bars->k0_full, L::kTileBytes);
      for (int hh = 0; hh < D / 64; ++hh)
        tma_load_3d_warp(smem + L::kKOff + hh * L::kHalfBytes, &map_k, &bars->k0_full, 64 * hh, 0, bh);
      // step j: V_j into V stage j % NS, K_{j+1} into K stage (j + 1) % NS.
      // Both stages were last used by step j - NS (V_{j-NS}; K_{j+1-NS},
      // whose S was issued in step j - NS); for j = NS - 1 the K stage held
      // K_0, released before the loop.
      constexpr int NS = kNSK;
      int issued = 0;
      bool ok = true;
      for (int j = 0; j < nkmax && ok; ++j) {
        const int s = j % NS, sk = (j + 1) % NS;
        const bool k_next = j + 1 < nkmax;
        if (j == NS - 1) ok = mbar_wait_warp(&bars->k0_empty, 0, abort_flag, p.status);
        if (ok && j >= NS)
          ok = mbar_wait_warp(&bars->step_done[s], (uint32_t)(j / NS - 1) & 1, abort_flag,
                              p.status);
        if (!ok) break;
        mbar_arrive_expect_tx_warp(&bars->kv_full[s], (k_next ? 2 : 1) * L::kTileBytes);
        for (int hh = 0; hh < D / 64; ++hh)
          tma_load_3d_warp(smem + L::kVOff + s * L::kTileBytes + hh * L::kHalfBytes, &map_v,
                      &bars->kv_full[s], 64 * hh, kBN * j, bh);
        if (k_next)
          for (int hh = 0; hh < D / 64; ++hh)
            tma_load_3d_warp(smem + L::kKOff + sk * L::kTileBytes + hh * L::kHalfBytes, &map_k,
                        &bars->kv_full[s], 64 * hh, kBN * (j + 1), bh);
        issued = j + 1;
      }
      if (!ok) {
        // aborted: let the copies already issued land before the CTA exits
        volatile int never = 0;
        const long long lim = kWaitLimitCycles / 4;
        for (int j = issued - 1; j >= 0 && j >= issued - NS; --j)
          mbar_wait(&bars->kv_full[j % NS], (uint32_t)(j / NS) & 1, &never, p.status, lim);
        mbar_wait(&bars->k0_full, 0, &never, p.status, lim);
        mbar_wait(&bars->q_full, 0, &never, p.status, lim);
        __syncwarp();
      }
    }
  } else if (warp == kWarpMMA) {
    // ------------------------------------------------------- MMA issuer --
    // The whole warp runs the issue loop (its waits and descriptors are
    // warp-uniform) and one elected lane issues each product and commit.
    {
      constexpr uint32_t kIdescS = idesc_bf16_f32(kBM, kBN, 0, 0);
      constexpr uint32_t kIdescPV = idesc_bf16_f32(kBM, D, 0, 1);
      const uint32_t q_addr = smem_u32(smem + L::kQOff);
      const uint32_t k_addr = smem_u32(smem + L::kKOff);
      const uint32_t v_addr = smem_u32(smem + L::kVOff);
      bool ok = __all_sync(0xffffffffu, mbar_wait(&bars->q_full, 0, abort_flag, p.status));
      bool any_issued = false;
      // Descriptors are built once; a K step only moves the start address
      // (the low 14-bit field, in 16-byte units, never carries: shared
      // addresses stay below 256 KB).  Rebuilding them per MMA made the
      // single issuing thread, not the tensor core, the bottleneck.
      const uint64_t desc_q = smem_desc_sw128(q_addr, 16, 1024);
      const uint64_t desc_k = smem_desc_sw128(k_addr, 16, 1024);
      // V: MN-major, LBO = distance between the two 64-column atoms (d = 128)
      const uint64_t desc_v = smem_desc_sw128(v_addr, D == 128 ? L::kHalfBytes : 0, 1024);
      auto issue_s = [&](int t, int s, int r) {
        // S_t = Q_t K^T over D in steps of 16 (32 bytes inside the swizzle
        // row), into the S region r
        const uint64_t a0 = desc_q + (uint64_t)((t * L::kTileBytes) >> 4);
        const uint64_t b0 = desc_k + (uint64_t)((s * L::kTileBytes) >> 4);
        const uint32_t d_tm = tmem + 256 * r;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t off = (uint64_t)((kk >> 2) * (L::kHalfBytes >> 4) + (kk & 3) * 2);
          umma_ss_warp(d_tm, a0 + off, b0 + off, kIdescS, kk > 0);
        }
        umma_commit_warp(&bars->s_full[r]);
      };
      auto issue_pv = [&](int t, int s, int j, int r) {
        // O_t += P_t V over 128 keys in steps of 16: P in TMEM region r (8
        // columns per 16 bf16 keys), V MN-major (d contiguous), 2048 bytes
        // per 16 keys
        const uint64_t b0 = desc_v + (uint64_t)((s * L::kTileBytes) >> 4);
        const uint32_t o_tm = tmem + 256 * t + 128, p_tm = tmem + 256 * r;
        umma_ts_warp(o_tm, p_tm, b0, kIdescPV, j > 0 ? 1u : 0u);
#pragma unroll
        for (int kk = 1; kk < kBN / 16; ++kk)
          umma_ts_warp(o_tm, p_tm + kk * 8, b0 + (uint64_t)(kk * (2048 >> 4)), kIdescPV, 1u);
      };
      constexpr int NS = kNSK;
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bars->k0_full, 0, abort_flag, p.status));
      if (ok) {
        tc_fence_after();
        for (int t = 0; t < kNQ; ++t)
          if (nkv[t] > 0) issue_s(t, 0, t);
        umma_commit_warp(&bars->k0_empty);
        any_issued = true;
      }
      for (int j = 0; j < nkmax && ok; ++j) {
        const int s = j % NS;
        const int jn = j + 1, sn = jn % NS;
        ok = __all_sync(0xffffffffu,
                       mbar_wait(&bars->kv_full[s], (uint32_t)(j / NS) & 1, abort_flag, p.status));
        if (!ok) break;
        tc_fence_after();
        if (kBal && j >= js) {
          // the long tile alone: S(j + 1) into the other region first
          if (jn < nkv[tl]) issue_s(tl, sn, s_region(tl, jn));
          ok = __all_sync(0xffffffffu, mbar_wait(&bars->p_full[s_region(tl, j)],
                                                 s_phase(tl, j) & 1, abort_flag, p.status));
          if (!ok) break;
          tc_fence_after();
          issue_pv(tl, s, j, s_region(tl, j));
          if (j == nkv[tl] - 1) umma_commit_warp(&bars->o_final[tl]);
          umma_commit_warp(&bars->pv_bar[tl]);
        } else {
          for (int t = 0; t < kNQ && ok; ++t) {
            if (j >= nkv[t]) continue;
            ok = __all_sync(0xffffffffu,
                            mbar_wait(&bars->p_full[t], (uint32_t)j & 1, abort_flag, p.status));
            if (!ok) break;
            tc_fence_after();
            issue_pv(t, s, j, t);
            if (j == nkv[t] - 1) umma_commit_warp(&bars->o_final[t]);
            if (jn < nkv[t]) issue_s(t, sn, s_region(t, jn));
          }
        }
        if (!ok) break;
        umma_commit_warp(&bars->step_done[s]);
      }
      if (!ok && any_issued) {
        // aborted: wait for the MMAs in flight before TMEM is released
        volatile int never = 0;
        umma_commit_warp(&bars->drain);
        __syncwarp();
        mbar_wait(&bars->drain, 0, &never, p.status, kWaitLimitCycles / 4);
        __syncwarp();
      }
    }
  } else if (warp < 4 * kNQ) {
    // ------------------------------------------------- softmax + epilogue --
    const int t = warp >> 2;  // query tile of this warpgroup
    const int r = threadIdx.x & 127;
    const int row = qt[t] * kBM + r;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t o_tm = tmem + lane_base + 256 * t + 128;
    if (nkv[t] > 0) {
      bool ok = __all_sync(0xffffffffu, mbar_wait(&bars->q_full, 0, abort_flag, p.status));
      // |q|^2 of this row: the swizzle permutes 16-byte chunks inside the
      // row's 128-byte line, which leaves the sum of squares unchanged.
      // Rows are 128 bytes apart, so thread r reads chunk c ^ (r & 7) in
      // round c: eight consecutive rows then cover all 32 banks (chunk c of
      // every row put a warp's 32 reads on the same four banks).
      float q_sq = 0.f;
      if (ok) {
        for (int hh = 0; hh < D / 64; ++hh) {
          const uint4* line = reinterpret_cast<const uint4*>(
              smem + L::kQOff + t * L::kTileBytes + hh * L::kHalfBytes + r * 128);
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint4 u = line[c ^ (r & 7)];
            const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              float lo = __uint_as_float(w4[e] << 16);
              float hi = __uint_as_float(w4[e] & 0xFFFF0000u);
              q_sq = fmaf(lo, lo, q_sq);
              q_sq = fmaf(hi, hi, q_sq);
            }
          }
        }
      }
      const float n = (float)(row + 1);
      const float tau = polar_tau(n, p.c.log_t0);
      const float scale2 = tau * kLog2e * rsqrtf((float)D);  // log2 units
      float m_ref = -INFINITY, l = 0.f, q2 = 0.f;
      for (int j = 0; j < nkv[t] && ok; ++j) {
        const int sr = s_region(t, j);
        ok = __all_sync(0xffffffffu, mbar_wait(&bars->s_full[sr], s_phase(t, j) & 1, abort_flag,
                                               p.status));
        if (!ok) break;
        tc_fence_after();
        const uint32_t s_tm = tmem + lane_base + 256 * sr;
        uint32_t sv[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(s_tm + 32 * c, sv[c]);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 4; ++c) reg_fence32(sv[c]);
        if (j == qt[t]) {
          // diagonal tile: key column c is visible iff c <= r
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (32 * c + e > r) sv[c][e] = __float_as_uint(-INFINITY);
        }
        // row max: three-input max, two chains
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            mx0 = fmax3(mx0, __uint_as_float(sv[c][e]), __uint_as_float(sv[c][e + 1]));
            mx1 = fmax3(mx1, __uint_as_float(sv[c][e + 2]), __uint_as_float(sv[c][e + 3]));
          }
        const float mt = fmaxf(mx0, mx1) * scale2;
        // tcgen05.ld/st are warp-collective: the rescale decision is taken
        // per warp; rows that do not need it use a factor of 1
        const bool need = mt > m_ref + kRescaleThreshold;
        if (__any_sync(0xffffffffu, need)) {
          const float alpha = need ? ex2_approx(m_ref - mt) : 1.0f;  // 0 on tile 0
          l *= alpha;
          q2 *= alpha * alpha;  // squared correction factor
          if (j > 0) {
            // O already holds P V of earlier tiles.  Normally the MMA that
            // produced S_j was issued after them, so they are complete here;
            // an S issued ahead of PV(j - 1) (one-tile steps past js) waits
            // for that product's own barrier.
            if (kBal && t == tl && j > js)
              ok = __all_sync(0xffffffffu, mbar_wait(&bars->pv_bar[t], (uint32_t)(j - 1 - js) & 1,
                                                     abort_flag, p.status));
#pragma unroll 1
            for (int c = 0; c < D / 32 && ok; ++c) {
              uint32_t ov[32];
              tmem_ld32(o_tm + 32 * c, ov);
              tmem_ld_wait();
              reg_fence32(ov);
#pragma unroll
              for (int e = 0; e < 32; ++e)
                ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
              tmem_st32(o_tm + 32 * c, ov);
            }
          }
          if (need) m_ref = mt;
        }
        if (!ok) break;
        // P over S in place: keys 2c', 2c'+1 -> TMEM column c' (bf16x2),
        // stored 32 keys at a time so P never needs its own registers.
        // Pairs of keys share packed fp32 instructions; sum p and sum p^2
        // run in two packed accumulators each.
        const float2 sc2 = make_float2(scale2, scale2);
        const float2 nm2 = make_float2(-m_ref, -m_ref);
        float2 la = make_float2(0.f, 0.f), lb = la, qa = la, qb = la;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            const float2 x0 = ffma2(make_float2(__uint_as_float(sv[c][e]),
                                                __uint_as_float(sv[c][e + 1])), sc2, nm2);
            const float2 x1 = ffma2(make_float2(__uint_as_float(sv[c][e + 2]),
                                                __uint_as_float(sv[c][e + 3])), sc2, nm2);
            const float2 p0 = make_float2(ex2_approx(x0.x), ex2_approx(x0.y));
            const float2 p1 = make_float2(ex2_approx(x1.x), ex2_approx(x1.y));
            la = fadd2(la, p0);
            lb = fadd2(lb, p1);
            qa = ffma2(p0, p0, qa);
            qb = ffma2(p1, p1, qb);
            pk[e / 2] = pack_bf16x2(p0.x, p0.y);
            pk[e / 2 + 1] = pack_bf16x2(p1.x, p1.y);
          }
          tmem_st16(s_tm + 16 * c, pk);
        }
        l += (la.x + la.y) + (lb.x + lb.y);
        q2 += (qa.x + qa.y) + (qb.x + qb.y);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_full[sr]);
      }
      // the row's memory stream, loaded into registers while the last
      // products finish, so that its latency is off the epilogue's path
      uint4 mrow[kBwd ? 1 : D / 8];
      if constexpr (!kBwd) {
        if (ok && row < p.T) {
          const uint4* mp = reinterpret_cast<const uint4*>(p.mem + ((size_t)bh * p.T + row) * D);
#pragma unroll
          for (int i = 0; i < D / 8; ++i) mrow[i] = __ldg(mp + i);
        } else {
#pragma unroll
          for (int i = 0; i < D / 8; ++i) mrow[i] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bars->o_final[t], 0, abort_flag, p.status));
      if (ok) {
        tc_fence_after();
        float acc_sq = 0.f;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t ov[32];
          tmem_ld32(o_tm + 32 * c, ov);
          tmem_ld_wait();
          reg_fence32(ov);
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float a = __uint_as_float(ov[e]);
            acc_sq = fmaf(a, a, acc_sq);
          }
        }
        if constexpr (kBwd) {
          bwd_row_epilogue<D>(p, o_tm, m_ref, l, q2, acc_sq, q_sq, n, row, bh, h, lane);
        } else {
        const RowResult res =
            polar_finish(m_ref * kLn2, l, q2, acc_sq, q_sq, n, D, p.c);
        const bool valid = row < p.T;
        const float* wv = p.w_count + (size_t)h * D;
        // The output tile is staged in this tile's Q buffer (its last reader,
        // the final S product, is done: O is final) in the 128-byte-swizzle
        // layout of the tensor map, then written by one TMA store per 64
        // columns: whole rows, coalesced, and rows past T are clipped by the
        // map.  16-byte chunk ch of row r sits at r * 128 + ((ch ^ (r & 7)) << 4).
        uint8_t* stage = smem + L::kQOff + t * L::kTileBytes;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t ov[32];
          tmem_ld32(o_tm + 32 * c, ov);
          tmem_ld_wait();
          reg_fence32(ov);
          const float4* wp = reinterpret_cast<const float4*>(wv + 32 * c);
          uint8_t* line = stage + (c >> 1) * L::kHalfBytes + r * 128;
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            const uint4 mu = mrow[4 * c + g];
            const float4 w0 = __ldg(wp + 2 * g), w1 = __ldg(wp + 2 * g + 1);
            const float wf[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
            const uint32_t mw[4] = {mu.x, mu.y, mu.z, mu.w};
            uint32_t o4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float m0 = __uint_as_float(mw[e] << 16);
              const float m1 = __uint_as_float(mw[e] & 0xFFFF0000u);
              const float a0 = __uint_as_float(ov[8 * g + 2 * e]);
              const float a1 = __uint_as_float(ov[8 * g + 2 * e + 1]);
              const float y0 = fmaf(a0, res.scale_u, fmaf(res.count, wf[2 * e], m0));
              const float y1 = fmaf(a1, res.scale_u, fmaf(res.count, wf[2 * e + 1], m1));
              o4[e] = pack_bf16x2(y0, y1);
            }
            const int ch = (c & 1) * 4 + g;
            *reinterpret_cast<uint4*>(line + ((ch ^ (r & 7)) << 4)) =
                make_uint4(o4[0], o4[1], o4[2], o4[3]);
          }
        }
        fence_proxy_async_smem();
        if (valid) {
          p.n_eff[(size_t)bh * p.T + row] = res.n_eff;
          if (p.conf) p.conf[(size_t)bh * p.T + row] = res.conf;
          if (p.stats)
            *reinterpret_cast<float2*>(p.stats + 2 * ((size_t)bh * p.T + row)) =
                make_float2(m_ref * kLn2 + logf(l), sqrtf(acc_sq) / l);
        }
        }  // forward epilogue
      }
      if constexpr (!kBwd) {
        // the staged tile is complete once every warp of the group is
        if (tile_bar_and(t, ok) && r == 0) {
          const uint8_t* stage = smem + L::kQOff + t * L::kTileBytes;
          for (int hh = 0; hh < D / 64; ++hh)
            tma_store_3d(&map_o, stage + hh * L::kHalfBytes, 64 * hh, kBM * qt[t], bh);
          tma_store_commit_wait_read();
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

template <int D, bool kBwd>
cudaError_t launch_d(const FwdArgs& a, const CUtensorMap& mq, const CUtensorMap& mk,
                     const CUtensorMap& mv, const CUtensorMap& mo, cudaStream_t s) {
  using L = Layout<D>;
  TcParams p;
  p.mem = static_cast<const __nv_bfloat16*>(a.mem);
  p.w_count = a.w_count;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.n_eff = a.n_eff;
  p.conf = a.conf;
  p.stats = a.stats;
  p.H = a.H;
  p.T = a.T;
  p.BH = a.B * a.H;
  p.n_qt = (a.T + kBM - 1) / kBM;
  p.n_pairs = (p.n_qt + kNQ - 1) / kNQ;
  p.head_group = p.BH;
  p.c = a.c;
  p.status = a.status;
  p.dout = static_cast<const __nv_bfloat16*>(a.dout);
  p.da = static_cast<__nv_bfloat16*>(a.da);
  p.grad_rows = a.grad_rows;
  p.dw_part = a.dw_part;
  const long long blocks = (long long)p.n_pairs * p.BH;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const bool bal = sms > 0 && blocks <= sms;
  // Head group of the multi-wave order: the largest divisor of B*H whose
  // heads' K and V fit a third of L2 (whole groups, so no group is a short
  // tail), one head when a single head's do not.  Measured: keyscale_16k
  // (8 MiB per head) 4 heads, needles_64k (32 MiB) 1 head, T = 8192 with 32
  // heads (4 MiB) 8 heads were the fastest groupings.
  p.head_group = l2_head_group(p.BH, 4.0 * (double)a.T * D);  // K and V, bf16
  auto kern = bal ? polar_fwd_tc_kernel<D, kBwd, true> : polar_fwd_tc_kernel<D, kBwd, false>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemBytes);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)blocks, kThreads, L::kSmemBytes, s>>>(mq, mk, mv, mo, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_tc(const FwdArgs& a, const CUtensorMap& mq, const CUtensorMap& mk,
                          const CUtensorMap& mv, const CUtensorMap& mo, cudaStream_t s) {
  if (a.dout != nullptr)
    return a.d == 64 ? launch_d<64, true>(a, mq, mk, mv, mo, s)
                     : launch_d<128, true>(a, mq, mk, mv, mo, s);
  return a.d == 64 ? launch_d<64, false>(a, mq, mk, mv, mo, s)
                   : launch_d<128, false>(a, mq, mk, mv, mo, s);
}

}  // namespace polar
