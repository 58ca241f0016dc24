// Paged, grouped-query decode split kernel on the tensor cores (bf16).
//
// "ATMA: Length-Invariant Language Modeling via Polar Attention and
// Gated-Delta Compression Memory", §2.2: the decode kernel reads paged KV
// blocks directly and one KV read serves the query heads of a group.  With G
// query heads per KV row the scores of a stage of 64 keys form a 64 x G
// product, and the accumulator update a G x d one: both go to tcgen05 with
// the keys (then d) on the TMEM lanes and the G heads, padded to 16, on the
// columns, so no thread reduces a dot product:
//   S^T (128 x 16)  = K_stage (rows 0-63 the stage's keys) . Qpad^T  (SS, K-major)
//   O^T (d x 16)   += V_stage^T (d x 64) . P^T (64 x 16)            (SS, A MN-major)
// Softmax threads 0-63 (one per key of the stage) take the G scores of their key,
// the heads' stage maxima come from a block reduction, and each thread keeps
// its share of l = sum p and Q2 = sum p^2; P^T (bf16) is written to shared
// memory in the operand layout.  The running maximum of a head is moved only
// when a stage exceeds it by more than 2^8 (log2 units); then l, Q2 and the
// head's column of O^T are rescaled by a and a^2 (squared correction factor).
//
// Roles (192 threads, two CTAs per SM): warps 0-3 softmax and the record,
// warp 4 MMA issuer and TMEM owner, warp 5 TMA producer.  The cache
// [num_pages, Hkv, page, d] is read as a 2-D tensor [num_pages * Hkv * page,
// d]; a stage gathers 64 / frag pieces of frag = min(page, 64) rows, each the
// rows of one (page, KV head) slice.  A piece past the split or on a page index outside
// the pool is loaded from rows beyond the tensor (zeros, no DRAM read); the
// keys of a stage that are masked have their V rows zeroed before the
// product (rows past a sequence's end may hold anything, and 0 * NaN is not
// 0).  Records match polar_decode_paged_split_kernel's (merged by the same
// combine kernel).
#include "polar_device.cuh"
#include "polar_internal.h"

namespace polar {

namespace {

constexpr int kPK = kPagedTcStageKeys;  // keys per stage (64)
constexpr int kPM = 128;        // M of the score product (rows kPK.. unused)
constexpr int kPN = 16;         // head columns (G padded; N of both products)
constexpr int kPThreads = 192;  // 6 warps
constexpr int kPWarpMMA = 4;
constexpr int kPWarpTMA = 5;
constexpr int kPTable = 256;    // block-table entries cached per window
constexpr uint32_t kPTmemCols = 64;  // S^T x3 at 0 / 16 / 48, O^T at 32
constexpr float kPLog2e = 1.4426950408889634f;
constexpr float kPLn2 = 0.6931471805599453f;
constexpr float kPRescale = 8.0f;  // log2 units
// S^T / P^T buffers in flight: the softmax of stage j may write P^T once
// the product of stage j - kPB has read its buffer, and S^T(i) may be
// issued up to kPB - 1 stages ahead of the last P V product.
constexpr int kPB = 3;
// TMEM column of S^T buffer b (O^T sits at columns 32..47)
__device__ __forceinline__ uint32_t st_col(int b) { return b == 2 ? 48u : 16u * (uint32_t)b; }

template <int NS>
struct PMisc {
  uint64_t full[NS], empty[NS];
  uint64_t s_full[kPB], p_full[kPB], pv_done[kPB], drain;
  uint32_t valid[NS][kPK / 32];  // page-validity bits of each stage's rows
  int tab[kPTable];
  float red[2][4][8];            // per-warp stage maxima
  uint32_t up[2][4];             // per warp: a logit passed its head's reference
  float lred[4][8], qred[4][8];
  uint32_t tmem_base;
  int abort_flag;
};

template <int D>
struct PLayout {
  static constexpr int kNS = D == 128 ? 3 : 6;       // 96 KB of K and V per CTA
  static constexpr int kAtoms = D / 64;              // 64-column swizzle atoms
  static constexpr int kAtomBytes = kPK * 128;       // one atom of a stage tile
  static constexpr int kTile = kPK * D * 2;          // K (or V) bytes per stage
  static constexpr int kQOff = 0;                    // Qpad [atoms][16 rows][128 B]
  static constexpr int kQAtom = kPN * 128;
  static constexpr int kPOff = kQOff + kAtoms * kQAtom;  // P^T [kPB][16][128 B]
  static constexpr int kPBuf = (kPK / 64) * kPN * 128;
  static constexpr int kKOff = (kPOff + kPB * kPBuf + 1023) / 1024 * 1024;
  static constexpr int kVOff = kKOff + kNS * kTile;
  static constexpr int kMiscOff = kVOff + kNS * kTile;
  static constexpr int kSmemBytes = kMiscOff + (int)sizeof(PMisc<kNS>) + 1024;
  // two CTAs per SM: one CTA's ring fills and drains while the other streams
  static_assert(2 * (kSmemBytes + 1024) <= 233472, "two CTAs per SM");
};

__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "r"(taddr)
               : "memory");
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(
                   taddr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
               "r"(r[7])
               : "memory");
}

__device__ __forceinline__ void reg_fence8(uint32_t (&r)[8]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7])
               :
               : "memory");
}

// Non-blocking probe of a phase (the issuer polls two barriers at once).
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Generic-proxy shared-memory writes made visible to the tensor core.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void softmax_bar() {
  asm volatile("bar.sync 1, 128;" ::: "memory");
}

// Named barrier of the 128 softmax threads that also ANDs a predicate over
// them: after a failed (aborted) wait every thread leaves the loop at the
// same barrier, so no barrier is left short of arrivals.
__device__ __forceinline__ bool softmax_bar_and(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}

struct PagedTcParams {
  const __nv_bfloat16* q;
  const int* table;
  const int* lens;
  float* partials;
  int Hq, Hkv, max_pages, num_pages, page_shift, frag, rows_total;
  int splits, chunk;
  polar_consts_t c;
  int* status;
};

template <int D, int G>
__global__ void __launch_bounds__(kPThreads, 2)
    polar_decode_paged_tc_kernel(const __grid_constant__ CUtensorMap map_k,
                                 const __grid_constant__ CUtensorMap map_v,
                                 const PagedTcParams p) {
  using L = PLayout<D>;
  constexpr int NS = L::kNS;
  static_assert(G >= 1 && G <= 8, "group size");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  PMisc<NS>& ms = *reinterpret_cast<PMisc<NS>*>(smem + L::kMiscOff);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x / p.Hkv, hkv = blockIdx.x % p.Hkv;
  const int split = blockIdx.y;
  const int page = 1 << p.page_shift;
  int n = p.lens[b];
  const int n_max = min(p.splits * p.chunk, p.max_pages << p.page_shift);
  if (n < 1 || n > n_max) {
    if (threadIdx.x == 0 && split == 0) atomicExch(p.status, 3);
    n = n < 1 ? 0 : n_max;
  }
  const int k0 = split * p.chunk;
  const int k1 = min(k0 + p.chunk, n);
  const int nst = k1 > k0 ? (k1 - k0 + kPK - 1) / kPK : 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&ms.full[i], 1);
      mbar_init(&ms.empty[i], 1);
    }
    for (int i = 0; i < kPB; ++i) {
      mbar_init(&ms.s_full[i], 1);
      mbar_init(&ms.p_full[i], 128);
      mbar_init(&ms.pv_done[i], 1);
    }
    mbar_init(&ms.drain, 1);
    ms.abort_flag = 0;
    fence_barrier_init();
  }
  // Qpad (the group's G query rows, zero rows up to 16) in the K-major
  // 128-byte-swizzle operand layout; the P^T buffers zeroed (their rows
  // G..15 stay zero).
  for (int i = threadIdx.x; i < L::kAtoms * kPN * 8; i += kPThreads) {
    const int atom = i / (kPN * 8), rem = i % (kPN * 8);
    const int row = rem >> 3, ch = rem & 7;
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (row < G)
      val = *reinterpret_cast<const uint4*>(
          p.q + ((size_t)b * p.Hq + (size_t)hkv * G + row) * D + atom * 64 + ch * 8);
    *reinterpret_cast<uint4*>(smem + L::kQOff + atom * L::kQAtom + row * 128 +
                              ((ch ^ (row & 7)) << 4)) = val;
  }
  for (int i = threadIdx.x; i < kPB * L::kPBuf / 16; i += kPThreads)
    *reinterpret_cast<uint4*>(smem + L::kPOff + i * 16) = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  if (warp == kPWarpMMA) tmem_alloc(&ms.tmem_base, kPTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ms.tmem_base;
  volatile int* abort_flag = &ms.abort_flag;

  if (warp == kPWarpTMA) {
    // ------------------------------------------------------ TMA producer --
    const int* tb = p.table + (size_t)b * p.max_pages;
    const int frag = p.frag;
    const int nfrag = kPK / frag;
    if (lane == 0) {
      tma_prefetch_desc(&map_k);
      tma_prefetch_desc(&map_v);
    }
    int wbase = -kPTable;
    int issued = 0;
    bool ok = true;
    for (int st = 0; st < nst && ok; ++st) {
      const int slot = st % NS;
      if (st >= NS)
        ok = __all_sync(0xffffffffu, mbar_wait(&ms.empty[slot], (uint32_t)(st / NS - 1) & 1,
                                               abort_flag, p.status));
      if (!ok) break;
      const int key0 = k0 + st * kPK;
      const int key_end = min(key0 + kPK, k1);
      const int lp_last = (key_end - 1) >> p.page_shift;
      if (lp_last >= wbase + kPTable) {
        wbase = key0 >> p.page_shift;
        for (int i = lane; i < kPTable; i += 32)
          ms.tab[i] = wbase + i < p.max_pages ? tb[wbase + i] : -1;
        __syncwarp();
      }
      if (lane == 0) {
        uint32_t mask[kPK / 32] = {};
        int ys[kPK / 8];
        for (int f = 0; f < nfrag; ++f) {
          const int key = key0 + f * frag;
          int y = p.rows_total;  // past the tensor: zeros
          if (key < key_end) {
            const int pg = ms.tab[(key >> p.page_shift) - wbase];
            if (pg >= 0 && pg < p.num_pages) {
              y = (int)(((long long)pg * p.Hkv + hkv) * page + (key & (page - 1)));
              const int r0 = f * frag;
              if (frag >= 32) {
                for (int w = r0 >> 5; w < (r0 + frag) >> 5; ++w) mask[w] = 0xffffffffu;
              } else {
                mask[r0 >> 5] |= ((1u << frag) - 1u) << (r0 & 31);
              }
            } else {
              atomicExch(p.status, 3);
            }
          }
          ys[f] = y;
        }
        for (int w = 0; w < kPK / 32; ++w) ms.valid[slot][w] = mask[w];
        mbar_arrive_expect_tx(&ms.full[slot], 2u * L::kTile);
        uint8_t* kd = smem + L::kKOff + slot * L::kTile;
        uint8_t* vd = smem + L::kVOff + slot * L::kTile;
        for (int f = 0; f < nfrag; ++f) {
#pragma unroll
          for (int a = 0; a < L::kAtoms; ++a) {
            const int off = a * L::kAtomBytes + f * frag * 128;
            tma_load_2d(kd + off, &map_k, &ms.full[slot], a * 64, ys[f]);
            tma_load_2d(vd + off, &map_v, &ms.full[slot], a * 64, ys[f]);
          }
        }
      }
      __syncwarp();
      issued = st + 1;
    }
    if (!ok && lane == 0) {
      // aborted: let the copies already issued land before the CTA exits
      volatile int never = 0;
      for (int st = issued - 1; st >= 0 && st >= issued - NS; --st)
        mbar_wait(&ms.full[st % NS], (uint32_t)(st / NS) & 1, &never, p.status,
                  kWaitLimitCycles / 4);
    }
  } else if (warp == kPWarpMMA) {
    // ------------------------------------------------------- MMA issuer --
    // The whole warp runs the loop (its probes and descriptors are
    // warp-uniform) and one elected lane issues each product and commit.
    if (nst > 0) {
      // S^T: M = 128 rows of K; rows 64-127 read the next 8 KB of shared
      // memory (the following atom, stage or V ring: in bounds) and land in
      // TMEM lanes 64-127, which no softmax thread uses
      constexpr uint32_t kIdS = idesc_bf16_f32(kPM, kPN, 0, 0);
      constexpr uint32_t kIdPV = idesc_bf16_f32(128, kPN, 1, 0);
      const uint64_t desc_q = smem_desc_sw128(smem_u32(smem + L::kQOff), 16, 1024);
      const uint64_t desc_p = smem_desc_sw128(smem_u32(smem + L::kPOff), 16, 1024);
      const uint64_t desc_k = smem_desc_sw128(smem_u32(smem + L::kKOff), 16, 1024);
      // V^T: MN-major A; the d = 128 tile has two 64-row atoms along M.  At
      // d = 64 the leading offset 0 makes rows 64-127 of O^T a copy of rows
      // 0-63 (never read).
      const uint64_t desc_v =
          smem_desc_sw128(smem_u32(smem + L::kVOff), D == 128 ? L::kAtomBytes : 0, 1024);
      auto issue_s = [&](int j) {
        const int slot = j % NS;
        const uint64_t a0 = desc_k + (uint64_t)((slot * L::kTile) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t ka = (uint64_t)((kk >> 2) * (L::kAtomBytes >> 4) + (kk & 3) * 2);
          const uint64_t kb = (uint64_t)((kk >> 2) * (L::kQAtom >> 4) + (kk & 3) * 2);
          umma_ss_warp(tmem + st_col(j % kPB), a0 + ka, desc_q + kb, kIdS, kk > 0);
        }
        umma_commit_warp(&ms.s_full[j % kPB]);
      };
      auto issue_pv = [&](int j) {
        const int slot = j % NS;
        const uint64_t a0 = desc_v + (uint64_t)((slot * L::kTile) >> 4);
        const uint64_t b0 = desc_p + (uint64_t)(((j % kPB) * L::kPBuf) >> 4);
#pragma unroll
        for (int kk = 0; kk < kPK / 16; ++kk) {
          const uint64_t kb = (uint64_t)((kk >> 2) * ((kPN * 128) >> 4) + (kk & 3) * 2);
          umma_ss_warp(tmem + 32, a0 + (uint64_t)(kk * (2048 >> 4)), b0 + kb, kIdPV,
                  (j > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit_warp(&ms.pv_done[j % kPB]);
        umma_commit_warp(&ms.empty[slot]);
      };
      // Issue S(i) as soon as stage i has landed (and its S^T buffer is
      // free: i <= pv + 1) and PV(j) as soon as P(j) is written, whichever
      // comes first: a stage's slot is then released when its own product
      // is done, not after the next stage has arrived.
      int ns = 0, np = 0;
      bool ok = true, any = false;
      long long t_last = clock64();
      while (np < nst) {
        bool prog = false;
        if (ns < nst && ns <= np + kPB - 1 &&
            __all_sync(0xffffffffu, mbar_test(&ms.full[ns % NS], (uint32_t)(ns / NS) & 1))) {
          tc_fence_after();
          issue_s(ns);
          ++ns;
          any = prog = true;
        }
        if (np < ns &&
            __all_sync(0xffffffffu, mbar_test(&ms.p_full[np % kPB], (uint32_t)(np / kPB) & 1))) {
          tc_fence_after();
          issue_pv(np);
          ++np;
          prog = true;
        }
        if (prog) {
          t_last = clock64();
        } else if (__any_sync(0xffffffffu, *abort_flag != 0)) {
          ok = false;
          break;
        } else if (__any_sync(0xffffffffu, clock64() - t_last > kWaitLimitCycles)) {
          if (lane == 0) {
            *abort_flag = 1;
            atomicExch(p.status, kStatusWaitTimeout);
          }
          ok = false;
          break;
        }
      }
      if (!ok && any) {
        // aborted: wait for the products in flight before TMEM is released
        volatile int never = 0;
        umma_commit_warp(&ms.drain);
        __syncwarp();
        mbar_wait(&ms.drain, 0, &never, p.status, kWaitLimitCycles / 4);
        __syncwarp();
      }
    }
  } else {
    // -------------------------------------------- softmax and the record --
    const int t = threadIdx.x;  // key of the stage; later the row dd of O^T
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const float scale2 = polar_tau((float)(n > 0 ? n : 1), p.c.log_t0) * kPLog2e *
                         rsqrtf((float)D);
    float m_ref[G], lsum[G], qsum[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      m_ref[g] = -INFINITY;
      lsum[g] = qsum[g] = 0.f;
    }
    uint8_t* pt = smem + L::kPOff;
    // byte offset of (head g, key t) in a P^T buffer: K-major, 128-byte swizzle
    const int p_atom = t >> 6, p_ch = (t & 63) >> 3, p_in = (t & 7) * 2;
    bool good = true;  // this thread's waits so far
    for (int j = 0; j < nst; ++j) {
      const int slot = j % NS;
      bool w = good && mbar_wait2(&ms.s_full[j % kPB], (uint32_t)(j / kPB) & 1, &ms.full[slot],
                                  (uint32_t)(j / NS) & 1, abort_flag, p.status);
      w = __all_sync(0xffffffffu, w);  // tcgen05.ld is warp-collective
      uint32_t r[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
      if (w) {
        tc_fence_after();
        tmem_ld8(tmem + lane_base + st_col(j % kPB), r);
        tmem_ld_wait();
        reg_fence8(r);
      }
      const int key = k0 + j * kPK + t;
      const bool mine = t < kPK;  // threads 64-127 hold no key of the stage
      const bool valid =
          mine && key < k1 && ((ms.valid[slot][(t & (kPK - 1)) >> 5] >> (t & 31)) & 1u);
      // The stage's maxima are needed only when some logit passes its head's
      // reference by more than the threshold (the first valid stage always
      // does: the reference starts at -inf); the block first agrees on that
      // with one vote, and computes the maxima only then.
      float x[G];
      bool up = false;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        x[g] = valid ? __uint_as_float(r[g]) * scale2 : -INFINITY;
        up = up || x[g] > m_ref[g] + kPRescale;
      }
      const bool wup = __any_sync(0xffffffffu, up);
      if (lane == 0) ms.up[j & 1][warp] = wup ? 1u : 0u;
      if (!softmax_bar_and(w)) {
        good = false;
        break;
      }
      float alpha[G];
#pragma unroll
      for (int g = 0; g < G; ++g) alpha[g] = 1.f;
      bool resc = false;
      if (ms.up[j & 1][0] | ms.up[j & 1][1] | ms.up[j & 1][2] | ms.up[j & 1][3]) {
        float bm[G];
#pragma unroll
        for (int g = 0; g < G; ++g) bm[g] = x[g];
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1)
#pragma unroll
          for (int g = 0; g < G; ++g) bm[g] = fmaxf(bm[g], __shfl_xor_sync(0xffffffffu, bm[g], o));
        if (lane == 0)
#pragma unroll
          for (int g = 0; g < G; ++g) ms.red[j & 1][warp][g] = bm[g];
        softmax_bar_and(true);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float mx = fmax3(fmaxf(ms.red[j & 1][0][g], ms.red[j & 1][1][g]),
                                 ms.red[j & 1][2][g], ms.red[j & 1][3][g]);
          if (mx > m_ref[g] + kPRescale || (m_ref[g] == -INFINITY && mx != -INFINITY)) {
            alpha[g] = m_ref[g] == -INFINITY ? 0.f : ex2_approx(m_ref[g] - mx);
            m_ref[g] = mx;
            lsum[g] *= alpha[g];
            qsum[g] *= alpha[g] * alpha[g];  // squared correction factor
            resc = true;
          }
        }
      }
      // P^T buffer j % kPB was read by the product of stage j - kPB
      if (j >= kPB)
        good = mbar_wait(&ms.pv_done[j % kPB], (uint32_t)(j / kPB - 1) & 1, abort_flag, p.status);
      if (good && mine) {
        uint8_t* pb = pt + (j % kPB) * L::kPBuf + p_atom * (kPN * 128);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float pv = valid ? ex2_approx(x[g] - m_ref[g]) : 0.f;
          lsum[g] += pv;
          qsum[g] = fmaf(pv, pv, qsum[g]);
          *reinterpret_cast<__nv_bfloat16*>(pb + g * 128 + ((p_ch ^ (g & 7)) << 4) + p_in) =
              __float2bfloat16_rn(pv);
        }
        if (!valid) {
          // the V row of a masked key may hold anything: zero it
          uint8_t* vr = smem + L::kVOff + slot * L::kTile + t * 128;
#pragma unroll
          for (int a = 0; a < L::kAtoms; ++a)
#pragma unroll
            for (int ch = 0; ch < 8; ++ch)
              *reinterpret_cast<uint4*>(vr + a * L::kAtomBytes + ch * 16) =
                  make_uint4(0u, 0u, 0u, 0u);
        }
      }
      if (resc && j >= 1) {
        // O^T holds stages < j (product j - 1 done): scale the moved heads
        bool w3 = good && mbar_wait(&ms.pv_done[(j - 1) % kPB], (uint32_t)((j - 1) / kPB) & 1,
                                    abort_flag, p.status);
        w3 = __all_sync(0xffffffffu, w3);
        if (w3) {
          tc_fence_after();
          uint32_t o[8];
          tmem_ld8(tmem + lane_base + 32, o);
          tmem_ld_wait();
          reg_fence8(o);
#pragma unroll
          for (int g = 0; g < G; ++g) o[g] = __float_as_uint(__uint_as_float(o[g]) * alpha[g]);
          tmem_st8(tmem + lane_base + 32, o);
          tmem_st_wait();
        }
        good = good && w3;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      if (good) mbar_arrive(&ms.p_full[j % kPB]);
    }
    // l and Q2 of each head over the 128 key lanes
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1)
#pragma unroll
      for (int g = 0; g < G; ++g) {
        lsum[g] += __shfl_xor_sync(0xffffffffu, lsum[g], o);
        qsum[g] += __shfl_xor_sync(0xffffffffu, qsum[g], o);
      }
    if (lane == 0)
#pragma unroll
      for (int g = 0; g < G; ++g) {
        ms.lred[warp][g] = lsum[g];
        ms.qred[warp][g] = qsum[g];
      }
    softmax_bar();
    float acc[G];
#pragma unroll
    for (int g = 0; g < G; ++g) acc[g] = 0.f;
    bool fin = good && nst > 0 &&
               mbar_wait(&ms.pv_done[(nst - 1) % kPB], (uint32_t)((nst - 1) / kPB) & 1,
                         abort_flag, p.status);
    fin = __all_sync(0xffffffffu, fin);
    if (nst > 0) {
      if (fin) {
        tc_fence_after();
        uint32_t o[8];
        tmem_ld8(tmem + lane_base + 32, o);
        tmem_ld_wait();
        reg_fence8(o);
#pragma unroll
        for (int g = 0; g < G; ++g) acc[g] = __uint_as_float(o[g]);
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float* rec =
          p.partials + (((size_t)b * p.Hq + (size_t)hkv * G + g) * p.splits + split) * (D + 4);
      if (t < D) rec[4 + t] = acc[g];
      if (t == 0) {
        rec[0] = m_ref[g] == -INFINITY ? -INFINITY : m_ref[g] * kPLn2;  // natural units
        rec[1] = ms.lred[0][g] + ms.lred[1][g] + ms.lred[2][g] + ms.lred[3][g];
        rec[2] = ms.qred[0][g] + ms.qred[1][g] + ms.qred[2][g] + ms.qred[3][g];
        rec[3] = 0.f;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kPWarpMMA) {
    tc_fence_after();
    tmem_dealloc(tmem, kPTmemCols);
  }
}

template <int D, int G>
cudaError_t paged_tc_d(const PagedArgs& a, const CUtensorMap& mk, const CUtensorMap& mv,
                       cudaStream_t s) {
  using L = PLayout<D>;
  PagedTcParams p;
  p.q = static_cast<const __nv_bfloat16*>(a.base.q);
  p.table = a.block_table;
  p.lens = a.base.seq_lens;
  p.partials = a.base.partials;
  p.Hq = a.base.H;
  p.Hkv = a.Hkv;
  p.max_pages = a.max_pages;
  p.num_pages = a.num_pages;
  p.page_shift = a.page_shift;
  const int page = 1 << a.page_shift;
  p.frag = page < kPK ? page : kPK;
  p.rows_total = (int)((long long)a.num_pages * a.Hkv * page);
  p.splits = a.base.splits;
  p.chunk = a.base.chunk;
  p.c = a.base.c;
  p.status = a.status;
  cudaError_t e = cudaFuncSetAttribute(polar_decode_paged_tc_kernel<D, G>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       L::kSmemBytes);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)(a.base.B * a.Hkv), (unsigned)a.base.splits);
  polar_decode_paged_tc_kernel<D, G><<<grid, kPThreads, L::kSmemBytes, s>>>(mk, mv, p);
  return cudaGetLastError();
}

template <int D>
cudaError_t paged_tc_g(const PagedArgs& a, const CUtensorMap& mk, const CUtensorMap& mv,
                       cudaStream_t s) {
  switch (a.base.H / a.Hkv) {
    case 1: return paged_tc_d<D, 1>(a, mk, mv, s);
    case 2: return paged_tc_d<D, 2>(a, mk, mv, s);
    case 4: return paged_tc_d<D, 4>(a, mk, mv, s);
    default: return paged_tc_d<D, 8>(a, mk, mv, s);
  }
}

}  // namespace

cudaError_t launch_decode_paged_tc(const PagedArgs& a, const CUtensorMap& mk,
                                   const CUtensorMap& mv, cudaStream_t s) {
  return a.base.d == 128 ? paged_tc_g<128>(a, mk, mv, s) : paged_tc_g<64>(a, mk, mv, s);
}

}  // namespace polar
