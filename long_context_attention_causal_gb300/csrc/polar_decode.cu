// Split-KV decode of causal Polar Attention, and the combine step.
//
// "ATMA: Length-Invariant Language Modeling via Polar Attention and
// Gated-Delta Compression Memory", §2.2: the decode kernel streams the KV
// cache; the streaming accumulators (running max m, l = sum p, Q2 = sum p^2,
// acc = sum p v) are associative under max-rebasing with a factor w on l and
// acc and w^2 on Q2 (the squared correction factors), so the cache is cut
// into chunks whose partial states merge exactly.  §2.1 gives the epilogue.
//
// Split kernel (HBM-bound): grid (B*H, splits), 256 threads.  A lane group
// of d*size/16 lanes owns one key row at a time and reads it with 16-byte
// loads (a bf16 d=128 row = 16 lanes); the dot product is reduced with
// xor-shuffles inside the group.  Each group carries its own streaming
// state over a batch of keys per step (loads for the next batch are issued
// before the current one is consumed); the CTA merges its groups through
// shared memory and writes one partial record {m, l, Q2, 0, acc[d]}.
//
// Combine kernel: grid B*H, d threads; merges the records and applies the
// epilogue with n = Tkv.  It is launched with programmatic dependent launch
// and waits on the split grid before reading the partials.
#include "polar_device.cuh"
#include "polar_internal.h"

namespace polar {

namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kU = 4;  // keys per lane group per batch
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <typename T>
struct Elem;
template <>
struct Elem<float> {
  static constexpr int kPerVec = 4;
  __device__ static void unpack(const uint4& u, float* f) {
    f[0] = __uint_as_float(u.x);
    f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z);
    f[3] = __uint_as_float(u.w);
  }
  __device__ static float to_float(float x) { return x; }
  __device__ static float from(float x) { return x; }
};
template <>
struct Elem<__nv_bfloat16> {
  static constexpr int kPerVec = 8;
  __device__ static void unpack(const uint4& u, float* f) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      f[2 * e] = __uint_as_float(w[e] << 16);
      f[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
    }
  }
  __device__ static float to_float(__nv_bfloat16 x) { return __bfloat162float(x); }
  __device__ static __nv_bfloat16 from(float x) { return __float2bfloat16_rn(x); }
};

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

template <int D, typename T>
__global__ void __launch_bounds__(kThreads, 3)
    polar_decode_split_kernel(const T* __restrict__ q, const T* __restrict__ k,
                              const T* __restrict__ v, float* __restrict__ partials,
                              int Tkv, int splits, int chunk, polar_consts_t c) {
  constexpr int EPL = Elem<T>::kPerVec;   // elements per lane per row
  constexpr int LPK = D / EPL;            // lanes per key row
  constexpr int KPW = 32 / LPK;           // keys per warp per step
  constexpr int G = kWarps * KPW;         // lane groups per CTA
  constexpr int STEP = G;                 // keys per CTA step
  __shared__ float sm_m[G], sm_l[G], sm_q2[G];
  __shared__ float sm_acc[G][D];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp_in_warp = lane / LPK, sub = lane % LPK;
  const int g = warp * KPW + grp_in_warp;
  const int bh = blockIdx.x;
  const int split = blockIdx.y;
  const int k0 = split * chunk;
  const int k1 = min(k0 + chunk, Tkv);
  const size_t kv_base = (size_t)bh * Tkv * D;

  // query fragment, pre-scaled into log2 units of the tempered logit
  const float n = (float)Tkv;
  const float scale2 = polar_tau(n, c.log_t0) * kLog2e * rsqrtf((float)D);
  float qf[EPL];
  Elem<T>::unpack(*reinterpret_cast<const uint4*>(q + (size_t)bh * D + sub * EPL), qf);
#pragma unroll
  for (int e = 0; e < EPL; ++e) qf[e] *= scale2;

  float m = -INFINITY, l = 0.f, q2 = 0.f;
  float acc[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) acc[e] = 0.f;

  const uint4* kp = reinterpret_cast<const uint4*>(k + kv_base) + sub;
  const uint4* vp = reinterpret_cast<const uint4*>(v + kv_base) + sub;
  constexpr int kRowVecs = D / EPL;  // uint4 per row

  uint4 kb[kU], vb[kU];
  auto load_batch = [&](int bstart) {
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int key = bstart + u * STEP + g;
      if (key < k1) {
        kb[u] = ld_stream(kp + (size_t)key * kRowVecs);
        vb[u] = ld_stream(vp + (size_t)key * kRowVecs);
      } else {
        kb[u] = make_uint4(0, 0, 0, 0);
        vb[u] = make_uint4(0, 0, 0, 0);
      }
    }
  };

  int b0 = k0;
  if (b0 < k1) load_batch(b0);
  for (; b0 < k1; b0 += kU * STEP) {
    uint4 kc[kU], vc[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      kc[u] = kb[u];
      vc[u] = vb[u];
    }
    if (b0 + kU * STEP < k1) load_batch(b0 + kU * STEP);
    float s[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      float kf[EPL];
      Elem<T>::unpack(kc[u], kf);
      float d0 = 0.f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) d0 = fmaf(qf[e], kf[e], d0);
#pragma unroll
      for (int o = LPK / 2; o > 0; o >>= 1) d0 += __shfl_xor_sync(0xffffffffu, d0, o);
      const int key = b0 + u * STEP + g;
      s[u] = key < k1 ? d0 : -INFINITY;
    }
    float bm = s[0];
#pragma unroll
    for (int u = 1; u < kU; ++u) bm = fmaxf(bm, s[u]);
    const float mn = fmaxf(m, bm);
    if (mn == -INFINITY) continue;  // this group saw no key in the batch
    const float alpha = ex2_approx(m - mn);
    l *= alpha;
    q2 *= alpha * alpha;  // squared correction factor
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] *= alpha;
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const float pu = ex2_approx(s[u] - mn);
      l += pu;
      q2 = fmaf(pu, pu, q2);
      float vf[EPL];
      Elem<T>::unpack(vc[u], vf);
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[e] = fmaf(pu, vf[e], acc[e]);
    }
    m = mn;
  }

  // merge the lane groups of this CTA
  if (sub == 0) {
    sm_m[g] = m;
    sm_l[g] = l;
    sm_q2[g] = q2;
  }
#pragma unroll
  for (int e = 0; e < EPL; ++e) sm_acc[g][sub * EPL + e] = acc[e];
  __syncthreads();
  float* rec = partials + ((size_t)bh * splits + split) * (D + 4);
  float M = -INFINITY;
#pragma unroll 4
  for (int x = 0; x < G; ++x) M = fmaxf(M, sm_m[x]);
  for (int x = threadIdx.x; x < D; x += kThreads) {
    float a = 0.f;
    if (M != -INFINITY) {
      for (int y = 0; y < G; ++y) a = fmaf(ex2_approx(sm_m[y] - M), sm_acc[y][x], a);
    }
    rec[4 + x] = a;
  }
  if (threadIdx.x == 0) {
    float L = 0.f, Q = 0.f;
    if (M != -INFINITY) {
      for (int y = 0; y < G; ++y) {
        const float wgt = ex2_approx(sm_m[y] - M);
        L = fmaf(wgt, sm_l[y], L);
        Q = fmaf(wgt * wgt, sm_q2[y], Q);
      }
    }
    rec[0] = M == -INFINITY ? -INFINITY : M * kLn2;  // natural units
    rec[1] = L;
    rec[2] = Q;
    rec[3] = 0.f;
  }
}

template <int D>
__device__ __forceinline__ float block_sum(float x, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = x;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int w = 0; w < D / 32; ++w) t += red[w];
  __syncthreads();
  return t;
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

// One CTA per (b, h), one thread per column.  The split records are read in
// parallel rather than one split after another: thread x takes the scalars
// of splits x, x + D, ... (maximum, then weights e^(m_s - M) into shared
// memory, D splits at a time), and every thread's accumulator loads of a
// chunk are independent, so the merge costs a few memory latencies instead
// of two per split.
template <int D, typename T>
__global__ void __launch_bounds__(D)
    polar_decode_combine_kernel(const float* __restrict__ partials, int splits,
                                const T* __restrict__ q, const T* __restrict__ mem,
                                const float* __restrict__ w_count, T* __restrict__ out,
                                float* __restrict__ n_eff, float* __restrict__ conf,
                                int H, int Tkv, const int* __restrict__ seq_lens,
                                polar_consts_t c) {
  __shared__ float red[D / 32];
  __shared__ float wgt[D];
  const int bh = blockIdx.x, h = bh % H, x = threadIdx.x;
  constexpr int R = D + 4;  // record stride
  // keys visible to this query: the cache length, or the sequence's length
  const int n_keys = seq_lens ? seq_lens[bh / H] : Tkv;
  const float qx = Elem<T>::to_float(q[(size_t)bh * D + x]);
  const float mx = Elem<T>::to_float(mem[(size_t)bh * D + x]);
  const float wx = w_count[(size_t)h * D + x];
  // the partials are written by the preceding grid (programmatic launch)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const float* rec = partials + (size_t)bh * splits * R;
  float M = -INFINITY;
  for (int s = x; s < splits; s += D) M = fmaxf(M, rec[(size_t)s * R]);
  M = warp_max(M);
  if ((x & 31) == 0) red[x >> 5] = M;
  __syncthreads();
#pragma unroll
  for (int w = 0; w < D / 32; ++w) M = fmaxf(M, red[w]);
  __syncthreads();
  if (M == -INFINITY || n_keys < 1) {
    // no key was visible (an invalid sequence length, flagged by the split
    // kernel): direction and count are zero, the memory stream passes
    out[(size_t)bh * D + x] = Elem<T>::from(mx);
    if (x == 0) {
      n_eff[bh] = 0.f;
      if (conf) conf[bh] = 0.f;
    }
    return;
  }
  float L = 0.f, Q = 0.f, a = 0.f;
  for (int s0 = 0; s0 < splits; s0 += D) {
    const int ns = min(D, splits - s0);
    if (x < ns) {
      const float* r = rec + (size_t)(s0 + x) * R;
      const float ms = r[0];
      // an empty split (m = -inf) weighs 0
      const float e = ms == -INFINITY ? 0.f : expf(ms - M);
      L = fmaf(e, r[1], L);
      Q = fmaf(e * e, r[2], Q);  // squared correction factor
      wgt[x] = e;
    }
    __syncthreads();
    const float* col = rec + (size_t)s0 * R + 4 + x;
    int u = 0;
    for (; u + 8 <= ns; u += 8) {
      float v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) v[k] = col[(size_t)(u + k) * R];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float e = wgt[u + k];
        a = fmaf(e, e != 0.f ? v[k] : 0.f, a);
      }
    }
    for (; u < ns; ++u) {
      const float e = wgt[u];
      a = fmaf(e, e != 0.f ? col[(size_t)u * R] : 0.f, a);
    }
    __syncthreads();
  }
  L = block_sum<D>(L, red);
  Q = block_sum<D>(Q, red);
  const float acc_sq = block_sum<D>(a * a, red);
  const float q_sq = block_sum<D>(qx * qx, red);
  const RowResult res = polar_finish(M, L, Q, acc_sq, q_sq, (float)n_keys, D, c);
  out[(size_t)bh * D + x] = Elem<T>::from(fmaf(a, res.scale_u, fmaf(res.count, wx, mx)));
  if (x == 0) {
    n_eff[bh] = res.n_eff;
    if (conf) conf[bh] = res.conf;
  }
}

template <int D, typename T>
cudaError_t split_d(const DecodeArgs& a, cudaStream_t s) {
  dim3 grid(a.B * a.H, a.splits);
  polar_decode_split_kernel<D, T><<<grid, kThreads, 0, s>>>(
      static_cast<const T*>(a.q), static_cast<const T*>(a.k), static_cast<const T*>(a.v),
      a.partials, a.Tkv, a.splits, a.chunk, a.c);
  return cudaGetLastError();
}

template <int D, typename T>
cudaError_t combine_d(const DecodeArgs& a, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.B * a.H);
  cfg.blockDim = dim3(D);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, polar_decode_combine_kernel<D, T>,
                            (const float*)a.partials, a.splits, static_cast<const T*>(a.q),
                            static_cast<const T*>(a.mem), a.w_count, static_cast<T*>(a.out),
                            a.n_eff, a.conf, a.H, a.Tkv, a.seq_lens, a.c);
}

// ------------------------------------------------------------------------
// Paged, grouped-query split kernel ("ATMA", §2.2: the decode kernel reads
// paged KV blocks directly and shares one KV read among the query heads of
// a group).  Grid (B * Hkv, splits), 288 threads: warps 0-7 compute, warp 8
// copies.  The cache is [num_pages, Hkv, page, d]; key j of sequence b is row
// j % page of page block_table[b][j / page], and the rows of one (page, KV
// head) are contiguous, so the copy warp streams them with cp.async.bulk
// into a 4-stage shared-memory ring (16 KB of K and 16 KB of V per stage):
// the bytes in flight do not depend on registers.  A CTA owns one
// (b, KV head, split) and all G query heads of the group: every K/V row it
// reads serves G dot products and G accumulators.
// Page indices and sequence lengths are checked on the device: a page
// outside the pool is not read (its keys are skipped) and a length outside
// [1, splits * chunk] is clamped; both record status 3.
constexpr int kPagedWarps = 8;                 // compute warps
constexpr int kPagedThreads = 32 * (kPagedWarps + 1);
constexpr int kPagedStages = 4;
constexpr int kStageBytes = 16384;             // per tensor per stage
constexpr int kTableWindow = 256;              // block-table entries cached

template <int D, typename T, int G>
struct PagedSmem {
  static constexpr int kRowBytes = D * (int)sizeof(T);
  static constexpr int kSK = kStageBytes / kRowBytes;  // keys per stage
  uint8_t k[kPagedStages][kStageBytes];
  uint8_t v[kPagedStages][kStageBytes];
  float acc[G][kPagedWarps][D];
  float m[G][kPagedWarps], l[G][kPagedWarps], q2[G][kPagedWarps];
  uint32_t valid[kPagedStages][(kSK + 31) / 32];
  int tab[kTableWindow];  // window of the sequence's block table
  uint64_t full[kPagedStages], empty[kPagedStages];
  int abort_flag;
};

template <int D, typename T, int G>
__global__ void __launch_bounds__(kPagedThreads, 1)
    polar_decode_paged_split_kernel(const T* __restrict__ q, const T* __restrict__ kp,
                                    const T* __restrict__ vp, const int* __restrict__ table,
                                    const int* __restrict__ lens, float* __restrict__ partials,
                                    int Hq, int Hkv, int max_pages, int num_pages,
                                    int page_shift, int splits, int chunk, polar_consts_t c,
                                    int* status) {
  using S = PagedSmem<D, T, G>;
  constexpr int EPL = Elem<T>::kPerVec;  // elements per lane per row
  constexpr int LPK = D / EPL;           // lanes per key row
  constexpr int KPW = 32 / LPK;          // key rows per warp per step
  constexpr int NG = kPagedWarps * KPW;  // lane groups
  constexpr int SK = S::kSK;             // keys per stage
  constexpr int KPG = SK / NG;           // keys per lane group per stage
  constexpr int UB = (G >= 8 ? 2 : 4) < KPG ? (G >= 8 ? 2 : 4) : KPG;  // score batch
  static_assert(KPG >= 1 && SK % NG == 0 && KPG % UB == 0, "stage shape");
  extern __shared__ __align__(128) uint8_t smem_raw[];
  S& sm = *reinterpret_cast<S*>(smem_raw);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x / Hkv, hkv = blockIdx.x % Hkv;
  const int split = blockIdx.y;
  const int page = 1 << page_shift;
  int n = lens[b];
  const int n_max = min(splits * chunk, max_pages << page_shift);
  if (n < 1 || n > n_max) {
    if (threadIdx.x == 0 && split == 0) atomicExch(status, 3);
    n = n < 1 ? 0 : n_max;
  }
  const int k0 = split * chunk;
  const int k1 = min(k0 + chunk, n);
  const int nst = k1 > k0 ? (k1 - k0 + SK - 1) / SK : 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kPagedStages; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], kPagedWarps);
    }
    sm.abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  volatile int* abort_flag = &sm.abort_flag;

  if (warp == kPagedWarps) {
    // ------------------------------------------------------- copy warp --
    // The whole warp walks the stages: it reloads a window of the block
    // table into shared memory (one load latency per kTableWindow pages
    // instead of one per stage); lane 0 builds the stage's pieces and issues
    // the bulk copies.
    const int* tb = table + (size_t)b * max_pages;
    constexpr int kFragMax = SK / 8;  // pages of >= 8 rows
    const int frag = page < SK ? page : SK;  // rows per contiguous piece
    int wbase = -kTableWindow;               // first logical page in the window
    int issued = 0;
    bool ok = true;
    for (int st = 0; st < nst && ok; ++st) {
      const int slot = st % kPagedStages;
      if (st >= kPagedStages)
        ok = __all_sync(0xffffffffu,
                        mbar_wait(&sm.empty[slot], (uint32_t)(st / kPagedStages - 1) & 1,
                                  abort_flag, status));
      if (!ok) break;
      const int key0 = k0 + st * SK;
      const int key_end = min(key0 + SK, k1);
      const int lp_last = (key_end - 1) >> page_shift;
      if (lp_last >= wbase + kTableWindow) {
        wbase = key0 >> page_shift;
        for (int i = lane; i < kTableWindow; i += 32)
          sm.tab[i] = wbase + i < max_pages ? tb[wbase + i] : -1;
        __syncwarp();
      }
      if (lane == 0) {
        int pg[kFragMax];
        uint32_t mask[(SK + 31) / 32] = {};
        uint32_t bytes = 0;
        int nf = 0;
        for (int key = key0; key < key_end; key += frag, ++nf) {
          const int p_phys = sm.tab[(key >> page_shift) - wbase];
          const bool valid = p_phys >= 0 && p_phys < num_pages;
          pg[nf] = valid ? p_phys : -1;
          if (valid) {
            bytes += 2u * frag * S::kRowBytes;
            const int kk = key - key0;
            if (frag >= 32) {
              for (int w = kk >> 5; w < (kk + frag) >> 5; ++w) mask[w] = 0xffffffffu;
            } else {
              mask[kk >> 5] |= ((1u << frag) - 1u) << (kk & 31);
            }
          } else {
            atomicExch(status, 3);
          }
        }
        for (int w = 0; w < (SK + 31) / 32; ++w) sm.valid[slot][w] = mask[w];
        mbar_arrive_expect_tx(&sm.full[slot], bytes);
        for (int f = 0; f < nf; ++f) {
          if (pg[f] < 0) continue;
          const int key = key0 + f * frag;
          const size_t row = ((size_t)pg[f] * Hkv + hkv) * page + (key & (page - 1));
          const uint32_t dst = (uint32_t)(f * frag * S::kRowBytes);
          bulk_g2s(sm.k[slot] + dst, kp + row * D, frag * S::kRowBytes, &sm.full[slot]);
          bulk_g2s(sm.v[slot] + dst, vp + row * D, frag * S::kRowBytes, &sm.full[slot]);
        }
      }
      __syncwarp();
      issued = st + 1;
    }
    if (!ok && lane == 0) {
      // aborted: let the copies already issued land before the CTA exits
      volatile int never = 0;
      for (int st = issued - 1; st >= 0 && st >= issued - kPagedStages; --st)
        mbar_wait(&sm.full[st % kPagedStages], (uint32_t)(st / kPagedStages) & 1, &never,
                  status, kWaitLimitCycles / 4);
    }
  } else {
    // ---------------------------------------------------- compute warps --
    // Dot products and accumulators run on pairs of columns with packed fp32
    // instructions (fma .f32x2): half the FMA instructions of scalar code.
    constexpr int EP2 = EPL / 2;
    const int g = warp * KPW + lane / LPK, sub = lane % LPK;
    const float scale2 =
        polar_tau((float)(n > 0 ? n : 1), c.log_t0) * kLog2e * rsqrtf((float)D);
    float2 qf[G][EP2];
#pragma unroll
    for (int gi = 0; gi < G; ++gi) {
      const int hq = hkv * G + gi;
      float t[EPL];
      Elem<T>::unpack(
          *reinterpret_cast<const uint4*>(q + ((size_t)b * Hq + hq) * D + sub * EPL), t);
#pragma unroll
      for (int e = 0; e < EP2; ++e) qf[gi][e] = make_float2(t[2 * e] * scale2, t[2 * e + 1] * scale2);
    }
    float m[G], l[G], q2[G];
    float2 acc[G][EP2];
#pragma unroll
    for (int gi = 0; gi < G; ++gi) {
      m[gi] = -INFINITY;
      l[gi] = q2[gi] = 0.f;
#pragma unroll
      for (int e = 0; e < EP2; ++e) acc[gi][e] = make_float2(0.f, 0.f);
    }
    bool ok = true;
    if constexpr (G * UB == LPK) {
      // Reduce-scatter form: the G x UB partial dot products of a sub-batch
      // are summed over the lane group with log2(LPK) halving exchanges, so
      // lane `sub` ends with the whole score of head sub / UB and key
      // sub % UB (15 shuffles instead of G * UB * log2(LPK)).  That lane
      // alone takes its exp and keeps its share of l and Q2; the UB x G
      // probabilities are then broadcast for the P V update.
      const int base = lane & ~(LPK - 1);  // first lane of this group
      const int my_g = sub / UB, my_u = sub % UB;
      float l_own = 0.f, q_own = 0.f;
      for (int st = 0; st < nst && ok; ++st) {
        const int slot = st % kPagedStages;
        ok = mbar_wait(&sm.full[slot], (uint32_t)(st / kPagedStages) & 1, abort_flag, status);
        if (!ok) break;
        const int key0 = k0 + st * SK;
#pragma unroll
        for (int u0 = 0; u0 < KPG; u0 += UB) {
          float v[G * UB];
          bool my_valid = false;
          bool valid_u[UB];
#pragma unroll
          for (int u = 0; u < UB; ++u) {
            const int kk = (u0 + u) * NG + g;
            const bool valid =
                key0 + kk < k1 && ((sm.valid[slot][kk >> 5] >> (kk & 31)) & 1u);
            valid_u[u] = valid;
            my_valid = my_u == u ? valid : my_valid;
            float kf[EPL];
            Elem<T>::unpack(
                *reinterpret_cast<const uint4*>(sm.k[slot] + kk * S::kRowBytes + sub * 16), kf);
#pragma unroll
            for (int gi = 0; gi < G; ++gi) {
              float2 dp = make_float2(0.f, 0.f);
#pragma unroll
              for (int e = 0; e < EP2; ++e)
                dp = ffma2(qf[gi][e], make_float2(kf[2 * e], kf[2 * e + 1]), dp);
              v[gi * UB + u] = dp.x + dp.y;
            }
          }
#pragma unroll
          for (int w = LPK / 2; w >= 1; w >>= 1) {
            const bool upper = (sub & w) != 0;
#pragma unroll
            for (int i = 0; i < w; ++i) {
              const float send = upper ? v[i] : v[i + w];
              const float keep = upper ? v[i + w] : v[i];
              v[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
            }
          }
          const float sc = my_valid ? v[0] : -INFINITY;
          float bm = sc;
#pragma unroll
          for (int o = 1; o < UB; o <<= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, o));
          float alpha[G], m_own = -INFINITY, a_own = 1.f;
#pragma unroll
          for (int gi = 0; gi < G; ++gi) {
            const float mn = fmaxf(m[gi], __shfl_sync(0xffffffffu, bm, base + gi * UB));
            alpha[gi] = mn == -INFINITY ? 1.f : ex2_approx(m[gi] - mn);
            m[gi] = mn;
            m_own = my_g == gi ? mn : m_own;
            a_own = my_g == gi ? alpha[gi] : a_own;
            const float2 a2 = make_float2(alpha[gi], alpha[gi]), z2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int e = 0; e < EP2; ++e) acc[gi][e] = ffma2(acc[gi][e], a2, z2);
          }
          const float pown = m_own == -INFINITY ? 0.f : ex2_approx(sc - m_own);
          l_own = fmaf(l_own, a_own, pown);
          q_own = fmaf(q_own, a_own * a_own, pown * pown);  // squared correction factor
#pragma unroll
          for (int u = 0; u < UB; ++u) {
            const int kk = (u0 + u) * NG + g;
            // rows of keys that were not copied hold stale shared memory:
            // read zeros instead (p = 0 there, and 0 * NaN would not be 0)
            const uint4 raw =
                valid_u[u] ? *reinterpret_cast<const uint4*>(sm.v[slot] + kk * S::kRowBytes + sub * 16)
                           : make_uint4(0u, 0u, 0u, 0u);
            float vf[EPL];
            Elem<T>::unpack(raw, vf);
#pragma unroll
            for (int gi = 0; gi < G; ++gi) {
              const float pu = __shfl_sync(0xffffffffu, pown, base + gi * UB + u);
              const float2 p2 = make_float2(pu, pu);
#pragma unroll
              for (int e = 0; e < EP2; ++e)
                acc[gi][e] = ffma2(p2, make_float2(vf[2 * e], vf[2 * e + 1]), acc[gi][e]);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[slot]);
      }
      // per-head l and Q2 from the lanes that own the head's keys
#pragma unroll
      for (int o = 1; o < UB; o <<= 1) {
        l_own += __shfl_xor_sync(0xffffffffu, l_own, o);
        q_own += __shfl_xor_sync(0xffffffffu, q_own, o);
      }
#pragma unroll
      for (int gi = 0; gi < G; ++gi) {
        l[gi] = __shfl_sync(0xffffffffu, l_own, base + gi * UB);
        q2[gi] = __shfl_sync(0xffffffffu, q_own, base + gi * UB);
      }
    } else {
      for (int st = 0; st < nst && ok; ++st) {
        const int slot = st % kPagedStages;
        ok = mbar_wait(&sm.full[slot], (uint32_t)(st / kPagedStages) & 1, abort_flag, status);
        if (!ok) break;
        const int key0 = k0 + st * SK;
        // keys of this stage in sub-batches of UB (the score batch costs G * UB
        // registers)
#pragma unroll
        for (int u0 = 0; u0 < KPG; u0 += UB) {
          float sc[G][UB];
#pragma unroll
          for (int u = 0; u < UB; ++u) {
            const int kk = (u0 + u) * NG + g;  // row of the stage
            const bool valid =
                key0 + kk < k1 && ((sm.valid[slot][kk >> 5] >> (kk & 31)) & 1u);
            float kf[EPL];
            Elem<T>::unpack(
                *reinterpret_cast<const uint4*>(sm.k[slot] + kk * S::kRowBytes + sub * 16), kf);
#pragma unroll
            for (int gi = 0; gi < G; ++gi) {
              float2 dp = make_float2(0.f, 0.f);
#pragma unroll
              for (int e = 0; e < EP2; ++e)
                dp = ffma2(qf[gi][e], make_float2(kf[2 * e], kf[2 * e + 1]), dp);
              float d0 = dp.x + dp.y;
#pragma unroll
              for (int o = LPK / 2; o > 0; o >>= 1) d0 += __shfl_xor_sync(0xffffffffu, d0, o);
              sc[gi][u] = valid ? d0 : -INFINITY;
            }
          }
#pragma unroll
          for (int gi = 0; gi < G; ++gi) {
            float bm = sc[gi][0];
#pragma unroll
            for (int u = 1; u < UB; ++u) bm = fmaxf(bm, sc[gi][u]);
            const float mn = fmaxf(m[gi], bm);
            if (mn == -INFINITY) continue;  // no visible key yet for the group
            const float alpha = ex2_approx(m[gi] - mn);
            l[gi] *= alpha;
            q2[gi] *= alpha * alpha;  // squared correction factor
            const float2 a2 = make_float2(alpha, alpha), z2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int e = 0; e < EP2; ++e) acc[gi][e] = ffma2(acc[gi][e], a2, z2);
            m[gi] = mn;
          }
#pragma unroll
          for (int u = 0; u < UB; ++u) {
            const int kk = (u0 + u) * NG + g;
            // rows of keys that were not copied hold stale shared memory
            const uint4 raw =
                sc[0][u] != -INFINITY
                    ? *reinterpret_cast<const uint4*>(sm.v[slot] + kk * S::kRowBytes + sub * 16)
                    : make_uint4(0u, 0u, 0u, 0u);
            float vf[EPL];
            Elem<T>::unpack(raw, vf);
#pragma unroll
            for (int gi = 0; gi < G; ++gi) {
              if (m[gi] == -INFINITY) continue;
              const float pu = ex2_approx(sc[gi][u] - m[gi]);  // 0 for skipped keys
              l[gi] += pu;
              q2[gi] = fmaf(pu, pu, q2[gi]);
              const float2 p2 = make_float2(pu, pu);
#pragma unroll
              for (int e = 0; e < EP2; ++e)
                acc[gi][e] = ffma2(p2, make_float2(vf[2 * e], vf[2 * e + 1]), acc[gi][e]);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[slot]);
      }
    }
    // merge the lane groups of each warp (shuffles), then the warps (smem)
#pragma unroll
    for (int gi = 0; gi < G; ++gi) {
#pragma unroll
      for (int o = LPK; o < 32; o <<= 1) {
        const float mo = __shfl_xor_sync(0xffffffffu, m[gi], o);
        const float lo = __shfl_xor_sync(0xffffffffu, l[gi], o);
        const float qo = __shfl_xor_sync(0xffffffffu, q2[gi], o);
        const float M = fmaxf(m[gi], mo);
        const float wa = M == -INFINITY ? 0.f : ex2_approx(m[gi] - M);
        const float wb = M == -INFINITY ? 0.f : ex2_approx(mo - M);
        l[gi] = wa * l[gi] + wb * lo;
        q2[gi] = wa * wa * q2[gi] + wb * wb * qo;
#pragma unroll
        for (int e = 0; e < EP2; ++e) {
          const float ax = __shfl_xor_sync(0xffffffffu, acc[gi][e].x, o);
          const float ay = __shfl_xor_sync(0xffffffffu, acc[gi][e].y, o);
          acc[gi][e] = make_float2(wa * acc[gi][e].x + wb * ax, wa * acc[gi][e].y + wb * ay);
        }
        m[gi] = M;
      }
      if (lane == 0) {
        sm.m[gi][warp] = m[gi];
        sm.l[gi][warp] = l[gi];
        sm.q2[gi][warp] = q2[gi];
      }
      if (lane < LPK) {
#pragma unroll
        for (int e = 0; e < EP2; ++e) {
          sm.acc[gi][warp][sub * EPL + 2 * e] = acc[gi][e].x;
          sm.acc[gi][warp][sub * EPL + 2 * e + 1] = acc[gi][e].y;
        }
      }
    }
  }
  __syncthreads();
  if (warp < kPagedWarps) {
    for (int idx = threadIdx.x; idx < G * D; idx += 32 * kPagedWarps) {
      const int gi = idx / D, x = idx % D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kPagedWarps; ++w) M = fmaxf(M, sm.m[gi][w]);
      float a = 0.f, L = 0.f, Q = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < kPagedWarps; ++w) {
          const float wt = ex2_approx(sm.m[gi][w] - M);
          a = fmaf(wt, sm.acc[gi][w][x], a);
          L = fmaf(wt, sm.l[gi][w], L);
          Q = fmaf(wt * wt, sm.q2[gi][w], Q);
        }
      }
      float* rec = partials + (((size_t)b * Hq + hkv * G + gi) * splits + split) * (D + 4);
      rec[4 + x] = a;
      if (x == 0) {
        rec[0] = M == -INFINITY ? -INFINITY : M * kLn2;  // natural units
        rec[1] = L;
        rec[2] = Q;
        rec[3] = 0.f;
      }
    }
  }
}

template <int D, typename T, int G>
cudaError_t paged_split_d(const PagedArgs& a, cudaStream_t s) {
  using S = PagedSmem<D, T, G>;
  const DecodeArgs& d = a.base;
  const int smem = (int)sizeof(S);
  cudaError_t e = cudaFuncSetAttribute(polar_decode_paged_split_kernel<D, T, G>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(d.B * a.Hkv, d.splits);
  polar_decode_paged_split_kernel<D, T, G><<<grid, kPagedThreads, smem, s>>>(
      static_cast<const T*>(d.q), static_cast<const T*>(a.k_pages),
      static_cast<const T*>(a.v_pages), a.block_table, d.seq_lens, d.partials, d.H, a.Hkv,
      a.max_pages, a.num_pages, a.page_shift, d.splits, d.chunk, d.c, a.status);
  return cudaGetLastError();
}

template <int D, typename T>
cudaError_t paged_split_g(const PagedArgs& a, cudaStream_t s) {
  switch (a.base.H / a.Hkv) {
    case 1: return paged_split_d<D, T, 1>(a, s);
    case 2: return paged_split_d<D, T, 2>(a, s);
    case 4: return paged_split_d<D, T, 4>(a, s);
    default: return paged_split_d<D, T, 8>(a, s);
  }
}

}  // namespace

cudaError_t launch_decode_split(const DecodeArgs& a, int dtype, cudaStream_t s) {
  if (dtype == POLAR_BF16)
    return a.d == 64 ? split_d<64, __nv_bfloat16>(a, s) : split_d<128, __nv_bfloat16>(a, s);
  return a.d == 64 ? split_d<64, float>(a, s) : split_d<128, float>(a, s);
}

cudaError_t launch_decode_combine(const DecodeArgs& a, int dtype, cudaStream_t s) {
  if (dtype == POLAR_BF16)
    return a.d == 64 ? combine_d<64, __nv_bfloat16>(a, s) : combine_d<128, __nv_bfloat16>(a, s);
  return a.d == 64 ? combine_d<64, float>(a, s) : combine_d<128, float>(a, s);
}

}  // namespace polar

namespace polar {
cudaError_t launch_decode_paged_split(const PagedArgs& a, int dtype, cudaStream_t s) {
  if (dtype == POLAR_BF16)
    return a.base.d == 64 ? paged_split_g<64, __nv_bfloat16>(a, s)
                          : paged_split_g<128, __nv_bfloat16>(a, s);
  return a.base.d == 64 ? paged_split_g<64, float>(a, s) : paged_split_g<128, float>(a, s);
}
}  // namespace polar
