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
__global__ void __launch_bounds__(kThreads)
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

template <int D, typename T>
__global__ void __launch_bounds__(D)
    polar_decode_combine_kernel(const float* __restrict__ partials, int splits,
                                const T* __restrict__ q, const T* __restrict__ mem,
                                const float* __restrict__ w_count, T* __restrict__ out,
                                float* __restrict__ n_eff, float* __restrict__ conf,
                                int H, int Tkv, polar_consts_t c) {
  __shared__ float red[D / 32];
  const int bh = blockIdx.x, h = bh % H, x = threadIdx.x;
  const float qx = Elem<T>::to_float(q[(size_t)bh * D + x]);
  const float mx = Elem<T>::to_float(mem[(size_t)bh * D + x]);
  const float wx = w_count[(size_t)h * D + x];
  // the partials are written by the preceding grid (programmatic launch)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const float* rec = partials + (size_t)bh * splits * (D + 4);
  float M = -INFINITY;
  for (int s = 0; s < splits; ++s) M = fmaxf(M, rec[(size_t)s * (D + 4)]);
  float L = 0.f, Q = 0.f, a = 0.f;
  for (int s = 0; s < splits; ++s) {
    const float* r = rec + (size_t)s * (D + 4);
    if (r[0] == -INFINITY) continue;  // empty split
    const float wgt = expf(r[0] - M);
    L = fmaf(wgt, r[1], L);
    Q = fmaf(wgt * wgt, r[2], Q);  // squared correction factor
    a = fmaf(wgt, r[4 + x], a);
  }
  const float acc_sq = block_sum<D>(a * a, red);
  const float q_sq = block_sum<D>(qx * qx, red);
  const RowResult res = polar_finish(M, L, Q, acc_sq, q_sq, (float)Tkv, D, c);
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
                            a.n_eff, a.conf, a.H, a.Tkv, a.c);
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
