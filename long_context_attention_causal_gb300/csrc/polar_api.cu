// C ABI of libpolarattn.so: argument validation, TMA descriptor encoding and
// kernel dispatch.  The declarations and the contract of every entry point
// are in include/polar_attn.h.
#include <cudaTypedefs.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <mutex>

#include "polar_device.cuh"
#include "polar_internal.h"

namespace polar {

// Kernel-side status word of each device (see polar_attn_device_status).
__device__ int g_status = 0;

namespace {

// Description of the last CUDA-level failure on this host thread.
thread_local char t_last_error[256] = "";

}  // namespace

void set_last_error(const char* msg) {
  std::snprintf(t_last_error, sizeof(t_last_error), "%s", msg ? msg : "");
}

namespace {

void note(const char* what, int code, const char* detail) {
  std::snprintf(t_last_error, sizeof(t_last_error), "%s failed (%d: %s)", what, code,
                detail ? detail : "");
}

int cuda_status(const char* what, cudaError_t e) {
  if (e == cudaSuccess) return POLAR_OK;
  note(what, (int)e, cudaGetErrorString(e));
  return POLAR_ERR_CUDA;
}

int* status_word() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return nullptr;
  return static_cast<int*>(p);
}

}  // namespace

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool consts_ok(const polar_consts_t& c) {
  return std::isfinite(c.log_t0) && c.log_t0 > 0.f && std::isfinite(c.kappa) &&
         c.kappa > 0.f && std::isfinite(c.sigma_k) && c.sigma_k >= 0.f &&
         std::isfinite(c.eps) && c.eps > 0.f && c.floor_order >= 0 && c.floor_order <= 2;
}

polar_consts_t defaults() {
  polar_consts_t c;
  c.log_t0 = 7.6246189861593985f;  // ln 2048
  c.kappa = 7.6246189861593985f;
  c.sigma_k = 1.0f;
  c.eps = 1e-6f;
  c.floor_order = 1;
  return c;
}

// The kernels are built for sm_103a only.
int check_device(int* num_sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return POLAR_ERR_DEVICE;
  int major = 0, minor = 0, sms = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return POLAR_ERR_DEVICE;
  if (major != 10 || minor != 3) return POLAR_ERR_DEVICE;
  if (num_sms) *num_sms = sms;
  return POLAR_OK;
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 3-D map over a [BH, T, d] bf16 tensor with a {64, rows, 1} box and 128-byte
// swizzle; out-of-range rows read as zeros.
bool make_map(CUtensorMap* map, const void* base, int BH, int T, int d, int rows = 128) {
  auto fn = encode_fn();
  if (!fn) {
    note("cudaGetDriverEntryPointByVersion(cuTensorMapEncodeTiled)", -1, "");
    return false;
  }
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)T, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)T * d * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r =
      fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
         estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) note("cuTensorMapEncodeTiled", (int)r, "");
  return r == CUDA_SUCCESS;
}

// 2-D map over a [rows, d] bf16 tensor with a {64, box_rows} box and
// 128-byte swizzle; rows past the end read as zeros.
bool make_map_2d(CUtensorMap* map, const void* base, long long rows, int d, int box_rows) {
  auto fn = encode_fn();
  if (!fn) {
    note("cudaGetDriverEntryPointByVersion(cuTensorMapEncodeTiled)", -1, "");
    return false;
  }
  cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)d * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r =
      fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
         estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) note("cuTensorMapEncodeTiled", (int)r, "");
  return r == CUDA_SUCCESS;
}

// bf16 prefill launch (tcgen05 kernel, 128-row TMA boxes for Q, K and V).
int launch_fwd_bf16(const FwdArgs& a, cudaStream_t s) {
  const int BH = a.B * a.H;
  CUtensorMap mq, mk, mv, mo;
  if (!make_map(&mq, a.q, BH, a.T, a.d) || !make_map(&mk, a.k, BH, a.T, a.d) ||
      !make_map(&mv, a.v, BH, a.T, a.d) || !make_map(&mo, a.out, BH, a.T, a.d))
    return POLAR_ERR_CUDA;
  return cuda_status("prefill (tcgen05) launch", launch_fwd_tc(a, mq, mk, mv, mo, s));
}

}  // namespace

// Split count of the decode: at least about eight waves of split CTAs
// (three 256-thread CTAs per SM) and, among the counts up to twice that
// minimum, the one whose last wave is fullest -- a partial last wave leaves
// SMs idle at the end of the stream (decode_32k: 10 splits, 11.2 waves,
// ran at 7.40 TB/s; 8 and 16 splits, 9.0 and 18.0 waves, at 7.55-7.58) --
// the smaller count on a tie; never under 512 keys per split.
int auto_splits(int BH, int Tkv, int num_sms) {
  const long long resident = (long long)(num_sms > 0 ? num_sms : 148) * 3;
  long long cap = (Tkv + 511) / 512;
  if (cap > 1024) cap = 1024;
  if (cap < 1) cap = 1;
  const long long bh = BH > 0 ? BH : 1;
  long long lo = (8 * resident + bh - 1) / bh;
  if (lo > cap) lo = cap;
  if (lo < 1) lo = 1;
  const long long hi = 2 * lo < cap ? 2 * lo : cap;
  long long best = lo;
  double best_fill = -1.0;
  for (long long s = lo; s <= hi; ++s) {
    const long long ctas = bh * s;
    const long long waves = (ctas + resident - 1) / resident;
    const double fill = (double)ctas / (double)(waves * resident);
    if (fill > best_fill + 1e-12) {
      best_fill = fill;
      best = s;
    }
  }
  return (int)best;
}

bool decode_sizes_ok(int B, int H, int Tkv, int d) {
  return B >= 0 && H >= 0 && Tkv >= 1 && Tkv <= (1 << 30) && (d == 64 || d == 128) &&
         (long long)B * H <= INT_MAX;
}

int l2_head_group(int BH, double per_head_bytes) {
  int dev = 0, l2 = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev);
  const double budget = l2 > 0 ? l2 / 3.0 : 40e6;
  const double fit = per_head_bytes > 0 ? budget / per_head_bytes : (double)BH;
  int g = fit >= BH ? BH : (fit >= 1.0 ? (int)fit : 1);
  for (int c = g; c > 0 && c > g - 64; --c)
    if (BH % c == 0) {
      g = c;
      break;
    }
  return g;
}

}  // namespace polar

using namespace polar;

extern "C" {

int polar_attn_version(void) { return 101; }

const char* polar_attn_last_error(void) { return t_last_error; }

int polar_attn_default_consts(polar_consts_t* c) {
  if (!c) return POLAR_ERR_INVALID;
  *c = defaults();
  return POLAR_OK;
}

const char* polar_attn_strerror(int status) {
  switch (status) {
    case POLAR_OK: return "ok";
    case POLAR_ERR_INVALID: return "invalid argument (null pointer, negative size or bad constant)";
    case POLAR_ERR_UNSUPPORTED: return "unsupported shape or dtype (d must be 64 or 128)";
    case POLAR_ERR_MISALIGNED: return "tensor pointer not 16-byte aligned";
    case POLAR_ERR_WORKSPACE: return "decode workspace missing or too small";
    case POLAR_ERR_CUDA: return "CUDA launch failed";
    case POLAR_ERR_DEVICE: return "no usable sm_103 device";
    default: return "unknown status";
  }
}

int polar_attn_fwd(const void* q, const void* k, const void* v, const void* mem,
                   const float* w_count, void* out, float* n_eff, float* conf, int B, int H,
                   int T, int d, int dtype, const polar_consts_t* c, void* stream) {
  if (B < 0 || H < 0 || T < 0) return POLAR_ERR_INVALID;
  if (dtype != POLAR_F32 && dtype != POLAR_BF16) return POLAR_ERR_UNSUPPORTED;
  if (d != 64 && d != 128) return POLAR_ERR_UNSUPPORTED;
  const polar_consts_t cc = c ? *c : defaults();
  if (!consts_ok(cc)) return POLAR_ERR_INVALID;
  if ((long long)B * H * T == 0) return POLAR_OK;
  if (!q || !k || !v || !mem || !w_count || !out || !n_eff) return POLAR_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(mem) ||
      !aligned16(w_count) || !aligned16(out))
    return POLAR_ERR_MISALIGNED;
  if ((long long)B * H > INT_MAX / 64 || T > (1 << 30)) return POLAR_ERR_UNSUPPORTED;
  int st = check_device(nullptr);
  if (st != POLAR_OK) return st;
  int* status = status_word();
  if (!status) return cuda_status("cudaGetSymbolAddress", cudaGetLastError());
  FwdArgs a{q, k, v, mem, w_count, out, n_eff, conf, B, H, T, d, cc, status};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (dtype == POLAR_BF16) return launch_fwd_bf16(a, s);
  e = launch_fwd_f32(a, s);
  return cuda_status("prefill (fp32) launch", e);
}

int polar_attn_fwd_stats(const void* q, const void* k, const void* v, const void* mem,
                         const float* w_count, void* out, float* n_eff, float* conf,
                         float* stats, int B, int H, int T, int d, int dtype,
                         const polar_consts_t* c, void* stream) {
  if (B < 0 || H < 0 || T < 0) return POLAR_ERR_INVALID;
  if (dtype != POLAR_BF16) {
    set_last_error("polar_attn_fwd_stats: bf16 only (fp32: polar_attn_fwd + polar_attn_bwd)");
    return POLAR_ERR_UNSUPPORTED;
  }
  if (d != 64 && d != 128) return POLAR_ERR_UNSUPPORTED;
  const polar_consts_t cc = c ? *c : defaults();
  if (!consts_ok(cc)) return POLAR_ERR_INVALID;
  if ((long long)B * H * T == 0) return POLAR_OK;
  if (!q || !k || !v || !mem || !w_count || !out || !n_eff || !conf || !stats)
    return POLAR_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(mem) ||
      !aligned16(w_count) || !aligned16(out) || (reinterpret_cast<uintptr_t>(stats) & 7u))
    return POLAR_ERR_MISALIGNED;
  if ((long long)B * H > INT_MAX / 64 || T > (1 << 30)) return POLAR_ERR_UNSUPPORTED;
  int st = check_device(nullptr);
  if (st != POLAR_OK) return st;
  int* status = status_word();
  if (!status) return cuda_status("cudaGetSymbolAddress", cudaGetLastError());
  FwdArgs a{q, k, v, mem, w_count, out, n_eff, conf, B, H, T, d, cc, status};
  a.stats = stats;
  return launch_fwd_bf16(a, static_cast<cudaStream_t>(stream));
}

int polar_attn_decode_num_splits(int B, int H, int Tkv, int d) {
  if (!decode_sizes_ok(B, H, Tkv, d)) return 0;
  int sms = 0;
  if (check_device(&sms) != POLAR_OK) sms = 148;
  const int BH = B * H > 0 ? B * H : 1;
  return auto_splits(BH, Tkv, sms);
}

size_t polar_attn_decode_workspace_bytes(int B, int H, int Tkv, int d, int num_splits) {
  if (!decode_sizes_ok(B, H, Tkv, d) || num_splits < 0) return 0;
  const int s = num_splits > 0 ? num_splits : polar_attn_decode_num_splits(B, H, Tkv, d);
  return (size_t)B * H * s * (d + 4) * sizeof(float);
}

int polar_attn_decode(const void* q, const void* k_cache, const void* v_cache, const void* mem,
                      const float* w_count, void* out, float* n_eff, float* conf, int B, int H,
                      int Tkv, int d, int dtype, const polar_consts_t* c, int num_splits,
                      void* workspace, size_t workspace_bytes, void* stream) {
  if (B < 0 || H < 0 || Tkv < 1 || num_splits < 0) return POLAR_ERR_INVALID;
  if (dtype != POLAR_F32 && dtype != POLAR_BF16) return POLAR_ERR_UNSUPPORTED;
  if (d != 64 && d != 128) return POLAR_ERR_UNSUPPORTED;
  if (!decode_sizes_ok(B, H, Tkv, d) || num_splits > 65535) return POLAR_ERR_UNSUPPORTED;
  const polar_consts_t cc = c ? *c : defaults();
  if (!consts_ok(cc)) return POLAR_ERR_INVALID;
  if ((long long)B * H == 0) return POLAR_OK;
  if (!q || !k_cache || !v_cache || !mem || !w_count || !out || !n_eff)
    return POLAR_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(mem) ||
      !aligned16(w_count) || !aligned16(out))
    return POLAR_ERR_MISALIGNED;
  int sms = 0;
  int st = check_device(&sms);
  if (st != POLAR_OK) return st;
  const int splits = num_splits > 0 ? num_splits : auto_splits(B * H, Tkv, sms);
  const size_t need = (size_t)B * H * splits * (d + 4) * sizeof(float);
  if (!workspace || workspace_bytes < need) return POLAR_ERR_WORKSPACE;
  if (!aligned16(workspace)) return POLAR_ERR_MISALIGNED;
  DecodeArgs a{q, k_cache, v_cache, mem, w_count, out, n_eff, conf, B, H, Tkv, d, cc,
               splits, (Tkv + splits - 1) / splits, static_cast<float*>(workspace)};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  st = cuda_status("decode split launch", launch_decode_split(a, dtype, s));
  if (st != POLAR_OK) return st;
  return cuda_status("decode combine launch", launch_decode_combine(a, dtype, s));
}

static bool paged_sizes_ok(int B, int Hq, int Hkv, int d, int max_seq_len) {
  if (B < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0) return false;
  const int G = Hq / Hkv;
  if (G != 1 && G != 2 && G != 4 && G != 8) return false;
  return (d == 64 || d == 128) && max_seq_len >= 1 && max_seq_len <= (1 << 30) &&
         (long long)B * Hq <= INT_MAX;
}

// Paged split count: a split CTA pays about six stages' time for its start
// and its record (the weight 6 fits sweeps at 32K tokens on 152 SMs, where
// 2, 4 and 8 query heads per KV head run fastest at 7, 7 and 9 splits), so
// prefer whole waves of CTAs that each stream at least 16 stages
// (16 KB of K per stage, counted for bf16 rows so that the workspace query
// and the call always agree).  A wave is two CTAs per SM, the residency of
// the bf16 tensor-core split kernel (the fp32 kernel runs one per SM).
static int auto_splits_paged(int BH, int max_seq_len, int d, int sms) {
  const int stage_keys = 16384 / (d * 2);
  const int stages = (max_seq_len + stage_keys - 1) / stage_keys;
  const int slots = 2 * sms;
  int best = 1;
  double best_eff = -1.0;
  for (int s = 1; s <= 256 && s <= stages; ++s) {
    const long long ctas = (long long)BH * s;
    const double waves = (double)ctas / slots;
    const double fill = waves / std::ceil(waves);
    const int per = (stages + s - 1) / s;
    if (per < 16 && s > 1) break;
    const double eff = fill * per / (per + 6.0);
    if (eff > best_eff + 1e-9) {
      best_eff = eff;
      best = s;
    }
  }
  return best;
}

int polar_attn_decode_paged_num_splits(int B, int Hkv, int max_seq_len, int d) {
  if (B < 0 || Hkv < 1 || max_seq_len < 1 || (d != 64 && d != 128)) return 0;
  int sms = 0;
  if (check_device(&sms) != POLAR_OK) sms = 148;
  const int BH = B * Hkv > 0 ? B * Hkv : 1;
  return auto_splits_paged(BH, max_seq_len, d, sms);
}

size_t polar_attn_decode_paged_workspace_bytes(int B, int Hq, int Hkv, int max_seq_len, int d,
                                               int num_splits) {
  if (!paged_sizes_ok(B, Hq, Hkv, d, max_seq_len) || num_splits < 0) return 0;
  const int s =
      num_splits > 0 ? num_splits : polar_attn_decode_paged_num_splits(B, Hkv, max_seq_len, d);
  return (size_t)B * Hq * s * (d + 4) * sizeof(float);
}

int polar_attn_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                            const int* block_table, const int* seq_lens, const void* mem,
                            const float* w_count, void* out, float* n_eff, float* conf, int B,
                            int Hq, int Hkv, int d, int page_size, int num_pages, int max_pages,
                            int max_seq_len, int dtype, const polar_consts_t* c, int num_splits,
                            void* workspace, size_t workspace_bytes, void* stream) {
  if (B < 0 || Hq < 1 || Hkv < 1 || num_splits < 0 || num_pages < 1 || max_pages < 1 ||
      max_seq_len < 1)
    return POLAR_ERR_INVALID;
  if (dtype != POLAR_F32 && dtype != POLAR_BF16) return POLAR_ERR_UNSUPPORTED;
  if (!paged_sizes_ok(B, Hq, Hkv, d, max_seq_len) || num_splits > 65535)
    return POLAR_ERR_UNSUPPORTED;
  if (page_size < 8 || page_size > 1024 || (page_size & (page_size - 1)) != 0)
    return POLAR_ERR_UNSUPPORTED;
  if ((long long)max_pages * page_size < max_seq_len) return POLAR_ERR_INVALID;
  const polar_consts_t cc = c ? *c : defaults();
  if (!consts_ok(cc)) return POLAR_ERR_INVALID;
  if (B == 0) return POLAR_OK;
  if (!q || !k_pages || !v_pages || !block_table || !seq_lens || !mem || !w_count || !out ||
      !n_eff)
    return POLAR_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(mem) ||
      !aligned16(w_count) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(block_table) & 3u) ||
      (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
    return POLAR_ERR_MISALIGNED;
  int sms = 0;
  int st = check_device(&sms);
  if (st != POLAR_OK) return st;
  const int splits = num_splits > 0 ? num_splits : auto_splits_paged(B * Hkv, max_seq_len, d, sms);
  const size_t need = (size_t)B * Hq * splits * (d + 4) * sizeof(float);
  if (!workspace || workspace_bytes < need) return POLAR_ERR_WORKSPACE;
  if (!aligned16(workspace)) return POLAR_ERR_MISALIGNED;
  int* status = status_word();
  if (!status) return cuda_status("cudaGetSymbolAddress", cudaGetLastError());
  // splits cover max_seq_len in whole pages
  int chunk = (max_seq_len + splits - 1) / splits;
  chunk = (chunk + page_size - 1) / page_size * page_size;
  int shift = 0;
  while ((1 << shift) < page_size) ++shift;
  PagedArgs a;
  a.base = DecodeArgs{q, nullptr, nullptr, mem, w_count, out, n_eff, conf, B, Hq, max_seq_len,
                      d, cc, splits, chunk, static_cast<float*>(workspace), seq_lens};
  a.k_pages = k_pages;
  a.v_pages = v_pages;
  a.block_table = block_table;
  a.Hkv = Hkv;
  a.page_shift = shift;
  a.num_pages = num_pages;
  a.max_pages = max_pages;
  a.status = status;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const long long rows = (long long)num_pages * Hkv * page_size;
  if (dtype == POLAR_BF16 && rows < INT_MAX) {
    // tensor-core split: the cache read as [rows, d] through two TMA maps
    CUtensorMap mk, mv;
    const int box = page_size < kPagedTcStageKeys ? page_size : kPagedTcStageKeys;
    if (!make_map_2d(&mk, k_pages, rows, d, box) || !make_map_2d(&mv, v_pages, rows, d, box))
      return POLAR_ERR_CUDA;
    st = cuda_status("paged decode split (tcgen05) launch", launch_decode_paged_tc(a, mk, mv, s));
  } else {
    st = cuda_status("paged decode split launch", launch_decode_paged_split(a, dtype, s));
  }
  if (st != POLAR_OK) return st;
  return cuda_status("paged decode combine launch", launch_decode_combine(a.base, dtype, s));
}

int polar_memory_step(float* state, const void* q, const void* k, const void* v,
                      const float* alpha, const float* beta, void* mem, int B, int H, int T,
                      int d, int dtype, float eps, void* stream) {
  if (B < 0 || H < 0 || T < 0 || !(eps > 0.f) || !std::isfinite(eps)) return POLAR_ERR_INVALID;
  if (dtype != POLAR_F32 && dtype != POLAR_BF16) return POLAR_ERR_UNSUPPORTED;
  if (d != 64 && d != 128) return POLAR_ERR_UNSUPPORTED;
  if ((long long)B * H > INT_MAX) return POLAR_ERR_UNSUPPORTED;
  if ((long long)B * H * T == 0) return POLAR_OK;
  if (!state || !q || !k || !v || !alpha || !beta || !mem) return POLAR_ERR_INVALID;
  if (!aligned16(state) || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(mem) ||
      (reinterpret_cast<uintptr_t>(alpha) & 3u) || (reinterpret_cast<uintptr_t>(beta) & 3u))
    return POLAR_ERR_MISALIGNED;
  int st = check_device(nullptr);
  if (st != POLAR_OK) return st;
  MemoryArgs a{state, q, k, v, alpha, beta, mem, B, H, T, d, eps};
  return cuda_status("memory step launch",
                     launch_memory_step(a, dtype, static_cast<cudaStream_t>(stream)));
}

size_t polar_attn_bwd_workspace_bytes(int B, int H, int T, int d) {
  if (B < 0 || H < 0 || T < 0 || (d != 64 && d != 128)) return 0;
  const size_t f32 = bwd_workspace_floats(B, H, T, d) * sizeof(float);
  const size_t tc = bwd_tc_layout(nullptr, B, H, T, d).bytes;
  return f32 > tc ? f32 : tc;
}

int polar_attn_bwd(const void* q, const void* k, const void* v, const float* w_count,
                   const void* dout, float* dq, float* dk, float* dv, float* dw_count, int B,
                   int H, int T, int d, int dtype, const polar_consts_t* c, void* workspace,
                   size_t workspace_bytes, void* stream) {
  if (B < 0 || H < 0 || T < 0) return POLAR_ERR_INVALID;
  if (dtype != POLAR_F32 && dtype != POLAR_BF16) return POLAR_ERR_UNSUPPORTED;
  if (d != 64 && d != 128) return POLAR_ERR_UNSUPPORTED;
  const polar_consts_t cc = c ? *c : defaults();
  if (!consts_ok(cc)) return POLAR_ERR_INVALID;
  if ((long long)B * H * T == 0) return POLAR_OK;
  if ((long long)B * H > INT_MAX / 64 || T > (1 << 28)) return POLAR_ERR_UNSUPPORTED;
  if (!q || !k || !v || !w_count || !dout || !dq || !dk || !dv || !dw_count)
    return POLAR_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dout) || !aligned16(dq) ||
      !aligned16(dk) || !aligned16(dv) || !aligned16(w_count) || !aligned16(dw_count))
    return POLAR_ERR_MISALIGNED;
  const size_t need = polar_attn_bwd_workspace_bytes(B, H, T, d);
  if (!workspace || workspace_bytes < need) return POLAR_ERR_WORKSPACE;
  if (!aligned16(workspace)) return POLAR_ERR_MISALIGNED;
  int st = check_device(nullptr);
  if (st != POLAR_OK) return st;
  BwdArgs a{q, k, v, dout, w_count, dq, dk, dv, dw_count, B, H, T, d, cc,
            static_cast<float*>(workspace), status_word()};
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == POLAR_F32) return cuda_status("backward launch", launch_bwd(a, dtype, s));
  // bf16: the forward kernel in backward mode, then the tensor-core tiles
  const BwdTcLayout w = bwd_tc_layout(workspace, B, H, T, d);
  if (!a.status) return cuda_status("status word", cudaErrorInvalidSymbol);
  CUtensorMap maps[4];
  const void* bases[4] = {q, k, v, w.da};
  for (int i = 0; i < 4; ++i)
    if (!make_map(&maps[i], bases[i], B * H, T, d)) return POLAR_ERR_CUDA;
  FwdArgs f{q, k, v, nullptr, w_count, nullptr, nullptr, nullptr, B, H, T, d, cc, a.status};
  f.dout = dout;
  f.da = w.da;
  f.grad_rows = w.rows;
  f.dw_part = w.dw_part;
  st = cuda_status("backward row pass",
                   launch_fwd_tc(f, maps[0], maps[1], maps[2], maps[0], s));
  if (st != POLAR_OK) return st;
  return cuda_status("backward tile launch", launch_bwd_tc(a, w, maps, s));
}

int polar_attn_bwd_stats(const void* q, const void* k, const void* v, const void* mem,
                         const float* w_count, const void* out, const float* n_eff,
                         const float* conf, const float* stats, const void* dout, float* dq,
                         float* dk, float* dv, float* dw_count, int B, int H, int T, int d,
                         int dtype, const polar_consts_t* c, void* workspace,
                         size_t workspace_bytes, void* stream) {
  if (B < 0 || H < 0 || T < 0) return POLAR_ERR_INVALID;
  if (dtype != POLAR_BF16) {
    set_last_error("polar_attn_bwd_stats: bf16 only (fp32: polar_attn_bwd)");
    return POLAR_ERR_UNSUPPORTED;
  }
  if (d != 64 && d != 128) return POLAR_ERR_UNSUPPORTED;
  const polar_consts_t cc = c ? *c : defaults();
  if (!consts_ok(cc)) return POLAR_ERR_INVALID;
  if ((long long)B * H * T == 0) return POLAR_OK;
  if ((long long)B * H > INT_MAX / 64 || T > (1 << 28)) return POLAR_ERR_UNSUPPORTED;
  if (!q || !k || !v || !mem || !w_count || !out || !n_eff || !conf || !stats || !dout || !dq ||
      !dk || !dv || !dw_count)
    return POLAR_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(mem) || !aligned16(out) ||
      !aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
      !aligned16(w_count) || !aligned16(dw_count) || (reinterpret_cast<uintptr_t>(stats) & 7u))
    return POLAR_ERR_MISALIGNED;
  const size_t need = polar_attn_bwd_workspace_bytes(B, H, T, d);
  if (!workspace || workspace_bytes < need) return POLAR_ERR_WORKSPACE;
  if (!aligned16(workspace)) return POLAR_ERR_MISALIGNED;
  int st = check_device(nullptr);
  if (st != POLAR_OK) return st;
  BwdArgs a{q, k, v, dout, w_count, dq, dk, dv, dw_count, B, H, T, d, cc,
            static_cast<float*>(workspace), status_word()};
  if (!a.status) return cuda_status("status word", cudaErrorInvalidSymbol);
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const BwdTcLayout w = bwd_tc_layout(workspace, B, H, T, d);
  CUtensorMap maps[4];
  const void* bases[4] = {q, k, v, w.da};
  for (int i = 0; i < 4; ++i)
    if (!make_map(&maps[i], bases[i], B * H, T, d)) return POLAR_ERR_CUDA;
  const SavedRows sv{out, mem, n_eff, conf, stats};
  st = cuda_status("backward row pass", launch_bwd_rows_saved(a, sv, w, s));
  if (st != POLAR_OK) return st;
  return cuda_status("backward tile launch", launch_bwd_tc(a, w, maps, s));
}

int polar_attn_combine(const float* partials, int num_splits, const void* q, const void* mem,
                       const float* w_count, void* out, float* n_eff, float* conf, int B, int H,
                       int Tkv, int d, int dtype, const polar_consts_t* c, void* stream) {
  if (B < 0 || H < 0 || Tkv < 1 || num_splits < 1) return POLAR_ERR_INVALID;
  if (dtype != POLAR_F32 && dtype != POLAR_BF16) return POLAR_ERR_UNSUPPORTED;
  if (d != 64 && d != 128) return POLAR_ERR_UNSUPPORTED;
  if (!decode_sizes_ok(B, H, Tkv, d)) return POLAR_ERR_UNSUPPORTED;
  const polar_consts_t cc = c ? *c : defaults();
  if (!consts_ok(cc)) return POLAR_ERR_INVALID;
  if ((long long)B * H == 0) return POLAR_OK;
  if (!partials || !q || !mem || !w_count || !out || !n_eff) return POLAR_ERR_INVALID;
  if (!aligned16(partials) || !aligned16(q) || !aligned16(mem) || !aligned16(w_count) ||
      !aligned16(out))
    return POLAR_ERR_MISALIGNED;
  int st = check_device(nullptr);
  if (st != POLAR_OK) return st;
  DecodeArgs a{q, nullptr, nullptr, mem, w_count, out, n_eff, conf, B, H, Tkv, d, cc,
               num_splits, 0, const_cast<float*>(partials)};
  return cuda_status("combine launch",
                     launch_decode_combine(a, dtype, static_cast<cudaStream_t>(stream)));
}

int polar_attn_device_status(int reset) {
  int v = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return -1;
  if (cudaMemcpyFromSymbol(&v, g_status, sizeof(int)) != cudaSuccess) return -1;
  if (reset) {
    const int z = 0;
    if (cudaMemcpyToSymbol(g_status, &z, sizeof(int)) != cudaSuccess) return -1;
  }
  return v;
}

int polar_attn_selftest_wait_timeout(int limit_us, void* stream) {
  if (limit_us < 1 || limit_us > 1000000) return POLAR_ERR_INVALID;
  int st = check_device(nullptr);
  if (st != POLAR_OK) return st;
  int khz = 0, dev = 0;
  cudaGetDevice(&dev);
  if (cudaDeviceGetAttribute(&khz, cudaDevAttrClockRate, dev) != cudaSuccess || khz <= 0)
    khz = 2000000;
  const long long cycles = (long long)khz * limit_us / 1000;
  int* status = status_word();
  if (!status) return cuda_status("cudaGetSymbolAddress", cudaGetLastError());
  return cuda_status("self-test launch",
                     launch_selftest_wait(cycles, status, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace polar {

namespace {
__global__ void selftest_wait_kernel(long long limit_cycles, int* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // nothing arrives on `bar`: the bounded wait must give up
    if (!mbar_wait(&bar, 0, &abort_flag, status, limit_cycles)) atomicExch(status, kStatusSelftest);
  }
}
}  // namespace

cudaError_t launch_selftest_wait(long long limit_cycles, int* status, cudaStream_t s) {
  selftest_wait_kernel<<<1, 32, 0, s>>>(limit_cycles, status);
  return cudaGetLastError();
}

}  // namespace polar
