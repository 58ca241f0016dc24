// Split-KV decode whose partial states live in a fixed, library-owned device
// array instead of a caller-provided workspace.
//
// Who needs it: callers that cannot allocate device memory when they run the
// decode step.  Typical cases are a host framework or plugin interface that
// owns all device memory and hands the kernel only its input and output
// buffers, and latency-critical serving loops where cudaMalloc (which may
// synchronise the whole device) is not allowed after start-up.  Such callers
// still pass q, the KV cache, mem, w_count and the outputs; the scratch for
// the split partials comes from the array below.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds POLAR_ATTN_STATIC_SCRATCH_BYTES of it until the process
// exits.  Its name in host code is only a host-side stand-in, never a device
// address, so the device address is looked up with cudaGetSymbolAddress
// once per device (with that device current) and cached.
#include <cstdio>
#include <mutex>

#include "polar_device.cuh"
#include "polar_internal.h"

namespace polar {

namespace {

constexpr size_t kScratchBytes = POLAR_ATTN_STATIC_SCRATCH_BYTES;

// Partials [B, H, splits, d + 4] of the most recent call on this device.
static __device__ __align__(256) float g_decode_scratch[kScratchBytes / sizeof(float)];

constexpr int kMaxDevices = 256;
std::mutex g_scratch_mu;
float* g_scratch_addr[kMaxDevices] = {};  // device address per device ordinal

// Device address of g_decode_scratch on device `dev` (the current device).
// The first call on a device resolves it; later calls reuse the cached value.
int scratch_address(int dev, float** out) {
  if (dev < 0 || dev >= kMaxDevices) return POLAR_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess || !p) {
      char msg[160];
      std::snprintf(msg, sizeof(msg), "cudaGetSymbolAddress(static decode scratch) failed (%d: %s)",
                    (int)e, cudaGetErrorString(e));
      set_last_error(msg);
      return POLAR_ERR_CUDA;
    }
    g_scratch_addr[dev] = static_cast<float*>(p);
  }
  *out = g_scratch_addr[dev];
  return POLAR_OK;
}

}  // namespace
}  // namespace polar

using namespace polar;

extern "C" int polar_attn_decode_static_scratch(const void* q, const void* k_cache,
                                                const void* v_cache, const void* mem,
                                                const float* w_count, void* out, float* n_eff,
                                                float* conf, int B, int H, int Tkv, int d,
                                                int dtype, const polar_consts_t* c,
                                                int num_splits, void* stream) {
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

  // one record of d + 4 floats per (b, h, split)
  const size_t rec_bytes = (size_t)(d + 4) * sizeof(float);
  const size_t per_split = (size_t)B * H * rec_bytes;
  int splits = num_splits;
  if (splits == 0) {
    // automatic choice, lowered until the partials fit the static array
    splits = auto_splits(B * H, Tkv, sms);
    const size_t fit = kScratchBytes / per_split;
    if ((size_t)splits > fit) splits = (int)fit;
  }
  if (splits < 1 || (size_t)splits * per_split > kScratchBytes) {
    char msg[200];
    std::snprintf(msg, sizeof(msg),
                  "decode partials need %zu bytes (B*H=%lld, splits=%d, d=%d) but the static "
                  "scratch holds %zu bytes",
                  (size_t)(splits < 1 ? 1 : splits) * per_split, (long long)B * H,
                  splits < 1 ? 1 : splits, d, kScratchBytes);
    set_last_error(msg);
    return POLAR_ERR_WORKSPACE;
  }

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return POLAR_ERR_DEVICE;
  float* scratch = nullptr;
  st = scratch_address(dev, &scratch);
  if (st != POLAR_OK) return st;

  // Every split record is fully written by the split kernel before the
  // combine reads it, so nothing in the array has to start at zero.
  DecodeArgs a{q, k_cache, v_cache, mem, w_count, out, n_eff, conf, B, H, Tkv, d, cc,
               splits, (Tkv + splits - 1) / splits, scratch};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_decode_split(a, dtype, s);
  if (e == cudaSuccess) e = launch_decode_combine(a, dtype, s);
  if (e != cudaSuccess) {
    char msg[160];
    std::snprintf(msg, sizeof(msg), "static-scratch decode launch failed (%d: %s)", (int)e,
                  cudaGetErrorString(e));
    set_last_error(msg);
    return POLAR_ERR_CUDA;
  }
  return POLAR_OK;
}
