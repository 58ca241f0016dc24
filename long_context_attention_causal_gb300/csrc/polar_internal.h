// Internal launch interface between the C ABI (polar_api.cu) and the kernel
// translation units.  Arguments here are already validated.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "polar_attn.h"

namespace polar {

struct FwdArgs {
  const void *q, *k, *v, *mem;
  const float* w_count;
  void* out;
  float* n_eff;
  float* conf;  // may be null
  int B, H, T, d;
  polar_consts_t c;
  int* status;  // device address of the library's status word
  float* stats = nullptr;  // optional [B, H, T, 2]: logsumexp, |a| (bf16 path)
  // Backward mode of the bf16 kernel (dout != null): instead of out, n_eff
  // and conf it writes dA, the per-row gradient record and the count * g
  // partials (polar_grad.cuh).
  const void* dout = nullptr;
  void* da = nullptr;
  float* grad_rows = nullptr;
  float* dw_part = nullptr;
};

struct DecodeArgs {
  const void *q, *k, *v, *mem;
  const float* w_count;
  void* out;
  float* n_eff;
  float* conf;  // may be null
  int B, H, Tkv, d;
  polar_consts_t c;
  int splits;      // >= 1
  int chunk;       // keys per split
  float* partials; // [B, H, splits, d + 4]
  const int* seq_lens = nullptr;  // [B] per-sequence key counts (paged), else Tkv
};

struct PagedArgs {
  DecodeArgs base;  // q, mem, out, n_eff, conf, w_count, partials; H = Hq, Tkv = max_seq_len
  const void *k_pages, *v_pages;  // [num_pages, Hkv, page, d]
  const int* block_table;         // [B, max_pages]
  int Hkv, page_shift, num_pages, max_pages;
  int* status;
};

struct MemoryArgs {
  float* state;                   // [B, H, d, d] fp32, updated in place
  const void *q, *k, *v;          // [B, H, T, d]
  const float *alpha, *beta;      // [B, H, T]
  void* mem;                      // [B, H, T, d]
  int B, H, T, d;
  float eps;
};

struct BwdArgs {
  const void *q, *k, *v, *dout;  // [B, H, T, d] of dtype
  const float* w_count;          // [H, d]
  float *dq, *dk, *dv;           // [B, H, T, d] fp32
  float* dw;                     // [H, d] fp32
  int B, H, T, d;
  polar_consts_t c;
  float* workspace;              // bwd_workspace_floats(...) floats
  int* status = nullptr;         // device status word (tensor-core path)
};

// Backward of the causal prefill, fp32 inputs (FP32 pipes).
size_t bwd_workspace_floats(int B, int H, int T, int d);
cudaError_t launch_bwd(const BwdArgs& a, int dtype, cudaStream_t s);

// Backward of the causal prefill, bf16 inputs (tensor cores).  The forward
// kernel in backward mode fills the workspace (dA, row records, count * g
// partials); the tile kernels then write dQ, dK, dV and dw.
struct BwdTcLayout {
  void* da;        // [BH, T, d] bf16
  float* rows;     // row records, pair blocks (polar_grad.cuh)
  float* dw_part;  // [BH, ceil(T / 32), d]
  size_t bytes;
};
BwdTcLayout bwd_tc_layout(void* workspace, int B, int H, int T, int d);
// Row pass of the backward from the forward's saved outputs (bf16): fills
// the same workspace as the forward kernel's backward mode.
struct SavedRows {
  const void *out, *mem;  // [B, H, T, d] bf16
  const float *n_eff, *conf, *stats;
};
cudaError_t launch_bwd_rows_saved(const BwdArgs& a, const SavedRows& sv, const BwdTcLayout& w,
                                  cudaStream_t s);
// maps: q, k, v, dA (128-row boxes)
cudaError_t launch_bwd_tc(const BwdArgs& a, const BwdTcLayout& w, const CUtensorMap* maps,
                          cudaStream_t s);

// Gated-delta memory steps over T tokens, state updated in place.
cudaError_t launch_memory_step(const MemoryArgs& a, int dtype, cudaStream_t s);

// Paged, grouped-query split kernel (combine: launch_decode_combine).
cudaError_t launch_decode_paged_split(const PagedArgs& a, int dtype, cudaStream_t s);
// The same split on the tensor cores (bf16; cache rows num_pages * Hkv * page
// addressable as int32).  mk, mv: 2-D maps [rows, d] with a {64, min(page,
// kPagedTcStageKeys)} box and 128-byte swizzle.
constexpr int kPagedTcStageKeys = 64;
cudaError_t launch_decode_paged_tc(const PagedArgs& a, const CUtensorMap& mk,
                                   const CUtensorMap& mv, cudaStream_t s);

// Heads per group in the multi-wave CTA orders of the tensor-core kernels
// (each group's streamed operands kept in L2): the largest divisor of BH
// whose heads' per_head_bytes fit a third of the current device's L2 (a
// short search below that bound; a near miss keeps the bound), at least 1.
int l2_head_group(int BH, double per_head_bytes);

// bf16 causal prefill on the tensor cores (tcgen05 + TMEM + TMA).
// map_o: the output [BH, T, d] with the same 128-row boxes (the forward
// epilogue's TMA store; unused in backward mode).
cudaError_t launch_fwd_tc(const FwdArgs& a, const CUtensorMap& map_q,
                          const CUtensorMap& map_k, const CUtensorMap& map_v,
                          const CUtensorMap& map_o, cudaStream_t s);

// fp32 causal prefill on the FP32 pipes.
cudaError_t launch_fwd_f32(const FwdArgs& a, cudaStream_t s);

// Split-KV decode: partial states per (b, h, split), then the combine.
cudaError_t launch_decode_split(const DecodeArgs& a, int dtype, cudaStream_t s);
cudaError_t launch_decode_combine(const DecodeArgs& a, int dtype, cudaStream_t s);

// Host helpers shared by the entry points (defined in polar_api.cu).
bool aligned16(const void* p);
bool consts_ok(const polar_consts_t& c);
polar_consts_t defaults();
int check_device(int* num_sms);
int auto_splits(int BH, int Tkv, int num_sms);
bool decode_sizes_ok(int B, int H, int Tkv, int d);
void set_last_error(const char* msg);

// Bounded-wait self test (one thread, a barrier nothing completes).
cudaError_t launch_selftest_wait(long long limit_cycles, int* status, cudaStream_t s);

}  // namespace polar
