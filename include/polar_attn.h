/*
 * polar_attn.h - C ABI of the GB300 (sm_103a) causal Polar Attention library
 * (libpolarattn.so).
 *
 * The operation is the fused causal Polar Attention forward of "ATMA:
 * Length-Invariant Language Modeling via Polar Attention and Gated-Delta
 * Compression Memory" (technical summaries):
 *   §2.1      out = content + count + memory (three additive streams);
 *   §2.1 (1)  direction channel: the sum of matched values projected onto the
 *             unit sphere, with a length temperature and an
 *             extreme-value-corrected null floor on the logits;
 *   §2.1 (2)  magnitude channel: participation ratio (inverse Simpson index)
 *             n_eff, gated by detection confidence, through a bounded,
 *             monotone, saturating tanh of log;
 *   §2.1 (3)  memory channel: an additive stream (an input here);
 *   §2.2      fused kernel: n_eff computed online with streaming accumulators
 *             and squared correction factors, O(block) memory;
 *   §2        decoder-only stack, hence causal attention.
 * The pages give no equations; this library computes the pinned reading, per
 * query row i of head h with n visible keys (n = i + 1 in prefill, n = Tkv in
 * decode):
 *   tau   = max(1, ln n / log_t0)
 *   s_j   = tau * (q_i . k_j) / sqrt(d)                       j < n
 *   p_j   = exp(s_j - m) / l,  m = max_j s_j,  l = sum_j exp(s_j - m)
 *   n_eff = 1 / sum_j p_j^2
 *   b     = tau * sigma_k * |q_i| / sqrt(d) * sqrt(2 ln n)     (null floor;
 *           floor_order 2: tau sigma_k |q_i|/sqrt(d) * [r - (ln ln n +
 *           ln 4 pi)/(2 r) + gamma/r], r = sqrt(2 ln n), the second-order
 *           expected maximum of n iid N(0,1); 0 at n = 1)
 *   conf  = sigmoid(m + ln l - b)
 *   u     = a / max(|a|, eps),  a = sum_j p_j v_j
 *   out_i = u + conf * tanh(ln n_eff / kappa) * w_count[h] + mem_i
 *
 * Conventions for every call:
 *   - All tensor pointers are DEVICE pointers owned by the caller, contiguous
 *     row-major, and 16-byte aligned.  The library allocates no device memory
 *     and keeps no host state between calls (TMA descriptors are built per
 *     call), so calls are thread-safe.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls
 *     enqueue work and return; they never synchronise.
 *   - The return value is a status (polar_status_t).  On any non-zero status
 *     nothing was launched (except POLAR_ERR_CUDA, reported by the launch
 *     itself).  Nothing aborts the process.
 *   - dtype selects the element type of q, k, v, mem and out: POLAR_F32 or
 *     POLAR_BF16.  n_eff, conf and w_count are always fp32.
 *   - d (head dimension) must be 64 or 128.
 */
#ifndef POLAR_ATTN_H
#define POLAR_ATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct polar_consts_t {
  float log_t0;  /* ln T0, temperature neutral length; default ln 2048 (§3:
                    training length 2K) */
  float kappa;   /* tanh-of-log saturation scale; default ln 2048 */
  float sigma_k; /* null-model std of a key component; default 1 */
  float eps;     /* guard of the unit-sphere projection; default 1e-6 */
  int floor_order; /* null floor: 1 = leading order sigma*sqrt(2 ln n)
                      (default; 0 is read as 1), 2 = second-order expected
                      maximum (Gumbel location + Euler-gamma shift) */
} polar_consts_t;

enum { POLAR_F32 = 0, POLAR_BF16 = 1 };

typedef enum polar_status_t {
  POLAR_OK = 0,
  POLAR_ERR_INVALID = 1,     /* null pointer, negative size, bad constant */
  POLAR_ERR_UNSUPPORTED = 2, /* d not in {64, 128}, unknown dtype, too large */
  POLAR_ERR_MISALIGNED = 3,  /* a tensor pointer not 16-byte aligned */
  POLAR_ERR_WORKSPACE = 4,   /* decode workspace missing or too small */
  POLAR_ERR_CUDA = 5,        /* the CUDA runtime refused the launch */
  POLAR_ERR_DEVICE = 6       /* no usable sm_103 device */
} polar_status_t;

/* Fill *c with the default constants (log_t0 = kappa = ln 2048, sigma_k = 1,
 * eps = 1e-6, floor_order = 1).  Always succeeds for a non-null c. */
int polar_attn_default_consts(polar_consts_t* c);

/*
 * Causal prefill (§2.1, §2.2).
 *   q, k, v, mem : [B, H, T, d] of dtype          (read)
 *   w_count      : [H, d] fp32                    (read; count direction per head)
 *   out          : [B, H, T, d] of dtype          (written)
 *   n_eff        : [B, H, T] fp32                 (written)
 *   conf         : [B, H, T] fp32 or NULL         (written if non-null; the gate)
 * B, H, T >= 0 (any zero: nothing to do, POLAR_OK).  Row i sees keys 0..i.
 * bf16 runs on the tensor cores (tcgen05, fp32 accumulation, P rounded to
 * bf16 for the PV product); fp32 runs on the FP32 pipes.  Memory beyond the
 * inputs and outputs: none (no T x T buffer, no workspace).
 */
int polar_attn_fwd(const void* q, const void* k, const void* v, const void* mem,
                   const float* w_count, void* out, float* n_eff, float* conf,
                   int B, int H, int T, int d, int dtype,
                   const polar_consts_t* c, void* stream);

/*
 * Causal prefill from HOST buffers: the results of polar_attn_fwd, with the
 * copies in and out overlapped with the kernels.  The (b, h) range is cut
 * into `num_pieces` runs of consecutive slices (0: automatic, about three
 * waves of prefill CTAs per piece, 2 to 8 pieces; at most 48), and the last run
 * is then cut in halves, quarters, ... down to one slice, since its kernel
 * and copy-out are all that runs after the last copy in; piece i is copied
 * in on an internal stream, computed once it has landed (even pieces on
 * `stream`, odd ones on an internal stream forked from it, so that two
 * pieces' kernels can overlap), and copied out on another internal stream
 * while later pieces compute.
 *   q, k, v, mem, w_count, out, n_eff, conf : HOST pointers, the shapes and
 *       dtypes of polar_attn_fwd (conf may be NULL).  Page-locked memory
 *       (cudaHostAlloc, cudaHostRegister) lets the copies run asynchronously
 *       and overlap; pageable memory gives the same results, serialised.
 *   workspace : polar_attn_fwd_host_workspace_bytes(B, H, T, d, dtype) bytes
 *       of device memory, 256-byte aligned, caller-owned: device copies of
 *       the inputs and outputs (contents on entry do not matter).
 * Stream-ordered: the work starts after what `stream` already holds, and
 * `stream` completes only after the last copy out; the host buffers hold
 * the results once `stream` has been synchronised, and must not be touched
 * before.  The kernel launches are those of polar_attn_fwd with B, H and
 * w_count narrowed to the piece, so each output element is bit-identical to
 * polar_attn_fwd's.  Calls on one device are enqueued one at a time (an
 * internal lock) and their copies in (and out) run in call order on shared
 * internal streams; a call waits only for its own `stream`, so consecutive
 * calls on two streams with two workspaces overlap (one call's copies in
 * with the previous call's last pieces and copies out), which keeps the
 * host link busy across steps.  Returns POLAR_ERR_WORKSPACE if workspace is
 * missing or too small, POLAR_ERR_MISALIGNED if it is not 256-byte aligned.
 */
int polar_attn_fwd_host(const void* q, const void* k, const void* v, const void* mem,
                        const float* w_count, void* out, float* n_eff, float* conf,
                        int B, int H, int T, int d, int dtype,
                        const polar_consts_t* c, int num_pieces, void* workspace,
                        size_t workspace_bytes, void* stream);

/* Workspace bytes of polar_attn_fwd_host (0 for invalid sizes). */
size_t polar_attn_fwd_host_workspace_bytes(int B, int H, int T, int d, int dtype);

/*
 * Split-KV decode (§2.1; §2.2 decode kernel): one query per (b, h) against a
 * cache of Tkv keys, all visible (n = Tkv; the cache holds the current token).
 *   q, mem           : [B, H, d] of dtype
 *   k_cache, v_cache : [B, H, Tkv, d] of dtype
 *   w_count          : [H, d] fp32
 *   out              : [B, H, d] of dtype;  n_eff, conf : [B, H] fp32
 *                      (conf may be NULL)
 *   num_splits       : chunks the cache is cut into (0 = automatic choice,
 *                      polar_attn_decode_num_splits); each chunk yields one
 *                      partial state, merged by the combine step
 *   workspace        : device buffer of at least
 *                      polar_attn_decode_workspace_bytes(B, H, Tkv, d,
 *                      num_splits) bytes, 16-byte aligned; it receives the
 *                      partials (layout below) and may be reused after the
 *                      stream has passed this call.
 * Launches the split kernel, then the combine kernel, on `stream`.
 * Tkv >= 1; B or H = 0 is a no-op.
 */
int polar_attn_decode(const void* q, const void* k_cache, const void* v_cache,
                      const void* mem, const float* w_count, void* out,
                      float* n_eff, float* conf, int B, int H, int Tkv, int d,
                      int dtype, const polar_consts_t* c, int num_splits,
                      void* workspace, size_t workspace_bytes, void* stream);

/* Split count chosen when num_splits = 0, for the current device.  Returns a
 * value >= 1, or 0 for invalid sizes. */
int polar_attn_decode_num_splits(int B, int H, int Tkv, int d);

/* Workspace bytes polar_attn_decode needs (num_splits = 0: automatic
 * choice).  Returns 0 for invalid sizes. */
size_t polar_attn_decode_workspace_bytes(int B, int H, int Tkv, int d,
                                         int num_splits);

/*
 * Combine step of split-KV decode: merges num_splits partial states per
 * (b, h) and applies the epilogue (null floor, gate, n_eff, count, direction,
 * memory) with n = Tkv.
 *   partials : [B, H, num_splits, d + 4] fp32.  Record of split s:
 *              { m, l, Q2, 0, acc[0..d) } with, over the split's keys j,
 *              l = sum exp(s_j - m), Q2 = sum exp(2 (s_j - m)),
 *              acc = sum exp(s_j - m) v_j, and m a reference logit (the
 *              running max); an empty split has m = -inf, l = Q2 = 0.
 *              Merging rebases each record on M = max m with weight
 *              w = exp(m - M): w on l and acc, w^2 on Q2 (§2.2, squared
 *              correction factors).
 *   q, mem   : [B, H, d] of dtype (q gives |q| for the null floor)
 *   other arguments as in polar_attn_decode.
 */
int polar_attn_combine(const float* partials, int num_splits, const void* q,
                       const void* mem, const float* w_count, void* out,
                       float* n_eff, float* conf, int B, int H, int Tkv, int d,
                       int dtype, const polar_consts_t* c, void* stream);

/*
 * Split-KV decode against a PAGED cache with grouped-query heads (ATMA §2.2:
 * the decode kernel reads paged KV blocks directly and shares each KV read
 * among the query heads of a group).
 *   q, mem      : [B, Hq, d] of dtype;  out : [B, Hq, d] of dtype
 *   k_pages,
 *   v_pages     : [num_pages, Hkv, page_size, d] of dtype (a page holds
 *                 page_size consecutive tokens of every KV head)
 *   block_table : [B, max_pages] int32, device: physical page of logical
 *                 page p of sequence b (entries past the sequence unused)
 *   seq_lens    : [B] int32, device: keys visible to sequence b (its cache
 *                 length, the current token included), in [1, max_seq_len]
 *   w_count     : [Hq, d] fp32;  n_eff, conf : [B, Hq] fp32 (conf may be NULL)
 * Query head h reads KV head h / (Hq / Hkv); Hq / Hkv must be 1, 2, 4 or 8.
 * page_size: a power of two in [8, 1024]; max_seq_len <= max_pages *
 * page_size (it sizes the splits).  Key j of sequence b is row j % page_size
 * of page block_table[b][j / page_size]; n = seq_lens[b] per sequence.
 * A page index outside [0, num_pages) is not read (its keys are skipped) and
 * a length outside [1, max_seq_len] is clamped on the device; either records
 * status 3 in polar_attn_device_status and leaves that row's result
 * meaningless (a row with no visible key returns out = mem, n_eff = conf = 0).
 * workspace: at least polar_attn_decode_paged_workspace_bytes(...) bytes;
 * num_splits = 0 chooses automatically.  Launches the paged split kernel
 * and the combine kernel on `stream`.  B = 0 is a no-op.  bf16 pools of
 * fewer than 2^31 rows (num_pages * Hkv * page_size) run the split on the
 * tensor cores (scores and P V in fp32 accumulation, P rounded to bf16, as
 * in the prefill); fp32, and larger bf16 pools, on the FP32 pipes.
 */
int polar_attn_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                            const int* block_table, const int* seq_lens,
                            const void* mem, const float* w_count, void* out,
                            float* n_eff, float* conf, int B, int Hq, int Hkv,
                            int d, int page_size, int num_pages, int max_pages,
                            int max_seq_len, int dtype, const polar_consts_t* c,
                            int num_splits, void* workspace,
                            size_t workspace_bytes, void* stream);

/* Split count polar_attn_decode_paged picks for num_splits = 0 (>= 1), or 0
 * for invalid sizes. */
int polar_attn_decode_paged_num_splits(int B, int Hkv, int max_seq_len, int d);

/* Workspace bytes of polar_attn_decode_paged: B * Hq * splits * (d + 4) * 4
 * (num_splits = 0: automatic choice).  0 for invalid sizes. */
size_t polar_attn_decode_paged_workspace_bytes(int B, int Hq, int Hkv,
                                               int max_seq_len, int d,
                                               int num_splits);

/*
 * Backward of the causal prefill: gradients of out (n_eff and conf are
 * diagnostics and carry none).  The pages train the model (ATMA §3) but
 * give no detail of the gradient; it follows from the forward pinned above:
 * through the unit-sphere projection, the softmax (with the count's
 * dependence on logsumexp and on Q2 = sum p^2), the null floor's dependence
 * on |q|, and count * w_count.  d out / d mem is the identity, so dmem is
 * the caller's dout (not written).
 *   q, k, v, dout : [B, H, T, d] of dtype (the forward's inputs)
 *   w_count       : [H, d] fp32
 *   dq, dk, dv    : [B, H, T, d] fp32 (written)
 *   dw_count      : [H, d] fp32 (written: sum over b and rows)
 *   workspace     : polar_attn_bwd_workspace_bytes(B, H, T, d) bytes,
 *                   device, 16-byte aligned, caller-owned; its contents
 *                   on entry do not affect the results
 * bf16 inputs run on the tensor cores: the prefill kernel recomputes each
 * row's streaming state and writes dA (bf16) and the row's gradient
 * scalars to the workspace, then dK/dV (per 128-key tile) and dQ (per
 * 128-query tile) take bf16 products of dA, P and dS with fp32
 * accumulation.  fp32 inputs run in fp32 on the FP32 pipes.
 * The bf16 path runs its dQ kernel beside the dK/dV kernel on a side stream
 * that the library keeps per device, forked from `stream` and joined back
 * into it with events (stream order is kept: later work on `stream` starts
 * after both).  That side stream is shared by every caller on the device:
 * backward calls on different caller streams of one device serialise on
 * it, and an eager backward call made while another thread captures a
 * backward (or polar_attn_bwd_stats) into a CUDA graph on the same device
 * may fail or break that capture; capturing itself is supported.
 * Returns POLAR_ERR_WORKSPACE if workspace_bytes is too small,
 * POLAR_ERR_MISALIGNED for pointers not 16-byte aligned; kernel-side wait
 * timeouts are reported by polar_attn_device_status.
 */
int polar_attn_bwd(const void* q, const void* k, const void* v, const float* w_count,
                   const void* dout, float* dq, float* dk, float* dv, float* dw_count,
                   int B, int H, int T, int d, int dtype, const polar_consts_t* c,
                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * Training pair for bf16 inputs: the forward that also keeps, per row, the
 * two statistics the backward needs (ATMA §2.2: the kernel's streaming
 * state), and the backward that starts from them instead of recomputing
 * the forward.
 * polar_attn_fwd_stats: as polar_attn_fwd (conf required), plus
 *   stats : [B, H, T, 2] fp32, 8-byte aligned (written): per row the
 *           logsumexp of the scaled logits, m + ln l, and |a|, the norm of
 *           a = sum_j p_j v_j before the unit-sphere projection.
 * polar_attn_bwd_stats: gradients as polar_attn_bwd, from the forward's
 *   inputs, its outputs out, n_eff, conf and stats, and dout.  The
 *   direction is recovered as u = out - count w_count - mem with
 *   count = conf tanh(ln n_eff / kappa), so out must be the forward's
 *   output for the same mem, w_count and constants.  Same workspace
 *   (polar_attn_bwd_workspace_bytes) and error codes as polar_attn_bwd.
 * Both return POLAR_ERR_UNSUPPORTED for fp32 inputs (fp32 callers use
 * polar_attn_fwd and polar_attn_bwd, which recomputes the forward).
 */
int polar_attn_fwd_stats(const void* q, const void* k, const void* v, const void* mem,
                         const float* w_count, void* out, float* n_eff, float* conf,
                         float* stats, int B, int H, int T, int d, int dtype,
                         const polar_consts_t* c, void* stream);
int polar_attn_bwd_stats(const void* q, const void* k, const void* v, const void* mem,
                         const float* w_count, const void* out, const float* n_eff,
                         const float* conf, const float* stats, const void* dout, float* dq,
                         float* dk, float* dv, float* dw_count, int B, int H, int T, int d,
                         int dtype, const polar_consts_t* c, void* workspace,
                         size_t workspace_bytes, void* stream);

/* Workspace bytes of polar_attn_bwd (the larger of the fp32 and bf16
 * paths' needs, about B * H * T * (d + 8) * 4).  0 for invalid sizes. */
size_t polar_attn_bwd_workspace_bytes(int B, int H, int T, int d);

/*
 * Gated-delta memory, in place (ATMA §2.1 item 3: the memory channel, a
 * gated delta rule with L2-normalised keys and queries that bound the
 * update's eigenvalues; §2.2: the in-place step kernel).  For each (b, h)
 * and each of T tokens in order:
 *   k^ = k / max(|k|, eps),  q^ = q / max(|q|, eps)
 *   S  <- alpha S (I - beta k^ k^T) + beta v k^T
 *   mem = S q^          (the memory stream polar_attn_fwd / decode add)
 *   state : [B, H, d, d] fp32, device, read and written in place (S maps
 *           keys to values: row i is value dimension i)
 *   q, k, v, mem : [B, H, T, d] of dtype (T = 1: one decode step)
 *   alpha, beta  : [B, H, T] fp32 gates, expected in [0, 1] (outside that
 *                  range the update is no longer contracting)
 * One read and one write of the state per call.  Tokens are processed in
 * sequence within a head; heads run in parallel.  eps > 0 (e.g. 1e-6).
 */
int polar_memory_step(float* state, const void* q, const void* k, const void* v,
                      const float* alpha, const float* beta, void* mem, int B,
                      int H, int T, int d, int dtype, float eps, void* stream);

/* Size of the library-owned device array used by
 * polar_attn_decode_static_scratch (8 MiB per GPU that loads the library). */
#define POLAR_ATTN_STATIC_SCRATCH_BYTES (8u * 1024u * 1024u)

/*
 * Split-KV decode that allocates nothing and takes no workspace.
 * (No counterpart on the pages: this is a service of the library.)
 * For callers that cannot allocate device memory at the time they decode,
 * e.g. a framework or plugin host that owns all device memory and passes the
 * kernel only its inputs and outputs, or a serving loop that forbids
 * cudaMalloc (which may synchronise the device) after start-up.
 * Same arguments and results as polar_attn_decode, without workspace and
 * workspace_bytes.  The split partials go to a file-scope device array of
 * POLAR_ATTN_STATIC_SCRATCH_BYTES that every GPU loading the library keeps
 * until the process exits.
 *   - Limit: B * H * splits * (d + 4) * 4 bytes must fit the array.  With
 *     num_splits = 0 the automatic split count is lowered until it fits;
 *     if even one split does not fit, or an explicit num_splits does not,
 *     the call returns POLAR_ERR_WORKSPACE (polar_attn_last_error gives the
 *     sizes) and launches nothing.
 *   - The first call on a device looks up the array's device address with
 *     cudaGetSymbolAddress (current device) and caches it; make that first
 *     call before any stream capture on that device.  The cached address
 *     does not survive cudaDeviceReset (the module, and with it the array,
 *     is loaded again, possibly elsewhere): do not call this entry point on
 *     a device after resetting it in the same process.
 *   - All calls on a device share the one array and it keeps the last call's
 *     partials.  Calls whose kernels overlap on the GPU (e.g. on two streams
 *     at once) race on it: serialise them.  Nothing in the array needs to
 *     start at zero; every record is written before it is read.
 *   - Calls no cudaMalloc, cudaFree or allocating library routine.
 */
int polar_attn_decode_static_scratch(const void* q, const void* k_cache,
                                     const void* v_cache, const void* mem,
                                     const float* w_count, void* out,
                                     float* n_eff, float* conf, int B, int H,
                                     int Tkv, int d, int dtype,
                                     const polar_consts_t* c, int num_splits,
                                     void* stream);

/* Static, never-null description of a status code. */
const char* polar_attn_strerror(int status);

/* Kernel-side status of the current device: every wait inside the kernels
 * has a time limit; a kernel whose wait runs out stops early and records a
 * non-zero code here (1 = a pipeline wait timed out, 2 = the self-test wait
 * timed out as intended, 3 = the paged decode met a page index or sequence
 * length outside its bounds).  Synchronises the device.  reset != 0 clears it.
 * Returns the code, or -1 if the device could not be queried. */
int polar_attn_device_status(int reset);

/* Self-test of the bounded wait: launches one thread that waits on a barrier
 * nothing will complete, with a limit of `limit_us` microseconds; the kernel
 * gives up, records code 2 and exits.  Used by tests to show a stuck wait
 * ends with a status instead of a hang. */
int polar_attn_selftest_wait_timeout(int limit_us, void* stream);

/* Text of the last CUDA-level failure (status POLAR_ERR_CUDA) seen by the
 * calling host thread: which call failed and the CUDA error.  Thread-local,
 * never null; "" when nothing has failed on this thread. */
const char* polar_attn_last_error(void);

/* Library ABI version (major * 100 + minor). */
int polar_attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* POLAR_ATTN_H */
