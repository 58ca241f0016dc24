// Causal prefill from host buffers: the (b, h) range is cut into pieces and
// each piece's copy in, kernel and copy out run on separate streams, so that
// the copies of one piece overlap the kernels of the others.  The kernels are
// the ones polar_attn_fwd launches (one launch per piece, alternately on the
// caller's stream and on an internal one forked from it); a piece is a run of
// consecutive (b, h) slices, contiguous in every tensor.
#include <cuda_runtime.h>

#include <climits>
#include <cstddef>
#include <cstdint>
#include <mutex>

#include "polar_internal.h"

namespace polar {
namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxPieces = 64;

// Per device: the copy streams and the events that order the pieces.
// Enqueueing is serialised by the mutex, so one set of events serves every
// call (a wait captures the event's last record when it is enqueued).
struct Pipeline {
  bool ready = false;
  cudaStream_t in = nullptr, out = nullptr, comp = nullptr;
  cudaEvent_t start = nullptr, done = nullptr;
  cudaEvent_t landed[kMaxPieces] = {}, computed[kMaxPieces] = {};
};

std::mutex g_mutex;
Pipeline g_pipe[kMaxDevices];

cudaError_t pipeline_init(Pipeline& p) {
  if (p.ready) return cudaSuccess;
  cudaError_t e = cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p.comp, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.start, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.done, cudaEventDisableTiming);
  for (int i = 0; i < kMaxPieces && e == cudaSuccess; ++i) {
    e = cudaEventCreateWithFlags(&p.landed[i], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.computed[i], cudaEventDisableTiming);
  }
  p.ready = (e == cudaSuccess);
  return e;
}

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

struct Regions {
  size_t q, k, v, mem, out, n_eff, conf, w, total;
};

Regions regions(int B, int H, int T, int d, int dtype) {
  const size_t es = dtype == POLAR_BF16 ? 2 : 4;
  const size_t big = round256((size_t)B * H * T * d * es);
  const size_t row = round256((size_t)B * H * T * sizeof(float));
  Regions r;
  r.q = 0;
  r.k = r.q + big;
  r.v = r.k + big;
  r.mem = r.v + big;
  r.out = r.mem + big;
  r.n_eff = r.out + big;
  r.conf = r.n_eff + row;
  r.w = r.conf + row;
  r.total = r.w + round256((size_t)H * d * sizeof(float));
  return r;
}

// A piece: batches [b0, b0 + nb) with all heads, or heads [h0, h0 + nh) of
// one batch b0.
struct Piece {
  int b0, nb, h0, nh;
};

int make_pieces(int B, int H, int T, int want, int sms, Piece* pcs) {
  if (want <= 0) {
    // Automatic: pieces of at least ~3 waves of prefill CTAs (two 128-row
    // tiles each), 2 to 8 of them before the last one is cut down.  Each
    // piece costs its copies' and launch's overheads and a partial last
    // wave, so at 16K tokens and 32 heads 3-4 pieces beat 6-8 (measured
    // 2.98 against 3.05 ms per call).
    const long long ctas = (long long)B * H * ((T + 255) / 256);
    long long n = ctas / (3LL * (sms > 0 ? sms : 148));
    want = (int)(n < 2 ? 2 : (n > 8 ? 8 : n));
  }
  if (want > kMaxPieces - 16) want = kMaxPieces - 16;
  int n = 0;
  if (want <= B) {
    const int per = (B + want - 1) / want;
    for (int b = 0; b < B; b += per) pcs[n++] = {b, per < B - b ? per : B - b, 0, H};
  } else {
    int groups = (want + B - 1) / B;
    if (groups > H) groups = H;
    const int per = (H + groups - 1) / groups;
    for (int b = 0; b < B && n < kMaxPieces; ++b)
      for (int h = 0; h < H && n < kMaxPieces; h += per)
        pcs[n++] = {b, 1, h, per < H - h ? per : H - h};
  }
  if (n > 1) {
    // Only the last piece's kernel and copy-out run after the last copy in
    // (the link is the bottleneck), so the last piece is cut in halves,
    // quarters, ... down to one (b, h) slice: the tail is one slice's
    // kernel and copy-out.  A batch run is cut into batches first, a
    // single batch into heads.
    Piece last = pcs[--n];
    while (n < kMaxPieces - 1) {
      if (last.nb > 1) {
        const int take = last.nb / 2;
        pcs[n++] = {last.b0, take, 0, H};
        last.b0 += take;
        last.nb -= take;
      } else if (last.nh > 1) {
        const int take = last.nh / 2;
        pcs[n++] = {last.b0, 1, last.h0, take};
        last.h0 += take;
        last.nh -= take;
      } else {
        break;
      }
    }
    pcs[n++] = last;
  }
  return n;
}

}  // namespace
}  // namespace polar

using namespace polar;

extern "C" {

size_t polar_attn_fwd_host_workspace_bytes(int B, int H, int T, int d, int dtype) {
  if (B < 0 || H < 0 || T < 0 || (d != 64 && d != 128)) return 0;
  if (dtype != POLAR_F32 && dtype != POLAR_BF16) return 0;
  return regions(B, H, T, d, dtype).total;
}

int polar_attn_fwd_host(const void* q, const void* k, const void* v, const void* mem,
                        const float* w_count, void* out, float* n_eff, float* conf, int B,
                        int H, int T, int d, int dtype, const polar_consts_t* c,
                        int num_pieces, void* workspace, size_t workspace_bytes,
                        void* stream) {
  if (B < 0 || H < 0 || T < 0 || num_pieces < 0) return POLAR_ERR_INVALID;
  if (dtype != POLAR_F32 && dtype != POLAR_BF16) return POLAR_ERR_UNSUPPORTED;
  if (d != 64 && d != 128) return POLAR_ERR_UNSUPPORTED;
  const polar_consts_t cc = c ? *c : defaults();
  if (!consts_ok(cc)) return POLAR_ERR_INVALID;
  if ((long long)B * H * T == 0) return POLAR_OK;
  if (!q || !k || !v || !mem || !w_count || !out || !n_eff) return POLAR_ERR_INVALID;
  if ((long long)B * H > INT_MAX / 64 || T > (1 << 30)) return POLAR_ERR_UNSUPPORTED;
  const Regions r = regions(B, H, T, d, dtype);
  if (!workspace || workspace_bytes < r.total) return POLAR_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return POLAR_ERR_MISALIGNED;
  int sms = 0;
  int st = check_device(&sms);
  if (st != POLAR_OK) return st;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev >= kMaxDevices) return POLAR_ERR_DEVICE;

  std::lock_guard<std::mutex> lock(g_mutex);
  Pipeline& p = g_pipe[dev];
  cudaError_t e = pipeline_init(p);
  if (e != cudaSuccess) {
    set_last_error("polar_attn_fwd_host: stream or event creation failed");
    return POLAR_ERR_CUDA;
  }
  Piece pcs[kMaxPieces];
  const int n = make_pieces(B, H, T, num_pieces, sms, pcs);

  char* ws = static_cast<char*>(workspace);
  const size_t es = dtype == POLAR_BF16 ? 2 : 4;
  const size_t slice = (size_t)T * d * es;  // bytes of one (b, h) slice of q/k/v/mem/out
  const size_t rowb = (size_t)T * sizeof(float);
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const char* hq = static_cast<const char*>(q);
  const char* hk = static_cast<const char*>(k);
  const char* hv = static_cast<const char*>(v);
  const char* hm = static_cast<const char*>(mem);
  char* ho = static_cast<char*>(out);
  char* hn = reinterpret_cast<char*>(n_eff);
  char* hc = reinterpret_cast<char*>(conf);

  // The copy streams start after the caller's earlier work on `stream`.
  e = cudaEventRecord(p.start, cs);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(p.in, p.start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(p.out, p.start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(p.comp, p.start, 0);
  // w_count lands before piece 0, which every kernel launch waits for
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(ws + r.w, w_count, (size_t)H * d * sizeof(float),
                        cudaMemcpyHostToDevice, p.in);
  int result = POLAR_OK;
  for (int i = 0; i < n && e == cudaSuccess && result == POLAR_OK; ++i) {
    const size_t bh0 = (size_t)pcs[i].b0 * H + pcs[i].h0;
    const size_t nbh = (size_t)pcs[i].nb * pcs[i].nh;
    const size_t off = bh0 * slice, len = nbh * slice;
    const size_t roff = bh0 * rowb, rlen = nbh * rowb;
    // One copy-in stream: pieces land one after another at the full copy
    // rate (two streams sharing the link delayed every piece; measured).
    cudaStream_t in = p.in;
    e = cudaMemcpyAsync(ws + r.q + off, hq + off, len, cudaMemcpyHostToDevice, in);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(ws + r.k + off, hk + off, len, cudaMemcpyHostToDevice, in);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(ws + r.v + off, hv + off, len, cudaMemcpyHostToDevice, in);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(ws + r.mem + off, hm + off, len, cudaMemcpyHostToDevice, in);
    if (e == cudaSuccess) e = cudaEventRecord(p.landed[i], in);
    // Pieces compute alternately on `stream` and on the internal compute
    // stream, so a piece's kernel starts as soon as its inputs have landed
    // even while the previous piece's last CTAs still run.
    cudaStream_t ks = (i & 1) ? p.comp : cs;
    if (e == cudaSuccess) e = cudaStreamWaitEvent(ks, p.landed[i], 0);
    if (e != cudaSuccess) break;
    const float* w = reinterpret_cast<const float*>(ws + r.w) + (size_t)pcs[i].h0 * d;
    result = polar_attn_fwd(ws + r.q + off, ws + r.k + off, ws + r.v + off, ws + r.mem + off,
                            w, ws + r.out + off, reinterpret_cast<float*>(ws + r.n_eff + roff),
                            conf ? reinterpret_cast<float*>(ws + r.conf + roff) : nullptr,
                            pcs[i].nb, pcs[i].nh, T, d, dtype, &cc, ks);
    if (result != POLAR_OK) break;
    e = cudaEventRecord(p.computed[i], ks);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(p.out, p.computed[i], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(ho + off, ws + r.out + off, len, cudaMemcpyDeviceToHost, p.out);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(hn + roff, ws + r.n_eff + roff, rlen, cudaMemcpyDeviceToHost, p.out);
    if (e == cudaSuccess && conf)
      e = cudaMemcpyAsync(hc + roff, ws + r.conf + roff, rlen, cudaMemcpyDeviceToHost, p.out);
  }
  // Whatever was enqueued on the internal streams, the caller's stream ends
  // after it.
  cudaError_t e2 = cudaEventRecord(p.done, p.in);
  if (e2 == cudaSuccess) e2 = cudaStreamWaitEvent(p.out, p.done, 0);
  if (e2 == cudaSuccess) e2 = cudaEventRecord(p.done, p.comp);
  if (e2 == cudaSuccess) e2 = cudaStreamWaitEvent(p.out, p.done, 0);
  if (e2 == cudaSuccess) e2 = cudaEventRecord(p.done, p.out);
  if (e2 == cudaSuccess) e2 = cudaStreamWaitEvent(cs, p.done, 0);
  if (result != POLAR_OK) return result;
  if (e == cudaSuccess) e = e2;
  if (e != cudaSuccess) {
    set_last_error("polar_attn_fwd_host: a copy or stream-ordering call failed");
    return POLAR_ERR_CUDA;
  }
  return POLAR_OK;
}

}  // extern "C"
