// Attention steps whose inputs and outputs live in host memory.
//
// The (batch, K/V head) pairs are independent problems, so the step is cut
// into slices of consecutive pairs and run as a three-stage pipeline:
//   copy-in stream   q, k, v (and dO) of slice c, host -> device
//   caller's stream  forward (and backward) kernels of slice c
//   copy-out stream  o, lse (and dq, dk, dv) of slice c, device -> host
// Events order each slice's stages; slice c's kernels run while slice c+1
// is copied in and slice c-1 is copied out. In the [B][H][N][d] layout a
// run of consecutive (b, h) pairs is one contiguous range of every tensor,
// so each tensor of a slice moves in one copy. The kernels are the device
// entry points' own, launched on the slice's sub-range; results do not
// depend on the slicing.
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <vector>

#include "../../include/fa.h"
#include "fa_common.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxChunks = 64;
constexpr int kDefaultChunks = 8;

// The library's own streams for one host thread on one device, created on
// first use and kept for the thread's lifetime (non-blocking: they never
// wait on the legacy default stream): copy-in, copy-out, and a side stream
// for the dQ sweep, which runs beside the dK/dV sweep.
struct CopyStreams {
  cudaStream_t in = nullptr;
  cudaStream_t out = nullptr;
  cudaStream_t side = nullptr;
};

cudaError_t make_stream(cudaStream_t* s) {
  if (*s != nullptr) return cudaSuccess;
  cudaError_t e = cudaStreamCreateWithFlags(s, cudaStreamNonBlocking);
  if (e != cudaSuccess) *s = nullptr;
  return e;
}

cudaError_t copy_streams(CopyStreams** out) {
  thread_local CopyStreams per_device[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  CopyStreams& cs = per_device[dev];
  if ((e = make_stream(&cs.in)) != cudaSuccess) return e;
  if ((e = make_stream(&cs.out)) != cudaSuccess) return e;
  if ((e = make_stream(&cs.side)) != cudaSuccess) return e;
  *out = &cs;
  return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Events of one call, released when the call returns (CUDA defers the
// release until the recorded work has completed).
struct Events {
  std::vector<cudaEvent_t> ev;
  ~Events() {
    for (cudaEvent_t e : ev) cudaEventDestroy(e);
  }
  cudaError_t make(cudaEvent_t* out) {
    cudaError_t e = cudaEventCreateWithFlags(out, cudaEventDisableTiming);
    if (e == cudaSuccess) ev.push_back(*out);
    return e;
  }
};

#define FA_TRY(expr)                         \
  do {                                       \
    cudaError_t e_ = (expr);                 \
    if (e_ != cudaSuccess) return e_;        \
  } while (0)

// Byte offset of row block [u0, u1) of a tensor with `per_unit` bytes per
// (batch, K/V head) pair.
struct Slice {
  size_t off, bytes;
};
Slice slice(long long u0, long long u1, size_t per_unit) {
  return {static_cast<size_t>(u0) * per_unit, static_cast<size_t>(u1 - u0) * per_unit};
}

const char* cptr(const void* p, size_t off) { return static_cast<const char*>(p) + off; }
char* mptr(void* p, size_t off) { return static_cast<char*>(p) + off; }

cudaError_t copy_in(void* dst, const void* src, Slice s, cudaStream_t st) {
  return cudaMemcpyAsync(mptr(dst, s.off), cptr(src, s.off), s.bytes, cudaMemcpyHostToDevice, st);
}
cudaError_t copy_out(void* dst, const void* src, Slice s, cudaStream_t st) {
  return cudaMemcpyAsync(mptr(dst, s.off), cptr(src, s.off), s.bytes, cudaMemcpyDeviceToHost, st);
}

// The pipeline; argument checks are done by the callers.
cudaError_t run_pipeline(const fa_tensors& h, const fa_tensors& dv, float* Dvec, bool with_bwd, int B,
                         int H, int Hkv, int N, int d, float scale, bool causal, int n_chunks,
                         cudaStream_t stream) {
  CopyStreams* cs = nullptr;
  FA_TRY(copy_streams(&cs));
  const int G = H / Hkv;
  const long long units = static_cast<long long>(B) * Hkv;  // (batch, K/V head) pairs
  const int C = static_cast<int>(n_chunks < units ? n_chunks : units);
  const size_t row_b = static_cast<size_t>(N) * d * 2;  // one head of a bf16 tensor
  const size_t q_unit = row_b * G, kv_unit = row_b;     // bytes per pair
  // lse, D per pair. A slice of them may start only 4-byte aligned (N and G
  // odd): every kernel reads and writes them one float at a time.
  const size_t r_unit = static_cast<size_t>(N) * G * 4;
  auto bounds = [&](int c, long long* u0, long long* u1) {
    *u0 = units * c / C;
    *u1 = units * (c + 1) / C;
  };

  Events evs;
  cudaEvent_t start, done;
  std::vector<cudaEvent_t> in_ready(C), fwd_done(C), pre_done(C), bwd_done(C), dq_done(C);
  FA_TRY(evs.make(&start));
  FA_TRY(evs.make(&done));
  for (int c = 0; c < C; ++c) {
    FA_TRY(evs.make(&in_ready[c]));
    FA_TRY(evs.make(&fwd_done[c]));
    if (with_bwd) {
      FA_TRY(evs.make(&pre_done[c]));
      FA_TRY(evs.make(&bwd_done[c]));
      FA_TRY(evs.make(&dq_done[c]));
    }
  }
  // Both copy streams start after the work already queued on `stream`.
  FA_TRY(cudaEventRecord(start, stream));
  FA_TRY(cudaStreamWaitEvent(cs->in, start, 0));
  FA_TRY(cudaStreamWaitEvent(cs->out, start, 0));

  cudaError_t err = cudaSuccess;
  // Stage 1: every slice's inputs, back to back.
  for (int c = 0; c < C && err == cudaSuccess; ++c) {
    long long u0, u1;
    bounds(c, &u0, &u1);
    const Slice sq = slice(u0, u1, q_unit), skv = slice(u0, u1, kv_unit);
    if ((err = copy_in(const_cast<void*>(dv.q), h.q, sq, cs->in)) != cudaSuccess) break;
    if ((err = copy_in(const_cast<void*>(dv.k), h.k, skv, cs->in)) != cudaSuccess) break;
    if ((err = copy_in(const_cast<void*>(dv.v), h.v, skv, cs->in)) != cudaSuccess) break;
    if (with_bwd && (err = copy_in(const_cast<void*>(dv.dO), h.dO, sq, cs->in)) != cudaSuccess) break;
    err = cudaEventRecord(in_ready[c], cs->in);
  }
  // Stage 2: the kernels of each slice, on the caller's stream.
  for (int c = 0; c < C && err == cudaSuccess; ++c) {
    long long u0, u1;
    bounds(c, &u0, &u1);
    const int bh = static_cast<int>((u1 - u0) * G);  // query heads in the slice
    const size_t oq = slice(u0, u1, q_unit).off, okv = slice(u0, u1, kv_unit).off;
    const size_t orow = slice(u0, u1, r_unit).off;
    float* lse = reinterpret_cast<float*>(mptr(dv.lse, orow));
    if ((err = cudaStreamWaitEvent(stream, in_ready[c], 0)) != cudaSuccess) break;
    err = fa::launch_fwd(cptr(dv.q, oq), cptr(dv.k, okv), cptr(dv.v, okv), mptr(dv.o, oq), lse, bh, G, N, d,
                         scale, causal, stream);
    if (err != cudaSuccess) break;
    if ((err = cudaEventRecord(fwd_done[c], stream)) != cudaSuccess) break;
    if (!with_bwd) continue;
    float* D = reinterpret_cast<float*>(mptr(Dvec, orow));
    err = fa::launch_bwd_preprocess(reinterpret_cast<const __nv_bfloat16*>(cptr(dv.o, oq)),
                                    reinterpret_cast<const __nv_bfloat16*>(cptr(dv.dO, oq)), D, bh, N, d,
                                    stream);
    if (err != cudaSuccess) break;
    // The dQ sweep needs only D: it runs on the side stream beside the
    // dK/dV sweep (and the next slice's kernels).
    if ((err = cudaEventRecord(pre_done[c], stream)) != cudaSuccess) break;
    if ((err = cudaStreamWaitEvent(cs->side, pre_done[c], 0)) != cudaSuccess) break;
    err = fa::launch_bwd_dkdv(cptr(dv.q, oq), cptr(dv.k, okv), cptr(dv.v, okv), cptr(dv.dO, oq),
                              mptr(dv.dk, okv), mptr(dv.dv, okv), lse, D, bh, G, N, d, scale, causal, stream);
    if (err != cudaSuccess) break;
    if ((err = cudaEventRecord(bwd_done[c], stream)) != cudaSuccess) break;
    err = fa::launch_bwd_dq(cptr(dv.q, oq), cptr(dv.k, okv), cptr(dv.v, okv), cptr(dv.dO, oq),
                            mptr(dv.dq, oq), lse, D, bh, G, N, d, scale, causal, cs->side);
    if (err != cudaSuccess) break;
    err = cudaEventRecord(dq_done[c], cs->side);
  }
  // Stage 3: every slice's outputs, each as soon as its kernels are done.
  for (int c = 0; c < C && err == cudaSuccess; ++c) {
    long long u0, u1;
    bounds(c, &u0, &u1);
    const Slice sq = slice(u0, u1, q_unit), skv = slice(u0, u1, kv_unit), sr = slice(u0, u1, r_unit);
    if ((err = cudaStreamWaitEvent(cs->out, fwd_done[c], 0)) != cudaSuccess) break;
    if ((err = copy_out(h.o, dv.o, sq, cs->out)) != cudaSuccess) break;
    if ((err = copy_out(h.lse, dv.lse, sr, cs->out)) != cudaSuccess) break;
    if (!with_bwd) continue;
    if ((err = cudaStreamWaitEvent(cs->out, bwd_done[c], 0)) != cudaSuccess) break;
    if ((err = copy_out(h.dk, dv.dk, skv, cs->out)) != cudaSuccess) break;
    if ((err = copy_out(h.dv, dv.dv, skv, cs->out)) != cudaSuccess) break;
    if ((err = cudaStreamWaitEvent(cs->out, dq_done[c], 0)) != cudaSuccess) break;
    err = copy_out(h.dq, dv.dq, sq, cs->out);
  }
  // Join: `stream` passes this point only after the copy streams and the
  // side stream have drained what this call queued on them, also after a
  // failure half-way.
  cudaError_t e1 = cudaEventRecord(done, cs->in);
  if (e1 == cudaSuccess) e1 = cudaStreamWaitEvent(stream, done, 0);
  cudaError_t e2 = cudaSuccess;
  for (cudaStream_t side : {cs->out, cs->side}) {
    cudaEvent_t ev;
    cudaError_t e = evs.make(&ev);
    if (e == cudaSuccess) e = cudaEventRecord(ev, side);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, ev, 0);
    if (e2 == cudaSuccess) e2 = e;
  }
  if (err != cudaSuccess) return err;
  return e1 != cudaSuccess ? e1 : e2;
}

// Row softmax of x [rows][n] fp32 from host memory, pipelined like the
// attention calls: slices of consecutive rows (each one contiguous range)
// are copied in, normalised and copied out on the three streams.
cudaError_t run_softmax_pipeline(const float* xh, float* yh, float* xd, float* yd, long long rows, int n,
                                 bool online, int n_chunks, cudaStream_t stream) {
  CopyStreams* cs = nullptr;
  FA_TRY(copy_streams(&cs));
  const int C = static_cast<int>(n_chunks < rows ? n_chunks : rows);
  const size_t row_bytes = static_cast<size_t>(n) * sizeof(float);
  Events evs;
  cudaEvent_t start, done;
  std::vector<cudaEvent_t> in_ready(C), out_ready(C);
  FA_TRY(evs.make(&start));
  FA_TRY(evs.make(&done));
  for (int c = 0; c < C; ++c) {
    FA_TRY(evs.make(&in_ready[c]));
    FA_TRY(evs.make(&out_ready[c]));
  }
  FA_TRY(cudaEventRecord(start, stream));
  FA_TRY(cudaStreamWaitEvent(cs->in, start, 0));
  FA_TRY(cudaStreamWaitEvent(cs->out, start, 0));
  auto bounds = [&](int c, long long* r0, long long* r1) {
    *r0 = rows * c / C;
    *r1 = rows * (c + 1) / C;
  };
  cudaError_t err = cudaSuccess;
  for (int c = 0; c < C && err == cudaSuccess; ++c) {
    long long r0, r1;
    bounds(c, &r0, &r1);
    const Slice sl = slice(r0, r1, row_bytes);
    if ((err = copy_in(xd, xh, sl, cs->in)) != cudaSuccess) break;
    err = cudaEventRecord(in_ready[c], cs->in);
  }
  for (int c = 0; c < C && err == cudaSuccess; ++c) {
    long long r0, r1;
    bounds(c, &r0, &r1);
    if ((err = cudaStreamWaitEvent(stream, in_ready[c], 0)) != cudaSuccess) break;
    err = fa::launch_softmax(xd + r0 * n, yd + r0 * n, r1 - r0, n, online, stream);
    if (err != cudaSuccess) break;
    err = cudaEventRecord(out_ready[c], stream);
  }
  for (int c = 0; c < C && err == cudaSuccess; ++c) {
    long long r0, r1;
    bounds(c, &r0, &r1);
    if ((err = cudaStreamWaitEvent(cs->out, out_ready[c], 0)) != cudaSuccess) break;
    err = copy_out(yh, yd, slice(r0, r1, row_bytes), cs->out);
  }
  cudaError_t e1 = cudaEventRecord(done, cs->in);
  if (e1 == cudaSuccess) e1 = cudaStreamWaitEvent(stream, done, 0);
  cudaEvent_t done_out;
  cudaError_t e2 = evs.make(&done_out);
  if (e2 == cudaSuccess) e2 = cudaEventRecord(done_out, cs->out);
  if (e2 == cudaSuccess) e2 = cudaStreamWaitEvent(stream, done_out, 0);
  if (err != cudaSuccess) return err;
  return e1 != cudaSuccess ? e1 : e2;
}

}  // namespace

namespace fa {

// The calling thread's side stream on the current device (see CopyStreams).
cudaError_t side_stream(cudaStream_t* out) {
  CopyStreams* cs = nullptr;
  cudaError_t e = copy_streams(&cs);
  if (e == cudaSuccess) *out = cs->side;
  return e;
}

}  // namespace fa

namespace {

int check_common(const fa_tensors* host, const fa_tensors* dev, bool with_bwd, int B, int H, int Hkv,
                 int N, int d, float scale, int n_chunks) {
  if (!host || !dev) return FA_ERR_INVALID_ARG;
  const void* hp[] = {host->q, host->k, host->v, host->o, host->lse};
  const void* dp[] = {dev->q, dev->k, dev->v, dev->o, dev->lse};
  for (const void* p : hp)
    if (!p) return FA_ERR_INVALID_ARG;
  for (const void* p : dp) {
    if (!p) return FA_ERR_INVALID_ARG;
    if (!aligned16(p)) return FA_ERR_MISALIGNED;
  }
  if (with_bwd) {
    const void* hb[] = {host->dO, host->dq, host->dk, host->dv};
    const void* db[] = {dev->dO, dev->dq, dev->dk, dev->dv};
    for (const void* p : hb)
      if (!p) return FA_ERR_INVALID_ARG;
    for (const void* p : db) {
      if (!p) return FA_ERR_INVALID_ARG;
      if (!aligned16(p)) return FA_ERR_MISALIGNED;
    }
  }
  if (B < 1 || H < 1 || N < 1 || Hkv < 1 || H % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || scale <= 0.f) return FA_ERR_INVALID_ARG;
  if (n_chunks < 0) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * H * N > INT_MAX) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

// Slices when the caller leaves the choice (n_chunks = 0): up to 8, but no
// more than keep every slice's dK/dV sweep (one CTA per K/V head and
// 128-key tile) at 1.5 or more CTAs per SM. Smaller slices leave SMs idle;
// their kernels lose more than the finer pipeline gains (measured: 32
// query over 8 K/V heads, N = 8192, runs best at 4 slices, 1.7 CTAs/SM).
int chunks_or_default(int n_chunks, int B, int Hkv, int N) {
  if (n_chunks > 0) return n_chunks > kMaxChunks ? kMaxChunks : n_chunks;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
    return kDefaultChunks;
  const long long ctas = static_cast<long long>(B) * Hkv * ((N + 127) / 128);
  const long long c = 2 * ctas / (3LL * sms);
  return static_cast<int>(c < 1 ? 1 : (c > kDefaultChunks ? kDefaultChunks : c));
}

}  // namespace

extern "C" {

int fa_fwd_host(const fa_tensors* host, const fa_tensors* dev, int B, int H, int Hkv, int N, int d,
                float scale, int causal, int n_chunks, void* stream) {
  const int st = check_common(host, dev, false, B, H, Hkv, N, d, scale, n_chunks);
  if (st != FA_OK) return st;
  const cudaError_t e = run_pipeline(*host, *dev, nullptr, false, B, H, Hkv, N, d, scale, causal != 0,
                                     chunks_or_default(n_chunks, B, Hkv, N), static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_fwd_bwd_host(const fa_tensors* host, const fa_tensors* dev, void* workspace, size_t ws_bytes, int B,
                    int H, int Hkv, int N, int d, float scale, int causal, int n_chunks, void* stream) {
  const int st = check_common(host, dev, true, B, H, Hkv, N, d, scale, n_chunks);
  if (st != FA_OK) return st;
  if (!workspace || ws_bytes < static_cast<size_t>(B) * H * N * sizeof(float)) return FA_ERR_WORKSPACE;
  if (!aligned16(workspace)) return FA_ERR_MISALIGNED;
  const cudaError_t e = run_pipeline(*host, *dev, static_cast<float*>(workspace), true, B, H, Hkv, N, d,
                                     scale, causal != 0, chunks_or_default(n_chunks, B, Hkv, N),
                                     static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_softmax_host(const float* x_host, float* y_host, float* x_dev, float* y_dev, long long rows, int n,
                    int online, int n_chunks, void* stream) {
  if (!x_host || !y_host || !x_dev || !y_dev || rows < 1 || n < 1 || n_chunks < 0) return FA_ERR_INVALID_ARG;
  if (rows > INT_MAX) return FA_ERR_UNSUPPORTED;
  if (((reinterpret_cast<uintptr_t>(x_dev) | reinterpret_cast<uintptr_t>(y_dev)) & 3u) != 0)
    return FA_ERR_MISALIGNED;
  const int C = n_chunks == 0 ? kDefaultChunks : (n_chunks > kMaxChunks ? kMaxChunks : n_chunks);
  const cudaError_t e = run_softmax_pipeline(x_host, y_host, x_dev, y_dev, rows, n, online != 0, C,
                                             static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // extern "C"
