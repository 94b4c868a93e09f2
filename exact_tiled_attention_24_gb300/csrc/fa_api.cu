// C ABI of the exact tiled attention library: argument checks, TMA
// descriptor construction and kernel dispatch. Declarations and the full
// contract are in include/fa.h.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>

#include "../../include/fa.h"
#include "fa_common.h"

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shared size/scale checks. Returns FA_OK or the status to report.
int check_sizes(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  const long long bh = static_cast<long long>(B) * H;
  // Grid sizes and row indices are 32-bit: BH * N rows must fit in int32.
  if (bh * N > INT_MAX) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

// Grouped-query heads: Hkv K/V heads, each shared by H / Hkv query heads.
int check_heads(int H, int Hkv) {
  if (Hkv < 1 || H % Hkv != 0) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

int check_scale(float scale) {
  if (!std::isfinite(scale) || scale <= 0.f) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

int map_cuda(cudaError_t e) { return e == cudaSuccess ? FA_OK : FA_ERR_CUDA; }

}  // namespace

extern "C" {

const char* fa_version(void) { return "0.1.0"; }

int fa_debug_checks(void) {
#ifdef FA_DEBUG
  return 1;
#else
  return 0;
#endif
}

const char* fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_MISALIGNED: return "FA_ERR_MISALIGNED";
    case FA_ERR_CUDA: return "FA_ERR_CUDA";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
    case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE";
    case FA_ERR_BAD_INDEX: return "FA_ERR_BAD_INDEX";
    case FA_ERR_BOUNDS: return "FA_ERR_BOUNDS";
    default: return "FA_ERR_UNKNOWN";
  }
}

int fa_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
               int Hkv, int N, int d, float scale, int causal, void* stream) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  int st = check_sizes(B, H, N, d);
  if (st != FA_OK) return st;
  if ((st = check_heads(H, Hkv)) != FA_OK) return st;
  if ((st = check_scale(scale)) != FA_OK) return st;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return FA_ERR_MISALIGNED;
  return map_cuda(fa::launch_fwd(q, k, v, o, lse, B * H, H / Hkv, N, d, scale, causal != 0,
                                 static_cast<cudaStream_t>(stream)));
}

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
           int d, float scale, int causal, void* stream) {
  return fa_fwd_gqa(q, k, v, o, lse, B, H, H, N, d, scale, causal, stream);
}

size_t fa_bwd_workspace_bytes(int B, int H, int N, int d) {
  if (check_sizes(B, H, N, d) != FA_OK) return 0;
  return static_cast<size_t>(B) * H * N * sizeof(float);
}

int fa_bwd_preprocess(const void* o, const void* dO, float* Dvec, int B, int H, int N, int d,
                      void* stream) {
  if (!o || !dO || !Dvec) return FA_ERR_INVALID_ARG;
  int st = check_sizes(B, H, N, d);
  if (st != FA_OK) return st;
  if (!aligned16(o) || !aligned16(dO) || !aligned16(Dvec)) return FA_ERR_MISALIGNED;
  return map_cuda(fa::launch_bwd_preprocess(static_cast<const __nv_bfloat16*>(o),
                                            static_cast<const __nv_bfloat16*>(dO), Dvec, B * H, N,
                                            d, static_cast<cudaStream_t>(stream)));
}

int fa_bwd_dkdv(const void* q, const void* k, const void* v, const void* dO, const float* lse,
                const float* Dvec, void* dk, void* dv, int B, int H, int Hkv, int N, int d,
                float scale, int causal, void* stream) {
  if (!q || !k || !v || !dO || !lse || !Dvec || !dk || !dv) return FA_ERR_INVALID_ARG;
  int st = check_sizes(B, H, N, d);
  if (st != FA_OK) return st;
  if ((st = check_heads(H, Hkv)) != FA_OK) return st;
  if ((st = check_scale(scale)) != FA_OK) return st;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dO) || !aligned16(lse) ||
      !aligned16(Dvec) || !aligned16(dk) || !aligned16(dv))
    return FA_ERR_MISALIGNED;
  return map_cuda(fa::launch_bwd_dkdv(q, k, v, dO, dk, dv, lse, Dvec, B * H, H / Hkv, N, d, scale,
                                      causal != 0, static_cast<cudaStream_t>(stream)));
}

int fa_bwd_dq(const void* q, const void* k, const void* v, const void* dO, const float* lse,
              const float* Dvec, void* dq, int B, int H, int Hkv, int N, int d, float scale,
              int causal, void* stream) {
  if (!q || !k || !v || !dO || !lse || !Dvec || !dq) return FA_ERR_INVALID_ARG;
  int st = check_sizes(B, H, N, d);
  if (st != FA_OK) return st;
  if ((st = check_heads(H, Hkv)) != FA_OK) return st;
  if ((st = check_scale(scale)) != FA_OK) return st;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dO) || !aligned16(lse) ||
      !aligned16(Dvec) || !aligned16(dq))
    return FA_ERR_MISALIGNED;
  return map_cuda(fa::launch_bwd_dq(q, k, v, dO, dq, lse, Dvec, B * H, H / Hkv, N, d, scale,
                                    causal != 0, static_cast<cudaStream_t>(stream)));
}

int fa_bwd_dq_d(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                float* Dvec, void* dq, int B, int H, int Hkv, int N, int d, float scale, int causal,
                void* stream) {
  if (!q || !k || !v || !o || !dO || !lse || !Dvec || !dq) return FA_ERR_INVALID_ARG;
  int st = check_sizes(B, H, N, d);
  if (st != FA_OK) return st;
  if ((st = check_heads(H, Hkv)) != FA_OK) return st;
  if ((st = check_scale(scale)) != FA_OK) return st;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dO) || !aligned16(lse) ||
      !aligned16(Dvec) || !aligned16(dq))
    return FA_ERR_MISALIGNED;
  return map_cuda(fa::launch_bwd_dq_d(q, k, v, o, dO, dq, lse, Dvec, B * H, H / Hkv, N, d, scale, causal != 0,
                                      static_cast<cudaStream_t>(stream)));
}

int fa_bwd_fuses_d(int B, int H, int Hkv, int N, int d) {
  if (check_sizes(B, H, N, d) != FA_OK || check_heads(H, Hkv) != FA_OK) return 0;
  return fa::bwd_fuse_d(B * H, H / Hkv, N) ? 1 : 0;
}

int fa_bwd_gqa(const void* q, const void* k, const void* v, const void* o, const void* dO,
               const float* lse, void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes,
               int B, int H, int Hkv, int N, int d, float scale, int causal, void* stream) {
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  int st = check_sizes(B, H, N, d);
  if (st != FA_OK) return st;
  if ((st = check_heads(H, Hkv)) != FA_OK) return st;
  if ((st = check_scale(scale)) != FA_OK) return st;
  if (!workspace || ws_bytes < fa_bwd_workspace_bytes(B, H, N, d)) return FA_ERR_WORKSPACE;
  // Every pointer is checked here, before the preprocess is launched, so
  // that an error leaves nothing queued (the stages repeat these checks).
  const void* ptrs[] = {q, k, v, o, dO, lse, dq, dk, dv, workspace};
  for (const void* p : ptrs)
    if (!aligned16(p)) return FA_ERR_MISALIGNED;
  float* Dvec = static_cast<float*>(workspace);
  if (fa::bwd_fuse_d(B * H, H / Hkv, N)) {  // D inside the dQ sweep, then dK/dV
    st = fa_bwd_dq_d(q, k, v, o, dO, lse, Dvec, dq, B, H, Hkv, N, d, scale, causal, stream);
    if (st != FA_OK) return st;
    return fa_bwd_dkdv(q, k, v, dO, lse, Dvec, dk, dv, B, H, Hkv, N, d, scale, causal, stream);
  }
  st = fa_bwd_preprocess(o, dO, Dvec, B, H, N, d, stream);
  if (st != FA_OK) return st;
  // The dQ sweep needs only D: it runs on the library's side stream, forked
  // from `stream` after the preprocess and joined back at the end, beside
  // the dK/dV sweep (the two grids then share one tail).
  cudaStream_t cs = static_cast<cudaStream_t>(stream), side = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  bool forked = fa::side_stream(&side) == cudaSuccess &&
                cudaEventCreateWithFlags(&fork, cudaEventDisableTiming) == cudaSuccess &&
                cudaEventCreateWithFlags(&join, cudaEventDisableTiming) == cudaSuccess &&
                cudaEventRecord(fork, cs) == cudaSuccess && cudaStreamWaitEvent(side, fork, 0) == cudaSuccess;
  if (!forked) {  // no side stream: the three stages in order on `stream`
    if (fork) cudaEventDestroy(fork);
    if (join) cudaEventDestroy(join);
    st = fa_bwd_dkdv(q, k, v, dO, lse, Dvec, dk, dv, B, H, Hkv, N, d, scale, causal, stream);
    if (st != FA_OK) return st;
    return fa_bwd_dq(q, k, v, dO, lse, Dvec, dq, B, H, Hkv, N, d, scale, causal, stream);
  }
  const int st_dkdv = fa_bwd_dkdv(q, k, v, dO, lse, Dvec, dk, dv, B, H, Hkv, N, d, scale, causal, stream);
  const int st_dq = fa_bwd_dq(q, k, v, dO, lse, Dvec, dq, B, H, Hkv, N, d, scale, causal, side);
  // Join even after a failed launch, so `stream` stays ordered after the side work.
  cudaError_t ej = cudaEventRecord(join, side);
  if (ej == cudaSuccess) ej = cudaStreamWaitEvent(cs, join, 0);
  cudaEventDestroy(fork);
  cudaEventDestroy(join);
  if (st_dkdv != FA_OK) return st_dkdv;
  if (st_dq != FA_OK) return st_dq;
  return map_cuda(ej);
}

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO,
           const float* lse, void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes,
           int B, int H, int N, int d, float scale, int causal, void* stream) {
  return fa_bwd_gqa(q, k, v, o, dO, lse, dq, dk, dv, workspace, ws_bytes, B, H, H, N, d, scale,
                    causal, stream);
}

static int softmax_rows(const float* x, float* y, long long rows, int n, bool online, void* stream) {
  if (!x || !y || rows < 1 || n < 1) return FA_ERR_INVALID_ARG;
  if (rows > INT_MAX) return FA_ERR_UNSUPPORTED;  // one CTA per row in a 1-D grid
  if (((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 3u) != 0)
    return FA_ERR_MISALIGNED;
  return map_cuda(fa::launch_softmax(x, y, rows, n, online, static_cast<cudaStream_t>(stream)));
}

int fa_softmax_safe(const float* x, float* y, long long rows, int n, void* stream) {
  return softmax_rows(x, y, rows, n, false, stream);
}

int fa_softmax_online(const float* x, float* y, long long rows, int n, void* stream) {
  return softmax_rows(x, y, rows, n, true, stream);
}

// ------------------------------------------------------------------ decode

size_t fa_decode_workspace_bytes(int B, int H, int d, int n_splits) {
  if (B < 1 || H < 1 || n_splits < 1 || (d != 64 && d != 128)) return 0;
  const size_t rows = static_cast<size_t>(n_splits) * B * H;
  const size_t o_bytes = (rows * d * sizeof(float) + 255) & ~static_cast<size_t>(255);
  return o_bytes + rows * sizeof(float);
}

int fa_decode_paged(const void* q, const void* k_cache, const void* v_cache, const int* block_table,
                    const int* seq_lens, void* o, float* lse, void* workspace, size_t ws_bytes, int B,
                    int H, int Hkv, int d, int num_blocks, int block_size, int max_blocks_per_seq,
                    float scale, int n_splits, void* stream) {
  if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !o || !lse) return FA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || num_blocks < 1 || block_size < 1 || max_blocks_per_seq < 1 || n_splits < 1)
    return FA_ERR_INVALID_ARG;
  int st = check_heads(H, Hkv);
  if (st != FA_OK) return st;
  if ((st = check_scale(scale)) != FA_OK) return st;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (B > 65535 || static_cast<long long>(Hkv) * ((H / Hkv + 15) / 16) > 65535 || n_splits > 4096)
    return FA_ERR_UNSUPPORTED;
  const long long ctx = static_cast<long long>(max_blocks_per_seq) * block_size;
  // The cache's token rows (num_blocks * Hkv * block_size) are indexed in
  // 32 bits on the device: fewer than 2^32 - 1 (512 GB of cache at d = 64).
  if (ctx > INT_MAX / 2 || static_cast<long long>(num_blocks) * Hkv * block_size >= 0xffffffffll)
    return FA_ERR_UNSUPPORTED;
  if (!workspace || ws_bytes < fa_decode_workspace_bytes(B, H, d, n_splits)) return FA_ERR_WORKSPACE;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o) ||
      !aligned16(workspace) || (reinterpret_cast<uintptr_t>(lse) & 3u) ||
      (reinterpret_cast<uintptr_t>(block_table) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
    return FA_ERR_MISALIGNED;
  const size_t rows = static_cast<size_t>(n_splits) * B * H;
  float* o_part = static_cast<float*>(workspace);
  float* lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                             ((rows * d * sizeof(float) + 255) & ~static_cast<size_t>(255)));
  return map_cuda(fa::launch_decode_paged(q, k_cache, v_cache, block_table, seq_lens, o, lse, o_part,
                                          lse_part, B, H, Hkv, d, num_blocks, block_size,
                                          max_blocks_per_seq, scale, n_splits,
                                          static_cast<cudaStream_t>(stream)));
}

int fa_attn_merge(const float* o_parts, const float* lse_parts, int n_parts, void* o, float* lse,
                  long long rows, int d, void* stream) {
  if (!o_parts || !lse_parts || !o || !lse || n_parts < 1 || rows < 1) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if ((rows + 7) / 8 > INT_MAX) return FA_ERR_UNSUPPORTED;
  if (!aligned16(o_parts) || !aligned16(o) || (reinterpret_cast<uintptr_t>(lse_parts) & 3u) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u))
    return FA_ERR_MISALIGNED;
  return map_cuda(fa::launch_attn_merge(o_parts, lse_parts, n_parts, o, lse, rows, d,
                                        static_cast<cudaStream_t>(stream)));
}

int fa_selftest_wait_limit(void* stream) {
  return map_cuda(fa::launch_wait_limit_selftest(static_cast<cudaStream_t>(stream)));
}

int fa_last_device_error(void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t ef = 0, eb = 0, ed = 0, et = 0, es = 0;
  if (fa::read_and_clear_fwd_error(&ef, s) != cudaSuccess) return FA_ERR_CUDA;
  if (fa::read_and_clear_bwd_error(&eb, s) != cudaSuccess) return FA_ERR_CUDA;
  if (fa::read_and_clear_decode_error(&ed, s) != cudaSuccess) return FA_ERR_CUDA;
  if (fa::read_and_clear_selftest_error(&et, s) != cudaSuccess) return FA_ERR_CUDA;
  if (fa::read_and_clear_softmax_error(&es, s) != cudaSuccess) return FA_ERR_CUDA;
  if (ef == 1 || eb == 1 || ed == 1 || et == 1) return FA_ERR_TIMEOUT;
  if (ef == 3 || eb == 3 || ed == 3 || es == 3) return FA_ERR_BOUNDS;
  if (ed == 2) return FA_ERR_BAD_INDEX;
  if (ef || eb || ed || et || es) return FA_ERR_TIMEOUT;
  return FA_OK;
}

}  // extern "C"
