// Allocation-free variant of the backward pass.
//
// fa_bwd needs device scratch (the fp32 row vector D = rowsum(dO ∘ O)) and
// expects the caller to provide it. Some callers cannot make
// that allocation: a host application that owns all device memory through
// its own fixed pool and gives plug-ins no allocator, a runtime that forbids
// device allocation after start-up (fixed memory budget, real-time loop), or
// code that must not take cudaMalloc's implicit device-wide synchronisation.
// fa_bwd_noalloc serves them: its scratch is a file-scope __device__ array
// of fixed size that lives in the library image, so the call itself
// allocates nothing.
//
// Properties of that array (also stated in include/fa.h):
//   * FA_BWD_NOALLOC_SCRATCH_BYTES bytes, held on every GPU that loads this
//     library until the process exits;
//   * shared by every call on a device: calls whose kernels overlap on the
//     GPU (other streams, other host threads) race on it;
//   * it keeps the last call's contents; the preprocess kernel rewrites D on
//     every call before anything reads it, so nothing stale is read.
// The array's device address is looked up once per device (with that device
// current) on the first call there.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "../../include/fa.h"
#include "fa_common.h"

namespace {

static __device__ __align__(256) unsigned char g_bwd_noalloc_scratch[FA_BWD_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch array on the current device (host code
// cannot use the array's name as an address), looked up on every call: a
// device reset reloads the module, and the array may then sit elsewhere.
// Returns nullptr on failure.
void* scratch_on_current_device() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_bwd_noalloc_scratch) != cudaSuccess) return nullptr;
  return p;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                              const void* dO, const float* lse, void* dq, void* dk, void* dv,
                              int B, int H, int N, int d, float scale, int causal, void* stream) {
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  // Same size and scale rules as fa_bwd; the workspace query returns 0 for
  // invalid sizes.
  const size_t need = fa_bwd_workspace_bytes(B, H, N, d);
  if (need == 0) return (B < 1 || H < 1 || N < 1) ? FA_ERR_INVALID_ARG : FA_ERR_UNSUPPORTED;
  if (!std::isfinite(scale) || scale <= 0.f) return FA_ERR_INVALID_ARG;
  if (need > FA_BWD_NOALLOC_SCRATCH_BYTES) return FA_ERR_WORKSPACE;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dO) ||
      !aligned16(lse) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return FA_ERR_MISALIGNED;
  void* scratch = scratch_on_current_device();
  if (!scratch) return FA_ERR_CUDA;
  float* Dvec = static_cast<float*>(scratch);
  const int BH = B * H;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (fa::bwd_fuse_d(BH, 1, N)) {  // the order fa_bwd takes for this shape, so the results match it
    if (fa::launch_bwd_dq_d(q, k, v, o, dO, dq, lse, Dvec, BH, 1, N, d, scale, causal != 0, s) != cudaSuccess)
      return FA_ERR_CUDA;
    if (fa::launch_bwd_dkdv(q, k, v, dO, dk, dv, lse, Dvec, BH, 1, N, d, scale, causal != 0, s) != cudaSuccess)
      return FA_ERR_CUDA;
    return FA_OK;
  }
  if (fa::launch_bwd_preprocess(static_cast<const __nv_bfloat16*>(o),
                                static_cast<const __nv_bfloat16*>(dO), Dvec, BH, N, d,
                                s) != cudaSuccess)
    return FA_ERR_CUDA;
  if (fa::launch_bwd_dkdv(q, k, v, dO, dk, dv, lse, Dvec, BH, 1, N, d, scale, causal != 0, s) !=
      cudaSuccess)
    return FA_ERR_CUDA;
  if (fa::launch_bwd_dq(q, k, v, dO, dq, lse, Dvec, BH, 1, N, d, scale, causal != 0, s) !=
      cudaSuccess)
    return FA_ERR_CUDA;
  return FA_OK;
}
