// Row softmax in fp32, two ways, as standalone bandwidth-bound kernels.
//
// Safe softmax (dcwnkz.com GPU-tricks article, appendix on softmax; CMU
// 10-423 L17–L18 notes, section 前置二：online softmax) subtracts the row
// maximum before exponentiating and so reads the row three times: once for
// the maximum, once for the sum of e^(x − m), once to write e^(x − m) / l.
// Online softmax (same CMU section) keeps the running maximum and the
// running denominator together in a single read, rescaling the denominator
// by e^(m_old − m_new) whenever the maximum grows, and needs two reads in all.
// Per element that is 3 loads + 1 store against 2 loads + 1 store, the
// 4:3 memory-traffic ratio the notes quote for this change.
//
// Each CTA owns one row and streams it from global memory in every pass
// (16-byte loads when the row is 16-byte aligned, else 4-byte ones). y may
// alias x: every element is read for the last time, by the thread that
// writes it, just before the write. Whether
// a re-read is served by DRAM or by L2 depends on how many bytes of rows are
// in flight: with 1 MB rows the re-reads miss the 126 MB L2, with short rows
// they hit it.
#include <cuda_runtime.h>

#include <cstdint>

#include "fa_common.h"
#include "fa_ptx.cuh"

namespace fa {

static __device__ uint32_t g_smx_err;

namespace sm {

constexpr int THREADS = 512;
constexpr int WARPS = THREADS / 32;
constexpr float LOG2E = 1.4426950408889634f;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Merge two (max, denominator) states: l is relative to m.
__device__ __forceinline__ void merge_ml(float& m, float& l, float m2, float l2) {
  const float mn = fmaxf(m, m2);
  if (mn == -INFINITY) return;  // both empty
  l = l * ex2((m - mn) * LOG2E) + l2 * ex2((m2 - mn) * LOG2E);
  m = mn;
}

__device__ __forceinline__ void warp_merge_ml(float& m, float& l) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float l2 = __shfl_xor_sync(0xffffffffu, l, o);
    merge_ml(m, l, m2, l2);
  }
}

// Block-wide reductions over THREADS threads through shared memory; every
// thread gets the result.
__device__ __forceinline__ float block_max(float v, float* red) {
  v = warp_max(v);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = (threadIdx.x & 31) < WARPS ? red[threadIdx.x & 31] : -INFINITY;
  r = warp_max(r);
  __syncthreads();
  return r;
}

__device__ __forceinline__ float block_sum(float v, float* red) {
  v = warp_sum(v);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = (threadIdx.x & 31) < WARPS ? red[threadIdx.x & 31] : 0.f;
  r = warp_sum(r);
  __syncthreads();
  return r;
}

__device__ __forceinline__ void block_merge_ml(float& m, float& l, float* red) {
  warp_merge_ml(m, l);
  if ((threadIdx.x & 31) == 0) {
    red[threadIdx.x >> 5] = m;
    red[WARPS + (threadIdx.x >> 5)] = l;
  }
  __syncthreads();
  const int w = threadIdx.x & 31;
  m = w < WARPS ? red[w] : -INFINITY;
  l = w < WARPS ? red[WARPS + w] : 0.f;
  warp_merge_ml(m, l);
  __syncthreads();
}

__device__ __forceinline__ float max4(float4 v) { return fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)); }

// Row access in units of U floats (U = 4: float4, U = 1: float).
template <int U>
struct Row;

template <>
struct Row<4> {
  using T = float4;
  static __device__ __forceinline__ float4 load(const float* p, long long i) {
    return reinterpret_cast<const float4*>(p)[i];
  }
  static __device__ __forceinline__ void store(float* p, long long i, float4 v) {
    __stcs(reinterpret_cast<float4*>(p) + i, v);
  }
  static __device__ __forceinline__ float vmax(float4 v) { return max4(v); }
  // Σ e^(v − m), as 2^((v − m)·log2 e): the difference first, so that v = m
  // gives exactly 1 whatever the magnitude of m.
  static __device__ __forceinline__ float vexpsum(float4 v, float m) {
    return ex2((v.x - m) * LOG2E) + ex2((v.y - m) * LOG2E) + ex2((v.z - m) * LOG2E) +
           ex2((v.w - m) * LOG2E);
  }
  static __device__ __forceinline__ float4 vnorm(float4 v, float m, float inv) {
    return make_float4(ex2((v.x - m) * LOG2E) * inv, ex2((v.y - m) * LOG2E) * inv,
                       ex2((v.z - m) * LOG2E) * inv, ex2((v.w - m) * LOG2E) * inv);
  }
};

template <>
struct Row<1> {
  using T = float;
  static __device__ __forceinline__ float load(const float* p, long long i) { return p[i]; }
  static __device__ __forceinline__ void store(float* p, long long i, float v) { __stcs(p + i, v); }
  static __device__ __forceinline__ float vmax(float v) { return v; }
  static __device__ __forceinline__ float vexpsum(float v, float m) { return ex2((v - m) * LOG2E); }
  static __device__ __forceinline__ float vnorm(float v, float m, float inv) {
    return ex2((v - m) * LOG2E) * inv;
  }
};

// Element i (in units of U floats) of row `row` lies inside the [rows][n]
// array (rows = the grid). Constant true outside the FA_DEBUG build.
template <int U>
__device__ __forceinline__ bool in_rows(long long row, int n, long long i) {
  return in_range(row * n + i * U, U, static_cast<long long>(gridDim.x) * n, &g_smx_err);
}

// Final pass, shared by both forms: y = e^(x − m) / l.
template <int U>
__device__ __forceinline__ void write_pass(const float* xr, float* yr, long long row, int n, long long nv,
                                           float m, float l) {
  using R = Row<U>;
  const float inv = 1.f / l;
#pragma unroll 4
  for (long long i = threadIdx.x; i < nv; i += THREADS)
    if (in_rows<U>(row, n, i)) R::store(yr, i, R::vnorm(R::load(xr, i), m, inv));
}

// Three passes: maximum, denominator, output.
template <int U>
__global__ void __launch_bounds__(THREADS) softmax_safe_kernel(const float* x, float* y, int n) {
  using R = Row<U>;
  __shared__ float red[2 * WARPS];
  const long long row = blockIdx.x;
  const float* xr = x + row * n;
  float* yr = y + row * n;
  const long long nv = n / U;
  float m = -INFINITY;
#pragma unroll 4
  for (long long i = threadIdx.x; i < nv; i += THREADS)
    if (in_rows<U>(row, n, i)) m = fmaxf(m, R::vmax(R::load(xr, i)));
  m = block_max(m, red);
  float l = 0.f;
#pragma unroll 4
  for (long long i = threadIdx.x; i < nv; i += THREADS)
    if (in_rows<U>(row, n, i)) l += R::vexpsum(R::load(xr, i), m);
  l = block_sum(l, red);
  write_pass<U>(xr, yr, row, n, nv, m, l);
}

// Two passes: maximum and denominator together (rescaling l when the
// maximum grows), then output.
template <int U>
__global__ void __launch_bounds__(THREADS) softmax_online_kernel(const float* x, float* y, int n) {
  using R = Row<U>;
  __shared__ float red[2 * WARPS];
  const long long row = blockIdx.x;
  const float* xr = x + row * n;
  float* yr = y + row * n;
  const long long nv = n / U;
  float m = -INFINITY, l = 0.f;
#pragma unroll 4
  for (long long i = threadIdx.x; i < nv; i += THREADS) {
    if (!in_rows<U>(row, n, i)) continue;
    const typename R::T v = R::load(xr, i);
    const float mn = fmaxf(m, R::vmax(v));
    if (mn == -INFINITY) continue;  // nothing but -inf so far
    l = l * ex2((m - mn) * LOG2E) + R::vexpsum(v, mn);
    m = mn;
  }
  block_merge_ml(m, l, red);
  write_pass<U>(xr, yr, row, n, nv, m, l);
}

}  // namespace sm

cudaError_t read_and_clear_softmax_error(uint32_t* out, cudaStream_t stream) {
  cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_smx_err, sizeof(uint32_t), 0, cudaMemcpyDeviceToHost,
                                            stream);
  if (e != cudaSuccess) return e;
  e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return e;
  const uint32_t zero = 0;
  e = cudaMemcpyToSymbolAsync(g_smx_err, &zero, sizeof(uint32_t), 0, cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(stream);
}

cudaError_t launch_softmax(const float* x, float* y, long long rows, int n, bool online,
                           cudaStream_t stream) {
  const bool vec = (n % 4 == 0) && ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 15u) == 0;
  const dim3 grid(static_cast<unsigned>(rows));
  if (online) {
    if (vec)
      sm::softmax_online_kernel<4><<<grid, sm::THREADS, 0, stream>>>(x, y, n);
    else
      sm::softmax_online_kernel<1><<<grid, sm::THREADS, 0, stream>>>(x, y, n);
  } else {
    if (vec)
      sm::softmax_safe_kernel<4><<<grid, sm::THREADS, 0, stream>>>(x, y, n);
    else
      sm::softmax_safe_kernel<1><<<grid, sm::THREADS, 0, stream>>>(x, y, n);
  }
  return cudaGetLastError();
}

}  // namespace fa
