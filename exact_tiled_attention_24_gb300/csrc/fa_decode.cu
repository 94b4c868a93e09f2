// Decode attention against a paged KV cache, split over the context, and the
// merge of partial attention results.
//
// Paged KV cache (CMU 10-423 L17–L18 notes, section 解碼端：PagedAttention):
// the cache is cut into blocks of a fixed number of tokens stored anywhere
// in memory; a block table maps a request's logical blocks to physical ones,
// and attention runs block by block. Decode ("07-16 下午" notes, section
// Prefill、Decode 与推理调度): each step brings one new token per request
// whose query attends to every cached token of that request, so the step
// reads the whole history of K and V and is bound by memory bandwidth.
//
// Merge ("07-16 下午" notes, section 长上下文与序列并行): partial softmax
// results over disjoint key blocks are combined by rescaling each block's
// normaliser and weighted sum by e^(m_block − m_global), not by adding
// separately normalised blocks. A partial result is kept as (o_s, lse_s)
// with o_s normalised within its block, so the combination is
//     lse = ln Σ_s e^(lse_s),   o = Σ_s e^(lse_s − lse) · o_s.
//
// Kernels:
//   decode_partial  one CTA per (context split, K/V head, request). It serves
//                   the G query heads that share the K/V head, so each K/V
//                   byte is read once per step. 64-key tiles of K and V are
//                   copied into shared memory by bulk copies (one per run of
//                   consecutive tokens inside a cache block), two tiles in
//                   flight; scores, the running (m, l) and the fp32 output
//                   rows stay on chip. Writes o_s (fp32) and lse_s per head.
//   merge           one warp per output row: the combination above.
// The work per byte is a few FMAs (G·d per key and head pair), far below the
// tensor-core ridge, so the products run on the FMA pipe.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "fa_common.h"
#include "fa_ptx.cuh"

namespace fa {

static __device__ uint32_t g_dec_err;

namespace dec {

constexpr int THREADS = 256;
constexpr int TK = 64;  // keys per tile
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.69314718055994531f;

template <int D, int GM>
struct Smem {
  static constexpr int ROW = D * 2;        // bytes of one key (or value) row
  static constexpr int TILE = TK * ROW;    // one K or V tile
  static constexpr int K_OFF = 0;          // K stages 0, 1
  static constexpr int V_OFF = 2 * TILE;   // V stages 0, 1
  static constexpr int Q_OFF = 4 * TILE;   // q rows fp32 [GM][D], times scale·log2 e
  static constexpr int P_OFF = Q_OFF + GM * D * 4;        // scores, then P: fp32 [GM][TK]
  static constexpr int ST_OFF = P_OFF + GM * TK * 4;      // m, l, alpha: fp32 [3][GM]
  static constexpr int TAB_OFF = ST_OFF + 3 * GM * 4;     // block-table slice, int32
  static constexpr int O_OFF = TAB_OFF + kDecodeMaxTable * 4;  // partial rows of key parts 1..
  static constexpr int PARTS = THREADS / D;               // key parts of the output pass
  static constexpr int BAR_OFF = O_OFF + (PARTS - 1) * GM * D * 4;
  static constexpr int BYTES = BAR_OFF + 2 * 8 + 16;
};

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

template <int D, int GM>
__global__ void __launch_bounds__(THREADS) decode_partial_kernel(
    const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k_cache,
    const __nv_bfloat16* __restrict__ v_cache, const int* __restrict__ block_table,
    const int* __restrict__ seq_lens, float* __restrict__ o_part, float* __restrict__ lse_part, int B,
    int H, int Hkv, int num_blocks, int bs, int max_blocks, float scale_log2) {
  using L = Smem<D, GM>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int S = gridDim.x;
  const int s = blockIdx.x, hk = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x;
  const int G = H / Hkv;
  uint32_t* err = &g_dec_err;

  // Context of request b, clamped to what its block-table row can address.
  int Lb = seq_lens[b];
  Lb = Lb < 0 ? 0 : (Lb > max_blocks * bs ? max_blocks * bs : Lb);
  const int n_tiles = (Lb + TK - 1) / TK;
  const int tps = (n_tiles + S - 1) / S;  // tiles per split
  const int tile0 = s * tps;
  const int tile1 = min(n_tiles, tile0 + tps);
  const size_t head0 = static_cast<size_t>(b) * H + static_cast<size_t>(hk) * G;  // first query head
  const size_t prow = static_cast<size_t>(s) * B * H + head0;                     // its partial row
  if (tile0 >= tile1) {  // no key in this split: o_s = 0, lse_s = -inf (weight 0 in the merge)
    for (int i = tid; i < G * D; i += THREADS) o_part[prow * D + i] = 0.f;
    if (tid < G) lse_part[prow + tid] = -INFINITY;
    return;
  }
  const int t_begin = tile0 * TK, t_end = min(Lb, tile1 * TK);
  const int blk0 = t_begin / bs;
  const int nblk = (t_end - 1) / bs + 1 - blk0;  // <= kDecodeMaxTable (checked on the host)

  uint8_t* sK = smem + L::K_OFF;
  uint8_t* sV = smem + L::V_OFF;
  float* sQ = reinterpret_cast<float*>(smem + L::Q_OFF);
  float* sP = reinterpret_cast<float*>(smem + L::P_OFF);
  float* sM = reinterpret_cast<float*>(smem + L::ST_OFF);
  float* sL = sM + GM;
  float* sA = sL + GM;
  int* sTab = reinterpret_cast<int*>(smem + L::TAB_OFF);
  float* sO = reinterpret_cast<float*>(smem + L::O_OFF);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);

  for (int i = tid; i < GM * D; i += THREADS) {
    const int g = i / D;
    sQ[i] = g < G ? __bfloat162float(q[(head0 + g) * D + (i % D)]) * scale_log2 : 0.f;
  }
  // Zero both stages: the tail rows of a partial tile then read as 0.
  for (int i = tid; i < 4 * L::TILE / 16; i += THREADS)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0u, 0u, 0u, 0u);
  for (int i = tid; i < nblk; i += THREADS) sTab[i] = block_table[static_cast<size_t>(b) * max_blocks + blk0 + i];
  if (tid < GM) {
    sM[tid] = -INFINITY;
    sL[tid] = 0.f;
  }
  if (tid == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    fence_mbar_init();
  }
  fence_async_smem();  // the zero fill before the bulk copies into the same bytes
  __syncthreads();

  // Thread 0: copy tile `tile` of K and V into stage st, one bulk copy per
  // run of consecutive tokens within a cache block. Entries outside
  // [0, num_blocks) are skipped (rows keep their old values) and reported.
  auto issue = [&](int tile, int st) {
    const int t0 = tile * TK, t1 = min(t_end, t0 + TK);
    uint32_t bytes = 0;
    for (int t = t0; t < t1;) {
      const int blk = sTab[t / bs - blk0];
      const int run = min(bs - t % bs, t1 - t);
      if (blk >= 0 && blk < num_blocks) bytes += static_cast<uint32_t>(run) * L::ROW;
      t += run;
    }
    mbar_arrive_expect_tx(&full[st], 2 * bytes);
    for (int t = t0; t < t1;) {
      const int blk = sTab[t / bs - blk0];
      const int off = t % bs;
      const int run = min(bs - off, t1 - t);
      if (blk >= 0 && blk < num_blocks) {
        const size_t src = ((static_cast<size_t>(blk) * Hkv + hk) * bs + off) * D;
        const uint32_t dst = static_cast<uint32_t>(t - t0) * L::ROW;
        bulk_load(sK + st * L::TILE + dst, k_cache + src, static_cast<uint32_t>(run) * L::ROW, &full[st]);
        bulk_load(sV + st * L::TILE + dst, v_cache + src, static_cast<uint32_t>(run) * L::ROW, &full[st]);
      } else {
        atomicExch(err, DEV_BAD_INDEX);
      }
      t += run;
    }
  };

  constexpr int PARTS = L::PARTS;
  constexpr int KP = TK / PARTS;  // keys per part in the output pass
  const int c = tid % D;          // output column of this thread
  const int part = tid / D;
  float acc[GM];
#pragma unroll
  for (int g = 0; g < GM; ++g) acc[g] = 0.f;

  if (tid == 0) issue(tile0, 0);
  int issued = 1;
  bool ok = true;
  int i = 0;
  for (int tile = tile0; tile < tile1; ++tile, ++i) {
    const int st = i & 1;
    if (tid == 0 && tile + 1 < tile1) {
      issue(tile + 1, st ^ 1);
      ++issued;
    }
    const bool waited = mbar_wait(&full[st], (i >> 1) & 1, err);
    if (__syncthreads_or(!waited)) {
      ok = false;
      break;
    }
    const int nk = min(t_end, (tile + 1) * TK) - tile * TK;
    // Scores (log2 units): thread -> key k, heads g = tid / TK + j·(THREADS / TK).
    // The 16-byte chunks of a row are visited in a rotated order so that the
    // threads of a phase hit distinct banks.
    {
      const int k = tid % TK;
      const uint4* kr = reinterpret_cast<const uint4*>(sK + st * L::TILE + k * L::ROW);
      for (int g = tid / TK; g < G; g += THREADS / TK) {
        const float* qr = sQ + g * D;
        float a = 0.f;
#pragma unroll 4
        for (int cc = 0; cc < D / 8; ++cc) {
          const int ch = (cc + k) & (D / 8 - 1);
          const uint4 kv = kr[ch];
          const float4 q0 = *reinterpret_cast<const float4*>(qr + ch * 8);
          const float4 q1 = *reinterpret_cast<const float4*>(qr + ch * 8 + 4);
          const __nv_bfloat162* k2 = reinterpret_cast<const __nv_bfloat162*>(&kv);
          const float2 f0 = __bfloat1622float2(k2[0]), f1 = __bfloat1622float2(k2[1]);
          const float2 f2 = __bfloat1622float2(k2[2]), f3 = __bfloat1622float2(k2[3]);
          a = fmaf(q0.x, f0.x, a);
          a = fmaf(q0.y, f0.y, a);
          a = fmaf(q0.z, f1.x, a);
          a = fmaf(q0.w, f1.y, a);
          a = fmaf(q1.x, f2.x, a);
          a = fmaf(q1.y, f2.y, a);
          a = fmaf(q1.z, f3.x, a);
          a = fmaf(q1.w, f3.y, a);
        }
        sP[g * TK + k] = k < nk ? a : -INFINITY;
      }
    }
    __syncthreads();
    // Online softmax per head (warp w takes heads w, w + 8, ...): raise m,
    // rescale l by 2^(m_old − m_new), P = 2^(s − m_new).
    {
      const int warp = tid >> 5, lane = tid & 31;
      for (int g = warp; g < G; g += THREADS / 32) {
        const float v0 = sP[g * TK + lane], v1 = sP[g * TK + lane + 32];
        const float m_old = sM[g];
        const float m_new = fmaxf(m_old, warp_max(fmaxf(v0, v1)));
        const float p0 = ex2(v0 - m_new), p1 = ex2(v1 - m_new);
        sP[g * TK + lane] = p0;
        sP[g * TK + lane + 32] = p1;
        const float sum = warp_sum(p0 + p1);
        if (lane == 0) {
          const float a = ex2(m_old - m_new);  // 0 on the first tile
          sA[g] = a;
          sL[g] = sL[g] * a + sum;
          sM[g] = m_new;
        }
      }
    }
    __syncthreads();
    // Output rows: thread -> column c, keys [part·KP, part·KP + KP).
    {
      const __nv_bfloat16* vt = reinterpret_cast<const __nv_bfloat16*>(sV + st * L::TILE);
#pragma unroll
      for (int g = 0; g < GM; ++g)
        if (g < G) acc[g] *= sA[g];
#pragma unroll 4
      for (int kk = 0; kk < KP; ++kk) {
        const int k = part * KP + kk;
        const float vv = __bfloat162float(vt[k * D + c]);
#pragma unroll
        for (int g = 0; g < GM; ++g)
          if (g < G) acc[g] = fmaf(sP[g * TK + k], vv, acc[g]);
      }
    }
    __syncthreads();  // stage st and sP are free for the next tiles
  }
  if (!ok) {
    // Let copies already issued land before the CTA exits (bounded).
    if (tid == 0)
      for (int j = i; j < issued; ++j) mbar_wait(&full[j & 1], (j >> 1) & 1, err);
    return;
  }
  // Sum the key parts and write o_s = u / l and lse_s = (m + log2 l)·ln 2.
  if (part > 0) {
#pragma unroll
    for (int g = 0; g < GM; ++g)
      if (g < G) sO[((part - 1) * GM + g) * D + c] = acc[g];
  }
  __syncthreads();
  if (part == 0) {
#pragma unroll
    for (int g = 0; g < GM; ++g) {
      if (g < G) {
        float u = acc[g];
        for (int p = 1; p < PARTS; ++p) u += sO[((p - 1) * GM + g) * D + c];
        o_part[(prow + g) * D + c] = u / sL[g];
      }
    }
  }
  if (tid < G) lse_part[prow + tid] = (sM[tid] + __log2f(sL[tid])) * LN2;
}

// One warp per output row: o = Σ_s e^(lse_s − lse) o_s, lse = ln Σ_s e^(lse_s).
template <int D>
__global__ void __launch_bounds__(256) merge_kernel(const float* __restrict__ o_parts,
                                                    const float* __restrict__ lse_parts, int S,
                                                    __nv_bfloat16* __restrict__ o, float* __restrict__ lse,
                                                    long long rows) {
  constexpr int CPL = D / 32;  // columns per lane
  const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  float m = -INFINITY;
  for (int s = lane; s < S; s += 32) m = fmaxf(m, lse_parts[s * rows + row]);
  m = warp_max(m);
  float l = 0.f;
  float acc[CPL];
#pragma unroll
  for (int j = 0; j < CPL; ++j) acc[j] = 0.f;
  if (m != -INFINITY) {
    for (int s = 0; s < S; ++s) {
      const float w = ex2((lse_parts[s * rows + row] - m) * LOG2E);
      l += w;
      const float* src = o_parts + (s * rows + row) * D + lane * CPL;
#pragma unroll
      for (int j = 0; j < CPL; ++j) acc[j] = fmaf(w, src[j], acc[j]);
    }
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
  for (int j = 0; j < CPL; j += 2)
    *reinterpret_cast<__nv_bfloat162*>(o + row * D + lane * CPL + j) =
        __floats2bfloat162_rn(acc[j] * inv, acc[j + 1] * inv);
  if (lane == 0) lse[row] = l > 0.f ? m + __logf(l) : -INFINITY;
}

template <int D, int GM>
static cudaError_t launch_partial_t(const void* q, const void* kc, const void* vc, const int* table,
                                    const int* seq_lens, float* o_part, float* lse_part, int B, int H,
                                    int Hkv, int num_blocks, int bs, int max_blocks, float scale, int S,
                                    cudaStream_t stream) {
  auto kern = decode_partial_kernel<D, GM>;
  const int smem = Smem<D, GM>::BYTES;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>(S), static_cast<unsigned>(Hkv), static_cast<unsigned>(B));
  kern<<<grid, THREADS, smem, stream>>>(static_cast<const __nv_bfloat16*>(q),
                                         static_cast<const __nv_bfloat16*>(kc),
                                         static_cast<const __nv_bfloat16*>(vc), table, seq_lens, o_part,
                                         lse_part, B, H, Hkv, num_blocks, bs, max_blocks,
                                         scale * LOG2E);
  return cudaGetLastError();
}

template <int D>
static cudaError_t launch_partial_d(const void* q, const void* kc, const void* vc, const int* table,
                                    const int* seq_lens, float* o_part, float* lse_part, int B, int H,
                                    int Hkv, int num_blocks, int bs, int max_blocks, float scale, int S,
                                    cudaStream_t stream) {
  const int G = H / Hkv;
  if (G <= 4)
    return launch_partial_t<D, 4>(q, kc, vc, table, seq_lens, o_part, lse_part, B, H, Hkv, num_blocks, bs,
                                  max_blocks, scale, S, stream);
  if (G <= 8)
    return launch_partial_t<D, 8>(q, kc, vc, table, seq_lens, o_part, lse_part, B, H, Hkv, num_blocks, bs,
                                  max_blocks, scale, S, stream);
  return launch_partial_t<D, 16>(q, kc, vc, table, seq_lens, o_part, lse_part, B, H, Hkv, num_blocks, bs,
                                 max_blocks, scale, S, stream);
}

}  // namespace dec

cudaError_t launch_attn_merge(const float* o_parts, const float* lse_parts, int S, void* o, float* lse,
                              long long rows, int d, cudaStream_t stream) {
  const unsigned blocks = static_cast<unsigned>((rows + 7) / 8);
  if (d == 64)
    dec::merge_kernel<64><<<blocks, 256, 0, stream>>>(o_parts, lse_parts, S,
                                                       static_cast<__nv_bfloat16*>(o), lse, rows);
  else
    dec::merge_kernel<128><<<blocks, 256, 0, stream>>>(o_parts, lse_parts, S,
                                                        static_cast<__nv_bfloat16*>(o), lse, rows);
  return cudaGetLastError();
}

cudaError_t launch_decode_paged(const void* q, const void* k_cache, const void* v_cache,
                                const int* block_table, const int* seq_lens, void* o, float* lse,
                                float* o_part, float* lse_part, int B, int H, int Hkv, int d,
                                int num_blocks, int block_size, int max_blocks, float scale, int S,
                                cudaStream_t stream) {
  cudaError_t e =
      d == 64 ? dec::launch_partial_d<64>(q, k_cache, v_cache, block_table, seq_lens, o_part, lse_part, B, H,
                                          Hkv, num_blocks, block_size, max_blocks, scale, S, stream)
              : dec::launch_partial_d<128>(q, k_cache, v_cache, block_table, seq_lens, o_part, lse_part, B,
                                           H, Hkv, num_blocks, block_size, max_blocks, scale, S, stream);
  if (e != cudaSuccess) return e;
  return launch_attn_merge(o_part, lse_part, S, o, lse, static_cast<long long>(B) * H, d, stream);
}

cudaError_t read_and_clear_decode_error(uint32_t* out, cudaStream_t stream) {
  cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_dec_err, sizeof(uint32_t), 0,
                                            cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return e;
  e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return e;
  const uint32_t zero = 0;
  e = cudaMemcpyToSymbolAsync(g_dec_err, &zero, sizeof(uint32_t), 0, cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(stream);
}

}  // namespace fa
