// Backward pass of exact attention by recomputation.
//
// The forward keeps only O and the per-row log-sum-exp; the backward never
// reads a stored attention matrix but rebuilds each P tile from Q, K and lse
// (CMU 10-423 L17–L18 notes, section "FlashAttention 本身", item 2:
// recompute the block when the backward needs it; dcwnkz.com GPU-tricks
// article, the recompute-instead-of-store trade-off, "选项 2"). With
// P = exp(scale·Q Kᵀ − lse) the gradients are
//     dV = Pᵀ dO,  dP = dO Vᵀ,  D_i = Σ_c dO_ic O_ic,  dS = P ∘ (dP − D),
//     dQ = scale · dS K,  dK = scale · dSᵀ Q.
//
// Three kernels:
//   preprocess  D = rowsum(dO ∘ O) and a zeroed fp32 dQ accumulator
//   main        one CTA per (head, 128-key tile): K_j, V_j stay in shared
//               memory, the CTA sweeps the 128-row query tiles (from the
//               diagonal on when causal). Sᵀ = K Qᵢᵀ and dPᵀ = V dOᵢᵀ land in
//               TMEM; the compute warps turn them into Pᵀ and dSᵀ (bf16,
//               written back into TMEM and, for dS, into shared memory);
//               dV += Pᵀ dOᵢ and dK += dSᵀ Qᵢ accumulate in TMEM for the
//               whole sweep; dQᵢ = dS K goes through TMEM and is added to
//               the fp32 accumulator with vector atomics.
//   dq_convert  dq = bf16(scale · dQ accumulator)
//
// Roles in the main kernel (192 threads): warp 0 TMA, warp 1 TMEM owner and
// MMA issuer, warps 2..5 compute (one thread per key row = TMEM lane).
// TMEM columns: dV 0.., dK 128.., S/P 256.., dP/dS 384..; dQᵢ reuses the S/P
// columns once the dV MMA that read P has completed.
#include <cuda_bf16.h>

#include "fa_common.h"
#include "fa_ptx.cuh"

namespace fa {

static __device__ uint32_t g_bwd_err;

namespace bwd {

// ------------------------------------------------------------ preprocess

template <int D>
__global__ void __launch_bounds__(256) preprocess_kernel(const __nv_bfloat16* __restrict__ o,
                                                         const __nv_bfloat16* __restrict__ dO,
                                                         float* __restrict__ Dvec,
                                                         float* __restrict__ dq_acc,
                                                         long long rows) {
  constexpr int TPR = D / 8;  // threads per row, 8 bf16 (16 bytes) each
  constexpr int RPB = 256 / TPR;
  const long long row = static_cast<long long>(blockIdx.x) * RPB + threadIdx.x / TPR;
  const int part = threadIdx.x % TPR;
  float acc = 0.f;
  if (row < rows) {
    const size_t off = static_cast<size_t>(row) * D + part * 8;
    const uint4 a = *reinterpret_cast<const uint4*>(o + off);
    const uint4 b = *reinterpret_cast<const uint4*>(dO + off);
    const __nv_bfloat162* ah = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* bh = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float2 fa2 = __bfloat1622float2(ah[t]);
      const float2 fb2 = __bfloat1622float2(bh[t]);
      acc = fmaf(fa2.x, fb2.x, acc);
      acc = fmaf(fa2.y, fb2.y, acc);
    }
    float4* z = reinterpret_cast<float4*>(dq_acc + off);
    z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int w = TPR / 2; w > 0; w >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, w);
  if (row < rows && part == 0) Dvec[row] = acc;
}

// ------------------------------------------------------------ dq convert

__global__ void __launch_bounds__(256) dq_convert_kernel(const float* __restrict__ acc,
                                                         __nv_bfloat16* __restrict__ dq,
                                                         long long n8, float scale) {
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const float4 a = reinterpret_cast<const float4*>(acc)[2 * i];
    const float4 b = reinterpret_cast<const float4*>(acc)[2 * i + 1];
    uint4 out;
    out.x = pack_bf16x2(a.x * scale, a.y * scale);
    out.y = pack_bf16x2(a.z * scale, a.w * scale);
    out.z = pack_bf16x2(b.x * scale, b.y * scale);
    out.w = pack_bf16x2(b.z * scale, b.w * scale);
    reinterpret_cast<uint4*>(dq)[i] = out;
  }
}

// ------------------------------------------------------------ main kernel

constexpr int BK = 128;  // keys per CTA
constexpr int BQ = 128;  // query rows per tile
constexpr int THREADS = 192;
constexpr uint32_t COL_DV = 0, COL_DK = 128, COL_S = 256, COL_DP = 384;

template <int D>
struct Smem {
  static constexpr int PANELS = D / 64;
  static constexpr int STAGES = 2;
  static constexpr int TILE = 128 * D * 2;
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = K_OFF + TILE;
  static constexpr int Q_OFF = V_OFF + TILE;
  static constexpr int DO_OFF = Q_OFF + STAGES * TILE;
  static constexpr int DS_OFF = DO_OFF + STAGES * TILE;
  static constexpr int DS_BYTES = BK * BQ * 2;
  static constexpr int LSE_OFF = DS_OFF + DS_BYTES;   // 128 floats (log2 units)
  static constexpr int DV_OFF = LSE_OFF + BQ * 4;     // 128 floats
  static constexpr int BAR_OFF = DV_OFF + BQ * 4;
  // kv_full, q_full[2], q_empty[2], sdp_full, ds_ready, mma2_done, dq_full, dq_free, final
  static constexpr int NBARS = 1 + 2 * STAGES + 6;
  static constexpr int TMEM_SLOT_OFF = BAR_OFF + NBARS * 8;
  static constexpr int BYTES = TMEM_SLOT_OFF + 16;
  static constexpr int ALLOC = BYTES + 1024;
};

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(THREADS, 1)
    bwd_main_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                    const __grid_constant__ CUtensorMap tdk,
                    const __grid_constant__ CUtensorMap tdv, const float* __restrict__ lse,
                    const float* __restrict__ Dvec, float* __restrict__ dq_acc, int BH, int N,
                    float scale, float scale_log2) {
  using L = Smem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sK = smem + L::K_OFF;
  uint8_t* sV = smem + L::V_OFF;
  uint8_t* sQ = smem + L::Q_OFF;
  uint8_t* sdO = smem + L::DO_OFF;
  uint8_t* sdS = smem + L::DS_OFF;
  float* sLse = reinterpret_cast<float*>(smem + L::LSE_OFF);
  float* sDv = reinterpret_cast<float*>(smem + L::DV_OFF);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint64_t* kv_full = bars;
  uint64_t* q_full = bars + 1;
  uint64_t* q_empty = q_full + L::STAGES;
  uint64_t* sdp_full = q_empty + L::STAGES;
  uint64_t* ds_ready = sdp_full + 1;
  uint64_t* mma2_done = ds_ready + 1;
  uint64_t* dq_full = mma2_done + 1;
  uint64_t* dq_free = dq_full + 1;
  uint64_t* final_bar = dq_free + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::TMEM_SLOT_OFF);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_kt = (N + BK - 1) / BK;
  const int n_qt = (N + BQ - 1) / BQ;
  const int kt = static_cast<int>(blockIdx.x) / BH;  // causal: heaviest key tile first
  const int bh = static_cast<int>(blockIdx.x) % BH;
  const int k0 = kt * BK;
  const int qt_begin = CAUSAL ? kt : 0;  // BQ == BK
  const int n_it = n_qt - qt_begin;
  (void)n_kt;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < L::STAGES; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);
    }
    mbar_init(sdp_full, 1);
    mbar_init(ds_ready, 4);
    mbar_init(mma2_done, 1);
    mbar_init(dq_full, 1);
    mbar_init(dq_free, 4);
    mbar_init(final_bar, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  uint32_t* err = &g_bwd_err;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tq);
      prefetch_tmap(&tk);
      prefetch_tmap(&tv);
      prefetch_tmap(&tdo);
      mbar_arrive_expect_tx(kv_full, 2 * L::TILE);
      for (int p = 0; p < L::PANELS; ++p) {
        tma_load_3d(sK + p * (BK * 128), &tk, kv_full, p * 64, k0, bh);
        tma_load_3d(sV + p * (BK * 128), &tv, kv_full, p * 64, k0, bh);
      }
      int issued = 0;
      for (int it = 0; it < n_it; ++it) {
        const int s = it % L::STAGES;
        if (!mbar_wait(&q_empty[s], ((it / L::STAGES) & 1) ^ 1, err)) break;
        const int q0 = (qt_begin + it) * BQ;
        mbar_arrive_expect_tx(&q_full[s], 2 * L::TILE);
        for (int p = 0; p < L::PANELS; ++p) {
          tma_load_3d(sQ + s * L::TILE + p * (BQ * 128), &tq, &q_full[s], p * 64, q0, bh);
          tma_load_3d(sdO + s * L::TILE + p * (BQ * 128), &tdo, &q_full[s], p * 64, q0, bh);
        }
        issued = it + 1;
      }
      mbar_wait(kv_full, 0, err);
      for (int it = max(0, issued - L::STAGES); it < issued; ++it)
        mbar_wait(&q_full[it % L::STAGES], (it / L::STAGES) & 1, err);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16(BK, BQ, false, false);  // Sᵀ, dPᵀ: 128x128, K = D
      constexpr uint32_t id_g = idesc_bf16(BK, D, false, true);    // dV, dK: B MN-major
      constexpr uint32_t id_q = idesc_bf16(BQ, D, true, true);     // dQ: A and B MN-major
      bool ok = mbar_wait(kv_full, 0, err);
      const uint32_t k_base = smem_u32(sK);
      const uint32_t v_base = smem_u32(sV);
      const uint32_t ds_base = smem_u32(sdS);
      for (int it = 0; it < n_it && ok; ++it) {
        const int s = it % L::STAGES;
        const uint32_t q_base = smem_u32(sQ + s * L::TILE);
        const uint32_t do_base = smem_u32(sdO + s * L::TILE);
        ok = mbar_wait(&q_full[s], (it / L::STAGES) & 1, err);
        if (ok && it > 0) ok = mbar_wait(dq_free, (it - 1) & 1, err);  // S/P columns free
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t poff = (ks / 4) * (128 * 128);
          const uint32_t kin = (ks % 4) * 16;
          mma_ss(tmem + COL_S, sdesc_kmajor(k_base + poff, kin), sdesc_kmajor(q_base + poff, kin),
                 id_s, ks > 0);
        }
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t poff = (ks / 4) * (128 * 128);
          const uint32_t kin = (ks % 4) * 16;
          mma_ss(tmem + COL_DP, sdesc_kmajor(v_base + poff, kin),
                 sdesc_kmajor(do_base + poff, kin), id_s, ks > 0);
        }
        tc_commit(sdp_full);
        ok = mbar_wait(ds_ready, it & 1, err);
        if (!ok) break;
        tc_fence_after();
        // dV += Pᵀ dOᵢ ; dK += dSᵀ Qᵢ   (A from TMEM, B MN-major in smem)
#pragma unroll
        for (int ks = 0; ks < BQ / 16; ++ks) {
          mma_ts(tmem + COL_DV, tmem + COL_S + ks * 8, sdesc_mnmajor(do_base, ks * 16, BQ * 128),
                 id_g, (it > 0 || ks > 0) ? 1u : 0u);
        }
#pragma unroll
        for (int ks = 0; ks < BQ / 16; ++ks) {
          mma_ts(tmem + COL_DK, tmem + COL_DP + ks * 8, sdesc_mnmajor(q_base, ks * 16, BQ * 128),
                 id_g, (it > 0 || ks > 0) ? 1u : 0u);
        }
        tc_commit(mma2_done);
        tc_commit(&q_empty[s]);
        // dQᵢ overwrites the S/P columns: only after the dV MMA has read P.
        ok = mbar_wait(mma2_done, it & 1, err);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < BK / 16; ++ks) {
          mma_ss(tmem + COL_S, sdesc_mnmajor(ds_base, ks * 16, BK * 128),
                 sdesc_mnmajor(k_base, ks * 16, BK * 128), id_q, ks > 0);
        }
        tc_commit(dq_full);
      }
      tc_commit(final_bar);
      mbar_wait(final_bar, 0, err);
    }
  } else {
    // ------------------------------------------------------------ compute
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // TMEM lane: key row (S, dP, dK, dV) or query row (dQ)
    const int key = k0 + r;
    const bool key_ok = key < N;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const float* lse_h = lse + static_cast<size_t>(bh) * N;
    const float* D_h = Dvec + static_cast<size_t>(bh) * N;
    float* dq_h = dq_acc + static_cast<size_t>(bh) * N * D;
    constexpr float LOG2E = 1.4426950408889634f;
    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
      const int qt = qt_begin + it;
      const int q0 = qt * BQ;
      // Stage this tile's lse (log2 units) and D; rows past N get lse=+inf (P = 0).
      named_bar_sync(1, 128);
      {
        const int q = q0 + r;
        sLse[r] = (q < N) ? lse_h[q] * LOG2E : INFINITY;
        sDv[r] = (q < N) ? D_h[q] : 0.f;
      }
      named_bar_sync(1, 128);
      ok = mbar_wait(sdp_full, it & 1, err);
      if (!ok) break;
      tc_fence_after();
      const uint32_t s_addr = tmem + lane_addr + COL_S;
      const uint32_t dp_addr = tmem + lane_addr + COL_DP;
      float p[BQ];
      {
        uint32_t raw[4][32];
        tmem_ld32(s_addr + 0, raw[0]);
        tmem_ld32(s_addr + 32, raw[1]);
        tmem_ld32(s_addr + 64, raw[2]);
        tmem_ld32(s_addr + 96, raw[3]);
        tmem_ld_wait();
        const bool diag = CAUSAL && (qt == kt);
#pragma unroll
        for (int c = 0; c < BQ; ++c) {
          float v = ex2(fmaf(__uint_as_float(raw[c / 32][c % 32]), scale_log2, -sLse[c]));
          if (!key_ok || (diag && c < r)) v = 0.f;
          p[c] = v;
        }
      }
      {
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < BQ; c += 32) {
#pragma unroll
          for (int t = 0; t < 16; ++t) pk[t] = pack_bf16x2(p[c + 2 * t], p[c + 2 * t + 1]);
          tmem_st16(s_addr + c / 2, pk);
        }
      }
      // dSᵀ = Pᵀ ∘ (dPᵀ − D): into TMEM (for dK) and shared memory (for dQ).
#pragma unroll
      for (int c = 0; c < BQ; c += 32) {
        uint32_t raw[32];
        tmem_ld32(dp_addr + c, raw);
        tmem_ld_wait();
        uint32_t pk[16];
#pragma unroll
        for (int t = 0; t < 16; ++t) {
          const float d0 = p[c + 2 * t] * (__uint_as_float(raw[2 * t]) - sDv[c + 2 * t]);
          const float d1 = p[c + 2 * t + 1] * (__uint_as_float(raw[2 * t + 1]) - sDv[c + 2 * t + 1]);
          pk[t] = pack_bf16x2(d0, d1);
        }
        tmem_st16(dp_addr + c / 2, pk);
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          const int col0 = c + ch * 8;
          const int panel = col0 / 64;
          const int chunk = (col0 % 64) / 8;
          *reinterpret_cast<uint4*>(sdS + panel * (BK * 128) + r * 128 + ((chunk ^ (r & 7)) * 16)) =
              make_uint4(pk[ch * 4], pk[ch * 4 + 1], pk[ch * 4 + 2], pk[ch * 4 + 3]);
        }
      }
      tmem_st_wait();
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ds_ready);
      // dQᵢ (unscaled) from TMEM, lane = query row, added into the accumulator.
      ok = mbar_wait(dq_full, it & 1, err);
      if (!ok) break;
      tc_fence_after();
      {
        const int q = q0 + r;
        float* dst = dq_h + static_cast<size_t>(q) * D;
#pragma unroll
        for (int c = 0; c < D; c += 32) {
          uint32_t raw[32];
          tmem_ld32(s_addr + c, raw);
          tmem_ld_wait();
          if (q < N) {
#pragma unroll
            for (int t = 0; t < 8; ++t) {
              atomicAdd(reinterpret_cast<float4*>(dst + c + 4 * t),
                        make_float4(__uint_as_float(raw[4 * t]), __uint_as_float(raw[4 * t + 1]),
                                    __uint_as_float(raw[4 * t + 2]),
                                    __uint_as_float(raw[4 * t + 3])));
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dq_free);
    }
    // -------------------------------------------------------------- epilogue
    // The last dq_full implies every MMA of this CTA has completed; the Q/dO
    // stage-0 buffers are free and serve as staging for dK and dV.
    named_bar_sync(1, 128);
    if (ok) {
      tc_fence_after();
      uint8_t* stage_dk = sQ;
      uint8_t* stage_dv = sdO;
#pragma unroll
      for (int c = 0; c < D; c += 32) {
        uint32_t a[32], b[32];
        tmem_ld32(tmem + lane_addr + COL_DK + c, a);
        tmem_ld32(tmem + lane_addr + COL_DV + c, b);
        tmem_ld_wait();
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          const int col0 = c + ch * 8;
          const int panel = col0 / 64;
          const int chunk = (col0 % 64) / 8;
          const int off = panel * (BK * 128) + r * 128 + ((chunk ^ (r & 7)) * 16);
          uint4 vk, vv;
          vk.x = pack_bf16x2(__uint_as_float(a[ch * 8 + 0]) * scale, __uint_as_float(a[ch * 8 + 1]) * scale);
          vk.y = pack_bf16x2(__uint_as_float(a[ch * 8 + 2]) * scale, __uint_as_float(a[ch * 8 + 3]) * scale);
          vk.z = pack_bf16x2(__uint_as_float(a[ch * 8 + 4]) * scale, __uint_as_float(a[ch * 8 + 5]) * scale);
          vk.w = pack_bf16x2(__uint_as_float(a[ch * 8 + 6]) * scale, __uint_as_float(a[ch * 8 + 7]) * scale);
          vv.x = pack_bf16x2(__uint_as_float(b[ch * 8 + 0]), __uint_as_float(b[ch * 8 + 1]));
          vv.y = pack_bf16x2(__uint_as_float(b[ch * 8 + 2]), __uint_as_float(b[ch * 8 + 3]));
          vv.z = pack_bf16x2(__uint_as_float(b[ch * 8 + 4]), __uint_as_float(b[ch * 8 + 5]));
          vv.w = pack_bf16x2(__uint_as_float(b[ch * 8 + 6]), __uint_as_float(b[ch * 8 + 7]));
          *reinterpret_cast<uint4*>(stage_dk + off) = vk;
          *reinterpret_cast<uint4*>(stage_dv + off) = vv;
        }
      }
      fence_async_smem();
    }
    named_bar_sync(1, 128);
    if (ok && warp == 2 && lane == 0) {
      for (int p = 0; p < L::PANELS; ++p) {
        tma_store_3d(&tdk, sQ + p * (BK * 128), p * 64, k0, bh);
        tma_store_3d(&tdv, sdO + p * (BK * 128), p * 64, k0, bh);
      }
      tma_store_commit();
      tma_store_wait_all();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool CAUSAL>
static cudaError_t launch_main_t(const CUtensorMap& tq, const CUtensorMap& tk,
                                 const CUtensorMap& tv, const CUtensorMap& tdo,
                                 const CUtensorMap& tdk, const CUtensorMap& tdv, const float* lse,
                                 const float* Dvec, float* dq_acc, int BH, int N, float scale,
                                 cudaStream_t stream) {
  auto kern = bwd_main_kernel<D, CAUSAL>;
  const int smem = Smem<D>::ALLOC;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int n_kt = (N + BK - 1) / BK;
  dim3 grid(static_cast<unsigned>(n_kt) * static_cast<unsigned>(BH));
  kern<<<grid, THREADS, smem, stream>>>(tq, tk, tv, tdo, tdk, tdv, lse, Dvec, dq_acc, BH, N, scale,
                                        scale * 1.4426950408889634f);
  return cudaGetLastError();
}

}  // namespace bwd

cudaError_t launch_bwd_preprocess(const __nv_bfloat16* o, const __nv_bfloat16* dO, float* Dvec,
                                  float* dq_acc, int BH, int N, int d, cudaStream_t stream) {
  const long long rows = static_cast<long long>(BH) * N;
  if (d == 64) {
    const long long blocks = (rows + 31) / 32;
    bwd::preprocess_kernel<64><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(o, dO, Dvec, dq_acc, rows);
  } else {
    const long long blocks = (rows + 15) / 16;
    bwd::preprocess_kernel<128><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(o, dO, Dvec, dq_acc, rows);
  }
  return cudaGetLastError();
}

cudaError_t launch_bwd_main(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const CUtensorMap& tdk,
                            const CUtensorMap& tdv, const float* lse, const float* Dvec,
                            float* dq_acc, int BH, int N, int d, float scale, bool causal,
                            cudaStream_t stream) {
  if (d == 64)
    return causal ? bwd::launch_main_t<64, true>(tq, tk, tv, tdo, tdk, tdv, lse, Dvec, dq_acc, BH, N, scale, stream)
                  : bwd::launch_main_t<64, false>(tq, tk, tv, tdo, tdk, tdv, lse, Dvec, dq_acc, BH, N, scale, stream);
  return causal ? bwd::launch_main_t<128, true>(tq, tk, tv, tdo, tdk, tdv, lse, Dvec, dq_acc, BH, N, scale, stream)
                : bwd::launch_main_t<128, false>(tq, tk, tv, tdo, tdk, tdv, lse, Dvec, dq_acc, BH, N, scale, stream);
}

cudaError_t launch_bwd_dq_convert(const float* dq_acc, __nv_bfloat16* dq, int BH, int N, int d,
                                  float scale, cudaStream_t stream) {
  const long long n8 = static_cast<long long>(BH) * N * d / 8;
  long long blocks = (n8 + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (blocks < 1) blocks = 1;
  bwd::dq_convert_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(dq_acc, dq, n8, scale);
  return cudaGetLastError();
}

cudaError_t read_and_clear_bwd_error(uint32_t* out, cudaStream_t stream) {
  cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_bwd_err, sizeof(uint32_t), 0,
                                            cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return e;
  e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return e;
  const uint32_t zero = 0;
  e = cudaMemcpyToSymbolAsync(g_bwd_err, &zero, sizeof(uint32_t), 0, cudaMemcpyHostToDevice,
                              stream);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(stream);
}

}  // namespace fa
