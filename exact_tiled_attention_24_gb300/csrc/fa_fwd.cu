// Forward pass of exact attention, computed tile by tile with online softmax.
//
// Method (CMU 10-423 L17–L18 notes, section "FlashAttention 本身"; dcwnkz.com
// GPU-tricks article, FlashAttention section and its six-score worked
// example): for one block of 128 query rows, sweep the keys/values in tiles
// of 128; keep per row the running max m, the running denominator l and the
// running weighted sum O; when a tile raises m, multiply l and O by
// e^(m_old - m_new) before adding the tile; divide by l once at the end.
// S = Q Kᵀ and P never leave the SM: S lives in tensor memory (TMEM), P is
// written back into TMEM as bf16 and fed straight to the P·V MMA.
//
// Roles inside one CTA (192 threads):
//   warp 0      TMA producer: Q once, then K_j / V_j into a 2-stage ring
//   warp 1      TMEM owner and MMA issuer (one elected lane)
//   warps 2..5  softmax: one thread per query row (TMEM lane), rescale of O,
//               epilogue (O / l -> bf16 -> TMA store, lse)
// TMEM columns: three S buffers at 0, 128, 256 (so S_{j+3} is only written
// after the P·V MMA that read buffer j%3 has completed), O at 384.
//
// Causal masking ("07-16 下午：分布式大模型训练与推理", section 自回归语言模型推理):
// query i sees keys j <= i; tiles above the diagonal are skipped, the
// diagonal tile is masked. Keys at or past N (ragged last tile) are masked.
#include <cuda_bf16.h>

#include "fa_common.h"
#include "fa_ptx.cuh"
#include "fa_tmap.h"

namespace fa {

static __device__ uint32_t g_fwd_err;

namespace fwd {

constexpr int BM = 128;       // query rows per CTA
constexpr int BN = 128;       // keys per tile
constexpr int NSB = 3;        // S buffers in TMEM
constexpr int THREADS = 192;  // 6 warps
constexpr uint32_t O_COL = 384;
constexpr int HEAD_GROUP = 8;

template <int D>
struct Smem {
  static constexpr int PANELS = D / 64;
  static constexpr int STAGES = 2;
  static constexpr int TILE_BYTES = BM * D * 2;  // = BN * D * 2
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + TILE_BYTES;
  static constexpr int V_OFF = K_OFF + STAGES * TILE_BYTES;
  static constexpr int BAR_OFF = V_OFF + STAGES * TILE_BYTES;
  // barriers: q_full, k_full[2], k_empty[2], v_full[2], v_empty[2],
  //           s_full[3], p_ready[3], pv_done[3], final
  static constexpr int NBARS = 1 + 4 * STAGES + 3 * NSB + 1;
  static constexpr int TMEM_SLOT_OFF = BAR_OFF + NBARS * 8;
  static constexpr int BYTES = TMEM_SLOT_OFF + 16;
  // Slack for 1024-byte alignment; at least 116 KB so that only one CTA
  // (and one 512-column TMEM allocation) is resident per SM.
  static constexpr int ALLOC = (BYTES + 1024) > 118784 ? (BYTES + 1024) : 118784;
};

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(THREADS, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap to,
                  float* __restrict__ lse, int BH, int N, float scale_log2) {
  using L = Smem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem + L::Q_OFF;
  uint8_t* sK = smem + L::K_OFF;
  uint8_t* sV = smem + L::V_OFF;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + L::STAGES;
  uint64_t* v_full = k_empty + L::STAGES;
  uint64_t* v_empty = v_full + L::STAGES;
  uint64_t* s_full = v_empty + L::STAGES;
  uint64_t* p_ready = s_full + NSB;
  uint64_t* pv_done = p_ready + NSB;
  uint64_t* final_bar = pv_done + NSB;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::TMEM_SLOT_OFF);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Heads in groups of HEAD_GROUP (their K/V stay in L2 while the group
  // runs); within a group the heaviest (causal) query tiles go first.
  const int n_qt = (N + BM - 1) / BM;
  int t, bh;
  grouped_tile_order(static_cast<int>(blockIdx.x), BH, n_qt, HEAD_GROUP, &t, &bh);
  const int qt = n_qt - 1 - t;
  const int q0 = qt * BM;
  const int n_kt_all = (N + BN - 1) / BN;
  const int n_kt = CAUSAL ? min(n_kt_all, qt + 1) : n_kt_all;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < L::STAGES; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int b = 0; b < NSB; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&p_ready[b], 4);
      mbar_init(&pv_done[b], 1);
    }
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
  uint32_t* err = &g_fwd_err;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tq);
      prefetch_tmap(&tk);
      prefetch_tmap(&tv);
      mbar_arrive_expect_tx(q_full, L::TILE_BYTES);
      for (int p = 0; p < L::PANELS; ++p) tma_load_3d(sQ + p * (BM * 128), &tq, q_full, p * 64, q0, bh);
      int issued = 0;
      bool ok = true;
      for (int j = 0; j < n_kt && ok; ++j) {
        const int s = j % L::STAGES;
        const uint32_t ph = (j / L::STAGES) & 1;
        ok = mbar_wait(&k_empty[s], ph ^ 1, err);
        if (!ok) break;
        mbar_arrive_expect_tx(&k_full[s], L::TILE_BYTES);
        for (int p = 0; p < L::PANELS; ++p)
          tma_load_3d(sK + s * L::TILE_BYTES + p * (BN * 128), &tk, &k_full[s], p * 64, j * BN, bh);
        ok = mbar_wait(&v_empty[s], ph ^ 1, err);
        if (!ok) break;
        mbar_arrive_expect_tx(&v_full[s], L::TILE_BYTES);
        for (int p = 0; p < L::PANELS; ++p)
          tma_load_3d(sV + s * L::TILE_BYTES + p * (BN * 128), &tv, &v_full[s], p * 64, j * BN, bh);
        issued = j + 1;
      }
      // Drain: never leave the CTA with copies still landing in its smem.
      mbar_wait(q_full, 0, err);
      for (int j = max(0, issued - L::STAGES); j < issued; ++j) {
        const int s = j % L::STAGES;
        const uint32_t ph = (j / L::STAGES) & 1;
        mbar_wait(&k_full[s], ph, err);
        mbar_wait(&v_full[s], ph, err);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16(BM, BN, false, false);
      constexpr uint32_t idesc_o = idesc_bf16(BM, D, false, true);
      bool ok = mbar_wait(q_full, 0, err);
      auto issue_s = [&](int jj) -> bool {
        const int s = jj % L::STAGES;
        if (!mbar_wait(&k_full[s], (jj / L::STAGES) & 1, err)) return false;
        tc_fence_after();
        const uint32_t d_tmem = tmem + (jj % NSB) * BN;
        const uint32_t q_base = smem_u32(sQ);
        const uint32_t k_base = smem_u32(sK + s * L::TILE_BYTES);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t poff = (ks / 4) * (BM * 128);
          mma_ss(d_tmem, sdesc_kmajor(q_base + poff, (ks % 4) * 16),
                 sdesc_kmajor(k_base + poff, (ks % 4) * 16), idesc_s, ks > 0);
        }
        tc_commit(&s_full[jj % NSB]);
        tc_commit(&k_empty[s]);
        return true;
      };
      for (int jj = 0; jj < min(NSB, n_kt) && ok; ++jj) ok = issue_s(jj);
      for (int j = 0; j < n_kt && ok; ++j) {
        const int s = j % L::STAGES;
        const int b = j % NSB;
        ok = mbar_wait(&v_full[s], (j / L::STAGES) & 1, err) &&
             mbar_wait(&p_ready[b], (j / NSB) & 1, err);
        if (!ok) break;
        tc_fence_after();
        const uint32_t v_base = smem_u32(sV + s * L::TILE_BYTES);
        const uint32_t p_tmem = tmem + b * BN;
#pragma unroll
        for (int ks = 0; ks < BN / 16; ++ks) {
          mma_ts(tmem + O_COL, p_tmem + ks * 8, sdesc_mnmajor(v_base, ks * 16, BN * 128), idesc_o,
                 (j > 0 || ks > 0) ? 1u : 0u);
        }
        tc_commit(&pv_done[b]);
        tc_commit(&v_empty[s]);
        // S_{j+2} reuses the buffer of P_{j-1}: wait until P V_{j-1} is done.
        if (j >= 1 && j + 2 < n_kt) {
          ok = mbar_wait(&pv_done[(j - 1) % NSB], ((j - 1) / NSB) & 1, err);
          if (ok) ok = issue_s(j + 2);
        }
      }
      // All issued MMAs complete before TMEM is released.
      tc_commit(final_bar);
      mbar_wait(final_bar, 0, err);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
    const int r = quarter * 32 + lane;
    const int qrow = q0 + r;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    float m = -INFINITY;  // running max, in log2 units of scaled scores
    float l = 0.f;        // running denominator
    bool ok = true;
    for (int j = 0; j < n_kt; ++j) {
      const int b = j % NSB;
      ok = mbar_wait(&s_full[b], (j / NSB) & 1, err);
      if (!ok) break;
      tc_fence_after();
      const uint32_t s_addr = tmem + lane_addr + b * BN;
      uint32_t raw[4][32];
      tmem_ld32(s_addr + 0, raw[0]);
      tmem_ld32(s_addr + 32, raw[1]);
      tmem_ld32(s_addr + 64, raw[2]);
      tmem_ld32(s_addr + 96, raw[3]);
      tmem_ld_wait();
      float x[BN];
#pragma unroll
      for (int c = 0; c < BN; ++c) x[c] = __uint_as_float(raw[c / 32][c % 32]);
      const int k0 = j * BN;
      const bool need_mask = (k0 + BN > N) || (CAUSAL && k0 + BN - 1 > q0);
      if (need_mask) {
#pragma unroll
        for (int c = 0; c < BN; ++c) {
          const int key = k0 + c;
          if (key >= N || (CAUSAL && key > qrow)) x[c] = -INFINITY;
        }
      }
      float mx0 = x[0], mx1 = x[1], mx2 = x[2], mx3 = x[3];
#pragma unroll
      for (int c = 4; c < BN; c += 4) {
        mx0 = fmaxf(mx0, x[c]);
        mx1 = fmaxf(mx1, x[c + 1]);
        mx2 = fmaxf(mx2, x[c + 2]);
        mx3 = fmaxf(mx3, x[c + 3]);
      }
      const float tile_max = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * scale_log2;
      const float m_new = fmaxf(m, tile_max);
      const float alpha = ex2(m - m_new);  // e^(m_old - m_new); 0 on the first tile
      float sum0 = 0.f, sum1 = 0.f;
      uint32_t pk[BN / 2];
#pragma unroll
      for (int c = 0; c < BN; c += 2) {
        const float p0 = ex2(fmaf(x[c], scale_log2, -m_new));
        const float p1 = ex2(fmaf(x[c + 1], scale_log2, -m_new));
        sum0 += p0;
        sum1 += p1;
        pk[c / 2] = pack_bf16x2(p0, p1);
      }
      l = l * alpha + (sum0 + sum1);
      m = m_new;
      // P (bf16) overwrites the first 64 columns of this S buffer.
#pragma unroll
      for (int c = 0; c < BN / 2; c += 16) {
        uint32_t part[16];
#pragma unroll
        for (int t = 0; t < 16; ++t) part[t] = pk[c + t];
        tmem_st16(s_addr + c, part);
      }
      // Rescale O by alpha once P V_{j-1} has landed (skipped when the whole
      // warp's rows kept their max, i.e. alpha == 1 everywhere).
      if (j > 0) {
        ok = mbar_wait(&pv_done[(j - 1) % NSB], ((j - 1) / NSB) & 1, err);
        if (!ok) break;
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
          const uint32_t o_addr = tmem + lane_addr + O_COL;
#pragma unroll
          for (int c = 0; c < D; c += 32) {
            uint32_t o[32];
            tmem_ld32(o_addr + c, o);
            tmem_ld_wait();
            uint32_t a[16], bb[16];
#pragma unroll
            for (int t = 0; t < 16; ++t) {
              a[t] = __float_as_uint(__uint_as_float(o[t]) * alpha);
              bb[t] = __float_as_uint(__uint_as_float(o[16 + t]) * alpha);
            }
            tmem_st16(o_addr + c, a);
            tmem_st16(o_addr + c + 16, bb);
          }
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_ready[b]);
    }
    // -------------------------------------------------------------- epilogue
    if (ok) ok = mbar_wait(&pv_done[(n_kt - 1) % NSB], ((n_kt - 1) / NSB) & 1, err);
    if (ok) {
      tc_fence_after();
      const float inv_l = 1.f / l;
      const uint32_t o_addr = tmem + lane_addr + O_COL;
#pragma unroll
      for (int c = 0; c < D; c += 32) {
        uint32_t o[32];
        tmem_ld32(o_addr + c, o);
        tmem_ld_wait();
        // 32 columns = 4 chunks of 16 bytes, written in the 128-byte swizzle.
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          const int col0 = c + ch * 8;
          const int panel = col0 / 64;
          const int chunk = (col0 % 64) / 8;
          uint4 val;
          val.x = pack_bf16x2(__uint_as_float(o[ch * 8 + 0]) * inv_l, __uint_as_float(o[ch * 8 + 1]) * inv_l);
          val.y = pack_bf16x2(__uint_as_float(o[ch * 8 + 2]) * inv_l, __uint_as_float(o[ch * 8 + 3]) * inv_l);
          val.z = pack_bf16x2(__uint_as_float(o[ch * 8 + 4]) * inv_l, __uint_as_float(o[ch * 8 + 5]) * inv_l);
          val.w = pack_bf16x2(__uint_as_float(o[ch * 8 + 6]) * inv_l, __uint_as_float(o[ch * 8 + 7]) * inv_l);
          *reinterpret_cast<uint4*>(sQ + panel * (BM * 128) + r * 128 + ((chunk ^ (r & 7)) * 16)) = val;
        }
      }
      if (qrow < N) {
        // lse in natural-log units: (m + log2 l) * ln 2
        lse[static_cast<size_t>(bh) * N + qrow] = (m + __log2f(l)) * 0.69314718055994531f;
      }
      fence_async_smem();
    }
    named_bar_sync(1, 128);
    if (ok && warp == 2 && lane == 0) {
      for (int p = 0; p < L::PANELS; ++p) tma_store_3d(&to, sQ + p * (BM * 128), p * 64, q0, bh);
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
static cudaError_t launch_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& to, float* lse, int BH, int N, float scale,
                            cudaStream_t stream) {
  auto kern = fa_fwd_kernel<D, CAUSAL>;
  const int smem = Smem<D>::ALLOC;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int n_qt = (N + BM - 1) / BM;
  dim3 grid(static_cast<unsigned>(n_qt) * static_cast<unsigned>(BH));
  const float scale_log2 = scale * 1.4426950408889634f;
  kern<<<grid, THREADS, smem, stream>>>(tq, tk, tv, to, lse, BH, N, scale_log2);
  return cudaGetLastError();
}

}  // namespace fwd

cudaError_t launch_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int BH,
                       int N, int d, float scale, bool causal, cudaStream_t stream) {
  CUtensorMap tq, tk, tv, to;
  if (!make_tmap_bf16(&tq, q, BH, N, d, fwd::BM) || !make_tmap_bf16(&tk, k, BH, N, d, fwd::BN) ||
      !make_tmap_bf16(&tv, v, BH, N, d, fwd::BN) || !make_tmap_bf16(&to, o, BH, N, d, fwd::BM))
    return cudaErrorInvalidValue;
  if (d == 64)
    return causal ? fwd::launch_t<64, true>(tq, tk, tv, to, lse, BH, N, scale, stream)
                  : fwd::launch_t<64, false>(tq, tk, tv, to, lse, BH, N, scale, stream);
  return causal ? fwd::launch_t<128, true>(tq, tk, tv, to, lse, BH, N, scale, stream)
                : fwd::launch_t<128, false>(tq, tk, tv, to, lse, BH, N, scale, stream);
}

cudaError_t read_and_clear_fwd_error(uint32_t* out, cudaStream_t stream) {
  cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_fwd_err, sizeof(uint32_t), 0,
                                            cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return e;
  e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return e;
  const uint32_t zero = 0;
  e = cudaMemcpyToSymbolAsync(g_fwd_err, &zero, sizeof(uint32_t), 0, cudaMemcpyHostToDevice,
                              stream);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(stream);
}

}  // namespace fa
