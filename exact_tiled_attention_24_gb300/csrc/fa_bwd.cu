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
//   main        one CTA per (head, 128-key tile): K_j and V_j stay in shared
//               memory while the CTA sweeps 64-row query tiles (from the
//               diagonal on when causal). Per tile: Sᵀ = K Qᵢᵀ and
//               dPᵀ = V dOᵢᵀ land in TMEM; the compute warps turn them into
//               Pᵀ and dSᵀ (bf16, written back into TMEM, dSᵀ also into shared
//               memory); dV += Pᵀ dOᵢ and dK += dSᵀ Qᵢ accumulate in TMEM over
//               the whole sweep; dQᵢᵀ = Kᵀ dSᵢᵀ lands in TMEM with the head
//               dimension on the lanes; the dQ warps restage it as [query][d]
//               rows in shared memory and add it to the fp32 accumulator with
//               bulk reductions.
//   dq_convert  dq = bf16(scale · dQ accumulator)
//
// Roles in the main kernel (448 threads): warp 0 TMA, warp 1 TMEM owner and
// MMA issuer, warps 2..9 compute (two warps per TMEM lane quarter, each
// owning half of the 64 query columns; thread = key row), warps 10..13 read
// dQᵀ out of TMEM. TMEM columns: dV 0.., dK 128.., two S buffers 256 and
// 320 (Sᵀ_{i+1} is ready while tile i's gradient products run), dP 384,
// dQᵀ 448. Products that reuse TMEM columns read by an earlier product are
// issued after it on the same thread, and tcgen05 MMAs execute in issue
// order.
#include <cuda_bf16.h>

#include "fa_common.h"
#include "fa_ptx.cuh"
#include "fa_tmap.h"

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

constexpr int BK = 128;  // keys per CTA (M of the S, dP, dV, dK products)
constexpr int BQ = 64;   // query rows per tile (N of S and dP, K of dV and dK)
constexpr int QST = 3;   // Q / dO stages: tiles i, i+1 in use while i+2 lands
constexpr int THREADS = 448;  // 14 warps
// TMEM columns (fp32 words): accumulators for dV and dK, two S buffers, dP
// and the dQᵀ tile.
constexpr uint32_t COL_DV = 0, COL_DK = 128, COL_S = 256, COL_DP = 384, COL_DQ = 448;
constexpr int HEAD_GROUP = 4;  // heads whose key tiles are scheduled together

template <int D>
struct Smem {
  static constexpr int PANELS = D / 64;
  static constexpr int KV_TILE = BK * D * 2;       // one K or V tile
  static constexpr int Q_TILE = BQ * D * 2;        // one Q or dO tile
  static constexpr int KV_PANEL = BK * 128;        // 64 columns of a K/V tile
  static constexpr int Q_PANEL = BQ * 128;         // 64 columns of a Q/dO tile
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = K_OFF + KV_TILE;
  static constexpr int Q_OFF = V_OFF + KV_TILE;
  static constexpr int DO_OFF = Q_OFF + QST * Q_TILE;
  static constexpr int DS_OFF = DO_OFF + QST * Q_TILE;
  static constexpr int DS_TILE = BK * BQ * 2;      // dSᵀ tile: 128 key rows x 64 queries
  static constexpr int STAT_OFF = DS_OFF + 2 * DS_TILE;
  static constexpr int STAT_BYTES = 8 * 64 * 4;    // per compute warp: 32 lse + 32 D
  static constexpr int DQ_STAGE_OFF = STAT_OFF + STAT_BYTES;
  static constexpr int DQ_STAGE_BYTES = 32 * D * 4;  // 32 query rows of fp32 dQ
  static constexpr int BAR_OFF = DQ_STAGE_OFF + DQ_STAGE_BYTES;
  // kv_full, q_full[QST], q_empty[QST], s_full[2], dp_full, ds_ready,
  // dq_full, dq_free, dq_done[2], final
  static constexpr int NBARS = 1 + 2 * QST + 2 + 1 + 1 + 1 + 1 + 2 + 1;
  static constexpr int TMEM_SLOT_OFF = BAR_OFF + NBARS * 8;
  static constexpr int BYTES = TMEM_SLOT_OFF + 16;
  static constexpr int ALLOC = (BYTES + 1024) > 118784 ? (BYTES + 1024) : 118784;
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
  float* sStat = reinterpret_cast<float*>(smem + L::STAT_OFF);
  float* sDqStage = reinterpret_cast<float*>(smem + L::DQ_STAGE_OFF);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint64_t* kv_full = bars;
  uint64_t* q_full = bars + 1;
  uint64_t* q_empty = q_full + QST;
  uint64_t* s_full = q_empty + QST;
  uint64_t* dp_full = s_full + 2;
  uint64_t* ds_ready = dp_full + 1;
  uint64_t* dq_full = ds_ready + 1;
  uint64_t* dq_free = dq_full + 1;
  uint64_t* dq_done = dq_free + 1;
  uint64_t* final_bar = dq_done + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::TMEM_SLOT_OFF);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_qt = (N + BQ - 1) / BQ;
  const int n_kt = (N + BK - 1) / BK;
  int kt, bh;  // causal: heaviest key tile (kt = 0) first within each head group
  grouped_tile_order(static_cast<int>(blockIdx.x), BH, n_kt, HEAD_GROUP, &kt, &bh);
  const int k0 = kt * BK;
  const int qt_begin = CAUSAL ? (k0 / BQ) : 0;  // first query tile with a visible pair
  const int n_it = n_qt - qt_begin;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < QST; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);
    }
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    mbar_init(dp_full, 1);
    mbar_init(ds_ready, 8);
    mbar_init(dq_full, 1);
    mbar_init(dq_free, 4);
    mbar_init(&dq_done[0], 1);
    mbar_init(&dq_done[1], 1);
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
      mbar_arrive_expect_tx(kv_full, 2 * L::KV_TILE);
      for (int p = 0; p < L::PANELS; ++p) {
        tma_load_3d(sK + p * L::KV_PANEL, &tk, kv_full, p * 64, k0, bh);
        tma_load_3d(sV + p * L::KV_PANEL, &tv, kv_full, p * 64, k0, bh);
      }
      int issued = 0;
      for (int it = 0; it < n_it; ++it) {
        const int s = it % QST;
        if (!mbar_wait(&q_empty[s], ((it / QST) & 1) ^ 1, err)) break;
        const int q0 = (qt_begin + it) * BQ;
        mbar_arrive_expect_tx(&q_full[s], 2 * L::Q_TILE);
        for (int p = 0; p < L::PANELS; ++p) {
          tma_load_3d(sQ + s * L::Q_TILE + p * L::Q_PANEL, &tq, &q_full[s], p * 64, q0, bh);
          tma_load_3d(sdO + s * L::Q_TILE + p * L::Q_PANEL, &tdo, &q_full[s], p * 64, q0, bh);
        }
        issued = it + 1;
      }
      mbar_wait(kv_full, 0, err);
      for (int it = max(0, issued - QST); it < issued; ++it)
        mbar_wait(&q_full[it % QST], (it / QST) & 1, err);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16(BK, BQ, false, false);  // Sᵀ, dPᵀ: K-major both
      constexpr uint32_t id_g = idesc_bf16(BK, D, false, true);    // dV, dK: A in TMEM, B MN-major
      constexpr uint32_t id_q = idesc_bf16(128, BQ, true, true);   // dQᵀ = Kᵀ dSᵀ: both MN-major
      const uint32_t k_base = smem_u32(sK);
      const uint32_t v_base = smem_u32(sV);
      // Sᵀ_i = K Q_iᵀ  (or dPᵀ_i = V dO_iᵀ): 128 keys x 64 queries, K = D.
      auto issue_kq = [&](uint32_t a_base, uint32_t b_base, uint32_t d_col) {
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          mma_ss(tmem + d_col, sdesc_kmajor(a_base + (ks / 4) * L::KV_PANEL, (ks % 4) * 16),
                 sdesc_kmajor(b_base + (ks / 4) * L::Q_PANEL, (ks % 4) * 16), id_s, ks > 0);
        }
      };
      bool ok = mbar_wait(kv_full, 0, err) && mbar_wait(&q_full[0], 0, err);
      if (ok) {
        tc_fence_after();
        issue_kq(k_base, smem_u32(sQ), COL_S);
        tc_commit(&s_full[0]);
        issue_kq(v_base, smem_u32(sdO), COL_DP);
        tc_commit(dp_full);
        if (n_it > 1) {
          ok = mbar_wait(&q_full[1], 0, err);
          if (ok) {
            tc_fence_after();
            issue_kq(k_base, smem_u32(sQ + L::Q_TILE), COL_S + BQ);
            tc_commit(&s_full[1]);
          }
        }
      }
      for (int i = 0; i < n_it && ok; ++i) {
        const int st = i % QST;
        const int b = i & 1;
        const uint32_t q_base = smem_u32(sQ + st * L::Q_TILE);
        const uint32_t do_base = smem_u32(sdO + st * L::Q_TILE);
        ok = mbar_wait(ds_ready, i & 1, err);
        if (!ok) break;
        tc_fence_after();
        // dV += Pᵀ dO_i and dK += dSᵀ Q_i. Pᵀ / dSᵀ are bf16 in TMEM: the two
        // 32-query halves sit at column offsets 0 and 32 of their buffers.
#pragma unroll
        for (int ks = 0; ks < BQ / 16; ++ks) {
          const uint32_t acol = (ks / 2) * 32 + (ks % 2) * 8;
          mma_ts(tmem + COL_DV, tmem + COL_S + b * BQ + acol,
                 sdesc_mnmajor(do_base, ks * 16, L::Q_PANEL), id_g, (i > 0 || ks > 0) ? 1u : 0u);
        }
#pragma unroll
        for (int ks = 0; ks < BQ / 16; ++ks) {
          const uint32_t acol = (ks / 2) * 32 + (ks % 2) * 8;
          mma_ts(tmem + COL_DK, tmem + COL_DP + acol, sdesc_mnmajor(q_base, ks * 16, L::Q_PANEL),
                 id_g, (i > 0 || ks > 0) ? 1u : 0u);
        }
        // dQᵀ_i = Kᵀ dSᵀ_i (head dim on TMEM lanes; with D = 64 lanes 64..127
        // hold unused products of the neighbouring V tile).
        if (i > 0) {
          ok = mbar_wait(dq_free, (i - 1) & 1, err);
          if (!ok) break;
          tc_fence_after();
        }
        const uint32_t ds_base = smem_u32(sdS + b * L::DS_TILE);
#pragma unroll
        for (int ks = 0; ks < BK / 16; ++ks) {
          mma_ss(tmem + COL_DQ, sdesc_mnmajor(k_base, ks * 16, L::KV_PANEL),
                 sdesc_mnmajor(ds_base, ks * 16, L::KV_PANEL), id_q, ks > 0);
        }
        tc_commit(dq_full);
        tc_commit(&dq_done[b]);
        tc_commit(&q_empty[st]);
        // Next tiles: dPᵀ_{i+1} reuses the dP columns after the dK product
        // that read dSᵀ_i; Sᵀ_{i+2} reuses buffer b after the dV product that
        // read Pᵀ_i (both issued above, executed in issue order).
        if (i + 1 < n_it) {
          issue_kq(v_base, smem_u32(sdO + ((i + 1) % QST) * L::Q_TILE), COL_DP);
          tc_commit(dp_full);
        }
        if (i + 2 < n_it) {
          const int s2 = (i + 2) % QST;
          ok = mbar_wait(&q_full[s2], ((i + 2) / QST) & 1, err);
          if (!ok) break;
          tc_fence_after();
          issue_kq(k_base, smem_u32(sQ + s2 * L::Q_TILE), COL_S + b * BQ);
          tc_commit(&s_full[b]);
        }
      }
      tc_commit(final_bar);
      mbar_wait(final_bar, 0, err);
    }
  } else if (warp < 10) {
    // ------------------------------------------------------------ compute
    // Warps 2..9: two warps per TMEM lane quarter, each owning 32 of the 64
    // query columns of a tile. Thread = key row r (TMEM lane).
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const int r = quarter * 32 + lane;
    const int key = k0 + r;
    const bool key_ok = key < N;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const float* lse_h = lse + static_cast<size_t>(bh) * N;
    const float* D_h = Dvec + static_cast<size_t>(bh) * N;
    float* my_lse = sStat + (warp - 2) * 64;
    float* my_D = my_lse + 32;
    constexpr float LOG2E = 1.4426950408889634f;
    bool ok = true;
    // lse and D of the next tile are loaded one tile ahead (registers), so
    // their global-memory latency is off the per-tile critical path.
    float lse_nx = INFINITY, D_nx = 0.f;
    {
      const int q = qt_begin * BQ + half * 32 + lane;
      if (q < N) {
        lse_nx = lse_h[q] * LOG2E;
        D_nx = D_h[q];
      }
    }
    for (int i = 0; i < n_it; ++i) {
      const int qt = qt_begin + i;
      const int q0 = qt * BQ + half * 32;  // first query of this warp's half
      const int b = i & 1;
      __syncwarp();
      my_lse[lane] = lse_nx;
      my_D[lane] = D_nx;
      __syncwarp();
      {
        const int q = q0 + BQ + lane;
        lse_nx = INFINITY;
        D_nx = 0.f;
        if (i + 1 < n_it && q < N) {
          lse_nx = lse_h[q] * LOG2E;
          D_nx = D_h[q];
        }
      }
      ok = mbar_wait(&s_full[b], (i >> 1) & 1, err);
      if (!ok) break;
      tc_fence_after();
      const uint32_t s_addr = tmem + lane_addr + COL_S + b * BQ + half * 32;
      const uint32_t dp_addr = tmem + lane_addr + COL_DP + half * 32;
      uint32_t raw[32];
      tmem_ld32(s_addr, raw);
      tmem_ld_wait();
      float p[32];
      const bool need_mask = !key_ok || (CAUSAL && q0 < k0 + BK);
#pragma unroll
      for (int c = 0; c < 32; c += 4) {
        const float4 l4 = *reinterpret_cast<const float4*>(my_lse + c);
        p[c + 0] = ex2(fmaf(__uint_as_float(raw[c + 0]), scale_log2, -l4.x));
        p[c + 1] = ex2(fmaf(__uint_as_float(raw[c + 1]), scale_log2, -l4.y));
        p[c + 2] = ex2(fmaf(__uint_as_float(raw[c + 2]), scale_log2, -l4.z));
        p[c + 3] = ex2(fmaf(__uint_as_float(raw[c + 3]), scale_log2, -l4.w));
      }
      if (need_mask) {
#pragma unroll
        for (int c = 0; c < 32; ++c)
          if (!key_ok || (CAUSAL && q0 + c < key)) p[c] = 0.f;
      }
      uint32_t pk[16];
#pragma unroll
      for (int t = 0; t < 16; ++t) pk[t] = pack_bf16x2(p[2 * t], p[2 * t + 1]);
      tmem_st16(s_addr, pk);
      // dSᵀ = Pᵀ ∘ (dPᵀ − D)
      ok = mbar_wait(dp_full, i & 1, err);
      if (!ok) break;
      tc_fence_after();
      tmem_ld32(dp_addr, raw);
      tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < 32; c += 4) {
        const float4 d4 = *reinterpret_cast<const float4*>(my_D + c);
        const float a0 = p[c + 0] * (__uint_as_float(raw[c + 0]) - d4.x);
        const float a1 = p[c + 1] * (__uint_as_float(raw[c + 1]) - d4.y);
        const float a2 = p[c + 2] * (__uint_as_float(raw[c + 2]) - d4.z);
        const float a3 = p[c + 3] * (__uint_as_float(raw[c + 3]) - d4.w);
        pk[c / 2] = pack_bf16x2(a0, a1);
        pk[c / 2 + 1] = pack_bf16x2(a2, a3);
      }
      tmem_st16(dp_addr, pk);
      // dSᵀ into shared memory for the dQ product: row = key, 64 queries of
      // 2 bytes = one 128-byte swizzled row; this half is chunks 4h..4h+3.
      if (i >= 2) {
        ok = mbar_wait(&dq_done[b], ((i - 2) >> 1) & 1, err);
        if (!ok) break;
      }
      uint8_t* ds_row = sdS + b * L::DS_TILE + r * 128;
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        const int chunk = half * 4 + ch;
        *reinterpret_cast<uint4*>(ds_row + ((chunk ^ (r & 7)) * 16)) =
            make_uint4(pk[ch * 4], pk[ch * 4 + 1], pk[ch * 4 + 2], pk[ch * 4 + 3]);
      }
      tmem_st_wait();
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ds_ready);
    }
    // -------------------------------------------------------------- epilogue
    // The last dQ product's completion implies every MMA of this CTA is done;
    // the Q and dO stage buffers then stage dK and dV for the TMA stores.
    if (ok) ok = mbar_wait(&dq_done[(n_it - 1) & 1], ((n_it - 1) >> 1) & 1, err);
    if (ok) {
      tc_fence_after();
#pragma unroll
      for (int cc = 0; cc < D / 2; cc += 32) {
        const int c = half * (D / 2) + cc;
        uint32_t a[32], bb[32];
        tmem_ld32(tmem + lane_addr + COL_DK + c, a);
        tmem_ld32(tmem + lane_addr + COL_DV + c, bb);
        tmem_ld_wait();
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          const int col0 = c + ch * 8;
          const int panel = col0 / 64;
          const int chunk = (col0 % 64) / 8;
          const int off = panel * L::KV_PANEL + r * 128 + ((chunk ^ (r & 7)) * 16);
          uint4 vk, vv;
          vk.x = pack_bf16x2(__uint_as_float(a[ch * 8 + 0]) * scale, __uint_as_float(a[ch * 8 + 1]) * scale);
          vk.y = pack_bf16x2(__uint_as_float(a[ch * 8 + 2]) * scale, __uint_as_float(a[ch * 8 + 3]) * scale);
          vk.z = pack_bf16x2(__uint_as_float(a[ch * 8 + 4]) * scale, __uint_as_float(a[ch * 8 + 5]) * scale);
          vk.w = pack_bf16x2(__uint_as_float(a[ch * 8 + 6]) * scale, __uint_as_float(a[ch * 8 + 7]) * scale);
          vv.x = pack_bf16x2(__uint_as_float(bb[ch * 8 + 0]), __uint_as_float(bb[ch * 8 + 1]));
          vv.y = pack_bf16x2(__uint_as_float(bb[ch * 8 + 2]), __uint_as_float(bb[ch * 8 + 3]));
          vv.z = pack_bf16x2(__uint_as_float(bb[ch * 8 + 4]), __uint_as_float(bb[ch * 8 + 5]));
          vv.w = pack_bf16x2(__uint_as_float(bb[ch * 8 + 6]), __uint_as_float(bb[ch * 8 + 7]));
          *reinterpret_cast<uint4*>(sQ + off) = vk;
          *reinterpret_cast<uint4*>(sdO + off) = vv;
        }
      }
      fence_async_smem();
    }
    named_bar_sync(1, 256);
    if (ok && warp == 2 && lane == 0) {
      for (int p = 0; p < L::PANELS; ++p) {
        tma_store_3d(&tdk, sQ + p * L::KV_PANEL, p * 64, k0, bh);
        tma_store_3d(&tdv, sdO + p * L::KV_PANEL, p * 64, k0, bh);
      }
      tma_store_commit();
      tma_store_wait_all();
    }
  } else {
    // ------------------------------------------------------------ dQ warps
    // Warps 10..13: read dQᵀ_i out of TMEM (lane = head-dim index, column =
    // query), release the TMEM columns, then stage 32 query rows at a time in
    // shared memory in the accumulator's [query][d] layout and add them to
    // the fp32 accumulator with one bulk reduction (rows q0.. are contiguous).
    const int quarter = warp & 3;
    const int dd = quarter * 32 + lane;
    const uint32_t dq_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + COL_DQ;
    float* acc_h = dq_acc + static_cast<size_t>(bh) * N * D;
    const bool active = (D == 128) || (quarter < 2);
    const bool issuer = (warp == 10 && lane == 0);
    for (int i = 0; i < n_it; ++i) {
      const bool got = mbar_wait(dq_full, i & 1, err);
      if (named_bar_any(2, 128, !got)) break;  // all four warps leave together
      tc_fence_after();
      uint32_t v[2][32];
      tmem_ld32(dq_addr, v[0]);
      tmem_ld32(dq_addr + 32, v[1]);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(dq_free);
      const int q0 = (qt_begin + i) * BQ;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int rows = min(32, N - (q0 + 32 * h));
        // the previous bulk reduction must have finished reading the stage
        if (issuer) bulk_wait_read_all();
        named_bar_sync(2, 128);
        if (rows > 0) {
          if (active) {
#pragma unroll
            for (int c = 0; c < 32; ++c) sDqStage[c * D + dd] = __uint_as_float(v[h][c]);
          }
          fence_async_smem();
        }
        named_bar_sync(2, 128);
        if (issuer && rows > 0) {
          bulk_reduce_add_f32(acc_h + static_cast<size_t>(q0 + 32 * h) * D, sDqStage,
                              static_cast<uint32_t>(rows) * D * 4u);
          tma_store_commit();
        }
      }
    }
    if (issuer) tma_store_wait_all();
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

cudaError_t launch_bwd_main(const void* q, const void* k, const void* v, const void* dO,
                            void* dk, void* dv, const float* lse, const float* Dvec,
                            float* dq_acc, int BH, int N, int d, float scale, bool causal,
                            cudaStream_t stream) {
  CUtensorMap tq, tk, tv, tdo, tdk, tdv;
  if (!make_tmap_bf16(&tq, q, BH, N, d, bwd::BQ) || !make_tmap_bf16(&tdo, dO, BH, N, d, bwd::BQ) ||
      !make_tmap_bf16(&tk, k, BH, N, d, bwd::BK) || !make_tmap_bf16(&tv, v, BH, N, d, bwd::BK) ||
      !make_tmap_bf16(&tdk, dk, BH, N, d, bwd::BK) || !make_tmap_bf16(&tdv, dv, BH, N, d, bwd::BK))
    return cudaErrorInvalidValue;
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
