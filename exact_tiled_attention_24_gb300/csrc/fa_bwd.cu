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
//   preprocess  D = rowsum(dO ∘ O).
//   dkdv        one CTA per (head, 128-key tile): K_j and V_j stay in shared
//               memory while the CTA sweeps 128-row query tiles (from the
//               diagonal on when causal). Per tile, Sᵀ = K Qᵢᵀ and
//               dPᵀ = V dOᵢᵀ land in TMEM; the compute warps turn them into
//               Pᵀ and dSᵀ (bf16, written back into TMEM) and
//               dV += Pᵀ dOᵢ, dK += dSᵀ Qᵢ accumulate in TMEM over the sweep.
//   dq          one CTA per (head, 128-row query tile): Q_i and dO_i are
//               copied into TMEM once and serve as the A operand while the
//               CTA sweeps 128-key tiles; S = Qᵢ Kⱼᵀ and dP = dOᵢ Vⱼᵀ are
//               recomputed, dS (bf16, TMEM) feeds dQ += dS Kⱼ, and dQ is
//               written once, in bf16, at the end.
// Computing dQ in its own sweep recomputes S and dP (seven products per
// query/key tile pair instead of five) but needs no cross-CTA reduction: on
// this part the fp32 reduction traffic of a dQ accumulated from every key
// tile (4 bytes x N x d per key tile) is bounded by L2 reduction throughput
// well below what the tensor cores need.
//
// Both sweep kernels use 128-wide tiles so that every product has N = 128
// (an MMA with N = 64 takes nearly as long as one with N = 128 on this part).
// Products that overwrite TMEM columns another product reads are issued
// after it on the same thread; tcgen05 MMAs execute in issue order.
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
                                                         long long rows) {
  constexpr int TPR = D / 8;  // threads per row, 8 bf16 (16 bytes) each
  constexpr int RPB = 256 / TPR;
  const long long row = static_cast<long long>(blockIdx.x) * RPB + threadIdx.x / TPR;
  const int part = threadIdx.x % TPR;
  float acc = 0.f;
  if (row < rows && in_range(static_cast<long long>(row) * D + part * 8, 8, rows * D, &g_bwd_err)) {
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
  }
#pragma unroll
  for (int w = TPR / 2; w > 0; w >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, w);
  if (row < rows && part == 0 && in_range(row, 1, rows, &g_bwd_err)) Dvec[row] = acc;
}

// ------------------------------------------------------- shared helpers

constexpr int TILE = 128;       // rows of every K, V, Q, dO tile
constexpr int MAX_HEAD_GROUP = 4;   // most heads whose tiles are scheduled together
constexpr int SWEEP_THREADS = 320;  // 10 warps: TMA, MMA, 8 compute

template <int D>
struct Tiles {
  static constexpr int PANELS = D / 64;
  static constexpr int BYTES = TILE * D * 2;  // one 128-row tile
  static constexpr int PANEL = TILE * 128;    // 64 columns x 128 rows
};

// Stage columns [c_begin, c_begin + NCOLS) of a [128 rows] fp32 tile held in
// TMEM (lane = row) as bf16, times `mul`, into a swizzled shared-memory tile
// (panels of 64 columns, dst_bytes in all) ready for a TMA store.
template <int NCOLS>
__device__ __forceinline__ void stage_tmem_rows_bf16(uint32_t taddr, uint8_t* dst, int r, int c_begin,
                                                     float mul, int dst_bytes, uint32_t* err) {
#pragma unroll
  for (int cc = 0; cc < NCOLS; cc += 32) {
    const int c = c_begin + cc;
    uint32_t a[32];
    tmem_ld32(taddr + c, a);
    tmem_ld_wait();
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) {
      const int col0 = c + ch * 8;
      const int panel = col0 / 64;
      const int chunk = (col0 % 64) / 8;
      uint4 v;
      v.x = pack_bf16x2(__uint_as_float(a[ch * 8 + 0]) * mul, __uint_as_float(a[ch * 8 + 1]) * mul);
      v.y = pack_bf16x2(__uint_as_float(a[ch * 8 + 2]) * mul, __uint_as_float(a[ch * 8 + 3]) * mul);
      v.z = pack_bf16x2(__uint_as_float(a[ch * 8 + 4]) * mul, __uint_as_float(a[ch * 8 + 5]) * mul);
      v.w = pack_bf16x2(__uint_as_float(a[ch * 8 + 6]) * mul, __uint_as_float(a[ch * 8 + 7]) * mul);
      const int off = panel * (TILE * 128) + r * 128 + ((chunk ^ (r & 7)) * 16);
      if (in_range(off, 16, dst_bytes, err)) *reinterpret_cast<uint4*>(dst + off) = v;
    }
  }
}

// Aligned shared-memory base; returns nullptr (and records an error) when
// the 1024-byte aligned layout does not fit the allocation.
__device__ __forceinline__ uint8_t* aligned_smem(uint8_t* raw, int bytes, int alloc) {
  const uint32_t pad = (1024u - (smem_u32(raw) & 1023u)) & 1023u;
  if (pad + static_cast<uint32_t>(bytes) > static_cast<uint32_t>(alloc)) {
    if (threadIdx.x == 0) atomicExch(&g_bwd_err, DEV_TIMEOUT);
    return nullptr;
  }
  return raw + pad;
}

constexpr int kMaxDynSmem = 232448;  // 227 KB per-block opt-in limit

// Dynamic allocation: the layout plus alignment slack, at least 116 KB so
// only one CTA (and one 512-column TMEM allocation) is resident per SM.
constexpr int alloc_for(int bytes) {
  return (bytes + 1024 <= kMaxDynSmem) ? (bytes + 1024 < 118784 ? 118784 : bytes + 1024) : kMaxDynSmem;
}

// ------------------------------------------------------------ dK, dV sweep

constexpr uint32_t KV_COL_DV = 0, KV_COL_DK = 128, KV_COL_S = 256, KV_COL_DP = 384;

template <int D>
struct DkdvSmem {
  using T = Tiles<D>;
  // Q tiles are read last by dK += dSᵀ Q, the product issued latest in a
  // tile's round, and first by the next-but-one Sᵀ: three Q stages keep the
  // load a full round ahead. dO is free one product after dV reads it.
  static constexpr int QST = 3;
  static constexpr int OST = 2;
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = K_OFF + T::BYTES;
  static constexpr int Q_OFF = V_OFF + T::BYTES;
  static constexpr int DO_OFF = Q_OFF + QST * T::BYTES;
  static constexpr int STAT_OFF = DO_OFF + OST * T::BYTES;
  static constexpr int STAT_BYTES = 2 * 2 * TILE * 4;  // two buffers of (lse, D) per query
  static constexpr int BAR_OFF = STAT_OFF + STAT_BYTES;
  // kv_full, in_full[QST] (Q_i and dO_i of tile i landed), q_empty[QST],
  // o_empty[OST], s_full, p_ready, dp_full, ds_ready, final
  static constexpr int NBARS = 1 + 2 * QST + OST + 5;
  static constexpr int TMEM_SLOT_OFF = BAR_OFF + NBARS * 8;
  static constexpr int BYTES = TMEM_SLOT_OFF + 16;
  static constexpr int ALLOC = alloc_for(BYTES);
  static_assert(BYTES <= kMaxDynSmem, "shared memory layout exceeds the per-block limit");
};

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(SWEEP_THREADS, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                    const __grid_constant__ CUtensorMap tdk,
                    const __grid_constant__ CUtensorMap tdv, const float* __restrict__ lse,
                    const float* __restrict__ Dvec, int BHkv, int G, int N, int head_group, float scale,
                    float scale_log2) {
  using L = DkdvSmem<D>;
  using T = Tiles<D>;
  constexpr int QST = L::QST;
  constexpr int OST = L::OST;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = aligned_smem(smem_raw, L::BYTES, L::ALLOC);
  if (smem == nullptr) return;
  uint8_t* sK = smem + L::K_OFF;
  uint8_t* sV = smem + L::V_OFF;
  uint8_t* sQ = smem + L::Q_OFF;
  uint8_t* sdO = smem + L::DO_OFF;
  float* sStat = reinterpret_cast<float*>(smem + L::STAT_OFF);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint64_t* kv_full = bars;
  uint64_t* in_full = bars + 1;
  uint64_t* q_empty = in_full + QST;
  uint64_t* o_empty = q_empty + QST;
  uint64_t* s_full = o_empty + OST;
  uint64_t* p_ready = s_full + 1;
  uint64_t* dp_full = p_ready + 1;
  uint64_t* ds_ready = dp_full + 1;
  uint64_t* final_bar = ds_ready + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::TMEM_SLOT_OFF);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_t = (N + TILE - 1) / TILE;
  int kt, bkv;  // causal: heaviest key tile (kt = 0) first within each head group
  grouped_tile_order(static_cast<int>(blockIdx.x), BHkv, n_t, head_group, &kt, &bkv);
  const int k0 = kt * TILE;
  const int qt_begin = CAUSAL ? kt : 0;  // first query tile with a visible pair
  const int n_q = n_t - qt_begin;        // query tiles swept per query head
  // Sweep tile it = (query head bkv·G + it / n_q, query tile qt_begin + it % n_q):
  // dK and dV of a shared K/V head sum over every query head of its group.
  const int n_it = G * n_q;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < QST; ++s) {
      mbar_init(&in_full[s], 1);
      mbar_init(&q_empty[s], 1);
    }
    for (int s = 0; s < OST; ++s) mbar_init(&o_empty[s], 1);
    mbar_init(s_full, 1);
    mbar_init(p_ready, 8);
    mbar_init(dp_full, 1);
    mbar_init(ds_ready, 8);
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
      mbar_arrive_expect_tx(kv_full, 2 * T::BYTES);
      for (int p = 0; p < T::PANELS; ++p) {
        tma_load_3d(sK + p * T::PANEL, &tk, kv_full, p * 64, k0, bkv);
        tma_load_3d(sV + p * T::PANEL, &tv, kv_full, p * 64, k0, bkv);
      }
      // Q_i and dO_i complete on one barrier, so the issuer waits once per
      // tile for its inputs.
      int issued = 0;
      int gq = 0, qi = 0;  // query head within the group, query tile index
      for (int it = 0; it < n_it; ++it) {
        const int q0 = (qt_begin + qi) * TILE;
        const int bh = bkv * G + gq;
        if (++qi == n_q) {
          qi = 0;
          ++gq;
        }
        const int sq = it % QST, so = it % OST;
        if (!mbar_wait(&q_empty[sq], ((it / QST) & 1) ^ 1, err)) break;
        if (!mbar_wait(&o_empty[so], ((it / OST) & 1) ^ 1, err)) break;
        mbar_arrive_expect_tx(&in_full[sq], 2 * T::BYTES);
        for (int p = 0; p < T::PANELS; ++p) {
          tma_load_3d(sQ + sq * T::BYTES + p * T::PANEL, &tq, &in_full[sq], p * 64, q0, bh);
          tma_load_3d(sdO + so * T::BYTES + p * T::PANEL, &tdo, &in_full[sq], p * 64, q0, bh);
        }
        issued = it + 1;
      }
      // No copy may still be in flight when the CTA exits.
      mbar_wait(kv_full, 0, err);
      for (int it = max(0, issued - QST); it < issued; ++it)
        mbar_wait(&in_full[it % QST], (it / QST) & 1, err);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    // Whole warp runs the loop (warp-uniform descriptors); one elected lane
    // issues MMAs and commits.
    constexpr uint32_t id_s = idesc_bf16(TILE, TILE, false, false);  // Sᵀ, dPᵀ: K-major both
    constexpr uint32_t id_g = idesc_bf16(TILE, D, false, true);      // dV, dK: A TMEM, B MN-major
    static_assert(QST == 3 && OST == 2, "descriptor selection assumes three Q and two dO stages");
    const uint64_t dK = sdesc_kmajor(smem_u32(sK), 0), dV = sdesc_kmajor(smem_u32(sV), 0);
    const uint64_t dQk0 = sdesc_kmajor(smem_u32(sQ), 0), dQk1 = sdesc_kmajor(smem_u32(sQ + T::BYTES), 0),
                   dQk2 = sdesc_kmajor(smem_u32(sQ + 2 * T::BYTES), 0);
    const uint64_t dOk0 = sdesc_kmajor(smem_u32(sdO), 0), dOk1 = sdesc_kmajor(smem_u32(sdO + T::BYTES), 0);
    const uint64_t dQm0 = sdesc_mnmajor(smem_u32(sQ), 0, T::PANEL);
    const uint64_t dQm1 = sdesc_mnmajor(smem_u32(sQ + T::BYTES), 0, T::PANEL);
    const uint64_t dQm2 = sdesc_mnmajor(smem_u32(sQ + 2 * T::BYTES), 0, T::PANEL);
    const uint64_t dOm0 = sdesc_mnmajor(smem_u32(sdO), 0, T::PANEL);
    const uint64_t dOm1 = sdesc_mnmajor(smem_u32(sdO + T::BYTES), 0, T::PANEL);
    auto sel3 = [](int st, uint64_t a, uint64_t b, uint64_t c) { return st == 0 ? a : (st == 1 ? b : c); };
    // Sᵀ = K Qᵀ (or dPᵀ = V dOᵀ): 128 keys x 128 queries, K = D; then commit.
    auto issue_kq = [&](uint64_t a, uint64_t b, uint32_t d_col, uint64_t* bar) {
      if (elect_one()) {
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          mma_ss(tmem + d_col, desc_add(a, kmajor_step(ks, T::PANEL)), desc_add(b, kmajor_step(ks, T::PANEL)),
                 id_s, ks > 0);
        tc_commit(bar);
      }
      __syncwarp();
    };
    // D_col += A(TMEM, 64-query halves at column offsets 0 and 64) · B (MN-major).
    auto issue_grad = [&](uint32_t d_col, uint32_t a_col, uint64_t b, uint32_t acc0, uint64_t* bar) {
      if (elect_one()) {
#pragma unroll
        for (int ks = 0; ks < TILE / 16; ++ks)
          mma_ts(tmem + d_col, tmem + a_col + (ks / 4) * 64 + (ks % 4) * 8, desc_add(b, mnmajor_step(ks)),
                 id_g, ks > 0 ? 1u : acc0);
        if (bar != nullptr) tc_commit(bar);
      }
      __syncwarp();
    };
    bool ok = mbar_wait_warp(kv_full, 0, err) && mbar_wait_warp(&in_full[0], 0, err);
    if (ok) {
      tc_fence_after();
      issue_kq(dK, dQk0, KV_COL_S, s_full);
      issue_kq(dV, dOk0, KV_COL_DP, dp_full);
    }
    // Round i: dV_i, Sᵀ_{i+1}, dK_i, dPᵀ_{i+1}. dV_i needs only Pᵀ_i, so it
    // and Sᵀ_{i+1} keep the tensor pipe busy while the compute warps turn
    // dPᵀ_i into dSᵀ_i. The wait for tile i+1's inputs comes first: it is
    // normally met already and overlaps the wait for Pᵀ_i.
    for (int i = 0; i < n_it && ok; ++i) {
      const int sq = i % QST, so = i % OST;
      const int sq1 = (i + 1) % QST, so1 = (i + 1) % OST;
      const uint32_t acc0 = i > 0 ? 1u : 0u;
      const bool more = i + 1 < n_it;
      if (more) {
        ok = mbar_wait_warp(&in_full[sq1], ((i + 1) / QST) & 1, err);
        if (!ok) break;
      }
      ok = mbar_wait_warp(p_ready, i & 1, err);
      if (!ok) break;
      tc_fence_after();
      // dV += Pᵀ dO_i (Pᵀ in the S columns); dO_i then has no further reader.
      issue_grad(KV_COL_DV, KV_COL_S, so ? dOm1 : dOm0, acc0, &o_empty[so]);
      // Sᵀ_{i+1} overwrites the S columns after the dV product read Pᵀ_i.
      if (more) issue_kq(dK, sel3(sq1, dQk0, dQk1, dQk2), KV_COL_S, s_full);
      ok = mbar_wait_warp(ds_ready, i & 1, err);
      if (!ok) break;
      tc_fence_after();
      // dK += dSᵀ Q_i (dSᵀ in the dP columns); Q_i then has no further reader.
      issue_grad(KV_COL_DK, KV_COL_DP, sel3(sq, dQm0, dQm1, dQm2), acc0, &q_empty[sq]);
      // dPᵀ_{i+1} overwrites the dP columns after the dK product read dSᵀ_i.
      if (more) issue_kq(dV, so1 ? dOk1 : dOk0, KV_COL_DP, dp_full);
    }
    if (elect_one()) tc_commit(final_bar);
    __syncwarp();
    mbar_wait_warp(final_bar, 0, err);
  } else {
    // ------------------------------------------------------------ compute
    // Warps 2..9: two warps per TMEM lane quarter; warp half h owns query
    // columns 64h..64h+63 of each tile. Thread = key row r (TMEM lane).
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const int ct = threadIdx.x - 64;  // 0..255 over the compute warps
    const int r = quarter * 32 + lane;
    const int key = k0 + r;
    const bool key_ok = key < N;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    constexpr float LOG2E = 1.4426950408889634f;
    // Per-tile (−lse·log2 e, −D) of the 128 queries, double-buffered in shared
    // memory: compute thread ct fills entry ct % 128 of lse (ct < 128) or of
    // D. A value is loaded one tile before it is stored, and only the store
    // reads the loaded register, so no warp waits on the load.
    // Stored negated (−lse·log2 e, −D) so that the packed pair arithmetic
    // below adds them; the products are the same as subtracting.
    const float stat_mul = ct < 128 ? -LOG2E : -1.f;
    const long long n_rows = static_cast<long long>(BHkv) * G * N;  // lse and D entries
    auto load_stat = [&](int tile) -> float {
      if (tile >= n_it) return ct < 128 ? INFINITY : 0.f;
      const int gq = tile / n_q;
      const int q = (qt_begin + tile - gq * n_q) * TILE + (ct & 127);
      const size_t row = static_cast<size_t>(bkv * G + gq) * N + q;
      const bool live = q < N && in_range(static_cast<long long>(row), 1, n_rows, err);
      if (ct < 128) return live ? lse[row] : INFINITY;
      return live ? Dvec[row] : 0.f;
    };
    if (in_range(ct, 1, 512, err)) sStat[ct] = load_stat(0) * stat_mul;  // buffer 0: lse[0..127], D[128..255]
    float stat_nx = load_stat(1);
    named_bar_sync(1, 256);
    bool ok = true;
    int qi = 0;  // query tile index of sweep tile i within its query head
    for (int i = 0; i < n_it; ++i) {
      const int q0 = (qt_begin + qi) * TILE + half * 64;  // first query of this warp's half
      if (++qi == n_q) qi = 0;
      const float* s_lse = sStat + (i & 1) * 256 + half * 64;
      const float* s_D = s_lse + 128;
      ok = mbar_wait(s_full, i & 1, err);
      if (!ok) break;
      tc_fence_after();
      const uint32_t s_addr = tmem + lane_addr + KV_COL_S + half * 64;
      const uint32_t dp_addr = tmem + lane_addr + KV_COL_DP + half * 64;
      float p[64];
      const bool masked = !key_ok || (CAUSAL && q0 < k0 + TILE);
      {
        uint32_t raw[64];
        tmem_ld64(s_addr, raw);
        tmem_ld_wait();
        const float2 sc2 = make_float2(scale_log2, scale_log2);
#pragma unroll
        for (int c = 0; c < 64; c += 4) {
          const float4 l4 = *reinterpret_cast<const float4*>(s_lse + c);  // −lse·log2 e
          const float2 e01 = ffma2(make_float2(__uint_as_float(raw[c + 0]), __uint_as_float(raw[c + 1])), sc2,
                                   make_float2(l4.x, l4.y));
          const float2 e23 = ffma2(make_float2(__uint_as_float(raw[c + 2]), __uint_as_float(raw[c + 3])), sc2,
                                   make_float2(l4.z, l4.w));
          p[c + 0] = ex2(e01.x);
          p[c + 1] = ex2(e01.y);
          p[c + 2] = ex2(e23.x);
          p[c + 3] = ex2(e23.y);
        }
      }
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        if (masked) {
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (!key_ok || (CAUSAL && q0 + 32 * h2 + c < key)) p[32 * h2 + c] = 0.f;
        }
        uint32_t pk[16];
#pragma unroll
        for (int t = 0; t < 16; ++t) pk[t] = pack_bf16x2(p[32 * h2 + 2 * t], p[32 * h2 + 2 * t + 1]);
        tmem_st16(s_addr + 16 * h2, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_ready);
      // dSᵀ = Pᵀ ∘ (dPᵀ − D), bf16 into this warp's own dP columns.
      ok = mbar_wait(dp_full, i & 1, err);
      if (!ok) break;
      tc_fence_after();
      {
        uint32_t raw[64];
        tmem_ld64(dp_addr, raw);
        tmem_ld_wait();
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 32; c += 4) {
            const float4 d4 = *reinterpret_cast<const float4*>(s_D + 32 * h2 + c);  // −D
            const float* pp = p + 32 * h2 + c;
            const uint32_t* rr = raw + 32 * h2 + c;
            const float2 ds01 = fmul2(make_float2(pp[0], pp[1]),
                                      fadd2(make_float2(__uint_as_float(rr[0]), __uint_as_float(rr[1])),
                                            make_float2(d4.x, d4.y)));
            const float2 ds23 = fmul2(make_float2(pp[2], pp[3]),
                                      fadd2(make_float2(__uint_as_float(rr[2]), __uint_as_float(rr[3])),
                                            make_float2(d4.z, d4.w)));
            pk[c / 2] = pack_bf16x2(ds01.x, ds01.y);
            pk[c / 2 + 1] = pack_bf16x2(ds23.x, ds23.y);
          }
          tmem_st16(dp_addr + 16 * h2, pk);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ds_ready);
      // Next tile's (lse, D) into the other buffer; its previous readers
      // passed the barrier at the end of the previous iteration.
      if (in_range(((i + 1) & 1) * 256 + ct, 1, 512, err)) sStat[((i + 1) & 1) * 256 + ct] = stat_nx * stat_mul;
      stat_nx = load_stat(i + 2);
      named_bar_sync(1, 256);
    }
    // -------------------------------------------------------------- epilogue
    // Wait for the last products; the stage-0 Q and dO buffers then stage
    // dK (scaled) and dV for the TMA stores.
    if (ok) ok = mbar_wait(final_bar, 0, err);
    if (ok) {
      tc_fence_after();
      stage_tmem_rows_bf16<D / 2>(tmem + lane_addr + KV_COL_DK, sQ, r, half * (D / 2), scale, T::BYTES, err);
      stage_tmem_rows_bf16<D / 2>(tmem + lane_addr + KV_COL_DV, sdO, r, half * (D / 2), 1.f, T::BYTES, err);
      fence_async_smem();
    }
    named_bar_sync(1, 256);
    if (ok && warp == 2 && lane == 0) {
      for (int p = 0; p < T::PANELS; ++p) {
        tma_store_3d(&tdk, sQ + p * T::PANEL, p * 64, k0, bkv);
        tma_store_3d(&tdv, sdO + p * T::PANEL, p * 64, k0, bkv);
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

// ------------------------------------------------------------------ dQ sweep

constexpr uint32_t Q_COL_S = 0, Q_COL_DP = 128, Q_COL_DQ = 256, Q_COL_Q = 384, Q_COL_DO = 448;

template <int D, bool FUSE_D>
struct DqSmem {
  using T = Tiles<D>;
  // Three K/V stages: 0 and 1 are dedicated; stage 2 is the Q/dO region,
  // free once Q and dO have been copied into TMEM.
  static constexpr int KST = 3;
  static constexpr int Q_OFF = 0;   // Q tile, then K of stage 2, then the dQ staging tile
  static constexpr int DO_OFF = Q_OFF + T::BYTES;  // dO tile, then V of stage 2
  static constexpr int K_OFF = DO_OFF + T::BYTES;  // K of stages 0, 1
  static constexpr int V_OFF = K_OFF + 2 * T::BYTES;  // V of stages 0, 1
  // FUSE_D: the O tile, and the two halves of each row's D (fp32 [2][128]).
  static constexpr int O_OFF = V_OFF + 2 * T::BYTES;
  static constexpr int RED_OFF = O_OFF + (FUSE_D ? T::BYTES : 0);
  static constexpr int BAR_OFF = RED_OFF + (FUSE_D ? 2 * TILE * 4 : 0);
  // q_full, s_go[KST], kv_empty[KST], a_ready, s_full, dp_full, ds_ready,
  // final
  static constexpr int NBARS = 1 + 2 * KST + 5;
  static constexpr int TMEM_SLOT_OFF = BAR_OFF + NBARS * 8;
  static constexpr int BYTES = TMEM_SLOT_OFF + 16;
  static constexpr int ALLOC = alloc_for(BYTES);
  static_assert(BYTES <= kMaxDynSmem, "shared memory layout exceeds the per-block limit");
};

// FUSE_D: the sweep also forms D = rowsum(dO ∘ O) for its query tile (O
// loaded beside Q and dO through `to`) and writes it to Dvec, instead of
// reading it there; the dK/dV sweep then runs after this one.
template <int D, bool CAUSAL, bool FUSE_D>
__global__ void __launch_bounds__(SWEEP_THREADS, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                  const __grid_constant__ CUtensorMap tdq, const __grid_constant__ CUtensorMap to,
                  const float* __restrict__ lse, float* __restrict__ Dvec, int BH, int G, int N,
                  int head_group, float scale, float scale_log2) {
  using L = DqSmem<D, FUSE_D>;
  using T = Tiles<D>;
  constexpr int KST = L::KST;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = aligned_smem(smem_raw, L::BYTES, L::ALLOC);
  if (smem == nullptr) return;
  uint8_t* sQ = smem + L::Q_OFF;
  uint8_t* sdO = smem + L::DO_OFF;
  // K and V tile of stage s
  auto kst = [&](int st) { return st < 2 ? smem + L::K_OFF + st * T::BYTES : sQ; };
  auto vst = [&](int st) { return st < 2 ? smem + L::V_OFF + st * T::BYTES : sdO; };
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  // s_go[j % KST]: the two things S_j waits for, in one barrier — K_j and
  // V_j have landed (the producer's byte-counted arrival) and the compute
  // warps hold S_{j-1} in registers, so S_j may overwrite its columns
  // (their 8 arrivals; for j = 0, made once Q and dO are in TMEM).
  uint64_t* q_full = bars;
  uint64_t* s_go = bars + 1;
  uint64_t* kv_empty = s_go + KST;
  uint64_t* a_ready = kv_empty + KST;  // Q and dO copied into TMEM
  uint64_t* s_full = a_ready + 1;
  uint64_t* dp_full = s_full + 1;
  uint64_t* ds_ready = dp_full + 1;
  uint64_t* final_bar = ds_ready + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::TMEM_SLOT_OFF);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_t = (N + TILE - 1) / TILE;
  int t, bh;  // causal: heaviest query tile (the last one) first within each head group
  grouped_tile_order(static_cast<int>(blockIdx.x), BH, n_t, head_group, &t, &bh);
  const int qt = n_t - 1 - t;
  const int q0 = qt * TILE;
  const int bkv = bh / G;  // K/V head shared by G consecutive query heads
  const int n_kv = CAUSAL ? qt + 1 : n_t;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < KST; ++s) {
      mbar_init(&s_go[s], 1 + 8);
      mbar_init(&kv_empty[s], 1);
    }
    mbar_init(a_ready, 8);
    mbar_init(s_full, 1);
    mbar_init(dp_full, 1);
    mbar_init(ds_ready, 8);
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
      mbar_arrive_expect_tx(q_full, (FUSE_D ? 3 : 2) * T::BYTES);
      for (int p = 0; p < T::PANELS; ++p) {
        tma_load_3d(sQ + p * T::PANEL, &tq, q_full, p * 64, q0, bh);
        tma_load_3d(sdO + p * T::PANEL, &tdo, q_full, p * 64, q0, bh);
        if (FUSE_D) tma_load_3d(smem + L::O_OFF + p * T::PANEL, &to, q_full, p * 64, q0, bh);
      }
      int issued = 0;
      for (int j = 0; j < n_kv; ++j) {
        const int s = j % KST;
        if (!mbar_wait(&kv_empty[s], ((j / KST) & 1) ^ 1, err)) break;
        // Stage 2 overlays Q and dO: first use waits for their copy to TMEM.
        if (j == 2 && !mbar_wait(a_ready, 0, err)) break;
        mbar_arrive_expect_tx(&s_go[s], 2 * T::BYTES);
        uint8_t* kd = kst(s);
        uint8_t* vd = vst(s);
        for (int p = 0; p < T::PANELS; ++p) {
          tma_load_3d(kd + p * T::PANEL, &tk, &s_go[s], p * 64, j * TILE, bkv);
          tma_load_3d(vd + p * T::PANEL, &tv, &s_go[s], p * 64, j * TILE, bkv);
        }
        issued = j + 1;
      }
      mbar_wait(q_full, 0, err);
      for (int j = max(0, issued - KST); j < issued; ++j)
        mbar_wait(&s_go[j % KST], (j / KST) & 1, err);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    // Whole warp runs the loop (warp-uniform descriptors); one elected lane
    // issues MMAs and commits.
    constexpr uint32_t id_s = idesc_bf16(TILE, TILE, false, false);  // S, dP: A TMEM, B K-major
    constexpr uint32_t id_q = idesc_bf16(TILE, D, false, true);      // dQ: A TMEM, B MN-major
    static_assert(KST == 3, "descriptor selection assumes three stages");
    const uint64_t dKk0 = sdesc_kmajor(smem_u32(kst(0)), 0), dKk1 = sdesc_kmajor(smem_u32(kst(1)), 0),
                   dKk2 = sdesc_kmajor(smem_u32(kst(2)), 0);
    const uint64_t dVk0 = sdesc_kmajor(smem_u32(vst(0)), 0), dVk1 = sdesc_kmajor(smem_u32(vst(1)), 0),
                   dVk2 = sdesc_kmajor(smem_u32(vst(2)), 0);
    const uint64_t dKm0 = sdesc_mnmajor(smem_u32(kst(0)), 0, T::PANEL),
                   dKm1 = sdesc_mnmajor(smem_u32(kst(1)), 0, T::PANEL),
                   dKm2 = sdesc_mnmajor(smem_u32(kst(2)), 0, T::PANEL);
    auto sel = [](int st, uint64_t a, uint64_t b, uint64_t c) { return st == 0 ? a : (st == 1 ? b : c); };
    // S = Q Kⱼᵀ (or dP = dO Vⱼᵀ): A = Q (dO) in TMEM, B = Kⱼ (Vⱼ) K-major.
    auto issue_ab = [&](uint32_t a_col, uint64_t b, uint32_t d_col, uint64_t* bar) {
      if (elect_one()) {
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          mma_ts(tmem + d_col, tmem + a_col + ks * 8, desc_add(b, kmajor_step(ks, T::PANEL)), id_s, ks > 0);
        tc_commit(bar);
      }
      __syncwarp();
    };
    bool ok = mbar_wait_warp(&s_go[0], 0, err);  // K_0, V_0 landed; Q, dO in TMEM
    if (ok) {
      tc_fence_after();
      issue_ab(Q_COL_Q, dKk0, Q_COL_S, s_full);
      issue_ab(Q_COL_DO, dVk0, Q_COL_DP, dp_full);
    }
    // Round j: S_{j+1} as soon as the compute warps hold S_j in registers,
    // then dQ += dS_j Kⱼ and dP_{j+1}; S_{j+1} keeps the tensor pipe busy
    // while dS_j is formed.
    for (int j = 0; j < n_kv && ok; ++j) {
      const int s = j % KST;
      const int s1 = (j + 1) % KST;
      const bool more = j + 1 < n_kv;
      if (more) {
        ok = mbar_wait_warp(&s_go[s1], ((j + 1) / KST) & 1, err);
        if (!ok) break;
        tc_fence_after();
        issue_ab(Q_COL_Q, sel(s1, dKk0, dKk1, dKk2), Q_COL_S, s_full);
      }
      ok = mbar_wait_warp(ds_ready, j & 1, err);
      if (!ok) break;
      tc_fence_after();
      // dQ += dS_j Kⱼ: A = dS in TMEM (bf16 in the dP columns, halves at
      // offsets 0 and 64), B = Kⱼ MN-major; then K_j and V_j are free.
      const uint64_t bk = sel(s, dKm0, dKm1, dKm2);
      if (elect_one()) {
#pragma unroll
        for (int ks = 0; ks < TILE / 16; ++ks)
          mma_ts(tmem + Q_COL_DQ, tmem + Q_COL_DP + (ks / 4) * 64 + (ks % 4) * 8,
                 desc_add(bk, mnmajor_step(ks)), id_q, (j > 0 || ks > 0) ? 1u : 0u);
        tc_commit(&kv_empty[s]);
      }
      __syncwarp();
      // dP_{j+1} overwrites the dP columns after the dQ product read dS_j.
      if (more) issue_ab(Q_COL_DO, sel(s1, dVk0, dVk1, dVk2), Q_COL_DP, dp_full);
    }
    if (elect_one()) tc_commit(final_bar);
    __syncwarp();
    mbar_wait_warp(final_bar, 0, err);
  } else {
    // ------------------------------------------------------------ compute
    // Warps 2..9: thread = query row r (TMEM lane); warp half h owns key
    // columns 64h..64h+63 of each tile.
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const int r = quarter * 32 + lane;
    const int q = q0 + r;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    constexpr float LOG2E = 1.4426950408889634f;
    const bool q_live = q < N && in_range(static_cast<long long>(bh) * N + q, 1, static_cast<long long>(BH) * N, err);
    const float lse2 = q_live ? lse[static_cast<size_t>(bh) * N + q] * LOG2E : 0.f;
    float Dq = (!FUSE_D && q_live) ? Dvec[static_cast<size_t>(bh) * N + q] : 0.f;
    float* red = reinterpret_cast<float*>(smem + L::RED_OFF);
    bool ok = mbar_wait(q_full, 0, err);
    if (ok) {
      // Copy this row of Q (half 0) or dO (half 1) into TMEM as bf16 pairs:
      // column c holds elements 2c (low half) and 2c + 1.
      const uint8_t* src = (half == 0 ? sQ : sdO);
      const uint32_t dst = tmem + lane_addr + (half == 0 ? Q_COL_Q : Q_COL_DO);
#pragma unroll
      for (int c16 = 0; c16 < D / 2; c16 += 16) {
        uint32_t w[16];
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          const int chunk = c16 / 4 + ch;  // 16-byte chunk = 8 elements = 4 columns
          const int panel = chunk / 8;
          const int off = panel * T::PANEL + r * 128 + (((chunk % 8) ^ (r & 7)) * 16);
          const uint4 v = in_range(off, 16, T::BYTES, err) ? *reinterpret_cast<const uint4*>(src + off)
                                                           : make_uint4(0u, 0u, 0u, 0u);
          w[ch * 4 + 0] = v.x;
          w[ch * 4 + 1] = v.y;
          w[ch * 4 + 2] = v.z;
          w[ch * 4 + 3] = v.w;
        }
        tmem_st16(dst + c16, w);
      }
      if constexpr (FUSE_D) {
        // This half's share of D for row r: columns 64h..64h+63 (32h.. at
        // d = 64) of O and dO, read before the dO tile is overwritten by
        // stage 2 of the K/V ring.
        constexpr int CPH = D / 16;  // 16-byte chunks per half row
        float acc = 0.f;
#pragma unroll
        for (int ch = 0; ch < CPH; ++ch) {
          const int chunk = half * CPH + ch;
          const int off = (chunk / 8) * T::PANEL + r * 128 + (((chunk % 8) ^ (r & 7)) * 16);
          if (!in_range(off, 16, T::BYTES, err)) continue;
          const uint4 a = *reinterpret_cast<const uint4*>(smem + L::O_OFF + off);
          const uint4 b = *reinterpret_cast<const uint4*>(sdO + off);
          const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
          for (int t2 = 0; t2 < 4; ++t2) {
            acc = fmaf(__uint_as_float(aw[t2] << 16), __uint_as_float(bw[t2] << 16), acc);
            acc = fmaf(__uint_as_float(aw[t2] & 0xffff0000u), __uint_as_float(bw[t2] & 0xffff0000u), acc);
          }
        }
        if (in_range(half * TILE + r, 1, 2 * TILE, err)) red[half * TILE + r] = acc;
      }
      tmem_st_wait();
      tc_fence_before();
    }
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(a_ready);
      mbar_arrive(&s_go[0]);
    }
    if constexpr (FUSE_D) {
      named_bar_sync(1, 256);  // both halves of every row written
      Dq = red[r] + red[TILE + r];
      if (ok && half == 0 && q_live) Dvec[static_cast<size_t>(bh) * N + q] = Dq;
    }
    for (int j = 0; j < n_kv && ok; ++j) {
      const int kb0 = j * TILE + half * 64;  // first key of this warp's half
      ok = mbar_wait(s_full, j & 1, err);
      if (!ok) break;
      tc_fence_after();
      const uint32_t s_addr = tmem + lane_addr + Q_COL_S + half * 64;
      const uint32_t dp_addr = tmem + lane_addr + Q_COL_DP + half * 64;
      float p[64];
      const bool masked = (kb0 + 64 > N) || (CAUSAL && kb0 + 63 > q0);
      uint32_t raw_s[64];
      tmem_ld64(s_addr, raw_s);
      tmem_ld_wait();
      // S_j is in registers: the next S may overwrite its columns.
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_go[(j + 1) % KST]);
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          const float2 e = ffma2(make_float2(__uint_as_float(raw_s[32 * h2 + c]),
                                             __uint_as_float(raw_s[32 * h2 + c + 1])),
                                 make_float2(scale_log2, scale_log2), make_float2(-lse2, -lse2));
          p[32 * h2 + c] = ex2(e.x);
          p[32 * h2 + c + 1] = ex2(e.y);
        }
        if (masked) {
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int key = kb0 + 32 * h2 + c;
            if (key >= N || (CAUSAL && key > q)) p[32 * h2 + c] = 0.f;
          }
        }
      }
      ok = mbar_wait(dp_full, j & 1, err);
      if (!ok) break;
      tc_fence_after();
      uint32_t raw[64];
      tmem_ld64(dp_addr, raw);
      tmem_ld_wait();
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        uint32_t pk[16];
#pragma unroll
        for (int t2 = 0; t2 < 16; ++t2) {
          const float* pp = p + 32 * h2 + 2 * t2;
          const uint32_t* rr = raw + 32 * h2 + 2 * t2;
          const float2 ds = fmul2(make_float2(pp[0], pp[1]),
                                  fadd2(make_float2(__uint_as_float(rr[0]), __uint_as_float(rr[1])),
                                        make_float2(-Dq, -Dq)));
          pk[t2] = pack_bf16x2(ds.x, ds.y);
        }
        tmem_st16(dp_addr + 16 * h2, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ds_ready);
    }
    // -------------------------------------------------------------- epilogue
    // dQ (scaled) in bf16, staged in the Q buffer (copied to TMEM long ago).
    if (ok) ok = mbar_wait(final_bar, 0, err);
    if (ok) {
      tc_fence_after();
      stage_tmem_rows_bf16<D / 2>(tmem + lane_addr + Q_COL_DQ, sQ, r, half * (D / 2), scale, T::BYTES, err);
      fence_async_smem();
    }
    named_bar_sync(1, 256);
    if (ok && warp == 2 && lane == 0) {
      for (int p = 0; p < T::PANELS; ++p) tma_store_3d(&tdq, sQ + p * T::PANEL, p * 64, q0, bh);
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
static cudaError_t launch_dkdv_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                 const CUtensorMap& tdo, const CUtensorMap& tdk,
                                 const CUtensorMap& tdv, const float* lse, const float* Dvec, int BHkv,
                                 int G, int N, float scale, cudaStream_t stream) {
  auto kern = bwd_dkdv_kernel<D, CAUSAL>;
  const int smem = DkdvSmem<D>::ALLOC;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int n_t = (N + TILE - 1) / TILE;
  dim3 grid(static_cast<unsigned>(n_t) * static_cast<unsigned>(BHkv));
  // A K/V head's CTAs re-read Q and dO of its G query heads (4·N·D·G bytes).
  const int group = head_group_for(4ll * N * D * G, MAX_HEAD_GROUP);
  kern<<<grid, SWEEP_THREADS, smem, stream>>>(tq, tk, tv, tdo, tdk, tdv, lse, Dvec, BHkv, G, N, group, scale,
                                               scale * 1.4426950408889634f);
  return cudaGetLastError();
}

template <int D, bool CAUSAL, bool FUSE_D>
static cudaError_t launch_dq_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                               const CUtensorMap& tdo, const CUtensorMap& tdq, const CUtensorMap& to,
                               const float* lse, float* Dvec, int BH, int G, int N, float scale,
                               cudaStream_t stream) {
  auto kern = bwd_dq_kernel<D, CAUSAL, FUSE_D>;
  const int smem = DqSmem<D, FUSE_D>::ALLOC;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int n_t = (N + TILE - 1) / TILE;
  dim3 grid(static_cast<unsigned>(n_t) * static_cast<unsigned>(BH));
  // A query head's CTAs re-read K and V of its K/V head, shared by G heads.
  const int group = head_group_for(4ll * N * D / G, MAX_HEAD_GROUP);
  kern<<<grid, SWEEP_THREADS, smem, stream>>>(tq, tk, tv, tdo, tdq, to, lse, Dvec, BH, G, N, group, scale,
                                               scale * 1.4426950408889634f);
  return cudaGetLastError();
}

template <bool FUSE_D>
static cudaError_t launch_dq(const void* q, const void* k, const void* v, const void* o, const void* dO,
                             void* dq, const float* lse, float* Dvec, int BH, int G, int N, int d,
                             float scale, bool causal, cudaStream_t stream) {
  CUtensorMap tq, tk, tv, tdo, tdq, to;
  const int T = TILE;
  const int BHkv = BH / G;
  if (!make_tmap_bf16(&tq, q, BH, N, d, T) || !make_tmap_bf16(&tdo, dO, BH, N, d, T) ||
      !make_tmap_bf16(&tk, k, BHkv, N, d, T) || !make_tmap_bf16(&tv, v, BHkv, N, d, T) ||
      !make_tmap_bf16(&tdq, dq, BH, N, d, T))
    return cudaErrorInvalidValue;
  if (!FUSE_D) to = tq;  // unused
  else if (!make_tmap_bf16(&to, o, BH, N, d, T)) return cudaErrorInvalidValue;
  if (d == 64)
    return causal ? launch_dq_t<64, true, FUSE_D>(tq, tk, tv, tdo, tdq, to, lse, Dvec, BH, G, N, scale, stream)
                  : launch_dq_t<64, false, FUSE_D>(tq, tk, tv, tdo, tdq, to, lse, Dvec, BH, G, N, scale, stream);
  return causal ? launch_dq_t<128, true, FUSE_D>(tq, tk, tv, tdo, tdq, to, lse, Dvec, BH, G, N, scale, stream)
                : launch_dq_t<128, false, FUSE_D>(tq, tk, tv, tdo, tdq, to, lse, Dvec, BH, G, N, scale, stream);
}

}  // namespace bwd

cudaError_t launch_bwd_preprocess(const __nv_bfloat16* o, const __nv_bfloat16* dO, float* Dvec,
                                  int BH, int N, int d, cudaStream_t stream) {
  const long long rows = static_cast<long long>(BH) * N;
  if (d == 64) {
    const long long blocks = (rows + 31) / 32;
    bwd::preprocess_kernel<64><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(o, dO, Dvec, rows);
  } else {
    const long long blocks = (rows + 15) / 16;
    bwd::preprocess_kernel<128><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(o, dO, Dvec, rows);
  }
  return cudaGetLastError();
}

cudaError_t launch_bwd_dkdv(const void* q, const void* k, const void* v, const void* dO, void* dk,
                            void* dv, const float* lse, const float* Dvec, int BH, int G, int N, int d,
                            float scale, bool causal, cudaStream_t stream) {
  CUtensorMap tq, tk, tv, tdo, tdk, tdv;
  const int T = bwd::TILE;
  const int BHkv = BH / G;
  if (!make_tmap_bf16(&tq, q, BH, N, d, T) || !make_tmap_bf16(&tdo, dO, BH, N, d, T) ||
      !make_tmap_bf16(&tk, k, BHkv, N, d, T) || !make_tmap_bf16(&tv, v, BHkv, N, d, T) ||
      !make_tmap_bf16(&tdk, dk, BHkv, N, d, T) || !make_tmap_bf16(&tdv, dv, BHkv, N, d, T))
    return cudaErrorInvalidValue;
  if (d == 64)
    return causal ? bwd::launch_dkdv_t<64, true>(tq, tk, tv, tdo, tdk, tdv, lse, Dvec, BHkv, G, N, scale, stream)
                  : bwd::launch_dkdv_t<64, false>(tq, tk, tv, tdo, tdk, tdv, lse, Dvec, BHkv, G, N, scale, stream);
  return causal ? bwd::launch_dkdv_t<128, true>(tq, tk, tv, tdo, tdk, tdv, lse, Dvec, BHkv, G, N, scale, stream)
                : bwd::launch_dkdv_t<128, false>(tq, tk, tv, tdo, tdk, tdv, lse, Dvec, BHkv, G, N, scale, stream);
}

cudaError_t launch_bwd_dq(const void* q, const void* k, const void* v, const void* dO, void* dq,
                          const float* lse, const float* Dvec, int BH, int G, int N, int d, float scale,
                          bool causal, cudaStream_t stream) {
  // D is only read in this form.
  return bwd::launch_dq<false>(q, k, v, nullptr, dO, dq, lse, const_cast<float*>(Dvec), BH, G, N, d, scale,
                               causal, stream);
}

cudaError_t launch_bwd_dq_d(const void* q, const void* k, const void* v, const void* o, const void* dO,
                            void* dq, const float* lse, float* Dvec, int BH, int G, int N, int d, float scale,
                            bool causal, cudaStream_t stream) {
  return bwd::launch_dq<true>(q, k, v, o, dO, dq, lse, Dvec, BH, G, N, d, scale, causal, stream);
}

bool bwd_fuse_d(int BH, int G, int N) {
  if (G != 1) return false;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
    return false;
  const long long ctas = static_cast<long long>(BH) * ((N + bwd::TILE - 1) / bwd::TILE);
  return ctas >= 4LL * sms;
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
