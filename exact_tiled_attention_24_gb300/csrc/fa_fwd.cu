// Forward pass of exact attention, computed tile by tile with online softmax.
//
// Method (CMU 10-423 L17–L18 notes, section "FlashAttention 本身"; dcwnkz.com
// GPU-tricks article, FlashAttention section and its six-score worked
// example): for a block of query rows, sweep the keys/values in tiles of
// 128; keep per row the running max m, the running denominator l and the
// running weighted sum O; when a tile raises m, multiply l and O by
// e^(m_old - m_new) before adding the tile; divide by l once at the end.
// S = Q Kᵀ and P never leave the SM: S lives in tensor memory (TMEM), P is
// written back into TMEM as bf16 and fed straight to the P·V MMA.
//
// One CTA owns two 128-row query tiles (Q0, Q1) of one head and sweeps the
// key/value tiles once for both ("ping-pong"): while one softmax group
// exponentiates its S tile, the tensor core runs the other group's products.
// Roles (320 threads):
//   warp 0      TMA producer: Q0, K_0 and Q1 once, then V_j with K_{j+1}
//               into 2-stage rings (one full and one empty barrier per pair)
//   warp 1      TMEM owner and MMA issuer (warp-uniform, one elected lane issues)
//   warps 2..5  softmax group 0 (Q0), one thread per query row (TMEM lane)
//   warps 6..9  softmax group 1 (Q1)
// TMEM columns: S0 0.., S1 128.., O0 256.., O1 384... The MMA order is
//   S0_0 S1_0 | PV0_0 S0_1 PV1_0 S1_1 | PV0_1 S0_2 ...
// S_g,j+1 overwrites the columns PV_g,j reads P from; it is issued after it
// on the same thread and tcgen05 MMAs execute in issue order.
//
// Rescaling: the exponent reference m of a row is raised to the running max
// only when the max has grown past it by more than RESCALE_LOG2 (in log2
// units); O and l are then multiplied by 2^(m_old - m_new) as in the worked
// example. Between raises P = 2^(s - m) may exceed 1 (at most 2^RESCALE_LOG2),
// which bf16 and the fp32 sums carry as well; the final O / l is the same
// quantity because numerator and denominator share the reference.
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

constexpr int BM = 128;       // query rows per tile (two tiles per CTA)
constexpr int BN = 128;       // keys per tile
constexpr int THREADS = 320;  // 10 warps
constexpr int MAX_HEAD_GROUP = 8;
constexpr float RESCALE_LOG2 = 8.f;

template <int D>
struct Smem {
  static constexpr int PANELS = D / 64;
  static constexpr int STAGES = 2;
  static constexpr int TILE_BYTES = BM * D * 2;  // = BN * D * 2
  static constexpr int PANEL = BM * 128;
  static constexpr int Q_OFF = 0;                // Q0, Q1 (later the O staging tiles)
  static constexpr int K_OFF = Q_OFF + 2 * TILE_BYTES;
  static constexpr int V_OFF = K_OFF + STAGES * TILE_BYTES;
  static constexpr int BAR_OFF = V_OFF + STAGES * TILE_BYTES;
  // q_full (Q0), k0_full, kv_full[2], kv_empty[2], s_full[2], p_ready[2]
  // (keys 0..63 of P), pv_done[2], final, p_hi[2] (keys 64..127), q1_full (Q1)
  static constexpr int NBARS = 2 + 2 * STAGES + 6 + 1 + 2 + 1;
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
                  float* __restrict__ lse, int BH, int G, int N, int head_group, float scale_log2) {
  using L = Smem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem + L::Q_OFF;
  uint8_t* sK = smem + L::K_OFF;
  uint8_t* sV = smem + L::V_OFF;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  // Step j of the sweep reads V_j and K_{j+1} (for S_{j+1}); the two are
  // loaded together and released together, so one full and one empty
  // barrier per slot serve both rings: slot j % 2 holds V_j in V stage
  // j % 2 and K_{j+1} in K stage (j + 1) % 2. K_0 has its own barrier.
  uint64_t* q_full = bars;
  uint64_t* k0_full = bars + 1;
  uint64_t* kv_full = bars + 2;                // [2]
  uint64_t* kv_empty = kv_full + L::STAGES;    // [2]
  uint64_t* s_full = kv_empty + L::STAGES;     // [2], one per group
  uint64_t* p_ready = s_full + 2;           // [2]
  uint64_t* pv_done = p_ready + 2;          // [2]
  uint64_t* final_bar = pv_done + 2;
  uint64_t* p_hi = final_bar + 1;           // [2]
  uint64_t* q1_full = p_hi + 2;  // Q1 (q_full: Q0): group 0's first S needs only Q0 and K_0
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::TMEM_SLOT_OFF);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Heads in groups of head_group (sized so that their K/V stay in L2 while
  // the group runs); within a group the heaviest (causal) query blocks go
  // first.
  const int n_qb = (N + 2 * BM - 1) / (2 * BM);  // blocks of two query tiles
  int t, bh;
  grouped_tile_order(static_cast<int>(blockIdx.x), BH, n_qb, head_group, &t, &bh);
  const int qb = n_qb - 1 - t;
  const int bkv = bh / G;  // K/V head shared by G consecutive query heads
  const int qrow0 = qb * 2 * BM;
  const int n_kt_all = (N + BN - 1) / BN;
  // key tiles per group: group g covers rows qrow0 + 128g .. + 127
  const int n_g0 = CAUSAL ? min(n_kt_all, 2 * qb + 1) : n_kt_all;
  const int n_g1 = CAUSAL ? min(n_kt_all, 2 * qb + 2) : n_kt_all;
  const int n_kt = n_g1;  // n_g1 >= n_g0 >= 1

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q1_full, 1);
    mbar_init(k0_full, 1);
    for (int s = 0; s < L::STAGES; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int g = 0; g < 2; ++g) {
      mbar_init(&s_full[g], 1);
      mbar_init(&p_ready[g], 4);
      mbar_init(&p_hi[g], 4);
      mbar_init(&pv_done[g], 1);
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
      // Q0 and K_0 first: group 0's first S needs only these two.
      mbar_arrive_expect_tx(q_full, L::TILE_BYTES);
      for (int p = 0; p < L::PANELS; ++p)
        tma_load_3d(sQ + p * L::PANEL, &tq, q_full, p * 64, qrow0, bh);
      mbar_arrive_expect_tx(k0_full, L::TILE_BYTES);
      for (int p = 0; p < L::PANELS; ++p)
        tma_load_3d(sK + p * L::PANEL, &tk, k0_full, p * 64, 0, bkv);
      mbar_arrive_expect_tx(q1_full, L::TILE_BYTES);
      for (int p = 0; p < L::PANELS; ++p)
        tma_load_3d(sQ + L::TILE_BYTES + p * L::PANEL, &tq, q1_full, p * 64, qrow0 + BM, bh);
      // Slot j: V_j and K_{j+1}, issued once step j - 2 (the prologue for
      // j = 1, whose S_0 read K_0) has released their stages.
      int issued = 0;
      for (int j = 0; j < n_kt; ++j) {
        const int sv = j % L::STAGES, sk = (j + 1) % L::STAGES;
        const bool has_k = j + 1 < n_kt;
        if (j >= 1 && !mbar_wait(&kv_empty[sv], ((j - 1) / 2) & 1, err)) break;
        mbar_arrive_expect_tx(&kv_full[sv], L::TILE_BYTES * (has_k ? 2 : 1));
        for (int p = 0; p < L::PANELS; ++p)
          tma_load_3d(sV + sv * L::TILE_BYTES + p * L::PANEL, &tv, &kv_full[sv], p * 64, j * BN, bkv);
        if (has_k)
          for (int p = 0; p < L::PANELS; ++p)
            tma_load_3d(sK + sk * L::TILE_BYTES + p * L::PANEL, &tk, &kv_full[sv], p * 64, (j + 1) * BN, bkv);
        issued = j + 1;
      }
      // Drain: never leave the CTA with copies still landing in its smem.
      mbar_wait(q_full, 0, err);
      mbar_wait(q1_full, 0, err);
      mbar_wait(k0_full, 0, err);
      for (int j = max(0, issued - L::STAGES); j < issued; ++j)
        mbar_wait(&kv_full[j % L::STAGES], (j / L::STAGES) & 1, err);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    // The whole warp runs this loop (descriptors stay warp-uniform, so the
    // per-MMA work is cheap even while the softmax warps saturate the issue
    // slots); one elected lane issues the MMAs and commits.
    constexpr uint32_t idesc_s = idesc_bf16(BM, BN, false, false);
    constexpr uint32_t idesc_o = idesc_bf16(BM, D, false, true);
    static_assert(L::STAGES == 2, "descriptor selection assumes two stages");
    const uint64_t dq0 = sdesc_kmajor(smem_u32(sQ), 0);
    const uint64_t dq1 = sdesc_kmajor(smem_u32(sQ + L::TILE_BYTES), 0);
    const uint64_t dk0 = sdesc_kmajor(smem_u32(sK), 0);
    const uint64_t dk1 = sdesc_kmajor(smem_u32(sK + L::TILE_BYTES), 0);
    const uint64_t dv0 = sdesc_mnmajor(smem_u32(sV), 0, L::PANEL);
    const uint64_t dv1 = sdesc_mnmajor(smem_u32(sV + L::TILE_BYTES), 0, L::PANEL);
    // S_g = Q_g K_jᵀ into the S columns of group g (K_j in stage s).
    auto issue_s = [&](int g, int s) {
      const uint64_t a = g ? dq1 : dq0, b = s ? dk1 : dk0;
      const uint32_t d = tmem + g * BN;
      if (elect_one()) {
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          mma_ss(d, desc_add(a, kmajor_step(ks, L::PANEL)), desc_add(b, kmajor_step(ks, L::PANEL)),
                 idesc_s, ks > 0);
        tc_commit(&s_full[g]);
      }
      __syncwarp();
    };
    // O_g += P_g V_j over keys 64·half .. 64·half + 63; P_g is bf16 in the
    // first 64 S columns of group g. The second half commits pv_done.
    auto issue_pv = [&](int g, int s, int half, uint32_t acc0) {
      const uint64_t b = s ? dv1 : dv0;
      const uint32_t d = tmem + 256 + g * 128;
      const uint32_t a = tmem + g * BN;
      if (elect_one()) {
#pragma unroll
        for (int k4 = 0; k4 < BN / 32; ++k4) {
          const int ks = half * (BN / 32) + k4;
          mma_ts(d, a + ks * 8, desc_add(b, mnmajor_step(ks)), idesc_o, ks > 0 ? 1u : acc0);
        }
        if (half == 1) tc_commit(&pv_done[g]);
      }
      __syncwarp();
    };
    auto commit = [&](uint64_t* bar) {
      if (elect_one()) tc_commit(bar);
      __syncwarp();
    };
    bool ok = mbar_wait_warp(q_full, 0, err) && mbar_wait_warp(k0_full, 0, err);
    if (ok) {
      tc_fence_after();
      issue_s(0, 0);
      ok = mbar_wait_warp(q1_full, 0, err);
    }
    if (ok) {
      tc_fence_after();
      issue_s(1, 0);
      commit(&kv_empty[1]);  // K_0 read: slot 1 (V_1, K_2) may load
    }
    for (int j = 0; j < n_kt && ok; ++j) {
      const int s = j % L::STAGES;
      const int s1 = (j + 1) % L::STAGES;
      // The data wait (V_j and K_{j+1}) comes first: it is normally met and
      // overlaps the wait for P_j, so no wait sits between two products.
      ok = mbar_wait_warp(&kv_full[s], (j / L::STAGES) & 1, err);
      if (!ok) break;
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        const int n_g = (g == 0) ? n_g0 : n_g1;
        if (j >= n_g) continue;
        // P·V on keys 0..63 as soon as that half of P is written, then on
        // keys 64..127: the tensor core starts while the softmax warps are
        // still on the second half.
        ok = mbar_wait_warp(&p_ready[g], j & 1, err);
        if (!ok) break;
        tc_fence_after();
        issue_pv(g, s, 0, j > 0 ? 1u : 0u);
        ok = mbar_wait_warp(&p_hi[g], j & 1, err);
        if (!ok) break;
        tc_fence_after();
        issue_pv(g, s, 1, 1u);
        if (j + 1 < n_g) issue_s(g, s1);
      }
      if (!ok) break;
      commit(&kv_empty[s]);  // V_j read by PV_j, K_{j+1} by S_{j+1}
    }
    commit(final_bar);
    mbar_wait_warp(final_bar, 0, err);
  } else {
    // ------------------------------------------------------------ softmax
    const int g = (warp - 2) >> 2;  // group
    const int quarter = warp & 3;   // TMEM lanes 32*quarter .. +31
    const int r = quarter * 32 + lane;
    const int q0 = qrow0 + g * BM;
    const int qrow = q0 + r;
    const int n_mine = (g == 0) ? n_g0 : n_g1;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t s_addr = tmem + lane_addr + g * BN;
    const uint32_t o_addr = tmem + lane_addr + 256 + g * 128;
    float m = -INFINITY;  // exponent reference (log2 units of scaled scores)
    float l = 0.f;        // running denominator relative to m
    bool ok = true;
    for (int j = 0; j < n_mine; ++j) {
      ok = mbar_wait(&s_full[g], j & 1, err);
      if (!ok) break;
      tc_fence_after();
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
      if ((k0 + BN > N) || (CAUSAL && k0 + BN - 1 > q0)) {
#pragma unroll
        for (int c = 0; c < BN; ++c) {
          const int key = k0 + c;
          if (key >= N || (CAUSAL && key > qrow)) x[c] = -INFINITY;
        }
      }
      // P for 32 columns from c on, relative to the reference -nm.x; bf16
      // into the S columns (P_j is read by the P·V product only after its
      // release), the fp32 values into the running sums. Packed fp32 pairs:
      // the scale-and-shift and the sums take one instruction per two
      // scores; four packed sums = eight independent chains.
      float2 sum[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) sum[u] = make_float2(0.f, 0.f);
      const float2 sc2 = make_float2(scale_log2, scale_log2);
      auto p_chunk = [&](int c, float2 nm2) {
        uint32_t pk[16];
#pragma unroll
        for (int t2 = 0; t2 < 16; ++t2) {
          const float2 e = ffma2(make_float2(x[c + 2 * t2], x[c + 2 * t2 + 1]), sc2, nm2);
          const float p0 = ex2(e.x);
          const float p1 = ex2(e.y);
          sum[t2 & 3] = fadd2(sum[t2 & 3], make_float2(p0, p1));
          pk[t2] = pack_bf16x2(p0, p1);
        }
        tmem_st16(s_addr + c / 2, pk);  // P (bf16) into the first 64 S columns
      };
      auto release = [&](uint64_t* bar) {  // this half of P is in TMEM
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar);
      };
      // The first half of P is formed against the current reference before
      // the tile maximum is known (the maximum is computed alongside); it
      // stands unless the maximum outgrew the reference by more than the
      // threshold, which is rare after the first tile. The first tile has
      // no reference yet.
      if (j > 0) {
        p_chunk(0, make_float2(-m, -m));
        p_chunk(32, make_float2(-m, -m));
      }
      // Eight independent max chains, two new scores per three-input max.
      float mx[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) mx[u] = fmaxf(x[u], x[8 + u]);
#pragma unroll
      for (int c = 16; c < BN; c += 16)
#pragma unroll
        for (int u = 0; u < 8; ++u) mx[u] = fmax3(mx[u], x[c + u], x[c + 8 + u]);
      const float tile_max = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]),
                                   fmaxf(mx[6], mx[7])) * scale_log2;
      // Raise the reference when the max outgrew it by more than the
      // threshold (always on the first tile, where m = -inf).
      const bool warp_raise = __any_sync(0xffffffffu, tile_max > m + RESCALE_LOG2);
      if (warp_raise) {
        const float m_new = fmaxf(m, tile_max);
        const float alpha = ex2(m - m_new);  // 0 on the first tile
        m = m_new;
        l *= alpha;
        // O *= alpha once P V_{j-1} has landed, before any of P_j is
        // released, since P V_j accumulates into O.
        if (j > 0) {
          ok = mbar_wait(&pv_done[g], (j - 1) & 1, err);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < D; c += 32) {
            uint32_t o[32];
            tmem_ld32(o_addr + c, o);
            tmem_ld_wait();
            uint32_t a[16], bb[16];
#pragma unroll
            for (int t2 = 0; t2 < 16; ++t2) {
              a[t2] = __float_as_uint(__uint_as_float(o[t2]) * alpha);
              bb[t2] = __float_as_uint(__uint_as_float(o[16 + t2]) * alpha);
            }
            tmem_st16(o_addr + c, a);
            tmem_st16(o_addr + c + 16, bb);
          }
        }
        // The first half again, against the new reference.
#pragma unroll
        for (int u = 0; u < 4; ++u) sum[u] = make_float2(0.f, 0.f);
        p_chunk(0, make_float2(-m, -m));
        p_chunk(32, make_float2(-m, -m));
      }
      release(&p_ready[g]);
      p_chunk(64, make_float2(-m, -m));
      p_chunk(96, make_float2(-m, -m));
      release(&p_hi[g]);
      l += ((sum[0].x + sum[0].y) + (sum[1].x + sum[1].y)) + ((sum[2].x + sum[2].y) + (sum[3].x + sum[3].y));
    }
    // -------------------------------------------------------------- epilogue
    if (ok) ok = mbar_wait(&pv_done[g], (n_mine - 1) & 1, err);
    uint8_t* stage = sQ + g * L::TILE_BYTES;  // Q_g is no longer read by any MMA
    if (ok) {
      tc_fence_after();
      const float inv_l = 1.f / l;
#pragma unroll
      for (int c = 0; c < D; c += 32) {
        uint32_t o[32];
        tmem_ld32(o_addr + c, o);
        tmem_ld_wait();
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
          const int off = g * L::TILE_BYTES + panel * L::PANEL + r * 128 + ((chunk ^ (r & 7)) * 16);
          if (in_range(off, 16, 2 * L::TILE_BYTES, err))  // the Q0, Q1 region
            *reinterpret_cast<uint4*>(sQ + off) = val;
        }
      }
      const long long lrow = static_cast<long long>(bh) * N + qrow;
      if (qrow < N && in_range(lrow, 1, static_cast<long long>(BH) * N, err)) {
        // lse in natural-log units: (m + log2 l) * ln 2
        lse[lrow] = (m + __log2f(l)) * 0.69314718055994531f;
      }
      fence_async_smem();
    }
    named_bar_sync(1 + g, 128);
    if (ok && (warp & 3) == 2 && lane == 0 && q0 < N) {
      for (int p = 0; p < L::PANELS; ++p) tma_store_3d(&to, stage + p * L::PANEL, p * 64, q0, bh);
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
                            const CUtensorMap& to, float* lse, int BH, int G, int N, float scale,
                            cudaStream_t stream) {
  auto kern = fa_fwd_kernel<D, CAUSAL>;
  const int smem = Smem<D>::ALLOC;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int n_qb = (N + 2 * BM - 1) / (2 * BM);
  dim3 grid(static_cast<unsigned>(n_qb) * static_cast<unsigned>(BH));
  const float scale_log2 = scale * 1.4426950408889634f;
  // K and V of one K/V head (4·N·D bytes) serve G query heads.
  const int group = head_group_for(4ll * N * D / G, MAX_HEAD_GROUP);
  kern<<<grid, THREADS, smem, stream>>>(tq, tk, tv, to, lse, BH, G, N, group, scale_log2);
  return cudaGetLastError();
}

}  // namespace fwd

cudaError_t launch_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int BH,
                       int G, int N, int d, float scale, bool causal, cudaStream_t stream) {
  CUtensorMap tq, tk, tv, to;
  const int BHkv = BH / G;
  if (!make_tmap_bf16(&tq, q, BH, N, d, fwd::BM) || !make_tmap_bf16(&tk, k, BHkv, N, d, fwd::BN) ||
      !make_tmap_bf16(&tv, v, BHkv, N, d, fwd::BN) || !make_tmap_bf16(&to, o, BH, N, d, fwd::BM))
    return cudaErrorInvalidValue;
  if (d == 64)
    return causal ? fwd::launch_t<64, true>(tq, tk, tv, to, lse, BH, G, N, scale, stream)
                  : fwd::launch_t<64, false>(tq, tk, tv, to, lse, BH, G, N, scale, stream);
  return causal ? fwd::launch_t<128, true>(tq, tk, tv, to, lse, BH, G, N, scale, stream)
                : fwd::launch_t<128, false>(tq, tk, tv, to, lse, BH, G, N, scale, stream);
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
