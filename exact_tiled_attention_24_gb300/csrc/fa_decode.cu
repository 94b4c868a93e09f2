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
//   decode_mma  one CTA per (context split, K/V head, request, 16 query
//               heads): both products of each 128-key tile on the tensor
//               cores; writes o_s (fp32) and lse_s per head.
//   merge       one warp per output row: the combination above.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "fa_common.h"
#include "fa_ptx.cuh"
#include "fa_tmap.h"

namespace fa {

static __device__ uint32_t g_dec_err;

namespace dec {

constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.69314718055994531f;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// One warp per output row: o = Σ_s e^(lse_s − lse) o_s, lse = ln Σ_s e^(lse_s).
// Lane i computes the weight of part i (of each group of 32), and the parts'
// output slices are loaded several at a time before any is used, so a row
// takes a few round trips to memory, not one per part. The sums run over the
// parts in order, the same arithmetic as one part after another.
template <int D>
__global__ void __launch_bounds__(256) merge_kernel(const float* __restrict__ o_parts,
                                                    const float* __restrict__ lse_parts, int S,
                                                    __nv_bfloat16* __restrict__ o, float* __restrict__ lse,
                                                    long long rows) {
  constexpr int CPL = D / 32;  // columns per lane: 4 (d = 128) or 2 (d = 64)
  constexpr int U = 16 / CPL;  // part slices in flight per lane (16 floats: the merge fits one wave)
  using Vec = typename std::conditional<CPL == 4, float4, float2>::type;
  const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  uint32_t* err = &g_dec_err;
  const long long prt = static_cast<long long>(S) * rows;  // rows of the partial results
  float m = -INFINITY;
  for (int s = lane; s < S; s += 32)
    if (in_range(s * rows + row, 1, prt, err)) m = fmaxf(m, lse_parts[s * rows + row]);
  m = warp_max(m);
  float l = 0.f;
  float acc[CPL];
#pragma unroll
  for (int j = 0; j < CPL; ++j) acc[j] = 0.f;
  if (m != -INFINITY) {
    for (int s0 = 0; s0 < S; s0 += 32) {
      const int sl = s0 + lane;
      float wl = 0.f;  // weight of part sl (0 for a part that is not there)
      if (sl < S && in_range(sl * rows + row, 1, prt, err)) wl = ex2((lse_parts[sl * rows + row] - m) * LOG2E);
      const int n = min(32, S - s0);
      for (int s1 = 0; s1 < n; s1 += U) {
        Vec v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const long long off = ((s0 + s1 + u) * rows + row) * D + lane * CPL;
          if (s1 + u < n && in_range(off, CPL, prt * D, err)) v[u] = *reinterpret_cast<const Vec*>(o_parts + off);
          else v[u] = Vec{};
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const float w = __shfl_sync(0xffffffffu, wl, s1 + u);
          if (s1 + u < n) {
            l += w;
            const float* x = reinterpret_cast<const float*>(&v[u]);
#pragma unroll
            for (int j = 0; j < CPL; ++j) acc[j] = fmaf(w, x[j], acc[j]);
          }
        }
      }
    }
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
  for (int j = 0; j < CPL; j += 2)
    if (in_range(row * D + lane * CPL + j, 2, rows * D, err))
      *reinterpret_cast<__nv_bfloat162*>(o + row * D + lane * CPL + j) =
          __floats2bfloat162_rn(acc[j] * inv, acc[j + 1] * inv);
  if (lane == 0 && in_range(row, 1, rows, err)) lse[row] = l > 0.f ? m + __logf(l) : -INFINITY;
}

}  // namespace dec

// ----------------------------------------------------------------------------
// The decode step on the tensor cores (d = 64 or 128, any cache block size).
//
// The work per K/V byte is small (G·d multiply-adds per key and head pair),
// but done on the FMA pipe its instruction stream, not HBM, sets the rate:
// converting bf16 rows, dot products and shuffles came to about 140 warp
// instructions per KB. Here both products of a 128-key tile run on the
// tensor core with the tile's keys as M, so the work per key is a few
// instructions of softmax:
//   Sᵀ = K Qᵀ    M = 128 keys, N = 16 query heads (padded), K = d; into TMEM
//   Oᵀ += Vᵀ Pᵀ  M = 128 dims (d = 64: padded by a zero panel), N = 16 heads,
//                K = 128 keys; accumulated in TMEM
// One thread per TMEM lane: lane r is key r of the tile in Sᵀ and dimension r
// in Oᵀ. K and V tiles reach shared memory in the 128-byte-swizzled K-major
// layout the products read, one of two ways:
//   boxes   block size a multiple of 8 dividing 128: each cache block of the
//           tile is its own TMA box (the cache viewed as (d, block_size,
//           num_blocks·Hkv)) at row offset block·block_size of the tile; a
//           block past the context or with a table entry outside
//           [0, num_blocks) is requested at an out-of-range coordinate, so
//           the box reads zeros and the entry is never dereferenced. Lane i
//           of the producer warp issues block i's box; the table entries
//           are loaded two tiles ahead, the first ones before the setup.
//   gather  any other block size: the producer warp's lanes look up each
//           token's block and copy its row in 16-byte pieces to the
//           swizzled position (zero fill for the same two cases). Each lane
//           arrives on the tile's barrier when its copies land, and the
//           issuer fences them for the tensor core after its wait. Below 8
//           tokens per block the lookups are loaded two tiles ahead.
// The softmax keeps one exponent reference per head, raised (and Oᵀ's column
// rescaled) when a key outgrows it by more than 2^8, as in the forward.
// Roles (224 threads): warp 0 loads K tiles, warp 1 V tiles (the whole
// warp: a lane per box, or four rows per lane to gather), warp 2 owns TMEM
// and issues the products, warps 3..6 run the softmax and the epilogue. Two
// or three CTAs share an SM.
namespace decmma {

constexpr int TK = 128;       // keys per tile (M of the score product)
constexpr int NH = 16;        // query heads per CTA (N of both products)
constexpr int THREADS = 224;  // 7 warps
constexpr float RESCALE_LOG2 = 8.f;

// Per-CTA configuration by the number of query heads GM the softmax keeps
// state for (4, 8 or 16). With up to 8 heads the state fits 80 registers,
// and three CTAs share an SM with one K stage, one V stage and one Pᵀ
// buffer each (more CTAs hide each one's start and finish better than
// deeper rings: measured 5930 against 5400 GB/s). With 16 heads, two CTAs
// with two K stages and two Pᵀ buffers.
template <int GM>
struct Cfg {
  static constexpr int CTAS = GM <= 8 ? 3 : 2;
  static constexpr int KST = CTAS == 3 ? 1 : 2, VST = 1, PB = CTAS == 3 ? 1 : 2;
};

// K tiles hold D / 64 panels of 64 columns; a V tile always holds two, so
// that Oᵀ = Vᵀ Pᵀ is an M = 128 product: at d = 64 its second panel stays
// zero, and rows 64..127 of Oᵀ are zero and never written out.
template <int D, int KST, int VST, int PB>
struct Smem {
  static constexpr int PANEL = TK * 128;   // 128 rows x 64 bf16 columns
  static constexpr int KPANELS = D / 64;
  static constexpr int K_TILE = KPANELS * PANEL;
  static constexpr int V_TILE = 2 * PANEL;
  static constexpr int QPANEL = NH * 128;  // 16 rows x 64 bf16 columns
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = K_OFF + KST * K_TILE;
  static constexpr int Q_OFF = V_OFF + VST * V_TILE;
  static constexpr int P_OFF = Q_OFF + KPANELS * QPANEL;   // Pᵀ: PB buffers x 2 panels (16 heads x 128 keys)
  static constexpr int RED_OFF = P_OFF + PB * 2 * QPANEL;  // [4 warps][NH] fp32
  static constexpr int BAR_OFF = RED_OFF + 4 * NH * 4;
  // q_full, k_full[KST], k_empty[KST], v_full[VST], v_empty[VST], s_full[2],
  // p_full[PB], p_empty[PB], o_done, final
  static constexpr int NBARS = 1 + 2 * KST + 2 * VST + 2 + 2 * PB + 2;
  static constexpr int TMEM_SLOT_OFF = BAR_OFF + NBARS * 8;
  static constexpr int BYTES = TMEM_SLOT_OFF + 16;
  static constexpr int ALLOC = BYTES + 1024;  // slack for 1024-byte alignment
};

// How K and V tiles reach shared memory. BOXES: one TMA box per cache block
// (a block size that is a multiple of 8 dividing 128, so boxes land on whole
// 8-row swizzle groups). Otherwise per-token 16-byte copies, with tk and tv
// unused and kc, vc read directly: GATHER looks up a tile's block-table
// entries after issuing the previous tile's copies; GATHER_AHEAD (block
// sizes below 8, where a tile needs 16 or more distinct entries) loads them
// two tiles ahead and the first ones before the CTA's setup.
enum TileLoad : int { BOXES = 0, GATHER = 1, GATHER_AHEAD = 2 };

template <int D, int GM, int LOAD>
__global__ void __launch_bounds__(THREADS, Cfg<GM>::CTAS) decode_mma_kernel(
    const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
    const __grid_constant__ CUtensorMap tv, const __nv_bfloat16* __restrict__ kc,
    const __nv_bfloat16* __restrict__ vc, const int* __restrict__ block_table,
    const int* __restrict__ seq_lens, float* __restrict__ o_part, float* __restrict__ lse_part,
    __nv_bfloat16* __restrict__ o_out, float* __restrict__ lse_out, int B, int H,
    int Hkv, int num_blocks, int bs, int max_blocks, float scale_log2) {
  constexpr int KST = Cfg<GM>::KST, VST = Cfg<GM>::VST, PB = Cfg<GM>::PB;
  constexpr bool GATHERED = LOAD != BOXES, AHEAD = LOAD == GATHER_AHEAD;
  using L = Smem<D, KST, VST, PB>;
  static_assert(Cfg<GM>::CTAS * (L::ALLOC + 1024) <= 233472, "the CTAs must fit an SM");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int S = gridDim.x;
  const int G_all = H / Hkv;
  const int n_chunk = (G_all + NH - 1) / NH;
  const int s = blockIdx.x, hk = blockIdx.y / n_chunk, chunk = blockIdx.y % n_chunk, b = blockIdx.z;
  const int G = min(GM, G_all - NH * chunk);  // query heads served by this CTA (GM covers them)
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  uint32_t* err = &g_dec_err;

  int Lb = in_range(b, 1, B, err) ? seq_lens[b] : 0;
  Lb = Lb < 0 ? 0 : (Lb > max_blocks * bs ? max_blocks * bs : Lb);
  const int n_tiles = (Lb + TK - 1) / TK;
  const int tps = (n_tiles + S - 1) / S;
  const int tile0 = s * tps;
  const int tile1 = min(n_tiles, tile0 + tps);
  const int head0 = b * H + hk * G_all + NH * chunk;        // first query head (row of q)
  const long long prow = static_cast<long long>(s) * B * H + head0;  // its partial row
  const long long part_rows = static_cast<long long>(S) * B * H;
  if (tile0 >= tile1) {  // no key in this split: o_s = 0, lse_s = -inf (weight 0 in the merge)
    for (int i = threadIdx.x; i < G * D; i += THREADS) {
      if (S == 1) {
        if (in_range(prow * D + i, 1, part_rows * D, err)) o_out[prow * D + i] = __float2bfloat16_rn(0.f);
      } else if (in_range(prow * D + i, 1, part_rows * D, err)) {
        o_part[prow * D + i] = 0.f;
      }
    }
    if (threadIdx.x < G && in_range(prow + threadIdx.x, 1, part_rows, err))
      (S == 1 ? lse_out : lse_part)[prow + threadIdx.x] = -INFINITY;
    return;
  }
  const int n_t = tile1 - tile0;
  const int t_end = min(Lb, tile1 * TK);  // keys at or past t_end are masked

  // GATHER_AHEAD: fetch() loads the block-table entries of rows lane,
  // lane + 32, lane + 64 and lane + 96 of a tile (0 past the context, -1 for
  // an index outside the table) into registers; the producer lanes use them
  // two tiles later. The first two tiles' loads are issued here, before the
  // CTA's setup.
  auto fetch = [&](int tile, int (&raw)[4]) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int t = tile * TK + lane + 32 * u;
      int e = 0;
      if (t < Lb) {
        const long long ti = static_cast<long long>(b) * max_blocks + t / bs;
        e = in_range(ti, 1, static_cast<long long>(B) * max_blocks, err) ? block_table[ti] : -1;
      }
      raw[u] = e;
    }
  };
  int raw_a[4] = {0, 0, 0, 0}, raw_b[4] = {0, 0, 0, 0};
  if (AHEAD && warp <= 1) {
    fetch(tile0, raw_a);
    if (n_t > 1) fetch(tile0 + 1, raw_b);
  }
  // BOXES: lane i of a producer warp holds the table entry of block i of a
  // tile (at most 16 blocks per tile), loaded two tiles ahead.
  const int bpt = TK / bs;  // blocks per tile
  auto fetch_box = [&](int tile) -> int {
    const int bi = tile * bpt + lane;
    int e = 0;
    if (lane < bpt && bi * bs < Lb) {
      const long long ti = static_cast<long long>(b) * max_blocks + bi;
      e = in_range(ti, 1, static_cast<long long>(B) * max_blocks, err) ? block_table[ti] : -1;
    }
    return e;
  };
  int box_a = 0, box_b = 0;
  if (LOAD == BOXES && warp <= 1) {
    box_a = fetch_box(tile0);
    if (n_t > 1) box_b = fetch_box(tile0 + 1);
  }

  uint8_t* sK = smem + L::K_OFF;
  uint8_t* sV = smem + L::V_OFF;
  uint8_t* sQ = smem + L::Q_OFF;
  uint8_t* sP = smem + L::P_OFF;
  float* red = reinterpret_cast<float*>(smem + L::RED_OFF);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;            // [KST]
  uint64_t* k_empty = k_full + KST;       // [KST]
  uint64_t* v_full = k_empty + KST;       // [VST]
  uint64_t* v_empty = v_full + VST;       // [VST]
  uint64_t* s_full = v_empty + VST;       // [2]
  uint64_t* p_full = s_full + 2;          // [PB]
  uint64_t* p_empty = p_full + PB;        // [PB]
  uint64_t* o_done = p_empty + PB;
  uint64_t* final_bar = o_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::TMEM_SLOT_OFF);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    // Gathered tiles: one arrival per producer lane once its copies landed.
    for (int i = 0; i < KST; ++i) {
      mbar_init(&k_full[i], GATHERED ? 32 : 1);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < VST; ++i) {
      mbar_init(&v_full[i], GATHERED ? 32 : 1);
      mbar_init(&v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) mbar_init(&s_full[i], 1);
    for (int i = 0; i < PB; ++i) {
      mbar_init(&p_full[i], 4);
      mbar_init(&p_empty[i], 1);
    }
    mbar_init(o_done, 1);
    mbar_init(final_bar, 1);
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, 64);  // Sᵀ buffers at columns 0 and 16, Oᵀ at 32
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // Loads of one 128-key tile of the cache: one box per cache block, lane i
  // of the producer warp issuing block i's box from its table entry `e`
  // (after lane 0 set the barrier's byte count).
  auto load_tile = [&](const CUtensorMap* map, uint8_t* dst, uint64_t* bar, int tile, int e, int bytes) {
    const int bi = tile * bpt + lane;
    int z = num_blocks * Hkv;  // out of range: the box reads zeros
    if (lane < bpt && bi * bs < Lb) {
      if (e >= 0 && e < num_blocks) z = e * Hkv + hk;
      else atomicExch(err, DEV_BAD_INDEX);
    }
    if (lane == 0) mbar_arrive_expect_tx(bar, bytes);
    __syncwarp();
    if (lane < bpt)
      for (int p = 0; p < L::KPANELS; ++p) tma_load_3d(dst + p * L::PANEL + lane * bs * 128, map, bar, p * 64, 0, z);
  };

  // The same tile by per-token copies, run by a whole warp. resolve() turns
  // fetched table entries of rows lane, lane + 32, lane + 64 and lane + 96
  // into cache row indices (token rows of d elements; NO_ROW past the
  // context or for a bad block index, zero fill); copy_tile() then moves
  // chunk c (16 bytes) of row r into the 128-byte-swizzled K-major layout
  // the products read: panel c / 8, at 128 r + 16 ((c mod 8) xor (r mod 8)).
  constexpr uint32_t NO_ROW = 0xffffffffu;  // the host keeps the cache below 2^32 - 1 rows
  const long long cache_elems = static_cast<long long>(num_blocks) * Hkv * bs * D;
  auto row_of = [&](int blk, int t, int bi) -> uint32_t {
    return (static_cast<uint32_t>(blk) * static_cast<uint32_t>(Hkv) + static_cast<uint32_t>(hk)) *
               static_cast<uint32_t>(bs) + static_cast<uint32_t>(t - bi * bs);
  };
  auto resolve = [&](int tile, const int (&raw)[4], uint32_t (&rows)[4]) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int t = tile * TK + lane + 32 * u;
      uint32_t row = NO_ROW;
      if (t < Lb) {
        const int blk = raw[u], bi = t / bs;
        if (blk >= 0 && blk < num_blocks)
          row = row_of(blk, t, bi);
        else
          atomicExch(err, DEV_BAD_INDEX);
      }
      rows[u] = row;
    }
  };
  // GATHER: the same rows with the entries loaded on the spot. (The two
  // forms stay apart: GATHER written as fetch() + resolve() measured 5%
  // slower at block sizes 12 to 48; its producer's instructions per tile
  // count there.)
  auto lookup = [&](int tile, uint32_t (&rows)[4]) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int t = tile * TK + lane + 32 * u;
      uint32_t row = NO_ROW;
      if (t < Lb) {
        const int bi = t / bs;
        const long long ti = static_cast<long long>(b) * max_blocks + bi;
        const int blk = in_range(ti, 1, static_cast<long long>(B) * max_blocks, err) ? block_table[ti] : -1;
        if (blk >= 0 && blk < num_blocks)
          row = row_of(blk, t, bi);
        else
          atomicExch(err, DEV_BAD_INDEX);
      }
      rows[u] = row;
    }
  };
  // Lane (c, rsub) copies chunk c of rows r = 32 u + r0 + RPI k + rsub. The
  // chunk's swizzled slot depends on r mod 8 = (RPI k + rsub) mod 8 only, so
  // the NX slots are computed once, and a copy costs a shuffle of the row
  // index, one multiply-add for the address and the copy itself.
  auto copy_tile = [&](const __nv_bfloat16* cache, uint8_t* dst, const uint32_t (&rows)[4]) {
    constexpr int CH = D / 8;     // 16-byte chunks per row
    constexpr int RPI = 32 / CH;  // rows per warp instruction
    constexpr int NX = 8 / RPI;   // warp instructions per 8-row swizzle period
    const int c = lane % CH, rsub = lane / CH;
    const char* src_lane = reinterpret_cast<const char*>(cache) + c * 16;
    uint8_t* dst_lane = dst + (c >> 3) * L::PANEL + rsub * 128;
    uint32_t slot[NX];
#pragma unroll
    for (int k = 0; k < NX; ++k) slot[k] = static_cast<uint32_t>(((c & 7) ^ ((k * RPI + rsub) & 7)) << 4);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
#pragma unroll 2
      for (int r0 = 0; r0 < 32; r0 += 8) {
#pragma unroll
        for (int k = 0; k < NX; ++k) {
          const int r1 = r0 + k * RPI;
          const uint32_t row = __shfl_sync(0xffffffffu, rows[u], r1 + rsub);
          const bool live = row != NO_ROW && in_range(static_cast<long long>(row) * D + c * 8, 8, cache_elems, err);
          const char* src = src_lane + static_cast<size_t>(live ? row : 0u) * (D * 2);
          cp_async_16(dst_lane + (32 * u + r1) * 128 + slot[k], src, live ? 16u : 0u);
        }
      }
    }
  };
  // Producer loop of the gathered path (NST stages; the whole warp). Each
  // lane's copies arrive on the tile's full barrier when they land (32
  // arrivals), so the lanes go straight on to the next tile's lookups; the
  // issuer fences the async proxy after its wait.
  auto gather_loop = [&](const __nv_bfloat16* cache, uint8_t* base, int stage_bytes, uint64_t* full,
                         uint64_t* empty, auto nst_c) {
    constexpr int NST = decltype(nst_c)::value;
    uint32_t cur[4], nxt[4] = {NO_ROW, NO_ROW, NO_ROW, NO_ROW};
    if (AHEAD)
      resolve(tile0, raw_a, cur);
    else
      lookup(tile0, cur);
    for (int j = 0; j < n_t; ++j) {
      const int st = j % NST;
      if (!mbar_wait_warp(&empty[st], ((j / NST) & 1) ^ 1, err)) break;
      copy_tile(cache, base + st * stage_bytes, cur);
      cp_async_arrive_noinc(&full[st]);
      if (AHEAD) {
        if (j + 1 < n_t) resolve(tile0 + j + 1, raw_b, cur);
        if (j + 2 < n_t) fetch(tile0 + j + 2, raw_b);
      } else {
        if (j + 1 < n_t) lookup(tile0 + j + 1, nxt);
#pragma unroll
        for (int u = 0; u < 4; ++u) cur[u] = nxt[u];
      }
    }
    cp_async_commit();
    cp_async_wait<0>();  // nothing may land after the CTA exits
  };

  if (GATHERED && warp <= 1) {
    // ------------------------------------ K (warp 0) and V (warp 1) producers
    if (warp == 0 && lane == 0) {
      prefetch_tmap(&tq);
      mbar_arrive_expect_tx(q_full, L::KPANELS * L::QPANEL);
      for (int p = 0; p < L::KPANELS; ++p) tma_load_3d(sQ + p * L::QPANEL, &tq, q_full, p * 64, head0, 0);
    }
    __syncwarp();
    if (warp == 0)
      gather_loop(kc, sK, L::K_TILE, k_full, k_empty, std::integral_constant<int, KST>{});
    else
      gather_loop(vc, sV, L::V_TILE, v_full, v_empty, std::integral_constant<int, VST>{});
    if (warp == 0 && lane == 0) mbar_wait(q_full, 0, err);
  } else if (warp == 0) {
    // --------------------------------------------------------- K producer
    if (lane == 0) {
      prefetch_tmap(&tq);
      prefetch_tmap(&tk);
      mbar_arrive_expect_tx(q_full, L::KPANELS * L::QPANEL);
      for (int p = 0; p < L::KPANELS; ++p) tma_load_3d(sQ + p * L::QPANEL, &tq, q_full, p * 64, head0, 0);
    }
    __syncwarp();
    int issued = 0, cur = box_a;
    for (int j = 0; j < n_t; ++j) {
      const int st = j % KST;
      if (!mbar_wait_warp(&k_empty[st], ((j / KST) & 1) ^ 1, err)) break;
      load_tile(&tk, sK + st * L::K_TILE, &k_full[st], tile0 + j, cur, L::K_TILE);
      issued = j + 1;
      cur = box_b;
      if (j + 2 < n_t) box_b = fetch_box(tile0 + j + 2);
    }
    if (lane == 0) {
      mbar_wait(q_full, 0, err);
      for (int j = max(0, issued - KST); j < issued; ++j) mbar_wait(&k_full[j % KST], (j / KST) & 1, err);
    }
  } else if (warp == 1) {
    // --------------------------------------------------------- V producer
    if (lane == 0) prefetch_tmap(&tv);
    __syncwarp();
    int issued = 0, cur = box_a;
    for (int j = 0; j < n_t; ++j) {
      const int st = j % VST;
      if (!mbar_wait_warp(&v_empty[st], ((j / VST) & 1) ^ 1, err)) break;
      load_tile(&tv, sV + st * L::V_TILE, &v_full[st], tile0 + j, cur, L::K_TILE);  // the real panels of the V tile
      issued = j + 1;
      cur = box_b;
      if (j + 2 < n_t) box_b = fetch_box(tile0 + j + 2);
    }
    if (lane == 0)
      for (int j = max(0, issued - VST); j < issued; ++j) mbar_wait(&v_full[j % VST], (j / VST) & 1, err);
  } else if (warp == 2) {
    // ---------------------------------------------------------- MMA issuer
    constexpr uint32_t idesc_s = idesc_bf16(TK, NH, false, false);  // A = K (K-major), B = Q (K-major)
    constexpr uint32_t idesc_o = idesc_bf16(128, NH, true, false);  // A = Vᵀ (MN-major, M = 128), B = Pᵀ (K-major)
    const uint64_t dq = sdesc_kmajor(smem_u32(sQ), 0);
    // Sᵀ_j = K_j Qᵀ into TMEM buffer j % 2. Issued one tile ahead of O: its
    // buffer's previous reader (the softmax of tile j - 2) released it before
    // P_{j-2}, which O_{j-2}, issued earlier, waited for.
    auto issue_s = [&](int j) -> bool {
      const int st = j % KST;
      if (!mbar_wait_warp(&k_full[st], (j / KST) & 1, err)) return false;
      tc_fence_after();
      if (GATHERED) fence_async_smem();  // the lanes' copies, for the tensor core
      const uint64_t dk = sdesc_kmajor(smem_u32(sK + st * L::K_TILE), 0);
      if (elect_one()) {
#pragma unroll
        for (int k16 = 0; k16 < D / 16; ++k16)
          mma_ss(tmem + (j & 1) * NH, desc_add(dk, kmajor_step(k16, L::PANEL)),
                 desc_add(dq, kmajor_step(k16, L::QPANEL)), idesc_s, k16 > 0);
        tc_commit(&s_full[j & 1]);
        tc_commit(&k_empty[st]);
      }
      __syncwarp();
      return true;
    };
    bool ok = mbar_wait_warp(q_full, 0, err) && issue_s(0);
    for (int j = 0; j < n_t && ok; ++j) {
      const int vs = j % VST, pb = j % PB;
      // The next tile's scores first, so its softmax can run while V_j lands.
      if (j + 1 < n_t && !issue_s(j + 1)) {
        ok = false;
        break;
      }
      ok = mbar_wait_warp(&v_full[vs], (j / VST) & 1, err) && mbar_wait_warp(&p_full[pb], (j / PB) & 1, err);
      if (!ok) break;
      tc_fence_after();
      if (GATHERED) fence_async_smem();
      const uint64_t dv = sdesc_mnmajor(smem_u32(sV + vs * L::V_TILE), 0, L::PANEL);
      const uint64_t dp = sdesc_kmajor(smem_u32(sP + pb * 2 * L::QPANEL), 0);
      if (elect_one()) {
#pragma unroll
        for (int k16 = 0; k16 < TK / 16; ++k16)
          mma_ss(tmem + 32, desc_add(dv, mnmajor_step(k16)), desc_add(dp, kmajor_step(k16, L::QPANEL)), idesc_o,
                 (j > 0 || k16 > 0) ? 1u : 0u);
        tc_commit(&v_empty[vs]);
        tc_commit(&p_empty[pb]);
        tc_commit(o_done);
      }
      __syncwarp();
    }
    if (elect_one()) tc_commit(final_bar);
    __syncwarp();
    mbar_wait_warp(final_bar, 0, err);
  } else {
    // ------------------------------------------------------ softmax (3..6)
    const int quarter = warp & 3;          // TMEM lanes 32*quarter .. +31
    const int r = quarter * 32 + lane;     // key of the tile in Sᵀ, dimension in Oᵀ
    const int wi = warp - 3;               // 0..3, index into the reduction scratch
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    // Pᵀ rows of padded heads (h >= G) are zero in both buffers for good;
    // at d = 64 so is the second panel of every V stage.
    for (int i = r; i < PB * 2 * NH * 64; i += 128) {
      const int h = (i / 64) % NH;
      if (h >= G) reinterpret_cast<uint16_t*>(sP)[i] = 0;
    }
    if (D == 64)
      for (int st = 0; st < VST; ++st)
        for (int i = r; i < L::PANEL / 16; i += 128)
          reinterpret_cast<uint4*>(sV + st * L::V_TILE + L::PANEL)[i] = make_uint4(0u, 0u, 0u, 0u);
    float m[GM], l[GM];
#pragma unroll
    for (int h = 0; h < GM; ++h) {
      m[h] = -INFINITY;
      l[h] = 0.f;
    }
    bool ok = true;
    for (int j = 0; j < n_t; ++j) {
      const int sb = j & 1, pb = j % PB;
      if (ok) ok = mbar_wait(&s_full[sb], (j >> 1) & 1, err);
      if (named_bar_any(1, 128, !ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t raw[16];
      tmem_ld16(tmem + lane_addr + sb * NH, raw);
      tmem_ld_wait();
      const bool live = (tile0 + j) * TK + r < t_end;
      float x[GM];
      bool need = false;
#pragma unroll
      for (int h = 0; h < GM; ++h) {
        x[h] = live && h < G ? __uint_as_float(raw[h]) * scale_log2 : -INFINITY;
        need |= x[h] > m[h] + RESCALE_LOG2;
      }
      if (named_bar_any(1, 128, need)) {
        // Raise every head's reference to its exact maximum so far.
#pragma unroll
        for (int h = 0; h < GM; ++h) {
          float v = x[h];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
          if (lane == 0) red[wi * NH + h] = v;
        }
        named_bar_sync(1, 128);
        float alpha[GM];
#pragma unroll
        for (int h = 0; h < GM; ++h) {
          const float tmax = fmaxf(fmaxf(red[h], red[NH + h]), fmaxf(red[2 * NH + h], red[3 * NH + h]));
          const float m_new = fmaxf(m[h], tmax);
          alpha[h] = m_new == -INFINITY ? 1.f : ex2(m[h] - m_new);  // 0 on a head's first key
          m[h] = m_new;
          l[h] *= alpha[h];
        }
        named_bar_sync(1, 128);  // the scratch is read before anyone rewrites it
        if (j > 0) {
          // Oᵀ columns *= alpha once O_{j-1} has landed (O_j accumulates into
          // it). When S_j completed, O_{j-2} had (it was issued before S_j), so
          // o_done is at most one phase behind and the parity wait is exact.
          ok = mbar_wait(o_done, (j - 1) & 1, err);
          tc_fence_after();
          if (ok) {
            uint32_t o[16];
            tmem_ld16(tmem + lane_addr + 32, o);
            tmem_ld_wait();
#pragma unroll
            for (int h = 0; h < GM; ++h) o[h] = __float_as_uint(__uint_as_float(o[h]) * alpha[h]);
            tmem_st16(tmem + lane_addr + 32, o);
          }
        }
      }
      // P_j (bf16) into Pᵀ buffer j % PB once O_{j-PB} has read it.
      if (ok) ok = mbar_wait(&p_empty[pb], ((j / PB) & 1) ^ 1, err);
      uint8_t* pbuf = sP + pb * 2 * L::QPANEL + (r / 64) * L::QPANEL;
#pragma unroll
      for (int h = 0; h < GM; ++h) {
        if (h >= G) break;
        const float pv = ex2(x[h] - m[h]);  // x = -inf (masked) gives 0
        l[h] += pv;
        const int off = h * 128 + ((((r % 64) >> 3) ^ (h & 7)) << 4) + (r & 7) * 2;
        if (in_range((r / 64) * L::QPANEL + off, 2, 2 * L::QPANEL, err))
          *reinterpret_cast<__nv_bfloat16*>(pbuf + off) = __float2bfloat16_rn(pv);
      }
      fence_async_smem();
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[pb]);
    }
    // ------------------------------------------------------------ epilogue
    // Wait for the issuer's final commit, not for o_done: with the scores
    // issued a tile ahead the softmax can finish its last tile while o_done
    // is two phases behind, and a parity wait would then match an earlier
    // completed phase. The final barrier has one phase only.
    if (ok) ok = mbar_wait(final_bar, 0, err);
    if (!named_bar_any(1, 128, !ok)) {
      tc_fence_after();
      // Every thread's partial denominators, summed per head.
#pragma unroll
      for (int h = 0; h < GM; ++h) {
        float v = l[h];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) red[wi * NH + h] = v;
      }
      named_bar_sync(1, 128);
      uint32_t o[16];
      tmem_ld16(tmem + lane_addr + 32, o);
      tmem_ld_wait();
#pragma unroll
      for (int h = 0; h < GM; ++h) {
        if (h >= G) break;
        const float lh = (red[h] + red[NH + h]) + (red[2 * NH + h] + red[3 * NH + h]);
        const long long orow = prow + h;
        // One split: this is the final row (o in bf16), and no merge runs.
        const float ov = __uint_as_float(o[h]) / lh, lv = (m[h] + __log2f(lh)) * dec::LN2;
        if (r < D && in_range(orow * D + r, 1, part_rows * D, err)) {
          if (S == 1) o_out[orow * D + r] = __float2bfloat16_rn(ov);
          else o_part[orow * D + r] = ov;
        }
        if (r == 0 && in_range(orow, 1, part_rows, err)) (S == 1 ? lse_out : lse_part)[orow] = lv;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 64);
  }
}

// TMA boxes serve a block size that is a multiple of 8 dividing 128 (each box
// lands on whole 1024-byte swizzle groups); other sizes gather per token.
inline bool boxes(int bs) { return bs % 8 == 0 && TK % bs == 0; }

// Output pointers of every launcher: o_part, lse_part take the split results
// (S > 1, merged afterwards); o_out, lse_out the final rows (S = 1).
struct Out {
  float* o_part;
  float* lse_part;
  __nv_bfloat16* o;
  float* lse;
};

template <int D, int GM, int LOAD>
static cudaError_t launch_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const void* kc,
                            const void* vc, const int* table, const int* seq_lens, const Out& out, int B, int H,
                            int Hkv, int num_blocks, int bs, int max_blocks, float scale, int S, cudaStream_t stream) {
  using C = Cfg<GM>;
  const int smem = Smem<D, C::KST, C::VST, C::PB>::ALLOC;
  auto kern = decode_mma_kernel<D, GM, LOAD>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int n_chunk = (H / Hkv + NH - 1) / NH;
  const dim3 grid(static_cast<unsigned>(S), static_cast<unsigned>(Hkv * n_chunk), static_cast<unsigned>(B));
  kern<<<grid, THREADS, smem, stream>>>(tq, tk, tv, static_cast<const __nv_bfloat16*>(kc),
                                        static_cast<const __nv_bfloat16*>(vc), table, seq_lens, out.o_part,
                                        out.lse_part, out.o, out.lse, B, H, Hkv, num_blocks, bs, max_blocks,
                                        scale * dec::LOG2E);
  return cudaGetLastError();
}

template <int D, int GM>
static cudaError_t launch_g(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const void* kc,
                            const void* vc, const int* table, const int* seq_lens, const Out& out, int B, int H,
                            int Hkv, int num_blocks, int bs, int max_blocks, float scale, int S, cudaStream_t stream) {
  if (boxes(bs))
    return launch_t<D, GM, BOXES>(tq, tk, tv, kc, vc, table, seq_lens, out, B, H, Hkv, num_blocks, bs, max_blocks,
                                  scale, S, stream);
  if (bs < 8)
    return launch_t<D, GM, GATHER_AHEAD>(tq, tk, tv, kc, vc, table, seq_lens, out, B, H, Hkv, num_blocks, bs,
                                         max_blocks, scale, S, stream);
  return launch_t<D, GM, GATHER>(tq, tk, tv, kc, vc, table, seq_lens, out, B, H, Hkv, num_blocks, bs, max_blocks,
                                 scale, S, stream);
}

template <int D>
static cudaError_t launch_d(const void* q, const void* kc, const void* vc, const int* table, const int* seq_lens,
                            const Out& out, int B, int H, int Hkv, int num_blocks, int bs, int max_blocks, float scale,
                            int S, cudaStream_t stream) {
  CUtensorMap tq, tk, tv;
  if (!make_tmap_bf16(&tq, q, 1, B * H, D, NH)) return cudaErrorInvalidValue;
  if (boxes(bs)) {
    if (!make_tmap_bf16(&tk, kc, num_blocks * Hkv, bs, D, bs) || !make_tmap_bf16(&tv, vc, num_blocks * Hkv, bs, D, bs))
      return cudaErrorInvalidValue;
  } else {
    tk = tq;  // unused: the gathered path reads the caches directly
    tv = tq;
  }
  const int G = H / Hkv;  // query heads per K/V head; CTAs take them 16 at a time
  if (G <= 4)
    return launch_g<D, 4>(tq, tk, tv, kc, vc, table, seq_lens, out, B, H, Hkv, num_blocks, bs, max_blocks, scale, S,
                          stream);
  if (G <= 8)
    return launch_g<D, 8>(tq, tk, tv, kc, vc, table, seq_lens, out, B, H, Hkv, num_blocks, bs, max_blocks, scale, S,
                          stream);
  return launch_g<D, 16>(tq, tk, tv, kc, vc, table, seq_lens, out, B, H, Hkv, num_blocks, bs, max_blocks, scale, S,
                         stream);
}

static cudaError_t launch(const void* q, const void* kc, const void* vc, const int* table, const int* seq_lens,
                          const Out& out, int B, int H, int Hkv, int d, int num_blocks, int bs, int max_blocks,
                          float scale, int S, cudaStream_t stream) {
  return d == 64 ? launch_d<64>(q, kc, vc, table, seq_lens, out, B, H, Hkv, num_blocks, bs, max_blocks, scale, S,
                                stream)
                 : launch_d<128>(q, kc, vc, table, seq_lens, out, B, H, Hkv, num_blocks, bs, max_blocks, scale, S,
                                 stream);
}

// Shapes this kernel serves (any block size).
inline bool serves(int d, int bs) { return (d == 64 || d == 128) && bs >= 1; }

}  // namespace decmma

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
  if (!decmma::serves(d, block_size)) return cudaErrorInvalidValue;
  const decmma::Out out{o_part, lse_part, static_cast<__nv_bfloat16*>(o), lse};
  cudaError_t e = decmma::launch(q, k_cache, v_cache, block_table, seq_lens, out, B, H, Hkv, d, num_blocks,
                                 block_size, max_blocks, scale, S, stream);
  if (e != cudaSuccess || S == 1) return e;  // one split: the kernel wrote o and lse
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
