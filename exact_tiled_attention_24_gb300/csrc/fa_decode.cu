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
//                   byte is read once per step (G > 16: one CTA per 16 of
//                   them, each reading the K/V head). 64-key tiles of K and V are
//                   copied into shared memory by bulk copies (one per run of
//                   consecutive tokens inside a cache block), three tiles in
//                   flight. Each warp owns 8 keys of every tile and keeps
//                   its own running (m, l) and fp32 output rows; the warps'
//                   states are merged once at the end. Writes o_s (fp32)
//                   and lse_s per head.
//   merge           one warp per output row: the combination above.
// The work per byte is a few FMAs (G·d per key and head pair), far below the
// tensor-core ridge, so the products run on the FMA pipe.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "fa_common.h"
#include "fa_ptx.cuh"
#include "fa_tmap.h"

namespace fa {

static __device__ uint32_t g_dec_err;

namespace dec {

constexpr int THREADS = 256;
constexpr int TK = 64;  // keys per tile
// Stages of the K/V ring. Two CTAs per SM with three 32 KB stages each keep
// ~128 KB of loads in flight per SM, what HBM latency under load needs.
constexpr int NST = 3;
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.69314718055994531f;

template <int D, int GM>
struct Smem {
  static constexpr int WARPS = THREADS / 32;
  static constexpr int ROW = D * 2;             // bytes of one key (or value) row
  static constexpr int TILE = TK * ROW;         // one K or V tile
  // Each warp streams its own 8 keys of every tile: stage st of warp w holds
  // their K rows then their V rows (after the loop, the stages hold the
  // warps' partial output rows).
  static constexpr int WSLOT = 2 * 8 * ROW;
  static constexpr int SLOT_OFF = 0;
  static constexpr int Q_OFF = NST * WARPS * WSLOT;  // q rows fp32 [GM][D], times scale·log2 e
  // Per-warp scratch: the scores, then the (p, p) pairs, of its 8 keys x 4
  // heads (64 floats), then the 4 heads' rescale factors.
  static constexpr int W_OFF = Q_OFF + GM * D * 4;
  static constexpr int W_BYTES = (8 * 4 * 2 + 4) * 4;
  static constexpr int ML_OFF = W_OFF + WARPS * W_BYTES;  // per-warp (m, l) per head: [WARPS][2][GM]
  static constexpr int TAB_OFF = ML_OFF + WARPS * 2 * GM * 4;  // block-table slice, int32
  static constexpr int BAR_OFF = TAB_OFF + kDecodeMaxTable * 4;
  // full[NST][WARPS] mbarriers, then fills so far per (stage, warp)
  static constexpr int CNT_OFF = BAR_OFF + NST * WARPS * 8;
  static constexpr int BYTES = CNT_OFF + NST * WARPS * 4 + 16;
  static_assert(WARPS * GM * D * 4 <= NST * WARPS * WSLOT, "the warps' partial rows must fit the idle stages");
};

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Two fp32 multiply-adds in one instruction: d = a * b + c, element-wise.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(*reinterpret_cast<unsigned long long*>(&d))
      : "l"(*reinterpret_cast<const unsigned long long*>(&a)),
        "l"(*reinterpret_cast<const unsigned long long*>(&b)),
        "l"(*reinterpret_cast<const unsigned long long*>(&c)));
  return d;
}

// bf16 pair (low half = first element) -> two floats, exactly.
__device__ __forceinline__ float2 bf2_to_f2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// Each warp owns keys 8w .. 8w + 7 of every tile: it streams their K and V
// rows through its own NST-slot ring (own mbarriers, refilled by itself as
// soon as it has read a slot) and keeps its own running (m, l) and output
// rows for the G heads. The warps never wait for one another inside the
// tile loop; their states are merged at the end with the same rescaling as
// the split merge. Two CTAs share an SM (the ring depth above assumes it),
// so the kernel is held to 128 registers a thread, except with 16 heads of
// 128 columns, whose accumulators would then spill.
template <int D, int GM>
__global__ void __launch_bounds__(THREADS, D * GM > 1024 ? 1 : 2) decode_partial_kernel(
    const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k_cache,
    const __nv_bfloat16* __restrict__ v_cache, const int* __restrict__ block_table,
    const int* __restrict__ seq_lens, float* __restrict__ o_part, float* __restrict__ lse_part, int B,
    int H, int Hkv, int num_blocks, int bs, int max_blocks, float scale_log2) {
  using L = Smem<D, GM>;
  constexpr int WARPS = L::WARPS;
  constexpr int CPL = D / 32;  // output columns per lane
  extern __shared__ __align__(1024) uint8_t smem[];
  const int S = gridDim.x;
  // blockIdx.y = (K/V head, chunk of at most 16 of its query heads)
  const int G_all = H / Hkv;
  const int n_chunk = (G_all + 15) / 16;
  const int s = blockIdx.x, hk = blockIdx.y / n_chunk, chunk = blockIdx.y % n_chunk, b = blockIdx.z;
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int G = min(16, G_all - 16 * chunk);  // query heads served by this CTA
  uint32_t* err = &g_dec_err;

  // Context of request b, clamped to what its block-table row can address.
  int Lb = in_range(b, 1, B, err) ? seq_lens[b] : 0;
  Lb = Lb < 0 ? 0 : (Lb > max_blocks * bs ? max_blocks * bs : Lb);
  const int n_tiles = (Lb + TK - 1) / TK;
  const int tps = (n_tiles + S - 1) / S;  // tiles per split
  const int tile0 = s * tps;
  const int tile1 = min(n_tiles, tile0 + tps);
  const size_t head0 = static_cast<size_t>(b) * H + static_cast<size_t>(hk) * G_all + 16 * chunk;  // first query head
  const size_t prow = static_cast<size_t>(s) * B * H + head0;                     // its partial row
  const long long part_rows = static_cast<long long>(S) * B * H;  // rows of o_part and lse_part
  if (tile0 >= tile1) {  // no key in this split: o_s = 0, lse_s = -inf (weight 0 in the merge)
    for (int i = tid; i < G * D; i += THREADS)
      if (in_range(static_cast<long long>(prow) * D + i, 1, part_rows * D, err)) o_part[prow * D + i] = 0.f;
    if (tid < G && in_range(static_cast<long long>(prow) + tid, 1, part_rows, err)) lse_part[prow + tid] = -INFINITY;
    return;
  }
  const int t_begin = tile0 * TK, t_end = min(Lb, tile1 * TK);
  const int blk0 = t_begin / bs;
  const int nblk = (t_end - 1) / bs + 1 - blk0;  // <= kDecodeMaxTable (checked on the host)

  uint8_t* sSlot = smem + L::SLOT_OFF + warp * L::WSLOT;  // this warp's slot of stage 0
  float* sQ = reinterpret_cast<float*>(smem + L::Q_OFF);
  float* sW = reinterpret_cast<float*>(smem + L::W_OFF + warp * L::W_BYTES);
  float* sML = reinterpret_cast<float*>(smem + L::ML_OFF);
  int* sTab = reinterpret_cast<int*>(smem + L::TAB_OFF);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF) + warp;  // [st * WARPS]
  int* fills = reinterpret_cast<int*>(smem + L::CNT_OFF) + warp;           // [st * WARPS]

  for (int i = tid; i < GM * D; i += THREADS) {
    const int g = i / D;
    const long long qi = static_cast<long long>(head0 + g) * D + (i % D);
    sQ[i] = g < G && in_range(qi, 1, static_cast<long long>(B) * H * D, err)
                ? __bfloat162float(q[qi]) * scale_log2
                : 0.f;
  }
  for (int i = tid; i < nblk; i += THREADS) {
    const long long ti = static_cast<long long>(b) * max_blocks + blk0 + i;
    if (in_range(i, 1, kDecodeMaxTable, err))
      sTab[i] = in_range(ti, 1, static_cast<long long>(B) * max_blocks, err) ? block_table[ti] : -1;
  }
  if (lane == 0) {
    for (int st = 0; st < NST; ++st) {
      fills[st * WARPS] = 0;
      mbar_init(&full[st * WARPS], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();

  // One warp: copy its 8 keys of tile `tile` (K rows, then V rows) into its
  // slot of stage st. Lane r takes the r-th run of consecutive tokens inside
  // one cache block. Entries outside [0, num_blocks) are never dereferenced:
  // their copies are skipped and the error is reported, and their rows of the
  // slot keep stale bytes, so the results of that request are undefined.
  // Only copied bytes are expected on the barrier.
  const bool single_run = (bs & 7) == 0;  // a warp's 8 keys never cross a block boundary
  const long long cache_elems = static_cast<long long>(num_blocks) * Hkv * bs * D;
  // Table entry blk may be read for rows [row0, row0 + nrows) of head hk.
  auto copy_ok = [&](int blk, int row0, int nrows) {
    return blk >= 0 && blk < num_blocks &&
           in_range((static_cast<long long>(blk) * Hkv + hk) * bs * D + static_cast<long long>(row0) * D,
                    static_cast<long long>(nrows) * D, cache_elems, err);
  };
  auto issue = [&](int tile, int st) {
    const int t0 = tile * TK + warp * 8, t1 = min(t_end, t0 + 8);
    if (single_run) {  // lane 0 alone: one table entry, two copies
      if (lane == 0) {
        ++fills[st * WARPS];
        uint32_t nbytes = 0;
        int blk = -1, off = 0;
        if (t0 < t1) {
          const int bi = t0 / bs;  // the only division per tile
          off = t0 - bi * bs;
          blk = in_range(bi - blk0, 1, nblk, err) ? sTab[bi - blk0] : -1;
          if (copy_ok(blk, off, t1 - t0)) nbytes = static_cast<uint32_t>(t1 - t0) * L::ROW;
          else atomicExch(err, DEV_BAD_INDEX);
        }
        mbar_arrive_expect_tx(&full[st * WARPS], 2 * nbytes);
        if (nbytes) {
          uint8_t* slot = sSlot + st * WARPS * L::WSLOT;
          const size_t src = ((static_cast<size_t>(blk) * Hkv + hk) * bs + off) * D;
          bulk_load(slot, k_cache + src, nbytes, &full[st * WARPS]);
          bulk_load(slot + 8 * L::ROW, v_cache + src, nbytes, &full[st * WARPS]);
        }
      }
      __syncwarp();
      return;
    }
    const int b0 = t0 / bs;  // the only division per tile
    const int nrun = t0 < t1 ? (t1 - 1) / bs - b0 + 1 : 0;
    uint32_t bytes = 0;
    for (int r = lane; r < nrun; r += 32) {
      const int blk = in_range(b0 + r - blk0, 1, nblk, err) ? sTab[b0 + r - blk0] : -1;
      const int rs = max(t0, (b0 + r) * bs), re = min(t1, (b0 + r + 1) * bs);
      if (copy_ok(blk, rs - (b0 + r) * bs, re - rs)) bytes += static_cast<uint32_t>(re - rs) * L::ROW;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) bytes += __shfl_xor_sync(0xffffffffu, bytes, o);
    if (lane == 0) {
      ++fills[st * WARPS];
      mbar_arrive_expect_tx(&full[st * WARPS], 2 * bytes);
    }
    __syncwarp();
    uint8_t* slot = sSlot + st * WARPS * L::WSLOT;
    for (int r = lane; r < nrun; r += 32) {
      const int blk = in_range(b0 + r - blk0, 1, nblk, err) ? sTab[b0 + r - blk0] : -1;
      const int rs = max(t0, (b0 + r) * bs), re = min(t1, (b0 + r + 1) * bs);
      if (copy_ok(blk, rs - (b0 + r) * bs, re - rs)) {
        const size_t src = ((static_cast<size_t>(blk) * Hkv + hk) * bs + (rs - (b0 + r) * bs)) * D;
        const uint32_t dst = static_cast<uint32_t>(rs - t0) * L::ROW;
        const uint32_t nbytes = static_cast<uint32_t>(re - rs) * L::ROW;
        bulk_load(slot + dst, k_cache + src, nbytes, &full[st * WARPS]);
        bulk_load(slot + 8 * L::ROW + dst, v_cache + src, nbytes, &full[st * WARPS]);
      } else {
        atomicExch(err, DEV_BAD_INDEX);
      }
    }
  };

  // Scores: 8 lanes per key (lane = 8·kw + dq); lane dq covers the 16-byte
  // chunks dq (and dq + 8 when d = 128) of the row, so the 8 lanes of a load
  // phase hit distinct banks. Four heads at a time; their q slices stay in
  // registers for the whole sweep when G <= 4.
  constexpr int CH = D / 64;
  const int dq = lane & 7, kw = lane >> 3;
  float2 qr[4][CH * 4];
  auto load_q = [&](int hg) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int ch = 0; ch < CH; ++ch) {
        const float* src = sQ + (hg * 4 + j) * D + (dq + 8 * ch) * 8;
#pragma unroll
        for (int i = 0; i < 4; ++i) qr[j][ch * 4 + i] = make_float2(src[2 * i], src[2 * i + 1]);
      }
  };
  if (GM == 4) load_q(0);

  // Per-warp state: lanes 8j .. 8j + 7 hold (m, l) of head 4·hg + j; every
  // lane holds output columns CPL·lane .. + CPL - 1 of every head.
  float m_run[GM / 4], l_run[GM / 4];
#pragma unroll
  for (int hg = 0; hg < GM / 4; ++hg) {
    m_run[hg] = -INFINITY;
    l_run[hg] = 0.f;
  }
  float2 acc[GM][CPL / 2];
#pragma unroll
  for (int g = 0; g < GM; ++g)
#pragma unroll
    for (int c = 0; c < CPL / 2; ++c) acc[g][c] = make_float2(0.f, 0.f);

  // The first NST tiles fill every slot of this warp.
  __syncthreads();  // barrier inits and the table slice are visible
  for (int j = 0; j < NST && tile0 + j < tile1; ++j) issue(tile0 + j, j);
  bool ok = true;
  int it = 0;
  for (int tile = tile0; tile < tile1; ++tile, ++it) {
    const int st = it % NST;
    ok = mbar_wait_warp(&full[st * WARPS], (it / NST) & 1, err);
    if (!ok) break;
    const int nk = min(t_end, (tile + 1) * TK) - tile * TK;
    const uint8_t* kt = sSlot + st * WARPS * L::WSLOT;  // this warp's 8 K rows, then its 8 V rows
    const uint32_t* vt = reinterpret_cast<const uint32_t*>(kt + 8 * L::ROW);
#pragma unroll
    for (int hg = 0; hg < GM / 4; ++hg) {
      if (hg * 4 >= G) continue;  // warp-uniform
      if (GM > 4) load_q(hg);
#pragma unroll
      for (int p = 0; p < 2; ++p) {
        const int kk = p * 4 + kw;  // key within the warp's eight
        const int k = warp * 8 + kk;
        float2 a[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) a[j] = make_float2(0.f, 0.f);
#pragma unroll
        for (int ch = 0; ch < CH; ++ch) {
          const uint4 kv = *reinterpret_cast<const uint4*>(kt + kk * L::ROW + (dq + 8 * ch) * 16);
          const float2 k0 = bf2_to_f2(kv.x), k1 = bf2_to_f2(kv.y), k2 = bf2_to_f2(kv.z), k3 = bf2_to_f2(kv.w);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            a[j] = fma2(k0, qr[j][ch * 4 + 0], a[j]);
            a[j] = fma2(k1, qr[j][ch * 4 + 1], a[j]);
            a[j] = fma2(k2, qr[j][ch * 4 + 2], a[j]);
            a[j] = fma2(k3, qr[j][ch * 4 + 3], a[j]);
          }
        }
        const float s0 = a[0].x + a[0].y, s1 = a[1].x + a[1].y;
        const float s2 = a[2].x + a[2].y, s3 = a[3].x + a[3].y;
        // Reduce-scatter over the key's 8 lanes: 4 shuffles leave lane pair
        // (dq, dq ^ 1) with the full score of head j = 2·bit2 + bit1.
        const bool hi = dq & 4, mid = dq & 2;
        const float t0 = __shfl_xor_sync(0xffffffffu, hi ? s0 : s2, 4);
        const float t1 = __shfl_xor_sync(0xffffffffu, hi ? s1 : s3, 4);
        const float a0 = (hi ? s2 : s0) + t0, a1 = (hi ? s3 : s1) + t1;
        float r = (mid ? a1 : a0) + __shfl_xor_sync(0xffffffffu, mid ? a0 : a1, 2);
        r += __shfl_xor_sync(0xffffffffu, r, 1);
        const int j = (hi ? 2 : 0) + (mid ? 1 : 0);
        // Rows past the context end hold stale bytes: their score is -inf
        // whatever r is.
        if ((dq & 1) == 0) sW[j * 8 + kk] = (k < nk && hg * 4 + j < G) ? r : -INFINITY;
      }
      __syncwarp();
      // Online softmax of the warp's 8 keys: lane = 8j + kk holds head j, key kk.
      float pr, al;
      {
        const int j = lane >> 3;
        const float sc = sW[lane];
        float mx = sc;
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        const float m_new = fmaxf(m_run[hg], mx);
        if (m_new == -INFINITY) {  // no key of this head seen by the warp yet
          pr = 0.f;
          al = 1.f;
        } else {
          pr = ex2(sc - m_new);
          al = ex2(m_run[hg] - m_new);
        }
        float sum = pr;
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        sum += __shfl_xor_sync(0xffffffffu, sum, 4);
        l_run[hg] = l_run[hg] * al + sum;
        m_run[hg] = m_new;
        (void)j;
      }
      __syncwarp();
      // (p, p) pairs, key-major: [kk][head j][2]; alphas of the 4 heads after.
      sW[((lane & 7) * 4 + (lane >> 3)) * 2] = pr;
      sW[((lane & 7) * 4 + (lane >> 3)) * 2 + 1] = pr;
      if ((lane & 7) == 0) sW[64 + (lane >> 3)] = al;
      __syncwarp();
      // Output columns: acc_j = α_j·acc_j + Σ_kk P_j,kk · V_kk[cols].
      {
        const float4 al4 = *reinterpret_cast<const float4*>(sW + 64);
        const float alj[4] = {al4.x, al4.y, al4.z, al4.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
          for (int c = 0; c < CPL / 2; ++c)
            acc[hg * 4 + j][c] = make_float2(acc[hg * 4 + j][c].x * alj[j], acc[hg * 4 + j][c].y * alj[j]);
        auto pv_key = [&](int kk) {
          const uint32_t* vr = vt + kk * (D / 2) + lane * (CPL / 2);
          float2 v[CPL / 2];
#pragma unroll
          for (int c = 0; c < CPL / 2; ++c) v[c] = bf2_to_f2(vr[c]);
          const float4 p01 = *reinterpret_cast<const float4*>(sW + kk * 8);
          const float4 p23 = *reinterpret_cast<const float4*>(sW + kk * 8 + 4);
          const float2 pp[4] = {make_float2(p01.x, p01.y), make_float2(p01.z, p01.w),
                                make_float2(p23.x, p23.y), make_float2(p23.z, p23.w)};
#pragma unroll
          for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int c = 0; c < CPL / 2; ++c) acc[hg * 4 + j][c] = fma2(v[c], pp[j], acc[hg * 4 + j][c]);
        };
        if (warp * 8 + 8 <= nk) {
          // All 8 rows hold copied keys (every tile but a context's last):
          // a branch-free loop whose shared-memory loads can be hoisted.
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) pv_key(kk);
        } else {
          // Rows past the context end were never copied (P is 0 there, and
          // their bytes may be anything): skip them, warp-uniformly.
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            if (warp * 8 + kk >= nk) break;
            pv_key(kk);
          }
        }
      }
      __syncwarp();  // the scratch is rewritten by the next head group
    }
    // This warp has read its slot of stage st: refill it.
    if (tile + NST < tile1) issue(tile + NST, st);
  }
  if (__syncthreads_or(!ok)) {
    // Let copies already issued land before the CTA exits (bounded).
    if (lane == 0)
      for (int st = 0; st < NST; ++st)
        if (fills[st * WARPS] > 0) mbar_wait(&full[st * WARPS], (fills[st * WARPS] - 1) & 1, err);
    return;
  }
  // Merge the warps' states per head: M = max_w m_w, L = Σ_w l_w 2^(m_w − M),
  // o = Σ_w acc_w 2^(m_w − M) / L, lse = (M + log2 L)·ln 2.
  float* sAcc = reinterpret_cast<float*>(smem + L::SLOT_OFF);  // [WARPS][GM][D]; the stages are idle
#pragma unroll
  for (int g = 0; g < GM; ++g)
#pragma unroll
    for (int c = 0; c < CPL / 2; ++c)
      *reinterpret_cast<float2*>(sAcc + (warp * GM + g) * D + lane * CPL + 2 * c) = acc[g][c];
#pragma unroll
  for (int hg = 0; hg < GM / 4; ++hg)
    if ((lane & 7) == 0) {
      sML[(warp * 2 + 0) * GM + hg * 4 + (lane >> 3)] = m_run[hg];
      sML[(warp * 2 + 1) * GM + hg * 4 + (lane >> 3)] = l_run[hg];
    }
  __syncthreads();
  for (int i = tid; i < G * D; i += THREADS) {
    const int g = i / D, c = i % D;
    float M = -INFINITY;
    for (int w = 0; w < WARPS; ++w) M = fmaxf(M, sML[(w * 2) * GM + g]);
    float Ls = 0.f, u = 0.f;
    for (int w = 0; w < WARPS; ++w) {
      const float mw = sML[(w * 2) * GM + g];
      if (mw == -INFINITY) continue;
      const float f = ex2(mw - M);
      Ls += sML[(w * 2 + 1) * GM + g] * f;
      u += sAcc[(w * GM + g) * D + c] * f;
    }
    if (in_range(static_cast<long long>(prow + g) * D + c, 1, part_rows * D, err)) o_part[(prow + g) * D + c] = u / Ls;
    if (c == 0 && in_range(static_cast<long long>(prow) + g, 1, part_rows, err))
      lse_part[prow + g] = (M + __log2f(Ls)) * LN2;
  }
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
    for (int s = 0; s < S; ++s) {
      if (!in_range((s * rows + row) * D + lane * CPL, CPL, prt * D, err)) continue;
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
    if (in_range(row * D + lane * CPL + j, 2, rows * D, err))
      *reinterpret_cast<__nv_bfloat162*>(o + row * D + lane * CPL + j) =
          __floats2bfloat162_rn(acc[j] * inv, acc[j + 1] * inv);
  if (lane == 0 && in_range(row, 1, rows, err)) lse[row] = l > 0.f ? m + __logf(l) : -INFINITY;
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
  const int n_chunk = (H / Hkv + 15) / 16;  // CTAs per K/V head (16 query heads each at most)
  const dim3 grid(static_cast<unsigned>(S), static_cast<unsigned>(Hkv * n_chunk), static_cast<unsigned>(B));
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

// ----------------------------------------------------------------------------
// The same decode step on the tensor cores (d = 64 or 128; cache blocks of
// 8, 16, 32, 64 or 128 tokens).
//
// The FMA-pipe kernel above issues about 140 warp instructions per KB of K/V
// (converting bf16 rows, 8-lane dot products, shuffles), and that instruction
// stream, not HBM, sets its rate. Here both products of a 128-key tile run on
// the tensor core with the tile's keys as M, so the work per key is a few
// instructions of softmax:
//   Sᵀ = K Qᵀ    M = 128 keys, N = 16 query heads (padded), K = d; into TMEM
//   Oᵀ += Vᵀ Pᵀ  M = 128 dims (d = 64: padded by a zero panel), N = 16 heads,
//                K = 128 keys; accumulated in TMEM
// One thread per TMEM lane: lane r is key r of the tile in Sᵀ and dimension r
// in Oᵀ. Each cache block of the tile arrives as its own TMA box (the cache
// viewed as (d, block_size, num_blocks·Hkv)), written at row offset
// block·block_size of the 128-row tile; a block past the context or with a
// table entry outside [0, num_blocks) is requested at an out-of-range
// coordinate, so the box reads zeros and the entry is never dereferenced.
// The softmax keeps one exponent reference per head, raised (and Oᵀ's column
// rescaled) when a key outgrows it by more than 2^8, as in the forward.
// Roles (224 threads): warp 0 loads K tiles (2 stages), warp 1 V tiles
// (1 stage), warp 2 owns TMEM and issues the products, warps 3..6 run the
// softmax and the epilogue. Two CTAs fit an SM.
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

template <int D, int GM>
__global__ void __launch_bounds__(THREADS, Cfg<GM>::CTAS) decode_mma_kernel(
    const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
    const __grid_constant__ CUtensorMap tv, const int* __restrict__ block_table,
    const int* __restrict__ seq_lens, float* __restrict__ o_part, float* __restrict__ lse_part, int B, int H,
    int Hkv, int num_blocks, int bs, int max_blocks, float scale_log2) {
  constexpr int KST = Cfg<GM>::KST, VST = Cfg<GM>::VST, PB = Cfg<GM>::PB;
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
    for (int i = threadIdx.x; i < G * D; i += THREADS)
      if (in_range(prow * D + i, 1, part_rows * D, err)) o_part[prow * D + i] = 0.f;
    if (threadIdx.x < G && in_range(prow + threadIdx.x, 1, part_rows, err)) lse_part[prow + threadIdx.x] = -INFINITY;
    return;
  }
  const int n_t = tile1 - tile0;
  const int t_end = min(Lb, tile1 * TK);  // keys at or past t_end are masked

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
    for (int i = 0; i < KST; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < VST; ++i) {
      mbar_init(&v_full[i], 1);
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

  // Loads of one 128-key tile of the cache: one box per cache block.
  const int bpt = TK / bs;  // blocks per tile
  auto load_tile = [&](const CUtensorMap* map, uint8_t* dst, uint64_t* bar, int tile) {  // D / 64 panels
    const int blk_first = tile * bpt;
    for (int i = 0; i < bpt; ++i) {
      const int bi = blk_first + i;
      int z = num_blocks * Hkv;  // out of range: the box reads zeros
      if (bi * bs < Lb) {
        const long long ti = static_cast<long long>(b) * max_blocks + bi;
        const int blk = in_range(ti, 1, static_cast<long long>(B) * max_blocks, err) ? block_table[ti] : -1;
        if (blk >= 0 && blk < num_blocks) z = blk * Hkv + hk;
        else atomicExch(err, DEV_BAD_INDEX);
      }
      for (int p = 0; p < L::KPANELS; ++p) tma_load_3d(dst + p * L::PANEL + i * bs * 128, map, bar, p * 64, 0, z);
    }
  };

  if (warp == 0) {
    // --------------------------------------------------------- K producer
    if (lane == 0) {
      prefetch_tmap(&tq);
      prefetch_tmap(&tk);
      mbar_arrive_expect_tx(q_full, L::KPANELS * L::QPANEL);
      for (int p = 0; p < L::KPANELS; ++p) tma_load_3d(sQ + p * L::QPANEL, &tq, q_full, p * 64, head0, 0);
      int issued = 0;
      for (int j = 0; j < n_t; ++j) {
        const int st = j % KST;
        if (!mbar_wait(&k_empty[st], ((j / KST) & 1) ^ 1, err)) break;
        mbar_arrive_expect_tx(&k_full[st], L::K_TILE);
        load_tile(&tk, sK + st * L::K_TILE, &k_full[st], tile0 + j);
        issued = j + 1;
      }
      mbar_wait(q_full, 0, err);
      for (int j = max(0, issued - KST); j < issued; ++j) mbar_wait(&k_full[j % KST], (j / KST) & 1, err);
    }
  } else if (warp == 1) {
    // --------------------------------------------------------- V producer
    if (lane == 0) {
      prefetch_tmap(&tv);
      int issued = 0;
      for (int j = 0; j < n_t; ++j) {
        const int st = j % VST;
        if (!mbar_wait(&v_empty[st], ((j / VST) & 1) ^ 1, err)) break;
        mbar_arrive_expect_tx(&v_full[st], L::K_TILE);  // the real panels of the V tile
        load_tile(&tv, sV + st * L::V_TILE, &v_full[st], tile0 + j);
        issued = j + 1;
      }
      for (int j = max(0, issued - VST); j < issued; ++j) mbar_wait(&v_full[j % VST], (j / VST) & 1, err);
    }
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
        if (r < D && in_range(orow * D + r, 1, part_rows * D, err)) o_part[orow * D + r] = __uint_as_float(o[h]) / lh;
        if (r == 0 && in_range(orow, 1, part_rows, err)) lse_part[orow] = (m[h] + __log2f(lh)) * dec::LN2;
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

template <int D, int GM>
static cudaError_t launch_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const int* table,
                            const int* seq_lens, float* o_part, float* lse_part, int B, int H, int Hkv,
                            int num_blocks, int bs, int max_blocks, float scale, int S, cudaStream_t stream) {
  using C = Cfg<GM>;
  const int smem = Smem<D, C::KST, C::VST, C::PB>::ALLOC;
  cudaError_t e = cudaFuncSetAttribute(decode_mma_kernel<D, GM>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int n_chunk = (H / Hkv + NH - 1) / NH;
  const dim3 grid(static_cast<unsigned>(S), static_cast<unsigned>(Hkv * n_chunk), static_cast<unsigned>(B));
  decode_mma_kernel<D, GM><<<grid, THREADS, smem, stream>>>(tq, tk, tv, table, seq_lens, o_part, lse_part, B, H, Hkv,
                                                         num_blocks, bs, max_blocks, scale * dec::LOG2E);
  return cudaGetLastError();
}

template <int D>
static cudaError_t launch_d(const void* q, const void* kc, const void* vc, const int* table, const int* seq_lens,
                            float* o_part, float* lse_part, int B, int H, int Hkv, int num_blocks, int bs,
                            int max_blocks, float scale, int S, cudaStream_t stream) {
  CUtensorMap tq, tk, tv;
  if (!make_tmap_bf16(&tq, q, 1, B * H, D, NH) || !make_tmap_bf16(&tk, kc, num_blocks * Hkv, bs, D, bs) ||
      !make_tmap_bf16(&tv, vc, num_blocks * Hkv, bs, D, bs))
    return cudaErrorInvalidValue;
  const int G = H / Hkv;  // query heads per K/V head; CTAs take them 16 at a time
  if (G <= 4)
    return launch_t<D, 4>(tq, tk, tv, table, seq_lens, o_part, lse_part, B, H, Hkv, num_blocks, bs, max_blocks,
                          scale, S, stream);
  if (G <= 8)
    return launch_t<D, 8>(tq, tk, tv, table, seq_lens, o_part, lse_part, B, H, Hkv, num_blocks, bs, max_blocks,
                          scale, S, stream);
  return launch_t<D, 16>(tq, tk, tv, table, seq_lens, o_part, lse_part, B, H, Hkv, num_blocks, bs, max_blocks,
                         scale, S, stream);
}

static cudaError_t launch(const void* q, const void* kc, const void* vc, const int* table, const int* seq_lens,
                          float* o_part, float* lse_part, int B, int H, int Hkv, int d, int num_blocks, int bs,
                          int max_blocks, float scale, int S, cudaStream_t stream) {
  return d == 64 ? launch_d<64>(q, kc, vc, table, seq_lens, o_part, lse_part, B, H, Hkv, num_blocks, bs,
                                max_blocks, scale, S, stream)
                 : launch_d<128>(q, kc, vc, table, seq_lens, o_part, lse_part, B, H, Hkv, num_blocks, bs,
                                 max_blocks, scale, S, stream);
}

// Shapes this kernel serves; the others take the FMA-pipe kernel.
inline bool serves(int d, int bs) { return (d == 64 || d == 128) && bs % 8 == 0 && TK % bs == 0; }

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
  if (decmma::serves(d, block_size)) {
    cudaError_t e = decmma::launch(q, k_cache, v_cache, block_table, seq_lens, o_part, lse_part, B, H, Hkv, d,
                                   num_blocks, block_size, max_blocks, scale, S, stream);
    if (e != cudaSuccess) return e;
    return launch_attn_merge(o_part, lse_part, S, o, lse, static_cast<long long>(B) * H, d, stream);
  }
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
