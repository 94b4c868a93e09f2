// Declarations shared by the C-ABI layer and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace fa {

// Heads whose tiles are scheduled together: the CTAs resident at one time
// then re-read one group's shared operand (K and V in the forward and the
// dQ sweep, Q and dO in the dK/dV sweep), and the group is sized so that
// operand stays in L2 (about 40 MB of the 129 MB). `bytes_per_head` is the
// shared operand's size per scheduled head.
constexpr long long kL2GroupBytes = 40ll << 20;
inline int head_group_for(long long bytes_per_head, int max_group) {
  long long g = bytes_per_head > 0 ? kL2GroupBytes / bytes_per_head : max_group;
  if (g > max_group) g = max_group;
  return g < 1 ? 1 : static_cast<int>(g);
}

// Kernel launchers. Pointers are device pointers to contiguous [BH][N][d]
// bf16 tensors (lse, Dvec: [BH][N] fp32); k, v, dk and dv hold BH / G heads,
// query head h reading K/V head h / G (G = 1: one K/V head per query head).
// Each launcher builds the TMA descriptors its kernel needs. Arguments are
// assumed validated by the caller. Return the launch (or descriptor) error.
cudaError_t launch_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int BH,
                       int G, int N, int d, float scale, bool causal, cudaStream_t stream);
cudaError_t launch_bwd_preprocess(const __nv_bfloat16* o, const __nv_bfloat16* dO, float* Dvec,
                                  int BH, int N, int d, cudaStream_t stream);
cudaError_t launch_bwd_dkdv(const void* q, const void* k, const void* v, const void* dO, void* dk,
                            void* dv, const float* lse, const float* Dvec, int BH, int G, int N, int d,
                            float scale, bool causal, cudaStream_t stream);
cudaError_t launch_bwd_dq(const void* q, const void* k, const void* v, const void* dO, void* dq,
                          const float* lse, const float* Dvec, int BH, int G, int N, int d, float scale,
                          bool causal, cudaStream_t stream);
// Whether the full backward forms D inside the dQ sweep and runs the dK/dV
// sweep after it, instead of a separate D pass and the two sweeps side by
// side: with one K/V head per query head (G = 1) and a dK/dV grid of at
// least four CTAs per SM. Measured: c4 2.354 against 2.382 ms, B=16 H=16
// N=2048 causal 0.795 against 0.821; with grouped-query heads or small
// grids the two sweeps sharing one tail is worth more than the D pass.
bool bwd_fuse_d(int BH, int G, int N);
// The dQ sweep that also forms D = rowsum(dO ∘ O) of its query tiles from o
// and writes it to Dvec (for a dK/dV sweep launched after it).
cudaError_t launch_bwd_dq_d(const void* q, const void* k, const void* v, const void* o, const void* dO,
                            void* dq, const float* lse, float* Dvec, int BH, int G, int N, int d, float scale,
                            bool causal, cudaStream_t stream);

// Row softmax of x [rows][n] fp32 into y (may alias x): three passes (safe)
// or two (online). One CTA per row.
cudaError_t launch_softmax(const float* x, float* y, long long rows, int n, bool online,
                           cudaStream_t stream);

// Decode of one new query row per request against a paged KV cache
// (k_cache, v_cache [num_blocks][Hkv][block_size][d] bf16), split over the
// context into S parts, partial results in o_part [S][B*H][d] fp32 and
// lse_part [S][B*H], then merged into o [B*H][d] bf16 and lse [B*H].
cudaError_t launch_decode_paged(const void* q, const void* k_cache, const void* v_cache,
                                const int* block_table, const int* seq_lens, void* o, float* lse,
                                float* o_part, float* lse_part, int B, int H, int Hkv, int d,
                                int num_blocks, int block_size, int max_blocks, float scale, int S,
                                cudaStream_t stream);
// Merge S partial attention results per row: o_parts [S][rows][d] fp32,
// lse_parts [S][rows] -> o [rows][d] bf16, lse [rows].
cudaError_t launch_attn_merge(const float* o_parts, const float* lse_parts, int S, void* o, float* lse,
                              long long rows, int d, cudaStream_t stream);

// The calling host thread's side stream on the current device (a
// non-blocking stream the library creates on first use and keeps).
cudaError_t side_stream(cudaStream_t* out);

// Device error words (one per translation unit): read, then clear.
cudaError_t launch_wait_limit_selftest(cudaStream_t stream);
cudaError_t read_and_clear_selftest_error(uint32_t* out, cudaStream_t stream);
cudaError_t read_and_clear_fwd_error(uint32_t* out, cudaStream_t stream);
cudaError_t read_and_clear_bwd_error(uint32_t* out, cudaStream_t stream);
cudaError_t read_and_clear_decode_error(uint32_t* out, cudaStream_t stream);
cudaError_t read_and_clear_softmax_error(uint32_t* out, cudaStream_t stream);

}  // namespace fa
