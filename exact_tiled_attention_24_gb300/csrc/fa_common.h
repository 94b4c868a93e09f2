// Declarations shared by the C-ABI layer and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace fa {

// Launch the forward kernel. Maps: q/k/v/o are [BH][N][d] bf16 with 64x128
// boxes. lse is [BH][N] fp32. Returns the launch error.
cudaError_t launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& to, float* lse, int BH, int N, int d, float scale,
                       bool causal, cudaStream_t stream);

// Backward stages (see fa_bwd.cu).
cudaError_t launch_bwd_preprocess(const __nv_bfloat16* o, const __nv_bfloat16* dO, float* Dvec,
                                  float* dq_acc, int BH, int N, int d, cudaStream_t stream);
cudaError_t launch_bwd_main(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const CUtensorMap& tdk,
                            const CUtensorMap& tdv, const float* lse, const float* Dvec,
                            float* dq_acc, int BH, int N, int d, float scale, bool causal,
                            cudaStream_t stream);
cudaError_t launch_bwd_dq_convert(const float* dq_acc, __nv_bfloat16* dq, int BH, int N, int d,
                                  float scale, cudaStream_t stream);

// Device error words (one per translation unit): read, then clear.
cudaError_t read_and_clear_fwd_error(uint32_t* out, cudaStream_t stream);
cudaError_t read_and_clear_bwd_error(uint32_t* out, cudaStream_t stream);

}  // namespace fa
