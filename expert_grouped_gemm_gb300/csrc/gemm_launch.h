// gemm_launch.h -- host entry points of the grouped GEMM kernels.
#pragma once
#include <cuda_runtime.h>

#include "gemm.h"

namespace moe {

// Tensor-core (tcgen05) grouped GEMM, bf16 operands. bn = 256 or 128 (tile width).
// Persistent grid of min(num_sms, max_tiles_hint) CTAs (hint <= 0: num_sms).
cudaError_t launch_tc_gemm(const GemmArgs& a, int bn, cudaStream_t st, int num_sms, int max_tiles_hint);

// CUDA-core grouped GEMM for fp32 operands (same GemmArgs semantics).
cudaError_t launch_simt_gemm_f32(const GemmArgs& a, cudaStream_t st);

}  // namespace moe
