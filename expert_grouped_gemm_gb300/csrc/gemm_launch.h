// gemm_launch.h -- host entry points of the grouped GEMM kernels.
#pragma once
#include <cuda_runtime.h>

#include "gemm.h"

namespace moe {

// Tensor-core (tcgen05) grouped GEMM, bf16 operands. bn = 256 or 128 (tile width).
// Persistent grid of min(num_sms, max_tiles_hint) CTAs (hint <= 0: num_sms).
cudaError_t launch_tc_gemm(const GemmArgs& a, int bn, cudaStream_t st, int num_sms, int max_tiles_hint);

// Weight-stationary variable-M store GEMM on CTA pairs (gemm_ws.cu): the output
// columns on the MMA's M dimension, each group's rows on N in chunks of up to 256
// (tile_rec2 records), so groups are padded to 16 rows rather than to row tiles.
bool ws_store_supported(const GemmArgs& a);
cudaError_t launch_ws_store(const GemmArgs& a, cudaStream_t st, int num_sms);

// CUDA-core grouped GEMM for fp32 operands (same GemmArgs semantics).
cudaError_t launch_simt_gemm_f32(const GemmArgs& a, cudaStream_t st);

}  // namespace moe
