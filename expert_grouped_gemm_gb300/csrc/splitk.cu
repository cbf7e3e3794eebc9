// splitk.cu -- the second pass of a K-split tensor-core GEMM: the fp32 partial
// outputs of the splits are added in split order (so the result does not depend
// on which CTA finished first) and the epilogue of the unsplit GEMM is applied.
// A K split is used when a GEMM has too few output tiles to occupy the GPU:
// the router GEMMs, and the expert forward GEMMs at decode-sized token counts.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

// 8 consecutive fp32 partial sums of split 0..S-1 at element offset i, added in order
// (four splits' loads are issued together before they are added, still in order)
__device__ __forceinline__ void sum_splits(const float* __restrict__ part, int64_t stride, int S, int64_t i, float* v) {
#pragma unroll
  for (int q = 0; q < 8; ++q) v[q] = 0.0f;
  for (int s0 = 0; s0 < S; s0 += 4) {
    float4 u[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (s0 + j < S) {
        const float4* p = reinterpret_cast<const float4*>(part + (s0 + j) * stride + i);
        u[2 * j] = p[0];
        u[2 * j + 1] = p[1];
      }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (s0 + j < S) {
        v[0] += u[2 * j].x; v[1] += u[2 * j].y; v[2] += u[2 * j].z; v[3] += u[2 * j].w;
        v[4] += u[2 * j + 1].x; v[5] += u[2 * j + 1].y; v[6] += u[2 * j + 1].z; v[7] += u[2 * j + 1].w;
      }
    }
  }
}

// out[r, n] = bf16(sum_s part[s][r][n]); rows marked as expert padding (pair_of_row < 0)
// are written as zeros. Thread per 8 columns, grid-stride over rows x column groups.
__global__ void __launch_bounds__(256) k_splitk_store(const float* __restrict__ part, int64_t stride, int S,
                                                      const int* __restrict__ nrows_dev, int nrows_const,
                                                      const int* __restrict__ pair_of_row, int N, int64_t ldo,
                                                      __nv_bfloat16* __restrict__ out) {
  pdl_wait();  // the previous kernel has completed and its writes are visible
  const int nrows = nrows_dev ? *nrows_dev : nrows_const;
  const int nv = N / 8;
  for (int64_t w = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; w < (int64_t)nrows * nv;
       w += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = w / nv;
    const int c = (int)(w - r * nv) * 8;
    float v[8];
    if (pair_of_row && pair_of_row[r] < 0) {
#pragma unroll
      for (int q = 0; q < 8; ++q) v[q] = 0.0f;
    } else {
      sum_splits(part, stride, S, r * N + c, v);
    }
    *reinterpret_cast<uint4*>(out + r * ldo + c) = f_to_bf16x8(v);
  }
}

// Expert gate/up: a = sum_s part[s][r][n], b = sum_s part[s][r][F + n];
// ab[r] = (a | b) and h[r] = silu(a) b in bf16, as the SwiGLU epilogue of the
// unsplit GEMM writes them; padding rows are zeros.
__global__ void __launch_bounds__(256) k_splitk_swiglu(const float* __restrict__ part, int64_t stride, int S,
                                                       const int* __restrict__ nrows_dev,
                                                       const int* __restrict__ pair_of_row, int F,
                                                       __nv_bfloat16* __restrict__ ab, __nv_bfloat16* __restrict__ h) {
  pdl_wait();  // the previous kernel has completed and its writes are visible
  const int nrows = *nrows_dev;
  const int nv = F / 8;
  for (int64_t w = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; w < (int64_t)nrows * nv;
       w += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = w / nv;
    const int c = (int)(w - r * nv) * 8;
    float a[8], b[8], hv[8];
    if (pair_of_row[r] < 0) {
#pragma unroll
      for (int q = 0; q < 8; ++q) a[q] = b[q] = 0.0f;
    } else {
      sum_splits(part, stride, S, r * 2 * F + c, a);
      sum_splits(part, stride, S, r * 2 * F + F + c, b);
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) hv[q] = a[q] * sigmoidf_(a[q]) * b[q];
    *reinterpret_cast<uint4*>(ab + r * 2 * F + c) = f_to_bf16x8(a);
    *reinterpret_cast<uint4*>(ab + r * 2 * F + F + c) = f_to_bf16x8(b);
    *reinterpret_cast<uint4*>(h + r * F + c) = f_to_bf16x8(hv);
  }
}

int grid_rows(int64_t max_rows, int n, int num_sms) {
  const int64_t work = max_rows * (n / 8);
  return (int)std::max<int64_t>(1, std::min<int64_t>((work + 255) / 256, (int64_t)num_sms * 8));
}

}  // namespace

cudaError_t launch_splitk_store(const float* part, int64_t stride, int S, const int* nrows_dev, int nrows_const,
                                int64_t max_rows, const int* pair_of_row, int N, int64_t ldo, void* out, int num_sms,
                                cudaStream_t st) {
  if (N % 8 || ldo % 8) return cudaErrorInvalidValue;
  MOE_LAUNCH(k_splitk_store, grid_rows(max_rows, N, num_sms), 256, 0, st, part, stride, S, nrows_dev, nrows_const,
                                                                  pair_of_row, N, ldo,
                                                                  reinterpret_cast<__nv_bfloat16*>(out));
  return cudaGetLastError();
}

cudaError_t launch_splitk_swiglu(const float* part, int64_t stride, int S, const int* nrows_dev, int64_t max_rows,
                                 const int* pair_of_row, int F, void* ab, void* h, int num_sms, cudaStream_t st) {
  if (F % 8) return cudaErrorInvalidValue;
  MOE_LAUNCH(k_splitk_swiglu, grid_rows(max_rows, F, num_sms), 256, 0, st, part, stride, S, nrows_dev, pair_of_row, F,
                                                                   reinterpret_cast<__nv_bfloat16*>(ab),
                                                                   reinterpret_cast<__nv_bfloat16*>(h));
  return cudaGetLastError();
}

}  // namespace moe
