// gemm_simt.cu -- fp32 grouped GEMM on the CUDA cores.
//
// The fp32 I/O configuration needs fp32-exact products: tensor-core tf32
// rounds operands to 10 mantissa bits, far outside a 1e-5 relative budget.
// This kernel computes the same GemmArgs problems as the tensor-core kernel
// with one thread per output element (two for paired SwiGLU halves) and a
// plain fp32 dot product, accumulated in ascending k.
#include "epilogue.cuh"
#include "gemm_launch.h"

namespace moe {

__global__ void simt_grouped_gemm_f32(const GemmArgs a) {
  pdl_wait();  // the previous kernel has completed and its writes are visible
  const float* A = reinterpret_cast<const float*>(a.A);
  const float* B0 = reinterpret_cast<const float*>(a.B0);
  const float* B1 = reinterpret_cast<const float*>(a.B1 ? a.B1 : a.B0);
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= a.N) return;
  float v0[1], v1[1];
  if (!a.var_k) {
    // one padded row per blockIdx.y (grid-stride)
    const int total_rows = a.row_off ? a.row_off[a.G] : a.rows_const;
    for (int r = blockIdx.y; r < total_rows; r += gridDim.y) {
      int g = 0;
      if (a.row_off) {  // last g with row_off[g] <= r
        int lo = 0, hi = a.G - 1;
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (a.row_off[mid] <= r) lo = mid; else hi = mid - 1;
        }
        g = lo;
      }
      const int rows_g = grp_rows(a, g);
      const int m = r - grp_off(a, g);
      float acc0 = 0.0f, acc1 = 0.0f;
      if (m < rows_g) {
        const float* ar = A + (int64_t)r * a.lda;
        for (int k = 0; k < a.K; ++k) {
          float b0, b1 = 0.0f;
          if (a.b_kmajor) {
            const bool second = a.k_split > 0 && k >= a.k_split;
            const float* Bm = second ? B1 : B0;
            const int kk = second ? k - a.k_split : k;
            b0 = Bm[((int64_t)g * a.N + n) * a.ldb + kk];
          } else {
            const int64_t br = ((int64_t)g * a.K + k) * a.ldb;
            b0 = B0[br + n];
            if (a.paired) b1 = B1[br + a.b1_col + n];
          }
          acc0 = fmaf(ar[k], b0, acc0);
          acc1 = fmaf(ar[k], b1, acc1);
        }
      }
      v0[0] = acc0;
      v1[0] = acc1;
      epilogue_apply<float, 1>(a, g, rows_g, m, n, v0, a.paired ? v1 : nullptr);
    }
  } else {
    const int g = blockIdx.z;
    const int rows_g = grp_rows(a, g);
    const int off = grp_off(a, g);
    for (int m = blockIdx.y; m < a.M; m += gridDim.y) {
      float acc0 = 0.0f, acc1 = 0.0f;
      for (int r = 0; r < rows_g; ++r) {
        const float av = A[(int64_t)(off + r) * a.lda + m];
        const int64_t br = (int64_t)(off + r) * a.ldb;
        acc0 = fmaf(av, B0[br + n], acc0);
        if (a.paired) acc1 = fmaf(av, B1[br + a.b1_col + n], acc1);
      }
      v0[0] = acc0;
      v1[0] = acc1;
      epilogue_apply<float, 1>(a, g, rows_g, m, n, v0, a.paired ? v1 : nullptr);
    }
  }
}

cudaError_t launch_simt_gemm_f32(const GemmArgs& a, cudaStream_t st) {
  dim3 block(64);
  dim3 grid((a.N + 63) / 64, 1, 1);
  if (!a.var_k) {
    grid.y = (unsigned)std::min<int64_t>(a.a_rows > 0 ? a.a_rows : 1, 65535);
  } else {
    grid.y = (unsigned)std::min(a.M, 65535);
    grid.z = (unsigned)a.G;
  }
  MOE_LAUNCH(simt_grouped_gemm_f32, grid, block, 0, st, a);
  return cudaGetLastError();
}

}  // namespace moe
