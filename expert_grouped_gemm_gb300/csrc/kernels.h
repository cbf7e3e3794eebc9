// kernels.h -- host launchers of the bandwidth kernels (routing, permutation,
// combine, scores, selection, compaction, router backward, dX reduce).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

namespace moe {

// part / nsplit / part_stride: the router GEMM's fp32 partial sums when it ran as a
// K split (null: logits already hold the sums). masks_clear: the caller has zeroed the
// chunk masks. logits_out / topk_idx_out / topk_w_out: optional second copies of the
// biased logits, indices and weights (the caller's own buffers), written by the kernel.
cudaError_t launch_route_topk(float* logits, const float* bias, int T, int E, int k, int* topk_idx, float* topk_w,
                              uint64_t* masks, cudaStream_t st, const float* part = nullptr, int nsplit = 1,
                              int64_t part_stride = 0, bool masks_clear = false, float* logits_out = nullptr,
                              int* topk_idx_out = nullptr, float* topk_w_out = nullptr);
cudaError_t launch_route_scan(const uint64_t* masks, int C, int E, int* count, int* offset, int* pad_off,
                              int* tile_off, int* chunk_base, int* pair_of_row, int* user_offsets, cudaStream_t st,
                              int* order = nullptr, int* tile_off2 = nullptr, int4* tile_rec = nullptr,
                              int4* ord_rec = nullptr, int4* tile_rec2 = nullptr);
cudaError_t launch_route_index(const uint64_t* masks, const int* chunk_base, const int* topk_idx, const int* offset,
                               const int* pad_off, int T, int E, int k, int* rowp_of_pair, int* row_of_pair,
                               int* pair_of_row, cudaStream_t st, int* row_of_pair_out = nullptr);
template <typename TIO>
cudaError_t launch_gather_rows(const void* x, const int* pair_of_row, const int* pad_total, int64_t Rmax, int H, int k,
                               void* x_perm, float* xnorm, int num_sms, cudaStream_t st);
template <typename TIO>
cudaError_t launch_combine(const void* y_pair, const int* rowp_of_pair, const float* topk_w, const void* sh_y, int T,
                           int H, int k, void* y, int num_sms, cudaStream_t st);

template <typename TIO>
cudaError_t launch_pair_score(const void* dy, const void* y_pair, const int* pair_of_row, const int* pad_total,
                              int64_t Rmax, const float* topk_w, const float* xnorm, int H, int k, float* g,
                              float* score, void* dy_perm, float* user_scores, int num_sms, cudaStream_t st);
cudaError_t launch_select(const float* score, const int* count, const int* pad_off, const int* quota, int E,
                          int* ret_cidx, int* ret_count, int* status, cudaStream_t st);
// K-split second pass (splitk.cu): ordered sums of the fp32 partials, then the
// epilogue of the unsplit GEMM (bf16 store, or the SwiGLU forward into ab and h).
// Rows: *nrows_dev when given, else nrows_const; max_rows bounds the grid.
cudaError_t launch_splitk_store(const float* part, int64_t stride, int S, const int* nrows_dev, int nrows_const,
                                int64_t max_rows, const int* pair_of_row, int N, int64_t ldo, void* out, int num_sms,
                                cudaStream_t st);
cudaError_t launch_splitk_swiglu(const float* part, int64_t stride, int S, const int* nrows_dev, int64_t max_rows,
                                 const int* pair_of_row, int F, void* ab, void* h, int num_sms, cudaStream_t st);
cudaError_t launch_ret_scan(const int* ret_count, int E, int* ret_offset, int* ret_pad_off, int* ret_tile_off,
                            int* ret_src, int* user_offsets, cudaStream_t st, int* order = nullptr,
                            int* ret_tile_off2 = nullptr, int4* tile_rec = nullptr, int4* ord_rec = nullptr,
                            int4* tile_rec2 = nullptr);
cudaError_t launch_ret_index(const int* topk_idx, const int* rowp_of_pair, const int* row_of_pair,
                             const int* ret_cidx, const int* ret_offset, const int* ret_pad_off, int64_t P,
                             int* ret_src, int* crow_of_pair, int* ret_rows, int* user_rows, int num_sms,
                             cudaStream_t st);
template <typename TIO>
cudaError_t launch_compact_rows(const int* ret_src, const int* ret_pad_total, int64_t Rmax, const int* pair_of_row,
                                const float* topk_w, const void* x, const void* ab, const void* h, const void* dy,
                                int H, int F, int k, void* x_c, void* ab_c, void* h_c, void* dy_c, int num_sms,
                                cudaStream_t st);
template <typename TIO>
cudaError_t launch_router_bwd(const float* g, const int* rowp_of_pair, const int* topk_idx, const float* topk_w,
                              int T, int Tpad, int E, int k, float* dl_sel, void* dl_dense, int num_sms,
                              cudaStream_t st);
template <typename TIO>
cudaError_t launch_transpose(const void* in, int R, int Cc, void* out, cudaStream_t st);
template <typename TIO>
cudaError_t launch_dx_reduce(const void* dx_pair, const int* crow_of_pair, const int* topk_idx, const float* dl_sel,
                             const void* wrT, const void* sh_dx, int T, int H, int k, void* dx, int num_sms,
                             cudaStream_t st);

cudaError_t launch_plan_quota(const int* count, int E, int64_t pairs, int64_t rho_num, int64_t rho_den,
                              const int* budget, int* quota, cudaStream_t st);

}  // namespace moe
