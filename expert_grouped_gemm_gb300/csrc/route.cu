// route.cu -- forward bandwidth kernels: top-k routing, deterministic
// histogram + scan, stable permutation, row gather and weighted combine.
//
// Routing follows issue "[MoE] Hot experts on RNGD during training (host
// dispatch, device expert graphs) #14", Proposal (routing and dispatch of
// token rows to experts, results scattered back), done here on the device:
//   * selection: per token the k largest biased fp32 logits, ties to the lower
//     expert index, slots in that order; weights = softmax renormalised over
//     the k selected logits, i.e. exp(l_j - l_max) / sum_j' exp(l_j' - l_max);
//   * placement: expert-contiguous rows, token order inside an expert, each
//     expert padded to 16 rows. Per 64-token chunk, a 64-bit mask per expert
//     records which tokens chose it, so a pair's rank inside its expert is a
//     popcount: no atomics on rows, identical result on every run.
#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kChunk = 64;  // tokens per routing chunk (one bit each in a uint64 mask)

// ------------------------------------------------------------------ top-k
// Warp per token (8 per block); lane l holds logits e = l + 32 i (i < EPL) in
// registers. The chunk masks (zeroed beforehand) get one bit per pair. ulogits,
// uidx, uw (each may be null) receive a second copy of what goes to logits,
// topk_idx and topk_w.
template <int EPL>
__global__ void __launch_bounds__(256) k_route_topk(float* logits, const float* bias, int T, int E, int k,
                                                    int* topk_idx, float* topk_w, uint64_t* masks,
                                                    const float* part, int nsplit, int64_t part_stride,
                                                    float* ulogits, int* uidx, float* uw) {
  pdl_wait();  // the previous kernel has completed and its writes are visible
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= T) return;
  float* lrow = logits + (int64_t)t * E;
  float v[EPL];
  float l[EPL];
  float bv_[EPL];  // the bias, loaded beside the logits rather than after them
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    bv_[i] = (bias && e < E) ? bias[e] : 0.0f;
  }
  if (part) {  // the router GEMM ran as a K split: its partial sums, added in split order
#pragma unroll
    for (int i = 0; i < EPL; ++i) l[i] = 0.0f;
    for (int s0 = 0; s0 < nsplit; s0 += 4) {
      float q[4][EPL];
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
          const int e = lane + 32 * i;
          q[j][i] = (s0 + j < nsplit && e < E) ? part[(s0 + j) * part_stride + (int64_t)t * E + e] : 0.0f;
        }
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int i = 0; i < EPL; ++i)
          if (s0 + j < nsplit) l[i] += q[j][i];
    }
  } else {
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      l[i] = e < E ? lrow[e] : 0.0f;
    }
  }
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    if (e < E) {
      const float x = l[i] + bv_[i];
      lrow[e] = x;                     // the biased logits the selection used
      if (ulogits) ulogits[(int64_t)t * E + e] = x;
      v[i] = (x != x) ? -INFINITY : x;  // NaN ranks last
    }
  }
  uint32_t taken = 0;  // bit i: expert lane + 32 i already selected (or absent)
#pragma unroll
  for (int i = 0; i < EPL; ++i)
    if (lane + 32 * i >= E) taken |= 1u << i;
  float lmax = 0.0f, sum = 0.0f;
  uint64_t* cmask = masks + (int64_t)(t / kChunk) * E;
  const uint64_t bit = 1ull << (t % kChunk);
  if (k <= 32) {
    // every lane sees each round's winner; lane j keeps slot j's expert and weight and
    // writes them itself, so no lane walks the k slots and nothing is read back
    int my_e = 0;
    float my_w = 0.0f;
    for (int j = 0; j < k; ++j) {
      float bv = -INFINITY;
      int be = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        if (!((taken >> i) & 1u) && (be == 0x7fffffff || v[i] > bv)) {  // e ascending: ties keep the first
          bv = v[i];
          be = e;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oe = __shfl_xor_sync(0xffffffffu, be, o);
        if (oe != 0x7fffffff && (be == 0x7fffffff || ov > bv || (ov == bv && oe < be))) {
          bv = ov;
          be = oe;
        }
      }
      if ((be & 31) == lane) taken |= 1u << (be >> 5);
      if (j == 0) lmax = bv;
      const float ex = expf(bv - lmax);
      sum += ex;  // the same order on every lane: slot 0 first
      if (lane == j) {
        my_e = be;
        my_w = ex;
      }
    }
    if (lane < k) {
      const int64_t q = (int64_t)t * k + lane;
      const float w = my_w * (1.0f / sum);
      topk_idx[q] = my_e;
      topk_w[q] = w;
      if (uidx) uidx[q] = my_e;
      if (uw) uw[q] = w;
      atomicOr(reinterpret_cast<unsigned long long*>(&cmask[my_e]), bit);
    }
    return;
  }
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int be = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      if (!((taken >> i) & 1u) && (be == 0x7fffffff || v[i] > bv)) {  // e ascending: ties keep the first
        bv = v[i];
        be = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oe = __shfl_xor_sync(0xffffffffu, be, o);
      if (oe != 0x7fffffff && (be == 0x7fffffff || ov > bv || (ov == bv && oe < be))) {
        bv = ov;
        be = oe;
      }
    }
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
    if (lane == 0) {
      if (j == 0) lmax = bv;
      const float ex = expf(bv - lmax);
      sum += ex;
      topk_idx[(int64_t)t * k + j] = be;
      topk_w[(int64_t)t * k + j] = ex;
      if (uidx) uidx[(int64_t)t * k + j] = be;
      atomicOr(reinterpret_cast<unsigned long long*>(&cmask[be]), bit);
    }
  }
  if (lane == 0) {
    const float inv = 1.0f / sum;
    for (int j = 0; j < k; ++j) {
      const float w = topk_w[(int64_t)t * k + j] * inv;
      topk_w[(int64_t)t * k + j] = w;
      if (uw) uw[(int64_t)t * k + j] = w;
    }
  }
}

// ------------------------------------------------------------------ scan
// One block of 1024 threads: expert e is handled by `parts` threads, each owning
// a contiguous range of chunks (parts = 1024 / E rounded down to a power of two).
__global__ void __launch_bounds__(1024) k_route_scan(const uint64_t* masks, int C, int E, int* count, int* offset,
                                                     int* pad_off, int* tile_off, int* chunk_base, int* pair_of_row,
                                                     int* user_offsets, int* order, int* tile_off2,
                                                     int4* tile_rec, int4* ord_rec, int4* tile_rec2) {
  pdl_wait();  // the previous kernel has completed and its writes are visible
  __shared__ int part_cnt[1024];
  int parts = 1;
  while (parts * 2 * E <= 1024) parts *= 2;
  const int tid = threadIdx.x;
  const int pe = tid % E, pp = tid / E;
  const bool worker = tid < parts * E;
  const int per = (C + parts - 1) / parts;
  const int c0 = pp * per, c1 = min(C, c0 + per);
  int pc = 0;
  if (worker)
    for (int cb = c0; cb < c1; cb += 8) {  // eight mask loads in flight, then their popcounts
      uint64_t m[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) m[j] = cb + j < c1 ? masks[(int64_t)(cb + j) * E + pe] : 0ull;
#pragma unroll
      for (int j = 0; j < 8; ++j) pc += __popcll(m[j]);
    }
  if (worker) part_cnt[pp * E + pe] = pc;
  __syncthreads();
  const int e = tid;
  int cnt = 0;
  if (e < E)
    for (int p = 0; p < parts; ++p) cnt += part_cnt[p * E + e];
  const int rank = order ? block_order_desc(cnt, E, order) : 0;
  const int pad = (cnt + 15) / 16 * 16;
  const int tiles = (cnt + 127) / 128;
  const int tiles2 = (cnt + 255) / 256;
  int4 tot;
  const int4 ex = block_excl_scan4(e < E ? make_int4(cnt, pad, tiles, tiles2) : make_int4(0, 0, 0, 0), &tot);
  const int oc = ex.x, op = ex.y, ot = ex.z, ot2 = ex.w;
  const int tot_c = tot.x, tot_p = tot.y, tot_t = tot.z, tot_t2 = tot.w;
  __shared__ int s_pad[1024];
  if (e < E) {
    count[e] = cnt;
    offset[e] = oc;
    pad_off[e] = op;
    tile_off[e] = ot;
    if (tile_off2) tile_off2[e] = ot2;
    if (user_offsets) user_offsets[e] = oc;
    s_pad[e] = op;
    for (int r = op + cnt; r < op + pad; ++r) pair_of_row[r] = -1;
    if (tile_rec)
      for (int j = 0; j < tiles; ++j) tile_rec[ot + j] = make_int4(e, j * 128, cnt, op);
    if (tile_rec2)
      for (int j = 0; j < tiles2; ++j) tile_rec2[ot2 + j] = make_int4(e, j * 256, cnt, op);
    if (ord_rec && order) ord_rec[rank] = make_int4(e, cnt, op, 0);
  }
  if (e == 0) {
    offset[E] = tot_c;
    pad_off[E] = tot_p;
    tile_off[E] = tot_t;
    if (tile_off2) tile_off2[E] = tot_t2;
    if (user_offsets) user_offsets[E] = tot_c;
  }
  __syncthreads();
  if (worker) {
    int run = s_pad[pe];
    for (int p = 0; p < pp; ++p) run += part_cnt[p * E + pe];
    for (int cb = c0; cb < c1; cb += 8) {
      uint64_t m[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) m[j] = cb + j < c1 ? masks[(int64_t)(cb + j) * E + pe] : 0ull;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (cb + j < c1) {
          chunk_base[(int64_t)(cb + j) * E + pe] = run;
          run += __popcll(m[j]);
        }
    }
  }
}

// ------------------------------------------------------------------ pair -> row
// grid = C chunks, block = 256.
__global__ void __launch_bounds__(256) k_route_index(const uint64_t* masks, const int* chunk_base, const int* topk_idx,
                                                     const int* offset, const int* pad_off, int T, int E, int k,
                                                     int* rowp_of_pair, int* row_of_pair, int* pair_of_row,
                                                     int* urow) {
  pdl_wait();  // the previous kernel has completed and its writes are visible
  extern __shared__ uint64_t sm[];  // masks[E] then bases[E]
  int* sbase = reinterpret_cast<int*>(sm + E);
  const int c = blockIdx.x;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    sm[e] = masks[(int64_t)c * E + e];
    sbase[e] = chunk_base[(int64_t)c * E + e];
  }
  __syncthreads();
  const int t0 = c * kChunk;
  const int ntok = min(kChunk, T - t0);
  for (int i = threadIdx.x; i < ntok * k; i += blockDim.x) {
    const int tl = i / k;
    const int64_t p = (int64_t)t0 * k + i;
    const int e = topk_idx[p];
    const int rank = __popcll(sm[e] & ((1ull << tl) - 1ull));
    const int prow = sbase[e] + rank;
    rowp_of_pair[p] = prow;
    const int r = offset[e] + (prow - pad_off[e]);
    row_of_pair[p] = r;
    if (urow) urow[p] = r;  // the caller's copy, when asked for
    pair_of_row[prow] = (int)p;
  }
}

// ------------------------------------------------------------------ gather
// Warp per padded row: x_perm[r] = x[token(r)] (zeros for pad rows); the warp
// that copies slot 0 of a token also writes ||x_t||_2.
template <typename TIO>
__global__ void __launch_bounds__(256) k_gather_rows(const TIO* x, const int* pair_of_row, const int* pad_total,
                                                     int H, int k, TIO* x_perm, float* xnorm) {
  pdl_wait();  // the previous kernel has completed and its writes are visible
  const int nrows = *pad_total;
  const int lane = threadIdx.x & 31;
  for (int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < nrows; r += (gridDim.x * blockDim.x) >> 5) {
    const int p = pair_of_row[r];
    TIO* dst = x_perm + (int64_t)r * H;
    float ss = 0.0f;
    if constexpr (sizeof(TIO) == 2) {
      const int nv = H / 8;
      if (p < 0) {
        for (int i = lane; i < nv; i += 32) reinterpret_cast<uint4*>(dst)[i] = make_uint4(0, 0, 0, 0);
      } else {
        const uint4* src = reinterpret_cast<const uint4*>(x + (int64_t)(p / k) * H);
        for (int i0 = lane; i0 < nv; i0 += 32 * 8) {  // eight loads in flight per lane, then their stores
          uint4 u[8];
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (i0 + 32 * j < nv) u[j] = src[i0 + 32 * j];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (i0 + 32 * j < nv) {
              reinterpret_cast<uint4*>(dst)[i0 + 32 * j] = u[j];
              float f[8];
              bf16x8_to_f(u[j], f);
#pragma unroll
              for (int q = 0; q < 8; ++q) ss = fmaf(f[q], f[q], ss);
            }
          }
        }
      }
    } else {
      if (p < 0) {
        for (int i = lane; i < H; i += 32) dst[i] = TIO(0);
      } else {
        const TIO* src = x + (int64_t)(p / k) * H;
        for (int i = lane; i < H; i += 32) {
          const float v = io<TIO>::to_f(src[i]);
          dst[i] = src[i];
          ss = fmaf(v, v, ss);
        }
      }
    }
    if (p >= 0 && (p % k) == 0) {
      ss = warp_sum(ss);
      if (lane == 0) xnorm[p / k] = sqrtf(ss);
    }
  }
}

// ------------------------------------------------------------------ combine
// y[t] = sum_j w[t,j] y_pair[row(t,j)] (+ shared y[t]), slots ascending.
// bf16: block per token, thread per 8-column slice; the k rows of a slice are
// loaded together (up to 8 at a time) before they are summed.
template <typename TIO>
__global__ void __launch_bounds__(256) k_combine(const TIO* __restrict__ y_pair, const int* __restrict__ rowp_of_pair,
                                                 const float* __restrict__ topk_w, const TIO* __restrict__ sh_y, int T,
                                                 int H, int k, TIO* __restrict__ y) {
  pdl_wait();  // the previous kernel has completed and its writes are visible
  if constexpr (sizeof(TIO) == 2) {
    const int nv = H / 8;
    for (int t = blockIdx.x; t < T; t += gridDim.x) {
      const int64_t p0 = (int64_t)t * k;
      for (int i = threadIdx.x; i < nv; i += blockDim.x) {
        float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        for (int j0 = 0; j0 < k; j0 += 8) {
          uint4 u[8];
#pragma unroll
          for (int jj = 0; jj < 8; ++jj)
            if (j0 + jj < k) u[jj] = reinterpret_cast<const uint4*>(y_pair + (int64_t)rowp_of_pair[p0 + j0 + jj] * H)[i];
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            if (j0 + jj < k) {
              const float w = topk_w[p0 + j0 + jj];
              float f[8];
              bf16x8_to_f(u[jj], f);
#pragma unroll
              for (int q = 0; q < 8; ++q) acc[q] = fmaf(w, f[q], acc[q]);
            }
          }
        }
        if (sh_y) {
          float f[8];
          bf16x8_to_f(reinterpret_cast<const uint4*>(sh_y + (int64_t)t * H)[i], f);
#pragma unroll
          for (int q = 0; q < 8; ++q) acc[q] += f[q];
        }
        reinterpret_cast<uint4*>(y + (int64_t)t * H)[i] = f_to_bf16x8(acc);
      }
    }
  } else {
    const int lane = threadIdx.x & 31;
    for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += (gridDim.x * blockDim.x) >> 5) {
      const int64_t p0 = (int64_t)t * k;
      for (int i = lane; i < H; i += 32) {
        float acc = 0.0f;
        for (int j = 0; j < k; ++j)
          acc = fmaf(topk_w[p0 + j], io<TIO>::to_f(y_pair[(int64_t)rowp_of_pair[p0 + j] * H + i]), acc);
        if (sh_y) acc += io<TIO>::to_f(sh_y[(int64_t)t * H + i]);
        y[(int64_t)t * H + i] = io<TIO>::cvt(acc);
      }
    }
  }
}

// bf16, k <= 8: persistent blocks, thread per 8-column slice. The next token's
// row indices and weights are loaded (by k threads, into registers) while this
// token's rows are in flight and handed over through shared memory at the token
// boundary, so no block stalls on an index load before its row loads. Same
// summation order as k_combine.
__global__ void __launch_bounds__(256, 4) k_combine_k8(const __nv_bfloat16* __restrict__ y_pair,
                                                    const int* __restrict__ rowp_of_pair, const float* __restrict__ topk_w,
                                                    const __nv_bfloat16* __restrict__ sh_y, int T, int H, int k,
                                                    __nv_bfloat16* __restrict__ y) {
  pdl_wait();  // the previous kernel has completed and its writes are visible
  __shared__ int s_row[2][8];
  __shared__ float s_w[2][8];
  const int tid = threadIdx.x, nv = H / 8;
  int t = blockIdx.x, buf = 0;
  if (tid < k && t < T) {
    s_row[0][tid] = rowp_of_pair[(int64_t)t * k + tid];
    s_w[0][tid] = topk_w[(int64_t)t * k + tid];
  }
  __syncthreads();
  for (; t < T; t += gridDim.x) {
    const int tn = t + gridDim.x;
    int r_next = 0;
    float w_next = 0.0f;
    if (tid < k && tn < T) {
      r_next = rowp_of_pair[(int64_t)tn * k + tid];
      w_next = topk_w[(int64_t)tn * k + tid];
    }
    for (int i = tid; i < nv; i += blockDim.x) {
      uint4 u[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (j < k) u[j] = reinterpret_cast<const uint4*>(y_pair + (int64_t)s_row[buf][j] * H)[i];
      float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (j < k) {
          float f[8];
          bf16x8_to_f(u[j], f);
          const float w = s_w[buf][j];
#pragma unroll
          for (int q = 0; q < 8; ++q) acc[q] = fmaf(w, f[q], acc[q]);
        }
      }
      if (sh_y) {
        float f[8];
        bf16x8_to_f(reinterpret_cast<const uint4*>(sh_y + (int64_t)t * H)[i], f);
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[q] += f[q];
      }
      reinterpret_cast<uint4*>(y + (int64_t)t * H)[i] = f_to_bf16x8(acc);
    }
    if (tid < k) {
      s_row[buf ^ 1][tid] = r_next;
      s_w[buf ^ 1][tid] = w_next;
    }
    __syncthreads();
    buf ^= 1;
  }
}

// ------------------------------------------------------------------ launchers
cudaError_t launch_route_topk(float* logits, const float* bias, int T, int E, int k, int* topk_idx, float* topk_w,
                              uint64_t* masks, cudaStream_t st, const float* part, int nsplit, int64_t part_stride,
                              bool masks_clear, float* logits_out, int* topk_idx_out, float* topk_w_out) {
  if (!masks_clear) {
    const int C = (T + kChunk - 1) / kChunk;
    const cudaError_t e = cudaMemsetAsync(masks, 0, (size_t)C * E * sizeof(uint64_t), st);
    if (e != cudaSuccess) return e;
  }
  const int grid = (T + 7) / 8;
  const int epl = (E + 31) / 32;
  if (epl <= 1) MOE_LAUNCH(k_route_topk<1>, grid, 256, 0, st, logits, bias, T, E, k, topk_idx, topk_w, masks, part, nsplit, part_stride,
                                 logits_out, topk_idx_out, topk_w_out);
  else if (epl <= 2) MOE_LAUNCH(k_route_topk<2>, grid, 256, 0, st, logits, bias, T, E, k, topk_idx, topk_w, masks, part, nsplit, part_stride,
                                 logits_out, topk_idx_out, topk_w_out);
  else if (epl <= 4) MOE_LAUNCH(k_route_topk<4>, grid, 256, 0, st, logits, bias, T, E, k, topk_idx, topk_w, masks, part, nsplit, part_stride,
                                 logits_out, topk_idx_out, topk_w_out);
  else if (epl <= 8) MOE_LAUNCH(k_route_topk<8>, grid, 256, 0, st, logits, bias, T, E, k, topk_idx, topk_w, masks, part, nsplit, part_stride,
                                 logits_out, topk_idx_out, topk_w_out);
  else if (epl <= 16) MOE_LAUNCH(k_route_topk<16>, grid, 256, 0, st, logits, bias, T, E, k, topk_idx, topk_w, masks, part, nsplit, part_stride,
                                 logits_out, topk_idx_out, topk_w_out);
  else MOE_LAUNCH(k_route_topk<32>, grid, 256, 0, st, logits, bias, T, E, k, topk_idx, topk_w, masks, part, nsplit, part_stride,
                                 logits_out, topk_idx_out, topk_w_out);
  return cudaGetLastError();
}

cudaError_t launch_route_scan(const uint64_t* masks, int C, int E, int* count, int* offset, int* pad_off,
                              int* tile_off, int* chunk_base, int* pair_of_row, int* user_offsets, cudaStream_t st,
                              int* order, int* tile_off2, int4* tile_rec, int4* ord_rec, int4* tile_rec2) {
  MOE_LAUNCH(k_route_scan, 1, 1024, 0, st, masks, C, E, count, offset, pad_off, tile_off, chunk_base, pair_of_row,
                                   user_offsets, order, tile_off2, tile_rec, ord_rec, tile_rec2);
  return cudaGetLastError();
}

cudaError_t launch_route_index(const uint64_t* masks, const int* chunk_base, const int* topk_idx, const int* offset,
                               const int* pad_off, int T, int E, int k, int* rowp_of_pair, int* row_of_pair,
                               int* pair_of_row, cudaStream_t st, int* row_of_pair_out) {
  const int C = (T + kChunk - 1) / kChunk;
  const size_t sm = E * (sizeof(uint64_t) + sizeof(int));
  MOE_LAUNCH(k_route_index, C, 256, sm, st, masks, chunk_base, topk_idx, offset, pad_off, T, E, k, rowp_of_pair,
             row_of_pair, pair_of_row, row_of_pair_out);
  return cudaGetLastError();
}

template <typename TIO>
cudaError_t launch_gather_rows(const void* x, const int* pair_of_row, const int* pad_total, int64_t Rmax, int H, int k,
                               void* x_perm, float* xnorm, int num_sms, cudaStream_t st) {
  const int64_t want = (Rmax + 7) / 8;
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)num_sms * 16));
  MOE_LAUNCH(k_gather_rows<TIO>, grid, 256, 0, st, reinterpret_cast<const TIO*>(x), pair_of_row, pad_total, H, k,
                                           reinterpret_cast<TIO*>(x_perm), xnorm);
  return cudaGetLastError();
}

template <typename TIO>
cudaError_t launch_combine(const void* y_pair, const int* rowp_of_pair, const float* topk_w, const void* sh_y, int T,
                           int H, int k, void* y, int num_sms, cudaStream_t st) {
  if (sizeof(TIO) == 2 && k <= 8) {
    int per_sm = 0;  // persistent: as many blocks as fit at once
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_combine_k8, 256, 0) != cudaSuccess || per_sm < 1)
      per_sm = 1;
    const int g = (int)std::max<int64_t>(1, std::min<int64_t>(T, (int64_t)num_sms * per_sm));
    MOE_LAUNCH(k_combine_k8, g, 256, 0, st, reinterpret_cast<const __nv_bfloat16*>(y_pair), rowp_of_pair, topk_w,
                                    reinterpret_cast<const __nv_bfloat16*>(sh_y), T, H, k,
                                    reinterpret_cast<__nv_bfloat16*>(y));
    return cudaGetLastError();
  }
  int grid;
  if (sizeof(TIO) == 2) {
    grid = (int)std::max<int64_t>(1, std::min<int64_t>(T, (int64_t)num_sms * 32));
  } else {
    const int64_t want = ((int64_t)T + 7) / 8;
    grid = (int)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)num_sms * 16));
  }
  MOE_LAUNCH(k_combine<TIO>, grid, 256, 0, st, reinterpret_cast<const TIO*>(y_pair), rowp_of_pair, topk_w,
                                       reinterpret_cast<const TIO*>(sh_y), T, H, k, reinterpret_cast<TIO*>(y));
  return cudaGetLastError();
}

template cudaError_t launch_gather_rows<float>(const void*, const int*, const int*, int64_t, int, int, void*, float*,
                                               int, cudaStream_t);
template cudaError_t launch_gather_rows<__nv_bfloat16>(const void*, const int*, const int*, int64_t, int, int, void*,
                                                       float*, int, cudaStream_t);
template cudaError_t launch_combine<float>(const void*, const int*, const float*, const void*, int, int, int, void*,
                                           int, cudaStream_t);
template cudaError_t launch_combine<__nv_bfloat16>(const void*, const int*, const float*, const void*, int, int, int,
                                                   void*, int, cudaStream_t);

}  // namespace moe
