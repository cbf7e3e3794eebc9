// backward.cu -- backward bandwidth kernels of the MoE block.
//
// Pair scores, quota selection and compaction follow "LRMoE: Demand-Side Load
// Re-Calibration for Efficient MoE Training on Memory-Constrained Nodes"
// (arXiv 2610.37720), Abstract: every token-expert pair gets a score that
// estimates its contribution to the expert update, each expert keeps the
// pairs within its quota, and the kept pairs are physically compacted so the
// backward grouped GEMMs run on smaller, variable-size groups. The metric
// itself is not given there; the score used is w * ||dY_t||_2 * ||x_t||_2.
// Ranking inside an expert is (score descending, token ascending); kept rows
// stay in row (= token) order.
#include "common.cuh"
#include "kernels.h"

namespace moe {

// ------------------------------------------------------------------ pair scores
// Warp per padded row r: g[r] = <dY_t, y_r>, score[r] = w ||dY_t|| ||x_t||, and
// (full mode) dy_perm[r] = w dY_t; pad rows of dy_perm are zeroed.
template <typename TIO>
__global__ void __launch_bounds__(256) k_pair_score(const TIO* dy, const TIO* y_pair, const int* pair_of_row,
                                                    const int* pad_total, const float* topk_w, const float* xnorm,
                                                    int H, int k, float* g, float* score, TIO* dy_perm,
                                                    float* user_scores) {
  pdl_wait();  // the previous kernel has completed and its writes are visible
  const int nrows = *pad_total;
  const int lane = threadIdx.x & 31;
  for (int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < nrows; r += (gridDim.x * blockDim.x) >> 5) {
    const int p = pair_of_row[r];
    if (p < 0) {
      if (dy_perm) {
        TIO* dst = dy_perm + (int64_t)r * H;
        for (int i = lane; i < H; i += 32) dst[i] = TIO(0);
      }
      continue;
    }
    const int t = p / k;
    const float w = topk_w[p];
    const TIO* dyr = dy + (int64_t)t * H;
    const TIO* yr = y_pair + (int64_t)r * H;
    TIO* dst = dy_perm ? dy_perm + (int64_t)r * H : nullptr;
    float ss = 0.0f, dot = 0.0f;
    if constexpr (sizeof(TIO) == 2) {
      const int nv = H / 8;
      for (int i0 = lane; i0 < nv; i0 += 32 * 4) {  // four column groups' loads in flight per lane
        uint4 ua[4], ub[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (i0 + 32 * j < nv) {
            ua[j] = reinterpret_cast<const uint4*>(dyr)[i0 + 32 * j];
            ub[j] = reinterpret_cast<const uint4*>(yr)[i0 + 32 * j];
          }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (i0 + 32 * j < nv) {
            float a[8], b[8];
            bf16x8_to_f(ua[j], a);
            bf16x8_to_f(ub[j], b);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              ss = fmaf(a[q], a[q], ss);
              dot = fmaf(a[q], b[q], dot);
              a[q] *= w;
            }
            if (dst) reinterpret_cast<uint4*>(dst)[i0 + 32 * j] = f_to_bf16x8(a);
          }
        }
      }
    } else {
      for (int i = lane; i < H; i += 32) {
        const float a = io<TIO>::to_f(dyr[i]);
        ss = fmaf(a, a, ss);
        dot = fmaf(a, io<TIO>::to_f(yr[i]), dot);
        if (dst) dst[i] = io<TIO>::cvt(w * a);
      }
    }
    ss = warp_sum(ss);
    dot = warp_sum(dot);
    if (lane == 0) {
      const float s = w * sqrtf(ss) * xnorm[t];
      g[r] = dot;
      score[r] = s;
      if (user_scores) user_scores[p] = s;
    }
  }
}

// ------------------------------------------------------------------ quota select
// Order-preserving map of an fp32 score to an unsigned key (larger score, larger key).
__device__ __forceinline__ uint32_t score_key(float s) {
  const uint32_t u = __float_as_uint(s);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

constexpr int kSelThreads = 512;
constexpr int kSelCache = 8192;  // keys of an expert kept in shared memory (rows past it are re-read)

// Block per expert. The kept rows are the q largest by (score descending, token
// ascending); rows of an expert are in token order, so among rows of equal score the
// earlier rows win. Steps: (1) a 4-pass MSB-first radix select over the 32-bit score
// keys finds the key of the q-th largest row and how many rows of exactly that key are
// still needed; each pass builds a 256-bin histogram of the rows that match the
// prefix found so far, and a suffix scan over the bins (in parallel) picks the bin the
// q-th row falls in; (2) one pass over the rows in row order keeps every row with a
// larger key and the first `need` rows with an equal key, and numbers the kept rows.
__global__ void __launch_bounds__(kSelThreads) k_select(const float* score, const int* count, const int* pad_off,
                                                        const int* quota, int* ret_cidx, int* ret_count,
                                                        int* status) {
  pdl_wait();  // the previous kernel has completed and its writes are visible
  __shared__ uint32_t s_key[kSelCache];
  __shared__ int hist[256];
  __shared__ int wtot[kSelThreads / 32];
  __shared__ uint32_t s_prefix;
  __shared__ int s_need;
  const int e = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cnt = count[e];
  const int base = pad_off[e];
  int q = cnt;
  if (quota) {
    const int qq = quota[e];
    if (qq < 0 && tid == 0) set_status(status, MOE_ERR_DEVICE_ARG);
    q = min(max(qq, 0), cnt);
  }
  const bool keep_all = (q == cnt), keep_none = (q == 0);
  const int cached = min(cnt, kSelCache);
  auto key_of = [&](int i) -> uint32_t { return i < kSelCache ? s_key[i] : score_key(score[base + i]); };
  uint32_t thr = 0;
  int need_eq = 0;
  if (!keep_all && !keep_none) {
    for (int i = tid; i < cached; i += kSelThreads) s_key[i] = score_key(score[base + i]);
    if (tid == 0) {
      s_prefix = 0;
      s_need = q;
    }
    uint32_t mask = 0;
    for (int d = 24; d >= 0; d -= 8) {
      if (tid < 256) hist[tid] = 0;
      __syncthreads();
      const uint32_t pre = s_prefix;
      for (int i = tid; i < cnt; i += kSelThreads) {
        const uint32_t kk = key_of(i);
        if ((kk & mask) == pre) atomicAdd(&hist[(kk >> d) & 0xFFu], 1);
      }
      __syncthreads();
      // suffix sums over the bins from the top: thread j holds bin 255 - j
      const int need = s_need;
      int v = tid < 256 ? hist[255 - tid] : 0, incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (lane == 31 && warp < 8) wtot[warp] = incl;
      __syncthreads();
      if (tid < 256) {
        for (int w2 = 0; w2 < warp; ++w2) incl += wtot[w2];
        const int excl = incl - v;
        if (excl < need && incl >= need) {  // exactly one bin holds the q-th largest row
          s_prefix = pre | ((uint32_t)(255 - tid) << d);
          s_need = need - excl;
        }
      }
      mask |= 0xFFu << d;
      __syncthreads();
    }
    thr = s_prefix;
    need_eq = s_need;
  }
  // number the kept rows in row order; rows with key == thr are kept while their rank
  // among the equal rows (in row order, i.e. token order) is below need_eq
  int carry_kept = 0, carry_eq = 0;
  for (int i0 = 0; i0 < cnt; i0 += kSelThreads) {
    const int i = i0 + tid;
    uint32_t kk = 0;
    if (i < cnt && !keep_all && !keep_none) kk = key_of(i);
    const int eq = (i < cnt && !keep_all && !keep_none && kk == thr) ? 1 : 0;
    int eq_tot;
    const int eq_rank = carry_eq + block_excl_scan(eq, &eq_tot);
    const bool kept = i < cnt && (keep_all || (!keep_none && (kk > thr || (eq && eq_rank < need_eq))));
    int kept_tot;
    const int pos = carry_kept + block_excl_scan(kept ? 1 : 0, &kept_tot);
    if (i < cnt) ret_cidx[base + i] = kept ? pos : -1;
    carry_kept += kept_tot;
    carry_eq += eq_tot;
  }
  if (tid == 0) ret_count[e] = q;
}

// One block of 1024 threads: offsets of the kept rows, exact and padded.
__global__ void __launch_bounds__(1024) k_ret_scan(const int* ret_count, int E, int* ret_offset, int* ret_pad_off,
                                                   int* ret_tile_off, int* ret_src, int* user_offsets, int* order,
                                                   int* ret_tile_off2, int4* tile_rec, int4* ord_rec,
                                                   int4* tile_rec2) {
  pdl_wait();  // the previous kernel has completed and its writes are visible
  const int e = threadIdx.x;
  const int cnt = e < E ? ret_count[e] : 0;
  const int rank = order ? block_order_desc(cnt, E, order) : 0;
  const int pad = (cnt + 15) / 16 * 16;
  const int tiles = (cnt + 127) / 128;
  const int tiles2 = (cnt + 255) / 256;
  int4 tot;
  const int4 ex = block_excl_scan4(make_int4(cnt, pad, tiles, tiles2), &tot);
  const int oc = ex.x, op = ex.y, ot = ex.z, ot2 = ex.w;
  const int tc = tot.x, tp = tot.y, tt = tot.z, tt2 = tot.w;
  if (ret_tile_off2 && e < E) ret_tile_off2[e] = ot2;
  if (ret_tile_off2 && e == 0) ret_tile_off2[E] = tt2;
  if (e < E) {
    ret_offset[e] = oc;
    ret_pad_off[e] = op;
    ret_tile_off[e] = ot;
    if (user_offsets) user_offsets[e] = oc;
    for (int r = op + cnt; r < op + pad; ++r) ret_src[r] = -1;
    if (tile_rec)
      for (int j = 0; j < tiles; ++j) tile_rec[ot + j] = make_int4(e, j * 128, cnt, op);
    if (tile_rec2)
      for (int j = 0; j < tiles2; ++j) tile_rec2[ot2 + j] = make_int4(e, j * 256, cnt, op);
    if (ord_rec && order) ord_rec[rank] = make_int4(e, cnt, op, 0);
  }
  if (e == 0) {
    ret_offset[E] = tc;
    ret_pad_off[E] = tp;
    ret_tile_off[E] = tt;
    if (user_offsets) user_offsets[E] = tc;
  }
}

// Thread per pair: compact row of each kept pair and the exposed kept-row list.
__global__ void k_ret_index(const int* topk_idx, const int* rowp_of_pair, const int* row_of_pair,
                            const int* ret_cidx, const int* ret_offset, const int* ret_pad_off, int64_t P,
                            int* ret_src, int* crow_of_pair, int* ret_rows, int* user_rows) {
  pdl_wait();  // the previous kernel has completed and its writes are visible
  for (int64_t p = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; p < P; p += (int64_t)gridDim.x * blockDim.x) {
    const int r = rowp_of_pair[p];
    const int c = ret_cidx[r];
    if (c >= 0) {
      const int e = topk_idx[p];
      const int crow = ret_pad_off[e] + c;
      ret_src[crow] = r;
      crow_of_pair[p] = crow;
      ret_rows[ret_offset[e] + c] = row_of_pair[p];
      if (user_rows) user_rows[ret_offset[e] + c] = row_of_pair[p];
    } else {
      crow_of_pair[p] = -1;
    }
  }
}

// Warp per compact row: copy x_t, a|b, h of the kept pair and write w dY_t. The four
// row segments go through one copy loop (so one set of registers serves them all); bf16
// rows move as 16-byte vectors with eight loads in flight per lane before their stores.
template <typename TIO>
__device__ __forceinline__ void zero_row(TIO* dst, int n, int lane) {
  if constexpr (sizeof(TIO) == 2) {
    for (int i = lane; i < n / 8; i += 32) reinterpret_cast<uint4*>(dst)[i] = make_uint4(0, 0, 0, 0);
  } else {
    for (int i = lane; i < n; i += 32) dst[i] = TIO(0);
  }
}

template <typename TIO>
__global__ void __launch_bounds__(256) k_compact_rows(const int* ret_src, const int* ret_pad_total,
                                                      const int* pair_of_row, const float* topk_w, const TIO* x,
                                                      const TIO* ab, const TIO* h, const TIO* dy, int H, int F, int k,
                                                      TIO* x_c, TIO* ab_c, TIO* h_c, TIO* dy_c) {
  pdl_wait();  // the previous kernel has completed and its writes are visible
  const int nrows = *ret_pad_total;
  const int lane = threadIdx.x & 31;
  for (int c = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; c < nrows; c += (gridDim.x * blockDim.x) >> 5) {
    const int src = ret_src[c];
    TIO* xd = x_c + (int64_t)c * H;
    TIO* abd = ab_c + (int64_t)c * 2 * F;
    TIO* hd = h_c + (int64_t)c * F;
    TIO* dyd = dy_c + (int64_t)c * H;
    if (src < 0) {
      zero_row(xd, H, lane);
      zero_row(abd, 2 * F, lane);
      zero_row(hd, F, lane);
      zero_row(dyd, H, lane);
      continue;
    }
    const int p = pair_of_row[src];
    const int t = p / k;
    const float w = topk_w[p];
#pragma unroll 1
    for (int seg = 0; seg < 4; ++seg) {
      const TIO* sp = seg == 0 ? x + (int64_t)t * H
                    : seg == 1 ? ab + (int64_t)src * 2 * F
                    : seg == 2 ? h + (int64_t)src * F
                               : dy + (int64_t)t * H;
      TIO* dp = seg == 0 ? xd : seg == 1 ? abd : seg == 2 ? hd : dyd;
      const int n = (seg == 0 || seg == 3) ? H : seg == 1 ? 2 * F : F;
      const bool scaled = seg == 3;  // w * dY_t, rounded once
      if constexpr (sizeof(TIO) == 2) {
        const int nv = n / 8;
        const uint4* s4 = reinterpret_cast<const uint4*>(sp);
        uint4* d4 = reinterpret_cast<uint4*>(dp);
#pragma unroll 1
        for (int i0 = lane; i0 < nv; i0 += 32 * 8) {
          uint4 u[8];
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (i0 + 32 * j < nv) u[j] = s4[i0 + 32 * j];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (i0 + 32 * j < nv) {
              if (scaled) {
                float a[8];
                bf16x8_to_f(u[j], a);
#pragma unroll
                for (int q = 0; q < 8; ++q) a[q] *= w;
                u[j] = f_to_bf16x8(a);
              }
              d4[i0 + 32 * j] = u[j];
            }
          }
        }
      } else {
        for (int i = lane; i < n; i += 32) dp[i] = scaled ? io<TIO>::cvt(w * io<TIO>::to_f(sp[i])) : sp[i];
      }
    }
  }
}

// ------------------------------------------------------------------ router backward
// Warp per token: dl_j = w_j (g_j - sum_i w_i g_i); dense row of dl (zeros off the
// selection) for the dW_router GEMM; rows in [T, Tpad) are zeroed.
template <typename TIO>
__global__ void __launch_bounds__(256) k_router_bwd(const float* g, const int* rowp_of_pair, const int* topk_idx,
                                                    const float* topk_w, int T, int Tpad, int E, int k,
                                                    float* dl_sel, TIO* dl_dense) {
  pdl_wait();  // the previous kernel has completed and its writes are visible
  const int lane = threadIdx.x & 31;
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < Tpad; t += (gridDim.x * blockDim.x) >> 5) {
    if (t >= T) {
      if (dl_dense)
        for (int e = lane; e < E; e += 32) dl_dense[(int64_t)t * E + e] = TIO(0);
      continue;
    }
    const int64_t p0 = (int64_t)t * k;
    float mean = 0.0f;
    for (int j = 0; j < k; ++j) mean = fmaf(topk_w[p0 + j], g[rowp_of_pair[p0 + j]], mean);
    if (lane == 0)
      for (int j = 0; j < k; ++j) dl_sel[p0 + j] = topk_w[p0 + j] * (g[rowp_of_pair[p0 + j]] - mean);
    if (dl_dense) {
      for (int e = lane; e < E; e += 32) {
        float v = 0.0f;
        for (int j = 0; j < k; ++j)
          if (topk_idx[p0 + j] == e) v = topk_w[p0 + j] * (g[rowp_of_pair[p0 + j]] - mean);
        dl_dense[(int64_t)t * E + e] = io<TIO>::cvt(v);
      }
    }
  }
}

// 32x32 tiled transpose: out[c][r] = in[r][c], in is [R, Cc].
template <typename TIO>
__global__ void k_transpose(const TIO* in, int R, int Cc, TIO* out) {
  pdl_wait();  // the previous kernel has completed and its writes are visible
  __shared__ TIO tile[32][33];
  const int bx = blockIdx.x * 32, by = blockIdx.y * 32;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int r = by + i, c = bx + threadIdx.x;
    if (r < R && c < Cc) tile[i][threadIdx.x] = in[(int64_t)r * Cc + c];
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int c = bx + i, r = by + threadIdx.x;
    if (r < R && c < Cc) out[(int64_t)c * R + r] = tile[threadIdx.x][i];
  }
}

// ------------------------------------------------------------------ dX reduce
// dX_t = sum_j [kept] dx_pair[crow(t,j)] + sum_j dl_j W_r[:,e_j] (+ shared dX_t),
// slots in order. bf16: block per token, thread per 8-column slice, the rows of
// up to 8 slots loaded together before they are summed.
template <typename TIO>
__global__ void __launch_bounds__(256) k_dx_reduce(const TIO* __restrict__ dx_pair, const int* __restrict__ crow_of_pair,
                                                   const int* __restrict__ topk_idx, const float* __restrict__ dl_sel,
                                                   const TIO* __restrict__ wrT, const TIO* __restrict__ sh_dx, int T,
                                                   int H, int k, TIO* __restrict__ dx) {
  pdl_wait();  // the previous kernel has completed and its writes are visible
  if constexpr (sizeof(TIO) == 2) {
    for (int t = blockIdx.x; t < T; t += gridDim.x) {
      const int64_t p0 = (int64_t)t * k;
      for (int i = threadIdx.x; i < H / 8; i += blockDim.x) {
        float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0}, f[8];
        for (int j0 = 0; j0 < k; j0 += 8) {
          uint4 u[8];
          int cr[8];
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            cr[jj] = (j0 + jj < k) ? crow_of_pair[p0 + j0 + jj] : -1;
            u[jj] = cr[jj] >= 0 ? reinterpret_cast<const uint4*>(dx_pair + (int64_t)cr[jj] * H)[i] : make_uint4(0, 0, 0, 0);
          }
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            if (cr[jj] >= 0) {
              bf16x8_to_f(u[jj], f);
#pragma unroll
              for (int q = 0; q < 8; ++q) acc[q] += f[q];
            }
          }
        }
        for (int j0 = 0; j0 < k; j0 += 8) {
          uint4 u[8];
#pragma unroll
          for (int jj = 0; jj < 8; ++jj)
            if (j0 + jj < k) u[jj] = reinterpret_cast<const uint4*>(wrT + (int64_t)topk_idx[p0 + j0 + jj] * H)[i];
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            if (j0 + jj < k) {
              const float d = dl_sel[p0 + j0 + jj];
              bf16x8_to_f(u[jj], f);
#pragma unroll
              for (int q = 0; q < 8; ++q) acc[q] = fmaf(d, f[q], acc[q]);
            }
          }
        }
        if (sh_dx) {
          bf16x8_to_f(reinterpret_cast<const uint4*>(sh_dx + (int64_t)t * H)[i], f);
#pragma unroll
          for (int q = 0; q < 8; ++q) acc[q] += f[q];
        }
        reinterpret_cast<uint4*>(dx + (int64_t)t * H)[i] = f_to_bf16x8(acc);
      }
    }
  } else {
    const int lane = threadIdx.x & 31;
    for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += (gridDim.x * blockDim.x) >> 5) {
      const int64_t p0 = (int64_t)t * k;
      for (int i = lane; i < H; i += 32) {
        float acc = 0.0f;
        for (int j = 0; j < k; ++j) {
          const int cr = crow_of_pair[p0 + j];
          if (cr >= 0) acc += io<TIO>::to_f(dx_pair[(int64_t)cr * H + i]);
        }
        for (int j = 0; j < k; ++j)
          acc = fmaf(dl_sel[p0 + j], io<TIO>::to_f(wrT[(int64_t)topk_idx[p0 + j] * H + i]), acc);
        if (sh_dx) acc += io<TIO>::to_f(sh_dx[(int64_t)t * H + i]);
        dx[(int64_t)t * H + i] = io<TIO>::cvt(acc);
      }
    }
  }
}

// ------------------------------------------------------------------ quota planner
// quota[e] = min(count[e], ceil(rho_num/rho_den * T*k/E)) (and <= budget[e] if given).
__global__ void k_plan_quota(const int* count, int E, int64_t pairs, int64_t rho_num, int64_t rho_den,
                             const int* budget, int* quota) {
  pdl_wait();  // the previous kernel has completed and its writes are visible
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= E) return;
  const int64_t den = rho_den * E;
  const int64_t q = (rho_num * pairs + den - 1) / den;
  int64_t v = count[e] < q ? count[e] : q;
  if (budget) v = v < budget[e] ? v : (budget[e] > 0 ? budget[e] : 0);
  quota[e] = (int)v;
}

// ------------------------------------------------------------------ launchers
cudaError_t launch_plan_quota(const int* count, int E, int64_t pairs, int64_t rho_num, int64_t rho_den,
                              const int* budget, int* quota, cudaStream_t st) {
  MOE_LAUNCH(k_plan_quota, (E + 255) / 256, 256, 0, st, count, E, pairs, rho_num, rho_den, budget, quota);
  return cudaGetLastError();
}

static int grid_for(int64_t warps, int num_sms) {
  const int64_t want = (warps + 7) / 8;
  return (int)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)num_sms * 16));
}

template <typename TIO>
cudaError_t launch_pair_score(const void* dy, const void* y_pair, const int* pair_of_row, const int* pad_total,
                              int64_t Rmax, const float* topk_w, const float* xnorm, int H, int k, float* g,
                              float* score, void* dy_perm, float* user_scores, int num_sms, cudaStream_t st) {
  MOE_LAUNCH(k_pair_score<TIO>, grid_for(Rmax, num_sms), 256, 0, st, reinterpret_cast<const TIO*>(dy), reinterpret_cast<const TIO*>(y_pair), pair_of_row, pad_total, topk_w, xnorm,
      H, k, g, score, reinterpret_cast<TIO*>(dy_perm), user_scores);
  return cudaGetLastError();
}

cudaError_t launch_select(const float* score, const int* count, const int* pad_off, const int* quota, int E,
                          int* ret_cidx, int* ret_count, int* status, cudaStream_t st) {
  MOE_LAUNCH(k_select, E, kSelThreads, 0, st, score, count, pad_off, quota, ret_cidx, ret_count, status);
  return cudaGetLastError();
}

cudaError_t launch_ret_scan(const int* ret_count, int E, int* ret_offset, int* ret_pad_off, int* ret_tile_off,
                            int* ret_src, int* user_offsets, cudaStream_t st, int* order, int* ret_tile_off2,
                            int4* tile_rec, int4* ord_rec, int4* tile_rec2) {
  MOE_LAUNCH(k_ret_scan, 1, 1024, 0, st, ret_count, E, ret_offset, ret_pad_off, ret_tile_off, ret_src, user_offsets, order,
                                 ret_tile_off2, tile_rec, ord_rec, tile_rec2);
  return cudaGetLastError();
}

cudaError_t launch_ret_index(const int* topk_idx, const int* rowp_of_pair, const int* row_of_pair,
                             const int* ret_cidx, const int* ret_offset, const int* ret_pad_off, int64_t P,
                             int* ret_src, int* crow_of_pair, int* ret_rows, int* user_rows, int num_sms,
                             cudaStream_t st) {
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>((P + 255) / 256, (int64_t)num_sms * 8));
  MOE_LAUNCH(k_ret_index, grid, 256, 0, st, topk_idx, rowp_of_pair, row_of_pair, ret_cidx, ret_offset, ret_pad_off, P,
                                    ret_src, crow_of_pair, ret_rows, user_rows);
  return cudaGetLastError();
}

template <typename TIO>
cudaError_t launch_compact_rows(const int* ret_src, const int* ret_pad_total, int64_t Rmax, const int* pair_of_row,
                                const float* topk_w, const void* x, const void* ab, const void* h, const void* dy,
                                int H, int F, int k, void* x_c, void* ab_c, void* h_c, void* dy_c, int num_sms,
                                cudaStream_t st) {
  MOE_LAUNCH(k_compact_rows<TIO>, grid_for(Rmax, num_sms), 256, 0, st, ret_src, ret_pad_total, pair_of_row, topk_w, reinterpret_cast<const TIO*>(x), reinterpret_cast<const TIO*>(ab),
      reinterpret_cast<const TIO*>(h), reinterpret_cast<const TIO*>(dy), H, F, k, reinterpret_cast<TIO*>(x_c),
      reinterpret_cast<TIO*>(ab_c), reinterpret_cast<TIO*>(h_c), reinterpret_cast<TIO*>(dy_c));
  return cudaGetLastError();
}

template <typename TIO>
cudaError_t launch_router_bwd(const float* g, const int* rowp_of_pair, const int* topk_idx, const float* topk_w,
                              int T, int Tpad, int E, int k, float* dl_sel, void* dl_dense, int num_sms,
                              cudaStream_t st) {
  MOE_LAUNCH(k_router_bwd<TIO>, grid_for(Tpad, num_sms), 256, 0, st, g, rowp_of_pair, topk_idx, topk_w, T, Tpad, E, k,
                                                             dl_sel, reinterpret_cast<TIO*>(dl_dense));
  return cudaGetLastError();
}

template <typename TIO>
cudaError_t launch_transpose(const void* in, int R, int Cc, void* out, cudaStream_t st) {
  dim3 grid((Cc + 31) / 32, (R + 31) / 32), block(32, 8);
  MOE_LAUNCH(k_transpose<TIO>, grid, block, 0, st, reinterpret_cast<const TIO*>(in), R, Cc, reinterpret_cast<TIO*>(out));
  return cudaGetLastError();
}

// bf16, k <= 8: warp per token, grid-stride. Lane j < k loads slot j's compact row,
// expert and router-logit gradient and shuffles hand them to the other lanes, so a warp
// needs no block barrier and many tokens are in flight per SM. Each lane owns 8
// consecutive columns per 256-column step and issues every slot's dx_pair and
// router-weight row loads of the step before it sums them. Same summation order as
// k_dx_reduce (kept slots ascending, then the router term slot by slot, then shared).
__global__ void __launch_bounds__(256) k_dx_reduce_k8(const __nv_bfloat16* __restrict__ dx_pair,
                                                      const int* __restrict__ crow_of_pair,
                                                      const int* __restrict__ topk_idx, const float* __restrict__ dl_sel,
                                                      const __nv_bfloat16* __restrict__ wrT,
                                                      const __nv_bfloat16* __restrict__ sh_dx, int T, int H, int k,
                                                      __nv_bfloat16* __restrict__ dx) {
  pdl_wait();  // the previous kernel has completed and its writes are visible
  const int lane = threadIdx.x & 31, wpb = blockDim.x >> 5;
  const int nv = H / 8;
  for (int t = blockIdx.x * wpb + (threadIdx.x >> 5); t < T; t += gridDim.x * wpb) {
    int c = -1, ex = 0;
    float d = 0.0f;
    if (lane < k) {
      c = crow_of_pair[(int64_t)t * k + lane];
      ex = topk_idx[(int64_t)t * k + lane];
      d = dl_sel[(int64_t)t * k + lane];
    }
    int cj[8], ej[8];
    float dj[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {  // lanes j >= k hold c = -1, d = 0
      cj[j] = __shfl_sync(0xffffffffu, c, j);
      ej[j] = __shfl_sync(0xffffffffu, ex, j);
      dj[j] = __shfl_sync(0xffffffffu, d, j);
    }
    for (int i = lane; i < nv; i += 32) {
      uint4 u[8], v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        u[j] = cj[j] >= 0 ? reinterpret_cast<const uint4*>(dx_pair + (int64_t)cj[j] * H)[i] : make_uint4(0, 0, 0, 0);
        v[j] = j < k ? reinterpret_cast<const uint4*>(wrT + (int64_t)ej[j] * H)[i] : make_uint4(0, 0, 0, 0);
      }
      float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0}, f[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (cj[j] >= 0) {
          bf16x8_to_f(u[j], f);
#pragma unroll
          for (int q = 0; q < 8; ++q) acc[q] += f[q];
        }
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (j < k) {
          bf16x8_to_f(v[j], f);
#pragma unroll
          for (int q = 0; q < 8; ++q) acc[q] = fmaf(dj[j], f[q], acc[q]);
        }
      }
      if (sh_dx) {
        bf16x8_to_f(reinterpret_cast<const uint4*>(sh_dx + (int64_t)t * H)[i], f);
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[q] += f[q];
      }
      reinterpret_cast<uint4*>(dx + (int64_t)t * H)[i] = f_to_bf16x8(acc);
    }
  }
}

template <typename TIO>
cudaError_t launch_dx_reduce(const void* dx_pair, const int* crow_of_pair, const int* topk_idx, const float* dl_sel,
                             const void* wrT, const void* sh_dx, int T, int H, int k, void* dx, int num_sms,
                             cudaStream_t st) {
  if (sizeof(TIO) == 2 && k <= 8) {
    // a warp per token in blocks of two warps, grid-stride with as many blocks as fit at
    // once: tokens spread over the SMs a warp at a time (blocks of eight warps left a
    // quarter of the SMs one block behind)
    constexpr int kThreads = 64;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_dx_reduce_k8, kThreads, 0) != cudaSuccess ||
        per_sm < 1)
      per_sm = 1;
    const int wpb = kThreads / 32;
    const int g =
        (int)std::max<int64_t>(1, std::min<int64_t>(((int64_t)T + wpb - 1) / wpb, (int64_t)num_sms * per_sm));
    MOE_LAUNCH(k_dx_reduce_k8, g, kThreads, 0, st, reinterpret_cast<const __nv_bfloat16*>(dx_pair), crow_of_pair, topk_idx, dl_sel,
                                      reinterpret_cast<const __nv_bfloat16*>(wrT),
                                      reinterpret_cast<const __nv_bfloat16*>(sh_dx), T, H, k,
                                      reinterpret_cast<__nv_bfloat16*>(dx));
    return cudaGetLastError();
  }
  const int grid = sizeof(TIO) == 2 ? (int)std::max<int64_t>(1, std::min<int64_t>(T, (int64_t)num_sms * 32))
                                    : grid_for(T, num_sms);
  MOE_LAUNCH(k_dx_reduce<TIO>, grid, 256, 0, st, reinterpret_cast<const TIO*>(dx_pair), crow_of_pair, topk_idx, dl_sel, reinterpret_cast<const TIO*>(wrT),
      reinterpret_cast<const TIO*>(sh_dx), T, H, k, reinterpret_cast<TIO*>(dx));
  return cudaGetLastError();
}

#define MOE_INST(TIO)                                                                                               \
  template cudaError_t launch_pair_score<TIO>(const void*, const void*, const int*, const int*, int64_t,           \
                                              const float*, const float*, int, int, float*, float*, void*, float*, \
                                              int, cudaStream_t);                                                  \
  template cudaError_t launch_compact_rows<TIO>(const int*, const int*, int64_t, const int*, const float*,         \
                                                const void*, const void*, const void*, const void*, int, int, int, \
                                                void*, void*, void*, void*, int, cudaStream_t);                    \
  template cudaError_t launch_router_bwd<TIO>(const float*, const int*, const int*, const float*, int, int, int,   \
                                              int, float*, void*, int, cudaStream_t);                              \
  template cudaError_t launch_transpose<TIO>(const void*, int, int, void*, cudaStream_t);                          \
  template cudaError_t launch_dx_reduce<TIO>(const void*, const int*, const int*, const float*, const void*,       \
                                             const void*, int, int, int, void*, int, cudaStream_t);
MOE_INST(float)
MOE_INST(__nv_bfloat16)
#undef MOE_INST

}  // namespace moe
