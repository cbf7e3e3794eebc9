// decode.cu -- the forward of the MoE layer for decode-sized token counts, fused
// into one persistent kernel (inference: nothing is kept for a backward).
//
// At a handful of tokens the layer is a weight stream: each token touches k experts,
// and their W_gate, W_up, W_down dominate the bytes. The unfused path runs a dozen
// short kernels whose launch, prologue and pipeline fill cost more than the stream.
// Here one cooperative launch (one CTA per SM, every CTA resident) runs four phases
// separated by grid-wide barriers:
//   R  router logits: CTA b computes logits[t, b], logits[t, b + G], ... over all of H
//      (CUDA cores), with the bias added;
//   G  every CTA takes the top-k and the renormalised softmax weights of every token
//      and builds the same slot table (the routed (token, expert) pairs sorted by
//      expert then token, then one slot per token for the shared expert); then units
//      (expert, 64 columns of F) stream all of H of W_gate and W_up through a ring of
//      four 32 KB shared-memory tiles (TMA, 128-byte swizzle) and meet the expert's
//      tokens in mma.sync m16n8k16 bf16 products with fp32 accumulation (gate and up in
//      two accumulators), and write h = silu(a) * b in bf16;
//   D  units (expert, 64 columns of H) stream all of F of W_down the same way and
//      write y for the expert's slots in fp32;
//   C  y[t] = sum_j w_tj y(t, j) (+ the shared expert), slots in order, rounded once.
// At most 16 tokens make the contractions 16 rows wide, so the weight stream, not the
// tensor rate, bounds them; no K is split, so no partial sums are reduced between
// phases. Every sum runs in a fixed order, so two calls give the same bits. Every wait
// (TMA landing, grid barrier) is bounded: a wait that runs out sets MOE_ERR_TIMEOUT in
// the status word and the kernel returns.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "decode.h"

namespace moe {

constexpr int kDecMaxT = 16;      // tokens (the mma M dimension)
constexpr int kDecThreads = 256;  // 8 warps: one 8-column n-tile of a 64-column unit each
constexpr int kDecStepRows = 256; // weight rows per ring step: four 64-row boxes
constexpr int kDecBufs = 6;       // weight tiles in flight per CTA
constexpr int kDecBoxRows = 64;
constexpr int kDecTileBytes = kDecStepRows * 128;            // 32 KB: 256 rows x 64 bf16
constexpr int kDecALd = kDecStepRows + 8;                    // A tile row stride (elements), padded
constexpr int kDecMaxE = 256;
constexpr int kDecMaxK = 16;  // T * k <= 256: one thread per routed pair when ranking them
constexpr int kDecMaxH = 4096;
constexpr uint64_t kDecWaitNs = 1000000000ull;                // 1 s

struct DecodeArgs {
  int T, H, F, E, k, Fs;
  const __nv_bfloat16* x;
  const __nv_bfloat16* w_router;
  const float* bias;
  __nv_bfloat16* y;
  int* topk_idx;      // workspace copy [T,k]
  float* topk_w;      // [T,k]
  int* user_idx;      // nullable
  float* user_w;      // nullable
  float* user_logits; // nullable [T,E]
  float* logits;      // [T][E] biased fp32 logits
  __nv_bfloat16* hbuf;  // [slots][Fm]
  float* ypair;       // [slots][H]
  float* part_g;      // [H / 256][slots][gate, up][Fm]: x Wg and x Wu over one 256-row chunk of H
  int smax;           // slot rows of part_g: T * k + T
  unsigned* sync;     // grid barrier counter (zeroed before the launch)
  int* status;
};

struct DecodeShared {
  __nv_bfloat16 a_tile[kDecMaxT * kDecALd];  // tokens x rows of the current step
  float red[kDecThreads / 32][kDecMaxT];     // router: one partial sum per warp and token
  int s_idx[kDecMaxT * kDecMaxK];
  float s_w[kDecMaxT * kDecMaxK];
  int slot_pair[kDecMaxT * kDecMaxK];        // routed slot -> pair t*k + j
  int slot_of_pair[kDecMaxT * kDecMaxK];
  int ex_id[kDecMaxT * kDecMaxK + 1];        // unit expert u -> expert id (shared: -1)
  int ex_first[kDecMaxT * kDecMaxK + 2];     // first slot of expert u; ex_first[n_u] = slots
  uint64_t bar[kDecBufs];
  int n_routed, n_u;
  int abort_flag;
};

// ------------------------------------------------------------------ small helpers
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2_trans(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}
// D = A (16x16, row) * B (16x8, col) + D, bf16 inputs, fp32 accumulators
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Grid-wide barrier number `phase` (1, 2, ...), in two halves so that a CTA can issue
// work between them: arrive (every CTA once: a release add after the CTA's own barrier)
// and wait (thread 0 polls with acquire loads). wait returns false when the wait ran
// out (or an earlier one did), after recording MOE_ERR_TIMEOUT.
__device__ __forceinline__ void dec_grid_arrive(const DecodeArgs& a, DecodeShared& sh) {
  __syncthreads();
  if (threadIdx.x == 0 && !sh.abort_flag)
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(a.sync), "r"(1u) : "memory");
}
__device__ bool dec_grid_wait(const DecodeArgs& a, DecodeShared& sh, unsigned phase) {
  if (threadIdx.x == 0 && !sh.abort_flag) {
    const unsigned target = phase * gridDim.x;
    if (ld_acquire_gpu(a.sync) < target) {
      const uint64_t t0 = globaltimer_ns();
      while (ld_acquire_gpu(a.sync) < target) {
        if (globaltimer_ns() - t0 > kDecWaitNs) {
          sh.abort_flag = 1;
          set_status(a.status, MOE_ERR_TIMEOUT);
          break;
        }
      }
    }
  }
  __syncthreads();
  return !sh.abort_flag;
}
__device__ __forceinline__ bool dec_grid_sync(const DecodeArgs& a, DecodeShared& sh, unsigned phase) {
  dec_grid_arrive(a, sh);
  return dec_grid_wait(a, sh, phase);
}

// d0 + d1 += (sh.a_tile, nrows columns) x (weight tile at wt, nrows rows x 64 columns):
// warp w takes the 16 x 8 block of columns 8w .. 8w+7 (rows = tokens). Even 16-row
// slices go to d0, odd ones to d1, so two mma chains are in flight; nrows is a multiple
// of 64.
__device__ __forceinline__ void step_mma(const DecodeShared& sh, uint32_t wt, int nrows, float (&d0)[4],
                                         float (&d1)[4]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t a_base = smem_u32(sh.a_tile);
#pragma unroll 2
  for (int kk = 0; kk < nrows; kk += 32) {
    uint32_t a0, a1, a2, a3, b0, b1, c0, c1, c2, c3, e0, e1;
    // A: matrices (rows 0-7, k 0-7), (8-15, 0-7), (0-7, 8-15), (8-15, 8-15)
    const int ar = lane & 15, ak = kk + ((lane >> 4) << 3);
    ldsm_x4(a_base + (uint32_t)((ar * kDecALd + ak) * 2), a0, a1, a2, a3);
    ldsm_x4(a_base + (uint32_t)((ar * kDecALd + ak + 16) * 2), c0, c1, c2, c3);
    // B: weight rows kk..kk+15, columns 8w..8w+7 (16-byte chunk w of each swizzled row)
    const int br = kk + (lane & 15), br2 = br + 16;
    ldsm_x2_trans(wt + (uint32_t)(br * 128 + ((warp ^ (br & 7)) << 4)), b0, b1);
    ldsm_x2_trans(wt + (uint32_t)(br2 * 128 + ((warp ^ (br2 & 7)) << 4)), e0, e1);
    mma_16816(d0, a0, a1, a2, a3, b0, b1);
    mma_16816(d1, c0, c1, c2, c3, e0, e1);
  }
}

// The weight ring: kDecBufs shared-memory tiles of at most 256 rows x 64 columns, filled
// by TMA in issue order and consumed in the same order. Every thread keeps the same copy
// of this state; thread 0 issues the copies.
struct Ring {
  int next_issue, next_use, inflight;
  uint32_t phase[kDecBufs];
};

__device__ __forceinline__ void ring_issue(DecodeShared& sh, uint8_t* tiles, Ring& r, const CUtensorMap* map,
                                           int row0, int col0, int nrows) {
  const int b = r.next_issue;
  r.next_issue = (b + 1) % kDecBufs;
  ++r.inflight;
  if (threadIdx.x == 0) {
    const int nbox = (nrows + kDecBoxRows - 1) / kDecBoxRows;
    fence_async_smem();  // this CTA's earlier reads of the buffer come before the copy
    mbar_arrive_expect_tx(&sh.bar[b], (uint32_t)(nbox * kDecBoxRows * 128));
    for (int x = 0; x < nbox; ++x)
      tma_load_2d(smem_u32(tiles + b * kDecTileBytes + x * kDecBoxRows * 128), map, smem_u32(&sh.bar[b]), col0,
                  row0 + x * kDecBoxRows);
  }
}

// Waits for the oldest tile in flight and returns its shared-memory address in wt; false
// after a wait ran out, once this CTA's other copies in flight have landed (so that its
// shared memory may be released).
__device__ __forceinline__ bool ring_wait(DecodeShared& sh, uint8_t* tiles, Ring& r, const DecodeArgs& a,
                                          uint32_t& wt) {
  const int b = r.next_use;
  const bool landed = mbar_wait_bounded(&sh.bar[b], r.phase[b], (volatile int*)&sh.abort_flag, kDecWaitNs);
  if (landed)
    r.phase[b] ^= 1u;
  else
    set_status(a.status, MOE_ERR_TIMEOUT);
  __syncthreads();
  if (sh.abort_flag) {
    if (threadIdx.x == 0)
      for (int q = landed ? 1 : 0; q < r.inflight; ++q) {
        const int bq = (b + q) % kDecBufs;
        mbar_wait_timed(&sh.bar[bq], r.phase[bq], 200000000ull);
      }
    __syncthreads();
    return false;
  }
  wt = smem_u32(tiles + b * kDecTileBytes);
  return true;
}

// After the barrier that ends the step: the oldest tile's buffer is free again.
__device__ __forceinline__ void ring_release(Ring& r) {
  r.next_use = (r.next_use + 1) % kDecBufs;
  --r.inflight;
}

// A tile of the current step: up to 16 rows (the unit's tokens) x 256 columns, two
// 16-byte pieces per thread, staged in registers one tile ahead.
__device__ __forceinline__ void a_store(DecodeShared& sh, const uint4 (&v)[2]) {
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int idx = threadIdx.x + q * kDecThreads, r = idx >> 5, c = idx & 31;
    *reinterpret_cast<uint4*>(sh.a_tile + r * kDecALd + c * 8) = v[q];
  }
}

// ------------------------------------------------------------------ the kernel
__global__ void __launch_bounds__(kDecThreads, 1)
    k_decode_fwd(const __grid_constant__ CUtensorMap tm_gate, const __grid_constant__ CUtensorMap tm_up,
                 const __grid_constant__ CUtensorMap tm_down, const __grid_constant__ CUtensorMap tm_sgate,
                 const __grid_constant__ CUtensorMap tm_sup, const __grid_constant__ CUtensorMap tm_sdown,
                 const DecodeArgs a) {
  extern __shared__ uint8_t dec_smem_raw[];
  uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dec_smem_raw) + 1023) & ~uintptr_t(1023));
  DecodeShared& sh = *reinterpret_cast<DecodeShared*>(tiles + kDecBufs * kDecTileBytes);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int T = a.T, H = a.H, F = a.F, E = a.E, k = a.k, Fs = a.Fs;
  const int Fm = max(F, Fs);
  const int G = gridDim.x;
  const int P = T * k;

  if (tid == 0) {
    for (int b = 0; b < kDecBufs; ++b) mbar_init(&sh.bar[b], 1);
    sh.abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  // ---------------------------------------------------------------- R: router logits
  // CTA b takes experts b, b + G, ...; thread i the rows 8i .. 8i+7 of each 2048-row
  // stretch of H (one column element of W_router per row, a 16-byte load of x per token)
  for (int e = blockIdx.x; e < E; e += G) {
    float acc[kDecMaxT];
#pragma unroll
    for (int t = 0; t < kDecMaxT; ++t) acc[t] = 0.0f;
    for (int r0 = tid * 8; r0 < H; r0 += kDecThreads * 8) {
      float wv[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) wv[q] = __bfloat162float(a.w_router[(int64_t)(r0 + q) * E + e]);
      uint4 xr[kDecMaxT];  // every token's 16 bytes in flight before the sums
#pragma unroll
      for (int t = 0; t < kDecMaxT; ++t)
        xr[t] = t < T ? *reinterpret_cast<const uint4*>(a.x + (int64_t)t * H + r0) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int t = 0; t < kDecMaxT; ++t) {
        float xv[8];
        bf16x8_to_f(xr[t], xv);
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[t] = fmaf(xv[q], wv[q], acc[t]);
      }
    }
    // a fixed butterfly inside each warp, then the eight warps in order, then the bias
#pragma unroll
    for (int t = 0; t < kDecMaxT; ++t) {
      float v = acc[t];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0 && t < T) sh.red[warp][t] = v;
    }
    __syncthreads();
    if (tid < T) {
      float l = 0.0f;
#pragma unroll
      for (int w = 0; w < kDecThreads / 32; ++w) l += sh.red[w][tid];
      l += a.bias ? a.bias[e] : 0.0f;
      a.logits[tid * E + e] = l;
      if (a.user_logits) a.user_logits[tid * E + e] = l;
    }
    __syncthreads();
  }
  if (!dec_grid_sync(a, sh, 1)) return;

  // ---------------------------------------------------------------- top-k and slots
  {
    // warp w takes tokens w, w + 8, ...: lane l holds the logits of experts l, l + 32, ...
    // as order-preserving keys (NaN reads as -inf, -0 as +0); each of k rounds takes the largest
    // key still free, ties to the lower expert index, with two warp reductions
    for (int t = warp; t < T; t += kDecThreads / 32) {
      float v[kDecMaxE / 32];
      uint32_t key[kDecMaxE / 32];
#pragma unroll
      for (int i = 0; i < kDecMaxE / 32; ++i) {
        const int e = lane + 32 * i;
        v[i] = e < E ? __ldcg(a.logits + t * E + e) : -INFINITY;
      }
      uint32_t free_mask = 0;
#pragma unroll
      for (int i = 0; i < kDecMaxE / 32; ++i) {
        float l = v[i];
        if (l != l) l = -INFINITY;
        if (l == 0.0f) l = 0.0f;  // -0 ties with +0
        v[i] = l;
        const uint32_t b = __float_as_uint(l);
        key[i] = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
        if (lane + 32 * i < E) free_mask |= 1u << i;
      }
      float lmax = 0.0f, sum = 0.0f, my_v = 0.0f;
      int my_e = 0;
      for (int j = 0; j < k; ++j) {
        uint32_t bk = 0;
        int bi = -1;
#pragma unroll
        for (int i = 0; i < kDecMaxE / 32; ++i)  // ascending i: a tie keeps the lower expert
          if (((free_mask >> i) & 1u) && (bi < 0 || key[i] > bk)) {
            bk = key[i];
            bi = i;
          }
        const uint32_t kmax = __reduce_max_sync(0xffffffffu, bi >= 0 ? bk : 0u);
        const int cand = (bi >= 0 && bk == kmax) ? lane + 32 * bi : 0x7fffffff;
        const int we = (int)__reduce_min_sync(0xffffffffu, (unsigned)cand);
        float wv = 0.0f;
#pragma unroll
        for (int i = 0; i < kDecMaxE / 32; ++i)
          if (lane + 32 * i == we) wv = v[i];
        wv = __shfl_sync(0xffffffffu, wv, we & 31);
        if ((we & 31) == lane) free_mask &= ~(1u << (we >> 5));
        if (j == 0) lmax = wv;
        sum += expf(wv - lmax);
        if (lane == j) {
          my_e = we;
          my_v = wv;
        }
      }
      if (lane < k) {
        const float wt = expf(my_v - lmax) * (1.0f / sum);
        sh.s_idx[t * k + lane] = my_e;
        sh.s_w[t * k + lane] = wt;
        if (blockIdx.x == 0) {
          a.topk_idx[t * k + lane] = my_e;
          a.topk_w[t * k + lane] = wt;
          if (a.user_idx) a.user_idx[t * k + lane] = my_e;
          if (a.user_w) a.user_w[t * k + lane] = wt;
        }
      }
    }
    __syncthreads();
    // routed slots: pairs sorted by (expert, token); a pair's rank is its slot
    if (tid < P) {
      const int e = sh.s_idx[tid];
      int rank = 0;
      for (int q = 0; q < P; ++q) {
        const int eq = sh.s_idx[q];
        rank += (eq < e) || (eq == e && q < tid);
      }
      sh.slot_pair[rank] = tid;
      sh.slot_of_pair[tid] = rank;
    }
    __syncthreads();
    // experts in slot order: a slot opens a new expert when its expert differs from the previous slot's
    const int first = (tid < P) && (tid == 0 || sh.s_idx[sh.slot_pair[tid]] != sh.s_idx[sh.slot_pair[tid - 1]]);
    int nfirst;
    const int u = block_excl_scan(first ? 1 : 0, &nfirst);
    if (first) {
      sh.ex_id[u] = sh.s_idx[sh.slot_pair[tid]];
      sh.ex_first[u] = tid;
    }
    if (tid == 0) {
      sh.n_routed = nfirst;
      sh.ex_first[nfirst] = P;
      int nu = nfirst;
      if (Fs > 0) {  // the shared expert: one slot per token after the routed ones
        sh.ex_id[nfirst] = -1;
        sh.ex_first[nfirst + 1] = P + T;
        ++nu;
      }
      sh.n_u = nu;
    }
    __syncthreads();
  }
  const int n_routed = sh.n_routed, n_u = sh.n_u;
  auto slot_tok = [&](int s) { return s < P ? sh.slot_pair[s] / k : s - P; };
  const int KC1 = (H + kDecStepRows - 1) / kDecStepRows;  // 256-row steps of H

  Ring ring;
  ring.next_issue = ring.next_use = ring.inflight = 0;
#pragma unroll
  for (int b = 0; b < kDecBufs; ++b) ring.phase[b] = 0;
  auto slot_rows = [&](int u, int& s0, int& ns) {
    s0 = sh.ex_first[u];
    ns = sh.ex_first[u + 1] - s0;
  };

  // ---------------------------------------------------------------- G: x Wg, x Wu per 256-row chunk
  // Steps (expert u, chunk kc of H, 64-column block fb of F_u, gate|up) in that order, an
  // even share of them per CTA: at any moment the CTAs stream neighbouring column blocks
  // of the same weight rows. Each step's 16 x 64 product (a 256-row partial sum) is
  // stored in part_g; phase H adds the chunks.
  {
    const int nfb_r = F / 64, nfb_s = Fs / 64;
    auto nfb = [&](int u) { return u < n_routed ? nfb_r : nfb_s; };
    const int64_t per_r = (int64_t)KC1 * nfb_r * 2;
    const int64_t total = (int64_t)n_routed * per_r + (Fs > 0 ? (int64_t)KC1 * nfb_s * 2 : 0);
    const int64_t s0 = total * blockIdx.x / G, s1 = total * (blockIdx.x + 1) / G;
    struct Cur {
      int u, kc, fb, gu;
    };
    auto at = [&](int64_t g) {
      Cur c;
      int64_t rem;
      if (g < (int64_t)n_routed * per_r) {
        c.u = (int)(g / per_r);
        rem = g - (int64_t)c.u * per_r;
      } else {
        c.u = n_routed;
        rem = g - (int64_t)n_routed * per_r;
      }
      const int nf2 = nfb(c.u) * 2;
      c.kc = (int)(rem / nf2);
      const int r2 = (int)(rem - (int64_t)c.kc * nf2);
      c.fb = r2 >> 1;
      c.gu = r2 & 1;
      return c;
    };
    auto advance = [&](Cur& c) {
      if (++c.gu == 2) {
        c.gu = 0;
        if (++c.fb == nfb(c.u)) {
          c.fb = 0;
          if (++c.kc == KC1) {
            c.kc = 0;
            ++c.u;
          }
        }
      }
    };
    auto issue = [&](const Cur& c) {
      const int k0 = c.kc * kDecStepRows, nrows = min(kDecStepRows, H - k0);
      if (c.u < n_routed)
        ring_issue(sh, tiles, ring, c.gu ? &tm_up : &tm_gate, sh.ex_id[c.u] * H + k0, c.fb * 64, nrows);
      else
        ring_issue(sh, tiles, ring, c.gu ? &tm_sup : &tm_sgate, k0, c.fb * 64, nrows);
    };
    // x rows of expert u's tokens, the 256 columns of chunk kc
    auto load_a = [&](int u, int kc, uint4 (&v)[2]) {
      const int k0 = kc * kDecStepRows, nk = min(kDecStepRows, H - k0);
      int sb, ns;
      slot_rows(u, sb, ns);
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int idx = tid + q * kDecThreads, r = idx >> 5, c = idx & 31;
        v[q] = make_uint4(0, 0, 0, 0);
        if (r < ns && c * 8 < nk) v[q] = *reinterpret_cast<const uint4*>(a.x + (int64_t)slot_tok(sb + r) * H + k0 + c * 8);
      }
    };
    if (s0 < s1) {
      Cur ic = at(s0);
      int64_t left = s1 - s0;
      for (; ring.inflight < kDecBufs && left > 0; --left, advance(ic)) issue(ic);
      Cur cc = at(s0);
      // the A tile after the current one: (u, kc + 1), else (u + 1, 0), if this CTA reaches it
      int nu = cc.u, nkc = cc.kc;
      int64_t ng = s0 - (int64_t)((cc.fb * 2) + cc.gu);  // first step of the current A tile
      uint4 av[2];
      load_a(cc.u, cc.kc, av);
      for (int64_t g = s0; g < s1; ++g, advance(cc)) {
        if (g == s0 || (cc.fb == 0 && cc.gu == 0)) {
          a_store(sh, av);  // the previous readers of the A tile passed the last barrier
          ng += nfb(nu) * 2;
          if (++nkc == KC1) {
            nkc = 0;
            ++nu;
          }
          if (ng < s1) load_a(nu, nkc, av);
        }
        uint32_t wt;
        if (!ring_wait(sh, tiles, ring, a, wt)) return;
        const int nrows = min(kDecStepRows, H - cc.kc * kDecStepRows);
        float d0[4] = {0, 0, 0, 0}, d1[4] = {0, 0, 0, 0};
        step_mma(sh, wt, nrows, d0, d1);
        int sb, ns;
        slot_rows(cc.u, sb, ns);
        const int col = cc.fb * 64 + warp * 8 + (lane & 3) * 2, r0 = lane >> 2;
        float* pg = a.part_g + ((int64_t)cc.kc * a.smax * 2 + cc.gu) * Fm + col;
        if (r0 < ns)
          *reinterpret_cast<float2*>(pg + (int64_t)(sb + r0) * 2 * Fm) = make_float2(d0[0] + d1[0], d0[1] + d1[1]);
        if (r0 + 8 < ns)
          *reinterpret_cast<float2*>(pg + (int64_t)(sb + r0 + 8) * 2 * Fm) =
              make_float2(d0[2] + d1[2], d0[3] + d1[3]);
        __syncthreads();  // this buffer (and, at an A step, the A tile) is free again
        ring_release(ring);
        if (left > 0) {
          issue(ic);
          advance(ic);
          --left;
        }
      }
    }
  }

  // ---------------------------------------------------------------- D: y = h Wd (its first copies)
  // Units (expert u, 64 columns hb of H), CTA b taking units b, b + G, ...; each streams
  // all F_u rows of W_down in 256-row steps. The first tiles are issued now, before the
  // barriers, so they land while phase H runs.
  const int nhb = H / 64;
  const int nunits_d = n_u * nhb;
  const int mine_d = nunits_d > (int)blockIdx.x ? (nunits_d - (int)blockIdx.x + G - 1) / G : 0;
  auto fu = [&](int u) { return u < n_routed ? F : Fs; };
  auto kc2 = [&](int u) { return (fu(u) + kDecStepRows - 1) / kDecStepRows; };
  struct DCur {
    int li, fk;
  };
  auto d_unit = [&](const DCur& c) { return (int)blockIdx.x + c.li * G; };
  auto d_advance = [&](DCur& c) {
    if (++c.fk == kc2(d_unit(c) / nhb)) {
      c.fk = 0;
      ++c.li;
    }
  };
  auto d_issue = [&](const DCur& c) {
    const int i = d_unit(c), u = i / nhb, hb = i % nhb, k0 = c.fk * kDecStepRows;
    const int nrows = min(kDecStepRows, fu(u) - k0);
    if (u < n_routed)
      ring_issue(sh, tiles, ring, &tm_down, sh.ex_id[u] * F + k0, hb * 64, nrows);
    else
      ring_issue(sh, tiles, ring, &tm_sdown, k0, hb * 64, nrows);
  };
  DCur dic{0, 0};
  dec_grid_arrive(a, sh);
  for (; ring.inflight < kDecBufs && dic.li < mine_d; d_advance(dic)) d_issue(dic);
  if (!dec_grid_wait(a, sh, 2)) {
    if (tid == 0)  // let the copies already issued land before the shared memory is released
      for (int q = 0; q < ring.inflight; ++q) {
        const int bq = (ring.next_use + q) % kDecBufs;
        mbar_wait_timed(&sh.bar[bq], ring.phase[bq], 200000000ull);
      }
    __syncthreads();
    return;
  }

  // ---------------------------------------------------------------- H: h = silu(sum_kc g) * (sum_kc u)
  {
    const int S = n_routed > 0 ? sh.ex_first[n_u] : 0;
    const int f8 = Fm / 8;
    // item idx -> CTA idx % G, so that a few items still use many SMs
    for (int idx = (int)blockIdx.x + G * tid; idx < S * f8; idx += G * kDecThreads) {
      const int sl = idx / f8, f = (idx - sl * f8) * 8;
      if (f >= (sl < P ? F : Fs)) continue;
      float gs[8], us[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) gs[q] = us[q] = 0.0f;
#pragma unroll 8
      for (int kc = 0; kc < KC1; ++kc) {  // chunks in order
        const float* pg = a.part_g + (((int64_t)kc * a.smax + sl) * 2) * Fm + f;
        const float4 g0 = __ldcg(reinterpret_cast<const float4*>(pg));
        const float4 g1 = __ldcg(reinterpret_cast<const float4*>(pg + 4));
        const float4 u0 = __ldcg(reinterpret_cast<const float4*>(pg + Fm));
        const float4 u1 = __ldcg(reinterpret_cast<const float4*>(pg + Fm + 4));
        gs[0] += g0.x; gs[1] += g0.y; gs[2] += g0.z; gs[3] += g0.w;
        gs[4] += g1.x; gs[5] += g1.y; gs[6] += g1.z; gs[7] += g1.w;
        us[0] += u0.x; us[1] += u0.y; us[2] += u0.z; us[3] += u0.w;
        us[4] += u1.x; us[5] += u1.y; us[6] += u1.z; us[7] += u1.w;
      }
      float h[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) h[q] = gs[q] * sigmoidf_(gs[q]) * us[q];
      *reinterpret_cast<uint4*>(a.hbuf + (int64_t)sl * Fm + f) = f_to_bf16x8(h);
    }
  }
  if (!dec_grid_sync(a, sh, 3)) {
    if (tid == 0)
      for (int q = 0; q < ring.inflight; ++q) {
        const int bq = (ring.next_use + q) % kDecBufs;
        mbar_wait_timed(&sh.bar[bq], ring.phase[bq], 200000000ull);
      }
    __syncthreads();
    return;
  }

  // ---------------------------------------------------------------- D: y = h Wd
  {
    // h rows of unit i's slots, the 256 columns of step fk
    auto load_a = [&](const DCur& c, uint4 (&v)[2]) {
      const int u = d_unit(c) / nhb, k0 = c.fk * kDecStepRows, nk = min(kDecStepRows, fu(u) - k0);
      int sb, ns;
      slot_rows(u, sb, ns);
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int idx = tid + q * kDecThreads, r = idx >> 5, c8 = idx & 31;
        v[q] = make_uint4(0, 0, 0, 0);
        if (r < ns && c8 * 8 < nk)
          v[q] = __ldcg(reinterpret_cast<const uint4*>(a.hbuf + (int64_t)(sb + r) * Fm + k0 + c8 * 8));
      }
    };
    float d0[4] = {0, 0, 0, 0}, d1[4] = {0, 0, 0, 0};
    uint4 av[2];
    DCur cc{0, 0}, ac{0, 0};
    if (mine_d > 0) load_a(ac, av);
    for (; cc.li < mine_d; d_advance(cc)) {
      a_store(sh, av);  // every step starts an A tile; its previous readers passed the last barrier
      d_advance(ac);
      if (ac.li < mine_d) load_a(ac, av);
      uint32_t wt;
      if (!ring_wait(sh, tiles, ring, a, wt)) return;
      const int i = d_unit(cc), u = i / nhb;
      step_mma(sh, wt, min(kDecStepRows, fu(u) - cc.fk * kDecStepRows), d0, d1);
      if (cc.fk + 1 == kc2(u)) {  // the unit's last step: its y rows
        const int hb = i % nhb;
        int sb, ns;
        slot_rows(u, sb, ns);
        const int col = hb * 64 + warp * 8 + (lane & 3) * 2, r0 = lane >> 2;
        if (r0 < ns)
          *reinterpret_cast<float2*>(a.ypair + (int64_t)(sb + r0) * H + col) = make_float2(d0[0] + d1[0], d0[1] + d1[1]);
        if (r0 + 8 < ns)
          *reinterpret_cast<float2*>(a.ypair + (int64_t)(sb + r0 + 8) * H + col) =
              make_float2(d0[2] + d1[2], d0[3] + d1[3]);
#pragma unroll
        for (int q = 0; q < 4; ++q) d0[q] = d1[q] = 0.0f;
      }
      __syncthreads();  // this buffer and the A tile are free again
      ring_release(ring);
      if (dic.li < mine_d) {
        d_issue(dic);
        d_advance(dic);
      }
    }
  }
  if (!dec_grid_sync(a, sh, 4)) return;

  // ---------------------------------------------------------------- C: combine
  for (int idx = blockIdx.x * kDecThreads + tid; idx < T * (H / 4); idx += G * kDecThreads) {
    const int t = idx / (H / 4), c = (idx % (H / 4)) * 4;
    float4 v[kDecMaxK];
#pragma unroll
    for (int j = 0; j < kDecMaxK; ++j)  // every slot's row loaded before the sum
      if (j < k) v[j] = __ldcg(reinterpret_cast<const float4*>(a.ypair + (int64_t)sh.slot_of_pair[t * k + j] * H + c));
    float acc[4] = {0, 0, 0, 0};
#pragma unroll
    for (int j = 0; j < kDecMaxK; ++j) {  // slots j ascending, then the shared expert
      if (j < k) {
        const float w = sh.s_w[t * k + j];
        acc[0] = fmaf(w, v[j].x, acc[0]);
        acc[1] = fmaf(w, v[j].y, acc[1]);
        acc[2] = fmaf(w, v[j].z, acc[2]);
        acc[3] = fmaf(w, v[j].w, acc[3]);
      }
    }
    if (Fs > 0) {
      const float4 sv = __ldcg(reinterpret_cast<const float4*>(a.ypair + (int64_t)(P + t) * H + c));
      acc[0] += sv.x;
      acc[1] += sv.y;
      acc[2] += sv.z;
      acc[3] += sv.w;
    }
    __nv_bfloat162* out = reinterpret_cast<__nv_bfloat162*>(a.y + (int64_t)t * H + c);
    out[0] = __floats2bfloat162_rn(acc[0], acc[1]);
    out[1] = __floats2bfloat162_rn(acc[2], acc[3]);
  }
}

// ------------------------------------------------------------------ host side
static PFN_cuTensorMapEncodeTiled_v12000 dec_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// [rows, cols] bf16, boxes of 64 rows x 64 columns, 128-byte swizzle
static bool dec_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols) {
  auto fn = dec_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)kDecBoxRows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// rows of the slot-indexed buffers: the T * k routed pairs and T shared-expert tokens
static int64_t dec_slots(int64_t T, int64_t k) { return T * k + T; }

size_t decode_scratch_bytes(int64_t T, int64_t H, int64_t F, int64_t E, int64_t k, int64_t Fs) {
  const int64_t Fm = F > Fs ? F : Fs, S = dec_slots(T, k), KC1 = (H + kDecStepRows - 1) / kDecStepRows;
  auto up = [](int64_t n) { return (size_t)((n + 255) / 256 * 256); };
  return up(T * E * 4) + up(S * Fm * 2) + up(S * H * 4) + up(KC1 * S * 2 * Fm * 4) + 256;
}

bool decode_supported(int64_t T, int64_t H, int64_t F, int64_t E, int64_t k, int64_t Fs) {
  return T >= 1 && T <= kDecMaxT && E <= kDecMaxE && k <= kDecMaxK && H <= kDecMaxH && F <= kDecMaxH &&
         Fs <= kDecMaxH && H % 64 == 0 && F % 64 == 0 && Fs % 64 == 0;
}

cudaError_t launch_decode_fwd(int T, int H, int F, int E, int k, int Fs, const void* x, const void* w_router,
                              const float* bias, const void* w_gate, const void* w_up, const void* w_down,
                              const void* ws_gate, const void* ws_up, const void* ws_down, void* y, int* topk_idx,
                              float* topk_w, int* user_idx, float* user_w, float* user_logits, void* scratch,
                              int* status, int num_sms, cudaStream_t st) {
  const int64_t Fm = F > Fs ? F : Fs, S = dec_slots(T, k), KC1 = (H + kDecStepRows - 1) / kDecStepRows;
  auto up = [](int64_t n) { return (int64_t)((n + 255) / 256 * 256); };
  char* b = static_cast<char*>(scratch);
  DecodeArgs a;
  a.T = T; a.H = H; a.F = F; a.E = E; a.k = k; a.Fs = Fs;
  a.x = static_cast<const __nv_bfloat16*>(x);
  a.w_router = static_cast<const __nv_bfloat16*>(w_router);
  a.bias = bias;
  a.y = static_cast<__nv_bfloat16*>(y);
  a.topk_idx = topk_idx;
  a.topk_w = topk_w;
  a.user_idx = user_idx;
  a.user_w = user_w;
  a.user_logits = user_logits;
  a.logits = reinterpret_cast<float*>(b);
  b += up((int64_t)T * E * 4);
  a.hbuf = reinterpret_cast<__nv_bfloat16*>(b);
  b += up(S * Fm * 2);
  a.ypair = reinterpret_cast<float*>(b);
  b += up(S * H * 4);
  a.part_g = reinterpret_cast<float*>(b);
  a.smax = (int)S;
  b += up(KC1 * S * 2 * Fm * 4);
  a.sync = reinterpret_cast<unsigned*>(b);
  a.status = status;
  cudaError_t e = cudaMemsetAsync(a.sync, 0, sizeof(unsigned), st);
  if (e != cudaSuccess) return e;
  CUtensorMap mg, mu, md, msg, msu, msd;
  bool ok = dec_map(&mg, w_gate, (int64_t)E * H, F) && dec_map(&mu, w_up, (int64_t)E * H, F) &&
            dec_map(&md, w_down, (int64_t)E * F, H);
  if (Fs > 0)
    ok = ok && dec_map(&msg, ws_gate, H, Fs) && dec_map(&msu, ws_up, H, Fs) && dec_map(&msd, ws_down, Fs, H);
  else
    msg = msu = msd = mg;  // unused without a shared expert
  if (!ok) return cudaErrorInvalidValue;
  const int smem = kDecBufs * kDecTileBytes + (int)sizeof(DecodeShared) + 1024;
  // once per device: the shared-memory attribute, and that one CTA per SM fits (all CTAs
  // of the cooperative grid must be resident at once)
  static std::mutex setup_mu;
  static bool ready[64] = {};
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  {
    std::lock_guard<std::mutex> lk(setup_mu);
    if (dev < 0 || dev >= 64 || !ready[dev]) {
      e = cudaFuncSetAttribute(k_decode_fwd, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return e;
      int per_sm = 0;
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_decode_fwd, kDecThreads, smem);
      if (e != cudaSuccess) return e;
      if (per_sm < 1) return cudaErrorInvalidConfiguration;
      if (dev >= 0 && dev < 64) ready[dev] = true;
    }
  }
  void* args[] = {&mg, &mu, &md, &msg, &msu, &msd, &a};
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(k_decode_fwd), dim3(num_sms), dim3(kDecThreads),
                                     args, (size_t)smem, st);
}

}  // namespace moe
