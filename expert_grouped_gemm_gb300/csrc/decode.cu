// decode.cu -- the forward of the MoE layer for decode-sized token counts, fused
// into one persistent kernel (inference: nothing is kept for a backward).
//
// At a handful of tokens the layer is a weight stream: each token touches k experts,
// and their W_gate, W_up, W_down dominate the bytes. The unfused path runs a dozen
// short kernels whose launch, prologue and pipeline fill cost more than the stream.
// Here one cooperative launch (one CTA per SM, every CTA resident) runs four phases
// separated by grid-wide barriers:
//   R  router logits: CTA b computes logits[t, 8b .. 8b+7] over all of H (CUDA cores),
//      with the bias added;
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
constexpr int kDecBufs = 4;       // weight tiles in flight per CTA
constexpr int kDecBoxRows = 64;
constexpr int kDecTileBytes = kDecStepRows * 128;            // 32 KB: 256 rows x 64 bf16
constexpr int kDecALd = kDecStepRows + 8;                    // A tile row stride (elements), padded
constexpr int kDecMaxE = 256;
constexpr int kDecMaxK = 16;  // T * k <= 256: one thread per routed pair when ranking them
constexpr int kDecMaxSlots = kDecMaxT * kDecMaxK + kDecMaxT;  // routed pairs + shared-expert tokens
constexpr int kDecRouterE = 8;                                // experts per router unit
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
  unsigned* sync;     // grid barrier counter (zeroed before the launch)
  int* status;
};

struct DecodeShared {
  __nv_bfloat16 a_tile[kDecMaxT * kDecALd];  // tokens x rows of the current step
  float red[32][kDecMaxT][kDecRouterE];      // router: partial sums of 32 row groups
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

// Grid-wide barrier number `phase` (1, 2, ...): every CTA arrives once; returns false
// when the wait ran out (or an earlier wait did), after recording MOE_ERR_TIMEOUT.
__device__ bool dec_grid_sync(const DecodeArgs& a, DecodeShared& sh, unsigned phase) {
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!sh.abort_flag) {
      __threadfence();
      atomicAdd(a.sync, 1u);
      const unsigned target = phase * gridDim.x;
      const uint64_t t0 = globaltimer_ns();
      while (ld_acquire_gpu(a.sync) < target) {
        if (globaltimer_ns() - t0 > kDecWaitNs) {
          sh.abort_flag = 1;
          set_status(a.status, MOE_ERR_TIMEOUT);
          break;
        }
        __nanosleep(32);
      }
      __threadfence();
    }
  }
  __syncthreads();
  return !sh.abort_flag;
}

// d += (sh.a_tile, nrows columns) x (weight tile at wt, nrows rows x 64 columns): warp w
// takes the 16 x 8 block of columns 8w .. 8w+7 (rows = tokens).
__device__ __forceinline__ void step_mma(const DecodeShared& sh, uint32_t wt, int nrows, float (&d)[4]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t a_base = smem_u32(sh.a_tile);
#pragma unroll 4
  for (int kk = 0; kk < nrows; kk += 16) {
    uint32_t a0, a1, a2, a3, b0, b1;
    // A: matrices (rows 0-7, k 0-7), (8-15, 0-7), (0-7, 8-15), (8-15, 8-15)
    const int ar = lane & 15, ak = kk + ((lane >> 4) << 3);
    ldsm_x4(a_base + (uint32_t)((ar * kDecALd + ak) * 2), a0, a1, a2, a3);
    // B: weight rows kk..kk+15, columns 8w..8w+7 (16-byte chunk w of each swizzled row)
    const int br = kk + (lane & 15);
    ldsm_x2_trans(wt + (uint32_t)(br * 128 + ((warp ^ (br & 7)) << 4)), b0, b1);
    mma_16816(d, a0, a1, a2, a3, b0, b1);
  }
}

// A weight-streaming phase: this CTA's units (blockIdx.x + li * gridDim.x < nunits), each
// a sequence of steps; step (unit i, s) is a tile of at most 256 weight rows x 64 columns
// (step_info: tensor map, first row, column, rows) that meets the A tile of the unit's
// tokens (needs_a(i, s): the step starts a new A tile; load_a / store_a move it through
// registers one A tile ahead). Four weight tiles are in flight. mma(i, s, wt, nrows)
// accumulates; done(i) writes the unit's result. Returns false after a wait ran out.
template <typename NSteps, typename StepInfo, typename NeedsA, typename LoadA, typename StoreA, typename Mma,
          typename Done>
__device__ bool stream_steps(DecodeShared& sh, uint8_t* tiles, uint32_t (&bar_phase)[kDecBufs], int nunits,
                             const DecodeArgs& a, NSteps nsteps, StepInfo step_info, NeedsA needs_a, LoadA load_a,
                             StoreA store_a, Mma mma, Done done) {
  const int G = gridDim.x;
  const int mine = nunits > (int)blockIdx.x ? (nunits - (int)blockIdx.x + G - 1) / G : 0;
  if (mine == 0) return true;
  auto unit = [&](int li) { return (int)blockIdx.x + li * G; };
  // cursor over this CTA's steps
  struct Cur {
    int li, s;
  };
  auto advance = [&](Cur& c) {
    if (++c.s >= nsteps(unit(c.li))) {
      c.s = 0;
      ++c.li;
    }
  };
  int slot_b = 0;  // ring slot of the next step to issue
  auto issue = [&](const Cur& c) {  // thread 0: the weight boxes of step c
    const CUtensorMap* map;
    int row0, col0, nrows;
    step_info(unit(c.li), c.s, map, row0, col0, nrows);
    const int b = slot_b;
    slot_b = (slot_b + 1) % kDecBufs;
    const int nbox = (nrows + kDecBoxRows - 1) / kDecBoxRows;
    if (nbox == 0) {
      mbar_arrive(&sh.bar[b]);
      return;
    }
    fence_async_smem();  // this CTA's earlier reads of the buffer come before the copy
    mbar_arrive_expect_tx(&sh.bar[b], (uint32_t)(nbox * kDecBoxRows * 128));
    for (int x = 0; x < nbox; ++x)
      tma_load_2d(smem_u32(tiles + b * kDecTileBytes + x * kDecBoxRows * 128), map, smem_u32(&sh.bar[b]), col0,
                  row0 + x * kDecBoxRows);
  };
  Cur ic{0, 0}, cc{0, 0}, ac{0, 0};  // issue, consume and A-load cursors
  int inflight = 0;
  if (threadIdx.x == 0)
    for (; inflight < kDecBufs && ic.li < mine; ++inflight, advance(ic)) issue(ic);
  __syncwarp();
  // every thread keeps the same issue cursor (thread 0 issued)
  if (threadIdx.x != 0)
    for (int q = 0; q < kDecBufs && ic.li < mine; ++q) advance(ic), ++inflight;
  uint4 av[2];
  load_a(unit(ac.li), ac.s, av);  // the first step always starts an A tile
  int b = 0;
  while (cc.li < mine) {
    const int i = unit(cc.li);
    if (needs_a(i, cc.s)) {
      store_a(av);  // the previous readers of the A tile passed the last barrier
      // the next step that starts an A tile, in flight during this one
      do advance(ac); while (ac.li < mine && !needs_a(unit(ac.li), ac.s));
      if (ac.li < mine) load_a(unit(ac.li), ac.s, av);
    }
    const bool landed = mbar_wait_bounded(&sh.bar[b], bar_phase[b], (volatile int*)&sh.abort_flag, kDecWaitNs);
    if (landed)
      bar_phase[b] ^= 1u;
    else
      set_status(a.status, MOE_ERR_TIMEOUT);
    __syncthreads();
    if (sh.abort_flag) {
      // let this CTA's copies still in flight land before its shared memory is released
      // (the pending phase of each buffer; this step's own only if it has not landed)
      if (threadIdx.x == 0)
        for (int q = landed ? 1 : 0; q < inflight; ++q) {
          const int bq = (b + q) % kDecBufs;
          mbar_wait_timed(&sh.bar[bq], bar_phase[bq], 200000000ull);
        }
      __syncthreads();
      return false;
    }
    const CUtensorMap* map;
    int row0, col0, nrows;
    step_info(i, cc.s, map, row0, col0, nrows);
    mma(i, cc.s, smem_u32(tiles + b * kDecTileBytes), nrows);
    const bool last = cc.s + 1 >= nsteps(i);
    if (last) done(i);
    __syncthreads();  // this buffer (and, at an A step, the A tile) is free again
    --inflight;
    if (ic.li < mine) {
      if (threadIdx.x == 0) issue(ic);
      advance(ic);
      ++inflight;
    }
    b = (b + 1) % kDecBufs;
    advance(cc);
  }
  return true;
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
  uint32_t bar_phase[kDecBufs] = {0, 0, 0, 0};

  // ---------------------------------------------------------------- R: router logits
  {
    // x[T][H] staged in the (still idle) weight ring: at most 16 x 4096 bf16 = 128 KB
    __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(tiles);
    const int EB = (E + kDecRouterE - 1) / kDecRouterE;
    if ((int)blockIdx.x < EB) {
      for (int i = tid; i < T * (H / 8); i += kDecThreads)
        reinterpret_cast<uint4*>(xs)[i] = reinterpret_cast<const uint4*>(a.x)[i];
      __syncthreads();
    }
    for (int eb = blockIdx.x; eb < EB; eb += G) {
      // thread: expert ec of the block, rows rg, rg + 32, ... (loads of 16 rows in flight)
      const int ec = tid & (kDecRouterE - 1), rg = tid / kDecRouterE, e = eb * kDecRouterE + ec;
      float acc[kDecMaxT];
#pragma unroll
      for (int t = 0; t < kDecMaxT; ++t) acc[t] = 0.0f;
      for (int r0 = rg; r0 < H; r0 += 32 * 16) {
        float wv[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const int r = r0 + 32 * q;
          wv[q] = (e < E && r < H) ? __bfloat162float(a.w_router[(int64_t)r * E + e]) : 0.0f;
        }
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const int r = r0 + 32 * q;
          if (r < H) {
#pragma unroll
            for (int t = 0; t < kDecMaxT; ++t)
              if (t < T) acc[t] = fmaf(__bfloat162float(xs[t * H + r]), wv[q], acc[t]);
          }
        }
      }
#pragma unroll
      for (int t = 0; t < kDecMaxT; ++t) sh.red[rg][t][ec] = acc[t];
      __syncthreads();
      if (tid < T * kDecRouterE) {  // the 32 row groups added in order, then the bias
        const int t = tid / kDecRouterE, c = tid % kDecRouterE, ee = eb * kDecRouterE + c;
        float l = 0.0f;
        for (int g = 0; g < 32; ++g) l += sh.red[g][t][c];
        if (ee < E) {
          l += a.bias ? a.bias[ee] : 0.0f;
          a.logits[t * E + ee] = l;
          if (a.user_logits) a.user_logits[t * E + ee] = l;
        }
      }
      __syncthreads();
    }
  }
  if (!dec_grid_sync(a, sh, 1)) return;

  // ---------------------------------------------------------------- top-k and slots
  {
    for (int t = warp; t < T; t += kDecThreads / 32) {
      float v[kDecMaxE / 32];
      uint32_t taken = 0;
#pragma unroll
      for (int i = 0; i < kDecMaxE / 32; ++i) {
        const int e = lane + 32 * i;
        if (e < E) {
          const float l = a.logits[t * E + e];
          v[i] = (l != l) ? -INFINITY : l;
        } else {
          v[i] = -INFINITY;
          taken |= 1u << i;
        }
      }
      float lmax = 0.0f, sum = 0.0f, my_w = 0.0f;
      int my_e = 0;
      for (int j = 0; j < k; ++j) {  // lane j keeps slot j (ties to the lower expert index)
        float bv = -INFINITY;
        int be = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < kDecMaxE / 32; ++i) {
          if (!((taken >> i) & 1u) && (be == 0x7fffffff || v[i] > bv)) {
            bv = v[i];
            be = lane + 32 * i;
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
        sum += ex;
        if (lane == j) {
          my_e = be;
          my_w = ex;
        }
      }
      if (lane < k) {
        const float wt = my_w * (1.0f / sum);
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

  // ---------------------------------------------------------------- G: h = silu(x Wg) * (x Wu)
  {
    // unit i -> (expert u, 64-column block fb of F_u); steps (kc, gate|up) over H
    const int nfb_r = F / 64;
    auto unit_of = [&](int i, int& u, int& fb) {
      if (i < n_routed * nfb_r) {
        u = i / nfb_r;
        fb = i % nfb_r;
      } else {
        u = n_routed;
        fb = i - n_routed * nfb_r;
      }
    };
    const int nunits = n_routed * nfb_r + (Fs > 0 ? Fs / 64 : 0);
    auto nsteps = [&](int) { return 2 * KC1; };
    auto step_info = [&](int i, int s, const CUtensorMap*& map, int& row0, int& col0, int& nrows) {
      int u, fb;
      unit_of(i, u, fb);
      const int kc = s >> 1, up = s & 1, k0 = kc * kDecStepRows;
      nrows = min(kDecStepRows, H - k0);
      col0 = fb * 64;
      if (u < n_routed) {
        map = up ? &tm_up : &tm_gate;
        row0 = sh.ex_id[u] * H + k0;
      } else {
        map = up ? &tm_sup : &tm_sgate;
        row0 = k0;
      }
    };
    auto needs_a = [&](int, int s) { return (s & 1) == 0; };
    auto load_a = [&](int i, int s, uint4 (&v)[2]) {  // x rows of the unit's tokens, the step's 256 columns
      int u, fb;
      unit_of(i, u, fb);
      const int k0 = (s >> 1) * kDecStepRows, nk = min(kDecStepRows, H - k0);
      const int s0 = sh.ex_first[u], ns = sh.ex_first[u + 1] - s0;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int idx = tid + q * kDecThreads, r = idx >> 5, c = idx & 31;
        v[q] = make_uint4(0, 0, 0, 0);
        if (r < ns && c * 8 < nk) v[q] = *reinterpret_cast<const uint4*>(a.x + (int64_t)slot_tok(s0 + r) * H + k0 + c * 8);
      }
    };
    auto store_a = [&](const uint4 (&v)[2]) {
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int idx = tid + q * kDecThreads, r = idx >> 5, c = idx & 31;
        *reinterpret_cast<uint4*>(sh.a_tile + r * kDecALd + c * 8) = v[q];
      }
    };
    float dg[4] = {0, 0, 0, 0}, du[4] = {0, 0, 0, 0};
    auto mma = [&](int, int s, uint32_t wt, int nrows) {
      if (s & 1) step_mma(sh, wt, nrows, du);
      else step_mma(sh, wt, nrows, dg);
    };
    auto done = [&](int i) {
      int u, fb;
      unit_of(i, u, fb);
      const int s0 = sh.ex_first[u], ns = sh.ex_first[u + 1] - s0;
      const int col = fb * 64 + warp * 8 + (lane & 3) * 2, r0 = lane >> 2;
      float h[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) h[q] = dg[q] * sigmoidf_(dg[q]) * du[q];
      if (r0 < ns)
        *reinterpret_cast<__nv_bfloat162*>(a.hbuf + (int64_t)(s0 + r0) * Fm + col) = __floats2bfloat162_rn(h[0], h[1]);
      if (r0 + 8 < ns)
        *reinterpret_cast<__nv_bfloat162*>(a.hbuf + (int64_t)(s0 + r0 + 8) * Fm + col) =
            __floats2bfloat162_rn(h[2], h[3]);
#pragma unroll
      for (int q = 0; q < 4; ++q) dg[q] = du[q] = 0.0f;
    };
    if (!stream_steps(sh, tiles, bar_phase, nunits, a, nsteps, step_info, needs_a, load_a, store_a, mma, done)) return;
  }
  if (!dec_grid_sync(a, sh, 2)) return;

  // ---------------------------------------------------------------- D: y = h Wd
  {
    const int nhb = H / 64;
    const int nunits = n_u * nhb;
    auto fu = [&](int u) { return u < n_routed ? F : Fs; };
    auto nsteps = [&](int i) { return (fu(i / nhb) + kDecStepRows - 1) / kDecStepRows; };
    auto step_info = [&](int i, int s, const CUtensorMap*& map, int& row0, int& col0, int& nrows) {
      const int u = i / nhb, hb = i % nhb, k0 = s * kDecStepRows;
      nrows = min(kDecStepRows, fu(u) - k0);
      col0 = hb * 64;
      if (u < n_routed) {
        map = &tm_down;
        row0 = sh.ex_id[u] * F + k0;
      } else {
        map = &tm_sdown;
        row0 = k0;
      }
    };
    auto needs_a = [&](int, int) { return true; };
    auto load_a = [&](int i, int s, uint4 (&v)[2]) {  // h rows of the unit's slots, the step's 256 columns
      const int u = i / nhb, k0 = s * kDecStepRows, nk = min(kDecStepRows, fu(u) - k0);
      const int s0 = sh.ex_first[u], ns = sh.ex_first[u + 1] - s0;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int idx = tid + q * kDecThreads, r = idx >> 5, c = idx & 31;
        v[q] = make_uint4(0, 0, 0, 0);
        if (r < ns && c * 8 < nk) v[q] = *reinterpret_cast<const uint4*>(a.hbuf + (int64_t)(s0 + r) * Fm + k0 + c * 8);
      }
    };
    auto store_a = [&](const uint4 (&v)[2]) {
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int idx = tid + q * kDecThreads, r = idx >> 5, c = idx & 31;
        *reinterpret_cast<uint4*>(sh.a_tile + r * kDecALd + c * 8) = v[q];
      }
    };
    float d[4] = {0, 0, 0, 0};
    auto mma = [&](int, int, uint32_t wt, int nrows) { step_mma(sh, wt, nrows, d); };
    auto done = [&](int i) {
      const int u = i / nhb, hb = i % nhb;
      const int s0 = sh.ex_first[u], ns = sh.ex_first[u + 1] - s0;
      const int col = hb * 64 + warp * 8 + (lane & 3) * 2, r0 = lane >> 2;
      if (r0 < ns) *reinterpret_cast<float2*>(a.ypair + (int64_t)(s0 + r0) * H + col) = make_float2(d[0], d[1]);
      if (r0 + 8 < ns) *reinterpret_cast<float2*>(a.ypair + (int64_t)(s0 + r0 + 8) * H + col) = make_float2(d[2], d[3]);
#pragma unroll
      for (int q = 0; q < 4; ++q) d[q] = 0.0f;
    };
    if (!stream_steps(sh, tiles, bar_phase, nunits, a, nsteps, step_info, needs_a, load_a, store_a, mma, done)) return;
  }
  if (!dec_grid_sync(a, sh, 3)) return;

  // ---------------------------------------------------------------- C: combine
  for (int idx = blockIdx.x * kDecThreads + tid; idx < T * (H / 4); idx += G * kDecThreads) {
    const int t = idx / (H / 4), c = (idx % (H / 4)) * 4;
    float4 v[kDecMaxK];
#pragma unroll
    for (int j = 0; j < kDecMaxK; ++j)  // every slot's row loaded before the sum
      if (j < k) v[j] = *reinterpret_cast<const float4*>(a.ypair + (int64_t)sh.slot_of_pair[t * k + j] * H + c);
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
      const float4 sv = *reinterpret_cast<const float4*>(a.ypair + (int64_t)(P + t) * H + c);
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

size_t decode_scratch_bytes(int64_t T, int64_t H, int64_t F, int64_t E, int64_t Fs) {
  const int64_t Fm = F > Fs ? F : Fs;
  auto up = [](int64_t n) { return (size_t)((n + 255) / 256 * 256); };
  return up(T * E * 4) + up((int64_t)kDecMaxSlots * Fm * 2) + up((int64_t)kDecMaxSlots * H * 4) + 256;
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
  const int64_t Fm = F > Fs ? F : Fs;
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
  b += up((int64_t)kDecMaxSlots * Fm * 2);
  a.ypair = reinterpret_cast<float*>(b);
  b += up((int64_t)kDecMaxSlots * H * 4);
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
