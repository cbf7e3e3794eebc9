// decode.cu -- the forward of the MoE layer for decode-sized token counts, fused
// into one persistent kernel (inference: nothing is kept for a backward).
//
// At a handful of tokens the layer is a weight stream: each token touches k experts,
// and their W_gate, W_up, W_down dominate the bytes. The unfused path runs a dozen
// short kernels whose launch, prologue and pipeline fill cost more than the stream.
// Here one cooperative launch (one CTA per SM, every CTA resident) runs these phases,
// separated by grid-wide barriers:
//   R  router logits: CTA (16-expert group, quarter of H) computes its block of
//      W_r^T x^T with mma.sync, a partial sum the top-k warps add in a fixed order;
//   K  every CTA takes the top-k and the renormalised softmax weights of every token
//      and builds the same slot table (the routed (token, expert) pairs sorted by
//      expert then token, then one slot per token for the shared expert);
//   G  x W_gate and x W_up: units (expert, column block of at most 768 columns) whose
//      steps are 32-row slices of H read end to end (a row block of the weight); each
//      CTA takes an even share of all steps (K split) and adds a unit's steps in
//      registers, storing the sums of a unit it streamed whole, or its piece of a
//      split unit;
//   H  h = silu(g) * u per slot, g and u the sums of each unit's pieces in CTA order;
//   D  y = h W_down: units (expert, 64 columns of H) taken round-robin, each streaming
//      all F_u rows in 256-row steps; its first copies are issued before phase H, so
//      they land while it runs;
//   C  y[t] = sum_j w_tj y(t, j) (+ the shared expert), slots in order, rounded once.
// The weight steps move through a ring of four 48 KB shared-memory tiles (TMA, 128-byte
// swizzle). One producer warp issues the copies as soon as a tile is free; eight
// consumer warps multiply (mma.sync m16n8k16, bf16 in, fp32 accumulators; warp w owns
// the 8-column n-tile w of every 64-column box) and free a tile as soon as each has
// read it, so that a tile is refilled without waiting for the block. At most 16 tokens
// make the contractions 16 rows wide: the weight stream, not the tensor rate, bounds
// them. Every sum runs in a fixed order, so two calls give the same bits. Every wait
// (TMA landing, a free tile, a grid barrier) is bounded: a wait that runs out sets
// MOE_ERR_TIMEOUT in the status word and the kernel returns.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "decode.h"

namespace moe {

constexpr int kDecMaxT = 16;                  // tokens (the mma M dimension)
constexpr int kDecThreads = 256;              // consumer threads: 8 warps
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kDecBlock = kDecThreads + 32;   // + the producer warp
constexpr int kDecBufs = 4;                   // ring tiles
constexpr int kDecTileBytes = 49152;          // one ring tile: 48 KB
// gate/up steps: 32 rows of H x up to 12 boxes of 64 columns side by side
constexpr int kDecGRows = 32;
constexpr int kDecGMaxBox = 12;
constexpr int kDecGBoxBytes = kDecGRows * 128;  // 4 KB
constexpr int kDecGMaxCols = kDecGMaxBox * 64;
// down steps: 256 rows of F_u x 64 columns of H (four 64-row boxes, 32 KB), then the
// step's A tile: the expert's h rows x the same 256 columns (four 16-row boxes, 8 KB)
constexpr int kDecStepRows = 256;
constexpr int kDecBoxRows = 64;
constexpr int kDecDABoxRows = 16;
constexpr int kDecDAOffset = 32768;
constexpr int kDecMaxE = 256;
constexpr int kDecRSlices = 4;  // router: row slices of H, each summed by its own CTAs
constexpr int kDecMaxK = 16;  // T * k <= 256: one thread per routed pair when ranking them
constexpr int kDecMaxH = 4096;
constexpr int kDecMaxGrid = 256;  // CTAs of one launch at most (one per SM)
constexpr uint64_t kDecWaitNs = 1000000000ull;  // 1 s

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
  float* logits;      // [kDecRSlices][T][E]: router partial sums over the row slices of H
  __nv_bfloat16* hbuf;  // [slots][Fm]
  float* ypair;       // [slots][H]
  float* part_g;      // [slots][gate, up][Fm]: x Wg and x Wu of a unit streamed by one CTA
  float* piece_g;     // [2 * kDecMaxGrid][gate, up][T][kDecGMaxCols]: pieces of split units
  unsigned* sync;     // grid barrier counter (zeroed by the caller before the launch)
  int* status;
  uint64_t wait_ns;   // limit of every wait (1 s; shorter in the self-test)
  unsigned stall;     // self-test: grid barrier number that needs one arrival more than the grid has (0: none)
};

struct DecodeShared {
  int s_idx[kDecMaxT * kDecMaxK];
  float s_w[kDecMaxT * kDecMaxK];
  int slot_pair[kDecMaxT * kDecMaxK];        // routed slot -> pair t*k + j
  int slot_of_pair[kDecMaxT * kDecMaxK];
  int ex_id[kDecMaxT * kDecMaxK + 1];        // unit expert u -> expert id (shared: -1)
  int ex_first[kDecMaxT * kDecMaxK + 2];     // first slot of expert u; ex_first[n_u] = slots
  int slot_u[kDecMaxT * kDecMaxK + kDecMaxT];  // slot -> unit expert u
  int cta_start[kDecMaxGrid + 1];            // first gate/up step of every CTA
  uint64_t full[kDecBufs];                   // a tile's copies landed
  uint64_t empty[kDecBufs];                  // every consumer warp has read the tile
  int n_routed, n_u;
  int h_ready;                               // phase H is done grid-wide: down A tiles may be copied
  int abort_flag;
};

// ------------------------------------------------------------------ small helpers
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
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
// barrier of the eight consumer warps only (the producer warp runs its own loop)
__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kDecThreads) : "memory"); }
// tx bytes expected on a barrier, without an arrival
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

// Grid-wide barrier number `phase` (1, 2, ...), in two halves so that a CTA can issue
// work between them: arrive (every CTA once: a release add after the CTA's own barrier)
// and wait (thread 0 polls with acquire loads). The CTA's own barrier covers all threads
// (kAll) before the producer warp starts its loop, the consumer warps after. wait
// returns false when the wait ran out (or an earlier one did), after recording
// MOE_ERR_TIMEOUT.
template <bool kAll>
__device__ __forceinline__ void block_sync() {
  if (kAll)
    __syncthreads();
  else
    consumer_sync();
}
// the same barrier, returning whether any participating thread passed true: every
// thread leaves with the same answer, even when another warp changes the flag it read
template <bool kAll>
__device__ __forceinline__ bool block_any(bool p) {
  if (kAll) return __syncthreads_or(p) != 0;
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred q, o;\n\tsetp.ne.u32 q, %1, 0;\n\tbar.red.or.pred o, 1, %2, q;\n\tselp.u32 %0, 1, 0, o;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)p), "n"(kDecThreads)
      : "memory");
  return r != 0;
}
template <bool kAll>
__device__ __forceinline__ void dec_grid_arrive(const DecodeArgs& a, DecodeShared& sh) {
  block_sync<kAll>();
  if (threadIdx.x == 0 && !sh.abort_flag)
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(a.sync), "r"(1u) : "memory");
}
template <bool kAll>
__device__ bool dec_grid_wait(const DecodeArgs& a, DecodeShared& sh, unsigned phase) {
  if (threadIdx.x == 0 && !sh.abort_flag) {
    const unsigned target = phase * gridDim.x + (phase == a.stall ? 1u : 0u);
    if (ld_acquire_gpu(a.sync) < target) {
      const uint64_t t0 = globaltimer_ns();
      while (ld_acquire_gpu(a.sync) < target) {
        if (globaltimer_ns() - t0 > a.wait_ns) {
          sh.abort_flag = 1;
          set_status(a.status, MOE_ERR_TIMEOUT);
          break;
        }
      }
    }
  }
  return !block_any<kAll>(*(volatile int*)&sh.abort_flag != 0);
}

// The steps of the gate/up phase; CTA c takes the steps [start(c), start(c + 1)), an
// even share, so a unit may be split between neighbouring CTAs (K split).
struct PhaseSteps {
  int64_t total;
  int G;
  __device__ int64_t start(int c) const { return total * c / G; }
  __device__ int cta_of(int64_t g) const { return (int)(((g + 1) * G - 1) / total); }  // last c with start(c) <= g
};
// The same in 32-bit arithmetic with the starts tabled (total * G < 2^31): for the
// reduce phase, which asks it for every item.
struct PhaseTable {
  const int* start;  // start[c], c <= G
  uint32_t total, G;
  __device__ int cta_of(uint32_t g) const { return (int)(((g + 1) * G - 1) / total); }
};

// Consumer wait for ring tile j (sequence number): its copies landed. False after the
// wait ran out or another role gave up.
__device__ __forceinline__ bool wait_full(DecodeShared& sh, const DecodeArgs& a, int j) {
  const int b = j % kDecBufs;
  if (mbar_wait_bounded(&sh.full[b], (uint32_t)((j / kDecBufs) & 1), (volatile int*)&sh.abort_flag, a.wait_ns))
    return true;
  set_status(a.status, MOE_ERR_TIMEOUT);
  return false;
}
// Consumer warp done with tile j.
__device__ __forceinline__ void release(DecodeShared& sh, int j) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&sh.empty[j % kDecBufs]);
}

// A gate/up step is read out of its tile into registers first (bf: box x, k16 half kq),
// so that the tile can be freed before the multiplications: warp w takes columns
// 8w .. 8w+7 of every box.
__device__ __forceinline__ void step_load_rows(uint32_t wt, int nbx, uint32_t (&bf)[2][kDecGMaxBox][2]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int kq = 0; kq < 2; ++kq) {
    const int br = kq * 16 + (lane & 15);
    const uint32_t boff = (uint32_t)(br * 128 + ((warp ^ (br & 7)) << 4));
#pragma unroll
    for (int x = 0; x < kDecGMaxBox; ++x)
      if (x < nbx) ldsm_x2_trans(wt + (uint32_t)(x * kDecGBoxBytes) + boff, bf[kq][x][0], bf[kq][x][1]);
  }
}
// acc[x] += A (16 rows x 32 columns, fragments in registers) x (box x: 32 rows x 64 columns)
// for the nbx boxes of the step; the nbx accumulators are independent chains.
__device__ __forceinline__ void step_mma_rows(int nbx, const uint32_t (&af)[2][4], const uint32_t (&bf)[2][kDecGMaxBox][2],
                                              float (&acc)[kDecGMaxBox][4]) {
#pragma unroll
  for (int kq = 0; kq < 2; ++kq)
#pragma unroll
    for (int x = 0; x < kDecGMaxBox; ++x)
      if (x < nbx) mma_16816(acc[x], af[kq][0], af[kq][1], af[kq][2], af[kq][3], bf[kq][x][0], bf[kq][x][1]);
}

// A down step read out of its tile into registers (16-row slice h of the nrows rows: A
// fragments fa[h] from the step's A tile at wt + kDecDAOffset, four swizzled 16-row
// boxes; B fragments fb[h] of the weight tile at wt), so that the tile can be freed
// before the multiplications. nrows is a multiple of 64.
__device__ __forceinline__ void step_load_down(uint32_t wt, int nrows, uint32_t (&fa)[16][4], uint32_t (&fb)[16][2]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t at = wt + kDecDAOffset;
  const int ar = lane & 15;
#pragma unroll
  for (int h = 0; h < 16; ++h) {
    const int k0 = 16 * h;
    if (k0 < nrows) {
      const int chunk = ((k0 & 63) >> 3) + (lane >> 4);  // 16-byte chunk of the A box row
      ldsm_x4(at + (uint32_t)((k0 >> 6) * (kDecDABoxRows * 128) + ar * 128 + ((chunk ^ (ar & 7)) << 4)), fa[h][0],
              fa[h][1], fa[h][2], fa[h][3]);
      const int br = k0 + (lane & 15);
      ldsm_x2_trans(wt + (uint32_t)(br * 128 + ((warp ^ (br & 7)) << 4)), fb[h][0], fb[h][1]);
    }
  }
}
// d0 + d1 += A x B over the step's 16-row slices: warp w takes columns 8w .. 8w+7; even
// slices go to d0, odd ones to d1.
__device__ __forceinline__ void step_mma_down(int nrows, const uint32_t (&fa)[16][4], const uint32_t (&fb)[16][2],
                                              float (&d0)[4], float (&d1)[4]) {
#pragma unroll
  for (int h = 0; h < 16; h += 2) {
    if (16 * h < nrows) {
      mma_16816(d0, fa[h][0], fa[h][1], fa[h][2], fa[h][3], fb[h][0], fb[h][1]);
      mma_16816(d1, fa[h + 1][0], fa[h + 1][1], fa[h + 1][2], fa[h + 1][3], fb[h + 1][0], fb[h + 1][1]);
    }
  }
}

// ------------------------------------------------------------------ the kernel
__global__ void __launch_bounds__(kDecBlock, 1)
    k_decode_fwd(const __grid_constant__ CUtensorMap tm_gate, const __grid_constant__ CUtensorMap tm_up,
                 const __grid_constant__ CUtensorMap tm_down, const __grid_constant__ CUtensorMap tm_sgate,
                 const __grid_constant__ CUtensorMap tm_sup, const __grid_constant__ CUtensorMap tm_sdown,
                 const __grid_constant__ CUtensorMap tm_h, const DecodeArgs a) {
  extern __shared__ uint8_t dec_smem_raw[];
  uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dec_smem_raw) + 1023) & ~uintptr_t(1023));
  DecodeShared& sh = *reinterpret_cast<DecodeShared*>(tiles + kDecBufs * kDecTileBytes);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool consumer = warp < kDecWarps;
  const int T = a.T, H = a.H, F = a.F, E = a.E, k = a.k, Fs = a.Fs;
  const int Fm = max(F, Fs);
  const int G = gridDim.x;
  const int P = T * k;

  if (tid == 0) {
    for (int b = 0; b < kDecBufs; ++b) {
      mbar_init(&sh.full[b], 1);
      mbar_init(&sh.empty[b], kDecWarps);
    }
    sh.abort_flag = 0;
    sh.h_ready = 0;
    fence_mbar_init();
  }
  __syncthreads();

  // ---------------------------------------------------------------- R: router logits
  // CTA (expert group eg of 16 experts, row slice sl of H) computes the 16 x T block of
  // logits^T = W_r^T x^T over its rows with mma.sync (experts as M, tokens as N), warp w
  // taking the 16-row blocks w, w + 8, ...; the eight warps are added in order and the
  // partial goes to a.logits[sl]. A slice's rows are read by the CTAs of all expert
  // groups at once, 32 bytes of each W_r row per CTA, so DRAM sees whole rows.
  {
    const int EG = (E + 15) / 16;
    const int nkb = H / 16, kbs = (nkb + kDecRSlices - 1) / kDecRSlices;  // 16-row blocks per slice
    for (int rb = blockIdx.x; rb < EG * kDecRSlices; rb += G) {
      const int eg = rb % EG, sl = rb / EG;
      const int kb0 = sl * kbs, kb1 = min(nkb, kb0 + kbs);
      const int g0 = lane >> 2, t4 = lane & 3;
      const int ea = eg * 16 + g0, eb = ea + 8;  // the two experts (M rows) of this lane
      float c[2][4] = {{0, 0, 0, 0}, {0, 0, 0, 0}};
      if (consumer) {
        auto wpair = [&](int e, int k) -> uint32_t {  // W_r[k][e], W_r[k + 1][e] packed
          if (e >= E) return 0u;
          const uint16_t lo = reinterpret_cast<const uint16_t*>(a.w_router)[(int64_t)k * E + e];
          const uint16_t hi = reinterpret_cast<const uint16_t*>(a.w_router)[(int64_t)(k + 1) * E + e];
          return (uint32_t)lo | ((uint32_t)hi << 16);
        };
#pragma unroll 4
        for (int kb = kb0 + warp; kb < kb1; kb += kDecWarps) {
          const int k0 = kb * 16 + 2 * t4;
          const uint32_t a0 = wpair(ea, k0), a1 = wpair(eb, k0), a2 = wpair(ea, k0 + 8), a3 = wpair(eb, k0 + 8);
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            const int t = nt * 8 + g0;
            if (nt * 8 < T) {
              uint32_t b0 = 0u, b1 = 0u;
              if (t < T) {
                b0 = *reinterpret_cast<const uint32_t*>(a.x + (int64_t)t * H + k0);
                b1 = *reinterpret_cast<const uint32_t*>(a.x + (int64_t)t * H + k0 + 8);
              }
              mma_16816(c[nt], a0, a1, a2, a3, b0, b1);
            }
          }
        }
      }
      // the warps' fragments, added in warp order (the idle ring holds them)
      float* red = reinterpret_cast<float*>(tiles);
      if (consumer)
#pragma unroll
        for (int q = 0; q < 8; ++q) red[(warp * 32 + lane) * 8 + q] = c[q >> 2][q & 3];
      __syncthreads();
      if (consumer) {
        const int ln = tid >> 3, q = tid & 7, nt = q >> 2, ci = q & 3;
        float v = 0.0f;
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) v += red[(w * 32 + ln) * 8 + q];
        // fragment element ci of lane ln: expert row (ln >> 2) + 8 (ci >> 1), token 2 (ln & 3) + (ci & 1)
        const int e = eg * 16 + (ln >> 2) + 8 * (ci >> 1), t = nt * 8 + 2 * (ln & 3) + (ci & 1);
        if (e < E && t < T) a.logits[((int64_t)sl * T + t) * E + e] = v;
      }
      __syncthreads();  // the ring is idle until the first copies; its readers are done here
    }
  }
  dec_grid_arrive<true>(a, sh);
  if (!dec_grid_wait<true>(a, sh, 1)) return;  // every thread, the producer warp too, leaves here

  // ---------------------------------------------------------------- K: top-k and slots
  {
    // warp w takes tokens w, w + 8, ...: lane l holds the logits of experts l, l + 32, ...
    // as order-preserving keys (NaN reads as -inf, -0 as +0); each of k rounds takes the
    // largest key still free, ties to the lower expert index, with two warp reductions
    for (int t = warp; consumer && t < T; t += kDecWarps) {
      float v[kDecMaxE / 32];
      uint32_t key[kDecMaxE / 32];
      float ps[kDecRSlices][kDecMaxE / 32];  // every slice's partial in flight before the sums
#pragma unroll
      for (int i = 0; i < kDecMaxE / 32; ++i) {
        const int e = lane + 32 * i;
#pragma unroll
        for (int q = 0; q < kDecRSlices; ++q) ps[q][i] = e < E ? __ldcg(a.logits + ((int64_t)q * T + t) * E + e) : 0.0f;
      }
#pragma unroll
      for (int i = 0; i < kDecMaxE / 32; ++i) {
        const int e = lane + 32 * i;
        float l = 0.0f;
#pragma unroll
        for (int q = 0; q < kDecRSlices; ++q) l += ps[q][i];  // slices in order, then the bias
        if (e < E) {
          l += a.bias ? a.bias[e] : 0.0f;
          if (blockIdx.x == 0 && a.user_logits) a.user_logits[t * E + e] = l;
        }
        v[i] = e < E ? l : -INFINITY;
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
    for (int u2 = tid; u2 < sh.n_u; u2 += kDecBlock)
      for (int q = sh.ex_first[u2]; q < sh.ex_first[u2 + 1]; ++q) sh.slot_u[q] = u2;
    __syncthreads();
  }
  const int n_routed = sh.n_routed, n_u = sh.n_u;
  auto slot_tok = [&](int s) { return s < P ? sh.slot_pair[s] / k : s - P; };

  // ---------------------------------------------------------------- step lists of both roles
  // G: units (expert u, column block cb of F_u); a unit's steps are its 32-row slices of
  // H, gate then up, each step the whole width of the block. CTA c takes the steps
  // [start(c), start(c + 1)) of all of them.
  const int nbox_r = F / 64, nbox_s = Fs / 64;
  const int ncb_r = (nbox_r + kDecGMaxBox - 1) / kDecGMaxBox, bpb_r = (nbox_r + ncb_r - 1) / ncb_r;
  const int ncb_s = nbox_s > 0 ? (nbox_s + kDecGMaxBox - 1) / kDecGMaxBox : 0;
  const int bpb_s = ncb_s > 0 ? (nbox_s + ncb_s - 1) / ncb_s : 1;
  const int RS = H / kDecGRows;  // 32-row slices of H
  const int SG = 2 * RS;         // steps per unit: the gate slices, then the up slices
  const PhaseSteps phg{(int64_t)(n_routed * ncb_r + ncb_s) * SG, G};
  const int64_t gs0 = phg.start(blockIdx.x), gs1 = phg.start(blockIdx.x + 1);
  for (int c = tid; c <= G; c += kDecBlock) sh.cta_start[c] = (int)phg.start(c);
  __syncthreads();  // every thread (the producer warp too) is still here
  const PhaseTable pht{sh.cta_start, (uint32_t)phg.total, (uint32_t)G};
  const int nG = (int)(gs1 - gs0);  // ring steps of this CTA's gate/up share
  auto g_unit = [&](int i, int& u, int& cb, int& nbx, int& bpb) {
    if (i < n_routed * ncb_r) {
      u = i / ncb_r;
      cb = i - u * ncb_r;
      bpb = bpb_r;
      nbx = min(bpb_r, nbox_r - cb * bpb_r);
    } else {
      u = n_routed;
      cb = i - n_routed * ncb_r;
      bpb = bpb_s;
      nbx = min(bpb_s, nbox_s - cb * bpb_s);
    }
  };
  // D: units (expert u, 64 columns hb of H), CTA b taking units b, b + G, ...; each
  // streams all F_u rows of W_down in 256-row steps.
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

  // ---------------------------------------------------------------- the producer warp
  if (!consumer) {
    if (lane != 0) return;
    int j = 0;            // ring sequence number of the next copy
    int ja = nG;          // sequence number of the next down step whose A tile is not issued
    DCur ac{0, 0};        // its cursor
    bool ok = true;
    auto h_ready = [&]() {
      int v;
      asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_u32(&sh.h_ready)) : "memory");
      return v != 0;
    };
    // the A tile of down step ja: h rows of the unit's slots x the step's 256 columns;
    // its arrival completes the step's barrier (the weights only announced their bytes)
    auto issue_a = [&]() {
      const int u = d_unit(ac) / nhb, k0 = ac.fk * kDecStepRows;
      const int nbox = (min(kDecStepRows, fu(u) - k0) + 63) / 64;
      const int b = ja % kDecBufs;
      mbar_arrive_expect_tx(&sh.full[b], (uint32_t)(nbox * kDecDABoxRows * 128));
      for (int x = 0; x < nbox; ++x)
        tma_load_2d(smem_u32(tiles + b * kDecTileBytes + kDecDAOffset + x * kDecDABoxRows * 128), &tm_h,
                    smem_u32(&sh.full[b]), k0 + x * 64, sh.ex_first[u]);
      ++ja;
      d_advance(ac);
    };
    // tile j's buffer free again (its previous use read by every consumer warp); A tiles
    // of down steps already issued go out meanwhile, once h is ready
    bool proxy_fenced = false;
    auto pump_a = [&](int upto) {
      if (ja < upto && h_ready()) {
        if (!proxy_fenced) {  // h was written by generic stores in other CTAs
          asm volatile("fence.proxy.async.global;" ::: "memory");
          proxy_fenced = true;
        }
        while (ja < upto) issue_a();
      }
    };
    auto acquire = [&](int jj) -> bool {
      const uint32_t bar = smem_u32(&sh.empty[jj % kDecBufs]);
      const uint32_t par = (uint32_t)(((jj / kDecBufs) & 1) ^ 1);
      uint64_t t0 = 0;
      uint32_t n = 0;
      while (!mbar_try_wait(bar, par)) {
        pump_a(jj);
        if ((++n & 63u) == 0) {
          if (*(volatile int*)&sh.abort_flag) return false;
          const uint64_t now = globaltimer_ns();
          if (t0 == 0)
            t0 = now;
          else if (now - t0 > a.wait_ns) {
            sh.abort_flag = 1;
            set_status(a.status, MOE_ERR_TIMEOUT);
            return false;
          }
        }
      }
      return true;
    };
    // gate/up steps
    if (nG > 0) {
      int ii = (int)(gs0 / SG), is = (int)(gs0 - (int64_t)ii * SG);
      for (int q = 0; q < nG; ++q, ++j) {
        if (!acquire(j)) {
          ok = false;
          break;
        }
        int u, cb, nbx, bpb;
        g_unit(ii, u, cb, nbx, bpb);
        const int gu = is >= RS ? 1 : 0, r0 = (is - gu * RS) * kDecGRows;
        const CUtensorMap* map = u < n_routed ? (gu ? &tm_up : &tm_gate) : (gu ? &tm_sup : &tm_sgate);
        const int b = j % kDecBufs;
        const int row0 = (u < n_routed ? sh.ex_id[u] * H : 0) + r0;
        fence_async_smem();
        mbar_arrive_expect_tx(&sh.full[b], (uint32_t)(nbx * kDecGBoxBytes));
        for (int x = 0; x < nbx; ++x)
          tma_load_2d(smem_u32(tiles + b * kDecTileBytes + x * kDecGBoxBytes), map, smem_u32(&sh.full[b]),
                      (cb * bpb + x) * 64, row0);
        if (++is == SG) {
          is = 0;
          ++ii;
        }
      }
    }
    // down steps: the weights as soon as a buffer is free, the A tiles once h is ready
    for (DCur dc{0, 0}; ok && dc.li < mine_d; d_advance(dc), ++j) {
      if (!acquire(j)) {
        ok = false;
        break;
      }
      const int i = d_unit(dc), u = i / nhb, hb = i % nhb, k0 = dc.fk * kDecStepRows;
      const int nbox = (min(kDecStepRows, fu(u) - k0) + kDecBoxRows - 1) / kDecBoxRows;
      const int b = j % kDecBufs;
      const CUtensorMap* map = u < n_routed ? &tm_down : &tm_sdown;
      const int row0 = (u < n_routed ? sh.ex_id[u] * F : 0) + k0;
      fence_async_smem();
      mbar_expect_tx(&sh.full[b], (uint32_t)(nbox * kDecBoxRows * 128));
      for (int x = 0; x < nbox; ++x)
        tma_load_2d(smem_u32(tiles + b * kDecTileBytes + x * kDecBoxRows * 128), map, smem_u32(&sh.full[b]), hb * 64,
                    row0 + x * kDecBoxRows);
      pump_a(j + 1);
    }
    // the A tiles still missing
    if (ok) {
      const uint64_t t0 = globaltimer_ns();
      while (ja < j) {
        pump_a(j);
        if (ja < j) {
          if (*(volatile int*)&sh.abort_flag) {
            ok = false;
            break;
          }
          if (globaltimer_ns() - t0 > a.wait_ns) {
            sh.abort_flag = 1;
            set_status(a.status, MOE_ERR_TIMEOUT);
            ok = false;
            break;
          }
        }
      }
    }
    if (!ok) {
      // on the way out after a failed wait: every copy issued lands before the shared
      // memory is released (a down step whose A tile never went out gets a plain arrival
      // in its place, so that its barrier completes on the weights' bytes alone)
      for (int q = j - kDecBufs < 0 ? 0 : j - kDecBufs; q < j; ++q) {
        const int b = q % kDecBufs;
        if (q >= ja) mbar_arrive(&sh.full[b]);
        mbar_wait_timed(&sh.full[b], (uint32_t)((q / kDecBufs) & 1), 200000000ull);
      }
    }
    return;
  }

  // ---------------------------------------------------------------- consumers
  auto slot_rows = [&](int u, int& s0, int& ns) {
    s0 = sh.ex_first[u];
    ns = sh.ex_first[u + 1] - s0;
  };
  int j = 0;  // ring sequence number of the next tile to read

  // ---------------------------------------------------------------- G: x Wg, x Wu
  // A unit's steps in this CTA are added in registers; at the end of the unit (or of the
  // CTA's share) the sums go to part_g (a unit streamed whole) or to piece slot 2c (the
  // CTA's first piece) or 2c + 1 (its last).
  {
    // A fragments of one 32-row slice of H (two k16 halves) for step st of unit i: rows =
    // the unit's tokens
    auto load_af = [&](int i, int st, uint32_t (&af)[2][4]) {
      int u, cb, nbx, bpb;
      g_unit(i, u, cb, nbx, bpb);
      int sb, ns;
      slot_rows(u, sb, ns);
      const int g0 = lane >> 2, t4 = lane & 3, k0 = (st >= RS ? st - RS : st) * kDecGRows;
      const __nv_bfloat16* x0 = a.x + (int64_t)slot_tok(sb + (g0 < ns ? g0 : 0)) * H;
      const __nv_bfloat16* x1 = a.x + (int64_t)slot_tok(sb + (g0 + 8 < ns ? g0 + 8 : 0)) * H;
#pragma unroll
      for (int kq = 0; kq < 2; ++kq) {
        const int kb = k0 + kq * 16 + 2 * t4;
        af[kq][0] = g0 < ns ? *reinterpret_cast<const uint32_t*>(x0 + kb) : 0u;
        af[kq][1] = g0 + 8 < ns ? *reinterpret_cast<const uint32_t*>(x1 + kb) : 0u;
        af[kq][2] = g0 < ns ? *reinterpret_cast<const uint32_t*>(x0 + kb + 8) : 0u;
        af[kq][3] = g0 + 8 < ns ? *reinterpret_cast<const uint32_t*>(x1 + kb + 8) : 0u;
      }
    };
    float acc[kDecGMaxBox][4];  // the gate or the up sums of the current unit
#pragma unroll
    for (int x = 0; x < kDecGMaxBox; ++x)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[x][q] = 0.0f;
    // the sums of unit i's gate (gu 0) or up (gu 1) steps in this CTA, to part_g (whole
    // unit) or its piece slot
    auto flush = [&](int i, int gu) {
      int u, cb, nbx, bpb;
      g_unit(i, u, cb, nbx, bpb);
      int sb, ns;
      slot_rows(u, sb, ns);
      const int64_t ub = (int64_t)i * SG, ue = ub + SG;
      const bool whole = ub >= gs0 && ue <= gs1;
      const int ps = ub <= gs0 ? 2 * (int)blockIdx.x : 2 * (int)blockIdx.x + 1;
      const int r0 = lane >> 2, cq = warp * 8 + (lane & 3) * 2;
#pragma unroll
      for (int x = 0; x < kDecGMaxBox; ++x) {
        if (x < nbx) {
#pragma unroll
          for (int h8 = 0; h8 < 2; ++h8) {
            const int r = r0 + 8 * h8;
            if (r < ns) {
              float* dst = whole ? a.part_g + ((int64_t)(sb + r) * 2 + gu) * Fm + (cb * bpb + x) * 64 + cq
                                 : a.piece_g + (((int64_t)ps * 2 + gu) * T + r) * kDecGMaxCols + x * 64 + cq;
              *reinterpret_cast<float2*>(dst) = make_float2(acc[x][2 * h8], acc[x][2 * h8 + 1]);
            }
          }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[x][q] = 0.0f;
      }
    };
    if (nG > 0) {
      int ci = (int)(gs0 / SG), cs = (int)(gs0 - (int64_t)ci * SG);  // unit and step of the tile
      int ai = ci, as = cs;  // the step whose A fragments are in an
      uint32_t af[2][4], an[2][4];
      load_af(ai, as, an);
      for (int64_t g = gs0; g < gs1; ++g, ++j) {
        // this step's A fragments, and the next step's in flight
#pragma unroll
        for (int kq = 0; kq < 2; ++kq)
#pragma unroll
          for (int q = 0; q < 4; ++q) af[kq][q] = an[kq][q];
        if (++as == SG) {
          as = 0;
          ++ai;
        }
        if (g + 1 < gs1) load_af(ai, as, an);
        if (!wait_full(sh, a, j)) break;  // the barrier below makes every warp leave
        int u, cb, nbx, bpb;
        g_unit(ci, u, cb, nbx, bpb);
        const uint32_t wt = smem_u32(tiles + (j % kDecBufs) * kDecTileBytes);
        uint32_t bf[2][kDecGMaxBox][2];
        step_load_rows(wt, nbx, bf);
        release(sh, j);  // the tile is in registers: its buffer can be refilled meanwhile
        step_mma_rows(nbx, af, bf, acc);
        if (g + 1 == gs1 || cs + 1 == RS || cs + 1 == SG) flush(ci, cs >= RS ? 1 : 0);
        if (++cs == SG) {
          cs = 0;
          ++ci;
        }
      }
    }
  }
  dec_grid_arrive<false>(a, sh);
  if (!dec_grid_wait<false>(a, sh, 2)) return;

  // ---------------------------------------------------------------- H: h = silu(g) * u
  // Item (slot sl, 4 columns f) with 8 lanes: for a unit one CTA streamed whole lane 0
  // reads part_g; for a split unit lane l adds the pieces of CTAs clo + l, clo + l + 8,
  // ... and a fixed butterfly adds the eight lanes.
  {
    const int S = sh.ex_first[n_u];
    const int f4 = Fm / 4, nitems = S * f4;
    const int grp = tid >> 3, sub = tid & 7;  // 32 groups per CTA
    const int passes = (nitems + 32 * G - 1) / (32 * G);
    for (int p = 0; p < passes; p += 2) {  // two items per group in flight
      int sl[2], fc[2];
      bool valid[2];
      float4 pgv[2][4], puv[2][4];
#pragma unroll
      for (int b2 = 0; b2 < 2; ++b2) {
        const int item = (int)blockIdx.x + G * (32 * (p + b2) + grp);
        sl[b2] = item / f4;
        fc[b2] = (item - sl[b2] * f4) * 4;
        valid[b2] = p + b2 < passes && item < nitems;
        int u = 0;
        if (valid[b2]) {
          u = sh.slot_u[sl[b2]];
          valid[b2] = fc[b2] < (u < n_routed ? F : Fs);
        }
#pragma unroll
        for (int m = 0; m < 4; ++m) pgv[b2][m] = puv[b2][m] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (!valid[b2]) continue;
        const int f = fc[b2];
        const int bpb = u < n_routed ? bpb_r : bpb_s;
        const int cb = (f >> 6) / bpb;
        const int i = (u < n_routed ? u * ncb_r : n_routed * ncb_r) + cb;
        const int ub = i * SG, um = ub + RS, ue = ub + SG;  // gate steps [ub, um), up steps [um, ue)
        const int clo = pht.cta_of((uint32_t)ub), chi = pht.cta_of((uint32_t)(ue - 1));
        if (clo == chi) {
          if (sub == 0) {
            const float* pg = a.part_g + (int64_t)sl[b2] * 2 * Fm + f;
            pgv[b2][0] = __ldcg(reinterpret_cast<const float4*>(pg));
            puv[b2][0] = __ldcg(reinterpret_cast<const float4*>(pg + Fm));
          }
        } else {
          const int row = sl[b2] - sh.ex_first[u], colp = f - cb * bpb * 64;
#pragma unroll
          for (int m = 0; m < 4; ++m) {  // up to 32 pieces in one round of loads
            const int q = clo + sub + 8 * m;
            if (q <= chi && pht.start[q] < pht.start[q + 1]) {
              const int ps = (q > clo || pht.start[clo] == ub) ? 2 * q : 2 * q + 1;
              const int lo = max(ub, pht.start[q]), hi = min(ue, pht.start[q + 1]);  // the piece's steps
              const float* pp = a.piece_g + ((int64_t)ps * 2 * T + row) * kDecGMaxCols + colp;
              if (lo < um) pgv[b2][m] = __ldcg(reinterpret_cast<const float4*>(pp));
              if (hi > um) puv[b2][m] = __ldcg(reinterpret_cast<const float4*>(pp + (int64_t)T * kDecGMaxCols));
            }
          }
          for (int q0 = clo + sub + 32; q0 <= chi; q0 += 8) {  // more than 32 pieces
            if (pht.start[q0] < pht.start[q0 + 1]) {
              const int lo = max(ub, pht.start[q0]), hi = min(ue, pht.start[q0 + 1]);
              const float* pp = a.piece_g + ((int64_t)2 * q0 * 2 * T + row) * kDecGMaxCols + colp;
              const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
              const float4 g4 = lo < um ? __ldcg(reinterpret_cast<const float4*>(pp)) : z4;
              const float4 u4 = hi > um ? __ldcg(reinterpret_cast<const float4*>(pp + (int64_t)T * kDecGMaxCols)) : z4;
              pgv[b2][3].x += g4.x; pgv[b2][3].y += g4.y; pgv[b2][3].z += g4.z; pgv[b2][3].w += g4.w;
              puv[b2][3].x += u4.x; puv[b2][3].y += u4.y; puv[b2][3].z += u4.z; puv[b2][3].w += u4.w;
            }
          }
        }
      }
#pragma unroll
      for (int b2 = 0; b2 < 2; ++b2) {
        float4 gs = pgv[b2][0], us = puv[b2][0];
#pragma unroll
        for (int m = 1; m < 4; ++m) {
          gs.x += pgv[b2][m].x; gs.y += pgv[b2][m].y; gs.z += pgv[b2][m].z; gs.w += pgv[b2][m].w;
          us.x += puv[b2][m].x; us.y += puv[b2][m].y; us.z += puv[b2][m].z; us.w += puv[b2][m].w;
        }
#pragma unroll
        for (int o = 4; o > 0; o >>= 1) {  // the eight lanes of the group, a fixed tree
          gs.x += __shfl_xor_sync(0xffffffffu, gs.x, o);
          gs.y += __shfl_xor_sync(0xffffffffu, gs.y, o);
          gs.z += __shfl_xor_sync(0xffffffffu, gs.z, o);
          gs.w += __shfl_xor_sync(0xffffffffu, gs.w, o);
          us.x += __shfl_xor_sync(0xffffffffu, us.x, o);
          us.y += __shfl_xor_sync(0xffffffffu, us.y, o);
          us.z += __shfl_xor_sync(0xffffffffu, us.z, o);
          us.w += __shfl_xor_sync(0xffffffffu, us.w, o);
        }
        if (valid[b2] && sub == 0) {
          const float h0 = gs.x * sigmoidf_(gs.x) * us.x, h1 = gs.y * sigmoidf_(gs.y) * us.y;
          const float h2 = gs.z * sigmoidf_(gs.z) * us.z, h3 = gs.w * sigmoidf_(gs.w) * us.w;
          __nv_bfloat162* dst = reinterpret_cast<__nv_bfloat162*>(a.hbuf + (int64_t)sl[b2] * Fm + fc[b2]);
          dst[0] = __floats2bfloat162_rn(h0, h1);
          dst[1] = __floats2bfloat162_rn(h2, h3);
        }
      }
    }
    // h is read next by the tensor-memory-access copies of other CTAs
    asm volatile("fence.proxy.async.global;" ::: "memory");
  }
  dec_grid_arrive<false>(a, sh);
  if (!dec_grid_wait<false>(a, sh, 3)) return;
  if (tid == 0) asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(smem_u32(&sh.h_ready)), "r"(1) : "memory");

  // ---------------------------------------------------------------- D: y = h W_down
  {
    float d0[4] = {0, 0, 0, 0}, d1[4] = {0, 0, 0, 0};
    for (DCur cc{0, 0}; cc.li < mine_d; d_advance(cc), ++j) {
      if (!wait_full(sh, a, j)) break;  // the barrier below makes every warp leave
      const int i = d_unit(cc), u = i / nhb;
      const uint32_t wt = smem_u32(tiles + (j % kDecBufs) * kDecTileBytes);
      const int nrows = min(kDecStepRows, fu(u) - cc.fk * kDecStepRows);
      uint32_t fa[16][4], fb[16][2];
      step_load_down(wt, nrows, fa, fb);
      release(sh, j);  // the tile is in registers: its buffer can be refilled meanwhile
      step_mma_down(nrows, fa, fb, d0, d1);
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
    }
  }
  dec_grid_arrive<false>(a, sh);
  if (!dec_grid_wait<false>(a, sh, 4)) return;

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

// [rows, cols] bf16, boxes of box_rows rows x 64 columns, 128-byte swizzle
static bool dec_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int box_rows) {
  auto fn = dec_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// rows of the slot-indexed buffers: the T * k routed pairs and T shared-expert tokens
static int64_t dec_slots(int64_t T, int64_t k) { return T * k + T; }

size_t decode_scratch_bytes(int64_t T, int64_t H, int64_t F, int64_t E, int64_t k, int64_t Fs) {
  const int64_t Fm = F > Fs ? F : Fs, S = dec_slots(T, k);
  auto up = [](int64_t n) { return (size_t)((n + 255) / 256 * 256); };
  return up(kDecRSlices * T * E * 4) + up(S * Fm * 2) + up(S * H * 4) + up(S * 2 * Fm * 4) +
         up((int64_t)2 * kDecMaxGrid * 2 * T * kDecGMaxCols * 4) + 256;
}

bool decode_supported(int64_t T, int64_t H, int64_t F, int64_t E, int64_t k, int64_t Fs) {
  return T >= 1 && T <= kDecMaxT && E <= kDecMaxE && k <= kDecMaxK && H <= kDecMaxH && F <= kDecMaxH &&
         Fs <= kDecMaxH && H % 64 == 0 && F % 64 == 0 && Fs % 64 == 0;
}

cudaError_t launch_decode_fwd(int T, int H, int F, int E, int k, int Fs, const void* x, const void* w_router,
                              const float* bias, const void* w_gate, const void* w_up, const void* w_down,
                              const void* ws_gate, const void* ws_up, const void* ws_down, void* y, int* topk_idx,
                              float* topk_w, int* user_idx, float* user_w, float* user_logits, void* scratch,
                              int* status, unsigned* sync, int num_sms, cudaStream_t st, unsigned stall,
                              uint64_t wait_ns) {
  const int64_t Fm = F > Fs ? F : Fs, S = dec_slots(T, k);
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
  b += up((int64_t)kDecRSlices * T * E * 4);
  a.hbuf = reinterpret_cast<__nv_bfloat16*>(b);
  b += up(S * Fm * 2);
  a.ypair = reinterpret_cast<float*>(b);
  b += up(S * H * 4);
  a.part_g = reinterpret_cast<float*>(b);
  b += up(S * 2 * Fm * 4);
  a.piece_g = reinterpret_cast<float*>(b);
  b += up((int64_t)2 * kDecMaxGrid * 2 * T * kDecGMaxCols * 4);
  a.status = status;
  a.sync = sync;  // zeroed by the caller on the same stream
  a.stall = stall;
  a.wait_ns = wait_ns;
  cudaError_t e = cudaSuccess;
  CUtensorMap mg, mu, md, msg, msu, msd, mh;
  bool ok = dec_map(&mg, w_gate, (int64_t)E * H, F, kDecGRows) && dec_map(&mu, w_up, (int64_t)E * H, F, kDecGRows) &&
            dec_map(&md, w_down, (int64_t)E * F, H, kDecBoxRows);
  if (Fs > 0)
    ok = ok && dec_map(&msg, ws_gate, H, Fs, kDecGRows) && dec_map(&msu, ws_up, H, Fs, kDecGRows) &&
         dec_map(&msd, ws_down, Fs, H, kDecBoxRows);
  else
    msg = msu = msd = mg;  // unused without a shared expert
  ok = ok && dec_map(&mh, a.hbuf, S, Fm, kDecDABoxRows);  // the A tiles of the down steps
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
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_decode_fwd, kDecBlock, smem);
      if (e != cudaSuccess) return e;
      if (per_sm < 1) return cudaErrorInvalidConfiguration;
      if (dev >= 0 && dev < 64) ready[dev] = true;
    }
  }
  void* args[] = {&mg, &mu, &md, &msg, &msu, &msd, &mh, &a};
  const int grid = num_sms < kDecMaxGrid ? num_sms : kDecMaxGrid;  // piece slots exist for kDecMaxGrid CTAs
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(k_decode_fwd), dim3(grid), dim3(kDecBlock),
                                     args, (size_t)smem, st);
}

}  // namespace moe
