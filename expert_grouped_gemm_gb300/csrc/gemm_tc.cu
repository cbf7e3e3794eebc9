// gemm_tc.cu -- persistent grouped GEMM on the 5th-generation tensor cores (sm_103a).
//
// Per CTA (64 + 32 * NEPI threads, one CTA per SM):
//   warp 0      TMA producer: loads A/B k-blocks of 64 into a STAGES-deep
//               ring of 128-byte-swizzled shared-memory tiles. An MN-major
//               operand (row-major [K, MN]) is read through a 3-D view
//               (64 columns, K rows, column chunk) so one bulk-tensor copy
//               fills all of its 64-column chunks.
//   warp 1      MMA issuer: tcgen05.mma (M=128, N=BN, K=16) into one of two
//               tensor-memory accumulators, commits free smem slots back.
//   warps 2..    NEPI epilogue warps (4, or 8 with two per TMEM lane quarter):
//               tcgen05.ld of the finished accumulator (one row per thread),
//               fused epilogue (SwiGLU fwd/bwd, store, dW), then the results
//               go through a 128-byte-swizzled staging tile in shared memory
//               and out with TMA bulk tensor stores of 32 rows x 64 columns (16
//               rows at a group's padded end, which is a multiple of 16, so a
//               store never reaches into another group's rows); or, for fp32
//               outputs (router logits, K-split partial sums), direct stores.
// Tiles (group, m-block, n-block, K split) come from device-side group offsets
// and per-tile records, so the host never learns the per-group row counts.
// Variable-K groups are visited heaviest first. Every barrier wait is bounded;
// a wait that runs out sets MOE_ERR_TIMEOUT in the status word, the CTA drains
// its own copies and MMAs, frees its tensor memory and returns.
#include <cudaTypedefs.h>

#include <mutex>

#include "epilogue.cuh"
#include "gemm_launch.h"

namespace moe {

constexpr int kStageRowBytes = 128;                   // 64 bf16 per staged row
constexpr int kStageTileBytes = 32 * kStageRowBytes;  // one warp's 32 rows x 64 columns (4 KB)

// CTAs per tile of the variable-M expert GEMMs (gate/up, down, dH, dX): 1 = one CTA per
// 128-row tile (default); 2 = CTA pair (cta_group::2, 256 rows by 256 columns; each CTA
// loads its 128 rows of A and half of B, so a k-block costs a CTA 32 KB instead of 48 KB
// and six stages fit in shared memory, but experts are padded to 256-row tiles). Pairs
// measured slower at the Qwen3 and GLM-4.5 shapes. The variable-K dW GEMMs use one CTA.
#ifndef MOE_VARM_CTAS
#define MOE_VARM_CTAS 1
#endif

template <int BN, int STAGES, int EPI_WARP_BYTES, int CTAS, int NEPI>
struct TcCfg {
  static constexpr int THREADS = 64 + 32 * NEPI;            // producer, MMA, NEPI epilogue warps
  static constexpr int A_BYTES = kTileM * kTileK * 2;       // 16 KB: this CTA's 128 rows
  static constexpr int B_BYTES = BN * kTileK * 2 / CTAS;    // this CTA's share of the BN columns
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;     // per CTA
  static constexpr int TILE_M = kTileM * CTAS;              // rows of one (pair) tile
  static constexpr int EPI_OFF = STAGES * STAGE_BYTES;
  static constexpr int BAR_OFF = EPI_OFF + NEPI * EPI_WARP_BYTES;
  static constexpr int SMEM = BAR_OFF + 256 + 1024;  // barriers + 1 KB alignment slack
  static constexpr uint32_t TMEM_COLS = 2 * BN;      // two accumulators
  static constexpr bool MN3D = (BN == 256);           // MN-major operands through 3-D views
};

// kb0 / kblocks: this tile's k-blocks (all of them without a K split); kb_last:
// the group's last k-block (variable K: the one a group's rows end in)
struct TileInfo {
  int g, m0, nt, rows, off, kblocks, kb0, kb_last, split;
};

template <int BN>
__device__ __forceinline__ int n_tiles(const GemmArgs& a) {
  const int w = a.paired ? BN / 2 : BN;
  return (a.N + w - 1) / w;
}

// The record behind tile t (one 16-byte load), when the schedule has records;
// the roles load the next tile's record while they work on the current one, so
// the load latency stays off their critical path.
template <int BN, int TILE_M>
__device__ __forceinline__ int4 load_tile_rec(const GemmArgs& a, int t, int NT) {
  if (a.ksplit > 1) t /= a.ksplit;
  if (a.var_k) {
    if (a.grp_rec) return __ldg(a.grp_rec + t / (((a.M + TILE_M - 1) / TILE_M) * NT));
  } else if (TILE_M == kTileM && a.tile_rec) {
    return __ldg(a.tile_rec + t / NT);
  } else if (TILE_M == 2 * kTileM && a.tile_rec2) {
    return __ldg(a.tile_rec2 + t / NT);
  }
  return make_int4(0, 0, 0, 0);
}

template <int BN, int TILE_M>
__device__ __forceinline__ TileInfo decode_tile(const GemmArgs& a, int t, int NT, int4 rec) {
  TileInfo ti;
  const int* toff = TILE_M == kTileM ? a.tile_off : a.tile_off2;
  const int ks = a.ksplit > 1 ? a.ksplit : 1;
  ti.split = t % ks;  // consecutive tiles are the splits of one output tile
  t /= ks;
  if (a.var_k) {
    const int MT = (a.M + TILE_M - 1) / TILE_M;
    const int gi = t / (MT * NT);
    const int rem = t - gi * MT * NT;
    ti.m0 = (rem / NT) * TILE_M;
    ti.nt = rem % NT;
    if (a.grp_rec) {
      ti.g = rec.x;
      ti.rows = rec.y;
      ti.off = rec.z;
    } else {
      ti.g = a.g_order ? a.g_order[gi] : gi;
      ti.rows = grp_rows(a, ti.g);
      ti.off = grp_off(a, ti.g);
    }
    ti.kblocks = (ti.rows + kTileK - 1) / kTileK;
  } else if ((TILE_M == kTileM && a.tile_rec) || (TILE_M == 2 * kTileM && a.tile_rec2)) {
    ti.nt = t - (t / NT) * NT;
    ti.g = rec.x;
    ti.m0 = rec.y;
    ti.rows = rec.z;
    ti.off = rec.w;
    ti.kblocks = a.K / kTileK;
  } else {
    const int u = t / NT;
    ti.nt = t - u * NT;
    int g = 0;
    if (toff) {  // last g with toff[g] <= u
      int lo = 0, hi = a.G - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (toff[mid] <= u) lo = mid; else hi = mid - 1;
      }
      g = lo;
      ti.m0 = (u - toff[g]) * TILE_M;
    } else {
      ti.m0 = u * TILE_M;
    }
    ti.g = g;
    ti.rows = grp_rows(a, g);
    ti.off = grp_off(a, g);
    ti.kblocks = a.K / kTileK;
  }
  ti.kb0 = 0;
  ti.kb_last = ti.kblocks - 1;
  if (ks > 1) {  // this split's share of the k-blocks
    const int per = (ti.kblocks + ks - 1) / ks;
    ti.kb0 = ti.split * per;
    ti.kblocks = max(0, min(per, ti.kblocks - ti.kb0));
  }
  return ti;
}

template <int BN, int TILE_M>
__device__ __forceinline__ int total_tiles(const GemmArgs& a) {
  const int NT = n_tiles<BN>(a);
  const int* toff = TILE_M == kTileM ? a.tile_off : a.tile_off2;
  const int ks = a.ksplit > 1 ? a.ksplit : 1;
  if (a.var_k) return a.G * ((a.M + TILE_M - 1) / TILE_M) * NT * ks;
  const int mt = toff ? toff[a.G] : (a.rows_const + TILE_M - 1) / TILE_M;
  return mt * NT * ks;
}

// ---------------------------------------------------------------- epilogue pieces
// Byte offset of 16-byte chunk j (0..7) of row r in a 128-byte-swizzled staging
// tile: the layout a TMA store with 128-byte swizzle reads.
__device__ __forceinline__ uint32_t stage_off(int r, int j) { return r * kStageRowBytes + ((j ^ (r & 7)) << 4); }

// SwiGLU backward: coalesced asynchronous copy of the a|b values of one
// 64-column chunk for one warp's 32 rows (eight threads per row, 16 bytes each)
// into the (a tile, b tile) pair at `buf`; rows at or past `rows_left` are skipped.
__device__ __forceinline__ void aux_prefetch(uint32_t buf, const __nv_bfloat16* ab, int64_t row0, int64_t ld, int N,
                                             int n0, int rows_left, int lane) {
  if (n0 < N) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = (lane >> 3) + 4 * i, j = lane & 7;
      if (r < rows_left) {
        const __nv_bfloat16* src = ab + (row0 + r) * ld + n0 + 8 * j;
        cp_async16(buf + stage_off(r, j), src);
        cp_async16(buf + kStageTileBytes + stage_off(r, j), src + N);
      }
    }
  }
  cp_async_commit();
}

template <int BN, int STAGES, int EPI_WARP_BYTES, int EPI, int CTAS, int NEPI>
__global__ void __launch_bounds__(64 + 32 * NEPI, 1)
    tc_grouped_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                    const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmO0,
                    const __grid_constant__ CUtensorMap tmO1, const __grid_constant__ CUtensorMap tmO0h,
                    const __grid_constant__ CUtensorMap tmO1h, const GemmArgs args) {
  using C = TcCfg<BN, STAGES, EPI_WARP_BYTES, CTAS, NEPI>;
  constexpr bool PAIR = CTAS == 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // In a CTA pair, rank 0 (the leader) issues the MMAs for both CTAs; each CTA
  // loads its own 128 rows of A and its half of the B columns, and its tensor
  // memory receives its own 128 rows of the accumulator.
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  const int cluster_id = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int num_clusters = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);   // the leader's producer arms it for both CTAs' bytes
      mbar_init(&empty[s], 1);  // one MMA commit (multicast to both CTAs of a pair)
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], NEPI * CTAS);  // one arrive per epilogue warp of each CTA
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    if constexpr (PAIR) tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
    else tmem_alloc(tmem_slot, C::TMEM_COLS);
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync_all();  // both CTAs' barriers exist before any remote arrive
  tc_fence_after();
  pdl_wait();  // the set-up above touched no global memory; everything below may read the previous kernel's outputs
  const uint32_t tmem_base = *tmem_slot;
  // leader barriers as seen from this CTA (shared::cluster addresses)
  const uint32_t full0 = PAIR ? mapa_shared(smem_u32(full), 0) : smem_u32(full);
  const uint32_t tempty0 = PAIR ? mapa_shared(smem_u32(tempty), 0) : smem_u32(tempty);

  const int NT = n_tiles<BN>(args);
  const int total = total_tiles<BN, C::TILE_M>(args);

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB0);
    tma_prefetch_desc(&tmB1);
    int stage = 0;
    uint32_t phase = 0;
    int issued_parity[STAGES];
#pragma unroll
    for (int s = 0; s < STAGES; ++s) issued_parity[s] = -1;
    bool ok = true;
    // Every TMA box of k-block kb of tile ti, loaded into the stage at sa with
    // completion on the barrier fb.
    auto issue = [&](const TileInfo& ti, int kb, uint32_t sa, uint32_t fb) {
      auto load2 = [&](uint32_t dst, const CUtensorMap* map, int c0, int c1) {
        if constexpr (PAIR) tma_load_2d_pair(dst, map, fb, c0, c1);
        else tma_load_2d(dst, map, fb, c0, c1);
      };
      auto load3 = [&](uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2) {
        if constexpr (PAIR) tma_load_3d_pair(dst, map, fb, c0, c1, c2);
        else tma_load_3d(dst, map, fb, c0, c1, c2);
      };
      const int m0c = ti.m0 + (int)rank * kTileM;  // this CTA's rows (var-M) / columns (var-K) of A
      const uint32_t sb = sa + C::A_BYTES;
      // A
      if (!args.var_k) {
        load2(sa, &tmA, kb * kTileK, ti.off + m0c);
      } else if (C::MN3D) {
        load3(sa, &tmA, 0, ti.off + kb * kTileK, m0c / 64);
      } else {
        load2(sa, &tmA, m0c, ti.off + kb * kTileK);
        load2(sa + 8192, &tmA, m0c + 64, ti.off + kb * kTileK);
      }
      // B (a pair splits the BN columns: rank 0 the first half, rank 1 the second)
      if (args.b_kmajor) {
        const bool second = args.k_split > 0 && kb * kTileK >= args.k_split;
        const int kk = second ? kb - args.k_split / kTileK : kb;
        load2(sb, second ? &tmB1 : &tmB0, kk * kTileK, ti.g * args.N + ti.nt * BN + (int)rank * (BN / CTAS));
      } else {
        const int brow = args.var_k ? ti.off + kb * kTileK : ti.g * args.K + kb * kTileK;
        if (C::MN3D) {
          if (args.paired) {  // halves of BN/2 columns: B0, then B1 at column offset b1_col
            if (!PAIR || rank == 0) load3(sb, &tmB0, 0, brow, ti.nt * (BN / 128));
            if (!PAIR || rank == 1)
              load3(PAIR ? sb : sb + BN / 2 * 128, &tmB1, 0, brow, args.b1_col / 64 + ti.nt * (BN / 128));
          } else {
            load3(sb, &tmB0, 0, brow, ti.nt * (BN / 64) + (int)rank * (BN / 64 / CTAS));
          }
        } else {
#pragma unroll
          for (int c = 0; c < BN / 64; ++c) {
            int col;
            const CUtensorMap* map = &tmB0;
            if (args.paired) {
              const int half = c / (BN / 128);
              col = ti.nt * (BN / 2) + (c % (BN / 128)) * 64;
              if (half) {
                map = &tmB1;
                col += args.b1_col;
              }
            } else {
              col = ti.nt * BN + c * 64;
            }
            load2(sb + c * 8192, map, col, brow);
          }
        }
      }
    };
    int4 rec = cluster_id < total ? load_tile_rec<BN, C::TILE_M>(args, cluster_id, NT) : make_int4(0, 0, 0, 0);
    for (int t = cluster_id; t < total && ok; t += num_clusters) {
      const TileInfo ti = decode_tile<BN, C::TILE_M>(args, t, NT, rec);
      if (t + num_clusters < total) rec = load_tile_rec<BN, C::TILE_M>(args, t + num_clusters, NT);
      for (int kb = ti.kb0; kb < ti.kb0 + ti.kblocks; ++kb) {
        if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        const uint32_t sa = smem_u32(smem + stage * C::STAGE_BYTES);
        const uint32_t fb = full0 + stage * 8;  // the leader's full barrier of this stage
        if (leader) mbar_arrive_expect_tx(&full[stage], CTAS * C::STAGE_BYTES);
        issued_parity[stage] = (int)phase;
        issue(ti, kb, sa, fb);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    // make sure no copy of ours is still landing in shared memory (the leader's
    // full barriers also count the peer's bytes)
    if (leader)
      for (int s = 0; s < STAGES; ++s)
        if (issued_parity[s] >= 0) mbar_wait_timed(&full[s], (uint32_t)issued_parity[s], 200000000ull);
  } else if (warp == 1 && lane == 0 && leader) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t idesc = idesc_bf16(C::TILE_M, BN, args.var_k, args.b_kmajor ? 0 : 1);
    // shared-memory descriptors of stage 0; a K-major operand advances 32 bytes per
    // k16 step, an MN-major one (a 3-D box of 64-row chunks) 2048 bytes
    const uint32_t sa0 = smem_u32(smem);
    const uint64_t adesc0 = args.var_k ? sdesc_sw128(sa0, 8192, 1024) : sdesc_sw128(sa0, 16, 1024);
    const uint64_t bdesc0 =
        args.b_kmajor ? sdesc_sw128(sa0 + C::A_BYTES, 16, 1024) : sdesc_sw128(sa0 + C::A_BYTES, 8192, 1024);
    const uint64_t astep = args.var_k ? 2048 >> 4 : 32 >> 4;
    const uint64_t bstep = args.b_kmajor ? 32 >> 4 : 2048 >> 4;
    auto mma = [&](uint32_t d, uint64_t a_desc, uint64_t b_desc, uint32_t accumulate) {
      if constexpr (PAIR) tc_mma_bf16_pair(d, a_desc, b_desc, idesc, accumulate);
      else tc_mma_bf16(d, a_desc, b_desc, idesc, accumulate);
    };
    int stage = 0;
    uint32_t phase = 0;
    int acc_i = 0;
    bool ok = true;
    int4 rec = cluster_id < total ? load_tile_rec<BN, C::TILE_M>(args, cluster_id, NT) : make_int4(0, 0, 0, 0);
    for (int t = cluster_id; t < total && ok; t += num_clusters) {
      const TileInfo ti = decode_tile<BN, C::TILE_M>(args, t, NT, rec);
      if (t + num_clusters < total) rec = load_tile_rec<BN, C::TILE_M>(args, t + num_clusters, NT);
      if (ti.kblocks == 0) continue;
      const int acc = acc_i & 1;
      const uint32_t acc_par = (uint32_t)((acc_i >> 1) & 1);
      const bool free_acc = PAIR ? mbar_wait_bounded_cluster(&tempty[acc], acc_par ^ 1u, abort_flag)
                                 : mbar_wait_bounded(&tempty[acc], acc_par ^ 1u, abort_flag);
      if (!free_acc) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
      for (int kb = ti.kb0; kb < ti.kb0 + ti.kblocks; ++kb) {
        if (!mbar_wait_bounded(&full[stage], phase, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // descriptors of this stage: the k16 steps only move the start address
        const uint64_t ad = adesc0 + (uint64_t)(stage * (C::STAGE_BYTES >> 4));
        const uint64_t bd = bdesc0 + (uint64_t)(stage * (C::STAGE_BYTES >> 4));
        const uint32_t acc0 = kb != ti.kb0 ? 1u : 0u;
        if (!(args.var_k && kb == ti.kb_last)) {  // full k-block: four k16 steps
          mma(d_tmem, ad, bd, acc0);
          mma(d_tmem, ad + astep, bd + bstep, 1u);
          mma(d_tmem, ad + 2 * astep, bd + 2 * bstep, 1u);
          mma(d_tmem, ad + 3 * astep, bd + 3 * bstep, 1u);
        } else {  // a variable-K group's last k-block: its rows rounded up to 16
          const int nk = (ti.rows - kb * kTileK + 15) / 16;
          for (int kk = 0; kk < nk; ++kk) mma(d_tmem, ad + kk * astep, bd + kk * bstep, kk != 0 ? 1u : acc0);
        }
        if constexpr (PAIR) tc_commit_pair_mc(&empty[stage]);
        else tc_commit(&empty[stage]);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      if constexpr (PAIR) tc_commit_pair_mc(&tfull[acc]);
      else tc_commit(&tfull[acc]);
      ++acc_i;
    }
    // wait until every MMA issued by this thread has completed
    if constexpr (PAIR) tc_commit_pair(drain);
    else tc_commit(drain);
    mbar_wait_timed(drain, 0, 200000000ull);
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may read
    const int row = q * 32 + lane;
    const int ew = warp - 2;  // epilogue warp index; with 8 warps, two share a lane quarter
    const uint32_t wstage = smem_u32(smem + C::EPI_OFF + ew * EPI_WARP_BYTES);
    constexpr bool tma_out = EPI != EPI_F32;
    constexpr bool bwd = EPI == EPI_SWIGLU_BWD;
    constexpr bool fwd = EPI == EPI_SWIGLU_FWD;
    // dW of a pair of weights (gate and up) with one staging tile per warp: dW_up goes
    // out through the tile after dW_gate's store has read it
    constexpr bool serial_pair = EPI == EPI_DW && EPI_WARP_BYTES < 2 * kStageTileBytes;
    const bool pair_later = serial_pair && args.paired;
    // staged outputs per chunk (the SwiGLU forward stages a|b, then h in the a tile)
    const int nout = (fwd || bwd || (EPI == EPI_DW && args.paired && !serial_pair)) ? 2 : 1;
    // one output alternates two staging sets when room allows; otherwise one set
    const int nbuf = (nout == 1 && EPI_WARP_BYTES >= 2 * kStageTileBytes) ? 2 : 1;
    // SwiGLU bwd: the a and b tiles of one chunk; da and db are staged in place over them
    const uint32_t aux_buf = wstage;
    const int W = args.paired ? BN / 2 : BN;                // output columns per tile
    const int CW = W / 64;                                  // 64-column chunks per tile
    constexpr int kSplit = NEPI / 4;                        // warps sharing one lane quarter
    const int c_begin = (ew / 4) * (CW / kSplit);           // this warp's chunks of the tile
    const int c_end = c_begin + CW / kSplit;
    const __nv_bfloat16* ab_aux = reinterpret_cast<const __nv_bfloat16*>(args.aux);
    int acc_i = 0;
    int sc = 0;  // staging sets used so far by this warp
    uint32_t ra[32], rb[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) rb[i] = 0u;  // only paired modes load it
    int4 rec = cluster_id < total ? load_tile_rec<BN, C::TILE_M>(args, cluster_id, NT) : make_int4(0, 0, 0, 0);
    for (int t = cluster_id; t < total; t += num_clusters) {
      TileInfo ti = decode_tile<BN, C::TILE_M>(args, t, NT, rec);
      if (t + num_clusters < total) rec = load_tile_rec<BN, C::TILE_M>(args, t + num_clusters, NT);
      ti.m0 += (int)rank * kTileM;  // this CTA's 128 rows of the (pair) tile
      const int m = ti.m0 + row;
      const int ncol0 = ti.nt * W;
      // rows of this tile that may be written, and the output row of this warp's box
      int lim;
      int64_t out_row0;
      if (args.var_k) {
        lim = args.M - ti.m0;
        out_row0 = (int64_t)ti.g * args.M + ti.m0 + q * 32;
      } else {
        lim = round_pad(ti.rows) - ti.m0;
        out_row0 = (int64_t)ti.off + ti.m0 + q * 32;
      }
      const int rows_left = lim - q * 32;                    // rows of this warp's 32 that are written
      const bool real = args.var_k || m < ti.rows;           // var-M rows past the group end are zero padding
      const int64_t aux_row0 = (int64_t)ti.off + ti.m0 + q * 32;
      if (bwd) {  // the previous tile's last da|db stores must have read the aux tiles
        if (lane == 0) bulk_wait_read_all();
        __syncwarp();
        aux_prefetch(aux_buf, ab_aux, aux_row0, args.ld_aux, args.N, ncol0 + c_begin * 64, rows_left, lane);
      }
      // variable-K group without rows, or a K split without k-blocks: the output is zero
      const bool empty_tile = ti.kblocks == 0;
      const int acc = acc_i & 1;
      if (!empty_tile) {
        const uint32_t acc_par = (uint32_t)((acc_i >> 1) & 1);
        if (!mbar_wait_bounded(&tfull[acc], acc_par, abort_flag)) break;
        tc_fence_after();
      }
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
      const bool live = !empty_tile && real;
      for (int c = c_begin; c < c_end; ++c) {
        const int n0 = ncol0 + c * 64;
        const bool store = rows_left > 0 && n0 < args.N;
        uint32_t set = wstage;
        if (tma_out && store && !bwd) {
          set = wstage + (nbuf == 2 ? (uint32_t)((sc & 1) * kStageTileBytes) : 0u);
          // the set must be free: the bulk stores that last used it have read it
          if (lane == 0) {
            if (nbuf == 2) bulk_wait_read_but1(); else bulk_wait_read_all();
          }
          __syncwarp();
        }
        if (bwd) {  // a|b of this chunk has landed
          cp_async_wait<0>();
          __syncwarp();
        }
        uint4 hpk[8];  // SwiGLU forward: h of this chunk, staged after a|b have been read
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {  // two 32-column halves of the chunk
          if (!empty_tile) {
            tmem_ld32_async(taddr + c * 64 + hh * 32, ra);
            if (args.paired) {  // gate and up columns of this half under one wait
              tmem_ld32_async(taddr + BN / 2 + c * 64 + hh * 32, rb);
              tmem_ld_wait(ra);
              tmem_ld_order(rb);
            } else {
              tmem_ld_wait(ra);
            }
          }
          if constexpr (!tma_out) {  // fp32: direct 16-byte stores, one row per thread
            const int nh = n0 + hh * 32;
            const bool row_ok = args.var_k ? m < args.M : m < ti.rows;
            if (row_ok && nh < args.N) {
              const int64_t orow = args.var_k ? (int64_t)ti.g * args.M + m : (int64_t)ti.off + m;
              float* o = reinterpret_cast<float*>(args.out0) + ti.split * args.part_stride + orow * args.ldo + nh;
              const int nv = min(32, args.N - nh);
#pragma unroll
              for (int half = 0; half < 2; ++half) {  // the paired second half goes to column N
                if (half && !args.paired) break;
                float* oh = o + (half ? args.N : 0);
                const uint32_t* r = half ? rb : ra;
                if (nv == 32 && (reinterpret_cast<uintptr_t>(oh) & 15) == 0) {
#pragma unroll
                  for (int i = 0; i < 32; i += 4)
                    *reinterpret_cast<uint4*>(oh + i) = empty_tile ? make_uint4(0, 0, 0, 0)
                                                                   : make_uint4(r[i], r[i + 1], r[i + 2], r[i + 3]);
                } else {
#pragma unroll
                  for (int i = 0; i < 32; ++i)
                    if (i < nv) oh[i] = empty_tile ? 0.0f : __uint_as_float(r[i]);
                }
              }
            }
            continue;
          }
#pragma unroll
          for (int g8 = 0; g8 < 4; ++g8) {
            const int j = hh * 4 + g8;  // 16-byte chunk of the staged 128-byte row
            float x0[8], x1[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              x0[i] = live ? __uint_as_float(ra[8 * g8 + i]) : 0.0f;
              x1[i] = live ? __uint_as_float(rb[8 * g8 + i]) : 0.0f;
            }
            if constexpr (fwd) {
              float h[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) h[i] = x0[i] * sigmoidf_(x0[i]) * x1[i];
              hpk[j] = f_to_bf16x8(h);
              if (store) {
                st_shared_v4(set + stage_off(lane, j), f_to_bf16x8(x0));
                st_shared_v4(set + kStageTileBytes + stage_off(lane, j), f_to_bf16x8(x1));
              }
            } else if constexpr (bwd) {
              float av[8], bv[8], da[8], db[8];
              bf16x8_to_f(ld_shared_v4(aux_buf + stage_off(lane, j)), av);
              bf16x8_to_f(ld_shared_v4(aux_buf + kStageTileBytes + stage_off(lane, j)), bv);
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const float s = sigmoidf_(av[i]);
                da[i] = x0[i] * bv[i] * s * (1.0f + av[i] * (1.0f - s));
                db[i] = x0[i] * av[i] * s;
              }
              if (store) {  // in place: each thread overwrites only what it just read
                st_shared_v4(aux_buf + stage_off(lane, j), f_to_bf16x8(da));
                st_shared_v4(aux_buf + kStageTileBytes + stage_off(lane, j), f_to_bf16x8(db));
              }
            } else {  // EPI_DW / EPI_STORE
              if (!store) continue;
              st_shared_v4(set + stage_off(lane, j), f_to_bf16x8(x0));
              if (nout > 1) st_shared_v4(set + kStageTileBytes + stage_off(lane, j), f_to_bf16x8(x1));
              else if (pair_later) hpk[j] = f_to_bf16x8(x1);
            }
          }
        }
        if (!tma_out) continue;
        if (!store) {
          if (bwd && c + 1 < c_end) {
            __syncwarp();
            aux_prefetch(aux_buf, ab_aux, aux_row0, args.ld_aux, args.N, n0 + 64, rows_left, lane);
          }
          continue;
        }
        ++sc;
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          // a | b (or da | db) go to the two halves of one a|b row; dW_up next to dW_gate
          const bool ab_row = fwd || bwd;
          const int c1 = ab_row ? args.N + n0 : n0;
          const bool full_box = rows_left >= 32;  // else a 16-row box ends at the group's padded end
          const CUtensorMap* o0 = full_box ? &tmO0 : &tmO0h;
          const CUtensorMap* o1 = ab_row ? o0 : (full_box ? &tmO1 : &tmO1h);
          tma_store_2d(o0, set, n0, (int)out_row0);
          if (nout > 1) tma_store_2d(o1, set + kStageTileBytes, c1, (int)out_row0);
          bulk_commit();
        }
        if (bwd && c + 1 < c_end) {  // the a|b tiles are free once da|db have been read out
          if (lane == 0) bulk_wait_read_all();
          __syncwarp();
          aux_prefetch(aux_buf, ab_aux, aux_row0, args.ld_aux, args.N, n0 + 64, rows_left, lane);
        }
        if (fwd || pair_later) {  // h (dW_up) goes out through the a (dW_gate) tile once it has been read
          if (lane == 0) bulk_wait_read_all();
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 8; ++j) st_shared_v4(set + stage_off(lane, j), hpk[j]);
          fence_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(rows_left >= 32 ? &tmO1 : &tmO1h, set, n0, (int)out_row0);
            bulk_commit();
          }
        }
      }
      if (!empty_tile) {  // this warp is done with the accumulator: tell the MMA issuer
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if constexpr (PAIR) mbar_arrive_cluster(tempty0 + acc * 8);
          else mbar_arrive(&tempty[acc]);
        }
        ++acc_i;
      }
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync_all();  // no CTA of the pair leaves while the other still uses it
  tc_fence_after();
  if (threadIdx.x == 0 && *abort_flag) set_status(args.status, MOE_ERR_TIMEOUT);
  if (warp == 2) {
    if constexpr (PAIR) tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    else tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------- host side

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// 2-D bf16 view [rows, cols] (cols contiguous) with box [box_rows, box_cols], 128-byte
// swizzle; out-of-bounds elements read as zero and are dropped on store.
static bool make_map_2d(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int box_cols, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D view of a row-major [rows, cols] bf16 matrix (cols a multiple of 64):
// (64 columns, row, 64-column chunk) with strides (2 B, cols*2 B, 128 B).
// A box (64, box_rows, box_chunks) lands in shared memory as box_chunks
// consecutive [box_rows][64] tiles: the MN-major operand layout.
static bool make_map_mn3d(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int box_rows, int box_chunks) {
  auto fn = encode_fn();
  if (!fn || cols % 64) return false;
  cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)(cols / 64)};
  cuuint64_t strides[2] = {(cuuint64_t)cols * 2, 128};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, (cuuint32_t)box_chunks};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, int STAGES, int EPI_WARP_BYTES, int EPI, int CTAS, int NEPI = 4>
static cudaError_t launch_cfg(const GemmArgs& a, cudaStream_t st, int num_sms) {
  using C = TcCfg<BN, STAGES, EPI_WARP_BYTES, CTAS, NEPI>;
  static_assert(C::SMEM <= 232448, "shared memory budget");
  static_assert(CTAS == 1 || BN == 256, "CTA pairs use the 256-column tile");
  static_assert(NEPI == 4 || NEPI == 8, "four or eight epilogue warps");
  if (a.epi != EPI) return cudaErrorInvalidValue;
  if (NEPI == 8 && ((a.paired ? BN / 2 : BN) / 64) % 2) return cudaErrorInvalidValue;
  auto kern = tc_grouped_gemm<BN, STAGES, EPI_WARP_BYTES, EPI, CTAS, NEPI>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  CUtensorMap mA, mB0, mB1, mO0, mO1, mO0h, mO1h;
  bool ok;
  if (!a.var_k)
    ok = make_map_2d(&mA, a.A, a.a_rows, a.lda, 64, kTileM);
  else if (C::MN3D)
    ok = make_map_mn3d(&mA, a.A, a.a_rows, a.lda, kTileK, kTileM / 64);
  else
    ok = make_map_2d(&mA, a.A, a.a_rows, a.lda, 64, kTileK);
  const void* b1 = a.B1 ? a.B1 : a.B0;
  if (a.b_kmajor) {  // each CTA loads BN/CTAS rows of B
    ok = ok && make_map_2d(&mB0, a.B0, a.b_rows, a.ldb, 64, BN / CTAS);
    ok = ok && make_map_2d(&mB1, b1, a.b_rows, a.ldb, 64, BN / CTAS);
  } else if (C::MN3D) {  // each CTA loads BN/CTAS columns of B (paired: one half each)
    const int chunks = (a.paired && CTAS == 1) ? BN / 128 : BN / 64 / CTAS;
    ok = ok && make_map_mn3d(&mB0, a.B0, a.b_rows, a.ldb, kTileK, chunks);
    ok = ok && make_map_mn3d(&mB1, b1, a.b_rows, a.ldb, kTileK, chunks);
  } else {
    ok = ok && make_map_2d(&mB0, a.B0, a.b_rows, a.ldb, 64, kTileK);
    ok = ok && make_map_2d(&mB1, b1, a.b_rows, a.ldb, 64, kTileK);
  }
  if (a.epi == EPI_F32) {
    mO0 = mO1 = mO0h = mO1h = mA;  // unused: fp32 outputs are stored directly
  } else {
    // output views: [out_rows, ld] for permuted / single-group outputs, [G*M, ld] for dW
    const int64_t orows = a.var_k ? (int64_t)a.G * a.M : a.out_rows;
    const void* o1 = a.out1 ? a.out1 : a.out0;
    const int64_t ld1 = (a.epi == EPI_SWIGLU_FWD) ? a.ldo1 : a.ldo;
    ok = ok && make_map_2d(&mO0, a.out0, orows, a.ldo, 64, 32) && make_map_2d(&mO0h, a.out0, orows, a.ldo, 64, 16);
    ok = ok && make_map_2d(&mO1, o1, orows, ld1, 64, 32) && make_map_2d(&mO1h, o1, orows, ld1, 64, 16);
  }
  if (!ok) return cudaErrorInvalidValue;
  if constexpr (CTAS == 1) {
    e = launch_pdl(kern, num_sms, C::THREADS, C::SMEM, st, mA, mB0, mB1, mO0, mO1, mO0h, mO1h, a);
    return e != cudaSuccess ? e : cudaGetLastError();
  } else {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // as many CTA pairs as can be resident at once (persistent schedule)
    cfg.gridDim = dim3(2 * (num_sms / 2));
    int max_clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&max_clusters, kern, &cfg) == cudaSuccess && max_clusters > 0 &&
        2 * max_clusters < (int)cfg.gridDim.x)
      cfg.gridDim = dim3(2 * max_clusters);
    e = cudaLaunchKernelEx(&cfg, kern, mA, mB0, mB1, mO0, mO1, mO0h, mO1h, a);
    return e != cudaSuccess ? e : cudaGetLastError();
  }
}

// Staging bytes one epilogue warp needs: nout 4 KB tiles (one output with room
// for two alternates two sets; the SwiGLU forward reuses its a tile for h),
// plus an a|b tile pair for the SwiGLU backward.
static int staging_bytes(const GemmArgs& a) {
  if (a.epi == EPI_F32) return 0;
  if (a.epi == EPI_SWIGLU_FWD) return 2 * kStageTileBytes;
  if (a.epi == EPI_SWIGLU_BWD) return 2 * kStageTileBytes;  // a|b tiles, da|db staged in place
  return kStageTileBytes;
}

cudaError_t launch_tc_gemm(const GemmArgs& a, int bn, cudaStream_t st, int num_sms, int /*max_tiles_hint*/) {
  const int need = staging_bytes(a);
  constexpr int kT = kStageTileBytes;
  if (bn == 128) {
    if (need > kT) return cudaErrorInvalidValue;
    if (a.epi == EPI_F32) return launch_cfg<128, 6, kT, EPI_F32, 1>(a, st, num_sms);
    if (a.epi == EPI_DW) return launch_cfg<128, 6, kT, EPI_DW, 1>(a, st, num_sms);
    return cudaErrorInvalidValue;
  }
  // 256-column tiles: the variable-M GEMMs as CTA pairs (or single CTAs), dW single CTAs
  switch (a.epi) {
#if MOE_VARM_CTAS == 2
    case EPI_SWIGLU_BWD:
      if (need > 4 * kT) return cudaErrorInvalidValue;
      return launch_cfg<256, 5, 4 * kT, EPI_SWIGLU_BWD, 2>(a, st, num_sms);
    case EPI_SWIGLU_FWD:
      if (need > 2 * kT) return cudaErrorInvalidValue;
      return launch_cfg<256, 6, 2 * kT, EPI_SWIGLU_FWD, 2>(a, st, num_sms);
    case EPI_STORE:
      if (need > 2 * kT) return cudaErrorInvalidValue;
      return launch_cfg<256, 6, 2 * kT, EPI_STORE, 2>(a, st, num_sms);
#else
    case EPI_SWIGLU_BWD:
      if (need > 2 * kT) return cudaErrorInvalidValue;
      return launch_cfg<256, 4, 2 * kT, EPI_SWIGLU_BWD, 1>(a, st, num_sms);
    case EPI_SWIGLU_FWD:
      if (need > 2 * kT) return cudaErrorInvalidValue;
      return launch_cfg<256, 4, 2 * kT, EPI_SWIGLU_FWD, 1>(a, st, num_sms);
    case EPI_STORE:
      if (need > 2 * kT) return cudaErrorInvalidValue;
      return launch_cfg<256, 4, 2 * kT, EPI_STORE, 1>(a, st, num_sms);
#endif
    case EPI_F32:  // fp32 partial sums of a K split (decode-sized expert GEMMs)
      return launch_cfg<256, 4, kT, EPI_F32, 1>(a, st, num_sms);
    case EPI_DW:  // short-K tiles: the epilogue sets the pace, so eight epilogue warps (4 KB staging each)
      if (need > kT) return cudaErrorInvalidValue;
      return launch_cfg<256, 4, kT, EPI_DW, 1, 8>(a, st, num_sms);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace moe
