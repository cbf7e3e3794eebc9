// gemm_tc.cu -- persistent grouped GEMM on the 5th-generation tensor cores (sm_103a).
//
// Per CTA (192 threads, one CTA per SM):
//   warp 0      TMA producer: loads A/B k-blocks of 64 into a STAGES-deep
//               ring of 128-byte-swizzled shared-memory tiles.
//   warp 1      MMA issuer: tcgen05.mma (M=128, N=BN, K=16) into one of two
//               tensor-memory accumulators, commits free smem slots back.
//   warps 2..5  epilogue: tcgen05.ld of the finished accumulator (one row per
//               thread), fused epilogue (SwiGLU fwd/bwd, store, dW), global stores.
// Tiles (group, m-block, n-block) are read from device-side group offsets, so
// the host never learns the per-expert row counts. Every barrier wait is
// bounded; a wait that runs out sets MOE_ERR_TIMEOUT in the status word, the
// CTA drains its own copies and MMAs, frees its tensor memory and returns.
#include <cudaTypedefs.h>

#include <mutex>

#include "epilogue.cuh"
#include "gemm_launch.h"

namespace moe {

constexpr int kThreads = 192;

template <int BN>
struct TcCfg {
  static constexpr int STAGES = (BN == 256) ? 4 : 6;
  static constexpr int A_BYTES = kTileM * kTileK * 2;  // 16 KB
  static constexpr int B_BYTES = BN * kTileK * 2;      // 32 KB (BN=256) / 16 KB
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int BAR_OFF = STAGES * STAGE_BYTES;
  static constexpr int SMEM = BAR_OFF + 256 + 1024;  // barriers + 1 KB alignment slack
  static constexpr uint32_t TMEM_COLS = 2 * BN;      // two accumulators
};

struct TileInfo {
  int g, m0, nt, rows, off, kblocks;
};

template <int BN>
__device__ __forceinline__ int n_tiles(const GemmArgs& a) {
  const int w = a.paired ? BN / 2 : BN;
  return (a.N + w - 1) / w;
}

template <int BN>
__device__ __forceinline__ TileInfo decode_tile(const GemmArgs& a, int t, int NT) {
  TileInfo ti;
  if (a.var_k) {
    const int MT = (a.M + kTileM - 1) / kTileM;
    ti.g = t / (MT * NT);
    const int rem = t - ti.g * MT * NT;
    ti.m0 = (rem / NT) * kTileM;
    ti.nt = rem % NT;
    ti.rows = grp_rows(a, ti.g);
    ti.off = grp_off(a, ti.g);
    ti.kblocks = (ti.rows + kTileK - 1) / kTileK;
  } else {
    const int u = t / NT;
    ti.nt = t - u * NT;
    int g = 0;
    if (a.tile_off) {  // last g with tile_off[g] <= u
      int lo = 0, hi = a.G - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.tile_off[mid] <= u) lo = mid; else hi = mid - 1;
      }
      g = lo;
      ti.m0 = (u - a.tile_off[g]) * kTileM;
    } else {
      ti.m0 = u * kTileM;
    }
    ti.g = g;
    ti.rows = grp_rows(a, g);
    ti.off = grp_off(a, g);
    ti.kblocks = a.K / kTileK;
  }
  return ti;
}

template <int BN>
__device__ __forceinline__ int total_tiles(const GemmArgs& a) {
  const int NT = n_tiles<BN>(a);
  if (a.var_k) return a.G * ((a.M + kTileM - 1) / kTileM) * NT;
  const int mt = a.tile_off ? a.tile_off[a.G] : (a.rows_const + kTileM - 1) / kTileM;
  return mt * NT;
}

template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    tc_grouped_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                    const __grid_constant__ CUtensorMap tmB1, const GemmArgs args) {
  using C = TcCfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* empty = full + C::STAGES;
  uint64_t* tfull = empty + C::STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 128);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int NT = n_tiles<BN>(args);
  const int total = total_tiles<BN>(args);

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB0);
    tma_prefetch_desc(&tmB1);
    int stage = 0;
    uint32_t phase = 0;
    int issued_parity[C::STAGES];
#pragma unroll
    for (int s = 0; s < C::STAGES; ++s) issued_parity[s] = -1;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      const TileInfo ti = decode_tile<BN>(args, t, NT);
      for (int kb = 0; kb < ti.kblocks; ++kb) {
        if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        uint8_t* sa = smem + stage * C::STAGE_BYTES;
        uint8_t* sb = sa + C::A_BYTES;
        const uint32_t fb = smem_u32(&full[stage]);
        mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
        issued_parity[stage] = (int)phase;
        if (!args.var_k) {
          tma_load_2d(smem_u32(sa), &tmA, fb, kb * kTileK, ti.off + ti.m0);
        } else {
          tma_load_2d(smem_u32(sa), &tmA, fb, ti.m0, ti.off + kb * kTileK);
          tma_load_2d(smem_u32(sa + 8192), &tmA, fb, ti.m0 + 64, ti.off + kb * kTileK);
        }
        if (args.b_kmajor) {
          const bool second = args.k_split > 0 && kb * kTileK >= args.k_split;
          const int kk = second ? kb - args.k_split / kTileK : kb;
          tma_load_2d(smem_u32(sb), second ? &tmB1 : &tmB0, fb, kk * kTileK, ti.g * args.N + ti.nt * BN);
        } else {
          const int brow = args.var_k ? ti.off + kb * kTileK : ti.g * args.K + kb * kTileK;
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
            tma_load_2d(smem_u32(sb + c * 8192), map, fb, col, brow);
          }
        }
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    // make sure no copy of ours is still landing in shared memory
    for (int s = 0; s < C::STAGES; ++s)
      if (issued_parity[s] >= 0) mbar_wait_timed(&full[s], (uint32_t)issued_parity[s], 200000000ull);
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t idesc = idesc_bf16(kTileM, BN, args.var_k, args.b_kmajor ? 0 : 1);
    int stage = 0;
    uint32_t phase = 0;
    int acc_i = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      const TileInfo ti = decode_tile<BN>(args, t, NT);
      if (ti.kblocks == 0) continue;
      const int acc = acc_i & 1;
      const uint32_t acc_par = (uint32_t)((acc_i >> 1) & 1);
      if (!mbar_wait_bounded(&tempty[acc], acc_par ^ 1u, abort_flag)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
      for (int kb = 0; kb < ti.kblocks; ++kb) {
        if (!mbar_wait_bounded(&full[stage], phase, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sa = smem_u32(smem + stage * C::STAGE_BYTES);
        const uint32_t sb = sa + C::A_BYTES;
        int nk = kTileK / 16;
        if (args.var_k && kb == ti.kblocks - 1) nk = (ti.rows - kb * kTileK + 15) / 16;
        for (int kk = 0; kk < nk; ++kk) {
          const uint64_t ad = args.var_k ? sdesc_sw128(sa + kk * 2048, 8192, 1024) : sdesc_sw128(sa + kk * 32, 16, 1024);
          const uint64_t bd =
              args.b_kmajor ? sdesc_sw128(sb + kk * 32, 16, 1024) : sdesc_sw128(sb + kk * 2048, 8192, 1024);
          tc_mma_bf16(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
        }
        tc_commit(&empty[stage]);
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      tc_commit(&tfull[acc]);
      ++acc_i;
    }
    // wait until every MMA issued by this thread has completed
    tc_commit(drain);
    mbar_wait_timed(drain, 0, 200000000ull);
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int row = q * 32 + lane;
    int acc_i = 0;
    float v0[32], v1[32];
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const TileInfo ti = decode_tile<BN>(args, t, NT);
      const int m = ti.m0 + row;
      if (ti.kblocks == 0) {  // variable-K group with no rows: its output is zero
#pragma unroll
        for (int i = 0; i < 32; ++i) v0[i] = v1[i] = 0.0f;
        if (args.paired) {
          for (int c = 0; c < BN / 64; ++c)
            epilogue_apply<__nv_bfloat16, 32>(args, ti.g, ti.rows, m, ti.nt * (BN / 2) + c * 32, v0, v1);
        } else {
          for (int c = 0; c < BN / 32; ++c)
            epilogue_apply<__nv_bfloat16, 32>(args, ti.g, ti.rows, m, ti.nt * BN + c * 32, v0, nullptr);
        }
        continue;
      }
      const int acc = acc_i & 1;
      const uint32_t acc_par = (uint32_t)((acc_i >> 1) & 1);
      if (!mbar_wait_bounded(&tfull[acc], acc_par, abort_flag)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
      if (args.paired) {
        for (int c = 0; c < BN / 64; ++c) {
          tmem_ld32(taddr + c * 32, v0);
          tmem_ld32(taddr + BN / 2 + c * 32, v1);
          epilogue_apply<__nv_bfloat16, 32>(args, ti.g, ti.rows, m, ti.nt * (BN / 2) + c * 32, v0, v1);
        }
      } else {
        for (int c = 0; c < BN / 32; ++c) {
          tmem_ld32(taddr + c * 32, v0);
          epilogue_apply<__nv_bfloat16, 32>(args, ti.g, ti.rows, m, ti.nt * BN + c * 32, v0, nullptr);
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
      ++acc_i;
    }
  }

  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) set_status(args.status, MOE_ERR_TIMEOUT);
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
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

// 2-D bf16 view [rows, cols] (cols contiguous), box [box_rows, box_cols], 128-byte swizzle,
// out-of-bounds elements read as zero.
static bool make_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int box_cols, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int BN>
static cudaError_t launch_bn(const GemmArgs& a, cudaStream_t st, int num_sms, int max_tiles_hint) {
  using C = TcCfg<BN>;
  cudaError_t e = cudaFuncSetAttribute(tc_grouped_gemm<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  CUtensorMap mA, mB0, mB1;
  bool ok;
  if (!a.var_k)
    ok = make_map(&mA, a.A, a.a_rows, a.lda, 64, kTileM);
  else
    ok = make_map(&mA, a.A, a.a_rows, a.lda, 64, kTileK);
  if (a.b_kmajor) {
    ok = ok && make_map(&mB0, a.B0, a.b_rows, a.ldb, 64, BN);
    ok = ok && make_map(&mB1, a.B1 ? a.B1 : a.B0, a.b_rows, a.ldb, 64, BN);
  } else {
    ok = ok && make_map(&mB0, a.B0, a.b_rows, a.ldb, 64, kTileK);
    ok = ok && make_map(&mB1, a.B1 ? a.B1 : a.B0, a.b_rows, a.ldb, 64, kTileK);
  }
  if (!ok) return cudaErrorInvalidValue;
  int grid = num_sms;
  if (max_tiles_hint > 0 && max_tiles_hint < grid) grid = max_tiles_hint;
  if (grid < 1) grid = 1;
  tc_grouped_gemm<BN><<<grid, kThreads, C::SMEM, st>>>(mA, mB0, mB1, a);
  return cudaGetLastError();
}

cudaError_t launch_tc_gemm(const GemmArgs& a, int bn, cudaStream_t st, int num_sms, int max_tiles_hint) {
  if (bn == 256) return launch_bn<256>(a, st, num_sms, max_tiles_hint);
  return launch_bn<128>(a, st, num_sms, max_tiles_hint);
}

}  // namespace moe
