// gemm_ws.cu -- weight-stationary grouped GEMM on CTA pairs (sm_103a), store epilogue.
//
// out[off_g + r, n] = sum_k act[off_g + r, k] W_g(k, n) for the rows r of group g: the
// variable-M store GEMMs (expert down, dX of the pairs). The product is formed
// transposed, D[n, r] = sum_k W_g(k, n) act[off_g + r, k]: a CTA pair (cta_group::2)
// puts 256 output columns on the MMA's M dimension, 128 per CTA, and a chunk of up to
// 256 of the group's rows on N, each CTA loading half of the chunk. A group is padded
// to 16 rows (the permuted layout; the MMA's N is that rounded up to 32) instead of to
// 128-row tiles, and a k-block costs each CTA 16 KB of weights and at most 16 KB of
// rows, so six stages fit in shared memory.
//
// Per CTA (192 threads, one CTA per SM, clusters of two):
//   warp 0      TMA producer (both CTAs; the leader's full barrier counts both CTAs' bytes)
//   warp 1      MMA issuer (leader only): tcgen05.mma.cta_group::2, M = 256, N = chunk rows
//   warps 2..5  epilogue: tcgen05.ld gives a thread one output column for 32 rows; 64
//               rows at a time go out transposed through a staging tile and a TMA store
// Every barrier wait is bounded as in the other tensor-core GEMM: a wait that runs out
// sets MOE_ERR_TIMEOUT, the CTA lets its own copies and MMAs finish, frees its tensor
// memory and returns.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "gemm_launch.h"

namespace moe {

namespace {

constexpr int kWsStages = 6;
constexpr int kWsABytes = 128 * kTileK * 2;  // 16 KB: this CTA's 128 output columns of W
constexpr int kWsBBytes = 128 * kTileK * 2;  // 16 KB: at most 128 rows, this CTA's half of a chunk
constexpr int kWsStageBytes = kWsABytes + kWsBBytes;
constexpr int kWsTileBytes = 64 * 32 * 2;    // one 64-row x 32-column bf16 staging tile
constexpr int kWsEpiOff = kWsStages * kWsStageBytes;
constexpr int kWsBarOff = kWsEpiOff + 4 * 2 * kWsTileBytes;  // two staging tiles per epilogue warp
constexpr int kWsSmem = kWsBarOff + 256 + 1024;               // barriers + 1 KB alignment slack
constexpr int kWsThreads = 192;
constexpr uint32_t kWsTmemCols = 512;  // two accumulators of up to 256 columns (rows of the chunk)
constexpr int kWsChunk = 256;          // rows of a chunk (one tile_rec2 record)
static_assert(kWsSmem <= 232448, "shared memory budget");

struct WsMaps {
  CUtensorMap w0, w1;  // weights: 128 output columns x 64 k of this CTA (w1: the second K half)
  CUtensorMap t[4];    // rows of act: 64 k x 128 / 64 / 32 / 16 rows
  CUtensorMap o64, o32, o16;  // out: 32 columns x 64 / 32 / 16 rows, no swizzle
};

struct WsTile {
  int g, m0, nrows, off, nt, n_mma;  // nrows: rows to store (16-padded); n_mma: MMA N (32-padded)
};

__device__ __forceinline__ WsTile ws_tile(const GemmArgs& a, int t, int NT, int4 rec) {
  WsTile w;
  w.nt = t % NT;
  w.g = rec.x;
  w.m0 = rec.y;
  w.off = rec.w;
  const int padded = (rec.z + kPadRows - 1) / kPadRows * kPadRows;
  w.nrows = min(kWsChunk, padded - w.m0);
  w.n_mma = (w.nrows + 31) / 32 * 32;
  return w;
}

__device__ __forceinline__ int4 ws_rec(const GemmArgs& a, int t, int NT) { return __ldg(a.tile_rec2 + t / NT); }

__device__ __forceinline__ void st_shared_b16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.b16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

__global__ void __launch_bounds__(kWsThreads, 1) ws_store_gemm(const __grid_constant__ WsMaps maps, const GemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kWsBarOff);
  uint64_t* empty = full + kWsStages;
  uint64_t* tfull = empty + kWsStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int cluster_id = (int)(blockIdx.x >> 1);
  const int num_clusters = (int)(gridDim.x >> 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kWsStages; ++s) {
      mbar_init(&full[s], 1);   // the leader's producer arms it for both CTAs' bytes
      mbar_init(&empty[s], 1);  // one MMA commit, multicast to both CTAs
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 4 * 2);  // one arrive per epilogue warp of each CTA
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) tmem_alloc_pair(tmem_slot, kWsTmemCols);
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers exist before any remote arrive
  tc_fence_after();
  pdl_wait();  // the set-up above touched no global memory
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t full0 = mapa_shared(smem_u32(full), 0);     // the leader's full barriers
  const uint32_t tempty0 = mapa_shared(smem_u32(tempty), 0);  // the leader's accumulator-free barriers

  const int NT = (args.N + 2 * 128 - 1) / (2 * 128);
  const int total = args.tile_off2[args.G] * NT;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    tma_prefetch_desc(&maps.w0);
    tma_prefetch_desc(&maps.w1);
    int stage = 0;
    uint32_t phase = 0;
    int issued_parity[kWsStages];
#pragma unroll
    for (int s = 0; s < kWsStages; ++s) issued_parity[s] = -1;
    bool ok = true;
    int4 rec = cluster_id < total ? ws_rec(args, cluster_id, NT) : make_int4(0, 0, 0, 0);
    for (int t = cluster_id; t < total && ok; t += num_clusters) {
      const WsTile w = ws_tile(args, t, NT, rec);
      if (t + num_clusters < total) rec = ws_rec(args, t + num_clusters, NT);
      const int h = w.n_mma / 2;                          // rows of this CTA's half (multiple of 16)
      const int r0 = w.off + w.m0 + (int)rank * h;        // first row of this CTA's half
      const int c0 = w.nt * 256 + (int)rank * 128;        // first output column of this CTA
      for (int kb = 0; kb < args.K / kTileK; ++kb) {
        if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        const uint32_t sa = smem_u32(smem + stage * kWsStageBytes);
        const uint32_t sb = sa + kWsABytes;
        const uint32_t fb = full0 + stage * 8;
        if (leader) mbar_arrive_expect_tx(&full[stage], 2u * (uint32_t)(kWsABytes + h * 128));
        issued_parity[stage] = (int)phase;
        // weights: this CTA's 128 output columns for k-block kb
        if (args.b_kmajor) {
          const bool second = args.k_split > 0 && kb * kTileK >= args.k_split;
          const int kk = second ? kb - args.k_split / kTileK : kb;
          tma_load_2d_pair(sa, second ? &maps.w1 : &maps.w0, fb, kk * kTileK, w.g * args.N + c0);
        } else {
          tma_load_3d_pair(sa, &maps.w0, fb, 0, w.g * args.K + kb * kTileK, c0 / 64);
        }
        // rows: h = 128 / 64 / 32 / 16-row boxes, packed from the top of the B tile
        int done = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int sz = 128 >> i;
          if (h - done >= sz) {
            tma_load_2d_pair(sb + (uint32_t)(done * 128), &maps.t[i], fb, kb * kTileK, r0 + done);
            done += sz;
          }
        }
        if (++stage == kWsStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    // no copy of ours may still be landing when the CTA leaves (the leader's full
    // barriers also count the peer's bytes)
    if (leader)
      for (int s = 0; s < kWsStages; ++s)
        if (issued_parity[s] >= 0) mbar_wait_timed(&full[s], (uint32_t)issued_parity[s], 200000000ull);
  } else if (warp == 1 && lane == 0 && leader) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t sa0 = smem_u32(smem);
    // A (weights): K-major rows of W (dX) or an MN-major [K, N] block in 64-column chunks (down)
    const uint64_t adesc0 = args.b_kmajor ? sdesc_sw128(sa0, 16, 1024) : sdesc_sw128(sa0, 8192, 1024);
    const uint64_t astep = args.b_kmajor ? 32 >> 4 : 2048 >> 4;
    const uint64_t bdesc0 = sdesc_sw128(sa0 + kWsABytes, 16, 1024);  // B (rows): K-major
    const uint64_t bstep = 32 >> 4;
    int stage = 0;
    uint32_t phase = 0;
    int acc_i = 0;
    bool ok = true;
    int4 rec = cluster_id < total ? ws_rec(args, cluster_id, NT) : make_int4(0, 0, 0, 0);
    for (int t = cluster_id; t < total && ok; t += num_clusters) {
      const WsTile w = ws_tile(args, t, NT, rec);
      if (t + num_clusters < total) rec = ws_rec(args, t + num_clusters, NT);
      const uint32_t idesc = idesc_bf16(256, w.n_mma, args.b_kmajor ? 0 : 1, 0);
      const int acc = acc_i & 1;
      const uint32_t acc_par = (uint32_t)((acc_i >> 1) & 1);
      if (!mbar_wait_bounded_cluster(&tempty[acc], acc_par ^ 1u, abort_flag)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + (uint32_t)(acc * 256);
      for (int kb = 0; kb < args.K / kTileK; ++kb) {
        if (!mbar_wait_bounded(&full[stage], phase, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t ad = adesc0 + (uint64_t)(stage * (kWsStageBytes >> 4));
        const uint64_t bd = bdesc0 + (uint64_t)(stage * (kWsStageBytes >> 4));
        tc_mma_bf16_pair(d_tmem, ad, bd, idesc, kb != 0 ? 1u : 0u);
        tc_mma_bf16_pair(d_tmem, ad + astep, bd + bstep, idesc, 1u);
        tc_mma_bf16_pair(d_tmem, ad + 2 * astep, bd + 2 * bstep, idesc, 1u);
        tc_mma_bf16_pair(d_tmem, ad + 3 * astep, bd + 3 * bstep, idesc, 1u);
        tc_commit_pair_mc(&empty[stage]);
        if (++stage == kWsStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      tc_commit_pair_mc(&tfull[acc]);
      ++acc_i;
    }
    tc_commit_pair(drain);  // wait until every MMA issued by this thread has completed
    mbar_wait_timed(drain, 0, 200000000ull);
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may read: output columns 32q..32q+31
    const uint32_t wst = smem_u32(smem + kWsEpiOff + (warp - 2) * 2 * kWsTileBytes);
    int acc_i = 0;
    int sc = 0;  // staging tiles used so far by this warp
    int4 rec = cluster_id < total ? ws_rec(args, cluster_id, NT) : make_int4(0, 0, 0, 0);
    for (int t = cluster_id; t < total; t += num_clusters) {
      const WsTile w = ws_tile(args, t, NT, rec);
      if (t + num_clusters < total) rec = ws_rec(args, t + num_clusters, NT);
      const int acc = acc_i & 1;
      const uint32_t acc_par = (uint32_t)((acc_i >> 1) & 1);
      if (!mbar_wait_bounded(&tfull[acc], acc_par, abort_flag)) break;
      tc_fence_after();
      const int col0 = w.nt * 256 + (int)rank * 128 + q * 32;  // this warp's 32 output columns
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * 256);
      for (int j = 0; j * 64 < w.nrows; ++j) {  // 64 rows of the chunk at a time
        const int rows_here = min(64, w.nrows - j * 64);  // 16, 32, 48 or 64
        uint32_t r0[32], r1[32];
        tmem_ld32_async(taddr + (uint32_t)(j * 64), r0);
        if (rows_here > 32) tmem_ld32_async(taddr + (uint32_t)(j * 64 + 32), r1);
        const uint32_t set = wst + (uint32_t)((sc & 1) * kWsTileBytes);
        if (lane == 0) bulk_wait_read_but1();  // the store that last used this tile has read it
        __syncwarp();
        tmem_ld_wait(r0);
        if (rows_here > 32) tmem_ld_order(r1);
        // thread `lane` holds column col0 + lane of the chunk's rows: row i goes to
        // staging row i, column lane (64-byte rows, the layout of the output box)
#pragma unroll
        for (int i = 0; i < 32; ++i)
          st_shared_b16(set + (uint32_t)(i * 64 + lane * 2),
                        __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(r0[i]))));
        if (rows_here > 32) {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            st_shared_b16(set + (uint32_t)((32 + i) * 64 + lane * 2),
                          __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(r1[i]))));
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          const int row = w.off + w.m0 + j * 64;
          if (rows_here == 64) {
            tma_store_2d(&maps.o64, set, col0, row);
          } else if (rows_here >= 32) {
            tma_store_2d(&maps.o32, set, col0, row);
            if (rows_here == 48) tma_store_2d(&maps.o16, set + 32 * 64, col0, row + 32);
          } else {
            tma_store_2d(&maps.o16, set, col0, row);
          }
          bulk_commit();
        }
        ++sc;
      }
      // this warp is done with the accumulator: tell the MMA issuer
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty0 + acc * 8);
      ++acc_i;
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // no CTA of the pair leaves while the other still uses it
  tc_fence_after();
  if (threadIdx.x == 0 && *abort_flag) set_status(args.status, MOE_ERR_TIMEOUT);
  if (warp == 2) tmem_dealloc_pair(tmem_base, kWsTmemCols);
}

// ---------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 ws_encode_fn() {
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

// 2-D bf16 view [rows, cols] (cols contiguous), box [box_rows, box_cols].
bool ws_map_2d(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int box_cols, int box_rows,
               CUtensorMapSwizzle swz) {
  auto fn = ws_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D view (64 columns, row, 64-column chunk) of a row-major [rows, cols] bf16 matrix;
// a box (64, box_rows, box_chunks) lands as box_chunks consecutive [box_rows][64] tiles.
bool ws_map_mn3d(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int box_rows, int box_chunks) {
  auto fn = ws_encode_fn();
  if (!fn || cols % 64) return false;
  cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)(cols / 64)};
  cuuint64_t strides[2] = {(cuuint64_t)cols * 2, 128};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, (cuuint32_t)box_chunks};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool ws_store_supported(const GemmArgs& a) {
  return !a.var_k && a.epi == EPI_STORE && a.tile_rec2 && a.tile_off2 && a.ksplit <= 1 && !a.paired &&
         a.K % kTileK == 0 && (a.b_kmajor ? (a.k_split % kTileK == 0) : (a.N % 64 == 0)) && a.ldo == a.N;
}

cudaError_t launch_ws_store(const GemmArgs& a, cudaStream_t st, int num_sms) {
  if (!ws_store_supported(a)) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(ws_store_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize, kWsSmem);
  if (e != cudaSuccess) return e;
  WsMaps maps;
  bool ok;
  const void* b1 = a.B1 ? a.B1 : a.B0;
  if (a.b_kmajor) {  // W_g rows (g*N + n), k contiguous: 128 rows x 64 k
    ok = ws_map_2d(&maps.w0, a.B0, a.b_rows, a.ldb, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) &&
         ws_map_2d(&maps.w1, b1, a.b_rows, a.ldb, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B);
  } else {  // W_g rows (g*K + k), n contiguous: 64 k x two 64-column chunks
    ok = ws_map_mn3d(&maps.w0, a.B0, a.b_rows, a.ldb, kTileK, 2);
    maps.w1 = maps.w0;
  }
  for (int i = 0; i < 4 && ok; ++i) ok = ws_map_2d(&maps.t[i], a.A, a.a_rows, a.lda, 64, 128 >> i, CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && ws_map_2d(&maps.o64, a.out0, a.out_rows, a.ldo, 32, 64, CU_TENSOR_MAP_SWIZZLE_NONE) &&
       ws_map_2d(&maps.o32, a.out0, a.out_rows, a.ldo, 32, 32, CU_TENSOR_MAP_SWIZZLE_NONE) &&
       ws_map_2d(&maps.o16, a.out0, a.out_rows, a.ldo, 32, 16, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (!ok) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kWsThreads);
  cfg.dynamicSmemBytes = kWsSmem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(2 * (num_sms / 2));
  // as many CTA pairs as can be resident at once (persistent schedule)
  int max_clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&max_clusters, ws_store_gemm, &cfg) == cudaSuccess && max_clusters > 0 &&
      2 * max_clusters < (int)cfg.gridDim.x)
    cfg.gridDim = dim3(2 * max_clusters);
  e = cudaLaunchKernelEx(&cfg, ws_store_gemm, maps, a);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace moe
