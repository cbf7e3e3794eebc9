// route_noalloc.cu -- the routing stage of moe_fwd for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc or hand over a workspace: code that runs
// inside an allocator-less runtime (an inference engine whose memory pool is
// fixed up front, a plugin that must not touch the caller's allocator, a
// process that has to stay inside a pre-sized memory budget). For them this
// entry point computes what moe_fwd reports about routing -- top-k experts and
// weights per token, per-expert offsets and the expert-contiguous row of every
// pair -- with all of its scratch memory in one file-scope device array of
// fixed size. Every GPU that loads the library keeps that array until the
// process exits.
//
// The router GEMM runs with the K split moe_fwd picks for the same dims (its
// fp32 partials live in the scratch, split 0 doubling as the logits buffer),
// so the results are bit-identical to moe_fwd's whenever that split fits; a
// smaller split is used otherwise, which changes only the fp32 summation
// order of the logits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "common.cuh"
#include "gemm_launch.h"
#include "kernels.h"

namespace moe {
int internal_check_dims(const moe_dims* d);
int internal_fail(int code, const char* msg);
void internal_count_launches(int n);
int internal_router_ksplit(const moe_dims* d, int sms);
}  // namespace moe

using namespace moe;

namespace {

// Size of the fixed scratch. What the routing stage keeps there, in bytes (each
// entry rounded up to 256): a status word; the router logits, 4*ks*T*E (ks = the
// router GEMM's K split, 1 without one); the per-64-token expert masks and row bases,
// 12*ceil(T/64)*E; per-expert counts and offsets, about 16*E; the padded row of
// every pair, 4*T*k; the pair of every padded row, 4*(T*k + 15*E). With ks = 1 the
// total is about 4*T*E + 12*ceil(T/64)*E + 8*T*k + 76*E bytes.
constexpr size_t kRouteScratchBytes = size_t(32) << 20;

static __device__ __align__(256) unsigned char g_route_scratch[kRouteScratchBytes];

size_t up256(size_t n) { return (n + 255) / 256 * 256; }

struct ScratchLayout {
  size_t status, logits, masks, chunk_base, count, offset, pad_off, tile_off, rowp, pair_of_row, total;
};

ScratchLayout scratch_layout(const moe_dims* d, int ks) {
  const size_t T = d->T, E = d->E, k = d->k, P = T * k, C = (T + 63) / 64, R = P + 15 * E;
  ScratchLayout L;
  size_t o = 0;
  L.status = o;      o += up256(sizeof(int));
  L.logits = o;      o += up256((size_t)ks * T * E * sizeof(float));
  L.masks = o;       o += up256(C * E * sizeof(uint64_t));
  L.chunk_base = o;  o += up256(C * E * sizeof(int));
  L.count = o;       o += up256(E * sizeof(int));
  L.offset = o;      o += up256((E + 1) * sizeof(int));
  L.pad_off = o;     o += up256((E + 1) * sizeof(int));
  L.tile_off = o;    o += up256((E + 1) * sizeof(int));
  L.rowp = o;        o += up256(P * sizeof(int));
  L.pair_of_row = o; o += up256(R * sizeof(int));
  L.total = o;
  return L;
}

// Device address of the scratch array in the current CUDA context. The lookup is
// done once per (device, context) and kept: a context that was torn down and made
// again (after cudaDeviceReset, for example) gets a fresh lookup, so a stale address
// is never used. The host-side name g_route_scratch is only a stand-in for the
// device symbol and must never be handed to a kernel.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);

CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}

int scratch_address(unsigned char** out) {
  static std::mutex mu;
  static std::map<std::pair<int, uintptr_t>, unsigned char*> addr;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return internal_fail(MOE_ERR_CUDA, "cudaGetDevice failed");
  CtxGetCurrentFn get_ctx = ctx_get_current();
  CUcontext ctx = nullptr;
  if (get_ctx) get_ctx(&ctx);
  std::lock_guard<std::mutex> lk(mu);
  if (ctx) {
    auto it = addr.find({dev, reinterpret_cast<uintptr_t>(ctx)});
    if (it != addr.end()) {
      *out = it->second;
      return MOE_OK;
    }
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_route_scratch);
  if (e != cudaSuccess || p == nullptr) {
    char msg[160];
    snprintf(msg, sizeof(msg), "cudaGetSymbolAddress(route scratch) failed: %s", cudaGetErrorString(e));
    return internal_fail(MOE_ERR_CUDA, msg);
  }
  // the lookup made the runtime's context current if it was not yet
  if (get_ctx && (ctx != nullptr || get_ctx(&ctx) == CUDA_SUCCESS) && ctx)
    addr[{dev, reinterpret_cast<uintptr_t>(ctx)}] = static_cast<unsigned char*>(p);
  *out = static_cast<unsigned char*>(p);
  return MOE_OK;
}

int sms_of_current_device() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  return n;
}

bool aligned(const void* p, int a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" MOE_API int moe_route_noalloc(const moe_dims* dims, void* stream, const void* x, const void* w_router,
                                         const float* router_bias, int32_t* topk_idx, float* topk_w,
                                         int32_t* expert_offsets, int32_t* row_of_pair, int32_t* device_status) {
  int rc = internal_check_dims(dims);
  if (rc) return rc;
  if (!x || !w_router || !topk_idx || !topk_w || !expert_offsets || !row_of_pair)
    return internal_fail(MOE_ERR_INVALID_ARG, "moe_route_noalloc: x, w_router and all four outputs are required");
  if (!aligned(x, 16) || !aligned(w_router, 16) || !aligned(router_bias, 4) || !aligned(topk_idx, 4) ||
      !aligned(topk_w, 4) || !aligned(expert_offsets, 4) || !aligned(row_of_pair, 4) || !aligned(device_status, 4))
    return internal_fail(MOE_ERR_INVALID_ARG, "moe_route_noalloc: misaligned pointer");
  const ScratchLayout L1 = scratch_layout(dims, 1);
  if (L1.total > kRouteScratchBytes) {
    char msg[240];
    snprintf(msg, sizeof(msg),
             "moe_route_noalloc: these dims need %zu bytes of routing scratch, more than the fixed %zu bytes "
             "(about 4*T*E + 12*ceil(T/64)*E + 8*T*k + 76*E bytes must fit; use moe_fwd with a workspace)",
             L1.total, kRouteScratchBytes);
    return internal_fail(MOE_ERR_UNSUPPORTED, msg);
  }
  unsigned char* base = nullptr;
  if ((rc = scratch_address(&base))) return rc;

  const int sms = sms_of_current_device();
  const int T = (int)dims->T, H = (int)dims->H, E = (int)dims->E, k = (int)dims->k;
  const int C = (T + 63) / 64;
  // moe_fwd's K split of the router GEMM; fewer splits if their partials do not fit
  int ks = internal_router_ksplit(dims, sms);
  while (ks > 1 && scratch_layout(dims, ks).total > kRouteScratchBytes) --ks;
  if (ks > 1) {  // the same normalisation moe_fwd applies: no split without k-blocks
    const int kblocks = H / 64;
    const int per = (kblocks + ks - 1) / ks;
    ks = (kblocks + per - 1) / per;
  }
  const ScratchLayout L = scratch_layout(dims, ks);

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int* status = device_status ? device_status : reinterpret_cast<int*>(base + L.status);
  float* logits = reinterpret_cast<float*>(base + L.logits);  // split s at logits + s*T*E
  uint64_t* masks = reinterpret_cast<uint64_t*>(base + L.masks);
  int* chunk_base = reinterpret_cast<int*>(base + L.chunk_base);
  int* count = reinterpret_cast<int*>(base + L.count);
  int* offset = reinterpret_cast<int*>(base + L.offset);
  int* pad_off = reinterpret_cast<int*>(base + L.pad_off);
  int* tile_off = reinterpret_cast<int*>(base + L.tile_off);
  int* rowp = reinterpret_cast<int*>(base + L.rowp);
  int* pair_of_row = reinterpret_cast<int*>(base + L.pair_of_row);

  auto cuda_fail = [](cudaError_t e, const char* what) {
    char msg[200];
    snprintf(msg, sizeof(msg), "moe_route_noalloc: %s: %s", what, cudaGetErrorString(e));
    return internal_fail(MOE_ERR_CUDA, msg);
  };
  // Only the status word must start at zero (the expert masks are cleared by the
  // top-k launcher): every other scratch entry is fully written by the kernel that
  // produces it before anything reads it, so what an earlier call left there is
  // never read.
  cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int), st);
  if (e != cudaSuccess) return cuda_fail(e, "clearing the status word");

  GemmArgs a;
  memset(&a, 0, sizeof(a));
  a.status = status;
  a.var_k = 0;
  a.G = 1;
  a.rows_const = T;
  a.K = H;
  a.N = E;
  a.A = x;
  a.lda = H;
  a.a_rows = T;
  a.B0 = w_router;
  a.ldb = E;
  a.b_rows = H;
  a.epi = EPI_F32;
  a.out0 = logits;
  a.ldo = E;
  if (ks > 1) {  // every split writes its fp32 partial sums; the top-k kernel adds them in split order
    a.ksplit = ks;
    a.part_stride = (int64_t)T * E;
  }
  e = dims->dtype == MOE_BF16 ? launch_tc_gemm(a, 128, st, sms, 0) : launch_simt_gemm_f32(a, st);
  if (e != cudaSuccess) return cuda_fail(e, "router GEMM");
  // with a split, the top-k kernel reads every split of a token's row before it writes
  // the biased logits over split 0 of that row (same thread, same elements)
  if ((e = launch_route_topk(logits, router_bias, T, E, k, topk_idx, topk_w, masks, st, ks > 1 ? logits : nullptr, ks,
                             (int64_t)T * E)) != cudaSuccess)
    return cuda_fail(e, "top-k");
  if ((e = launch_route_scan(masks, C, E, count, offset, pad_off, tile_off, chunk_base, pair_of_row, expert_offsets,
                             st)) != cudaSuccess)
    return cuda_fail(e, "expert scan");
  if ((e = launch_route_index(masks, chunk_base, topk_idx, offset, pad_off, T, E, k, rowp, row_of_pair, pair_of_row,
                              st)) != cudaSuccess)
    return cuda_fail(e, "pair rows");
  internal_count_launches(4);
  return MOE_OK;
}
