// route_noalloc.cu -- the routing stage of moe_fwd for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc or hand over a workspace: code that runs
// inside an allocator-less runtime (an inference engine whose memory pool is
// fixed up front, a plugin that must not touch the caller's allocator, a
// process that has to stay inside a pre-sized memory budget). For them this
// entry point computes exactly what moe_fwd reports about routing -- top-k
// experts and weights per token, per-expert offsets and the expert-contiguous
// row of every pair -- with all of its scratch memory in one file-scope
// device array of fixed size. Every GPU that loads the library keeps that
// array until the process exits.
#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include "common.cuh"
#include "gemm_launch.h"
#include "kernels.h"

namespace moe {
int internal_check_dims(const moe_dims* d);
int internal_fail(int code, const char* msg);
void internal_count_launches(int n);
}  // namespace moe

using namespace moe;

namespace {

// Largest scratch the routing stage may use: biased fp32 logits [T,E], the
// per-chunk expert masks and row bases, the per-expert counters and the
// padded pair/row maps. T*E <= 1,048,576 with k <= 8 fits (e.g. T=8192, E=128).
constexpr size_t kRouteScratchBytes = size_t(8) << 20;

static __device__ __align__(256) unsigned char g_route_scratch[kRouteScratchBytes];

size_t up256(size_t n) { return (n + 255) / 256 * 256; }

struct ScratchLayout {
  size_t status, logits, masks, chunk_base, count, offset, pad_off, tile_off, rowp, pair_of_row, total;
};

ScratchLayout scratch_layout(const moe_dims* d) {
  const size_t T = d->T, E = d->E, k = d->k, P = T * k, C = (T + 63) / 64, R = P + 15 * E;
  ScratchLayout L;
  size_t o = 0;
  L.status = o;      o += up256(sizeof(int));
  L.logits = o;      o += up256(T * E * sizeof(float));
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

// Device address of the scratch array on the current device, looked up once
// per device. The host-side name g_route_scratch is only a stand-in for the
// device symbol and must never be handed to a kernel.
int scratch_address(unsigned char** out) {
  static std::mutex mu;
  static std::unordered_map<int, unsigned char*> addr;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return internal_fail(MOE_ERR_CUDA, "cudaGetDevice failed");
  std::lock_guard<std::mutex> lk(mu);
  auto it = addr.find(dev);
  if (it != addr.end()) {
    *out = it->second;
    return MOE_OK;
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_route_scratch);
  if (e != cudaSuccess || p == nullptr) {
    char msg[160];
    snprintf(msg, sizeof(msg), "cudaGetSymbolAddress(route scratch) failed: %s", cudaGetErrorString(e));
    return internal_fail(MOE_ERR_CUDA, msg);
  }
  addr[dev] = static_cast<unsigned char*>(p);
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
  const ScratchLayout L = scratch_layout(dims);
  if (L.total > kRouteScratchBytes) {
    char msg[200];
    snprintf(msg, sizeof(msg),
             "moe_route_noalloc: these dims need %zu bytes of routing scratch, more than the fixed %zu bytes "
             "(keep T*E <= 1048576 with k <= 8, or use moe_fwd with a workspace)",
             L.total, kRouteScratchBytes);
    return internal_fail(MOE_ERR_UNSUPPORTED, msg);
  }
  unsigned char* base = nullptr;
  if ((rc = scratch_address(&base))) return rc;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int T = (int)dims->T, H = (int)dims->H, E = (int)dims->E, k = (int)dims->k;
  const int C = (T + 63) / 64;
  int* status = device_status ? device_status : reinterpret_cast<int*>(base + L.status);
  float* logits = reinterpret_cast<float*>(base + L.logits);
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
  // Only the status word must start at zero: every other scratch entry is
  // fully written by the kernel that produces it before anything reads it.
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
  e = dims->dtype == MOE_BF16 ? launch_tc_gemm(a, 128, st, sms_of_current_device(), 0) : launch_simt_gemm_f32(a, st);
  if (e != cudaSuccess) return cuda_fail(e, "router GEMM");
  if ((e = launch_route_topk(logits, router_bias, T, E, k, topk_idx, topk_w, masks, st)) != cudaSuccess)
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
