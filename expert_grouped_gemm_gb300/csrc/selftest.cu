// selftest.cu -- exercises the bounded mbarrier wait that every pipelined
// kernel of the library relies on, without faulting or hanging the GPU.
//
// One thread initialises an mbarrier that expects one arrival. With arrive = 1
// it arrives first and the wait returns at once; with arrive = 0 nothing ever
// arrives, the wait gives up after limit_ns and the kernel records
// MOE_ERR_TIMEOUT -- the same path a GEMM CTA takes when a producer or the
// MMA issuer stops making progress. The kernel then returns normally, so the
// context stays usable.
#include <cuda_runtime.h>

#include "common.cuh"

namespace moe {
int internal_fail(int code, const char* msg);
void internal_count_launches(int n);
}  // namespace moe

using namespace moe;

namespace {

__global__ void k_wait_probe(int arrive_first, unsigned long long limit_ns, int* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (arrive_first) mbar_arrive(&bar);
    const bool ok = mbar_wait_bounded(&bar, 0, &abort_flag, limit_ns);
    *status = ok ? MOE_OK : MOE_ERR_TIMEOUT;
  }
}

}  // namespace

extern "C" MOE_API int moe_selftest_wait(void* stream, int arrive, int64_t limit_us, int32_t* device_status) {
  if (!device_status) return internal_fail(MOE_ERR_INVALID_ARG, "moe_selftest_wait: device_status is null");
  if (limit_us < 1 || limit_us > 1000000)
    return internal_fail(MOE_ERR_INVALID_ARG, "moe_selftest_wait: limit_us must be in [1, 1000000]");
  k_wait_probe<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(arrive ? 1 : 0,
                                                               (unsigned long long)limit_us * 1000ull, device_status);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return internal_fail(MOE_ERR_CUDA, cudaGetErrorString(e));
  internal_count_launches(1);
  return MOE_OK;
}
