// decode.h -- host side of the fused decode forward (decode.cu).
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace moe {

// dims the fused kernel handles: 1 <= T <= 16, E <= 256, k <= 16, H, F, Fs <= 4096 (multiples of 64)
bool decode_supported(int64_t T, int64_t H, int64_t F, int64_t E, int64_t k, int64_t Fs);
// bytes of device scratch it needs (logits, h, per-slot y, gate/up partial sums per 256-row
// chunk of H, a barrier counter)
size_t decode_scratch_bytes(int64_t T, int64_t H, int64_t F, int64_t E, int64_t k, int64_t Fs);
// one cooperative launch of num_sms CTAs on st; sync is the grid-barrier counter, zeroed by
// the caller on st before the launch. Self-test only: stall (1..4) makes that grid barrier
// need one arrival more than the grid has, and wait_ns bounds every wait.
cudaError_t launch_decode_fwd(int T, int H, int F, int E, int k, int Fs, const void* x, const void* w_router,
                              const float* bias, const void* w_gate, const void* w_up, const void* w_down,
                              const void* ws_gate, const void* ws_up, const void* ws_down, void* y, int* topk_idx,
                              float* topk_w, int* user_idx, float* user_w, float* user_logits, void* scratch,
                              int* status, unsigned* sync, int num_sms, cudaStream_t st, unsigned stall = 0,
                              uint64_t wait_ns = 1000000000ull);

}  // namespace moe
