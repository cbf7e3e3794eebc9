/*
 * moe.h -- C ABI of the GB300 MoE expert-block library (libmoe_gb300.so).
 *
 * One MoE layer on one GPU: router -> top-k -> permute -> grouped SwiGLU
 * expert MLP -> weighted combine (moe_fwd); per-pair scores and optional
 * per-expert quota selection with physical compaction (moe_select_retained);
 * dX, dW_expert and dW_router with the same grouped GEMMs (moe_bwd).
 *
 * Sources of the operations (three web pages on one subject):
 *   [I14]   issue "[MoE] Hot experts on RNGD during training (host dispatch,
 *           device expert graphs) #14", sections Proposal and Scope.
 *   [PR44]  pull request "PR #44" (HostMLP(keep_graph=True)), section Changes.
 *   [LRMoE] "LRMoE: Demand-Side Load Re-Calibration for Efficient MoE Training
 *           on Memory-Constrained Nodes" (arXiv 2610.37720), Abstract.
 *
 * Conventions that hold for every call:
 *   - All tensor arguments are DEVICE pointers to row-major, contiguous
 *     buffers owned by the caller. The library allocates and frees no device
 *     memory; the caller passes a workspace of moe_workspace_size() bytes
 *     (256-byte aligned) that carries the state saved by moe_fwd for
 *     moe_select_retained and moe_bwd.
 *   - Element type of x, weights, y, dy, dx and every dW is dims.dtype
 *     (MOE_BF16 or MOE_F32); router_bias, top-k weights, logits and scores are
 *     float32; indices, offsets and quotas are int32. Accumulation is fp32.
 *   - stream is a cudaStream_t passed as void*. Every call only enqueues work
 *     and never synchronises the host (moe_read_status excepted). moe_bwd runs
 *     its router-gradient and dX-reduce kernels on a stream the library keeps
 *     for the workspace, forked from `stream` and joined back into it with
 *     events, so all of a call's work comes after earlier work on `stream` and
 *     before later work on it, and a fwd / select / bwd sequence can be
 *     captured in a CUDA graph (make a workspace's first moe_bwd call outside
 *     a capture: it creates that stream). The stream and its two events live as
 *     long as the process.
 *   - Return values: MOE_OK or a negative moe_status. Arguments are validated
 *     on the host before anything is enqueued; on error nothing is enqueued
 *     and moe_last_error() describes the failure. Errors found by the GPU
 *     (a bounded wait that ran out, a negative quota) are written to a status
 *     word in the workspace and reported by moe_read_status().
 *   - Calls on one workspace must be serialised by the caller (same stream or
 *     explicit events). Different workspaces are independent.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1,  /* bad dims, null required pointer, misaligned buffer */
  MOE_ERR_UNSUPPORTED = -2,  /* valid but not supported by this library (e.g. H % 64 != 0 in bf16) */
  MOE_ERR_CUDA = -3,         /* a CUDA runtime/driver call failed */
  MOE_ERR_WORKSPACE = -4,    /* workspace null, too small or misaligned */
  MOE_ERR_STATE = -5,        /* call order violated (bwd before fwd, x differs from fwd's x, ...) */
  MOE_ERR_TIMEOUT = -6,      /* device: a bounded wait inside a kernel ran out */
  MOE_ERR_DEVICE_ARG = -7    /* device: an argument read on the GPU was invalid (negative quota) */
} moe_status;

typedef enum { MOE_BF16 = 0, MOE_F32 = 1 } moe_dtype;

/* dims.flags */
#define MOE_FROZEN 1u   /* experts and router frozen ([I14] Scope: LoRA first): no dW of any
                           expert, router or shared expert is computed; dX stays complete */
#define MOE_RECOMPUTE 2u /* [PR44] keep_graph=False: the backward (or the retention select)
                           re-derives a|b, h and y_pair from the saved permuted rows instead
                           of using the forward's; results are bitwise the same */

typedef struct moe_dims {
  int64_t T;         /* tokens */
  int64_t H;         /* hidden size */
  int64_t F;         /* routed expert intermediate size */
  int64_t E;         /* routed experts */
  int64_t k;         /* experts per token, 1 <= k <= E <= 1024 */
  int64_t F_shared;  /* always-on shared expert intermediate size; 0 = none */
  int32_t dtype;     /* moe_dtype */
  uint32_t flags;    /* MOE_FROZEN | MOE_RECOMPUTE */
} moe_dims;

/*
 * moe_workspace_size -- bytes of device workspace needed for these dims.
 * Host-only (no CUDA call). Validates dims: T,H,F,E,k >= 1, k <= E <= 1024,
 * F_shared >= 0; bf16 additionally needs H % 64 == 0, F % 64 == 0,
 * F_shared % 64 == 0 and E % 16 == 0 (tensor-core tiles and 16-byte TMA
 * rows). Returns MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED otherwise.
 */
MOE_API int moe_workspace_size(const moe_dims* dims, size_t* bytes);

/*
 * moe_fwd -- forward of the MoE layer ([I14] Proposal: routing, dispatch of
 * rows to experts, expert forward, results scattered back).
 *   logits[t,e] = x[t,:] . w_router[:,e] + router_bias[e]   (fp32)
 *   top-k of logits per token, ties to the lower expert index, slot order
 *   by logit descending; topk_w = softmax over all E renormalised over the k
 *   selected experts.
 *   Pairs (t,j) are placed expert-contiguously, token order inside an expert.
 *   For each pair: a = x_t W_gate[e], b = x_t W_up[e], h = silu(a)*b,
 *   y_pair = h W_down[e]; y[t] = sum_j topk_w[t,j] y_pair(t,j)
 *   + shared expert silu(x ws_gate)*(x ws_up) ws_down when F_shared > 0.
 * Inputs:  x[T,H], w_router[H,E], router_bias[E] (float, nullable = zero),
 *          w_gate[E,H,F], w_up[E,H,F], w_down[E,F,H],
 *          ws_gate[H,Fs], ws_up[H,Fs], ws_down[Fs,H] (null iff F_shared == 0).
 * Output:  y[T,H].
 * Optional outputs (nullable): topk_idx[T,k] int32, topk_w[T,k] float,
 *          expert_offsets[E+1] int32 (exclusive prefix of per-expert counts),
 *          row_of_pair[T*k] int32 (row of pair t*k+j in expert-contiguous order),
 *          logits[T,E] float (the biased fp32 logits the selection used).
 * The workspace keeps the routing, the permuted rows and the activations
 * a, b, h, y_pair ([PR44] Changes: the forward keeps what the backward
 * reuses), plus the x and weight pointers, which must stay valid and
 * unmodified until moe_bwd.
 */
MOE_API int moe_fwd(const moe_dims* dims, void* ws, size_t ws_bytes, void* stream,
            const void* x, const void* w_router, const float* router_bias,
            const void* w_gate, const void* w_up, const void* w_down,
            const void* ws_gate, const void* ws_up, const void* ws_down,
            void* y,
            int32_t* topk_idx, float* topk_w, int32_t* expert_offsets,
            int32_t* row_of_pair, float* logits);

/*
 * moe_fwd_decode -- the forward of moe_fwd for decode-sized token counts, fused into
 * one persistent kernel, for inference ([I14] Evidence: per-token latency with 1..8
 * routed experts at inference time). At a handful of tokens the layer is a weight
 * stream; this call reads each touched expert's W_gate, W_up and W_down from HBM once,
 * with no other launch than its own.
 *   Computes what moe_fwd computes: y, and optionally the top-k experts, weights and
 *   the biased fp32 router logits the selection used. The router logits are summed in
 *   another order than moe_fwd's, so an index can differ from moe_fwd's at a near tie.
 * Needs dims.dtype == MOE_BF16, 1 <= T <= 16, E <= 256, k <= 16 and H, F,
 * F_shared <= 4096; other dims return MOE_ERR_UNSUPPORTED (use moe_fwd).
 * Inputs and outputs as moe_fwd (y[T,H]; topk_idx[T,k] int32, topk_w[T,k] float,
 * logits[T,E] float nullable). The workspace is the one moe_workspace_size() gives
 * for these dims. Nothing is kept for a backward: moe_select_retained / moe_bwd on
 * this workspace return MOE_ERR_STATE until the next moe_fwd.
 * Every wait inside the kernel is bounded; one that runs out writes MOE_ERR_TIMEOUT
 * to the workspace status word (moe_read_status).
 */
MOE_API int moe_fwd_decode(const moe_dims* dims, void* ws, size_t ws_bytes, void* stream,
                           const void* x, const void* w_router, const float* router_bias,
                           const void* w_gate, const void* w_up, const void* w_down,
                           const void* ws_gate, const void* ws_up, const void* ws_down,
                           void* y, int32_t* topk_idx, float* topk_w, float* logits);

/*
 * moe_select_retained -- per-pair scores and per-expert quota selection with
 * physical compaction ([LRMoE] Abstract: a per-pair estimate of the
 * contribution to the expert update, pairs selected within per-expert
 * quotas, physically compacted for smaller variable-size grouped GEMMs).
 *   score(t,j) = topk_w[t,j] * ||dy_t||_2 * ||x_t||_2
 *   q_e = min(quota[e], count_e); per expert the q_e pairs with the largest
 *   (score, then lower token) are kept and copied, in row order, into
 *   compact buffers used by moe_bwd(use_retained=1).
 * Inputs:  dy[T,H]; quota[E] int32 device (null = keep every pair). A
 *          negative quota entry sets MOE_ERR_DEVICE_ARG in the status word
 *          and is treated as 0.
 * Optional outputs (nullable): retained_offsets[E+1] int32 (exclusive prefix
 *          of kept counts), retained_rows[T*k] int32 (kept rows, in the
 *          expert-contiguous row numbering of moe_fwd's row_of_pair, listed
 *          expert by expert in ascending row order; entries past the total
 *          are left untouched), scores[T*k] float (per pair t*k+j).
 * Requires a prior moe_fwd on this workspace.
 */
MOE_API int moe_select_retained(const moe_dims* dims, void* ws, size_t ws_bytes, void* stream,
                        const void* dy, const int32_t* quota,
                        int32_t* retained_offsets, int32_t* retained_rows, float* scores);

/*
 * moe_bwd -- backward of L = <dy, y> ([I14] Proposal: dx and, for full
 * fine-tuning, dW; [LRMoE] Abstract: the expert backward runs on the
 * retained, compacted pairs).
 *   Expert part over kept pairs (all pairs when use_retained == 0):
 *     dy_r = w_r dy_t; dh = dy_r W_down[e]^T; da = dh*b*s(a)*(1+a(1-s(a)));
 *     db = dh*silu(a); dx_r = da W_gate[e]^T + db W_up[e]^T;
 *     dW_gate[e] = sum x_t^T da, dW_up[e] = sum x_t^T db, dW_down[e] = sum h^T dy_r.
 *   Router part over all pairs: g = <dy_t, y_pair>, dl[t,e_j] = w_j (g_j - sum_i w_i g_i),
 *     dx_t += dl_t w_router^T, dw_router = x^T dl (no gradient to router_bias).
 *   Shared expert: full backward with dy (never subject to retention).
 *   dx[T,H] = expert part + router part + shared part.
 * Inputs:  dy[T,H]; x must be the pointer given to moe_fwd (else MOE_ERR_STATE);
 *          use_retained = 1 needs a prior moe_select_retained on the same dy.
 * Outputs: dx[T,H]; unless MOE_FROZEN: dw_router[H,E], dw_gate[E,H,F],
 *          dw_up[E,H,F], dw_down[E,F,H] and, with a shared expert,
 *          dws_gate[H,Fs], dws_up[H,Fs], dws_down[Fs,H]. dW buffers are
 *          overwritten (experts with no kept pair get zeros); they must be
 *          null when MOE_FROZEN is set.
 */
MOE_API int moe_bwd(const moe_dims* dims, void* ws, size_t ws_bytes, void* stream,
            const void* dy, const void* x, int use_retained,
            void* dx, void* dw_router, void* dw_gate, void* dw_up, void* dw_down,
            void* dws_gate, void* dws_up, void* dws_down);

/*
 * moe_route_noalloc -- the routing stage of moe_fwd without any device
 * allocation and without a workspace. It is for callers that cannot call
 * cudaMalloc or lend the library memory: a runtime whose device memory pool
 * is fixed up front, a plugin that must not touch its host's allocator, a
 * process held to a pre-sized memory budget. The pages this library follows
 * have no counterpart to it; it exists only for those callers.
 *   Computes the routing moe_fwd reports through its optional outputs:
 *   router logits x w_router + router_bias (fp32), top-k experts per token
 *   (ties to the lower index), softmax-renormalised weights, per-expert
 *   exclusive offsets and the expert-contiguous row of every pair. The router
 *   GEMM runs with the same K split as moe_fwd whenever its fp32 partial sums
 *   fit in the scratch, and the results are then bit-identical to moe_fwd's;
 *   otherwise it runs with fewer splits, the logits are summed in another
 *   order, and an index may differ from moe_fwd's at a near tie.
 * Inputs:  x[T,H], w_router[H,E] (dims.dtype), router_bias[E] float (nullable).
 * Outputs (all required, device): topk_idx[T,k] int32, topk_w[T,k] float,
 *          expert_offsets[E+1] int32, row_of_pair[T*k] int32;
 *          device_status (nullable, one int32 on the device): set to MOE_OK,
 *          or to MOE_ERR_TIMEOUT if a bounded wait inside a kernel ran out.
 * Scratch: one fixed array of 32 MiB in the library's device memory (every
 *          GPU that loads the library holds it until the process exits).
 *          Without a K split the call needs about
 *          4*T*E + 12*ceil(T/64)*E + 8*T*k + 76*E bytes of it (each of ten
 *          entries rounded up to 256 bytes); a K split of ks parts adds
 *          4*(ks-1)*T*E. Dims that do not fit without a split are rejected with
 *          MOE_ERR_UNSUPPORTED before any work (T=8192, E=128, k=8 needs 9.1 MB
 *          with its split of 2; at k = 8 the largest T that fits is about
 *          55,800 for E=128, 256,000 for E=16 and 7,600 for E=1024).
 *          Every call on a device uses the same array and leaves its
 *          contents behind (nothing an earlier call left is ever read): calls
 *          that overlap on the GPU (two streams, or two threads without
 *          ordering) race on it and must be serialised.
 * The first call in each CUDA context looks up the array's device address
 * (cudaGetSymbolAddress) and keeps it; make that first call before any stream
 * capture. Calls no cudaMalloc/cudaFree or allocating library routine.
 */
MOE_API int moe_route_noalloc(const moe_dims* dims, void* stream, const void* x, const void* w_router,
                              const float* router_bias, int32_t* topk_idx, float* topk_w,
                              int32_t* expert_offsets, int32_t* row_of_pair, int32_t* device_status);

/*
 * moe_plan_quota -- per-expert retention quotas planned on the device from the
 * routing of the last moe_fwd ([LRMoE] Abstract: the forward plans retention
 * quotas under resource constraints).
 *   quota[e] = min(count_e, ceil(rho_num / rho_den * T*k / E)), and at most
 *   budget[e] when budget (int32 [E] device, nullable) is given (negative
 *   budgets count as 0). quota[E] int32 device output, usable directly by
 *   moe_select_retained. 0 <= rho_num <= 2^20, 1 <= rho_den <= 2^20.
 */
MOE_API int moe_plan_quota(const moe_dims* dims, void* ws, size_t ws_bytes, void* stream, int64_t rho_num,
                           int64_t rho_den, const int32_t* budget, int32_t* quota);

/*
 * moe_selftest_wait -- checks, on the GPU, the bounded barrier wait that every
 * pipelined kernel of the library uses. A one-thread kernel waits on an
 * mbarrier; with arrive != 0 it arrives first and *device_status becomes
 * MOE_OK, with arrive == 0 nothing arrives, the wait gives up after limit_us
 * (1 .. 1,000,000) and *device_status becomes MOE_ERR_TIMEOUT. The kernel
 * always returns, so the context stays usable. device_status: one int32 on the device.
 */
MOE_API int moe_selftest_wait(void* stream, int arrive, int64_t limit_us, int32_t* device_status);

/*
 * moe_selftest_decode_wait -- checks, on the GPU, the failure path of the fused decode
 * kernel: runs moe_fwd_decode (same arguments, same rules; no optional outputs) with
 * grid barrier `barrier` (1 = after the router, 2 = after gate/up, 3 = after h,
 * 4 = after down) needing one arrival more than the grid has, and every wait inside
 * the kernel bounded by limit_us (1 .. 1,000,000) instead of 1 s. That wait runs out,
 * the kernel writes MOE_ERR_TIMEOUT to the workspace status word (moe_read_status),
 * every warp leaves and the kernel returns with its copies landed: the context stays
 * usable and the next moe_fwd_decode on the workspace computes normally. y is left
 * unspecified.
 */
MOE_API int moe_selftest_decode_wait(const moe_dims* dims, void* ws, size_t ws_bytes, void* stream,
                                     const void* x, const void* w_router, const float* router_bias,
                                     const void* w_gate, const void* w_up, const void* w_down,
                                     const void* ws_gate, const void* ws_up, const void* ws_down, void* y,
                                     int barrier, int64_t limit_us);

/*
 * moe_read_status -- synchronises `stream` and returns the device status word
 * of the workspace (MOE_OK, MOE_ERR_TIMEOUT or MOE_ERR_DEVICE_ARG), then
 * clears it. Returns MOE_ERR_CUDA if the synchronisation itself failed.
 */
MOE_API int moe_read_status(void* ws, void* stream);

/* moe_last_error -- thread-local message describing the last non-OK return. */
MOE_API const char* moe_last_error(void);

/*
 * moe_workspace_entry -- diagnostic: name, byte offset and byte size of the
 * i-th buffer of the workspace layout for these dims (host-only). Lets tests
 * read saved intermediates (e.g. "ab" = a|b per padded row, "h", "y_pair",
 * "pad_off") after a call. Returns MOE_ERR_INVALID_ARG once i is past the
 * last entry. The layout is internal and may change between builds.
 */
MOE_API int moe_workspace_entry(const moe_dims* dims, int i, const char** name, size_t* offset, size_t* bytes);

/*
 * moe_kernel_launches -- number of CUDA kernels this library has launched in
 * this process so far (all workspaces, all streams). Host-only.
 */
MOE_API int64_t moe_kernel_launches(void);

/*
 * moe_timing_enable / moe_timing_read -- optional per-kernel-family timing.
 * When enabled (on != 0), the library brackets every grouped-GEMM launch and
 * every group of bandwidth-kernel launches with CUDA events recorded on the
 * caller's stream and keeps them. moe_timing_read synchronises those events
 * and writes, per family (0 = grouped GEMMs, 1 = bandwidth kernels), the total
 * milliseconds and the number of bracketed spans, then forgets them. Returns
 * MOE_OK or MOE_ERR_CUDA. Off by default; enabling adds two event records per
 * span. Process-wide (not per workspace); not for use during graph capture.
 */
MOE_API int moe_timing_enable(int on);
MOE_API int moe_timing_read(double ms_out[2], int64_t launches_out[2]);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
