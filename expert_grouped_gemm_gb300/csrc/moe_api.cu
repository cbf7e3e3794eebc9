// moe_api.cu -- the C ABI: validation, workspace carve-up, kernel sequencing.
//
// moe_fwd / moe_select_retained / moe_bwd only enqueue kernels on the caller's
// stream. Host-side call-order state (which x the forward saw, whether a
// selection was made and for which dy) lives in a small registry keyed by the
// workspace pointer; the activations themselves stay in the workspace.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <unordered_map>
#include <vector>

#include "common.cuh"
#include "decode.h"
#include "gemm_launch.h"
#include "kernels.h"
#include "layout.h"

using namespace moe;

namespace {

thread_local std::string g_err;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}

#define CK(call)                                                                                  \
  do {                                                                                            \
    cudaError_t e_ = (call);                                                                      \
    if (e_ != cudaSuccess) return fail(MOE_ERR_CUDA, "%s: %s", #call, cudaGetErrorString(e_));    \
  } while (0)

// Every kernel launch of the library goes through CKL, which also counts it.
std::atomic<int64_t> g_launches{0};
#define CKL(call)      \
  do {                 \
    g_launches += 1;   \
    CK(call);          \
  } while (0)

// ------------------------------------------------------------------ validation
int check_dims(const moe_dims* d) {
  if (!d) return fail(MOE_ERR_INVALID_ARG, "dims is null");
  if (d->T < 1 || d->H < 1 || d->F < 1 || d->E < 1 || d->k < 1)
    return fail(MOE_ERR_INVALID_ARG, "T, H, F, E, k must be >= 1");
  if (d->k > d->E) return fail(MOE_ERR_INVALID_ARG, "k (%lld) > E (%lld)", (long long)d->k, (long long)d->E);
  if (d->E > 1024) return fail(MOE_ERR_UNSUPPORTED, "E > 1024");
  if (d->F_shared < 0) return fail(MOE_ERR_INVALID_ARG, "F_shared < 0");
  if (d->dtype != MOE_BF16 && d->dtype != MOE_F32) return fail(MOE_ERR_INVALID_ARG, "unknown dtype %d", d->dtype);
  if (d->flags & ~(MOE_FROZEN | MOE_RECOMPUTE)) return fail(MOE_ERR_INVALID_ARG, "unknown flags 0x%x", d->flags);
  const int64_t P = d->T * d->k;
  if (P + 16 * d->E >= (1ll << 31) - 1024) return fail(MOE_ERR_UNSUPPORTED, "T*k too large for int32 row indices");
  if (d->H >= (1 << 24) || d->F >= (1 << 24) || d->F_shared >= (1 << 24))
    return fail(MOE_ERR_UNSUPPORTED, "H/F too large");
  if (d->dtype == MOE_BF16) {
    if (d->H % 64 || d->F % 64 || d->F_shared % 64)
      return fail(MOE_ERR_UNSUPPORTED, "bf16 needs H, F, F_shared multiples of 64");
    if (d->E % 16) return fail(MOE_ERR_UNSUPPORTED, "bf16 needs E multiple of 16");
  }
  return MOE_OK;
}

WsLayout make_layout(const moe_dims* d) {
  WsLayout L;
  L.T = d->T;
  L.H = d->H;
  L.F = d->F;
  L.E = d->E;
  L.k = d->k;
  L.Fs = d->F_shared;
  L.P = d->T * d->k;
  L.Rmax = L.P + 15 * L.E;
  L.Tpad = (L.T + 15) / 16 * 16;
  L.C = (L.T + 63) / 64;
  L.es = d->dtype == MOE_BF16 ? 2 : 4;
  const int64_t es = L.es, T = L.T, H = L.H, F = L.F, E = L.E, k = L.k, Fs = L.Fs, P = L.P, R = L.Rmax,
                Tp = L.Tpad, C = L.C;
  L.Rdec = std::min<int64_t>(R, P + 15 * std::min<int64_t>(E, P));
  {  // K-split partials: room for kMaxSplit splits of every GEMM that may be split on a GPU of up to
     // kSplitMaxSms SMs (the split needs at most half the SMs busy without it)
    auto few = [](int64_t tiles) { return tiles * 2 <= kSplitMaxSms; };
    const int64_t act = std::min<int64_t>(E, P) + P / 128;  // bound on 128-row expert tiles
    int64_t per = 0;
    if (few(((T + 127) / 128) * ((E + 127) / 128))) per = std::max(per, T * E);        // router logits
    if (few(((H + 127) / 128) * ((E + 127) / 128))) per = std::max(per, H * E);        // router dW
    if (few(act * ((F + 127) / 128))) per = std::max(per, L.Rdec * 2 * F);            // expert gate/up
    if (few(act * ((H + 255) / 256))) per = std::max(per, L.Rdec * H);                // expert down
    L.part_elems = per * kMaxSplit;
  }
  const int64_t sizes[] = {
      256,                       // status (the decode kernel's barrier counter at byte 16)
      C * E * 8,                 // masks (right after status: one memset clears both)
      T * E * 4,                 // logits
      T * k * 4, T * k * 4,      // topk idx, w
      T * 4,                     // xnorm
      C * E * 4,                 // chunk_base
      E * 4, (E + 1) * 4, (E + 1) * 4, (E + 1) * 4,  // count offset pad_off tile_off
      P * 4, P * 4, R * 4,       // rowp_of_pair row_of_pair pair_of_row
      R * H * es, R * 2 * F * es, R * F * es, R * H * es,  // x_perm ab h y_pair
      Tp * 2 * Fs * es, Tp * Fs * es, Tp * H * es,         // sh_ab sh_h sh_y
      R * 4, R * 4, R * H * es,  // g score dy_perm
      R * 4, E * 4, (E + 1) * 4, (E + 1) * 4, (E + 1) * 4, R * 4, P * 4, P * 4,  // ret_*
      R * H * es, R * 2 * F * es, R * F * es, R * H * es,  // x_c ab_c h_c dy_c
      R * 2 * F * es, R * H * es,  // dab dx_pair
      Tp * E * es, T * k * 4, E * H * es,  // dl dl_sel wrT
      Tp * 2 * Fs * es, Tp * H * es,       // sh_dab sh_dx
      E * 4, E * 4,                        // order ret_order
      (E + 1) * 4, (E + 1) * 4,            // tile_off2 ret_tile_off2
      (P / 128 + E + 1) * 16, (P / 128 + E + 1) * 16,  // tile_rec ret_tile_rec
      E * 16, E * 16,                                  // ord_rec ret_ord_rec
      L.part_elems * 4,                                // part
      (P / 256 + E + 1) * 16, (P / 256 + E + 1) * 16,  // tile_rec2 ret_tile_rec2
      (int64_t)(d->dtype == MOE_BF16 && decode_supported(T, H, F, E, k, Fs)  // decode scratch (T <= 16)
                    ? decode_scratch_bytes(T, H, F, E, k, Fs)
                    : 0),
  };
  L.n = (int)(sizeof(sizes) / sizeof(sizes[0]));
  size_t off = 0;
  for (int i = 0; i < L.n; ++i) {
    L.off[i] = off;
    off += ((size_t)sizes[i] + 255) / 256 * 256;
  }
  L.total = off;
  return L;
}

// Names of the workspace entries, in layout order (kept in step with make_ptrs).
const char* const kEntryNames[] = {
    "status", "masks", "logits", "topk_idx", "topk_w", "xnorm", "chunk_base", "count", "offset", "pad_off",
    "tile_off", "rowp_of_pair", "row_of_pair", "pair_of_row", "x_perm", "ab", "h", "y_pair", "sh_ab", "sh_h",
    "sh_y", "g", "score", "dy_perm", "ret_cidx", "ret_count", "ret_offset", "ret_pad_off", "ret_tile_off",
    "ret_src", "crow_of_pair", "ret_rows", "x_c", "ab_c", "h_c", "dy_c", "dab", "dx_pair", "dl", "dl_sel", "wrT",
    "sh_dab", "sh_dx", "order", "ret_order", "tile_off2", "ret_tile_off2", "tile_rec", "ret_tile_rec", "ord_rec",
    "ret_ord_rec", "part", "tile_rec2", "ret_tile_rec2", "decode"};

WsPtrs make_ptrs(const WsLayout& L, void* ws) {
  char* b = static_cast<char*>(ws);
  int i = 0;
  auto nx = [&]() { return static_cast<void*>(b + L.off[i++]); };
  WsPtrs p;
  p.status = (int*)nx();
  p.masks = (uint64_t*)nx();
  p.logits = (float*)nx();
  p.topk_idx = (int*)nx();
  p.topk_w = (float*)nx();
  p.xnorm = (float*)nx();
  p.chunk_base = (int*)nx();
  p.count = (int*)nx();
  p.offset = (int*)nx();
  p.pad_off = (int*)nx();
  p.tile_off = (int*)nx();
  p.rowp_of_pair = (int*)nx();
  p.row_of_pair = (int*)nx();
  p.pair_of_row = (int*)nx();
  p.x_perm = nx();
  p.ab = nx();
  p.h = nx();
  p.y_pair = nx();
  p.sh_ab = nx();
  p.sh_h = nx();
  p.sh_y = nx();
  p.g = (float*)nx();
  p.score = (float*)nx();
  p.dy_perm = nx();
  p.ret_cidx = (int*)nx();
  p.ret_count = (int*)nx();
  p.ret_offset = (int*)nx();
  p.ret_pad_off = (int*)nx();
  p.ret_tile_off = (int*)nx();
  p.ret_src = (int*)nx();
  p.crow_of_pair = (int*)nx();
  p.ret_rows = (int*)nx();
  p.x_c = nx();
  p.ab_c = nx();
  p.h_c = nx();
  p.dy_c = nx();
  p.dab = nx();
  p.dx_pair = nx();
  p.dl = nx();
  p.dl_sel = (float*)nx();
  p.wrT = nx();
  p.sh_dab = nx();
  p.sh_dx = nx();
  p.order = (int*)nx();
  p.ret_order = (int*)nx();
  p.tile_off2 = (int*)nx();
  p.ret_tile_off2 = (int*)nx();
  p.tile_rec = (int4*)nx();
  p.ret_tile_rec = (int4*)nx();
  p.ord_rec = (int4*)nx();
  p.ret_ord_rec = (int4*)nx();
  p.part = (float*)nx();
  p.tile_rec2 = (int4*)nx();
  p.ret_tile_rec2 = (int4*)nx();
  p.decode = nx();
  return p;
}

// ------------------------------------------------------------------ call-order state
struct State {
  moe_dims d;
  bool fwd_done = false;
  const void *x = nullptr, *w_router = nullptr, *w_gate = nullptr, *w_up = nullptr, *w_down = nullptr;
  const void *ws_gate = nullptr, *ws_up = nullptr, *ws_down = nullptr;
  bool sel_done = false;
  const void* sel_dy = nullptr;
};
std::mutex g_mu;
std::unordered_map<void*, State> g_state;

// A stream of the workspace's own for the backward's router-gradient and dX-reduce
// kernels, which run beside the dW GEMMs: forked from the caller's stream by `fork`
// after the dX GEMMs and joined back by `join` before the router dW GEMM, so the
// call's work stays ordered on (and capturable from) the caller's stream.
#ifndef MOE_BWD_OVERLAP
#define MOE_BWD_OVERLAP 1  // 0: every backward kernel on the caller's stream
#endif
struct Side {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
std::unordered_map<void*, Side> g_side;  // guarded by g_mu

cudaError_t side_for(void* ws, Side* out) {
  std::lock_guard<std::mutex> lk(g_mu);
  Side& sd = g_side[ws];
  if (!sd.s) {
    cudaError_t e = cudaStreamCreateWithFlags(&sd.s, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&sd.fork, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&sd.join, cudaEventDisableTiming);
    if (e != cudaSuccess) {
      if (sd.fork) cudaEventDestroy(sd.fork);
      if (sd.s) cudaStreamDestroy(sd.s);
      sd = Side();
      return e;
    }
  }
  *out = sd;
  return cudaSuccess;
}

bool same_dims(const moe_dims& a, const moe_dims& b) {
  return a.T == b.T && a.H == b.H && a.F == b.F && a.E == b.E && a.k == b.k && a.F_shared == b.F_shared &&
         a.dtype == b.dtype && a.flags == b.flags;
}

int check_ws(const moe_dims* d, void* ws, size_t ws_bytes, WsLayout* L) {
  int rc = check_dims(d);
  if (rc) return rc;
  if (!ws) return fail(MOE_ERR_WORKSPACE, "workspace is null");
  if (reinterpret_cast<uintptr_t>(ws) & 255) return fail(MOE_ERR_WORKSPACE, "workspace not 256-byte aligned");
  *L = make_layout(d);
  if (ws_bytes < L->total)
    return fail(MOE_ERR_WORKSPACE, "workspace too small: %zu < %zu bytes", ws_bytes, L->total);
  return MOE_OK;
}

int check_ptr(const void* p, const char* name, bool required, int align = 16) {
  if (!p) return required ? fail(MOE_ERR_INVALID_ARG, "%s is null", name) : MOE_OK;
  if (reinterpret_cast<uintptr_t>(p) % align) return fail(MOE_ERR_INVALID_ARG, "%s not %d-byte aligned", name, align);
  return MOE_OK;
}

int num_sms_current() {
  static std::mutex mu;
  static std::unordered_map<int, int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  std::lock_guard<std::mutex> lk(mu);
  auto it = cache.find(dev);
  if (it != cache.end()) return it->second;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  cache[dev] = n;
  return n;
}

// ------------------------------------------------------------------ optional timing
struct Timing {
  std::mutex mu;
  bool on = false;
  struct Rec {
    cudaEvent_t a, b;
    int fam;
  };
  std::vector<Rec> recs;
  std::vector<cudaEvent_t> pool;
  cudaEvent_t get() {
    if (!pool.empty()) {
      cudaEvent_t e = pool.back();
      pool.pop_back();
      return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
  }
} g_timing;

struct Span {
  cudaStream_t st;
  int fam;
  cudaEvent_t a = nullptr;
  Span(cudaStream_t s, int f) : st(s), fam(f) {
    std::lock_guard<std::mutex> lk(g_timing.mu);
    if (g_timing.on) {
      a = g_timing.get();
      cudaEventRecord(a, st);
    }
  }
  ~Span() {
    if (!a) return;
    std::lock_guard<std::mutex> lk(g_timing.mu);
    cudaEvent_t b = g_timing.get();
    cudaEventRecord(b, st);
    g_timing.recs.push_back({a, b, fam});
  }
};

enum { FAM_GEMM = 0, FAM_BW = 1 };

// ------------------------------------------------------------------ GEMM helpers
// 1: the variable-M store GEMMs (expert down, dX of the pairs) run weight-stationary on
// CTA pairs (gemm_ws.cu) where their shapes allow. Parity-green, measured slower than the
// single-CTA kernel at the Qwen3 shape, so off by default.
#ifndef MOE_WS
#define MOE_WS 0
#endif

cudaError_t run_gemm(const GemmArgs& a, int bf16, int bn, cudaStream_t st, int sms) {
  Span sp(st, FAM_GEMM);
  if (bf16 && MOE_WS && bn == 256 && ws_store_supported(a)) return launch_ws_store(a, st, sms);
  if (bf16) return launch_tc_gemm(a, bn, st, sms, 0);
  return launch_simt_gemm_f32(a, st);
}

// K split of a GEMM with `tiles` output tiles of `kblocks` k-blocks: used only when
// the tiles alone would leave at least half of the SMs idle, and only as far as the
// partial buffer holds `elems` fp32 per split. No split is left without k-blocks.
int ksplit_for(const WsLayout& L, int64_t tiles, int kblocks, int sms, int64_t elems) {
  if (tiles <= 0 || tiles * 2 > sms || kblocks < 2 || elems <= 0) return 1;
  int ks = (int)std::min<int64_t>({(int64_t)sms / tiles, (int64_t)kblocks, (int64_t)kMaxSplit, L.part_elems / elems});
  if (ks < 2) return 1;
  const int per = (kblocks + ks - 1) / ks;
  return (kblocks + per - 1) / per;
}

GemmArgs base_args(int* status) {
  GemmArgs a;
  memset(&a, 0, sizeof(a));
  a.status = status;
  return a;
}

}  // namespace

// The expert forward GEMMs: gate/up with fused SwiGLU, down, and the shared
// expert. moe_fwd runs them; in MOE_RECOMPUTE mode the retention select or the
// backward runs them again (same kernels, same inputs: the same bits).
int expert_forward_gemms(const WsLayout& L, const WsPtrs& p, int bf, int sms, cudaStream_t st, const void* w_gate,
                         const void* w_up, const void* w_down, const void* ws_gate, const void* ws_up,
                         const void* ws_down, const void* x) {
  const int T = (int)L.T, H = (int)L.H, F = (int)L.F, E = (int)L.E, Fs = (int)L.Fs;
  const bool shared = L.Fs > 0;
  const int64_t act_tiles = std::min<int64_t>(L.E, L.P) + L.P / 128;  // bound on 128-row expert tiles
  // expert gate/up with fused SwiGLU
  {
    GemmArgs a = base_args(p.status);
    a.var_k = 0;
    a.G = E;
    a.rows = p.count;
    a.row_off = p.pad_off;
    a.tile_off = p.tile_off;
    a.tile_rec = p.tile_rec;
    a.tile_rec2 = p.tile_rec2;
    a.tile_off2 = p.tile_off2;
    a.K = H;
    a.N = F;
    a.paired = 1;
    a.A = p.x_perm;
    a.lda = H;
    a.a_rows = L.Rmax;
    a.B0 = w_gate;
    a.B1 = w_up;
    a.ldb = F;
    a.b_rows = L.E * L.H;
    a.epi = EPI_SWIGLU_FWD;
    a.out0 = p.ab;
    a.ldo = 2 * F;
    a.out1 = p.h;
    a.ldo1 = F;
    a.zero_pad = 1;
    a.out_rows = L.Rmax;
    const int ks = bf ? ksplit_for(L, act_tiles * ((F + 127) / 128), H / kTileK, sms, L.Rdec * 2 * F) : 1;
    if (ks > 1) {  // decode-sized: K split into fp32 partials, then the SwiGLU epilogue in a second pass
      a.epi = EPI_F32;
      a.out0 = p.part;
      a.out1 = nullptr;
      a.ksplit = ks;
      a.part_stride = L.Rdec * 2 * F;
      CKL(run_gemm(a, bf, 256, st, sms));
      Span sp(st, FAM_BW);
      CKL(launch_splitk_swiglu(p.part, L.Rdec * 2 * F, ks, p.pad_off + E, L.Rdec, p.pair_of_row, F, p.ab, p.h, sms,
                               st));
    } else {
      CKL(run_gemm(a, bf, 256, st, sms));
    }
  }
  // expert down
  {
    GemmArgs a = base_args(p.status);
    a.var_k = 0;
    a.G = E;
    a.rows = p.count;
    a.row_off = p.pad_off;
    a.tile_off = p.tile_off;
    a.tile_rec = p.tile_rec;
    a.tile_rec2 = p.tile_rec2;
    a.tile_off2 = p.tile_off2;
    a.K = F;
    a.N = H;
    a.A = p.h;
    a.lda = F;
    a.a_rows = L.Rmax;
    a.B0 = w_down;
    a.ldb = H;
    a.b_rows = L.E * L.F;
    a.epi = EPI_STORE;
    a.out0 = p.y_pair;
    a.ldo = H;
    a.zero_pad = 1;
    a.out_rows = L.Rmax;
    const int ks = bf ? ksplit_for(L, act_tiles * ((H + 255) / 256), F / kTileK, sms, L.Rdec * H) : 1;
    if (ks > 1) {
      a.epi = EPI_F32;
      a.out0 = p.part;
      a.ksplit = ks;
      a.part_stride = L.Rdec * H;
      CKL(run_gemm(a, bf, 256, st, sms));
      Span sp(st, FAM_BW);
      CKL(launch_splitk_store(p.part, L.Rdec * H, ks, p.pad_off + E, 0, L.Rdec, p.pair_of_row, H, H, p.y_pair, sms,
                              st));
    } else {
      CKL(run_gemm(a, bf, 256, st, sms));
    }
  }
  if (shared) {
    GemmArgs a = base_args(p.status);
    a.var_k = 0;
    a.G = 1;
    a.rows_const = T;
    a.K = H;
    a.N = Fs;
    a.paired = 1;
    a.A = x;
    a.lda = H;
    a.a_rows = T;
    a.B0 = ws_gate;
    a.B1 = ws_up;
    a.ldb = Fs;
    a.b_rows = H;
    a.epi = EPI_SWIGLU_FWD;
    a.out0 = p.sh_ab;
    a.ldo = 2 * Fs;
    a.out1 = p.sh_h;
    a.ldo1 = Fs;
    a.zero_pad = 1;
    a.out_rows = L.Tpad;
    CKL(run_gemm(a, bf, 256, st, sms));
    GemmArgs b = base_args(p.status);
    b.var_k = 0;
    b.G = 1;
    b.rows_const = T;
    b.K = Fs;
    b.N = H;
    b.A = p.sh_h;
    b.lda = Fs;
    b.a_rows = L.Tpad;
    b.B0 = ws_down;
    b.ldb = H;
    b.b_rows = Fs;
    b.epi = EPI_STORE;
    b.out0 = p.sh_y;
    b.ldo = H;
    b.zero_pad = 1;
    b.out_rows = L.Tpad;
    CKL(run_gemm(b, bf, 256, st, sms));
  }
  return MOE_OK;
}

// Hooks for the other translation units of the library (not part of the C ABI).
namespace moe {
int internal_check_dims(const moe_dims* d) { return check_dims(d); }
// The K split moe_fwd uses for the router logits GEMM at these dims on a GPU of `sms` SMs
// (1: none). Valid dims only.
int internal_router_ksplit(const moe_dims* d, int sms) {
  if (d->dtype != MOE_BF16) return 1;
  const WsLayout L = make_layout(d);
  return ksplit_for(L, ((L.T + 127) / 128) * ((L.E + 127) / 128), (int)(L.H / kTileK), sms, L.T * L.E);
}
int internal_fail(int code, const char* msg) { return fail(code, "%s", msg); }
void internal_count_launches(int n) { g_launches += n; }
}  // namespace moe

// ====================================================================== C ABI
extern "C" {

const char* moe_last_error(void) { return g_err.c_str(); }

int moe_workspace_size(const moe_dims* dims, size_t* bytes) {
  int rc = check_dims(dims);
  if (rc) return rc;
  if (!bytes) return fail(MOE_ERR_INVALID_ARG, "bytes is null");
  *bytes = make_layout(dims).total;
  return MOE_OK;
}

int moe_workspace_entry(const moe_dims* dims, int i, const char** name, size_t* offset, size_t* bytes) {
  int rc = check_dims(dims);
  if (rc) return rc;
  const WsLayout L = make_layout(dims);
  const int n = (int)(sizeof(kEntryNames) / sizeof(kEntryNames[0]));
  if (n != L.n) return fail(MOE_ERR_UNSUPPORTED, "workspace entry table out of step");
  if (i < 0 || i >= n) return fail(MOE_ERR_INVALID_ARG, "entry %d out of range [0, %d)", i, n);
  if (name) *name = kEntryNames[i];
  if (offset) *offset = L.off[i];
  if (bytes) *bytes = (i + 1 < n ? L.off[i + 1] : L.total) - L.off[i];
  return MOE_OK;
}

int64_t moe_kernel_launches(void) { return g_launches.load(); }

int moe_plan_quota(const moe_dims* dims, void* ws, size_t ws_bytes, void* stream, int64_t rho_num, int64_t rho_den,
                   const int32_t* budget, int32_t* quota) {
  WsLayout L;
  int rc = check_ws(dims, ws, ws_bytes, &L);
  if (rc) return rc;
  if ((rc = check_ptr(quota, "quota", true, 4)) || (rc = check_ptr(budget, "budget", false, 4))) return rc;
  if (rho_num < 0 || rho_den < 1 || rho_num > (1ll << 20) || rho_den > (1ll << 20))
    return fail(MOE_ERR_INVALID_ARG, "need 0 <= rho_num <= 2^20 and 1 <= rho_den <= 2^20");
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_state.find(ws);
    if (it == g_state.end() || !it->second.fwd_done)
      return fail(MOE_ERR_STATE, "moe_plan_quota before moe_fwd on this workspace");
    if (!same_dims(it->second.d, *dims)) return fail(MOE_ERR_STATE, "dims differ from moe_fwd's");
  }
  const WsPtrs p = make_ptrs(L, ws);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Span sp(st, FAM_BW);
  CKL(launch_plan_quota(p.count, (int)L.E, L.P, rho_num, rho_den, budget, quota, st));
  return MOE_OK;
}

int moe_timing_enable(int on) {
  std::lock_guard<std::mutex> lk(g_timing.mu);
  g_timing.on = on != 0;
  return MOE_OK;
}

int moe_timing_read(double ms_out[2], int64_t launches_out[2]) {
  std::lock_guard<std::mutex> lk(g_timing.mu);
  double ms[2] = {0, 0};
  int64_t n[2] = {0, 0};
  int rc = MOE_OK;
  for (auto& r : g_timing.recs) {
    if (cudaEventSynchronize(r.b) != cudaSuccess) rc = fail(MOE_ERR_CUDA, "event sync failed");
    float t = 0.f;
    if (cudaEventElapsedTime(&t, r.a, r.b) == cudaSuccess) {
      ms[r.fam] += t;
      n[r.fam] += 1;
    }
    g_timing.pool.push_back(r.a);
    g_timing.pool.push_back(r.b);
  }
  g_timing.recs.clear();
  if (ms_out) {
    ms_out[0] = ms[0];
    ms_out[1] = ms[1];
  }
  if (launches_out) {
    launches_out[0] = n[0];
    launches_out[1] = n[1];
  }
  return rc;
}

int moe_read_status(void* ws, void* stream) {
  if (!ws) return fail(MOE_ERR_WORKSPACE, "workspace is null");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int v = 0;
  CK(cudaMemcpyAsync(&v, ws, sizeof(int), cudaMemcpyDeviceToHost, st));
  CK(cudaStreamSynchronize(st));
  const int zero = 0;
  CK(cudaMemcpyAsync(ws, &zero, sizeof(int), cudaMemcpyHostToDevice, st));
  CK(cudaStreamSynchronize(st));
  if (v != MOE_OK) fail(v, "device status %d", v);
  return v;
}

int moe_fwd(const moe_dims* dims, void* ws, size_t ws_bytes, void* stream, const void* x, const void* w_router,
            const float* router_bias, const void* w_gate, const void* w_up, const void* w_down, const void* ws_gate,
            const void* ws_up, const void* ws_down, void* y, int32_t* topk_idx, float* topk_w,
            int32_t* expert_offsets, int32_t* row_of_pair, float* logits) {
  WsLayout L;
  int rc = check_ws(dims, ws, ws_bytes, &L);
  if (rc) return rc;
  const bool shared = dims->F_shared > 0;
  if ((rc = check_ptr(x, "x", true)) || (rc = check_ptr(w_router, "w_router", true)) ||
      (rc = check_ptr(router_bias, "router_bias", false, 4)) || (rc = check_ptr(w_gate, "w_gate", true)) ||
      (rc = check_ptr(w_up, "w_up", true)) || (rc = check_ptr(w_down, "w_down", true)) ||
      (rc = check_ptr(y, "y", true)) || (rc = check_ptr(topk_idx, "topk_idx", false, 4)) ||
      (rc = check_ptr(topk_w, "topk_w", false, 4)) || (rc = check_ptr(expert_offsets, "expert_offsets", false, 4)) ||
      (rc = check_ptr(row_of_pair, "row_of_pair", false, 4)) || (rc = check_ptr(logits, "logits", false, 4)))
    return rc;
  if (shared) {
    if ((rc = check_ptr(ws_gate, "ws_gate", true)) || (rc = check_ptr(ws_up, "ws_up", true)) ||
        (rc = check_ptr(ws_down, "ws_down", true)))
      return rc;
  } else if (ws_gate || ws_up || ws_down) {
    return fail(MOE_ERR_INVALID_ARG, "shared-expert weights given but F_shared == 0");
  }

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const WsPtrs p = make_ptrs(L, ws);
  const int bf = dims->dtype == MOE_BF16;
  const int sms = num_sms_current();
  const int T = (int)L.T, H = (int)L.H, F = (int)L.F, E = (int)L.E, k = (int)L.k, Fs = (int)L.Fs;

  // the status word and the routing chunk masks (the next entry) start at zero
  CK(cudaMemsetAsync(p.status, 0, L.off[2] - L.off[0], st));

  // router logits = x W_r  (fp32 out; bias added by the top-k kernel)
  const int rks = moe::internal_router_ksplit(dims, sms);
  {
    GemmArgs a = base_args(p.status);
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
    a.out0 = p.logits;
    a.ldo = E;
    if (rks > 1) {  // few tiles: K split, the top-k kernel adds the partial sums
      a.ksplit = rks;
      a.out0 = p.part;
      a.part_stride = (int64_t)T * E;
    }
    CKL(run_gemm(a, bf, 128, st, sms));
  }
  {
    Span sp(st, FAM_BW);
    CKL(launch_route_topk(p.logits, router_bias, T, E, k, p.topk_idx, p.topk_w, p.masks, st,
                          rks > 1 ? p.part : nullptr, rks, (int64_t)T * E, /*masks_clear=*/true, logits, topk_idx,
                          topk_w));
    CKL(launch_route_scan(p.masks, (int)L.C, E, p.count, p.offset, p.pad_off, p.tile_off, p.chunk_base, p.pair_of_row,
                         expert_offsets, st, p.order, p.tile_off2, p.tile_rec, p.ord_rec, p.tile_rec2));
    CKL(launch_route_index(p.masks, p.chunk_base, p.topk_idx, p.offset, p.pad_off, T, E, k, p.rowp_of_pair,
                          p.row_of_pair, p.pair_of_row, st, row_of_pair));
    if (bf)
      CKL(launch_gather_rows<__nv_bfloat16>(x, p.pair_of_row, p.pad_off + E, L.Rmax, H, k, p.x_perm, p.xnorm, sms, st));
    else
      CKL(launch_gather_rows<float>(x, p.pair_of_row, p.pad_off + E, L.Rmax, H, k, p.x_perm, p.xnorm, sms, st));
  }
  if ((rc = expert_forward_gemms(L, p, bf, sms, st, w_gate, w_up, w_down, ws_gate, ws_up, ws_down, x))) return rc;
  {
    Span sp(st, FAM_BW);
    if (bf)
      CKL(launch_combine<__nv_bfloat16>(p.y_pair, p.rowp_of_pair, p.topk_w, shared ? p.sh_y : nullptr, T, H, k, y, sms,
                                       st));
    else
      CKL(launch_combine<float>(p.y_pair, p.rowp_of_pair, p.topk_w, shared ? p.sh_y : nullptr, T, H, k, y, sms, st));
  }

  std::lock_guard<std::mutex> lk(g_mu);
  State& s = g_state[ws];
  s = State();
  s.d = *dims;
  s.fwd_done = true;
  s.x = x;
  s.w_router = w_router;
  s.w_gate = w_gate;
  s.w_up = w_up;
  s.w_down = w_down;
  s.ws_gate = ws_gate;
  s.ws_up = ws_up;
  s.ws_down = ws_down;
  return MOE_OK;
}

// moe_fwd_decode and its self-test: stall (1..4) makes that grid barrier of the kernel
// unreachable, wait_ns bounds every wait inside it.
static int fwd_decode_impl(const moe_dims* dims, void* ws, size_t ws_bytes, void* stream, const void* x,
                           const void* w_router, const float* router_bias, const void* w_gate, const void* w_up,
                           const void* w_down, const void* ws_gate, const void* ws_up, const void* ws_down, void* y,
                           int32_t* topk_idx, float* topk_w, float* logits, unsigned stall, uint64_t wait_ns) {
  WsLayout L;
  int rc = check_ws(dims, ws, ws_bytes, &L);
  if (rc) return rc;
  if (dims->dtype != MOE_BF16) return fail(MOE_ERR_UNSUPPORTED, "moe_fwd_decode: bf16 only");
  if (!decode_supported(L.T, L.H, L.F, L.E, L.k, L.Fs))
    return fail(MOE_ERR_UNSUPPORTED,
                "moe_fwd_decode: needs T <= 16, E <= 256, k <= 16 and H, F, F_shared <= 4096 (T=%lld E=%lld k=%lld)",
                (long long)L.T, (long long)L.E, (long long)L.k);
  const bool shared = dims->F_shared > 0;
  if ((rc = check_ptr(x, "x", true)) || (rc = check_ptr(w_router, "w_router", true)) ||
      (rc = check_ptr(router_bias, "router_bias", false, 4)) || (rc = check_ptr(w_gate, "w_gate", true)) ||
      (rc = check_ptr(w_up, "w_up", true)) || (rc = check_ptr(w_down, "w_down", true)) ||
      (rc = check_ptr(y, "y", true)) || (rc = check_ptr(topk_idx, "topk_idx", false, 4)) ||
      (rc = check_ptr(topk_w, "topk_w", false, 4)) || (rc = check_ptr(logits, "logits", false, 4)))
    return rc;
  if (shared) {
    if ((rc = check_ptr(ws_gate, "ws_gate", true)) || (rc = check_ptr(ws_up, "ws_up", true)) ||
        (rc = check_ptr(ws_down, "ws_down", true)))
      return rc;
  } else if (ws_gate || ws_up || ws_down) {
    return fail(MOE_ERR_INVALID_ARG, "shared-expert weights given but F_shared == 0");
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const WsPtrs p = make_ptrs(L, ws);
  // one memset for the status word and, 16 bytes further in the same 256-byte entry,
  // the decode kernel's grid-barrier counter
  unsigned* dec_sync = reinterpret_cast<unsigned*>(reinterpret_cast<char*>(p.status) + 16);
  CK(cudaMemsetAsync(p.status, 0, 32, st));
  g_launches += 1;
  CK(launch_decode_fwd((int)L.T, (int)L.H, (int)L.F, (int)L.E, (int)L.k, (int)L.Fs, x, w_router, router_bias, w_gate,
                       w_up, w_down, ws_gate, ws_up, ws_down, y, p.topk_idx, p.topk_w, topk_idx, topk_w, logits,
                       p.decode, p.status, dec_sync, num_sms_current(), st, stall, wait_ns));
  // inference only: the routing buffers no longer hold a forward the backward could use
  std::lock_guard<std::mutex> lk(g_mu);
  g_state[ws] = State();
  return MOE_OK;
}

int moe_fwd_decode(const moe_dims* dims, void* ws, size_t ws_bytes, void* stream, const void* x, const void* w_router,
                   const float* router_bias, const void* w_gate, const void* w_up, const void* w_down,
                   const void* ws_gate, const void* ws_up, const void* ws_down, void* y, int32_t* topk_idx,
                   float* topk_w, float* logits) {
  return fwd_decode_impl(dims, ws, ws_bytes, stream, x, w_router, router_bias, w_gate, w_up, w_down, ws_gate, ws_up,
                         ws_down, y, topk_idx, topk_w, logits, 0u, 1000000000ull);
}

int moe_selftest_decode_wait(const moe_dims* dims, void* ws, size_t ws_bytes, void* stream, const void* x,
                             const void* w_router, const float* router_bias, const void* w_gate, const void* w_up,
                             const void* w_down, const void* ws_gate, const void* ws_up, const void* ws_down,
                             void* y, int barrier, int64_t limit_us) {
  if (barrier < 1 || barrier > 4) return fail(MOE_ERR_INVALID_ARG, "moe_selftest_decode_wait: barrier must be 1..4");
  if (limit_us < 1 || limit_us > 1000000)
    return fail(MOE_ERR_INVALID_ARG, "moe_selftest_decode_wait: limit_us must be 1..1000000");
  return fwd_decode_impl(dims, ws, ws_bytes, stream, x, w_router, router_bias, w_gate, w_up, w_down, ws_gate, ws_up,
                         ws_down, y, nullptr, nullptr, nullptr, (unsigned)barrier, (uint64_t)limit_us * 1000ull);
}

int moe_select_retained(const moe_dims* dims, void* ws, size_t ws_bytes, void* stream, const void* dy,
                        const int32_t* quota, int32_t* retained_offsets, int32_t* retained_rows, float* scores) {
  WsLayout L;
  int rc = check_ws(dims, ws, ws_bytes, &L);
  if (rc) return rc;
  if ((rc = check_ptr(dy, "dy", true)) || (rc = check_ptr(quota, "quota", false, 4)) ||
      (rc = check_ptr(retained_offsets, "retained_offsets", false, 4)) ||
      (rc = check_ptr(retained_rows, "retained_rows", false, 4)) || (rc = check_ptr(scores, "scores", false, 4)))
    return rc;
  State s;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_state.find(ws);
    if (it == g_state.end() || !it->second.fwd_done)
      return fail(MOE_ERR_STATE, "moe_select_retained before moe_fwd on this workspace");
    if (!same_dims(it->second.d, *dims)) return fail(MOE_ERR_STATE, "dims differ from moe_fwd's");
    s = it->second;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const WsPtrs p = make_ptrs(L, ws);
  const int bf = dims->dtype == MOE_BF16;
  const int sms = num_sms_current();
  const int H = (int)L.H, F = (int)L.F, E = (int)L.E, k = (int)L.k;
  if (dims->flags & MOE_RECOMPUTE)  // scores and compaction read y_pair, a|b and h: re-derive them
    if ((rc = expert_forward_gemms(L, p, bf, sms, st, s.w_gate, s.w_up, s.w_down, s.ws_gate, s.ws_up, s.ws_down, s.x)))
      return rc;
  {
    Span sp(st, FAM_BW);
    if (bf)
      CKL(launch_pair_score<__nv_bfloat16>(dy, p.y_pair, p.pair_of_row, p.pad_off + E, L.Rmax, p.topk_w, p.xnorm, H, k,
                                          p.g, p.score, nullptr, scores, sms, st));
    else
      CKL(launch_pair_score<float>(dy, p.y_pair, p.pair_of_row, p.pad_off + E, L.Rmax, p.topk_w, p.xnorm, H, k, p.g,
                                  p.score, nullptr, scores, sms, st));
    CKL(launch_select(p.score, p.count, p.pad_off, quota, E, p.ret_cidx, p.ret_count, p.status, st));
    CKL(launch_ret_scan(p.ret_count, E, p.ret_offset, p.ret_pad_off, p.ret_tile_off, p.ret_src, retained_offsets, st,
                        p.ret_order, p.ret_tile_off2, p.ret_tile_rec, p.ret_ord_rec, p.ret_tile_rec2));
    CKL(launch_ret_index(p.topk_idx, p.rowp_of_pair, p.row_of_pair, p.ret_cidx, p.ret_offset, p.ret_pad_off, L.P,
                        p.ret_src, p.crow_of_pair, p.ret_rows, retained_rows, sms, st));
    if (bf)
      CKL(launch_compact_rows<__nv_bfloat16>(p.ret_src, p.ret_pad_off + E, L.Rmax, p.pair_of_row, p.topk_w, s.x, p.ab,
                                            p.h, dy, H, F, k, p.x_c, p.ab_c, p.h_c, p.dy_c, sms, st));
    else
      CKL(launch_compact_rows<float>(p.ret_src, p.ret_pad_off + E, L.Rmax, p.pair_of_row, p.topk_w, s.x, p.ab, p.h, dy,
                                    H, F, k, p.x_c, p.ab_c, p.h_c, p.dy_c, sms, st));
  }
  std::lock_guard<std::mutex> lk(g_mu);
  State& sr = g_state[ws];
  sr.sel_done = true;
  sr.sel_dy = dy;
  return MOE_OK;
}

int moe_bwd(const moe_dims* dims, void* ws, size_t ws_bytes, void* stream, const void* dy, const void* x,
            int use_retained, void* dx, void* dw_router, void* dw_gate, void* dw_up, void* dw_down, void* dws_gate,
            void* dws_up, void* dws_down) {
  WsLayout L;
  int rc = check_ws(dims, ws, ws_bytes, &L);
  if (rc) return rc;
  const bool frozen = dims->flags & MOE_FROZEN;
  const bool shared = dims->F_shared > 0;
  if ((rc = check_ptr(dy, "dy", true)) || (rc = check_ptr(x, "x", true)) || (rc = check_ptr(dx, "dx", true)))
    return rc;
  if (frozen) {
    if (dw_router || dw_gate || dw_up || dw_down || dws_gate || dws_up || dws_down)
      return fail(MOE_ERR_INVALID_ARG, "dW pointers must be null with MOE_FROZEN");
  } else {
    if ((rc = check_ptr(dw_router, "dw_router", true)) || (rc = check_ptr(dw_gate, "dw_gate", true)) ||
        (rc = check_ptr(dw_up, "dw_up", true)) || (rc = check_ptr(dw_down, "dw_down", true)))
      return rc;
    if (shared) {
      if ((rc = check_ptr(dws_gate, "dws_gate", true)) || (rc = check_ptr(dws_up, "dws_up", true)) ||
          (rc = check_ptr(dws_down, "dws_down", true)))
        return rc;
    } else if (dws_gate || dws_up || dws_down) {
      return fail(MOE_ERR_INVALID_ARG, "shared-expert gradients given but F_shared == 0");
    }
  }
  State s;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_state.find(ws);
    if (it == g_state.end() || !it->second.fwd_done) return fail(MOE_ERR_STATE, "moe_bwd before moe_fwd on this workspace");
    if (!same_dims(it->second.d, *dims)) return fail(MOE_ERR_STATE, "dims differ from moe_fwd's");
    if (it->second.x != x) return fail(MOE_ERR_STATE, "x differs from the tensor moe_fwd saw");
    if (use_retained && (!it->second.sel_done || it->second.sel_dy != dy))
      return fail(MOE_ERR_STATE, "use_retained needs moe_select_retained on the same dy first");
    s = it->second;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const WsPtrs p = make_ptrs(L, ws);
  const int bf = dims->dtype == MOE_BF16;
  const int sms = num_sms_current();
  const int T = (int)L.T, H = (int)L.H, F = (int)L.F, E = (int)L.E, k = (int)L.k, Fs = (int)L.Fs;

  // choose full or compact buffers
  const int* rows = p.count;
  const int* roff = p.pad_off;
  const int* toff = p.tile_off;
  const int* toff2 = p.tile_off2;
  const int4* trec = p.tile_rec;
  const int4* trec2 = p.tile_rec2;
  const void* xs = p.x_perm;
  const void* abs_ = p.ab;
  const void* hs = p.h;
  const void* dys = p.dy_perm;
  const int* crow = p.rowp_of_pair;
  if (use_retained) {
    rows = p.ret_count;
    roff = p.ret_pad_off;
    toff = p.ret_tile_off;
    trec = p.ret_tile_rec;
    trec2 = p.ret_tile_rec2;
    toff2 = p.ret_tile_off2;
    xs = p.x_c;
    abs_ = p.ab_c;
    hs = p.h_c;
    dys = p.dy_c;
    crow = p.crow_of_pair;
  }
  if ((dims->flags & MOE_RECOMPUTE) && !use_retained) {
    // the backward re-derives a|b, h and y_pair from the saved permuted rows (with
    // use_retained the selection already did, before it compacted them)
    if ((rc = expert_forward_gemms(L, p, bf, sms, st, s.w_gate, s.w_up, s.w_down, s.ws_gate, s.ws_up, s.ws_down, x)))
      return rc;
  }
  if (!use_retained) {
    // router-gradient dots g (and scores) over all pairs plus the w*dY rows;
    // with use_retained the selection already produced g for this dy
    Span sp(st, FAM_BW);
    if (bf)
      CKL(launch_pair_score<__nv_bfloat16>(dy, p.y_pair, p.pair_of_row, p.pad_off + E, L.Rmax, p.topk_w, p.xnorm, H, k,
                                          p.g, p.score, p.dy_perm, nullptr, sms, st));
    else
      CKL(launch_pair_score<float>(dy, p.y_pair, p.pair_of_row, p.pad_off + E, L.Rmax, p.topk_w, p.xnorm, H, k, p.g,
                                  p.score, p.dy_perm, nullptr, sms, st));
  }
  // dH = dy W_down^T with fused SwiGLU backward -> dAB
  {
    GemmArgs a = base_args(p.status);
    a.var_k = 0;
    a.G = E;
    a.rows = rows;
    a.row_off = roff;
    a.tile_off = toff;
    a.tile_rec = trec;
    a.tile_rec2 = trec2;
    a.tile_off2 = toff2;
    a.K = H;
    a.N = F;
    a.A = dys;
    a.lda = H;
    a.a_rows = L.Rmax;
    a.B0 = s.w_down;
    a.ldb = H;
    a.b_rows = L.E * L.F;
    a.b_kmajor = 1;
    a.epi = EPI_SWIGLU_BWD;
    a.aux = abs_;
    a.ld_aux = 2 * F;
    a.out0 = p.dab;
    a.ldo = 2 * F;
    a.zero_pad = 1;
    a.out_rows = L.Rmax;
    CKL(run_gemm(a, bf, 256, st, sms));
  }
  // dx_pair = [da | db] [W_gate ; W_up]^T
  {
    GemmArgs a = base_args(p.status);
    a.var_k = 0;
    a.G = E;
    a.rows = rows;
    a.row_off = roff;
    a.tile_off = toff;
    a.tile_rec = trec;
    a.tile_rec2 = trec2;
    a.tile_off2 = toff2;
    a.K = 2 * F;
    a.N = H;
    a.A = p.dab;
    a.lda = 2 * F;
    a.a_rows = L.Rmax;
    a.B0 = s.w_gate;
    a.B1 = s.w_up;
    a.ldb = F;
    a.b_rows = L.E * L.H;
    a.b_kmajor = 1;
    a.k_split = F;
    a.epi = EPI_STORE;
    a.out0 = p.dx_pair;
    a.ldo = H;
    a.zero_pad = 1;
    a.out_rows = L.Rmax;
    CKL(run_gemm(a, bf, 256, st, sms));
  }
  if (shared) {
    GemmArgs a = base_args(p.status);
    a.var_k = 0;
    a.G = 1;
    a.rows_const = T;
    a.K = H;
    a.N = Fs;
    a.A = dy;
    a.lda = H;
    a.a_rows = T;
    a.B0 = s.ws_down;
    a.ldb = H;
    a.b_rows = Fs;
    a.b_kmajor = 1;
    a.epi = EPI_SWIGLU_BWD;
    a.aux = p.sh_ab;
    a.ld_aux = 2 * Fs;
    a.out0 = p.sh_dab;
    a.ldo = 2 * Fs;
    a.zero_pad = 1;
    a.out_rows = L.Tpad;
    CKL(run_gemm(a, bf, 256, st, sms));
    GemmArgs b = base_args(p.status);
    b.var_k = 0;
    b.G = 1;
    b.rows_const = T;
    b.K = 2 * Fs;
    b.N = H;
    b.A = p.sh_dab;
    b.lda = 2 * Fs;
    b.a_rows = L.Tpad;
    b.B0 = s.ws_gate;
    b.B1 = s.ws_up;
    b.ldb = Fs;
    b.b_rows = H;
    b.b_kmajor = 1;
    b.k_split = Fs;
    b.epi = EPI_STORE;
    b.out0 = p.sh_dx;
    b.ldo = H;
    b.zero_pad = 1;
    b.out_rows = L.Tpad;
    CKL(run_gemm(b, bf, 256, st, sms));
  }
  // The router gradient and the dX reduce touch nothing the dW GEMMs read or write, so
  // they can run on the side stream beside the dW GEMMs. That pays while the dW GEMMs
  // leave HBM bandwidth and power to spare, i.e. while the dW gate/up GEMM at the mean
  // load of r = T k / E rows per expert sits below the ridge: r H 2F flops over
  // 2 (r H + r 2F + H 2F) bytes against 1.94 PFLOP/s / 6.78 TB/s = 287 flop/B (GB300,
  // bf16, measured). Kept on `st` while per-family timing is on, so that every span
  // brackets its own kernels.
  bool timing;
  {
    std::lock_guard<std::mutex> lk(g_timing.mu);
    timing = g_timing.on;
  }
  const double r_mean = (double)L.P / (double)L.E;
  const double dw_flop_per_byte = r_mean * (double)L.H * (2.0 * L.F) /
                                  (r_mean * ((double)L.H + 2.0 * L.F) + (double)L.H * (2.0 * L.F));
  const bool overlap = MOE_BWD_OVERLAP && !frozen && !timing && dw_flop_per_byte < 287.0;
  Side side;
  cudaStream_t bs = st;
  if (overlap) {
    CK(side_for(ws, &side));
    CK(cudaEventRecord(side.fork, st));
    CK(cudaStreamWaitEvent(side.s, side.fork, 0));
    bs = side.s;
  }
  {
    Span sp(bs, FAM_BW);
    if (bf) {
      CKL(launch_router_bwd<__nv_bfloat16>(p.g, p.rowp_of_pair, p.topk_idx, p.topk_w, T, (int)L.Tpad, E, k, p.dl_sel,
                                          frozen ? nullptr : p.dl, sms, bs));
      CKL(launch_transpose<__nv_bfloat16>(s.w_router, H, E, p.wrT, bs));
      CKL(launch_dx_reduce<__nv_bfloat16>(p.dx_pair, crow, p.topk_idx, p.dl_sel, p.wrT, shared ? p.sh_dx : nullptr, T,
                                         H, k, dx, sms, bs));
    } else {
      CKL(launch_router_bwd<float>(p.g, p.rowp_of_pair, p.topk_idx, p.topk_w, T, (int)L.Tpad, E, k, p.dl_sel,
                                  frozen ? nullptr : p.dl, sms, bs));
      CKL(launch_transpose<float>(s.w_router, H, E, p.wrT, bs));
      CKL(launch_dx_reduce<float>(p.dx_pair, crow, p.topk_idx, p.dl_sel, p.wrT, shared ? p.sh_dx : nullptr, T, H, k,
                                 dx, sms, bs));
    }
  }
  if (overlap) CK(cudaEventRecord(side.join, bs));
  if (!frozen) {
    // dW_gate[e] = x_e^T da_e, dW_up[e] = x_e^T db_e   (rows of the group are the reduction)
    {
      GemmArgs a = base_args(p.status);
      a.var_k = 1;
      a.G = E;
      a.rows = rows;
      a.row_off = roff;
      a.M = H;
      a.N = F;
      a.paired = 1;
      a.A = xs;
      a.lda = H;
      a.a_rows = L.Rmax;
      a.B0 = p.dab;
      a.B1 = p.dab;
      a.ldb = 2 * F;
      a.b_rows = L.Rmax;
      a.b1_col = F;
      a.epi = EPI_DW;
      a.out0 = dw_gate;
      a.out1 = dw_up;
      a.ldo = F;
      a.out_gstride = L.H * L.F;
      a.g_order = use_retained ? p.ret_order : p.order;
      a.grp_rec = use_retained ? p.ret_ord_rec : p.ord_rec;
      CKL(run_gemm(a, bf, 256, st, sms));
    }
    // dW_down[e] = h_e^T dy_e
    {
      GemmArgs a = base_args(p.status);
      a.var_k = 1;
      a.G = E;
      a.rows = rows;
      a.row_off = roff;
      a.M = F;
      a.N = H;
      a.A = hs;
      a.lda = F;
      a.a_rows = L.Rmax;
      a.B0 = dys;
      a.ldb = H;
      a.b_rows = L.Rmax;
      a.epi = EPI_DW;
      a.out0 = dw_down;
      a.ldo = H;
      a.out_gstride = L.F * L.H;
      a.g_order = use_retained ? p.ret_order : p.order;
      a.grp_rec = use_retained ? p.ret_ord_rec : p.ord_rec;
      CKL(run_gemm(a, bf, 256, st, sms));
    }
    // dW_router = x^T dl (dl from the router gradient: the side stream joins here)
    if (overlap) CK(cudaStreamWaitEvent(st, side.join, 0));
    {
      GemmArgs a = base_args(p.status);
      a.var_k = 1;
      a.G = 1;
      a.rows_const = T;
      a.M = H;
      a.N = E;
      a.A = x;
      a.lda = H;
      a.a_rows = T;
      a.B0 = p.dl;
      a.ldb = E;
      a.b_rows = L.Tpad;
      a.epi = EPI_DW;
      a.out0 = dw_router;
      a.ldo = E;
      const int ks = bf ? ksplit_for(L, ((L.H + 127) / 128) * ((L.E + 127) / 128), (T + kTileK - 1) / kTileK, sms,
                                     L.H * L.E)
                        : 1;
      if (ks > 1) {  // few tiles, long K (all tokens): K split, then an ordered sum into bf16
        a.epi = EPI_F32;
        a.out0 = p.part;
        a.ksplit = ks;
        a.part_stride = L.H * L.E;
        CKL(run_gemm(a, bf, 128, st, sms));
        Span sp(st, FAM_BW);
        CKL(launch_splitk_store(p.part, L.H * L.E, ks, nullptr, H, H, nullptr, E, E, dw_router, sms, st));
      } else {
        CKL(run_gemm(a, bf, 128, st, sms));
      }
    }
    if (shared) {
      GemmArgs a = base_args(p.status);
      a.var_k = 1;
      a.G = 1;
      a.rows_const = T;
      a.M = H;
      a.N = Fs;
      a.paired = 1;
      a.A = x;
      a.lda = H;
      a.a_rows = T;
      a.B0 = p.sh_dab;
      a.B1 = p.sh_dab;
      a.ldb = 2 * Fs;
      a.b_rows = L.Tpad;
      a.b1_col = Fs;
      a.epi = EPI_DW;
      a.out0 = dws_gate;
      a.out1 = dws_up;
      a.ldo = Fs;
      CKL(run_gemm(a, bf, 256, st, sms));
      GemmArgs b = base_args(p.status);
      b.var_k = 1;
      b.G = 1;
      b.rows_const = T;
      b.M = Fs;
      b.N = H;
      b.A = p.sh_h;
      b.lda = Fs;
      b.a_rows = L.Tpad;
      b.B0 = dy;
      b.ldb = H;
      b.b_rows = T;
      b.epi = EPI_DW;
      b.out0 = dws_down;
      b.ldo = H;
      CKL(run_gemm(b, bf, 256, st, sms));
    }
  }
  return MOE_OK;
}

}  // extern "C"
