// epilogue.cuh -- output stage shared by the tensor-core and SIMT grouped GEMMs.
//
// A thread hands over NV consecutive accumulator columns [n0, n0+NV) of one
// output row (plus the matching columns of the second half when paired) and
// the epilogue applies the GEMM's fused operation and stores the result.
#pragma once
#include "common.cuh"
#include "gemm.h"

namespace moe {

__device__ __forceinline__ int grp_rows(const GemmArgs& a, int g) { return a.rows ? a.rows[g] : a.rows_const; }
__device__ __forceinline__ int grp_off(const GemmArgs& a, int g) { return a.row_off ? a.row_off[g] : 0; }
__device__ __forceinline__ int round_pad(int r) { return (r + kPadRows - 1) / kPadRows * kPadRows; }

template <typename TIO, int NV>
__device__ __forceinline__ void store_vals(TIO* dst, const float* v, int nvalid) {
  if constexpr (sizeof(TIO) == 2 && NV % 8 == 0) {
    if (nvalid == NV && (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
#pragma unroll
      for (int i = 0; i < NV; i += 8) *reinterpret_cast<uint4*>(dst + i) = f_to_bf16x8(v + i);
      return;
    }
  }
#pragma unroll
  for (int i = 0; i < NV; ++i)
    if (i < nvalid) dst[i] = io<TIO>::cvt(v[i]);
}

template <typename TIO, int NV>
__device__ __forceinline__ void load_vals(const TIO* src, float* v, int nvalid) {
  if constexpr (sizeof(TIO) == 2 && NV % 8 == 0) {
    if (nvalid == NV && (reinterpret_cast<uintptr_t>(src) & 15) == 0) {
#pragma unroll
      for (int i = 0; i < NV; i += 8) bf16x8_to_f(*reinterpret_cast<const uint4*>(src + i), v + i);
      return;
    }
  }
#pragma unroll
  for (int i = 0; i < NV; ++i) v[i] = (i < nvalid) ? io<TIO>::ld(src + i) : 0.0f;
}

// m: row inside the group (var-M) or output row index (var-K).
template <typename TIO, int NV>
__device__ __forceinline__ void epilogue_apply(const GemmArgs& a, int g, int rows_g, int m, int n0, float* v0,
                                               float* v1) {
  const int nvalid = min(NV, a.N - n0);
  if (nvalid <= 0) return;
  if (!a.var_k) {
    const bool real = m < rows_g;
    if (!real) {
      if (!a.zero_pad || m >= round_pad(rows_g)) return;
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        v0[i] = 0.0f;
        if (v1) v1[i] = 0.0f;
      }
    }
    const int64_t gr = (int64_t)grp_off(a, g) + m;
    switch (a.epi) {
      case EPI_SWIGLU_FWD: {
        TIO* ab = reinterpret_cast<TIO*>(a.out0) + gr * a.ldo;
        TIO* hh = reinterpret_cast<TIO*>(a.out1) + gr * a.ldo1;
        float h[NV];
#pragma unroll
        for (int i = 0; i < NV; ++i) h[i] = v0[i] * sigmoidf_(v0[i]) * v1[i];
        store_vals<TIO, NV>(ab + n0, v0, nvalid);
        store_vals<TIO, NV>(ab + a.N + n0, v1, nvalid);
        store_vals<TIO, NV>(hh + n0, h, nvalid);
        break;
      }
      case EPI_STORE: {
        store_vals<TIO, NV>(reinterpret_cast<TIO*>(a.out0) + gr * a.ldo + n0, v0, nvalid);
        break;
      }
      case EPI_SWIGLU_BWD: {
        const TIO* ab = reinterpret_cast<const TIO*>(a.aux) + gr * a.ld_aux;
        float av[NV], bv[NV], da[NV], db[NV];
        load_vals<TIO, NV>(ab + n0, av, nvalid);
        load_vals<TIO, NV>(ab + a.N + n0, bv, nvalid);
#pragma unroll
        for (int i = 0; i < NV; ++i) {
          const float s = sigmoidf_(av[i]);
          da[i] = real ? v0[i] * bv[i] * s * (1.0f + av[i] * (1.0f - s)) : 0.0f;
          db[i] = real ? v0[i] * av[i] * s : 0.0f;
        }
        TIO* o = reinterpret_cast<TIO*>(a.out0) + gr * a.ldo;
        store_vals<TIO, NV>(o + n0, da, nvalid);
        store_vals<TIO, NV>(o + a.N + n0, db, nvalid);
        break;
      }
      case EPI_F32: {
        float* o = reinterpret_cast<float*>(a.out0) + gr * a.ldo + n0;
#pragma unroll
        for (int i = 0; i < NV; ++i)
          if (i < nvalid) o[i] = v0[i];
        break;
      }
      default:
        break;
    }
  } else {
    if (m >= a.M) return;
    const int64_t base = (int64_t)g * a.out_gstride + (int64_t)m * a.ldo + n0;
    store_vals<TIO, NV>(reinterpret_cast<TIO*>(a.out0) + base, v0, nvalid);
    if (a.paired) store_vals<TIO, NV>(reinterpret_cast<TIO*>(a.out1) + base, v1, nvalid);
  }
}

}  // namespace moe
