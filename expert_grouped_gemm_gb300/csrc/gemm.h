// gemm.h -- one description for every grouped GEMM of the MoE block.
//
// Two schedules:
//   variable M (var_k = 0): group g owns rows [row_off[g], row_off[g] + rows[g])
//     of a permuted activation buffer A[*, K]; D_g[m, n] = sum_k A[row_off[g]+m, k] * B_g[k, n].
//     Used for the expert forward (gate/up, down) and the backward dH and dX GEMMs.
//   variable K (var_k = 1): the group's rows are the reduction dimension;
//     D_g[m, n] = sum_{r < rows[g]} A[row_off[g]+r, m] * B[row_off[g]+r, n].
//     Used for the per-expert weight gradients X^T dH.
// Every permuted buffer stores each group padded to a multiple of 16 rows with
// zero rows, so a 16-row slice past a group's end contributes nothing.
#pragma once
#include <stdint.h>

namespace moe {

enum Epi : int {
  EPI_SWIGLU_FWD = 0,  // var-M, paired: out0 = ab [rows, 2N] (a | b), out1 = h = silu(a)*b [rows, N]
  EPI_STORE = 1,       // var-M: out0 [rows, ldo] in the I/O type
  EPI_SWIGLU_BWD = 2,  // var-M: acc = dh; aux = ab [rows, 2N]; out0 = dAB [rows, 2N] (da | db)
  EPI_DW = 3,          // var-K: out0 (+ out1 when paired) [G][M][ldo] in the I/O type
  EPI_F32 = 4,         // fp32 out0 [rows, ldo] (var-M rows of the group; var-K rows g*M + m); with a K
                       // split, split s writes out0 + s * part_stride and a reduce pass adds the splits
                       // in order; paired: the second half at column N
};

constexpr int kPadRows = 16;  // per-group row padding of permuted buffers
constexpr int kTileM = 128;   // tensor-core tile rows
constexpr int kTileK = 64;    // tensor-core k-block (one 128-byte swizzle row of bf16)
constexpr int kMaxSplit = 16; // largest K split of a tensor-core GEMM
constexpr int kSplitMaxSms = 256;  // the workspace holds K-split partials for GPUs of up to this many SMs

struct GemmArgs {
  // schedule
  int var_k;
  int G;
  const int* rows;      // [G] rows per group, or null: single group of rows_const rows
  const int* row_off;   // [G+1] padded row offsets (prefix), or null: 0
  const int* tile_off;  // [G+1] prefix of ceil(rows/128) per group (var-M), or null (single group)
  const int* tile_off2; // [G+1] prefix of ceil(rows/256) per group (var-M, two-CTA tiles), or null
  int rows_const;
  int M;                // var-K: output rows
  int N;                // output columns (per half when paired)
  int K;                // var-M: reduction length (multiple of 64)
  int paired;           // two B halves -> two accumulators per output element
  // operands; every operand is a row-major 2-D view [rows, ld] (elements)
  const void* A;
  int64_t lda, a_rows;
  const void* B0;
  const void* B1;
  int64_t ldb, b_rows;
  int b_kmajor;         // var-M: 1 -> B_g rows are (g*N + n) with k contiguous; 0 -> rows (g*K + k), n contiguous
  int b1_col;           // paired var-K: column offset of the second half in B1
  int k_split;          // var-M K-major: k in [0, k_split) reads B0, the rest B1 at k - k_split (0 = none)
  // epilogue
  int epi;
  void* out0;
  void* out1;
  int64_t ldo;          // out0 / out1 leading dim
  int64_t ldo1;         // out1 leading dim for EPI_SWIGLU_FWD (h)
  int64_t out_gstride;  // var-K: elements between groups
  const void* aux;
  int64_t ld_aux;
  int zero_pad;         // var-M: write zeros in rows [rows_g, round16(rows_g))
  int64_t out_rows;     // rows of the out0 / out1 2-D views (tensor-core stores are clipped there)
  const int* g_order;   // var-K: order in which groups are scheduled (heaviest first), or null
  // Tile records (read with one 16-byte load instead of a search): var-M, one per
  // 128-row block {group, first row within the group, rows, row offset}; var-K,
  // one per scheduled group {group, rows, row offset, 0}. Null: derive from the above.
  const int4* tile_rec;
  const int4* grp_rec;
  const int4* tile_rec2;  // var-M, CTA-pair tiles: one record per 256-row block, same fields as tile_rec
  // K split (tensor cores, EPI_F32 only): every tile's k-blocks are divided over ksplit
  // CTAs (0 or 1: none); a split without k-blocks writes zeros
  int ksplit;
  int64_t part_stride;  // elements between the fp32 outputs of consecutive splits
  int* status;
};

}  // namespace moe
