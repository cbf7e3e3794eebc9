// layout.h -- workspace layout of one MoE layer and the device pointers into it.
//
// Row-indexed activation buffers are "permuted": expert e owns padded rows
// [pad_off[e], pad_off[e+1]) where pad_off is the exclusive prefix of
// round_up(count[e], 16); the rows past count[e] are zero. Rmax = T*k + 15*E
// bounds every padded total. Shared-expert buffers hold Tpad = round_up(T, 16)
// rows (zero past T).
#pragma once
#include <stddef.h>
#include <stdint.h>

namespace moe {

struct WsPtrs {
  int* status;
  float* logits;        // [T,E] biased fp32 logits
  int* topk_idx;        // [T,k]
  float* topk_w;        // [T,k]
  float* xnorm;         // [T]
  uint64_t* masks;      // [C,E] per 64-token chunk: bit t of expert e = token t picked e
  int* chunk_base;      // [C,E] first padded row of chunk c's pairs of expert e
  int* count;           // [E]
  int* offset;          // [E+1] exact offsets
  int* pad_off;         // [E+1] padded offsets
  int* tile_off;        // [E+1] prefix of ceil(count/128)
  int* rowp_of_pair;    // [P] padded row of pair p
  int* row_of_pair;     // [P] exact row of pair p
  int* pair_of_row;     // [Rmax] pair of padded row (-1 for pad rows)
  void* x_perm;         // [Rmax,H]
  void* ab;             // [Rmax,2F]  a | b
  void* h;              // [Rmax,F]
  void* y_pair;         // [Rmax,H]
  void* sh_ab;          // [Tpad,2Fs]
  void* sh_h;           // [Tpad,Fs]
  void* sh_y;           // [Tpad,H]
  float* g;             // [Rmax] <dY_t, y_r> per padded row
  float* score;         // [Rmax]
  void* dy_perm;        // [Rmax,H] w * dY_t (all pairs)
  int* ret_cidx;        // [Rmax] index of a kept row inside its expert's kept list, -1 if dropped
  int* ret_count;       // [E]
  int* ret_offset;      // [E+1]
  int* ret_pad_off;     // [E+1]
  int* ret_tile_off;    // [E+1]
  int* ret_src;         // [Rmax] source padded row of compact row (-1 for pad rows)
  int* crow_of_pair;    // [P] compact row of pair p, -1 if dropped
  int* ret_rows;        // [P] exact kept rows, expert by expert
  void* x_c;            // [Rmax,H]   compact copies
  void* ab_c;           // [Rmax,2F]
  void* h_c;            // [Rmax,F]
  void* dy_c;           // [Rmax,H]
  void* dab;            // [Rmax,2F]  da | db
  void* dx_pair;        // [Rmax,H]
  void* dl;             // [Tpad,E] dense router logit gradient (I/O type)
  float* dl_sel;        // [T,k]
  void* wrT;            // [E,H] router weight transposed
  void* sh_dab;         // [Tpad,2Fs]
  void* sh_dx;          // [Tpad,H]
  int* order;           // [E] experts by count, descending (dW scheduling order)
  int* ret_order;       // [E] experts by kept count, descending
  int* tile_off2;       // [E+1] prefix of ceil(count/256) (two-CTA tiles)
  int* ret_tile_off2;   // [E+1] prefix of ceil(kept/256)
  int4* tile_rec;       // [P/128 + E] per 128-row block: {expert, first row in the group, count, pad_off}
  int4* ret_tile_rec;   // same for the kept rows
  int4* ord_rec;        // [E] experts in dW order: {expert, count, pad_off, 0}
  int4* ret_ord_rec;    // same for the kept rows
  float* part;          // fp32 partial sums of a K-split GEMM, split after split
  int4* tile_rec2;      // [P/256 + E] per 256-row block (CTA-pair tiles): {expert, first row, count, pad_off}
  int4* ret_tile_rec2;  // same for the kept rows
  void* decode;         // scratch of the fused decode forward (T <= 16 only; empty otherwise)
};

struct WsLayout {
  int64_t T, H, F, E, k, Fs, P, Rmax, Tpad, C;
  int64_t Rdec;        // padded permuted rows actually used: T*k + 15*min(E, T*k)
  int64_t part_elems;  // fp32 elements of the K-split partial buffer (0: no split possible)
  int es;  // bytes per I/O element
  size_t total;
  size_t off[64];
  int n;
};

}  // namespace moe
