// Closed forms of the block topology (George Lin's blog, MoE training post,
// section 1.3 "hybrid BCSR-COO format" and "transpose indices").  Shared by
// the topology kernel and the fused dispatch kernel.
//
// Every array entry is a function of the padded offsets po[0..E] and the
// block edge B (128, or 64 / 256 for the block-size ablation) alone:
//   row block r lies in expert e(r) = the e with po[e] <= B r < po[e+1];
//   BCSR position q = r*nb + j holds column e(r)*nb + j;
//   in transposed order expert e's blocks fill the same range
//   [nb*rb_e, nb*rb_{e+1}) (rb_e = po[e]/B), column jj of the expert
//   holding its R_e rows consecutively.
#pragma once

#include "common.cuh"

namespace dmoe {

__device__ __forceinline__ int topo_expert_of_row(const int32_t* po, int E, int32_t row_elem) {
  // first e with po[e+1] > row_elem
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (po[mid + 1] > row_elem) hi = mid;
    else lo = mid + 1;
  }
  return lo;
}

// Number of entries topology_entries() walks (the longest array).
__host__ __device__ inline int64_t topology_items(int E, int nb, int R_max, int nnz_max) {
  const int64_t a = nnz_max, b = static_cast<int64_t>(R_max) + 1, c = static_cast<int64_t>(E) * nb + 1;
  return a > b ? (a > c ? a : c) : (b > c ? b : c);
}

// Writes entries i0, i0 + stride, ... of every topology array from po (any
// memory the caller can read; shared memory in both kernels).  R_max =
// P_max / B and nnz_max = R_max * nb size the arrays; entries past the
// current P are filled so that row_offsets stays non-decreasing.  With tpe
// (T_e per expert) and row_fill non-null, row_fill[r] = the rows of row
// block r that hold tokens: min(B, T_e - (B r - po[e])), 0 past P.
__device__ __forceinline__ void topology_entries(const int32_t* po, const int32_t* tpe, int E, int B, int nb,
                                                 int R_max, int nnz_max, int32_t* __restrict__ row_fill,
                                                 int32_t* __restrict__ row_offsets,
                                                 int32_t* __restrict__ column_indices,
                                                 int32_t* __restrict__ row_indices,
                                                 int32_t* __restrict__ column_offsets_t,
                                                 int32_t* __restrict__ row_indices_t,
                                                 int32_t* __restrict__ block_offsets_t, int64_t i0, int64_t stride) {
  const int32_t P = po[E];
  const int32_t R = min(P / B, R_max);
  const int32_t nnz = R * nb;
  const int32_t ncols = E * nb;
  const int64_t n_items = topology_items(E, nb, R_max, nnz_max);
  for (int64_t ii = i0; ii < n_items; ii += stride) {
    const int32_t i = static_cast<int32_t>(ii);
    if (i <= R_max) row_offsets[i] = min(i, R) * nb;
    if (row_fill && tpe && i < R_max) {
      int32_t f = 0;
      if (i < R) {
        const int e = topo_expert_of_row(po, E, i * B);
        f = min(B, tpe[e] - (i * B - po[e]));
      }
      row_fill[i] = f;
    }
    if (i < nnz) {
      const int32_t r = i / nb;
      const int32_t j = i - r * nb;
      const int e = topo_expert_of_row(po, E, r * B);
      column_indices[i] = e * nb + j;
      row_indices[i] = r;
      // transposed entry i lies in the same expert's range
      const int32_t rb = po[e] / B;
      const int32_t Re = po[e + 1] / B - rb;
      const int32_t local = i - rb * nb;
      const int32_t jj = local / Re;
      const int32_t r_in = local - jj * Re;
      row_indices_t[i] = rb + r_in;
      block_offsets_t[i] = (rb + r_in) * nb + jj;
    }
    if (i <= ncols) {
      if (i == ncols) {
        column_offsets_t[i] = nnz;
      } else {
        const int e = i / nb;
        const int32_t jj = i - e * nb;
        const int32_t rb = po[e] / B;
        const int32_t Re = po[e + 1] / B - rb;
        column_offsets_t[i] = rb * nb + jj * Re;
      }
    }
  }
}

}  // namespace dmoe
