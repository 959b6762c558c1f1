// a3: block topology + transpose metadata in a single kernel (George Lin's
// blog, MoE training post, section 1.3 "hybrid BCSR-COO format" and
// "transpose indices"; section 1.4: topology and transpose metadata are built
// by one kernel to avoid several launches).
//
// Every array entry has a closed form in the padded offsets, so each thread
// writes its entries independently (grid-stride loop, no synchronisation):
//   row block r lies in expert e(r) = the e with po[e] <= 128 r < po[e+1];
//   BCSR position q = r*nb + j holds column e(r)*nb + j;
//   in transposed order expert e's blocks fill the same range
//   [nb*rb_e, nb*rb_{e+1}) (rb_e = po[e]/128), column jj of the expert
//   holding its R_e rows consecutively.
// A few hundred KB of int32 writes: launch-latency bound.
#include "common.cuh"

namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ int expert_of_row(const int32_t* s_po, int E, int32_t row_elem) {
  // first e with s_po[e+1] > row_elem
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (s_po[mid + 1] > row_elem) hi = mid;
    else lo = mid + 1;
  }
  return lo;
}

__global__ void __launch_bounds__(kThreads)
    build_topology_kernel(const int32_t* __restrict__ padded_offsets, int E, int nb, int R_max, int nnz_max,
                          int32_t* __restrict__ row_offsets, int32_t* __restrict__ column_indices,
                          int32_t* __restrict__ row_indices, int32_t* __restrict__ column_offsets_t,
                          int32_t* __restrict__ row_indices_t, int32_t* __restrict__ block_offsets_t,
                          int32_t* __restrict__ nnz_dev, int32_t* __restrict__ P_dev) {
  extern __shared__ int32_t s_po[];  // [E+1]
  dmoe::pdl_wait();
  dmoe::pdl_launch_dependents();
  for (int e = threadIdx.x; e <= E; e += kThreads) s_po[e] = padded_offsets[e];
  __syncthreads();
  const int32_t P = s_po[E];
  const int32_t R = min(P / DMOE_BLOCK, R_max);
  const int32_t nnz = R * nb;
  const int32_t ncols = E * nb;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    *nnz_dev = nnz;
    *P_dev = P;
  }
  const int32_t n_items = max(max(nnz_max, R_max + 1), ncols + 1);
  for (int32_t i = blockIdx.x * kThreads + threadIdx.x; i < n_items; i += gridDim.x * kThreads) {
    if (i <= R_max) row_offsets[i] = min(i, R) * nb;
    if (i < nnz) {
      const int32_t r = i / nb;
      const int32_t j = i - r * nb;
      const int e = expert_of_row(s_po, E, r * DMOE_BLOCK);
      column_indices[i] = e * nb + j;
      row_indices[i] = r;
      // transposed entry i lies in the same expert's range
      const int32_t rb = s_po[e] / DMOE_BLOCK;
      const int32_t Re = s_po[e + 1] / DMOE_BLOCK - rb;
      const int32_t local = i - rb * nb;
      const int32_t jj = local / Re;
      const int32_t ii = local - jj * Re;
      row_indices_t[i] = rb + ii;
      block_offsets_t[i] = (rb + ii) * nb + jj;
    }
    if (i <= ncols) {
      if (i == ncols) {
        column_offsets_t[i] = nnz;
      } else {
        const int e = i / nb;
        const int32_t jj = i - e * nb;
        const int32_t rb = s_po[e] / DMOE_BLOCK;
        const int32_t Re = s_po[e + 1] / DMOE_BLOCK - rb;
        column_offsets_t[i] = rb * nb + jj * Re;
      }
    }
  }
}

}  // namespace

DMOE_API dmoe_status dmoe_build_topology(const int32_t* padded_offsets, const dmoe_topology* topo,
                                         dmoe_stream_t stream) {
  if (!padded_offsets || !topo) return DMOE_ERR_INVALID_ARG;
  const dmoe_topology& t = *topo;
  if (t.E < 1 || t.E > 1024 || t.F < DMOE_BLOCK || (t.F % DMOE_BLOCK) || t.P_max < 0 ||
      (t.P_max % DMOE_BLOCK))
    return DMOE_ERR_INVALID_ARG;
  const int nb = t.F / DMOE_BLOCK;
  const int64_t R_max = t.P_max / DMOE_BLOCK;
  if (static_cast<int64_t>(t.nnz_max) != R_max * nb || R_max * nb > 0x7fffffffLL ||
      static_cast<int64_t>(t.E) * nb > 0x7ffffffeLL)
    return DMOE_ERR_INVALID_ARG;
  if (!t.row_offsets || !t.column_offsets_t || !t.nnz_dev || !t.P_dev) return DMOE_ERR_INVALID_ARG;
  if (t.nnz_max > 0 && (!t.column_indices || !t.row_indices || !t.row_indices_t || !t.block_offsets_t))
    return DMOE_ERR_INVALID_ARG;
  dmoe::DeviceInfo di;
  dmoe_status s = dmoe::device_info(&di);
  if (s != DMOE_OK) return s;
  const int64_t n_items = std::max<int64_t>(std::max<int64_t>(t.nnz_max, R_max + 1), int64_t(t.E) * nb + 1);
  int blocks = static_cast<int>((n_items + kThreads - 1) / kThreads);
  blocks = std::min(blocks, di.sm_count * 8);
  cudaError_t e = dmoe::launch_pdl(build_topology_kernel, dim3(blocks), dim3(kThreads), (t.E + 1) * sizeof(int32_t),
                                   dmoe::as_stream(stream), padded_offsets, t.E, nb, static_cast<int>(R_max),
                                   t.nnz_max, t.row_offsets, t.column_indices, t.row_indices, t.column_offsets_t,
                                   t.row_indices_t, t.block_offsets_t, t.nnz_dev, t.P_dev);
  if (e != cudaSuccess) return dmoe::cuda_status(e);
  dmoe::count_launches(1);
  return DMOE_OK;
}
