// a3: block topology + transpose metadata in a single kernel (George Lin's
// blog, MoE training post, section 1.3 "hybrid BCSR-COO format" and
// "transpose indices"; section 1.4: topology and transpose metadata are built
// by one kernel to avoid several launches).  Every entry has a closed form in
// the padded offsets (topology.cuh), so each thread writes its entries
// independently (grid-stride loop, no synchronisation).  A few hundred KB of
// int32 writes: launch-latency bound.
#include "topology.cuh"

namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
    build_topology_kernel(const int32_t* __restrict__ padded_offsets, const int32_t* __restrict__ tokens_per_expert,
                          int E, int B, int nb, int R_max, int nnz_max, int32_t* __restrict__ row_fill,
                          int32_t* __restrict__ row_offsets, int32_t* __restrict__ column_indices,
                          int32_t* __restrict__ row_indices, int32_t* __restrict__ column_offsets_t,
                          int32_t* __restrict__ row_indices_t, int32_t* __restrict__ block_offsets_t,
                          int32_t* __restrict__ nnz_dev, int32_t* __restrict__ P_dev) {
  extern __shared__ int32_t s_po[];  // [E+1] padded offsets, then [E] tokens per expert
  int32_t* s_tpe = s_po + E + 1;
  dmoe::pdl_wait();
  dmoe::pdl_launch_dependents();
  for (int e = threadIdx.x; e <= E; e += kThreads) s_po[e] = padded_offsets[e];
  if (tokens_per_expert)
    for (int e = threadIdx.x; e < E; e += kThreads) s_tpe[e] = tokens_per_expert[e];
  __syncthreads();
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    const int32_t P = s_po[E];
    *nnz_dev = min(P / B, R_max) * nb;
    *P_dev = P;
  }
  dmoe::topology_entries(s_po, tokens_per_expert ? s_tpe : nullptr, E, B, nb, R_max, nnz_max, row_fill, row_offsets,
                         column_indices, row_indices, column_offsets_t,
                         row_indices_t, block_offsets_t, static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x,
                         static_cast<int64_t>(gridDim.x) * kThreads);
}

}  // namespace

DMOE_API dmoe_status dmoe_build_topology(const int32_t* padded_offsets, const int32_t* tokens_per_expert,
                                         const dmoe_topology* topo, dmoe_stream_t stream) {
  if (!padded_offsets || !topo) return DMOE_ERR_INVALID_ARG;
  const dmoe_topology& t = *topo;
  const int B = t.block ? t.block : DMOE_BLOCK;
  if (B != 64 && B != 128 && B != 256) return DMOE_ERR_INVALID_ARG;
  if (t.E < 1 || t.E > 1024 || t.F < B || (t.F % B) || (t.F % DMOE_BLOCK) || t.P_max < 0 || (t.P_max % B))
    return DMOE_ERR_INVALID_ARG;
  const int nb = t.F / B;
  const int64_t R_max = t.P_max / B;
  if (static_cast<int64_t>(t.nnz_max) != R_max * nb || R_max * nb > 0x7fffffffLL ||
      static_cast<int64_t>(t.E) * nb > 0x7ffffffeLL)
    return DMOE_ERR_INVALID_ARG;
  if (!t.row_offsets || !t.column_offsets_t || !t.nnz_dev || !t.P_dev) return DMOE_ERR_INVALID_ARG;
  if (t.nnz_max > 0 && (!t.column_indices || !t.row_indices || !t.row_indices_t || !t.block_offsets_t))
    return DMOE_ERR_INVALID_ARG;
  dmoe::DeviceInfo di;
  dmoe_status s = dmoe::device_info(&di);
  if (s != DMOE_OK) return s;
  const int64_t n_items = dmoe::topology_items(t.E, nb, static_cast<int>(R_max), t.nnz_max);
  int blocks = static_cast<int>((n_items + kThreads - 1) / kThreads);
  blocks = std::min(blocks, di.sm_count * 8);
  cudaError_t e = dmoe::launch_pdl(build_topology_kernel, dim3(blocks), dim3(kThreads),
                                   (2 * t.E + 1) * sizeof(int32_t), dmoe::as_stream(stream), padded_offsets,
                                   tokens_per_expert, t.E, B, nb, static_cast<int>(R_max), t.nnz_max, t.row_fill,
                                   t.row_offsets, t.column_indices, t.row_indices, t.column_offsets_t,
                                   t.row_indices_t, t.block_offsets_t, t.nnz_dev, t.P_dev);
  if (e != cudaSuccess) return dmoe::cuda_status(e);
  dmoe::count_launches(1);
  return DMOE_OK;
}
