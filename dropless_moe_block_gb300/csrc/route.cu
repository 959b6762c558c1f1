// a1: top-k router (George Lin's blog, MoE training post, section 1.1: a gate
// network assigns each token to experts), and its backward: the gradient of
// the gate weights with respect to the logits.  One warp per token: the row
// of E logits sits in registers (E/32 per lane), softmax statistics and k
// rounds of warp arg-max run with shuffles.  Memory-bound: T*E*4 bytes read
// (and written, for the backward).
#include <math.h>

#include "route.cuh"

namespace {

constexpr int kWarpsPerBlock = 8;

template <int NPL>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    route_topk_kernel(const float* __restrict__ logits, int T, int E, int k, int renorm,
                      int32_t* __restrict__ expert_idx, float* __restrict__ gate_w) {
  dmoe::pdl_wait();
  dmoe::pdl_launch_dependents();
  const int t = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  dmoe::route_token<NPL>(logits + static_cast<int64_t>(t) * E, E, k, renorm, expert_idx + static_cast<int64_t>(t) * k,
                         gate_w + static_cast<int64_t>(t) * k, lane, [](int) {});
}

template <int NPL>
cudaError_t launch(const float* logits, int T, int E, int k, int renorm, int32_t* ei, float* gw,
                   cudaStream_t st) {
  const int blocks = (T + kWarpsPerBlock - 1) / kWarpsPerBlock;
  return dmoe::launch_pdl(route_topk_kernel<NPL>, dim3(blocks), dim3(kWarpsPerBlock * 32), 0, st, logits, T, E, k,
                          renorm, ei, gw);
}

// Gradient of the gate weights w.r.t. the logits (the chosen set is locally
// constant).  With c = sum_j d_gate[j] * gate_w[j] and G_e the d_gate of the
// slot holding expert e (0 if e was not chosen):
//   plain softmax weights:  d z_e = p_e (G_e - c)
//   renormalised weights:   d z_e = w_e (G_e - c) for chosen e, 0 otherwise
// (the renormalised weights are a softmax over the chosen logits alone).
template <int NPL>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    route_topk_backward_kernel(const float* __restrict__ logits, const int32_t* __restrict__ expert_idx,
                               const float* __restrict__ gate_w, const float* __restrict__ d_gate, int T, int E,
                               int k, int renorm, float* __restrict__ d_logits, int32_t* err) {
  dmoe::pdl_wait();
  dmoe::pdl_launch_dependents();
  const int t = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  const float* row = logits + static_cast<int64_t>(t) * E;
  float v[NPL], g[NPL], w[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = i * 32 + lane;
    const float x = e < E ? __ldg(row + e) : -INFINITY;
    v[i] = isnan(x) ? -INFINITY : x;
    g[i] = 0.f;
    w[i] = 0.f;
  }
  // slot values scattered to the lanes owning their experts; c on the side
  const int64_t a0 = static_cast<int64_t>(t) * k;
  float c = 0.f;
  for (int j = 0; j < k; ++j) {
    const int e = __ldg(expert_idx + a0 + j);
    const float gj = __ldg(d_gate + a0 + j);
    const float wj = __ldg(gate_w + a0 + j);
    c = fmaf(gj, wj, c);
    if (e < 0 || e >= E) {
      if (lane == 0) dmoe::raise_error(err, DMOE_SITE_ROUTE_INDEX | DMOE_ERR_DEVICE);
      continue;
    }
    if ((e & 31) == lane) {
#pragma unroll
      for (int i = 0; i < NPL; ++i)
        if (i == (e >> 5)) {
          g[i] = gj;
          w[i] = wj;
        }
    }
  }
  float* out = d_logits + static_cast<int64_t>(t) * E;
  if (renorm) {
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const int e = i * 32 + lane;
      if (e < E) out[e] = w[i] * (g[i] - c);
    }
    return;
  }
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < NPL; ++i) m = fmaxf(m, v[i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < NPL; ++i)
    if (i * 32 + lane < E) s += expf(v[i] - m);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  const float inv_s = 1.f / s;
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = i * 32 + lane;
    if (e < E) out[e] = expf(v[i] - m) * inv_s * (g[i] - c);
  }
}

template <int NPL>
cudaError_t launch_bwd(const float* logits, const int32_t* ei, const float* gw, const float* dg, int T, int E, int k,
                       int renorm, float* dl, int32_t* err, cudaStream_t st) {
  const int blocks = (T + kWarpsPerBlock - 1) / kWarpsPerBlock;
  return dmoe::launch_pdl(route_topk_backward_kernel<NPL>, dim3(blocks), dim3(kWarpsPerBlock * 32), 0, st, logits,
                          ei, gw, dg, T, E, k, renorm, dl, err);
}

}  // namespace

DMOE_API dmoe_status dmoe_route_topk(const float* logits, int T, int E, int k, int renormalize,
                                     int32_t* expert_idx, float* gate_w, dmoe_stream_t stream) {
  if (T < 0 || E < 1 || E > 1024 || k < 1 || k > E) return DMOE_ERR_INVALID_ARG;
  if (T == 0) return DMOE_OK;
  if (!logits || !expert_idx || !gate_w) return DMOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(logits) | reinterpret_cast<uintptr_t>(expert_idx) |
       reinterpret_cast<uintptr_t>(gate_w)) & 3u)
    return DMOE_ERR_INVALID_ARG;
  dmoe::DeviceInfo di;
  dmoe_status s = dmoe::device_info(&di);
  if (s != DMOE_OK) return s;
  cudaStream_t st = dmoe::as_stream(stream);
  const int r = renormalize ? 1 : 0;
  cudaError_t e;
  if (E <= 32) e = launch<1>(logits, T, E, k, r, expert_idx, gate_w, st);
  else if (E <= 64) e = launch<2>(logits, T, E, k, r, expert_idx, gate_w, st);
  else if (E <= 128) e = launch<4>(logits, T, E, k, r, expert_idx, gate_w, st);
  else if (E <= 256) e = launch<8>(logits, T, E, k, r, expert_idx, gate_w, st);
  else if (E <= 512) e = launch<16>(logits, T, E, k, r, expert_idx, gate_w, st);
  else e = launch<32>(logits, T, E, k, r, expert_idx, gate_w, st);
  if (e != cudaSuccess) return dmoe::cuda_status(e);
  dmoe::count_launches(1);
  return DMOE_OK;
}

DMOE_API dmoe_status dmoe_route_topk_backward(const float* logits, const int32_t* expert_idx, const float* gate_w,
                                              const float* d_gate, int T, int E, int k, int renormalize,
                                              float* d_logits, dmoe_stream_t stream) {
  if (T < 0 || E < 1 || E > 1024 || k < 1 || k > E) return DMOE_ERR_INVALID_ARG;
  if (T == 0) return DMOE_OK;
  if (!logits || !expert_idx || !gate_w || !d_gate || !d_logits) return DMOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(logits) | reinterpret_cast<uintptr_t>(expert_idx) |
       reinterpret_cast<uintptr_t>(gate_w) | reinterpret_cast<uintptr_t>(d_gate) |
       reinterpret_cast<uintptr_t>(d_logits)) & 3u)
    return DMOE_ERR_INVALID_ARG;
  dmoe::DeviceInfo di;
  dmoe_status s = dmoe::device_info(&di);
  if (s != DMOE_OK) return s;
  cudaStream_t st = dmoe::as_stream(stream);
  const int r = renormalize ? 1 : 0;
  cudaError_t e;
  if (E <= 32) e = launch_bwd<1>(logits, expert_idx, gate_w, d_gate, T, E, k, r, d_logits, di.err_word, st);
  else if (E <= 64) e = launch_bwd<2>(logits, expert_idx, gate_w, d_gate, T, E, k, r, d_logits, di.err_word, st);
  else if (E <= 128) e = launch_bwd<4>(logits, expert_idx, gate_w, d_gate, T, E, k, r, d_logits, di.err_word, st);
  else if (E <= 256) e = launch_bwd<8>(logits, expert_idx, gate_w, d_gate, T, E, k, r, d_logits, di.err_word, st);
  else if (E <= 512) e = launch_bwd<16>(logits, expert_idx, gate_w, d_gate, T, E, k, r, d_logits, di.err_word, st);
  else e = launch_bwd<32>(logits, expert_idx, gate_w, d_gate, T, E, k, r, d_logits, di.err_word, st);
  if (e != cudaSuccess) return dmoe::cuda_status(e);
  dmoe::count_launches(1);
  return DMOE_OK;
}
