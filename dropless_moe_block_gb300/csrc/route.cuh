// Top-k routing of one token by one warp (George Lin's blog, MoE training
// post, section 1.1: the gate assigns each token to experts).  Shared by the
// router kernel and the fused dispatch kernel.
#pragma once

#include <math.h>

#include "common.cuh"

namespace dmoe {

// a "better" than b: larger logit, or equal logit and lower expert id
__device__ __forceinline__ bool route_better(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// The whole warp routes the token whose E fp32 logits start at `row` (global
// or shared memory; E <= 32 * NPL; lane l holds experts l, l + 32, ...):
// softmax, then k rounds of warp arg-max.  Lane 0 writes out_i[j]
// (descending weight) and out_w[j]
// (the softmax probability, renormalised over the k chosen when renorm)
// and calls on_pick(e) once per chosen expert.  NaN logits count as -inf.
template <int NPL, class OnPick>
__device__ __forceinline__ void route_token(const float* __restrict__ row, int E, int k, int renorm,
                                            int32_t* __restrict__ out_i, float* __restrict__ out_w, int lane,
                                            OnPick on_pick) {
  float v[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = i * 32 + lane;
    const float x = e < E ? row[e] : -INFINITY;
    v[i] = isnan(x) ? -INFINITY : x;
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

  uint32_t taken = 0;
  float sel = 0.f;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const int e = i * 32 + lane;
      if (e < E && !((taken >> i) & 1u) && route_better(v[i], e, bv, bi)) {
        bv = v[i];
        bi = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (route_better(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    const float p = expf(bv - m) * inv_s;
    sel += p;
    if (lane == 0) {
      out_i[j] = bi;
      out_w[j] = p;
      on_pick(bi);
    }
  }
  if (renorm) {
    __syncwarp();
    const float inv = 1.f / sel;
    for (int j = lane; j < k; j += 32) out_w[j] *= inv;
  }
}

}  // namespace dmoe
