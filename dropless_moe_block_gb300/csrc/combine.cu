// a6/a11: un-permute + top-k weighted combine, and a7: its backward.
// The inverse of the permutation of section 1.4 of George Lin's blog post on
// MoE training: rows return from expert-grouped order to batch order and the
// k expert outputs of each token are summed with their gate weights.
// Both kernels are HBM-bound row gathers/scatters with 16-byte vectors, one
// warp per output row.
#include <cuda_bf16.h>

#include "common.cuh"

namespace {

constexpr int kWarps = 8;

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float (&f)[8]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 p = __bfloat1622float2(h[i]);
    f[2 * i] = p.x;
    f[2 * i + 1] = p.y;
  }
}

__device__ __forceinline__ uint4 f32_to_bf16x8(const float (&f)[8]) {
  uint4 u;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  return u;
}

// One warp per token.  KMAX > 0: the token's k <= KMAX source rows and gate
// weights are read and checked once, then every 16-byte column chunk issues
// its k row loads together (two chunks per loop trip); KMAX = 0 serves any k
// with the per-slot loop.  Either way the fp32 sum runs in slot order.
template <int KMAX>
__global__ void __launch_bounds__(kWarps * 32)
    unpermute_combine_kernel(const uint16_t* __restrict__ y_perm, int n_rows, const int32_t* __restrict__ dest_row,
                             const float* __restrict__ gate_w, int T, int d, int k, uint16_t* __restrict__ y,
                             int32_t* err) {
  dmoe::pdl_wait();
  dmoe::pdl_launch_dependents();
  const int t = blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  const int nvec = d >> 3;
  const uint4* src = reinterpret_cast<const uint4*>(y_perm);
  uint4* dst = reinterpret_cast<uint4*>(y) + static_cast<int64_t>(t) * nvec;
  const int64_t a0 = static_cast<int64_t>(t) * k;
  if constexpr (KMAX > 0) {
    int64_t off[KMAX > 0 ? KMAX : 1];
    float w[KMAX > 0 ? KMAX : 1];
    bool ok[KMAX > 0 ? KMAX : 1];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      ok[j] = false;
      off[j] = 0;
      w[j] = 0.f;
      if (j < k) {
        const int32_t p = __ldg(dest_row + a0 + j);
        if (p < 0 || p >= n_rows) {
          if (lane == 0) dmoe::raise_error(err, DMOE_SITE_COMBINE_INDEX | DMOE_ERR_DEVICE);
        } else {
          ok[j] = true;
          off[j] = static_cast<int64_t>(p) * nvec;
          w[j] = gate_w ? __ldg(gate_w + a0 + j) : 1.f;
        }
      }
    }
#pragma unroll 2
    for (int v = lane; v < nvec; v += 32) {
      uint4 u[KMAX > 0 ? KMAX : 1];
#pragma unroll
      for (int j = 0; j < KMAX; ++j)
        if (ok[j]) u[j] = __ldg(src + off[j] + v);
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        if (!ok[j]) continue;
        float f[8];
        bf16x8_to_f32(u[j], f);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = fmaf(w[j], f[i], acc[i]);
      }
      dst[v] = f32_to_bf16x8(acc);
    }
  } else {
#pragma unroll 2
    for (int v = lane; v < nvec; v += 32) {
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
      for (int j = 0; j < k; ++j) {
        const int32_t p = __ldg(dest_row + a0 + j);
        if (p < 0 || p >= n_rows) {
          if (v == lane) dmoe::raise_error(err, DMOE_SITE_COMBINE_INDEX | DMOE_ERR_DEVICE);
          continue;
        }
        const float w = gate_w ? __ldg(gate_w + a0 + j) : 1.f;
        float f[8];
        bf16x8_to_f32(__ldg(src + static_cast<int64_t>(p) * nvec + v), f);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = fmaf(w, f[i], acc[i]);
      }
      dst[v] = f32_to_bf16x8(acc);
    }
  }
}

__global__ void __launch_bounds__(kWarps * 32)
    combine_backward_kernel(const uint16_t* __restrict__ dy, const uint16_t* __restrict__ y_perm,
                            const int32_t* __restrict__ src_of_row, const float* __restrict__ gate_w,
                            const int32_t* __restrict__ P_dev, int d, int k, int P_max, int64_t A,
                            uint16_t* __restrict__ dy_perm, float* __restrict__ d_gate, int32_t* err) {
  dmoe::pdl_wait();
  dmoe::pdl_launch_dependents();
  const int p = blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (p >= P_max || p >= __ldg(P_dev)) return;
  const int nvec = d >> 3;
  uint4* out = reinterpret_cast<uint4*>(dy_perm) + static_cast<int64_t>(p) * nvec;
  const int32_t a = __ldg(src_of_row + p);
  if (a >= A) {
    if (lane == 0) dmoe::raise_error(err, DMOE_SITE_COMBINE_INDEX | DMOE_ERR_DEVICE);
  }
  if (a < 0 || a >= A) {
    for (int v = lane; v < nvec; v += 32) out[v] = make_uint4(0, 0, 0, 0);
    return;
  }
  const int64_t t = a / k;
  const float w = gate_w ? __ldg(gate_w + a) : 1.f;
  const uint4* g = reinterpret_cast<const uint4*>(dy) + t * nvec;
  const uint4* yp = y_perm ? reinterpret_cast<const uint4*>(y_perm) + static_cast<int64_t>(p) * nvec : nullptr;
  float dot = 0.f;
#pragma unroll 4
  for (int v = lane; v < nvec; v += 32) {
    float f[8];
    bf16x8_to_f32(__ldg(g + v), f);
    if (d_gate) {
      float q[8];
      bf16x8_to_f32(__ldg(yp + v), q);
#pragma unroll
      for (int i = 0; i < 8; ++i) dot = fmaf(f[i], q[i], dot);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) f[i] *= w;
    out[v] = f32_to_bf16x8(f);
  }
  if (d_gate) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
    if (lane == 0) d_gate[a] = dot;
  }
}

}  // namespace

DMOE_API dmoe_status dmoe_unpermute_combine(const uint16_t* y_perm, int n_rows, const int32_t* dest_row,
                                            const float* gate_w, int T, int d, int k, uint16_t* y,
                                            dmoe_stream_t stream) {
  if (T < 0 || d < 8 || (d & 7) || k < 1 || n_rows < 0) return DMOE_ERR_INVALID_ARG;
  if (T == 0) return DMOE_OK;
  if (!y_perm || !dest_row || !y) return DMOE_ERR_INVALID_ARG;
  if (!dmoe::aligned16(y_perm) || !dmoe::aligned16(y) || (reinterpret_cast<uintptr_t>(dest_row) & 3) ||
      (reinterpret_cast<uintptr_t>(gate_w) & 3))
    return DMOE_ERR_INVALID_ARG;
  dmoe::DeviceInfo di;
  dmoe_status s = dmoe::device_info(&di);
  if (s != DMOE_OK) return s;
  const int blocks = (T + kWarps - 1) / kWarps;
  auto kern = k <= 1 ? unpermute_combine_kernel<1>
            : k <= 2 ? unpermute_combine_kernel<2>
            : k <= 4 ? unpermute_combine_kernel<4>
            : k <= 8 ? unpermute_combine_kernel<8>
                     : unpermute_combine_kernel<0>;
  cudaError_t e = dmoe::launch_pdl(kern, dim3(blocks), dim3(kWarps * 32), 0, dmoe::as_stream(stream), y_perm,
                                   n_rows, dest_row, gate_w, T, d, k, y, di.err_word);
  if (e != cudaSuccess) return dmoe::cuda_status(e);
  dmoe::count_launches(1);
  return DMOE_OK;
}

DMOE_API dmoe_status dmoe_combine_backward(const uint16_t* dy, const uint16_t* y_perm, const int32_t* src_of_row,
                                           const float* gate_w, const int32_t* P_dev, int T, int d, int k,
                                           int P_max, uint16_t* dy_perm, float* d_gate, dmoe_stream_t stream) {
  if (T < 0 || d < 8 || (d & 7) || k < 1 || P_max < 0 || (P_max % 64)) return DMOE_ERR_INVALID_ARG;
  if (P_max == 0) return DMOE_OK;
  if (!src_of_row || !P_dev || !dy_perm || (T > 0 && !dy)) return DMOE_ERR_INVALID_ARG;
  if (d_gate && !y_perm) return DMOE_ERR_INVALID_ARG;
  if (!dmoe::aligned16(dy) || !dmoe::aligned16(y_perm) || !dmoe::aligned16(dy_perm) ||
      (reinterpret_cast<uintptr_t>(gate_w) & 3) || (reinterpret_cast<uintptr_t>(d_gate) & 3))
    return DMOE_ERR_INVALID_ARG;
  dmoe::DeviceInfo di;
  dmoe_status s = dmoe::device_info(&di);
  if (s != DMOE_OK) return s;
  const int blocks = (P_max + kWarps - 1) / kWarps;
  cudaError_t e = dmoe::launch_pdl(combine_backward_kernel, dim3(blocks), dim3(kWarps * 32), 0,
                                   dmoe::as_stream(stream), dy, y_perm, src_of_row, gate_w, P_dev, d, k, P_max,
                                   static_cast<int64_t>(T) * k, dy_perm, d_gate, di.err_word);
  if (e != cudaSuccess) return dmoe::cuda_status(e);
  dmoe::count_launches(1);
  return DMOE_OK;
}
