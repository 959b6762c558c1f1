// f1: the router's linear gate fused into top-k routing (George Lin's blog
// post on MoE training, section 1.1: a gate network sends each token to
// experts).
//
// One cluster of CS CTAs (CS = 1, 2 or 4) per tile of 64 tokens; CTA r of
// the cluster sums K slices [r nk / CS, (r + 1) nk / CS) of the d / 64 (64
// tokens per tile and the split over d both serve to fill the GPU: the
// product is small):
//   warp 0     TMA producer: 64-wide K slices of x (64 token rows) and of
//              w_gate (EP = E rounded up to a power of two >= 32 rows; rows
//              past E read as zeros) into a ring of 4-6 128B-swizzled stages
//   warp 1     TMEM allocator and single-thread tcgen05.mma issuer
//              (M = 64, N = EP, K = 16 per instruction, fp32 in TMEM; row m
//              of the accumulator sits in TMEM lane 32 (m / 16) + m % 16)
//   warps 2-5  TMEM -> shared memory: lanes 0-15 of warp q hold the partial
//              logits of tokens 16 q .. 16 q + 15 (in the freed ring)
//   all 14     after a cluster barrier, CTA r owns rows [r 64 / CS,
//              (r + 1) 64 / CS): it adds the CS partial tiles of its rows in
//              rank order through distributed shared memory, writes those
//              logits to global memory and routes those tokens, one warp per
//              token, with the routine dmoe_route_topk uses (the same result
//              for the same logits); a second cluster barrier keeps every
//              tile alive until all reads of it are done.
// Every mbarrier wait is bounded; on expiry the kernel records
// DMOE_SITE_GEMM_WAIT | DMOE_ERR_TIMEOUT, the cluster writes nothing, frees
// its TMEM and returns (every thread still passes both cluster barriers).
#include <algorithm>
#include <atomic>

#include "route.cuh"
#include "tc.cuh"
#include "tmap.cuh"

namespace {

using dmoe::tc::smem_u32;

constexpr int kTileT = 64;    // tokens per CTA (M = 64 MMAs)
constexpr int kSliceK = 64;   // K per stage (one 128-byte swizzle row)
constexpr int kWarpsG = 14;
constexpr int kThreadsG = 32 * kWarpsG;
constexpr uint32_t kSliceX = kTileT * kSliceK * 2;  // 8 KB

template <int NPL, int CS>
struct GatePlan {
  static constexpr int EP = 32 * NPL;  // MMA N and TMEM columns
  static constexpr uint32_t STAGE = kSliceX + EP * kSliceK * 2;
  // about 96 KB of ring (two CTAs per SM) where four stages fit in it
  static constexpr int FIT = static_cast<int>(96 * 1024 / STAGE);
  static constexpr int STAGES = FIT < 4 ? 4 : (FIT > 6 ? 6 : FIT);
  static constexpr int LD = EP + 1;  // logits tile row (floats, padded: conflict-free column writes)
  static constexpr int ROWS = kTileT / CS;  // rows each CTA of the cluster reduces and routes
  static constexpr size_t SMEM = 1024 + STAGES * STAGE + 256;
  static_assert(STAGE % 1024 == 0, "stages stay 1024-byte aligned");
  static_assert(kTileT * LD * 4 <= STAGES * STAGE, "the logits tile must fit in the operand ring");
};

template <int NPL, int CS>
__global__ void __launch_bounds__(kThreadsG, 1)
    gate_route_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w, int T,
                      int d, int E, int k, int renorm, float* __restrict__ logits, int32_t* __restrict__ expert_idx,
                      float* __restrict__ gate_w, int32_t* err) {
  using namespace dmoe::tc;
  using PL = GatePlan<NPL, CS>;
  constexpr uint32_t IDESC = idesc_bf16(kTileT, PL::EP, false, false);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + PL::STAGES * PL::STAGE);
  uint64_t* empty = full + PL::STAGES;
  uint64_t* tfull = empty + PL::STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tfull + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* tile = reinterpret_cast<float*>(smem);  // [kTileT][LD], once the MMAs are done

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = CS > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int t0 = (blockIdx.x / CS) * kTileT;
  const int nk = d / kSliceK;
  const int k0 = nk * rank / CS;        // this CTA's K slices
  const int k1 = nk * (rank + 1) / CS;
  if (threadIdx.x == 0) {
    for (int s = 0; s < PL::STAGES; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    mbar_init(tfull, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&map_x);
    tma_prefetch_map(&map_w);
  }
  if (warp == 1) tmem_alloc(tmem_slot, PL::EP);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  dmoe::pdl_wait();
  dmoe::pdl_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {
      uint32_t phase = 0;
      for (int i = k0, s = 0; i < k1; ++i) {
        if (!mbar_wait(empty + s, phase ^ 1u, abort_flag)) {
          dmoe::raise_error(err, DMOE_SITE_GEMM_WAIT | DMOE_ERR_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        uint8_t* sx = smem + s * PL::STAGE;
        mbar_arrive_expect_tx(full + s, PL::STAGE);
        tma_load_2d(sx, &map_x, full + s, i * kSliceK, t0);
        tma_load_2d(sx + kSliceX, &map_w, full + s, i * kSliceK, 0);
        if (++s == PL::STAGES) {
          s = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      uint32_t phase = 0;
      bool ok = true;
      for (int i = k0, s = 0; i < k1; ++i) {
        if (!mbar_wait(full + s, phase, abort_flag)) {
          ok = false;
          break;
        }
        fence_after_sync();
        const uint32_t sa = smem_u32(smem + s * PL::STAGE);
        const uint64_t adesc = sdesc_sw128(sa, 16, 1024);
        const uint64_t bdesc = sdesc_sw128(sa + kSliceX, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < kSliceK / 16; ++kk)
          mma_bf16(tmem, adesc + 2 * kk, bdesc + 2 * kk, IDESC, (i > k0 || kk > 0) ? 1u : 0u);
        mma_commit(empty + s);
        if (++s == PL::STAGES) {
          s = 0;
          phase ^= 1u;
        }
      }
      if (ok) {
        mma_commit(tfull);
      } else {
        dmoe::raise_error(err, DMOE_SITE_GEMM_WAIT | DMOE_ERR_TIMEOUT);
        *abort_flag = 1;
      }
    }
  } else if (warp < 6) {
    // TMEM lane quadrant q = warp % 4: lanes 0-15 hold tokens 16 q .. 16 q + 15
    const int quad = warp & 3;
    if (mbar_wait(tfull, 0, abort_flag)) {
      fence_after_sync();
      float* row = tile + (quad * 16 + (lane & 15)) * PL::LD;
#pragma unroll
      for (int c = 0; c < NPL; ++c) {
        float v[32];
        tmem_ld32(tmem + (static_cast<uint32_t>(quad * 32) << 16) + c * 32, v);
        tmem_ld_wait();
        if (lane < 16) {
#pragma unroll
          for (int j = 0; j < 32; ++j) row[c * 32 + j] = v[j];
        }
      }
    } else if (lane == 0) {
      dmoe::raise_error(err, DMOE_SITE_GEMM_WAIT | DMOE_ERR_TIMEOUT);
      *abort_flag = 1;
    }
  }
  fence_before_sync();
  // every partial tile (and abort flag) of the cluster is written
  if (CS > 1) cluster_sync();
  else __syncthreads();
  bool ok = *abort_flag == 0;
  if (CS > 1) {
    const uint32_t fa = smem_u32(const_cast<int*>(abort_flag));
#pragma unroll
    for (int q = 0; q < CS; ++q)
      if (q != rank) ok = ok && dsmem_ld_s32(dsmem_addr(fa, q)) == 0;
  }
  const int r0 = rank * PL::ROWS;  // this CTA's rows of the tile
  const int rows = min(PL::ROWS, T - t0 - r0);
  if (CS > 1 && ok) {
    // the CS partial sums of each logit of rows r0 .. r0 + rows - 1, added
    // in rank order into this CTA's tile (no other CTA reads these rows here)
    const uint32_t base = smem_u32(tile);
    for (int i = threadIdx.x; i < rows * E; i += kThreadsG) {
      const int r = r0 + i / E;
      const int e = i - (i / E) * E;
      const uint32_t off = static_cast<uint32_t>((r * PL::LD + e) * 4);
      float acc = 0.f;
#pragma unroll
      for (int q = 0; q < CS; ++q) acc += q == rank ? tile[r * PL::LD + e] : dsmem_ld_f32(dsmem_addr(base + off, q));
      tile[r * PL::LD + e] = acc;
    }
  }
  // no CTA of the cluster reads another's tile after this point
  if (CS > 1) cluster_sync();
  if (ok && rows > 0) {
    for (int i = threadIdx.x; i < rows * E; i += kThreadsG) {
      const int r = r0 + i / E;
      const int e = i - (i / E) * E;
      logits[static_cast<int64_t>(t0 + r) * E + e] = tile[r * PL::LD + e];
    }
    for (int r = r0 + warp; r < r0 + rows; r += kWarpsG) {
      const int64_t t = t0 + r;
      dmoe::route_token<NPL>(tile + r * PL::LD, E, k, renorm, expert_idx + t * k, gate_w + t * k, lane,
                             [](int) {});
    }
  }
  if (warp == 1) {
    fence_after_sync();
    tmem_dealloc(tmem, PL::EP);
  }
}

template <int NPL, int CS>
cudaError_t launch_gate(const CUtensorMap& mx, const CUtensorMap& mw, int T, int d, int E, int k, int renorm,
                        float* logits, int32_t* expert_idx, float* gate_w, const dmoe::DeviceInfo& di,
                        cudaStream_t st) {
  auto kern = gate_route_kernel<NPL, CS>;
  const size_t smem = GatePlan<NPL, CS>::SMEM;
  static std::atomic<uint64_t> opted{0};
  const uint64_t bit = di.device < 64 ? (uint64_t(1) << di.device) : 0;
  if (!bit || !(opted.load(std::memory_order_acquire) & bit)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    if (bit) opted.fetch_or(bit, std::memory_order_acq_rel);
  }
  const int tiles = (T + kTileT - 1) / kTileT;
  if (CS == 1)
    return dmoe::launch_pdl(kern, dim3(tiles), dim3(kThreadsG), smem, st, mx, mw, T, d, E, k, renorm, logits,
                            expert_idx, gate_w, di.err_word);
  return dmoe::launch_pdl_cluster(kern, dim3(tiles * CS), dim3(kThreadsG), smem, st, CS, mx, mw, T, d, E, k, renorm,
                                  logits, expert_idx, gate_w, di.err_word);
}

template <int NPL>
cudaError_t launch_gate_split(int cs, const CUtensorMap& mx, const CUtensorMap& mw, int T, int d, int E, int k,
                              int renorm, float* logits, int32_t* expert_idx, float* gate_w,
                              const dmoe::DeviceInfo& di, cudaStream_t st) {
  if (cs == 4) return launch_gate<NPL, 4>(mx, mw, T, d, E, k, renorm, logits, expert_idx, gate_w, di, st);
  if (cs == 2) return launch_gate<NPL, 2>(mx, mw, T, d, E, k, renorm, logits, expert_idx, gate_w, di, st);
  return launch_gate<NPL, 1>(mx, mw, T, d, E, k, renorm, logits, expert_idx, gate_w, di, st);
}

}  // namespace

DMOE_API dmoe_status dmoe_gate_route_topk(const uint16_t* x, const uint16_t* w_gate, int T, int d, int E, int k,
                                          int renormalize, float* logits, int32_t* expert_idx, float* gate_w,
                                          dmoe_stream_t stream) {
  if (T < 0 || d < kSliceK || (d % kSliceK) || E < 1 || E > 256 || k < 1 || k > E) return DMOE_ERR_INVALID_ARG;
  if (T == 0) return DMOE_OK;
  if (!x || !w_gate || !logits || !expert_idx || !gate_w) return DMOE_ERR_INVALID_ARG;
  if (!dmoe::aligned16(x) || !dmoe::aligned16(w_gate) ||
      ((reinterpret_cast<uintptr_t>(logits) | reinterpret_cast<uintptr_t>(expert_idx) |
        reinterpret_cast<uintptr_t>(gate_w)) & 3u))
    return DMOE_ERR_INVALID_ARG;
  dmoe::DeviceInfo di;
  dmoe_status s = dmoe::device_info(&di);
  if (s != DMOE_OK) return s;
  const int npl = E <= 32 ? 1 : E <= 64 ? 2 : E <= 128 ? 4 : 8;
  CUtensorMap mx, mw;
  if (!dmoe::make_map(&mx, x, static_cast<uint64_t>(T), static_cast<uint64_t>(d), kSliceK, kTileT) ||
      !dmoe::make_map(&mw, w_gate, static_cast<uint64_t>(E), static_cast<uint64_t>(d), kSliceK, 32 * npl))
    return DMOE_ERR_CUDA;
  cudaStream_t st = dmoe::as_stream(stream);
  const int r = renormalize ? 1 : 0;
  // split d over a cluster of 2 or 4 CTAs while the tiles alone leave SMs
  // idle and every CTA keeps at least two K slices
  const int tiles = (T + kTileT - 1) / kTileT;
  const int nk = d / kSliceK;
  int cs = 1;
  while (cs < 4 && static_cast<int64_t>(tiles) * cs < di.sm_count && nk >= 4 * cs) cs *= 2;
  cudaError_t e;
  switch (npl) {
    case 1: e = launch_gate_split<1>(cs, mx, mw, T, d, E, k, r, logits, expert_idx, gate_w, di, st); break;
    case 2: e = launch_gate_split<2>(cs, mx, mw, T, d, E, k, r, logits, expert_idx, gate_w, di, st); break;
    case 4: e = launch_gate_split<4>(cs, mx, mw, T, d, E, k, r, logits, expert_idx, gate_w, di, st); break;
    default: e = launch_gate_split<8>(cs, mx, mw, T, d, E, k, r, logits, expert_idx, gate_w, di, st); break;
  }
  if (e != cudaSuccess) return dmoe::cuda_status(e);
  dmoe::count_launches(1);
  return DMOE_OK;
}
