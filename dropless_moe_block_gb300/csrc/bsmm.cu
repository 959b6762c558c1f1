// a4/a8 SDD, a5 DSD, a10 DSD^T and a9 DSTD: the block-sparse products of
// George Lin's blog post on MoE training, section 1.2 (the expert MLP as
// SDD -> activation -> DSD) and section 1.3 (128x128 blocks, BCSR row walk,
// transpose index for the weight gradient).
//
// One persistent, warp-specialised tcgen05 kernel template serves all four:
//   warp 0      TMA producer (whole warp): the lanes fetch up to 32 block
//               indices of the topology at once, lane 0 issues the TMA loads
//               of 64-wide K slices of A and B into a ring of 128B-swizzled
//               shared-memory stages (mbarrier complete_tx), and, for the
//               backward SDD, the stored forward blocks the epilogue needs
//   warp 1      TMEM allocator + single-thread tcgen05.mma issuer
//               (M=128, N=128, K=16 per instruction, fp32 accumulator)
//   warps 2-5   epilogue: tcgen05.ld of the accumulator, fused activation /
//               activation gradient, bf16 stores
// Each output tile is one 128x128 block (SDD) or one 128x128 tile of a dense
// output; two TMEM accumulators per CTA let the epilogue of tile i overlap the
// MMAs of tile i+1.  Tiles are assigned round-robin over a grid of one CTA
// per SM; every role decodes its next tile while it works on the current one.
// Every mbarrier wait is bounded (kWaitLimitNs); on expiry the kernel records
// DMOE_SITE_GEMM_WAIT | DMOE_ERR_TIMEOUT, stops all roles, frees its TMEM and
// returns.
//
// Operand majors (a "K-major" tile has K contiguous; "MN-major" has M or N
// contiguous), with Sb the [nnz,128,128] block array:
//   SDD  (b_trans=0): A = X [P,K] K-major,   B = W [K,E*F] MN-major
//   SDD  (b_trans=1): A = X [P,K] K-major,   B = W [E*F,K] K-major
//   DSD             : A = Sb K-major,        B = W [E*F,N] MN-major
//   DSD^T           : A = Sb K-major,        B = W [N,E*F] K-major
//   DSTD (c_trans=0): A = Sb^T MN-major,     B = D [P,N]  MN-major
//   DSTD (c_trans=1): A = D^T MN-major,      B = Sb       MN-major
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <math.h>

#include <atomic>
#include <mutex>

#include "tc.cuh"

namespace {

using dmoe::tc::smem_u32;

enum Op : int { OP_SDD = 0, OP_DSD = 1, OP_DSDT = 2, OP_DSTD = 3, OP_DSTDT = 4 };

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int BK = 64;
constexpr int UMMA_K = 16;
constexpr uint32_t TILE_BYTES = BM * BK * 2;  // 16 KB: one 128 x 64 bf16 operand slice
constexpr uint32_t HALF_BYTES = TILE_BYTES / 2;
constexpr uint32_t BLOCK_BYTES = BM * BN * 2;  // 32 KB: one 128 x 128 bf16 block
constexpr int kEpiWarps = 8;  // two per TMEM lane quadrant, 64 columns each
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr size_t kSmemLimit = 232448;  // opt-in dynamic shared memory per CTA
constexpr size_t kSmemReserve = 1024 + 512;

struct Params {
  CUtensorMap map_a;
  CUtensorMap map_b;
  CUtensorMap map_a2;
  CUtensorMap map_b2;
  CUtensorMap map_aux0;
  const int32_t* row_offsets;
  const int32_t* column_indices;
  const int32_t* row_indices;
  const int32_t* column_offsets_t;
  const int32_t* row_indices_t;
  const int32_t* block_offsets_t;
  const int32_t* nnz_dev;
  const int32_t* P_dev;
  int nb;         // F / 128
  int K;          // SDD reduction length
  int N;          // dense width (DSD, DSD^T, DSTD)
  int EF;         // E * F
  int ntn;        // tiles along N
  int max_tiles;  // host bound on the tile count
  int second;  // DSD^T: a second (S2, B2) pair accumulates into the same tile
  uint16_t* out0;
  uint16_t* out1;
  uint16_t* out2;
  const uint16_t* aux0;  // stored forward blocks read by the SwiGLU' epilogue
  const uint16_t* aux1;
  int32_t* err;
};

struct Tile {
  int kiters;  // 64-wide K slices
  int a, b, c;  // op-specific coordinates
  int nblk;     // blocks walked along K (DSD / DSD^T / DSTD)
};

template <int OP>
__device__ __forceinline__ int num_tiles(const Params& p) {
  int n;
  if (OP == OP_SDD) n = __ldg(p.nnz_dev);
  else if (OP == OP_DSD || OP == OP_DSDT) n = (__ldg(p.P_dev) / BM) * p.ntn;
  else n = (p.EF / BM) * p.ntn;
  return n < p.max_tiles ? (n > 0 ? n : 0) : p.max_tiles;
}

template <int OP>
__device__ __forceinline__ Tile decode(const Params& p, int t) {
  Tile tl;
  if (OP == OP_SDD) {
    tl.a = t;                            // block q
    tl.b = __ldg(p.row_indices + t);     // row block r
    tl.c = __ldg(p.column_indices + t);  // column block c
    tl.kiters = p.K / BK;
    tl.nblk = 0;
  } else if (OP == OP_DSD || OP == OP_DSDT) {
    const int r = t / p.ntn;
    const int q0 = __ldg(p.row_offsets + r);
    const int n = __ldg(p.row_offsets + r + 1) - q0;
    tl.a = r;
    tl.b = t - r * p.ntn;  // n tile
    tl.c = q0;
    tl.nblk = n;
    tl.kiters = n * (BM / BK) * (p.second ? 2 : 1);
  } else {
    const int c = t / p.ntn;
    const int j0 = __ldg(p.column_offsets_t + c);
    const int n = __ldg(p.column_offsets_t + c + 1) - j0;
    tl.a = c;
    tl.b = t - c * p.ntn;  // n tile (DSTD) / m tile (DSTD^T)
    tl.c = j0;
    tl.nblk = n;
    tl.kiters = n * (BM / BK);
  }
  return tl;
}

// TMA loads of one K slice.  For the block-walking ops, v0 / v1 are the
// per-block topology values (DSD, DSD^T: column block; DSTD: BCSR position
// and row block), blk the BCSR position, half the 64-row half of the block.
template <int OP, bool DUAL, bool B_MN>
__device__ __forceinline__ void load_slice(const Params& p, const Tile& tl, int i, int blk, int v0, int v1,
                                           int half, int pass, uint8_t* sa, uint8_t* sb, uint8_t* sb2,
                                           uint64_t* bar) {
  using namespace dmoe::tc;
  if (OP == OP_SDD) {
    const int k0 = i * BK;
    tma_load_2d(sa, &p.map_a, bar, k0, tl.b * BM);
    if (B_MN) {
      tma_load_2d(sb, &p.map_b, bar, tl.c * BN, k0);
      tma_load_2d(sb + HALF_BYTES, &p.map_b, bar, tl.c * BN + 64, k0);
      if (DUAL) {
        tma_load_2d(sb2, &p.map_b2, bar, tl.c * BN, k0);
        tma_load_2d(sb2 + HALF_BYTES, &p.map_b2, bar, tl.c * BN + 64, k0);
      }
    } else {
      tma_load_2d(sb, &p.map_b, bar, k0, tl.c * BN);
    }
  } else if (OP == OP_DSD || OP == OP_DSDT) {
    const CUtensorMap* ma = pass ? &p.map_a2 : &p.map_a;
    const CUtensorMap* mb = pass ? &p.map_b2 : &p.map_b;
    tma_load_2d(sa, ma, bar, half * BK, blk * BM);
    if (OP == OP_DSD) {
      const int krow = v0 * BM + half * BK;
      tma_load_2d(sb, mb, bar, tl.b * BN, krow);
      tma_load_2d(sb + HALF_BYTES, mb, bar, tl.b * BN + 64, krow);
    } else {
      tma_load_2d(sb, mb, bar, v0 * BM + half * BK, tl.b * BN);
    }
  } else {
    const int srow = v0 * BM + half * BK;  // K rows inside the block array
    const int drow = v1 * BM + half * BK;  // K rows of the dense operand
    if (OP == OP_DSTD) {
      tma_load_2d(sa, &p.map_a, bar, 0, srow);
      tma_load_2d(sa + HALF_BYTES, &p.map_a, bar, 64, srow);
      tma_load_2d(sb, &p.map_b, bar, tl.b * BN, drow);
      tma_load_2d(sb + HALF_BYTES, &p.map_b, bar, tl.b * BN + 64, drow);
    } else {
      tma_load_2d(sa, &p.map_a, bar, tl.b * BM, drow);
      tma_load_2d(sa + HALF_BYTES, &p.map_a, bar, tl.b * BM + 64, drow);
      tma_load_2d(sb, &p.map_b, bar, 0, srow);
      tma_load_2d(sb + HALF_BYTES, &p.map_b, bar, 64, srow);
    }
  }
}

__device__ __forceinline__ float gelu_f(float x) { return 0.5f * x * (1.f + erff(x * 0.70710678118654752f)); }

__device__ __forceinline__ float gelu_grad_f(float x) {
  return 0.5f * (1.f + erff(x * 0.70710678118654752f)) + x * 0.39894228040143268f * expf(-0.5f * x * x);
}

__device__ __forceinline__ float sigmoid_f(float x) { return 1.f / (1.f + expf(-x)); }

__device__ __forceinline__ void unpack8(const uint4& u, float* f) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 q = __bfloat1622float2(h[i]);
    f[2 * i] = q.x;
    f[2 * i + 1] = q.y;
  }
}

__device__ __forceinline__ uint4 pack8(const float* f) {
  uint4 u;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  return u;
}

// 32 bf16 of row `row`, columns c0..c0+31, of a block staged in shared memory
// by two 128B-swizzled TMA boxes (columns 0-63 and 64-127, 16 KB each): the
// 16-byte chunk j of a 128-byte row sits at chunk j ^ (row % 8), so the 8
// rows of a quarter-warp hit 8 different bank groups.
__device__ __forceinline__ void load32_staged(const uint8_t* blk, int row, int c0, float* v) {
  const uint8_t* box = blk + (c0 >> 6) * HALF_BYTES * 2 + row * 128;
  const int j0 = (c0 & 63) >> 3;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint4 u = *reinterpret_cast<const uint4*>(box + (((j0 + j) ^ (row & 7)) << 4));
    unpack8(u, v + 8 * j);
  }
}

// 32 fp32 accumulator columns of this thread's TMEM lane, waited for in the
// same asm statement so that no use of the registers can move above the wait.
__device__ __forceinline__ void tmem_load32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
        "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
        "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory plan of one instantiation: the operand ring, the staged
// forward blocks of GELU' (double-buffered, 128B-swizzled TMA boxes) and one
// 32 x 32 bf16 slab (2 KB, 64B-swizzled) per epilogue warp, through which
// each output chunk is transposed into row-contiguous global stores.
template <int EPI>
struct Plan {
  static constexpr bool DUAL = EPI == DMOE_EPI_SWIGLU_FWD;
  static constexpr int AUX = EPI == DMOE_EPI_GELU_BWD ? 1 : 0;  // staged by TMA
  static constexpr uint32_t STAGE_BYTES = TILE_BYTES * (DUAL ? 3 : 2);
  static constexpr uint32_t AUX_BYTES = 2u * AUX * BLOCK_BYTES;
  static constexpr uint32_t SLAB = 32 * 32 * 2;
  static constexpr uint32_t OUT_BYTES = kEpiWarps * SLAB;
  static constexpr int STAGES_FIT =
      static_cast<int>((kSmemLimit - kSmemReserve - AUX_BYTES - OUT_BYTES) / STAGE_BYTES);
  static constexpr int STAGES = STAGES_FIT > 6 ? 6 : STAGES_FIT;
  static constexpr size_t SMEM =
      static_cast<size_t>(STAGES) * STAGE_BYTES + AUX_BYTES + OUT_BYTES + kSmemReserve;
  static_assert(STAGES >= 4, "shared-memory plan leaves fewer than four stages");
  static_assert(SMEM <= kSmemLimit, "shared-memory plan too large");
};

// Row and column of element (0, 0) of the 32 x 32 output chunk that the
// warp owning TMEM lane quadrant `quad` stores for columns c0..c0+31, and
// the output's row pitch in elements.
template <int OP>
__device__ __forceinline__ int64_t chunk_origin(const Params& p, const Tile& tl, int quad, int c0, int* pitch) {
  if (OP == OP_SDD) {
    *pitch = BN;
    return static_cast<int64_t>(tl.a) * (BM * BN) + (quad * 32) * BN + c0;
  }
  if (OP == OP_DSD || OP == OP_DSDT || OP == OP_DSTD) {
    *pitch = p.N;
    return (static_cast<int64_t>(tl.a) * BM + quad * 32) * p.N + static_cast<int64_t>(tl.b) * BN + c0;
  }
  *pitch = p.EF;
  return (static_cast<int64_t>(tl.b) * BM + quad * 32) * p.EF + static_cast<int64_t>(tl.a) * BN + c0;
}

// Stores a 32 x 32 bf16 chunk held one row per lane: each lane writes its
// 64-byte row into the warp's 64B-swizzled slab (16-byte chunk j of row r at
// j ^ ((r >> 1) & 3): conflict-free), then the warp reads it back four lanes
// per row and writes 8 full 64-byte row segments per instruction.
__device__ __forceinline__ void store_chunk(uint8_t* slab, int lane, const float* v, uint16_t* out, int64_t origin,
                                            int pitch) {
  uint8_t* rowp = slab + lane * 64;
  const int sw = (lane >> 1) & 3;
#pragma unroll
  for (int j = 0; j < 4; ++j) *reinterpret_cast<uint4*>(rowp + ((j ^ sw) << 4)) = pack8(v + 8 * j);
  __syncwarp();
  const int cj = lane & 3;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = i * 8 + (lane >> 2);
    const uint4 u = *reinterpret_cast<const uint4*>(slab + r * 64 + ((cj ^ ((r >> 1) & 3)) << 4));
    *reinterpret_cast<uint4*>(out + origin + static_cast<int64_t>(r) * pitch + cj * 8) = u;
  }
  __syncwarp();
}

template <int OP, int EPI, bool B_MN>
__global__ void __launch_bounds__(kThreads, 1) bsmm_kernel(const __grid_constant__ Params p) {
  using namespace dmoe::tc;
  using PL = Plan<EPI>;
  constexpr bool DUAL = PL::DUAL;
  constexpr int AUX = PL::AUX;
  constexpr bool A_MN = (OP == OP_DSTD || OP == OP_DSTDT);
  constexpr int STAGES = PL::STAGES;
  constexpr uint32_t STAGE_BYTES = PL::STAGE_BYTES;
  constexpr uint32_t ACC_COLS = DUAL ? 256 : 128;
  constexpr uint32_t TMEM_COLS = 2 * ACC_COLS;
  constexpr uint32_t IDESC = idesc_bf16(BM, BN, A_MN, B_MN);
  // per-UMMA_K advance of the descriptor start address (16-byte units)
  constexpr uint64_t A_STEP = A_MN ? (UMMA_K * 128) >> 4 : (UMMA_K * 2) >> 4;
  constexpr uint64_t B_STEP = B_MN ? (UMMA_K * 128) >> 4 : (UMMA_K * 2) >> 4;
  constexpr uint32_t A_LBO = A_MN ? HALF_BYTES : 16;
  constexpr uint32_t B_LBO = B_MN ? HALF_BYTES : 16;
  constexpr bool WALK = OP != OP_SDD;  // K walks blocks of the topology

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* aux_smem = smem + STAGES * STAGE_BYTES;  // [2][AUX][32 KB]
  uint8_t* out_smem = aux_smem + PL::AUX_BYTES;     // [kEpiWarps][2 KB]
  uint64_t* full = reinterpret_cast<uint64_t*>(out_smem + PL::OUT_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* afull = tempty + 2;
  uint64_t* aempty = afull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(aempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull + a, 1);
      mbar_init(tempty + a, kEpiWarps);
      mbar_init(afull + a, 1);
      mbar_init(aempty + a, kEpiWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&p.map_a);
    tma_prefetch_map(&p.map_b);
  }
  if (warp == 1) tmem_alloc(tmem_slot, TMEM_COLS);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  const int ntiles = num_tiles<OP>(p);
  const int G = gridDim.x;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    int stage = 0;
    uint32_t phase = 0;
    uint32_t aslot = 0, aphase = 0;
    bool ok = true;
    int t = blockIdx.x;
    Tile cur = t < ntiles ? decode<OP>(p, t) : Tile{};
    // lane 0 claims the next stage and issues its loads
    auto issue = [&](const Tile& tl, int i, int blk, int v0, int v1, int half, int pass) {
      if (lane == 0) {
        ok = mbar_wait(empty + stage, phase ^ 1u, abort_flag);
        if (ok) {
          uint8_t* sa = smem + stage * STAGE_BYTES;
          mbar_arrive_expect_tx(full + stage, STAGE_BYTES);
          load_slice<OP, DUAL, B_MN>(p, tl, i, blk, v0, v1, half, pass, sa, sa + TILE_BYTES, sa + 2 * TILE_BYTES,
                                     full + stage);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (++stage == STAGES) {
        stage = 0;
        phase ^= 1u;
      }
    };
    while (t < ntiles && ok) {
      const int tn = t + G;
      const Tile nxt = tn < ntiles ? decode<OP>(p, tn) : Tile{};  // in flight while this tile issues
      if (AUX > 0) {
        if (lane == 0) {
          ok = mbar_wait(aempty + aslot, aphase ^ 1u, abort_flag);
          if (ok) {
            uint8_t* dst = aux_smem + aslot * (AUX * BLOCK_BYTES);
            mbar_arrive_expect_tx(afull + aslot, AUX * BLOCK_BYTES);
            tma_load_2d(dst, &p.map_aux0, afull + aslot, 0, cur.a * BM);
            tma_load_2d(dst + HALF_BYTES * 2, &p.map_aux0, afull + aslot, 64, cur.a * BM);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (++aslot == 2) {
          aslot = 0;
          aphase ^= 1u;
        }
      }
      if (!WALK) {
        for (int i = 0; i < cur.kiters && ok; ++i) issue(cur, i, 0, 0, 0, 0, 0);
      } else {
        const int passes = (OP == OP_DSDT && p.second) ? 2 : 1;
        for (int pass = 0; pass < passes && ok; ++pass) {
          for (int base = 0; base < cur.nblk && ok; base += 32) {
            // up to 32 blocks' topology values fetched at once, one per lane
            int my0 = 0, my1 = 0;
            if (base + lane < cur.nblk) {
              const int j = cur.c + base + lane;
              if (OP == OP_DSD || OP == OP_DSDT) {
                my0 = __ldg(p.column_indices + j);
              } else {
                my0 = __ldg(p.block_offsets_t + j);
                my1 = __ldg(p.row_indices_t + j);
              }
            }
            const int cnt = min(32, cur.nblk - base);
            for (int bb = 0; bb < cnt && ok; ++bb) {
              const int v0 = __shfl_sync(0xffffffffu, my0, bb);
              const int v1 = __shfl_sync(0xffffffffu, my1, bb);
              const int blk = cur.c + base + bb;
              issue(cur, 0, blk, v0, v1, 0, pass);
              if (ok) issue(cur, 0, blk, v0, v1, 1, pass);
            }
          }
        }
      }
      cur = nxt;
      t = tn;
    }
    if (!ok && lane == 0) {
      dmoe::raise_error(p.err, DMOE_SITE_GEMM_WAIT | DMOE_ERR_TIMEOUT);
      *abort_flag = 1;
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // --------------------------------------------------------- MMA issue
      int stage = 0;
      uint32_t phase = 0;
      uint32_t acc = 0, acc_phase = 0;
      bool ok = true;
      int t = blockIdx.x;
      int kit = t < ntiles ? decode<OP>(p, t).kiters : 0;
      while (t < ntiles && ok) {
        const int tn = t + G;
        const int kit_next = tn < ntiles ? decode<OP>(p, tn).kiters : 0;
        if (kit > 0) {
          if (!mbar_wait(tempty + acc, acc_phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          fence_after_sync();
          const uint32_t d0 = tmem_base + acc * ACC_COLS;
          for (int i = 0; i < kit; ++i) {
            if (!mbar_wait(full + stage, phase, abort_flag)) {
              ok = false;
              break;
            }
            fence_after_sync();
            const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
            const uint64_t adesc = sdesc_sw128(sa, A_LBO, 1024);
            const uint64_t bdesc = sdesc_sw128(sa + TILE_BYTES, B_LBO, 1024);
            const uint64_t b2desc = sdesc_sw128(sa + 2 * TILE_BYTES, B_LBO, 1024);
#pragma unroll
            for (int kk = 0; kk < BK / UMMA_K; ++kk) {
              const uint32_t accum = (i > 0 || kk > 0) ? 1u : 0u;
              mma_bf16(d0, adesc + A_STEP * kk, bdesc + B_STEP * kk, IDESC, accum);
              if (DUAL) mma_bf16(d0 + 128, adesc + A_STEP * kk, b2desc + B_STEP * kk, IDESC, accum);
            }
            mma_commit(empty + stage);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          mma_commit(tfull + acc);
          if (++acc == 2) {
            acc = 0;
            acc_phase ^= 1u;
          }
        }
        kit = kit_next;
        t = tn;
      }
      if (!ok) {
        dmoe::raise_error(p.err, DMOE_SITE_GEMM_WAIT | DMOE_ERR_TIMEOUT);
        *abort_flag = 1;
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;               // TMEM lanes 32*quad .. 32*quad+31
    const int col0 = ((warp - 2) >> 2) * 64;  // this warp's 64 of the 128 columns
    const int row = quad * 32 + lane;
    uint8_t* slab = out_smem + (warp - 2) * PL::SLAB;
    uint32_t acc = 0, acc_phase = 0;
    uint32_t aslot = 0, aphase = 0;
    bool ok = true;
    int t = blockIdx.x;
    Tile cur = t < ntiles ? decode<OP>(p, t) : Tile{};
    while (t < ntiles) {
      const int tn = t + G;
      const Tile nxt = tn < ntiles ? decode<OP>(p, tn) : Tile{};
      if (cur.kiters == 0) {
        const float z[32] = {};
        for (int c0 = col0; c0 < col0 + 64; c0 += 32) {
          int pitch;
          const int64_t org = chunk_origin<OP>(p, cur, quad, c0, &pitch);
          store_chunk(slab, lane, z, p.out0, org, pitch);
        }
        cur = nxt;
        t = tn;
        continue;
      }
      uint4 a0[8], a1[8];  // SwiGLU': this row's 64 columns of both stored forward blocks
      if (EPI == DMOE_EPI_SWIGLU_BWD) {
        const int64_t off = static_cast<int64_t>(cur.a) * (BM * BN) + row * BN + col0;
        const uint4* r0 = reinterpret_cast<const uint4*>(p.aux0 + off);
        const uint4* r1 = reinterpret_cast<const uint4*>(p.aux1 + off);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          a0[j] = __ldg(r0 + j);
          a1[j] = __ldg(r1 + j);
        }
      }
      if (!mbar_wait(tfull + acc, acc_phase, abort_flag)) {
        ok = false;
        break;
      }
      const uint8_t* aux = aux_smem + aslot * (AUX * BLOCK_BYTES);
      if (AUX > 0 && !mbar_wait(afull + aslot, aphase, abort_flag)) {
        ok = false;
        break;
      }
      fence_after_sync();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + acc * ACC_COLS;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int c0 = col0 + 32 * h;
        int pitch;
        const int64_t org = chunk_origin<OP>(p, cur, quad, c0, &pitch);
        float v[32];
        tmem_load32(tbase + c0, v);
        if (EPI == DMOE_EPI_STORE) {
          store_chunk(slab, lane, v, p.out0, org, pitch);
        } else if (EPI == DMOE_EPI_GELU_FWD) {
          store_chunk(slab, lane, v, p.out0, org, pitch);
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = gelu_f(v[j]);
          store_chunk(slab, lane, v, p.out1, org, pitch);
        } else if (EPI == DMOE_EPI_SWIGLU_FWD) {
          float v3[32];
          tmem_load32(tbase + 128 + c0, v3);
          store_chunk(slab, lane, v, p.out0, org, pitch);
          store_chunk(slab, lane, v3, p.out1, org, pitch);
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = v[j] * sigmoid_f(v[j]) * v3[j];
          store_chunk(slab, lane, v, p.out2, org, pitch);
        } else if (EPI == DMOE_EPI_GELU_BWD) {
          float hh[32];
          load32_staged(aux, row, c0, hh);
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] *= gelu_grad_f(hh[j]);
          store_chunk(slab, lane, v, p.out0, org, pitch);
        } else {  // SWIGLU_BWD
          float h1[32], h3[32];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            unpack8(a0[4 * h + j], h1 + 8 * j);
            unpack8(a1[4 * h + j], h3 + 8 * j);
          }
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float sg = sigmoid_f(h1[j]);
            const float g = v[j];
            h3[j] = g * h3[j] * sg * (1.f + h1[j] * (1.f - sg));
            v[j] = g * h1[j] * sg;
          }
          store_chunk(slab, lane, h3, p.out0, org, pitch);
          store_chunk(slab, lane, v, p.out1, org, pitch);
        }
      }
      fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(tempty + acc);
        if (AUX > 0) mbar_arrive(aempty + aslot);
      }
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
      if (AUX > 0 && ++aslot == 2) {
        aslot = 0;
        aphase ^= 1u;
      }
      cur = nxt;
      t = tn;
    }
    if (!ok && lane == 0) {
      dmoe::raise_error(p.err, DMOE_SITE_GEMM_WAIT | DMOE_ERR_TIMEOUT);
      *abort_flag = 1;
    }
  }

  fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    fence_after_sync();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// Row-major bf16 matrix [rows, cols]; box = box_cols (inner) x box_rows.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_cols, uint32_t box_rows,
              CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool topo_ok(const dmoe_topology* t) {
  if (!t) return false;
  if (t->E < 1 || t->E > 1024 || t->F < DMOE_BLOCK || (t->F % DMOE_BLOCK) || t->P_max < 0 ||
      (t->P_max % DMOE_BLOCK))
    return false;
  const int64_t nb = t->F / DMOE_BLOCK;
  if (static_cast<int64_t>(t->nnz_max) != static_cast<int64_t>(t->P_max / DMOE_BLOCK) * nb) return false;
  if (static_cast<int64_t>(t->nnz_max) * DMOE_BLOCK > 0x7fffffffLL) return false;
  return t->row_offsets && t->column_indices && t->row_indices && t->column_offsets_t && t->row_indices_t &&
         t->block_offsets_t && t->nnz_dev && t->P_dev;
}

void fill_topo(Params& p, const dmoe_topology* t) {
  p.row_offsets = t->row_offsets;
  p.column_indices = t->column_indices;
  p.row_indices = t->row_indices;
  p.column_offsets_t = t->column_offsets_t;
  p.row_indices_t = t->row_indices_t;
  p.block_offsets_t = t->block_offsets_t;
  p.nnz_dev = t->nnz_dev;
  p.P_dev = t->P_dev;
  p.nb = t->F / DMOE_BLOCK;
  p.EF = t->E * t->F;
}

template <int OP, int EPI, bool B_MN>
dmoe_status launch(const Params& p, const dmoe::DeviceInfo& di, cudaStream_t st) {
  if (p.max_tiles <= 0) return DMOE_OK;
  auto kern = bsmm_kernel<OP, EPI, B_MN>;
  const size_t smem = Plan<EPI>::SMEM;
  // the dynamic shared-memory opt-in, once per instantiation and device
  static std::atomic<uint64_t> opted{0};
  const uint64_t bit = di.device < 64 ? (uint64_t(1) << di.device) : 0;
  if (!bit || !(opted.load(std::memory_order_acquire) & bit)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return dmoe::cuda_status(e);
    if (bit) opted.fetch_or(bit, std::memory_order_acq_rel);
  }
  const int grid = std::min(di.sm_count, p.max_tiles);
  kern<<<grid, kThreads, smem, st>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return dmoe::cuda_status(e);
  dmoe::count_launches(1);
  return DMOE_OK;
}

bool a16(const void* p) { return dmoe::aligned16(p); }

}  // namespace

DMOE_API dmoe_status dmoe_sdd(const uint16_t* A, const uint16_t* B, const uint16_t* B2, int K, int b_trans,
                              const dmoe_topology* topo, int epilogue, const uint16_t* aux0, const uint16_t* aux1,
                              uint16_t* out0, uint16_t* out1, uint16_t* out2, dmoe_stream_t stream) {
  if (!topo_ok(topo) || K < BK || (K % BK) || !A || !B || !out0) return DMOE_ERR_INVALID_ARG;
  if (!a16(A) || !a16(B) || !a16(B2) || !a16(aux0) || !a16(aux1) || !a16(out0) || !a16(out1) || !a16(out2))
    return DMOE_ERR_INVALID_ARG;
  switch (epilogue) {
    case DMOE_EPI_STORE: break;
    case DMOE_EPI_GELU_FWD:
      if (!out1) return DMOE_ERR_INVALID_ARG;
      break;
    case DMOE_EPI_SWIGLU_FWD:
      if (!B2 || !out1 || !out2) return DMOE_ERR_INVALID_ARG;
      if (b_trans) return DMOE_ERR_UNSUPPORTED;
      break;
    case DMOE_EPI_GELU_BWD:
      if (!aux0) return DMOE_ERR_INVALID_ARG;
      break;
    case DMOE_EPI_SWIGLU_BWD:
      if (!aux0 || !aux1 || !out1) return DMOE_ERR_INVALID_ARG;
      break;
    default: return DMOE_ERR_INVALID_ARG;
  }
  dmoe::DeviceInfo di;
  dmoe_status s = dmoe::device_info(&di);
  if (s != DMOE_OK) return s;
  if (topo->nnz_max == 0) return DMOE_OK;
  Params p{};
  fill_topo(p, topo);
  p.K = K;
  p.max_tiles = topo->nnz_max;
  p.aux0 = aux0;
  p.aux1 = aux1;
  p.err = di.err_word;
  if (!make_map(&p.map_a, A, topo->P_max, K, BK, BM)) return DMOE_ERR_CUDA;
  if (!b_trans) {
    if (!make_map(&p.map_b, B, K, p.EF, 64, BK)) return DMOE_ERR_CUDA;
    if (epilogue == DMOE_EPI_SWIGLU_FWD && !make_map(&p.map_b2, B2, K, p.EF, 64, BK)) return DMOE_ERR_CUDA;
  } else {
    if (!make_map(&p.map_b, B, p.EF, K, BK, BN)) return DMOE_ERR_CUDA;
  }
  const uint64_t srows = static_cast<uint64_t>(topo->nnz_max) * BM;
  if (epilogue == DMOE_EPI_GELU_BWD && !make_map(&p.map_aux0, aux0, srows, BN, 64, BM)) return DMOE_ERR_CUDA;
  p.out0 = out0;
  p.out1 = out1;
  p.out2 = out2;
  cudaStream_t st = dmoe::as_stream(stream);
  const bool bmn = !b_trans;
  switch (epilogue) {
    case DMOE_EPI_SWIGLU_FWD: return launch<OP_SDD, DMOE_EPI_SWIGLU_FWD, true>(p, di, st);
    case DMOE_EPI_GELU_FWD:
      return bmn ? launch<OP_SDD, DMOE_EPI_GELU_FWD, true>(p, di, st)
                 : launch<OP_SDD, DMOE_EPI_GELU_FWD, false>(p, di, st);
    case DMOE_EPI_GELU_BWD:
      return bmn ? launch<OP_SDD, DMOE_EPI_GELU_BWD, true>(p, di, st)
                 : launch<OP_SDD, DMOE_EPI_GELU_BWD, false>(p, di, st);
    case DMOE_EPI_SWIGLU_BWD:
      return bmn ? launch<OP_SDD, DMOE_EPI_SWIGLU_BWD, true>(p, di, st)
                 : launch<OP_SDD, DMOE_EPI_SWIGLU_BWD, false>(p, di, st);
    default:
      return bmn ? launch<OP_SDD, DMOE_EPI_STORE, true>(p, di, st) : launch<OP_SDD, DMOE_EPI_STORE, false>(p, di, st);
  }
}

DMOE_API dmoe_status dmoe_dsd(const dmoe_topology* topo, const uint16_t* S, const uint16_t* Bm, int N, uint16_t* C,
                              dmoe_stream_t stream) {
  if (!topo_ok(topo) || N < BN || (N % BN) || !S || !Bm || !C) return DMOE_ERR_INVALID_ARG;
  if (!a16(S) || !a16(Bm) || !a16(C)) return DMOE_ERR_INVALID_ARG;
  dmoe::DeviceInfo di;
  dmoe_status s = dmoe::device_info(&di);
  if (s != DMOE_OK) return s;
  if (topo->nnz_max == 0) return DMOE_OK;
  Params p{};
  fill_topo(p, topo);
  p.N = N;
  p.ntn = N / BN;
  p.max_tiles = (topo->P_max / BM) * p.ntn;
  p.err = di.err_word;
  if (!make_map(&p.map_a, S, static_cast<uint64_t>(topo->nnz_max) * BM, BM, BK, BM)) return DMOE_ERR_CUDA;
  if (!make_map(&p.map_b, Bm, p.EF, N, 64, BK)) return DMOE_ERR_CUDA;
  p.out0 = C;
  return launch<OP_DSD, DMOE_EPI_STORE, true>(p, di, dmoe::as_stream(stream));
}

DMOE_API dmoe_status dmoe_dsd_t(const dmoe_topology* topo, const uint16_t* S, const uint16_t* Bm,
                                const uint16_t* S2, const uint16_t* Bm2, int N, uint16_t* C, dmoe_stream_t stream) {
  if (!topo_ok(topo) || N < BN || (N % BN) || !S || !Bm || !C) return DMOE_ERR_INVALID_ARG;
  if ((S2 == nullptr) != (Bm2 == nullptr)) return DMOE_ERR_INVALID_ARG;
  if (!a16(S) || !a16(Bm) || !a16(S2) || !a16(Bm2) || !a16(C)) return DMOE_ERR_INVALID_ARG;
  dmoe::DeviceInfo di;
  dmoe_status s = dmoe::device_info(&di);
  if (s != DMOE_OK) return s;
  if (topo->nnz_max == 0) return DMOE_OK;
  Params p{};
  fill_topo(p, topo);
  p.N = N;
  p.ntn = N / BN;
  p.max_tiles = (topo->P_max / BM) * p.ntn;
  p.second = S2 ? 1 : 0;
  p.err = di.err_word;
  const uint64_t srows = static_cast<uint64_t>(topo->nnz_max) * BM;
  if (!make_map(&p.map_a, S, srows, BM, BK, BM)) return DMOE_ERR_CUDA;
  if (!make_map(&p.map_b, Bm, N, p.EF, BK, BN)) return DMOE_ERR_CUDA;
  if (S2) {
    if (!make_map(&p.map_a2, S2, srows, BM, BK, BM)) return DMOE_ERR_CUDA;
    if (!make_map(&p.map_b2, Bm2, N, p.EF, BK, BN)) return DMOE_ERR_CUDA;
  }
  p.out0 = C;
  return launch<OP_DSDT, DMOE_EPI_STORE, false>(p, di, dmoe::as_stream(stream));
}

DMOE_API dmoe_status dmoe_dstd(const dmoe_topology* topo, const uint16_t* S, const uint16_t* D, int N, int c_trans,
                               uint16_t* C, dmoe_stream_t stream) {
  if (!topo_ok(topo) || N < BN || (N % BN) || !S || !D || !C) return DMOE_ERR_INVALID_ARG;
  if (!a16(S) || !a16(D) || !a16(C)) return DMOE_ERR_INVALID_ARG;
  dmoe::DeviceInfo di;
  dmoe_status s = dmoe::device_info(&di);
  if (s != DMOE_OK) return s;
  Params p{};
  fill_topo(p, topo);
  p.N = N;
  p.ntn = N / BN;
  p.max_tiles = (p.EF / BM) * p.ntn;
  p.err = di.err_word;
  const uint64_t srows = static_cast<uint64_t>(topo->nnz_max > 0 ? topo->nnz_max : 1) * BM;
  const uint64_t drows = topo->P_max > 0 ? topo->P_max : BM;
  // with no rows at all every tile has K = 0 and only zeros are written;
  // the maps then describe valid placeholder extents that are never read
  if (!c_trans) {
    if (!make_map(&p.map_a, S, srows, BM, 64, BK)) return DMOE_ERR_CUDA;
    if (!make_map(&p.map_b, D, drows, N, 64, BK)) return DMOE_ERR_CUDA;
    p.out0 = C;
    return launch<OP_DSTD, DMOE_EPI_STORE, true>(p, di, dmoe::as_stream(stream));
  }
  if (!make_map(&p.map_a, D, drows, N, 64, BK)) return DMOE_ERR_CUDA;
  if (!make_map(&p.map_b, S, srows, BM, 64, BK)) return DMOE_ERR_CUDA;
  p.out0 = C;
  return launch<OP_DSTDT, DMOE_EPI_STORE, true>(p, di, dmoe::as_stream(stream));
}
