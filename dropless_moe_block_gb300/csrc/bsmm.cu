// a4/a8 SDD, a5 DSD, a10 DSD^T and a9 DSTD: the block-sparse products of
// George Lin's blog post on MoE training, section 1.2 (the expert MLP as
// SDD -> activation -> DSD) and section 1.3 (128x128 blocks, BCSR row walk,
// transpose index for the weight gradient).
//
// One persistent, warp-specialised tcgen05 kernel template serves all four:
//   warp 0      TMA producer (whole warp): the lanes fetch up to 32 block
//               indices of the topology at once, lane 0 issues the TMA loads
//               of 64-wide K slices of A and B into a ring of 128B-swizzled
//               shared-memory stages (mbarrier complete_tx)
//   warp 1      TMEM allocator + single-thread tcgen05.mma issuer
//               (M=128, N=BN, K=16 per instruction, fp32 accumulator)
//   warps 2-9   epilogue, two warps per TMEM lane quadrant: tcgen05.ld of
//               the accumulator, fused activation / activation gradient (the
//               backward reads the stored forward blocks with coalesced loads
//               a tile ahead and turns them into rows through the warp's
//               slab), bf16 chunks written into the warp's 64B-swizzled
//               slabs and sent out by coalesced 16-byte stores
// A tile is 128 rows x BN columns, BN = 128 or 256 (chosen per call from
// the tile count); with BN = 256 an SDD tile is two adjacent nonzero blocks
// of one row, and the SwiGLU SDD runs W1 and W3 as the two halves of one
// N = 256 product.  Two TMEM accumulators per CTA let the epilogue of tile
// i overlap the MMAs of tile i+1.  CTA pairs (2-CTA clusters) run M = 256
// tiles as single cta_group::2 operations, 256 x 256, or 256 x 512 as two
// sub-tiles whose N = 256 operations share each K step's A slice (NS = 2:
// the two accumulators fill the tensor memory, so the MMAs of the next tile
// start on sub-tile 0 as soon as the epilogue has drained it, and sub-tile
// 1's first K steps wait in their ring stages until it is drained too).
// Tiles are assigned round-robin over a grid of one CTA per SM (or pair);
// every role decodes its next tiles ahead.  Every mbarrier wait is bounded
// (kWaitLimitNs); on expiry the kernel records DMOE_SITE_GEMM_WAIT |
// DMOE_ERR_TIMEOUT, stops all roles, frees its TMEM and returns.
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
#include "tmap.cuh"

namespace {

using dmoe::tc::smem_u32;

enum Op : int { OP_SDD = 0, OP_DSD = 1, OP_DSDT = 2, OP_DSTD = 3, OP_DSTDT = 4 };

constexpr int BM = 128;  // tile rows = TMEM lanes
constexpr int BK = 64;   // K slice per pipeline stage (one 128-byte swizzle row)
constexpr int BLK = 128;  // default block edge of the sparse format (64 and 256 also served)
constexpr int UMMA_K = 16;
constexpr uint32_t SLICE_BYTES = BM * BK * 2;    // 16 KB: 128 rows x 64 K of bf16
constexpr uint32_t ATOM_BYTES = 64 * BK * 2;     // 8 KB: 64 MN x 64 K (MN-major box)
constexpr int kEpiWarps = 8;  // two per TMEM lane quadrant
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr size_t kSmemLimit = 232448;  // opt-in dynamic shared memory per CTA
constexpr size_t kSmemReserve = 1024 + 512;
// CTA-pair products over row blocks: the pair-row table (one word per
// expert and one for the totals) for up to kPairMaxE experts
constexpr int kPairMaxE = 256;
constexpr size_t kPairTabBytes = ((kPairMaxE + 1) * 4 + 15) / 16 * 16;

std::atomic<int> g_tile_n{0};  // 0 = choose per call, else forced 128 / 256
// CTA pairs: 0 = choose per call, 1 = never, 2 = where allowed (256 x 256
// pair tiles), 3 = where allowed, with 256 x 512 tiles (two sub-tiles) where
// the shape allows those
std::atomic<int> g_pair{0};

struct Params {
  CUtensorMap map_a;
  CUtensorMap map_b;
  CUtensorMap map_a2;
  CUtensorMap map_b2;
  CUtensorMap map_a64;   // A (and the second pair's A) in 64-row boxes: a CTA's half of a lone row block
  CUtensorMap map_a2_64;
  uint16_t* out[3];  // outputs out0..out2 (row-major bf16)
  int64_t ldo;       // their row pitch in elements
  const int32_t* row_offsets;
  const int32_t* column_indices;
  const int32_t* row_indices;
  const int32_t* column_offsets_t;
  const int32_t* row_indices_t;
  const int32_t* block_offsets_t;
  const int32_t* nnz_dev;
  const int32_t* P_dev;
  const int32_t* row_fill;  // rows holding tokens per row block (NULL: all full)
  int blk;        // block edge B of the format: 64, 128 or 256
  int bsh;        // log2(B)
  int tm;         // tile rows: min(B, 128)
  int nb;         // F / B
  int K;          // SDD reduction length
  int N;          // dense width (DSD, DSD^T, DSTD)
  int EF;         // E * F
  int E;          // experts
  int ntn;        // tiles along the dense width (CTA pairs: 256-wide pair tiles)
  int max_tiles;  // host bound on the tile count
  int second;     // DSD^T: a second (S2, B2) pair accumulates into the same tile
  const uint16_t* aux0;  // stored forward blocks read by the backward epilogues
  const uint16_t* aux1;
  int32_t* err;
};

struct Tile {
  int kiters;  // 64-wide K slices
  int a, b, c;  // op-specific coordinates
  int nblk;     // blocks walked along K (DSD / DSD^T / DSTD)
  int m64;      // M = 64 MMAs: 64-row blocks, or a tile with at most 64 tokens
  int ro, co;   // row / column offset of the tile inside its block
  int single;   // CTA pair: the pair tile covers one row block (an expert's odd last one),
                // 64 of its rows per CTA (M = 128 pair MMAs)
  int ld0, ld1, ld2;  // topology values loaded by decode(), turned into fields by finish()
};

// Pair rows of the CTA-pair products that walk row blocks (SDD, DSD,
// DSD^T): the two CTAs of a pair take row blocks 2j and 2j + 1 of one expert
// (the same weights); the last one, when the expert has an odd count, is
// split over the pair, 64 rows per CTA (M = 128 pair MMAs).
// Table entry e (0..E) packs the first row block (high 16 bits) and the
// first pair row (low 16 bits) of expert e; entry E holds the totals.  Built
// by warp 0 from the transposed column offsets: expert e's first column
// block lists one block per row block of e.
__device__ void build_pair_table(const Params& p, uint32_t* tab, int lane) {
  int carry_pr = 0, carry_rb = 0;
  for (int base = 0; base < p.E; base += 32) {
    const int e = base + lane;
    int nrb = 0;
    if (e < p.E) {
      const int c = e * p.nb;
      nrb = __ldg(p.column_offsets_t + c + 1) - __ldg(p.column_offsets_t + c);
    }
    int ipr = (nrb + 1) >> 1, irb = nrb;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int upr = __shfl_up_sync(0xffffffffu, ipr, o);
      const int urb = __shfl_up_sync(0xffffffffu, irb, o);
      if (lane >= o) {
        ipr += upr;
        irb += urb;
      }
    }
    if (e < p.E) tab[e + 1] = (static_cast<uint32_t>(carry_rb + irb) << 16) | static_cast<uint32_t>(carry_pr + ipr);
    carry_pr += __shfl_sync(0xffffffffu, ipr, 31);
    carry_rb += __shfl_sync(0xffffffffu, irb, 31);
  }
  if (lane == 0) tab[0] = 0;
}

struct PairRow {
  int e;       // expert
  int rb;      // first row block of the pair
  int single;  // the expert's last, odd row block: no second one
};

// Pair row pr of expert e.
__device__ __forceinline__ PairRow pair_row_of(const uint32_t* tab, int e, int pr) {
  PairRow q;
  q.e = e;
  q.rb = static_cast<int>(tab[e] >> 16) + 2 * (pr - static_cast<int>(tab[e] & 0xffffu));
  q.single = q.rb + 1 == static_cast<int>(tab[e + 1] >> 16);
  return q;
}

// Pair row pr (< the total in tab[E]): its expert is the last e whose first
// pair row is <= pr (experts without rows own no pair row).
__device__ __forceinline__ int pair_expert(const uint32_t* tab, int E, int pr) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (static_cast<int>(tab[mid] & 0xffffu) <= pr) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Pair rows per rasterisation group of the CTA-pair row-walking products
// (groups of 4 or 8 for DSD / DSD^T, whose rows are whole rows of blocks,
// measured more weight traffic from HBM, not less).
constexpr int kPairRaster = 16;

// Tile t of the pair-row x cols grid, rasterised by expert: an expert's
// tiles form groups of up to kPairRaster pair rows with the columns outer
// and the rows inner, so the pairs working at the same time share weight
// columns (one expert's) while the group's rows stay in L2, and the weights
// are streamed from HBM about once per group.  Every expert has the same
// `cols` column tiles, so expert e's tiles start at its first pair row
// times cols.
__device__ __forceinline__ PairRow pair_raster(const uint32_t* tab, int E, int t, int cols, int& c) {
  const int e = pair_expert(tab, E, t / cols);
  const int pr0 = static_cast<int>(tab[e] & 0xffffu);
  const int npr = static_cast<int>(tab[e + 1] & 0xffffu) - pr0;
  int l = t - pr0 * cols;
  const int g = l / (kPairRaster * cols);
  const int gr0 = g * kPairRaster;
  const int gh = min(kPairRaster, npr - gr0);
  l -= gr0 * cols;
  c = l / gh;
  return pair_row_of(tab, e, pr0 + gr0 + l % gh);
}

// Output columns of one SDD tile (the SwiGLU tile runs W1 | W3 as the two
// halves of an N = 256 product, so it covers 128 output columns).
template <int BN, bool DUAL>
__host__ __device__ constexpr int sdd_cols_per_tile() {
  return DUAL ? 128 : BN;
}

template <int OP, int BN, bool DUAL>
__device__ __forceinline__ int num_tiles(const Params& p) {
  int n;
  if (OP == OP_SDD) n = (__ldg(p.P_dev) / p.tm) * (p.nb * p.blk / sdd_cols_per_tile<BN, DUAL>());
  else if (OP == OP_DSD || OP == OP_DSDT) n = (__ldg(p.P_dev) / p.tm) * p.ntn;
  else if (OP == OP_DSTD) n = (p.EF / BM) * p.ntn;
  else n = (p.EF / BN) * p.ntn;
  return n < p.max_tiles ? (n > 0 ? n : 0) : p.max_tiles;
}

// Row blocks per rasterisation group of the row-walking products.
constexpr int kRasterRows = 8;

// Tile t of a rows x cols grid, visited in groups of kRasterRows rows with
// the columns outer and the rows inner inside a group: concurrent CTAs then
// share each weight column tile (L2 hits) while a group's A rows stay in L2.
__device__ __forceinline__ void raster(int t, int rows, int cols, int& r, int& c) {
  const int per_group = kRasterRows * cols;
  const int g = t / per_group;
  const int r0 = g * kRasterRows;
  const int rg = min(kRasterRows, rows - r0);
  const int l = t - g * per_group;
  r = r0 + l % rg;
  c = l / rg;
}

// Row tiles of the row-walking products (P / tile rows).
template <int OP, int BN, bool DUAL>
__device__ __forceinline__ int tile_rows(const Params& p, int ntiles) {
  if (OP == OP_SDD) return ntiles / (p.nb * p.blk / sdd_cols_per_tile<BN, DUAL>());
  if (OP == OP_DSD || OP == OP_DSDT) return ntiles / p.ntn;
  return 0;
}

// NS = 2 (CTA pairs only): tile t is a pair of horizontally adjacent
// sub-tiles sharing their A rows; decode() returns the first (the column tile
// counts it sees are those of the sub-tile pairs), second_sub() the second.
template <int OP, int BN, bool DUAL, bool PAIR, int NS = 1>
__device__ __forceinline__ Tile decode(const Params& p, int t, int rows, int rank, const uint32_t* tab) {
  Tile tl;
  tl.ro = 0;
  tl.co = 0;
  tl.single = 0;
  if (OP == OP_SDD) {
    // row tile rt (tm rows), column tile ct of the expert; every row block
    // holds its expert's nb blocks, so block (r, j) sits at BCSR position
    // r*nb + j.  CTA pair: pair row rt, this CTA's row block of it.
    constexpr int cols = NS * sdd_cols_per_tile<BN, DUAL>();
    int rt = 0, ct;
    PairRow pq{};
    if (PAIR) pq = pair_raster(tab, p.E, t, p.nb * p.blk / cols, ct);
    else raster(t, rows, p.nb * p.blk / cols, rt, ct);
    const int lc = ct * cols;  // first output column inside the expert
    int r;
    if (PAIR) {
      tl.single = pq.single;
      r = pq.rb + (pq.single ? 0 : rank);
      tl.b = r;  // row tile = row block (B = 128)
    } else {
      const int row0 = rt * p.tm;
      r = row0 >> p.bsh;
      tl.ro = row0 - (r << p.bsh);
      tl.b = rt;  // row tile
    }
    const int q = r * p.nb + (lc >> p.bsh);
    tl.co = lc & (p.blk - 1);
    tl.a = q;                                                   // first block
    tl.ld0 = __ldg(p.column_indices + q);                       // its weight column block
    tl.ld1 = (PAIR || p.blk == 64 || p.row_fill == nullptr) ? 0 : __ldg(p.row_fill + r);
    tl.kiters = p.K / BK;
    tl.nblk = 0;
  } else if (OP == OP_DSD || OP == OP_DSDT) {
    // walked in reverse (last row tiles, i.e. last experts, first): in a
    // layer step the SDD before them walks forward, so the blocks of the
    // experts it reached last are still in L2 when these tiles start; and
    // the backward SDD after the forward DSD starts on the experts whose
    // weight rows the DSD read last
    int rt = 0, nt;
    PairRow q{};
    if (PAIR) q = pair_raster(tab, p.E, rows * p.ntn - 1 - t, p.ntn, nt);
    else raster(rows * p.ntn - 1 - t, rows, p.ntn, rt, nt);
    int r;
    if (PAIR) {
      tl.single = q.single;
      r = q.rb + (q.single ? 0 : rank);
      tl.a = r;  // row tile = row block (B = 128)
    } else {
      const int row0 = rt * p.tm;
      r = row0 >> p.bsh;
      tl.ro = row0 - (r << p.bsh);
      tl.a = rt;  // row tile
    }
    tl.ld0 = __ldg(p.row_offsets + r);
    tl.ld1 = __ldg(p.row_offsets + r + 1);
    tl.ld2 = (PAIR || p.blk == 64 || p.row_fill == nullptr) ? 0 : __ldg(p.row_fill + r);
    tl.b = nt * NS;  // n tile
  } else {
    // DSTD: 128 weight columns (column block cb from column co; two blocks
    // cb, cb + 1 when B = 64), n tile.  DSTD^T: BN weight columns, m tile.
    // CTA pair: DSTD takes 128-column groups 2g and 2g + 1 (one expert, the
    // same K walk), DSTD^T m tiles 2m and 2m + 1 of one column group.
    int cg, b;
    if (PAIR && OP == OP_DSTD) {
      const int g = t / p.ntn;
      cg = 2 * g + rank;
      b = t - g * p.ntn;
    } else {
      cg = t / p.ntn;
      b = t - cg * p.ntn;
      if (PAIR) b = 2 * b + rank;
    }
    const int c0 = cg * (OP == OP_DSTD ? BM : BN * NS);
    const int cb = c0 >> p.bsh;
    tl.ld0 = __ldg(p.column_offsets_t + cb);
    tl.ld1 = __ldg(p.column_offsets_t + cb + 1);
    tl.co = c0 - (cb << p.bsh);
    tl.a = OP == OP_DSTD ? cg : cg * NS;
    tl.b = OP == OP_DSTD ? b * NS : b;
  }
  return tl;
}

// The second sub-tile of a finished NS = 2 tile: the next column tile of the
// same rows and the same K walk.  SDD: the next output block(s) of the row
// block and the weight columns after the first sub-tile's (an expert's
// blocks of a row sit at consecutive BCSR positions and weight column
// blocks).  DSTD^T: the next BN weight columns, blocks further along the
// same row blocks of the expert.  DSD, DSD^T, DSTD: the next n tile.
template <int OP, int BN, bool DUAL>
__device__ __forceinline__ Tile second_sub(const Params& p, Tile tl) {
  if (OP == OP_SDD) {
    constexpr int cols = sdd_cols_per_tile<BN, DUAL>();
    tl.a += cols >> p.bsh;
    tl.c += cols;
  } else if (OP == OP_DSTDT) {
    tl.a += 1;
    tl.co += BN;
  } else {
    tl.b += 1;
  }
  return tl;
}

// The fields of a decoded tile that depend on its loaded topology values.
// decode() only issues the loads; each role finishes a tile one iteration
// after decoding it, so the loads' latency passes during the current tile's
// work instead of stalling the tile boundary.  (A row block with at most 64
// tokens runs M = 64 MMAs; 64-row blocks always do.)
template <int OP, bool PAIR>
__device__ __forceinline__ void finish(const Params& p, Tile& tl) {
  if (OP == OP_SDD) {
    tl.c = (tl.ld0 << p.bsh) + tl.co;  // first weight column
    tl.m64 = PAIR ? 0 : (p.blk == 64 ? 1 : (p.row_fill != nullptr && tl.ld1 - tl.ro <= 64));
  } else if (OP == OP_DSD || OP == OP_DSDT) {
    const int n = tl.ld1 - tl.ld0;
    tl.c = tl.ld0;
    tl.nblk = n;
    tl.kiters = n * (p.blk >> 6) * (p.second ? 2 : 1);
    tl.m64 = PAIR ? 0 : (p.blk == 64 ? 1 : (p.row_fill != nullptr && tl.ld2 - tl.ro <= 64));
  } else {
    const int n = tl.ld1 - tl.ld0;
    tl.c = tl.ld0;
    tl.nblk = n;
    tl.kiters = n * (p.blk >> 6);
    tl.m64 = 0;  // M runs over weight columns here; the padding is along K
  }
}

// TMA loads of one K slice into A (16 KB) and B (BN x 64: 16 or 32 KB; a
// CTA of a pair loads its half of B, BN / 2 x 64).  MN-major operands are
// stored as 64-wide atoms of 64 MN x 64 K, ATOM_BYTES apart.  For the
// block-walking ops, v0 / v1 are the per-block topology values (DSD, DSD^T:
// column block; DSTD: BCSR position and row block), blk the BCSR position,
// kk the 64-row slice of the block.  ld(dst, map, x, y) issues one box.
// with_a = false loads B only (the second sub-tile of an NS = 2 tile).
template <int OP, bool DUAL, bool B_MN, int BN, bool PAIR, typename LD>
__device__ __forceinline__ void load_slice(const Params& p, const Tile& tl, int i, int blk, int v0, int v1,
                                           int kk, int pass, uint8_t* sa, uint8_t* sb, int rank, bool with_a,
                                           LD&& ld) {
  // B atoms (or rows) of this CTA: all BN, or the half [rank BN/2, (rank+1) BN/2)
  constexpr int ATOMS = (PAIR ? BN / 2 : BN) / 64;
  const int j0 = PAIR ? rank * ATOMS : 0;
  const int bsh = p.bsh;
  // a lone row block of a CTA pair: this CTA's 64 of its rows
  const bool half = PAIR && tl.single;
  const int a_off = half ? 64 * rank : 0;
  if (OP == OP_SDD) {
    const int k0 = i * BK;
    if (with_a) ld(sa, half ? &p.map_a64 : &p.map_a, k0, tl.b * p.tm + a_off);
    if (B_MN) {
      if (DUAL && half) {
        // an M = 128 pair MMA keeps output columns 0-127 (rank 0's B) in
        // TMEM lanes 0-63 and 128-255 (rank 1's) in lanes 64-127: rank r
        // loads W1 and W3 columns 64 r .. 64 r + 63, so that every lane
        // holds matching W1 and W3 results
        ld(sb, &p.map_b, tl.c + 64 * rank, k0);
        ld(sb + ATOM_BYTES, &p.map_b2, tl.c + 64 * rank, k0);
      } else if (DUAL && PAIR) {
        // W1 | W3 halves of the N = 256 product: rank 0 loads W1, rank 1 W3
        const CUtensorMap* mb = rank ? &p.map_b2 : &p.map_b;
        ld(sb, mb, tl.c, k0);
        ld(sb + ATOM_BYTES, mb, tl.c + 64, k0);
      } else if (DUAL) {
        ld(sb, &p.map_b, tl.c, k0);
        ld(sb + ATOM_BYTES, &p.map_b, tl.c + 64, k0);
        ld(sb + 2 * ATOM_BYTES, &p.map_b2, tl.c, k0);
        ld(sb + 3 * ATOM_BYTES, &p.map_b2, tl.c + 64, k0);
      } else {
#pragma unroll
        for (int j = 0; j < ATOMS; ++j) ld(sb + j * ATOM_BYTES, &p.map_b, tl.c + 64 * (j0 + j), k0);
      }
    } else {
      ld(sb, &p.map_b, k0, tl.c + 64 * j0);
    }
  } else if (OP == OP_DSD || OP == OP_DSDT) {
    const CUtensorMap* ma = half ? (pass ? &p.map_a2_64 : &p.map_a64) : (pass ? &p.map_a2 : &p.map_a);
    const CUtensorMap* mb = pass ? &p.map_b2 : &p.map_b;
    if (with_a) ld(sa, ma, kk * BK, (blk << bsh) + tl.ro + a_off);
    const int krow = (v0 << bsh) + kk * BK;  // weight rows (DSD) / columns (DSD^T)
    if (OP == OP_DSD) {
#pragma unroll
      for (int j = 0; j < ATOMS; ++j) ld(sb + j * ATOM_BYTES, mb, tl.b * BN + 64 * (j0 + j), krow);
    } else {
      ld(sb, mb, krow, tl.b * BN + 64 * j0);
    }
  } else {
    const int drow = (v1 << bsh) + kk * BK;  // K rows of the dense operand
    // 64-column atom j of the tile's weight columns inside the block array:
    // block v0 + (co + 64 j) / B, column (co + 64 j) % B, rows kk*64..
    // (B a power of two: shifts and masks on the single issuing thread)
    auto srow = [&](int j) { return ((v0 + ((tl.co + 64 * j) >> bsh)) << bsh) + kk * BK; };
    auto scol = [&](int j) { return (tl.co + 64 * j) & ((1 << bsh) - 1); };
    if (OP == OP_DSTD) {
      if (with_a) {
        ld(sa, &p.map_a, scol(0), srow(0));
        ld(sa + ATOM_BYTES, &p.map_a, scol(1), srow(1));
      }
#pragma unroll
      for (int j = 0; j < ATOMS; ++j) ld(sb + j * ATOM_BYTES, &p.map_b, tl.b * BN + 64 * (j0 + j), drow);
    } else {
      if (with_a) {
        ld(sa, &p.map_a, tl.b * BM, drow);
        ld(sa + ATOM_BYTES, &p.map_a, tl.b * BM + 64, drow);
      }
      // the tile's columns of one row block sit in adjacent blocks of that row
#pragma unroll
      for (int j = 0; j < ATOMS; ++j) ld(sb + j * ATOM_BYTES, &p.map_b, scol(j0 + j), srow(j0 + j));
    }
  }
}

__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// Packed two-lane fp32 arithmetic of the sm_100 family: one instruction
// yields two independent results, each rounded as the scalar operation.
__device__ __forceinline__ float2 f2_fma(float2 a, float2 b, float2 c) {
  float2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(reinterpret_cast<uint64_t&>(d))
      : "l"(reinterpret_cast<uint64_t&>(a)), "l"(reinterpret_cast<uint64_t&>(b)), "l"(reinterpret_cast<uint64_t&>(c)));
  return d;
}

__device__ __forceinline__ float2 f2_mul(float2 a, float2 b) {
  float2 d;
  asm("mul.rn.f32x2 %0, %1, %2;"
      : "=l"(reinterpret_cast<uint64_t&>(d))
      : "l"(reinterpret_cast<uint64_t&>(a)), "l"(reinterpret_cast<uint64_t&>(b)));
  return d;
}

__device__ __forceinline__ float2 f2_splat(float v) { return make_float2(v, v); }

__device__ __forceinline__ float ex2_approx(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// The exact (erf) GELU, gelu(x) = x Phi(x), and its derivative
// gelu'(x) = Phi(x) + x phi(x), of two accumulator values with packed
// arithmetic.  Phi comes from the erfc approximation of Abramowitz & Stegun,
// Handbook of Mathematical Functions, formula 7.1.26 (|error| <= 1.5e-7):
//   erfc(z) ~= t (a1 + t (a2 + t (a3 + t (a4 + t a5)))) exp(-z^2),
//   t = 1 / (1 + p z),  z = |x| / sqrt(2) >= 0,
// with the coefficients halved so that the product is Phi(-|x|) directly.
// exp(-z^2) = exp(-x^2 / 2) = 2^(-x^2 log2(e) / 2) also gives the density
// phi(x) = exp(-x^2 / 2) / sqrt(2 pi).  Phi(x) = 1 - Phi(-|x|) for x >= 0
// and Phi(-|x|) for x < 0, chosen by a select (no cancellation in the left
// tail).
__device__ __forceinline__ void gelu_pair(float2 x, float2& gelu, float2& dgelu) {
  const float2 ax = make_float2(fabsf(x.x), fabsf(x.y));
  const float2 u = f2_fma(ax, f2_splat(0.3275911f * 0.70710678118654752f), f2_splat(1.f));
  const float2 t = make_float2(rcp_approx(u.x), rcp_approx(u.y));
  float2 q = f2_fma(t, f2_splat(0.5f * 1.061405429f), f2_splat(0.5f * -1.453152027f));
  q = f2_fma(t, q, f2_splat(0.5f * 1.421413741f));
  q = f2_fma(t, q, f2_splat(0.5f * -0.284496736f));
  q = f2_fma(t, q, f2_splat(0.5f * 0.254829592f));
  q = f2_mul(q, t);
  const float2 s = f2_mul(f2_mul(x, x), f2_splat(-0.5f * 1.44269504088896341f));
  const float2 e = make_float2(ex2_approx(s.x), ex2_approx(s.y));
  const float2 h = f2_mul(q, e);                                  // Phi(-|x|)
  const float2 omh = f2_fma(h, f2_splat(-1.f), f2_splat(1.f));     // 1 - Phi(-|x|)
  const float2 cdf = make_float2(x.x < 0.f ? h.x : omh.x, x.y < 0.f ? h.y : omh.y);
  dgelu = f2_fma(f2_mul(x, f2_splat(0.39894228040143268f)), e, cdf);  // Phi + x phi
  gelu = f2_mul(x, cdf);
}


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

// Shared-memory plan of one instantiation: the operand ring and two 32 x 32
// bf16 slabs (2 KB each, 64B-swizzled) per epilogue warp.  A CTA of a pair
// holds half of each B slice, and the pair-row table.  NS = 2: each stage
// holds the B slices of both sub-tiles after the shared A slice.
template <int EPI, int BN, bool PAIR, int NS = 1>
struct Plan {
  static constexpr bool DUAL = EPI == DMOE_EPI_SWIGLU_FWD;
  static constexpr uint32_t B_BYTES = (PAIR ? BN / 2 : BN) * BK * 2;  // one sub-tile's B slice
  static constexpr uint32_t STAGE_BYTES = SLICE_BYTES + NS * B_BYTES;
  static constexpr uint32_t SLAB = 32 * 32 * 2;
  static constexpr uint32_t OUT_BYTES = kEpiWarps * 2 * SLAB;
  static constexpr size_t TAB_BYTES = PAIR ? kPairTabBytes : 0;
  static constexpr int STAGES_FIT =
      static_cast<int>((kSmemLimit - kSmemReserve - TAB_BYTES - OUT_BYTES) / STAGE_BYTES);
  static constexpr int STAGES = STAGES_FIT > 6 ? 6 : STAGES_FIT;
  static constexpr size_t SMEM = static_cast<size_t>(STAGES) * STAGE_BYTES + OUT_BYTES + TAB_BYTES + kSmemReserve;
  static_assert(STAGES >= 4, "shared-memory plan leaves fewer than four stages");
  static_assert(SMEM <= kSmemLimit, "shared-memory plan too large");
  static_assert(!DUAL || BN == 256, "the SwiGLU SDD runs W1 | W3 as one N = 256 product");
  static_assert(!PAIR || BN == 256, "a CTA pair runs M = 256 x N = 256 products");
  static_assert(NS == 1 || (NS == 2 && PAIR), "two sub-tiles per tile: CTA pairs only");
};

// Output coordinates (column x, row y) of element (tile row 0, tile column
// cc) in the output's tensor map.  SDD writes B x B blocks, seen as a
// [nnz_max * B, B] matrix: the tile starts at row ro, column co of block
// tl.a and a 32-column chunk never crosses a block.
template <int OP, int BN>
__device__ __forceinline__ void chunk_xy(const Params& p, const Tile& tl, int cc, int* x, int* y) {
  if (OP == OP_SDD) {
    const int c = tl.co + cc;
    *x = c & (p.blk - 1);
    *y = ((tl.a + (c >> p.bsh)) << p.bsh) + tl.ro;
  } else if (OP == OP_DSD || OP == OP_DSDT) {
    *x = tl.b * BN + cc;
    *y = tl.a * p.tm;
  } else if (OP == OP_DSTD) {
    *x = tl.b * BN + cc;
    *y = tl.a * BM;
  } else {
    *x = tl.a * BN + cc;
    *y = tl.b * BM;
  }
}

// Tile row held by TMEM lane r (0..31) of lane quadrant quad.  An M = 128
// accumulator keeps row 32 quad + r there; an M = 64 one keeps rows 16 quad +
// r in lanes r < 16 and nothing in lanes 16..31, which then stand for the
// block's padding rows 64 + 16 quad + (r - 16) (written as the results of
// all-zero rows).
// `layout`: 0 for an M = 128 accumulator (and each CTA's half of an M =
// 256 pair one), 1 for an M = 64 one, 2 + rank for a CTA pair's M = 128
// accumulator, whose CTA of rank r keeps rows 64 r + m (m < 64) in TMEM lanes
// m and 64 + m (the first and second half of the columns; measured on this
// GPU with a probe of one MMA), so quadrant quad holds rows
// 64 r + 32 (quad & 1) + r.
__device__ __forceinline__ int tile_row(int quad, int r, int layout) {
  if (layout == 0) return 32 * quad + r;
  if (layout == 1) return r < 16 ? 16 * quad + r : 48 + 16 * quad + r;
  return 64 * (layout - 2) + 32 * (quad & 1) + r;
}

// Output chunks.  A 32 x 32 bf16 chunk held one row per lane (lane r = TMEM
// lane 32 quad + r) goes to global memory through the warp's slab: each lane
// writes its 64-byte row into the slab (16-byte piece j of row r at piece
// j ^ ((r >> 1) & 3), free of bank conflicts), then every lane reads back
// 16-byte pieces of other rows, so that each store instruction writes whole
// row segments: 8 rows x 64 bytes (one chunk) or 4 rows x 128 bytes (two
// chunks side by side).  Plain coalesced stores: no proxy fence, no bulk
// group to wait for before the slab is reused.  Rows at or past `rows`
// (tile_row(quad, r, layout)) do not exist and are skipped.  `flip` stores the
// rows pairwise swapped (a second slab read in the same instruction as the
// first then hits the other half of the banks).
__device__ __forceinline__ void slab_put(uint8_t* slab, int lane, const float* v, int flip = 0) {
  uint8_t* rowp = slab + (lane ^ flip) * 64;
  const int sw = (lane >> 1) & 3;
#pragma unroll
  for (int j = 0; j < 4; ++j) *reinterpret_cast<uint4*>(rowp + ((j ^ sw) << 4)) = pack8(v + 8 * j);
}

__device__ __forceinline__ uint4 slab_get(const uint8_t* slab, int r, int j, int flip = 0) {
  return *reinterpret_cast<const uint4*>(slab + (r ^ flip) * 64 + ((j ^ ((r >> 1) & 3)) << 4));
}

// One chunk at columns x .. x + 31 of output rows y0 + tile_row(quad, ., layout).
__device__ __forceinline__ void write_chunk(uint8_t* slab, int lane, const float* v, uint16_t* out, int64_t ld, int x,
                                            int y0, int quad, int layout, int rows) {
  slab_put(slab, lane, v);
  __syncwarp();
  const int j = lane & 3;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = 8 * i + (lane >> 2);
    const uint4 q = slab_get(slab, r, j);
    const int tr = tile_row(quad, r, layout);
    if (tr < rows) *reinterpret_cast<uint4*>(out + static_cast<int64_t>(y0 + tr) * ld + x + 8 * j) = q;
  }
  __syncwarp();
}

// Two chunks side by side (columns x .. x + 63), through the warp's two slabs.
__device__ __forceinline__ void write_chunk2(uint8_t* slabs, int lane, const float* v, const float* w, uint16_t* out,
                                             int64_t ld, int x, int y0, int quad, int layout, int rows,
                                             uint32_t slab_bytes) {
  slab_put(slabs, lane, v);
  slab_put(slabs + slab_bytes, lane, w, 1);
  __syncwarp();
  const int j = lane & 7;
  const uint8_t* sl = slabs + (j >> 2) * slab_bytes;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = 4 * i + (lane >> 3);
    const uint4 q = slab_get(sl, r, j & 3, j >> 2);
    const int tr = tile_row(quad, r, layout);
    if (tr < rows) *reinterpret_cast<uint4*>(out + static_cast<int64_t>(y0 + tr) * ld + x + 8 * j) = q;
  }
  __syncwarp();
}

// 2 x 32 fp32 accumulator columns of this thread's TMEM lane (two loads,
// one wait).
__device__ __forceinline__ void tmem_load32x2(uint32_t ta, uint32_t tb, float* va, float* vb) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%64];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, "
      "%48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%65];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
        "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
        "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]),
        "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]),
        "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]),
        "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]),
        "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(ta), "r"(tb)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    va[i] = __uint_as_float(r[i]);
    vb[i] = __uint_as_float(r[32 + i]);
  }
}

// CTA pairs (PAIR): the grid is made of 2-CTA clusters; rank 0 of each pair
// issues the M = 256 pair MMAs for both CTAs.  Each CTA's producer loads its
// own A rows and its half of B into its own ring and counts the bytes on
// rank 0's full barrier (rank 0 announces the pair's total); rank 0's MMA
// commits release the stage in both CTAs and signal both CTAs' accumulator
// barriers; both CTAs' epilogue warps drain their own TMEM rows and arrive on
// rank 0's accumulator-empty barrier.
template <int OP, int EPI, bool B_MN, int BN, bool PAIR, int NS>
__global__ void __launch_bounds__(kThreads, 1) bsmm_kernel(const __grid_constant__ Params p) {
  using namespace dmoe::tc;
  using PL = Plan<EPI, BN, PAIR, NS>;
  constexpr bool DUAL = PL::DUAL;
  constexpr bool A_MN = (OP == OP_DSTD || OP == OP_DSTDT);
  constexpr bool ROWWALK = (OP == OP_SDD || OP == OP_DSD || OP == OP_DSDT);
  constexpr int STAGES = PL::STAGES;
  constexpr uint32_t STAGE_BYTES = PL::STAGE_BYTES;
  constexpr uint32_t ACC_COLS = BN;
  constexpr uint32_t TMEM_COLS = 2 * ACC_COLS;
  constexpr uint32_t IDESC = idesc_bf16(PAIR ? 2 * BM : BM, BN, A_MN, B_MN);
  // M = 64 for row blocks with at most 64 tokens (the A operand's first 64
  // rows; the accumulator then fills TMEM lanes 16 q .. 16 q + 15 of each
  // lane quadrant q); single-CTA tiles only
  constexpr uint32_t IDESC64 = idesc_bf16(64, BN, A_MN, B_MN);
  // a CTA pair's lone row block: M = 128 pair MMAs, 64 rows from each CTA
  constexpr uint32_t IDESC_HALF = idesc_bf16(BM, BN, A_MN, B_MN);
  // per-UMMA_K advance of the descriptor start address (16-byte units)
  constexpr uint64_t A_STEP = A_MN ? (UMMA_K * 128) >> 4 : (UMMA_K * 2) >> 4;
  constexpr uint64_t B_STEP = B_MN ? (UMMA_K * 128) >> 4 : (UMMA_K * 2) >> 4;
  constexpr uint32_t A_LBO = A_MN ? ATOM_BYTES : 16;
  constexpr uint32_t B_LBO = B_MN ? ATOM_BYTES : 16;
  constexpr bool WALK = OP != OP_SDD;  // K walks blocks of the topology
  // output columns per tile and per epilogue warp (SwiGLU: one block, both
  // halves of the accumulator feed each output column)
  constexpr int OUT_COLS = sdd_cols_per_tile<BN, DUAL>();
  constexpr int WARP_COLS = OUT_COLS / 2;
  constexpr int NCH = WARP_COLS / 32;  // 32-column chunks per epilogue warp
  // stored forward blocks read by the backward epilogues, and how many
  // chunks of them are loaded into registers ahead of their use
  constexpr int NAUX = EPI == DMOE_EPI_GELU_BWD ? 1 : (EPI == DMOE_EPI_SWIGLU_BWD ? 2 : 0);
  constexpr int PD = NAUX == 2 && NCH > 2 ? 2 : NCH;
  static_assert(NAUX == 0 || OP == OP_SDD, "stored-block epilogues belong to the SDD");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* out_smem = smem + STAGES * STAGE_BYTES;  // [kEpiWarps][2][2 KB]
  uint32_t* pair_tab = reinterpret_cast<uint32_t*>(out_smem + PL::OUT_BYTES);  // CTA pairs over row blocks
  uint64_t* full = reinterpret_cast<uint64_t*>(out_smem + PL::OUT_BYTES + PL::TAB_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = PAIR ? static_cast<int>(cluster_ctarank()) : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull + a, 1);
      mbar_init(tempty + a, PAIR ? 2 * kEpiWarps : kEpiWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&p.map_a);
    tma_prefetch_map(&p.map_b);
  }
  if (warp == 1) {
    if (PAIR) tmem_alloc_pair(tmem_slot, TMEM_COLS);
    else tmem_alloc(tmem_slot, TMEM_COLS);
  }
  fence_before_sync();
  // a pair's barriers are initialised before either CTA touches the other's
  if (PAIR) cluster_sync();
  else __syncthreads();
  fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  // everything above overlaps the previous kernel; its outputs are read below
  dmoe::pdl_wait();
  dmoe::pdl_launch_dependents();
  int rows;  // row tiles (CTA pairs: pair rows) of the row-walking products
  if (PAIR && ROWWALK) {
    if (warp == 0) build_pair_table(p, pair_tab, lane);
    __syncthreads();
    rows = static_cast<int>(pair_tab[p.E] & 0xffffu);
  } else if (ROWWALK) {
    rows = __ldg(p.P_dev) / p.tm;
  } else {
    rows = 0;
  }
  int ntiles;
  if (ROWWALK) {
    // the row-walking products visit whole rows only (rows x tiles per row)
    const int per_row = OP == OP_SDD ? p.nb * p.blk / (NS * sdd_cols_per_tile<BN, DUAL>()) : p.ntn;
    rows = min(rows, p.max_tiles / per_row);
    ntiles = rows * per_row;
  } else {
    const int n = (OP == OP_DSTD ? p.EF / (PAIR ? 2 * BM : BM) : p.EF / (NS * BN)) * p.ntn;
    ntiles = min(n, p.max_tiles);
  }
  // tiles are dealt round-robin over the grid's CTAs, or over its pairs
  const int G = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  const int unit = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  // decode(): address arithmetic and the tile's topology loads; fin(): the
  // fields that depend on the loaded values (see finish())
  auto dec = [&](int tt) { return decode<OP, BN, DUAL, PAIR, NS>(p, tt, rows, rank, pair_tab); };
  auto fin = [&](Tile tl) {
    finish<OP, PAIR>(p, tl);
    return tl;
  };
  // NS = 2: a finished tile's second sub-tile (the first one otherwise)
  auto sub1 = [&](const Tile& tl) { return NS == 2 ? second_sub<OP, BN, DUAL>(p, tl) : tl; };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    int t = unit;
    Tile cur = t < ntiles ? fin(dec(t)) : Tile{};
    const int kslices = p.blk >> 6;  // 64-row K slices per block
    // rank 0's full barriers count both CTAs' bytes (shared::cluster address)
    const uint32_t full_pair = PAIR ? dsmem_addr(smem_u32(full), 0) : 0u;
    // lane 0 claims the next stage and issues its loads (NS = 2: A once,
    // then the B slices of both sub-tiles tl and tl1)
    auto issue = [&](const Tile& tl, const Tile& tl1, int i, int blk, int v0, int v1, int kk, int pass) {
      if (lane == 0) {
        ok = mbar_wait(empty + stage, phase ^ 1u, abort_flag);
        if (ok) {
          uint8_t* sa = smem + stage * STAGE_BYTES;
          if (PAIR) {
            if (rank == 0)
              // A: 2 x 128 rows, or 2 x 64 rows of a lone row block
              mbar_arrive_expect_tx(full + stage, (tl.single ? 1u : 2u) * SLICE_BYTES + 2u * NS * PL::B_BYTES);
            const uint32_t bar = full_pair + 8u * stage;
            auto ldp = [&](void* dst, const CUtensorMap* m, int x, int y) { tma_load_2d_pair(dst, m, bar, x, y); };
            load_slice<OP, DUAL, B_MN, BN, PAIR>(p, tl, i, blk, v0, v1, kk, pass, sa, sa + SLICE_BYTES, rank, true,
                                                 ldp);
            if (NS == 2)
              load_slice<OP, DUAL, B_MN, BN, PAIR>(p, tl1, i, blk, v0, v1, kk, pass, sa,
                                                   sa + SLICE_BYTES + PL::B_BYTES, rank, false, ldp);
          } else {
            uint64_t* bar = full + stage;
            mbar_arrive_expect_tx(bar, STAGE_BYTES);
            load_slice<OP, DUAL, B_MN, BN, PAIR>(
                p, tl, i, blk, v0, v1, kk, pass, sa, sa + SLICE_BYTES, rank, true,
                [&](void* dst, const CUtensorMap* m, int x, int y) { tma_load_2d(dst, m, bar, x, y); });
          }
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (++stage == STAGES) {
        stage = 0;
        phase ^= 1u;
      }
    };
    // topology values of up to 32 blocks of a tile, one per lane, from its
    // block `base` on
    auto fetch = [&](const Tile& tl, int base, int& m0, int& m1) {
      m0 = 0;
      m1 = 0;
      if (WALK && base + lane < tl.nblk) {
        const int j = tl.c + base + lane;
        if (OP == OP_DSD || OP == OP_DSDT) {
          m0 = __ldg(p.column_indices + j);
        } else {
          m0 = __ldg(p.block_offsets_t + j);
          m1 = __ldg(p.row_indices_t + j);
        }
      }
    };
    // tile t+G is decoded and its first index batch fetched one tile ahead,
    // tile t+2G decoded two tiles ahead, so no TMA issue waits on metadata
    Tile nxt = t + G < ntiles ? fin(dec(t + G)) : Tile{};
    int c0v, c1v;
    fetch(cur, 0, c0v, c1v);
    while (t < ntiles && ok) {
      const int t2 = t + 2 * G;
      Tile nxt2 = t2 < ntiles ? dec(t2) : Tile{};
      int n0v = 0, n1v = 0;
      if (t + G < ntiles) fetch(nxt, 0, n0v, n1v);
      const Tile cur1 = sub1(cur);
      if (!WALK) {
        for (int i = 0; i < cur.kiters && ok; ++i) issue(cur, cur1, i, 0, 0, 0, 0, 0);
      } else {
        const int passes = (OP == OP_DSDT && p.second) ? 2 : 1;
        for (int pass = 0; pass < passes && ok; ++pass) {
          for (int base = 0; base < cur.nblk && ok; base += 32) {
            int my0 = c0v, my1 = c1v;
            if (base > 0) fetch(cur, base, my0, my1);
            const int cnt = min(32, cur.nblk - base);
            for (int bb = 0; bb < cnt && ok; ++bb) {
              const int v0 = __shfl_sync(0xffffffffu, my0, bb);
              const int v1 = __shfl_sync(0xffffffffu, my1, bb);
              const int blk = cur.c + base + bb;
              for (int kk = 0; kk < kslices && ok; ++kk) issue(cur, cur1, 0, blk, v0, v1, kk, pass);
            }
          }
        }
      }
      cur = nxt;
      if (t2 < ntiles) finish<OP, PAIR>(p, nxt2);
      nxt = nxt2;
      c0v = n0v;
      c1v = n1v;
      t += G;
    }
    // CTA pair: every stage this CTA filled has been consumed (the MMA
    // commits that release them have all arrived) before it may exit
    if (PAIR && ok && lane == 0) {
      for (int s = 0; s < STAGES && ok; ++s) {
        ok = mbar_wait(empty + stage, phase ^ 1u, abort_flag);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (!ok && lane == 0) {
      dmoe::raise_error(p.err, DMOE_SITE_GEMM_WAIT | DMOE_ERR_TIMEOUT);
      *abort_flag = 1;
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // --------------------------------------------------------- MMA issue
      int stage = 0;
      uint32_t phase = 0;
      uint32_t acc = 0, acc_phase = 0;
      bool ok = true;
      int t = unit;
      Tile cur = t < ntiles ? fin(dec(t)) : Tile{};
      while (t < ntiles && ok) {
        const int tn = t + G;
        Tile nxt = tn < ntiles ? dec(tn) : Tile{};
        const int kit = cur.kiters;
        const uint32_t idesc = PAIR ? (cur.single ? IDESC_HALF : IDESC) : (cur.m64 ? IDESC64 : IDESC);
        if (NS == 2 && kit > 0) {
          // the two sub-tiles' accumulators, TMEM columns 0.. and ACC_COLS..:
          // sub-tile 0 starts once the epilogue has drained its columns of
          // the previous tile; sub-tile 1's MMAs of the first K slices wait
          // in their (still held) ring stages until its columns are drained
          // too, then catch up
          if (!mbar_wait_cluster(tempty, acc_phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          fence_after_sync();
          bool free1 = false;
          int held = 0;  // K slices 0 .. held - 1 wait for sub-tile 1's columns
          const int hstage = stage;
          auto mmas = [&](uint32_t d, int st, uint32_t boff, bool first) {
            const uint32_t sa = smem_u32(smem + st * STAGE_BYTES);
            const uint64_t adesc = sdesc_sw128(sa, A_LBO, 1024);
            const uint64_t bdesc = sdesc_sw128(sa + SLICE_BYTES + boff, B_LBO, 1024);
#pragma unroll
            for (int kk = 0; kk < BK / UMMA_K; ++kk)
              mma_bf16_pair(d, adesc + A_STEP * kk, bdesc + B_STEP * kk, idesc, (!first || kk > 0) ? 1u : 0u);
          };
          auto catch_up = [&]() {
            for (int j = 0; j < held; ++j) {
              const int st = (hstage + j) % STAGES;
              mmas(tmem_base + ACC_COLS, st, PL::B_BYTES, j == 0);
              mma_commit_pair(empty + st);
            }
            held = 0;
          };
          for (int i = 0; i < kit; ++i) {
            if (!mbar_wait(full + stage, phase, abort_flag)) {
              ok = false;
              break;
            }
            fence_after_sync();
            mmas(tmem_base, stage, 0, i == 0);
            if (!free1 && mbar_try_wait_cluster(tempty + 1, acc_phase ^ 1u)) free1 = true;
            if (!free1 && held + 1 == STAGES) {
              // every stage is held: the producer cannot go on before these
              if (!mbar_wait_cluster(tempty + 1, acc_phase ^ 1u, abort_flag)) {
                ok = false;
                break;
              }
              free1 = true;
            }
            if (free1) {
              fence_after_sync();
              catch_up();
              mmas(tmem_base + ACC_COLS, stage, PL::B_BYTES, i == 0);
              mma_commit_pair(empty + stage);
            } else {
              ++held;
            }
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          if (held > 0) {
            if (!mbar_wait_cluster(tempty + 1, acc_phase ^ 1u, abort_flag)) {
              ok = false;
              break;
            }
            fence_after_sync();
            catch_up();
          }
          mma_commit_pair(tfull);
          acc_phase ^= 1u;
        } else if (kit > 0) {
          const bool drained = PAIR ? mbar_wait_cluster(tempty + acc, acc_phase ^ 1u, abort_flag)
                                    : mbar_wait(tempty + acc, acc_phase ^ 1u, abort_flag);
          if (!drained) {
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
            const uint64_t bdesc = sdesc_sw128(sa + SLICE_BYTES, B_LBO, 1024);
#pragma unroll
            for (int kk = 0; kk < BK / UMMA_K; ++kk) {
              if (PAIR)
                mma_bf16_pair(d0, adesc + A_STEP * kk, bdesc + B_STEP * kk, idesc, (i > 0 || kk > 0) ? 1u : 0u);
              else
                mma_bf16(d0, adesc + A_STEP * kk, bdesc + B_STEP * kk, idesc, (i > 0 || kk > 0) ? 1u : 0u);
            }
            if (PAIR) mma_commit_pair(empty + stage);
            else mma_commit(empty + stage);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          if (PAIR) mma_commit_pair(tfull + acc);
          else mma_commit(tfull + acc);
          if (++acc == 2) {
            acc = 0;
            acc_phase ^= 1u;
          }
        }
        if (tn < ntiles) finish<OP, PAIR>(p, nxt);
        cur = nxt;
        t = tn;
      }
      if (!ok) {
        dmoe::raise_error(p.err, DMOE_SITE_GEMM_WAIT | DMOE_ERR_TIMEOUT);
        *abort_flag = 1;
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;                      // TMEM lanes 32*quad .. 32*quad+31
    const int col0 = ((warp - 2) >> 2) * WARP_COLS;  // this warp's output columns
    uint8_t* const slabs = out_smem + (warp - 2) * 2 * PL::SLAB;  // two 2 KB slabs of this warp
    // the accumulator-empty barriers the MMA issuer waits on (rank 0's)
    const uint32_t tempty_pair = PAIR ? dsmem_addr(smem_u32(tempty), 0) : 0u;
    // rows of a tile (64 for 64-row blocks)
    const int tile_h = (OP == OP_SDD || OP == OP_DSD || OP == OP_DSDT) ? p.tm : BM;
    uint32_t acc = 0, acc_phase = 0;
    bool ok = true;
    int t = unit;
    Tile cur = t < ntiles ? fin(dec(t)) : Tile{};
    // Chunk h of the stored forward blocks, read coalesced: lane l holds the
    // 16-byte segment (l & 3) of rows 8 i + (l >> 2), i = 0..3 (eight whole
    // 64-byte row segments per load); aux_rows() turns it into one row per
    // lane through the warp's slab.  Register slot h % PD, refilled with
    // chunk h + PD of the same tile once chunk h is consumed.  The blocks of
    // the next tile are meanwhile brought into L2 by one bulk prefetch, so
    // no load is in flight across tiles (and the register loads hit L2).
    // The chunks of a tile this warp drains: chunk h covers output columns
    // ocol(h) .. ocol(h) + 31 of the tile, read from TMEM columns tcol(h)
    // (SwiGLU: H3 hcol3 further on), of rows tile_row(quad, lane, layout).
    // A CTA pair's lone row block (M = 128 pair MMA) keeps half the columns
    // per lane half, so each warp has half as many chunks there.
    const int hw = (warp - 2) >> 2;  // which half of the lane quadrant's columns
    auto lone = [&](const Tile& tl) { return PAIR && tl.single; };
    auto layout_of = [&](const Tile& tl) { return lone(tl) ? 2 + rank : tl.m64; };
    auto nchunks = [&](const Tile& tl) { return lone(tl) ? (DUAL ? 1 : NCH / 2) : NCH; };
    auto ocol = [&](const Tile& tl, int h) {
      if (!lone(tl)) return col0 + 32 * h;
      return DUAL ? (quad >> 1) * 64 + hw * 32 : (quad >> 1) * 128 + hw * 64 + 32 * h;
    };
    auto tcol = [&](const Tile& tl, int h) {
      if (!lone(tl)) return col0 + 32 * h;
      return DUAL ? hw * 32 : hw * 64 + 32 * h;
    };
    uint4 pf0[PD][4], pf1[PD][4];
    auto prefetch = [&](const Tile& tl, int h, int slot) {
      const int c = tl.co + ocol(tl, h);
      const int lay = layout_of(tl);
      const int64_t off = ((static_cast<int64_t>(tl.a) + (c >> p.bsh)) << (2 * p.bsh)) +
                          (static_cast<int64_t>(tl.ro) << p.bsh) + (c & (p.blk - 1)) + (lane & 3) * 8;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        int tr = tile_row(quad, i * 8 + (lane >> 2), lay);
        if (tr >= p.tm) tr = 0;  // no such row in a 64-row tile: any row of it (the value is multiplied by 0)
        const int64_t o = off + (static_cast<int64_t>(tr) << p.bsh);
        pf0[slot][i] = __ldg(reinterpret_cast<const uint4*>(p.aux0 + o));
        if (NAUX == 2) pf1[slot][i] = __ldg(reinterpret_cast<const uint4*>(p.aux1 + o));
      }
    };
    auto aux_rows = [&](const uint4 (&q)[4], float* f, uint8_t* slab) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = i * 8 + (lane >> 2);
        *reinterpret_cast<uint4*>(slab + r * 64 + (((lane & 3) ^ ((r >> 1) & 3)) << 4)) = q[i];
      }
      __syncwarp();
      const int sw = (lane >> 1) & 3;
#pragma unroll
      for (int j = 0; j < 4; ++j) unpack8(*reinterpret_cast<const uint4*>(slab + lane * 64 + ((j ^ sw) << 4)), f + 8 * j);
      __syncwarp();
    };
    auto prefetch_l2 = [&](const Tile& tl) {
      if (warp == 2 && lane == 0) {
        // the tile's rows of its blocks: whole blocks when they are at most
        // as wide as the tile, else rows ro .. ro + tm - 1 of one block
        constexpr int cols = NS * sdd_cols_per_tile<BN, DUAL>();
        const uint32_t bytes = static_cast<uint32_t>(cols > p.blk ? cols : p.blk) * p.tm * 2;
        const int64_t off = (static_cast<int64_t>(tl.a) * p.blk + tl.ro) * p.blk;
        dmoe::tc::bulk_prefetch_l2(p.aux0 + off, bytes);
        if (NAUX == 2) dmoe::tc::bulk_prefetch_l2(p.aux1 + off, bytes);
      }
    };
    // this warp is done reading accumulator acc: called right after the
    // last TMEM load of a tile (or sub-tile), before that chunk's math and
    // stores, so the MMA issuer gets the columns back as early as possible
    auto release = [&]() {
      fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        if (PAIR) mbar_arrive_cluster(tempty_pair + 8u * acc);
        else mbar_arrive(tempty + acc);
      }
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    };
    if (NAUX > 0 && t < ntiles) prefetch_l2(cur);
    while (t < ntiles) {
      const int tn = t + G;
      Tile nxt = tn < ntiles ? dec(tn) : Tile{};
      if (NAUX > 0 && tn < ntiles) prefetch_l2(nxt);
      // NS = 2: sub-tile 0 from accumulator columns 0.., then sub-tile 1
      // from ACC_COLS.. (both complete at the tile's one commit); each
      // hands its columns back as soon as it is drained
      for (int sub = 0; sub < NS; ++sub) {
        const Tile cs = sub ? sub1(cur) : cur;
        const int nch = nchunks(cs);
        if (NAUX > 0) {
#pragma unroll
          for (int h = 0; h < PD; ++h)
            if (h < nch) prefetch(cs, h, h);  // in flight during the accumulator wait
        }
        if (cs.kiters == 0) {
          const float z[32] = {};
          for (int cc = col0; cc < col0 + WARP_COLS; cc += 32) {
            int x, y0;
            chunk_xy<OP, BN>(p, cs, cc, &x, &y0);
            write_chunk(slabs, lane, z, p.out[0], p.ldo, x, y0, quad, 0, tile_h);
          }
          continue;
        }
        if (sub == 0 && !(PAIR ? mbar_wait_cluster(tfull + acc, acc_phase, abort_flag)
                               : mbar_wait(tfull + acc, acc_phase, abort_flag))) {
          ok = false;
          break;
        }
        fence_after_sync();
        const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + acc * ACC_COLS;
        const int lay = layout_of(cs);
        const bool pad_lanes = lay == 1 && lane >= 16;  // an M = 64 tile's padding rows: results of zero rows
        if (EPI == DMOE_EPI_STORE) {
          // two chunks per step, both read from TMEM under one wait
          static_assert(EPI != DMOE_EPI_STORE || NCH % 2 == 0, "store epilogue walks chunk pairs");
#pragma unroll
          for (int h = 0; h < NCH; h += 2) {
            if (h >= nch) break;
            int x, y0, x2, y2;  // the two chunks may sit in different blocks (SDD)
            chunk_xy<OP, BN>(p, cs, ocol(cs, h), &x, &y0);
            chunk_xy<OP, BN>(p, cs, ocol(cs, h + 1), &x2, &y2);
            float v[32], w[32];
            tmem_load32x2(tbase + tcol(cs, h), tbase + tcol(cs, h + 1), v, w);
            if (h + 2 >= nch) release();  // the accumulator's last columns are in registers
            if (pad_lanes) {
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                v[j] = 0.f;
                w[j] = 0.f;
              }
            }
            if (x2 == x + 32 && y2 == y0) {
              write_chunk2(slabs, lane, v, w, p.out[0], p.ldo, x, y0, quad, lay, tile_h, PL::SLAB);
            } else {
              write_chunk(slabs, lane, v, p.out[0], p.ldo, x, y0, quad, lay, tile_h);
              write_chunk(slabs, lane, w, p.out[0], p.ldo, x2, y2, quad, lay, tile_h);
            }
          }
        } else {
          const int h3 = lone(cs) ? 64 : BLK;  // SwiGLU: H3's TMEM columns after H1's
#pragma unroll
          for (int h = 0; h < NCH; ++h) {
            if (h >= nch) break;
            int x, y0;
            chunk_xy<OP, BN>(p, cs, ocol(cs, h), &x, &y0);
            float v[32];
            tmem_load32(tbase + tcol(cs, h), v);
            if (EPI != DMOE_EPI_SWIGLU_FWD && h + 1 >= nch) release();
            if (pad_lanes) {
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = 0.f;
            }
            if (EPI == DMOE_EPI_GELU_FWD) {
              float g[32];
#pragma unroll
              for (int j = 0; j < 32; j += 2) {
                float2 ge, dg;
                gelu_pair(make_float2(v[j], v[j + 1]), ge, dg);
                g[j] = dg.x;  // gelu'
                g[j + 1] = dg.y;
                v[j] = ge.x;  // gelu
                v[j + 1] = ge.y;
              }
              write_chunk(slabs, lane, g, p.out[0], p.ldo, x, y0, quad, lay, tile_h);
              write_chunk(slabs, lane, v, p.out[1], p.ldo, x, y0, quad, lay, tile_h);
            } else if (EPI == DMOE_EPI_SWIGLU_FWD) {
              float v3[32], g[32];
              tmem_load32(tbase + h3 + tcol(cs, h), v3);
              if (h + 1 >= nch) release();
              if (pad_lanes) {
#pragma unroll
                for (int j = 0; j < 32; ++j) v3[j] = 0.f;
              }
#pragma unroll
              for (int j = 0; j < 32; j += 2) {
                const float2 h1 = make_float2(v[j], v[j + 1]);
                const float2 h3v = make_float2(v3[j], v3[j + 1]);
                // sigmoid(h1) = 1 / (1 + 2^(-h1 log2(e))); for large negative h1
                // the power is +inf and rcp.approx(+inf) = +0
                const float2 q = f2_mul(h1, f2_splat(-1.44269504088896341f));
                const float2 d = make_float2(1.f + ex2_approx(q.x), 1.f + ex2_approx(q.y));
                const float2 sg = make_float2(rcp_approx(d.x), rcp_approx(d.y));
                const float2 si = f2_mul(h1, sg);                                                // silu(h1) = da/dh3
                const float2 f = f2_fma(h1, f2_fma(sg, f2_splat(-1.f), f2_splat(1.f)), f2_splat(1.f));
                const float2 ga = f2_mul(f2_mul(h3v, sg), f);                                    // da/dh1
                const float2 a = f2_mul(h3v, si);                                                // a
                g[j] = ga.x;
                g[j + 1] = ga.y;
                v[j] = si.x;
                v[j + 1] = si.y;
                v3[j] = a.x;
                v3[j + 1] = a.y;
              }
              write_chunk(slabs, lane, g, p.out[0], p.ldo, x, y0, quad, lay, tile_h);
              write_chunk(slabs, lane, v, p.out[1], p.ldo, x, y0, quad, lay, tile_h);
              write_chunk(slabs, lane, v3, p.out[2], p.ldo, x, y0, quad, lay, tile_h);
            } else {  // GELU_BWD, SWIGLU_BWD: out_i = acc * aux_i
              float a[32];
              uint8_t* sl = slabs;
              aux_rows(pf0[h % PD], a, sl);
              if (NAUX == 1 && h + PD < nch) prefetch(cs, h + PD, h % PD);
#pragma unroll
              for (int j = 0; j < 32; ++j) a[j] *= v[j];
              write_chunk(sl, lane, a, p.out[0], p.ldo, x, y0, quad, lay, tile_h);
              if (NAUX == 2) {
                aux_rows(pf1[h % PD], a, sl);
                if (h + PD < nch) prefetch(cs, h + PD, h % PD);
#pragma unroll
                for (int j = 0; j < 32; ++j) a[j] *= v[j];
                write_chunk(sl, lane, a, p.out[1], p.ldo, x, y0, quad, lay, tile_h);
              }
            }
          }
        }
      }
      if (!ok) break;
      if (tn < ntiles) finish<OP, PAIR>(p, nxt);
      cur = nxt;
      t = tn;
    }
    if (!ok && lane == 0) {
      dmoe::raise_error(p.err, DMOE_SITE_GEMM_WAIT | DMOE_ERR_TIMEOUT);
      *abort_flag = 1;
    }
  }

  __syncwarp();
  fence_before_sync();
  // a CTA of a pair leaves only once the other no longer reads or signals
  // its shared memory
  if (PAIR) cluster_sync();
  else __syncthreads();
  if (warp == 1) {
    fence_after_sync();
    if (PAIR) tmem_dealloc_pair(tmem_base, TMEM_COLS);
    else tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host side

using dmoe::make_map;

// Output i [rows, cols] written by the epilogue (row-major; every output of
// a call has the same row pitch).
bool make_out_map(Params& p, int i, void* base, uint64_t rows, uint64_t cols) {
  (void)rows;
  p.out[i] = static_cast<uint16_t*>(base);
  p.ldo = static_cast<int64_t>(cols);
  return true;
}

// Block edge of a topology (0 stands for the default 128).
int topo_block(const dmoe_topology* t) { return t->block ? t->block : DMOE_BLOCK; }

bool topo_ok(const dmoe_topology* t) {
  if (!t) return false;
  const int B = topo_block(t);
  if (B != 64 && B != 128 && B != 256) return false;
  // F a multiple of 128 as well: the weight-gradient tiles cover 128 columns
  if (t->E < 1 || t->E > 1024 || t->F < B || (t->F % B) || (t->F % DMOE_BLOCK) || t->P_max < 0 || (t->P_max % B))
    return false;
  const int64_t nb = t->F / B;
  if (static_cast<int64_t>(t->nnz_max) != static_cast<int64_t>(t->P_max / B) * nb) return false;
  if (static_cast<int64_t>(t->nnz_max) * B > 0x7fffffffLL) return false;
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
  p.row_fill = t->row_fill;
  p.blk = topo_block(t);
  p.bsh = p.blk == 64 ? 6 : (p.blk == 128 ? 7 : 8);
  p.tm = p.blk < BM ? p.blk : BM;
  p.nb = t->F / p.blk;
  p.EF = t->E * t->F;
  p.E = t->E;
}

// 256-column tiles when allowed and there are still at least three waves of
// them; the setting of dmoe_set_tile_n overrides the choice.
bool wide_tiles(bool allowed, int64_t tiles256, int sms, bool prefer = true) {
  if (!allowed) return false;
  const int forced = g_tile_n.load(std::memory_order_relaxed);
  if (forced == 128) return false;
  if (forced == 256) return true;
  return prefer && tiles256 >= 3 * static_cast<int64_t>(sms);
}

// CTA pairs for a call: only with 128-row blocks, at most kPairMaxE experts
// and fewer than 2^16 row blocks (the pair-row table), 256-wide tiles the
// shape allows (`shape_ok`), and a device that can hold 2-CTA clusters of
// the kernel.  By default (dmoe_set_pair 0) DSD, DSD^T and the weight
// gradients pair wherever allowed (measured faster at every workload, e.g.
// MoE-XS DSD 40.9 -> 38.5 us, the skewed workload's DSTD 189 -> 167 us),
// the SDDs when the experts average at least three row blocks (their
// tiles were slower on pairs at MoE-XS and skewed: 51 -> 59 and 189 -> 192
// us forward); `any_rows` marks the products that pair at any row count.
// The setting forces pairs off (1) or on where allowed (2, 3).
bool use_pair(const dmoe_topology* t, bool shape_ok, bool any_rows = false) {
  const int B = topo_block(t);
  const int64_t R = t->P_max / B;
  if (B != 128 || t->E > kPairMaxE || R >= 65536 || !shape_ok || (t->F % 256)) return false;
  const int mode = g_pair.load(std::memory_order_relaxed);
  if (mode == 1) return false;
  if (mode >= 2) return true;
  return any_rows || R >= 3 * static_cast<int64_t>(t->E);
}

// Two sub-tiles per pair tile (256 x 512: the A slice of each K step feeds
// two N = 256 MMAs, so a pair loads a quarter fewer operand bytes per flop)
// for a CTA-pair call whose shape gives an even count of 256-wide column
// tiles inside each expert (`shape_ok`).  The two accumulators then fill the
// tensor memory, so the next tile's MMAs wait until the epilogue has
// drained sub-tile 0: by default only for the plain store epilogue (the
// SDD epilogues with activations, a second output or stored factors drain
// slower and made their products slower, e.g. the SwiGLU backward SDD of
// the Mixtral-shaped layer 1364 -> 1604 us), where the tile's K walk has at
// least 8 slices of 64 (the skewed workload's weight gradients, 6 slices
// per expert, were 22% slower) and the doubled tiles still make at least
// three waves over the pairs.  Setting 3 forces them wherever allowed, 1
// and 2 never.
bool use_ns2(bool shape_ok, bool store_epilogue, int64_t k_slices, int64_t tiles, int sms) {
  if (!shape_ok) return false;
  const int mode = g_pair.load(std::memory_order_relaxed);
  if (mode == 3) return true;
  if (mode != 0) return false;
  return store_epilogue && k_slices >= 8 && tiles >= 3 * static_cast<int64_t>(sms / 2);
}

// Pair rows of a routing, at most: each expert's row blocks in pairs, one
// row block alone when its count is odd.
int64_t pair_rows_max(const dmoe_topology* t) { return (t->P_max / DMOE_BLOCK + t->E) / 2; }

template <int OP, int EPI, bool B_MN, int BN, bool PAIR, int NS = 1>
dmoe_status launch(const Params& p, const dmoe::DeviceInfo& di, cudaStream_t st) {
  if (p.max_tiles <= 0) return DMOE_OK;
  auto kern = bsmm_kernel<OP, EPI, B_MN, BN, PAIR, NS>;
  const size_t smem = Plan<EPI, BN, PAIR, NS>::SMEM;
  // the dynamic shared-memory opt-in and, for pairs, the number of 2-CTA
  // clusters that fit on the device, once per instantiation and device
  static std::atomic<uint64_t> opted{0};
  static std::atomic<int> clusters[64];
  const uint64_t bit = di.device < 64 ? (uint64_t(1) << di.device) : 0;
  if (!bit || !(opted.load(std::memory_order_acquire) & bit)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return dmoe::cuda_status(e);
    if (PAIR) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(static_cast<unsigned>(di.sm_count & ~1));
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = smem;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
      if (e != cudaSuccess) return dmoe::cuda_status(e);
      if (n < 1) return DMOE_ERR_UNSUPPORTED;
      if (bit) clusters[di.device].store(n, std::memory_order_relaxed);
    }
    if (bit) opted.fetch_or(bit, std::memory_order_acq_rel);
  }
  cudaError_t e;
  if (PAIR) {
    const int n = bit ? clusters[di.device].load(std::memory_order_relaxed) : di.sm_count / 2;
    const int grid = 2 * std::min(n, p.max_tiles);
    e = dmoe::launch_pdl_cluster(kern, dim3(grid), dim3(kThreads), smem, st, 2, p);
  } else {
    const int grid = std::min(di.sm_count, p.max_tiles);
    e = dmoe::launch_pdl(kern, dim3(grid), dim3(kThreads), smem, st, p);
  }
  if (e != cudaSuccess) return dmoe::cuda_status(e);
  dmoe::count_launches(1);
  return DMOE_OK;
}

// SDD instantiation for an epilogue, B major and tile width (pairs: 256,
// or 256 x 512 with ns2).
template <int EPI>
dmoe_status launch_sdd(const Params& p, const dmoe::DeviceInfo& di, cudaStream_t st, bool b_mn, bool wide,
                       bool pair, bool ns2) {
  if (pair && ns2)
    return b_mn ? launch<OP_SDD, EPI, true, 256, true, 2>(p, di, st) : launch<OP_SDD, EPI, false, 256, true, 2>(p, di, st);
  if (pair) return b_mn ? launch<OP_SDD, EPI, true, 256, true>(p, di, st) : launch<OP_SDD, EPI, false, 256, true>(p, di, st);
  if (b_mn)
    return wide ? launch<OP_SDD, EPI, true, 256, false>(p, di, st) : launch<OP_SDD, EPI, true, 128, false>(p, di, st);
  return wide ? launch<OP_SDD, EPI, false, 256, false>(p, di, st) : launch<OP_SDD, EPI, false, 128, false>(p, di, st);
}

bool a16(const void* p) { return dmoe::aligned16(p); }

}  // namespace

DMOE_API dmoe_status dmoe_set_tile_n(int bn) {
  if (bn != 0 && bn != 128 && bn != 256) return DMOE_ERR_INVALID_ARG;
  g_tile_n.store(bn, std::memory_order_relaxed);
  return DMOE_OK;
}

DMOE_API dmoe_status dmoe_set_pair(int mode) {
  if (mode < 0 || mode > 3) return DMOE_ERR_INVALID_ARG;
  g_pair.store(mode, std::memory_order_relaxed);
  return DMOE_OK;
}

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
  const int64_t row_tiles = topo->P_max / p.tm;
  const int F = topo->F;
  p.max_tiles = static_cast<int>(row_tiles * (F / 128));
  p.aux0 = aux0;
  p.aux1 = aux1;
  p.err = di.err_word;
  // the output blocks as [nnz_max * B, B] matrices
  const uint64_t orows = static_cast<uint64_t>(topo->nnz_max) * p.blk;
  if (!make_out_map(p, 0, out0, orows, p.blk)) return DMOE_ERR_CUDA;
  if (out1 && !make_out_map(p, 1, out1, orows, p.blk)) return DMOE_ERR_CUDA;
  if (out2 && !make_out_map(p, 2, out2, orows, p.blk)) return DMOE_ERR_CUDA;
  // the backward epilogues load two stored blocks per 256-column tile; with a
  // short K they outrun the tile's MMAs, so they go wide only from K = 1024
  const bool bwd = epilogue == DMOE_EPI_GELU_BWD || epilogue == DMOE_EPI_SWIGLU_BWD;
  const bool pair = use_pair(topo, true);
  const bool wide = epilogue != DMOE_EPI_SWIGLU_FWD && !pair &&
                    wide_tiles(F % 256 == 0, row_tiles * (F / 256), di.sm_count, !bwd || K >= 1024);
  const int bn_b = wide ? 256 : 128;  // B rows loaded per K slice (K-major B; a pair CTA's half: 128)
  if (!make_map(&p.map_a, A, topo->P_max, K, BK, BM)) return DMOE_ERR_CUDA;
  if (pair && !make_map(&p.map_a64, A, topo->P_max, K, BK, BM / 2)) return DMOE_ERR_CUDA;
  if (!b_trans) {
    if (!make_map(&p.map_b, B, K, p.EF, 64, BK)) return DMOE_ERR_CUDA;
    if (epilogue == DMOE_EPI_SWIGLU_FWD && !make_map(&p.map_b2, B2, K, p.EF, 64, BK)) return DMOE_ERR_CUDA;
  } else {
    if (!make_map(&p.map_b, B, p.EF, K, BK, bn_b)) return DMOE_ERR_CUDA;
  }
  cudaStream_t st = dmoe::as_stream(stream);
  // pair rows x (128 output columns for SwiGLU's W1 | W3 tiles, else 256;
  // twice that with two sub-tiles)
  const int sub_cols = epilogue == DMOE_EPI_SWIGLU_FWD ? 128 : 256;
  const bool ns2 = pair && use_ns2(F % (2 * sub_cols) == 0, epilogue == DMOE_EPI_STORE, K / BK,
                                   pair_rows_max(topo) * (F / (2 * sub_cols)), di.sm_count);
  if (pair) p.max_tiles = static_cast<int>(pair_rows_max(topo) * (F / ((ns2 ? 2 : 1) * sub_cols)));
  if (epilogue == DMOE_EPI_SWIGLU_FWD) {
    if (ns2) return launch<OP_SDD, DMOE_EPI_SWIGLU_FWD, true, 256, true, 2>(p, di, st);
    return pair ? launch<OP_SDD, DMOE_EPI_SWIGLU_FWD, true, 256, true>(p, di, st)
                : launch<OP_SDD, DMOE_EPI_SWIGLU_FWD, true, 256, false>(p, di, st);
  }
  if (wide) p.max_tiles = static_cast<int>(row_tiles * (F / 256));
  switch (epilogue) {
    case DMOE_EPI_GELU_FWD: return launch_sdd<DMOE_EPI_GELU_FWD>(p, di, st, !b_trans, wide, pair, ns2);
    case DMOE_EPI_GELU_BWD: return launch_sdd<DMOE_EPI_GELU_BWD>(p, di, st, !b_trans, wide, pair, ns2);
    case DMOE_EPI_SWIGLU_BWD: return launch_sdd<DMOE_EPI_SWIGLU_BWD>(p, di, st, !b_trans, wide, pair, ns2);
    default: return launch_sdd<DMOE_EPI_STORE>(p, di, st, !b_trans, wide, pair, ns2);
  }
}

DMOE_API dmoe_status dmoe_dsd(const dmoe_topology* topo, const uint16_t* S, const uint16_t* Bm, int N, uint16_t* C,
                              dmoe_stream_t stream) {
  if (!topo_ok(topo) || N < BLK || (N % BLK) || !S || !Bm || !C) return DMOE_ERR_INVALID_ARG;
  if (!a16(S) || !a16(Bm) || !a16(C)) return DMOE_ERR_INVALID_ARG;
  dmoe::DeviceInfo di;
  dmoe_status s = dmoe::device_info(&di);
  if (s != DMOE_OK) return s;
  if (topo->nnz_max == 0) return DMOE_OK;
  Params p{};
  fill_topo(p, topo);
  p.N = N;
  if (!make_out_map(p, 0, C, topo->P_max, N)) return DMOE_ERR_CUDA;
  p.err = di.err_word;
  const int64_t rows = topo->P_max / p.tm;
  const bool pair = use_pair(topo, N % 256 == 0, true);
  const bool wide = pair || wide_tiles(N % 256 == 0, rows * (N / 256), di.sm_count);
  const bool ns2 = pair && use_ns2(N % 512 == 0, true, topo->F / BK, pair_rows_max(topo) * (N / 512), di.sm_count);
  p.ntn = N / (ns2 ? 512 : (wide ? 256 : 128));
  p.max_tiles = static_cast<int>((pair ? pair_rows_max(topo) : rows) * p.ntn);
  if (!make_map(&p.map_a, S, static_cast<uint64_t>(topo->nnz_max) * p.blk, p.blk, BK, BM)) return DMOE_ERR_CUDA;
  if (pair && !make_map(&p.map_a64, S, static_cast<uint64_t>(topo->nnz_max) * p.blk, p.blk, BK, BM / 2))
    return DMOE_ERR_CUDA;
  if (!make_map(&p.map_b, Bm, p.EF, N, 64, BK)) return DMOE_ERR_CUDA;
  cudaStream_t st = dmoe::as_stream(stream);
  if (ns2) return launch<OP_DSD, DMOE_EPI_STORE, true, 256, true, 2>(p, di, st);
  if (pair) return launch<OP_DSD, DMOE_EPI_STORE, true, 256, true>(p, di, st);
  return wide ? launch<OP_DSD, DMOE_EPI_STORE, true, 256, false>(p, di, st)
              : launch<OP_DSD, DMOE_EPI_STORE, true, 128, false>(p, di, st);
}

DMOE_API dmoe_status dmoe_dsd_t(const dmoe_topology* topo, const uint16_t* S, const uint16_t* Bm,
                                const uint16_t* S2, const uint16_t* Bm2, int N, uint16_t* C, dmoe_stream_t stream) {
  if (!topo_ok(topo) || N < BLK || (N % BLK) || !S || !Bm || !C) return DMOE_ERR_INVALID_ARG;
  if ((S2 == nullptr) != (Bm2 == nullptr)) return DMOE_ERR_INVALID_ARG;
  if (!a16(S) || !a16(Bm) || !a16(S2) || !a16(Bm2) || !a16(C)) return DMOE_ERR_INVALID_ARG;
  dmoe::DeviceInfo di;
  dmoe_status s = dmoe::device_info(&di);
  if (s != DMOE_OK) return s;
  if (topo->nnz_max == 0) return DMOE_OK;
  Params p{};
  fill_topo(p, topo);
  p.N = N;
  p.second = S2 ? 1 : 0;
  if (!make_out_map(p, 0, C, topo->P_max, N)) return DMOE_ERR_CUDA;
  p.err = di.err_word;
  const int64_t rows = topo->P_max / p.tm;
  const bool pair = use_pair(topo, N % 256 == 0, true);
  const bool wide = pair || wide_tiles(N % 256 == 0, rows * (N / 256), di.sm_count);
  const bool ns2 = pair && use_ns2(N % 512 == 0, true, (topo->F / BK) * (S2 ? 2 : 1),
                                   pair_rows_max(topo) * (N / 512), di.sm_count);
  p.ntn = N / (ns2 ? 512 : (wide ? 256 : 128));
  p.max_tiles = static_cast<int>((pair ? pair_rows_max(topo) : rows) * p.ntn);
  const int bn = pair ? 128 : (wide ? 256 : 128);  // B rows per K slice (a pair CTA loads its half)
  const uint64_t srows = static_cast<uint64_t>(topo->nnz_max) * p.blk;
  if (!make_map(&p.map_a, S, srows, p.blk, BK, BM)) return DMOE_ERR_CUDA;
  if (pair && !make_map(&p.map_a64, S, srows, p.blk, BK, BM / 2)) return DMOE_ERR_CUDA;
  if (!make_map(&p.map_b, Bm, N, p.EF, BK, bn)) return DMOE_ERR_CUDA;
  if (S2) {
    if (!make_map(&p.map_a2, S2, srows, p.blk, BK, BM)) return DMOE_ERR_CUDA;
    if (pair && !make_map(&p.map_a2_64, S2, srows, p.blk, BK, BM / 2)) return DMOE_ERR_CUDA;
    if (!make_map(&p.map_b2, Bm2, N, p.EF, BK, bn)) return DMOE_ERR_CUDA;
  }
  cudaStream_t st = dmoe::as_stream(stream);
  if (ns2) return launch<OP_DSDT, DMOE_EPI_STORE, false, 256, true, 2>(p, di, st);
  if (pair) return launch<OP_DSDT, DMOE_EPI_STORE, false, 256, true>(p, di, st);
  return wide ? launch<OP_DSDT, DMOE_EPI_STORE, false, 256, false>(p, di, st)
              : launch<OP_DSDT, DMOE_EPI_STORE, false, 128, false>(p, di, st);
}

DMOE_API dmoe_status dmoe_dstd(const dmoe_topology* topo, const uint16_t* S, const uint16_t* D, int N, int c_trans,
                               uint16_t* C, dmoe_stream_t stream) {
  if (!topo_ok(topo) || N < BLK || (N % BLK) || !S || !D || !C) return DMOE_ERR_INVALID_ARG;
  if (!a16(S) || !a16(D) || !a16(C)) return DMOE_ERR_INVALID_ARG;
  dmoe::DeviceInfo di;
  dmoe_status s = dmoe::device_info(&di);
  if (s != DMOE_OK) return s;
  Params p{};
  fill_topo(p, topo);
  p.N = N;
  // the weight gradient [E*F, N], or [N, E*F] transposed
  if (!(c_trans ? make_out_map(p, 0, C, N, p.EF) : make_out_map(p, 0, C, p.EF, N)))
    return DMOE_ERR_CUDA;
  p.err = di.err_word;
  const uint64_t srows = static_cast<uint64_t>(topo->nnz_max > 0 ? topo->nnz_max : 1) * p.blk;
  const uint64_t drows = topo->P_max > 0 ? topo->P_max : BM;
  const int64_t cols = p.EF / BM;  // 128-column groups of the weight columns
  cudaStream_t st = dmoe::as_stream(stream);
  // with no rows at all every tile has K = 0 and only zeros are written;
  // the maps then describe valid placeholder extents that are never read
  // CTA pairs: 256 weight columns (two column blocks of one expert when
  // F % 256 == 0) x 256 dense columns per pair tile
  const bool pair = use_pair(topo, N % 256 == 0, true);
  // K slices of an average expert's tile (its rows, padded, over 64)
  const int64_t k_avg = topo->P_max / topo->E / BK;
  if (!c_trans) {
    const bool wide = pair || wide_tiles(N % 256 == 0, cols * (N / 256), di.sm_count);
    const bool ns2 = pair && use_ns2(N % 512 == 0, true, k_avg, (cols / 2) * (N / 512), di.sm_count);
    p.ntn = N / (ns2 ? 512 : (wide ? 256 : 128));
    p.max_tiles = static_cast<int>((pair ? cols / 2 : cols) * p.ntn);
    if (!make_map(&p.map_a, S, srows, p.blk, 64, BK)) return DMOE_ERR_CUDA;
    if (!make_map(&p.map_b, D, drows, N, 64, BK)) return DMOE_ERR_CUDA;
    if (ns2) return launch<OP_DSTD, DMOE_EPI_STORE, true, 256, true, 2>(p, di, st);
    if (pair) return launch<OP_DSTD, DMOE_EPI_STORE, true, 256, true>(p, di, st);
    return wide ? launch<OP_DSTD, DMOE_EPI_STORE, true, 256, false>(p, di, st)
                : launch<OP_DSTD, DMOE_EPI_STORE, true, 128, false>(p, di, st);
  }
  // DSTD^T: a 256-column tile stays inside one expert when F % 256 == 0
  const bool wide = pair || wide_tiles(topo->F % 256 == 0, (cols / 2) * (N / 128), di.sm_count);
  // two sub-tiles: 512 weight columns of one expert when F % 512 == 0
  const bool ns2 = pair && use_ns2(topo->F % 512 == 0, true, k_avg, (cols / 4) * (N / 256), di.sm_count);
  p.ntn = pair ? N / 256 : N / BM;  // m tiles (pairs of them)
  p.max_tiles = static_cast<int>((ns2 ? cols / 4 : (wide ? cols / 2 : cols)) * p.ntn);
  if (!make_map(&p.map_a, D, drows, N, 64, BK)) return DMOE_ERR_CUDA;
  if (!make_map(&p.map_b, S, srows, p.blk, 64, BK)) return DMOE_ERR_CUDA;
  if (ns2) return launch<OP_DSTDT, DMOE_EPI_STORE, true, 256, true, 2>(p, di, st);
  if (pair) return launch<OP_DSTDT, DMOE_EPI_STORE, true, 256, true>(p, di, st);
  return wide ? launch<OP_DSTDT, DMOE_EPI_STORE, true, 256, false>(p, di, st)
              : launch<OP_DSTDT, DMOE_EPI_STORE, true, 128, false>(p, di, st);
}
