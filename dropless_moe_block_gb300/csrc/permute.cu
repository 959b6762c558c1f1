// a2: permute + pad in one kernel (George Lin's blog, MoE training post,
// section 1.4: tokens are reordered from batch order into expert-grouped order
// and every group is padded to a multiple of the 128-row block, section 1.3).
//
// One cooperative launch of G = #SMs blocks, each owning a contiguous chunk of
// the A = T*k assignments:
//   1. the chunk's first source rows start loading into shared memory
//      (cp.async), and one warp gives every assignment of the chunk its
//      expert and its stable rank among the chunk's assignments to that
//      expert (warp match + popc, ascending a), which also yields the
//      chunk's expert histogram -> ws
//   2. grid barrier (bounded spin)
//   3. every block reduces the G histograms: totals T_e, its own prefix per
//      expert, padded offsets (block 0 publishes them)
//   4. dest_row / src_of_row: padded offset + the block's prefix + the rank
//   5. pad rows are zeroed (spread evenly over all blocks), then the rows
//      are copied with 16-byte vectors, the staged ones from shared memory.
// The copy moves T*k*d*2 bytes in and out and dominates: HBM-bound.
#include <cooperative_groups.h>

#include <atomic>
#include <mutex>

#include "route.cuh"
#include "topology.cuh"

namespace {

__device__ __forceinline__ int64_t lmin(int64_t a, int64_t b) { return a < b ? a : b; }

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxE = 1024;
constexpr int kDestCap = 4096;  // chunk destinations kept in shared memory
constexpr int kRowBatch = 8;    // rows each warp moves per batch (loads in flight together)
constexpr int kScratchInts = 4096;     // prefix partials: [groups][E] totals and prefixes, 2 x 2048
constexpr int kScratchBytes = kScratchInts * 4;
constexpr int kStageMax = 176 * 1024;  // dynamic shared memory for the chunk's staged source rows

struct WsLayout {
  unsigned int* arrive;  // grid barrier: arrivals
  unsigned int* depart;  // grid barrier: departures (last one resets both)
  int32_t* hist;         // [G][E]
};

constexpr size_t kWsHeader = 256;

__host__ __device__ inline WsLayout ws_layout(void* ws) {
  char* b = static_cast<char*>(ws);
  return WsLayout{reinterpret_cast<unsigned int*>(b), reinterpret_cast<unsigned int*>(b + 128),
                  reinterpret_cast<int32_t*>(b + kWsHeader)};
}

// Self-resetting grid barrier of the G blocks of the grid: each block
// waits until `target` arrivals (G; the self-test asks for one more, which
// never comes) or until limit_ns has passed, polling the counter with
// acquire loads (no sleep between polls, no fence after the wait).  Every
// block departs later, with grid_barrier_depart, whether its wait completed
// or gave up, and the last of the G to depart (all of them have then arrived
// and left the spin) puts both counters back to 0, so the workspace is ready
// for the next call after a timeout too; departing at the end of the block's
// work keeps that atomic round trip off the path between the barrier and
// the prefix.  Returns false when this block's wait gave up.
__device__ __forceinline__ unsigned int ld_acquire_gpu(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ bool grid_barrier(unsigned int* arrive, unsigned int target, uint64_t limit_ns, int32_t* err) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    __threadfence();
    atomicAdd(arrive, 1u);
    const uint64_t t0 = dmoe::globaltimer_ns();
    uint32_t it = 0;
    while (ld_acquire_gpu(arrive) < target) {
      if ((++it & 63u) == 0 && dmoe::globaltimer_ns() - t0 > limit_ns) {
        ok = 0;
        dmoe::raise_error(err, DMOE_SITE_PERMUTE_BARRIER | DMOE_ERR_TIMEOUT);
        break;
      }
    }
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

// A block leaves the barrier once it no longer needs it (at the end of its
// work, or when its wait gave up); the last of the G blocks to leave (all of
// them have then passed or abandoned the spin) puts both counters back to 0.
__device__ __forceinline__ void grid_barrier_depart(unsigned int* arrive, unsigned int* depart) {
  if (threadIdx.x == 0 && atomicAdd(depart, 1u) == gridDim.x - 1) {
    atomicExch(arrive, 0u);
    atomicExch(depart, 0u);
  }
}

// Per-block shared state of the permutation.
struct PermuteSmem {
  int32_t cnt[kMaxE];       // histogram, then the block's prefix (running rank base when not pre-ranked)
  int32_t tot[kMaxE];       // T_e
  int32_t off[kMaxE + 1];   // padded offsets
  int32_t padc[kMaxE + 1];  // exclusive scan of pad rows
  int32_t dest[kDestCap];   // this chunk's (expert, rank) pairs, then its destination rows (if it fits)
};

// The chunk's first `n` source rows, loaded by cp.async into shared memory
// (one commit group, waited for before the copy), `nvec` 16-byte vectors each.
struct Staged {
  const uint4* rows;
  int n;
};

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// (expert, rank inside the chunk) of an assignment, kept in one word: the
// expert in the low 10 bits (E <= 1024), the rank above; -1 for an expert
// id outside [0, E).
constexpr int kExpertBits = 10;

// Phases 2-5 for this block's chunk [a0, a1) of the assignments, whose
// expert histogram is in sm.cnt (every block of the grid calls it).
// Returns false when the grid barrier gave up (the error word is set).
__device__ bool permute_tail(PermuteSmem& sm, const uint16_t* __restrict__ x,
                             const int32_t* __restrict__ expert_idx, int d, int E, int k, int B, int P_max,
                             int32_t* __restrict__ tokens_per_expert, int32_t* __restrict__ padded_offsets,
                             int32_t* __restrict__ dest_row, int32_t* __restrict__ src_of_row,
                             uint16_t* __restrict__ x_perm, int32_t* __restrict__ P_dev, const WsLayout& L,
                             int32_t* err, int64_t a0, int64_t a1, int32_t* scratch, bool ranked = false,
                             Staged staged = Staged{}, unsigned int barrier_extra = 0,
                             uint64_t limit_ns = dmoe::kWaitLimitNs) {
  int32_t* s_cnt = sm.cnt;
  int32_t* s_tot = sm.tot;
  int32_t* s_off = sm.off;
  int32_t* s_padc = sm.padc;
  int32_t* s_dest = sm.dest;
  const int G = gridDim.x;
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  for (int e = tid; e < E; e += kThreads) L.hist[static_cast<int64_t>(b) * E + e] = s_cnt[e];

  // 2. all histograms visible
  if (!grid_barrier(L.arrive, G + barrier_extra, limit_ns, err)) {
    grid_barrier_depart(L.arrive, L.depart);
    return false;
  }

  // 3. totals and this block's prefix per expert.  Thread groups split the
  //    G histograms (16-byte loads of 4 experts when E % 4 == 0), every
  //    thread keeping several loads in flight; each group's partial sums go
  //    to the scratch ([groups][E] each, groups * E <= 2048) and are added
  //    up per expert in a second pass (no contended shared atomics).
  {
    const int vec = (E % 4 == 0) ? 4 : 1;
    const int lanes = (E + vec - 1) / vec;  // threads per histogram row
    const int groups = lanes >= kThreads ? 1 : kThreads / lanes;
    const int g = tid / lanes;
    int32_t* ptot = scratch;
    int32_t* ppre = scratch + kScratchInts / 2;
    if (g < groups) {
      for (int q = tid % lanes; q < lanes; q += (groups == 1 ? kThreads : lanes)) {
        int tot[4] = {0, 0, 0, 0}, pre[4] = {0, 0, 0, 0};
        if (vec == 4) {
          const int4* h4 = reinterpret_cast<const int4*>(L.hist);
#pragma unroll 8
          for (int bb = g; bb < G; bb += groups) {
            const int4 h = __ldcg(h4 + static_cast<int64_t>(bb) * lanes + q);
            const int m = bb < b;
            tot[0] += h.x; tot[1] += h.y; tot[2] += h.z; tot[3] += h.w;
            pre[0] += m * h.x; pre[1] += m * h.y; pre[2] += m * h.z; pre[3] += m * h.w;
          }
        } else {
#pragma unroll 8
          for (int bb = g; bb < G; bb += groups) {
            const int h = __ldcg(L.hist + static_cast<int64_t>(bb) * E + q);
            tot[0] += h;
            pre[0] += (bb < b) * h;
          }
        }
        for (int i = 0; i < vec; ++i) {
          ptot[g * E + q * vec + i] = tot[i];
          ppre[g * E + q * vec + i] = pre[i];
        }
      }
    }
    __syncthreads();
    for (int e = tid; e < E; e += kThreads) {
      int32_t te = 0, pe = 0;
      for (int gg = 0; gg < groups; ++gg) {
        te += ptot[gg * E + e];
        pe += ppre[gg * E + e];
      }
      s_tot[e] = te;
      s_cnt[e] = pe;
    }
  }
  __syncthreads();
  if (tid < 32) {
    // exclusive scans of padded sizes and of pad rows, 32 experts at a time
    int32_t carry_off = 0, carry_pad = 0;
    for (int base = 0; base < E; base += 32) {
      const int e = base + tid;
      const int32_t te = e < E ? s_tot[e] : 0;
      const int32_t pe = (te + B - 1) / B * B;
      int32_t io = pe, ip = pe - te;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t uo = __shfl_up_sync(0xffffffffu, io, o);
        const int32_t up = __shfl_up_sync(0xffffffffu, ip, o);
        if (tid >= o) {
          io += uo;
          ip += up;
        }
      }
      if (e < E) {
        s_off[e + 1] = carry_off + io;
        s_padc[e + 1] = carry_pad + ip;
      }
      carry_off += __shfl_sync(0xffffffffu, io, 31);
      carry_pad += __shfl_sync(0xffffffffu, ip, 31);
    }
    if (tid == 0) {
      s_off[0] = 0;
      s_padc[0] = 0;
    }
  }
  __syncthreads();
  const int32_t P = s_off[E];
  if (b == 0) {
    for (int e = tid; e < E; e += kThreads) tokens_per_expert[e] = s_tot[e];
    for (int e = tid; e <= E; e += kThreads) padded_offsets[e] = s_off[e];
    if (tid == 0) *P_dev = P;
  }

  // 4. destination rows of this chunk.  Pre-ranked: every assignment's
  //    (expert, rank) is in s_dest, so each thread places its own; else one
  //    warp ranks the chunk 32 assignments at a time (stable, ascending a).
  const int rows = static_cast<int>(a1 - a0);
  const bool dest_in_smem = rows <= kDestCap;
  if (ranked) {
    for (int i = tid; i < rows; i += kThreads) {
      const int32_t er = s_dest[i];
      int32_t dest = -1;
      if (er >= 0) {
        const int e = er & ((1 << kExpertBits) - 1);
        dest = s_off[e] + s_cnt[e] + (er >> kExpertBits);
      }
      const int64_t a = a0 + i;
      dest_row[a] = dest;
      if (dest >= 0) src_of_row[dest] = static_cast<int32_t>(a);
      s_dest[i] = dest;
    }
  } else if (tid < 32) {
    const unsigned lt = (1u << tid) - 1u;
    for (int64_t base = a0; base < a1; base += 32) {
      const int64_t a = base + tid;
      int e = a < a1 ? expert_idx[a] : -1;
      if (e >= E) e = -1;
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      const int rank = __popc(peers & lt);
      const int cnt = __popc(peers);
      int32_t dest = -1;
      if (e >= 0) dest = s_off[e] + s_cnt[e] + rank;
      __syncwarp();
      if (e >= 0 && rank == 0) s_cnt[e] += cnt;
      __syncwarp();
      if (a < a1) {
        dest_row[a] = dest;
        if (dest >= 0) src_of_row[dest] = static_cast<int32_t>(a);
        if (dest_in_smem) s_dest[a - a0] = dest;
      }
    }
  }
  __syncthreads();

  // 5a. zero pad rows and mark them in src_of_row; pad row indices are
  //     spread evenly over the blocks, one warp per row (stores only, so
  //     they go out ahead of the copy's loads)
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int nvec = d >> 3;
  const uint4* xv = reinterpret_cast<const uint4*>(x);
  uint4* pv = reinterpret_cast<uint4*>(x_perm);
  const int32_t npad = s_padc[E];
  const int32_t pchunk = (npad + G - 1) / G;
  const int32_t q0 = min(npad, b * pchunk);
  const int32_t q1 = min(npad, q0 + pchunk);
  for (int32_t q = q0 + warp; q < q1; q += kWarps) {
    // expert owning pad index q: last e with s_padc[e] <= q
    int lo = 0, hi = E - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_padc[mid] <= q) lo = mid;
      else hi = mid - 1;
    }
    const int32_t row = s_off[lo] + s_tot[lo] + (q - s_padc[lo]);
    uint4* dstp = pv + static_cast<int64_t>(row) * nvec;
    for (int v = lane; v < nvec; v += 32) dstp[v] = make_uint4(0, 0, 0, 0);
    if (lane == 0) src_of_row[row] = -1;
  }

  // 5b. rows staged in shared memory: 16-byte vectors of one row per warp
  if (staged.n > 0) {
    cp_async_wait_all();
    __syncthreads();
    for (int r = warp; r < staged.n; r += kWarps) {
      const int32_t dest = dest_in_smem ? s_dest[r] : dest_row[a0 + r];
      if (dest < 0) continue;
      uint4* dstp = pv + static_cast<int64_t>(dest) * nvec;
      const uint4* srcp = staged.rows + static_cast<int64_t>(r) * nvec;
      for (int v = lane; v < nvec; v += 32) dstp[v] = srcp[v];
    }
  }

  // 5c. the other rows from global memory: warp per row, 16-byte vectors
  //     per lane, kRowBatch rows per warp with all their loads in flight
  //     together
  for (int r0 = staged.n + warp * kRowBatch; r0 < rows; r0 += kWarps * kRowBatch) {
    int64_t src[kRowBatch], dst[kRowBatch];
#pragma unroll
    for (int j = 0; j < kRowBatch; ++j) {
      const int r = r0 + j;
      const int32_t dest = r < rows ? (dest_in_smem ? s_dest[r] : dest_row[a0 + r]) : -1;
      src[j] = dest >= 0 ? ((a0 + r) / k) * nvec : -1;
      dst[j] = dest >= 0 ? static_cast<int64_t>(dest) * nvec : -1;
    }
    for (int v = lane; v < nvec; v += 32) {
      uint4 u[kRowBatch];
#pragma unroll
      for (int j = 0; j < kRowBatch; ++j)
        if (src[j] >= 0) u[j] = __ldg(xv + src[j] + v);
#pragma unroll
      for (int j = 0; j < kRowBatch; ++j)
        if (dst[j] >= 0) pv[dst[j] + v] = u[j];
    }
  }
  // rows P .. P_max-1 hold nothing
  for (int64_t r = P + static_cast<int64_t>(b) * kThreads + tid; r < P_max; r += static_cast<int64_t>(G) * kThreads)
    src_of_row[r] = -1;
  grid_barrier_depart(L.arrive, L.depart);
  return true;
}

__global__ void __launch_bounds__(kThreads)
    permute_pad_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ expert_idx, int T, int d,
                       int E, int k, int B, int P_max, int32_t* __restrict__ tokens_per_expert,
                       int32_t* __restrict__ padded_offsets, int32_t* __restrict__ dest_row,
                       int32_t* __restrict__ src_of_row, uint16_t* __restrict__ x_perm, int32_t* __restrict__ P_dev,
                       void* ws, int32_t* err, int stage_bytes, unsigned int barrier_extra, uint64_t limit_ns) {
  __shared__ PermuteSmem sm;
  // dynamic shared memory: the prefix scratch, then stage_bytes for source rows
  extern __shared__ uint4 dyn[];
  int32_t* scratch = reinterpret_cast<int32_t*>(dyn);
  uint4* stage = dyn + kScratchBytes / 16;
  dmoe::pdl_wait();
  dmoe::pdl_launch_dependents();
  const int G = gridDim.x;
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  const int64_t A = static_cast<int64_t>(T) * k;
  const int64_t chunk = (A + G - 1) / G;
  const int64_t a0 = lmin(A, b * chunk);
  const int64_t a1 = lmin(A, a0 + chunk);
  const int rows = static_cast<int>(a1 - a0);

  // 1a. the chunk's expert ids are loaded (registers), then the chunk's
  //     source rows start moving into shared memory (they do not depend on
  //     the routing, and arrive while the grid barrier and the prefix run);
  //     the id loads go first so that they do not queue behind the rows
  constexpr int kIds = kDestCap / kThreads;
  const bool ranked = rows <= kDestCap;
  int ids[kIds];
  if (ranked) {
#pragma unroll
    for (int j = 0; j < kIds; ++j) {
      const int i = tid + j * kThreads;
      ids[j] = i < rows ? expert_idx[a0 + i] : 0;
    }
  }
  const int nvec = d >> 3;
  Staged st;
  st.rows = stage;
  st.n = min(rows, stage_bytes / (nvec * 16));
  if (st.n > 0) {
    const uint4* xv = reinterpret_cast<const uint4*>(x);
    for (int i = tid; i < st.n * nvec; i += kThreads) {
      const int r = i / nvec;
      const int v = i - r * nvec;
      cp_async16(stage + i, xv + ((a0 + r) / k) * nvec + v);
    }
    cp_async_commit();
  }
  // 1b. histogram; with the chunk's destinations in shared memory, also the
  //     (expert, rank) of each assignment: the expert ids land in s_dest,
  //     then one warp ranks them 32 at a time (stable, ascending a)
  for (int e = tid; e < E; e += kThreads) sm.cnt[e] = 0;
  if (ranked) {
#pragma unroll
    for (int j = 0; j < kIds; ++j) {
      const int i = tid + j * kThreads;
      if (i < rows) {
        const int e = ids[j];
        const bool good = e >= 0 && e < E;
        if (!good) dmoe::raise_error(err, DMOE_SITE_PERMUTE_EXPERT_ID | DMOE_ERR_DEVICE);
        sm.dest[i] = good ? e : -1;
      }
    }
    __syncthreads();
    if (tid < 32) {
      const unsigned lt = (1u << tid) - 1u;
      for (int base = 0; base < rows; base += 32) {
        const int i = base + tid;
        const int e = i < rows ? sm.dest[i] : -1;
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        const int rank = __popc(peers & lt);
        int32_t er = -1;
        if (e >= 0) er = ((sm.cnt[e] + rank) << kExpertBits) | e;
        __syncwarp();
        if (e >= 0 && rank == 0) sm.cnt[e] += __popc(peers);
        __syncwarp();
        if (i < rows) sm.dest[i] = er;
      }
    }
  } else {
    __syncthreads();
    for (int64_t a = a0 + tid; a < a1; a += kThreads) {
      const int e = expert_idx[a];
      if (e >= 0 && e < E) atomicAdd(&sm.cnt[e], 1);
      else dmoe::raise_error(err, DMOE_SITE_PERMUTE_EXPERT_ID | DMOE_ERR_DEVICE);
    }
  }
  __syncthreads();
  permute_tail(sm, x, expert_idx, d, E, k, B, P_max, tokens_per_expert, padded_offsets, dest_row, src_of_row,
               x_perm, P_dev, ws_layout(ws), err, a0, a1, scratch, ranked, st, barrier_extra, limit_ns);
}

// a1 + a2 (+ a3) in one cooperative launch (the dispatch of the layer):
// block b routes tokens [b*tc, (b+1)*tc) (tc = ceil(T / G)) one warp per
// token, counting its picks in the shared histogram, then runs the
// permutation on the assignments of those tokens, and finally (with_topo)
// every block writes its share of the topology from the padded offsets it
// already holds.
template <int NPL>
__global__ void __launch_bounds__(kThreads)
    dispatch_kernel(const float* __restrict__ logits, const uint16_t* __restrict__ x, int T, int d, int E, int k,
                    int renorm, int P_max, int32_t* __restrict__ expert_idx, float* __restrict__ gate_w,
                    int32_t* __restrict__ tokens_per_expert, int32_t* __restrict__ padded_offsets,
                    int32_t* __restrict__ dest_row, int32_t* __restrict__ src_of_row, uint16_t* __restrict__ x_perm,
                    int32_t* __restrict__ P_dev, const dmoe_topology topo, int with_topo, void* ws, int32_t* err) {
  __shared__ PermuteSmem sm;
  extern __shared__ int32_t scratch[];  // kScratchBytes: the prefix partials
  dmoe::pdl_wait();
  dmoe::pdl_launch_dependents();
  const int G = gridDim.x;
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int64_t tc = (static_cast<int64_t>(T) + G - 1) / G;
  const int64_t t0 = lmin(T, b * tc);
  const int64_t t1 = lmin(T, t0 + tc);

  for (int e = tid; e < E; e += kThreads) sm.cnt[e] = 0;
  __syncthreads();
  for (int64_t t = t0 + warp; t < t1; t += kWarps)
    dmoe::route_token<NPL>(logits + t * E, E, k, renorm, expert_idx + t * k, gate_w + t * k, lane,
                           [&](int e) { atomicAdd(&sm.cnt[e], 1); });
  __syncthreads();
  const int B = with_topo && topo.block ? topo.block : DMOE_BLOCK;
  if (!permute_tail(sm, x, expert_idx, d, E, k, B, P_max, tokens_per_expert, padded_offsets, dest_row, src_of_row,
                    x_perm, P_dev, ws_layout(ws), err, t0 * k, t1 * k, scratch) ||
      !with_topo)
    return;
  const int nb = topo.F / B;
  const int R_max = topo.P_max / B;
  if (b == 0 && tid == 0) {
    const int32_t P = sm.off[E];
    *topo.nnz_dev = min(P / B, R_max) * nb;
    *topo.P_dev = P;
  }
  dmoe::topology_entries(sm.off, sm.tot, E, B, nb, R_max, topo.nnz_max, topo.row_fill, topo.row_offsets,
                         topo.column_indices, topo.row_indices, topo.column_offsets_t, topo.row_indices_t,
                         topo.block_offsets_t,
                         static_cast<int64_t>(b) * kThreads + tid, static_cast<int64_t>(G) * kThreads);
}

// Opts a kernel of this file into `bytes` of dynamic shared memory, once per
// kernel and device (the static PermuteSmem plus the scratch already pass
// the default limit).
template <auto KERN>
dmoe_status smem_optin(int bytes, const dmoe::DeviceInfo& di) {
  static std::atomic<uint64_t> opted{0};  // one set of device bits per kernel
  const uint64_t bit = di.device < 64 ? (uint64_t(1) << di.device) : 0;
  if (bit && (opted.load(std::memory_order_acquire) & bit)) return DMOE_OK;
  const cudaError_t e = cudaFuncSetAttribute(KERN, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return dmoe::cuda_status(e);
  if (bit) opted.fetch_or(bit, std::memory_order_acq_rel);
  return DMOE_OK;
}

}  // namespace

DMOE_API size_t dmoe_permute_pad_workspace_size(int T, int k, int E) {
  (void)T;
  (void)k;
  dmoe::DeviceInfo di;
  if (dmoe::device_info(&di) != DMOE_OK) return 0;
  if (E < 1) return 0;
  return kWsHeader + static_cast<size_t>(di.sm_count) * static_cast<size_t>(E) * sizeof(int32_t);
}

namespace {

// Checks and launches permute_pad_kernel; barrier_extra / limit_ns are 0 /
// the library's wait limit except in the barrier self-test.
dmoe_status launch_permute(const uint16_t* x, const int32_t* expert_idx, int T, int d, int E, int k, int block,
                           int P_max, int32_t* tokens_per_expert, int32_t* padded_offsets, int32_t* dest_row,
                           int32_t* src_of_row, uint16_t* x_perm, int32_t* P_dev, void* ws, size_t ws_bytes,
                           dmoe_stream_t stream, unsigned int barrier_extra, uint64_t limit_ns) {
  if (T < 0 || d < 8 || (d & 7) || E < 1 || E > kMaxE || k < 1 || k > E) return DMOE_ERR_INVALID_ARG;
  if (block != 64 && block != 128 && block != 256) return DMOE_ERR_INVALID_ARG;
  if (static_cast<int64_t>(T) * k > 0x7fffffffLL) return DMOE_ERR_INVALID_ARG;
  if (P_max < dmoe_padded_rows_max_block(T, k, E, block) || (P_max % block)) return DMOE_ERR_INVALID_ARG;
  if (!tokens_per_expert || !padded_offsets || !P_dev || !ws) return DMOE_ERR_INVALID_ARG;
  if (T > 0 && (!x || !expert_idx || !dest_row || !src_of_row || !x_perm)) return DMOE_ERR_INVALID_ARG;
  if (P_max > 0 && (!src_of_row || !x_perm)) return DMOE_ERR_INVALID_ARG;
  if (!dmoe::aligned16(x) || !dmoe::aligned16(x_perm) || !dmoe::aligned16(ws)) return DMOE_ERR_INVALID_ARG;
  dmoe::DeviceInfo di;
  dmoe_status s = dmoe::device_info(&di);
  if (s != DMOE_OK) return s;
  const size_t need = kWsHeader + static_cast<size_t>(di.sm_count) * E * sizeof(int32_t);
  if (ws_bytes < need) return DMOE_ERR_INVALID_ARG;

  const int G = di.sm_count;
  // shared memory for the chunk's source rows when all of them fit in
  // kStageMax (opt-in once per device); larger chunks stream through
  // registers only
  const int64_t chunk_rows = (static_cast<int64_t>(T) * k + G - 1) / G;
  const int stage_bytes = chunk_rows * d * 2 <= kStageMax ? static_cast<int>(chunk_rows * d * 2) : 0;
  const int dyn_bytes = kScratchBytes + stage_bytes;
  s = smem_optin<permute_pad_kernel>(kScratchBytes + kStageMax, di);
  if (s != DMOE_OK) return s;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, permute_pad_kernel, kThreads, dyn_bytes) != cudaSuccess)
    return dmoe::cuda_status(cudaErrorUnknown);
  if (per_sm < 1) return DMOE_ERR_UNSUPPORTED;
  int32_t* err = di.err_word;
  // cooperative (the grid barrier needs every block resident) and with
  // programmatic dependent launch (its prologue may overlap the router's tail)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(G);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = dyn_bytes;
  cfg.stream = dmoe::as_stream(stream);
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = cudaLaunchKernelEx(&cfg, permute_pad_kernel, x, expert_idx, T, d, E, k, block, P_max,
                                     tokens_per_expert, padded_offsets, dest_row, src_of_row, x_perm, P_dev, ws, err,
                                     stage_bytes, barrier_extra, limit_ns);
  if (e != cudaSuccess) return dmoe::cuda_status(e);
  dmoe::count_launches(1);
  return DMOE_OK;
}

}  // namespace

DMOE_API dmoe_status dmoe_permute_pad_block(const uint16_t* x, const int32_t* expert_idx, int T, int d, int E,
                                            int k, int block, int P_max, int32_t* tokens_per_expert,
                                            int32_t* padded_offsets, int32_t* dest_row, int32_t* src_of_row,
                                            uint16_t* x_perm, int32_t* P_dev, void* ws, size_t ws_bytes,
                                            dmoe_stream_t stream) {
  return launch_permute(x, expert_idx, T, d, E, k, block, P_max, tokens_per_expert, padded_offsets, dest_row,
                        src_of_row, x_perm, P_dev, ws, ws_bytes, stream, 0u, dmoe::kWaitLimitNs);
}

DMOE_API dmoe_status dmoe_selftest_permute_timeout(const uint16_t* x, const int32_t* expert_idx, int T, int d,
                                                   int E, int k, int P_max, int32_t* tokens_per_expert,
                                                   int32_t* padded_offsets, int32_t* dest_row, int32_t* src_of_row,
                                                   uint16_t* x_perm, int32_t* P_dev, void* ws, size_t ws_bytes,
                                                   int64_t limit_ns, dmoe_stream_t stream) {
  if (limit_ns < 1000 || limit_ns > static_cast<int64_t>(dmoe::kWaitLimitNs)) return DMOE_ERR_INVALID_ARG;
  return launch_permute(x, expert_idx, T, d, E, k, DMOE_BLOCK, P_max, tokens_per_expert, padded_offsets, dest_row,
                        src_of_row, x_perm, P_dev, ws, ws_bytes, stream, 1u, static_cast<uint64_t>(limit_ns));
}

DMOE_API dmoe_status dmoe_permute_pad(const uint16_t* x, const int32_t* expert_idx, int T, int d, int E,
                                      int k, int P_max, int32_t* tokens_per_expert, int32_t* padded_offsets,
                                      int32_t* dest_row, int32_t* src_of_row, uint16_t* x_perm,
                                      int32_t* P_dev, void* ws, size_t ws_bytes, dmoe_stream_t stream) {
  return dmoe_permute_pad_block(x, expert_idx, T, d, E, k, DMOE_BLOCK, P_max, tokens_per_expert, padded_offsets,
                                dest_row, src_of_row, x_perm, P_dev, ws, ws_bytes, stream);
}

namespace {

template <int NPL>
dmoe_status launch_dispatch(void** args, const dmoe::DeviceInfo& di, cudaStream_t st) {
  const int G = di.sm_count;
  const dmoe_status so = smem_optin<dispatch_kernel<NPL>>(kScratchBytes, di);
  if (so != DMOE_OK) return so;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dispatch_kernel<NPL>, kThreads, kScratchBytes) !=
      cudaSuccess)
    return dmoe::cuda_status(cudaErrorUnknown);
  if (per_sm < 1) return DMOE_ERR_UNSUPPORTED;
  // cooperative and with programmatic dependent launch, as the permutation
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(G);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kScratchBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(dispatch_kernel<NPL>), args);
  if (e != cudaSuccess) return dmoe::cuda_status(e);
  dmoe::count_launches(1);
  return DMOE_OK;
}

}  // namespace

DMOE_API dmoe_status dmoe_dispatch(const float* logits, const uint16_t* x, int T, int d, int E, int k,
                                   int renormalize, int P_max, int32_t* expert_idx, float* gate_w,
                                   int32_t* tokens_per_expert, int32_t* padded_offsets, int32_t* dest_row,
                                   int32_t* src_of_row, uint16_t* x_perm, int32_t* P_dev, const dmoe_topology* topo,
                                   void* ws, size_t ws_bytes, dmoe_stream_t stream) {
  if (T < 0 || d < 8 || (d & 7) || E < 1 || E > kMaxE || k < 1 || k > E) return DMOE_ERR_INVALID_ARG;
  if (static_cast<int64_t>(T) * k > 0x7fffffffLL) return DMOE_ERR_INVALID_ARG;
  const int B = topo && topo->block ? topo->block : DMOE_BLOCK;
  if (B != 64 && B != 128 && B != 256) return DMOE_ERR_INVALID_ARG;
  if (P_max < dmoe_padded_rows_max_block(T, k, E, B) || (P_max % B)) return DMOE_ERR_INVALID_ARG;
  dmoe_topology tv{};
  if (topo) {
    const dmoe_topology& t = *topo;
    if (t.E != E || t.P_max != P_max || t.F < B || (t.F % B) || (t.F % DMOE_BLOCK)) return DMOE_ERR_INVALID_ARG;
    const int64_t nb = t.F / B;
    const int64_t R_max = P_max / B;
    if (static_cast<int64_t>(t.nnz_max) != R_max * nb || R_max * nb > 0x7fffffffLL ||
        static_cast<int64_t>(E) * nb > 0x7ffffffeLL)
      return DMOE_ERR_INVALID_ARG;
    if (!t.row_offsets || !t.column_offsets_t || !t.nnz_dev || !t.P_dev) return DMOE_ERR_INVALID_ARG;
    if (t.nnz_max > 0 && (!t.column_indices || !t.row_indices || !t.row_indices_t || !t.block_offsets_t))
      return DMOE_ERR_INVALID_ARG;
    tv = t;
  }
  const int with_topo = topo ? 1 : 0;
  if (!tokens_per_expert || !padded_offsets || !P_dev || !ws) return DMOE_ERR_INVALID_ARG;
  if (T > 0 && (!logits || !x || !expert_idx || !gate_w || !dest_row || !src_of_row || !x_perm))
    return DMOE_ERR_INVALID_ARG;
  if (P_max > 0 && (!src_of_row || !x_perm)) return DMOE_ERR_INVALID_ARG;
  if (!dmoe::aligned16(x) || !dmoe::aligned16(x_perm) || !dmoe::aligned16(ws)) return DMOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(logits) | reinterpret_cast<uintptr_t>(expert_idx) |
       reinterpret_cast<uintptr_t>(gate_w)) & 3u)
    return DMOE_ERR_INVALID_ARG;
  dmoe::DeviceInfo di;
  dmoe_status s = dmoe::device_info(&di);
  if (s != DMOE_OK) return s;
  const size_t need = kWsHeader + static_cast<size_t>(di.sm_count) * E * sizeof(int32_t);
  if (ws_bytes < need) return DMOE_ERR_INVALID_ARG;

  const int r = renormalize ? 1 : 0;
  int32_t* err = di.err_word;
  void* args[] = {(void*)&logits,     (void*)&x,         (void*)&T,          (void*)&d,
                  (void*)&E,          (void*)&k,         (void*)&r,          (void*)&P_max,
                  (void*)&expert_idx, (void*)&gate_w,    (void*)&tokens_per_expert, (void*)&padded_offsets,
                  (void*)&dest_row,   (void*)&src_of_row, (void*)&x_perm,    (void*)&P_dev,
                  (void*)&tv,         (void*)&with_topo, (void*)&ws,         (void*)&err};
  cudaStream_t st = dmoe::as_stream(stream);
  if (E <= 32) return launch_dispatch<1>(args, di, st);
  if (E <= 64) return launch_dispatch<2>(args, di, st);
  if (E <= 128) return launch_dispatch<4>(args, di, st);
  if (E <= 256) return launch_dispatch<8>(args, di, st);
  if (E <= 512) return launch_dispatch<16>(args, di, st);
  return launch_dispatch<32>(args, di, st);
}

// ---------------------------------------------------------------------------
// Permute + pad for callers that cannot allocate device memory.
//
// Some callers of this library only ever hand it the tensors it reads and
// writes: a plugin interface that passes inputs and outputs but no
// workspace, a runtime whose device memory is planned once at start-up with
// no allocator reachable from the call site, or a latency-critical path
// where a cudaMalloc (which may synchronise the device) is not acceptable.
// For them this entry point runs the same permute_pad_kernel, but its
// scratch (barrier counters + per-block histograms) lives in the static
// device array below instead of a caller-provided workspace.
//
// Limits: E <= kNoAllocMaxE experts and a device with at most
// kNoAllocMaxBlocks SMs (the cooperative grid has one block per SM); the
// array is 256 + 256*256*4 bytes = 262,400 bytes, which every GPU that
// loads the library keeps until the process exits.
// ---------------------------------------------------------------------------

namespace {

constexpr int kNoAllocMaxE = 256;
constexpr int kNoAllocMaxBlocks = 256;
constexpr size_t kNoAllocBytes = kWsHeader + static_cast<size_t>(kNoAllocMaxBlocks) * kNoAllocMaxE * sizeof(int32_t);

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

// Device address of g_noalloc_scratch, looked up once per device with that
// device current (in host code the symbol itself is only a host-side handle).
constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kNoAllocMaxDevices];

dmoe_status noalloc_scratch(int dev, void** out) {
  if (dev < 0 || dev >= kNoAllocMaxDevices) return DMOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) return dmoe::cuda_status(e == cudaSuccess ? cudaErrorUnknown : e);
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return DMOE_OK;
}

}  // namespace

DMOE_API dmoe_status dmoe_permute_pad_noalloc(const uint16_t* x, const int32_t* expert_idx, int T, int d, int E,
                                              int k, int P_max, int32_t* tokens_per_expert,
                                              int32_t* padded_offsets, int32_t* dest_row, int32_t* src_of_row,
                                              uint16_t* x_perm, int32_t* P_dev, dmoe_stream_t stream) {
  if (T < 0 || d < 8 || (d & 7) || E < 1 || k < 1 || k > E) return DMOE_ERR_INVALID_ARG;
  if (E > kNoAllocMaxE) return DMOE_ERR_INVALID_ARG;  // beyond the static scratch
  if (static_cast<int64_t>(T) * k > 0x7fffffffLL) return DMOE_ERR_INVALID_ARG;
  if (P_max < dmoe_padded_rows_max(T, k, E) || (P_max % DMOE_BLOCK)) return DMOE_ERR_INVALID_ARG;
  if (!tokens_per_expert || !padded_offsets || !P_dev) return DMOE_ERR_INVALID_ARG;
  if (T > 0 && (!x || !expert_idx || !dest_row || !src_of_row || !x_perm)) return DMOE_ERR_INVALID_ARG;
  if (P_max > 0 && (!src_of_row || !x_perm)) return DMOE_ERR_INVALID_ARG;
  if (!dmoe::aligned16(x) || !dmoe::aligned16(x_perm)) return DMOE_ERR_INVALID_ARG;
  dmoe::DeviceInfo di;
  dmoe_status s = dmoe::device_info(&di);
  if (s != DMOE_OK) return s;
  if (di.sm_count > kNoAllocMaxBlocks) return DMOE_ERR_INVALID_ARG;  // beyond the static scratch
  void* ws = nullptr;
  s = noalloc_scratch(di.device, &ws);
  if (s != DMOE_OK) return s;
  cudaStream_t st = dmoe::as_stream(stream);
  // the barrier counters must start at zero; the histograms are rewritten
  // by every call before they are read
  cudaError_t e = cudaMemsetAsync(ws, 0, kWsHeader, st);
  if (e != cudaSuccess) return dmoe::cuda_status(e);
  int per_sm = 0;
  s = smem_optin<permute_pad_kernel>(kScratchBytes + kStageMax, di);
  if (s != DMOE_OK) return s;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, permute_pad_kernel, kThreads, kScratchBytes) !=
      cudaSuccess)
    return dmoe::cuda_status(cudaErrorUnknown);
  if (per_sm < 1) return DMOE_ERR_UNSUPPORTED;
  const int G = di.sm_count;
  int32_t* err = di.err_word;
  int block = DMOE_BLOCK;
  int stage_bytes = 0;  // no staged rows: the static shared memory only
  unsigned int barrier_extra = 0;
  uint64_t limit_ns = dmoe::kWaitLimitNs;
  void* args[] = {(void*)&x,          (void*)&expert_idx, (void*)&T,          (void*)&d,
                  (void*)&E,          (void*)&k,          (void*)&block,      (void*)&P_max,
                  (void*)&tokens_per_expert, (void*)&padded_offsets, (void*)&dest_row, (void*)&src_of_row,
                  (void*)&x_perm,     (void*)&P_dev,      (void*)&ws,         (void*)&err,
                  (void*)&stage_bytes, (void*)&barrier_extra, (void*)&limit_ns};
  e = cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(permute_pad_kernel), dim3(G), dim3(kThreads), args,
                                  kScratchBytes, st);
  if (e != cudaSuccess) return dmoe::cuda_status(e);
  dmoe::count_launches(1);
  return DMOE_OK;
}
