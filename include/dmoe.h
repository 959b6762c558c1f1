/*
 * dmoe.h -- C ABI of the GB300 (sm_103a) dropless MoE block.
 *
 * The operations follow section 1 ("MegaBlocks") of George Lin's blog post on
 * MoE training systems (MegaBlocks / FlexMoE / fused comm-comp):
 *   1.1  a gate network routes every token to experts, with no capacity;
 *   1.2  the experts' two-layer MLP is one block-sparse product:
 *        SDD (layer 1) -> activation -> DSD (layer 2);
 *   1.3  128x128 blocks, groups padded to a multiple of 128, hybrid BCSR-COO
 *        topology plus a transpose index; DSTD gives the weight gradients;
 *   1.4  one kernel permutes and pads, one kernel builds the topology.
 *
 * Notation: T tokens, d model width, E experts, F hidden width of one expert
 * (a multiple of 128), k experts per token, A = T*k assignments
 * (a = t*k + j), T_e tokens of expert e, P = sum_e ceil(T_e/128)*128 padded
 * rows, R = P/128 row blocks, nb = F/128 column blocks per expert,
 * nnz = R*nb nonzero blocks.
 *
 * Conventions shared by every call:
 *  - bf16 tensors are passed as uint16_t bit patterns; fp32 as float;
 *    indices as int32_t.  All matrices are row-major and dense
 *    (leading dimension = number of columns).
 *  - Every pointer argument is a DEVICE pointer owned by the caller, unless
 *    stated otherwise.  The library allocates no device memory.  Scratch is
 *    passed in as (ws, ws_bytes) with a *_workspace_size query.
 *  - Every call takes a CUDA stream (cudaStream_t passed as void*; NULL is
 *    the legacy default stream) and is asynchronous.  Sizes that depend on
 *    the routing (P, nnz) stay on the device; no call synchronises.
 *  - Device pointers must be 16-byte aligned; sizes are validated on the
 *    host before anything is launched.  An invalid argument returns
 *    DMOE_ERR_INVALID_ARG and launches nothing.
 *  - Kernels never trap.  A problem found on the device (an expert id out
 *    of range, a wait that gave up) sets a sticky device error word that
 *    dmoe_get_error() reads.
 *  - On first use on a device the library looks up, with that device
 *    current, the device addresses of its own device globals (the error
 *    word, the no-alloc scratch) and keeps them for the life of the
 *    process; a cudaDeviceReset in the calling process invalidates them,
 *    and the library must not be called after one.
 *  - Calls are stateless and may be issued from several host threads,
 *    with two exceptions: dmoe_set_tile_n and dmoe_set_pair change
 *    process-wide settings, and dmoe_permute_pad_noalloc works in one
 *    static scratch area (its entry says how concurrent calls must be
 *    serialised).
 */
#ifndef DMOE_H_
#define DMOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DMOE_BLOCK 128

typedef void* dmoe_stream_t; /* a cudaStream_t */

typedef enum dmoe_status {
  DMOE_OK = 0,
  DMOE_ERR_INVALID_ARG = 1, /* bad pointer, size or alignment; nothing launched */
  DMOE_ERR_UNSUPPORTED = 2, /* valid request this build does not handle (e.g. not sm_103) */
  DMOE_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed */
  DMOE_ERR_TIMEOUT = 4,     /* (device word) a bounded wait gave up */
  DMOE_ERR_DEVICE = 5       /* (device word) bad data found on the device */
} dmoe_status;

/* Device error word codes (low 8 bits = dmoe_status, upper bits = site). */
#define DMOE_SITE_PERMUTE_BARRIER (1 << 8)
#define DMOE_SITE_PERMUTE_EXPERT_ID (2 << 8)
#define DMOE_SITE_GEMM_WAIT (3 << 8)
#define DMOE_SITE_COMBINE_INDEX (4 << 8)
#define DMOE_SITE_ROUTE_INDEX (5 << 8)
#define DMOE_SITE_SELFTEST (6 << 8)

/* Block-sparse topology (section 1.3, hybrid BCSR-COO + transpose index).
 * Plain device arrays, all int32, owned by the caller; filled by
 * dmoe_build_topology and read by the block-sparse products.
 *   row_offsets      [P_max/128 + 1]  BCSR: blocks of row r are
 *                                     row_offsets[r] .. row_offsets[r+1]-1
 *   column_indices   [nnz_max]        BCSR column block of each block
 *   row_indices      [nnz_max]        materialised row block (COO view)
 *   column_offsets_t [E*F/128 + 1]    transpose index: blocks of column c are
 *                                     entries column_offsets_t[c] .. [c+1]-1
 *   row_indices_t    [nnz_max]        row block of each transposed entry
 *   block_offsets_t  [nnz_max]        BCSR position of each transposed entry
 *   nnz_dev, P_dev   [1]              nnz and P of the current routing
 *   row_fill         [P_max/128]      rows of row block r that hold tokens
 *                                     (1..128; 0 past P/128); may be NULL,
 *                                     which the products read as "all full"
 * Host fields: E, F (multiple of 128 and of the block), P_max (multiple of
 * the block, >= P), nnz_max = (P_max/B)*(F/B), block B = 64, 128 or 256 (0
 * means 128: the page's choice; 64 and 256 re-run its block-size ablation).
 * With block B every "128" below reads B: blocks are B x B, row block r is
 * rows B r .. B r + B - 1.  Entries past nnz (or past P/128+1 for
 * row_offsets) are written with the value at the end of the valid range
 * (row_offsets) or left untouched (the others). */
typedef struct dmoe_topology {
  int32_t* row_offsets;
  int32_t* column_indices;
  int32_t* row_indices;
  int32_t* column_offsets_t;
  int32_t* row_indices_t;
  int32_t* block_offsets_t;
  int32_t* nnz_dev;
  int32_t* P_dev;
  int32_t* row_fill;
  int32_t E;
  int32_t F;
  int32_t P_max;
  int32_t nnz_max;
  int32_t block;
} dmoe_topology;

/* SDD epilogues (section 1.2: the activation between SDD and DSD is fused
 * into SDD).  acc = the fp32 block product; outputs are bf16 blocks.  The
 * forward epilogues store, besides the activation, its partial derivatives
 * with respect to the pre-activations (computed in fp32 from the
 * accumulators), which is all the backward pass needs of them:
 *   STORE:       out0 = acc
 *   GELU_FWD:    h = acc:  out0 = gelu'(h), out1 = gelu(h)
 *   SWIGLU_FWD:  needs B2; h1 = A*B, h3 = A*B2, a = silu(h1) * h3:
 *                out0 = da/dh1 = h3 * silu'(h1), out1 = da/dh3 = silu(h1),
 *                out2 = a
 *   GELU_BWD:    aux0 = the GELU_FWD out0 blocks;  out0 = acc * aux0
 *   SWIGLU_BWD:  aux0, aux1 = the SWIGLU_FWD out0, out1 blocks;
 *                out0 = acc * aux0 (dh1), out1 = acc * aux1 (dh3)
 * gelu is the exact erf form x*Phi(x), gelu' = Phi(x) + x*phi(x);
 * silu(x) = x*sigmoid(x), silu' = sigmoid(x) * (1 + x*(1 - sigmoid(x))). */
typedef enum dmoe_epilogue {
  DMOE_EPI_STORE = 0,
  DMOE_EPI_GELU_FWD = 1,
  DMOE_EPI_SWIGLU_FWD = 2,
  DMOE_EPI_GELU_BWD = 3,
  DMOE_EPI_SWIGLU_BWD = 4
} dmoe_epilogue;

/* ---------------------------------------------------------------- utility */

/* Library version string (static storage). */
const char* dmoe_version(void);

/* Message for a status code (static storage). */
const char* dmoe_status_string(int status);

/* Largest P any routing of T tokens x k slots over E experts can produce:
 * 128*floor((T*k + 127*min(E, T*k)) / 128).  Host-only, no CUDA call. */
int64_t dmoe_padded_rows_max(int T, int k, int E);

/* The same bound for groups padded to a multiple of `block` (64, 128 or
 * 256; -1 for other values). */
int64_t dmoe_padded_rows_max_block(int T, int k, int E, int block);

/* Read the device error word of the current device (synchronous: waits for
 * the device).  *code_out receives 0 or (site | dmoe_status); with clear != 0
 * the word is reset to 0.  Returns DMOE_OK or DMOE_ERR_CUDA. */
dmoe_status dmoe_get_error(int32_t* code_out, int clear);

/* Number of kernels this library has launched in this process (host
 * counter, for accounting). */
int64_t dmoe_launch_count(void);

/* Diagnostic of the failure path every bounded wait of the library takes:
 * one warp waits on a device flag that nothing ever sets, with the same
 * %globaltimer-bounded spin as the kernels' waits (whose limit is 1 s), for
 * limit_ns nanoseconds; then it sets DMOE_SITE_SELFTEST | DMOE_ERR_TIMEOUT in
 * the device error word and returns, leaving the context usable.  Requires
 * 1000 <= limit_ns <= 1e9 (DMOE_ERR_INVALID_ARG otherwise, nothing
 * launched).  Asynchronous on `stream`: the timeout shows in the error word
 * once the stream has reached it (dmoe_get_error synchronises). */
dmoe_status dmoe_selftest_bounded_wait(int64_t limit_ns, dmoe_stream_t stream);

/* Tile width of the block-sparse products (dmoe_sdd, dmoe_dsd, dmoe_dsd_t,
 * dmoe_dstd): 0 (default) lets each call choose 128 or 256 output columns
 * per tile from its shape (256 when the shape allows it and still gives at
 * least three waves of tiles); 128 or 256 forces that width wherever the
 * shape allows it.  Process-wide; returns DMOE_ERR_INVALID_ARG for other
 * values.  Host-only, no CUDA call. */
dmoe_status dmoe_set_tile_n(int bn);

/* CTA pairs in the block-sparse products.  A paired call launches 2-CTA
 * thread-block clusters: the two CTAs (two SMs) run one M = 256 x N = 256
 * tile as a single tensor-core operation (tcgen05 cta_group::2), each
 * holding its own 128 rows of A and half of B in shared memory.  Rows pair
 * within an expert: SDD / DSD / DSD^T take two row blocks of one expert
 * (an expert's odd last row block is split over the pair, 64 rows per
 * CTA, as one M = 128 operation), DSTD two
 * column blocks, DSTD^T two 128-row slices of the dense operand.  A call
 * can pair with 128-row blocks, E <= 256, fewer than 65536 row blocks, F a
 * multiple of 256 and, for DSD / DSD^T / DSTD, N a multiple of 256.
 * A pair tile can also be 256 x 512: two N = 256 operations per K step
 * share the step's A slice, so the pair loads a quarter fewer operand
 * bytes per flop (the two accumulators then fill the SM's tensor memory,
 * and the epilogue hands each half back as soon as it is drained).  That
 * needs an even count of 256-wide column tiles inside each expert: F a
 * multiple of 512 (SDD except SwiGLU, DSTD^T), N a multiple of 512 (DSD,
 * DSD^T, DSTD); the SwiGLU SDD (128 output columns per sub-tile) only F a
 * multiple of 256.
 *   mode 0 (default): DSD, DSD^T and DSTD pair wherever allowed; the SDDs
 *                     when the experts average at least three row blocks
 *                     (P_max / 128 >= 3 E);
 *                     256 x 512 pair tiles for the plain store epilogue
 *                     (DSD, DSD^T, DSTD, the store SDD) where allowed, the
 *                     tile's K walk has at least 8 slices of 64 (for the
 *                     weight gradients: an average expert's padded rows /
 *                     64) and the wider tiles still make at least three
 *                     waves over the device's SM pairs;
 *   mode 1:           never pair;
 *   mode 2:           pair wherever allowed, 256 x 256 pair tiles only;
 *   mode 3:           pair wherever allowed, 256 x 512 pair tiles wherever
 *                     allowed.
 * Results are the same either way (within the products' rounding).
 * Process-wide; returns DMOE_ERR_INVALID_ARG for other modes.  Host-only,
 * no CUDA call. */
dmoe_status dmoe_set_pair(int mode);

/* ------------------------------------------------------------ a1 routing */

/* Top-k router (section 1.1).  For every token t: softmax over the E fp32
 * logits; the k experts with the largest logits (equal logits: lower expert
 * id first) in descending order go to expert_idx[t*k + j]; gate_w[t*k + j]
 * is the softmax probability of that expert, divided by the sum of the k
 * chosen probabilities when renormalize != 0.  Logits must be finite.
 *   logits      [T, E] fp32 (device, read)
 *   expert_idx  [T, k] int32 (device, written)
 *   gate_w      [T, k] fp32  (device, written)
 * Requires 1 <= k <= E <= 1024, T >= 0 (T == 0 launches nothing). */
dmoe_status dmoe_route_topk(const float* logits, int T, int E, int k, int renormalize,
                            int32_t* expert_idx, float* gate_w, dmoe_stream_t stream);

/* Router backward: gradient of the gate weights of dmoe_route_topk with
 * respect to the logits (section 1.1's gate network, trained through the
 * weights it hands the combine; the top-k choice itself is piecewise
 * constant and carries no gradient).  For token t, with p the softmax of
 * its logits, c = sum_j d_gate[j] * gate_w[j] and G_e the d_gate of the
 * slot holding expert e (0 if e was not chosen):
 *   renormalize == 0:  d_logits[t, e] = p_e (G_e - c)
 *   renormalize != 0:  d_logits[t, e] = gate_w(e) (G_e - c) if e was
 *                      chosen, else 0.
 *   logits, expert_idx, gate_w: as given to / returned by dmoe_route_topk
 *   d_gate   [T, k] fp32 (e.g. from dmoe_combine_backward)
 *   d_logits [T, E] fp32 (written)
 * An expert id outside [0, E) is skipped and sets
 * DMOE_SITE_ROUTE_INDEX | DMOE_ERR_DEVICE. */
dmoe_status dmoe_route_topk_backward(const float* logits, const int32_t* expert_idx,
                                     const float* gate_w, const float* d_gate, int T, int E,
                                     int k, int renormalize, float* d_logits,
                                     dmoe_stream_t stream);

/* Linear gate fused into the router (section 1.1's gate network; the
 * optional fusion of the router GEMM into the router).  For every token t:
 *   logits[t, e] = sum_c x[t, c] * w_gate[e, c]   (bf16 products, fp32 sum
 *                                                   on the tensor cores)
 * then exactly what dmoe_route_topk does with those fp32 logits (same
 * choice, tie rule, weights and renormalisation, bit for bit).
 *   x           [T, d] bf16, row-major (device, read; 16-byte aligned)
 *   w_gate      [E, d] bf16, row-major: one d-vector per expert (device,
 *               read; 16-byte aligned)
 *   logits      [T, E] fp32 (device, written; what dmoe_route_topk_backward
 *               later needs)
 *   expert_idx  [T, k] int32, gate_w [T, k] fp32 (device, written)
 * Requires d a multiple of 64, 1 <= k <= E <= 256, T >= 0 (T == 0 launches
 * nothing).  A bounded wait that gives up sets
 * DMOE_SITE_GEMM_WAIT | DMOE_ERR_TIMEOUT and leaves the outputs unwritten.
 * The gradients of the gate's own GEMM (d_logits . w_gate into dx and
 * d_logits^T . x for w_gate) are plain dense GEMMs left to the caller. */
dmoe_status dmoe_gate_route_topk(const uint16_t* x, const uint16_t* w_gate, int T, int d, int E, int k,
                                 int renormalize, float* logits, int32_t* expert_idx, float* gate_w,
                                 dmoe_stream_t stream);

/* ------------------------------------------------------- a2 permute + pad */

/* Bytes of scratch dmoe_permute_pad needs on the current device. */
size_t dmoe_permute_pad_workspace_size(int T, int k, int E);

/* Permute + pad in one kernel (section 1.4; padding rule of section 1.3).
 * Groups the A assignments by expert -- stable: ascending a inside a
 * group -- and pads every group to a multiple of 128 rows.
 *   x                 [T, d] bf16 (read)
 *   expert_idx        [T, k] int32 (read), values in [0, E)
 *   tokens_per_expert [E] int32: T_e
 *   padded_offsets    [E+1] int32: exclusive scan of ceil(T_e/128)*128
 *   dest_row          [A] int32: row of assignment a
 *   src_of_row        [P_max] int32: assignment held by row p, -1 for pad
 *                     rows and for rows P .. P_max-1
 *   x_perm            [P_max, d] bf16: row p = x[src_of_row[p] / k];
 *                     pad rows are zero; rows P .. P_max-1 untouched
 *   P_dev             [1] int32: P
 *   ws, ws_bytes      scratch of dmoe_permute_pad_workspace_size() bytes,
 *                     zero-filled before its first use; every call leaves
 *                     it ready for the next one (its barrier counters back
 *                     at zero), including a call whose grid barrier timed
 *                     out: every block departs the barrier, waited or not,
 *                     and the last one resets the counters.
 * P_max must be >= dmoe_padded_rows_max(T, k, E).  d must be a multiple of
 * 8.  An expert id outside [0, E) sets the device error word
 * (DMOE_SITE_PERMUTE_EXPERT_ID | DMOE_ERR_DEVICE); that assignment is then
 * not placed (dest_row = -1).  Uses a cooperative launch with a bounded
 * grid-wide barrier (DMOE_SITE_PERMUTE_BARRIER | DMOE_ERR_TIMEOUT on
 * expiry).  Calls sharing one ws must not overlap. */
dmoe_status dmoe_permute_pad(const uint16_t* x, const int32_t* expert_idx, int T, int d, int E,
                             int k, int P_max, int32_t* tokens_per_expert,
                             int32_t* padded_offsets, int32_t* dest_row, int32_t* src_of_row,
                             uint16_t* x_perm, int32_t* P_dev, void* ws, size_t ws_bytes,
                             dmoe_stream_t stream);

/* dmoe_permute_pad with every group padded to a multiple of `block` (64,
 * 128 or 256: the block sizes of the page's ablation) instead of 128.
 * P_max >= dmoe_padded_rows_max_block(T, k, E, block), a multiple of block. */
dmoe_status dmoe_permute_pad_block(const uint16_t* x, const int32_t* expert_idx, int T, int d, int E, int k,
                                   int block, int P_max, int32_t* tokens_per_expert, int32_t* padded_offsets,
                                   int32_t* dest_row, int32_t* src_of_row, uint16_t* x_perm, int32_t* P_dev,
                                   void* ws, size_t ws_bytes, dmoe_stream_t stream);

/* Diagnostic of the permutation's grid barrier on its failure path: runs
 * dmoe_permute_pad on the given arguments (the same checks, outputs and
 * workspace) with a barrier that waits for one arrival more than the grid
 * has, so every block gives up after limit_ns nanoseconds, records
 * DMOE_SITE_PERMUTE_BARRIER | DMOE_ERR_TIMEOUT in the device error word and
 * writes nothing past the barrier (the outputs are left as they were,
 * except ws).  The workspace is left ready for the next call, as after any
 * call.  Requires 1000 <= limit_ns <= 1e9 (DMOE_ERR_INVALID_ARG otherwise,
 * nothing launched). */
dmoe_status dmoe_selftest_permute_timeout(const uint16_t* x, const int32_t* expert_idx, int T, int d, int E,
                                          int k, int P_max, int32_t* tokens_per_expert, int32_t* padded_offsets,
                                          int32_t* dest_row, int32_t* src_of_row, uint16_t* x_perm,
                                          int32_t* P_dev, void* ws, size_t ws_bytes, int64_t limit_ns,
                                          dmoe_stream_t stream);

/* Permute + pad that allocates nothing and takes no workspace.  The page
 * has no counterpart to this call: it exists for callers of this library
 * that cannot allocate device memory -- a plugin interface that hands the
 * library only its input and output tensors, a runtime whose device memory
 * is planned once at start-up with no allocator reachable where the layer
 * runs, or a latency-critical path that cannot afford the implicit device
 * synchronisation a cudaMalloc may bring.
 * Arguments, outputs and results are exactly those of dmoe_permute_pad,
 * minus (ws, ws_bytes): the scratch is a static device array inside the
 * library (262,400 bytes, held by every GPU that loads the library until
 * the process exits).
 * Limits: E <= 256 and a device with at most 256 SMs; larger requests
 * return DMOE_ERR_INVALID_ARG and launch nothing.
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture.  Every call clears the array's barrier
 * counters (cudaMemsetAsync on the given stream) and rewrites its
 * histograms; all calls on a device share the one array, so calls that
 * overlap on the GPU (different streams, or several host threads) race
 * and must be serialised by the caller.  Calls no cudaMalloc / cudaFree. */
dmoe_status dmoe_permute_pad_noalloc(const uint16_t* x, const int32_t* expert_idx, int T, int d,
                                     int E, int k, int P_max, int32_t* tokens_per_expert,
                                     int32_t* padded_offsets, int32_t* dest_row,
                                     int32_t* src_of_row, uint16_t* x_perm, int32_t* P_dev,
                                     dmoe_stream_t stream);

/* ----------------------------------------------------------- a3 topology */

/* Topology + transpose metadata in one kernel (sections 1.3 and 1.4).
 * Reads padded_offsets [E+1] (device) and fills every array of *topo (see
 * dmoe_topology) and topo->nnz_dev, topo->P_dev.  Row block r belongs to
 * the expert e with padded_offsets[e] <= 128*r < padded_offsets[e+1] and
 * holds column blocks e*nb .. e*nb+nb-1; the transpose index lists blocks
 * by column, then row, ascending.  With tokens_per_expert [E] (device, may
 * be NULL) and topo->row_fill set, row_fill is written too.  topo itself is
 * a host pointer. */
dmoe_status dmoe_build_topology(const int32_t* padded_offsets, const int32_t* tokens_per_expert,
                                const dmoe_topology* topo, dmoe_stream_t stream);

/* --------------------------------------------- a1 + a2 + a3 fused dispatch */

/* Router, permute + pad and (optionally) topology in one cooperative launch
 * (section 1.4 builds the permutation and the topology metadata in fused
 * kernels to save launches; here the top-k router joins them).  Computes
 * exactly what dmoe_route_topk, then dmoe_permute_pad, then (topo != NULL)
 * dmoe_build_topology compute, with the same arguments and results; the
 * assignments are split among the blocks by token (each block routes its
 * own tokens and counts their experts without reading expert_idx back).
 *   logits [T, E] fp32, x [T, d] bf16 (read); expert_idx, gate_w [T, k],
 *   tokens_per_expert [E], padded_offsets [E+1], dest_row [T*k],
 *   src_of_row [P_max], x_perm [P_max, d], *P_dev (written); with topo,
 *   every array of *topo plus *topo->nnz_dev and *topo->P_dev (written;
 *   topo->E == E and topo->P_max == P_max required).
 *   P_max >= dmoe_padded_rows_max_block(T, k, E, B), a multiple of B, where B
 *   is topo->block (128 without topo).
 *   ws / ws_bytes: as for dmoe_permute_pad (dmoe_permute_pad_workspace_size,
 *   zero-filled before first use, left reusable); calls sharing a ws must
 *   not overlap on the GPU.
 * Requires 1 <= k <= E <= 1024, d a multiple of 8, x / x_perm / ws 16-byte
 * aligned.  Out-of-range arguments: DMOE_ERR_INVALID_ARG, nothing launched.
 * A grid barrier that gives up sets the error word (DMOE_SITE_PERMUTE_BARRIER
 * | DMOE_ERR_TIMEOUT) and leaves the outputs incomplete. */
dmoe_status dmoe_dispatch(const float* logits, const uint16_t* x, int T, int d, int E, int k, int renormalize,
                          int P_max, int32_t* expert_idx, float* gate_w, int32_t* tokens_per_expert,
                          int32_t* padded_offsets, int32_t* dest_row, int32_t* src_of_row, uint16_t* x_perm,
                          int32_t* P_dev, const dmoe_topology* topo, void* ws, size_t ws_bytes,
                          dmoe_stream_t stream);

/* ------------------------------------------------ a4/a8 SDD (+ epilogue) */

/* Sampled dense x dense -> block-sparse (section 1.2).  For every nonzero
 * block q = (r, c) of topo:
 *   acc[q] = A[128r .. 128r+127, 0..K-1] * Bn[0..K-1, 128c .. 128c+127]
 * where Bn = B ([K, E*F]) when b_trans == 0, and Bn = B^T with B
 * [E*F, K] when b_trans != 0.  B2 (same layout as B, SWIGLU_FWD only)
 * gives the second accumulator.  The epilogue (dmoe_epilogue) maps the
 * accumulators to bf16 output blocks [nnz_max, 128, 128] (block q at
 * q*16384, row-major); aux0/aux1 are blocks of the same shape.
 *   A  [P_max, K] bf16;  K a multiple of 64.
 * Unused pointers may be NULL. */
dmoe_status dmoe_sdd(const uint16_t* A, const uint16_t* B, const uint16_t* B2, int K,
                     int b_trans, const dmoe_topology* topo, int epilogue, const uint16_t* aux0,
                     const uint16_t* aux1, uint16_t* out0, uint16_t* out1, uint16_t* out2,
                     dmoe_stream_t stream);

/* ------------------------------------------------------------- a5 DSD */

/* Block-sparse x dense -> dense (section 1.2, layer 2; BCSR row walk of
 * section 1.3):  C[P, N] = S * Bm, S the [P, E*F] matrix given by its
 * blocks S [nnz_max, 128, 128] and topo; Bm [E*F, N] bf16; C [P_max, N]
 * bf16 (rows P .. P_max-1 untouched).  N a multiple of 128. */
dmoe_status dmoe_dsd(const dmoe_topology* topo, const uint16_t* S, const uint16_t* Bm, int N,
                     uint16_t* C, dmoe_stream_t stream);

/* ------------------------------------------------------------ a10 DSD^T */

/* DSD with the transposed dense operand (backward data gradient through
 * layer 1):  C[P, N] = S * Bm^T (+ S2 * Bm2^T), Bm and Bm2 [N, E*F] bf16,
 * S and S2 blocks with the same topology.  S2/Bm2 may both be NULL.
 * C [P_max, N] bf16.  N a multiple of 128. */
dmoe_status dmoe_dsd_t(const dmoe_topology* topo, const uint16_t* S, const uint16_t* Bm,
                       const uint16_t* S2, const uint16_t* Bm2, int N, uint16_t* C,
                       dmoe_stream_t stream);

/* ------------------------------------------------------------- a9 DSTD */

/* Transposed block-sparse x dense -> dense (section 1.3, weight gradient
 * through the transpose index):  G = S^T * D, S [P, E*F] by blocks, D
 * [P_max, N] bf16 (rows < P read).  c_trans == 0: C = G, [E*F, N];
 * c_trans != 0: C = G^T, [N, E*F].  Columns of S with no block (experts
 * without tokens) give zero rows/columns of C.  N a multiple of 128. */
dmoe_status dmoe_dstd(const dmoe_topology* topo, const uint16_t* S, const uint16_t* D, int N,
                      int c_trans, uint16_t* C, dmoe_stream_t stream);

/* ------------------------------------------------ a6/a11 un-permute+combine */

/* Return rows to batch order and combine the k slots of each token:
 *   y[t] = sum_{j<k} w[t*k+j] * y_perm[dest_row[t*k+j]]   (fp32 sum, j order)
 * with w = gate_w, or w = 1 when gate_w is NULL.
 *   y_perm [n_rows, d] bf16, dest_row [A] int32, gate_w [A] fp32 or NULL,
 *   y [T, d] bf16.  d a multiple of 8.  A dest_row entry outside
 *   [0, n_rows) contributes nothing and sets
 *   DMOE_SITE_COMBINE_INDEX | DMOE_ERR_DEVICE. */
dmoe_status dmoe_unpermute_combine(const uint16_t* y_perm, int n_rows, const int32_t* dest_row,
                                   const float* gate_w, int T, int d, int k, uint16_t* y,
                                   dmoe_stream_t stream);

/* ------------------------------------------------------ a7 combine backward */

/* Gradient of dmoe_unpermute_combine with respect to y_perm and gate_w:
 *   dy_perm[p] = w[a] * dy[a / k] for the row p holding assignment a
 *                (a = src_of_row[p] >= 0), 0 for pad rows p < P;
 *   d_gate[a]  = <dy[a / k], y_perm[p]>  (fp32 dot product).
 * w = gate_w, or 1 when gate_w is NULL (then d_gate may be NULL too).
 *   dy [T, d] bf16, y_perm [P_max, d] bf16 (may be NULL when d_gate is
 *   NULL), src_of_row [P_max] int32, P_dev [1] int32 (device),
 *   dy_perm [P_max, d] bf16 (rows P .. P_max-1 untouched), d_gate [A] fp32.
 * A src_of_row entry >= T*k is treated as a pad row and sets
 * DMOE_SITE_COMBINE_INDEX | DMOE_ERR_DEVICE.
 * This call is an addition to the page's list: the backward needs it. */
dmoe_status dmoe_combine_backward(const uint16_t* dy, const uint16_t* y_perm,
                                  const int32_t* src_of_row, const float* gate_w,
                                  const int32_t* P_dev, int T, int d, int k, int P_max,
                                  uint16_t* dy_perm, float* d_gate, dmoe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DMOE_H_ */
