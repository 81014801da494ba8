/*
 * flux_gb300.h -- C ABI of the GB300 (sm_103a) fused GEMM + tensor-parallel
 * collective library.
 *
 * What it computes.  The dense tensor-parallel MLP of FLUX ("FLUX: Fast
 * Software-based Communication Overlap On GPUs Through Kernel Fusion", paper
 * review, section 三 "技术架构", subsection "MLP 前向传播"):
 *     Output1 = GEMM(AllGather(X), W1)          flux_ag_gemm
 *     Output2 = ReduceScatter(GEMM(Output1, W2)) flux_gemm_rs
 * and the MoE variant of COMET (COMET article, section "COMET 的技术原理":
 * the shared tensor is cut along the token dimension, tokens are gathered to
 * experts, expert outputs are combined back per token):
 *     top-k gate (router scores -> expert ids, softmax weights) flux_moe_topk_gate
 *     routing (histogram + prefix sum + stable permutation)  flux_moe_route
 *     AllGather + gather-by-expert + grouped GEMM            flux_moe_ag_grouped_gemm
 *     grouped GEMM + top-k weighted combine + ReduceScatter  flux_moe_grouped_gemm_rs
 * and the same two layers under an expert-parallel x tensor-parallel split of
 * the experts (COMET's EP x TP ratio, same section):
 *     dispatch by expert + grouped GEMM                     flux_moe_ep_dispatch_gemm
 *     grouped GEMM + top-k weighted combine to the owners    flux_moe_ep_gemm_combine
 * plus the plain non-split GEMM that the effective-communication-time metric
 * ECT = OverallTime - GEMM_non-split is measured against (paper review,
 * section 三, "核心公式"): flux_gemm.  The operator list is the one the Flux
 * quick start exercises (Flux tool page, section "快速开始": gemm_only,
 * ag_gemm, gemm_rs, moe_ag_scatter, moe_gather_rs).
 *
 * Tensor-parallel ranks are VIRTUAL: the R ranks of one call are R sets of
 * buffers in the memory of the one GPU the call runs on.  The "communication"
 * is tile movement between those buffers inside one fused kernel, gated by
 * per-shard ready flags; nothing is sent between GPUs.
 *
 * Conventions shared by every entry point
 *   - Every buffer argument is caller-owned.  Pointers documented "device" are
 *     device (or managed) memory of the current CUDA device; arrays of R
 *     pointers ("x_shards" etc.) are HOST arrays holding R device pointers.
 *     The library allocates no device memory and keeps no pointer after the
 *     call returns (it does keep a per-process cache of kernel attributes).
 *   - Matrices are row-major; the leading dimension equals the row length.
 *   - dtype selects fp16 (IEEE binary16) or bf16 for every 16-bit operand
 *     and output; accumulation is always fp32 in tensor memory, rounding of
 *     16-bit outputs is to nearest even.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*,
 *     NULL = the legacy default stream).
 *   - Argument errors return at once with nothing launched.  A CUDA launch
 *     failure returns FLUX_ERR_CUDA (flux_last_cuda_error() gives the code).
 *     Errors found on the device (a bounded wait that ran out) are recorded
 *     in the workspace header and returned by flux_get_status().
 *   - 16-byte alignment is required for every base pointer, and every row
 *     pitch must be a multiple of 16 bytes (so inner dimensions are multiples
 *     of 8 elements).  Violations return FLUX_ERR_UNSUPPORTED; there is no
 *     fallback path.
 *   - Workspaces must be 256-byte aligned, at least flux_*workspace_size()
 *     bytes, and zero-filled once before first use (flux_workspace_init).
 *     Every successful call leaves its workspace zero again.  Calls that share
 *     one workspace must be ordered on the GPU (same stream or events); calls
 *     that overlap on the GPU need separate workspaces.
 */
#ifndef FLUX_GB300_H
#define FLUX_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FLUX_MAX_RANKS 16
#define FLUX_MAX_EXPERTS 1024

typedef enum {
  FLUX_OK = 0,
  FLUX_ERR_INVALID_ARG = 1, /* null pointer, negative or inconsistent size, R out of range */
  FLUX_ERR_UNSUPPORTED = 2, /* alignment / pitch / divisibility rule not met */
  FLUX_ERR_WORKSPACE = 3,   /* workspace null, misaligned or smaller than required */
  FLUX_ERR_CUDA = 4,        /* a CUDA runtime or driver call failed */
  FLUX_ERR_TIMEOUT = 5,     /* device: a ready flag or pipeline wait exceeded timeout_ns */
  FLUX_ERR_NO_DEVICE = 6    /* current device is not an sm_100-family (tcgen05) GPU */
} flux_status_t;

typedef enum { FLUX_F16 = 0, FLUX_BF16 = 1 } flux_dtype_t;

typedef enum {
  FLUX_OP_GEMM = 0,
  FLUX_OP_AG_GEMM = 1,
  FLUX_OP_GEMM_RS = 2,
  FLUX_OP_MOE_AG = 3,
  FLUX_OP_MOE_RS = 4,
  FLUX_OP_MLP = 5,        /* flux_mlp_ag_rs */
  FLUX_OP_MOE_LAYERS = 6, /* flux_moe_layers */
  FLUX_OP_MOE_EP_AG = 7,  /* flux_moe_ep_dispatch_gemm */
  FLUX_OP_MOE_EP_RS = 8,  /* flux_moe_ep_gemm_combine */
  FLUX_OP_AG_GEMM_PUSH = 9 /* flux_ag_gemm with opts->ag_push (the push form) */
} flux_op_t;

/* Optional per-call settings; pass NULL for the defaults. */
typedef struct {
  uint32_t epoch;       /* AG ops: shard s is ready when ready_flags[s] >= epoch (default 1) */
  uint32_t reserved0;
  uint64_t timeout_ns;  /* bound on every device-side wait (0 = 2 s) */
  int32_t num_ctas;     /* persistent grid size (0 = one CTA per SM) */
  int32_t group_n;      /* tile raster: n-tiles per band (0 = 4 for AllGather + GEMM, else 8) */
  int32_t tiles_per_group; /* GEMM-RS: output tiles per rank-group (0 = grid size) */
  int32_t deterministic_rs; /* GEMM-RS: nonzero = add the ranks' fp32 partials in ascending
                               rank order (bit-reproducible; slower: the adds of one tile
                               are serialised over the ranks) */
  int32_t moe_pull_gather;  /* MoE layer0: nonzero = the GEMM's producer warps gather each
                               A tile's token rows themselves (single CTAs, 128 x 256
                               tiles); 0 (default) = the epilogue warps of every CTA
                               copy a share of the grouped rows into the workspace
                               while CTA pairs compute 256 x 512 tiles, each once its
                               rows' ready counts are in */
  int32_t moe_stage_ctas;   /* MoE layer0 staged: how many CTAs' epilogue warps copy rows
                               (0 = all); the push form of AllGather + GEMM: how many
                               CTAs copy rows before they compute (0 = all; fewer = a
                               communication / computation split of the grid, the
                               others compute from the start) */
  int32_t rs_tile;          /* GEMM-RS on whole units (dynamic schedule): 0 = the
                               library's choice; 1 = regions of 4 CTAs, 256 x 512
                               CTA-pair tiles with one 512-column accumulator, B shared
                               by multicast between the two pairs; 2 = regions of 8
                               CTAs, 256 x 256 pair tiles with two accumulators (the
                               fp32 adds of one tile overlap the next tile's MMAs), A
                               and B shared by multicast between the four pairs; 3 = as
                               1, but a region claims one output tile and computes all
                               R ranks' partials of it back to back (the tile's fp32
                               rows stay in L2 between the partials) */
  int32_t moe_l1_ranks;     /* MoE layer1 with tp > 1 ranks per expert group: how many
                               ranks' partials of one 256 x 512 tile a CTA pair computes
                               back to back into one TMEM accumulator before its
                               gate-weighted adds into the token rows (a divisor of tp;
                               the units are claimed at run time from a counter in the
                               workspace).  0 = tp (all ranks of the group: one add per
                               slot; the default); 1 = none: every rank's partial is
                               added on its own, from 256 x 256 tiles with two
                               accumulators (256 x 512 from 48 k-slices per rank on) */
  void* trace;              /* optional per-unit trace (device memory, NULL = off): every
                               CTA of the fused kernel records, per work item, eight
                               64-bit words -- a tag (unit id + 1 in bits 0..31, rank
                               in 32..39, first k-slice in 40..63) and %globaltimer
                               stamps (ns): producer start / last issue, MMA
                               accumulator free / first operands in / last commit,
                               epilogue accumulator full / done.  Words 0 and 1
                               hold the grid size and the records per CTA,
                               (trace_words - 8) / (8 * grid); CTA b's records
                               start at word 8 + 8 * b * (records per CTA); later
                               items of a CTA are dropped; the caller zeroes the
                               buffer.  Dense ops and MoE layers (not the
                               cluster ReduceScatter of few rows, not the pull
                               gather of MoE layer0).  Compiled out when the
                               library is built with -DFLUX_TRACE=0. */
  uint64_t trace_words;     /* size of `trace` in 64-bit words */
  int32_t ag_push;          /* AllGather + GEMM: nonzero = the push form.  Copy CTAs first
                               push every shard's rows (after its ready flag) into one
                               gathered copy of X in the workspace and count each 128-row
                               block; the GEMM tiles wait for their block's count and load A
                               from the copy.  0 (default) = the pull form: each tile loads
                               its A rows from the owning shard after the shard's flag.
                               Needs flux_workspace_size(FLUX_OP_AG_GEMM_PUSH, ...) and the
                               dynamic schedule; moe_stage_ctas sets the copy CTAs. */
  int32_t debug_probe;      /* checked build only (libflux_gb300_checked.so, see
                               flux_checks_enabled): nonzero makes the kernel fail one
                               check on purpose (report: FLUX_ERR_INVALID_ARG, wait site
                               13, arg0 = 15, arg1 = this value), to show that checks
                               report; ignored by the regular build */
  int32_t moe_static_schedule; /* MoE layer0 (staged form): nonzero = the static unit
                               schedule (CTA pair i takes units i, i + pairs, ...);
                               0 (default) = the dynamic one: each pair claims its next
                               unit from a counter in the workspace while it computes
                               the current one, so pairs that drew cheaper units (the
                               half-wide last column tile, an expert's partial last
                               rows) take more of them */
  int32_t rs_group;         /* GEMM-RS on regions of 4 CTAs (rs_tile 1): how many ranks'
                               partials of one output tile a region computes back to
                               back into one TMEM accumulator before it adds the sum
                               into the owner's fp32 rows (a divisor of R; 0 = the
                               library's choice, 1 = every rank's partial added on its
                               own).  Fewer adds and accumulator hand-overs, longer
                               work units; the summation order of the ranks changes
                               (results within the fp32 rounding of the adds) */
  int32_t acc_whole;        /* tiles with one 512-column accumulator (256 x 512 pair tiles):
                               nonzero = the next tile's MMAs wait until the epilogue has
                               read the whole accumulator; 0 (default) = the epilogue hands
                               back its first 256 columns early and the next tile's first
                               k-slices (as many as the operand ring holds) run their
                               MMAs into those columns meanwhile.  Same results. */
} flux_opts_t;

/* What flux_get_status found in a workspace header. */
typedef struct {
  uint32_t status; /* flux_status_t of the first device-side error, 0 if none */
  uint32_t where;  /* which wait gave up: 1 ready flag, 2 smem slot free, 3 smem slot full,
                      4 accumulator free, 5 accumulator full, 6 drain,
                      7 deterministic GEMM-RS turn, 8 staged MoE rows of an m-tile,
                      9 next unit of the dynamic schedule (dense ops, MoE layer0), 10 a cluster
                      of an unexpected shape under the dynamic schedule, 11 MoE
                      layer1's grid barrier before the token rows are converted,
                      12 the exchange of a cluster ReduceScatter (GEMM-RS of few
                      rows), 13 a failed check of the checked build */
  uint32_t arg0;   /* flag wait: shard index; pipeline waits: CTA index */
  uint32_t arg1;   /* flag wait: last flag value seen; pipeline waits: stage / buffer */
} flux_device_report_t;

/* ---------------------------------------------------------------- housekeeping */

/* Version of this ABI (major * 10000 + minor * 100 + patch). */
int flux_version(void);

/* 1 in the checked build of the library (libflux_gb300_checked.so, compiled
 * with -DFLUX_CHECKS=1), 0 in the regular one.  In the checked build every
 * TMA coordinate and every global store or add of the kernels is checked
 * against the tensor it addresses; a failed check ends the call with
 * FLUX_ERR_INVALID_ARG (reported by flux_get_status: wait site 13, arg0 the
 * check -- 1 A row, 2 A k, 3 B column, 4 B k, 5 output row, 6 output
 * column, 7 fp32 row or token, 8 fp32 column, 9 owner rank, 15 the
 * requested probe -- and arg1 the offending value) and the access is
 * skipped, or, for a load, moved to the tensor's origin.  No check traps. */
int flux_checks_enabled(void);

/* sizeof(flux_opts_t) as this library was compiled: a binding checks its own
 * copy of the struct against it before passing options. */
size_t flux_opts_size(void);

/* Human-readable name of a status code (static string, never NULL). */
const char* flux_status_string(flux_status_t s);

/* The cudaError_t of the most recent FLUX_ERR_CUDA on the calling thread. */
int flux_last_cuda_error(void);

/* Bytes of workspace a dense op needs (FLUX_OP_GEMM / AG_GEMM / GEMM_RS / MLP).
 * M, N, K as in the op's own signature (FLUX_OP_MLP: M, H, F).  Every dense op
 * needs the 256-byte status header; GEMM-RS adds per-tile arrival counters and
 * the fp32 accumulation buffer of the owners' row chunks (M x N floats).  Each
 * op then adds the mailboxes of its dynamic unit schedule: 4 x (2 U + 384)
 * bytes rounded up to 256, U = R x ceil(M / 512) x ceil(N_r / 512) work units
 * (N_r = the op's output columns per rank).  With that area the op runs on
 * every SM (clusters of CTA pairs, 4 preferred, units claimed at run time);
 * given only the header (GEMM, AG-GEMM) or only header + counters +
 * accumulators (GEMM-RS), it runs its static schedule on 4-CTA clusters.  The
 * MLP needs the larger of its two calls' workspaces.  Returns 0 for an unknown
 * op or invalid sizes. */
size_t flux_workspace_size(flux_op_t op, int R, int M, int N, int K);

/* Launch shape of a dense op's whole-tile kernel on the current device: CTAs
 * per (preferred) cluster and its persistent grid -- the dynamic schedule's
 * grid when that launch form is available, else the CTAs of 4-CTA clusters
 * resident at once.  FLUX_OP_GEMM / AG_GEMM / GEMM_RS / MLP; other ops return
 * FLUX_ERR_INVALID_ARG. */
flux_status_t flux_launch_info(flux_op_t op, flux_dtype_t dtype, int* cluster_ctas,
                               int* resident_ctas);

/* Bytes of workspace a MoE op needs (FLUX_OP_MOE_AG / MOE_RS / MOE_LAYERS / MOE_EP_AG /
 * MOE_EP_RS); 0 for an unknown op or invalid sizes. */
size_t flux_moe_workspace_size(flux_op_t op, int R, int T, int H, int F, int E, int topk);

/* Zero `bytes` of a workspace on `stream` (cudaMemsetAsync). */
flux_status_t flux_workspace_init(void* workspace, size_t bytes, void* stream);

/* Synchronise `stream`, then read the device status of `workspace`.
 * Returns FLUX_OK or the first device-side error recorded by a call that used
 * this workspace.  If `report` is non-NULL it receives the details.  After an
 * error the whole workspace (`bytes`) is zeroed again, so it can be reused. */
flux_status_t flux_get_status(void* workspace, size_t bytes, void* stream,
                              flux_device_report_t* report);

/* ---------------------------------------------------------------- dense ops */

/* Plain non-split GEMM: C[M x N] = A[M x K] . B[K x N].
 * The GEMM_non-split baseline of ECT (paper review, section 三, "核心公式").
 * A, B, C device; K = 0 writes zeros.  At most 128 rows (M divisible by 4 or
 * 8, K / S a multiple of 8 and at least 256 for S = 8 or 4 K slices), given
 * the workspace flux_workspace_size(FLUX_OP_GEMM, 1, M, N, K) asks for then:
 * K is split into S slices whose fp32 partials are summed on chip (the
 * few-row GEMM + ReduceScatter form of flux_gemm_rs, the slices in place of
 * ranks); with less workspace, or opts->num_ctas set, the whole-tile form
 * runs. */
flux_status_t flux_gemm(int M, int N, int K, flux_dtype_t dtype, const void* A, const void* B,
                        void* C, void* workspace, size_t workspace_bytes, const flux_opts_t* opts,
                        void* stream);

/* Output1_r = GEMM(AllGather(X), W1_r) for r in [0, R)
 * (paper review, section 三, "MLP 前向传播", first GEMM; AllGather overlap,
 * section 三 "AllGather 重叠").
 *   x_shards[s]  device, [M/R x K]: the rows [s M/R, (s+1) M/R) of X owned by rank s
 *   w_shards[r]  device, [K x N/R]: rank r's column block of W1
 *   out[r]       device, [M x N/R]: rank r's Output1
 *   ready_flags  device uint32[R] or NULL: the kernel pulls a tile of X_s only
 *                after reading ready_flags[s] >= opts->epoch (acquire, gpu
 *                scope); NULL means every shard is ready.  A flag that never
 *                becomes ready ends the call with FLUX_ERR_TIMEOUT (reported by
 *                flux_get_status) after opts->timeout_ns.
 * Requires 1 <= R <= FLUX_MAX_RANKS, M and N divisible by R, (M/R) % 8 == 0,
 * K % 8 == 0, (N/R) % 8 == 0. */
flux_status_t flux_ag_gemm(int R, int M, int N, int K, flux_dtype_t dtype,
                           const void* const* x_shards, const void* const* w_shards,
                           void* const* out, const uint32_t* ready_flags, void* workspace,
                           size_t workspace_bytes, const flux_opts_t* opts, void* stream);

/* Output2_o = rows [o M/R, (o+1) M/R) of sum_r A_r . B_r, for o in [0, R)
 * (paper review, section 三, "MLP 前向传播", second GEMM; ReduceScatter overlap,
 * section 三 "ReduceScatter 重叠").
 *   a_shards[r]  device, [M x K/R]: rank r's column block of Output1
 *   b_shards[r]  device, [K/R x N]: rank r's row block of W2
 *   out[o]       device, [M/R x N]: owner rank o's row chunk of the reduced product
 * Every rank's partial tile is accumulated in fp32 into the owner's chunk of
 * the workspace; the last partial to arrive converts the tile to 16 bits and
 * stores it in out[owner].  Few rows (M <= 128, R = 4 or 8, no num_ctas or
 * deterministic_rs option, every 256-column tile on a resident 4-CTA
 * cluster): a cluster of 4 CTAs computes the R partials of a tile and reduces
 * them through distributed shared memory instead, summing in a fixed order
 * (repeat calls give the same bits) without touching the workspace's
 * accumulators.  Requires M and K divisible by R, (K/R) % 8 == 0, N % 8 == 0. */
flux_status_t flux_gemm_rs(int R, int M, int N, int K, flux_dtype_t dtype,
                           const void* const* a_shards, const void* const* b_shards,
                           void* const* out, void* workspace, size_t workspace_bytes,
                           const flux_opts_t* opts, void* stream);

/* The dense tensor-parallel MLP in one call: both GEMMs of the paper review's
 * "MLP 前向传播" (section 三), with no activation between them (the pages
 * give none):
 *   h[r]   = GEMM(AllGather(X), W1_r)            as flux_ag_gemm(R, M, F, H)
 *   out[o] = rows of sum_r GEMM(h[r], W2_r)      as flux_gemm_rs(R, M, H, F)
 *   x_shards[s]  device, [M/R x H];  w1_shards[r] device, [H x F/R]
 *   h[r]         device, [M x F/R]: Output1, written and then read by the call
 *   w2_shards[r] device, [F/R x H];  out[o] device, [M/R x H]
 *   ready_flags  as in flux_ag_gemm
 * Workspace: flux_workspace_size(FLUX_OP_MLP, R, M, H, F).  opts apply to both
 * GEMMs.  Requirements: those of the two calls. */
flux_status_t flux_mlp_ag_rs(int R, int M, int H, int F, flux_dtype_t dtype,
                             const void* const* x_shards, const void* const* w1_shards,
                             void* const* h, const void* const* w2_shards, void* const* out,
                             const uint32_t* ready_flags, void* workspace, size_t workspace_bytes,
                             const flux_opts_t* opts, void* stream);

/* GEMM + ReduceScatter that allocates nothing and takes no workspace.
 * No counterpart in the FLUX or COMET pages: it exists for callers that cannot
 * allocate device memory or hand over a workspace (plugin hosts and inference
 * runtimes whose device-memory budget is fixed before serving starts, wrappers
 * without an allocator).  Same arguments, results and requirements as
 * flux_gemm_rs, minus the workspace.  Scratch comes from a 256-byte aligned
 * __device__ array of FLUX_NOALLOC_SCRATCH_BYTES inside the library, held by
 * every GPU that loads the library until the process exits.
 *   - Returns FLUX_ERR_WORKSPACE, launching nothing, when
 *     flux_workspace_size(FLUX_OP_GEMM_RS, R, M, N, K) exceeds that size.
 *   - The first call on a device looks up the array's device address (with
 *     that device current); make it before any stream capture begins.
 *   - All calls on a device share the array and it keeps the last call's
 *     contents; each call checks its arguments first (a refused call leaves
 *     the stream and the array alone), then zeroes the part it uses on
 *     `stream`.  Calls that overlap on the GPU race on it: order them (one
 *     stream or events).
 *   - Device-side status (flux_get_status) is not available for these calls. */
#define FLUX_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
flux_status_t flux_gemm_rs_noalloc(int R, int M, int N, int K, flux_dtype_t dtype,
                                   const void* const* a_shards, const void* const* b_shards,
                                   void* const* out, const flux_opts_t* opts, void* stream);

/* ---------------------------------------------------------------- MoE ops */

/* Top-k gate of T tokens over E experts from fp32 router scores.  The pages
 * name the Mixture-of-Experts layer (COMET article, "COMET 是什么") but not
 * its gate; this is the plain one:
 *   logits        device float32[T x E]
 *   topk_ids      device int32[T x topk]: the topk largest scores of the token,
 *                 largest first, equal scores in ascending expert order (a NaN
 *                 score counts as -inf)
 *   topk_weights  device float32[T x topk]: softmax over the chosen scores,
 *                 exp(s_j - s_0) / sum_i exp(s_i - s_0) in fp32 with expf (the
 *                 softmax over all E renormalised over the chosen k); if the
 *                 largest chosen score s_0 is infinite, the chosen scores equal
 *                 to it share the weight equally and the rest get 0
 * The ids are exact (decided on the fp32 scores); deterministic.  Requires
 * 1 <= topk <= E <= FLUX_MAX_EXPERTS; bad sizes or NULL buffers (T > 0) return
 * FLUX_ERR_INVALID_ARG. */
flux_status_t flux_moe_topk_gate(int T, int E, int topk, const float* logits, int32_t* topk_ids,
                                 float* topk_weights, void* stream);

/* Routing of T tokens with topk experts each (COMET article, section
 * "COMET 的技术原理", token-dimension decomposition).  Slot s = t*topk + k.
 *   topk_ids     device int32[T*topk], values in [0, E)
 *   counts       device int32[E]      slots per expert
 *   offsets      device int32[E+1]    exclusive prefix sum, offsets[E] = T*topk
 *   slot_to_row  device int32[T*topk] offsets[id[s]] + #{s' < s : id[s'] = id[s]}
 *   row_to_slot  device int32[T*topk] the inverse permutation (rows grouped by expert)
 * Bit-exact and deterministic.  An id outside [0, E) is counted nowhere and
 * makes the call record FLUX_ERR_INVALID_ARG in `workspace` (which must then
 * hold at least 256 bytes; may be NULL to skip the check). */
flux_status_t flux_moe_route(int T, int E, int topk, const int32_t* topk_ids, int32_t* counts,
                             int32_t* offsets, int32_t* slot_to_row, int32_t* row_to_slot,
                             void* workspace, size_t workspace_bytes, void* stream);

/* MoE layer0: H_r[row] = AllGather(X)[token(row)] . W1_r[expert(row)] for r in [0, R),
 * rows in the grouped (expert-sorted) order of flux_moe_route, which this call
 * runs first and whose outputs it writes to counts/offsets/slot_to_row/row_to_slot.
 *   x_shards[s]   device, [T/R x H]: token rows owned by rank s
 *   w1_shards[r]  device, [E x H x F/R]: rank r's column block of every expert's W1
 *   topk_ids      device int32[T x topk]
 *   h_out[r]      device, [T*topk x F/R]
 *   ready_flags   as in flux_ag_gemm (per token shard), or NULL
 * By default the rows are gathered once, inside the same kernel, into a
 * grouped copy [T*topk x H] in the workspace (flux_moe_workspace_size
 * FLUX_OP_MOE_AG counts it), each 256-row tile published by a ready count
 * that its GEMM tiles wait for; opts->moe_pull_gather selects the gather in
 * the GEMM's producer warps instead (no copy).
 * Requires T and F divisible by R, H % 8 == 0, (F/R) % 8 == 0, 1 <= E <= FLUX_MAX_EXPERTS. */
flux_status_t flux_moe_ag_grouped_gemm(int R, int T, int H, int F, int E, int topk,
                                       flux_dtype_t dtype, const void* const* x_shards,
                                       const void* const* w1_shards, const int32_t* topk_ids,
                                       void* const* h_out, int32_t* counts, int32_t* offsets,
                                       int32_t* slot_to_row, int32_t* row_to_slot,
                                       const uint32_t* ready_flags, void* workspace,
                                       size_t workspace_bytes, const flux_opts_t* opts,
                                       void* stream);

/* MoE layer1: Out_o[t] = sum_r sum_k topk_weights[t,k] . (H_r[slot_to_row[t*topk+k]] .
 * W2_r[topk_ids[t,k]]) for the tokens t in [o T/R, (o+1) T/R) owned by rank o.
 *   h_shards[r]   device, [T*topk x F/R]: layer0 output of rank r, grouped order
 *   w2_shards[r]  device, [E x F/R x H]: rank r's row block of every expert's W2
 *   topk_ids      device int32[T x topk]; topk_weights device float32[T x topk]
 *   offsets, slot_to_row, row_to_slot: the routing that ordered h_shards
 *                 (from flux_moe_route or layer0), or all three NULL to have
 *                 this call recompute them in its workspace
 *   out[o]        device, [T/R x H]
 * Contributions are accumulated in fp32 in the workspace (gate-weighted adds
 * in each tile's epilogue).  With rank groups (the default when an expert
 * group has several ranks) every (token, 512-column tile) receives a known
 * number of adds, and the add that completes it converts it to 16 bits and
 * zeroes it.  Otherwise (one add per rank, or a slot whose expert id is out
 * of range, routed nowhere) the CTAs of the launch meet at a grid-wide
 * barrier when every tile is done (the launch is sized so that all of them
 * are resident at once; a kernel of another stream that holds SMs the whole
 * time can delay it until timeout_ns, FLUX_ERR_TIMEOUT at wait site 11) and
 * each converts a share of the token rows.  Tiles are 256 x 256 on CTA
 * pairs with two accumulators (each tile's adds overlap the next tile), or,
 * for reductions of 48 or more 64-deep k-slices (F/R > 3008, also the
 * per-rank length of flux_moe_ep_gemm_combine), 256 x 512 with one.
 * Requires T and F divisible by R, (F/R) % 8 == 0, H % 8 == 0. */
flux_status_t flux_moe_grouped_gemm_rs(int R, int T, int H, int F, int E, int topk,
                                       flux_dtype_t dtype, const void* const* h_shards,
                                       const void* const* w2_shards, const int32_t* topk_ids,
                                       const float* topk_weights, const int32_t* offsets,
                                       const int32_t* slot_to_row, const int32_t* row_to_slot,
                                       void* const* out, void* workspace, size_t workspace_bytes,
                                       const flux_opts_t* opts, void* stream);

/* The MoE layer in one call: routing, layer0 and layer1 (COMET article,
 * "COMET 的技术原理"; the pages give no activation between the layers, so
 * there is none):
 *   h[r]   = flux_moe_ag_grouped_gemm output (grouped rows, [T*topk x F/R])
 *   out[o] = flux_moe_grouped_gemm_rs of h with the same routing ([T/R x H])
 * The routing (counts, offsets, slot_to_row, row_to_slot) is kept in the
 * workspace: flux_moe_workspace_size(FLUX_OP_MOE_LAYERS, ...).  Other arguments
 * and requirements as in the two calls. */
flux_status_t flux_moe_layers(int R, int T, int H, int F, int E, int topk, flux_dtype_t dtype,
                              const void* const* x_shards, const void* const* w1_shards,
                              const void* const* w2_shards, const int32_t* topk_ids,
                              const float* topk_weights, void* const* h, void* const* out,
                              const uint32_t* ready_flags, void* workspace,
                              size_t workspace_bytes, const flux_opts_t* opts, void* stream);

/* ---------------------------------------------------------------- MoE, EP x TP split
 *
 * The R ranks form EP = R / tp expert groups of tp ranks (COMET article,
 * "COMET 的技术原理": the EP x TP ratio of the MoE layer).  Group g holds
 * experts [g E/EP, (g+1) E/EP); rank r = g tp + t holds block t (F/tp wide)
 * of each of them.  tp = R is the tensor-parallel layout of
 * flux_moe_ag_grouped_gemm / flux_moe_grouped_gemm_rs (same results); tp = 1
 * is pure expert parallel: every expert whole on one rank, and each routed
 * token row dispatched to that rank alone.
 * Workspace: flux_moe_workspace_size(FLUX_OP_MOE_EP_AG / FLUX_OP_MOE_EP_RS,
 * ...), which does not depend on tp.  Requires R % tp == 0, E % (R/tp) == 0,
 * F % tp == 0, T % R == 0, H % 8 == 0, (F/tp) % 8 == 0.  Invalid sizes or a
 * NULL buffer return FLUX_ERR_INVALID_ARG; unaligned buffers
 * FLUX_ERR_UNSUPPORTED. */

/* EP layer0: h_out[r][row] = X[token(row)] . W1[r][expert(row) - g E/EP] for
 * the grouped-order rows of group g's experts, rows [offsets[g E/EP],
 * offsets[(g+1) E/EP]); the call runs flux_moe_route first and writes
 * counts/offsets/slot_to_row/row_to_slot as that call does.
 *   x_shards[s]   device, [T/R x H]: token rows owned by rank s
 *   w1_shards[r]  device, [E/EP x H x F/tp]: column block t of group g's experts
 *   h_out[r]      device, [T*topk x F/tp]: only group g's rows are written (with
 *                 H == 0 the whole buffer is zeroed), so ranks of different
 *                 groups with the same t may pass one buffer
 *   ready_flags   as in flux_ag_gemm (per token shard), or NULL */
flux_status_t flux_moe_ep_dispatch_gemm(int R, int tp, int T, int H, int F, int E, int topk,
                                        flux_dtype_t dtype, const void* const* x_shards,
                                        const void* const* w1_shards, const int32_t* topk_ids,
                                        void* const* h_out, int32_t* counts, int32_t* offsets,
                                        int32_t* slot_to_row, int32_t* row_to_slot,
                                        const uint32_t* ready_flags, void* workspace,
                                        size_t workspace_bytes, const flux_opts_t* opts,
                                        void* stream);

/* EP layer1 + combine: Out_o[t] = sum_k topk_weights[t,k] . sum over the tp ranks
 * r of expert e = topk_ids[t,k]'s group of (h_shards[r][slot_to_row[t*topk+k]] .
 * W2[r][e - g E/EP]), for the tokens t in [o T/R, (o+1) T/R) owned by rank o.
 *   h_shards[r]   device, [T*topk x F/tp]: rows of group g's experts are read
 *   w2_shards[r]  device, [E/EP x F/tp x H]: row block t of group g's experts
 *   offsets, slot_to_row, row_to_slot: the routing that ordered h_shards, or all
 *                 three NULL to have this call recompute them in its workspace
 *   out[o]        device, [T/R x H]
 * The tp*topk contributions to a token row are added in fp32 in the workspace;
 * the last one converts the row to 16 bits. */
flux_status_t flux_moe_ep_gemm_combine(int R, int tp, int T, int H, int F, int E, int topk,
                                       flux_dtype_t dtype, const void* const* h_shards,
                                       const void* const* w2_shards, const int32_t* topk_ids,
                                       const float* topk_weights, const int32_t* offsets,
                                       const int32_t* slot_to_row, const int32_t* row_to_slot,
                                       void* const* out, void* workspace, size_t workspace_bytes,
                                       const flux_opts_t* opts, void* stream);

/* ---------------------------------------------------------------- tuning
 *
 * Per-problem launch options chosen by measurement (FLUX paper review,
 * "关键优化": the fused kernel's tile is searched per problem; COMET article,
 * "动态负载平衡": precompiled variants picked at run time by token count and
 * parallel layout).  Each flux_tune_* call runs its op on the given buffers
 * with every candidate option set (one warm-up and five timed calls each, on
 * `stream`, synchronising it), records the fastest for that problem -- this
 * device, the op, the dtype and the sizes -- in a process-wide table, and
 * copies it to *best (may be NULL).  Afterwards a call of the same op and
 * problem with opts == NULL uses the recorded options; passing opts overrides
 * the table.  The outputs hold the result of the last candidate run; a
 * candidate that fails (argument, launch or device-side error) ends the call
 * with that status and records nothing.  Arguments as in the op itself.
 * Candidates:
 *   AllGather + GEMM          group_n in {2, 4, 8, 16}
 *   GEMM + ReduceScatter      group_n in {4, 8, 16} x tiles_per_group in {0, 2};
 *                             the stream-K (decode) form: num_ctas in
 *                             {0, SMs, 7/8 SMs, SMs / 2}
 *   MoE layer0 (any tp)       staged with group_n 8 or 16, or moe_pull_gather
 *   MoE layer1 (any tp)       group_n in {4, 8, 16}
 * flux_moe_ag_grouped_gemm / flux_moe_grouped_gemm_rs are the tp = R
 * problems of the two MoE tuners. */
flux_status_t flux_tune_ag_gemm(int R, int M, int N, int K, flux_dtype_t dtype,
                                const void* const* x_shards, const void* const* w_shards,
                                void* const* out, const uint32_t* ready_flags, void* workspace,
                                size_t workspace_bytes, void* stream, flux_opts_t* best);
flux_status_t flux_tune_gemm_rs(int R, int M, int N, int K, flux_dtype_t dtype,
                                const void* const* a_shards, const void* const* b_shards,
                                void* const* out, void* workspace, size_t workspace_bytes,
                                void* stream, flux_opts_t* best);
flux_status_t flux_tune_moe_layer0(int R, int tp, int T, int H, int F, int E, int topk,
                                   flux_dtype_t dtype, const void* const* x_shards,
                                   const void* const* w1_shards, const int32_t* topk_ids,
                                   void* const* h_out, int32_t* counts, int32_t* offsets,
                                   int32_t* slot_to_row, int32_t* row_to_slot,
                                   const uint32_t* ready_flags, void* workspace,
                                   size_t workspace_bytes, void* stream, flux_opts_t* best);
flux_status_t flux_tune_moe_layer1(int R, int tp, int T, int H, int F, int E, int topk,
                                   flux_dtype_t dtype, const void* const* h_shards,
                                   const void* const* w2_shards, const int32_t* topk_ids,
                                   const float* topk_weights, const int32_t* offsets,
                                   const int32_t* slot_to_row, const int32_t* row_to_slot,
                                   void* const* out, void* workspace, size_t workspace_bytes,
                                   void* stream, flux_opts_t* best);

/* Forget every recorded problem / how many are recorded. */
void flux_tune_clear(void);
int flux_tune_count(void);

#ifdef __cplusplus
}
#endif

#endif /* FLUX_GB300_H */
