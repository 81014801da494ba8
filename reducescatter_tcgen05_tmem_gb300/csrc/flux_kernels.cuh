// Persistent, warp-specialised tcgen05 GEMM with fused tensor-parallel
// collectives over R virtual ranks (all ranks' buffers live on this GPU).
//
//   producer warp(s)  TMA (or cp.async row gather) of A/B k-slices into a
//                     shared-memory ring; for AllGather, the A tile is pulled
//                     from the rank that owns its rows only after that rank's
//                     ready flag is seen (acquire)
//   MMA warp          one thread issues tcgen05.mma (fp32 accumulators in
//                     TMEM); accumulators are double-buffered in the 512 TMEM
//                     columns so the epilogue of one tile overlaps the main
//                     loop of the next
//   epilogue warps    tcgen05.ld TMEM -> registers, then one of:
//                       STORE        convert to 16 bits, store (AllGather-GEMM, plain GEMM)
//                       REDUCE       fp32 add into the owner rank's row chunk of the
//                                    workspace; the last partial converts and stores
//                                    (GEMM + ReduceScatter)
//                       MOE_GATHER   STORE with A rows gathered by expert (MoE layer0)
//                       MOE_SCATTER  gate-weighted fp32 add into the owning token row;
//                                    after a grid-wide barrier every CTA converts a
//                                    share of the token rows (MoE layer1); the
//                                    _WIDE form runs 256 x 512 tiles (long K)
//                       MOE_STAGED   STORE for MoE layer0 whose A rows were first
//                                    gathered into a grouped staging buffer by every
//                                    CTA of the same launch (per-tile ready counters)
//                       RS_CLUSTER   GEMM + ReduceScatter of few rows (M <= 128, the
//                                    decode shapes): a cluster of 4 CTAs computes all
//                                    R partials of one 128 x 256 tile (R / 4 each, in
//                                    separate accumulators), then reduces them through
//                                    distributed shared memory, each CTA into the rows
//                                    of the owner ranks it serves (no fp32 workspace)
//
// PAIR = 1: one CTA computes a 128 x 256 tile with tcgen05.mma.cta_group::1
//           (4-stage ring of 48 KB: A 128x64 + B 64x256); two 256-column
//           accumulators, so the epilogue of one tile overlaps the next.
// PAIR = 2: a cluster of two CTAs computes a 256 x 512 tile with two
//           tcgen05.mma.cta_group::2 (M 256, N 256) per 16-deep k step, issued
//           by the even CTA.  Each CTA holds its own 128 rows of A and, of each
//           256-column half of the tile, its own 128 columns of B (4-stage ring
//           of 48 KB).  Per unit of tensor work an SM then requests half the
//           operand bytes of the PAIR = 1 tile: the load path (TMA requests in
//           flight per SM), not the tensor pipe, is what bounds these kernels.
//           The 128 x 512 fp32 accumulator of a CTA fills all 512 TMEM
//           columns, so the MMAs of the next tile wait for the epilogue.
//           Both CTAs' TMA loads complete on the even CTA's "full" barrier,
//           whose producer expects the bytes of both.  Commits are multicast
//           to both CTAs' "empty" and "accumulator full" barriers; both CTAs'
//           epilogue warps arrive on the even CTA's "accumulator empty" barrier.
// CL = 4:   a cluster of two such pairs stacked along M (a 512 x 512 unit).
//           CTAs r and r^2 need the same B columns, so each issues half of
//           them (the 256-column half h = r / 2) as a TMA multicast to both;
//           every CTA's bytes still complete on its own pair's even-CTA
//           barrier.  A stage may be refilled only when both pairs' MMAs have
//           read it: each "empty" barrier counts one commit per pair.
//
// MoE layer1, CL = 2: a CTA pair computes a 256 x 256 tile inside one expert.
// MoE layer0, two forms:
//   MOE_GATHER, CL = 1: the producer gathers the A rows with cp.async, whose
//     completion can only be signalled in the issuing CTA, so single CTAs.
//   MOE_STAGED, CL = 2: every CTA first copies a share of the grouped A rows
//     into a staging buffer and counts each finished 32-row block on its
//     m-unit's ready counter; then CTA pairs compute 256 x 512 tiles whose
//     producers wait for their unit's count and load A by TMA.
//
// RS_CLUSTER, CL = 4: four independent single-CTA (PAIR = 1) 128 x 256
// tiles per cluster, one n-tile per cluster; the cluster only serves the
// distributed-shared-memory reduction of the partials.
//
// The template parameter CL is the number of CTAs of a cluster (1, 2 or 4);
// PAIR = min(CL, 2) is the tcgen05 CTA group (1 for RS_CLUSTER) and
// MC = CL / PAIR the pairs that share B (dense modes only).
//
// Dynamic schedule (dense modes, CL = 4, KParams::dyn): clusters of 4 CTAs fit
// on only part of the SMs (144 of 152 on GB300), so the kernel is launched with
// CTA pairs as the cluster size and 4 as the preferred one.  Every aligned group
// of 4 CTAs (a "region") is then either one 4-CTA cluster or two pair clusters.
// The region computes one 512 x 512 unit at a time either way: pair clusters
// load their own B instead of sharing it by multicast.  Regions claim units from
// a counter in the workspace header, so that the slower pair regions take fewer
// of them; the region's first CTA claims the next unit a few k-slices before
// its current one ends and writes it into the region's mailbox in the
// workspace, from which every role of the region's CTAs reads its units.  In
// store mode the last units are claimed as two 256-column halves each.
// CL = 8 (store mode, dynamic schedule only): regions of four pairs, two
// stacked along M and two side by side along N (512 x 1024 units); in an
// 8-CTA cluster CTA r shares B with r ^ 2 and A with r ^ 4, each issuing half
// of the shared boxes as multicasts (A in two 64-row boxes); where an 8-CTA
// cluster does not fit the region runs as four pair clusters.
//
// Every wait is bounded: after timeout_ns (or an iteration cap) the thread
// records FLUX_ERR_TIMEOUT in the workspace header, raises the per-call abort
// word, and the CTA drains its in-flight copies and MMAs, frees TMEM and exits.
#pragma once

#include "flux_ptx.cuh"

// Per-unit tracing: every work item of a CTA can record %globaltimer stamps of
// its roles into a caller buffer (KParams::trace).  Built in by default; build
// with -DFLUX_TRACE=0 to compile it out.
#ifndef FLUX_TRACE
#define FLUX_TRACE 1
#endif
// Checked build (-DFLUX_CHECKS=1, libflux_gb300_checked.so): every TMA
// coordinate and every global store or add of the kernels is checked against
// the tensor it addresses; a failed check records FLUX_ERR_INVALID_ARG with
// the check's code and the offending value (wait site W_CHECK) and the access
// is skipped (stores, adds) or moved to a safe coordinate (loads, whose bytes
// the stage barrier expects).  The regular build compiles the checks out.
#ifndef FLUX_CHECKS
#define FLUX_CHECKS 0
#endif

namespace flux {

constexpr int BM = 128;  // rows of A per CTA (TMEM lanes)
constexpr int BN = 256;  // tile columns (MMA N)
constexpr int BK = 64;   // k-slice per pipeline stage (one 128-byte swizzle row of 16-bit data)
constexpr int UK = 16;   // K of one tcgen05.mma kind::f16
constexpr int A_STAGE = BM * BK * 2;  // 16 KB
constexpr int B_BOX_N = 64;           // 64 columns = 128 bytes, one swizzle span
constexpr int TMEM_COLS = 2 * BN;     // all 512 TMEM columns: fp32 accumulators
constexpr int MAXR = 16;
constexpr int EPI_WARPS = 4;
constexpr int GATHER_LAG = 2;         // cp.async groups in flight before a stage is published

// Epilogue staging for the fp32 reduce modes, 8 KB per epilogue warp.
//   REDUCE: two 4 KB buffers, each a 32-row x 32-float box in the 128-byte
//           swizzled layout of the accumulator tensor map (one tensor bulk
//           reduce per buffer; the swizzle keeps the row-per-thread stores
//           free of bank conflicts).
//   MOE_SCATTER: 32 rows of 32 floats, each row padded to 144 bytes (written
//           by the row's thread, read back row-contiguously for the
//           vector atomic adds into the rows' tokens).
constexpr int STG_BOX = 32 * 32 * 4;
constexpr int STG_PITCH = 144;
constexpr int STG_WARP = 2 * STG_BOX;
static_assert(32 * STG_PITCH <= STG_WARP, "row staging fits");

// Tile geometry: PAIR CTAs form one tcgen05 CTA group (M = 128 PAIR), and NM
// MMAs of N = 256 cover the tile's columns at every 16-deep k step.
//   <1,1> 128 x 256, B 256 columns per CTA, 4 stages of 48 KB, 2 accumulators
//   <2,1> 256 x 256, B 128 columns per CTA, 6 stages of 32 KB, 2 accumulators
//   <2,2> 256 x 512, B 256 columns per CTA, 4 stages of 48 KB, 1 accumulator
template <int PAIR, int NM, int EW = EPI_WARPS>
struct Geo {
  static constexpr int TILE_M = BM * PAIR;             // rows of one tile
  static constexpr int TILE_N = BN * NM;               // columns of one tile
  static constexpr int N_MMA = NM;                     // N = 256 MMAs per 16-deep k step
  static constexpr int B_BOXES = TILE_N / PAIR / B_BOX_N;  // 64-column B boxes per CTA and stage
  static constexpr int B_STAGE = B_BOXES * B_BOX_N * BK * 2;
  // the ring gives up the room the epilogue warps beyond four stage in
  static constexpr int STAGES = (192 * 1024 - (EW - EPI_WARPS) * STG_WARP) / (A_STAGE + B_STAGE);
  static constexpr int ACC_BUFS = 2 / NM;              // accumulators in the 512 TMEM columns
  static constexpr int ACC_COLS = TILE_N;              // TMEM columns of one accumulator
  static constexpr int SMEM = STAGES * (A_STAGE + B_STAGE) + EW * STG_WARP + 1024 /*align*/ +
                              512 /*barriers*/;
  static_assert(ACC_BUFS * ACC_COLS == TMEM_COLS, "TMEM budget");
};
constexpr int cmax(int a, int b) { return a > b ? a : b; }
constexpr int SMEM_BYTES = cmax(Geo<1, 1>::SMEM, cmax(Geo<2, 1>::SMEM, Geo<2, 2>::SMEM));

// First output column of B box j (0..3) of CTA `cta` in a tile starting at
// column n0.  A single CTA holds columns n0 .. n0+255 in order; a pair splits
// each 256-column half h of its tile, CTA c holding n0 + 256h + 128c + [0, 128),
// so that the two halves of one N = 256 MMA sit at the same shared-memory
// offset in both CTAs.
template <int PAIR>
__device__ __forceinline__ int b_box_col(int n0, int cta, int j) {
  return PAIR == 2 ? n0 + (j >> 1) * BN + cta * (BN / 2) + (j & 1) * B_BOX_N : n0 + j * B_BOX_N;
}

// Boxes (bit j) that start inside the N columns; the others are not loaded
// (their shared-memory slots keep stale data that only feeds columns >= N,
// which are never stored).  In a CTA pair a CTA with no column of the tile
// still loads box 0 (from the tile's first column; the results are never
// stored): the pair's MMAs wait only for the bytes its "full" barrier
// expects, so a CTA that loaded nothing into a stage (no rows of the unit
// either) could be lapped by two rounds of that stage and then wait for a
// phase of its "empty" barrier that parity cannot tell apart.
template <int PAIR, int NBOX>
__device__ __forceinline__ uint32_t b_box_mask(int N, int n0, int cta) {
  uint32_t m = 0;
#pragma unroll
  for (int j = 0; j < NBOX; ++j)
    if (b_box_col<PAIR>(n0, cta, j) < N) m |= 1u << j;
  if (PAIR == 2 && m == 0) m = 1u;
  return m;
}

enum Mode {
  MODE_STORE = 0,
  MODE_REDUCE = 1,
  MODE_MOE_GATHER = 2,
  MODE_MOE_SCATTER = 3,
  MODE_MOE_STAGED = 4,
  MODE_RS_CLUSTER = 5,
  // MOE_SCATTER on 256 x 512 pair tiles with one accumulator: for long
  // reductions (the accumulator's fp32 drain is short against the tile's main
  // loop and the wider tile receives fewer bytes per MMA), and for rank
  // groups whose partials are summed in TMEM before the adds (rs_group)
  MODE_MOE_SCATTER_WIDE = 6
};
// MoE layer1 (gate-weighted adds into the token rows), any tile form
__host__ __device__ constexpr bool is_scatter(int mode) {
  return mode == MODE_MOE_SCATTER || mode == MODE_MOE_SCATTER_WIDE;
}
__host__ __device__ constexpr bool is_moe(int mode) {
  return mode == MODE_MOE_GATHER || is_scatter(mode) || mode == MODE_MOE_STAGED;
}
// MOE_STAGED: rows per staging block (one ready count).  Small, so that the
// rows of the first units are spread over every copying CTA and ready early
// (8 rows: 10 us less per call than 32 at the MoE workload's sizes)
constexpr int STAGE_BLK = 8;
// MOE_STAGED with xcols: column tiles per group in the unit order (see
// decode_moe).  At the MoE workload's sizes (28 tiles per expert) groups of
// 4 / 8 / 16 / 28 gave 605 / 612 / 621 / 639 us: the fewer weight tiles in
// use at once, the better
constexpr int XCOL_GROUP = 4;
constexpr int STAGE_UNROLL = 16;  // MOE_STAGED: 16-byte loads in flight per lane

// device status header at the start of every workspace (256 bytes)
// H_CLAIM / H_EXIT: dynamic schedule's unit counter and count of finished
// CTAs (the last CTA out zeroes both and the mailboxes).  H_GRID /
// H_GRID_EXIT: MoE layer1's grid barrier before the row conversion and its
// exit count (the last CTA out zeroes both).
enum HdrField {
  H_STATUS = 0, H_WHERE = 1, H_ARG0 = 2, H_ARG1 = 3, H_ABORT = 4,
  H_CLAIM = 8, H_EXIT = 9, H_GRID = 10, H_GRID_EXIT = 11,
  H_FAST = 12  // dynamic schedule: regions that run as one full cluster (registered at start)
};
enum WaitSite {
  W_FLAG = 1,
  W_EMPTY = 2,
  W_FULL = 3,
  W_TEMPTY = 4,
  W_TFULL = 5,
  W_DRAIN = 6,
  W_TURN = 7,
  W_STAGE = 8,
  W_SCHED = 9,  // dynamic schedule: the region's next unit
  W_SHAPE = 10, // dynamic schedule: a cluster of an unexpected size or CTA order
  W_GRID = 11,  // MoE layer1: every CTA's adds in before the rows are converted
  W_XCHG = 12,  // cluster ReduceScatter: peers' rings free / partial rows received
  W_CHECK = 13  // checked build: a coordinate or address check failed (arg0 = CheckCode)
};
// What a failed check of the checked build was about (report arg0).
enum CheckCode {
  CK_A_ROW = 1,     // A box start row outside its tensor (or the shard index outside [0, R))
  CK_A_K = 2,       // A box k coordinate outside [0, K) or not 16-byte aligned
  CK_B_COL = 3,     // B box column outside [0, N) or not 16-byte aligned
  CK_B_K = 4,       // B box k coordinate outside [0, K)
  CK_OUT_ROW = 5,   // output row outside its buffer
  CK_OUT_COL = 6,   // output column outside its row (or not 16-byte aligned)
  CK_ACC_ROW = 7,   // fp32 accumulation row outside [0, M) (GEMM-RS) or token outside [0, T)
  CK_ACC_COL = 8,   // fp32 accumulation column outside [0, N)
  CK_OWNER = 9,     // owner rank outside [0, R)
  CK_PROBE = 15     // the deliberate failure requested by flux_opts_t.debug_probe
};
constexpr uint32_t ST_TIMEOUT = 5;
constexpr uint32_t ST_INVALID = 1;

struct KParams {
  CUtensorMap tmA[MAXR];   // per-rank A operand maps (K-major, 128B swizzle)
  CUtensorMap tmB[MAXR];   // per-rank B operand maps (N-major, 128B swizzle)
  CUtensorMap tmAcc;       // REDUCE: fp32 accumulation rows [M x N], 32 x 32 boxes
  CUtensorMap tmOut[MAXR]; // store modes: per-rank 16-bit outputs, 64-column x 32-row boxes
  void* out[MAXR];         // per-rank outputs
  const void* xsrc[MAXR];  // MOE_GATHER: per-shard token rows
  int R;
  int M;                   // rows of the A row space (AG: gathered rows; MoE: T*topk)
  int N;                   // output columns of one rank
  int K;                   // reduction length of one rank
  int Mt, Nt, KT;          // scheduled tiles along M (TILE_M rows), N, and k-slices
  int ldo;                 // output row pitch (elements)
  int rows_per_rank;       // AG: rows per X shard; RS: rows per owner chunk; MoE: tokens per rank
  int a_box_m;             // rows per A TMA box (AG)
  int group_n;             // raster band width in n-tiles
  int tiles_per_group;     // REDUCE: output tiles per rank-group
  int stream_k;            // REDUCE: 1 = contiguous k-step ranges per CTA
  int deterministic;       // REDUCE: ranks add their partials in ascending order
  int num_units;           // dense modes: number of work units
  int Nt_tile;             // REDUCE: output tiles (TILE_N columns) per row block, for the counters
  int num_claims;          // dynamic schedule: claim ids (units; see split_from, rs_group)
  int split_from;          // dynamic schedule, store mode: units from here on are claimed as
                           // two 256-column halves (num_units: none); reduce mode with
                           // rank groups: group claims from here on are claimed rank by rank
  long long total_ksteps;  // REDUCE stream-K: num_units * KT
  const uint32_t* flags;   // AG ready flags (nullptr = all ready)
  uint32_t epoch;
  uint32_t seq;            // per-call id, written to the abort word on error
  uint64_t timeout_ns;
  uint32_t* hdr;           // workspace header
  uint32_t* counters;      // REDUCE arrival counters
  float* acc;              // REDUCE / MOE_SCATTER fp32 accumulation rows
  // MoE routing (device arrays)
  const int32_t* offsets;      // [E+1]
  const int32_t* row_to_slot;  // [T*topk]
  const int32_t* tile_off;     // [E+1] first m-tile of each expert
  const float* topk_w;         // [T*topk]
  void* stage;                 // MOE_STAGED: grouped A rows [T*topk x H], 16-bit;
                               // push AG-GEMM: the gathered X [M x K], 16-bit
  uint32_t* unit_cnt;          // MOE_STAGED: finished staging blocks per m-unit (zeroed by routing);
                               // push AG-GEMM: copied 128-row blocks (one count each)
  int stage_ctas;              // MOE_STAGED / push: CTAs that copy rows before computing (0 = all)
  int push;                    // STORE: the push form of AllGather + GEMM (see push_rows)
  int push_rows_total;         // push: rows of X (the shards' rows back to back)
  int push_shard_rows;         // push: rows per X shard (the producers see one gathered shard)
  int E, topk, T, H;
  int moe_tp;  // MoE: ranks per expert group (R: tensor parallel, 1: expert parallel)
  int moe_el;  // MoE: experts per group; rank g moe_tp + t holds block t of group g's experts
  int moe_order;  // MoE: unit order (see decode_moe)
  // per-unit trace (nullptr = off): trace_words 64-bit words, TR_FIELDS per record
  unsigned long long* trace;
  long long trace_words;
  // dense CL = 4 kernels: units claimed at run time (see the dynamic schedule above)
  int dyn;
  int mbox_cap;    // mailbox entries per region
  uint32_t* mbox;  // [gridDim / 4 regions x mbox_cap] claimed unit + 1, or MBOX_DONE
  // regions made of pair clusters (slower: no multicast) stop claiming once at
  // most this many claims are left, and at most as many full-cluster regions
  // have registered, so that the faster regions take the last units (0 = off)
  int claim_reserve;
  // GEMM-RS, dynamic schedule: a claim is one output tile, and the region runs
  // the R ranks' partials of it back to back (R items per claim)
  int rs_tile_major;
  int rs_group;      // REDUCE, dynamic: ranks whose partials of one tile a region sums in
                     // TMEM before one drain (1 = each rank's partial drained on its own)
  int rs_direct;     // REDUCE, rs_group == R: a group's sum is the tile's result and is
                     // stored in the owner's 16-bit rows (tmOut[owner]) without fp32 rows
  int debug_probe;  // checked build: nonzero makes CTA 0 fail one check (CK_PROBE) on purpose
  int acc_halves;   // one 512-column accumulator: handed back in two 256-column halves
  // MOE_SCATTER_WIDE with rank groups: arrivals per (token, 512-column tile)
  // [T x row_tiles] (nullptr: the end-of-call pass converts every token
  // row).  The add that brings a tile of a token to row_arrivals (topk x
  // the group count per slot) converts it and zeroes it and its count.
  uint32_t* row_cnt;
  int row_tiles;
  int row_arrivals;
  // MOE_STAGED: the output columns of an expert group's ranks side by side
  // (N = moe_tp x xcols), xcols columns per rank, a multiple of 64: a column
  // tile may span two ranks (each 64-column B box and output box lies in
  // one); units carry no rank.  0: tiles within one rank's columns
  int xcols;
};

constexpr uint32_t MBOX_DONE = 0xFFFFFFFFu;
// k-slices before the end of its current unit at which a region claims the next
// (the other CTAs of the region read it when they finish the current unit)
constexpr int CLAIM_AHEAD = 8;

struct Ctl {
  uint32_t* hdr;
  uint32_t seq;
  uint64_t flag_timeout;
  uint64_t pipe_timeout;
};

__device__ __forceinline__ bool aborted(const Ctl& c) {
  return ld_volatile_u32(c.hdr + H_ABORT) == c.seq;
}

static __device__ __noinline__ void raise_error(const Ctl& c, uint32_t code, uint32_t where,
                                                uint32_t a0, uint32_t a1) {
  if (atomicCAS(c.hdr + H_STATUS, 0u, code) == 0u) {
    c.hdr[H_WHERE] = where;
    c.hdr[H_ARG0] = a0;
    c.hdr[H_ARG1] = a1;
  }
  __threadfence();
  atomicExch(c.hdr + H_ABORT, c.seq);
}

// Checked build: true when `cond` holds; otherwise records the failure (first
// error wins, the call is aborted so that the other roles leave) and returns
// false.  Always true in the regular build.
__device__ __forceinline__ bool check_ok(const Ctl& c, bool cond, uint32_t code, uint32_t value) {
#if FLUX_CHECKS
  if (!cond) raise_error(c, ST_INVALID, W_CHECK, code, value);
  return cond;
#else
  (void)c; (void)code; (void)value;
  return true;
#endif
}

// Waits that have not finished within this many SM cycles start the (slow)
// checks of the global timer and the abort word; a healthy pipeline never gets
// there, so the hot path costs one probe per iteration.
constexpr long long LAZY_CHECK_CYCLES = 1ll << 20;

// Bounded mbarrier wait.  0 = phase completed, 1 = timed out (recorded),
// 2 = another thread aborted this call.  `check_abort` = false is used by the
// final drains, which must outlive an abort.
static __device__ __noinline__ int wait_bar_slow(uint32_t bar, uint32_t parity, const Ctl& c,
                                                 uint32_t where, uint32_t arg1, bool check_abort) {
  const long long c0 = clock64();
  uint64_t t0 = 0;
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return 0;
    if ((it & 63u) == 0u && (clock64() - c0 > LAZY_CHECK_CYCLES || it > (1u << 24))) {
      if (t0 == 0) t0 = globaltimer();
      if (check_abort && aborted(c)) return 2;
      if (globaltimer() - t0 > c.pipe_timeout || it > (1u << 30)) {
        raise_error(c, ST_TIMEOUT, where, blockIdx.x, arg1);
        return 1;
      }
    }
  }
}

__device__ __forceinline__ int wait_bar(uint32_t bar, uint32_t parity, const Ctl& c,
                                        uint32_t where, uint32_t arg1, bool check_abort = true) {
  if (mbar_try_wait(bar, parity)) return 0;
  return wait_bar_slow(bar, parity, c, where, arg1, check_abort);
}

// Drain form of wait_bar_remote: ignores the abort word (the copies being
// waited for must land even when the call aborted).
static __device__ __noinline__ int wait_bar_remote_drain(uint32_t bar, uint32_t parity,
                                                         const Ctl& c, uint32_t where, uint32_t arg1) {
  const long long c0 = clock64();
  uint64_t t0 = 0;
  for (uint32_t it = 1;; ++it) {
    if (mbar_test_wait(bar, parity)) return 0;
    if ((it & 255u) == 0u && (clock64() - c0 > LAZY_CHECK_CYCLES || it > (1u << 24))) {
      if (t0 == 0) t0 = globaltimer();
      if (globaltimer() - t0 > c.pipe_timeout || it > (1u << 30)) {
        raise_error(c, ST_TIMEOUT, where, blockIdx.x, arg1);
        return 1;
      }
    }
  }
}

// The same bound for a barrier completed by another CTA of the cluster: polled
// with the non-blocking test_wait.
static __device__ __noinline__ int wait_bar_remote(uint32_t bar, uint32_t parity, const Ctl& c,
                                                   uint32_t where, uint32_t arg1) {
  if (mbar_test_wait(bar, parity)) return 0;
  const long long c0 = clock64();
  uint64_t t0 = 0;
  for (uint32_t it = 1;; ++it) {
    if (mbar_test_wait(bar, parity)) return 0;
    if ((it & 255u) == 0u && (clock64() - c0 > LAZY_CHECK_CYCLES || it > (1u << 24))) {
      if (t0 == 0) t0 = globaltimer();
      if (aborted(c)) return 2;
      if (globaltimer() - t0 > c.pipe_timeout || it > (1u << 30)) {
        raise_error(c, ST_TIMEOUT, where, blockIdx.x, arg1);
        return 1;
      }
    }
  }
}

// Bounded wait for ready_flags[s] >= epoch (acquire at gpu scope).  True when ready.
static __device__ __noinline__ bool wait_flag(const uint32_t* flags, int s, uint32_t epoch,
                                              const Ctl& c) {
  uint32_t v = ld_acquire_u32(flags + s);
  if (v >= epoch) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    __nanosleep(128);
    v = ld_acquire_u32(flags + s);
    if (v >= epoch) return true;
    if ((it & 7u) == 0u) {
      if (aborted(c)) return false;
      if (globaltimer() - t0 > c.flag_timeout || it > (1u << 28)) {
        raise_error(c, ST_TIMEOUT, W_FLAG, static_cast<uint32_t>(s), v);
        return false;
      }
    }
  }
}

// Bounded wait until *cnt >= target (acquire at gpu scope): the deterministic
// GEMM-RS turn of one rank on one 32-row quarter (W_TURN), or the staged rows
// of one MoE m-unit (W_STAGE).  True when reached.
static __device__ __noinline__ bool wait_count(const uint32_t* cnt, uint32_t target, const Ctl& c,
                                               uint32_t where) {
  uint32_t v = ld_acquire_u32(cnt);
  if (v >= target) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    __nanosleep(64);
    v = ld_acquire_u32(cnt);
    if (v >= target) return true;
    if ((it & 7u) == 0u) {
      if (aborted(c)) return false;
      if (globaltimer() - t0 > c.pipe_timeout || it > (1u << 28)) {
        raise_error(c, ST_TIMEOUT, where, target, v);
        return false;
      }
    }
  }
}

// ---------------------------------------------------------------- tile schedule
// Band raster: bands of `group_n` n-tiles; inside a band the m-tile index runs
// fastest, so the CTAs of one wave share a few B column tiles and sweep A.
__device__ __forceinline__ void raster(int t, int Mt, int Nt, int group_n, int& mt, int& nt) {
  const int band = Mt * group_n;
  const int g = t / band;
  const int local = t - g * band;
  mt = local % Mt;
  nt = g * group_n + local / Mt;
}

struct Work {
  int r;       // rank whose operands feed the tile
  int mt, nt;  // scheduled tile coordinates (mt counts TILE_M-row tiles)
  int n0, n_end;  // the item's output columns [n0, n_end) (a tile, or half of one)
  int m0;      // first A row of THIS CTA's part of the tile
  int row_end; // rows >= row_end are not part of the tile's problem
  int e;       // expert (MoE)
  int k0, k1;  // k-slice range of this item
  int tile;    // linear 128-row output-tile id of this CTA's part (REDUCE counters)
  int rsub;    // rank groups / tile-major GEMM-RS: place of this rank's partial in the
               // tile's rank group
  int rcnt;    // rank groups / tile-major GEMM-RS: the group's size
  int uid;     // the unit (or claim) id the item came from (traces)
};

// Trace record of one work item of one CTA: eight 64-bit words.
//   0  tag: unit id + 1 (bits 0..31), rank (32..39), k-slice range start (40..63)
//   1  producer: the item's first k-slice may be issued (flags and claims done)
//   2  producer: its last k-slice issued
//   3  MMA (even CTA of a pair): the accumulator is free
//   4  MMA: the first k-slice's operands have landed
//   5  MMA: the last k-slice's MMAs issued and committed
//   6  epilogue (first epilogue warp): the accumulator is full
//   7  epilogue: the item's stores or adds are issued (for GEMM-RS, its
//      arrival counted and, if last, its rows converted)
// The first eight words are a header (word 0: gridDim.x, word 1: records per
// CTA); the records of CTA b start at trace + 8 + b * items * 8, items =
// (trace_words - 8) / (8 * gridDim.x); items beyond that are not recorded.
enum TraceField {
  TR_TAG = 0, TR_PROD_START = 1, TR_PROD_END = 2, TR_MMA_ACC = 3, TR_MMA_FIRST = 4,
  TR_MMA_END = 5, TR_EPI_FULL = 6, TR_EPI_END = 7, TR_FIELDS = 8
};

// Record field `f` of this CTA's item `item` (no-op without a trace buffer).
__device__ __forceinline__ void trace_put(const KParams& p, int item, int f, unsigned long long v) {
#if FLUX_TRACE
  if (p.trace == nullptr) return;
  const long long per_cta = (p.trace_words - TR_FIELDS) / (TR_FIELDS * static_cast<long long>(gridDim.x));
  if (item >= per_cta) return;
  p.trace[TR_FIELDS + (static_cast<long long>(blockIdx.x) * per_cta + item) * TR_FIELDS + f] = v;
#endif
}
__device__ __forceinline__ void trace_now(const KParams& p, int item, int f) {
#if FLUX_TRACE
  if (p.trace != nullptr) trace_put(p, item, f, globaltimer());
#endif
}
__device__ __forceinline__ void trace_tag(const KParams& p, int item, const Work& w) {
#if FLUX_TRACE
  if (p.trace != nullptr)
    trace_put(p, item, TR_TAG,
              (static_cast<unsigned long long>(static_cast<uint32_t>(w.uid + 1))) |
                  (static_cast<unsigned long long>(w.r & 0xFF) << 32) |
                  (static_cast<unsigned long long>(w.k0 & 0xFFFFFF) << 40));
#endif
}

// Shape of the work of one cluster of CL CTAs (128 rows of A per CTA).
//   dense modes, CL 2 / 4: CTA pairs with 256 x 512 tiles (MC pairs share B)
//   MOE_SCATTER, CL 2: one CTA pair, 256 x 256 tiles (_WIDE: 256 x 512)
//   MOE_GATHER: single CTAs only (cp.async row gather)
//   MOE_STAGED, CL 2: one CTA pair, 256 x 512 tiles
template <int MODE, int CL>
struct Unit {
  static constexpr bool DENSE = MODE == MODE_STORE || MODE == MODE_REDUCE;
  // RS_CLUSTER: every CTA of the cluster runs its own 128 x 256 tiles
  static constexpr int PAIR = (CL >= 2 && MODE != MODE_RS_CLUSTER) ? 2 : 1;
  // GEMM-RS in regions of 8: 256 x 256 pair tiles (two accumulators, so the
  // fp32 adds of one tile overlap the next tile's MMAs); the other dense and
  // wide forms: 256 x 512 pair tiles
  static constexpr int NM =
      (MODE == MODE_REDUCE && CL == 8) ? 1
      : ((DENSE || MODE == MODE_MOE_STAGED || MODE == MODE_MOE_SCATTER_WIDE) && PAIR == 2) ? 2 : 1;
  static constexpr int EW = EPI_WARPS;
  // pairs side by side along N (share A by multicast) and stacked along M
  // (share B by multicast)
  static constexpr int PN = (DENSE && CL == 8) ? 2 : 1;
  static constexpr int PM = MODE == MODE_RS_CLUSTER ? 1 : CL / PAIR / PN;
  static constexpr int MC = PM;
  static constexpr int ROWS = BM * PAIR * PM;
  using G = Geo<PAIR, NM, EW>;
  static constexpr int UNIT_N = G::TILE_N * PN;
  static_assert(DENSE || MC == 1, "MoE tiles: no B sharing between pairs");
  static_assert(MODE != MODE_MOE_GATHER || CL == 1, "MoE layer0 gather: single CTAs");
  static_assert(MODE != MODE_MOE_STAGED || CL == 2, "MoE layer0 staged: CTA pairs");
};

template <int MODE, int DT, int CL>
struct KernelShape {
  // the cp.async row gather (single-CTA MoE layer0) takes four producer warps
  static constexpr bool CPASYNC_GATHER = MODE == MODE_MOE_GATHER && CL == 1;
  static constexpr int PRODUCER_WARPS = CPASYNC_GATHER ? 4 : 1;
  static constexpr int MMA_WARP = PRODUCER_WARPS;
  static constexpr int EPI_WARP0 = PRODUCER_WARPS + 1;
  static constexpr int EPI = EPI_WARPS;
  static constexpr int THREADS = 32 * (PRODUCER_WARPS + 1 + EPI);
  static constexpr int FULL_COUNT = CPASYNC_GATHER ? (BM + 1) : 1;
};

// AllGather / plain GEMM: unit -> (rank, m-tile, n-tile).  Ranks are the
// outer loop; inside a rank the m order is rotated so that rank r starts with
// the rows it owns (the local shard is the first to be ready) and then walks
// the other ranks' shards in ring order.  `cta` is the CTA's rank in its
// cluster; it holds rows m0 .. m0+127 of the unit.
template <int CL>
__device__ __forceinline__ Work decode_store(const KParams& p, int u, int cta) {
  constexpr int TM = Unit<MODE_STORE, CL>::ROWS;
  Work w;
  const int per_rank = p.Mt * p.Nt;
  w.r = u / per_rank;
  int mt, nt;
  raster(u - w.r * per_rank, p.Mt, p.Nt, p.group_n, mt, nt);
  const int mt_per_shard = p.rows_per_rank / TM;
  if (mt_per_shard > 0 && p.rows_per_rank % TM == 0) mt = (mt + w.r * mt_per_shard) % p.Mt;
  using U = Unit<MODE_STORE, CL>;
  const int pr = cta / U::PAIR;  // pair of the region
  w.mt = mt;
  w.nt = nt;
  w.n0 = nt * U::UNIT_N + (pr / U::PM) * U::G::TILE_N;
  w.n_end = min(p.N, w.n0 + U::G::TILE_N);
  w.m0 = mt * TM + (pr % U::PM) * (BM * U::PAIR) + (cta % U::PAIR) * BM;
  w.row_end = p.M;
  w.e = 0;
  w.k0 = 0;
  w.k1 = p.KT;
  w.tile = 0;
  w.rsub = 0;
  w.rcnt = 1;
  w.uid = u;
  return w;
}

// GEMM + ReduceScatter: unit -> (tile group, rank, tile).  The R partials of
// one output tile are `tiles_per_group` units apart, so with a strided
// persistent schedule they land in consecutive waves while the owner's fp32
// tile is still in L2.
template <int CL>
__device__ __forceinline__ Work decode_reduce(const KParams& p, int u, int cta) {
  constexpr int TM = Unit<MODE_REDUCE, CL>::ROWS;
  Work w;
  const int tiles = p.Mt * p.Nt;
  const int TG = p.tiles_per_group;
  const int full_groups = tiles / TG;
  int t;
  if (u < full_groups * TG * p.R) {
    const int g = u / (TG * p.R);
    const int rem = u - g * TG * p.R;
    w.r = rem / TG;
    t = g * TG + (rem - w.r * TG);
  } else {
    const int tl = tiles - full_groups * TG;
    const int rem = u - full_groups * TG * p.R;
    w.r = rem / tl;
    t = full_groups * TG + (rem - w.r * tl);
  }
  raster(t, p.Mt, p.Nt, p.group_n, w.mt, w.nt);
  using U = Unit<MODE_REDUCE, CL>;
  const int pr = cta / U::PAIR;  // pair of the region
  w.n0 = w.nt * U::UNIT_N + (pr / U::PM) * U::G::TILE_N;
  w.n_end = min(p.N, w.n0 + U::G::TILE_N);
  w.m0 = w.mt * TM + (pr % U::PM) * (BM * U::PAIR) + (cta % U::PAIR) * BM;
  // counters: 128-row block x output tile (TILE_N columns) of this CTA's part
  w.tile = (w.m0 / BM) * p.Nt_tile + w.n0 / U::G::TILE_N;
  w.row_end = p.M;
  w.e = 0;
  w.k0 = 0;
  w.k1 = p.KT;
  w.rsub = 0;
  w.rcnt = 1;
  w.uid = u;
  return w;
}

// MoE: unit -> (rank, grouped m-unit, n-tile); the expert of an m-unit comes
// from the device table of each expert's first unit (units of BM * CL rows)
// written by the routing kernel.  `cta` picks the 128-row part of the unit.
// An m-unit of expert e runs on the moe_tp ranks of e's group g = e / moe_el
// (ranks g moe_tp + [0, moe_tp)), each with its block of the expert's weight
// (local expert e % moe_el).  Tensor parallel: one group of R ranks; expert
// parallel: R groups of one rank.  Unit order (moe_order):
//   0  rank outermost, then bands of group_n n-tiles with the m-tile fastest
//   1  rank innermost: the ranks' tiles of one (m, n) are consecutive units
//   2  band outermost, then rank, then the m-tile fastest inside the band
//   3  expert outermost, then n-tile, then the expert's m-units, rank fastest:
//      the weight blocks of one expert column tile and the expert's rows are
//      in use together, and each is read while the other stays in L2.  With
//      xcols (no rank index) the column tiles take the ranks' place in groups
//      of XCOL_GROUP: expert, group, m-unit, tile of the group fastest, so
//      that consecutive units share the rows (in L2) and not a weight tile
//      (streamed from DRAM: units that start together on one weight tile all
//      wait on the same misses)
//   5  rank innermost, then the n-tiles of one m-unit, then the m-units: the
//      rows of an m-unit serve all its column tiles while they are in L2
template <int CL>
__device__ __forceinline__ Work decode_moe(const KParams& p, int u, int total_mt, int cta, int tile_n) {
  Work w;
  const int per_rank = total_mt * p.Nt;
  int tr, t;  // rank inside the expert's group; the unit's index among that rank's
  int gmt, nt;
  int lo = 0, hi = p.E;  // the m-unit's expert: largest e with tile_off[e] <= gmt
  if (p.moe_order == 3 && p.xcols > 0) {
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(p.tile_off + mid) * p.Nt <= u) lo = mid; else hi = mid;
    }
    const int t0 = __ldg(p.tile_off + lo);
    const int ke = __ldg(p.tile_off + lo + 1) - t0;  // >= 1: u lies in this expert's units
    const int local = u - t0 * p.Nt;
    const int full = p.Nt / XCOL_GROUP;  // whole groups of column tiles
    int g0, gs, rem;                     // the group's first tile and size; the unit inside it
    if (local < full * XCOL_GROUP * ke) {
      const int g = local / (XCOL_GROUP * ke);
      g0 = g * XCOL_GROUP;
      gs = XCOL_GROUP;
      rem = local - g * XCOL_GROUP * ke;
    } else {
      g0 = full * XCOL_GROUP;
      gs = p.Nt - g0;
      rem = local - full * XCOL_GROUP * ke;
    }
    gmt = t0 + rem / gs;
    nt = g0 + (rem - (rem / gs) * gs);
    tr = 0;
  } else if (p.moe_order == 3) {
    const int per_mt = p.Nt * p.moe_tp;  // units per m-unit
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(p.tile_off + mid) * per_mt <= u) lo = mid; else hi = mid;
    }
    const int t0 = __ldg(p.tile_off + lo);
    const int ke = __ldg(p.tile_off + lo + 1) - t0;  // >= 1: u lies in this expert's units
    const int local = u - t0 * per_mt;
    nt = local / (ke * p.moe_tp);
    const int rem = local - nt * ke * p.moe_tp;
    gmt = t0 + rem / p.moe_tp;
    tr = rem - (rem / p.moe_tp) * p.moe_tp;
  } else {
    if (p.moe_order == 1 || p.moe_order == 5) {
      tr = u % p.moe_tp;
      t = u / p.moe_tp;
    } else if (p.moe_order == 2) {
      const int gn = p.group_n;
      const int full = p.Nt / gn;              // full bands
      const int band = total_mt * gn;          // one rank's units in a full band
      const int done = full * band * p.moe_tp;
      if (u < done) {
        const int g = u / (band * p.moe_tp);
        const int rem = u - g * band * p.moe_tp;
        tr = rem / band;
        t = g * band + (rem - tr * band);
      } else {
        const int tail = total_mt * (p.Nt - full * gn);
        const int rem = u - done;
        tr = rem / tail;
        t = full * band + (rem - tr * tail);
      }
    } else {
      tr = u / per_rank;
      t = u - tr * per_rank;
    }
    if (p.moe_order == 5) {
      gmt = t / p.Nt;
      nt = t - gmt * p.Nt;
    } else {
      // m-tile fastest inside bands of group_n n-tiles
      raster(t, total_mt, p.Nt, p.group_n, gmt, nt);
    }
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(p.tile_off + mid) <= gmt) lo = mid; else hi = mid;
    }
  }
  const int grp = lo / p.moe_el;
  w.r = grp * p.moe_tp + tr;
  w.e = lo - grp * p.moe_el;  // index into rank r's experts
  const int e_off = __ldg(p.offsets + lo);
  w.m0 = e_off + (gmt - __ldg(p.tile_off + lo)) * (BM * CL) + cta * BM;
  w.row_end = __ldg(p.offsets + lo + 1);
  w.mt = gmt;
  w.nt = nt;
  w.n0 = nt * tile_n;
  w.n_end = min(p.N, w.n0 + tile_n);
  w.k0 = 0;
  w.k1 = p.KT;
  w.tile = 0;
  w.rsub = 0;
  w.rcnt = 1;
  return w;
}

// GEMM-RS with rank groups (rs_group = G > 1): claim c stands for the G units
// of one output tile whose ranks form group rg; the claims follow the unit
// order of decode_reduce with the ranks taken G at a time (rank group rg of
// tile group g: units g TG R + (rg G + j) TG + t, j < G).  Returns the unit
// of the claim's j-th rank.
__device__ __forceinline__ int rs_group_unit(const KParams& p, int c, int j) {
  const int G = p.rs_group, RG = p.R / G;
  const int tiles = p.Mt * p.Nt;
  const int TG = p.tiles_per_group;
  const int full_groups = tiles / TG;
  const int full_claims = full_groups * TG * RG;
  int base, tgg, rem;
  if (c < full_claims) {
    const int g = c / (TG * RG);
    rem = c - g * TG * RG;
    base = g * TG * p.R;
    tgg = TG;
  } else {
    rem = c - full_claims;
    base = full_groups * TG * p.R;
    tgg = tiles - full_groups * TG;
  }
  const int rg = rem / tgg, t = rem - rg * tgg;
  return base + (rg * G + j) * tgg + t;
}

// Iterates the items of this CTA identically in every role.  All CTAs of a
// cluster (of a region, under the dynamic schedule) walk the same units
// (region index = blockIdx / CL).  `cta` is the CTA's part of the unit.
// Static schedule: units u, u + stride, ... of the persistent grid.  Dynamic
// schedule: the units the region's mailbox receives, in order; `warp_uniform`
// (a whole warp calls next) makes lane 0 read the mailbox for the warp.
template <int MODE, int CL>
struct ItemIter {
  // dense tiles in regions of two or four pairs; the staged MoE layer0 in
  // regions of one pair (its unit count comes from the device tile table)
  static constexpr bool DYN_OK =
      (Unit<MODE, CL>::DENSE && (CL == 4 || CL == 8)) ||
      ((MODE == MODE_MOE_STAGED || MODE == MODE_MOE_SCATTER_WIDE) && CL == 2);
  // rank groups summed in TMEM (rs_group > 1): GEMM-RS, and MoE layer1 on
  // 256 x 512 tiles with the ranks innermost in the unit order (moe_order 1)
  static constexpr bool GROUPS = MODE == MODE_REDUCE || MODE == MODE_MOE_SCATTER_WIDE;
  const KParams& p;
  const Ctl* ctl;
  int total_mt;      // MoE: device-computed number of m-tiles
  int num_units;
  long long pos, end;  // stream-K k-step range
  int u, stride, cta;
  bool dyn, warp_uniform;
  uint32_t* box;     // dynamic: the region's mailbox
  int taken;         // dynamic: mailbox entries read so far
  int sub;           // tile-major GEMM-RS / rank groups: next rank of the tile
  int cur_claim;     // tile-major GEMM-RS / rank groups: the claim this region took last
  int msplit;        // MoE layer1 rank groups: group claims from here on go out rank by rank

  __device__ ItemIter(const KParams& p_, int total_mt_, int cta_, const Ctl* ctl_ = nullptr,
                      bool warp_uniform_ = false)
      : p(p_), ctl(ctl_), total_mt(total_mt_), cta(cta_), warp_uniform(warp_uniform_) {
    if (is_moe(MODE)) {
      num_units = total_mt * p.Nt * (p.xcols > 0 ? 1 : p.moe_tp);
    } else {
      num_units = p.num_units;
    }
    sub = 0;
    cur_claim = 0;
    u = blockIdx.x / CL;
    stride = gridDim.x / CL;
    msplit = 0;
    if (MODE == MODE_MOE_SCATTER_WIDE && p.rs_group > 1) {
      // the last split_from group claims (a count, 0 = none) go out rank by rank
      const int groups = num_units / p.rs_group;
      msplit = groups > p.split_from ? groups - p.split_from : 0;
    }
    dyn = DYN_OK && p.dyn != 0 && ctl != nullptr;
    box = dyn ? p.mbox + static_cast<size_t>(u) * p.mbox_cap : nullptr;
    taken = 0;
    if (MODE == MODE_REDUCE && p.stream_k) {
      const long long L = p.total_ksteps;
      pos = L * u / stride;
      end = L * (u + 1) / stride;
    }
  }

  // dynamic schedule: how many claim ids the counter hands out
  __device__ int claims() const {
    if (MODE == MODE_MOE_SCATTER_WIDE && p.rs_group > 1)
      return msplit + (num_units / p.rs_group - msplit) * p.rs_group;
    return is_moe(MODE) ? num_units : p.num_claims;
  }

  __device__ bool next(Work& w) {
    if (MODE == MODE_RS_CLUSTER) {
      // the cluster's n-tile u; this CTA's ranks cta, cta + CL, ...
      const int r = cta + taken * CL;
      if (u >= p.Nt || r >= p.R) return false;
      ++taken;
      w.r = r;
      w.mt = 0;
      w.nt = u;
      w.n0 = u * BN;
      w.n_end = min(p.N, w.n0 + BN);
      w.m0 = 0;
      w.row_end = p.M;
      w.e = 0;
      w.k0 = 0;
      w.k1 = p.KT;
      w.tile = 0;
      w.rsub = 0;
      w.rcnt = 1;
      w.uid = u * MAXR + r;
      return true;
    }
    if (DYN_OK && dyn) {
      if (GROUPS && sub > 0) {
        // the next rank of the tile this region claimed (tile-major: all R
        // ranks; rank groups: the group's G)
        const int cnt = p.rs_tile_major ? p.R : p.rs_group;
        if (MODE == MODE_REDUCE)
          w = decode_reduce<CL>(p, p.rs_tile_major ? cur_claim * p.R + sub : rs_group_unit(p, cur_claim, sub),
                                cta);
        else
          w = decode_moe<CL>(p, cur_claim * cnt + sub, total_mt, cta, Unit<MODE, CL>::G::TILE_N);
        w.rsub = sub;
        w.rcnt = cnt;
        w.uid = cur_claim;
        if (++sub == cnt) sub = 0;
        return true;
      }
      uint32_t v = 0;
      if (!warp_uniform || (threadIdx.x & 31) == 0) {
        // bounded: a timeout is recorded, an abort ends the walk
        if (wait_count(box + taken, 1u, *ctl, W_SCHED)) v = ld_acquire_u32(box + taken);
      }
      if (warp_uniform) v = __shfl_sync(0xFFFFFFFFu, v, 0);
      ++taken;
      if (v == 0u || v == MBOX_DONE) return false;
      const int id = static_cast<int>(v - 1u);
      if (MODE == MODE_STORE) {
        if (CL != 4 || id < p.split_from) {
          w = decode_store<CL>(p, id, cta);
        } else {
          // the last units are claimed as two 256-column halves
          const int half = (id - p.split_from) & 1;
          w = decode_store<CL>(p, p.split_from + ((id - p.split_from) >> 1), cta);
          w.n0 += half * BN;
          w.n_end = min(w.n_end, w.n0 + BN);
        }
      } else if (MODE == MODE_MOE_SCATTER_WIDE && p.rs_group > 1) {
        // rank innermost: the group of claim c is units c G .. c G + G - 1
        const int G = p.rs_group;
        if (id >= msplit) {
          const int j = id - msplit;
          w = decode_moe<CL>(p, (msplit + j / G) * G + j % G, total_mt, cta, Unit<MODE, CL>::G::TILE_N);
        } else {
          cur_claim = id;
          w = decode_moe<CL>(p, id * G, total_mt, cta, Unit<MODE, CL>::G::TILE_N);
          w.rsub = 0;
          w.rcnt = G;
          sub = 1;
        }
      } else if (is_moe(MODE)) {
        w = decode_moe<CL>(p, id, total_mt, cta, Unit<MODE, CL>::G::TILE_N);
      } else if (p.rs_tile_major) {
        // claim id = output tile; its rank 0 now, the other ranks next
        cur_claim = id;
        w = decode_reduce<CL>(p, id * p.R, cta);
        w.rsub = 0;
        w.rcnt = p.R;
        sub = p.R > 1 ? 1 : 0;
      } else if (MODE == MODE_REDUCE && p.rs_group > 1 && id >= p.split_from) {
        // the last rank groups are claimed rank by rank (their partials added
        // one by one), so that the regions run out of work at about the same time
        const int j = id - p.split_from;
        w = decode_reduce<CL>(p, rs_group_unit(p, p.split_from + j / p.rs_group, j % p.rs_group), cta);
      } else if (MODE == MODE_REDUCE && p.rs_group > 1) {
        // claim id = one tile's rank group; its first rank now, the others next
        cur_claim = id;
        w = decode_reduce<CL>(p, rs_group_unit(p, id, 0), cta);
        w.rsub = 0;
        w.rcnt = p.rs_group;
        sub = 1;
      } else {
        w = decode_reduce<CL>(p, id, cta);
      }
      w.uid = id;
      return true;
    }
    if (MODE == MODE_REDUCE && p.stream_k) {
      if (pos >= end) return false;
      const int unit = static_cast<int>(pos / p.KT);
      const int k0 = static_cast<int>(pos - static_cast<long long>(unit) * p.KT);
      long long k1 = k0 + (end - pos);
      if (k1 > p.KT) k1 = p.KT;
      w = decode_reduce<CL>(p, unit, cta);
      w.k0 = k0;
      w.k1 = static_cast<int>(k1);
      w.uid = unit;
      pos += k1 - k0;
      return true;
    }
    if (u >= num_units) return false;
    if (MODE == MODE_STORE) w = decode_store<CL>(p, u, cta);
    else if (MODE == MODE_REDUCE) w = decode_reduce<CL>(p, u, cta);
    else w = decode_moe<CL>(p, u, total_mt, cta, Unit<MODE, CL>::G::TILE_N);
    w.uid = u;
    u += stride;
    return true;
  }
};

// Dynamic schedule: the region's first CTA writes its next claim id (+ 1)
// into entry j of the region's mailbox, or MBOX_DONE once the counter has run
// out or the mailbox is full (then the other regions take the remaining
// claims: the mailboxes together hold more entries than there are claims).
// The counter hands out ids below num_claims: the host's count for the dense
// ops, the device-computed unit count for MoE layer0.  Store mode: ids from
// split_from on are the two 256-column halves of the last units; a half
// without columns is skipped here.
template <int MODE, int CL>
__device__ __forceinline__ void claim_unit(const KParams& p, uint32_t* box, int j, bool slow,
                                           int num_claims) {
  if (j >= p.mbox_cap) return;  // past the region's DONE entry: never read, never written
  uint32_t v = MBOX_DONE;
  bool stop = false;
  if (slow && p.claim_reserve > 0) {
    // leave the last claims to the full-cluster regions (one each at most);
    // they registered before their first claim and claim until the counter
    // runs out, so no unit is left behind
    const uint32_t fast = min(ld_volatile_u32(p.hdr + H_FAST), static_cast<uint32_t>(p.claim_reserve));
    const uint32_t seen = ld_volatile_u32(p.hdr + H_CLAIM);
    stop = fast > 0 && seen + fast >= static_cast<uint32_t>(num_claims);
  }
  if (j < p.mbox_cap - 1 && !stop) {
    for (;;) {
      const uint32_t u = atomicAdd(p.hdr + H_CLAIM, 1u);
      if (u >= static_cast<uint32_t>(num_claims)) break;
      const int id = static_cast<int>(u);
      // the second half of a last unit narrower than 257 columns has no columns
      if (MODE == MODE_STORE && CL == 4 && id >= p.split_from && ((id - p.split_from) & 1) &&
          decode_store<CL>(p, p.split_from + ((id - p.split_from) >> 1), 0).n0 + BN >= p.N)
        continue;
      v = u + 1u;
      break;
    }
  }
  st_release_u32(box + j, v);
}

// Where a CTA sits.  vrank: its 128-row part of the unit (0 .. CL-1); hw_rank,
// hw_cl: its rank in, and the size of, the cluster it was launched in (under
// the dynamic schedule a region may be two pair clusters); mc2: the unit's two
// pairs share B by multicast (one cluster holds both).
struct Pos {
  int vrank;
  int hw_rank;
  int hw_cl;
  bool mc2;
};

// ---------------------------------------------------------------- roles
struct Smem {
  uint8_t* a;       // STAGES x A_STAGE
  uint8_t* b;       // STAGES x B_STAGE
  uint64_t* full;   // [STAGES] this CTA's operands landed
  uint64_t* empty;  // [STAGES] the MMAs reading the stage completed
  uint64_t* tfull;  // [2]
  uint64_t* tempty; // [2]
  uint64_t* thalf;  // [2] the accumulator's first 256 columns read (acc_halves)
  uint64_t* drain;  // [1]
  uint32_t* tmem_slot;
  uint32_t* misc;   // [2] dynamic schedule: cluster-shape check, last CTA out
  uint64_t* xbar;   // [2] RS_CLUSTER: peers' rings free, partial rows received
  uint8_t* stg;     // EPI_WARPS x STG_WARP epilogue staging (1024-byte aligned)
};

// Bytes the odd CTA of a pair loads for one stage of work item `w` (the even
// CTA's view of the item): its 128 rows of A and its columns of B.
template <int MODE, class G>
__device__ __forceinline__ uint32_t pair_peer_bytes(const KParams& p, const Work& w) {
  const int m0 = w.m0 + BM;
  int nbox_a = m0 < w.row_end ? 1 : 0;
  uint32_t a = nbox_a * A_STAGE;
  if (MODE == MODE_STORE && nbox_a)
    a = ((min(m0 + BM, w.row_end) - m0 + p.a_box_m - 1) / p.a_box_m) * p.a_box_m * BK * 2;
  const uint32_t mask = b_box_mask<2, G::B_BOXES>(w.n_end, w.n0, 1);
  return a + __popc(mask) * B_BOX_N * BK * 2;
}

// The k-slices [kb, ke) of work item `w` (TMA producer thread).  MC2: the
// pairs of a 4-CTA cluster share B by multicast (compile-time, so that the
// per-slice loop carries no branch on it).  False when a wait gave up.
template <int MODE, int CL, bool MC2>
__device__ __forceinline__ bool produce_ksteps(const KParams& p, const Smem& s, const Ctl& c,
                                               const Work& w, int kb, int ke, int nbox_a,
                                               uint32_t bmask, uint32_t bytes, int n0, int cta,
                                               int half, uint16_t mc_mask, int hw_rank,
                                               uint32_t& stage, uint32_t& phase, uint32_t& issued) {
  // PN = 2: this CTA and its N neighbour (hw_rank ^ 4) hold the same A rows;
  // each issues one of the two 64-row A boxes as a multicast to both
  constexpr bool MCA = Unit<MODE, CL>::PN == 2;
  const uint16_t mask_a = static_cast<uint16_t>((1u << hw_rank) | (1u << (hw_rank ^ 4)));
  const int a_half = (hw_rank >> 2) & 1;
  constexpr int PAIR = Unit<MODE, CL>::PAIR;
  using G = typename Unit<MODE, CL>::G;
  // the item's B boxes: tensor map and column (only the k coordinate moves
  // in the loop; the single issuing thread's per-slice work stays short)
  const CUtensorMap* bmap[G::B_BOXES];
  int bcol[G::B_BOXES];
#pragma unroll
  for (int j = 0; j < G::B_BOXES; ++j) {
    const int nc = b_box_col<PAIR>(n0, cta, j);
    int n = nc < w.n_end ? nc : n0;  // the padding box of a CTA without columns
    // (a padding box may start up to a tile past N: the load reads fill values)
    if (!check_ok(c, n >= 0 && n < p.N + Unit<MODE, CL>::G::TILE_N && (n & 7) == 0 && w.r >= 0 && w.r < p.R,
                  CK_B_COL, static_cast<uint32_t>(n)))
      n = 0;
    int br = w.r;
    if (MODE == MODE_MOE_STAGED && p.xcols > 0) {
      // the box's rank in the expert group, and its column in that rank's block
      const int t = n / p.xcols;
      br += t;
      n -= t * p.xcols;
      if (!check_ok(c, br < p.R, CK_B_COL, static_cast<uint32_t>(br))) br = w.r;
    }
    bmap[j] = &p.tmB[br];
    bcol[j] = n;
  }
  // store mode: shard and shard row of the item's first A box (the next boxes
  // step from there; a box never spans two shards)
  int a_sh0 = 0, a_lrow0 = 0;
  if (MODE == MODE_STORE) {
    a_sh0 = w.m0 / p.rows_per_rank;
    a_lrow0 = w.m0 - a_sh0 * p.rows_per_rank;
  }
  for (int k = kb; k < ke; ++k) {
    // The empty barrier is completed by a remote commit whenever another CTA's
    // MMAs read the stage; the producer still waits in try_wait rather than
    // polling with test_wait: the polling thread's issue slots cost more than
    // a late wake-up (full step 7.80-7.87 against 7.95-8.01 ms, AG-GEMM and
    // MoE layer1 6-7 % faster)
    if (wait_bar(smem_u32(&s.empty[stage]), phase ^ 1u, c, W_EMPTY, stage) != 0) return false;
    const uint32_t fb = smem_u32(&s.full[stage]);
    if (PAIR == 1 || cta == 0) mbar_arrive_expect_tx(fb, bytes);
    // barrier in the even CTA of this CTA's pair
    const uint32_t fbc = PAIR == 2 ? mapa_shared(fb, static_cast<uint32_t>(hw_rank & ~1)) : fb;
    const uint32_t sa = smem_u32(s.a + stage * A_STAGE);
    const uint32_t sb = smem_u32(s.b + stage * G::B_STAGE);
    const int kc = k * BK;
    if (MODE == MODE_STORE) {
      int bsh = a_sh0, blrow = a_lrow0;
      for (int bx = 0; bx < nbox_a; ++bx) {
        if (bx > 0) {
          blrow += p.a_box_m;
          if (blrow >= p.rows_per_rank) {
            blrow -= p.rows_per_rank;
            ++bsh;
          }
        }
        if (MCA && MC2 && bx != a_half) continue;  // the N neighbour multicasts this box
        const int row = w.m0 + bx * p.a_box_m;
        int sh = bsh, lrow = blrow;
        int kx = kc;
        if (!check_ok(c, row >= 0 && sh < p.R && sh * p.rows_per_rank + lrow == row, CK_A_ROW,
                      static_cast<uint32_t>(row)))
          sh = lrow = 0;
        if (!check_ok(c, kc >= 0 && kc < p.K && (kc & 7) == 0, CK_A_K, static_cast<uint32_t>(kc))) kx = 0;
        if (MCA && MC2)
          tma_load_2d_pair_mc(sa + bx * p.a_box_m * BK * 2, &p.tmA[sh], fbc, kx, lrow, mask_a);
        else if (PAIR == 2)
          tma_load_2d_pair(sa + bx * p.a_box_m * BK * 2, &p.tmA[sh], fbc, kx, lrow);
        else
          tma_load_2d(sa + bx * p.a_box_m * BK * 2, &p.tmA[sh], fb, kx, lrow);
      }
    } else if (nbox_a) {
      // (checked build: a box outside the tensor is recorded and moved to its origin)
      int ar = w.r, am0 = w.m0, ak = kc;
      if (!check_ok(c, ar >= 0 && ar < p.R && am0 >= 0 && am0 < p.M, CK_A_ROW, static_cast<uint32_t>(am0)))
        ar = am0 = 0;
      if (!check_ok(c, ak >= 0 && ak < p.K && (ak & 7) == 0, CK_A_K, static_cast<uint32_t>(ak))) ak = 0;
      if (MCA) {
        // two 64-row boxes (the map's box is 64 rows); with a 8-CTA cluster
        // each of the two N neighbours issues one of them to both
        for (int bx = 0; bx < 2; ++bx) {
          if (MC2 && bx != a_half) continue;
          if (MC2)
            tma_load_2d_pair_mc(sa + bx * 64 * BK * 2, &p.tmA[ar], fbc, ak, am0 + bx * 64, mask_a);
          else
            tma_load_2d_pair(sa + bx * 64 * BK * 2, &p.tmA[ar], fbc, ak, am0 + bx * 64);
        }
      } else if (PAIR == 2) {
        tma_load_2d_pair(sa, &p.tmA[ar], fbc, ak, am0);
      } else {
        tma_load_2d(sa, &p.tmA[ar], fb, ak, am0);
      }
    }
#pragma unroll
    for (int j = 0; j < G::B_BOXES; ++j) {
      if (!((bmask >> j) & 1u)) continue;
      // the pair stacked with this one multicasts the other half of the boxes
      if (MC2 && (j * 2) / G::B_BOXES != half) continue;
      check_ok(c, kc >= 0 && kc < p.K, CK_B_K, static_cast<uint32_t>(kc));
      const uint32_t dst = sb + j * B_BOX_N * BK * 2;
      if (is_scatter(MODE) || MODE == MODE_MOE_STAGED) {
        if (PAIR == 2) tma_load_3d_pair(dst, bmap[j], fbc, bcol[j], kc, w.e);
        else tma_load_3d(dst, bmap[j], fb, bcol[j], kc, w.e);
      } else if (PAIR == 2) {
        if (MC2) tma_load_2d_pair_mc(dst, bmap[j], fbc, bcol[j], kc, mc_mask);
        else tma_load_2d_pair(dst, bmap[j], fbc, bcol[j], kc);
      } else {
        tma_load_2d(dst, bmap[j], fb, bcol[j], kc);
      }
    }
    ++issued;
    if (++stage == G::STAGES) { stage = 0; phase ^= 1u; }
  }
  return true;
}

// TMA producer (one thread).  Under the dynamic schedule the producer of a
// region's first CTA also claims the region's units.
template <int MODE, int CL>
__device__ void producer_tma(const KParams& p, const Smem& s, const Ctl& c, int total_mt,
                             const Pos& ps) {
  constexpr int PAIR = Unit<MODE, CL>::PAIR;
  constexpr int MC = Unit<MODE, CL>::MC;
  using G = typename Unit<MODE, CL>::G;
  const int cta = ps.vrank & (PAIR - 1);  // position in the pair
  const bool mc2 = MC == 2 && ps.mc2;     // B shared with the other pair by multicast
  const int half = (ps.hw_rank / PAIR) % 2;  // mc2: the B half this CTA multicasts
  // mc2: this CTA and the one holding the same B columns in the other tile
  const uint16_t mc_mask = static_cast<uint16_t>((1u << ps.hw_rank) | (1u << (ps.hw_rank ^ PAIR)));
  ItemIter<MODE, CL> iter(p, total_mt, ps.vrank, &c);
  const bool leader = iter.dyn && ps.vrank == 0;
  const bool slow_region = !ps.mc2;  // a region of pair clusters (no multicast)
  int claimed = 0;  // mailbox entries the leader has written
  if (leader) {
    if (!slow_region) atomicAdd(p.hdr + H_FAST, 1u);  // before its first claim
    claim_unit<MODE, CL>(p, iter.box, claimed++, slow_region, iter.claims());
  }
  Work w;
  uint32_t stage = 0, phase = 0;
  uint32_t issued = 0;
  uint32_t ready = (p.flags == nullptr) ? 0xFFFFFFFFu : 0u;
  int staged_mt = -1;  // MOE_STAGED: the last m-unit whose rows were seen staged
  bool ok = true;
  int item = 0;  // trace record index
  while (ok && iter.next(w)) {
    int nbox_a = w.m0 < w.row_end ? 1 : 0;  // a CTA part wholly past the last row loads no A
    if (MODE == MODE_MOE_STAGED && nbox_a && w.mt != staged_mt) {
      // every 32-row block of the unit must be staged (acquire), then be
      // visible to the TMA reads of this thread
      const int rows_u = min(BM * CL, w.row_end - (w.m0 - cta * BM));
      const uint32_t target = static_cast<uint32_t>((rows_u + STAGE_BLK - 1) / STAGE_BLK);
      if (!wait_count(p.unit_cnt + w.mt, target, c, W_STAGE)) break;
      fence_proxy_async_global();
      staged_mt = w.mt;
    }
    if (MODE == MODE_STORE) {
      nbox_a = 0;
      if (w.m0 < w.row_end) {
        if (p.push) {
          // push form: this part's 128-row block of the gathered copy must be
          // complete (acquire), then visible to this thread's TMA reads
          if (!wait_count(p.unit_cnt + w.m0 / BM, 1u, c, W_STAGE)) break;
          fence_proxy_async_global();
        } else {
          // shards covering the valid rows of this CTA's part must be published first
          const int last_row = min(w.m0 + BM, w.row_end) - 1;
          const int s0 = w.m0 / p.rows_per_rank, s1 = last_row / p.rows_per_rank;
          for (int sh = s0; sh <= s1 && ok; ++sh) {
            if (!((ready >> sh) & 1u)) {
              if (!wait_flag(p.flags, sh, p.epoch, c)) ok = false;
              else ready |= 1u << sh;
            }
          }
          if (!ok) break;
          if (p.flags != nullptr) fence_proxy_async_global();
        }
        nbox_a = (min(w.m0 + BM, w.row_end) - w.m0 + p.a_box_m - 1) / p.a_box_m;
      }
    }
    const int n0 = w.n0;
    const uint32_t bmask = b_box_mask<PAIR, G::B_BOXES>(w.n_end, n0, cta);
    uint32_t bytes = ((MODE == MODE_STORE) ? nbox_a * p.a_box_m * BK * 2 : nbox_a * A_STAGE) +
                     __popc(bmask) * B_BOX_N * BK * 2;
    if (PAIR == 2 && cta == 0) {
      // the even CTA's barrier also counts the odd CTA's bytes of the same stage
      bytes += pair_peer_bytes<MODE, G>(p, w);
    }
    trace_tag(p, item, w);
    trace_now(p, item, TR_PROD_START);
    // k-slices up to the claim point, the leader's claim of the region's
    // next unit, then the rest (no per-slice branch on either)
    // (one claim per item the mailbox hands out: under the tile-major GEMM-RS
    // schedule the next tile is claimed during the last rank's item)
    const bool claims_here = leader && w.rsub + 1 >= w.rcnt;
    const int claim_k = claims_here ? max(w.k0, w.k1 - CLAIM_AHEAD) : w.k1;
    for (int seg = 0; seg < 2 && ok; ++seg) {
      const int kb = seg == 0 ? w.k0 : claim_k, ke = seg == 0 ? claim_k : w.k1;
      if (seg == 1 && claims_here) claim_unit<MODE, CL>(p, iter.box, claimed++, slow_region, iter.claims());
      if (kb >= ke) continue;
      if constexpr (MC == 2) {
        ok = mc2 ? produce_ksteps<MODE, CL, true>(p, s, c, w, kb, ke, nbox_a, bmask, bytes, n0, cta, half,
                                                  mc_mask, ps.hw_rank, stage, phase, issued)
                 : produce_ksteps<MODE, CL, false>(p, s, c, w, kb, ke, nbox_a, bmask, bytes, n0, cta,
                                                   half, mc_mask, ps.hw_rank, stage, phase, issued);
      } else {
        ok = produce_ksteps<MODE, CL, false>(p, s, c, w, kb, ke, nbox_a, bmask, bytes, n0, cta, half,
                                             mc_mask, ps.hw_rank, stage, phase, issued);
      }
    }
    trace_now(p, item, TR_PROD_END);
    ++item;
  }
  // drain: every issued copy must land before the CTA may exit.  The odd CTA of
  // a pair cannot see its copies complete (they count on the even CTA's
  // barrier); it waits until the MMAs that read its last fill of each stage
  // completed, which implies the fill landed (bounded, like every wait).
  for (uint32_t st = 0; st < G::STAGES; ++st) {
    const uint32_t fills = issued / G::STAGES + (st < issued % G::STAGES ? 1u : 0u);
    if (fills == 0) continue;
    if (PAIR == 2 && cta != 0) {
      // (with mc2 the empty barrier also waits for the other pair, whose
      // multicast copies land here too)
      wait_bar_remote_drain(smem_u32(&s.empty[st]), (fills - 1u) & 1u, c, W_DRAIN, st);
    } else {
      wait_bar(smem_u32(&s.full[st]), (fills - 1u) & 1u, c, W_DRAIN, st, false);
    }
  }
}

// cp.async row-gather producer for MoE layer0 (all producer threads).  Eight
// consecutive threads copy one 128-byte row of a k-slice (16 bytes each), so a
// warp instruction moves four whole rows; thread t serves rows 16i + t/8
// (i = 0..7) of the A tile, each from the token row of the rank that owns it,
// into the 128B-swizzled layout the MMA descriptor expects.  Thread 0 also
// issues the B tile by TMA.
template <int NPROD>
__device__ void producer_gather(const KParams& p, const Smem& s, const Ctl& c, int total_mt) {
  using G = typename Unit<MODE_MOE_GATHER, 1>::G;
  ItemIter<MODE_MOE_GATHER, 1> iter(p, total_mt, 0);
  const int tid = threadIdx.x;  // producer warps are warps 0 .. NPROD/32-1
  Work w;
  uint32_t stage = 0, phase = 0, issued = 0;
  int pending = 0;  // stages whose cp.async group is committed but not yet published
  uint32_t ready = (p.flags == nullptr) ? 0xFFFFFFFFu : 0u;
  bool ok = true;
  const char* any_src = static_cast<const char*>(p.xsrc[0]);
  static_assert(NPROD == BM, "one producer thread per 16-byte chunk of 16 rows");
  constexpr int ROWS_PER_PASS = NPROD / 8;
  constexpr int PASSES = BM / ROWS_PER_PASS;
  const int sub = tid >> 3;   // row within a pass
  const int chunk = tid & 7;  // 16-byte chunk of the 128-byte row
  while (ok && iter.next(w)) {
    // my rows of this tile (nullptr: past the expert's last row)
    const char* src[PASSES];
#pragma unroll
    for (int i = 0; i < PASSES; ++i) {
      const int row = w.m0 + i * ROWS_PER_PASS + sub;
      src[i] = nullptr;
      if (row < w.row_end) {
        const int slot = __ldg(p.row_to_slot + row);
        const int tok = slot / p.topk;
        const int sh = tok / p.rows_per_rank;
        if (!((ready >> sh) & 1u)) {
          if (!wait_flag(p.flags, sh, p.epoch, c)) ok = false;
          else ready |= 1u << sh;
        }
        src[i] = static_cast<const char*>(p.xsrc[sh]) +
                 static_cast<size_t>(tok - sh * p.rows_per_rank) * p.H * 2 + chunk * 16;
      }
    }
    if (!ok) break;
    const int nbox_b = min(G::B_BOXES, (p.N - w.nt * BN + B_BOX_N - 1) / B_BOX_N);
    const uint32_t bytes_b = nbox_b * B_BOX_N * BK * 2;
    for (int k = w.k0; k < w.k1; ++k) {
      const int wr = wait_bar(smem_u32(&s.empty[stage]), phase ^ 1u, c, W_EMPTY, stage);
      if (wr != 0) { ok = false; break; }
      const uint32_t fb = smem_u32(&s.full[stage]);
      const uint32_t sa = smem_u32(s.a + stage * A_STAGE);
      const uint32_t sb = smem_u32(s.b + stage * G::B_STAGE);
      const int kc = k * BK;
      if (tid == 0) {
        mbar_arrive_expect_tx(fb, bytes_b);
        for (int j = 0; j < nbox_b; ++j)
          tma_load_3d(sb + j * B_BOX_N * BK * 2, &p.tmB[w.r], fb, w.nt * BN + j * B_BOX_N, kc, w.e);
      }
      {
        const bool col_ok = kc + chunk * 8 < p.H;
#pragma unroll
        for (int i = 0; i < PASSES; ++i) {
          const int r = i * ROWS_PER_PASS + sub;
          const uint32_t dst = sa + r * 128 + ((chunk ^ (r & 7)) << 4);
          if (src[i] != nullptr && col_ok) cp_async_16(dst, src[i] + static_cast<size_t>(kc) * 2);
          else cp_async_zero_16(dst, any_src);
        }
      }
      cp_async_commit();
      ++issued;
      ++pending;
      if (pending > GATHER_LAG) {
        cp_async_wait<GATHER_LAG>();
        fence_proxy_async_smem();
        const uint32_t old_stage = (stage + G::STAGES - GATHER_LAG) % G::STAGES;
        mbar_arrive(smem_u32(&s.full[old_stage]));
        --pending;
      }
      if (++stage == G::STAGES) { stage = 0; phase ^= 1u; }
    }
  }
  // publish what is still pending (also on abort, so the copies are complete)
  cp_async_wait<0>();
  fence_proxy_async_smem();
  for (; pending > 0; --pending) {
    const uint32_t old_stage = (stage + G::STAGES - pending) % G::STAGES;
    mbar_arrive(smem_u32(&s.full[old_stage]));
  }
  if (tid == 0) {
    for (uint32_t st = 0; st < G::STAGES; ++st) {
      const uint32_t fills = issued / G::STAGES + (st < issued % G::STAGES ? 1u : 0u);
      if (fills > 0) wait_bar(smem_u32(&s.full[st]), (fills - 1u) & 1u, c, W_DRAIN, st, false);
    }
  }
}

// MMA issuer (one thread; with pairs only in the even CTA of each pair).
template <int MODE, int DT, int CL>
__device__ void mma_issuer(const KParams& p, const Smem& s, const Ctl& c, uint32_t tmem_base,
                           int total_mt, const Pos& ps) {
  constexpr int PAIR = Unit<MODE, CL>::PAIR;
  using G = typename Unit<MODE, CL>::G;
  constexpr uint32_t IDESC = idesc_f16(DT, BM * PAIR, BN, 0, 1);
  // stage release reaches every CTA of the cluster (with a multicast B every
  // CTA's shared memory is filled by both pairs); the accumulator-full signal
  // only this pair
  const uint16_t EMPTY_MASK = static_cast<uint16_t>((1u << ps.hw_cl) - 1u);
  const uint16_t pair_mask = static_cast<uint16_t>(0x3u << (ps.hw_rank & ~1));
  // One 512-column accumulator (acc_halves): the epilogue hands back its first
  // 256 columns before the rest, and the next tile's first k-slices (as many
  // as the ring holds) issue their half-0 MMAs before the whole accumulator is
  // free; their half-1 MMAs follow once it is.  Each half still accumulates
  // its k-slices in order, so the results are those of the plain order.
  constexpr bool SPLIT = G::ACC_BUFS == 1 && G::N_MMA == 2;
  // GEMM-RS with rank groups (rs_group > 1): the group's ranks accumulate into
  // one accumulator back to back; only the last one hands it to the epilogue
  const bool grouped = ItemIter<MODE, CL>::GROUPS && p.rs_group > 1;
  ItemIter<MODE, CL> iter(p, total_mt, ps.vrank, &c);
  Work w;
  uint32_t stage = 0, phase = 0;
  int it = 0;    // accumulator hand-overs so far
  int item = 0;  // trace record index
  bool any = false;
  bool ok = true;
  while (ok && iter.next(w)) {
    const uint32_t b = it % G::ACC_BUFS;
    const uint32_t use = static_cast<uint32_t>(it / G::ACC_BUFS);
    const uint32_t d = tmem_base + b * G::ACC_COLS;
    const bool cont = grouped && w.rsub > 0;               // adds onto the group's sum
    const bool last = !grouped || w.rsub + 1 >= w.rcnt;   // hands the sum over
    // 256-column halves of the tile that start below N (a half wholly past N
    // has nothing to compute; its accumulator columns are never stored)
    const int n_live = (G::N_MMA > 1 && w.n0 + BN >= w.n_end) ? 1 : G::N_MMA;
    int pre = 0;  // leading k-slices whose half-0 MMAs were issued early
    if (SPLIT && !cont && p.acc_halves && use > 0 && n_live == 2) {
      if ((PAIR == 2 ? wait_bar_remote(smem_u32(&s.thalf[b]), (use & 1u) ^ 1u, c, W_TEMPTY, b + 2)
                     : wait_bar(smem_u32(&s.thalf[b]), (use & 1u) ^ 1u, c, W_TEMPTY, b + 2)) != 0)
        break;
      trace_now(p, item, TR_MMA_ACC);
      tc_fence_after();
      pre = min(G::STAGES, w.k1 - w.k0);
      uint32_t st = stage, ph = phase;
      for (int j = 0; j < pre; ++j) {
        if (wait_bar(smem_u32(&s.full[st]), ph, c, W_FULL, st) != 0) { ok = false; break; }
        if (j == 0) trace_now(p, item, TR_MMA_FIRST);
        tc_fence_after();
        const uint32_t sa = smem_u32(s.a + st * A_STAGE);
        const uint32_t sb = smem_u32(s.b + st * G::B_STAGE);
#pragma unroll
        for (int kk = 0; kk < BK / UK; ++kk) {
          const uint64_t ad = sdesc_sw128(sa + kk * UK * 2, 16, 1024);
          const uint64_t bd = sdesc_sw128(sb + kk * UK * 128, BK * 128, 1024);
          const uint32_t acc = (j > 0 || kk > 0) ? 1u : 0u;
          if (PAIR == 2) umma2_f16(d, ad, bd, IDESC, acc);
          else umma_f16(d, ad, bd, IDESC, acc);
        }
        if (++st == G::STAGES) { st = 0; ph ^= 1u; }
      }
      if (!ok) break;
    }
    if (!cont && (PAIR == 2 ? wait_bar_remote(smem_u32(&s.tempty[b]), (use & 1u) ^ 1u, c, W_TEMPTY, b)
                            : wait_bar(smem_u32(&s.tempty[b]), (use & 1u) ^ 1u, c, W_TEMPTY, b)) != 0)
      break;
    if (pre == 0) trace_now(p, item, TR_MMA_ACC);
    tc_fence_after();
    for (int k = w.k0; k < w.k1; ++k) {
      const bool early = k - w.k0 < pre;  // its stage is known full, its half 0 issued
      if (!early) {
        if (wait_bar(smem_u32(&s.full[stage]), phase, c, W_FULL, stage) != 0) { ok = false; break; }
        if (k == w.k0) trace_now(p, item, TR_MMA_FIRST);
        tc_fence_after();
      }
      const uint32_t sa = smem_u32(s.a + stage * A_STAGE);
      const uint32_t sb = smem_u32(s.b + stage * G::B_STAGE);
#pragma unroll
      for (int kk = 0; kk < BK / UK; ++kk) {
        // A: K-major rows of 128 B, 8-row groups 1024 B apart; a 16-wide k step is +32 B.
        const uint64_t ad = sdesc_sw128(sa + kk * UK * 2, 16, 1024);
        const uint32_t acc = (cont || k > w.k0 || kk > 0) ? 1u : 0u;
#pragma unroll
        for (int h = 0; h < G::N_MMA; ++h) {
          if (h >= n_live) break;
          if (SPLIT && h == 0 && early) continue;
          // B: N-major; 64-column (128 B) panels BK*128 B apart, 8-k-row groups
          // 1024 B apart; a 16-deep k step is 16 rows = +2048 B.  MMA h of a
          // pair reads panels 2h, 2h+1 and writes TMEM columns 256h ..
          const uint64_t bd =
              sdesc_sw128(sb + h * (BN / PAIR) * BK * 2 + kk * UK * 128, BK * 128, 1024);
          if (PAIR == 2) umma2_f16(d + h * BN, ad, bd, IDESC, acc);
          else umma_f16(d + h * BN, ad, bd, IDESC, acc);
        }
      }
      if (PAIR == 2) umma2_commit_mc(smem_u32(&s.empty[stage]), EMPTY_MASK);
      else umma_commit(smem_u32(&s.empty[stage]));
      any = true;
      if (++stage == G::STAGES) { stage = 0; phase ^= 1u; }
    }
    if (!ok) break;
    trace_now(p, item, TR_MMA_END);
    ++item;
    if (!last) continue;
    if (PAIR == 2) umma2_commit_mc(smem_u32(&s.tfull[b]), pair_mask);
    else umma_commit(smem_u32(&s.tfull[b]));
    ++it;
  }
  if (any) {
    if (PAIR == 2) umma2_commit(smem_u32(s.drain));
    else umma_commit(smem_u32(s.drain));
    wait_bar(smem_u32(s.drain), 0, c, W_DRAIN, 0, false);
  }
}

// epilogue helpers -----------------------------------------------------------
// Store one 64-column chunk of a warp's 32 rows as 16-bit values: every
// thread stages its row (128 bytes) in the warp's staging rows, then the rows
// are read back so that eight lanes cover one row and each warp instruction
// writes four whole 128-byte rows.  Rows >= rows_valid and columns >=
// ncols_valid (a multiple of 8) are not written.
template <int DT>
__device__ __forceinline__ void store_rows_chunk64(void* out, int ldo, long long row0, int rows_valid,
                                                   int col0, int ncols_valid, uint32_t sstg, int lane,
                                                   const uint32_t (&v)[32], const uint32_t (&u)[32]) {
  const uint32_t srow = sstg + lane * STG_PITCH;
  __syncwarp();  // the previous chunk's read-back is done
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    const uint32_t(&x)[32] = g < 4 ? v : u;
    const int b = (g & 3) * 8;
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                 ::"r"(srow + g * 16),
                   "r"(pack2<DT>(__uint_as_float(x[b + 0]), __uint_as_float(x[b + 1]))),
                   "r"(pack2<DT>(__uint_as_float(x[b + 2]), __uint_as_float(x[b + 3]))),
                   "r"(pack2<DT>(__uint_as_float(x[b + 4]), __uint_as_float(x[b + 5]))),
                   "r"(pack2<DT>(__uint_as_float(x[b + 6]), __uint_as_float(x[b + 7])))
                 : "memory");
  }
  __syncwarp();
  const int cc = (lane & 7) * 8;  // 16-bit column inside the chunk
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int rr = i * 4 + (lane >> 3);
    uint32_t a, b, c, d;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(a), "=r"(b), "=r"(c), "=r"(d) : "r"(sstg + rr * STG_PITCH + (lane & 7) * 16)
                 : "memory");
    if (rr < rows_valid && cc < ncols_valid) {
      uint16_t* dst = static_cast<uint16_t*>(out) + (row0 + rr) * ldo + col0 + cc;
      *reinterpret_cast<uint4*>(dst) = make_uint4(a, b, c, d);
    }
  }
}

// Gate-weighted scatter-add of one 32-column chunk of a warp's 32 rows: every
// thread stages its row (times its gate) in the warp's staging rows, then the
// rows are read back so that eight lanes cover one 128-byte row and each
// warp instruction adds four whole rows into their tokens' fp32 rows with
// red.global.add.v4.f32 (the load/store path, clear of the TMA queue that
// feeds the main loop).  Rows with row_ok == false add nothing.
__device__ __forceinline__ float as_f32(uint32_t x) { return __uint_as_float(x); }
__device__ __forceinline__ float as_f32(float x) { return x; }

template <class T>
__device__ __forceinline__ void scatter_add_chunk(float* acc, int ld_acc, int col0, int ncols_valid,
                                                  uint32_t sstg, int lane, int tok, bool row_ok,
                                                  float gate, const T (&v)[32]) {
  const uint32_t srow = sstg + lane * STG_PITCH;
  __syncwarp();  // the previous chunk's read-back is done
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    const float a = as_f32(v[g * 4 + 0]) * gate, b = as_f32(v[g * 4 + 1]) * gate;
    const float c = as_f32(v[g * 4 + 2]) * gate, d = as_f32(v[g * 4 + 3]) * gate;
    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(srow + g * 16), "f"(a), "f"(b),
                 "f"(c), "f"(d) : "memory");
  }
  __syncwarp();
  const int cc = (lane & 7) * 4;  // float column inside the chunk
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int rr = i * 4 + (lane >> 3);  // row of the warp's 32
    const int t = __shfl_sync(0xFFFFFFFFu, tok, rr);
    const int ok = __shfl_sync(0xFFFFFFFFu, row_ok ? 1 : 0, rr);
    float x0, x1, x2, x3;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(x0), "=f"(x1), "=f"(x2), "=f"(x3) : "r"(sstg + rr * STG_PITCH + cc * 4)
                 : "memory");
    if (ok && cc < ncols_valid) {
      float* dst = acc + static_cast<long long>(t) * ld_acc + col0 + cc;
      asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "f"(x0), "f"(x1),
                   "f"(x2), "f"(x3) : "memory");
    }
  }
}

// Convert 8 consecutive fp32 accumulators (L2) to 16 bits, store them, and
// zero the accumulators for the next call.
template <int DT>
__device__ __forceinline__ void convert8(float* src, uint16_t* dst) {
  const float4 a = ld_cg_f4(src);
  const float4 b = ld_cg_f4(src + 4);
  uint4 q;
  q.x = pack2<DT>(a.x, a.y);
  q.y = pack2<DT>(a.z, a.w);
  q.z = pack2<DT>(b.x, b.y);
  q.w = pack2<DT>(b.z, b.w);
  *reinterpret_cast<uint4*>(dst) = q;
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  st_cg_f4(src, z);
  st_cg_f4(src + 4, z);
}

// MoE layer1 with rank groups: convert the token tiles of the warp's slots in
// `todo` (bit i: slot of lane i, token tok of that lane) whose last add has
// landed: the fp32 row's columns [n0, n0 + ncols) of the tile go to the
// owner's 16-bit output row and are zeroed.  Two tiles at a time, 16 lanes
// each, 32 columns per lane (four 8-column chunks).
template <int DT>
__device__ __forceinline__ void convert_token_tiles(const KParams& p, const Ctl& c, uint32_t todo, int tok,
                                                    int n0, int ncols, int lane) {
  const int half = lane >> 4, hl = lane & 15;
  const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
  while (todo != 0u) {
    const int r0 = __ffs(todo) - 1;
    todo &= todo - 1u;
    int r1 = -1;
    if (todo != 0u) {
      r1 = __ffs(todo) - 1;
      todo &= todo - 1u;
    }
    const int mine = half == 0 ? r0 : r1;
    const int t = __shfl_sync(0xFFFFFFFFu, tok, mine < 0 ? 0 : mine);
    if (mine < 0) continue;  // (the second half of the warp has no tile this round)
    const int o = t / p.rows_per_rank;
    const int lt = t - o * p.rows_per_rank;
    if (!check_ok(c, o >= 0 && o < p.R, CK_OWNER, static_cast<uint32_t>(o))) continue;
    float* src = p.acc + static_cast<long long>(t) * p.N + n0;
    uint16_t* dst = static_cast<uint16_t*>(p.out[o]) + static_cast<long long>(lt) * p.ldo + n0;
    float4 a[4], b[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int col = (j * 16 + hl) * 8;  // 8-column chunk of this lane
      if (col < ncols) {
        a[j] = ld_cg_f4(src + col);
        b[j] = ld_cg_f4(src + col + 4);
      }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int col = (j * 16 + hl) * 8;
      if (col < ncols) {
        uint4 q;
        q.x = pack2<DT>(a[j].x, a[j].y);
        q.y = pack2<DT>(a[j].z, a[j].w);
        q.z = pack2<DT>(b[j].x, b[j].y);
        q.w = pack2<DT>(b[j].z, b[j].w);
        *reinterpret_cast<uint4*>(dst + col) = q;
        st_cg_f4(src + col, zero);
        st_cg_f4(src + col + 4, zero);
      }
    }
  }
}

template <int MODE, int DT, int CL>
__device__ void epilogue(const KParams& p, const Smem& s, const Ctl& c, uint32_t tmem_base,
                         int total_mt, int warp, const Pos& ps) {
  constexpr int PAIR = Unit<MODE, CL>::PAIR;
  const int cta = ps.vrank & (PAIR - 1);
  const int lane = threadIdx.x & 31;
  const int q = warp & 3;  // TMEM lane quarter this warp may access
  ItemIter<MODE, CL> iter(p, total_mt, ps.vrank, &c, true);
  Work w;
  int it = 0;
  // the accumulator-empty barrier lives in the even CTA of a pair
  const uint32_t tempty0 = (PAIR == 2 && cta != 0)
                               ? mapa_shared(smem_u32(&s.tempty[0]), static_cast<uint32_t>(ps.hw_rank & ~1))
                               : smem_u32(&s.tempty[0]);
  const uint32_t sstg = smem_u32(s.stg + q * STG_WARP);
  using G = typename Unit<MODE, CL>::G;
  constexpr bool SPLIT = G::ACC_BUFS == 1 && G::N_MMA == 2;
  const uint32_t thalf0 = (PAIR == 2 && cta != 0)
                              ? mapa_shared(smem_u32(&s.thalf[0]), static_cast<uint32_t>(ps.hw_rank & ~1))
                              : smem_u32(&s.thalf[0]);
  // the first epilogue warp records the trace stamps
  const bool tracer = warp == KernelShape<MODE, DT, CL>::EPI_WARP0 && lane == 0;
  int nst = 0;  // tensor bulk stores this warp has committed
  // GEMM-RS with rank groups: only a group's last item hands over the
  // accumulator, holding the sum of the group's partials
  const bool grouped = ItemIter<MODE, CL>::GROUPS && p.rs_group > 1;
  // every slot routed (the routing's last offset is T*topk): the token tiles
  // are converted as their last add lands, else by the end-of-call pass
  const bool count_rows = MODE == MODE_MOE_SCATTER_WIDE && p.row_cnt != nullptr &&
                          __ldg(p.offsets + p.E) == p.T * p.topk;
  int item = -1;  // trace record index
  while (iter.next(w)) {
    ++item;
    if (grouped && w.rsub + 1 < w.rcnt) continue;
    const uint32_t b = it % G::ACC_BUFS;
    const uint32_t use = static_cast<uint32_t>(it / G::ACC_BUFS);
    // one 512-column accumulator: once this warp's loads of its first 256
    // columns have completed, say so (every item, whether or not the MMA
    // side uses it, so that the barrier's phases follow the items)
    bool half_out = !SPLIT;
    auto free_half = [&]() {
      if (half_out) return;
      half_out = true;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (PAIR == 2 && cta != 0) mbar_arrive_remote(thalf0 + b * 8);
        else mbar_arrive(smem_u32(&s.thalf[b]));
      }
    };
    // one lane waits so that the whole warp takes the same exit decision
    // before the warp-collective tcgen05.ld below
    int wr = 0;
    if (lane == 0)
      wr = (PAIR == 2 && cta != 0) ? wait_bar_remote(smem_u32(&s.tfull[b]), use & 1u, c, W_TFULL, b)
                                   : wait_bar(smem_u32(&s.tfull[b]), use & 1u, c, W_TFULL, b);
    wr = __shfl_sync(0xFFFFFFFFu, wr, 0);
    if (wr != 0) break;
    if (tracer) trace_now(p, item, TR_EPI_FULL);
    tc_fence_after();
    const int row0 = w.m0 + q * 32;       // first of this warp's 32 rows
    const int row = row0 + lane;           // row of the A row space held by this thread
    const bool row_ok = row < w.row_end;
    const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + b * G::ACC_COLS;
    const int n0 = w.n0;
    const int ncols = w.n_end - n0;
    // per-row routing data
    float gate = 1.0f;
    int tok = 0;
    if (is_scatter(MODE) && row_ok) {
      const int slot = __ldg(p.row_to_slot + row);
      tok = slot / p.topk;
      gate = __ldg(p.topk_w + slot);
    }
    // GEMM-RS whose group holds all R ranks: the sum is the tile's result and
    // goes to the owner's 16-bit rows like an AllGather tile (no fp32 rows,
    // no arrival count); the owner's rows hold whole 128-row CTA parts
    const bool direct = MODE == MODE_REDUCE && p.rs_direct && grouped && w.rcnt == p.R;
    const int orank = MODE == MODE_REDUCE ? w.m0 / max(p.rows_per_rank, 1) : w.r;  // output tensor
    const int orow0 = MODE == MODE_REDUCE ? row0 - orank * p.rows_per_rank : row0;  // its row
    if (MODE == MODE_STORE || MODE == MODE_MOE_GATHER || MODE == MODE_MOE_STAGED || direct) {
      // 64 columns at a time: two TMEM loads, one row-contiguous store pass
      for (int ch = 0; ch < G::TILE_N / 64; ++ch) {
        if (ch * 64 == BN) free_half();
        if (ch * 64 >= ncols) break;  // warp-uniform
        uint32_t v[32], u[32];
        tmem_ld_32x32b_x32(taddr + ch * 64, v);
        tmem_ld_32x32b_x32(taddr + ch * 64 + 32, u);
        if (row0 >= w.row_end) continue;  // none of this warp's rows is in the tile
        // the box's output tensor and column (xcols: the rank whose block holds it)
        int crank = orank, ccol = n0 + ch * 64;
        if (MODE == MODE_MOE_STAGED && p.xcols > 0) {
          const int t = ccol / p.xcols;
          crank += t;
          ccol -= t * p.xcols;
        }
        // (checked build: a box outside the rank's output is recorded and not written)
        if (!check_ok(c, crank >= 0 && crank < p.R && row0 >= 0 && row0 < p.M, CK_OUT_ROW,
                      static_cast<uint32_t>(row0)) ||
            !check_ok(c, ccol >= 0 && ccol < p.ldo && (ccol & 7) == 0, CK_OUT_COL, static_cast<uint32_t>(ccol)))
          continue;
        if (row0 + 32 <= w.row_end || w.row_end == p.M) {
          // the warp's 32 x 64 box, staged in the 128-byte swizzled layout of
          // the output map, goes out as one tensor bulk store (rows past the
          // tensor are clipped); two staging boxes per warp alternate
          const uint32_t buf = sstg + (nst & 1) * STG_BOX;
          if (nst >= 2) {
            if (lane == 0) bulk_wait_read<1>();
            __syncwarp();
          }
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            const uint32_t(&x)[32] = g < 4 ? v : u;
            const int b = (g & 3) * 8;
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                         ::"r"(buf + lane * 128 + ((g ^ (lane & 7)) << 4)),
                           "r"(pack2<DT>(__uint_as_float(x[b + 0]), __uint_as_float(x[b + 1]))),
                           "r"(pack2<DT>(__uint_as_float(x[b + 2]), __uint_as_float(x[b + 3]))),
                           "r"(pack2<DT>(__uint_as_float(x[b + 4]), __uint_as_float(x[b + 5]))),
                           "r"(pack2<DT>(__uint_as_float(x[b + 6]), __uint_as_float(x[b + 7])))
                         : "memory");
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&p.tmOut[crank], buf, ccol, orow0);
            bulk_commit();
          }
          ++nst;
        } else {
          // the warp's rows run past this tile's last row into rows of another
          // tile (MoE: the next expert's): plain row stores up to the last row,
          // through the staging rows once no bulk store still reads them
          if (nst > 0) {
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
          }
          store_rows_chunk64<DT>(p.out[crank], p.ldo, orow0, w.row_end - row0, ccol, ncols - ch * 64, sstg,
                                 lane, v, u);
        }
      }
      if (direct && nst > 0) {
        // the fp32 path of the next item stages from its first box on: this
        // item's stores must have read their staging boxes (their writes
        // complete before the warp leaves, below)
        if (lane == 0) bulk_wait_read_all();
        __syncwarp();
      }
    } else {
      // fp32 adds: into this tile's own rows (REDUCE) or the rows' tokens,
      // gate-weighted (MOE_SCATTER)
      const int key = MODE == MODE_REDUCE ? row : tok;
      if (MODE == MODE_REDUCE && p.deterministic && row0 < w.row_end) {
        // ranks add in ascending order: wait until every lower rank's k-slices
        // of this quarter are in (its adds were fenced before it counted them)
        int ok_turn = 1;
        if (lane == 0)
          ok_turn = wait_count(p.counters + (static_cast<size_t>(w.tile) * 4 + q),
                               static_cast<uint32_t>(w.r) * static_cast<uint32_t>(p.KT), c,
                               W_TURN) ? 1 : 0;
        ok_turn = __shfl_sync(0xFFFFFFFFu, ok_turn, 0);
        __syncwarp();  // the lanes' adds are ordered after lane 0's acquire
        if (!ok_turn) break;  // TMEM stays held: the MMA side times out too
      }
      if constexpr (MODE == MODE_REDUCE) {
        // each 32 x 32 fp32 box of the warp goes out as one tensor bulk
        // reduce-add (the TMA engine reads the staged box and adds it in L2);
        // two staging boxes per warp alternate
        if (row0 < w.row_end) {
          for (int ch = 0; ch < G::TILE_N / 32; ++ch) {
            if (ch * 32 == BN) free_half();
            if (ch * 32 >= ncols) break;  // warp-uniform
            uint32_t v[32];
            tmem_ld_32x32b_x32(taddr + ch * 32, v);
            // (checked build: a box outside the fp32 rows is recorded and not added)
            if (!check_ok(c, row0 >= 0 && row0 < p.M, CK_ACC_ROW, static_cast<uint32_t>(row0)) ||
                !check_ok(c, n0 + ch * 32 >= 0 && n0 + ch * 32 < p.N && ((n0 + ch * 32) & 3) == 0, CK_ACC_COL,
                          static_cast<uint32_t>(n0 + ch * 32)))
              continue;
            const uint32_t buf = sstg + (ch & 1) * STG_BOX;
            if (ch >= 2) {
              if (lane == 0) bulk_wait_read<1>();
              __syncwarp();
            }
#pragma unroll
            for (int g = 0; g < 8; ++g)
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                           ::"r"(buf + lane * 128 + ((g ^ (lane & 7)) << 4)), "r"(v[g * 4 + 0]),
                             "r"(v[g * 4 + 1]), "r"(v[g * 4 + 2]), "r"(v[g * 4 + 3]) : "memory");
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_reduce_add_2d(&p.tmAcc, buf, n0 + ch * 32, row0);
              bulk_commit();
            }
          }
        }
      } else {
        // (checked build: a token outside [0, T) or a tile outside the row is
        // recorded and not added)
        const bool tok_ok = check_ok(c, !row_ok || (key >= 0 && key < p.T), CK_ACC_ROW, static_cast<uint32_t>(key));
        const bool col_ok = check_ok(c, n0 >= 0 && n0 < p.N, CK_ACC_COL, static_cast<uint32_t>(n0));
        for (int ch = 0; ch < G::TILE_N / 32; ++ch) {
          if (ch * 32 == BN) free_half();
          if (ch * 32 >= ncols || !col_ok) break;  // warp-uniform
          uint32_t v[32];
          tmem_ld_32x32b_x32(taddr + ch * 32, v);
          scatter_add_chunk(p.acc, p.N, n0 + ch * 32, ncols - ch * 32, sstg, lane, key, row_ok && tok_ok, gate, v);
        }
      }
    }
    // hand the accumulator back to the MMA warp
    free_half();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
      if (PAIR == 2 && cta != 0) mbar_arrive_remote(tempty0 + b * 8);
      else mbar_arrive(smem_u32(&s.tempty[b]));
    }
    ++it;
    if (tracer && (MODE != MODE_REDUCE || direct)) trace_now(p, item, TR_EPI_END);

    if (MODE == MODE_MOE_SCATTER_WIDE && grouped && count_rows && ncols > 0) {
      // this tile's adds of the warp's 32 slots are issued: make them visible,
      // then count each slot's token tile; the add that completes a token
      // tile converts it (after the accumulator went back, so the next
      // tile's MMAs do not wait for it)
      __syncwarp();
      __threadfence();
      __syncwarp();
      const int tile = n0 / G::TILE_N;
      bool done = false;
      if (row_ok && tok >= 0 && tok < p.T) {
        uint32_t* cnt = p.row_cnt + static_cast<size_t>(tok) * p.row_tiles + tile;
        done = atomicAdd(cnt, 1u) + 1u == static_cast<uint32_t>(p.row_arrivals);
        if (done) *cnt = 0u;  // no other add of this call reaches the tile
      }
      const uint32_t todo = __ballot_sync(0xFFFFFFFFu, done);
      if (todo != 0u) {
        __threadfence();  // the other adds to those tiles, before this warp reads them
        convert_token_tiles<DT>(p, c, todo, tok, n0, ncols, lane);
      }
    }

    if (MODE == MODE_REDUCE && !direct) {
      // arrival counter of this tile's 32-row quarter counts k-slices; quarters
      // wholly past the last row, and the parts of a region past the last
      // column (no tile of their own), have nothing to count
      if (row0 >= w.row_end || ncols <= 0) {
        if (tracer) trace_now(p, item, TR_EPI_END);
        continue;
      }
      // the box reduces of this quarter have completed
      if (lane == 0) bulk_wait_all();
      __syncwarp();
      __threadfence();
      __syncwarp();
      // (a rank group's sum counts the k-slices of all its ranks)
      const uint32_t nk = static_cast<uint32_t>(w.k1 - w.k0) * static_cast<uint32_t>(grouped ? w.rcnt : 1);
      const uint32_t target = static_cast<uint32_t>(p.R) * static_cast<uint32_t>(p.KT);
      uint32_t* cnt = p.counters + (static_cast<size_t>(w.tile) * 4 + q);
      uint32_t old = 0;
      if (lane == 0) old = atomicAdd(cnt, nk);
      old = __shfl_sync(0xFFFFFFFFu, old, 0);
      if (old + nk == target) {
        __threadfence();
        for (int i = 0; i < 32; ++i) {
          const int grow = w.m0 + q * 32 + i;
          if (grow >= w.row_end) break;
          const int o = grow / p.rows_per_rank;
          const int lr = grow - o * p.rows_per_rank;
          if (!check_ok(c, o >= 0 && o < p.R, CK_OWNER, static_cast<uint32_t>(o))) break;
#pragma unroll
          for (int c0 = 0; c0 < G::TILE_N; c0 += 256) {
            const int col = n0 + c0 + lane * 8;
            if (col < p.N && check_ok(c, col >= 0 && (col & 7) == 0, CK_OUT_COL, static_cast<uint32_t>(col)))
              convert8<DT>(p.acc + static_cast<long long>(grow) * p.N + col,
                           static_cast<uint16_t*>(p.out[o]) + static_cast<long long>(lr) * p.ldo + col);
          }
        }
        if (lane == 0) atomicExch(cnt, 0u);
      }
      if (tracer) trace_now(p, item, TR_EPI_END);
    }
  }
  if (nst > 0) {
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }
}

// RS_CLUSTER epilogue (the EPI_WARPS epilogue warps of every CTA).  The tile's
// rows are the M <= 128 activation rows; owner rank o holds rows
// [o M/R, (o+1) M/R), and CTA d of the cluster reduces the owners d, d + CL,
// ... (M / CL rows).  Each CTA holds one fp32 accumulator per rank it
// computed (ranks cta, cta + CL, ...).
//   1. once its accumulators are complete, its MMAs are done and its operand
//      ring is free: it tells every CTA of the cluster (xbar[0], CL arrivals);
//   2. when every ring is free, each thread (one row) adds its row of the
//      accumulators and writes it into slot `cta` of the ring of the CTA that
//      reduces the row's owner (st.shared::cluster), then arrives there
//      (xbar[1], M arrivals per CTA, release at cluster scope);
//   3. when its M rows are in, the CTA adds the CL slots in slot order,
//      converts to 16 bits and stores its owners' rows.
// Exchange layout in each ring: slot c (0 .. CL-1) of M / CL rows x 256 fp32.
template <int DT, int CL>
__device__ void epilogue_rs_cluster(const KParams& p, const Smem& s, const Ctl& c, uint32_t tmem_base,
                                    int warp, const Pos& ps) {
  using G = typename Unit<MODE_RS_CLUSTER, CL>::G;
  constexpr int ROWB = BN * 4;  // bytes of one fp32 row of the tile
  const int lane = threadIdx.x & 31;
  const int q = warp & 3;  // TMEM lane quarter: rows 32q .. 32q + 31
  const int cta = ps.vrank;
  const int nacc = (p.R - cta + CL - 1) / CL;  // accumulators of this CTA
  const int rows_o = p.M / p.R;                // rows per owner rank
  const int rows_d = p.M / CL;                 // rows each CTA reduces
  const uint32_t ring = smem_u32(s.a);
  const uint32_t xfree = smem_u32(&s.xbar[0]), xrows = smem_u32(&s.xbar[1]);
  const int n0 = static_cast<int>(blockIdx.x / CL) * BN;

  // 1. this CTA's partials are complete (each accumulator is used once)
  int ok = 1;
  if (lane == 0) {
    for (int b = 0; b < nacc && ok; ++b)
      if (wait_bar(smem_u32(&s.tfull[b]), 0u, c, W_TFULL, static_cast<uint32_t>(b)) != 0) ok = 0;
  }
  ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
  if (!ok) return;  // recorded; the peers' bounded waits see the abort
  tc_fence_after();
  if (q == 0 && lane == 0)
    for (int d = 0; d < CL; ++d) mbar_arrive_remote(mapa_shared(xfree, static_cast<uint32_t>(d)));

  // 2. every ring of the cluster is free: send each row to its reducer
  if (lane == 0) ok = wait_bar_remote(xfree, 0u, c, W_XCHG, 0u) == 0 ? 1 : 0;
  ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
  if (!ok) return;
  const int row = q * 32 + lane;
  const bool valid = row < p.M;
  uint32_t dst = 0;
  int dcta = 0;
  if (valid) {
    const int o = row / rows_o;
    dcta = o % CL;
    const int lr = (o / CL) * rows_o + (row - o * rows_o);
    dst = mapa_shared(ring + static_cast<uint32_t>((cta * rows_d + lr) * ROWB), static_cast<uint32_t>(dcta));
  }
  const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
  for (int ch = 0; ch < BN / 32; ++ch) {
    uint32_t v[32];
    tmem_ld_32x32b_x32(taddr + ch * 32, v);  // warp-collective: every lane, valid row or not
    if (nacc > 1) {
      uint32_t u[32];
      tmem_ld_32x32b_x32(taddr + G::ACC_COLS + ch * 32, u);
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) + __uint_as_float(u[i]));
    }
    if (valid) {
#pragma unroll
      for (int g = 0; g < 8; ++g)
        st_shared_cluster_f4(dst + ch * 128 + g * 16, __uint_as_float(v[4 * g]), __uint_as_float(v[4 * g + 1]),
                             __uint_as_float(v[4 * g + 2]), __uint_as_float(v[4 * g + 3]));
    }
  }
  if (valid) mbar_arrive_remote(mapa_shared(xrows, static_cast<uint32_t>(dcta)));

  // 3. this CTA's rows from every CTA of the cluster: add, convert, store
  if (lane == 0) ok = wait_bar_remote(xrows, 0u, c, W_XCHG, 1u) == 0 ? 1 : 0;
  ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
  if (!ok) return;
  fence_acq_rel_cluster();
  const int tid = q * 32 + lane;  // 0 .. 127
  // items: (row lr, 8-column group g); a warp covers one row's 32 groups
  for (int item = tid; item < rows_d * (BN / 8); item += EPI_WARPS * 32) {
    const int lr = item / (BN / 8), g = item % (BN / 8);
    const int col = n0 + g * 8;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int sc = 0; sc < CL; ++sc) {
      const uint32_t a = ring + static_cast<uint32_t>((sc * rows_d + lr) * ROWB + g * 32);
      float x[8];
      asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                   : "=f"(x[0]), "=f"(x[1]), "=f"(x[2]), "=f"(x[3]) : "r"(a) : "memory");
      asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                   : "=f"(x[4]), "=f"(x[5]), "=f"(x[6]), "=f"(x[7]) : "r"(a + 16) : "memory");
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] += x[i];
    }
    const int o = cta + (lr / rows_o) * CL;
    const int orow = lr - (lr / rows_o) * rows_o;
    if (col < p.N && check_ok(c, o >= 0 && o < p.R && orow < rows_o, CK_OWNER, static_cast<uint32_t>(o))) {
      uint4 qv;
      qv.x = pack2<DT>(acc[0], acc[1]);
      qv.y = pack2<DT>(acc[2], acc[3]);
      qv.z = pack2<DT>(acc[4], acc[5]);
      qv.w = pack2<DT>(acc[6], acc[7]);
      *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out[o]) + static_cast<long long>(orow) * p.ldo + col) = qv;
    }
  }
}

// MoE layer1, after every role of this CTA is done: the CTAs of the launch
// meet at a grid-wide barrier (the launch is sized so that all of them are
// resident at once; the wait is bounded), which makes every gate-weighted add
// of the call visible; then each CTA converts a share of the fp32 token rows
// to 16 bits into the owner ranks' outputs and zeroes them for the next call.
// The last CTA out resets the barrier's counters.  `flag` is a shared word.
template <int DT>
__device__ void finish_token_rows(const KParams& p, const Ctl& c, uint32_t* flag) {
  __threadfence();  // this thread's adds, before the CTA's arrival
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(p.hdr + H_GRID, 1u);
    *flag = wait_count(p.hdr + H_GRID, gridDim.x, c, W_GRID) ? 1u : 0u;
  }
  __syncthreads();
  if (*flag != 0u) {
    // 8 columns per chunk; a thread takes FIN_BATCH chunks a grid-stride
    // apart per round and issues all their loads before any store
    constexpr int FIN_BATCH = 4;
    const int chunks = p.H / 8;
    const long long total = static_cast<long long>(p.T) * chunks;
    const long long step = static_cast<long long>(gridDim.x) * blockDim.x;
    const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
    for (long long i0 = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i0 < total;
         i0 += step * FIN_BATCH) {
      float4 a[FIN_BATCH], b[FIN_BATCH];
#pragma unroll
      for (int j = 0; j < FIN_BATCH; ++j) {
        const long long i = i0 + j * step;
        if (i < total) {
          const int t = static_cast<int>(i / chunks);
          const float* src = p.acc + static_cast<long long>(t) * p.N + (i - static_cast<long long>(t) * chunks) * 8;
          a[j] = ld_cg_f4(src);
          b[j] = ld_cg_f4(src + 4);
        }
      }
#pragma unroll
      for (int j = 0; j < FIN_BATCH; ++j) {
        const long long i = i0 + j * step;
        if (i < total) {
          const int t = static_cast<int>(i / chunks);
          const int col = static_cast<int>(i - static_cast<long long>(t) * chunks) * 8;
          const int o = t / p.rows_per_rank;
          const int lt = t - o * p.rows_per_rank;
          if (!check_ok(c, o >= 0 && o < p.R, CK_OWNER, static_cast<uint32_t>(o))) continue;
          uint4 q;
          q.x = pack2<DT>(a[j].x, a[j].y);
          q.y = pack2<DT>(a[j].z, a[j].w);
          q.z = pack2<DT>(b[j].x, b[j].y);
          q.w = pack2<DT>(b[j].z, b[j].w);
          *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out[o]) + static_cast<long long>(lt) * p.ldo + col) = q;
          float* src = p.acc + static_cast<long long>(t) * p.N + col;
          st_cg_f4(src, zero);
          st_cg_f4(src + 4, zero);
        }
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(p.hdr + H_GRID_EXIT, 1u) + 1u == gridDim.x) {
      // every CTA has passed the barrier and converted its rows
      p.hdr[H_GRID] = 0u;
      p.hdr[H_GRID_EXIT] = 0u;
    }
  }
}

// AllGather + GEMM, push form: the first stage_ctas CTAs (all by default)
// push the rows of every shard into the gathered copy of X, one 128-row block
// at a time (blocks dealt to those CTAs in turn, ascending, so that the
// first units' rows come first); a warp copies a row with 16-byte loads, 16
// in flight per lane, after the ready flag of the shard that owns it.  When
// the whole CTA is done with a block it counts the block (release); the GEMM
// producers of the same launch wait for that count.  Block b of the copy
// holds rows [128 b, 128 b + 128) of the concatenated shards.
static __device__ void push_rows(const KParams& p, const Ctl& c) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = static_cast<int>(blockDim.x >> 5);
  const int chunks = p.K / 8;  // 16-byte chunks per row
  uint32_t ready = (p.flags == nullptr) ? 0xFFFFFFFFu : 0u;
  const int nblk = (p.push_rows_total + BM - 1) / BM;
  const int copiers = p.stage_ctas > 0 ? min(p.stage_ctas, static_cast<int>(gridDim.x))
                                       : static_cast<int>(gridDim.x);
  if (static_cast<int>(blockIdx.x) >= copiers) return;
  for (int blk = blockIdx.x; blk < nblk; blk += copiers) {
    const int row0 = blk * BM;
    const int nrows = min(BM, p.push_rows_total - row0);
    int ok = 1;
    for (int rr = warp; rr < nrows && ok; rr += nwarps) {
      const int row = row0 + rr;
      const int sh = row / p.push_shard_rows;
      if (!((ready >> sh) & 1u)) {
        if (lane == 0) ok = wait_flag(p.flags, sh, p.epoch, c) ? 1 : 0;
        ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
        if (!ok) break;
        ready |= 1u << sh;
      }
      const uint4* src = reinterpret_cast<const uint4*>(
          static_cast<const char*>(p.xsrc[sh]) + static_cast<size_t>(row - sh * p.push_shard_rows) * p.K * 2);
      uint4* dst = reinterpret_cast<uint4*>(static_cast<char*>(p.stage) + static_cast<size_t>(row) * p.K * 2);
      for (int c0 = 0; c0 < chunks; c0 += 32 * STAGE_UNROLL) {
        uint4 v[STAGE_UNROLL];
#pragma unroll
        for (int j = 0; j < STAGE_UNROLL; ++j) {
          const int ch = c0 + j * 32 + lane;
          if (ch < chunks) v[j] = __ldg(src + ch);
        }
#pragma unroll
        for (int j = 0; j < STAGE_UNROLL; ++j) {
          const int ch = c0 + j * 32 + lane;
          if (ch < chunks) dst[ch] = v[j];
        }
      }
    }
    // the block's rows, written by every thread, become visible (also to the
    // readers' TMA) before its count
    __threadfence();
    fence_proxy_async_global();
    if (!__syncthreads_and(ok)) return;  // a shard flag timed out (recorded)
    if (threadIdx.x == 0) atomicAdd(p.unit_cnt + blk, 1u);
  }
}

// MoE layer0, staged: the epilogue warps of the first stage_ctas CTAs (all
// CTAs by default) copy the grouped rows while the producer and MMA warps
// start on the units whose rows are in (the epilogue warps have nothing else
// to do until the CTA's first accumulator is full).  Blocks of STAGE_BLK
// grouped rows, in ascending m-unit order, are dealt to those CTAs in turn
// (so the first units' rows are spread over all of them); a warp
// copies one row at a time (the token row of the shard that owns it, after
// that shard's ready flag) into the staging buffer, 16 loads of 16 bytes in
// flight per lane.  When the group's warps are done with a block (named
// barrier 1), its count goes to the unit's ready counter (release), which the
// GEMM producers wait for.  False when a shard's flag timed out (recorded).
__device__ __forceinline__ bool group_all(int v, int nthreads) {
  int r;
  asm volatile("{\n\t.reg .pred a, b;\n\tsetp.ne.s32 a, %1, 0;\n\t"
               "bar.red.and.pred b, 1, %2, a;\n\tselp.s32 %0, 1, 0, b;\n\t}"
               : "=r"(r) : "r"(v), "r"(nthreads) : "memory");
  return r != 0;
}

template <int CL>
__device__ bool stage_rows(const KParams& p, const Ctl& c, int total_mt, int warp, int nwarps) {
  constexpr int UROWS = BM * CL;
  constexpr int BLKS = UROWS / STAGE_BLK;
  const int lane = threadIdx.x & 31;
  const int chunks = p.H / 8;  // 16-byte chunks per row
  uint32_t ready = (p.flags == nullptr) ? 0xFFFFFFFFu : 0u;
  const int items = total_mt * BLKS;
  const int copiers = p.stage_ctas > 0 ? min(p.stage_ctas, static_cast<int>(gridDim.x))
                                       : static_cast<int>(gridDim.x);
  if (static_cast<int>(blockIdx.x) >= copiers) return true;
  for (int i = blockIdx.x; i < items; i += copiers) {
    const int gmt = i / BLKS, b = i - (i / BLKS) * BLKS;
    int lo = 0, hi = p.E;  // the unit's expert: largest e with tile_off[e] <= gmt
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(p.tile_off + mid) <= gmt) lo = mid; else hi = mid;
    }
    const int row_end = __ldg(p.offsets + lo + 1);
    const int row0 = __ldg(p.offsets + lo) + (gmt - __ldg(p.tile_off + lo)) * UROWS + b * STAGE_BLK;
    if (row0 >= row_end) continue;  // the same decision in every thread
    const int nrows = min(STAGE_BLK, row_end - row0);
    int ok = 1;
    for (int rr = warp; rr < nrows && ok; rr += nwarps) {
      const int row = row0 + rr;
      const int tok = __ldg(p.row_to_slot + row) / p.topk;
      const int sh = tok / p.rows_per_rank;
      if (!((ready >> sh) & 1u)) {
        if (lane == 0) ok = wait_flag(p.flags, sh, p.epoch, c) ? 1 : 0;
        ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
        if (!ok) break;
        ready |= 1u << sh;
      }
      const uint4* src = reinterpret_cast<const uint4*>(
          static_cast<const char*>(p.xsrc[sh]) +
          static_cast<size_t>(tok - sh * p.rows_per_rank) * p.H * 2);
      uint4* dst = reinterpret_cast<uint4*>(static_cast<char*>(p.stage) +
                                            static_cast<size_t>(row) * p.H * 2);
      for (int c0 = 0; c0 < chunks; c0 += 32 * STAGE_UNROLL) {
        uint4 v[STAGE_UNROLL];
#pragma unroll
        for (int j = 0; j < STAGE_UNROLL; ++j) {
          const int ch = c0 + j * 32 + lane;
          if (ch < chunks) v[j] = __ldg(src + ch);
        }
#pragma unroll
        for (int j = 0; j < STAGE_UNROLL; ++j) {
          const int ch = c0 + j * 32 + lane;
          if (ch < chunks) dst[ch] = v[j];
        }
      }
    }
    // the block's rows, written by every thread, become visible (also to the
    // readers' TMA) before its count
    __threadfence();
    fence_proxy_async_global();
    if (!group_all(ok, nwarps * 32)) return false;
    if (warp == 0 && lane == 0) atomicAdd(p.unit_cnt + gmt, 1u);
  }
  return true;
}

// ---------------------------------------------------------------- kernel

template <int MODE, int DT, int CL>
__global__ void __launch_bounds__(KernelShape<MODE, DT, CL>::THREADS, 1)
fused_gemm_kernel(const __grid_constant__ KParams p) {
  using KS = KernelShape<MODE, DT, CL>;
  constexpr int PAIR = Unit<MODE, CL>::PAIR;
  constexpr int MC = Unit<MODE, CL>::MC;
  using G = typename Unit<MODE, CL>::G;
  static_assert(CL == 1 || CL == 2 || CL == 4 || CL == 8, "cluster of 1, 2, 4 or 8 CTAs");
  static_assert(MC <= 2, "at most two tiles share a B box");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  Smem s;
  s.a = base;
  s.b = base + G::STAGES * A_STAGE;
  s.stg = base + G::STAGES * (A_STAGE + G::B_STAGE);
  uint64_t* bars = reinterpret_cast<uint64_t*>(s.stg + KS::EPI * STG_WARP);
  s.full = bars;
  s.empty = bars + G::STAGES;
  s.tfull = bars + 2 * G::STAGES;
  s.tempty = bars + 2 * G::STAGES + 2;
  s.drain = bars + 2 * G::STAGES + 4;
  s.tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * G::STAGES + 5);
  s.misc = s.tmem_slot + 1;
  s.xbar = bars + 2 * G::STAGES + 7;
  s.thalf = bars + 2 * G::STAGES + 9;

  const int warp = threadIdx.x >> 5;
  const bool dyn = ItemIter<MODE, CL>::DYN_OK && p.dyn != 0;
  Pos ps;
  ps.hw_rank = CL > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  ps.hw_cl = CL > 1 ? static_cast<int>(cluster_nctarank()) : 1;
  // dynamic schedule: the CTA's part of the unit is its place in the region of
  // CL CTAs, whichever cluster size the launch gave the region
  ps.vrank = dyn ? static_cast<int>(blockIdx.x % CL) : ps.hw_rank;
  ps.mc2 = ps.hw_cl == CL;
  const int cta = ps.vrank & (PAIR - 1);
  Ctl c;
  c.hdr = p.hdr;
  c.seq = p.seq;
  c.flag_timeout = p.timeout_ns;
  c.pipe_timeout = 2 * p.timeout_ns + 10000000ull;

  if (threadIdx.x == 0) {
    // the dynamic schedule expects clusters of CL or PAIR CTAs made of
    // consecutive, aligned CTA indices
    s.misc[0] = (dyn && ((ps.hw_cl != CL && ps.hw_cl != PAIR) ||
                         ps.hw_rank != static_cast<int>(blockIdx.x % ps.hw_cl))) ? 1u : 0u;
    s.misc[1] = 0u;
    for (int i = 0; i < G::STAGES; ++i) {
      mbar_init(smem_u32(&s.full[i]), KS::FULL_COUNT);
      // one commit per pair that reads the stage
      mbar_init(smem_u32(&s.empty[i]), (MC == 2 && ps.mc2) ? ps.hw_cl / PAIR : 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&s.tfull[i]), 1);
      mbar_init(smem_u32(&s.tempty[i]), KS::EPI * PAIR);
      mbar_init(smem_u32(&s.thalf[i]), KS::EPI * PAIR);
    }
    mbar_init(smem_u32(s.drain), 1);
    if (MODE == MODE_RS_CLUSTER) {
      mbar_init(smem_u32(&s.xbar[0]), CL);                          // rings free
      mbar_init(smem_u32(&s.xbar[1]), static_cast<uint32_t>(p.M));  // rows received
    }
    fence_mbar_init();
  }
  if (warp == KS::MMA_WARP) {
    if (PAIR == 2) {
      tmem_alloc2(smem_u32(s.tmem_slot), TMEM_COLS);
      tmem_relinquish2();
    } else {
      tmem_alloc(smem_u32(s.tmem_slot), TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (CL > 1) cluster_sync();  // peer barriers initialised and TMEM allocated in every CTA
  tc_fence_after();
  const uint32_t tmem_base = *s.tmem_slot;
  bool run = true;
  if (dyn) {
    // one decision for the whole cluster: any CTA of an unexpected shape stops them all
    for (int r = 0; r < ps.hw_cl; ++r)
      if (ld_shared_cluster_u32(mapa_shared(smem_u32(s.misc), static_cast<uint32_t>(r))) != 0u)
        run = false;
    if (!run && threadIdx.x == 0 && ps.hw_rank == 0)
      raise_error(c, ST_INVALID, W_SHAPE, blockIdx.x, static_cast<uint32_t>(ps.hw_cl));
  }

  if (p.debug_probe != 0 && blockIdx.x == 0 && threadIdx.x == 0)
    check_ok(c, false, CK_PROBE, static_cast<uint32_t>(p.debug_probe));  // checked build only
#if FLUX_TRACE
  if (p.trace != nullptr && blockIdx.x == 0 && threadIdx.x == 0 && p.trace_words >= TR_FIELDS) {
    p.trace[0] = gridDim.x;
    p.trace[1] = (p.trace_words - TR_FIELDS) / (TR_FIELDS * static_cast<long long>(gridDim.x));
  }
#endif
  int total_mt = 0;
  if (is_moe(MODE)) total_mt = __ldg(p.tile_off + p.E);
  if constexpr (MODE == MODE_STORE) {
    if (p.push && run) push_rows(p, c);
  }

  const int lane = threadIdx.x & 31;
  if (warp == 0 && lane < p.R) {
    // bring this call's tensor maps into the TMA descriptor cache
    tma_prefetch_desc(&p.tmB[lane]);
    if (!KS::CPASYNC_GATHER) tma_prefetch_desc(&p.tmA[lane]);
  }
  if (!run) {
    // (the cluster shape check failed: recorded above; no role runs)
  } else if (warp < KS::PRODUCER_WARPS) {
    if constexpr (KS::CPASYNC_GATHER) {
      producer_gather<KS::PRODUCER_WARPS * 32>(p, s, c, total_mt);
    } else if (lane == 0) {
      producer_tma<MODE, CL>(p, s, c, total_mt, ps);
    }
  } else if (warp == KS::MMA_WARP) {
    // the even CTA of a pair issues the MMAs for both
    if (lane == 0 && cta == 0) mma_issuer<MODE, DT, CL>(p, s, c, tmem_base, total_mt, ps);
    __syncwarp();
  } else if constexpr (MODE == MODE_RS_CLUSTER) {
    epilogue_rs_cluster<DT, CL>(p, s, c, tmem_base, warp, ps);
  } else {
    // (staged MoE layer0: the copy first; after a shard flag timed out the
    // epilogue still runs, its waits give up as the producer's do)
    if constexpr (MODE == MODE_MOE_STAGED)
      stage_rows<CL>(p, c, total_mt, warp - KS::EPI_WARP0, KS::EPI);
    epilogue<MODE, DT, CL>(p, s, c, tmem_base, total_mt, warp, ps);
  }

  tc_fence_before();
  __syncthreads();
  if (CL > 1) cluster_sync();  // no CTA frees TMEM or leaves while another still works
  if (warp == KS::MMA_WARP) {
    tc_fence_after();
    if (PAIR == 2) tmem_dealloc2(tmem_base, TMEM_COLS);
    else tmem_dealloc(tmem_base, TMEM_COLS);
  }
  if constexpr (is_scatter(MODE)) {
    // (with rank groups and every slot routed the epilogues converted the rows)
    const bool counted = MODE == MODE_MOE_SCATTER_WIDE && p.rs_group > 1 && p.row_cnt != nullptr &&
                         __ldg(p.offsets + p.E) == p.T * p.topk;
    if (!counted) finish_token_rows<DT>(p, c, s.misc + 1);
  }
  if (dyn) {
    // The last CTA to finish clears the schedule (counter, exit count and
    // mailboxes) so that the workspace is zero again for the next call.  Every
    // CTA's claims and mailbox reads come before its exit count.
    if (threadIdx.x == 0) {
      __threadfence();
      s.misc[1] = (atomicAdd(p.hdr + H_EXIT, 1u) + 1u == gridDim.x) ? 1u : 0u;
    }
    __syncthreads();
    if (s.misc[1] != 0u) {
      __threadfence();
      const int n = static_cast<int>(gridDim.x / CL) * p.mbox_cap;
      for (int i = threadIdx.x; i < n; i += blockDim.x) p.mbox[i] = 0u;
      if (MODE == MODE_STORE && p.push)
        for (int i = threadIdx.x; i < (p.push_rows_total + BM - 1) / BM; i += blockDim.x) p.unit_cnt[i] = 0u;
      if (threadIdx.x == 0) {
        p.hdr[H_CLAIM] = 0u;
        p.hdr[H_EXIT] = 0u;
        p.hdr[H_FAST] = 0u;
      }
    }
  }
}

}  // namespace flux
