// Dense entry points: plain GEMM, AllGather + GEMM, GEMM + ReduceScatter.
#include <mutex>

#include "flux_host.h"
#include "flux_kernels.cuh"
#include "flux_launch.cuh"

namespace flux {
namespace {

template <int MODE, int CL>
flux_status_t launch_dt(flux_dtype_t dt, const KParams& p, int grid, cudaStream_t s) {
  return dt == FLUX_BF16 ? Launcher<MODE, 1, CL>::launch(p, grid, s)
                         : Launcher<MODE, 0, CL>::launch(p, grid, s);
}

template <int MODE, int CL>
int grid_dt(flux_dtype_t dt, const DeviceInfo& dev, const flux_opts_t* opts, long long units) {
  return dt == FLUX_BF16 ? grid_for<MODE, 1, CL>(dev, opts, units)
                         : grid_for<MODE, 0, CL>(dev, opts, units);
}

template <int MODE, int CL>
int grid_dyn_dt(flux_dtype_t dt, const DeviceInfo& dev) {
  return dt == FLUX_BF16 ? Launcher<MODE, 1, CL>::max_ctas_dyn(dev)
                         : Launcher<MODE, 0, CL>::max_ctas_dyn(dev);
}

template <int MODE, int CL>
flux_status_t launch_dyn_dt(flux_dtype_t dt, const KParams& p, int grid, cudaStream_t s) {
  return dt == FLUX_BF16 ? Launcher<MODE, 1, CL>::launch_dyn(p, grid, s)
                         : Launcher<MODE, 0, CL>::launch_dyn(p, grid, s);
}

// Dense whole-tile kernels: on the static schedule, clusters of two CTA pairs
// stacked along M (512 x 512 per cluster, B multicast between the pairs); on
// the dynamic schedule, store mode runs regions of four pairs (512 x 1024: A
// multicast between the pairs side by side along N as well) where 8-CTA
// clusters fit and pairs elsewhere; reduce mode regions of two pairs.
constexpr int DENSE_CL = 4;
constexpr int DENSE_CL8 = 8;
// GEMM-RS form of the whole-unit dynamic schedule when opts->rs_tile is 0
// (1: regions of 4, 256 x 512 pair tiles; 2: regions of 8, 256 x 256 pair tiles)
constexpr int DEFAULT_RS_TILE = 1;
// GEMM-RS on regions of 4: ranks whose partials of one tile are summed in TMEM
// before the fp32 adds (see rs_group in the kernel parameters).  At 4096 x
// 49152 x 12288 over 8 ranks, against each rank's partial added on its own:
// 1, 2, 4, 8 ranks 3255-3263, 3056-3107, 3045-3062, 2971-3023 us alone; the
// whole step (power-limited) best with 4
constexpr int DEFAULT_RS_GROUP = 4;
// GEMM-RS of few rows: clusters of 4 CTAs reduce the R partials of a tile
// through distributed shared memory (each CTA computes R / 4 partials)
constexpr int RS_CLUSTER_CL = 4;
using DenseUnit = Unit<MODE_STORE, DENSE_CL>;
using DenseGeo = DenseUnit::G;

bool valid_dtype(flux_dtype_t dt) { return dt == FLUX_F16 || dt == FLUX_BF16; }

void fill_common(KParams& p, const flux_opts_t* opts, void* ws) {
  p.timeout_ns = (opts && opts->timeout_ns) ? opts->timeout_ns : DEFAULT_TIMEOUT_NS;
  p.epoch = (opts && opts->epoch) ? opts->epoch : 1u;
  p.group_n = (opts && opts->group_n > 0) ? opts->group_n : 8;
  p.seq = next_seq();
  p.hdr = static_cast<uint32_t*>(ws);
  p.trace = opts ? static_cast<unsigned long long*>(opts->trace) : nullptr;
  p.trace_words = (opts && opts->trace) ? static_cast<long long>(opts->trace_words) : 0;
  p.debug_probe = opts ? opts->debug_probe : 0;
  p.acc_halves = (opts && opts->acc_whole) ? 0 : 1;
}

flux_status_t zero_outputs(void* const* out, int n, size_t bytes, cudaStream_t s) {
  for (int i = 0; i < n; ++i) {
    cudaError_t e = cudaMemsetAsync(out[i], 0, bytes, s);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return FLUX_OK;
}

size_t rs_counter_bytes(int M, int N) {
  const size_t Mt = (M + BM - 1) / BM, Nt = (N + BN - 1) / BN;
  return round_up(Mt * Nt * 4 * sizeof(uint32_t), WS_ALIGN);
}

// GEMM-RS workspace without the dynamic schedule's mailboxes: header, arrival
// counters, fp32 owner rows (the least a call accepts; it then runs the static
// schedule).
size_t rs_min_bytes(int M, int N) {
  return WS_HEADER + rs_counter_bytes(M, N) + static_cast<size_t>(M) * N * sizeof(float);
}

flux_status_t gemm_rs_impl(int R, int M, int N, int K, flux_dtype_t dtype,
                           const void* const* a_shards, long long lda, const void* const* b_shards,
                           void* const* out, void* workspace, size_t workspace_bytes,
                           const flux_opts_t* opts, void* stream);

// K slices of the few-row plain GEMM (0 = not split): at most 128 rows, each
// slice at least 256 deep and a multiple of 8, the rows dividing into S chunks.
int gemm_k_split(int M, int N, int K) {
  if (M < 1 || M > BM || N < 1 || N % 8) return 0;
  for (int S : {8, 4})
    if (M % S == 0 && K % (8 * S) == 0 && K / S >= 256) return S;
  return 0;
}

// Whole 512 x 512 units of a dense op over R ranks with `cols` output columns each.
long long dense_units(int R, int M, int cols) {
  return static_cast<long long>(R) * ((M + DenseUnit::ROWS - 1) / DenseUnit::ROWS) *
         ((cols + DenseGeo::TILE_N - 1) / DenseGeo::TILE_N);
}

// Mailboxes of the dynamic schedule: C <= U + MAX_REGIONS claims (the last
// units of a store-mode op are claimed as two halves, at most one per region)
// over g <= MAX_REGIONS regions of 2 ceil(C / g) + 2 entries each: at most
// 2 U + 6 MAX_REGIONS entries.
size_t sched_bytes(long long units) {
  return round_up(static_cast<size_t>(2 * units + 6 * MAX_REGIONS) * sizeof(uint32_t), WS_ALIGN);
}

// Set up the dynamic schedule of a dense CL = 4 launch if the workspace has
// room for its mailboxes at `mbox` and the launch form is available; returns
// its grid, or 0 (then the static schedule runs).
template <int MODE, int CL>
int setup_dyn(KParams& p, flux_dtype_t dt, const DeviceInfo& dev, const flux_opts_t* opts,
              uint8_t* mbox, size_t room) {
  if (room < sched_bytes(p.num_units)) return 0;
  int grid = grid_dyn_dt<MODE, CL>(dt, dev);
  if (opts && opts->num_ctas > 0 && opts->num_ctas < grid) grid = opts->num_ctas - opts->num_ctas % CL;
  if (grid < CL) return 0;
  const long long regions = grid / CL;
  if (regions > p.num_units) {
    grid = static_cast<int>(p.num_units) * CL;
  }
  const long long g = grid / CL;
  // store mode, regions of 4: the last g units are claimed as two 256-column
  // halves, so that the last wave of units ends more evenly over the regions.
  // (Regions of 8 take no halves: there a half unit, every pair computing a
  // 256-column half of its tile, still takes 90 % of a whole unit's time --
  // the k-slices of the ring are latency-bound below that much work.)
  p.split_from = p.num_units;
  if (MODE == MODE_STORE && CL == 4)
    p.split_from = static_cast<int>(p.num_units > g ? p.num_units - g : 0);
  p.num_claims = p.num_units + (p.num_units - p.split_from);
  p.dyn = 1;
  // regions of pair clusters leave the last claims to the full-cluster ones
  {
    const int full = (dt == FLUX_BF16 ? Launcher<MODE, 1, CL>::max_ctas(dev)
                                      : Launcher<MODE, 0, CL>::max_ctas(dev)) / CL;
    p.claim_reserve = (opts && opts->num_ctas > 0) ? 0 : full;
  }
  p.mbox_cap = static_cast<int>(2 * ((p.num_claims + g - 1) / g) + 2);
  p.mbox = reinterpret_cast<uint32_t*>(mbox);
  return grid;
}

// Push form of AllGather + GEMM: per 128-row block a ready count, then the
// gathered copy of X [M x K] (16-bit), after the header and the mailboxes.
size_t push_counter_bytes(int M) { return round_up(static_cast<size_t>((M + BM - 1) / BM) * 4, WS_ALIGN); }

}  // namespace
}  // namespace flux

using namespace flux;

extern "C" size_t flux_workspace_size(flux_op_t op, int R, int M, int N, int K) {
  if (R < 1 || R > FLUX_MAX_RANKS || M < 0 || N < 0 || K < 0) return 0;
  switch (op) {
    case FLUX_OP_AG_GEMM_PUSH:
      return WS_HEADER + sched_bytes(dense_units(R, M, N / R)) + push_counter_bytes(M) +
             round_up(static_cast<size_t>(M) * K * 2, WS_ALIGN);
    case FLUX_OP_GEMM: {
      const size_t plain = WS_HEADER + sched_bytes(dense_units(R, M, N / R));
      // few rows: the split-K form needs the GEMM + ReduceScatter workspace
      const int S = R == 1 ? gemm_k_split(M, N, K) : 0;
      if (S == 0) return plain;
      const size_t split = rs_min_bytes(M, N) + sched_bytes(dense_units(S, M, N));
      return split > plain ? split : plain;
    }
    case FLUX_OP_AG_GEMM:
      return WS_HEADER + sched_bytes(dense_units(R, M, N / R));
    case FLUX_OP_GEMM_RS:
      return rs_min_bytes(M, N) + sched_bytes(dense_units(R, M, N));
    case FLUX_OP_MLP: {  // (R, M, H, F): its AG-GEMM (R, M, F, H), then its GEMM-RS (R, M, H, F)
      const size_t ag = flux_workspace_size(FLUX_OP_AG_GEMM, R, M, K, N);
      const size_t rs = flux_workspace_size(FLUX_OP_GEMM_RS, R, M, N, K);
      return ag > rs ? ag : rs;
    }
    default:
      return 0;
  }
}

extern "C" flux_status_t flux_launch_info(flux_op_t op, flux_dtype_t dtype, int* cluster_ctas,
                                          int* resident_ctas) {
  if (!valid_dtype(dtype) || cluster_ctas == nullptr || resident_ctas == nullptr)
    return FLUX_ERR_INVALID_ARG;
  DeviceInfo dev;
  flux_status_t st = current_device(&dev);
  if (st != FLUX_OK) return st;
  int cl = 0, cap = 0;
  switch (op) {
    case FLUX_OP_GEMM:
    case FLUX_OP_AG_GEMM:
      cl = DENSE_CL8;
      cap = grid_dyn_dt<MODE_STORE, DENSE_CL8>(dtype, dev);
      if (cap == 0) {
        cl = DENSE_CL;
        cap = grid_dt<MODE_STORE, DENSE_CL>(dtype, dev, nullptr, 1LL << 30);
      }
      break;
    case FLUX_OP_GEMM_RS:
    case FLUX_OP_MLP:
      cl = DENSE_CL;
      cap = grid_dyn_dt<MODE_REDUCE, DENSE_CL>(dtype, dev);
      if (cap == 0) cap = grid_dt<MODE_REDUCE, DENSE_CL>(dtype, dev, nullptr, 1LL << 30);
      break;
    default:
      return FLUX_ERR_INVALID_ARG;
  }
  if (cap == 0) return FLUX_ERR_CUDA;
  *cluster_ctas = cl;
  *resident_ctas = cap;
  return FLUX_OK;
}

bool flux::rs_uses_stream_k(int R, int M, int N, int sm, bool deterministic) {
  const long long units128 = static_cast<long long>((M + BM - 1) / BM) * ((N + BN - 1) / BN) * R;
  return units128 < 4LL * sm && !deterministic;
}

extern "C" flux_status_t flux_ag_gemm(int R, int M, int N, int K, flux_dtype_t dtype,
                                      const void* const* x_shards, const void* const* w_shards,
                                      void* const* out, const uint32_t* ready_flags,
                                      void* workspace, size_t workspace_bytes,
                                      const flux_opts_t* opts, void* stream) {
  if (R < 1 || R > FLUX_MAX_RANKS || M < 0 || N < 0 || K < 0 || !valid_dtype(dtype))
    return FLUX_ERR_INVALID_ARG;
  if (M % R || N % R) return FLUX_ERR_INVALID_ARG;
  if (x_shards == nullptr || w_shards == nullptr || out == nullptr) return FLUX_ERR_INVALID_ARG;
  flux_status_t st = check_workspace(workspace, workspace_bytes, WS_HEADER);
  if (st != FLUX_OK) return st;
  flux_opts_t tuned;
  if (opts == nullptr && tuned_opts(FLUX_OP_AG_GEMM, {R, M, N, K, 0, 0, 0, 0}, dtype, &tuned))
    opts = &tuned;
  const int rows = M / R, Nr = N / R;
  if (M == 0 || Nr == 0) return FLUX_OK;
  for (int r = 0; r < R; ++r) {
    if (x_shards[r] == nullptr || w_shards[r] == nullptr || out[r] == nullptr)
      return FLUX_ERR_INVALID_ARG;
    if (!aligned16(x_shards[r]) || !aligned16(w_shards[r]) || !aligned16(out[r]))
      return FLUX_ERR_UNSUPPORTED;
  }
  if (K % 8 || Nr % 8) return FLUX_ERR_UNSUPPORTED;
  int box_m = BM;
  if (R > 1) {
    box_m = 0;
    for (int b = BM; b >= 8; b >>= 1)
      if (rows % b == 0) { box_m = b; break; }
    if (box_m == 0) return FLUX_ERR_UNSUPPORTED;
  }
  DeviceInfo dev;
  if ((st = current_device(&dev)) != FLUX_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (K == 0) return zero_outputs(out, R, static_cast<size_t>(M) * Nr * 2, s);

  KParams p{};
  for (int r = 0; r < R; ++r) {
    if ((st = encode_2d(&p.tmA[r], dtype, x_shards[r], K, rows, static_cast<uint64_t>(K) * 2, BK,
                        box_m)) != FLUX_OK)
      return st;
    if ((st = encode_2d(&p.tmB[r], dtype, w_shards[r], Nr, K, static_cast<uint64_t>(Nr) * 2, B_BOX_N,
                        BK)) != FLUX_OK)
      return st;
    p.out[r] = out[r];
    if ((st = encode_2d(&p.tmOut[r], dtype, out[r], Nr, M, static_cast<uint64_t>(Nr) * 2, 64, 32)) != FLUX_OK)
      return st;
  }
  p.R = R;
  p.M = M;
  p.N = Nr;
  p.K = K;
  p.Mt = (M + DenseUnit::ROWS - 1) / DenseUnit::ROWS;
  p.Nt = (Nr + DenseGeo::TILE_N - 1) / DenseGeo::TILE_N;
  p.KT = (K + BK - 1) / BK;
  p.ldo = Nr;
  p.rows_per_rank = rows;
  p.a_box_m = box_m;
  p.num_units = R * p.Mt * p.Nt;
  p.flags = ready_flags;
  fill_common(p, opts, workspace);
  // bands of 4 n-tiles (2048 columns) measured best for the 512 x 512 units
  if (!(opts && opts->group_n > 0)) p.group_n = 4;
  if (opts && opts->ag_push) {
    // Push form: copy CTAs push every shard's rows into one gathered copy of X
    // in the workspace (a ready count per 128-row block); the tiles load A
    // from that copy, so the producers see a single shard of M rows.
    const size_t sched = sched_bytes(dense_units(R, M, Nr));
    const size_t need = flux_workspace_size(FLUX_OP_AG_GEMM_PUSH, R, M, N, K);
    if (workspace_bytes < need) return FLUX_ERR_WORKSPACE;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    p.unit_cnt = reinterpret_cast<uint32_t*>(ws + WS_HEADER + sched);
    p.stage = ws + WS_HEADER + sched + push_counter_bytes(M);
    p.push = 1;
    p.push_rows_total = M;
    p.push_shard_rows = rows;
    p.stage_ctas = opts->moe_stage_ctas > 0 ? opts->moe_stage_ctas : 0;
    p.rows_per_rank = M;
    for (int r = 0; r < R; ++r) p.xsrc[r] = x_shards[r];
    KParams q = p;
    if ((st = encode_2d(&q.tmA[0], dtype, p.stage, K, M, static_cast<uint64_t>(K) * 2, BK, 64)) != FLUX_OK)
      return st;
    q.a_box_m = 64;
    q.Nt = (Nr + Unit<MODE_STORE, DENSE_CL8>::UNIT_N - 1) / Unit<MODE_STORE, DENSE_CL8>::UNIT_N;
    q.num_units = R * q.Mt * q.Nt;
    if (!(opts && opts->group_n > 0)) q.group_n = 2;
    const int g8 = setup_dyn<MODE_STORE, DENSE_CL8>(q, dtype, dev, opts, ws + WS_HEADER, sched);
    if (g8 > 0 && launch_dyn_dt<MODE_STORE, DENSE_CL8>(dtype, q, g8, s) == FLUX_OK) return FLUX_OK;
    if ((st = encode_2d(&p.tmA[0], dtype, p.stage, K, M, static_cast<uint64_t>(K) * 2, BK, BM)) != FLUX_OK)
      return st;
    p.a_box_m = BM;
    const int dgrid = setup_dyn<MODE_STORE, DENSE_CL>(p, dtype, dev, opts, ws + WS_HEADER, sched);
    if (dgrid > 0 && launch_dyn_dt<MODE_STORE, DENSE_CL>(dtype, p, dgrid, s) == FLUX_OK) return FLUX_OK;
    return FLUX_ERR_UNSUPPORTED;  // the push form runs on the dynamic schedule only
  }
  // dynamic schedule over every SM when the workspace holds its mailboxes:
  // regions of 8 CTAs (512 x 1024 units, 64-row A boxes that must not
  // straddle two shards), else regions of 4
  if (R == 1 || rows % 64 == 0) {
    KParams q = p;
    for (int r = 0; r < R; ++r)
      if ((st = encode_2d(&q.tmA[r], dtype, x_shards[r], K, rows, static_cast<uint64_t>(K) * 2, BK,
                          64)) != FLUX_OK)
        return st;
    q.a_box_m = 64;
    q.Nt = (Nr + Unit<MODE_STORE, DENSE_CL8>::UNIT_N - 1) / Unit<MODE_STORE, DENSE_CL8>::UNIT_N;
    q.num_units = R * q.Mt * q.Nt;
    // bands of 2 n-units (2048 columns), as 4 for the 512-column units
    if (!(opts && opts->group_n > 0)) q.group_n = 2;
    const int g8 = setup_dyn<MODE_STORE, DENSE_CL8>(q, dtype, dev, opts,
                                                    static_cast<uint8_t*>(workspace) + WS_HEADER,
                                                    workspace_bytes - WS_HEADER);
    if (g8 > 0 && launch_dyn_dt<MODE_STORE, DENSE_CL8>(dtype, q, g8, s) == FLUX_OK) return FLUX_OK;
  }
  const int dgrid = setup_dyn<MODE_STORE, DENSE_CL>(p, dtype, dev, opts,
                                          static_cast<uint8_t*>(workspace) + WS_HEADER,
                                          workspace_bytes - WS_HEADER);
  if (dgrid > 0) {
    if (launch_dyn_dt<MODE_STORE, DENSE_CL>(dtype, p, dgrid, s) == FLUX_OK) return FLUX_OK;
    p.dyn = 0;  // launch form refused: the static schedule below
    p.mbox = nullptr;
    p.mbox_cap = 0;
  }
  const int grid = grid_dt<MODE_STORE, DENSE_CL>(dtype, dev, opts, p.num_units);
  if (grid == 0) return FLUX_ERR_CUDA;
  return launch_dt<MODE_STORE, DENSE_CL>(dtype, p, grid, s);
}

extern "C" flux_status_t flux_gemm(int M, int N, int K, flux_dtype_t dtype, const void* A,
                                   const void* B, void* C, void* workspace,
                                   size_t workspace_bytes, const flux_opts_t* opts, void* stream) {
  // Few rows: one 128-row tile leaves most SMs idle, so K is split into S
  // slices that play the ranks of a GEMM + ReduceScatter (slice s: columns
  // [s K/S, (s+1) K/S) of A, the same rows of B), whose partials are summed in
  // fp32 -- inside 4-CTA clusters through distributed shared memory where the
  // n-tiles fit, else by k-slice ranges over the grid -- and "owner" o writes
  // rows [o M/S, (o+1) M/S) of C.
  const int S = gemm_k_split(M, N, K);
  if (S > 1 && valid_dtype(dtype) && !(opts && opts->num_ctas > 0) && workspace != nullptr &&
      workspace_bytes >= rs_min_bytes(M, N) && A != nullptr && B != nullptr && C != nullptr &&
      aligned16(A) && aligned16(B) && aligned16(C)) {
    const int Ks = K / S;
    const void* a[FLUX_MAX_RANKS];
    const void* b[FLUX_MAX_RANKS];
    void* c[FLUX_MAX_RANKS];
    for (int s = 0; s < S; ++s) {
      a[s] = static_cast<const uint16_t*>(A) + static_cast<size_t>(s) * Ks;
      b[s] = static_cast<const uint16_t*>(B) + static_cast<size_t>(s) * Ks * N;
      c[s] = static_cast<uint16_t*>(C) + static_cast<size_t>(s) * (M / S) * N;
    }
    return gemm_rs_impl(S, M, N, K, dtype, a, K, b, c, workspace, workspace_bytes, opts, stream);
  }
  const void* a[1] = {A};
  const void* b[1] = {B};
  void* c[1] = {C};
  return flux_ag_gemm(1, M, N, K, dtype, a, b, c, nullptr, workspace, workspace_bytes, opts, stream);
}

namespace flux {
namespace {

// GEMM + ReduceScatter; `lda` is the row pitch of every A shard in elements
// (K / R for separate shard buffers; the full K when the shards are column
// slices of one matrix, as in the split-K plain GEMM).
flux_status_t gemm_rs_impl(int R, int M, int N, int K, flux_dtype_t dtype,
                           const void* const* a_shards, long long lda, const void* const* b_shards,
                           void* const* out, void* workspace, size_t workspace_bytes,
                           const flux_opts_t* opts, void* stream) {
  if (R < 1 || R > FLUX_MAX_RANKS || M < 0 || N < 0 || K < 0 || !valid_dtype(dtype))
    return FLUX_ERR_INVALID_ARG;
  if (M % R || K % R) return FLUX_ERR_INVALID_ARG;
  if (a_shards == nullptr || b_shards == nullptr || out == nullptr) return FLUX_ERR_INVALID_ARG;
  flux_status_t st = check_workspace(workspace, workspace_bytes, rs_min_bytes(M, N));
  if (st != FLUX_OK) return st;
  flux_opts_t tuned;
  if (opts == nullptr && tuned_opts(FLUX_OP_GEMM_RS, {R, M, N, K, 0, 0, 0, 0}, dtype, &tuned))
    opts = &tuned;
  if (M == 0 || N == 0) return FLUX_OK;
  const int Kr = K / R, rows = M / R;
  for (int r = 0; r < R; ++r) {
    if (a_shards[r] == nullptr || b_shards[r] == nullptr || out[r] == nullptr)
      return FLUX_ERR_INVALID_ARG;
    if (!aligned16(a_shards[r]) || !aligned16(b_shards[r]) || !aligned16(out[r]))
      return FLUX_ERR_UNSUPPORTED;
  }
  if (Kr % 8 || N % 8) return FLUX_ERR_UNSUPPORTED;
  DeviceInfo dev;
  if ((st = current_device(&dev)) != FLUX_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (Kr == 0) return zero_outputs(out, R, static_cast<size_t>(rows) * N * 2, s);

  KParams p{};
  for (int r = 0; r < R; ++r) {
    if ((st = encode_2d(&p.tmA[r], dtype, a_shards[r], Kr, M, static_cast<uint64_t>(lda) * 2, BK,
                        BM)) != FLUX_OK)
      return st;
    if ((st = encode_2d(&p.tmB[r], dtype, b_shards[r], N, Kr, static_cast<uint64_t>(N) * 2, B_BOX_N,
                        BK)) != FLUX_OK)
      return st;
    p.out[r] = out[r];
  }
  p.R = R;
  p.M = M;
  p.N = N;
  p.K = Kr;
  p.KT = (Kr + BK - 1) / BK;
  p.ldo = N;
  p.rows_per_rank = rows;
  p.a_box_m = BM;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.counters = reinterpret_cast<uint32_t*>(ws + WS_HEADER);
  p.acc = reinterpret_cast<float*>(ws + WS_HEADER + rs_counter_bytes(M, N));
  if ((st = encode_2d_f32(&p.tmAcc, p.acc, N, M, static_cast<uint64_t>(N) * 4, 32, 32)) != FLUX_OK)
    return st;
  fill_common(p, opts, workspace);

  // Few tiles per SM (decode shapes): single-CTA 128 x 256 tiles and an equal
  // contiguous range of k-slices per CTA (tiles split along K add into the same
  // fp32 owner tile).  Otherwise: whole 512 x 512 units on clusters of two CTA
  // pairs, strided over a persistent grid.
  const int sm = (opts && opts->num_ctas > 0) ? opts->num_ctas : dev.sm_count;
  // deterministic_rs: whole tiles (no k split), each rank's partial of a tile
  // on consecutive units (tile-major), added in ascending rank order
  p.deterministic = (opts && opts->deterministic_rs) ? 1 : 0;
  // At most 128 rows and 4 or 8 ranks, every 256-column tile on a resident
  // cluster of 4 CTAs (no grid given): the cluster computes the tile's R
  // partials and reduces them through distributed shared memory into the
  // owners' rows -- no fp32 workspace traffic, no atomics.
  if (!p.deterministic && !(opts && opts->num_ctas > 0) && M <= BM && (R == 4 || R == 8)) {
    const int nt = (N + BN - 1) / BN;
    const int cap = grid_dt<MODE_RS_CLUSTER, RS_CLUSTER_CL>(dtype, dev, nullptr, 1LL << 30);
    if (cap > 0 && nt * RS_CLUSTER_CL <= cap) {
      p.Mt = 1;
      p.Nt = nt;
      p.num_units = nt;
      p.stream_k = 0;
      return launch_dt<MODE_RS_CLUSTER, RS_CLUSTER_CL>(dtype, p, nt * RS_CLUSTER_CL, s);
    }
  }
  if (rs_uses_stream_k(R, M, N, sm, p.deterministic != 0)) {
    p.Nt = (N + BN - 1) / BN;
    p.Mt = (M + BM - 1) / BM;
    p.num_units = p.Mt * p.Nt * R;
    p.total_ksteps = static_cast<long long>(p.num_units) * p.KT;
    p.stream_k = 1;
    const int cap = grid_dt<MODE_REDUCE, 1>(dtype, dev, opts, p.total_ksteps);
    if (cap == 0) return FLUX_ERR_CUDA;
    long long per = p.total_ksteps / cap;
    int grid = per >= 4 ? cap : static_cast<int>((p.total_ksteps + 3) / 4);
    if (grid < 1) grid = 1;
    // Default grid: whole units per CTA when that still keeps three quarters
    // of the CTAs busy.  No unit is then split along K, so fewer partial tiles
    // end the call with fp32 adds (decode 128 x 8192 x 28672: 256 units on 128
    // CTAs, 112 -> 102 us).
    if (!(opts && opts->num_ctas > 0) && grid == cap) {
      for (int g = cap; g >= (3 * cap + 3) / 4; --g) {
        if (p.num_units % g == 0) {
          grid = g;
          break;
        }
      }
    }
    p.tiles_per_group = p.Mt * p.Nt;
    p.Nt_tile = p.Nt;
    return launch_dt<MODE_REDUCE, 1>(dtype, p, grid, s);
  }
  using RsUnit = Unit<MODE_REDUCE, DENSE_CL>;
  p.Nt = (N + RsUnit::G::TILE_N - 1) / RsUnit::G::TILE_N;
  p.Nt_tile = p.Nt;
  p.Mt = (M + RsUnit::ROWS - 1) / RsUnit::ROWS;
  const int tiles = p.Mt * p.Nt;
  p.num_units = tiles * R;
  p.total_ksteps = static_cast<long long>(p.num_units) * p.KT;
  p.stream_k = 0;
  auto tiles_per_group = [&](int grid, int cl, int ntiles) {
    const int tg = p.deterministic ? 1
                  : (opts && opts->tiles_per_group > 0) ? opts->tiles_per_group : grid / cl;
    return tg < ntiles ? tg : ntiles;
  };
  if (!p.deterministic) {
    // dynamic schedule over every SM when the workspace holds its mailboxes
    // (the deterministic order keeps the static schedule: its waits point at
    // lower units, which must already sit on resident clusters).
    const size_t off = rs_min_bytes(M, N);
    const size_t room = workspace_bytes > off ? workspace_bytes - off : 0;
    const int form = (opts && opts->rs_tile > 0) ? opts->rs_tile : DEFAULT_RS_TILE;
    if (form == 2) {
      // regions of 8 CTAs: four pairs of 256 x 256 tiles (two accumulators
      // each) on the same 512 x 512 units, A shared by multicast between the
      // pairs side by side along N (two 64-row boxes), B between the pairs
      // stacked along M
      using U8 = Unit<MODE_REDUCE, DENSE_CL8>;
      KParams q = p;
      for (int r = 0; r < R; ++r)
        if ((st = encode_2d(&q.tmA[r], dtype, a_shards[r], Kr, M, static_cast<uint64_t>(lda) * 2, BK,
                            64)) != FLUX_OK)
          return st;
      q.Nt = (N + U8::UNIT_N - 1) / U8::UNIT_N;
      q.Nt_tile = (N + U8::G::TILE_N - 1) / U8::G::TILE_N;
      q.Mt = (M + U8::ROWS - 1) / U8::ROWS;
      const int tiles8 = q.Mt * q.Nt;
      q.num_units = tiles8 * R;
      q.total_ksteps = static_cast<long long>(q.num_units) * q.KT;
      q.stream_k = 0;
      const int g8 = setup_dyn<MODE_REDUCE, DENSE_CL8>(q, dtype, dev, opts, ws + off, room);
      if (g8 > 0) {
        q.tiles_per_group = tiles_per_group(g8, DENSE_CL8, tiles8);
        if (launch_dyn_dt<MODE_REDUCE, DENSE_CL8>(dtype, q, g8, s) == FLUX_OK) return FLUX_OK;
      }
    }
    // regions of 4 CTAs: two pairs of 256 x 512 tiles stacked along M, B
    // shared by multicast
    const int dgrid = setup_dyn<MODE_REDUCE, DENSE_CL>(p, dtype, dev, opts, ws + off, room);
    if (dgrid > 0 && form == 3) {
      // tile-major: one claim per output tile, whose R partials the region
      // computes back to back (units u = tile * R + rank)
      p.rs_tile_major = 1;
      p.tiles_per_group = 1;
      p.num_claims = tiles;
      const int g = dgrid / DENSE_CL;
      p.mbox_cap = 2 * ((tiles + g - 1) / g) + 2;
      if (launch_dyn_dt<MODE_REDUCE, DENSE_CL>(dtype, p, dgrid, s) == FLUX_OK) return FLUX_OK;
      p.rs_tile_major = 0;
    }
    if (dgrid > 0) {
      p.tiles_per_group = tiles_per_group(dgrid, DENSE_CL, tiles);
      // rank groups: a region sums the partials of G ranks of one tile in
      // TMEM and drains the sum once (one fp32 add per G partials)
      const int G = (opts && opts->rs_group > 0) ? opts->rs_group : DEFAULT_RS_GROUP;
      if (G > 1 && R % G == 0) {
        // the last g group claims go out rank by rank: G times as many claims,
        // each a single rank's unit
        const int g = dgrid / DENSE_CL;
        const int groups = p.num_units / G;
        p.rs_group = G;
        p.split_from = groups > g ? groups - g : 0;
        p.num_claims = p.split_from + (groups - p.split_from) * G;
        p.mbox_cap = 2 * ((p.num_claims + g - 1) / g) + 2;
        // a group of all R ranks sums the whole tile: stored straight into the
        // owner's 16-bit rows when every 128-row CTA part lies in one owner
        if (G == R && rows % BM == 0) {
          bool ok = true;
          for (int o = 0; o < R && ok; ++o)
            ok = encode_2d(&p.tmOut[o], dtype, out[o], N, rows, static_cast<uint64_t>(N) * 2, 64, 32) ==
                 FLUX_OK;
          p.rs_direct = ok ? 1 : 0;
        }
      }
      if (launch_dyn_dt<MODE_REDUCE, DENSE_CL>(dtype, p, dgrid, s) == FLUX_OK) return FLUX_OK;
      p.rs_group = 1;
      p.rs_direct = 0;
      p.split_from = p.num_units;
      p.dyn = 0;  // launch form refused: the static schedule below
      p.mbox = nullptr;
      p.mbox_cap = 0;
    }
  }
  const int grid = grid_dt<MODE_REDUCE, DENSE_CL>(dtype, dev, opts, p.num_units);
  if (grid == 0) return FLUX_ERR_CUDA;
  p.tiles_per_group = tiles_per_group(grid, DENSE_CL, tiles);
  return launch_dt<MODE_REDUCE, DENSE_CL>(dtype, p, grid, s);
}

}  // namespace
}  // namespace flux

extern "C" flux_status_t flux_gemm_rs(int R, int M, int N, int K, flux_dtype_t dtype,
                                      const void* const* a_shards, const void* const* b_shards,
                                      void* const* out, void* workspace, size_t workspace_bytes,
                                      const flux_opts_t* opts, void* stream) {
  return gemm_rs_impl(R, M, N, K, dtype, a_shards, R >= 1 ? K / R : 0, b_shards, out, workspace,
                      workspace_bytes, opts, stream);
}

extern "C" flux_status_t flux_mlp_ag_rs(int R, int M, int H, int F, flux_dtype_t dtype,
                                        const void* const* x_shards, const void* const* w1_shards,
                                        void* const* h, const void* const* w2_shards,
                                        void* const* out, const uint32_t* ready_flags,
                                        void* workspace, size_t workspace_bytes,
                                        const flux_opts_t* opts, void* stream) {
  if (h == nullptr) return FLUX_ERR_INVALID_ARG;
  // validate both calls before launching either (the least each accepts: the
  // GEMM-RS part; the AG-GEMM needs only the header)
  if (R < 1 || R > FLUX_MAX_RANKS || M < 0 || H < 0 || F < 0 || M % R || F % R ||
      !valid_dtype(dtype))
    return FLUX_ERR_INVALID_ARG;
  flux_status_t st = check_workspace(workspace, workspace_bytes, rs_min_bytes(M, H));
  if (st != FLUX_OK) return st;
  if ((st = flux_ag_gemm(R, M, F, H, dtype, x_shards, w1_shards, h, ready_flags, workspace,
                         workspace_bytes, opts, stream)) != FLUX_OK)
    return st;
  return flux_gemm_rs(R, M, H, F, dtype, reinterpret_cast<const void* const*>(h), w2_shards, out,
                      workspace, workspace_bytes, opts, stream);
}
