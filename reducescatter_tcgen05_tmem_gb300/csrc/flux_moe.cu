// MoE entry points: the top-k gate, routing (histogram, prefix sum, stable
// permutation), AllGather + gather-by-expert + grouped GEMM (layer0), and
// grouped GEMM + gate-weighted combine + ReduceScatter by token (layer1), in
// the tensor-parallel layout and under an EP x TP split of the experts.
#include <math.h>

#include <algorithm>
#include <mutex>

#include "flux_host.h"
#include "flux_kernels.cuh"
#include "flux_launch.cuh"

namespace flux {

constexpr int ROUTE_THREADS = 1024;
// CTAs per cluster of the grouped GEMMs; the tile-offset table of each
// counts units of BM * CL rows inside an expert.
//   layer0: single CTAs, A rows gathered with cp.async (eight threads per
//     128-byte row).  Measured alternatives: two CTAs sharing B by multicast
//     (slower; multicast does not lower the bytes an SM receives) and CTA
//     pairs gathering rows with TMA tile::gather4 (2.7x slower: 32 gather
//     operations per stage cost the TMA unit far more than one 128-row box).
//   layer1: CTA pairs.  With several ranks per expert group (tensor
//     parallel), 256 x 512 tiles whose ranks' partials are summed in TMEM
//     before one add (MODE_MOE_SCATTER_WIDE with rank groups, the default);
//     with one rank per group (or on request, moe_l1_ranks 1): 256 x 256
//     tiles with two accumulators, so that the fp32 adds of one tile overlap
//     the main loop of the next, and from MOE1_WIDE_KT k-slices on 256 x 512
//     tiles with one accumulator.  Measured at T 4096, H 4096, F 14336, 8
//     experts, top-2: with 28 k-slices per tile and per rank the wide tile
//     alone is 13 % slower (0.76 -> 0.87 ms: the MMAs wait for each drain),
//     with 224 (expert parallel, one rank per expert) 14 % faster (0.78 ->
//     0.67 ms); the 8-rank groups make the tensor-parallel layer 224 k-slices
//     per drain too.
//   layer0 staged (the default): the epilogue warps copy the grouped rows
//     into the workspace while CTA pairs with 256 x 512 tiles load them by
//     TMA (see MODE_MOE_STAGED; 256 x 256 measured slower).
// layer1 rank groups: claim the last groups rank by rank (measured slower with
// 8-rank groups, 713-718 against 654 us: a quarter of the work then drains
// rank by rank)
constexpr int MOE1_SPLIT_TAIL = 0;
constexpr int MOE0_CL = 1;
constexpr int MOE0S_CL = 2;
constexpr int MOE1_CL = 2;
constexpr int MOE1_WIDE_KT = 48;  // layer1 k-slices from which the wide tile is taken
constexpr int ROUTE_CHUNK = 4096;  // expert ids staged in shared memory per pass
constexpr int ROUTE_WARPS = ROUTE_THREADS / 32;
constexpr int ROUTE_PAR_E = 64;    // up to this many experts all warps share the permutation

// Exclusive block-wide prefix sum of one int per thread (blockDim.x == 1024).
__device__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, w, o);
      if (lane >= o) w += y;
    }
    warp_sums[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const int before = (warp > 0 ? warp_sums[warp - 1] : 0) + x - v;
  if (total) *total = warp_sums[31];
  __syncthreads();
  return before;
}

// One CTA: counts[e], offsets[e] (exclusive prefix sum), the stable
// permutation slot_to_row / row_to_slot (rows grouped by expert, ascending slot
// order inside an expert) and, if tile_off != nullptr, the first unit of
// `unit_rows` rows of each expert in the grouped GEMM; with unit_cnt !=
// nullptr the ready counters of those units are zeroed for the staged layer0.
// Ids outside [0, E) are not routed; their slot_to_row entry is -1 and
// FLUX_ERR_INVALID_ARG is recorded in hdr.
__global__ void __launch_bounds__(ROUTE_THREADS, 1)
moe_route_kernel(const int32_t* __restrict__ ids, int n, int E, int32_t* counts,
                 int32_t* offsets, int32_t* slot_to_row, int32_t* row_to_slot, int32_t* tile_off,
                 int unit_rows, uint32_t* unit_cnt, uint32_t* hdr) {
  __shared__ int hist[FLUX_MAX_EXPERTS];
  __shared__ int base[FLUX_MAX_EXPERTS];
  __shared__ int warp_sums[32];
  __shared__ int totals[2];
  __shared__ int stage[ROUTE_CHUNK];
  __shared__ int warp_base[ROUTE_WARPS][ROUTE_PAR_E];
  const int tid = threadIdx.x;
  for (int e = tid; e < E; e += ROUTE_THREADS) hist[e] = 0;
  __syncthreads();
  int bad = 0;
  for (int s = tid; s < n; s += ROUTE_THREADS) {
    const int e = ids[s];
    if (e >= 0 && e < E) atomicAdd(&hist[e], 1);
    else bad = 1;
  }
  bad = __syncthreads_or(bad);
  // E <= 1024 = blockDim: one expert per thread
  const int cnt = tid < E ? hist[tid] : 0;
  const int off = block_exclusive_scan(cnt, warp_sums, &totals[0]);
  const int ntile = (cnt + unit_rows - 1) / unit_rows;
  const int toff = block_exclusive_scan(ntile, warp_sums, &totals[1]);
  if (tid < E) {
    counts[tid] = cnt;
    offsets[tid] = off;
    base[tid] = off;
    if (tile_off) tile_off[tid] = toff;
  }
  if (tid == 0) {
    offsets[E] = totals[0];
    if (tile_off) tile_off[E] = totals[1];
  }
  if (unit_cnt)
    for (int i = tid; i < totals[1]; i += ROUTE_THREADS) unit_cnt[i] = 0u;
  __syncthreads();
  // stable permutation: row(slot) = offsets[e] + number of earlier slots of
  // expert e.  Slots are taken 32 at a time; __match_any_sync ranks the lanes
  // of one expert inside a group.
  const int lane = tid & 31, warp = tid >> 5;
  for (int c0 = 0; c0 < n; c0 += ROUTE_CHUNK) {
    const int cn = min(ROUTE_CHUNK, n - c0);
    for (int i = tid; i < cn; i += ROUTE_THREADS) stage[i] = ids[c0 + i];
    __syncthreads();
    if (E <= ROUTE_PAR_E) {
      // every warp takes a contiguous run of the chunk: count per expert,
      // scan the counts over the warps (in slot order), then place
      const int per = ((cn + ROUTE_WARPS * 32 - 1) / (ROUTE_WARPS * 32)) * 32;
      const int lo = warp * per, hi = min(cn, lo + per);
      for (int e = lane; e < E; e += 32) warp_base[warp][e] = 0;
      __syncwarp();
      for (int i0 = lo; i0 < hi; i0 += 32) {
        const int i = i0 + lane;
        const int e = i < hi ? stage[i] : -1;
        const bool valid = i < hi && e >= 0 && e < E;
        const unsigned mask = __match_any_sync(0xFFFFFFFFu, valid ? e : -1 - lane);
        if (valid && lane == __ffs(mask) - 1) warp_base[warp][e] += __popc(mask);
        __syncwarp();
      }
      __syncthreads();
      if (tid < E) {
        int run = base[tid];
        for (int w = 0; w < ROUTE_WARPS; ++w) {
          const int c = warp_base[w][tid];
          warp_base[w][tid] = run;
          run += c;
        }
        base[tid] = run;
      }
      __syncthreads();
      for (int i0 = lo; i0 < hi; i0 += 32) {
        const int i = i0 + lane;
        const int e = i < hi ? stage[i] : -1;
        const bool valid = i < hi && e >= 0 && e < E;
        const unsigned mask = __match_any_sync(0xFFFFFFFFu, valid ? e : -1 - lane);
        const int rank = __popc(mask & ((1u << lane) - 1u));
        if (valid) {
          const int row = warp_base[warp][e] + rank;
          slot_to_row[c0 + i] = row;
          row_to_slot[row] = c0 + i;
        } else if (i < hi) {
          slot_to_row[c0 + i] = -1;
        }
        __syncwarp();
        if (valid && lane == __ffs(mask) - 1) warp_base[warp][e] += __popc(mask);
        __syncwarp();
      }
    } else if (tid < 32) {
      // many experts: the first warp walks the chunk in order
      for (int i0 = 0; i0 < cn; i0 += 32) {
        const int i = i0 + lane;
        const int e = i < cn ? stage[i] : -1;
        const bool valid = i < cn && e >= 0 && e < E;
        // invalid lanes get distinct keys so they never group with a real expert
        const int key = valid ? e : -1 - lane;
        const unsigned mask = __match_any_sync(0xFFFFFFFFu, key);
        const int rank = __popc(mask & ((1u << lane) - 1u));
        if (valid) {
          const int row = base[e] + rank;
          slot_to_row[c0 + i] = row;
          row_to_slot[row] = c0 + i;
        } else if (i < cn) {
          slot_to_row[c0 + i] = -1;
        }
        __syncwarp();
        if (valid && lane == __ffs(mask) - 1) base[e] += __popc(mask);
        __syncwarp();
      }
    }
    __syncthreads();
  }
  if (bad && hdr != nullptr && tid == 0) atomicCAS(hdr + H_STATUS, 0u, ST_INVALID);
}

constexpr int GATE_WARPS = 8;  // tokens per CTA at a time (one warp each)

// Top-k gate, one warp per token.  The token's scores are staged in shared
// memory (a NaN becomes -inf); topk rounds of a warp-wide arg-max (largest
// score, then lowest expert id) pick the experts, each chosen score marked NaN
// so that later rounds skip it; the chosen scores are then turned into
// softmax weights in fp32: exp(s_j - s_0) / sum over the chosen, s_0 the
// largest, or, when s_0 is infinite, equal shares among the scores equal to
// it.  The weights array holds the chosen scores between the two passes.
__global__ void __launch_bounds__(GATE_WARPS * 32)
moe_topk_gate_kernel(const float* __restrict__ logits, int T, int E, int topk,
                     int32_t* __restrict__ ids, float* __restrict__ weights) {
  extern __shared__ float gate_scores[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float* sv = gate_scores + warp * E;
  for (int t = blockIdx.x * GATE_WARPS + warp; t < T; t += gridDim.x * GATE_WARPS) {
    const float* row = logits + static_cast<size_t>(t) * E;
    for (int e = lane; e < E; e += 32) {
      const float v = __ldg(row + e);
      sv[e] = (v != v) ? -INFINITY : v;
    }
    __syncwarp();
    int32_t* id_out = ids + static_cast<size_t>(t) * topk;
    float* w_out = weights + static_cast<size_t>(t) * topk;
    float top = 0.0f;
    for (int j = 0; j < topk; ++j) {
      float best = -INFINITY;
      int bi = E;  // no candidate yet; any unchosen score, even -inf, beats it
      for (int e = lane; e < E; e += 32) {
        const float v = sv[e];
        if (v != v) continue;  // chosen in an earlier round
        if (v > best || (v == best && e < bi)) {
          best = v;
          bi = e;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ob = __shfl_xor_sync(0xFFFFFFFFu, best, o);
        const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
        if (ob > best || (ob == best && oi < bi)) {
          best = ob;
          bi = oi;
        }
      }
      // (best, bi) is the same in every lane: a total order has one maximum,
      // and j < topk <= E leaves at least one unchosen score
      if (j == 0) top = best;
      if (lane == 0) {
        id_out[j] = bi;
        w_out[j] = best;
      }
      if (lane == (bi & 31)) sv[bi] = NAN;
      __syncwarp();
    }
    const bool inf_top = isinf(top);
    float zsum = 0.0f;
    for (int j = lane; j < topk; j += 32) {
      const float sj = w_out[j];
      const float z = inf_top ? (sj == top ? 1.0f : 0.0f) : expf(sj - top);
      w_out[j] = z;
      zsum += z;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) zsum += __shfl_xor_sync(0xFFFFFFFFu, zsum, o);
    for (int j = lane; j < topk; j += 32) w_out[j] = w_out[j] / zsum;
    __syncwarp();
  }
}

// tile_off[e] = sum_{e' < e} ceil(count_e' / unit_rows) from a given offsets array.
__global__ void tile_offsets_kernel(const int32_t* offsets, int E, int unit_rows, int32_t* tile_off) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  int acc = 0;
  for (int e = 0; e < E; ++e) {
    tile_off[e] = acc;
    const int c = offsets[e + 1] - offsets[e];
    acc += (c > 0 ? (c + unit_rows - 1) / unit_rows : 0);
  }
  tile_off[E] = acc;
}

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

// Sizes every MoE layout accepts (the workspace does not depend on the split).
bool moe_common_ok(int R, int T, int H, int F, int E, int topk) {
  return R >= 1 && R <= FLUX_MAX_RANKS && T >= 0 && H >= 0 && F >= 0 && E >= 1 &&
         E <= FLUX_MAX_EXPERTS && topk >= 1 && topk <= E && T % R == 0 &&
         static_cast<long long>(T) * topk < (1ll << 31);
}

// EP x TP split: R / tp expert groups of tp ranks; each group holds E / (R/tp)
// experts, each rank of a group an F/tp block of them.  tp = R is the
// tensor-parallel layout, tp = 1 pure expert parallel.
bool moe_split_ok(int R, int tp, int T, int H, int F, int E, int topk) {
  return moe_common_ok(R, T, H, F, E, topk) && tp >= 1 && tp <= R && R % tp == 0 &&
         E % (R / tp) == 0 && F % tp == 0;
}

bool moe_shape_ok(int R, int T, int H, int F, int E, int topk) {
  return moe_split_ok(R, R, T, H, F, E, topk);
}

size_t a256(size_t v) { return round_up(v, WS_ALIGN); }

// workspace layout (offsets from the start): header, tile table, then the
// layer1 part (MOE_RS, MOE_LAYERS), then the layer0 part (MOE_AG,
// MOE_LAYERS), so that the one-call layer finds each part where the single
// calls put it
struct MoeWs {
  size_t tile_off, counts, offsets, s2r, r2s, acc, row_cnt, unit_cnt, stage, mbox, mbox_bytes, mbox1, mbox1_bytes,
      total;
};

// Dynamic schedule of the staged layer0: at most this many regions (CTA pairs).
constexpr int MOE0_MAX_REGIONS = 256;

// Bound on the staged layer0's units for any EP x TP split of these sizes:
// m-units of BM * MOE0S_CL rows (one partial m-unit per expert at most) times
// ceil(F / tp / 512) * tp <= ceil(F / 512) + R column tiles over the ranks
// (ceil(F / 512) with the ranks' columns side by side).
long long moe0_unit_bound(int R, int T, int F, int E, int topk) {
  const long long n = static_cast<long long>(T) * topk;
  const long long mts = (n + BM * MOE0S_CL - 1) / (BM * MOE0S_CL) + E;
  return mts * ((F + 2 * BN - 1) / (2 * BN) + R);
}

MoeWs moe_layout(flux_op_t op, int R, int T, int H, int F, int E, int topk) {
  MoeWs w{};
  const size_t n = static_cast<size_t>(T) * topk;
  size_t o = WS_HEADER;
  w.tile_off = o;
  o += a256((E + 1) * sizeof(int32_t));
  if (op == FLUX_OP_MOE_RS || op == FLUX_OP_MOE_LAYERS) {
    // routing recomputed here when the caller passes none
    w.counts = o;
    o += a256(E * sizeof(int32_t));
    w.offsets = o;
    o += a256((E + 1) * sizeof(int32_t));
    w.s2r = o;
    o += a256(n * sizeof(int32_t));
    w.r2s = o;
    o += a256(n * sizeof(int32_t));
    w.acc = o;
    o += a256(static_cast<size_t>(T) * H * sizeof(float));
    // rank groups: adds per (token, 512-column tile) of the fp32 rows
    w.row_cnt = o;
    o += a256(static_cast<size_t>(T) * ((H + 2 * BN - 1) / (2 * BN)) * sizeof(uint32_t));
    // mailboxes of layer1's dynamic schedule (rank groups on 256 x 512 tiles):
    // at most 2 U + 4 MOE0_MAX_REGIONS entries for U = (ceil(T*topk / 256) + E)
    // ceil(H / 512) R units (every rank of an expert's group computes all H
    // columns of its partial) over any EP x TP split
    const long long u1 = (static_cast<long long>((n + BM * MOE0S_CL - 1) / (BM * MOE0S_CL)) + E) *
                         ((H + 2 * BN - 1) / (2 * BN)) * R;
    w.mbox1 = o;
    w.mbox1_bytes = a256(static_cast<size_t>(2 * u1 + 4 * MOE0_MAX_REGIONS) * sizeof(uint32_t));
    o += w.mbox1_bytes;
  }
  if (op == FLUX_OP_MOE_AG || op == FLUX_OP_MOE_LAYERS) {
    // staged layer0: one ready counter per m-unit of BM * MOE0S_CL rows, and
    // the grouped A rows [T*topk x H] (16-bit)
    const size_t units = (n + BM * MOE0S_CL - 1) / (BM * MOE0S_CL) + static_cast<size_t>(E);
    w.unit_cnt = o;
    o += a256(units * sizeof(uint32_t));
    w.stage = o;
    o += a256(n * static_cast<size_t>(H) * 2);
    // mailboxes of the dynamic unit schedule: g regions of 2 ceil(U / g) + 2
    // entries, at most 2 U + 4 MOE0_MAX_REGIONS
    w.mbox = o;
    w.mbox_bytes = a256(static_cast<size_t>(2 * moe0_unit_bound(R, T, F, E, topk) + 4 * MOE0_MAX_REGIONS) *
                        sizeof(uint32_t));
    o += w.mbox_bytes;
  }
  w.total = o;
  return w;
}

flux_status_t launch_route(const int32_t* ids, int n, int E, int32_t* counts, int32_t* offsets,
                           int32_t* s2r, int32_t* r2s, int32_t* tile_off, int unit_rows,
                           uint32_t* unit_cnt, uint32_t* hdr, cudaStream_t s) {
  moe_route_kernel<<<1, ROUTE_THREADS, 0, s>>>(ids, n, E, counts, offsets, s2r, r2s, tile_off,
                                               unit_rows, unit_cnt, hdr);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? FLUX_OK : cuda_fail(e);
}

}  // namespace
}  // namespace flux

using namespace flux;

extern "C" size_t flux_moe_workspace_size(flux_op_t op, int R, int T, int H, int F, int E,
                                          int topk) {
  if (op == FLUX_OP_MOE_EP_AG || op == FLUX_OP_MOE_EP_RS) {
    // any EP x TP split of these sizes; the call itself checks the split
    if (!moe_common_ok(R, T, H, F, E, topk)) return 0;
    return moe_layout(op == FLUX_OP_MOE_EP_AG ? FLUX_OP_MOE_AG : FLUX_OP_MOE_RS, R, T, H, F, E,
                      topk).total;
  }
  if (!moe_shape_ok(R, T, H, F, E, topk)) return 0;
  if (op != FLUX_OP_MOE_AG && op != FLUX_OP_MOE_RS && op != FLUX_OP_MOE_LAYERS) return 0;
  return moe_layout(op, R, T, H, F, E, topk).total;
}

extern "C" flux_status_t flux_moe_topk_gate(int T, int E, int topk, const float* logits,
                                            int32_t* topk_ids, float* topk_weights,
                                            void* stream) {
  if (T < 0 || E < 1 || E > FLUX_MAX_EXPERTS || topk < 1 || topk > E ||
      static_cast<long long>(T) * E >= (1ll << 40) ||
      static_cast<long long>(T) * topk >= (1ll << 31))
    return FLUX_ERR_INVALID_ARG;
  if (T > 0 && (logits == nullptr || topk_ids == nullptr || topk_weights == nullptr))
    return FLUX_ERR_INVALID_ARG;
  DeviceInfo dev;
  flux_status_t st = current_device(&dev);
  if (st != FLUX_OK) return st;
  if (T == 0) return FLUX_OK;
  const long long want = (static_cast<long long>(T) + GATE_WARPS - 1) / GATE_WARPS;
  const int grid = static_cast<int>(std::min<long long>(want, 8ll * dev.sm_count));
  const size_t smem = static_cast<size_t>(GATE_WARPS) * E * sizeof(float);  // <= 32 KB
  moe_topk_gate_kernel<<<grid, GATE_WARPS * 32, smem, static_cast<cudaStream_t>(stream)>>>(
      logits, T, E, topk, topk_ids, topk_weights);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? FLUX_OK : cuda_fail(e);
}

extern "C" flux_status_t flux_moe_route(int T, int E, int topk, const int32_t* topk_ids,
                                        int32_t* counts, int32_t* offsets, int32_t* slot_to_row,
                                        int32_t* row_to_slot, void* workspace,
                                        size_t workspace_bytes, void* stream) {
  if (T < 0 || E < 1 || E > FLUX_MAX_EXPERTS || topk < 1 ||
      static_cast<long long>(T) * topk >= (1ll << 31))
    return FLUX_ERR_INVALID_ARG;
  if (counts == nullptr || offsets == nullptr) return FLUX_ERR_INVALID_ARG;
  const int n = T * topk;
  if (n > 0 && (topk_ids == nullptr || slot_to_row == nullptr || row_to_slot == nullptr))
    return FLUX_ERR_INVALID_ARG;
  if (workspace != nullptr) {
    flux_status_t st = check_workspace(workspace, workspace_bytes, WS_HEADER);
    if (st != FLUX_OK) return st;
  }
  DeviceInfo dev;
  flux_status_t st = current_device(&dev);
  if (st != FLUX_OK) return st;
  return launch_route(topk_ids, n, E, counts, offsets, slot_to_row, row_to_slot, nullptr, BM,
                      nullptr,
                      static_cast<uint32_t*>(workspace), static_cast<cudaStream_t>(stream));
}

namespace flux {
namespace {

// Layer0 for an EP x TP split (tp ranks per expert group; tp = R is tensor
// parallel).  Rank r = g tp + t: w1_shards[r] [E/EP x H x F/tp] holds column
// block t of the experts of group g, and h_out[r] [T*topk x F/tp] receives the
// rows of those experts (the other rows are left as they were, so ranks of
// different groups may share one buffer).  `ws_op` names the layout of the
// workspace (MOE_AG, or MOE_LAYERS inside the one-call layer).
flux_status_t moe_layer0_impl(
    flux_op_t ws_op, int tp, int R, int T, int H, int F, int E, int topk, flux_dtype_t dtype,
    const void* const* x_shards, const void* const* w1_shards, const int32_t* topk_ids,
    void* const* h_out, int32_t* counts, int32_t* offsets, int32_t* slot_to_row,
    int32_t* row_to_slot, const uint32_t* ready_flags, void* workspace, size_t workspace_bytes,
    const flux_opts_t* opts, void* stream) {
  if (!moe_split_ok(R, tp, T, H, F, E, topk) || (dtype != FLUX_F16 && dtype != FLUX_BF16))
    return FLUX_ERR_INVALID_ARG;
  if (x_shards == nullptr || w1_shards == nullptr || h_out == nullptr || counts == nullptr ||
      offsets == nullptr || slot_to_row == nullptr || row_to_slot == nullptr ||
      (T > 0 && topk_ids == nullptr))
    return FLUX_ERR_INVALID_ARG;
  const MoeWs L = moe_layout(ws_op, R, T, H, F, E, topk);
  flux_status_t st = check_workspace(workspace, workspace_bytes, L.total);
  if (st != FLUX_OK) return st;
  flux_opts_t tuned;
  if (opts == nullptr && tuned_opts(FLUX_OP_MOE_AG, {R, tp, T, H, F, E, topk, 0}, dtype, &tuned))
    opts = &tuned;
  const bool pull = opts != nullptr && opts->moe_pull_gather != 0;
  const int cl = pull ? MOE0_CL : MOE0S_CL;
  // output columns per rank and experts per rank's weight block
  const int Fr = F / tp, EB = E / (R / tp), rows = T / R, n = T * topk;
  for (int r = 0; r < R; ++r) {
    if (x_shards[r] == nullptr || w1_shards[r] == nullptr || h_out[r] == nullptr)
      return FLUX_ERR_INVALID_ARG;
    if (!aligned16(x_shards[r]) || !aligned16(w1_shards[r]) || !aligned16(h_out[r]))
      return FLUX_ERR_UNSUPPORTED;
  }
  if (H % 8 || Fr % 8) return FLUX_ERR_UNSUPPORTED;
  DeviceInfo dev;
  if ((st = current_device(&dev)) != FLUX_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* tile_off = reinterpret_cast<int32_t*>(ws + L.tile_off);
  uint32_t* unit_cnt = pull ? nullptr : reinterpret_cast<uint32_t*>(ws + L.unit_cnt);
  if ((st = launch_route(topk_ids, n, E, counts, offsets, slot_to_row, row_to_slot, tile_off,
                         BM * cl, unit_cnt, static_cast<uint32_t*>(workspace), s)) != FLUX_OK)
    return st;
  if (n == 0 || Fr == 0) return FLUX_OK;
  if (H == 0) {
    for (int r = 0; r < R; ++r) {
      cudaError_t e = cudaMemsetAsync(h_out[r], 0, static_cast<size_t>(n) * Fr * 2, s);
      if (e != cudaSuccess) return cuda_fail(e);
    }
    return FLUX_OK;
  }
  KParams p{};
  void* stage = ws + L.stage;
  CUtensorMap tm_stage;
  if (!pull &&
      (st = encode_2d(&tm_stage, dtype, stage, H, n, static_cast<uint64_t>(H) * 2, BK, BM)) != FLUX_OK)
    return st;
  for (int r = 0; r < R; ++r) {
    if ((st = encode_3d(&p.tmB[r], dtype, w1_shards[r], Fr, H, EB, B_BOX_N, BK)) != FLUX_OK) return st;
    if (!pull) p.tmA[r] = tm_stage;  // every rank reads the one staged copy of the rows
    p.out[r] = h_out[r];
    if ((st = encode_2d(&p.tmOut[r], dtype, h_out[r], Fr, n, static_cast<uint64_t>(Fr) * 2, 64, 32)) != FLUX_OK)
      return st;
    p.xsrc[r] = x_shards[r];
  }
  p.stage = stage;
  p.unit_cnt = unit_cnt;
  p.stage_ctas = (opts && opts->moe_stage_ctas > 0) ? opts->moe_stage_ctas : 0;
  p.moe_tp = tp;
  p.moe_el = EB;
  // expert outermost, then column tile, then the expert's m-units with the
  // ranks fastest: an expert's rows and one column tile of its weight blocks
  // stay in L2 while they are used (DRAM read per call at the MoE workload's
  // sizes 1.42 GB, 1.5 % faster than the m-fastest order over all experts:
  // 1.52 GB)
  p.moe_order = 3;
  // staged: the 512-column tiles run over the group's ranks' columns side by
  // side where every 64-column box lies in one rank (F/tp a multiple of 64),
  // so a rank block of 3.5 tiles leaves no half-wide tile (at the MoE
  // workload's sizes a half tile's k-loop took 89 % of a whole one's time)
  const bool xcols = !pull && Fr % B_BOX_N == 0;
  p.xcols = xcols ? Fr : 0;
  p.R = R;
  p.M = n;
  p.N = xcols ? tp * Fr : Fr;
  p.K = H;
  p.Nt = pull ? (Fr + BN - 1) / BN : (p.N + 2 * BN - 1) / (2 * BN);  // 256- / 512-column tiles
  p.KT = (H + BK - 1) / BK;
  p.ldo = Fr;
  p.rows_per_rank = rows;
  p.flags = ready_flags;
  p.offsets = offsets;
  p.row_to_slot = row_to_slot;
  p.tile_off = tile_off;
  p.E = E;
  p.topk = topk;
  p.T = T;
  p.H = H;
  p.timeout_ns = (opts && opts->timeout_ns) ? opts->timeout_ns : DEFAULT_TIMEOUT_NS;
  p.epoch = (opts && opts->epoch) ? opts->epoch : 1u;
  p.group_n = (opts && opts->group_n > 0) ? opts->group_n : 8;
  p.seq = next_seq();
  p.hdr = static_cast<uint32_t*>(workspace);
  p.trace = opts ? static_cast<unsigned long long*>(opts->trace) : nullptr;
  p.trace_words = (opts && opts->trace) ? static_cast<long long>(opts->trace_words) : 0;
  p.debug_probe = opts ? opts->debug_probe : 0;
  p.acc_halves = (opts && opts->acc_whole) ? 0 : 1;
  const long long max_units =
      (static_cast<long long>((n + BM * cl - 1) / (BM * cl)) + E) * p.Nt *
      static_cast<long long>(xcols ? 1 : tp);
  if (pull) {
    const int grid = grid_dt<MODE_MOE_GATHER, MOE0_CL>(dtype, dev, opts, max_units);
    if (grid == 0) return FLUX_ERR_CUDA;
    return launch_dt<MODE_MOE_GATHER, MOE0_CL>(dtype, p, grid, s);
  }
  const int grid = grid_dt<MODE_MOE_STAGED, MOE0S_CL>(dtype, dev, opts, max_units);
  if (grid == 0) return FLUX_ERR_CUDA;
  const long long g = grid / MOE0S_CL;
  const long long cap = 2 * ((max_units + g - 1) / g) + 2;
  if (!(opts && opts->moe_static_schedule) && g <= MOE0_MAX_REGIONS &&
      static_cast<size_t>(g * cap) * sizeof(uint32_t) <= L.mbox_bytes) {
    // dynamic: each pair's producer claims the pair's next unit from the
    // counter (units differ in cost: a half-wide last column tile, the
    // experts' partial last m-units), so the last wave ends evenly
    p.dyn = 1;
    p.mbox = reinterpret_cast<uint32_t*>(ws + L.mbox);
    p.mbox_cap = static_cast<int>(cap);
    p.claim_reserve = 0;
  }
  return launch_dt<MODE_MOE_STAGED, MOE0S_CL>(dtype, p, grid, s);
}

// Layer1 for an EP x TP split.  Rank r = g tp + t: h_shards[r] [T*topk x F/tp]
// (only the rows of group g's experts are read) and w2_shards[r]
// [E/EP x F/tp x H] (row block t of group g's experts); every (token, k) slot
// adds tp partials.
flux_status_t moe_layer1_impl(
    int tp, int R, int T, int H, int F, int E, int topk, flux_dtype_t dtype,
    const void* const* h_shards, const void* const* w2_shards, const int32_t* topk_ids,
    const float* topk_weights, const int32_t* offsets, const int32_t* slot_to_row,
    const int32_t* row_to_slot, void* const* out, void* workspace, size_t workspace_bytes,
    const flux_opts_t* opts, void* stream) {
  if (!moe_split_ok(R, tp, T, H, F, E, topk) || (dtype != FLUX_F16 && dtype != FLUX_BF16))
    return FLUX_ERR_INVALID_ARG;
  const bool given = offsets != nullptr;
  if (given != (slot_to_row != nullptr) || given != (row_to_slot != nullptr))
    return FLUX_ERR_INVALID_ARG;
  if (h_shards == nullptr || w2_shards == nullptr || out == nullptr ||
      (T > 0 && (topk_ids == nullptr || topk_weights == nullptr)))
    return FLUX_ERR_INVALID_ARG;
  const MoeWs L = moe_layout(FLUX_OP_MOE_RS, R, T, H, F, E, topk);
  flux_status_t st = check_workspace(workspace, workspace_bytes, L.total);
  if (st != FLUX_OK) return st;
  flux_opts_t tuned;
  if (opts == nullptr && tuned_opts(FLUX_OP_MOE_RS, {R, tp, T, H, F, E, topk, 0}, dtype, &tuned))
    opts = &tuned;
  // reduction length per rank and experts per rank's weight block
  const int Fr = F / tp, EB = E / (R / tp), rows = T / R, n = T * topk;
  for (int r = 0; r < R; ++r) {
    if (h_shards[r] == nullptr || w2_shards[r] == nullptr || out[r] == nullptr)
      return FLUX_ERR_INVALID_ARG;
    if (!aligned16(h_shards[r]) || !aligned16(w2_shards[r]) || !aligned16(out[r]))
      return FLUX_ERR_UNSUPPORTED;
  }
  if (H % 8 || Fr % 8) return FLUX_ERR_UNSUPPORTED;
  DeviceInfo dev;
  if ((st = current_device(&dev)) != FLUX_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (T == 0 || H == 0) return FLUX_OK;
  if (Fr == 0) {
    for (int r = 0; r < R; ++r) {
      cudaError_t e = cudaMemsetAsync(out[r], 0, static_cast<size_t>(rows) * H * 2, s);
      if (e != cudaSuccess) return cuda_fail(e);
    }
    return FLUX_OK;
  }
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* tile_off = reinterpret_cast<int32_t*>(ws + L.tile_off);
  if (!given) {
    offsets = reinterpret_cast<int32_t*>(ws + L.offsets);
    row_to_slot = reinterpret_cast<int32_t*>(ws + L.r2s);
    if ((st = launch_route(topk_ids, n, E, reinterpret_cast<int32_t*>(ws + L.counts),
                           const_cast<int32_t*>(offsets), reinterpret_cast<int32_t*>(ws + L.s2r),
                           const_cast<int32_t*>(row_to_slot), tile_off, BM * MOE1_CL, nullptr,
                           static_cast<uint32_t*>(workspace), s)) != FLUX_OK)
      return st;
  } else {
    tile_offsets_kernel<<<1, 32, 0, s>>>(offsets, E, BM * MOE1_CL, tile_off);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e);
  }
  KParams p{};
  for (int r = 0; r < R; ++r) {
    if ((st = encode_2d(&p.tmA[r], dtype, h_shards[r], Fr, n, static_cast<uint64_t>(Fr) * 2, BK,
                        BM)) != FLUX_OK)
      return st;
    if ((st = encode_3d(&p.tmB[r], dtype, w2_shards[r], H, Fr, EB, B_BOX_N, BK)) != FLUX_OK) return st;
    p.out[r] = out[r];
  }
  p.moe_tp = tp;
  p.moe_el = EB;
  p.moe_order = 0;  // rank outermost: concurrent tiles add into different token rows
  p.R = R;
  p.M = n;
  p.N = H;
  p.K = Fr;
  p.KT = (Fr + BK - 1) / BK;
  const bool wide = p.KT >= MOE1_WIDE_KT;
  // rank groups (moe_l1_ranks; default all tp ranks of the expert group): a
  // CTA pair computes the partials of rg ranks of one 256 x 512 tile back to
  // back into one TMEM accumulator (rank-innermost claims on the dynamic
  // schedule) and makes one gate-weighted add per slot for the group.  At
  // T 4096, H 4096, F 14336, 8 experts, top-2, 8 ranks: 654 against 697 us
  // with one 256 x 256 tile and one add per rank (groups of 4: 716 us, the
  // last wave of 4-rank claims idles 13 % of the call)
  const int rg = (opts && opts->moe_l1_ranks > 0) ? opts->moe_l1_ranks : tp;
  if (opts && opts->moe_l1_ranks > 0 && tp % opts->moe_l1_ranks) return FLUX_ERR_INVALID_ARG;
  const bool grouped = tp > 1 && rg > 1;
  const int tile_n = (wide || grouped) ? 2 * BN : BN;
  p.Nt = (H + tile_n - 1) / tile_n;
  p.ldo = H;
  p.rows_per_rank = rows;
  p.offsets = offsets;
  p.row_to_slot = row_to_slot;
  p.tile_off = tile_off;
  p.topk_w = topk_weights;
  p.E = E;
  p.topk = topk;
  p.T = T;
  p.H = H;
  p.acc = reinterpret_cast<float*>(ws + L.acc);
  p.timeout_ns = (opts && opts->timeout_ns) ? opts->timeout_ns : DEFAULT_TIMEOUT_NS;
  p.epoch = (opts && opts->epoch) ? opts->epoch : 1u;
  p.group_n = (opts && opts->group_n > 0) ? opts->group_n : 8;
  p.seq = next_seq();
  p.hdr = static_cast<uint32_t*>(workspace);
  p.trace = opts ? static_cast<unsigned long long*>(opts->trace) : nullptr;
  p.trace_words = (opts && opts->trace) ? static_cast<long long>(opts->trace_words) : 0;
  p.debug_probe = opts ? opts->debug_probe : 0;
  p.acc_halves = (opts && opts->acc_whole) ? 0 : 1;
  const long long max_units =
      (static_cast<long long>((n + BM * MOE1_CL - 1) / (BM * MOE1_CL)) + E) * p.Nt *
      static_cast<long long>(tp);
  if (grouped) {
    const int grid = grid_dt<MODE_MOE_SCATTER_WIDE, MOE1_CL>(dtype, dev, opts, max_units);
    if (grid == 0) return FLUX_ERR_CUDA;
    const long long g = grid / MOE1_CL;
    const long long cap = 2 * ((max_units + g - 1) / g) + 2;
    // (the area holds 2 U + 4 MOE0_MAX_REGIONS entries, U >= max_units)
    if (g > MOE0_MAX_REGIONS || static_cast<size_t>(g * cap) * sizeof(uint32_t) > L.mbox1_bytes)
      return FLUX_ERR_WORKSPACE;
    // rank innermost (a group's ranks are consecutive units), then the column
    // tiles of one m-unit (650 against 664 us with the m-units fastest)
    p.moe_order = 5;
    p.rs_group = rg;
    // each (token, column tile) receives topk x tp / rg adds; the last one
    // converts it and no end-of-call pass runs (634-635 against 654-655 us
    // with the pass at the MoE workload's sizes)
    p.row_cnt = reinterpret_cast<uint32_t*>(ws + L.row_cnt);
    p.row_tiles = (H + 2 * BN - 1) / (2 * BN);
    p.row_arrivals = topk * (tp / rg);
    p.split_from = MOE1_SPLIT_TAIL ? static_cast<int>(g) : 0;  // group claims split rank by rank
    p.dyn = 1;
    p.mbox = reinterpret_cast<uint32_t*>(ws + L.mbox1);
    p.mbox_cap = static_cast<int>(cap);
    p.claim_reserve = 0;
    return launch_dt<MODE_MOE_SCATTER_WIDE, MOE1_CL>(dtype, p, grid, s);
  }
  if (wide) {
    const int grid = grid_dt<MODE_MOE_SCATTER_WIDE, MOE1_CL>(dtype, dev, opts, max_units);
    if (grid == 0) return FLUX_ERR_CUDA;
    return launch_dt<MODE_MOE_SCATTER_WIDE, MOE1_CL>(dtype, p, grid, s);
  }
  const int grid = grid_dt<MODE_MOE_SCATTER, MOE1_CL>(dtype, dev, opts, max_units);
  if (grid == 0) return FLUX_ERR_CUDA;
  return launch_dt<MODE_MOE_SCATTER, MOE1_CL>(dtype, p, grid, s);
}

}  // namespace
}  // namespace flux

extern "C" flux_status_t flux_moe_ag_grouped_gemm(
    int R, int T, int H, int F, int E, int topk, flux_dtype_t dtype, const void* const* x_shards,
    const void* const* w1_shards, const int32_t* topk_ids, void* const* h_out, int32_t* counts,
    int32_t* offsets, int32_t* slot_to_row, int32_t* row_to_slot, const uint32_t* ready_flags,
    void* workspace, size_t workspace_bytes, const flux_opts_t* opts, void* stream) {
  return moe_layer0_impl(FLUX_OP_MOE_AG, R, R, T, H, F, E, topk, dtype, x_shards, w1_shards,
                         topk_ids, h_out,
                         counts, offsets, slot_to_row, row_to_slot, ready_flags, workspace,
                         workspace_bytes, opts, stream);
}

extern "C" flux_status_t flux_moe_grouped_gemm_rs(
    int R, int T, int H, int F, int E, int topk, flux_dtype_t dtype, const void* const* h_shards,
    const void* const* w2_shards, const int32_t* topk_ids, const float* topk_weights,
    const int32_t* offsets, const int32_t* slot_to_row, const int32_t* row_to_slot,
    void* const* out, void* workspace, size_t workspace_bytes, const flux_opts_t* opts,
    void* stream) {
  return moe_layer1_impl(R, R, T, H, F, E, topk, dtype, h_shards, w2_shards, topk_ids,
                         topk_weights, offsets, slot_to_row, row_to_slot, out, workspace,
                         workspace_bytes, opts, stream);
}

extern "C" flux_status_t flux_moe_ep_dispatch_gemm(
    int R, int tp, int T, int H, int F, int E, int topk, flux_dtype_t dtype,
    const void* const* x_shards, const void* const* w1_shards, const int32_t* topk_ids,
    void* const* h_out, int32_t* counts, int32_t* offsets, int32_t* slot_to_row,
    int32_t* row_to_slot, const uint32_t* ready_flags, void* workspace, size_t workspace_bytes,
    const flux_opts_t* opts, void* stream) {
  return moe_layer0_impl(FLUX_OP_MOE_AG, tp, R, T, H, F, E, topk, dtype, x_shards, w1_shards,
                         topk_ids, h_out,
                         counts, offsets, slot_to_row, row_to_slot, ready_flags, workspace,
                         workspace_bytes, opts, stream);
}

extern "C" flux_status_t flux_moe_ep_gemm_combine(
    int R, int tp, int T, int H, int F, int E, int topk, flux_dtype_t dtype,
    const void* const* h_shards, const void* const* w2_shards, const int32_t* topk_ids,
    const float* topk_weights, const int32_t* offsets, const int32_t* slot_to_row,
    const int32_t* row_to_slot, void* const* out, void* workspace, size_t workspace_bytes,
    const flux_opts_t* opts, void* stream) {
  return moe_layer1_impl(tp, R, T, H, F, E, topk, dtype, h_shards, w2_shards, topk_ids,
                         topk_weights, offsets, slot_to_row, row_to_slot, out, workspace,
                         workspace_bytes, opts, stream);
}

extern "C" flux_status_t flux_moe_layers(int R, int T, int H, int F, int E, int topk,
                                         flux_dtype_t dtype, const void* const* x_shards,
                                         const void* const* w1_shards,
                                         const void* const* w2_shards, const int32_t* topk_ids,
                                         const float* topk_weights, void* const* h,
                                         void* const* out, const uint32_t* ready_flags,
                                         void* workspace, size_t workspace_bytes,
                                         const flux_opts_t* opts, void* stream) {
  if (!moe_shape_ok(R, T, H, F, E, topk) || h == nullptr) return FLUX_ERR_INVALID_ARG;
  const MoeWs L = moe_layout(FLUX_OP_MOE_LAYERS, R, T, H, F, E, topk);
  flux_status_t st = check_workspace(workspace, workspace_bytes, L.total);
  if (st != FLUX_OK) return st;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* counts = reinterpret_cast<int32_t*>(ws + L.counts);
  int32_t* offsets = reinterpret_cast<int32_t*>(ws + L.offsets);
  int32_t* s2r = reinterpret_cast<int32_t*>(ws + L.s2r);
  int32_t* r2s = reinterpret_cast<int32_t*>(ws + L.r2s);
  // layer0 writes its routing into layer1's part of the workspace
  if ((st = moe_layer0_impl(FLUX_OP_MOE_LAYERS, R, R, T, H, F, E, topk, dtype, x_shards,
                            w1_shards, topk_ids, h, counts, offsets, s2r, r2s, ready_flags,
                            workspace, workspace_bytes, opts, stream)) != FLUX_OK)
    return st;
  return flux_moe_grouped_gemm_rs(R, T, H, F, E, topk, dtype, reinterpret_cast<const void* const*>(h),
                                  w2_shards, topk_ids, topk_weights, offsets, s2r, r2s, out,
                                  workspace, workspace_bytes, opts, stream);
}
