// Per-problem launch-option table and the calls that fill it by measurement.
//
// The pages tune FLUX's communication tile per shape (FLUX paper review,
// "关键优化": the tile size of the fused kernel is searched per problem) and
// let COMET pick among precompiled fused variants at run time by token count
// and parallel layout (COMET article, "动态负载平衡").  Here every variant is
// already compiled in; what a problem may choose is its launch options: the
// raster band width, the GEMM-RS rank grouping, the stream-K grid, and for
// MoE layer0 the staged or producer-side gather.  flux_tune_* time the
// candidates on the caller's stream and record the fastest for that problem
// (device, op, sizes, dtype); an entry point called with opts == NULL uses
// the recorded options of its problem, if any.
#include <algorithm>
#include <array>
#include <map>
#include <mutex>
#include <vector>

#include "flux_host.h"

namespace flux {
namespace {

using Key = std::array<int, 11>;  // device, op, dtype, up to 8 sizes

std::mutex g_mu;
std::map<Key, flux_opts_t> g_table;

Key make_key(flux_op_t op, const std::array<int, 8>& dims, flux_dtype_t dt) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
  Key k{};
  k[0] = dev;
  k[1] = static_cast<int>(op);
  k[2] = static_cast<int>(dt);
  for (int i = 0; i < 8; ++i) k[3 + i] = dims[i];
  return k;
}

// Median device time (ms) of `iters` calls of `run` on `s`, after one warm-up
// call; a failing call (launch or device status) ends the measurement.
template <class F>
flux_status_t time_call(F&& run, cudaStream_t s, void* workspace, size_t workspace_bytes,
                        int iters, float* ms) {
  flux_status_t st = run();
  if (st != FLUX_OK) return st;
  cudaEvent_t a, b;
  cudaError_t e = cudaEventCreate(&a);
  if (e != cudaSuccess) return cuda_fail(e);
  if ((e = cudaEventCreate(&b)) != cudaSuccess) {
    cudaEventDestroy(a);
    return cuda_fail(e);
  }
  std::vector<float> t;
  for (int i = 0; i < iters && st == FLUX_OK; ++i) {
    cudaEventRecord(a, s);
    st = run();
    cudaEventRecord(b, s);
    if ((e = cudaEventSynchronize(b)) != cudaSuccess) {
      st = cuda_fail(e);
      break;
    }
    float v = 0.f;
    cudaEventElapsedTime(&v, a, b);
    t.push_back(v);
  }
  cudaEventDestroy(a);
  cudaEventDestroy(b);
  if (st != FLUX_OK) return st;
  // a device-side error (a bounded wait that gave up) fails the candidate
  flux_device_report_t rep{};
  st = flux_get_status(workspace, workspace_bytes, s, &rep);
  if (st != FLUX_OK) return st;
  std::sort(t.begin(), t.end());
  *ms = t[t.size() / 2];
  return FLUX_OK;
}

constexpr int TUNE_ITERS = 5;

// Times every candidate, records and returns the fastest.
template <class F>
flux_status_t pick(flux_op_t op, const std::array<int, 8>& dims, flux_dtype_t dt,
                   const std::vector<flux_opts_t>& cands, F&& run_with, cudaStream_t s,
                   void* workspace, size_t workspace_bytes, flux_opts_t* best) {
  float best_ms = 0.f;
  int best_i = -1;
  for (size_t i = 0; i < cands.size(); ++i) {
    float ms = 0.f;
    const flux_opts_t* o = &cands[i];
    flux_status_t st = time_call([&] { return run_with(o); }, s, workspace, workspace_bytes,
                                 TUNE_ITERS, &ms);
    if (st != FLUX_OK) return st;
    if (best_i < 0 || ms < best_ms) {
      best_ms = ms;
      best_i = static_cast<int>(i);
    }
  }
  if (best_i < 0) return FLUX_ERR_INVALID_ARG;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    g_table[make_key(op, dims, dt)] = cands[best_i];
  }
  if (best) *best = cands[best_i];
  return FLUX_OK;
}

flux_opts_t base_opts() {
  flux_opts_t o{};
  return o;
}

}  // namespace

bool tuned_opts(flux_op_t op, const std::array<int, 8>& dims, flux_dtype_t dt, flux_opts_t* out) {
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = g_table.find(make_key(op, dims, dt));
  if (it == g_table.end()) return false;
  *out = it->second;
  return true;
}

}  // namespace flux

using namespace flux;

extern "C" void flux_tune_clear(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_table.clear();
}

extern "C" int flux_tune_count(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  return static_cast<int>(g_table.size());
}

extern "C" flux_status_t flux_tune_ag_gemm(int R, int M, int N, int K, flux_dtype_t dtype,
                                           const void* const* x_shards,
                                           const void* const* w_shards, void* const* out,
                                           const uint32_t* ready_flags, void* workspace,
                                           size_t workspace_bytes, void* stream,
                                           flux_opts_t* best) {
  std::vector<flux_opts_t> cands;
  for (int g : {2, 4, 8, 16}) {
    flux_opts_t o = base_opts();
    o.group_n = g;
    cands.push_back(o);
  }
  return pick(FLUX_OP_AG_GEMM, {R, M, N, K, 0, 0, 0, 0}, dtype, cands,
              [&](const flux_opts_t* o) {
                return flux_ag_gemm(R, M, N, K, dtype, x_shards, w_shards, out, ready_flags,
                                    workspace, workspace_bytes, o, stream);
              },
              static_cast<cudaStream_t>(stream), workspace, workspace_bytes, best);
}

extern "C" flux_status_t flux_tune_gemm_rs(int R, int M, int N, int K, flux_dtype_t dtype,
                                           const void* const* a_shards,
                                           const void* const* b_shards, void* const* out,
                                           void* workspace, size_t workspace_bytes, void* stream,
                                           flux_opts_t* best) {
  DeviceInfo dev;
  flux_status_t st = current_device(&dev);
  if (st != FLUX_OK) return st;
  if (R < 1 || M < 0 || N < 0) return FLUX_ERR_INVALID_ARG;
  std::vector<flux_opts_t> cands;
  if (rs_uses_stream_k(R, M, N, dev.sm_count, false)) {
    // stream-K: the grid (0 = whole units per CTA where three quarters stay busy)
    for (int g : {0, dev.sm_count, dev.sm_count * 7 / 8, dev.sm_count / 2}) {
      flux_opts_t o = base_opts();
      o.num_ctas = g;
      cands.push_back(o);
    }
  } else {
    for (int form : {1, 2})
      for (int g : {4, 8, 16})
        for (int tg : {0, 2}) {
          flux_opts_t o = base_opts();
          // regions of 4 with 256 x 512 pair tiles, or of 8 with 256 x 256
          o.rs_tile = form;
          o.group_n = g;
          // 0: one rank group per wave; 2: pairs of tiles (the R partials of a
          // tile in consecutive units)
          o.tiles_per_group = tg;
          cands.push_back(o);
        }
    // regions of 4: how many ranks' partials of a tile are summed in TMEM
    for (int rg : {1, 2, 8}) {
      if (R % rg) continue;
      flux_opts_t o = base_opts();
      o.rs_tile = 1;
      o.rs_group = rg;
      cands.push_back(o);
    }
  }
  return pick(FLUX_OP_GEMM_RS, {R, M, N, K, 0, 0, 0, 0}, dtype, cands,
              [&](const flux_opts_t* o) {
                return flux_gemm_rs(R, M, N, K, dtype, a_shards, b_shards, out, workspace,
                                    workspace_bytes, o, stream);
              },
              static_cast<cudaStream_t>(stream), workspace, workspace_bytes, best);
}

extern "C" flux_status_t flux_tune_moe_layer0(
    int R, int tp, int T, int H, int F, int E, int topk, flux_dtype_t dtype,
    const void* const* x_shards, const void* const* w1_shards, const int32_t* topk_ids,
    void* const* h_out, int32_t* counts, int32_t* offsets, int32_t* slot_to_row,
    int32_t* row_to_slot, const uint32_t* ready_flags, void* workspace, size_t workspace_bytes,
    void* stream, flux_opts_t* best) {
  std::vector<flux_opts_t> cands;
  for (int g : {8, 16}) {
    flux_opts_t o = base_opts();
    o.group_n = g;
    cands.push_back(o);  // staged copy, CTA pairs, dynamic unit schedule
  }
  {
    flux_opts_t o = base_opts();
    o.moe_static_schedule = 1;  // staged copy, CTA pairs, static unit schedule
    cands.push_back(o);
  }
  {
    flux_opts_t o = base_opts();
    o.moe_pull_gather = 1;  // producer-side gather, single CTAs
    cands.push_back(o);
  }
  return pick(FLUX_OP_MOE_AG, {R, tp, T, H, F, E, topk, 0}, dtype, cands,
              [&](const flux_opts_t* o) {
                return flux_moe_ep_dispatch_gemm(R, tp, T, H, F, E, topk, dtype, x_shards,
                                                 w1_shards, topk_ids, h_out, counts, offsets,
                                                 slot_to_row, row_to_slot, ready_flags,
                                                 workspace, workspace_bytes, o, stream);
              },
              static_cast<cudaStream_t>(stream), workspace, workspace_bytes, best);
}

extern "C" flux_status_t flux_tune_moe_layer1(
    int R, int tp, int T, int H, int F, int E, int topk, flux_dtype_t dtype,
    const void* const* h_shards, const void* const* w2_shards, const int32_t* topk_ids,
    const float* topk_weights, const int32_t* offsets, const int32_t* slot_to_row,
    const int32_t* row_to_slot, void* const* out, void* workspace, size_t workspace_bytes,
    void* stream, flux_opts_t* best) {
  std::vector<flux_opts_t> cands;
  // partials of how many ranks a CTA pair sums on chip (1: none, tp: the
  // whole group, tp / 2: half groups, twice the units for the same adds x 2)
  std::vector<int> groups = {1};
  if (tp > 1) groups.push_back(tp);
  if (tp % 2 == 0 && tp / 2 > 1) groups.push_back(tp / 2);
  for (int rg : groups)
    for (int g : {4, 8, 16}) {
      flux_opts_t o = base_opts();
      o.group_n = g;
      o.moe_l1_ranks = rg;
      cands.push_back(o);
    }
  return pick(FLUX_OP_MOE_RS, {R, tp, T, H, F, E, topk, 0}, dtype, cands,
              [&](const flux_opts_t* o) {
                return flux_moe_ep_gemm_combine(R, tp, T, H, F, E, topk, dtype, h_shards,
                                                w2_shards, topk_ids, topk_weights, offsets,
                                                slot_to_row, row_to_slot, out, workspace,
                                                workspace_bytes, o, stream);
              },
              static_cast<cudaStream_t>(stream), workspace, workspace_bytes, best);
}
