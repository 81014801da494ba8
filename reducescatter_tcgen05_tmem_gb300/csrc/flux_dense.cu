// Dense entry points: plain GEMM, AllGather + GEMM, GEMM + ReduceScatter.
#include <mutex>

#include "flux_host.h"
#include "flux_kernels.cuh"

namespace flux {
namespace {

template <int MODE, int DT>
flux_status_t launch(const KParams& p, int grid, cudaStream_t stream) {
  using KS = KernelShape<MODE, DT>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(fused_gemm_kernel<MODE, DT>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  });
  if (attr_err != cudaSuccess) return cuda_fail(attr_err);
  fused_gemm_kernel<MODE, DT><<<grid, KS::THREADS, SMEM_BYTES, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? FLUX_OK : cuda_fail(e);
}

template <int MODE>
flux_status_t launch_dt(flux_dtype_t dt, const KParams& p, int grid, cudaStream_t s) {
  return dt == FLUX_BF16 ? launch<MODE, 1>(p, grid, s) : launch<MODE, 0>(p, grid, s);
}

bool valid_dtype(flux_dtype_t dt) { return dt == FLUX_F16 || dt == FLUX_BF16; }

void fill_common(KParams& p, const flux_opts_t* opts, void* ws) {
  p.timeout_ns = (opts && opts->timeout_ns) ? opts->timeout_ns : DEFAULT_TIMEOUT_NS;
  p.epoch = (opts && opts->epoch) ? opts->epoch : 1u;
  p.group_n = (opts && opts->group_n > 0) ? opts->group_n : 8;
  p.seq = next_seq();
  p.hdr = static_cast<uint32_t*>(ws);
}

int grid_size(const DeviceInfo& d, const flux_opts_t* opts, long long work) {
  int g = (opts && opts->num_ctas > 0) ? opts->num_ctas : d.sm_count;
  if (work < g) g = static_cast<int>(work);
  return g < 1 ? 1 : g;
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

}  // namespace
}  // namespace flux

using namespace flux;

extern "C" size_t flux_workspace_size(flux_op_t op, int R, int M, int N, int K) {
  if (R < 1 || R > FLUX_MAX_RANKS || M < 0 || N < 0 || K < 0) return 0;
  switch (op) {
    case FLUX_OP_GEMM:
    case FLUX_OP_AG_GEMM:
      return WS_HEADER;
    case FLUX_OP_GEMM_RS:
      return WS_HEADER + rs_counter_bytes(M, N) + static_cast<size_t>(M) * N * sizeof(float);
    default:
      return 0;
  }
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
  }
  p.R = R;
  p.M = M;
  p.N = Nr;
  p.K = K;
  p.Mt = (M + BM - 1) / BM;
  p.Nt = (Nr + BN - 1) / BN;
  p.KT = (K + BK - 1) / BK;
  p.ldo = Nr;
  p.rows_per_rank = rows;
  p.a_box_m = box_m;
  p.num_units = R * p.Mt * p.Nt;
  p.flags = ready_flags;
  fill_common(p, opts, workspace);
  return launch_dt<MODE_STORE>(dtype, p, grid_size(dev, opts, p.num_units), s);
}

extern "C" flux_status_t flux_gemm(int M, int N, int K, flux_dtype_t dtype, const void* A,
                                   const void* B, void* C, void* workspace,
                                   size_t workspace_bytes, const flux_opts_t* opts, void* stream) {
  const void* a[1] = {A};
  const void* b[1] = {B};
  void* c[1] = {C};
  return flux_ag_gemm(1, M, N, K, dtype, a, b, c, nullptr, workspace, workspace_bytes, opts, stream);
}

extern "C" flux_status_t flux_gemm_rs(int R, int M, int N, int K, flux_dtype_t dtype,
                                      const void* const* a_shards, const void* const* b_shards,
                                      void* const* out, void* workspace, size_t workspace_bytes,
                                      const flux_opts_t* opts, void* stream) {
  if (R < 1 || R > FLUX_MAX_RANKS || M < 0 || N < 0 || K < 0 || !valid_dtype(dtype))
    return FLUX_ERR_INVALID_ARG;
  if (M % R || K % R) return FLUX_ERR_INVALID_ARG;
  if (a_shards == nullptr || b_shards == nullptr || out == nullptr) return FLUX_ERR_INVALID_ARG;
  const size_t need = flux_workspace_size(FLUX_OP_GEMM_RS, R, M, N, K);
  flux_status_t st = check_workspace(workspace, workspace_bytes, need);
  if (st != FLUX_OK) return st;
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
    if ((st = encode_2d(&p.tmA[r], dtype, a_shards[r], Kr, M, static_cast<uint64_t>(Kr) * 2, BK,
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
  p.Mt = (M + BM - 1) / BM;
  p.Nt = (N + BN - 1) / BN;
  p.KT = (Kr + BK - 1) / BK;
  p.ldo = N;
  p.rows_per_rank = rows;
  p.a_box_m = BM;
  const int tiles = p.Mt * p.Nt;
  p.num_units = tiles * R;
  p.total_ksteps = static_cast<long long>(p.num_units) * p.KT;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.counters = reinterpret_cast<uint32_t*>(ws + WS_HEADER);
  p.acc = reinterpret_cast<float*>(ws + WS_HEADER + rs_counter_bytes(M, N));
  fill_common(p, opts, workspace);

  // Few tiles per SM (decode shapes): give every CTA an equal contiguous range
  // of k-slices (tiles split along K add into the same fp32 owner tile).
  // Otherwise: whole tiles, strided over a persistent grid.
  int grid;
  const int sm = (opts && opts->num_ctas > 0) ? opts->num_ctas : dev.sm_count;
  if (p.num_units < 4 * sm) {
    p.stream_k = 1;
    long long per = p.total_ksteps / sm;
    grid = per >= 4 ? sm : static_cast<int>((p.total_ksteps + 3) / 4);
    if (grid < 1) grid = 1;
  } else {
    p.stream_k = 0;
    grid = grid_size(dev, opts, p.num_units);
  }
  int tg = (opts && opts->tiles_per_group > 0) ? opts->tiles_per_group : grid;
  p.tiles_per_group = tg < tiles ? tg : tiles;
  return launch_dt<MODE_REDUCE>(dtype, p, grid, s);
}
