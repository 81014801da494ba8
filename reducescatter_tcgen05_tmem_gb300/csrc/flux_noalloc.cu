// GEMM + ReduceScatter for callers that cannot provide a workspace.
//
// Some callers have no way to allocate device memory for us: plugin hosts and
// inference runtimes that fix their device-memory budget at start-up and refuse
// allocations once requests are being served (an allocation there can stall or
// fail in the middle of a request), and thin wrappers that have no allocator of
// their own to call.  This entry point serves them with a scratch buffer that
// is part of the library image itself: a file-scope __device__ array that every
// GPU which loads the library holds until the process exits.
//
// Limits and rules of use:
//   * The scratch is FLUX_NOALLOC_SCRATCH_BYTES (16 MiB).  A problem whose
//     GEMM + ReduceScatter workspace (flux_workspace_size(FLUX_OP_GEMM_RS, ...))
//     is larger is rejected with FLUX_ERR_WORKSPACE before anything is launched.
//   * The first call on a device looks up the device address of the array
//     (with that device current) and caches it; make that first call before
//     any stream capture begins.
//   * Every call on a device shares the one array, and the array keeps what
//     the last call left in it.  Each call therefore zeroes the part it uses
//     (an asynchronous memset on `stream`) before the kernel runs.  Calls that
//     overlap on the GPU (different streams without ordering between them)
//     race on the array and give wrong results: order them.
//   * Nothing here calls cudaMalloc, cudaFree or any other allocating routine.
#include <mutex>

#include "flux_host.h"

namespace flux {
namespace {

constexpr size_t kScratchBytes = FLUX_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// The scratch itself.  In host code this name is only a host-side stand-in for
// the symbol, never a device address: the address comes from
// cudaGetSymbolAddress below.
__device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

void* g_scratch_ptr[kMaxDevices];
bool g_scratch_ready[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of the scratch on the current device (looked up once per device).
flux_status_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return FLUX_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ready[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e);
    g_scratch_ptr[dev] = p;
    g_scratch_ready[dev] = true;
  }
  *out = g_scratch_ptr[dev];
  return FLUX_OK;
}

}  // namespace
}  // namespace flux

using namespace flux;

extern "C" flux_status_t flux_gemm_rs_noalloc(int R, int M, int N, int K, flux_dtype_t dtype,
                                              const void* const* a_shards,
                                              const void* const* b_shards, void* const* out,
                                              const flux_opts_t* opts, void* stream) {
  const size_t need = flux_workspace_size(FLUX_OP_GEMM_RS, R, M, N, K);
  if (need == 0) return FLUX_ERR_INVALID_ARG;
  if (need > kScratchBytes) return FLUX_ERR_WORKSPACE;
  if (M % R || K % R || a_shards == nullptr || b_shards == nullptr || out == nullptr ||
      (dtype != FLUX_F16 && dtype != FLUX_BF16))
    return FLUX_ERR_INVALID_ARG;
  // Every check flux_gemm_rs makes on the arguments comes first, so that a
  // call that is going to be refused leaves the stream and the shared array
  // alone.
  const int Kr = K / R;
  if (M > 0 && N > 0) {
    for (int r = 0; r < R; ++r) {
      if (a_shards[r] == nullptr || b_shards[r] == nullptr || out[r] == nullptr)
        return FLUX_ERR_INVALID_ARG;
      if (!aligned16(a_shards[r]) || !aligned16(b_shards[r]) || !aligned16(out[r]))
        return FLUX_ERR_UNSUPPORTED;
    }
    if (Kr % 8 || N % 8) return FLUX_ERR_UNSUPPORTED;
  }
  DeviceInfo dev;
  flux_status_t st = current_device(&dev);
  if (st != FLUX_OK) return st;
  void* scratch = nullptr;
  if ((st = scratch_address(&scratch)) != FLUX_OK) return st;
  // Nothing to reduce (empty output, or a zero-length K that only zero-fills
  // the outputs): the scratch is not used, so it is not cleared either.
  if (M > 0 && N > 0 && Kr > 0) {
    // the header, arrival counters and fp32 accumulators must start at zero
    cudaError_t e = cudaMemsetAsync(scratch, 0, need, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return flux_gemm_rs(R, M, N, K, dtype, a_shards, b_shards, out, scratch, need, opts, stream);
}
