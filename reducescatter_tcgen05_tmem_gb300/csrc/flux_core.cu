// Housekeeping entry points of the C ABI and the host helpers of flux_host.h.
#include <atomic>
#include <mutex>

#include <cudaTypedefs.h>

#include "flux_host.h"

#ifndef FLUX_CHECKS
#define FLUX_CHECKS 0
#endif

namespace flux {

namespace {
thread_local int g_last_cuda_error = 0;
std::atomic<uint32_t> g_seq{0};

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_err = cudaSuccess;

constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
bool g_dev_ok[kMaxDevices];
std::mutex g_dev_mu;

CUtensorMapDataType map_type(flux_dtype_t dt) {
  return dt == FLUX_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
}

flux_status_t encoder(PFN_cuTensorMapEncodeTiled_v12000* fn) {
  std::call_once(g_encode_once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    g_encode_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                                    cudaEnableDefault, &q);
    if (g_encode_err == cudaSuccess && q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  if (g_encode == nullptr) return cuda_fail(g_encode_err != cudaSuccess ? g_encode_err : cudaErrorNotSupported);
  *fn = g_encode;
  return FLUX_OK;
}
}  // namespace

flux_status_t cuda_fail(cudaError_t e) {
  g_last_cuda_error = static_cast<int>(e);
  return FLUX_ERR_CUDA;
}

uint32_t next_seq() {
  uint32_t v;
  do { v = g_seq.fetch_add(1) + 1; } while (v == 0);
  return v;
}

flux_status_t current_device(DeviceInfo* info) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return FLUX_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (!g_dev_ok[dev]) {
    DeviceInfo d{};
    d.device = dev;
    int v = 0;
    if ((e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
      return cuda_fail(e);
    d.max_smem_optin = static_cast<size_t>(v);
    g_dev[dev] = d;
    g_dev_ok[dev] = true;
  }
  *info = g_dev[dev];
  // The kernels are built for sm_103a only (tcgen05 / TMEM / TMA).
  if (info->cc_major != 10 || info->cc_minor != 3) return FLUX_ERR_NO_DEVICE;
  return FLUX_OK;
}

flux_status_t encode_2d(CUtensorMap* map, flux_dtype_t dt, const void* base, uint64_t inner,
                        uint64_t outer, uint64_t row_pitch_bytes, uint32_t box_inner,
                        uint32_t box_outer) {
  PFN_cuTensorMapEncodeTiled_v12000 fn;
  flux_status_t st = encoder(&fn);
  if (st != FLUX_OK) return st;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_pitch_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(map, map_type(dt), 2, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
  return FLUX_OK;
}

flux_status_t encode_2d_f32(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                            uint64_t row_pitch_bytes, uint32_t box_inner, uint32_t box_outer) {
  PFN_cuTensorMapEncodeTiled_v12000 fn;
  flux_status_t st = encoder(&fn);
  if (st != FLUX_OK) return st;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_pitch_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box,
                  es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
  return FLUX_OK;
}

flux_status_t encode_3d(CUtensorMap* map, flux_dtype_t dt, const void* base, uint64_t d0,
                        uint64_t d1, uint64_t d2, uint32_t box0, uint32_t box1) {
  PFN_cuTensorMapEncodeTiled_v12000 fn;
  flux_status_t st = encoder(&fn);
  if (st != FLUX_OK) return st;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
  cuuint32_t box[3] = {box0, box1, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(map, map_type(dt), 3, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
  return FLUX_OK;
}

flux_status_t check_workspace(const void* ws, size_t have, size_t need) {
  if (ws == nullptr) return FLUX_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) % WS_ALIGN) != 0) return FLUX_ERR_WORKSPACE;
  if (have < need) return FLUX_ERR_WORKSPACE;
  return FLUX_OK;
}

}  // namespace flux

using namespace flux;

extern "C" int flux_version(void) { return 200; }

extern "C" int flux_checks_enabled(void) { return FLUX_CHECKS ? 1 : 0; }

extern "C" size_t flux_opts_size(void) { return sizeof(flux_opts_t); }

extern "C" const char* flux_status_string(flux_status_t s) {
  switch (s) {
    case FLUX_OK: return "FLUX_OK";
    case FLUX_ERR_INVALID_ARG: return "FLUX_ERR_INVALID_ARG";
    case FLUX_ERR_UNSUPPORTED: return "FLUX_ERR_UNSUPPORTED";
    case FLUX_ERR_WORKSPACE: return "FLUX_ERR_WORKSPACE";
    case FLUX_ERR_CUDA: return "FLUX_ERR_CUDA";
    case FLUX_ERR_TIMEOUT: return "FLUX_ERR_TIMEOUT";
    case FLUX_ERR_NO_DEVICE: return "FLUX_ERR_NO_DEVICE";
  }
  return "FLUX_ERR_UNKNOWN";
}

extern "C" int flux_last_cuda_error(void) { return g_last_cuda_error; }

extern "C" flux_status_t flux_workspace_init(void* workspace, size_t bytes, void* stream) {
  if (workspace == nullptr || bytes < WS_HEADER) return FLUX_ERR_WORKSPACE;
  cudaError_t e = cudaMemsetAsync(workspace, 0, bytes, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FLUX_OK : cuda_fail(e);
}

extern "C" flux_status_t flux_get_status(void* workspace, size_t bytes, void* stream,
                                         flux_device_report_t* report) {
  if (workspace == nullptr || bytes < WS_HEADER) return FLUX_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e);
  uint32_t h[4] = {0, 0, 0, 0};
  e = cudaMemcpy(h, workspace, sizeof(h), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e);
  if (report != nullptr) {
    report->status = h[0];
    report->where = h[1];
    report->arg0 = h[2];
    report->arg1 = h[3];
  }
  if (h[0] != 0) {
    // the failed call left partial sums and counters behind: start clean
    e = cudaMemsetAsync(workspace, 0, bytes, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e);
    return static_cast<flux_status_t>(h[0]);
  }
  return FLUX_OK;
}
