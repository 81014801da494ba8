// Host-side helpers shared by the C-ABI entry points: device checks, tensor
// map encoding, argument validation and the per-call launch bookkeeping.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <array>

#include "../../include/flux_gb300.h"

namespace flux {

constexpr size_t WS_HEADER = 256;  // status header at the start of every workspace
constexpr size_t WS_ALIGN = 256;
// Dynamic schedule of the dense kernels: at most this many regions of 4 CTAs.
constexpr int MAX_REGIONS = 64;

struct DeviceInfo {
  int device;
  int sm_count;
  int cc_major, cc_minor;
  size_t max_smem_optin;
};

// Current device's properties (cached); FLUX_ERR_NO_DEVICE if it has no tcgen05.
flux_status_t current_device(DeviceInfo* info);

// Remember a failing cudaError_t for flux_last_cuda_error() and return FLUX_ERR_CUDA.
flux_status_t cuda_fail(cudaError_t e);

// Fresh per-call id (never 0) written into the abort word if the call aborts.
uint32_t next_seq();

// 2-D row-major tensor [outer x inner] of 16-bit elements with 128-byte swizzle.
flux_status_t encode_2d(CUtensorMap* map, flux_dtype_t dt, const void* base, uint64_t inner,
                        uint64_t outer, uint64_t row_pitch_bytes, uint32_t box_inner,
                        uint32_t box_outer);

// 2-D row-major fp32 tensor with 128-byte swizzle (the accumulation rows of the
// reduce epilogue).
flux_status_t encode_2d_f32(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                            uint64_t row_pitch_bytes, uint32_t box_inner, uint32_t box_outer);

// 3-D row-major tensor [d2 x d1 x d0] of 16-bit elements with 128-byte swizzle.
flux_status_t encode_3d(CUtensorMap* map, flux_dtype_t dt, const void* base, uint64_t d0,
                        uint64_t d1, uint64_t d2, uint32_t box0, uint32_t box1);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Validate a workspace pointer and size.
flux_status_t check_workspace(const void* ws, size_t have, size_t need);

// Default timeout when opts is NULL or timeout_ns == 0.
constexpr uint64_t DEFAULT_TIMEOUT_NS = 2000000000ull;

// Launch options recorded by flux_tune_* for one problem (this device, op,
// dtype and up to eight sizes); false if that problem was never tuned.
bool tuned_opts(flux_op_t op, const std::array<int, 8>& dims, flux_dtype_t dt, flux_opts_t* out);

// Whether flux_gemm_rs takes its stream-K form (single CTAs, k-slices split
// evenly over the grid) for this problem on a GPU with `sm` SMs.
bool rs_uses_stream_k(int R, int M, int N, int sm, bool deterministic);

}  // namespace flux
