// Host-side launch of one instantiation of the fused kernel: sets the shared
// memory attribute once, sizes CTA-pair grids to the clusters that fit at
// once, and launches on the caller's stream.
#pragma once

#include <cstdio>
#include <cstdlib>
#include <mutex>

#include "flux_host.h"
#include "flux_kernels.cuh"

namespace flux {

// FLUX_DEBUG=1 in the environment prints each launch's configuration to stderr.
inline bool debug_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("FLUX_DEBUG");
    return v != nullptr && v[0] != '\0' && v[0] != '0';
  }();
  return on;
}

template <int MODE, int DT, int CL>
struct Launcher {
  // Largest grid (CTAs) that is resident at once; 0 on error.
  static int max_ctas(const DeviceInfo& dev) {
    static std::once_flag once;
    static cudaError_t err = cudaSuccess;
    static int ctas = 0;
    std::call_once(once, [&dev] {
      err = cudaFuncSetAttribute(fused_gemm_kernel<MODE, DT, CL>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
      if (err != cudaSuccess) return;
      if (CL == 1) {
        ctas = dev.sm_count;
        return;
      }
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(CL * (dev.sm_count / CL), 1, 1);
      cfg.blockDim = dim3(KernelShape<MODE, DT, CL>::THREADS, 1, 1);
      cfg.dynamicSmemBytes = SMEM_BYTES;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = CL;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int clusters = 0;
      err = cudaOccupancyMaxActiveClusters(&clusters, fused_gemm_kernel<MODE, DT, CL>, &cfg);
      ctas = clusters * CL;
      if (debug_enabled())
        std::fprintf(stderr, "[flux] mode %d dtype %d cluster %d: %d clusters resident at once\n",
                     MODE, DT, CL, clusters);
    });
    if (err != cudaSuccess) {
      cuda_fail(err);
      return 0;
    }
    return ctas;
  }

  // Dynamic schedule (dense CL = 4 kernels): the grid when clusters are CTA
  // pairs with CL as the preferred size, a multiple of CL of at most
  // 4 * MAX_REGIONS CTAs; 0 if this launch form is not available.
  static int max_ctas_dyn(const DeviceInfo& dev) {
    static_assert(CL == 4 || CL == 8, "regions of two or four CTA pairs");
    if (max_ctas(dev) <= 0) return 0;  // sets the shared memory attribute
    static std::once_flag once;
    static int ctas = 0;
    std::call_once(once, [&dev] {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2 * (dev.sm_count / 2), 1, 1);
      cfg.blockDim = dim3(KernelShape<MODE, DT, CL>::THREADS, 1, 1);
      cfg.dynamicSmemBytes = SMEM_BYTES;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int clusters = 0;
      if (cudaOccupancyMaxActiveClusters(&clusters, fused_gemm_kernel<MODE, DT, CL>, &cfg) !=
          cudaSuccess) {
        (void)cudaGetLastError();
        clusters = 0;
      }
      int g = clusters * 2;
      g -= g % CL;
      if (g > CL * MAX_REGIONS) g = CL * MAX_REGIONS;
      ctas = g;
      if (debug_enabled())
        std::fprintf(stderr, "[flux] mode %d dtype %d: %d CTA pairs resident at once (dynamic grid %d)\n",
                     MODE, DT, clusters, g);
    });
    return ctas;
  }

  static flux_status_t launch_dyn(const KParams& p, int grid, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(KernelShape<MODE, DT, CL>::THREADS, 1, 1);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributePreferredClusterDimension;
    attr[1].val.preferredClusterDim.x = CL;
    attr[1].val.preferredClusterDim.y = 1;
    attr[1].val.preferredClusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (debug_enabled())
      std::fprintf(stderr,
                   "[flux] mode %d dtype %d: dynamic schedule, grid %d (pairs, preferred %d), units %d, "
                   "mailbox %d per region, tiles %d x %d, k-slices %d\n",
                   MODE, DT, grid, CL, p.num_units, p.mbox_cap, p.Mt, p.Nt, p.KT);
    cudaError_t e = cudaLaunchKernelEx(&cfg, fused_gemm_kernel<MODE, DT, CL>, p);
    return e == cudaSuccess ? FLUX_OK : cuda_fail(e);
  }

  static flux_status_t launch(const KParams& p, int grid, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(KernelShape<MODE, DT, CL>::THREADS, 1, 1);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = CL > 1 ? 1 : 0;
    if (debug_enabled())
      std::fprintf(stderr,
                   "[flux] mode %d dtype %d cluster %d: grid %d x %d threads, %d B smem, units %d, "
                   "tiles %d x %d, k-slices %d, stream-k %d\n",
                   MODE, DT, CL, grid, KernelShape<MODE, DT, CL>::THREADS, SMEM_BYTES,
                   p.num_units, p.Mt, p.Nt, p.KT, p.stream_k);
    cudaError_t e = cudaLaunchKernelEx(&cfg, fused_gemm_kernel<MODE, DT, CL>, p);
    return e == cudaSuccess ? FLUX_OK : cuda_fail(e);
  }
};

// Grid for `units` work units of CL CTAs each, capped at the resident CTAs
// (or opts->num_ctas); a multiple of CL, at least CL.
template <int MODE, int DT, int CL>
int grid_for(const DeviceInfo& dev, const flux_opts_t* opts, long long units) {
  int cap = Launcher<MODE, DT, CL>::max_ctas(dev);
  if (cap <= 0) return 0;
  if (opts && opts->num_ctas > 0 && opts->num_ctas < cap) cap = opts->num_ctas;
  long long g = units * CL;
  if (g > cap) g = cap;
  g -= g % CL;
  if (g < CL) g = CL;
  return static_cast<int>(g);
}

}  // namespace flux
