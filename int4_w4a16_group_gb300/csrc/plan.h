// Host-side launch planning shared by the streaming kernels: per-device occupancy data of a
// kernel (resident CTAs per SM, resident clusters per cluster size) and the split over K that
// fills the GPU's CTA slots best.
#pragma once
#include <cuda_runtime.h>

#include "internal.h"

namespace w4a16 {

constexpr int kMaxCluster = 16;

struct LaunchData {
  int occ;                             // resident CTAs per SM
  int max_clusters[kMaxCluster + 1];   // resident clusters per cluster size
};
using LaunchCache = PerDeviceOnce<LaunchData>;

template <typename Kern>
cudaError_t launch_data(Kern kern, int smem, int threads, LaunchCache& cache,
                        const DeviceInfo& di, const LaunchData** out) {
  return cache.get(di.device, [&](LaunchData& d) {
    cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (r != cudaSuccess) return r;
    r = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (r != cudaSuccess) return r;
    int occ = 0;
    r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, threads, smem);
    if (r != cudaSuccess) return r;
    d.occ = occ < 1 ? 1 : occ;
    for (int ck = 1; ck <= kMaxCluster; ++ck) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(1, ck, 1);
      cfg.blockDim = dim3(threads, 1, 1);
      cfg.dynamicSmemBytes = smem;
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeClusterDimension;
      at[0].val.clusterDim.x = 1;
      at[0].val.clusterDim.y = ck;
      at[0].val.clusterDim.z = 1;
      cfg.attrs = at;
      cfg.numAttrs = 1;
      int nc = 0;
      if (cudaOccupancyMaxActiveClusters(&nc, kern, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        nc = 0;
      }
      d.max_clusters[ck] = nc;
    }
    return cudaSuccess;
  }, out);
}

// Split over K for `units` clusters (column tiles x row slices): the cluster size whose waves of
// resident clusters fill the GPU's CTA slots best, each rank keeping at least two stages. *eff
// receives the filled fraction of the slots over those waves.
inline int plan_split(const LaunchData& ld, long long units, int stages, const DeviceInfo& di,
                      double* eff) {
  const double slots = (double)di.sm_count * ld.occ;
  int CK = 1;
  double best = -1.0;
  for (int ck = 1; ck <= kMaxCluster; ++ck) {
    if (ck > 1 && stages / ck < 2) break;
    const int nc = ld.max_clusters[ck];
    if (nc <= 0) continue;
    const long long waves = (units + nc - 1) / nc;
    const double e = (double)units * ck / ((double)waves * slots);
    if (e > best * 1.02) {
      best = e;
      CK = ck;
    }
  }
  if (eff) *eff = best;
  return CK;
}

}  // namespace w4a16
