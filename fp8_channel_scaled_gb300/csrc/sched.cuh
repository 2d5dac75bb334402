// sched.cuh -- tile order of the persistent tile kernels.
#pragma once

namespace fp8g {

// Grouped rasterisation: tiles are visited in groups of `group_m` consecutive
// M blocks, walking N within a group, so the CTAs resident at one time share
// few x row-blocks and few w column-blocks and re-read them from L2 (the
// grouped tile order of the "Kimi K3 (256k)" page, SM90 WGMMA paragraph).
__device__ __forceinline__ void tile_coords(int t, int num_m, int num_n, int group_m, int& mb,
                                            int& nb) {
  const int per_group = group_m * num_n;
  const int g = t / per_group;
  const int first_m = g * group_m;
  const int gsize = min(num_m - first_m, group_m);
  const int r = t - g * per_group;
  mb = first_m + r % gsize;
  nb = r / gsize;
}

}  // namespace fp8g
