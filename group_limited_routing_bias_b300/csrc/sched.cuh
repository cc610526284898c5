// Tile schedule over experts shared by the persistent expert GEMMs: every
// CTA reads the expert row offsets into shared memory and forms the prefix of
// tiles per expert, so a tile index maps to (expert, feature tile, token tile)
// with a binary search.
#pragma once

#include <cstdint>

namespace beam {

struct TileSched {
  int off[257];  // expert row offsets
  int tp[257];   // prefix of tiles (or token tiles) per expert
};

// Prefix over experts of ceil(rows_e / rows_per_tile) * mult, computed by warp 0.
__device__ __forceinline__ void tile_sched_prologue(const int32_t *offsets, int E, int rows_per_tile,
                                             int mult, TileSched &s) {
  for (int i = threadIdx.x; i <= E; i += blockDim.x) s.off[i] = offsets[i];
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int per = (E + 31) / 32;
    const int e0 = lane * per;
    int local = 0;
    for (int e = e0; e < e0 + per && e < E; ++e)
      local += (s.off[e + 1] - s.off[e] + rows_per_tile - 1) / rows_per_tile * mult;
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - local;
    for (int e = e0; e < e0 + per && e < E; ++e) {
      s.tp[e] = run;
      run += (s.off[e + 1] - s.off[e] + rows_per_tile - 1) / rows_per_tile * mult;
    }
    if (lane == 31) s.tp[E] = incl;
  }
  __syncthreads();
}

__device__ __forceinline__ int tile_sched_expert(const TileSched &s, int E, int v) {
  int lo = 0, hi = E;  // last e with tp[e] <= v
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s.tp[mid] <= v) lo = mid;
    else hi = mid;
  }
  return lo;
}

}  // namespace beam
