// Dispatch of the Beam MoE block: the T*k (token, slot) entries are counted
// per expert, offsets are the exclusive scan of the counts, and every entry
// gets a row in expert-major order that keeps ascending entry order inside an
// expert (a stable counting sort).  Then the x rows are gathered into that
// order so each expert's rows are contiguous for the grouped GEMMs.
//
//   permute_small_kernel   one CTA, when T*k fits one chunk: all three steps below
//   permute_count_kernel   one CTA per chunk of 4096 entries: histogram
//   permute_scan_kernel    one CTA: per-chunk bases and expert offsets
//   permute_scatter_kernel one CTA per chunk: warp-ordered ranks -> slots
//   permute_scatter_rows_kernel  all SMs: each token's x row to its k slots (16-byte
//                          vectors, one warp per 2 KB segment of a row)
//   permute_scatter_rows_scaled_kernel  the same as f16 scaled per token (one
//                          warp per token), for the token-major packed GEMMs
#include <cuda_fp16.h>

#include "moe_internal.cuh"
#include "rowscale.cuh"

namespace beam {

namespace {

constexpr int kChunkThreads = 1024;
constexpr int kEntriesPerWarp = kPermuteChunk / (kChunkThreads / 32);  // 128

__global__ void __launch_bounds__(kChunkThreads)
    permute_count_kernel(const int32_t *__restrict__ idx, int Tk, int E, int32_t *__restrict__ counts,
                         uint32_t *status) {
  extern __shared__ int cnt[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  const int base = blockIdx.x * kPermuteChunk;
  bool bad = false;
  for (int j = threadIdx.x; j < kPermuteChunk; j += blockDim.x) {
    const int n = base + j;
    if (n >= Tk) break;
    const int e = idx[n];
    if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);
    else bad = true;
  }
  if (bad) atomicOr(status, (uint32_t)MOE_DEV_BAD_INDEX);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) counts[(size_t)blockIdx.x * E + e] = cnt[e];
}

// Exclusive block scan of one value per thread (blockDim.x <= 1024).
__device__ int block_exclusive_scan(int v, int *warp_sums) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    int s = lane < nw ? warp_sums[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, s, off);
      if (lane >= off) s += o;
    }
    if (lane < nw) warp_sums[lane] = s;  // inclusive sums of warps
  }
  __syncthreads();
  const int before = warp == 0 ? 0 : warp_sums[warp - 1];
  return before + incl - v;
}

__global__ void __launch_bounds__(256)
    permute_scan_kernel(const int32_t *__restrict__ counts, int nchunks, int E,
                        int32_t *__restrict__ bases, int32_t *__restrict__ offsets) {
  __shared__ int warp_sums[32];
  const int e = threadIdx.x;
  int total = 0;
  if (e < E)
    for (int c = 0; c < nchunks; ++c) {
      const int v = counts[(size_t)c * E + e];
      bases[(size_t)c * E + e] = total;
      total += v;
    }
  const int start = block_exclusive_scan(e < E ? total : 0, warp_sums);
  if (e < E) {
    for (int c = 0; c < nchunks; ++c) bases[(size_t)c * E + e] += start;
    offsets[e] = start;
    if (e == E - 1) offsets[E] = start + total;
  }
}

__global__ void __launch_bounds__(kChunkThreads)
    permute_scatter_kernel(const int32_t *__restrict__ idx, int Tk, int E,
                           const int32_t *__restrict__ bases, int32_t *__restrict__ slot_of,
                           int32_t *__restrict__ row_src) {
  extern __shared__ int wcnt[];  // [32 warps][E]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < 32 * E; i += blockDim.x) wcnt[i] = 0;
  __syncthreads();
  const int wbase = blockIdx.x * kPermuteChunk + warp * kEntriesPerWarp;
  int *mine = wcnt + warp * E;
  // pass A: per-warp counts, in entry order
  for (int sub = 0; sub < kEntriesPerWarp; sub += 32) {
    const int n = wbase + sub + lane;
    int e = n < Tk ? idx[n] : -1;
    if (e < 0 || e >= E) e = -1;
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && lane == __ffs(peers) - 1) mine[e] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  // per expert: the chunk's base plus the counts of the warps before
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = bases[(size_t)blockIdx.x * E + e];
    for (int w = 0; w < 32; ++w) {
      const int c = wcnt[w * E + e];
      wcnt[w * E + e] = run;
      run += c;
    }
  }
  __syncthreads();
  // pass B: slot = running base + rank among equal experts in this group of 32
  const uint32_t lt = (1u << lane) - 1u;
  for (int sub = 0; sub < kEntriesPerWarp; sub += 32) {
    const int n = wbase + sub + lane;
    int e = n < Tk ? idx[n] : -1;
    if (e < 0 || e >= E) e = -1;
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    int slot = -1;
    if (e >= 0) slot = mine[e] + __popc(peers & lt);
    __syncwarp();
    if (e >= 0 && lane == __ffs(peers) - 1) mine[e] += __popc(peers);
    __syncwarp();
    if (n < Tk) {
      slot_of[n] = slot;
      if (slot >= 0) row_src[slot] = n;
    }
  }
}

// All of count, scan and scatter in one CTA, for batches of at most one chunk
// (T*k <= 4096 entries, e.g. decode): per-warp counts in entry order, per
// expert totals and their exclusive scan, then the same warp-ordered slots as
// the multi-CTA path.
__global__ void __launch_bounds__(kChunkThreads)
    permute_small_kernel(const int32_t *__restrict__ idx, int Tk, int E,
                         int32_t *__restrict__ offsets, int32_t *__restrict__ slot_of,
                         int32_t *__restrict__ row_src, uint32_t *status) {
  extern __shared__ int wcnt[];  // [32 warps][E]
  __shared__ int warp_sums[32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < 32 * E; i += blockDim.x) wcnt[i] = 0;
  __syncthreads();
  const int wbase = warp * kEntriesPerWarp;
  int *mine = wcnt + warp * E;
  bool bad = false;
  for (int sub = 0; sub < kEntriesPerWarp; sub += 32) {
    const int n = wbase + sub + lane;
    int e = n < Tk ? idx[n] : -1;
    if (n < Tk && (e < 0 || e >= E)) bad = true;
    if (e < 0 || e >= E) e = -1;
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && lane == __ffs(peers) - 1) mine[e] += __popc(peers);
    __syncwarp();
  }
  if (bad) atomicOr(status, (uint32_t)MOE_DEV_BAD_INDEX);
  __syncthreads();
  // per expert: total over warps, then the exclusive scan over experts
  int total = 0;
  if (threadIdx.x < E)
    for (int w = 0; w < 32; ++w) total += wcnt[w * E + threadIdx.x];
  const int start = block_exclusive_scan(threadIdx.x < E ? total : 0, warp_sums);
  if (threadIdx.x < E) {
    int run = start;
    for (int w = 0; w < 32; ++w) {
      const int c = wcnt[w * E + threadIdx.x];
      wcnt[w * E + threadIdx.x] = run;
      run += c;
    }
    offsets[threadIdx.x] = start;
    if (threadIdx.x == E - 1) offsets[E] = start + total;
  }
  __syncthreads();
  const uint32_t lt = (1u << lane) - 1u;
  for (int sub = 0; sub < kEntriesPerWarp; sub += 32) {
    const int n = wbase + sub + lane;
    int e = n < Tk ? idx[n] : -1;
    if (e < 0 || e >= E) e = -1;
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    int slot = -1;
    if (e >= 0) slot = mine[e] + __popc(peers & lt);
    __syncwarp();
    if (e >= 0 && lane == __ffs(peers) - 1) mine[e] += __popc(peers);
    __syncwarp();
    if (n < Tk) {
      slot_of[n] = slot;
      if (slot >= 0) row_src[slot] = n;
    }
  }
}

// Copies x rows into permuted order, in token order: token t's row is read
// once and written to every permuted row that holds one of its entries
// (slot_of[t*k + j]; dropped entries have slot -1).  Reading x once matters
// when x is larger than L2 (prefill: an expert-ordered gather would fetch each
// row from DRAM up to k times).  One warp per (token, 128-vector segment of its row): each lane loads its
// four 16-byte vectors of the segment first, then stores them to the token's
// k slots, so a warp has all its loads in flight at once and a small batch
// still spreads over many warps.
constexpr int kScatterSeg = 128;  // 16-byte vectors per warp task (4 per lane)

__global__ void __launch_bounds__(256)
    permute_scatter_rows_kernel(const uint4 *__restrict__ x, const int32_t *__restrict__ slot_of,
                                int T, int top_k, int vec_per_row, uint4 *__restrict__ x_perm) {
  const int lane = threadIdx.x & 31;
  const int segs = (vec_per_row + kScatterSeg - 1) / kScatterSeg;
  const long ntasks = (long)T * segs;
  const long nwarps = (long)gridDim.x * (blockDim.x >> 5);
  for (long w = (long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); w < ntasks; w += nwarps) {
    const int t = (int)(w / segs);
    const int v0 = (int)(w - (long)t * segs) * kScatterSeg + lane;
    const int my_slot = lane < top_k ? __ldg(slot_of + (size_t)t * top_k + lane) : -1;
    const uint4 *src = x + (size_t)t * vec_per_row;
    uint4 q[kScatterSeg / 32];
#pragma unroll
    for (int i = 0; i < kScatterSeg / 32; ++i) {
      const int v = v0 + 32 * i;
      q[i] = v < vec_per_row ? src[v] : make_uint4(0u, 0u, 0u, 0u);
    }
    for (int j = 0; j < top_k; ++j) {
      const int slot = __shfl_sync(0xffffffffu, my_slot, j);  // the same in every lane
      if (slot < 0) continue;
      uint4 *dst = x_perm + (size_t)slot * vec_per_row;
#pragma unroll
      for (int i = 0; i < kScatterSeg / 32; ++i)
        if (v0 + 32 * i < vec_per_row) dst[v0 + 32 * i] = q[i];
    }
  }
}

// The same copy as f16 scaled by a power of two per token (rowscale.cuh):
// one warp per token finds the row's largest magnitude, then converts and
// writes the row to the token's slots; lane j records xscale and clears hmax
// of slot j.  The second pass reads the row again, from L2.
__global__ void __launch_bounds__(256)
    permute_scatter_rows_scaled_kernel(const uint4 *__restrict__ x,
                                       const int32_t *__restrict__ slot_of, int T, int top_k,
                                       int vec_per_row, uint4 *__restrict__ x_perm, float *xscale,
                                       uint32_t *hmax) {
  const int lane = threadIdx.x & 31;
  const long nwarps = (long)gridDim.x * (blockDim.x >> 5);
  for (long t = (long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < T; t += nwarps) {
    const int my_slot = lane < top_k ? __ldg(slot_of + (size_t)t * top_k + lane) : -1;
    const uint4 *src = x + (size_t)t * vec_per_row;
    uint32_t m = 0;
#pragma unroll 8
    for (int v = lane; v < vec_per_row; v += 32) m = bf16x8_absmax_bits(src[v], m);
    m = max(m & 0xFFFFu, m >> 16);
    m = __reduce_max_sync(0xffffffffu, m);
    const int sx = row_scale_exp(m >> 7);
    const float sc = ldexpf(1.0f, sx);
    for (int v0 = 0; v0 < vec_per_row; v0 += 32 * 4) {
      uint4 q[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int v = v0 + 32 * i + lane;
        q[i] = v < vec_per_row ? bf16x8_to_f16x8_scaled(src[v], sc) : make_uint4(0u, 0u, 0u, 0u);
      }
      for (int j = 0; j < top_k; ++j) {
        const int slot = __shfl_sync(0xffffffffu, my_slot, j);  // the same in every lane
        if (slot < 0) continue;
        uint4 *dst = x_perm + (size_t)slot * vec_per_row;
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (v0 + 32 * i + lane < vec_per_row) dst[v0 + 32 * i + lane] = q[i];
      }
    }
    if (my_slot >= 0) {
      xscale[my_slot] = ldexpf(1.0f, -sx);
      hmax[my_slot] = 0u;
    }
  }
}

}  // namespace

moe_status launch_permute(const moe_dims &d, const int32_t *topk_idx, const void *x, void *x_perm,
                          int32_t *expert_offsets, int32_t *slot_of, int32_t *row_src,
                          int32_t *counts, int32_t *bases, uint32_t *status, cudaStream_t stream,
                          GatherMode gather, float *xscale, uint32_t *hmax) {
  const int Tk = d.T * d.top_k;
  const int nchunks = std::max(1, (Tk + kPermuteChunk - 1) / kPermuteChunk);
  const int scatter_smem = 32 * d.E * 4;  // at most 32 KB (E <= 256): no opt-in needed
  if (nchunks == 1) {
    permute_small_kernel<<<1, kChunkThreads, scatter_smem, stream>>>(topk_idx, Tk, d.E,
                                                                     expert_offsets, slot_of,
                                                                     row_src, status);
  } else {
    permute_count_kernel<<<nchunks, kChunkThreads, d.E * 4, stream>>>(topk_idx, Tk, d.E, counts,
                                                                       status);
    permute_scan_kernel<<<1, 256, 0, stream>>>(counts, nchunks, d.E, bases, expert_offsets);
    permute_scatter_kernel<<<nchunks, kChunkThreads, scatter_smem, stream>>>(
        topk_idx, Tk, d.E, bases, slot_of, row_src);
  }
  if (Tk > 0 && gather == kGatherF16Scaled) {
    const int blocks = (int)std::max<long>(1, std::min<long>(((long)d.T + 7) / 8, device_sm_count() * 8));
    permute_scatter_rows_scaled_kernel<<<blocks, 256, 0, stream>>>(
        static_cast<const uint4 *>(x), slot_of, d.T, d.top_k, d.H / 8, static_cast<uint4 *>(x_perm),
        xscale, hmax);
  } else if (Tk > 0 && gather == kGatherBf16) {
    const long tasks = (long)d.T * ((d.H / 8 + kScatterSeg - 1) / kScatterSeg);
    const int blocks = (int)std::max<long>(1, std::min<long>((tasks + 7) / 8, device_sm_count() * 8));
    permute_scatter_rows_kernel<<<blocks, 256, 0, stream>>>(
        static_cast<const uint4 *>(x), slot_of, d.T, d.top_k, d.H / 8,
        static_cast<uint4 *>(x_perm));
  }
  return cudaPeekAtLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace beam
