// MMA-tiled layout of bf16 expert weights (moe_pack_bf16): a matrix
// [E, N, K] (N output rows, K contiguous) becomes tiles of 128 rows x 64 k,
// each stored as the 16 KB image the expert GEMMs keep in shared memory
// (128-byte rows in 8-row groups, 16-byte chunk c of row r at position
// c XOR (r mod 8)), ordered expert, then 128-row block, then k block.  A tile
// then arrives with one contiguous bulk copy instead of 128 row requests, and
// a CTA streaming one 128-row block over K reads a contiguous region.
#include "moe_internal.cuh"

namespace beam {

namespace {

__global__ void __launch_bounds__(256)
    pack_bf16_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst, int N, int K,
                     size_t nchunks) {
  const int kc_per_row = K / 8;  // 16-byte chunks per row
  const int ktiles = K / 64;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < nchunks;
       i += (size_t)gridDim.x * blockDim.x) {
    const size_t row = i / kc_per_row;  // e * N + n
    const int kc = (int)(i - row * kc_per_row);
    const size_t rblk = row / 128;  // (e * N + n) / 128 = e * N/128 + n / 128, N % 128 == 0
    const int r = (int)(row % 128);
    const int kt = kc / 8, c = kc % 8;
    const size_t tile = rblk * ktiles + kt;
    dst[tile * 1024 + (r / 8) * 64 + (r % 8) * 8 + (c ^ (r % 8))] = src[i];
  }
}

}  // namespace

moe_status launch_pack_bf16(int E, int N, int K, const void *src, void *dst, cudaStream_t stream) {
  const size_t nchunks = (size_t)E * N * (K / 8);
  if (nchunks == 0) return MOE_OK;
  const int blocks = (int)std::min<size_t>((nchunks + 255) / 256, (size_t)device_sm_count() * 16);
  pack_bf16_kernel<<<blocks, 256, 0, stream>>>(static_cast<const uint4 *>(src),
                                               static_cast<uint4 *>(dst), N, K, nchunks);
  return cudaPeekAtLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace beam
