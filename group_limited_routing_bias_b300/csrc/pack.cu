// MMA-tiled layout of bf16 expert weights (moe_pack_bf16): a matrix
// [E, N, K] (N output rows, K contiguous) becomes tiles of 128 rows x 64 k,
// each stored as the 16 KB image the expert GEMMs keep in shared memory
// (128-byte rows in 8-row groups, 16-byte chunk c of row r at position
// c XOR (r mod 8)), ordered expert, then 128-row block, then k block.  A tile
// then arrives with one contiguous bulk copy instead of 128 row requests, and
// a CTA streaming one 128-row block over K reads a contiguous region.
//
// The packed formats use the same tile grid and order with plain row-major
// tiles (the converter warps write the swizzled operand image themselves):
//   NVFP4 (moe_pack_nvfp4): 4608 bytes per tile, the 128 rows' 32 code bytes
//     (64 k, two per byte) row after row, then their four e4m3 block scales;
//   FP8 (moe_pack_fp8): 8192 bytes per tile, 64 code bytes per row.
// The row-major packed weights give each 64-wide K slice of a row only 32 or
// 64 contiguous bytes, and streaming them as 128-row boxes of such segments
// leaves the decode GEMMs far below HBM bandwidth.
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

// One thread per (row, k block): 32 code bytes and 4 scale bytes.
__global__ void __launch_bounds__(256)
    pack_nvfp4_kernel(const uint8_t *__restrict__ q, const uint8_t *__restrict__ s,
                      uint8_t *__restrict__ dst, int K, size_t nitems) {
  const int ktiles = K / 64;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < nitems;
       i += (size_t)gridDim.x * blockDim.x) {
    const size_t row = i / ktiles;  // e * N + n
    const int kt = (int)(i - row * ktiles);
    const size_t tile = (row / 128) * ktiles + kt;
    const int r = (int)(row % 128);
    uint8_t *t = dst + tile * 4608;
    const uint4 *src = reinterpret_cast<const uint4 *>(q + row * (K / 2) + kt * 32);
    uint4 *d = reinterpret_cast<uint4 *>(t + r * 32);
    d[0] = src[0];
    d[1] = src[1];
    *reinterpret_cast<uint32_t *>(t + 128 * 32 + r * 4) =
        *reinterpret_cast<const uint32_t *>(s + row * (K / 16) + kt * 4);
  }
}

// One thread per 16-byte chunk of codes.
__global__ void __launch_bounds__(256)
    pack_fp8_kernel(const uint4 *__restrict__ q, uint4 *__restrict__ dst, int K, size_t nchunks) {
  const int kc_per_row = K / 16;
  const int ktiles = K / 64;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < nchunks;
       i += (size_t)gridDim.x * blockDim.x) {
    const size_t row = i / kc_per_row;
    const int kc = (int)(i - row * kc_per_row);
    const int kt = kc / 4, c = kc % 4;
    const size_t tile = (row / 128) * ktiles + kt;
    dst[tile * 512 + (row % 128) * 4 + c] = q[i];
  }
}

int pack_blocks(size_t items) {
  return (int)std::min<size_t>((items + 255) / 256, (size_t)device_sm_count() * 16);
}

}  // namespace

moe_status launch_pack_nvfp4(int E, int N, int K, const uint8_t *q, const uint8_t *s, uint8_t *dst,
                             cudaStream_t stream) {
  const size_t nitems = (size_t)E * N * (K / 64);
  if (nitems == 0) return MOE_OK;
  pack_nvfp4_kernel<<<pack_blocks(nitems), 256, 0, stream>>>(q, s, dst, K, nitems);
  return cudaPeekAtLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status launch_pack_fp8(int E, int N, int K, const uint8_t *q, uint8_t *dst, cudaStream_t stream) {
  const size_t nchunks = (size_t)E * N * (K / 16);
  if (nchunks == 0) return MOE_OK;
  pack_fp8_kernel<<<pack_blocks(nchunks), 256, 0, stream>>>(reinterpret_cast<const uint4 *>(q),
                                                            reinterpret_cast<uint4 *>(dst), K, nchunks);
  return cudaPeekAtLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status launch_pack_bf16(int E, int N, int K, const void *src, void *dst, cudaStream_t stream) {
  const size_t nchunks = (size_t)E * N * (K / 8);
  if (nchunks == 0) return MOE_OK;
  const int blocks = (int)std::min<size_t>((nchunks + 255) / 256, (size_t)device_sm_count() * 16);
  pack_bf16_kernel<<<blocks, 256, 0, stream>>>(static_cast<const uint4 *>(src),
                                               static_cast<uint4 *>(dst), N, K, nchunks);
  return cudaPeekAtLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace beam
