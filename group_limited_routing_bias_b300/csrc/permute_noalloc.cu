// moe_permute_noalloc: the dispatch step for callers that cannot allocate
// device memory, neither through cudaMalloc nor through a workspace they own.
//
// Who needs this: code that runs as a plug-in inside a host framework which
// owns all device memory and hands the plug-in only its input and output
// tensors, and serving loops that forbid any allocation after start-up
// (cudaMalloc can synchronise the device and stall every stream).
//
// The scratch that moe_permute takes from the caller's workspace (per-chunk
// expert counts and bases, plus a status word) lives here in one file-scope
// device array instead.  Every GPU that loads this library holds the array
// until the process exits.
#include <mutex>

#include "moe_internal.cuh"

namespace beam {
namespace {

constexpr size_t kNoAllocScratchBytes = 1u << 20;  // 1 MiB
static __device__ __align__(256) unsigned char g_permute_scratch[kNoAllocScratchBytes];

// Device address of g_permute_scratch, looked up once per device.
void *scratch_address(moe_status *st) {
  static std::mutex mu;
  static void *addr[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    *st = MOE_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_permute_scratch) != cudaSuccess || !p) {
      *st = MOE_ERR_CUDA;
      return nullptr;
    }
    addr[dev] = p;
  }
  *st = MOE_OK;
  return addr[dev];
}

}  // namespace
}  // namespace beam

using namespace beam;

namespace {
constexpr size_t kNoAllocHeaderBytes = 256;  // status word, then the tables
}

extern "C" moe_status moe_permute_noalloc(const moe_dims *dims, const int32_t *topk_idx,
                                          const void *x, void *x_perm, int32_t *expert_offsets,
                                          int32_t *slot_of, int32_t *row_src,
                                          moe_stream_t stream) {
  moe_status st = moe_check_dims(dims);
  if (st != MOE_OK) return st;
  if (dims->T == 0) return MOE_OK;
  for (const void *p : {(const void *)topk_idx, x, (const void *)x_perm,
                        (const void *)expert_offsets, (const void *)slot_of,
                        (const void *)row_src})
    if (!p || (reinterpret_cast<uintptr_t>(p) & 15u)) return MOE_ERR_INVALID_ARG;
  const size_t Tk = (size_t)dims->T * dims->top_k;
  const size_t nchunks = std::max<size_t>(1, (Tk + kPermuteChunk - 1) / kPermuteChunk);
  const size_t table = ((nchunks * dims->E * sizeof(int32_t)) + 255) & ~(size_t)255;
  if (kNoAllocHeaderBytes + 2 * table > kNoAllocScratchBytes) return MOE_ERR_UNSUPPORTED;
  char *base = static_cast<char *>(scratch_address(&st));
  if (st != MOE_OK) return st;
  // Every word of the counts and bases tables is written before it is read
  // within one call, so nothing is cleared between calls.
  uint32_t *status = reinterpret_cast<uint32_t *>(base);
  int32_t *counts = reinterpret_cast<int32_t *>(base + kNoAllocHeaderBytes);
  int32_t *bases = reinterpret_cast<int32_t *>(base + kNoAllocHeaderBytes + table);
  return launch_permute(*dims, topk_idx, x, x_perm, expert_offsets, slot_of, row_src, counts, bases,
                        status, reinterpret_cast<cudaStream_t>(stream));
}
