// Auxiliary-loss-free balancing of the Beam MoE router: after a batch is
// routed, each expert's selection bias moves one step against its load
// ("Beam 1.0": DeepSeek-V3's auxiliary-loss-free balancing with a cosine decay
// of the expert-bias updates).  Readings (the page gives no formula):
//   load_e  = entries (token, slot) routed to expert e in the batch
//   gamma_t = gamma_max * (1 + cos(pi * step / total_steps)) / 2, step clamped
//   bias[e] += gamma_t * sign(T*k/E - load_e)
// One CTA: a shared-memory histogram of topk_idx, then one thread per expert.
// Integer counts make the result independent of the atomics' order.
#include <cmath>

#include "moe_internal.cuh"

namespace beam {
namespace {

__global__ void __launch_bounds__(1024)
    bias_update_kernel(const int32_t *__restrict__ idx, long n, int E, double mean, float gamma,
                       float *__restrict__ bias) {
  __shared__ int load[256];
  for (int e = threadIdx.x; e < E; e += blockDim.x) load[e] = 0;
  __syncthreads();
  for (long i = threadIdx.x; i < n; i += blockDim.x) {
    const int e = __ldg(idx + i);
    if (e >= 0 && e < E) atomicAdd(&load[e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const double diff = mean - (double)load[e];
    const float sgn = diff > 0 ? 1.0f : (diff < 0 ? -1.0f : 0.0f);
    bias[e] = bias[e] + gamma * sgn;
  }
}

}  // namespace
}  // namespace beam

using namespace beam;

extern "C" moe_status moe_bias_update(const moe_dims *dims, const int32_t *topk_idx, float *bias,
                                      double gamma_max, int step, int total_steps,
                                      float *gamma_used, moe_stream_t stream) {
  moe_status st = moe_check_dims(dims);
  if (st != MOE_OK) return st;
  if (!bias || (reinterpret_cast<uintptr_t>(bias) & 3u)) return MOE_ERR_INVALID_ARG;
  if (dims->T > 0 && (!topk_idx || (reinterpret_cast<uintptr_t>(topk_idx) & 3u)))
    return MOE_ERR_INVALID_ARG;
  if (!(gamma_max >= 0.0) || total_steps < 0) return MOE_ERR_INVALID_ARG;
  double frac = total_steps > 0 ? (double)step / (double)total_steps : 1.0;
  frac = frac < 0.0 ? 0.0 : (frac > 1.0 ? 1.0 : frac);
  const float gamma = (float)(gamma_max * 0.5 * (1.0 + std::cos(M_PI * frac)));
  if (gamma_used) *gamma_used = gamma;
  const long n = (long)dims->T * dims->top_k;
  const double mean = (double)n / (double)dims->E;
  bias_update_kernel<<<1, 1024, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      topk_idx, n, dims->E, mean, gamma, bias);
  return cudaPeekAtLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
