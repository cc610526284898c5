// Expert MLPs of the Beam MoE block over the permuted rows: each expert is a
// SwiGLU MLP ("Hugging Face releases Beam ...", third paragraph):
//   h = silu(X_e . W_gate[e]^T) * (X_e . W_up[e]^T)
//   y_partial = topk_w * (h . W_down[e]^T)
//
// Both GEMMs run on the tcgen05 skeleton with the weight rows as the MMA's
// M side (128 output features per tile) and the expert's token rows as the N
// side (BN rows, 16..256, chosen from the mean rows per expert).  At decode
// sizes this streams each touched expert's weights once through shared
// memory while the few token rows ride along; at prefill sizes BN = 256.
// Gate and up share one B tile and accumulate into two tensor-memory blocks,
// so silu(g) * u is formed in the epilogue without another pass; the down
// projection scales each token row by its routing weight in its epilogue.
#include "moe_internal.cuh"
#include "tc_gemm.cuh"

namespace beam {

namespace {

template <int CH>
__device__ __forceinline__ void tmem_ld_chunk(uint32_t taddr, uint32_t (&r)[CH]);
template <>
__device__ __forceinline__ void tmem_ld_chunk<32>(uint32_t taddr, uint32_t (&r)[32]) {
  tmem_ld32(taddr, r);
}
template <>
__device__ __forceinline__ void tmem_ld_chunk<16>(uint32_t taddr, uint32_t (&r)[16]) {
  tmem_ld16(taddr, r);
}

struct ExpertSched {
  int off[257];  // expert row offsets
  int tt[257];   // prefix of token tiles per expert
};

template <int BN_, bool GATEUP>
struct ExpertGemm {
  static constexpr int BN = BN_;
  static constexpr int NA = GATEUP ? 2 : 1;
  static constexpr int NBUF = (2 * NA * BN <= 512) ? 2 : 1;
  static constexpr int STAGE_BYTES = StageGeom<BN, NA>::kBytes;
  static constexpr int STAGES_FIT =
      (kSmemLimit - kSmemReserve - (int)sizeof(ExpertSched)) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 12 ? 12 : STAGES_FIT;
  static_assert(STAGES >= 2, "pipeline needs two stages");

  struct Params {
    CUtensorMap tmap_a0;  // weights [E * a_rows, K]: W_gate or W_down
    CUtensorMap tmap_a1;  // W_up (gate/up only)
    CUtensorMap tmap_b;   // token rows [Tk, K]: x_perm or h
    const int32_t *offsets;
    const int32_t *row_src;
    const float *topk_w;
    __nv_bfloat16 *out;  // h [Tk, I] or y_partial [Tk, H]
    int E, out_cols, a_rows, ksteps, mt;
    uint32_t *status;
  };
  using Sched = ExpertSched;
  struct Tile {
    int row0, nrows, arow0, m;
  };

  __device__ static void prologue(const Params &p, Sched &s) {
    for (int i = threadIdx.x; i <= p.E; i += blockDim.x) s.off[i] = p.offsets[i];
    __syncthreads();
    if (threadIdx.x < 32) {
      const int lane = threadIdx.x;
      const int per = (p.E + 31) / 32;
      const int e0 = lane * per;
      int local = 0;
      for (int e = e0; e < e0 + per && e < p.E; ++e) local += (s.off[e + 1] - s.off[e] + BN - 1) / BN;
      int incl = local;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      int run = incl - local;
      for (int e = e0; e < e0 + per && e < p.E; ++e) {
        s.tt[e] = run;
        run += (s.off[e + 1] - s.off[e] + BN - 1) / BN;
      }
      if (lane == 31) s.tt[p.E] = incl;
    }
    __syncthreads();
  }
  __device__ static int num_tiles(const Params &p, const Sched &s) { return s.tt[p.E] * p.mt; }
  __device__ static Tile tile(const Params &p, const Sched &s, int t) {
    const int tti = t / p.mt, m = t - tti * p.mt;
    int lo = 0, hi = p.E;  // last e with tt[e] <= tti
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s.tt[mid] <= tti) lo = mid;
      else hi = mid;
    }
    const int e = lo;
    const int row0 = s.off[e] + (tti - s.tt[e]) * BN;
    const int nrows = min(BN, s.off[e + 1] - row0);
    return Tile{row0, nrows, e * p.a_rows + m * kTileM, m};
  }
  __device__ static int num_k(const Params &p, const Tile &) { return p.ksteps; }
  __device__ static void load(const Params &p, const Tile &t, int k, uint8_t *stage, uint64_t *bar) {
    tma_load_2d(stage, &p.tmap_a0, bar, k * kTileK, t.arow0);
    if (GATEUP) tma_load_2d(stage + kATileBytes, &p.tmap_a1, bar, k * kTileK, t.arow0);
    tma_load_2d(stage + NA * kATileBytes, &p.tmap_b, bar, k * kTileK, t.row0);
  }
  __device__ static void epilogue(const Params &p, const Tile &t, uint32_t taddr, int row) {
    constexpr int CH = BN < 32 ? BN : 32;
    const int f = t.m * kTileM + row;
    for (int c = 0; c < t.nrows; c += CH) {
      uint32_t g[CH];
      tmem_ld_chunk<CH>(taddr + c, g);
      if (GATEUP) {
        uint32_t u[CH];
        tmem_ld_chunk<CH>(taddr + BN + c, u);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < CH; ++j) {
          if (c + j < t.nrows) {
            const float gv = __uint_as_float(g[j]);
            const float uv = __uint_as_float(u[j]);
            const float hv = gv / (1.0f + __expf(-gv)) * uv;
            p.out[(size_t)(t.row0 + c + j) * p.out_cols + f] = __float2bfloat16_rn(hv);
          }
        }
      } else {
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < CH; ++j) {
          if (c + j < t.nrows) {
            const int r = t.row0 + c + j;
            const float w = __ldg(p.topk_w + __ldg(p.row_src + r));
            p.out[(size_t)r * p.out_cols + f] = __float2bfloat16_rn(__uint_as_float(g[j]) * w);
          }
        }
      }
    }
  }
};

template <class P>
moe_status launch_gemm(const typename P::Params &prm, int grid, cudaStream_t stream) {
  constexpr int smem = smem_bytes_for<P>();
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(tc_gemm_kernel<P>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
    attr_set = true;
  }
  tc_gemm_kernel<P><<<grid, 256, smem, stream>>>(prm);
  return cudaPeekAtLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

template <int BN>
moe_status launch_experts_bn(const moe_dims &d, const moe_experts &ex, const void *x_perm,
                             const int32_t *offsets, const int32_t *row_src, const float *topk_w,
                             void *y_partial, __nv_bfloat16 *h, uint32_t *status,
                             cudaStream_t stream) {
  const long Tk = (long)d.T * d.top_k;
  const long max_tt = Tk / BN + std::min<long>(d.E, Tk);
  const int sms = device_sm_count();
  {
    using P = ExpertGemm<BN, true>;
    typename P::Params prm;
    if (!make_tmap_bf16_2d(&prm.tmap_a0, ex.w_gate, d.H, (uint64_t)d.E * d.I, kTileM) ||
        !make_tmap_bf16_2d(&prm.tmap_a1, ex.w_up, d.H, (uint64_t)d.E * d.I, kTileM) ||
        !make_tmap_bf16_2d(&prm.tmap_b, x_perm, d.H, Tk, BN))
      return MOE_ERR_CUDA;
    prm.offsets = offsets;
    prm.row_src = row_src;
    prm.topk_w = topk_w;
    prm.out = h;
    prm.E = d.E;
    prm.out_cols = d.I;
    prm.a_rows = d.I;
    prm.ksteps = d.H / kTileK;
    prm.mt = d.I / kTileM;
    prm.status = status;
    const int grid = (int)std::max<long>(1, std::min<long>(sms, max_tt * prm.mt));
    const moe_status st = launch_gemm<P>(prm, grid, stream);
    if (st != MOE_OK) return st;
  }
  {
    using P = ExpertGemm<BN, false>;
    typename P::Params prm;
    if (!make_tmap_bf16_2d(&prm.tmap_a0, ex.w_down, d.I, (uint64_t)d.E * d.H, kTileM) ||
        !make_tmap_bf16_2d(&prm.tmap_b, h, d.I, Tk, BN))
      return MOE_ERR_CUDA;
    prm.tmap_a1 = prm.tmap_a0;
    prm.offsets = offsets;
    prm.row_src = row_src;
    prm.topk_w = topk_w;
    prm.out = static_cast<__nv_bfloat16 *>(y_partial);
    prm.E = d.E;
    prm.out_cols = d.H;
    prm.a_rows = d.H;
    prm.ksteps = d.I / kTileK;
    prm.mt = d.H / kTileM;
    prm.status = status;
    const int grid = (int)std::max<long>(1, std::min<long>(sms, max_tt * prm.mt));
    return launch_gemm<P>(prm, grid, stream);
  }
}

// ------------------------------------------------------------------ combine

__global__ void __launch_bounds__(128)
    combine_kernel(const uint4 *__restrict__ y_partial, const int32_t *__restrict__ slot_of,
                   int top_k, int vec_per_row, uint4 *__restrict__ y) {
  __shared__ int slots[16];
  const int t = blockIdx.x;
  if (threadIdx.x < top_k) slots[threadIdx.x] = slot_of[(size_t)t * top_k + threadIdx.x];
  __syncthreads();
  for (int v = threadIdx.x; v < vec_per_row; v += blockDim.x) {
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    for (int j = 0; j < top_k; ++j) {
      const int s = slots[j];
      if (s < 0) continue;
      const uint4 q = y_partial[(size_t)s * vec_per_row + v];
      const __nv_bfloat162 *b = reinterpret_cast<const __nv_bfloat162 *>(&q);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(b[i]);
        acc[2 * i] += f.x;
        acc[2 * i + 1] += f.y;
      }
    }
    uint4 o;
    __nv_bfloat162 *ob = reinterpret_cast<__nv_bfloat162 *>(&o);
#pragma unroll
    for (int i = 0; i < 4; ++i) ob[i] = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
    y[(size_t)t * vec_per_row + v] = o;
  }
}

}  // namespace

moe_status launch_experts(const moe_dims &d, const moe_experts &ex, const void *x_perm,
                          const int32_t *expert_offsets, const int32_t *row_src,
                          const float *topk_w, void *y_partial, __nv_bfloat16 *h,
                          uint32_t *status, cudaStream_t stream) {
  if (ex.dtype != MOE_W_BF16) return MOE_ERR_NOT_IMPLEMENTED;
  switch (expert_bn(d)) {
    case 16: return launch_experts_bn<16>(d, ex, x_perm, expert_offsets, row_src, topk_w, y_partial, h, status, stream);
    case 32: return launch_experts_bn<32>(d, ex, x_perm, expert_offsets, row_src, topk_w, y_partial, h, status, stream);
    case 64: return launch_experts_bn<64>(d, ex, x_perm, expert_offsets, row_src, topk_w, y_partial, h, status, stream);
    case 128: return launch_experts_bn<128>(d, ex, x_perm, expert_offsets, row_src, topk_w, y_partial, h, status, stream);
    default: return launch_experts_bn<256>(d, ex, x_perm, expert_offsets, row_src, topk_w, y_partial, h, status, stream);
  }
}

moe_status launch_combine(const moe_dims &d, const void *y_partial, const int32_t *slot_of, void *y,
                          cudaStream_t stream) {
  if (d.T == 0) return MOE_OK;
  combine_kernel<<<d.T, 128, 0, stream>>>(static_cast<const uint4 *>(y_partial), slot_of, d.top_k,
                                          d.H / 8, static_cast<uint4 *>(y));
  return cudaPeekAtLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace beam
