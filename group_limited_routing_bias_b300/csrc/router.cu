// Router of the Beam MoE block: sigmoid scores with a per-expert selection
// bias and group-limited top-k ("Hugging Face releases Beam ...", third
// paragraph; "Reflection Releases Beam ...", section "Where Beam Saves and
// Where the Memory Bill Comes In"; "Beam 1.0" for the bias).
//
// Three kernels:
//   1. router_split_kernel: the fp32 router weight W is split into three bf16
//      matrices hi + mid + lo == W exactly, laid side by side as W3 [E, 3H].
//   2. tc_gemm_kernel<RouterLogits>: logits = x . W3^T on tcgen05 tensor
//      cores.  x is bf16 and each part has 8 significant bits, so every
//      product is exact in the fp32 accumulator.  For small T the K range is
//      split over CTAs and the partial sums are added in a fixed order later.
//   3. router_topk_kernel: one warp per token; sigmoid, bias, group top-2
//      sums, top groups and top experts by warp shuffles in registers.
#include "moe_internal.cuh"
#include "tc_gemm.cuh"

namespace beam {

// Eight consecutive weights per thread: two 16-byte loads, three 16-byte stores.
__global__ void router_split_kernel(const float4 *__restrict__ w, uint4 *__restrict__ w3, int E,
                                    int H) {
  const int vec_per_row = H / 8;
  const size_t n = (size_t)E * vec_per_row;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x) {
    const int e = (int)(i / vec_per_row), v = (int)(i % vec_per_row);
    const float4 a = w[2 * i], b = w[2 * i + 1];
    const float src[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t hi[4], mid[4], lo[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float r0[2], r1[2], r2[2];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const float x = src[2 * j + q];
        r0[q] = __bfloat162float(__float2bfloat16_rn(x));
        const float d1 = x - r0[q];  // exact: x and its bf16 rounding share the top bits
        r1[q] = __bfloat162float(__float2bfloat16_rn(d1));
        r2[q] = d1 - r1[q];  // exact, at most 8 significant bits, so exact in bf16
      }
      const __nv_bfloat162 h2 = __floats2bfloat162_rn(r0[0], r0[1]);
      const __nv_bfloat162 m2 = __floats2bfloat162_rn(r1[0], r1[1]);
      const __nv_bfloat162 l2 = __floats2bfloat162_rn(r2[0], r2[1]);
      hi[j] = *reinterpret_cast<const uint32_t *>(&h2);
      mid[j] = *reinterpret_cast<const uint32_t *>(&m2);
      lo[j] = *reinterpret_cast<const uint32_t *>(&l2);
    }
    uint4 *row = w3 + (size_t)e * 3 * vec_per_row;
    row[v] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    row[vec_per_row + v] = make_uint4(mid[0], mid[1], mid[2], mid[3]);
    row[2 * vec_per_row + v] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  }
}

// logits partial sums: D[token, expert] over one K range of [x x x] . [hi mid lo]^T
//
// The tensor cores' fp32 accumulation does not round to nearest at every step:
// over the 960 MMAs of a full K range (3 H = 15360 products) the logits of a
// T = 16384 batch drifted by up to 1.2e-4 from the exact sums (mean 2e-5),
// while split-K partials of 16 MMAs stayed within 2e-6.  So each CTA's K range
// is cut into chunks of kChunkSlices 64-wide slices: every chunk starts a fresh
// accumulator, and the epilogue adds the chunks in order, in fp32 with
// round-to-nearest, into running sums kept in tensor memory next to the
// accumulator; the last chunk's sum is the CTA's partial.
constexpr int kChunkSlices = 8;  // 32 MMAs of K = 16 per accumulator

template <int BN_>
struct RouterLogits {
  static constexpr int BN = BN_;
  static constexpr int NA = 1;
  static constexpr int NBUF = 1;
  static constexpr int STAGES = 4;
  static constexpr int EXTRA_TMEM_COLS = BN;  // running sums over the chunks
  struct Params {
    CUtensorMap tmap_x;   // bf16 [T, H], box {64, 128}
    CUtensorMap tmap_w3;  // bf16 [E, 3H], box {64, BN}
    float *partial;       // fp32 [ksplit, T, E]
    int T, E, H, ksteps, ksplit;
    uint32_t *status;
  };
  struct Sched {
    int unused;
  };
  struct Tile {
    int m0, kbeg, kend, split;
    bool first, last;  // first and last chunk of the CTA's K range
  };
  static constexpr bool CONVERT = false;
  static constexpr bool F16 = false;
  static constexpr int RAW_BYTES = 0;
  static constexpr int RSTAGES = 0;
  static constexpr int TX_BYTES = StageGeom<BN, NA>::kOperandBytes;
  __device__ static void convert(const Params &, const Tile &, int, uint8_t *, int) {}
  __device__ static void prologue(const Params &, Sched &) {}
  // K range of this CTA's split
  __device__ static int split_begin(const Params &p, int s) { return (int)((long)p.ksteps * s / p.ksplit); }
  // One M tile per CTA (grid.x = M tiles, grid.y = splits); its tiles are the
  // chunks of its K range, t = blockIdx.x + chunk * gridDim.x.
  __device__ static int num_tiles(const Params &p, const Sched &) {
    const int s = blockIdx.y;
    const int nk = split_begin(p, s + 1) - split_begin(p, s);
    return gridDim.x * ((nk + kChunkSlices - 1) / kChunkSlices);
  }
  __device__ static Tile tile(const Params &p, const Sched &, int t) {
    const int s = blockIdx.y;
    const int kb = split_begin(p, s), ke = split_begin(p, s + 1);
    const int g = (int)gridDim.x;
    const int chunk = t / g;
    const int cb = kb + chunk * kChunkSlices;
    const int ce = min(cb + kChunkSlices, ke);
    return Tile{(t % g) * kTileM, cb, ce, s, chunk == 0, ce == ke};
  }
  __device__ static int num_k(const Params &, const Tile &t) { return t.kend - t.kbeg; }
  __device__ static void load(const Params &p, const Tile &t, int k, uint8_t *stage, uint64_t *bar) {
    const int kk = t.kbeg + k;
    const int hsteps = p.H / kTileK;
    tma_load_2d(stage, &p.tmap_x, bar, (kk % hsteps) * kTileK, t.m0);
    tma_load_2d(stage + kATileBytes, &p.tmap_w3, bar, kk * kTileK, 0);
  }
  __device__ static void epilogue(const Params &p, const Tile &t, uint32_t taddr, int row) {
    const int token = t.m0 + row;
    const uint32_t run = taddr + BN;  // NBUF == 1: the running sums follow the accumulator
    bool stored = false;
    for (int c = 0; c < BN; c += 32) {
      if (c >= p.E) break;
      uint32_t r[32];
      tmem_ld32(taddr + c, r);
      if (!t.first) {
        uint32_t a[32];
        tmem_ld32(run + c, a);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j)
          r[j] = __float_as_uint(__fadd_rn(__uint_as_float(a[j]), __uint_as_float(r[j])));
      } else {
        tmem_wait_ld();
      }
      if (!t.last) {
        tmem_st32(run + c, r);
        stored = true;
      } else if (token < p.T) {
        float4 *dst = reinterpret_cast<float4 *>(p.partial + ((size_t)t.split * p.T + token) * p.E + c);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          dst[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                               __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
      }
    }
    if (stored) tmem_wait_st();
  }
};

// ------------------------------------------------------------------ top-k

struct TopkArgs {
  const float *partial;  // [ksplit, T, E]
  const float *bias;     // [E]
  float *logits;         // [T, E] or null: the summed logits the selection uses
  int32_t *topk_idx;     // [T, k]
  float *topk_w;         // [T, k]
  int T, E, n_group, topk_group, top_k, ksplit;
  int log2_gsize;
  float routed_scale;
};

// Merge (a1 >= a2) with (b1 >= b2) into the two largest of the four.
__device__ __forceinline__ void top2_merge(float &a1, float &a2, float b1, float b2) {
  const float hi = fmaxf(a1, b1);
  const float lo = fmaxf(fminf(a1, b1), fmaxf(a2, b2));
  a1 = hi;
  a2 = lo;
}

// One CTA per TPB tokens.  First all 256 threads add the K-split partial
// logits of the CTA's tokens into shared memory, splits added in split order;
// every load is issued unconditionally from a clamped address (a split past
// ksplit adds exactly +0.0), so all of a thread's loads are in flight at once.
// Then one warp per token does the selection.  Lane l holds experts
// e = l + 32 i, i = 0..7.  With a K split (small T) each CTA takes one token,
// so a thread waits on one round trip for its kMaxRouterSplit loads.
template <int TPB>
__global__ void __launch_bounds__(256) router_topk_kernel(TopkArgs a) {
  constexpr int NS = 8;
  __shared__ float logits_s[TPB][256];
  const int lane = threadIdx.x & 31;
  const int gsize = 1 << a.log2_gsize;
  const int t0 = blockIdx.x * TPB;
  {
    const int e = threadIdx.x;  // blockDim.x == 256 >= E
    float acc[TPB];
#pragma unroll
    for (int j = 0; j < TPB; ++j) acc[j] = 0.f;
    if (e < a.E) {
      if constexpr (TPB == 1) {
        float v[kMaxRouterSplit];
#pragma unroll
        for (int sp = 0; sp < kMaxRouterSplit; ++sp) {
          const int spc = sp < a.ksplit ? sp : a.ksplit - 1;
          v[sp] = __ldg(a.partial + ((size_t)spc * a.T + t0) * a.E + e);
        }
#pragma unroll
        for (int sp = 0; sp < kMaxRouterSplit; ++sp) acc[0] += sp < a.ksplit ? v[sp] : 0.f;
      } else {  // TPB > 1 is only launched without a K split
#pragma unroll
        for (int j = 0; j < TPB; ++j)
          acc[j] = __ldg(a.partial + (size_t)min(t0 + j, a.T - 1) * a.E + e);
      }
    }
#pragma unroll
    for (int j = 0; j < TPB; ++j) {
      logits_s[j][e] = acc[j];
      if (a.logits && e < a.E && t0 + j < a.T) a.logits[(size_t)(t0 + j) * a.E + e] = acc[j];
    }
  }
  __syncthreads();
  if ((threadIdx.x >> 5) >= TPB) return;
  const int t = t0 + (threadIdx.x >> 5);
  if (t < a.T) {
    float s[NS], sb[NS];
#pragma unroll
    for (int i = 0; i < NS; ++i) {
      const int e = lane + 32 * i;
      if (e < a.E) {
        const float l = logits_s[threadIdx.x >> 5][e];
        s[i] = 1.0f / (1.0f + expf(-l));
        sb[i] = s[i] + a.bias[e];
      } else {
        s[i] = 0.f;
        sb[i] = -INFINITY;
      }
    }
    // ---- group scores: sum of the two largest biased scores per group
    float g1[NS], g2[NS];
#pragma unroll
    for (int i = 0; i < NS; ++i) {
      g1[i] = sb[i];
      g2[i] = -INFINITY;
    }
    const int seg = gsize < 32 ? gsize : 32;  // lanes per group inside one slot
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      if (off < seg) {
#pragma unroll
        for (int i = 0; i < NS; ++i) {
          const float o1 = __shfl_xor_sync(0xffffffffu, g1[i], off);
          const float o2 = __shfl_xor_sync(0xffffffffu, g2[i], off);
          top2_merge(g1[i], g2[i], o1, o2);
        }
      }
    }
    // a group wider than 32 spans gsize/32 consecutive slots: tree-merge them
    // into the group's first slot (static register indices only)
    if (gsize >= 64) {
#pragma unroll
      for (int i = 0; i < NS; i += 2) top2_merge(g1[i], g2[i], g1[i + 1], g2[i + 1]);
    }
    if (gsize >= 128) {
#pragma unroll
      for (int i = 0; i < NS; i += 4) top2_merge(g1[i], g2[i], g1[i + 2], g2[i + 2]);
    }
    if (gsize >= 256) top2_merge(g1[0], g2[0], g1[4], g2[4]);
    // lane j (< n_group) fetches the score of group j
    float my_gs = -INFINITY;
#pragma unroll
    for (int i = 0; i < NS; ++i) {
      const int first_e = lane * gsize;  // first expert of group `lane`
      const int src = first_e & 31;
      const float v = __shfl_sync(0xffffffffu, g1[i] + g2[i], src);
      if (lane < a.n_group && (first_e >> 5) == i) my_gs = v;
    }
    // rank of group `lane`: groups with a larger score, or equal and lower index
    int rank = 0;
    for (int j = 0; j < a.n_group; ++j) {
      const float v = __shfl_sync(0xffffffffu, my_gs, j);
      if (v > my_gs || (v == my_gs && j < lane)) ++rank;
    }
    const uint32_t kept = __ballot_sync(0xffffffffu, lane < a.n_group && rank < a.topk_group);

    // ---- top-k experts among the kept groups (descending, ties to lower index)
    float cand[NS];
#pragma unroll
    for (int i = 0; i < NS; ++i) {
      const int e = lane + 32 * i;
      cand[i] = (e < a.E && ((kept >> (e >> a.log2_gsize)) & 1u)) ? sb[i] : -INFINITY;
    }
    float wsum = 0.f, my_s = 0.f;
    int my_e = 0;
    for (int r = 0; r < a.top_k; ++r) {
      float bv = -INFINITY;
      int be = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < NS; ++i) {
        const int e = lane + 32 * i;
        if (cand[i] > bv) {  // slots ascend in e, so a tie keeps the lower index
          bv = cand[i];
          be = e;
        }
      }
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int oe = __shfl_xor_sync(0xffffffffu, be, off);
        if (ov > bv || (ov == bv && oe < be)) {
          bv = ov;
          be = oe;
        }
      }
      float sv = 0.f;
      if ((be & 31) == lane) {
#pragma unroll
        for (int i = 0; i < NS; ++i)
          if (i == (be >> 5)) {
            sv = s[i];
            cand[i] = -INFINITY;
          }
      }
      sv = __shfl_sync(0xffffffffu, sv, be & 31);
      wsum += sv;
      if (lane == r) {
        my_s = sv;
        my_e = be;
      }
    }
    if (lane < a.top_k) {
      a.topk_idx[(size_t)t * a.top_k + lane] = my_e;
      a.topk_w[(size_t)t * a.top_k + lane] = a.routed_scale * my_s / wsum;
    }
  }
}

// ------------------------------------------------------------------ host side

template <int BN>
static moe_status launch_router_gemm(const RouterPlan &rp, const void *x, const __nv_bfloat16 *w3,
                                     float *partial, uint32_t *status, cudaStream_t stream) {
  using P = RouterLogits<BN>;
  typename P::Params prm;
  if (!make_tmap_bf16_2d(&prm.tmap_x, x, rp.H, rp.T, kTileM)) return MOE_ERR_CUDA;
  if (!make_tmap_bf16_2d(&prm.tmap_w3, w3, 3 * rp.H, rp.E, BN)) return MOE_ERR_CUDA;
  prm.partial = partial;
  prm.T = rp.T;
  prm.E = rp.E;
  prm.H = rp.H;
  prm.ksteps = 3 * rp.H / kTileK;
  prm.ksplit = rp.ksplit;
  prm.status = status;
  constexpr int smem = smem_bytes_for<P>();
  if (ensure_smem_limit((const void *)tc_gemm_kernel<P>, smem) != MOE_OK) return MOE_ERR_CUDA;
  dim3 grid((rp.T + kTileM - 1) / kTileM, rp.ksplit);
  tc_gemm_kernel<P><<<grid, 256, smem, stream>>>(prm);
  return cudaPeekAtLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status launch_route(const moe_dims &d, const void *x, const float *w_router, const float *bias,
                        int32_t *topk_idx, float *topk_w, const RouterPlan &rp,
                        __nv_bfloat16 *w3, float *partial, uint32_t *status, cudaStream_t stream,
                        float *logits) {
  {
    const size_t n = (size_t)d.E * d.H / 8;
    const int blocks = (int)std::min<size_t>((n + 255) / 256, 4096);
    router_split_kernel<<<blocks, 256, 0, stream>>>(reinterpret_cast<const float4 *>(w_router),
                                                    reinterpret_cast<uint4 *>(w3), d.E, d.H);
    if (cudaPeekAtLastError() != cudaSuccess) return MOE_ERR_CUDA;
  }
  moe_status st;
  if (rp.BN == 32) st = launch_router_gemm<32>(rp, x, w3, partial, status, stream);
  else if (rp.BN == 64) st = launch_router_gemm<64>(rp, x, w3, partial, status, stream);
  else if (rp.BN == 128) st = launch_router_gemm<128>(rp, x, w3, partial, status, stream);
  else st = launch_router_gemm<256>(rp, x, w3, partial, status, stream);
  if (st != MOE_OK) return st;

  TopkArgs a;
  a.partial = partial;
  a.bias = bias;
  a.logits = logits;
  a.topk_idx = topk_idx;
  a.topk_w = topk_w;
  a.T = d.T;
  a.E = d.E;
  a.n_group = d.n_group;
  a.topk_group = d.topk_group;
  a.top_k = d.top_k;
  a.ksplit = rp.ksplit;
  a.log2_gsize = ilog2(d.E / d.n_group);
  a.routed_scale = d.routed_scale;
  if (rp.ksplit > 1)
    router_topk_kernel<1><<<d.T, 256, 0, stream>>>(a);
  else
    router_topk_kernel<8><<<(d.T + 7) / 8, 256, 0, stream>>>(a);
  return cudaPeekAtLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace beam
