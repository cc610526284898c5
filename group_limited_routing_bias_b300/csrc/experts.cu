// Expert MLPs of the Beam MoE block over the permuted rows: each expert is a
// SwiGLU MLP ("Hugging Face releases Beam ...", third paragraph):
//   h = silu(X_e . W_gate[e]^T) * (X_e . W_up[e]^T)
//   y_partial = topk_w * (h . W_down[e]^T)
//
// Both GEMMs run on the tcgen05 skeleton in one of two orientations.  Up to
// 1023 (token, expert) rows per call, the weight rows are the MMA's M side
// (128 output features per tile) and the expert's token rows the N side (BN
// rows, 16..256, from the mean rows per expert): at decode sizes this streams
// each touched expert's weights once through shared memory while the few
// token rows ride along.  From 1024 rows up, the token-major tiles below put
// 128 token rows on M and 256 weight rows on N.
// Gate and up share one B tile and accumulate into two tensor-memory blocks,
// so silu(g) * u is formed in the epilogue without another pass; the down
// projection scales each token row by its routing weight in its epilogue.
#include "moe_internal.cuh"
#include "sched.cuh"
#include "tc_gemm.cuh"

namespace beam {

namespace {

template <int CH>
__device__ __forceinline__ void tmem_ld_chunk(uint32_t taddr, uint32_t (&r)[CH]);
template <>
__device__ __forceinline__ void tmem_ld_chunk<32>(uint32_t taddr, uint32_t (&r)[32]) {
  tmem_ld32(taddr, r);
}

template <int BN_, bool GATEUP>
struct ExpertGemm {
  static constexpr int BN = BN_;
  static constexpr int NA = GATEUP ? 2 : 1;
  static constexpr int NBUF = (2 * NA * BN <= 512) ? 2 : 1;
  // Up to 64 token rows, two 64-wide K slices per stage: every weight row then
  // arrives as 256 contiguous bytes per stage (2% more HBM bandwidth at decode).
  static constexpr int KSUB = BN <= 64 ? 2 : 1;
  static constexpr int STAGE_BYTES = StageGeom<BN, NA>::kBytes * KSUB;
  static constexpr int STAGES_FIT =
      (kSmemLimit - kSmemReserve - (int)sizeof(TileSched)) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_FIT > 12 ? 12 : STAGES_FIT;
  static_assert(STAGES >= 2, "pipeline needs two stages");
  static constexpr bool DYNAMIC = true;  // tiles taken from a global counter
  // The down GEMM is launched as a programmatic dependent of gate/up: its CTAs
  // start on SMs that gate/up no longer needs, and each down tile waits only
  // for its own expert's h rows (counted per expert as the gate/up epilogue
  // warps store them), so the gate/up tail and the launch gap overlap work.
  static constexpr bool PDL_PRIMARY = GATEUP;
  static constexpr bool PDL_SECONDARY = !GATEUP;

  struct Params {
    CUtensorMap tmap_a0;  // weights [E * a_rows, K]: W_gate or W_down
    CUtensorMap tmap_a1;  // W_up (gate/up only)
    CUtensorMap tmap_b;   // token rows [Tk, K]: x_perm or h, box of BN rows
    CUtensorMap tmap_bh;  // the same rows, box of BN / 2 rows
    const int32_t *offsets;
    const int32_t *row_src;
    const float *topk_w;
    __nv_bfloat16 *out;  // h [Tk, I] or y_partial [Tk, H]
    int E, out_cols, a_rows, ksteps, mt;
    uint32_t *status;
    // MMA-tiled weights (moe_pack_bf16), or null: each 128 x 64 tile is one
    // contiguous 16 KB copy instead of a 2-D TMA box
    const uint8_t *wp0, *wp1;
    int ktiles;  // 64-wide k blocks per weight row
    uint32_t *sched_counters;  // dynamic tile schedule (workspace header)
    uint32_t *expert_done;     // [E] gate/up epilogue warps done per expert (workspace header)
    int up_mt;                 // gate/up feature tiles per token tile (down: readiness target)
  };
  using Sched = TileSched;
  struct Tile {
    int row0, nrows, arow0, m, e, ntt;  // ntt: token tiles of expert e
  };
  static constexpr bool CONVERT = false;
  static constexpr bool F16 = false;
  static constexpr int RAW_BYTES = 0;
  static constexpr int RSTAGES = 0;
  __device__ static void convert(const Params &, const Tile &, int, uint8_t *, int) {}

  // Token rows a tile loads: a tile of at most BN / 2 rows loads the half box
  // (the MMA still reads BN rows; the columns of rows past the tile's own are
  // never stored), so an expert of up to BN rows streams its weights once at
  // the cost of a BN / 2 box.
  __device__ static int box_rows(const Tile &t) { return t.nrows <= BN / 2 ? BN / 2 : BN; }
  __device__ static uint32_t tx_bytes(const Params &, const Tile &t) {
    return (uint32_t)KSUB * (NA * kATileBytes + box_rows(t) * kTileK * 2);
  }

  __device__ static void prologue(const Params &p, Sched &s) {
    tile_sched_prologue(p.offsets, p.E, BN, 1, s);
  }
  __device__ static int num_tiles(const Params &p, const Sched &s) { return s.tp[p.E] * p.mt; }
  __device__ static Tile tile(const Params &p, const Sched &s, int t) {
    const int tti = t / p.mt, m = t - tti * p.mt;
    const int e = tile_sched_expert(s, p.E, tti);
    const int row0 = s.off[e] + (tti - s.tp[e]) * BN;
    const int nrows = min(BN, s.off[e + 1] - row0);
    return Tile{row0, nrows, e * p.a_rows + m * kTileM, m, e, s.tp[e + 1] - s.tp[e]};
  }
  // gate/up: each epilogue warp publishes its 32 features of h for the tile
  // (release: its stores before the count, for the down GEMM's TMA reads)
  __device__ static void tile_done(const Params &p, const Tile &t) {
    if constexpr (GATEUP) {
      asm volatile("fence.proxy.async.global;" ::: "memory");
      __threadfence();
      atomicAdd(p.expert_done + t.e, 1u);
    }
  }
  // down: wait until every gate/up tile of the expert (4 epilogue warps each)
  // has been published, then order the TMA reads of h after that
  __device__ static bool tile_ready(const Params &p, const Tile &t, volatile int *abort) {
    if constexpr (GATEUP) {
      return true;
    } else {
      const uint32_t need = 4u * (uint32_t)p.up_mt * (uint32_t)t.ntt;
      const uint32_t *cnt = p.expert_done + t.e;
      if (ld_acquire_gpu(cnt) < need) {
        const uint64_t t0 = global_timer_ns();
        while (ld_acquire_gpu(cnt) < need) {
          if (*abort) return false;
          if (global_timer_ns() - t0 > kWaitLimitNs) {
            *abort = 1;
            atomicOr(p.status, (uint32_t)MOE_DEV_TIMEOUT);
            return false;
          }
          __nanosleep(100);
        }
      }
      asm volatile("fence.proxy.async.global;" ::: "memory");
      return true;
    }
  }
  // down, last CTA: every count has been consumed; zero them for the next call
  __device__ static void last_cta(const Params &p) {
    if constexpr (!GATEUP)
      for (int e = 0; e < p.E; ++e) p.expert_done[e] = 0;
  }
  __device__ static int num_k(const Params &p, const Tile &) { return p.ksteps; }
  __device__ static void load(const Params &p, const Tile &t, int k, uint8_t *stage, uint64_t *bar) {
#pragma unroll
    for (int sub = 0; sub < KSUB; ++sub) {
      uint8_t *st = stage + sub * StageGeom<BN, NA>::kBytes;
      const int kb = k * KSUB + sub;
      if (p.wp0) {
        const size_t tile = (size_t)(t.arow0 / kTileM) * p.ktiles + kb;
        bulk_load(st, p.wp0 + tile * kATileBytes, kATileBytes, bar);
        if (GATEUP) bulk_load(st + kATileBytes, p.wp1 + tile * kATileBytes, kATileBytes, bar);
      } else {
        tma_load_2d(st, &p.tmap_a0, bar, kb * kTileK, t.arow0);
        if (GATEUP) tma_load_2d(st + kATileBytes, &p.tmap_a1, bar, kb * kTileK, t.arow0);
      }
      tma_load_2d(st + NA * kATileBytes, box_rows(t) == BN ? &p.tmap_b : &p.tmap_bh, bar,
                  kb * kTileK, t.row0);
    }
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

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&v);
}

// Token-major expert GEMM for larger batches: 128 token rows of one expert on
// the MMA's M side, 256 weight rows on the N side.  Gate/up: the N side is the
// 128 gate rows and the 128 up rows of the same 128 features, so each thread
// of the epilogue owns one token row and holds both g and u of its features;
// it writes h as 16-byte vectors.  Down: 256 output features per tile, the
// row's routing weight is one scalar per thread.  Two 256-column accumulators
// double-buffer the 512 tensor-memory columns.  Tiles of one expert run
// feature-tile-major so the token tiles that share a weight tile are
// scheduled side by side and read it from L2.
template <bool GATEUP>
struct ExpertGemmTM {
  static constexpr int BN = 256;
  static constexpr int NA = 1;
  static constexpr int NBUF = 2;
  static constexpr int STAGES = 4;
  static constexpr int FW = GATEUP ? 128 : 256;  // output features per tile

  struct Params {
    CUtensorMap tmap_a;   // token rows [Tk, K]: x_perm or h, box {64, 128}
    CUtensorMap tmap_a32, tmap_a64;  // the same rows, boxes {64, 32} and {64, 64}
    CUtensorMap tmap_b0;  // W_gate [E*I, H] box {64,128}, or W_down [E*H, I] box {64,256}
    CUtensorMap tmap_b1;  // W_up [E*I, H] box {64,128} (gate/up only)
    const int32_t *offsets;
    const int32_t *row_src;
    const float *topk_w;
    __nv_bfloat16 *out;  // h [Tk, I] or y_partial [Tk, H]
    int E, out_cols, b_rows, ksteps, nf;
    uint32_t *status;
    const uint8_t *wp0, *wp1;  // MMA-tiled weights (moe_pack_bf16), or null
    int ktiles;                // 64-wide k blocks per weight row
  };
  using Sched = TileSched;
  struct Tile {
    int row0, nrows, brow0, f;
  };
  static constexpr bool CONVERT = false;
  static constexpr bool F16 = false;
  static constexpr int RAW_BYTES = 0;
  static constexpr int RSTAGES = 0;
  __device__ static void convert(const Params &, const Tile &, int, uint8_t *, int) {}

  __device__ static void prologue(const Params &p, Sched &s) {
    tile_sched_prologue(p.offsets, p.E, kTileM, p.nf, s);
  }
  __device__ static int num_tiles(const Params &p, const Sched &s) { return s.tp[p.E]; }
  __device__ static Tile tile(const Params &p, const Sched &s, int t) {
    const int e = tile_sched_expert(s, p.E, t);
    const int ntt = (s.off[e + 1] - s.off[e] + kTileM - 1) / kTileM;
    const int local = t - s.tp[e];
    const int f = local / ntt, tt = local - f * ntt;
    const int row0 = s.off[e] + tt * kTileM;
    return Tile{row0, min(kTileM, s.off[e + 1] - row0), e * p.b_rows + f * FW, f};
  }
  __device__ static int num_k(const Params &p, const Tile &) { return p.ksteps; }
  __device__ static uint32_t tx_bytes(const Params &, const Tile &t) {
    return act_box_rows(t.nrows) * kTileK * 2 + 2 * kATileBytes;
  }
  __device__ static void load(const Params &p, const Tile &t, int k, uint8_t *stage, uint64_t *bar) {
    const int ar = act_box_rows(t.nrows);
    tma_load_2d(stage, ar == 32 ? &p.tmap_a32 : ar == 64 ? &p.tmap_a64 : &p.tmap_a, bar, k * kTileK,
                t.row0);
    if (p.wp0) {  // 16 KB tiles: gate then up, or two 128-row blocks of W_down
      const size_t t0 = (size_t)(t.brow0 / kTileM) * p.ktiles + k;
      bulk_load(stage + kATileBytes, p.wp0 + t0 * kATileBytes, kATileBytes, bar);
      if (GATEUP)
        bulk_load(stage + 2 * kATileBytes, p.wp1 + t0 * kATileBytes, kATileBytes, bar);
      else
        bulk_load(stage + 2 * kATileBytes, p.wp0 + (t0 + p.ktiles) * kATileBytes, kATileBytes, bar);
    } else if (GATEUP) {
      tma_load_2d(stage + kATileBytes, &p.tmap_b0, bar, k * kTileK, t.brow0);
      tma_load_2d(stage + 2 * kATileBytes, &p.tmap_b1, bar, k * kTileK, t.brow0);
    } else {
      tma_load_2d(stage + kATileBytes, &p.tmap_b0, bar, k * kTileK, t.brow0);
    }
  }
  __device__ static void epilogue(const Params &p, const Tile &t, uint32_t taddr, int row) {
    const bool valid = row < t.nrows;
    __nv_bfloat16 *dst = p.out + (size_t)(t.row0 + row) * p.out_cols + t.f * FW;
    if (GATEUP) {
#pragma unroll 1
      for (int c = 0; c < FW; c += 32) {
        uint32_t g[32], u[32];
        tmem_ld32(taddr + c, g);
        tmem_ld32(taddr + FW + c, u);
        tmem_wait_ld();
        if (valid) {
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float g0 = __uint_as_float(g[2 * j]), g1 = __uint_as_float(g[2 * j + 1]);
            const float h0 = g0 / (1.0f + __expf(-g0)) * __uint_as_float(u[2 * j]);
            const float h1 = g1 / (1.0f + __expf(-g1)) * __uint_as_float(u[2 * j + 1]);
            pk[j] = pack_bf16x2(h0, h1);
          }
          uint4 *d4 = reinterpret_cast<uint4 *>(dst + c);
#pragma unroll
          for (int q = 0; q < 4; ++q) d4[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        }
      }
    } else {
      const float w = valid ? __ldg(p.topk_w + __ldg(p.row_src + t.row0 + row)) : 0.f;
#pragma unroll 1
      for (int c = 0; c < FW; c += 32) {
        uint32_t a[32];
        tmem_ld32(taddr + c, a);
        tmem_wait_ld();
        if (valid) {
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j)
            pk[j] = pack_bf16x2(__uint_as_float(a[2 * j]) * w, __uint_as_float(a[2 * j + 1]) * w);
          uint4 *d4 = reinterpret_cast<uint4 *>(dst + c);
#pragma unroll
          for (int q = 0; q < 4; ++q) d4[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        }
      }
    }
  }
};

template <class P>
moe_status launch_gemm(const typename P::Params &prm, int grid, cudaStream_t stream) {
  constexpr int smem = smem_bytes_for<P>();
  if (ensure_smem_limit((const void *)tc_gemm_kernel<P>, smem) != MOE_OK) return MOE_ERR_CUDA;
  if constexpr (PdlSecondaryOf<P>::value) {
    // A programmatic dependent of the previous launch.  Its CTAs never share an
    // SM with the primary's (each needs more than half the shared memory).
    static_assert(smem > kSmemLimit / 2, "dependent launch must not share SMs with its primary");
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, tc_gemm_kernel<P>, prm) != cudaSuccess) return MOE_ERR_CUDA;
  } else {
    tc_gemm_kernel<P><<<grid, 256, smem, stream>>>(prm);
  }
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
        !make_tmap_bf16_2d(&prm.tmap_b, x_perm, d.H, Tk, BN) ||
        !make_tmap_bf16_2d(&prm.tmap_bh, x_perm, d.H, Tk, BN / 2))
      return MOE_ERR_CUDA;
    prm.offsets = offsets;
    prm.row_src = row_src;
    prm.topk_w = topk_w;
    prm.out = h;
    prm.E = d.E;
    prm.out_cols = d.I;
    prm.a_rows = d.I;
    prm.ksteps = d.H / (kTileK * P::KSUB);
    prm.mt = d.I / kTileM;
    prm.status = status;
    prm.sched_counters = status + kSchedCounterWord;
    prm.expert_done = status + kExpertDoneWord;
    prm.up_mt = prm.mt;
    const bool tiled = ex.layout == MOE_LAYOUT_TILED;
    prm.wp0 = tiled ? static_cast<const uint8_t *>(ex.w_gate) : nullptr;
    prm.wp1 = tiled ? static_cast<const uint8_t *>(ex.w_up) : nullptr;
    prm.ktiles = d.H / kTileK;
    const int grid = (int)std::max<long>(1, std::min<long>(sms, max_tt * prm.mt));
    const moe_status st = launch_gemm<P>(prm, grid, stream);
    if (st != MOE_OK) return st;
  }
  {
    using P = ExpertGemm<BN, false>;
    typename P::Params prm;
    if (!make_tmap_bf16_2d(&prm.tmap_a0, ex.w_down, d.I, (uint64_t)d.E * d.H, kTileM) ||
        !make_tmap_bf16_2d(&prm.tmap_b, h, d.I, Tk, BN) ||
        !make_tmap_bf16_2d(&prm.tmap_bh, h, d.I, Tk, BN / 2))
      return MOE_ERR_CUDA;
    prm.tmap_a1 = prm.tmap_a0;
    prm.offsets = offsets;
    prm.row_src = row_src;
    prm.topk_w = topk_w;
    prm.out = static_cast<__nv_bfloat16 *>(y_partial);
    prm.E = d.E;
    prm.out_cols = d.H;
    prm.a_rows = d.H;
    prm.ksteps = d.I / (kTileK * P::KSUB);
    prm.mt = d.H / kTileM;
    prm.status = status;
    prm.sched_counters = status + kSchedCounterWord + 2;  // runs alongside gate/up's
    prm.expert_done = status + kExpertDoneWord;
    prm.up_mt = d.I / kTileM;
    const bool tiled = ex.layout == MOE_LAYOUT_TILED;
    prm.wp0 = tiled ? static_cast<const uint8_t *>(ex.w_down) : nullptr;
    prm.wp1 = nullptr;
    prm.ktiles = d.I / kTileK;
    const int grid = (int)std::max<long>(1, std::min<long>(sms, max_tt * prm.mt));
    return launch_gemm<P>(prm, grid, stream);
  }
}

moe_status launch_experts_token_major(const moe_dims &d, const moe_experts &ex, const void *x_perm,
                                      const int32_t *offsets, const int32_t *row_src,
                                      const float *topk_w, void *y_partial, __nv_bfloat16 *h,
                                      uint32_t *status, cudaStream_t stream) {
  const long Tk = (long)d.T * d.top_k;
  const long max_tt = Tk / kTileM + std::min<long>(d.E, Tk);
  const int sms = device_sm_count();
  {
    using P = ExpertGemmTM<true>;
    typename P::Params prm;
    if (!make_tmap_bf16_2d(&prm.tmap_a, x_perm, d.H, Tk, kTileM) ||
        !make_tmap_bf16_2d(&prm.tmap_a32, x_perm, d.H, Tk, 32) ||
        !make_tmap_bf16_2d(&prm.tmap_a64, x_perm, d.H, Tk, 64) ||
        !make_tmap_bf16_2d(&prm.tmap_b0, ex.w_gate, d.H, (uint64_t)d.E * d.I, 128) ||
        !make_tmap_bf16_2d(&prm.tmap_b1, ex.w_up, d.H, (uint64_t)d.E * d.I, 128))
      return MOE_ERR_CUDA;
    prm.offsets = offsets;
    prm.row_src = row_src;
    prm.topk_w = topk_w;
    prm.out = h;
    prm.E = d.E;
    prm.out_cols = d.I;
    prm.b_rows = d.I;
    prm.ksteps = d.H / kTileK;
    prm.nf = d.I / P::FW;
    prm.status = status;
    const bool tiled = ex.layout == MOE_LAYOUT_TILED;
    prm.wp0 = tiled ? static_cast<const uint8_t *>(ex.w_gate) : nullptr;
    prm.wp1 = tiled ? static_cast<const uint8_t *>(ex.w_up) : nullptr;
    prm.ktiles = d.H / kTileK;
    const int grid = (int)std::max<long>(1, std::min<long>(sms, max_tt * prm.nf));
    const moe_status st = launch_gemm<P>(prm, grid, stream);
    if (st != MOE_OK) return st;
  }
  {
    using P = ExpertGemmTM<false>;
    typename P::Params prm;
    if (!make_tmap_bf16_2d(&prm.tmap_a, h, d.I, Tk, kTileM) ||
        !make_tmap_bf16_2d(&prm.tmap_a32, h, d.I, Tk, 32) ||
        !make_tmap_bf16_2d(&prm.tmap_a64, h, d.I, Tk, 64) ||
        !make_tmap_bf16_2d(&prm.tmap_b0, ex.w_down, d.I, (uint64_t)d.E * d.H, 256))
      return MOE_ERR_CUDA;
    prm.tmap_b1 = prm.tmap_b0;
    prm.offsets = offsets;
    prm.row_src = row_src;
    prm.topk_w = topk_w;
    prm.out = static_cast<__nv_bfloat16 *>(y_partial);
    prm.E = d.E;
    prm.out_cols = d.H;
    prm.b_rows = d.H;
    prm.ksteps = d.I / kTileK;
    prm.nf = d.H / P::FW;
    prm.status = status;
    const bool tiled = ex.layout == MOE_LAYOUT_TILED;
    prm.wp0 = tiled ? static_cast<const uint8_t *>(ex.w_down) : nullptr;
    prm.wp1 = nullptr;
    prm.ktiles = d.I / kTileK;
    const int grid = (int)std::max<long>(1, std::min<long>(sms, max_tt * prm.nf));
    return launch_gemm<P>(prm, grid, stream);
  }
}

// ------------------------------------------------------------------ combine

// One thread per (token, 8 consecutive columns): the k slot rows are loaded
// together, summed in fp32 in slot order and rounded once to bf16.
__global__ void __launch_bounds__(128)
    combine_kernel(const uint4 *__restrict__ y_partial, const int32_t *__restrict__ slot_of,
                   int T, int top_k, int vec_per_row, uint4 *__restrict__ y) {
  const long i = blockIdx.x * (long)blockDim.x + threadIdx.x;
  if (i >= (long)T * vec_per_row) return;
  const int t = (int)(i / vec_per_row), v = (int)(i % vec_per_row);
  const int32_t *so = slot_of + (size_t)t * top_k;
  float acc[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) acc[q] = 0.f;
  uint4 vals[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    if (j < top_k) {
      const int s = __ldg(so + j);
      vals[j] = s >= 0 ? __ldg(y_partial + (size_t)s * vec_per_row + v) : make_uint4(0, 0, 0, 0);
    }
  }
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    if (j < top_k) {
      const __nv_bfloat162 *b = reinterpret_cast<const __nv_bfloat162 *>(&vals[j]);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 f = __bfloat1622float2(b[q]);
        acc[2 * q] += f.x;
        acc[2 * q + 1] += f.y;
      }
    }
  }
  uint4 o;
  __nv_bfloat162 *ob = reinterpret_cast<__nv_bfloat162 *>(&o);
#pragma unroll
  for (int q = 0; q < 4; ++q) ob[q] = __floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]);
  y[i] = o;
}

}  // namespace

moe_status launch_experts(const moe_dims &d, const moe_experts &ex, const void *x_perm,
                          const int32_t *expert_offsets, const int32_t *row_src,
                          const float *topk_w, void *y_partial, __nv_bfloat16 *h,
                          uint32_t *status, cudaStream_t stream) {
  if (ex.dtype != MOE_W_BF16) return MOE_ERR_NOT_IMPLEMENTED;
  // Token-major tiles from 1024 (token, expert) rows up.  Measured on B300
  // (expert stage, Beam shape): 1.98 vs 2.21 ms at T=256 (top-8), 2.53 vs
  // 3.09 ms at T=1024, 2.74 vs 3.34 ms at T=2048; at T=64 the weights-on-M
  // tiles are ahead (1.354 vs 1.370 ms).
  if ((long)d.T * d.top_k >= 1024 && d.H % 256 == 0)
    return launch_experts_token_major(d, ex, x_perm, expert_offsets, row_src, topk_w, y_partial, h,
                                      status, stream);
  switch (expert_tile_rows(d)) {
    case 32: return launch_experts_bn<32>(d, ex, x_perm, expert_offsets, row_src, topk_w, y_partial, h, status, stream);
    case 64: return launch_experts_bn<64>(d, ex, x_perm, expert_offsets, row_src, topk_w, y_partial, h, status, stream);
    case 128: return launch_experts_bn<128>(d, ex, x_perm, expert_offsets, row_src, topk_w, y_partial, h, status, stream);
    default: return launch_experts_bn<256>(d, ex, x_perm, expert_offsets, row_src, topk_w, y_partial, h, status, stream);
  }
}

moe_status launch_combine(const moe_dims &d, const void *y_partial, const int32_t *slot_of, void *y,
                          cudaStream_t stream) {
  if (d.T == 0) return MOE_OK;
  const long n = (long)d.T * (d.H / 8);
  combine_kernel<<<(unsigned)((n + 127) / 128), 128, 0, stream>>>(
      static_cast<const uint4 *>(y_partial), slot_of, d.T, d.top_k, d.H / 8, static_cast<uint4 *>(y));
  return cudaPeekAtLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace beam
