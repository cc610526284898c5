// Expert MLPs with packed NVFP4 or FP8 weights for small and mid-size batches:
// weights on the MMA's M side, dequantised straight into tensor memory
// (tc_gemm_wtmem.cuh), the expert's token rows on N.  Same block as
// experts.cu ("Hugging Face releases Beam ...", third paragraph: SwiGLU
// experts; "Reflection Releases Beam ...", section "Where Beam Saves and Where
// the Memory Bill Comes In": NVFP4 and FP8 checkpoints):
//   h = silu(X_e . W_gate[e]^T) * (X_e . W_up[e]^T)
//   y_partial = topk_w * (h . W_down[e]^T)
//
// Operands are bf16 on both sides, so the activations keep bf16's range: a
// weight e2m1 * e4m3 (at most six significant bits, in [2^-10, 2688]) or an
// e4m3 code is exact in bf16.  A converter thread dequantises one weight row
// of a 64-wide K slice: e2m1 (or e4m3) pairs to f16 pairs by the hardware
// conversion, times the f16 block scale (exact), widened to fp32 and packed to
// bf16 pairs (exact).  The NVFP4 global scale and the FP8 row scales multiply
// the fp32 accumulator in the epilogue.  x_perm and h stay bf16.
//
// Tiles, schedule and the gate/up -> down hand-off are those of the bf16
// weights-on-M GEMMs in experts.cu: tiles are taken from a global counter,
// the down GEMM is a programmatic dependent of gate/up and each down tile
// waits (bounded) until its expert's h rows are published.
#include "moe_internal.cuh"
#include "sched.cuh"
#include "tc_gemm_wtmem.cuh"

namespace beam {

namespace {

// Two f16 values -> the same two values as bf16 (exact for every value
// produced here: at most 11 significant bits are never needed, all are normal
// or zero in bf16's range).
__device__ __forceinline__ uint32_t f16x2_to_bf16x2(uint32_t h) {
  float lo, hi;
  asm("{\n\t.reg .b16 l, u;\n\tmov.b32 {l, u}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, u;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(h));
  uint32_t o;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(o) : "f"(hi), "f"(lo));
  return o;
}

// One NVFP4 weight row of a 64-wide K slice: 32 code bytes (even k in the low
// nibble) and the four e4m3 scales of its 16-k blocks -> 32 bf16 pairs.
__device__ __forceinline__ void nvfp4_row_bf16(uint4 c0, uint4 c1, uint32_t scales,
                                               uint32_t (&out)[32]) {
  uint32_t s16[4];
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const uint32_t byte = (scales >> (8 * b)) & 0xFFu;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(s16[b]) : "h"((uint16_t)(byte | (byte << 8))));
  }
  const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {  // word i: k 8i .. 8i + 7, block i / 2
    uint32_t h0, h1, h2, h3;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
        : "r"(w[i]));
    const uint32_t s = s16[i >> 1];
    asm("mul.rn.f16x2 %0, %0, %1;" : "+r"(h0) : "r"(s));
    asm("mul.rn.f16x2 %0, %0, %1;" : "+r"(h1) : "r"(s));
    asm("mul.rn.f16x2 %0, %0, %1;" : "+r"(h2) : "r"(s));
    asm("mul.rn.f16x2 %0, %0, %1;" : "+r"(h3) : "r"(s));
    out[4 * i + 0] = f16x2_to_bf16x2(h0);
    out[4 * i + 1] = f16x2_to_bf16x2(h1);
    out[4 * i + 2] = f16x2_to_bf16x2(h2);
    out[4 * i + 3] = f16x2_to_bf16x2(h3);
  }
}

// One FP8 weight row of a 64-wide K slice: 64 e4m3 codes -> 32 bf16 pairs.
__device__ __forceinline__ void fp8_row_bf16(const uint8_t *codes, uint32_t (&out)[32]) {
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    const uint4 q = *reinterpret_cast<const uint4 *>(codes + 16 * v);
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t lo, hi;
      asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(lo) : "h"((uint16_t)(w[i] & 0xFFFFu)));
      asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(hi) : "h"((uint16_t)(w[i] >> 16)));
      out[8 * v + 2 * i] = f16x2_to_bf16x2(lo);
      out[8 * v + 2 * i + 1] = f16x2_to_bf16x2(hi);
    }
  }
}

// Raw layouts of one 128-row A tile of a K slice in a ring slot, per format.
// Row-major NVFP4 arrives as TMA boxes: codes [128][32 B], then scale boxes
// [128][16 B] (the 16 scales of 256 k; this slice's four at (k % 4) * 4).
struct WtNvfp4 {
  static constexpr bool kTiled = false, kPerRowScale = false;
  static constexpr int kTileBytes = 128 * 48;
  __device__ static void convert(const uint8_t *t, int k, int r, uint32_t (&out)[32]) {
    const uint4 *c = reinterpret_cast<const uint4 *>(t + r * 32);
    const uint32_t sc = *reinterpret_cast<const uint32_t *>(t + 128 * 32 + r * 16 + (k & 3) * 4);
    nvfp4_row_bf16(c[0], c[1], sc, out);
  }
};
// Tiled NVFP4 (moe_pack_nvfp4): codes [128][32 B], then scales [128][4 B].
struct WtNvfp4Tiled {
  static constexpr bool kTiled = true, kPerRowScale = false;
  static constexpr int kTileBytes = 4608;
  __device__ static void convert(const uint8_t *t, int, int r, uint32_t (&out)[32]) {
    const uint4 *c = reinterpret_cast<const uint4 *>(t + r * 32);
    const uint32_t sc = *reinterpret_cast<const uint32_t *>(t + 128 * 32 + r * 4);
    nvfp4_row_bf16(c[0], c[1], sc, out);
  }
};
// FP8, row-major (TMA box) or tiled (moe_pack_fp8): codes [128][64 B].
struct WtFp8 {
  static constexpr bool kTiled = false, kPerRowScale = true;
  static constexpr int kTileBytes = 8192;
  __device__ static void convert(const uint8_t *t, int, int r, uint32_t (&out)[32]) {
    fp8_row_bf16(t + r * 64, out);
  }
};
struct WtFp8Tiled : WtFp8 {
  static constexpr bool kTiled = true;
};

struct WtParams {
  CUtensorMap tmap_b;    // token rows [Tk, K] bf16 (x_perm or h), box {64, BN}
  CUtensorMap tmap_bh;   // the same rows, box {64, BN / 2}
  CUtensorMap tmap_q0;   // row-major codes of W_gate or W_down
  CUtensorMap tmap_q1;   // row-major codes of W_up
  CUtensorMap tmap_s0;   // row-major NVFP4 scales of W_gate or W_down
  CUtensorMap tmap_s1;   // ... of W_up
  const uint8_t *wt0, *wt1;  // tiled layouts (maps unused)
  int ktiles;                // K slices per 128-row block (tiled)
  const float *g0, *g1;      // NVFP4 globals [E]; FP8 row scales [E, N]
  int scale_rows;            // N for FP8 row scales, 0 for NVFP4
  const int32_t *offsets;
  const int32_t *row_src;
  const float *topk_w;
  __nv_bfloat16 *out;  // h [Tk, I] or y_partial [Tk, H]
  int E, out_cols, w_rows, ksteps, mt;
  uint32_t *status;
  uint32_t *sched_counters;  // dynamic tile schedule (workspace header)
  uint32_t *expert_done;     // [E] gate/up epilogue warps done per expert (workspace header)
  int up_mt;                 // gate/up feature tiles per token tile (down: readiness target)
};

__device__ __forceinline__ float wt_scale(const float *g, int scale_rows, int e, int n) {
  return __ldg(g + (size_t)e * (scale_rows > 0 ? scale_rows : 1) + (scale_rows > 0 ? n : 0));
}

template <class Fmt, int BN_, bool GATEUP>
struct ExpertGemmWT {
  static constexpr int BN = BN_;
  static constexpr int NA = GATEUP ? 2 : 1;
  static constexpr int NBUF = 2 * NA * BN <= 256 ? 2 : 1;  // leave columns for the A stages
  static constexpr int KS = kWtTilesPerStep / NA;           // 64-wide K slices per step
  // stages of four A tiles: what tensor memory holds beside the accumulators (at most 4)
  static constexpr int AST_FIT = (512 - NBUF * NA * BN) / (kWtTilesPerStep * 32);
  static constexpr int AST = AST_FIT > 4 ? 4 : AST_FIT;
  static constexpr int RAW_BYTES = kWtTilesPerStep * Fmt::kTileBytes;
  // activation ring: up to 6 steps ahead (they come from L2 with a long
  // latency), in at most half the shared memory
  static constexpr int B_SLOT = KS * BN * kTileK * 2;
  static constexpr int BS_FIT = (kSmemLimit / 2) / B_SLOT;
  static constexpr int BS = BS_FIT > 6 ? 6 : BS_FIT < 2 ? 2 : BS_FIT;
  // raw ring: what shared memory holds beside the activation slots (at most 8 steps)
  static constexpr int RS_FIT =
      (kSmemLimit - 2048 - (int)sizeof(TileSched) - BS * KS * BN * kTileK * 2) / RAW_BYTES;
  static constexpr int RS = RS_FIT > 8 ? 8 : RS_FIT;
  static_assert(AST >= 2 && RS >= 2, "pipeline depth");
  static constexpr bool DYNAMIC = true;
  static constexpr bool PDL_PRIMARY = GATEUP;
  static constexpr bool PDL_SECONDARY = !GATEUP;

  using Params = WtParams;
  using Sched = TileSched;
  struct Tile {
    int row0, nrows, arow0, m, e, ntt;  // ntt: token tiles of expert e
  };

  __device__ static int box_rows(const Tile &t) { return t.nrows <= BN / 2 ? BN / 2 : BN; }
  __device__ static void prologue(const Params &p, Sched &s) {
    tile_sched_prologue(p.offsets, p.E, BN, 1, s);
  }
  __device__ static int num_tiles(const Params &p, const Sched &s) { return s.tp[p.E] * p.mt; }
  __device__ static Tile tile(const Params &p, const Sched &s, int t) {
    const int tti = t / p.mt, m = t - tti * p.mt;
    const int e = tile_sched_expert(s, p.E, tti);
    const int row0 = s.off[e] + (tti - s.tp[e]) * BN;
    return Tile{row0, min(BN, s.off[e + 1] - row0), e * p.w_rows + m * kTileM, m, e,
                s.tp[e + 1] - s.tp[e]};
  }
  __device__ static int num_steps(const Params &p, const Tile &) { return p.ksteps / KS; }
  __device__ static uint32_t b_tx_bytes(const Params &, const Tile &t) {
    return (uint32_t)(KS * box_rows(t) * kTileK * 2);
  }
  // the step's KS activation tiles, each BN rows x 64 k (128-byte swizzle)
  __device__ static void load_b(const Params &p, const Tile &t, int s, uint8_t *bslot,
                                uint64_t *bar) {
    const CUtensorMap *m = box_rows(t) == BN ? &p.tmap_b : &p.tmap_bh;
#pragma unroll
    for (int j = 0; j < KS; ++j)
      tma_load_2d(bslot + j * (BN * kTileK * 2), m, bar, (s * KS + j) * kTileK, t.row0);
  }
  // the step's four weight tiles, tile j * NA + a = slice j, matrix a
  __device__ static void load_raw(const Params &p, const Tile &t, int s, uint8_t *raw,
                                  uint64_t *bar) {
#pragma unroll
    for (int j = 0; j < KS; ++j) {
      const int k = s * KS + j;
#pragma unroll
      for (int a = 0; a < NA; ++a) {
        uint8_t *dst = raw + (j * NA + a) * Fmt::kTileBytes;
        if constexpr (Fmt::kTiled) {
          const uint8_t *w = a == 0 ? p.wt0 : p.wt1;
          bulk_load(dst, w + ((size_t)(t.arow0 / kTileM) * p.ktiles + k) * Fmt::kTileBytes,
                    Fmt::kTileBytes, bar);
        } else if constexpr (Fmt::kPerRowScale) {
          tma_load_2d(dst, a == 0 ? &p.tmap_q0 : &p.tmap_q1, bar, k * 64, t.arow0);
        } else {
          tma_load_2d(dst, a == 0 ? &p.tmap_q0 : &p.tmap_q1, bar, k * 32, t.arow0);
          tma_load_2d(dst + 128 * 32, a == 0 ? &p.tmap_s0 : &p.tmap_s1, bar, (k >> 2) * 16,
                      t.arow0);
        }
      }
    }
  }
  __device__ static void convert_row(const Params &, const Tile &, int s, const uint8_t *raw,
                                     int j, int a, int row, uint32_t (&out)[32]) {
    Fmt::convert(raw + (j * NA + a) * Fmt::kTileBytes, s * KS + j, row, out);
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
  __device__ static void epilogue(const Params &p, const Tile &t, uint32_t taddr, int row) {
    const int f = t.m * kTileM + row;  // output feature of this thread
    const float ga = wt_scale(p.g0, p.scale_rows, t.e, f);
    const float gb = GATEUP ? wt_scale(p.g1, p.scale_rows, t.e, f) : 0.f;
    for (int c = 0; c < t.nrows; c += 16) {
      uint32_t a[16];
      tmem_ld16(taddr + c, a);
      if (GATEUP) {
        uint32_t u[16];
        tmem_ld16(taddr + BN + c, u);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          if (c + j < t.nrows) {
            const float gv = __uint_as_float(a[j]) * ga;
            const float hv = gv / (1.0f + __expf(-gv)) * (__uint_as_float(u[j]) * gb);
            p.out[(size_t)(t.row0 + c + j) * p.out_cols + f] = __float2bfloat16_rn(hv);
          }
        }
      } else {
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          if (c + j < t.nrows) {
            const int r = t.row0 + c + j;
            const float w = __ldg(p.topk_w + __ldg(p.row_src + r)) * ga;
            p.out[(size_t)r * p.out_cols + f] = __float2bfloat16_rn(__uint_as_float(a[j]) * w);
          }
        }
      }
    }
  }
};

template <class P>
moe_status launch_wt(const WtParams &prm, int grid, cudaStream_t stream) {
  constexpr int smem = wt_smem_bytes<P>();
  static_assert(smem <= kSmemLimit, "shared memory budget");
  // the down GEMM runs as a programmatic dependent: its CTAs must never share
  // an SM with a gate/up CTA (each needs more than half the shared memory)
  static_assert(smem > kSmemLimit / 2, "dependent launch must not share SMs with its primary");
  if (ensure_smem_limit((const void *)wt_gemm_kernel<P>, smem) != MOE_OK) return MOE_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kWtThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = P::PDL_SECONDARY ? 1 : 0;
  if (cudaLaunchKernelEx(&cfg, wt_gemm_kernel<P>, prm) != cudaSuccess) return MOE_ERR_CUDA;
  return cudaPeekAtLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// Weight operands of one GEMM (w1/s1: W_up, or the same tensor again for down).
template <class Fmt>
bool wt_weights(WtParams &prm, const void *w0, const void *s0, const void *w1, const void *s1,
                int K, long rows) {
  if constexpr (Fmt::kTiled) {
    prm.wt0 = static_cast<const uint8_t *>(w0);
    prm.wt1 = static_cast<const uint8_t *>(w1);
    prm.ktiles = K / kTileK;
    return true;
  } else {
    prm.wt0 = prm.wt1 = nullptr;
    prm.ktiles = 0;
    const CUtensorMapDataType U8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
    if (Fmt::kPerRowScale)
      return make_tmap_2d(&prm.tmap_q0, w0, U8, 1, K, rows, 64, 128, false) &&
             make_tmap_2d(&prm.tmap_q1, w1, U8, 1, K, rows, 64, 128, false);
    return make_tmap_2d(&prm.tmap_q0, w0, U8, 1, K / 2, rows, 32, 128, false) &&
           make_tmap_2d(&prm.tmap_q1, w1, U8, 1, K / 2, rows, 32, 128, false) &&
           make_tmap_2d(&prm.tmap_s0, s0, U8, 1, K / 16, rows, 16, 128, false) &&
           make_tmap_2d(&prm.tmap_s1, s1, U8, 1, K / 16, rows, 16, 128, false);
  }
}

template <class Fmt, int BN>
moe_status launch_wt_bn(const moe_dims &d, const moe_experts &ex, const void *x_perm,
                        const int32_t *offsets, const int32_t *row_src, const float *topk_w,
                        void *y_partial, __nv_bfloat16 *h, uint32_t *status, cudaStream_t stream) {
  const long Tk = (long)d.T * d.top_k;
  const long max_tt = Tk / BN + std::min<long>(d.E, Tk);
  const int sms = device_sm_count();
  {
    WtParams prm{};
    const long rows = (long)d.E * d.I;
    if (!make_tmap_bf16_2d(&prm.tmap_b, x_perm, d.H, Tk, BN) ||
        !make_tmap_bf16_2d(&prm.tmap_bh, x_perm, d.H, Tk, BN / 2) ||
        !wt_weights<Fmt>(prm, ex.w_gate, ex.s_gate, ex.w_up, ex.s_up, d.H, rows))
      return MOE_ERR_CUDA;
    prm.g0 = ex.g_gate;
    prm.g1 = ex.g_up;
    prm.scale_rows = Fmt::kPerRowScale ? d.I : 0;
    prm.offsets = offsets;
    prm.row_src = row_src;
    prm.topk_w = topk_w;
    prm.out = h;
    prm.E = d.E;
    prm.out_cols = d.I;
    prm.w_rows = d.I;
    prm.ksteps = d.H / kTileK;
    prm.mt = d.I / kTileM;
    prm.status = status;
    prm.sched_counters = status + kSchedCounterWord;
    prm.expert_done = status + kExpertDoneWord;
    prm.up_mt = prm.mt;
    const int grid = (int)std::max<long>(1, std::min<long>(sms, max_tt * prm.mt));
    const moe_status st = launch_wt<ExpertGemmWT<Fmt, BN, true>>(prm, grid, stream);
    if (st != MOE_OK) return st;
  }
  {
    WtParams prm{};
    const long rows = (long)d.E * d.H;
    if (!make_tmap_bf16_2d(&prm.tmap_b, h, d.I, Tk, BN) ||
        !make_tmap_bf16_2d(&prm.tmap_bh, h, d.I, Tk, BN / 2) ||
        !wt_weights<Fmt>(prm, ex.w_down, ex.s_down, ex.w_down, ex.s_down, d.I, rows))
      return MOE_ERR_CUDA;
    prm.g0 = ex.g_down;
    prm.g1 = ex.g_down;
    prm.scale_rows = Fmt::kPerRowScale ? d.H : 0;
    prm.offsets = offsets;
    prm.row_src = row_src;
    prm.topk_w = topk_w;
    prm.out = static_cast<__nv_bfloat16 *>(y_partial);
    prm.E = d.E;
    prm.out_cols = d.H;
    prm.w_rows = d.H;
    prm.ksteps = d.I / kTileK;
    prm.mt = d.H / kTileM;
    prm.status = status;
    prm.sched_counters = status + kSchedCounterWord + 2;  // runs alongside gate/up's
    prm.expert_done = status + kExpertDoneWord;
    prm.up_mt = d.I / kTileM;
    const int grid = (int)std::max<long>(1, std::min<long>(sms, max_tt * prm.mt));
    return launch_wt<ExpertGemmWT<Fmt, BN, false>>(prm, grid, stream);
  }
}

template <class Fmt>
moe_status launch_wt_fmt(const moe_dims &d, const moe_experts &ex, const void *x_perm,
                         const int32_t *offsets, const int32_t *row_src, const float *topk_w,
                         void *y_partial, __nv_bfloat16 *h, uint32_t *status, cudaStream_t stream) {
  switch (expert_tile_rows(d)) {
    case 32: return launch_wt_bn<Fmt, 32>(d, ex, x_perm, offsets, row_src, topk_w, y_partial, h, status, stream);
    case 64: return launch_wt_bn<Fmt, 64>(d, ex, x_perm, offsets, row_src, topk_w, y_partial, h, status, stream);
    default: return launch_wt_bn<Fmt, 128>(d, ex, x_perm, offsets, row_src, topk_w, y_partial, h, status, stream);
  }
}

}  // namespace

// The K loops run in steps of four 64-wide slices per matrix pair (gate/up:
// 2 slices of H, down: 4 slices of I).
bool packed_wt_applies(const moe_dims &d) {
  return expert_tile_rows(d) <= kPackedWtMaxRows && d.H % 128 == 0 && d.I % 256 == 0;
}

moe_status launch_experts_packed_wt(const moe_dims &d, const moe_experts &ex, const void *x_perm,
                                    const int32_t *expert_offsets, const int32_t *row_src,
                                    const float *topk_w, void *y_partial, __nv_bfloat16 *h,
                                    uint32_t *status, cudaStream_t stream) {
  const bool tiled = ex.layout == MOE_LAYOUT_TILED;
  if (ex.dtype == MOE_W_FP8)
    return tiled ? launch_wt_fmt<WtFp8Tiled>(d, ex, x_perm, expert_offsets, row_src, topk_w,
                                             y_partial, h, status, stream)
                 : launch_wt_fmt<WtFp8>(d, ex, x_perm, expert_offsets, row_src, topk_w, y_partial,
                                        h, status, stream);
  if (ex.dtype == MOE_W_NVFP4)
    return tiled ? launch_wt_fmt<WtNvfp4Tiled>(d, ex, x_perm, expert_offsets, row_src, topk_w,
                                               y_partial, h, status, stream)
                 : launch_wt_fmt<WtNvfp4>(d, ex, x_perm, expert_offsets, row_src, topk_w,
                                          y_partial, h, status, stream);
  return MOE_ERR_NOT_IMPLEMENTED;
}

}  // namespace beam
