// Expert MLPs with packed NVFP4 or FP8 weights for small and mid-size batches:
// weights on the MMA's M side, dequantised straight into tensor memory
// (tc_gemm_wtmem.cuh), the expert's token rows on N.  Same block as
// experts.cu ("Hugging Face releases Beam ...", third paragraph: SwiGLU
// experts; "Reflection Releases Beam ...", section "Where Beam Saves and Where
// the Memory Bill Comes In": NVFP4 and FP8 checkpoints):
//   h = silu(X_e . W_gate[e]^T) * (X_e . W_up[e]^T)
//   y_partial = topk_w * (h . W_down[e]^T)
//
// Operands are f16 on both sides.  A weight e2m1 * e4m3 (at most six
// significant bits, in [2^-10, 2688]) or an e4m3 code is exact in f16: a
// converter thread dequantises one weight row of a 64-wide K slice, e2m1 (or
// e4m3) pairs to f16 pairs by the hardware conversion, times the f16 block
// scale (exact).  The activations keep bf16's range through one power-of-two
// scale per token row (rowscale.cuh): the epilogue multiplies each
// accumulator column by its row's inverse factor, together with the NVFP4
// global or the FP8 row scale.
//
// Tiles are taken from a global counter as in the bf16 weights-on-M GEMMs of
// experts.cu.  The gate/up epilogue writes bf16 h and gathers each row's
// largest |h|; a small kernel running beside gate/up (a programmatic
// dependent of it) rescales an expert's rows of h to f16 in place as soon as
// the expert's gate/up tiles are done, and publishes them; the down GEMM (a
// programmatic dependent of that kernel) starts as gate/up's CTAs leave
// their SMs and each down tile waits (bounded) for its expert's rows.
#include <cuda_fp16.h>

#include "moe_internal.cuh"
#include "rowscale.cuh"
#include "sched.cuh"
#include "tc_gemm_wtmem.cuh"

namespace beam {

namespace {

// Half h of one NVFP4 weight row of a 64-wide K slice: 16 code bytes (k 32h ..
// 32h + 31, even k in the low nibble) and the e4m3 scales of its two 16-k
// blocks (bytes 2h, 2h + 1 of `scales`) -> 16 f16 pairs.
__device__ __forceinline__ void nvfp4_half_f16(uint4 c, uint32_t scales, int h,
                                               uint32_t (&out)[16]) {
  uint32_t s16[2];
#pragma unroll
  for (int b = 0; b < 2; ++b) {
    const uint32_t byte = (scales >> (8 * (2 * h + b))) & 0xFFu;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(s16[b]) : "h"((uint16_t)(byte | (byte << 8))));
  }
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {  // word i: k 32h + 8i .. + 7, block i / 2 of the half
    uint32_t h0, h1, h2, h3;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
        : "r"(w[i]));
    const uint32_t sc = s16[i >> 1];
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(out[4 * i + 0]) : "r"(h0), "r"(sc));
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(out[4 * i + 1]) : "r"(h1), "r"(sc));
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(out[4 * i + 2]) : "r"(h2), "r"(sc));
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(out[4 * i + 3]) : "r"(h3), "r"(sc));
  }
}

// Half of one FP8 weight row of a 64-wide K slice: 32 e4m3 codes (two 16-byte
// vectors) -> 16 f16 pairs.
__device__ __forceinline__ void fp8_half_f16(const uint4 *codes, uint32_t (&out)[16]) {
#pragma unroll
  for (int v = 0; v < 2; ++v) {
    const uint4 q = codes[v];
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(out[8 * v + 2 * i]) : "h"((uint16_t)(w[i] & 0xFFFFu)));
      asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(out[8 * v + 2 * i + 1]) : "h"((uint16_t)(w[i] >> 16)));
    }
  }
}

// Rows of x_perm (bf16 [rows, K]) -> f16 rows scaled by a power of two each
// (see above); rscale[r] receives the inverse factor and hmax[r] is cleared
// for the gate/up epilogue's maxima.  dst may equal src (each value is read
// and written by one lane).  One warp per row.  Launched as an ordinary
// kernel; the gate/up GEMM is its programmatic dependent.
__global__ void __launch_bounds__(256) rows_f16_scaled_kernel(const __nv_bfloat16 *src,
                                                              __half *dst, int rows, int K,
                                                              float *rscale, uint32_t *hmax) {
  // the gate/up GEMM may start streaming weights; it reads x16 only after
  // this kernel has completed
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int r = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  const uint4 *s4 = reinterpret_cast<const uint4 *>(src + (size_t)r * K);
  uint4 *d4 = reinterpret_cast<uint4 *>(dst + (size_t)r * K);
  const int n4 = K / 8;
  uint32_t m = 0;  // largest |bf16| bit pattern of the lane's values (per half)
#pragma unroll 8
  for (int i = lane; i < n4; i += 32) m = bf16x8_absmax_bits(s4[i], m);
  m = max(m & 0xFFFFu, m >> 16);
  m = __reduce_max_sync(0xffffffffu, m);
  const int sx = row_scale_exp(m >> 7);  // bf16 and fp32 share the exponent field
  const float sc = ldexpf(1.0f, sx);
#pragma unroll 8
  for (int i = lane; i < n4; i += 32) d4[i] = bf16x8_to_f16x8_scaled(s4[i], sc);
  if (lane == 0) {
    rscale[r] = ldexpf(1.0f, -sx);
    hmax[r] = 0u;
  }
}

// Rows of h (bf16 [Tk, K], in place) -> f16 scaled by the power of two that
// their largest magnitude hmax[r] (fp32 bits, gathered by the gate/up
// epilogue) asks for; hscale[r] receives the inverse factor.  A programmatic
// dependent of the gate/up GEMM that runs beside it: CTA b takes experts b,
// b + grid, ...; for each it waits (bounded) until every gate/up epilogue
// warp of the expert has counted (4 per feature tile and token tile of bn
// rows), rescales the expert's rows (one warp per row, four warps) and counts
// once more, which publishes them to the down GEMM's TMA reads.
__global__ void __launch_bounds__(128) h_rows_f16_scaled_kernel(
    __nv_bfloat16 *h, const int32_t *offsets, int E, int K, int bn, int up_mt,
    const uint32_t *hmax, float *hscale, uint32_t *expert_done, uint32_t *status) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ int ok;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int e = blockIdx.x; e < E; e += gridDim.x) {
    const int r0 = __ldg(offsets + e), r1 = __ldg(offsets + e + 1);
    if (r1 == r0) continue;
    if (threadIdx.x == 0) {
      const uint32_t need = 4u * (uint32_t)up_mt * (uint32_t)((r1 - r0 + bn - 1) / bn);
      ok = 1;
      if (ld_acquire_gpu(expert_done + e) < need) {
        const uint64_t t0 = global_timer_ns();
        while (ld_acquire_gpu(expert_done + e) < need) {
          if (ld_acquire_gpu(status) & (uint32_t)MOE_DEV_TIMEOUT) {
            ok = 0;  // a GEMM gave up: so does this
            break;
          }
          if (global_timer_ns() - t0 > kWaitLimitNs) {
            atomicOr(status, (uint32_t)MOE_DEV_TIMEOUT);
            ok = 0;
            break;
          }
          __nanosleep(200);
        }
      }
    }
    __syncthreads();
    if (!ok) return;
    for (int r = r0 + warp; r < r1; r += 4) {
      const float inv = rescale_row_inplace(h + (size_t)r * K, K, __ldcg(hmax + r), lane);
      if (lane == 0) hscale[r] = inv;
    }
    asm volatile("fence.proxy.async.global;" ::: "memory");
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      atomicAdd(expert_done + e, 1u);
    }
  }
}

// Raw layouts of one 128-row A tile of a K slice in a ring slot, per format.
// A converter thread first loads all its row's packed bytes into registers
// (load), then converts the row in two halves of 32 k (convert).
struct WtRow {
  uint4 q[4];   // NVFP4: q[0..1] = 32 code bytes; FP8: 64 code bytes
  uint32_t sc;  // NVFP4: the four e4m3 block scales of the slice
};
// Row-major NVFP4 arrives as TMA boxes: codes [128][32 B], then scale boxes
// [128][16 B] (the 16 scales of 256 k; this slice's four at (k % 4) * 4).
struct WtNvfp4 {
  static constexpr bool kTiled = false, kPerRowScale = false;
  static constexpr int kTileBytes = 128 * 48;
  __device__ static void load(const uint8_t *t, int k, int r, WtRow &w) {
    w.q[0] = reinterpret_cast<const uint4 *>(t + r * 32)[0];
    w.q[1] = reinterpret_cast<const uint4 *>(t + r * 32)[1];
    w.sc = *reinterpret_cast<const uint32_t *>(t + 128 * 32 + r * 16 + (k & 3) * 4);
  }
  __device__ static void convert(const WtRow &w, int h, uint32_t (&out)[16]) {
    nvfp4_half_f16(w.q[h], w.sc, h, out);
  }
};
// Tiled NVFP4 (moe_pack_nvfp4): codes [128][32 B], then scales [128][4 B].
struct WtNvfp4Tiled : WtNvfp4 {
  static constexpr bool kTiled = true;
  static constexpr int kTileBytes = 4608;
  __device__ static void load(const uint8_t *t, int, int r, WtRow &w) {
    w.q[0] = reinterpret_cast<const uint4 *>(t + r * 32)[0];
    w.q[1] = reinterpret_cast<const uint4 *>(t + r * 32)[1];
    w.sc = *reinterpret_cast<const uint32_t *>(t + 128 * 32 + r * 4);
  }
};
// FP8, row-major (TMA box) or tiled (moe_pack_fp8): codes [128][64 B].
struct WtFp8 {
  static constexpr bool kTiled = false, kPerRowScale = true;
  static constexpr int kTileBytes = 8192;
  __device__ static void load(const uint8_t *t, int, int r, WtRow &w) {
#pragma unroll
    for (int v = 0; v < 4; ++v) w.q[v] = reinterpret_cast<const uint4 *>(t + r * 64)[v];
  }
  __device__ static void convert(const WtRow &w, int h, uint32_t (&out)[16]) {
    fp8_half_f16(&w.q[2 * h], out);
  }
};
struct WtFp8Tiled : WtFp8 {
  static constexpr bool kTiled = true;
};

struct WtParams {
  CUtensorMap tmap_b;    // scaled f16 token rows [Tk, K] (x16 or h), box {64, BN}
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
  const float *bscale;  // [Tk] inverse row factor of the B operand (x16 or h)
  uint32_t *hmax;       // [Tk] gate/up: largest |h| of each row (fp32 bits)
  int E, out_cols, w_rows, ksteps, mt;
  uint32_t *status;
  uint32_t *sched_counters;  // dynamic tile schedule (workspace header)
  uint32_t *expert_done;     // [E] gate/up epilogue warps done per expert (workspace header)
  int up_mt;                 // gate/up feature tiles per token tile
};

__device__ __forceinline__ float wt_scale(const float *g, int scale_rows, int e, int n) {
  return __ldg(g + (size_t)e * (scale_rows > 0 ? scale_rows : 1) + (scale_rows > 0 ? n : 0));
}

template <class Fmt, int BN_, bool GATEUP>
struct ExpertGemmWT {
  static constexpr int BN = BN_;
  static constexpr int NA = GATEUP ? 2 : 1;
  // two accumulator sets only while three A stages still fit beside them: the
  // converters are the bound, and with two stages they wait for the MMA to
  // free one every step
  static constexpr int NBUF = 512 - 2 * NA * BN >= 3 * kWtTilesPerStep * 32 ? 2 : 1;
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
  // raw ring: what shared memory holds beside the activation slots (at most 8
  // steps), leaving 2 KB of the SM free so that a CTA of the h rescaling
  // kernel fits beside this one
  static constexpr int RS_FIT =
      (kSmemLimit - 2048 - (int)sizeof(TileSched) - BS * KS * BN * kTileK * 2 - 2048) / RAW_BYTES;
  static constexpr int RS = RS_FIT > 8 ? 8 : RS_FIT;
  static_assert(AST >= 2 && RS >= 2, "pipeline depth");
  static constexpr bool DYNAMIC = true;
  // every launch of the chain x16 rescaling -> gate/up -> h rescaling -> down
  // is a programmatic dependent of the one before: gate/up reads x16 after
  // waiting for its kernel to complete, down each expert's h once published
  static constexpr bool PDL_PRIMARY = true;
  static constexpr bool PDL_SECONDARY = true;
  static constexpr bool PDL_WAIT_B = GATEUP;

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
  using Row = WtRow;
  __device__ static void load_row(const Params &, const Tile &, int s, const uint8_t *raw, int j,
                                  int a, int row, Row &w) {
    Fmt::load(raw + (j * NA + a) * Fmt::kTileBytes, s * KS + j, row, w);
  }
  __device__ static void convert_half(const Row &w, int h, uint32_t (&out)[16]) {
    Fmt::convert(w, h, out);
  }
  // gate/up: each epilogue warp counts its 32 features of h for the tile (its
  // stores and row maxima before the count); the h rescaling kernel waits for
  // the expert's count to complete
  __device__ static void tile_done(const Params &p, const Tile &t) {
    if constexpr (GATEUP) {
      __threadfence();
      atomicAdd(p.expert_done + t.e, 1u);
    }
  }
  // down: wait until the rescaling kernel has published the expert's f16 h
  // rows (one count beyond the gate/up warps'), then order the TMA reads of h
  // after that
  __device__ static bool tile_ready(const Params &p, const Tile &t, volatile int *abort) {
    if constexpr (GATEUP) {
      return true;
    } else {
      const uint32_t need = 4u * (uint32_t)p.up_mt * (uint32_t)t.ntt + 1u;
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
  // Accumulator column n is token row row0 + n scaled by the row's factor:
  // multiplied back by bscale first (exact), then by the weight scales.  Lane
  // l loads the factors of rows row0 + l, row0 + 32 + l, ... once per tile;
  // each column takes them from its lane with a shuffle.
  __device__ static void epilogue(const Params &p, const Tile &t, uint32_t taddr, int row) {
    constexpr int NG = BN / 32;  // 32-row groups of the tile
    const int f = t.m * kTileM + row;  // output feature of this thread
    const int lane = row & 31;
    const float ga = wt_scale(p.g0, p.scale_rows, t.e, f);
    const float gb = GATEUP ? wt_scale(p.g1, p.scale_rows, t.e, f) : 0.f;
    float bs_l[NG], tw_l[NG];
#pragma unroll
    for (int i = 0; i < NG; ++i) {
      const int n = i * 32 + lane;
      bs_l[i] = tw_l[i] = 0.f;
      if (n < t.nrows) {
        const int r = t.row0 + n;
        bs_l[i] = __ldcg(p.bscale + r);
        if (!GATEUP) tw_l[i] = __ldg(p.topk_w + __ldg(p.row_src + r));
      }
    }
#pragma unroll
    for (int i = 0; i < NG; ++i) {
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int c = i * 32 + hf * 16;
        if (c >= t.nrows) break;
        uint32_t a[16];
        tmem_ld16(taddr + c, a);
        if (GATEUP) {
          uint32_t u[16];
          tmem_ld16(taddr + BN + c, u);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float bs = __shfl_sync(0xffffffffu, bs_l[i], hf * 16 + j);
            uint32_t mag = 0;
            if (c + j < t.nrows) {
              const float gv = __uint_as_float(a[j]) * bs * ga;
              const float hv = gv / (1.0f + __expf(-gv)) * (__uint_as_float(u[j]) * bs * gb);
              const __nv_bfloat16 hb = __float2bfloat16_rn(hv);
              p.out[(size_t)(t.row0 + c + j) * p.out_cols + f] = hb;
              mag = __float_as_uint(fabsf(__bfloat162float(hb)));
            }
            // the row's largest |h| over this warp's 32 features, one atomic per row
            mag = __reduce_max_sync(0xffffffffu, mag);
            if (lane == j && c + j < t.nrows) atomicMax(p.hmax + t.row0 + c + j, mag);
          }
        } else {
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float bs = __shfl_sync(0xffffffffu, bs_l[i], hf * 16 + j);
            const float w = __shfl_sync(0xffffffffu, tw_l[i], hf * 16 + j) * ga;
            if (c + j < t.nrows)
              p.out[(size_t)(t.row0 + c + j) * p.out_cols + f] =
                  __float2bfloat16_rn(__uint_as_float(a[j]) * bs * w);
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
  cfg.numAttrs = 1;
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
                        void *y_partial, const PackedWtScratch &scr, uint32_t *status,
                        cudaStream_t stream) {
  const long Tk = (long)d.T * d.top_k;
  const long max_tt = Tk / BN + std::min<long>(d.E, Tk);
  const int sms = device_sm_count();
  __nv_bfloat16 *h = static_cast<__nv_bfloat16 *>(scr.h);
  if (launch_rows_f16_scaled(x_perm, scr.x16, Tk, d.H, scr.xscale, scr.hmax, stream) != MOE_OK)
    return MOE_ERR_CUDA;
  // the tensor maps only move 2-byte elements: the bf16 maps serve the f16 rows
  {
    WtParams prm{};
    const long rows = (long)d.E * d.I;
    if (!make_tmap_bf16_2d(&prm.tmap_b, scr.x16, d.H, Tk, BN) ||
        !make_tmap_bf16_2d(&prm.tmap_bh, scr.x16, d.H, Tk, BN / 2) ||
        !wt_weights<Fmt>(prm, ex.w_gate, ex.s_gate, ex.w_up, ex.s_up, d.H, rows))
      return MOE_ERR_CUDA;
    prm.g0 = ex.g_gate;
    prm.g1 = ex.g_up;
    prm.scale_rows = Fmt::kPerRowScale ? d.I : 0;
    prm.offsets = offsets;
    prm.row_src = row_src;
    prm.topk_w = topk_w;
    prm.out = h;
    prm.bscale = scr.xscale;
    prm.hmax = scr.hmax;
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
    // h rows -> scaled f16 in place, expert by expert beside gate/up: one
    // CTA of 128 threads per SM fits beside a gate/up or a down CTA (registers)
    const int grid = std::max(1, std::min(sms, d.E));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(128);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, h_rows_f16_scaled_kernel, h, offsets, d.E, d.I, BN,
                           d.I / kTileM, (const uint32_t *)scr.hmax, scr.hscale,
                           status + kExpertDoneWord, status) != cudaSuccess ||
        cudaPeekAtLastError() != cudaSuccess)
      return MOE_ERR_CUDA;
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
    prm.bscale = scr.hscale;
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
                         void *y_partial, const PackedWtScratch &scr, uint32_t *status,
                         cudaStream_t stream) {
  switch (expert_tile_rows(d)) {
    case 32: return launch_wt_bn<Fmt, 32>(d, ex, x_perm, offsets, row_src, topk_w, y_partial, scr, status, stream);
    case 64: return launch_wt_bn<Fmt, 64>(d, ex, x_perm, offsets, row_src, topk_w, y_partial, scr, status, stream);
    default: return launch_wt_bn<Fmt, 128>(d, ex, x_perm, offsets, row_src, topk_w, y_partial, scr, status, stream);
  }
}

}  // namespace

moe_status launch_rows_f16_scaled(const void *x_perm, void *x16, long rows, int K, float *xscale,
                                  uint32_t *hmax, cudaStream_t stream) {
  if (rows == 0) return MOE_OK;
  rows_f16_scaled_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16 *>(x_perm), static_cast<__half *>(x16), (int)rows, K, xscale,
      hmax);
  return cudaPeekAtLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// The K loops run in steps of four 64-wide slices per matrix pair (gate/up:
// 2 slices of H, down: 4 slices of I).
bool packed_wt_applies(const moe_dims &d) {
  return expert_tile_rows(d) <= kPackedWtMaxRows && d.H % 128 == 0 && d.I % 256 == 0;
}

moe_status launch_experts_packed_wt(const moe_dims &d, const moe_experts &ex, const void *x_perm,
                                    const int32_t *expert_offsets, const int32_t *row_src,
                                    const float *topk_w, void *y_partial,
                                    const PackedWtScratch &scr, uint32_t *status,
                                    cudaStream_t stream) {
  const bool tiled = ex.layout == MOE_LAYOUT_TILED;
  if (ex.dtype == MOE_W_FP8)
    return tiled ? launch_wt_fmt<WtFp8Tiled>(d, ex, x_perm, expert_offsets, row_src, topk_w,
                                             y_partial, scr, status, stream)
                 : launch_wt_fmt<WtFp8>(d, ex, x_perm, expert_offsets, row_src, topk_w, y_partial,
                                        scr, status, stream);
  if (ex.dtype == MOE_W_NVFP4)
    return tiled ? launch_wt_fmt<WtNvfp4Tiled>(d, ex, x_perm, expert_offsets, row_src, topk_w,
                                               y_partial, scr, status, stream)
                 : launch_wt_fmt<WtNvfp4>(d, ex, x_perm, expert_offsets, row_src, topk_w,
                                          y_partial, scr, status, stream);
  return MOE_ERR_NOT_IMPLEMENTED;
}

}  // namespace beam
