// Expert MLPs with packed low-precision weights ("Reflection Releases Beam
// ...", section "Where Beam Saves and Where the Memory Bill Comes In": BF16,
// FP8 and NVFP4 checkpoints; NVFP4 for Blackwell).
//   NVFP4: a weight is e2m1(code) * e4m3(block scale) * fp32 global, one scale
//          per 16 consecutive k, one global per expert and matrix.
//   FP8:   a weight is e4m3(code) * fp32 row scale, one scale per output row
//          (the pages give no FP8 layout; a per-row scale keeps the
//          dequantisation exact, since it factors out of the K sum).
// Both formats follow the same pipeline below; a format policy supplies the
// raw-slot layout, the raw loads, the converter and the epilogue scale.
//
// The activations stay 16-bit (W4A16).  The product e2m1 * e4m3 has at most
// six significant bits and lies in [2^-10, 2688], so it is exact in f16; the
// global scale, a per-matrix constant, is applied to the fp32 accumulator in
// the epilogue (for FP8 the row scale does the same job, and e4m3 is exact
// in f16).  The MMAs therefore run kind::f16 with f16 operands: the
// producer TMA-loads the packed codes and their scales into a deep raw ring,
// eight converter warps turn each 64-wide K slice into an f16 operand tile
// with the 128-byte swizzle (hardware e2m1x2 and e4m3x2 conversions, one
// f16x2 multiply per code pair) and free the raw slot at once, and the
// activations arrive by TMA as f16 rows scaled by a power of two each
// (rowscale.cuh): x_perm scaled in the dispatch gather, h written in bf16
// with its row maxima by the gate/up epilogue, then rescaled in place by a
// small kernel between the two GEMMs.  The epilogues multiply each row's
// inverse factor back into the accumulator.
//
// Two tile shapes: token rows on M with 256 weight rows on N (from 64 token
// rows per call up), and weights on M with the tokens on N for the smallest
// batches.  Both stream each touched expert's packed weights once per token
// tile.  (Batches whose expert tiles hold at most 64 rows run the
// tensor-memory GEMMs of experts_packed_wt.cu instead.)
#include <cuda_fp16.h>

#include "moe_internal.cuh"
#include "rowscale.cuh"
#include "sched.cuh"
#include "tc_gemm.cuh"

namespace beam {

namespace {

constexpr int kPackedRowBytes = kTileK / 2;  // NVFP4: 32 bytes of e2m1 pairs per row per K slice
constexpr int kScaleBoxBytes = 16;           // NVFP4: one scale box = 16 scales = 256 k = 4 K slices
constexpr int kFp8RowBytes = kTileK;         // FP8: 64 e4m3 codes per row per K slice

// Half of one 64-wide K slice of one weight row: 16 bytes of e2m1 pairs (even
// k in the low nibble) and the two e4m3 block scales that cover them -> 32 f16
// values, written as four 16-byte chunks (4*half .. 4*half+3) at the
// 128-byte-swizzle positions of row r.
__device__ __forceinline__ void fp4_half_row_to_f16(const uint8_t *packed16, uint32_t scales2,
                                                    uint8_t *dst_row, int r, int half) {
  const uint4 p = *reinterpret_cast<const uint4 *>(packed16);
  const uint32_t w[4] = {p.x, p.y, p.z, p.w};
  uint32_t s2[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const uint32_t b = (scales2 >> (8 * j)) & 0xFFu;
    const uint16_t pair = (uint16_t)(b | (b << 8));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(s2[j]) : "h"(pair));
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t o0, o1, o2, o3;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(o0), "=r"(o1), "=r"(o2), "=r"(o3)
        : "r"(w[i]));
    const uint32_t sc = s2[i >> 1];  // codes 8i..8i+7 of this half lie in block i/2
    asm("mul.rn.f16x2 %0, %0, %1;" : "+r"(o0) : "r"(sc));
    asm("mul.rn.f16x2 %0, %0, %1;" : "+r"(o1) : "r"(sc));
    asm("mul.rn.f16x2 %0, %0, %1;" : "+r"(o2) : "r"(sc));
    asm("mul.rn.f16x2 %0, %0, %1;" : "+r"(o3) : "r"(sc));
    const int chunk = 4 * half + i;
    *reinterpret_cast<uint4 *>(dst_row + ((chunk ^ (r & 7)) << 4)) = make_uint4(o0, o1, o2, o3);
  }
}

// Half of one 64-wide K slice of one FP8 weight row: 32 e4m3 codes -> 32 f16
// (exact), four 16-byte chunks at the swizzle positions of row r.
__device__ __forceinline__ void fp8_half_row_to_f16(const uint8_t *codes32, uint8_t *dst_row, int r,
                                                    int half) {
  const uint4 a = *reinterpret_cast<const uint4 *>(codes32);
  const uint4 b = *reinterpret_cast<const uint4 *>(codes32 + 16);
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {  // chunk i: codes 8i..8i+7 = words 2i, 2i+1
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const uint32_t word = w[2 * i + j];
      asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(o[2 * j]) : "h"((uint16_t)(word & 0xFFFFu)));
      asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(o[2 * j + 1]) : "h"((uint16_t)(word >> 16)));
    }
    const int chunk = 4 * half + i;
    *reinterpret_cast<uint4 *>(dst_row + ((chunk ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

struct Fp4Params;

// NVFP4: raw slot = codes [NW][32 B], then scale boxes [NW][16 B]; the epilogue
// scale is the expert's global.
struct Nvfp4Format {
  static constexpr bool kPerRowScale = false;
  static constexpr bool kTiled = false;
  static constexpr int kRawRowBytes = kPackedRowBytes + kScaleBoxBytes;
  template <int NW>
  __device__ static void load_rows(uint8_t *raw, int first_row, const CUtensorMap *q,
                                   const CUtensorMap *s, uint64_t *bar, int k, int wrow) {
    tma_load_2d(raw + first_row * kPackedRowBytes, q, bar, k * kPackedRowBytes, wrow);
    tma_load_2d(raw + NW * kPackedRowBytes + first_row * kScaleBoxBytes, s, bar,
                (k >> 2) * kScaleBoxBytes, wrow);
  }
  template <int NW, int NTHR>
  __device__ static void convert(const uint8_t *raw, uint8_t *dst, int k, int ctid) {
#pragma unroll
    for (int it = ctid; it < 2 * NW; it += NTHR) {
      const int r = it >> 1, half = it & 1;
      const uint32_t sc = *reinterpret_cast<const uint16_t *>(
          raw + NW * kPackedRowBytes + r * kScaleBoxBytes + (k & 3) * 4 + half * 2);
      fp4_half_row_to_f16(raw + r * kPackedRowBytes + half * 16, sc, dst + r * 128, r, half);
    }
  }
};

// FP8: raw slot = codes [NW][64 B]; the epilogue scale is per output row.
struct Fp8Format {
  static constexpr bool kPerRowScale = true;
  static constexpr bool kTiled = false;
  static constexpr int kRawRowBytes = kFp8RowBytes;
  template <int NW>
  __device__ static void load_rows(uint8_t *raw, int first_row, const CUtensorMap *q,
                                   const CUtensorMap *, uint64_t *bar, int k, int wrow) {
    tma_load_2d(raw + first_row * kFp8RowBytes, q, bar, k * kFp8RowBytes, wrow);
  }
  template <int NW, int NTHR>
  __device__ static void convert(const uint8_t *raw, uint8_t *dst, int, int ctid) {
#pragma unroll
    for (int it = ctid; it < 2 * NW; it += NTHR) {
      const int r = it >> 1, half = it & 1;
      fp8_half_row_to_f16(raw + r * kFp8RowBytes + half * 32, dst + r * 128, r, half);
    }
  }
};

// NVFP4, tiled layout (moe_pack_nvfp4): a raw slot holds NW / 128 whole tiles
// as they lie in HBM, each the 128 rows' codes [128][32 B] then their scales
// [128][4 B] (the four blocks of this K slice), loaded with one bulk copy per
// tile.
struct Nvfp4TiledFormat {
  static constexpr bool kPerRowScale = false;
  static constexpr bool kTiled = true;
  static constexpr int kRawRowBytes = kPackedRowBytes + 4;
  static constexpr int kTileBytes = kTileM * kRawRowBytes;  // 4608
  template <int NW, int NTHR>
  __device__ static void convert(const uint8_t *raw, uint8_t *dst, int, int ctid) {
#pragma unroll
    for (int it = ctid; it < 2 * NW; it += NTHR) {
      const int r = it >> 1, half = it & 1;
      const uint8_t *tile = raw + (r / kTileM) * kTileBytes;
      const int rr = r % kTileM;
      const uint32_t sc =
          *reinterpret_cast<const uint16_t *>(tile + kTileM * kPackedRowBytes + rr * 4 + half * 2);
      fp4_half_row_to_f16(tile + rr * kPackedRowBytes + half * 16, sc, dst + r * 128, r, half);
    }
  }
};

// FP8, tiled layout (moe_pack_fp8): a tile is [128][64 B], so NW / 128 tiles
// side by side are exactly the row-major raw slot and the converter is the
// same; only the load differs.
struct Fp8TiledFormat : Fp8Format {
  static constexpr bool kTiled = true;
  static constexpr int kTileBytes = kTileM * kFp8RowBytes;  // 8192
};

// Raw loads of one tiled weight block: the tile of 128-row block `rblk` and K
// slice k of a tiled tensor with `ktiles` K slices per row block.
template <class Fmt>
__device__ __forceinline__ void load_tile(uint8_t *raw, const uint8_t *w, int rblk, int ktiles,
                                          int k, uint64_t *bar) {
  bulk_load(raw, w + ((size_t)rblk * ktiles + k) * Fmt::kTileBytes, Fmt::kTileBytes, bar);
}

__device__ __forceinline__ uint32_t pack_bf16x2_(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&v);
}

template <int CH>
__device__ __forceinline__ void tmem_ld_n(uint32_t taddr, uint32_t (&r)[CH]);
template <>
__device__ __forceinline__ void tmem_ld_n<32>(uint32_t taddr, uint32_t (&r)[32]) {
  tmem_ld32(taddr, r);
}
template <>
__device__ __forceinline__ void tmem_ld_n<16>(uint32_t taddr, uint32_t (&r)[16]) {
  tmem_ld16(taddr, r);
}

struct Fp4Params {
  CUtensorMap tmap_act;  // f16 token rows [Tk, K] (x or h), 128-byte swizzle
  CUtensorMap tmap_act32, tmap_act64;  // token-major tiles: the same rows, 32- and 64-row boxes
  CUtensorMap tmap_q0;   // packed codes [E*N, K/2] of W_gate or W_down
  CUtensorMap tmap_q1;   // packed codes of W_up (gate/up only)
  CUtensorMap tmap_s0;   // e4m3 scales [E*N, K/16] of W_gate or W_down
  CUtensorMap tmap_s1;   // scales of W_up
  const uint8_t *wt0;    // tiled layouts: tiles of W_gate or W_down (the maps above unused)
  const uint8_t *wt1;    // tiles of W_up (gate/up only)
  int ktiles;            // tiled layouts: K slices per 128-row block
  const float *g0;       // NVFP4: global scales [E] (gate or down); FP8: row scales [E, N]
  const float *g1;       // the same for up
  int scale_rows;        // N for FP8 row scales (index e * N + n), 0 for NVFP4 (index e)
  const int32_t *offsets;
  const int32_t *row_src;
  const float *topk_w;
  void *out;  // h bf16 [Tk, I] or y_partial bf16 [Tk, H]
  const float *bscale;  // [Tk] inverse row factor of the activations (x16 or h, rowscale.cuh)
  uint32_t *hmax;       // [Tk] gate/up: largest |h| of each row (fp32 bits)
  int E, out_cols, w_rows, ksteps, mt;
  uint32_t *status;
};

// ---------------------------------------------------------------- weights on M (small batches)

__device__ __forceinline__ float weight_scale(const float *g, int scale_rows, int e, int n) {
  return __ldg(g + (size_t)e * (scale_rows > 0 ? scale_rows : 1) + (scale_rows > 0 ? n : 0));
}

template <class Fmt, int BN_, bool GATEUP>
struct ExpertGemmFP4 {
  static constexpr int BN = BN_;
  static constexpr int NA = GATEUP ? 2 : 1;
  static constexpr int NW = NA * kTileM;  // weight rows dequantised per stage
  static constexpr bool CONVERT = true;
  static constexpr int CONVERT_WARPS = 8;
  static constexpr int CGROUPS = 1;
  static constexpr bool F16 = true;
  static constexpr int RAW_BYTES = NW * Fmt::kRawRowBytes;
  static constexpr int TX_BYTES = BN * kTileK * 2;  // the activation tile; raw bytes on their own ring
  static constexpr int NBUF = (2 * NA * BN <= 512) ? 2 : 1;
  static constexpr int OPERAND_BYTES = StageGeom<BN, NA>::kBytes;
  static constexpr int STAGES = OPERAND_BYTES * 3 <= 110 * 1024 ? 3 : 2;
  static constexpr int RSTAGES_FIT =
      (kSmemLimit - kSmemReserve - (int)sizeof(TileSched) - STAGES * OPERAND_BYTES) / RAW_BYTES;
  static constexpr int RSTAGES = (RSTAGES_FIT > 16 ? 16 : RSTAGES_FIT) / CGROUPS * CGROUPS;
  static_assert(RSTAGES >= 2, "raw ring needs two slots");

  using Params = Fp4Params;
  using Sched = TileSched;
  struct Tile {
    int row0, nrows, arow0, m, e;
  };

  __device__ static void prologue(const Params &p, Sched &s) { tile_sched_prologue(p.offsets, p.E, BN, 1, s); }
  __device__ static int num_tiles(const Params &p, const Sched &s) { return s.tp[p.E] * p.mt; }
  __device__ static Tile tile(const Params &p, const Sched &s, int t) {
    const int tti = t / p.mt, m = t - tti * p.mt;
    const int e = tile_sched_expert(s, p.E, tti);
    const int row0 = s.off[e] + (tti - s.tp[e]) * BN;
    return Tile{row0, min(BN, s.off[e + 1] - row0), e * p.w_rows + m * kTileM, m, e};
  }
  __device__ static int num_k(const Params &p, const Tile &) { return p.ksteps; }
  __device__ static void load(const Params &p, const Tile &t, int k, uint8_t *stage, uint64_t *bar) {
    tma_load_2d(stage + NA * kATileBytes, &p.tmap_act, bar, k * kTileK, t.row0);
  }
  __device__ static void load_raw(const Params &p, const Tile &t, int k, uint8_t *raw,
                                  uint64_t *raw_bar) {
    if constexpr (Fmt::kTiled) {
      load_tile<Fmt>(raw, p.wt0, t.arow0 / kTileM, p.ktiles, k, raw_bar);
      if (GATEUP) load_tile<Fmt>(raw + Fmt::kTileBytes, p.wt1, t.arow0 / kTileM, p.ktiles, k, raw_bar);
    } else {
      Fmt::template load_rows<NW>(raw, 0, &p.tmap_q0, &p.tmap_s0, raw_bar, k, t.arow0);
      if (GATEUP)
        Fmt::template load_rows<NW>(raw, kTileM, &p.tmap_q1, &p.tmap_s1, raw_bar, k, t.arow0);
    }
  }
  __device__ static void convert(const Params &, const Tile &, int k, uint8_t *stage,
                                 const uint8_t *raw, int ctid) {
    // A tiles: gate rows 0..127, up rows 128..255; a converter group per slice
    Fmt::template convert<NW, 32 * CONVERT_WARPS / CGROUPS>(raw, stage, k, ctid);
  }
  __device__ static void epilogue(const Params &p, const Tile &t, uint32_t taddr, int row) {
    constexpr int CH = BN < 32 ? BN : 32;
    const int f = t.m * kTileM + row;
    const float ga = weight_scale(p.g0, p.scale_rows, t.e, f);
    const float gb = GATEUP ? weight_scale(p.g1, p.scale_rows, t.e, f) : 0.f;
    for (int c = 0; c < t.nrows; c += CH) {
      uint32_t a[CH];
      tmem_ld_n<CH>(taddr + c, a);
      if (GATEUP) {
        uint32_t u[CH];
        tmem_ld_n<CH>(taddr + BN + c, u);
        tmem_wait_ld();
        __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(p.out);
#pragma unroll
        for (int j = 0; j < CH; ++j) {
          uint32_t mag = 0;
          if (c + j < t.nrows) {
            const int r = t.row0 + c + j;
            const float bs = __ldg(p.bscale + r);
            const float gv = __uint_as_float(a[j]) * bs * ga;
            const float hv = gv / (1.0f + __expf(-gv)) * (__uint_as_float(u[j]) * bs * gb);
            const __nv_bfloat16 hb = __float2bfloat16_rn(hv);
            out[(size_t)r * p.out_cols + f] = hb;
            mag = __float_as_uint(fabsf(__bfloat162float(hb)));
          }
          // the row's largest |h| over this warp's 32 features, one atomic per row
          mag = __reduce_max_sync(0xffffffffu, mag);
          if ((row & 31) == j && c + j < t.nrows) atomicMax(p.hmax + t.row0 + c + j, mag);
        }
      } else {
        tmem_wait_ld();
        __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(p.out);
#pragma unroll
        for (int j = 0; j < CH; ++j) {
          if (c + j < t.nrows) {
            const int r = t.row0 + c + j;
            const float w = __ldg(p.topk_w + __ldg(p.row_src + r)) * ga;
            out[(size_t)r * p.out_cols + f] =
                __float2bfloat16_rn(__uint_as_float(a[j]) * __ldg(p.bscale + r) * w);
          }
        }
      }
    }
  }
};

// ---------------------------------------------------------------- token rows on M (large batches)

template <class Fmt, bool GATEUP>
struct ExpertGemmTMFP4 {
  static constexpr int BN = 256;
  static constexpr int NA = 1;
  static constexpr int NW = 256;
  static constexpr int CGROUPS = 2;  // two converter groups on alternate K slices
  static constexpr bool CONVERT = true;
  static constexpr bool F16 = true;
  static constexpr int RAW_BYTES = NW * Fmt::kRawRowBytes;
  static constexpr int NBUF = 2;
  static constexpr int STAGES = 3;
  static constexpr int RSTAGES_FIT = (kSmemLimit - kSmemReserve - (int)sizeof(TileSched) -
                                      STAGES * StageGeom<BN, NA>::kBytes) / RAW_BYTES;
  static constexpr int RSTAGES = (RSTAGES_FIT > 16 ? 16 : RSTAGES_FIT) / CGROUPS * CGROUPS;
  static_assert(RSTAGES >= 2, "raw ring needs two slots");
  static constexpr int FW = GATEUP ? 128 : 256;
  // gate/up -> h rescaling -> down, each a programmatic dependent of the one
  // before: down streams and converts weights at once, its activation
  // producer waits for the rescaled h
  static constexpr bool PDL_PRIMARY = GATEUP;
  static constexpr bool PDL_SECONDARY = !GATEUP;
  static constexpr bool PDL_WAIT_B = !GATEUP;

  using Params = Fp4Params;
  using Sched = TileSched;
  struct Tile {
    int row0, nrows, brow0, f, e;
  };

  __device__ static void prologue(const Params &p, Sched &s) {
    tile_sched_prologue(p.offsets, p.E, kTileM, p.mt, s);
  }
  __device__ static int num_tiles(const Params &p, const Sched &s) { return s.tp[p.E]; }
  __device__ static Tile tile(const Params &p, const Sched &s, int t) {
    const int e = tile_sched_expert(s, p.E, t);
    const int ntt = (s.off[e + 1] - s.off[e] + kTileM - 1) / kTileM;
    const int local = t - s.tp[e];
    const int f = local / ntt, tt = local - f * ntt;
    const int row0 = s.off[e] + tt * kTileM;
    return Tile{row0, min(kTileM, s.off[e + 1] - row0), e * p.w_rows + f * FW, f, e};
  }
  __device__ static int num_k(const Params &p, const Tile &) { return p.ksteps; }
  __device__ static uint32_t tx_bytes(const Params &, const Tile &t) {
    return act_box_rows(t.nrows) * kTileK * 2;
  }
  __device__ static void load(const Params &p, const Tile &t, int k, uint8_t *stage, uint64_t *bar) {
    const int ar = act_box_rows(t.nrows);
    tma_load_2d(stage, ar == 32 ? &p.tmap_act32 : ar == 64 ? &p.tmap_act64 : &p.tmap_act, bar,
                k * kTileK, t.row0);
  }
  __device__ static void load_raw(const Params &p, const Tile &t, int k, uint8_t *raw,
                                  uint64_t *raw_bar) {
    if constexpr (Fmt::kTiled) {
      // gate/up: the gate and up tiles of one 128-row block; down: two blocks
      const int rblk = t.brow0 / kTileM;
      load_tile<Fmt>(raw, p.wt0, rblk, p.ktiles, k, raw_bar);
      if (GATEUP) load_tile<Fmt>(raw + Fmt::kTileBytes, p.wt1, rblk, p.ktiles, k, raw_bar);
      else load_tile<Fmt>(raw + Fmt::kTileBytes, p.wt0, rblk + 1, p.ktiles, k, raw_bar);
    } else if (GATEUP) {
      Fmt::template load_rows<NW>(raw, 0, &p.tmap_q0, &p.tmap_s0, raw_bar, k, t.brow0);
      Fmt::template load_rows<NW>(raw, kTileM, &p.tmap_q1, &p.tmap_s1, raw_bar, k, t.brow0);
    } else {
      Fmt::template load_rows<NW>(raw, 0, &p.tmap_q0, &p.tmap_s0, raw_bar, k, t.brow0);
    }
  }
  __device__ static void convert(const Params &, const Tile &, int k, uint8_t *stage,
                                 const uint8_t *raw, int ctid) {
    // B tile: 256 weight rows; each converter group converts its own slices
    Fmt::template convert<NW, 32 * kConvertWarps / CGROUPS>(raw, stage + kATileBytes, k, ctid);
  }
  __device__ static void epilogue(const Params &p, const Tile &t, uint32_t taddr, int row) {
    const bool valid = row < t.nrows;
    const int n0 = t.f * FW;  // first output feature of the tile
    // this thread's token row: its inverse activation factor (rowscale.cuh;
    // for down written by the kernel this launch depends on: read from L2)
    const float bs = valid ? __ldcg(p.bscale + t.row0 + row) : 0.f;
    if (GATEUP) {
      __nv_bfloat16 *dst =
          static_cast<__nv_bfloat16 *>(p.out) + (size_t)(t.row0 + row) * p.out_cols + n0;
      float hmax = 0.f;
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
            const int n = n0 + c + 2 * j;
            const float g0 = __uint_as_float(g[2 * j]) * bs * weight_scale(p.g0, p.scale_rows, t.e, n);
            const float g1 =
                __uint_as_float(g[2 * j + 1]) * bs * weight_scale(p.g0, p.scale_rows, t.e, n + 1);
            const float h0 = g0 / (1.0f + __expf(-g0)) *
                             (__uint_as_float(u[2 * j]) * bs * weight_scale(p.g1, p.scale_rows, t.e, n));
            const float h1 = g1 / (1.0f + __expf(-g1)) *
                             (__uint_as_float(u[2 * j + 1]) * bs *
                              weight_scale(p.g1, p.scale_rows, t.e, n + 1));
            pk[j] = pack_bf16x2_(h0, h1);
            const __nv_bfloat162 hb = *reinterpret_cast<const __nv_bfloat162 *>(&pk[j]);
            hmax = fmaxf(hmax, fmaxf(fabsf(__low2float(hb)), fabsf(__high2float(hb))));
          }
          uint4 *d4 = reinterpret_cast<uint4 *>(dst + c);
#pragma unroll
          for (int q = 0; q < 4; ++q) d4[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        }
      }
      if (valid) atomicMax(p.hmax + t.row0 + row, __float_as_uint(hmax));
    } else {
      const float w = valid ? __ldg(p.topk_w + __ldg(p.row_src + t.row0 + row)) : 0.f;
      __nv_bfloat16 *dst =
          static_cast<__nv_bfloat16 *>(p.out) + (size_t)(t.row0 + row) * p.out_cols + n0;
#pragma unroll 1
      for (int c = 0; c < FW; c += 32) {
        uint32_t a[32];
        tmem_ld32(taddr + c, a);
        tmem_wait_ld();
        if (valid) {
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int n = n0 + c + 2 * j;
            pk[j] = pack_bf16x2_(
                __uint_as_float(a[2 * j]) * bs * w * weight_scale(p.g0, p.scale_rows, t.e, n),
                __uint_as_float(a[2 * j + 1]) * bs * w * weight_scale(p.g0, p.scale_rows, t.e, n + 1));
          }
          uint4 *d4 = reinterpret_cast<uint4 *>(dst + c);
#pragma unroll
          for (int q = 0; q < 4; ++q) d4[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        }
      }
    }
  }
};

// ---------------------------------------------------------------- host side

template <class P>
moe_status launch_fp4(const Fp4Params &prm, int grid, cudaStream_t stream) {
  constexpr int smem = smem_bytes_for<P>();
  static_assert(smem <= kSmemLimit, "shared memory budget");
  if (ensure_smem_limit((const void *)tc_gemm_kernel<P>, smem) != MOE_OK) return MOE_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads_for<P>());
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = PdlSecondaryOf<P>::value ? 1 : 0;
  if (cudaLaunchKernelEx(&cfg, tc_gemm_kernel<P>, prm) != cudaSuccess) return MOE_ERR_CUDA;
  return cudaPeekAtLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// Rows of h (bf16 [rows, K], in place) -> f16 scaled per row by the factor
// the gate/up epilogues' maxima ask for (rowscale.cuh); hscale[r] receives
// the inverse factor.  A programmatic dependent of gate/up: it lets the down
// GEMM's launch begin, then waits for gate/up to complete.  One warp per row.
__global__ void __launch_bounds__(256) h_rows_rescale_kernel(__nv_bfloat16 *h, long rows, int K,
                                                             const uint32_t *hmax, float *hscale) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const long nwarps = (long)gridDim.x * (blockDim.x >> 5);
  for (long r = (long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += nwarps) {
    const float inv = rescale_row_inplace(h + r * K, K, __ldcg(hmax + r), lane);
    if (lane == 0) hscale[r] = inv;
  }
}

moe_status launch_h_rescale(const moe_dims &d, const PackedWtScratch &scr, cudaStream_t stream) {
  const long Tk = (long)d.T * d.top_k;
  const int grid = (int)std::max<long>(1, std::min<long>((Tk + 7) / 8, (long)device_sm_count() * 8));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, h_rows_rescale_kernel, static_cast<__nv_bfloat16 *>(scr.h), Tk, d.I,
                         (const uint32_t *)scr.hmax, scr.hscale) != cudaSuccess)
    return MOE_ERR_CUDA;
  return cudaPeekAtLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

bool make_act_map(CUtensorMap *m, const void *base, int K, long rows, int box_rows) {
  return make_tmap_2d(m, base, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, K, rows, 64, box_rows, true);
}

// Raw-weight tensor maps of one weight tensor [rows, K]: NVFP4 codes [rows, K/2]
// and scales [rows, K/16]; FP8 codes [rows, K] (no scale map: row scales are
// read by the epilogue).
template <class Fmt>
bool make_weight_maps(CUtensorMap *q, CUtensorMap *s, const void *qp, const void *sp, int K,
                      long rows, int box_rows) {
  if (Fmt::kPerRowScale) {
    const bool ok = make_tmap_2d(q, qp, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K, rows, kFp8RowBytes,
                                 box_rows, false);
    *s = *q;
    return ok;
  }
  return make_tmap_2d(q, qp, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K / 2, rows, kPackedRowBytes,
                      box_rows, false) &&
         make_tmap_2d(s, sp, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K / 16, rows, kScaleBoxBytes,
                      box_rows, false);
}

// Weight operands of one GEMM: tensor maps of the row-major codes and scales
// (w1/s1: W_up, or the same tensor again for down), or the tiled pointers.
template <class Fmt>
bool set_weights(Fp4Params &prm, const void *w0, const void *s0, const void *w1, const void *s1,
                 int K, long rows, int box_rows) {
  if constexpr (Fmt::kTiled) {
    prm.wt0 = static_cast<const uint8_t *>(w0);
    prm.wt1 = static_cast<const uint8_t *>(w1);
    prm.ktiles = K / kTileK;
    return true;
  } else {
    prm.wt0 = prm.wt1 = nullptr;
    prm.ktiles = 0;
    if (!make_weight_maps<Fmt>(&prm.tmap_q0, &prm.tmap_s0, w0, s0, K, rows, box_rows)) return false;
    if (w1 == w0) {
      prm.tmap_q1 = prm.tmap_q0;
      prm.tmap_s1 = prm.tmap_s0;
      return true;
    }
    return make_weight_maps<Fmt>(&prm.tmap_q1, &prm.tmap_s1, w1, s1, K, rows, box_rows);
  }
}

Fp4Params base_params(const moe_dims &d, const int32_t *offsets, const int32_t *row_src,
                      const float *topk_w, uint32_t *status) {
  Fp4Params prm;
  prm.offsets = offsets;
  prm.row_src = row_src;
  prm.topk_w = topk_w;
  prm.E = d.E;
  prm.status = status;
  return prm;
}

template <class Fmt, int BN>
moe_status launch_packed_small(const moe_dims &d, const moe_experts &ex, const int32_t *offsets,
                               const int32_t *row_src, const float *topk_w, void *y_partial,
                               const PackedWtScratch &scr, uint32_t *status, cudaStream_t stream) {
  const long Tk = (long)d.T * d.top_k;
  const long max_tt = Tk / BN + std::min<long>(d.E, Tk);
  const int sms = device_sm_count();
  {
    Fp4Params prm = base_params(d, offsets, row_src, topk_w, status);
    const long rows = (long)d.E * d.I;
    if (!make_act_map(&prm.tmap_act, scr.x16, d.H, Tk, BN) ||
        !set_weights<Fmt>(prm, ex.w_gate, ex.s_gate, ex.w_up, ex.s_up, d.H, rows, kTileM))
      return MOE_ERR_CUDA;
    prm.g0 = ex.g_gate;
    prm.g1 = ex.g_up;
    prm.scale_rows = Fmt::kPerRowScale ? d.I : 0;
    prm.out = scr.h;
    prm.bscale = scr.xscale;
    prm.hmax = scr.hmax;
    prm.out_cols = d.I;
    prm.w_rows = d.I;
    prm.ksteps = d.H / kTileK;
    prm.mt = d.I / kTileM;
    const int grid = (int)std::max<long>(1, std::min<long>(sms, max_tt * prm.mt));
    const moe_status st = launch_fp4<ExpertGemmFP4<Fmt, BN, true>>(prm, grid, stream);
    if (st != MOE_OK) return st;
  }
  if (launch_h_rescale(d, scr, stream) != MOE_OK) return MOE_ERR_CUDA;
  {
    Fp4Params prm = base_params(d, offsets, row_src, topk_w, status);
    const long rows = (long)d.E * d.H;
    if (!make_act_map(&prm.tmap_act, scr.h, d.I, Tk, BN) ||
        !set_weights<Fmt>(prm, ex.w_down, ex.s_down, ex.w_down, ex.s_down, d.I, rows, kTileM))
      return MOE_ERR_CUDA;
    prm.g0 = ex.g_down;
    prm.g1 = ex.g_down;
    prm.scale_rows = Fmt::kPerRowScale ? d.H : 0;
    prm.out = y_partial;
    prm.bscale = scr.hscale;
    prm.out_cols = d.H;
    prm.w_rows = d.H;
    prm.ksteps = d.I / kTileK;
    prm.mt = d.H / kTileM;
    const int grid = (int)std::max<long>(1, std::min<long>(sms, max_tt * prm.mt));
    return launch_fp4<ExpertGemmFP4<Fmt, BN, false>>(prm, grid, stream);
  }
}

template <class Fmt>
moe_status launch_packed_large(const moe_dims &d, const moe_experts &ex, const int32_t *offsets,
                               const int32_t *row_src, const float *topk_w, void *y_partial,
                               const PackedWtScratch &scr, uint32_t *status, cudaStream_t stream) {
  const long Tk = (long)d.T * d.top_k;
  const long max_tt = Tk / kTileM + std::min<long>(d.E, Tk);
  const int sms = device_sm_count();
  {
    using P = ExpertGemmTMFP4<Fmt, true>;
    Fp4Params prm = base_params(d, offsets, row_src, topk_w, status);
    const long rows = (long)d.E * d.I;
    if (!make_act_map(&prm.tmap_act, scr.x16, d.H, Tk, kTileM) ||
        !make_act_map(&prm.tmap_act32, scr.x16, d.H, Tk, 32) ||
        !make_act_map(&prm.tmap_act64, scr.x16, d.H, Tk, 64) ||
        !set_weights<Fmt>(prm, ex.w_gate, ex.s_gate, ex.w_up, ex.s_up, d.H, rows, 128))
      return MOE_ERR_CUDA;
    prm.g0 = ex.g_gate;
    prm.g1 = ex.g_up;
    prm.scale_rows = Fmt::kPerRowScale ? d.I : 0;
    prm.out = scr.h;
    prm.bscale = scr.xscale;
    prm.hmax = scr.hmax;
    prm.out_cols = d.I;
    prm.w_rows = d.I;
    prm.ksteps = d.H / kTileK;
    prm.mt = d.I / P::FW;
    const int grid = (int)std::max<long>(1, std::min<long>(sms, max_tt * prm.mt));
    const moe_status st = launch_fp4<P>(prm, grid, stream);
    if (st != MOE_OK) return st;
  }
  if (launch_h_rescale(d, scr, stream) != MOE_OK) return MOE_ERR_CUDA;
  {
    using P = ExpertGemmTMFP4<Fmt, false>;
    Fp4Params prm = base_params(d, offsets, row_src, topk_w, status);
    const long rows = (long)d.E * d.H;
    if (!make_act_map(&prm.tmap_act, scr.h, d.I, Tk, kTileM) ||
        !make_act_map(&prm.tmap_act32, scr.h, d.I, Tk, 32) ||
        !make_act_map(&prm.tmap_act64, scr.h, d.I, Tk, 64) ||
        !set_weights<Fmt>(prm, ex.w_down, ex.s_down, ex.w_down, ex.s_down, d.I, rows, 256))
      return MOE_ERR_CUDA;
    prm.g0 = ex.g_down;
    prm.g1 = ex.g_down;
    prm.scale_rows = Fmt::kPerRowScale ? d.H : 0;
    prm.out = y_partial;
    prm.bscale = scr.hscale;
    prm.out_cols = d.H;
    prm.w_rows = d.H;
    prm.ksteps = d.I / kTileK;
    prm.mt = d.H / P::FW;
    const int grid = (int)std::max<long>(1, std::min<long>(sms, max_tt * prm.mt));
    return launch_fp4<P>(prm, grid, stream);
  }
}

template <class Fmt>
moe_status launch_packed(const moe_dims &d, const moe_experts &ex, const int32_t *offsets,
                         const int32_t *row_src, const float *topk_w, void *y_partial,
                         const PackedWtScratch &scr, uint32_t *status, cudaStream_t stream) {
  // Token-major tiles from 64 (token, expert) rows up: with the weights on N
  // one MMA covers 256 weight rows, and the converter groups keep two K slices
  // in flight.  Measured on B300 (expert stage, tiled NVFP4): 0.94 vs 1.07 ms
  // at T=64 (top-8), 1.35 vs 2.11 ms at T=256, 1.88 vs 3.61 ms at T=1024; the
  // weights-on-M tiles stay for the smallest batches (T=1: 0.14 vs 0.17 ms).
  if ((long)d.T * d.top_k >= 64 && d.H % 256 == 0)
    return launch_packed_large<Fmt>(d, ex, offsets, row_src, topk_w, y_partial, scr, status, stream);
  switch (expert_bn(d)) {
    case 16: return launch_packed_small<Fmt, 16>(d, ex, offsets, row_src, topk_w, y_partial, scr, status, stream);
    case 32: return launch_packed_small<Fmt, 32>(d, ex, offsets, row_src, topk_w, y_partial, scr, status, stream);
    case 64: return launch_packed_small<Fmt, 64>(d, ex, offsets, row_src, topk_w, y_partial, scr, status, stream);
    case 128: return launch_packed_small<Fmt, 128>(d, ex, offsets, row_src, topk_w, y_partial, scr, status, stream);
    default: return launch_packed_small<Fmt, 256>(d, ex, offsets, row_src, topk_w, y_partial, scr, status, stream);
  }
}

}  // namespace

moe_status launch_experts_fp4(const moe_dims &d, const moe_experts &ex,
                              const int32_t *expert_offsets, const int32_t *row_src,
                              const float *topk_w, void *y_partial, const PackedWtScratch &scr,
                              uint32_t *status, cudaStream_t stream) {
  const bool tiled = ex.layout == MOE_LAYOUT_TILED;
  if (ex.dtype == MOE_W_FP8)
    return tiled ? launch_packed<Fp8TiledFormat>(d, ex, expert_offsets, row_src, topk_w, y_partial,
                                                 scr, status, stream)
                 : launch_packed<Fp8Format>(d, ex, expert_offsets, row_src, topk_w, y_partial, scr,
                                            status, stream);
  return tiled ? launch_packed<Nvfp4TiledFormat>(d, ex, expert_offsets, row_src, topk_w, y_partial,
                                                 scr, status, stream)
               : launch_packed<Nvfp4Format>(d, ex, expert_offsets, row_src, topk_w, y_partial, scr,
                                            status, stream);
}

}  // namespace beam
