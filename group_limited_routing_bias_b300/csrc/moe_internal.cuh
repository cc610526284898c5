// Declarations shared by the translation units of libbeam_moe.so: launch
// plans, the workspace layout, and tensor-map creation.
#pragma once

#include <algorithm>
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "beam_moe.h"

namespace beam {

constexpr int kTargetCtas = 148;       // B300 SM count; sizes the router's K split
constexpr int kPermuteChunk = 4096;    // entries per permute CTA (32 warps x 128)
constexpr size_t kHeaderBytes = 2048;  // workspace status header
// Header layout (uint32 words): [0] the device status word; [32..35] the
// counters of the dynamic tile schedule (next tile, finished CTAs) of the
// gate/up and the down GEMM; [64, 64 + E) per-expert counts of published
// gate/up tiles.  All zero between calls.
constexpr size_t kSchedCounterWord = 32;
constexpr size_t kExpertDoneWord = 64;
constexpr int kMaxRouterSplit = 60;    // router K split; the top-k kernel adds the partials

inline int ilog2(int v) {
  int r = 0;
  while ((1 << (r + 1)) <= v) ++r;
  return r;
}

// ------------------------------------------------------------------ plans

struct RouterPlan {
  int T, E, H;
  int BN;      // MMA N: next of 32/64/128/256 at or above E
  int ksplit;  // CTAs along K (partial sums added in order by the top-k kernel)
};

inline RouterPlan make_router_plan(const moe_dims &d) {
  RouterPlan p;
  p.T = d.T;
  p.E = d.E;
  p.H = d.H;
  p.BN = d.E <= 32 ? 32 : d.E <= 64 ? 64 : d.E <= 128 ? 128 : 256;
  const int mt = std::max(1, (d.T + 127) / 128);
  const int ksteps = 3 * d.H / 64;
  p.ksplit = std::max(1, std::min({kTargetCtas / mt, ksteps / 4, kMaxRouterSplit}));
  return p;
}

// Expert GEMM plan: N of the MMA (token rows per tile) from the mean rows per expert.
inline int expert_bn(const moe_dims &d) {
  const long rows = (long)d.T * d.top_k;
  const long mean = (rows + d.E - 1) / d.E;
  return mean <= 16 ? 16 : mean <= 32 ? 32 : mean <= 64 ? 64 : mean <= 128 ? 128 : 256;
}

// Token rows per tile of the bf16 weights-on-M GEMMs: twice the mean class up
// to 64, so an expert holding a few times the mean rows (common at decode,
// where the selection bias concentrates the load) still streams its weights
// once; a tile of at most half that loads a half-height activation box.  The
// wider MMAs cost little: these GEMMs are bound by the weight stream (an
// M = 128, N = 32 MMA takes 16 clocks, N = 16 nine).
inline int expert_tile_rows(const moe_dims &d) {
  const int bn = expert_bn(d);
  return bn <= 32 ? 2 * bn : bn;
}

// ------------------------------------------------------------------ workspace

struct WsLayout {
  size_t w3 = 0, partial = 0;                       // router
  size_t topk_idx = 0, topk_w = 0;                  // forward only
  size_t counts = 0, bases = 0;                     // permute
  size_t offsets = 0, slot_of = 0, row_src = 0, x_perm = 0;  // forward only
  size_t h = 0;                                     // experts
  size_t x16 = 0;                                   // experts, NVFP4 or FP8 only
  size_t xscale = 0, hmax = 0, hscale = 0;          // experts and forward, NVFP4 or FP8 only
  size_t xq = 0, xs = 0, hq = 0, hs = 0;            // experts and forward, W4A4 only
  size_t y_partial = 0;                             // forward only
  size_t total = 0;
};

inline WsLayout ws_layout(const moe_dims &d, moe_op op, moe_wdtype wdtype = MOE_W_BF16) {
  WsLayout L;
  size_t off = kHeaderBytes;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += (bytes + 255) & ~(size_t)255;
    return o;
  };
  const size_t Tk = (size_t)d.T * d.top_k;
  const bool fwd = op == MOE_OP_FORWARD;
  if (op == MOE_OP_ROUTE || fwd) {
    const RouterPlan rp = make_router_plan(d);
    L.w3 = take((size_t)d.E * 3 * d.H * 2);
    L.partial = take((size_t)rp.ksplit * d.T * d.E * 4);
  }
  if (fwd) {
    L.topk_idx = take(Tk * 4);
    L.topk_w = take(Tk * 4);
  }
  if (op == MOE_OP_PERMUTE || fwd) {
    const size_t nchunks = std::max<size_t>(1, (Tk + kPermuteChunk - 1) / kPermuteChunk);
    L.counts = take(nchunks * d.E * 4);
    L.bases = take(nchunks * d.E * 4);
  }
  const bool a4 = wdtype == MOE_W_NVFP4_A4;
  if (fwd) {
    L.offsets = take((size_t)(d.E + 1) * 4);
    L.slot_of = take(Tk * 4);
    L.row_src = take(Tk * 4);
    if (!a4) L.x_perm = take(Tk * d.H * 2);
  }
  if (a4 && (op == MOE_OP_EXPERTS || fwd)) {
    L.xq = take(Tk * d.H / 2);
    L.xs = take(Tk * d.H / 16);
    L.hq = take(Tk * d.I / 2);
    L.hs = take(Tk * d.I / 16);
  } else if (op == MOE_OP_EXPERTS || fwd) {
    L.h = take(Tk * d.I * 2);
  }
  if (op == MOE_OP_EXPERTS && wdtype != MOE_W_BF16 && !a4) L.x16 = take(Tk * d.H * 2);
  if ((op == MOE_OP_EXPERTS || fwd) && wdtype != MOE_W_BF16 && !a4) {
    L.xscale = take(Tk * 4);
    L.hmax = take(Tk * 4);
    L.hscale = take(Tk * 4);
  }
  if (fwd) L.y_partial = take(Tk * d.H * 2);
  L.total = off;
  return L;
}

// ------------------------------------------------------------------ tensor maps

// 2-D bf16 tensor [outer, inner] (inner contiguous), box {64, box_outer},
// 128-byte swizzle, zero fill out of bounds.
bool make_tmap_bf16_2d(CUtensorMap *map, const void *base, uint64_t inner, uint64_t outer,
                       uint32_t box_outer);

// Any 2-D tensor [outer, inner] with a {box_inner, box_outer} box; 128-byte
// swizzle or none; zero fill out of bounds.
bool make_tmap_2d(CUtensorMap *map, const void *base, CUtensorMapDataType dtype, int elem_bytes,
                  uint64_t inner, uint64_t outer, uint32_t box_inner, uint32_t box_outer,
                  bool swizzle128);

int device_sm_count();

// Raises `kernel`'s dynamic shared memory limit to `bytes` on the current
// device.  The attribute is per device, so this runs once per (kernel,
// device) pair; safe to call from several host threads.
moe_status ensure_smem_limit(const void *kernel, int bytes);

// ------------------------------------------------------------------ launchers

// logits (nullable): receives the fp32 logits [T, E] the selection is made from.
moe_status launch_route(const moe_dims &d, const void *x, const float *w_router, const float *bias,
                        int32_t *topk_idx, float *topk_w, const RouterPlan &rp,
                        __nv_bfloat16 *w3, float *partial, uint32_t *status, cudaStream_t stream,
                        float *logits = nullptr);

// What the dispatch does with x after sorting: copy rows in bf16, copy them
// as f16 scaled by a power of two per token (operands of the token-major
// packed-weight GEMMs, rowscale.cuh; xscale and hmax as for
// launch_rows_f16_scaled), or nothing (W4A4 quantises while gathering, in
// launch_quantize_nvfp4).
enum GatherMode { kGatherBf16 = 0, kGatherF16Scaled = 1, kGatherNone = 2 };

moe_status launch_permute(const moe_dims &d, const int32_t *topk_idx, const void *x, void *x_perm,
                          int32_t *expert_offsets, int32_t *slot_of, int32_t *row_src,
                          int32_t *counts, int32_t *bases, uint32_t *status, cudaStream_t stream,
                          GatherMode gather = kGatherBf16, float *xscale = nullptr,
                          uint32_t *hmax = nullptr);

// NVFP4 quantisation of bf16 rows.  With row_src, output row r (r < offsets[E],
// read on the device) is x[row_src[r] / top_k]; otherwise row r is x[r], r < rows.
moe_status launch_quantize_nvfp4(const void *x, const int32_t *row_src, const int32_t *offsets,
                                 int E, int top_k, int rows, int cols, float g, uint8_t *q,
                                 uint8_t *s, cudaStream_t stream);

// NVFP4 quantisation of bf16 token rows x [T, cols], each written to the
// permuted rows slot_of[t*top_k + j] (skipping -1): the forward's gather.
moe_status launch_quantize_scatter_nvfp4(const void *x, const int32_t *slot_of, int T, int top_k,
                                         int cols, float g, uint8_t *q, uint8_t *s,
                                         cudaStream_t stream);

// NVFP4 weights and activations: xq/xs the quantised permuted rows, hq/hs
// scratch for the quantised h.
moe_status launch_experts_w4a4(const moe_dims &d, const moe_experts &ex, const uint8_t *xq,
                               const uint8_t *xs, const int32_t *offsets, const int32_t *row_src,
                               const float *topk_w, void *y_partial, uint8_t *hq, uint8_t *hs,
                               uint32_t *status, cudaStream_t stream);

moe_status launch_experts(const moe_dims &d, const moe_experts &ex, const void *x_perm,
                          const int32_t *expert_offsets, const int32_t *row_src,
                          const float *topk_w, void *y_partial, __nv_bfloat16 *h,
                          uint32_t *status, cudaStream_t stream);


// NVFP4 or FP8 weights, small and mid-size batches: weights dequantised into
// tensor memory, token rows on the MMA's N side, f16 operands with one
// power-of-two scale per token row (experts_packed_wt.cu).  x_perm is bf16
// [Tk, H]; x16 receives its scaled f16 copy (may equal x_perm: converted in
// place); h [Tk, I] holds bf16 h, then its scaled f16 copy; xscale, hmax and
// hscale are [Tk] scratch.  Used while the token tiles hold at most
// kPackedWtMaxRows rows.
// x_perm rows (bf16 [rows, K]) -> x16 (f16, may equal x_perm) scaled by a
// power of two per row (rowscale.cuh); xscale[r] = the inverse factor, and
// hmax[r] cleared for the gate/up epilogues' row maxima of h.
moe_status launch_rows_f16_scaled(const void *x_perm, void *x16, long rows, int K, float *xscale,
                                  uint32_t *hmax, cudaStream_t stream);

struct PackedWtScratch {
  void *x16;
  void *h;
  float *xscale;
  uint32_t *hmax;
  float *hscale;
};
// NVFP4 or FP8 expert weights, the GEMMs with the dequantised weights in
// shared memory (experts_packed.cu; token-major tiles from 64 rows up): scr
// as above, with scr.x16 already holding the scaled f16 rows and xscale,
// hmax set (launch_rows_f16_scaled or the scaled gather).
moe_status launch_experts_fp4(const moe_dims &d, const moe_experts &ex,
                              const int32_t *expert_offsets, const int32_t *row_src,
                              const float *topk_w, void *y_partial, const PackedWtScratch &scr,
                              uint32_t *status, cudaStream_t stream);
constexpr int kPackedWtMaxRows = 64;
bool packed_wt_applies(const moe_dims &d);
moe_status launch_experts_packed_wt(const moe_dims &d, const moe_experts &ex, const void *x_perm,
                                    const int32_t *expert_offsets, const int32_t *row_src,
                                    const float *topk_w, void *y_partial,
                                    const PackedWtScratch &scr, uint32_t *status,
                                    cudaStream_t stream);

// bf16 [E, N, K] -> MMA-tiled layout (see moe_pack_bf16 in beam_moe.h).
moe_status launch_pack_bf16(int E, int N, int K, const void *src, void *dst, cudaStream_t stream);

// NVFP4 codes [E, N, K/2] + scales [E, N, K/16], or FP8 codes [E, N, K] -> the
// tiled layouts (see moe_pack_nvfp4 / moe_pack_fp8 in beam_moe.h).
moe_status launch_pack_nvfp4(int E, int N, int K, const uint8_t *q, const uint8_t *s, uint8_t *dst,
                             cudaStream_t stream);
moe_status launch_pack_fp8(int E, int N, int K, const uint8_t *q, uint8_t *dst, cudaStream_t stream);

// n bf16 values -> f16 (n even).

moe_status launch_combine(const moe_dims &d, const void *y_partial, const int32_t *slot_of, void *y,
                          cudaStream_t stream);

}  // namespace beam
