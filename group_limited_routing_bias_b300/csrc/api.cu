// C ABI of libbeam_moe.so (declared in include/beam_moe.h): argument checks,
// workspace carving, tensor-map encoding, and the launch sequence of each
// entry point.  Every check happens before the first launch; nothing here
// allocates device memory or synchronises (except moe_workspace_status).
#include <mutex>
#include <set>
#include <utility>

#include "moe_internal.cuh"

namespace beam {

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool is_pow2(int v) { return v > 0 && (v & (v - 1)) == 0; }

bool finite_positive(float v) { return v > 0.0f && v <= 3.402823466e38f; }

}  // namespace

bool make_tmap_2d(CUtensorMap *map, const void *base, CUtensorMapDataType dtype, int elem_bytes,
                  uint64_t inner, uint64_t outer, uint32_t box_inner, uint32_t box_outer,
                  bool swizzle128) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || outer == 0) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * (uint64_t)elem_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, dtype, 2, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tmap_bf16_2d(CUtensorMap *map, const void *base, uint64_t inner, uint64_t outer,
                       uint32_t box_outer) {
  return make_tmap_2d(map, base, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, inner, outer, 64, box_outer,
                      true);
}

int device_sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return kTargetCtas;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = kTargetCtas;
    cached[dev] = n;
  }
  return cached[dev];
}

moe_status ensure_smem_limit(const void *kernel, int bytes) {
  static std::mutex mu;
  static std::set<std::pair<const void *, int>> done;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (done.count({kernel, dev})) return MOE_OK;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  done.insert({kernel, dev});
  return MOE_OK;
}

}  // namespace beam

using namespace beam;

namespace {

moe_status check_dims(const moe_dims *d) {
  if (!d) return MOE_ERR_INVALID_ARG;
  if (d->T < 0 || d->H <= 0 || d->E <= 0 || d->I <= 0 || d->n_group <= 0 || d->top_k <= 0 ||
      d->topk_group <= 0)
    return MOE_ERR_INVALID_ARG;
  if (d->E % d->n_group != 0 || d->topk_group > d->n_group) return MOE_ERR_INVALID_ARG;
  const int gsize = d->E / d->n_group;
  if (d->top_k > d->topk_group * gsize) return MOE_ERR_INVALID_ARG;
  if (!(d->routed_scale == d->routed_scale)) return MOE_ERR_INVALID_ARG;  // NaN
  if (d->H % 128 != 0 || d->I % 128 != 0) return MOE_ERR_UNSUPPORTED;
  if (d->E > 256 || d->E % 32 != 0 || d->n_group > 32 || gsize < 2 || !is_pow2(gsize))
    return MOE_ERR_UNSUPPORTED;
  if (d->top_k > 16) return MOE_ERR_UNSUPPORTED;
  if ((long long)d->T * d->top_k >= (1ll << 31)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

moe_status check_ws(const moe_dims *d, moe_op op, const void *ws, size_t ws_bytes,
                    moe_wdtype wdtype = MOE_W_BF16) {
  if (!ws || !aligned16(ws)) return MOE_ERR_WORKSPACE;
  if (ws_bytes < ws_layout(*d, op, wdtype).total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

template <class T>
T *at(void *ws, size_t off) {
  return reinterpret_cast<T *>(static_cast<char *>(ws) + off);
}

uint32_t *status_word(void *ws) { return static_cast<uint32_t *>(ws); }

bool ptrs_ok(std::initializer_list<const void *> ps) {
  for (const void *p : ps)
    if (!p || !aligned16(p)) return false;
  return true;
}

moe_status check_experts(const moe_dims *d, const moe_experts *ex) {
  if (!ex) return MOE_ERR_INVALID_ARG;
  if (ex->layout != MOE_LAYOUT_ROWMAJOR && ex->layout != MOE_LAYOUT_TILED) return MOE_ERR_INVALID_ARG;
  const bool tiled = ex->layout == MOE_LAYOUT_TILED;
  if (tiled && ex->dtype == MOE_W_NVFP4_A4) return MOE_ERR_UNSUPPORTED;
  if (ex->dtype == MOE_W_BF16) {
    if (!ptrs_ok({ex->w_gate, ex->w_up, ex->w_down})) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
  }
  if (ex->dtype == MOE_W_NVFP4 || ex->dtype == MOE_W_NVFP4_A4) {
    if (!ptrs_ok({ex->w_gate, ex->w_up, ex->w_down})) return MOE_ERR_INVALID_ARG;
    if (!tiled && !ptrs_ok({ex->s_gate, ex->s_up, ex->s_down})) return MOE_ERR_INVALID_ARG;
    if (ex->dtype == MOE_W_NVFP4_A4 &&
        !(finite_positive(ex->x_global) && finite_positive(ex->h_global)))
      return MOE_ERR_INVALID_ARG;
    for (const float *g : {ex->g_gate, ex->g_up, ex->g_down})
      if (!g || (reinterpret_cast<uintptr_t>(g) & 3u)) return MOE_ERR_INVALID_ARG;
    // one TMA box of block scales spans 16 bytes = 256 k
    if (d->H % 256 != 0 || d->I % 256 != 0) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
  }
  if (ex->dtype == MOE_W_FP8) {
    if (!ptrs_ok({ex->w_gate, ex->w_up, ex->w_down})) return MOE_ERR_INVALID_ARG;
    for (const float *g : {ex->g_gate, ex->g_up, ex->g_down})
      if (!g || (reinterpret_cast<uintptr_t>(g) & 3u)) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
  }
  return MOE_ERR_INVALID_ARG;
}

}  // namespace

extern "C" {

int moe_version(void) { return 100; }

const char *moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape";
    case MOE_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE: return "device-side error recorded in the workspace status word";
    case MOE_ERR_NOT_IMPLEMENTED: return "not implemented";
  }
  return "unknown status";
}

moe_status moe_check_dims(const moe_dims *dims) { return check_dims(dims); }

size_t moe_workspace_size(const moe_dims *dims, moe_wdtype wdtype, moe_op op) {
  if (check_dims(dims) != MOE_OK) return 0;
  if (wdtype != MOE_W_BF16 && wdtype != MOE_W_NVFP4 && wdtype != MOE_W_FP8 &&
      wdtype != MOE_W_NVFP4_A4)
    return 0;
  if (op < MOE_OP_ROUTE || op > MOE_OP_FORWARD) return 0;
  return ws_layout(*dims, op, wdtype).total;
}

moe_status moe_workspace_init(void *ws, moe_stream_t stream) {
  if (!ws) return MOE_ERR_WORKSPACE;
  return cudaMemsetAsync(ws, 0, kHeaderBytes, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

moe_status moe_workspace_status(const void *ws, moe_stream_t stream, uint32_t *out_bits) {
  if (!ws || !out_bits) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint32_t bits = 0;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemcpy(&bits, ws, sizeof bits, cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  *out_bits = bits;
  return bits ? MOE_ERR_DEVICE : MOE_OK;
}

moe_status moe_route(const moe_dims *dims, const void *x, const float *w_router, const float *bias,
                     int32_t *topk_idx, float *topk_w, void *ws, size_t ws_bytes,
                     moe_stream_t stream) {
  moe_status st = check_dims(dims);
  if (st != MOE_OK) return st;
  if (dims->T == 0) return MOE_OK;
  if (!ptrs_ok({x, w_router, bias, topk_idx, topk_w})) return MOE_ERR_INVALID_ARG;
  if ((st = check_ws(dims, MOE_OP_ROUTE, ws, ws_bytes)) != MOE_OK) return st;
  const WsLayout L = ws_layout(*dims, MOE_OP_ROUTE);
  return launch_route(*dims, x, w_router, bias, topk_idx, topk_w, make_router_plan(*dims),
                      at<__nv_bfloat16>(ws, L.w3), at<float>(ws, L.partial), status_word(ws),
                      reinterpret_cast<cudaStream_t>(stream));
}

moe_status moe_route_logits(const moe_dims *dims, const void *x, const float *w_router,
                            const float *bias, int32_t *topk_idx, float *topk_w, float *logits,
                            void *ws, size_t ws_bytes, moe_stream_t stream) {
  moe_status st = check_dims(dims);
  if (st != MOE_OK) return st;
  if (dims->T == 0) return MOE_OK;
  if (!ptrs_ok({x, w_router, bias, topk_idx, topk_w, logits})) return MOE_ERR_INVALID_ARG;
  if ((st = check_ws(dims, MOE_OP_ROUTE, ws, ws_bytes)) != MOE_OK) return st;
  const WsLayout L = ws_layout(*dims, MOE_OP_ROUTE);
  return launch_route(*dims, x, w_router, bias, topk_idx, topk_w, make_router_plan(*dims),
                      at<__nv_bfloat16>(ws, L.w3), at<float>(ws, L.partial), status_word(ws),
                      reinterpret_cast<cudaStream_t>(stream), logits);
}

moe_status moe_permute(const moe_dims *dims, const int32_t *topk_idx, const void *x, void *x_perm,
                       int32_t *expert_offsets, int32_t *slot_of, int32_t *row_src, void *ws,
                       size_t ws_bytes, moe_stream_t stream) {
  moe_status st = check_dims(dims);
  if (st != MOE_OK) return st;
  if (dims->T == 0) return MOE_OK;
  if (!ptrs_ok({topk_idx, x, x_perm, expert_offsets, slot_of, row_src})) return MOE_ERR_INVALID_ARG;
  if ((st = check_ws(dims, MOE_OP_PERMUTE, ws, ws_bytes)) != MOE_OK) return st;
  const WsLayout L = ws_layout(*dims, MOE_OP_PERMUTE);
  return launch_permute(*dims, topk_idx, x, x_perm, expert_offsets, slot_of, row_src,
                        at<int32_t>(ws, L.counts), at<int32_t>(ws, L.bases), status_word(ws),
                        reinterpret_cast<cudaStream_t>(stream));
}

moe_status moe_experts_swiglu(const moe_dims *dims, const moe_experts *experts, const void *x_perm,
                              const int32_t *expert_offsets, const int32_t *row_src,
                              const float *topk_w, void *y_partial, void *ws, size_t ws_bytes,
                              moe_stream_t stream) {
  moe_status st = check_dims(dims);
  if (st != MOE_OK) return st;
  if (dims->T == 0) return MOE_OK;
  if ((st = check_experts(dims, experts)) != MOE_OK) return st;
  if (!ptrs_ok({x_perm, expert_offsets, row_src, topk_w, y_partial})) return MOE_ERR_INVALID_ARG;
  if ((st = check_ws(dims, MOE_OP_EXPERTS, ws, ws_bytes, experts->dtype)) != MOE_OK) return st;
  const WsLayout L = ws_layout(*dims, MOE_OP_EXPERTS, experts->dtype);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (experts->dtype == MOE_W_NVFP4_A4) {
    uint8_t *xq = at<uint8_t>(ws, L.xq), *xs = at<uint8_t>(ws, L.xs);
    const int Tk = dims->T * dims->top_k;
    if ((st = launch_quantize_nvfp4(x_perm, nullptr, nullptr, dims->E, dims->top_k, Tk, dims->H,
                                    experts->x_global, xq, xs, s)) != MOE_OK)
      return st;
    return launch_experts_w4a4(*dims, *experts, xq, xs, expert_offsets, row_src, topk_w, y_partial,
                               at<uint8_t>(ws, L.hq), at<uint8_t>(ws, L.hs), status_word(ws), s);
  }
  if (experts->dtype != MOE_W_BF16) {
    const PackedWtScratch scr{at<void>(ws, L.x16), at<void>(ws, L.h), at<float>(ws, L.xscale),
                              at<uint32_t>(ws, L.hmax), at<float>(ws, L.hscale)};
    if (packed_wt_applies(*dims))
      return launch_experts_packed_wt(*dims, *experts, x_perm, expert_offsets, row_src, topk_w,
                                      y_partial, scr, status_word(ws), s);
    if ((st = launch_rows_f16_scaled(x_perm, scr.x16, (long)dims->T * dims->top_k, dims->H,
                                     scr.xscale, scr.hmax, s)) != MOE_OK)
      return st;
    return launch_experts_fp4(*dims, *experts, expert_offsets, row_src, topk_w, y_partial, scr,
                              status_word(ws), s);
  }
  return launch_experts(*dims, *experts, x_perm, expert_offsets, row_src, topk_w, y_partial,
                        at<__nv_bfloat16>(ws, L.h), status_word(ws), s);
}

moe_status moe_combine(const moe_dims *dims, const void *y_partial, const int32_t *slot_of, void *y,
                       moe_stream_t stream) {
  moe_status st = check_dims(dims);
  if (st != MOE_OK) return st;
  if (dims->T == 0) return MOE_OK;
  if (!ptrs_ok({y_partial, slot_of, y})) return MOE_ERR_INVALID_ARG;
  return launch_combine(*dims, y_partial, slot_of, y, reinterpret_cast<cudaStream_t>(stream));
}

moe_status moe_forward(const moe_dims *dims, const void *x, const float *w_router,
                       const float *bias, const moe_experts *experts, void *y, int32_t *topk_idx,
                       float *topk_w, void *ws, size_t ws_bytes, moe_stream_t stream) {
  moe_status st = check_dims(dims);
  if (st != MOE_OK) return st;
  if (dims->T == 0) return MOE_OK;
  if ((st = check_experts(dims, experts)) != MOE_OK) return st;
  if (!ptrs_ok({x, w_router, bias, y})) return MOE_ERR_INVALID_ARG;
  if ((topk_idx && !aligned16(topk_idx)) || (topk_w && !aligned16(topk_w)))
    return MOE_ERR_INVALID_ARG;
  if ((st = check_ws(dims, MOE_OP_FORWARD, ws, ws_bytes, experts->dtype)) != MOE_OK) return st;
  const moe_dims &d = *dims;
  const WsLayout L = ws_layout(d, MOE_OP_FORWARD, experts->dtype);
  const bool a4 = experts->dtype == MOE_W_NVFP4_A4;
  const bool packed = experts->dtype != MOE_W_BF16 && !a4;
  // packed weights: small and mid-size batches dequantise into tensor memory,
  // large ones run the token-major GEMMs; both on f16 activations with a
  // power-of-two scale per row
  const bool packed_wt = packed && packed_wt_applies(d);
  const bool fp4 = packed && !packed_wt;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t *idx = topk_idx ? topk_idx : at<int32_t>(ws, L.topk_idx);
  float *w = topk_w ? topk_w : at<float>(ws, L.topk_w);
  uint32_t *status = status_word(ws);
  if ((st = launch_route(d, x, w_router, bias, idx, w, make_router_plan(d),
                         at<__nv_bfloat16>(ws, L.w3), at<float>(ws, L.partial), status, s)) != MOE_OK)
    return st;
  void *x_perm = at<void>(ws, L.x_perm);
  int32_t *offsets = at<int32_t>(ws, L.offsets);
  int32_t *slot_of = at<int32_t>(ws, L.slot_of);
  int32_t *row_src = at<int32_t>(ws, L.row_src);
  // the gather writes x_perm in bf16, or as f16 scaled per token for the
  // token-major packed-weight GEMMs; W4A4 quantises each token once and
  // writes it to its slots
  const GatherMode gm = a4 ? kGatherNone : fp4 ? kGatherF16Scaled : kGatherBf16;
  if ((st = launch_permute(d, idx, x, x_perm, offsets, slot_of, row_src, at<int32_t>(ws, L.counts),
                           at<int32_t>(ws, L.bases), status, s, gm, at<float>(ws, L.xscale),
                           at<uint32_t>(ws, L.hmax))) != MOE_OK)
    return st;
  void *y_partial = at<void>(ws, L.y_partial);
  if (a4) {
    uint8_t *xq = at<uint8_t>(ws, L.xq), *xs = at<uint8_t>(ws, L.xs);
    if ((st = launch_quantize_scatter_nvfp4(x, slot_of, d.T, d.top_k, d.H, experts->x_global, xq,
                                            xs, s)) != MOE_OK)
      return st;
    st = launch_experts_w4a4(d, *experts, xq, xs, offsets, row_src, w, y_partial,
                             at<uint8_t>(ws, L.hq), at<uint8_t>(ws, L.hs), status, s);
  } else if (packed_wt) {
    // x_perm is scaled to f16 in place
    const PackedWtScratch scr{x_perm, at<void>(ws, L.h), at<float>(ws, L.xscale),
                              at<uint32_t>(ws, L.hmax), at<float>(ws, L.hscale)};
    st = launch_experts_packed_wt(d, *experts, x_perm, offsets, row_src, w, y_partial, scr, status,
                                  s);
  } else if (fp4) {
    const PackedWtScratch scr{x_perm, at<void>(ws, L.h), at<float>(ws, L.xscale),
                              at<uint32_t>(ws, L.hmax), at<float>(ws, L.hscale)};
    st = launch_experts_fp4(d, *experts, offsets, row_src, w, y_partial, scr, status, s);
  } else {
    st = launch_experts(d, *experts, x_perm, offsets, row_src, w, y_partial,
                        at<__nv_bfloat16>(ws, L.h), status, s);
  }
  if (st != MOE_OK) return st;
  return launch_combine(d, y_partial, slot_of, y, s);
}

moe_status moe_pack_bf16(int E, int N, int K, const void *src, void *dst, moe_stream_t stream) {
  if (E < 0 || N < 0 || K < 0 || N % 128 != 0 || K % 64 != 0) return MOE_ERR_INVALID_ARG;
  if ((size_t)E * N * K == 0) return MOE_OK;
  if (!ptrs_ok({src, dst}) || src == dst) return MOE_ERR_INVALID_ARG;
  return launch_pack_bf16(E, N, K, src, dst, reinterpret_cast<cudaStream_t>(stream));
}

moe_status moe_pack_nvfp4(int E, int N, int K, const uint8_t *q, const uint8_t *s, uint8_t *dst,
                          moe_stream_t stream) {
  if (E < 0 || N < 0 || K < 0 || N % 128 != 0 || K % 64 != 0) return MOE_ERR_INVALID_ARG;
  if ((size_t)E * N * K == 0) return MOE_OK;
  if (!ptrs_ok({q, s, dst}) || dst == q || dst == s) return MOE_ERR_INVALID_ARG;
  return launch_pack_nvfp4(E, N, K, q, s, dst, reinterpret_cast<cudaStream_t>(stream));
}

moe_status moe_pack_fp8(int E, int N, int K, const uint8_t *q, uint8_t *dst, moe_stream_t stream) {
  if (E < 0 || N < 0 || K < 0 || N % 128 != 0 || K % 64 != 0) return MOE_ERR_INVALID_ARG;
  if ((size_t)E * N * K == 0) return MOE_OK;
  if (!ptrs_ok({q, dst}) || dst == q) return MOE_ERR_INVALID_ARG;
  return launch_pack_fp8(E, N, K, q, dst, reinterpret_cast<cudaStream_t>(stream));
}

moe_status moe_quantize_nvfp4(int rows, int cols, const void *x, float g, uint8_t *q, uint8_t *s,
                              moe_stream_t stream) {
  if (rows < 0 || cols <= 0 || cols % 16 != 0 || !finite_positive(g)) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  if (!ptrs_ok({x, q, s})) return MOE_ERR_INVALID_ARG;
  return launch_quantize_nvfp4(x, nullptr, nullptr, 0, 1, rows, cols, g, q, s,
                               reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
