/*
 * beam_moe.h — C ABI of the B300 (sm_103a) forward pass of Beam's
 * Mixture-of-Experts block.
 *
 * The layer (Reflection's Beam; "Hugging Face releases Beam ..." third
 * paragraph, and "Reflection Releases Beam ...", section "Where Beam Saves and
 * Where the Memory Bill Comes In"): 256 experts per layer, each a SwiGLU MLP
 * with intermediate size 2,560, hidden size 5,120; a sigmoid router with a
 * per-expert selection bias ("Beam 1.0", auxiliary-loss-free balancing) keeps
 * the best 4 of 8 groups of 32 experts and picks the top 8 experts inside
 * them; the routed weights are normalised and scaled by 2.5; no shared expert.
 *
 * Conventions for every call below
 *   - All tensor pointers are DEVICE pointers on the current CUDA device,
 *     16-byte aligned (256 recommended), row-major and densely packed.  The
 *     caller owns every buffer; the library allocates no device memory and
 *     keeps no pointer after a call returns.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream) and never synchronise, except moe_workspace_status.
 *   - Argument errors return before anything is launched.  A failed launch
 *     returns MOE_ERR_CUDA.  Errors found on the device (an expert index out of
 *     range, an internal wait that ran past its time limit) set bits in the
 *     status word at the start of the workspace; read it with
 *     moe_workspace_status after the stream has finished.
 *   - Workspaces must be at least moe_workspace_size(...) bytes and their
 *     first 2048 bytes zeroed once before first use (moe_workspace_init);
 *     calls leave them zeroed again (they hold the status word and the
 *     counters of the expert GEMMs' tile schedule).  After a call that
 *     returned an error or set a device status bit, zero them again
 *     (moe_workspace_init) before reusing the workspace.
 *     A workspace may be reused by consecutive calls on one stream; calls
 *     that run concurrently need separate workspaces.
 *   - Shape limits: H % 128 == 0, I % 128 == 0, E <= 256 with E % 32 == 0,
 *     E % n_group == 0, group size E / n_group a power of two >= 2,
 *     n_group <= 32, 1 <= topk_group <= n_group, 1 <= top_k <= 16 and
 *     top_k <= topk_group * group size, 0 <= T and T * top_k < 2^31.
 *   - T == 0 is a no-op: the call returns MOE_OK after checking the dims and
 *     reads no pointer.
 *   - Inputs must be finite.  Selection compares fp32 scores; equal scores go
 *     to the lower group index, then to the lower expert index.
 *
 * Layouts (T tokens, H hidden, E experts, I intermediate, k = top_k)
 *   x           bf16  [T, H]
 *   w_router    fp32  [E, H]            one row per expert
 *   bias        fp32  [E]               selection bias (selection only)
 *   topk_idx    int32 [T, k]            descending biased score
 *   topk_w      fp32  [T, k]            routed weights, sum to routed_scale
 *   expert_offsets int32 [E + 1]        rows of expert e are
 *                                       [offsets[e], offsets[e+1]) in the
 *                                       permuted order
 *   slot_of     int32 [T * k]           permuted row of entry t*k + j
 *   row_src     int32 [T * k]           entry t*k + j held by permuted row r
 *   x_perm      bf16  [T * k, H]        x rows in permuted (expert-major,
 *                                       then entry-ascending) order
 *   y_partial   bf16  [T * k, H]        routed-weight-scaled expert output
 *                                       per permuted row
 *   y           bf16  [T, H]            block output
 *   bf16 experts: w_gate, w_up [E, I, H]; w_down [E, H, I]   (out x in)
 *   NVFP4 experts: w_* packed e2m1 uint8 [E, N, K/2] with the even k in the
 *                  low nibble, s_* e4m3 uint8 [E, N, K/16] (one scale per 16
 *                  consecutive k), g_* fp32 [E] global scales; the weight is
 *                  e2m1 * e4m3 * global.  (N, K) = (I, H) for gate and up,
 *                  (H, I) for down.  Needs H % 256 == 0 and I % 256 == 0.
 *   NVFP4 W4A4:    the NVFP4 layouts above, plus x_global and h_global in
 *                  moe_experts; the activations are quantised as in
 *                  moe_quantize_nvfp4, the GEMMs accumulate in fp32, and h is
 *                  held as NVFP4 between them.
 *   FP8 experts:   w_* e4m3 uint8 [E, N, K]; g_* fp32 [E, N], one scale per
 *                  output row (the pages give no FP8 layout: this is the plain
 *                  reading that keeps dequantisation exact); s_* unused.
 *                  The weight is e4m3 * g[e, n].
 */
#ifndef BEAM_MOE_H
#define BEAM_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *moe_stream_t; /* identical to cudaStream_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,     /* null/misaligned pointer or bad shape        */
  MOE_ERR_UNSUPPORTED = 2,     /* shape outside the limits above              */
  MOE_ERR_WORKSPACE = 3,       /* workspace missing or too small              */
  MOE_ERR_CUDA = 4,            /* a CUDA call or kernel launch failed         */
  MOE_ERR_DEVICE = 5,          /* the workspace status word is non-zero       */
  MOE_ERR_NOT_IMPLEMENTED = 6
} moe_status;

/* Expert weight formats.  MOE_W_NVFP4_A4 takes NVFP4 weights as MOE_W_NVFP4
 * and also quantises the activations (x before gate/up, h before down) to
 * NVFP4, so both GEMMs run on the block-scaled fp4 tensor cores (W4A4). */
typedef enum { MOE_W_BF16 = 0, MOE_W_NVFP4 = 1, MOE_W_FP8 = 2, MOE_W_NVFP4_A4 = 3 } moe_wdtype;

/* Which entry point a workspace is sized for. */
typedef enum {
  MOE_OP_ROUTE = 0,
  MOE_OP_PERMUTE = 1,
  MOE_OP_EXPERTS = 2,
  MOE_OP_FORWARD = 3
} moe_op;

/* Bits of the device status word (first 4 bytes of a workspace). */
#define MOE_DEV_TIMEOUT 0x1   /* an internal wait ran past its limit        */
#define MOE_DEV_BAD_INDEX 0x2 /* an expert index outside [0, E) was skipped */

typedef struct {
  int T;              /* tokens in this call                               */
  int H;              /* hidden size (Beam: 5120)                          */
  int E;              /* routed experts (Beam: 256)                        */
  int n_group;        /* expert groups (Beam: 8)                           */
  int topk_group;     /* groups kept per token (Beam: 4)                   */
  int top_k;          /* experts per token (Beam: 8)                       */
  int I;              /* SwiGLU intermediate size (Beam: 2560)             */
  float routed_scale; /* factor on the normalised weights (Beam: 2.5)      */
} moe_dims;

typedef struct {
  moe_wdtype dtype;
  const void *w_gate, *w_up, *w_down;    /* bf16, packed e2m1 (NVFP4) or e4m3 (FP8) */
  const uint8_t *s_gate, *s_up, *s_down; /* e4m3 block scales (NVFP4 only)          */
  const float *g_gate, *g_up, *g_down;   /* fp32 [E] globals (NVFP4), [E, N] row
                                            scales (FP8)                            */
  float x_global, h_global;              /* MOE_W_NVFP4_A4 only: static fp32 global
                                            scales of the x and h quantisers (finite,
                                            > 0; see moe_quantize_nvfp4)            */
  int layout;                            /* MOE_LAYOUT_ROWMAJOR, or MOE_LAYOUT_TILED
                                            for weights packed by moe_pack_bf16,
                                            moe_pack_nvfp4 or moe_pack_fp8          */
} moe_experts;

/* Layout of the expert weights.  MOE_LAYOUT_TILED applies to MOE_W_BF16
 * (w_* written by moe_pack_bf16), MOE_W_NVFP4 (w_* written by moe_pack_nvfp4,
 * which holds the block scales too: s_* are then unused and may be NULL) and
 * MOE_W_FP8 (w_* written by moe_pack_fp8; g_* as for row-major).  MOE_W_NVFP4_A4
 * takes row-major weights only (MOE_ERR_UNSUPPORTED otherwise). */
#define MOE_LAYOUT_ROWMAJOR 0 /* [E, N, K] as in the layouts above                */
#define MOE_LAYOUT_TILED 1    /* the tiled layouts written by the moe_pack_* calls */

/* Library version, major * 10000 + minor * 100 + patch. */
int moe_version(void);

/* Human-readable name of a status code (static string). */
const char *moe_status_string(moe_status s);

/* Checks dims against the shape limits above; MOE_OK if supported. */
moe_status moe_check_dims(const moe_dims *dims);

/* Bytes of workspace that entry point `op` needs for these dims (0 if the
 * dims are unsupported).  Includes the 2048-byte status header. */
size_t moe_workspace_size(const moe_dims *dims, moe_wdtype wdtype, moe_op op);

/* Zeroes the 2048-byte status header of a workspace (asynchronous). */
moe_status moe_workspace_init(void *ws, moe_stream_t stream);

/* Synchronises `stream`, then copies the workspace status word into
 * *out_bits (0 = no device error).  Returns MOE_ERR_DEVICE if it is set. */
moe_status moe_workspace_status(const void *ws, moe_stream_t stream, uint32_t *out_bits);

/*
 * Router: sigmoid scores, per-expert selection bias, group-limited top-k.
 * ("Hugging Face releases Beam ...", third paragraph: top 8 experts from the
 * top 4 of 8 groups of 32; "Reflection Releases Beam ...", section "Where Beam
 * Saves ...": sigmoid scores, DeepSeek-V3 group limits, normalised and scaled
 * by 2.5; "Beam 1.0": per-expert bias of auxiliary-loss-free balancing.)
 *   logit[t,e] = sum_h x[t,h] * w_router[e,h]      (fp32 accumulation)
 *   s = sigmoid(logit); s' = s + bias[e]           (s' selects, s weighs)
 *   group score = sum of the two largest s' of the group
 *   keep the topk_group best groups; take the top_k largest s' among their
 *   experts; topk_w = routed_scale * s / sum of the chosen s.
 * Outputs topk_idx [T,k] and topk_w [T,k].  Workspace: MOE_OP_ROUTE.
 */
moe_status moe_route(const moe_dims *dims, const void *x, const float *w_router,
                     const float *bias, int32_t *topk_idx, float *topk_w, void *ws,
                     size_t ws_bytes, moe_stream_t stream);

/*
 * moe_route with one more output: logits fp32 [T, E] receives the router
 * logits x . w_router^T from which the selection above was made, exactly the
 * values the sigmoid is applied to (the same fp32 sums, in the same order).
 * Routing outputs are identical to moe_route's.  For inspection of the
 * router and for losses on its logits; the pages define the logit as the
 * router's dot product ("Reflection Releases Beam ...", section "Where Beam
 * Saves ...": sigmoid scores over the router's output).  Workspace: MOE_OP_ROUTE.
 */
moe_status moe_route_logits(const moe_dims *dims, const void *x, const float *w_router,
                            const float *bias, int32_t *topk_idx, float *topk_w, float *logits,
                            void *ws, size_t ws_bytes, moe_stream_t stream);

/*
 * Dispatch: sorts the T*k (token, slot) entries by expert, stably (entries of
 * one expert keep ascending t*k + j order), and gathers x rows into that order.
 * (The pages: tokens must reach the experts they selected — "Beam Turns
 * Frontier-Scale Openness Into an Infrastructure Decision", section "Sparse
 * compute still requires dense planning".)
 * Outputs expert_offsets [E+1], slot_of [T*k], row_src [T*k], x_perm [T*k,H].
 * Entries with an index outside [0,E) set MOE_DEV_BAD_INDEX and are dropped.
 * Workspace: MOE_OP_PERMUTE.
 */
moe_status moe_permute(const moe_dims *dims, const int32_t *topk_idx, const void *x,
                       void *x_perm, int32_t *expert_offsets, int32_t *slot_of,
                       int32_t *row_src, void *ws, size_t ws_bytes, moe_stream_t stream);

/*
 * Expert MLPs over the permuted rows ("Hugging Face releases Beam ...", third
 * paragraph: each expert a SwiGLU MLP with intermediate size 2,560):
 *   h = silu(x_perm . W_gate[e]^T) * (x_perm . W_up[e]^T)     (h kept in bf16)
 *   y_partial[r] = topk_w[row_src[r]] * (h . W_down[e]^T)      (stored bf16)
 * for every permuted row r of expert e.  fp32 accumulation on tensor cores.
 * With NVFP4 or FP8 weights (MOE_W_NVFP4, MOE_W_FP8) the GEMMs run on f16
 * operands: the dequantised weights are exact in f16, and x_perm and h keep
 * bf16's range by one power-of-two scale per row (each row's largest
 * magnitude brought into [2^14, 2^15), multiplied back out of the fp32
 * accumulator), so the results are those of bf16 activations up to values
 * below 2^-28 of their row's largest.  topk_w is indexed by entry (t*k + j).
 * Workspace: MOE_OP_EXPERTS.
 */
moe_status moe_experts_swiglu(const moe_dims *dims, const moe_experts *experts,
                              const void *x_perm, const int32_t *expert_offsets,
                              const int32_t *row_src, const float *topk_w, void *y_partial,
                              void *ws, size_t ws_bytes, moe_stream_t stream);

/*
 * Combine: y[t] = sum over j = 0..k-1, in that order, of y_partial[slot_of[t*k+j]],
 * summed in fp32 and rounded once to bf16.  No shared expert enters the sum
 * ("Reflection Releases Beam ...", section "Where Beam Saves ...": there is no
 * shared expert).  Deterministic.  Needs no workspace.
 */
moe_status moe_combine(const moe_dims *dims, const void *y_partial, const int32_t *slot_of,
                       void *y, moe_stream_t stream);

/*
 * The whole block: moe_route, moe_permute, moe_experts_swiglu and moe_combine
 * in sequence on `stream`, with every intermediate in the workspace.  The
 * block as the pages state it: "Hugging Face releases Beam ...", third
 * paragraph (256 experts per layer, each a SwiGLU MLP of intermediate size
 * 2,560; the top 8 experts from the top 4 of 8 groups of 32), and "Reflection
 * Releases Beam ...", section "Where Beam Saves and Where the Memory Bill
 * Comes In" (sigmoid router, outputs normalised and scaled by 2.5, no shared
 * expert).
 * topk_idx / topk_w may be NULL; when given they receive the routing.
 * Workspace: MOE_OP_FORWARD.
 */
moe_status moe_forward(const moe_dims *dims, const void *x, const float *w_router,
                       const float *bias, const moe_experts *experts, void *y, int32_t *topk_idx,
                       float *topk_w, void *ws, size_t ws_bytes, moe_stream_t stream);

/*
 * Auxiliary-loss-free load balancing ("Beam 1.0": the router's per-expert bias
 * follows DeepSeek-V3's auxiliary-loss-free balancing with a cosine decay of
 * the expert-bias updates).  After a batch is routed (topk_idx [T,k] from
 * moe_route or moe_forward), moves every expert's selection bias one step
 * against its load:
 *   load_e  = number of entries of topk_idx equal to e
 *   gamma_t = gamma_max * (1 + cos(pi * step / total_steps)) / 2,
 *             step clamped to [0, total_steps]
 *   bias[e] += gamma_t * sign(T*k/E - load_e)      (sign(0) = 0)
 * The page names the method, not the formula: this is the plain reading.
 * bias fp32 [E] is updated in place on `stream`; *gamma_used (nullable)
 * receives gamma_t as applied (fp32).  Entries outside [0, E) are ignored.
 * Needs no workspace; results do not depend on thread timing.
 */
moe_status moe_bias_update(const moe_dims *dims, const int32_t *topk_idx, float *bias,
                           double gamma_max, int step, int total_steps, float *gamma_used,
                           moe_stream_t stream);

/*
 * NVFP4 quantisation of activations, the step MOE_W_NVFP4_A4 applies to x
 * before the gate/up GEMM and to h before the down GEMM.  The pages give only
 * "NVFP4 for Blackwell" ("Reflection Releases Beam ...", section "Where Beam
 * Saves and Where the Memory Bill Comes In"); the reading here is the
 * weights' two-level format with a static per-tensor global scale g:
 * for every block of 16 consecutive values v of a row, in fp32 (IEEE
 * division and multiplication, round to nearest even):
 *   amax = max |v|;  s = e4m3(amax / (6 g)) saturating at 448;
 *   scale = value(s) * g;  code_i = e2m1(v_i / scale) saturating at +-6
 *   (all codes 0 when scale == 0).  The value of a code is e2m1 * e4m3 * g.
 *   x  bf16 [rows, cols] (cols % 16 == 0), g finite and > 0
 *   q  uint8 [rows, cols/2]: two codes per byte, even column in the low nibble
 *   s  uint8 [rows, cols/16]: e4m3 scale codes
 * Needs no workspace.  rows == 0 is a no-op.
 */
moe_status moe_quantize_nvfp4(int rows, int cols, const void *x, float g, uint8_t *q, uint8_t *s,
                              moe_stream_t stream);

/*
 * Packs one bf16 weight tensor [E, N, K] (row-major, K contiguous: W_gate or
 * W_up with N = I, K = H; W_down with N = H, K = I) into the MMA-tiled layout
 * that moe_experts.layout = MOE_LAYOUT_TILED expects: tiles of 128 rows x 64 k,
 * each stored as the 16 KB image the expert GEMMs hold in shared memory (the
 * 128-byte swizzle: 16-byte chunk c of row r at position c XOR (r mod 8) of the
 * row), ordered expert, 128-row block, k block.  Same size as the source.  A
 * tile then streams from HBM as one contiguous copy; results are bit for bit
 * those of the row-major layout.  The pages give no weight layout (a
 * load-time preparation step of this implementation, like the NVFP4 packing).
 *   Needs N % 128 == 0, K % 64 == 0, src and dst distinct and 16-byte aligned.
 *   Asynchronous on `stream`; needs no workspace.
 */
moe_status moe_pack_bf16(int E, int N, int K, const void *src, void *dst, moe_stream_t stream);

/*
 * Packs one NVFP4 weight tensor (codes q uint8 [E, N, K/2], even k in the low
 * nibble, and e4m3 block scales s uint8 [E, N, K/16], as in the NVFP4 layout
 * above) into the tiled layout that moe_experts.layout = MOE_LAYOUT_TILED
 * expects for MOE_W_NVFP4: tiles of 128 rows x 64 k, ordered expert, 128-row
 * block, k block; a tile is 4608 bytes, the 128 rows' codes (32 bytes per row,
 * row after row) followed by their scales (4 bytes per row, row after row).
 * dst holds E * N * K * 9 / 16 bytes.  Each tile then streams from HBM as one
 * contiguous copy instead of 256 short row segments; results are bit for bit
 * those of the row-major layout.  A load-time preparation step of this
 * implementation (the pages give no weight layout).
 *   Needs N % 128 == 0, K % 64 == 0, all pointers 16-byte aligned, dst
 *   distinct from q and s.  Asynchronous on `stream`; needs no workspace.
 */
moe_status moe_pack_nvfp4(int E, int N, int K, const uint8_t *q, const uint8_t *s, uint8_t *dst,
                          moe_stream_t stream);

/*
 * Packs one FP8 weight tensor (e4m3 codes uint8 [E, N, K]) into the tiled
 * layout that moe_experts.layout = MOE_LAYOUT_TILED expects for MOE_W_FP8:
 * tiles of 128 rows x 64 k (8192 bytes, 64 bytes per row, row after row),
 * ordered expert, 128-row block, k block.  dst holds E * N * K bytes; the row
 * scales g_* keep their [E, N] layout.  Results are bit for bit those of the
 * row-major layout.
 *   Needs N % 128 == 0, K % 64 == 0, q and dst 16-byte aligned and distinct.
 *   Asynchronous on `stream`; needs no workspace.
 */
moe_status moe_pack_fp8(int E, int N, int K, const uint8_t *q, uint8_t *dst, moe_stream_t stream);

/*
 * moe_permute_noalloc — the dispatch of moe_permute for callers that cannot
 * allocate device memory at all: a plug-in inside a host framework that owns
 * every device buffer and passes it only its inputs and outputs, or a serving
 * loop that forbids allocations after start-up (cudaMalloc may synchronise the
 * device).  The pages have no counterpart to this entry point.
 *   Same inputs, outputs and layouts as moe_permute, but no workspace: its
 *   scratch (per-chunk expert counts and bases) lives in one 1 MiB device
 *   array inside the library, which every GPU that loads the library holds
 *   until the process exits.
 *   Limit: 256 + 2 * round_up(4 * E * ceil(T*k / 4096), 256) bytes must fit
 *   in 1 MiB (a 256-byte header, then two tables, each rounded up to 256
 *   bytes), i.e. T*k <= 2,093,056 entries at E = 256 and <= 16,769,024 at
 *   E = 32; larger calls return MOE_ERR_UNSUPPORTED before launching
 *   anything.
 *   The first call on each device looks up the array's device address with
 *   that device current and keeps it for the life of the process; make that
 *   first call before any stream capture.  The address belongs to the
 *   device's primary context: do not call this entry point from another
 *   driver context, or after cudaDeviceReset (which may reload the library's
 *   device code at another address).
 *   All calls share the one array: calls that overlap on the GPU (other
 *   streams, other host threads) race and corrupt each other's results.
 *   Out-of-range expert indices are dropped as in moe_permute, but no status
 *   word is kept: check expert_offsets[E] == T*k instead.
 */
moe_status moe_permute_noalloc(const moe_dims *dims, const int32_t *topk_idx, const void *x,
                               void *x_perm, int32_t *expert_offsets, int32_t *slot_of,
                               int32_t *row_src, moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* BEAM_MOE_H */
