// Expert MLPs with NVFP4 weights AND NVFP4 activations (W4A4) on the
// block-scaled fp4 tensor cores of sm_103a.
//
// The pages ship Beam as an NVFP4 checkpoint for Blackwell ("Reflection
// Releases Beam ...", section "Where Beam Saves and Where the Memory Bill
// Comes In"); this path also quantises the activations to NVFP4 (readings in
// nvfp4_quant.cuh) so both GEMM operands are e2m1 codes with one ue4m3 scale
// per 16 k, which tcgen05.mma kind::mxf4nvf4 consumes directly:
//   D[m, n] = sum_k e2m1(a[m,k]) * sfa[m, k/16] * e2m1(b[n,k]) * sfb[n, k/16]
// and the two fp32 global scales multiply D in the epilogue.
//
// Token-major tiles: 128 token rows of one expert on the MMA's M side, 256
// weight rows on N.  Gate/up puts the 128 gate rows and the 128 up rows of the
// same 128 features on N, so the epilogue forms h = silu(g) * u per token row
// and quantises it to NVFP4 (16 consecutive features per scale) for the down
// GEMM.  Down scales each token row by its routing weight and stores bf16.
//
// One CTA per SM, persistent; 640 threads:
//   warp 0 lane 0 : TMA producer (codes with the 128-byte swizzle, scales plain)
//   warp 1        : MMA issuer (the warp converged, one elected lane issuing):
//                   copies each stage's scales to tensor memory
//                   (tcgen05.cp) and issues the four K=64 MMAs of the stage
//   warps 2, 3    : scale arrangers, alternate K slices: rearrange the stage's
//                   scale bytes in shared memory into the 32 x 16-byte blocks
//                   that tcgen05.cp.32x128b.warpx4 copies to tensor memory (row
//                   m of a 128-row block goes to byte (m % 32) * 16 + (m / 32) * 4,
//                   its four 16-k scales in consecutive bytes); warp 2 also
//                   allocates tensor memory
//   warps 4..19   : epilogue, four warps per 32-lane quarter of the accumulator
// Tensor memory: accumulator columns [0, 256); stage s keeps its scales at
// columns 256 + 48 s: A in the first 16 (4 per MMA), B in the next 32 (8 per
// MMA, one column per 32 rows of N).  A stage's scale columns are rewritten
// only after the MMAs that read them have completed (the producer refills a
// stage only after their commit).
#include "moe_internal.cuh"
#include "nvfp4_quant.cuh"
#include "ptx.cuh"
#include "sched.cuh"
#include "tc_gemm.cuh"

namespace beam {

namespace {

constexpr int kW4M = 128;                          // token rows per tile (MMA M)
constexpr int kW4N = 256;                          // weight rows per tile (MMA N)
constexpr int kW4RowBytes = 128;                   // 256 fp4 values: one K slice
constexpr int kW4ABytes = kW4M * kW4RowBytes;      // 16 KB
constexpr int kW4BBytes = kW4N * kW4RowBytes;      // 32 KB
constexpr int kW4SfABytes = kW4M * 16;             // 2 KB: 16 scales per row per slice
constexpr int kW4SfBBytes = kW4N * 16;             // 4 KB
constexpr int kW4Stage = kW4ABytes + kW4BBytes + kW4SfABytes + kW4SfBBytes;  // 55296
constexpr int kW4Stages = 4;
constexpr int kW4EpiWarps = 16;
constexpr int kW4Threads = 128 + 32 * kW4EpiWarps;
constexpr uint32_t kW4TmemCols = 512;
constexpr uint32_t kW4SfCol0 = 256;
constexpr uint32_t kW4SfStride = 48;
static_assert(kW4Stage % 1024 == 0, "stage must keep 1024-byte alignment");
static_assert(kW4SfCol0 + kW4Stages * kW4SfStride <= kW4TmemCols, "tensor memory overflow");

constexpr int kW4SmemBytes = 1024 + kW4Stages * kW4Stage + 256 + (int)sizeof(TileSched);
static_assert(kW4SmemBytes <= kSmemLimit, "shared memory overflow");

// kind::mxf4nvf4 instruction descriptor: A and B e2m1 (format 1), ue4m3
// scales (bit 23 clear), scale-factor ids 0, K-major, dense K = 64.
__host__ __device__ constexpr uint32_t w4_idesc(int M, int N) {
  return (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Shared-memory descriptor of a 32-row x 16-byte block with no swizzle
// (8-row core matrices 128 bytes apart), the source of tcgen05.cp.32x128b.
__device__ __forceinline__ uint64_t sf_desc(uint32_t smem_addr) {
  uint64_t d = (uint64_t)((smem_addr & 0x3FFFF) >> 4);
  d |= (uint64_t)(128 >> 4) << 16;
  d |= (uint64_t)(128 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  return d;
}

__device__ __forceinline__ void tmem_cp_sf(uint32_t taddr, uint64_t desc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc)
               : "memory");
}

__device__ __forceinline__ void umma_fp4(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t sfa, uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X "
      "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2_w4(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&v);
}

struct W4Params {
  CUtensorMap tm_a, tm_sa;    // activation codes [Tk, K/2] box {128,128} sw128; scales [Tk, K/16] box {16,128}
  CUtensorMap tm_b0, tm_sb0;  // gate (box {128,128}/{16,128}) or down (box {128,256}/{16,256})
  CUtensorMap tm_b1, tm_sb1;  // up (gate/up only)
  const int32_t *offsets;
  const int32_t *row_src;
  const float *topk_w;
  const float *gw0, *gw1;  // weight globals [E]: gate (or down), up
  float ga;                // global scale of the activation operand
  float gh;                // global scale of the h quantiser (gate/up)
  uint8_t *hq, *hs;        // gate/up output: h codes [Tk, I/2], scales [Tk, I/16]
  __nv_bfloat16 *y;        // down output: y_partial [Tk, H]
  int E, ksteps, nf, b_rows, out_cols;
  uint32_t *status;
};

struct W4Tile {
  int e, f, row0, nrows, brow0;
};

template <bool GATEUP>
__device__ __forceinline__ W4Tile w4_tile(const W4Params &p, const TileSched &s, int t) {
  constexpr int FW = GATEUP ? 128 : 256;  // output features per tile
  const int e = tile_sched_expert(s, p.E, t);
  const int ntt = (s.off[e + 1] - s.off[e] + kW4M - 1) / kW4M;
  const int local = t - s.tp[e];
  const int f = local / ntt, tt = local - f * ntt;  // token tiles inner: weight tile reuse in L2
  const int row0 = s.off[e] + tt * kW4M;
  return W4Tile{e, f, row0, min(kW4M, s.off[e + 1] - row0), e * p.b_rows + f * FW};
}

// Rearranges the 16 scale bytes of each row of a 128*nblk-row slice (row-major,
// 16 bytes per row, as TMA delivered it) into per-MMA 512-byte blocks:
// block (j * nblk + b) holds, for rows 128 b .. 128 b + 127, the 4 scales of
// MMA j.  In place; the whole warp takes part.
template <int NBLK>
__device__ __forceinline__ void w4_arrange_sf(uint8_t *sf, int lane) {
  uint4 v[NBLK][4];
#pragma unroll
  for (int b = 0; b < NBLK; ++b)
#pragma unroll
    for (int m1 = 0; m1 < 4; ++m1)
      v[b][m1] = *reinterpret_cast<const uint4 *>(sf + (b * 128 + m1 * 32 + lane) * 16);
  __syncwarp();
#pragma unroll
  for (int b = 0; b < NBLK; ++b) {
    *reinterpret_cast<uint4 *>(sf + (0 * NBLK + b) * 512 + lane * 16) =
        make_uint4(v[b][0].x, v[b][1].x, v[b][2].x, v[b][3].x);
    *reinterpret_cast<uint4 *>(sf + (1 * NBLK + b) * 512 + lane * 16) =
        make_uint4(v[b][0].y, v[b][1].y, v[b][2].y, v[b][3].y);
    *reinterpret_cast<uint4 *>(sf + (2 * NBLK + b) * 512 + lane * 16) =
        make_uint4(v[b][0].z, v[b][1].z, v[b][2].z, v[b][3].z);
    *reinterpret_cast<uint4 *>(sf + (3 * NBLK + b) * 512 + lane * 16) =
        make_uint4(v[b][0].w, v[b][1].w, v[b][2].w, v[b][3].w);
  }
}

template <bool GATEUP>
__global__ void __launch_bounds__(kW4Threads, 1) w4a4_gemm_kernel(const __grid_constant__ W4Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t *stages = smem_raw + pad;
  uint64_t *full = reinterpret_cast<uint64_t *>(stages + kW4Stages * kW4Stage);
  uint64_t *empty = full + kW4Stages;
  uint64_t *sfready = empty + kW4Stages;  // a stage's scale factors are arranged
  uint64_t *tfull = sfready + kW4Stages;
  uint64_t *tempty = tfull + 1;
  uint64_t *drain = tempty + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  TileSched *sched = reinterpret_cast<TileSched *>(stages + kW4Stages * kW4Stage + 256);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kW4Stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&sfready[s], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, kW4EpiWarps);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, kW4TmemCols);
    tmem_relinquish();
  }
  tile_sched_prologue(p.offsets, p.E, kW4M, p.nf, *sched);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int ntiles = sched->tp[p.E];

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      int stage = 0;
      uint32_t ph = 0, issued = 0, par = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < ntiles; t += gridDim.x) {
        const W4Tile tile = w4_tile<GATEUP>(p, *sched, t);
        for (int k = 0; k < p.ksteps; ++k) {
          if (!mbar_wait(&empty[stage], ph ^ 1u, abort_flag, p.status)) {
            ok = false;
            break;
          }
          uint8_t *st = stages + stage * kW4Stage;
          uint64_t *bar = &full[stage];
          mbar_arrive_expect_tx(bar, kW4Stage);
          tma_load_2d(st, &p.tm_a, bar, k * kW4RowBytes, tile.row0);
          tma_load_2d(st + kW4ABytes + kW4BBytes, &p.tm_sa, bar, k * 16, tile.row0);
          uint8_t *sfb = st + kW4ABytes + kW4BBytes + kW4SfABytes;
          if (GATEUP) {
            tma_load_2d(st + kW4ABytes, &p.tm_b0, bar, k * kW4RowBytes, tile.brow0);
            tma_load_2d(st + kW4ABytes + kW4BBytes / 2, &p.tm_b1, bar, k * kW4RowBytes, tile.brow0);
            tma_load_2d(sfb, &p.tm_sb0, bar, k * 16, tile.brow0);
            tma_load_2d(sfb + kW4SfBBytes / 2, &p.tm_sb1, bar, k * 16, tile.brow0);
          } else {
            tma_load_2d(st + kW4ABytes, &p.tm_b0, bar, k * kW4RowBytes, tile.brow0);
            tma_load_2d(sfb, &p.tm_sb0, bar, k * 16, tile.brow0);
          }
          issued |= 1u << stage;
          par = (par & ~(1u << stage)) | (ph << stage);
          if (++stage == kW4Stages) {
            stage = 0;
            ph ^= 1u;
          }
        }
      }
      if (!ok) {  // let every copy in flight land before the CTA exits
        for (int s = 0; s < kW4Stages; ++s)
          if (issued & (1u << s)) mbar_drain_wait(&full[s], (par >> s) & 1u);
      }
    }
  } else if (warp == 1) {
    {
      // ---------------- MMA issuer: scale copies to tensor memory, then the
      // MMAs; the whole warp runs the loop converged and one elected lane issues
      constexpr uint32_t kIdesc = w4_idesc(kW4M, kW4N);
      int stage = 0;
      uint32_t ph = 0, bph = 0;
      bool ok = true, any = false;
      const bool leader = elect_one();
      for (int t = blockIdx.x; ok && t < ntiles; t += gridDim.x) {
        ok = __all_sync(0xffffffffu, mbar_wait(tempty, bph ^ 1u, abort_flag, p.status));
        if (!ok) break;
        tc_fence_after();
        for (int k = 0; k < p.ksteps; ++k) {
          const bool got = mbar_wait(&full[stage], ph, abort_flag, p.status) &&
                           mbar_wait(&sfready[stage], ph, abort_flag, p.status);
          ok = __all_sync(0xffffffffu, got);
          if (!ok) break;
          tc_fence_after();
          if (leader) {
            uint8_t *st = stages + stage * kW4Stage;
            const uint8_t *sfa = st + kW4ABytes + kW4BBytes;
            const uint8_t *sfb = sfa + kW4SfABytes;
            const uint32_t sf_t = tmem_base + kW4SfCol0 + stage * kW4SfStride;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              tmem_cp_sf(sf_t + 4 * j, sf_desc(smem_u32(sfa + j * 512)));
              tmem_cp_sf(sf_t + 16 + 8 * j, sf_desc(smem_u32(sfb + (2 * j) * 512)));
              tmem_cp_sf(sf_t + 16 + 8 * j + 4, sf_desc(smem_u32(sfb + (2 * j + 1) * 512)));
            }
            const uint64_t adesc = umma_desc_sw128(smem_u32(st));
            const uint64_t bdesc = umma_desc_sw128(smem_u32(st + kW4ABytes));
#pragma unroll
            for (int j = 0; j < 4; ++j)
              umma_fp4(tmem_base, adesc + 2 * j, bdesc + 2 * j, kIdesc, sf_t + 4 * j,
                       sf_t + 16 + 8 * j, (k | j) != 0 ? 1u : 0u);
            umma_commit(&empty[stage]);
          }
          __syncwarp();
          any = true;
          if (++stage == kW4Stages) {
            stage = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        if (leader) umma_commit(tfull);
        __syncwarp();
        bph ^= 1u;
      }
      if (!ok && any && leader) {  // wait for the tensor cores before the memory is released
        umma_commit(drain);
        mbar_drain_wait(drain, 0);
      }
      __syncwarp();
    }
  } else if (warp == 2 || warp == 3) {
    // ---------------- scale arrangers: warp 2 takes the even K slices of the
    // CTA's sequence, warp 3 the odd ones, so arranging one slice overlaps the
    // MMA issue of the previous one.
    int stage = 0, n = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < ntiles; t += gridDim.x) {
      for (int k = 0; k < p.ksteps; ++k, ++n) {
        if ((n & 1) == warp - 2) {
          const bool got = mbar_wait(&full[stage], ph, abort_flag, p.status);
          if (!__all_sync(0xffffffffu, got)) {
            ok = false;
            break;
          }
          uint8_t *sfa = stages + stage * kW4Stage + kW4ABytes + kW4BBytes;
          w4_arrange_sf<1>(sfa, lane);
          w4_arrange_sf<2>(sfa + kW4SfABytes, lane);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sfready[stage]);
        }
        if (++stage == kW4Stages) {
          stage = 0;
          ph ^= 1u;
        }
      }
    }
  } else if (warp >= 4) {
    // ---------------- epilogue: four warps per 32-lane quarter, each with a
    // quarter of the tile's output columns.  A warp copies its accumulator
    // columns into registers and releases tensor memory at once, so the next
    // tile's MMAs overlap the SwiGLU / quantisation / stores below.
    const int q = warp & 3;
    const int part = (warp - 4) >> 2;  // 0..3
    const int row = q * 32 + lane;
    const uint32_t tq = tmem_base + ((uint32_t)(q * 32) << 16);
    uint32_t bph = 0;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
      const W4Tile tile = w4_tile<GATEUP>(p, *sched, t);
      bool ok = mbar_wait(tfull, bph, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, ok)) break;
      bph ^= 1u;
      const bool live = q * 32 < tile.nrows;  // this quarter holds rows of the tile
      uint32_t a[64];
      if (live) {
        tc_fence_after();
        if (GATEUP) {  // gate columns [32 part, +32), up columns 128 + the same
          tmem_ld32(tq + part * 32, *reinterpret_cast<uint32_t(*)[32]>(&a[0]));
          tmem_ld32(tq + 128 + part * 32, *reinterpret_cast<uint32_t(*)[32]>(&a[32]));
        } else {  // output columns [64 part, +64)
          tmem_ld32(tq + part * 64, *reinterpret_cast<uint32_t(*)[32]>(&a[0]));
          tmem_ld32(tq + part * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&a[32]));
        }
        tmem_wait_ld();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty);
      if (!live) continue;
      const bool valid = row < tile.nrows;
      const size_t grow = (size_t)(tile.row0 + row);
      if (GATEUP) {
        const float sg = p.ga * __ldg(p.gw0 + tile.e);
        const float su = p.ga * __ldg(p.gw1 + tile.e);
        const float six_gh = 6.0f * p.gh;
        uint32_t cw[4];
        uint32_t scw = 0;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          float *h = reinterpret_cast<float *>(&a[c * 16]);  // h overwrites g
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float gv = __uint_as_float(a[c * 16 + i]) * sg;
            const float uv = __uint_as_float(a[32 + c * 16 + i]) * su;
            h[i] = __fdividef(gv, 1.0f + __expf(-gv)) * uv;
          }
          uint2 codes;
          const uint32_t sc =
              nvfp4_quantize_block(*reinterpret_cast<float(*)[16]>(h), six_gh, p.gh, codes);
          cw[2 * c] = codes.x;
          cw[2 * c + 1] = codes.y;
          scw |= sc << (8 * c);
        }
        if (valid) {
          const int feat0 = tile.f * 128 + part * 32;
          *reinterpret_cast<uint4 *>(p.hq + grow * (p.out_cols / 2) + feat0 / 2) =
              make_uint4(cw[0], cw[1], cw[2], cw[3]);
          *reinterpret_cast<uint16_t *>(p.hs + grow * (p.out_cols / 16) + feat0 / 16) =
              (uint16_t)scw;
        }
      } else if (valid) {
        const float w = __ldg(p.topk_w + __ldg(p.row_src + tile.row0 + row));
        const float sc = p.ga * __ldg(p.gw0 + tile.e) * w;
        uint4 *d4 = reinterpret_cast<uint4 *>(p.y + grow * p.out_cols + tile.f * 256 + part * 64);
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          uint32_t pk[4];
#pragma unroll
          for (int j = 0; j < 4; ++j)
            pk[j] = pack_bf16x2_w4(__uint_as_float(a[8 * v + 2 * j]) * sc,
                                   __uint_as_float(a[8 * v + 2 * j + 1]) * sc);
          d4[v] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kW4TmemCols);
  }
}

// Rows of bf16 x -> NVFP4 codes and scales; one warp per row, one 16-value
// block per lane and step.  With row_src, output row r quantises
// x[row_src[r] / top_k] for r < offsets[E] (the dispatch's gather);
// without, row r quantises x[r] for r < rows.
__global__ void __launch_bounds__(256)
    quantize_rows_kernel(const uint4 *__restrict__ x, const int32_t *__restrict__ row_src,
                         const int32_t *__restrict__ offsets, int E, int top_k, int rows, int cols,
                         float g, uint2 *__restrict__ q, uint8_t *__restrict__ s) {
  const int n = row_src ? offsets[E] : rows;
  const int lane = threadIdx.x & 31;
  const int nwarps = gridDim.x * (blockDim.x >> 5);
  const int nblk = cols / 16;
  const float six_g = 6.0f * g;
  for (int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < n; r += nwarps) {
    const int src = row_src ? row_src[r] / top_k : r;
    const uint4 *xr = x + (size_t)src * (cols / 8);
    for (int b = lane; b < nblk; b += 32) {
      const uint4 lo = xr[2 * b], hi = xr[2 * b + 1];
      const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
      float v[16];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[i]));
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
      }
      uint2 codes;
      const uint32_t sc = nvfp4_quantize_block(v, six_g, g, codes);
      q[(size_t)r * nblk + b] = codes;
      s[(size_t)r * nblk + b] = (uint8_t)sc;
    }
  }
}

// The dispatch's form for the forward pass: token t is quantised once and its
// codes and scales are written to every permuted row that holds one of its
// entries (slot_of[t*k + j]; dropped entries have slot -1).  One warp per
// (token, 32 blocks of its row), one 16-value block per lane, so a small batch
// still spreads over many warps.
__global__ void __launch_bounds__(256)
    quantize_scatter_kernel(const uint4 *__restrict__ x, const int32_t *__restrict__ slot_of,
                            int T, int top_k, int cols, float g, uint2 *__restrict__ q,
                            uint8_t *__restrict__ s) {
  const int lane = threadIdx.x & 31;
  const long nwarps = (long)gridDim.x * (blockDim.x >> 5);
  const int nblk = cols / 16;
  const int segs = (nblk + 31) / 32;
  const float six_g = 6.0f * g;
  for (long w = (long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); w < (long)T * segs;
       w += nwarps) {
    const int t = (int)(w / segs);
    const uint4 *xr = x + (size_t)t * (cols / 8);
    const int my_slot = lane < top_k ? __ldg(slot_of + (size_t)t * top_k + lane) : -1;
    {  // whole warp: the slots are shuffled
      const int b = (int)(w - (long)t * segs) * 32 + lane;
      uint2 codes = make_uint2(0u, 0u);
      uint8_t sc = 0;
      if (b < nblk) {
        const uint4 lo = xr[2 * b], hi = xr[2 * b + 1];
        const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
        float v[16];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[i]));
          v[2 * i] = f.x;
          v[2 * i + 1] = f.y;
        }
        sc = (uint8_t)nvfp4_quantize_block(v, six_g, g, codes);
      }
      for (int j = 0; j < top_k; ++j) {
        const int slot = __shfl_sync(0xffffffffu, my_slot, j);
        if (slot >= 0 && b < nblk) {
          q[(size_t)slot * nblk + b] = codes;
          s[(size_t)slot * nblk + b] = sc;
        }
      }
    }
  }
}

}  // namespace

moe_status launch_quantize_scatter_nvfp4(const void *x, const int32_t *slot_of, int T, int top_k,
                                         int cols, float g, uint8_t *q, uint8_t *s,
                                         cudaStream_t stream) {
  if (T <= 0) return MOE_OK;
  const long tasks = (long)T * ((cols / 16 + 31) / 32);
  const int blocks = (int)std::max<long>(1, std::min<long>((tasks + 7) / 8, device_sm_count() * 8));
  quantize_scatter_kernel<<<blocks, 256, 0, stream>>>(static_cast<const uint4 *>(x), slot_of, T,
                                                     top_k, cols, g, reinterpret_cast<uint2 *>(q),
                                                     s);
  return cudaPeekAtLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status launch_quantize_nvfp4(const void *x, const int32_t *row_src, const int32_t *offsets,
                                 int E, int top_k, int rows, int cols, float g, uint8_t *q,
                                 uint8_t *s, cudaStream_t stream) {
  if (rows <= 0) return MOE_OK;
  const int blocks = std::max(1, std::min((rows + 7) / 8, device_sm_count() * 8));
  quantize_rows_kernel<<<blocks, 256, 0, stream>>>(static_cast<const uint4 *>(x), row_src, offsets,
                                                  E, top_k, rows, cols, g,
                                                  reinterpret_cast<uint2 *>(q), s);
  return cudaPeekAtLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status launch_experts_w4a4(const moe_dims &d, const moe_experts &ex, const uint8_t *xq,
                               const uint8_t *xs, const int32_t *offsets, const int32_t *row_src,
                               const float *topk_w, void *y_partial, uint8_t *hq, uint8_t *hs,
                               uint32_t *status, cudaStream_t stream) {
  const uint64_t Tk = (uint64_t)d.T * d.top_k;
  const uint64_t E = d.E, H = d.H, I = d.I;
  if (ensure_smem_limit((const void *)w4a4_gemm_kernel<true>, kW4SmemBytes) != MOE_OK ||
      ensure_smem_limit((const void *)w4a4_gemm_kernel<false>, kW4SmemBytes) != MOE_OK)
    return MOE_ERR_CUDA;
  const CUtensorMapDataType U8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const int grid = device_sm_count();

  W4Params g{};
  bool ok = make_tmap_2d(&g.tm_a, xq, U8, 1, H / 2, Tk, 128, 128, true) &&
            make_tmap_2d(&g.tm_sa, xs, U8, 1, H / 16, Tk, 16, 128, false) &&
            make_tmap_2d(&g.tm_b0, ex.w_gate, U8, 1, H / 2, E * I, 128, 128, true) &&
            make_tmap_2d(&g.tm_sb0, ex.s_gate, U8, 1, H / 16, E * I, 16, 128, false) &&
            make_tmap_2d(&g.tm_b1, ex.w_up, U8, 1, H / 2, E * I, 128, 128, true) &&
            make_tmap_2d(&g.tm_sb1, ex.s_up, U8, 1, H / 16, E * I, 16, 128, false);
  if (!ok) return MOE_ERR_CUDA;
  g.offsets = offsets;
  g.row_src = row_src;
  g.topk_w = topk_w;
  g.gw0 = ex.g_gate;
  g.gw1 = ex.g_up;
  g.ga = ex.x_global;
  g.gh = ex.h_global;
  g.hq = hq;
  g.hs = hs;
  g.E = d.E;
  g.ksteps = d.H / 256;
  g.nf = d.I / 128;
  g.b_rows = d.I;
  g.out_cols = d.I;
  g.status = status;
  w4a4_gemm_kernel<true><<<grid, kW4Threads, kW4SmemBytes, stream>>>(g);
  if (cudaPeekAtLastError() != cudaSuccess) return MOE_ERR_CUDA;

  W4Params dn{};
  ok = make_tmap_2d(&dn.tm_a, hq, U8, 1, I / 2, Tk, 128, 128, true) &&
       make_tmap_2d(&dn.tm_sa, hs, U8, 1, I / 16, Tk, 16, 128, false) &&
       make_tmap_2d(&dn.tm_b0, ex.w_down, U8, 1, I / 2, E * H, 128, 256, true) &&
       make_tmap_2d(&dn.tm_sb0, ex.s_down, U8, 1, I / 16, E * H, 16, 256, false);
  if (!ok) return MOE_ERR_CUDA;
  dn.tm_b1 = dn.tm_b0;
  dn.tm_sb1 = dn.tm_sb0;
  dn.offsets = offsets;
  dn.row_src = row_src;
  dn.topk_w = topk_w;
  dn.gw0 = ex.g_down;
  dn.gw1 = ex.g_down;
  dn.ga = ex.h_global;
  dn.gh = 1.0f;
  dn.y = static_cast<__nv_bfloat16 *>(y_partial);
  dn.E = d.E;
  dn.ksteps = d.I / 256;
  dn.nf = d.H / 256;
  dn.b_rows = d.H;
  dn.out_cols = d.H;
  dn.status = status;
  w4a4_gemm_kernel<false><<<grid, kW4Threads, kW4SmemBytes, stream>>>(dn);
  return cudaPeekAtLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace beam
