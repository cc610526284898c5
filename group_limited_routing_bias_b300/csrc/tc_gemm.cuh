// Warp-specialised tcgen05 GEMM skeleton for sm_103a.
//
// One CTA (256 threads) per SM, persistent over tiles.  Each tile computes
// NA accumulators D_a[128 x BN] (fp32, tensor memory) = A_a[128 x K] . B[BN x K]^T,
// with every operand K-major bf16 staged by TMA in 64-wide K slices with the
// 128-byte swizzle.
//   warp 0 lane 0 : TMA producer, STAGES-deep shared-memory ring
//   warp 1        : MMA issuer (tcgen05.mma, M=128, N=BN, K=16 per instruction),
//                   the whole warp converged, one elected lane issuing
//   warp 2        : tensor-memory allocation / release
//   warps 4..7    : epilogue; warp 4+q reads accumulator rows 32q..32q+31
// The accumulators are double-buffered in tensor memory when they fit, so
// the epilogue of one tile overlaps the main loop of the next.
//
// Problems whose weights arrive packed (NVFP4) add a converter role and a
// second ring: warp 0 TMA-loads the packed bytes of each K slice into a deep
// raw ring (RSTAGES), warp 3 the activation tile into the operand ring;
//   warps 8..     : P::CONVERT_WARPS converter warps (optional, default 8) in
//                   P::CGROUPS groups (optional, default 1) taking alternate
//                   K slices (two groups dequantise two slices at once; faster
//                   for the large-batch tiles): wait for a slice's raw
//                   bytes, dequantise them into the operand slot's swizzled
//                   weight tile, release the raw slot at once, fence the
//                   generic proxy against the tensor cores' async proxy, then
//                   signal the MMA.
// The raw ring is refilled as soon as a slice is converted, so the bytes in
// flight are not held back by MMA completion.
//
// Tile schedule: by default CTA b takes tiles b, b + grid, b + 2 grid, ...
// A problem with P::DYNAMIC (bf16 problems) instead has its producer take the
// next tile from a global counter (P::Params::sched_counters[0]) as it starts
// loading it, and hand the index to the MMA and epilogue roles through a
// kTileRing-deep ring in shared memory, so SMs that stream faster take more
// tiles and the tail shrinks.  The last CTA to finish zeroes both counters
// (sched_counters[1] counts finished CTAs), so they start at zero for the next
// launch; they must be zero before the first.
//
// Optional hooks for a producer/consumer pair of launches (the decode gate/up
// and down GEMMs), all default off:
//   static constexpr bool PDL_PRIMARY;    every CTA allows the next launch (a
//                                         programmatic dependent) to start once
//                                         SMs free up (griddepcontrol.launch_dependents)
//   static constexpr bool PDL_SECONDARY;  launched as that dependent: the CTAs wait
//                                         for the primary grid only before exiting
//   static constexpr bool PDL_WAIT_B;     (CONVERT) the activation producer waits
//                                         for the primary grid before its first load
//   static bool tile_ready(const Params&, const Tile&, volatile int *abort)
//                                         producer, before a tile's first load
//                                         (false: gave up, the CTA aborts)
//   static void tile_done(const Params&, const Tile&)
//                                         lane 0 of each of the four epilogue warps,
//                                         after the warp stored its rows of the tile
//   static void last_cta(const Params&)   the last CTA to finish (dynamic schedule)
//
// A problem class P supplies the shapes and the tile schedule:
//   static constexpr int BN, NA, STAGES, NBUF, TX_BYTES (or a tx_bytes hook, below);
//   static constexpr bool CONVERT, F16;   (packed weights; f16 instead of bf16 operands)
//   static constexpr int KSUB;            (optional, default 1: 64-wide K slices per stage;
//                                          two let each weight row arrive as 256 contiguous
//                                          bytes per stage, which HBM streams better)
//   static constexpr int RSTAGES, RAW_BYTES;  (CONVERT: raw ring depth and slot size)
//   struct Params { ...; uint32_t *status; };  struct Sched;  struct Tile;
//   static void prologue(const Params&, Sched&)   (all threads; may __syncthreads)
//   static int  num_tiles(const Params&, const Sched&)
//   static Tile tile(const Params&, const Sched&, int t)
//   static int  num_k(const Params&, const Tile&)
//   static void load(const Params&, const Tile&, int k, uint8_t *stage, uint64_t *bar)
//   static uint32_t tx_bytes(const Params&, const Tile&)  (optional: the bytes load()
//                                          brings for that tile, when not TX_BYTES)
//   static void epilogue(const Params&, const Tile&, uint32_t taddr, int row)
//   static constexpr int EXTRA_TMEM_COLS;  (optional, default 0: tensor-memory
//                                          columns after the NBUF accumulators,
//                                          at taddr - buf * NA * BN + NBUF * NA * BN)
//   CONVERT problems load the operand ring's activation tile with load() and the
//   raw ring with
//   static void load_raw(const Params&, const Tile&, int k, uint8_t *raw, uint64_t *raw_bar)
//   static void convert(const Params&, const Tile&, int k, uint8_t *stage, const uint8_t *raw,
//                       int ctid)   (ctid: thread within its converter group)
#pragma once

#include <type_traits>
#include <utility>

#include "ptx.cuh"

namespace beam {

constexpr int kTileM = 128;
constexpr int kTileK = 64;                       // bf16 elements per 128-byte row
constexpr int kATileBytes = kTileM * kTileK * 2;  // 16 KB
constexpr int kSmemLimit = 232448;                // 227 KB dynamic shared memory
constexpr int kSmemReserve = 4096;                // alignment slack + barriers

template <int BN, int NA>
struct StageGeom {
  static constexpr int kOperandBytes = NA * kATileBytes + BN * kTileK * 2;
  static constexpr int kBytes = kOperandBytes;
  static_assert(kBytes % 1024 == 0, "stage must keep 1024-byte alignment");
};

template <class P, class = void>
struct KSubOf {
  static constexpr int value = 1;
};
template <class P>
struct KSubOf<P, std::void_t<decltype(P::KSUB)>> {
  static constexpr int value = P::KSUB;
};

// A stage holds KSUB consecutive 64-wide K slices, each laid out as StageGeom.
template <class P>
__host__ __device__ constexpr int stage_bytes_of() {
  return StageGeom<P::BN, P::NA>::kBytes * KSubOf<P>::value;
}

template <class P>
__host__ __device__ constexpr int raw_ring_bytes_of() {
  return P::CONVERT ? P::RSTAGES * P::RAW_BYTES : 0;
}

template <class P>
__host__ __device__ constexpr int smem_bytes_for() {
  return kSmemReserve + P::STAGES * stage_bytes_of<P>() + raw_ring_bytes_of<P>() +
         (int)sizeof(typename P::Sched);
}

constexpr int kConvertWarps = 8;

// Converter groups taking alternate K slices (optional P::CGROUPS, default 1).
template <class P, class = void>
struct CGroupsOf {
  static constexpr int value = 1;
};
template <class P>
struct CGroupsOf<P, std::void_t<decltype(P::CGROUPS)>> {
  static constexpr int value = P::CGROUPS;
};

// Converter warps (optional P::CONVERT_WARPS, default kConvertWarps).
template <class P, class = void>
struct ConvertWarpsOf {
  static constexpr int value = kConvertWarps;
};
template <class P>
struct ConvertWarpsOf<P, std::void_t<decltype(P::CONVERT_WARPS)>> {
  static constexpr int value = P::CONVERT_WARPS;
};

template <class P, class = void>
struct DynamicOf {
  static constexpr bool value = false;
};
template <class P>
struct DynamicOf<P, std::void_t<decltype(P::DYNAMIC)>> {
  static constexpr bool value = P::DYNAMIC;
};

constexpr int kTileRing = 4;

template <class P, class = void>
struct PdlPrimaryOf {
  static constexpr bool value = false;
};
template <class P>
struct PdlPrimaryOf<P, std::void_t<decltype(P::PDL_PRIMARY)>> {
  static constexpr bool value = P::PDL_PRIMARY;
};
template <class P, class = void>
struct PdlSecondaryOf {
  static constexpr bool value = false;
};
template <class P>
struct PdlSecondaryOf<P, std::void_t<decltype(P::PDL_SECONDARY)>> {
  static constexpr bool value = P::PDL_SECONDARY;
};
// Optional P::PDL_WAIT_B (with CONVERT): the activation tiles are the output
// of the launch this one depends on; the activation producer alone waits for
// it (griddepcontrol.wait) before its first load, the weights stream at once.
template <class P, class = void>
struct PdlWaitBOf {
  static constexpr bool value = false;
};
template <class P>
struct PdlWaitBOf<P, std::void_t<decltype(P::PDL_WAIT_B)>> {
  static constexpr bool value = P::PDL_WAIT_B;
};
template <class P, class = void>
struct HasTileReady : std::false_type {};
template <class P>
struct HasTileReady<P, std::void_t<decltype(P::tile_ready(std::declval<const typename P::Params &>(),
                                                           std::declval<const typename P::Tile &>(),
                                                           std::declval<volatile int *>()))>>
    : std::true_type {};
template <class P, class = void>
struct HasTileDone : std::false_type {};
template <class P>
struct HasTileDone<P, std::void_t<decltype(P::tile_done(std::declval<const typename P::Params &>(),
                                                         std::declval<const typename P::Tile &>()))>>
    : std::true_type {};
template <class P, class = void>
struct HasLastCta : std::false_type {};
template <class P>
struct HasLastCta<P, std::void_t<decltype(P::last_cta(std::declval<const typename P::Params &>()))>>
    : std::true_type {};

// Tensor-memory columns a problem keeps beyond its accumulators (optional
// P::EXTRA_TMEM_COLS, default 0), at [NBUF * NA * BN, + EXTRA) of every lane.
template <class P, class = void>
struct ExtraTmemOf {
  static constexpr int value = 0;
};
template <class P>
struct ExtraTmemOf<P, std::void_t<decltype(P::EXTRA_TMEM_COLS)>> {
  static constexpr int value = P::EXTRA_TMEM_COLS;
};

template <class P>
__host__ __device__ constexpr int threads_for() {
  return P::CONVERT ? 256 + 32 * ConvertWarpsOf<P>::value : 256;
}

template <class P, class = void>
struct HasTxBytes : std::false_type {};
template <class P>
struct HasTxBytes<P, std::void_t<decltype(P::tx_bytes(std::declval<const typename P::Params &>(),
                                                       std::declval<const typename P::Tile &>()))>>
    : std::true_type {};

template <class P>
__device__ __forceinline__ uint32_t tx_bytes_of(const typename P::Params &p, const typename P::Tile &t) {
  if constexpr (HasTxBytes<P>::value) return P::tx_bytes(p, t);
  else return P::TX_BYTES;
}

// Token rows of the activation box that a token-major tile loads: the MMA
// always reads 128 rows, but rows past the tile's own are never stored, so a
// tile of a few rows loads a 32- or 64-row box and leaves the rest stale.
__host__ __device__ constexpr int act_box_rows(int nrows) {
  return nrows <= 32 ? 32 : nrows <= 64 ? 64 : 128;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

template <class P>
__global__ void __launch_bounds__(threads_for<P>(), 1)
    tc_gemm_kernel(const __grid_constant__ typename P::Params p) {
  constexpr int STAGE = stage_bytes_of<P>();
  constexpr uint32_t kAccCols = P::NA * P::BN;
  constexpr uint32_t kTmemCols = tmem_cols_pow2(P::NBUF * kAccCols + ExtraTmemOf<P>::value);
  constexpr uint32_t kIdesc = P::F16 ? umma_idesc_f16(kTileM, P::BN) : umma_idesc_bf16(kTileM, P::BN);
  static_assert(P::NBUF * kAccCols + ExtraTmemOf<P>::value <= 512, "tensor memory overflow");
  constexpr int CG = CGroupsOf<P>::value;
  constexpr int kGroupWarps = ConvertWarpsOf<P>::value / CG;
  static_assert(ConvertWarpsOf<P>::value % CG == 0, "converter groups must split the converter warps");
  // Barrier waits go by phase parity, which is unambiguous only while a waiter
  // is at most one phase behind.  A group reaching slice n must already know
  // that slice n - RSTAGES (same raw slot) landed, and that the MMA of slice
  // n - 2 STAGES (same operand slot, two uses back) completed: both hold when
  // the earlier slice is the group's own (RSTAGES a multiple of the group
  // count) and when its previous slice's wait covers it (STAGES >= groups).
  static_assert(CG == 1 || (P::RSTAGES % CG == 0 && P::STAGES >= CG),
                "converter groups need RSTAGES % groups == 0 and STAGES >= groups");
  static_assert(KSubOf<P>::value == 1 || !P::CONVERT, "several K slices per stage: bf16 path only");
  static_assert(P::BN % 16 == 0 && P::BN >= 16 && P::BN <= 256, "invalid MMA N");
  constexpr bool DYN = DynamicOf<P>::value;
  static_assert(!DYN || !P::CONVERT, "dynamic tile schedule: problems without converters only");

  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t *stages = smem_raw + pad;
  constexpr int RS = P::CONVERT ? P::RSTAGES : 1;
  uint8_t *raws = stages + P::STAGES * STAGE;  // raw ring (CONVERT only)
  uint64_t *full = reinterpret_cast<uint64_t *>(raws + raw_ring_bytes_of<P>());
  uint64_t *empty = full + P::STAGES;
  uint64_t *tfull = empty + P::STAGES;
  uint64_t *tempty = tfull + P::NBUF;
  uint64_t *ready = tempty + P::NBUF;  // converters -> MMA (CONVERT only)
  uint64_t *raw_full = ready + P::STAGES;
  uint64_t *raw_empty = raw_full + RS;
  uint64_t *drain = raw_empty + RS;
  uint64_t *tr_full = drain + 1;  // tile ring (DYNAMIC only)
  uint64_t *tr_empty = tr_full + kTileRing;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tr_empty + kTileRing);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  volatile int *tring = abort_flag + 1;
  static_assert((3 * P::STAGES + 2 * P::NBUF + 2 * RS + 1 + 2 * kTileRing) * 8 + 8 +
                        4 * kTileRing <= 1024,
                "barrier area");
  typename P::Sched *sched = reinterpret_cast<typename P::Sched *>(
      raws + raw_ring_bytes_of<P>() + 1024);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < P::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < P::NBUF; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4);
    }
    for (int s = 0; s < P::STAGES; ++s) mbar_init(&ready[s], kGroupWarps);
    for (int s = 0; s < RS; ++s) {
      mbar_init(&raw_full[s], 1);
      mbar_init(&raw_empty[s], kGroupWarps);
    }
    mbar_init(drain, 1);
    for (int s = 0; s < kTileRing; ++s) {
      mbar_init(&tr_full[s], 1);
      mbar_init(&tr_empty[s], 1 + 4);  // the MMA thread and the four epilogue warps
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  P::prologue(p, *sched);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int ntiles = P::num_tiles(p, *sched);
  if constexpr (PdlPrimaryOf<P>::value) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // Tile feed.  `cur` is the static cursor; slot / tph index the tile ring.
  // The producer publishes each tile it takes (-1 at the end); consumers read
  // them in order (whole_warp: every lane waits, lane 0 releases the slot).
  auto produce_tile = [&](int &cur, int &slot, uint32_t &tph, bool &ok) -> int {
    if constexpr (!DYN) {
      const int t = cur;
      cur += gridDim.x;
      return t < ntiles ? t : -1;
    } else {
      int t = (int)atomicAdd(p.sched_counters, 1u);
      if (t >= ntiles) t = -1;
      if (!mbar_wait(&tr_empty[slot], tph ^ 1u, abort_flag, p.status)) {
        ok = false;
        return -1;
      }
      tring[slot] = t;
      mbar_arrive(&tr_full[slot]);
      if (++slot == kTileRing) {
        slot = 0;
        tph ^= 1u;
      }
      return t;
    }
  };
  auto consume_tile = [&](int &cur, int &slot, uint32_t &tph, bool &ok, bool whole_warp) -> int {
    if constexpr (!DYN) {
      const int t = cur;
      cur += gridDim.x;
      return t < ntiles ? t : -1;
    } else {
      bool got = mbar_wait(&tr_full[slot], tph, abort_flag, p.status);
      if (whole_warp) got = __all_sync(0xffffffffu, got);
      if (!got) {
        ok = false;
        return -1;
      }
      const int t = tring[slot];
      if (whole_warp) __syncwarp();
      if (!whole_warp || lane == 0) mbar_arrive(&tr_empty[slot]);
      if (++slot == kTileRing) {
        slot = 0;
        tph ^= 1u;
      }
      return t;
    }
  };

  if (warp == 0 || (P::CONVERT && warp == 3)) {
    if (lane == 0) {
      // ---------------- TMA producers.  Without conversion warp 0 fills the
      // operand ring.  With it, warp 0 streams packed weights into the raw ring
      // (gated only by the converters freeing raw slots) and warp 3 issues the
      // activation tiles into the operand ring (gated by MMA completion).
      const bool raw_role = P::CONVERT && warp == 0;
      if constexpr (P::CONVERT && PdlWaitBOf<P>::value) {
        if (!raw_role) asm volatile("griddepcontrol.wait;" ::: "memory");
      }
      int stage = 0, cur = blockIdx.x, tslot = 0;
      uint32_t ph = 0, issued = 0, par = 0, tph = 0;
      bool ok = true;
      for (int t = produce_tile(cur, tslot, tph, ok); ok && t >= 0;
           t = produce_tile(cur, tslot, tph, ok)) {
        const typename P::Tile tile = P::tile(p, *sched, t);
        const int nk = P::num_k(p, tile);
        if constexpr (HasTileReady<P>::value) {
          if (!P::tile_ready(p, tile, abort_flag)) {
            ok = false;
            break;
          }
        }
        for (int k = 0; k < nk; ++k) {
          if constexpr (P::CONVERT) {
            if (raw_role) {
              if (!mbar_wait(&raw_empty[stage], ph ^ 1u, abort_flag, p.status)) {
                ok = false;
                break;
              }
              mbar_arrive_expect_tx(&raw_full[stage], P::RAW_BYTES);
              P::load_raw(p, tile, k, raws + stage * P::RAW_BYTES, &raw_full[stage]);
            } else {
              if (!mbar_wait(&empty[stage], ph ^ 1u, abort_flag, p.status)) {
                ok = false;
                break;
              }
              mbar_arrive_expect_tx(&full[stage], tx_bytes_of<P>(p, tile));
              P::load(p, tile, k, stages + stage * STAGE, &full[stage]);
            }
          } else {
            if (!mbar_wait(&empty[stage], ph ^ 1u, abort_flag, p.status)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&full[stage], tx_bytes_of<P>(p, tile));
            P::load(p, tile, k, stages + stage * STAGE, &full[stage]);
          }
          issued |= 1u << stage;
          par = (par & ~(1u << stage)) | (ph << stage);
          if (++stage == (raw_role ? RS : P::STAGES)) {
            stage = 0;
            ph ^= 1u;
          }
        }
      }
      if (!ok) {  // let every copy still in flight land before the CTA exits
        uint64_t *bars = raw_role ? raw_full : full;
        for (int s = 0; s < (raw_role ? RS : P::STAGES); ++s)
          if (issued & (1u << s)) mbar_drain_wait(&bars[s], (par >> s) & 1u);
      }
    }
  } else if (warp == 1) {
    {
      // ---------------- MMA issuer: the whole warp runs the loop converged, so
      // descriptors and addresses stay warp-uniform, and one elected lane issues
      // (a lone issuing lane competes for issue slots and slows the MMAs)
      int stage = 0, buf = 0, cur = blockIdx.x, tslot = 0;
      uint32_t ph = 0, bph = 0, tph = 0;
      bool ok = true, any = false;
      const bool leader = elect_one();
      for (int t = consume_tile(cur, tslot, tph, ok, true); ok && t >= 0;
           t = consume_tile(cur, tslot, tph, ok, true)) {
        const typename P::Tile tile = P::tile(p, *sched, t);
        const int nk = P::num_k(p, tile);
        ok = __all_sync(0xffffffffu, mbar_wait(&tempty[buf], bph ^ 1u, abort_flag, p.status));
        if (!ok) break;
        tc_fence_after();
        const uint32_t d0 = tmem_base + buf * kAccCols;
        for (int k = 0; k < nk; ++k) {
          bool got = mbar_wait(&full[stage], ph, abort_flag, p.status) &&
                     (!P::CONVERT || mbar_wait(&ready[stage], ph, abort_flag, p.status));
          ok = __all_sync(0xffffffffu, got);
          if (!ok) break;
          tc_fence_after();
          if (leader) {
#pragma unroll
            for (int sub = 0; sub < KSubOf<P>::value; ++sub) {
              const uint32_t sa =
                  smem_u32(stages + stage * STAGE) + sub * StageGeom<P::BN, P::NA>::kBytes;
              const uint64_t bdesc = umma_desc_sw128(sa + P::NA * kATileBytes);
#pragma unroll
              for (int kk = 0; kk < kTileK / 16; ++kk) {
#pragma unroll
                for (int a = 0; a < P::NA; ++a) {
                  const uint64_t adesc = umma_desc_sw128(sa + a * kATileBytes);
                  umma_bf16(d0 + a * P::BN, adesc + 2 * kk, bdesc + 2 * kk, kIdesc,
                            (k | kk | sub) != 0 ? 1u : 0u);
                }
              }
            }
            umma_commit(&empty[stage]);
          }
          __syncwarp();
          any = true;
          if (++stage == P::STAGES) {
            stage = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        if (leader) umma_commit(&tfull[buf]);
        __syncwarp();
        if (++buf == P::NBUF) {
          buf = 0;
          bph ^= 1u;
        }
      }
      if (!ok && any && leader) {  // wait for the tensor cores before the memory is released
        umma_commit(drain);
        mbar_drain_wait(drain, 0);
      }
      __syncwarp();
    }
  } else if (P::CONVERT && warp >= 8) {
    // ---------------- converters: raw packed weights -> swizzled operand tile
    const int group = CG == 1 ? 0 : (warp - 8) / kGroupWarps;
    const int gtid = threadIdx.x - 256 - group * 32 * kGroupWarps;
    int stage = 0, rstage = 0, n = 0;
    uint32_t ph = 0, rph = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < ntiles; t += gridDim.x) {
      const typename P::Tile tile = P::tile(p, *sched, t);
      const int nk = P::num_k(p, tile);
      for (int k = 0; k < nk; ++k, ++n) {
        if (CG == 1 || n % CG == group) {
          // the raw slice has landed, and the operand slot it goes to is free
          bool got = mbar_wait(&raw_full[rstage], rph, abort_flag, p.status) &&
                     mbar_wait(&empty[stage], ph ^ 1u, abort_flag, p.status);
          got = __all_sync(0xffffffffu, got);
          if (!got) {
            ok = false;
            break;
          }
          if constexpr (P::CONVERT)
            P::convert(p, tile, k, stages + stage * STAGE, raws + rstage * P::RAW_BYTES, gtid);
          __syncwarp();
          if (lane == 0) mbar_arrive(&raw_empty[rstage]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&ready[stage]);
        }
        if (++rstage == RS) {
          rstage = 0;
          rph ^= 1u;
        }
        if (++stage == P::STAGES) {
          stage = 0;
          ph ^= 1u;
        }
      }
    }
  } else if (warp >= 4 && warp < 8) {
    // ---------------- epilogue
    const int q = warp & 3;
    const int row = q * 32 + lane;
    int buf = 0, cur = blockIdx.x, tslot = 0;
    uint32_t bph = 0, tph = 0;
    bool fed = true;
    for (int t = consume_tile(cur, tslot, tph, fed, true); fed && t >= 0;
         t = consume_tile(cur, tslot, tph, fed, true)) {
      const typename P::Tile tile = P::tile(p, *sched, t);
      bool ok = mbar_wait(&tfull[buf], bph, abort_flag, p.status);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + buf * kAccCols;
      P::epilogue(p, tile, taddr, row);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[buf]);
      if constexpr (HasTileDone<P>::value) {
        if (lane == 0) P::tile_done(p, tile);
      }
      if (++buf == P::NBUF) {
        buf = 0;
        bph ^= 1u;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (DYN) {
    if (threadIdx.x == 0) {
      __threadfence();
      if (atomicAdd(p.sched_counters + 1, 1u) == gridDim.x - 1) {
        p.sched_counters[0] = 0;  // every CTA has taken its last tile
        p.sched_counters[1] = 0;
        if constexpr (HasLastCta<P>::value) P::last_cta(p);
        __threadfence();
      }
    }
  }
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
  // A dependent launch: order this grid's completion after the primary's.
  if constexpr (PdlSecondaryOf<P>::value) asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace beam
