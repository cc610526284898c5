// Warp-specialised tcgen05 GEMM for packed weights whose dequantised form is
// the MMA's A operand in TENSOR memory (sm_103a).
//
// Each tile computes NA accumulators D_a[128 x BN] (fp32, tensor memory) =
// W_a[128 x K] . X[BN x K]^T: 128 weight rows of one expert on the MMA's M
// side (gate and up rows for NA = 2), the expert's token rows on N.  Issued
// by an elected lane of a converged warp, a kind::f16 MMA with M = 128, N = 32
// and A in tensor memory takes 16 clocks (N = 16: 9, N = 64: 32), the tensor
// rate; with A in shared memory an N = 32 MMA takes 40 clocks, bound by
// shared-memory reads of A, and the dequantised weights would cross shared
// memory twice (the converters' store, the MMA's read).  Here the converters
// write the weights into tensor memory with tcgen05.st; shared memory only
// carries the packed bytes and the small activation tiles.
//
// The K loop runs in steps of KS 64-wide slices, KS * NA = 4 A tiles of 128
// rows x 64 k per step.  A barrier wait right after a commit costs a few
// hundred clocks (it returns once the committed MMAs are done), so each step
// carries 16 MMAs per wait and commit.
//
// One CTA per SM, persistent, 768 threads:
//   warp 0 lane 0 : weight producer: each step's packed weights into a deep
//                   raw ring (RS steps), freed by the converters
//   warp 3 lane 0 : activation producer: the step's KS activation tiles (BN
//                   token rows x 64 k, 128-byte swizzle, the MMA's B operand)
//                   into a B ring of BS steps, freed by the MMA's commits, so
//                   the activations are fetched well before the step is due
//   warp 1        : MMA issuer, converged, one elected lane issuing:
//                   tcgen05.mma kind::f16 (f16 operands) with A from tensor
//                   memory; one wait and one commit per step
//   warp 2        : tensor-memory allocation / release (all 512 columns)
//   warps 4..7    : epilogue; warp 4+q reads accumulator rows 32q..32q+31
//   warps 8..23   : converters, four warpgroups; group g dequantises A tile g
//                   of every step (slice g / NA, matrix g % NA); thread (q,
//                   lane) takes weight row 32q + lane (tensor-memory lane
//                   quarter q) into 32 columns of the stage.  After the B tiles
//                   have landed too, the group signals the stage full.
// Tensor memory: accumulators [0, NBUF * NA * BN); then AST stages of
// 4 * 32 columns (four A tiles of 128 rows x 64 k in f16 pairs).
//
// Every wait is bounded (ptx.cuh); on expiry the CTA records MOE_DEV_TIMEOUT,
// lets its copies and MMAs drain, frees tensor memory and returns.
//
// A problem class P supplies:
//   static constexpr int BN, NA, KS, NBUF, AST, RS, BS, RAW_BYTES;   (RAW_BYTES: one step)
//   static constexpr bool DYNAMIC, PDL_PRIMARY, PDL_SECONDARY, PDL_WAIT_B;
//   struct Params { ...; uint32_t *status; uint32_t *sched_counters; };
//   struct Sched; struct Tile;
//   static void prologue(const Params&, Sched&)
//   static int  num_tiles(const Params&, const Sched&)
//   static Tile tile(const Params&, const Sched&, int t)
//   static int  num_steps(const Params&, const Tile&)
//   static uint32_t b_tx_bytes(const Params&, const Tile&)       (one step)
//   static void load_b(const Params&, const Tile&, int s, uint8_t *bslot, uint64_t *bar)
//                                       (KS tiles of BN rows x 128 bytes)
//   static void load_raw(const Params&, const Tile&, int s, uint8_t *raw, uint64_t *bar)
//   struct Row;                         (one weight row's packed bytes in registers)
//   static void load_row(const Params&, const Tile&, int s, const uint8_t *raw, int j,
//                        int a, int row, Row&)   (slice j of the step, matrix a)
//   static void convert_half(const Row&, int h, uint32_t (&out)[16])
//                                       (f16 pairs of k 32h .. 32h + 31)
//   static void epilogue(const Params&, const Tile&, uint32_t taddr, int row)
//   optional tile_ready / tile_done / last_cta hooks as in tc_gemm.cuh.
#pragma once

#include "tc_gemm.cuh"

namespace beam {

constexpr int kWtConvWarps = 16;
constexpr int kWtThreads = 256 + 32 * kWtConvWarps;
constexpr int kWtTilesPerStep = 4;  // A tiles (128 rows x 64 k) per step = converter groups

template <class P>
__host__ __device__ constexpr int wt_b_slot_bytes() {
  return P::KS * P::BN * kTileK * 2;  // KS tiles of BN rows x 128 bytes
}

// Dynamic shared memory of a CTA: the two rings, barriers and schedule, and
// at least half the SM's shared memory, so that no two CTAs (each holding all
// 512 tensor-memory columns) ever share an SM, nor a down CTA started early by
// the programmatic dependent launch an SM still running gate/up.
template <class P>
__host__ __device__ constexpr int wt_smem_bytes() {
  constexpr int need = 1024 + P::BS * wt_b_slot_bytes<P>() + P::RS * P::RAW_BYTES + 1024 +
                       (int)sizeof(typename P::Sched);
  constexpr int half = kSmemLimit / 2 + 1024;
  return need > half ? need : half;
}

template <class P>
__global__ void __launch_bounds__(kWtThreads, 1)
    wt_gemm_kernel(const __grid_constant__ typename P::Params p) {
  constexpr int NA = P::NA, BN = P::BN, KS = P::KS, RS = P::RS, AST = P::AST, BS = P::BS;
  constexpr int BSLOT = wt_b_slot_bytes<P>();
  constexpr uint32_t kAccCols = NA * BN;
  constexpr uint32_t kACol0 = P::NBUF * kAccCols;
  constexpr uint32_t kStageCols = kWtTilesPerStep * 32;
  constexpr uint32_t kTmemCols = 512;
  constexpr uint32_t kIdesc = umma_idesc_f16(kTileM, BN);
  constexpr bool DYN = P::DYNAMIC;
  static_assert(KS * NA == kWtTilesPerStep, "a step holds four A tiles");
  static_assert(kACol0 + AST * kStageCols <= kTmemCols, "tensor memory overflow");
  static_assert(BSLOT % 1024 == 0 && P::RAW_BYTES % 128 == 0, "slot alignment");
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "invalid MMA N");
  static_assert(AST >= 2 && RS >= 2 && BS >= 2, "pipeline depth");
  constexpr uint32_t kConvWarpsPerStep = kWtConvWarps;  // every group takes part in every step

  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t *bslots = smem_raw + pad;
  uint8_t *raws = bslots + BS * BSLOT;
  uint8_t *bar_area = raws + RS * P::RAW_BYTES;
  uint64_t *raw_full = reinterpret_cast<uint64_t *>(bar_area);
  uint64_t *raw_empty = raw_full + RS;
  uint64_t *b_full = raw_empty + RS;
  uint64_t *b_empty = b_full + BS;   // B slot free (the MMA's commit)
  uint64_t *a_full = b_empty + BS;   // A stage written and its step's B tiles landed
  uint64_t *a_empty = a_full + AST;  // A stage free (the MMA's commit)
  uint64_t *tfull = a_empty + AST;
  uint64_t *tempty = tfull + P::NBUF;
  uint64_t *drain = tempty + P::NBUF;
  uint64_t *tr_full = drain + 1;
  uint64_t *tr_empty = tr_full + kTileRing;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tr_empty + kTileRing);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  volatile int *tring = abort_flag + 1;
  static_assert((2 * RS + 2 * BS + 2 * AST + 2 * P::NBUF + 1 + 2 * kTileRing) * 8 + 8 + 4 * kTileRing <= 1024,
                "barrier area");
  typename P::Sched *sched = reinterpret_cast<typename P::Sched *>(bar_area + 1024);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < RS; ++s) {
      mbar_init(&raw_full[s], 1);
      mbar_init(&raw_empty[s], kConvWarpsPerStep);
    }
    for (int s = 0; s < BS; ++s) {
      mbar_init(&b_full[s], 1);
      mbar_init(&b_empty[s], 1);
    }
    for (int s = 0; s < AST; ++s) {
      mbar_init(&a_full[s], kConvWarpsPerStep);
      mbar_init(&a_empty[s], 1);
    }
    for (int b = 0; b < P::NBUF; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4);
    }
    mbar_init(drain, 1);
    for (int s = 0; s < kTileRing; ++s) {
      mbar_init(&tr_full[s], 1);
      // the MMA thread, the activation producer, the epilogue and converter warps
      mbar_init(&tr_empty[s], 1 + 1 + 4 + kWtConvWarps);
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
  if constexpr (P::PDL_PRIMARY) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // Tile feed (as in tc_gemm.cuh): static cursor, or the weight producer's
  // dynamic picks handed to every other role through a ring in shared memory.
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

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- weight producer (weights are static: it streams ahead
      // without waiting for anything but free raw slots)
      int rs = 0, cur = blockIdx.x, tslot = 0;
      uint32_t ph = 0, issued = 0, par = 0, tph = 0;
      bool ok = true;
      for (int t = produce_tile(cur, tslot, tph, ok); ok && t >= 0;
           t = produce_tile(cur, tslot, tph, ok)) {
        const typename P::Tile tile = P::tile(p, *sched, t);
        const int ns = P::num_steps(p, tile);
        for (int s = 0; s < ns; ++s) {
          if (!mbar_wait(&raw_empty[rs], ph ^ 1u, abort_flag, p.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&raw_full[rs], P::RAW_BYTES);
          P::load_raw(p, tile, s, raws + rs * P::RAW_BYTES, &raw_full[rs]);
          issued |= 1u << rs;
          par = (par & ~(1u << rs)) | (ph << rs);
          if (++rs == RS) {
            rs = 0;
            ph ^= 1u;
          }
        }
      }
      if (!ok) {  // let every copy still in flight land before the CTA exits
        for (int s = 0; s < RS; ++s)
          if (issued & (1u << s)) mbar_drain_wait(&raw_full[s], (par >> s) & 1u);
      }
    }
  } else if (warp == 3) {
    if (lane == 0) {
      // ---------------- activation producer (a down tile's h rows are read only
      // once tile_ready says they have been published; with PDL_WAIT_B the
      // activations are the previous launch's output: this thread alone waits
      // for it to complete, while the weights already stream and convert)
      if constexpr (P::PDL_WAIT_B) asm volatile("griddepcontrol.wait;" ::: "memory");
      int bs = 0, cur = blockIdx.x, tslot = 0;
      uint32_t ph = 0, issued = 0, par = 0, tph = 0;
      bool ok = true;
      for (int t = consume_tile(cur, tslot, tph, ok, false); ok && t >= 0;
           t = consume_tile(cur, tslot, tph, ok, false)) {
        const typename P::Tile tile = P::tile(p, *sched, t);
        if constexpr (HasTileReady<P>::value) {
          if (!P::tile_ready(p, tile, abort_flag)) {
            ok = false;
            break;
          }
        }
        const int ns = P::num_steps(p, tile);
        const uint32_t tx = P::b_tx_bytes(p, tile);
        for (int s = 0; s < ns; ++s) {
          if (!mbar_wait(&b_empty[bs], ph ^ 1u, abort_flag, p.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&b_full[bs], tx);
          P::load_b(p, tile, s, bslots + bs * BSLOT, &b_full[bs]);
          issued |= 1u << bs;
          par = (par & ~(1u << bs)) | (ph << bs);
          if (++bs == BS) {
            bs = 0;
            ph ^= 1u;
          }
        }
      }
      if (!ok) {
        for (int s = 0; s < BS; ++s)
          if (issued & (1u << s)) mbar_drain_wait(&b_full[s], (par >> s) & 1u);
      }
    }
  } else if (warp == 1) {
    {
      // ---------------- MMA issuer: the whole warp runs the loop converged,
      // so descriptors and addresses stay warp-uniform; one elected lane
      // issues.  One wait (a_full covers the B tiles too) and one commit per step.
      int as = 0, bs = 0, buf = 0, cur = blockIdx.x, tslot = 0;
      uint32_t aph = 0, bph = 0, tph = 0;
      bool ok = true, any = false;
      const uint32_t b0 = smem_u32(bslots);
      const bool leader = elect_one();
      for (int t = consume_tile(cur, tslot, tph, ok, true); ok && t >= 0;
           t = consume_tile(cur, tslot, tph, ok, true)) {
        const typename P::Tile tile = P::tile(p, *sched, t);
        const int ns = P::num_steps(p, tile);
        ok = __all_sync(0xffffffffu, mbar_wait(&tempty[buf], bph ^ 1u, abort_flag, p.status));
        if (!ok) break;
        tc_fence_after();
        const uint32_t d0 = tmem_base + buf * kAccCols;
        // The commit that frees stage s is issued halfway through step s + 1's
        // MMAs, not right after step s: a barrier wait that follows a commit
        // at once stalls until the tensor core has drained, and it would then
        // sit idle while the next step is waited for and issued.
        int prev = -1, prevb = -1;  // stage and B slot whose commit is still due
        for (int s = 0; s < ns; ++s) {
          ok = __all_sync(0xffffffffu, mbar_wait(&a_full[as], aph, abort_flag, p.status));
          if (!ok) break;
          tc_fence_after();
          const uint32_t bst = b0 + bs * BSLOT;
          const uint32_t acol = tmem_base + kACol0 + as * kStageCols;
          if (leader) {
#pragma unroll
            for (int j = 0; j < KS; ++j) {
              if (j == KS / 2 && prev >= 0) {
                umma_commit(&a_empty[prev]);
                umma_commit(&b_empty[prevb]);
              }
              const uint64_t bdesc = umma_desc_sw128(bst + j * (BN * kTileK * 2));
#pragma unroll
              for (int kk = 0; kk < kTileK / 16; ++kk) {
#pragma unroll
                for (int a = 0; a < NA; ++a)
                  umma_f16_tmem_a(d0 + a * BN, acol + (j * NA + a) * 32 + 8 * kk, bdesc + 2 * kk,
                                   kIdesc, (s | j | kk) != 0 ? 1u : 0u);
              }
            }
          }
          __syncwarp();
          prev = as;
          prevb = bs;
          any = true;
          if (++as == AST) {
            as = 0;
            aph ^= 1u;
          }
          if (++bs == BS) bs = 0;
        }
        if (leader && prev >= 0) {
          umma_commit(&a_empty[prev]);
          umma_commit(&b_empty[prevb]);
        }
        __syncwarp();
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
  } else if (warp >= 8) {
    // ---------------- converters: packed weights -> f16 A stages in tensor memory
    const int g = (warp - 8) >> 2;  // warpgroup = A tile of the step
    const int q = warp & 3;         // tensor-memory lane quarter
    const int row = q * 32 + lane;
    const int j = g / NA, a = g % NA;  // slice of the step, matrix
    const uint32_t tq = tmem_base + ((uint32_t)(q * 32) << 16) + kACol0 + g * 32;
    int rs = 0, as = 0, bs = 0, cur = blockIdx.x, tslot = 0;
    uint32_t rph = 0, aph = 0, bph2 = 0, tph = 0;
    bool ok = true;
    for (int t = consume_tile(cur, tslot, tph, ok, true); ok && t >= 0;
         t = consume_tile(cur, tslot, tph, ok, true)) {
      const typename P::Tile tile = P::tile(p, *sched, t);
      const int ns = P::num_steps(p, tile);
      for (int s = 0; s < ns; ++s) {
        bool got = mbar_wait(&raw_full[rs], rph, abort_flag, p.status) &&
                   mbar_wait(&a_empty[as], aph ^ 1u, abort_flag, p.status);
        got = __all_sync(0xffffffffu, got);
        if (!got) {
          ok = false;
          break;
        }
        tc_fence_after();
        // the row's packed bytes into registers, then two halves of 32 k, the
        // first half's store running while the second half converts.  The
        // ring slot goes back to the producer only once the converted values
        // exist: an mbarrier arrival does not wait for the thread's
        // shared-memory loads still in flight (releasing the slot right after
        // the loads let the next TMA copy overwrite bytes not yet read)
        typename P::Row w;
        P::load_row(p, tile, s, raws + rs * P::RAW_BYTES, j, a, row, w);
        uint32_t v[16];
        P::convert_half(w, 0, v);
        tmem_st16(tq + as * kStageCols, v);
        P::convert_half(w, 1, v);
        tmem_st16(tq + as * kStageCols + 16, v);
        __syncwarp();
        if (lane == 0) mbar_arrive(&raw_empty[rs]);
        tmem_wait_st();
        // the stage is complete for the MMA once its B tiles have landed too:
        // one warp checks (the stage completes only with every warp's arrival,
        // so the MMA thread's wait on it covers the B tiles)
        if (warp == 8) {
          got = mbar_wait(&b_full[bs], bph2, abort_flag, p.status);
          got = __all_sync(0xffffffffu, got);
          if (!got) {
            ok = false;
            break;
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_full[as]);
        if (++rs == RS) {
          rs = 0;
          rph ^= 1u;
        }
        if (++as == AST) {
          as = 0;
          aph ^= 1u;
        }
        if (++bs == BS) {
          bs = 0;
          bph2 ^= 1u;
        }
      }
    }
  } else if (warp >= 4) {
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
  if constexpr (P::PDL_SECONDARY) asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace beam
