// Two-CTA (cta_group::2) variant of the warp-specialised tcgen05 GEMM.
//
// A cluster of two CTAs on neighbouring SMs computes one 256 x BN tile:
// CTA r of the pair holds rows 128r..128r+127 of A and half of B's BN rows in
// its own shared memory, and its own 128 rows of the fp32 accumulator in its
// own tensor memory.  The even CTA (the leader) issues every
// tcgen05.mma.cta_group::2 (M=256); the tensor cores read the A and B halves
// of both CTAs.  Per CTA a stage is 16 KB of A plus BN/2 rows of B, a third
// less than the one-CTA kernel for the same work, so more stages fit and less
// data crosses from L2 per FLOP.
//   warp 0 lane 0 (both CTAs): TMA loads of the CTA's halves; completion is
//                              signalled on the leader's full barrier
//   warp 1 lane 0 (leader)    : MMA issuer; commits are multicast to both CTAs
//   warp 2 (both)             : collective tensor-memory allocation / release
//   warps 4..7 (both)         : epilogue of the CTA's 128 rows; they release the
//                              accumulator on the leader's barrier
// Every wait is bounded as in tc_gemm.cuh.
//
// A problem class P supplies BN (total N), STAGES, NBUF, Params (with status),
// Sched, Tile, prologue, num_tiles (pair tiles), tile, num_k,
//   load(p, tile, k, uint8_t *stage, uint32_t leader_full_bar, int rank)
//   epilogue(p, tile, taddr, row, rank)
#pragma once

#include "tc_gemm.cuh"

namespace beam {

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// shared::cluster address of the variable at shared::cta address `addr` in CTA `rank`
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t d;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(addr), "r"(rank));
  return d;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::
          : "memory");
}

// TMA load into this CTA's shared memory, completion signalled on the mbarrier
// at shared::cluster address `bar` (the leader CTA's).
__device__ __forceinline__ void tma_load_2d_cg2(void *dst, const CUtensorMap *map, uint32_t bar,
                                                int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

__device__ __forceinline__ void umma_bf16_cg2(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives once on the mbarrier at the same offset in every CTA of `mask` when
// the pair's MMAs issued so far have completed.
__device__ __forceinline__ void umma_commit_cg2(uint64_t *bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_u32(bar)),
      "h"(mask)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

__device__ __forceinline__ void tmem_alloc_cg2(uint32_t *dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish_cg2() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_cg2(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

template <class P>
__host__ __device__ constexpr int stage_bytes_cg2() {
  return kATileBytes + (P::BN / 2) * kTileK * 2;
}

template <class P>
__host__ __device__ constexpr int smem_bytes_cg2() {
  return kSmemReserve + P::STAGES * stage_bytes_cg2<P>() + (int)sizeof(typename P::Sched);
}

template <class P>
__global__ void __launch_bounds__(256, 1)
    tc_gemm2_kernel(const __grid_constant__ typename P::Params p) {
  constexpr int STAGE = stage_bytes_cg2<P>();
  constexpr uint32_t kAccCols = P::BN;
  constexpr uint32_t kTmemCols = tmem_cols_pow2(P::NBUF * kAccCols);
  constexpr uint32_t kIdesc = umma_idesc_bf16(2 * kTileM, P::BN);
  static_assert(P::NBUF * kAccCols <= 512, "accumulators exceed tensor memory");
  static_assert(P::BN % 32 == 0 && P::BN <= 256, "invalid MMA N for M=256");
  static_assert(STAGE % 1024 == 0, "stage must keep 1024-byte alignment");

  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t *stages = smem_raw + pad;
  uint64_t *full = reinterpret_cast<uint64_t *>(stages + P::STAGES * STAGE);
  uint64_t *empty = full + P::STAGES;
  uint64_t *tfull = empty + P::STAGES;
  uint64_t *tempty = tfull + P::NBUF;
  uint64_t *drain = tempty + P::NBUF;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  typename P::Sched *sched =
      reinterpret_cast<typename P::Sched *>(stages + P::STAGES * STAGE + 1024);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < P::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < P::NBUF; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 8);  // four epilogue warps in each CTA of the pair
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 2) {
    tmem_alloc_cg2(tmem_slot, kTmemCols);
    tmem_relinquish_cg2();
  }
  P::prologue(p, *sched);
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers exist before any remote arrive or multicast
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int ntiles = P::num_tiles(p, *sched);
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer (both CTAs)
      int stage = 0;
      uint32_t ph = 0, issued = 0, par = 0;
      bool ok = true;
      for (int t = pair; ok && t < ntiles; t += npairs) {
        const typename P::Tile tile = P::tile(p, *sched, t);
        const int nk = P::num_k(p, tile);
        for (int k = 0; k < nk; ++k) {
          if (!mbar_wait(&empty[stage], ph ^ 1u, abort_flag, p.status)) {
            ok = false;
            break;
          }
          if (leader) mbar_arrive_expect_tx(&full[stage], 2 * STAGE);  // both CTAs' halves
          P::load(p, tile, k, stages + stage * STAGE, mapa_shared(smem_u32(&full[stage]), 0), rank);
          issued |= 1u << stage;
          par = (par & ~(1u << stage)) | (ph << stage);
          if (++stage == P::STAGES) {
            stage = 0;
            ph ^= 1u;
          }
        }
      }
      if (!ok && leader) {  // the leader's full barriers count both CTAs' bytes
        for (int s = 0; s < P::STAGES; ++s)
          if (issued & (1u << s)) mbar_drain_wait(&full[s], (par >> s) & 1u);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------- MMA issuer (leader only)
      int stage = 0, buf = 0;
      uint32_t ph = 0, bph = 0;
      bool ok = true, any = false;
      for (int t = pair; ok && t < ntiles; t += npairs) {
        const typename P::Tile tile = P::tile(p, *sched, t);
        const int nk = P::num_k(p, tile);
        if (!mbar_wait(&tempty[buf], bph ^ 1u, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d0 = tmem_base + buf * kAccCols;
        for (int k = 0; k < nk; ++k) {
          if (!mbar_wait(&full[stage], ph, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(stages + stage * STAGE);
          const uint64_t adesc = umma_desc_sw128(sa);
          const uint64_t bdesc = umma_desc_sw128(sa + kATileBytes);
#pragma unroll
          for (int kk = 0; kk < kTileK / 16; ++kk)
            umma_bf16_cg2(d0, adesc + 2 * kk, bdesc + 2 * kk, kIdesc, (k | kk) != 0 ? 1u : 0u);
          umma_commit_cg2(&empty[stage], 0x3);
          any = true;
          if (++stage == P::STAGES) {
            stage = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_cg2(&tfull[buf], 0x3);
        if (++buf == P::NBUF) {
          buf = 0;
          bph ^= 1u;
        }
      }
      if (!ok && any) {
        umma_commit_cg2(drain, 0x1);
        mbar_drain_wait(drain, 0);
      }
    }
  } else if (warp >= 4) {
    // ---------------- epilogue (both CTAs, each its own 128 rows)
    const int q = warp & 3;
    const int row = q * 32 + lane;
    int buf = 0;
    uint32_t bph = 0;
    for (int t = pair; t < ntiles; t += npairs) {
      const typename P::Tile tile = P::tile(p, *sched, t);
      bool ok = mbar_wait(&tfull[buf], bph, abort_flag, p.status);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + buf * kAccCols;
      P::epilogue(p, tile, taddr, row, (int)rank);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[buf]), 0));
      if (++buf == P::NBUF) {
        buf = 0;
        bph ^= 1u;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // no MMA, copy or remote arrive of the pair is still in flight
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc_cg2(tmem_base, kTmemCols);
  }
}

}  // namespace beam
