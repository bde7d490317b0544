// The GEMM of tile_gemm.cuh on CTA pairs: tcgen05.mma.cta_group::2 with
// M = 256 (128 rows in each CTA of a 2-CTA cluster) and N = 256.
//
// Each CTA streams its own 128x64 A box and its half (128 of the 256
// columns) of the B tile into a 6-stage ring (7 for the forward's instance,
// which needs no store boxes); the pair's tensor cores share the two B
// halves, so every SM moves 32 KiB per 64-deep k-block instead of 48 KiB,
// and more stages fit in shared memory. The even CTA's producer
// expects the bytes of both CTAs on its full barrier, the odd CTA's TMA
// loads complete on that barrier, and the even CTA's single MMA thread
// issues the MMAs and releases both CTAs' stages and accumulators with
// multicast commits. Each CTA's epilogue warps read their own 128 TMEM lanes
// and report to the even CTA that the accumulator buffer may be reused.
//
// With gradient filtering the pair leaves out a k-block only when both CTAs'
// tiles skip it: the dW mask stays 128 rows x 256 vocabulary ids (both
// halves of a dW group read the same dZ tile), the dH mask becomes 256 rows
// x 256 ids (the two halves are two row tiles). A tile whose k-blocks are
// all left out takes no accumulator at all.
#pragma once

#include "tile_gemm.cuh"

namespace flce {

constexpr int kPairStages = 6;
constexpr int kPairStagesLse = 7;     // launches of EPI_LSE problems only: no store boxes
constexpr uint32_t kPairBBytes = (kBN / 2) * kBK * 2;           // 16 KiB: this CTA's half of B
constexpr uint32_t kPairStageBytes = kABytes + kPairBBytes;      // 32 KiB

// The epilogue's TMA store boxes take the room of one more stage; EPI_LSE
// stores nothing through shared memory, so the forward's instance uses that
// room for a seventh stage.
__host__ __device__ constexpr int pair_stages(int modes) { return modes == kModesForward ? kPairStagesLse : kPairStages; }
__host__ __device__ constexpr uint32_t pair_epi_bytes(int modes) { return modes == kModesForward ? 0u : kEpiBytes; }
__host__ __device__ constexpr uint32_t pair_smem_bytes(int modes) {
  return 1024 + pair_stages(modes) * kPairStageBytes + pair_epi_bytes(modes) + kBarrierBytes;
}
static_assert(pair_smem_bytes(kModesBackward) <= 232448 && pair_smem_bytes(kModesForward) <= 232448,
              "shared memory of the pair kernel");
static_assert((2 * kPairStagesLse + 5) * 8 + 8 <= kBarrierBytes, "barrier area of the pair kernel");

// The tiles one pair handles, in the order it handles them. A pair takes
// every stride-th tile from unit0. With groups > 1 the pairs are cut into
// that many runs of consecutive pairs, and run k starts its list k/groups of
// the way in: the problems of one launch then run side by side (the fused
// optimizer's memory-heavy epilogues overlap the other problems' MMAs),
// while neighbouring pairs still take neighbouring tiles and share operands
// in L2. Every role of the pair walks the same order.
struct TileOrder {
  int unit0, stride, count, rot;
  __device__ TileOrder(int unit0_, int stride_, int num_tiles, int groups)
      : unit0(unit0_), stride(stride_), count(0), rot(0) {
    count = unit0 < num_tiles ? (num_tiles - 1 - unit0) / stride + 1 : 0;
    if (groups > 1 && count > 0) rot = (int)((int64_t)count * ((int64_t)unit0 * groups / stride) / groups);
  }
  __device__ int tile(int j) const {
    int jj = j + rot;
    if (jj >= count) jj -= count;
    return unit0 + jj * stride;
  }
};

// kSkip: some problem of the launch leaves out filtered k-blocks. Launches
// without filtering use the kSkip = false instance, whose k-loops carry no
// skip test at all. kModes: the epilogue set (kModesForward,
// kModesBackward or kModesBackwardAdamw), which also fixes the ring depth.
template <bool kSkip, int kModes>
__global__ void __launch_bounds__(kGemmThreads, 1) flce_gemm_pair_kernel(const __grid_constant__ GemmLaunch L) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  constexpr int kStg = pair_stages(kModes);
  uint8_t* epi_smem = smem + kStg * kPairStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(epi_smem + pair_epi_bytes(kModes));
  uint64_t* full_bar = bars;                        // [kStg] (used in the even CTA)
  uint64_t* empty_bar = bars + kStg;         // [kStg]
  uint64_t* acc_full = bars + 2 * kStg;      // [2]
  uint64_t* acc_empty = bars + 2 * kStg + 2; // [2] (used in the even CTA)
  uint64_t* drain_bar = bars + 2 * kStg + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStg + 5);
  volatile uint32_t* abort_flag = tmem_slot + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_tiles = L.tile_end[L.n_probs - 1];
  const uint64_t wait_limit_ns = L.prob[0].wait_limit_ns;
  uint32_t* const status = L.prob[0].status;
  const int rank = (int)ptx::cluster_ctarank();
  const bool leader = rank == 0;
  const int unit0 = blockIdx.x / 2;
  const int unit_stride = gridDim.x / 2;
  constexpr uint16_t kBoth = 3;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStg; ++s) {
      ptx::mbar_init(&full_bar[s], 1);
      ptx::mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&acc_full[b], 1);
      ptx::mbar_init(&acc_empty[b], 8);           // 4 epilogue warps in each CTA
    }
    ptx::mbar_init(drain_bar, 1);
    *abort_flag = 0u;
    ptx::fence_mbarrier_init();
    for (int q = 0; q < L.n_probs; ++q) {
      ptx::prefetch_tmap(&L.tm_a[q]);
      ptx::prefetch_tmap(&L.tm_b[q]);
      ptx::prefetch_tmap(&L.tm_out[q]);
    }
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(tmem_slot, kTmemCols);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync_all();                          // both CTAs' barriers exist
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // The prologue above touches only shared memory, TMEM and the kernel
  // parameters, so it may overlap the end of the previous GEMM launch (which
  // may have written this launch's operands): every thread waits for that
  // launch before its first global-memory access. The next launch may start
  // its own prologue as soon as an SM frees up.
  ptx::wait_prior_grids();
  if (threadIdx.x == 0) ptx::launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ producer (both CTAs)
    if (lane == 0) {
      const uint32_t full_leader = ptx::map_to_rank(&full_bar[0], 0);
      const uint32_t smem_base = ptx::smem_u32(smem);
      uint32_t stage = 0, phase = 0, issued = 0;
      bool ok = true;
      const TileOrder ord(unit0, unit_stride, num_tiles, L.order_groups);
      for (int j = 0; j < ord.count && ok; ++j) {
        int pi, mt, nt;
        const int tl = decode_tile(L, ord.tile(j), pi);
        const GemmParams& p = L.prob[pi];
        tile_coords(p, tl, 2, rank, mt, nt);
        const bool may_skip = kSkip && p.skip_by_flags != 0;
        const uint64_t keep = may_skip ? tile_keep(p, mt - rank, 2) : ~0ull;
        // Everything the k-loop needs, read from the parameters once per tile
        // and pinned in registers: the single producer thread issues a TMA
        // copy every few hundred cycles, and re-reading parameters between
        // the copies measurably slowed the whole pipeline.
        const uint64_t tmA = ptx::pin(reinterpret_cast<uint64_t>(&L.tm_a[pi]));
        const uint64_t tmB = ptx::pin(reinterpret_cast<uint64_t>(&L.tm_b[pi]));
        const int32_t a_mn = ptx::pin(p.a_mn), b_mn = ptx::pin(p.b_mn);
        const int32_t a_m = ptx::pin(p.a_m0 + mt * kBM), a_k = ptx::pin(p.a_k0);
        const int32_t b_n = ptx::pin(p.b_n0 + nt * kBN + rank * (kBN / 2)), b_k = ptx::pin(p.b_k0);
        const int32_t k_blocks = ptx::pin(p.k_blocks);
        // k-block kb reads keep-mask unit kb >> unit_shift (a dH unit spans
        // 256 staging columns = 4 k-blocks, a dW unit 128 rows = 2): a shift,
        // since a division by a pinned value would be a software division
        // on every k-block.
        static_assert(kBN / kBK == 4 && kBM / kBK == 2, "keep-mask units of 4 and 2 k-blocks");
        const int32_t unit_shift = kSkip ? ptx::pin(p.flags_a_is_rows ? 2 : 1) : 0;
        for (int kb = 0; kb < k_blocks; ++kb) {
          if (kSkip && may_skip && ((keep >> (kb >> unit_shift)) & 1ull) == 0ull) continue;
          if (!ptx::mbar_wait_bounded(&empty_bar[stage], phase ^ 1u, wait_limit_ns, abort_flag)) {
            record_timeout(status, abort_flag);
            ok = false;
            break;
          }
          const uint32_t sa = smem_base + stage * kPairStageBytes;
          const uint32_t sb = sa + kABytes;
          const uint32_t fb = full_leader + stage * 8u;
          if (leader) ptx::mbar_arrive_expect_tx(&full_bar[stage], 2 * kPairStageBytes);
          const int32_t kc = kb * kBK;
          if (a_mn == kMnBox3d) {
            ptx::tma_load_3d_pair(sa, tmA, 0, a_k + kc, a_m >> 6, fb);
          } else if (a_mn) {
            ptx::tma_load_2d_pair(sa, tmA, a_m, a_k + kc, fb);
            ptx::tma_load_2d_pair(sa + 8192, tmA, a_m + 64, a_k + kc, fb);
          } else {
            ptx::tma_load_2d_pair(sa, tmA, a_k + kc, a_m, fb);
          }
          if (b_mn == kMnBox3d) {
            ptx::tma_load_3d_pair(sb, tmB, 0, b_k + kc, b_n >> 6, fb);
          } else if (b_mn) {
            ptx::tma_load_2d_pair(sb, tmB, b_n, b_k + kc, fb);
            ptx::tma_load_2d_pair(sb + 8192, tmB, b_n + 64, b_k + kc, fb);
          } else {
            ptx::tma_load_2d_pair(sb, tmB, b_k + kc, b_n, fb);
          }
          ++issued;
          if (++stage == kStg) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok && leader) {
        // The even CTA's full barriers count both CTAs' bytes: once a phase
        // completes, no copy of that phase is still landing in either CTA.
        // Stage s was last filled in the current phase if s < stage, in the
        // previous one otherwise (if `issued` ever reached it).
        volatile uint32_t never = 0u;
        for (uint32_t s = 0; s < (uint32_t)kStg; ++s)
          if (s < issued) ptx::mbar_wait_bounded(&full_bar[s], s < stage ? phase : (phase ^ 1u), 100000000ull, &never);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (lane == 0 && leader) {
      const uint32_t smem_base = ptx::smem_u32(smem);
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      const TileOrder ord(unit0, unit_stride, num_tiles, L.order_groups);
      int i = 0;                                      // accumulators used so far
      for (int j = 0; j < ord.count && ok; ++j) {
        int pi, mt, nt;
        const int tl = decode_tile(L, ord.tile(j), pi);
        const GemmParams& p = L.prob[pi];
        tile_coords(p, tl, 2, rank, mt, nt);
        const bool may_skip = kSkip && p.skip_by_flags != 0;
        const uint64_t keep = may_skip ? tile_keep(p, mt, 2) : ~0ull;   // mt: the even CTA's m-tile
        // A tile with every k-block filtered out needs no accumulator: the
        // epilogue writes it without reading TMEM, and both sides skip the
        // hand-off for it.
        if (kSkip && may_skip && keep == 0ull) continue;
        const uint32_t idesc = (uint32_t)ptx::pin((int32_t)ptx::idesc_bf16_f32(2 * kBM, kBN, p.a_mn != 0, p.b_mn != 0));
        const uint32_t buf = i & 1, use = i >> 1;
        ++i;
        if (!ptx::mbar_wait_bounded(&acc_empty[buf], (use & 1u) ^ 1u, wait_limit_ns, abort_flag)) {
          record_timeout(status, abort_flag);
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * kBN;
        uint32_t accumulate = 0;
        const bool a_mn = ptx::pin(p.a_mn) != 0, b_mn = ptx::pin(p.b_mn) != 0;
        const int k_blocks = ptx::pin(p.k_blocks);
        const int32_t unit_shift = kSkip ? ptx::pin(p.flags_a_is_rows ? 2 : 1) : 0;   // as in the producer
        for (int kb = 0; kb < k_blocks; ++kb) {
          if (kSkip && may_skip && ((keep >> (kb >> unit_shift)) & 1ull) == 0ull) continue;
          if (!ptx::mbar_wait_bounded(&full_bar[stage], phase, wait_limit_ns, abort_flag)) {
            record_timeout(status, abort_flag);
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t a_addr = smem_base + stage * kPairStageBytes;
          const uint32_t b_addr = a_addr + kABytes;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            const uint64_t adesc = a_mn ? ptx::smem_desc_sw128(a_addr + k * 2048, 8192, 1024)
                                        : ptx::smem_desc_sw128(a_addr + k * 32, 16, 1024);
            const uint64_t bdesc = b_mn ? ptx::smem_desc_sw128(b_addr + k * 2048, 8192, 1024)
                                        : ptx::smem_desc_sw128(b_addr + k * 32, 16, 1024);
            ptx::mma_bf16_ss_pair(d_tmem, adesc, bdesc, idesc, accumulate);
            accumulate = 1;
          }
          ptx::mma_commit_pair_multicast(&empty_bar[stage], kBoth);
          if (++stage == kStg) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        ptx::mma_commit_pair_multicast(&acc_full[buf], kBoth);
      }
      // Every MMA issued has completed once the drain barrier flips.
      ptx::mma_commit_pair_multicast(drain_bar, 1);
      volatile uint32_t never = 0u;
      ptx::mbar_wait_bounded(drain_bar, 0u, 100000000ull, &never);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;
    uint8_t* my_boxes = epi_smem + q * 2 * kEpiBoxBytes;
    uint32_t ebuf = 0;
    const TileOrder ord(unit0, unit_stride, num_tiles, L.order_groups);
    int i = 0;                                        // accumulators used so far
    for (int j = 0; j < ord.count; ++j) {
      int pi, mt, nt;
      const int tl = decode_tile(L, ord.tile(j), pi);
      const GemmParams& p = L.prob[pi];
      const CUtensorMap* tmOut = &L.tm_out[pi];
      tile_coords(p, tl, 2, rank, mt, nt);
      // A tile with no accumulator (see the MMA issuer) is written without
      // waiting for one and releases nothing.
      const bool no_acc = kSkip && p.skip_by_flags != 0 && tile_keep(p, mt - rank, 2) == 0ull;
      uint32_t buf = 0;
      if (!no_acc) {
        buf = i & 1;
        const uint32_t use = i >> 1;
        ++i;
        if (!ptx::mbar_wait_bounded(&acc_full[buf], use & 1u, wait_limit_ns, abort_flag)) {
          record_timeout(status, abort_flag);
          break;
        }
        ptx::tc_fence_after();
      }
      const uint32_t taddr = tmem_base + buf * kBN + ((uint32_t)(q * 32) << 16);
      const AccRelease rel{&acc_empty[buf], ptx::map_to_rank(&acc_empty[buf], 0), !leader, no_acc};
      epilogue_tile<kModes>(p, tmOut, mt, nt, taddr, q, lane, my_boxes, ebuf, rel, 2);
    }
    if (lane == 0) ptx::bulk_wait_group<0>();
    __syncwarp();
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync_all();                          // the pair is done with both CTAs' TMEM and smem
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc_pair(tmem_base, kTmemCols);
}

}  // namespace flce
