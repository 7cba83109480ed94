// gemm_pair.cu -- block-scaled MXFP8 GEMM on block pairs (tcgen05 cta_group::2).
//
// "Low-Precision GPU Programming", section "Scale ownership and the GEMM
// dataflow": Y = sum over 32-element K blocks b of S_A[i,b] S_B[j,b] times
// the block's dot product, each block's scale product kept inside the outer
// sum and applied by the tensor core (kind::mxf8f6f4.block_scale, E8M0
// scales from tensor memory), FP32 accumulation in tensor memory, FP32 or
// BF16 epilogue.  Every MMA spans the tensor cores of the two blocks of a
// cluster: M = 256 per instruction, block r holding
// rows 128r..128r+127 of A and of the accumulator, and half of the B tile
// (N rows 128r..128r+127) in its shared memory.  Per block and stage that is
// 32 KB of operands instead of 48 KB, so six stages fit (five next to the
// group table of the grouped modes), and one warp of block 0 issues the
// MMAs of both SMs.
//
//   warp 0 (both blocks)  TMA producer: A, B half, A scales, B scales into
//                         this block's ring; every copy completes on block
//                         0's `full` barrier (cta_group::2 tensor copies).
//   warp 1                both blocks allocate tensor memory together; in
//                         block 0 the warp copies scales to tensor memory and
//                         issues the pair MMAs (one elected lane), then
//                         multicasts the stage release to both blocks'
//                         `empty` barriers.
//   warps 2..9 (both)     epilogue on the block's own 128 accumulator rows,
//                         releasing the accumulator to block 0's barrier.
//                         With the fused epilogue: warps 4..11, warps 2 and
//                         3 idle (they complete the first warpgroup, whose
//                         registers go to the epilogue warpgroups).
// The work decomposition (tiles.cuh) has three modes: dense, grouped by rows of A
// (mixture-of-experts forward and data gradient) and grouped along K (the
// per-expert weight gradient).  All waits are bounded; a final cluster
// barrier keeps either block alive until its partner no longer touches its
// memory.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "epilogue.cuh"
#include "groups.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "status.cuh"
#include "tiles.cuh"

namespace mx {
namespace {

constexpr int kRowsPerBlock = 128;   // accumulator rows per block (256 per pair)
constexpr int kPairN = 256;          // columns of a pair tile
constexpr int kBK = kTileK;          // K per stage = four scale blocks
constexpr int kPEpiWarps = 8;
// Warp layout.  Plain epilogue: warp 0 producer, warp 1 MMA, warps 2-9
// epilogue, ten warps.  Either way a block has three warps on some of the
// SM's four sub-partition register files (16384 registers each), so a
// thread gets at most 168 at launch, which the plain kernels need and the
// fused epilogue (128 FP32 accumulator values plus bias and activation)
// exceeds.  Fused epilogue: twelve warps; the first warpgroup (producer,
// MMA, two idle warps) gives registers up and the two epilogue warpgroups
// take them, within the block's launch allocation.  (The grouped modes
// measured slower in the twelve-warp form, so it is kept to the fused,
// dense kernel.)
template <bool FUSED>
struct PairWarps {
  static constexpr int kFirstEpi = FUSED ? 4 : 2;
  static constexpr int kThreads = (kFirstEpi + kPEpiWarps) * 32;
};
constexpr int kPLaunchRegs = 168;
constexpr int kPLowRegs = 88;
constexpr int kPHighRegs = 208;
static_assert(kPLaunchRegs * 3 * 32 <= 16384, "launch registers per sub-partition");
static_assert(4 * 32 * kPLowRegs + kPEpiWarps * 32 * kPHighRegs <=
                  PairWarps<true>::kThreads * kPLaunchRegs,
              "register reallocation within the launch allocation");
constexpr uint32_t kPTmemCols = 512;
constexpr uint16_t kBoth = 0x3;
constexpr uint16_t kLeaderOnly = 0x1;
static_assert(kRowsPerBlock == kTileM, "tile rows");

template <bool GROUPED>
struct PairCfg {
  static constexpr int kStages = GROUPED ? 5 : 6;
  static constexpr int kABytes = kRowsPerBlock * kBK;    // 16 KB
  static constexpr int kBBytes = (kPairN / 2) * kBK;     // 16 KB, this block's half of B
  static constexpr int kSfaBytes = 512;                  // this block's 128 rows x 4 blocks
  static constexpr int kSfbBytes = 1024;                 // all 256 columns x 4 blocks
  // bytes one stage's four tensor copies of both blocks deliver, with the A
  // and B codes stored in a_bits / b_bits per element (8, or 4 / 6 packed:
  // an unpacking copy counts the bytes it reads, not the padded container
  // bytes it writes to shared memory)
  static __device__ __forceinline__ uint32_t pair_tx(int32_t a_bits, int32_t b_bits) {
    return 2u * (static_cast<uint32_t>(kABytes * a_bits / 8) +
                 static_cast<uint32_t>(kBBytes * b_bits / 8) + kSfaBytes + kSfbBytes);
  }
  static constexpr int kSfSlotCols = 4 + 8;
  static constexpr int kSfBaseCol = kPairN;              // after the accumulator
  static_assert(kSfBaseCol + kStages * kSfSlotCols <= int(kPTmemCols), "tensor memory budget");
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + kStages * kABytes;
  static constexpr int kOffSfa = kOffB + kStages * kBBytes;
  static constexpr int kOffSfb = kOffSfa + kStages * kSfaBytes;
  static constexpr int kOffEpi = kOffSfb + kStages * kSfbBytes;
  static constexpr int kOffBar = kOffEpi + kPEpiWarps * 2048;
  static constexpr int kNumBars = 2 * kStages + 3;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kOffGroup = kOffMisc + 64;
  static constexpr int kSmemBytes =
      kOffGroup + (GROUPED ? int(sizeof(GroupSmem)) : 0) + 1024;  // + alignment slack
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

template <int MODE, bool FUSED>
__global__ void __launch_bounds__(PairWarps<FUSED>::kThreads, 1)
    mx_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmap_a,
                        const __grid_constant__ CUtensorMap tmap_b,
                        const __grid_constant__ CUtensorMap tmap_sa,
                        const __grid_constant__ CUtensorMap tmap_sb, const GemmParams p) {
  constexpr bool GROUPED = MODE != kModeDense;
  using C = PairCfg<GROUPED>;
  constexpr int kPStages = C::kStages;
  constexpr int kFirstEpi = PairWarps<FUSED>::kFirstEpi;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem + C::kOffA;
  uint8_t* sB = smem + C::kOffB;
  uint8_t* sSfa = smem + C::kOffSfa;
  uint8_t* sSfb = smem + C::kOffSfb;
  uint8_t* sEpi = smem + C::kOffEpi;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* empty = full + kPStages;
  uint64_t* acc_full = empty + kPStages;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* mma_done = acc_empty + 1;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile uint32_t* s_abort = reinterpret_cast<volatile uint32_t*>(smem + C::kOffMisc + 4);
  GroupSmem* gs = reinterpret_cast<GroupSmem*>(smem + C::kOffGroup);

  const uint32_t warp = warp_id();
  const uint32_t lane = lane_id();
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int64_t cluster_id = blockIdx.x / 2;
  const int64_t num_clusters = gridDim.x / 2;

  if (warp == 0) {
    if (lane == 0) {
      for (int s = 0; s < kPStages; ++s) {
        mbar_init(&full[s], 1);   // block 0's: its producer's arrive + both blocks' bytes
        mbar_init(&empty[s], 1);  // one multicast commit per use
      }
      mbar_init(acc_full, 1);
      mbar_init(acc_empty, 2 * kPEpiWarps);  // one arrival per epilogue warp of the pair
      mbar_init(mma_done, 1);
      *s_abort = 0u;
      fence_mbarrier_init();
      tma_prefetch_desc(&tmap_a);
      tma_prefetch_desc(&tmap_b);
      tma_prefetch_desc(&tmap_sa);
      tma_prefetch_desc(&tmap_sb);
    }
    __syncwarp();
    if constexpr (GROUPED) {
      pdl_wait();  // the offsets may be written by the previous kernel
      // grouped along K the offsets split the p.k tokens of the contraction
      group_tile_prefix(p.offsets, p.groups, MODE == kModeGroupK ? p.k : p.m, gs->off, gs->tiles,
                        &gs->valid, 2, gs->units);
    }
  }
  if (warp == 1) {
    tmem_alloc_pair(s_tmem, kPTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before_sync();
  cluster_sync();  // barriers and group tables of both blocks exist before any cross-block use
  tc_fence_after_sync();
  const uint32_t tmem_base = *s_tmem;
  pdl_wait();  // operands and output may belong to the previous kernel of the stream
  pdl_launch_dependents();

  const int64_t n_tiles = (p.n + kPairN - 1) / kPairN;
  const int64_t m_units = (p.m + 2 * kRowsPerBlock - 1) / (2 * kRowsPerBlock);
  int64_t num_units;
  if constexpr (GROUPED) {
    // grouped along K, the 128-padded token segments must fit in A and B
    const bool fits = MODE != kModeGroupK ||
                      (gs->valid && static_cast<int64_t>(gs->tiles[p.groups]) * kBK <= p.lda &&
                       static_cast<int64_t>(gs->tiles[p.groups]) * kBK <= p.ldb);
    if (!gs->valid || !fits) {
      if (blockIdx.x == 0 && threadIdx.x == 0) record_device_status(p.status, MX_DEV_BAD_OFFSETS);
      num_units = 0;
    } else if constexpr (MODE == kModeGroupK) {
      num_units = static_cast<int64_t>(p.groups) * m_units * n_tiles;
    } else {
      num_units = static_cast<int64_t>(gs->units[p.groups]) * n_tiles;
    }
  } else {
    num_units = m_units * n_tiles;
  }

  // Each role's code sits under its own register reallocation, so the
  // compiler allocates it within that role's share.
  if constexpr (FUSED) {
    if (warp < kFirstEpi) setmaxnreg_dec<kPLowRegs>();
  }
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Whole warp; one elected lane issues (warp-uniform operands).  Every
    // block always issues all four copies with full boxes (padding rows and
    // out-of-range scale tiles are zero-filled or never stored), so block
    // 0's expected byte count is the same for every stage.
    const uint32_t full_leader0 = cluster_map(&full[0], 0);
    const uint32_t stage_tx = C::pair_tx(p.a_bits, p.b_bits);
    uint32_t stage = 0, phase = 0;
    int64_t issued = 0;
    bool ok = true;
    for (int64_t u = cluster_id; u < num_units && ok; u += num_clusters) {
      const TileInfo ti = tile_info<kPairN, MODE, 2>(p, u, n_tiles, rank, gs);
      const int32_t a_row = static_cast<int32_t>(ti.m0);
      const int32_t b_row = static_cast<int32_t>(ti.b_row0 + rank * (kPairN / 2));
      const int32_t kt_count = (ti.k_blocks + 3) / 4;
      for (int32_t kt = 0; kt < kt_count; ++kt) {
        if (!mbar_wait_warp(&empty[stage], phase ^ 1u, s_abort, p.status, p.wait_limit_ns)) {
          ok = false;
          break;
        }
        if (elect_one()) {
          if (leader) mbar_arrive_expect_tx(&full[stage], stage_tx);
          const uint32_t bar = full_leader0 + stage * 8u;
          tma_load_2d_pair(sA + stage * C::kABytes, &tmap_a, bar,
                           static_cast<int32_t>(ti.a_kx0) + kt * kBK, a_row);
          tma_load_2d_pair(sB + stage * C::kBBytes, &tmap_b, bar,
                           static_cast<int32_t>(ti.b_kx0) + kt * kBK, b_row);
          tma_load_3d_pair(sSfa + stage * C::kSfaBytes, &tmap_sa, bar, 0, ti.sfa_kt0 + kt,
                           ti.sfa_rt);
          tma_load_3d_pair(sSfb + stage * C::kSfbBytes, &tmap_sb, bar, 0, ti.sfb_kt0 + kt,
                           ti.sfb_rt);
        }
        __syncwarp();
        ++issued;
        if (++stage == kPStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    // Drain: wait until block 0 has consumed every fill of this block's
    // ring, so no copy into it and no commit arrival on it is still pending.
    for (int s = 0; s < kPStages; ++s) {
      const int64_t fills = issued > s ? (issued - s + kPStages - 1) / kPStages : 0;
      if (fills)
        mbar_wait_warp(&empty[s], static_cast<uint32_t>((fills - 1) & 1), s_abort, p.status,
                       p.wait_limit_ns, true);
    }
  } else if (warp == 1 && leader) {
    // ------------------------------------------------------------ MMA issuer (block 0)
    // Whole warp computes the operands; one elected lane issues.
    constexpr uint32_t kHiOperand = smem_desc_hi(1024, 2);
    constexpr uint32_t kHiScale = smem_desc_hi(128, 0);
    const uint32_t a_lo0 = smem_desc_lo(smem_u32(sA), 16);
    const uint32_t b_lo0 = smem_desc_lo(smem_u32(sB), 16);
    const uint32_t sfa_lo0 = smem_desc_lo(smem_u32(sSfa), 0);
    const uint32_t sfb_lo0 = smem_desc_lo(smem_u32(sSfb), 0);
    const uint32_t idesc0 = mxf8_idesc(p.fa, p.fb, 2 * kRowsPerBlock, kPairN, 0, 0);
    const uint32_t acc_full_peer = cluster_map(acc_full, 1);
    // Grouped along K every group has its own contraction length; a group
    // without tokens has none (its output tile is written as zeros).
    const uint32_t group_units = static_cast<uint32_t>(m_units * n_tiles);
    int32_t k_blocks = static_cast<int32_t>((p.k + 31) / 32);
    uint32_t stage = 0, phase = 0, acc_phase = 0;
    bool ok = true;
    for (int64_t u = cluster_id; u < num_units && ok; u += num_clusters) {
      if constexpr (MODE == kModeGroupK) {
        const int g = static_cast<int>(static_cast<uint32_t>(u) / group_units);
        k_blocks = (gs->off[g + 1] - gs->off[g] + 31) / 32;
      }
      const int32_t kt_count = (k_blocks + 3) / 4;
      const int32_t kt_full = k_blocks / 4;
      if (!mbar_wait_warp(acc_empty, acc_phase ^ 1u, s_abort, p.status, p.wait_limit_ns)) break;
      tc_fence_after_sync();
      for (int32_t kt = 0; kt < kt_count; ++kt) {
        if (!mbar_wait_warp(&full[stage], phase, s_abort, p.status, p.wait_limit_ns)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t sf_tmem = tmem_base + C::kSfBaseCol + stage * C::kSfSlotCols;
        const uint32_t sfa_lo = sfa_lo0 + stage * (C::kSfaBytes >> 4);
        const uint32_t sfb_lo = sfb_lo0 + stage * (C::kSfbBytes >> 4);
        const uint32_t a_lo = a_lo0 + stage * (C::kABytes >> 4);
        const uint32_t b_lo = b_lo0 + stage * (C::kBBytes >> 4);
        const uint32_t kb_here =
            kt < kt_full ? 4u : static_cast<uint32_t>(k_blocks - kt * 4);
        if (elect_one()) {
          tc_cp_pair_32x128b_warpx4(sf_tmem, sfa_lo, kHiScale);
          tc_cp_pair_32x128b_warpx4(sf_tmem + 4, sfb_lo, kHiScale);
          tc_cp_pair_32x128b_warpx4(sf_tmem + 8, sfb_lo + (512 >> 4), kHiScale);
#pragma unroll
          for (uint32_t kb = 0; kb < 4; ++kb) {
            if (kb < kb_here)
              tc_mma_pair_mxf8(tmem_base, a_lo + 2u * kb, kHiOperand, b_lo + 2u * kb, kHiOperand,
                               idesc0 | (kb << 4) | (kb << 29), sf_tmem, sf_tmem + 4,
                               (kt > 0 || kb > 0) ? 1u : 0u);
          }
          tc_commit_pair_multicast(&empty[stage], kBoth);
        }
        __syncwarp();
        if (++stage == kPStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      if (elect_one()) {
        if (kt_count > 0) {
          tc_commit_pair_multicast(acc_full, kBoth);
        } else {
          // nothing to accumulate: both epilogues write zeros
          mbar_arrive(acc_full);
          mbar_arrive_cluster(acc_full_peer);
        }
      }
      __syncwarp();
      acc_phase ^= 1u;
    }
    // Every MMA (they also write block 1's tensor memory) completes before
    // either block releases tensor memory.
    if (elect_one()) {
      tc_commit_pair_multicast(mma_done, kLeaderOnly);
      mbar_wait(mma_done, 0, s_abort, p.status, p.wait_limit_ns, true);
    }
    __syncwarp();
  } else if (warp >= kFirstEpi) {
    // ------------------------------------------------------------ epilogue (both blocks)
    if constexpr (FUSED) setmaxnreg_inc<kPHighRegs>();
    const uint32_t q = warp & 3u;
    const uint32_t half = (warp - kFirstEpi) >> 2;
    uint8_t* stage_buf = sEpi + (warp - kFirstEpi) * 2048;
    const uint32_t acc_empty_leader = cluster_map(acc_empty, 0);
    uint32_t acc_phase = 0;
    for (int64_t u = cluster_id; u < num_units; u += num_clusters) {
      const TileInfo ti = tile_info<kPairN, MODE, 2>(p, u, n_tiles, rank, gs);
      const bool got = mbar_wait(acc_full, acc_phase, s_abort, p.status, p.wait_limit_ns);
      if (!__all_sync(0xffffffffu, got)) break;
      tc_fence_after_sync();
      const uint32_t t_row = tmem_base + ((q * 32u) << 16) + half * (kPairN / 2);
      epilogue_share<kPairN, FUSED>(p, t_row, ti.y_row0 + q * 32, ti.n0 + half * (kPairN / 2),
                                    ti.m_end, stage_buf, lane, ti.k_blocks == 0, [&] {
                                      tc_fence_before_sync();
                                      __syncwarp();
                                      if (lane == 0) mbar_arrive_relaxed_cluster(acc_empty_leader);
                                    });
      acc_phase ^= 1u;
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  cluster_sync();  // the partner no longer touches this block's memory
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, kPTmemCols);
  }
}

template <int MODE, bool FUSED>
cudaError_t launch_pair_impl(const GemmParams& p, const CUtensorMap& ta, const CUtensorMap& tb,
                             const CUtensorMap& tsa, const CUtensorMap& tsb, int num_sms,
                             cudaStream_t stream) {
  using C = PairCfg<MODE != kModeDense>;
  auto kern = mx_gemm_pair_kernel<MODE, FUSED>;
  static PerDeviceOnce setup;
  cudaError_t err = setup.run([&]() -> cudaError_t {
    // The register increase in the kernel waits for registers the first
    // warpgroup returns; it only completes if the block is launched with
    // the allocation the shares were computed for.
    if (FUSED) {
      cudaFuncAttributes fa;
      const cudaError_t e = cudaFuncGetAttributes(&fa, kern);
      if (e != cudaSuccess) return e;
      if (fa.numRegs != kPLaunchRegs) return cudaErrorInvalidConfiguration;
    }
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  });
  if (err != cudaSuccess) return err;
  const int64_t n_tiles = (p.n + kPairN - 1) / kPairN;
  const int64_t m_tiles = (p.m + kRowsPerBlock - 1) / kRowsPerBlock;
  // upper bound of the pair units (grouped by rows: every group may add a
  // partial unit; grouped along K: every group covers the whole output)
  int64_t units = ((m_tiles + 1) / 2) * n_tiles;
  if (MODE == kModeGroupM) units = ((m_tiles + p.groups + 1) / 2 + p.groups) * n_tiles;
  if (MODE == kModeGroupK) units *= p.groups;
  if (units == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1] = pdl_attribute();
  cfg.blockDim = dim3(PairWarps<FUSED>::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;  // the occupancy query below sees the cluster shape only
  int max_clusters = num_sms / 2;
  cfg.gridDim = dim3(static_cast<unsigned>(max_clusters * 2));
  int active = 0;
  if (cudaOccupancyMaxActiveClusters(&active, kern, &cfg) == cudaSuccess && active > 0)
    max_clusters = ::min(max_clusters, active);
  const int64_t clusters = units < max_clusters ? units : max_clusters;
  cfg.gridDim = dim3(static_cast<unsigned>(clusters * 2));
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, ta, tb, tsa, tsb, p);
}

}  // namespace

cudaError_t launch_gemm_pair(const GemmParams& p, const CUtensorMap& tmap_a,
                             const CUtensorMap& tmap_b, const CUtensorMap& tmap_sa,
                             const CUtensorMap& tmap_sb, int num_sms, cudaStream_t stream) {
  if (p.bias != nullptr || p.act != 0) {  // fused epilogue: dense GEMMs only
    if (p.mode != kModeDense) return cudaErrorNotSupported;
    return launch_pair_impl<kModeDense, true>(p, tmap_a, tmap_b, tmap_sa, tmap_sb, num_sms,
                                              stream);
  }
  if (p.mode == kModeGroupM)
    return launch_pair_impl<kModeGroupM, false>(p, tmap_a, tmap_b, tmap_sa, tmap_sb, num_sms,
                                                stream);
  if (p.mode == kModeGroupK)
    return launch_pair_impl<kModeGroupK, false>(p, tmap_a, tmap_b, tmap_sa, tmap_sb, num_sms,
                                                stream);
  return launch_pair_impl<kModeDense, false>(p, tmap_a, tmap_b, tmap_sa, tmap_sb, num_sms, stream);
}

}  // namespace mx
