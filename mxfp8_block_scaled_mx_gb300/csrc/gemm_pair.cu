// gemm_pair.cu -- block-scaled MXFP8 GEMM on block pairs (tcgen05 cta_group::2).
//
// Same computation as gemm.cu ("Low-Precision GPU Programming", section
// "Scale ownership and the GEMM dataflow": each 32-element K block keeps its
// scale product inside the outer sum), but every MMA spans the tensor cores
// of the two blocks of a cluster: M = 256 per instruction, block r holding
// rows 128r..128r+127 of A and of the accumulator, and half of the B tile
// (N rows 128r..128r+127) in its shared memory.  Per block and stage that is
// 32 KB of operands instead of 48 KB, so six stages fit, and one thread in
// block 0 issues the MMAs of both SMs.
//
//   warp 0 (both blocks)  TMA producer: A, B half, A scales, B scales into
//                         this block's ring; every copy completes on block
//                         0's `full` barrier (cta_group::2 tensor copies).
//   warp 1                both blocks allocate tensor memory together; in
//                         block 0 one lane copies scales to tensor memory and
//                         issues the pair MMAs, then multicasts the stage
//                         release to both blocks' `empty` barriers.
//   warps 2..9 (both)     epilogue on the block's own 128 accumulator rows,
//                         releasing the accumulator to block 0's barrier.
// All waits are bounded; a final cluster barrier keeps either block alive
// until its partner no longer touches its memory.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "epilogue.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "status.cuh"

namespace mx {
namespace {

constexpr int kRowsPerBlock = 128;   // accumulator rows per block (256 per pair)
constexpr int kPairN = 256;          // columns of a pair tile
constexpr int kBK = 128;             // K per stage = four scale blocks
constexpr int kPStages = 6;
constexpr int kPEpiWarps = 8;
constexpr int kPThreads = 64 + kPEpiWarps * 32;
constexpr uint32_t kPTmemCols = 512;
constexpr uint16_t kBoth = 0x3;
constexpr uint16_t kLeaderOnly = 0x1;

struct PairCfg {
  static constexpr int kABytes = kRowsPerBlock * kBK;    // 16 KB
  static constexpr int kBBytes = (kPairN / 2) * kBK;     // 16 KB, this block's half of B
  static constexpr int kSfaBytes = 512;                  // this block's 128 rows x 4 blocks
  static constexpr int kSfbBytes = 1024;                 // all 256 columns x 4 blocks
  static constexpr uint32_t kPairTx = 2u * (kABytes + kBBytes + kSfaBytes + kSfbBytes);
  static constexpr int kSfSlotCols = 4 + 8;
  static constexpr int kSfBaseCol = kPairN;              // after the accumulator
  static_assert(kSfBaseCol + kPStages * kSfSlotCols <= int(kPTmemCols), "tensor memory budget");
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + kPStages * kABytes;
  static constexpr int kOffSfa = kOffB + kPStages * kBBytes;
  static constexpr int kOffSfb = kOffSfa + kPStages * kSfaBytes;
  static constexpr int kOffEpi = kOffSfb + kPStages * kSfbBytes;
  static constexpr int kOffBar = kOffEpi + kPEpiWarps * 2048;
  static constexpr int kNumBars = 2 * kPStages + 3;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 64 + 1024;  // + alignment slack
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

struct PairTile {
  int64_t m0;       // this block's first accumulator row
  int64_t n0;       // first column of the pair tile
  int32_t b_row;    // first row of this block's half of the B tile
  int32_t sfa_rt;   // 128-row scale tile of this block's A rows
  int32_t sfb_rt0;  // first of the two 128-row scale tiles of B
};

// Pair unit u: banded raster over 256-row m-units (band_m / 2 units per
// band, n outer inside a band) so a band of A stays in L2 while B streams.
__device__ __forceinline__ PairTile pair_tile(const GemmParams& p, int64_t u, int64_t n_tiles,
                                              uint32_t rank) {
  const int64_t m_units = (p.m + 2 * kRowsPerBlock - 1) / (2 * kRowsPerBlock);
  const int64_t band_units = p.band_m / 2 > 0 ? p.band_m / 2 : 1;
  const int64_t band_size = band_units * n_tiles;
  const int64_t band = u / band_size;
  const int64_t within = u - band * band_size;
  const int64_t in_band = ::min(band_units, m_units - band * band_units);
  const int64_t n_blk = within / in_band;
  const int64_t mu = band * band_units + (within - n_blk * in_band);
  PairTile t;
  t.m0 = mu * 2 * kRowsPerBlock + rank * kRowsPerBlock;
  t.n0 = n_blk * kPairN;
  t.b_row = static_cast<int32_t>(t.n0 + rank * (kPairN / 2));
  t.sfa_rt = static_cast<int32_t>(mu * 2 + rank);
  t.sfb_rt0 = static_cast<int32_t>(t.n0 / 128);
  return t;
}

template <bool FUSED>
__global__ void __launch_bounds__(kPThreads, 1)
    mx_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmap_a,
                        const __grid_constant__ CUtensorMap tmap_b,
                        const __grid_constant__ CUtensorMap tmap_sa,
                        const __grid_constant__ CUtensorMap tmap_sb, const GemmParams p) {
  using C = PairCfg;
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

  const uint32_t warp = warp_id();
  const uint32_t lane = lane_id();
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int64_t cluster_id = blockIdx.x / 2;
  const int64_t num_clusters = gridDim.x / 2;

  if (warp == 0 && lane == 0) {
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
  if (warp == 1) {
    tmem_alloc_pair(s_tmem, kPTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before_sync();
  cluster_sync();  // barriers of both blocks exist before any cross-block use
  tc_fence_after_sync();
  const uint32_t tmem_base = *s_tmem;

  const int64_t n_tiles = (p.n + kPairN - 1) / kPairN;
  const int64_t num_units = ((p.m + 2 * kRowsPerBlock - 1) / (2 * kRowsPerBlock)) * n_tiles;
  const int32_t k_tiles = static_cast<int32_t>((p.k + kBK - 1) / kBK);
  const int32_t k_blocks = static_cast<int32_t>(p.k / 32);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Whole warp; one elected lane issues (warp-uniform operands).
    const uint32_t full_leader0 = cluster_map(&full[0], 0);
    uint32_t stage = 0, phase = 0;
    int64_t issued = 0;
    bool ok = true;
    for (int64_t u = cluster_id; u < num_units && ok; u += num_clusters) {
      const PairTile t = pair_tile(p, u, n_tiles, rank);
      for (int32_t kt = 0; kt < k_tiles; ++kt) {
        if (!mbar_wait_warp(&empty[stage], phase ^ 1u, s_abort, p.status, p.wait_limit_ns)) {
          ok = false;
          break;
        }
        if (elect_one()) {
          if (leader) mbar_arrive_expect_tx(&full[stage], C::kPairTx);
          const uint32_t bar = full_leader0 + stage * 8u;
          const int32_t kx = kt * kBK;
          tma_load_2d_pair(sA + stage * C::kABytes, &tmap_a, bar, kx, static_cast<int32_t>(t.m0));
          tma_load_2d_pair(sB + stage * C::kBBytes, &tmap_b, bar, kx, t.b_row);
          tma_load_3d_pair(sSfa + stage * C::kSfaBytes, &tmap_sa, bar, 0, kt, t.sfa_rt);
          tma_load_3d_pair(sSfb + stage * C::kSfbBytes, &tmap_sb, bar, 0, kt, t.sfb_rt0);
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
    const int32_t kt_full = k_blocks / 4;
    uint32_t stage = 0, phase = 0, acc_phase = 0;
    bool ok = true;
    for (int64_t u = cluster_id; u < num_units && ok; u += num_clusters) {
      if (!mbar_wait_warp(acc_empty, acc_phase ^ 1u, s_abort, p.status, p.wait_limit_ns)) break;
      tc_fence_after_sync();
      for (int32_t kt = 0; kt < k_tiles; ++kt) {
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
      if (elect_one()) tc_commit_pair_multicast(acc_full, kBoth);
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
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogue (both blocks)
    const uint32_t q = warp & 3u;
    const uint32_t half = (warp - 2) >> 2;
    uint8_t* stage_buf = sEpi + (warp - 2) * 2048;
    const uint32_t acc_empty_leader = cluster_map(acc_empty, 0);
    uint32_t acc_phase = 0;
    for (int64_t u = cluster_id; u < num_units; u += num_clusters) {
      const PairTile t = pair_tile(p, u, n_tiles, rank);
      const bool got = mbar_wait(acc_full, acc_phase, s_abort, p.status, p.wait_limit_ns);
      if (!__all_sync(0xffffffffu, got)) break;
      tc_fence_after_sync();
      const uint32_t t_row = tmem_base + ((q * 32u) << 16) + half * (kPairN / 2);
      epilogue_share<kPairN, FUSED>(p, t_row, t.m0 + q * 32, t.n0 + half * (kPairN / 2), p.m,
                                    stage_buf, lane, false, [&] {
                                      tc_fence_before_sync();
                                      __syncwarp();
                                      if (lane == 0) mbar_arrive_cluster(acc_empty_leader);
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

template <bool FUSED>
cudaError_t launch_pair_impl(const GemmParams& p, const CUtensorMap& ta, const CUtensorMap& tb,
                             const CUtensorMap& tsa, const CUtensorMap& tsb, int num_sms,
                             cudaStream_t stream) {
  auto kern = mx_gemm_pair_kernel<FUSED>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               PairCfg::kSmemBytes);
    if (err != cudaSuccess) return err;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  const int64_t units =
      ((p.m + 2 * kRowsPerBlock - 1) / (2 * kRowsPerBlock)) * ((p.n + kPairN - 1) / kPairN);
  if (units == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = PairCfg::kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int max_clusters = num_sms / 2;
  cfg.gridDim = dim3(static_cast<unsigned>(max_clusters * 2));
  int active = 0;
  if (cudaOccupancyMaxActiveClusters(&active, kern, &cfg) == cudaSuccess && active > 0)
    max_clusters = ::min(max_clusters, active);
  const int64_t clusters = units < max_clusters ? units : max_clusters;
  cfg.gridDim = dim3(static_cast<unsigned>(clusters * 2));
  return cudaLaunchKernelEx(&cfg, kern, ta, tb, tsa, tsb, p);
}

}  // namespace

cudaError_t launch_gemm_pair(const GemmParams& p, const CUtensorMap& tmap_a,
                             const CUtensorMap& tmap_b, const CUtensorMap& tmap_sa,
                             const CUtensorMap& tmap_sb, int num_sms, cudaStream_t stream) {
  if (p.groups > 0) return cudaErrorNotSupported;
  if (p.bias != nullptr || p.act != 0)
    return launch_pair_impl<true>(p, tmap_a, tmap_b, tmap_sa, tmap_sb, num_sms, stream);
  return launch_pair_impl<false>(p, tmap_a, tmap_b, tmap_sa, tmap_sb, num_sms, stream);
}

}  // namespace mx
