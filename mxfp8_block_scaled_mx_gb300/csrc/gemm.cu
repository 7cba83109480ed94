// gemm.cu -- block-scaled MXFP8 GEMM on the fifth-generation tensor cores.
//
// "Low-Precision GPU Programming" (leetllm.com), section "Scale ownership
// and the GEMM dataflow": with 32-element blocks along K the scale product
// of each block stays inside the outer sum,
//     Y[i,j] = sum_b S_A[i,b] S_B[j,b] sum_{k in b} A~[i,k] B~[j,k],
// and block-scaled matrix instructions consume the scale operands directly.
// Here that instruction is tcgen05.mma.kind::mxf8f6f4.block_scale: one MMA
// covers K = 32 (one scale block), takes E4M3/E5M2 (or E2M3/E3M2/E2M1)
// operands from shared memory and E8M0 scales from tensor memory, and
// accumulates in FP32 in tensor memory.  This is the one-block kernel; the
// default for every mode is the block-pair kernel of gemm_pair.cu, which
// shares the work decomposition (tiles.cuh) and the epilogue.
//
// Structure (one persistent block of 10 warps per SM):
//   warp 0      TMA producer: A and B code tiles (128-byte swizzle) with
//               cp.async.bulk.tensor, the 512-byte scale units with
//               cp.async.bulk, into a ring of kStages shared-memory slots
//               guarded by full/empty mbarriers.
//   warp 1      allocates tensor memory; issues tcgen05.cp (scales ->
//               tensor memory) and tcgen05.mma, and releases each slot with
//               tcgen05.commit.
//   Both run as warp-wide loops in which one elected lane issues the copies
//   and tensor-core instructions, so their operands are warp-uniform.
//   warps 2..9  epilogue: tcgen05.ld of the FP32 accumulator into registers
//               (two warps per 32-lane quarter, half the columns each), early
//               release of the accumulator (one relaxed arrive per warp),
//               then (optionally) the FP32 bias and SiLU of the kernel
//               contract's epilogue, conversion to FP32/BF16 (RNE), staging
//               through shared memory and coalesced 64-byte row segments,
//               masked at the matrix (or group) edge.
// With 128-wide tiles the accumulator is double-buffered in tensor memory
// so the epilogue of one tile overlaps the main loop of the next.
//
// Clusters of CM = 2 blocks take two m-tiles of the same n-tile: each block
// loads its own A tile and half of the shared B tile, multicasting that half
// to both blocks, so B crosses from L2 once per pair.  A stage is released
// only when both blocks' MMAs are done with it (the MMA commit arrives on
// the empty barrier of both blocks).
//
// Grouped (mixture-of-experts) modes walk (group, m-tile, n-tile) triples;
// group offsets are read on the device and turned into a tile prefix by
// every block, so the host never synchronizes.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "epilogue.cuh"
#include "groups.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "status.cuh"
#include "tiles.cuh"

namespace mx {
namespace {

constexpr int BM = kTileM;
constexpr int BK = kTileK;
constexpr int kEpiWarps = 8;       // two per tensor-memory lane quarter
constexpr int kThreads = 64 + kEpiWarps * 32;
constexpr int kEpiStageBytes = 2048;  // per epilogue warp: 32 rows x 64 bytes
constexpr uint32_t kTmemCols = 512;

template <int BN, bool GROUPED>
struct Cfg {
  static constexpr int kStages = BN == 128 ? (GROUPED ? 5 : 6) : 4;
  static constexpr int kAccStages = BN == 128 ? 2 : 1;
  static constexpr int kABytes = BM * BK;
  static constexpr int kBBytes = BN * BK;
  static constexpr int kSfbUnits = BN / 128;
  static constexpr int kSfaCols = 4;
  static constexpr int kSfSlotCols = 4 + 4 * kSfbUnits;
  static constexpr int kSfBaseCol = kAccStages * BN;
  static_assert(kSfBaseCol + kStages * kSfSlotCols <= int(kTmemCols), "tensor memory budget");
  // shared memory layout (offsets from a 1024-aligned base)
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + kStages * kABytes;
  static constexpr int kOffSfa = kOffB + kStages * kBBytes;
  static constexpr int kOffSfb = kOffSfa + kStages * 512;
  static constexpr int kOffEpi = kOffSfb + kStages * kSfbUnits * 512;
  static constexpr int kOffBar = kOffEpi + kEpiWarps * kEpiStageBytes;
  static constexpr int kNumBars = 2 * kStages + 2 * kAccStages + 1;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kOffGroup = kOffMisc + 64;
  static constexpr int kSmemBytes =
      kOffGroup + (GROUPED ? int(sizeof(GroupSmem)) : 0) + 1024;  // + alignment slack
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

template <int BN, int MODE, int CM, bool FUSED>
__global__ void __launch_bounds__(kThreads, 1)
    mx_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                   const __grid_constant__ CUtensorMap tmap_b, const GemmParams p) {
  constexpr bool GROUPED = MODE != kModeDense;
  using C = Cfg<BN, GROUPED>;
  static_assert(CM == 1 || CM == 2, "cluster size");
  constexpr uint16_t kPairMask = 0x3;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem + C::kOffA;
  uint8_t* sB = smem + C::kOffB;
  uint8_t* sSfa = smem + C::kOffSfa;
  uint8_t* sSfb = smem + C::kOffSfb;
  uint8_t* sEpi = smem + C::kOffEpi;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* full = bars;
  uint64_t* empty = bars + C::kStages;
  uint64_t* acc_full = bars + 2 * C::kStages;
  uint64_t* acc_empty = acc_full + C::kAccStages;
  uint64_t* mma_done = acc_empty + C::kAccStages;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile uint32_t* s_abort = reinterpret_cast<volatile uint32_t*>(smem + C::kOffMisc + 4);
  GroupSmem* gs = reinterpret_cast<GroupSmem*>(smem + C::kOffGroup);

  const uint32_t warp = warp_id();
  const uint32_t lane = lane_id();
  const uint32_t rank = CM > 1 ? cluster_ctarank() : 0u;
  const int64_t cluster_id = blockIdx.x / CM;
  const int64_t num_clusters = gridDim.x / CM;

  if (warp == 0) {
    if (lane == 0) {
      for (int s = 0; s < C::kStages; ++s) {
        mbar_init(&full[s], 1);
        mbar_init(&empty[s], CM);  // one MMA commit from every block of the cluster
      }
      for (int s = 0; s < C::kAccStages; ++s) {
        mbar_init(&acc_full[s], 1);
        mbar_init(&acc_empty[s], kEpiWarps);  // one arrival per epilogue warp
      }
      mbar_init(mma_done, 1);
      *s_abort = 0u;
      fence_mbarrier_init();
      tma_prefetch_desc(&tmap_a);
      tma_prefetch_desc(&tmap_b);
    }
    __syncwarp();
    if constexpr (GROUPED) {
      // grouped along K the offsets split the p.k tokens of the contraction
      group_tile_prefix(p.offsets, p.groups, MODE == kModeGroupK ? p.k : p.m, gs->off, gs->tiles,
                        &gs->valid, CM, gs->units);
    }
  }
  if (warp == 1) {
    tmem_alloc(s_tmem, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  // Barriers of every block of the cluster must be initialized before any
  // block multicasts into them.
  if constexpr (CM > 1) {
    cluster_sync();
  } else {
    __syncthreads();
  }
  tc_fence_after_sync();
  const uint32_t tmem_base = *s_tmem;

  const int64_t n_tiles = (p.n + BN - 1) / BN;
  int64_t num_units;
  if constexpr (GROUPED) {
    // grouped along K, the 128-padded token segments must fit in A and B
    const bool fits = MODE != kModeGroupK ||
                      (gs->valid && static_cast<int64_t>(gs->tiles[p.groups]) * BK <= p.lda &&
                       static_cast<int64_t>(gs->tiles[p.groups]) * BK <= p.ldb);
    if (!gs->valid || !fits) {
      if (blockIdx.x == 0 && threadIdx.x == 0) record_device_status(p.status, MX_DEV_BAD_OFFSETS);
      num_units = 0;
    } else if constexpr (MODE == kModeGroupK) {
      num_units = static_cast<int64_t>(p.groups) * ((p.m + BM * CM - 1) / (BM * CM)) * n_tiles;
    } else {
      num_units = static_cast<int64_t>(gs->units[p.groups]) * n_tiles;
    }
  } else {
    num_units = ((p.m + BM * CM - 1) / (BM * CM)) * n_tiles;
  }

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The whole warp runs the loop and waits; one elected lane issues the
    // copies (warp-uniform operands, see elect_one).
    uint32_t stage = 0, phase = 0;
    int64_t issued = 0;  // stage fills issued so far
    bool ok = true;
    for (int64_t u = cluster_id; u < num_units && ok; u += num_clusters) {
      const TileInfo ti = tile_info<BN, MODE, CM>(p, u, n_tiles, rank, gs);
      int sfb_units = 0;
#pragma unroll
      for (int j = 0; j < C::kSfbUnits; ++j)
        if (ti.n0 + 128 * j < p.n) ++sfb_units;
      const uint32_t tx =
          C::kABytes + C::kBBytes + (ti.sfa_unit >= 0 ? 512u : 0u) + 512u * sfb_units;
      const uint8_t* sfa_src = p.sa + (ti.sfa_unit >= 0 ? ti.sfa_unit : 0) * 512;
      const uint8_t* sfb_src = p.sb + ti.sfb_unit * 512;
      const int64_t sfb_stride = ti.sfb_step * 512;
      const int32_t a_row = static_cast<int32_t>(ti.m0);
      const int32_t b_row = static_cast<int32_t>(ti.b_row0 + rank * (BN / CM));
      const int32_t kt_count = (ti.k_blocks + 3) / 4;
      for (int32_t kt = 0; kt < kt_count; ++kt) {
        if (!mbar_wait_warp(&empty[stage], phase ^ 1u, s_abort, p.status, p.wait_limit_ns)) {
          ok = false;
          break;
        }
        if (elect_one()) {
          mbar_arrive_expect_tx(&full[stage], tx);
          const int32_t kx_a = static_cast<int32_t>(ti.a_kx0) + kt * BK;
          const int32_t kx_b = static_cast<int32_t>(ti.b_kx0) + kt * BK;
          tma_load_2d(sA + stage * C::kABytes, &tmap_a, &full[stage], kx_a, a_row);
          if constexpr (CM > 1) {
            // this block's half of the shared B tile, delivered to both blocks
            tma_load_2d_multicast(sB + stage * C::kBBytes + rank * (C::kBBytes / CM), &tmap_b,
                                  &full[stage], kx_b, b_row, kPairMask);
          } else {
            tma_load_2d(sB + stage * C::kBBytes, &tmap_b, &full[stage], kx_b, b_row);
          }
          if (ti.sfa_unit >= 0) bulk_load(sSfa + stage * 512, sfa_src, 512, &full[stage]);
          for (int j = 0; j < sfb_units; ++j)
            bulk_load(sSfb + (stage * C::kSfbUnits + j) * 512, sfb_src + j * sfb_stride, 512,
                      &full[stage]);
        }
        __syncwarp();
        ++issued;
        sfa_src += 512;
        sfb_src += 512;
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    // Drain: every copy into this block's shared memory must land before
    // the block exits.
    for (int s = 0; s < C::kStages; ++s) {
      const int64_t fills = issued > s ? (issued - s + C::kStages - 1) / C::kStages : 0;
      if (fills)
        mbar_wait_warp(&full[s], static_cast<uint32_t>((fills - 1) & 1), s_abort, p.status,
                       p.wait_limit_ns, true);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop and computes the operands; one elected
    // lane (always the same one, so its commits track its own MMAs) issues
    // the scale copies, the MMAs and the commits.  Descriptor halves and
    // instruction descriptors are precomputed; the loop does 32-bit adds.
    constexpr uint32_t kHiOperand = smem_desc_hi(1024, 2);  // 8-row groups 1 KB apart, 128B swizzle
    constexpr uint32_t kHiScale = smem_desc_hi(128, 0);     // 32 rows x 16 B, no swizzle
    const uint32_t a_lo0 = smem_desc_lo(smem_u32(sA), 16);
    const uint32_t b_lo0 = smem_desc_lo(smem_u32(sB), 16);
    const uint32_t sfa_lo0 = smem_desc_lo(smem_u32(sSfa), 0);
    const uint32_t sfb_lo0 = smem_desc_lo(smem_u32(sSfb), 0);
    const uint32_t idesc0 = mxf8_idesc(p.fa, p.fb, BM, BN, 0, 0);
    // Grouped along K every group has its own contraction length; a group
    // without tokens has none (its output tile is written as zeros).
    const uint32_t group_units =
        static_cast<uint32_t>(((p.m + BM * CM - 1) / (BM * CM)) * n_tiles);
    int32_t k_blocks = static_cast<int32_t>(p.k / 32);
    uint32_t stage = 0, phase = 0;
    uint32_t acc = 0, acc_phase = 0;
    bool ok = true;
    for (int64_t u = cluster_id; u < num_units && ok; u += num_clusters) {
      if constexpr (MODE == kModeGroupK) {
        const int g = static_cast<int>(static_cast<uint32_t>(u) / group_units);
        k_blocks = (gs->off[g + 1] - gs->off[g] + 31) / 32;
      }
      const int32_t kt_count = (k_blocks + 3) / 4;
      const int32_t kt_full = k_blocks / 4;  // k-tiles with all four scale blocks
      if (!mbar_wait_warp(&acc_empty[acc], acc_phase ^ 1u, s_abort, p.status, p.wait_limit_ns))
        break;
      tc_fence_after_sync();
      const uint32_t d_tmem = tmem_base + acc * BN;
      for (int32_t kt = 0; kt < kt_count; ++kt) {
        if (!mbar_wait_warp(&full[stage], phase, s_abort, p.status, p.wait_limit_ns)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t sf_tmem = tmem_base + C::kSfBaseCol + stage * C::kSfSlotCols;
        const uint32_t a_lo = a_lo0 + stage * (C::kABytes >> 4);
        const uint32_t b_lo = b_lo0 + stage * (C::kBBytes >> 4);
        const uint32_t sfa_lo = sfa_lo0 + stage * (512 >> 4);
        const uint32_t sfb_lo = sfb_lo0 + stage * C::kSfbUnits * (512 >> 4);
        const uint32_t sfb_tmem = sf_tmem + C::kSfaCols;
        if (elect_one()) {
          tc_cp_32x128b_warpx4_lohi(sf_tmem, sfa_lo, kHiScale);
#pragma unroll
          for (int j = 0; j < C::kSfbUnits; ++j)
            tc_cp_32x128b_warpx4_lohi(sfb_tmem + 4 * j, sfb_lo + j * (512 >> 4), kHiScale);
          // +32 bytes along K inside the 128-byte swizzled row = +2 in the
          // 16-byte address field; block kb's scales are byte kb of the
          // scale columns (scale-factor ids in the instruction descriptor).
          if (kt < kt_full) {
            tc_mma_mxf8_lohi(d_tmem, a_lo, kHiOperand, b_lo, kHiOperand, idesc0, sf_tmem,
                             sfb_tmem, kt > 0 ? 1u : 0u);
#pragma unroll
            for (uint32_t kb = 1; kb < 4; ++kb)
              tc_mma_mxf8_lohi(d_tmem, a_lo + 2u * kb, kHiOperand, b_lo + 2u * kb, kHiOperand,
                               idesc0 | (kb << 4) | (kb << 29), sf_tmem, sfb_tmem, 1u);
          } else {
            const uint32_t kb_here = static_cast<uint32_t>(k_blocks - kt * 4);
            for (uint32_t kb = 0; kb < kb_here; ++kb)
              tc_mma_mxf8_lohi(d_tmem, a_lo + 2u * kb, kHiOperand, b_lo + 2u * kb, kHiOperand,
                               idesc0 | (kb << 4) | (kb << 29), sf_tmem, sfb_tmem,
                               (kt > 0 || kb > 0) ? 1u : 0u);
          }
          if constexpr (CM > 1) {
            tc_commit_multicast(&empty[stage], kPairMask);
          } else {
            tc_commit(&empty[stage]);
          }
        }
        __syncwarp();
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      if (elect_one()) {
        if (kt_count > 0) {
          tc_commit(&acc_full[acc]);
        } else {
          mbar_arrive(&acc_full[acc]);  // nothing to accumulate: the epilogue writes zeros
        }
      }
      __syncwarp();
      if (++acc == C::kAccStages) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    // Every issued tensor-core operation must finish before tensor memory
    // is released.
    if (elect_one()) {
      tc_commit(mma_done);
      mbar_wait(mma_done, 0, s_abort, p.status, p.wait_limit_ns, true);
    }
    __syncwarp();
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogue
    // Eight warps: warp w reads lane quarter w % 4 (rows 32*(w%4) ..) and
    // column half (w - 2) / 4 of the accumulator.  Each warp first pulls its
    // whole share out of tensor memory into registers (FP32, or packed BF16),
    // releases the accumulator to the MMA warp, and only then converts and
    // stores through a 2 KB shared staging buffer, so the stores overlap the
    // next tile's main loop.
    constexpr int kCols = BN / 2;                  // accumulator columns per warp
    const uint32_t q = warp & 3u;
    const uint32_t half = (warp - 2) >> 2;
    uint8_t* stage_buf = sEpi + (warp - 2) * kEpiStageBytes;
    uint32_t acc = 0, acc_phase = 0;
    for (int64_t u = cluster_id; u < num_units; u += num_clusters) {
      const TileInfo ti = tile_info<BN, MODE, CM>(p, u, n_tiles, rank, gs);
      const bool got = mbar_wait(&acc_full[acc], acc_phase, s_abort, p.status, p.wait_limit_ns);
      if (!__all_sync(0xffffffffu, got)) break;
      tc_fence_after_sync();
      const uint32_t t_row = tmem_base + ((q * 32u) << 16) + acc * BN + half * kCols;
      const int64_t grow0 = ti.y_row0 + q * 32;
      const int64_t gcol0 = ti.n0 + half * kCols;
      epilogue_share<BN, FUSED>(p, t_row, grow0, gcol0, ti.m_end, stage_buf, lane, ti.k_blocks == 0,
                                [&] {
                                  tc_fence_before_sync();
                                  __syncwarp();
                                  if (lane == 0) mbar_arrive_relaxed(&acc_empty[acc]);
                                });
      if (++acc == C::kAccStages) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, kTmemCols);
  }
  // No block of the cluster may exit while its peer can still multicast
  // into its shared memory or arrive on its barriers.
  if constexpr (CM > 1) cluster_sync();
}

__global__ void wait_selftest_kernel(uint32_t* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ uint32_t abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbarrier_init();
    // Nothing ever arrives on `bar`: the wait must give up by itself.
    mbar_wait(&bar, 0, &abort_flag, status, limit_ns);
  }
}

template <int BN, int MODE, int CM, bool FUSED = false>
cudaError_t launch_impl(const GemmParams& p, const CUtensorMap& ta, const CUtensorMap& tb,
                        int num_sms, cudaStream_t stream) {
  using C = Cfg<BN, MODE != kModeDense>;
  auto kern = mx_gemm_kernel<BN, MODE, CM, FUSED>;
  // The attribute is per function and device; set it once per device.
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (err != cudaSuccess) return err;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  const int64_t n_tiles = (p.n + BN - 1) / BN;
  const int64_t m_tiles = (p.m + BM - 1) / BM;
  // upper bound of the work units (grouped by rows: every group may add a
  // partial unit; grouped along K: every group covers the whole output)
  int64_t units = ((m_tiles + CM - 1) / CM) * n_tiles;
  if (MODE == kModeGroupM) units = ((m_tiles + p.groups + CM - 1) / CM + p.groups) * n_tiles;
  if (MODE == kModeGroupK) units *= p.groups;
  if (units == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CM;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int max_clusters = num_sms / CM;
  if (CM > 1) {
    cfg.gridDim = dim3(static_cast<unsigned>(max_clusters * CM));
    int active = 0;
    if (cudaOccupancyMaxActiveClusters(&active, kern, &cfg) == cudaSuccess && active > 0)
      max_clusters = ::min(max_clusters, active);
  }
  const int64_t clusters = units < max_clusters ? units : max_clusters;
  cfg.gridDim = dim3(static_cast<unsigned>(clusters * CM));
  return cudaLaunchKernelEx(&cfg, kern, ta, tb, p);
}

template <int MODE>
cudaError_t launch_mode(const GemmParams& p, const CUtensorMap& ta, const CUtensorMap& tb,
                        int block_n, int cluster_m, int num_sms, cudaStream_t stream) {
  if (block_n == 256)
    return cluster_m == 2 ? launch_impl<256, MODE, 2>(p, ta, tb, num_sms, stream)
                          : launch_impl<256, MODE, 1>(p, ta, tb, num_sms, stream);
  return cluster_m == 2 ? launch_impl<128, MODE, 2>(p, ta, tb, num_sms, stream)
                        : launch_impl<128, MODE, 1>(p, ta, tb, num_sms, stream);
}

}  // namespace

int gemm_default_block_n(const GemmParams& p) {
  (void)p;
  return 256;
}

cudaError_t launch_gemm(const GemmParams& p, const CUtensorMap& ta, const CUtensorMap& tb,
                        int block_n, int cluster_m, int num_sms, cudaStream_t stream) {
  if (p.bias != nullptr || p.act != 0) {  // fused epilogue: dense GEMMs only
    if (p.mode != kModeDense) return cudaErrorNotSupported;
    if (block_n == 256)
      return cluster_m == 2 ? launch_impl<256, kModeDense, 2, true>(p, ta, tb, num_sms, stream)
                            : launch_impl<256, kModeDense, 1, true>(p, ta, tb, num_sms, stream);
    return cluster_m == 2 ? launch_impl<128, kModeDense, 2, true>(p, ta, tb, num_sms, stream)
                          : launch_impl<128, kModeDense, 1, true>(p, ta, tb, num_sms, stream);
  }
  if (p.mode == kModeGroupM)
    return launch_mode<kModeGroupM>(p, ta, tb, block_n, cluster_m, num_sms, stream);
  if (p.mode == kModeGroupK)
    return launch_mode<kModeGroupK>(p, ta, tb, block_n, cluster_m, num_sms, stream);
  return launch_mode<kModeDense>(p, ta, tb, block_n, cluster_m, num_sms, stream);
}

cudaError_t launch_wait_selftest(uint32_t* status, uint64_t limit_ns, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace mx
