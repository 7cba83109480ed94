// ptx.cuh -- hand-written inline-PTX wrappers for sm_103a: mbarrier, TMA
// (cp.async.bulk / cp.async.bulk.tensor), and the fifth-generation tensor
// core instructions (tcgen05.alloc / cp / mma / commit / ld).
#pragma once

#include <cstdint>

#include "status.cuh"

namespace mx {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }
__device__ __forceinline__ uint32_t warp_id() { return threadIdx.x >> 5; }

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbarrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase of `parity` to complete.  Gives up when the
// block-wide abort flag is raised (unless `drain`) or after `limit_ns`
// nanoseconds; on a timeout it records MX_DEV_TIMEOUT in the device status
// word and raises the abort flag so every other role of the block stops
// waiting too.  `drain` waits are used at teardown for work already in
// flight (copies, MMAs), which completes by itself, so they ignore the
// abort flag and only honour the time limit.  Returns false when the wait
// gave up.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          volatile uint32_t* abort_flag, uint32_t* status,
                                          uint64_t limit_ns, bool drain = false) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  uint32_t spins = 0;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((++spins & 63u) == 0) {
      if (!drain && *abort_flag) return false;
      if (global_timer_ns() - t0 > limit_ns) {
        record_device_status(status, MX_DEV_TIMEOUT);
        *abort_flag = 1u;
        return false;
      }
    }
  }
}

// One lane of a fully active warp (the same lane every time).  Tensor-core
// and TMA instructions are issued by this lane while the whole warp computes
// their operands, so the operands are warp-uniform and no per-instruction
// conversion into uniform registers is needed.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred;
  asm volatile(
      "{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

// Register reallocation between the warpgroups of a block: every warp of a
// warpgroup executes the same instruction.  A decrease returns registers to
// the block's pool; an increase waits until the pool holds them, so the
// warpgroups' new shares must sum to at most the block's launch allocation
// (threads x registers per thread at launch).
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_dec() {
  static_assert(N >= 24 && N <= 256 && N % 8 == 0, "register count");
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_inc() {
  static_assert(N >= 24 && N <= 256 && N % 8 == 0, "register count");
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// mbar_wait by every lane of a warp; the verdict is made warp-uniform (a
// lane that gave up makes the whole warp give up).
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity,
                                               volatile uint32_t* abort_flag, uint32_t* status,
                                               uint64_t limit_ns, bool drain = false) {
  const bool got = mbar_wait(bar, parity, abort_flag, status, limit_ns, drain);
  return __all_sync(0xffffffffu, got);
}

// ---------------------------------------------------------------- programmatic dependent launch

// The library's kernels are launched with programmatic stream serialization:
// a kernel may start (on SMs its predecessor in the stream has left) while
// that predecessor is still running, so its set-up (barriers, tensor memory,
// descriptor prefetch) overlaps the predecessor's tail.  pdl_wait() blocks
// until the predecessor has completed and its memory operations are
// visible; every kernel calls it before its first global memory access.
// pdl_launch_dependents() allows the next kernel of the stream to start
// launching.  Without the launch attribute both are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- clusters

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Full cluster barrier (every thread of every block of the cluster).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}

// ---------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// 2-D tiled tensor load global -> shared, completing on `bar` (tx bytes).
// x is the innermost (contiguous) coordinate; it must be a multiple of
// 16 elements for 8-bit data.
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const void* tmap, uint64_t* bar,
                                            int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}

// ---------------------------------------------------------------- tcgen05

__device__ __forceinline__ void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Load 32 consecutive 32-bit columns of this warp's 32 tensor-memory lanes:
// thread t receives lane (quarter*32 + t), columns [col, col + 32).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32"
      " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15,"
      " %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31},"
      " [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- descriptors

// Shared-memory matrix descriptor of the tcgen05 instructions, as two
// 32-bit halves.  Low half: start address and leading byte offset (16-byte
// units); high half: stride byte offset (16-byte units), version 1 (bit 46
// of the 64-bit descriptor) and the swizzle mode in bits 61..63 (0 none,
// 2 = 128-byte swizzle).
__device__ __forceinline__ uint32_t smem_desc_lo(uint32_t saddr, uint32_t lbo_bytes) {
  return ((saddr >> 4) & 0x3FFFu) | (((lbo_bytes >> 4) & 0x3FFFu) << 16);
}
__host__ __device__ constexpr uint32_t smem_desc_hi(uint32_t sbo_bytes, uint32_t swizzle_mode) {
  return ((sbo_bytes >> 4) & 0x3FFFu) | (1u << 14) | ((swizzle_mode & 0x7u) << 29);
}

// Instruction descriptor of kind::mxf8f6f4 with block scaling: K-major A
// and B, dense, E8M0 scale format, scale-factor byte ids for A and B.
// fmt codes: 0 = E4M3, 1 = E5M2, 3 = E2M3, 4 = E3M2, 5 = E2M1.
__host__ __device__ constexpr uint32_t mxf8_idesc(uint32_t fa, uint32_t fb, uint32_t m,
                                                  uint32_t n, uint32_t sfa_id, uint32_t sfb_id) {
  return (sfb_id & 3u) << 4 | (fa & 7u) << 7 | (fb & 7u) << 10 | ((n >> 3) & 0x3Fu) << 17 |
         1u << 23 | ((m >> 4) & 0x1Fu) << 24 | (sfa_id & 3u) << 29;
}

// ---------------------------------------------------------------- block pairs
// (cta_group::2: one MMA spans the tensor cores of both blocks of a
// two-block cluster; rank 0 issues it)

// Address of the same shared-memory variable in block `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_map(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}

// Arrive without memory-ordering semantics: for releasing tensor memory
// that this thread finished reading with tcgen05.ld + tcgen05.wait::ld and
// a tcgen05.fence::before_thread_sync.  A release arrive would also wait
// until this thread's earlier global stores are visible, which the
// accumulator handoff does not need.
__device__ __forceinline__ void mbar_arrive_relaxed_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

// Arrive (count one) on an mbarrier given by its cluster address.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

// Tiled loads into this block's shared memory that complete on an mbarrier
// of either block of the pair (given by cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void* smem_dst, const void* tmap,
                                                 uint32_t bar_cluster, int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar_cluster), "r"(x), "r"(y)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d_pair(void* smem_dst, const void* tmap,
                                                 uint32_t bar_cluster, int32_t x, int32_t y,
                                                 int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar_cluster), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// Executed by one warp of each block of the pair, collectively.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(slot)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// Scale copy of the pair: each block's shared-memory matrix (same offset)
// goes to the same tensor-memory address of that block.
__device__ __forceinline__ void tc_cp_pair_32x128b_warpx4(uint32_t taddr, uint32_t lo,
                                                          uint32_t hi) {
  asm volatile(
      "{\n\t.reg .b64 d;\n\tmov.b64 d, {%1, %2};\n\t"
      "tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], d;\n\t}" ::"r"(taddr),
      "r"(lo), "r"(hi)
      : "memory");
}

// M = 256 MMA over the pair: A rows 0..127 from block 0's shared memory and
// 128..255 from block 1's (same offset); B's N rows split likewise; each
// block accumulates its 128 rows in its own tensor memory with its own
// scale factors.
__device__ __forceinline__ void tc_mma_pair_mxf8(uint32_t d_tmem, uint32_t a_lo, uint32_t a_hi,
                                                 uint32_t b_lo, uint32_t b_hi, uint32_t idesc,
                                                 uint32_t sfa_tmem, uint32_t sfb_tmem,
                                                 uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 da, db;\n\t"
      "mov.b64 da, {%1, %2};\n\t"
      "mov.b64 db, {%3, %4};\n\t"
      "setp.ne.b32 p, %8, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X"
      " [%0], da, db, %5, [%6], [%7], p;\n\t}" ::"r"(d_tmem),
      "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem),
      "r"(accumulate)
      : "memory");
}

// Completion of the pair's tensor-core work so far arrives on the mbarrier
// at the same offset in every block of `cta_mask`.
__device__ __forceinline__ void tc_commit_pair_multicast(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}

}  // namespace mx
