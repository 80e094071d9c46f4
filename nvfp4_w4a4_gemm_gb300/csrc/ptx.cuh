// Inline-PTX helpers for sm_103a: mbarriers with bounded waits, TMA bulk
// copies, tcgen05 (TMEM alloc, MMA, commit, loads, smem->tmem copy) and the
// FP4/FP8 conversions.  Everything here is a thin wrapper over one PTX
// instruction (or a short fixed sequence of them).
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace nv4 {

// ----------------------------------------------------------- error word ----
// Status word of the translation unit that includes this header (internal
// linkage: each .cu file has its own copy and exports host accessors for
// it).  Word 0 = first error code, word 1 = which wait gave up.
enum : uint32_t { kDevErrNone = 0, kDevErrInvalidArg = 1, kDevErrTimeout = 4 };
static __device__ uint32_t g_dev_status[2] = {0u, 0u};
// Spin limit for every bounded wait of the translation unit, in %globaltimer
// nanoseconds (2 s); like the status word, each .cu file has its own copy and
// its own host setter (nvfp4_set_wait_limit_ns calls all of them).
static __device__ uint64_t g_wait_limit_ns = 2000000000ull;

__device__ __forceinline__ void report_error(uint32_t code, uint32_t where) {
  if (atomicCAS(&g_dev_status[0], 0u, code) == 0u) g_dev_status[1] = where;
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------- mbarrier ----
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// One elected lane of a fully converged warp (elect.sync).  Issue points of
// asynchronous work (TMA, tcgen05.mma / cp / commit) use it so the issuing
// warp stays converged: a single lane running a loop of its own, with
// shared-memory polls between MMAs, was measured to stall the tensor pipe
// (about 2.8x lower MMA throughput).
__device__ __forceinline__ bool elect_one() {
  uint32_t pred;
  asm volatile("{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}" : "=r"(pred));
  return pred != 0;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
               : "memory");
}
// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start while the preceding kernel of its stream runs;
// griddepcontrol.wait blocks the calling thread until that kernel has
// completed and its writes are visible.  launch_dependents lets the next
// such kernel start (it has no effect on other launches).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// n arrivals at once (a barrier whose phase other threads complete one by one)
__device__ __forceinline__ void mbar_arrive_n(uint64_t* bar, uint32_t n) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(bar)), "r"(n)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
// Adds `bytes` to the transaction count of the current phase (no arrival).
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: returns false (and records a timeout) when the phase has not
// completed within the device-wide limit.  `aborted` lets a CTA stop waiting
// as soon as another of its warps has given up.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t where,
                                          volatile int* aborted) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  const uint64_t limit = g_wait_limit_ns;
  uint32_t n = 0;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((++n & 255u) == 0u) {
      if (aborted != nullptr && *aborted) return false;
      if (globaltimer() - t0 > limit) {
        report_error(kDevErrTimeout, where);
        if (aborted != nullptr) *aborted = 1;
        return false;
      }
    }
  }
}

// mbar_wait executed by a whole converged warp; the result is warp-uniform
// (false in every lane if any lane gave up).
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity, uint32_t where,
                                               volatile int* aborted) {
  const bool ok = mbar_wait(bar, parity, where, aborted);
  return __all_sync(0xffffffffu, ok);
}

// ------------------------------------------------------------------ TMA ----
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* d) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(d)) : "memory");
}
// 2D tiled tensor load global -> shared, completion on an mbarrier.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* desc, uint64_t* bar, int32_t x,
                                            int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(desc)), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}
// 3D tiled tensor load (used for per-expert stacked weights).
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* desc, uint64_t* bar, int32_t x,
                                            int32_t y, int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], "
      "[%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(desc)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}
// Plain bulk copy global -> shared (16-byte aligned, size multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// -------------------------------------------------------------- tcgen05 ----
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Arrive on `bar` once all tcgen05 operations issued so far by this thread
// have completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}
// Block-scaled FP4 MMA: D[tmem] (+)= (A*sfa) x (B*sfb)^T, K = 64 per issue.
// kind::mxf4nvf4 with 4 scales per row per issue (16-element blocks, E4M3 or
// UE8M0 scales as the instruction descriptor says).
__device__ __forceinline__ void mma_nvf4_4x(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}
// MXFP4: kind::mxf4, 2 UE8M0 scales per row per issue (32-element blocks).
__device__ __forceinline__ void mma_mxf4_2x(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}
// BF16 MMA (kind::f16), K = 16 per issue, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// FP8 MMA (kind::f8f6f4, element types from the instruction descriptor),
// K = 32 per issue, fp32 accumulate, no block scales.
__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Copy a 128-row x 16-byte scale tile from shared memory (described by an
// smem matrix descriptor) into 4 TMEM columns, replicated to all 4 lane
// quarters (32 lanes x 128 bits, warpx4).
__device__ __forceinline__ void tmem_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
// Load 32 lanes x 16 consecutive 32-bit columns (one row per thread).
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
// 16 TMEM lanes x 64 columns (shape 16x256b, 8 repetitions): thread t gets,
// for j = 0..7, r[4j], r[4j+1] = lane t/4, columns 8j + 2(t%4) + {0, 1} and
// r[4j+2], r[4j+3] = lane 8 + t/4, the same columns.
__device__ __forceinline__ void tmem_ld_16x256b_x8(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor (tcgen05 format): start address, leading
// and stride byte offsets (all >> 4), descriptor version 1 at bit 46 and the
// swizzle mode in bits 61..63 (2 = 128-byte swizzle, 0 = none).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t swizzle) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)(swizzle & 7u) << 61;
  return d;
}

// ------------------------------------- clusters: CTA pairs, shared data --
// Two CTAs of a 2-CTA cluster run one tcgen05 MMA stream together: the even
// rank (the leader) issues MMAs, scale copies and commits for both, each CTA
// keeps its half of the operands in its own shared memory and its half of
// the accumulator in its own TMEM.  The decode layer's 4-CTA clusters share
// the quantized tokens with CTA-to-CTA bulk copies.  Shared-memory addresses
// of any CTA of the cluster are reached through the cluster window (mapa).
__device__ __forceinline__ uint32_t cta_rank_in_cluster() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(smem_u32(p)), "r"(rank));
  return out;
}
// Bulk copy (async proxy) of `bytes` (a multiple of 16, both addresses 16-byte
// aligned) from this CTA's shared memory into the shared memory of a CTA of
// the cluster; the bytes complete on that CTA's mbarrier `bar_caddr`.
__device__ __forceinline__ void bulk_copy_to_cta(uint32_t dst_caddr, const void* src, uint32_t bytes,
                                                 uint32_t bar_caddr) {
  asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   dst_caddr),
               "r"(smem_u32(src)), "r"(bytes), "r"(bar_caddr)
               : "memory");
}
// The two halves of a cluster barrier, for threads that have work to do
// between announcing they are here and needing everyone else to be.  The
// arrival has no memory ordering: enough after fence_mbar_init when the
// barriers' initialization is all the other CTAs need to see.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
// Every thread of every CTA of the cluster (release / acquire at cluster scope).
__device__ __forceinline__ void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// One arrival on an mbarrier of any CTA of the cluster (cluster address).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t caddr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(caddr) : "memory");
}
// The same arrival with release at CTA scope only: it does not wait for the
// thread's earlier global stores to become visible to the cluster.  Enough
// when what the arrival hands over is TMEM this thread has finished reading
// (tcgen05.wait::ld, then tcgen05.fence::before_thread_sync).
__device__ __forceinline__ void mbar_arrive_cluster_cta(uint32_t caddr) {
  asm volatile("mbarrier.arrive.release.cta.shared::cluster.b64 _, [%0];" ::"r"(caddr) : "memory");
}
// try_wait with acquire at cluster scope: for barriers that other CTAs of
// the cluster arrive on (their writes before the arrival become visible).
__device__ __forceinline__ bool mbar_try_wait_cl(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait (as mbar_wait) on a barrier that receives remote arrivals.
__device__ __forceinline__ bool mbar_wait_cl(uint64_t* bar, uint32_t parity, uint32_t where, volatile int* aborted) {
  if (mbar_try_wait_cl(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  const uint64_t limit = g_wait_limit_ns;
  uint32_t n = 0;
  while (true) {
    if (mbar_try_wait_cl(bar, parity)) return true;
    if ((++n & 255u) == 0u) {
      if (aborted != nullptr && *aborted) return false;
      if (globaltimer() - t0 > limit) {
        report_error(kDevErrTimeout, where);
        if (aborted != nullptr) *aborted = 1;
        return false;
      }
    }
  }
}
__device__ __forceinline__ bool mbar_wait_cl_warp(uint64_t* bar, uint32_t parity, uint32_t where,
                                                  volatile int* aborted) {
  const bool ok = mbar_wait_cl(bar, parity, where, aborted);
  return __all_sync(0xffffffffu, ok);
}
// 2D tiled tensor load into this CTA's shared memory whose completion bytes
// go to an mbarrier of either CTA of the pair (`bar_caddr`, cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* desc, uint32_t bar_caddr, int32_t x,
                                                 int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, {%3, "
      "%4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(desc)), "r"(bar_caddr), "r"(x), "r"(y)
      : "memory");
}
// The 3D form (per-expert stacked weights of a grouped GEMM).
__device__ __forceinline__ void tma_load_3d_pair(void* dst, const CUtensorMap* desc, uint32_t bar_caddr, int32_t x,
                                                 int32_t y, int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, {%3, "
      "%4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(desc)), "r"(bar_caddr), "r"(x), "r"(y), "r"(z)
      : "memory");
}
// Arrival on named barrier `id` without waiting (the barrier completes when
// `n` threads have arrived or synced on it).
__device__ __forceinline__ void named_bar_arrive(uint32_t id, uint32_t n) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}
// Barrier `id` (1..15) over the first `n` threads that reach it (whole warps).
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
// Generic-proxy shared-memory writes of this thread become visible to later
// async-proxy (TMA, tensor core) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// TMEM allocation shared by the pair: executed by one warp of EACH CTA.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// Arrive on an mbarrier of either CTA (cluster address) once the pair's
// tcgen05 operations issued so far by this thread have completed.
__device__ __forceinline__ void tc_commit_pair(uint32_t bar_caddr) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar_caddr)
               : "memory");
}
// Pair MMAs: M = 256 rows, 128 from each CTA's shared memory (same offset),
// B's N rows split in halves the same way, D in each CTA's own TMEM.
__device__ __forceinline__ void mma_nvf4_4x_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                 uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_mxf4_2x_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                 uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Block-scaled FP8 MMA on a CTA pair (kind::mxf8f6f4, one UE8M0 scale per
// row per 32 elements), K = 32 per issue, fp32 accumulate.
__device__ __forceinline__ void mma_mxf8_1x_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                 uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}
// Scale-tile copy in both CTAs of the pair: each CTA's shared memory at the
// descriptor's address into its own TMEM at taddr (replicated to all 4 lane
// quarters, as tmem_cp_32x128b_x4).
__device__ __forceinline__ void tmem_cp_32x128b_x4_pair(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// ---------------------------------------------------------- conversions ----
// Two fp32 -> one byte of two E2M1 codes, RNE + satfinite: `lo` goes to bits
// 0..3 and `hi` to bits 4..7.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
  uint32_t out;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
      : "=r"(out)
      : "f"(hi), "f"(lo));
  return out;
}
// 8 bf16 (4 packed words) times s2 = {s, s}: f32x2 multiplies, each product
// rounded to nearest fp32, then E2M1 codes (RNE, satfinite) packed into one
// word, element 2i in the low nibble of byte i.
__device__ __forceinline__ uint32_t bf16x8_mul_e2m1(const uint4& w, uint64_t s2) {
  uint32_t out;
#define NV4_E2M1_PAIR(W, T)                                                   \
  "shl.b32 lo, " W ", 16;\n\tand.b32 hi, " W ", 0xFFFF0000;\n\t"             \
  "mov.b64 x, {lo, hi};\n\tmul.rn.f32x2 p, x, %5;\n\tmov.b64 {lo, hi}, p;\n\t" \
  "cvt.rn.satfinite.e2m1x2.f32 " T ", hi, lo;\n\t"
  asm("{\n\t.reg .b64 x, p;\n\t.reg .b32 lo, hi;\n\t.reg .b8 t0, t1, t2, t3;\n\t"
      NV4_E2M1_PAIR("%1", "t0") NV4_E2M1_PAIR("%2", "t1") NV4_E2M1_PAIR("%3", "t2") NV4_E2M1_PAIR("%4", "t3")
      "mov.b32 %0, {t0, t1, t2, t3};\n\t}"
      : "=r"(out)
      : "r"(w.x), "r"(w.y), "r"(w.z), "r"(w.w), "l"(s2));
#undef NV4_E2M1_PAIR
  return out;
}
// The same with two products per element, each rounded to nearest fp32:
// E2M1(RN(RN(x * r) * s)) (r2 = {r, r}, s2 = {s, s}).
__device__ __forceinline__ uint32_t bf16x8_mul2_e2m1(const uint4& w, uint64_t r2, uint64_t s2) {
  uint32_t out;
#define NV4_E2M1_PAIR2(W, T)                                                                       \
  "shl.b32 lo, " W ", 16;\n\tand.b32 hi, " W ", 0xFFFF0000;\n\t"                                  \
  "mov.b64 x, {lo, hi};\n\tmul.rn.f32x2 p, x, %5;\n\tmul.rn.f32x2 p, p, %6;\n\tmov.b64 {lo, hi}, p;\n\t" \
  "cvt.rn.satfinite.e2m1x2.f32 " T ", hi, lo;\n\t"
  asm("{\n\t.reg .b64 x, p;\n\t.reg .b32 lo, hi;\n\t.reg .b8 t0, t1, t2, t3;\n\t"
      NV4_E2M1_PAIR2("%1", "t0") NV4_E2M1_PAIR2("%2", "t1") NV4_E2M1_PAIR2("%3", "t2") NV4_E2M1_PAIR2("%4", "t3")
      "mov.b32 %0, {t0, t1, t2, t3};\n\t}"
      : "=r"(out)
      : "r"(w.x), "r"(w.y), "r"(w.z), "r"(w.w), "l"(r2), "l"(s2));
#undef NV4_E2M1_PAIR2
  return out;
}
// Packed pairs of fp32 (low word = first element) and their element-wise
// IEEE round-to-nearest arithmetic (f32x2 instructions: one issue for two
// results, each rounded exactly as the scalar instruction would).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 f2_unpack(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
// Per-half max of magnitudes of two bf16 pairs (max.xorsign.abs: the result's
// sign bits carry no meaning, its magnitudes are max(|a|, |b|)).
__device__ __forceinline__ uint32_t bf16x2_absmax(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// 32-byte global store of 8 words (256-bit; the address must be 32-byte aligned).
__device__ __forceinline__ void stg_256(void* p, const uint32_t* w) {
  asm volatile("st.global.v8.u32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]),
               "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}
// 32-byte streaming global load (256-bit; the address must be 32-byte aligned).
__device__ __forceinline__ void ldg_stream32(const void* p, uint4& a, uint4& b) {
  asm volatile("ld.global.nc.L1::no_allocate.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z), "=r"(b.w)
               : "l"(p));
}
// One byte of two E2M1 codes -> two exact halves (low nibble -> .x).
__device__ __forceinline__ uint32_t cvt_e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t out;
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(out) : "r"(byte));
  return out;
}
// fp32 -> E4M3 byte (sign in bit 7), RNE + satfinite.
__device__ __forceinline__ uint32_t cvt_e4m3(float v) {
  uint32_t out;
  asm("{\n\t.reg .b16 t;\n\tcvt.rn.satfinite.e4m3x2.f32 t, %1, %2;\n\tcvt.u32.u16 %0, t;\n\t}"
      : "=r"(out)
      : "f"(0.0f), "f"(v));
  return out & 0xFFu;
}
// E4M3 byte -> exact fp32 (via f16x2).
__device__ __forceinline__ float e4m3_to_f32(uint32_t byte) {
  uint32_t h2;
  asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(h2) : "r"(byte));
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu)));
}

}  // namespace nv4
