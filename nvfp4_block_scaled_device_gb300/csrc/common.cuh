// Device-side helpers shared by the NVFP4 kernels: inline-PTX wrappers for
// mbarriers, TMA, tcgen05 (tensor memory, MMA, copies), bounded waits and the
// FP4/FP8 conversions.  sm_103a only.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace nvfp4 {

// Error code written to the device status word when a wait gives up; the
// value is kErrTimeout * 100 + a site number.
constexpr int kErrTimeout = 6;

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ bool elect_one()
{
    uint32_t pred = 0;
    asm volatile(
        "{\n .reg .b32 r;\n .reg .pred p;\n"
        " elect.sync r|p, 0xffffffff;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(pred));
    return pred != 0;
}

// ------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits give up after about kWaitLimitCycles SM clock cycles (~2 s at
// 2 GHz): the SM cycle counter is cheap to read, and a healthy wait never
// comes near the limit.
constexpr uint64_t kWaitLimitCycles = 4000000000ull;

// Bounded wait that ignores the abort flag (used while tearing down).
__device__ __forceinline__ void mbar_wait_teardown(uint32_t bar, uint32_t parity)
{
    const uint64_t t0 = clock64();
    while (!mbar_try_wait(bar, parity) && (uint64_t)(clock64() - t0) < kWaitLimitCycles / 8) {
    }
}

// Per-warpgroup register budget (all four warps of a warpgroup execute the
// same instruction).  The block's registers are split per SM sub-partition,
// one warp of each warpgroup per sub-partition: the decreases must free what
// the increases take.
template <uint32_t kRegs>
__device__ __forceinline__ void setmaxnreg_dec()
{
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegs));
}
template <uint32_t kRegs>
__device__ __forceinline__ void setmaxnreg_inc()
{
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegs));
}

// ------------------------------------------------------------------ TMA
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t x, int32_t y, uint64_t cache_hint)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "l"(cache_hint)
        : "memory");
}

// tma_load_2d for an SM pair: the copy lands in this CTA's shared memory and
// completes its bytes on `bar_cluster`, an mbarrier of either CTA of the pair
// (a shared::cluster address), so both CTAs' copies of a stage can report
// to one barrier of the pair's leader.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster,
                                                 int32_t x, int32_t y, uint64_t cache_hint)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y), "l"(cache_hint)
        : "memory");
}

// 1-D form of tma_load_2d_pair (element coordinate x).
__device__ __forceinline__ void tma_load_1d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster,
                                                 int32_t x, uint64_t cache_hint)
{
    asm volatile(
        "cp.async.bulk.tensor.1d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%3}], [%2], %4;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "l"(cache_hint)
        : "memory");
}

// 1-D bulk copy global -> shared (16-B aligned addresses, size % 16 == 0).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Programmatic dependent launch.  A kernel launched with the
// programmatic-serialization attribute may start while the previous kernel
// of the stream is still running: griddep_wait() returns once that kernel
// has completed and its memory operations are visible (at once without such
// a dependency).  griddep_launch_dependents() lets the next kernel of the
// stream be scheduled before this one completes.
__device__ __forceinline__ void griddep_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void griddep_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// -------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05 format, version 1).
//   start, lbo, sbo in bytes; layout: 0 none, 2 = 128-byte swizzle.
__device__ __forceinline__ uint64_t make_smem_desc(uint32_t start, uint32_t lbo, uint32_t sbo, uint32_t layout)
{
    uint64_t d = 0;
    d |= (uint64_t)((start >> 4) & 0x3FFF);
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;  // descriptor version for tcgen05
    d |= (uint64_t)(layout & 7) << 61;
    return d;
}

__device__ __forceinline__ uint64_t desc_from(uint32_t lo, uint32_t hi)
{
    return ((uint64_t)hi << 32) | lo;
}

// Block-scaled MMA: D[tmem] (+)= A[smem] * B[smem]^T with per-16 UE4M3
// scales of A and B read from tensor memory; E2M1 operands, fp32 accumulate.
__device__ __forceinline__ void mma_mxf4nvf4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                             uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate)
{
    asm volatile(
        "{\n .reg .pred p;\n"
        " setp.ne.b32 p, %6, 0;\n"
        " tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n"
        "}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// Copy one 512-byte scale tile (32 rows x 16 bytes in shared memory) into
// tensor memory: 4 columns, replicated into all four 32-lane quarters.
__device__ __forceinline__ void tmem_copy_sf(uint32_t taddr, uint64_t src_desc)
{
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(src_desc) : "memory");
}

// ---- warp-wide issue: the whole (converged) warp executes these; one
// elected lane (the lowest active lane, the same in every call) issues.
// Issuing tcgen05 and TMA instructions from a converged warp lets them
// pipeline; from a lone lane of a diverged warp each one stalls the issuer
// for roughly the instruction's execution time.
__device__ __forceinline__ void mma_mxf4nvf4_warp(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                  uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate)
{
    asm volatile(
        "{\n .reg .pred p, e;\n .reg .b32 r;\n"
        " setp.ne.b32 p, %6, 0;\n"
        " elect.sync r|e, 0xffffffff;\n"
        " @e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n"
        "}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tmem_copy_sf_warp(uint32_t taddr, uint64_t src_desc)
{
    asm volatile(
        "{\n .reg .pred e;\n .reg .b32 r;\n elect.sync r|e, 0xffffffff;\n"
        " @e tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;\n}" ::"r"(taddr),
        "l"(src_desc)
        : "memory");
}

__device__ __forceinline__ void mma_commit_warp(uint32_t bar)
{
    asm volatile(
        "{\n .reg .pred e;\n .reg .b32 r;\n elect.sync r|e, 0xffffffff;\n"
        " @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx_warp(uint32_t bar, uint32_t bytes)
{
    asm volatile(
        "{\n .reg .pred e;\n .reg .b32 r;\n elect.sync r|e, 0xffffffff;\n"
        " @e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n}" ::"r"(bar),
        "r"(bytes)
        : "memory");
}

__device__ __forceinline__ void tma_load_2d_warp(uint32_t dst, const CUtensorMap* map, uint32_t bar, int32_t x,
                                                 int32_t y, uint64_t cache_hint)
{
    asm volatile(
        "{\n .reg .pred e;\n .reg .b32 r;\n elect.sync r|e, 0xffffffff;\n"
        " @e cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5;\n}" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "l"(cache_hint)
        : "memory");
}

__device__ __forceinline__ void bulk_load_warp(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar)
{
    asm volatile(
        "{\n .reg .pred e;\n .reg .b32 r;\n elect.sync r|e, 0xffffffff;\n"
        " @e cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n}" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Warp-wide waits.  The whole warp polls, converged: a vote makes each
// poll's outcome warp-uniform and a round of polls runs inside one asm block.
// A wait that leaves some lanes spinning while others idle (one lane polling
// for the warp) slows the tensor pipe's intake of the MMA-issuing warp, even
// from another sub-partition; a converged warp does not.  With kSleep the
// polls carry a suspend-time hint, so a warp waiting through a whole tile
// (the epilogue) mostly sleeps.  Between rounds the warp checks, uniformly,
// the CTA's abort flag and the time limit (see mbar_wait).
constexpr uint32_t kFastPolls = 256;
constexpr uint32_t kSleepPolls = 16;
constexpr uint32_t kSuspendHintNs = 20000;

template <bool kSleep>
__device__ __forceinline__ bool mbar_poll_warp(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    if (kSleep)
        asm volatile(
            "{\n .reg .pred p, q;\n .reg .u32 n;\n mov.u32 n, 0;\n"
            "POLL_%=:\n"
            " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %4;\n"
            " vote.sync.all.pred p, p, 0xffffffff;\n"
            " @p bra.uni DONE_%=;\n"
            " add.u32 n, n, 1;\n"
            " setp.lt.u32 q, n, %3;\n"
            " @q bra.uni POLL_%=;\n"
            "DONE_%=:\n"
            " selp.u32 %0, 1, 0, p;\n}"
            : "=r"(ok)
            : "r"(bar), "r"(parity), "n"(kSleepPolls), "r"(kSuspendHintNs)
            : "memory");
    else
        asm volatile(
            "{\n .reg .pred p, q;\n .reg .u32 n;\n mov.u32 n, 0;\n"
            "POLL_%=:\n"
            " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            " vote.sync.all.pred p, p, 0xffffffff;\n"
            " @p bra.uni DONE_%=;\n"
            " add.u32 n, n, 1;\n"
            " setp.lt.u32 q, n, %3;\n"
            " @q bra.uni POLL_%=;\n"
            "DONE_%=:\n"
            " selp.u32 %0, 1, 0, p;\n}"
            : "=r"(ok)
            : "r"(bar), "r"(parity), "n"(kFastPolls)
            : "memory");
    return ok != 0;
}

// As mbar_poll_warp, with cluster-scope acquire (phases completed by the
// other CTA of the pair).
template <bool kSleep>
__device__ __forceinline__ bool mbar_poll_cluster_warp(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    if (kSleep)
        asm volatile(
            "{\n .reg .pred p, q;\n .reg .u32 n;\n mov.u32 n, 0;\n"
            "POLL_%=:\n"
            " mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %4;\n"
            " vote.sync.all.pred p, p, 0xffffffff;\n"
            " @p bra.uni DONE_%=;\n"
            " add.u32 n, n, 1;\n"
            " setp.lt.u32 q, n, %3;\n"
            " @q bra.uni POLL_%=;\n"
            "DONE_%=:\n"
            " selp.u32 %0, 1, 0, p;\n}"
            : "=r"(ok)
            : "r"(bar), "r"(parity), "n"(kSleepPolls), "r"(kSuspendHintNs)
            : "memory");
    else
        asm volatile(
            "{\n .reg .pred p, q;\n .reg .u32 n;\n mov.u32 n, 0;\n"
            "POLL_%=:\n"
            " mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
            " vote.sync.all.pred p, p, 0xffffffff;\n"
            " @p bra.uni DONE_%=;\n"
            " add.u32 n, n, 1;\n"
            " setp.lt.u32 q, n, %3;\n"
            " @q bra.uni POLL_%=;\n"
            "DONE_%=:\n"
            " selp.u32 %0, 1, 0, p;\n}"
            : "=r"(ok)
            : "r"(bar), "r"(parity), "n"(kFastPolls)
            : "memory");
    return ok != 0;
}

// Bounded warp-wide wait (converged throughout).  On giving up it raises the
// CTA's abort flag and records kErrTimeout*100 + site in the device status
// word (a timeout), or leaves them as they are (another warp gave up first);
// returns false.
template <bool kSleep = false>
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* status,
                                               int site)
{
    if (mbar_poll_warp<kSleep>(bar, parity)) return true;
    const uint64_t t0 = clock64();
    for (;;) {
        if (mbar_poll_warp<kSleep>(bar, parity)) return true;
        // every lane reads the flag and the clock; lane 0's verdict is the warp's
        int stop = *abort_flag ? 1 : ((uint64_t)(clock64() - t0) > kWaitLimitCycles ? 2 : 0);
        stop = __shfl_sync(0xffffffffu, stop, 0);
        if (stop != 0) {
            if (stop == 2 && (threadIdx.x & 31) == 0) {
                *abort_flag = 1;
                if (status) atomicCAS(status, 0, kErrTimeout * 100 + site);
            }
            __syncwarp();
            return false;
        }
    }
}

// As mbar_wait_warp, with cluster-scope acquire.
template <bool kSleep = false>
__device__ __forceinline__ bool mbar_wait_cluster_warp(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* status,
                                                       int site)
{
    if (mbar_poll_cluster_warp<kSleep>(bar, parity)) return true;
    const uint64_t t0 = clock64();
    for (;;) {
        if (mbar_poll_cluster_warp<kSleep>(bar, parity)) return true;
        // every lane reads the flag and the clock; lane 0's verdict is the warp's
        int stop = *abort_flag ? 1 : ((uint64_t)(clock64() - t0) > kWaitLimitCycles ? 2 : 0);
        stop = __shfl_sync(0xffffffffu, stop, 0);
        if (stop != 0) {
            if (stop == 2 && (threadIdx.x & 31) == 0) {
                *abort_flag = 1;
                if (status) atomicCAS(status, 0, kErrTimeout * 100 + site);
            }
            __syncwarp();
            return false;
        }
    }
}

// Bounded barrier of a group of warps (warp-converged calls): each warp
// arrives on a shared-memory counter and waits until it reaches target (the
// group's warp count for a first barrier, twice that for a second one);
// memory before the arrival is visible to every warp after the wait.  A warp
// gives up when the CTA's abort flag is raised or after the time limit (then
// recording a timeout and raising the flag itself); returns false then.
__device__ __forceinline__ bool epi_sync(int* counter, int target, volatile int* abort_flag, int* status, int site)
{
    int ok = 1;
    __syncwarp();
    if ((threadIdx.x & 31) == 0) {
        __threadfence_block();
        atomicAdd(counter, 1);
        const uint64_t t0 = clock64();
        while (*reinterpret_cast<volatile int*>(counter) < target) {
            if (*abort_flag) {
                ok = 0;
                break;
            }
            if ((uint64_t)(clock64() - t0) > kWaitLimitCycles) {
                *abort_flag = 1;
                if (status) atomicCAS(status, 0, kErrTimeout * 100 + site);
                ok = 0;
                break;
            }
        }
        __threadfence_block();
    }
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Arrive on an mbarrier once all tcgen05 operations issued so far by this
// thread have completed.
__device__ __forceinline__ void mma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// Load 32 consecutive fp32 columns of this warp's 32 tensor-memory lanes.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v)
{
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 32; i++) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_ld_wait()
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ------------------------------------------------------- clusters (2-SM)
__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Address of the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_cta(uint32_t addr, uint32_t rank)
{
    uint32_t out;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(addr), "r"(rank));
    return out;
}

__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Arrive on an mbarrier of another CTA of the cluster (cluster-scope release).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// 2-SM (cta_group::2) tensor-core operations: issued by the pair's even CTA
// for both CTAs; operands sit at the same shared/tensor-memory addresses in
// both.  The whole (converged) warp executes these; one lane issues.
__device__ __forceinline__ void tmem_alloc2(uint32_t dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish2()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc2(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void mma2_mxf4nvf4_warp(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                   uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate)
{
    asm volatile(
        "{\n .reg .pred p, e;\n .reg .b32 r;\n"
        " setp.ne.b32 p, %6, 0;\n"
        " elect.sync r|e, 0xffffffff;\n"
        " @e tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n"
        "}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tmem_copy_sf2_warp(uint32_t taddr, uint64_t src_desc)
{
    asm volatile(
        "{\n .reg .pred e;\n .reg .b32 r;\n elect.sync r|e, 0xffffffff;\n"
        " @e tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;\n}" ::"r"(taddr),
        "l"(src_desc)
        : "memory");
}

// Arrive on the mbarrier at offset `bar` of every CTA in `cta_mask` once all
// 2-SM tensor-core operations issued so far have completed.
__device__ __forceinline__ void mma_commit2_mc_warp(uint32_t bar, uint16_t cta_mask)
{
    asm volatile(
        "{\n .reg .pred e;\n .reg .b32 r;\n elect.sync r|e, 0xffffffff;\n"
        " @e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n}" ::"r"(
            bar),
        "h"(cta_mask)
        : "memory");
}

// ------------------------------------------------- fused stage issue
// One full K stage (4 K-steps of 64): its 12 scale-tile copies shared ->
// tensor memory (A, B rows 0-127, B rows 128-255 per K-step), its 4 MMAs
// and the commit that frees the stage, all from one asm block with a single
// elect.sync.  The warp stays converged from the first instruction to the
// last: issuing each tensor-core instruction from its own elected block, or
// any branch between them, slows the tensor pipe's intake.
//   acc: accumulator (tensor memory)     sfc: this stage's first scale column
//   f_lo / sf_hi: scale-tile descriptor of the stage (16-byte units in lo)
//   a_lo / b_lo / sw_hi: A and B code descriptors of the stage
//   acc0: accumulate into acc for the first K-step (0 = overwrite)
//   bar: mbarrier the commit arrives on
// Layout assumed: scale tiles of one K-step 512 B apart, the B tiles at
// +2048 and +4096 bytes; code K-steps 32 bytes apart; scale columns per
// K-step: A at +0, B rows 0-127 at +4, B rows 128-255 at +8, 12 per K-step.
__device__ __forceinline__ void stage_issue_1sm(uint32_t acc, uint32_t sfc, uint32_t f_lo, uint32_t sf_hi,
                                                uint32_t a_lo, uint32_t b_lo, uint32_t sw_hi, uint32_t idesc,
                                                uint32_t acc0, uint32_t bar)
{
    asm volatile(
        "{\n"
        " .reg .pred e, p, pt;\n"
        " .reg .b32 r, t, lo;\n"
        " .reg .b64 d, da, db;\n"
        " elect.sync r|e, 0xffffffff;\n"
        " setp.ne.b32 p, %8, 0;\n"
        " setp.eq.b32 pt, 0, 0;\n"
        " add.u32 t, %1, 0; add.u32 lo, %2, 0; mov.b64 d, {lo, %3};\n"
        " @e tcgen05.cp.cta_group::1.32x128b.warpx4 [t], d;\n"
        " add.u32 t, %1, 4; add.u32 lo, %2, 128; mov.b64 d, {lo, %3};\n"
        " @e tcgen05.cp.cta_group::1.32x128b.warpx4 [t], d;\n"
        " add.u32 t, %1, 8; add.u32 lo, %2, 256; mov.b64 d, {lo, %3};\n"
        " @e tcgen05.cp.cta_group::1.32x128b.warpx4 [t], d;\n"
        " add.u32 t, %1, 12; add.u32 lo, %2, 32; mov.b64 d, {lo, %3};\n"
        " @e tcgen05.cp.cta_group::1.32x128b.warpx4 [t], d;\n"
        " add.u32 t, %1, 16; add.u32 lo, %2, 160; mov.b64 d, {lo, %3};\n"
        " @e tcgen05.cp.cta_group::1.32x128b.warpx4 [t], d;\n"
        " add.u32 t, %1, 20; add.u32 lo, %2, 288; mov.b64 d, {lo, %3};\n"
        " @e tcgen05.cp.cta_group::1.32x128b.warpx4 [t], d;\n"
        " add.u32 t, %1, 24; add.u32 lo, %2, 64; mov.b64 d, {lo, %3};\n"
        " @e tcgen05.cp.cta_group::1.32x128b.warpx4 [t], d;\n"
        " add.u32 t, %1, 28; add.u32 lo, %2, 192; mov.b64 d, {lo, %3};\n"
        " @e tcgen05.cp.cta_group::1.32x128b.warpx4 [t], d;\n"
        " add.u32 t, %1, 32; add.u32 lo, %2, 320; mov.b64 d, {lo, %3};\n"
        " @e tcgen05.cp.cta_group::1.32x128b.warpx4 [t], d;\n"
        " add.u32 t, %1, 36; add.u32 lo, %2, 96; mov.b64 d, {lo, %3};\n"
        " @e tcgen05.cp.cta_group::1.32x128b.warpx4 [t], d;\n"
        " add.u32 t, %1, 40; add.u32 lo, %2, 224; mov.b64 d, {lo, %3};\n"
        " @e tcgen05.cp.cta_group::1.32x128b.warpx4 [t], d;\n"
        " add.u32 t, %1, 44; add.u32 lo, %2, 352; mov.b64 d, {lo, %3};\n"
        " @e tcgen05.cp.cta_group::1.32x128b.warpx4 [t], d;\n"
        " add.u32 lo, %4, 0; mov.b64 da, {lo, %6}; add.u32 lo, %5, 0; mov.b64 db, {lo, %6};\n"
        " add.u32 t, %1, 0; add.u32 r, %1, 4;\n"
        " @e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], da, db, %7, [t], [r], p;\n"
        " add.u32 lo, %4, 2; mov.b64 da, {lo, %6}; add.u32 lo, %5, 2; mov.b64 db, {lo, %6};\n"
        " add.u32 t, %1, 12; add.u32 r, %1, 16;\n"
        " @e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], da, db, %7, [t], [r], pt;\n"
        " add.u32 lo, %4, 4; mov.b64 da, {lo, %6}; add.u32 lo, %5, 4; mov.b64 db, {lo, %6};\n"
        " add.u32 t, %1, 24; add.u32 r, %1, 28;\n"
        " @e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], da, db, %7, [t], [r], pt;\n"
        " add.u32 lo, %4, 6; mov.b64 da, {lo, %6}; add.u32 lo, %5, 6; mov.b64 db, {lo, %6};\n"
        " add.u32 t, %1, 36; add.u32 r, %1, 40;\n"
        " @e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], da, db, %7, [t], [r], pt;\n"
        " @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%9];\n"
        "}\n"
        ::"r"(acc), "r"(sfc), "r"(f_lo), "r"(sf_hi), "r"(a_lo), "r"(b_lo), "r"(sw_hi), "r"(idesc), "r"(acc0),
        "r"(bar)
        : "memory");
}

// The same for an SM pair (cta_group::2): the copies and MMAs act on both
// CTAs' shared and tensor memory, and the commit arrives on `bar` in every
// CTA of `cta_mask`.
__device__ __forceinline__ void stage_issue_2sm(uint32_t acc, uint32_t sfc, uint32_t f_lo, uint32_t sf_hi,
                                                uint32_t a_lo, uint32_t b_lo, uint32_t sw_hi, uint32_t idesc,
                                                uint32_t acc0, uint32_t bar, uint16_t cta_mask)
{
    asm volatile(
        "{\n"
        " .reg .pred e, p, pt;\n"
        " .reg .b32 r, t, lo;\n"
        " .reg .b64 d, da, db;\n"
        " elect.sync r|e, 0xffffffff;\n"
        " setp.ne.b32 p, %8, 0;\n"
        " setp.eq.b32 pt, 0, 0;\n"
        " add.u32 t, %1, 0; add.u32 lo, %2, 0; mov.b64 d, {lo, %3};\n"
        " @e tcgen05.cp.cta_group::2.32x128b.warpx4 [t], d;\n"
        " add.u32 t, %1, 4; add.u32 lo, %2, 128; mov.b64 d, {lo, %3};\n"
        " @e tcgen05.cp.cta_group::2.32x128b.warpx4 [t], d;\n"
        " add.u32 t, %1, 8; add.u32 lo, %2, 256; mov.b64 d, {lo, %3};\n"
        " @e tcgen05.cp.cta_group::2.32x128b.warpx4 [t], d;\n"
        " add.u32 t, %1, 12; add.u32 lo, %2, 32; mov.b64 d, {lo, %3};\n"
        " @e tcgen05.cp.cta_group::2.32x128b.warpx4 [t], d;\n"
        " add.u32 t, %1, 16; add.u32 lo, %2, 160; mov.b64 d, {lo, %3};\n"
        " @e tcgen05.cp.cta_group::2.32x128b.warpx4 [t], d;\n"
        " add.u32 t, %1, 20; add.u32 lo, %2, 288; mov.b64 d, {lo, %3};\n"
        " @e tcgen05.cp.cta_group::2.32x128b.warpx4 [t], d;\n"
        " add.u32 t, %1, 24; add.u32 lo, %2, 64; mov.b64 d, {lo, %3};\n"
        " @e tcgen05.cp.cta_group::2.32x128b.warpx4 [t], d;\n"
        " add.u32 t, %1, 28; add.u32 lo, %2, 192; mov.b64 d, {lo, %3};\n"
        " @e tcgen05.cp.cta_group::2.32x128b.warpx4 [t], d;\n"
        " add.u32 t, %1, 32; add.u32 lo, %2, 320; mov.b64 d, {lo, %3};\n"
        " @e tcgen05.cp.cta_group::2.32x128b.warpx4 [t], d;\n"
        " add.u32 t, %1, 36; add.u32 lo, %2, 96; mov.b64 d, {lo, %3};\n"
        " @e tcgen05.cp.cta_group::2.32x128b.warpx4 [t], d;\n"
        " add.u32 t, %1, 40; add.u32 lo, %2, 224; mov.b64 d, {lo, %3};\n"
        " @e tcgen05.cp.cta_group::2.32x128b.warpx4 [t], d;\n"
        " add.u32 t, %1, 44; add.u32 lo, %2, 352; mov.b64 d, {lo, %3};\n"
        " @e tcgen05.cp.cta_group::2.32x128b.warpx4 [t], d;\n"
        " add.u32 lo, %4, 0; mov.b64 da, {lo, %6}; add.u32 lo, %5, 0; mov.b64 db, {lo, %6};\n"
        " add.u32 t, %1, 0; add.u32 r, %1, 4;\n"
        " @e tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], da, db, %7, [t], [r], p;\n"
        " add.u32 lo, %4, 2; mov.b64 da, {lo, %6}; add.u32 lo, %5, 2; mov.b64 db, {lo, %6};\n"
        " add.u32 t, %1, 12; add.u32 r, %1, 16;\n"
        " @e tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], da, db, %7, [t], [r], pt;\n"
        " add.u32 lo, %4, 4; mov.b64 da, {lo, %6}; add.u32 lo, %5, 4; mov.b64 db, {lo, %6};\n"
        " add.u32 t, %1, 24; add.u32 r, %1, 28;\n"
        " @e tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], da, db, %7, [t], [r], pt;\n"
        " add.u32 lo, %4, 6; mov.b64 da, {lo, %6}; add.u32 lo, %5, 6; mov.b64 db, {lo, %6};\n"
        " add.u32 t, %1, 36; add.u32 r, %1, 40;\n"
        " @e tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], da, db, %7, [t], [r], pt;\n"
        " @e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%9], %10;\n"
        "}\n"
        ::"r"(acc), "r"(sfc), "r"(f_lo), "r"(sf_hi), "r"(a_lo), "r"(b_lo), "r"(sw_hi), "r"(idesc), "r"(acc0),
        "r"(bar), "h"(cta_mask)
        : "memory");
}

// ---------------------------------------------------- FP4 / FP8 convert
// Eight fp32 values -> eight E2M1 codes (round-to-nearest-even, saturating),
// v[0] in the lowest nibble.
__device__ __forceinline__ uint32_t cvt_e2m1x8(const float* v)
{
    uint32_t out;
    asm volatile(
        "{\n .reg .b8 b0, b1, b2, b3;\n"
        " cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
        " cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
        " cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n"
        " cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
        " mov.b32 %0, {b0, b1, b2, b3};\n}"
        : "=r"(out)
        : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
    return out;
}

// Non-negative fp32 -> E4M3 byte (round-to-nearest-even, saturating at 448).
__device__ __forceinline__ uint32_t cvt_e4m3(float s)
{
    uint16_t out;
    asm volatile("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(out) : "f"(0.0f), "f"(s));
    return out & 0xFFu;
}

// E4M3 byte -> fp32 (exact).
__device__ __forceinline__ float e4m3_to_f32(uint32_t b)
{
    uint32_t h2;
    uint16_t in = (uint16_t)(b & 0xFFu);
    asm volatile("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
    return __half2float(__ushort_as_half((uint16_t)(h2 & 0xFFFFu)));
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float bf16_round(float v)
{
    return __bfloat162float(__float2bfloat16_rn(v));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t a = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
    uint32_t b = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
    return a | (b << 16);
}

// Two binary32 values -> bf16x2, each rounded to nearest even (lo in the
// low half): pack_bf16x2 in one instruction.
__device__ __forceinline__ uint32_t cvt_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Sum of two bf16x2, each half rounded to nearest even once.  For bf16
// operands this equals rounding their binary32 sum to bf16: that sum is
// exact when the exponents differ by at most 15, and otherwise the smaller
// operand lies far below half an ulp of the larger, which both roundings
// then return.
__device__ __forceinline__ uint32_t add_bf16x2(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Byte offset of scale (row r, scale column c) in the 128x4-tile layout.
__device__ __forceinline__ int64_t sf_offset(int64_t r, int64_t c, int64_t kb_pad)
{
    return ((r >> 7) * (kb_pad >> 2) + (c >> 2)) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4 + (c & 3);
}

// Correctly rounded binary32 quotient a / b for many a and one b > 0
// (normal, with a / b far from overflow and underflow), from the correctly
// rounded reciprocal y = RN(1/b): q0 = RN(a*y), the remainder
// r = a - b*q0 is exact in one FMA, and RN(q0 + r*y) = RN(a/b)
// (P. Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Dev. 34(1), 1990: quotient refinement
// with a correctly rounded reciprocal).
__device__ __forceinline__ float div_by_recip(float a, float b, float y)
{
    const float q0 = __fmul_rn(a, y);
    // t = q0*b - a, the negated remainder, so that the final sum keeps the
    // sign of a zero quotient: a = -0 gives q0 = -0, t = +0, -t*y + q0 = -0
    const float t = __fmaf_rn(q0, b, -a);
    return __fmaf_rn(-t, y, q0);
}

// Quantize one 16-element block held as two halves of 8 in lanes l, l^1:
// shared helper so every kernel takes bit-identical decisions.
//   v: this lane's 8 values; g: global scale.  Returns this lane's 8 codes
//   (32 bits) and writes the block's scale byte to *sc.
// Arithmetic (binary32, one rounding per step): d = 6*g, s = E4M3(amax16/d),
// den = E4M3val(s)*g, code_i = E2M1(v_i/den).
__device__ __forceinline__ uint32_t quant_half_block(const float* v, float g, float amax16, uint32_t* sc_out)
{
    // d, its reciprocal: the same for every block of a tensor (hoisted out of
    // the callers' loops); amax16 / d by the quotient refinement above
    // (a quotient below 2^-126 would round to a zero scale either way)
    const float d = __fmul_rn(6.0f, g);
    const float s_raw = div_by_recip(amax16, d, __frcp_rn(d));
    const uint32_t sc = cvt_e4m3(s_raw);
    *sc_out = sc;
    if (sc == 0) return 0u;
    const float den = __fmul_rn(e4m3_to_f32(sc), g);
    const float y = __frcp_rn(den);
    float q[8];
#pragma unroll
    for (int i = 0; i < 8; i++) q[i] = div_by_recip(v[i], den, y);
    return cvt_e2m1x8(q);
}

}  // namespace nvfp4
