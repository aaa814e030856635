// Inline-PTX building blocks for sm_103a: mbarriers, TMA (cp.async.bulk.tensor),
// tcgen05 (TMEM allocation, MMA, copies, loads) and the descriptors they take.
#pragma once

#include <cuda.h>  // CUtensorMap (type only; the driver is reached through the runtime)
#include <stdint.h>

namespace dg {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ----------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar_addr, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(bar_addr), "r"(parity)
        : "memory");
    return ok != 0;
}

// As mbar_try_wait, with cluster-scope acquire: for barriers that the other CTA
// of a cluster arrives on after its own writes.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar_addr, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(bar_addr), "r"(parity)
        : "memory");
    return ok != 0;
}

// Per-CTA control block for bounded waits: when any wait runs out it raises
// `abort` (shared memory) so every other role of the CTA stops waiting too,
// and records the failure in the caller's status word.
struct WaitCtl {
    volatile int *abort;   // shared-memory flag
    int32_t *status;       // device status word or nullptr
    uint64_t timeout_ns;
};

template <bool CLUSTER = false>
static __device__ __noinline__ bool mbar_wait_slow(uint32_t bar_addr, uint32_t parity, WaitCtl ctl,
                                            int32_t timeout_flag) {
    const uint64_t t0 = global_timer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 64; ++i)
            if (CLUSTER ? mbar_try_wait_cluster(bar_addr, parity) : mbar_try_wait(bar_addr, parity))
                return true;
        if (*ctl.abort) return false;
        if (global_timer_ns() - t0 > ctl.timeout_ns) {
            *ctl.abort = 1;
            if (ctl.status) atomicOr(ctl.status, timeout_flag);
            return false;
        }
    }
}

// Wait for the phase of `bar` with the given parity to complete.  Returns false
// (and the CTA is aborting) if the time limit ran out or another role aborted.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, const WaitCtl &ctl,
                                          int32_t timeout_flag) {
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait(a, parity)) return true;
    return mbar_wait_slow(a, parity, ctl, timeout_flag);
}

// Waits for copies already issued to land whatever the abort flag says (a CTA
// must not leave while a copy into its shared memory is in flight); gives up
// after the time limit.
__device__ __forceinline__ void mbar_wait_drain(uint64_t *bar, uint32_t parity, const WaitCtl &ctl) {
    const uint32_t a = smem_u32(bar);
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(a, parity))
        if (global_timer_ns() - t0 > ctl.timeout_ns) return;
}

// As mbar_wait, with cluster-scope acquire (arrivals come from the peer CTA).
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t *bar, uint32_t parity, const WaitCtl &ctl,
                                                  int32_t timeout_flag) {
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait_cluster(a, parity)) return true;
    return mbar_wait_slow<true>(a, parity, ctl, timeout_flag);
}

// One lane of the converged warp (the lowest active lane).  The issuing
// loops of the producer and MMA warps run on all 32 lanes, so their
// warp-uniform operands (descriptors, coordinates, TMEM addresses) stay in
// uniform registers, and only the issue itself is guarded by this election.
__device__ __forceinline__ bool elect_one() {
    uint32_t pred;
    asm volatile(
        "{\n\t.reg .pred P;\n\t"
        "elect.sync _|P, 0xffffffff;\n\t"
        "selp.u32 %0, 1, 0, P;\n\t}\n"
        : "=r"(pred));
    return pred != 0;
}

// Warp-uniform outcome of a bounded wait that every lane performs.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t *bar, uint32_t parity, const WaitCtl &ctl,
                                               int32_t timeout_flag) {
    return __all_sync(0xFFFFFFFFu, mbar_wait(bar, parity, ctl, timeout_flag));
}

__device__ __forceinline__ bool mbar_wait_cluster_warp(uint64_t *bar, uint32_t parity, const WaitCtl &ctl,
                                                       int32_t timeout_flag) {
    return __all_sync(0xFFFFFFFFu, mbar_wait_cluster(bar, parity, ctl, timeout_flag));
}

// ----------------------------------------------------------------- clusters

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_nctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}

// Address of the same shared-memory location in the CTA of cluster rank `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

// Arrive on a peer CTA's mbarrier with the default (release, CTA-scope)
// semantics.  For a CTA pair's hand-offs where what the arrival announces is
// local to the arriving CTA's SM (its own shared memory already made visible to
// the async proxy by fence.proxy.async, or its own TMEM reads completed by
// tcgen05.wait::ld and ordered by tcgen05.fence::before_thread_sync) and the
// peer only issues the tcgen05 operation that later touches that SM's storage.
// About 80 cycles instead of 400 or more for the cluster-scope release, which
// waits for this thread's outstanding memory traffic.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Programmatic dependent launch: let the next grid in the stream start launching
// (its CTAs run up to their own wait), and wait until the grids this one depends
// on have completed with their memory visible.
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Named CTA barrier `id` (1..15) over `count` threads: wait, or only arrive.
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t count) {
    asm volatile("barrier.cta.sync.aligned %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void named_bar_arrive(uint32_t id, uint32_t count) {
    asm volatile("barrier.cta.arrive.aligned %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// All threads of all CTAs of the cluster (release/acquire ordering).
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ----------------------------------------------------------------- proxies

// Make generic-proxy writes to shared memory visible to the async proxy
// (TMA stores, tcgen05.cp, tcgen05.mma operand reads).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ----------------------------------------------------------------- TMA

// Fetch [p, p + bytes) from global memory into L2 (no data returned; p and bytes
// multiples of 16).  One request for a whole row segment keeps the DRAM reads
// long and contiguous.
__device__ __forceinline__ void prefetch_l2_bulk(const void *p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(p)), "r"(bytes)
                 : "memory");
}

// 32-byte global load (p 32-byte aligned), cached at L2 only.
// L2 prefetch of the 128-byte line holding p, from this thread.
__device__ __forceinline__ void prefetch_l2_line(const void *p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<uint64_t>(p)) : "memory");
}

__device__ __forceinline__ void ld_global_cg_v8(const void *p, uint32_t (&r)[8]) {
    asm volatile("ld.global.cg.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "l"(reinterpret_cast<uint64_t>(p)));
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(void *smem_dst, const CUtensorMap *map, uint64_t *bar,
                                            int32_t x, int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// TMA load into this CTA's shared memory whose completion is counted on an
// mbarrier of either CTA of the pair (cluster address `bar_cluster`).
__device__ __forceinline__ void tma_load_2d_pair(void *smem_dst, const CUtensorMap *map,
                                                 uint32_t bar_cluster, int32_t x, int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster)
        : "memory");
}

// 3-D tiled load: box {x extent, y extent, z extent} lands as z slabs of y rows.
// With the K-blocked operand view (x = K within a 128-K block, y = row, z =
// K-block) one load fills the consecutive stages of a ring slot.
__device__ __forceinline__ void tma_load_3d(void *smem_dst, const CUtensorMap *map, uint64_t *bar,
                                            int32_t x, int32_t y, int32_t z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

// As tma_load_3d, completing on an mbarrier given by its cluster address
// (the leader CTA's barrier in a CTA pair).
__device__ __forceinline__ void tma_load_3d_pair(void *smem_dst, const CUtensorMap *map,
                                                 uint32_t bar_cluster, int32_t x, int32_t y, int32_t z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar_cluster)
        : "memory");
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, const void *smem_src,
                                             int32_t x, int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(x), "r"(y), "r"(smem_u32(smem_src))
        : "memory");
}

// TMA reduce: the box in shared memory is added element-wise to the tensor in
// global memory (the addition is done at L2, in the tensor map's type; FP32
// adds round to nearest even).
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap *map, const void *smem_src, int32_t x,
                                                  int32_t y) {
    asm volatile(
        "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(x), "r"(y), "r"(smem_u32(smem_src))
        : "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

template <int N>
__device__ __forceinline__ void bulk_wait_group() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// ----------------------------------------------------------------- cp.async (plain asynchronous copies)

// Copies 4 bytes from global to shared memory asynchronously; a src_bytes of 0
// reads nothing and writes zeros.
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

// At most N of this thread's most recent cp.async groups are still in flight.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// cp_async_wait with a run-time count (0..7; larger counts wait for 7).
__device__ __forceinline__ void cp_async_wait_dyn(int n) {
    switch (n) {
        case 0: cp_async_wait<0>(); break;
        case 1: cp_async_wait<1>(); break;
        case 2: cp_async_wait<2>(); break;
        case 3: cp_async_wait<3>(); break;
        case 4: cp_async_wait<4>(); break;
        case 5: cp_async_wait<5>(); break;
        case 6: cp_async_wait<6>(); break;
        default: cp_async_wait<7>(); break;
    }
}

// ----------------------------------------------------------------- tcgen05

// TMEM allocation: one full warp executes these.  The allocated base address
// (lane 0, first column) is written to `dst` in shared memory.
__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrive (once) on `bar` when every tcgen05 async operation this thread has
// issued so far (mma, cp) has completed.
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// ---- CTA-pair (cta_group::2) forms: the pair's two SMs act as one MMA unit.
// Allocation is collective (one warp in each CTA); the leader issues the MMAs,
// which read A rows 0-127 / B rows 0..N/2-1 from the leader's shared memory and
// A rows 128-255 / B rows N/2..N-1 from the peer's (same offsets), and write
// each CTA's 128 rows of D into its own TMEM.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t *dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst)),
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

// Arrive on the mbarrier at this offset in every CTA of `cta_mask` when all
// tcgen05 operations this thread issued so far have completed.
__device__ __forceinline__ void tc_commit_pair(uint64_t *bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(cta_mask)
        : "memory");
}

__device__ __forceinline__ void tc_mma_mxf8_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                 uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                                 uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;\n\t}\n" ::"r"(
            d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
        : "memory");
}

// Copies each CTA's own shared-memory source into its own TMEM (issued by the leader).
__device__ __forceinline__ void tc_cp_32x128b_warpx4_pair(uint32_t taddr, uint64_t src_desc) {
    asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(src_desc)
                 : "memory");
}

// 64 rows of 16 bytes: rows 0-31 to lanes 0-31 of quadrants 0 and 1, rows 32-63
// to quadrants 2 and 3 (each CTA of the pair, from its own shared memory).
__device__ __forceinline__ void tc_cp_64x128b_warpx2_01_23_pair(uint32_t taddr, uint64_t src_desc) {
    asm volatile("tcgen05.cp.cta_group::2.64x128b.warpx2::01_23 [%0], %1;" ::"r"(taddr), "l"(src_desc)
                 : "memory");
}

// D(tmem) (+)= A(smem) * B(smem)^T with UE8M0 block scales read from TMEM,
// one scale per 32 K-elements of each row of A and of B.
__device__ __forceinline__ void tc_mma_mxf8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;\n\t}\n" ::"r"(
            d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
        : "memory");
}

// D(tmem) (+)= A(smem) * B(smem)^T without scales (FP8 inputs, FP32 accumulate).
__device__ __forceinline__ void tc_mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Copy 32 rows x 128 bits from shared memory into TMEM, replicated into all
// four 32-lane sub-partitions.
__device__ __forceinline__ void tc_cp_32x128b_warpx4(uint32_t taddr, uint64_t src_desc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(src_desc)
                 : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 32 lanes x 16 consecutive 32-bit columns: thread t of the warp receives
// lane (base lane + t), columns col..col+15.
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

// Ties the registers produced by tcgen05.ld to the wait that makes them valid.
__device__ __forceinline__ void reg_fence16(uint32_t (&r)[16]) {
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])::"memory");
}

// ----------------------------------------------------------------- descriptors

// Shared-memory matrix descriptor (tcgen05 form): start address, leading and
// stride byte offsets (all >> 4), the fixed version field (bit 46), base
// offset 0, and the swizzle mode in bits 61-63.
enum : uint32_t { kSwizzleNone = 0, kSwizzle128B = 2, kSwizzle64B = 4, kSwizzle32B = 6 };

__device__ __forceinline__ uint64_t make_smem_desc(uint32_t saddr, uint32_t lbo_bytes,
                                                   uint32_t sbo_bytes, uint32_t swizzle) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(swizzle & 0x7u) << 61;
    return d;
}

// K-major operand tile whose rows are 128 bytes (128 FP8 K-elements), written
// by TMA with 128-byte swizzle: 8-row groups are 1024 bytes apart.
__device__ __forceinline__ uint64_t make_desc_kmajor_sw128(uint32_t saddr) {
    return make_smem_desc(saddr, 16, 1024, kSwizzle128B);
}

// Source of a 32x128b tcgen05.cp: 32 rows of 16 bytes, contiguous, no
// swizzle (8-row core matrices 128 bytes apart).
__device__ __forceinline__ uint64_t make_desc_sf_32x128b(uint32_t saddr) {
    return make_smem_desc(saddr, 0, 128, kSwizzleNone);
}

// Instruction descriptor, block-scaled FP8 x FP8 (E4M3 both), FP32 accumulate,
// K-major A and B, UE8M0 scales.  sf_id_a / sf_id_b choose which byte of the
// 32-bit TMEM scale word is used.
__host__ __device__ constexpr uint32_t make_idesc_mxf8(uint32_t m, uint32_t n, uint32_t sf_id_a,
                                                       uint32_t sf_id_b) {
    return ((sf_id_b & 3u) << 4)      // B scale-factor byte
           | (0u << 7)                // A format: E4M3
           | (0u << 10)               // B format: E4M3
           | ((n >> 3) << 17)         // N / 8
           | (1u << 23)               // scale format: UE8M0
           | ((m >> 4) << 24)         // M / 16
           | ((sf_id_a & 3u) << 29);  // A scale-factor byte
}

// Instruction descriptor, FP8 x FP8 (E4M3 both) without scales, FP32 accumulate.
__host__ __device__ constexpr uint32_t make_idesc_f8(uint32_t m, uint32_t n) {
    return (1u << 4)            // D format: FP32
           | (0u << 7) | (0u << 10) | ((n >> 3) << 17) | ((m >> 4) << 24);
}

}  // namespace dg
