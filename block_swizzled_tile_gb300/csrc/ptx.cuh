// Device primitives for sm_103a written as inline PTX: mbarriers with bounded
// waits, TMA tile loads, cp.async, and the tcgen05 family (TMEM allocation,
// MMA, commit, TMEM loads, shared->TMEM copies).
//
// The buffered mainloop these serve is the GB300 counterpart of the
// multi-buffered L1/L0 pipelines of "Block Dispatch Policies"
// (MmadAtlasA2Pingpong / MmadAtlasA2Preload / MmadAtlasA2PreloadAsync):
// there, buffers are handed between the copy and the cube unit; here shared
// memory stages are handed between a TMA producer and the tcgen05 issuer by
// mbarriers, and TMEM accumulators between the issuer and the epilogue.
#pragma once
#include <cstdint>
#include <cuda.h>

namespace bst {

// ----------------------------------------------------------------- misc ----

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// 1 in exactly one lane of the (converged) warp -- the lowest active one, so
// lane 0 of a full warp -- 0 elsewhere.  The MMA loops run on the whole warp
// and issue from the elected lane: a tcgen05.mma group issued by a lone lane
// of a diverged warp and followed by an mbarrier wait costs about 320 ns per
// k-block on sm_103a whatever its size, against about 200 ns (128 x 128
// pieces) to 260 ns (128 x 256, the tensor time) from a converged warp.
__device__ __forceinline__ uint32_t elect_one() {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .b32 r;\n\t.reg .pred p;\n\t"
        "elect.sync r|p, 0xffffffff;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok));
    return ok;
}

__device__ __forceinline__ uint32_t lane_id() {
    uint32_t l;
    asm volatile("mov.u32 %0, %laneid;" : "=r"(l));
    return l;
}

// ------------------------------------------------------------- mbarrier ----

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// makes barrier initialisation visible to the async proxy (TMA, tcgen05)
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// `count` arrivals at once (on behalf of threads that take no part in this phase)
__device__ __forceinline__ void mbar_arrive_cnt(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

// adds `bytes` to the barrier's expected transaction count without arriving
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar_addr, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar_addr), "r"(parity)
        : "memory");
    return ok != 0;
}

// try_wait with a suspend-time hint: a thread whose phase is not complete is
// parked (for at most hint_ns) instead of re-polling, and wakes when the phase
// completes
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar_addr, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar_addr), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Error word layout (one per device, in the library's own __device__ memory).
enum : uint32_t {
    kErrTimeout = 1u,       // a bounded wait gave up
    kErrGroups = 2u,        // grouped sizes inconsistent with total rows
    kErrTraceOverflow = 4u, // more tasks than the debug map buffer holds
};

struct WaitCtl {
    volatile int* abort_flag;   // shared: set once any wait of this CTA gave up
    uint64_t timeout_ns;
    uint32_t* err_word;         // global: [0] flags, [1] block, [2] where
};

// Waits for the phase with parity `parity` of `bar` to complete.  Gives up
// after ctl.timeout_ns (measured on %globaltimer) or a hard iteration cap,
// raising the CTA's abort flag and recording the failure; returns false then,
// and also as soon as another role of the CTA has aborted.
static __device__ __noinline__ bool mbar_wait_slow(uint64_t* bar, uint32_t parity, WaitCtl ctl, uint32_t where) {
    const uint32_t a = smem_u32(bar);
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1; it < (1u << 24); ++it) {
        if (mbar_try_wait_sleep(a, parity, 20000u)) return true;
        if (*ctl.abort_flag) return false;
        if (globaltimer_ns() - t0 > ctl.timeout_ns) break;
    }
    *ctl.abort_flag = 1;
    if (atomicOr(&ctl.err_word[0], kErrTimeout) == 0) {
        ctl.err_word[1] = blockIdx.x;
        ctl.err_word[2] = where;
    }
    return false;
}

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, WaitCtl ctl, uint32_t where) {
    const uint32_t a = smem_u32(bar);
#pragma unroll 1
    for (uint32_t i = 0; i < 16; ++i)
        if (mbar_try_wait(a, parity)) return true;
    return mbar_wait_slow(bar, parity, ctl, where);
}

// The same wait with acquire semantics at cluster scope: used where the
// phase is completed by a release arrival of another CTA of the cluster
// whose shared-memory writes the waiting side then consumes.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar_addr, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar_addr), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ void fence_acq_rel_cluster() { asm volatile("fence.acq_rel.cluster;" ::: "memory"); }

__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, WaitCtl ctl, uint32_t where) {
    const uint32_t a = smem_u32(bar);
#pragma unroll 1
    for (uint32_t i = 0; i < 16; ++i)
        if (mbar_try_wait_cluster(a, parity)) return true;
    // the slow path observes the phase with cta-scope acquire; the fence
    // extends it to the cluster
    const bool ok = mbar_wait_slow(bar, parity, ctl, where);
    fence_acq_rel_cluster();
    return ok;
}

// Wait used only while shutting down after an abort: ignores the abort flag,
// still gives up after the time limit.
static __device__ __noinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
    const uint32_t a = smem_u32(bar);
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 0; it < (1u << 24); ++it) {
        if (mbar_try_wait_sleep(a, parity, 20000u)) return true;
        if (globaltimer_ns() - t0 > timeout_ns) return false;
    }
    return false;
}

// ------------------------------------------- programmatic dependent launch --

// Waits until every grid this one depends on (launched before it on the
// stream with programmatic serialization) has completed and its memory is
// visible; a no-op when the kernel was launched without that attribute.
// Nothing before it may touch global memory written by earlier work.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Lets the next grid on the stream be scheduled (it still waits for this one
// to complete before it touches memory).
__device__ __forceinline__ void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ------------------------------------------------------------------ TMA ----

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* m) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// Tensor maps rewritten on the device (grouped slice-K: one map per group,
// its base moved to the group's first K element and its K extent cut to the
// group's size, so TMA fills the group's ragged last k-block with zeros).
// The map lives in global memory; the writer releases it to the tensor-map
// proxy and every thread that issues copies with it acquires it first.
__device__ __forceinline__ void tmap_replace_address(void* gmap, uint64_t addr) {
    asm volatile("tensormap.replace.tile.global_address.global.b1024.b64 [%0], %1;" ::"l"(gmap), "l"(addr) : "memory");
}
template <int ORD>
__device__ __forceinline__ void tmap_replace_dim(void* gmap, uint32_t extent) {
    asm volatile("tensormap.replace.tile.global_dim.global.b1024.b32 [%0], %1, %2;" ::"l"(gmap), "n"(ORD),
                 "r"(extent)
                 : "memory");
}
__device__ __forceinline__ void tmap_release() {
    asm volatile("fence.proxy.tensormap::generic.release.gpu;" ::: "memory");
}
__device__ __forceinline__ void tmap_acquire(const void* gmap) {
    asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(gmap) : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* m, uint64_t* bar, int32_t x, int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(x), "r"(y)
        );
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* m, uint64_t* bar, int32_t x, int32_t y,
                                            int32_t z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
        );
}

// orders this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA / tcgen05) accesses
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// brings the 128-byte line holding `p` into L2 (no register result, no TMA)
__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// ------------------------------------------------------------- cp.async ----

// 4-byte global->shared copy; src_bytes 0 writes zeros instead of reading
__device__ __forceinline__ void cp_async_4(void* dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
                 );
}

// V-byte (4, 8 or 16) asynchronous copy into shared memory; bytes past
// src_bytes (<= V) are zero-filled, and with src_bytes = 0 nothing is read
template <uint32_t V>
__device__ __forceinline__ void cp_async_v(void* dst, const void* src, uint32_t src_bytes) {
    static_assert(V == 4 || V == 8 || V == 16, "cp.async size");
    asm volatile("cp.async.ca.shared.global [%0], [%1], %2, %3;" ::"r"(smem_u32(dst)), "l"(src), "n"(V),
                 "r"(src_bytes));
}

// waits until every cp.async issued by this thread has landed
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// the barrier receives one arrival (counted in its expected count) when all
// earlier cp.async of this thread have landed
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
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

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor (tcgen05 "matrix descriptor"): start
// address, leading- and stride-dimension byte offsets (all >> 4), the fixed
// version bits 46-48 = 0b001, base offset 0, and the swizzle mode in bits
// 61-63 (0 = none, 2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes,
                                              uint32_t swizzle) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(swizzle & 7u) << 61;
    return d;
}
constexpr uint32_t kSwizzleNone = 0;
constexpr uint32_t kSwizzle128B = 2;

// Instruction descriptor for kind::f16 (fp16/bf16 in, fp32 accumulator):
// bits 4-5 D format (1 = f32), 7-9 / 10-12 A / B format (0 = f16, 1 = bf16),
// 15 / 16 A / B major (0 = K, 1 = MN), 17-22 N >> 3, 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_f16(uint32_t ab_fmt, uint32_t a_mn, uint32_t b_mn, uint32_t M,
                                                 uint32_t N) {
    return (1u << 4) | (ab_fmt << 7) | (ab_fmt << 10) | (a_mn << 15) | (b_mn << 16) | ((N >> 3) << 17) |
           ((M >> 4) << 24);
}

// Instruction descriptor for kind::mxf8f6f4 with block scaling: bits 4-5
// scale-factor byte of B, 7-9 / 10-12 A / B format (0 = e4m3), 17-22 N >> 3,
// 23 scale type (1 = UE8M0), 24-28 M >> 4, 29-30 scale-factor byte of A.
__host__ __device__ constexpr uint32_t idesc_mxf8(uint32_t M, uint32_t N, uint32_t sf_id) {
    return (sf_id << 4) | (0u << 7) | (0u << 10) | ((N >> 3) << 17) | (1u << 23) | ((M >> 4) << 24) |
           (sf_id << 29);
}

__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        );
}

__device__ __forceinline__ void umma_mxf8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        );
}

// arrive once on `bar` when every tcgen05 operation issued so far by this
// thread has completed
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 );
}

// 32 lanes x 128 bits from shared memory into TMEM, replicated to all four
// 32-lane quarters of the accumulator
__device__ __forceinline__ void tmem_cp_32x128b_warpx4(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc));
}

// each thread of the warp reads 32 consecutive 32-bit columns of its own lane;
// the wait for completion sits in the same asm statement so that no use of the
// destination registers can be scheduled before the data has arrived
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// the same for 16 consecutive columns
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// each thread writes 32 consecutive 32-bit columns of its own lane; waits
// until the write is done (a later tcgen05.ld of the columns sees it)
__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n\t"
        "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
        "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
        "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

// ------------------------------------------------- CTA pairs (clusters) ----
// Two CTAs of a cluster of 2 form a CTA pair whose tcgen05 MMA (cta_group::2)
// reads A rows 0-127 and half of B from the leader's (rank 0) shared memory,
// A rows 128-255 and the other half of B from the peer's, and writes the
// accumulator rows of each CTA into that CTA's TMEM.

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %clusterid.x;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t num_clusters_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %nclusterid.x;" : "=r"(r));
    return r;
}

// shared::cluster address of the object at shared::cta address `a` in CTA `rank`
__device__ __forceinline__ uint32_t map_to_cta(uint32_t a, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}

__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The same barrier with a relaxed arrival: it orders execution only, so the
// arrival does not wait for this thread's earlier memory operations (global
// stores in particular) to become visible cluster-wide.
__device__ __forceinline__ void cluster_sync_relaxed_arrive() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Release fence at cluster scope restricted to this CTA's shared-memory
// accesses: orders them before a following relaxed arrival on another CTA's
// barrier.  A release arrival orders every earlier memory access of the
// thread, and on GB300 waits about a microsecond for the SM's outstanding
// global traffic (operand loads in flight included); this one does not.
__device__ __forceinline__ void fence_release_smem_cluster() {
    asm volatile("fence.release.sync_restrict::shared::cta.cluster;" ::: "memory");
}

// arrive on an mbarrier given by its shared::cluster address (own or peer CTA)
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx_cluster(uint32_t cluster_addr, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cluster.shared::cluster.b64 _, [%0], %1;" ::"r"(cluster_addr),
                 "r"(bytes)
                 : "memory");
}

// Remote arrivals that publish no data (the arriving thread has only read
// shared memory the barrier guards): relaxed, so the arrival does not wait
// for the thread's earlier memory operations to become visible cluster-wide.
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx_cluster_relaxed(uint32_t cluster_addr, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.relaxed.cluster.shared::cluster.b64 _, [%0], %1;" ::"r"(cluster_addr),
                 "r"(bytes)
                 : "memory");
}

// Cluster launch control: asks the hardware to cancel a cluster of this grid
// that has not started yet.  The 16-byte response is written to `resp` in
// every CTA of the cluster and counted (16 bytes) on the barrier at the same
// offset in each.  No request may follow one whose response said "none".
__device__ __forceinline__ void clc_try_cancel_multicast(void* resp, uint64_t* bar) {
    asm volatile(
        "clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes.multicast::cluster::all.b128 "
        "[%0], [%1];" ::"r"(smem_u32(resp)),
        "r"(smem_u32(bar))
        : "memory");
}

// The x index of the first CTA of the cluster a response cancelled, or
// 0xFFFFFFFF when it cancelled none.
__device__ __forceinline__ uint32_t clc_cancelled_ctaid_x(const void* resp) {
    uint32_t ok, x = 0xFFFFFFFFu;
    asm volatile(
        "{\n\t.reg .b128 r;\n\t.reg .pred p;\n\t"
        "ld.shared.b128 r, [%2];\n\t"
        "clusterlaunchcontrol.query_cancel.is_canceled.pred.b128 p, r;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t"
        "@p clusterlaunchcontrol.query_cancel.get_first_ctaid::x.b32.b128 %1, r;\n\t}"
        : "=r"(ok), "+r"(x)
        : "r"(smem_u32(resp))
        : "memory");
    return ok ? x : 0xFFFFFFFFu;
}

// TMA tile load into this CTA's shared memory whose completion is counted on
// an mbarrier of either CTA of the pair (cluster address)
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* m, uint32_t bar_cluster, int32_t x,
                                                 int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
        "%4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(bar_cluster), "r"(x), "r"(y));
}

__device__ __forceinline__ void tma_load_3d_pair(void* dst, const CUtensorMap* m, uint32_t bar_cluster, int32_t x,
                                                 int32_t y, int32_t z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
        "%4, %5}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(bar_cluster), "r"(x), "r"(y), "r"(z));
}

// collective over the pair: executed by one warp in each of the two CTAs
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

__device__ __forceinline__ void umma_f16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                              uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

// MXFP8 MMA of a CTA pair (M = 256): as umma_mxf8, with A rows 0-127 and
// the first half of B in the leader's shared memory and the rest in the
// peer's.  Each CTA's tensor memory holds the accumulator rows and the A
// scale factors of its own 128 rows and the B scale factors of all N columns,
// at the same addresses in both CTAs.
__device__ __forceinline__ void umma_mxf8_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                               uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate));
}

// The pair's shared -> tensor memory copy (issued by the leader): the source
// descriptor addresses the same offset in both CTAs' shared memory, and each
// CTA's tensor memory receives the lines of its own shared memory.
__device__ __forceinline__ void tmem_cp_32x128b_warpx4_pair(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc));
}

// arrive once on the barrier at the same shared offset in every CTA of
// cta_mask when all tcgen05 operations issued so far by this thread are done
__device__ __forceinline__ void umma_commit_pair_mc(uint64_t* bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(cta_mask));
}

// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned)
// from this CTA's shared memory into the shared memory of a CTA of the
// cluster; completion is counted in bytes on `bar_cluster` (a barrier of the
// destination CTA).  The source must have been written through the generic
// proxy and fenced (fence.proxy.async) before the copy is issued.
__device__ __forceinline__ void bulk_copy_to_cluster(uint32_t dst_cluster, const void* src, uint32_t bytes,
                                                     uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst_cluster),
        "r"(smem_u32(src)), "r"(bytes), "r"(bar_cluster)
        : "memory");
}

__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// global -> this CTA's shared memory, bytes a multiple of 16, both addresses
// 16-byte aligned; completes on bar
__device__ __forceinline__ void bulk_load_global(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// this CTA's shared memory -> global (a bulk group; see bulk_commit_group)
__device__ __forceinline__ void bulk_store_global(void* dst, const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_u32(src)),
                 "r"(bytes)
                 : "memory");
}

// at most three committed bulk groups may still be reading their sources
__device__ __forceinline__ void bulk_wait_read_3() { asm volatile("cp.async.bulk.wait_group.read 3;" ::: "memory"); }

// every committed bulk group has completed
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// waits until every committed bulk copy of this thread has finished reading its source
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

}  // namespace bst
