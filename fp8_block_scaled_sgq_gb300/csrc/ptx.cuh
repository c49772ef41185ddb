// Inline-PTX building blocks for sm_103a: mbarriers, TMA, tcgen05 (UMMA,
// TMEM), programmatic dependent launch, and a bounded wait.
#pragma once
#include <cstdint>
#include <cuda.h>

namespace sgq {
namespace ptx {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t)::"memory");
    return t;
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
// Non-blocking probe of a phase (no suspend).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\n"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0u;
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\n"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Fences between the generic proxy and the async proxy (TMA / tcgen05).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ TMA
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* m) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* m, int32_t x,
                                            int32_t y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// ------------------------------------------------------------------ cp.async
// 4-byte global -> shared copy through the LSU async path (Ampere-style).
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
// Waits until at most n of this thread's committed groups are still pending.
__device__ __forceinline__ void cp_async_wait_pending(int n) {
    switch (n) {
        case 0: asm volatile("cp.async.wait_group 0;" ::: "memory"); break;
        case 1: asm volatile("cp.async.wait_group 1;" ::: "memory"); break;
        case 2: asm volatile("cp.async.wait_group 2;" ::: "memory"); break;
        case 3: asm volatile("cp.async.wait_group 3;" ::: "memory"); break;
        case 4: asm volatile("cp.async.wait_group 4;" ::: "memory"); break;
        case 5: asm volatile("cp.async.wait_group 5;" ::: "memory"); break;
        case 6: asm volatile("cp.async.wait_group 6;" ::: "memory"); break;
        default: asm volatile("cp.async.wait_group 7;" ::: "memory"); break;
    }
}

// ------------------------------------------------------------------ PDL
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------------ tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
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
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Arrives on `bar` once every tcgen05 op issued so far by this thread is done.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     bar)
                 : "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, FP8 operands, fp32 accumulator.
__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Block-scaled variant: one UE8M0 scale per row per 32-wide K chunk, read
// from TMEM at sfa / sfb (byte selected by the sf ids in idesc).
__device__ __forceinline__ void mma_mxf8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %6, 0;\n"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X"
        " [%0], %1, %2, %3, [%4], [%5], p;\n}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}
// SMEM (32 rows x 16 bytes) -> TMEM, replicated into all four 32-lane quadrants.
__device__ __forceinline__ void tmem_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
                 : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 32 lanes x N consecutive 32-bit columns; thread t gets lane (base_lane + t).
template <int N>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, uint32_t (&r)[N]);

template <>
__device__ __forceinline__ void tmem_ld<4>(uint32_t taddr, uint32_t (&r)[4]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr));
}
template <>
__device__ __forceinline__ void tmem_ld<8>(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
}
template <>
__device__ __forceinline__ void tmem_ld<16>(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
template <>
__device__ __forceinline__ void tmem_ld<32>(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
        "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

// ------------------------------------------------------------------ predicated issue
// Variants executed by a whole converged warp; only lanes with `pred` != 0
// perform the operation.  Keeping the warp converged lets the compiler keep
// descriptors and addresses warp-uniform, which makes tcgen05/TMA issue much
// cheaper than from a diverged single-lane branch.  Callers pass one fixed
// lane so that MMAs and the commits that track them come from one thread.
__device__ __forceinline__ void mma_f8_if(uint32_t pred, uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n.reg .pred p, q;\nsetp.ne.b32 p, %5, 0;\nsetp.ne.b32 q, %4, 0;\n"
        "@p tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, q;\n}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(pred)
        : "memory");
}
__device__ __forceinline__ void mma_mxf8_if(uint32_t pred, uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n.reg .pred p, q;\nsetp.ne.b32 p, %7, 0;\nsetp.ne.b32 q, %6, 0;\n"
        "@p tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X"
        " [%0], %1, %2, %3, [%4], [%5], q;\n}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate), "r"(pred)
        : "memory");
}
__device__ __forceinline__ void tmem_cp_32x128b_x4_if(uint32_t pred, uint32_t taddr, uint64_t sdesc) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %2, 0;\n"
        "@p tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;\n}" ::"r"(taddr), "l"(sdesc), "r"(pred)
        : "memory");
}
__device__ __forceinline__ void tc_commit_if(uint32_t pred, uint32_t bar) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %1, 0;\n"
        "@p tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}" ::"r"(bar),
        "r"(pred)
        : "memory");
}
__device__ __forceinline__ void mbar_arrive_if(uint32_t pred, uint32_t bar) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %1, 0;\n@p mbarrier.arrive.shared::cta.b64 _, [%0];\n}" ::"r"(bar),
        "r"(pred)
        : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx_if(uint32_t pred, uint32_t bar, uint32_t bytes) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %2, 0;\n"
        "@p mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n}" ::"r"(bar), "r"(bytes), "r"(pred)
        : "memory");
}
__device__ __forceinline__ void tma_load_2d_if(uint32_t pred, uint32_t dst, const CUtensorMap* m, int32_t x,
                                               int32_t y, uint32_t bar) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %5, 0;\n"
        "@p cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];\n}" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(bar), "r"(pred)
        : "memory");
}


// ------------------------------------------------------------------ elected issue
// A converged warp elects one lane (elect.sync) to issue; with the whole warp
// active the same lane is elected every time, so MMAs and the commit that
// tracks them come from one thread.

// One block-scaled 128-wide K stage: the A and B scale-factor copies into
// TMEM (B in two 128-row copies), then four K = 32 MMAs (byte j of each scale
// word for MMA j) accumulating into d; the first starts over when acc == 0.
__device__ __forceinline__ void mx_stage2_elect(uint32_t d, uint64_t a, uint64_t b, uint32_t i0, uint32_t i1,
                                                uint32_t i2, uint32_t i3, uint32_t sfa_t, uint32_t sfb_t,
                                                uint64_t sfa_d, uint64_t sfb_d, uint32_t acc) {
    asm volatile(
        "{\n.reg .pred e, q, t;\n.reg .b64 a1, a2, a3, b1, b2, b3, s2;\n.reg .b32 t2;\n"
        "elect.sync _|e, 0xffffffff;\n"
        "setp.ne.b32 q, %9, 0;\n"
        "setp.eq.u32 t, %0, %0;\n"
        "add.s64 a1, %1, 2;\nadd.s64 a2, %1, 4;\nadd.s64 a3, %1, 6;\n"
        "add.s64 b1, %2, 2;\nadd.s64 b2, %2, 4;\nadd.s64 b3, %2, 6;\n"
        "add.s64 s2, %11, 32;\nadd.u32 t2, %8, 4;\n"
        "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%7], %10;\n"
        "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%8], %11;\n"
        "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [t2], s2;\n"
        "@e tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%7], [%8], q;\n"
        "@e tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], a1, b1, %4, [%7], [%8], t;\n"
        "@e tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], a2, b2, %5, [%7], [%8], t;\n"
        "@e tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], a3, b3, %6, [%7], [%8], t;\n}" ::"r"(d),
        "l"(a), "l"(b), "r"(i0), "r"(i1), "r"(i2), "r"(i3), "r"(sfa_t), "r"(sfb_t), "r"(acc), "l"(sfa_d), "l"(sfb_d)
        : "memory");
}
// mx_stage2_elect for a CTA pair (.cta_group::2, issued by the leader CTA):
// each CTA's scale words go from its own shared memory to its own TMEM (same
// addresses), and the M = 256 MMAs read A rows 0-127 and B rows 0 .. N/2-1
// from the leader's shared memory, the rest from the peer's at the same offsets.
__device__ __forceinline__ void mx_stage2_elect_pair(uint32_t d, uint64_t a, uint64_t b, uint32_t i0, uint32_t i1,
                                                     uint32_t i2, uint32_t i3, uint32_t sfa_t, uint32_t sfb_t,
                                                     uint64_t sfa_d, uint64_t sfb_d, uint32_t acc) {
    asm volatile(
        "{\n.reg .pred e, q, t;\n.reg .b64 a1, a2, a3, b1, b2, b3, s2;\n.reg .b32 t2;\n"
        "elect.sync _|e, 0xffffffff;\n"
        "setp.ne.b32 q, %9, 0;\n"
        "setp.eq.u32 t, %0, %0;\n"
        "add.s64 a1, %1, 2;\nadd.s64 a2, %1, 4;\nadd.s64 a3, %1, 6;\n"
        "add.s64 b1, %2, 2;\nadd.s64 b2, %2, 4;\nadd.s64 b3, %2, 6;\n"
        "add.s64 s2, %11, 32;\nadd.u32 t2, %8, 4;\n"
        "@e tcgen05.cp.cta_group::2.32x128b.warpx4 [%7], %10;\n"
        "@e tcgen05.cp.cta_group::2.32x128b.warpx4 [%8], %11;\n"
        "@e tcgen05.cp.cta_group::2.32x128b.warpx4 [t2], s2;\n"
        "@e tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%7], [%8], q;\n"
        "@e tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], a1, b1, %4, [%7], [%8], t;\n"
        "@e tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], a2, b2, %5, [%7], [%8], t;\n"
        "@e tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], a3, b3, %6, [%7], [%8], t;\n}" ::"r"(d),
        "l"(a), "l"(b), "r"(i0), "r"(i1), "r"(i2), "r"(i3), "r"(sfa_t), "r"(sfb_t), "r"(acc), "l"(sfa_d), "l"(sfb_d)
        : "memory");
}
// Pair commit from one elected lane: arrives on `bar` (same offset) in both
// CTAs when the leader's earlier tcgen05 ops are done.
__device__ __forceinline__ void commit_pair_elect(uint32_t bar) {
    asm volatile(
        "{\n.reg .pred e;\nelect.sync _|e, 0xffffffff;\n"
        "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n}" ::"r"(
            bar),
        "h"(static_cast<uint16_t>(3))
        : "memory");
}
// Pair commit arriving on this (the leader) CTA's `bar` only.
__device__ __forceinline__ void commit_pair_local_elect(uint32_t bar) {
    asm volatile(
        "{\n.reg .pred e;\nelect.sync _|e, 0xffffffff;\n"
        "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}" ::"r"(bar)
        : "memory");
}
// Commit (arrive on `bar` when this lane's earlier tcgen05 ops are done).
__device__ __forceinline__ void commit_elect(uint32_t bar) {
    asm volatile(
        "{\n.reg .pred e;\nelect.sync _|e, 0xffffffff;\n"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}" ::"r"(bar)
        : "memory");
}

// ------------------------------------------------------------------ CTA pairs
// A cluster of two CTAs (ranks 0 and 1) drives one tcgen05 unit pair: rank 0
// (the leader) issues every MMA, scale copy and commit with .cta_group::2;
// both CTAs allocate the same TMEM columns.  A pair-issued op reads operand
// A rows 0-127 and the first half of the B columns from the leader's shared
// memory and the rest from the peer's, at the same offsets; the scale copy
// fills each CTA's TMEM from its own shared memory; each CTA's accumulator
// holds its 128 rows and all N columns.
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Shared-memory address of the same variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa(uint32_t smem_addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
    return r;
}
// Atomic add with acquire-release semantics at GPU scope: publishes what
// happened before it (including what a preceding bar.sync ordered) and, for
// the thread that sees the final count, makes the other adders' writes visible.
__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t* p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}
// Orders this thread's generic-proxy memory accesses (all state spaces)
// with its later async-proxy ones (bulk copies, TMA).
__device__ __forceinline__ void fence_proxy_async_all() { asm volatile("fence.proxy.async;" ::: "memory"); }
// Load with acquire semantics at GPU scope (a spin on another CTA's count).
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
// 32-byte global store (the address must be 32-byte aligned).
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t (&w)[8]) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]), "r"(w[1]),
                 "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Split cluster barrier: a relaxed arrive (nothing to publish beyond what a
// fence.mbarrier_init already released) and the matching wait, taken later.
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Arrive (release at cluster scope) on an mbarrier given by its cluster address.
__device__ __forceinline__ void mbar_arrive_cluster_if(uint32_t pred, uint32_t cluster_bar) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %1, 0;\n"
        "@p mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];\n}" ::"r"(cluster_bar), "r"(pred)
        : "memory");
}
// Bounded-wait building block with cluster-scope acquire.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\n"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0u;
}
__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t cluster_addr) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(cluster_addr) : "memory");
    return v;
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t cluster_addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(cluster_addr) : "memory");
    return v;
}
__device__ __forceinline__ void st_cluster_f32(uint32_t cluster_addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(cluster_addr), "f"(v) : "memory");
}
__device__ __forceinline__ void st_cluster_u32(uint32_t cluster_addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}
// TMA tile load into this CTA's shared memory whose completion is signalled
// on an mbarrier of either CTA of the pair (cluster address).
__device__ __forceinline__ void tma_load_2d_pair_if(uint32_t pred, uint32_t dst, const CUtensorMap* m, int32_t x,
                                                    int32_t y, uint32_t cluster_bar) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %5, 0;\n"
        "@p cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];\n}" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(cluster_bar), "r"(pred)
        : "memory");
}

// Bulk copy (async proxy) of `bytes` (a multiple of 16, both addresses
// 16-byte aligned) from global memory into this CTA's shared memory,
// completing `bytes` of transactions on the CTA's mbarrier `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// Bulk copy (async proxy) of `bytes` (a multiple of 16, both addresses
// 16-byte aligned) from this CTA's shared memory to global memory, tracked
// by the thread's bulk async-groups (bulk_commit, bulk_wait_all).
__device__ __forceinline__ void bulk_store(void* dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until every committed bulk group of this thread is complete (its
// writes performed, its shared-memory source free again).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Bulk copy (async proxy) of `bytes` (multiple of 16) from this CTA's shared
// memory to another CTA's, completing `bytes` of transactions on an mbarrier
// in the destination CTA.  Used as a cheap cross-CTA signal with payload: the
// copy's completion also orders this thread's earlier shared-memory writes
// (published to the async proxy by fence.proxy.async) before the receiver.
__device__ __forceinline__ void bulk_copy_to_cluster_if(uint32_t pred, uint32_t dst_cluster, uint32_t src_cta,
                                                        uint32_t bytes, uint32_t cluster_bar) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "@p cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n}" ::"r"(
            dst_cluster),
        "r"(src_cta), "r"(bytes), "r"(cluster_bar), "r"(pred)
        : "memory");
}

// tcgen05 forms for one CTA (CG = 1) or a CTA pair (CG = 2).  Every tcgen05
// instruction of a kernel uses the same group size.
template <int CG>
__device__ __forceinline__ void tmem_alloc_g(uint32_t dst_smem, uint32_t ncols) {
    if constexpr (CG == 1)
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                     : "memory");
    else
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                     : "memory");
}
template <int CG>
__device__ __forceinline__ void tmem_relinquish_g() {
    if constexpr (CG == 1)
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    else
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
template <int CG>
__device__ __forceinline__ void tmem_dealloc_g(uint32_t taddr, uint32_t ncols) {
    if constexpr (CG == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
    else
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
template <int CG>
__device__ __forceinline__ void mma_f8_g_if(uint32_t pred, uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
    if constexpr (CG == 1) {
        mma_f8_if(pred, d_tmem, adesc, bdesc, idesc, accumulate);
    } else {
        asm volatile(
            "{\n.reg .pred p, q;\nsetp.ne.b32 p, %5, 0;\nsetp.ne.b32 q, %4, 0;\n"
            "@p tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, q;\n}" ::"r"(d_tmem),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(pred)
            : "memory");
    }
}
template <int CG>
__device__ __forceinline__ void mma_mxf8_g_if(uint32_t pred, uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                              uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                              uint32_t accumulate) {
    if constexpr (CG == 1) {
        mma_mxf8_if(pred, d_tmem, adesc, bdesc, idesc, sfa_tmem, sfb_tmem, accumulate);
    } else {
        asm volatile(
            "{\n.reg .pred p, q;\nsetp.ne.b32 p, %7, 0;\nsetp.ne.b32 q, %6, 0;\n"
            "@p tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X"
            " [%0], %1, %2, %3, [%4], [%5], q;\n}" ::"r"(d_tmem),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate), "r"(pred)
            : "memory");
    }
}
template <int CG>
__device__ __forceinline__ void tmem_cp_g_if(uint32_t pred, uint32_t taddr, uint64_t sdesc) {
    if constexpr (CG == 1) {
        tmem_cp_32x128b_x4_if(pred, taddr, sdesc);
    } else {
        asm volatile(
            "{\n.reg .pred p;\nsetp.ne.b32 p, %2, 0;\n"
            "@p tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;\n}" ::"r"(taddr), "l"(sdesc), "r"(pred)
            : "memory");
    }
}
// Commit: CG = 1 arrives on this CTA's `bar`; CG = 2 arrives on `bar` (same
// offset) in both CTAs of the pair.
template <int CG>
__device__ __forceinline__ void tc_commit_g_if(uint32_t pred, uint32_t bar) {
    if constexpr (CG == 1) {
        tc_commit_if(pred, bar);
    } else {
        asm volatile(
            "{\n.reg .pred p;\nsetp.ne.b32 p, %1, 0;\n"
            "@p tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %2;\n}" ::"r"(
                bar),
            "r"(pred), "h"(static_cast<uint16_t>(3))
            : "memory");
    }
}
// Commit arriving on this CTA's `bar` only (pair form: the leader's own barrier).
template <int CG>
__device__ __forceinline__ void tc_commit_local_g_if(uint32_t pred, uint32_t bar) {
    if constexpr (CG == 1) {
        tc_commit_if(pred, bar);
    } else {
        asm volatile(
            "{\n.reg .pred p;\nsetp.ne.b32 p, %1, 0;\n"
            "@p tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}" ::"r"(bar),
            "r"(pred)
            : "memory");
    }
}

// ------------------------------------------------------------------ descriptors
// Shared-memory matrix descriptor (tcgen05 form): start >> 4 in [0,14),
// leading byte offset >> 4 in [16,30), stride byte offset >> 4 in [32,46),
// descriptor version 1 at bit 46, layout (swizzle) in [61,64).
enum : uint32_t { kLayoutNone = 0, kLayoutSw128 = 2 };
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes,
                                              uint32_t layout) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(layout & 7u) << 61;
    return d;
}

// Instruction descriptor, kind::f8f6f4: fp32 D, E4M3 A and B, both K-major.
__host__ __device__ constexpr uint32_t idesc_f8(uint32_t M, uint32_t N) {
    return (1u << 4)              // D format: f32
           | (0u << 7)            // A: E4M3
           | (0u << 10)           // B: E4M3
           | ((N >> 3) << 17)     // N / 8
           | ((M >> 4) << 24);    // M / 16
}
// Instruction descriptor, kind::mxf8f6f4 block-scaled: E4M3 A and B, K-major,
// UE8M0 scale factors; the A/B scale-factor ids are or-ed in per MMA.
__host__ __device__ constexpr uint32_t idesc_mxf8(uint32_t M, uint32_t N) {
    return (0u << 7) | (0u << 10) | ((N >> 3) << 17) | (1u << 23)  // scale format UE8M0
           | ((M >> 4) << 24);
}
__device__ __forceinline__ uint32_t idesc_sf_ids(uint32_t idesc, uint32_t a_id, uint32_t b_id) {
    return idesc | ((b_id & 3u) << 4) | ((a_id & 3u) << 29);
}

}  // namespace ptx
}  // namespace sgq
