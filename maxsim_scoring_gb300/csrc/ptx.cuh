// Inline-PTX wrappers for the sm_103a features the kernels use: mbarriers,
// TMA tensor loads, tensor memory (tcgen05.alloc / ld) and the 5th-generation
// tensor-core MMA (tcgen05.mma, kind::f16, fp32 accumulation in TMEM).
#pragma once

#include <cstdint>
#include <cuda.h>

namespace maxsim {

// ---------------------------------------------------------------- basics

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void named_barrier_sync(uint32_t id, uint32_t nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Move registers between the warpgroups of a CTA: every warp of a
// warpgroup executes the same call. inc waits until the pool the block was
// launched with can supply the new count.
template <uint32_t kRegs>
__device__ __forceinline__ void regs_release() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegs));
}

template <uint32_t kRegs>
__device__ __forceinline__ void regs_claim() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegs));
}

// (x0, x1) *= (s0, s1) with one packed instruction (mul.rn.f32x2: each lane
// rounded as a plain fp32 multiply).
__device__ __forceinline__ void mul2_rn(float& x0, float& x1, float s0, float s1) {
    asm("{\n\t.reg .b64 a, b, d;\n\t"
        "mov.b64 a, {%0, %1};\n\t"
        "mov.b64 b, {%2, %3};\n\t"
        "mul.rn.f32x2 d, a, b;\n\t"
        "mov.b64 {%0, %1}, d;\n\t}"
        : "+f"(x0), "+f"(x1)
        : "f"(s0), "f"(s1));
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.b32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// ---------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled bulk tensor load into this CTA's shared memory; completion is
// signalled on `bar` as transaction bytes. x = innermost coordinate (elements).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int32_t x,
                                            int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// Same, with an L2 eviction-priority hint (policy from createpolicy).
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap* map, uint32_t bar, int32_t x,
                                                 int32_t y, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
        "%3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ---------------------------------------------------------------- clusters

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Address, in the shared::cluster window, of the same shared-memory offset in
// the CTA of rank `rank`.
__device__ __forceinline__ uint32_t map_shared_rank(uint32_t smem_addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
    return r;
}

// Arrive (release, cluster scope) on an mbarrier given by its shared::cluster address.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Arrive on an mbarrier given by its shared::cluster address, with the
// default (CTA-scope) release: enough when the only accesses to order are
// tensor-memory reads, which tcgen05.fence::before_thread_sync orders before
// this arrive. A cluster-scope release would first wait for every earlier
// memory operation of the thread (global stores included) to become visible
// to the cluster.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.b32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// All threads of every CTA of the cluster.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- tensor memory

// Warp-wide: allocate `ncols` TMEM columns (power of two >= 32); the base
// address is written to shared memory at `dst`.
// kGroup = 2: a CTA pair allocates the same columns in both CTAs (one warp of
// each CTA executes it); a kernel uses one group size for all tcgen05 ops.
template <int kGroup = 1>
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols) {
    if constexpr (kGroup == 1)
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst), "r"(ncols)
                     : "memory");
    else
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst), "r"(ncols)
                     : "memory");
}

template <int kGroup = 1>
__device__ __forceinline__ void tmem_relinquish() {
    if constexpr (kGroup == 1)
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    else
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

template <int kGroup = 1>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    if constexpr (kGroup == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
    else
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (f16 / bf16 inputs), fp32 D.
// kGroup = 2: issued by the pair's even CTA; A's rows and D's lanes are split
// between the two CTAs (128 each, same smem / TMEM offsets), B's N rows are
// split in halves (the first N/2 from the even CTA).
template <int kGroup = 1>
__device__ __forceinline__ void mma_f16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
    if constexpr (kGroup == 1)
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
            : "memory");
}

// Same as mma_f16_ss with each descriptor given as its two 32-bit words.
template <int kGroup = 1>
__device__ __forceinline__ void mma_f16_ss_words(uint32_t d_tmem, uint32_t a_lo, uint32_t a_hi, uint32_t b_lo,
                                                 uint32_t b_hi, uint32_t idesc, uint32_t accumulate) {
    if constexpr (kGroup == 1)
        asm volatile(
            "{\n\t.reg .pred p;\n\t.reg .b64 da, db;\n\t"
            "setp.ne.b32 p, %6, 0;\n\t"
            "mov.b64 da, {%1, %2};\n\t"
            "mov.b64 db, {%3, %4};\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, p;\n\t}" ::"r"(d_tmem),
            "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\t.reg .b64 da, db;\n\t"
            "setp.ne.b32 p, %6, 0;\n\t"
            "mov.b64 da, {%1, %2};\n\t"
            "mov.b64 db, {%3, %4};\n\t"
            "tcgen05.mma.cta_group::2.kind::f16 [%0], da, db, %5, p;\n\t}" ::"r"(d_tmem),
            "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate)
            : "memory");
}

// MMA chains issued by one elected lane of the calling warp. Every lane of
// the warp calls them with the same (warp-uniform) arguments; elect.sync with
// a full mask always picks the same lane, so the chains and the commits that
// track them come from one thread. Issuing a whole chain from one asm block
// keeps the tensor pipe fed: one instruction per block would cost more issue
// cycles than a 128 x 128 x 16 MMA takes to run.
//
// A K = 128 chain: eight K = 16 steps into d. A and B are K-major with the
// 128-byte swizzle; a step advances both descriptors by 32 bytes (2 in the
// 16-byte address field) and the fifth step moves to the next 64-element
// atom, kAAtom16 / kBAtom16 (atom bytes >> 4) further on. The first step
// accumulates into d only if `accumulate` is nonzero.
#define MAXSIM_CHAIN8(GROUP)                                                               \
    "{\n\t.reg .pred e, p0, pt;\n\t"                                                      \
    ".reg .b64 a1, a2, a3, a4, a5, a6, a7, b1, b2, b3, b4, b5, b6, b7;\n\t"               \
    "setp.ne.b32 p0, %4, 0;\n\t"                                                          \
    "setp.eq.b32 pt, %4, %4;\n\t"                                                         \
    "add.s64 a1, %1, 2;\n\tadd.s64 a2, %1, 4;\n\tadd.s64 a3, %1, 6;\n\t"                  \
    "add.s64 a4, %1, %5;\n\tadd.s64 a5, %1, %6;\n\tadd.s64 a6, %1, %7;\n\tadd.s64 a7, %1, %8;\n\t" \
    "add.s64 b1, %2, 2;\n\tadd.s64 b2, %2, 4;\n\tadd.s64 b3, %2, 6;\n\t"                  \
    "add.s64 b4, %2, %9;\n\tadd.s64 b5, %2, %10;\n\tadd.s64 b6, %2, %11;\n\tadd.s64 b7, %2, %12;\n\t" \
    "elect.sync _|e, 0xffffffff;\n\t"                                                     \
    "@e tcgen05.mma.cta_group::" GROUP ".kind::f16 [%0], %1, %2, %3, p0;\n\t"            \
    "@e tcgen05.mma.cta_group::" GROUP ".kind::f16 [%0], a1, b1, %3, pt;\n\t"            \
    "@e tcgen05.mma.cta_group::" GROUP ".kind::f16 [%0], a2, b2, %3, pt;\n\t"            \
    "@e tcgen05.mma.cta_group::" GROUP ".kind::f16 [%0], a3, b3, %3, pt;\n\t"            \
    "@e tcgen05.mma.cta_group::" GROUP ".kind::f16 [%0], a4, b4, %3, pt;\n\t"            \
    "@e tcgen05.mma.cta_group::" GROUP ".kind::f16 [%0], a5, b5, %3, pt;\n\t"            \
    "@e tcgen05.mma.cta_group::" GROUP ".kind::f16 [%0], a6, b6, %3, pt;\n\t"            \
    "@e tcgen05.mma.cta_group::" GROUP ".kind::f16 [%0], a7, b7, %3, pt;\n\t}"

template <int kGroup, uint32_t kAAtom16, uint32_t kBAtom16>
__device__ __forceinline__ void mma_chain8_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                              uint32_t accumulate) {
    if constexpr (kGroup == 1)
        asm volatile(MAXSIM_CHAIN8("1")::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(accumulate), "n"(kAAtom16),
                     "n"(kAAtom16 + 2), "n"(kAAtom16 + 4), "n"(kAAtom16 + 6), "n"(kBAtom16), "n"(kBAtom16 + 2),
                     "n"(kBAtom16 + 4), "n"(kBAtom16 + 6)
                     : "memory");
    else
        asm volatile(MAXSIM_CHAIN8("2")::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(accumulate), "n"(kAAtom16),
                     "n"(kAAtom16 + 2), "n"(kAAtom16 + 4), "n"(kAAtom16 + 6), "n"(kBAtom16), "n"(kBAtom16 + 2),
                     "n"(kBAtom16 + 4), "n"(kBAtom16 + 6)
                     : "memory");
}
#undef MAXSIM_CHAIN8

// A K = 64 chain (one atom, four K = 16 steps), same conventions.
#define MAXSIM_CHAIN4(GROUP)                                                    \
    "{\n\t.reg .pred e, p0, pt;\n\t.reg .b64 a1, a2, a3, b1, b2, b3;\n\t"      \
    "setp.ne.b32 p0, %4, 0;\n\t"                                               \
    "setp.eq.b32 pt, %4, %4;\n\t"                                              \
    "add.s64 a1, %1, 2;\n\tadd.s64 a2, %1, 4;\n\tadd.s64 a3, %1, 6;\n\t"       \
    "add.s64 b1, %2, 2;\n\tadd.s64 b2, %2, 4;\n\tadd.s64 b3, %2, 6;\n\t"       \
    "elect.sync _|e, 0xffffffff;\n\t"                                          \
    "@e tcgen05.mma.cta_group::" GROUP ".kind::f16 [%0], %1, %2, %3, p0;\n\t" \
    "@e tcgen05.mma.cta_group::" GROUP ".kind::f16 [%0], a1, b1, %3, pt;\n\t" \
    "@e tcgen05.mma.cta_group::" GROUP ".kind::f16 [%0], a2, b2, %3, pt;\n\t" \
    "@e tcgen05.mma.cta_group::" GROUP ".kind::f16 [%0], a3, b3, %3, pt;\n\t}"

template <int kGroup>
__device__ __forceinline__ void mma_chain4_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                              uint32_t accumulate) {
    if constexpr (kGroup == 1)
        asm volatile(MAXSIM_CHAIN4("1")::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(accumulate) : "memory");
    else
        asm volatile(MAXSIM_CHAIN4("2")::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(accumulate) : "memory");
}
#undef MAXSIM_CHAIN4

// One K = 16 step, same conventions.
template <int kGroup>
__device__ __forceinline__ void mma_step_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
    if constexpr (kGroup == 1)
        asm volatile(
            "{\n\t.reg .pred e, p0;\n\t"
            "setp.ne.b32 p0, %4, 0;\n\t"
            "elect.sync _|e, 0xffffffff;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p0;\n\t}" ::"r"(d),
            "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred e, p0;\n\t"
            "setp.ne.b32 p0, %4, 0;\n\t"
            "elect.sync _|e, 0xffffffff;\n\t"
            "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p0;\n\t}" ::"r"(d),
            "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
            : "memory");
}

// tcgen05.commit from the elected lane (the lane that issued the chains).
template <int kGroup = 1>
__device__ __forceinline__ void mma_commit_elect(uint32_t bar, uint16_t cta_mask = 3) {
    if constexpr (kGroup == 1)
        asm volatile(
            "{\n\t.reg .pred e;\n\t"
            "elect.sync _|e, 0xffffffff;\n\t"
            "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred e;\n\t"
            "elect.sync _|e, 0xffffffff;\n\t"
            "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], "
            "%1;\n\t}" ::"r"(bar),
            "h"(cta_mask)
            : "memory");
}

// Arrive on `bar` once every tcgen05 operation issued so far by this thread
// has completed. kGroup = 2: the arrival goes to the barrier at the same
// offset in every CTA of the pair selected by cta_mask (bit r = rank r).
template <int kGroup = 1>
__device__ __forceinline__ void mma_commit(uint32_t bar, uint16_t cta_mask = 3) {
    if constexpr (kGroup == 1)
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                     : "memory");
    else
        asm volatile(
            "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
                bar),
            "h"(cta_mask)
            : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 32 consecutive fp32 columns of this thread's TMEM lane (32x32b shape: warp w
// of a warpgroup reads lanes 32*(w%4) .. 32*(w%4)+31).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t* r = reinterpret_cast<uint32_t*>(v);
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

// 16 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[32]) {
    uint32_t* r = reinterpret_cast<uint32_t*>(v);
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

// 32 (or 16) consecutive fp32 columns of this thread's TMEM lane, and their
// maximum computed on the way out of tensor memory (tcgen05.ld.red, .max:
// NaN columns are ignored as by max.f32; all-NaN gives NaN).
#define MAXSIM_R32 \
    "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}"
__device__ __forceinline__ float tmem_ldmax32(uint32_t taddr, float (&v)[32]) {
    uint32_t* r = reinterpret_cast<uint32_t*>(v);
    float m;
    asm volatile("tcgen05.ld.red.sync.aligned.32x32b.x32.max.f32 " MAXSIM_R32 ", %32, [%33];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                   "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
                   "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
                   "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=f"(m)
                 : "r"(taddr));
    return m;
}
#undef MAXSIM_R32

__device__ __forceinline__ float tmem_ldmax16(uint32_t taddr, float (&v)[32]) {
    uint32_t* r = reinterpret_cast<uint32_t*>(v);
    float m;
    asm volatile(
        "tcgen05.ld.red.sync.aligned.32x32b.x16.max.f32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, %16, [%17];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=f"(m)
        : "r"(taddr));
    return m;
}

// ---------------------------------------------------------------- INT8 -> f16

// Eight signed bytes (w0: elements 0-3, w1: elements 4-7, little-endian) to
// eight binary16 values, exactly. Each byte b is biased to u = b + 128, placed
// as the low mantissa byte of the binary16 1024.0 (exponent 10, unit ulp), so
// the half is 1024 + u, and 1152 = 1024 + 128 is subtracted: the result is b.
__device__ __forceinline__ uint32_t i8x2_to_f16x2(uint32_t biased, uint32_t selector) {
    uint32_t h, d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(h) : "r"(biased), "r"(0x64646464u), "r"(selector));
    asm("sub.f16x2 %0, %1, %2;" : "=r"(d) : "r"(h), "r"(0x64806480u));
    return d;
}

__device__ __forceinline__ uint4 i8x8_to_f16x8(uint32_t w0, uint32_t w1) {
    const uint32_t u0 = w0 ^ 0x80808080u, u1 = w1 ^ 0x80808080u;
    uint4 r;
    r.x = i8x2_to_f16x2(u0, 0x4140u);  // bytes 0, 1
    r.y = i8x2_to_f16x2(u0, 0x4342u);  // bytes 2, 3
    r.z = i8x2_to_f16x2(u1, 0x4140u);
    r.w = i8x2_to_f16x2(u1, 0x4342u);
    return r;
}

// ---------------------------------------------------------------- descriptors

// Shared-memory matrix descriptor for a K-major operand stored with the
// 128-byte swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart
// (stride byte offset), base 1024-byte aligned. Layout of the 64-bit word:
// [0,14) start address >> 4, [16,30) leading byte offset >> 4 (unused for a
// swizzled K-major operand), [32,46) stride byte offset >> 4, [46,48) fixed
// version 1, [49,52) base offset, [61,64) swizzle mode (2 = 128-byte).
__device__ __forceinline__ uint64_t sdesc_k_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(1) << 16;
    d |= static_cast<uint64_t>(1024 >> 4) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// Instruction descriptor for kind::f16 with fp32 accumulation, both operands
// K-major: [4,6) D format (1 = f32), [7,10) A format, [10,13) B format
// (0 = f16, 1 = bf16), [15] / [16] A / B major (0 = K), [17,23) N >> 3,
// [24,29) M >> 4.
__host__ __device__ constexpr uint32_t idesc_f16_f32(uint32_t ab_format, uint32_t M, uint32_t N) {
    return (1u << 4) | (ab_format << 7) | (ab_format << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

}  // namespace maxsim
