// tc.cuh -- sm_103a building blocks: mbarrier, bulk async copies, tcgen05
// (TMEM allocation, MMA, commit, TMEM load/store) and shared-memory matrix
// descriptors.  Hand-written inline PTX; no CUTLASS / CuTe.
//
// Shared-memory operand layouts used throughout (bf16, no swizzle): operands
// are tiled into 8 x 16-byte "core matrices" (8 rows of 8 consecutive
// elements, 128 contiguous bytes).
//   K-major  (the reduction index k is contiguous inside a core matrix):
//       byte(r, k)  = (r/8)*RSTRIDE + (k/8)*KSTRIDE + (r%8)*16 + (k%8)*2
//   MN-major (the row index m (or n) is contiguous inside a core matrix):
//       byte(mn, k) = (mn/8)*MNSTRIDE + (k/8)*KSTRIDE + (k%8)*16 + (mn%8)*2
// For this no-swizzle ("interleaved") form the descriptor takes, in both
// majors, the K-direction core-matrix stride as its leading-dimension byte
// offset and the M/N-direction stride as its stride-dimension byte offset
// (checked on hardware by kda_selftest_tcgen05).  Every layout in this library
// keeps the k-groups 128 bytes apart, so one K=16 MMA step advances the
// descriptor start address by 256 bytes.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>

namespace kda {

// ----------------------------------------------------------------------------- addresses
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// byte offset of element (r, k) of a K-major operand
__host__ __device__ constexpr uint32_t kmaj_off(uint32_t r, uint32_t k, uint32_t kstride,
                                                uint32_t rstride) {
    return (r >> 3) * rstride + (k >> 3) * kstride + (r & 7u) * 16u + (k & 7u) * 2u;
}
// byte offset of element (mn, k) of an MN-major operand
__host__ __device__ constexpr uint32_t mnmaj_off(uint32_t mn, uint32_t k, uint32_t kstride,
                                                 uint32_t mnstride) {
    return (mn >> 3) * mnstride + (k >> 3) * kstride + (k & 7u) * 16u + (mn & 7u) * 2u;
}

// ----------------------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_addr(bar))
        : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
            smem_addr(bar)),
        "r"(bytes)
        : "memory");
}
__device__ __forceinline__ uint32_t mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok;
}
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ uint32_t mbar_test_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok;
}

// Limits below this are test settings (kda_set_wait_limit_ns): such a wait
// polls without suspending, so that any wait that does not complete at once
// gives up, whatever the hardware's suspend time of try_wait.
constexpr uint64_t kShortWaitNs = 1000000ull;

// Wait for the phase with the given parity to complete.  Bounded: returns
// false (and the caller must report a timeout and unwind) after `limit_ns`.
// The retry loop is kept rolled: it is inlined at every wait, and unrolled
// copies cost instruction-cache misses in the large fused kernel (measured).
// All lanes of a converged warp read the barrier and the global timer in the
// same instructions, so they return the same answer.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
    const bool poll = limit_ns < kShortWaitNs;
    if (!poll && mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
#pragma unroll 1
    for (uint32_t i = 1;; ++i) {
        if (poll ? mbar_test_wait(bar, parity) : mbar_try_wait(bar, parity)) return true;
        if ((i & 15u) == 0 && global_ns() - t0 > limit_ns) return false;
    }
}

// The library's per-device status block (kda_api.cu): word 0 holds the status
// bits, words 2-3 the limit in ns of the bounded waits that can give up on the
// way (2 s unless kda_set_wait_limit_ns changed it).  Kernels read it once, at
// the start.
__device__ __forceinline__ uint64_t wait_limit_ns(const int* status) {
    return *reinterpret_cast<const volatile unsigned long long*>(status + 2);
}
// Limit of the waits a CTA makes for its own copies and MMAs before it exits
// after giving up: longer than any limit a caller sets, so that nothing the CTA
// started is still writing its shared or tensor memory when it leaves.
constexpr uint64_t kDrainLimitNs = 4000000000ull;
// Wait (bounded by kDrainLimitNs) for the phase; used only to drain.
__device__ __forceinline__ bool mbar_drain(uint64_t* bar, uint32_t parity) {
    return mbar_wait(bar, parity, kDrainLimitNs);
}

// ----------------------------------------------------------------------------- bulk copies
// Global -> shared bulk copy completing on an mbarrier (16-byte aligned
// addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}
// Same copy with an L2 cache policy for the source lines (see l2_policy).
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], "
        "[%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}
// L2 cache policies for the hinted copies and stores: data streamed once is
// marked evict_first, data written now and read back soon evict_last.
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
__device__ __forceinline__ uint64_t l2_policy_evict_normal() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}
// Hint: bring `bytes` (multiple of 16) at `src` into L2 ahead of use.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
// bulk async-groups of the calling thread (bulk and tensor stores to global memory)
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// wait until at most N of the thread's groups are still reading their shared-memory source
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// wait until at most N of the thread's groups are still incomplete (writes not yet performed)
template <int N>
__device__ __forceinline__ void bulk_wait() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}
// ----------------------------------------------------------------------------- fences
// order async-proxy (bulk copy) global accesses with the thread's generic-proxy ones
__device__ __forceinline__ void fence_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ----------------------------------------------------------------------------- TMEM
// Allocation / deallocation are warp-collective.  The allocated base address
// (lane 0, first column) is written to shared memory at `dst`.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(dst)),
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
// TMEM address of (lane, column).
__device__ __forceinline__ uint32_t taddr(uint32_t base, uint32_t lane, uint32_t col) {
    return base + (lane << 16) + col;
}

// 32 lanes x 32-bit, 16 / 32 consecutive columns per thread (thread i of the
// warp reads lane (warp%4)*32 + i).  The registers are only valid after
// tmem_wait_ld; tmem_wait_ld16/32 also tie the registers to the wait so the
// compiler cannot read them early.
__device__ __forceinline__ void tmem_ld16(uint32_t ta, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%"
        "15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(ta));
}
__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void reg_fence16(uint32_t (&r)[16]) {
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]));
}
// Load 16 columns and wait (self-contained).
__device__ __forceinline__ void tmem_load16(uint32_t ta, uint32_t (&r)[16]) {
    tmem_ld16(ta, r);
    tmem_wait_ld();
    reg_fence16(r);
}
__device__ __forceinline__ void tmem_st16(uint32_t ta, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%"
        "14,%15,%16};" ::"r"(ta),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ----------------------------------------------------------------------------- MMA
// Shared-memory matrix descriptor, no swizzle: start address, leading-
// dimension byte offset (= K-direction core-matrix stride), stride-dimension
// byte offset (= M/N-direction core-matrix stride), all >> 4, and the fixed
// 0b001 field at bits 46..48 that tcgen05 descriptors carry.  Same meaning for
// K-major and MN-major operands (the major-ness is in the instruction
// descriptor).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t kstride, uint32_t mnstride) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((kstride >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((mnstride >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}
// Instruction descriptor for kind::f16 with bf16 A/B and fp32 accumulation:
// D format at bits 4..5 (1 = f32), A / B formats at 7..9 / 10..12 (1 = bf16),
// A / B major-ness at bits 15 / 16 (1 = MN-major), N>>3 at 17..22, M>>4 at 24..28.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(uint32_t M, uint32_t N, bool a_mn, bool b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) |
           ((b_mn ? 1u : 0u) << 16) | ((N >> 3) << 17) | ((M >> 4) << 24);
}
// D[tmem] (+)= A[smem] * B[smem]; issued by a single thread.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// True on exactly one lane of the (converged) warp.
__device__ __forceinline__ bool elect_one() {
    uint32_t is_leader;
    asm volatile(
        "{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(is_leader));
    return is_leader != 0;
}
// D[tmem] (+)= A[tmem] * B[smem]: A is read from tensor memory (lane = row m,
// 32-bit column c holds the two bf16 elements 2c (low half) and 2c+1 along K).
__device__ __forceinline__ void mma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive once on `bar` when every MMA issued so far by this thread completes.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_addr(bar))
        : "memory");
}

// ----------------------------------------------------------------------------- transcendentals
// Hardware base-2 exponential / logarithm (PTX ex2.approx / lg2.approx).
// The hardware base-2 exponential and logarithm (one MUFU operation each), with
// subnormal inputs and results flushed to zero.  Their one user, the chunk
// kernel's gate, never depends on a subnormal: the logarithm's inputs lie in
// (1, 2], 2^-|x| is subnormal only where 1 + 2^-|x| already rounds to 1, and the
// decays are at least e^-10 (the library rejects lower_bound < -10).
__device__ __forceinline__ float hw_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float hw_log2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ----------------------------------------------------------------------------- misc
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_to_f(uint16_t u) { return __uint_as_float(((uint32_t)u) << 16); }

__device__ __forceinline__ void st_shared_v4(uint32_t saddr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(saddr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

}  // namespace kda
