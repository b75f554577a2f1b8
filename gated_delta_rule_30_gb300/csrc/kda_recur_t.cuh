// kda_recur_t.cuh -- the transposed recurrence body, shared by the stand-alone
// transposed recurrence kernel (kda_recur_t.cu) and the fused kernel
// (kda_fused.cu).
//
// Transposed recurrence kernel of the KDA forward pass: the
// sequential chunk-to-chunk state update for one whole (sequence, head).  Used
// when there are enough (sequence, head) pairs to fill the GPU; with few long
// sequences the value-sliced kernel in kda_recur.cu spreads each pair over
// more SMs instead.
//
// The state is kept transposed, S^T (value channel v on the 128 TMEM lanes,
// key channel k on 128 fp32 columns), so that the small, per-chunk matrices
// are the tcgen05 A operands (read from TMEM) and the chunk record's wide
// matrices are B operands read in place from shared memory.  Per chunk i, with
// the record written by the chunk kernel:
//   X^T   = S^T . [W ; scale*Qhat]^T        (MMA1: A = bf16 S^T in TMEM, N = 128, K = 128,
//                                            into accumulator X[i % 2])
//   Delta = U - X_W                         (v_new; bf16 Delta^T to TMEM)
//   S^T  += Delta^T . Ktilde                (MMA2s: N = 128, K = 64; S^T was decayed by
//                                            Diag(exp(G_last)) beforehand)
//   X_Q  += Delta^T . Aqk_hi^T + Delta^T . Aqk_lo^T   (MMA2o: N = 64, K = 64, twice)
//   O^T   = X_Q
// This is the gated delta rule unrolled over the chunk
// (reading of "Flashkda Delta Attention", "Core Kernel API": recurrent state
// updates of delta attention).  A K=16 tcgen05 MMA costs about 44 cycles for
// N <= 64 on GB300 and 67 at N = 128, so wide MMAs on the chain (8 + 4
// instructions per chunk) replace the ~12 narrow ones a value-sliced
// formulation needs there.  Only MMA1, Delta and MMA2s are on the sequential
// chain: MMA2o runs while the next snapshot is taken.
//
// Warp roles (448 threads): warps 0-7 are chain warps -- warp w owns TMEM lane
// quarter w % 4 (32 value channels) and half w / 4 of the columns it touches
// (state columns, or the chunk's tokens) and takes the snapshot and Delta;
// warp 8 streams whole records with one bulk copy each into a 2-stage ring;
// warp 9 issues the MMAs; warps 10-13 (one per lane quarter) move the outputs
// of chunk i out of X[i % 2] while later chunks run, transposing them through
// shared memory into whole 256-byte token rows, and release X[i % 2] for
// MMA1(i + 2).  Every mbarrier wait is bounded; on timeout the CTA records
// kStatusTimeout, stops, drains its own copies and frees TMEM.
#pragma once
#include <cuda_runtime.h>

#include "kda_internal.h"
#include "tc.cuh"

namespace kda {
namespace recur_t {


constexpr int kEpiWarps = 8;
constexpr int kOutWarps = 4;
constexpr int kThreads = 32 * (kEpiWarps + 2 + kOutWarps);
constexpr int kWarpProducer = kEpiWarps, kWarpMma = kEpiWarps + 1, kWarpOut0 = kEpiWarps + 2;
constexpr int kStages = 2;
constexpr uint32_t kStageBytes = kRecBytes;          // a whole record per stage
constexpr uint32_t kTileO = kChunk * kDim * 2;       // output tile, bf16 [64 tokens][128 v]
constexpr uint32_t kSmemO = kStages * kStageBytes;   // two output tiles
constexpr uint32_t kSmemBytes = kSmemO + 2 * kTileO;
// TMEM columns
constexpr uint32_t kColS = 0;      // S^T, fp32, 128 columns
constexpr uint32_t kColX0 = 128;   // X[0] = [X_W | X_Q] (+ the output updates), 128 columns
constexpr uint32_t kColSb = 256;   // bf16 S^T snapshot (A of MMA1), 64 columns
constexpr uint32_t kColDb = 320;   // bf16 Delta^T (A of MMA2s / MMA2o), 32 columns
constexpr uint32_t kColX1 = 384;   // X[1]
constexpr uint32_t kTmemCols = 512;
__device__ __forceinline__ uint32_t col_x(int i) { return (i & 1) ? kColX1 : kColX0; }

struct RecurTArgs {
    void* out;  // bf16 [tokens, H, 128]
    const void* h0;
    void* hT;
    int h0_dtype;  // kda_dtype_t of h0 / hT (KDA_DTYPE_NONE: absent)
    int hT_dtype;
    int H;
    int N;
    const int32_t* flags;
    const int32_t* chunk_off;
    const ChunkInfo* info;
    const uint8_t* records;
    int* status;
};

// One thread's 64 state elements S[k0 + j][v] (j < 64, row stride kDim), in
// the caller's dtype; the dtype branch is taken once, outside the loops.
template <typename T>
__device__ __forceinline__ void state_ld64(const void* p, size_t base, uint32_t (&r)[64]) {
    const T* s = reinterpret_cast<const T*>(p) + base;
#pragma unroll
    for (int j = 0; j < 64; ++j) {
        if constexpr (sizeof(T) == 4)
            r[j] = __float_as_uint(s[(size_t)j * kDim]);
        else
            r[j] = __float_as_uint(__bfloat162float(s[(size_t)j * kDim]));
    }
}
template <typename T>
__device__ __forceinline__ void state_st16(void* p, size_t base, const uint32_t (&r)[16]) {
    T* s = reinterpret_cast<T*>(p) + base;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        if constexpr (sizeof(T) == 4)
            s[(size_t)j * kDim] = __uint_as_float(r[j]);
        else
            s[(size_t)j * kDim] = __float2bfloat16_rn(__uint_as_float(r[j]));
    }
}

// The barrier after the initial state load uses id bar_all + kBarStateOffset.
constexpr uint32_t kBarStateOffset = 4;
// Barrier over the kThreads threads of the recurrence block (and its
// non-waiting arrival).
__device__ __forceinline__ void all_sync(uint32_t bar_id) {
    asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "n"(kThreads) : "memory");
}
__device__ __forceinline__ void all_arrive(uint32_t bar_id) {
    asm volatile("bar.arrive %0, %1;" ::"r"(bar_id), "n"(kThreads) : "memory");
}
__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
// Wait (bounded by `limit` ns) until *flag is non-zero.
__device__ __forceinline__ bool wait_flag(const int* flag, uint64_t limit) {
    if (ld_acquire_gpu(flag) != 0) return true;
    const uint64_t t0 = global_ns();
    while (true) {
        for (int i = 0; i < 16; ++i) {
            __nanosleep(64);
            if (ld_acquire_gpu(flag) != 0) return true;
        }
        if (global_ns() - t0 > limit) return false;
    }
}

// Each record reaches its ring slot in two parts.  Part A (W and scale*Q o E,
// U^T, exp(G_last)) is what a chunk needs first, and its readers are done once
// the chunk's Delta is computed; part B ((K o F)^T and scale*Aqk) is needed only
// for the state update and the outputs.  So part A of chunk i + 2 is copied as
// soon as chunk i has computed Delta, over a chunk ahead of its use, and part B
// once chunk i's MMAs are done: a record copy no longer has to fit in one
// chunk's processing time (with the fused launch's memory traffic it did not).
constexpr uint32_t kPartA0 = kRecWQ, kPartA0Bytes = kRecKT - kRecWQ;        // W, Q
constexpr uint32_t kPartA1 = kRecUT, kPartA1Bytes = kRecBytes - kRecUT;     // U^T, gamma
constexpr uint32_t kPartB = kRecKT, kPartBBytes = kRecUT - kRecKT;          // K^T, Aqk hi/lo
static_assert(kPartA0Bytes + kPartA1Bytes + kPartBBytes == kRecBytes, "record parts");
static_assert(kRecWQ == 0 && kRecKT < kRecAQ && kRecAQ < kRecAQL && kRecAQL < kRecUT &&
                  kRecUT < kRecGam,
              "part A = [0, KT) + [UT, end), part B = [KT, UT)");

// Small per-block state that lives outside the dynamic shared-memory area.
// full/fullB: parts A/B of a record landed; emptyA: part A of the slot read
// (Delta computed); empty: the slot's MMAs done; s_ready[r]: round r of the snapshot written (key
// channels 64 h + 32 r .. + 31 of both halves h); mma1: X^T ready;
// d_ready: Delta^T written; mma2s: state updated; mma2o[b]: outputs of the
// chunk in X[b] complete; x_free[b]: the output warps have read X[b];
// tile_full[b]: output tile b is written; mma_done: every MMA the block
// issued has completed (waited for once, before TMEM is freed)
struct RecurTShared {
    uint64_t full[kStages], fullB[kStages], emptyA[kStages], empty[kStages], s_ready[2], mma1,
        d_ready, mma2s, mma2o[2], x_free[2], tile_full[2], mma_done;
    uint32_t tmem_base;
    int s_abort;
};

// 8 / 16 packed columns to TMEM (one lane per thread)
__device__ __forceinline__ void tmem_st8(uint32_t ta, const uint32_t (&r)[8]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(ta),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
        : "memory");
}

// Bounded wait that records a timeout and raises the CTA's abort flag.  When a
// whole warp waits, its lanes see the same barrier state and time in the same
// instructions, so they leave the loop together.
#define WAIT_OR_ABORT(bar, parity)                  \
    if (!mbar_wait((bar), (parity), lim)) {         \
        atomicOr(P.status, kStatusTimeout);         \
        S.s_abort = 1;                             \
        break;                                      \
    }

// The recurrence of (sequence, head) pair `pair` on kThreads threads (thread
// index `tid`), with the shared-memory area `sm` (kSmemBytes, 1024-byte
// aligned) and the small state `S`, synchronised by named barriers `bar_all`
// and bar_all + kBarStateOffset (mbarriers elsewhere).  With `ready` non-null the record
// of (chunk c, head h) is copied only once ready[c * H + h] is set.
__device__ __forceinline__ void recur_t_body(const RecurTArgs& P, uint8_t* sm, RecurTShared& S,
                                             const int tid, const uint32_t bar_all,
                                             const int pair, const int* ready) {
    if (P.flags[0] != 1) return;
    // a CTA that already gave up on a bounded wait poisons the launch: skip the
    // rest (decided once, so every thread takes the same path)
    if (tid == 0) S.s_abort = (*((volatile int*)P.status) & kStatusTimeout) ? 1 : 0;
    all_sync(bar_all);
    if (S.s_abort) return;
    const uint64_t lim = wait_limit_ns(P.status);  // of every wait that may give up
    const int H = P.H;
    const int h = pair % H;
    const int n = pair / H;
    const int c_begin = P.chunk_off[n];
    const int nchunks = P.chunk_off[n + 1] - c_begin;
    const int warp = tid >> 5, lane = tid & 31;
    const size_t state_base = ((size_t)n * H + h) * kDim * kDim;
    // The chain warps issue their initial-state loads first, so the DRAM
    // latency overlaps the TMEM allocation and barrier set-up.  Thread (q, hc)
    // holds S^T[v][k] = h0[k][v] for v = 32 q + lane and its 64 k.
    uint32_t st0[64];
    if (warp < kEpiWarps) {
        const size_t b0 = state_base + (size_t)(64 * (warp >> 2)) * kDim + 32 * (warp & 3) + lane;
        if (P.h0_dtype == KDA_DTYPE_FP32)
            state_ld64<float>(P.h0, b0, st0);
        else if (P.h0_dtype == KDA_DTYPE_BF16)
            state_ld64<__nv_bfloat16>(P.h0, b0, st0);
        else
#pragma unroll
            for (int j = 0; j < 64; ++j) st0[j] = 0u;
    }

    if (warp == 0) {
        tmem_alloc(&S.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&S.full[s], 1);
            mbar_init(&S.fullB[s], 1);
            mbar_init(&S.emptyA[s], 32 * kEpiWarps);
            mbar_init(&S.empty[s], 1);
        }
        mbar_init(&S.s_ready[0], 32 * kEpiWarps);
        mbar_init(&S.s_ready[1], 32 * kEpiWarps);
        mbar_init(&S.mma1, 1);
        mbar_init(&S.d_ready, 32 * kEpiWarps);
        mbar_init(&S.mma2s, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&S.mma2o[b], 1);
            mbar_init(&S.x_free[b], 32 * kOutWarps);
            mbar_init(&S.tile_full[b], 32 * kOutWarps);
        }
        mbar_init(&S.mma_done, 1);
        mbar_fence_init();
        S.s_abort = 0;
    }
    tc_fence_before();
    all_sync(bar_all);
    tc_fence_after();
    const uint32_t tbase = S.tmem_base;

    if (warp < kEpiWarps) {
        // -------------------------------------------------------- epilogue warps
        const int q = warp & 3, hc = warp >> 2;
        const int v = 32 * q + lane;  // value channel = TMEM lane
        const uint32_t lane_base = taddr(tbase, 32u * q, 0);
        // initial state (loaded above) to TMEM
#pragma unroll
        for (int c0 = 0; c0 < 64; c0 += 16)
            tmem_st16(lane_base + kColS + 64 * hc + c0,
                      *reinterpret_cast<const uint32_t(*)[16]>(st0 + c0));
        tmem_wait_st();
        tc_fence_before();
        all_sync(bar_all + kBarStateOffset);
        tc_fence_after();

        int i = 0;
        for (; i < nchunks; ++i) {
            const int s = i % kStages;
            const uint32_t ph = (uint32_t)(i & 1);
            const uint8_t* st = sm + s * kStageBytes;
            WAIT_OR_ABORT(&S.full[s], (uint32_t)((i / kStages) & 1));
            // snapshot in two rounds of 32 key channels: the bf16 S^T columns
            // MMA1 reads are written and signalled first (MMA1 starts on round 0's
            // K-steps while round 1 is converted); the chunk decay
            // S^T <- S^T Diag(gamma), which only MMA2s needs, follows off that path
            // (the wait::st before d_ready covers its stores)
            {
                const float4* gam4 =
                    reinterpret_cast<const float4*>(st + kRecGam) + 16 * hc;  // 64 channels
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const uint32_t c0 = 64 * hc + 32 * r;  // first key channel of the round
                    uint32_t x[2][16];
                    tmem_ld16(lane_base + kColS + c0, x[0]);
                    tmem_ld16(lane_base + kColS + c0 + 16, x[1]);
                    tmem_wait_ld();
                    reg_fence16(x[0]);
                    reg_fence16(x[1]);
                    uint32_t pk[16];
#pragma unroll
                    for (int u = 0; u < 16; ++u)
                        pk[u] = pack_bf16(__uint_as_float(x[u >> 3][(2 * u) & 15]),
                                          __uint_as_float(x[u >> 3][(2 * u + 1) & 15]));
                    tmem_st16(lane_base + kColSb + c0 / 2, pk);
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(&S.s_ready[r]);
#pragma unroll
                    for (int g = 0; g < 2; ++g) {
#pragma unroll
                        for (int w = 0; w < 4; ++w) {
                            const float4 g4 = gam4[8 * r + 4 * g + w];
                            x[g][4 * w + 0] = __float_as_uint(__uint_as_float(x[g][4 * w + 0]) * g4.x);
                            x[g][4 * w + 1] = __float_as_uint(__uint_as_float(x[g][4 * w + 1]) * g4.y);
                            x[g][4 * w + 2] = __float_as_uint(__uint_as_float(x[g][4 * w + 2]) * g4.z);
                            x[g][4 * w + 3] = __float_as_uint(__uint_as_float(x[g][4 * w + 3]) * g4.w);
                        }
                        tmem_st16(lane_base + kColS + c0 + 16 * g, x[g]);
                    }
                }
            }
            // Delta^T[v][t] = U[t][v] - X_W[v][t] for this thread's 32 tokens
            uint32_t uw[16];
            {
                const uint4* up = reinterpret_cast<const uint4*>(st + kRecUT + v * 128 + 64 * hc);
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const uint4 x = up[w];
                    uw[4 * w + 0] = x.x;
                    uw[4 * w + 1] = x.y;
                    uw[4 * w + 2] = x.z;
                    uw[4 * w + 3] = x.w;
                }
            }
            WAIT_OR_ABORT(&S.mma1, ph);
            tc_fence_after();
            {
                uint32_t r[2][16];
                tmem_ld16(lane_base + col_x(i) + 32 * hc, r[0]);
                tmem_ld16(lane_base + col_x(i) + 32 * hc + 16, r[1]);
                tmem_wait_ld();
                reg_fence16(r[0]);
                reg_fence16(r[1]);
                uint32_t pk[16];
#pragma unroll
                for (int u = 0; u < 32; u += 2) {
                    const uint32_t uu = uw[u / 2];
                    const float x0 = __uint_as_float(r[u >> 4][u & 15]);
                    const float x1 = __uint_as_float(r[u >> 4][(u & 15) + 1]);
                    pk[u / 2] = pack_bf16(bf16_lo(uu) - x0, bf16_hi(uu) - x1);
                }
                tmem_st16(lane_base + kColDb + 16 * hc, pk);
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&S.d_ready);
                // gamma and U^T are read and MMA1 (the reader of W, Q) has completed:
                // part A of the slot may take chunk i + 2's
                mbar_arrive(&S.emptyA[s]);
            }
            WAIT_OR_ABORT(&S.mma2s, ph);
            tc_fence_after();
        }
        if (!*((volatile int*)&S.s_abort)) {
            if (P.hT_dtype != KDA_DTYPE_NONE) {
#pragma unroll
                for (int c0 = 0; c0 < 64; c0 += 16) {
                    uint32_t r[16];
                    tmem_load16(lane_base + kColS + 64 * hc + c0, r);
                    const size_t b0 = state_base + (size_t)(64 * hc + c0) * kDim + v;
                    if (P.hT_dtype == KDA_DTYPE_FP32)
                        state_st16<float>(P.hT, b0, r);
                    else
                        state_st16<__nv_bfloat16>(P.hT, b0, r);
                }
            }
        }
    } else {
        // matches the chain warps' barrier after the initial state; the producer
        // only arrives (it touches no TMEM), so the first record copies overlap
        // the state load
        // (its own barrier id: the producer may reach the final barrier first)
        tc_fence_before();
        if (warp == kWarpProducer)
            all_arrive(bar_all + kBarStateOffset);
        else
            all_sync(bar_all + kBarStateOffset);
        tc_fence_after();
        if (warp == kWarpProducer) {
            // ---------------------------------------------------- producer
            if (lane == 0) {
                int fillsA[kStages] = {0, 0}, fillsB[kStages] = {0, 0};
                // a record is dead once copied: its lines may leave L2 first
                const uint64_t pol_rec = l2_policy_evict_first();
                constexpr int kAhead = kStages + 2;  // records pulled into L2 ahead
                if (!ready)
                    for (int i = 0; i < kAhead && i < nchunks; ++i)
                        bulk_prefetch_l2(P.records + ((size_t)(c_begin + i) * H + h) * kRecBytes,
                                         kRecBytes);
                for (int i = 0; i < nchunks; ++i) {
                    const int s = i % kStages;
                    uint8_t* dst = sm + s * kStageBytes;
                    const uint8_t* rec = P.records + ((size_t)(c_begin + i) * H + h) * kRecBytes;
                    // part A once the chunk last in this slot has computed its Delta
                    if (fillsA[s] > 0) WAIT_OR_ABORT(&S.emptyA[s], (uint32_t)((fillsA[s] - 1) & 1));
                    if (*((volatile int*)&S.s_abort)) break;
                    if (!ready && i + kAhead < nchunks)
                        bulk_prefetch_l2(
                            P.records + ((size_t)(c_begin + i + kAhead) * H + h) * kRecBytes,
                            kRecBytes);
                    if (ready) {
                        // the record is written by a chunk-kernel worker of the same launch
                        if (!wait_flag(ready + (size_t)(c_begin + i) * H + h, lim)) {
                            atomicOr(P.status, kStatusTimeout);
                            S.s_abort = 1;
                            break;
                        }
                        // the acquired view of the record before the bulk copy's reads
                        fence_async_global();
                    }
                    mbar_arrive_expect_tx(&S.full[s], kPartA0Bytes + kPartA1Bytes);
                    bulk_g2s_hint(dst + kPartA0, rec + kPartA0, kPartA0Bytes, &S.full[s], pol_rec);
                    bulk_g2s_hint(dst + kPartA1, rec + kPartA1, kPartA1Bytes, &S.full[s], pol_rec);
                    ++fillsA[s];
                    // part B once that chunk's MMAs are done
                    if (fillsB[s] > 0) WAIT_OR_ABORT(&S.empty[s], (uint32_t)((fillsB[s] - 1) & 1));
                    if (*((volatile int*)&S.s_abort)) break;
                    mbar_arrive_expect_tx(&S.fullB[s], kPartBBytes);
                    bulk_g2s_hint(dst + kPartB, rec + kPartB, kPartBBytes, &S.fullB[s], pol_rec);
                    ++fillsB[s];
                }
                // drain: every issued fill must have landed before the CTA exits
                for (int s = 0; s < kStages; ++s) {
                    if (fillsA[s] > 0 && !mbar_drain(&S.full[s], (uint32_t)((fillsA[s] - 1) & 1)))
                        atomicOr(P.status, kStatusTimeout);
                    if (fillsB[s] > 0 && !mbar_drain(&S.fullB[s], (uint32_t)((fillsB[s] - 1) & 1)))
                        atomicOr(P.status, kStatusTimeout);
                }
            }
        } else if (warp == kWarpMma) {
            // ---------------------------------------------------- MMA issuer
            const uint32_t idesc1 = idesc_bf16_f32(128, 128, false, true);
            const uint32_t idesc2 = idesc_bf16_f32(128, 128, false, false);
            const uint32_t idesc3 = idesc_bf16_f32(128, 64, false, false);
            const uint32_t st0 = smem_addr(sm);
            // B operands of stage 0; stage s adds s * kStageBytes to the address
            // field (bytes >> 4), one K=16 step adds 256 B (16)
            const uint64_t dWQ0 = smem_desc(st0 + kRecWQ, 128, 2048);
            const uint64_t dKT0 = smem_desc(st0 + kRecKT, 128, 1024);
            const uint64_t dAQ0 = smem_desc(st0 + kRecAQ, 128, 1024);   // Aqk hi
            const uint64_t dAQL0 = smem_desc(st0 + kRecAQL, 128, 1024); // Aqk lo
            constexpr uint64_t kStageStep = kStageBytes >> 4;
            for (int i = 0; i < nchunks; ++i) {
                const int s = i % kStages;
                const uint32_t ph = (uint32_t)(i & 1);
                const uint64_t so = (uint64_t)s * kStageStep;
                const uint32_t tX = tbase + col_x(i);
                WAIT_OR_ABORT(&S.full[s], (uint32_t)((i / kStages) & 1));
                // X[i % 2] still holds the outputs of chunk i - 2 until they are read
                if (i >= 2) WAIT_OR_ABORT(&S.x_free[i & 1], (uint32_t)(((i - 2) >> 1) & 1));
                // MMA1 in two halves: the K-steps of snapshot round 0 (key channels
                // 0-31 and 64-95) as soon as it lands, then those of round 1
                WAIT_OR_ABORT(&S.s_ready[0], ph);
                tc_fence_after();
                if (elect_one()) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int kk = (j & 1) + 4 * (j >> 1);  // 0, 1, 4, 5
                        mma_bf16_ta(tX, tbase + kColSb + 8 * kk, dWQ0 + so + 16u * kk, idesc1,
                                    j > 0 ? 1u : 0u);
                    }
                }
                __syncwarp();
                WAIT_OR_ABORT(&S.s_ready[1], ph);
                tc_fence_after();
                if (elect_one()) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int kk = 2 + (j & 1) + 4 * (j >> 1);  // 2, 3, 6, 7
                        mma_bf16_ta(tX, tbase + kColSb + 8 * kk, dWQ0 + so + 16u * kk, idesc1, 1u);
                    }
                    mma_commit(&S.mma1);
                }
                __syncwarp();
                WAIT_OR_ABORT(&S.d_ready, ph);
                WAIT_OR_ABORT(&S.fullB[s], (uint32_t)((i / kStages) & 1));
                tc_fence_after();
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_bf16_ta(tbase + kColS, tbase + kColDb + 8 * kk, dKT0 + so + 16u * kk,
                                    idesc2, 1u);
                    mma_commit(&S.mma2s);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_bf16_ta(tX + 64, tbase + kColDb + 8 * kk, dAQ0 + so + 16u * kk, idesc3,
                                    1u);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_bf16_ta(tX + 64, tbase + kColDb + 8 * kk, dAQL0 + so + 16u * kk,
                                    idesc3, 1u);
                    mma_commit(&S.mma2o[i & 1]);
                    mma_commit(&S.empty[s]);
                }
                __syncwarp();
            }
            // every MMA issued above has completed before TMEM is freed (after
            // a normal end the consumers already waited for them; after giving
            // up some may still be running)
            if (elect_one()) mma_commit(&S.mma_done);
            __syncwarp();
            if (!mbar_drain(&S.mma_done, 0)) atomicOr(P.status, kStatusTimeout);
        } else {
            // ---------------------------------------------------- output warps
            const int q = warp & 3;          // TMEM lane quarter
            const int v = 32 * q + lane;     // value channel
            const int ot = tid - 32 * kWarpOut0;  // 0..127
            for (int i = 0; i < nchunks; ++i) {
                const int b = i & 1;
                WAIT_OR_ABORT(&S.mma2o[b], (uint32_t)((i >> 1) & 1));
                tc_fence_after();
                __nv_bfloat16* tile = reinterpret_cast<__nv_bfloat16*>(sm + kSmemO + b * kTileO);
#pragma unroll
                for (int c0 = 0; c0 < 64; c0 += 32) {
                    uint32_t r[2][16];
                    tmem_ld16(taddr(tbase, 32u * q, col_x(i) + 64 + c0), r[0]);
                    tmem_ld16(taddr(tbase, 32u * q, col_x(i) + 64 + c0 + 16), r[1]);
                    tmem_wait_ld();
                    reg_fence16(r[0]);
                    reg_fence16(r[1]);
#pragma unroll
                    for (int u = 0; u < 32; ++u)
                        tile[(c0 + u) * kDim + v] = __float2bfloat16_rn(__uint_as_float(r[u >> 4][u & 15]));
                }
                tc_fence_before();
                mbar_arrive(&S.x_free[b]);  // MMA1(i + 2) may overwrite X[b]
                // the whole tile is written (every thread arrives for chunk i only
                // after its stores of chunk i - 1, so tile b is free again here)
                mbar_arrive(&S.tile_full[b]);
                WAIT_OR_ABORT(&S.tile_full[b], (uint32_t)((i >> 1) & 1));
                const ChunkInfo ci = P.info[c_begin + i];
#pragma unroll
                for (int it = 0; it < (int)(kTileO / 16) / (32 * kOutWarps); ++it) {
                    const int e = ot + 32 * kOutWarps * it;  // 16-byte piece
                    const int t = e >> 4, piece = e & 15;
                    if (t < ci.len)
                        reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(P.out) +
                                                 ((size_t)(ci.tok0 + t) * H + h) * kDim)[piece] =
                            reinterpret_cast<const uint4*>(tile + t * kDim)[piece];
                }
            }
        }
    }
    tc_fence_before();
    all_sync(bar_all);
    if (warp == 0) tmem_dealloc(tbase, kTmemCols);
}


#undef WAIT_OR_ABORT

inline RecurTArgs make_recur_t_args(const Problem& p, const Workspace& ws, int* status) {
    RecurTArgs a;
    a.out = p.out;
    a.h0 = p.h0;
    a.hT = p.hT;
    a.h0_dtype = p.h0_dtype;
    a.hT_dtype = p.hT_dtype;
    a.H = p.H;
    a.N = p.N;
    a.flags = ws.flags;
    a.chunk_off = ws.chunk_off;
    a.info = ws.info;
    a.records = ws.records;
    a.status = status;
    return a;
}

}  // namespace recur_t
}  // namespace kda
