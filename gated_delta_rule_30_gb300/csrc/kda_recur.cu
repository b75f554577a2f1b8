// kda_recur.cu -- recurrence kernel of the KDA forward pass: the sequential
// chunk-to-chunk state update for one (sequence, head, value slice).
//
// Per chunk, with S the K x VS state slice entering it (fp32, kept in TMEM:
// lane = key channel, column = value channel) and the chunk record written by
// the chunk kernel:
//   X     = [W ; scale*Qhat] . S                  (tcgen05, M=128, K=128)
//   Delta = U - X[0:64]                           (v_new, fp32 -> bf16)
//   S     = Diag(exp(G_last)) S + Ktilde^T . Delta   (tcgen05, M=128, K=64)
//   O     = X[64:128] + scale*Aqk . Delta         (tcgen05, accumulated in X;
//                                                  Aqk as a bf16 hi + lo pair)
// which is the unrolled gated delta rule over the chunk (reading of "Flashkda
// Delta Attention", "Core Kernel API": recurrent state updates; the value
// dimension splits exactly because column j of S, Delta and O depends only on
// column j).  The decay is applied in TMEM while the bf16 snapshot of S used
// by the first product is taken, so each chunk costs two dependent MMA
// rounds.
//
// Warp roles (256 threads): warps 0-3 own the 4 TMEM lane quarters (state
// snapshot / decay, Delta for rows 0-63, state I/O); warp 4 streams records
// with bulk copies into a 2- or 3-stage ring (and prefetches upcoming records
// into L2); warp 5 issues the MMAs; warps 6-7 (lane quarters 2-3, the output
// rows of X) write the outputs of chunk j from X[j % 2] while later chunks
// run and then release that buffer to the MMA warp.  Only X = [W;Q].S, Delta
// and the state update are on the sequential chain; the output update for
// chunk i has its own barriers and is issued right after the state update, so
// the tensor pipe (which runs a CTA's MMAs in issue order) executes it while
// the next snapshot is taken.  Every mbarrier wait is bounded; on timeout the
// CTA records kStatusTimeout, stops, waits (bounded) for its own copies and
// frees TMEM.
//
// Map mode (kMap, segmented path): the grid holds twice the slices of each
// (segment, head).  Slices [0, 128/VS) start from a zero state and give X, the
// state the segment reaches from zero; slices [128/VS, 256/VS) start from the
// identity with U taken as zero (Delta = -X[0:64]) and give the linear part M
// of the segment's state map, since each value column evolves by
// s <- (Diag(gamma) - Ktilde^T W) s + Ktilde^T u.  No outputs are formed
// (the output product and the output warps are skipped); the final slice is
// stored as X [k][v] or as M^T [j][k].
#include <cuda_runtime.h>

#include <type_traits>

#include "kda_internal.h"
#include "tc.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;

template <int VS>
struct RecurLayout {
    // the first kRecOperands bytes mirror the record: WQ, KT, AQ hi, AQ lo
    static constexpr uint32_t kStageWQ = kRecWQ;
    static constexpr uint32_t kStageKT = kRecKT;
    static constexpr uint32_t kStageAQ = kRecAQ;
    static constexpr uint32_t kStageAQL = kRecAQL;
    static constexpr uint32_t kStageUT = kRecOperands;               // VS x 128 B
    static constexpr uint32_t kStageGam = kRecOperands + VS * 128;   // 512 B
    static constexpr uint32_t kStageBytes = kStageGam + 512;
    // ring depth: three stages when they fit next to the snapshot and Delta buffers
    static constexpr int kStages = (3 * kStageBytes + VS * 256 + 2 * VS * 128 <= 232448) ? 3 : 2;
    static constexpr uint32_t kSb = kStages * kStageBytes;  // S snapshot, K=128 x N=VS, MN-major
    static constexpr uint32_t kDb = kSb + VS * 256;         // 2 x Delta, K=64 x N=VS, MN-major
    static constexpr uint32_t kBytes = kDb + 2 * VS * 128;
    static constexpr uint32_t kLoadBytes = kRecOperands + VS * 128 + 512;
    static constexpr uint32_t kTmemCols = (3 * VS <= 128) ? 128 : (3 * VS <= 256 ? 256 : 512);
};

struct RecurArgs {
    void* out;  // bf16 [tokens, H, 128]
    const void* h0;
    void* hT;
    int H;
    int N;
    const int32_t* flags;
    const int32_t* chunk_off;
    const ChunkInfo* info;
    const uint8_t* records;
    int* status;
};

template <typename T>
struct StateIO;
template <>
struct StateIO<float> {
    static __device__ __forceinline__ void load16(const void* base, size_t off, uint32_t (&r)[16]) {
        const float4* p = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(base) + off);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 x = p[i];
            r[4 * i + 0] = __float_as_uint(x.x);
            r[4 * i + 1] = __float_as_uint(x.y);
            r[4 * i + 2] = __float_as_uint(x.z);
            r[4 * i + 3] = __float_as_uint(x.w);
        }
    }
    static __device__ __forceinline__ void store16(void* base, size_t off, const uint32_t (&r)[16]) {
        float4* p = reinterpret_cast<float4*>(reinterpret_cast<float*>(base) + off);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            p[i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                               __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
    }
};
template <>
struct StateIO<__nv_bfloat16> {
    static __device__ __forceinline__ void load16(const void* base, size_t off, uint32_t (&r)[16]) {
        const uint4* p =
            reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(base) + off);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const uint4 x = p[i];
            const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                r[8 * i + 2 * j] = __float_as_uint(bf16_lo(w[j]));
                r[8 * i + 2 * j + 1] = __float_as_uint(bf16_hi(w[j]));
            }
        }
    }
    static __device__ __forceinline__ void store16(void* base, size_t off, const uint32_t (&r)[16]) {
        uint4* p = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(base) + off);
#pragma unroll
        for (int i = 0; i < 2; ++i)
            p[i] = make_uint4(pack_bf16(__uint_as_float(r[8 * i + 0]), __uint_as_float(r[8 * i + 1])),
                              pack_bf16(__uint_as_float(r[8 * i + 2]), __uint_as_float(r[8 * i + 3])),
                              pack_bf16(__uint_as_float(r[8 * i + 4]), __uint_as_float(r[8 * i + 5])),
                              pack_bf16(__uint_as_float(r[8 * i + 6]), __uint_as_float(r[8 * i + 7])));
    }
};
struct NoState {};

// Bounded wait that records a timeout and raises the CTA's abort flag.  When a
// whole warp waits, its lanes see the same barrier state and time in the same
// instructions, so they leave the loop together.
#define WAIT_OR_ABORT(bar, parity)                  \
    if (!mbar_wait((bar), (parity), lim)) {         \
        atomicOr(P.status, kStatusTimeout);         \
        s_abort = 1;                             \
        break;                                      \
    }

// H0 / HT: float, __nv_bfloat16 or NoState; kMap: map mode (H0 = NoState, HT = float)
template <int VS, typename H0, typename HT, bool kMap = false>
__global__ void __launch_bounds__(kThreads, 1) recur_kernel(const RecurArgs P) {
    using L = RecurLayout<VS>;
    constexpr int kSlices = kDim / VS;
    constexpr int kGridSlices = kMap ? 2 * kSlices : kSlices;
    extern __shared__ __align__(1024) uint8_t sm[];
    // full/empty: record ring; s_ready: snapshot written; mma1: X = [W;Q].S done;
    // d_ready: Delta written; mma2s: state update done; mma2o[b]: output update
    // of the chunk in X[b] done; x_free[b]: the output warps have read X[b];
    // mma_done: every MMA the CTA issued has completed (before TMEM is freed)
    constexpr int NS = L::kStages;
    __shared__ uint64_t full[NS], empty[NS], s_ready, mma1, d_ready, mma2s, mma2o[2], x_free[2],
        mma_done;
    __shared__ uint32_t tmem_base;
    __shared__ int s_abort;

    if (P.flags[0] != 1) return;
    // a CTA that already gave up on a bounded wait poisons the launch: skip the
    // rest (decided once, so every thread takes the same path)
    if (threadIdx.x == 0) s_abort = (*((volatile int*)P.status) & kStatusTimeout) ? 1 : 0;
    __syncthreads();
    if (s_abort) return;
    const uint64_t lim = wait_limit_ns(P.status);  // of every wait that may give up
    const int H = P.H;
    const int gslice = blockIdx.x % kGridSlices;
    const bool lin = kMap && gslice >= kSlices;  // map mode: this CTA evolves the identity
    const int slice = lin ? gslice - kSlices : gslice;
    const int nh = blockIdx.x / kGridSlices;
    const int h = nh % H;
    const int n = nh / H;
    const int v0 = slice * VS;
    const int c_begin = P.chunk_off[n];
    const int nchunks = P.chunk_off[n + 1] - c_begin;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // ---------------------------------------------------------------- set-up
    if (warp == 0) {
        tmem_alloc(&tmem_base, L::kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(&s_ready, 128);
        mbar_init(&mma1, 1);
        mbar_init(&d_ready, 64);
        mbar_init(&mma2s, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&mma2o[b], 1);
            mbar_init(&x_free[b], 64);
        }
        mbar_init(&mma_done, 1);
        mbar_fence_init();
        s_abort = 0;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tmem_base;
    const uint32_t tS = tbase;  // columns [0, VS); X[b] at [VS (1 + b), VS (2 + b))
    const size_t state_base = (kMap ? (size_t)nh * 2 + (lin ? 1 : 0) : (size_t)nh) * kDim * kDim;

    // initial state -> TMEM (thread = key channel)
    if (warp < 4) {
        const int ch = tid;
#pragma unroll
        for (int c0 = 0; c0 < VS; c0 += 16) {
            uint32_t r[16];
            if constexpr (kMap) {
#pragma unroll
                for (int u = 0; u < 16; ++u)
                    r[u] = (lin && ch == v0 + c0 + u) ? __float_as_uint(1.f) : 0u;
            } else if constexpr (std::is_same<H0, NoState>::value) {
#pragma unroll
                for (int u = 0; u < 16; ++u) r[u] = 0u;
            } else {
                StateIO<H0>::load16(P.h0, state_base + (size_t)ch * kDim + v0 + c0, r);
            }
            tmem_st16(taddr(tS, 32u * warp, (uint32_t)c0), r);
        }
        tmem_wait_st();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (warp == 4) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int fills[NS];
            for (int s = 0; s < NS; ++s) fills[s] = 0;
            constexpr int kAhead = NS + 2;  // records pulled into L2 this many chunks ahead
            for (int i = 0; i < kAhead && i < nchunks; ++i)
                bulk_prefetch_l2(P.records + ((size_t)(c_begin + i) * H + h) * kRecBytes,
                                 kRecBytes);
            for (int i = 0; i < nchunks; ++i) {
                const int s = i % NS;
                if (fills[s] > 0) WAIT_OR_ABORT(&empty[s], (uint32_t)((fills[s] - 1) & 1));
                if (*((volatile int*)&s_abort)) break;
                if (i + kAhead < nchunks)
                    bulk_prefetch_l2(
                        P.records + ((size_t)(c_begin + i + kAhead) * H + h) * kRecBytes,
                        kRecBytes);
                uint8_t* st = sm + s * L::kStageBytes;
                const uint8_t* rec = P.records + ((size_t)(c_begin + i) * H + h) * kRecBytes;
                mbar_arrive_expect_tx(&full[s], L::kLoadBytes);
                bulk_g2s(st, rec, kRecOperands, &full[s]);
                bulk_g2s(st + L::kStageUT, rec + kRecUT + v0 * 128, VS * 128, &full[s]);
                bulk_g2s(st + L::kStageGam, rec + kRecGam, 512, &full[s]);
                ++fills[s];
            }
            // drain: every issued fill must have landed before the CTA exits
            for (int s = 0; s < NS; ++s)
                if (fills[s] > 0 && !mbar_drain(&full[s], (uint32_t)((fills[s] - 1) & 1)))
                    atomicOr(P.status, kStatusTimeout);
        }
    } else if (warp == 5) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs the loop (descriptors stay warp-uniform); one
        // elected lane issues.  Per chunk i the critical chain is
        //   MMA1(i): X = [W;Q].S  ->  (Delta)  ->  MMA2s(i): S += Kt^T.Delta
        // and the output update MMA2o(i): X[64:] += Aqk.Delta (hi and lo) has
        // its own barrier, so the next snapshot never waits for it.
        const uint32_t idesc1 = idesc_bf16_f32(128, VS, true, true);
        const uint32_t idesc2 = idesc_bf16_f32(128, VS, false, true);
        // Descriptors of stage 0 / Delta buffer 0; the other stage (buffer) is
        // the same descriptor with its start-address field (bytes >> 4) moved by
        // the stage (buffer) size, and one K=16 step moves it by 256 B (16).
        const uint64_t dSb = smem_desc(smem_addr(sm + L::kSb), 128, 2048);
        const uint64_t dDb0 = smem_desc(smem_addr(sm + L::kDb), 128, 1024);
        const uint32_t st0 = smem_addr(sm);
        const uint64_t dWQ0 = smem_desc(st0 + L::kStageWQ, 128, 2048);
        const uint64_t dKT0 = smem_desc(st0 + L::kStageKT, 128, 1024);
        // [* ; Aqk] operands: rows 0..63 start 8 KB before the data and only
        // feed X rows 0..63, which are dead once Delta is formed
        const uint64_t dAQ0 = smem_desc(st0 + L::kStageAQ - 8192, 128, 1024);
        const uint64_t dAQL0 = smem_desc(st0 + L::kStageAQL - 8192, 128, 1024);
        constexpr uint64_t kStageStep = L::kStageBytes >> 4;
        constexpr uint64_t kDbStep = (VS * 128) >> 4;
        auto issue_out = [&](int j) {  // MMA2o(j)
            const uint64_t so = (uint64_t)(j % NS) * kStageStep;
            const uint64_t dd = dDb0 + (uint64_t)(j & 1) * kDbStep;
            const uint32_t tXj = tbase + VS * (1 + (j & 1));
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tXj, dAQ0 + so + 16u * kk, dd + 16u * kk, idesc2, 1u);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tXj, dAQL0 + so + 16u * kk, dd + 16u * kk, idesc2, 1u);
                mma_commit(&mma2o[j & 1]);
                mma_commit(&empty[j % NS]);
            }
            __syncwarp();
        };
        int i = 0;
        for (; i < nchunks; ++i) {
            const int s = i % NS;
            const uint32_t ph = (uint32_t)(i & 1);
            const uint32_t tX = tbase + VS * (1 + (i & 1));
            WAIT_OR_ABORT(&full[s], (uint32_t)((i / NS) & 1));
            // X[i % 2] still holds the outputs of chunk i - 2 until they are read
            if (!kMap && i >= 2) WAIT_OR_ABORT(&x_free[i & 1], (uint32_t)(((i - 2) >> 1) & 1));
            WAIT_OR_ABORT(&s_ready, ph);
            tc_fence_after();
            const uint64_t so = (uint64_t)s * kStageStep;
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16(tX, dWQ0 + so + 16u * kk, dSb + 16u * kk, idesc1, kk > 0 ? 1u : 0u);
                mma_commit(&mma1);
            }
            __syncwarp();
            WAIT_OR_ABORT(&d_ready, ph);
            tc_fence_after();
            const uint64_t dd = dDb0 + (uint64_t)(i & 1) * kDbStep;
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tS, dKT0 + so + 16u * kk, dd + 16u * kk, idesc2, 1u);
                mma_commit(&mma2s);
                // map mode: no output product; the stage is free once the state update has read it
                if (kMap) mma_commit(&empty[s]);
            }
            __syncwarp();
            if (!kMap) issue_out(i);
        }
        // every MMA issued above has completed before TMEM is freed (after a
        // normal end the consumers already waited for them; after giving up
        // some may still be running)
        if (elect_one()) mma_commit(&mma_done);
        __syncwarp();
        if (!mbar_drain(&mma_done, 0)) atomicOr(P.status, kStatusTimeout);
    } else if (warp < 4) {
        // ------------------------------------------------------------ state / epilogue warps
        const int row = tid;  // TMEM lane: key channel for S, token row for X
        int i = 0;
        for (; i < nchunks; ++i) {
            const int s = i % NS;
            const uint32_t ph = (uint32_t)(i & 1);
            const uint8_t* st = sm + s * L::kStageBytes;
            WAIT_OR_ABORT(&full[s], (uint32_t)((i / NS) & 1));
            // snapshot S (bf16, MN-major B operand K=128 x N=VS) and decay it in TMEM
            {
                const float gam = reinterpret_cast<const float*>(st + L::kStageGam)[row];
#pragma unroll
                for (int c0 = 0; c0 < VS; c0 += 16) {
                    uint32_t r[16];
                    tmem_load16(taddr(tS, 32u * warp, (uint32_t)c0), r);
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        const uint32_t* x = r + 8 * half;
                        st_shared_v4(smem_addr(sm + L::kSb +
                                               mnmaj_off(c0 + 8 * half, row, 128, 2048)),
                                     pack_bf16(__uint_as_float(x[0]), __uint_as_float(x[1])),
                                     pack_bf16(__uint_as_float(x[2]), __uint_as_float(x[3])),
                                     pack_bf16(__uint_as_float(x[4]), __uint_as_float(x[5])),
                                     pack_bf16(__uint_as_float(x[6]), __uint_as_float(x[7])));
                    }
#pragma unroll
                    for (int u = 0; u < 16; ++u) r[u] = __float_as_uint(__uint_as_float(r[u]) * gam);
                    tmem_st16(taddr(tS, 32u * warp, (uint32_t)c0), r);
                }
                tmem_wait_st();
                fence_async_smem();
                tc_fence_before();
                mbar_arrive(&s_ready);
            }
            if (warp < 2) {
                // Delta = U - X[0:64] for token row `row`, into Db[i & 1]
                const uint16_t* ut = reinterpret_cast<const uint16_t*>(st + L::kStageUT);
                uint32_t u_pk[VS / 2];  // U[row][c], two bf16 per register, read before waiting
#pragma unroll
                for (int c = 0; c < VS; c += 2)
                    u_pk[c / 2] = lin ? 0u
                                      : ((uint32_t)ut[c * 64 + row] |
                                         ((uint32_t)ut[(c + 1) * 64 + row] << 16));
                WAIT_OR_ABORT(&mma1, ph);
                tc_fence_after();
                const uint32_t tX = tbase + VS * (1 + (i & 1));
                uint8_t* db = sm + L::kDb + (i & 1) * (VS * 128);
#pragma unroll
                for (int c0 = 0; c0 < VS; c0 += 16) {
                    uint32_t r[16];
                    tmem_load16(taddr(tX, 32u * warp, (uint32_t)c0), r);
                    float d[16];
#pragma unroll
                    for (int u = 0; u < 16; ++u) {
                        const uint32_t pk = u_pk[(c0 + u) / 2];
                        d[u] = ((u & 1) ? bf16_hi(pk) : bf16_lo(pk)) - __uint_as_float(r[u]);
                    }
#pragma unroll
                    for (int half = 0; half < 2; ++half)
                        st_shared_v4(smem_addr(db + mnmaj_off(c0 + 8 * half, row, 128, 1024)),
                                     pack_bf16(d[8 * half + 0], d[8 * half + 1]),
                                     pack_bf16(d[8 * half + 2], d[8 * half + 3]),
                                     pack_bf16(d[8 * half + 4], d[8 * half + 5]),
                                     pack_bf16(d[8 * half + 6], d[8 * half + 7]));
                }
                fence_async_smem();
                tc_fence_before();
                mbar_arrive(&d_ready);
            }
            WAIT_OR_ABORT(&mma2s, ph);
            tc_fence_after();
        }
        if (!*((volatile int*)&s_abort)) {
            if constexpr (kMap) {
                const int ch = row;
#pragma unroll
                for (int c0 = 0; c0 < VS; c0 += 16) {
                    uint32_t r[16];
                    tmem_load16(taddr(tS, 32u * warp, (uint32_t)c0), r);
                    if (lin) {  // M^T[j][k]: a warp's 32 key channels are 32 consecutive words
                        float* mt = reinterpret_cast<float*>(P.hT) + state_base;
#pragma unroll
                        for (int u = 0; u < 16; ++u)
                            mt[(size_t)(v0 + c0 + u) * kDim + ch] = __uint_as_float(r[u]);
                    } else {
                        StateIO<float>::store16(P.hT, state_base + (size_t)ch * kDim + v0 + c0, r);
                    }
                }
            } else if constexpr (!std::is_same<HT, NoState>::value) {
                const int ch = row;
#pragma unroll
                for (int c0 = 0; c0 < VS; c0 += 16) {
                    uint32_t r[16];
                    tmem_load16(taddr(tS, 32u * warp, (uint32_t)c0), r);
                    StateIO<HT>::store16(P.hT, state_base + (size_t)ch * kDim + v0 + c0, r);
                }
            }
        }
    } else if (!kMap) {
        // ------------------------------------------------------------ output warps
        // warps 6 and 7 (TMEM lane quarters 2 and 3: rows 64..127 of X) write
        // the outputs of chunk j from X[j % 2], then release that buffer
        const int t = 32 * (warp & 3) - 64 + lane;  // token row of the chunk
        for (int j = 0; j < nchunks; ++j) {
            WAIT_OR_ABORT(&mma2o[j & 1], (uint32_t)((j >> 1) & 1));
            tc_fence_after();
            const ChunkInfo cj = P.info[c_begin + j];
            const uint32_t tXj = tbase + VS * (1 + (j & 1));
#pragma unroll
            for (int c0 = 0; c0 < VS; c0 += 32) {
                uint32_t r[2][16];
                tmem_ld16(taddr(tXj, 32u * (warp & 3), (uint32_t)c0), r[0]);
                tmem_ld16(taddr(tXj, 32u * (warp & 3), (uint32_t)c0 + 16u), r[1]);
                tmem_wait_ld();
                reg_fence16(r[0]);
                reg_fence16(r[1]);
                if (t < cj.len) {
                    uint4* dst = reinterpret_cast<uint4*>(
                        reinterpret_cast<__nv_bfloat16*>(P.out) +
                        ((size_t)(cj.tok0 + t) * H + h) * kDim + v0 + c0);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint32_t* x = r[q >> 1] + 8 * (q & 1);
                        dst[q] = make_uint4(pack_bf16(__uint_as_float(x[0]), __uint_as_float(x[1])),
                                            pack_bf16(__uint_as_float(x[2]), __uint_as_float(x[3])),
                                            pack_bf16(__uint_as_float(x[4]), __uint_as_float(x[5])),
                                            pack_bf16(__uint_as_float(x[6]), __uint_as_float(x[7])));
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&x_free[j & 1]);  // MMA1(j + 2) may overwrite X[j % 2]
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, L::kTmemCols);
}

template <int VS, typename H0, typename HT, bool kMap = false>
cudaError_t launch_recur_t(const Problem& p, const RecurArgs& a, cudaStream_t st) {
    using L = RecurLayout<VS>;
    auto kern = recur_kernel<VS, H0, HT, kMap>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
    if (e != cudaSuccess) return e;
    const long long blocks = (long long)p.N * p.H * (kDim / VS) * (kMap ? 2 : 1);
    kern<<<(unsigned)blocks, kThreads, L::kBytes, st>>>(a);
    return cudaGetLastError();
}

template <int VS, typename H0>
cudaError_t launch_recur_h0(const Problem& p, const RecurArgs& a, cudaStream_t st) {
    switch (p.hT_dtype) {
        case KDA_DTYPE_FP32: return launch_recur_t<VS, H0, float>(p, a, st);
        case KDA_DTYPE_BF16: return launch_recur_t<VS, H0, __nv_bfloat16>(p, a, st);
        default: return launch_recur_t<VS, H0, NoState>(p, a, st);
    }
}

template <int VS>
cudaError_t launch_recur_vs(const Problem& p, const RecurArgs& a, cudaStream_t st) {
    switch (p.h0_dtype) {
        case KDA_DTYPE_FP32: return launch_recur_h0<VS, float>(p, a, st);
        case KDA_DTYPE_BF16: return launch_recur_h0<VS, __nv_bfloat16>(p, a, st);
        default: return launch_recur_h0<VS, NoState>(p, a, st);
    }
}

}  // namespace

int recur_slice_width(const Problem& p, int num_sms) {
    // Split the value dimension only as far as needed to fill the GPU: each
    // slice re-reads the shared operands of its chunk, so fewer slices means
    // less on-chip traffic.
    const long long pairs = (long long)p.N * p.H;
    if (pairs >= 2LL * num_sms) return 128;
    if (pairs * 2 >= num_sms) return 64;
    return 32;
}

namespace {
RecurArgs recur_args(const Problem& p, const Workspace& ws, int* status) {
    RecurArgs a;
    a.out = p.out;
    a.h0 = p.h0;
    a.hT = p.hT;
    a.H = p.H;
    a.N = p.N;
    a.flags = ws.flags;
    a.chunk_off = ws.chunk_off;
    a.info = ws.info;
    a.records = ws.records;
    a.status = status;
    return a;
}
}  // namespace

cudaError_t launch_recur_sliced(const Problem& p, const Workspace& ws, int* status,
                                cudaStream_t st, int vs) {
    if (p.N == 0 || p.H == 0) return cudaSuccess;
    const RecurArgs a = recur_args(p, ws, status);
    if (vs == 0) {
        int dev = 0, sms = 148;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        vs = recur_slice_width(p, sms);
    }
    switch (vs) {
        case 128: return launch_recur_vs<128>(p, a, st);
        case 64: return launch_recur_vs<64>(p, a, st);
        default: return launch_recur_vs<32>(p, a, st);
    }
}

cudaError_t launch_recur_maps(const Problem& p, const Workspace& ws, int* status,
                              cudaStream_t st) {
    if (p.N == 0 || p.H == 0) return cudaSuccess;
    RecurArgs a = recur_args(p, ws, status);
    a.out = nullptr;
    a.h0 = nullptr;
    a.hT = ws.seg_maps;
    // one 128-wide slice for X and one for M per (segment, head)
    return launch_recur_t<128, NoState, float, true>(p, a, st);
}

bool recur_prefers_transposed(const Problem& p, int num_sms) {
    // The transposed kernel runs one CTA per (sequence, head) and does a chunk
    // in fewer, wider MMAs; measured on GB300 it is the faster one from about
    // half a CTA per SM up (128 pairs x 32 chunks: 0.096 vs 0.111 ms), while
    // 32 pairs x 1024 chunks take 2.0 ms transposed against 1.1 ms sliced.
    return 2LL * p.N * p.H >= num_sms;
}

int recur_choose(const Problem& p, int kind) {
    if (kind == 1 || kind == 2) return kind;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return recur_prefers_transposed(p, sms) ? 2 : 1;
}

cudaError_t launch_recur(const Problem& p, const Workspace& ws, int* status, cudaStream_t st,
                         int kind) {
    return recur_choose(p, kind) == 2 ? launch_recur_transposed(p, ws, status, st)
                                      : launch_recur_sliced(p, ws, status, st);
}

}  // namespace kda
