// kda_bwd.cu -- backward pass of the KDA forward: the gradients of
// L = <dout, out> + <dS_final, final_state> with respect to q, k, v, g, beta,
// A_log, dt_bias and the initial state, token-recurrent, in fp32.
//
// Forward of one (sequence, head) pair, per token (the operation of kda_fwd,
// "Flashkda Delta Attention", "Core Kernel API"; the gate is the same reading
// of A_log, dt_bias and lower_bound):
//   x = g_t + dt_bias,  pre = -exp(A_log) softplus(x),  a = exp(max(pre, lower_bound))
//   S~ = Diag(a) S,  r = S~^T k,  u = beta (v - r),  S' = S~ + k u^T,  o = scale S'^T q.
// Reverse mode of one token, given dS (the gradient of S'):
//   dq = scale S' dO                 dS += scale q dO^T
//   du = dS^T k     dk = dS u        dv = beta du      dbeta = du . (v - r)
//   dr = -beta du   dk += S~ dr      dS~ = dS + k dr^T
//   da = rowsum(dS~ o S)             dS (of the state before the token) = Diag(a) dS~
//   dpre = [pre >= lower_bound] da a     dA_log += pre dpre
//   dx = -exp(A_log) dpre sigmoid(x)     dg = dx,  ddt_bias += dx.
// The clamp passes its gradient to the argument it returns, at a tie to pre.
//
// The state recursion, forward and backward, is independent per value column:
// r, u, du and dr of column j need column j of S and dS only.  Only the
// outputs dq, dk, da and dbeta sum over value columns.  So one (sequence,
// head) pair runs on a cluster of four CTAs, each holding a 32-column slice of
// S and dS in registers (warp w: columns 4w..4w+3 of the slice; lane l: key
// rows 4l..4l+3).  A column sum over the 128 key channels is one warp's
// butterfly, so the per-token chain has no block-wide barrier.  The row sums
// are taken per token in shared memory over the eight warps, then over the
// four CTAs through distributed shared memory, in a fixed order (the results
// are deterministic).
//
// Each CTA first runs the forward over the pair's tokens, storing its slice of
// the state entering tokens 0 and 8 of every 16-token segment (checkpoints,
// fp32, workspace).  It then takes the segments last to first: from the
// token-8 checkpoint it recomputes the states entering tokens 8..15 into
// shared memory and walks those tokens backwards, then does the same for
// tokens 0..7 from the token-0 checkpoint.  Forward steps run two tokens per
// column-sum butterfly (pair_u).  Forward work per token is thus about 1.9
// state updates; the backward walk is the rest.
// With the q/k normalisation flag the rows of q and k are staged normalised,
// and a row kernel applies the normalisation's chain rule to dq and dk after.
// This is the token-recurrent form of the backward pass, the plain GPU
// counterpart of the fp64 reverse-mode oracle.
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "kda.h"
#include "kda_internal.h"
#include "kda_bwd_status.h"

namespace kda {
namespace bwd {

namespace cg = cooperative_groups;

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kSlices = 4;                 // CTAs per pair (the cluster)
constexpr int kVs = kDim / kSlices;        // value columns per CTA (32)
constexpr int kSeg = 16;                   // tokens per checkpoint segment
constexpr int kHalf = 8;                   // tokens walked per recomputation
constexpr int kSliceElems = kDim * kVs;    // 4096 floats per state slice
constexpr int kChunkSegs = 4;              // segments per low-memory checkpoint (64 tokens)
constexpr int kScratchSlots = 256;         // low-memory replay slots (>= CTAs resident at once)
constexpr int kPart = 388;                 // dq[128] | dk[128] | da[128] | dbeta, padded

// Dynamic shared memory of one CTA (byte offsets).
constexpr int kSmSt = 0;                                         // float4 [kHalf][4][kThreads]
constexpr int kSmQ = kSmSt + kHalf * 4 * kThreads * 16;          // float [kSeg][128]
constexpr int kSmK = kSmQ + kSeg * kDim * 4;                     // float [kSeg][128]
constexpr int kSmA = kSmK + kSeg * kDim * 4;                     // float [kSeg][128] decays
constexpr int kSmX = kSmA + kSeg * kDim * 4;                     // float [kSeg][128] g + dt_bias
constexpr int kSmV = kSmX + kSeg * kDim * 4;                     // float [kSeg][kVs]
constexpr int kSmDO = kSmV + kSeg * kVs * 4;                     // float [kSeg][kVs]
constexpr int kSmB = kSmDO + kSeg * kVs * 4;                     // float [kSeg]
constexpr int kSmSlot = kSmB + kSeg * 4;                         // float [2][kWarps][kPart]
constexpr int kSmPart = kSmSlot + 2 * kWarps * kPart * 4;        // float [2][kHalf][kPart]
constexpr int kSmemBytes = kSmPart + 2 * kHalf * kPart * 4;
static_assert(kSmemBytes <= 227 * 1024, "shared memory of the backward kernel");
// more than half of an SM's 228 KB: one CTA per SM at a time, so fewer CTAs are
// resident than there are low-memory replay slots (the launch checks the SM count)
static_assert(2 * kSmemBytes > 228 * 1024, "the replay-slot pool assumes one CTA per SM");
static_assert(kSmQ % 16 == 0 && kSmV % 16 == 0 && kSmDO % 16 == 0 && kSmSlot % 16 == 0 &&
                  kSmPart % 16 == 0 && (kPart * 4) % 16 == 0,
              "float4 areas must be 16-byte aligned");

struct BwdArgs {
    const __nv_bfloat16* q;
    const __nv_bfloat16* k;
    const __nv_bfloat16* v;
    const __nv_bfloat16* g;
    const __nv_bfloat16* beta;
    const __nv_bfloat16* dout;
    const float* A_log;
    const float* dt_bias;
    float lower_bound;
    float scale;
    const void* h0;          // [N, H, K, V] bf16 / fp32, or null
    int h0_fp32;
    const float* dhT;        // [N, H, K, V] fp32, or null
    const int32_t* cu;       // [N + 1], or null (N sequences of T tokens)
    int qk_norm;             // q and k rows used as x / sqrt(|x|^2 + eps)
    int N, H, T;
    long long total;         // tokens over all sequences
    float* dq;
    float* dk;
    float* dv;
    float* dg;
    float* dbeta;
    float* dh0;              // [N, H, K, V] fp32, or null
    float* part_dA;          // [N * H][kSlices]
    float* part_ddt;         // [N * H][K]
    float* ckpt;             // [slots][H][kSlices][2][kSliceElems]; low-memory:
                             // [slots64][H][kSlices][kSliceElems]
    float* scratch;          // low-memory: [kScratchSlots][2 kChunkSegs][kSliceElems]
    int* pool;               // low-memory: slot-in-use bitmap (kScratchSlots bits), zero at launch
    int* status;
};

// Checkpoint slots (two states each: entering tokens 0 and 8 of a 16-token
// segment) of sequence n start at floor(cu[n] / 16) + n: consecutive
// sequences' ranges cannot overlap (sequence n has at most floor(L / 16) + 1
// segments), and all fit in floor(total / 16) + N + 1 slots.
__host__ __device__ inline long long ckpt_slots(long long total, long long N) {
    return total / kSeg + N + 1;
}
// Low-memory mode: one state per 64-token chunk, slots from floor(cu[n] / 64) + n.
__host__ __device__ inline long long ckpt64_slots(long long total, long long N) {
    return total / (kSeg * kChunkSegs) + N + 1;
}

__device__ __forceinline__ float softplus(float x) {
    return fmaxf(x, 0.f) + log1pf(expf(-fabsf(x)));
}

// Gate of one (token, channel): pre-clamp log-decay and the decay itself.
__device__ __forceinline__ void gate(float x, float expA, float lb, float& pre, float& a) {
    pre = -expA * softplus(x);
    a = expf(fmaxf(pre, lb));
}

// Column sums over the 32 lanes of a warp, every lane ending with the same
// sums.  Reduce-scatter, then gather: lanes exchange half of their partial
// sums with the lane 16 apart (each keeping two columns), then half again with
// the lane 8 apart (one column), sum that column over the 8 lanes that share
// it by a butterfly (each step adds the same two values on both partners, so
// the 8 lanes agree), and finally read the other columns' sums from lanes of
// the groups that hold them: 10 shuffles instead of 20 for a plain butterfly.
__device__ __forceinline__ void warp_sum4(float (&p)[4]) {
    const int lane = threadIdx.x & 31;
    const bool hi4 = lane & 16, hi3 = lane & 8;
    float q0 = hi4 ? p[2] : p[0], q1 = hi4 ? p[3] : p[1];
    q0 += __shfl_xor_sync(0xffffffffu, hi4 ? p[0] : p[2], 16);
    q1 += __shfl_xor_sync(0xffffffffu, hi4 ? p[1] : p[3], 16);
    // q0, q1: columns 2 hi4 + 0, 2 hi4 + 1
    float w = hi3 ? q1 : q0;
    w += __shfl_xor_sync(0xffffffffu, hi3 ? q0 : q1, 8);
    // w: column 2 hi4 + hi3
    w += __shfl_xor_sync(0xffffffffu, w, 4);
    w += __shfl_xor_sync(0xffffffffu, w, 2);
    w += __shfl_xor_sync(0xffffffffu, w, 1);
#pragma unroll
    for (int m = 0; m < 4; ++m) p[m] = __shfl_sync(0xffffffffu, w, (m >> 1) * 16 + (m & 1) * 8 + (lane & 7));
}

__device__ __forceinline__ void ld4(const float* p, float (&x)[4]) {
    const float4 t = *reinterpret_cast<const float4*>(p);
    x[0] = t.x; x[1] = t.y; x[2] = t.z; x[3] = t.w;
}
__device__ __forceinline__ void st4(float* p, const float (&x)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
}

// One forward token on this thread's 4 x 4 piece of the state slice.
__device__ __forceinline__ void fwd_token(float (&S)[4][4], const float (&a)[4],
                                          const float (&kk)[4], const float (&vv)[4], float b) {
    float p[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) p[m] = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            S[i][m] *= a[i];
            p[m] = fmaf(S[i][m], kk[i], p[m]);
        }
    warp_sum4(p);
    float u[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) u[m] = b * (vv[m] - p[m]);
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int m = 0; m < 4; ++m) S[i][m] = fmaf(kk[i], u[m], S[i][m]);
}

// Column sums of eight values per lane (see warp_sum4): reduce-scatter over
// the lane bits 4, 3 and 2 (four, two and one shuffles), a butterfly over the
// four lanes that share a value, then the gather: 17 shuffles instead of 40.
__device__ __forceinline__ void warp_sum8(float (&p)[8]) {
    const int lane = threadIdx.x & 31;
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
    // value index bits: bit 2 <- lane bit 4, bit 1 <- lane bit 3, bit 0 <- lane bit 2
    float q[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float keep = b4 ? p[4 + j] : p[j], send = b4 ? p[j] : p[4 + j];
        q[j] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
    float r[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const float keep = b3 ? q[2 + j] : q[j], send = b3 ? q[j] : q[2 + j];
        r[j] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
    float w = b2 ? r[1] : r[0];
    w += __shfl_xor_sync(0xffffffffu, b2 ? r[0] : r[1], 4);
    w += __shfl_xor_sync(0xffffffffu, w, 2);
    w += __shfl_xor_sync(0xffffffffu, w, 1);
#pragma unroll
    for (int m = 0; m < 8; ++m) p[m] = __shfl_sync(0xffffffffu, w, m * 4 + (lane & 3));
}

// Split cluster barrier: arrive (releasing this thread's shared-memory writes
// to the other CTAs of the cluster), then later wait (acquiring theirs).
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

// Two forward tokens t and t + 1 with one column-sum butterfly.  The decayed
// state of token t + 1 is a1 o (a0 o S + k0 u0^T), so
//   r1 = (a1 o a0 o S)^T k1 + c u0,  c = sum_i a1_i k0_i k1_i:
// both column sums and c come from the state before token t, and only the
// scalar correction c u0 waits for u0.  Computes u0 and u1 and leaves
// S = a0 o S (the decayed state of token t).
__device__ __forceinline__ void pair_u(float (&S)[4][4], const float (&a0)[4], const float (&k0)[4],
                                       const float (&v0)[4], float b0, const float (&a1)[4],
                                       const float (&k1)[4], const float (&v1)[4], float b1,
                                       float (&u0)[4], float (&u1)[4]) {
    float p[8], ak1[4], c = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        ak1[i] = a1[i] * k1[i];
        c = fmaf(ak1[i], k0[i], c);
    }
#pragma unroll
    for (int m = 0; m < 8; ++m) p[m] = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            S[i][m] *= a0[i];
            p[m] = fmaf(S[i][m], k0[i], p[m]);
            p[4 + m] = fmaf(S[i][m], ak1[i], p[4 + m]);
        }
    warp_sum8(p);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        u0[m] = b0 * (v0[m] - p[m]);
        u1[m] = b1 * (v1[m] - p[4 + m] - c * u0[m]);
    }
}

// S += k u^T, and S = a o S + k u^T.
__device__ __forceinline__ void add_ku(float (&S)[4][4], const float (&kk)[4], const float (&u)[4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int m = 0; m < 4; ++m) S[i][m] = fmaf(kk[i], u[m], S[i][m]);
}
__device__ __forceinline__ void decay_add_ku(float (&S)[4][4], const float (&a)[4],
                                             const float (&kk)[4], const float (&u)[4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int m = 0; m < 4; ++m) S[i][m] = fmaf(kk[i], u[m], a[i] * S[i][m]);
}

// One segment's token data as loaded from global memory (bf16 bit patterns),
// held in registers so that the loads of the next segment overlap the work on
// the current one.  Thread t: channels 8 (t % 16) .. + 7 of token t / 16 of k,
// g and q; threads 0..63 eight values of v, threads 64..127 of dout (this
// CTA's value columns); threads 128..143 the beta of one token.  Zero past len.
struct Fetched {
    uint4 k, g, q, vd;
    float beta;
};

__device__ __forceinline__ void fetch_segment(const BwdArgs& P, long long row0, int h, int len,
                                              int col0, bool with_q, int tid, Fetched& F) {
    const int H = P.H;
    const int t = tid >> 4, c8 = (tid & 15) * 8;
    F.k = F.g = F.q = F.vd = make_uint4(0u, 0u, 0u, 0u);
    F.beta = 0.f;
    if (t < len) {
        const long long off = ((row0 + t) * H + h) * kDim + c8;
        F.k = *reinterpret_cast<const uint4*>(P.k + off);
        F.g = *reinterpret_cast<const uint4*>(P.g + off);
        if (with_q) F.q = *reinterpret_cast<const uint4*>(P.q + off);
    }
    if (tid < 128) {
        const int piece = tid & 63, tv = piece >> 2, cv = (piece & 3) * 8;
        if (tv < len && (tid < 64 || with_q)) {
            const __nv_bfloat16* src = tid < 64 ? P.v : P.dout;
            F.vd = *reinterpret_cast<const uint4*>(src + ((row0 + tv) * H + h) * kDim + col0 + cv);
        }
    } else if (tid < 128 + kSeg && tid - 128 < len) {
        F.beta = __bfloat162float(P.beta[(row0 + (tid - 128)) * H + h]);
    }
}

// Writes fetched token data to shared memory as fp32: k, q, the gate argument
// x = g + dt_bias and the decay a of all 128 key channels, v and dout of this
// CTA's columns, beta.  dtb: dt_bias of the thread's eight channels.
// with_q: also q and dout.
__device__ __forceinline__ void store_segment(uint8_t* sm, const Fetched& F, const float (&dtb)[8],
                                              float expA, float lb, bool with_q, bool qk_norm,
                                              int tid) {
    const int t = tid >> 4, c8 = (tid & 15) * 8;
    const __nv_bfloat16* kb = reinterpret_cast<const __nv_bfloat16*>(&F.k);
    const __nv_bfloat16* gb = reinterpret_cast<const __nv_bfloat16*>(&F.g);
    const __nv_bfloat16* qb = reinterpret_cast<const __nv_bfloat16*>(&F.q);
    float kk[8], xx[8], aa[8], qq[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        kk[e] = __bfloat162float(kb[e]);
        qq[e] = __bfloat162float(qb[e]);
        xx[e] = __bfloat162float(gb[e]) + dtb[e];
        float pre;
        gate(xx[e], expA, lb, pre, aa[e]);
    }
    if (qk_norm) {
        // a token's 128 channels sit on the 16 lanes of one half-warp
        float sk = 0.f, sq = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            sk = fmaf(kk[e], kk[e], sk);
            sq = fmaf(qq[e], qq[e], sq);
        }
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) {
            sk += __shfl_xor_sync(0xffffffffu, sk, o);
            sq += __shfl_xor_sync(0xffffffffu, sq, o);
        }
        const float ik = 1.f / sqrtf(sk + kL2NormEps), iq = 1.f / sqrtf(sq + kL2NormEps);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            kk[e] *= ik;
            qq[e] *= iq;
        }
    }
    const int base = t * kDim + c8;
#pragma unroll
    for (int e = 0; e < 8; e += 4) {
        *reinterpret_cast<float4*>(sm + kSmK + 4 * (base + e)) =
            make_float4(kk[e], kk[e + 1], kk[e + 2], kk[e + 3]);
        *reinterpret_cast<float4*>(sm + kSmA + 4 * (base + e)) =
            make_float4(aa[e], aa[e + 1], aa[e + 2], aa[e + 3]);
        *reinterpret_cast<float4*>(sm + kSmX + 4 * (base + e)) =
            make_float4(xx[e], xx[e + 1], xx[e + 2], xx[e + 3]);
        if (with_q)
            *reinterpret_cast<float4*>(sm + kSmQ + 4 * (base + e)) =
                make_float4(qq[e], qq[e + 1], qq[e + 2], qq[e + 3]);
    }
    if (tid < 128) {
        if (tid < 64 || with_q) {
            const int piece = tid & 63, tv = piece >> 2, cv = (piece & 3) * 8;
            const __nv_bfloat16* vb = reinterpret_cast<const __nv_bfloat16*>(&F.vd);
            float* dst = reinterpret_cast<float*>(sm + (tid < 64 ? kSmV : kSmDO)) + tv * kVs + cv;
            *reinterpret_cast<float4*>(dst) =
                make_float4(__bfloat162float(vb[0]), __bfloat162float(vb[1]),
                            __bfloat162float(vb[2]), __bfloat162float(vb[3]));
            *reinterpret_cast<float4*>(dst + 4) =
                make_float4(__bfloat162float(vb[4]), __bfloat162float(vb[5]),
                            __bfloat162float(vb[6]), __bfloat162float(vb[7]));
        }
    } else if (tid < 128 + kSeg) {
        reinterpret_cast<float*>(sm + kSmB)[tid - 128] = F.beta;
    }
}

// The thread's 4 x 4 piece of a state slice in the checkpoint / shared-memory
// layouts: four float4 (one per key row), each array ordered [row][thread] so
// that a warp's accesses are contiguous.
__device__ __forceinline__ void save_piece(float4* base, const float (&S)[4][4], int tid) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
        base[i * kThreads + tid] = make_float4(S[i][0], S[i][1], S[i][2], S[i][3]);
}
__device__ __forceinline__ void load_piece(const float4* base, float (&S)[4][4], int tid) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float4 t = base[i * kThreads + tid];
        S[i][0] = t.x; S[i][1] = t.y; S[i][2] = t.z; S[i][3] = t.w;
    }
}

// One cluster of kSlices CTAs per (sequence, head) pair; CTA rank r holds
// value columns 32 r .. 32 r + 31 and writes dq, dk, dg of key channels
// 32 r .. 32 r + 31.
// kLowMem: checkpoints every 64 tokens, each chunk replayed into a scratch slot
// (a template parameter, so the default kernel carries none of that code).
template <bool kLowMem>
__global__ void __cluster_dims__(kSlices, 1, 1) __launch_bounds__(kThreads, 1)
    bwd_kernel(const BwdArgs P) {
    extern __shared__ __align__(16) uint8_t sm[];
    cg::cluster_group cluster = cg::this_cluster();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rank = (int)cluster.block_rank();
    const long long pair = blockIdx.x / kSlices;
    const int H = P.H;
    const int n = (int)(pair / H), h = (int)(pair % H);
    const int col0 = rank * kVs;
    const float lb = P.lower_bound;

    // sequence bounds; a malformed cu_seqlens leaves the pair empty and sets the status
    long long row0;
    int L;
    if (P.cu) {
        const int c0 = P.cu[n], c1 = P.cu[n + 1];
        const bool ok = P.cu[0] == 0 && (long long)P.cu[P.N] == P.total && 0 <= c0 && c0 <= c1 &&
                        (long long)c1 <= P.total;
        if (!ok && rank == 0 && tid == 0) atomicOr(P.status, kStatusDeviceInput);
        row0 = ok ? c0 : 0;
        L = ok ? c1 - c0 : 0;
    } else {
        row0 = (long long)n * P.T;
        L = P.T;
    }
    const float expA = expf(P.A_log[h]);
    float dtb[8];  // dt_bias of the eight channels this thread stages
#pragma unroll
    for (int e = 0; e < 8; ++e) dtb[e] = P.dt_bias[(long long)h * kDim + (tid & 15) * 8 + e];
    const float* qs = reinterpret_cast<const float*>(sm + kSmQ);
    const float* ks = reinterpret_cast<const float*>(sm + kSmK);
    const float* as = reinterpret_cast<const float*>(sm + kSmA);
    const float* xs = reinterpret_cast<const float*>(sm + kSmX);
    const float* vs = reinterpret_cast<const float*>(sm + kSmV);
    const float* dos = reinterpret_cast<const float*>(sm + kSmDO);
    const float* bs = reinterpret_cast<const float*>(sm + kSmB);
    float4* st = reinterpret_cast<float4*>(sm + kSmSt);
    float* slot = reinterpret_cast<float*>(sm + kSmSlot);
    float* part = reinterpret_cast<float*>(sm + kSmPart);

    // this thread's piece: key rows 4 lane + i, value columns col0 + 4 warp + m
    const long long soff = pair * kDim * kDim + (long long)(4 * lane) * kDim + col0 + 4 * warp;
    float S[4][4], dS[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (!P.h0) {
#pragma unroll
            for (int m = 0; m < 4; ++m) S[i][m] = 0.f;
        } else if (P.h0_fp32) {
            ld4(static_cast<const float*>(P.h0) + soff + i * kDim, S[i]);
        } else {
            const uint2 r =
                *reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(P.h0) + soff + i * kDim);
            const __nv_bfloat16* rb = reinterpret_cast<const __nv_bfloat16*>(&r);
#pragma unroll
            for (int m = 0; m < 4; ++m) S[i][m] = __bfloat162float(rb[m]);
        }
        if (P.dhT) ld4(P.dhT + soff + i * kDim, dS[i]);
        else {
#pragma unroll
            for (int m = 0; m < 4; ++m) dS[i][m] = 0.f;
        }
    }

    const int nseg = (L + kSeg - 1) / kSeg;
    const long long slot0 = row0 / kSeg + n;
    const long long slot64 = row0 / (kSeg * kChunkSegs) + n;
    // Low-memory mode: a replay slot for this CTA, claimed in the pool's
    // occupancy bitmap (kScratchSlots bits in 32-bit words).  At most one CTA per
    // SM is resident, so fewer than half the bits are ever set and every read of
    // the bitmap shows free bits; a claim that loses a race retries with the
    // word's newer value.  All loops are bounded.
    __shared__ int s_scratch;
    if (kLowMem) {
        if (tid == 0) {
            unsigned* bits = reinterpret_cast<unsigned*>(P.pool);
            constexpr int kWords = kScratchSlots / 32;
            int got = -1;
            for (int pass = 0; pass < 64 && got < 0; ++pass) {
                for (int w = 0; w < kWords && got < 0; ++w) {
                    const int word = (int)((blockIdx.x + (unsigned)w) % kWords);
                    unsigned cur = atomicOr(bits + word, 0u);
                    for (int tries = 0; tries < 32 && cur != 0xffffffffu; ++tries) {
                        const unsigned bit = 1u << (__ffs(~cur) - 1);
                        const unsigned old = atomicOr(bits + word, bit);
                        if (!(old & bit)) {
                            got = word * 32 + __ffs(bit) - 1;
                            break;
                        }
                        cur = old | bit;
                    }
                }
            }
            if (got < 0) {  // not reachable while fewer CTAs than slots are resident
                atomicOr(P.status, kStatusScratch);
                got = 0;
            }
            s_scratch = got;
        }
        __syncthreads();
    }
    // checkpoint of segment s: the state entering token 8 half of the segment
    // (low-memory: in this CTA's replay slot, by the segment's place in its chunk)
    auto ckpt_at = [&](int s, int half) {
        if (kLowMem)
            return reinterpret_cast<float4*>(
                P.scratch + ((long long)s_scratch * 2 * kChunkSegs + (s % kChunkSegs) * 2 + half) *
                                kSliceElems);
        return reinterpret_cast<float4*>(
            P.ckpt + ((((slot0 + s) * H + h) * kSlices + rank) * 2 + half) * (long long)kSliceElems);
    };
    // low-memory: the state entering 64-token chunk c
    auto ckpt64_at = [&](int c) {
        return reinterpret_cast<float4*>(
            P.ckpt + (((slot64 + c) * H + h) * kSlices + rank) * (long long)kSliceElems);
    };
    Fetched F;

    // 1. forward sweep: the states entering tokens 0 and 8 of every segment
    //    (the last segment's tokens are replayed by the walk, so the sweep
    //    stops before them); the next segment's loads are in flight while a
    //    segment is swept.  Checkpoints are read back later by this same thread.
    if (nseg > 1) fetch_segment(P, row0, h, kSeg, col0, false, tid, F);
    for (int s = 0; s < nseg; ++s) {
        if (!kLowMem) save_piece(ckpt_at(s, 0), S, tid);
        else if (s % kChunkSegs == 0) save_piece(ckpt64_at(s / kChunkSegs), S, tid);
        if (s == nseg - 1) break;
        __syncthreads();
        store_segment(sm, F, dtb, expA, lb, false, P.qk_norm != 0, tid);
        if (s + 2 < nseg)
            fetch_segment(P, row0 + (long long)(s + 1) * kSeg, h, kSeg, col0, false, tid, F);
        __syncthreads();
        for (int t = 0; t < kSeg; t += 2) {
            if (t == kHalf && !kLowMem) save_piece(ckpt_at(s, 1), S, tid);
            float a0[4], k0[4], v0[4], a1[4], k1[4], v1[4], u0[4], u1[4];
            ld4(as + t * kDim + 4 * lane, a0);
            ld4(ks + t * kDim + 4 * lane, k0);
            ld4(vs + t * kVs + 4 * warp, v0);
            ld4(as + (t + 1) * kDim + 4 * lane, a1);
            ld4(ks + (t + 1) * kDim + 4 * lane, k1);
            ld4(vs + (t + 1) * kVs + 4 * warp, v1);
            pair_u(S, a0, k0, v0, bs[t], a1, k1, v1, bs[t + 1], u0, u1);
            add_ku(S, k0, u0);
            decay_add_ku(S, a1, k1, u1);
        }
    }

    // 2. backward walk, segments last to first, each in two halves.  The row
    //    sums of a half are taken over the cluster after the next half's
    //    states are recomputed, which hides the cluster barrier's latency.
    float accA = 0.f, accB = 0.f;  // dA_log and ddt_bias of key channel 32 rank + lane
    int cb = 0;                    // part[] buffer of the current half
    bool pend = false;             // a walked half whose row sums are not yet taken
    long long p_row = 0;           // its first token's row
    int p_len = 0, p_cb = 0;
    float p_x = 0.f;               // gate argument of (its token warp, channel 32 rank + lane)
    auto finish_half = [&]() {
        cluster_wait();
        if (warp < p_len) {
            const int c = rank * kVs + lane;
            const long long row = p_row + warp;
            float sq = 0.f, sk = 0.f, sa = 0.f, sb = 0.f;
#pragma unroll
            for (int r = 0; r < kSlices; ++r) {
                const float* rp =
                    cluster.map_shared_rank(part + (p_cb * kHalf + warp) * kPart, (unsigned)r);
                sq += rp[c];
                sk += rp[kDim + c];
                sa += rp[2 * kDim + c];
                sb += rp[3 * kDim];
            }
            const long long off = (row * H + h) * kDim + c;
            float pre, a;
            gate(p_x, expA, lb, pre, a);
            const float dpre = pre >= lb ? sa * a : 0.f;
            accA = fmaf(pre, dpre, accA);
            const float dx = -expA * dpre / (1.f + expf(-p_x));
            accB += dx;
            P.dq[off] = sq;
            P.dk[off] = sk;
            P.dg[off] = dx;
            if (rank == 0 && lane == 0) P.dbeta[row * H + h] = sb;
        }
        pend = false;
    };

    // C: the checkpoint the current half is replayed from; Cn: the next half's.
    // Halves are walked in the order (s, 1), (s, 0), (s - 1, 1), ...; the last
    // segment has no token-8 checkpoint, so its upper half replays from token 0.
    float C[4][4], Cn[4][4];
    if (nseg > 0) {
        fetch_segment(P, row0 + (long long)(nseg - 1) * kSeg, h, L - (nseg - 1) * kSeg, col0,
                      true, tid, F);
        if (!kLowMem) load_piece(ckpt_at(nseg - 1, 0), C, tid);
    }
    for (int s = nseg - 1; s >= 0; --s) {
        const int len = min(kSeg, L - s * kSeg);
        const long long rs = row0 + (long long)s * kSeg;
        if (kLowMem && (s == nseg - 1 || s % kChunkSegs == kChunkSegs - 1)) {
            // entering 64-token chunk c from above: replay it from its checkpoint,
            // writing the token-0 and token-8 states of its segments 4c .. s into
            // the replay slot (the same operations as the sweep, so the same bits)
            const int c = s / kChunkSegs;
            float R[4][4];
            Fetched G;
            load_piece(ckpt64_at(c), R, tid);
            for (int s2 = c * kChunkSegs; s2 <= s; ++s2) {
                save_piece(ckpt_at(s2, 0), R, tid);
                if (s2 == nseg - 1) break;  // the last segment is walked from its token 0
                __syncthreads();
                fetch_segment(P, row0 + (long long)s2 * kSeg, h, kSeg, col0, false, tid, G);
                store_segment(sm, G, dtb, expA, lb, false, P.qk_norm != 0, tid);
                __syncthreads();
                const int tend = s2 == s ? kHalf : kSeg;  // segment s needs its token-8 state only
                for (int t = 0; t < tend; t += 2) {
                    if (t == kHalf) save_piece(ckpt_at(s2, 1), R, tid);
                    float a0[4], k0[4], v0[4], a1[4], k1[4], v1[4], u0[4], u1[4];
                    ld4(as + t * kDim + 4 * lane, a0);
                    ld4(ks + t * kDim + 4 * lane, k0);
                    ld4(vs + t * kVs + 4 * warp, v0);
                    ld4(as + (t + 1) * kDim + 4 * lane, a1);
                    ld4(ks + (t + 1) * kDim + 4 * lane, k1);
                    ld4(vs + (t + 1) * kVs + 4 * warp, v1);
                    pair_u(R, a0, k0, v0, bs[t], a1, k1, v1, bs[t + 1], u0, u1);
                    add_ku(R, k0, u0);
                    decay_add_ku(R, a1, k1, u1);
                }
                if (tend == kHalf) save_piece(ckpt_at(s2, 1), R, tid);
            }
            // the half walked first replays from this segment's token-8 state
            // (token 0 for the last segment)
            load_piece(ckpt_at(s, s < nseg - 1 ? 1 : 0), C, tid);
        }
        __syncthreads();
        store_segment(sm, F, dtb, expA, lb, true, P.qk_norm != 0, tid);
        if (s > 0) fetch_segment(P, rs - kSeg, h, kSeg, col0, true, tid, F);
        __syncthreads();
        for (int half = len > kHalf ? 1 : 0; half >= 0; --half) {
            const int t0 = half * kHalf, t1 = min(len, t0 + kHalf);
            {   // states entering tokens t0 .. t1 - 1, from the checkpoint
                float R[4][4];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int m = 0; m < 4; ++m) R[i][m] = C[i][m];
                // the next half's checkpoint is loaded while this one is walked
                if (half == 1) load_piece(ckpt_at(s, 0), Cn, tid);
                else if (s > 0) load_piece(ckpt_at(s - 1, 1), Cn, tid);
                // replay tokens tr .. t1 - 2, two at a time where possible
                const int tr = (half == 1 && s < nseg - 1) ? kHalf : 0;
                for (int t = tr; t < t1;) {
                    if (t >= t0) save_piece(st + (t - t0) * 4 * kThreads, R, tid);
                    if (t + 1 >= t1) break;
                    if (t + 2 < t1) {
                        float a0[4], k0[4], v0[4], a1[4], k1[4], v1[4], u0[4], u1[4];
                        ld4(as + t * kDim + 4 * lane, a0);
                        ld4(ks + t * kDim + 4 * lane, k0);
                        ld4(vs + t * kVs + 4 * warp, v0);
                        ld4(as + (t + 1) * kDim + 4 * lane, a1);
                        ld4(ks + (t + 1) * kDim + 4 * lane, k1);
                        ld4(vs + (t + 1) * kVs + 4 * warp, v1);
                        pair_u(R, a0, k0, v0, bs[t], a1, k1, v1, bs[t + 1], u0, u1);
                        add_ku(R, k0, u0);
                        if (t + 1 >= t0) save_piece(st + (t + 1 - t0) * 4 * kThreads, R, tid);
                        decay_add_ku(R, a1, k1, u1);
                        t += 2;
                    } else {
                        float a[4], kk[4], vv[4];
                        ld4(as + t * kDim + 4 * lane, a);
                        ld4(ks + t * kDim + 4 * lane, kk);
                        ld4(vs + t * kVs + 4 * warp, vv);
                        fwd_token(R, a, kk, vv, bs[t]);
                        t += 1;
                    }
                }
            }
            const float x_here = t0 + warp < t1 ? xs[(t0 + warp) * kDim + rank * kVs + lane] : 0.f;
            if (pend) finish_half();
            for (int t = t1 - 1; t >= t0; --t) {
                float a[4], kk[4], qq[4], vv[4], oo[4], Sp[4][4];
                ld4(as + t * kDim + 4 * lane, a);
                ld4(ks + t * kDim + 4 * lane, kk);
                ld4(qs + t * kDim + 4 * lane, qq);
                ld4(vs + t * kVs + 4 * warp, vv);
                ld4(dos + t * kVs + 4 * warp, oo);
                const float b = bs[t];
                load_piece(st + (t - t0) * 4 * kThreads, Sp, tid);
                // S~ = Diag(a) S and r = S~^T k; dS += scale q dO^T and du = dS^T k
                // (one butterfly for both column sums)
                float St[4][4], red[8];
#pragma unroll
                for (int m = 0; m < 8; ++m) red[m] = 0.f;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float sq = P.scale * qq[i];
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        St[i][m] = a[i] * Sp[i][m];
                        red[m] = fmaf(St[i][m], kk[i], red[m]);
                        dS[i][m] = fmaf(sq, oo[m], dS[i][m]);
                        red[4 + m] = fmaf(dS[i][m], kk[i], red[4 + m]);
                    }
                }
                warp_sum8(red);
                float e[4], u[4], du[4], dr[4], dbp = 0.f;
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    e[m] = vv[m] - red[m];
                    u[m] = b * e[m];
                    du[m] = red[4 + m];
                    dbp = fmaf(du[m], e[m], dbp);
                    dr[m] = -b * du[m];
                }
                float dqp[4], dkp[4], dap[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    // o = scale S'^T q with S' = S~ + k u^T
                    float x = 0.f;
#pragma unroll
                    for (int m = 0; m < 4; ++m) x = fmaf(fmaf(kk[i], u[m], St[i][m]), oo[m], x);
                    dqp[i] = P.scale * x;
                    // dk = dS u + S~ dr; then dS~ = dS + k dr^T
                    float y = 0.f;
#pragma unroll
                    for (int m = 0; m < 4; ++m) y = fmaf(dS[i][m], u[m], y);
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        y = fmaf(St[i][m], dr[m], y);
                        dS[i][m] = fmaf(kk[i], dr[m], dS[i][m]);
                    }
                    dkp[i] = y;
                    // da = rowsum(dS~ o S); dS = Diag(a) dS~
                    float z = 0.f;
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        z = fmaf(dS[i][m], Sp[i][m], z);
                        dS[i][m] *= a[i];
                    }
                    dap[i] = z;
                }
                if (lane == 0) {
                    const float dvv[4] = {b * du[0], b * du[1], b * du[2], b * du[3]};
                    st4(P.dv + ((rs + t) * H + h) * kDim + col0 + 4 * warp, dvv);
                }
                // row sums: this warp's share, then the CTA's in a fixed warp order
                float* sl = slot + ((t & 1) * kWarps + warp) * kPart;
                st4(sl + 4 * lane, dqp);
                st4(sl + kDim + 4 * lane, dkp);
                st4(sl + 2 * kDim + 4 * lane, dap);
                if (lane == 0) sl[3 * kDim] = dbp;
                __syncthreads();
                const float* src = slot + (t & 1) * kWarps * kPart;
                float* dst = part + (cb * kHalf + (t - t0)) * kPart;
                if (tid < 3 * kDim / 2) {
                    float2 acc = *reinterpret_cast<const float2*>(src + 2 * tid);
#pragma unroll
                    for (int w = 1; w < kWarps; ++w) {
                        const float2 x = *reinterpret_cast<const float2*>(src + w * kPart + 2 * tid);
                        acc.x += x.x;
                        acc.y += x.y;
                    }
                    *reinterpret_cast<float2*>(dst + 2 * tid) = acc;
                } else if (tid == 3 * kDim / 2) {
                    float acc = src[3 * kDim];
#pragma unroll
                    for (int w = 1; w < kWarps; ++w) acc += src[w * kPart + 3 * kDim];
                    dst[3 * kDim] = acc;
                }
            }
            // the CTA's row sums of this half are in part[cb]: publish them
            cluster_arrive();
            pend = true;
            p_row = rs + t0;
            p_len = t1 - t0;
            p_cb = cb;
            p_x = x_here;
            cb ^= 1;
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int m = 0; m < 4; ++m) C[i][m] = Cn[i][m];
        }
    }
    if (pend) finish_half();

    // 3. dS is now the gradient of the initial state
    if (P.dh0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) st4(P.dh0 + soff + i * kDim, dS[i]);
    }
    // per-pair sums of dA_log and ddt_bias, in a fixed order
    __syncthreads();
    slot[warp * 32 + lane] = accB;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) accA += __shfl_xor_sync(0xffffffffu, accA, o);
    if (lane == 0) slot[kThreads + warp] = accA;
    __syncthreads();
    if (tid < 32) {
        float x = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) x += slot[w * 32 + tid];
        P.part_ddt[pair * kDim + rank * kVs + tid] = x;
    } else if (tid == 32) {
        float x = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) x += slot[kThreads + w];
        P.part_dA[pair * kSlices + rank] = x;
    }
    // no CTA leaves while a peer may still read its shared memory; the replay
    // slot goes back to the pool once every thread's scratch stores are visible
    if (kLowMem) __threadfence();
    cluster.sync();
    if (kLowMem && tid == 0)
        atomicAnd(reinterpret_cast<unsigned*>(P.pool) + s_scratch / 32, ~(1u << (s_scratch % 32)));
}

// dA_log [H] and ddt_bias [H, K]: the per-pair sums added over the sequences
// (and CTAs) in a fixed order.
__global__ void bwd_param_kernel(const float* __restrict__ part_dA,
                                 const float* __restrict__ part_ddt, int N, int H,
                                 float* __restrict__ dA_log, float* __restrict__ ddt_bias) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= H * (kDim + 1)) return;
    const int h = i / (kDim + 1), c = i % (kDim + 1);
    float x = 0.f;
    if (c < kDim) {
        for (int n = 0; n < N; ++n) x += part_ddt[((long long)n * H + h) * kDim + c];
        ddt_bias[(long long)h * kDim + c] = x;
    } else {
        for (int n = 0; n < N; ++n)
            for (int r = 0; r < kSlices; ++r) x += part_dA[((long long)n * H + h) * kSlices + r];
        dA_log[h] = x;
    }
}

// Chain rule through the q/k normalisation, in place: for every (token, head)
// row of x (q or k, bf16) with n = sqrt(|x|^2 + eps) and xhat = x / n, the
// gradient dxhat that the backward kernel wrote becomes
// dx = (dxhat - xhat (xhat . dxhat)) / n.  One warp per row, four channels a lane.
__global__ void __launch_bounds__(256) bwd_l2norm_kernel(const __nv_bfloat16* __restrict__ q,
                                                         const __nv_bfloat16* __restrict__ k,
                                                         float* __restrict__ dq,
                                                         float* __restrict__ dk, long long rows) {
    const long long row = blockIdx.x * 8ll + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const __nv_bfloat16* x = blockIdx.y == 0 ? q : k;
    float* dx = blockIdx.y == 0 ? dq : dk;
    const uint2 xr = *reinterpret_cast<const uint2*>(x + row * kDim + 4 * lane);
    const __nv_bfloat16* xb = reinterpret_cast<const __nv_bfloat16*>(&xr);
    float xv[4], d[4];
    ld4(dx + row * kDim + 4 * lane, d);
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        xv[e] = __bfloat162float(xb[e]);
        ss = fmaf(xv[e], xv[e], ss);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float inv = 1.f / sqrtf(ss + kL2NormEps);
    float dot = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        xv[e] *= inv;
        dot = fmaf(xv[e], d[e], dot);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
#pragma unroll
    for (int e = 0; e < 4; ++e) d[e] = (d[e] - xv[e] * dot) * inv;
    st4(dx + row * kDim + 4 * lane, d);
}

}  // namespace bwd
}  // namespace kda

// ============================================================================= host side
namespace kda {
namespace bwd {
namespace {

constexpr size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Workspace: per-pair partial sums, then (low-memory) the slot pool and the
// replay slots, then the checkpoints.
size_t ws_bytes(long long total, long long N, long long H, bool low_mem) {
    const size_t pairs = (size_t)N * (size_t)H;
    size_t b = align256(pairs * kSlices * sizeof(float)) + align256(pairs * kDim * sizeof(float));
    if (low_mem)
        return b + align256(kScratchSlots * sizeof(int)) +
               (size_t)kScratchSlots * 2 * kChunkSegs * kSliceElems * sizeof(float) +
               (size_t)ckpt64_slots(total, N) * (size_t)H * kSlices * kSliceElems * sizeof(float);
    return b + (size_t)ckpt_slots(total, N) * (size_t)H * kSlices * 2 * kSliceElems * sizeof(float);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace bwd
}  // namespace kda

using namespace kda;

extern "C" size_t kda_bwd_workspace_size(int32_t B, int32_t T, int32_t H, int32_t num_seqs,
                                         int32_t has_cu_seqlens, uint32_t flags) {
    clear_error();
    if (B < 1 || T < 0 || H < 1 || (has_cu_seqlens && (B != 1 || num_seqs < 0)) ||
        (flags & ~(uint32_t)(KDA_FWD_QK_L2NORM | KDA_BWD_LOW_MEMORY))) {
        set_error(KDA_ERR_INVALID_ARGUMENT, "invalid sizes or flags");
        return 0;
    }
    const long long N = has_cu_seqlens ? num_seqs : B;
    return bwd::ws_bytes((long long)B * T, N, H, (flags & KDA_BWD_LOW_MEMORY) != 0);
}

extern "C" kda_status_t kda_bwd(const void* q, const void* k, const void* v, const void* g,
                                const void* beta, float scale, const float* A_log,
                                const float* dt_bias, float lower_bound,
                                const void* initial_state, kda_dtype_t initial_dtype,
                                const void* dout, const float* dfinal_state,
                                const int32_t* cu_seqlens, int32_t num_seqs, int32_t B,
                                int32_t T, int32_t H, int32_t K, int32_t V, float* dq, float* dk,
                                float* dv, float* dg, float* dbeta, float* dA_log,
                                float* ddt_bias, float* dinitial_state, uint32_t flags,
                                void* workspace, size_t workspace_bytes_, void* stream) {
    using bwd::aligned16;
    clear_error();
    if (flags & ~(uint32_t)(KDA_FWD_QK_L2NORM | KDA_BWD_LOW_MEMORY))
        return set_error(KDA_ERR_INVALID_ARGUMENT, "unknown flag bits");
    const bool low_mem = (flags & KDA_BWD_LOW_MEMORY) != 0;
    if (K != kDim || V != kDim)
        return set_error(KDA_ERR_INVALID_ARGUMENT, "K and V must both be 128");
    if (B < 1 || T < 0 || H < 1)
        return set_error(KDA_ERR_INVALID_ARGUMENT, "need B >= 1, T >= 0, H >= 1");
    if (cu_seqlens && B != 1)
        return set_error(KDA_ERR_INVALID_ARGUMENT, "cu_seqlens requires B == 1");
    if (cu_seqlens && num_seqs < 0)
        return set_error(KDA_ERR_INVALID_ARGUMENT, "num_seqs must be >= 0");
    if (initial_dtype != KDA_DTYPE_NONE && initial_dtype != KDA_DTYPE_BF16 &&
        initial_dtype != KDA_DTYPE_FP32)
        return set_error(KDA_ERR_INVALID_ARGUMENT, "initial_state dtype must be NONE, BF16 or FP32");
    if ((initial_state == nullptr) != (initial_dtype == KDA_DTYPE_NONE))
        return set_error(KDA_ERR_INVALID_ARGUMENT, "initial_state pointer and dtype disagree");
    if (!std::isfinite(scale)) return set_error(KDA_ERR_INVALID_ARGUMENT, "scale must be finite");
    if (!std::isfinite(lower_bound) || lower_bound > 0.f)
        return set_error(KDA_ERR_INVALID_ARGUMENT, "lower_bound must be finite and <= 0");
    const long long total = (long long)B * T;
    if (total > (long long)INT32_MAX - 64)
        return set_error(KDA_ERR_INVALID_ARGUMENT, "B * T too large");
    const long long N = cu_seqlens ? num_seqs : B;
    if ((long long)N * H * bwd::kSlices > (long long)INT32_MAX)
        return set_error(KDA_ERR_INVALID_ARGUMENT, "too many (sequence, head) pairs");
    if ((total * H + 7) / 8 > (long long)INT32_MAX)
        return set_error(KDA_ERR_INVALID_ARGUMENT, "too many (token, head) rows");
    if (total > 0) {
        if (!q || !k || !v || !g || !beta || !dout || !dq || !dk || !dv || !dg || !dbeta)
            return set_error(KDA_ERR_INVALID_ARGUMENT,
                             "q, k, v, g, beta, dout and the token gradients must be non-null");
        if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(dout) ||
            !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(dg))
            return set_error(KDA_ERR_INVALID_ARGUMENT,
                             "q, k, v, g, dout, dq, dk, dv and dg must be 16-byte aligned");
        if ((reinterpret_cast<uintptr_t>(beta) & 1u) || (reinterpret_cast<uintptr_t>(dbeta) & 3u))
            return set_error(KDA_ERR_INVALID_ARGUMENT,
                             "beta must be 2-byte and dbeta 4-byte aligned");
    }
    if (!A_log || !dt_bias || !dA_log || !ddt_bias)
        return set_error(KDA_ERR_INVALID_ARGUMENT,
                         "A_log, dt_bias, dA_log and ddt_bias must be non-null");
    if ((initial_state && !aligned16(initial_state)) || (dfinal_state && !aligned16(dfinal_state)) ||
        (dinitial_state && !aligned16(dinitial_state)))
        return set_error(KDA_ERR_INVALID_ARGUMENT, "states and their gradients must be 16-byte aligned");
    if (cu_seqlens && (reinterpret_cast<uintptr_t>(cu_seqlens) & 3u))
        return set_error(KDA_ERR_INVALID_ARGUMENT, "cu_seqlens must be 4-byte aligned");
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const size_t need = bwd::ws_bytes(total, N, H, low_mem);
    if (N > 0 && workspace) {
        if (workspace_bytes_ < need)
            return set_error(KDA_ERR_INVALID_ARGUMENT,
                             "workspace smaller than kda_bwd_workspace_size()");
        if (reinterpret_cast<uintptr_t>(workspace) & 255u)
            return set_error(KDA_ERR_INVALID_ARGUMENT, "workspace must be 256-byte aligned");
    }
    int* status = device_status_ptr();  // before any allocation: nothing to undo on failure
    if (!status) return KDA_ERR_CUDA;
    void* ws = workspace;
    bool owned = false;
    if (N > 0 && !ws) {
        cudaError_t e = cudaMallocAsync(&ws, need, st);
        if (e != cudaSuccess) return cuda_error(e, "cudaMallocAsync(workspace)");
        owned = true;
    }
    cudaError_t e = cudaSuccess;
    if (N > 0) {
        const size_t pairs = (size_t)N * (size_t)H;
        uint8_t* p = static_cast<uint8_t*>(ws);
        bwd::BwdArgs a;
        a.q = static_cast<const __nv_bfloat16*>(q);
        a.k = static_cast<const __nv_bfloat16*>(k);
        a.v = static_cast<const __nv_bfloat16*>(v);
        a.g = static_cast<const __nv_bfloat16*>(g);
        a.beta = static_cast<const __nv_bfloat16*>(beta);
        a.dout = static_cast<const __nv_bfloat16*>(dout);
        a.A_log = A_log;
        a.dt_bias = dt_bias;
        a.lower_bound = lower_bound;
        a.scale = scale;
        a.h0 = initial_state;
        a.h0_fp32 = initial_dtype == KDA_DTYPE_FP32;
        a.dhT = dfinal_state;
        a.cu = cu_seqlens;
        a.qk_norm = (flags & KDA_FWD_QK_L2NORM) != 0;
        a.N = (int)N;
        a.H = H;
        a.T = T;
        a.total = total;
        a.dq = dq;
        a.dk = dk;
        a.dv = dv;
        a.dg = dg;
        a.dbeta = dbeta;
        a.dh0 = dinitial_state;
        a.part_dA = reinterpret_cast<float*>(p);
        p += bwd::align256(pairs * bwd::kSlices * sizeof(float));
        a.part_ddt = reinterpret_cast<float*>(p);
        p += bwd::align256(pairs * kDim * sizeof(float));
        a.pool = nullptr;
        a.scratch = nullptr;
        if (low_mem) {
            a.pool = reinterpret_cast<int*>(p);
            p += bwd::align256(bwd::kScratchSlots * sizeof(int));
            a.scratch = reinterpret_cast<float*>(p);
            p += (size_t)bwd::kScratchSlots * 2 * bwd::kChunkSegs * bwd::kSliceElems * sizeof(float);
        }
        a.ckpt = reinterpret_cast<float*>(p);
        a.status = status;
        auto kernel = low_mem ? bwd::bwd_kernel<true> : bwd::bwd_kernel<false>;
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 bwd::kSmemBytes);
        // every replay slot free at launch; more slots than SMs
        if (e == cudaSuccess && low_mem) {
            int dev = 0, sms = 0;
            e = cudaGetDevice(&dev);
            if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            if (e == cudaSuccess && sms > bwd::kScratchSlots) {
                if (owned) cudaFreeAsync(ws, st);
                return set_error(KDA_ERR_UNSUPPORTED, "more SMs than low-memory replay slots");
            }
            if (e == cudaSuccess)
                e = cudaMemsetAsync(a.pool, 0, bwd::kScratchSlots * sizeof(int), st);
        }
        if (e == cudaSuccess) {
            kernel<<<(unsigned)(pairs * bwd::kSlices), bwd::kThreads, bwd::kSmemBytes, st>>>(a);
            e = cudaGetLastError();
        }
    }
    if (e == cudaSuccess) {
        const int outs = H * (kDim + 1);
        bwd::bwd_param_kernel<<<(outs + 255) / 256, 256, 0, st>>>(
            static_cast<const float*>(ws), reinterpret_cast<const float*>(
                static_cast<const uint8_t*>(ws) +
                bwd::align256((size_t)N * H * bwd::kSlices * sizeof(float))),
            (int)N, H, dA_log, ddt_bias);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess && (flags & KDA_FWD_QK_L2NORM) && total > 0) {
        const long long rows = total * H;  // (rows + 7) / 8 <= INT32_MAX, checked above
        bwd::bwd_l2norm_kernel<<<dim3((unsigned)((rows + 7) / 8), 2), 256, 0, st>>>(
            static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k), dq, dk,
            rows);
        e = cudaGetLastError();
    }
    kda_status_t rc = e == cudaSuccess ? KDA_OK : cuda_error(e, "backward kernel launch");
    if (owned) {
        cudaError_t f = cudaFreeAsync(ws, st);
        if (f != cudaSuccess && rc == KDA_OK) rc = cuda_error(f, "cudaFreeAsync(workspace)");
    }
    return rc;
}
