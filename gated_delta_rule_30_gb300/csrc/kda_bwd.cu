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
// the state entering every 16-token segment (checkpoints, fp32, workspace).
// It then takes the segments last to first: from the segment's checkpoint it
// recomputes the states entering tokens 8..15 into shared memory, walks those
// tokens backwards, then does the same for tokens 0..7.  Forward work per
// token is thus 2.5 state updates; the backward walk is the rest.
// This is the token-recurrent form of the backward pass, the plain GPU
// counterpart of the fp64 reverse-mode oracle.
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "kda.h"
#include "kda_internal.h"

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
constexpr int kPart = 388;                 // dq[128] | dk[128] | da[128] | dbeta, padded

// Dynamic shared memory of one CTA (byte offsets).
constexpr int kSmSt = 0;                                         // float4 [kHalf][4][kThreads]
constexpr int kSmQ = kSmSt + kHalf * 4 * kThreads * 16;          // float [kSeg][128]
constexpr int kSmK = kSmQ + kSeg * kDim * 4;                     // float [kSeg][128]
constexpr int kSmA = kSmK + kSeg * kDim * 4;                     // float [kSeg][128] decays
constexpr int kSmV = kSmA + kSeg * kDim * 4;                     // float [kSeg][kVs]
constexpr int kSmDO = kSmV + kSeg * kVs * 4;                     // float [kSeg][kVs]
constexpr int kSmB = kSmDO + kSeg * kVs * 4;                     // float [kSeg]
constexpr int kSmSlot = kSmB + kSeg * 4;                         // float [2][kWarps][kPart]
constexpr int kSmPart = kSmSlot + 2 * kWarps * kPart * 4;        // float [2][kHalf][kPart]
constexpr int kSmemBytes = kSmPart + 2 * kHalf * kPart * 4;
static_assert(kSmemBytes <= 227 * 1024, "shared memory of the backward kernel");
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
    float* ckpt;             // [slots][H][kSlices][kSliceElems]
    int* status;
};

// Checkpoint slots of sequence n start at floor(cu[n] / 16) + n: consecutive
// sequences' ranges cannot overlap (sequence n has at most floor(L / 16) + 1
// segments), and all fit in floor(total / 16) + N + 1 slots.
__host__ __device__ inline long long ckpt_slots(long long total, long long N) {
    return total / kSeg + N + 1;
}

__device__ __forceinline__ float softplus(float x) {
    return fmaxf(x, 0.f) + log1pf(expf(-fabsf(x)));
}

// Gate of one (token, channel): pre-clamp log-decay and the decay itself.
__device__ __forceinline__ void gate(float x, float expA, float lb, float& pre, float& a) {
    pre = -expA * softplus(x);
    a = expf(fmaxf(pre, lb));
}

// Column sums over the 32 lanes of a warp (all lanes end with the same sums:
// each butterfly step adds the same two values on both partners).
__device__ __forceinline__ void warp_sum4(float (&p)[4]) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
#pragma unroll
        for (int m = 0; m < 4; ++m) p[m] += __shfl_xor_sync(0xffffffffu, p[m], o);
    }
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

// Stages one segment's token data in shared memory as fp32: q, k and the
// decays a of all 128 key channels, v and dout of this CTA's value columns,
// beta.  Rows at or past len are zero (never used).  with_q: also q and dout.
__device__ __forceinline__ void stage_segment(const BwdArgs& P, uint8_t* sm, long long row0,
                                              int h, int len, int col0, float expA,
                                              bool with_q, int tid) {
    float* qs = reinterpret_cast<float*>(sm + kSmQ);
    float* ks = reinterpret_cast<float*>(sm + kSmK);
    float* as = reinterpret_cast<float*>(sm + kSmA);
    float* vs = reinterpret_cast<float*>(sm + kSmV);
    float* dos = reinterpret_cast<float*>(sm + kSmDO);
    float* bs = reinterpret_cast<float*>(sm + kSmB);
    const int H = P.H;
    {   // 16 tokens x 128 channels = 256 pieces of 8 channels, one per thread
        const int t = tid >> 4, c8 = (tid & 15) * 8;
        float kq[8], qq[8], aa[8];
        if (t < len) {
            const long long off = ((row0 + t) * H + h) * kDim + c8;
            const uint4 kr = *reinterpret_cast<const uint4*>(P.k + off);
            const uint4 gr = *reinterpret_cast<const uint4*>(P.g + off);
            const __nv_bfloat16* kb = reinterpret_cast<const __nv_bfloat16*>(&kr);
            const __nv_bfloat16* gb = reinterpret_cast<const __nv_bfloat16*>(&gr);
            const float* dtb = P.dt_bias + (long long)h * kDim + c8;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                kq[e] = __bfloat162float(kb[e]);
                float pre;
                gate(__bfloat162float(gb[e]) + dtb[e], expA, P.lower_bound, pre, aa[e]);
            }
            if (with_q) {
                const uint4 qr = *reinterpret_cast<const uint4*>(P.q + off);
                const __nv_bfloat16* qb = reinterpret_cast<const __nv_bfloat16*>(&qr);
#pragma unroll
                for (int e = 0; e < 8; ++e) qq[e] = __bfloat162float(qb[e]);
            }
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) kq[e] = qq[e] = aa[e] = 0.f;
        }
#pragma unroll
        for (int e = 0; e < 8; e += 4) {
            *reinterpret_cast<float4*>(ks + t * kDim + c8 + e) =
                make_float4(kq[e], kq[e + 1], kq[e + 2], kq[e + 3]);
            *reinterpret_cast<float4*>(as + t * kDim + c8 + e) =
                make_float4(aa[e], aa[e + 1], aa[e + 2], aa[e + 3]);
            if (with_q)
                *reinterpret_cast<float4*>(qs + t * kDim + c8 + e) =
                    make_float4(qq[e], qq[e + 1], qq[e + 2], qq[e + 3]);
        }
    }
    // v and dout: 16 tokens x 32 columns = 64 pieces of 8 each
    if (tid < 128 && (tid < 64 || with_q)) {
        const int piece = tid & 63, t = piece >> 2, c8 = (piece & 3) * 8;
        const __nv_bfloat16* src = tid < 64 ? P.v : P.dout;
        float* dst = tid < 64 ? vs : dos;
        float x[8];
        if (t < len) {
            const uint4 r = *reinterpret_cast<const uint4*>(src + ((row0 + t) * H + h) * kDim +
                                                           col0 + c8);
            const __nv_bfloat16* rb = reinterpret_cast<const __nv_bfloat16*>(&r);
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = __bfloat162float(rb[e]);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = 0.f;
        }
        *reinterpret_cast<float4*>(dst + t * kVs + c8) = make_float4(x[0], x[1], x[2], x[3]);
        *reinterpret_cast<float4*>(dst + t * kVs + c8 + 4) = make_float4(x[4], x[5], x[6], x[7]);
    } else if (tid >= 128 && tid < 128 + kSeg) {
        const int t = tid - 128;
        bs[t] = t < len ? __bfloat162float(P.beta[(row0 + t) * H + h]) : 0.f;
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
    const float* qs = reinterpret_cast<const float*>(sm + kSmQ);
    const float* ks = reinterpret_cast<const float*>(sm + kSmK);
    const float* as = reinterpret_cast<const float*>(sm + kSmA);
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
    auto ckpt_at = [&](int s) {
        return reinterpret_cast<float4*>(P.ckpt + (((slot0 + s) * H + h) * kSlices + rank) *
                                                      (long long)kSliceElems);
    };

    // 1. forward sweep: the state entering every segment (the last segment's
    //    tokens are replayed by the walk, so the sweep stops before them)
    for (int s = 0; s < nseg; ++s) {
        save_piece(ckpt_at(s), S, tid);  // read back later by this same thread
        if (s == nseg - 1) break;
        __syncthreads();
        stage_segment(P, sm, row0 + (long long)s * kSeg, h, kSeg, col0, expA, false, tid);
        __syncthreads();
        for (int t = 0; t < kSeg; ++t) {
            float a[4], kk[4], vv[4];
            ld4(as + t * kDim + 4 * lane, a);
            ld4(ks + t * kDim + 4 * lane, kk);
            ld4(vs + t * kVs + 4 * warp, vv);
            fwd_token(S, a, kk, vv, bs[t]);
        }
    }

    // 2. backward walk, segments last to first, each in two halves
    float accA = 0.f, accB = 0.f;  // dA_log and ddt_bias of key channel 32 rank + lane
    int cb = 0;                    // part[] buffer of the current half
    for (int s = nseg - 1; s >= 0; --s) {
        const int len = min(kSeg, L - s * kSeg);
        const long long rs = row0 + (long long)s * kSeg;
        __syncthreads();
        stage_segment(P, sm, rs, h, len, col0, expA, true, tid);
        __syncthreads();
        for (int half = len > kHalf ? 1 : 0; half >= 0; --half) {
            const int t0 = half * kHalf, t1 = min(len, t0 + kHalf);
            {   // states entering tokens t0 .. t1 - 1, from the checkpoint
                float R[4][4];
                load_piece(ckpt_at(s), R, tid);
                for (int t = 0; t < t1; ++t) {
                    if (t >= t0) save_piece(st + (t - t0) * 4 * kThreads, R, tid);
                    if (t + 1 < t1) {
                        float a[4], kk[4], vv[4];
                        ld4(as + t * kDim + 4 * lane, a);
                        ld4(ks + t * kDim + 4 * lane, kk);
                        ld4(vs + t * kVs + 4 * warp, vv);
                        fwd_token(R, a, kk, vv, bs[t]);
                    }
                }
            }
            for (int t = t1 - 1; t >= t0; --t) {
                float a[4], kk[4], qq[4], vv[4], oo[4], Sp[4][4];
                ld4(as + t * kDim + 4 * lane, a);
                ld4(ks + t * kDim + 4 * lane, kk);
                ld4(qs + t * kDim + 4 * lane, qq);
                ld4(vs + t * kVs + 4 * warp, vv);
                ld4(dos + t * kVs + 4 * warp, oo);
                const float b = bs[t];
                load_piece(st + (t - t0) * 4 * kThreads, Sp, tid);
                // recompute: S~ = Diag(a) S, r = S~^T k, u = beta (v - r)
                float St[4][4], r[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        St[i][m] = a[i] * Sp[i][m];
                        r[m] = fmaf(St[i][m], kk[i], r[m]);
                    }
                warp_sum4(r);
                float e[4], u[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    e[m] = vv[m] - r[m];
                    u[m] = b * e[m];
                }
                // o = scale S'^T q
                float dqp[4], dkp[4], dap[4], du[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float x = 0.f;
#pragma unroll
                    for (int m = 0; m < 4; ++m) x = fmaf(fmaf(kk[i], u[m], St[i][m]), oo[m], x);
                    dqp[i] = P.scale * x;
                    const float sq = P.scale * qq[i];
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        dS[i][m] = fmaf(sq, oo[m], dS[i][m]);
                        du[m] = fmaf(dS[i][m], kk[i], du[m]);
                    }
                }
                // S' = S~ + k u^T
                warp_sum4(du);
                float dbp = 0.f, dr[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    dbp = fmaf(du[m], e[m], dbp);
                    dr[m] = -b * du[m];
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float x = 0.f;
#pragma unroll
                    for (int m = 0; m < 4; ++m) x = fmaf(dS[i][m], u[m], x);
                    // r = S~^T k
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        x = fmaf(St[i][m], dr[m], x);
                        dS[i][m] = fmaf(kk[i], dr[m], dS[i][m]);
                    }
                    dkp[i] = x;
                    // S~ = Diag(a) S
                    float y = 0.f;
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        y = fmaf(dS[i][m], Sp[i][m], y);
                        dS[i][m] *= a[i];
                    }
                    dap[i] = y;
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
            // the pair's row sums over the four CTAs; then the per-channel outputs
            cluster.sync();
            if (t0 + warp < t1) {
                const int c = rank * kVs + lane;
                const long long row = rs + t0 + warp;
                float sq = 0.f, sk = 0.f, sa = 0.f, sb = 0.f;
#pragma unroll
                for (int r = 0; r < kSlices; ++r) {
                    const float* rp =
                        cluster.map_shared_rank(part + (cb * kHalf + warp) * kPart, (unsigned)r);
                    sq += rp[c];
                    sk += rp[kDim + c];
                    sa += rp[2 * kDim + c];
                    sb += rp[3 * kDim];
                }
                const long long off = (row * H + h) * kDim + c;
                const float x = __bfloat162float(P.g[off]) + P.dt_bias[(long long)h * kDim + c];
                float pre, a;
                gate(x, expA, lb, pre, a);
                const float dpre = pre >= lb ? sa * a : 0.f;
                accA = fmaf(pre, dpre, accA);
                const float dx = -expA * dpre / (1.f + expf(-x));
                accB += dx;
                P.dq[off] = sq;
                P.dk[off] = sk;
                P.dg[off] = dx;
                if (rank == 0 && lane == 0) P.dbeta[row * H + h] = sb;
            }
            cb ^= 1;
        }
    }

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
    // no CTA leaves while a peer may still read its shared memory
    cluster.sync();
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

}  // namespace bwd
}  // namespace kda

// ============================================================================= host side
namespace kda {
namespace bwd {
namespace {

constexpr size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

size_t ws_bytes(long long total, long long N, long long H) {
    const size_t pairs = (size_t)N * (size_t)H;
    return align256(pairs * kSlices * sizeof(float)) + align256(pairs * kDim * sizeof(float)) +
           (size_t)ckpt_slots(total, N) * (size_t)H * kSlices * kSliceElems * sizeof(float);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace bwd
}  // namespace kda

using namespace kda;

extern "C" size_t kda_bwd_workspace_size(int32_t B, int32_t T, int32_t H, int32_t num_seqs,
                                         int32_t has_cu_seqlens) {
    clear_error();
    if (B < 1 || T < 0 || H < 1 || (has_cu_seqlens && (B != 1 || num_seqs < 0))) {
        set_error(KDA_ERR_INVALID_ARGUMENT, "invalid sizes");
        return 0;
    }
    const long long N = has_cu_seqlens ? num_seqs : B;
    return bwd::ws_bytes((long long)B * T, N, H);
}

extern "C" kda_status_t kda_bwd(const void* q, const void* k, const void* v, const void* g,
                                const void* beta, float scale, const float* A_log,
                                const float* dt_bias, float lower_bound,
                                const void* initial_state, kda_dtype_t initial_dtype,
                                const void* dout, const float* dfinal_state,
                                const int32_t* cu_seqlens, int32_t num_seqs, int32_t B,
                                int32_t T, int32_t H, int32_t K, int32_t V, float* dq, float* dk,
                                float* dv, float* dg, float* dbeta, float* dA_log,
                                float* ddt_bias, float* dinitial_state, void* workspace,
                                size_t workspace_bytes_, void* stream) {
    using bwd::aligned16;
    clear_error();
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
    const size_t need = bwd::ws_bytes(total, N, H);
    void* ws = workspace;
    bool owned = false;
    if (N > 0) {
        if (!ws) {
            cudaError_t e = cudaMallocAsync(&ws, need, st);
            if (e != cudaSuccess) return cuda_error(e, "cudaMallocAsync(workspace)");
            owned = true;
        } else {
            if (workspace_bytes_ < need)
                return set_error(KDA_ERR_INVALID_ARGUMENT,
                                 "workspace smaller than kda_bwd_workspace_size()");
            if (reinterpret_cast<uintptr_t>(ws) & 255u)
                return set_error(KDA_ERR_INVALID_ARGUMENT, "workspace must be 256-byte aligned");
        }
    }
    int* status = device_status_ptr();
    if (!status) return KDA_ERR_CUDA;
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
        a.ckpt = reinterpret_cast<float*>(p);
        a.status = status;
        e = cudaFuncSetAttribute(bwd::bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 bwd::kSmemBytes);
        if (e == cudaSuccess) {
            bwd::bwd_kernel<<<(unsigned)(pairs * bwd::kSlices), bwd::kThreads, bwd::kSmemBytes,
                              st>>>(a);
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
    kda_status_t rc = e == cudaSuccess ? KDA_OK : cuda_error(e, "backward kernel launch");
    if (owned) {
        cudaError_t f = cudaFreeAsync(ws, st);
        if (f != cudaSuccess && rc == KDA_OK) rc = cuda_error(f, "cudaFreeAsync(workspace)");
    }
    return rc;
}
