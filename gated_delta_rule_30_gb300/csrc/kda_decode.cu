// kda_decode.cu -- single-token step of the KDA forward pass (T = 1 per
// sequence, no cu_seqlens): the recurrence applied to one token,
//   S' = (I - beta k k^T) Diag(alpha) S + beta k v^T,   o = scale * S'^T q,
// with log alpha = max(-exp(A_log[h]) * softplus(g + dt_bias[h]), lower_bound)
// per key channel (reading of "Flashkda Delta Attention", "Core Kernel API":
// the recurrent state update of delta attention, taken one token at a time).
//
// With one token there is no chunk to factor: the step is a pass over the
// 128 x 128 state, bound by reading and writing it.  One CTA of 128 threads
// per (sequence, head): the pair's state (one contiguous 64 KB / 32 KB block)
// arrives in shared memory by one bulk copy, thread v updates value column v
// there (a row k of S is 128 consecutive elements, so the column accesses of a
// warp hit distinct banks),
//   r_v  = sum_k alpha_k S[k][v] k_k
//   S'[k][v] = alpha_k S[k][v] + k_k beta (v_v - r_v)
//   o_v  = scale * sum_k S'[k][v] q_k
// in fp32, and one bulk store writes the final state back.  In place (final
// state == initial state) is safe: the store starts after every read.  The
// bulk-copy wait is bounded; on timeout the CTA records kStatusTimeout, waits
// once more for its copy (with the longer drain limit) and writes nothing.
// With q/k normalisation (kda_fwd_ex) q and k are first scaled to
// x / sqrt(|x|^2 + eps) by a block reduction, in fp32.
#include <cuda_runtime.h>

#include <type_traits>

#include "kda_internal.h"
#include "tc.cuh"

namespace kda {
namespace {

constexpr int kDecThreads = kDim;  // one thread per value column

struct DecodeArgs {
    const __nv_bfloat16* q;
    const __nv_bfloat16* k;
    const __nv_bfloat16* v;
    const __nv_bfloat16* g;
    const __nv_bfloat16* beta;
    const float* A_log;
    const float* dt_bias;
    float lower_bound;
    float scale;
    int qk_norm;  // normalise q and k to unit L2 norm first
    __nv_bfloat16* out;
    const void* h0;
    void* hT;
    int H;
};

struct NoState {};

// T: the state's element type in memory (float or __nv_bfloat16; with no
// initial state, the final state's); H0 / HT: T or NoState.
template <typename T, typename H0, typename HT>
__global__ void __launch_bounds__(kDecThreads) decode_kernel(const DecodeArgs P, int* status) {
    extern __shared__ __align__(128) uint8_t smraw[];
    T* sS = reinterpret_cast<T*>(smraw);  // the pair's state, [k][v]
    __shared__ float sA[kDim];             // alpha_k
    __shared__ float sK[kDim];             // k_k
    __shared__ float sQ[kDim];             // q_k
    __shared__ float sRed[2][kDecThreads / 32];  // per-warp sums of k^2, q^2 (q/k normalisation)
    __shared__ uint64_t bar;
    __shared__ int s_fail;
    constexpr uint32_t kStateBytes = kDim * kDim * sizeof(T);
    const int H = P.H;
    const int n = blockIdx.x / H;
    const int h = blockIdx.x - n * H;
    const int t = threadIdx.x;               // value column v, and key channel for the loads
    const uint64_t lim = wait_limit_ns(status);  // of the state-copy wait
    const size_t row = (size_t)n * H + h;    // token row of the [N, 1, H, 128] tensors
    const size_t sbase = row * kDim * kDim;  // state [N, H, 128, 128]

    if (t == 0) {
        s_fail = 0;
        if constexpr (!std::is_same<H0, NoState>::value) {
            mbar_init(&bar, 1);
            mbar_fence_init();
            mbar_arrive_expect_tx(&bar, kStateBytes);
            bulk_g2s(sS, reinterpret_cast<const T*>(P.h0) + sbase, kStateBytes, &bar);
        }
    }
    // gate of key channel t while the state lands:
    // la = max(-exp(A_log) * softplus(x), lower_bound)
    {
        const float x = __bfloat162float(P.g[row * kDim + t]) + P.dt_bias[h * kDim + t];
        const float sp = fmaxf(x, 0.f) + log1pf(expf(-fabsf(x)));
        sA[t] = expf(fmaxf(-expf(P.A_log[h]) * sp, P.lower_bound));
        float kv = __bfloat162float(P.k[row * kDim + t]);
        float qv = __bfloat162float(P.q[row * kDim + t]);
        if (P.qk_norm) {
            // x / sqrt(|x|^2 + eps) for x = k and q: block sums of the squares
            float a = kv * kv, b = qv * qv;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                a += __shfl_xor_sync(0xffffffffu, a, o);
                b += __shfl_xor_sync(0xffffffffu, b, o);
            }
            if ((t & 31) == 0) {
                sRed[0][t >> 5] = a;
                sRed[1][t >> 5] = b;
            }
            __syncthreads();
            a = 0.f;
            b = 0.f;
#pragma unroll
            for (int w = 0; w < kDecThreads / 32; ++w) {
                a += sRed[0][w];
                b += sRed[1][w];
            }
            kv *= rsqrtf(a + kL2NormEps);
            qv *= rsqrtf(b + kL2NormEps);
        }
        sK[t] = kv;
        sQ[t] = qv;
    }
    const float beta = __bfloat162float(P.beta[row]);
    const float vv = __bfloat162float(P.v[row * kDim + t]);
    if constexpr (std::is_same<H0, NoState>::value) {
#pragma unroll 8
        for (int k = 0; k < kDim; ++k) sS[k * kDim + t] = T(0.f);
    }
    __syncthreads();  // barrier initialised (and state zeroed), gate visible
    if constexpr (!std::is_same<H0, NoState>::value) {
        if (!mbar_wait(&bar, 0, lim)) {
            atomicOr(status, kStatusTimeout);
            s_fail = 1;
        }
        __syncthreads();
        if (s_fail) {
            // gave up: wait once more, with the longer drain limit, for the copy in
            // flight so that it never lands after the CTA has left
            if (t == 0) mbar_drain(&bar, 0);
            return;
        }
    }

    float r = 0.f;
#pragma unroll 8
    for (int k = 0; k < kDim; ++k) r = fmaf(sA[k] * float(sS[k * kDim + t]), sK[k], r);
    const float d = beta * (vv - r);
    float o = 0.f;
#pragma unroll 8
    for (int k = 0; k < kDim; ++k) {
        const float sn = fmaf(sK[k], d, sA[k] * float(sS[k * kDim + t]));
        o = fmaf(sn, sQ[k], o);
        if constexpr (!std::is_same<HT, NoState>::value) sS[k * kDim + t] = T(sn);
    }
    P.out[row * kDim + t] = __float2bfloat16_rn(P.scale * o);
    if constexpr (!std::is_same<HT, NoState>::value) {
        fence_async_smem();
        __syncthreads();
        if (t == 0) {
            asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                             reinterpret_cast<T*>(P.hT) + sbase),
                         "r"(smem_addr(sS)), "r"(kStateBytes)
                         : "memory");
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
            asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
        }
    }
}

template <typename T, typename H0, typename HT>
cudaError_t launch_dec(const Problem& p, const DecodeArgs& a, int* status, cudaStream_t st) {
    constexpr uint32_t kStateBytes = kDim * kDim * sizeof(T);
    auto kern = decode_kernel<T, H0, HT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kStateBytes);
    if (e != cudaSuccess) return e;
    const long long blocks = (long long)p.N * p.H;
    kern<<<(unsigned)blocks, kDecThreads, kStateBytes, st>>>(a, status);
    return cudaGetLastError();
}

}  // namespace

bool decode_applies(const Problem& p) { return p.cu == nullptr && p.T == 1 && p.N > 0; }

cudaError_t launch_decode(const Problem& p, int* status, cudaStream_t st) {
    if (p.N == 0 || p.H == 0) return cudaSuccess;
    DecodeArgs a;
    a.q = reinterpret_cast<const __nv_bfloat16*>(p.q);
    a.k = reinterpret_cast<const __nv_bfloat16*>(p.k);
    a.v = reinterpret_cast<const __nv_bfloat16*>(p.v);
    a.g = reinterpret_cast<const __nv_bfloat16*>(p.g);
    a.beta = reinterpret_cast<const __nv_bfloat16*>(p.beta);
    a.A_log = p.A_log;
    a.dt_bias = p.dt_bias;
    a.lower_bound = p.lower_bound;
    a.scale = p.scale;
    a.qk_norm = p.qk_norm ? 1 : 0;
    a.out = reinterpret_cast<__nv_bfloat16*>(p.out);
    a.h0 = p.h0;
    a.hT = p.hT;
    a.H = p.H;
    using F = float;
    using B = __nv_bfloat16;
    const kda_dtype_t d0 = p.h0_dtype, d1 = p.hT_dtype;
    if (d0 == KDA_DTYPE_FP32 && d1 == KDA_DTYPE_FP32) return launch_dec<F, F, F>(p, a, status, st);
    if (d0 == KDA_DTYPE_FP32) return launch_dec<F, F, NoState>(p, a, status, st);
    if (d0 == KDA_DTYPE_BF16 && d1 == KDA_DTYPE_BF16) return launch_dec<B, B, B>(p, a, status, st);
    if (d0 == KDA_DTYPE_BF16) return launch_dec<B, B, NoState>(p, a, status, st);
    if (d1 == KDA_DTYPE_FP32) return launch_dec<F, NoState, F>(p, a, status, st);
    if (d1 == KDA_DTYPE_BF16) return launch_dec<B, NoState, B>(p, a, status, st);
    return launch_dec<F, NoState, NoState>(p, a, status, st);
}

}  // namespace kda
