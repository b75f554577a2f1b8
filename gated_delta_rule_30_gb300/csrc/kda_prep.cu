// kda_prep.cu -- chunk kernel of the KDA forward pass: everything that does
// not depend on the running state, for one 64-token chunk of one head.
//
// For the chunk's tokens t = 0..63 (padding t >= len behaves as q = k = v = 0,
// beta = 0, log-decay 0) and key channel c, with alpha_t = exp(la_t),
//   la_t      = max(-exp(A_log[h]) * softplus(g_t + dt_bias[h]), lower_bound)
//   E_t       = prod_{s<=t} alpha_s               = exp(G_t)
//   F_t       = prod_{t<s<=63} alpha_s            = exp(G_last - G_t)
//   A[i][j]   = beta_i sum_c k_ic k_jc exp(G_ic - G_jc)       (j < i)
//   Aqk[i][j] = sum_c q_ic k_jc exp(G_ic - G_jc)              (j <= i)
//   T         = (I + A)^-1 (unit lower triangular)
//   W         = T diag(beta) (K o E),  U = T diag(beta) V
// and writes W, scale*(Q o E), (K o F)^T, scale*Aqk (as a bf16 hi/lo pair),
// U^T and exp(G_last) in
// the layout of one record (see kda_internal.h).  This is the chunkwise form
// of the gated delta rule (reading of "Flashkda Delta Attention", "Core Kernel
// API"; the pages give only the call), with the exponentials of G differences
// factored per 16-token sub-block so that no factor overflows fp32/bf16:
// for rows in sub-block a the reference point is token m_a = 16a + 7,
//   left_i  = x_i o exp(G_i - G_{m_a})     (x = k or q),
//   right_j = k_j o exp(G_{m_a} - G_j)     (j < 16(a+1)),
// so |exponent| <= 8 |lower_bound| inside a sub-block and <= 0 across them.
//
// Work split (128 threads, thread = key channel): the gate, decays and every
// scaled operand are elementwise over tokens for a fixed channel; the four
// score products (one per row sub-block, M=128 rows = k and q rows of that
// sub-block, N = 16(a+1) key tokens, K = 128 channels), and the two WY
// products (M = 128 channels, N = 64 tokens, K = 64 tokens) run on tcgen05
// with fp32 accumulators in TMEM; the triangular inverse is fp32 forward
// substitution (thread j owns column j of T).
#include <cuda_runtime.h>

#include "kda_internal.h"
#include "tc.cuh"

namespace kda {
namespace {

constexpr int kThreads = 128;
// shared memory map (bytes)
constexpr uint32_t kSmQ = 0, kSmK = 16384, kSmV = 32768, kSmG = 49152;  // staging tiles [64][128]
constexpr uint32_t kSmLeft = 0;       // 32 KB   (aliases staging after it is consumed)
constexpr uint32_t kSmR = 32768;      // 40 KB   R_0..R_3
constexpr uint32_t kSmVbT = 73728;    // 16 KB   (beta V)^T, K-major, M = 128 value channels, K = 64
constexpr uint32_t kSmKbT = 90112;    // 16 KB   (beta K o E)^T
constexpr uint32_t kSmA = 0;          // fp32 [64][kAStride] (aliases Left after the score MMAs)
constexpr uint32_t kSmTT = 32768;     // 8 KB    T^T as MN-major B operand (aliases R)
constexpr uint32_t kSmBytes = 106496;
constexpr int kAStride = 68;
// R_a (16(a+1) rows x 256 B) starts at 2048 a (a+1): 0, 4096, 12288, 24576
__host__ __device__ constexpr uint32_t r_off(int a) { return 2048u * a * (a + 1); }
// score block a occupies TMEM columns [8 a (a+1), 8 (a+1)(a+2)): 0, 16, 48, 96
__host__ __device__ constexpr uint32_t d_col(int a) { return 8u * a * (a + 1); }
constexpr uint32_t kTmemCols = 256;

struct PrepArgs {
    const __nv_bfloat16* q;
    const __nv_bfloat16* k;
    const __nv_bfloat16* v;
    const __nv_bfloat16* g;
    const __nv_bfloat16* beta;
    const float* A_log;
    const float* dt_bias;
    float lower_bound;
    float scale;
    int H;
    int N;
    const int32_t* flags;
    const int32_t* chunk_off;
    const ChunkInfo* info;
    uint8_t* records;
    int* status;
};

__device__ __forceinline__ float lds_bf16(const uint8_t* base, uint32_t off) {
    return bf16_to_f(*reinterpret_cast<const uint16_t*>(base + off));
}

__device__ __forceinline__ void stg_v4(uint8_t* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    *reinterpret_cast<uint4*>(p) = make_uint4(a, b, c, d);
}

__global__ void __launch_bounds__(kThreads, 2) prep_kernel(const PrepArgs P) {
    extern __shared__ __align__(1024) uint8_t sm[];
    __shared__ float sBeta[kChunk];
    __shared__ uint64_t bar;
    __shared__ uint32_t tmem_base;
    __shared__ int s_abort;

    if (P.flags[0] != 1) return;
    // a CTA that already gave up on a bounded wait poisons the launch: skip the rest
    if (*((volatile int*)P.status) & kStatusTimeout) return;
    const int H = P.H;
    const int chunk = blockIdx.x / H;
    const int h = blockIdx.x - chunk * H;
    if (chunk >= P.chunk_off[P.N]) return;
    const ChunkInfo ci = P.info[chunk];
    const int tok0 = ci.tok0, len = ci.len;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int ch = tid;
    uint8_t* rec = P.records + ((size_t)chunk * H + h) * kRecBytes;

    // ---------------------------------------------------------------- staging
    {
        const __nv_bfloat16* srcs[4] = {P.q, P.k, P.v, P.g};
        const uint32_t dsts[4] = {kSmQ, kSmK, kSmV, kSmG};
#pragma unroll
        for (int x = 0; x < 4; ++x) {
#pragma unroll
            for (int it = 0; it < 8; ++it) {
                const int c = tid + kThreads * it;
                const int row = c >> 4, col = c & 15;
                const bool ok = row < len;
                const __nv_bfloat16* src =
                    srcs[x] + ((size_t)(ok ? tok0 + row : tok0) * H + h) * kDim + col * 8;
                cp_async16_zfill(sm + dsts[x] + row * 256 + col * 16, src, ok);
            }
        }
        if (tid < kChunk)
            sBeta[tid] = tid < len ? __bfloat162float(P.beta[(size_t)(tok0 + tid) * H + h]) : 0.f;
        if (warp == 0) {
            tmem_alloc(&tmem_base, kTmemCols);
            tmem_relinquish();
        }
        if (tid == 0) {
            mbar_init(&bar, 1);
            mbar_fence_init();
            s_abort = 0;
        }
        cp_async_wait_all();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }
    const uint32_t tbase = tmem_base;

    // ---------------------------------------------------------------- gate + decays
    float al[kChunk];
    {
        const float dtb = P.dt_bias[h * kDim + ch];
        const float negA = -__expf(P.A_log[h]);
        const float lb = P.lower_bound;
#pragma unroll
        for (int t = 0; t < kChunk; ++t) {
            const float x = lds_bf16(sm, kSmG + t * 256 + ch * 2) + dtb;
            const float sp = fmaxf(x, 0.f) + __logf(1.f + __expf(-fabsf(x)));
            const float la = fmaxf(negA * sp, lb);
            al[t] = (t < len) ? __expf(la) : 1.f;
        }
    }
    uint32_t qp[kChunk / 2], kp[kChunk / 2];
#pragma unroll
    for (int t = 0; t < kChunk; t += 2) {
        qp[t / 2] = pack_bf16(lds_bf16(sm, kSmQ + t * 256 + ch * 2),
                              lds_bf16(sm, kSmQ + (t + 1) * 256 + ch * 2));
        kp[t / 2] = pack_bf16(lds_bf16(sm, kSmK + t * 256 + ch * 2),
                              lds_bf16(sm, kSmK + (t + 1) * 256 + ch * 2));
    }
#define KV(t) ((t) & 1 ? bf16_hi(kp[(t) / 2]) : bf16_lo(kp[(t) / 2]))
#define QV(t) ((t) & 1 ? bf16_hi(qp[(t) / 2]) : bf16_lo(qp[(t) / 2]))
    {
        // prefix pass: (beta K o E)^T to smem, scale * (Q o E) and exp(G_last) to the record
        float E = 1.f;
#pragma unroll
        for (int tg = 0; tg < 8; ++tg) {
            float kb[8], qh[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int t = tg * 8 + u;
                E *= al[t];
                kb[u] = sBeta[t] * KV(t) * E;
                qh[u] = P.scale * QV(t) * E;
            }
            st_shared_v4(smem_addr(sm + kSmKbT + kmaj_off(ch, tg * 8, 128, 1024)),
                         pack_bf16(kb[0], kb[1]), pack_bf16(kb[2], kb[3]), pack_bf16(kb[4], kb[5]),
                         pack_bf16(kb[6], kb[7]));
            stg_v4(rec + kRecWQ + mnmaj_off(64 + tg * 8, ch, 128, 2048), pack_bf16(qh[0], qh[1]),
                   pack_bf16(qh[2], qh[3]), pack_bf16(qh[4], qh[5]), pack_bf16(qh[6], qh[7]));
        }
        reinterpret_cast<float*>(rec + kRecGam)[ch] = E;
        // suffix pass: (K o F)^T to the record
        float F = 1.f;
#pragma unroll
        for (int tg = 7; tg >= 0; --tg) {
            float kt[8];
#pragma unroll
            for (int u = 7; u >= 0; --u) {
                const int t = tg * 8 + u;
                kt[u] = KV(t) * F;
                F *= al[t];
            }
            stg_v4(rec + kRecKT + kmaj_off(ch, tg * 8, 128, 1024), pack_bf16(kt[0], kt[1]),
                   pack_bf16(kt[2], kt[3]), pack_bf16(kt[4], kt[5]), pack_bf16(kt[6], kt[7]));
        }
        // (beta V)^T (thread = value channel)
#pragma unroll
        for (int tg = 0; tg < 8; ++tg) {
            float vb[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int t = tg * 8 + u;
                vb[u] = sBeta[t] * lds_bf16(sm, kSmV + t * 256 + ch * 2);
            }
            st_shared_v4(smem_addr(sm + kSmVbT + kmaj_off(ch, tg * 8, 128, 1024)),
                         pack_bf16(vb[0], vb[1]), pack_bf16(vb[2], vb[3]), pack_bf16(vb[4], vb[5]),
                         pack_bf16(vb[6], vb[7]));
        }
    }
    __syncthreads();  // staging fully consumed; Left / R may now overwrite it

    // ---------------------------------------------------------------- score operands
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        const int b0 = 16 * a;
        // left factors exp(G_i - G_{m_a}) for the 16 tokens of sub-block a (m_a = b0 + 7)
        float lf[16];
        {
            float run = 1.f;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                run *= al[b0 + u];
                lf[u] = run;  // prod_{s=b0}^{b0+u}
            }
            const float inv = 1.f / lf[7];
#pragma unroll
            for (int u = 0; u < 7; ++u) lf[u] *= inv;
            lf[7] = 1.f;
            run = 1.f;
#pragma unroll
            for (int u = 8; u < 16; ++u) {
                run *= al[b0 + u];
                lf[u] = run;  // prod_{s=m_a+1}^{b0+u}
            }
        }
        // rows 32a .. 32a+15: k-left; 32a+16 .. 32a+31: q-left (MN-major, LBO 2048, SBO 128)
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            float kl[8], ql[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int t = b0 + half * 8 + u;
                kl[u] = KV(t) * lf[half * 8 + u];
                ql[u] = QV(t) * lf[half * 8 + u];
            }
            st_shared_v4(smem_addr(sm + kSmLeft + mnmaj_off(32 * a + 8 * half, ch, 128, 2048)),
                         pack_bf16(kl[0], kl[1]), pack_bf16(kl[2], kl[3]), pack_bf16(kl[4], kl[5]),
                         pack_bf16(kl[6], kl[7]));
            st_shared_v4(smem_addr(sm + kSmLeft + mnmaj_off(32 * a + 16 + 8 * half, ch, 128, 2048)),
                         pack_bf16(ql[0], ql[1]), pack_bf16(ql[2], ql[3]), pack_bf16(ql[4], ql[5]),
                         pack_bf16(ql[6], ql[7]));
        }
        // right operand R_a[j] = k_j o exp(G_{m_a} - G_j), j < 16(a+1)
        float rf[64];
        {
            const int m = b0 + 7;
            rf[m] = 1.f;
            float run = 1.f;
#pragma unroll
            for (int j = m - 1; j >= 0; --j) {
                run *= al[j + 1];
                rf[j] = run;  // prod_{s=j+1}^{m}
            }
            run = 1.f;
#pragma unroll
            for (int j = b0 + 15; j > m; --j) {
                rf[j] = run;  // prod_{s=j+1}^{b0+15}
                run *= al[j];
            }
            const float inv = 1.f / run;  // run = prod_{s=m+1}^{b0+15}
#pragma unroll
            for (int j = m + 1; j <= b0 + 15; ++j) rf[j] *= inv;
        }
#pragma unroll
        for (int jg = 0; jg < 2 * (a + 1); ++jg) {
            float r8[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) r8[u] = KV(jg * 8 + u) * rf[jg * 8 + u];
            st_shared_v4(smem_addr(sm + kSmR + r_off(a) + mnmaj_off(jg * 8, ch, 128, 2048)),
                         pack_bf16(r8[0], r8[1]), pack_bf16(r8[2], r8[3]), pack_bf16(r8[4], r8[5]),
                         pack_bf16(r8[6], r8[7]));
        }
    }
#undef KV
#undef QV
    fence_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---------------------------------------------------------------- score MMAs
    if (tid == 0) {
        tc_fence_after();
        const uint32_t left = smem_addr(sm + kSmLeft);
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const uint32_t idesc = idesc_bf16_f32(128, 16 * (a + 1), true, true);
            const uint32_t right = smem_addr(sm + kSmR + r_off(a));
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_bf16(tbase + d_col(a), smem_desc(left + kk * 256, 128, 2048),
                         smem_desc(right + kk * 256, 128, 2048), idesc, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bar);
    }
    if (!mbar_wait(&bar, 0)) {
        atomicOr(P.status, kStatusTimeout);
        s_abort = 1;
    }
    tc_fence_after();
    __syncthreads();
    if (s_abort) goto teardown;

    // ---------------------------------------------------------------- score read-out
    {
        const int a = warp;
        const bool is_k = lane < 16;
        const int i = 16 * a + (lane & 15);
        float row[64];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            uint32_t r[16];
            tmem_load16(taddr(tbase, 32u * a, d_col(a) + 16u * c), r);
#pragma unroll
            for (int u = 0; u < 16; ++u) row[16 * c + u] = __uint_as_float(r[u]);
        }
        float* sA = reinterpret_cast<float*>(sm + kSmA);
        if (is_k) {
            const float b = sBeta[i];
#pragma unroll
            for (int j = 0; j < 64; ++j) sA[i * kAStride + j] = (j < i) ? b * row[j] : 0.f;
        } else {
#pragma unroll
            for (int jg = 0; jg < 8; ++jg) {
                float hi[8], lo[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int j = jg * 8 + u;
                    const float o = (j <= i) ? P.scale * row[j] : 0.f;
                    hi[u] = __bfloat162float(__float2bfloat16_rn(o));
                    lo[u] = o - hi[u];
                }
                stg_v4(rec + kRecAQ + kmaj_off(i, jg * 8, 128, 1024), pack_bf16(hi[0], hi[1]),
                       pack_bf16(hi[2], hi[3]), pack_bf16(hi[4], hi[5]), pack_bf16(hi[6], hi[7]));
                stg_v4(rec + kRecAQL + kmaj_off(i, jg * 8, 128, 1024), pack_bf16(lo[0], lo[1]),
                       pack_bf16(lo[2], lo[3]), pack_bf16(lo[4], lo[5]), pack_bf16(lo[6], lo[7]));
            }
        }
    }
    tc_fence_before();
    __syncthreads();

    // ---------------------------------------------------------------- T = (I + A)^-1
    if (tid < kChunk) {
        const int j = tid;
        const float* sA = reinterpret_cast<const float*>(sm + kSmA);
        float tcol[kChunk];
#pragma unroll
        for (int l = 0; l < kChunk; ++l) tcol[l] = (l == j) ? 1.f : 0.f;
#pragma unroll
        for (int i = 1; i < kChunk; ++i) {
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int l = 0; l < i; l += 4) {
                const float4 a4 = *reinterpret_cast<const float4*>(sA + i * kAStride + l);
                acc[0] = fmaf(a4.x, tcol[l], acc[0]);
                if (l + 1 < i) acc[1] = fmaf(a4.y, tcol[l + 1], acc[1]);
                if (l + 2 < i) acc[2] = fmaf(a4.z, tcol[l + 2], acc[2]);
                if (l + 3 < i) acc[3] = fmaf(a4.w, tcol[l + 3], acc[3]);
            }
            const float s = (acc[0] + acc[1]) + (acc[2] + acc[3]);
            tcol[i] = (i > j) ? -s : tcol[i];
        }
        // T^T as MN-major B operand: element (n = t, k = j), LBO 1024, SBO 128
#pragma unroll
        for (int tg = 0; tg < 8; ++tg)
            st_shared_v4(smem_addr(sm + kSmTT + mnmaj_off(tg * 8, j, 128, 1024)),
                         pack_bf16(tcol[tg * 8 + 0], tcol[tg * 8 + 1]),
                         pack_bf16(tcol[tg * 8 + 2], tcol[tg * 8 + 3]),
                         pack_bf16(tcol[tg * 8 + 4], tcol[tg * 8 + 5]),
                         pack_bf16(tcol[tg * 8 + 6], tcol[tg * 8 + 7]));
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---------------------------------------------------------------- W^T, U^T MMAs
    if (tid == 0) {
        tc_fence_after();
        const uint32_t idesc = idesc_bf16_f32(128, 64, false, true);
        const uint32_t bT = smem_addr(sm + kSmTT);
        const uint32_t aK = smem_addr(sm + kSmKbT);
        const uint32_t aV = smem_addr(sm + kSmVbT);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            mma_bf16(tbase + 0, smem_desc(aK + kk * 256, 128, 1024),
                     smem_desc(bT + kk * 256, 128, 1024), idesc, kk > 0 ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            mma_bf16(tbase + 64, smem_desc(aV + kk * 256, 128, 1024),
                     smem_desc(bT + kk * 256, 128, 1024), idesc, kk > 0 ? 1u : 0u);
        mma_commit(&bar);
    }
    if (!mbar_wait(&bar, 1)) {
        atomicOr(P.status, kStatusTimeout);
        s_abort = 1;
    }
    tc_fence_after();
    __syncthreads();
    if (s_abort) goto teardown;

    // ---------------------------------------------------------------- W, U^T to the record
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint32_t r[16];
        tmem_load16(taddr(tbase, 32u * warp, 16u * c), r);  // W[16c + u][ch]
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const uint32_t* x = r + 8 * half;
            stg_v4(rec + kRecWQ + mnmaj_off(16 * c + 8 * half, ch, 128, 2048),
                   pack_bf16(__uint_as_float(x[0]), __uint_as_float(x[1])),
                   pack_bf16(__uint_as_float(x[2]), __uint_as_float(x[3])),
                   pack_bf16(__uint_as_float(x[4]), __uint_as_float(x[5])),
                   pack_bf16(__uint_as_float(x[6]), __uint_as_float(x[7])));
        }
        tmem_load16(taddr(tbase, 32u * warp, 64u + 16u * c), r);  // U[16c + u][ch]
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const uint32_t* x = r + 8 * half;
            stg_v4(rec + kRecUT + ch * 128 + (16 * c + 8 * half) * 2,
                   pack_bf16(__uint_as_float(x[0]), __uint_as_float(x[1])),
                   pack_bf16(__uint_as_float(x[2]), __uint_as_float(x[3])),
                   pack_bf16(__uint_as_float(x[4]), __uint_as_float(x[5])),
                   pack_bf16(__uint_as_float(x[6]), __uint_as_float(x[7])));
        }
    }

teardown:
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, kTmemCols);
}

}  // namespace

cudaError_t launch_prep(const Problem& p, const Workspace& ws, int* status, cudaStream_t st) {
    if (p.max_chunks == 0 || p.H == 0) return cudaSuccess;
    cudaError_t e =
        cudaFuncSetAttribute(prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmBytes);
    if (e != cudaSuccess) return e;
    PrepArgs a;
    a.q = reinterpret_cast<const __nv_bfloat16*>(p.q);
    a.k = reinterpret_cast<const __nv_bfloat16*>(p.k);
    a.v = reinterpret_cast<const __nv_bfloat16*>(p.v);
    a.g = reinterpret_cast<const __nv_bfloat16*>(p.g);
    a.beta = reinterpret_cast<const __nv_bfloat16*>(p.beta);
    a.A_log = p.A_log;
    a.dt_bias = p.dt_bias;
    a.lower_bound = p.lower_bound;
    a.scale = p.scale;
    a.H = p.H;
    a.N = p.N;
    a.flags = ws.flags;
    a.chunk_off = ws.chunk_off;
    a.info = ws.info;
    a.records = ws.records;
    a.status = status;
    const long long blocks = (long long)p.max_chunks * p.H;
    prep_kernel<<<(unsigned)blocks, kThreads, kSmBytes, st>>>(a);
    return cudaGetLastError();
}

}  // namespace kda
