// kda_prep.cuh -- the chunk kernel's worker body, shared by the stand-alone
// chunk kernel (kda_prep.cu) and the fused kernel (kda_fused.cu).
//
// The chunk kernel of the KDA forward pass: everything that does
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
// U^T and exp(G_last) in the layout of one record (see kda_internal.h).  This
// is the chunkwise form of the gated delta rule (reading of "Flashkda Delta
// Attention", "Core Kernel API"; the pages give only the call), with the
// exponentials of G differences factored per 16-token sub-block so that no
// factor overflows fp32/bf16: for rows in sub-block a the reference point is
// token m_a = 16a + 7,
//   left_i  = x_i o exp(G_i - G_{m_a})     (x = k or q),
//   right_j = k_j o exp(G_{m_a} - G_j)     (j < 16(a+1)),
// so |exponent| <= 8 |lower_bound| inside a sub-block and <= 0 across them.
// Every exp(G_i - G_j) is a product of the alphas between i and j, so the
// only transcendentals are those of the gate itself.
//
// The kernel is persistent (two CTAs per SM, each looping over (chunk, head)
// items): once an item's last MMA has read shared memory, the copies of the
// next item's q, k, v, g are issued, so they land while the current item's
// results are written out.
//
// Work split (256 threads): for the gate, the decays and the scaled operands
// thread (c, h) owns key channel c = tid % 128 and the 32 tokens of half
// h = tid / 128 of the chunk (products that cross the halves are exchanged
// through shared memory).  The score products (M = 128 rows = the k and q
// rows of the four sub-blocks, N = 16 + 32 + 48 + 64 = 160 columns holding
// the four right operands side by side, K = 128 channels; the rows of
// sub-block a only read the columns of its own right operand) and the two WY
// products (M = 128 channels, N = 64 tokens,
// K = 64 tokens) run on tcgen05 with fp32 accumulators in TMEM.  The
// triangular inverse is blocked: the four 16 x 16 diagonal blocks by forward
// substitution (two warps), then the off-diagonal blocks by 2 x 2 block
// recursion (T_10, T_32, then the lower-left 32 x 32 block), in fp32 shared memory.
#pragma once
#include <cuda.h>  // CUtensorMap (the encoder is fetched at run time)
#include <cuda_runtime.h>

#include "kda_internal.h"
#include "tc.cuh"

namespace kda {
namespace prep {


constexpr int kThreads = 256;
// shared memory map (bytes)
constexpr uint32_t kSmQ = 0, kSmK = 16384, kSmG = 49152;  // staging tiles, row-major [64 t][128 c]
// V^T as the A operand of U^T = V^T diag(beta) T^T: the v tile lands row-major and
// is moved in place (v_to_operand) into the MN-major core-matrix layout (8 value
// channels x 8 tokens per 128 B; token groups 128 B apart, channel groups 1024 B
// apart): byte(v, t) = (v/8)*1024 + t*16 + (v%8)*2
constexpr uint32_t kSmV = 73728;      // 16 KB   (live until the WY MMAs)
constexpr uint32_t kSmLeft = 0;       // 32 KB   (aliases the q, k tiles once they are consumed)
constexpr uint32_t kSmR = 32768;      // 40 KB   R_0..R_3 (aliases the g tile)
constexpr uint32_t kSmKbT = 90112;    // 16 KB   (K o E)^T, K-major, M = 128 key channels, K = 64
constexpr uint32_t kSmBytes = 106496;
// after the score MMAs (alias Left / R)
constexpr int kStr = 68;              // fp32 row stride of the 64 x 64 tiles
constexpr uint32_t kSmA = 0;          // A^T (beta-scaled, strictly lower A), fp32 [64][kStr]
constexpr uint32_t kSmT = 17408;      // T, fp32 [64][kStr]
constexpr uint32_t kSmX = 34816;      // products of the inverse's recursion, fp32 (<= 32 x kXb)
constexpr uint32_t kSmTT = 40960;     // T^T as MN-major B operand, bf16 8 KB
// R_a (16(a+1) rows x 256 B) starts at 2048 a (a+1): 0, 4096, 12288, 24576
__host__ __device__ constexpr uint32_t r_off(int a) { return 2048u * a * (a + 1); }
// score block a occupies TMEM columns [8 a (a+1), 8 (a+1)(a+2)): 0, 16, 48, 96
__host__ __device__ constexpr uint32_t d_col(int a) { return 8u * a * (a + 1); }
constexpr uint32_t kTmemCols = 256;
// The thread that issues the U^T tensor stores and, in the fused launch,
// publishes the ready flags: lane 0 of warp 2, a q-row warp of the score
// read-out, which has slack there while warps 0 and 1 invert the diagonal
// blocks (the bulk-group waits must come from the issuing thread; thread 0 is on
// every critical path, and a GPU-scope release taken there stalled its whole
// worker: fused launch 1.40 -> 1.23 ms with the workers alone).
constexpr int kStoreTid = 64;


struct PrepArgs {
    // TMA descriptors of q, k, v, g viewed as [tokens][H][128] bf16 with a box of
    // 64 tokens x 1 head x 128 channels (one 16 KB row-major tile per copy); tm_ut: the U^T block
    // of every record as [record][128 value channels][64 tokens] bf16 with a box of
    // one record's block, 128-byte swizzled in shared memory (written by TMA store)
    CUtensorMap tm_q, tm_k, tm_v, tm_g, tm_ut;
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
    int qk_norm;  // normalise each q and k row (token) to unit L2 norm first
    int hint_records;  // store records with an L2 evict_last policy (read back soon, fused launch)
    const int32_t* flags;
    const int32_t* chunk_off;
    const ChunkInfo* info;
    uint8_t* records;
    int* status;
};

__device__ __forceinline__ float lds_bf16(const uint8_t* base, uint32_t off) {
    return bf16_to_f(*reinterpret_cast<const uint16_t*>(base + off));
}
// 16-byte record store with the L2 policy `pol` (see l2_policy_evict_last)
__device__ __forceinline__ void stg_v4(uint8_t* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d,
                                       uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v4.b32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "r"(a),
                 "r"(b), "r"(c), "r"(d), "l"(pol)
                 : "memory");
}
__device__ __forceinline__ void sts_v4f(uint32_t saddr, const float (&x)[8]) {
    st_shared_v4(saddr, pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]), pack_bf16(x[4], x[5]),
                 pack_bf16(x[6], x[7]));
}
__device__ __forceinline__ void stg_v4f(uint8_t* p, const float (&x)[8], uint64_t pol) {
    stg_v4(p, pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]), pack_bf16(x[4], x[5]),
           pack_bf16(x[6], x[7]), pol);
}

// Factors of the right score operands, produced eight tokens at a time (the
// arrays of a whole sub-block would hold up to 48 more registers at the phase
// with the most live values).  For a reference token m of this half's tokens
// (local indices), the factor of token u is exp(G_m - G_u):
//   u <= m: prod_{s=u+1}^{m} alpha_s, a running product taken downwards from m;
//   u >  m: 1 / prod_{s=m+1}^{u} alpha_s, taken as (prod_{s=u+1}^{e} alpha_s) /
//           (prod_{s=m+1}^{e} alpha_s) over the tokens up to the group's end e.
// back8(al, g, run, f): tokens 8g + 7 down to 8g of a downward run (run is the
// product from the token above the group up to m; f[i] is token 8g + i).
__device__ __forceinline__ void back8(const float (&al)[32], int g, float& run, float (&f)[8],
                                      bool first) {
    // (g is a compile-time constant at every call)
#pragma unroll
    for (int i = 7; i >= 0; --i) {
        if (!(first && i == 7)) run *= al[8 * g + i + 1];
        f[i] = run;
    }
}
// fwd8(al, g, f): tokens 8g .. 8g + 7 after the reference 8g - 1:
// f[i] = 1 / prod_{s=8g}^{8g+i} alpha_s.
__device__ __forceinline__ void fwd8(const float (&al)[32], int g, float (&f)[8]) {
    float run = 1.f;
#pragma unroll
    for (int i = 7; i >= 0; --i) {
        f[i] = run;
        run *= al[8 * g + i];
    }
    const float inv = 1.f / run;
#pragma unroll
    for (int i = 0; i < 8; ++i) f[i] *= inv;
}

// The v tile lands row-major ([64 tokens][128 channels], 256-byte rows); the U
// MMA reads it as the MN-major operand of kSmV.  The move permutes 16-byte
// chunks (token t, channel group c8) -> (c8, t), in place, on 256 threads: every
// thread first loads four chunks (v_tile_load), the caller synchronises, then
// every thread writes them (v_tile_store).  A quarter-warp moves an 8 x 8 block
// of chunks, lane i taking chunk (t0 + i, c0 + (i + s) % 8) at step s, so that
// neither the reads (rows 256 B apart) nor the writes (groups 1024 B apart) meet
// a bank conflict.  Tokens t >= len are written as zeros.
__device__ __forceinline__ void v_chunk(int tid, int j, int& t, int& c8) {
    const int qw = tid >> 3, i = tid & 7;
    const int blk = qw >> 1, s = 4 * (qw & 1) + j;
    t = 8 * (blk & 7) + i;
    c8 = 8 * (blk >> 3) + ((i + s) & 7);
}
__device__ __forceinline__ void v_tile_load(const uint8_t* tile, int tid, int len, uint4 (&x)[4]) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        int t, c8;
        v_chunk(tid, j, t, c8);
        x[j] = t < len ? *reinterpret_cast<const uint4*>(tile + t * 256 + c8 * 16)
                       : make_uint4(0u, 0u, 0u, 0u);
    }
}
__device__ __forceinline__ void v_tile_store(uint8_t* tile, int tid, const uint4 (&x)[4]) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        int t, c8;
        v_chunk(tid, j, t, c8);
        *reinterpret_cast<uint4*>(tile + c8 * 1024 + t * 16) = x[j];
    }
}

// Per-worker state that lives outside the dynamic shared-memory area.
struct PrepShared {
    float sBeta[kChunk];
    float sRn[2][kChunk];  // 1 / |row| of the q (0) and k (1) rows, with q/k normalisation
    float sTot[2][kDim];  // product of each half's alphas
    float sQf[2][kDim];   // prod_{s=32}^{39} and prod_{s=32}^{55} alpha_s
    uint64_t bar;       // MMA completion
    uint64_t bar_g;     // g tile landed
    uint64_t bar_qkv;   // q, k, v tiles landed
    uint32_t tmem_base;
    int s_abort;
    int pending;  // with `ready`: the item whose flag waits for its U^T store (kStoreTid)
};

// Barrier over the kThreads threads of one worker.
__device__ __forceinline__ void sub_sync(uint32_t bar_id) {
    asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "n"(kThreads) : "memory");
}
// One TMA tile copy (box of the tensor map at coordinates {x, y, z}) into shared
// memory, completing on `bar`.
// The inputs are read once: the copies mark their lines evict_first in L2.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z,
                                            uint64_t* bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar)), "l"(pol)
        : "memory");
}
// TMA tensor store of one box from shared memory, in the thread's bulk async-group.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, int x, int y, int z,
                                             const void* src, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group.L2::cache_hint [%0, {%1, %2, %3}], "
        "[%4], %5;" ::"l"(reinterpret_cast<uint64_t>(map)),
        "r"(x), "r"(y), "r"(z), "r"(smem_addr(src)), "l"(pol)
        : "memory");
}
// Row `ch` (64 bf16 values, 128 B) of a 128 x 64 tile in the 128-byte swizzled
// layout the tensor store reads: 16-byte chunk j of row ch sits in slot
// j ^ (ch % 8), so the eight rows a quarter-warp writes fall in distinct banks.
// r[c][u] holds the value of column 16 c + u.
__device__ __forceinline__ void sts_row_swizzled(uint8_t* tile, int ch, const uint32_t (&r)[4][16]) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint32_t* x = &r[j >> 1][8 * (j & 1)];
        st_shared_v4(smem_addr(tile + ch * 128 + ((j ^ (ch & 7)) << 4)),
                     pack_bf16(__uint_as_float(x[0]), __uint_as_float(x[1])),
                     pack_bf16(__uint_as_float(x[2]), __uint_as_float(x[3])),
                     pack_bf16(__uint_as_float(x[4]), __uint_as_float(x[5])),
                     pack_bf16(__uint_as_float(x[6]), __uint_as_float(x[7])));
    }
}
__device__ __forceinline__ void st_relaxed_gpu(int* p, int v) {
    asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Publish ready[item] = 1 once every store of that record is performed: the
// calling thread's tensor stores (waited for), then, through a GPU-scope fence,
// everything ordered before this thread.  (The fence costs about a thousand
// cycles of the SM's progress, wherever it is taken; batching several flags
// behind one fence did not shorten the fused launch.)
__device__ __forceinline__ void publish_flag(int* ready, int item) {
    bulk_wait<0>();
    fence_async_global();
    __threadfence();
    st_relaxed_gpu(ready + item, 1);
}

// Off-diagonal part of T = (I + A)^-1 from its four diagonal 16 x 16 blocks
// (already in sT), by 2 x 2 block recursion on all kThreads threads:
//   T_10 = -T_11 A_10 T_00  and  T_32 = -T_33 A_32 T_22   (steps A1, A2), after
//   which T_lo = T[0:32][0:32] and T_hi = T[32:64][32:64] are the inverses of
//   the two diagonal halves, then
//   T[32:64][0:32] = -T_hi A[32:64][0:32] T_lo             (steps B1, B2).
// In B1 each warp owns four columns j and sums only c >= its first column (T_lo
// is lower triangular); in B2 each warp owns four rows i and sums only c <= its
// last row (T_hi is lower triangular).  sAT[l][i] = A[i][l]; sX is scratch.
constexpr int kXs = 18;   // row stride of the 16 x 16 products in sX
constexpr int kXb = 34;   // row stride of the 32 x 32 product in sX
__device__ __forceinline__ void offdiag_inverse(const float* sAT, float* sT, float* sX, int tid,
                                                uint32_t bar_id) {
    const int warp = tid >> 5, lane = tid & 31;
    {
        // A1: X = A_ab T_bb for (a, b) = (1, 0) (threads 0-127) and (3, 2) (128-255);
        // thread: row i, columns j, j + 1
        const int blk = tid >> 7, i = tid & 15, j = ((tid >> 4) & 7) * 2;
        const int r0 = 16 + 32 * blk, c0 = 32 * blk;
        float x0 = 0.f, x1 = 0.f;
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            const float av = sAT[(c0 + c) * kStr + r0 + i];
            const float2 tv = *reinterpret_cast<const float2*>(sT + (c0 + c) * kStr + c0 + j);
            x0 = fmaf(av, tv.x, x0);
            x1 = fmaf(av, tv.y, x1);
        }
        *reinterpret_cast<float2*>(sX + blk * 16 * kXs + i * kXs + j) = make_float2(x0, x1);
    }
    sub_sync(bar_id);
    {
        // A2: T_ab = -T_aa X; thread: rows i, i + 1, column j
        const int blk = tid >> 7, j = tid & 15, i = ((tid >> 4) & 7) * 2;
        const int r0 = 16 + 32 * blk, c0 = 32 * blk;
        float y0 = 0.f, y1 = 0.f;
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            const float xv = sX[blk * 16 * kXs + c * kXs + j];
            y0 = fmaf(sT[(r0 + i) * kStr + r0 + c], xv, y0);
            y1 = fmaf(sT[(r0 + i + 1) * kStr + r0 + c], xv, y1);
        }
        sT[(r0 + i) * kStr + c0 + j] = -y0;
        sT[(r0 + i + 1) * kStr + c0 + j] = -y1;
    }
    sub_sync(bar_id);
    {
        // B1: X = A[32:64][0:32] T_lo; warp w: columns 4w .. 4w + 3 (lanes 16-31 the
        // upper pair), rows 2 (lane % 16) and + 1
        const int i = (lane & 15) * 2, j = 4 * warp + 2 * (lane >> 4);
        float x00 = 0.f, x01 = 0.f, x10 = 0.f, x11 = 0.f;
#pragma unroll 4
        for (int c = 4 * warp; c < 32; ++c) {
            const float2 av = *reinterpret_cast<const float2*>(sAT + c * kStr + 32 + i);
            const float2 tv = *reinterpret_cast<const float2*>(sT + c * kStr + j);
            x00 = fmaf(av.x, tv.x, x00);
            x01 = fmaf(av.x, tv.y, x01);
            x10 = fmaf(av.y, tv.x, x10);
            x11 = fmaf(av.y, tv.y, x11);
        }
        *reinterpret_cast<float2*>(sX + i * kXb + j) = make_float2(x00, x01);
        *reinterpret_cast<float2*>(sX + (i + 1) * kXb + j) = make_float2(x10, x11);
    }
    sub_sync(bar_id);
    {
        // B2: T[32:64][0:32] = -T_hi X; warp w: rows 4w .. 4w + 3 (lanes 16-31 the
        // upper pair), columns 2 (lane % 16) and + 1
        const int i = 4 * warp + 2 * (lane >> 4), j = (lane & 15) * 2;
        float y00 = 0.f, y01 = 0.f, y10 = 0.f, y11 = 0.f;
        const float* t0p = sT + (32 + i) * kStr + 32;
#pragma unroll 4
        for (int c = 0; c < 4 * warp + 4; ++c) {
            const float2 xv = *reinterpret_cast<const float2*>(sX + c * kXb + j);
            const float t0 = t0p[c], t1 = t0p[kStr + c];
            y00 = fmaf(t0, xv.x, y00);
            y01 = fmaf(t0, xv.y, y01);
            y10 = fmaf(t1, xv.x, y10);
            y11 = fmaf(t1, xv.y, y11);
        }
        *reinterpret_cast<float2*>(sT + (32 + i) * kStr + j) = make_float2(-y00, -y01);
        *reinterpret_cast<float2*>(sT + (33 + i) * kStr + j) = make_float2(-y10, -y11);
    }
    sub_sync(bar_id);
}

// One chunk-kernel worker: `kThreads` threads (thread index `tid`), the
// shared-memory area `sm` (kSmBytes, 1024-byte aligned) and the small state
// `S`, synchronised by named barrier `bar_id` (and `bar_k`, over the half of
// the worker's warps that read the key rows of the scores).  It processes the (chunk, head)
// items first_item, first_item + item_stride, ...; with `ready` non-null it
// publishes ready[item] = 1 (release, GPU scope) once an item's record is
// complete.
//
// QKN: normalise the q and k rows first (P.qk_norm); a template parameter so
// that the common kernels carry none of that code (the worker's instruction
// footprint matters when two copies share an SM).
template <bool QKN>
__device__ __forceinline__ void prep_body(const PrepArgs& P, uint8_t* sm, PrepShared& S,
                                          const int tid, const uint32_t bar_id,
                                          const uint32_t bar_k, const int first_item,
                                          const int item_stride, int* ready,
                                          const bool relinquish) {

    if (P.flags[0] != 1) return;
    // L2 policies: the inputs are streamed once; the records are read back soon
    // by the fused launch's recurrence (elsewhere they outgrow L2: no hint)
    const uint64_t pol_in = l2_policy_evict_first();
    const uint64_t pol_rec = P.hint_records ? l2_policy_evict_last() : l2_policy_evict_normal();
    // a CTA that already gave up on a bounded wait poisons the launch: skip the
    // rest (decided once, so every thread of the worker takes the same path)
    if (tid == 0) {
        S.s_abort = (*((volatile int*)P.status) & kStatusTimeout) ? 1 : 0;
        // the swizzled U^T staging tile needs a 1024-byte aligned area
        if (smem_addr(sm) & 1023u) {
            atomicOr(P.status, kStatusLayout);
            S.s_abort = 1;
        }
    }
    sub_sync(bar_id);
    if (S.s_abort) return;
    const uint64_t lim = wait_limit_ns(P.status);  // of every wait that may give up
    const int H = P.H;
    const int n_items = P.chunk_off[P.N] * H;  // valid (chunk, head) pairs
    int item = first_item;
    if (item >= n_items) return;
    const int warp = tid >> 5, lane = tid & 31;
    const int ch = tid & (kDim - 1);
    const int half = tid >> 7;
    const int t0 = 32 * half;  // first token of this thread's half

    // Issue the tile copies of one item's g (on its own barrier: the g tile's
    // area is free once the previous item's score MMA has read it, so it is
    // requested that early and the gate can start at once) and of its q, k, v
    // (once the previous item's WY MMAs are done), and set its beta.  Rows past
    // the end of the tensor read as zeros; rows past the chunk's length (the
    // next sequence's tokens) are zeroed after landing.
    auto stage_g = [&](int tok0, int hh) {  // thread 0
        mbar_arrive_expect_tx(&S.bar_g, kChunk * kDim * 2);
        tma_load_3d(sm + kSmG, &P.tm_g, 0, hh, tok0, &S.bar_g, pol_in);
    };
    auto stage_qkv = [&](int tok0, int hh, float beta_t) {
        if (tid == 0) {
            mbar_arrive_expect_tx(&S.bar_qkv, 3 * kChunk * kDim * 2);
            tma_load_3d(sm + kSmQ, &P.tm_q, 0, hh, tok0, &S.bar_qkv, pol_in);
            tma_load_3d(sm + kSmK, &P.tm_k, 0, hh, tok0, &S.bar_qkv, pol_in);
            tma_load_3d(sm + kSmV, &P.tm_v, 0, hh, tok0, &S.bar_qkv, pol_in);
        }
        if (tid < kChunk) S.sBeta[tid] = beta_t;
    };
    auto load_beta = [&](const ChunkInfo& c, int hh) -> float {
        return (tid < c.len) ? __bfloat162float(P.beta[(size_t)(c.tok0 + tid) * H + hh]) : 0.f;
    };

    if (warp == 0) {
        tmem_alloc(&S.tmem_base, kTmemCols);
        if (relinquish) tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&S.bar, 1);
        mbar_init(&S.bar_g, 1);
        mbar_init(&S.bar_qkv, 1);
        mbar_fence_init();
        S.s_abort = 0;
        S.pending = -1;
    }
    int chunk = item / H;
    int h = item - chunk * H;
    ChunkInfo ci = P.info[chunk];
    if (tid == 0) stage_g(ci.tok0, h);
    stage_qkv(ci.tok0, h, tid < kChunk ? load_beta(ci, h) : 0.f);
    float dtb = P.dt_bias[h * kDim + ch];
    float alog = P.A_log[h];
    tc_fence_before();
    sub_sync(bar_id);
    tc_fence_after();
    const uint32_t tbase = S.tmem_base;
    // phases of bar_g / bar_qkv the next waits expect, and the copies issued and
    // not yet waited for
    uint32_t gph = 0, qph = 0;
    bool g_out = true, qkv_out = true;
    int drain_mma = -1;     // after giving up on an MMA wait: the S.bar phase still owed

    for (;;) {
    const int len = ci.len;
    uint8_t* rec = P.records + ((size_t)chunk * H + h) * kRecBytes;
    const int next = item + item_stride;
    const bool has_next = next < n_items;
    const int chunk_n = has_next ? next / H : chunk;
    const int h_n = has_next ? next - chunk_n * H : h;
    // first token of the next item, for its early g copy (thread 0)
    const int tok0_n = (tid == 0 && has_next) ? P.info[chunk_n].tok0 : 0;
    if (mbar_wait(&S.bar_g, gph, lim)) {
        g_out = false;
        gph ^= 1u;
    } else {
        atomicOr(P.status, kStatusTimeout);
        S.s_abort = 1;
    }
    sub_sync(bar_id);
    if (S.s_abort) break;

    // ---------------------------------------------------------------- gate (32 tokens)
    float al[32];
    {
        // In base 2: x2 = (g + dt_bias) log2(e); softplus(x) log2(e) = max(x2, 0) +
        // log2(1 + 2^-|x2|); log2(alpha) = max(-exp(A_log) * that, lower_bound log2(e)).
        constexpr float kLog2e = 1.4426950408889634f;
        const float dtb2 = dtb * kLog2e;
        const float negA = -__expf(alog);
        const float lb2 = P.lower_bound * kLog2e;
        float prod = 1.f;
#pragma unroll
        for (int u = 0; u < 32; ++u) {
            const int t = t0 + u;
            const float x2 = fmaf(lds_bf16(sm, kSmG + t * 256 + ch * 2), kLog2e, dtb2);
            const float sp2 = fmaxf(x2, 0.f) + hw_log2(1.f + hw_exp2(-fabsf(x2)));
            const float a = hw_exp2(fmaxf(negA * sp2, lb2));
            al[u] = (t < len) ? a : 1.f;
            prod *= al[u];
            if (half == 1 && u == 7) S.sQf[0][ch] = prod;   // prod_{32}^{39}
            if (half == 1 && u == 23) S.sQf[1][ch] = prod;  // prod_{32}^{55}
        }
        S.sTot[half][ch] = prod;
    }
    if (mbar_wait(&S.bar_qkv, qph, lim)) {
        qkv_out = false;
        qph ^= 1u;
    } else {
        atomicOr(P.status, kStatusTimeout);
        S.s_abort = 1;
    }
    if (len < kChunk && !qkv_out) {
        // zero the rows of tokens past the chunk's end in the q, k tiles (the v tile's
        // are zeroed when it is moved into the operand layout)
        for (int e = tid; e < 2 * kChunk * 16; e += kThreads) {
            const int tile = e / (kChunk * 16), r = (e / 16) % kChunk, piece = e & 15;
            if (r >= len)
                *reinterpret_cast<uint4*>(sm + tile * 16384 + r * 256 + piece * 16) =
                    make_uint4(0u, 0u, 0u, 0u);
        }
    }
    // the previous item's U^T tensor store has read the (K o E)^T area, which the
    // prefix pass below rewrites
    if (tid == kStoreTid) bulk_wait_read<0>();
    sub_sync(bar_id);           // q, k, v, S.sTot, S.sQf visible
    if (S.s_abort) break;
    uint32_t qp[16], kp[16];
    if (QKN) {
        // 1 / sqrt(|x|^2 + eps) of each q row (r < 64) and k row (r >= 64), two
        // threads per row; zeroed padding rows stay zero
        {
            const int r = tid >> 1, hf = tid & 1;
            const uint4* rowp = reinterpret_cast<const uint4*>(
                sm + (r < kChunk ? kSmQ : kSmK) + (r & (kChunk - 1)) * 256 + hf * 128);
            float ss = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w) {
                const uint4 x = rowp[w];
                const uint32_t e[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    ss = fmaf(bf16_lo(e[j]), bf16_lo(e[j]), ss);
                    ss = fmaf(bf16_hi(e[j]), bf16_hi(e[j]), ss);
                }
            }
            ss += __shfl_xor_sync(0xffffffffu, ss, 1);
            if (hf == 0) S.sRn[r / kChunk][r & (kChunk - 1)] = rsqrtf(ss + kL2NormEps);
        }
        sub_sync(bar_id);
        // the normalised rows, rounded to bf16 like the inputs
#pragma unroll
        for (int u = 0; u < 32; u += 2) {
            const int t = t0 + u;
            qp[u / 2] = pack_bf16(lds_bf16(sm, kSmQ + t * 256 + ch * 2) * S.sRn[0][t],
                                  lds_bf16(sm, kSmQ + (t + 1) * 256 + ch * 2) * S.sRn[0][t + 1]);
            kp[u / 2] = pack_bf16(lds_bf16(sm, kSmK + t * 256 + ch * 2) * S.sRn[1][t],
                                  lds_bf16(sm, kSmK + (t + 1) * 256 + ch * 2) * S.sRn[1][t + 1]);
        }
    } else {
#pragma unroll
        for (int u = 0; u < 32; u += 2) {
            const int t = t0 + u;
            qp[u / 2] = pack_bf16(lds_bf16(sm, kSmQ + t * 256 + ch * 2),
                                  lds_bf16(sm, kSmQ + (t + 1) * 256 + ch * 2));
            kp[u / 2] = pack_bf16(lds_bf16(sm, kSmK + t * 256 + ch * 2),
                                  lds_bf16(sm, kSmK + (t + 1) * 256 + ch * 2));
        }
    }
#define KV(u) ((u) & 1 ? bf16_hi(kp[(u) / 2]) : bf16_lo(kp[(u) / 2]))
#define QV(u) ((u) & 1 ? bf16_hi(qp[(u) / 2]) : bf16_lo(qp[(u) / 2]))
    const float P0 = S.sTot[0][ch], P1 = S.sTot[1][ch];
    {
        // prefix pass: (K o E)^T to smem, scale * (Q o E) to the record (beta
        // enters the WY products through the shared operand diag(beta) T^T)
        float E = half ? P0 : 1.f;
#pragma unroll
        for (int tg = 0; tg < 4; ++tg) {
            float kb[8], qh[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int uu = tg * 8 + u;
                E *= al[uu];
                kb[u] = KV(uu) * E;
                qh[u] = P.scale * QV(uu) * E;
            }
            sts_v4f(smem_addr(sm + kSmKbT + kmaj_off(ch, t0 + tg * 8, 128, 1024)), kb);
            stg_v4f(rec + kRecWQ + mnmaj_off(64 + t0 + tg * 8, ch, 128, 2048), qh, pol_rec);
        }
        if (half == 0) reinterpret_cast<float*>(rec + kRecGam)[ch] = P0 * P1;
        // suffix pass: (K o F)^T to the record
        float F = half ? 1.f : P1;
#pragma unroll
        for (int tg = 3; tg >= 0; --tg) {
            float kt[8];
#pragma unroll
            for (int u = 7; u >= 0; --u) {
                const int uu = tg * 8 + u;
                kt[u] = KV(uu) * F;
                F *= al[uu];
            }
            stg_v4f(rec + kRecKT + kmaj_off(ch, t0 + tg * 8, 128, 1024), kt, pol_rec);
        }
    }
    sub_sync(bar_id);  // staging fully consumed; Left / R may now overwrite it

    // ---------------------------------------------------------------- score operands
    {
        // left factors exp(G_i - G_{m_a}) for this half's two sub-blocks
#pragma unroll
        for (int bl = 0; bl < 2; ++bl) {
            const int a = 2 * half + bl;  // global sub-block
            const int u0 = 16 * bl;       // its first local token
            // (eight tokens at a time: tokens u0 .. u0 + 7 relative to the reference
            // u0 + 7, then u0 + 8 .. u0 + 15)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                float lf[8];
                float run = 1.f;
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    run *= al[u0 + hh * 8 + u];
                    lf[u] = run;
                }
                if (hh == 0) {
                    const float inv = 1.f / lf[7];
#pragma unroll
                    for (int u = 0; u < 7; ++u) lf[u] *= inv;
                    lf[7] = 1.f;
                }
                float kl[8], ql[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    kl[u] = KV(u0 + hh * 8 + u) * lf[u];
                    ql[u] = QV(u0 + hh * 8 + u) * lf[u];
                }
                sts_v4f(smem_addr(sm + kSmLeft + mnmaj_off(16 * a + 8 * hh, ch, 128, 2048)), kl);
                sts_v4f(smem_addr(sm + kSmLeft + mnmaj_off(64 + 16 * a + 8 * hh, ch, 128, 2048)),
                        ql);
            }
        }
        // right operands inside this half: R_{2h} rows [32h, 32h+16), R_{2h+1} rows [32h, 32h+32)
        {
            // R_{2h}: reference local token 7 (groups 0 down, then group 1 up);
            // R_{2h+1}: reference 23 (groups 2, 1, 0 down, then group 3 up)
            const int a0 = 2 * half, a1 = 2 * half + 1;
            auto put = [&](int a, int g, const float (&f)[8]) {
                float r8[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) r8[u] = KV(g * 8 + u) * f[u];
                sts_v4f(smem_addr(sm + kSmR + r_off(a) + mnmaj_off(t0 + g * 8, ch, 128, 2048)), r8);
            };
            float f[8];
            float run = 1.f;
            back8(al, 0, run, f, true);
            put(a0, 0, f);
            fwd8(al, 1, f);
            put(a0, 1, f);
            run = 1.f;
            back8(al, 2, run, f, true);
            put(a1, 2, f);
            back8(al, 1, run, f, false);
            put(a1, 1, f);
            back8(al, 0, run, f, false);
            put(a1, 0, f);
            fwd8(al, 3, f);
            put(a1, 3, f);
        }
        if (half == 0) {
            // R_2 and R_3 rows [0, 32): prod_{j+1}^{31} alpha (local) times the
            // second half's prod_{32}^{m_a} alpha
            const float q2 = S.sQf[0][ch], q3 = S.sQf[1][ch];
            float run = 1.f;
#pragma unroll
            for (int jg = 3; jg >= 0; --jg) {  // prod_{s=u+1}^{31} alpha_s, downwards
                float sfx[8];
#pragma unroll
                for (int u = 7; u >= 0; --u) {
                    sfx[u] = run;
                    run *= al[jg * 8 + u];
                }
                float r2[8], r3[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const float kv = KV(jg * 8 + u) * sfx[u];
                    r2[u] = kv * q2;
                    r3[u] = kv * q3;
                }
                sts_v4f(smem_addr(sm + kSmR + r_off(2) + mnmaj_off(jg * 8, ch, 128, 2048)), r2);
                sts_v4f(smem_addr(sm + kSmR + r_off(3) + mnmaj_off(jg * 8, ch, 128, 2048)), r3);
            }
        }
    }
#undef KV
#undef QV
    fence_async_smem();
    tc_fence_before();
    sub_sync(bar_id);

    // ---------------------------------------------------------------- score MMAs
    if (tid == 0) {
        // R_0..R_3 are contiguous with one 2048-B stride between 8-row groups and
        // their TMEM columns d_col(a) follow the same order, so all four score
        // blocks are one MMA with N = 16 + 32 + 48 + 64 = 160 (8 instructions).
        tc_fence_after();
        const uint64_t dl = smem_desc(smem_addr(sm + kSmLeft), 128, 2048);
        const uint64_t dr = smem_desc(smem_addr(sm + kSmR), 128, 2048);
        const uint32_t idesc = idesc_bf16_f32(128, 160, true, true);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
            mma_bf16(tbase, dl + 16u * kk, dr + 16u * kk, idesc, kk > 0 ? 1u : 0u);
        mma_commit(&S.bar);
    }
    if (!mbar_wait(&S.bar, 0, lim)) {
        atomicOr(P.status, kStatusTimeout);
        S.s_abort = 1;
    }
    tc_fence_after();
    sub_sync(bar_id);
    if (S.s_abort) {
        drain_mma = 0;
        break;
    }
    // the score MMA has read R, which covers the g tile: request the next item's g
    if (has_next) {
        if (tid == 0) stage_g(tok0_n, h_n);
        g_out = true;
    }

    // ---------------------------------------------------------------- score read-out
    // TMEM lane quarter w % 4 holds k rows (quarters 0, 1) or q rows (2, 3) of
    // tokens 32 (w % 2) .. + 31, i.e. sub-blocks a_lo = 2 (w % 2) (lanes 0-15)
    // and a_lo + 1 (lanes 16-31); warps w and w + 4 split that row's columns j.
    {
        const int qd = warp & 3, hj = warp >> 2;
        const bool is_k = qd < 2;
        const int i = 32 * (qd & 1) + lane;  // token of this row
        const int a_lo = 2 * (qd & 1);
        const bool upper = lane >= 16;       // row of sub-block a_lo + 1
        const int jw = (qd & 1) ? 32 : 16;   // columns per warp
        float* sAT = reinterpret_cast<float*>(sm + kSmA);
        const float f = is_k ? S.sBeta[i] : P.scale;
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            if (rr * 16 >= jw) break;
            const int jb = jw * hj + 16 * rr;
            uint32_t r0[16], r1[16];
            tmem_ld16(taddr(tbase, 32u * qd, d_col(a_lo) + (uint32_t)jb), r0);
            tmem_ld16(taddr(tbase, 32u * qd, d_col(a_lo + 1) + (uint32_t)jb), r1);
            tmem_wait_ld();
            reg_fence16(r0);
            reg_fence16(r1);
            float val[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const int j = jb + u;
                const float x = __uint_as_float(upper ? r1[u] : r0[u]);
                val[u] = (is_k ? (j < i) : (j <= i)) ? f * x : 0.f;
            }
            if (is_k) {
                // A^T[j][i] = beta_i A[i][j] (column-major A: the inverse reads columns)
#pragma unroll
                for (int u = 0; u < 16; ++u) sAT[(jb + u) * kStr + i] = val[u];
            } else {
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    float hi[8], lo[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        hi[u] = __bfloat162float(__float2bfloat16_rn(val[8 * hh + u]));
                        lo[u] = val[8 * hh + u] - hi[u];
                    }
                    stg_v4f(rec + kRecAQ + kmaj_off(i, jb + 8 * hh, 128, 1024), hi, pol_rec);
                    stg_v4f(rec + kRecAQL + kmaj_off(i, jb + 8 * hh, 128, 1024), lo, pol_rec);
                }
            }
        }
        float* sT = reinterpret_cast<float*>(sm + kSmT);
        if (!is_k) {
            if (qd == 2) {
                // tokens 0..31 attend to no key in 32..63: zero those record columns
#pragma unroll
                for (int jg = 0; jg < 2; ++jg) {
                    const int j0 = 32 + 16 * hj + 8 * jg;
                    stg_v4(rec + kRecAQ + kmaj_off(i, j0, 128, 1024), 0u, 0u, 0u, 0u, pol_rec);
                    stg_v4(rec + kRecAQL + kmaj_off(i, j0, 128, 1024), 0u, 0u, 0u, 0u, pol_rec);
                }
            }
            // zero the strictly upper 16 x 16 blocks of T (q-row warps, while the
            // k-row warps invert the diagonal blocks)
            const int qt = 64 * hj + 32 * (qd - 2) + lane;  // 0..127
            for (int e = qt; e < 6 * 256; e += 128) {
                const int blk = e >> 8, r = (e >> 4) & 15, c = e & 15;
                const int a = blk < 3 ? 0 : (blk < 5 ? 1 : 2);
                const int b = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
                sT[(16 * a + r) * kStr + 16 * b + c] = 0.f;
            }
            if (ready && tid == kStoreTid && S.pending >= 0) {
                // the previous item's U^T store has completed (a gate phase and more
                // ago): publish its record (every other store of it is ordered before
                // by the barriers since)
                publish_flag(ready, S.pending);
                S.pending = -1;
            }
        } else {
            // A^T is complete once the four k-row warps have stored it; warps 0 and 1
            // then invert the four 16 x 16 diagonal blocks of I + A by forward
            // substitution (lanes 0-15 one block, 16-31 the next; lane = column j),
            // overlapping the q-row warps' record stores
            asm volatile("bar.sync %0, %1;" ::"r"(bar_k), "n"(kThreads / 2) : "memory");
            if (warp < 2) {
                const int o = 16 * (2 * warp + (lane >> 4)), j = lane & 15;
                const float* sA = sAT;  // sA[l][i] = A[i][l]
                float tc[16];
#pragma unroll
                for (int l = 0; l < 16; ++l) tc[l] = (l == j) ? 1.f : 0.f;
#pragma unroll
                for (int ii = 1; ii < 16; ++ii) {
                    float s0 = 0.f, s1 = 0.f;
#pragma unroll
                    for (int l = 0; l < ii; ++l) {
                        if (l & 1)
                            s1 = fmaf(sA[(o + l) * kStr + o + ii], tc[l], s1);
                        else
                            s0 = fmaf(sA[(o + l) * kStr + o + ii], tc[l], s0);
                    }
                    if (ii > j) tc[ii] = -(s0 + s1);
                }
#pragma unroll
                for (int ii = 0; ii < 16; ++ii) sT[(o + ii) * kStr + o + j] = tc[ii];
            }
        }
    }
    tc_fence_before();
    sub_sync(bar_id);

    // the next item's chunk info and per-head parameters, loaded here (the
    // register-heavy phases are over) so they arrive long before the staging
    const ChunkInfo ci_n = P.info[chunk_n];
    const float dtb_n = P.dt_bias[h_n * kDim + ch];
    const float alog_n = P.A_log[h_n];

    // ---------------------------------------------------------------- T = (I + A)^-1
    {
        const float* sAT = reinterpret_cast<const float*>(sm + kSmA);  // sAT[l][i] = A[i][l]
        float* sT = reinterpret_cast<float*>(sm + kSmT);
        float* sX = reinterpret_cast<float*>(sm + kSmX);
        // (diagonal blocks: inverted above, after the score read-out)
        offdiag_inverse(sAT, sT, sX, tid, bar_id);
        // the v tile into the operand layout (its copy landed with q and k)
        {
            uint4 vx[4];
            v_tile_load(sm + kSmV, tid, len, vx);
            sub_sync(bar_id);
            v_tile_store(sm + kSmV, tid, vx);
        }
        // diag(beta) T^T as MN-major B operand: element (n = t, k = s) = beta_s T[t][s],
        // k-groups 128 B, n-groups 1024 B
#pragma unroll
        for (int it = 0; it < 2; ++it) {
            const int e = tid + kThreads * it;   // 512 vectors: (t-group, s)
            const int s = e & 63, tg = e >> 6;
            const float bs = S.sBeta[s];
            float x[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) x[u] = sT[(tg * 8 + u) * kStr + s] * bs;
            sts_v4f(smem_addr(sm + kSmTT + mnmaj_off(tg * 8, s, 128, 1024)), x);
        }
    }
    fence_async_smem();
    tc_fence_before();
    sub_sync(bar_id);

    // ---------------------------------------------------------------- W^T, U^T MMAs
    if (tid == 0) {
        tc_fence_after();
        const uint32_t idesc_w = idesc_bf16_f32(128, 64, false, true);  // A K-major
        const uint32_t idesc_u = idesc_bf16_f32(128, 64, true, true);   // A MN-major (V tile)
        const uint32_t bT = smem_addr(sm + kSmTT);
        const uint32_t aK = smem_addr(sm + kSmKbT);
        const uint32_t aV = smem_addr(sm + kSmV);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            mma_bf16(tbase + 0, smem_desc(aK + kk * 256, 128, 1024),
                     smem_desc(bT + kk * 256, 128, 1024), idesc_w, kk > 0 ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            mma_bf16(tbase + 64, smem_desc(aV + kk * 256, 128, 1024),
                     smem_desc(bT + kk * 256, 128, 1024), idesc_u, kk > 0 ? 1u : 0u);
        mma_commit(&S.bar);
    }
    if (!mbar_wait(&S.bar, 1, lim)) {
        atomicOr(P.status, kStatusTimeout);
        S.s_abort = 1;
    }
    tc_fence_after();
    sub_sync(bar_id);
    if (S.s_abort) {
        drain_mma = 1;
        break;
    }

    // the staging area of q, k, v is free again: start the next item's copies
    float beta_n = 0.f;
    if (has_next && tid < kChunk) beta_n = load_beta(ci_n, h_n);
    if (has_next) {
        stage_qkv(ci_n.tok0, h_n, beta_n);
        qkv_out = true;
    }

    // ---------------------------------------------------------------- W (warps 0-3), U^T (4-7)
    // W goes to the record with coalesced stores; U^T (one 128-byte record row per
    // value channel) is staged in the (K o E)^T area, which the W MMA has finished
    // reading, and written by one TMA store; the next item's prefix pass, the
    // area's next writer, starts after thread 0 has seen the store read it.
    {
        const bool is_w = warp < 4;
        const uint32_t col0 = is_w ? 0u : 64u;
        uint32_t r[4][16];  // all four loads in flight before one wait
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld16(taddr(tbase, 32u * (warp & 3), col0 + 16u * c), r[c]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 4; ++c) reg_fence16(r[c]);
        if (is_w) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    float x[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) x[u] = __uint_as_float(r[c][8 * hh + u]);
                    stg_v4f(rec + kRecWQ + mnmaj_off(16 * c + 8 * hh, ch, 128, 2048), x, pol_rec);
                }
            }
        } else {
            sts_row_swizzled(sm + kSmKbT, ch, r);
            fence_async_smem();
        }
    }
    // the barrier orders every thread's record stores and U^T staging before the
    // tensor store and the flag release
    sub_sync(bar_id);
    if (tid == kStoreTid) {
        tma_store_3d(&P.tm_ut, 0, 0, chunk * H + h, sm + kSmKbT, pol_rec);
        bulk_commit();
        // the flag follows once the store has completed (next item's read-out, or
        // the exit)
        if (ready) S.pending = item;
    }
    if (!has_next) break;
    item = next;
    chunk = chunk_n;
    h = h_n;
    ci = ci_n;
    dtb = dtb_n;
    alog = alog_n;
    tc_fence_before();
    }  // item loop

    if (tid == kStoreTid) {
        // the last U^T store, then the last flag
        bulk_wait<0>();
        if (ready && S.pending >= 0) publish_flag(ready, S.pending);
    }
    if (tid == 0) {
        // an aborted worker waits (bounded) for its own tile copies before leaving
        if (g_out) mbar_drain(&S.bar_g, gph);
        if (qkv_out) mbar_drain(&S.bar_qkv, qph);
    }
    // ... and for an MMA it stopped waiting for, before its TMEM is freed
    if (drain_mma >= 0 && tid == 0) mbar_drain(&S.bar, (uint32_t)drain_mma);
    tc_fence_before();
    sub_sync(bar_id);
    if (warp == 0) tmem_dealloc(tbase, kTmemCols);
}


// cuTensorMapEncodeTiled, fetched from the driver once.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
inline EncodeTiledFn encode_tiled_fn() {
    static EncodeTiledFn fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            f = nullptr;
        return reinterpret_cast<EncodeTiledFn>(f);
    }();
    return fn;
}
// [tokens][H][128] bf16 -> tiles of 64 tokens x 1 head x 128 channels.
inline bool encode_tile_map(CUtensorMap* m, const void* base, int64_t tokens, int H) {
    const EncodeTiledFn enc = encode_tiled_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)kDim, (cuuint64_t)H, (cuuint64_t)tokens};
    const cuuint64_t strides[2] = {(cuuint64_t)kDim * 2, (cuuint64_t)H * kDim * 2};  // bytes
    const cuuint32_t box[3] = {(cuuint32_t)kDim, 1u, (cuuint32_t)kChunk};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The U^T block of every record: {64 tokens, 128 value channels, n_rec records},
// rows 128 B apart, records kRecBytes apart -> boxes of one record's 64 x 128,
// 128-byte swizzled in shared memory.
inline bool encode_ut_map(CUtensorMap* m, uint8_t* records, int64_t n_rec) {
    const EncodeTiledFn enc = encode_tiled_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)kChunk, (cuuint64_t)kDim, (cuuint64_t)n_rec};
    const cuuint64_t strides[2] = {(cuuint64_t)kChunk * 2, (cuuint64_t)kRecBytes};  // bytes
    const cuuint32_t box[3] = {(cuuint32_t)kChunk, (cuuint32_t)kDim, 1u};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, records + kRecUT, dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Arguments of the chunk kernel; false if a tensor map cannot be built.
inline bool make_prep_args(const Problem& p, const Workspace& ws, int* status, PrepArgs& a) {
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
    a.qk_norm = p.qk_norm ? 1 : 0;
    a.hint_records = 0;
    a.flags = ws.flags;
    a.chunk_off = ws.chunk_off;
    a.info = ws.info;
    a.records = ws.records;
    a.status = status;
    return encode_tile_map(&a.tm_q, p.q, p.total_tokens, p.H) &&
           encode_tile_map(&a.tm_k, p.k, p.total_tokens, p.H) &&
           encode_tile_map(&a.tm_v, p.v, p.total_tokens, p.H) &&
           encode_tile_map(&a.tm_g, p.g, p.total_tokens, p.H) &&
           encode_ut_map(&a.tm_ut, ws.records, (int64_t)p.max_chunks * p.H);
}

}  // namespace prep
}  // namespace kda
