// kda_segmented.cu -- chunk-parallel state passing for few, long sequences.
//
// The chunked recurrence is sequential over a sequence's chunks, so with few
// (sequence, head) pairs most SMs would idle.  Over any run of chunks the
// state update is affine in the state entering it, the same map for every
// value column (reading of "Flashkda Delta Attention", "Core Kernel API": the
// recurrent state update; per chunk s <- (Diag(gamma) - Ktilde^T W) s +
// Ktilde^T u for each value column s):
//   S_end = M S_start + X,
// with X the state reached from zero and M the image of the identity when U
// is taken as zero.  The path, per call:
//   1. seg_schedule_kernel: split each sequence's chunks into `segs`
//      contiguous segments (possibly empty) -> segment chunk offsets;
//   2. the chunk kernel, as on every path (records per (chunk, head));
//   3. map pass (kda_recur.cu, map mode): X and M of every (segment, head), all
//      segments at once;
//   4. seg_scan_kernel: per (sequence, head, 8 value columns), in fp32,
//      S_0 = initial state, S_{j+1} = M_j S_j + X_j; writes every segment's
//      entering state and the final state;
//   5. the value-sliced recurrence over the segments as independent
//      pseudo-sequences, each starting from its entering state: the outputs.
// Work is about three recurrences instead of one, spread over `segs` times as
// many CTAs.
#include <cuda_runtime.h>

#include "kda_internal.h"
#include "tc.cuh"

namespace kda {
namespace {

constexpr int kMaxSegments = 32;
constexpr int kMinSegments = 4;        // automatic selection: at least this many ...
constexpr int kMinSegmentChunks = 16;  // ... segments of at least this many chunks

constexpr int kScanCols = 8;  // value columns per scan CTA
constexpr int kScanSlices = kDim / kScanCols;
constexpr int kScanThreads = 256;  // thread = (key row r, 4 of the CTA's 8 columns)
constexpr uint32_t kMapBytes = kDim * kDim * sizeof(float);
constexpr uint32_t kScanSmem = 2 * kMapBytes + kDim * kScanCols * sizeof(float);

int num_sms() {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms;
}

__global__ void seg_schedule_kernel(const int32_t* __restrict__ chunk_off, int N, int P,
                                    int32_t* __restrict__ seg_off) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long total = (long long)N * P;
    if (i < total) {
        const int n = (int)(i / P), j = (int)(i % P);
        const int off = chunk_off[n];
        const int c = chunk_off[n + 1] - off;
        seg_off[i] = off + (int)(((long long)j * c) / P);
    } else if (i == total) {
        seg_off[total] = chunk_off[N];
    }
}

struct ScanArgs {
    const float* maps;
    float* start;
    const void* h0;
    void* hT;
    int h0_dtype;
    int hT_dtype;
    int H;
    int P;
    const int32_t* flags;
    int* status;
};

__global__ void __launch_bounds__(kScanThreads, 1) seg_scan_kernel(const ScanArgs A) {
    extern __shared__ __align__(128) uint8_t sm[];
    float* Mt = reinterpret_cast<float*>(sm);                 // [2][128][128]: M^T, double-buffered
    float* S = reinterpret_cast<float*>(sm + 2 * kMapBytes);  // [128][8]: the state slice
    __shared__ uint64_t bar[2];
    __shared__ int s_abort;
    if (A.flags[0] != 1) return;
    if (threadIdx.x == 0) s_abort = (*((volatile int*)A.status) & kStatusTimeout) ? 1 : 0;
    __syncthreads();
    if (s_abort) return;
    const uint64_t lim = wait_limit_ns(A.status);  // of the copy waits that may give up

    const int H = A.H, P = A.P;
    const int slice = blockIdx.x % kScanSlices;
    const int nh = blockIdx.x / kScanSlices;
    const int h = nh % H, n = nh / H;
    const int t = threadIdx.x, r = t & (kDim - 1), cq = (t >> 7) * 4;
    const int c = slice * kScanCols + cq;  // first of this thread's 4 value columns
    constexpr size_t KK = (size_t)kDim * kDim;
    const size_t sidx = ((size_t)n * H + h) * KK + (size_t)r * kDim + c;  // into h0 / hT
    auto maps_of = [&](int j) { return A.maps + (((size_t)n * P + j) * H + h) * 2 * KK; };

    if (t == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        mbar_fence_init();
        mbar_arrive_expect_tx(&bar[0], kMapBytes);
        bulk_g2s(Mt, maps_of(0) + KK, kMapBytes, &bar[0]);
    }
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);  // state entering the first segment
    if (A.h0_dtype == KDA_DTYPE_FP32) {
        s = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(A.h0) + sidx);
    } else if (A.h0_dtype == KDA_DTYPE_BF16) {
        const uint2 w =
            *reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(A.h0) + sidx);
        s = make_float4(bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y));
    }
    *reinterpret_cast<float4*>(S + r * kScanCols + cq) = s;
    __syncthreads();  // barriers initialised, S written

    float4 x_next = *reinterpret_cast<const float4*>(maps_of(0) + (size_t)r * kDim + c);  // X_0
    int j = 0;
    for (; j < P; ++j) {
        const int b = j & 1;
        // the other buffer was last read in step j - 1, which every thread has left
        if (t == 0 && j + 1 < P) {
            mbar_arrive_expect_tx(&bar[b ^ 1], kMapBytes);
            bulk_g2s(Mt + (b ^ 1) * KK, maps_of(j + 1) + KK, kMapBytes, &bar[b ^ 1]);
        }
        float4 acc = x_next;  // X_j; X_{j+1} is fetched while this step computes
        if (j + 1 < P)
            x_next = *reinterpret_cast<const float4*>(maps_of(j + 1) + (size_t)r * kDim + c);
        *reinterpret_cast<float4*>(A.start + (((size_t)n * P + j) * H + h) * KK +
                                   (size_t)r * kDim + c) = s;
        if (!mbar_wait(&bar[b], (uint32_t)((j >> 1) & 1), lim)) {
            atomicOr(A.status, kStatusTimeout);
            s_abort = 1;
        }
        const float* M = Mt + b * KK;
#pragma unroll 8
        for (int k = 0; k < kDim; ++k) {
            const float m = M[k * kDim + r];  // M[r][k]
            const float4 x = *reinterpret_cast<const float4*>(S + k * kScanCols + cq);
            acc.x = fmaf(m, x.x, acc.x);
            acc.y = fmaf(m, x.y, acc.y);
            acc.z = fmaf(m, x.z, acc.z);
            acc.w = fmaf(m, x.w, acc.w);
        }
        __syncthreads();  // every thread has read S and Mt[b]
        if (s_abort) break;
        *reinterpret_cast<float4*>(S + r * kScanCols + cq) = acc;
        s = acc;
        __syncthreads();  // S_{j+1} visible
    }
    if (j < P) {
        // gave up: wait once more, with the longer drain limit, for the copy
        // step j timed out on and for the one issued in step j before leaving
        if (t == 0) {
            mbar_drain(&bar[j & 1], (uint32_t)((j >> 1) & 1));
            if (j + 1 < P) mbar_drain(&bar[(j + 1) & 1], (uint32_t)(((j + 1) >> 1) & 1));
        }
        return;
    }
    if (A.hT_dtype == KDA_DTYPE_FP32) {
        *reinterpret_cast<float4*>(reinterpret_cast<float*>(A.hT) + sidx) = s;
    } else if (A.hT_dtype == KDA_DTYPE_BF16) {
        *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(A.hT) + sidx) =
            make_uint2(pack_bf16(s.x, s.y), pack_bf16(s.z, s.w));
    }
}

// The segments as a problem of their own: N * segs pseudo-sequences whose
// chunk offsets are the segment offsets.
void segment_view(const Problem& p, const Workspace& ws, Problem& pv, Workspace& wv) {
    pv = p;
    pv.N = p.N * ws.segs;
    wv = ws;
    wv.chunk_off = ws.seg_off;
}

}  // namespace

int segment_count(int64_t N, int64_t H, int64_t max_chunks, int kind) {
    if ((kind != 0 && kind != 4) || N <= 0 || H <= 0 || max_chunks <= 0) return 0;
    if (N * H * kMaxSegments > (int64_t)INT32_MAX / 2) return 0;
    const int64_t sms = num_sms();
    const int64_t fill = sms / (2 * N * H);  // map and output passes: two CTAs per (segment, head)
    const int64_t per_seq = max_chunks / N;  // chunks per sequence (the mean, for packed input)
    int64_t P = fill < kMaxSegments ? fill : kMaxSegments;
    if (kind == 0) {
        const int64_t by_len = per_seq / kMinSegmentChunks;
        if (by_len < P) P = by_len;
        return P >= kMinSegments ? (int)P : 0;
    }
    // forced: with more (sequence, head) pairs than half the SMs the segments
    // would not run side by side and their states (192 KB per segment and
    // head) would only cost memory, so the unsplit path runs instead
    if (fill == 0) return 0;
    const int64_t by_len = per_seq / 2;
    if (by_len < P) P = by_len;
    return P >= 2 ? (int)P : 2;
}

cudaError_t launch_seg_schedule(const Problem& p, const Workspace& ws, cudaStream_t st) {
    const long long n = (long long)p.N * ws.segs + 1;
    const int threads = 256;
    seg_schedule_kernel<<<(unsigned)((n + threads - 1) / threads), threads, 0, st>>>(
        ws.chunk_off, p.N, ws.segs, ws.seg_off);
    return cudaGetLastError();
}

cudaError_t launch_seg_maps(const Problem& p, const Workspace& ws, int* status, cudaStream_t st) {
    Problem pv;
    Workspace wv;
    segment_view(p, ws, pv, wv);
    return launch_recur_maps(pv, wv, status, st);
}

cudaError_t launch_seg_scan(const Problem& p, const Workspace& ws, int* status, cudaStream_t st) {
    if (p.N == 0 || p.H == 0) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(seg_scan_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kScanSmem);
    if (e != cudaSuccess) return e;
    ScanArgs a;
    a.maps = ws.seg_maps;
    a.start = ws.seg_start;
    a.h0 = p.h0;
    a.hT = p.hT;
    a.h0_dtype = p.h0_dtype;
    a.hT_dtype = p.hT_dtype;
    a.H = p.H;
    a.P = ws.segs;
    a.flags = ws.flags;
    a.status = status;
    const long long blocks = (long long)p.N * p.H * kScanSlices;
    seg_scan_kernel<<<(unsigned)blocks, kScanThreads, kScanSmem, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_seg_outputs(const Problem& p, const Workspace& ws, int* status,
                               cudaStream_t st) {
    Problem pv;
    Workspace wv;
    segment_view(p, ws, pv, wv);
    pv.h0 = ws.seg_start;
    pv.h0_dtype = KDA_DTYPE_FP32;
    pv.hT = nullptr;  // the scan wrote the final state
    pv.hT_dtype = KDA_DTYPE_NONE;
    // the narrowest value slices that still run in one wave
    const long long pairs = (long long)pv.N * pv.H;
    const long long sms = num_sms();
    const int vs = pairs * 4 <= sms ? 32 : (pairs * 2 <= sms ? 64 : 128);
    return launch_recur_sliced(pv, wv, status, st, vs);
}

}  // namespace kda
