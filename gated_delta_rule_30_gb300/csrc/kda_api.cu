// kda_api.cu -- C ABI (include/kda.h): argument validation, workspace
// carve-up, the device-side schedule of 64-token chunks, and the launch
// sequence schedule -> chunk kernel -> recurrence kernel on the caller's
// stream.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdio>
#include <atomic>
#include <cstring>
#include <mutex>

#include "kda.h"
#include "kda_internal.h"
#include "kda_bwd_status.h"

namespace kda {

// ----------------------------------------------------------------------------- errors
namespace {
thread_local char g_msg[512] = {0};
thread_local int g_last_path = 0;  // kda_last_path
}  // namespace

kda_status_t set_error(kda_status_t s, const char* msg) {
    std::snprintf(g_msg, sizeof g_msg, "%s", msg);
    return s;
}
kda_status_t cuda_error(cudaError_t e, const char* where) {
    std::snprintf(g_msg, sizeof g_msg, "%s: %s", where, cudaGetErrorString(e));
    return KDA_ERR_CUDA;
}
void clear_error() { g_msg[0] = 0; }

// ----------------------------------------------------------------------------- status block
// Four ints per device.  Word 0: bit kStatusDeviceInput (malformed cu_seqlens
// seen by the schedule kernel) and bit kStatusTimeout (a bounded wait gave
// up).  Words 2-3: the limit, in ns, of the device-side waits that can give up
// (little-endian 64-bit; 2 s = 0x77359400), read by the kernels through
// wait_limit_ns (tc.cuh).
__device__ __align__(16) int g_kda_status[4] = {0, 0, 2000000000, 0};

int* device_status_ptr() {
    static std::mutex mu;
    static int* ptrs[128] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) {
        set_error(KDA_ERR_CUDA, "cudaGetDevice failed");
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (!ptrs[dev]) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_kda_status);
        if (e != cudaSuccess) {
            cuda_error(e, "cudaGetSymbolAddress(status)");
            return nullptr;
        }
        ptrs[dev] = static_cast<int*>(p);
    }
    return ptrs[dev];
}

// ----------------------------------------------------------------------------- workspace
namespace {
constexpr size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
}  // namespace

namespace {
// segmented path: segment offsets, X and M^T per (segment, head), entering states
size_t segment_area_bytes(int64_t N, int64_t H, int segs) {
    if (segs <= 0) return 0;
    const size_t nseg = (size_t)N * segs;
    return align256((nseg + 1) * sizeof(int32_t)) + nseg * (size_t)H * 3 * kDim * kDim * sizeof(float);
}
}  // namespace

size_t workspace_bytes(int64_t max_chunks, int64_t N, int64_t H, int segs) {
    return 256 + align256((size_t)(N + 1) * sizeof(int32_t)) +
           align256((size_t)max_chunks * sizeof(ChunkInfo)) +
           (size_t)max_chunks * (size_t)H * kRecBytes + align256(ready_bytes(max_chunks, H)) +
           segment_area_bytes(N, H, segs);
}

Workspace carve_workspace(void* base, int64_t max_chunks, int64_t N, int64_t H, int segs) {
    uint8_t* p = static_cast<uint8_t*>(base);
    Workspace w;
    w.flags = reinterpret_cast<int32_t*>(p);
    p += 256;
    w.chunk_off = reinterpret_cast<int32_t*>(p);
    p += align256((size_t)(N + 1) * sizeof(int32_t));
    w.info = reinterpret_cast<ChunkInfo*>(p);
    p += align256((size_t)max_chunks * sizeof(ChunkInfo));
    w.records = p;
    p += (size_t)max_chunks * (size_t)H * kRecBytes;
    w.ready = reinterpret_cast<int32_t*>(p);
    p += align256(ready_bytes(max_chunks, H));
    w.segs = segs > 0 ? segs : 0;
    w.seg_off = nullptr;
    w.seg_maps = nullptr;
    w.seg_start = nullptr;
    if (w.segs > 0) {
        const size_t nseg = (size_t)N * w.segs;
        w.seg_off = reinterpret_cast<int32_t*>(p);
        p += align256((nseg + 1) * sizeof(int32_t));
        w.seg_maps = reinterpret_cast<float*>(p);
        p += nseg * (size_t)H * 2 * kDim * kDim * sizeof(float);
        w.seg_start = reinterpret_cast<float*>(p);
    }
    return w;
}

// ----------------------------------------------------------------------------- schedule
namespace {

constexpr int kSchedThreads = 1024;

// Builds chunk_off[N+1] (chunks per sequence, prefix-summed) and the chunk
// table from cu_seqlens (or from B sequences of length T).  Validates
// cu_seqlens: 0 = cu[0] <= ... <= cu[N] = total_tokens; on a violation it sets
// flags[0] = 0 (every later kernel then does nothing) and the status bit.
__global__ void __launch_bounds__(kSchedThreads) schedule_kernel(
    const int32_t* __restrict__ cu, int N, int T, long long total_tokens, long long max_chunks,
    int32_t* __restrict__ flags, int32_t* __restrict__ chunk_off, ChunkInfo* __restrict__ info,
    int* __restrict__ status) {
    __shared__ int32_t warp_sums[32];
    __shared__ int s_bad;
    __shared__ int32_t s_carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        s_bad = 0;
        s_carry = 0;
    }
    __syncthreads();
    if (cu) {
        if (tid == 0 && (cu[0] != 0 || (long long)cu[N] != total_tokens)) s_bad = 1;
        for (int n = tid; n < N; n += kSchedThreads)
            if (cu[n + 1] < cu[n]) s_bad = 1;
    }
    __syncthreads();
    if (s_bad) {
        if (tid == 0) {
            flags[0] = 0;
            atomicOr(status, kStatusDeviceInput);
        }
        return;
    }
    for (int base = 0; base < N; base += kSchedThreads) {
        const int n = base + tid;
        const int len = (n < N) ? (cu ? cu[n + 1] - cu[n] : T) : 0;
        const int nc = (len + kChunk - 1) / kChunk;
        int x = nc;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_sums[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int w = warp_sums[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += y;
            }
            warp_sums[lane] = w;
        }
        __syncthreads();
        const int excl = x - nc + (warp > 0 ? warp_sums[warp - 1] : 0);
        const int carry = s_carry;
        if (n < N) chunk_off[n] = carry + excl;
        __syncthreads();
        if (tid == 0) s_carry = carry + warp_sums[31];
        __syncthreads();
    }
    const int total = s_carry;
    if (tid == 0) {
        chunk_off[N] = total;
        flags[0] = (total <= max_chunks) ? 1 : 0;
    }
    if (total > max_chunks) return;
    // chunk table, one chunk per thread: chunk c belongs to the last sequence n
    // with chunk_off[n] <= c (empty sequences share their successor's offset)
    for (int c = tid; c < total; c += kSchedThreads) {
        int lo = 0, hi = N - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (chunk_off[mid] <= c) lo = mid;
            else hi = mid - 1;
        }
        const int j = c - chunk_off[lo];  // chunk index within sequence lo
        const int len = cu ? cu[lo + 1] - cu[lo] : T;
        ChunkInfo ci;
        ci.tok0 = (cu ? cu[lo] : lo * T) + j * kChunk;
        ci.len = min(kChunk, len - j * kChunk);
        info[c] = ci;
    }
}

}  // namespace

cudaError_t launch_schedule(const Problem& p, const Workspace& ws, int* status, cudaStream_t st) {
    schedule_kernel<<<1, kSchedThreads, 0, st>>>(p.cu, p.N, p.T, (long long)p.total_tokens,
                                                 (long long)p.max_chunks, ws.flags, ws.chunk_off,
                                                 ws.info, status);
    return cudaGetLastError();
}

// ----------------------------------------------------------------------------- validation
namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

kda_status_t build_problem(Problem& p, const void* q, const void* k, const void* v, const void* g,
                           const void* beta, float scale, void* out, const float* A_log,
                           const float* dt_bias, float lower_bound, const void* h0,
                           kda_dtype_t h0_dtype, void* hT, kda_dtype_t hT_dtype,
                           const int32_t* cu, int32_t num_seqs, int32_t B, int32_t T, int32_t H,
                           int32_t K, int32_t V) {
    if (K != kDim || V != kDim)
        return set_error(KDA_ERR_INVALID_ARGUMENT, "K and V must both be 128");
    if (B < 1 || T < 0 || H < 1) return set_error(KDA_ERR_INVALID_ARGUMENT, "need B >= 1, T >= 0, H >= 1");
    if (cu && B != 1) return set_error(KDA_ERR_INVALID_ARGUMENT, "cu_seqlens requires B == 1");
    if (cu && num_seqs < 0) return set_error(KDA_ERR_INVALID_ARGUMENT, "num_seqs must be >= 0");
    if (h0_dtype != KDA_DTYPE_NONE && h0_dtype != KDA_DTYPE_BF16 && h0_dtype != KDA_DTYPE_FP32)
        return set_error(KDA_ERR_INVALID_ARGUMENT, "initial_state dtype must be NONE, BF16 or FP32");
    if (hT_dtype != KDA_DTYPE_NONE && hT_dtype != KDA_DTYPE_BF16 && hT_dtype != KDA_DTYPE_FP32)
        return set_error(KDA_ERR_INVALID_ARGUMENT, "final_state dtype must be NONE, BF16 or FP32");
    if ((h0 == nullptr) != (h0_dtype == KDA_DTYPE_NONE))
        return set_error(KDA_ERR_INVALID_ARGUMENT, "initial_state pointer and dtype disagree");
    if ((hT == nullptr) != (hT_dtype == KDA_DTYPE_NONE))
        return set_error(KDA_ERR_INVALID_ARGUMENT, "final_state pointer and dtype disagree");
    if (h0 && hT && h0_dtype != hT_dtype)
        return set_error(KDA_ERR_INVALID_ARGUMENT,
                         "initial_state and final_state must have the same dtype");
    if (!std::isfinite(scale)) return set_error(KDA_ERR_INVALID_ARGUMENT, "scale must be finite");
    if (!std::isfinite(lower_bound) || lower_bound > 0.f)
        return set_error(KDA_ERR_INVALID_ARGUMENT, "lower_bound must be finite and <= 0");
    if (lower_bound < -10.f)
        return set_error(KDA_ERR_UNSUPPORTED,
                         "lower_bound below -10 is outside the sub-block decay factorisation range");
    const int64_t total = (int64_t)B * T;
    if (total > (int64_t)INT32_MAX - 64)
        return set_error(KDA_ERR_INVALID_ARGUMENT, "B * T too large");
    const int32_t N = cu ? num_seqs : B;
    if (total > 0) {
        if (!q || !k || !v || !g || !beta || !out)
            return set_error(KDA_ERR_INVALID_ARGUMENT, "q, k, v, g, beta and out must be non-null");
        if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(out))
            return set_error(KDA_ERR_INVALID_ARGUMENT, "q, k, v, g and out must be 16-byte aligned");
        if ((reinterpret_cast<uintptr_t>(beta) & 1u) != 0)
            return set_error(KDA_ERR_INVALID_ARGUMENT, "beta must be 2-byte aligned");
    }
    if (N > 0 && (!A_log || !dt_bias))
        return set_error(KDA_ERR_INVALID_ARGUMENT, "A_log and dt_bias must be non-null");
    if ((h0 && !aligned16(h0)) || (hT && !aligned16(hT)))
        return set_error(KDA_ERR_INVALID_ARGUMENT, "states must be 16-byte aligned");
    if (h0 && hT && h0 != hT) {
        const size_t bytes = (size_t)N * H * kDim * kDim * (h0_dtype == KDA_DTYPE_FP32 ? 4 : 2);
        const uintptr_t a0 = reinterpret_cast<uintptr_t>(h0), b0 = reinterpret_cast<uintptr_t>(hT);
        if (a0 < b0 + bytes && b0 < a0 + bytes)
            return set_error(KDA_ERR_INVALID_ARGUMENT,
                             "initial_state and final_state overlap without being identical");
    }
    if (cu && (reinterpret_cast<uintptr_t>(cu) & 3u))
        return set_error(KDA_ERR_INVALID_ARGUMENT, "cu_seqlens must be 4-byte aligned");
    p.q = q;
    p.k = k;
    p.v = v;
    p.g = g;
    p.beta = beta;
    p.scale = scale;
    p.out = out;
    p.A_log = A_log;
    p.dt_bias = dt_bias;
    p.lower_bound = lower_bound;
    p.h0 = h0;
    p.h0_dtype = h0_dtype;
    p.hT = hT;
    p.hT_dtype = hT_dtype;
    p.cu = cu;
    p.N = N;
    p.B = B;
    p.T = T;
    p.H = H;
    p.total_tokens = total;
    // sum_n ceil(L_n / 64) <= floor((total + 63 N) / 64)
    p.max_chunks = (total + (int64_t)(kChunk - 1) * N) / kChunk;
    p.qk_norm = false;
    return KDA_OK;
}

constexpr int kMaxStageEvents = 6;
cudaEvent_t g_stage_events[kMaxStageEvents] = {nullptr};
int g_stage_count = 0;  // 0: off
std::atomic<int> g_recur_kind{0};  // kda_set_recurrence_kernel (process-wide)

void stage_mark(int i, cudaStream_t st) {
    if (i < g_stage_count) cudaEventRecord(g_stage_events[i], st);
}

// The single-token step takes a problem when the selection is automatic and it
// applies; it reads and writes only the caller's tensors (no workspace).
bool takes_decode(const Problem& p, int kind) { return kind == 0 && decode_applies(p); }

kda_status_t run(const Problem& p, void* workspace, size_t workspace_size, cudaStream_t st) {
    if (p.N == 0) return KDA_OK;
    int* status = device_status_ptr();
    if (!status) return KDA_ERR_CUDA;
    const int sel = g_recur_kind.load();  // one reading of the selection for the whole call
    if (takes_decode(p, sel)) {
        // one token per sequence: a single pass over the states, no chunk records
        stage_mark(0, st);
        cudaError_t e = launch_decode(p, status, st);
        stage_mark(1, st);
        stage_mark(2, st);
        stage_mark(3, st);
        g_last_path = 4;
        return e == cudaSuccess ? KDA_OK : cuda_error(e, "kernel launch");
    }
    const int segs = segment_count(p.N, p.H, p.max_chunks, sel);
    const size_t need = workspace_bytes(p.max_chunks, p.N, p.H, segs);
    void* ws_ptr = workspace;
    bool owned = false;
    if (!ws_ptr) {
        cudaError_t e = cudaMallocAsync(&ws_ptr, need, st);
        if (e != cudaSuccess) return cuda_error(e, "cudaMallocAsync(workspace)");
        owned = true;
    } else {
        if (workspace_size < need)
            return set_error(KDA_ERR_INVALID_ARGUMENT, "workspace smaller than kda_workspace_size()");
        if (reinterpret_cast<uintptr_t>(ws_ptr) & 255u)
            return set_error(KDA_ERR_INVALID_ARGUMENT, "workspace must be 256-byte aligned");
    }
    const Workspace ws = carve_workspace(ws_ptr, p.max_chunks, p.N, p.H, segs);
    stage_mark(0, st);
    cudaError_t e = launch_schedule(p, ws, status, st);
    if (segs > 0) {
        // few long sequences: segments scanned in parallel (kda_segmented.cu)
        if (e == cudaSuccess) e = launch_seg_schedule(p, ws, st);
        stage_mark(1, st);
        if (e == cudaSuccess) e = launch_prep(p, ws, status, st);
        stage_mark(2, st);
        if (e == cudaSuccess) e = launch_seg_maps(p, ws, status, st);
        stage_mark(3, st);
        if (e == cudaSuccess) e = launch_seg_scan(p, ws, status, st);
        stage_mark(4, st);
        if (e == cudaSuccess) e = launch_seg_outputs(p, ws, status, st);
        stage_mark(5, st);
        g_last_path = 5;
        kda_status_t rc = e == cudaSuccess ? KDA_OK : cuda_error(e, "kernel launch");
        if (owned) {
            cudaError_t f = cudaFreeAsync(ws_ptr, st);
            if (f != cudaSuccess && rc == KDA_OK) rc = cuda_error(f, "cudaFreeAsync(workspace)");
        }
        return rc;
    }
    stage_mark(1, st);
    // kind 3 asks for the fused launch; automatic selection takes it for few,
    // long sequences
    bool fused = false;
    if (e == cudaSuccess && (sel == 3 || sel == 0) && fused_eligible(p, sel == 3)) {
        e = launch_fused(p, ws, status, st);
        if (e == cudaErrorCooperativeLaunchTooLarge || e == cudaErrorNotSupported) {
            cudaGetLastError();  // not resident on this device right now: run the two kernels
            e = cudaSuccess;
        } else {
            fused = true;
        }
    }
    if (!fused) {
        const int kind = recur_choose(p, sel == 3 ? 2 : sel);
        if (e == cudaSuccess) e = launch_prep(p, ws, status, st);
        stage_mark(2, st);
        if (e == cudaSuccess) e = launch_recur(p, ws, status, st, kind);
        g_last_path = kind;
    } else {
        stage_mark(2, st);
        g_last_path = 3;
    }
    stage_mark(3, st);
    kda_status_t rc = KDA_OK;
    if (e != cudaSuccess) rc = cuda_error(e, "kernel launch");
    if (owned) {
        cudaError_t f = cudaFreeAsync(ws_ptr, st);
        if (f != cudaSuccess && rc == KDA_OK) rc = cuda_error(f, "cudaFreeAsync(workspace)");
    }
    return rc;
}

}  // namespace
}  // namespace kda

// ============================================================================= C ABI
using namespace kda;

extern "C" kda_status_t kda_fwd(const void* q, const void* k, const void* v, const void* g,
                                const void* beta, float scale, void* out, const float* A_log,
                                const float* dt_bias, float lower_bound, const void* initial_state,
                                kda_dtype_t initial_dtype, void* final_state,
                                kda_dtype_t final_dtype, const int32_t* cu_seqlens,
                                int32_t num_seqs, int32_t B, int32_t T, int32_t H, int32_t K,
                                int32_t V, void* stream) {
    clear_error();
    Problem p;
    kda_status_t rc = build_problem(p, q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound,
                                    initial_state, initial_dtype, final_state, final_dtype,
                                    cu_seqlens, num_seqs, B, T, H, K, V);
    if (rc != KDA_OK) return rc;
    return run(p, nullptr, 0, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" kda_status_t kda_fwd_ws(const void* q, const void* k, const void* v, const void* g,
                                   const void* beta, float scale, void* out, const float* A_log,
                                   const float* dt_bias, float lower_bound,
                                   const void* initial_state, kda_dtype_t initial_dtype,
                                   void* final_state, kda_dtype_t final_dtype,
                                   const int32_t* cu_seqlens, int32_t num_seqs, int32_t B,
                                   int32_t T, int32_t H, int32_t K, int32_t V, void* workspace,
                                   size_t workspace_bytes_, void* stream) {
    clear_error();
    Problem p;
    kda_status_t rc = build_problem(p, q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound,
                                    initial_state, initial_dtype, final_state, final_dtype,
                                    cu_seqlens, num_seqs, B, T, H, K, V);
    if (rc != KDA_OK) return rc;
    if (!workspace && p.N > 0)
        return set_error(KDA_ERR_INVALID_ARGUMENT, "workspace must be non-null");
    return run(p, workspace, workspace_bytes_, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" kda_status_t kda_fwd_ex(const void* q, const void* k, const void* v, const void* g,
                                   const void* beta, float scale, void* out, const float* A_log,
                                   const float* dt_bias, float lower_bound,
                                   const void* initial_state, kda_dtype_t initial_dtype,
                                   void* final_state, kda_dtype_t final_dtype,
                                   const int32_t* cu_seqlens, int32_t num_seqs, int32_t B,
                                   int32_t T, int32_t H, int32_t K, int32_t V, uint32_t flags,
                                   void* workspace, size_t workspace_bytes_, void* stream) {
    clear_error();
    if (flags & ~(uint32_t)KDA_FWD_QK_L2NORM)
        return set_error(KDA_ERR_INVALID_ARGUMENT, "unknown flag bits");
    Problem p;
    kda_status_t rc = build_problem(p, q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound,
                                    initial_state, initial_dtype, final_state, final_dtype,
                                    cu_seqlens, num_seqs, B, T, H, K, V);
    if (rc != KDA_OK) return rc;
    p.qk_norm = (flags & KDA_FWD_QK_L2NORM) != 0;
    return run(p, workspace, workspace ? workspace_bytes_ : 0,
               reinterpret_cast<cudaStream_t>(stream));
}

extern "C" size_t kda_workspace_size(int32_t B, int32_t T, int32_t H, int32_t num_seqs,
                                     int32_t has_cu_seqlens) {
    clear_error();
    if (B < 1 || T < 0 || H < 1 || (has_cu_seqlens && (B != 1 || num_seqs < 0))) {
        set_error(KDA_ERR_INVALID_ARGUMENT, "invalid sizes");
        return 0;
    }
    const int64_t N = has_cu_seqlens ? num_seqs : B;
    const int sel = g_recur_kind.load();
    // the single-token step uses no workspace: report the smallest valid size
    if (sel == 0 && !has_cu_seqlens && T == 1) return 256;
    const int64_t total = (int64_t)B * T;
    const int64_t max_chunks = (total + (int64_t)(kChunk - 1) * N) / kChunk;
    return workspace_bytes(max_chunks, N, H, segment_count(N, H, max_chunks, sel));
}

extern "C" kda_status_t kda_device_status(void* stream) {
    clear_error();
    int* status = device_status_ptr();
    if (!status) return KDA_ERR_CUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_error(e, "cudaStreamSynchronize");
    int host = 0;
    e = cudaMemcpyFromSymbol(&host, g_kda_status, sizeof(int));
    if (e != cudaSuccess) return cuda_error(e, "read status");
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_kda_status, &zero, sizeof(int));
    if (e != cudaSuccess) return cuda_error(e, "clear status");
    if (host & kStatusLayout)
        return set_error(KDA_ERR_CUDA, "a kernel's shared-memory area was not 1024-byte aligned");
    if (host & kStatusScratch)
        return set_error(KDA_ERR_CUDA, "the backward pass found no free low-memory replay slot");
    if (host & kStatusTimeout) return set_error(KDA_ERR_TIMEOUT, "a bounded device wait timed out");
    if (host & kStatusDeviceInput)
        return set_error(KDA_ERR_DEVICE_INPUT, "malformed cu_seqlens detected on the device");
    return KDA_OK;
}

extern "C" const char* kda_status_string(kda_status_t s) {
    switch (s) {
        case KDA_OK: return "KDA_OK";
        case KDA_ERR_INVALID_ARGUMENT: return "KDA_ERR_INVALID_ARGUMENT";
        case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA";
        case KDA_ERR_TIMEOUT: return "KDA_ERR_TIMEOUT";
        case KDA_ERR_DEVICE_INPUT: return "KDA_ERR_DEVICE_INPUT";
        default: return "KDA_ERR_UNKNOWN";
    }
}

extern "C" const char* kda_last_error_message(void) { return kda::g_msg; }

extern "C" int kda_last_path(void) { return kda::g_last_path; }

extern "C" int kda_abi_version(void) { return KDA_ABI_VERSION; }

extern "C" kda_status_t kda_set_recurrence_kernel(int32_t kind) {
    clear_error();
    if (kind < 0 || kind > 4)
        return set_error(KDA_ERR_INVALID_ARGUMENT, "kind must be 0, 1, 2, 3 or 4");
    g_recur_kind.store(kind);
    return KDA_OK;
}

extern "C" kda_status_t kda_set_wait_limit_ns(uint64_t limit_ns) {
    clear_error();
    if (limit_ns == 0 || limit_ns > 2000000000ull)
        return set_error(KDA_ERR_INVALID_ARGUMENT, "limit_ns must be in [1, 2e9]");
    if (!device_status_ptr()) return KDA_ERR_CUDA;
    cudaError_t e = cudaMemcpyToSymbol(g_kda_status, &limit_ns, sizeof(limit_ns), 2 * sizeof(int));
    if (e != cudaSuccess) return cuda_error(e, "set wait limit");
    return KDA_OK;
}

extern "C" kda_status_t kda_set_stage_events(void* const* events, int32_t count) {
    clear_error();
    if (events == nullptr || count == 0) {
        g_stage_count = 0;
        return KDA_OK;
    }
    if (count != 4 && count != kMaxStageEvents)
        return set_error(KDA_ERR_INVALID_ARGUMENT, "count must be 0, 4 or 6");
    for (int i = 0; i < count; ++i)
        if (!events[i]) return set_error(KDA_ERR_INVALID_ARGUMENT, "null event");
    for (int i = 0; i < count; ++i) g_stage_events[i] = static_cast<cudaEvent_t>(events[i]);
    g_stage_count = count;
    return KDA_OK;
}
