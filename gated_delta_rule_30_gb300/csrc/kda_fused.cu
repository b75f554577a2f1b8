// kda_fused.cu -- one cooperative launch that runs the chunk kernel and the
// recurrence at the same time, for problems with few, long sequences.
//
// The recurrence of a (sequence, head) pair is a chain of dependent steps: it
// leaves most of an SM idle, while the chunk kernel is throughput-bound.  Run
// one after the other, their times add; run together they overlap.  Blocks
// [0, R) of the launch (R = number of (sequence, head) pairs) each run the
// transposed recurrence of one pair; the remaining blocks each host two
// chunk-kernel workers of 256 threads (the same work split, registers and
// shared memory as two CTAs of the stand-alone chunk kernel) that walk the
// (chunk, head) items in chunk-major order, so records appear in the order
// the recurrences consume them.  A worker publishes ready[item] = 1 with a
// GPU-scope release after all of the item's record stores; the recurrence's
// producer warp waits (bounded) for the flag, then copies the record.
//
// The launch is cooperative, one block per SM, so every block is resident at
// once and the waits always end; workers never wait on recurrence blocks.
#include "kda_prep.cuh"
#include "kda_recur_t.cuh"


namespace kda {
namespace {

constexpr int kFusedThreads = 2 * prep::kThreads;  // 512: two workers, or one recurrence
constexpr uint32_t kWorkerSmem = 2 * prep::kSmBytes;
constexpr uint32_t kFusedSmem = kWorkerSmem > recur_t::kSmemBytes ? kWorkerSmem
                                                                  : recur_t::kSmemBytes;
static_assert(recur_t::kThreads <= kFusedThreads, "recurrence role needs more threads");
static_assert(prep::kSmBytes % 1024 == 0, "worker areas must stay 1024-byte aligned");

struct FusedArgs {
    prep::PrepArgs p;
    recur_t::RecurTArgs r;
    int* ready;  // [max_chunks * H]
    int n_rec;   // blocks running a recurrence (one per pair)
};

template <bool QKN>
__global__ void __launch_bounds__(kFusedThreads, 1) fused_kernel(const __grid_constant__ FusedArgs A) {
    extern __shared__ __align__(1024) uint8_t sm[];
    __shared__ prep::PrepShared ps[2];
    __shared__ recur_t::RecurTShared rs;
    if ((int)blockIdx.x < A.n_rec) {
        // barrier 1 spans the recurrence's threads; the rest of the block leaves
        if ((int)threadIdx.x >= recur_t::kThreads) return;
        recur_t::recur_t_body(A.r, sm, rs, threadIdx.x, 1u, blockIdx.x, A.ready);
    } else {
        const int workers = 2 * ((int)gridDim.x - A.n_rec);
        const int w0 = 2 * ((int)blockIdx.x - A.n_rec);
        // both workers share the SM's TMEM (256 columns each); neither gives up
        // the allocation permit before the other has allocated.  Each worker's
        // shared-memory area, barriers and role are compile-time constants, so
        // the block holds two copies of the worker's code: one copy with
        // run-time parameters needs more registers and ran 12% slower.
        // (named barriers: 1 and 2 span each worker, 3 and 4 its key-row warps)
        if ((int)threadIdx.x < prep::kThreads)
            prep::prep_body<QKN>(A.p, sm, ps[0], threadIdx.x, 1u, 3u, w0, workers, A.ready,
                                 false);
        else
            prep::prep_body<QKN>(A.p, sm + prep::kSmBytes, ps[1], threadIdx.x - prep::kThreads,
                                 2u, 4u, w0 + 1, workers, A.ready, false);
    }
}

}  // namespace

bool fused_eligible(const Problem& p, bool forced) {
    int dev = 0, sms = 0, coop = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
    if (!coop || p.N == 0 || p.H == 0 || p.max_chunks == 0) return false;
    const long long pairs = (long long)p.N * p.H;
    // the recurrences may take at most a quarter of the SMs (forced: all but one)
    if (forced ? pairs >= sms : 4 * pairs > sms) return false;
    // with few chunks per sequence there is little to overlap
    if (!forced && p.max_chunks < 8 * p.N) return false;
    const auto kern = p.qk_norm ? fused_kernel<true> : fused_kernel<false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kFusedSmem) !=
        cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kFusedThreads, kFusedSmem) !=
        cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return per_sm >= 1;
}

cudaError_t launch_fused(const Problem& p, const Workspace& ws, int* status, cudaStream_t st) {
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaError_t e = cudaMemsetAsync(ws.ready, 0, ready_bytes(p.max_chunks, p.H), st);
    if (e != cudaSuccess) return e;
    FusedArgs a;
    if (!prep::make_prep_args(p, ws, status, a.p)) return cudaErrorInvalidValue;
    a.p.hint_records = 1;  // the recurrence reads each record back within a few chunks
    a.r = recur_t::make_recur_t_args(p, ws, status);
    a.ready = ws.ready;
    a.n_rec = p.N * p.H;
    void* args[] = {&a};
    const auto kern = p.qk_norm ? fused_kernel<true> : fused_kernel<false>;
    return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(kern), dim3(sms),
                                       dim3(kFusedThreads), args, kFusedSmem, st);
}

}  // namespace kda
