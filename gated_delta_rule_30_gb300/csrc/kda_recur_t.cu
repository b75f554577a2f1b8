// kda_recur_t.cu -- stand-alone transposed recurrence kernel (the body and its
// design notes are in kda_recur_t.cuh): one CTA per (sequence, head).
#include "kda_recur_t.cuh"

namespace kda {
namespace {

using namespace recur_t;

__global__ void __launch_bounds__(kThreads, 1) recur_t_kernel(const RecurTArgs P) {
    extern __shared__ __align__(1024) uint8_t sm[];
    __shared__ RecurTShared S;
    // barrier 0 over the whole CTA is __syncthreads
    recur_t_body(P, sm, S, threadIdx.x, 0u, blockIdx.x, nullptr);
}

}  // namespace

cudaError_t launch_recur_transposed(const Problem& p, const Workspace& ws, int* status,
                                   cudaStream_t st) {
    if (p.N == 0 || p.H == 0) return cudaSuccess;
    const RecurTArgs a = make_recur_t_args(p, ws, status);
    cudaError_t e = cudaFuncSetAttribute(recur_t_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    const long long blocks = (long long)p.N * p.H;
    recur_t_kernel<<<(unsigned)blocks, kThreads, kSmemBytes, st>>>(a);
    return cudaGetLastError();
}

}  // namespace kda
