// kda_prep.cu -- stand-alone chunk kernel of the KDA forward pass (the worker
// body and its design notes are in kda_prep.cuh).
#include "kda_prep.cuh"

namespace kda {
namespace {

using namespace prep;

template <bool QKN>
__global__ void __launch_bounds__(kThreads, 2) prep_kernel(const __grid_constant__ PrepArgs P) {
    extern __shared__ __align__(1024) uint8_t sm[];
    __shared__ PrepShared S;
    // barrier 0 over the whole 256-thread CTA is __syncthreads; barrier 1 spans
    // the warps that read the key rows of the scores
    prep_body<QKN>(P, sm, S, threadIdx.x, 0u, 1u, blockIdx.x, gridDim.x, nullptr, true);
}

}  // namespace

cudaError_t launch_prep(const Problem& p, const Workspace& ws, int* status, cudaStream_t st) {
    if (p.max_chunks == 0 || p.H == 0) return cudaSuccess;
    const auto kern = p.qk_norm ? prep_kernel<true> : prep_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmBytes);
    if (e != cudaSuccess) return e;
    PrepArgs a;
    if (!make_prep_args(p, ws, status, a)) return cudaErrorInvalidValue;
    // persistent: two CTAs per SM, each looping over (chunk, head) items
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long items = (long long)p.max_chunks * p.H;
    const long long blocks = items < 2LL * sms ? items : 2LL * sms;
    kern<<<(unsigned)blocks, kThreads, kSmBytes, st>>>(a);
    return cudaGetLastError();
}

}  // namespace kda
