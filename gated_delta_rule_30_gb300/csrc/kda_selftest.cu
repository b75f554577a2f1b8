// kda_selftest.cu -- checks the tcgen05 operand layouts the KDA kernels rely
// on: one M=128 x N x K bf16 MMA with fp32 accumulation in TMEM for each
// combination of K-major / MN-major A and B (no swizzle, k-groups 128 bytes
// apart), read back with tcgen05.ld by four warps.
#include <cuda_runtime.h>

#include "kda.h"
#include "kda_internal.h"
#include "tc.cuh"

namespace kda {

namespace {

constexpr int kSelftestSmem = 2 * 32768 + 2 * 65536;

__global__ void __launch_bounds__(128, 1)
    selftest_kernel(const __nv_bfloat16* __restrict__ a, const __nv_bfloat16* __restrict__ b,
                    float* __restrict__ d, int N, int K, int ncols, int* __restrict__ status) {
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ uint64_t bar;
    __shared__ uint32_t tmem_base;
    uint8_t* sAk = smem;
    uint8_t* sAm = smem + 32768;
    uint8_t* sBk = smem + 65536;
    uint8_t* sBm = smem + 131072;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t kbytes = (uint32_t)K * 16u;  // stride of 8 rows (or 8 mn) when k-groups are inner
    for (int idx = tid; idx < 128 * K; idx += 128) {
        const int m = idx / K, k = idx % K;
        const __nv_bfloat16 val = a[idx];
        *reinterpret_cast<__nv_bfloat16*>(sAk + kmaj_off(m, k, 128, kbytes)) = val;
        *reinterpret_cast<__nv_bfloat16*>(sAm + mnmaj_off(m, k, 128, kbytes)) = val;
    }
    for (int idx = tid; idx < K * N; idx += 128) {
        const int k = idx / N, n = idx % N;
        const __nv_bfloat16 val = b[idx];
        *reinterpret_cast<__nv_bfloat16*>(sBk + kmaj_off(n, k, 128, kbytes)) = val;
        *reinterpret_cast<__nv_bfloat16*>(sBm + mnmaj_off(n, k, 128, kbytes)) = val;
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base, (uint32_t)ncols);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&bar, 1);
        mbar_fence_init();
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tmem_base;
    bool ok = true;
    for (int combo = 0; combo < 4; ++combo) {
        const bool a_mn = (combo == 1 || combo == 3);
        const bool b_mn = (combo == 1 || combo == 2);
        if (tid == 0) {
            const uint32_t idesc = idesc_bf16_f32(128, (uint32_t)N, a_mn, b_mn);
            const uint32_t abase = smem_addr(a_mn ? sAm : sAk);
            const uint32_t bbase = smem_addr(b_mn ? sBm : sBk);
            for (int kk = 0; kk < K / 16; ++kk) {
                // both layouts keep k-groups 128 B apart and 8-row groups K*16 B apart
                mma_bf16(tbase, smem_desc(abase + kk * 256, 128, kbytes),
                         smem_desc(bbase + kk * 256, 128, kbytes), idesc, kk > 0 ? 1u : 0u);
            }
            mma_commit(&bar);
        }
        if (!mbar_drain(&bar, (uint32_t)(combo & 1))) {
            ok = false;
            atomicOr(status, 1);
        }
        tc_fence_after();
        if (ok) {
            for (int c0 = 0; c0 < N; c0 += 16) {
                uint32_t r[16];
                tmem_load16(taddr(tbase, (uint32_t)(warp * 32), (uint32_t)c0), r);
                float* row = d + ((size_t)combo * 128 + warp * 32 + lane) * N + c0;
#pragma unroll
                for (int i = 0; i < 16; ++i) row[i] = __uint_as_float(r[i]);
            }
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (!ok) break;
    }
    if (warp == 0) tmem_dealloc(tbase, (uint32_t)ncols);
}

}  // namespace

kda_status_t selftest_tcgen05(const void* a, const void* b, float* d, int N, int K,
                              cudaStream_t stream) {
    if (!a || !b || !d) return set_error(KDA_ERR_INVALID_ARGUMENT, "selftest: null pointer");
    if (N < 16 || N > 256 || N % 16 || K < 16 || K > 128 || K % 16)
        return set_error(KDA_ERR_INVALID_ARGUMENT, "selftest: N must be 16..256 (step 16), K 16..128 (step 16)");
    int ncols = 32;
    while (ncols < N) ncols *= 2;
    int* status = device_status_ptr();
    if (!status) return KDA_ERR_CUDA;
    cudaError_t e = cudaFuncSetAttribute(selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSelftestSmem);
    if (e != cudaSuccess) return cuda_error(e, "selftest: cudaFuncSetAttribute");
    selftest_kernel<<<1, 128, kSelftestSmem, stream>>>(
        reinterpret_cast<const __nv_bfloat16*>(a), reinterpret_cast<const __nv_bfloat16*>(b), d, N,
        K, ncols, status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_error(e, "selftest: launch");
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_error(e, "selftest: synchronize");
    return KDA_OK;
}

}  // namespace kda

extern "C" kda_status_t kda_selftest_tcgen05(const void* a, const void* b, float* d, int32_t N,
                                             int32_t K, void* stream) {
    kda::clear_error();
    return kda::selftest_tcgen05(a, b, d, N, K, reinterpret_cast<cudaStream_t>(stream));
}
