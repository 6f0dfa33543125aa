// selftest.cu -- a self-test of the failure path of the library's bounded waits.
//
// Every pipeline wait in the kernels (mbarrier phases, the fused GEMMs'
// readiness counters) gives up after a %globaltimer limit, records
// MOE_DEV_ERR_TIMEOUT in a device error word and lets the kernel finish, so a
// fault elsewhere never hangs the GPU. moe_selftest_wait_timeout runs that
// path on purpose: one thread waits on a flag that nothing sets.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/moe.h"
#include "kernels.cuh"
#include "ptx.cuh"

static __device__ int32_t g_never_set;       // stays 0: nothing sets it
static __device__ uint32_t g_selftest_err;   // the self-test's device error word

static __global__ void selftest_wait_kernel(unsigned long long limit_ns)
{
    __shared__ int abort_flag;
    abort_flag = 0;
    moe::wait_count(&g_never_set, 1, &abort_flag, &g_selftest_err, limit_ns);
}

extern "C" moe_status moe_selftest_wait_timeout(int32_t limit_ms, moe_stream_t stream)
{
    if (limit_ms < 1 || limit_ms > 4000) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    const uint32_t zero = 0;
    uint32_t word = 0;
    if (cudaMemcpyToSymbolAsync(g_selftest_err, &zero, sizeof zero, 0, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    selftest_wait_kernel<<<1, 1, 0, s>>>((unsigned long long)limit_ms * 1000000ull);
    moe::count_launch();
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemcpyFromSymbolAsync(&word, g_selftest_err, sizeof word, 0, cudaMemcpyDeviceToHost, s) !=
            cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return MOE_ERR_CUDA;
    return (word & moe::MOE_DEV_ERR_TIMEOUT) ? MOE_ERR_TIMEOUT : MOE_OK;
}
