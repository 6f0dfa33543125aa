// combine.cu -- the "combine" of the DisagMoE summary (section 2.2): the
// gate-weighted expert outputs, already scaled and scattered to
// slot[rank][token] by GEMM1, are summed back into token order.
//
// out[t,:] = bf16( ((slot[0,t,:] + slot[1,t,:]) + ...) + slot[n-1,t,:] )
// An fp32 left fold in fixed slot (= expert rank) order, no atomics, so the
// result does not depend on scheduling. HBM-bound: each thread streams 8
// consecutive columns (two 16-byte loads per slot, one 16-byte store), and
// the slot reads are marked evict-first because nothing reads them again.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kCombineThreads = 256;

__global__ void __launch_bounds__(kCombineThreads)
combine_kernel(const float* __restrict__ slot, int n_slots, uint16_t* __restrict__ out, int64_t TH)
{
    pdl_wait();
    pdl_launch_dependents();
    const int64_t n_vec = TH / 8;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < n_vec; v += stride) {
        const float4* s0 = reinterpret_cast<const float4*>(slot) + 2 * v;
        float4 a = __ldcs(s0);
        float4 b = __ldcs(s0 + 1);
        for (int j = 1; j < n_slots; ++j) {
            const float4* sj = reinterpret_cast<const float4*>(slot + (int64_t)j * TH) + 2 * v;
            const float4 c = __ldcs(sj);
            const float4 d = __ldcs(sj + 1);
            a.x = a.x + c.x; a.y = a.y + c.y; a.z = a.z + c.z; a.w = a.w + c.w;
            b.x = b.x + d.x; b.y = b.y + d.y; b.z = b.z + d.z; b.w = b.w + d.w;
        }
        __nv_bfloat162 p0 = __floats2bfloat162_rn(a.x, a.y);
        __nv_bfloat162 p1 = __floats2bfloat162_rn(a.z, a.w);
        __nv_bfloat162 p2 = __floats2bfloat162_rn(b.x, b.y);
        __nv_bfloat162 p3 = __floats2bfloat162_rn(b.z, b.w);
        uint4 o;
        o.x = *reinterpret_cast<uint32_t*>(&p0);
        o.y = *reinterpret_cast<uint32_t*>(&p1);
        o.z = *reinterpret_cast<uint32_t*>(&p2);
        o.w = *reinterpret_cast<uint32_t*>(&p3);
        reinterpret_cast<uint4*>(out)[v] = o;
    }
}

}  // namespace

cudaError_t launch_combine(const float* slot, int32_t n_slots, uint16_t* out, int64_t T, int32_t H,
                           int num_sms, cudaStream_t s)
{
    const int64_t TH = T * (int64_t)H;
    if (TH == 0) return cudaSuccess;
    const int64_t n_vec = TH / 8;
    int64_t blocks = (n_vec + kCombineThreads - 1) / kCombineThreads;
    const int64_t cap = (int64_t)num_sms * 8;   // 8 resident blocks of 256 per SM
    if (blocks > cap) blocks = cap;
    return launch_pdl(combine_kernel, dim3((unsigned)blocks), dim3(kCombineThreads), 0, s, slot, n_slots, out, TH);
}

}  // namespace moe
