// route.cu -- router: gate logits, top-k and gate weights per token.
//
// The pages name top-k routing (DisagMoE summary, section 2.2) but give no
// formula. This kernel computes the readings stated in include/moe.h:
// fp32 logits in the canonical order, top-k on the logits (ties to the lower
// expert id), softmax over the k selected.
//
// Canonical order on the GPU. A warp owns a group of NT tokens; its lane L
// is the canonical lane L: it owns the 8-element chunks c = L, L+32, ... of
// the hidden dimension, accumulates fmaf(x[h], Wg[h,e], acc) over them in
// increasing h for every expert e of the current expert block, and the 32
// lane sums are combined with an xor butterfly (strides 16, 8, 4, 2, 1).
// That is bit for bit the order the oracle restates.
//
// Memory. x is streamed once from HBM with 16-byte loads (a warp reads 512
// contiguous bytes per token per step). Wg is staged in shared memory in a
// lane-major layout, [step m][element i][expert octet q][lane L] of uint4
// (8 bf16 experts), so that the 32 lanes of a warp read 512 contiguous bytes
// (no bank conflicts). For large H*E the gate is staged in slices of H.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kRouteWarps = 16;
constexpr int kRouteThreads = kRouteWarps * 32;
constexpr int kSliceBytes = 64 * 1024;   // shared-memory budget for one gate slice

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Stage gate rows of m-steps [m0, m0 + ms_count) and experts [e0, e0 + EB)
// into the lane-major layout. Rows >= H and experts >= E are zero.
template <int EB>
__device__ void stage_gate(uint4* wg_s, const uint16_t* __restrict__ Wg, int H, int E, int m0,
                           int ms_count, int e0)
{
    constexpr int Q = EB / 8;
    const int total = ms_count * 8 * Q * 32;
    const bool vec = (E % 8 == 0);
    for (int idx = threadIdx.x; idx < total; idx += blockDim.x) {
        int L = idx & 31;
        int rest = idx >> 5;
        int q = rest % Q;
        rest /= Q;
        int i = rest & 7;
        int ms = rest >> 3;
        int h = (m0 + ms) * 256 + 8 * L + i;
        int e = e0 + 8 * q;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (h < H) {
            const uint16_t* src = Wg + (int64_t)h * E + e;
            if (vec && e + 8 <= E) {
                v = __ldg(reinterpret_cast<const uint4*>(src));
            } else {
                uint16_t t[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) t[u] = (e + u < E) ? src[u] : (uint16_t)0;
                v.x = t[0] | ((uint32_t)t[1] << 16);
                v.y = t[2] | ((uint32_t)t[3] << 16);
                v.z = t[4] | ((uint32_t)t[5] << 16);
                v.w = t[6] | ((uint32_t)t[7] << 16);
            }
        }
        wg_s[idx] = v;
    }
}

template <int EB, int NT>
__global__ void __launch_bounds__(kRouteThreads, 1) route_kernel(RouteArgs a, int ms_per_slice)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    constexpr int Q = EB / 8;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int H = a.H, E = a.E, k = a.k;
    const int n_chunks = H / 8;
    const int n_steps = (n_chunks + 31) / 32;
    const int n_slices = (n_steps + ms_per_slice - 1) / ms_per_slice;
    const int n_eblocks = (E + EB - 1) / EB;
    const bool stage_once = (n_slices == 1 && n_eblocks == 1);

    uint4* wg_s = reinterpret_cast<uint4*>(smem_raw);
    float* logit_s = reinterpret_cast<float*>(smem_raw + (size_t)ms_per_slice * 8 * Q * 32 * 16);
    float* my_logits = logit_s + (size_t)warp * NT * E;

    if (stage_once) {
        stage_gate<EB>(wg_s, a.Wg, H, E, 0, n_steps, 0);
        __syncthreads();
    }

    const int64_t tokens_per_iter = (int64_t)kRouteWarps * NT;
    for (int64_t tg = blockIdx.x; tg * tokens_per_iter < a.T; tg += gridDim.x) {
        const int64_t t0 = tg * tokens_per_iter + (int64_t)warp * NT;
        for (int eb = 0; eb < n_eblocks; ++eb) {
            float acc[NT][EB];
#pragma unroll
            for (int tt = 0; tt < NT; ++tt)
#pragma unroll
                for (int e = 0; e < EB; ++e) acc[tt][e] = 0.0f;

            for (int sl = 0; sl < n_slices; ++sl) {
                const int m0 = sl * ms_per_slice;
                const int ms_count = min(ms_per_slice, n_steps - m0);
                if (!stage_once) {
                    __syncthreads();
                    stage_gate<EB>(wg_s, a.Wg, H, E, m0, ms_count, eb * EB);
                    __syncthreads();
                }
                for (int ms = 0; ms < ms_count; ++ms) {
                    const int c = (m0 + ms) * 32 + lane;
                    uint4 xv[NT];
#pragma unroll
                    for (int tt = 0; tt < NT; ++tt) {
                        const int64_t t = t0 + tt;
                        xv[tt] = make_uint4(0, 0, 0, 0);
                        if (c < n_chunks && t < a.T)
                            xv[tt] = __ldg(reinterpret_cast<const uint4*>(a.x + t * H + 8 * c));
                    }
                    const uint4* wrow = wg_s + (size_t)ms * 8 * Q * 32 + lane;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        float xf[NT];
#pragma unroll
                        for (int tt = 0; tt < NT; ++tt) {
                            uint32_t word = (i < 2) ? xv[tt].x : (i < 4) ? xv[tt].y
                                          : (i < 6) ? xv[tt].z : xv[tt].w;
                            xf[tt] = (i & 1) ? bf16_hi(word) : bf16_lo(word);
                        }
#pragma unroll
                        for (int q = 0; q < Q; ++q) {
                            const uint4 w = wrow[(i * Q + q) * 32];
                            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                const float wl = bf16_lo(ww[u]);
                                const float wh = bf16_hi(ww[u]);
#pragma unroll
                                for (int tt = 0; tt < NT; ++tt) {
                                    acc[tt][8 * q + 2 * u] = fmaf(xf[tt], wl, acc[tt][8 * q + 2 * u]);
                                    acc[tt][8 * q + 2 * u + 1] =
                                        fmaf(xf[tt], wh, acc[tt][8 * q + 2 * u + 1]);
                                }
                            }
                        }
                    }
                }
            }
            // xor butterfly over the 32 canonical lanes, strides 16..1
#pragma unroll
            for (int tt = 0; tt < NT; ++tt) {
#pragma unroll
                for (int e = 0; e < EB; ++e) {
                    float v = acc[tt][e];
#pragma unroll
                    for (int s = 16; s >= 1; s >>= 1) v = v + __shfl_xor_sync(0xffffffffu, v, s);
                    const int eg = eb * EB + e;
                    if (lane == 0 && eg < E) {
                        if (a.bias) v = v + a.bias[eg];
                        my_logits[tt * E + eg] = v;
                    }
                }
            }
        }
        __syncwarp();

        // top-k per token: each lane scans experts e = lane, lane+32, ...;
        // a warp argmax (larger value, ties to the lower id) picks each rank.
        for (int tt = 0; tt < NT; ++tt) {
            const int64_t t = t0 + tt;
            if (t >= a.T) break;
            const float* l = my_logits + tt * E;
            uint32_t taken = 0;   // bit u: expert lane + 32u already selected
            int sel_e[8];
            float sel_l[8];
            for (int j = 0; j < k; ++j) {
                float bv = 0.0f;
                int be = -1;
                for (int u = 0; lane + 32 * u < E; ++u) {
                    if (taken & (1u << u)) continue;
                    const float v = l[lane + 32 * u];
                    if (be < 0 || v > bv) { bv = v; be = lane + 32 * u; }
                }
#pragma unroll
                for (int s = 16; s >= 1; s >>= 1) {
                    const float ov = __shfl_xor_sync(0xffffffffu, bv, s);
                    const int oe = __shfl_xor_sync(0xffffffffu, be, s);
                    const bool better = (oe >= 0) && (be < 0 || ov > bv || (ov == bv && oe < be));
                    if (better) { bv = ov; be = oe; }
                }
                if ((be & 31) == lane) taken |= 1u << (be >> 5);
                sel_e[j < 8 ? j : 7] = be;
                sel_l[j < 8 ? j : 7] = bv;
            }
            if (lane == 0) {
                const float m = sel_l[0];
                float ex[8];
                float den = 0.0f;
                for (int j = 0; j < k; ++j) {
                    ex[j] = expf(sel_l[j] - m);
                    den = den + ex[j];
                }
                for (int j = 0; j < k; ++j) {
                    a.topk_idx[t * k + j] = sel_e[j];
                    a.topk_w[t * k + j] = ex[j] / den;
                }
            }
        }
        __syncwarp();
    }
}

template <int EB, int NT>
cudaError_t launch_route_t(const RouteArgs& a, int num_sms, cudaStream_t s)
{
    constexpr int Q = EB / 8;
    const int n_steps = (a.H / 8 + 31) / 32;
    const int step_bytes = 8 * Q * 32 * 16;   // one m-step of the gate slice
    int ms = kSliceBytes / step_bytes;
    if (ms < 1) ms = 1;
    if (ms > n_steps) ms = n_steps;
    const size_t smem = (size_t)ms * step_bytes + (size_t)kRouteWarps * NT * a.E * sizeof(float);
    auto kern = route_kernel<EB, NT>;
    cudaError_t err =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    const int64_t groups = (a.T + (int64_t)kRouteWarps * NT - 1) / ((int64_t)kRouteWarps * NT);
    const int grid = (int)(groups < num_sms ? groups : num_sms);
    kern<<<grid, kRouteThreads, smem, s>>>(a, ms);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_route(const RouteArgs& a, int num_sms, cudaStream_t s)
{
    if (a.T == 0) return cudaSuccess;
    if (a.E <= 8) return launch_route_t<8, 4>(a, num_sms, s);
    if (a.E <= 16) return launch_route_t<16, 2>(a, num_sms, s);
    if (a.E <= 32) return launch_route_t<32, 2>(a, num_sms, s);
    return launch_route_t<64, 1>(a, num_sms, s);
}

}  // namespace moe
