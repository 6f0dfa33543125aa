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
// Three kernels compute this order.
//
// route_stream_kernel (E <= 8, the gate fits shared memory): see its own
// comment below; TMA-fed per-warp pipelines and mixed-precision FMAs.
//
// route_cluster_kernel (8 < E <= 64). The canonical lanes are
// independent until the butterfly, and lanes L and L' with L = L' (mod CS)
// meet only in its last log2(CS) levels (strides CS/2 .. 1). So a cluster of
// CS CTAs splits the canonical lanes: CTA `rank` owns the lanes L = rank (mod
// CS). Each CTA keeps only its part of the gate, H*E*2/CS bytes, resident in
// shared memory for the whole kernel (CS is the smallest power of two that
// makes it fit), and streams only its own 16-byte chunks of x. The butterfly
// levels with stride >= CS run inside the CTA (a transpose-reduce: at each
// stride a lane keeps half of its values and adds its partner's copy of that
// half, so every sum has the butterfly's operands); the CS-1 remote partial
// sums then go to rank 0 through distributed shared memory, which finishes
// the levels CS/2 .. 1 in the same tree. x arrives through a ring of three
// 256-element steps in shared memory, filled with asynchronous 16-byte copies
// two steps ahead, so HBM latency is hidden without registers. A thread holds
// NT tokens x EW experts of fp32 accumulators; the warps of a CTA are split
// into expert and token subgroups.
//
// route_kernel (E > 64, or a gate too large for the other two): one CTA per
// SM, warp lane L = canonical lane L, the gate staged in 64 KB slices of H for
// every group of tokens.
//
// The last two stage Wg in a lane-major layout, [step m][element i][expert octet q]
// [lane] of uint4 (8 bf16 experts), so the lanes of a warp read consecutive
// 16-byte words (no bank conflicts).
#include <cooperative_groups.h>
#include <cstdint>
#include <cstring>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/moe.h"
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
    pdl_wait();
    pdl_launch_dependents();
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
            // without renormalisation the denominator runs over all E experts
            float den_all = 0.0f;
            if (!a.renorm) {
                for (int u = 0; lane + 32 * u < E; ++u) den_all += expf(l[lane + 32 * u] - sel_l[0]);
#pragma unroll
                for (int st = 16; st >= 1; st >>= 1) den_all += __shfl_xor_sync(0xffffffffu, den_all, st);
            }
            if (lane == 0) {
                const float m = sel_l[0];
                float ex[8];
                float den = 0.0f;
                for (int j = 0; j < k; ++j) {
                    ex[j] = expf(sel_l[j] - m);
                    den = den + ex[j];
                }
                if (!a.renorm) den = den_all;
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
    return launch_pdl(kern, dim3(grid), dim3(kRouteThreads), smem, s, a, ms);
}

// ------------------------------------------------------ cluster router --

namespace cg = cooperative_groups;

constexpr int kCWarps = 16;
constexpr int kCThreads = kCWarps * 32;
constexpr int kRing = 3;                       // x ring depth, in steps
constexpr size_t kSmemBudget = 220 * 1024;     // dynamic shared memory per CTA
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

template <int CS_, int EW_, int EWG_, int NT_, bool WF32_, int MINB_>
struct CShape {
    static constexpr int CS = CS_;                  // CTAs per cluster (canonical lane split)
    static constexpr int EW = EW_;                  // experts per thread
    static constexpr int EWG = EWG_;                // expert subgroups of warps
    static constexpr int NT = NT_;                  // tokens per thread
    static constexpr bool WF32 = WF32_;             // gate kept as fp32 (else bf16) in smem
    static constexpr int MINB = MINB_;              // CTAs per SM the registers must allow
    static constexpr int LC = 32 / CS;              // canonical lanes per CTA
    static constexpr int EB = EW * EWG;             // experts held (E padded)
    static constexpr int VW = WF32 ? 4 : 8;         // experts per 16-byte gate word
    static constexpr int QV = EB / VW;              // gate words per (step, element, lane)
    static constexpr int TS = kCWarps / EWG;        // token subgroups of warps
    static constexpr int TB = TS * CS * NT;         // tokens per group
    static constexpr int TBO = TB / CS;             // tokens of a group finished by each rank
    static constexpr int GATE_STEP_U4 = 8 * QV * LC;
    static constexpr int X_STEP_U4 = TB * LC;
    static constexpr int LOG_LC = LC == 32 ? 5 : LC == 16 ? 4 : LC == 8 ? 3 : 2;
    static constexpr int LOG_QV = QV == 1 ? 0 : QV == 2 ? 1 : QV == 4 ? 2 : QV == 8 ? 3 : 4;
    static_assert((1 << LOG_QV) == QV && (1 << LOG_LC) == LC, "power-of-two shapes");

    static size_t smem_bytes(int H, int E)
    {
        const size_t n_steps = (size_t)(H / 8 + 31) / 32;
        return n_steps * GATE_STEP_U4 * 16 + (size_t)kRing * X_STEP_U4 * 16 +
               (size_t)CS * TBO * EB * 4 + (size_t)TBO * E * 4;
    }
};

// Transpose-reduce of N values per lane over strides St, St/2, .., 1. While
// N > 1 a lane keeps the half selected by its stride bit and adds the
// partner's copy of that half; once N == 1 it is a plain butterfly step.
template <int N, int St>
__device__ __forceinline__ void transpose_reduce(float* v, int lane)
{
    if constexpr (N > 1) {
        const bool up = (lane & St) != 0;
#pragma unroll
        for (int i = 0; i < N / 2; ++i) {
            const float send = up ? v[i] : v[i + N / 2];
            const float keep = up ? v[i + N / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(kFull, send, St);
        }
        if constexpr (St > 1) transpose_reduce<N / 2, St / 2>(v, lane);
    } else {
        v[0] = v[0] + __shfl_xor_sync(kFull, v[0], St);
        if constexpr (St > 1) transpose_reduce<1, St / 2>(v, lane);
    }
}

// After transpose_reduce<N, LC/2>, the lane with sub-lane r holds experts
// first .. first + count - 1 of its N; `writer` marks one lane per set.
template <int N, int LC>
__device__ __forceinline__ void reduced_slots(int r, int& first, int& count, bool& writer)
{
    int n = N, base = 0, dup = 0;
#pragma unroll
    for (int st = LC / 2; st >= 1; st >>= 1) {
        if (n > 1) {
            if (r & st) base += n / 2;
            n /= 2;
        } else {
            dup |= st;
        }
    }
    first = base;
    count = n;
    writer = (r & dup) == 0;
}

// The gate words of this CTA's canonical lanes, all steps, into shared memory:
// layout [step m][element i][word q][sub-lane r]; word q holds experts
// VW*q .. VW*q+VW-1 of hidden row h = 256 m + 8 (r*CS + rank) + i.
template <class S>
__device__ void stage_gate_cluster(uint4* gate, const uint16_t* __restrict__ Wg, int H, int E, int n_steps,
                                   int rank)
{
    const int total = n_steps * S::GATE_STEP_U4;
    auto coords = [&](int idx, int& h, int& e) {
        const int rr = idx & (S::LC - 1);
        const int rest = idx >> S::LOG_LC;
        const int q = rest & (S::QV - 1);
        const int i = (rest >> S::LOG_QV) & 7;
        const int m = rest >> (S::LOG_QV + 3);
        h = m * 256 + 8 * (rr * S::CS + rank) + i;
        e = S::VW * q;
    };
    if constexpr (!S::WF32) {
        const bool vec = (E % 8 == 0);
        for (int idx = threadIdx.x; idx < total; idx += kCThreads) {
            int h, e;
            coords(idx, h, e);
            if (vec) {
                const bool in = (h < H) && (e + 8 <= E);
                cp_async_16(smem_u32(gate + idx), in ? Wg + (int64_t)h * E + e : Wg, in ? 16u : 0u);
            } else {
                uint32_t w[4] = {0, 0, 0, 0};
                if (h < H)
                    for (int u = 0; u < 8 && e + u < E; ++u)
                        w[u >> 1] |= (uint32_t)Wg[(int64_t)h * E + e + u] << (16 * (u & 1));
                gate[idx] = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
    } else {
        // fp32 words: loads issued in batches of 8 per thread, then widened
        const bool vec = (E % 4 == 0);
        constexpr int B = 8;
        for (int base = threadIdx.x; base < total; base += B * kCThreads) {
            uint2 raw[B];
#pragma unroll
            for (int b = 0; b < B; ++b) {
                const int idx = base + b * kCThreads;
                raw[b] = make_uint2(0, 0);
                if (idx < total) {
                    int h, e;
                    coords(idx, h, e);
                    if (h < H) {
                        const uint16_t* src = Wg + (int64_t)h * E + e;
                        if (vec && e + 4 <= E) {
                            raw[b] = __ldg(reinterpret_cast<const uint2*>(src));
                        } else {
                            uint32_t w[2] = {0, 0};
                            for (int u = 0; u < 4 && e + u < E; ++u)
                                w[u >> 1] |= (uint32_t)src[u] << (16 * (u & 1));
                            raw[b] = make_uint2(w[0], w[1]);
                        }
                    }
                }
            }
#pragma unroll
            for (int b = 0; b < B; ++b) {
                const int idx = base + b * kCThreads;
                if (idx < total)
                    reinterpret_cast<float4*>(gate)[idx] =
                        make_float4(bf16_lo(raw[b].x), bf16_hi(raw[b].x), bf16_lo(raw[b].y), bf16_hi(raw[b].y));
            }
        }
    }
}

template <class S>
__global__ void __launch_bounds__(kCThreads, S::MINB) route_cluster_kernel(RouteArgs a)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    pdl_wait();
    pdl_launch_dependents();
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = S::CS > 1 ? (int)cluster.block_rank() : 0;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int r = lane & (S::LC - 1);      // this CTA's canonical lane r*CS + rank
    const int slot = lane >> S::LOG_LC;    // token slot within the warp
    const int eg = warp % S::EWG;
    const int ts = warp / S::EWG;
    const int H = a.H, E = a.E, k = a.k;
    const int n_steps = (H / 8 + 31) / 32;
    const int n_chunks = H / 8;

    uint4* gate = reinterpret_cast<uint4*>(smem_raw);
    uint4* ring = gate + (size_t)n_steps * S::GATE_STEP_U4;
    float* red = reinterpret_cast<float*>(ring + kRing * S::X_STEP_U4);   // [CS][TBO][EB]
    float* logit_s = red + S::CS * S::TBO * S::EB;                       // [TBO][E]

    const int64_t n_clusters = gridDim.x / S::CS;
    const int64_t group_stride = n_clusters * S::TB;
    int64_t t0 = (int64_t)(blockIdx.x / S::CS) * S::TB;
    if (t0 >= a.T) return;   // the whole cluster leaves together

    stage_gate_cluster<S>(gate, a.Wg, H, E, n_steps, rank);

    // x of one step for the group starting at g0 into ring slot `sl`
    auto stage_x = [&](int sl, int64_t g0, int m) {
#pragma unroll
        for (int j = 0; j < (S::X_STEP_U4 + kCThreads - 1) / kCThreads; ++j) {
            const int idx = threadIdx.x + j * kCThreads;
            if (idx < S::X_STEP_U4) {
                const int64_t t = g0 + (idx >> S::LOG_LC);
                const int c = m * 32 + (idx & (S::LC - 1)) * S::CS + rank;
                const bool in = (t < a.T) && (c < n_chunks);
                cp_async_16(smem_u32(ring + sl * S::X_STEP_U4 + idx), in ? a.x + t * H + 8 * c : a.x,
                            in ? 16u : 0u);
            }
        }
    };
    // prefetch cursor, kRing-1 steps ahead (commit groups: prologue 0..kRing-2,
    // step number s commits s + kRing - 1; the bf16 gate copies are in group 0)
    int64_t pf_t0 = t0;
    int pf_m = 0, pf_slot = 0;
    auto pf_issue = [&]() {
        if (pf_t0 < a.T) {
            stage_x(pf_slot, pf_t0, pf_m);
            if (++pf_m == n_steps) { pf_m = 0; pf_t0 += group_stride; }
            if (++pf_slot == kRing) pf_slot = 0;
        }
    };
#pragma unroll
    for (int j = 0; j < kRing - 1; ++j) {
        pf_issue();
        cp_async_commit();
    }

    int first, count;
    bool writer;
    reduced_slots<S::EW, S::LC>(r, first, count, writer);
    constexpr int MAXC = S::EW / S::LC > 0 ? S::EW / S::LC : 1;
    auto tok = [&](int jt) { return (ts * S::CS + slot) * S::NT + jt; };

    float acc[S::NT][S::EW];
    int cur_slot = 0;
    while (t0 < a.T) {
#pragma unroll
        for (int jt = 0; jt < S::NT; ++jt)
#pragma unroll
            for (int e = 0; e < S::EW; ++e) acc[jt][e] = 0.0f;

        for (int m = 0; m < n_steps; ++m) {
            __syncthreads();   // the previous step is done: its ring slot is free
            pf_issue();
            cp_async_commit();
            cp_async_wait<kRing - 1>();   // x of this step (and the gate) has landed
            __syncthreads();

            const uint4* xs = ring + cur_slot * S::X_STEP_U4 + ((ts * S::CS + slot) * S::NT) * S::LC + r;
            const uint4* gs = gate + (size_t)m * S::GATE_STEP_U4 + (eg * (S::EW / S::VW)) * S::LC + r;
            uint4 xv[S::NT];
#pragma unroll
            for (int jt = 0; jt < S::NT; ++jt) xv[jt] = xs[jt * S::LC];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float xf[S::NT];
#pragma unroll
                for (int jt = 0; jt < S::NT; ++jt) {
                    const uint32_t word = (i < 2) ? xv[jt].x : (i < 4) ? xv[jt].y
                                        : (i < 6) ? xv[jt].z : xv[jt].w;
                    xf[jt] = (i & 1) ? bf16_hi(word) : bf16_lo(word);
                }
#pragma unroll
                for (int q = 0; q < S::EW / S::VW; ++q) {
                    const uint4 w = gs[(i * S::QV + q) * S::LC];
                    float wf[S::VW];
                    if constexpr (S::WF32) {
                        wf[0] = __uint_as_float(w.x); wf[1] = __uint_as_float(w.y);
                        wf[2] = __uint_as_float(w.z); wf[3] = __uint_as_float(w.w);
                    } else {
                        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            wf[2 * u] = bf16_lo(ww[u]);
                            wf[2 * u + 1] = bf16_hi(ww[u]);
                        }
                    }
#pragma unroll
                    for (int u = 0; u < S::VW; ++u)
#pragma unroll
                        for (int jt = 0; jt < S::NT; ++jt)
                            acc[jt][S::VW * q + u] = fmaf(xf[jt], wf[u], acc[jt][S::VW * q + u]);
                }
            }
            if (++cur_slot == kRing) cur_slot = 0;
        }

        // butterfly levels with stride >= CS, inside the CTA
#pragma unroll
        for (int jt = 0; jt < S::NT; ++jt) transpose_reduce<S::EW, S::LC / 2>(acc[jt], r);
        const int e_base = eg * S::EW + first;

        // each rank finishes the tokens tt with tt mod CS == rank: every rank
        // sends it its partial sums (its own included)
        cluster.sync();   // the owners are done with the previous group's partial sums
        if (writer) {
#pragma unroll
            for (int jt = 0; jt < S::NT; ++jt) {
                const int tt = tok(jt);
                float* dst = (S::CS > 1 ? cluster.map_shared_rank(red, tt % S::CS) : red) +
                             (rank * S::TBO + tt / S::CS) * S::EB + e_base;
#pragma unroll
                for (int c = 0; c < MAXC; ++c)
                    if (c < count) dst[c] = acc[jt][c];
            }
        }
        cluster.sync();   // every partial sum has arrived at its owner
        // butterfly levels with stride < CS across the ranks, then the bias
        for (int idx = threadIdx.x; idx < S::TBO * E; idx += kCThreads) {
            const int u = idx / E, e = idx - u * E;
            float v[S::CS];
#pragma unroll
            for (int rho = 0; rho < S::CS; ++rho) v[rho] = red[(rho * S::TBO + u) * S::EB + e];
#pragma unroll
            for (int st = S::CS / 2; st >= 1; st >>= 1) {
                float nv[S::CS];
#pragma unroll
                for (int rho = 0; rho < S::CS; ++rho) nv[rho] = v[rho] + v[rho ^ st];
#pragma unroll
                for (int rho = 0; rho < S::CS; ++rho) v[rho] = nv[rho];
            }
            float l = v[0];
            if (a.bias) l = l + a.bias[e];
            logit_s[idx] = l;
        }
        __syncthreads();
        // top-k of this rank's tokens, one warp per token: each lane scans experts
        // e = lane, lane+32; a warp argmax (larger value, ties to the lower id).
        for (int u = warp; u < S::TBO; u += kCWarps) {
            const int64_t t = t0 + (int64_t)u * S::CS + rank;
            if (t >= a.T) break;
            const float* l = logit_s + u * E;
            uint32_t taken = 0;
            int sel_e[8];
            float sel_l[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (j >= k) break;
                float bv = 0.0f;
                int be = -1;
                for (int uu = 0; lane + 32 * uu < E; ++uu) {
                    if (taken & (1u << uu)) continue;
                    const float v = l[lane + 32 * uu];
                    if (be < 0 || v > bv) { bv = v; be = lane + 32 * uu; }
                }
#pragma unroll
                for (int st = 16; st >= 1; st >>= 1) {
                    const float ov = __shfl_xor_sync(kFull, bv, st);
                    const int oe = __shfl_xor_sync(kFull, be, st);
                    const bool better = (oe >= 0) && (be < 0 || ov > bv || (ov == bv && oe < be));
                    if (better) { bv = ov; be = oe; }
                }
                if ((be & 31) == lane) taken |= 1u << (be >> 5);
                sel_e[j] = be;
                sel_l[j] = bv;
            }
            // without renormalisation the denominator runs over all E experts
            float den_all = 0.0f;
            if (!a.renorm) {
                for (int uu = 0; lane + 32 * uu < E; ++uu) den_all += expf(l[lane + 32 * uu] - sel_l[0]);
#pragma unroll
                for (int st = 16; st >= 1; st >>= 1) den_all += __shfl_xor_sync(kFull, den_all, st);
            }
            if (lane == 0) {
                const float mx = sel_l[0];
                float ex[8];
                float den = 0.0f;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (j >= k) break;
                    ex[j] = expf(sel_l[j] - mx);
                    den = den + ex[j];
                }
                if (!a.renorm) den = den_all;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (j >= k) break;
                    a.topk_idx[t * k + j] = sel_e[j];
                    a.topk_w[t * k + j] = ex[j] / den;
                }
            }
        }
        t0 += group_stride;
    }
    cp_async_wait<0>();   // nothing in flight at exit
    if (S::CS > 1) cluster.sync();   // no rank leaves while another may still read its smem
}

template <class S>
cudaError_t launch_cluster(const RouteArgs& a, int num_sms, cudaStream_t s)
{
    const size_t smem = S::smem_bytes(a.H, a.E);
    auto kern = route_cluster_kernel<S>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    const int64_t groups = (a.T + S::TB - 1) / S::TB;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kCThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = S::CS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;   // the occupancy query sees the cluster shape only
    int64_t clusters = (int64_t)num_sms * S::MINB / S::CS;
    cfg.gridDim = dim3((unsigned)(clusters * S::CS));
    int max_clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&max_clusters, kern, &cfg) == cudaSuccess && max_clusters > 0)
        clusters = max_clusters;
    if (clusters > groups) clusters = groups;
    if (clusters < 1) clusters = 1;
    cfg.gridDim = dim3((unsigned)(clusters * S::CS));
    cfg.numAttrs = 2;
    err = cudaLaunchKernelEx(&cfg, kern, a);
    if (err != cudaSuccess) return err;
    count_launch();
    return cudaGetLastError();
}

// The first cluster shape (in the order given) whose shared memory fits.
template <int EW, int EWG, int NT, int MINB, int CS0>
cudaError_t launch_cluster_any(const RouteArgs& a, int num_sms, cudaStream_t s, bool& launched)
{
    launched = true;
#define MOE_TRY_SHAPE(CS, F32)                                                                 \
    if ((CS) >= CS0 && CShape<CS, EW, EWG, NT, F32, MINB>::smem_bytes(a.H, a.E) <= kSmemBudget) \
        return launch_cluster<CShape<CS, EW, EWG, NT, F32, MINB>>(a, num_sms, s);
    // clusters of 8 are placed on fewer SMs (15 clusters, 120 SMs, measured),
    // so a bf16 gate in a cluster of <= 4 beats an fp32 gate in a cluster of 8
    MOE_TRY_SHAPE(2, true)
    MOE_TRY_SHAPE(4, true)
    MOE_TRY_SHAPE(2, false)
    MOE_TRY_SHAPE(4, false)
    MOE_TRY_SHAPE(8, true)
    MOE_TRY_SHAPE(8, false)
#undef MOE_TRY_SHAPE
    launched = false;
    return cudaSuccess;
}


// ----------------------------------------------------- streaming router --
//
// route_stream_kernel (E <= 8). One CTA per SM; every warp is an independent
// pipeline over groups of NT tokens, so no CTA barrier couples the warps once
// they run. Lane L of a warp is the canonical lane L.
//
// Gate. Kept bf16 in shared memory as the gate viewed as a [H/8][64] matrix
// (row c = the 8 hidden rows of chunk c, 8 experts each) in 128-byte-swizzled
// rows: chunk c's element i sits at byte c*128 + ((i ^ (c & 7)) << 4). The
// 32 lanes of a warp read 32 consecutive chunks at one element, which the
// swizzle spreads over all banks. With E == 8 the gate arrives by one TMA
// copy per 256-element step, each completing its own mbarrier, so a warp
// starts on step 0 while later steps are still in flight; otherwise (E < 8,
// rows are not 16 bytes) threads stage it with plain stores.
//
// x. Each warp streams its tokens through a ring of D steps in shared memory,
// one TMA copy (NT token rows x 256 elements) per step, D-1 steps ahead of
// use. Bulk copies keep enough bytes in flight per SM to cover HBM latency,
// which per-thread copies, limited by the outstanding-miss tracking of the
// load path, did not (measured).
//
// FMAs. The mixed-precision form fma.rn.f32.bf16 takes the bf16 operands as
// they are: widening bf16 to fp32 is exact and the product is rounded once
// with the add, so each step is fmaf on the widened values, bit for bit, in
// the canonical order. After a group's steps a transpose-reduce (the
// butterfly's operands and tree) leaves every logit on one lane (two with
// NT == 8), and the top-k runs as a shuffle argmax among the lanes that hold
// one token's logits.

// acc[e] = fma(x, g[e], acc[e]) for the 8 experts of one hidden element: x is
// half XH of the x word, g[e] half e&1 of gate word e>>1.
#define MOE_FMA8_BF16(XH)                                                                    \
    asm("{\n\t.reg .b16 xl, xh, g0, g1, g2, g3, g4, g5, g6, g7;\n\t"                        \
        "mov.b32 {xl, xh}, %8;\n\t"                                                            \
        "mov.b32 {g0, g1}, %9;\n\t"                                                            \
        "mov.b32 {g2, g3}, %10;\n\t"                                                           \
        "mov.b32 {g4, g5}, %11;\n\t"                                                           \
        "mov.b32 {g6, g7}, %12;\n\t"                                                           \
        "fma.rn.f32.bf16 %0, " XH ", g0, %0;\n\t"                                              \
        "fma.rn.f32.bf16 %1, " XH ", g1, %1;\n\t"                                              \
        "fma.rn.f32.bf16 %2, " XH ", g2, %2;\n\t"                                              \
        "fma.rn.f32.bf16 %3, " XH ", g3, %3;\n\t"                                              \
        "fma.rn.f32.bf16 %4, " XH ", g4, %4;\n\t"                                              \
        "fma.rn.f32.bf16 %5, " XH ", g5, %5;\n\t"                                              \
        "fma.rn.f32.bf16 %6, " XH ", g6, %6;\n\t"                                              \
        "fma.rn.f32.bf16 %7, " XH ", g7, %7;\n\t}"                                             \
        : "+f"(acc[0]), "+f"(acc[1]), "+f"(acc[2]), "+f"(acc[3]), "+f"(acc[4]), "+f"(acc[5]),    \
          "+f"(acc[6]), "+f"(acc[7])                                                             \
        : "r"(xw), "r"(g.x), "r"(g.y), "r"(g.z), "r"(g.w))
template <int HALF>
__device__ __forceinline__ void fma8_bf16(float (&acc)[8], uint32_t xw, const uint4& g)
{
    if constexpr (HALF) MOE_FMA8_BF16("xh");
    else MOE_FMA8_BF16("xl");
}
#undef MOE_FMA8_BF16

template <int NT_, int D_, int NW_>
struct SShape {
    static constexpr int NT = NT_;   // tokens per warp group (rows of one x copy)
    static constexpr int D = D_;     // x ring depth per warp, in steps
    static constexpr int NW = NW_;   // warps per CTA
    static constexpr int THREADS = NW * 32;
    static constexpr int SLOT_BYTES = NT * 512;   // NT rows x 256 bf16
    static size_t smem_bytes(int H)
    {
        const size_t n_steps = (size_t)(H / 8 + 31) / 32;
        return 1024 + n_steps * 4096 + (size_t)NW * D * SLOT_BYTES + (n_steps + (size_t)NW * D) * 8 + 16;
    }
};

template <class S>
__global__ void __launch_bounds__(S::THREADS, 1)
    route_stream_kernel(const __grid_constant__ CUtensorMap gmap, const __grid_constant__ CUtensorMap xmap,
                        RouteArgs a, int gate_tma, int n_sl)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    pdl_wait();
    pdl_launch_dependents();
    constexpr int NT = S::NT, D = S::D, NW = S::NW;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int H = a.H, E = a.E, k = a.k;
    const int n_steps = (H / 8 + 31) / 32;

    unsigned char* gate = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);   // [m][32][128 B]
    unsigned char* ring_all = gate + (size_t)n_steps * 4096;
    unsigned char* ring = ring_all + (size_t)warp * D * S::SLOT_BYTES;               // [slot][token][512 B]
    uint64_t* gbar = reinterpret_cast<uint64_t*>(ring_all + (size_t)NW * D * S::SLOT_BYTES);
    uint64_t* xbar = gbar + n_steps + warp * D;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gbar + n_steps + NW * D);

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        if (gate_tma)
            for (int m = 0; m < n_steps; ++m) mbar_init(smem_u32(gbar + m), 1);
        for (int b = 0; b < NW * D; ++b) mbar_init(smem_u32(gbar + n_steps + b), 1);
        fence_barrier_init();
    }
    // expert slice: with n_sl > 1 a CTA computes the logits of experts
    // 8*slice .. 8*slice+7 only; CTAs b = n_sl*r .. n_sl*r+n_sl-1 (one stream
    // r) take the same tokens at the same time, so x is read from HBM about once
    const int slice = blockIdx.x % n_sl;
    if (n_sl > 1) {
        for (int h = threadIdx.x; h < n_steps * 256; h += S::THREADS) {
            const int c = h >> 3, i = h & 7;
            const bool in = h < H;
            cp_async_16(smem_u32(gate + (size_t)c * 128 + ((i ^ (c & 7)) << 4)),
                        in ? a.Wg + (int64_t)h * E + 8 * slice : a.Wg, in ? 16u : 0u);
        }
        cp_async_commit();
        cp_async_wait<0>();
    } else if (!gate_tma) {
        for (int h = threadIdx.x; h < n_steps * 256; h += S::THREADS) {
            uint32_t w[4] = {0, 0, 0, 0};
            if (h < H)
                for (int e = 0; e < E; ++e)
                    w[e >> 1] |= (uint32_t)a.Wg[(int64_t)h * E + e] << (16 * (e & 1));
            const int c = h >> 3, i = h & 7;
            *reinterpret_cast<uint4*>(gate + (size_t)c * 128 + ((i ^ (c & 7)) << 4)) =
                make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
    __syncthreads();   // barriers initialised (and a plainly staged gate visible)
    if (gate_tma && threadIdx.x == 0) {
        for (int m = 0; m < n_steps; ++m) {
            mbar_arrive_expect_tx(smem_u32(gbar + m), 4096);
            tma_load_2d(smem_u32(gate + (size_t)m * 4096), &gmap, 0, 32 * m, smem_u32(gbar + m));
        }
    }

    // token groups: warp w of stream r takes g = r + n_streams * (w + NW * j), j = 0, 1, ..
    const int64_t G = (a.T + NT - 1) / NT;
    const int n_streams = gridDim.x / n_sl;
    const int64_t g_first = blockIdx.x / n_sl + (int64_t)n_streams * warp;
    const int64_t g_stride = (int64_t)n_streams * NW;

    // prefetch cursor, D-1 steps ahead; lane 0 issues the copies
    int64_t pf_g = g_first;
    int pf_m = 0, pf_slot = 0;
    auto pf_issue = [&]() {
        if (pf_g < G) {
            if (lane == 0) {
                // the slot was last read a step ago (the __syncwarp before
                // this call): order those reads before the async-proxy write
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                const uint32_t bar = smem_u32(xbar + pf_slot);
                mbar_arrive_expect_tx(bar, S::SLOT_BYTES);
                tma_load_2d(smem_u32(ring + (size_t)pf_slot * S::SLOT_BYTES), &xmap, 256 * pf_m,
                            (int32_t)(pf_g * NT), bar);
            }
            if (++pf_m == n_steps) { pf_m = 0; pf_g += g_stride; }
            if (++pf_slot == D) pf_slot = 0;
        }
    };
#pragma unroll
    for (int j = 0; j < D - 1; ++j) pf_issue();

    // this lane's gate words: chunk 32m + lane, element i at gl + m*4096 + (i ^ (lane & 7))*16
    const unsigned char* gl = gate + lane * 128;
    const int sw = lane & 7;

    // the lanes that hold one token's logits after the reduce
    constexpr int NV = NT * 8 > 32 ? NT * 8 / 32 : 1;       // logits per lane
    constexpr int LOG_DUP = NT == 1 ? 2 : NT == 2 ? 1 : 0;   // lanes holding copies
    constexpr int SL = 32 / NT;                              // lanes per token
    static_assert(NT == 1 || NT == 2 || NT == 4 || NT == 8, "NT in {1, 2, 4, 8}");
    const int vbase = NV * (lane >> LOG_DUP);
    const int my_tt = vbase >> 3;
    const int e0 = vbase & 7;

    int cur = 0;
    uint32_t phases = 0;   // bit s: parity of the next completion of slot s
    bool first = true;
    for (int64_t g = g_first; g < G; g += g_stride) {
        float acc[NT][8];
#pragma unroll
        for (int tt = 0; tt < NT; ++tt)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[tt][e] = 0.0f;

        for (int m = 0; m < n_steps; ++m) {
            __syncwarp();   // every lane is done with the slot the next copy overwrites
            pf_issue();
            if (gate_tma && first) mbar_wait(smem_u32(gbar + m), 0, abort_flag, a.err);
            mbar_wait(smem_u32(xbar + cur), (phases >> cur) & 1u, abort_flag, a.err);
            phases ^= 1u << cur;
            const unsigned char* xs = ring + (size_t)cur * S::SLOT_BYTES + lane * 16;
            uint4 xv[NT];
#pragma unroll
            for (int tt = 0; tt < NT; ++tt) xv[tt] = *reinterpret_cast<const uint4*>(xs + tt * 512);
            const unsigned char* gs = gl + (size_t)m * 4096;
#pragma unroll
            for (int q = 0; q < 4; ++q) {   // elements 2q, 2q+1: word q of each x chunk
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const uint4 gw = *reinterpret_cast<const uint4*>(gs + (((2 * q + half) ^ sw) << 4));
#pragma unroll
                    for (int tt = 0; tt < NT; ++tt) {
                        const uint32_t w = q == 0 ? xv[tt].x : q == 1 ? xv[tt].y : q == 2 ? xv[tt].z : xv[tt].w;
                        if (half) fma8_bf16<1>(acc[tt], w, gw);
                        else fma8_bf16<0>(acc[tt], w, gw);
                    }
                }
            }
            if (++cur == D) cur = 0;
        }
        first = false;

        // the butterfly over the 32 canonical lanes, as a transpose-reduce:
        // afterwards this lane holds logits e0 .. e0+NV-1 of token my_tt
        float v[NT * 8];
#pragma unroll
        for (int tt = 0; tt < NT; ++tt)
#pragma unroll
            for (int e = 0; e < 8; ++e) v[tt * 8 + e] = acc[tt][e];
        transpose_reduce<NT * 8, 16>(v, lane);
        if (n_sl > 1) {
            // this slice's logits (bias added) for the top-k pass
            const int64_t t = g * NT + my_tt;
            if ((lane & ((1 << LOG_DUP) - 1)) == 0 && t < a.T) {
#pragma unroll
                for (int u = 0; u < NV; ++u) {
                    const int e = 8 * slice + e0 + u;
                    float l = v[u];
                    if (a.bias) l = l + a.bias[e];
                    a.logits[t * E + e] = l;
                }
            }
            continue;
        }
        float l[NV];
#pragma unroll
        for (int u = 0; u < NV; ++u) {
            l[u] = v[u];
            if (a.bias && e0 + u < E) l[u] = l[u] + a.bias[e0 + u];
        }

        // top-k: k rounds of an argmax over the token's lanes (larger logit,
        // ties to the lower id); the winner's holder marks it taken
        uint32_t taken = 0;
        int sel_e[8];
        float sel_l[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (j >= k) break;
            float bv = 0.0f;
            int be = -1;
#pragma unroll
            for (int u = 0; u < NV; ++u) {
                const bool ok = (e0 + u < E) && !((taken >> u) & 1u);
                if (ok && (be < 0 || l[u] > bv)) { bv = l[u]; be = e0 + u; }
            }
#pragma unroll
            for (int st = 1; st < SL; st <<= 1) {
                const float ov = __shfl_xor_sync(kFull, bv, st);
                const int oe = __shfl_xor_sync(kFull, be, st);
                const bool better = (oe >= 0) && (be < 0 || ov > bv || (ov == bv && oe < be));
                if (better) { bv = ov; be = oe; }
            }
            if (be >= e0 && be < e0 + NV) taken |= 1u << (be - e0);
            sel_e[j] = be;
            sel_l[j] = bv;
        }
        const float mx = sel_l[0];
        // without renormalisation the denominator runs over all E experts
        float den_all = 0.0f;
        if (!a.renorm) {
#pragma unroll
            for (int u = 0; u < NV; ++u)
                if (e0 + u < E && (lane & ((1 << LOG_DUP) - 1)) == 0) den_all = den_all + expf(l[u] - mx);
#pragma unroll
            for (int st = 1; st < SL; st <<= 1) den_all = den_all + __shfl_xor_sync(kFull, den_all, st);
        }
        const int64_t t = g * NT + my_tt;
        if ((lane & (SL - 1)) == 0 && t < a.T) {
            float ex[8];
            float den = 0.0f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (j >= k) break;
                ex[j] = expf(sel_l[j] - mx);
                den = den + ex[j];
            }
            if (!a.renorm) den = den_all;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (j >= k) break;
                a.topk_idx[t * k + j] = sel_e[j];
                a.topk_w[t * k + j] = ex[j] / den;
            }
        }
    }
    // every x copy a warp issued, it also waited for; a warp without tokens
    // never waited on the gate: no CTA exits while its copies may still land
    if (gate_tma && threadIdx.x == 0)
        for (int m = 0; m < n_steps; ++m) mbar_wait_drain(smem_u32(gbar + m), 0);
}

// Top-k and gate weights from the [T, E] logits the sliced router wrote. A
// warp takes 4 tokens, 8 lanes per token; lane r of a token holds experts
// r*E/8 .. r*E/8 + E/8 - 1 (E is a multiple of 8, at most 256). k rounds of
// an argmax (larger logit, ties to the lower id) over the token's 8 lanes.
// PMAX bounds E/8 at compile time, so the per-lane loops are no longer than
// the logits a lane holds.
template <int PMAX>
__global__ void route_topk_kernel(RouteArgs a)
{
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int r = lane & 7;
    const int E = a.E, k = a.k;
    const int per = E >> 3;   // logits per lane
    const int64_t t = ((int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * 4 + (lane >> 3);
    const bool live = t < a.T;
    const int e_lo = r * per;
    float lv[PMAX];
    const float* src = a.logits + t * E + e_lo;
    if ((per & 3) == 0) {   // 16-byte aligned runs of 4
#pragma unroll
        for (int u = 0; u < PMAX; u += 4) {
            float4 q = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            if (live && u < per) q = *reinterpret_cast<const float4*>(src + u);
            lv[u] = q.x; lv[u + 1] = q.y; lv[u + 2] = q.z; lv[u + 3] = q.w;
        }
    } else {
#pragma unroll
        for (int u = 0; u < PMAX; ++u) lv[u] = (live && u < per) ? src[u] : 0.0f;
    }
    uint32_t taken = 0;
    int sel_e[8];
    float sel_l[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        if (j >= k) break;
        float bv = 0.0f;
        int be = -1;
#pragma unroll
        for (int u = 0; u < PMAX; ++u)
            if (u < per && !((taken >> u) & 1u) && (be < 0 || lv[u] > bv)) { bv = lv[u]; be = e_lo + u; }
#pragma unroll
        for (int st = 1; st < 8; st <<= 1) {
            const float ov = __shfl_xor_sync(kFull, bv, st);
            const int oe = __shfl_xor_sync(kFull, be, st);
            const bool better = (oe >= 0) && (be < 0 || ov > bv || (ov == bv && oe < be));
            if (better) { bv = ov; be = oe; }
        }
        if (be >= e_lo && be < e_lo + per) taken |= 1u << (be - e_lo);
        sel_e[j] = be;
        sel_l[j] = bv;
    }
    const float mx = sel_l[0];
    // without renormalisation the denominator runs over all E experts
    float den_all = 0.0f;
    if (!a.renorm) {
#pragma unroll
        for (int u = 0; u < PMAX; ++u)
            if (u < per) den_all = den_all + expf(lv[u] - mx);
#pragma unroll
        for (int st = 1; st < 8; st <<= 1) den_all = den_all + __shfl_xor_sync(kFull, den_all, st);
    }
    if (r == 0 && live) {
        float ex[8];
        float den = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (j >= k) break;
            ex[j] = expf(sel_l[j] - mx);
            den = den + ex[j];
        }
        if (!a.renorm) den = den_all;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (j >= k) break;
            a.topk_idx[t * k + j] = sel_e[j];
            a.topk_w[t * k + j] = ex[j] / den;
        }
    }
}

// Returns false (nothing launched) when a tensor map cannot be made. With
// E > 8 (a multiple of 8, a.logits set) the experts are split in slices of 8
// over the CTAs of a stream and a second kernel takes the top-k.
template <class S>
bool launch_stream(const RouteArgs& a, int num_sms, cudaStream_t s, cudaError_t& err)
{
    const int n_sl = a.E > 8 ? a.E / 8 : 1;
    CUtensorMap gmap, xmap;
    std::memset(&gmap, 0, sizeof(gmap));
    // x as a bf16 [T, H] matrix, box {256, NT}: one step of NT token rows
    if (!encode_map_2d(&xmap, a.x, (uint64_t)a.H, (uint64_t)a.T, 256, S::NT, 0)) return false;
    // the gate Wg[H, 8] as a bf16 [H/8, 64] matrix, box {64, 32}, 128-byte swizzle
    const bool gate_tma = a.E == 8 && encode_map_2d(&gmap, a.Wg, 64, (uint64_t)a.H / 8, 64, 32, 128);
    const size_t smem = S::smem_bytes(a.H);
    auto kern = route_stream_kernel<S>;
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return true;
    // one CTA per SM; the token groups are dealt round-robin over the streams
    // (n_sl CTAs each), so every SM gets within one of the same number
    const int64_t G = (a.T + S::NT - 1) / S::NT;
    int64_t n_streams = num_sms / n_sl;
    if (n_streams > G) n_streams = G;
    if (n_streams < 1) n_streams = 1;
    err = launch_pdl(kern, dim3((unsigned)(n_streams * n_sl)), dim3(S::THREADS), smem, s, gmap, xmap, a,
                     gate_tma ? 1 : 0, n_sl);
    if (err != cudaSuccess || n_sl == 1) return true;
    const dim3 blocks((unsigned)((a.T + 31) / 32));   // 8 warps x 4 tokens
    if (n_sl <= 4)
        err = launch_pdl(route_topk_kernel<4>, blocks, dim3(256), 0, s, a);
    else if (n_sl <= 8)
        err = launch_pdl(route_topk_kernel<8>, blocks, dim3(256), 0, s, a);
    else if (n_sl <= 16)
        err = launch_pdl(route_topk_kernel<16>, blocks, dim3(256), 0, s, a);
    else
        err = launch_pdl(route_topk_kernel<32>, blocks, dim3(256), 0, s, a);
    return true;
}

}  // namespace

namespace {

constexpr size_t kStreamBudget = 227 * 1024;
// Twelve warps: the mixed-precision FMA needs more than two warps per
// scheduler to approach its issue rate (measured: 8 -> 12 warps,
// DeepSeek-shaped 244 -> 232 us; E = 8 unchanged).
using StreamShape = SShape<8, 3, 12>;

// Whether some cluster shape of this expert bucket fits shared memory (the
// smallest one: a cluster of 8 with a bf16 gate).
bool cluster_fits(int32_t H, int32_t E)
{
    if (E <= 8 || E > 64) return false;
    // the shapes launch_cluster_any tries for each bucket, at CS = 8, bf16 gate
    if (E <= 16) return CShape<8, 16, 1, 2, false, 1>::smem_bytes(H, E) <= kSmemBudget;
    if (E <= 32) return CShape<8, 16, 2, 4, false, 1>::smem_bytes(H, E) <= kSmemBudget;
    return CShape<8, 16, 4, 4, false, 1>::smem_bytes(H, E) <= kSmemBudget;
}

}  // namespace

int route_variant(int32_t H, int32_t E, bool has_logits)
{
    const bool stream_fits = StreamShape::smem_bytes(H) <= kStreamBudget;
    if (E <= 8 && stream_fits) return MOE_ROUTER_STREAM;
    if (E > 8 && has_logits && E % 8 == 0 && stream_fits) return MOE_ROUTER_SLICED;
    if (cluster_fits(H, E)) return MOE_ROUTER_CLUSTER;
    return MOE_ROUTER_BLOCK;
}

cudaError_t launch_route(const RouteArgs& a, int num_sms, cudaStream_t s)
{
    if (a.T == 0) return cudaSuccess;
    cudaError_t err = cudaSuccess;
    const int variant = route_variant(a.H, a.E, a.logits != nullptr);
    // (launch_stream returns false only if a tensor map cannot be encoded;
    // then the block router below runs)
    if ((variant == MOE_ROUTER_STREAM || variant == MOE_ROUTER_SLICED) &&
        launch_stream<StreamShape>(a, num_sms, s, err))
        return err;
    if (variant == MOE_ROUTER_CLUSTER) {
        bool launched = false;
        if (a.E <= 16) err = launch_cluster_any<16, 1, 2, 1, 2>(a, num_sms, s, launched);
        else if (a.E <= 32) err = launch_cluster_any<16, 2, 4, 1, 2>(a, num_sms, s, launched);
        else err = launch_cluster_any<16, 4, 4, 1, 2>(a, num_sms, s, launched);
        if (launched) return err;
    }
    if (a.E <= 8) return launch_route_t<8, 4>(a, num_sms, s);
    if (a.E <= 16) return launch_route_t<16, 2>(a, num_sms, s);
    if (a.E <= 32) return launch_route_t<32, 2>(a, num_sms, s);
    return launch_route_t<64, 1>(a, num_sms, s);
}

// The shared expert's sigmoid gate: one warp per token, fp32 dot product (the
// lane sums and a butterfly; no integer depends on it), then 1/(1+exp(-d)).
__global__ void shared_gate_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ wsg,
                                   float* __restrict__ scale, int64_t T, int32_t H)
{
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < T; t += warps) {
        float d = 0.0f;
        for (int c = lane; c < H / 8; c += 32) {
            const uint4 xv = __ldg(reinterpret_cast<const uint4*>(x + t * H + 8 * c));
            const uint4 wv = __ldg(reinterpret_cast<const uint4*>(wsg + 8 * c));
            const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w}, ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                d = fmaf(bf16_lo(xw[u]), bf16_lo(ww[u]), d);
                d = fmaf(bf16_hi(xw[u]), bf16_hi(ww[u]), d);
            }
        }
#pragma unroll
        for (int st = 16; st >= 1; st >>= 1) d += __shfl_xor_sync(0xffffffffu, d, st);
        if (lane == 0) scale[t] = 1.0f / (1.0f + expf(-d));
    }
}

cudaError_t launch_shared_gate(const uint16_t* x, const uint16_t* wsg, float* scale, int64_t T,
                               int32_t H, int num_sms, cudaStream_t s)
{
    if (T == 0) return cudaSuccess;
    const int64_t blocks_needed = (T + 7) / 8;
    const int64_t cap = (int64_t)num_sms * 8;
    return launch_pdl(shared_gate_kernel, dim3((unsigned)(blocks_needed < cap ? blocks_needed : cap)), dim3(256), 0,
                      s, x, wsg, scale, T, H);
}

}  // namespace moe
