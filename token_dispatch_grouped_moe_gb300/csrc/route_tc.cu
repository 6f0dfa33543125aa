// route_tc.cu -- the router's gate GEMM on the tensor cores, with the expert
// ids still exactly those of the canonical fp32 order.
//
// The pages name top-k routing (DisagMoE summary, section 2.2) and give no
// kernel. The ids are defined by fp32 logits summed in the canonical order
// (include/moe.h): 8-element chunks, chunk c on lane c mod 32, fma in
// increasing h, then an xor butterfly over the 32 lane sums. That order costs
// H*E fp32 FMAs per token, which for E = 64 is far more than the HBM time of
// reading x. Here the logits are first computed on the tensor cores, and each
// token's selection is proven equal to the canonical one, or the token is
// recomputed in the canonical order:
//
//   1. route_tc_prep_kernel: the gate transposed to WgT[NP][H] (K-major rows
//      per expert, zero rows up to NP = E rounded up to 16) and the sums of
//      squares from which each column's 2-norm ||w_e|| follows, rounded up.
//   2. route_tc_kernel: per 128-token tile, TMA streams x and WgT through an
//      ring of 8 stages (4 when two CTAs share an SM); one thread issues tcgen05.mma (K = 16) into a fresh TMEM
//      partial [128 x NP] every 64 of H (one k-block, four MMAs). The
//      epilogue warps (one thread per token) add the partials in fp32 in k
//      order, the fast logit f_e, and read their token's row of each x tile
//      from shared memory for ||x_t||^2 (fp32, every step rounded upward).
//   3. The bound. With p_h = x_h w_he (exact in fp32) and S = sum_h p_h:
//        canonical:  |l - S| <= gamma(H/32 + 5) sum|p|        (fp32 RN)
//        fast:       |f - S| <= (4 u_mma + gamma(H/64)) sum|p|
//      where u_mma bounds one K = 16 tensor-core step relative to the
//      magnitudes it adds (|C| + sum |a_i b_i|): products exact, then at most
//      17 terms aligned and truncated to fp32, 2^-18 taken (twice the 17 *
//      2^-23 of that model; checked against exact sums on the GPU by a test).
//      sum|p| <= ||x_t|| ||w_e|| (Cauchy-Schwarz). So |f_e - l_e| <= B_t for
//      every expert, B_t from ||x_t|| and max_e ||w_e|| (plus the bias add).
//   4. The main kernel writes f (bias added) and B_t to the workspace.
//      route_tc_select_kernel (eight lanes per token) takes the top k+1 by
//      fast logit (ties to the lower id). If every consecutive gap among them
//      exceeds 2 B_t, the canonical logits have the same order there and
//      every other expert is below the k selected: the ids and ranks are the
//      canonical ones, and the weights are a softmax of the fast logits
//      (within the fp32 rounding of the canonical ones; weights are compared
//      with a tolerance).
//   5. Otherwise only the ambiguous runs are recomputed in the canonical order
//      (lane L = canonical lane L, fmaf in increasing h, the butterfly) by
//      the fix kernel (a warp per listed token, or below 8192 tokens a block
//      whose warps share its run members): the positions whose gap to a
//      neighbour is at most
//      2 B_t, the run at the k / k+1 boundary extended by every expert within
//      2 B_t below it (chained). Each run is more than 2 B_t away from every
//      other expert, so ordering run members by their canonical logits and
//      the others by their fast logits is the canonical order.
#include <cstdint>
#include <cstring>
#include <cmath>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/moe.h"
#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kTcTile = 128;      // tokens per tile (MMA M)
constexpr int kTcBK = 64;         // k-block (one 128-byte swizzle row of bf16)
constexpr int kTcStagesMax = 8;   // one CTA per SM: 8 stages; two CTAs per SM: 4 each
constexpr int kTcTmemCols = 256;  // up to two CTAs per SM share the 512 TMEM columns
constexpr int kTcThreads = 192;   // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int kTcABytes = kTcTile * kTcBK * 2;   // 16 KB
constexpr int kTcPartKB = 1;      // k-blocks per TMEM partial (4 MMAs of K = 16)
constexpr int kTcPrepRows = 64;   // gate rows per block of the prep kernel
constexpr int kSelectThreads = 128;   // the striding select kernel: 4 warps of 4 tokens per block
constexpr int kFixThreads = 128;      // the block fix kernel: 4 warps per listed token
// From this many tokens the select and fix steps take a warp per group and a
// warp per listed token (many listed tokens, short member lists); below, the
// striding select kernel and a block per listed token (measured on GB300,
// DeepSeek-shaped E = 64: T = 4096 route 44 -> 36 us, T = 32768 83 -> 110 us
// the other way round).
constexpr int64_t kTcManyTokens = 8192;

// A stage holds the x tile (128 token rows x 64 of H) and the gate tile (NP
// expert rows x 64 of H), both K-major in 128-byte-swizzled rows; one MMA per
// K = 16 step multiplies them into a TMEM partial of NP columns. A partial
// buffer is NP columns rounded up to a multiple of 32.
template <int NP>
struct TcCfg {
    static constexpr int B_BYTES = NP * kTcBK * 2;
    static constexpr int STAGE = kTcABytes + B_BYTES;   // a multiple of 1024
    static constexpr int PB_COLS = (NP + 31) / 32 * 32;
    static constexpr int NB = kTcTmemCols / PB_COLS > 8 ? 8 : kTcTmemCols / PB_COLS;
    static constexpr uint32_t IDESC = idesc_bf16_f32(kTcTile, NP, false, false);
    static_assert(STAGE % 1024 == 0, "stages stay 1024-byte aligned");
    static_assert(NB >= 2 && NB <= 8, "two to eight partial buffers");
};

struct TcSmem {
    uint64_t full[kTcStagesMax];
    uint64_t empty[kTcStagesMax];
    uint64_t pfull[8];
    uint64_t pempty[8];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
    float wmax;
};

template <int NP, int STAGES>
constexpr size_t tc_smem_bytes()
{
    return 1024 + (size_t)STAGES * TcCfg<NP>::STAGE + sizeof(TcSmem);
}

// 32 lanes x 16 columns of 32-bit TMEM cells (thread i: lane base + i).
__device__ __forceinline__ void tmem_ld_x16(uint32_t taddr, uint32_t* v)
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
          "=r"(v[14]), "=r"(v[15])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ float bf16f(uint16_t v) { return __uint_as_float((uint32_t)v << 16); }

// ------------------------------------------------------------------ prep --

// Block b: gate rows h in [64 b, 64 b + 64) (read contiguously), transposed
// through shared memory to WgT[e][h] (rows e >= E zero), and the sums of
// squares of those 64 values per expert, wpart[b][e], in fp32 rounded upward
// at every step (so never below the exact sum; added in h order, and the main
// kernel adds the blocks in b order: the same bits on every run). Block 0
// also zeroes the count of listed tokens.
__global__ void __launch_bounds__(256) route_tc_prep_kernel(const uint16_t* __restrict__ Wg, int32_t H, int32_t E,
                                                            int32_t NP, uint16_t* __restrict__ wgt,
                                                            float* __restrict__ wpart, int32_t* __restrict__ n_exact)
{
    pdl_wait();
    pdl_launch_dependents();
    __shared__ uint16_t tile[kTcPrepRows][64 + 2];
    const int h0 = blockIdx.x * kTcPrepRows;
    // 64 rows of E bf16 are contiguous: 8 at a time (E is a multiple of 8)
    const uint4* src = reinterpret_cast<const uint4*>(Wg + (int64_t)h0 * E);
    for (int i = threadIdx.x; i < kTcPrepRows * E / 8; i += blockDim.x) {
        const uint4 v = src[i];
        const int hh = (8 * i) / E, e = 8 * i - hh * E;
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            tile[hh][e + 2 * q] = (uint16_t)(w[q] & 0xFFFFu);
            tile[hh][e + 2 * q + 1] = (uint16_t)(w[q] >> 16);
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < kTcPrepRows * NP; i += blockDim.x) {
        const int e = i / kTcPrepRows, hh = i - e * kTcPrepRows;
        wgt[(int64_t)e * H + h0 + hh] = e < E ? tile[hh][e] : (uint16_t)0;
    }
    if (threadIdx.x < NP) {
        const int e = threadIdx.x;
        float ss = 0.0f;
        if (e < E)
            for (int hh = 0; hh < kTcPrepRows; ++hh) {
                const float f = bf16f(tile[hh][e]);
                ss = __fmaf_ru(f, f, ss);
            }
        wpart[(int64_t)blockIdx.x * NP + e] = ss;
    }
    if (blockIdx.x == 0 && threadIdx.x < 2) n_exact[threadIdx.x] = 0;   // listed tokens, listed pairs
}

// ------------------------------------------------------------------ main --

template <int NP, int kTcStages>
__global__ void __launch_bounds__(kTcThreads, 2)
route_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW, const RouteArgs a,
                const RouteTcArgs c)
{
    using C = TcCfg<NP>;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t tiles = (raw + 1023u) & ~1023u;
    TcSmem* st = reinterpret_cast<TcSmem*>(smem_raw + (tiles - raw) + (size_t)kTcStages * C::STAGE);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = a.E;
    const int n_kb = a.H / kTcBK;
    const int n_tiles = (int)((a.T + kTcTile - 1) / kTcTile);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kTcStages; ++s) {
            mbar_init(smem_u32(&st->full[s]), 1);
            // freed by the MMA's commit and by the four epilogue warps, which
            // read their token rows of x from the stage (||x_t||^2)
            mbar_init(smem_u32(&st->empty[s]), 5);
        }
        for (int b = 0; b < C::NB; ++b) {
            mbar_init(smem_u32(&st->pfull[b]), 1);
            mbar_init(smem_u32(&st->pempty[b]), 4);
        }
        mbar_init(smem_u32(&st->drain), 1);
        st->abort = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmW);
    }
    if (warp == 1) {
        tmem_alloc<1>(smem_u32(&st->tmem_base), kTcTmemCols);
        tmem_relinquish<1>();
    }
    pdl_wait();
    pdl_launch_dependents();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = st->tmem_base;
    volatile int* abort = &st->abort;

    if (warp == 0) {
        // ============================== TMA producer ==============================
        int stage = 0, issued = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
            for (int kb = 0; kb < n_kb; ++kb) {
                if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&st->empty[stage]), phase ^ 1u, abort, a.err))) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    const uint32_t full = smem_u32(&st->full[stage]);
                    const uint32_t dst = tiles + stage * C::STAGE;
                    mbar_arrive_expect_tx(full, C::STAGE);
                    tma_load_2d(dst, &tmX, kb * kTcBK, tile * kTcTile, full);
                    tma_load_2d(dst + kTcABytes, &tmW, kb * kTcBK, 0, full);
                }
                __syncwarp();
                ++issued;
                if (++stage == kTcStages) { stage = 0; phase ^= 1u; }
            }
        }
        if (!ok && lane == 0) {
            int s = stage;
            uint32_t ph = phase;
            for (int i = 0; i < min(issued, kTcStages); ++i) {
                if (s == 0) { s = kTcStages - 1; ph ^= 1u; } else { --s; }
                mbar_wait_drain(smem_u32(&st->full[s]), ph);
            }
        }
    } else if (warp == 1) {
        // ============================== MMA issuer ================================
        if (lane == 0) {
            int stage = 0, pb = 0;
            uint32_t phase = 0, pphase = 0;
            bool ok = true, any = false;
            for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
                for (int kb = 0; kb < n_kb; ++kb) {
                    const int in_part = kb % kTcPartKB;   // a partial starts afresh every kTcPartKB k-blocks
                    if (!mbar_wait(smem_u32(&st->full[stage]), phase, abort, a.err) ||
                        (in_part == 0 && !mbar_wait(smem_u32(&st->pempty[pb]), pphase ^ 1u, abort, a.err))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_base = tiles + stage * C::STAGE;
                    const uint32_t b_base = a_base + kTcABytes;
                    const uint32_t d = tmem + pb * C::PB_COLS;
                    const bool part_end = in_part == kTcPartKB - 1 || kb == n_kb - 1;
#pragma unroll
                    for (int kk = 0; kk < kTcBK / 16; ++kk) {
                        const uint64_t ad = smem_desc_sw128(a_base + kk * 32, 16, 1024);
                        const uint64_t bd = smem_desc_sw128(b_base + kk * 32, 16, 1024);
                        tc_mma_f16<1>(d, ad, bd, C::IDESC, (in_part | kk) != 0 ? 1u : 0u);
                    }
                    any = true;
                    tc_commit<1>(smem_u32(&st->empty[stage]));
                    if (part_end) tc_commit<1>(smem_u32(&st->pfull[pb]));
                    if (++stage == kTcStages) { stage = 0; phase ^= 1u; }
                    if (part_end && ++pb == C::NB) { pb = 0; pphase ^= 1u; }
                }
            }
            if (!ok && any) {
                tc_commit<1>(smem_u32(&st->drain));
                mbar_wait_drain(smem_u32(&st->drain), 0);
            }
        }
        __syncwarp();
    } else {
        // ============================== epilogue ==================================
        const int ew = warp & 3;   // TMEM lane quarter of this warp
        const int r = ew * 32 + lane;
        const uint32_t lane_off = (uint32_t)(ew * 32) << 16;
        if (warp == 2) {
            // the largest column norm of the gate: the prep kernel's per-block
            // sums of squares added in block order and the square root, all
            // rounded upward (an upper bound); computed while the first tile
            // streams in, shared with the other epilogue warps by a named barrier
            const int nblk = a.H / kTcPrepRows;
            float m = 0.0f;
            for (int e = lane; e < E; e += 32) {
                float ss = 0.0f;
                for (int b = 0; b < nblk; ++b) ss = __fadd_ru(ss, c.wpart[(int64_t)b * NP + e]);
                m = fmaxf(m, __fsqrt_ru(ss));
            }
            for (int sh = 16; sh > 0; sh >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, sh));
            if (lane == 0) st->wmax = m;
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");   // the four epilogue warps
        const float wmax = st->wmax;
        const int n_part = (n_kb + kTcPartKB - 1) / kTcPartKB;
        int pb = 0, xstage = 0;
        uint32_t pphase = 0, xphase = 0;
        const unsigned char* tiles_ptr = smem_raw + (tiles - raw);
        for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
            float s[NP];
#pragma unroll
            for (int e = 0; e < NP; ++e) s[e] = 0.0f;
            float sumsq = 0.0f;
            bool ok = true;
            for (int q = 0; q < n_part; ++q) {
                // this thread's token row of the stage's x tile: ||x_t||^2 in
                // fp32 with every step rounded upward (never below the exact sum)
                for (int u = 0; u < kTcPartKB; ++u) {
                    if (q * kTcPartKB + u >= n_kb) break;
                    if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&st->full[xstage]), xphase, abort, a.err))) {
                        ok = false;
                        break;
                    }
                    const unsigned char* row = tiles_ptr + (size_t)xstage * C::STAGE + r * 128;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint4 v = *reinterpret_cast<const uint4*>(row + ((j ^ (r & 7)) << 4));
                        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            const float lo = __uint_as_float(w4[h] << 16), hi = __uint_as_float(w4[h] & 0xFFFF0000u);
                            sumsq = __fmaf_ru(lo, lo, sumsq);
                            sumsq = __fmaf_ru(hi, hi, sumsq);
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&st->empty[xstage]));
                    if (++xstage == kTcStages) { xstage = 0; xphase ^= 1u; }
                }
                if (!ok) break;
                if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&st->pfull[pb]), pphase, abort, a.err))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t src = tmem + lane_off + pb * C::PB_COLS;
                uint32_t v[NP];
#pragma unroll
                for (int u = 0; u + 32 <= NP; u += 32)
                    tmem_ld_32x32b_x32(src + u, *reinterpret_cast<uint32_t(*)[32]>(v + u));
                if (NP % 32) tmem_ld_x16(src + (NP / 32) * 32, v + (NP / 32) * 32);
                tc_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&st->pempty[pb]));
                // the fp32 sums of the partials, in k order
#pragma unroll
                for (int e = 0; e < NP; ++e) s[e] = s[e] + __uint_as_float(v[e]);
                if (++pb == C::NB) { pb = 0; pphase ^= 1u; }
            }
            if (!ok) break;
            const int64_t t = (int64_t)tile * kTcTile + r;
            if (t >= a.T) continue;
            // ||x_t|| rounded up, then B_t
            const float xnorm = __fsqrt_ru(sumsq);
            float fmax_abs = 0.0f;
            float4* dst = reinterpret_cast<float4*>(c.fast + t * E);   // E % 8 == 0: 32-byte aligned rows
#pragma unroll
            for (int e = 0; e < NP; e += 4) {
                if (e >= E) break;
                float v[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    v[u] = s[e + u];
                    if (a.bias) v[u] = v[u] + a.bias[e + u];
                    fmax_abs = fmaxf(fmax_abs, fabsf(v[u]));
                }
                dst[e / 4] = make_float4(v[0], v[1], v[2], v[3]);
            }
            float bnd = c.c_tot * xnorm * wmax * (1.0f + 0x1p-16f);
            // the bias add on either side rounds once more
            if (a.bias) bnd = bnd + 0x1p-22f * (fmax_abs + bnd);
            c.bound[t] = bnd;
            if (c.dbg_fast) {
#pragma unroll
                for (int e = 0; e < NP; ++e)
                    if (e < E) c.dbg_fast[t * E + e] = s[e];
                c.dbg_bound[t] = c.c_fast * xnorm * wmax;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<1>(tmem, kTcTmemCols);
    }
}

// ---------------------------------------------------------------- select --

// The canonical logits of experts e0 and e1 (e1 < 0: none) for one token,
// computed by the whole warp: lane L is canonical lane L, taking its chunks
// c = L, L + 32, ... in increasing order, fmaf in increasing h, then the xor
// butterfly; loads for eight chunks of both experts issued together.
__device__ __forceinline__ void canonical_pair(const uint16_t* xrow, const uint16_t* wgt, int H, int e0, int e1,
                                               int lane, float& l0, float& l1)
{
    const uint4* xr = reinterpret_cast<const uint4*>(xrow);
    const uint4* w0 = reinterpret_cast<const uint4*>(wgt + (int64_t)e0 * H);
    const uint4* w1 = reinterpret_cast<const uint4*>(wgt + (int64_t)(e1 < 0 ? e0 : e1) * H);
    const int n_ch = H / 8;
    float a0 = 0.0f, a1 = 0.0f;
    for (int c0 = lane; c0 < n_ch; c0 += 32 * 8) {
        uint4 xv[8], v0[8], v1[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const int ch = c0 + 32 * m;
            if (ch < n_ch) {
                xv[m] = xr[ch];
                v0[m] = w0[ch];
                v1[m] = w1[ch];
            }
        }
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            if (c0 + 32 * m >= n_ch) break;
            const uint32_t xs[4] = {xv[m].x, xv[m].y, xv[m].z, xv[m].w};
            const uint32_t p0[4] = {v0[m].x, v0[m].y, v0[m].z, v0[m].w};
            const uint32_t p1[4] = {v1[m].x, v1[m].y, v1[m].z, v1[m].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float xl = __uint_as_float(xs[q] << 16), xh = __uint_as_float(xs[q] & 0xFFFF0000u);
                a0 = __fmaf_rn(xl, __uint_as_float(p0[q] << 16), a0);
                a0 = __fmaf_rn(xh, __uint_as_float(p0[q] & 0xFFFF0000u), a0);
                a1 = __fmaf_rn(xl, __uint_as_float(p1[q] << 16), a1);
                a1 = __fmaf_rn(xh, __uint_as_float(p1[q] & 0xFFFF0000u), a1);
            }
        }
    }
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) {
        a0 = a0 + __shfl_xor_sync(0xffffffffu, a0, s);
        a1 = a1 + __shfl_xor_sync(0xffffffffu, a1, s);
    }
    l0 = a0;
    l1 = a1;
}

// Eight lanes per token (four tokens per warp), lane r holding the fast
// logits of experts r*E/8 .. (r+1)*E/8 - 1. The top k+1 by fast logit (ties to
// the lower id), then the proof: every consecutive gap among them above 2 B_t.
// Proven tokens are written at once. For the others, the ambiguous runs
// (positions whose gap to a neighbour is at most 2 B_t; the run at the k/k+1
// boundary extended by every expert within 2 B_t below it, chained) are
// recomputed in the canonical order by the whole warp, and the final order
// takes the canonical logit of every run member and the fast logit of every
// other expert: each run is separated from the rest by more than 2 B_t, so
// this order is the canonical one.
template <int PMAX>
__device__ __forceinline__ void select_group(const RouteArgs& a, const RouteTcArgs& c, int64_t grp)
{
    const int lane = threadIdx.x & 31;
    const int r = lane & 7, sub = lane >> 3;
    const int E = a.E, k = a.k;
    const int per = E >> 3;
    const int64_t t = grp * 4 + sub;
    const bool live = t < a.T;
    const int e_lo = r * per;
    const unsigned gmask = 0xFFu << (8 * sub);
    float lv[PMAX];
#pragma unroll
    for (int u = 0; u < PMAX; ++u) lv[u] = (live && u < per) ? c.fast[t * E + e_lo + u] : 0.0f;
    const float B = live ? c.bound[t] : 0.0f;
    const float B2 = 2.0f * B;
    const int kk1 = k < E ? k + 1 : E;
    uint32_t taken = 0;
    int sel[9];
    float selv[9];
#pragma unroll
    for (int j = 0; j < 9; ++j) {
        sel[j] = -1;
        selv[j] = 0.0f;
        if (j >= kk1) continue;
        float bv = 0.0f;
        int be = -1;
#pragma unroll
        for (int u = 0; u < PMAX; ++u)
            if (u < per && !((taken >> u) & 1u) && (be < 0 || lv[u] > bv)) { bv = lv[u]; be = e_lo + u; }
#pragma unroll
        for (int st = 1; st < 8; st <<= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, st);
            const int oe = __shfl_xor_sync(0xffffffffu, be, st);
            if (oe >= 0 && (be < 0 || ov > bv || (ov == bv && oe < be))) { bv = ov; be = oe; }
        }
        if (be >= e_lo && be < e_lo + per) taken |= 1u << (be - e_lo);
        sel[j] = be;
        selv[j] = bv;
    }
    // ambiguous gaps among the top k+1
    uint32_t amb = 0;   // bit j: gap between positions j and j+1 is at most 2 B_t
#pragma unroll
    for (int j = 0; j < 8; ++j)
        if (j + 1 < kk1 && !(selv[j] - selv[j + 1] > B2)) amb |= 1u << j;
    if (c.force_exact) amb = (1u << (kk1 - 1)) - 1u;
    const bool proven = live && amb == 0 && !c.force_exact;
    const float mx = selv[0];
    float den_all = 0.0f;
    if (!a.renorm) {
#pragma unroll
        for (int u = 0; u < PMAX; ++u)
            if (u < per) den_all = den_all + expf(lv[u] - mx);
#pragma unroll
        for (int st = 1; st < 8; st <<= 1) den_all = den_all + __shfl_xor_sync(0xffffffffu, den_all, st);
    }
    if (proven && r == 0) {
        float ex[8], den = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (j >= k) break;
            ex[j] = expf(selv[j] - mx);
            den = den + ex[j];
        }
        if (!a.renorm) den = den_all;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (j >= k) break;
            a.topk_idx[t * k + j] = sel[j];
            a.topk_w[t * k + j] = ex[j] / den;
        }
    }
    // the run members (a 64-bit mask of experts; positions of the top list
    // plus, for the boundary run, the chained experts below it)
    uint64_t cand = 0;
    bool need = live && (amb != 0 || c.force_exact);
    if (need) {
#pragma unroll
        for (int j = 0; j < 9; ++j)
            if (j < kk1 && (((amb >> j) & 1u) || (j > 0 && ((amb >> (j - 1)) & 1u)))) cand |= 1ull << sel[j];
        if (c.force_exact || !a.renorm)
            cand = E == 64 ? ~0ull : ((1ull << E) - 1ull);
        else if (k < E && ((amb >> (k - 1)) & 1u)) {
            // the boundary run goes below position k: chain downwards
            float lo = selv[k];
            for (int it = 0; it < 64; ++it) {
                uint32_t add = 0;
                float nlo = lo;
#pragma unroll
                for (int u = 0; u < PMAX; ++u)
                    if (u < per && !((taken >> u) & 1u) && !((cand >> (e_lo + u)) & 1ull) && lv[u] >= lo - B2) {
                        add |= 1u << u;
                        nlo = fminf(nlo, lv[u]);
                    }
                uint64_t m = 0;
#pragma unroll
                for (int u = 0; u < PMAX; ++u)
                    if ((add >> u) & 1u) m |= 1ull << (e_lo + u);
#pragma unroll
                for (int st = 1; st < 8; st <<= 1) {
                    m |= ((uint64_t)__shfl_xor_sync(gmask, (uint32_t)(m >> 32), st) << 32) |
                         __shfl_xor_sync(gmask, (uint32_t)m, st);
                    nlo = fminf(nlo, __shfl_xor_sync(gmask, nlo, st));
                }
                if (m == 0) break;
                cand |= m;
                lo = nlo;
            }
        }
    }
    // list the token: its runs and its top list, for the fix kernel
    if (need && r == 0) {
        const int slot = atomicAdd(c.n_exact, 1);
        c.flag_tok[slot] = (int32_t)t;
        c.flag_cand[slot] = cand;
#pragma unroll
        for (int j = 0; j < 9; ++j) {
            c.flag_sel[(int64_t)slot * 9 + j] = sel[j];
            c.flag_selv[(int64_t)slot * 9 + j] = selv[j];
        }
        if (c.pairs) {
            // its (token, member pair) work items for the pairs kernel
            const int np = (__popcll((long long)cand) + 1) >> 1;
            const int pb = atomicAdd(c.n_exact + 1, np);
            for (int q = 0; q < np; ++q) c.pairs[pb + q] = slot * 32 + q;
        }
    }
}

// Four tokens per warp (select_group), one group per warp: from 8192 tokens.
template <int PMAX>
__global__ void __launch_bounds__(256) route_tc_select_kernel(const RouteArgs a, const RouteTcArgs c)
{
    pdl_wait();
    pdl_launch_dependents();
    select_group<PMAX>(a, c, (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5));
}

// Below 8192 tokens: the warps of a grid sized to the resident blocks stride
// over the groups, so the selection runs in one wave.
template <int PMAX>
__global__ void __launch_bounds__(kSelectThreads) route_tc_select_stride_kernel(const RouteArgs a,
                                                                                const RouteTcArgs c)
{
    pdl_wait();
    pdl_launch_dependents();
    const int64_t n_groups = (a.T + 3) / 4;
    const int64_t warps = (int64_t)gridDim.x * (kSelectThreads / 32);
    for (int64_t grp = (int64_t)blockIdx.x * (kSelectThreads / 32) + (threadIdx.x >> 5); grp < n_groups; grp += warps)
        select_group<PMAX>(a, c, grp);
}

// The final order of one recomputed token (one thread): the top list (ids,
// fast logits; the run members among them take their canonical logits from
// lg) and the run members below it (canonical logits), ties to the lower id;
// writes the k ids and weights (without renormalisation every expert is a
// run member, so the denominator runs over canonical logits throughout).
__device__ __forceinline__ void order_token(const RouteArgs& a, int64_t t, uint64_t cm, const int* id0,
                                            const float* key0, int kk1, const float* lg)
{
    const int E = a.E, k = a.k;
    float key[9];
    int id[9];
    for (int j = 0; j < kk1; ++j) {
        id[j] = id0[j];
        key[j] = key0[j];
    }
    uint64_t extra = cm;
    for (int j = 0; j < kk1; ++j) {
        if ((cm >> id[j]) & 1ull) key[j] = lg[id[j]];
        extra &= ~(1ull << id[j]);
    }
    int osel[8];
    float ov[8];
    uint32_t used = 0;
    uint64_t used_x = 0;
    for (int j = 0; j < k; ++j) {
        float bv = 0.0f;
        int be = -1, bi = -1;
        for (int q = 0; q < kk1; ++q)
            if (!((used >> q) & 1u) && (be < 0 || key[q] > bv || (key[q] == bv && id[q] < be))) {
                bv = key[q];
                be = id[q];
                bi = q;
            }
        uint64_t rx = extra & ~used_x;
        while (rx) {
            const int e = __ffsll((long long)rx) - 1;
            rx &= rx - 1;
            if (be < 0 || lg[e] > bv || (lg[e] == bv && e < be)) {
                bv = lg[e];
                be = e;
                bi = 64 + e;
            }
        }
        if (bi >= 64) used_x |= 1ull << (bi - 64); else used |= 1u << bi;
        osel[j] = be;
        ov[j] = bv;
    }
    const float m0 = ov[0];
    float ex[8], den = 0.0f;
    for (int j = 0; j < k; ++j) {
        ex[j] = expf(ov[j] - m0);
        den = den + ex[j];
    }
    if (!a.renorm) {
        den = 0.0f;
        for (int e = 0; e < E; ++e) den = den + expf(lg[e] - m0);
    }
    for (int j = 0; j < k; ++j) {
        a.topk_idx[t * k + j] = osel[j];
        a.topk_w[t * k + j] = ex[j] / den;
    }
}

// Below 8192 tokens, a block per listed token: its warps share the run
// members (warp w takes the pairs w, w + 4, ... of the member list; each
// pair's canonical logits by the whole warp, two experts per pass), then
// thread 0 orders the top list and the run members below it (canonical
// logits for run members, fast logits otherwise) and writes the k ids and
// weights. A token's members thus cost about one pass, not one per pair.
__global__ void __launch_bounds__(kFixThreads) route_tc_fix_block_kernel(const RouteArgs a, const RouteTcArgs c)
{
    pdl_wait();
    pdl_launch_dependents();
    __shared__ float lg[64];
    __shared__ int mem_s[64];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = *c.n_exact;
    const int E = a.E, k = a.k;
    const int kk1 = k < E ? k + 1 : E;
    for (int i = blockIdx.x; i < n; i += gridDim.x) {
        const int64_t t = c.flag_tok[i];
        const uint64_t cm = c.flag_cand[i];
        // the members in increasing id order
        int n_mem = 0;
        if (threadIdx.x == 0) {
            uint64_t rest = cm;
            while (rest) {
                mem_s[n_mem++] = __ffsll((long long)rest) - 1;
                rest &= rest - 1;
            }
        }
        n_mem = __popcll((long long)cm);
        __syncthreads();
        const uint16_t* xrow = a.x + t * a.H;
        for (int q = 2 * warp; q < n_mem; q += 2 * (kFixThreads / 32)) {
            const int e0 = mem_s[q];
            const int e1 = q + 1 < n_mem ? mem_s[q + 1] : -1;
            float l0, l1;
            canonical_pair(xrow, c.wgt, a.H, e0, e1, lane, l0, l1);
            if (lane == 0) {
                lg[e0] = a.bias ? l0 + a.bias[e0] : l0;
                if (e1 >= 0) lg[e1] = a.bias ? l1 + a.bias[e1] : l1;
            }
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            float key[9];
            int id[9];
            for (int j = 0; j < kk1; ++j) {
                id[j] = c.flag_sel[(int64_t)i * 9 + j];
                key[j] = c.flag_selv[(int64_t)i * 9 + j];
            }
            uint64_t extra = cm;
            for (int j = 0; j < kk1; ++j) {
                if ((cm >> id[j]) & 1ull) key[j] = lg[id[j]];
                extra &= ~(1ull << id[j]);
            }
            int osel[8];
            float ov[8];
            uint32_t used = 0;
            uint64_t used_x = 0;
            for (int j = 0; j < k; ++j) {
                float bv = 0.0f;
                int be = -1, bi = -1;
                for (int q = 0; q < kk1; ++q)
                    if (!((used >> q) & 1u) && (be < 0 || key[q] > bv || (key[q] == bv && id[q] < be))) {
                        bv = key[q];
                        be = id[q];
                        bi = q;
                    }
                uint64_t rx = extra & ~used_x;
                while (rx) {
                    const int e = __ffsll((long long)rx) - 1;
                    rx &= rx - 1;
                    if (be < 0 || lg[e] > bv || (lg[e] == bv && e < be)) {
                        bv = lg[e];
                        be = e;
                        bi = 64 + e;
                    }
                }
                if (bi >= 64) used_x |= 1ull << (bi - 64); else used |= 1u << bi;
                osel[j] = be;
                ov[j] = bv;
            }
            const float m0 = ov[0];
            float ex[8], den = 0.0f;
            for (int j = 0; j < k; ++j) {
                ex[j] = expf(ov[j] - m0);
                den = den + ex[j];
            }
            if (!a.renorm) {
                // every expert is a run member here: canonical logits throughout
                den = 0.0f;
                for (int e = 0; e < E; ++e) den = den + expf(lg[e] - m0);
            }
            for (int j = 0; j < k; ++j) {
                a.topk_idx[t * k + j] = osel[j];
                a.topk_w[t * k + j] = ex[j] / den;
            }
        }
        __syncthreads();
    }
}

// From 8192 tokens the fix step is balanced over (listed token, pair of run
// members) work items, which the select kernel lists: a warp per item
// computes the pair's canonical logits into lg_buf[token slot][expert], so a
// token with a long member list spreads over several warps; then
// route_tc_order_kernel finishes each token.
__global__ void __launch_bounds__(256) route_tc_pairs_kernel(const RouteArgs a, const RouteTcArgs c)
{
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int n_pairs = c.n_exact[1];
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); w < n_pairs; w += warps) {
        const int ent = c.pairs[w];
        const int i = ent >> 5, q = ent & 31;   // token slot, pair of its members
        const int64_t t = c.flag_tok[i];
        uint64_t m = c.flag_cand[i];
        for (int u = 0; u < 2 * q; ++u) m &= m - 1;   // drop the members of the pairs before
        const int e0 = __ffsll((long long)m) - 1;
        m &= m - 1;
        const int e1 = m ? __ffsll((long long)m) - 1 : -1;
        float l0, l1;
        canonical_pair(a.x + t * a.H, c.wgt, a.H, e0, e1, lane, l0, l1);
        if (lane == 0) {
            float* lg = c.lg_buf + (int64_t)i * 64;
            lg[e0] = a.bias ? l0 + a.bias[e0] : l0;
            if (e1 >= 0) lg[e1] = a.bias ? l1 + a.bias[e1] : l1;
        }
    }
}

// A thread per listed token: its final order from the pairs kernel's logits.
// Token i goes to block i mod gridDim.x, so a few thousand tokens spread over
// every SM (the work per token is a short serial chain of dependent loads).
__global__ void __launch_bounds__(64) route_tc_order_kernel(const RouteArgs a, const RouteTcArgs c)
{
    pdl_wait();
    pdl_launch_dependents();
    const int n = c.n_exact[0];
    const int kk1 = a.k < a.E ? a.k + 1 : a.E;
    for (int64_t i = blockIdx.x + (int64_t)gridDim.x * threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        order_token(a, c.flag_tok[i], c.flag_cand[i], c.flag_sel + i * 9, c.flag_selv + i * 9, kk1,
                    c.lg_buf + i * 64);
}

// The fast-path constants: c_fast bounds |f - S| and c_tot |f - l| per unit
// of ||x_t|| ||w_e|| (see the file comment), rounded up.
void tc_constants(int32_t H, RouteTcArgs* c)
{
    const double u = std::ldexp(1.0, -24);
    const double u_mma = std::ldexp(1.0, -18);
    auto gamma = [&](double n) { return n * u / (1.0 - n * u); };
    const double n_kb = H / (double)kTcBK;
    const double n_part = std::ceil(n_kb / kTcPartKB);
    const double steps = 4.0 * kTcPartKB;   // K = 16 MMA steps in one partial
    const double chain = steps * u_mma * (1.0 + 1e-3);
    const double cf = chain + gamma(n_part) * (1.0 + chain);
    const double cc = gamma(H / 32.0 + 5.0);
    c->c_fast = (float)(cf * (1.0 + 1e-6));
    c->c_tot = (float)((cf + cc) * (1.0 + 1e-6));
}

template <int NP, int STAGES>
cudaError_t launch_tc_s(const RouteArgs& a, const RouteTcArgs& c, const CUtensorMap& mx, const CUtensorMap& mw,
                        int grid, cudaStream_t s)
{
    constexpr size_t smem = tc_smem_bytes<NP, STAGES>();
    auto kern = route_tc_kernel<NP, STAGES>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    return launch_pdl(kern, dim3(grid), dim3(kTcThreads), smem, s, mx, mw, a, c);
}

// One CTA per 128-token tile: with at most one tile per SM, 8 stages in one
// CTA; with more tiles, two CTAs of 4 stages share an SM, so that every tile
// runs at once (measured: DeepSeek-shaped T = 32768, 256 tiles, main kernel
// 34 -> 28 us; T = 16384, 128 tiles, 8 stages 4 us faster than 4).
template <int NP>
cudaError_t launch_tc(const RouteArgs& a, const RouteTcArgs& c, int num_sms, cudaStream_t s)
{
    CUtensorMap mx, mw;
    if (!encode_map_2d(&mx, a.x, (uint64_t)a.H, (uint64_t)a.T, kTcBK, kTcTile, 128) ||
        !encode_map_2d(&mw, c.wgt, (uint64_t)a.H, (uint64_t)NP, kTcBK, NP, 128))
        return cudaErrorInvalidValue;
    const int64_t n_tiles = (a.T + kTcTile - 1) / kTcTile;
    if (n_tiles <= num_sms) return launch_tc_s<NP, 8>(a, c, mx, mw, (int)n_tiles, s);
    const int grid = (int)(n_tiles < 2 * num_sms ? n_tiles : 2 * num_sms);
    return launch_tc_s<NP, 4>(a, c, mx, mw, grid, s);
}

}  // namespace

bool route_tc_supported(int64_t T, int32_t H, int32_t E)
{
    return E >= 8 && E <= 64 && E % 8 == 0 && H % kTcBK == 0 && T >= kRouteTcMinTokens;
}

int route_tc_np(int32_t E) { return (E + 15) / 16 * 16; }

cudaError_t launch_route_tc(const RouteArgs& a, RouteTcArgs c, int num_sms, cudaStream_t s)
{
    if (a.T == 0) return cudaSuccess;
    const int NP = route_tc_np(a.E);
    tc_constants(a.H, &c);
    cudaError_t err = launch_pdl(route_tc_prep_kernel, dim3((unsigned)(a.H / kTcPrepRows)), dim3(256), 0, s, a.Wg,
                                 a.H, a.E, NP, c.wgt, c.wpart, c.n_exact);
    if (err != cudaSuccess) return err;
    if (NP == 16) err = launch_tc<16>(a, c, num_sms, s);
    else if (NP == 32) err = launch_tc<32>(a, c, num_sms, s);
    else if (NP == 48) err = launch_tc<48>(a, c, num_sms, s);
    else if (NP == 64) err = launch_tc<64>(a, c, num_sms, s);
    else return cudaErrorInvalidValue;
    if (err != cudaSuccess) return err;
    if (a.T < kTcManyTokens) c.pairs = nullptr;   // the block fix kernel takes whole tokens
    if (a.T >= kTcManyTokens) {
        // many tokens: a warp per 4-token group (which lists the recomputed
        // tokens' member pairs), a warp per listed pair, a thread per listed token
        const dim3 blocks((unsigned)((a.T + 31) / 32));   // 8 warps x 4 tokens
        err = a.E <= 32 ? launch_pdl(route_tc_select_kernel<4>, blocks, dim3(256), 0, s, a, c)
                        : launch_pdl(route_tc_select_kernel<8>, blocks, dim3(256), 0, s, a, c);
        if (err != cudaSuccess) return err;
        err = launch_pdl(route_tc_pairs_kernel, dim3((unsigned)(8 * num_sms)), dim3(256), 0, s, a, c);
        if (err != cudaSuccess) return err;
        return launch_pdl(route_tc_order_kernel, dim3((unsigned)(8 * num_sms)), dim3(64), 0, s, a, c);
    }
    // fewer: the resident blocks stride over the groups (one wave), then a
    // block per listed token
    auto sel = a.E <= 32 ? route_tc_select_stride_kernel<4> : route_tc_select_stride_kernel<8>;
    int per_sm = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, sel, kSelectThreads, 0);
    if (err != cudaSuccess) return err;
    const int64_t need = (a.T + 4 * (kSelectThreads / 32) - 1) / (4 * (kSelectThreads / 32));
    const int64_t resident = (int64_t)num_sms * (per_sm > 0 ? per_sm : 1);
    err = launch_pdl(sel, dim3((unsigned)(need < resident ? need : resident)), dim3(kSelectThreads), 0, s, a, c);
    if (err != cudaSuccess) return err;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, route_tc_fix_block_kernel, kFixThreads, 0);
    if (err != cudaSuccess) return err;
    return launch_pdl(route_tc_fix_block_kernel, dim3((unsigned)(num_sms * (per_sm > 0 ? per_sm : 1))),
                      dim3(kFixThreads), 0, s, a, c);
}

}  // namespace moe
