// permute.cu -- dispatch: a deterministic, stable counting sort of the
// R = T*k routed assignments by expert, plus the GEMM tile table.
//
// "Dispatch" is the step that sends each token to its k experts (DisagMoE
// summary, section 2.2). On one GPU it is an index permutation: positions
// p = offsets[e] .. offsets[e+1]-1 hold, in increasing f, the assignments
// f = t*k + j routed to expert e. Only integer work: the result is bit-exact.
//
// Two phases over fixed chunks of f (kChunk assignments per block):
//   1. histogram: per-chunk expert counts -> hist[chunk][e];
//   2. scatter: each block reads the whole (small) hist table to get the
//      global counts, the exclusive scan over experts and the count of each
//      expert in earlier chunks; then it ranks its own assignments stably
//      (warp match + per-warp counts in warp order) and writes src_row and
//      inv_pos. Block 0 also writes counts, offsets and the tile table.
// No float arithmetic and no order-dependent atomics: the integer atomics in
// the histogram only count. While every chunk's block fits on the GPU at once
// both phases run in one cooperative launch with a grid barrier between them
// (one launch fewer on the path); larger inputs take two launches.
#include <cooperative_groups.h>
#include <cstdint>
#include <cuda_runtime.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kChunk = 2048;
constexpr int kHistThreads = 256;
constexpr int kScatterThreads = 1024;
constexpr int kScatterWarps = kScatterThreads / 32;
constexpr int kMaxE = 256;

// Phase 1 for this block's chunk (any block size).
__device__ __forceinline__ void hist_body(const PermuteArgs& a)
{
    __shared__ int hist_s[kMaxE];
    for (int e = threadIdx.x; e < a.E; e += blockDim.x) hist_s[e] = 0;
    __syncthreads();
    const int64_t f0 = (int64_t)blockIdx.x * kChunk;
    const int64_t f1 = min(f0 + kChunk, a.R);
    for (int64_t f = f0 + threadIdx.x; f < f1; f += blockDim.x) {
        const int id = a.topk_idx[f];
        if (id >= 0 && id < a.E)
            atomicAdd(&hist_s[id], 1);
        else
            report_error(a.err, MOE_DEV_ERR_BAD_EXPERT);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < a.E; e += blockDim.x)
        a.hist[(int64_t)blockIdx.x * a.E + e] = hist_s[e];
}

__global__ void __launch_bounds__(kHistThreads) perm_hist_kernel(PermuteArgs a)
{
    pdl_wait();
    pdl_launch_dependents();
    hist_body(a);
}

// Exclusive scan of vals[0..n) in place by warp 0 (n <= 256); returns total.
__device__ int warp0_exclusive_scan(int* vals, int n)
{
    __shared__ int total_s;
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        const int per = (n + 31) / 32;
        const int b = lane * per;
        int local = 0;
        for (int i = 0; i < per; ++i)
            if (b + i < n) local += vals[b + i];
        int incl = local;
#pragma unroll
        for (int s = 1; s < 32; s <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, incl, s);
            if (lane >= s) incl += o;
        }
        int run = incl - local;
        for (int i = 0; i < per; ++i)
            if (b + i < n) {
                const int v = vals[b + i];
                vals[b + i] = run;
                run += v;
            }
        if (lane == 31) total_s = incl;
    }
    __syncthreads();
    const int total = total_s;
    __syncthreads();   // total_s may be rewritten by the next call
    return total;
}

// Phase 2 for this block's chunk (kScatterThreads threads).
__device__ __forceinline__ void scatter_body(const PermuteArgs& a, int n_chunks)
{
    __shared__ int total_s[kMaxE];
    __shared__ int base_s[kMaxE];      // next free position of each expert for this block
    __shared__ int tiles_s[kMaxE];
    __shared__ int wc_s[kScatterWarps][kMaxE];   // per-warp expert counts of one round
    const int E = a.E;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // 1. global totals and this block's per-expert start, from the hist table
    {
        const int subs = kScatterThreads / E >= 1 ? kScatterThreads / E : 1;
        int* part_tot = &wc_s[0][0];                 // reuse as scratch [subs][E] (fits: subs*E <= 1024*... )
        int* part_before = &wc_s[0][0] + (kScatterWarps * kMaxE) / 2;
        for (int i = tid; i < subs * E; i += blockDim.x) {
            const int e = i % E, sub = i / E;
            int tot = 0, before = 0;
            for (int c = sub; c < n_chunks; c += subs) {
                const int v = a.hist[(int64_t)c * E + e];
                tot += v;
                if (c < (int)blockIdx.x) before += v;
            }
            part_tot[i] = tot;
            part_before[i] = before;
        }
        __syncthreads();
        for (int e = tid; e < E; e += blockDim.x) {
            int tot = 0, before = 0;
            for (int sub = 0; sub < subs; ++sub) {
                tot += part_tot[sub * E + e];
                before += part_before[sub * E + e];
            }
            total_s[e] = tot;
            base_s[e] = before;
            tiles_s[e] = (tot + kTileM - 1) / kTileM;
        }
        __syncthreads();
    }
    if (blockIdx.x == 0)
        for (int e = tid; e < E; e += blockDim.x) a.counts[e] = total_s[e];
    __syncthreads();
    const int R_valid = warp0_exclusive_scan(total_s, E);   // total_s := offsets
    const int n_tiles = warp0_exclusive_scan(tiles_s, E);   // tiles_s := tile_start
    for (int e = tid; e < E; e += blockDim.x) base_s[e] += total_s[e];
    if (blockIdx.x == 0) {
        for (int e = tid; e < E; e += blockDim.x) {
            a.offsets[e] = total_s[e];
            a.tile_start[e] = tiles_s[e];
        }
        if (tid == 0) {
            a.offsets[E] = R_valid;
            a.tile_start[E] = n_tiles;
        }
    }
    for (int i = tid; i < kScatterWarps * kMaxE; i += blockDim.x) (&wc_s[0][0])[i] = 0;
    __syncthreads();

    // 2. stable ranks inside this block's chunk, one round of 1024 f at a time
    const int64_t f0 = (int64_t)blockIdx.x * kChunk;
    const int64_t f1 = min(f0 + kChunk, a.R);
    for (int64_t fr = f0; fr < f1; fr += kScatterThreads) {
        const int64_t f = fr + tid;
        int id = -1;
        if (f < f1) {
            id = a.topk_idx[f];
            if (id < 0 || id >= E) id = -1;   // reported by the histogram kernel
        }
        const unsigned peers = __match_any_sync(0xffffffffu, id);
        const int leader = __ffs(peers) - 1;
        const int lane_rank = __popc(peers & ((1u << lane) - 1u));
        if (id >= 0 && lane == leader) wc_s[warp][id] = __popc(peers);
        __syncthreads();
        int warp_before = 0;
        if (id >= 0 && lane == leader)
            for (int w = 0; w < warp; ++w) warp_before += wc_s[w][id];
        warp_before = __shfl_sync(0xffffffffu, warp_before, leader);
        if (id >= 0) {
            const int p = base_s[id] + warp_before + lane_rank;
            a.src_row[p] = (int32_t)f;
            a.inv_pos[f] = p;
        }
        __syncthreads();
        for (int e = tid; e < E; e += blockDim.x) {
            int s = 0;
            for (int w = 0; w < kScatterWarps; ++w) s += wc_s[w][e];
            base_s[e] += s;
        }
        __syncthreads();
        if (id >= 0 && lane == leader) wc_s[warp][id] = 0;
        __syncthreads();
    }
}

__global__ void __launch_bounds__(kScatterThreads) perm_scatter_kernel(PermuteArgs a, int n_chunks)
{
    pdl_wait();
    pdl_launch_dependents();
    scatter_body(a, n_chunks);
}

// Both phases; launched cooperatively (all blocks resident) so the grid
// barrier between them completes.
__global__ void __launch_bounds__(kScatterThreads) perm_fused_kernel(PermuteArgs a, int n_chunks)
{
    pdl_launch_dependents();   // (a cooperative launch: it starts after the kernel before it)
    hist_body(a);
    __threadfence();
    cooperative_groups::this_grid().sync();
    scatter_body(a, n_chunks);
}

// x_perm[p] = x[src_row[p] / k] for p < offsets[E] (the valid positions;
// fewer than R only if some expert ids were out of range). src_row null means
// the identity (f = p); r_valid null means all R rows. One warp per row,
// 16-byte loads and stores: an HBM-bound copy.
__global__ void gather_rows_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ src_row,
                                   const int32_t* __restrict__ r_valid, uint16_t* __restrict__ x_perm,
                                   int64_t R, int64_t T, int32_t H, int32_t k, uint32_t* err)
{
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int vec_per_row = H / 8;
    const int64_t n = r_valid ? min((int64_t)*r_valid, R) : R;
    for (int64_t p = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); p < n; p += warps) {
        const int64_t t = (src_row ? (int64_t)src_row[p] : p) / k;
        if (t < 0 || t >= T) {
            if (lane == 0) report_error(err, MOE_DEV_ERR_BOUNDS);
            continue;
        }
        const uint4* src = reinterpret_cast<const uint4*>(x + t * H);
        uint4* dst = reinterpret_cast<uint4*>(x_perm + p * H);
        for (int v = lane; v < vec_per_row; v += 32) dst[v] = __ldg(src + v);
    }
}

// x_perm by token: a warp per token reads its row of x once and writes it to
// the token's k dispatch positions (inv_pos[t*k + j], for the valid ids), 4 KB
// of the row at a time in registers. Every x_perm row p < *r_valid is the
// position of exactly one valid assignment, so each is written once, with the
// same bytes as the gather by src_row; x is read once instead of k times.
__global__ void __launch_bounds__(256) scatter_rows_kernel(const uint16_t* __restrict__ x,
                                                           const int32_t* __restrict__ topk_idx,
                                                           const int32_t* __restrict__ inv_pos,
                                                           const int32_t* __restrict__ r_valid,
                                                           uint16_t* __restrict__ x_perm, int64_t T, int32_t H,
                                                           int32_t k, int32_t E, uint32_t* err)
{
    pdl_wait();
    pdl_launch_dependents();
    constexpr int U = 8;   // 16-byte words a lane holds: 4 KB of the row per pass
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int vec_per_row = H / 8;
    const int64_t n_valid = *r_valid;
    for (int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < T; t += warps) {
        // lane j < k: the position of assignment j of this token, or -1
        int p = -1;
        if (lane < k) {
            const int id = topk_idx[t * k + lane];
            if (id >= 0 && id < E) {
                p = inv_pos[t * k + lane];
                if (p < 0 || p >= n_valid) {
                    report_error(err, MOE_DEV_ERR_BOUNDS);
                    p = -1;
                }
            }
        }
        const uint4* src = reinterpret_cast<const uint4*>(x + t * H);
        for (int v0 = 0; v0 < vec_per_row; v0 += 32 * U) {
            uint4 r[U];
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (v0 + 32 * u + lane < vec_per_row) r[u] = __ldg(src + v0 + 32 * u + lane);
            for (int j = 0; j < k; ++j) {
                const int pj = __shfl_sync(0xffffffffu, p, j);
                if (pj < 0) continue;
                uint4* dst = reinterpret_cast<uint4*>(x_perm + (int64_t)pj * H);
#pragma unroll
                for (int u = 0; u < U; ++u)
                    if (v0 + 32 * u + lane < vec_per_row) dst[v0 + 32 * u + lane] = r[u];
            }
        }
    }
}

__global__ void tile_table_kernel(const int32_t* __restrict__ offsets, int32_t G,
                                  int32_t* __restrict__ tile_start)
{
    __shared__ int tiles_s[kMaxE];
    pdl_wait();
    pdl_launch_dependents();
    for (int g = threadIdx.x; g < G; g += blockDim.x)
        tiles_s[g] = (offsets[g + 1] - offsets[g] + kTileM - 1) / kTileM;
    __syncthreads();
    const int n = warp0_exclusive_scan(tiles_s, G);
    for (int g = threadIdx.x; g < G; g += blockDim.x) tile_start[g] = tiles_s[g];
    if (threadIdx.x == 0) tile_start[G] = n;
}

}  // namespace

int permute_num_chunks(int64_t R) { return (int)((R + kChunk - 1) / kChunk); }

cudaError_t launch_permute(const PermuteArgs& a, cudaStream_t s)
{
    const int n = permute_num_chunks(a.R);
    if (n == 0) {
        // no assignments: zero counts/offsets/tile table via one tiny block
        return launch_pdl(perm_scatter_kernel, dim3(1), dim3(kScatterThreads), 0, s, a, 0);
    }
    // one cooperative launch while every chunk's block can be resident at once
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, perm_fused_kernel, kScatterThreads, 0) ==
            cudaSuccess &&
        n <= sms * per_sm) {
        PermuteArgs args = a;
        int n_chunks = n;
        void* params[] = {&args, &n_chunks};
        const cudaError_t e = cudaLaunchCooperativeKernel((const void*)perm_fused_kernel, dim3(n),
                                                          dim3(kScatterThreads), params, 0, s);
        if (e == cudaSuccess) count_launch();
        return e;
    }
    const cudaError_t err = launch_pdl(perm_hist_kernel, dim3(n), dim3(kHistThreads), 0, s, a);
    if (err != cudaSuccess) return err;
    return launch_pdl(perm_scatter_kernel, dim3(n), dim3(kScatterThreads), 0, s, a, n);
}

cudaError_t launch_gather_rows(const uint16_t* x, const int32_t* src_row, const int32_t* r_valid,
                               uint16_t* x_perm, int64_t R, int64_t T, int32_t H, int32_t k,
                               uint32_t* err, int num_sms, cudaStream_t s)
{
    if (R == 0) return cudaSuccess;
    const int64_t blocks_needed = (R + 7) / 8;
    const int grid = (int)(blocks_needed < (int64_t)num_sms * 8 ? blocks_needed : (int64_t)num_sms * 8);
    return launch_pdl(gather_rows_kernel, dim3(grid), dim3(256), 0, s, x, src_row, r_valid, x_perm, R, T, H, k,
                      err);
}

cudaError_t launch_scatter_rows(const uint16_t* x, const int32_t* topk_idx, const int32_t* inv_pos,
                                const int32_t* r_valid, uint16_t* x_perm, int64_t T, int32_t H, int32_t k,
                                int32_t E, uint32_t* err, int num_sms, cudaStream_t s)
{
    if (T == 0) return cudaSuccess;
    const int64_t blocks_needed = (T + 7) / 8;
    const int grid = (int)(blocks_needed < (int64_t)num_sms * 8 ? blocks_needed : (int64_t)num_sms * 8);
    return launch_pdl(scatter_rows_kernel, dim3(grid), dim3(256), 0, s, x, topk_idx, inv_pos, r_valid, x_perm, T,
                      H, k, E, err);
}

cudaError_t launch_tile_table(const int32_t* offsets, int32_t G, int32_t* tile_start, cudaStream_t s)
{
    return launch_pdl(tile_table_kernel, dim3(1), dim3(256), 0, s, offsets, G, tile_start);
}

}  // namespace moe
