// kernels.cuh -- launchers of the layer's kernels (host side), shared by the
// kernel files and the C ABI (api.cu). Internal to the library.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/moe.h"

namespace moe {

// The host checks of a moe_dims that every entry point shares (null, signs,
// k <= E, the supported sizes); MOE_OK or the status to return.
moe_status check_dims(const moe_dims* d);
// MOE_DEBUG=1 (read once): every entry point synchronises and checks.
bool debug_mode();

constexpr int kTileM = 128;   // GEMM M tile (routed rows per tile)
// GEMM K per pipeline stage: 64 bf16 (128-byte A rows, 128-byte swizzle, 4
// stages of 48 KB) or 32 (64-byte rows, 64-byte swizzle, 9 stages of 24 KB).
// 32 keeps more bytes in flight per SM but measured half the throughput
// (Mixtral-shaped layer 3.46 -> 5.92 ms), so 64.
constexpr int kGemmBK = 64;

struct RouteArgs {
    const uint16_t* x;     // [T,H] bf16 bits
    const uint16_t* Wg;    // [H,E]
    const float* bias;     // [E] or null
    int32_t* topk_idx;     // [T,k]
    float* topk_w;         // [T,k]
    int64_t T;
    int32_t H, E, k;
    int32_t renorm = 1;    // 1: softmax over the k selected; 0: over all E
    uint32_t* err = nullptr;   // device error word (a bounded wait that ran out), or null
    float* logits = nullptr;   // [T,E] fp32 scratch for E > 8 (the sliced router), or null
};
cudaError_t launch_route(const RouteArgs& a, int num_sms, cudaStream_t s);
// The router kernel launch_route runs for these sizes (MOE_ROUTER_*);
// has_logits: a [T,E] logits scratch is passed (the layer call).
int route_variant(int32_t H, int32_t E, bool has_logits);

// The tensor-core router (route_tc.cu): the gate GEMM on tcgen05, each
// token's selection proven equal to the canonical fp32 order's by an error
// bound, or recomputed in that order. Scratch from the layer's workspace.
constexpr int64_t kRouteTcMinTokens = 512;   // below: one tile per CTA is too few
struct RouteTcArgs {
    uint16_t* wgt;          // [NP, H] the gate transposed (NP = E rounded up to 16)
    float* wpart;           // [H/64, NP] sums of squares of the gate's columns per 64 rows, rounded up
    float* fast;            // [T, E] the tensor-core logits (bias added)
    float* bound;           // [T] B_t: |fast - canonical| <= B_t for every expert of token t
    int32_t* n_exact;       // [2] tokens listed for the canonical recomputation, their member pairs
    int32_t* pairs = nullptr;   // [32 T] listed (token slot * 32 + pair) work items, or null
    float* lg_buf = nullptr;    // [T, 64] canonical logits of the listed tokens' run members
    int32_t* flag_tok;      // [T] the listed tokens
    uint64_t* flag_cand;    // [T] their run members (bit e)
    int32_t* flag_sel;      // [T, 9] their top k+1 by fast logit
    float* flag_selv;       // [T, 9] and those fast logits
    float c_fast = 0.0f;    // bound constants (set by the launcher)
    float c_tot = 0.0f;
    int32_t force_exact = 0;     // recompute every token (test hook)
    float* dbg_fast = nullptr;   // [T, E] the fast logits before the bias (test hook), or null
    float* dbg_bound = nullptr;  // [T] c_fast ||x_t|| max_e ||w_e|| (test hook)
};
bool route_tc_supported(int64_t T, int32_t H, int32_t E);
int route_tc_np(int32_t E);
cudaError_t launch_route_tc(const RouteArgs& a, RouteTcArgs c, int num_sms, cudaStream_t s);

// A TMA tensor map of a row-major bf16 matrix [outer, inner] with box
// {box_inner, box_outer}, a 128- or 64-byte swizzle or none (swizzle_bytes
// 128, 64 or 0); out-of-bounds elements
// read as zero. False if the driver entry point or the encoding fails.
bool encode_map_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
                   uint32_t box_outer, int swizzle_bytes);

// scale[t] = 1 / (1 + exp(-x[t] . wsg)) (the shared expert's sigmoid gate)
cudaError_t launch_shared_gate(const uint16_t* x, const uint16_t* wsg, float* scale, int64_t T,
                               int32_t H, int num_sms, cudaStream_t s);

struct PermuteArgs {
    const int32_t* topk_idx;   // [R]
    int32_t* counts;           // [E]
    int32_t* offsets;          // [E+1]
    int32_t* src_row;          // [R]
    int32_t* inv_pos;          // [R]
    int32_t* tile_start;       // [E+1]  (M-tile prefix of the GEMMs)
    int32_t* hist;             // [num_chunks, E] scratch
    uint32_t* err;
    int64_t R;
    int32_t E;
};
int permute_num_chunks(int64_t R);
cudaError_t launch_permute(const PermuteArgs& a, cudaStream_t s);

// x_perm[p] = x[src_row[p] / k] for p < *r_valid (r_valid = &offsets[E]);
// src_row null = identity, r_valid null = all R rows.
cudaError_t launch_gather_rows(const uint16_t* x, const int32_t* src_row, const int32_t* r_valid,
                               uint16_t* x_perm, int64_t R, int64_t T, int32_t H, int32_t k,
                               uint32_t* err, int num_sms, cudaStream_t s);
// The same x_perm from the token side: x[t] to x_perm[inv_pos[t*k + j]] for
// every j whose id topk_idx[t*k + j] is in [0, E); x read once per token.
cudaError_t launch_scatter_rows(const uint16_t* x, const int32_t* topk_idx, const int32_t* inv_pos,
                                const int32_t* r_valid, uint16_t* x_perm, int64_t T, int32_t H, int32_t k,
                                int32_t E, uint32_t* err, int num_sms, cudaStream_t s);

cudaError_t launch_tile_table(const int32_t* offsets, int32_t G, int32_t* tile_start,
                              cudaStream_t s);

// GEMM0 + SwiGLU with A gathered from x by TMA gather4 (kGemm0Gather) or read
// from the dispatch-ordered copy x_perm (kGemm0Dense); GEMM1 + weighted scatter
// (kGemm1Scatter), or GEMM1 + weighted scatter + the combine done by the last
// of the n_slots contributions to each (token, 256-column tile) (kGemm1Combine).
// kGemm0CpGather: GEMM0 whose A rows are gathered from x by a producer warp
// with 16-byte cp.async copies (no x_perm).
// kFusedScatter / kFusedCombine: GEMM0 (dense A) and GEMM1 (scatter / combine)
// in one persistent launch; a GEMM1 tile waits (bounded) until the GEMM0 tiles
// of its (expert, M tile) have published their rows of h.
enum GemmMode { kGemm0Gather = 0, kGemm1Scatter = 1, kGemm0Dense = 2, kGemm1Combine = 3,
                kGemm0CpGather = 4, kFusedScatter = 5, kFusedCombine = 6 };

struct GemmArgs {
    int32_t M;                   // rows in dispatched order (R, or T for a dense expert)
    int32_t N;                   // GEMM0: F (per W1 / W3);  GEMM1: H
    int32_t K;                   // GEMM0: H;  GEMM1: F
    int32_t G;                   // groups (experts)
    int32_t k;                   // experts per token: token = f / k, rank = f % k
    int64_t T;                   // tokens
    const int32_t* tile_start;   // [G+1] or null (then G == 1: one group of M rows)
    const int32_t* offsets;      // [G+1] or null (then G == 1)
    const int32_t* src_row;      // [M] or null (identity)
    const float* topk_w;         // GEMM1: [M] by f, or null (weight 1)
    __nv_bfloat16* h_out;        // GEMM0: [M, N]
    const uint16_t* x;           // kGemm0CpGather: x [T, K] (A rows gathered by token)
    float* slot;                 // GEMM1: slot array [n_slots, T, N]; rank j goes to slot_j0 + j
    int32_t slot_j0;             // GEMM1: first slot of this launch (the shared expert: k)
    int32_t n_slots;             // kGemm1Combine: contributions summed per (token, N tile)
    int32_t n_tickets;           // kGemm1Combine: arrivals per (token, N tile) before the sum
                                 // (n_slots, or 1 when the other slots were written earlier)
    int32_t* arrive;             // kGemm1Combine: [T, ceil(N/256)] tickets, zero before the first launch
    uint16_t* out;               // kGemm1Combine: [T, N] bf16 layer output
    int32_t* ready;              // fused, GEMM1 args: [M tiles] count of GEMM0 warps done, zero first
    int32_t ready_target;        // fused, GEMM1 args: count that makes an M tile's h complete
    // kGemm0Dense with the dispatch copy inside the launch (copy_ready non-null):
    // warp 6 copies row r of x_perm from x[src_row[r] / k] for the rows
    // r < offsets[G], in 4 KB pieces, counting each finished piece on its
    // 128-row tile; the producer loads a tile once all its pieces are counted
    uint16_t* copy_dst;          // x_perm [M, K], the A operand of this launch
    int32_t* copy_ready;         // [128-row tiles] pieces copied, zero before the launch
    uint32_t* err;
};

// tmA: kGemm0CpGather -> unused (A comes from args.x);
//      kGemm0Gather -> x [T,H] (box 64 x 1, gathered); kGemm0Dense -> x_perm
// [M,H] (box 64 x 128); kGemm1Scatter -> h [M,F] (box 64 x 128).
// tmB0/tmB1: GEMM0 -> W1 / W3 viewed as [G*H, F]; GEMM1 -> W2 viewed as [G*F, H]
// (tmB1 unused). All boxes 64 wide with 128-byte swizzle.
// cta_group 2: one MMA of 256 x 256 over a CTA pair (a 2-CTA cluster), each
// CTA staging half of A's rows and half of B's columns; kGemm0Dense,
// kGemm1Scatter and kGemm1Combine only.
cudaError_t launch_grouped_gemm(int mode, const CUtensorMap& tmA, const CUtensorMap& tmB0,
                                const CUtensorMap& tmB1, const GemmArgs& a, int num_sms,
                                cudaStream_t s, int cta_group = 1);
// Both GEMMs in one launch: a0 / tmA, tmB0, tmB1 as for kGemm0Dense; a1 / tmA1
// (h) and tmB2 (W2) as for GEMM1. mode is kFusedScatter or kFusedCombine.
cudaError_t launch_grouped_gemm_fused(int mode, const CUtensorMap& tmA, const CUtensorMap& tmB0,
                                      const CUtensorMap& tmB1, const CUtensorMap& tmA1,
                                      const CUtensorMap& tmB2, const GemmArgs& a0, const GemmArgs& a1,
                                      int num_sms, cudaStream_t s);

// Counts one kernel launch issued by this library (read with moe_launch_count).
void count_launch();

// Launches kern<<<grid, block, smem, s>>>(args...) with programmatic stream
// serialization (the kernel may start before the previous kernel in the stream
// ends; it calls pdl_wait() before touching global memory) and counts it.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args)
{
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
    if (e == cudaSuccess) count_launch();
    return e;
}

cudaError_t launch_combine(const float* slot, int32_t n_slots, uint16_t* out, int64_t T, int32_t H,
                           int num_sms, cudaStream_t s);

}  // namespace moe
