/*
 * moe.h -- C ABI of the GB300 (sm_103a) MoE FFN layer forward.
 *
 * The layer: top-k routing, dispatch of the routed (token, expert) pairs into
 * per-expert groups, a SwiGLU expert FFN per group (GEMM0 + SwiGLU split
 * along the token dimension M, GEMM1 split along the hidden dimension N),
 * and the gate-weighted combine back to token order. The parts are those
 * named in the DisagMoE summary (gist.science, "Resumo Tecnico: DisagMoE",
 * section 2.2, "Alinhamento de Estagios": top-k experts, dispatch, combine)
 * and on the COMET page (nav.superapi.store/en/comet, "COMET's Technical
 * Principles", "Tensor Decomposition": Layer 0 split along M, Layer 1 along
 * N). The pages give no formulas; the readings used here are:
 *   - logits l[t,e] = sum_h x[t,h] Wg[h,e] in fp32 in one canonical order
 *     (8-element chunks, chunk c on lane c mod 32, fma in increasing h, then
 *     an xor butterfly over the 32 lane sums with strides 16, 8, 4, 2, 1),
 *     plus bias[e] when a bias is given;
 *   - top-k on the logits, descending, ties to the lower expert id; the rank
 *     of an expert is its selection position;
 *   - gate weights = softmax over the k selected logits;
 *   - expert e: y = (silu(x W1[e]) * (x W3[e])) W2[e], silu(a) = a/(1+e^-a);
 *   - out[t] = sum over ranks j = 0..k-1 (in that order) of w[t,j] y_j,
 *     plus the always-on shared expert (weight 1) when F_shared > 0.
 *
 * Conventions (every entry point):
 *   - Tensors are row-major and contiguous: x[T,H], Wg[H,E], W1/W3[E,H,F],
 *     W2[E,F,H]; shared expert W1s/W3s[H,Fs], W2s[Fs,H]. bf16 tensors are
 *     passed as moe_bf16 (raw bf16 bits).
 *   - Every pointer is a device pointer owned by the caller; the library
 *     allocates no memory and keeps no per-call state. Scratch memory is the
 *     caller's workspace `ws` of at least moe_workspace_size(dims) bytes,
 *     256-byte aligned. Two calls that share a workspace must not overlap.
 *   - Calls are asynchronous on `stream`. Argument checks run on the host
 *     before any launch and return MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED
 *     / MOE_ERR_WORKSPACE without launching. A launch failure returns
 *     MOE_ERR_CUDA. Errors found on the device (an expert id outside
 *     [0, E), a bounded wait that ran out) are OR-ed into the error word at
 *     the start of `ws` and read by moe_check(); with the environment
 *     variable MOE_DEBUG=1 every entry point synchronises and checks.
 *   - Supported shapes (else MOE_ERR_UNSUPPORTED): 1 <= k <= min(E, 8),
 *     E <= 256, H and F (and F_shared) multiples of 64, T*k < 2^31.
 *     T == 0 is a valid no-op. Pointers must be 16-byte aligned.
 *   - Results are bit-identical from run to run (no float atomics).
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t moe_bf16;                 /* raw bf16 bits */
typedef struct CUstream_st* moe_stream_t;  /* the same type as cudaStream_t */
typedef struct CUevent_st* moe_event_t;    /* the same type as cudaEvent_t */

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,   /* null pointer, negative size, bad id (device) */
    MOE_ERR_UNSUPPORTED = 2,   /* shape outside the supported set */
    MOE_ERR_WORKSPACE = 3,     /* workspace missing, too small or misaligned */
    MOE_ERR_CUDA = 4,          /* a CUDA runtime / driver call failed */
    MOE_ERR_TIMEOUT = 5,       /* a bounded device wait ran out (device) */
    MOE_ERR_DEVICE_BOUNDS = 6  /* a device index check failed (device) */
} moe_status;

typedef struct {
    int64_t T;         /* tokens */
    int32_t H;         /* hidden size */
    int32_t F;         /* expert FFN width */
    int32_t E;         /* routed experts */
    int32_t k;         /* experts per token */
    int32_t F_shared;  /* shared expert FFN width; 0 = no shared expert */
} moe_dims;

/* Optional per-stage timing: each non-null event is recorded on the stream
 * at that point of moe_layer_forward. */
typedef struct {
    moe_event_t before_route;
    moe_event_t before_permute;
    moe_event_t before_gemm0;      /* routed GEMM0 + SwiGLU */
    moe_event_t before_gemm1;      /* routed GEMM1 + weighted scatter */
    moe_event_t before_shared;     /* shared-expert GEMM0 + GEMM1 (if any) */
    moe_event_t before_combine;
    moe_event_t after_combine;
} moe_stage_events;

/* Gating variants (readings of this library; the pages give no gate formula).
 * A null moe_gating* means {renormalize = 1, shared_gate = NULL}. */
typedef struct {
    int32_t renormalize;          /* 1: weights = softmax over the k selected logits;
                                     0: softmax over all E logits at the selected ids
                                        (the k weights then sum to less than 1) */
    const moe_bf16* shared_gate;  /* [H] or NULL: scale the shared expert's output by
                                     sigmoid(x[t] . shared_gate) instead of 1 */
} moe_gating;

/* Optional routing outputs of moe_layer_forward; each null field is kept in
 * the workspace instead. Sizes: [T*k], [T*k], [E], [E+1], [T*k], [T*k]. */
typedef struct {
    int32_t* topk_idx;
    float* topk_w;
    int32_t* counts;
    int32_t* offsets;
    int32_t* src_row;
    int32_t* inv_pos;
} moe_routing_out;

/* Library-wide options (moe_set_option / moe_get_option). */
enum {
    /* How GEMM0 obtains the routed token rows (its A operand):
     *   MOE_GEMM0_A_PERMUTED   (default) the dispatch step copies them into
     *                          dispatch order (x_perm, in the workspace) and
     *                          GEMM0 loads dense 128-row TMA tiles;
     *   MOE_GEMM0_A_TMA_GATHER the GEMM0 producer warp gathers them straight
     *                          from x with TMA gather4, 4 rows per instruction;
     *   MOE_GEMM0_A_CP_GATHER  a GEMM0 producer warp gathers them straight
     *                          from x with 16-byte cp.async copies.
     * All give bit-identical results. */
    MOE_OPT_GEMM0_A = 0,
    MOE_GEMM0_A_PERMUTED = 0,
    MOE_GEMM0_A_TMA_GATHER = 1,
    MOE_GEMM0_A_CP_GATHER = 2,
    /* Where moe_layer_forward sums the k weighted expert rows of a token:
     *   MOE_COMBINE_AUTO     (default) fused when the last GEMM1 to run (the
     *                        shared expert's if any, else the routed one) has
     *                        K >= 4096, else separate;
     *   MOE_COMBINE_FUSED    in GEMM1's epilogue: each row takes an integer
     *                        ticket per (token, 256-column tile) and the last
     *                        one sums the token's slots in rank order;
     *   MOE_COMBINE_SEPARATE a streaming combine kernel after the GEMMs.
     * Both sum the same fp32 values in the same order: bit-identical. */
    MOE_OPT_COMBINE = 1,
    MOE_COMBINE_AUTO = 0,
    MOE_COMBINE_FUSED = 1,
    MOE_COMBINE_SEPARATE = 2,
    /* Whether moe_layer_forward runs the routed experts' two GEMMs as one
     * persistent launch (GEMM1 tiles start as soon as the GEMM0 tiles of their
     * expert and 128-row block have written h; no launch boundary, no GEMM0
     * tail) or as two launches. Only with MOE_GEMM0_A_PERMUTED.
     *   MOE_GEMM_FUSION_AUTO (default) the table in the library's layer call
     *                        (by shape; see moe_layer_forward);
     *   MOE_GEMM_FUSION_ON / MOE_GEMM_FUSION_OFF force it.
     * Same arithmetic either way: bit-identical. */
    MOE_OPT_GEMM_FUSION = 2,
    MOE_GEMM_FUSION_AUTO = 0,
    MOE_GEMM_FUSION_ON = 1,
    MOE_GEMM_FUSION_OFF = 2,
    /* How many CTAs share one tensor-core MMA in the expert GEMMs that read a
     * dense A operand (GEMM0 over x_perm, every GEMM1, the shared expert):
     *   MOE_CTA_GROUP_AUTO (default) the table in the library's layer call
     *                      (by rows per expert and GEMM; see moe_layer_plan);
     *   MOE_CTA_GROUP_ONE  one CTA per 128 x 256 MMA tile;
     *   MOE_CTA_GROUP_PAIR a 2-CTA cluster per 256 x 256 MMA tile
     *                      (tcgen05 cta_group::2): each CTA stages 128 rows
     *                      of A and half of B's columns.
     * The gathered GEMM0 forms and the one-launch GEMM pair always run one CTA
     * per MMA. */
    MOE_OPT_CTA_GROUP = 3,
    MOE_CTA_GROUP_AUTO = 0,
    MOE_CTA_GROUP_ONE = 1,
    MOE_CTA_GROUP_PAIR = 2,
    /* Who copies the routed token rows into dispatch order (x_perm) when
     * GEMM0 reads them from there (MOE_GEMM0_A_PERMUTED, two GEMM launches):
     *   MOE_X_PERM_COPY_AUTO   (default) the table (see moe_layer_plan): the
     *                          kernel, which measured as fast on GB300;
     *   MOE_X_PERM_COPY_INLINE a spare warp of every GEMM0 CTA, while the
     *                          GEMM runs: each 128-row tile is computed as
     *                          soon as its rows are copied (counted per
     *                          tile), so the copy overlaps the tensor work;
     *   MOE_X_PERM_COPY_KERNEL a copy kernel before GEMM0.
     * The same bytes either way: bit-identical. */
    MOE_OPT_X_PERM_COPY = 4,
    MOE_X_PERM_COPY_AUTO = 0,
    MOE_X_PERM_COPY_INLINE = 1,
    MOE_X_PERM_COPY_KERNEL = 2,
    /* Which router moe_layer_forward runs:
     *   MOE_ROUTER_OPT_AUTO   (default) the table (see moe_layer_plan): the
     *                         tensor-core router for 16 <= E <= 64 (E a
     *                         multiple of 8) from T = 8192, where it measured
     *                         faster, else an FMA router;
     *   MOE_ROUTER_OPT_FMA    the FMA routers (the canonical order itself);
     *   MOE_ROUTER_OPT_TENSOR the tensor-core router wherever it applies
     *                         (8 <= E <= 64, E a multiple of 8, T >= 512).
     * The expert ids and their order are the same bit for bit either way
     * (the tensor-core router proves each token's selection against the
     * canonical order, or recomputes the token in it); the gate weights agree
     * to fp32 rounding (a softmax of logits whose summation order differs). */
    MOE_OPT_ROUTER = 5,
    MOE_ROUTER_OPT_AUTO = 0,
    MOE_ROUTER_OPT_FMA = 1,
    MOE_ROUTER_OPT_TENSOR = 2
};

/* Sets a library-wide option for later calls (all devices and threads).
 * Returns MOE_ERR_INVALID_ARG for an unknown option or value. Do not change
 * options while another thread is inside a call. */
moe_status moe_set_option(int option, int value);

/* Current value of an option, or -1 for an unknown option. */
int moe_get_option(int option);

/* Router kernels (moe_plan.router). All select the same experts in the same
 * order bit for bit; the FMA routers (0..3) also give the same logits. */
enum {
    MOE_ROUTER_STREAM = 0,   /* E <= 8: TMA-fed per-warp pipelines, top-k fused */
    MOE_ROUTER_SLICED = 1,   /* E > 8, a multiple of 8, inside moe_layer_forward: expert
                              * slices of 8 per CTA, logits to the workspace, top-k pass */
    MOE_ROUTER_CLUSTER = 2,  /* 8 < E <= 64: canonical lanes split over a CTA cluster */
    MOE_ROUTER_BLOCK = 3,    /* anything else: one CTA per SM, gate staged in slices */
    MOE_ROUTER_TENSOR = 4    /* inside moe_layer_forward, 8 <= E <= 64, E % 8 == 0: the
                              * gate GEMM on tcgen05; each token's top-k proven equal to
                              * the canonical order's by an error bound (ties and near
                              * ties recomputed in the canonical order) */
};

/* The configuration moe_layer_forward runs for a shape under the current
 * options: the library's per-shape table, fixed before any launch. */
typedef struct {
    int32_t router;        /* MOE_ROUTER_* */
    int32_t gemm0_a;       /* MOE_GEMM0_A_* in effect */
    int32_t combine;       /* MOE_COMBINE_FUSED or MOE_COMBINE_SEPARATE */
    int32_t gemm_fusion;   /* MOE_GEMM_FUSION_ON or MOE_GEMM_FUSION_OFF */
    int32_t tile_m;        /* grouped GEMM tile rows (routed rows per tile; 256 for a CTA pair) */
    int32_t tile_n;        /* grouped GEMM MMA N (GEMM0: half W1, half W3) */
    int32_t tile_k;        /* K per pipeline stage */
    int32_t stages;        /* shared-memory pipeline stages */
    int32_t cta_group;     /* CTAs per MMA (tcgen05 cta_group) of the routed GEMM0; tile_m
                            * and stages describe it */
    int32_t cta_group_gemm1; /* the same for the routed GEMM1 (a second launch; 1 when both
                              * GEMMs share one launch) */
    int32_t x_perm_copy;   /* MOE_X_PERM_COPY_INLINE or _KERNEL; 0 when GEMM0 does not read x_perm */
} moe_plan;

/* Fills *plan for `dims` (host only: no device work, no launch). Returns
 * MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED for shapes moe_layer_forward
 * rejects. */
moe_status moe_layer_plan(const moe_dims* dims, moe_plan* plan);

/* Self-test of the failure path every pipeline wait takes: one device thread
 * waits, bounded by limit_ms (1..4000) of %globaltimer time, on a device flag
 * that nothing sets, gives up, and reports it through a device error word.
 * Returns MOE_ERR_TIMEOUT when that happened (the expected outcome), MOE_OK if
 * the wait somehow completed, MOE_ERR_CUDA on a launch or copy error. The
 * device stays usable. Synchronises `stream`. */
moe_status moe_selftest_wait_timeout(int32_t limit_ms, moe_stream_t stream);

/* Test hook of the tensor-core router (MOE_ROUTER_TENSOR): routes x with it
 * as moe_layer_forward would, writing topk_idx[T,k] / topk_w[T,k] and
 * optionally
 *   fast_logits[T,E]  the tensor-core logits (before the bias),
 *   fast_bound[T]     the bound used for the tensor-core part of the error,
 *                     c_fast ||x_t|| max_e ||w_e||, so that a caller can check
 *                     |fast_logits - exact| <= fast_bound,
 *   n_exact           how many tokens took the canonical recomputation
 *                     (reading it synchronises `stream`).
 * force_exact != 0 sends every token through the canonical recomputation.
 * ws is a moe_layer_forward workspace for dims. MOE_ERR_UNSUPPORTED where the
 * tensor-core router does not apply. Not needed for normal use. */
moe_status moe_selftest_route_tc(const moe_dims* dims, const moe_bf16* x, const moe_bf16* Wg,
                                 const float* bias, int32_t renormalize, int32_t force_exact,
                                 int32_t* topk_idx, float* topk_w, float* fast_logits,
                                 float* fast_bound, int64_t* n_exact, void* ws, size_t ws_bytes,
                                 moe_stream_t stream);

/* Library version (major*10000 + minor*100 + patch). */
int moe_version(void);

/* Number of CUDA kernels this library has launched in this process (all
 * threads, devices and streams) since it was loaded: each kernel launch of
 * every call counts once; memsets and copies do not. A caller takes the
 * difference around a region to count what that region launched. */
uint64_t moe_launch_count(void);

/* Text for a status code. Never null. */
const char* moe_status_string(int status);

/* Workspace bytes that every entry point below accepts for `dims`.
 * Returns 0 for invalid dims. */
size_t moe_workspace_size(const moe_dims* dims);

/* Synchronises `stream`, reads and clears the device error word at the start
 * of `ws`, and returns the status it holds (MOE_OK if none). */
moe_status moe_check(void* ws, moe_stream_t stream);

/*
 * Router (top-k gating).
 * In:  x[T,H], Wg[H,E] (bf16); bias[E] (f32, may be null).
 * Out: topk_idx[T,k] (int32, expert ids in rank order), topk_w[T,k] (f32,
 *      the softmax of the selected logits, in rank order).
 * The logits are computed in the canonical fp32 order given above, so the ids
 * are bit-exact against any implementation of that order.
 */
moe_status moe_route(const moe_dims* dims, const moe_bf16* x, const moe_bf16* Wg, const float* bias,
                     int32_t* topk_idx, float* topk_w, moe_stream_t stream);

/* moe_route with a gating variant (gating->renormalize; shared_gate unused). */
moe_status moe_route_ex(const moe_dims* dims, const moe_bf16* x, const moe_bf16* Wg, const float* bias,
                        const moe_gating* gating, int32_t* topk_idx, float* topk_w, moe_stream_t stream);

/*
 * Dispatch: stable counting sort of the R = T*k assignments f = t*k + j by
 * expert id topk_idx[f] (the "dispatch" of the DisagMoE summary, 2.2).
 * In:  topk_idx[R] (int32).
 * Out: counts[E]; offsets[E+1] (exclusive scan, offsets[E] = R);
 *      src_row[R] (src_row[p] = f, experts in increasing order, f increasing
 *      within an expert); inv_pos[R] (inv_pos[f] = p).
 *      x_perm[R,H] (bf16, may be null): x_perm[p] = x[src_row[p] / k]; x
 *      must be given when x_perm is.
 * An id outside [0, E) sets MOE_ERR_INVALID_ARG in the device error word and
 * that assignment is skipped (no out-of-bounds write).
 * Also writes the GEMM tile table into `ws` for a later moe_expert_ffn /
 * moe_layer_forward on the same workspace.
 */
moe_status moe_permute(const moe_dims* dims, const int32_t* topk_idx, int32_t* counts,
                       int32_t* offsets, int32_t* src_row, int32_t* inv_pos, const moe_bf16* x,
                       moe_bf16* x_perm, void* ws, size_t ws_bytes, moe_stream_t stream);

/*
 * Dispatch with no workspace: the same results as moe_permute (counts,
 * offsets, src_row, inv_pos and the optional x_perm, bit for bit), for
 * callers that cannot provide scratch memory -- a host framework that gives
 * its plug-ins no allocator or scratch hook, or a service whose device memory
 * budget is fixed at start-up and which must not allocate while serving.
 * The pages have no counterpart to this entry point; it is an interface
 * convenience of this library.
 * Scratch: a fixed 1 MiB array inside the library, one per GPU, held until
 * the process exits. Shapes whose per-chunk histogram (ceil(T*k / 2048) * E
 * ints) exceeds 261632 ints are rejected with MOE_ERR_UNSUPPORTED before any
 * launch (for example E = 64 allows T*k up to 8,372,224).
 * The first call on a device looks up the array's device address with that
 * device current; make it before any stream capture on the device. The
 * address is cached for the life of the device's context: calling
 * cudaDeviceReset after the first call is not supported. All calls
 * on a device share the array, which keeps the last call's contents (nothing
 * in it needs to start at zero); calls that overlap on the GPU race on it and
 * must be serialised by the caller. No memory is allocated by this call.
 * The shape checks are moe_permute's. An expert id outside [0, E) is
 * skipped (offsets[E] then ends below T*k); there is no device error word.
 * With MOE_DEBUG=1 the call synchronises and returns MOE_ERR_CUDA if a
 * launch faulted.
 */
moe_status moe_permute_static(const moe_dims* dims, const int32_t* topk_idx, int32_t* counts,
                              int32_t* offsets, int32_t* src_row, int32_t* inv_pos,
                              const moe_bf16* x, moe_bf16* x_perm, moe_stream_t stream);

/*
 * Expert FFN over the dispatched groups: for every position p of expert e
 * (offsets[e] <= p < offsets[e+1]) with f = src_row[p], t = f / k, j = f % k:
 *   h[p]      = silu(x[t] W1[e]) * (x[t] W3[e])     (GEMM0 + SwiGLU, h in bf16)
 *   slot[j,t] = w * (h[p] W2[e])                    (GEMM1 + weighted scatter)
 * with w = topk_w[f], or 1 when topk_w is null.
 * In:  x[T,H]; src_row[R] (null = identity: f = p); offsets[E+1] (null = one
 *      group holding all R rows; then E must be 1); W1/W3[E,H,F], W2[E,F,H].
 * Out: slot[k,T,H] (f32). Every (j, t) slot is written exactly once.
 * Call with dims {T, H, F=Fs, E=1, k=1} and null src_row/offsets/topk_w to
 * run a dense (shared) expert into slot[0].
 */
moe_status moe_expert_ffn(const moe_dims* dims, const moe_bf16* x, const int32_t* src_row,
                          const int32_t* offsets, const moe_bf16* W1, const moe_bf16* W3,
                          const moe_bf16* W2, const float* topk_w, float* slot, void* ws,
                          size_t ws_bytes, moe_stream_t stream);

/*
 * Combine (the "combine" of the DisagMoE summary, 2.2): out[t,:] =
 * bf16( ((slot[0,t,:] + slot[1,t,:]) + ...) + slot[n_slots-1,t,:] ), an fp32
 * left fold in slot order, no atomics.
 * In:  slot[n_slots,T,H] (f32), 1 <= n_slots <= 9.  Out: out[T,H] (bf16).
 */
moe_status moe_combine(const moe_dims* dims, const float* slot, int32_t n_slots, moe_bf16* out,
                       moe_stream_t stream);

/*
 * The whole layer: route -> permute -> expert FFN (routed; then the shared
 * expert when dims->F_shared > 0) -> combine.
 * In:  x, Wg, bias (nullable), W1, W3, W2; W1s/W3s/W2s (needed iff F_shared > 0).
 * Out: out[T,H] (bf16); routing (nullable) receives the routing tensors.
 * events (nullable) are recorded at the stage boundaries.
 */
moe_status moe_layer_forward(const moe_dims* dims, const moe_bf16* x, const moe_bf16* Wg,
                             const float* bias, const moe_bf16* W1, const moe_bf16* W3,
                             const moe_bf16* W2, const moe_bf16* W1s, const moe_bf16* W3s,
                             const moe_bf16* W2s, moe_bf16* out, const moe_routing_out* routing,
                             void* ws, size_t ws_bytes, const moe_stage_events* events,
                             moe_stream_t stream);

/* moe_layer_forward with a gating variant (nullable; see moe_gating). A
 * shared_gate needs F_shared > 0; its [H] vector must be 16-byte aligned. */
moe_status moe_layer_forward_ex(const moe_dims* dims, const moe_bf16* x, const moe_bf16* Wg,
                                const float* bias, const moe_gating* gating, const moe_bf16* W1,
                                const moe_bf16* W3, const moe_bf16* W2, const moe_bf16* W1s,
                                const moe_bf16* W3s, const moe_bf16* W2s, moe_bf16* out,
                                const moe_routing_out* routing, void* ws, size_t ws_bytes,
                                const moe_stage_events* events, moe_stream_t stream);

/*
 * The whole layer from and to host memory: x_host[T,H] in, out_host[T,H] out
 * (bf16), every weight already on the device. The tokens are split into
 * n_chunks consecutive chunks (0: the library's choice, else 1..64) and the
 * chunks are pipelined: while the layer runs on chunk c (on `stream`), the
 * host-to-device copy of chunk c+1 and the device-to-host copy of chunk c-1
 * run on two copy streams the library keeps per device. Tokens are
 * independent (routing and the expert GEMMs of a row do not depend on the
 * other rows in its chunk) and every chunk runs the router family the whole
 * batch would, so every output row is bit for bit the one moe_layer_forward
 * gives for the whole batch. One exception: when the whole batch takes the
 * tensor-core router and a caller-chosen n_chunks leaves a chunk below the
 * 512 tokens that router needs, that chunk takes the FMA routers: the same
 * ids and dispatch, gate weights within fp32 rounding (the library's own
 * chunk choice never does this).
 *
 * x_host and out_host should be page-locked (cudaHostAlloc /
 * cudaHostRegister); pageable memory works but its copies do not overlap.
 * x_dev and out_dev are caller-owned device staging buffers of T*H bf16
 * each, 16-byte aligned; on return x_dev holds x and out_dev the output.
 * ws is moe_workspace_size(dims) bytes (the whole batch's), as for
 * moe_layer_forward. The call is stream-ordered on `stream`: it starts after
 * the work already queued there, and work queued there afterwards starts
 * once out_host holds the result (synchronize the stream before reading it).
 * Errors: the argument checks of moe_layer_forward (MOE_ERR_INVALID_ARG for
 * a null or misaligned pointer or n_chunks outside 0..64); MOE_ERR_CUDA if a
 * copy, an event or a launch fails, after which out_host is unspecified (work
 * queued on `stream` afterwards still waits for every copy already queued).
 * Concurrent calls from several host threads on one device share the copy
 * streams and are serialized by them (correct, not overlapped).
 */
moe_status moe_layer_forward_host(const moe_dims* dims, const moe_bf16* x_host, const moe_bf16* Wg,
                                  const float* bias, const moe_bf16* W1, const moe_bf16* W3,
                                  const moe_bf16* W2, const moe_bf16* W1s, const moe_bf16* W3s,
                                  const moe_bf16* W2s, moe_bf16* out_host, moe_bf16* x_dev,
                                  moe_bf16* out_dev, int32_t n_chunks, void* ws, size_t ws_bytes,
                                  moe_stream_t stream);

/* The chunk count moe_layer_forward_host uses for n_chunks = 0 (host only). */
int32_t moe_host_chunks(const moe_dims* dims);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
