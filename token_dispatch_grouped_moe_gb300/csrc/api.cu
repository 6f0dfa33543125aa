// api.cu -- the C ABI of include/moe.h: argument checks, workspace layout,
// TMA descriptors and the launch sequence of the layer. Host code only.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>
#include <algorithm>

#include <nvtx3/nvToolsExt.h>

#include "../../include/moe.h"
#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kVersion = 300;   // 0.3.0
constexpr int kMaxDevices = 64;

// ---------------------------------------------------------------- tracing --

// An NVTX range over the host code that enqueues one stage: a profiler or
// tracer that records NVTX (ncu --nvtx, Nsight Systems) attributes each
// kernel to the stage that launched it ("moe/route", "moe/gemm0", ...). With
// no tool attached, a push/pop pair is a couple of branches (NVTX v3 is
// header-only and loads no library unless a tool asks for it).
struct Range {
    explicit Range(const char* name) { nvtxRangePushA(name); }
    ~Range() { nvtxRangePop(); }
    void next(const char* name)   // close this range and open the next stage's
    {
        nvtxRangePop();
        nvtxRangePushA(name);
    }
    Range(const Range&) = delete;
    Range& operator=(const Range&) = delete;
};

// ------------------------------------------------------------ device info --

std::atomic<int> g_num_sms[kMaxDevices];
std::atomic<int> g_gemm0_a{MOE_GEMM0_A_PERMUTED};
std::atomic<int> g_combine{MOE_COMBINE_AUTO};
std::atomic<int> g_gemm_fusion{MOE_GEMM_FUSION_AUTO};
std::atomic<int> g_cta_group{MOE_CTA_GROUP_AUTO};
std::atomic<int> g_x_perm_copy{MOE_X_PERM_COPY_AUTO};
std::atomic<int> g_router{MOE_ROUTER_OPT_AUTO};
std::atomic<unsigned long long> g_launch_count{0};

int num_sms_current()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    int n = g_num_sms[dev].load(std::memory_order_relaxed);
    if (n > 0) return n;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        return -1;
    g_num_sms[dev].store(n, std::memory_order_relaxed);
    return n;
}

// ---------------------------------------------------------- tensor maps --

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

}  // namespace

bool encode_map_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
                   uint32_t box_outer, int swizzle_bytes)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * 2};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                    : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                          : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

namespace {

// The grouped GEMM's operands, bf16 [outer, inner] (inner contiguous);
// out-of-bounds elements read as zero.
// A (K-major rows): box {kGemmBK, box_rows}, swizzle = one A row (kGemmBK * 2 bytes).
bool make_map_a(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_rows)
{
    return encode_map_2d(m, base, inner, outer, kGemmBK, box_rows, kGemmBK * 2);
}
// B (weights, N contiguous): box {64 columns, kGemmBK k-rows}, 128-byte swizzle.
bool make_map_b(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer)
{
    return encode_map_2d(m, base, inner, outer, 64, kGemmBK, 128);
}

// The per-shape table of moe_layer_forward (all entries measured on GB300):
//  - router: by E and the gate's shared-memory size (route_variant);
//  - combine, automatic: fused into GEMM1's epilogue when the last GEMM1 to
//    run has K >= 4096 (Mixtral F = 14336, Qwen2 shared F = 20480), where the
//    epilogue work hides behind a long main loop; separate for short tiles
//    (DeepSeek F = 1408: fused GEMM1 0.42 -> 0.81 ms at T = 16384, k = 6);
//  - GEMM fusion, automatic: both routed GEMMs in one launch below 512 routed
//    rows per expert on average, where the GEMMs are short and
//    weight-bandwidth bound and the GEMM0 tail and launch boundary weigh
//    (DeepSeek-shaped T = 1024: 0.273 -> 0.259 ms per layer, T = 4096:
//    0.484 -> 0.467 ms); from 512 rows per expert up (Qwen2, DeepSeek
//    T = 32768, Mixtral) the two forms measured the same;
//  - CTAs per MMA (dense-A GEMMs, not in the one-launch pair): a 2-CTA
//    cluster per 256 x 256 x 64 tile (tcgen05 cta_group::2, 6 stages of 32 KB
//    in each CTA) for GEMM0 from 1024 dispatched rows per expert on average
//    and for GEMM1 from 512; else one CTA per 128 x 256 x 64 tile (4 stages of
//    48 KB). Measured per layer, one CTA -> pairs: DeepSeek T = 32768 2.87 ->
//    2.76 ms (GEMM1 0.80 -> 0.72), T = 16384 1.49 -> 1.43, Qwen2 2.55 -> 2.49
//    (GEMM0 0.85 -> 0.87: 512 rows per expert pad more in 256-row tiles),
//    Mixtral 3.53 -> 3.51. Zipf routing needs no reordering: the static
//    schedule spreads every expert's tiles over all SMs (Mixtral-Zipf measured
//    as fast as uniform routing).
// CTAs per MMA for an expert GEMM over `rows` dispatched rows in `groups`
// experts (option, else the table): a pair's 256-row tiles pad each expert to
// a multiple of 256 rows, which costs GEMM0 more than the pair gains below
// 1024 rows per expert; GEMM1 gains more (its short K leaves a 4-stage ring
// of 48 KB exposed at every tile) and takes pairs from 512.
int cta_group_for(int64_t rows, int32_t groups, bool gemm1)
{
    const int opt = g_cta_group.load();
    if (opt == MOE_CTA_GROUP_ONE) return 1;
    if (opt == MOE_CTA_GROUP_PAIR) return 2;
    return rows >= (int64_t)(gemm1 ? 512 : 1024) * groups ? 2 : 1;
}

moe_plan plan_of(const moe_dims& d)
{
    moe_plan p{};
    p.router = route_variant(d.H, d.E, /*has_logits=*/true);
    const int router_opt = g_router.load();
    // the tensor-core router (the ids are the same either way): forced by the
    // option wherever it applies, else where it measured faster than the FMA
    // routers on GB300: E >= 16 from 4096 tokens (DeepSeek-shaped T = 4096:
    // 44 -> 36 us, T = 16384: 107 -> 55 us, T = 32768: 206 -> 83 us; Qwen2-
    // shaped T = 4096: 68 -> 60 us). Below that, and for E = 8, the FMA
    // routers are as fast or faster (Mixtral-shaped 27 vs 45 us, DeepSeek-
    // shaped T = 1024 26 vs 36 us).
    if (route_tc_supported(d.T, d.H, d.E) &&
        (router_opt == MOE_ROUTER_OPT_TENSOR ||
         (router_opt == MOE_ROUTER_OPT_AUTO && d.E >= 16 && d.T >= 4096)))
        p.router = MOE_ROUTER_TENSOR;
    p.gemm0_a = g_gemm0_a.load();
    const int combine_opt = g_combine.load();
    const int32_t k_last = d.F_shared > 0 ? d.F_shared : d.F;
    p.combine = (combine_opt == MOE_COMBINE_FUSED || (combine_opt == MOE_COMBINE_AUTO && k_last >= 4096))
                    ? MOE_COMBINE_FUSED : MOE_COMBINE_SEPARATE;
    const int fusion_opt = g_gemm_fusion.load();
    const bool fuse = p.gemm0_a == MOE_GEMM0_A_PERMUTED &&
                      (fusion_opt == MOE_GEMM_FUSION_ON ||
                       (fusion_opt == MOE_GEMM_FUSION_AUTO && d.T * (int64_t)d.k < (int64_t)512 * d.E));
    p.gemm_fusion = fuse ? MOE_GEMM_FUSION_ON : MOE_GEMM_FUSION_OFF;
    p.cta_group = (p.gemm0_a == MOE_GEMM0_A_PERMUTED && !fuse)
                      ? cta_group_for(d.T * (int64_t)d.k, d.E, false) : 1;
    p.cta_group_gemm1 = fuse ? 1 : cta_group_for(d.T * (int64_t)d.k, d.E, true);
    if (p.gemm0_a == MOE_GEMM0_A_PERMUTED) {
        const int opt = g_x_perm_copy.load();
        // measured no faster inline (the copy's bulk loads share each SM's TMA
        // unit with the GEMM's operand loads): the kernel unless asked
        p.x_perm_copy = (!fuse && opt == MOE_X_PERM_COPY_INLINE) ? MOE_X_PERM_COPY_INLINE : MOE_X_PERM_COPY_KERNEL;
    }
    p.tile_m = p.cta_group == 2 ? 2 * kTileM : kTileM;
    p.tile_n = 256;
    p.tile_k = 64;
    p.stages = p.cta_group == 2 ? 6 : 4;
    return p;
}

// ------------------------------------------------------------ workspace --

size_t al256(size_t x) { return (x + 255) & ~(size_t)255; }

struct Layout {
    size_t err, tile, hist, idx, w, counts, offsets, src, inv, xp, h, hs, slot, arrive, sgate, logits, ready;
    size_t tc_wgt, tc_wnorm, tc_nflag, tc_tok, tc_cand, tc_ftok, tc_fcand, tc_fsel, tc_fselv, tc_pairs, tc_lg,
        total;
};

Layout layout_of(const moe_dims& d)
{
    const size_t T = (size_t)d.T, R = (size_t)d.T * d.k;
    const size_t E = (size_t)d.E;
    Layout L;
    size_t o = 0;
    L.err = o; o += 256;
    L.tile = o; o += al256((E + 2) * 4);
    L.hist = o; o += al256((size_t)permute_num_chunks((int64_t)R) * E * 4);
    L.idx = o; o += al256(R * 4);
    L.w = o; o += al256(R * 4);
    L.counts = o; o += al256(E * 4);
    L.offsets = o; o += al256((E + 1) * 4);
    L.src = o; o += al256(R * 4);
    L.inv = o; o += al256(R * 4);
    L.xp = o; o += al256(R * (size_t)d.H * 2);
    L.h = o; o += al256(R * (size_t)d.F * 2);
    L.hs = o; o += al256(T * (size_t)d.F_shared * 2);
    L.slot = o; o += al256(((size_t)d.k + (d.F_shared > 0 ? 1 : 0)) * T * (size_t)d.H * 4);
    L.arrive = o; o += al256(T * (size_t)((d.H + 255) / 256) * 4);
    L.sgate = o; o += al256(T * 4);
    L.logits = o; o += al256(E > 8 ? T * E * 4 : 0);   // the sliced router's logits
    L.ready = o; o += al256(((R + kTileM - 1) / kTileM + E + 1) * 4);   // fused GEMMs: per M tile
    // the tensor-core router: transposed gate, column norms, the list of
    // tokens recomputed in the canonical order
    const bool tc = route_tc_supported((int64_t)T, d.H, d.E) || (d.E >= 8 && d.E <= 64 && d.E % 8 == 0);
    const size_t np = tc ? (size_t)route_tc_np(d.E) : 0;
    L.tc_wgt = o; o += al256(np * (size_t)d.H * 2);
    L.tc_wnorm = o; o += al256(np * (size_t)(d.H / 64) * 4);
    L.tc_nflag = o; o += al256(tc ? 4 : 0);
    L.tc_tok = o; o += al256(tc ? T * 4 : 0);                  // per-token bound
    L.tc_cand = o; o += al256(tc ? T * (size_t)d.E * 4 : 0);   // fast logits
    L.tc_ftok = o; o += al256(tc ? T * 4 : 0);                  // listed tokens
    L.tc_fcand = o; o += al256(tc ? T * 8 : 0);
    L.tc_fsel = o; o += al256(tc ? T * 9 * 4 : 0);
    L.tc_fselv = o; o += al256(tc ? T * 9 * 4 : 0);
    L.tc_pairs = o; o += al256(tc ? T * 32 * 4 : 0);                // (token, member pair) items
    L.tc_lg = o; o += al256(tc ? T * 64 * 4 : 0);                   // their canonical logits
    L.total = o;
    return L;
}

// ----------------------------------------------------------- validation --

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

moe_status check_ws(const moe_dims& d, void* ws, size_t ws_bytes)
{
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return MOE_ERR_WORKSPACE;
    if (ws_bytes < layout_of(d).total) return MOE_ERR_WORKSPACE;
    return MOE_OK;
}

moe_status finish(cudaError_t e, void* ws, cudaStream_t s)
{
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    if (debug_mode()) {
        if (ws) return moe_check(ws, (moe_stream_t)s);
        if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
    }
    return MOE_OK;
}

#define MOE_TRY(expr)                                  \
    do {                                               \
        cudaError_t e_ = (expr);                       \
        if (e_ != cudaSuccess) return MOE_ERR_CUDA;    \
    } while (0)

#define MOE_TRY_STATUS(expr)                           \
    do {                                               \
        moe_status s_ = (expr);                        \
        if (s_ != MOE_OK) return s_;                   \
    } while (0)

unsigned char* bytes(void* p) { return static_cast<unsigned char*>(p); }

// The two grouped GEMMs of one expert set (routed or shared). GEMM0 reads its
// A rows from x_rows ([M,H], already in dispatch order) when given, else it
// gathers them from x with TMA gather4.
// With `fused` (the layer path), GEMM1 also finishes the combine: slot is the
// whole [n_slots, T, H] array, this launch writes slots slot_j0 .. slot_j0+k-1,
// and the last contribution to each (token, 256-column tile) writes out.
// GEMM1 + combine: the row holding the last of n_tickets arrivals per
// (token, N tile) sums n_slots slots from slot 0 (n_tickets 0 = n_slots).
struct FusedCombine {
    bool on;
    int32_t slot_j0, n_slots;
    int32_t* arrive;
    uint16_t* out;
    int32_t n_tickets = 0;
};

RouteTcArgs tc_args_of(const Layout& L, unsigned char* w)
{
    RouteTcArgs c;
    c.wgt = reinterpret_cast<uint16_t*>(w + L.tc_wgt);
    c.wpart = reinterpret_cast<float*>(w + L.tc_wnorm);
    c.n_exact = reinterpret_cast<int32_t*>(w + L.tc_nflag);
    c.bound = reinterpret_cast<float*>(w + L.tc_tok);
    c.fast = reinterpret_cast<float*>(w + L.tc_cand);
    c.flag_tok = reinterpret_cast<int32_t*>(w + L.tc_ftok);
    c.flag_cand = reinterpret_cast<uint64_t*>(w + L.tc_fcand);
    c.flag_sel = reinterpret_cast<int32_t*>(w + L.tc_fsel);
    c.flag_selv = reinterpret_cast<float*>(w + L.tc_fselv);
    c.pairs = reinterpret_cast<int32_t*>(w + L.tc_pairs);
    c.lg_buf = reinterpret_cast<float*>(w + L.tc_lg);
    return c;
}

moe_status run_expert_gemms(const moe_dims& d, int32_t M, int32_t F, int32_t G, int32_t k,
                            const uint16_t* x, const uint16_t* x_rows, const int32_t* src_row,
                            const int32_t* tile_start, const int32_t* offsets, const uint16_t* W1,
                            const uint16_t* W3, const uint16_t* W2, const float* topk_w, float* slot,
                            uint16_t* h, uint32_t* err, int sms, cudaStream_t s, moe_event_t ev_mid,
                            const FusedCombine& fc = FusedCombine{false, 0, 0, nullptr, nullptr},
                            bool cp_gather = false, int32_t* ready = nullptr, int cta_group0 = 1,
                            int cta_group1 = 1, int32_t* copy_ready = nullptr, uint16_t* copy_dst = nullptr)
{
    if (M == 0) {
        if (ev_mid) MOE_TRY(cudaEventRecord((cudaEvent_t)ev_mid, s));
        return MOE_OK;
    }
    CUtensorMap mx, m1, m3, mh, m2;
    const bool dense = (x_rows != nullptr);
    const bool ok_a = dense ? make_map_a(&mx, x_rows, (uint64_t)d.H, (uint64_t)M, 128)
                            : make_map_a(&mx, x, (uint64_t)d.H, (uint64_t)d.T, 1);
    if (!ok_a ||
        !make_map_b(&m1, W1, (uint64_t)F, (uint64_t)G * d.H) ||
        !make_map_b(&m3, W3, (uint64_t)F, (uint64_t)G * d.H) ||
        !make_map_a(&mh, h, (uint64_t)F, (uint64_t)M, 128) ||
        !make_map_b(&m2, W2, (uint64_t)d.H, (uint64_t)G * F))
        return MOE_ERR_CUDA;
    GemmArgs a{};
    a.M = M;
    a.G = G;
    a.k = k;
    a.T = d.T;
    a.tile_start = tile_start;
    a.offsets = offsets;
    a.src_row = src_row;
    a.err = err;
    // GEMM0 + SwiGLU: [rows, H] x [H, F] (W1 and W3) -> h [rows, F]
    a.N = F;
    a.K = d.H;
    a.h_out = reinterpret_cast<__nv_bfloat16*>(h);
    a.x = x;
    if (ready && dense) {
        // both GEMMs in one launch: GEMM1 tiles wait for their rows of h
        GemmArgs b = a;
        b.N = d.H;
        b.K = F;
        b.h_out = nullptr;
        b.topk_w = topk_w;
        b.slot = slot;
        b.slot_j0 = fc.on ? fc.slot_j0 : 0;
        b.n_slots = fc.n_slots;
        b.n_tickets = fc.n_tickets ? fc.n_tickets : fc.n_slots;
        b.arrive = fc.arrive;
        b.out = fc.out;
        b.ready = ready;
        b.ready_target = 4 * ((F + 127) / 128);   // 4 epilogue warps x GEMM0 N tiles
        MOE_TRY(cudaMemsetAsync(ready, 0, (size_t)((M + kTileM - 1) / kTileM + G + 1) * 4, s));
        Range r("moe/gemm0+gemm1");
        MOE_TRY(launch_grouped_gemm_fused(fc.on ? kFusedCombine : kFusedScatter, mx, m1, m3, mh, m2, a, b,
                                          sms, s));
        if (ev_mid) MOE_TRY(cudaEventRecord((cudaEvent_t)ev_mid, s));
        return MOE_OK;
    }
    if (copy_ready) {
        // GEMM0's copy warps fill x_perm (copy_dst) from x while the GEMM runs
        if (!dense || !src_row || !tile_start || !copy_dst) return MOE_ERR_INVALID_ARG;
        MOE_TRY(cudaMemsetAsync(copy_ready, 0, (size_t)((M + kTileM - 1) / kTileM + G + 1) * 4, s));
        a.copy_ready = copy_ready;
        a.copy_dst = copy_dst;
    }
    Range r("moe/gemm0");
    MOE_TRY(launch_grouped_gemm(dense ? kGemm0Dense : cp_gather ? kGemm0CpGather : kGemm0Gather, mx, m1,
                                m3, a, sms, s, dense ? cta_group0 : 1));
    r.next("moe/gemm1");
    a.copy_ready = nullptr;
    a.copy_dst = nullptr;
    if (ev_mid) MOE_TRY(cudaEventRecord((cudaEvent_t)ev_mid, s));
    // GEMM1 + weighted scatter: h [rows, F] x W2 [F, H] -> slot[rank][token]
    a.N = d.H;
    a.K = F;
    a.h_out = nullptr;
    a.topk_w = topk_w;
    a.slot = slot;
    a.slot_j0 = fc.on ? fc.slot_j0 : 0;
    a.n_slots = fc.n_slots;
    a.n_tickets = fc.n_tickets ? fc.n_tickets : fc.n_slots;
    a.arrive = fc.arrive;
    a.out = fc.out;
    MOE_TRY(launch_grouped_gemm(fc.on ? kGemm1Combine : kGemm1Scatter, mh, m2, m2, a, sms, s, cta_group1));
    return MOE_OK;
}

void record(moe_event_t ev, cudaStream_t s)
{
    if (ev) cudaEventRecord((cudaEvent_t)ev, s);
}

}  // namespace

void count_launch() { g_launch_count.fetch_add(1, std::memory_order_relaxed); }

bool debug_mode()
{
    static const bool on = [] {
        const char* v = std::getenv("MOE_DEBUG");
        return v && v[0] && std::strcmp(v, "0") != 0;
    }();
    return on;
}

// The two copy streams of moe_layer_forward_host (host-to-device and
// device-to-host), created on first use for each device and kept until exit.
struct CopyStreams {
    cudaStream_t h2d = nullptr, d2h = nullptr;
};
CopyStreams g_copy[kMaxDevices];
std::mutex g_copy_mu;

bool copy_streams(cudaStream_t* h2d, cudaStream_t* d2h)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    std::lock_guard<std::mutex> lock(g_copy_mu);
    CopyStreams& c = g_copy[dev];
    if (!c.h2d && cudaStreamCreateWithFlags(&c.h2d, cudaStreamNonBlocking) != cudaSuccess) {
        c.h2d = nullptr;
        return false;
    }
    if (!c.d2h && cudaStreamCreateWithFlags(&c.d2h, cudaStreamNonBlocking) != cudaSuccess) {
        c.d2h = nullptr;
        return false;
    }
    *h2d = c.h2d;
    *d2h = c.d2h;
    return true;
}

// Chunks of moe_layer_forward_host when the caller leaves the choice to the
// library: at least 8192 tokens each, at most three. A chunk pays the layer's
// fixed costs again (launches, the GEMMs' last partial wave, another pass
// over the expert weights), which a smaller chunk does not earn back through
// the copies it hides. Measured on GB300 (ms per call, host link ~0.33 ms per
// 64 MiB each way): Mixtral-shaped T = 8192: 1 chunk 3.97, 2 chunks 3.97,
// 4 chunks 4.77 (the layer alone: 3.28 ms at T = 8192, 1.80 at T = 4096);
// DeepSeek-shaped T = 32768: 1 chunk 3.99, 2: 3.47, 3: 3.42, 4: 3.50;
// Qwen2-shaped T = 4096: 1 chunk 2.76, 2: 3.08.
int32_t host_chunks_of(const moe_dims& d)
{
    const int64_t n = d.T / 8192;
    return (int32_t)(n < 1 ? 1 : n > 3 ? 3 : n);
}

moe_status check_dims(const moe_dims* d)
{
    if (!d) return MOE_ERR_INVALID_ARG;
    if (d->T < 0 || d->H <= 0 || d->F <= 0 || d->E <= 0 || d->k <= 0 || d->F_shared < 0)
        return MOE_ERR_INVALID_ARG;
    if (d->k > d->E) return MOE_ERR_INVALID_ARG;
    if (d->k > 8 || d->E > 256) return MOE_ERR_UNSUPPORTED;
    if (d->H % 64 || d->F % 64 || d->F_shared % 64) return MOE_ERR_UNSUPPORTED;
    if (d->T * (int64_t)d->k >= ((int64_t)1 << 31)) return MOE_ERR_UNSUPPORTED;
    if ((int64_t)d->E * d->H >= ((int64_t)1 << 31) || (int64_t)d->E * d->F >= ((int64_t)1 << 31))
        return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

}  // namespace moe

namespace moe {

// The layer call with an optional router override (router_force >= 0): the
// host-buffer call runs every chunk with the router kernel family the whole
// batch would take, so that a chunk's gate weights are the whole batch's
// (the FMA routers share their bits; the tensor-core router's proven tokens
// take weights from its own logits).
moe_status layer_forward_impl(const moe_dims* dims, const moe_bf16* x, const moe_bf16* Wg, const float* bias,
                              const moe_gating* gating, const moe_bf16* W1, const moe_bf16* W3,
                              const moe_bf16* W2, const moe_bf16* W1s, const moe_bf16* W3s, const moe_bf16* W2s,
                              moe_bf16* out, const moe_routing_out* routing, void* ws, size_t ws_bytes,
                              const moe_stage_events* events, moe_stream_t stream, int router_force)
{
    MOE_TRY_STATUS(check_dims(dims));
    MOE_TRY_STATUS(check_ws(*dims, ws, ws_bytes));
    const moe_dims& d = *dims;
    if (d.T == 0) return MOE_OK;
    if (!x || !Wg || !W1 || !W3 || !W2 || !out) return MOE_ERR_INVALID_ARG;
    if (d.F_shared > 0 && (!W1s || !W3s || !W2s)) return MOE_ERR_INVALID_ARG;
    const void* ptrs[] = {x, Wg, W1, W3, W2, out};
    for (const void* p : ptrs)
        if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
    if (d.F_shared > 0 && (!aligned16(W1s) || !aligned16(W3s) || !aligned16(W2s)))
        return MOE_ERR_INVALID_ARG;
    const moe_bf16* shared_gate = gating ? gating->shared_gate : nullptr;
    if (shared_gate && (d.F_shared == 0 || !aligned16(shared_gate))) return MOE_ERR_INVALID_ARG;
    const int sms = num_sms_current();
    if (sms <= 0) return MOE_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    const Layout L = layout_of(d);
    unsigned char* w = bytes(ws);
    uint32_t* err = reinterpret_cast<uint32_t*>(w + L.err);
    auto pick_i = [&](int32_t* user, size_t off) { return user ? user : reinterpret_cast<int32_t*>(w + off); };
    int32_t* idx = pick_i(routing ? routing->topk_idx : nullptr, L.idx);
    float* tw = (routing && routing->topk_w) ? routing->topk_w : reinterpret_cast<float*>(w + L.w);
    int32_t* counts = pick_i(routing ? routing->counts : nullptr, L.counts);
    int32_t* offsets = pick_i(routing ? routing->offsets : nullptr, L.offsets);
    int32_t* src = pick_i(routing ? routing->src_row : nullptr, L.src);
    int32_t* inv = pick_i(routing ? routing->inv_pos : nullptr, L.inv);
    int32_t* tile = reinterpret_cast<int32_t*>(w + L.tile);
    float* slot = reinterpret_cast<float*>(w + L.slot);
    const int64_t R = d.T * d.k;
    const int32_t n_slots = d.k + (d.F_shared > 0 ? 1 : 0);
    int32_t* arrive = reinterpret_cast<int32_t*>(w + L.arrive);
    moe_plan plan = plan_of(d);
    if (router_force == MOE_ROUTER_TENSOR && route_tc_supported(d.T, d.H, d.E))
        plan.router = MOE_ROUTER_TENSOR;
    else if (router_force >= 0 && router_force != MOE_ROUTER_TENSOR)
        plan.router = route_variant(d.H, d.E, /*has_logits=*/true);
    const bool fused = plan.combine == MOE_COMBINE_FUSED;
    // GEMM1 counts contributions per (token, 256-column tile); with a shared
    // expert its GEMM1 runs last and is the only arrival (no counting)
    if (fused && d.F_shared == 0)
        MOE_TRY(cudaMemsetAsync(arrive, 0, (size_t)d.T * ((d.H + 255) / 256) * 4, s));

    Range layer_range("moe/layer_forward");
    Range stage("moe/route");
    record(events ? events->before_route : nullptr, s);
    RouteArgs ra{x, Wg, bias, idx, tw, d.T, d.H, d.E, d.k};
    ra.renorm = gating ? (gating->renormalize != 0) : 1;
    ra.err = err;
    ra.logits = reinterpret_cast<float*>(w + L.logits);
    if (plan.router == MOE_ROUTER_TENSOR)
        MOE_TRY(launch_route_tc(ra, tc_args_of(L, w), sms, s));
    else
        MOE_TRY(launch_route(ra, sms, s));

    stage.next("moe/permute");
    record(events ? events->before_permute : nullptr, s);
    PermuteArgs pa{idx, counts, offsets, src, inv, tile, reinterpret_cast<int32_t*>(w + L.hist), err,
                   R, d.E};
    MOE_TRY(launch_permute(pa, s));

    const bool permuted = (plan.gemm0_a == MOE_GEMM0_A_PERMUTED);
    const bool cp_gather = (plan.gemm0_a == MOE_GEMM0_A_CP_GATHER);
    uint16_t* xp = reinterpret_cast<uint16_t*>(w + L.xp);
    // x_perm: copied by GEMM0's copy warps while it runs, or by a kernel first
    const bool copy_inline = permuted && plan.x_perm_copy == MOE_X_PERM_COPY_INLINE;
    if (permuted && !copy_inline)
        MOE_TRY(launch_scatter_rows(x, idx, inv, offsets + d.E, xp, d.T, d.H, d.k, d.E, err, sms, s));

    // both routed GEMMs in one launch (dense A only)
    const bool fuse_gemms = plan.gemm_fusion == MOE_GEMM_FUSION_ON;

    stage.next("moe/experts");
    record(events ? events->before_gemm0 : nullptr, s);
    MOE_TRY_STATUS(run_expert_gemms(d, (int32_t)R, d.F, d.E, d.k, x, permuted ? xp : nullptr, src,
                                    tile, offsets, W1, W3, W2, tw, slot,
                                    reinterpret_cast<uint16_t*>(w + L.h), err, sms, s,
                                    events ? events->before_gemm1 : nullptr,
                                    // with a shared expert, only its GEMM1 (the last) combines
                                    FusedCombine{fused && d.F_shared == 0, 0, n_slots, arrive, out}, cp_gather,
                                    fuse_gemms ? reinterpret_cast<int32_t*>(w + L.ready) : nullptr,
                                    plan.cta_group, plan.cta_group_gemm1,
                                    copy_inline ? reinterpret_cast<int32_t*>(w + L.ready) : nullptr,
                                    copy_inline ? xp : nullptr));

    stage.next("moe/shared_expert");
    record(events ? events->before_shared : nullptr, s);
    if (d.F_shared > 0) {
        // the sigmoid gate, if any, is the shared expert's row weight in GEMM1
        float* sgate = nullptr;
        if (shared_gate) {
            sgate = reinterpret_cast<float*>(w + L.sgate);
            MOE_TRY(launch_shared_gate(x, shared_gate, sgate, d.T, d.H, sms, s));
        }
        // identity dispatch: every token, in token order, weight 1
        MOE_TRY_STATUS(run_expert_gemms(d, (int32_t)d.T, d.F_shared, 1, 1, x,
                                        (permuted || cp_gather) ? x : nullptr,
                                        nullptr, nullptr, nullptr, W1s, W3s, W2s, sgate,
                                        fused ? slot : slot + (size_t)d.k * d.T * d.H,
                                        reinterpret_cast<uint16_t*>(w + L.hs), err, sms, s, nullptr,
                                        // every routed slot is written: one arrival each
                                        FusedCombine{fused, d.k, n_slots, arrive, out, 1}, false, nullptr,
                                        (permuted || cp_gather) ? cta_group_for(d.T, 1, false) : 1,
                                        cta_group_for(d.T, 1, true)));
    }

    stage.next("moe/combine");
    record(events ? events->before_combine : nullptr, s);
    if (!fused)   // else GEMM1's epilogue finished it (the last contribution)
        MOE_TRY(launch_combine(slot, n_slots, out, d.T, d.H, sms, s));
    record(events ? events->after_combine : nullptr, s);
    return finish(cudaSuccess, ws, s);
}

}  // namespace moe

using namespace moe;

extern "C" {

int moe_version(void) { return kVersion; }

uint64_t moe_launch_count(void) { return g_launch_count.load(std::memory_order_relaxed); }

const char* moe_status_string(int status)
{
    switch (status) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: invalid argument";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: shape not supported";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE: workspace missing, too small or misaligned";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA: a CUDA call failed";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT: a bounded device wait ran out";
    case MOE_ERR_DEVICE_BOUNDS: return "MOE_ERR_DEVICE_BOUNDS: a device index check failed";
    default: return "unknown moe_status";
    }
}

moe_status moe_set_option(int option, int value)
{
    if (option == MOE_OPT_GEMM0_A) {
        if (value != MOE_GEMM0_A_PERMUTED && value != MOE_GEMM0_A_TMA_GATHER &&
            value != MOE_GEMM0_A_CP_GATHER)
            return MOE_ERR_INVALID_ARG;
        g_gemm0_a.store(value);
        return MOE_OK;
    }
    if (option == MOE_OPT_COMBINE) {
        if (value != MOE_COMBINE_AUTO && value != MOE_COMBINE_FUSED && value != MOE_COMBINE_SEPARATE)
            return MOE_ERR_INVALID_ARG;
        g_combine.store(value);
        return MOE_OK;
    }
    if (option == MOE_OPT_GEMM_FUSION) {
        if (value != MOE_GEMM_FUSION_AUTO && value != MOE_GEMM_FUSION_ON && value != MOE_GEMM_FUSION_OFF)
            return MOE_ERR_INVALID_ARG;
        g_gemm_fusion.store(value);
        return MOE_OK;
    }
    if (option == MOE_OPT_CTA_GROUP) {
        if (value != MOE_CTA_GROUP_AUTO && value != MOE_CTA_GROUP_ONE && value != MOE_CTA_GROUP_PAIR)
            return MOE_ERR_INVALID_ARG;
        g_cta_group.store(value);
        return MOE_OK;
    }
    if (option == MOE_OPT_X_PERM_COPY) {
        if (value != MOE_X_PERM_COPY_AUTO && value != MOE_X_PERM_COPY_INLINE && value != MOE_X_PERM_COPY_KERNEL)
            return MOE_ERR_INVALID_ARG;
        g_x_perm_copy.store(value);
        return MOE_OK;
    }
    if (option == MOE_OPT_ROUTER) {
        if (value != MOE_ROUTER_OPT_AUTO && value != MOE_ROUTER_OPT_FMA && value != MOE_ROUTER_OPT_TENSOR)
            return MOE_ERR_INVALID_ARG;
        g_router.store(value);
        return MOE_OK;
    }
    return MOE_ERR_INVALID_ARG;
}

int moe_get_option(int option)
{
    if (option == MOE_OPT_GEMM0_A) return g_gemm0_a.load();
    if (option == MOE_OPT_COMBINE) return g_combine.load();
    if (option == MOE_OPT_GEMM_FUSION) return g_gemm_fusion.load();
    if (option == MOE_OPT_CTA_GROUP) return g_cta_group.load();
    if (option == MOE_OPT_X_PERM_COPY) return g_x_perm_copy.load();
    if (option == MOE_OPT_ROUTER) return g_router.load();
    return -1;
}

moe_status moe_layer_plan(const moe_dims* dims, moe_plan* plan)
{
    MOE_TRY_STATUS(check_dims(dims));
    if (!plan) return MOE_ERR_INVALID_ARG;
    *plan = plan_of(*dims);
    return MOE_OK;
}

size_t moe_workspace_size(const moe_dims* dims)
{
    if (check_dims(dims) != MOE_OK) return 0;
    return layout_of(*dims).total;
}

moe_status moe_check(void* ws, moe_stream_t stream)
{
    if (!ws) return MOE_ERR_WORKSPACE;
    cudaStream_t s = (cudaStream_t)stream;
    uint32_t word = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemcpy(&word, ws, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
    if (word != 0 && cudaMemset(ws, 0, sizeof word) != cudaSuccess) return MOE_ERR_CUDA;
    if (word & MOE_DEV_ERR_TIMEOUT) return MOE_ERR_TIMEOUT;
    if (word & MOE_DEV_ERR_BAD_EXPERT) return MOE_ERR_INVALID_ARG;
    if (word & MOE_DEV_ERR_BOUNDS) return MOE_ERR_DEVICE_BOUNDS;
    return MOE_OK;
}

moe_status moe_route(const moe_dims* dims, const moe_bf16* x, const moe_bf16* Wg, const float* bias,
                     int32_t* topk_idx, float* topk_w, moe_stream_t stream)
{
    return moe_route_ex(dims, x, Wg, bias, nullptr, topk_idx, topk_w, stream);
}

moe_status moe_route_ex(const moe_dims* dims, const moe_bf16* x, const moe_bf16* Wg, const float* bias,
                        const moe_gating* gating, int32_t* topk_idx, float* topk_w, moe_stream_t stream)
{
    MOE_TRY_STATUS(check_dims(dims));
    if (dims->T == 0) return MOE_OK;
    if (!x || !Wg || !topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(Wg)) return MOE_ERR_INVALID_ARG;
    const int sms = num_sms_current();
    if (sms <= 0) return MOE_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    Range r("moe/route");
    RouteArgs a{x, Wg, bias, topk_idx, topk_w, dims->T, dims->H, dims->E, dims->k};
    a.renorm = gating ? (gating->renormalize != 0) : 1;
    return finish(launch_route(a, sms, s), nullptr, s);
}

moe_status moe_permute(const moe_dims* dims, const int32_t* topk_idx, int32_t* counts,
                       int32_t* offsets, int32_t* src_row, int32_t* inv_pos, const moe_bf16* x,
                       moe_bf16* x_perm, void* ws, size_t ws_bytes, moe_stream_t stream)
{
    MOE_TRY_STATUS(check_dims(dims));
    MOE_TRY_STATUS(check_ws(*dims, ws, ws_bytes));
    if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
    const int64_t R = dims->T * dims->k;
    if (R > 0 && (!topk_idx || !src_row || !inv_pos)) return MOE_ERR_INVALID_ARG;
    if (x_perm && (!x || !aligned16(x) || !aligned16(x_perm))) return MOE_ERR_INVALID_ARG;
    const int sms = num_sms_current();
    if (sms <= 0) return MOE_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    const Layout L = layout_of(*dims);
    uint32_t* err = reinterpret_cast<uint32_t*>(bytes(ws) + L.err);
    PermuteArgs a{topk_idx, counts, offsets, src_row, inv_pos,
                  reinterpret_cast<int32_t*>(bytes(ws) + L.tile),
                  reinterpret_cast<int32_t*>(bytes(ws) + L.hist), err, R, dims->E};
    Range r("moe/permute");
    MOE_TRY(launch_permute(a, s));
    if (x_perm)
        MOE_TRY(launch_scatter_rows(x, topk_idx, inv_pos, offsets + dims->E, x_perm, dims->T, dims->H, dims->k,
                                    dims->E, err, sms, s));
    return finish(cudaSuccess, ws, s);
}

moe_status moe_expert_ffn(const moe_dims* dims, const moe_bf16* x, const int32_t* src_row,
                          const int32_t* offsets, const moe_bf16* W1, const moe_bf16* W3,
                          const moe_bf16* W2, const float* topk_w, float* slot, void* ws,
                          size_t ws_bytes, moe_stream_t stream)
{
    MOE_TRY_STATUS(check_dims(dims));
    MOE_TRY_STATUS(check_ws(*dims, ws, ws_bytes));
    if (dims->T == 0) return MOE_OK;
    if (!x || !W1 || !W3 || !W2 || !slot) return MOE_ERR_INVALID_ARG;
    if (!offsets && dims->E != 1) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(W1) || !aligned16(W3) || !aligned16(W2) || !aligned16(slot))
        return MOE_ERR_INVALID_ARG;
    const int sms = num_sms_current();
    if (sms <= 0) return MOE_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    const Layout L = layout_of(*dims);
    uint32_t* err = reinterpret_cast<uint32_t*>(bytes(ws) + L.err);
    int32_t* tile = nullptr;
    if (offsets) {
        tile = reinterpret_cast<int32_t*>(bytes(ws) + L.tile);
        MOE_TRY(launch_tile_table(offsets, dims->E, tile, s));
    }
    const int32_t R = (int32_t)(dims->T * dims->k);
    const uint16_t* x_rows = nullptr;
    const int a_opt = g_gemm0_a.load();
    // the layer's table decides whether both GEMMs share one launch (dense A)
    // and who copies x_perm
    const moe_plan plan = plan_of(*dims);
    uint16_t* copy_dst = nullptr;
    if (a_opt == MOE_GEMM0_A_CP_GATHER && !src_row && dims->k == 1) {
        x_rows = x;   // identity dispatch: x is already in dispatch order
    } else if (a_opt == MOE_GEMM0_A_PERMUTED) {
        if (!src_row && dims->k == 1) {
            x_rows = x;   // identity dispatch: x is already in dispatch order
        } else {
            uint16_t* xp = reinterpret_cast<uint16_t*>(bytes(ws) + L.xp);
            if (plan.x_perm_copy == MOE_X_PERM_COPY_INLINE && src_row && tile)
                copy_dst = xp;   // GEMM0's copy warps fill it
            else
                MOE_TRY(launch_gather_rows(x, src_row, offsets ? offsets + dims->E : nullptr, xp, R,
                                           dims->T, dims->H, dims->k, err, sms, s));
            x_rows = xp;
        }
    }
    const bool fuse_gemms = x_rows && plan.gemm_fusion == MOE_GEMM_FUSION_ON;
    MOE_TRY_STATUS(run_expert_gemms(*dims, R, dims->F, dims->E, dims->k, x, x_rows, src_row, tile,
                                    offsets, W1, W3, W2, topk_w, slot,
                                    reinterpret_cast<uint16_t*>(bytes(ws) + L.h), err, sms, s,
                                    nullptr, FusedCombine{false, 0, 0, nullptr, nullptr},
                                    a_opt == MOE_GEMM0_A_CP_GATHER,
                                    fuse_gemms ? reinterpret_cast<int32_t*>(bytes(ws) + L.ready) : nullptr,
                                    plan.cta_group, plan.cta_group_gemm1,
                                    copy_dst ? reinterpret_cast<int32_t*>(bytes(ws) + L.ready) : nullptr,
                                    copy_dst));
    return finish(cudaSuccess, ws, s);
}

moe_status moe_combine(const moe_dims* dims, const float* slot, int32_t n_slots, moe_bf16* out,
                       moe_stream_t stream)
{
    MOE_TRY_STATUS(check_dims(dims));
    if (dims->T == 0) return MOE_OK;
    if (!slot || !out || n_slots < 1 || n_slots > 9) return MOE_ERR_INVALID_ARG;
    if (!aligned16(slot) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
    const int sms = num_sms_current();
    if (sms <= 0) return MOE_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    Range r("moe/combine");
    return finish(launch_combine(slot, n_slots, out, dims->T, dims->H, sms, s), nullptr, s);
}

moe_status moe_layer_forward(const moe_dims* dims, const moe_bf16* x, const moe_bf16* Wg,
                             const float* bias, const moe_bf16* W1, const moe_bf16* W3,
                             const moe_bf16* W2, const moe_bf16* W1s, const moe_bf16* W3s,
                             const moe_bf16* W2s, moe_bf16* out, const moe_routing_out* routing,
                             void* ws, size_t ws_bytes, const moe_stage_events* events,
                             moe_stream_t stream)
{
    return moe_layer_forward_ex(dims, x, Wg, bias, nullptr, W1, W3, W2, W1s, W3s, W2s, out, routing,
                                ws, ws_bytes, events, stream);
}

moe_status moe_layer_forward_ex(const moe_dims* dims, const moe_bf16* x, const moe_bf16* Wg,
                                const float* bias, const moe_gating* gating, const moe_bf16* W1,
                                const moe_bf16* W3, const moe_bf16* W2, const moe_bf16* W1s,
                                const moe_bf16* W3s, const moe_bf16* W2s, moe_bf16* out,
                                const moe_routing_out* routing, void* ws, size_t ws_bytes,
                                const moe_stage_events* events, moe_stream_t stream)
{
    return layer_forward_impl(dims, x, Wg, bias, gating, W1, W3, W2, W1s, W3s, W2s, out, routing, ws, ws_bytes,
                              events, stream, -1);
}

int32_t moe_host_chunks(const moe_dims* dims)
{
    if (check_dims(dims) != MOE_OK) return 0;
    return host_chunks_of(*dims);
}

moe_status moe_layer_forward_host(const moe_dims* dims, const moe_bf16* x_host, const moe_bf16* Wg,
                                  const float* bias, const moe_bf16* W1, const moe_bf16* W3,
                                  const moe_bf16* W2, const moe_bf16* W1s, const moe_bf16* W3s,
                                  const moe_bf16* W2s, moe_bf16* out_host, moe_bf16* x_dev,
                                  moe_bf16* out_dev, int32_t n_chunks, void* ws, size_t ws_bytes,
                                  moe_stream_t stream)
{
    MOE_TRY_STATUS(check_dims(dims));
    MOE_TRY_STATUS(check_ws(*dims, ws, ws_bytes));
    const moe_dims& d = *dims;
    if (d.T == 0) return MOE_OK;
    if (!x_host || !out_host || !x_dev || !out_dev) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x_dev) || !aligned16(out_dev)) return MOE_ERR_INVALID_ARG;
    if (n_chunks < 0 || n_chunks > 64) return MOE_ERR_INVALID_ARG;
    Range range("moe/layer_forward_host");
    const int32_t n = n_chunks == 0 ? host_chunks_of(d) : n_chunks;
    // every chunk takes the router family of the whole batch
    const int batch_router = plan_of(d).router;
    // chunk c: tokens [c*base, min(T, (c+1)*base)), base a multiple of 128
    int64_t base = (d.T + n - 1) / n;
    base = (base + 127) / 128 * 128;
    const int32_t n_used = (int32_t)((d.T + base - 1) / base);
    cudaStream_t s = (cudaStream_t)stream, h2d = nullptr, d2h = nullptr;
    if (!copy_streams(&h2d, &d2h)) return MOE_ERR_CUDA;
    // events of this call (released by the runtime once they have completed)
    std::vector<cudaEvent_t> ev(2 * (size_t)n_used + 2, nullptr);
    struct Release {
        std::vector<cudaEvent_t>& e;
        ~Release()
        {
            for (cudaEvent_t x : e)
                if (x) cudaEventDestroy(x);
        }
    } release{ev};
    for (cudaEvent_t& e : ev) MOE_TRY(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
    cudaEvent_t ev_start = ev[0], ev_done = ev[1];
    // on every return, also after a failure part way, later work on the
    // caller's stream waits for every copy this call queued (so the caller may
    // reuse its buffers once the stream has drained)
    struct Join {
        cudaStream_t s, h2d, d2h;
        cudaEvent_t e_h2d, e_d2h;
        bool armed = true;
        ~Join()
        {
            if (!armed) return;
            if (cudaEventRecord(e_h2d, h2d) == cudaSuccess) cudaStreamWaitEvent(s, e_h2d, 0);
            if (cudaEventRecord(e_d2h, d2h) == cudaSuccess) cudaStreamWaitEvent(s, e_d2h, 0);
        }
    } join{s, h2d, d2h, ev_start, ev_done};   // (ev_start may be recorded again: earlier waits keep their record)
    // the copies start after the work already queued on the caller's stream
    MOE_TRY(cudaEventRecord(ev_start, s));
    MOE_TRY(cudaStreamWaitEvent(h2d, ev_start, 0));
    MOE_TRY(cudaStreamWaitEvent(d2h, ev_start, 0));
    const size_t row = (size_t)d.H * sizeof(moe_bf16);
    for (int32_t c = 0; c < n_used; ++c) {
        const int64_t t0 = c * base, tc = std::min<int64_t>(base, d.T - t0);
        MOE_TRY(cudaMemcpyAsync(x_dev + t0 * d.H, x_host + t0 * d.H, (size_t)tc * row, cudaMemcpyHostToDevice,
                                h2d));
        MOE_TRY(cudaEventRecord(ev[2 + 2 * c], h2d));
    }
    for (int32_t c = 0; c < n_used; ++c) {
        const int64_t t0 = c * base, tc = std::min<int64_t>(base, d.T - t0);
        moe_dims dc = d;
        dc.T = tc;
        MOE_TRY(cudaStreamWaitEvent(s, ev[2 + 2 * c], 0));
        MOE_TRY_STATUS(layer_forward_impl(&dc, x_dev + t0 * d.H, Wg, bias, nullptr, W1, W3, W2, W1s, W3s, W2s,
                                          out_dev + t0 * d.H, nullptr, ws, ws_bytes, nullptr, stream,
                                          batch_router));
        MOE_TRY(cudaEventRecord(ev[3 + 2 * c], s));
        MOE_TRY(cudaStreamWaitEvent(d2h, ev[3 + 2 * c], 0));
        MOE_TRY(cudaMemcpyAsync(out_host + t0 * d.H, out_dev + t0 * d.H, (size_t)tc * row, cudaMemcpyDeviceToHost,
                                d2h));
    }
    // later work on the caller's stream waits for the last copy to the host
    // (the copies to the device are done: every chunk's layer call waited on them)
    join.armed = false;
    MOE_TRY(cudaEventRecord(ev_done, d2h));
    MOE_TRY(cudaStreamWaitEvent(s, ev_done, 0));
    return finish(cudaSuccess, ws, s);
}

moe_status moe_selftest_route_tc(const moe_dims* dims, const moe_bf16* x, const moe_bf16* Wg,
                                 const float* bias, int32_t renormalize, int32_t force_exact,
                                 int32_t* topk_idx, float* topk_w, float* fast_logits,
                                 float* fast_bound, int64_t* n_exact, void* ws, size_t ws_bytes,
                                 moe_stream_t stream)
{
    MOE_TRY_STATUS(check_dims(dims));
    MOE_TRY_STATUS(check_ws(*dims, ws, ws_bytes));
    const moe_dims& d = *dims;
    if (!route_tc_supported(d.T, d.H, d.E)) return MOE_ERR_UNSUPPORTED;
    if (!x || !Wg || !topk_idx || !topk_w || !aligned16(x) || !aligned16(Wg)) return MOE_ERR_INVALID_ARG;
    if ((fast_logits == nullptr) != (fast_bound == nullptr)) return MOE_ERR_INVALID_ARG;
    const int sms = num_sms_current();
    if (sms <= 0) return MOE_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    const Layout L = layout_of(d);
    unsigned char* w = bytes(ws);
    RouteArgs ra{x, Wg, bias, topk_idx, topk_w, d.T, d.H, d.E, d.k};
    ra.renorm = renormalize != 0;
    ra.err = reinterpret_cast<uint32_t*>(w + L.err);
    RouteTcArgs c = tc_args_of(L, w);
    c.force_exact = force_exact != 0;
    c.dbg_fast = fast_logits;
    c.dbg_bound = fast_bound;
    MOE_TRY(launch_route_tc(ra, c, sms, s));
    if (n_exact) {
        int32_t n = 0;
        MOE_TRY(cudaMemcpyAsync(&n, c.n_exact, sizeof n, cudaMemcpyDeviceToHost, s));
        MOE_TRY(cudaStreamSynchronize(s));
        *n_exact = n;
    }
    return finish(cudaSuccess, ws, s);
}

}  // extern "C"
