// grouped_gemm.cu -- the two expert GEMMs of the layer on the 5th-generation
// tensor cores (tcgen05 + TMEM), one persistent warp-specialised kernel
// template with two epilogues.
//
// The COMET page splits the first expert GEMM ("Layer 0") along the token
// dimension M and the second ("Layer 1") along the hidden dimension N
// ("COMET's Technical Principles", "Tensor Decomposition"), and runs the GEMM
// thread blocks on asynchronous TMA loads ("Thread Block Isolation"). Here,
// on one GPU with every expert local:
//   GEMM0 + SwiGLU: M tiles are 128 dispatched rows of one expert. Two ways to
//     fetch those token rows (the A operand):
//       kGemm0Dense  - one TMA box per stage from x_perm, the token rows
//                      already gathered into dispatch order by the permute
//                      step (an HBM-bound copy);
//       kGemm0Gather - the producer warp gathers the rows of x itself with
//                      TMA gather4 (4 rows per instruction, indices from
//                      src_row), so no permuted copy of x is written;
//       kGemm0CpGather - a second producer warp gathers the rows with 16-byte
//                      cp.async copies straight into the 128-byte-swizzled
//                      tile (32 per lane per stage), waits for them two stages
//                      later, fences them into the async proxy and only then
//                      arrives on the stage's barrier (which also counts the
//                      TMA bytes of B). No x_perm round trip through HBM.
//     Both gather forms measured ~0.5 PFLOP/s on GB300 against ~1.7 for the
//     dense form: 128 scattered 128-byte rows per stage do not arrive fast
//     enough for one CTA, whatever issues them. kGemm0Dense is the default.
//     B is [W1 | W3] for one 128-wide slice of F: one 128x256 MMA tile gives
//     both x W1 and x W3, and the epilogue writes h = silu(x W1) * (x W3) in
//     bf16.
//   GEMM1 + weighted scatter (mode kGemm1Scatter): A = h rows (plain TMA tile),
//     B = W2 for one 256-wide slice of H (the N split). The epilogue scales
//     each row by its gate weight and writes it to slot[rank][token] (f32):
//     every slot is written exactly once, so the later combine is a fixed
//     rank-order sum with no float atomics.
//   GEMM1 + combine (mode kGemm1Combine): the same, then each row takes an
//     integer ticket for its (token, N tile); the row that takes the last of
//     the n_slots tickets sums the token's slots in rank order (fp32, the
//     same left fold as the separate combine kernel) and writes the bf16
//     output. Which row is last depends on scheduling; the sum does not.
//
// Kernel shape: one CTA per SM (224 threads, ~221 KB of shared memory),
// persistent over a static schedule of (expert, N tile, M tile) work items
// read from the device tile table (no host sync). Roles:
//   warp 0      TMA producer: 4-stage ring of {A 128x64, B 64x256} bf16 tiles,
//               128-byte swizzle, one mbarrier pair per stage.
//   warp 1      TMEM allocator (512 columns) and MMA issuer (one thread):
//               tcgen05.mma.cta_group::1.kind::f16, M=128 N=256 K=16, f32
//               accumulators in TMEM, double-buffered (2 x 256 columns) so the
//               epilogue of one tile overlaps the main loop of the next.
//   warps 2..5  epilogue: tcgen05.ld 32 lanes x 32 columns at a time.
//   warp 6      cp.async row gather (kGemm0CpGather), or the dispatch copy
//               x -> x_perm inside a kGemm0Dense launch (copy_ready set): 4 KB
//               pieces through a 6-slot shared-memory ring, counted per
//               128-row tile; the producer waits for a tile's count.
// CTA pairs (template argument PAIR; dense-A GEMM0 and GEMM1): a 2-CTA cluster
// shares one tcgen05.mma.cta_group::2 of M=256 N=256 K=16. Each CTA stages its
// 128 rows of A and half of B's columns (6 stages of 32 KB); both CTAs' TMA
// boxes complete on the rank-0 CTA's stage barrier; rank 0 issues the MMAs and
// its commits arrive on the barriers of both CTAs (multicast); the peer's
// epilogue releases a TMEM buffer on rank 0's barrier. TMEM (512 columns) is
// one collective allocation at the same address in both CTAs. Work items are
// 256-row tiles; rank 0 takes the first 128 rows, rank 1 the rest.
// Every wait is bounded (ptx.cuh); on a timeout the CTA drains what it
// issued, frees its TMEM and exits with the error recorded.
#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int BM = kTileM;   // 128
constexpr int BN = 256;      // MMA N (GEMM0: 128 of W1 + 128 of W3)
constexpr int BK = kGemmBK;  // K per stage: one A row of BK bf16 = one swizzle span
constexpr int A_ROW = BK * 2;                // bytes: 64 (64-byte swizzle) or 128 (128-byte)
static_assert(BK == 32 || BK == 64, "A rows are one 64- or 128-byte swizzle span");
constexpr int A_BYTES = BM * BK * 2;         // 8 KB (BK 32) or 16 KB
constexpr int B_CHUNK_BYTES = BK * 128;      // one 64-column slice of B: BK k-rows x 128 B
constexpr int NUM_THREADS = 224;   // 7 warps: TMA, MMA, 4 x epilogue, row gather
constexpr int GATHER_LAG = 2;      // stages a gathered A tile is given to land
constexpr int MAX_GROUPS = 257;
constexpr int TMEM_COLS = 512;
constexpr int COPY_PIECE = 4096;   // dispatch copy: bytes per piece of a row
constexpr int COPY_SLOTS = 6;      // dispatch copy: pieces in flight per CTA

// One CTA per MMA (PAIR false): a stage holds A 128 x BK and all BN columns of
// B. A CTA pair (PAIR true, tcgen05 cta_group::2): one MMA of 256 x BN over
// both CTAs, each staging its 128 rows of A and its BN / 2 columns of B, so a
// stage is 32 KB instead of 48 KB and 6 stages fit where 4 did.
template <bool PAIR>
struct Cfg {
    static constexpr int B_COLS = PAIR ? BN / 2 : BN;   // columns of B staged by this CTA
    static constexpr int B_BYTES = B_COLS * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = PAIR ? 6 : (BK == 32 ? 9 : 4);
    static constexpr int TILE_ROWS = PAIR ? 2 * BM : BM;   // rows of one work item
    static constexpr uint32_t IDESC = idesc_bf16_f32(TILE_ROWS, BN, /*a_mn_major=*/false, /*b_mn_major=*/true);
};

template <int STAGES>
struct SmemTail {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
    int tile_start[MAX_GROUPS + 1];
    int offsets[MAX_GROUPS + 1];
    int tok[BM];                      // kGemm0CpGather: token of each row of the current tile
    int tile128[MAX_GROUPS + 1];      // first 128-row tile of each group (the copy counters' index)
    uint64_t cbar[COPY_SLOTS];        // dispatch copy: one barrier per ring slot
};

// The dispatch copy's ring follows the tail, 128-byte aligned.
template <bool PAIR>
__host__ __device__ constexpr size_t ring_offset()
{
    return ((size_t)Cfg<PAIR>::STAGES * Cfg<PAIR>::STAGE_BYTES + sizeof(SmemTail<Cfg<PAIR>::STAGES>) + 127) &
           ~(size_t)127;
}
template <bool PAIR>
__host__ __device__ constexpr size_t smem_bytes()
{
    return 1024 /*align slack*/ + ring_offset<PAIR>() + (size_t)COPY_SLOTS * COPY_PIECE;
}
static_assert(smem_bytes<false>() <= 227 * 1024 && smem_bytes<true>() <= 227 * 1024, "shared memory");

struct Work {
    int g, row0, rows, n_tile;
};

// Work item w of the static schedule: expert-major, then N tile, then M tile.
// ts is the table of TILE_ROWS-row tiles; this CTA's rows start `sub` rows into
// the tile (a pair's rank-1 CTA: 128) and may be none (rows <= 0).
template <int TILE_ROWS>
__device__ __forceinline__ Work decode_work(int w, int n_tiles, const int* ts, const int* offs, int G, int sub)
{
    int lo = 0, hi = G;   // ts[lo]*n <= w < ts[hi]*n
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (ts[mid] * n_tiles <= w) lo = mid; else hi = mid;
    }
    Work r;
    r.g = lo;
    const int mt = ts[lo + 1] - ts[lo];
    const int wl = w - ts[lo] * n_tiles;
    r.n_tile = wl / mt;
    const int ml = wl - r.n_tile * mt;
    r.row0 = offs[lo] + ml * TILE_ROWS + sub;
    r.rows = min(BM, offs[lo + 1] - r.row0);
    return r;
}

// The fused combine of the rows whose (token, 256-column tile) this warp
// finished (bit i of `todo`: lane i's row, token t on that lane): out[t, n0 +
// 8l .. 8l+7] = bf16 of the left fold slot[0] + slot[1] + ... + slot[ns-1] in
// fp32, lane l taking columns 8l .. 8l+7, for ns <= NS. Every slot load of a
// batch of CB rows is issued before the first add, so a batch costs one
// memory round trip (a fold that loads slot j only after adding slot j-1
// costs ns of them).
template <int NS, int CB>
__device__ __forceinline__ void combine_rows(unsigned todo, int64_t t, const float* slot, uint16_t* out, int n0,
                                             int N1, int64_t T, int ns)
{
    const int c = 8 * (threadIdx.x & 31);
    const int64_t TN = T * (int64_t)N1;
    const bool col_ok = n0 + c < N1;
    while (todo) {
        int64_t tt[CB];
#pragma unroll
        for (int u = 0; u < CB; ++u) {
            tt[u] = -1;
            if (todo) {   // warp-uniform: todo is a ballot
                const int src_lane = __ffs(todo) - 1;
                todo &= todo - 1;
                tt[u] = __shfl_sync(0xffffffffu, t, src_lane);
            }
        }
        if (!col_ok) continue;
        float4 v[CB][NS][2];
#pragma unroll
        for (int u = 0; u < CB; ++u) {
            if (tt[u] < 0) continue;
            const float* src = slot + tt[u] * N1 + n0 + c;
#pragma unroll
            for (int j = 0; j < NS; ++j) {
                if (j < ns) {
                    v[u][j][0] = __ldcg(reinterpret_cast<const float4*>(src + j * TN));
                    v[u][j][1] = __ldcg(reinterpret_cast<const float4*>(src + j * TN + 4));
                }
            }
        }
#pragma unroll
        for (int u = 0; u < CB; ++u) {
            if (tt[u] < 0) continue;
            float4 a0 = v[u][0][0], a1 = v[u][0][1];
#pragma unroll
            for (int j = 1; j < NS; ++j) {
                if (j >= ns) break;
                a0.x = a0.x + v[u][j][0].x; a0.y = a0.y + v[u][j][0].y;
                a0.z = a0.z + v[u][j][0].z; a0.w = a0.w + v[u][j][0].w;
                a1.x = a1.x + v[u][j][1].x; a1.y = a1.y + v[u][j][1].y;
                a1.z = a1.z + v[u][j][1].z; a1.w = a1.w + v[u][j][1].w;
            }
            __nv_bfloat162 p0 = __floats2bfloat162_rn(a0.x, a0.y);
            __nv_bfloat162 p1 = __floats2bfloat162_rn(a0.z, a0.w);
            __nv_bfloat162 p2 = __floats2bfloat162_rn(a1.x, a1.y);
            __nv_bfloat162 p3 = __floats2bfloat162_rn(a1.z, a1.w);
            uint4 o;
            o.x = *reinterpret_cast<uint32_t*>(&p0);
            o.y = *reinterpret_cast<uint32_t*>(&p1);
            o.z = *reinterpret_cast<uint32_t*>(&p2);
            o.w = *reinterpret_cast<uint32_t*>(&p3);
            *reinterpret_cast<uint4*>(out + tt[u] * N1 + n0 + c) = o;
        }
    }
}

template <int MODE, bool PAIR>
__global__ void __launch_bounds__(NUM_THREADS, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                    const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmA1,
                    const __grid_constant__ CUtensorMap tmB2, const GemmArgs args, const GemmArgs args1)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t tiles_addr = (raw_addr + 1023u) & ~1023u;
    unsigned char* tiles = smem_raw + (tiles_addr - raw_addr);
    using C = Cfg<PAIR>;
    constexpr int STAGES = C::STAGES;
    constexpr int STAGE_BYTES = C::STAGE_BYTES;
    constexpr int CG = PAIR ? 2 : 1;   // tcgen05 CTA group
    SmemTail<STAGES>* st = reinterpret_cast<SmemTail<STAGES>*>(tiles + (size_t)STAGES * STAGE_BYTES);

    // FUSED: work items [0, total0) are GEMM0 (dense A) tiles, the rest GEMM1
    // tiles (args1, maps tmA1 / tmB2); a GEMM1 tile waits until every GEMM0
    // tile of its (expert, M tile) has published its rows of h
    constexpr bool FUSED = (MODE == kFusedScatter || MODE == kFusedCombine);
    constexpr bool IS_GEMM0 = (MODE == kGemm0Gather || MODE == kGemm0Dense || MODE == kGemm0CpGather);
    constexpr bool HAS_GEMM0 = IS_GEMM0 || FUSED;
    constexpr bool COMBINE = (MODE == kGemm1Combine || MODE == kFusedCombine);
    constexpr bool CP_GATHER = (MODE == kGemm0CpGather);
    constexpr bool GATHER = (MODE == kGemm0Gather);
    static_assert(!PAIR || MODE == kGemm0Dense || MODE == kGemm1Scatter || MODE == kGemm1Combine,
                  "CTA pairs run the dense-A GEMM0 and the GEMM1 modes");
    static_assert(!PAIR || BK == 64, "CTA pairs use 128-byte rows of A");
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = args.G;
    // a pair walks the schedule together: both CTAs take the same work items,
    // rank 0 the first 128 rows of each and rank 1 the next 128
    const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
    const int unit = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
    const int n_units = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;
    const int sub = (int)rank * BM;

    // ---- set-up
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            // with cp.async rows, a stage is full after the TMA bytes of B and
            // the gather warp's arrival
            mbar_init(smem_u32(&st->full[s]), CP_GATHER ? 2 : 1);
            mbar_init(smem_u32(&st->empty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&st->tfull[a]), 1);
            // the epilogue warps release a TMEM buffer: 4 here, 4 more from the peer
            mbar_init(smem_u32(&st->tempty[a]), PAIR ? 8 : 4);
        }
        mbar_init(smem_u32(&st->drain), 1);
        for (int c = 0; c < COPY_SLOTS; ++c) mbar_init(smem_u32(&st->cbar[c]), 1);
        st->abort = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB0);
        if (HAS_GEMM0) tma_prefetch_desc(&tmB1);
        if (FUSED) {
            tma_prefetch_desc(&tmA1);
            tma_prefetch_desc(&tmB2);
        }
    }
    if (warp == 1) {
        tmem_alloc<CG>(smem_u32(&st->tmem_base), TMEM_COLS);
        tmem_relinquish<CG>();
    }
    // launched with programmatic stream serialization: the set-up above is
    // on-chip only; the tile table and every operand are read after the
    // kernel before this one has completed
    pdl_wait();
    pdl_launch_dependents();
    if (PAIR) {
        // the table of 256-row tiles, from the group offsets (warp 0: a scan)
        if (warp == 0) {
            if (args.tile_start == nullptr) {
                if (lane == 0) {
                    st->offsets[0] = 0;
                    st->offsets[1] = args.M;
                    st->tile128[0] = 0;
                    st->tile128[1] = (args.M + BM - 1) / BM;
                }
            } else {
                for (int i = lane; i <= G; i += 32) {
                    st->offsets[i] = args.offsets[i];
                    st->tile128[i] = args.tile_start[i];
                }
            }
            __syncwarp();
            const int per = (G + 31) / 32;
            const int g0 = lane * per;
            auto tiles_of = [&](int g) {
                return (st->offsets[g + 1] - st->offsets[g] + C::TILE_ROWS - 1) / C::TILE_ROWS;
            };
            int mine = 0;
            for (int i = 0; i < per; ++i)
                if (g0 + i < G) mine += tiles_of(g0 + i);
            int incl = mine;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, d);
                if (lane >= d) incl += v;
            }
            int run = incl - mine;
            for (int i = 0; i < per; ++i) {
                if (g0 + i < G) {
                    st->tile_start[g0 + i] = run;
                    run += tiles_of(g0 + i);
                }
            }
            if (lane == 31) st->tile_start[G] = incl;
        }
    } else if (args.tile_start == nullptr) {
        if (threadIdx.x == 0) {
            st->tile_start[0] = st->tile128[0] = 0;
            st->tile_start[1] = st->tile128[1] = (args.M + BM - 1) / BM;
            st->offsets[0] = 0;
            st->offsets[1] = args.M;
        }
    } else {
        for (int i = threadIdx.x; i <= G; i += blockDim.x) {
            st->tile_start[i] = st->tile128[i] = args.tile_start[i];
            st->offsets[i] = args.offsets[i];
        }
    }
    tc_fence_before();
    // a pair: both CTAs' barriers are initialised before either signals the other's
    if (PAIR) cluster_sync(); else __syncthreads();
    tc_fence_after();

    const uint32_t tmem_base = st->tmem_base;
    // pass 0 (this mode's GEMM, or GEMM0 when fused) and pass 1 (GEMM1 when fused)
    const int n_out0 = HAS_GEMM0 ? BN / 2 : BN;   // output columns per tile
    const int n_tiles0 = (args.N + n_out0 - 1) / n_out0;
    const int total0 = st->tile_start[G] * n_tiles0;
    const int n_tiles1 = FUSED ? (args1.N + BN - 1) / BN : 0;
    const int total = total0 + st->tile_start[G] * n_tiles1;
    const int k_blocks0 = args.K / BK;
    const int k_blocks1 = FUSED ? args1.K / BK : 0;
    volatile int* abort = &st->abort;

    if (warp == 0) {
        // ============================ TMA producer ============================
        int stage = 0;
        uint32_t phase = 0;
        int issued = 0;
        bool ok = true;
        for (int w = unit; w < total && ok; w += n_units) {
            const bool p1 = FUSED && w >= total0;
            const int n_tiles = p1 ? n_tiles1 : n_tiles0;
            const int k_blocks = p1 ? k_blocks1 : k_blocks0;
            const Work wk = decode_work<C::TILE_ROWS>(p1 ? w - total0 : w, n_tiles, st->tile_start, st->offsets,
                                                     G, sub);
            if (p1) {
                // the rows of h this tile reads: every GEMM0 tile of (expert, M tile)
                // must have stored and published them
                const int mt = st->tile_start[wk.g] + (wk.row0 - st->offsets[wk.g]) / BM;
                bool ready = true;
                if (lane == 0) ready = wait_count(args1.ready + mt, args1.ready_target, abort, args.err);
                if (!__shfl_sync(0xffffffffu, ready, 0)) {
                    ok = false;
                    break;
                }
                if (lane == 0) asm volatile("fence.proxy.async.global;" ::: "memory");
                __syncwarp();
            }
            int tok[4] = {0, 0, 0, 0};
            if (GATHER) {
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int p = wk.row0 + min(4 * lane + r, wk.rows - 1);
                    const int f = args.src_row ? args.src_row[p] : p;
                    int t = f / args.k;
                    if (f < 0 || t >= args.T) {
                        report_error(args.err, MOE_DEV_ERR_BOUNDS);
                        t = 0;
                    }
                    tok[r] = t;
                }
            }
            if (MODE == kGemm0Dense && args.copy_ready != nullptr && wk.rows > 0) {
                // this tile's A rows come from the launch's copy warps: wait until
                // every piece of them is counted, then read them through TMA
                const int mt = st->tile128[wk.g] + (wk.row0 - st->offsets[wk.g]) / BM;
                const int ppr = (args.K * 2 + COPY_PIECE - 1) / COPY_PIECE;
                bool ready = true;
                if (lane == 0) ready = wait_count(args.copy_ready + mt, wk.rows * ppr, abort, args.err);
                if (!__shfl_sync(0xffffffffu, ready, 0)) {
                    ok = false;
                    break;
                }
                if (lane == 0) asm volatile("fence.proxy.async.global;" ::: "memory");
                __syncwarp();
            }
            const int b_row = wk.g * (p1 ? args1.K : args.K);
            for (int kb = 0; kb < k_blocks; ++kb) {
                // every lane waits; the outcome is made warp-uniform
                if (!__all_sync(0xffffffffu,
                                mbar_wait(smem_u32(&st->empty[stage]), phase ^ 1u, abort, args.err))) {
                    ok = false;
                    break;
                }
                const uint32_t full = smem_u32(&st->full[stage]);
                const uint32_t a_dst = tiles_addr + stage * STAGE_BYTES;
                const uint32_t b_dst = a_dst + A_BYTES;
                if constexpr (PAIR) {
                    // both CTAs' boxes complete on the leader's barrier, which
                    // expects the bytes of the two
                    if (lane == 0) {
                        if (rank == 0) mbar_arrive_expect_tx(full, 2 * STAGE_BYTES);
                        const uint32_t bar = mapa_shared(full, 0);
                        tma_load_2d_pair(a_dst, &tmA, kb * BK, wk.row0, bar);
                        if (HAS_GEMM0) {
                            // rank 0 stages the W1 half of B, rank 1 the W3 half
                            const CUtensorMap* mb = rank == 0 ? &tmB0 : &tmB1;
                            const int n0 = wk.n_tile * (BN / 2);
                            tma_load_2d_pair(b_dst, mb, n0, b_row + kb * BK, bar);
                            tma_load_2d_pair(b_dst + B_CHUNK_BYTES, mb, n0 + 64, b_row + kb * BK, bar);
                        } else {
                            const int n0 = wk.n_tile * BN + (int)rank * (BN / 2);
                            tma_load_2d_pair(b_dst, &tmB0, n0, b_row + kb * BK, bar);
                            tma_load_2d_pair(b_dst + B_CHUNK_BYTES, &tmB0, n0 + 64, b_row + kb * BK, bar);
                        }
                    }
                    __syncwarp();
                    ++issued;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                    continue;
                }
                if (lane == 0) mbar_arrive_expect_tx(full, CP_GATHER ? C::B_BYTES : STAGE_BYTES);
                __syncwarp();
                if (GATHER)
                    tma_gather4(a_dst + lane * 4 * A_ROW, &tmA, kb * BK, tok[0], tok[1], tok[2], tok[3], full);
                else if (!CP_GATHER && lane == 0)
                    tma_load_2d(a_dst, p1 ? &tmA1 : &tmA, kb * BK, wk.row0, full);
                if (HAS_GEMM0 && !p1) {
                    if (lane == 0) {
                        const int n0 = wk.n_tile * (BN / 2);
                        tma_load_2d(b_dst + 0 * B_CHUNK_BYTES, &tmB0, n0, b_row + kb * BK, full);
                        tma_load_2d(b_dst + 1 * B_CHUNK_BYTES, &tmB0, n0 + 64, b_row + kb * BK, full);
                        tma_load_2d(b_dst + 2 * B_CHUNK_BYTES, &tmB1, n0, b_row + kb * BK, full);
                        tma_load_2d(b_dst + 3 * B_CHUNK_BYTES, &tmB1, n0 + 64, b_row + kb * BK, full);
                    }
                } else {
                    if (lane == 0) {
                        const int n0 = wk.n_tile * BN;
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            tma_load_2d(b_dst + j * B_CHUNK_BYTES, p1 ? &tmB2 : &tmB0, n0 + 64 * j,
                                        b_row + kb * BK, full);
                    }
                }
                ++issued;
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
        }
        if (PAIR && ok) {
            // the tensor-core commits that free this CTA's stages come from the
            // leader; wait for the last of them to land before the CTA may exit
            for (int i = 0; i < STAGES; ++i) {
                if (!__all_sync(0xffffffffu,
                                mbar_wait(smem_u32(&st->empty[stage]), phase ^ 1u, abort, args.err)))
                    break;
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
        }
        if (!PAIR && !ok && lane == 0) {
            // drain: wait (bounded) for the loads still in flight
            int s = stage;
            uint32_t ph = phase;
            for (int i = 0; i < min(issued, STAGES); ++i) {
                if (s == 0) { s = STAGES - 1; ph ^= 1u; } else { --s; }
                mbar_wait_drain(smem_u32(&st->full[s]), ph);
            }
        }
    } else if (warp == 1) {
        // ============================ MMA issuer ==============================
        // (a pair: the rank-0 CTA issues for both)
        if (lane == 0 && rank == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            bool any = false;
            for (int w = unit; w < total && ok; w += n_units) {
                const int k_blocks = (FUSED && w >= total0) ? k_blocks1 : k_blocks0;
                if (!mbar_wait<PAIR>(smem_u32(&st->tempty[acc]), acc_phase ^ 1u, abort, args.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (int kb = 0; kb < k_blocks; ++kb) {
                    if (!mbar_wait(smem_u32(&st->full[stage]), phase, abort, args.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_base = tiles_addr + stage * STAGE_BYTES;
                    const uint32_t b_base = a_base + A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        // K-major A: each K step of 16 is 32 bytes further along the row
                        const uint64_t ad = BK == 64 ? smem_desc_sw128(a_base + kk * 32, 16, 1024)
                                                     : smem_desc_sw64(a_base + kk * 32, 16, 512);
                        const uint64_t bd = smem_desc_sw128(b_base + kk * 16 * 128, B_CHUNK_BYTES, 1024);
                        tc_mma_f16<CG>(d_tmem, ad, bd, C::IDESC, (kb | kk) != 0 ? 1u : 0u);
                    }
                    any = true;
                    tc_commit<CG>(smem_u32(&st->empty[stage]));
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                tc_commit<CG>(smem_u32(&st->tfull[acc]));
                if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
            }
            if (!ok && any) {
                // drain: every MMA issued so far must finish before TMEM is freed
                if (PAIR) tc_commit_pair_local(smem_u32(&st->drain));
                else tc_commit(smem_u32(&st->drain));
                mbar_wait_drain(smem_u32(&st->drain), 0);
            }
        }
        __syncwarp();
    } else if (warp == 6) {
        // ========================= A row gather (cp.async) ======================
        if (CP_GATHER) {
            int stage = 0, done_stage = 0;
            uint32_t phase = 0;
            int pending = 0;   // stages issued whose rows are not yet published
            bool ok = true;
            constexpr int CPR = A_ROW / 16;   // 16-byte chunks per A row (4 or 8)
            const int c = lane % CPR;         // this lane's chunk of a row
            const int rsub = lane / CPR;      // row within a group of 32 / CPR
            auto publish_oldest = [&]() {
                // the oldest pending stage's copies have landed (this lane's): make
                // them visible to the tensor cores, then arrive once for the warp
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&st->full[done_stage]));
                if (++done_stage == STAGES) done_stage = 0;
                --pending;
            };
            const int n_tiles = n_tiles0;
            const int k_blocks = k_blocks0;
            for (int w = blockIdx.x; w < total && ok; w += gridDim.x) {
                const Work wk = decode_work<BM>(w, n_tiles, st->tile_start, st->offsets, G, 0);
                __syncwarp();   // the previous tile's rows are no longer read
                for (int rr = lane; rr < BM; rr += 32) {
                    const int p = wk.row0 + min(rr, wk.rows - 1);
                    const int f = args.src_row ? args.src_row[p] : p;
                    int t = f / args.k;
                    if (f < 0 || t >= args.T) {
                        report_error(args.err, MOE_DEV_ERR_BOUNDS);
                        t = 0;
                    }
                    st->tok[rr] = t;
                }
                __syncwarp();
                for (int kb = 0; kb < k_blocks; ++kb) {
                    if (!__all_sync(0xffffffffu,
                                    mbar_wait(smem_u32(&st->empty[stage]), phase ^ 1u, abort, args.err))) {
                        ok = false;
                        break;
                    }
                    const uint32_t a_dst = tiles_addr + stage * STAGE_BYTES;
                    const uint16_t* xk = args.x + kb * BK + c * 8;
#pragma unroll 8
                    for (int q = 0; q < BM / (32 / CPR); ++q) {
                        const int r = (32 / CPR) * q + rsub;
                        const uint16_t* src = xk + (int64_t)st->tok[r] * args.K;
                        // the swizzle of the TMA / tensor-core layout: 16-byte chunk
                        // index XOR row bits (128-byte rows: r mod 8; 64-byte: (r/2) mod 4)
                        const int swz = BK == 64 ? (r & 7) : ((r >> 1) & 3);
                        const uint32_t dst = a_dst + r * A_ROW + ((c ^ swz) << 4);
                        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src)
                                     : "memory");
                    }
                    asm volatile("cp.async.commit_group;" ::: "memory");
                    ++pending;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                    if (pending > GATHER_LAG) {
                        asm volatile("cp.async.wait_group %0;" ::"n"(GATHER_LAG) : "memory");
                        publish_oldest();
                    }
                }
            }
            // the last stages (and, after an abort, whatever is in flight)
            asm volatile("cp.async.wait_group 0;" ::: "memory");
            while (pending > 0) publish_oldest();
        } else if (MODE == kGemm0Dense && args.copy_ready != nullptr) {
            // ===================== dispatch copy: x -> x_perm =====================
            // The rows of x_perm in 4 KB pieces, piece p = (row, part) taken by
            // CTA p mod gridDim.x, so every CTA works from the first rows on and
            // the first experts' tiles are ready first. A piece arrives in a
            // ring slot by a bulk copy, goes out with 16-byte stores, and is
            // counted on its 128-row tile after a proxy fence (the tile is read
            // back through TMA).
            unsigned char* ring = tiles + ring_offset<PAIR>();
            const uint32_t ring_addr = smem_u32(ring);
            const int64_t rows = st->offsets[G];            // rows with a valid expert
            const int row_bytes = args.K * 2;
            const int ppr = (row_bytes + COPY_PIECE - 1) / COPY_PIECE;
            const int64_t total = rows * ppr;
            const int64_t first = blockIdx.x, stride = gridDim.x;
            auto piece = [&](int64_t j, int64_t& r, int& part, int& bytes) {
                const int64_t p = first + j * stride;
                r = p / ppr;
                part = (int)(p - r * ppr);
                bytes = min(COPY_PIECE, row_bytes - part * COPY_PIECE);
                return p < total;
            };
            auto issue = [&](int64_t j) {
                int64_t r;
                int part, bytes;
                if (!piece(j, r, part, bytes) || lane != 0) return;
                const int f = args.src_row[r];
                int64_t t = f / args.k;
                if (f < 0 || t >= args.T) {
                    report_error(args.err, MOE_DEV_ERR_BOUNDS);
                    t = 0;
                }
                const int slot = (int)(j % COPY_SLOTS);
                const uint32_t bar = smem_u32(&st->cbar[slot]);
                mbar_arrive_expect_tx(bar, (uint32_t)bytes);
                bulk_load(ring_addr + slot * COPY_PIECE,
                          args.x + t * args.K + (int64_t)part * (COPY_PIECE / 2), (uint32_t)bytes, bar);
            };
            for (int q = 0; q < COPY_SLOTS; ++q) issue(q);
            // counts the pieces j0 .. j-1 (copied, not yet counted) on their tiles,
            // after one fence for all of them: lane q takes piece j0 + q
            int64_t j0 = 0;
            auto publish = [&](int64_t j_end) {
                asm volatile("fence.proxy.async.global;" ::: "memory");
                __threadfence();
                __syncwarp();
                int64_t r;
                int part, bytes;
                if (j0 + lane < j_end && piece(j0 + lane, r, part, bytes)) {
                    int lo = 0, hi = G;   // the group of row r: offsets[lo] <= r < offsets[lo + 1]
                    while (hi - lo > 1) {
                        const int mid = (lo + hi) >> 1;
                        if (st->offsets[mid] <= r) lo = mid; else hi = mid;
                    }
                    atomicAdd(args.copy_ready + st->tile128[lo] + (int)((r - st->offsets[lo]) / BM), 1);
                }
                j0 = j_end;
            };
            int64_t j = 0;
            for (;; ++j) {
                int64_t r;
                int part, bytes;
                if (!piece(j, r, part, bytes)) break;
                const int slot = (int)(j % COPY_SLOTS);
                const uint32_t parity = (uint32_t)((j / COPY_SLOTS) & 1);
                if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&st->cbar[slot]), parity, abort, args.err)))
                    break;
                // the piece into registers (at most 4 KB: 8 x 16 bytes a lane), the
                // slot refilled at once, then the stores
                const uint4* src = reinterpret_cast<const uint4*>(ring + slot * COPY_PIECE);
                const int n16 = bytes / 16;
                uint4 v[COPY_PIECE / 512];
#pragma unroll
                for (int u = 0; u < COPY_PIECE / 512; ++u)
                    if (lane + 32 * u < n16) v[u] = src[lane + 32 * u];
                __syncwarp();
                if (lane == 0) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                issue(j + COPY_SLOTS);
                uint4* dst = reinterpret_cast<uint4*>(args.copy_dst + r * args.K + (int64_t)part * (COPY_PIECE / 2));
#pragma unroll
                for (int u = 0; u < COPY_PIECE / 512; ++u)
                    if (lane + 32 * u < n16) dst[lane + 32 * u] = v[u];
                if (j + 1 - j0 == COPY_SLOTS) publish(j + 1);
            }
            publish(j);   // the last pieces (after an abort: those copied before it)
            // after an abort: the pieces still in flight land before the CTA exits
            if (lane == 0) {
                for (int64_t q = j; q < j + COPY_SLOTS; ++q) {
                    int64_t r;
                    int part, bytes;
                    if (!piece(q, r, part, bytes)) break;
                    mbar_wait_drain(smem_u32(&st->cbar[q % COPY_SLOTS]), (uint32_t)((q / COPY_SLOTS) & 1));
                }
            }
        }
    } else {
        // ============================== epilogue ==============================
        const int ew = warp & 3;               // TMEM lane quarter this warp may access
        const int r = ew * 32 + lane;          // row of the tile
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int w = unit; w < total; w += n_units) {
            const bool p1 = FUSED && w >= total0;
            const int n_tiles = p1 ? n_tiles1 : n_tiles0;
            const Work wk = decode_work<C::TILE_ROWS>(p1 ? w - total0 : w, n_tiles, st->tile_start, st->offsets,
                                                     G, sub);
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&st->tfull[acc]), acc_phase, abort, args.err)))
                break;
            tc_fence_after();
            const uint32_t t_row = tmem_base + ((uint32_t)(ew * 32) << 16) + acc * BN;
            const bool valid = r < wk.rows;
            const int p = wk.row0 + r;
            if (HAS_GEMM0 && !p1) {
                const int n0 = wk.n_tile * (BN / 2);
#pragma unroll 1
                for (int c = 0; c < BN / 2; c += 32) {
                    uint32_t va[32], vb[32];
                    tmem_ld_32x32b_x32(t_row + c, va);
                    tmem_ld_32x32b_x32(t_row + BN / 2 + c, vb);
                    tc_wait_ld();
                    if (valid && n0 + c < args.N) {
                        uint32_t packed[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const float a0 = __uint_as_float(va[2 * i]);
                            const float a1 = __uint_as_float(va[2 * i + 1]);
                            const float b0 = __uint_as_float(vb[2 * i]);
                            const float b1 = __uint_as_float(vb[2 * i + 1]);
                            const float g0 = a0 / (1.0f + __expf(-a0)) * b0;
                            const float g1 = a1 / (1.0f + __expf(-a1)) * b1;
                            __nv_bfloat162 hv = __floats2bfloat162_rn(g0, g1);
                            packed[i] = *reinterpret_cast<uint32_t*>(&hv);
                        }
                        // 64 bytes of this row: two whole-sector stores
                        __nv_bfloat16* dst = args.h_out + (int64_t)p * args.N + n0 + c;
#pragma unroll
                        for (int i = 0; i < 2; ++i)
                            st_global_v8(dst + 16 * i, packed[8 * i], packed[8 * i + 1], packed[8 * i + 2],
                                         packed[8 * i + 3], packed[8 * i + 4], packed[8 * i + 5],
                                         packed[8 * i + 6], packed[8 * i + 7]);
                    }
                }
                if constexpr (FUSED) {
                    // publish this warp's 32 rows of the tile to the GEMM1 tiles
                    // that read them with TMA (generic stores -> async-proxy reads)
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                    __threadfence();
                    __syncwarp();
                    if (lane == 0) {
                        const int mt = st->tile_start[wk.g] + (wk.row0 - st->offsets[wk.g]) / BM;
                        atomicAdd(args1.ready + mt, 1);
                    }
                }
            } else {
                const int n0 = wk.n_tile * BN;
                const int N1 = FUSED ? args1.N : args.N;
                const float* topk_w = FUSED ? args1.topk_w : args.topk_w;
                int64_t t = 0;
                int j = 0;
                float wt = 1.0f;
                bool ok_row = valid;
                if (valid) {
                    const int f = args.src_row ? args.src_row[p] : p;
                    t = f / args.k;
                    j = f - (int)t * args.k;
                    if (f < 0 || t >= args.T) {
                        report_error(args.err, MOE_DEV_ERR_BOUNDS);
                        ok_row = false;
                    } else if (topk_w) {
                        wt = topk_w[f];
                    }
                }
                float* dst_row = (FUSED ? args1.slot : args.slot) +
                                 ((int64_t)((FUSED ? args1.slot_j0 : args.slot_j0) + j) * args.T + t) * N1 + n0;
#pragma unroll 1
                for (int c = 0; c < BN; c += 32) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(t_row + c, v);
                    tc_wait_ld();
                    if (ok_row && n0 + c < N1) {
                        // 128 bytes of this row: four whole-sector stores
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            uint32_t o[8];
#pragma unroll
                            for (int u = 0; u < 8; ++u)
                                o[u] = __float_as_uint(wt * __uint_as_float(v[8 * i + u]));
                            st_global_v8(dst_row + c + 8 * i, o[0], o[1], o[2], o[3], o[4], o[5], o[6],
                                         o[7]);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                // TMEM free for the MMA (a pair's: on the leader's barrier)
                if (PAIR && rank != 0) mbar_arrive_remote(mapa_shared(smem_u32(&st->tempty[acc]), 0));
                else mbar_arrive(smem_u32(&st->tempty[acc]));
            }
            if (COMBINE && (!FUSED || p1)) {
                // publish this row's slot segment, then take a ticket for its
                // (token, N tile); the holder of the last ticket finishes it
                const int N1 = FUSED ? args1.N : args.N;
                const int n_slots = FUSED ? args1.n_slots : args.n_slots;
                const int n_tickets = FUSED ? args1.n_tickets : args.n_tickets;
                float* slot = FUSED ? args1.slot : args.slot;
                uint16_t* out = FUSED ? args1.out : args.out;
                int32_t* arrive = FUSED ? args1.arrive : args.arrive;
                int64_t t = -1;
                bool last = false;
                if (valid) {
                    const int f = args.src_row ? args.src_row[p] : p;
                    if (f >= 0 && f / args.k < args.T) {
                        t = f / args.k;
                        if (n_tickets == 1) {
                            last = true;   // the only arrival: every other slot was written before
                        } else {
                            __threadfence();
                            last = atomicAdd(arrive + t * n_tiles + wk.n_tile, 1) == n_tickets - 1;
                        }
                    }
                }
                // the warp sums its finished rows together: lane l takes columns
                // 8l .. 8l+7, so each slot row is read as one coalesced 1 KB line
                unsigned todo = __ballot_sync(0xffffffffu, last);
                if (todo) {
                    __threadfence();
                    const int n0 = wk.n_tile * BN;
                    // batches: 4 rows of <= 2 slots, 2 rows of <= 6, else one row of <= 9
                    if (n_slots <= 2) combine_rows<2, 4>(todo, t, slot, out, n0, N1, args.T, n_slots);
                    else if (n_slots <= 6) combine_rows<6, 2>(todo, t, slot, out, n0, N1, args.T, n_slots);
                    else combine_rows<9, 1>(todo, t, slot, out, n0, N1, args.T, n_slots);
                }
            }
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
    }

    // ---- teardown: every role is done (or has drained after an abort)
    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) {
        // after an abort, give the copies and commits already issued for this
        // CTA (some by the other CTA) time to land; then neither CTA leaves
        // while the other may still use its shared memory or TMEM
        if (threadIdx.x == 0 && *abort) sleep_ns(1000000);
        cluster_sync();
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<CG>(tmem_base, TMEM_COLS);
    }
}

using GemmKernel = void (*)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap,
                           const CUtensorMap, const GemmArgs, const GemmArgs);

// CTA-pair kernels: how many pairs can be resident at once (shared memory and
// the GPCs' SM pairs decide), looked up once per kernel and device.
constexpr int kMaxPairDevices = 64;
std::atomic<int> g_pair_clusters[3][kMaxPairDevices];

cudaError_t launch_pair(int slot, GemmKernel kern, const CUtensorMap& tmA, const CUtensorMap& tmB0,
                        const CUtensorMap& tmB1, const GemmArgs& a, int num_sms, cudaStream_t s)
{
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)smem_bytes<true>());
    if (err != cudaSuccess) return err;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = smem_bytes<true>();
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int dev = 0;
    err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxPairDevices) return cudaErrorInvalidDevice;
    int clusters = g_pair_clusters[slot][dev].load(std::memory_order_relaxed);
    if (clusters <= 0) {
        cfg.gridDim = dim3((unsigned)(num_sms & ~1));
        err = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
        if (err != cudaSuccess) return err;
        if (clusters <= 0) return cudaErrorInvalidConfiguration;
        g_pair_clusters[slot][dev].store(clusters, std::memory_order_relaxed);
    }
    clusters = clusters < num_sms / 2 ? clusters : num_sms / 2;
    if (clusters <= 0) return cudaErrorInvalidConfiguration;
    cfg.gridDim = dim3((unsigned)(2 * clusters));
    cfg.numAttrs = 2;   // the cached occupancy query above saw the cluster shape only
    err = cudaLaunchKernelEx(&cfg, kern, tmA, tmB0, tmB1, tmB0, tmB0, a, a);
    if (err == cudaSuccess) count_launch();
    return err;
}

}  // namespace

cudaError_t launch_grouped_gemm_fused(int mode, const CUtensorMap& tmA, const CUtensorMap& tmB0,
                                      const CUtensorMap& tmB1, const CUtensorMap& tmA1,
                                      const CUtensorMap& tmB2, const GemmArgs& a0, const GemmArgs& a1,
                                      int num_sms, cudaStream_t s)
{
    if (a0.M == 0) return cudaSuccess;
    if (a0.G < 1 || a0.G > MAX_GROUPS - 1) return cudaErrorInvalidValue;
    if (a0.K % BK != 0) return cudaErrorInvalidValue;
    const bool fused = (mode == kFusedScatter || mode == kFusedCombine);
    if (fused && (a1.K % BK != 0 || a1.ready == nullptr)) return cudaErrorInvalidValue;
    // the in-launch dispatch copy: dense GEMM0 over a routed tile table only
    if (a0.copy_ready && (mode != kGemm0Dense || !a0.copy_dst || !a0.src_row || !a0.tile_start || !a0.x))
        return cudaErrorInvalidValue;
    GemmKernel kern;
    if (mode == kGemm0Gather) kern = grouped_gemm_kernel<kGemm0Gather, false>;
    else if (mode == kGemm0Dense) kern = grouped_gemm_kernel<kGemm0Dense, false>;
    else if (mode == kGemm1Scatter) kern = grouped_gemm_kernel<kGemm1Scatter, false>;
    else if (mode == kGemm1Combine) kern = grouped_gemm_kernel<kGemm1Combine, false>;
    else if (mode == kGemm0CpGather) kern = grouped_gemm_kernel<kGemm0CpGather, false>;
    else if (mode == kFusedScatter) kern = grouped_gemm_kernel<kFusedScatter, false>;
    else if (mode == kFusedCombine) kern = grouped_gemm_kernel<kFusedCombine, false>;
    else return cudaErrorInvalidValue;
    constexpr size_t smem = smem_bytes<false>();
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    return launch_pdl(kern, dim3(num_sms), dim3(NUM_THREADS), smem, s, tmA, tmB0, tmB1, tmA1, tmB2, a0, a1);
}

cudaError_t launch_grouped_gemm(int mode, const CUtensorMap& tmA, const CUtensorMap& tmB0,
                                const CUtensorMap& tmB1, const GemmArgs& a, int num_sms,
                                cudaStream_t s, int cta_group)
{
    if (mode == kFusedScatter || mode == kFusedCombine) return cudaErrorInvalidValue;
    if (cta_group == 1) return launch_grouped_gemm_fused(mode, tmA, tmB0, tmB1, tmB0, tmB0, a, a, num_sms, s);
    if (cta_group != 2) return cudaErrorInvalidValue;
    if (a.M == 0) return cudaSuccess;
    if (a.G < 1 || a.G > MAX_GROUPS - 1 || a.K % BK != 0) return cudaErrorInvalidValue;
    if (a.copy_ready && (mode != kGemm0Dense || !a.copy_dst || !a.src_row || !a.tile_start || !a.x))
        return cudaErrorInvalidValue;
    if (mode == kGemm0Dense) return launch_pair(0, grouped_gemm_kernel<kGemm0Dense, true>, tmA, tmB0, tmB1, a, num_sms, s);
    if (mode == kGemm1Scatter)
        return launch_pair(1, grouped_gemm_kernel<kGemm1Scatter, true>, tmA, tmB0, tmB1, a, num_sms, s);
    if (mode == kGemm1Combine)
        return launch_pair(2, grouped_gemm_kernel<kGemm1Combine, true>, tmA, tmB0, tmB1, a, num_sms, s);
    return cudaErrorInvalidValue;   // the gathered-A GEMM0 forms run one CTA per MMA
}

}  // namespace moe
