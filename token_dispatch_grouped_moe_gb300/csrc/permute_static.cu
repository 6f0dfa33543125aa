// permute_static.cu -- the dispatch step without a caller workspace.
//
// moe_permute needs scratch memory for its per-chunk expert histogram, and
// takes it from the caller's workspace. Some callers have no way to provide
// one: a host framework that owns all device memory and gives its plug-ins no
// allocator and no scratch hook, or a service whose device memory budget is
// fixed at start-up and which forbids allocating (or growing a pool) once it
// is serving, because an allocation can block and synchronise the device.
// moe_permute_static serves them: its scratch is a fixed array in this file
// (kStaticScratchBytes per GPU, held by every GPU that loads the library
// until the process exits), and it allocates nothing itself.
//
// Rules of this entry point:
//   - The first call on a device looks up the device address of the array
//     (cudaGetSymbolAddress, with that device current) and caches it; make
//     that first call before any stream capture on the device. The cached
//     address lives as long as the device's context: a cudaDeviceReset after
//     the first call is not supported (the module is loaded afresh and the
//     array may move).
//   - The same shape rules as moe_permute (check_dims), and with MOE_DEBUG=1
//     the call synchronises and reports a launch fault as MOE_ERR_CUDA.
//   - All calls on a device share the one array and it keeps the contents of
//     the last call. Nothing in it has to start at zero: every call writes
//     the part it reads. Calls that overlap on the GPU (other streams, other
//     host threads) race on the array: serialise them.
//   - Shapes whose histogram does not fit in the array are rejected with
//     MOE_ERR_UNSUPPORTED before anything is launched.
//   - There is no error word: an expert id outside [0, E) is skipped, so
//     offsets[E] ends below T*k, which is how the caller detects it.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "../../include/moe.h"
#include "kernels.cuh"

namespace {

constexpr size_t kStaticScratchBytes = 1u << 20;   // 1 MiB per GPU
constexpr int kStaticScratchInts = (int)(kStaticScratchBytes / sizeof(int32_t));
constexpr int kTileTableInts = 512;                 // tile table (E + 1 <= 257) first
constexpr int kMaxDevices = 64;

std::atomic<int32_t*> g_scratch_dev[kMaxDevices];
std::atomic<int> g_sms_dev[kMaxDevices];
std::mutex g_setup;

}  // namespace

// The scratch array. Only host code needs its device address (below); it is
// never dereferenced on the host.
static __device__ __align__(256) int32_t g_dispatch_scratch[kStaticScratchInts];

namespace {

// Device address of g_dispatch_scratch and the SM count, for the current
// device; looked up once per device.
moe_status static_scratch(int32_t** ptr, int* sms)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
    int32_t* p = g_scratch_dev[dev].load(std::memory_order_acquire);
    if (!p) {
        std::lock_guard<std::mutex> lock(g_setup);
        p = g_scratch_dev[dev].load(std::memory_order_acquire);
        if (!p) {
            void* addr = nullptr;
            if (cudaGetSymbolAddress(&addr, g_dispatch_scratch) != cudaSuccess || !addr)
                return MOE_ERR_CUDA;
            int n = 0;
            if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
                return MOE_ERR_CUDA;
            g_sms_dev[dev].store(n, std::memory_order_relaxed);
            p = static_cast<int32_t*>(addr);
            g_scratch_dev[dev].store(p, std::memory_order_release);
        }
    }
    *ptr = p;
    *sms = g_sms_dev[dev].load(std::memory_order_relaxed);
    return MOE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" moe_status moe_permute_static(const moe_dims* dims, const int32_t* topk_idx,
                                         int32_t* counts, int32_t* offsets, int32_t* src_row,
                                         int32_t* inv_pos, const moe_bf16* x, moe_bf16* x_perm,
                                         moe_stream_t stream)
{
    // the same shape rules as moe_permute, then the array's limit
    const moe_status dims_ok = moe::check_dims(dims);
    if (dims_ok != MOE_OK) return dims_ok;
    const moe_dims& d = *dims;
    const int64_t R = d.T * d.k;
    const int64_t hist_ints = (int64_t)moe::permute_num_chunks(R) * d.E;
    if (hist_ints > kStaticScratchInts - kTileTableInts) return MOE_ERR_UNSUPPORTED;
    if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
    if (R > 0 && (!topk_idx || !src_row || !inv_pos)) return MOE_ERR_INVALID_ARG;
    if (x_perm && (!x || !aligned16(x) || !aligned16(x_perm))) return MOE_ERR_INVALID_ARG;

    int32_t* scratch = nullptr;
    int sms = 0;
    const moe_status st = static_scratch(&scratch, &sms);
    if (st != MOE_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    moe::PermuteArgs a{topk_idx, counts, offsets, src_row, inv_pos,
                       scratch,                    // tile table
                       scratch + kTileTableInts,   // per-chunk histogram
                       nullptr,                    // no error word (see above)
                       R, d.E};
    if (moe::launch_permute(a, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (x_perm && moe::launch_gather_rows(x, src_row, offsets + d.E, x_perm, R, d.T, d.H, d.k, nullptr,
                                          sms, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (moe::debug_mode()) {
        // MOE_DEBUG=1: wait for the launches and report a fault they raised
        if (cudaStreamSynchronize(s) != cudaSuccess || cudaGetLastError() != cudaSuccess)
            return MOE_ERR_CUDA;
    }
    return MOE_OK;
}
