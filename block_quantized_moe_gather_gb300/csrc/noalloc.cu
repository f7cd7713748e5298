// Allocation-free variant of the expert permutation (bq_moe_permute_noalloc).
//
// Some callers cannot hand the library a workspace: for example a host
// integration whose device memory is owned and fully reserved by another
// framework's allocator, or a latency-critical loop that must not call
// cudaMalloc (which can fail there, or synchronise the device).  This entry
// point runs the same histogram / scan / placement kernels as
// bq_moe_permute, but their scratch (the per-chunk expert histograms) is a
// fixed array in device memory that is part of the library image.
//
// Behaviour a caller must know:
//  - The array holds kNoAllocScratchInts int32 values (256 KiB) on every GPU
//    that loads the library, until the process exits.  Requests whose
//    histograms need more (ceil(T*k / 256) * E ints) are rejected with
//    BQ_ERR_SHAPE before anything is launched.
//  - The first call on a device looks up the array's device address on that
//    device (cudaGetSymbolAddress, with that device current).  Make this
//    first call before any stream capture.
//  - Every call on a device shares the one array and leaves its contents
//    behind.  The kernels write every scratch entry they later read, so
//    nothing has to start at zero.  Two calls whose kernels overlap on the
//    GPU (different streams, no ordering between them) race on the array
//    and give wrong results; order them on one stream or with events.
//  - No cudaMalloc, cudaFree or other allocating routine is called.
#include <mutex>

#include "moe_internal.cuh"

namespace {

constexpr int kNoAllocScratchInts = 65536;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) int32_t g_permute_scratch[kNoAllocScratchInts];

int32_t* g_scratch_addr[kMaxDevices];   // device address of g_permute_scratch, per device
std::mutex g_scratch_mutex;

// Device address of the scratch array on the current device (looked up once).
bq_status scratch_on_current_device(int32_t** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return bq::fail(BQ_ERR_CUDA, "bq_moe_permute_noalloc: cudaGetDevice failed");
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_permute_scratch);
        if (e != cudaSuccess || !p)
            return bq::fail(BQ_ERR_CUDA, "bq_moe_permute_noalloc: cudaGetSymbolAddress on device %d: %s", dev,
                            cudaGetErrorString(e));
        g_scratch_addr[dev] = static_cast<int32_t*>(p);
    }
    *out = g_scratch_addr[dev];
    return BQ_OK;
}

}  // namespace

extern "C" bq_status bq_moe_permute_noalloc(const int32_t* ids, int32_t T, int32_t k, int32_t E, int32_t* counts,
                                            int32_t* offsets, int32_t* perm_token, int32_t* perm_slot,
                                            int32_t* inv, bq_stream_t stream) {
    bq_status s = bq::validate_route("bq_moe_permute_noalloc", T, E, k);
    if (s != BQ_OK) return s;
    if (!counts || !offsets || (T > 0 && (!ids || !perm_token || !perm_slot || !inv)))
        return bq::fail(BQ_ERR_NULL, "bq_moe_permute_noalloc: NULL pointer");
    // validate_route bounds T * k by INT32_MAX, so the int product below cannot wrap
    const size_t need = bq::permute_scratch_bytes(T * k, E) / sizeof(int32_t);
    if (need > (size_t)kNoAllocScratchInts)
        return bq::fail(BQ_ERR_SHAPE,
                        "bq_moe_permute_noalloc: T*k = %d with E = %d needs %zu scratch ints; the built-in "
                        "array holds %d (use bq_moe_permute with a workspace)",
                        T * k, E, need, kNoAllocScratchInts);
    if ((s = bq::check_arch()) != BQ_OK) return s;
    int32_t* scratch = nullptr;
    if ((s = scratch_on_current_device(&scratch)) != BQ_OK) return s;
    bq::launch_permute(ids, nullptr, T, k, E, counts, offsets, perm_token, perm_slot, nullptr, inv, scratch,
                       (cudaStream_t)stream);
    return bq::check_launch("bq_moe_permute_noalloc");
}
