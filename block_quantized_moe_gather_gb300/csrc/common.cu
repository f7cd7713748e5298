// Status strings, last-error messages, the device status word and the
// architecture check shared by every entry point.
#include <stdarg.h>
#include <stdio.h>

#include <atomic>
#include <mutex>

#include "bq_internal.cuh"

namespace {

thread_local char g_last_error[512] = "";

// One status word per device; kernels record the first error code seen.
__device__ int32_t g_device_status = 0;

constexpr int kMaxDevices = 64;
int g_arch_ok[kMaxDevices];          // 0 unknown, 1 ok, -1 wrong arch
int32_t* g_status_ptr[kMaxDevices];  // device address of g_device_status
std::mutex g_mutex;
std::atomic<uint64_t> g_launches{0};
thread_local cudaEvent_t g_stage_start[BQ_STAGE_COUNT];
thread_local cudaEvent_t g_stage_stop[BQ_STAGE_COUNT];

}  // namespace

namespace bq {

bq_status fail(bq_status s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    return s;
}

bq_status check_arch() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return fail(BQ_ERR_CUDA, "cudaGetDevice failed");
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_arch_ok[dev] == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return fail(BQ_ERR_CUDA, "cannot query compute capability of device %d", dev);
        g_arch_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
        if (g_arch_ok[dev] == 1) {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) {
                g_arch_ok[dev] = 0;
                return fail(BQ_ERR_CUDA, "cudaGetSymbolAddress(status word) failed on device %d", dev);
            }
            g_status_ptr[dev] = static_cast<int32_t*>(p);
        }
    }
    if (g_arch_ok[dev] != 1)
        return fail(BQ_ERR_ARCH, "device %d is not compute capability 10.3 (sm_103a build)", dev);
    return BQ_OK;
}

int32_t* device_status_ptr() {
    int dev = 0;
    cudaGetDevice(&dev);
    return (dev >= 0 && dev < kMaxDevices) ? g_status_ptr[dev] : nullptr;
}

void note_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

void stage_begin(int stage, cudaStream_t st) {
    if (g_stage_start[stage]) cudaEventRecord(g_stage_start[stage], st);
}

void stage_end(int stage, cudaStream_t st) {
    if (g_stage_stop[stage]) cudaEventRecord(g_stage_stop[stage], st);
}

bq_status check_launch(const char* what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(BQ_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
    return BQ_OK;
}

}  // namespace bq

extern "C" {

const char* bq_status_string(bq_status s) {
    switch (s) {
        case BQ_OK: return "BQ_OK";
        case BQ_ERR_NULL: return "BQ_ERR_NULL: a required pointer is NULL";
        case BQ_ERR_SHAPE: return "BQ_ERR_SHAPE: a size is out of range or not divisible";
        case BQ_ERR_ALIGN: return "BQ_ERR_ALIGN: a pointer is not aligned";
        case BQ_ERR_FORMAT: return "BQ_ERR_FORMAT: unknown or mismatched weight format";
        case BQ_ERR_WORKSPACE: return "BQ_ERR_WORKSPACE: workspace missing or too small";
        case BQ_ERR_CUDA: return "BQ_ERR_CUDA: a CUDA call failed";
        case BQ_ERR_DEVICE: return "BQ_ERR_DEVICE: the device status word was set";
        case BQ_ERR_ARCH: return "BQ_ERR_ARCH: device is not compute capability 10.3";
    }
    return "unknown bq_status";
}

const char* bq_last_error(void) { return g_last_error; }

bq_status bq_set_stage_events(int32_t stage, void* start_event, void* stop_event) {
    if (stage < 0 || stage >= BQ_STAGE_COUNT) return bq::fail(BQ_ERR_SHAPE, "bq_set_stage_events: stage %d", stage);
    g_stage_start[stage] = static_cast<cudaEvent_t>(start_event);
    g_stage_stop[stage] = static_cast<cudaEvent_t>(stop_event);
    return BQ_OK;
}

uint64_t bq_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

bq_status bq_device_status(bq_stream_t stream, int32_t* code) {
    if (!code) return bq::fail(BQ_ERR_NULL, "bq_device_status: code is NULL");
    bq_status s = bq::check_arch();
    if (s != BQ_OK) return s;
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return bq::fail(BQ_ERR_CUDA, "stream sync: %s", cudaGetErrorString(e));
    int32_t v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof(v)) != cudaSuccess ||
        cudaMemcpyToSymbol(g_device_status, &zero, sizeof(zero)) != cudaSuccess)
        return bq::fail(BQ_ERR_CUDA, "reading the device status word failed");
    *code = v;
    if (v != BQ_DEV_OK) return bq::fail(BQ_ERR_DEVICE, "device status code %d", v);
    return BQ_OK;
}

}  // extern "C"
