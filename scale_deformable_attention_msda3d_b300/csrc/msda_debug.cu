// Debug build support (compiled with -DMSDA_DEBUG_BOUNDS into libmsda_debug.so): the record
// of the first out-of-range corner row any kernel met, and a self-test that writes a
// made-up record through the same device function the kernels use, so that the reporting
// path can be exercised without any out-of-range access.  In the normal build the entry
// points below only report that the checks are not compiled in.
#include <mutex>

#include "common.cuh"

namespace msda {

#ifdef MSDA_DEBUG_BOUNDS

namespace {

// One record per device (every GPU that loads the library holds its own copy); zero at
// load, cleared by debug_record_take.
static __device__ DebugRecord g_debug_record;

constexpr int kMaxDevices = 64;
std::mutex g_lock;
DebugRecord *g_record_ptr[kMaxDevices] = {};

__global__ void debug_selftest_kernel(const __grid_constant__ Params p, long long row,
                                      long long item, int sample) {
    // the check fails for an out-of-range row and records it; nothing is accessed
    (void)row_ok(p, row, item, sample);
}

}  // namespace

cudaError_t debug_record(DebugRecord **ptr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> guard(g_lock);
    if (!g_record_ptr[dev]) {
        // host code may not use the variable's name as an address: ask the runtime for the
        // device address of this device's copy (once per device, with it current)
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_debug_record);
        if (e != cudaSuccess) return e;
        g_record_ptr[dev] = static_cast<DebugRecord *>(p);
    }
    *ptr = g_record_ptr[dev];
    return cudaSuccess;
}

cudaError_t debug_record_take(DebugRecord *out) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return e;
    e = cudaMemcpyFromSymbol(out, g_debug_record, sizeof(DebugRecord));
    if (e != cudaSuccess) return e;
    const DebugRecord zero = {};
    return cudaMemcpyToSymbol(g_debug_record, &zero, sizeof(DebugRecord));
}

cudaError_t launch_debug_selftest(const Params &p, long long row, long long item, int sample,
                                  cudaStream_t s) {
    debug_selftest_kernel<<<1, 1, 0, s>>>(p, row, item, sample);
    return cudaGetLastError();
}

#else

cudaError_t debug_record(DebugRecord **ptr) {
    *ptr = nullptr;
    return cudaErrorNotSupported;
}
cudaError_t debug_record_take(DebugRecord *) { return cudaErrorNotSupported; }
cudaError_t launch_debug_selftest(const Params &, long long, long long, int, cudaStream_t) {
    return cudaErrorNotSupported;
}

#endif

}  // namespace msda
