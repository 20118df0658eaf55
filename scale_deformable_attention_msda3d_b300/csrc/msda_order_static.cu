// Query order without any allocation: the histogram and key scratch of msda_query_order
// live in a fixed array in this library's device image instead of a caller workspace.
//
// Who needs this: code that must not call cudaMalloc (or any allocator) on its path, for
// example a real-time loop that forbids allocation after start-up, a plugin whose host
// framework owns every device allocation, or a caller that cannot find a place to keep a
// workspace between calls.  They pass the input and output buffers and nothing else.
//
// The array below is in device memory of every GPU that loads the library and stays there
// until the process exits.  Calls share it: two calls whose work overlaps on the GPU (on
// different streams, or from different host threads) race on it and can give wrong
// orders.  Each call clears the histogram part itself before use.
#include <cstdint>
#include <mutex>

#include "common.cuh"

namespace msda {

namespace {

// Largest problem the fixed scratch holds: B <= kStaticOrderBatches and
// B * Nq <= kStaticOrderQueries (4 MB of keys plus 1 MB of histograms).
constexpr long long kStaticOrderBatches = 64;
constexpr long long kStaticOrderQueries = 1LL << 20;
constexpr long long kStaticOrderInts = kStaticOrderBatches * kOrderBuckets + kStaticOrderQueries;

static __device__ __align__(256) int g_order_scratch[kStaticOrderInts];

constexpr int kMaxDevices = 64;
std::mutex g_lock;
int *g_scratch_ptr[kMaxDevices] = {};

}  // namespace

cudaError_t static_order_scratch(int **ptr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> guard(g_lock);
    if (!g_scratch_ptr[dev]) {
        // host code may not use the array's name as an address: ask the runtime for the
        // device address of this device's copy (once per device, with it current)
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_order_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = static_cast<int *>(p);
    }
    *ptr = g_scratch_ptr[dev];
    return cudaSuccess;
}

bool static_order_fits(long long B, long long Nq) {
    return B <= kStaticOrderBatches && B * Nq <= kStaticOrderQueries;
}

cudaError_t launch_query_order_static(int ndim, const Params &p, int *order, cudaStream_t s) {
    int *scratch = nullptr;
    cudaError_t e = static_order_scratch(&scratch);
    if (e != cudaSuccess) return e;
    int *hist = scratch;
    int *keys = scratch + kStaticOrderBatches * kOrderBuckets;
    return launch_query_order(ndim, p, order, hist, keys, s);
}

}  // namespace msda
