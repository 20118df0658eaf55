// Locality-aware query order: a permutation of each batch's queries that puts queries
// whose samples land close together next to each other, so that the lane groups, warps
// and CTAs that run at the same time read overlapping value rows (L1 / L2 reuse).  The
// core's result does not depend on the order; only which items run side by side does.
//
// Key of a query: the Morton (Z-order) code of the mean of its finite sampling locations
// (all heads, levels and points), on a 64 x 64 (2D) or 16 x 16 x 16 (3D) grid over the
// normalised [0, 1] square / cube (4096 buckets per batch).  The permutation is a counting sort by key:
//   1. keys (one warp per query) + per-batch histogram (global integer atomics),
//   2. per-batch exclusive scan of the histogram (one CTA per batch),
//   3. scatter: each query takes the next slot of its bucket (atomic cursor).
// Queries with equal keys end up in arbitrary (run-dependent) relative order.
#include "common.cuh"

namespace msda {

namespace {

// Spreads the low `bits` bits of v so that bit k moves to bit k * stride.
__device__ __forceinline__ unsigned spread(unsigned v, int bits, int stride) {
    unsigned r = 0;
    for (int k = 0; k < bits; ++k) r |= ((v >> k) & 1u) << (k * stride);
    return r;
}

__device__ __forceinline__ unsigned cell(float mean, int bits) {
    const float c = fminf(fmaxf(mean, 0.f), 1.f) * static_cast<float>(1 << bits);
    const unsigned i = static_cast<unsigned>(c);
    return i >= (1u << bits) ? (1u << bits) - 1u : i;
}

// One warp per query: the lanes read the query's samples (contiguous) in turn, sum the
// finite ones and reduce across the warp.
template <int NDIM>
__global__ void __launch_bounds__(256)
order_keys(const float *__restrict__ loc, long long n_queries, int per_query, int *hist,
           int *keys, long long Nq) {
    const long long pos = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (pos >= n_queries) return;  // whole warps leave together
    const float *src = loc + pos * per_query * NDIM;
    float sum[NDIM];
#pragma unroll
    for (int k = 0; k < NDIM; ++k) sum[k] = 0.f;
    float n = 0.f;
    for (int s = lane; s < per_query; s += 32) {
        float v[NDIM];
        bool fin = true;
#pragma unroll
        for (int k = 0; k < NDIM; ++k) {
            v[k] = __ldcs(src + s * NDIM + k);
            fin = fin && isfinite(v[k]);
        }
        if (fin) {
#pragma unroll
            for (int k = 0; k < NDIM; ++k) sum[k] += v[k];
            n += 1.f;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
        for (int k = 0; k < NDIM; ++k) sum[k] += __shfl_xor_sync(kFull, sum[k], o);
        n += __shfl_xor_sync(kFull, n, o);
    }
    if (lane != 0) return;
    unsigned key;
    if (n == 0.f) {
        key = kOrderBuckets - 1;  // no finite sample: last bucket
    } else {
        constexpr int BITS = NDIM == 2 ? kOrderBits2d : kOrderBits3d;
        key = 0;
#pragma unroll
        for (int k = 0; k < NDIM; ++k) key |= spread(cell(sum[k] / n, BITS), BITS, NDIM) << k;
    }
    const long long b = pos / Nq;
    keys[pos] = static_cast<int>(key);
    atomicAdd(hist + b * kOrderBuckets + key, 1);
}

// Exclusive prefix sum of one batch's histogram, in place (1024 threads, one CTA per batch,
// kOrderBuckets / 1024 consecutive buckets per thread).
__global__ void __launch_bounds__(1024) order_scan(int *hist) {
    constexpr int PER = kOrderBuckets / 1024;
    __shared__ int warp_tot[32];
    int *h = hist + static_cast<long long>(blockIdx.x) * kOrderBuckets + threadIdx.x * PER;
    int local = 0;
    for (int i = 0; i < PER; ++i) local += h[i];
    // inclusive scan of `local` over the block
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = warp_tot[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(kFull, w, o);
            if (lane >= o) w += y;
        }
        warp_tot[lane] = w;  // inclusive warp prefix
    }
    __syncthreads();
    int run = x - local + (warp > 0 ? warp_tot[warp - 1] : 0);  // exclusive prefix of this thread
    for (int i = 0; i < PER; ++i) {
        const int c = h[i];
        h[i] = run;
        run += c;
    }
}

__global__ void __launch_bounds__(256)
order_scatter(const int *keys, long long n_queries, long long Nq, int *hist, int *order) {
    const long long pos = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (pos >= n_queries) return;
    const long long b = pos / Nq;
    const int slot = atomicAdd(hist + b * kOrderBuckets + keys[pos], 1);
    order[b * Nq + slot] = static_cast<int>(pos - b * Nq);
}

}  // namespace

cudaError_t launch_query_order(int ndim, const Params &p, int *order, int *hist, int *keys,
                               cudaStream_t s) {
    const long long n = p.B * p.Nq;
    if (n == 0) return cudaSuccess;
    // every grid size is checked before the first enqueue: a rejected call leaves nothing
    // on the stream
    const long long warps_blocks = (n * 32 + 255) / 256;
    if (warps_blocks > 0x7fffffffLL || p.B > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const unsigned blocks = static_cast<unsigned>((n + 255) / 256);
    cudaError_t e = cudaMemsetAsync(hist, 0, sizeof(int) * p.B * kOrderBuckets, s);
    if (e != cudaSuccess) return e;
    const int per_query = p.M * p.L * p.P;
    if (ndim == 2)
        order_keys<2><<<static_cast<unsigned>(warps_blocks), 256, 0, s>>>(p.loc, n, per_query,
                                                                         hist, keys, p.Nq);
    else
        order_keys<3><<<static_cast<unsigned>(warps_blocks), 256, 0, s>>>(p.loc, n, per_query,
                                                                         hist, keys, p.Nq);
    order_scan<<<static_cast<unsigned>(p.B), 1024, 0, s>>>(hist);
    order_scatter<<<blocks, 256, 0, s>>>(keys, n, p.Nq, hist, order);
    return cudaGetLastError();
}

}  // namespace msda
