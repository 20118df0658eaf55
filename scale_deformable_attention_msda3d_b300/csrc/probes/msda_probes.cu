// Microbenchmarks of the on-chip rates that bound the libmsda kernels (built into
// libmsda_probes.so, separate from the library; bench.py --probe runs them).  Each kernel
// moves 128-byte rows -- one fp32 D=32 head slice, the encoder workload's value row -- at
// random positions drawn by a counter-based hash, the access pattern of the corner gather:
//
//   gather_rows<VB>     random rows read from a buffer (L1-, L2- or HBM-resident by its
//                       size), VB = 16 or 32 bytes per lane, 128 / VB lanes per row
//   reduce_rows         random rows reduced into a buffer with red.global.add.v4.f32
//                       (8 lanes per row; one L2 request per row)
//   smem_atomic_rows    random rows of a 247-row shared-memory tile (the coarsest encoder
//                       level, 13 x 19) updated with per-channel shared-memory atomics
//   smem_owner_rows     the same tile updated without atomics: each lane group owns the
//                       rows congruent to its index and updates only those (plain
//                       shared-memory load, add, store)
//   tma_gather_rows     random rows copied into shared memory by cp.async.bulk (one
//                       128-byte bulk copy per row, completion on an mbarrier)
//   tma_gather4_rows    random rows copied into shared memory by the tensor copy's
//                       four-row gather mode (cp.async.bulk.tensor ... tile::gather4: four
//                       rows of a 2D tensor map per copy), four stages per warp in flight,
//                       each row then read from shared memory by the warp
//
// Every wait is bounded: a wait that runs out of iterations sets *err and the kernel
// returns after waiting (again bounded) for its own copies.  The host side only launches
// kernels; timing is done by the caller with CUDA events.
#include <cstdint>
#include <cuda.h>  // CUtensorMap and its enums (the encoder is fetched at run time)
#include <cuda_runtime.h>

namespace {

__device__ __forceinline__ unsigned hash32(unsigned x) {
    x ^= x >> 16;
    x *= 0x7feb352du;
    x ^= x >> 15;
    x *= 0x846ca68bu;
    x ^= x >> 16;
    return x;
}

// random row in [0, n): the high half of hash * n
__device__ __forceinline__ unsigned pick(unsigned key, unsigned n) {
    return __umulhi(hash32(key), n);
}

template <int VB>
__global__ void __launch_bounds__(256) gather_rows(const char *__restrict__ buf, unsigned n_rows,
                                                   int iters, unsigned seed, float *sink) {
    constexpr int G = 128 / VB;
    const unsigned tid = blockIdx.x * blockDim.x + threadIdx.x;
    const unsigned grp = tid / G, sub = tid % G;
    float acc = 0.f;
#pragma unroll 4
    for (int i = 0; i < iters; ++i) {
        const unsigned r = pick(grp * 7919u + i * 104729u + seed, n_rows);
        const char *p = buf + static_cast<size_t>(r) * 128 + sub * VB;
        if constexpr (VB == 16) {
            const float4 v = __ldg(reinterpret_cast<const float4 *>(p));
            acc += (v.x + v.y) + (v.z + v.w);
        } else {
            uint4 a, b;
            asm volatile("ld.global.nc.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                         : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y),
                           "=r"(b.z), "=r"(b.w)
                         : "l"(p));
            acc += (__uint_as_float(a.x) + __uint_as_float(a.y)) +
                   (__uint_as_float(a.z) + __uint_as_float(a.w)) +
                   (__uint_as_float(b.x) + __uint_as_float(b.y)) +
                   (__uint_as_float(b.z) + __uint_as_float(b.w));
        }
    }
    sink[tid] = acc;
}

__global__ void __launch_bounds__(256) reduce_rows(float *buf, unsigned n_rows, int iters,
                                                   unsigned seed) {
    const unsigned tid = blockIdx.x * blockDim.x + threadIdx.x;
    const unsigned grp = tid / 8, sub = tid % 8;
    const float w = 1e-3f * (sub + 1);
#pragma unroll 4
    for (int i = 0; i < iters; ++i) {
        const unsigned r = pick(grp * 7919u + i * 104729u + seed, n_rows);
        atomicAdd(reinterpret_cast<float4 *>(buf + static_cast<size_t>(r) * 32 + sub * 4),
                  make_float4(w, w, w, w));
    }
}

constexpr int kTileRows = 247;   // 13 x 19
constexpr int kRowFloats = 32;

__global__ void __launch_bounds__(256) smem_atomic_rows(int iters, unsigned seed, float *sink) {
    __shared__ float tile[kTileRows * kRowFloats];
    for (int i = threadIdx.x; i < kTileRows * kRowFloats; i += blockDim.x) tile[i] = 0.f;
    __syncthreads();
    const unsigned tid = blockIdx.x * blockDim.x + threadIdx.x;
    const unsigned grp = tid / 8, sub = threadIdx.x % 8;
    const float w = 1e-3f * (sub + 1);
#pragma unroll 4
    for (int i = 0; i < iters; ++i) {
        const unsigned r = pick(grp * 7919u + i * 104729u + seed, kTileRows);
        float *d = tile + r * kRowFloats + sub * 4;
        atomicAdd(d, w);
        atomicAdd(d + 1, w);
        atomicAdd(d + 2, w);
        atomicAdd(d + 3, w);
    }
    __syncthreads();
    sink[tid] = tile[threadIdx.x % (kTileRows * kRowFloats)];
}

__global__ void __launch_bounds__(256) smem_owner_rows(int iters, unsigned seed, float *sink) {
    __shared__ float4 tile[kTileRows * kRowFloats / 4];
    for (int i = threadIdx.x; i < kTileRows * kRowFloats / 4; i += blockDim.x)
        tile[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    __syncthreads();
    const unsigned tid = blockIdx.x * blockDim.x + threadIdx.x;
    const unsigned g = threadIdx.x / 8, sub = threadIdx.x % 8;
    const unsigned ngroups = blockDim.x / 8;
    const unsigned owned = (kTileRows - g + ngroups - 1) / ngroups;  // rows g, g + ngroups, ...
    const float w = 1e-3f * (sub + 1);
    for (int i = 0; i < iters; ++i) {
        const unsigned r = g + ngroups * pick(tid * 7919u + i * 104729u + seed, owned);
        float4 *d = tile + r * (kRowFloats / 4) + sub;
        float4 v = *d;
        v.x += w; v.y += w; v.z += w; v.w += w;
        *d = v;
    }
    __syncthreads();
    const float4 v = tile[threadIdx.x % (kTileRows * kRowFloats / 4)];
    sink[tid] = v.x + v.w;
}

// One warp per batch of 32 rows: lane k issues the bulk copy of row k into shared memory;
// lane 0 waits on the mbarrier for all 32 x 128 bytes.
constexpr unsigned kWaitLimit = 1u << 22;

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    for (unsigned it = 0; it < kWaitLimit; ++it) {
        uint32_t done;
        asm volatile("{\n\t.reg .pred p;\n\t"
                     "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                     "selp.u32 %0, 1, 0, p;\n\t}"
                     : "=r"(done) : "r"(bar), "r"(parity) : "memory");
        if (done) return true;
    }
    return false;
}

__global__ void __launch_bounds__(128) tma_gather_rows(const char *__restrict__ buf,
                                                       unsigned n_rows, int iters, unsigned seed,
                                                       float *sink, int *err) {
    __shared__ __align__(128) char rows[4][32 * 128];
    __shared__ __align__(8) unsigned long long bars[4];
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t bar = static_cast<uint32_t>(__cvta_generic_to_shared(&bars[warp]));
    const uint32_t dst0 = static_cast<uint32_t>(__cvta_generic_to_shared(&rows[warp][0]));
    if (lane == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(bar) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    const unsigned gw = (blockIdx.x * blockDim.x + threadIdx.x) / 32;
    float acc = 0.f;
    bool ok = true;
    for (int i = 0; i < iters && ok; ++i) {
        if (lane == 0)
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                         :: "r"(bar), "r"(32u * 128u) : "memory");
        __syncwarp();
        const unsigned r = pick(gw * 7919u + i * 104729u + lane * 31u + seed, n_rows);
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
                     "[%0], [%1], 128, [%2];"
                     :: "r"(dst0 + lane * 128), "l"(buf + static_cast<size_t>(r) * 128), "r"(bar)
                     : "memory");
        ok = mbar_wait(bar, i & 1);
        acc += reinterpret_cast<const float *>(&rows[warp][0])[lane];
        __syncwarp();
        // the next batch's bulk copies (async proxy) overwrite what was just read
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (!ok) {
        atomicExch(err, 1);
        // the copies of this batch may still be in flight: wait for them (bounded) before
        // the block's shared memory goes away
        (void)mbar_wait(bar, (iters - 1) & 1);
    }
    sink[blockIdx.x * blockDim.x + threadIdx.x] = acc;
}

// Four-row gathers: each warp keeps kG4Stages batches in flight; a batch is kG4Ops
// tile::gather4 copies (issued by lanes 0 .. kG4Ops-1, 4 rows of 128 bytes each) completing
// on the stage's mbarrier.  The warp then reads the batch's rows from shared memory (one
// 16-byte slice per lane per row group, as the forward's lane groups would) and re-issues
// the stage.
constexpr int kG4Warps = 4, kG4Stages = 4, kG4Ops = 4;
constexpr unsigned kG4BatchBytes = kG4Ops * 4 * 128;

__global__ void __launch_bounds__(kG4Warps * 32)
tma_gather4_rows(const __grid_constant__ CUtensorMap map, unsigned n_rows, int iters,
                 unsigned seed, float *sink, int *err) {
    __shared__ __align__(128) char rows[kG4Warps][kG4Stages][kG4BatchBytes];
    __shared__ __align__(8) unsigned long long bars[kG4Warps][kG4Stages];
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t bar0 = static_cast<uint32_t>(__cvta_generic_to_shared(&bars[warp][0]));
    if (lane == 0) {
        for (int s = 0; s < kG4Stages; ++s)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(bar0 + 8u * s) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    const unsigned gw = (blockIdx.x * blockDim.x + threadIdx.x) / 32;
    // batch i goes to stage i % kG4Stages
    auto issue = [&](int i) {
        const int s = i % kG4Stages;
        const uint32_t bar = bar0 + 8u * s;
        if (lane == 0)
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                         :: "r"(bar), "r"(kG4BatchBytes) : "memory");
        __syncwarp();
        if (lane < kG4Ops) {
            const unsigned key = (gw * 7919u + i * 104729u + lane * 31u + seed) * 4u;
            const int r0 = static_cast<int>(pick(key, n_rows));
            const int r1 = static_cast<int>(pick(key + 1u, n_rows));
            const int r2 = static_cast<int>(pick(key + 2u, n_rows));
            const int r3 = static_cast<int>(pick(key + 3u, n_rows));
            const uint32_t dst =
                static_cast<uint32_t>(__cvta_generic_to_shared(&rows[warp][s][lane * 4 * 128]));
            asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4"
                         ".mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5, %6}], [%7];"
                         :: "r"(dst), "l"(reinterpret_cast<uint64_t>(&map)), "r"(0), "r"(r0),
                            "r"(r1), "r"(r2), "r"(r3), "r"(bar)
                         : "memory");
        }
    };
    int issued = 0;
    for (; issued < kG4Stages && issued < iters; ++issued) issue(issued);
    float acc = 0.f;
    bool ok = true;
    int i = 0;
    for (; i < iters; ++i) {
        const int s = i % kG4Stages;
        ok = mbar_wait(bar0 + 8u * s, (i / kG4Stages) & 1);
        if (!ok) break;
        const float4 *st = reinterpret_cast<const float4 *>(&rows[warp][s][0]);
#pragma unroll
        for (int k = 0; k < static_cast<int>(kG4BatchBytes / 512); ++k) {
            const float4 v = st[k * 32 + lane];
            acc += (v.x + v.y) + (v.z + v.w);
        }
        __syncwarp();
        // the stage's next copies (async proxy) overwrite what was just read
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        if (issued < iters) issue(issued++);
    }
    if (!ok) {
        atomicExch(err, 1);
        // batches i .. issued-1 may still be in flight: wait for them (bounded) before the
        // block's shared memory goes away
        for (int j = i; j < issued; ++j)
            (void)mbar_wait(bar0 + 8u * (j % kG4Stages), (j / kG4Stages) & 1);
    }
    sink[blockIdx.x * blockDim.x + threadIdx.x] = acc;
}

// The tensor map of a buffer of n_rows rows of 32 fp32 (128 bytes), one row per box, for
// the four-row gather.  The encoder comes from the driver at run time (no libcuda link).
cudaError_t row_tensor_map(void *buf, unsigned n_rows, CUtensorMap *map) {
    using Encode = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
    static Encode encode = nullptr;
    if (encode == nullptr) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        const cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn,
                                                               12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr)
            return e != cudaSuccess ? e : cudaErrorNotSupported;
        encode = reinterpret_cast<Encode>(fn);
    }
    const cuuint64_t dims[2] = {32, n_rows};
    const cuuint64_t strides[1] = {128};
    const cuuint32_t box[2] = {32, 1};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, buf, dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

extern "C" {

// kind: 0 gather16, 1 gather32, 2 reduce, 3 smem atomic, 4 smem owner, 5 tma gather,
// 6 tma four-row gather.  Returns the CUDA launch status.  buf / n_rows: the row buffer
// (unused by kinds 3, 4); sink: one float per thread of the grid (blocks * threads); err:
// one int (kinds 5, 6).
int msda_probe_launch(int kind, void *buf, unsigned n_rows, int blocks, int iters,
                      unsigned seed, float *sink, int *err, void *stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    switch (kind) {
        case 0: gather_rows<16><<<blocks, 256, 0, s>>>(static_cast<const char *>(buf), n_rows, iters, seed, sink); break;
        case 1: gather_rows<32><<<blocks, 256, 0, s>>>(static_cast<const char *>(buf), n_rows, iters, seed, sink); break;
        case 2: reduce_rows<<<blocks, 256, 0, s>>>(static_cast<float *>(buf), n_rows, iters, seed); break;
        case 3: smem_atomic_rows<<<blocks, 256, 0, s>>>(iters, seed, sink); break;
        case 4: smem_owner_rows<<<blocks, 256, 0, s>>>(iters, seed, sink); break;
        case 5: tma_gather_rows<<<blocks, 128, 0, s>>>(static_cast<const char *>(buf), n_rows, iters, seed, sink, err); break;
        case 6: {
            // rows must start 16-byte aligned for the tensor map (the buffer is 256-byte
            // aligned, rows are 128 bytes)
            if ((reinterpret_cast<uintptr_t>(buf) & 127u) != 0 || n_rows == 0)
                return static_cast<int>(cudaErrorInvalidValue);
            CUtensorMap map;
            const cudaError_t e = row_tensor_map(buf, n_rows, &map);
            if (e != cudaSuccess) return static_cast<int>(e);
            tma_gather4_rows<<<blocks, kG4Warps * 32, 0, s>>>(map, n_rows, iters, seed, sink, err);
            break;
        }
        default: return static_cast<int>(cudaErrorInvalidValue);
    }
    return static_cast<int>(cudaGetLastError());
}

// Threads per block of a probe kind (the caller sizes sink as blocks * this).
int msda_probe_block(int kind) { return kind == 5 ? 128 : kind == 6 ? kG4Warps * 32 : 256; }

}  // extern "C"
