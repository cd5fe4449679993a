// fc_internal.cuh -- helpers shared by the CUDA translation units of the library (not part of the
// C ABI).  sm_103a only.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fusechain.h"

namespace fc {

// Record a CUDA error for fuse_last_cuda_error() and return FUSE_ECUDA.
int record_cuda_error(cudaError_t e);

// FUSE_OK if the last launch on this thread succeeded, else FUSE_ECUDA (error recorded).
inline int check_launch() {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? FUSE_OK : record_cuda_error(e);
}

// ----------------------------------------------------------------- programmatic dependent launch
// Every kernel of this library is launched with programmatic stream serialization allowed: it may
// be scheduled while the kernel before it on the stream is still finishing, which hides the launch
// latency between back-to-back kernels.  In exchange every kernel calls pdl_begin() before it
// touches global memory: griddepcontrol.wait returns once the preceding grid has completed and its
// writes are visible (at once if there is no such grid), so stream order is kept for every byte.
// launch_dependents lets the next kernel be scheduled as soon as every CTA of this one has started.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_begin() {
    pdl_trigger();
    pdl_wait();
}
// Start `bytes` of global memory at `ptr` on their way into L2 (both 16-byte aligned; nothing to
// wait for).  Issued before pdl_wait(), it overlaps a kernel's first DRAM reads with the end of
// the preceding kernel: L2 is the point of coherence of the device's memory, so the loads after
// pdl_wait() still return what the preceding kernel wrote, only sooner.
__device__ __forceinline__ void prefetch_l2_bulk(const void* ptr, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(ptr), "r"(bytes) : "memory");
}
// Kernels with a set-up phase that touches no global memory (mbarrier init, TMEM allocation,
// tensor-map prefetch) call pdl_trigger() at entry and pdl_wait() after the set-up, so the set-up
// overlaps the end of the preceding kernel.

// Launch `kernel` on `grid` x `block` threads with `smem` bytes of dynamic shared memory on `st`,
// programmatic serialization allowed, as clusters of `cluster_x` CTAs when cluster_x > 1.
// FUSE_OK, or FUSE_ECUDA with the error recorded.
template <typename... KArgs, typename... Args>
int launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, int cluster_x,
               Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[2];
    unsigned n = 0;
    at[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
    if (cluster_x > 1) {
        at[n].id = cudaLaunchAttributeClusterDimension;
        at[n].val.clusterDim.x = static_cast<unsigned>(cluster_x);
        at[n].val.clusterDim.y = 1;
        at[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = at;
    cfg.numAttrs = n;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
    if (e != cudaSuccess) return record_cuda_error(e);
    return check_launch();
}

// Streaming-multiprocessor count of the current device (cached per device).
int sm_count();
// Opt `kernel` into `bytes` of dynamic shared memory on the current device (and, with
// max_shared_carveout, into the largest shared-memory carveout) once per device: a kernel
// attribute belongs to a device's context, so every device a process launches on needs its own.
// Returns FUSE_OK or the recorded CUDA error.
int opt_in_smem(const void* kernel, int bytes, bool max_shared_carveout = false);

// Device address of the watchdog word on the current device (nullptr on failure).  Kernels with
// bounded waits take it as a parameter and set it when a wait runs out.
int* watchdog_flag();

// Occupancy-derived blocks per SM for a kernel at a block size (cached by caller as needed).
template <typename K>
int blocks_per_sm(K kernel, int block, size_t dyn_smem = 0) {
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kernel, block, dyn_smem) != cudaSuccess) {
        (void)cudaGetLastError();
        return 1;
    }
    return b > 0 ? b : 1;
}

// Fill a kernel record from the runtime's attributes of `kernel` launched with (block, dyn_smem),
// each CTA allocating `tmem_cols` tensor-memory columns.
int describe_kernel(const void* kernel, const char* name, int block, int dyn_smem,
                    fuse_kernel_record* out, int tmem_cols = 0);

inline bool is_aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// ----------------------------------------------------------------------- storage types
template <int DT> struct Storage;
template <> struct Storage<FUSE_F32> { using T = float; };
template <> struct Storage<FUSE_F16> { using T = __half; };
template <> struct Storage<FUSE_BF16> { using T = __nv_bfloat16; };

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__half v) { return __half2float(v); }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __half from_f32<__half>(float v) { return __float2half_rn(v); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

// A 16-byte vector of storage elements, unpacked to fp32 and packed back (nearest-even).
template <typename T> struct Vec16;
template <> struct Vec16<float> {
    static constexpr int N = 4;
    __device__ __forceinline__ static void unpack(const uint4& r, float* f) {
        f[0] = __uint_as_float(r.x); f[1] = __uint_as_float(r.y);
        f[2] = __uint_as_float(r.z); f[3] = __uint_as_float(r.w);
    }
    __device__ __forceinline__ static uint4 pack(const float* f) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                          __float_as_uint(f[3]));
    }
};
template <> struct Vec16<__half> {
    static constexpr int N = 8;
    __device__ __forceinline__ static void unpack(const uint4& r, float* f) {
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
            float2 t = __half22float2(h);
            f[2 * i] = t.x; f[2 * i + 1] = t.y;
        }
    }
    __device__ __forceinline__ static uint4 pack(const float* f) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __half2 h = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
            w[i] = *reinterpret_cast<uint32_t*>(&h);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
};
template <> struct Vec16<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ __forceinline__ static void unpack(const uint4& r, float* f) {
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            // bf16 -> fp32 is exact: the 16 bits become the high half of the fp32 pattern
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
    __device__ __forceinline__ static uint4 pack(const float* f) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
            w[i] = *reinterpret_cast<uint32_t*>(&h);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
};

// Streaming (evict-first) 16-byte global accesses: each byte of a chain is touched once.
__device__ __forceinline__ uint4 ld_stream(const uint4* p) { return __ldcs(p); }
__device__ __forceinline__ void st_stream(uint4* p, const uint4& v) { __stcs(p, v); }

// 32-byte vectors (8 fp32 or 16 fp16/bf16 values) with streaming 256-bit ld/st.global.cs (sm_100+)
template <typename T> struct Vec32 {
    static constexpr int N = 32 / sizeof(T);
    __device__ __forceinline__ static void load(const T* p, float* f) {
        uint32_t w[8];
        asm volatile("ld.global.cs.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                     : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]),
                       "=r"(w[6]), "=r"(w[7])
                     : "l"(p));
        Vec16<T>::unpack(make_uint4(w[0], w[1], w[2], w[3]), f);
        Vec16<T>::unpack(make_uint4(w[4], w[5], w[6], w[7]), f + N / 2);
    }
    __device__ __forceinline__ static void store(T* p, const float* f) {
        const uint4 lo = Vec16<T>::pack(f), hi = Vec16<T>::pack(f + N / 2);
        asm volatile("st.global.cs.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(lo.x),
                     "r"(lo.y), "r"(lo.z), "r"(lo.w), "r"(hi.x), "r"(hi.y), "r"(hi.z), "r"(hi.w)
                     : "memory");
    }
};

}  // namespace fc
