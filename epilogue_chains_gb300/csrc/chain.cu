// chain.cu -- the pointwise chain y = f_{K-1}(...f_0(x)), f_s(v) = [ReLU](a_s*v + b_s).
//
// [C05] §3 "API / experiment shape" names the three forms built here:
//   naive  -- one stage kernel per s, the intermediate passes through global memory;
//   fused  -- one kernel that loops s = 0..K-1 in registers and writes once;
//   fat    -- the fused kernel plus C05_FAT_TEMPS (48) live temporaries summed into a sink, a
//             probe of the register-pressure cliff ([C05] §6.2: blocks/SM 6 -> 1 on sm_120).
// [OFCG] §3.2 gives their byte ledgers: 2*K*N*b unfused, 2*N*b fused.
//
// GB300 design: the work is pure HBM streaming (8 B/element for fp32, 2 flops per stage), so the
// kernels are shaped for DRAM efficiency, not ALU: one 32-byte vector per thread (256-bit
// ld/st.global.cs, sm_100+), an exact grid of many short CTAs (measured on GB300 to match
// cudaMemcpy at this size, where persistent grid-stride loops and TMA bulk-copy pipelines were
// slower), and stage coefficients in a __grid_constant__ parameter read from the constant bank.
#include <mutex>

#include "fc_internal.cuh"

namespace fc {
namespace {

constexpr int kBlock = 256;

struct ChainParams {
    const void* x;
    void* y;
    int64_t n;      // elements
    int64_t head;   // scalar elements before the 32-byte-aligned body
    int64_t nvec;   // 32-byte vectors in the body (fused/unfused); the fat probe reads the same
                    // body in groups of 4 elements
    int K;
    int prefetch;   // 1: start this CTA's input on its way into L2 before the grid-dependency wait
    int64_t ahead;  // with prefetch: also start the input of CTA blockIdx.x + ahead (the CTA that
                    // takes this slot one wave later); 0 = none
    uint32_t relu_mask;
    float a[FUSE_MAX_STAGES];
    float b[FUSE_MAX_STAGES];
};

__device__ float g_fat_sink;  // written only on an impossible bit pattern: keeps the fat sum live

// One stage, rounded twice (fl32(fl32(a*v) + b)), then ReLU(t) = t > 0 ? t : +0.
__device__ __forceinline__ float stage_apply(float v, float a, float b, bool relu) {
    float t = __fadd_rn(__fmul_rn(a, v), b);
    return relu ? (t > 0.0f ? t : 0.0f) : t;
}

template <int E, bool kOneStage>
__device__ __forceinline__ void run_chain(float (&f)[E], const ChainParams& p) {
    const int K = kOneStage ? 1 : p.K;
    for (int s = 0; s < K; ++s) {
        const float a = p.a[s];
        const float b = p.b[s];
        const bool relu = (p.relu_mask >> s) & 1u;
#pragma unroll
        for (int e = 0; e < E; ++e) f[e] = stage_apply(f[e], a, b, relu);
    }
}

// Thread g handles: head element g (if g < head), vector g (if g < nvec), tail element g.
template <typename T, bool kOneStage>
__device__ __forceinline__ void chain_body(const ChainParams& p) {
    using V = Vec32<T>;
    constexpr int E = V::N;
    const T* x = static_cast<const T*>(p.x);
    T* y = static_cast<T*>(p.y);
    const int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (g < p.nvec) {
        float f[E];
        V::load(x + p.head + g * E, f);
        run_chain<E, kOneStage>(f, p);
        V::store(y + p.head + g * E, f);
    }
    if (g < p.head) {
        float f[1] = {to_f32(x[g])};
        run_chain<1, kOneStage>(f, p);
        y[g] = from_f32<T>(f[0]);
    }
    const int64_t t = p.head + p.nvec * E + g;
    if (t < p.n) {
        float f[1] = {to_f32(x[t])};
        run_chain<1, kOneStage>(f, p);
        y[t] = from_f32<T>(f[0]);
    }
}

// This CTA's share of the 32-byte-aligned body on its way into L2 while the preceding kernel may
// still run, then the grid-dependency wait (before any global-memory load or store).  The share of
// the CTA one wave later goes too: at the start of a launch the first wave then has two waves of
// input in flight across the grid-dependency release, and in steady state every CTA finds its
// input already on its way (measured at N = 2^24: 21.0 -> 20.1 us per call; one wave ahead only
// for the first wave gains half of that, two waves ahead or twice the distance lose it again).
// Not for an unfused stage after the first: its input is the intermediate the preceding stage is
// writing, already in L2 or about to be overwritten, and fetching it from DRAM early only adds
// traffic (measured: the K = 8 unfused chain at N = 2^24 went from 104 to 113 us with it).
template <typename T>
__device__ __forceinline__ void prefetch_then_wait(const ChainParams& p) {
    pdl_trigger();
    if (p.prefetch && threadIdx.x == 0) {
        for (int w = 0; w < (p.ahead > 0 ? 2 : 1); ++w) {
            const int64_t v0 = (static_cast<int64_t>(blockIdx.x) + w * p.ahead) * kBlock;
            const int64_t nv = p.nvec - v0 < kBlock ? p.nvec - v0 : kBlock;
            if (nv > 0)
                prefetch_l2_bulk(static_cast<const T*>(p.x) + p.head + v0 * Vec32<T>::N,
                                 static_cast<uint32_t>(nv) * 32u);
        }
    }
    pdl_wait();
}

template <typename T>
__global__ void __launch_bounds__(kBlock) chain_fused_kernel(const __grid_constant__ ChainParams p) {
    prefetch_then_wait<T>(p);
    chain_body<T, false>(p);
}

template <typename T>
__global__ void __launch_bounds__(kBlock) chain_stage_kernel(const __grid_constant__ ChainParams p) {
    prefetch_then_wait<T>(p);
    chain_body<T, true>(p);
}

// CTAs of the element kernels resident on the whole device at once (one wave).
template <typename T>
int64_t resident_ctas() {
    static const int occ = blocks_per_sm(chain_fused_kernel<T>, kBlock);
    return static_cast<int64_t>(sm_count()) * occ;
}

// ---------------------------------------------------------------------------------- fat probe
// Each element carries FUSE_FAT_TEMPS temporaries t_j, updated every stage as t_j <- t_j*a_s + v
// and summed into a sink at the end.  The stage loop has a run-time trip count, so all
// temporaries of the 4 elements a thread holds (4 x 48 = 192 fp32) are live across it.
template <int E>
__device__ __forceinline__ float fat_group(float (&v)[E], const ChainParams& p) {
    float t[E][FUSE_FAT_TEMPS];
#pragma unroll
    for (int e = 0; e < E; ++e)
#pragma unroll
        for (int j = 0; j < FUSE_FAT_TEMPS; ++j) t[e][j] = v[e] * (1.0f + j * (1.0f / 64.0f));
    for (int s = 0; s < p.K; ++s) {
        const float a = p.a[s];
        const float b = p.b[s];
        const bool relu = (p.relu_mask >> s) & 1u;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            v[e] = stage_apply(v[e], a, b, relu);
#pragma unroll
            for (int j = 0; j < FUSE_FAT_TEMPS; ++j) t[e][j] = __fmaf_rn(t[e][j], a, v[e]);
        }
    }
    float acc = 0.0f;
#pragma unroll
    for (int e = 0; e < E; ++e)
#pragma unroll
        for (int j = 0; j < FUSE_FAT_TEMPS; ++j) acc += t[e][j];
    return acc;
}

template <typename T>
__global__ void __launch_bounds__(kBlock, 1) chain_fat_kernel(const __grid_constant__ ChainParams p) {
    pdl_begin();  // before any global-memory access (programmatic dependent launch)
    const T* x = static_cast<const T*>(p.x);
    T* y = static_cast<T*>(p.y);
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t nthr = static_cast<int64_t>(gridDim.x) * blockDim.x;
    float sink = 0.0f;

    // groups of 4 consecutive elements (the body is 32-byte aligned, so 4 elements are aligned
    // to 4*sizeof(T)); head and tail one element at a time
    const int64_t body = p.nvec * Vec32<T>::N;
    const int64_t groups = body / 4;
    const int64_t tail0 = p.head + groups * 4;
    for (int64_t i = tid; i < p.head; i += nthr) {
        float v[1] = {to_f32(x[i])};
        sink += fat_group<1>(v, p);
        y[i] = from_f32<T>(v[0]);
    }
    for (int64_t i = tail0 + tid; i < p.n; i += nthr) {
        float v[1] = {to_f32(x[i])};
        sink += fat_group<1>(v, p);
        y[i] = from_f32<T>(v[0]);
    }
    const T* xb = x + p.head;
    T* yb = y + p.head;
    for (int64_t g = tid; g < groups; g += nthr) {
        float v[4];
        if constexpr (sizeof(T) == 4) {
            uint4 r = ld_stream(reinterpret_cast<const uint4*>(xb) + g);
            Vec16<float>::unpack(r, v);
        } else {
            uint2 r = __ldcs(reinterpret_cast<const uint2*>(xb) + g);
            const T* h = reinterpret_cast<const T*>(&r);
#pragma unroll
            for (int e = 0; e < 4; ++e) v[e] = to_f32(h[e]);
        }
        sink += fat_group<4>(v, p);
        if constexpr (sizeof(T) == 4) {
            st_stream(reinterpret_cast<uint4*>(yb) + g, Vec16<float>::pack(v));
        } else {
            T h[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) h[e] = from_f32<T>(v[e]);
            __stcs(reinterpret_cast<uint2*>(yb) + g, *reinterpret_cast<uint2*>(h));
        }
    }
    if (__float_as_uint(sink) == 0x7fbadbadu) g_fat_sink = sink;
}

// ---------------------------------------------------------------------------------- host side
// Split [0, n) into a scalar head up to the first 32-byte boundary, 32-byte vectors, and a scalar
// tail, when x and y sit at the same offset modulo 32 bytes; otherwise all elements are scalar.
template <typename T>
void partition(ChainParams& p, const void* x, const void* y) {
    const uintptr_t xo = reinterpret_cast<uintptr_t>(x) % 32, yo = reinterpret_cast<uintptr_t>(y) % 32;
    if (xo == yo) {
        int64_t head = xo ? static_cast<int64_t>((32 - xo) / sizeof(T)) : 0;
        if (head > p.n) head = p.n;
        p.head = head;
        p.nvec = (p.n - head) / Vec32<T>::N;
    } else {
        p.head = p.n;
        p.nvec = 0;
    }
}

template <typename T>
unsigned exact_grid(const ChainParams& p) {
    int64_t units = p.nvec;
    const int64_t tail = p.n - p.head - p.nvec * Vec32<T>::N;
    if (p.head > units) units = p.head;
    if (tail > units) units = tail;
    const int64_t g = ceil_div(units, kBlock);
    return static_cast<unsigned>(g < 1 ? 1 : g);
}

template <typename T>
int launch_chain(const ChainParams& base, int mode, cudaStream_t stream) {
    ChainParams p = base;
    p.prefetch = 1;
    p.ahead = resident_ctas<T>();
    partition<T>(p, p.x, p.y);
    if (mode == FUSE_FUSED) {
        return launch_pdl(chain_fused_kernel<T>, dim3(exact_grid<T>(p)), dim3(kBlock), 0, stream, 1, p);
    }
    if (mode == FUSE_FAT) {
        static const int occ = blocks_per_sm(chain_fat_kernel<T>, kBlock);
        const int64_t want = ceil_div(ceil_div(p.n, 4), kBlock);
        const int64_t cap = static_cast<int64_t>(sm_count()) * occ;
        const unsigned grid = static_cast<unsigned>(want < 1 ? 1 : (want < cap ? want : cap));
        return launch_pdl(chain_fat_kernel<T>, dim3(grid), dim3(kBlock), 0, stream, 1, p);
    }
    // FUSE_UNFUSED: stage s is its own launch; stage 0 reads x, every later stage reads and
    // rewrites y in place, so each intermediate makes a full round trip through global memory.
    for (int s = 0; s < base.K; ++s) {
        ChainParams q = base;
        q.K = 1;
        q.a[0] = base.a[s];
        q.b[0] = base.b[s];
        q.relu_mask = (base.relu_mask >> s) & 1u;
        if (s > 0) q.x = base.y;
        q.prefetch = s == 0;
        q.ahead = s == 0 ? resident_ctas<T>() : 0;
        partition<T>(q, q.x, q.y);
        const int rc = launch_pdl(chain_stage_kernel<T>, dim3(exact_grid<T>(q)), dim3(kBlock), 0, stream, 1, q);
        if (rc != FUSE_OK) return rc;
    }
    return FUSE_OK;
}

}  // namespace

// report entries of this translation unit
int chain_report_count() { return 5; }
int chain_report(int i, fuse_kernel_record* out) {
    switch (i) {
        case 0: return describe_kernel((const void*)chain_fused_kernel<float>,
                                       "chain_fused_kernel<f32>", kBlock, 0, out);
        case 1: return describe_kernel((const void*)chain_stage_kernel<float>,
                                       "chain_stage_kernel<f32> (unfused stage)", kBlock, 0, out);
        case 2: return describe_kernel((const void*)chain_fat_kernel<float>,
                                       "chain_fat_kernel<f32> (48 live temps)", kBlock, 0, out);
        case 3: return describe_kernel((const void*)chain_fused_kernel<__nv_bfloat16>,
                                       "chain_fused_kernel<bf16>", kBlock, 0, out);
        case 4: return describe_kernel((const void*)chain_fat_kernel<__nv_bfloat16>,
                                       "chain_fat_kernel<bf16> (48 live temps)", kBlock, 0, out);
        default: return FUSE_EINVAL;
    }
}

}  // namespace fc

extern "C" int fuse_chain_run(const fuse_stage* stages, int K, const void* x, void* y, int64_t n,
                              int dtype, int mode, fuse_stream_t stream) {
    using namespace fc;
    if (!stages || K < 1 || K > FUSE_MAX_STAGES || n < 0) return FUSE_EINVAL;
    if (dtype != FUSE_F32 && dtype != FUSE_F16 && dtype != FUSE_BF16) return FUSE_EINVAL;
    if (mode != FUSE_FUSED && mode != FUSE_UNFUSED && mode != FUSE_FAT) return FUSE_EINVAL;
    for (int s = 0; s < K; ++s)
        if (stages[s].op != FUSE_OP_AFFINE && stages[s].op != FUSE_OP_AFFINE_RELU) return FUSE_EINVAL;
    if (n == 0) return FUSE_OK;
    if (!x || !y) return FUSE_EINVAL;
    const size_t eb = dtype == FUSE_F32 ? 4 : 2;
    if (!is_aligned(x, eb) || !is_aligned(y, eb)) return FUSE_EALIGN;
    const uintptr_t xa = reinterpret_cast<uintptr_t>(x), ya = reinterpret_cast<uintptr_t>(y);
    const uintptr_t bytes = static_cast<uintptr_t>(n) * eb;
    if (xa != ya && xa < ya + bytes && ya < xa + bytes) return FUSE_EINVAL;  // partial overlap

    ChainParams p{};
    p.x = x;
    p.y = y;
    p.n = n;
    p.K = K;
    for (int s = 0; s < K; ++s) {
        p.a[s] = stages[s].a;
        p.b[s] = stages[s].b;
        if (stages[s].op == FUSE_OP_AFFINE_RELU) p.relu_mask |= 1u << s;
    }
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    switch (dtype) {
        case FUSE_F32: return launch_chain<float>(p, mode, st);
        case FUSE_F16: return launch_chain<__half>(p, mode, st);
        default: return launch_chain<__nv_bfloat16>(p, mode, st);
    }
}

namespace fc {
namespace {
// Per-device helper streams and events of fuse_chain_run_host(), created at the first call on a
// device and kept for the life of the process.
struct HostPipe {
    std::mutex mu;
    bool ready = false;
    cudaStream_t s_in = nullptr, s_out = nullptr;
    cudaEvent_t entry = nullptr, in = nullptr, run = nullptr, out = nullptr;
};
HostPipe g_pipes[64];

int host_pipe_init(HostPipe& hp) {
    if (hp.ready) return FUSE_OK;
    cudaError_t e;
    if ((e = cudaStreamCreateWithFlags(&hp.s_in, cudaStreamNonBlocking)) != cudaSuccess ||
        (e = cudaStreamCreateWithFlags(&hp.s_out, cudaStreamNonBlocking)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&hp.entry, cudaEventDisableTiming)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&hp.in, cudaEventDisableTiming)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&hp.run, cudaEventDisableTiming)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&hp.out, cudaEventDisableTiming)) != cudaSuccess)
        return record_cuda_error(e);
    hp.ready = true;
    return FUSE_OK;
}
}  // namespace
}  // namespace fc

extern "C" int fuse_chain_run_host(const fuse_stage* stages, int K, const void* x_host, void* y_host,
                                   int64_t n, int dtype, int mode, void* x_dev, void* y_dev, int slices,
                                   fuse_stream_t stream) {
    using namespace fc;
    if (!stages || K < 1 || K > FUSE_MAX_STAGES || n < 0 || slices < 1 || slices > 64) return FUSE_EINVAL;
    if (dtype != FUSE_F32 && dtype != FUSE_F16 && dtype != FUSE_BF16) return FUSE_EINVAL;
    if (mode != FUSE_FUSED && mode != FUSE_UNFUSED && mode != FUSE_FAT) return FUSE_EINVAL;
    if (n == 0) return FUSE_OK;
    if (!x_host || !y_host || !x_dev || !y_dev) return FUSE_EINVAL;
    const int64_t eb = dtype == FUSE_F32 ? 4 : 2;
    const uintptr_t xa = reinterpret_cast<uintptr_t>(x_dev), ya = reinterpret_cast<uintptr_t>(y_dev);
    const uintptr_t bytes = static_cast<uintptr_t>(n * eb);
    if (xa != ya && xa < ya + bytes && ya < xa + bytes) return FUSE_EINVAL;  // partial overlap
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return record_cuda_error(e);
    if (dev < 0 || dev >= 64) return FUSE_EUNSUPPORTED;
    HostPipe& hp = g_pipes[dev];
    std::lock_guard<std::mutex> lock(hp.mu);
    int rc = host_pipe_init(hp);
    if (rc != FUSE_OK) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    auto ok = [&](cudaError_t err) { return err == cudaSuccess ? FUSE_OK : record_cuda_error(err); };
    // the copies start after the work already queued on `stream`
    if ((rc = ok(cudaEventRecord(hp.entry, st))) || (rc = ok(cudaStreamWaitEvent(hp.s_in, hp.entry, 0))) ||
        (rc = ok(cudaStreamWaitEvent(hp.s_out, hp.entry, 0))))
        return rc;
    // Slice boundaries in whole 32-byte vectors (each slice keeps the vector path of the whole
    // call).  The first slice's copy in and the last slice's copy out overlap nothing, so with
    // three or more slices those two are a quarter of the size of the others (weights 1, 4, ...,
    // 4, 1): the pipeline fills and drains on small pieces.
    const int64_t wsum = slices >= 3 ? 4 * (slices - 2) + 2 : slices;
    auto bound = [&](int i) -> int64_t {   // first element of slice i (i = slices -> n)
        if (i <= 0) return 0;
        if (i >= slices) return n;
        const int64_t w = slices >= 3 ? 1 + 4 * (i - 1) : i;
        const int64_t e = static_cast<int64_t>(static_cast<double>(n) * static_cast<double>(w) /
                                               static_cast<double>(wsum));
        const int64_t a = e / 32 * 32;
        return a < n ? a : n;
    };
    for (int i = 0; i < slices; ++i) {
        const int64_t lo = bound(i), hi = bound(i + 1);
        if (hi <= lo) continue;
        const int64_t cnt = hi - lo;
        const size_t off = static_cast<size_t>(lo * eb), len = static_cast<size_t>(cnt * eb);
        if ((rc = ok(cudaMemcpyAsync(static_cast<char*>(x_dev) + off, static_cast<const char*>(x_host) + off, len,
                                     cudaMemcpyHostToDevice, hp.s_in))) ||
            (rc = ok(cudaEventRecord(hp.in, hp.s_in))) || (rc = ok(cudaStreamWaitEvent(st, hp.in, 0))))
            return rc;
        if ((rc = fuse_chain_run(stages, K, static_cast<const char*>(x_dev) + off, static_cast<char*>(y_dev) + off,
                                 cnt, dtype, mode, stream)))
            return rc;
        if ((rc = ok(cudaEventRecord(hp.run, st))) || (rc = ok(cudaStreamWaitEvent(hp.s_out, hp.run, 0))) ||
            (rc = ok(cudaMemcpyAsync(static_cast<char*>(y_host) + off, static_cast<const char*>(y_dev) + off, len,
                                     cudaMemcpyDeviceToHost, hp.s_out))))
            return rc;
    }
    // `stream` resumes once the last slice is back in host memory
    if ((rc = ok(cudaEventRecord(hp.out, hp.s_out))) || (rc = ok(cudaStreamWaitEvent(st, hp.out, 0)))) return rc;
    return FUSE_OK;
}

extern "C" int64_t fuse_chain_bytes(int K, int64_t n, int dtype, int mode) {
    if (K < 1 || K > FUSE_MAX_STAGES || n < 0) return FUSE_EINVAL;
    if (dtype != FUSE_F32 && dtype != FUSE_F16 && dtype != FUSE_BF16) return FUSE_EINVAL;
    const int64_t b = dtype == FUSE_F32 ? 4 : 2;
    // [OFCG] §3.2: every kernel reads N*b and writes N*b.
    if (mode == FUSE_UNFUSED) return 2 * static_cast<int64_t>(K) * n * b;
    if (mode == FUSE_FUSED || mode == FUSE_FAT) return 2 * n * b;
    return FUSE_EINVAL;
}
