// silu_mul.cu -- y = SiLU(gate) * up, fused (one pass) and unfused (two kernels).
//
// "AIGC fundamentals | operator fusion and CUDA Graph", appendix launch_model [F3]: in the
// per-layer kernel list of a decoder, the gate/up projection is one GEMM and "SiLU + multiply"
// one fused kernel, where the unfused list runs a SiLU kernel and an element-wise multiply
// kernel.  SiLU(v) = v * logistic(v) = v / (1 + e^-v).  Byte ledgers (b = element bytes,
// N = rows * cols): fused reads g and u and writes y, 3 N b; unfused writes s = SiLU(g) and reads
// it back, 2 N b + 3 N b = 5 N b.
//
// GB300 design: pure HBM streaming, shaped like the pointwise chain: one 32-byte vector of gate,
// one of up and one of y per thread (256-bit ld/st.global.cs), an exact grid of short CTAs.  g and
// u share a row stride, so the two halves of one merged gate/up GEMM output [rows, 2 cols] are
// read in place.  SiLU in fp32: one ex2 and one reciprocal on the SFU per element (2 SFU ops per
// 2-byte element keep the SFU below the HBM time at bf16).
#include "fc_internal.cuh"

namespace fc {
namespace {

constexpr int kBlock = 256;

// Steps: the fused kernel computes y = SiLU(g) * u; the unfused form runs kSilu (y = SiLU(g),
// rounded to the storage type) then kMul (y = y * u).
enum Step : int { kFused = 0, kSilu = 1, kMul = 2 };

struct SiluParams {
    const void* g;
    const void* u;
    void* y;
    int64_t rows, cols, ld;  // g and u: row stride ld elements; y: row stride cols
    int64_t vpr;             // 32-byte vectors per row (vector path)
    int64_t nvec;            // rows * vpr
    int64_t ahead;           // vector path: CTAs one wave later, whose input is prefetched too
};

__device__ __forceinline__ float ex2_approx(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// v / (1 + e^-v) with e^-v = 2^(-v log2 e).  Far negative v: e^-v -> +inf, the reciprocal -> 0,
// so the result is -0; far positive v: e^-v -> 0 and the result is v.
__device__ __forceinline__ float silu_f32(float v) {
    constexpr float kLog2e = 1.4426950408889634f;
    const float e = ex2_approx(-v * kLog2e);
    return v * rcp_approx(1.0f + e);
}

template <int STEP>
__device__ __forceinline__ float apply(float gv, float uv, float yv) {
    if (STEP == kFused) return silu_f32(gv) * uv;
    if (STEP == kSilu) return silu_f32(gv);
    return yv * uv;
}

// The inputs CTA `cta` reads from DRAM (g and u; u alone for the multiply step, whose y is the
// intermediate the preceding step just wrote) on their way into L2: one contiguous range per row
// its vectors touch, at most two (a CTA's vectors cross at most one row boundary when a row holds
// at least a CTA's worth of them; narrower rows are left to the loads).  Ranges start on 32-byte
// vector boundaries and are whole vectors long.
template <typename T, int STEP>
__device__ __forceinline__ void prefetch_share(const SiluParams& p, int64_t cta) {
    const int64_t t0 = cta * kBlock;
    if (t0 >= p.nvec) return;
    const int64_t t1 = t0 + kBlock < p.nvec ? t0 + kBlock : p.nvec;
    constexpr int E = Vec32<T>::N;
    int64_t t = t0;
    for (int seg = 0; seg < 2 && t < t1; ++seg) {
        const int64_t row = t / p.vpr;
        const int64_t end = t1 < (row + 1) * p.vpr ? t1 : (row + 1) * p.vpr;
        const int64_t src = row * p.ld + (t - row * p.vpr) * E;
        const uint32_t bytes = static_cast<uint32_t>(end - t) * 32u;
        if (STEP != kMul) prefetch_l2_bulk(static_cast<const T*>(p.g) + src, bytes);
        if (STEP != kSilu) prefetch_l2_bulk(static_cast<const T*>(p.u) + src, bytes);
        t = end;
    }
}

// Before the grid-dependency wait, the CTA's own inputs and those of the CTA one wave later start
// on their way into L2 while the preceding kernel may still run (the pointwise chain's scheme).
template <typename T, int STEP>
__global__ void __launch_bounds__(kBlock) silu_mul_vec_kernel(const __grid_constant__ SiluParams p) {
    pdl_trigger();
    if (threadIdx.x == 0) {
        prefetch_share<T, STEP>(p, blockIdx.x);
        if (p.ahead > 0) prefetch_share<T, STEP>(p, static_cast<int64_t>(blockIdx.x) + p.ahead);
    }
    pdl_wait();  // before any global-memory load or store (programmatic dependent launch)
    using V = Vec32<T>;
    constexpr int E = V::N;
    const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (t >= p.nvec) return;
    const int64_t row = t / p.vpr;
    const int64_t c = (t - row * p.vpr) * E;
    const int64_t src = row * p.ld + c, dst = row * p.cols + c;
    float a[E], b[E];
    if (STEP == kMul) {
        V::load(static_cast<const T*>(p.y) + dst, a);
        V::load(static_cast<const T*>(p.u) + src, b);
#pragma unroll
        for (int e = 0; e < E; ++e) a[e] = apply<kMul>(0.0f, b[e], a[e]);
    } else {
        V::load(static_cast<const T*>(p.g) + src, a);
        if (STEP == kFused) V::load(static_cast<const T*>(p.u) + src, b);
#pragma unroll
        for (int e = 0; e < E; ++e) a[e] = apply<STEP>(a[e], STEP == kFused ? b[e] : 0.0f, 0.0f);
    }
    V::store(static_cast<T*>(p.y) + dst, a);
}

// Element-wise variant for shapes or pointers the 32-byte vectors do not fit.
template <typename T, int STEP>
__global__ void __launch_bounds__(kBlock) silu_mul_scalar_kernel(const __grid_constant__ SiluParams p) {
    pdl_begin();  // before any global-memory access (programmatic dependent launch)
    const int64_t n = p.rows * p.cols;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const T* g = static_cast<const T*>(p.g);
    const T* u = static_cast<const T*>(p.u);
    T* y = static_cast<T*>(p.y);
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
        const int64_t row = i / p.cols, c = i - row * p.cols;
        const int64_t src = row * p.ld + c;
        const float gv = STEP == kMul ? 0.0f : to_f32(g[src]);
        const float uv = STEP == kSilu ? 0.0f : to_f32(u[src]);
        const float yv = STEP == kMul ? to_f32(y[i]) : 0.0f;
        y[i] = from_f32<T>(apply<STEP>(gv, uv, yv));
    }
}

template <typename T, int STEP>
int launch(const SiluParams& p, bool vec, cudaStream_t st) {
    if (vec) {
        const int64_t grid = ceil_div(p.nvec, kBlock);
        if (grid > 0x7fffffffLL) return FUSE_EUNSUPPORTED;
        static const int occ = blocks_per_sm(silu_mul_vec_kernel<T, STEP>, kBlock);
        SiluParams q = p;
        q.ahead = static_cast<int64_t>(sm_count()) * occ;
        return launch_pdl(silu_mul_vec_kernel<T, STEP>, dim3(static_cast<unsigned>(grid)), dim3(kBlock), 0, st, 1, q);
    } else {
        int64_t grid = ceil_div(p.rows * p.cols, kBlock);
        const int64_t cap = static_cast<int64_t>(sm_count()) * (2048 / kBlock) * 4;
        if (grid > cap) grid = cap;
        return launch_pdl(silu_mul_scalar_kernel<T, STEP>, dim3(static_cast<unsigned>(grid)), dim3(kBlock), 0, st,
                          1, p);
    }
}

template <typename T>
int run(const SiluParams& p, bool vec, int mode, cudaStream_t st) {
    if (mode == FUSE_FUSED) return launch<T, kFused>(p, vec, st);
    int rc = launch<T, kSilu>(p, vec, st);
    if (rc) return rc;
    return launch<T, kMul>(p, vec, st);
}

bool overlaps(const void* a, int64_t a_bytes, const void* b, int64_t b_bytes) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + static_cast<uintptr_t>(b_bytes) && y < x + static_cast<uintptr_t>(a_bytes);
}

}  // namespace

int silu_report_count() { return 2; }
int silu_report(int i, fuse_kernel_record* out) {
    switch (i) {
        case 0: return describe_kernel((const void*)silu_mul_vec_kernel<__nv_bfloat16, kFused>,
                                       "silu_mul_vec_kernel<bf16> (fused)", kBlock, 0, out);
        case 1: return describe_kernel((const void*)silu_mul_vec_kernel<__nv_bfloat16, kSilu>,
                                       "silu_mul_vec_kernel<bf16> (unfused SiLU step)", kBlock, 0, out);
        default: return FUSE_EINVAL;
    }
}

}  // namespace fc

extern "C" int fuse_silu_mul(const void* g, const void* u, int64_t ld, void* y, int64_t rows,
                             int64_t cols, int dtype, int mode, fuse_stream_t stream) {
    using namespace fc;
    if (rows < 0 || cols < 0 || ld < cols) return FUSE_EINVAL;
    if (dtype != FUSE_F32 && dtype != FUSE_F16 && dtype != FUSE_BF16) return FUSE_EINVAL;
    if (mode != FUSE_FUSED && mode != FUSE_UNFUSED) return FUSE_EINVAL;
    if (rows == 0 || cols == 0) return FUSE_OK;
    if (!g || !u || !y) return FUSE_EINVAL;
    const int64_t eb = dtype == FUSE_F32 ? 4 : 2;
    if (rows > (int64_t(1) << 40) / ld) return FUSE_EUNSUPPORTED;
    if (!is_aligned(g, eb) || !is_aligned(u, eb) || !is_aligned(y, eb)) return FUSE_EALIGN;
    // y must not overlap up (the unfused form writes y before it reads up); it may be gate itself
    // only when both are dense (ld == cols), element i then being read before it is written
    const int64_t in_bytes = ((rows - 1) * ld + cols) * eb, out_bytes = rows * cols * eb;
    if (overlaps(y, out_bytes, u, in_bytes)) return FUSE_EINVAL;
    if (overlaps(y, out_bytes, g, in_bytes) && !(y == g && ld == cols)) return FUSE_EINVAL;
    SiluParams p{g, u, y, rows, cols, ld, 0, 0, 0};
    const int64_t E = 32 / eb;
    const bool vec = cols % E == 0 && ld % E == 0 && is_aligned(g, 32) && is_aligned(u, 32) &&
                     is_aligned(y, 32);
    if (vec) {
        p.vpr = cols / E;
        p.nvec = rows * p.vpr;
    }
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (dtype == FUSE_F32) return run<float>(p, vec, mode, st);
    if (dtype == FUSE_F16) return run<__half>(p, vec, mode, st);
    return run<__nv_bfloat16>(p, vec, mode, st);
}

extern "C" int64_t fuse_silu_mul_bytes(int64_t rows, int64_t cols, int dtype, int mode) {
    if (rows < 0 || cols < 0) return FUSE_EINVAL;
    if (dtype != FUSE_F32 && dtype != FUSE_F16 && dtype != FUSE_BF16) return FUSE_EINVAL;
    const int64_t n = rows * cols, b = dtype == FUSE_F32 ? 4 : 2;
    if (mode == FUSE_FUSED) return 3 * n * b;    // read g, u; write y
    if (mode == FUSE_UNFUSED) return 5 * n * b;  // SiLU: read g, write s; mul: read s, u, write y
    return FUSE_EINVAL;
}
