// rmsnorm.cu -- RMSNorm, fused (one pass) and unfused (four kernels); and residual add + RMSNorm.
//
// [OFCG] §3.2 and fusion_lab [A2]: unfused RMSNorm is x*x -> reduce-mean -> x*r -> *g, each step
// a kernel that reads and writes HBM; fused it is one pass.  Per row i:
//     r_i = 1/sqrt(mean_j x_ij^2 + eps),   y_ij = (x_ij * r_i) * w_j.
// [OFCG] appendix launch_model [F3] also fuses the residual add into the RMSNorm that follows
// it: h = x + r (the new residual stream, written out), y = RMSNorm(h) * w, one pass, against a
// residual-add kernel followed by the four RMSNorm kernels unfused.
//
// GB300 design (fused): one CTA per row, the whole row in registers (16-byte vector loads, VPT
// vectors per thread, 512 threads for rows of 4096), a warp-shuffle reduction followed by a
// shared-memory reduction across the CTA's warps, then the scaled row written with 16-byte
// streaming stores.  x (and the residual) are read from HBM exactly once; w (16 KB at hidden 4096)
// stays in L1/L2.  An exact grid of short CTAs lets the hardware scheduler balance rows over the
// SMs: a persistent grid that prefetched the next row into registers lost ~8 % to its last,
// partial round of rows.  Instead, before its grid-dependency wait each CTA starts its own row and
// the row of the CTA one wave later on their way into L2 (bulk prefetches), so a launch's first
// reads overlap the end of the launch before it.
#include <cuda.h>

#include <mutex>

#include "fc_internal.cuh"

namespace fc {
namespace {

constexpr int kRowThreadsScalar = 512;
constexpr int kEwBlock = 256;

template <int THREADS>
__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    constexpr int W = THREADS / 32;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float t = 0.0f;
#pragma unroll
    for (int k = 0; k < W; ++k) t += red[k];
    return t;
}

// One CTA per row.  ADD: the row is h = x + res (one fp32 rounding per element), stored to h
// before it is normalised; h may be x or res itself (each element is read before the same thread
// writes it).  Rows are whole 16-byte vectors (hidden % 4 == 0, 16-byte aligned bases).
// Before the grid-dependency wait, the row's input, and that of row + ahead (the row this slot
// takes one wave later; ahead = 0: none), start on their way into L2 while the preceding kernel
// may still run.
template <int THR, int VPT, bool ADD>
__global__ void __launch_bounds__(THR) rmsnorm_row_kernel(const float* x, const float* res,
                                                          const float* __restrict__ w, float* h,
                                                          float* __restrict__ y, int hidden, float eps,
                                                          int ahead) {
    pdl_trigger();
    const int64_t row = blockIdx.x;
    if (threadIdx.x == 0) {
        const uint32_t bytes = static_cast<uint32_t>(hidden) * 4u;
        prefetch_l2_bulk(x + row * hidden, bytes);
        if (ADD) prefetch_l2_bulk(res + row * hidden, bytes);
        if (ahead > 0 && row + ahead < gridDim.x) {
            prefetch_l2_bulk(x + (row + ahead) * hidden, bytes);
            if (ADD) prefetch_l2_bulk(res + (row + ahead) * hidden, bytes);
        }
    }
    pdl_wait();  // before any global-memory load or store (programmatic dependent launch)
    __shared__ float red[THR / 32];
    const int nv = hidden / 4;
    const float4* xr = reinterpret_cast<const float4*>(x + row * hidden);
    float4 v[VPT];
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int idx = threadIdx.x + k * THR;
        v[k] = idx < nv ? __ldcs(xr + idx) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (ADD) {
        const float4* rr = reinterpret_cast<const float4*>(res + row * hidden);
        float4* hr = reinterpret_cast<float4*>(h + row * hidden);
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int idx = threadIdx.x + k * THR;
            if (idx < nv) {
                const float4 b = __ldcs(rr + idx);
                v[k].x = __fadd_rn(v[k].x, b.x); v[k].y = __fadd_rn(v[k].y, b.y);
                v[k].z = __fadd_rn(v[k].z, b.z); v[k].w = __fadd_rn(v[k].w, b.w);
                __stcs(hr + idx, v[k]);
            }
        }
    }
    float ss = 0.0f;
#pragma unroll
    for (int k = 0; k < VPT; ++k)
        ss += v[k].x * v[k].x + v[k].y * v[k].y + v[k].z * v[k].z + v[k].w * v[k].w;
    const float total = block_sum<THR>(ss, red);
    const float r = rsqrtf(__fdiv_rn(total, static_cast<float>(hidden)) + eps);
    const float4* wv = reinterpret_cast<const float4*>(w);
    float4* yr = reinterpret_cast<float4*>(y + row * hidden);
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int idx = threadIdx.x + k * THR;
        if (idx < nv) {
            const float4 g = __ldg(wv + idx);
            float4 o;
            o.x = __fmul_rn(__fmul_rn(v[k].x, r), g.x);
            o.y = __fmul_rn(__fmul_rn(v[k].y, r), g.y);
            o.z = __fmul_rn(__fmul_rn(v[k].z, r), g.z);
            o.w = __fmul_rn(__fmul_rn(v[k].w, r), g.w);
            __stcs(yr + idx, o);
        }
    }
}

// Element-wise variant for rows that are not whole 16-byte vectors (odd hidden or offsets).
template <int EPT, bool ADD>
__global__ void __launch_bounds__(kRowThreadsScalar) rmsnorm_fused_scalar_kernel(
    const float* x, const float* res, const float* __restrict__ w, float* h, float* __restrict__ y,
    int hidden, float eps) {
    pdl_begin();  // before any global-memory access (programmatic dependent launch)
    __shared__ float red[kRowThreadsScalar / 32];
    const int64_t row = blockIdx.x;
    const float* xr = x + row * hidden;
    float* yr = y + row * hidden;
    float v[EPT];
    float ss = 0.0f;
#pragma unroll
    for (int k = 0; k < EPT; ++k) {
        const int j = threadIdx.x + k * kRowThreadsScalar;
        v[k] = j < hidden ? xr[j] : 0.0f;
        if (ADD && j < hidden) {
            v[k] = __fadd_rn(v[k], res[row * hidden + j]);
            h[row * hidden + j] = v[k];
        }
        ss += v[k] * v[k];
    }
    const float total = block_sum<kRowThreadsScalar>(ss, red);
    const float r = rsqrtf(__fdiv_rn(total, static_cast<float>(hidden)) + eps);
#pragma unroll
    for (int k = 0; k < EPT; ++k) {
        const int j = threadIdx.x + k * kRowThreadsScalar;
        if (j < hidden) yr[j] = __fmul_rn(__fmul_rn(v[k], r), w[j]);
    }
}

// ------------------------------------------------------------------------- unfused kernels
// (0, residual form only) h = x + res
__global__ void __launch_bounds__(kEwBlock) residual_add_kernel(const float* x, const float* res,
                                                                float* h, int64_t n, bool vec) {
    pdl_begin();  // before any global-memory access (programmatic dependent launch)
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t nthr = static_cast<int64_t>(gridDim.x) * blockDim.x;
    int64_t done = 0;
    if (vec) {
        const int64_t nv = n / 4;
        for (int64_t i = tid; i < nv; i += nthr) {
            float4 a = __ldcs(reinterpret_cast<const float4*>(x) + i);
            const float4 b = __ldcs(reinterpret_cast<const float4*>(res) + i);
            a.x = __fadd_rn(a.x, b.x); a.y = __fadd_rn(a.y, b.y);
            a.z = __fadd_rn(a.z, b.z); a.w = __fadd_rn(a.w, b.w);
            __stcs(reinterpret_cast<float4*>(h) + i, a);
        }
        done = nv * 4;
    }
    for (int64_t i = done + tid; i < n; i += nthr) h[i] = __fadd_rn(x[i], res[i]);
}

// (1) sq = x*x   (2) ms = rowmean(sq)   (3) t = x * rsqrt(ms + eps)   (4) y = t * w
__global__ void __launch_bounds__(kEwBlock) rms_square_kernel(const float* __restrict__ x,
                                                              float* __restrict__ y, int64_t n,
                                                              bool vec) {
    pdl_begin();  // before any global-memory access (programmatic dependent launch)
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t nthr = static_cast<int64_t>(gridDim.x) * blockDim.x;
    int64_t done = 0;
    if (vec) {
        const int64_t nv = n / 4;
        for (int64_t i = tid; i < nv; i += nthr) {
            float4 a = __ldcs(reinterpret_cast<const float4*>(x) + i);
            a.x = __fmul_rn(a.x, a.x); a.y = __fmul_rn(a.y, a.y);
            a.z = __fmul_rn(a.z, a.z); a.w = __fmul_rn(a.w, a.w);
            __stcs(reinterpret_cast<float4*>(y) + i, a);
        }
        done = nv * 4;
    }
    for (int64_t i = done + tid; i < n; i += nthr) y[i] = __fmul_rn(x[i], x[i]);
}

__global__ void __launch_bounds__(kRowThreadsScalar) rms_rowmean_kernel(
    const float* __restrict__ sq, float* __restrict__ ms, int hidden) {
    pdl_begin();  // before any global-memory access (programmatic dependent launch)
    __shared__ float red[kRowThreadsScalar / 32];
    const int64_t row = blockIdx.x;
    const float* r = sq + row * hidden;
    float acc = 0.0f;
    for (int j = threadIdx.x; j < hidden; j += kRowThreadsScalar) acc += __ldcs(r + j);
    const float total = block_sum<kRowThreadsScalar>(acc, red);
    if (threadIdx.x == 0) ms[row] = __fdiv_rn(total, static_cast<float>(hidden));
}

__global__ void __launch_bounds__(kEwBlock) rms_scale_kernel(const float* __restrict__ x,
                                                             const float* __restrict__ ms,
                                                             float* __restrict__ y, int64_t n,
                                                             int hidden, float eps, bool vec) {
    pdl_begin();  // before any global-memory access (programmatic dependent launch)
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t nthr = static_cast<int64_t>(gridDim.x) * blockDim.x;
    if (vec) {  // hidden % 4 == 0: a vector never straddles two rows
        const int64_t nv = n / 4;
        const int vpr = hidden / 4;
        for (int64_t i = tid; i < nv; i += nthr) {
            const float r = rsqrtf(__ldg(ms + i / vpr) + eps);
            float4 a = __ldcs(reinterpret_cast<const float4*>(x) + i);
            a.x = __fmul_rn(a.x, r); a.y = __fmul_rn(a.y, r);
            a.z = __fmul_rn(a.z, r); a.w = __fmul_rn(a.w, r);
            __stcs(reinterpret_cast<float4*>(y) + i, a);
        }
        return;
    }
    for (int64_t i = tid; i < n; i += nthr) y[i] = __fmul_rn(x[i], rsqrtf(ms[i / hidden] + eps));
}

__global__ void __launch_bounds__(kEwBlock) rms_weight_kernel(float* __restrict__ y,
                                                              const float* __restrict__ w,
                                                              int64_t n, int hidden, bool vec) {
    pdl_begin();  // before any global-memory access (programmatic dependent launch)
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t nthr = static_cast<int64_t>(gridDim.x) * blockDim.x;
    if (vec) {
        const int64_t nv = n / 4;
        const int vpr = hidden / 4;
        for (int64_t i = tid; i < nv; i += nthr) {
            const float4 g = __ldg(reinterpret_cast<const float4*>(w) + i % vpr);
            float4 a = __ldcs(reinterpret_cast<const float4*>(y) + i);
            a.x = __fmul_rn(a.x, g.x); a.y = __fmul_rn(a.y, g.y);
            a.z = __fmul_rn(a.z, g.z); a.w = __fmul_rn(a.w, g.w);
            __stcs(reinterpret_cast<float4*>(y) + i, a);
        }
        return;
    }
    for (int64_t i = tid; i < n; i += nthr) y[i] = __fmul_rn(y[i], w[i % hidden]);
}

template <int THR, int VPT, bool ADD>
int launch_fused_vec(const float* x, const float* res, const float* w, float* h, float* y,
                     int64_t rows, int hidden, float eps, cudaStream_t st) {
    // The residual form reads two rows per CTA: prefetching the next wave's rows as well measured
    // no faster (22.34 -> 22.31 us at [2048, 4096]) and read 7 % more from DRAM (lines evicted
    // before their use), so it prefetches its own rows only.
    static const int occ = blocks_per_sm(rmsnorm_row_kernel<THR, VPT, ADD>, THR);
    const int ahead = ADD ? 0 : sm_count() * occ;
    return launch_pdl(rmsnorm_row_kernel<THR, VPT, ADD>, dim3(static_cast<unsigned>(rows)), dim3(THR), 0, st, 1, x, res, w, h, y, hidden, eps, ahead);
}

template <int EPT, bool ADD>
int launch_fused_scalar(const float* x, const float* res, const float* w, float* h, float* y,
                        int64_t rows, int hidden, float eps, cudaStream_t st) {
    return launch_pdl(rmsnorm_fused_scalar_kernel<EPT, ADD>, dim3(static_cast<unsigned>(rows)), dim3(kRowThreadsScalar), 0, st, 1, x, res, w, h, y, hidden, eps);
}

// The fused form for hidden <= 16384: the row lives in registers (VPT float4 or EPT floats per
// thread).  With ADD the row is x + res and is also stored to h.
template <bool ADD>
int fused_dispatch(const float* x, const float* res, const float* w, float* h, float* y,
                   int64_t rows, int H, float eps, bool vec, cudaStream_t st) {
    if (H > 16384) return FUSE_EUNSUPPORTED;
    if (vec) {
        const int nv = H / 4;
        if (nv <= 128) return launch_fused_vec<128, 1, ADD>(x, res, w, h, y, rows, H, eps, st);
        if (nv <= 256) return launch_fused_vec<256, 1, ADD>(x, res, w, h, y, rows, H, eps, st);
        if (nv <= 512) return launch_fused_vec<512, 1, ADD>(x, res, w, h, y, rows, H, eps, st);
        if (nv <= 1024) return launch_fused_vec<512, 2, ADD>(x, res, w, h, y, rows, H, eps, st);
        if (nv <= 2048) return launch_fused_vec<512, 4, ADD>(x, res, w, h, y, rows, H, eps, st);
        return launch_fused_vec<512, 8, ADD>(x, res, w, h, y, rows, H, eps, st);
    }
    if (H <= 1 * kRowThreadsScalar) return launch_fused_scalar<1, ADD>(x, res, w, h, y, rows, H, eps, st);
    if (H <= 2 * kRowThreadsScalar) return launch_fused_scalar<2, ADD>(x, res, w, h, y, rows, H, eps, st);
    if (H <= 4 * kRowThreadsScalar) return launch_fused_scalar<4, ADD>(x, res, w, h, y, rows, H, eps, st);
    if (H <= 8 * kRowThreadsScalar) return launch_fused_scalar<8, ADD>(x, res, w, h, y, rows, H, eps, st);
    if (H <= 16 * kRowThreadsScalar) return launch_fused_scalar<16, ADD>(x, res, w, h, y, rows, H, eps, st);
    return launch_fused_scalar<32, ADD>(x, res, w, h, y, rows, H, eps, st);
}

unsigned ew_grid(int64_t units) {
    const int64_t cap = static_cast<int64_t>(sm_count()) * (2048 / kEwBlock);
    int64_t g = ceil_div(units, kEwBlock);
    if (g > cap) g = cap;
    return static_cast<unsigned>(g < 1 ? 1 : g);
}

}  // namespace

// The four unfused RMSNorm kernels on x (the residual form passes h as x); y != x.
int unfused_steps(const float* x, const float* w, float* y, float* ms, int64_t rows, int H,
                  float eps, bool vec, cudaStream_t st) {
    const int64_t n = rows * H;
    const bool fvec = is_aligned(x, 16) && is_aligned(y, 16);
    int rc = launch_pdl(rms_square_kernel, dim3(ew_grid(fvec ? n / 4 : n)), dim3(kEwBlock), 0, st, 1, x, y, n, fvec);
    if (rc) return rc;
    if ((rc = launch_pdl(rms_rowmean_kernel, dim3(static_cast<unsigned>(rows)), dim3(kRowThreadsScalar), 0, st, 1, y, ms, H))) return rc;
    if ((rc = launch_pdl(rms_scale_kernel, dim3(ew_grid(vec ? n / 4 : n)), dim3(kEwBlock), 0, st, 1, x, ms, y, n, H, eps, vec))) return rc;
    return launch_pdl(rms_weight_kernel, dim3(ew_grid(vec ? n / 4 : n)), dim3(kEwBlock), 0, st, 1, y, w, n, H, vec);
}

int rmsnorm_report_count() { return 4; }
int rmsnorm_report(int i, fuse_kernel_record* out) {
    switch (i) {
        case 0: return describe_kernel((const void*)rmsnorm_row_kernel<512, 2, false>,
                                       "rmsnorm_row_kernel<512 thr, VPT=2> (hidden 4096)", 512, 0, out);
        case 3: return describe_kernel((const void*)rmsnorm_row_kernel<512, 2, true>,
                                       "rmsnorm_row_kernel<512 thr, VPT=2, +residual> (hidden 4096)",
                                       512, 0, out);
        case 1: return describe_kernel((const void*)rms_rowmean_kernel,
                                       "rms_rowmean_kernel (unfused step 2)", kRowThreadsScalar, 0, out);
        case 2: return describe_kernel((const void*)rms_scale_kernel,
                                       "rms_scale_kernel (unfused step 3)", kEwBlock, 0, out);
        default: return FUSE_EINVAL;
    }
}

}  // namespace fc

extern "C" size_t fuse_rmsnorm_workspace_bytes(int64_t rows, int64_t hidden, int mode) {
    (void)hidden;
    if (rows < 0) return 0;
    return mode == FUSE_UNFUSED ? static_cast<size_t>(rows) * sizeof(float) : 0;
}

extern "C" int fuse_rmsnorm(const float* x, const float* w, float* y, int64_t rows, int64_t hidden,
                            float eps, int mode, void* workspace, size_t ws_bytes,
                            fuse_stream_t stream) {
    using namespace fc;
    if (rows < 0 || hidden < 1 || hidden > 65536 || !(eps >= 0.0f)) return FUSE_EINVAL;
    if (mode != FUSE_FUSED && mode != FUSE_UNFUSED) return FUSE_EINVAL;
    if (rows > 2147483647LL) return FUSE_EUNSUPPORTED;
    if (rows == 0) return FUSE_OK;
    if (!x || !w || !y) return FUSE_EINVAL;
    if (!is_aligned(x, 4) || !is_aligned(w, 4) || !is_aligned(y, 4)) return FUSE_EALIGN;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int H = static_cast<int>(hidden);
    const bool vec = (H % 4 == 0) && is_aligned(x, 16) && is_aligned(y, 16) && is_aligned(w, 16);

    if (mode == FUSE_FUSED) return fused_dispatch<false>(x, nullptr, w, nullptr, y, rows, H, eps, vec, st);

    // FUSE_UNFUSED: four kernels; the N-sized intermediates live in y, the row means in workspace.
    if (!workspace || ws_bytes < fuse_rmsnorm_workspace_bytes(rows, hidden, mode)) return FUSE_EWORKSPACE;
    if (!is_aligned(workspace, 4)) return FUSE_EALIGN;
    if (x == y) return FUSE_EINVAL;  // step 3 re-reads x after step 1 overwrote y
    return unfused_steps(x, w, y, static_cast<float*>(workspace), rows, H, eps, vec, st);
}

extern "C" int fuse_add_rmsnorm(const float* x, const float* r, const float* w, float* h, float* y,
                                int64_t rows, int64_t hidden, float eps, int mode, void* workspace,
                                size_t ws_bytes, fuse_stream_t stream) {
    using namespace fc;
    if (rows < 0 || hidden < 1 || hidden > 65536 || !(eps >= 0.0f)) return FUSE_EINVAL;
    if (mode != FUSE_FUSED && mode != FUSE_UNFUSED) return FUSE_EINVAL;
    if (rows > 2147483647LL) return FUSE_EUNSUPPORTED;
    if (rows == 0) return FUSE_OK;
    if (!x || !r || !w || !h || !y) return FUSE_EINVAL;
    if (y == x || y == r || y == h) return FUSE_EINVAL;  // h may be x or r (in place), y may not
    if (!is_aligned(x, 4) || !is_aligned(r, 4) || !is_aligned(w, 4) || !is_aligned(h, 4) ||
        !is_aligned(y, 4))
        return FUSE_EALIGN;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int H = static_cast<int>(hidden);
    const bool vec = (H % 4 == 0) && is_aligned(x, 16) && is_aligned(r, 16) && is_aligned(h, 16) &&
                     is_aligned(y, 16) && is_aligned(w, 16);
    if (mode == FUSE_FUSED) return fused_dispatch<true>(x, r, w, h, y, rows, H, eps, vec, st);

    // FUSE_UNFUSED: the residual-add kernel, then the four RMSNorm kernels on h.
    if (!workspace || ws_bytes < fuse_rmsnorm_workspace_bytes(rows, hidden, mode)) return FUSE_EWORKSPACE;
    if (!is_aligned(workspace, 4)) return FUSE_EALIGN;
    const int64_t n = rows * hidden;
    const bool avec = is_aligned(x, 16) && is_aligned(r, 16) && is_aligned(h, 16);
    const int rc = launch_pdl(residual_add_kernel, dim3(ew_grid(avec ? n / 4 : n)), dim3(kEwBlock), 0, st, 1, x, r, h, n, avec);
    if (rc) return rc;
    return unfused_steps(h, w, y, static_cast<float*>(workspace), rows, H, eps, vec, st);
}

extern "C" int64_t fuse_add_rmsnorm_bytes(int64_t rows, int64_t hidden, int mode) {
    if (rows < 0 || hidden < 1) return FUSE_EINVAL;
    const int64_t n = rows * hidden, b = 4;
    // fused: read x and r, write h and y, read w once
    if (mode == FUSE_FUSED) return 4 * n * b + hidden * b;
    // unfused: add (r x, r r, w h) + the four RMSNorm kernels on h (7 N b + row means + w)
    if (mode == FUSE_UNFUSED) return 10 * n * b + 2 * rows * b + hidden * b;
    return FUSE_EINVAL;
}

extern "C" int64_t fuse_rmsnorm_bytes(int64_t rows, int64_t hidden, int mode) {
    if (rows < 0 || hidden < 1) return FUSE_EINVAL;
    const int64_t n = rows * hidden, b = 4;
    // fused: read x, write y, read w once
    if (mode == FUSE_FUSED) return 2 * n * b + hidden * b;
    // unfused: sq (r x, w y) + mean (r y, w ms) + scale (r x, r ms, w y) + weight (r y, r w, w y)
    if (mode == FUSE_UNFUSED) return 7 * n * b + 2 * rows * b + hidden * b;
    return FUSE_EINVAL;
}

// ------------------------------------------------------------------------- allocation-free entry
// The four-kernel unfused RMSNorm with its row statistics in a fixed, library-owned device array
// instead of a caller workspace, for callers that cannot allocate device memory.  The array lives
// for the life of the process on every device that loads this library.
namespace {
constexpr int64_t kStaticMaxRows = 65536;  // 256 KiB of fp32 row statistics
__device__ __align__(256) float g_rms_static_ms[kStaticMaxRows];

// The driver's process-unique id of the calling thread's current context (0 if there is none
// or the driver entry points are missing).  Driver calls are reached through the runtime's entry
// point query, so the library needs no link against libcuda.
unsigned long long current_context_id() {
    using GetCurrentFn = CUresult (*)(CUcontext*);
    using GetIdFn = CUresult (*)(CUcontext, unsigned long long*);
    static GetCurrentFn get_current = nullptr;
    static GetIdFn get_id = nullptr;
    static bool looked = false;
    if (!looked) {  // called under the entry point's mutex
        looked = true;
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrentFn>(p);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetIdFn>(p);
        (void)cudaGetLastError();
    }
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}
}  // namespace


extern "C" int fuse_rmsnorm_unfused_static(const float* x, const float* w, float* y, int64_t rows,
                                           int64_t hidden, float eps, fuse_stream_t stream) {
    using namespace fc;
    if (rows < 0 || hidden < 1 || hidden > 65536 || !(eps >= 0.0f)) return FUSE_EINVAL;
    if (rows > kStaticMaxRows) return FUSE_EUNSUPPORTED;
    if (rows == 0) return FUSE_OK;
    if (!x || !w || !y || x == y) return FUSE_EINVAL;
    if (!is_aligned(x, 4) || !is_aligned(w, 4) || !is_aligned(y, 4)) return FUSE_EALIGN;

    // Host code cannot use the array's name as a device address: look the address up once per
    // device, with that device current, and keep it for as long as that device's context lives.
    // The cache is keyed by the driver's unique context id, so after cudaDeviceReset() (a new
    // primary context, into which the module is loaded again, maybe at another address) the next
    // call looks the address up afresh instead of launching on a stale pointer.
    static std::mutex mu;
    static float* dev_ms[64] = {nullptr};
    static unsigned long long dev_ctx[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return record_cuda_error(e);
    if (dev < 0 || dev >= 64) return FUSE_EUNSUPPORTED;
    float* ms = nullptr;
    {
        std::lock_guard<std::mutex> lock(mu);
        unsigned long long ctx = current_context_id();
        if (!dev_ms[dev] || ctx == 0 || ctx != dev_ctx[dev]) {
            void* p = nullptr;
            e = cudaGetSymbolAddress(&p, g_rms_static_ms);
            if (e != cudaSuccess) return record_cuda_error(e);
            dev_ms[dev] = static_cast<float*>(p);
            dev_ctx[dev] = current_context_id();  // the lookup made the device's context current
        }
        ms = dev_ms[dev];
    }

    // Same four kernels as the unfused mode of fuse_rmsnorm().  Every row statistic the later
    // kernels read is written by the row-mean kernel of the same call, so nothing is cleared.
    const int H = static_cast<int>(hidden);
    const bool vec = (H % 4 == 0) && is_aligned(x, 16) && is_aligned(y, 16) && is_aligned(w, 16);
    return unfused_steps(x, w, y, ms, rows, H, eps, vec, reinterpret_cast<cudaStream_t>(stream));
}
