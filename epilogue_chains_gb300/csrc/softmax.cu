// softmax.cu -- causal attention-score softmax over the last axis of s[BH, S, S] (bf16).
//
// [OFCG] fusion_lab [E]: softmax is max -> subtract -> exp -> sum -> divide over a row; unfused,
// each step reads (and the elementwise ones write) the whole score tensor: 8 copies of it,
// against 2 fused ([A3]).  §3.5: query i sees keys j <= i; skipping whole key blocks of a T x T
// tiling leaves the fraction (n_b + 1)/(2 n_b) of the blocks to read.
//
// GB300 design (fused): one warp per row, the row's kept columns loaded as 16 B vectors (8 bf16)
// straight into registers, a warp-shuffle max and sum (no shared memory, no block barrier), the
// exponentials kept in registers, one 16 B streaming store per 8 outputs.  With skip tile T,
// row i loads only the columns < (floor(i/T)+1)*T and writes zeros past them without reading.
#include <math.h>

#include "fc_internal.cuh"

namespace fc {
namespace {

constexpr int kWarpsPerBlock = 8;
constexpr int kSmBlock = 32 * kWarpsPerBlock;
constexpr int kEwBlock = 256;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <typename OutT> struct OutVec;
template <> struct OutVec<__nv_bfloat16> {  // 8 outputs = one 16 B store
    __device__ __forceinline__ static void store(__nv_bfloat16* row, int v, const float* f) {
        __stcs(reinterpret_cast<uint4*>(row) + v, Vec16<__nv_bfloat16>::pack(f));
    }
    __device__ __forceinline__ static void zero(__nv_bfloat16* row, int v) {
        __stcs(reinterpret_cast<uint4*>(row) + v, make_uint4(0, 0, 0, 0));
    }
};
template <> struct OutVec<float> {  // 8 outputs = two 16 B stores
    __device__ __forceinline__ static void store(float* row, int v, const float* f) {
        __stcs(reinterpret_cast<float4*>(row) + 2 * v, make_float4(f[0], f[1], f[2], f[3]));
        __stcs(reinterpret_cast<float4*>(row) + 2 * v + 1, make_float4(f[4], f[5], f[6], f[7]));
    }
    __device__ __forceinline__ static void zero(float* row, int v) {
        __stcs(reinterpret_cast<float4*>(row) + 2 * v, make_float4(0.f, 0.f, 0.f, 0.f));
        __stcs(reinterpret_cast<float4*>(row) + 2 * v + 1, make_float4(0.f, 0.f, 0.f, 0.f));
    }
};

// Fused, register-resident: S % 8 == 0 and S <= 256 * VPL.
template <int VPL, typename OutT>
__global__ void __launch_bounds__(kSmBlock) softmax_fused_kernel(
    const __nv_bfloat16* __restrict__ s, OutT* __restrict__ p, int64_t rows, int S, float scale,
    int skip_tile) {
    const int lane = threadIdx.x % 32;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + threadIdx.x / 32;
    if (row >= rows) return;
    const int i = static_cast<int>(row % S);  // query index inside its (batch, head)
    const int ncols = skip_tile > 0 ? min(S, (i / skip_tile + 1) * skip_tile) : S;
    const int nvec_load = ncols / 8;
    const int nvec = S / 8;
    const uint4* srow = reinterpret_cast<const uint4*>(s + row * S);
    OutT* prow = p + row * S;

    float f[VPL][8];
#pragma unroll
    for (int u = 0; u < VPL; ++u) {
        const int v = lane + 32 * u;
        uint4 r = make_uint4(0, 0, 0, 0);
        if (v < nvec_load) r = __ldcs(srow + v);
        Vec16<__nv_bfloat16>::unpack(r, f[u]);
    }
    float mx = -INFINITY;
#pragma unroll
    for (int u = 0; u < VPL; ++u) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int col = 8 * (lane + 32 * u) + e;
            const float z = f[u][e] * scale;
            f[u][e] = z;
            if (col <= i) mx = fmaxf(mx, z);
        }
    }
    mx = warp_max(mx);
    float sum = 0.0f;
#pragma unroll
    for (int u = 0; u < VPL; ++u) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int col = 8 * (lane + 32 * u) + e;
            const float ev = col <= i ? __expf(f[u][e] - mx) : 0.0f;
            f[u][e] = ev;
            sum += ev;
        }
    }
    sum = warp_sum(sum);
    const float inv = __frcp_rn(sum);
#pragma unroll
    for (int u = 0; u < VPL; ++u) {
        const int v = lane + 32 * u;
        if (v < nvec) {
            if (v < nvec_load) {
#pragma unroll
                for (int e = 0; e < 8; ++e) f[u][e] = __fmul_rn(f[u][e], inv);
                OutVec<OutT>::store(prow, v, f[u]);
            } else {
                OutVec<OutT>::zero(prow, v);
            }
        }
    }
}

// Fused, any S (<= 8192) and any alignment: pass 1 folds the row into a running (max, sum) per
// lane and merges the lanes; pass 2 re-reads the kept scores and writes every output.
template <typename OutT>
__global__ void __launch_bounds__(kSmBlock) softmax_fused_generic_kernel(
    const __nv_bfloat16* __restrict__ s, OutT* __restrict__ p, int64_t rows, int S, float scale,
    int skip_tile) {
    const int lane = threadIdx.x % 32;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + threadIdx.x / 32;
    if (row >= rows) return;
    const int i = static_cast<int>(row % S);
    const int ncols = skip_tile > 0 ? min(S, (i / skip_tile + 1) * skip_tile) : S;
    const __nv_bfloat16* srow = s + row * S;
    OutT* prow = p + row * S;
    float m = -INFINITY, l = 0.0f;
    for (int j = lane; j < ncols && j <= i; j += 32) {
        const float z = __bfloat162float(srow[j]) * scale;
        const float mn = fmaxf(m, z);
        l = l * __expf(m - mn) + __expf(z - mn);
        m = mn;
    }
    const float M = warp_max(m);
    l = (m == -INFINITY) ? 0.0f : l * __expf(m - M);
    const float inv = __frcp_rn(warp_sum(l));
    for (int j = lane; j < S; j += 32) {
        float v = 0.0f;
        if (j <= i) v = __fmul_rn(__expf(__bfloat162float(srow[j]) * scale - M), inv);
        prow[j] = from_f32<OutT>(v);
    }
}

// ------------------------------------------------------------------------- unfused kernels
// (1) m = rowmax(scale*s)  (2) d = bf16(scale*s - m), -inf where j > i  (3) e = bf16(exp d)
// (4) l = rowsum(e)        (5) p = bf16(e / l)
// Step 2 folds scale and mask into the subtraction, so no mask tensor exists ([OFCG] [A3] notes
// that a materialised mask would add another full copy of the score tensor).
__global__ void __launch_bounds__(kSmBlock) sm_rowmax_kernel(const __nv_bfloat16* __restrict__ s,
                                                             float* __restrict__ m, int64_t rows,
                                                             int S, float scale) {
    const int lane = threadIdx.x % 32;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + threadIdx.x / 32;
    if (row >= rows) return;
    const int i = static_cast<int>(row % S);
    const __nv_bfloat16* r = s + row * S;
    float mx = -INFINITY;
    for (int j = lane; j < S; j += 32) {
        const float z = __bfloat162float(__ldcs(r + j)) * scale;  // whole row read, as unfused
        if (j <= i) mx = fmaxf(mx, z);
    }
    mx = warp_max(mx);
    if (lane == 0) m[row] = mx;
}

__global__ void __launch_bounds__(kEwBlock) sm_sub_kernel(const __nv_bfloat16* __restrict__ s,
                                                          const float* __restrict__ m,
                                                          __nv_bfloat16* __restrict__ d,
                                                          int64_t n, int S, float scale) {
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t nthr = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t k = tid; k < n; k += nthr) {
        const int64_t row = k / S;
        const int j = static_cast<int>(k - row * S);
        const int i = static_cast<int>(row % S);
        const float z = __bfloat162float(__ldcs(s + k)) * scale;
        d[k] = j <= i ? __float2bfloat16_rn(z - __ldg(m + row)) : __float2bfloat16_rn(-INFINITY);
    }
}

__global__ void __launch_bounds__(kEwBlock) sm_exp_kernel(__nv_bfloat16* __restrict__ d, int64_t n) {
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t nthr = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t k = tid; k < n; k += nthr) d[k] = __float2bfloat16_rn(expf(__bfloat162float(d[k])));
}

__global__ void __launch_bounds__(kSmBlock) sm_rowsum_kernel(const __nv_bfloat16* __restrict__ e,
                                                             float* __restrict__ l, int64_t rows,
                                                             int S) {
    const int lane = threadIdx.x % 32;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + threadIdx.x / 32;
    if (row >= rows) return;
    const __nv_bfloat16* r = e + row * S;
    float acc = 0.0f;
    for (int j = lane; j < S; j += 32) acc += __bfloat162float(__ldcs(r + j));
    acc = warp_sum(acc);
    if (lane == 0) l[row] = acc;
}

__global__ void __launch_bounds__(kEwBlock) sm_div_kernel(__nv_bfloat16* __restrict__ e,
                                                          const float* __restrict__ l, int64_t n,
                                                          int S) {
    const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t nthr = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t k = tid; k < n; k += nthr)
        e[k] = __float2bfloat16_rn(__fdiv_rn(__bfloat162float(e[k]), __ldg(l + k / S)));
}

unsigned ew_grid(int64_t units) {
    const int64_t cap = static_cast<int64_t>(sm_count()) * (2048 / kEwBlock);
    int64_t g = ceil_div(units, kEwBlock);
    if (g > cap) g = cap;
    return static_cast<unsigned>(g < 1 ? 1 : g);
}

template <typename OutT>
int launch_fused(const __nv_bfloat16* s, OutT* p, int64_t rows, int S, float scale, int tile,
                 bool vec, cudaStream_t st) {
    const unsigned grid = static_cast<unsigned>(ceil_div(rows, kWarpsPerBlock));
    if (vec) {
        const int vpl = static_cast<int>(ceil_div(S / 8, 32));
        if (vpl <= 1) softmax_fused_kernel<1, OutT><<<grid, kSmBlock, 0, st>>>(s, p, rows, S, scale, tile);
        else if (vpl <= 2) softmax_fused_kernel<2, OutT><<<grid, kSmBlock, 0, st>>>(s, p, rows, S, scale, tile);
        else if (vpl <= 4) softmax_fused_kernel<4, OutT><<<grid, kSmBlock, 0, st>>>(s, p, rows, S, scale, tile);
        else softmax_fused_kernel<8, OutT><<<grid, kSmBlock, 0, st>>>(s, p, rows, S, scale, tile);
    } else {
        softmax_fused_generic_kernel<OutT><<<grid, kSmBlock, 0, st>>>(s, p, rows, S, scale, tile);
    }
    return check_launch();
}

}  // namespace

int softmax_report_count() { return 4; }
int softmax_report(int i, fuse_kernel_record* out) {
    switch (i) {
        case 0: return describe_kernel((const void*)softmax_fused_kernel<8, __nv_bfloat16>,
                                       "softmax_fused_kernel<VPL=8,bf16> (S 2048)", kSmBlock, 0, out);
        case 1: return describe_kernel((const void*)softmax_fused_generic_kernel<__nv_bfloat16>,
                                       "softmax_fused_generic_kernel<bf16>", kSmBlock, 0, out);
        case 2: return describe_kernel((const void*)sm_sub_kernel,
                                       "sm_sub_kernel (unfused step 2)", kEwBlock, 0, out);
        case 3: return describe_kernel((const void*)sm_rowmax_kernel,
                                       "sm_rowmax_kernel (unfused step 1)", kSmBlock, 0, out);
        default: return FUSE_EINVAL;
    }
}

}  // namespace fc

extern "C" size_t fuse_causal_softmax_workspace_bytes(int64_t batch_heads, int64_t S, int mode) {
    if (batch_heads < 0 || S < 0 || mode != FUSE_UNFUSED) return 0;
    return 2 * static_cast<size_t>(batch_heads) * static_cast<size_t>(S) * sizeof(float);
}

extern "C" int fuse_causal_softmax(const void* s, void* p, int64_t batch_heads, int64_t S,
                                   float scale, int skip_tile, int out_dtype, int mode,
                                   void* workspace, size_t ws_bytes, fuse_stream_t stream) {
    using namespace fc;
    if (batch_heads < 0 || S < 1 || S > 8192 || !isfinite(scale)) return FUSE_EINVAL;
    if (skip_tile < 0 || (skip_tile > 0 && skip_tile % 8 != 0)) return FUSE_EINVAL;
    if (out_dtype != FUSE_BF16 && out_dtype != FUSE_F32) return FUSE_EINVAL;
    if (mode != FUSE_FUSED && mode != FUSE_UNFUSED) return FUSE_EINVAL;
    const int64_t rows = batch_heads * S;
    if (ceil_div(rows, kWarpsPerBlock) > 2147483647LL) return FUSE_EUNSUPPORTED;
    if (rows == 0) return FUSE_OK;
    if (!s || !p) return FUSE_EINVAL;
    if (!is_aligned(s, 2) || !is_aligned(p, out_dtype == FUSE_F32 ? 4 : 2)) return FUSE_EALIGN;
    const char* sb = static_cast<const char*>(s);
    const char* pb = static_cast<const char*>(p);
    const int64_t n = rows * S;
    const int64_t sbytes = n * 2, pbytes = n * (out_dtype == FUSE_F32 ? 4 : 2);
    if (sb < pb + pbytes && pb < sb + sbytes) return FUSE_EINVAL;  // s and p must not overlap
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int Si = static_cast<int>(S);
    const __nv_bfloat16* sp = static_cast<const __nv_bfloat16*>(s);

    if (mode == FUSE_FUSED) {
        const bool vec = (Si % 8 == 0) && Si <= 2048 && is_aligned(s, 16) && is_aligned(p, 16);
        if (out_dtype == FUSE_BF16)
            return launch_fused(sp, static_cast<__nv_bfloat16*>(p), rows, Si, scale, skip_tile, vec, st);
        return launch_fused(sp, static_cast<float*>(p), rows, Si, scale, skip_tile, vec, st);
    }

    // FUSE_UNFUSED: five kernels over whole rows; intermediates are bf16 in p.
    if (skip_tile != 0 || out_dtype != FUSE_BF16) return FUSE_EUNSUPPORTED;
    if (!workspace || ws_bytes < fuse_causal_softmax_workspace_bytes(batch_heads, S, mode))
        return FUSE_EWORKSPACE;
    if (!is_aligned(workspace, 4)) return FUSE_EALIGN;
    float* m = static_cast<float*>(workspace);
    float* l = m + rows;
    __nv_bfloat16* d = static_cast<__nv_bfloat16*>(p);
    const unsigned rgrid = static_cast<unsigned>(ceil_div(rows, kWarpsPerBlock));
    int rc;
    sm_rowmax_kernel<<<rgrid, kSmBlock, 0, st>>>(sp, m, rows, Si, scale);
    if ((rc = check_launch())) return rc;
    sm_sub_kernel<<<ew_grid(n), kEwBlock, 0, st>>>(sp, m, d, n, Si, scale);
    if ((rc = check_launch())) return rc;
    sm_exp_kernel<<<ew_grid(n), kEwBlock, 0, st>>>(d, n);
    if ((rc = check_launch())) return rc;
    sm_rowsum_kernel<<<rgrid, kSmBlock, 0, st>>>(d, l, rows, Si);
    if ((rc = check_launch())) return rc;
    sm_div_kernel<<<ew_grid(n), kEwBlock, 0, st>>>(d, l, n, Si);
    return check_launch();
}

extern "C" int64_t fuse_causal_softmax_bytes(int64_t batch_heads, int64_t S, int skip_tile,
                                             int out_dtype, int mode) {
    if (batch_heads < 0 || S < 1 || skip_tile < 0) return FUSE_EINVAL;
    if (out_dtype != FUSE_BF16 && out_dtype != FUSE_F32) return FUSE_EINVAL;
    const int64_t rows = batch_heads * S, n = rows * S;
    const int64_t ob = out_dtype == FUSE_F32 ? 4 : 2;
    if (mode == FUSE_UNFUSED) {
        // [OFCG] [A3]: max 1, sub 2, exp 2, sum 1, div 2 copies of the bf16 score tensor, plus the
        // fp32 row statistics (m written once, read once; l written once, read once)
        return 8 * n * 2 + 4 * rows * 4;
    }
    if (mode != FUSE_FUSED) return FUSE_EINVAL;
    // every output is written once; row i reads its first ncols(i) scores
    int64_t read_cols = 0;
    for (int64_t i = 0; i < S; ++i) {
        int64_t c = S;
        if (skip_tile > 0) {
            c = (i / skip_tile + 1) * skip_tile;
            if (c > S) c = S;
        }
        read_cols += c;
    }
    return batch_heads * read_cols * 2 + n * ob;
}
