// softmax.cu -- causal attention-score softmax over the last axis of s[BH, S, S] (bf16).
//
// [OFCG] fusion_lab [E]: softmax is max -> subtract -> exp -> sum -> divide over a row; unfused,
// each step reads (and the elementwise ones write) the whole score tensor: 8 copies of it,
// against 2 fused ([A3]).  §3.5: query i sees keys j <= i; skipping whole key blocks of a T x T
// tiling leaves the fraction (n_b + 1)/(2 n_b) of the scores to read.
//
// GB300 design (fused): persistent warps, one row per warp at a time.  The bulk-copy engine (TMA,
// cp.async.bulk) streams each row's kept columns into a per-warp two-stage shared-memory ring, so
// a warp computes row r while its next two rows land, at no register cost; the row is then held
// in registers as 32-byte vectors (16 bf16).  Each lane's vectors are classified against the diagonal:
// fully kept vectors run an unmasked path, the one diagonal vector a masked path, and masked
// vectors do no arithmetic (and, with skip tile T, are not even read).  exp(z - m) is computed as
// 2^(t - m') with t = s * (scale * log2 e) -- one multiply, one subtract, one ex2 per element.
// Max and sum are warp-shuffle reductions: a row never leaves its warp, so no shared memory or
// block barrier is needed.
#include <math.h>

#include "fc_internal.cuh"
#include "fc_ptx.cuh"

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
// 2^x, the MUFU instruction (relative error ~2^-22; ftz: subnormal results flush to +0)
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void ld32(const void* p, uint32_t (&w)[8]) {
    asm volatile("ld.global.cs.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]),
                   "=r"(w[6]), "=r"(w[7])
                 : "l"(p));
}
__device__ __forceinline__ void st32(void* p, const uint32_t (&w)[8]) {
    asm volatile("st.global.cs.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(w[0]),
                 "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}
// 16 bf16 (8 words) -> 16 fp32 (exact)
__device__ __forceinline__ void unpack16(const uint32_t (&w)[8], float* f) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        f[2 * k] = __uint_as_float(w[k] << 16);
        f[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
}

// 16 outputs of one 32-byte input vector
template <typename OutT> struct Out16;
template <> struct Out16<__nv_bfloat16> {  // one 32-byte store
    __device__ __forceinline__ static void store(__nv_bfloat16* row, int v, const float* f) {
        uint32_t w[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * k], f[2 * k + 1]);
            w[k] = *reinterpret_cast<uint32_t*>(&h);
        }
        st32(row + 16 * v, w);
    }
    __device__ __forceinline__ static void zero(__nv_bfloat16* row, int v) {
        const uint32_t w[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        st32(row + 16 * v, w);
    }
};
template <> struct Out16<float> {  // two 32-byte stores
    __device__ __forceinline__ static void store(float* row, int v, const float* f) {
        uint32_t w[8];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int k = 0; k < 8; ++k) w[k] = __float_as_uint(f[8 * h + k]);
            st32(row + 16 * v + 8 * h, w);
        }
    }
    __device__ __forceinline__ static void zero(float* row, int v) {
        const uint32_t w[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        st32(row + 16 * v, w);
        st32(row + 16 * v + 8, w);
    }
};

__device__ __forceinline__ int load_vectors(int i, int S, int skip_tile) {
    const int ncols = skip_tile > 0 ? min(S, (i / skip_tile + 1) * skip_tile) : S;
    return ncols / 16;  // S and skip_tile are multiples of 16 on this path
}

// Fused, persistent, TMA-fed: S % 16 == 0, S <= 512 * VPL, 32-byte aligned rows.
// Warp w owns a ring of kStages row buffers in shared memory; lane 0 asks the bulk-copy engine for
// the kept columns of each row it will process next (one cp.async.bulk per row, completion counted
// on the stage's mbarrier), so the warp computes row r while rows r + nw and r + 2 nw are landing.
constexpr int kStages = 2;

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}
__device__ __forceinline__ void lds32(uint32_t addr, uint32_t (&w)[8]) {
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]) : "r"(addr));
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7]) : "r"(addr + 16));
}

size_t fused_smem_bytes(int S) {
    return static_cast<size_t>(kWarpsPerBlock) * kStages * (static_cast<size_t>(S) * 2 + 8);
}

template <int VPL, typename OutT>
__global__ void __launch_bounds__(kSmBlock, 2) softmax_fused_kernel(
    const __nv_bfloat16* __restrict__ s, OutT* __restrict__ p, int64_t rows, int S, float c,
    int skip_tile, int* flag) {
    pdl_begin();  // before any global-memory access (programmatic dependent launch)
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t rowbytes = static_cast<uint32_t>(S) * 2;
    const uint32_t wbuf = smem_addr(smem) + warp * kStages * rowbytes;
    const uint32_t bars = smem_addr(smem) + kWarpsPerBlock * kStages * rowbytes + warp * kStages * 8;
    const int64_t nw = static_cast<int64_t>(gridDim.x) * kWarpsPerBlock;
    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + warp;
    const int nvec = S / 16;

    if (lane == 0) {
#pragma unroll
        for (int st = 0; st < kStages; ++st) mbar_init(bars + 8 * st, 1);
        fence_mbar_init();
    }
    __syncwarp();
    auto issue = [&](int64_t r, int st) {  // lane 0
        const uint32_t bytes = 32u * load_vectors(static_cast<int>(r % S), S, skip_tile);
        mbar_arrive_expect_tx(bars + 8 * st, bytes);
        bulk_g2s(wbuf + st * rowbytes, s + r * S, bytes, bars + 8 * st);
    };
    uint32_t pending = 0, phase = 0;  // per stage: a copy is in flight / parity of its next phase
#pragma unroll
    for (int st = 0; st < kStages; ++st) {
        const int64_t r = r0 + st * nw;
        if (r < rows) {
            if (lane == 0) issue(r, st);
            pending |= 1u << st;
        }
    }

    int st = 0;
    for (int64_t row = r0; row < rows; row += nw, st = (st + 1) % kStages) {
        if (!mbar_wait_bounded(bars + 8 * st, (phase >> st) & 1u, flag)) {
            // give up: let the copies still in flight land (bounded) before the CTA exits
            for (int k = 0; k < kStages; ++k)
                if ((pending >> k) & 1u) (void)mbar_wait_drain(bars + 8 * k, (phase >> k) & 1u);
            return;
        }
        phase ^= 1u << st;
        pending &= ~(1u << st);

        const int i = static_cast<int>(row % S);
        const int kv = i / 16;  // vectors < kv are fully kept, kv holds the diagonal
        uint32_t cur[VPL][8];
#pragma unroll
        for (int u = 0; u < VPL; ++u) {
            const int v = lane + 32 * u;
            if (v <= kv) lds32(wbuf + st * rowbytes + 32 * v, cur[u]);
        }
        __syncwarp();  // every lane has read the stage: it may be refilled
        if (row + kStages * nw < rows) {
            if (lane == 0) issue(row + kStages * nw, st);
            pending |= 1u << st;
        }

        float m = -INFINITY;
#pragma unroll
        for (int u = 0; u < VPL; ++u) {
            const int v = lane + 32 * u;
            if (v <= kv) {
                float f[16];
                unpack16(cur[u], f);
                if (v < kv) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) m = fmaxf(m, f[e] * c);
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        if (16 * v + e <= i) m = fmaxf(m, f[e] * c);
                }
            }
        }
        m = warp_max(m);

        float ev[VPL][16];
        float sum = 0.0f;
#pragma unroll
        for (int u = 0; u < VPL; ++u) {
            const int v = lane + 32 * u;
            if (v <= kv) {
                unpack16(cur[u], ev[u]);
                if (v < kv) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        ev[u][e] = ex2(ev[u][e] * c - m);
                        sum += ev[u][e];
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        ev[u][e] = (16 * v + e <= i) ? ex2(ev[u][e] * c - m) : 0.0f;
                        sum += ev[u][e];
                    }
                }
            }
        }
        sum = warp_sum(sum);
        const float inv = __frcp_rn(sum);

        OutT* prow = p + row * S;
#pragma unroll
        for (int u = 0; u < VPL; ++u) {
            const int v = lane + 32 * u;
            if (v < nvec) {
                if (v <= kv) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) ev[u][e] = __fmul_rn(ev[u][e], inv);
                    Out16<OutT>::store(prow, v, ev[u]);
                } else {
                    Out16<OutT>::zero(prow, v);
                }
            }
        }
    }
}

// Fused, any S (<= 8192) and any alignment: pass 1 folds the kept scores into a running
// (max, sum) per lane and merges the lanes; pass 2 re-reads them and writes every output.
template <typename OutT>
__global__ void __launch_bounds__(kSmBlock) softmax_fused_generic_kernel(
    const __nv_bfloat16* __restrict__ s, OutT* __restrict__ p, int64_t rows, int S, float c,
    int skip_tile) {
    pdl_begin();  // before any global-memory access (programmatic dependent launch)
    const int lane = threadIdx.x % 32;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + threadIdx.x / 32;
    if (row >= rows) return;
    const int i = static_cast<int>(row % S);
    const int ncols = skip_tile > 0 ? min(S, (i / skip_tile + 1) * skip_tile) : S;
    const __nv_bfloat16* srow = s + row * S;
    OutT* prow = p + row * S;
    float m = -INFINITY, l = 0.0f;
    for (int j = lane; j < ncols && j <= i; j += 32) {
        const float t = __bfloat162float(srow[j]) * c;
        const float mn = fmaxf(m, t);
        l = l * ex2(m - mn) + ex2(t - mn);
        m = mn;
    }
    const float M = warp_max(m);
    l = (m == -INFINITY) ? 0.0f : l * ex2(m - M);
    const float inv = __frcp_rn(warp_sum(l));
    for (int j = lane; j < S; j += 32) {
        float v = 0.0f;
        if (j <= i) v = __fmul_rn(ex2(__bfloat162float(srow[j]) * c - M), inv);
        prow[j] = from_f32<OutT>(v);
    }
}

// ------------------------------------------------------------------------- unfused kernels
// (1) m = rowmax(scale*s)  (2) d = bf16(scale*s - m), -inf where j > i  (3) e = bf16(exp d)
// (4) l = rowsum(e)        (5) p = bf16(e * (1/l))
// Step 2 folds scale and mask into the subtraction, so no mask tensor exists ([OFCG] [A3] notes
// that a materialised mask would add another full copy of the score tensor).  Every step streams
// whole rows with 32-byte vectors when S % 16 == 0 and the tensors are 32-byte aligned.
template <bool VEC>
__global__ void __launch_bounds__(kSmBlock) sm_rowmax_kernel(const __nv_bfloat16* __restrict__ s,
                                                             float* __restrict__ m, int64_t rows,
                                                             int S, float scale) {
    pdl_begin();  // before any global-memory access (programmatic dependent launch)
    const int lane = threadIdx.x % 32;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + threadIdx.x / 32;
    if (row >= rows) return;
    const int i = static_cast<int>(row % S);
    const __nv_bfloat16* r = s + row * S;
    float mx = -INFINITY;
    if (VEC) {
        for (int v = lane; v < S / 16; v += 32) {
            uint32_t w[8];
            ld32(r + 16 * v, w);
            float f[16];
            unpack16(w, f);
#pragma unroll
            for (int e = 0; e < 16; ++e)
                if (16 * v + e <= i) mx = fmaxf(mx, f[e] * scale);
        }
    } else {
        for (int j = lane; j < S; j += 32) {
            const float z = __bfloat162float(r[j]) * scale;
            if (j <= i) mx = fmaxf(mx, z);
        }
    }
    mx = warp_max(mx);
    if (lane == 0) m[row] = mx;
}

template <bool VEC>
__global__ void __launch_bounds__(kEwBlock) sm_sub_kernel(const __nv_bfloat16* __restrict__ s,
                                                          const float* __restrict__ m,
                                                          __nv_bfloat16* __restrict__ d,
                                                          int64_t n, int S, float scale) {
    pdl_begin();  // before any global-memory access (programmatic dependent launch)
    const int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (VEC) {
        const int64_t vpr = S / 16;
        if (g >= n / 16) return;
        const int64_t row = g / vpr;
        const int j0 = static_cast<int>(g - row * vpr) * 16;
        const int i = static_cast<int>(row % S);
        const float mr = __ldg(m + row);
        uint32_t w[8];
        ld32(s + 16 * g, w);
        float f[16];
        unpack16(w, f);
#pragma unroll
        for (int e = 0; e < 16; ++e) f[e] = (j0 + e <= i) ? f[e] * scale - mr : -INFINITY;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * k], f[2 * k + 1]);
            w[k] = *reinterpret_cast<uint32_t*>(&h);
        }
        st32(d + 16 * g, w);
        return;
    }
    if (g >= n) return;
    const int64_t row = g / S;
    const int j = static_cast<int>(g - row * S);
    const int i = static_cast<int>(row % S);
    const float z = __bfloat162float(s[g]) * scale;
    d[g] = __float2bfloat16_rn(j <= i ? z - __ldg(m + row) : -INFINITY);
}

template <bool VEC>
__global__ void __launch_bounds__(kEwBlock) sm_exp_kernel(__nv_bfloat16* __restrict__ d, int64_t n) {
    pdl_begin();  // before any global-memory access (programmatic dependent launch)
    const int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (VEC) {
        if (g >= n / 16) return;
        uint32_t w[8];
        ld32(d + 16 * g, w);
        float f[16];
        unpack16(w, f);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            __nv_bfloat162 h = __floats2bfloat162_rn(expf(f[2 * k]), expf(f[2 * k + 1]));
            w[k] = *reinterpret_cast<uint32_t*>(&h);
        }
        st32(d + 16 * g, w);
        return;
    }
    if (g < n) d[g] = __float2bfloat16_rn(expf(__bfloat162float(d[g])));
}

template <bool VEC>
__global__ void __launch_bounds__(kSmBlock) sm_rowsum_kernel(const __nv_bfloat16* __restrict__ e,
                                                             float* __restrict__ l, int64_t rows,
                                                             int S) {
    pdl_begin();  // before any global-memory access (programmatic dependent launch)
    const int lane = threadIdx.x % 32;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * kWarpsPerBlock + threadIdx.x / 32;
    if (row >= rows) return;
    const __nv_bfloat16* r = e + row * S;
    float acc = 0.0f;
    if (VEC) {
        for (int v = lane; v < S / 16; v += 32) {
            uint32_t w[8];
            ld32(r + 16 * v, w);
            float f[16];
            unpack16(w, f);
#pragma unroll
            for (int k = 0; k < 16; ++k) acc += f[k];
        }
    } else {
        for (int j = lane; j < S; j += 32) acc += __bfloat162float(r[j]);
    }
    acc = warp_sum(acc);
    if (lane == 0) l[row] = acc;
}

template <bool VEC>
__global__ void __launch_bounds__(kEwBlock) sm_div_kernel(__nv_bfloat16* __restrict__ e,
                                                          const float* __restrict__ l, int64_t n,
                                                          int S) {
    pdl_begin();  // before any global-memory access (programmatic dependent launch)
    const int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (VEC) {
        if (g >= n / 16) return;
        const float inv = __frcp_rn(__ldg(l + g / (S / 16)));  // one reciprocal per vector
        uint32_t w[8];
        ld32(e + 16 * g, w);
        float f[16];
        unpack16(w, f);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            __nv_bfloat162 h = __floats2bfloat162_rn(__fmul_rn(f[2 * k], inv), __fmul_rn(f[2 * k + 1], inv));
            w[k] = *reinterpret_cast<uint32_t*>(&h);
        }
        st32(e + 16 * g, w);
        return;
    }
    if (g < n) e[g] = __float2bfloat16_rn(__fmul_rn(__bfloat162float(e[g]), __frcp_rn(__ldg(l + g / S))));
}

unsigned grid_for(int64_t units, int block) {
    const int64_t g = ceil_div(units, block);
    return static_cast<unsigned>(g < 1 ? 1 : g);
}

template <int VPL, typename OutT>
int launch_vec(const __nv_bfloat16* s, OutT* p, int64_t rows, int S, float c, int tile,
               cudaStream_t st) {
    const size_t smem = fused_smem_bytes(S);
    const int attr_rc = opt_in_smem((const void*)softmax_fused_kernel<VPL, OutT>,
                                    static_cast<int>(fused_smem_bytes(512 * VPL)));
    if (attr_rc != FUSE_OK) return attr_rc;
    int* flag = watchdog_flag();
    if (!flag) return FUSE_ECUDA;
    const int occ = blocks_per_sm(softmax_fused_kernel<VPL, OutT>, kSmBlock, smem);
    int64_t grid = ceil_div(rows, kWarpsPerBlock);
    const int64_t cap = static_cast<int64_t>(sm_count()) * occ;
    if (grid > cap) grid = cap;
    return launch_pdl(softmax_fused_kernel<VPL, OutT>, dim3(static_cast<unsigned>(grid)), dim3(kSmBlock), smem, st, 1, s, p, rows, S, c, tile, flag);
}

template <typename OutT>
int launch_fused(const __nv_bfloat16* s, OutT* p, int64_t rows, int S, float c, int tile, bool vec,
                 cudaStream_t st) {
    if (vec) {
        const int vpl = static_cast<int>(ceil_div(S / 16, 32));
        if (vpl <= 1) return launch_vec<1, OutT>(s, p, rows, S, c, tile, st);
        if (vpl <= 2) return launch_vec<2, OutT>(s, p, rows, S, c, tile, st);
        return launch_vec<4, OutT>(s, p, rows, S, c, tile, st);
    }
    return launch_pdl(softmax_fused_generic_kernel<OutT>, dim3(grid_for(rows, kWarpsPerBlock)), dim3(kSmBlock), 0, st, 1, s, p, rows, S, c, tile);
}

template <bool VEC>
int launch_unfused(const __nv_bfloat16* s, __nv_bfloat16* d, float* m, float* l, int64_t rows,
                   int S, float scale, cudaStream_t st) {
    const int64_t n = rows * S;
    const int64_t units = VEC ? n / 16 : n;
    const unsigned rgrid = grid_for(rows, kWarpsPerBlock);
    int rc;
    if ((rc = launch_pdl(sm_rowmax_kernel<VEC>, dim3(rgrid), dim3(kSmBlock), 0, st, 1, s, m, rows, S, scale))) return rc;
    if ((rc = launch_pdl(sm_sub_kernel<VEC>, dim3(grid_for(units, kEwBlock)), dim3(kEwBlock), 0, st, 1, s, m, d, n, S, scale))) return rc;
    if ((rc = launch_pdl(sm_exp_kernel<VEC>, dim3(grid_for(units, kEwBlock)), dim3(kEwBlock), 0, st, 1, d, n))) return rc;
    if ((rc = launch_pdl(sm_rowsum_kernel<VEC>, dim3(rgrid), dim3(kSmBlock), 0, st, 1, d, l, rows, S))) return rc;
    return launch_pdl(sm_div_kernel<VEC>, dim3(grid_for(units, kEwBlock)), dim3(kEwBlock), 0, st, 1, d, l, n, S);
}

}  // namespace

int softmax_report_count() { return 4; }
int softmax_report(int i, fuse_kernel_record* out) {
    switch (i) {
        case 0: return describe_kernel((const void*)softmax_fused_kernel<4, __nv_bfloat16>,
                                       "softmax_fused_kernel<VPL=4,bf16> (S 2048)", kSmBlock,
                                       static_cast<int>(fused_smem_bytes(2048)), out);
        case 1: return describe_kernel((const void*)softmax_fused_generic_kernel<__nv_bfloat16>,
                                       "softmax_fused_generic_kernel<bf16>", kSmBlock, 0, out);
        case 2: return describe_kernel((const void*)sm_sub_kernel<true>,
                                       "sm_sub_kernel (unfused step 2)", kEwBlock, 0, out);
        case 3: return describe_kernel((const void*)sm_rowmax_kernel<true>,
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
    if (skip_tile < 0 || (skip_tile > 0 && skip_tile % 16 != 0)) return FUSE_EINVAL;
    if (out_dtype != FUSE_BF16 && out_dtype != FUSE_F32) return FUSE_EINVAL;
    if (mode != FUSE_FUSED && mode != FUSE_UNFUSED) return FUSE_EINVAL;
    const int64_t rows = batch_heads * S;
    if (ceil_div(rows * S, kEwBlock) > 2147483647LL) return FUSE_EUNSUPPORTED;
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
    const bool vec = (Si % 16 == 0) && is_aligned(s, 32) && is_aligned(p, 32);

    if (mode == FUSE_FUSED) {
        const float c = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
        const bool reg = vec && Si <= 2048;
        if (out_dtype == FUSE_BF16)
            return launch_fused(sp, static_cast<__nv_bfloat16*>(p), rows, Si, c, skip_tile, reg, st);
        return launch_fused(sp, static_cast<float*>(p), rows, Si, c, skip_tile, reg, st);
    }

    // FUSE_UNFUSED: five kernels over whole rows; intermediates are bf16 in p.
    if (skip_tile != 0 || out_dtype != FUSE_BF16) return FUSE_EUNSUPPORTED;
    if (!workspace || ws_bytes < fuse_causal_softmax_workspace_bytes(batch_heads, S, mode))
        return FUSE_EWORKSPACE;
    if (!is_aligned(workspace, 4)) return FUSE_EALIGN;
    float* m = static_cast<float*>(workspace);
    float* l = m + rows;
    __nv_bfloat16* d = static_cast<__nv_bfloat16*>(p);
    if (vec) return launch_unfused<true>(sp, d, m, l, rows, Si, scale, st);
    return launch_unfused<false>(sp, d, m, l, rows, Si, scale, st);
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
