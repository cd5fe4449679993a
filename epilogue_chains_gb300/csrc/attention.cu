// attention.cu -- causal attention that never materialises the S x S score matrix.
//
// "AIGC fundamentals | operator fusion and CUDA Graph" §6.3 and its reading list: the score tensor
// of the causal softmax row ([B, H, S, S] = 1 GiB at B=8, H=16, S=2048) disappears altogether when
// the softmax is fused into the attention itself and normalised online (FlashAttention,
// arXiv:2205.14135), which also skips the masked half of the scores.  Per (batch, head) slice:
//     O = softmax(scale Q K^T, keys j <= query i) V,   Q, K, V, O bf16 [S, D].
//
// GB300 design: one CTA per 128-row query tile, heaviest (most key blocks) tiles first, 192
// threads in three roles.
//  * warp 0 (one lane) loads Q once and then, per 128-key block j, K_j and V_j with TMA
//    (128-byte swizzle; single buffers: K_j+1 streams in as soon as S_j is computed, V_j+1 as
//    soon as PV_j is);
//  * warp 1 owns TMEM (512 columns: two 128-column score buffers and the D-column output
//    accumulator) and issues the tcgen05 MMAs: S_j = Q K_j^T (M 128, N 128, bf16, K-major both)
//    into score buffer j % 2, and O += P_j V_j (M 128, N D, P K-major from shared memory, V
//    MN-major) -- S_j+1 is issued before PV_j, so the next scores are computed while the softmax
//    warps work on the current ones;
//  * warps 2-5 (one TMEM lane quadrant each, one query row per thread) read the scores with
//    tcgen05.ld, mask the diagonal block, keep the running row maximum m and sum l in base-2
//    units, write P = 2^(s c - m) as bf16 into shared memory in the MMA's swizzled layout, and
//    rescale the O accumulator in TMEM only when the maximum has grown by more than 2^8 since it
//    was last applied (P stays <= 256, exact in the final O / l).  After the last block they
//    divide O by l and store it.
// All waits are bounded (watchdog); a CTA whose wait runs out drains its MMAs and copies and
// frees its TMEM before it returns.
#include <math.h>

#include <mutex>

#include "fc_internal.cuh"
#include "fc_ptx.cuh"
#include "fc_tc.cuh"

namespace fc {
namespace {

constexpr int kAttnQ = 128;          // query rows per CTA
constexpr int kAttnK = 128;          // keys per block
constexpr int kAttnThreads = 192;    // producer, MMA, 4 softmax warps
constexpr float kRescaleLog2 = 8.0f; // rescale O only when the row maximum grew by more than this

template <int D>
struct AttnLayout {
    static constexpr int ATOMS = D / 64;                   // 128-byte swizzle atoms along D
    static constexpr uint32_t REGION = 128 * 128;          // 128 rows x 128 B
    static constexpr uint32_t Q_BYTES = kAttnQ * D * 2;
    static constexpr uint32_t K_BYTES = kAttnK * D * 2;
    static constexpr uint32_t V_BYTES = kAttnK * D * 2;
    static constexpr uint32_t P_BYTES = kAttnQ * kAttnK * 2;
    static constexpr uint32_t OFF_Q = 0;
    static constexpr uint32_t OFF_K = OFF_Q + Q_BYTES;
    static constexpr uint32_t OFF_V = OFF_K + K_BYTES;
    static constexpr uint32_t OFF_P = OFF_V + V_BYTES;
    static constexpr uint32_t OFF_BAR = OFF_P + P_BYTES;
    static constexpr int N_BARS = 12;
    static constexpr uint32_t OFF_HOLD = OFF_BAR + N_BARS * 8;
    static constexpr uint32_t SMEM = OFF_HOLD + 16 + 1024;  // + alignment slack
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t O_COL = 2 * kAttnK;
    static_assert(O_COL + D <= TMEM_COLS, "score buffers and O must fit in TMEM");
};

struct AttnArgs {
    int BH, S;
    float c;               // scale * log2(e): scores in base-2 units
    __nv_bfloat16* O;
    int* flag;
};

__device__ __forceinline__ float ex2f(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

template <int D>
__global__ void __launch_bounds__(kAttnThreads, 1) attn_fwd_kernel(
    const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
    const __grid_constant__ CUtensorMap mV, const __grid_constant__ AttnArgs a) {
    using L = AttnLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (smem_addr(smem_raw) + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - smem_addr(smem_raw));
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t bar0 = base + L::OFF_BAR;
    const uint32_t q_full = bar0, k_full = bar0 + 8, k_empty = bar0 + 16, v_full = bar0 + 24,
                   v_empty = bar0 + 32, p_full = bar0 + 72, o_done = bar0 + 80, drain = bar0 + 88;
    auto s_full = [&](int b) { return bar0 + 40u + 8u * b; };
    auto s_free = [&](int b) { return bar0 + 56u + 8u * b; };
    int* flag = a.flag;

    const int ntile = a.S / kAttnQ;
    const int t = blockIdx.x;
    const int qt = ntile - 1 - t / a.BH;   // heaviest query tiles first
    const int bh = t % a.BH;
    const int nb = qt + 1;                 // key blocks 0..qt (causal)
    const int row0 = bh * a.S + qt * kAttnQ;
    const int krow0 = bh * a.S;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(k_full, 1);
        mbar_init(k_empty, 1);
        mbar_init(v_full, 1);
        mbar_init(v_empty, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(s_full(b), 1);
            mbar_init(s_free(b), 4);
        }
        mbar_init(p_full, 4);
        mbar_init(o_done, 1);
        mbar_init(drain, 1);
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(base + L::OFF_HOLD, L::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gbase + L::OFF_HOLD);

    if (warp == 0) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0) {
            prefetch_map(&mQ);
            prefetch_map(&mK);
            prefetch_map(&mV);
            mbar_arrive_expect_tx(q_full, L::Q_BYTES);
            for (int c = 0; c < L::ATOMS; ++c)
                tma_load_2d(base + L::OFF_Q + c * L::REGION, &mQ, 64 * c, row0, q_full);
            int k_loads = 0, v_loads = 0;
            bool ok = true;
            for (int j = 0; j < nb && ok; ++j) {
                if (j > 0 && !mbar_wait_bounded(k_empty, (j - 1) & 1, flag)) { ok = false; break; }
                mbar_arrive_expect_tx(k_full, L::K_BYTES);
                for (int c = 0; c < L::ATOMS; ++c)
                    tma_load_2d(base + L::OFF_K + c * L::REGION, &mK, 64 * c, krow0 + j * kAttnK, k_full);
                ++k_loads;
                if (j > 0 && !mbar_wait_bounded(v_empty, (j - 1) & 1, flag)) { ok = false; break; }
                mbar_arrive_expect_tx(v_full, L::V_BYTES);
                for (int c = 0; c < L::ATOMS; ++c)
                    tma_load_2d(base + L::OFF_V + c * L::REGION, &mV, 64 * c, krow0 + j * kAttnK, v_full);
                ++v_loads;
            }
            if (!ok) {  // let the copies in flight land before the CTA's shared memory goes away
                (void)mbar_wait_drain(q_full, 0);
                if (k_loads) (void)mbar_wait_drain(k_full, (k_loads - 1) & 1);
                if (v_loads) (void)mbar_wait_drain(v_full, (v_loads - 1) & 1);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idS = idesc_f16(kAttnQ, kAttnK, false, false, true);
            constexpr uint32_t idO = idesc_f16(kAttnQ, D, false, true, true);
            bool issued = false;
            auto issue_s = [&](int j) -> bool {
                const int b = j & 1;
                if (!mbar_wait_bounded(k_full, j & 1, flag)) return false;
                if (j >= 2 && !mbar_wait_bounded(s_free(b), ((j - 2) >> 1) & 1, flag)) return false;
                tc_fence_after();
#pragma unroll
                for (int s = 0; s < D / 16; ++s) {
                    const uint32_t off = (s / 4) * L::REGION + (s % 4) * 32;
                    tc_mma(tmem + b * kAttnK, smem_desc_sw128(base + L::OFF_Q + off, 16, 1024),
                           smem_desc_sw128(base + L::OFF_K + off, 16, 1024), idS, s > 0 ? 1u : 0u);
                }
                tc_commit(s_full(b));
                tc_commit(k_empty);
                issued = true;
                return true;
            };
            auto issue_pv = [&](int j) -> bool {
                if (!mbar_wait_bounded(p_full, j & 1, flag)) return false;
                if (!mbar_wait_bounded(v_full, j & 1, flag)) return false;
                tc_fence_after();
#pragma unroll
                for (int s = 0; s < kAttnK / 16; ++s) {
                    const uint32_t poff = (s / 4) * L::REGION + (s % 4) * 32;
                    tc_mma(tmem + L::O_COL, smem_desc_sw128(base + L::OFF_P + poff, 16, 1024),
                           smem_desc_sw128(base + L::OFF_V + s * 2048, L::REGION, 1024), idO,
                           (j > 0 || s > 0) ? 1u : 0u);
                }
                tc_commit(o_done);
                tc_commit(v_empty);
                issued = true;
                return true;
            };
            bool ok = mbar_wait_bounded(q_full, 0, flag);
            if (ok) ok = issue_s(0);
            for (int j = 0; ok && j < nb; ++j) {
                if (j + 1 < nb && !issue_s(j + 1)) { ok = false; break; }
                ok = issue_pv(j);
            }
            if (!ok && issued) {  // MMAs in flight must finish before TMEM is freed
                tc_commit(drain);
                (void)mbar_wait_drain(drain, 0);
            }
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- softmax warps
        const int qd = warp % 4;
        const int r = 32 * qd + lane;                       // query row within the tile
        const uint32_t lanes = static_cast<uint32_t>(32 * qd) << 16;
        float m_used = -INFINITY, l = 0.0f;
        bool ok = true;
        // tcgen05.ld/st are warp-collective: every wait outcome is made warp-uniform before them
        for (int j = 0; j < nb; ++j) {
            const int b = j & 1;
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(s_full(b), (j >> 1) & 1, flag))) {
                ok = false;
                break;
            }
            tc_fence_after();
            float s[kAttnK];
#pragma unroll
            for (int k = 0; k < kAttnK / 32; ++k) tmem_ld32(tmem + lanes + b * kAttnK + 32 * k, s + 32 * k);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(s_free(b));   // the score buffer may be overwritten now

            const bool diag = (j == nb - 1);
            float mx = -INFINITY;
#pragma unroll
            for (int k = 0; k < kAttnK; ++k) {
                const float x = (diag && k > r) ? -INFINITY : s[k] * a.c;
                s[k] = x;
                mx = fmaxf(mx, x);
            }
            float alpha = 1.0f;
            bool rescale = false;
            if (mx > m_used + kRescaleLog2) {   // always true for the first block (m_used = -inf)
                if (j > 0) {
                    alpha = ex2f(m_used - mx);
                    rescale = true;
                }
                m_used = mx;
            }
            float sum = 0.0f;
            uint32_t pk[kAttnK / 2];
#pragma unroll
            for (int k = 0; k < kAttnK; k += 2) {
                const float p0 = ex2f(s[k] - m_used), p1 = ex2f(s[k + 1] - m_used);
                sum += p0 + p1;
                pk[k / 2] = pack_bf16x2(p0, p1);
            }
            l = l * alpha + sum;

            // PV_{j-1} must be complete: the P buffer is free and O holds blocks 0..j-1
            if (j > 0) {
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(o_done, (j - 1) & 1, flag))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
            }
            if (__any_sync(0xffffffffu, rescale)) {   // rows without a new maximum scale by 1
#pragma unroll 1
                for (int k = 0; k < D / 32; ++k) {
                    float o[32];
                    tmem_ld32(tmem + lanes + L::O_COL + 32 * k, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] *= alpha;
                    tmem_st32(tmem + lanes + L::O_COL + 32 * k, o);
                }
                tmem_st_wait();
            }
            // P row r, keys 0..127: 16 chunks of 8 keys; chunk ch lies in 64-key atom ch / 8 at
            // 16-byte slot (ch % 8) ^ (r % 8) of the row (128-byte swizzle)
            uint8_t* prow = gbase + L::OFF_P + r * 128;
#pragma unroll
            for (int ch = 0; ch < kAttnK / 8; ++ch) {
                uint4* dst = reinterpret_cast<uint4*>(prow + (ch >> 3) * L::REGION + (((ch & 7) ^ (r & 7)) << 4));
                *dst = make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
            }
            fence_async_smem();   // the generic-proxy P writes become visible to the tensor core
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full);
        }
        if (ok && __all_sync(0xffffffffu, mbar_wait_bounded(o_done, (nb - 1) & 1, flag))) {
            tc_fence_after();
            const float inv = 1.0f / l;
            __nv_bfloat16* orow = a.O + static_cast<int64_t>(row0 + r) * D;
#pragma unroll 1
            for (int k = 0; k < D / 32; ++k) {
                float o[32];
                tmem_ld32(tmem + lanes + L::O_COL + 32 * k, o);
                tmem_ld_wait();
                uint4* dst = reinterpret_cast<uint4*>(orow + 32 * k);
#pragma unroll
                for (int v = 0; v < 4; ++v)
                    dst[v] = make_uint4(pack_bf16x2(o[8 * v] * inv, o[8 * v + 1] * inv),
                                        pack_bf16x2(o[8 * v + 2] * inv, o[8 * v + 3] * inv),
                                        pack_bf16x2(o[8 * v + 4] * inv, o[8 * v + 5] * inv),
                                        pack_bf16x2(o[8 * v + 6] * inv, o[8 * v + 7] * inv));
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, L::TMEM_COLS);
    }
}

// Dynamic shared memory of a launch: the layout's, but at least 120 KB so that one CTA runs per SM
// for every D (each CTA allocates all 512 TMEM columns).
template <int D>
constexpr uint32_t attn_launch_smem() {
    return AttnLayout<D>::SMEM > 120u * 1024u ? AttnLayout<D>::SMEM : 120u * 1024u;
}

// Opt the kernel into its shared-memory size on the current device (once per device).
template <int D>
int attn_attr() {
    static std::mutex mu;
    static bool done[64] = {false};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return record_cuda_error(e);
    if (dev < 0 || dev >= 64) return FUSE_EUNSUPPORTED;
    std::lock_guard<std::mutex> lock(mu);
    if (!done[dev]) {
        e = cudaFuncSetAttribute(attn_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(attn_launch_smem<D>()));
        if (e != cudaSuccess) return record_cuda_error(e);
        done[dev] = true;
    }
    return FUSE_OK;
}

template <int D>
int launch_attn(const void* q, const void* k, const void* v, void* o, int bh, int S, float scale,
                cudaStream_t st) {
    const int rc = attn_attr<D>();
    if (rc != FUSE_OK) return rc;
    const int64_t rows = static_cast<int64_t>(bh) * S;
    CUtensorMap mQ, mK, mV;
    if (!make_map(&mQ, q, rows, D, 64, kAttnQ, true) || !make_map(&mK, k, rows, D, 64, kAttnK, true) ||
        !make_map(&mV, v, rows, D, 64, kAttnK, true))
        return FUSE_ECUDA;
    int* flag = watchdog_flag();
    if (!flag) return FUSE_ECUDA;
    AttnArgs args{bh, S, scale * 1.4426950408889634f, static_cast<__nv_bfloat16*>(o), flag};
    const unsigned grid = static_cast<unsigned>(rows / kAttnQ);
    attn_fwd_kernel<D><<<grid, kAttnThreads, attn_launch_smem<D>(), st>>>(mQ, mK, mV, args);
    return check_launch();
}

bool overlap(const void* a, const void* b, int64_t bytes) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + static_cast<uintptr_t>(bytes) && y < x + static_cast<uintptr_t>(bytes);
}

}  // namespace

int attn_report_count() { return 1; }
int attn_report(int i, fuse_kernel_record* out) {
    if (i != 0) return FUSE_EINVAL;
    const int rc = attn_attr<256>();
    if (rc != FUSE_OK) return rc;
    return describe_kernel((const void*)attn_fwd_kernel<256>,
                           "attn_fwd_kernel<D=256> (tcgen05, no score matrix)", kAttnThreads,
                           static_cast<int>(attn_launch_smem<256>()), out);
}

}  // namespace fc

extern "C" int fuse_attention(const void* q, const void* k, const void* v, void* o, int64_t bh,
                              int64_t S, int64_t D, float scale, fuse_stream_t stream) {
    using namespace fc;
    if (bh < 0 || S < 0 || !(scale > 0.0f) || !isfinite(scale)) return FUSE_EINVAL;
    if (D != 64 && D != 128 && D != 256) return FUSE_EUNSUPPORTED;
    if (bh == 0 || S == 0) return FUSE_OK;
    if (!q || !k || !v || !o) return FUSE_EINVAL;
    if (S % kAttnQ != 0 || bh * S > 2147483647LL) return FUSE_EUNSUPPORTED;
    if (!is_aligned(q, 16) || !is_aligned(k, 16) || !is_aligned(v, 16) || !is_aligned(o, 16))
        return FUSE_EALIGN;
    const int64_t bytes = bh * S * D * 2;
    if (overlap(o, q, bytes) || overlap(o, k, bytes) || overlap(o, v, bytes)) return FUSE_EINVAL;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int B = static_cast<int>(bh), SS = static_cast<int>(S);
    if (D == 64) return launch_attn<64>(q, k, v, o, B, SS, scale, st);
    if (D == 128) return launch_attn<128>(q, k, v, o, B, SS, scale, st);
    return launch_attn<256>(q, k, v, o, B, SS, scale, st);
}

extern "C" int64_t fuse_attention_bytes(int64_t bh, int64_t S, int64_t D) {
    if (bh < 0 || S < 0 || D < 1) return FUSE_EINVAL;
    return 4 * bh * S * D * 2;   // read Q, K, V once, write O once (bf16)
}

extern "C" int64_t fuse_attention_flops(int64_t bh, int64_t S, int64_t D) {
    if (bh < 0 || S < 0 || D < 1) return FUSE_EINVAL;
    // Q K^T and P V over the visible (i, j <= i) pairs: 2 * 2 * D flops per pair
    return 4 * D * (S * (S + 1) / 2) * bh;
}
