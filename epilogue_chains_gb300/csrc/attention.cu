// attention.cu -- causal attention that never materialises the S x S score matrix.
//
// "AIGC fundamentals | operator fusion and CUDA Graph" §6.3 and its reading list: the score tensor
// of the causal softmax row ([B, H, S, S] = 1 GiB at B=8, H=16, S=2048) disappears altogether when
// the softmax is fused into the attention itself and normalised online (FlashAttention,
// arXiv:2205.14135), which also skips the masked half of the scores.  Per (batch, head) slice:
//     O = softmax(scale Q K^T, keys j <= query i) V,   Q, K, V, O bf16 [S, D].
//
// GB300 design: one CTA per 128-row query tile, heaviest (most key blocks) tiles first; two CTAs
// with adjacent tiles of one slice form a cluster and multicast the key/value blocks they share.
// Keys go in blocks of 128 (the MMA re-reads the whole Q tile from shared memory for every block,
// so longer blocks cost less shared-memory bandwidth per flop), which at a head size of 256 leaves
// room for one K, one V and one P buffer (Q 64 KB + K 64 KB + V 64 KB + P 32 KB) and two score
// buffers in TMEM (2 x 128 score columns + 256 O columns).  320 threads in three roles:
//  * warp 0: lane 0 loads Q once and the K blocks, lane 1 the V blocks (TMA, 128-byte swizzle),
//    each as soon as its buffer is free (K_j+1 once S_j is computed, V_j+1 once PV_j is);
//  * warp 1 owns TMEM and issues the tcgen05 MMAs: S_j = Q K_j^T (M 128, N 128, bf16, K-major
//    both) into score buffer j % 2, and O += P_j V_j (M 128, N D, P K-major, V MN-major), in the
//    order S_0, S_1, PV_0, S_2, PV_1, ... so the next scores are computed while the softmax warps
//    work on the current ones;
//  * warps 2-9 (two per TMEM lane quadrant, one query row per thread, each warp half of a
//    block's keys and half of O's columns) read the scores with tcgen05.ld, mask the diagonal
//    blocks, keep the running row maximum m and sum l in base-2 units, write P = 2^(s c - m) as
//    bf16 into shared memory in the MMA's swizzled layout, and rescale their half of the O
//    accumulator in TMEM only when the maximum has grown by more than 2^8 since it was last
//    applied (P stays <= 256, exact in the final O / l).  After the last block they divide O by
//    l and store it.
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
constexpr int kKVStages = 1;         // K and V buffers (each a ring of this many blocks)
constexpr int kPBuf = 1;             // P buffers in shared memory
constexpr int kAttnSoftmaxWarps = 8; // two per TMEM lane quadrant, each exponentiating 32 keys
constexpr int kAttnThreads = 32 * (2 + kAttnSoftmaxWarps);
constexpr float kRescaleLog2 = 8.0f; // rescale O only when the row maximum grew by more than this
constexpr int kSBuf = 2;             // score buffers in TMEM: S_j+kSBuf-1 is computed before PV_j

// Shared memory: Q (128 x D), two K and two V stages (64 keys x D each) and two P buffers
// (128 x 64 bf16), all in 128-byte-swizzled 64-column atoms.  TMEM: two 64-column score buffers
// and the D-column O accumulator.
template <int D>
struct AttnLayout {
    static constexpr int ATOMS = D / 64;                   // 128-byte swizzle atoms along D
    static constexpr uint32_t Q_REGION = kAttnQ * 128;     // one atom of Q: 128 rows x 128 B
    static constexpr uint32_t KV_REGION = kAttnK * 128;    // one atom of a K or V block
    static constexpr uint32_t Q_BYTES = kAttnQ * D * 2;
    static constexpr uint32_t KV_BYTES = kAttnK * D * 2;
    static constexpr uint32_t P_BYTES = kAttnQ * kAttnK * 2;
    static constexpr uint32_t OFF_Q = 0;
    static constexpr uint32_t OFF_K = OFF_Q + Q_BYTES;                 // + stage * KV_BYTES
    static constexpr uint32_t OFF_V = OFF_K + kKVStages * KV_BYTES;    // + stage * KV_BYTES
    static constexpr uint32_t OFF_P = OFF_V + kKVStages * KV_BYTES;    // + buffer * P_BYTES
    static constexpr uint32_t OFF_BAR = OFF_P + kPBuf * P_BYTES;
    static constexpr int N_BARS = 3 + 4 * kKVStages + 2 * kPBuf + 2 * kSBuf;
    static constexpr uint32_t OFF_HOLD = OFF_BAR + N_BARS * 8;
    static constexpr uint32_t SMEM = OFF_HOLD + 16 + 1024;       // + alignment slack
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t O_COL = 256;
    static_assert(kSBuf * kAttnK <= O_COL && O_COL + D <= TMEM_COLS, "TMEM budget");
    static_assert(SMEM <= 232448, "shared-memory budget");
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

template <int D, int CL>
__global__ void __launch_bounds__(kAttnThreads, 1) attn_fwd_kernel(
    const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
    const __grid_constant__ CUtensorMap mV, const __grid_constant__ AttnArgs a) {
    using L = AttnLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (smem_addr(smem_raw) + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - smem_addr(smem_raw));
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    // barriers: q_full, drain, l_ready, then per K/V stage k_full, k_empty, v_full, v_empty, per
    // P buffer p_full, o_done, per score buffer s_full, s_free.  A ring of n buffers used by
    // blocks j = 0, 1, ...: buffer j % n, completion number j / n, parity (j / n) & 1.
    const uint32_t bar0 = base + L::OFF_BAR;
    const uint32_t q_full = bar0, drain = bar0 + 8, l_ready = bar0 + 16;
    constexpr int KV = kKVStages, PB = kPBuf, SB = kSBuf;
    auto k_full = [&](int i) { return bar0 + 8u * (3 + i); };
    auto k_empty = [&](int i) { return bar0 + 8u * (3 + KV + i); };
    auto v_full = [&](int i) { return bar0 + 8u * (3 + 2 * KV + i); };
    auto v_empty = [&](int i) { return bar0 + 8u * (3 + 3 * KV + i); };
    auto p_full = [&](int i) { return bar0 + 8u * (3 + 4 * KV + i); };
    auto o_done = [&](int i) { return bar0 + 8u * (3 + 4 * KV + PB + i); };
    auto s_full = [&](int i) { return bar0 + 8u * (3 + 4 * KV + 2 * PB + i); };
    auto s_free = [&](int i) { return bar0 + 8u * (3 + 4 * KV + 2 * PB + SB + i); };
    int* flag = a.flag;

    // CL = 2: the two CTAs of a cluster take adjacent query tiles 2u, 2u + 1 of one slice and
    // share the key blocks both need: each loads half of every shared K and V block and
    // multicasts it to both, halving the L2 traffic of the key/value stream.  Heaviest tiles first.
    const int ntile = a.S / kAttnQ;
    const uint32_t rank = CL > 1 ? cluster_rank() : 0u;
    const int group = blockIdx.x / CL;
    const int u = ntile / CL - 1 - group / a.BH;
    const int bh = group % a.BH;
    const int qt = CL * u + static_cast<int>(rank);
    constexpr int kBlocksPerTile = kAttnQ / kAttnK;
    const int nb = (qt + 1) * kBlocksPerTile;             // key blocks up to the diagonal
    const int nshared = (CL * u + 1) * kBlocksPerTile;    // needed by every CTA of the cluster
    const int row0 = bh * a.S + qt * kAttnQ;
    const int krow0 = bh * a.S;
    constexpr uint16_t kAll = static_cast<uint16_t>((1u << CL) - 1u);
    constexpr int kAtomsPerCta = L::ATOMS / CL;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int i = 0; i < KV; ++i) {
            mbar_init(k_full(i), 1);
            mbar_init(k_empty(i), CL);   // a shared block is free once every CTA is done with it
            mbar_init(v_full(i), 1);
            mbar_init(v_empty(i), CL);
        }
        for (int i = 0; i < PB; ++i) {
            mbar_init(p_full(i), kAttnSoftmaxWarps);
            mbar_init(o_done(i), 1);
        }
        for (int i = 0; i < SB; ++i) {
            mbar_init(s_full(i), 1);
            mbar_init(s_free(i), kAttnSoftmaxWarps);
        }
        mbar_init(drain, 1);
        mbar_init(l_ready, kAttnSoftmaxWarps);
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(base + L::OFF_HOLD, L::TMEM_COLS);
    tc_fence_before();
    if (CL > 1) cluster_sync();   // the peer's multicast copies and commits find initialised barriers
    else __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gbase + L::OFF_HOLD);

    if (warp == 0) {
        // ---------------------------------------------------------------- TMA producers
        // lane 0 loads Q and the K blocks, lane 1 the V blocks, each into a two-stage ring: block
        // j + 2 streams in while blocks j and j + 1 are being used
        if (lane < 2) {
            const bool is_k = lane == 0;
            const CUtensorMap* map = is_k ? &mK : &mV;
            const uint32_t off = is_k ? L::OFF_K : L::OFF_V;
            prefetch_map(map);
            if (is_k) {
                prefetch_map(&mQ);
                mbar_arrive_expect_tx(q_full, L::Q_BYTES);
                for (int c = 0; c < L::ATOMS; ++c)
                    tma_load_2d(base + L::OFF_Q + c * L::Q_REGION, &mQ, 64 * c, row0, q_full);
            }
            int loads = 0;
            for (int j = 0; j < nb; ++j) {
                const int st = j % KV;
                const uint32_t full = is_k ? k_full(st) : v_full(st);
                const uint32_t empty = is_k ? k_empty(st) : v_empty(st);
                if (j >= KV && !mbar_wait_bounded(empty, ((j - KV) / KV) & 1, flag)) break;
                mbar_arrive_expect_tx(full, L::KV_BYTES);
                const int y = krow0 + j * kAttnK;
                const uint32_t dst = base + off + st * L::KV_BYTES;
                if (CL > 1 && j < nshared) {
                    for (int c = kAtomsPerCta * rank; c < kAtomsPerCta * (rank + 1); ++c)
                        tma_load_2d_mc(dst + c * L::KV_REGION, map, 64 * c, y, full, kAll);
                } else {
                    for (int c = 0; c < L::ATOMS; ++c) tma_load_2d(dst + c * L::KV_REGION, map, 64 * c, y, full);
                }
                ++loads;
            }
            if (loads < nb) {  // let the copies in flight land before the shared memory goes away
                if (is_k) (void)mbar_wait_drain(q_full, 0);
                for (int j = loads - KV < 0 ? 0 : loads - KV; j < loads; ++j)
                    (void)mbar_wait_drain(is_k ? k_full(j % KV) : v_full(j % KV), (j / KV) & 1);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        // order: S_0, S_1, S_2, PV_0, S_3, PV_1, ...: the scores of the next two blocks are
        // computed while the softmax warps work on the current ones
        if (lane == 0) {
            constexpr uint32_t idS = idesc_f16(kAttnQ, kAttnK, false, false, true);
            constexpr uint32_t idO = idesc_f16(kAttnQ, D, false, true, true);
            bool issued = false;
            auto issue_s = [&](int j) -> bool {
                const int st = j % KV, sb = j % SB;
                if (!mbar_wait_bounded(k_full(st), (j / KV) & 1, flag)) return false;
                if (j >= SB && !mbar_wait_bounded(s_free(sb), ((j - SB) / SB) & 1, flag)) return false;
                tc_fence_after();
                const uint32_t kb = base + L::OFF_K + st * L::KV_BYTES;
#pragma unroll
                for (int s = 0; s < D / 16; ++s)   // K = 16 steps: atom s / 4, 32 B apart within it
                    tc_mma(tmem + sb * kAttnK,
                           smem_desc_sw128(base + L::OFF_Q + (s / 4) * L::Q_REGION + (s % 4) * 32, 16, 1024),
                           smem_desc_sw128(kb + (s / 4) * L::KV_REGION + (s % 4) * 32, 16, 1024), idS,
                           s > 0 ? 1u : 0u);
                tc_commit(s_full(sb));
                if (CL > 1 && j < nshared) tc_commit_mc(k_empty(st), kAll);   // free in every CTA
                else tc_commit(k_empty(st));
                issued = true;
                return true;
            };
            auto issue_pv = [&](int j) -> bool {
                const int st = j % KV, pi = j % PB;
                if (!mbar_wait_bounded(p_full(pi), (j / PB) & 1, flag)) return false;
                if (!mbar_wait_bounded(v_full(st), (j / KV) & 1, flag)) return false;
                tc_fence_after();
                const uint32_t pb = base + L::OFF_P + pi * L::P_BYTES;
                const uint32_t vb = base + L::OFF_V + st * L::KV_BYTES;
#pragma unroll
                for (int s = 0; s < kAttnK / 16; ++s)   // K = 16 keys: P atom s / 4; V rows 16 s..
                    tc_mma(tmem + L::O_COL, smem_desc_sw128(pb + (s / 4) * L::Q_REGION + (s % 4) * 32, 16, 1024),
                           smem_desc_sw128(vb + s * 2048, L::KV_REGION, 1024), idO,
                           (j > 0 || s > 0) ? 1u : 0u);
                tc_commit(o_done(pi));
                if (CL > 1 && j < nshared) tc_commit_mc(v_empty(st), kAll);
                else tc_commit(v_empty(st));
                issued = true;
                return true;
            };
            bool ok = mbar_wait_bounded(q_full, 0, flag);
            for (int j = 0; ok && j < SB - 1 && j < nb; ++j) ok = issue_s(j);
            for (int j = 0; ok && j < nb; ++j) {
                if (j + SB - 1 < nb && !issue_s(j + SB - 1)) { ok = false; break; }
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
        // Warp w serves TMEM lane quadrant w % 4 (query rows 32 (w % 4) + lane) and half hh of each
        // block's keys and of O's columns.  Both warps of a quadrant read the whole score row, so
        // they reach the same row maximum without exchanging it; each exponentiates and writes its
        // 32 keys of P and keeps the partial row sum of its own keys.
        const int qd = warp % 4;
        const int hh = (warp - 2) / 4;
        const int r = 32 * qd + lane;                        // query row within the tile
        const int qrow = qt * kAttnQ + r;                    // query index within the slice
        const uint32_t lanes = static_cast<uint32_t>(32 * qd) << 16;
        const float c = a.c;
        float m_used = -INFINITY, l = 0.0f;                  // m_used in base-2 units
        bool ok = true;
        // tcgen05.ld/st are warp-collective: every wait outcome is made warp-uniform before them
        for (int j = 0; j < nb; ++j) {
            const int pi = j % PB, sb = j % SB;
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(s_full(sb), (j / SB) & 1, flag))) {
                ok = false;
                break;
            }
            tc_fence_after();
            // own keys HK hh .. HK hh + HK - 1, then the other half (for the row maximum only)
            constexpr int HK = kAttnK / 2;
            float s[HK], so[HK];
            const uint32_t sbase = tmem + lanes + sb * kAttnK;
#pragma unroll
            for (int k = 0; k < HK / 32; ++k) {
                tmem_ld32(sbase + HK * hh + 32 * k, s + 32 * k);
                tmem_ld32(sbase + HK * (1 - hh) + 32 * k, so + 32 * k);
            }
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(s_free(sb));   // the score buffer may be overwritten now

            // keys with index > query index are masked (only in the blocks at the diagonal)
            const int lim = qrow - j * kAttnK;           // last visible key of this block
            const bool masked = lim < kAttnK - 1;
            const int k0 = HK * hh, ko = HK * (1 - hh);
            float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int k = 0; k < HK; ++k) {
                const float x = (masked && k0 + k > lim) ? -INFINITY : s[k];
                const float y = (masked && ko + k > lim) ? -INFINITY : so[k];
                mx4[k & 3] = fmaxf(mx4[k & 3], fmaxf(x, y));
            }
            const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * c;
            float alpha = 1.0f;
            bool rescale = false;
            if (mx > m_used + kRescaleLog2) {   // always true for the first block (m_used = -inf)
                if (j > 0) {
                    alpha = ex2f(m_used - mx);
                    rescale = true;
                }
                m_used = mx;
            }
            // p = 2^(s c - m) for this warp's HK keys, two at a time
            const float2 c2 = make_float2(c, c), nm2 = make_float2(-m_used, -m_used);
            float2 sum2 = make_float2(0.0f, 0.0f);
            uint32_t pk[HK / 2];
#pragma unroll
            for (int k = 0; k < HK; k += 2) {
                const float2 x = __ffma2_rn(make_float2(s[k], s[k + 1]), c2, nm2);
                float2 p = make_float2(ex2f(x.x), ex2f(x.y));
                if (masked) {
                    if (k0 + k > lim) p.x = 0.0f;
                    if (k0 + k + 1 > lim) p.y = 0.0f;
                }
                sum2 = __fadd2_rn(sum2, p);
                pk[k / 2] = pack_bf16x2(p.x, p.y);
            }
            l = l * alpha + (sum2.x + sum2.y);

            // P buffer pi was last read by PV_{j-PB}
            if (j >= PB) {
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(o_done(pi), ((j - PB) / PB) & 1, flag))) {
                    ok = false;
                    break;
                }
            }
            if (__any_sync(0xffffffffu, rescale)) {   // rows without a new maximum scale by 1
                // O must hold blocks 0..j-1 exactly: PV_{j-1} complete (PV_j is not issued yet)
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(o_done((j - 1) % PB), ((j - 1) / PB) & 1, flag))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll 1
                for (int k = 0; k < D / 64; ++k) {
                    const uint32_t col = L::O_COL + (D / 2) * hh + 32 * k;
                    float o[32];
                    tmem_ld32(tmem + lanes + col, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] *= alpha;
                    tmem_st32(tmem + lanes + col, o);
                }
                tmem_st_wait();
            }
            // P row r, this warp's keys: 16-byte chunks ch (8 keys each) lie in 64-key atom ch / 8
            // at slot (ch % 8) ^ (r % 8) of the row (128-byte swizzle)
            uint8_t* prow = gbase + L::OFF_P + pi * L::P_BYTES + r * 128;
#pragma unroll
            for (int q = 0; q < HK / 8; ++q) {
                const int ch = (HK / 8) * hh + q;
                uint4* dst = reinterpret_cast<uint4*>(prow + (ch / 8) * L::Q_REGION + (((ch % 8) ^ (r & 7)) << 4));
                *dst = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
            }
            fence_async_smem();   // the generic-proxy P writes become visible to the tensor core
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full(pi));
        }
        const int last = nb - 1;
        if (ok && __all_sync(0xffffffffu, mbar_wait_bounded(o_done(last % PB), (last / PB) & 1, flag))) {
            tc_fence_after();
            // the row sum is the sum of the two halves' partial sums; P is free now, so the
            // softmax warps exchange them there (a bounded mbarrier wait, not a named barrier:
            // a warp that gave up earlier must not leave its partner blocked)
            float* lx = reinterpret_cast<float*>(gbase + L::OFF_P);
            lx[hh * kAttnQ + r] = l;
            __syncwarp();
            if (lane == 0) mbar_arrive(l_ready);
            const bool got = __all_sync(0xffffffffu, mbar_wait_bounded(l_ready, 0, flag));
            const float inv = 1.0f / (l + lx[(1 - hh) * kAttnQ + r]);
            if (got) {
                __nv_bfloat16* orow = a.O + static_cast<int64_t>(row0 + r) * D + (D / 2) * hh;
#pragma unroll 1
                for (int k = 0; k < D / 64; ++k) {
                    float o[32];
                    tmem_ld32(tmem + lanes + L::O_COL + (D / 2) * hh + 32 * k, o);
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
    }
    tc_fence_before();
    // no CTA leaves while its peer may still multicast into its shared memory or commit to its
    // barriers
    if (CL > 1) cluster_sync();
    else __syncthreads();
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
template <int D, int CL>
int attn_attr() {
    static std::mutex mu;
    static bool done[64] = {false};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return record_cuda_error(e);
    if (dev < 0 || dev >= 64) return FUSE_EUNSUPPORTED;
    std::lock_guard<std::mutex> lock(mu);
    if (!done[dev]) {
        e = cudaFuncSetAttribute(attn_fwd_kernel<D, CL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(attn_launch_smem<D>()));
        if (e != cudaSuccess) return record_cuda_error(e);
        done[dev] = true;
    }
    return FUSE_OK;
}

template <int D, int CL>
int launch_attn(const CUtensorMap& mQ, const CUtensorMap& mK, const CUtensorMap& mV,
                const AttnArgs& args, cudaStream_t st) {
    const int rc = attn_attr<D, CL>();
    if (rc != FUSE_OK) return rc;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(static_cast<int64_t>(args.BH) * args.S / kAttnQ));
    cfg.blockDim = dim3(kAttnThreads);
    cfg.dynamicSmemBytes = attn_launch_smem<D>();
    cfg.stream = st;
    cudaLaunchAttribute attrs[1];
    attrs[0].id = cudaLaunchAttributeClusterDimension;
    attrs[0].val.clusterDim.x = CL;
    attrs[0].val.clusterDim.y = 1;
    attrs[0].val.clusterDim.z = 1;
    cfg.attrs = attrs;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, attn_fwd_kernel<D, CL>, mQ, mK, mV, args);
    if (e != cudaSuccess) return record_cuda_error(e);
    return check_launch();
}

template <int D>
int run_attn(const void* q, const void* k, const void* v, void* o, int bh, int S, float scale,
             cudaStream_t st) {
    const int64_t rows = static_cast<int64_t>(bh) * S;
    CUtensorMap mQ, mK, mV;
    if (!make_map(&mQ, q, rows, D, 64, kAttnQ, true) || !make_map(&mK, k, rows, D, 64, kAttnK, true) ||
        !make_map(&mV, v, rows, D, 64, kAttnK, true))
        return FUSE_ECUDA;
    int* flag = watchdog_flag();
    if (!flag) return FUSE_ECUDA;
    const AttnArgs args{bh, S, scale * 1.4426950408889634f, static_cast<__nv_bfloat16*>(o), flag};
    // pairs of adjacent query tiles share their key/value stream when the tiles pair up and the
    // head splits into two halves of 64-wide swizzle atoms
    if (D >= 128 && (S / kAttnQ) % 2 == 0) return launch_attn<D, 2>(mQ, mK, mV, args, st);
    return launch_attn<D, 1>(mQ, mK, mV, args, st);
}

bool overlap(const void* a, const void* b, int64_t bytes) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + static_cast<uintptr_t>(bytes) && y < x + static_cast<uintptr_t>(bytes);
}

}  // namespace

int attn_report_count() { return 1; }
int attn_report(int i, fuse_kernel_record* out) {
    if (i != 0) return FUSE_EINVAL;
    const int rc = attn_attr<256, 2>();
    if (rc != FUSE_OK) return rc;
    const int r2 = describe_kernel((const void*)attn_fwd_kernel<256, 2>,
                                   "attn_fwd_kernel<D=256> (tcgen05, 2-CTA K/V multicast)", kAttnThreads,
                                   static_cast<int>(attn_launch_smem<256>()), out);
    if (r2 == FUSE_OK) out->cluster_size = 2;
    return r2;
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
    if (D == 64) return run_attn<64>(q, k, v, o, B, SS, scale, st);
    if (D == 128) return run_attn<128>(q, k, v, o, B, SS, scale, st);
    return run_attn<256>(q, k, v, o, B, SS, scale, st);
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
