// attention.cu -- causal attention that never materialises the S x S score matrix.
//
// "AIGC fundamentals | operator fusion and CUDA Graph" §6.3 and its reading list: the score tensor
// of the causal softmax row ([B, H, S, S] = 1 GiB at B=8, H=16, S=2048) disappears altogether when
// the softmax is fused into the attention itself and normalised online (FlashAttention,
// arXiv:2205.14135), which also skips the masked half of the scores.  Per (batch, head) slice:
//     O = softmax(scale Q K^T, keys j <= query i) V,   Q, K, V, O bf16 [S, D].
//
// GB300 design, two kernels sharing the softmax code:
//  * attn_persist_kernel (D = 128, 256 with an even number of 128-row query tiles, the
//    benchmarked case): two CTAs of a cluster run as one 2-SM MMA unit over a pair of adjacent
//    query tiles, P goes from the softmax warps to the PV MMA through TMEM, and each cluster stays
//    resident over a list of tile pairs.  Described at the kernel.
//  * attn_fwd_kernel (D = 64, or an odd tile count): one CTA per 128-row query tile.  Keys go in
//    blocks of 128 (the MMA re-reads the whole Q tile from shared memory for every block, so longer
//    blocks cost less shared-memory bandwidth per flop), which at a head size of 256 leaves room
//    for one K, one V and one P buffer (Q 64 KB + K 64 KB + V 64 KB + P 32 KB) and two score
//    buffers in TMEM (2 x 128 score columns + 256 O columns).  352 threads in four roles:
//     - warps 0 and 2: lane 0 of warp 0 loads Q once and the K blocks, lane 0 of warp 2 the V
//       blocks (TMA, 128-byte swizzle), each as soon as its buffer is free (K_j+1 once S_j is
//       computed, V_j+1 once PV_j is);
//     - warp 1 owns TMEM and issues the tcgen05 MMAs: S_j = Q K_j^T (M 128, N 128, bf16, K-major
//       both) into score buffer j % 2, and O += P_j V_j (M 128, N D, P K-major, V MN-major), in
//       the order S_0, S_1, PV_0, S_2, PV_1, ... so the next scores are computed while the softmax
//       warps work on the current ones;
//     - warps 3-10 (two per TMEM lane quadrant, one query row per thread, each warp half of a
//       block's keys and half of O's columns) read the scores with tcgen05.ld, mask the diagonal
//       block, keep the running row maximum m and sum l in base-2 units, write P = 2^(s c - m) as
//       bf16 into shared memory in the MMA's swizzled layout, and rescale their half of the O
//       accumulator in TMEM only when the maximum has grown by more than 2^8 since it was last
//       applied (P stays <= 256, exact in the final O / l).  After the last block they divide O
//       by l and store it.
// Work runs in groups of 16 (batch, head) slices, heaviest tiles first within a group, so the
// tiles in flight together share their slices' key and value blocks in L2 (order_item()); the
// persistent kernel's clusters take that order through host-balanced item lists (build_sched()).
// All waits are bounded (watchdog); a CTA whose wait runs out drains its MMAs and copies and
// frees its TMEM before it returns.
#include <math.h>

#include <mutex>
#include <vector>

#include "fc_internal.cuh"
#include "fc_ptx.cuh"
#include "fc_tc.cuh"

namespace fc {
namespace {

constexpr int kAttnQ = 128;          // query rows per CTA
constexpr int kAttnK = 128;          // keys per block
constexpr int kKVStages = 1;         // K and V buffers (each a ring of this many blocks)
constexpr int kPBuf = 1;             // P buffers in shared memory
constexpr int kAttnSoftmaxWarps = 8; // two per TMEM lane quadrant, each exponentiating half a block's keys
// One-CTA kernel: warp 0: Q and K loads; warp 1: MMA issue; warp 2: V loads; warps 3-10: softmax.
// Every producer and the MMA issuer own a warp: a thread parked in an mbarrier wait parks its
// whole warp.
constexpr int kAttnThreads = 32 * (3 + kAttnSoftmaxWarps);
constexpr float kRescaleLog2 = 8.0f; // rescale O only when the row maximum grew by more than this
constexpr int kSBuf = 2;             // score buffers in TMEM: S_j+kSBuf-1 is computed before PV_j

// One-CTA kernel.  Shared memory: Q (128 x D), kKVStages K and V blocks (128 keys x D each) and
// kPBuf P buffers (128 x 128 bf16), all in 128-byte-swizzled 64-column atoms.  TMEM: kSBuf
// 128-column score buffers and the D-column O accumulator.
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

// Work order: item i of `per_head` items per (batch, head) slice, heaviest item (index 0 of a
// slice) ... lightest.  Slices go in groups of kOrderGroup: within a group the items run heaviest
// first across all of the group's slices, then the next group.  The group's key/value blocks
// (kOrderGroup x 2 x S x D x 2 B: 32 MiB at S = 2048, D = 256) stay in L2 while its items run, and
// every group ends with its lightest items, so the grid ends with short work instead of with the
// heaviest items of the last slices.
constexpr int kOrderGroup = 16;
__host__ __device__ __forceinline__ void order_item(int i, int per_head, int BH, int& bh, int& heavy_rank) {
    const int g = i / (kOrderGroup * per_head);
    const int gs = BH - g * kOrderGroup < kOrderGroup ? BH - g * kOrderGroup : kOrderGroup;   // slices in this group
    const int r = i - g * kOrderGroup * per_head;
    heavy_rank = r / gs;                                       // 0 = heaviest
    bh = g * kOrderGroup + r % gs;
}

// Per-cluster item lists of the persistent 2-SM kernel, passed as a kernel parameter.  Cluster c
// runs items item[first[c]] .. item[first[c + 1] - 1] (indices into the order_item() order, in
// increasing order).  n == 0: no list (more items or clusters than it holds), cluster c runs items
// c, c + C, c + 2C, ... of C clusters.
constexpr int kSchedClusters = 96;   // >= the 2-SM clusters resident on GB300 (76)
constexpr int kSchedItems = 4096;
struct AttnSched {
    int n;
    uint16_t first[kSchedClusters + 1];
    uint16_t item[kSchedItems];
};

// Per-warpgroup register budgets (the block is launched with 128 per thread).
template <int N> __device__ __forceinline__ void setmaxnreg_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N> __device__ __forceinline__ void setmaxnreg_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
// Wait until at most one committed bulk store group still reads its shared-memory source.
__device__ __forceinline__ void bulk_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }

__device__ __forceinline__ float max3f(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Keys k0 + k of a block at or past the diagonal that the lane's row does not see (k0 + k > lim)
// become -inf in place, one compare and select per key, so that the plain maximum and exponential
// below serve every block: a masked key gives -inf to the maximum and 2^-inf = +0 as its weight,
// the same maxima, weights and sums, bit for bit, as leaving it out.  (A separate masked copy of
// the maximum and exponential code, run once or twice per tile pair, came back to the SM's
// instruction cache every time and took twice as long as this.)
template <int HK>
__device__ __forceinline__ void mask_block(float (&v)[HK], int k0, int lim) {
    const int th = lim - k0;   // key k0 + k is visible iff k <= th
#pragma unroll
    for (int k = 0; k < HK; ++k) v[k] = k > th ? -INFINITY : v[k];
}

// Row maximum over this thread's HK scores s (keys k0 + k) and its partner warp's HK scores so
// (keys ko + k); with MASK, keys past `lim` (the last visible key of the block) are left out.
// Four independent chains of three-input maxima.
template <int HK, bool MASK>
__device__ __forceinline__ float block_row_max(const float (&s)[HK], const float (&so)[HK], int k0, int ko,
                                               int lim) {
    float m[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
    for (int k = 0; k < HK; ++k) {
        const float x = (MASK && k0 + k > lim) ? -INFINITY : s[k];
        const float y = (MASK && ko + k > lim) ? -INFINITY : so[k];
        m[k & 3] = max3f(m[k & 3], x, y);
    }
    return fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3]));
}

// p = 2^(s c - m) for this thread's HK keys, two at a time, packed to bf16 pairs; with MASK,
// keys past `lim` give p = 0.  Returns the (unrounded) sum of p as two partial sums.
template <int HK, bool MASK>
__device__ __forceinline__ float2 block_exp2(const float (&s)[HK], int k0, int lim, float c, float m,
                                             uint32_t (&pk)[HK / 2]) {
    const float2 c2 = make_float2(c, c), nm2 = make_float2(-m, -m);
    float2 sum2 = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int k = 0; k < HK; k += 2) {
        const float2 x = __ffma2_rn(make_float2(s[k], s[k + 1]), c2, nm2);
        float2 p = make_float2(ex2f(x.x), ex2f(x.y));
        if (MASK) {
            if (k0 + k > lim) p.x = 0.0f;
            if (k0 + k + 1 > lim) p.y = 0.0f;
        }
        sum2 = __fadd2_rn(sum2, p);
        pk[k / 2] = pack_bf16x2(p.x, p.y);
    }
    return sum2;
}

// The same two steps for a block at or past the diagonal, where key k of the block is visible to
// the lane's row iff k <= lim.  A warp's 32 lanes hold 32 consecutive rows, so their limits are
// base + lane with base = lim - lane a multiple of 32, and every aligned chunk of 32 keys is, for
// the whole warp, either visible (ks + 31 <= base), masked (ks > base + 31) or the one band where
// key ks + e is visible for lanes e <= lane (ks == base).  Branching per chunk on those
// warp-uniform cases keeps the per-element mask to that band and skips masked chunks (the
// softmax is issue-bound, and the element-wise mask of block_row_max / block_exp2 with MASK
// more than doubled a diagonal block's softmax time); maxima and sums are theirs, bit for bit
// (masked keys contribute -inf to the maximum and +0, in the same order, to the sum).
template <int HK>
__device__ __forceinline__ float block_row_max_diag(const float (&s)[HK], const float (&so)[HK], int k0, int ko,
                                                    int base, int lane) {
    float m[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
    auto chunk = [&](const float (&v)[HK], int ks, int c) {
        if (ks + 31 <= base) {
#pragma unroll
            for (int e = 0; e < 32; ++e) m[e & 3] = fmaxf(m[e & 3], v[32 * c + e]);
        } else if (ks == base) {
#pragma unroll
            for (int e = 0; e < 32; ++e) m[e & 3] = fmaxf(m[e & 3], e > lane ? -INFINITY : v[32 * c + e]);
        }
    };
#pragma unroll
    for (int c = 0; c < HK / 32; ++c) {
        chunk(s, k0 + 32 * c, c);
        chunk(so, ko + 32 * c, c);
    }
    return fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3]));
}

template <int HK>
__device__ __forceinline__ float2 block_exp2_diag(const float (&s)[HK], int k0, int base, int lane, float c,
                                                  float m, uint32_t (&pk)[HK / 2]) {
    const float2 c2 = make_float2(c, c), nm2 = make_float2(-m, -m);
    float2 sum2 = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int cc = 0; cc < HK / 32; ++cc) {
        const int ks = k0 + 32 * cc;
        if (ks + 31 <= base) {
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
                const int k = 32 * cc + e;
                const float2 x = __ffma2_rn(make_float2(s[k], s[k + 1]), c2, nm2);
                const float2 p = make_float2(ex2f(x.x), ex2f(x.y));
                sum2 = __fadd2_rn(sum2, p);
                pk[k / 2] = pack_bf16x2(p.x, p.y);
            }
        } else if (ks == base) {
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
                const int k = 32 * cc + e;
                const float2 x = __ffma2_rn(make_float2(s[k], s[k + 1]), c2, nm2);
                float2 p = make_float2(ex2f(x.x), ex2f(x.y));
                if (e > lane) p.x = 0.0f;
                if (e + 1 > lane) p.y = 0.0f;
                sum2 = __fadd2_rn(sum2, p);
                pk[k / 2] = pack_bf16x2(p.x, p.y);
            }
        } else {
#pragma unroll
            for (int e = 0; e < 32; e += 2) pk[(32 * cc + e) / 2] = 0u;
        }
    }
    return sum2;
}

template <int D>
__global__ void __launch_bounds__(kAttnThreads, 1) attn_fwd_kernel(
    const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
    const __grid_constant__ CUtensorMap mV, const __grid_constant__ AttnArgs a) {
    pdl_trigger();  // the set-up below touches no global memory; pdl_wait() follows it
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

    const int ntile = a.S / kAttnQ;
    int bh, heavy;
    order_item(static_cast<int>(blockIdx.x), ntile, a.BH, bh, heavy);
    const int qt = ntile - 1 - heavy;
    constexpr int kBlocksPerTile = kAttnQ / kAttnK;
    const int nb = (qt + 1) * kBlocksPerTile;             // key blocks up to the diagonal
    const int row0 = bh * a.S + qt * kAttnQ;
    const int krow0 = bh * a.S;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int i = 0; i < KV; ++i) {
            mbar_init(k_full(i), 1);
            mbar_init(k_empty(i), 1);
            mbar_init(v_full(i), 1);
            mbar_init(v_empty(i), 1);
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
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gbase + L::OFF_HOLD);
    pdl_wait();  // the preceding kernel has completed: global memory may be touched

    if (warp == 0 || warp == 2) {
        // ---------------------------------------------------------------- TMA producers
        // warp 0 loads Q and the K blocks, warp 2 the V blocks (lane 0 of each), each into its ring
        if (lane == 0) {
            const bool is_k = warp == 0;
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
                for (int c = 0; c < L::ATOMS; ++c) tma_load_2d(dst + c * L::KV_REGION, map, 64 * c, y, full);
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
                tc_commit(k_empty(st));
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
                tc_commit(v_empty(st));
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
        const int hh = (warp - 3) / 4;
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

            // keys with index > query index are masked: only in the blocks at and past the
            // tile's diagonal (j >= qt), a condition uniform over the CTA
            const int lim = qrow - j * kAttnK;           // last visible key of this block
            const bool diag = j >= qt;
            const int k0 = HK * hh, ko = HK * (1 - hh);
            const float mx = (diag ? block_row_max_diag<HK>(s, so, k0, ko, lim - lane, lane)
                                   : block_row_max<HK, false>(s, so, k0, ko, lim)) * c;
            float alpha = 1.0f;
            bool rescale = false;
            if (mx > m_used + kRescaleLog2) {   // always true for the first block (m_used = -inf)
                if (j > 0) {
                    alpha = ex2f(m_used - mx);
                    rescale = true;
                }
                m_used = mx;
            }
            // p = 2^(s c - m) for this warp's HK keys
            uint32_t pk[HK / 2];
            const float2 sum2 = diag ? block_exp2_diag<HK>(s, k0, lim - lane, lane, c, m_used, pk)
                                     : block_exp2<HK, false>(s, k0, lim, c, m_used, pk);
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
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, L::TMEM_COLS);
    }
}

// ================================================================== 2-SM variant (D = 128, 256)
// The two CTAs of a cluster hold adjacent query tiles 2u and 2u + 1 of one slice and act as one
// MMA unit (tcgen05 .cta_group::2, M = 256): S = Q K^T takes rows 0-127 of Q from CTA 0 and rows
// 128-255 from CTA 1 and keys 0-63 of the block from CTA 0, keys 64-127 from CTA 1; O += P V
// takes P's rows the same way and V's columns 0..D/2-1 from CTA 0, D/2..D-1 from CTA 1.  Each CTA
// so holds half of every key and value block: two K and two V stages fit next to Q at D = 256
// (Q 64 KB + K 2 x 32 KB + V 2 x 32 KB), and the MMAs read half as many B-operand bytes per flop
// from each CTA's shared memory.  P never touches shared memory: the softmax warps store it as
// bf16 into TMEM and the PV MMA takes its A operand from there.  TMEM (512 columns per CTA):
// S at 0-127 (one buffer: S_j+1 is computed as soon as both CTAs have read S_j), P at 128-255
// (two buffers of 64 columns, 128 bf16 keys each), O at 256-511.  The pair walks key blocks
// 0 .. 2u + 1 together (tile 2u finds block 2u + 1 fully masked).
// Warp roles are given at the persistent kernel below, the only kernel on this layout.
// K and V ring depths (K_j+2 is loaded once S_j has completed, V_j+2 once PV_j has).
constexpr int kPairK = 2, kPairV = 2;
// Warps that read out and store each item's O (one per TMEM lane quadrant).
constexpr int kAttnReadoutWarps = 4;

template <int D>
struct PairLayout {
    static constexpr int QATOMS = D / 64;                      // 64-column swizzle atoms of Q and K
    static constexpr int VATOMS = D / 128;                     // atoms of this CTA's V columns
    static constexpr uint32_t Q_REGION = kAttnQ * 128;         // one Q atom: 128 rows x 128 B
    static constexpr uint32_t KH_REGION = (kAttnK / 2) * 128;  // one atom of a K half: 64 keys x 128 B
    static constexpr uint32_t V_REGION = kAttnK * 128;         // one atom of a V half: 128 keys x 128 B
    static constexpr uint32_t Q_BYTES = kAttnQ * D * 2;
    static constexpr uint32_t KH_BYTES = (kAttnK / 2) * D * 2;
    static constexpr uint32_t VH_BYTES = kAttnK * (D / 2) * 2;
    static constexpr uint32_t OFF_Q = 0;
    static constexpr uint32_t OFF_K = OFF_Q + Q_BYTES;                 // + stage * KH_BYTES
    static constexpr uint32_t OFF_V = OFF_K + kPairK * KH_BYTES;       // + stage * VH_BYTES
    // output staging: two boxes per output warp, each 32 rows x 64 columns of bf16 (one
    // 128-byte-swizzled box of the O tensor map), written to global memory by TMA stores
    static constexpr uint32_t ST_WARP = 32 * 128;
    static constexpr uint32_t OFF_ST = OFF_V + kPairV * VH_BYTES;
    static constexpr uint32_t OFF_LX = OFF_ST + 2 * kAttnReadoutWarps * ST_WARP;   // row sums, 2 x 128 fp32
    static constexpr uint32_t OFF_BAR = OFF_LX + 2 * kAttnQ * 4;
    // q_full, drain, l_ready, s_full, s_free, p_full[2], o_done[2], k_full[KS], k_empty[KS],
    // v_full[VS], v_empty[VS], q_empty, o_free, lx_free
    static constexpr int N_BARS = 9 + 2 * kPairK + 2 * kPairV + 3;
    static constexpr uint32_t OFF_HOLD = OFF_BAR + N_BARS * 8;
    static constexpr uint32_t SMEM = OFF_HOLD + 16 + 1024;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t S_COL = 0, P_COL = 128, O_COL = 256;
    static_assert(D == 128 || D == 256, "2-SM attention handles D = 128 and 256");
    static_assert(S_COL + kAttnK <= P_COL && P_COL + 2 * (kAttnK / 2) <= O_COL && O_COL + D <= TMEM_COLS,
                  "TMEM budget");
    static_assert(SMEM <= 232448, "shared-memory budget");
};

// ================================================================== persistent 2-SM variant
// The 2-SM pipeline above in a persistent kernel: each cluster stays resident and walks its list
// of tile pairs (AttnSched), so the set-up (TMEM allocation, barriers) happens once and every
// ring (K, V, S, P) runs on across items: the next item's Q, K and V stream in while the current
// item finishes.  Roles (512 threads per CTA):
//   warp 0, lane 0: this CTA's half of every K block (TMA), and with an item's last K block the
//     next item's Q rows into L2; warp 2, lane 0: its half of every V block; warp 3, lane 0: its
//     128 Q rows.  The bytes of both CTAs complete on CTA 0's barriers.
//     Q gets a warp of its own because the next item's Q may only overwrite the current one once
//     the current item's last S has completed (q_empty), and the K and V rings must not wait.
//   warp 1 of CTA 0: every MMA of the pair, per item in the order S_0, S_1, PV_0, S_2, PV_1, ...;
//     its commits signal both CTAs' barriers.
//   warps 4-11: softmax of this CTA's 128 query rows (two warps per TMEM lane quadrant, each
//     exponentiating half of a block's keys and rescaling half of O's columns); they release S
//     and publish P on CTA 0's barriers, and after an item's last block its row sums (l_ready).
//   warps 12-15: the output: once an item's last PV has completed, each reads its lane
//     quadrant's 32 rows of O from TMEM, divides them by the row sums and arrives on o_free as
//     soon as all of them have left TMEM (the next item's PV_0, which overwrites O with
//     accumulate off, waits for it), then stores them (staged in shared memory, TMA box stores).
//     Meanwhile the softmax warps go on with the next item's S blocks, so its S MMAs fill the
//     tensor pipe while O is read out.
// Register budgets per warpgroup (setmaxnreg; launched at 128 per thread): producers and MMA
// issuer 48, softmax 160, output 144 -- 48 x 128 + 160 x 256 + 144 x 128 = 65,536, all the CTA is
// launched with.
constexpr int kPersistThreads = 32 * (4 + kAttnSoftmaxWarps + kAttnReadoutWarps);

template <int D>
__global__ void __launch_bounds__(kPersistThreads, 1) attn_persist_kernel(
    const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mKh,
    const __grid_constant__ CUtensorMap mV,
    const __grid_constant__ CUtensorMap mO, const __grid_constant__ AttnArgs a,
    const __grid_constant__ AttnSched sch) {
    pdl_trigger();  // the set-up below touches no global memory; pdl_wait() follows it
    using L = PairLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (smem_addr(smem_raw) + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - smem_addr(smem_raw));
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    // barriers: q_full, drain, l_ready, s_full, s_free, p_full[2], o_done[2], K ring, V ring,
    // then q_empty and o_free
    const uint32_t bar0 = base + L::OFF_BAR;
    const uint32_t q_full = bar0, drain = bar0 + 8, l_ready = bar0 + 16, s_full = bar0 + 24,
                   s_free = bar0 + 32;
    constexpr int KS = kPairK, VS = kPairV;
    auto p_full = [&](int b) { return bar0 + 8u * (5 + b); };
    auto o_done = [&](int b) { return bar0 + 8u * (7 + b); };
    auto k_full = [&](int i) { return bar0 + 8u * (9 + i); };
    auto k_empty = [&](int i) { return bar0 + 8u * (9 + KS + i); };
    auto v_full = [&](int i) { return bar0 + 8u * (9 + 2 * KS + i); };
    auto v_empty = [&](int i) { return bar0 + 8u * (9 + 2 * KS + VS + i); };
    const uint32_t q_empty = bar0 + 8u * (L::N_BARS - 3), o_free = bar0 + 8u * (L::N_BARS - 2);
    const uint32_t lx_free = bar0 + 8u * (L::N_BARS - 1);
    int* flag = a.flag;

    const int ntile = a.S / kAttnQ;
    const int per_head = ntile / 2;
    const int n_items = a.BH * per_head;
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;
    const int cid = blockIdx.x / 2, ncl = gridDim.x / 2;
    const int my_first = sch.n ? sch.first[cid] : 0;
    const int my_items = sch.n ? sch.first[cid + 1] - my_first
                               : (cid < n_items ? (n_items - cid + ncl - 1) / ncl : 0);
    // item t of this cluster -> slice, pair index u, key blocks, first query row
    auto item = [&](int t, int& bh, int& u, int& nb) {
        int heavy;
        order_item(sch.n ? static_cast<int>(sch.item[my_first + t]) : cid + t * ncl, per_head, a.BH, bh, heavy);
        u = per_head - 1 - heavy;
        nb = (2 * u + 2) * (kAttnQ / kAttnK);
    };

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        mbar_init(o_free, 2 * kAttnReadoutWarps);   // both CTAs' output warps (CTA 0's copy)
        mbar_init(lx_free, kAttnReadoutWarps);      // this CTA's output warps have read the row sums
        mbar_init(drain, 1);
        mbar_init(l_ready, kAttnSoftmaxWarps);
        mbar_init(s_full, 1);
        mbar_init(s_free, 2 * kAttnSoftmaxWarps);   // both CTAs' softmax warps (CTA 0's copy)
        for (int b = 0; b < 2; ++b) {
            mbar_init(p_full(b), 2 * kAttnSoftmaxWarps);
            mbar_init(o_done(b), 1);
        }
        for (int i = 0; i < KS; ++i) {
            mbar_init(k_full(i), 1);
            mbar_init(k_empty(i), 1);
        }
        for (int i = 0; i < VS; ++i) {
            mbar_init(v_full(i), 1);
            mbar_init(v_empty(i), 1);
        }
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc_pair(base + L::OFF_HOLD, L::TMEM_COLS);
    tc_fence_before();
    cluster_sync();   // both CTAs' barriers exist before either signals the other
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gbase + L::OFF_HOLD);
    // The cluster's first item's Q rows and first key and value blocks on their way into L2 while
    // the preceding kernel may still run (an L2 fill changes no data, whoever writes these lines
    // before the grid-dependency wait returns).
    if (lane == 0 && my_items > 0 && (warp == 0 || warp == 2 || warp == 3)) {
        int bh, u, nb;
        item(0, bh, u, nb);
        if (warp == 3) {
            const int row0 = bh * a.S + (2 * u + static_cast<int>(rank)) * kAttnQ;
            for (int c = 0; c < L::QATOMS; ++c) tma_prefetch_2d(&mQ, 64 * c, row0);
        } else if (warp == 0) {
            for (int j = 0; j < nb && j < kPairK; ++j)
                for (int c = 0; c < L::QATOMS; ++c)
                    tma_prefetch_2d(&mKh, 64 * c, bh * a.S + j * kAttnK + static_cast<int>(rank) * (kAttnK / 2));
        } else {
            for (int j = 0; j < nb && j < kPairV; ++j)
                for (int c = 0; c < L::VATOMS; ++c)
                    tma_prefetch_2d(&mV, static_cast<int>(rank) * (D / 2) + 64 * c, bh * a.S + j * kAttnK);
        }
    }
    pdl_wait();  // the preceding kernel has completed: global memory may be touched

    if (warp < 4) {
        // ================================================ warpgroup 0: producers and MMA issuer
        setmaxnreg_dec<48>();
        if (warp == 0 || warp == 2) {
            // ---------------------------------------------------------------- K / V producers
            if (lane == 0) {
                const bool is_k = warp == 0;
                prefetch_map(is_k ? &mKh : &mV);
                const int R = is_k ? KS : VS;
                int g = 0;   // blocks loaded so far, over all items
                bool ok = true;
                for (int t = 0; ok && t < my_items; ++t) {
                    int bh, u, nb;
                    item(t, bh, u, nb);
                    const int krow0 = bh * a.S;
                    for (int j = 0; j < nb; ++j, ++g) {
                        const int st = g % R;
                        const uint32_t full = is_k ? k_full(st) : v_full(st);
                        const uint32_t empty = is_k ? k_empty(st) : v_empty(st);
                        if (g >= R && !mbar_wait_bounded(empty, ((g - R) / R) & 1, flag)) { ok = false; break; }
                        if (leader) mbar_arrive_expect_tx(full, 2 * (is_k ? L::KH_BYTES : L::VH_BYTES));
                        const uint32_t full_cl = mapa_shared(full, 0);
                        if (is_k) {
                            const int y = krow0 + j * kAttnK + static_cast<int>(rank) * (kAttnK / 2);
                            for (int c = 0; c < L::QATOMS; ++c)
                                tma_load_2d_pair(base + L::OFF_K + st * L::KH_BYTES + c * L::KH_REGION, &mKh, 64 * c, y,
                                                 full_cl);
                            // the next item's Q rows into L2 once this item's last K block is on its
                            // way, about two blocks before the Q producer loads them
                            if (j == nb - 1 && t + 1 < my_items) {
                                int nbh, nu, nnb;
                                item(t + 1, nbh, nu, nnb);
                                const int qrow = nbh * a.S + (2 * nu + static_cast<int>(rank)) * kAttnQ;
                                for (int c = 0; c < L::QATOMS; ++c) tma_prefetch_2d(&mQ, 64 * c, qrow);
                            }
                        } else {
                            const int y = krow0 + j * kAttnK;
                            for (int c = 0; c < L::VATOMS; ++c)
                                tma_load_2d_pair(base + L::OFF_V + st * L::VH_BYTES + c * L::V_REGION, &mV,
                                                 static_cast<int>(rank) * (D / 2) + 64 * c, y, full_cl);
                        }
                    }
                }
                if (!ok && leader)   // both CTAs' copies in flight complete on CTA 0's barriers
                    for (int h = g - R < 0 ? 0 : g - R; h < g; ++h)
                        (void)mbar_wait_drain(is_k ? k_full(h % R) : v_full(h % R), (h / R) & 1);
            }
            __syncwarp();
        } else if (warp == 3) {
            // ---------------------------------------------------------------- Q producer
            if (lane == 0) {
                prefetch_map(&mQ);
                const uint32_t qf = mapa_shared(q_full, 0);
                // Each item's rows are looked up (list and order, a few hundred cycles) one item ahead,
                // so the load follows the q_empty wait at once.
                int row0 = 0;
                if (my_items > 0) {
                    int bh, u, nb;
                    item(0, bh, u, nb);
                    row0 = bh * a.S + (2 * u + static_cast<int>(rank)) * kAttnQ;
                }
                int t = 0;
                for (; t < my_items; ++t) {
                    // the previous item's last S has completed in both CTAs
                    if (t >= 1 && !mbar_wait_bounded(q_empty, (t - 1) & 1, flag)) break;
                    if (leader) mbar_arrive_expect_tx(q_full, 2 * L::Q_BYTES);
                    for (int c = 0; c < L::QATOMS; ++c)
                        tma_load_2d_pair(base + L::OFF_Q + c * L::Q_REGION, &mQ, 64 * c, row0, qf);
                    // the next item's rows (its Q reaches L2 by the K producer's prefetch, two blocks
                    // before this item's last S frees the buffer)
                    if (t + 1 < my_items) {
                        int bh, u, nb;
                        item(t + 1, bh, u, nb);
                        row0 = bh * a.S + (2 * u + static_cast<int>(rank)) * kAttnQ;
                    }
                }
                if (t < my_items && t >= 1 && leader) (void)mbar_wait_drain(q_full, (t - 1) & 1);
            }
            __syncwarp();
        } else {
            // ---------------------------------------------------------------- MMA issuer (CTA 0)
            if (leader && lane == 0) {
                constexpr uint32_t idS = idesc_f16(2 * kAttnQ, kAttnK, false, false, true);
                constexpr uint32_t idO = idesc_f16(2 * kAttnQ, D, false, true, true);
                bool issued = false;
                // S_j and PV_j of item t are global block g = (blocks of earlier items) + j
                auto issue_s = [&](int t, int j, int g, int nb) -> bool {
                    const int st = g % KS;
                    if (j == 0 && !mbar_wait_bounded(q_full, t & 1, flag)) return false;
                    if (!mbar_wait_bounded(k_full(st), (g / KS) & 1, flag)) return false;
                    // both CTAs have read the previous S into registers
                    if (g >= 1 && !mbar_wait_bounded(s_free, (g - 1) & 1, flag)) return false;
                    tc_fence_after();
                    const uint32_t kb = base + L::OFF_K + st * L::KH_BYTES;
#pragma unroll
                    for (int s = 0; s < D / 16; ++s)
                        tc_mma_pair(tmem + L::S_COL,
                                    smem_desc_sw128(base + L::OFF_Q + (s / 4) * L::Q_REGION + (s % 4) * 32, 16, 1024),
                                    smem_desc_sw128(kb + (s / 4) * L::KH_REGION + (s % 4) * 32, 16, 1024), idS,
                                    s > 0 ? 1u : 0u);
                    tc_commit_pair_mc(s_full, 0x3);
                    tc_commit_pair_mc(k_empty(st), 0x3);
                    if (j == nb - 1) tc_commit_pair_mc(q_empty, 0x3);   // the item's Q is no longer read
                    issued = true;
                    return true;
                };
                auto issue_pv = [&](int t, int j, int g) -> bool {
                    const int st = g % VS, pb = g % 2;
                    if (!mbar_wait_bounded(p_full(pb), (g / 2) & 1, flag)) return false;
                    // the previous item's O has been read out by both CTAs
                    if (j == 0 && t >= 1 && !mbar_wait_bounded(o_free, (t - 1) & 1, flag)) return false;
                    if (!mbar_wait_bounded(v_full(st), (g / VS) & 1, flag)) return false;
                    tc_fence_after();
                    const uint32_t vb = base + L::OFF_V + st * L::VH_BYTES;
#pragma unroll
                    for (int s = 0; s < kAttnK / 16; ++s)
                        tc_mma_pair_ts(tmem + L::O_COL, tmem + L::P_COL + (kAttnK / 2) * pb + 8 * s,
                                       smem_desc_sw128(vb + s * 2048, L::V_REGION, 1024), idO,
                                       (j > 0 || s > 0) ? 1u : 0u);
                    tc_commit_pair_mc(o_done(pb), 0x3);
                    tc_commit_pair_mc(v_empty(st), 0x3);
                    issued = true;
                    return true;
                };
                // S_0, then for every block g (over all items) S_g+1 before PV_g: the next scores are
                // computed while the softmax warps work on the current ones, across item boundaries
                // too (the next item's S_0 precedes the current item's last PV)
                // The item after the S cursor's is looked up (nb_next) once the cursor's item has
                // issued its S_0, while the queued MMAs run; when the PV cursor moves on, the S cursor
                // is already on that item (S runs one block ahead), so its block count is nbs.
                bool ok = my_items > 0;
                int ts = 0, js = 0, nbs = 0, tp = 0, jp = 0, nbp = 0, nb_next = 0, bh_, u_;
                if (ok) {
                    item(0, bh_, u_, nbs);
                    nbp = nbs;
                    ok = issue_s(0, 0, 0, nbs);
                    js = 1;
                    if (my_items > 1) item(1, bh_, u_, nb_next);
                }
                for (int g = 0; ok && tp < my_items; ++g) {
                    if (js == nbs && ts + 1 < my_items) {   // the S cursor moves to the next item
                        ++ts;
                        js = 0;
                        nbs = nb_next;
                    }
                    if (js < nbs) {
                        if (!issue_s(ts, js, g + 1, nbs)) { ok = false; break; }
                        if (++js == 1 && ts + 1 < my_items) item(ts + 1, bh_, u_, nb_next);
                    }
                    if (!issue_pv(tp, jp, g)) { ok = false; break; }
                    if (++jp == nbp && ++tp < my_items) {
                        jp = 0;
                        nbp = nbs;
                    }
                }
                if (!ok && issued) {  // MMAs in flight must finish before TMEM is freed
                    tc_commit_pair(drain);
                    (void)mbar_wait_drain(drain, 0);
                }
            }
            __syncwarp();
        }
    } else if (warp < 4 + kAttnSoftmaxWarps) {
        setmaxnreg_inc<160>();
        // ---------------------------------------------------------------- softmax warps
        // Warp w serves TMEM lane quadrant w % 4 (query rows 32 (w % 4) + lane of this CTA's tile)
        // and half hh of each block's keys and of O's columns.
        const int qd = warp % 4;
        const int hh = (warp - 4) / 4;
        const int r = 32 * qd + lane;
        const uint32_t lanes = static_cast<uint32_t>(32 * qd) << 16;
        const float c = a.c;
        const uint32_t s_free0 = mapa_shared(s_free, 0);
        const uint32_t p_full_a = mapa_shared(p_full(0), 0), p_full_b = mapa_shared(p_full(1), 0);
        float* lx = reinterpret_cast<float*>(gbase + L::OFF_LX);
        bool ok = true;
        int g = 0;   // global block index
        for (int t = 0; ok && t < my_items; ++t) {
            int bh, u, nb;
            item(t, bh, u, nb);
            const int qt = 2 * u + static_cast<int>(rank);
            const int qrow = qt * kAttnQ + r;
            float m_used = -INFINITY, l = 0.0f;
            // tcgen05.ld/st are warp-collective: every wait outcome is made warp-uniform before them
            for (int j = 0; j < nb; ++j, ++g) {
                const int pb = g % 2;
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(s_full, g & 1, flag))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                constexpr int HK = kAttnK / 2;
                float s[HK], so[HK];
                const uint32_t sbase = tmem + lanes + L::S_COL;
#pragma unroll
                for (int k = 0; k < HK / 32; ++k) {
                    tmem_ld32(sbase + HK * hh + 32 * k, s + 32 * k);
                    tmem_ld32(sbase + HK * (1 - hh) + 32 * k, so + 32 * k);
                }
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(s_free0);   // S may be overwritten now

                const int lim = qrow - j * kAttnK;           // last visible key of this block
                const bool diag = j >= qt;
                const int k0 = HK * hh, ko = HK * (1 - hh);
                const bool past = j > qt;   // every key of the block lies past this CTA's rows
                if (diag && !past) {
                    mask_block<HK>(s, k0, lim);
                    mask_block<HK>(so, ko, lim);
                }
                const float mx = past ? -INFINITY : block_row_max<HK, false>(s, so, k0, ko, lim) * c;
                float alpha = 1.0f;
                bool rescale = false;
                if (mx > m_used + kRescaleLog2) {
                    if (j > 0) {
                        alpha = ex2f(m_used - mx);
                        rescale = true;
                    }
                    m_used = mx;
                }
                uint32_t pk[HK / 2];
                float2 sum2 = make_float2(0.0f, 0.0f);
                if (past) {
#pragma unroll
                    for (int i = 0; i < HK / 2; ++i) pk[i] = 0u;
                } else {
                    sum2 = block_exp2<HK, false>(s, k0, lim, c, m_used, pk);
                }
                l = l * alpha + (sum2.x + sum2.y);

                // P buffer pb was last read by PV of global block g - 2
                if (g >= 2) {
                    if (!__all_sync(0xffffffffu, mbar_wait_bounded(o_done(pb), ((g - 2) / 2) & 1, flag))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                }
                if (__any_sync(0xffffffffu, rescale)) {
                    // O must hold blocks 0..j-1 of this item exactly: PV of block g - 1 complete
                    if (!__all_sync(0xffffffffu, mbar_wait_bounded(o_done((g - 1) % 2), ((g - 1) / 2) & 1, flag))) {
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
                }
                tmem_st32(tmem + lanes + L::P_COL + HK * pb + (HK / 2) * hh, reinterpret_cast<const float*>(pk));
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(pb ? p_full_b : p_full_a);
            }
            if (!ok) break;
            // the item's row sums (this warp's half of the keys) for the output warps, once they
            // have read the previous item's
            if (t >= 1 && !__all_sync(0xffffffffu, mbar_wait_bounded(lx_free, (t - 1) & 1, flag))) {
                ok = false;
                break;
            }
            lx[hh * kAttnQ + r] = l;
            __syncwarp();
            if (lane == 0) mbar_arrive(l_ready);
        }
    } else {
        // ---------------------------------------------------------------- output warps
        setmaxnreg_inc<144>();   // 48 x 128 + 160 x 256 + 144 x 128 = 65,536 (the launch's 512 x 128)
        // Warp 12 + q reads TMEM lane quadrant q: rows 32 q + lane of this CTA's tile, all of O's
        // columns, 64 at a time (chunk k), and stores them (scaled by 1 / l, bf16) through its two
        // staging boxes (row = lane, 16-byte pieces in the 128-byte swizzle of the O tensor map)
        // with TMA box stores; a box is written again only once the store from it two chunks
        // earlier has read it.  O leaves TMEM as early as the registers allow: chunks 0 .. NCH - 3
        // go straight to their boxes, chunk NCH - 2 is held packed to bf16 pairs and chunk
        // NCH - 1 as fp32, and o_free is signalled once all of them are read, so the next item's
        // PV_0 overwrites O while the last two chunks are staged and stored.
        constexpr int NCH = D / 64;
        const int ow = warp - 4 - kAttnSoftmaxWarps;
        const int qd = warp % 4;
        const int r = 32 * qd + lane;
        const uint32_t lanes = static_cast<uint32_t>(32 * qd) << 16;
        const float* lx = reinterpret_cast<const float*>(gbase + L::OFF_LX);
        const uint32_t o_free0 = mapa_shared(o_free, 0);
        auto stage_box = [&](int k, int orow0, const uint32_t (&w)[32]) {
            const int box = 2 * ow + (k & 1);
            uint8_t* stage = gbase + L::OFF_ST + box * L::ST_WARP;
            if (lane == 0) bulk_wait_read1();   // the store from this box two chunks ago has read it
            __syncwarp();
#pragma unroll
            for (int v = 0; v < 8; ++v)
                *reinterpret_cast<uint4*>(stage + lane * 128 + ((v ^ (lane & 7)) * 16)) =
                    make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
            fence_async_smem();   // generic-proxy writes become visible to the TMA engine
            __syncwarp();
            if (lane == 0) {
                tma_store_2d(&mO, 64 * k, orow0, base + L::OFF_ST + box * L::ST_WARP);
                bulk_commit();
            }
        };
        auto pack = [&](const float (&o)[64], float inv, uint32_t (&w)[32]) {
#pragma unroll
            for (int v = 0; v < 32; ++v) w[v] = pack_bf16x2(o[2 * v] * inv, o[2 * v + 1] * inv);
        };
        bool ok = true;
        int g = 0;
        for (int t = 0; ok && t < my_items; ++t) {
            int bh, u, nb;
            item(t, bh, u, nb);
            const int qt = 2 * u + static_cast<int>(rank);
            g += nb;
            const int g_last = g - 1;   // the item's last PV
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(l_ready, t & 1, flag)) ||
                !__all_sync(0xffffffffu, mbar_wait_bounded(o_done(g_last % 2), (g_last / 2) & 1, flag))) {
                ok = false;
                break;
            }
            tc_fence_after();
            const float inv = 1.0f / (lx[r] + lx[kAttnQ + r]);
            __syncwarp();
            if (lane == 0) mbar_arrive(lx_free);
            const int orow0 = bh * a.S + qt * kAttnQ + 32 * qd;
            float o[64];
            uint32_t w[32], held[32];
#pragma unroll 1
            for (int k = 0; k < NCH - 2; ++k) {
                tmem_ld32(tmem + lanes + L::O_COL + 64 * k, o);
                tmem_ld32(tmem + lanes + L::O_COL + 64 * k + 32, o + 32);
                tmem_ld_wait();
                pack(o, inv, w);
                stage_box(k, orow0, w);
            }
            tmem_ld32(tmem + lanes + L::O_COL + 64 * (NCH - 2), o);
            tmem_ld32(tmem + lanes + L::O_COL + 64 * (NCH - 2) + 32, o + 32);
            tmem_ld_wait();
            pack(o, inv, held);
            tmem_ld32(tmem + lanes + L::O_COL + 64 * (NCH - 1), o);
            tmem_ld32(tmem + lanes + L::O_COL + 64 * (NCH - 1) + 32, o + 32);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(o_free0);   // the next item's PV_0 may overwrite O
            stage_box(NCH - 2, orow0, held);
            pack(o, inv, w);
            stage_box(NCH - 1, orow0, w);
        }
        if (lane == 0) bulk_wait0();   // the output stores have completed
        __syncwarp();
    }
    tc_fence_before();
    // neither CTA leaves while its peer may still read its shared memory or TMEM (MMA operands),
    // write into it (copies) or signal its barriers
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, L::TMEM_COLS);
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
int launch_attn(const CUtensorMap& mQ, const CUtensorMap& mK, const CUtensorMap& mV,
                const AttnArgs& args, cudaStream_t st) {
    const int rc = attn_attr<D>();
    if (rc != FUSE_OK) return rc;
    return launch_pdl(attn_fwd_kernel<D>, dim3(static_cast<unsigned>(static_cast<int64_t>(args.BH) * args.S / kAttnQ)), dim3(kAttnThreads), attn_launch_smem<D>(), st, 1, mQ, mK, mV, args);
}

// Balanced item lists for `ncl` clusters: the items, in order_item() order, go one after another
// to the cluster whose estimated finish time is earliest (the order a shared work queue would hand
// them out in), so the clusters finish together; a plain round-robin leaves the busiest cluster
// ~14 % above the mean at [128, 2048, 256] on 76 clusters.  Estimated cost of an item: 10 per key
// block plus 8 for its fixed costs (what an item boundary adds, the wait for the next Q and for
// the output release, measured at 0.75 of a block).  Lists are cached per shape.
void build_sched(int BH, int per_head, int ncl, AttnSched* out) {
    out->n = 0;
    const int64_t n = static_cast<int64_t>(BH) * per_head;
    if (n > kSchedItems || ncl > kSchedClusters || ncl < 1) return;
    int64_t load[kSchedClusters] = {0};
    int count[kSchedClusters] = {0};
    static thread_local uint8_t owner[kSchedItems];
    static thread_local int16_t nblk[kSchedItems];
    std::vector<int> mine[kSchedClusters];
    for (int i = 0; i < static_cast<int>(n); ++i) {
        int c = 0;
        for (int j = 1; j < ncl; ++j)
            if (load[j] < load[c]) c = j;
        int bh, heavy;
        order_item(i, per_head, BH, bh, heavy);
        nblk[i] = static_cast<int16_t>(2 * (per_head - 1 - heavy) + 2);
        load[c] += 10 * nblk[i] + 8;
        owner[i] = static_cast<uint8_t>(c);
        mine[c].push_back(i);
        ++count[c];
    }
    // Assigned one after another, the group's last items (the lightest are still 2 key blocks)
    // leave the estimated loads a few per cent apart (up to 3.4 us above the mean at [128, 2048,
    // 256] on 76 clusters).  Evening them out: an item of the busiest cluster trades places with a
    // lighter item of the same slice group (so it still runs while that group's key and value
    // blocks are in L2) in the idlest cluster, the pair that best halves their gap, until no trade
    // narrows it (0.8 us above the mean on the same case).
    const int per_group = kOrderGroup * per_head;
    for (int it = 0; it < 8 * ncl; ++it) {
        int cmax = 0, cmin = 0;
        for (int c = 1; c < ncl; ++c) {
            if (load[c] > load[cmax]) cmax = c;
            if (load[c] < load[cmin]) cmin = c;
        }
        const int64_t gap = load[cmax] - load[cmin];
        int ia = -1, ib = -1;
        int64_t best = 0, best_d = 0;
        for (int x = 0; x < static_cast<int>(mine[cmax].size()); ++x)
            for (int y = 0; y < static_cast<int>(mine[cmin].size()); ++y) {
                const int a = mine[cmax][x], b = mine[cmin][y];
                if (a / per_group != b / per_group) continue;
                const int64_t d = 10 * (nblk[a] - nblk[b]);
                if (d <= 0 || d >= gap) continue;
                const int64_t score = gap - 2 * d < 0 ? 2 * d - gap : gap - 2 * d;
                if (ia < 0 || score < best) {
                    ia = x;
                    ib = y;
                    best = score;
                    best_d = d;
                }
            }
        if (ia < 0) break;
        const int a = mine[cmax][ia], b = mine[cmin][ib];
        mine[cmax][ia] = b;
        mine[cmin][ib] = a;
        owner[a] = static_cast<uint8_t>(cmin);
        owner[b] = static_cast<uint8_t>(cmax);
        load[cmax] -= best_d;
        load[cmin] += best_d;
    }
    out->first[0] = 0;
    for (int c = 0; c < ncl; ++c) out->first[c + 1] = static_cast<uint16_t>(out->first[c] + count[c]);
    int fill[kSchedClusters];
    for (int c = 0; c < ncl; ++c) fill[c] = out->first[c];
    for (int i = 0; i < static_cast<int>(n); ++i) out->item[fill[owner[i]]++] = static_cast<uint16_t>(i);
    out->n = static_cast<int>(n);
}

struct SchedEntry {
    int BH = 0, per_head = 0, ncl = 0;
    AttnSched s;
};

// Copies the cached list for (BH, per_head, ncl) into *out, building it on first use.
void get_sched(int BH, int per_head, int ncl, AttnSched* out) {
    static std::mutex mu;
    static SchedEntry cache[8];
    static int next = 0;
    std::lock_guard<std::mutex> lock(mu);
    for (const SchedEntry& e : cache)
        if (e.ncl == ncl && e.BH == BH && e.per_head == per_head) {
            *out = e.s;
            return;
        }
    SchedEntry& e = cache[next];
    next = (next + 1) % 8;
    e.BH = BH;
    e.per_head = per_head;
    e.ncl = ncl;
    build_sched(BH, per_head, ncl, &e.s);
    *out = e.s;
}

// Sets the persistent kernel's shared-memory attribute once per device and returns (through *n)
// how many of its clusters can be resident at once.
template <int D>
int persist_setup(int* n_out) {
    static std::mutex mu;
    static int clusters[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return record_cuda_error(e);
    if (dev < 0 || dev >= 64) return FUSE_EUNSUPPORTED;
    std::lock_guard<std::mutex> lock(mu);
    if (clusters[dev] == 0) {
        e = cudaFuncSetAttribute(attn_persist_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(PairLayout<D>::SMEM));
        if (e != cudaSuccess) return record_cuda_error(e);
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * static_cast<unsigned>(sm_count()));
        cfg.blockDim = dim3(kPersistThreads);
        cfg.dynamicSmemBytes = PairLayout<D>::SMEM;
        cudaLaunchAttribute attrs[1];
        attrs[0].id = cudaLaunchAttributeClusterDimension;
        attrs[0].val.clusterDim.x = 2;
        attrs[0].val.clusterDim.y = 1;
        attrs[0].val.clusterDim.z = 1;
        cfg.attrs = attrs;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, attn_persist_kernel<D>, &cfg) != cudaSuccess || n < 1) {
            (void)cudaGetLastError();
            n = sm_count() / 2;
        }
        clusters[dev] = n;
    }
    *n_out = clusters[dev];
    return FUSE_OK;
}

// Persistent 2-SM kernel: as many clusters as can be resident (at most one per tile pair).
template <int D>
int launch_persist(const void* q, const void* k, const void* v, const AttnArgs& args, cudaStream_t st) {
    int resident = 0;
    const int rc = persist_setup<D>(&resident);
    if (rc != FUSE_OK) return rc;
    const int64_t rows = static_cast<int64_t>(args.BH) * args.S;
    const int64_t items = rows / kAttnQ / 2;
    const int ncl = static_cast<int>(items < resident ? items : resident);
    CUtensorMap mQ, mKh, mV, mO;
    if (!make_map(&mQ, q, rows, D, 64, kAttnQ, true) || !make_map(&mKh, k, rows, D, 64, kAttnK / 2, true) ||
        !make_map(&mV, v, rows, D, 64, kAttnK, true) || !make_map(&mO, args.O, rows, D, 64, 32, true))
        return FUSE_ECUDA;
    static thread_local AttnSched sch;
    get_sched(args.BH, args.S / kAttnQ / 2, ncl, &sch);
    return launch_pdl(attn_persist_kernel<D>, dim3(2 * static_cast<unsigned>(ncl)), dim3(kPersistThreads),
                      PairLayout<D>::SMEM, st, 2, mQ, mKh, mV, mO, args, sch);
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
    // adjacent query tiles run as 2-SM pairs when they pair up and the head splits into two
    // halves of 64-wide swizzle atoms
    if constexpr (D >= 128) {
        if ((S / kAttnQ) % 2 == 0) return launch_persist<D>(q, k, v, args, st);
    }
    return launch_attn<D>(mQ, mK, mV, args, st);
}

bool overlap(const void* a, const void* b, int64_t bytes) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + static_cast<uintptr_t>(bytes) && y < x + static_cast<uintptr_t>(bytes);
}

}  // namespace

int attn_report_count() { return 1; }
int attn_report(int i, fuse_kernel_record* out) {
    if (i != 0) return FUSE_EINVAL;
    int resident = 0;
    const int rc = persist_setup<256>(&resident);
    if (rc != FUSE_OK) return rc;
    const int r2 = describe_kernel((const void*)attn_persist_kernel<256>,
                                   "attn_persist_kernel<D=256> (tcgen05 2-SM, M=256, persistent)",
                                   kPersistThreads, static_cast<int>(PairLayout<256>::SMEM), out,
                                   static_cast<int>(PairLayout<256>::TMEM_COLS));
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

extern "C" int64_t fuse_attention_schedule(int64_t bh, int64_t S, int clusters, int32_t* first,
                                           int32_t* items) {
    using namespace fc;
    if (bh < 1 || S < 2 * kAttnQ || S % (2 * kAttnQ) != 0 || clusters < 1 || !first || !items) return FUSE_EINVAL;
    const int64_t per_head = S / (2 * kAttnQ);
    if (clusters > kSchedClusters || bh * per_head > kSchedItems) return FUSE_EUNSUPPORTED;
    static thread_local AttnSched sch;
    build_sched(static_cast<int>(bh), static_cast<int>(per_head), clusters, &sch);
    if (sch.n == 0) return FUSE_EUNSUPPORTED;
    for (int c = 0; c <= clusters; ++c) first[c] = sch.first[c];
    for (int i = 0; i < sch.n; ++i) items[i] = sch.item[i];
    return sch.n;
}

extern "C" int64_t fuse_attention_flops(int64_t bh, int64_t S, int64_t D) {
    if (bh < 0 || S < 0 || D < 1) return FUSE_EINVAL;
    // Q K^T and P V over the visible (i, j <= i) pairs: 2 * 2 * D flops per pair
    return 4 * D * (S * (S + 1) / 2) * bh;
}
