// gemm.cu -- fp16 GEMM with the bias + GELU + residual epilogue applied from TMEM, under every cut
// plan of the four-stage chain mm -> +bias -> GELU -> +residual.
//
// [K4] §① prices this chain (chain_mlp_epilogue, fp16) under the cut plans [1,1,1,1], [1,3],
// [2,2] and [4]: every cut writes the intermediate (C, C', C'') back to HBM and reads it again;
// plan [4] reads A, B, bias and R once and writes Y once.  §⑥ adds the decode shape M = 16, where
// the GEMM is bound by reading the 4096 x 4096 weight.  [OFCG] §5.2 names the same fusion
// "epilogue fusion": the GEMM's output is written once, already in its final form.
//
// GB300 design.
//  * M > 64: one persistent CTA per SM, warp-specialised.  Warp 0 drives TMA (128B-swizzled
//    tiles, a 4-stage mbarrier ring); warp 1 owns TMEM and issues tcgen05.mma (M=128, N=256,
//    K=16, fp16 in, fp32 accumulate), committing each stage back to the producer and each
//    finished tile to the epilogue; warps 2-5 drain the accumulator with tcgen05.ld, 64 columns
//    at a time, add bias, apply GELU(erf), add the residual (brought in by TMA while the MMAs
//    run) and TMA-store fp16 Y.  The accumulator is double-buffered in TMEM (2 x 256 columns), so
//    the epilogue of tile i overlaps the main loop of tile i+1.  A is consumed K-major, B
//    ([K,N], N contiguous) MN-major, both straight from their row-major layouts.
//  * M <= 64 (decode): swap A and B so N fills the 128-row MMA dimension and M becomes the MMA's
//    N (16..64); split K across an 8-CTA cluster, reduce the eight fp32 partial tiles through
//    distributed shared memory (no global workspace) and apply the epilogue there.
//  * Cut plans: the GEMM kernel stops after the first stage segment and stores that fp16
//    intermediate; a vectorised tail kernel applies each later segment in place in Y.
//  * Every mbarrier wait is bounded; a wait that runs out raises the watchdog word, the CTA lets
//    its copies and MMAs in flight finish (bounded), frees its TMEM and returns.
#include <cudaTypedefs.h>
#include <math.h>

#include <mutex>

#include "fc_internal.cuh"
#include "fc_ptx.cuh"

namespace fc {
namespace {

// ------------------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int x, int y, uint32_t src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(src)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void prefetch_map(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t holder, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(holder), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// arrive (once) on `bar` when every tcgen05.mma issued so far by this thread has completed
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
        "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor (tcgen05): 128B swizzle, start/leading/stride in 16 B units.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo & 0x3FFFFu) >> 4) << 16;
    d |= static_cast<uint64_t>((sbo & 0x3FFFFu) >> 4) << 32;
    d |= static_cast<uint64_t>(1) << 46;  // descriptor version for tcgen05
    d |= static_cast<uint64_t>(2) << 61;  // SWIZZLE_128B
    return d;
}
// Instruction descriptor, kind::f16: fp16 A and B, fp32 D, dense.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool a_mn_major, bool b_mn_major) {
    return (1u << 4) | (static_cast<uint32_t>(a_mn_major) << 15) |
           (static_cast<uint32_t>(b_mn_major) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

// ------------------------------------------------------------------------------ epilogue math
// Stages of the chain after the GEMM: 1 = +bias, 2 = GELU(erf), 3 = +residual.
__device__ __forceinline__ float gelu_erf(float v) {
    return 0.5f * v * (1.0f + erff(v * 0.70710678118654752f));
}
// apply stages first..last (inclusive, 1..3) to v
__device__ __forceinline__ float apply_stages(float v, int first, int last, float b, float r) {
    if (first <= 1 && last >= 1) v += b;
    if (first <= 2 && last >= 2) v = gelu_erf(v);
    if (first <= 3 && last >= 3) v += r;
    return v;
}

__device__ __forceinline__ void unpack_h8(const uint4& u, float* f) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 t = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}
__device__ __forceinline__ uint4 pack_h8(const float* f) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __half2 h = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
        w[i] = *reinterpret_cast<uint32_t*>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// =============================================================================== main kernel
constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int kMainThreads = 192;              // 6 warps
constexpr uint32_t A_STAGE = BM * BK * 2;      // 16 KB
constexpr uint32_t B_BOX = 64 * BK * 2;        // 8 KB: 64 N x 64 K
constexpr uint32_t B_STAGE = BN * BK * 2;      // 32 KB
constexpr uint32_t E_BUF = 32 * 64 * 2;        // 4 KB: 32 rows x 64 cols
constexpr uint32_t OFF_A = 0;
constexpr uint32_t OFF_B = OFF_A + STAGES * A_STAGE;
constexpr uint32_t OFF_E = OFF_B + STAGES * B_STAGE;
constexpr uint32_t OFF_BAR = OFF_E + 4 * 2 * E_BUF;
// barriers: full[4], empty[4], acc_full[2], acc_empty[2], rbar[4][2], drain[1]
constexpr uint32_t N_BARS = STAGES * 2 + 2 + 2 + 8 + 1;
constexpr uint32_t OFF_HOLD = OFF_BAR + N_BARS * 8;
constexpr uint32_t MAIN_SMEM = OFF_HOLD + 16 + 1024;  // + alignment slack
constexpr uint32_t TMEM_COLS = 2 * BN;

struct MainArgs {
    int M, N, K;
    int tiles_m, tiles_n;
    int epi;             // last stage applied in this kernel: 0 (C), 1 (C'), 2 (C''), 3 (Y)
    const __half* bias;
    int* flag;
};

__device__ __forceinline__ void tile_coords(int t, int tiles_m, int& m0, int& n0) {
    m0 = (t % tiles_m) * BM;
    n0 = (t / tiles_m) * BN;
}

__global__ void __launch_bounds__(kMainThreads, 1) gemm_tc_kernel(
    const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
    const __grid_constant__ CUtensorMap mapR, const __grid_constant__ CUtensorMap mapY,
    const __grid_constant__ MainArgs args) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (smem_addr(smem_raw) + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - smem_addr(smem_raw));
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t bar0 = base + OFF_BAR;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto accf_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
    auto acce_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
    auto r_bar = [&](int ew, int j) { return bar0 + 8u * (2 * STAGES + 4 + 2 * ew + j); };
    const uint32_t drain_bar = bar0 + 8u * (N_BARS - 1);
    const uint32_t holder = base + OFF_HOLD;
    const int total_tiles = args.tiles_m * args.tiles_n;
    const int nk = (args.K + BK - 1) / BK;
    int* flag = args.flag;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf_bar(b), 1);
            mbar_init(acce_bar(b), 4);
        }
        for (int ew = 0; ew < 4; ++ew)
            for (int j = 0; j < 2; ++j) mbar_init(r_bar(ew, j), 1);
        mbar_init(drain_bar, 1);
        fence_mbar_init();
        prefetch_map(&mapA);
        prefetch_map(&mapB);
        prefetch_map(&mapR);
        prefetch_map(&mapY);
    }
    if (warp == 1) tmem_alloc(holder, TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(gbase + OFF_HOLD);

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        int stage = 0;
        uint32_t phase = 0, inflight = 0, issue_par = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
            int m0, n0;
            tile_coords(t, args.tiles_m, m0, n0);
            for (int kb = 0; kb < nk; ++kb) {
                if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, flag)) { ok = false; break; }
                inflight &= ~(1u << stage);  // its previous load was consumed
                if (lane == 0) {
                    mbar_arrive_expect_tx(full_bar(stage), A_STAGE + B_STAGE);
                    tma_load_2d(base + OFF_A + stage * A_STAGE, &mapA, kb * BK, m0, full_bar(stage));
#pragma unroll
                    for (int j = 0; j < BN / 64; ++j)
                        tma_load_2d(base + OFF_B + stage * B_STAGE + j * B_BOX, &mapB, n0 + 64 * j,
                                    kb * BK, full_bar(stage));
                }
                inflight |= 1u << stage;
                issue_par = (issue_par & ~(1u << stage)) | (phase << stage);
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
        }
        if (!ok) {  // let loads in flight land before this CTA can exit
            for (int s = 0; s < STAGES; ++s)
                if ((inflight >> s) & 1u) (void)mbar_wait_bounded(full_bar(s), (issue_par >> s) & 1u, flag, kWaitBudget / 8);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        constexpr uint32_t idesc = idesc_f16(BM, BN, false, true);
        int stage = 0, acc = 0;
        uint32_t phase = 0, acc_phase = 0;
        bool ok = true, issued = false;
        for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
            if (!mbar_wait_bounded(acce_bar(acc), acc_phase ^ 1u, flag)) { ok = false; break; }
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + acc * BN;
            for (int kb = 0; kb < nk; ++kb) {
                if (!mbar_wait_bounded(full_bar(stage), phase, flag)) { ok = false; break; }
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t a0 = base + OFF_A + stage * A_STAGE;
                    const uint32_t b0 = base + OFF_B + stage * B_STAGE;
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k) {
                        // A: K-major rows of 128 B, 8-row groups 1024 B apart; +32 B per K=16 step
                        const uint64_t ad = smem_desc_sw128(a0 + 32u * k, 16u, 1024u);
                        // B: MN-major, 64-wide N boxes 8 KB apart (LBO), 8-row K groups 1024 B
                        // apart (SBO); +16 rows (2048 B) per K=16 step
                        const uint64_t bd = smem_desc_sw128(b0 + 2048u * k, B_BOX, 1024u);
                        tc_mma(d_tmem, ad, bd, idesc, (kb > 0 || k > 0) ? 1u : 0u);
                    }
                    tc_commit(empty_bar(stage));  // frees the stage once these MMAs are done
                }
                issued = true;
                __syncwarp();
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
            if (!ok) break;
            if (lane == 0) tc_commit(accf_bar(acc));
            __syncwarp();
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
        if (!ok && issued) {  // MMAs in flight must finish before TMEM is freed
            if (lane == 0) tc_commit(drain_bar);
            __syncwarp();
            (void)mbar_wait_bounded(drain_bar, 0, flag, kWaitBudget / 8);
        }
    } else {
        // ------------------------------------------------------------ epilogue (warps 2-5)
        const int q = warp % 4;            // TMEM lane quadrant: rows 32q..32q+31 of the tile
        const int ew = warp - 2;           // index of this warp's buffers
        const uint32_t ebuf0 = base + OFF_E + ew * 2 * E_BUF;
        uint8_t* gebuf0 = gbase + OFF_E + ew * 2 * E_BUF;
        const bool need_r = args.epi >= 3;
        int acc = 0;
        uint32_t acc_phase = 0;
        int g = 0;  // chunk counter of this warp (4 per tile)
        bool ok = true;
        auto issue_r = [&](int gi, int t) {  // residual chunk gi (of tile t) -> buffer gi % 2
            int m0, n0;
            tile_coords(t, args.tiles_m, m0, n0);
            const int c = gi % 4;
            mbar_arrive_expect_tx(r_bar(ew, gi % 2), E_BUF);
            tma_load_2d(ebuf0 + (gi % 2) * E_BUF, &mapR, n0 + 64 * c, m0 + 32 * q, r_bar(ew, gi % 2));
        };
        uint32_t r_inflight = 0, r_par = 0;  // per buffer: a residual load in flight / its parity
        auto note_r = [&](int gi) {
            r_inflight |= 1u << (gi % 2);
            r_par = (r_par & ~(1u << (gi % 2))) | (static_cast<uint32_t>((gi / 2) & 1) << (gi % 2));
        };
        if (need_r && static_cast<int>(blockIdx.x) < total_tiles) {
            if (lane == 0) issue_r(0, blockIdx.x);
            note_r(0);
        }
        for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
            int m0, n0;
            tile_coords(t, args.tiles_m, m0, n0);
            if (!mbar_wait_bounded(accf_bar(acc), acc_phase, flag)) { ok = false; break; }
            tc_fence_after();
            for (int c = 0; c < BN / 64; ++c, ++g) {
                const int buf = g % 2;
                // next chunk's residual into the other buffer, once the store that last used it
                // has finished reading it
                const bool has_next = (c + 1 < BN / 64) || (t + static_cast<int>(gridDim.x) < total_tiles);
                if (lane == 0) bulk_wait_read0();
                __syncwarp();
                if (need_r && has_next) {
                    if (lane == 0) issue_r(g + 1, c + 1 < BN / 64 ? t : t + static_cast<int>(gridDim.x));
                    note_r(g + 1);
                }
                float v[64];
                const uint32_t tcol = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + acc * BN + 64 * c;
                tmem_ld32(tcol, v);
                tmem_ld32(tcol + 32, v + 32);
                tmem_ld_wait();
                if (c == BN / 64 - 1) {  // the accumulator buffer is drained: hand it back
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(acce_bar(acc));
                }
                if (need_r) {
                    if (!mbar_wait_bounded(r_bar(ew, buf), (g / 2) & 1, flag)) { ok = false; break; }
                    r_inflight &= ~(1u << buf);
                }
                // row `lane` of this warp's 32 rows; its 64 columns are 8 swizzled 16 B chunks
                uint8_t* rowp = gebuf0 + buf * E_BUF + lane * 128;
                const int ncol0 = n0 + 64 * c;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    float bv[8] = {0, 0, 0, 0, 0, 0, 0, 0};
                    if (args.epi >= 1 && ncol0 + 8 * j < args.N)
                        unpack_h8(__ldg(reinterpret_cast<const uint4*>(args.bias + ncol0 + 8 * j)), bv);
                    uint4* chunk = reinterpret_cast<uint4*>(rowp + 16 * (j ^ (lane & 7)));
                    float rv[8] = {0, 0, 0, 0, 0, 0, 0, 0};
                    if (need_r) unpack_h8(*chunk, rv);
                    float o[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) o[e] = apply_stages(v[8 * j + e], 1, args.epi, bv[e], rv[e]);
                    *chunk = pack_h8(o);
                }
                fence_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(&mapY, ncol0, m0 + 32 * q, ebuf0 + buf * E_BUF);
                    bulk_commit();
                }
            }
            if (!ok) break;
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
        if (lane == 0) bulk_wait0();
        if (!ok) {
            for (int j = 0; j < 2; ++j)
                if ((r_inflight >> j) & 1u)
                    (void)mbar_wait_bounded(r_bar(ew, j), (r_par >> j) & 1u, flag, kWaitBudget / 8);
        }
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, TMEM_COLS);
}

// =============================================================================== decode kernel
// Y^T[N, M] = B^T[N, K] A^T[K, M] for M <= 64: MMA M = 128 rows of N, MMA N = NM >= M.
constexpr int DEC_SPLIT = 8;    // K split = cluster size
constexpr int DEC_STAGES = 4;
constexpr int kDecThreads = 128;
constexpr uint32_t DEC_BT_STAGE = 128 * BK * 2;  // 16 KB: two 64-wide N boxes

struct DecodeArgs {
    int M, N, K;
    int kb_per_split;   // k-blocks of 64 per CTA
    int epi;
    const __half* bias;
    const __half* R;
    __half* Y;
    int* flag;
};

template <int NM>
struct DecodeLayout {
    static constexpr uint32_t A_ST = NM * BK * 2;
    static constexpr uint32_t OFF_BT = 0;
    static constexpr uint32_t OFF_AS = OFF_BT + DEC_STAGES * DEC_BT_STAGE;
    static constexpr uint32_t OFF_P = OFF_AS + DEC_STAGES * A_ST;       // fp32 partial [NM][128]
    static constexpr uint32_t OFF_BAR = OFF_P + NM * 128 * 4;
    static constexpr uint32_t N_BARS = 2 * DEC_STAGES + 2;           // full, empty, acc, drain
    static constexpr uint32_t OFF_HOLD = OFF_BAR + N_BARS * 8;
    static constexpr uint32_t SMEM = OFF_HOLD + 16 + 1024;
    static constexpr uint32_t TCOLS = NM <= 32 ? 32 : 64;
};

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ float ld_dsmem_f32(uint32_t local_addr, uint32_t rank) {
    uint32_t remote;
    float v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

template <int NM>
__global__ void __launch_bounds__(kDecThreads) gemm_decode_kernel(
    const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
    const __grid_constant__ DecodeArgs args) {
    using L = DecodeLayout<NM>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (smem_addr(smem_raw) + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - smem_addr(smem_raw));
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t rank = cluster_rank();                  // K split index
    const int n0 = (blockIdx.x / DEC_SPLIT) * 128;          // 128 output columns of Y
    const int kb0 = static_cast<int>(rank) * args.kb_per_split;
    const int nk_all = (args.K + BK - 1) / BK;
    const int nk = max(0, min(args.kb_per_split, nk_all - kb0));
    const uint32_t bar0 = base + L::OFF_BAR;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (DEC_STAGES + s); };
    const uint32_t acc_bar = bar0 + 8u * (2 * DEC_STAGES);
    const uint32_t drain_bar = acc_bar + 8u;
    const uint32_t holder = base + L::OFF_HOLD;
    float* part = reinterpret_cast<float*>(gbase + L::OFF_P);  // [NM][128]
    int* flag = args.flag;

    if (threadIdx.x == 0) {
        for (int s = 0; s < DEC_STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        mbar_init(acc_bar, 1);
        mbar_init(drain_bar, 1);
        fence_mbar_init();
        prefetch_map(&mapA);
        prefetch_map(&mapB);
    }
    if (warp == 1) tmem_alloc(holder, L::TCOLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(gbase + L::OFF_HOLD);
    bool ok = true;

    if (warp == 0) {
        uint32_t inflight = 0, issue_par = 0, phase = 0;
        int stage = 0;
        for (int kb = 0; kb < nk; ++kb) {
            if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, flag)) { ok = false; break; }
            inflight &= ~(1u << stage);
            if (lane == 0) {
                mbar_arrive_expect_tx(full_bar(stage), DEC_BT_STAGE + L::A_ST);
                const int k = (kb0 + kb) * BK;
                tma_load_2d(base + L::OFF_BT + stage * DEC_BT_STAGE, &mapB, n0, k, full_bar(stage));
                tma_load_2d(base + L::OFF_BT + stage * DEC_BT_STAGE + B_BOX, &mapB, n0 + 64, k, full_bar(stage));
                tma_load_2d(base + L::OFF_AS + stage * L::A_ST, &mapA, k, 0, full_bar(stage));
            }
            inflight |= 1u << stage;
            issue_par = (issue_par & ~(1u << stage)) | (phase << stage);
            if (++stage == DEC_STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok)
            for (int s = 0; s < DEC_STAGES; ++s)
                if ((inflight >> s) & 1u) (void)mbar_wait_bounded(full_bar(s), (issue_par >> s) & 1u, flag, kWaitBudget / 8);
    } else if (warp == 1) {
        constexpr uint32_t idesc = idesc_f16(128, NM, true, false);
        uint32_t phase = 0;
        int stage = 0;
        bool issued = false;
        for (int kb = 0; kb < nk; ++kb) {
            if (!mbar_wait_bounded(full_bar(stage), phase, flag)) { ok = false; break; }
            tc_fence_after();
            if (lane == 0) {
                const uint32_t bt0 = base + L::OFF_BT + stage * DEC_BT_STAGE;
                const uint32_t a0 = base + L::OFF_AS + stage * L::A_ST;
#pragma unroll
                for (int k = 0; k < BK / 16; ++k) {
                    // MMA A = B^T tile: MN-major (N contiguous), N boxes of 64 are 8 KB apart
                    const uint64_t ad = smem_desc_sw128(bt0 + 2048u * k, B_BOX, 1024u);
                    // MMA B = A rows: K-major, NM rows of 128 B
                    const uint64_t bd = smem_desc_sw128(a0 + 32u * k, 16u, 1024u);
                    tc_mma(tmem_base, ad, bd, idesc, (kb > 0 || k > 0) ? 1u : 0u);
                }
                tc_commit(empty_bar(stage));
            }
            issued = true;
            __syncwarp();
            if (++stage == DEC_STAGES) { stage = 0; phase ^= 1u; }
        }
        if (ok) {
            if (lane == 0) tc_commit(acc_bar);
            __syncwarp();
        } else if (issued) {
            if (lane == 0) tc_commit(drain_bar);
            __syncwarp();
            (void)mbar_wait_bounded(drain_bar, 0, flag, kWaitBudget / 8);
        }
    }
    // all four warps: accumulator (TMEM lane = output column n0 + 32*warp + lane) -> smem partial
    {
        const bool have = nk > 0;
        bool got = true;
        if (have) got = mbar_wait_bounded(acc_bar, 0, flag);
        tc_fence_after();
        float v[NM];
        if (have && got) {
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * warp) << 16);
#pragma unroll
            for (int c = 0; c < NM; c += 16) tmem_ld16(taddr + c, v + c);
            tmem_ld_wait();
        } else {
#pragma unroll
            for (int c = 0; c < NM; ++c) v[c] = 0.0f;
        }
#pragma unroll
        for (int c = 0; c < NM; ++c) part[c * 128 + 32 * warp + lane] = v[c];
    }
    tc_fence_before();
    cluster_sync();  // every CTA of the cluster has its partial in shared memory

    // CTA `rank` reduces output columns [n0 + 16*rank, n0 + 16*rank + 16) for all NM rows
    {
        constexpr int COLS = 128 / DEC_SPLIT;  // 16
        const uint32_t part_addr = smem_addr(part);
        for (int idx = threadIdx.x; idx < COLS * NM; idx += kDecThreads) {
            const int m = idx / COLS;
            const int nl = static_cast<int>(rank) * COLS + idx % COLS;
            float s = 0.0f;
#pragma unroll
            for (int r = 0; r < DEC_SPLIT; ++r)
                s += ld_dsmem_f32(part_addr + 4u * (m * 128 + nl), static_cast<uint32_t>(r));
            const int n = n0 + nl;
            if (m < args.M && n < args.N) {
                const float b = args.epi >= 1 ? __half2float(args.bias[n]) : 0.0f;
                const float rr = args.epi >= 3 ? __half2float(args.R[static_cast<int64_t>(m) * args.N + n]) : 0.0f;
                args.Y[static_cast<int64_t>(m) * args.N + n] = __float2half_rn(apply_stages(s, 1, args.epi, b, rr));
            }
        }
    }
    cluster_sync();  // no CTA leaves while another still reads its partial
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, L::TCOLS);
}

// =============================================================================== tail kernel
// Y <- h(stages first..last applied to Y), 8 halves per thread (N % 8 == 0).
__global__ void __launch_bounds__(256) epi_tail_kernel(__half* __restrict__ Y, const __half* __restrict__ bias,
                                                       const __half* __restrict__ R, int64_t M, int N,
                                                       int first, int last) {
    const int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t total = M * N / 8;
    if (g >= total) return;
    const int n = static_cast<int>((g * 8) % N);
    float v[8], bv[8] = {0, 0, 0, 0, 0, 0, 0, 0}, rv[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    uint4* yp = reinterpret_cast<uint4*>(Y) + g;
    unpack_h8(*yp, v);
    if (first <= 1 && last >= 1) unpack_h8(__ldg(reinterpret_cast<const uint4*>(bias + n)), bv);
    if (last >= 3) unpack_h8(__ldcs(reinterpret_cast<const uint4*>(R) + g), rv);
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = apply_stages(v[e], first, last, bv[e], rv[e]);
    *yp = pack_h8(v);
}

// =============================================================================== host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::mutex mu;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            (void)cudaGetLastError();
    }
    return fn;
}

// 2-D fp16 tensor [rows, cols] row-major, box [box_rows, box_cols], 128B swizzle
bool make_map(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols, int box_cols, int box_rows) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
                     estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool overlap(const void* a, int64_t abytes, const void* b, int64_t bbytes) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + static_cast<uintptr_t>(bbytes) && y < x + static_cast<uintptr_t>(abytes);
}

template <int NM>
int launch_decode(const CUtensorMap& mA, const CUtensorMap& mB, const DecodeArgs& a, cudaStream_t st) {
    using L = DecodeLayout<NM>;
    static const bool attr = cudaFuncSetAttribute(gemm_decode_kernel<NM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                  static_cast<int>(L::SMEM)) == cudaSuccess;
    if (!attr) return check_launch();
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ceil_div(a.N, 128) * DEC_SPLIT));
    cfg.blockDim = dim3(kDecThreads);
    cfg.dynamicSmemBytes = L::SMEM;
    cfg.stream = st;
    cudaLaunchAttribute attrs[1];
    attrs[0].id = cudaLaunchAttributeClusterDimension;
    attrs[0].val.clusterDim.x = DEC_SPLIT;
    attrs[0].val.clusterDim.y = 1;
    attrs[0].val.clusterDim.z = 1;
    cfg.attrs = attrs;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_decode_kernel<NM>, mA, mB, a);
    if (e != cudaSuccess) return record_cuda_error(e);
    return check_launch();
}

// GEMM + the stages 1..epi, fp16 result into Y
int launch_gemm(const void* A, const void* B, const void* bias, const void* R, void* Y, int64_t M,
                int64_t N, int64_t K, int epi, cudaStream_t st) {
    int* flag = watchdog_flag();
    if (!flag) return FUSE_ECUDA;
    CUtensorMap mA, mB;
    if (M <= 64) {
        const int NM = M <= 16 ? 16 : (M <= 32 ? 32 : 64);
        if (!make_map(&mA, A, M, K, 64, NM) || !make_map(&mB, B, K, N, 64, 64)) return FUSE_ECUDA;
        DecodeArgs a;
        a.M = static_cast<int>(M);
        a.N = static_cast<int>(N);
        a.K = static_cast<int>(K);
        const int nk = static_cast<int>(ceil_div(K, BK));
        a.kb_per_split = static_cast<int>(ceil_div(nk, DEC_SPLIT));
        a.epi = epi;
        a.bias = static_cast<const __half*>(bias);
        a.R = static_cast<const __half*>(R);
        a.Y = static_cast<__half*>(Y);
        a.flag = flag;
        if (NM == 16) return launch_decode<16>(mA, mB, a, st);
        if (NM == 32) return launch_decode<32>(mA, mB, a, st);
        return launch_decode<64>(mA, mB, a, st);
    }
    CUtensorMap mR, mY;
    if (!make_map(&mA, A, M, K, 64, BM) || !make_map(&mB, B, K, N, 64, 64) ||
        !make_map(&mR, epi >= 3 ? R : Y, M, N, 64, 32) || !make_map(&mY, Y, M, N, 64, 32))
        return FUSE_ECUDA;
    static const bool attr = cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                  static_cast<int>(MAIN_SMEM)) == cudaSuccess;
    if (!attr) return check_launch();
    MainArgs a;
    a.M = static_cast<int>(M);
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    a.tiles_m = static_cast<int>(ceil_div(M, BM));
    a.tiles_n = static_cast<int>(ceil_div(N, BN));
    a.epi = epi;
    a.bias = static_cast<const __half*>(bias);
    a.flag = flag;
    const int tiles = a.tiles_m * a.tiles_n;
    const int grid = tiles < sm_count() ? tiles : sm_count();
    gemm_tc_kernel<<<grid, kMainThreads, MAIN_SMEM, st>>>(mA, mB, mR, mY, a);
    return check_launch();
}

int launch_tail(void* Y, const void* bias, const void* R, int64_t M, int64_t N, int first, int last,
                cudaStream_t st) {
    const int64_t units = M * N / 8;
    epi_tail_kernel<<<static_cast<unsigned>(ceil_div(units, 256)), 256, 0, st>>>(
        static_cast<__half*>(Y), static_cast<const __half*>(bias), static_cast<const __half*>(R), M,
        static_cast<int>(N), first, last);
    return check_launch();
}

}  // namespace

int gemm_report_count() { return 3; }
int gemm_report(int i, fuse_kernel_record* out) {
    switch (i) {
        case 0: return describe_kernel((const void*)gemm_tc_kernel, "gemm_tc_kernel (128x256 tcgen05)",
                                       kMainThreads, static_cast<int>(MAIN_SMEM), out);
        case 1: return describe_kernel((const void*)gemm_decode_kernel<16>,
                                       "gemm_decode_kernel<16> (swap-AB, split-K x8)", kDecThreads,
                                       static_cast<int>(DecodeLayout<16>::SMEM), out);
        case 2: return describe_kernel((const void*)epi_tail_kernel, "epi_tail_kernel (unfused plans)", 256, 0, out);
        default: return FUSE_EINVAL;
    }
}

}  // namespace fc

extern "C" int fuse_gemm_epilogue_plan(const void* A, const void* B, const void* bias, const void* R,
                                       void* Y, int64_t M, int64_t N, int64_t Kdim, uint32_t cut_mask,
                                       fuse_stream_t stream) {
    using namespace fc;
    if (M < 0 || N < 0 || Kdim < 0 || cut_mask > 7u) return FUSE_EINVAL;
    if (M == 0 || N == 0) return FUSE_OK;
    if (Kdim == 0) return FUSE_EUNSUPPORTED;
    if (!A || !B || !bias || !R || !Y) return FUSE_EINVAL;
    if (N % 8 != 0 || Kdim % 8 != 0) return FUSE_EALIGN;  // 16-byte row strides for TMA
    if (!is_aligned(A, 16) || !is_aligned(B, 16) || !is_aligned(bias, 16) || !is_aligned(R, 16) ||
        !is_aligned(Y, 16))
        return FUSE_EALIGN;
    if (M > 2147483647LL || N > 2147483647LL || Kdim > 2147483647LL) return FUSE_EUNSUPPORTED;
    const int64_t ybytes = M * N * 2;
    if (overlap(Y, ybytes, A, M * Kdim * 2) || overlap(Y, ybytes, B, Kdim * N * 2) ||
        overlap(Y, ybytes, bias, N * 2) || overlap(Y, ybytes, R, M * N * 2))
        return FUSE_EINVAL;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // segments of the chain (stage 0 = mm, 1 = bias, 2 = gelu, 3 = residual)
    int first = 0;
    while (first < 4) {
        int last = first;
        while (last < 3 && !((cut_mask >> last) & 1u)) ++last;
        const int rc = first == 0 ? launch_gemm(A, B, bias, R, Y, M, N, Kdim, last, st)
                                  : launch_tail(Y, bias, R, M, N, first, last, st);
        if (rc != FUSE_OK) return rc;
        first = last + 1;
    }
    return FUSE_OK;
}

extern "C" int fuse_gemm_epilogue(const void* A, const void* B, const void* bias, const void* R, void* Y,
                                  int64_t M, int64_t N, int64_t Kdim, fuse_stream_t stream) {
    return fuse_gemm_epilogue_plan(A, B, bias, R, Y, M, N, Kdim, 0u, stream);
}

extern "C" int64_t fuse_gemm_bytes(int64_t M, int64_t N, int64_t Kdim, uint32_t cut_mask) {
    if (M < 0 || N < 0 || Kdim < 0 || cut_mask > 7u) return FUSE_EINVAL;
    // [K4] §① traffic: A, B, bias and R are read once in any plan, Y written once; every cut adds
    // one write and one read of an M x N fp16 intermediate.
    const int cuts = static_cast<int>((cut_mask & 1u) + ((cut_mask >> 1) & 1u) + ((cut_mask >> 2) & 1u));
    return 2 * (M * Kdim + Kdim * N + N + M * N + M * N + 2 * static_cast<int64_t>(cuts) * M * N);
}
