// gemm_decode.cu -- the GEMM chain mm -> +bias -> GELU -> +residual for a few rows (M <= 64, the
// decode shape of [K4] §⑥: M = 16 against a 4096 x 4096 fp16 weight), where reading the weight
// once bounds the time.
//
// GB300 design: swap A and B so the weight's N fills the 128-row MMA dimension and M becomes the
// MMA's N (16, 32 or 64); split K over an 8-CTA cluster (256 CTAs for N = 4096, one wave at two
// CTAs per SM); every CTA streams its 128-column x K/8 slab of the weight through a 5-stage TMA
// ring (M <= 16) into tcgen05 MMAs (fp32 accumulator in TMEM), then sends each of the eight column
// slices of its partial to the CTA that owns that slice (st.async into the owner's shared memory,
// completion on its mbarrier).  The owner sums the eight partials in rank order and applies the
// epilogue: no global workspace, no cluster barrier after the main loop.  In a stream of decode
// calls the time goes to waiting for the preceding call (its grid completing releases this one
// ~1.7 us after its last CTA ends), the weight stream and the exchange; so nothing but the TMA
// issue sits between the grid-dependency wait and the first load (the epilogue's bias and
// residual loads belong to the warps idle during the main loop), and with FUSE_GEMM_STATIC_B the
// first ring of weight boxes is already on its way before that wait.  Every mbarrier wait is
// bounded (watchdog).
#include <cudaTypedefs.h>
#include <math.h>

#include "fc_internal.cuh"
#include "fc_ptx.cuh"
#include "fc_tc.cuh"
#include "gemm_epi.cuh"

namespace fc {
namespace {

constexpr int BK = 64;                          // K per pipeline stage
constexpr uint32_t B_BOX = 64 * BK * 2;         // 8 KB: one 64 N x 64 K box of the weight

// =============================================================================== decode kernel
// Y^T[N, M] = B^T[N, K] A^T[K, M] for M <= 64: MMA M = 128 rows of N, MMA N = NM >= M.
constexpr int DEC_SPLIT = 8;    // K split = cluster size
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
    int b_static;       // 1: B is not written by the work queued before this call (see below)
};

template <int NM>
struct DecodeLayout {
    // 5 x 18 KB for M <= 16 keeps two CTAs per SM (2 x 100 KB), so the whole grid is resident
    static constexpr int STAGES = NM <= 16 ? 5 : (NM <= 32 ? 4 : 3);
    static constexpr uint32_t A_ST = NM * BK * 2;
    static constexpr uint32_t OFF_BT = 0;
    static constexpr uint32_t OFF_AS = OFF_BT + STAGES * DEC_BT_STAGE;
    // fp32 partials received from every CTA of the cluster for this CTA's column slice:
    // [source rank][slice column][output row], DEC_SPLIT x (128 / DEC_SPLIT) x NM
    static constexpr uint32_t OFF_P = OFF_AS + STAGES * A_ST;
    static constexpr uint32_t OFF_BAR = OFF_P + NM * 128 * 4;
    static constexpr uint32_t N_BARS = 2 * STAGES + 3;               // full, empty, acc, drain, recv
    static constexpr uint32_t OFF_HOLD = OFF_BAR + N_BARS * 8;
    static constexpr uint32_t SMEM = OFF_HOLD + 16 + 1024;
    static constexpr uint32_t TCOLS = NM <= 32 ? 32 : 64;
};

// Store four floats into the shared memory of a CTA of the cluster (`remote` and `remote_bar` are
// shared::cluster addresses); the bytes count toward that CTA's mbarrier transaction.
__device__ __forceinline__ void st_async_v4(uint32_t remote, float a, float b, float c, float d,
                                            uint32_t remote_bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];"
                 ::"r"(remote), "f"(a), "f"(b), "f"(c), "f"(d), "r"(remote_bar)
                 : "memory");
}
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

template <int NM>
__global__ void __launch_bounds__(kDecThreads) gemm_decode_kernel(
    const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
    const __grid_constant__ DecodeArgs args) {
    pdl_trigger();  // the set-up below touches no global memory; pdl_wait() follows it
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
    auto empty_bar = [&](int s) { return bar0 + 8u * (L::STAGES + s); };
    const uint32_t acc_bar = bar0 + 8u * (2 * L::STAGES);
    const uint32_t drain_bar = acc_bar + 8u;
    const uint32_t recv_bar = drain_bar + 8u;
    const uint32_t holder = base + L::OFF_HOLD;
    const float* recv = reinterpret_cast<const float*>(gbase + L::OFF_P);  // [DEC_SPLIT][COLS][NM]
    int* flag = args.flag;

    if (threadIdx.x == 0) {
        for (int s = 0; s < L::STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        mbar_init(acc_bar, 1);
        mbar_init(drain_bar, 1);
        mbar_init(recv_bar, 1);
        fence_mbar_init();
        // every CTA of the cluster sends this CTA one slice of its partial (NM x COLS fp32)
        mbar_arrive_expect_tx(recv_bar, static_cast<uint32_t>(128 * NM * 4));
        prefetch_map(&mapA);
        prefetch_map(&mapB);
        if (args.b_static) {
            // The caller vouches that nothing queued before this call writes B: the first ring of
            // weight boxes is loaded now, while the preceding kernel may still run (A, which it may
            // have written, follows after the grid-dependency wait; each stage's barrier expects
            // both, so no MMA starts before A is current).
            for (int kb = 0; kb < nk && kb < L::STAGES; ++kb) {
                const int k = (kb0 + kb) * BK;
                mbar_arrive_expect_tx(full_bar(kb), DEC_BT_STAGE + L::A_ST);
                tma_load_2d(base + L::OFF_BT + kb * DEC_BT_STAGE, &mapB, n0, k, full_bar(kb));
                tma_load_2d(base + L::OFF_BT + kb * DEC_BT_STAGE + B_BOX, &mapB, n0 + 64, k, full_bar(kb));
            }
        } else {
            // Start this CTA's whole weight slice on its way into L2 while the preceding kernel
            // may still run: an L2 prefetch returns nothing to the SM, and L2 is where that
            // kernel's writes land, so the loads after pdl_wait() read current data, only sooner.
            for (int kb = 0; kb < nk; ++kb) {
                const int k = (kb0 + kb) * BK;
                tma_prefetch_2d(&mapB, n0, k);
                tma_prefetch_2d(&mapB, n0 + 64, k);
                tma_prefetch_2d(&mapA, k, 0);
            }
        }
    }
    if (warp == 1) tmem_alloc(holder, L::TCOLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // Peers may send into this CTA's shared memory only once its receive barrier exists: the
    // cluster barrier is arrived at here and waited on just before the first send, so the wait
    // overlaps the main loop.  Every thread reaches both on every path.
    cluster_arrive();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(gbase + L::OFF_HOLD);
    bool ok = true;
    pdl_wait();  // the preceding kernel has completed: global memory may be touched

    // After the K reduction CTA `rank` finishes output columns [n0 + COLS*rank, +COLS) of all NM
    // rows, in units of one column and four consecutive rows: unit idx = uthread + kDecThreads*u
    // is slice column idx / (NM/4), rows 4*(idx % (NM/4)) .. +3.  Units go to warps 2 and 3 first
    // (uthread = threadIdx.x ^ 64), which have nothing to do during the main loop and load the
    // bias and residual values of their units now, so that latency hides under it; the TMA and
    // MMA warps (0 and 1) hold units only when there are more than 64 (M > 16) and load theirs
    // after their loops, so no global load delays the first TMA issue or the first MMA.
    constexpr int COLS = 128 / DEC_SPLIT;  // 16
    constexpr int UNITS = NM * COLS / 4;
    constexpr int UPT = (UNITS + kDecThreads - 1) / kDecThreads;
    const int uthread = static_cast<int>(threadIdx.x) ^ 64;
    float eb[UPT], er[UPT][4];
    auto load_units = [&]() {
#pragma unroll
        for (int u = 0; u < UPT; ++u) {
            const int idx = uthread + kDecThreads * u;
            const int n = n0 + COLS * static_cast<int>(rank) + idx / (NM / 4);
            const int m0 = 4 * (idx % (NM / 4));
            const bool valid = idx < UNITS && n < args.N;
            eb[u] = valid && args.epi >= 1 ? __half2float(__ldg(args.bias + n)) : 0.0f;
#pragma unroll
            for (int i = 0; i < 4; ++i)
                er[u][i] = valid && args.epi >= 3 && m0 + i < args.M
                               ? __half2float(__ldcs(args.R + static_cast<int64_t>(m0 + i) * args.N + n))
                               : 0.0f;
        }
    };
    if (warp >= 2) load_units();

    if (warp == 0) {
        uint32_t inflight = 0, issue_par = 0, phase = 0;
        int stage = 0;
        for (int kb = 0; kb < nk; ++kb) {
            // stages whose weight boxes went out before the grid-dependency wait only need A (their
            // barriers are fresh, so there is nothing to wait for, and the loop cannot stop before
            // every such stage has its A: each of their barriers completes)
            const bool early = args.b_static && kb < L::STAGES;
            if (!early && !mbar_wait_bounded(empty_bar(stage), phase ^ 1u, flag)) { ok = false; break; }
            inflight &= ~(1u << stage);
            if (lane == 0) {
                const int k = (kb0 + kb) * BK;
                if (!early) {
                    mbar_arrive_expect_tx(full_bar(stage), DEC_BT_STAGE + L::A_ST);
                    tma_load_2d(base + L::OFF_BT + stage * DEC_BT_STAGE, &mapB, n0, k, full_bar(stage));
                    tma_load_2d(base + L::OFF_BT + stage * DEC_BT_STAGE + B_BOX, &mapB, n0 + 64, k, full_bar(stage));
                }
                tma_load_2d(base + L::OFF_AS + stage * L::A_ST, &mapA, k, 0, full_bar(stage));
            }
            inflight |= 1u << stage;
            issue_par = (issue_par & ~(1u << stage)) | (phase << stage);
            if (++stage == L::STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok)
            for (int s = 0; s < L::STAGES; ++s)
                if ((inflight >> s) & 1u) (void)mbar_wait_drain(full_bar(s), (issue_par >> s) & 1u);
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
            if (++stage == L::STAGES) { stage = 0; phase ^= 1u; }
        }
        if (ok) {
            if (lane == 0) tc_commit(acc_bar);
            __syncwarp();
        } else if (issued) {
            if (lane == 0) tc_commit(drain_bar);
            __syncwarp();
            (void)mbar_wait_drain(drain_bar, 0);
        }
    }
    if (warp < 2) load_units();
    // All four warps: thread (warp, lane) holds output column n0 + 32*warp + lane of this CTA's
    // partial (its TMEM lane) for all NM rows and sends it to the CTA that owns that column's slice,
    // into row `rank` of that CTA's receive buffer.
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
            for (int c = 0; c < NM; ++c) v[c] = 0.0f;   // after a failed wait: zeros, still sent
        }
        const int col = 32 * warp + lane;
        const uint32_t owner = static_cast<uint32_t>(col / COLS);
        const uint32_t dst = mapa_shared(
            smem_addr(recv) + 4u * static_cast<uint32_t>((static_cast<int>(rank) * COLS + col % COLS) * NM), owner);
        const uint32_t dst_bar = mapa_shared(recv_bar, owner);
        cluster_wait();   // every CTA of the cluster has initialised its receive barrier
#pragma unroll
        for (int c = 0; c < NM; c += 4) st_async_v4(dst + 4u * c, v[c], v[c + 1], v[c + 2], v[c + 3], dst_bar);
    }

    // This CTA's slice: the DEC_SPLIT partials summed in rank order, then the epilogue.  If the
    // wait gives up (another wait of the launch failed), the peers still send their slices on every
    // path: wait for them without the flag (bounded) so none lands after this CTA has exited.
    const bool received = mbar_wait_bounded(recv_bar, 0, flag);
    if (!received) (void)mbar_wait_drain(recv_bar, 0, kWaitBudget);
    if (received) {
#pragma unroll
        for (int u = 0; u < UPT; ++u) {
            const int idx = uthread + kDecThreads * u;
            if (idx >= UNITS) break;
            const int c = idx / (NM / 4);
            const int m0 = 4 * (idx % (NM / 4));
            float4 sum = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
            for (int r = 0; r < DEC_SPLIT; ++r) {
                const float4 p = *reinterpret_cast<const float4*>(recv + (r * COLS + c) * NM + m0);
                sum.x += p.x;
                sum.y += p.y;
                sum.z += p.z;
                sum.w += p.w;
            }
            const int n = n0 + COLS * static_cast<int>(rank) + c;
            if (n < args.N) {
                const float2 lo = apply_stages2(make_float2(sum.x, sum.y), 1, args.epi, make_float2(eb[u], eb[u]),
                                                make_float2(er[u][0], er[u][1]));
                const float2 hi = apply_stages2(make_float2(sum.z, sum.w), 1, args.epi, make_float2(eb[u], eb[u]),
                                                make_float2(er[u][2], er[u][3]));
                const float o[4] = {lo.x, lo.y, hi.x, hi.y};
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (m0 + i < args.M) args.Y[static_cast<int64_t>(m0 + i) * args.N + n] = __float2half_rn(o[i]);
            }
        }
    }
    // TMEM is freed once every thread's reads of it have completed.  No cluster barrier: a CTA's
    // shared memory is written by its peers only until its own receive barrier completes.
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, L::TCOLS);
}

template <int NM>
int launch_decode(const CUtensorMap& mA, const CUtensorMap& mB, const DecodeArgs& a, cudaStream_t st) {
    using L = DecodeLayout<NM>;
    // all of an SM's shared memory as shared (not L1) lets two decode CTAs share an SM, so the
    // whole grid (ceil(N/128) x 8 CTAs) is resident in one wave (CTA start stamps: the 256 CTAs
    // of N = 4096 start within ~1.2 us, two per SM on 148 SMs; the occupancy API, which reports
    // one CTA per SM for kernels that allocate tensor memory, undercounts)
    const int rc = opt_in_smem((const void*)gemm_decode_kernel<NM>, static_cast<int>(L::SMEM), true);
    if (rc != FUSE_OK) return rc;
    return launch_pdl(gemm_decode_kernel<NM>, dim3(static_cast<unsigned>(ceil_div(a.N, 128) * DEC_SPLIT)), dim3(kDecThreads), L::SMEM, st, DEC_SPLIT, mA, mB, a);
}

// Clusters of the decode kernel that can be resident at once (0 if the query fails).
template <int NM>
int decode_max_active_clusters() {
    using L = DecodeLayout<NM>;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(DEC_SPLIT * 32));
    cfg.blockDim = dim3(kDecThreads);
    cfg.dynamicSmemBytes = L::SMEM;
    cudaLaunchAttribute attrs[1];
    attrs[0].id = cudaLaunchAttributeClusterDimension;
    attrs[0].val.clusterDim.x = DEC_SPLIT;
    attrs[0].val.clusterDim.y = 1;
    attrs[0].val.clusterDim.z = 1;
    cfg.attrs = attrs;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_decode_kernel<NM>, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

}  // namespace

// Y = stages 1..epi of the chain applied to A @ B, for M <= 64 (FUSE_OK or an error status).
int launch_decode_gemm(const void* A, const void* B, const void* bias, const void* R, void* Y, int64_t M,
                       int64_t N, int64_t K, int epi, bool b_static, cudaStream_t st) {
    int* flag = watchdog_flag();
    if (!flag) return FUSE_ECUDA;
    CUtensorMap mA, mB;
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
    a.b_static = b_static ? 1 : 0;
    if (NM == 16) return launch_decode<16>(mA, mB, a, st);
    if (NM == 32) return launch_decode<32>(mA, mB, a, st);
    return launch_decode<64>(mA, mB, a, st);
}

// Kernel record of the M = 16 decode kernel.
int decode_report(fuse_kernel_record* out) {
    // the launch configuration's attributes, as a launch sets them (shared-memory carveout included)
    if (const int ra = opt_in_smem((const void*)gemm_decode_kernel<16>, static_cast<int>(DecodeLayout<16>::SMEM), true);
        ra != FUSE_OK)
        return ra;
    const int rc = describe_kernel((const void*)gemm_decode_kernel<16>,
                                   "gemm_decode_kernel<16> (swap-AB, split-K x8)", kDecThreads,
                                   static_cast<int>(DecodeLayout<16>::SMEM), out,
                                   static_cast<int>(DecodeLayout<16>::TCOLS));
    if (rc == FUSE_OK) {
        out->cluster_size = DEC_SPLIT;
        out->max_active_clusters = decode_max_active_clusters<16>();
    }
    return rc;
}

}  // namespace fc
