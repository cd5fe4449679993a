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
//  * M > 64: persistent 2-CTA clusters, one CTA per SM, warp-specialised.  The two CTAs of a
//    cluster act as one MMA unit (tcgen05 .cta_group::2): each holds its own 128 rows of A and one
//    half (128 columns) of the B tile per stage, and the even CTA issues M = 256, N = 256, K = 16
//    MMAs (fp16 in, fp32 accumulate) whose rows 0-127 accumulate in its TMEM and rows 128-255 in
//    its peer's.  Warp 0 drives TMA (128B-swizzled tiles, a 6-stage mbarrier ring, both CTAs'
//    bytes completing on the even CTA's barriers); warp 1 of the even CTA issues the MMAs,
//    committing each stage back to both producers and each finished tile to both epilogues;
//    warps 2-9 of each CTA drain its accumulator with tcgen05.ld, 32 columns at a time, add bias
//    (handed out by shuffles), apply GELU(erf) and add the residual (prefetched one 64-column chunk
//    ahead), with global loads and stores coalesced through a small shared-memory tile per warp.
//    The accumulator is double-buffered in TMEM (2 x 256 columns), so the epilogue of tile i
//    overlaps the main loop of tile i+1.  With a caller workspace the tiles of the last, partial
//    wave are split over K between two pairs that exchange partial sums (described at unit_of).
//    A is consumed K-major, B ([K,N], N contiguous) MN-major, both straight from their row-major
//    layouts.
//  * M <= 64 (decode): gemm_decode.cu.
//  * Cut plans: the GEMM kernel stops after the first stage segment and stores that fp16
//    intermediate; a vectorised tail kernel (the segment's stages a template parameter) applies
//    each later segment in place in Y.
//  * Every mbarrier wait is bounded; a wait that runs out raises the watchdog word, the CTA lets
//    its copies and MMAs in flight finish (bounded), frees its TMEM and returns.
#include <cudaTypedefs.h>
#include <math.h>

#include <atomic>
#include <mutex>

#include "fc_internal.cuh"
#include "fc_ptx.cuh"
#include "fc_tc.cuh"
#include "gemm_epi.cuh"

namespace fc {

// the decode kernel (gemm_decode.cu)
int launch_decode_gemm(const void* A, const void* B, const void* bias, const void* R, void* Y, int64_t M,
                       int64_t N, int64_t K, int epi, bool b_static, cudaStream_t st);
int decode_report(fuse_kernel_record* out);

namespace {

// =============================================================================== main kernel
// A CTA pair computes a 256 x BN output tile with M = 256 MMAs (cta_group::2): each CTA holds its
// own 128 rows of A and one half (BN / 2 columns) of B per stage.
constexpr int BM = 128, BN = 256, BK = 64, STAGES = 6;
constexpr int kEpiWarps = 8;                   // two per TMEM lane quadrant
constexpr int kMainThreads = 32 * (2 + kEpiWarps);
constexpr uint32_t A_STAGE = BM * BK * 2;      // 16 KB
constexpr uint32_t B_BOX = 64 * BK * 2;        // 8 KB: 64 N x 64 K
constexpr uint32_t B_STAGE = (BN / 2) * BK * 2;  // 16 KB: this CTA's half of the B tile
constexpr uint32_t OFF_A = 0;
constexpr uint32_t OFF_B = OFF_A + STAGES * A_STAGE;
constexpr uint32_t OFF_BAR = OFF_B + STAGES * B_STAGE;
// barriers: full[STAGES], empty[STAGES], acc_full[2], acc_empty[2], part_written, part_read, drain,
// role
constexpr uint32_t N_BARS = STAGES * 2 + 2 + 2 + 2 + 1 + 1;
constexpr uint32_t OFF_HOLD = OFF_BAR + N_BARS * 8;   // TMEM address (4 bytes)
constexpr uint32_t OFF_ROLE = OFF_HOLD + 4;           // split tile: this CTA's ticket role
// epilogue staging: per epilogue warp one 32-row x 128-byte tile (16-byte chunk j of row r at
// slot j ^ (r % 8)), through which it transposes between its row-per-lane TMEM layout and
// coalesced global accesses
constexpr uint32_t STAGE_WARP = 32 * 128;
constexpr uint32_t OFF_STAGE = (OFF_HOLD + 16 + 127) / 128 * 128;
constexpr uint32_t MAIN_SMEM = OFF_STAGE + kEpiWarps * STAGE_WARP + 1024;  // + alignment slack
static_assert(MAIN_SMEM <= 232448, "shared-memory budget");
constexpr uint32_t TMEM_COLS = 2 * BN;

struct MainArgs {
    int M, N, K;
    int pair_rows;       // ceil(tiles_m / 2): a CTA pair covers two adjacent 128-row tiles
    int tiles_n;
    int full_units;      // pair tiles computed over the whole K by one pair
    int units;           // full_units + 2 * (split tiles): each later tile is split over K in two
    int nk_split;        // first k-block of the second K half of a split tile
    int epi;             // last stage applied in this kernel: 0 (C), 1 (C'), 2 (C''), 3 (Y)
    const __half* bias;
    const __half* R;
    __half* Y;
    float* part;         // split tiles: raw fp32 sums, [slot][K half][rank] x 128 x 256
    unsigned long long* ticket;   // split tiles: [slot][rank] ticket word, (epoch << 32) | count
    int* full;           // split tiles: [slot][rank] = epoch once a leaving part's sums are complete
    int epoch;           // this call's tag for the ticket and full words (never 0)
    long long partner_window;   // SM cycles a first part waits for the other's ticket
    int* flag;
};

// Work unit u of a CTA pair -> output rows [m0, m0+128) of this CTA (rank r of the pair takes the
// r-th of two adjacent 128-row tiles), columns [n0, n0+256) shared by the pair, k-blocks
// [kb0, kb1).  The first full_units units are whole pair tiles; the pair tiles of the last,
// partial wave are split over K into two units (part 0: the first half of K, part 1: the second),
// so that the wave spreads over twice as many SMs (wave quantisation: 256 pair tiles on 76 pairs
// would otherwise leave two thirds of the SMs idle for the last tile time).  The two parts
// exchange fp32 partial sums through global memory; normally each finishes one column half of the
// tile (part p adds the other part's sums of columns 128p..128p+127 and applies the epilogue
// there, with all eight epilogue warps).  Which part finishes what is settled by a ticket
// (split_ticket) so that neither part ever waits for one that has not started: the parts need
// not be resident at the same time.  Splitting N instead does not help: an M = 256, N = 128 MMA
// takes as long as an N = 256 one on this hardware.
struct Unit {
    int m0, n0, kb0, kb1;
    int part;   // -1: whole tile; 0 or 1: K half of a split tile
    int slot;   // split tile index
};
constexpr int kGroupRows = 16;   // pair rows per band of the tile order
__device__ __forceinline__ Unit unit_of(int u, const MainArgs& a, uint32_t rank, int nk) {
    Unit r;
    int t = u;
    r.part = -1;
    r.slot = 0;
    r.kb0 = 0;
    r.kb1 = nk;
    if (u >= a.full_units) {
        const int s = u - a.full_units;
        t = a.full_units + s / 2;
        r.slot = s / 2;
        r.part = s % 2;
        r.kb0 = r.part ? a.nk_split : 0;
        r.kb1 = r.part ? nk : a.nk_split;
    }
    // Tiles run in groups of kGroupRows pair rows, column by column within a group, so that the
    // tiles in flight share a band of A that stays in L2 (16 x 256 rows of A at K = 4096 are
    // 32 MB) while B is streamed once per band; with one band (M <= 4096) this is plain
    // column-major order.  Walking all of M per column instead re-reads A from DRAM for every
    // column of tiles once A outgrows L2 (measured at M = 32768: 5.7x the ledger's bytes).
    const int per_group = kGroupRows * a.tiles_n;
    const int g = t / per_group, first = g * kGroupRows;
    const int rows = a.pair_rows - first < kGroupRows ? a.pair_rows - first : kGroupRows;
    const int i = t - g * per_group;
    r.m0 = (2 * (first + i % rows) + static_cast<int>(rank)) * BM;
    r.n0 = (i / rows) * BN;
    return r;
}

// Roles of the two parts of a split tile, per CTA rank, from its ticket word (epoch << 32 | count;
// any other epoch reads as count 0).  Each part first publishes the raw sums of the other part's
// column half, then takes its ticket:
//  * count 2: the other part took its ticket first and published its sums before: both finish
//    their own column half (kRoleNormal);
//  * count 1: first.  The other part may not have started (it need not be resident), so this one
//    waits for it a bounded while (kPartnerWindow); if it takes its ticket meanwhile, kRoleNormal.
//    Otherwise the first claims the word (count kLeft) and leaves the whole tile to the other:
//    it publishes its sums of its own half too, then the full word (kRoleLeft);
//  * count kLeft + 1: the other part left: wait for its full word (it is running, so the wait
//    ends) and finish both halves (kRoleAlone).
// Nobody waits for a party that has not taken its ticket, so no pair of clusters needs to be
// co-resident.  The party that sees the final count resets the word to 0 (the full word is reset
// by its reader), so a completed call leaves the workspace as it found it: a CUDA graph replay,
// which reuses its epoch, starts from zeros.
constexpr int kRoleFailed = 0, kRoleNormal = 1, kRoleLeft = 2, kRoleAlone = 3;
constexpr unsigned long long kLeft = 0x100;
constexpr long long kPartnerWindow = 100000;   // SM cycles, ~50 us (default)

__device__ __forceinline__ unsigned long long ld_relaxed_gpu_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ int split_ticket(unsigned long long* tw, int epoch, long long window) {
    const unsigned long long E = static_cast<unsigned long long>(static_cast<unsigned>(epoch)) << 32;
    unsigned long long old = ld_relaxed_gpu_u64(tw), nw;
    for (;;) {
        nw = (old & 0xffffffff00000000ull) == E ? old + 1 : (E | 1ull);
        const unsigned long long prev = atomicCAS(tw, old, nw);
        if (prev == old) break;
        old = prev;
    }
    const unsigned long long cnt = nw & 0xffffffffull;
    if (cnt == 2) return kRoleNormal;
    if (cnt == kLeft + 1) {
        atomicExch(tw, 0ull);
        return kRoleAlone;
    }
    if (cnt != 1) return kRoleFailed;
    const long long t0 = clock64();
    while (clock64() - t0 < window) {
        if (ld_relaxed_gpu_u64(tw) == (E | 2ull)) {
            atomicExch(tw, 0ull);
            return kRoleNormal;
        }
    }
    const unsigned long long prev = atomicCAS(tw, E | 1ull, E | kLeft);
    if (prev == (E | 1ull)) return kRoleLeft;
    if (prev == (E | 2ull)) {
        atomicExch(tw, 0ull);
        return kRoleNormal;
    }
    return kRoleFailed;
}

__global__ void __launch_bounds__(kMainThreads, 1) gemm_tc_kernel(
    const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
    const __grid_constant__ MainArgs args) {
    pdl_trigger();  // the set-up below touches no global memory; pdl_wait() follows it
    extern __shared__ uint8_t smem_raw[];
    const uint32_t base = (smem_addr(smem_raw) + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - smem_addr(smem_raw));
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t bar0 = base + OFF_BAR;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto accf_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
    auto acce_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
    const uint32_t drain_bar = bar0 + 8u * (N_BARS - 2);
    // the eight epilogue warps of a split unit have written (read) the exchanged partial sums
    const uint32_t part_written = bar0 + 8u * (N_BARS - 4), part_read = bar0 + 8u * (N_BARS - 3);
    const uint32_t role_bar = bar0 + 8u * (N_BARS - 1);
    const uint32_t holder = base + OFF_HOLD;
    const int total_units = args.units;
    const int nk = (args.K + BK - 1) / BK;
    int* flag = args.flag;
    const uint32_t rank = cluster_rank();
    const int cid = blockIdx.x / 2;            // CTA pair (cluster) index
    const int nclusters = gridDim.x / 2;
    // k-blocks this pair runs in all (both CTAs run the same sequence)
    int total_kb = 0;
    for (int u = cid; u < total_units; u += nclusters) {
        const Unit w = unit_of(u, args, rank, nk);
        total_kb += w.kb1 - w.kb0;
    }

    // The even CTA of the pair (rank 0) issues the MMAs.  Its full barriers count the bytes both
    // CTAs load for a stage; every CTA's empty and accumulator-full barriers are signalled by the
    // leader's commits (multicast); its accumulator-empty barriers collect the epilogue warps of
    // both CTAs.
    const bool leader = rank == 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf_bar(b), 1);
            mbar_init(acce_bar(b), 2 * kEpiWarps);
        }
        mbar_init(drain_bar, 1);
        mbar_init(part_written, kEpiWarps);
        mbar_init(part_read, kEpiWarps);
        mbar_init(role_bar, 1);
        fence_mbar_init();
        prefetch_map(&mapA);
        prefetch_map(&mapB);
    }
    if (warp == 1) tmem_alloc_pair(holder, TMEM_COLS);
    tc_fence_before();
    cluster_sync();  // both CTAs' barriers exist before either signals the other
    tc_fence_after();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(gbase + OFF_HOLD);
    pdl_wait();  // the preceding kernel has completed: global memory may be touched

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        int stage = 0;
        uint32_t phase = 0, inflight = 0, issue_par = 0;
        bool ok = true;
        for (int u = cid; u < total_units && ok; u += nclusters) {
            const Unit w = unit_of(u, args, rank, nk);
            for (int kb = w.kb0; kb < w.kb1; ++kb) {
                // the stage is free in both CTAs (each MMA commit arrives on both empty barriers)
                if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, flag)) { ok = false; break; }
                inflight &= ~(1u << stage);  // its previous load was consumed
                if (lane == 0) {
                    // this CTA's 128 rows of A and its half of the B tile's columns; both CTAs'
                    // bytes complete on the leader's full barrier
                    if (leader) mbar_arrive_expect_tx(full_bar(stage), 2 * (A_STAGE + B_STAGE));
                    const uint32_t full_cl = mapa_shared(full_bar(stage), 0);
                    tma_load_2d_pair(base + OFF_A + stage * A_STAGE, &mapA, kb * BK, w.m0, full_cl);
                    for (int j = 0; j < B_STAGE / B_BOX; ++j)
                        tma_load_2d_pair(base + OFF_B + stage * B_STAGE + j * B_BOX, &mapB,
                                         w.n0 + static_cast<int>(rank) * (BN / 2) + 64 * j, kb * BK, full_cl);
                }
                inflight |= 1u << stage;
                issue_par = (issue_par & ~(1u << stage)) | (phase << stage);
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
        }
        if (!ok && leader) {  // let both CTAs' loads in flight land before either can exit
            for (int s = 0; s < STAGES; ++s)
                if ((inflight >> s) & 1u) (void)mbar_wait_drain(full_bar(s), (issue_par >> s) & 1u);
        }
    } else if (warp == 1 && leader) {
        // ------------------------------------------------------------ MMA issuer
        constexpr uint32_t idesc = idesc_f16(2 * BM, BN, false, true);
        int stage = 0, acc = 0;
        uint32_t phase = 0, acc_phase = 0;
        bool ok = true, issued = false;
        int kg = 0;  // k-blocks issued so far by this CTA (the same sequence in both CTAs)
        for (int u = cid; u < total_units && ok; u += nclusters) {
            const Unit w = unit_of(u, args, rank, nk);
            if (!mbar_wait_bounded(acce_bar(acc), acc_phase ^ 1u, flag)) { ok = false; break; }
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + acc * BN;
            for (int kb = w.kb0; kb < w.kb1; ++kb) {
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
                        // apart (SBO); +16 rows (2048 B) per K=16 step; the peer's half sits at
                        // the same offsets in its shared memory
                        const uint64_t bd = smem_desc_sw128(b0 + 2048u * k, B_BOX, 1024u);
                        tc_mma_pair(d_tmem, ad, bd, idesc, (kb > w.kb0 || k > 0) ? 1u : 0u);
                    }
                    // frees the stage in both CTAs once these MMAs are done -- unless no later load
                    // uses it
                    if (kg + STAGES < total_kb) tc_commit_pair_mc(empty_bar(stage), 0x3);
                }
                ++kg;
                issued = true;
                __syncwarp();
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
            if (!ok) break;
            if (lane == 0) tc_commit_pair_mc(accf_bar(acc), 0x3);   // both CTAs' accumulators
            __syncwarp();
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
        if (!ok && issued) {  // MMAs in flight must finish before TMEM is freed
            if (lane == 0) tc_commit_pair(drain_bar);
            __syncwarp();
            (void)mbar_wait_drain(drain_bar, 0);
        }
    } else if (warp >= 2) {
        // ------------------------------------------------------------ epilogue (warps 2-9)
        // Warp w drains TMEM lane quadrant q = w % 4 (rows 32q..32q+31 of the unit) and one half
        // of the unit's 64-column chunks; after tcgen05.ld each thread holds one row.  Global
        // memory is accessed coalesced (8 lanes per 128-byte row segment, 4 rows per instruction)
        // and transposed through the warp's staging tile: the residual chunk is loaded that way
        // one chunk ahead, written to the tile and read back by rows; the fp16 results are
        // written to the tile by rows and stored by row segments.
        // Split tiles exchange raw fp32 sums through the caller's workspace; which part finishes
        // which columns is settled by a ticket (split_ticket).
        constexpr int CH = 64;
        constexpr int PER = (BN / CH) / 2;   // chunks of each warp per unit
        const int q = warp % 4;
        const int h = (warp - 2) / 4;
        const bool need_r = args.epi >= 3;
        uint8_t* stage = gbase + OFF_STAGE + (warp - 2) * STAGE_WARP;
        const int cr = lane / 8, cj = lane % 8;   // coalesced layout: row cr + 4 i, 16-byte chunk cj
        auto st_row = [&](int r, int j, const uint4& v) {
            *reinterpret_cast<uint4*>(stage + r * 128 + ((j ^ (r & 7)) * 16)) = v;
        };
        auto ld_row = [&](int r, int j) {
            return *reinterpret_cast<const uint4*>(stage + r * 128 + ((j ^ (r & 7)) * 16));
        };
        int acc = 0;
        uint32_t acc_phase = 0;
        bool ok = true;
        uint4 rnext[8];
        // Whole tiles: this warp finishes chunks h*PER and h*PER + 1.  Split tiles (part p): the
        // warp owns chunk c1 = 2p + h of this part's column half and chunk c0 = 2(1 - p) + h of
        // the other's; it first stores its raw sums of c0 for the other part, then finishes c1
        // with the other part's sums of it (and c0 too when this part finishes the tile alone).
        auto first_r_chunk = [&](const Unit& w) { return w.part < 0 ? h * PER : 2 * w.part + h; };
        auto load_r = [&](int u, int c) {  // residual chunk c of unit u, coalesced layout
            const Unit w = unit_of(u, args, rank, nk);
            const int col = w.n0 + CH * c + 8 * cj;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int row = w.m0 + 32 * q + cr + 4 * i;
                rnext[i] = make_uint4(0, 0, 0, 0);
                if (row < args.M && col < args.N)
                    rnext[i] = __ldcs(reinterpret_cast<const uint4*>(args.R + static_cast<int64_t>(row) * args.N + col));
            }
        };
        // Raw partial sums of a split unit, one region per slot, K half and CTA rank (128 x 256
        // fp32), laid out for rows held one per lane: float4 j (columns 4j..4j+3) of 32-column
        // group g of this warp's row `lane` sits at [q][g][j][lane], so a warp instruction covers
        // 512 contiguous bytes both when one part writes it and when the other reads it.
        auto part_at = [&](const Unit& w, int part, int g, int j) {
            return reinterpret_cast<float4*>(args.part) +
                   ((((static_cast<int64_t>(w.slot * 2 + part) * 2 + static_cast<int>(rank)) * 4 + q) * 8 + g) * 8 + j) * 32 + lane;
        };
        auto ticket_word = [&](const Unit& w) { return args.ticket + w.slot * 2 + static_cast<int>(rank); };
        auto full_word = [&](const Unit& w) { return args.full + w.slot * 2 + static_cast<int>(rank); };
        // This warp is done reading accumulator buffer `acc`: hand it back to the MMA issuer.
        auto release_acc = [&]() {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(mapa_shared(acce_bar(acc), 0));   // the leader's
        };
        // The raw fp32 sums of chunk c into this part's region.
        auto store_raw = [&](const Unit& w, int c, bool release) {
#pragma unroll 1
            for (int g = 0; g < 2; ++g) {
                float v[32];
                tmem_ld32(tmem_base + (static_cast<uint32_t>(32 * q) << 16) + acc * BN + CH * c + 32 * g, v);
                tmem_ld_wait();
                if (release && g == 1) release_acc();
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    __stcg(part_at(w, w.part, 2 * c + g, j), make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]));
            }
        };
        // Finish chunk c of unit w: accumulator (+ the other part's sums of it when `other` >= 0),
        // then the stages with bias (lanes 16*bslot.. hold it) and the residual (staged from rnext,
        // which holds this chunk's residual on entry; the residual chunk (nu, nc) is loaded next,
        // none if nu < 0), stored to Y.  `release`: hand the accumulator back after the last read.
        auto finish_chunk = [&](const Unit& w, int c, int bslot, int other, bool release, int nu, int nc,
                                const uint2& bl) {
            const int ncol0 = w.n0 + CH * c;
            // the residual chunk into the staging tile (each thread then reads its own row's
            // segments there and overwrites each with its result); then the next chunk's load
            if (need_r) {
#pragma unroll
                for (int i = 0; i < 8; ++i) st_row(cr + 4 * i, cj, rnext[i]);
                __syncwarp();
                if (nu >= 0) load_r(nu, nc);
            }
            // two 32-column halves of the chunk, one tcgen05.ld each
#pragma unroll 1
            for (int g = 0; g < 2; ++g) {
                float v[32];
                tmem_ld32(tmem_base + (static_cast<uint32_t>(32 * q) << 16) + acc * BN + CH * c + 32 * g, v);
                tmem_ld_wait();
                if (release && g == 1) release_acc();
                if (other >= 0) {   // add the other part's partial sums
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float4 t = __ldcg(part_at(w, other, 2 * c + g, j));
                        v[4 * j] += t.x;
                        v[4 * j + 1] += t.y;
                        v[4 * j + 2] += t.z;
                        v[4 * j + 3] += t.w;
                    }
                }
                // the 32 columns' stages in one branch-free block per stage count (the count
                // is uniform per launch), so the 16 independent GELU chains interleave
                auto finish = [&](auto last_c) {
                    constexpr int LAST = decltype(last_c)::value;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        float bv[8];
                        {
                            const int src = 16 * bslot + (32 * g + 8 * j) / 4;   // lane holding these columns
                            uint4 b8;
                            b8.x = __shfl_sync(0xffffffffu, bl.x, src);
                            b8.y = __shfl_sync(0xffffffffu, bl.y, src);
                            b8.z = __shfl_sync(0xffffffffu, bl.x, src + 1);
                            b8.w = __shfl_sync(0xffffffffu, bl.y, src + 1);
                            unpack_h8(b8, bv);
                        }
                        float rv[8] = {0, 0, 0, 0, 0, 0, 0, 0};
                        if constexpr (LAST >= 3) unpack_h8(ld_row(lane, 4 * g + j), rv);
                        float o[8];
#pragma unroll
                        for (int e = 0; e < 8; e += 2) {
                            const float2 r2 = apply_stages2_upto<LAST>(make_float2(v[8 * j + e], v[8 * j + e + 1]),
                                                                       make_float2(bv[e], bv[e + 1]),
                                                                       make_float2(rv[e], rv[e + 1]));
                            o[e] = r2.x;
                            o[e + 1] = r2.y;
                        }
                        st_row(lane, 4 * g + j, pack_h8(o));
                    }
                };
                switch (args.epi) {
                    case 3: finish(IntC<3>{}); break;
                    case 2: finish(IntC<2>{}); break;
                    case 1: finish(IntC<1>{}); break;
                    default: finish(IntC<0>{}); break;
                }
            }
            __syncwarp();
            {
                const int col = ncol0 + 8 * cj;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int row = w.m0 + 32 * q + cr + 4 * i;
                    const uint4 t = ld_row(cr + 4 * i, cj);
                    if (row < args.M && col < args.N)
                        __stcs(reinterpret_cast<uint4*>(args.Y + static_cast<int64_t>(row) * args.N + col), t);
                }
            }
            __syncwarp();
        };
        if (need_r && cid < total_units) load_r(cid, first_r_chunk(unit_of(cid, args, rank, nk)));
        for (int u = cid; u < total_units && ok; u += nclusters) {
            const Unit w = unit_of(u, args, rank, nk);
            const bool split = w.part >= 0;
            const int nu = u + nclusters < total_units ? u + nclusters : -1;     // next unit
            const int nc = nu >= 0 ? first_r_chunk(unit_of(nu, args, rank, nk)) : 0;
            // the bias values of this warp's two chunks, four per lane (lanes 16k..16k+15: its
            // k-th chunk; split units: k = 0 for c1, k = 1 for c0), fetched while the unit's MMAs
            // run and handed to every lane by shuffles, so no load latency sits in the element loop
            uint2 bl = make_uint2(0, 0);
            {
                const int k = lane / 16;
                const int c = split ? (k == 0 ? 2 * w.part + h : 2 * (1 - w.part) + h) : h * PER + k;
                const int col = w.n0 + CH * c + 4 * (lane % 16);
                if (args.epi >= 1 && col < args.N) bl = __ldg(reinterpret_cast<const uint2*>(args.bias + col));
            }
            if (!mbar_wait_bounded(accf_bar(acc), acc_phase, flag)) { ok = false; break; }
            tc_fence_after();
            if (!split) {
                for (int cc = 0; cc < PER; ++cc) {
                    const bool last = cc + 1 == PER;
                    finish_chunk(w, h * PER + cc, cc, -1, last, last ? nu : u, last ? nc : h * PER + cc + 1, bl);
                }
            } else {
                const int p = w.part;
                const int c0 = 2 * (1 - p) + h, c1 = 2 * p + h;
                // (1) the other part's column half: raw sums into this part's region
                store_raw(w, c0, false);
                __syncwarp();
                if (lane == 0) mbar_arrive(part_written);
                // (2) one thread takes the tile's ticket once all eight warps have written; the
                // ticket decides who finishes what, and nobody waits on a party that has not taken
                // its ticket yet (which might not even be resident)
                if (warp == 2 && lane == 0) {
                    int role = kRoleFailed;
                    if (mbar_wait_bounded(part_written, 0, flag)) {
                        __threadfence();
                        role = split_ticket(ticket_word(w), args.epoch, args.partner_window);
                        __threadfence();
                    }
                    *reinterpret_cast<volatile int*>(gbase + OFF_ROLE) = role;
                    mbar_arrive(role_bar);
                }
                if (!mbar_wait_bounded(role_bar, 0, flag)) { ok = false; break; }
                const int role = *reinterpret_cast<volatile int*>(gbase + OFF_ROLE);
                if (role == kRoleFailed) { ok = false; break; }
                fence_acq_rel_gpu();   // the other part's sums, published before its ticket
                if (role == kRoleLeft) {
                    // the other part finishes the whole tile: leave it this part's other half too
                    store_raw(w, c1, true);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(part_read);
                    if (warp == 2 && lane == 0 && mbar_wait_bounded(part_read, 0, flag)) {
                        __threadfence();
                        st_release_gpu(full_word(w), args.epoch);
                    }
                    __syncwarp();
                } else if (role == kRoleNormal) {
                    finish_chunk(w, c1, 0, 1 - p, true, nu, nc, bl);
                } else {   // kRoleAlone: the other part left both halves of its sums
                    if (!__all_sync(0xffffffffu, flag_wait_bounded(full_word(w), args.epoch, flag))) {
                        ok = false;
                        break;
                    }
                    finish_chunk(w, c1, 0, 1 - p, false, u, c0, bl);
                    finish_chunk(w, c0, 1, 1 - p, true, nu, nc, bl);
                    // all eight warps have read the sums: clear the word for a later call (a graph
                    // replay reuses its epoch)
                    if (lane == 0) mbar_arrive(part_read);
                    if (warp == 2 && lane == 0 && mbar_wait_bounded(part_read, 0, flag)) *full_word(w) = 0;
                    __syncwarp();
                }
            }
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
        __syncwarp();
    }
    tc_fence_before();
    cluster_sync();  // neither CTA leaves while its peer may still write into its shared memory
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem_base, TMEM_COLS);
}

// =============================================================================== tail kernel
// Y <- h(stages first..last applied to Y), 8 halves per thread (N % 8 == 0).
template <int FIRST, int LAST>
__global__ void __launch_bounds__(256) epi_tail_kernel(__half* __restrict__ Y, const __half* __restrict__ bias,
                                                       const __half* __restrict__ R, int64_t M, int N) {
    pdl_begin();  // before any global-memory access (programmatic dependent launch)
    const int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t total = M * N / 8;
    if (g >= total) return;
    const int n = static_cast<int>((g * 8) % N);
    float v[8], bv[8] = {0, 0, 0, 0, 0, 0, 0, 0}, rv[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    uint4* yp = reinterpret_cast<uint4*>(Y) + g;
    unpack_h8(*yp, v);
    if constexpr (FIRST <= 1 && LAST >= 1) unpack_h8(__ldg(reinterpret_cast<const uint4*>(bias + n)), bv);
    if constexpr (LAST >= 3) unpack_h8(__ldcs(reinterpret_cast<const uint4*>(R) + g), rv);
    // stages FIRST..LAST fixed at compile time: one branch-free block for the eight values
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
        float2 x = make_float2(v[e], v[e + 1]);
        if constexpr (FIRST <= 1 && LAST >= 1) x = __fadd2_rn(x, make_float2(bv[e], bv[e + 1]));
        if constexpr (FIRST <= 2 && LAST >= 2) x = gelu_erf2(x);
        if constexpr (LAST >= 3) x = __fadd2_rn(x, make_float2(rv[e], rv[e + 1]));
        v[e] = x.x;
        v[e + 1] = x.y;
    }
    *yp = pack_h8(v);
}

// =============================================================================== host side

bool overlap(const void* a, int64_t abytes, const void* b, int64_t bbytes) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + static_cast<uintptr_t>(bbytes) && y < x + static_cast<uintptr_t>(abytes);
}

int main_attr() {
    return opt_in_smem((const void*)gemm_tc_kernel, static_cast<int>(MAIN_SMEM));
}

// 2-CTA clusters that can be resident at once (a cluster needs both its CTAs in one GPC, so an
// odd SM count in a GPC leaves an SM out); persistent launches use exactly this many.
int max_active_pairs() {
    static std::mutex mu;
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        (void)cudaGetLastError();
        return sm_count() / 2;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (cached[dev] == 0 && main_attr() == FUSE_OK) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * static_cast<unsigned>(sm_count()));
        cfg.blockDim = dim3(kMainThreads);
        cfg.dynamicSmemBytes = MAIN_SMEM;
        cudaLaunchAttribute attrs[1];
        attrs[0].id = cudaLaunchAttributeClusterDimension;
        attrs[0].val.clusterDim.x = 2;
        attrs[0].val.clusterDim.y = 1;
        attrs[0].val.clusterDim.z = 1;
        cfg.attrs = attrs;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, gemm_tc_kernel, &cfg) != cudaSuccess || n < 1) {
            (void)cudaGetLastError();
            n = sm_count() / 2;
        }
        cached[dev] = n;
    }
    return cached[dev] > 0 ? cached[dev] : sm_count() / 2;
}

// Split-K workspace: a 2 KB header (the ticket words, one per split tile and CTA rank, then the
// full words), then the raw fp32 partial sums of the split tiles, 128 x 256 per K half and CTA.
constexpr int kSplitMaxTiles = 64;
constexpr int64_t kSplitHeader = 2048;
constexpr int64_t kSplitFullOffset = 8 * 2 * kSplitMaxTiles;
constexpr int64_t kSplitTileBytes = 2LL * 2LL * BM * BN * 4;
static_assert(kSplitFullOffset + 4 * 2 * kSplitMaxTiles <= kSplitHeader, "ticket and full words fit the header");

int64_t split_ws_bytes(int tiles) {
    const int t = tiles < kSplitMaxTiles ? tiles : kSplitMaxTiles;
    return kSplitHeader + t * kSplitTileBytes;
}

std::atomic<long long> g_partner_window{kPartnerWindow};

// Tag of one call for the ticket and full words: never 0, different from the tags of recent calls.
int next_epoch() {
    static std::atomic<unsigned> counter{0};
    unsigned e = counter.fetch_add(1, std::memory_order_relaxed) % 0x7fffffffu;
    return static_cast<int>(e) + 1;
}

// GEMM + the stages 1..epi, fp16 result into Y.  `ws` (ws_bytes, zero-filled before its first use)
// lets the last, partial wave of tiles be split over K; without it that wave runs whole tiles.
int launch_gemm(const void* A, const void* B, const void* bias, const void* R, void* Y, int64_t M,
                int64_t N, int64_t K, int epi, void* ws, size_t ws_bytes, bool b_static, cudaStream_t st) {
    int* flag = watchdog_flag();
    if (!flag) return FUSE_ECUDA;
    CUtensorMap mA, mB;
    if (M <= 64) return launch_decode_gemm(A, B, bias, R, Y, M, N, K, epi, b_static, st);
    if (!make_map(&mA, A, M, K, 64, BM) || !make_map(&mB, B, K, N, 64, 64)) return FUSE_ECUDA;
    if (const int rc = main_attr(); rc != FUSE_OK) return rc;
    MainArgs a;
    a.M = static_cast<int>(M);
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    a.pair_rows = static_cast<int>(ceil_div(ceil_div(M, BM), 2));
    a.tiles_n = static_cast<int>(ceil_div(N, BN));
    a.epi = epi;
    a.bias = static_cast<const __half*>(bias);
    a.R = static_cast<const __half*>(R);
    a.Y = static_cast<__half*>(Y);
    a.flag = flag;
    const int tiles = a.pair_rows * a.tiles_n;             // pair tiles (256 rows x 256 cols)
    const int pairs = max_active_pairs();
    const int nk = static_cast<int>(ceil_div(K, BK));
    // split the last, partial wave over K when its halves still fit in one wave (each pair then
    // runs at most one split unit, its last) and the caller gave room for the partial sums
    const int tail = tiles % pairs;
    const bool split = tiles > pairs && tail != 0 && 2 * tail <= pairs && tail <= kSplitMaxTiles && nk >= 2 &&
                       ws != nullptr && is_aligned(ws, 256) &&
                       static_cast<int64_t>(ws_bytes) >= kSplitHeader + tail * kSplitTileBytes;
    const int clusters = tiles < pairs ? tiles : pairs;
    a.full_units = split ? tiles - tail : tiles;
    a.units = a.full_units + 2 * (tiles - a.full_units);
    a.nk_split = nk / 2;
    a.ticket = split ? static_cast<unsigned long long*>(ws) : nullptr;
    a.full = split ? reinterpret_cast<int*>(static_cast<uint8_t*>(ws) + kSplitFullOffset) : nullptr;
    a.part = split ? reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + kSplitHeader) : nullptr;
    a.epoch = split ? next_epoch() : 1;
    a.partner_window = g_partner_window.load(std::memory_order_relaxed);
    return launch_pdl(gemm_tc_kernel, dim3(static_cast<unsigned>(2 * clusters)), dim3(kMainThreads), MAIN_SMEM, st,
                      2, mA, mB, a);
}

int launch_tail(void* Y, const void* bias, const void* R, int64_t M, int64_t N, int first, int last,
                cudaStream_t st) {
    const int64_t units = M * N / 8;
    const dim3 grid(static_cast<unsigned>(ceil_div(units, 256)));
    __half* y = static_cast<__half*>(Y);
    const __half* b = static_cast<const __half*>(bias);
    const __half* r = static_cast<const __half*>(R);
    const int n = static_cast<int>(N);
    switch (first * 4 + last) {   // segments of the chain after a cut: stages first..last
        case 1 * 4 + 1: return launch_pdl(epi_tail_kernel<1, 1>, grid, dim3(256), 0, st, 1, y, b, r, M, n);
        case 1 * 4 + 2: return launch_pdl(epi_tail_kernel<1, 2>, grid, dim3(256), 0, st, 1, y, b, r, M, n);
        case 1 * 4 + 3: return launch_pdl(epi_tail_kernel<1, 3>, grid, dim3(256), 0, st, 1, y, b, r, M, n);
        case 2 * 4 + 2: return launch_pdl(epi_tail_kernel<2, 2>, grid, dim3(256), 0, st, 1, y, b, r, M, n);
        case 2 * 4 + 3: return launch_pdl(epi_tail_kernel<2, 3>, grid, dim3(256), 0, st, 1, y, b, r, M, n);
        case 3 * 4 + 3: return launch_pdl(epi_tail_kernel<3, 3>, grid, dim3(256), 0, st, 1, y, b, r, M, n);
        default: return FUSE_EINVAL;
    }
}

}  // namespace

int gemm_report_count() { return 3; }
int gemm_report(int i, fuse_kernel_record* out) {
    switch (i) {
        case 0: {
            if (const int ra = main_attr(); ra != FUSE_OK) return ra;
            const int rc = describe_kernel((const void*)gemm_tc_kernel,
                                           "gemm_tc_kernel (2-CTA cluster, 128x256 tcgen05)",
                                           kMainThreads, static_cast<int>(MAIN_SMEM), out,
                                           static_cast<int>(TMEM_COLS));
            if (rc == FUSE_OK) {
                out->cluster_size = 2;
                out->max_active_clusters = max_active_pairs();
            }
            return rc;
        }
        case 1: return decode_report(out);
        case 2: return describe_kernel((const void*)epi_tail_kernel<1, 3>, "epi_tail_kernel<1,3> (unfused plans)", 256, 0, out);
        default: return FUSE_EINVAL;
    }
}

}  // namespace fc

extern "C" int fuse_gemm_epilogue_ws(const void* A, const void* B, const void* bias, const void* R, void* Y,
                                     int64_t M, int64_t N, int64_t Kdim, uint32_t cut_mask, void* workspace,
                                     size_t ws_bytes, fuse_stream_t stream) {
    using namespace fc;
    if (M < 0 || N < 0 || Kdim < 0 || (cut_mask & ~(7u | FUSE_GEMM_STATIC_B)) != 0u) return FUSE_EINVAL;
    const bool b_static = (cut_mask & FUSE_GEMM_STATIC_B) != 0u;
    cut_mask &= 7u;
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
    if (workspace && ws_bytes > 0) {
        const int64_t wb = static_cast<int64_t>(ws_bytes);
        if (overlap(workspace, wb, Y, ybytes) || overlap(workspace, wb, A, M * Kdim * 2) ||
            overlap(workspace, wb, B, Kdim * N * 2) || overlap(workspace, wb, bias, N * 2) ||
            overlap(workspace, wb, R, M * N * 2))
            return FUSE_EINVAL;
    }
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // segments of the chain (stage 0 = mm, 1 = bias, 2 = gelu, 3 = residual)
    int first = 0;
    while (first < 4) {
        int last = first;
        while (last < 3 && !((cut_mask >> last) & 1u)) ++last;
        const int rc = first == 0 ? launch_gemm(A, B, bias, R, Y, M, N, Kdim, last, workspace, ws_bytes, b_static, st)
                                  : launch_tail(Y, bias, R, M, N, first, last, st);
        if (rc != FUSE_OK) return rc;
        first = last + 1;
    }
    return FUSE_OK;
}

extern "C" int fuse_gemm_epilogue_plan(const void* A, const void* B, const void* bias, const void* R,
                                       void* Y, int64_t M, int64_t N, int64_t Kdim, uint32_t cut_mask,
                                       fuse_stream_t stream) {
    return fuse_gemm_epilogue_ws(A, B, bias, R, Y, M, N, Kdim, cut_mask, nullptr, 0, stream);
}

extern "C" int fuse_gemm_epilogue(const void* A, const void* B, const void* bias, const void* R, void* Y,
                                  int64_t M, int64_t N, int64_t Kdim, fuse_stream_t stream) {
    return fuse_gemm_epilogue_ws(A, B, bias, R, Y, M, N, Kdim, 0u, nullptr, 0, stream);
}

extern "C" int fuse_debug_split_window(int64_t cycles) {
    if (cycles < 0 || cycles > 2000000000LL) return FUSE_EINVAL;
    fc::g_partner_window.store(cycles, std::memory_order_relaxed);
    return FUSE_OK;
}

extern "C" size_t fuse_gemm_workspace_bytes(int64_t M, int64_t N, int64_t Kdim) {
    using namespace fc;
    if (M <= 64 || N <= 0 || Kdim <= 0) return 0;   // the decode kernel needs none
    const int64_t tiles = ceil_div(ceil_div(M, BM), 2) * ceil_div(N, BN);
    return static_cast<size_t>(split_ws_bytes(tiles > kSplitMaxTiles ? kSplitMaxTiles : static_cast<int>(tiles)));
}

extern "C" int64_t fuse_gemm_bytes(int64_t M, int64_t N, int64_t Kdim, uint32_t cut_mask) {
    if (M < 0 || N < 0 || Kdim < 0 || cut_mask > 7u) return FUSE_EINVAL;
    // [K4] §① traffic: A, B, bias and R are read once in any plan, Y written once; every cut adds
    // one write and one read of an M x N fp16 intermediate.
    const int cuts = static_cast<int>((cut_mask & 1u) + ((cut_mask >> 1) & 1u) + ((cut_mask >> 2) & 1u));
    return 2 * (M * Kdim + Kdim * N + N + M * N + M * N + 2 * static_cast<int64_t>(cuts) * M * N);
}
