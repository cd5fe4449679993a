/*
 * fusechain.h -- C ABI of the vertical-fusion library for one NVIDIA GB300 (sm_103a).
 *
 * A chain of K dependent operators runs as ONE kernel that reads its inputs from HBM once, keeps
 * every intermediate in registers or shared memory and writes only the final output.  Each chain
 * also has an explicit unfused mode (one kernel per stage, intermediates through global memory)
 * so that the byte ledgers of the pages can be checked against measured DRAM traffic.
 *
 * Sources (web pages; cited by title and section):
 *   [K4]   "K4 walkthrough: the three ledgers of fusion -- bytes, launches, registers"
 *   [C05]  "C-05 Kernel Fusion cost boundary: less write-back vs register pressure and occupancy"
 *   [OFCG] "AIGC fundamentals | operator fusion and CUDA Graph"
 *
 * Conventions for every entry point below:
 *   - Compute calls are stream-ordered and asynchronous: they validate their arguments on the
 *     host, enqueue kernels on `stream` (NULL = the legacy default stream) and return.  None of
 *     them synchronizes.
 *   - Pointers named as device pointers must be device (or managed) memory that stays valid until
 *     the enqueued work finishes; the caller owns all of it.  Host pointers (stage arrays, output
 *     records) are read or written before the call returns.
 *   - No compute entry point allocates memory.  Unfused modes that need row statistics take a
 *     caller workspace whose size the matching *_workspace_bytes() call returns.
 *   - All tensors are dense, row-major and contiguous.
 *   - Return value: FUSE_OK (0) or a negative fuse_status.  FUSE_ECUDA means the launch itself
 *     failed (cudaGetLastError() after the launch); the CUDA error string is then available from
 *     fuse_last_cuda_error().  No C++ exception crosses this boundary.
 *   - The library is thread-compatible: concurrent calls on different streams are allowed.
 */
#ifndef FUSECHAIN_H
#define FUSECHAIN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st* fuse_stream_t;

typedef enum {
    FUSE_OK = 0,
    FUSE_EINVAL = -1,         /* null pointer, size <= 0, K out of range, bad enum value     */
    FUSE_EALIGN = -2,         /* alignment / leading-dimension rule of the call not met       */
    FUSE_EUNSUPPORTED = -3,   /* a size or combination this build does not implement          */
    FUSE_ECUDA = -4,          /* a CUDA launch or runtime call failed                         */
    FUSE_ETIMEOUT = -5,       /* a bounded device-side wait ran out (watchdog)                */
    FUSE_EWORKSPACE = -6      /* workspace pointer missing or smaller than required           */
} fuse_status;

typedef enum { FUSE_F32 = 0, FUSE_F16 = 1, FUSE_BF16 = 2 } fuse_dtype;

typedef enum {
    FUSE_FUSED = 0,           /* one kernel for the whole chain                                */
    FUSE_UNFUSED = 1,         /* one kernel per stage, intermediates through global memory     */
    FUSE_FAT = 2              /* fused + a deliberately register-heavy live-temporary probe    */
} fuse_mode;

typedef enum {
    FUSE_OP_AFFINE = 0,       /* v <- a*v + b                                                  */
    FUSE_OP_AFFINE_RELU = 1   /* v <- max(a*v + b, +0)  (t > 0 ? t : +0)                       */
} fuse_op;

#define FUSE_MAX_STAGES 32
#define FUSE_FAT_TEMPS 48     /* live fp32 temporaries per element in FUSE_FAT mode ([C05] §3) */

/*
 * One operator of a chain.  [K4] introduction and §③: a Stage states how many elements it
 * writes, how many elements it reads from outside the chain (weights, bias, residual, or the
 * chain input for the first stage), its FLOPs and the registers it keeps live when fused.
 * fuse_chain_run() executes `op`, `a`, `b`; fuse_ledger() reads the other fields.
 */
typedef struct {
    int32_t op;               /* fuse_op                                                       */
    float a;                  /* multiplier (fp32)                                             */
    float b;                  /* addend (fp32)                                                 */
    int64_t writes;           /* elements written                                              */
    int64_t ext_reads;        /* elements read from outside the chain                          */
    int64_t flops;            /* floating-point operations                                     */
    int32_t live_regs;        /* registers live per thread when fused                          */
} fuse_stage;

/* ===================================================================== pointwise chain
 * [C05] §3 (API / experiment shape): stage s computes y = a_s*y + b_s (ReLU on the even stages
 * in the pages' sweep); the fused kernel loops s = 0..K-1 in registers and writes once; the
 * naive form launches one stage kernel per s and passes the intermediate through global memory;
 * the fat form is the fused kernel plus FUSE_FAT_TEMPS live temporaries summed into a sink.
 * [OFCG] §3.2 gives the byte ledger: unfused 2*K*N*b, fused 2*N*b.
 *
 * Arithmetic: every stage rounds twice in fp32, t = fl32(fl32(a*v) + b) (no FMA contraction),
 * then ReLU if op == FUSE_OP_AFFINE_RELU.  Values are loaded from `dtype` exactly and every value
 * stored to global memory is rounded (nearest-even) to `dtype`: FUSED and FAT store once, so
 * they give bit-identical y; UNFUSED stores after every stage, so it equals them for FUSE_F32
 * and, for 16-bit storage, equals the chain applied one stage at a time.
 *
 *   stages  host array of K stages (1 <= K <= FUSE_MAX_STAGES)
 *   x       device pointer, n elements of `dtype` (input; may equal y, may not partially overlap)
 *   y       device pointer, n elements of `dtype` (output)
 *   n       element count, n >= 0 (n == 0 enqueues nothing)
 *   dtype   FUSE_F32, FUSE_F16 or FUSE_BF16 (storage type; math is fp32)
 *   mode    FUSE_FUSED: 1 launch, reads x once, writes y once.
 *           FUSE_UNFUSED: K launches; stage 0 reads x and writes y, stage s > 0 reads y and
 *             writes y in place (the intermediate round-trips through global memory each stage).
 *           FUSE_FAT: 1 launch of the register-heavy probe; y identical to FUSED.
 * Alignment: any element-aligned pointers work; the 32-byte vector path is used where x and y
 * share their offset modulo 32 bytes.
 */
int fuse_chain_run(const fuse_stage* stages, int K, const void* x, void* y, int64_t n,
                   int dtype, int mode, fuse_stream_t stream);
/* The same chain for data in host memory: the call a host-side caller makes with its own buffers.
 * x_host is copied to the device, the chain runs there, and y comes back to y_host.  The vector
 * is cut into `slices` (1..64) pieces of whole 32-byte vectors, and each piece's copy in, kernel(s)
 * and copy out are ordered by events, so both copy directions overlap the kernels and each other.
 *   x_host, y_host  host memory of n elements of `dtype` (page-locked, from cudaHostAlloc or
 *           cudaHostRegister, for the copies to run asynchronously; pageable memory works, but its
 *           copies wait for the host)
 *   x_dev, y_dev    device scratch of n elements each, owned by the caller (overwritten; may be
 *           the same buffer, may not partially overlap); the call allocates nothing
 *   stages, K, n, dtype, mode  as fuse_chain_run()
 * Stream order: the copies start after the work queued on `stream` before the call, the kernels
 * run on `stream`, and `stream` continues only after the last piece is back in y_host (read
 * y_host after synchronizing `stream`).  The copies run on two helper streams that the library
 * creates at the first call on each device (with five events) and keeps until the process exits;
 * calls from several host threads are serialized on them.
 */
int fuse_chain_run_host(const fuse_stage* stages, int K, const void* x_host, void* y_host,
                        int64_t n, int dtype, int mode, void* x_dev, void* y_dev, int slices,
                        fuse_stream_t stream);

/* ===================================================================== RMSNorm
 * [OFCG] §3.2 and fusion_lab [A2]: RMSNorm unfused is four passes (x*x, reduce-mean, x*r, *g),
 * fused is one.  Computes, per row i,
 *     r_i = 1 / sqrt(mean_j x_ij^2 + eps),   y_ij = (x_ij * r_i) * w_j
 * with fp32 storage and fp32 accumulation.
 *
 *   x, y    device fp32 [rows, hidden];  w  device fp32 [hidden]
 *   rows >= 0, 1 <= hidden <= 65536, eps >= 0
 *   mode    FUSE_FUSED: one kernel, one CTA per row with the row kept in registers
 *           (hidden <= 16384 in this build; larger -> FUSE_EUNSUPPORTED).
 *           FUSE_UNFUSED: four kernels: sq = x^2 -> y;  ms = rowmean(y) -> workspace;
 *             t = x * rsqrt(ms + eps) -> y;  y = y * w  (in place).  Requires y != x.
 *   workspace / ws_bytes: device scratch for the unfused row statistics; at least
 *           fuse_rmsnorm_workspace_bytes(rows, hidden, mode) bytes; may be NULL for FUSED.
 */
int fuse_rmsnorm(const float* x, const float* w, float* y, int64_t rows, int64_t hidden,
                 float eps, int mode, void* workspace, size_t ws_bytes, fuse_stream_t stream);
size_t fuse_rmsnorm_workspace_bytes(int64_t rows, int64_t hidden, int mode);

/* Allocation-free variant of the unfused RMSNorm (the pages have no counterpart: this entry point
 * exists for callers, not for the method).  Some callers cannot allocate device memory at the
 * point where they call: a host that hands this library a fixed memory budget and owns every
 * allocation in it, or a latency-critical loop where cudaMalloc (which can synchronize the device
 * and take unbounded time) is not allowed.  This call takes no workspace and allocates nothing:
 * its row statistics live in one library-owned __device__ array of FUSE_RMSNORM_STATIC_MAX_ROWS
 * floats (256 KiB), which every GPU that loads the library keeps until the process exits.
 * Same arithmetic, kernels and output as fuse_rmsnorm(..., FUSE_UNFUSED, ...).
 *   rows > FUSE_RMSNORM_STATIC_MAX_ROWS -> FUSE_EUNSUPPORTED (nothing launched); y != x.
 * The first call on each device looks up the array's device address (cudaGetSymbolAddress) with
 * that device current; make that first call before any stream capture.  The address is kept per
 * device context: after cudaDeviceReset() the next call on that device (a new context) looks it
 * up again, so make that call before any capture too.  All calls share the
 * array and it keeps the last call's contents, so calls that may overlap on the GPU (different
 * streams, or different host threads on one device) race; serialize them.
 */
#define FUSE_RMSNORM_STATIC_MAX_ROWS 65536
int fuse_rmsnorm_unfused_static(const float* x, const float* w, float* y, int64_t rows,
                                int64_t hidden, float eps, fuse_stream_t stream);

/* ===================================================================== residual add + RMSNorm
 * [OFCG] appendix launch_model [F3]: after fusion a decoder layer runs "residual + RMSNorm" as one
 * kernel where the unfused layer runs a residual-add kernel and four RMSNorm kernels.  Per row i:
 *     h_ij = x_ij + r_ij  (one fp32 rounding; the new residual stream, written out),
 *     y_ij = (h_ij * rsqrt(mean_j h_ij^2 + eps)) * w_j   (RMSNorm of h as fuse_rmsnorm()).
 *   x, r, h, y  device fp32 [rows, hidden]; w device fp32 [hidden].  h may be x or r itself (in
 *           place); y must differ from x, r and h.  Otherwise no two of them may overlap.
 *   mode    FUSE_FUSED: one kernel, reads x and r once, writes h and y once (4 N b + 4 hidden);
 *             hidden <= 16384 (larger -> FUSE_EUNSUPPORTED).
 *           FUSE_UNFUSED: five kernels, h = x + r, then the four RMSNorm kernels of fuse_rmsnorm()
 *             on h (10 N b + row means + w).  Needs workspace of
 *             fuse_rmsnorm_workspace_bytes(rows, hidden, FUSE_UNFUSED) bytes.
 * Numerics: h is bit-identical in both modes; y as fuse_rmsnorm() (fp32 accumulation).
 */
int fuse_add_rmsnorm(const float* x, const float* r, const float* w, float* h, float* y,
                     int64_t rows, int64_t hidden, float eps, int mode, void* workspace,
                     size_t ws_bytes, fuse_stream_t stream);

/* ===================================================================== SiLU(gate) * up
 * [OFCG] appendix launch_model [F3]: "SiLU + multiply" fused into one kernel after the gate/up
 * GEMM, where the unfused layer runs a SiLU kernel and an element-wise multiply kernel.
 *     y_ij = SiLU(g_ij) * u_ij,   SiLU(v) = v / (1 + e^-v).
 *   g, u    device [rows, cols] of `dtype` with a common row stride ld >= cols elements (the two
 *           halves of one merged [rows, 2 cols] gate/up output: g = base, u = base + cols,
 *           ld = 2 cols; separate dense tensors: ld = cols).  This is the one strided operand
 *           layout of the library.
 *   y       device [rows, cols], dense.  y must not overlap u; it may be g itself when ld == cols.
 *   dtype   FUSE_F32 / FUSE_F16 / FUSE_BF16 storage, fp32 math (SiLU via exp2 and reciprocal on
 *           the special-function unit: about 2^-21 relative error before the final rounding).
 *   mode    FUSE_FUSED: one kernel (3 N b).  FUSE_UNFUSED: two kernels, s = SiLU(g) stored in y
 *           (rounded to dtype), then y = s * u (5 N b).
 * The 32-byte vector path needs cols and ld multiples of 32 bytes and 32-byte aligned pointers;
 * other shapes use an element-wise kernel.
 */
int fuse_silu_mul(const void* g, const void* u, int64_t ld, void* y, int64_t rows, int64_t cols,
                  int dtype, int mode, fuse_stream_t stream);

/* ===================================================================== causal softmax
 * [OFCG] fusion_lab [E] (max -> subtract -> exp -> sum -> divide over the last axis), §3.5
 * (causal mask: query i sees keys j <= i; block-granular skipping) and [A3] (8 copies of the
 * score tensor unfused vs 2 fused).  For every row i of every (batch*head):
 *     z_j = scale * s_ij (j <= i),  p_ij = exp(z_j - max z) / sum exp(z - max z),  p_ij = +0 (j > i)
 * fp32 math, bf16 input, bf16 (nearest-even) or fp32 output.
 *
 *   s          device bf16 [batch_heads, S, S]
 *   p          device [batch_heads, S, S] of out_dtype (FUSE_BF16 or FUSE_F32)
 *   S          1 <= S <= 8192
 *   skip_tile  0: every row reads all S scores (masked ones are ignored);
 *              T > 0 (a multiple of 16): row i reads only the columns < (floor(i/T)+1)*T, i.e.
 *              the key blocks of a T x T block-causal tiling that are not fully masked.
 *              Output values do not depend on skip_tile.  FUSED mode only.
 *   scale      any finite value
 *   mode       FUSE_FUSED: one kernel, one warp per row, row kept in registers (32-byte vectors
 *              when S % 16 == 0, S <= 2048 and s, p are 32-byte aligned; otherwise a two-pass
 *              element-wise kernel that re-reads the kept scores).
 *              FUSE_UNFUSED: five kernels over whole rows; the three elementwise intermediates
 *              (scaled-and-shifted scores, exponentials) are bf16 and live in p; the row max
 *              and row sum (fp32) live in the workspace.  skip_tile must be 0.
 */
int fuse_causal_softmax(const void* s, void* p, int64_t batch_heads, int64_t S, float scale,
                        int skip_tile, int out_dtype, int mode, void* workspace,
                        size_t ws_bytes, fuse_stream_t stream);
size_t fuse_causal_softmax_workspace_bytes(int64_t batch_heads, int64_t S, int mode);

/* ===================================================================== GEMM epilogue chain
 * [K4] §① chain_mlp_epilogue: the chain mm -> +bias -> GELU -> +residual in fp16, priced under the
 * cut plans [1,1,1,1], [1,3], [2,2], [4]; §⑥ the decode shape M = 16.  [OFCG] §5.2: epilogue
 * fusion writes the GEMM output once, already in its final form.  Computes
 *     Y = fp16( GELU( A @ B + bias ) + R ),   GELU(v) = v/2 (1 + erf(v / sqrt 2)),
 * with fp16 inputs, fp32 accumulation (tcgen05 tensor cores) and fp32 epilogue math.
 *
 *   A     device fp16 [M, Kdim] row-major;   B  device fp16 [Kdim, N] row-major (N contiguous)
 *   bias  device fp16 [N];   R, Y  device fp16 [M, N] row-major.  Y must not overlap any input.
 *   Rules: N % 8 == 0 and Kdim % 8 == 0 (16-byte row strides), every pointer 16-byte aligned
 *          (FUSE_EALIGN otherwise); M, N, Kdim <= 2^31 - 1; Kdim >= 1.  Ragged tiles are handled.
 *   M > 64:  persistent 128 x 256-tile kernel, one CTA per SM.
 *   M <= 64: decode kernel (swap A/B, split K over an 8-CTA cluster, reduction in distributed
 *            shared memory).
 * fuse_gemm_epilogue() is plan [4]: one kernel, reads A, B, bias, R once, writes Y once.
 * fuse_gemm_epilogue_plan(): cut_mask bit i (i = 0, 1, 2) places a kernel boundary after stage i
 * (0 = mm, 1 = +bias, 2 = GELU): [1,1,1,1] = 7, [1,3] = 1, [2,2] = 2, [4] = 0; all 8 masks
 * are accepted.  Each cut stores the intermediate (C, C', C'') as fp16 in Y and the next kernel
 * reads it back in place, so the plan's DRAM traffic is fuse_gemm_bytes() and its numerics round
 * to fp16 exactly at the cuts.  No workspace is needed (fuse_gemm_epilogue_ws() takes an optional
 * one that balances the last wave of tiles).
 */
/* Flag for the cut_mask argument of fuse_gemm_epilogue_plan/_ws (OR it in): the caller vouches
 * that no work queued on the stream before the call writes B (a weight, as in a decode loop).
 * The decode kernel (M <= 64) then loads its first ring of weight boxes while the preceding kernel
 * may still run, instead of after waiting for it; A, bias and R are still read only after that
 * wait.  Results are unchanged; if something queued before the call does write B, the call may
 * read B's old contents.  Ignored for M > 64. */
#define FUSE_GEMM_STATIC_B 0x100u
int fuse_gemm_epilogue(const void* A, const void* B, const void* bias, const void* R, void* Y,
                       int64_t M, int64_t N, int64_t Kdim, fuse_stream_t stream);
int fuse_gemm_epilogue_plan(const void* A, const void* B, const void* bias, const void* R, void* Y,
                            int64_t M, int64_t N, int64_t Kdim, uint32_t cut_mask,
                            fuse_stream_t stream);
/* The same with a caller workspace (the library allocates nothing).  With it, when the tiles do
 * not fill a whole number of waves of the persistent kernel and the last, partial wave would leave
 * at least half of the SM pairs idle, each tile of that wave is split over K between two SM pairs,
 * which exchange fp32 partial sums through the workspace and each apply the epilogue to one half of
 * the tile's columns.  A ticket in the workspace decides who finishes what, and neither pair waits
 * for one that has not started: if the other pair is late (other work holds the SMs it would run
 * on), the first leaves its sums and the other finishes the whole tile.  Results equal the
 * unsplit kernel's up to fp32 summation order.
 *   cut_mask   the plan (bits 0..2, as fuse_gemm_epilogue_plan), optionally | FUSE_GEMM_STATIC_B;
 *              any other bit: FUSE_EINVAL.
 *   workspace  device memory of at least fuse_gemm_workspace_bytes(M, N, Kdim) bytes, 256-byte
 *              aligned, zero-filled before its first use (every completed call leaves it so; after
 *              a call that failed with FUSE_ETIMEOUT, zero it again); not shared with a call that
 *              may run at the same time.  NULL, or smaller, or misaligned: no split (still
 *              correct).  Must not overlap any operand (FUSE_EINVAL).
 */
int fuse_gemm_epilogue_ws(const void* A, const void* B, const void* bias, const void* R, void* Y,
                          int64_t M, int64_t N, int64_t Kdim, uint32_t cut_mask, void* workspace,
                          size_t ws_bytes, fuse_stream_t stream);
/* Test hook of the split tiles: how long (SM cycles, 0 <= cycles <= 2e9; default 100000) the first
 * part of a split tile waits for the other part's ticket before it leaves the whole tile to it.
 * 0 makes every first part leave, so the path where one part finishes a tile alone runs on every
 * split tile; results are the same up to fp32 summation order.  Applies to calls launched after
 * it (process-wide); FUSE_EINVAL outside the range. */
int fuse_debug_split_window(int64_t cycles);
/* Workspace bytes for fuse_gemm_epilogue_ws (0 when no split can apply, e.g. M <= 64): a 2 KB
 * header and 512 KB of fp32 partial sums per split tile, for at most 64 tiles. */
size_t fuse_gemm_workspace_bytes(int64_t M, int64_t N, int64_t Kdim);
/* [K4] §① traffic of a plan, in bytes: 2 * (M*K + K*N + N + 2*M*N + 2*cuts*M*N). */
int64_t fuse_gemm_bytes(int64_t M, int64_t N, int64_t Kdim, uint32_t cut_mask);

/* ===================================================================== attention, no score matrix
 * "AIGC fundamentals | operator fusion and CUDA Graph" §6.3 and its reading list (FlashAttention):
 * the causal softmax's S x S score tensor is never written; the softmax is fused into the
 * attention and normalised online.  Per slice b of batch x heads:
 *     O_b = softmax(scale Q_b K_b^T with keys j <= query i) V_b.
 *   q, k, v, o  device bf16 [bh, S, D] row-major, 16-byte aligned; o must not overlap q, k, v.
 *   S       a multiple of 128 (else FUSE_EUNSUPPORTED); D in {64, 128, 256} (else
 *           FUSE_EUNSUPPORTED); bh * S < 2^31.
 *   scale   > 0 (1/sqrt(D) for the usual attention).
 * One kernel (tcgen05 MMAs, scores and output accumulator in TMEM).  P is rounded to bf16 before
 * it multiplies V and O is rounded once to bf16; scores and sums are fp32.
 */
int fuse_attention(const void* q, const void* k, const void* v, void* o, int64_t bh, int64_t S,
                   int64_t D, float scale, fuse_stream_t stream);
/* Algorithmic DRAM bytes (read Q, K, V, write O once: 8 bh S D) and useful flops (2 x 2 D per
 * visible query-key pair: 2 D bh S (S + 1)) of one fuse_attention() call. */
int64_t fuse_attention_bytes(int64_t bh, int64_t S, int64_t D);
int64_t fuse_attention_flops(int64_t bh, int64_t S, int64_t D);
/* The work lists of the persistent 2-SM attention kernel (host arithmetic, no GPU needed).  Its
 * items are pairs of adjacent 128-row query tiles: item i of bh * (S / 256) covers slice and tile
 * pair as ordered in groups of 16 slices, heaviest pair first within a group; an item with pair
 * index u reads 2u + 2 key blocks.  Items go, in that order, to the cluster with the earliest
 * estimated finish (10 per key block + 8 per item); then, while it narrows their gap, the
 * busiest cluster trades an item for a lighter one of the same 16-slice group with the idlest.
 * Cluster c runs items[first[c]] .. items[first[c + 1] - 1], in increasing order.
 *   first   host int32 [clusters + 1];  items  host int32 [bh * S / 256]
 *   S a multiple of 256; 1 <= clusters <= 96; bh * S / 256 <= 4096 (the kernel falls back to a
 *   round-robin assignment beyond these, and so does this call: FUSE_EUNSUPPORTED).
 * Returns the number of items, or a negative FUSE_E* code. */
int64_t fuse_attention_schedule(int64_t bh, int64_t S, int clusters, int32_t* first, int32_t* items);

/* ===================================================================== ledgers
 * [K4] §① traffic(): a cut plan splits the K stages into consecutive kernels (cut_mask bit i =
 * a kernel boundary after stage i).  Each kernel reads the previous kernel's output (the
 * `writes` of the stage just before it, if any) plus the ext_reads of its stages, and writes
 * the `writes` of its last stage.  Bytes = elements * elem_bytes.  reg_peak is the largest sum
 * of live_regs over the stages of one kernel; flops is the plain sum.
 */
typedef struct {
    int64_t bytes;
    int64_t launches;
    int64_t reg_peak;
    int64_t flops;
} fuse_ledger_t;

int fuse_ledger(const fuse_stage* stages, int K, uint32_t cut_mask, int elem_bytes,
                fuse_ledger_t* out);

/* [K4] §② time_estimate / best_plan: a roofline + launch cost model over cut plans.  For every
 * kernel of a plan:  t = max(mem, compute) + launch,  mem = bytes / hbm_bytes_per_s (the ledger
 * bytes above), compute = flops / flops_per_s; when the kernel's live_regs sum exceeds reg_limit
 * the memory time is multiplied by spill_penalty ([K4] §③).  fuse_plan_time() returns a plan's
 * total in *seconds; fuse_best_plan() enumerates all 2^(K-1) cut masks and returns the cheapest
 * (ties go to the lower mask).  Host only, no CUDA call. */
typedef struct {
    double hbm_bytes_per_s;
    double flops_per_s;
    double launch_s;
    double spill_penalty;
    int32_t reg_limit;
} fuse_cost_model;

int fuse_plan_time(const fuse_stage* stages, int K, uint32_t cut_mask, int elem_bytes,
                   const fuse_cost_model* model, double* seconds);
int fuse_best_plan(const fuse_stage* stages, int K, int elem_bytes, const fuse_cost_model* model,
                   uint32_t* best_mask, double* best_seconds);

/* "AIGC fundamentals | operator fusion and CUDA Graph" §3.4: timeline of n_kernels kernels on one
 * stream.  Eager: the host spends t_launch per submission and does not wait; kernel i starts at
 * max(end of kernel i-1, (i+1) t_launch) and runs t_exec.  Graph: one submission, then the GPU
 * front end spends t_dispatch per node.  Outputs (any time unit, the inputs' own): *eager = total
 * eager time, *eager_idle = the GPU's idle part of it, *graph = total graph time.  Host only. */
int fuse_launch_model(int64_t n_kernels, double t_launch, double t_exec, double t_dispatch,
                      double* eager, double* eager_idle, double* graph);

/* Algorithmic DRAM bytes of one call of the entry points above (what the kernel must move at
 * minimum; the unfused forms count every intermediate round trip).  Negative = fuse_status. */
int64_t fuse_chain_bytes(int K, int64_t n, int dtype, int mode);
int64_t fuse_rmsnorm_bytes(int64_t rows, int64_t hidden, int mode);
int64_t fuse_causal_softmax_bytes(int64_t batch_heads, int64_t S, int skip_tile, int out_dtype,
                                  int mode);
int64_t fuse_add_rmsnorm_bytes(int64_t rows, int64_t hidden, int mode);
int64_t fuse_silu_mul_bytes(int64_t rows, int64_t cols, int dtype, int mode);

/* ===================================================================== reports and status
 * [K4] §③ and [C05] §6.2: registers per thread, spills and blocks per SM decide when fusion
 * loses.  fuse_kernel_report() describes one kernel variant as launched by this library.
 */
typedef struct {
    char name[64];
    int32_t regs_per_thread;
    int32_t local_bytes_per_thread;   /* local memory (spills + local arrays)                   */
    int32_t static_smem_bytes;
    int32_t dynamic_smem_bytes;       /* as launched                                            */
    int32_t block_threads;            /* as launched                                            */
    int32_t blocks_per_sm;            /* CTAs one SM holds at once: the least of what threads,
                                         registers, shared memory (with the 1 KB each CTA reserves)
                                         and tensor-memory columns allow                          */
    int32_t max_threads_per_block;
    int32_t cluster_size;             /* CTAs per thread-block cluster as launched (1 = none)    */
    int32_t max_active_clusters;      /* clusters resident at once per the occupancy API (0 if no
                                         cluster); like blocks_per_sm_api, conservative for kernels
                                         that allocate tensor memory                              */
    int32_t blocks_per_sm_api;        /* cudaOccupancyMaxActiveBlocksPerMultiprocessor's answer.
                                         For kernels that allocate tensor memory it is 1 whatever
                                         their shared memory, while the hardware runs as many CTAs
                                         as blocks_per_sm (CTA start stamps of the decode GEMM:
                                         two per SM, its 256 CTAs in one wave on 148 SMs)         */
    int32_t tmem_cols;                /* tensor-memory columns one CTA allocates (0: none)        */
    /* What ptxas -v printed for this kernel when the library was built (the same figures as
     * fuse_ptxas_entry(); -1 each if the build kept no record of the kernel):                   */
    int32_t ptxas_registers;
    int32_t stack_bytes;              /* per-thread stack frame                                  */
    int32_t spill_store_bytes;        /* bytes of register spill stores per thread               */
    int32_t spill_load_bytes;         /* bytes of register spill loads per thread                */
    char symbol[256];                 /* mangled device symbol ("" if the runtime cannot name it) */
} fuse_kernel_record;

/* The ptxas -v record of every kernel entry compiled into this library ([K4] §③ and [C05] §6.2:
 * a fused kernel that needs more registers than the SM grants spills, and the spill traffic is
 * the cost that decides against fusing).  The build parses its own ptxas output into a table
 * linked into the library, so these two calls are host only and need no GPU.
 *   fuse_ptxas_count() = number of entries; fuse_ptxas_entry(i, out) fills *out for entry i
 *   (FUSE_EINVAL if out is NULL or i is out of range). */
typedef struct {
    char symbol[256];                 /* mangled entry name as ptxas printed it                 */
    int32_t registers;
    int32_t stack_bytes;
    int32_t spill_store_bytes;
    int32_t spill_load_bytes;
} fuse_ptxas_record;
int fuse_ptxas_count(void);
int fuse_ptxas_entry(int index, fuse_ptxas_record* out);

/* Number of kernel variants fuse_kernel_report() knows (index 0 .. count-1). */
int fuse_kernel_count(void);
/* Fill *out for variant `index` (needs a CUDA device; the current device is used). */
int fuse_kernel_report(int index, fuse_kernel_record* out);

/* CUDA-graph capture of this library's calls ("AIGC fundamentals | operator fusion and CUDA
 * Graph" §3.4: one submission for N kernels; §6.4: shapes and addresses are frozen, no host
 * synchronisation inside).  Typical use, e.g. an unfused plan whose kernels are launch-bound:
 *     fuse_graph_begin(s); fuse_chain_run(..., FUSE_UNFUSED, s); fuse_graph_end(s, &g);
 *     fuse_graph_launch(g, s);  ...  fuse_graph_destroy(g);
 *   fuse_graph_begin(stream)   stream must not be NULL (the legacy stream cannot be captured).
 *       Makes every kernel of the library resident on the current device first (once per
 *       device), then starts a thread-local capture.  Calls of this library issued on `stream`
 *       until fuse_graph_end() are recorded, not run.  Do not call fuse_check() or anything that
 *       synchronizes while capturing (the capture fails; fuse_graph_end() then reports it).
 *   fuse_graph_end(stream, &g) ends the capture and instantiates it; *g is NULL on error.  If a
 *       call inside the capture returned an error, end the capture anyway and drop the result.
 *   fuse_graph_launch(g, stream) replays the recorded kernels in order on any stream, with the
 *       same pointers, sizes and parameters; update inputs in place between replays.
 *   fuse_graph_kernel_count(g) = the number of kernel nodes (launches per replay).
 *   fuse_graph_destroy(g) frees the executable graph (NULL is ignored); the caller owns g. */
typedef struct fuse_graph_s* fuse_graph_t;
int fuse_graph_begin(fuse_stream_t stream);
int fuse_graph_end(fuse_stream_t stream, fuse_graph_t* out);
int fuse_graph_launch(fuse_graph_t graph, fuse_stream_t stream);
int fuse_graph_kernel_count(fuse_graph_t graph);
void fuse_graph_destroy(fuse_graph_t graph);

const char* fuse_strerror(int status);
/* Message of the last CUDA error seen by this library on this thread ("" if none). */
const char* fuse_last_cuda_error(void);
/* Synchronize `stream`, then return FUSE_ETIMEOUT if a device watchdog fired since the last
 * check (and clear it), FUSE_ECUDA if the stream reported an error, else FUSE_OK. */
int fuse_check(fuse_stream_t stream);
/* Test hook of the watchdog: one thread waits on an mbarrier that nothing arrives on, for
 * budget_cycles SM clock cycles (0 <= budget_cycles < 2^31), then records the timeout and
 * returns normally; the next fuse_check() returns FUSE_ETIMEOUT.  It faults and traps nothing
 * and leaves the context usable (the same bounded wait guards every mbarrier wait of the GEMM). */
int fuse_debug_expire_wait(int64_t budget_cycles, fuse_stream_t stream);

/* Library version, (major << 16) | minor. */
int fuse_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FUSECHAIN_H */
