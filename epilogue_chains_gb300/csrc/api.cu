// api.cu -- status, error strings, device queries and the kernel report of the C ABI.
#include <stdio.h>
#include <string.h>

#include <mutex>
#include <vector>

#include "fc_internal.cuh"
#include "fc_tc.cuh"

namespace fc {

// per-translation-unit report tables (defined next to their kernels)
int chain_report_count();
int chain_report(int i, fuse_kernel_record* out);
int rmsnorm_report_count();
int rmsnorm_report(int i, fuse_kernel_record* out);
int softmax_report_count();
int softmax_report(int i, fuse_kernel_record* out);
int gemm_report_count();
int gemm_report(int i, fuse_kernel_record* out);
int silu_report_count();
int silu_report(int i, fuse_kernel_record* out);
int attn_report_count();
int attn_report(int i, fuse_kernel_record* out);
int watchdog_take();  // 1 if a bounded device wait expired since the last call (and clears it)

namespace {
thread_local char t_last_error[256] = "";
}

int record_cuda_error(cudaError_t e) {
    snprintf(t_last_error, sizeof(t_last_error), "%s: %s", cudaGetErrorName(e),
             cudaGetErrorString(e));
    // A failed runtime call also leaves its error as the thread's "last error"; clear it (where it
    // is not sticky) so that it is not reported again by the next call's launch check.
    (void)cudaGetLastError();
    return FUSE_ECUDA;
}

int sm_count() {
    static std::mutex mu;
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return 1;
    }
    if (dev < 0 || dev >= 64) return 1;
    std::lock_guard<std::mutex> lock(mu);
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            (void)cudaGetLastError();
            n = 1;
        }
        cached[dev] = n > 0 ? n : 1;
    }
    return cached[dev];
}

int opt_in_smem(const void* kernel, int bytes, bool max_shared_carveout) {
    struct Done {
        const void* kernel;
        int dev, bytes;
    };
    static std::mutex mu;
    static std::vector<Done> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return record_cuda_error(e);
    std::lock_guard<std::mutex> lock(mu);
    for (const Done& d : done)
        if (d.kernel == kernel && d.dev == dev && d.bytes >= bytes) return FUSE_OK;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && max_shared_carveout)
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 static_cast<int>(cudaSharedmemCarveoutMaxShared));
    if (e != cudaSuccess) return record_cuda_error(e);
    done.push_back({kernel, dev, bytes});
    return FUSE_OK;
}

// The ptxas -v table of this build (generated from the build's own ptxas output and linked in).
extern const fuse_ptxas_record kPtxasTable[];
extern const int kPtxasCount;

int describe_kernel(const void* kernel, const char* name, int block, int dyn_smem,
                    fuse_kernel_record* out, int tmem_cols) {
    if (!out) return FUSE_EINVAL;
    memset(out, 0, sizeof(*out));
    snprintf(out->name, sizeof(out->name), "%s", name);
    out->ptxas_registers = out->stack_bytes = out->spill_store_bytes = out->spill_load_bytes = -1;
    const char* sym = nullptr;
    if (cudaFuncGetName(&sym, kernel) == cudaSuccess && sym) {
        snprintf(out->symbol, sizeof(out->symbol), "%s", sym);
        for (int i = 0; i < kPtxasCount; ++i) {
            if (strcmp(kPtxasTable[i].symbol, out->symbol) != 0) continue;
            out->ptxas_registers = kPtxasTable[i].registers;
            out->stack_bytes = kPtxasTable[i].stack_bytes;
            out->spill_store_bytes = kPtxasTable[i].spill_store_bytes;
            out->spill_load_bytes = kPtxasTable[i].spill_load_bytes;
            break;
        }
    } else {
        (void)cudaGetLastError();
    }
    cudaFuncAttributes a;
    cudaError_t e = cudaFuncGetAttributes(&a, kernel);
    if (e != cudaSuccess) return record_cuda_error(e);
    out->regs_per_thread = a.numRegs;
    out->local_bytes_per_thread = static_cast<int32_t>(a.localSizeBytes);
    out->static_smem_bytes = static_cast<int32_t>(a.sharedSizeBytes);
    out->dynamic_smem_bytes = dyn_smem;
    out->block_threads = block;
    out->max_threads_per_block = a.maxThreadsPerBlock;
    out->tmem_cols = tmem_cols;
    // above the default 48 KB a launch opts in to its dynamic shared memory first; do the same so
    // the answer does not depend on whether the kernel has been launched in this process yet
    if (dyn_smem > a.maxDynamicSharedSizeBytes) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_smem);
        if (e != cudaSuccess) return record_cuda_error(e);
    }
    int b = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kernel, block, dyn_smem);
    if (e != cudaSuccess) return record_cuda_error(e);
    out->blocks_per_sm_api = b;
    // residency from the SM's own limits: threads, blocks, registers (allocated per warp in units
    // of 256), shared memory (each CTA also reserves some) and the 512 tensor-memory columns
    int dev = 0, thr = 0, blk = 0, regs = 0, smem = 0, rsv = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&thr, cudaDevAttrMaxThreadsPerMultiProcessor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&blk, cudaDevAttrMaxBlocksPerMultiprocessor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&regs, cudaDevAttrMaxRegistersPerMultiprocessor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&rsv, cudaDevAttrReservedSharedMemoryPerBlock, dev)) != cudaSuccess)
        return record_cuda_error(e);
    const int warps = (block + 31) / 32;
    const int regs_per_warp = (a.numRegs * 32 + 255) / 256 * 256;
    int n = blk;
    n = n < thr / block ? n : thr / block;
    if (regs_per_warp > 0) n = n < regs / (regs_per_warp * warps) ? n : regs / (regs_per_warp * warps);
    const int per_cta = dyn_smem + static_cast<int>(a.sharedSizeBytes) + rsv;
    n = n < smem / per_cta ? n : smem / per_cta;
    if (tmem_cols > 0) n = n < 512 / tmem_cols ? n : 512 / tmem_cols;
    out->blocks_per_sm = n;
    out->cluster_size = 1;
    out->max_active_clusters = 0;
    return FUSE_OK;
}

namespace {
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
}  // namespace

bool make_map(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols, int box_cols,
              int box_rows, bool bf16) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                     const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace fc

namespace {
struct ReportTable {
    int (*count)();
    int (*get)(int, fuse_kernel_record*);
};
const ReportTable kTables[] = {
    {fc::chain_report_count, fc::chain_report},
    {fc::rmsnorm_report_count, fc::rmsnorm_report},
    {fc::softmax_report_count, fc::softmax_report},
    {fc::gemm_report_count, fc::gemm_report},
    {fc::silu_report_count, fc::silu_report},
    {fc::attn_report_count, fc::attn_report},
};
}  // namespace

extern "C" int fuse_kernel_count(void) {
    int n = 0;
    for (const auto& t : kTables) n += t.count();
    return n;
}

extern "C" int fuse_kernel_report(int index, fuse_kernel_record* out) {
    if (!out || index < 0) return FUSE_EINVAL;
    for (const auto& t : kTables) {
        const int c = t.count();
        if (index < c) return t.get(index, out);
        index -= c;
    }
    return FUSE_EINVAL;
}

extern "C" int fuse_ptxas_count(void) { return fc::kPtxasCount; }

extern "C" int fuse_ptxas_entry(int index, fuse_ptxas_record* out) {
    if (!out || index < 0 || index >= fc::kPtxasCount) return FUSE_EINVAL;
    *out = fc::kPtxasTable[index];
    return FUSE_OK;
}

extern "C" const char* fuse_strerror(int status) {
    switch (status) {
        case FUSE_OK: return "ok";
        case FUSE_EINVAL: return "invalid argument";
        case FUSE_EALIGN: return "alignment or leading-dimension rule not met";
        case FUSE_EUNSUPPORTED: return "unsupported size or combination";
        case FUSE_ECUDA: return "CUDA launch or runtime error";
        case FUSE_ETIMEOUT: return "bounded device wait expired (watchdog)";
        case FUSE_EWORKSPACE: return "workspace missing or too small";
        default: return "unknown status";
    }
}

extern "C" const char* fuse_last_cuda_error(void) { return fc::t_last_error; }

extern "C" int fuse_check(fuse_stream_t stream) {
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fc::record_cuda_error(e);
    if (fc::watchdog_take()) return FUSE_ETIMEOUT;
    return FUSE_OK;
}

extern "C" int fuse_version(void) { return (1 << 16) | 0; }
