// watchdog.cu -- the device watchdog word and its test hook.
//
// Every spin-wait in this library's kernels is bounded (fc::mbar_wait_bounded).  A wait that runs
// out sets this word instead of trapping or hanging; the kernel then unwinds normally, so the
// context stays usable and the host learns of it through fuse_check() as FUSE_ETIMEOUT.
#include <mutex>

#include "fc_internal.cuh"
#include "fc_ptx.cuh"

__device__ int g_fc_watchdog;

namespace fc {

// Device address of the watchdog word on the current device (looked up once per device).
int* watchdog_flag() {
    static std::mutex mu;
    static int* cached[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        (void)cudaGetLastError();
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (!cached[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_fc_watchdog) != cudaSuccess) {
            (void)cudaGetLastError();
            return nullptr;
        }
        cached[dev] = static_cast<int*>(p);
    }
    return cached[dev];
}

int watchdog_take() {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_fc_watchdog, sizeof(int)) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    if (v) {
        const int zero = 0;
        (void)cudaMemcpyToSymbol(g_fc_watchdog, &zero, sizeof(int));
    }
    return v != 0;
}

namespace {
// One thread waits on an mbarrier that nobody arrives on; the bounded wait gives up after
// `budget` cycles, raises the flag and the kernel returns.
__global__ void watchdog_probe_kernel(int* flag, long long budget) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_addr(&bar);
    mbar_init(b, 1);
    fence_mbar_init();
    (void)mbar_wait_bounded(b, 0, flag, budget);
}
}  // namespace

}  // namespace fc

extern "C" int fuse_debug_expire_wait(int64_t budget_cycles, fuse_stream_t stream) {
    if (budget_cycles < 0 || budget_cycles >= (int64_t(1) << 31)) return FUSE_EINVAL;
    int* flag = fc::watchdog_flag();
    if (!flag) return FUSE_ECUDA;
    fc::watchdog_probe_kernel<<<1, 1, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        flag, static_cast<long long>(budget_cycles));
    return fc::check_launch();
}
