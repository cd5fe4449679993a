// gemm.cu -- fp16 GEMM + bias + GELU + residual (tcgen05 / TMEM / TMA).  Kernels land here.
#include "fc_internal.cuh"

namespace fc {
int gemm_report_count() { return 0; }
int gemm_report(int, fuse_kernel_record*) { return FUSE_EINVAL; }
}  // namespace fc
