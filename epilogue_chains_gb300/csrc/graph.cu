// graph.cu -- CUDA-graph capture and replay of this library's calls.
//
// "AIGC fundamentals | operator fusion and CUDA Graph" §3.4: a graph turns N host submissions
// into one, while the GPU front end still walks the N kernel nodes; §6.4: what was captured is
// frozen (shapes, addresses) and nothing inside may hand control back to the host.  The capture
// wraps whatever the caller issues on one stream between fuse_graph_begin() and fuse_graph_end()
// (any mode of any entry point); replay re-runs those kernels with the same arguments.
#include <mutex>
#include <new>

#include "fc_internal.cuh"

struct fuse_graph_s {
    cudaGraphExec_t exec = nullptr;
    int kernels = 0;
};

namespace fc {
namespace {

// Make every kernel of the library resident on the current device before a capture starts, so
// that no lazy module load and no first-use lookup happens while the stream is capturing.
int preload_current_device() {
    static std::mutex mu;
    static bool done[64] = {false};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return record_cuda_error(e);
    if (dev < 0 || dev >= 64) return FUSE_EUNSUPPORTED;
    std::lock_guard<std::mutex> lock(mu);
    if (done[dev]) return FUSE_OK;
    if (!watchdog_flag()) return FUSE_ECUDA;
    (void)sm_count();
    const int n = fuse_kernel_count();
    for (int i = 0; i < n; ++i) {
        fuse_kernel_record r;
        const int rc = fuse_kernel_report(i, &r);
        if (rc != FUSE_OK) return rc;
    }
    done[dev] = true;
    return FUSE_OK;
}

}  // namespace
}  // namespace fc

extern "C" int fuse_graph_begin(fuse_stream_t stream) {
    if (!stream) return FUSE_EINVAL;  // the legacy default stream cannot be captured
    const int rc = fc::preload_current_device();
    if (rc != FUSE_OK) return rc;
    cudaError_t e = cudaStreamBeginCapture(reinterpret_cast<cudaStream_t>(stream),
                                           cudaStreamCaptureModeThreadLocal);
    return e == cudaSuccess ? FUSE_OK : fc::record_cuda_error(e);
}

extern "C" int fuse_graph_end(fuse_stream_t stream, fuse_graph_t* out) {
    if (!stream || !out) return FUSE_EINVAL;
    *out = nullptr;
    cudaGraph_t graph = nullptr;
    cudaError_t e = cudaStreamEndCapture(reinterpret_cast<cudaStream_t>(stream), &graph);
    if (e != cudaSuccess) {
        if (graph) (void)cudaGraphDestroy(graph);
        return fc::record_cuda_error(e);
    }
    size_t n = 0;
    e = cudaGraphGetNodes(graph, nullptr, &n);
    int kernels = 0;
    if (e == cudaSuccess && n > 0) {
        cudaGraphNode_t* nodes = new (std::nothrow) cudaGraphNode_t[n];
        if (!nodes) {
            (void)cudaGraphDestroy(graph);
            return FUSE_EUNSUPPORTED;
        }
        e = cudaGraphGetNodes(graph, nodes, &n);
        for (size_t i = 0; e == cudaSuccess && i < n; ++i) {
            cudaGraphNodeType t;
            e = cudaGraphNodeGetType(nodes[i], &t);
            if (e == cudaSuccess && t == cudaGraphNodeTypeKernel) ++kernels;
        }
        delete[] nodes;
    }
    cudaGraphExec_t exec = nullptr;
    if (e == cudaSuccess) e = cudaGraphInstantiate(&exec, graph, 0);
    (void)cudaGraphDestroy(graph);
    if (e != cudaSuccess) return fc::record_cuda_error(e);
    fuse_graph_s* g = new (std::nothrow) fuse_graph_s;
    if (!g) {
        (void)cudaGraphExecDestroy(exec);
        return FUSE_EUNSUPPORTED;
    }
    g->exec = exec;
    g->kernels = kernels;
    *out = g;
    return FUSE_OK;
}

extern "C" int fuse_graph_launch(fuse_graph_t g, fuse_stream_t stream) {
    if (!g || !g->exec) return FUSE_EINVAL;
    cudaError_t e = cudaGraphLaunch(g->exec, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FUSE_OK : fc::record_cuda_error(e);
}

extern "C" int fuse_graph_kernel_count(fuse_graph_t g) { return g ? g->kernels : FUSE_EINVAL; }

extern "C" void fuse_graph_destroy(fuse_graph_t g) {
    if (!g) return;
    if (g->exec) (void)cudaGraphExecDestroy(g->exec);
    delete g;
}
