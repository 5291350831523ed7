// graph.cu -- one convolution training step (forward, then backward) recorded
// as a CUDA graph and replayed with a single launch.
//
// A captured graph fixes a sequence of kernels and the addresses they read and
// write, not the values, and a family counts as capturable only when replay
// reproduces the eager result bit for bit (LibreYOLO documentation, page "Grafy
// CUDA", sections "Co jest przechwytywane" and "Obsługa inferencji").  A step of
// this library is a handful of kernels (operand preparation, the conv passes,
// the shard-order reductions); for a small convolution their launch latency is
// the whole cost, so the step is captured once on a private stream and replayed
// on the caller's stream.  The graph is bound to the buffers given at creation.
// Every kernel of the step is deterministic, so a replay equals the eager calls
// exactly.
#include "common.cuh"

#include <new>

struct hc_step_graph_s {
    cudaGraph_t graph;
    cudaGraphExec_t exec;
};

extern "C" hc_status hc_conv2d_step_graph_create(const hc_conv_desc* d, const float* x, const float* w,
                                                 const float* bias, float* y, const float* gy, float* gx, float* gw,
                                                 float* gb, void* ws_fwd, size_t ws_fwd_bytes, void* ws_bwd,
                                                 size_t ws_bwd_bytes, hc_step_graph* out) {
    if (!out) return HC_ERR_INVALID_ARG;
    *out = nullptr;
    if (!d || !x || !w || !y || !gy) return HC_ERR_INVALID_ARG;
    cudaStream_t s;
    if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) return HC_ERR_CUDA;
    // relaxed: the first call of a kernel family sets its shared-memory attribute
    // and may look up the tensor-map encoder, which are host calls, not stream work
    if (cudaStreamBeginCapture(s, cudaStreamCaptureModeRelaxed) != cudaSuccess) {
        cudaStreamDestroy(s);
        return HC_ERR_CUDA;
    }
    // with separate workspaces the backward pass reads x's operand copy from the
    // forward one where the algorithm keeps one (the results equal
    // hc_conv2d_bwd's bit for bit); a shared buffer would be overwritten first
    const char *f0 = (const char*)ws_fwd, *b0 = (const char*)ws_bwd;
    const bool apart = !f0 || !b0 || f0 + ws_fwd_bytes <= b0 || b0 + ws_bwd_bytes <= f0;
    hc_status st = hc_conv2d_fwd(d, x, w, bias, y, ws_fwd, ws_fwd_bytes, (void*)s);
    if (st == HC_OK)
        st = apart ? hc_conv2d_bwd_reuse(d, x, w, gy, gx, gw, gb, nullptr, nullptr, ws_bwd, ws_bwd_bytes, ws_fwd,
                                         ws_fwd_bytes, (void*)s, HC_ALGO_AUTO)
                   : hc_conv2d_bwd(d, x, w, gy, gx, gw, gb, nullptr, nullptr, ws_bwd, ws_bwd_bytes, (void*)s);
    cudaGraph_t g = nullptr;
    const cudaError_t e = cudaStreamEndCapture(s, &g);
    cudaStreamDestroy(s);
    if (st != HC_OK || e != cudaSuccess || !g) {
        if (g) cudaGraphDestroy(g);
        cudaGetLastError();
        return st != HC_OK ? st : HC_ERR_CUDA;
    }
    cudaGraphExec_t ex;
    if (cudaGraphInstantiate(&ex, g, 0) != cudaSuccess) {
        cudaGraphDestroy(g);
        cudaGetLastError();
        return HC_ERR_CUDA;
    }
    hc_step_graph h = new (std::nothrow) hc_step_graph_s{g, ex};
    if (!h) {
        cudaGraphExecDestroy(ex);
        cudaGraphDestroy(g);
        return HC_ERR_CUDA;
    }
    *out = h;
    return HC_OK;
}

extern "C" hc_status hc_step_graph_launch(hc_step_graph g, void* stream) {
    if (!g) return HC_ERR_INVALID_ARG;
    return cudaGraphLaunch(g->exec, (cudaStream_t)stream) == cudaSuccess ? HC_OK : HC_ERR_CUDA;
}

extern "C" hc_status hc_step_graph_destroy(hc_step_graph g) {
    if (!g) return HC_OK;
    const bool ok = cudaGraphExecDestroy(g->exec) == cudaSuccess && cudaGraphDestroy(g->graph) == cudaSuccess;
    delete g;
    return ok ? HC_OK : HC_ERR_CUDA;
}
