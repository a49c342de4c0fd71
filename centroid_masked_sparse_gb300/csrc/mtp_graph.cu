// CUDA graphs of the masked calls: record one call with fixed buffers, replay it
// with a single launch.  The counterpart of the fixed-size graphs of
// Gemma4Proposer._setup_centroids_cuda_graphs ("Add Gemma4 MTP speculative
// decoding with centroids masking", vLLM spec_decode/gemma4.py); the calls are
// capture-safe by construction (no allocation, no host synchronisation, a fixed
// launch sequence chained by programmatic dependent launches, which the graph
// keeps as programmatic edges).
#include <new>

#include "internal.h"

struct mtp_graph {
    cudaGraph_t graph;
    cudaGraphExec_t exec;
    int device;   // the descriptor's device, current while the graph is launched
};

namespace {

mtp_status run_call(const mtp_head_desc *desc, int32_t finish, const void *hidden, int32_t batch, void *out0,
                    void *out1, void *ws, size_t ws_bytes, void *stream)
{
    if (finish == MTP_FINISH_ARGMAX)
        return mtp_masked_topk_tokens(desc, hidden, batch, (int32_t *)out0, (float *)out1, ws, ws_bytes, stream);
    if (finish == MTP_FINISH_SCATTER)
        return mtp_masked_scatter_logits(desc, hidden, batch, (float *)out0, ws, ws_bytes, stream);
    return mtp_select_and_score(desc, hidden, batch, (float *)out0, (int32_t *)out1, ws, ws_bytes, stream);
}

}  // namespace

extern "C" {

mtp_status mtp_graph_capture(const mtp_head_desc *desc, int32_t finish, const void *hidden, int32_t batch,
                             void *out0, void *out1, void *workspace, size_t workspace_bytes, void *stream,
                             mtp_graph **graph)
{
    if (!graph) return MTP_ERR_NULL;
    *graph = nullptr;
    if (!stream) return MTP_ERR_NULL;
    if (finish != MTP_FINISH_ARGMAX && finish != MTP_FINISH_SCATTER && finish != MTP_FINISH_PAIR)
        return MTP_ERR_SHAPE;
    if (batch < 1) return MTP_ERR_SHAPE;
    // eagerly once: validates everything and does the one-time per-device work
    // (kernel attributes, occupancy queries, tensor-map encoder lookup) outside the capture
    mtp_status st = run_call(desc, finish, hidden, batch, out0, out1, workspace, workspace_bytes, stream);
    if (st != MTP_OK) return st;
    const mtp::DeviceScope dev(desc->device);
    if (!dev.ok) return MTP_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal) != cudaSuccess) return MTP_ERR_CUDA;
    st = run_call(desc, finish, hidden, batch, out0, out1, workspace, workspace_bytes, stream);
    cudaGraph_t g = nullptr;
    const cudaError_t e = cudaStreamEndCapture(s, &g);
    if (st != MTP_OK || e != cudaSuccess || !g) {
        if (g) cudaGraphDestroy(g);
        cudaGetLastError();
        return st != MTP_OK ? st : MTP_ERR_CUDA;
    }
    cudaGraphExec_t x = nullptr;
    if (cudaGraphInstantiate(&x, g, 0) != cudaSuccess) {
        cudaGraphDestroy(g);
        cudaGetLastError();
        return MTP_ERR_CUDA;
    }
    mtp_graph *h = new (std::nothrow) mtp_graph{g, x, desc->device};
    if (!h) {
        cudaGraphExecDestroy(x);
        cudaGraphDestroy(g);
        return MTP_ERR_CUDA;
    }
    *graph = h;
    return MTP_OK;
}

mtp_status mtp_graph_launch(const mtp_graph *graph, void *stream)
{
    if (!graph) return MTP_ERR_NULL;
    const mtp::DeviceScope dev(graph->device);
    if (!dev.ok) return MTP_ERR_CUDA;
    return cudaGraphLaunch(graph->exec, (cudaStream_t)stream) == cudaSuccess ? MTP_OK : MTP_ERR_CUDA;
}

mtp_status mtp_graph_destroy(mtp_graph *graph)
{
    if (!graph) return MTP_OK;
    const cudaError_t a = cudaGraphExecDestroy(graph->exec);
    const cudaError_t b = cudaGraphDestroy(graph->graph);
    delete graph;
    return (a == cudaSuccess && b == cudaSuccess) ? MTP_OK : MTP_ERR_CUDA;
}

}  // extern "C"
