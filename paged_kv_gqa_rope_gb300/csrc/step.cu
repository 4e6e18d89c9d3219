// A whole decode step behind one call (RoPE/append then decode, chained by
// programmatic dependent launch) and its capture into a replayable CUDA
// graph ("nano-vllm notes - Llama": the serving loop's decode step, captured
// in a CUDA graph); the prefill step likewise (RoPE/append then the varlen
// causal prefill, "nano-vllm notes - Llama", prepare_prefill).
#include <cuda_runtime.h>

#include <new>

#include "pa.h"

struct pa_step_graph {
    cudaGraphExec_t exec;  // the captured kernels carry their arguments
};

extern "C" int pa_decode_step(void *q, void *k, const void *v, const int32_t *positions,
                              const int32_t *slot_mapping, const void *rope_table,
                              int max_positions, const pa_cache_t *cache, int layer,
                              const int32_t *block_tables, int max_blocks_per_seq,
                              const int32_t *context_lens, int num_seqs, int n_heads,
                              int n_kv_heads, int head_dim, float scale, void *workspace,
                              size_t workspace_bytes, void *out, int32_t *dev_status,
                              pa_stream_t stream) {
    int rc = pa_rope_kv_write(q, k, v, positions, slot_mapping, num_seqs, n_heads, n_kv_heads,
                              head_dim, rope_table, max_positions, cache, layer, dev_status,
                              stream);
    if (rc != PA_OK) return rc;
    return pa_decode(q, cache, layer, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                     n_heads, n_kv_heads, head_dim, scale, workspace, workspace_bytes, out,
                     dev_status, stream);
}

extern "C" int pa_prefill_step(void *q, void *k, const void *v, const int32_t *positions,
                               const int32_t *slot_mapping, const void *rope_table,
                               int max_positions, const pa_cache_t *cache, int layer,
                               const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                               const int32_t *block_tables, int max_blocks_per_seq, int num_seqs,
                               int total_q, int max_seqlen_q, int n_heads, int n_kv_heads,
                               int head_dim, float scale, void *out, int32_t *dev_status,
                               pa_stream_t stream) {
    int rc = pa_rope_kv_write(q, k, v, positions, slot_mapping, total_q, n_heads, n_kv_heads,
                              head_dim, rope_table, max_positions, cache, layer, dev_status,
                              stream);
    if (rc != PA_OK) return rc;
    return pa_prefill_varlen(q, total_q, cache, layer, cu_seqlens_q, cu_seqlens_k, block_tables,
                             max_blocks_per_seq, num_seqs, max_seqlen_q, n_heads, n_kv_heads,
                             head_dim, scale, out, dev_status, stream);
}

namespace {

// True if p is host memory the device can copy from asynchronously
// (page-locked: allocated by cudaHostAlloc / cudaMallocHost or registered).
bool page_locked(const void *p) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return at.type == cudaMemoryTypeHost;
}

}  // namespace

extern "C" int pa_step_graph_create_io(
    pa_step_graph_t *graph, void *q, void *k, const void *v, const int32_t *positions,
    const int32_t *slot_mapping, const void *rope_table, int max_positions,
    const pa_cache_t *cache, int layer, const int32_t *block_tables, int max_blocks_per_seq,
    const int32_t *context_lens, int num_seqs, int n_heads, int n_kv_heads, int head_dim,
    float scale, void *workspace, size_t workspace_bytes, void *out, int32_t *dev_status,
    const void *host_in, void *dev_in, size_t in_bytes, void *host_out) {
    if (!graph) return PA_ERR_INVALID;
    *graph = nullptr;
    if (in_bytes > 0 && (!host_in || !dev_in)) return PA_ERR_INVALID;
    if (in_bytes > 0 && !page_locked(host_in)) return PA_ERR_INVALID;
    if (host_out && (!out || num_seqs <= 0 || !page_locked(host_out))) return PA_ERR_INVALID;
    const size_t out_bytes =
        host_out ? (size_t)num_seqs * (size_t)n_heads * (size_t)head_dim * 2 : 0;
    cudaStream_t cs = nullptr;
    if (cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess) {
        cudaGetLastError();
        return PA_ERR_CUDA;
    }
    int rc = PA_OK;
    cudaGraph_t g = nullptr;
    cudaGraphExec_t exec = nullptr;
    if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeRelaxed) != cudaSuccess) {
        rc = PA_ERR_CUDA;
    } else {
        if (in_bytes > 0 &&
            cudaMemcpyAsync(dev_in, host_in, in_bytes, cudaMemcpyHostToDevice, cs) != cudaSuccess)
            rc = PA_ERR_CUDA;
        if (rc == PA_OK)
            rc = pa_decode_step(q, k, v, positions, slot_mapping, rope_table, max_positions,
                                cache, layer, block_tables, max_blocks_per_seq, context_lens,
                                num_seqs, n_heads, n_kv_heads, head_dim, scale, workspace,
                                workspace_bytes, out, dev_status, cs);
        if (rc == PA_OK && out_bytes > 0 &&
            cudaMemcpyAsync(host_out, out, out_bytes, cudaMemcpyDeviceToHost, cs) != cudaSuccess)
            rc = PA_ERR_CUDA;
        // End the capture whatever happened, so the stream is usable again.
        if (cudaStreamEndCapture(cs, &g) != cudaSuccess && rc == PA_OK) rc = PA_ERR_CUDA;
    }
    if (rc == PA_OK && cudaGraphInstantiate(&exec, g, 0) != cudaSuccess) rc = PA_ERR_CUDA;
    if (g) cudaGraphDestroy(g);
    cudaStreamDestroy(cs);
    if (rc != PA_OK) {
        if (exec) cudaGraphExecDestroy(exec);
        cudaGetLastError();
        return rc;
    }
    pa_step_graph *h = new (std::nothrow) pa_step_graph;
    if (!h) {
        cudaGraphExecDestroy(exec);
        return PA_ERR_CUDA;
    }
    h->exec = exec;
    *graph = h;
    return PA_OK;
}

extern "C" int pa_step_graph_create(pa_step_graph_t *graph, void *q, void *k, const void *v,
                                    const int32_t *positions, const int32_t *slot_mapping,
                                    const void *rope_table, int max_positions,
                                    const pa_cache_t *cache, int layer,
                                    const int32_t *block_tables, int max_blocks_per_seq,
                                    const int32_t *context_lens, int num_seqs, int n_heads,
                                    int n_kv_heads, int head_dim, float scale, void *workspace,
                                    size_t workspace_bytes, void *out, int32_t *dev_status) {
    return pa_step_graph_create_io(graph, q, k, v, positions, slot_mapping, rope_table,
                                   max_positions, cache, layer, block_tables, max_blocks_per_seq,
                                   context_lens, num_seqs, n_heads, n_kv_heads, head_dim, scale,
                                   workspace, workspace_bytes, out, dev_status, nullptr, nullptr,
                                   0, nullptr);
}

extern "C" int pa_step_graph_launch(pa_step_graph_t graph, pa_stream_t stream) {
    if (!graph) return PA_ERR_INVALID;
    return cudaGraphLaunch(graph->exec, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

extern "C" int pa_step_graph_destroy(pa_step_graph_t graph) {
    if (!graph) return PA_ERR_INVALID;
    const bool ok = cudaGraphExecDestroy(graph->exec) == cudaSuccess;
    delete graph;
    return ok ? PA_OK : PA_ERR_CUDA;
}
