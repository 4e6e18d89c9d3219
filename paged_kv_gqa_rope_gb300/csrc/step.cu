// A whole decode step behind one call (RoPE/append then decode, chained by
// programmatic dependent launch) and its capture into a replayable CUDA
// graph ("nano-vllm notes - Llama": the serving loop's decode step, captured
// in a CUDA graph); the prefill step likewise (RoPE/append then the varlen
// causal prefill, "nano-vllm notes - Llama", prepare_prefill).
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <new>

#include "common.cuh"
#include "internal.h"
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

// The device's address of page-locked host memory mapped into its address
// space (all cudaHostAlloc memory under unified addressing), else null.
void *mapped_ptr(const void *p) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// n bytes from src to dst (both 16-byte aligned), one 16-byte piece per
// thread and pass, the last n % 16 bytes by block 0.  The step graph's
// host <-> device copies: this kernel reads or writes the mapped host
// buffer itself, so the copy is one kernel node instead of a copy-engine
// transfer with its own set-up latency.  Launched as a dependent of the
// kernel before it (whose writes it waits for).  It does not let the next
// kernel launch early: the input copy writes the decode kernel's context
// lengths and block tables, which that kernel reads before its own
// grid-dependency wait, so the RoPE/append kernel between them must not
// start (and let the decode kernel start) before this copy has finished.
__global__ void __launch_bounds__(256)
    copy_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst, size_t n16,
                const uint8_t *__restrict__ src_b, uint8_t *__restrict__ dst_b, size_t n) {
    pa::griddep_wait();
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += stride)
        dst[i] = src[i];
    if (blockIdx.x == 0)
        for (size_t i = n16 * 16 + threadIdx.x; i < n; i += blockDim.x) dst_b[i] = src_b[i];
}

int copy_by_kernel(const void *src, void *dst, size_t n, cudaStream_t st) {
    const size_t n16 = n / 16;
    const int blocks =
        (int)std::max<size_t>(1, std::min<size_t>((n16 + 255) / 256, (size_t)pa::sm_count() * 4));
    pa::launch_dependent(copy_kernel, dim3(blocks), dim3(256), 0, st,
                         static_cast<const uint4 *>(src), static_cast<uint4 *>(dst), n16,
                         static_cast<const uint8_t *>(src), static_cast<uint8_t *>(dst), n);
    return pa::launch_status();
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
        // The copies: a kernel on the mapped host buffer when there is one
        // (and every address is 16-byte aligned), else a copy-engine copy.
        if (in_bytes > 0) {
            const void *src = mapped_ptr(host_in);
            if (src && aligned16(src) && aligned16(dev_in))
                rc = copy_by_kernel(src, dev_in, in_bytes, cs);
            else if (cudaMemcpyAsync(dev_in, host_in, in_bytes, cudaMemcpyHostToDevice, cs) !=
                     cudaSuccess)
                rc = PA_ERR_CUDA;
        }
        if (rc == PA_OK)
            rc = pa_decode_step(q, k, v, positions, slot_mapping, rope_table, max_positions,
                                cache, layer, block_tables, max_blocks_per_seq, context_lens,
                                num_seqs, n_heads, n_kv_heads, head_dim, scale, workspace,
                                workspace_bytes, out, dev_status, cs);
        if (rc == PA_OK && out_bytes > 0) {
            void *dst = mapped_ptr(host_out);
            if (dst && aligned16(dst) && aligned16(out))
                rc = copy_by_kernel(out, dst, out_bytes, cs);
            else if (cudaMemcpyAsync(host_out, out, out_bytes, cudaMemcpyDeviceToHost, cs) !=
                     cudaSuccess)
                rc = PA_ERR_CUDA;
        }
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
