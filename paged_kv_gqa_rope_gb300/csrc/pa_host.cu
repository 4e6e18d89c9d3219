// Host entry points of libpa: the cache pool, the metadata of a prefill call
// or a decode step, the RoPE table, error strings and device checks.
#include <math.h>
#include <string.h>

#include <mutex>
#include <vector>

#include "internal.h"

namespace pa {

int sm_count() {
    static int counts[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (counts[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        counts[dev] = n;
    }
    return counts[dev];
}

EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

bool make_cache_map(CUtensorMap *map, const pa_cache_t *c, int box_halves, int box_rows) {
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return false;
    const uint64_t d = c->head_dim, hk = c->n_kv_heads;
    const uint64_t rows = (uint64_t)c->num_blocks * c->block_size;
    cuuint64_t dims[5] = {64, d / 64, hk, rows, 2ull * c->layers};
    cuuint64_t strides[4] = {128, d * 2, hk * d * 2, (uint64_t)c->layer_stride * 2};
    cuuint32_t box[5] = {64, (cuuint32_t)box_halves, 1, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 5, c->base, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     // L2 fetches of one (token, KV head) row: 2 * head_dim bytes
                     d >= 128 ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B
                              : CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 5-D fp16 map of layer `layer`'s K and V planes: {64, D/64, Hk, rows, 2},
// box {64, D/64, 1, 16, 2}: one copy brings a block's K tile then its V
// tile (each as make_cache_map's box of the whole row would).
bool make_cache_pair_map(CUtensorMap *map, const pa_cache_t *c, int layer) {
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return false;
    const uint64_t d = c->head_dim, hk = c->n_kv_heads;
    const uint64_t rows = (uint64_t)c->num_blocks * c->block_size;
    cuuint64_t dims[5] = {64, d / 64, hk, rows, 2};
    cuuint64_t strides[4] = {128, d * 2, hk * d * 2, (uint64_t)c->kv_stride * 2};
    cuuint32_t box[5] = {64, (cuuint32_t)(d / 64), 1, (cuuint32_t)c->block_size, 2};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 5,
                     static_cast<__half *>(c->base) + (size_t)layer * c->layer_stride, dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     d >= 128 ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B
                              : CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace pa

using namespace pa;

namespace {

// A block id whose slots block * block_size .. + block_size - 1 are int32.
bool slot_fits(int32_t block, int block_size) {
    return block >= 0 && ((int64_t)block + 1) * block_size - 1 <= INT32_MAX;
}

}  // namespace

extern "C" {

size_t pa_cache_bytes(int layers, int num_blocks, int block_size, int n_kv_heads, int head_dim) {
    if (layers <= 0 || num_blocks <= 0 || block_size <= 0 || n_kv_heads <= 0 || head_dim <= 0)
        return 0;
    return (size_t)2 * layers * num_blocks * block_size * n_kv_heads * head_dim * sizeof(__half);
}

int pa_alloc_cache(pa_cache_t *out, int layers, int num_blocks, int block_size, int n_kv_heads,
                   int head_dim, void *device_base) {
    if (!out) return PA_ERR_INVALID;
    memset(out, 0, sizeof(*out));
    const size_t bytes = pa_cache_bytes(layers, num_blocks, block_size, n_kv_heads, head_dim);
    if (bytes == 0) return PA_ERR_INVALID;
    if ((int64_t)num_blocks * block_size > INT32_MAX) return PA_ERR_INVALID;  // slots are int32
    if (block_size != kBlockSize || (head_dim != 64 && head_dim != 128)) return PA_ERR_UNSUPPORTED;
    if (device_base && (reinterpret_cast<uintptr_t>(device_base) & 255u)) return PA_ERR_INVALID;
    void *base = device_base;
    if (!base) {
        if (cudaMalloc(&base, bytes) != cudaSuccess) {
            cudaGetLastError();
            return PA_ERR_CUDA;
        }
        out->owns = 1;
    }
    out->base = base;
    out->layers = layers;
    out->num_blocks = num_blocks;
    out->block_size = block_size;
    out->n_kv_heads = n_kv_heads;
    out->head_dim = head_dim;
    out->layer_stride = (int64_t)num_blocks * block_size * n_kv_heads * head_dim;
    out->kv_stride = out->layer_stride * layers;
    return PA_OK;
}

int pa_free_cache(pa_cache_t *cache) {
    if (!cache) return PA_ERR_INVALID;
    int rc = PA_OK;
    if (cache->owns && cache->base && cudaFree(cache->base) != cudaSuccess) rc = PA_ERR_CUDA;
    memset(cache, 0, sizeof(*cache));
    return rc;
}

int pa_prepare_prefill(int num_seqs, const int32_t *num_cached, const int32_t *num_new,
                       const int32_t *block_tables, int max_blocks_per_seq, int block_size,
                       int32_t *positions, int32_t *slot_mapping, int32_t *cu_seqlens_q,
                       int32_t *cu_seqlens_k, int32_t *max_seqlen_q, int32_t *max_seqlen_k) {
    if (num_seqs < 0 || block_size <= 0 || max_blocks_per_seq < 0) return PA_ERR_INVALID;
    if (num_seqs > 0 && (!num_cached || !num_new || !block_tables || !cu_seqlens_q ||
                         !cu_seqlens_k))
        return PA_ERR_INVALID;
    // First pass: validate everything before writing any output.
    int64_t total = 0, total_k = 0;
    for (int s = 0; s < num_seqs; ++s) {
        const int64_t start = num_cached[s], n = num_new[s];
        if (start < 0 || n < 0) return PA_ERR_INVALID;
        const int64_t end = start + n;
        if (end > INT32_MAX) return PA_ERR_INVALID;
        if (n > 0 && (end - 1) / block_size >= max_blocks_per_seq) return PA_ERR_INVALID;
        total += n;
        total_k += end;  // cu_seqlens_k is int32 too
        if (total > INT32_MAX || total_k > INT32_MAX) return PA_ERR_INVALID;
        for (int64_t lb = start / block_size; n > 0 && lb <= (end - 1) / block_size; ++lb)
            if (!slot_fits(block_tables[(int64_t)s * max_blocks_per_seq + lb], block_size))
                return PA_ERR_INVALID;
    }
    if (total > 0 && (!positions || !slot_mapping)) return PA_ERR_INVALID;
    int32_t mq = 0, mk = 0, t = 0;
    if (cu_seqlens_q) cu_seqlens_q[0] = 0;  // both may be NULL when num_seqs == 0
    if (cu_seqlens_k) cu_seqlens_k[0] = 0;
    for (int s = 0; s < num_seqs; ++s) {
        const int32_t start = num_cached[s], n = num_new[s], end = start + n;
        const int32_t *row = block_tables + (int64_t)s * max_blocks_per_seq;
        for (int32_t p = start; p < end; ++p, ++t) {
            positions[t] = p;
            slot_mapping[t] = row[p / block_size] * block_size + p % block_size;
        }
        cu_seqlens_q[s + 1] = cu_seqlens_q[s] + n;
        cu_seqlens_k[s + 1] = cu_seqlens_k[s] + end;
        if (n > mq) mq = n;
        if (end > mk) mk = end;
    }
    if (max_seqlen_q) *max_seqlen_q = mq;
    if (max_seqlen_k) *max_seqlen_k = mk;
    return PA_OK;
}

int pa_prepare_decode(int num_seqs, const int32_t *num_cached, const int32_t *block_tables,
                      int max_blocks_per_seq, int block_size, int32_t *positions,
                      int32_t *slot_mapping, int32_t *context_lens) {
    if (num_seqs < 0 || block_size <= 0 || max_blocks_per_seq < 0) return PA_ERR_INVALID;
    if (num_seqs == 0) return PA_OK;
    if (!num_cached || !block_tables || !positions || !slot_mapping || !context_lens)
        return PA_ERR_INVALID;
    for (int s = 0; s < num_seqs; ++s) {
        const int64_t p = num_cached[s];
        if (p < 0 || p >= INT32_MAX || p / block_size >= max_blocks_per_seq) return PA_ERR_INVALID;
        if (!slot_fits(block_tables[(int64_t)s * max_blocks_per_seq + p / block_size], block_size))
            return PA_ERR_INVALID;
    }
    for (int s = 0; s < num_seqs; ++s) {
        const int32_t p = num_cached[s];
        positions[s] = p;
        slot_mapping[s] =
            block_tables[(int64_t)s * max_blocks_per_seq + p / block_size] * block_size +
            p % block_size;
        context_lens[s] = p + 1;
    }
    return PA_OK;
}

size_t pa_rope_table_bytes(int max_positions, int head_dim) {
    if (max_positions <= 0 || head_dim <= 0 || (head_dim & 1)) return 0;
    return (size_t)max_positions * (head_dim / 2) * 2 * sizeof(float);
}

int pa_rope_table_init(void *device_table, int max_positions, int head_dim, double theta,
                       pa_stream_t stream) {
    const size_t bytes = pa_rope_table_bytes(max_positions, head_dim);
    if (!device_table || bytes == 0 || !aligned16(device_table) || !(theta > 1.0))
        return PA_ERR_INVALID;
    const int half = head_dim / 2;
    // theta_i = 1 / theta^(2i/d); angle = m * theta_i; cos/sin in double,
    // each rounded once to float ("Meta Llama source deep-dive", 3.3).
    std::vector<double> inv(half);
    for (int i = 0; i < half; ++i) inv[i] = 1.0 / pow(theta, (double)(2 * i) / (double)head_dim);
    std::vector<float> host((size_t)max_positions * half * 2);
    for (int m = 0; m < max_positions; ++m) {
        float *row = host.data() + (size_t)m * half * 2;
        for (int i = 0; i < half; ++i) {
            const double ang = (double)m * inv[i];
            row[2 * i] = (float)cos(ang);
            row[2 * i + 1] = (float)sin(ang);
        }
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(device_table, host.data(), bytes, cudaMemcpyHostToDevice, st) !=
            cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess) {
        cudaGetLastError();
        return PA_ERR_CUDA;
    }
    return PA_OK;
}

const char *pa_strerror(int code) {
    switch (code) {
        case PA_OK: return "ok";
        case PA_ERR_INVALID: return "invalid argument";
        case PA_ERR_UNSUPPORTED: return "unsupported shape or device";
        case PA_ERR_CUDA: return "CUDA runtime error";
        case PA_ERR_WORKSPACE: return "decode workspace too small";
        default: return "unknown error";
    }
}

int pa_check_device(void) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return PA_ERR_CUDA;
    }
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
        cudaGetLastError();
        return PA_ERR_CUDA;
    }
    return (major == 10 && minor == 3) ? PA_OK : PA_ERR_UNSUPPORTED;
}

}  // extern "C"
