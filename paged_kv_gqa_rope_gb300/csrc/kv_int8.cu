// The int8 KV pool ("Meta Llama source deep-dive", 8.4: a quantised KV
// cache; the scheme is this library's, see include/pa.h): allocation and
// the RoPE + append kernel that quantises each appended K/V row.
//
// Like rope_kv_write_kernel (same per-token grid), one thread handles one
// 16-byte piece (8 fp16 values) of one head row; the D/8 threads of a K or V
// row (consecutive lanes of one warp) reduce the row's absolute maximum with
// shuffles, then each writes its 8 codes and the first the row's scale.
#include <string.h>

#include "common.cuh"
#include "internal.h"

namespace pa {
namespace {

struct RopeI8Args {
    __half *q;
    __half *k;
    const __half *v;
    const int32_t *positions;
    const int32_t *slots;
    const float2 *table;  // [max_pos][d/2] {cos, sin}
    int8_t *kcodes;       // K code plane of the layer: [num_slots][Hk][d]
    int8_t *vcodes;
    float *kscales;       // K scale plane of the layer: [num_blocks][Hk][16]
    float *vscales;
    int64_t num_slots;
    int32_t *status;
    int num_tokens, n_heads, n_kv_heads, max_pos;
};

// One code: clamp(rint(x / scale)), ties to even, 0 for a zero scale.
__device__ __forceinline__ int code_of(float x, float scale) {
    if (!(scale > 0.f)) return 0;
    const int q = __float2int_rn(__fdiv_rn(x, scale));
    return max(-127, min(127, q));
}

template <int D>
__global__ void __launch_bounds__(256) rope_kv_write_i8_kernel(const RopeI8Args a) {
    griddep_launch_dependents();
    constexpr int kPieces = D / 8;  // 16-byte pieces per head row (a power of two <= 16)
    const int rows = a.n_heads + 2 * a.n_kv_heads;
    const int t = (int)(blockIdx.z * gridDim.y + blockIdx.y);
    if (t >= a.num_tokens) return;  // the whole CTA
    const int idx = (int)(blockIdx.x * blockDim.x + threadIdx.x);  // piece within the token
    // Threads past the token's last row (whole rows of them) still take part
    // in the row reductions below; they read row 0 and write nothing.
    const bool live = idx < rows * kPieces;
    const int i = live ? idx : idx % kPieces;
    const int piece = i % kPieces;
    const int row = i / kPieces;

    const int pos = __ldg(a.positions + t);
    const bool pos_ok = pos >= 0 && pos < a.max_pos;
    if (live && !pos_ok && row == 0 && piece == 0) report(a.status, PA_DEV_BAD_POSITION);
    const int slot = __ldg(a.slots + t);
    const bool write_cache = live && pos_ok && slot >= 0 && slot < a.num_slots;
    if (live && pos_ok && slot >= a.num_slots && row == 0 && piece == 0)
        report(a.status, PA_DEV_BAD_SLOT);

    const int Hk = a.n_kv_heads;
    uint4 x = make_uint4(0, 0, 0, 0);
    if (row < a.n_heads + Hk) {
        // Q or K row: rotate in place
        const bool is_q = row < a.n_heads;
        __half *base = is_q ? a.q + ((int64_t)t * a.n_heads + row) * D
                            : a.k + ((int64_t)t * Hk + (row - a.n_heads)) * D;
        uint4 *p = reinterpret_cast<uint4 *>(base) + piece;
        if (pos_ok) {
            const float4 *cs = reinterpret_cast<const float4 *>(a.table + (int64_t)pos * (D / 2) +
                                                                piece * 4);
            x = rope_rotate8(*p, __ldg(cs), __ldg(cs + 1));
            if (live) *p = x;
        }
    } else {
        const int h = row - a.n_heads - Hk;
        x = __ldg(reinterpret_cast<const uint4 *>(a.v + ((int64_t)t * Hk + h) * D) + piece);
    }
    // |x| maximum over the row's kPieces lanes (aligned groups of a warp)
    float v[8];
    {
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const __half2 h = *reinterpret_cast<const __half2 *>(&w[j]);
            v[2 * j] = __low2float(h);
            v[2 * j + 1] = __high2float(h);
        }
    }
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(v[j]));
#pragma unroll
    for (int off = kPieces / 2; off >= 1; off >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));

    if (row >= a.n_heads && write_cache) {
        const bool is_k = row < a.n_heads + Hk;
        const int h = is_k ? row - a.n_heads : row - a.n_heads - Hk;
        const float scale = __fdiv_rn(amax, 127.f);
        uint32_t lo = 0, hi = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            lo |= (uint32_t)(code_of(v[j], scale) & 0xff) << (8 * j);
            hi |= (uint32_t)(code_of(v[4 + j], scale) & 0xff) << (8 * j);
        }
        int8_t *codes = (is_k ? a.kcodes : a.vcodes) + ((int64_t)slot * Hk + h) * D;
        reinterpret_cast<uint2 *>(codes)[piece] = make_uint2(lo, hi);
        if (piece == 0) {
            const int64_t blk = slot / kBlockSize;
            (is_k ? a.kscales : a.vscales)[(blk * Hk + h) * kBlockSize + slot % kBlockSize] = scale;
        }
    }
}

size_t codes_bytes(int layers, int num_blocks, int block_size, int n_kv_heads, int head_dim) {
    return (size_t)2 * layers * num_blocks * block_size * n_kv_heads * head_dim;
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" size_t pa_cache_i8_bytes(int layers, int num_blocks, int block_size, int n_kv_heads,
                                    int head_dim) {
    if (layers <= 0 || num_blocks <= 0 || block_size <= 0 || n_kv_heads <= 0 || head_dim <= 0)
        return 0;
    const size_t c = (codes_bytes(layers, num_blocks, block_size, n_kv_heads, head_dim) + 255) &
                     ~(size_t)255;
    return c + (size_t)2 * layers * num_blocks * n_kv_heads * block_size * sizeof(float);
}

extern "C" int pa_alloc_cache_i8(pa_cache_i8_t *out, int layers, int num_blocks, int block_size,
                                 int n_kv_heads, int head_dim, void *device_base) {
    if (!out) return PA_ERR_INVALID;
    memset(out, 0, sizeof(*out));
    const size_t bytes = pa_cache_i8_bytes(layers, num_blocks, block_size, n_kv_heads, head_dim);
    if (bytes == 0) return PA_ERR_INVALID;
    if ((int64_t)num_blocks * block_size > INT32_MAX) return PA_ERR_INVALID;
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
    const size_t c = (codes_bytes(layers, num_blocks, block_size, n_kv_heads, head_dim) + 255) &
                     ~(size_t)255;
    out->codes = static_cast<int8_t *>(base);
    out->scales = reinterpret_cast<float *>(static_cast<uint8_t *>(base) + c);
    out->layers = layers;
    out->num_blocks = num_blocks;
    out->block_size = block_size;
    out->n_kv_heads = n_kv_heads;
    out->head_dim = head_dim;
    return PA_OK;
}

extern "C" int pa_free_cache_i8(pa_cache_i8_t *cache) {
    if (!cache) return PA_ERR_INVALID;
    int rc = PA_OK;
    if (cache->owns && cache->codes && cudaFree(cache->codes) != cudaSuccess) rc = PA_ERR_CUDA;
    memset(cache, 0, sizeof(*cache));
    return rc;
}

extern "C" int pa_rope_kv_write_i8(void *q, void *k, const void *v, const int32_t *positions,
                                   const int32_t *slot_mapping, int num_tokens, int n_heads,
                                   int n_kv_heads, int head_dim, const void *rope_table,
                                   int max_positions, const pa_cache_i8_t *cache, int layer,
                                   int32_t *dev_status, pa_stream_t stream) {
    if (num_tokens < 0 || n_heads <= 0 || n_kv_heads <= 0 || n_heads % n_kv_heads != 0 ||
        max_positions <= 0)
        return PA_ERR_INVALID;
    if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (!cache || !cache->codes || !cache->scales || layer < 0 || layer >= cache->layers ||
        cache->n_kv_heads != n_kv_heads || cache->head_dim != head_dim ||
        cache->block_size != kBlockSize || cache->num_blocks <= 0)
        return PA_ERR_INVALID;
    if (num_tokens == 0) return PA_OK;
    if (!q || !k || !v || !positions || !slot_mapping || !rope_table) return PA_ERR_INVALID;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(rope_table))
        return PA_ERR_INVALID;
    if ((int64_t)num_tokens * (n_heads + 2 * n_kv_heads) * (head_dim / 8) > (int64_t)1 << 40)
        return PA_ERR_INVALID;

    const int64_t slots = (int64_t)cache->num_blocks * kBlockSize;
    const int64_t code_plane = slots * n_kv_heads * head_dim;
    const int64_t scale_plane = (int64_t)cache->num_blocks * n_kv_heads * kBlockSize;
    RopeI8Args a;
    a.q = static_cast<__half *>(q);
    a.k = static_cast<__half *>(k);
    a.v = static_cast<const __half *>(v);
    a.positions = positions;
    a.slots = slot_mapping;
    a.table = static_cast<const float2 *>(rope_table);
    a.kcodes = cache->codes + (int64_t)layer * code_plane;
    a.vcodes = cache->codes + (int64_t)(cache->layers + layer) * code_plane;
    a.kscales = cache->scales + (int64_t)layer * scale_plane;
    a.vscales = cache->scales + (int64_t)(cache->layers + layer) * scale_plane;
    a.num_slots = slots;
    a.status = dev_status;
    a.num_tokens = num_tokens;
    a.n_heads = n_heads;
    a.n_kv_heads = n_kv_heads;
    a.max_pos = max_positions;

    const dim3 grid = token_grid(num_tokens, (n_heads + 2 * n_kv_heads) * (head_dim / 8));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (head_dim == 128)
        rope_kv_write_i8_kernel<128><<<grid, kTokenThreads, 0, st>>>(a);
    else
        rope_kv_write_i8_kernel<64><<<grid, kTokenThreads, 0, st>>>(a);
    return launch_status();
}
