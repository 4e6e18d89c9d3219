// Steps a1 + a2: rotary embedding of the new tokens' Q/K in place and the
// append of their K/V to the paged cache through slot_mapping
// ("Meta Llama source deep-dive", 3.3 apply_rotary_emb and 3.5 step 2;
// "nano-vllm notes - Llama", slot_mapping).
//
// One thread moves one 16-byte piece (8 fp16 = 4 rotation pairs) of one head
// row.  A token has n_heads Q rows, n_kv_heads K rows and n_kv_heads V rows;
// consecutive threads take consecutive pieces, so every warp reads and writes
// whole 128-byte lines.  The grid has one row of CTAs per token (blockIdx.y,
// and blockIdx.z past 65535 tokens), each CTA 256 pieces of it, so the row
// and piece of a thread come from shifts, not divisions (one piece per
// thread measured faster than two or four with their loads issued first).  The kernel is
// bound by HBM: it reads Q, K and V once and writes Q, K, cache K and cache
// V once.
#include "common.cuh"
#include "internal.h"

namespace pa {
namespace {

struct RopeArgs {
    __half *q;
    __half *k;
    const __half *v;
    const int32_t *positions;
    const int32_t *slots;
    const float2 *table;  // [max_pos][d/2] {cos, sin}
    __half *kcache;       // K plane of the layer: [num_slots][Hk][d]
    __half *vcache;
    int64_t num_slots;
    int32_t *status;
    int num_tokens, n_heads, n_kv_heads, max_pos;
};

template <int D>
__global__ void __launch_bounds__(kTokenThreads) rope_kv_write_kernel(const RopeArgs a) {
    // The decode or prefill kernel that follows may start its set-up now; it
    // waits (griddepcontrol.wait) for this kernel's writes before using them.
    griddep_launch_dependents();
    constexpr int kPieces = D / 8;  // 16-byte pieces per head row
    const int rows = a.n_heads + 2 * a.n_kv_heads;
    const int t = (int)(blockIdx.z * gridDim.y + blockIdx.y);
    const int i = (int)(blockIdx.x * blockDim.x + threadIdx.x);  // piece within the token
    if (t >= a.num_tokens || i >= rows * kPieces) return;
    const int piece = i % kPieces;
    const int row = i / kPieces;

    const int pos = __ldg(a.positions + t);
    if (pos < 0 || pos >= a.max_pos) {
        if (row == 0 && piece == 0) report(a.status, PA_DEV_BAD_POSITION);
        return;
    }
    const int slot = __ldg(a.slots + t);
    const bool write_cache = slot >= 0 && slot < a.num_slots;
    if (slot >= a.num_slots && row == 0 && piece == 0) report(a.status, PA_DEV_BAD_SLOT);

    const int Hk = a.n_kv_heads;
    if (row < a.n_heads + Hk) {
        // Q or K row: rotate in place (and append K).
        const bool is_q = row < a.n_heads;
        __half *base = is_q ? a.q + ((int64_t)t * a.n_heads + row) * D
                            : a.k + ((int64_t)t * Hk + (row - a.n_heads)) * D;
        uint4 *p = reinterpret_cast<uint4 *>(base) + piece;
        const float4 *cs = reinterpret_cast<const float4 *>(a.table + (int64_t)pos * (D / 2) +
                                                            piece * 4);
        const uint4 r = rope_rotate8(*p, __ldg(cs), __ldg(cs + 1));
        *p = r;
        if (!is_q && write_cache) {
            const int h = row - a.n_heads;
            reinterpret_cast<uint4 *>(a.kcache + ((int64_t)slot * Hk + h) * D)[piece] = r;
        }
    } else if (write_cache) {
        const int h = row - a.n_heads - Hk;
        const uint4 x =
            __ldg(reinterpret_cast<const uint4 *>(a.v + ((int64_t)t * Hk + h) * D) + piece);
        reinterpret_cast<uint4 *>(a.vcache + ((int64_t)slot * Hk + h) * D)[piece] = x;
    }
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" int pa_rope_kv_write(void *q, void *k, const void *v, const int32_t *positions,
                                const int32_t *slot_mapping, int num_tokens, int n_heads,
                                int n_kv_heads, int head_dim, const void *rope_table,
                                int max_positions, const pa_cache_t *cache, int layer,
                                int32_t *dev_status, pa_stream_t stream) {
    if (num_tokens < 0 || n_heads <= 0 || n_kv_heads <= 0 || n_heads % n_kv_heads != 0 ||
        max_positions <= 0)
        return PA_ERR_INVALID;
    if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (!cache_ok(cache, layer, n_kv_heads, head_dim)) return PA_ERR_INVALID;
    if (num_tokens == 0) return PA_OK;
    if (!q || !k || !v || !positions || !slot_mapping || !rope_table) return PA_ERR_INVALID;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(rope_table))
        return PA_ERR_INVALID;
    if ((int64_t)num_tokens * (n_heads + 2 * n_kv_heads) * (head_dim / 8) > (int64_t)1 << 40)
        return PA_ERR_INVALID;

    RopeArgs a;
    a.q = static_cast<__half *>(q);
    a.k = static_cast<__half *>(k);
    a.v = static_cast<const __half *>(v);
    a.positions = positions;
    a.slots = slot_mapping;
    a.table = static_cast<const float2 *>(rope_table);
    a.kcache = cache_plane(cache, 0, layer);
    a.vcache = cache_plane(cache, 1, layer);
    a.num_slots = (int64_t)cache->num_blocks * cache->block_size;
    a.status = dev_status;
    a.num_tokens = num_tokens;
    a.n_heads = n_heads;
    a.n_kv_heads = n_kv_heads;
    a.max_pos = max_positions;

    const dim3 grid = token_grid(num_tokens, (n_heads + 2 * n_kv_heads) * (head_dim / 8));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (head_dim == 128)
        rope_kv_write_kernel<128><<<grid, kTokenThreads, 0, st>>>(a);
    else
        rope_kv_write_kernel<64><<<grid, kTokenThreads, 0, st>>>(a);
    return launch_status();
}
