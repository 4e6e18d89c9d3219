// Steps a1 + a2: rotary embedding of the new tokens' Q/K in place and the
// append of their K/V to the paged cache through slot_mapping
// ("Meta Llama source deep-dive", 3.3 apply_rotary_emb and 3.5 step 2;
// "nano-vllm notes - Llama", slot_mapping).
//
// Two kernels do the same work.  Small batches: one thread moves one 16-byte
// piece (8 fp16 = 4 rotation pairs) of one head row.  A token has n_heads Q
// rows, n_kv_heads K rows and n_kv_heads V rows; consecutive threads take
// consecutive pieces, so every warp reads and writes whole 128-byte lines.
// The grid has one row of CTAs per token (blockIdx.y, and blockIdx.z past
// 65535 tokens), each CTA 256 pieces of it, so the row and piece of a thread
// come from shifts, not divisions (one piece per thread measured faster than
// two or four with their loads issued first).
// Batches of at least eight tokens per SM: the staged kernel below, whose bulk
// copies keep more bytes in flight than one 16-byte load per thread can
// (the 16-sequence prefill's 1.39 GB: 289 -> 237 us).  Both are bound by
// HBM: they read Q, K and V once and write Q, K, cache K and cache V once.
#include <algorithm>
#include <mutex>

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
    // This kernel is itself launched as a dependent: it reads and writes
    // nothing before the kernel ahead of it (the previous step's attention
    // kernel, which reads the cache and Q, or the step graph's input copy)
    // has finished.
    griddep_launch_dependents();
    griddep_wait();
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


// 1-D bulk copy global -> shared, completing on `bar` (size and both
// addresses multiples of 16 bytes).
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes,
                                          uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// The same work with the loads staged in shared memory: a CTA takes tokens
// t = blockIdx.x, + gridDim.x, ...; one thread brings a token's Q, K and V
// rows (three contiguous runs) into one of two stages with bulk copies while
// the CTA works on the other stage, so the loads in flight do not hold
// registers.  Each thread then rotates 16-byte pieces from shared memory and
// stores them as the per-piece kernel does.
template <int D>
__global__ void __launch_bounds__(kTokenThreads) rope_kv_write_staged_kernel(const RopeArgs a) {
    griddep_launch_dependents();
    griddep_wait();
    extern __shared__ __align__(16) uint8_t smem[];
    constexpr int kPieces = D / 8;
    const int H = a.n_heads, Hk = a.n_kv_heads, rows = H + 2 * Hk;
    const uint32_t qb = (uint32_t)H * D * 2, kb = (uint32_t)Hk * D * 2, stage = qb + 2 * kb;
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + 2 * stage);
    if (threadIdx.x == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        fence_barrier_init();
    }
    __syncthreads();
    auto issue = [&](int t, int s) {
        uint8_t *dst = smem + s * stage;
        mbar_arrive_expect_tx(&bar[s], stage);
        bulk_load(dst, a.q + (int64_t)t * H * D, qb, &bar[s]);
        bulk_load(dst + qb, a.k + (int64_t)t * Hk * D, kb, &bar[s]);
        bulk_load(dst + qb + kb, a.v + (int64_t)t * Hk * D, kb, &bar[s]);
    };
    int t = (int)blockIdx.x;
    if (t < a.num_tokens && threadIdx.x == 0) issue(t, 0);
    int k = 0;
    bool ok = true;
    for (; t < a.num_tokens; t += (int)gridDim.x, ++k) {
        const int s = k & 1;
        const int tn = t + (int)gridDim.x;
        if (threadIdx.x == 0 && tn < a.num_tokens) issue(tn, s ^ 1);
        // every thread of the CTA takes the same decision
        ok = __syncthreads_and(mbar_wait(&bar[s], (k >> 1) & 1));
        if (!ok) break;
        const int pos = __ldg(a.positions + t);
        const int slot = __ldg(a.slots + t);
        const bool pos_ok = pos >= 0 && pos < a.max_pos;
        const bool write_cache = slot >= 0 && slot < a.num_slots;
        if (threadIdx.x == 0) {
            if (!pos_ok)
                report(a.status, PA_DEV_BAD_POSITION);
            else if (slot >= a.num_slots)
                report(a.status, PA_DEV_BAD_SLOT);
        }
        if (pos_ok) {
            const uint4 *src = reinterpret_cast<const uint4 *>(smem + s * stage);
            const float4 *tab = reinterpret_cast<const float4 *>(a.table + (int64_t)pos * (D / 2));
            for (int i = threadIdx.x; i < rows * kPieces; i += blockDim.x) {
                const int row = i / kPieces, piece = i % kPieces;
                const uint4 x = src[i];
                if (row < H + Hk) {
                    const uint4 r =
                        rope_rotate8(x, __ldg(tab + piece * 2), __ldg(tab + piece * 2 + 1));
                    if (row < H) {
                        reinterpret_cast<uint4 *>(a.q + ((int64_t)t * H + row) * D)[piece] = r;
                    } else {
                        const int h = row - H;
                        reinterpret_cast<uint4 *>(a.k + ((int64_t)t * Hk + h) * D)[piece] = r;
                        if (write_cache)
                            reinterpret_cast<uint4 *>(a.kcache +
                                                      ((int64_t)slot * Hk + h) * D)[piece] = r;
                    }
                } else if (write_cache) {
                    const int h = row - H - Hk;
                    reinterpret_cast<uint4 *>(a.vcache + ((int64_t)slot * Hk + h) * D)[piece] = x;
                }
            }
        }
        __syncthreads();  // the stage may be refilled
    }
    if (!ok && threadIdx.x == 0) {
        report(a.status, PA_DEV_TIMEOUT);
        // leave no copy in flight: the stages that have one outstanding
        mbar_wait(&bar[k & 1], (k >> 1) & 1);
        if (t + (int)gridDim.x < a.num_tokens) mbar_wait(&bar[(k + 1) & 1], ((k + 1) >> 1) & 1);
    }
}

constexpr size_t kStagedRopeSmem = 100 * 1024;

// The staged kernels' shared-memory limit, raised once per device.
bool staged_attr_set() {
    static std::mutex mu;
    static bool done[64] = {false};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    std::lock_guard<std::mutex> lock(mu);
    if (done[dev]) return true;
    if (cudaFuncSetAttribute(rope_kv_write_staged_kernel<128>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kStagedRopeSmem) !=
            cudaSuccess ||
        cudaFuncSetAttribute(rope_kv_write_staged_kernel<64>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kStagedRopeSmem) !=
            cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    done[dev] = true;
    return true;
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

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // Staged loads for batches of at least eight tokens per SM (a prefill)
    // when two stages of a token's rows leave room for at least two CTAs per
    // SM; smaller batches (decode: a 256-sequence batch measured 7.5 us
    // per-piece against 8.5 us staged) spread each token's pieces over
    // several CTAs instead.
    const size_t stage = (size_t)(n_heads + 2 * n_kv_heads) * head_dim * 2;
    const size_t smem = 2 * stage + 16;
    if (num_tokens >= 8 * sm_count() && smem <= kStagedRopeSmem) {
        if (!staged_attr_set()) return PA_ERR_CUDA;
        int per_sm = 0;
        const void *fn = head_dim == 128 ? (const void *)rope_kv_write_staged_kernel<128>
                                         : (const void *)rope_kv_write_staged_kernel<64>;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kTokenThreads, smem) !=
                cudaSuccess ||
            per_sm < 1) {
            cudaGetLastError();
            return PA_ERR_CUDA;
        }
        const int grid = (int)std::min<int64_t>(num_tokens, (int64_t)sm_count() * per_sm);
        if (head_dim == 128)
            launch_dependent(rope_kv_write_staged_kernel<128>, dim3(grid), dim3(kTokenThreads),
                             smem, st, a);
        else
            launch_dependent(rope_kv_write_staged_kernel<64>, dim3(grid), dim3(kTokenThreads),
                             smem, st, a);
        return launch_status();
    }
    const dim3 grid = token_grid(num_tokens, (n_heads + 2 * n_kv_heads) * (head_dim / 8));
    if (head_dim == 128)
        launch_dependent(rope_kv_write_kernel<128>, grid, dim3(kTokenThreads), 0, st, a);
    else
        launch_dependent(rope_kv_write_kernel<64>, grid, dim3(kTokenThreads), 0, st, a);
    return launch_status();
}
