// Host-side helpers shared by the translation units of libpa.
#pragma once

#include <utility>

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa.h"

namespace pa {

// Tokens per cache block the kernels are built for.
constexpr int kBlockSize = 16;

// Widest block table the kernels accept: a sequence's length bound
// max_blocks_per_seq * kBlockSize must fit in int32.
constexpr int kMaxBlocksPerSeq = INT32_MAX / kBlockSize;

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline bool cache_ok(const pa_cache_t *c, int layer, int n_kv_heads, int head_dim) {
    return c && c->base && aligned16(c->base) && c->block_size == kBlockSize &&
           c->n_kv_heads == n_kv_heads && c->head_dim == head_dim && layer >= 0 &&
           layer < c->layers && c->num_blocks > 0;
}

// Device pointer to element [kv][layer][0][0][0][0] of the pool.
inline __half *cache_plane(const pa_cache_t *c, int kv, int layer) {
    return static_cast<__half *>(c->base) + (int64_t)kv * c->kv_stride +
           (int64_t)layer * c->layer_stride;
}

// Launch-time error of the last kernel -> pa_status.
inline int launch_status() {
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

// Number of SMs of the current device (cached per device).
int sm_count();

// Launch `kernel` with programmatic stream serialization: it may start while
// the previous kernel in the stream finishes, and must call griddep_wait()
// before it reads anything that kernel writes.  An error is left for
// launch_status().
template <typename... Params, typename... Args>
inline void launch_dependent(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t st, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// cuTensorMapEncodeTiled obtained from the driver at run time (the library
// does not link libcuda, so it loads on machines without a GPU).
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled();

// 5-D fp16 tensor map over one K or V plane set of the pool, viewed as
//   dim0 = 64 elements of a row        (contiguous)
//   dim1 = head_dim / 64 halves        (stride 128 B)
//   dim2 = n_kv_heads                  (stride head_dim * 2 B)
//   dim3 = num_blocks * block_size rows (stride n_kv_heads * head_dim * 2 B)
//   dim4 = 2 * layers planes            (stride num_blocks * block_size * Hk * d * 2 B)
// with a box of {64, box_halves, 1, box_rows, 1} and 128-byte swizzle.
// Plane index of (kv, layer) is kv * layers + layer.  Returns false on error.
bool make_cache_map(CUtensorMap *map, const pa_cache_t *c, int box_halves, int box_rows);

// Grid of the per-token kernels (RoPE/append): x = chunks of kTokenThreads
// pieces of one token, y (and z past 65535 tokens) = token.
constexpr int kTokenThreads = 256;
inline dim3 token_grid(int num_tokens, int pieces_per_token) {
    const unsigned chunks = (unsigned)((pieces_per_token + kTokenThreads - 1) / kTokenThreads);
    const unsigned y = (unsigned)(num_tokens < 65535 ? num_tokens : 65535);
    const unsigned z = (unsigned)((num_tokens + 65534) / 65535);
    return dim3(chunks, y, z);
}
// The same view of one layer with dim4 = its 2 planes (K, V; stride
// kv_stride) and a box of {64, head_dim / 64, 1, block_size, 2}: a block's
// whole K tile, then its V tile, in one copy.
bool make_cache_pair_map(CUtensorMap *map, const pa_cache_t *c, int layer);

}  // namespace pa
