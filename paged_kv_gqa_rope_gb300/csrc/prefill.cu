// Step a3: varlen causal prefill over the paged cache on the tcgen05 tensor
// cores ("Meta Llama source deep-dive", 3.5: scores = q k^T / sqrt(d),
// softmax in fp32, times V; 3.8: a cached prefix of start_pos keys is fully
// visible and the new tokens see each other causally; "personal chatgpt 22 -
// llama2 generate", section 2: M_ij = 0 for j <= i; "nano-vllm notes -
// Llama", prepare_prefill: cu_seqlens_q / cu_seqlens_k delimit the flattened
// stream and block_tables locate every key, prefix and new, in the cache).
//
// One CTA computes one 128-row tile of queries of one sequence and one Q
// head.  Row i of tile t sits at absolute position p + 128 t + i (p = cached
// prefix length) and sees keys 0 .. p + 128 t + i; key tiles of 128 keys
// (8 cache blocks) past the last row's position are never loaded, and only
// the tiles that reach past the first row's position are masked.
//
// Roles (192 threads):
//   warps 0-3  softmax: thread i owns query row i, which is TMEM lane i;
//   warp 4     producer: TMA loads of the Q tile and of the K / V tiles, one
//              16-token block (x two 64-column halves) at a time, gathered
//              through the block table into a 2-stage ring;
//   warp 5     MMA issuer (one thread) and TMEM owner.
// Tensor memory (512 columns): three 128-column score buffers S0..S2 and the
// output accumulator O at column 384.  Per key tile j:
//   S[j%3]  = Q . K_j^T                 tcgen05.mma, both operands in smem
//   softmax reads S[j%3], writes P = 2^(s*scale*log2e - m) as fp16 over it
//   O      += P . V_j                   tcgen05.mma, A = P from TMEM
// The running maximum m only moves when a tile raises it by more than 8 (in
// log2 units): P then stays <= 256 and O (in TMEM) is rescaled only on those
// tiles, after the previous P.V has finished.  The row sum accumulates the
// fp16-rounded P, so a constant V comes back exactly.
//
// Bound: tensor cores.  Algorithmic FLOPs = 4 * d * H * (number of visible
// (query, key) pairs).
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace pa {
namespace {

constexpr int kBM = 128;  // query rows per tile
constexpr int kBN = 128;  // keys per tile
constexpr int kBlocksPerTile = kBN / kBlockSize;
constexpr int kSoftmaxWarps = 4;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kThreads = 6 * 32;
constexpr int kTmemCols = 512;
constexpr int kOCol = 384;  // TMEM column of the O accumulator
constexpr float kRescaleThreshold = 8.0f;

struct PrefillArgs {
    const int32_t *cu_q;
    const int32_t *cu_k;
    const int32_t *block_tables;
    __half *out;
    int32_t *status;
    float scale_log2;
    int B, H, g, maxb, num_blocks, plane_k, plane_v, tiles_max, total_q;
};

template <int D>
struct PL {
    static constexpr int kHalf = kBM * 128;         // one 64-column half of a 128-row tile
    static constexpr int kTile = kHalf * (D / 64);  // Q, K or V tile bytes
    static constexpr int kQ = 0;
    static constexpr int kK = kQ + kTile;       // 2 stages
    static constexpr int kV = kK + 2 * kTile;   // 2 stages
    static constexpr int kBar = kV + 2 * kTile;
    static constexpr int kBytes = kBar + 256;
};

// barrier slots inside the barrier area
enum {
    B_Q = 0,
    B_KFULL = 1,    // 2
    B_KEMPTY = 3,   // 2
    B_VFULL = 5,    // 2
    B_VEMPTY = 7,   // 2
    B_VFIXED = 9,
    B_SFULL = 10,   // 3
    B_PREADY = 13,  // 3
    B_ODONE = 16,   // 3
    B_DRAIN = 19,
    B_COUNT = 20
};

__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int c0, int c1, int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
        "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }
__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap qmap,
                   const __grid_constant__ CUtensorMap kvmap, const PrefillArgs a) {
    using L = PL<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + L::kBar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar + B_COUNT);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // ---- which tile: heavy (late) query tiles first, heads fastest
    const int per_tile = a.H * a.B;
    const int t = a.tiles_max - 1 - (int)(blockIdx.x / per_tile);
    const int rem = (int)(blockIdx.x % per_tile);
    const int s = rem / a.H, h = rem - (rem / a.H) * a.H;
    const int q_begin = __ldg(a.cu_q + s), q_end = __ldg(a.cu_q + s + 1);
    const int k_len = __ldg(a.cu_k + s + 1) - __ldg(a.cu_k + s);
    const int L_q = q_end - q_begin;
    if (L_q < 0 || k_len < L_q || k_len > a.maxb * kBlockSize || q_begin < 0 ||
        q_end > a.total_q) {
        if (t == 0 && h == 0 && tid == 0) report(a.status, PA_DEV_BAD_LENGTH);
        return;
    }
    // Rows past the grid's tiles (L_q above the max_seqlen_q bound) are not
    // computed; the sequence is reported.
    if (L_q > a.tiles_max * kBM && t == 0 && h == 0 && tid == 0)
        report(a.status, PA_DEV_BAD_LENGTH);
    const int q0 = t * kBM;
    if (q0 >= L_q) return;  // whole CTA

    const int p = k_len - L_q;
    const int rows_valid = min(kBM, L_q - q0);
    const int kv_end = p + q0 + rows_valid;  // keys 0 .. kv_end-1 are visible to some row
    const int n = (kv_end + kBN - 1) / kBN;
    const int nblk_k = (k_len + kBlockSize - 1) / kBlockSize;
    const int kvh = h / a.g;
    const bool fix_tail = (k_len % kBlockSize) != 0 && (nblk_k - 1) / kBlocksPerTile == n - 1;

    if (tid == 0) {
        mbar_init(&bar[B_Q], 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar[B_KFULL + i], 1);
            mbar_init(&bar[B_KEMPTY + i], 1);
            mbar_init(&bar[B_VFULL + i], 1);
            mbar_init(&bar[B_VEMPTY + i], 1);
        }
        mbar_init(&bar[B_VFIXED], 1);
        for (int i = 0; i < 3; ++i) {
            mbar_init(&bar[B_SFULL + i], 1);
            mbar_init(&bar[B_PREADY + i], kSoftmaxWarps * 32);
            mbar_init(&bar[B_ODONE + i], 1);
        }
        mbar_init(&bar[B_DRAIN], 1);
        fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        tc::alloc(tmem_slot, kTmemCols);
        tc::relinquish();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kProducerWarp) {
        // ======================= producer: Q once, then K/V tiles
        const int32_t *row = a.block_tables + (int64_t)s * a.maxb;
        const int oob_row = a.num_blocks * kBlockSize;  // zero-filled by TMA
        auto block_row = [&](int j) -> int {            // cache row of lane's block in tile j
            const int lb = j * kBlocksPerTile + lane;
            if (lane >= kBlocksPerTile || lb >= nblk_k) return oob_row;
            const int blk = __ldg(row + lb);
            if (blk < 0 || blk >= a.num_blocks) {
                report(a.status, PA_DEV_BAD_BLOCK);
                return oob_row;
            }
            return blk * kBlockSize;
        };
        int ok = 1;
        if (lane == 0) {
            tma_prefetch_desc(&qmap);
            tma_prefetch_desc(&kvmap);
            mbar_arrive_expect_tx(&bar[B_Q], L::kTile);
            for (int hf = 0; hf < D / 64; ++hf)
                tma_load_4d(smem + L::kQ + hf * L::kHalf, &qmap, &bar[B_Q], 0, hf, h,
                            q_begin + q0);
        }
        int rows_cur = block_row(0);
        int issued = 0;
        for (int j = 0; j < n && ok; ++j) {
            const int rows_next = j + 1 < n ? block_row(j + 1) : 0;
            const int st = j & 1;
            const uint32_t ph = (j >> 1) & 1;
            int r8[kBlocksPerTile];
#pragma unroll
            for (int b = 0; b < kBlocksPerTile; ++b) r8[b] = __shfl_sync(0xffffffffu, rows_cur, b);
            if (lane == 0) {
                ok = mbar_wait(&bar[B_KEMPTY + st], ph ^ 1);
                if (ok) {
                    uint8_t *kt = smem + L::kK + st * L::kTile;
                    mbar_arrive_expect_tx(&bar[B_KFULL + st], L::kTile);
#pragma unroll
                    for (int b = 0; b < kBlocksPerTile; ++b)
                        for (int hf = 0; hf < D / 64; ++hf)
                            tma_load_5d(kt + hf * L::kHalf + b * kBlockSize * 128, &kvmap,
                                        &bar[B_KFULL + st], 0, hf, kvh, r8[b], a.plane_k);
                    ok = mbar_wait(&bar[B_VEMPTY + st], ph ^ 1);
                }
                if (ok) {
                    uint8_t *vt = smem + L::kV + st * L::kTile;
                    mbar_arrive_expect_tx(&bar[B_VFULL + st], L::kTile);
#pragma unroll
                    for (int b = 0; b < kBlocksPerTile; ++b)
                        for (int hf = 0; hf < D / 64; ++hf)
                            tma_load_5d(vt + hf * L::kHalf + b * kBlockSize * 128, &kvmap,
                                        &bar[B_VFULL + st], 0, hf, kvh, r8[b], a.plane_v);
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (ok && fix_tail && j == n - 1) {
                // Rows of the sequence's last block past k_len are never
                // written and may hold NaN bits; P is 0 there but 0 * NaN is
                // not, so they are cleared before P.V reads the tile.
                if (lane == 0) ok = mbar_wait(&bar[B_VFULL + st], ph);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (ok) {
                    uint8_t *vt = smem + L::kV + st * L::kTile;
                    const int b_in = (nblk_k - 1) % kBlocksPerTile;
                    const int r0 = k_len % kBlockSize;
                    const int nrows = kBlockSize - r0;
                    const int pieces = nrows * (D / 64) * 8;  // 16-byte pieces
                    for (int i = lane; i < pieces; i += 32) {
                        const int line = i >> 3, piece = i & 7;
                        const int hf = line / nrows, r = r0 + line % nrows;
                        *reinterpret_cast<uint4 *>(vt + hf * L::kHalf +
                                                   (b_in * kBlockSize + r) * 128 + piece * 16) =
                            make_uint4(0, 0, 0, 0);
                    }
                    tc::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bar[B_VFIXED]);
                }
            }
            rows_cur = rows_next;
            issued = j + 1;
        }
        if (lane == 0) {
            if (!ok) report(a.status, PA_DEV_TIMEOUT);
            // Leave no copy in flight: the last tiles' loads have landed.
            for (int j = max(0, issued - 2); j < issued; ++j) {
                mbar_wait(&bar[B_KFULL + (j & 1)], (j >> 1) & 1);
                mbar_wait(&bar[B_VFULL + (j & 1)], (j >> 1) & 1);
            }
        }
    } else if (warp == kMmaWarp) {
        // ======================= MMA issuer (one thread)
        if (lane == 0) {
            constexpr uint32_t kIdescQK = tc::idesc_f16(kBM, kBN, false, false);
            constexpr uint32_t kIdescPV = tc::idesc_f16(kBM, D, false, true);
            const uint32_t q_base = smem_u32(smem + L::kQ);
            bool ok = mbar_wait(&bar[B_Q], 0);
            auto issue_s = [&](int jj) -> bool {
                const int st = jj & 1;
                if (!mbar_wait(&bar[B_KFULL + st], (jj >> 1) & 1)) return false;
                tc::fence_after();
                const uint32_t k_base = smem_u32(smem + L::kK + st * L::kTile);
                const uint32_t d_tmem = tmem + (jj % 3) * kBN;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * L::kHalf + (kk & 3) * 32;
                    tc::mma_ss(d_tmem, tc::smem_desc_sw128(q_base + off, 16, 1024),
                               tc::smem_desc_sw128(k_base + off, 16, 1024), kIdescQK, kk > 0);
                }
                tc::commit(&bar[B_SFULL + jj % 3]);
                tc::commit(&bar[B_KEMPTY + st]);
                return true;
            };
            if (ok) ok = issue_s(0);
            if (ok && n > 1) ok = issue_s(1);
            for (int j = 0; j < n && ok; ++j) {
                const int b3 = j % 3, st = j & 1;
                ok = mbar_wait(&bar[B_PREADY + b3], (j / 3) & 1);
                if (!ok) break;
                ok = (fix_tail && j == n - 1) ? mbar_wait(&bar[B_VFIXED], 0)
                                              : mbar_wait(&bar[B_VFULL + st], (j >> 1) & 1);
                if (!ok) break;
                tc::fence_after();
                const uint32_t v_base = smem_u32(smem + L::kV + st * L::kTile);
                const uint32_t p_tmem = tmem + b3 * kBN;
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk)
                    tc::mma_ts(tmem + kOCol, p_tmem + kk * 8,
                               tc::smem_desc_sw128(v_base + kk * 16 * 128, L::kHalf, 1024),
                               kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
                tc::commit(&bar[B_ODONE + b3]);
                tc::commit(&bar[B_VEMPTY + st]);
                if (j + 2 < n) {
                    // S(j+2) overwrites the buffer P(j-1) was read from.
                    if (j >= 1) ok = mbar_wait(&bar[B_ODONE + (j - 1) % 3], ((j - 1) / 3) & 1);
                    if (ok) ok = issue_s(j + 2);
                }
            }
            if (!ok) report(a.status, PA_DEV_TIMEOUT);
            // Nothing of ours may still be running when the CTA frees TMEM.
            tc::commit(&bar[B_DRAIN]);
            mbar_wait(&bar[B_DRAIN], 0);
        }
        __syncwarp();
    } else {
        // ======================= softmax warps: thread = query row
        const int r = tid;
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        const int apos = p + q0 + r;
        const int key_lim = min(apos, k_len - 1);  // last key this row may see
        const float sl2 = a.scale_log2;
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < n; ++j) {
            const int b3 = j % 3;
            ok = __all_sync(0xffffffffu, mbar_wait(&bar[B_SFULL + b3], (j / 3) & 1));
            if (!ok) break;
            tc::fence_after();
            const uint32_t s_tmem = tmem + lane_base + b3 * kBN;
            uint32_t sr[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c) tc::ld32(s_tmem + c * 32, sr[c]);
            float mx = -INFINITY;
            const bool masked = j * kBN + kBN - 1 > p + q0;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    if (masked && j * kBN + c * 32 + i > key_lim) sr[c][i] = f2u(-INFINITY);
                    mx = fmaxf(mx, u2f(sr[c][i]));
                }
            }
            const float m_tile = mx * sl2;
            const bool raise = m_tile > m_used + kRescaleThreshold;
            float alpha = 1.f;
            if (raise) {
                alpha = ex2(m_used - m_tile);  // 0 on the first tile
                l *= alpha;
                m_used = m_tile;
            }
            if (j > 0 && __any_sync(0xffffffffu, raise)) {
                // O must hold P(j-1).V(j-1) before it is scaled.
                ok = __all_sync(0xffffffffu,
                                mbar_wait(&bar[B_ODONE + (j - 1) % 3], ((j - 1) / 3) & 1));
                if (!ok) break;
                tc::fence_after();
                const uint32_t o_tmem = tmem + lane_base + kOCol;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t orr[32];
                    tc::ld32(o_tmem + c * 32, orr);
#pragma unroll
                    for (int i = 0; i < 32; ++i) orr[i] = f2u(u2f(orr[i]) * alpha);
                    tc::st32(o_tmem + c * 32, orr);
                }
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float p0 = ex2(fmaf(u2f(sr[c][2 * i]), sl2, -m_used));
                    const float p1 = ex2(fmaf(u2f(sr[c][2 * i + 1]), sl2, -m_used));
                    const __half2 hp = __floats2half2_rn(p0, p1);
                    l += __low2float(hp) + __high2float(hp);
                    pk[i] = *reinterpret_cast<const uint32_t *>(&hp);
                }
                tc::st16(s_tmem + c * 16, pk);
            }
            tc::wait_st();
            tc::fence_before();
            mbar_arrive(&bar[B_PREADY + b3]);
        }
        if (ok)
            ok = __all_sync(0xffffffffu,
                            mbar_wait(&bar[B_ODONE + (n - 1) % 3], ((n - 1) / 3) & 1));
        if (ok) {
            tc::fence_after();
            const uint32_t o_tmem = tmem + lane_base + kOCol;
            const float inv = l > 0.f ? 1.f / l : 0.f;
            uint4 *dst = reinterpret_cast<uint4 *>(a.out +
                                                   ((int64_t)(q_begin + q0 + r) * a.H + h) * D);
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t orr[32];
                tc::ld32(o_tmem + c * 32, orr);
                if (r < rows_valid) {
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const __half2 hv = __floats2half2_rn(u2f(orr[v * 8 + 2 * e]) * inv,
                                                                 u2f(orr[v * 8 + 2 * e + 1]) * inv);
                            w[e] = *reinterpret_cast<const uint32_t *>(&hv);
                        }
                        dst[c * 4 + v] = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            }
        } else if (lane == 0) {
            report(a.status, PA_DEV_TIMEOUT);
        }
    }

    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (warp == kMmaWarp) tc::dealloc(tmem, kTmemCols);
}

// 4-D fp16 map of q or out [T][H][D]: {64, D/64, H, T}, box {64, 1, 1, 128}.
bool make_rows_map(CUtensorMap *map, const void *base, int T, int H, int D) {
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return false;
    cuuint64_t dims[4] = {64, (cuuint64_t)(D / 64), (cuuint64_t)H, (cuuint64_t)T};
    cuuint64_t strides[3] = {128, (cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
    cuuint32_t box[4] = {64, 1, 1, kBM};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, const_cast<void *>(base), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
int launch_prefill(const CUtensorMap &qmap, const CUtensorMap &kvmap, const PrefillArgs &a,
                   cudaStream_t st) {
    // At least 116 KB of shared memory keeps one CTA per SM, so no CTA
    // waits in tcgen05.alloc for another's 512 TMEM columns.
    const size_t smem = (PL<D>::kBytes > 116 * 1024 ? PL<D>::kBytes : 116 * 1024) + 1024;
    static std::mutex mu;
    static bool attr_set[64] = {false};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PA_ERR_CUDA;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!attr_set[dev]) {
            if (cudaFuncSetAttribute(prefill_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)smem) != cudaSuccess) {
                cudaGetLastError();
                return PA_ERR_CUDA;
            }
            attr_set[dev] = true;
        }
    }
    const int64_t grid = (int64_t)a.tiles_max * a.H * a.B;
    if (grid > 0x7fffffff) return PA_ERR_UNSUPPORTED;
    prefill_kernel<D><<<(unsigned)grid, kThreads, smem, st>>>(qmap, kvmap, a);
    return launch_status();
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" int pa_prefill_varlen(const void *q, int total_q, const pa_cache_t *cache, int layer,
                                 const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                                 const int32_t *block_tables, int max_blocks_per_seq,
                                 int num_seqs, int max_seqlen_q, int n_heads, int n_kv_heads,
                                 int head_dim, float scale, void *out, int32_t *dev_status,
                                 pa_stream_t stream) {
    if (n_heads <= 0 || n_kv_heads <= 0 || n_heads % n_kv_heads != 0 || num_seqs < 0 ||
        total_q < 0 || max_seqlen_q < 0 || max_blocks_per_seq <= 0 || !(scale >= 0.f))
        return PA_ERR_INVALID;
    if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (!cache_ok(cache, layer, n_kv_heads, head_dim)) return PA_ERR_INVALID;
    if (num_seqs == 0 || max_seqlen_q == 0 || total_q == 0) return PA_OK;
    if (!q || !out || !cu_seqlens_q || !cu_seqlens_k || !block_tables) return PA_ERR_INVALID;
    if (!aligned16(q) || !aligned16(out)) return PA_ERR_INVALID;

    CUtensorMap qmap, kvmap;
    if (!make_rows_map(&qmap, q, total_q, n_heads, head_dim) ||
        !make_cache_map(&kvmap, cache, 1, kBlockSize))
        return PA_ERR_CUDA;
    if (scale == 0.f) scale = 1.0f / sqrtf((float)head_dim);

    PrefillArgs a;
    a.cu_q = cu_seqlens_q;
    a.cu_k = cu_seqlens_k;
    a.block_tables = block_tables;
    a.out = static_cast<__half *>(out);
    a.status = dev_status;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.B = num_seqs;
    a.H = n_heads;
    a.g = n_heads / n_kv_heads;
    a.maxb = max_blocks_per_seq;
    a.num_blocks = cache->num_blocks;
    a.plane_k = layer;
    a.plane_v = cache->layers + layer;
    a.tiles_max = (max_seqlen_q + kBM - 1) / kBM;
    a.total_q = total_q;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return head_dim == 128 ? launch_prefill<128>(qmap, kvmap, a, st)
                           : launch_prefill<64>(qmap, kvmap, a, st);
}
