// Step a4: single-token GQA decode against the paged cache
// ("personal chatgpt 22 - llama2 generate", section 3: the new query attends
// to the whole cached history with no mask; "nano-vllm notes - Llama",
// prepare_decode: context_lens include the token just appended;
// "Meta Llama source deep-dive", 3.4 repeat_kv: Q head h reads KV head h/g).
//
// Work decomposition.  Every (sequence s, KV head h) pair owns
// ceil(context_lens[s] / 16) KV blocks and a few units (after them; before
// them in the int8 kernel) that stand for the pair's fixed cost (its merge
// and output, about the time of ten fp16 or eight int8 blocks' streaming);
// laid end to end, pair after pair, they form one line of W units.  The
// persistent grid of G CTAs cuts that line into G equal ranges, so every CTA
// has about the same work whatever the mix of context lengths (a CTA with
// many short pairs streams fewer blocks).  A CTA walks its range as segments (the part of one pair that
// falls in it; a segment of a pair's cost units alone has no block and is
// skipped).  A pair whose blocks lie inside one range is finished there; a
// pair whose blocks are cut by range ends is finished by the CTA that
// completes its last piece: each piece leaves (max, sum, unnormalised O) in
// the workspace (record slot 0 if the pair's blocks began before the CTA's
// range, 1 if they begin in it and go on past it), and the last to arrive
// merges the 2-3 pieces by an online softmax and resets the pair's arrival
// counter to zero; if the pieces of the others have all arrived when a CTA
// reaches the end of its last segment, that CTA closes the pair from its own
// partial results without leaving a record.
//
// Inside a CTA one producer warp streams the K and V block tiles (16 tokens x
// head_dim fp16 of one KV head; one TMA copy brings both) into a ring of
// shared-memory stages; four consumer warps take the blocks of a segment in
// turn (two CTAs per SM for the fp16 cache).  Each warp
// computes, with warp-level tensor-core MMAs,
//     S^T (16 tokens x 8 heads) = K (16 x d) . Q^T (d x 8 heads)
// so the g Q heads that share the KV head form the N = 8 dimension and each
// K/V byte is read once for the whole group; the online softmax runs on the
// accumulator fragments with warp shuffles; P is rounded to fp16 (the row sum
// accumulates the rounded values), transposed in registers (movmatrix) and
// multiplied into
//     O^T (d x 8 heads) += V^T (d x 16 tokens) . P^T (16 tokens x 8 heads).
// The four warps' (max, sum, O) are merged through shared memory at the end
// of each segment.
//
// The int8 cache (pa_decode_i8) runs the same kernel with I8 = true: the
// stages hold code tiles and scales, and each consumer warp builds the MMA
// fragments from the codes in registers (see the int8 branch below); four
// CTAs per SM.
//
// Bound: HBM.  Algorithmic bytes = sum_s context_lens[s] * Hk * d * 2 (K, V)
// * 2 B; everything else (Q, O, tables, partial records) is < 0.5 % of it.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace pa {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kMaxSeqs = 4096;
constexpr int kGroupPad = 8;   // MMA N: Q heads per KV head, padded
constexpr int kMaxGrid = 608;  // CTAs the workspace has record slots for (4 per SM)

struct DecodeArgs {
    const __half *q;              // [B][H][D]
    const int32_t *block_tables;  // [B][maxb]
    const int32_t *context_lens;  // [B]
    __half *out;                  // [B][H][D]
    int32_t *counters;            // [B][Hk] arrival counters (zero between calls)
    float *rec;                   // [grid][2][8][D + 4]: O (unnormalised), m, l
    int32_t *status;
    float scale_log2;             // scale * log2(e)
    int B, H, Hk, g, maxb, num_blocks;
};

// Shared memory of one ring stage.  fp16 cache: the K and V tiles of one
// (block, KV head) as TMA writes them (128-byte swizzle).  int8 cache: the
// K and V codes (16 rows of D bytes each; 128-byte swizzle at D = 128), and
// apart from them, in a ring of their own, the 16 K and 16 V scales.
template <int D, bool I8 = false>
struct Layout {
    static constexpr int kTileBytes = kBlockSize * D * 2;  // one fp16 K or V block tile
    static constexpr int kCodeBytes = kBlockSize * D;      // one int8 K or V block tile
    static constexpr int kStageBytes = I8 ? 2 * kCodeBytes : 2 * kTileBytes;
    static constexpr int kScaleBytes = I8 ? 2 * kBlockSize * 4 : 0;
    // int8: the segment's Q^T fragments [D/16][32 lanes][2 words], shared by
    // the consumer warps (read per block instead of held in registers)
    static constexpr int kQsmBytes = I8 ? (D / 16) * 32 * 8 : 0;
    static constexpr int kRec = D + 4;                     // floats per head record
};

// int8 codes enter the tensor core as fp16 code + kCodeBias (byte ^ 0x80,
// i.e. code + 128, as the low mantissa byte of 1024.0: exact); the bias is
// taken out of the fp32 results.
constexpr float kCodeBias = 1152.f;

// First block index of CTA c's range: floor(W * c / G).
__device__ __forceinline__ int64_t range_start(int64_t W, int c, int G) { return W * c / G; }

// The CTA whose range holds block index idx: the largest c with
// floor(W c / G) <= idx, i.e. ceil((idx + 1) G / W) - 1.
__device__ __forceinline__ int cta_of(int64_t idx, int64_t W, int G) {
    return (int)(((idx + 1) * G + W - 1) / W) - 1;
}

// Units of the line that stand for one pair's fixed cost: ten after its
// blocks for the fp16 kernel, eight before them for the int8 kernel (whose
// blocks stream twice as fast and whose merges cost more of them).  Before
// its blocks, the units fall to the CTA that holds the pair's first block,
// the CTA that closes or merges a cut pair at the end of its range: that
// measured better for the int8 kernel (ragged_decode 485 -> 463 us), after
// them better for the fp16 one (757 -> 753 us).  fp16 ragged_decode took
// 753, 740 and 742 us with 4, 10 and 16 units (gqa_decode_70b 88.6, 88.6
// and 89.4 us; mha_decode_7b 164.8, 164.4 and 164.5 us).
constexpr int kPairCost = 10;
constexpr int kPairCostI8 = 8;

// Segment of the line starting at `pos` (< end): its pair, its nu units and
// the nb blocks among them (blocks b0 .. b0 + nb - 1 of the pair, nb = 0 for
// a segment of cost units alone); the pair's blocks are the units
// [pair_start, pair_end), its kCost cost units before them (kFront) or
// after them.
struct Segment {
    int s, kvh, b0, nb, nu, ctx;
    int64_t pair_start, pair_end;
};

template <int kCost, bool kFront>
__device__ __forceinline__ Segment segment_at(int64_t pos, int64_t end, const int64_t *prefix,
                                              int B, const int32_t *context_lens) {
    int lo = 0, hi = B - 1;  // largest s with prefix[s] <= pos
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (prefix[mid] <= pos)
            lo = mid;
        else
            hi = mid - 1;
    }
    Segment g;
    g.s = lo;
    g.ctx = __ldg(context_lens + lo);
    const int nblk = (g.ctx + kBlockSize - 1) / kBlockSize;
    const int span = kCost + nblk;
    const int64_t rem = pos - prefix[lo];
    g.kvh = (int)(rem / span);
    const int u0 = (int)(rem - (int64_t)g.kvh * span);  // unit of the pair
    const int64_t base = prefix[lo] + (int64_t)g.kvh * span;
    const int lead = kFront ? kCost : 0;  // units before the blocks
    g.pair_start = base + lead;
    g.pair_end = g.pair_start + nblk;
    g.nu = (int)(min(end, base + span) - pos);
    const int first = max(u0, lead), last = min(u0 + g.nu, lead + nblk);  // units of blocks
    g.nb = max(0, last - first);
    g.b0 = min(first - lead, nblk);
    return g;
}

// Byte offset inside a K or V block tile written by TMA with 128-byte
// swizzle: row r (token) of the tile holds D/64 lines of 128 B; line
// index = r * (D/64) + half; the 16-byte piece p of a line is stored at
// position p ^ (line % 8).
template <int D>
__device__ __forceinline__ uint32_t tile_offset(int row, int piece16) {
    const int half = piece16 >> 3;
    const int line = row * (D / 64) + half;
    return (uint32_t)(line * 128 + (((piece16 & 7) ^ (line & 7)) << 4));
}

// Byte offset of 16-byte chunk c of row r of an int8 code tile: rows of
// 128 bytes with 128-byte swizzle at D = 128, plain rows at D = 64.
template <int D>
__device__ __forceinline__ uint32_t code_offset(int r, int c) {
    if constexpr (D == 128)
        return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
    else
        return (uint32_t)(r * D + c * 16);
}

// 4-D tiled load (the int8 code map) into shared memory.
__device__ __forceinline__ void tma_load_4d_u8(void *dst, const CUtensorMap *map, uint64_t *bar,
                                               int c0, int c1, int c2, int c3, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
        "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}

// L2 policy for data read once: its lines are the first to go, so that the
// small data read by every launch (context lengths, block tables, Q, the
// pieces' records) stays in L2 while the cache streams through.
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 5-D tiled load (the fp16 cache map) into shared memory with an L2 policy.
__device__ __forceinline__ void tma_load_5d_hint(void *dst, const CUtensorMap *map, uint64_t *bar,
                                                 int c0, int c1, int c2, int c3, int c4,
                                                 uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4),
        "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}

// 3-D tiled load (the int8 scale map) into shared memory.
// (No evict-first policy here: a block's 64-byte scale rows of two KV heads
// share a 128-byte L2 line, which the other head's copy then reads from L2;
// with the policy the int8 kernels read the scales twice from DRAM.)
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}

// int8: four CTAs per SM (96 registers; the Q fragments live in shared
// memory): the per-block consumer work, not the bytes in flight, bounds the
// int8 pipeline, so more consumer warps pay.
// Online-softmax merge factors of n partial results of head h, given as
// (max, sum) in column h of the rows of m and l (row stride kGroupPad):
// M = max_i m_i; f_i = 2^(m_i - M) replaces m_i (all zero when every m_i is
// -inf, an empty part); L = sum_i f_i l_i goes to l[h] and M to
// l[kGroupPad + h].  O = sum_i f_i O_i is then the merged numerator.
// Every merge of partial results (warps, pieces) sums in index order with
// explicit fused multiply-adds, so a pair's output has the same bits
// whichever CTA, and which of the merge paths, combines its pieces.
__device__ __forceinline__ float piece_factor(float m, float M) {
    return M == -INFINITY ? 0.f : ex2(m - M);
}
__device__ __forceinline__ void merge_factors(float *m, float *l, int h, int n) {
    float M = -INFINITY;
    for (int i = 0; i < n; ++i) M = fmaxf(M, m[i * kGroupPad + h]);
    float Lsum = 0.f;
    for (int i = 0; i < n; ++i) {
        const float f = piece_factor(m[i * kGroupPad + h], M);
        m[i * kGroupPad + h] = f;
        Lsum = __fmaf_rn(f, l[i * kGroupPad + h], Lsum);
    }
    l[h] = Lsum;
    l[kGroupPad + h] = M;
}

// 16-byte asynchronous copy global -> shared through L2 only (the source is
// written by other CTAs of the launch), and the wait for this thread's.
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void fence_acq_rel_gpu() {
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
}
__device__ __forceinline__ int ld_acquire_gpu(const int *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// The pair's output rows from its pieces' records, by one warp (the warp of
// the last piece to arrive, while the rest of its CTA goes on).  Per head:
// the pieces' maximum M (lanes load the pieces' maxima together), then, for
// pieces in groups of 32 (lane j holding piece i0 + j's factor 2^(m - M) and
// sum), the row sum and the O of the head's D columns (lane = column within
// each run of 32) accumulated in piece order, the O values of four pieces
// loaded at a time (two for the int8 kernel, whose registers are capped).
template <int D, bool I8>
__device__ void warp_merge_records(const DecodeArgs &a, const Segment &sg, int64_t W, int G,
                                   int lane) {
    constexpr int kRec = D + 4;
    constexpr int kRuns = D / 32;
    constexpr int kBatch = I8 ? 2 : 4;
    const int c_first = cta_of(sg.pair_start, W, G), c_last = cta_of(sg.pair_end - 1, W, G);
    const int nrec = c_last - c_first + 1;
    auto rec_of = [&](int i, int h) -> const float * {
        const int c = c_first + i;
        const int sl = sg.pair_start <= range_start(W, c, G) ? 0 : 1;
        return a.rec + ((int64_t)(c * 2 + sl) * kGroupPad + h) * kRec;
    };
    for (int h = 0; h < a.g; ++h) {
        float M = -INFINITY;
        for (int i0 = 0; i0 < nrec; i0 += 32)
            if (i0 + lane < nrec) M = fmaxf(M, __ldcg(rec_of(i0 + lane, h) + D));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        float Lsum = 0.f;
        float O[kRuns];
#pragma unroll
        for (int r = 0; r < kRuns; ++r) O[r] = 0.f;
        for (int i0 = 0; i0 < nrec; i0 += 32) {
            const int n = min(32, nrec - i0);
            float fi = 0.f, li = 0.f;
            if (lane < n) {
                const float *r = rec_of(i0 + lane, h);
                fi = piece_factor(__ldcg(r + D), M);
                li = __ldcg(r + D + 1);
            }
            for (int j0 = 0; j0 < n; j0 += kBatch) {
                float x[kBatch][kRuns];
#pragma unroll
                for (int jj = 0; jj < kBatch; ++jj) {
                    const float *r = rec_of(i0 + min(j0 + jj, n - 1), h);
#pragma unroll
                    for (int rr = 0; rr < kRuns; ++rr)
                        x[jj][rr] = j0 + jj < n ? __ldcg(r + rr * 32 + lane) : 0.f;
                }
#pragma unroll
                for (int jj = 0; jj < kBatch; ++jj) {
                    const float f = __shfl_sync(0xffffffffu, fi, (j0 + jj) & 31);
                    const float l = __shfl_sync(0xffffffffu, li, (j0 + jj) & 31);
                    if (j0 + jj < n) {
                        Lsum = __fmaf_rn(f, l, Lsum);
#pragma unroll
                        for (int rr = 0; rr < kRuns; ++rr) O[rr] = __fmaf_rn(f, x[jj][rr], O[rr]);
                    }
                }
            }
        }
#pragma unroll
        for (int rr = 0; rr < kRuns; ++rr)
            a.out[((int64_t)sg.s * a.H + sg.kvh * a.g + h) * D + rr * 32 + lane] =
                __float2half_rn(Lsum > 0.f ? O[rr] / Lsum : 0.f);
    }
}

template <int D, int NSTAGE, bool I8>
__global__ void __launch_bounds__(kThreads, I8 ? 4 : 2)
    decode_kernel(const __grid_constant__ CUtensorMap kvmap,
                  const __grid_constant__ CUtensorMap smap, const DecodeArgs a) {
    // Consumer warp w takes blocks w, w+4, ... of a segment, and segments end
    // with a barrier of all consumer warps.  With NSTAGE a multiple of the
    // warp count, every use of a stage within a segment belongs to the same
    // warp, so a warp never waits on a stage whose previous fill another warp
    // has not consumed yet (the mbarrier parity would alias that wait onto
    // the earlier, completed phase).
    static_assert(NSTAGE % kConsumerWarps == 0, "stages must be a multiple of consumer warps");
    constexpr int kCost = I8 ? kPairCostI8 : kPairCost;
    using L = Layout<D, I8>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *stages = smem;
    uint8_t *scale_ring = smem + NSTAGE * L::kStageBytes;  // int8: [NSTAGE][K 16, V 16] floats
    uint8_t *qsm = scale_ring + NSTAGE * L::kScaleBytes;      // int8: Q^T fragments
    uint64_t *full = reinterpret_cast<uint64_t *>(qsm + L::kQsmBytes);
    uint64_t *empty = full + NSTAGE;
    int *stage_bad = reinterpret_cast<int *>(empty + NSTAGE);
    float *sm_o = reinterpret_cast<float *>(stage_bad + NSTAGE);  // [4][8][D]
    float *sm_m = sm_o + kConsumerWarps * kGroupPad * D;           // [4][8]
    float *sm_l = sm_m + kConsumerWarps * kGroupPad;               // [4][8]
    float *sm_pm = sm_l + kConsumerWarps * kGroupPad;              // [4][8] pieces' (max,
    float *sm_pl = sm_pm + kConsumerWarps * kGroupPad;             // [4][8]  sum) per head
    int *sm_flag = reinterpret_cast<int *>(sm_pl + kConsumerWarps * kGroupPad);  // [4]
    int64_t *prefix = reinterpret_cast<int64_t *>(sm_flag + 4);    // [B + 1]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int B = a.B;
    const int cta = blockIdx.x;

    // -------- blocks per sequence (all KV heads) and their prefix sum
    for (int s = tid; s < B; s += kThreads) {
        const int ctx = __ldg(a.context_lens + s);
        int64_t n = 0;
        if (ctx >= 1 && ctx <= a.maxb * kBlockSize)
            n = (int64_t)((ctx + kBlockSize - 1) / kBlockSize + kCost) * a.Hk;
        else if (cta == 0)
            report(a.status, PA_DEV_BAD_LENGTH);
        prefix[s + 1] = n;
    }
    if (tid < NSTAGE) stage_bad[tid] = 0;
    if (tid == 0) {
        prefix[0] = 0;
        sm_flag[0] = sm_flag[1] = 0;
        for (int i = 0; i < NSTAGE; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        fence_barrier_init();
    }
    __syncthreads();
    if (warp == 0) {  // inclusive scan of prefix[1..B] by one warp
        int64_t carry = 0;
        for (int base = 1; base <= B; base += 32) {
            const int i = base + lane;
            int64_t v = i <= B ? prefix[i] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int64_t t = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += t;
            }
            if (i <= B) prefix[i] = v + carry;
            carry += __shfl_sync(0xffffffffu, v, 31);
        }
    }
    __syncthreads();
    // Everything above read only call metadata; Q and the cache may still be
    // being written by the RoPE/append kernel before this one.
    griddep_wait();
    // The kernel after this one (the next step's RoPE/append, the step
    // graph's output copy) may be launched now: it waits for this grid to
    // finish before it touches memory, and this grid's CTAs are all resident
    // (one persistent wave), so its launch latency hides under this kernel.
    griddep_launch_dependents();
    const int64_t W = prefix[B];
    // With fewer blocks than CTAs only the first W CTAs get a (one-block)
    // range, so that every range is non-empty and a pair cut into pieces
    // counts exactly one arrival per CTA between its first and last.
    const int G = (int)(W < (int64_t)gridDim.x ? W : (int64_t)gridDim.x);
    if (cta >= G) return;
    const int64_t start = range_start(W, cta, G), end = range_start(W, cta + 1, G);

    if (warp == kConsumerWarps) {
        // ================= producer warp: TMA block tiles into the ring
        if (lane == 0) {
            tma_prefetch_desc(&kvmap);
            if constexpr (I8) tma_prefetch_desc(&smap);
        }
        int gblk = 0;
        bool abort = false;
        const uint64_t pol = l2_evict_first();
        for (int64_t pos = start; pos < end && !abort;) {
            const Segment sg = segment_at<kCost, I8>(pos, end, prefix, B, a.context_lens);
            const int32_t *row = a.block_tables + (int64_t)sg.s * a.maxb + sg.b0;
            for (int w0 = 0; w0 < sg.nb && !abort; w0 += 32) {
                const int cnt = min(32, sg.nb - w0);
                const int my_blk = lane < cnt ? __ldg(row + w0 + lane) : 0;
                for (int j = 0; j < cnt; ++j) {
                    const int blk = __shfl_sync(0xffffffffu, my_blk, j);
                    const int stage = gblk % NSTAGE;
                    const uint32_t ph = (gblk / NSTAGE) & 1;
                    int ok = 1;
                    if (lane == 0) {
                        ok = mbar_wait(&empty[stage], ph ^ 1);
                        if (!ok) {
                            report(a.status, PA_DEV_TIMEOUT);
                        } else if (blk >= 0 && blk < a.num_blocks) {
                            // One copy brings the block's K and V tiles (the
                            // maps' outer dimension is the layer's K and V
                            // planes); the int8 scales come in a second.
                            uint8_t *dst = stages + stage * L::kStageBytes;
                            if constexpr (I8) {
                                mbar_arrive_expect_tx(&full[stage],
                                                      L::kStageBytes + L::kScaleBytes);
                                tma_load_4d_u8(dst, &kvmap, &full[stage], 0, sg.kvh,
                                               blk * kBlockSize, 0, pol);
                                tma_load_3d(scale_ring + stage * L::kScaleBytes, &smap,
                                            &full[stage], 0, blk * a.Hk + sg.kvh, 0);
                            } else {
                                mbar_arrive_expect_tx(&full[stage], L::kStageBytes);
                                tma_load_5d_hint(dst, &kvmap, &full[stage], 0, 0, sg.kvh,
                                                 blk * kBlockSize, 0, pol);
                            }
                        } else {
                            report(a.status, PA_DEV_BAD_BLOCK);
                            stage_bad[stage] = 1;
                            mbar_arrive(&full[stage]);
                        }
                    }
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok) {
                        abort = true;
                        break;
                    }
                    ++gblk;
                }
            }
            pos += sg.nu;
        }
        // Leave no copy in flight: wait (bounded) for the last stages issued.
        if (lane == 0) {
            for (int i = max(0, gblk - NSTAGE); i < gblk; ++i)
                mbar_wait(&full[i % NSTAGE], (i / NSTAGE) & 1);
        }
        return;
    }

    // ===================== consumer warps
    const int head = lane >> 2;  // B-operand column (Q head in group)
    const int quad = lane & 3;
    const int h0 = 2 * quad;     // accumulator columns held by this lane
    constexpr int kCons = kConsumerWarps * 32;
    int gblk = 0;
    for (int64_t pos = start; pos < end;) {
        const Segment sg = segment_at<kCost, I8>(pos, end, prefix, B, a.context_lens);
        const int s = sg.s, kvh = sg.kvh, b0 = sg.b0, nb = sg.nb, ctx = sg.ctx;
        if (nb == 0) {  // cost units alone
            pos += sg.nu;
            continue;
        }

        // Q^T fragments (B operand).  fp16 cache: Q[head][16kk + 2*quad + {0,1}]
        // and + 8.  int8 cache: the k order of the K fragments built from the
        // codes (i8_k_fragment), and qbias = kCodeBias * sum over d of Q for
        // this lane's two accumulator columns (heads h0, h0 + 1).
        uint32_t qb[D / 16][2];
        float qbias0 = 0.f, qbias1 = 0.f;
        {
            const bool hv = head < a.g;
            const uint32_t *qrow = reinterpret_cast<const uint32_t *>(
                a.q + ((int64_t)s * a.H + kvh * a.g + (hv ? head : 0)) * D);
            if constexpr (I8) {
                float part = 0.f;
#pragma unroll
                for (int m = 0; m < D / 64; ++m) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int d = 16 * ((D / 64) * quad + m) + 4 * i;
                        const uint2 w = hv ? __ldg(reinterpret_cast<const uint2 *>(qrow) + d / 4)
                                           : make_uint2(0u, 0u);
                        // Q[d], Q[d + 2] and Q[d + 1], Q[d + 3]; every consumer
                        // warp writes the same values, so no warp waits for another
                        st_shared_v2(smem_u32(qsm) + ((4 * m + i) * 32 + lane) * 8,
                                     __byte_perm(w.x, w.y, 0x5410), __byte_perm(w.x, w.y, 0x7632));
                        const float2 f0 = __half22float2(*reinterpret_cast<const __half2 *>(&w.x));
                        const float2 f1 = __half22float2(*reinterpret_cast<const __half2 *>(&w.y));
                        part += (f0.x + f0.y) + (f1.x + f1.y);
                    }
                }
                part += __shfl_xor_sync(0xffffffffu, part, 1);
                part += __shfl_xor_sync(0xffffffffu, part, 2);  // lanes 4h .. 4h+3: head h
                qbias0 = kCodeBias * __shfl_sync(0xffffffffu, part, 8 * quad);
                qbias1 = kCodeBias * __shfl_sync(0xffffffffu, part, 8 * quad + 4);
                __syncwarp();
            } else {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    qb[kk][0] = hv ? __ldg(qrow + kk * 8 + quad) : 0u;
                    qb[kk][1] = hv ? __ldg(qrow + kk * 8 + 4 + quad) : 0u;
                }
            }
        }
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
        float o[D / 16][4];
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
        // int8: sum over the last block's tokens of P as fed to P.V, per
        // column.  P.V on biased codes adds kCodeBias times it to O; it is
        // taken out again when O is rescaled for the next block, so O never
        // carries more than one block's bias.
        float pl0 = 0.f, pl1 = 0.f;

        bool abort = false;
        for (int j = warp; j < nb; j += kConsumerWarps) {
            const int gb = gblk + j;
            const int stage = gb % NSTAGE;
            if (!mbar_wait(&full[stage], (gb / NSTAGE) & 1)) {
                if (lane == 0) report(a.status, PA_DEV_TIMEOUT);
                abort = true;
                break;
            }
            const int bad = stage_bad[stage];
            const uint32_t kt = smem_u32(stages + stage * L::kStageBytes);
            const int tok = (b0 + j) * kBlockSize + head;  // token of score row `head`
            if constexpr (I8) {
                // This lane's codes, read once (the stage is then free again):
                // K rows head and head + 8, chunks (D/64) quad + m; V tokens
                // 2 quad + {0, 1, 8, 9}, the D/8 columns from head * D/8.
                uint32_t kw[2][D / 16];
                float ks0 = 0.f, ks1 = 0.f, vs0 = 0.f, vs1 = 0.f;
                if (!bad) {
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
#pragma unroll
                        for (int m = 0; m < D / 64; ++m) {
                            const uint4 x =
                                ld_shared_v4(kt + code_offset<D>(head + 8 * r, (D / 64) * quad + m));
                            kw[r][4 * m] = x.x ^ 0x80808080u;
                            kw[r][4 * m + 1] = x.y ^ 0x80808080u;
                            kw[r][4 * m + 2] = x.z ^ 0x80808080u;
                            kw[r][4 * m + 3] = x.w ^ 0x80808080u;
                        }
                    }
                    const uint32_t sc = smem_u32(scale_ring + stage * L::kScaleBytes) + head * 4;
                    ks0 = ld_shared_f32(sc);
                    ks1 = ld_shared_f32(sc + 32);
                    vs0 = ld_shared_f32(sc + kBlockSize * 4);
                    vs1 = ld_shared_f32(sc + kBlockSize * 4 + 32);
                }
                if (bad) {
                    __syncwarp();
                    if (lane == 0) {
                        stage_bad[stage] = 0;
                        mbar_arrive(&empty[stage]);
                    }
                } else {
                    // S^T on codes + kCodeBias (exact in fp16); the bias adds
                    // kCodeBias * sum(Q) to every score of a column.
                    float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t af[4] = {__byte_perm(kw[0][kk], 0x64u, 0x4240),
                                                __byte_perm(kw[1][kk], 0x64u, 0x4240),
                                                __byte_perm(kw[0][kk], 0x64u, 0x4341),
                                                __byte_perm(kw[1][kk], 0x64u, 0x4341)};
                        const uint2 qf = ld_shared_v2(smem_u32(qsm) + (kk * 32 + lane) * 8);
                        mma_16816(sc, af, qf.x, qf.y);
                    }
                    float x0 = (sc[0] - qbias0) * (ks0 * a.scale_log2);
                    float x1 = (sc[1] - qbias1) * (ks0 * a.scale_log2);
                    float x2 = (sc[2] - qbias0) * (ks1 * a.scale_log2);
                    float x3 = (sc[3] - qbias1) * (ks1 * a.scale_log2);
                    // a never-written slot's codes and scales may hold any bits
                    if (tok >= ctx) {
                        x0 = x1 = -INFINITY;
                        vs0 = 0.f;
                    }
                    if (tok + 8 >= ctx) {
                        x2 = x3 = -INFINITY;
                        vs1 = 0.f;
                    }
                    float bm0 = fmaxf(x0, x2), bm1 = fmaxf(x1, x3);
#pragma unroll
                    for (int off = 4; off < 32; off <<= 1) {
                        bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, off));
                        bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, off));
                    }
                    const float mn0 = fmaxf(m0, bm0), mn1 = fmaxf(m1, bm1);
                    const float al0 = ex2(m0 - mn0), al1 = ex2(m1 - mn1);
                    m0 = mn0;
                    m1 = mn1;
                    // the row sum adds P; P.V multiplies each token's P by its
                    // V scale (the codes stand for code * scale)
                    const float e0 = ex2(x0 - mn0), e1 = ex2(x1 - mn1);
                    const float e2 = ex2(x2 - mn0), e3 = ex2(x3 - mn1);
                    l0 = l0 * al0 + e0 + e2;
                    l1 = l1 * al1 + e1 + e3;
                    const __half2 p01 = __floats2half2_rn(e0 * vs0, e1 * vs0);
                    const __half2 p23 = __floats2half2_rn(e2 * vs1, e3 * vs1);
                    const uint32_t pb0 = movmatrix_trans(*reinterpret_cast<const uint32_t *>(&p01));
                    const uint32_t pb1 = movmatrix_trans(*reinterpret_cast<const uint32_t *>(&p23));
                    // V codes only now (fewer registers live at once), then
                    // the stage is free again
                    uint32_t vw[4][D / 32];
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        const int t = 2 * quad + (v & 1) + 8 * (v >> 1);
                        if constexpr (D == 128) {
                            const uint4 x = ld_shared_v4(kt + L::kCodeBytes + code_offset<D>(t, head));
                            vw[v][0] = x.x ^ 0x80808080u;
                            vw[v][1] = x.y ^ 0x80808080u;
                            vw[v][2] = x.z ^ 0x80808080u;
                            vw[v][3] = x.w ^ 0x80808080u;
                        } else {
                            const uint2 x = ld_shared_v2(kt + L::kCodeBytes + t * D + head * (D / 8));
                            vw[v][0] = x.x ^ 0x80808080u;
                            vw[v][1] = x.y ^ 0x80808080u;
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[stage]);
                    const float c0 = -kCodeBias * pl0 * al0, c1 = -kCodeBias * pl1 * al1;
#pragma unroll
                    for (int mt = 0; mt < D / 16; ++mt) {
                        o[mt][0] = fmaf(o[mt][0], al0, c0);
                        o[mt][1] = fmaf(o[mt][1], al1, c1);
                        o[mt][2] = fmaf(o[mt][2], al0, c0);
                        o[mt][3] = fmaf(o[mt][3], al1, c1);
                        // V^T rows head*D/8 + 2 mt (+1), tokens 2 quad + {0,1}
                        // (+8): byte 2 mt % 4 (+1) of word mt / 2 of each token
                        const uint32_t sel = (mt & 1) ? 0x7362u : 0x5140u;
                        const uint32_t t01 = __byte_perm(vw[0][mt >> 1], vw[1][mt >> 1], sel);
                        const uint32_t t89 = __byte_perm(vw[2][mt >> 1], vw[3][mt >> 1], sel);
                        const uint32_t af[4] = {__byte_perm(t01, 0x64u, 0x4140),
                                                __byte_perm(t01, 0x64u, 0x4342),
                                                __byte_perm(t89, 0x64u, 0x4140),
                                                __byte_perm(t89, 0x64u, 0x4342)};
                        mma_16816(o[mt], af, pb0, pb1);
                    }
                    // this block's column sums of P, on the tensor core: 1 . P^T
                    const uint32_t ones[4] = {0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u};
                    float ps[4] = {0.f, 0.f, 0.f, 0.f};
                    mma_16816(ps, ones, pb0, pb1);
                    pl0 = ps[0];
                    pl1 = ps[1];
                }
            } else {
                if (!bad) {
                    const uint32_t vt = kt + L::kTileBytes;
                    float sc[4] = {0.f, 0.f, 0.f, 0.f};
                    const int krow = (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        uint32_t af[4];
                        ldmatrix_x4(af, kt + tile_offset<D>(krow, kk * 2 + (lane >> 4)));
                        mma_16816(sc, af, qb[kk][0], qb[kk][1]);
                    }
                    float x0 = sc[0] * a.scale_log2, x1 = sc[1] * a.scale_log2;
                    float x2 = sc[2] * a.scale_log2, x3 = sc[3] * a.scale_log2;
                    if (tok >= ctx) x0 = x1 = -INFINITY;
                    if (tok + 8 >= ctx) x2 = x3 = -INFINITY;
                    float bm0 = fmaxf(x0, x2), bm1 = fmaxf(x1, x3);
#pragma unroll
                    for (int off = 4; off < 32; off <<= 1) {
                        bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, off));
                        bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, off));
                    }
                    const float mn0 = fmaxf(m0, bm0), mn1 = fmaxf(m1, bm1);
                    const float al0 = ex2(m0 - mn0), al1 = ex2(m1 - mn1);
                    m0 = mn0;
                    m1 = mn1;
                    const __half2 p01 = __floats2half2_rn(ex2(x0 - mn0), ex2(x1 - mn1));
                    const __half2 p23 = __floats2half2_rn(ex2(x2 - mn0), ex2(x3 - mn1));
                    l0 = l0 * al0 + __low2float(p01) + __low2float(p23);
                    l1 = l1 * al1 + __high2float(p01) + __high2float(p23);
                    const uint32_t pb0 = movmatrix_trans(*reinterpret_cast<const uint32_t *>(&p01));
                    const uint32_t pb1 = movmatrix_trans(*reinterpret_cast<const uint32_t *>(&p23));
                    const int vrow = (lane & 7) + (lane >> 4) * 8;
                    // Rows of V past the context (the tail of a sequence's last
                    // block) are never written and may hold any bits, NaN
                    // included; P is 0 there, but 0 * NaN is not, so those
                    // tokens' lanes of the V^T fragment are cleared.
                    const int valid = ctx - (b0 + j) * kBlockSize;  // tokens in this block
                    uint32_t keep01 = 0xffffffffu, keep89 = 0xffffffffu;
                    if (valid < kBlockSize) {
                        const int t0 = 2 * quad;
                        keep01 = (t0 < valid ? 0x0000ffffu : 0u) | (t0 + 1 < valid ? 0xffff0000u : 0u);
                        keep89 = (t0 + 8 < valid ? 0x0000ffffu : 0u) | (t0 + 9 < valid ? 0xffff0000u : 0u);
                    }
#pragma unroll
                    for (int mt = 0; mt < D / 16; ++mt) {
                        o[mt][0] *= al0;
                        o[mt][1] *= al1;
                        o[mt][2] *= al0;
                        o[mt][3] *= al1;
                        uint32_t af[4];
                        ldmatrix_x4_trans(af, vt + tile_offset<D>(vrow, mt * 2 + ((lane >> 3) & 1)));
                        af[0] &= keep01;
                        af[1] &= keep01;
                        af[2] &= keep89;
                        af[3] &= keep89;
                        mma_16816(o[mt], af, pb0, pb1);
                    }
                }
                __syncwarp();
                if (lane == 0) {
                    if (bad) stage_bad[stage] = 0;
                    mbar_arrive(&empty[stage]);
                }
            }
        }
        // A timed-out wait leaves the ring out of step: every consumer warp
        // learns of it at the barrier below and the CTA stops after this segment.
        if (__any_sync(0xffffffffu, abort) && lane == 0) atomicOr(sm_flag + 1, 1);
        gblk += nb;

#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, off);
            l1 += __shfl_xor_sync(0xffffffffu, l1, off);
        }
        if (lane < 4) {
            sm_m[warp * kGroupPad + h0] = m0;
            sm_m[warp * kGroupPad + h0 + 1] = m1;
            sm_l[warp * kGroupPad + h0] = l0;
            sm_l[warp * kGroupPad + h0 + 1] = l1;
        }
        float *ow = sm_o + (warp * kGroupPad + h0) * D;
        if constexpr (I8) {
            // rows head * D/8 + 2 mt and + 1 of O^T; the last block's bias out
            const float c0 = kCodeBias * pl0, c1 = kCodeBias * pl1;
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
                const int d = head * (D / 8) + 2 * mt;
                ow[d] = o[mt][0] - c0;
                ow[D + d] = o[mt][1] - c1;
                ow[d + 1] = o[mt][2] - c0;
                ow[D + d + 1] = o[mt][3] - c1;
            }
        } else {
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
                const int d = mt * 16 + head;
                ow[d] = o[mt][0];
                ow[D + d] = o[mt][1];
                ow[d + 8] = o[mt][2];
                ow[D + d + 8] = o[mt][3];
            }
        }
        // (a whole pair's segment starts at the pair's first block unless
        // cost units come before the blocks)
        const bool whole = I8 ? b0 == 0 && b0 + nb == sg.pair_end - sg.pair_start
                              : pos == sg.pair_start && pos + nb == sg.pair_end;
        // A cut pair: its pieces are those of CTAs c_first .. c_last.  On the
        // CTA's last segment, if every other piece has already arrived on the
        // pair's counter, this piece is the last, and the pair is merged from
        // this CTA's partial results and the other pieces' records, with no
        // record, fence or arrival of its own.  (The counter is read here; its
        // value is needed after the barrier.)
        int c_first = 0, c_last = 0, nrec = 1, arrived = -1;
        bool may_close = false;
        if (!whole) {
            c_first = cta_of(sg.pair_start, W, G);
            c_last = cta_of(sg.pair_end - 1, W, G);
            nrec = c_last - c_first + 1;
            may_close = pos + sg.nu == end && nrec <= kConsumerWarps;
            if (may_close && tid == 0) arrived = ld_acquire_gpu(a.counters + s * a.Hk + kvh);
        }
        named_barrier_sync(1, kCons);
        abort = sm_flag[1] != 0;
        if (tid < a.g) merge_factors(sm_m, sm_l, tid, kConsumerWarps);
        if (tid == 0) sm_flag[2] = may_close && arrived == nrec - 1;
        named_barrier_sync(1, kCons);
        const bool close = sm_flag[2] != 0;
        const bool last_seg = pos + sg.nu == end;

        if (whole) {
            for (int idx = tid; idx < a.g * D; idx += kCons) {
                const int h = idx / D, d = idx - (idx / D) * D;
                float O = 0.f;
#pragma unroll
                for (int wv = 0; wv < kConsumerWarps; ++wv)
                    O = __fmaf_rn(sm_m[wv * kGroupPad + h], sm_o[(wv * kGroupPad + h) * D + d], O);
                const float Lsum = sm_l[h];
                a.out[((int64_t)s * a.H + kvh * a.g + h) * D + d] =
                    __float2half_rn(Lsum > 0.f ? O / Lsum : 0.f);
            }
            named_barrier_sync(1, kCons);  // the smem merge area is free again
        } else {
            // A piece of a cut pair.  Unless it closes the pair, it leaves the
            // CTA's record of it (slot 0 for the CTA's first segment, 1 for its
            // last) and arrives on the pair's counter after a release fence
            // (one thread, after the barrier that follows every thread's
            // record stores); the piece that arrives last merges the pair.
            bool merge = close;
            if (!close) {
                // slot 0 for a pair whose blocks began before this range (with
                // cost units after the blocks: this CTA's first segment)
                const int slot = (I8 ? sg.pair_start <= start : pos == start) ? 0 : 1;
                float *myrec = a.rec + ((int64_t)(cta * 2 + slot) * kGroupPad) * L::kRec;
                for (int idx = tid; idx < a.g * D; idx += kCons) {
                    const int h = idx / D, d = idx - (idx / D) * D;
                    float O = 0.f;
#pragma unroll
                    for (int wv = 0; wv < kConsumerWarps; ++wv)
                        O = __fmaf_rn(sm_m[wv * kGroupPad + h], sm_o[(wv * kGroupPad + h) * D + d],
                                      O);
                    float *r = myrec + h * L::kRec;
                    r[d] = O;
                    if (d == 0) {
                        r[D] = sm_l[kGroupPad + h];
                        r[D + 1] = sm_l[h];
                    }
                }
                named_barrier_sync(1, kCons);
                if (!last_seg) {
                    // Mid-range: warp 0 alone arrives (and, in the rare case
                    // that this piece is the last, merges the pair from the
                    // records) while the other warps go on with the next
                    // segment.
                    if (warp == 0) {
                        int last = 0;
                        if (lane == 0) {
                            fence_acq_rel_gpu();
                            const int prev = atomicAdd(a.counters + s * a.Hk + kvh, 1);
                            last = prev == nrec - 1;
                            if (last) fence_acq_rel_gpu();
                        }
                        if (__shfl_sync(0xffffffffu, last, 0)) {
                            warp_merge_records<D, I8>(a, sg, W, G, lane);
                            if (lane == 0) a.counters[s * a.Hk + kvh] = 0;
                        }
                    }
                } else {
                    // The CTA's last segment: every warp waits for the arrival.
                    if (tid == 0) {
                        fence_acq_rel_gpu();
                        const int prev = atomicAdd(a.counters + s * a.Hk + kvh, 1);
                        const int last = prev == nrec - 1;
                        if (last) fence_acq_rel_gpu();
                        sm_flag[0] = last;
                    }
                    named_barrier_sync(1, kCons);
                    merge = sm_flag[0] != 0;
                }
            }
            if (merge && nrec <= kConsumerWarps) {
                // Pieces i = 0 .. nrec-1 of the pair (CTA c_first + i), from
                // their records, except this CTA's own when it closes the pair:
                // (max, sum) per head from the merge factors above, O from the
                // four warps' partial O.
                if constexpr (!I8) {
                    // fp16: each thread loads the records' O values of its
                    // elements into registers first, then their (max, sum), so
                    // the loads overlap.
                    const int own = close ? cta - c_first : -1;
                    constexpr int kEl = kGroupPad * D / kCons;
                    constexpr int kPass = kEl;
#pragma unroll 1
                    for (int k0 = 0; k0 < kEl; k0 += kPass) {
                        float x[kConsumerWarps][kPass];
#pragma unroll
                        for (int i = 0; i < kConsumerWarps; ++i) {
                            const int c = c_first + i;
                            const int sl = sg.pair_start <= range_start(W, c, G) ? 0 : 1;
                            const float *pb = a.rec + (int64_t)(c * 2 + sl) * kGroupPad * L::kRec;
#pragma unroll
                            for (int k = 0; k < kPass; ++k) {
                                const int idx = tid + (k0 + k) * kCons, h = idx / D,
                                          d = idx - h * D;
                                x[i][k] = i < nrec && i != own && idx < a.g * D
                                              ? __ldcg(pb + h * L::kRec + d)
                                              : 0.f;
                            }
                        }
                        if (k0 == 0) {
                            if (tid < nrec * a.g) {
                                const int i = tid / a.g, h = tid - (tid / a.g) * a.g;
                                float pm, pl;
                                if (i == own) {
                                    pm = sm_l[kGroupPad + h];
                                    pl = sm_l[h];
                              } else {
                                    const int c = c_first + i;
                                    const int sl = sg.pair_start <= range_start(W, c, G) ? 0 : 1;
                                    const float *r =
                                        a.rec + ((int64_t)(c * 2 + sl) * kGroupPad + h) * L::kRec;
                                    pm = __ldcg(r + D);
                                    pl = __ldcg(r + D + 1);
                                }
                                sm_pm[i * kGroupPad + h] = pm;
                                sm_pl[i * kGroupPad + h] = pl;
                            }
                            named_barrier_sync(1, kCons);
                            if (tid < a.g) merge_factors(sm_pm, sm_pl, tid, nrec);
                            named_barrier_sync(1, kCons);
                        }
#pragma unroll
                        for (int k = 0; k < kPass; ++k) {
                            const int idx = tid + (k0 + k) * kCons, h = idx / D, d = idx - h * D;
                            if (idx < a.g * D) {
                                float Oown = 0.f;
                                if (own >= 0) {
#pragma unroll
                                    for (int wv = 0; wv < kConsumerWarps; ++wv)
                                        Oown = __fmaf_rn(sm_m[wv * kGroupPad + h],
                                                         sm_o[(wv * kGroupPad + h) * D + d], Oown);
                                }
                                float O = 0.f;
#pragma unroll
                                for (int i = 0; i < kConsumerWarps; ++i)
                                    if (i < nrec)
                                        O = __fmaf_rn(sm_pm[i * kGroupPad + h],
                                                      i == own ? Oown : x[i][k], O);
                                const float Lsum = sm_pl[h];
                                a.out[((int64_t)s * a.H + kvh * a.g + h) * D + d] =
                                    __float2half_rn(Lsum > 0.f ? O / Lsum : 0.f);
                            }
                        }
                    }
                  } else {
                    // int8 (registers capped for four CTAs per SM): this CTA's own
                    // O goes to registers first; the records' O rows are then
                    // copied into the partial-O area (piece i's g rows where warp
                    // i's were) by asynchronous copies, one round trip for all of
                    // them, beside the loads of their (max, sum).
                    const int own = close ? cta - c_first : -1;
                    constexpr int kEl = kGroupPad * D / kCons;
                    float oown[kEl];
#pragma unroll
                    for (int k = 0; k < kEl; ++k) {
                        const int idx = tid + k * kCons, h = idx / D, d = idx - h * D;
                        oown[k] = 0.f;
                        if (own >= 0 && idx < a.g * D) {
#pragma unroll
                            for (int wv = 0; wv < kConsumerWarps; ++wv)
                                oown[k] = __fmaf_rn(sm_m[wv * kGroupPad + h],
                                                    sm_o[(wv * kGroupPad + h) * D + d], oown[k]);
                        }
                    }
                    named_barrier_sync(1, kCons);  // the partial O is read: its area is free
                    constexpr int kChunks = D / 4;  // 16-byte pieces of a row
                    for (int i = 0; i < nrec; ++i) {
                        if (i == own) continue;
                        const int c = c_first + i;
                        const int sl = sg.pair_start <= range_start(W, c, G) ? 0 : 1;
                        const float *pb = a.rec + (int64_t)(c * 2 + sl) * kGroupPad * L::kRec;
                        for (int ch = tid; ch < a.g * kChunks; ch += kCons) {
                            const int h = ch / kChunks, d = (ch - h * kChunks) * 4;
                            cp_async16(sm_o + (i * kGroupPad + h) * D + d, pb + h * L::kRec + d);
                        }
                    }
                    cp_async_commit();
                    if (tid < nrec * a.g) {
                        const int i = tid / a.g, h = tid - (tid / a.g) * a.g;
                        float pm, pl;
                        if (i == own) {
                            pm = sm_l[kGroupPad + h];
                            pl = sm_l[h];
                        } else {
                            const int c = c_first + i;
                            const int sl = sg.pair_start <= range_start(W, c, G) ? 0 : 1;
                            const float *r =
                                a.rec + ((int64_t)(c * 2 + sl) * kGroupPad + h) * L::kRec;
                            pm = __ldcg(r + D);
                            pl = __ldcg(r + D + 1);
                        }
                        sm_pm[i * kGroupPad + h] = pm;
                        sm_pl[i * kGroupPad + h] = pl;
                    }
                    cp_async_wait_all();
                    named_barrier_sync(1, kCons);
                    if (tid < a.g) merge_factors(sm_pm, sm_pl, tid, nrec);
                    named_barrier_sync(1, kCons);
#pragma unroll
                    for (int k = 0; k < kEl; ++k) {
                        const int idx = tid + k * kCons, h = idx / D, d = idx - h * D;
                        if (idx < a.g * D) {
                            float O = 0.f;
#pragma unroll
                            for (int i = 0; i < kConsumerWarps; ++i)
                                if (i < nrec)
                                    O = __fmaf_rn(sm_pm[i * kGroupPad + h],
                                                  i == own ? oown[k]
                                                           : sm_o[(i * kGroupPad + h) * D + d],
                                                  O);
                            const float Lsum = sm_pl[h];
                            a.out[((int64_t)s * a.H + kvh * a.g + h) * D + d] =
                                __float2half_rn(Lsum > 0.f ? O / Lsum : 0.f);
                        }
                    }
                }
                if (tid == 0) a.counters[s * a.Hk + kvh] = 0;
            } else if (merge) {
                // More pieces (a long pair over a narrow grid), from the
                // records: one element at a time.
                for (int idx = tid; idx < a.g * D; idx += kCons) {
                    const int h = idx / D, d = idx - (idx / D) * D;
                    auto rec_of = [&](int c) -> const float * {
                        const int sl = sg.pair_start <= range_start(W, c, G) ? 0 : 1;
                        return a.rec + ((int64_t)(c * 2 + sl) * kGroupPad + h) * L::kRec;
                    };
                    float M = -INFINITY;
                    for (int c = c_first; c <= c_last; ++c) M = fmaxf(M, __ldcg(rec_of(c) + D));
                    float O = 0.f, Lsum = 0.f;
                    for (int c = c_first; c <= c_last; ++c) {
                        const float *r = rec_of(c);
                        const float f = piece_factor(__ldcg(r + D), M);
                        Lsum = __fmaf_rn(f, __ldcg(r + D + 1), Lsum);
                        O = __fmaf_rn(f, __ldcg(r + d), O);
                    }
                    a.out[((int64_t)s * a.H + kvh * a.g + h) * D + d] =
                        __float2half_rn(Lsum > 0.f ? O / Lsum : 0.f);
                }
                if (tid == 0) a.counters[s * a.Hk + kvh] = 0;
            }
        }
        pos += sg.nu;
        if (abort) break;
    }
}

template <int D, int NSTAGE, bool I8>
size_t decode_smem_bytes(int B) {
    return 1024 + (size_t)NSTAGE * Layout<D, I8>::kStageBytes +
           (size_t)NSTAGE * Layout<D, I8>::kScaleBytes + Layout<D, I8>::kQsmBytes +
           2 * NSTAGE * sizeof(uint64_t) +
           NSTAGE * sizeof(int) + (size_t)kConsumerWarps * kGroupPad * (D + 4) * sizeof(float) +
           4 * sizeof(int) + 8 + (size_t)(B + 1) * sizeof(int64_t);
}

constexpr int kStages = 8;

template <int D, int NSTAGE, bool I8>
int launch_decode_stages(const CUtensorMap &map, const CUtensorMap &smap, const DecodeArgs &a,
                         int max_grid, cudaStream_t st) {
    const size_t smem = decode_smem_bytes<D, NSTAGE, I8>(a.B);
    // The kernel may use up to the shared memory of kMaxSeqs sequences; the
    // limit is raised once per device.  The grid is sized from this call's
    // shared memory, so small batches get more CTAs (bytes in flight) per SM.
    static std::mutex mu;
    static bool attr_set[64] = {false};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PA_ERR_CUDA;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!attr_set[dev]) {
            if (cudaFuncSetAttribute(decode_kernel<D, NSTAGE, I8>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)decode_smem_bytes<D, NSTAGE, I8>(kMaxSeqs)) !=
                cudaSuccess) {
                cudaGetLastError();
                return PA_ERR_CUDA;
            }
            attr_set[dev] = true;
        }
    }
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_kernel<D, NSTAGE, I8>,
                                                      kThreads, smem) != cudaSuccess ||
        per_sm < 1) {
        cudaGetLastError();
        return PA_ERR_CUDA;
    }
    const int grid = min(sm_count() * per_sm, max_grid);
    if (grid < 1) return PA_ERR_CUDA;
    launch_dependent(decode_kernel<D, NSTAGE, I8>, dim3(grid), dim3(kThreads), smem, st, map, smap,
                     a);
    return launch_status();
}

template <int D>
int launch_decode(const CUtensorMap &map, const DecodeArgs &a, int max_grid, cudaStream_t st) {
    // (no scale map on the fp16 path: the kernel never reads it)
    // 8 stages of 8 KB at d=128 and two CTAs per SM (the register budget
    // allows two) keep 128 KB of K/V in flight per SM; 4 stages, or 12-16
    // stages at one CTA per SM, measured slower on all decode workloads.
    return launch_decode_stages<D, kStages, false>(map, map, a, max_grid, st);
}

// int8 cache: a stage holds half the bytes; 8 stages at four CTAs per SM.
constexpr int kStagesI8 = 8;

size_t counters_bytes(int B, int Hk) {
    return ((size_t)B * Hk * sizeof(int32_t) + 255) & ~(size_t)255;
}
size_t cta_record_bytes(int D) { return (size_t)2 * kGroupPad * (D + 4) * sizeof(float); }

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" size_t pa_decode_workspace_bytes(int num_seqs, int n_heads, int n_kv_heads,
                                            int head_dim) {
    if (num_seqs <= 0 || n_heads <= 0 || n_kv_heads <= 0 || head_dim <= 0) return 0;
    return counters_bytes(num_seqs, n_kv_heads) + (size_t)kMaxGrid * cta_record_bytes(head_dim);
}

namespace pa {
namespace {

// The argument checks of pa_decode that do not involve the workspace, in
// the order pa_decode makes them.  PA_OK with num_seqs == 0 means "nothing
// to do".
int check_decode_args(const void *q, const pa_cache_t *cache, int layer,
                      const int32_t *block_tables, int max_blocks_per_seq,
                      const int32_t *context_lens, int num_seqs, int n_heads, int n_kv_heads,
                      int head_dim, float scale, const void *out) {
    if (num_seqs < 0 || n_heads <= 0 || n_kv_heads <= 0 || n_heads % n_kv_heads != 0 ||
        max_blocks_per_seq <= 0 || max_blocks_per_seq > kMaxBlocksPerSeq || !(scale >= 0.f))
        return PA_ERR_INVALID;
    if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (n_heads / n_kv_heads > kGroupPad || num_seqs > kMaxSeqs) return PA_ERR_UNSUPPORTED;
    if (!cache_ok(cache, layer, n_kv_heads, head_dim)) return PA_ERR_INVALID;
    if (num_seqs == 0) return PA_OK;
    if (!q || !block_tables || !context_lens || !out) return PA_ERR_INVALID;
    if (!aligned16(q) || !aligned16(out)) return PA_ERR_INVALID;
    return PA_OK;
}

}  // namespace
}  // namespace pa

extern "C" int pa_decode(const void *q, const pa_cache_t *cache, int layer,
                         const int32_t *block_tables, int max_blocks_per_seq,
                         const int32_t *context_lens, int num_seqs, int n_heads, int n_kv_heads,
                         int head_dim, float scale, void *workspace, size_t workspace_bytes,
                         void *out, int32_t *dev_status, pa_stream_t stream) {
    const int rc = check_decode_args(q, cache, layer, block_tables, max_blocks_per_seq,
                                     context_lens, num_seqs, n_heads, n_kv_heads, head_dim, scale,
                                     out);
    if (rc != PA_OK || num_seqs == 0) return rc;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return PA_ERR_INVALID;
    const size_t cnt = counters_bytes(num_seqs, n_kv_heads);
    if (workspace_bytes < cnt + cta_record_bytes(head_dim)) return PA_ERR_WORKSPACE;
    // A smaller workspace only narrows the grid.
    const size_t slots = (workspace_bytes - cnt) / cta_record_bytes(head_dim);
    const int max_grid = (int)(slots < (size_t)kMaxGrid ? slots : (size_t)kMaxGrid);

    CUtensorMap map;
    if (!make_cache_pair_map(&map, cache, layer)) return PA_ERR_CUDA;
    if (scale == 0.f) scale = 1.0f / sqrtf((float)head_dim);

    DecodeArgs a;
    a.q = static_cast<const __half *>(q);
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.out = static_cast<__half *>(out);
    a.counters = static_cast<int32_t *>(workspace);
    a.rec = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + cnt);
    a.status = dev_status;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.B = num_seqs;
    a.H = n_heads;
    a.Hk = n_kv_heads;
    a.g = n_heads / n_kv_heads;
    a.maxb = max_blocks_per_seq;
    a.num_blocks = cache->num_blocks;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return head_dim == 128 ? launch_decode<128>(map, a, max_grid, st)
                           : launch_decode<64>(map, a, max_grid, st);
}

// ---------------------------------------------------------------- int8 cache

namespace pa {
namespace {

// 4-D uint8 map of layer `layer`'s codes: {head_dim bytes, Hk, num_blocks *
// 16 rows, 2 planes (K, V)}, box {head_dim, 1, 16, 2}: one copy brings a
// block's K and V code tiles.  128-byte swizzle at head_dim 128 (the
// consumers' 16-byte reads of a block tile then fall in distinct banks),
// none at 64; L2 fetches of one row's size.
bool make_codes_map(CUtensorMap *map, const pa_cache_i8_t *c, int layer) {
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return false;
    const cuuint64_t D = c->head_dim, Hk = c->n_kv_heads;
    const cuuint64_t rows = (cuuint64_t)c->num_blocks * c->block_size;
    const cuuint64_t plane = rows * Hk * D;  // bytes of one layer's K (or V) codes
    cuuint64_t dims[4] = {D, Hk, rows, 2};
    cuuint64_t strides[3] = {D, Hk * D, (cuuint64_t)c->layers * plane};
    cuuint32_t box[4] = {(cuuint32_t)D, 1, (cuuint32_t)kBlockSize, 2};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, c->codes + (size_t)layer * plane, dims,
               strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               D == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
               D == 128 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B : CU_TENSOR_MAP_L2_PROMOTION_L2_64B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D float32 map of layer `layer`'s scales: {16, num_blocks * Hk, 2 planes
// (K, V)}, box {16, 1, 2}: one copy brings a (block, KV head)'s 16 K and 16
// V scales.
bool make_scales_map(CUtensorMap *map, const pa_cache_i8_t *c, int layer) {
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return false;
    const cuuint64_t n = (cuuint64_t)c->num_blocks * c->n_kv_heads;
    const cuuint64_t plane = n * kBlockSize;  // floats of one layer's K (or V) scales
    cuuint64_t dims[3] = {(cuuint64_t)kBlockSize, n, 2};
    cuuint64_t strides[2] = {kBlockSize * 4, (cuuint64_t)c->layers * plane * 4};
    cuuint32_t box[3] = {(cuuint32_t)kBlockSize, 1, 2};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, c->scales + (size_t)layer * plane, dims,
               strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace
}  // namespace pa

extern "C" int pa_decode_i8(const void *q, const pa_cache_i8_t *cache, int layer,
                            const int32_t *block_tables, int max_blocks_per_seq,
                            const int32_t *context_lens, int num_seqs, int n_heads,
                            int n_kv_heads, int head_dim, float scale, void *workspace,
                            size_t workspace_bytes, void *out, int32_t *dev_status,
                            pa_stream_t stream) {
    if (num_seqs < 0 || n_heads <= 0 || n_kv_heads <= 0 || n_heads % n_kv_heads != 0 ||
        max_blocks_per_seq <= 0 || max_blocks_per_seq > kMaxBlocksPerSeq || !(scale >= 0.f))
        return PA_ERR_INVALID;
    if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (n_heads / n_kv_heads > kGroupPad || num_seqs > kMaxSeqs) return PA_ERR_UNSUPPORTED;
    if (!cache || !cache->codes || !cache->scales || layer < 0 || layer >= cache->layers ||
        cache->n_kv_heads != n_kv_heads || cache->head_dim != head_dim ||
        cache->block_size != kBlockSize || cache->num_blocks <= 0)
        return PA_ERR_INVALID;
    if (num_seqs == 0) return PA_OK;
    if (!q || !block_tables || !context_lens || !out || !workspace) return PA_ERR_INVALID;
    if (!aligned16(q) || !aligned16(out) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return PA_ERR_INVALID;
    const size_t cnt = counters_bytes(num_seqs, n_kv_heads);
    if (workspace_bytes < cnt + cta_record_bytes(head_dim)) return PA_ERR_WORKSPACE;
    const size_t slots = (workspace_bytes - cnt) / cta_record_bytes(head_dim);
    const int max_grid = (int)(slots < (size_t)kMaxGrid ? slots : (size_t)kMaxGrid);

    CUtensorMap map, smap;
    if (!make_codes_map(&map, cache, layer) || !make_scales_map(&smap, cache, layer))
        return PA_ERR_CUDA;
    if (scale == 0.f) scale = 1.0f / sqrtf((float)head_dim);

    DecodeArgs a;
    a.q = static_cast<const __half *>(q);
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.out = static_cast<__half *>(out);
    a.counters = static_cast<int32_t *>(workspace);
    a.rec = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + cnt);
    a.status = dev_status;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.B = num_seqs;
    a.H = n_heads;
    a.Hk = n_kv_heads;
    a.g = n_heads / n_kv_heads;
    a.maxb = max_blocks_per_seq;
    a.num_blocks = cache->num_blocks;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return head_dim == 128
               ? launch_decode_stages<128, kStagesI8, true>(map, smap, a, max_grid, st)
               : launch_decode_stages<64, kStagesI8, true>(map, smap, a, max_grid, st);
}

// ---------------------------------------------------------------- no-alloc variant
//
// For callers that cannot give the library device memory: the workspace of
// pa_decode is taken from one fixed array of this translation unit.  Host
// code never uses the array's name as an address (on the host it only
// names a stand-in); the device address comes from cudaGetSymbolAddress,
// looked up once per device with that device current.

static __device__ __align__(256) uint8_t g_noalloc_scratch[PA_DECODE_NOALLOC_SCRATCH_BYTES];

namespace pa {
namespace {

// cuCtxGetCurrent, obtained from the driver at run time like
// cuTensorMapEncodeTiled (the library does not link libcuda).
using CtxGetCurrentFn = CUresult (*)(CUcontext *);
CtxGetCurrentFn ctx_get_current() {
    static CtxGetCurrentFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult r;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                             &r) == cudaSuccess &&
            r == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(p);
    });
    return fn;
}

// Per device: the context the array's address was looked up in, and the
// address.  A device reset (or any re-creation of the primary context)
// loads the module again, possibly at another address; the context handle
// then differs and the address is looked up again.
struct NoallocSlot {
    CUcontext ctx = nullptr;
    void *ptr = nullptr;
};
std::mutex g_noalloc_mu;
NoallocSlot g_noalloc[64];

int noalloc_scratch(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return PA_ERR_CUDA;
    }
    // The current context may not exist yet on the first call: the symbol
    // lookup below creates it, and the context is read again after it.
    CtxGetCurrentFn get_ctx = ctx_get_current();
    CUcontext ctx = nullptr;
    if (get_ctx && get_ctx(&ctx) != CUDA_SUCCESS) ctx = nullptr;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    NoallocSlot &slot = g_noalloc[dev];
    if (!slot.ptr || !ctx || slot.ctx != ctx) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return PA_ERR_CUDA;
        }
        if (!ctx && get_ctx && get_ctx(&ctx) != CUDA_SUCCESS) ctx = nullptr;
        slot.ptr = p;
        slot.ctx = ctx;
    }
    *out = slot.ptr;
    return PA_OK;
}

}  // namespace
}  // namespace pa

extern "C" int pa_decode_noalloc(const void *q, const pa_cache_t *cache, int layer,
                                 const int32_t *block_tables, int max_blocks_per_seq,
                                 const int32_t *context_lens, int num_seqs, int n_heads,
                                 int n_kv_heads, int head_dim, float scale, void *out,
                                 int32_t *dev_status, pa_stream_t stream) {
    // The same checks, in the same order, as pa_decode, before anything is
    // enqueued: the two entry points return the same codes for the same
    // arguments.
    const int rc = check_decode_args(q, cache, layer, block_tables, max_blocks_per_seq,
                                     context_lens, num_seqs, n_heads, n_kv_heads, head_dim, scale,
                                     out);
    if (rc != PA_OK || num_seqs == 0) return rc;
    const size_t need = pa_decode_workspace_bytes(num_seqs, n_heads, n_kv_heads, head_dim);
    if (need == 0) return PA_ERR_INVALID;
    if (need > PA_DECODE_NOALLOC_SCRATCH_BYTES) return PA_ERR_WORKSPACE;
    void *scratch = nullptr;
    const int src = noalloc_scratch(&scratch);
    if (src != PA_OK) return src;
    // Counters must start at zero; an earlier call that stopped early may
    // have left some behind.
    if (cudaMemsetAsync(scratch, 0, counters_bytes(num_seqs, n_kv_heads),
                        static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return PA_ERR_CUDA;
    }
    return pa_decode(q, cache, layer, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                     n_heads, n_kv_heads, head_dim, scale, scratch, need, out, dev_status, stream);
}
