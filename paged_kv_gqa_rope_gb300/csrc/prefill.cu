// Step a3: varlen causal prefill over the paged cache on the tcgen05 tensor
// cores ("Meta Llama source deep-dive", 3.5: scores = q k^T / sqrt(d),
// softmax in fp32, times V; 3.8: a cached prefix of start_pos keys is fully
// visible and the new tokens see each other causally; "personal chatgpt 22 -
// llama2 generate", section 2: M_ij = 0 for j <= i; "nano-vllm notes -
// Llama", prepare_prefill: cu_seqlens_q / cu_seqlens_k delimit the flattened
// stream and block_tables locate every key, prefix and new, in the cache).
//
// Work unit: 256 query rows (two 128-row tiles) of one sequence and one Q
// head; both tiles read the same K/V tiles, so each K/V byte brought to the
// SM serves 256 rows (a paged K/V tile takes a few microseconds to arrive,
// and the rings that hide that fit in shared memory only at this rate).
// Row i of a sequence with a cached prefix of p keys sits at absolute
// position p + i and sees keys 0 .. p + i; key tiles of 128 keys (8 cache
// blocks) past a tile's last row are never loaded, and only the tiles that
// reach past a tile's first row are masked.
//
// Schedule: units are ordered (sequence, head, row pair from the last to the
// first) and handed out in that order by a global work counter to the CTAs
// of a persistent grid as they become free, so the CTAs running at any moment
// work on neighbouring units, mostly of the same heads, and read each K/V
// tile from L2 rather than each from HBM; the sequences are listed from the
// costliest to the cheapest and within a head the costliest pair goes first,
// so the cheap units close the list, which evens out the CTAs' ends.  When
// the scheduler takes a unit it asks L2 for the unit's Q tiles, so their
// later load into shared memory is an L2 hit.
//
// Pipeline.  Tensor memory (512 columns): S_0 | S_1 | O_0 | O_1, the score
// tile of each query tile (128 keys) and its output accumulator.  Per key
// tile the softmax of tile t reads S_t in two 64-column halves and writes
// each half's P as fp16 over the first 32 columns of the half, handing the
// first half to the tensor core at once; O_t += P.V runs in the same two
// halves, and each half of the next key tile's scores (N = 64) goes into
// its half of S_t as soon as the P.V that reads that half's P is issued
// (tcgen05.mma operations issued by one thread execute in issue order).
// So the next tile's first-half scores are computed while the softmax works
// on this tile's second half.  Each query tile has its own MMA thread, so
// one tile's softmax runs while the tensor core works on the other's P.V
// and scores, and neither tile's MMAs wait behind the other's
// synchronisation.
//
// Roles (512 threads, 128 registers each):
//   warps 0-3, 4-7   softmax of query tile 0 / 1 (thread i owns row i =
//                    TMEM lane i): running maximum and sum, P = 2^(s * scale
//                    * log2 e - m) in fp16
//   warp 8           producer of the Q tiles and the K tiles, and scheduler:
//                    takes the CTA's next unit from the launch's work counter
//                    into a ring in shared memory; warp 10 producer of the V
//                    tiles: TMA loads of one 16-token block x 64-column half
//                    at a time, gathered through the block table into rings
//                    (K: 3 stages, V: 2 at head_dim 128)
//   warps 9, 11      MMA issuers of query tile 0 / 1 (one thread each);
//                    warp 9 owns the TMEM
//   warps 12-15      output: O_t / l of a finished tile to global memory,
//                    while the softmax warpgroups work on the next unit
// The running maximum only moves when a half tile raises it by more than 8
// (log2 units), so P <= 256 and O is rescaled (in TMEM) only then.  The row
// sum adds P in fp32 before its rounding to fp16 (the two differ by far
// less than the output's own fp16 rounding).
//
// Bound: tensor cores.  Algorithmic FLOPs = 4 * d * H * (number of visible
// (query, key) pairs).
#include <atomic>
#include <climits>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tcgen05.cuh"

namespace pa {
namespace {

constexpr int kBM = 128;   // query rows per tile
constexpr int kBN = 128;   // keys per K/V tile
constexpr int kBlocksPerTile = kBN / kBlockSize;
constexpr int kUnitRows = 2 * kBM;
constexpr int kProducerWarp = 8;   // also the scheduler
constexpr int kMmaWarp = 9;        // query tile 0; warp 11 issues tile 1's
constexpr int kVProducerWarp = 10;
constexpr int kMma1Warp = 11;
constexpr int kEpilogueWarp = 12;  // warps 12-15
constexpr int kThreads = 16 * 32;  // 128 registers per thread
constexpr int kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;
constexpr int kMaxSeqs = 2048;
constexpr int kRing = 6;             // scheduled units buffered per CTA
constexpr int kRingConsumers = 15;   // warps that read every ring entry
constexpr int kSchedSlots = 64;      // launches that may run at the same time

// Work counters of the dynamic unit schedule, one pair per launch slot: the
// next unit to hand out, and the CTAs that took their last unit (the last of
// them resets both for the slot's next launch).
__device__ int g_sched_next[kSchedSlots];
__device__ int g_sched_done[kSchedSlots];

struct PrefillArgs {
    const int32_t *cu_q;
    const int32_t *cu_k;
    const int32_t *block_tables;
    __half *out;
    int32_t *status;
    float scale_log2;
    int B, H, g, maxb, num_blocks, plane_k, plane_v, max_seqlen_q, total_q;
    int sched;  // launch slot of the work counters
};

// Shared memory: a small area of barriers, the unit ring, row sums and the
// sequence table at the start of the window (16-byte aligned), then, from
// the next 1024-byte boundary (128-byte swizzle), the operand tiles.
constexpr int kRingOff = 432;                    // barriers + TMEM slot before it
constexpr int kSeenOff = kRingOff + kRing * 32;  // int [8]: K / V tiles seen per stage
constexpr int kLsumOff = kSeenOff + 32;          // float [2 tiles][128]: row sums
constexpr int kTabOff = kLsumOff + 2 * 128 * 4;  // int4 [B + 1]: sequence table
// int [B] after the table: sequence of each table row (ranked batches)
__host__ __device__ __forceinline__ int misc_bytes(int B, bool ranked) {
    return (kTabOff + (B + 1) * 16 + (ranked ? B * 4 : 0) + 15) & ~15;
}

template <int D, int KS, int VS>
struct PL {
    static constexpr int kQHalf = kBM * 128;          // one 64-column half of a Q tile
    static constexpr int kQTile = kQHalf * (D / 64);
    static constexpr int kKVHalf = kBN * 128;         // one 64-column half of a K/V tile
    static constexpr int kKVTile = kKVHalf * (D / 64);
    static constexpr int kQ = 0;                      // 2 query tiles
    static constexpr int kK = 2 * kQTile;             // KS stages
    static constexpr int kV = kK + KS * kKVTile;      // VS stages
    static constexpr int kTiles = kV + VS * kKVTile;
    // The window: the small area, at most 1008 bytes to the 1024-byte
    // boundary (the window starts 16-byte aligned), the tiles.
    static size_t bytes(int B, bool ranked) {
        return (size_t)misc_bytes(B, ranked) + 1008 + (size_t)kTiles;
    }
};

// TMEM columns: the score tile of query tile t at t * 128 (its P over the
// first 64 columns), O_t at 256 + t * D.
__device__ __forceinline__ uint32_t s_col(int t) { return (uint32_t)(t * kBN); }
__device__ __forceinline__ uint32_t o_col(int t, int D) { return (uint32_t)(2 * kBN + t * D); }

enum {
    B_QFULL = 0,    // per query tile
    B_QEMPTY = 2,   // per query tile
    B_KFULL = 4,    // up to 3 K stages
    B_KEMPTY = 7,   // up to 3
    B_VFULL = 10,   // up to 3 V stages
    B_VEMPTY = 13,  // up to 3
    B_VFIXED = 16,  // up to 3: a V tile whose tail rows were cleared
    B_SFULL = 19,   // [tile][half]: scores of the half written
    B_PHALF = 23,   // per query tile: P of the first 64 keys written
    B_PREADY = 25,  // per query tile: P of all 128 keys written
    B_OHALF = 27,   // per query tile: the P.V of the first 64 keys done
    B_ODONE = 29,   // per query tile: the P.V of the other 64 keys done
    B_OUNIT = 31,   // per query tile: the unit's last P.V done
    B_OFREE = 33,   // per query tile: O_t read out
    B_LREADY = 35,  // per query tile: row sums of a unit written
    B_LFREE = 37,   // per query tile: row sums read
    B_DRAIN = 39,   // per query tile
    B_UFULL = 41,   // kRing: unit ring entry written
    B_UEMPTY = 47,  // kRing: entry read by every consumer warp
    B_COUNT = 53
};
static_assert(B_UEMPTY == B_UFULL + kRing && B_COUNT == B_UEMPTY + kRing, "ring barriers");
static_assert(B_COUNT * 8 + 4 <= kRingOff, "barrier area");

// Highest K or V tile of a stage that an MMA thread has seen land: written
// with release order after the thread's wait on the tile's barrier, read
// with acquire order, and only ever raised, so (unlike a barrier's phase
// parity) a value cannot be mistaken for an older one.
__device__ __forceinline__ void seen_raise(int *p, int tile) {
    asm volatile("red.release.cta.shared::cta.max.s32 [%0], %1;" ::"r"(smem_u32(p)), "r"(tile)
                 : "memory");
}
__device__ __forceinline__ int seen_read(const int *p) {
    int v;
    asm volatile("ld.acquire.cta.shared::cta.s32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
    return v;
}
// Until tile `tile` of the stage has been seen to land (false after
// kWaitLimitNs).
__device__ __forceinline__ bool seen_wait(const int *p, int tile) {
    if (seen_read(p) >= tile) return true;
    const uint64_t t0 = globaltimer_ns();
    while (seen_read(p) < tile) {
        __nanosleep(64);
        if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
    }
    return true;
}

__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int c0, int c1, int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
        "r"(smem_u32(bar))
        : "memory");
}

// Prefetch one 4-D box into L2 (no shared memory, no completion tracking).
__device__ __forceinline__ void tma_prefetch_4d(const CUtensorMap *map, int c0, int c1, int c2,
                                                int c3) {
    asm volatile(
        "cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }
__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }

// Scores of columns c0 .. c0 + 63 (sa: c0 .., sb: c0 + 32 ..) past the last
// visible column kl become -inf (diagonal tiles only).
__device__ __forceinline__ void mask_cols(uint32_t (&sa)[32], uint32_t (&sb)[32], int c0, int kl) {
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        if (c0 + i > kl) sa[i] = f2u(-INFINITY);
        if (c0 + 32 + i > kl) sb[i] = f2u(-INFINITY);
    }
}

// Maximum of 64 scores (sa: columns c0 .., sb: c0 + 32 ..).
__device__ __forceinline__ float half_max(const uint32_t (&sa)[32], const uint32_t (&sb)[32]) {
    float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
        m0 = fmax3(m0, u2f(sa[i]), u2f(sa[i + 1]));
        m1 = fmax3(m1, u2f(sa[i + 2]), u2f(sa[i + 3]));
        m2 = fmax3(m2, u2f(sb[i]), u2f(sb[i + 1]));
        m3 = fmax3(m3, u2f(sb[i + 2]), u2f(sb[i + 3]));
    }
    return fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
}

// P = 2^(s * scale_log2 - m) of 64 scores as fp16 pairs (pa: columns c0 ..,
// pb: c0 + 32 ..); la / lb add the fp32 values (packed pairs) before their
// rounding.  Pairs of columns go through one packed fp32 FMA and add.
__device__ __forceinline__ void exp_half(const uint32_t (&sa)[32], const uint32_t (&sb)[32],
                                         uint64_t sl2x2, float m, uint32_t (&pa)[16],
                                         uint32_t (&pb)[16], uint64_t &la, uint64_t &lb) {
    const uint64_t negm = f2_pack(-m, -m);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        float a0, a1, b0, b1;
        f2_unpack(f2_fma(f2_pack(u2f(sa[2 * i]), u2f(sa[2 * i + 1])), sl2x2, negm), a0, a1);
        f2_unpack(f2_fma(f2_pack(u2f(sb[2 * i]), u2f(sb[2 * i + 1])), sl2x2, negm), b0, b1);
        a0 = ex2(a0);
        a1 = ex2(a1);
        b0 = ex2(b0);
        b1 = ex2(b1);
        la = f2_add(la, f2_pack(a0, a1));
        lb = f2_add(lb, f2_pack(b0, b1));
        pa[i] = pack_half2(a0, a1);
        pb[i] = pack_half2(b0, b1);
    }
}

// Shape of row pair k of a sequence with L_q query rows and a prefix of p.
// When L_q is not a multiple of 256 the odd rows form the first pair (rows
// 0 .. L_q mod 256 - 1): a pair with an empty or short second tile then
// sees the fewest keys, instead of the most as the sequence's last rows.
struct PairShape {
    int q0;     // first row of the pair
    int rv[2];  // valid rows of query tile 0 / 1
    int n[2];   // key tiles of query tile 0 / 1 (0 for an empty tile)
    // Selects instead of a run-time index keep the shape in registers.
    __device__ __forceinline__ int tiles(int t) const { return t ? n[1] : n[0]; }
    __device__ __forceinline__ int rows(int t) const { return t ? rv[1] : rv[0]; }
};

__device__ __forceinline__ PairShape pair_shape(int p, int L_q, int k) {
    PairShape ps;
    const int rem = L_q % kUnitRows;
    const int off = rem == 0 ? 0 : rem - kUnitRows;  // where pair 0 would start
    ps.q0 = max(0, off + k * kUnitRows);
    const int rows = off + (k + 1) * kUnitRows - ps.q0;
    ps.rv[0] = min(kBM, rows);
    ps.rv[1] = max(0, rows - kBM);
    ps.n[0] = (p + ps.q0 + ps.rv[0] + kBN - 1) / kBN;
    ps.n[1] = ps.rv[1] > 0 ? (p + ps.q0 + kBM + ps.rv[1] + kBN - 1) / kBN : 0;
    return ps;
}

struct SeqInfo {
    int q_begin, L_q, k_len;
};

__device__ __forceinline__ SeqInfo seq_info(const PrefillArgs &a, int s) {
    SeqInfo si;
    si.q_begin = __ldg(a.cu_q + s);
    si.L_q = __ldg(a.cu_q + s + 1) - si.q_begin;
    si.k_len = __ldg(a.cu_k + s + 1) - __ldg(a.cu_k + s);
    return si;
}

__device__ __forceinline__ bool seq_ok(const PrefillArgs &a, const SeqInfo &si) {
    return si.L_q >= 0 && si.k_len >= si.L_q && si.k_len <= a.maxb * kBlockSize &&
           si.q_begin >= 0 && si.q_begin + si.L_q <= a.total_q;
}

// Work unit idx of the list ordered (sequence, head, row pair from the last
// to the first).  CTAs take units from the list in order as they finish
// others, so the CTAs running at any moment work on neighbouring units,
// mostly of the same heads, and share those heads' K/V tiles in L2; within a
// head the costliest pair comes first, and the sequences are listed from
// the costliest to the cheapest (batches of up to kThreads sequences), so
// the list ends on cheap units.  `tab` is the shared-memory sequence table:
// tab[i] = {units of rows before i, q_begin, L_q, k_len} of sequence
// seqid[i] (i itself when seqid is null), tab[B].x = all units.
struct UnitIter {
    int u;  // unit index
    int s, h, k;
    SeqInfo si;
    int p;
    PairShape ps;

    // Unit idx from the sequence table (the scheduler decodes each unit once).
    __device__ __forceinline__ void decode(int B, const int4 *tab, const int *seqid, int idx) {
        u = idx;
        if (u >= tab[B].x) return;
        int lo = 0, hi = B - 1;  // largest s with tab[s].x <= u
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (tab[mid].x <= u)
                lo = mid;
            else
                hi = mid - 1;
        }
        const int4 e = tab[lo];
        s = seqid ? seqid[lo] : lo;
        si.q_begin = e.y;
        si.L_q = e.z;
        si.k_len = e.w;
        const int npairs = (si.L_q + kUnitRows - 1) / kUnitRows;
        const int rem = u - e.x;
        h = rem / npairs;
        k = npairs - 1 - (rem - h * npairs);
    }
    // A decoded unit in a ring entry: {u, s, h, k}, {q_begin, L_q, k_len, 0}.
    __device__ __forceinline__ void store(int4 *e) const {
        e[0] = make_int4(u, s, h, k);
        e[1] = make_int4(si.q_begin, si.L_q, si.k_len, 0);
    }
    __device__ __forceinline__ void load(const int4 *e) {
        const int4 x = e[0], y = e[1];
        u = x.x;
        s = x.y;
        h = x.z;
        k = x.w;
        si.q_begin = y.x;
        si.L_q = y.y;
        si.k_len = y.z;
        p = si.k_len - si.L_q;
        ps = pair_shape(p, si.L_q, k);
    }
    __device__ __forceinline__ bool valid(int total) const { return u < total; }
    __device__ __forceinline__ int nmax() const { return max(ps.n[0], ps.n[1]); }
    // The last K/V tile holds the sequence's last block, which ends inside
    // the block: its V rows past k_len are cleared before P.V reads them.
    __device__ __forceinline__ bool fix_tail() const {
        const int nblk_k = (si.k_len + kBlockSize - 1) / kBlockSize;
        return (si.k_len % kBlockSize) != 0 && (nblk_k - 1) / kBlocksPerTile == nmax() - 1;
    }
};

// A CTA that has taken its last unit; the last such CTA of the launch clears
// the slot's counters for the next launch that uses it.
__device__ __forceinline__ void sched_finish(int slot) {
    __threadfence();
    if (atomicAdd(&g_sched_done[slot], 1) == (int)gridDim.x - 1) {
        atomicExch(&g_sched_next[slot], 0);
        atomicExch(&g_sched_done[slot], 0);
    }
}

template <int D, int KS, int VS>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap qmap,
                   const __grid_constant__ CUtensorMap kvmap, const PrefillArgs a) {
    using L = PL<D, KS, VS>;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int B = a.B;
    const bool ranked = B <= kThreads;
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem_raw);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar + B_COUNT);
    int4 *tab = reinterpret_cast<int4 *>(smem_raw + kTabOff);
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + misc_bytes(B, ranked) + 1023) &
        ~static_cast<uintptr_t>(1023));

    // ---- sequence table: lengths and the running count of units
    for (int s = tid; s < B; s += kThreads) {
        const SeqInfo si = seq_info(a, s);
        int c = 0;
        if (seq_ok(a, si)) {
            c = ((si.L_q + kUnitRows - 1) / kUnitRows) * a.H;
            if (si.L_q > a.max_seqlen_q && blockIdx.x == 0) report(a.status, PA_DEV_BAD_LENGTH);
        } else if (blockIdx.x == 0) {
            report(a.status, PA_DEV_BAD_LENGTH);
        }
        tab[s].y = si.q_begin;
        tab[s].z = si.L_q;
        tab[s].w = si.k_len;
        tab[s + 1].x = c;  // units of sequence s, summed below
    }
    if (tid == 0) tab[0].x = 0;
    __syncthreads();
    // ---- sequences from the costliest (visible query-key pairs) to the
    // cheapest: rank by counting, one sequence per thread
    int *seqid = reinterpret_cast<int *>(tab + B + 1);
    if (ranked) {
        int4 mine = make_int4(0, 0, 0, 0);
        int rank = 0;
        if (tid < B) {
            mine = make_int4(tab[tid + 1].x, tab[tid].y, tab[tid].z, tab[tid].w);
            auto cost = [](int units, int L_q, int k_len) -> long long {
                return units > 0 ? (long long)L_q * (2ll * k_len - L_q) : 0ll;
            };
            const long long c = cost(mine.x, mine.z, mine.w);
            for (int o = 0; o < B; ++o) {
                const long long co = cost(tab[o + 1].x, tab[o].z, tab[o].w);
                rank += (co > c || (co == c && o < tid)) ? 1 : 0;
            }
        }
        __syncthreads();
        if (tid < B) {
            tab[rank].y = mine.y;
            tab[rank].z = mine.z;
            tab[rank].w = mine.w;
            tab[rank + 1].x = mine.x;
            seqid[rank] = tid;
        }
        __syncthreads();
    }
    if (warp == 0) {
        int carry = 0;
        for (int base = 1; base <= B; base += 32) {
            const int i = base + lane;
            int v = i <= B ? tab[i].x : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int t = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += t;
            }
            if (i <= B) tab[i].x = v + carry;
            carry += __shfl_sync(0xffffffffu, v, 31);
        }
    }
    __syncthreads();
    // ---- unit ring: entry 0 taken here, the rest by the K producer warp
    int4 *uring = reinterpret_cast<int4 *>(smem_raw + kRingOff);  // 2 x int4 per entry
    const int total_units = tab[B].x;
    if (tid == 0) {
        UnitIter u0;
        u0.decode(B, tab, ranked ? seqid : nullptr,
                  min(atomicAdd(&g_sched_next[a.sched], 1), total_units));
        u0.store(uring);
    }
    __syncthreads();
    if (uring[0].x >= total_units) {  // no unit left for this CTA
        if (tid == 0) sched_finish(a.sched);
        return;
    }

    if (tid == 0) {
        // a K or V stage is free once both MMA threads are done with it
        for (int i = 0; i < KS; ++i) {
            mbar_init(&bar[B_KFULL + i], 1);
            mbar_init(&bar[B_KEMPTY + i], 2);
        }
        for (int i = 0; i < VS; ++i) {
            mbar_init(&bar[B_VFULL + i], 1);
            mbar_init(&bar[B_VEMPTY + i], 2);
            mbar_init(&bar[B_VFIXED + i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar[B_QFULL + i], 1);
            mbar_init(&bar[B_QEMPTY + i], 1);
            mbar_init(&bar[B_SFULL + 2 * i], 1);
            mbar_init(&bar[B_SFULL + 2 * i + 1], 1);
            mbar_init(&bar[B_PHALF + i], 128);
            mbar_init(&bar[B_PREADY + i], 128);
            mbar_init(&bar[B_OHALF + i], 1);
            mbar_init(&bar[B_ODONE + i], 1);
            mbar_init(&bar[B_OUNIT + i], 1);
            mbar_init(&bar[B_OFREE + i], 128);
            mbar_init(&bar[B_LREADY + i], 128);
            mbar_init(&bar[B_LFREE + i], 128);
        }
        mbar_init(&bar[B_DRAIN], 1);
        mbar_init(&bar[B_DRAIN + 1], 1);
        for (int i = 0; i < 8; ++i) reinterpret_cast<int *>(smem_raw + kSeenOff)[i] = -1;
        for (int i = 0; i < kRing; ++i) {
            mbar_init(&bar[B_UFULL + i], 1);
            mbar_init(&bar[B_UEMPTY + i], kRingConsumers);
        }
        fence_barrier_init();
        mbar_arrive(&bar[B_UFULL]);  // entry 0 is in place
    }
    if (warp == kMmaWarp) {
        tc::alloc(tmem_slot, kTmemCols);
        tc::relinquish();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    // The set-up above read only call metadata; Q and the cache may still be
    // being written by the RoPE/append kernel before this one.
    griddep_wait();
    const uint32_t tmem = *tmem_slot;
    const int oob_row = a.num_blocks * kBlockSize;  // zero-filled by TMA

    float *lsum = reinterpret_cast<float *>(smem_raw + kLsumOff);
    // Unit of ring entry i for a whole warp: every lane waits and reads,
    // lane 0 releases the entry (one arrival per warp).
    auto take = [&](int i) -> UnitIter {
        const int slot = i % kRing;
        UnitIter u;
        u.u = INT_MAX;
        const bool ok = __all_sync(0xffffffffu, mbar_wait(&bar[B_UFULL + slot], (i / kRing) & 1));
        if (ok) u.load(uring + 2 * slot);
        __syncwarp();
        if (lane == 0) {
            if (ok)
                mbar_arrive(&bar[B_UEMPTY + slot]);
            else
                report(a.status, PA_DEV_TIMEOUT);
        }
        return u;
    };

    // The same for one thread of a consumer warp (the MMA issuer).
    auto take0 = [&](int i) -> UnitIter {
        const int slot = i % kRing;
        UnitIter u;
        u.u = INT_MAX;
        if (!mbar_wait(&bar[B_UFULL + slot], (i / kRing) & 1)) {
            report(a.status, PA_DEV_TIMEOUT);
            return u;
        }
        u.load(uring + 2 * slot);
        mbar_arrive(&bar[B_UEMPTY + slot]);
        return u;
    };

    if (warp >= kEpilogueWarp) {
        // ======================= output warpgroup: thread = query row of the
        // finished tile.  It reads O_t once the unit's last P.V of the tile
        // completed, releases O_t to the next unit and stores O_t / l; the
        // softmax warpgroups meanwhile work on the next unit.
        const int r = tid - kEpilogueWarp * 32;  // TMEM lane
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        bool ok = true;
        int un0 = 0, un1 = 0;  // earlier units with rows in query tile 0 / 1
        int ui = 0;            // ring entry
        for (UnitIter u = take(0); u.valid(total_units) && ok; u = take(++ui)) {
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                int &un = t ? un1 : un0;
                if (!ok || u.ps.tiles(t) == 0) continue;
                ok = __all_sync(0xffffffffu, mbar_wait(&bar[B_LREADY + t], un & 1) &&
                                                 mbar_wait(&bar[B_OUNIT + t], un & 1));
                if (!ok) continue;
                tc::fence_after();
                const float l = lsum[t * 128 + r];
                mbar_arrive(&bar[B_LFREE + t]);
                const float inv = l > 0.f ? 1.f / l : 0.f;
                const bool row_valid = r < u.ps.rows(t);
                uint4 *dst = reinterpret_cast<uint4 *>(
                    a.out + ((int64_t)(u.si.q_begin + u.ps.q0 + t * kBM + r) * a.H + u.h) * D);
                // 32 columns at a time; O_t is released once its last columns
                // are read.
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t orr[32];
                    tc::ld32(tmem + lane_base + o_col(t, D) + c * 32, orr);
                    if (c == D / 32 - 1) {
                        tc::fence_before();
                        mbar_arrive(&bar[B_OFREE + t]);  // the next unit may overwrite O_t
                    }
                    uint32_t h[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        h[i] = pack_half2(u2f(orr[2 * i]) * inv, u2f(orr[2 * i + 1]) * inv);
                    if (row_valid) {
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            dst[c * 4 + v] = make_uint4(h[4 * v], h[4 * v + 1], h[4 * v + 2], h[4 * v + 3]);
                    }
                }
                ++un;
            }
        }
        if (!ok && lane == 0) report(a.status, PA_DEV_TIMEOUT);
    } else if (warp >= kProducerWarp) {
      if (warp == kProducerWarp || warp == kVProducerWarp) {
        // ======================= producers: Q and K tiles (warp 8), V tiles
        // (warp 10), each as soon as its own ring has room
        const bool is_v = warp == kVProducerWarp;
        const int full0 = is_v ? B_VFULL : B_KFULL;
        const int empty0 = is_v ? B_VEMPTY : B_KEMPTY;
        const int nst = is_v ? VS : KS;  // ring depth
        const int plane = is_v ? a.plane_v : a.plane_k;
        uint8_t *const ring = smem + (is_v ? L::kV : L::kK);
        int ok = 1;
        if (lane == 0) {
            if (!is_v) tma_prefetch_desc(&qmap);
            tma_prefetch_desc(&kvmap);
        }
        // Cache row of this lane's block (lanes 0-7) of key tile j of unit u.
        auto block_row = [&](const UnitIter &u, int j) -> int {
            const int nblk_k = (u.si.k_len + kBlockSize - 1) / kBlockSize;
            const int lb = j * kBlocksPerTile + lane;
            if (lane >= kBlocksPerTile || lb >= nblk_k) return oob_row;
            const int blk = __ldg(a.block_tables + (int64_t)u.s * a.maxb + lb);
            if (blk < 0 || blk >= a.num_blocks) {
                if (!is_v) report(a.status, PA_DEV_BAD_BLOCK);
                return oob_row;
            }
            return blk * kBlockSize;
        };
        int kvc = 0, qn0 = 0, qn1 = 0;  // K/V tiles, Q tiles per query tile, loaded so far
        int ui = 0;                     // ring entry
        // The K producer is also the scheduler: as it starts a unit it takes
        // the CTA's next unit from the launch's work counter into the next
        // ring entry (one unit ahead hides the counter's latency, and no more
        // is claimed, so the CTAs' last units end close together), and asks
        // L2 for that unit's Q tiles.  The ring ends with one entry past the
        // last unit.
        auto schedule = [&](int i) -> UnitIter {
            const int slot = i % kRing;
            int okw = 1;
            if (lane == 0) {
                if (i >= kRing) okw = mbar_wait(&bar[B_UEMPTY + slot], ((i / kRing) - 1) & 1);
                UnitIter v;
                v.decode(B, tab, ranked ? seqid : nullptr,
                         okw ? min(atomicAdd(&g_sched_next[a.sched], 1), total_units)
                             : total_units);
                v.store(uring + 2 * slot);
                mbar_arrive(&bar[B_UFULL + slot]);
                if (v.u >= total_units) {
                    sched_finish(a.sched);
                } else {
                    const PairShape ps = pair_shape(v.si.k_len - v.si.L_q, v.si.L_q, v.k);
                    for (int t = 0; t < 2 && ps.rows(t) > 0; ++t)
                        for (int hf = 0; hf < D / 64; ++hf)
                            tma_prefetch_4d(&qmap, 0, hf, v.h, v.si.q_begin + ps.q0 + t * kBM);
                }
            }
            ok = __shfl_sync(0xffffffffu, okw, 0) && ok;
            __syncwarp();
            UnitIter v;
            v.load(uring + 2 * slot);
            return v;
        };
        UnitIter u, un;
        if (is_v) {
            u = take(0);
        } else {
            u.load(uring);  // entry 0, written in the set-up
        }
        int rows_cur = u.valid(total_units) ? block_row(u, 0) : 0;
        while (u.valid(total_units) && ok) {
            if (!is_v) un = schedule(ui + 1);
            const int nmax = u.nmax();
            const int kvh = u.h / a.g;
            const int q0 = u.ps.q0;
            const bool fix_tail = is_v && u.fix_tail();
            for (int j = 0; j < nmax && ok; ++j) {
                int rows_next;
                if (j + 1 < nmax) {
                    rows_next = block_row(u, j + 1);
                } else {  // the next unit: its first block rows are looked up early
                    if (is_v) un = take(ui + 1);
                    rows_next = un.valid(total_units) ? block_row(un, 0) : 0;
                }
                const int idx = kvc + j;
                const int st = idx % nst;
                const uint32_t ph = (idx / nst) & 1;
                int rr[kBlocksPerTile];
#pragma unroll
                for (int b = 0; b < kBlocksPerTile; ++b)
                    rr[b] = __shfl_sync(0xffffffffu, rows_cur, b);
                if (lane == 0) {
                    ok = mbar_wait(&bar[empty0 + st], ph ^ 1);
                    if (ok) {
                        uint8_t *dst = ring + st * L::kKVTile;
                        mbar_arrive_expect_tx(&bar[full0 + st], L::kKVTile);
#pragma unroll
                        for (int b = 0; b < kBlocksPerTile; ++b)
                            for (int hf = 0; hf < D / 64; ++hf)
                                tma_load_5d(dst + hf * L::kKVHalf + b * kBlockSize * 128, &kvmap,
                                            &bar[full0 + st], 0, hf, kvh, rr[b], plane);
                    }
                }
                if (!is_v && j == 0 && lane == 0) {
                    // Q tiles after K_0: K_0's stage frees earlier than a Q
                    // buffer, which waits for its tile's last scores of the
                    // unit before.
#pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        int &qn = t ? qn1 : qn0;
                        if (!ok || u.ps.tiles(t) == 0) continue;
                        if (qn > 0) ok = mbar_wait(&bar[B_QEMPTY + t], (qn - 1) & 1);
                        if (!ok) continue;
                        mbar_arrive_expect_tx(&bar[B_QFULL + t], L::kQTile);
                        for (int hf = 0; hf < D / 64; ++hf)
                            tma_load_4d(smem + L::kQ + t * L::kQTile + hf * L::kQHalf, &qmap,
                                        &bar[B_QFULL + t], 0, hf, u.h,
                                        u.si.q_begin + q0 + t * kBM);
                        ++qn;
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (ok && fix_tail && j == nmax - 1) {
                    // Rows of the sequence's last block past k_len are never
                    // written and may hold NaN bits; P is 0 there but 0 * NaN
                    // is not, so they are cleared before P.V reads the tile.
                    if (lane == 0) ok = mbar_wait(&bar[B_VFULL + st], ph);
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (ok) {
                        uint8_t *vt = smem + L::kV + st * L::kKVTile;
                        const int nblk_k = (u.si.k_len + kBlockSize - 1) / kBlockSize;
                        const int b_in = (nblk_k - 1) % kBlocksPerTile;
                        const int r0 = u.si.k_len % kBlockSize;
                        const int nrows = kBlockSize - r0;
                        const int pieces = nrows * (D / 64) * 8;  // 16-byte pieces
                        for (int i = lane; i < pieces; i += 32) {
                            const int line = i >> 3, piece = i & 7;
                            const int hf = line / nrows, r = r0 + line % nrows;
                            *reinterpret_cast<uint4 *>(vt + hf * L::kKVHalf +
                                                       (b_in * kBlockSize + r) * 128 + piece * 16) =
                                make_uint4(0, 0, 0, 0);
                        }
                        tc::fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&bar[B_VFIXED + st]);
                    }
                }
                rows_cur = rows_next;
            }
            kvc += nmax;
            u = un;
            ++ui;
        }
        if (lane == 0) {
            if (!ok) report(a.status, PA_DEV_TIMEOUT);
            // Leave no copy in flight: the last tiles' loads have landed.
            for (int i = max(0, kvc - nst); i < kvc; ++i)
                mbar_wait(&bar[full0 + i % nst], (i / nst) & 1);
            if (!is_v && qn0 > 0) mbar_wait(&bar[B_QFULL], (qn0 - 1) & 1);
            if (!is_v && qn1 > 0) mbar_wait(&bar[B_QFULL + 1], (qn1 - 1) & 1);
        }
      } else {
        // ======================= MMA issuers: one thread per query tile (warp 9
        // tile 0, warp 11 tile 1), so one tile's waits and commits overlap
        // the other's MMAs (an MMA's issue holds its thread for about its
        // run time).  Per key tile j of its tile: O_t += P.V over the first
        // 64 keys as soon as the softmax has written their P, then over the
        // other 64, then S_t(j + 1) = Q_t.K_(j+1)^T into the same TMEM (the
        // P.V was issued first by this thread: tcgen05.mma operations issued
        // by one thread execute in issue order).
        const int t = warp == kMma1Warp ? 1 : 0;
        if (lane == 0) {
            constexpr uint32_t kIdescQK = tc::idesc_f16(kBM, kBN / 2, false, false);
            constexpr uint32_t kIdescPV = tc::idesc_f16(kBM, D, false, true);
            // Shared-memory descriptors of the operand buffers, built once; a
            // k-step only adds its byte offset / 16 to the start-address field.
            const uint64_t dq = tc::smem_desc_sw128(smem_u32(smem + L::kQ + t * L::kQTile), 16, 1024);
            const uint64_t dk0 = tc::smem_desc_sw128(smem_u32(smem + L::kK), 16, 1024);
            const uint64_t dv0 = tc::smem_desc_sw128(smem_u32(smem + L::kV), L::kKVHalf, 1024);
            bool ok = true;
            int kvc = 0;  // K/V tiles of earlier units
            int g = 0;    // score tiles of this query tile in earlier units
            int un = 0;   // earlier units with rows in this tile
            int fix0 = 0, fix1 = 0, fix2 = 0;  // cleared V tiles per V stage
            // Scores of keys 64x .. 64x + 63 of K/V tile kvi (K stage kvi % KS)
            // into columns 64x .. 64x + 63 of S_t.
            auto issue_s = [&](int kvi, int x) {
                const uint64_t dk =
                    dk0 + (uint64_t)(((kvi % KS) * L::kKVTile + x * (kBN / 2) * 128) >> 4);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    tc::mma_ss(tmem + s_col(t) + x * (kBN / 2),
                               dq + (uint64_t)(((kk >> 2) * L::kQHalf + (kk & 3) * 32) >> 4),
                               dk + (uint64_t)(((kk >> 2) * L::kKVHalf + (kk & 3) * 32) >> 4),
                               kIdescQK, kk > 0);
                tc::commit(&bar[B_SFULL + 2 * t + x]);
            };
            // Releases of K/V tile j of a unit: a tile used by both query
            // tiles is released once by each thread, one used by this tile
            // alone twice by this thread, so no thread waits for a tile it
            // does not read.  (A thread releases a tile only after seeing it
            // loaded, and the stage's next load needs both releases: neither
            // thread can release a stage's next tile before the other has
            // released the current one.)
            auto release = [&](int full_bar, int j, int n, int n_o) {
                if (j < n) tc::commit(&bar[full_bar]);
                if (j < n && j >= n_o) tc::commit(&bar[full_bar]);
            };
            // A wait on a stage barrier by phase parity is exact only while
            // the barrier's previous phase is complete (the next cannot
            // complete before this thread releases the tile).  A thread that
            // skipped the stage's previous tile (the other query tile's last
            // key tile, or a unit with no rows of this tile) has not seen it
            // land: it would pass at once while that load is still in flight.
            // So before such a wait it checks the stage's seen counter, which
            // both threads raise after each wait.  The previous tile of a
            // stage lies in an earlier unit only for the first KS (or VS)
            // tiles of a unit; for K tile 0 the Q wait below gives the same.
            int *const kseen = reinterpret_cast<int *>(smem_raw + kSeenOff);
            int *const vseen = kseen + 4;
            int ui = 0;  // ring entry
            for (UnitIter u = take0(0); u.valid(total_units) && ok; u = take0(++ui)) {
                const int n = u.ps.tiles(t);
                const int n_o = u.ps.tiles(1 - t);
                const int nmax = u.nmax();
                const bool fix_tail = u.fix_tail();
                if (n > 0) {
                    // ---- K tile 0: the tile's first scores
                    // (Q_t first: the producer loads a unit's Q tiles only
                    // after its K tile 0, whose stage it takes only once the
                    // stage's previous tile has landed and been released, so
                    // the parity wait on K tile 0 that follows is exact)
                    ok = mbar_wait(&bar[B_QFULL + t], un & 1) &&
                         mbar_wait(&bar[B_KFULL + kvc % KS], (kvc / KS) & 1);
                    if (!ok) break;
                    seen_raise(kseen + kvc % KS, kvc);
                    tc::fence_after();
                    issue_s(kvc, 0);
                    issue_s(kvc, 1);
                    if (n == 1) tc::commit(&bar[B_QEMPTY + t]);  // Q_t done
                    release(B_KEMPTY + kvc % KS, 0, n, n_o);
                }
                for (int j = 0; j < n && ok; ++j) {
                    const int kvi = kvc + j;
                    const int vs = kvi % VS;
                    const int G = g + j;  // this score tile
                    // V tile j (its tail rows cleared first when it holds the
                    // sequence's last block)
                    const bool fixed = fix_tail && j == nmax - 1;
                    const bool next_s = j + 1 < n;
                    if (j < VS && kvi >= VS) ok = seen_wait(vseen + vs, kvi - VS);
                    ok = ok && mbar_wait2(fixed ? &bar[B_VFIXED + vs] : &bar[B_VFULL + vs],
                                          fixed ? (vs == 0 ? fix0 : vs == 1 ? fix1 : fix2) & 1
                                                : (kvi / VS) & 1,
                                          &bar[B_PHALF + t], G & 1);
                    if (ok) seen_raise(vseen + vs, kvi);
                    if (ok && next_s) {
                        const int kn = kvi + 1;
                        if (j + 1 < KS && kn >= KS) ok = seen_wait(kseen + kn % KS, kn - KS);
                        ok = ok && mbar_wait(&bar[B_KFULL + kn % KS], (kn / KS) & 1);
                        if (ok) seen_raise(kseen + kn % KS, kn);
                    }
                    // The unit's first P.V overwrites O_t: the output warpgroup
                    // must have read the previous unit's.
                    if (ok && j == 0 && un > 0) ok = mbar_wait(&bar[B_OFREE + t], (un - 1) & 1);
                    if (!ok) break;
                    tc::fence_after();
                    const uint64_t dv = dv0 + (uint64_t)((vs * L::kKVTile) >> 4);
                    // P of the first 64 keys sits in columns 0 .. 31, of the
                    // other 64 in columns 64 .. 95: each half of the next
                    // scores can go in as soon as the P.V that reads the
                    // half's P is issued
#pragma unroll
                    for (int kk = 0; kk < kBN / 32; ++kk)
                        tc::mma_ts(tmem + o_col(t, D), tmem + s_col(t) + kk * 8,
                                   dv + (uint64_t)((kk * 16 * 128) >> 4), kIdescPV,
                                   (j > 0 || kk > 0) ? 1u : 0u);
                    tc::commit(&bar[B_OHALF + t]);
                    if (next_s) issue_s(kvi + 1, 0);
                    ok = mbar_wait(&bar[B_PREADY + t], G & 1);
                    if (!ok) break;
                    tc::fence_after();
#pragma unroll
                    for (int kk = 0; kk < kBN / 32; ++kk)
                        tc::mma_ts(tmem + o_col(t, D), tmem + s_col(t) + kBN / 2 + kk * 8,
                                   dv + (uint64_t)(((kBN / 2 + kk * 16) * 128) >> 4), kIdescPV, 1u);
                    tc::commit(&bar[B_ODONE + t]);
                    if (j == n - 1) tc::commit(&bar[B_OUNIT + t]);
                    if (next_s) {
                        issue_s(kvi + 1, 1);
                        if (j + 2 == n) tc::commit(&bar[B_QEMPTY + t]);  // Q_t done
                    }
                    release(B_VEMPTY + vs, j, n, n_o);
                    if (next_s) release(B_KEMPTY + (kvi + 1) % KS, j + 1, n, n_o);
                    if (fixed) {
                        fix0 += vs == 0;
                        fix1 += vs == 1;
                        fix2 += vs == 2;
                    }
                }
                // the unit's cleared V tile, when only the other tile reads it
                if (ok && fix_tail && n < nmax) {
                    const int vs = (kvc + nmax - 1) % VS;
                    fix0 += vs == 0;
                    fix1 += vs == 1;
                    fix2 += vs == 2;
                }
                kvc += nmax;
                if (n > 0) {
                    g += n;
                    ++un;
                }
            }
            if (!ok) report(a.status, PA_DEV_TIMEOUT);
            // Nothing of ours may still be running when the CTA frees TMEM.
            tc::commit(&bar[B_DRAIN + t]);
            mbar_wait(&bar[B_DRAIN + t], 0);
        }
        __syncwarp();
      }
    } else {
        // ======================= softmax warpgroups: thread = query row
        const int t = warp >> 2;      // query tile of this warpgroup
        const int r = tid - t * 128;  // row in the tile = TMEM lane
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t s_tmem = tmem + lane_base + s_col(t);
        const uint32_t o_tmem = tmem + lane_base + o_col(t, D);
        const float sl2 = a.scale_log2;
        const uint64_t sl2x2 = f2_pack(sl2, sl2);
        bool ok = true;
        int g = 0;   // score tiles of this query tile in earlier units
        int un = 0;  // earlier units with rows in this query tile
        int ui = 0;  // ring entry
        for (UnitIter u = take(0); u.valid(total_units) && ok; u = take(++ui)) {
            const int n = u.ps.tiles(t);
            if (n == 0) continue;
            const int first_row = u.p + u.ps.q0 + t * kBM;  // position of row 0
            const int key_lim = min(first_row + r, u.si.k_len - 1);
            float m_used = -INFINITY, l = 0.f;
            for (int j = 0; j < n && ok; ++j) {
                const int G = g + j;
                const bool masked = j * kBN + kBN - 1 > first_row;
                // Each 64-column half is read from TMEM once with its 32
                // columns' maxima (tcgen05.ld.red; a masked half takes the
                // maximum after masking), then its P is written over the
                // score tile's first columns and handed to the P.V at once
                // (the first half on B_PHALF, so the tensor core starts on it
                // while the second is computed).
#pragma unroll 1
                for (int hf = 0; hf < 2; ++hf) {
                    ok = __all_sync(0xffffffffu, mbar_wait(&bar[B_SFULL + 2 * t + hf], G & 1));
                    if (!ok) break;
                    tc::fence_after();
                    uint32_t sa[32], sb[32];
                    float ma, mb;
                    tc::ld32_max_issue(s_tmem + hf * 64, sa, ma);
                    tc::ld32_max_issue(s_tmem + hf * 64 + 32, sb, mb);
                    tc::wait_ld(sa, sb, ma, mb);
                    float mx = fmaxf(ma, mb);
                    if (masked) {
                        mask_cols(sa, sb, j * kBN + hf * 64, key_lim);
                        mx = half_max(sa, sb);
                    }
                    const float m_t = mx * sl2;
                    const bool up = m_t > m_used + kRescaleThreshold;
                    float f = 1.f;
                    if (up) {
                        f = ex2(m_used - m_t);  // 0 on the first half
                        l *= f;
                        m_used = m_t;
                    }
                    if ((j > 0 || hf == 1) && __any_sync(0xffffffffu, up)) {
                        // O_t holds P.V made with the old maximum: it is scaled
                        // down to the new one by the whole warp (TMEM loads
                        // and stores are warp-wide; rows that keep their
                        // maximum scale by 1) once the P.V issued for the
                        // half before this one is done: the previous tile's
                        // second half for the first half, this tile's first
                        // half for the second.  (The P.V before that one
                        // completed before this half's scores, issued after it.)
                        ok = __all_sync(0xffffffffu,
                                        hf == 0 ? mbar_wait(&bar[B_ODONE + t], (G - 1) & 1)
                                                : mbar_wait(&bar[B_OHALF + t], G & 1));
                        if (!ok) break;
                        tc::fence_after();
#pragma unroll 1
                        for (int c = 0; c < D / 32; ++c) {
                            uint32_t orr[32];
                            tc::ld32(o_tmem + c * 32, orr);
#pragma unroll
                            for (int i = 0; i < 32; ++i) orr[i] = f2u(u2f(orr[i]) * f);
                            tc::st32(o_tmem + c * 32, orr);
                        }
                    }
                    {
                        uint64_t la = 0, lb = 0;  // packed partial row sums (+0.0f pairs)
                        uint32_t pa[16], pb[16];
                        exp_half(sa, sb, sl2x2, m_used, pa, pb, la, lb);
                        // P of this half over the first 32 of its 64 columns
                        tc::st16(s_tmem + hf * 64, pa);
                        tc::st16(s_tmem + hf * 64 + 16, pb);
                        float x0, x1, y0, y1;
                        f2_unpack(la, x0, x1);
                        f2_unpack(lb, y0, y1);
                        l += (x0 + x1) + (y0 + y1);
                    }
                    tc::wait_st();
                    tc::fence_before();
                    mbar_arrive(&bar[(hf == 0 ? B_PHALF : B_PREADY) + t]);
                }
            }
            if (!ok) break;
            // The row sum goes to the output warpgroup, which waits for the
            // unit's last P.V; this warpgroup goes on to the next unit (once
            // the previous unit's row sum has been read).
            if (un > 0) {
                ok = __all_sync(0xffffffffu, mbar_wait(&bar[B_LFREE + t], (un - 1) & 1));
                if (!ok) break;
            }
            lsum[t * 128 + r] = l;
            mbar_arrive(&bar[B_LREADY + t]);
            ++un;
            g += n;
        }
        if (!ok && lane == 0) report(a.status, PA_DEV_TIMEOUT);
    }

    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    if (warp == kMmaWarp) tc::dealloc(tmem, kTmemCols);
}

// 4-D fp16 map of q [T][H][D]: {64, D/64, H, T}, box {64, 1, 1, 128}.
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

constexpr size_t kSmemLimit = 227 * 1024;  // opt-in dynamic shared memory per CTA

template <int D, int KS, int VS>
size_t prefill_smem(int B) {
    // At least 116 KB keeps one CTA per SM, so no CTA waits in tcgen05.alloc
    // for another's 512 TMEM columns.
    const size_t need = PL<D, KS, VS>::bytes(B, B <= kThreads);
    return need > 116 * 1024 ? need : 116 * 1024;
}

template <int D, int KS, int VS>
int launch_prefill_stages(const CUtensorMap &qmap, const CUtensorMap &kvmap,
                          const PrefillArgs &a, cudaStream_t st) {
    static std::mutex mu;
    static bool attr_set[64] = {false};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PA_ERR_CUDA;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!attr_set[dev]) {
            if (cudaFuncSetAttribute(prefill_kernel<D, KS, VS>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)kSmemLimit) != cudaSuccess) {
                cudaGetLastError();
                return PA_ERR_CUDA;
            }
            attr_set[dev] = true;
        }
    }
    const int grid = sm_count();
    if (grid < 1) return PA_ERR_CUDA;
    launch_dependent(prefill_kernel<D, KS, VS>, dim3(grid), dim3(kThreads),
                     prefill_smem<D, KS, VS>(a.B), st, qmap, kvmap, a);
    return launch_status();
}

// Ring depths: two K and two V stages at head_dim 128 (a third stage of
// either fits only for small batches and measured slower on the 16-sequence
// prefill), three of each at head_dim 64, where the tiles are half the size.
template <int D>
int launch_prefill(const CUtensorMap &qmap, const CUtensorMap &kvmap, const PrefillArgs &a,
                   cudaStream_t st) {
    if constexpr (D == 64) {
        return launch_prefill_stages<64, 3, 3>(qmap, kvmap, a, st);
    } else {
        if (prefill_smem<D, 2, 2>(a.B) <= kSmemLimit)
            return launch_prefill_stages<D, 2, 2>(qmap, kvmap, a, st);
        return PA_ERR_UNSUPPORTED;
    }
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
        total_q < 0 || max_seqlen_q < 0 || max_blocks_per_seq <= 0 ||
        max_blocks_per_seq > kMaxBlocksPerSeq || !(scale >= 0.f))
        return PA_ERR_INVALID;
    if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (num_seqs > kMaxSeqs) return PA_ERR_UNSUPPORTED;
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
    a.max_seqlen_q = max_seqlen_q;
    a.total_q = total_q;
    static std::atomic<unsigned> launches{0};
    a.sched = (int)(launches.fetch_add(1) % kSchedSlots);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return head_dim == 128 ? launch_prefill<128>(qmap, kvmap, a, st)
                           : launch_prefill<64>(qmap, kvmap, a, st);
}
