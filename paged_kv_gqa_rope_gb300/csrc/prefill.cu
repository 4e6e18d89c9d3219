// Step a3: varlen causal prefill over the paged cache on the tcgen05 tensor
// cores ("Meta Llama source deep-dive", 3.5: scores = q k^T / sqrt(d),
// softmax in fp32, times V; 3.8: a cached prefix of start_pos keys is fully
// visible and the new tokens see each other causally; "personal chatgpt 22 -
// llama2 generate", section 2: M_ij = 0 for j <= i; "nano-vllm notes -
// Llama", prepare_prefill: cu_seqlens_q / cu_seqlens_k delimit the flattened
// stream and block_tables locate every key, prefix and new, in the cache).
//
// Work unit: 256 query rows (two 128-row tiles) of one sequence and one Q
// head.  Row i of a sequence with a cached prefix of p keys sits at
// absolute position p + i and sees keys 0 .. p + i; key tiles of 128 keys
// (8 cache blocks) past a tile's last row are never loaded, and only the
// tiles that reach past a tile's first row are masked.
//
// Schedule: units are ordered (sequence, head, row pair from the last to the
// first) and handed out in that order by a global work counter to the CTAs
// of a persistent grid as they become free, so the CTAs running at any moment
// work on neighbouring units, mostly of the same heads, and read each K/V
// tile from L2 rather than each from HBM; the sequences are listed from the
// costliest to the cheapest and within a head the costliest pair goes first,
// so the cheap units close the list, which evens out the CTAs' ends.
//
// Roles (512 threads):
//   warps 0-3   softmax of query tile 0 (thread i owns row i = TMEM lane i)
//   warps 4-7   softmax of query tile 1
//   warp 8      producer of the two Q tiles and the K tiles, warp 10 of the
//               V tiles: TMA loads of one 16-token block x 64-column half
//               at a time, gathered through the block table into rings (K:
//               2 stages, V: 3 when shared memory allows, else 2), each
//               refilled as soon as its own slot is free
//   warp 9      MMA issuer (one thread) and TMEM owner
//   warp 11     scheduler: takes the CTA's next units from the launch's
//               work counter into a ring in shared memory
//   warps 12-15 output: O_t / l of a finished tile to global memory, while
//               the softmax warpgroups already work on the next unit
// Tensor memory (512 columns): S0 | S1 | O0 | O1 (128 columns per score
// tile, head_dim per O).  Per key tile j the MMA thread issues, in order,
//   O0 += P0 . V_j   (A = P0 from TMEM, once softmax_0 wrote it over S0)
//   S0  = Q0 . K_j+1^T (same TMEM as P0: tcgen05.mma operations issued by
//                       one thread execute in issue order, so the P.V has
//                       read P0 before S0 is written; no wait in between)
//   O1 += P1 . V_j,  S1 = Q1 . K_j+1^T
// so softmax_0 works on S0(j+1) while the tensor core runs tile 1's MMAs and
// softmax_1 while it runs tile 0's.  Each P_t.V_j runs in two halves of 64
// keys: the first as soon as the softmax has written P for them, the second
// once the whole tile's P is written.  Every MMA has N = 128 (M = 128,
// K = 16): a tcgen05.mma takes about 96 cycles at any N up to 128, so wide
// tiles use the tensor core better.  The running maximum only moves when a
// half tile raises it by more than 8 (log2 units), so P <= 256 and O is
// rescaled (in TMEM) only then.  The row sum adds P in fp32 before its
// rounding to fp16 (the two differ by far less than the output's own fp16
// rounding).
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

constexpr int kBM = 128;  // query rows per tile
constexpr int kBN = 128;  // keys per tile
constexpr int kBlocksPerTile = kBN / kBlockSize;
constexpr int kUnitRows = 2 * kBM;
constexpr int kKStages = 2;  // K ring; the V ring has VS = 2 or 3 stages
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kVProducerWarp = 10;
constexpr int kEpilogueWarp = 12;  // warps 12-15
constexpr int kThreads = 16 * 32;  // 128 registers per thread, no spills
constexpr int kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;
constexpr int kMaxSeqs = 2048;
constexpr int kSchedWarp = 11;
constexpr int kRing = 8;             // scheduled units buffered per CTA
constexpr int kRingConsumers = 15;   // warps that read every ring entry
constexpr int kRingByte = 512;       // offset of the ring (kRing x 32 bytes) in the barrier area
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

template <int D, int VS>
struct PL {
    static constexpr int kQHalf = kBM * 128;          // one 64-column half of a Q tile
    static constexpr int kQTile = kQHalf * (D / 64);
    static constexpr int kKVHalf = kBN * 128;         // one 64-column half of a K/V tile
    static constexpr int kKVTile = kKVHalf * (D / 64);
    static constexpr int kQ = 0;                      // 2 query tiles
    static constexpr int kK = 2 * kQTile;             // kKStages stages
    static constexpr int kV = kK + kKStages * kKVTile;  // VS stages
    static constexpr int kBar = kV + VS * kKVTile;
    static constexpr int kLsum = kBar + 1024;         // float [2 tiles][2 units][128]: row sums
    static constexpr int kSeqId = kLsum + 2048;       // int [kThreads]: sequence of each table row
    static constexpr int kTab = kSeqId + 4 * kThreads;  // int4 [B + 1]: sequence table
    static size_t bytes(int B) { return (size_t)kTab + (size_t)(B + 1) * 16; }
    static constexpr int kOCol = 2 * kBN;             // O_t at kOCol + t * D
};

// TMEM column of the score tile of query tile t.
__device__ __forceinline__ uint32_t s_col(int t) { return (uint32_t)(t * kBN); }

enum {
    B_QFULL = 0,    // per query tile
    B_QEMPTY = 2,   // per query tile
    B_KFULL = 4,    // kKStages
    B_KEMPTY = 6,   // kKStages
    B_VFULL = 8,    // up to 3 V stages
    B_VEMPTY = 11,  // up to 3
    B_VFIXED = 14,  // up to 3: a V tile whose tail rows were cleared
    B_SFULL = 17,   // per query tile
    B_PREADY = 19,  // per query tile
    B_ODONE = 21,   // per query tile
    B_OFREE = 23,   // per query tile
    B_DRAIN = 25,
    B_LREADY = 26,  // per query tile and unit parity: row sums written
    B_UFULL = 30,   // kRing: unit ring entry written
    B_UEMPTY = 38,  // kRing: entry read by every consumer warp
    B_KSTART = 46,  // the K producer started a unit
    B_PHALF = 47,   // per query tile: P of the score tile's first 64 keys written
    B_OHALF = 49,   // per query tile: the P.V of those 64 keys done
    B_COUNT = 51
};
static_assert(B_COUNT * 8 + 4 <= kRingByte && kRingByte + kRing * 32 <= 1024, "barrier area");

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
struct PairShape {
    int rv[2];  // valid rows of query tile 0 / 1
    int n[2];   // key tiles of query tile 0 / 1 (0 for an empty tile)
    // Selects instead of a run-time index keep the shape in registers.
    __device__ __forceinline__ int tiles(int t) const { return t ? n[1] : n[0]; }
    __device__ __forceinline__ int rows(int t) const { return t ? rv[1] : rv[0]; }
};

__device__ __forceinline__ PairShape pair_shape(int p, int L_q, int k) {
    PairShape ps;
    const int q0 = k * kUnitRows;
    ps.rv[0] = min(kBM, L_q - q0);
    ps.rv[1] = max(0, min(kBM, L_q - q0 - kBM));
    ps.n[0] = (p + q0 + ps.rv[0] + kBN - 1) / kBN;
    ps.n[1] = ps.rv[1] > 0 ? (p + q0 + kBM + ps.rv[1] + kBN - 1) / kBN : 0;
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

template <int D, int VS>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap qmap,
                   const __grid_constant__ CUtensorMap kvmap, const PrefillArgs a) {
    using L = PL<D, VS>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + L::kBar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar + B_COUNT);
    int4 *tab = reinterpret_cast<int4 *>(smem + L::kTab);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int B = a.B;

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
    int *seqid = reinterpret_cast<int *>(smem + L::kSeqId);
    const bool ranked = B <= kThreads;
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
    // ---- unit ring: entry 0 taken here, the rest by the scheduler warp
    int4 *uring = reinterpret_cast<int4 *>(smem + L::kBar + kRingByte);  // 2 x int4 per entry
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
        for (int i = 0; i < kKStages; ++i) {
            mbar_init(&bar[B_KFULL + i], 1);
            mbar_init(&bar[B_KEMPTY + i], 1);
        }
        for (int i = 0; i < VS; ++i) {
            mbar_init(&bar[B_VFULL + i], 1);
            mbar_init(&bar[B_VEMPTY + i], 1);
            mbar_init(&bar[B_VFIXED + i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar[B_QFULL + i], 1);
            mbar_init(&bar[B_QEMPTY + i], 1);
            mbar_init(&bar[B_SFULL + i], 1);
            mbar_init(&bar[B_PREADY + i], 128);
            mbar_init(&bar[B_PHALF + i], 128);
            mbar_init(&bar[B_OHALF + i], 1);
            mbar_init(&bar[B_ODONE + i], 1);
            mbar_init(&bar[B_OFREE + i], 128);
            mbar_init(&bar[B_LREADY + 2 * i], 128);
            mbar_init(&bar[B_LREADY + 2 * i + 1], 128);
        }
        mbar_init(&bar[B_DRAIN], 1);
        for (int i = 0; i < kRing; ++i) {
            mbar_init(&bar[B_UFULL + i], 1);
            mbar_init(&bar[B_UEMPTY + i], kRingConsumers);
        }
        mbar_init(&bar[B_KSTART], 1);
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

    float *lsum = reinterpret_cast<float *>(smem + L::kLsum);
    // Unit of ring entry i, for one thread of a consumer warp (the MMA
    // issuer): waits for the entry and releases it (one arrival per warp).
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
    // The same for a whole warp: every lane waits and reads, lane 0 releases.
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

    if (warp >= kEpilogueWarp) {
        // ======================= output warpgroup: thread = query row of the
        // finished tile.  It reads O_t once the unit's last P.V completed,
        // releases O_t to the next unit and stores O_t / l; the softmax
        // warpgroups meanwhile work on the next unit.
        const int r = tid - kEpilogueWarp * 32;  // TMEM lane
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        bool ok = true;
        int g0 = 0, g1 = 0;    // score tiles of query tile 0 / 1 in earlier units
        int un0 = 0, un1 = 0;  // earlier units with rows in query tile 0 / 1
        int ui = 0;            // ring entry
        for (UnitIter u = take(0); u.valid(total_units) && ok; u = take(++ui)) {
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                const int n = u.ps.tiles(t);
                int &g = t ? g1 : g0;
                int &un = t ? un1 : un0;
                if (!ok || n == 0) continue;
                const int slot = 2 * t + (un & 1);
                ok = __all_sync(0xffffffffu,
                                mbar_wait(&bar[B_LREADY + slot], (un >> 1) & 1) &&
                                    mbar_wait(&bar[B_ODONE + t], (g + n - 1) & 1));
                if (!ok) continue;
                tc::fence_after();
                const float l = lsum[slot * 128 + r];
                const float inv = l > 0.f ? 1.f / l : 0.f;
                const bool row_valid = r < u.ps.rows(t);
                uint4 *dst = reinterpret_cast<uint4 *>(
                    a.out + ((int64_t)(u.si.q_begin + u.k * kUnitRows + t * kBM + r) * a.H + u.h) * D);
                // 32 columns at a time; O_t is released once its last columns
                // are read.
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t orr[32];
                    tc::ld32(tmem + lane_base + L::kOCol + t * D + c * 32, orr);
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
                g += n;
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
        const int nst = is_v ? VS : kKStages;  // ring depth
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
        UnitIter u = take(0), un;
        int rows_cur = u.valid(total_units) ? block_row(u, 0) : 0;
        while (u.valid(total_units) && ok) {
            // Starting u lets the scheduler take the unit after it: one unit
            // ahead is enough to hide the counter's latency, and no more is
            // claimed, so the CTAs' last units end close together.
            if (!is_v && lane == 0) mbar_arrive(&bar[B_KSTART]);
            const int nmax = max(u.ps.n[0], u.ps.n[1]);
            const int kvh = u.h / a.g;
            const int q0 = u.k * kUnitRows;
            const int nblk_k = (u.si.k_len + kBlockSize - 1) / kBlockSize;
            const bool fix_tail = is_v && (u.si.k_len % kBlockSize) != 0 &&
                                  (nblk_k - 1) / kBlocksPerTile == nmax - 1;
            for (int j = 0; j < nmax && ok; ++j) {
                int rows_next;
                if (j + 1 < nmax) {
                    rows_next = block_row(u, j + 1);
                } else {  // the next unit: its first block rows are looked up early
                    un = take(++ui);
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
                    // buffer, which waits for its tile's last S of the unit before.
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
        }
        if (lane == 0) {
            if (!ok) report(a.status, PA_DEV_TIMEOUT);
            // Leave no copy in flight: the last tiles' loads have landed.
            for (int i = max(0, kvc - nst); i < kvc; ++i)
                mbar_wait(&bar[full0 + i % nst], (i / nst) & 1);
            if (!is_v && qn0 > 0) mbar_wait(&bar[B_QFULL], (qn0 - 1) & 1);
            if (!is_v && qn1 > 0) mbar_wait(&bar[B_QFULL + 1], (qn1 - 1) & 1);
        }
      } else if (warp == kMmaWarp) {
        // ======================= MMA issuer (one thread)
        if (lane == 0) {
            constexpr uint32_t kIdescQK = tc::idesc_f16(kBM, kBN, false, false);
            constexpr uint32_t kIdescPV = tc::idesc_f16(kBM, D, false, true);
            bool ok = true;
            int kvc = 0;
            int fixc0 = 0, fixc1 = 0, fixc2 = 0;  // cleared V tiles per V stage
            int gt[2] = {0, 0};       // score tiles of query tile t in earlier units
            int units_t[2] = {0, 0};  // earlier units with a non-empty tile t
            // Shared-memory descriptors of every operand buffer, built once; a
            // k-step only adds its byte offset / 16 to the start-address field.
            const uint64_t dq0 = tc::smem_desc_sw128(smem_u32(smem + L::kQ), 16, 1024);
            const uint64_t dk0 = tc::smem_desc_sw128(smem_u32(smem + L::kK), 16, 1024);
            const uint64_t dv0 = tc::smem_desc_sw128(smem_u32(smem + L::kV), L::kKVHalf, 1024);
            // S_t for key tile j of unit u, K from ring stage st.  Its TMEM held
            // P_t of the previous score tile: the P.V that read it was issued
            // earlier by this thread, and tcgen05.mma operations issued by one
            // thread run in issue order.  After the unit's last S_t the Q_t
            // buffer is released to the next unit.
            auto issue_s = [&](const UnitIter &u, int t, int j, int st) {
                const uint64_t dq = dq0 + (uint64_t)((t * L::kQTile) >> 4);
                const uint64_t dk = dk0 + (uint64_t)((st * L::kKVTile) >> 4);
                const uint32_t d_tmem = tmem + s_col(t);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    tc::mma_ss(d_tmem, dq + (uint64_t)(((kk >> 2) * L::kQHalf + (kk & 3) * 32) >> 4),
                               dk + (uint64_t)(((kk >> 2) * L::kKVHalf + (kk & 3) * 32) >> 4),
                               kIdescQK, kk > 0);
                tc::commit(&bar[B_SFULL + t]);
                if (j + 1 == u.ps.tiles(t)) tc::commit(&bar[B_QEMPTY + t]);
            };
            // Both tiles' scores for key tile j of this unit (K from its stage).
            auto issue_s_tile = [&](const UnitIter &u, int j) -> bool {
                const int idx = kvc + j;
                const int st = idx % kKStages;
                if (!mbar_wait(&bar[B_KFULL + st], (idx / kKStages) & 1)) return false;
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    if (j >= u.ps.tiles(t)) continue;
                    if (!mbar_wait(&bar[B_QFULL + t], (t ? units_t[1] : units_t[0]) & 1)) return false;
                    tc::fence_after();
                    issue_s(u, t, j, st);
                }
                tc::commit(&bar[B_KEMPTY + st]);
                return true;
            };
            int ui = 0;  // ring entry
            for (UnitIter u = take0(0); u.valid(total_units) && ok; u = take0(++ui)) {
                const int nmax = max(u.ps.n[0], u.ps.n[1]);
                const int nblk_k = (u.si.k_len + kBlockSize - 1) / kBlockSize;
                const bool fix_tail = (u.si.k_len % kBlockSize) != 0 &&
                                      (nblk_k - 1) / kBlocksPerTile == nmax - 1;
                ok = issue_s_tile(u, 0);
                for (int j = 0; j < nmax && ok; ++j) {
                    const int idx = kvc + j;
                    const int st = idx % VS;               // V stage of tile j
                    const int st1 = (idx + 1) % kKStages;  // K stage of tile j+1
                    // A stage is refilled only after its tile was consumed, so
                    // per-stage barriers never run two phases ahead.
                    ok = (fix_tail && j == nmax - 1)
                             ? mbar_wait(&bar[B_VFIXED + st],
                                         (st == 0 ? fixc0++ : st == 1 ? fixc1++ : fixc2++) & 1)
                             : mbar_wait(&bar[B_VFULL + st], (idx / VS) & 1);
                    tc::fence_after();
                    const uint64_t dv = dv0 + (uint64_t)((st * L::kKVTile) >> 4);
                    bool k_next = false;  // K of tile j+1 waited for
                    // Tile 0's P.V then its next scores, then tile 1's: each
                    // softmax warpgroup works while the tensor core runs the
                    // other tile's MMAs.
                    const int t_last = j < u.ps.n[1] ? 1 : 0;  // last tile to read V_j
#pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        if (!ok || j >= u.ps.n[t]) continue;
                        const int G = gt[t] + j;
                        // P.V in two halves of 64 keys: the first as soon as
                        // the softmax has written P for them, the second when
                        // the whole tile's P is in TMEM.
                        ok = mbar_wait(&bar[B_PHALF + t], G & 1);
                        if (ok && j == 0 && units_t[t] > 0)
                            ok = mbar_wait(&bar[B_OFREE + t], (units_t[t] - 1) & 1);
                        tc::fence_after();
                        if (!ok) continue;
#pragma unroll
                        for (int kk = 0; kk < kBN / 32; ++kk)
                            tc::mma_ts(tmem + L::kOCol + t * D, tmem + s_col(t) + kk * 8,
                                       dv + (uint64_t)((kk * 16 * 128) >> 4), kIdescPV,
                                       (j > 0 || kk > 0) ? 1u : 0u);
                        tc::commit(&bar[B_OHALF + t]);
                        ok = mbar_wait(&bar[B_PREADY + t], G & 1);
                        tc::fence_after();
                        if (!ok) continue;
#pragma unroll
                        for (int kk = kBN / 32; kk < kBN / 16; ++kk)
                            tc::mma_ts(tmem + L::kOCol + t * D, tmem + s_col(t) + kk * 8,
                                       dv + (uint64_t)((kk * 16 * 128) >> 4), kIdescPV, 1u);
                        tc::commit(&bar[B_ODONE + t]);
                        if (t == t_last) tc::commit(&bar[B_VEMPTY + st]);  // V_j free
                        if (j + 1 < u.ps.n[t]) {
                            if (!k_next) {
                                ok = mbar_wait(&bar[B_KFULL + st1], ((idx + 1) / kKStages) & 1);
                                tc::fence_after();
                                k_next = true;
                            }
                            if (ok) issue_s(u, t, j + 1, st1);
                        }
                    }
                    if (!ok) break;
                    if (k_next) tc::commit(&bar[B_KEMPTY + st1]);
                }
                kvc += nmax;
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    gt[t] += u.ps.n[t];
                    if (u.ps.n[t] > 0) ++units_t[t];
                }
            }
            if (!ok) report(a.status, PA_DEV_TIMEOUT);
            // Nothing of ours may still be running when the CTA frees TMEM.
            tc::commit(&bar[B_DRAIN]);
            mbar_wait(&bar[B_DRAIN], 0);
        }
        __syncwarp();
      } else if (warp == kSchedWarp) {
        // ======================= scheduler (one thread): takes the CTA's next
        // unit from the launch's work counter into the ring once the K
        // producer started the one before, ending with one past the last unit
        if (lane == 0) {
            bool ok = true;
            for (int i = 1;; ++i) {
                const int slot = i % kRing;
                ok = mbar_wait(&bar[B_KSTART], (i - 1) & 1);
                if (ok && i >= kRing) ok = mbar_wait(&bar[B_UEMPTY + slot], ((i / kRing) - 1) & 1);
                UnitIter u;
                u.decode(B, tab, ranked ? seqid : nullptr,
                         ok ? min(atomicAdd(&g_sched_next[a.sched], 1), total_units) : total_units);
                u.store(uring + 2 * slot);
                mbar_arrive(&bar[B_UFULL + slot]);
                if (u.u >= total_units) break;
            }
            if (!ok) report(a.status, PA_DEV_TIMEOUT);
            sched_finish(a.sched);
        }
        __syncwarp();
      }
    } else {
        // ======================= softmax warpgroups: thread = query row
        const int t = warp >> 2;      // query tile of this warpgroup
        const int r = tid - t * 128;  // row in the tile = TMEM lane
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t o_tmem = tmem + lane_base + L::kOCol + t * D;
        const float sl2 = a.scale_log2;
        bool ok = true;
        int g = 0;   // score tiles of this query tile in earlier units
        int un = 0;  // earlier units with rows in this query tile
        const uint32_t s_tmem = tmem + lane_base + s_col(t);
        int ui = 0;  // ring entry
        for (UnitIter u = take(0); u.valid(total_units) && ok; u = take(++ui)) {
            const int n = u.ps.tiles(t);
            if (n == 0) continue;
            const int first_row = u.p + u.k * kUnitRows + t * kBM;  // position of row 0
            const int key_lim = min(first_row + r, u.si.k_len - 1);
            float m_used = -INFINITY, l = 0.f;
            for (int j = 0; j < n; ++j) {
                const int G = g + j;
                ok = __all_sync(0xffffffffu, mbar_wait(&bar[B_SFULL + t], G & 1));
                if (!ok) break;
                tc::fence_after();
                const bool masked = j * kBN + kBN - 1 > first_row;
                const int kl = key_lim - j * kBN;  // last visible column of this tile
                const uint64_t sl2x2 = f2_pack(sl2, sl2);
                // Each 64-column half is read from TMEM once: its maximum, then
                // P over S; then the half goes to the P.V (keys 0-63 on
                // B_PHALF, the rest on B_PREADY), so the tensor core starts on
                // the first half while the second is computed.  A half that
                // raises the running maximum past the threshold (rare after a
                // row's first tile) first scales O_t down to it: O_t then holds
                // the earlier tiles' P.V, and for the second half also this
                // tile's first-half P.V, made with the old maximum.
#pragma unroll 1
                for (int hf = 0; hf < 2; ++hf) {
                    // The TMEM load returns each 32 columns' maximum too
                    // (tcgen05.ld.red); a masked tile takes it after masking.
                    uint32_t sa[32], sb[32];
                    float ma, mb;
                    tc::ld32_max_issue(s_tmem + hf * 64, sa, ma);
                    tc::ld32_max_issue(s_tmem + hf * 64 + 32, sb, mb);
                    tc::wait_ld(sa, sb, ma, mb);
                    float mx = fmaxf(ma, mb);
                    if (masked) {
                        mask_cols(sa, sb, hf * 64, kl);
                        mx = half_max(sa, sb);
                    }
                    const float m_t = mx * sl2;
                    const bool up = m_t > m_used + kRescaleThreshold;
                    float a = 1.f;
                    if (up) {
                        a = ex2(m_used - m_t);  // 0 on the first tile
                        l *= a;
                        m_used = m_t;
                    }
                    if ((j > 0 || hf == 1) && __any_sync(0xffffffffu, up)) {
                        // O_t must hold the P.V it is scaled with (normally
                        // complete: the previous tile's was issued before S_t).
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
                            for (int i = 0; i < 32; ++i) orr[i] = f2u(u2f(orr[i]) * a);
                            tc::st32(o_tmem + c * 32, orr);
                        }
                    }
                    {
                        uint64_t la = 0, lb = 0;  // packed partial row sums (+0.0f pairs)
                        uint32_t pa[16], pb[16];
                        exp_half(sa, sb, sl2x2, m_used, pa, pb, la, lb);
                        tc::st16(s_tmem + hf * 32, pa);
                        tc::st16(s_tmem + hf * 32 + 16, pb);
                        float x0, x1, y0, y1;
                        f2_unpack(la, x0, x1);
                        f2_unpack(lb, y0, y1);
                        l += (x0 + x1) + (y0 + y1);
                    }
                    tc::wait_st();
                    tc::fence_before();
                    mbar_arrive(&bar[hf == 0 ? B_PHALF + t : B_PREADY + t]);
                }
                if (!ok) break;
            }
            if (!ok) break;
            // The row sum goes to the output warpgroup, which waits for the
            // unit's last P.V; this warpgroup goes on to the next unit.
            lsum[(2 * t + (un & 1)) * 128 + r] = l;
            mbar_arrive(&bar[B_LREADY + 2 * t + (un & 1)]);
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

template <int D, int VS>
size_t prefill_smem(int B) {
    // At least 116 KB keeps one CTA per SM, so no CTA waits in tcgen05.alloc
    // for another's 512 TMEM columns.
    const size_t need = PL<D, VS>::bytes(B) + 1024;
    return need > 116 * 1024 ? need : 116 * 1024;
}

template <int D, int VS>
int launch_prefill_vs(const CUtensorMap &qmap, const CUtensorMap &kvmap, const PrefillArgs &a,
                      cudaStream_t st) {
    static std::mutex mu;
    static bool attr_set[64] = {false};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PA_ERR_CUDA;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!attr_set[dev]) {
            if (cudaFuncSetAttribute(prefill_kernel<D, VS>,
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
    launch_dependent(prefill_kernel<D, VS>, dim3(grid), dim3(kThreads), prefill_smem<D, VS>(a.B),
                     st, qmap, kvmap, a);
    return launch_status();
}

// Three V stages when the batch's prefix table leaves room for them (they
// hide the ~3 us a paged V tile takes to arrive); two otherwise.
template <int D>
int launch_prefill(const CUtensorMap &qmap, const CUtensorMap &kvmap, const PrefillArgs &a,
                   cudaStream_t st) {
    if (prefill_smem<D, 3>(a.B) <= kSmemLimit) return launch_prefill_vs<D, 3>(qmap, kvmap, a, st);
    if (prefill_smem<D, 2>(a.B) <= kSmemLimit) return launch_prefill_vs<D, 2>(qmap, kvmap, a, st);
    return PA_ERR_UNSUPPORTED;
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
