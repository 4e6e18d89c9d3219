/*
 * pa.h - C ABI of the paged-KV GQA attention hot path for GB300 (sm_103a).
 *
 * The four steps of one attention layer of a Llama-2-style paged-KV engine:
 *
 *   pa_rope_kv_write   rotary embedding of the new tokens' Q and K at their
 *                      true positions, and the write of their K/V into the
 *                      block-paged cache through slot_mapping;
 *   pa_prefill_varlen  causal attention over a flattened stream of new
 *                      tokens (cu_seqlens_q / cu_seqlens_k), reading any
 *                      cached prefix through block_tables;
 *   pa_decode          attention of one new query per sequence against all
 *                      of its cached K/V, Q heads grouped onto KV heads;
 *   pa_alloc_cache     the block pool itself.
 *
 * plus host-side metadata builders (positions, cu_seqlens, slot_mapping,
 * context_lens) and the RoPE table.
 *
 * Conventions for every entry point:
 *  - Pointers documented "device" are CUDA device pointers owned by the
 *    caller (the library never frees them); "host" pointers are plain host
 *    memory.  All tensors are dense and row-major in the stated shape.
 *  - fp16 is IEEE binary16 (stored as uint16_t bits); metadata is int32.
 *  - Device work is enqueued on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream) and is asynchronous: no entry point synchronises the
 *    stream except pa_rope_table_init.
 *  - The return value is a pa_status code.  Arguments are checked on the
 *    host before anything is enqueued; an invalid call returns
 *    PA_ERR_INVALID / PA_ERR_UNSUPPORTED and touches no memory.
 *  - Device-side checks: metadata values that only exist on the device
 *    (slots, positions, block ids, lengths) are range-checked by the
 *    kernels.  A bad value is never dereferenced; the kernel skips the
 *    access and ORs a PA_DEV_* bit into *dev_status (a caller-owned device
 *    int32, may be NULL to skip reporting).  The caller reads it after the
 *    stream has finished and clears it when it wants to.
 *  - Nothing aborts, traps or waits without a bound; every wait inside a
 *    kernel gives up after about a second and reports PA_DEV_TIMEOUT.
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef void *pa_stream_t; /* cudaStream_t */

/* Return codes. */
enum pa_status {
    PA_OK = 0,
    PA_ERR_INVALID = 1,     /* bad shape, null pointer, misalignment, ... */
    PA_ERR_UNSUPPORTED = 2, /* valid but not built: head_dim, block_size, group size, device */
    PA_ERR_CUDA = 3,        /* a CUDA runtime call failed (launch, copy, malloc) */
    PA_ERR_WORKSPACE = 4    /* the decode workspace is smaller than the call needs */
};

/* Bits that kernels OR into *dev_status. */
enum pa_device_status {
    PA_DEV_BAD_SLOT = 1,      /* slot_mapping entry >= num_blocks * block_size */
    PA_DEV_BAD_POSITION = 2,  /* position < 0 or >= the RoPE table's rows */
    PA_DEV_BAD_BLOCK = 4,     /* block_tables entry outside [0, num_blocks) */
    PA_DEV_BAD_LENGTH = 8,    /* cu_seqlens / context_lens inconsistent or too long */
    PA_DEV_TIMEOUT = 16,      /* a bounded wait inside a kernel gave up */
    PA_DEV_WORKSPACE = 32     /* more decode chunks than the workspace holds */
};

/*
 * The paged KV cache: one fp16 pool laid out as
 *     [2 (K, V)][layers][num_blocks][block_size][n_kv_heads][head_dim]
 * ("nano-vllm notes - Llama", allocate_kv_cache).  Physical slot
 * `slot` of layer l is block slot / block_size, row slot % block_size.
 */
typedef struct {
    void *base;           /* device pointer to element [0][0][0][0][0][0] */
    int32_t layers;
    int32_t num_blocks;
    int32_t block_size;   /* tokens per block; 16 is the built size */
    int32_t n_kv_heads;
    int32_t head_dim;     /* 64 or 128 */
    int32_t owns;         /* 1 if pa_alloc_cache allocated base */
    int64_t layer_stride; /* elements between consecutive layers */
    int64_t kv_stride;    /* elements between the K and the V plane */
} pa_cache_t;

/* Bytes of the pool: 2 * layers * num_blocks * block_size * n_kv_heads *
 * head_dim * 2 (fp16).  0 for non-positive arguments. */
size_t pa_cache_bytes(int layers, int num_blocks, int block_size, int n_kv_heads, int head_dim);

/* Describe a pool.  With device_base == NULL the library cudaMallocs
 * pa_cache_bytes(...) bytes (contents undefined) and sets owns = 1;
 * otherwise it wraps the caller's allocation (at least that many bytes,
 * 256-byte aligned) and sets owns = 0.  Errors: PA_ERR_INVALID (shape,
 * alignment, out == NULL), PA_ERR_UNSUPPORTED (block_size != 16, head_dim
 * not 64/128), PA_ERR_CUDA (allocation failed). */
int pa_alloc_cache(pa_cache_t *out, int layers, int num_blocks, int block_size,
                   int n_kv_heads, int head_dim, void *device_base);

/* Free the pool if the library owns it; clears *cache either way. */
int pa_free_cache(pa_cache_t *cache);

/*
 * Metadata of one prefill call ("nano-vllm notes - Llama", prepare_prefill),
 * host to host.  For sequence s with num_cached[s] tokens already cached and
 * num_new[s] new ones, its new tokens sit at positions
 * num_cached[s] .. num_cached[s]+num_new[s]-1 and are written to slot
 * block_tables[s][pos / block_size] * block_size + pos % block_size.
 *   block_tables   host int32 [num_seqs][max_blocks_per_seq]
 *   positions      host int32 [sum num_new]          (output)
 *   slot_mapping   host int32 [sum num_new]          (output)
 *   cu_seqlens_q   host int32 [num_seqs + 1]         (output)
 *   cu_seqlens_k   host int32 [num_seqs + 1]         (output; seqlen_k = cached + new)
 *   max_seqlen_q/k host int32 scalars               (output, may be NULL)
 * Returns PA_ERR_INVALID for negative lengths, a block table row too short
 * for its sequence, a needed entry that is negative or whose slots pass
 * INT32_MAX, or totals (sum num_new, sum cached + new) past INT32_MAX.
 * Nothing is written on error.
 */
int pa_prepare_prefill(int num_seqs, const int32_t *num_cached, const int32_t *num_new,
                       const int32_t *block_tables, int max_blocks_per_seq, int block_size,
                       int32_t *positions, int32_t *slot_mapping, int32_t *cu_seqlens_q,
                       int32_t *cu_seqlens_k, int32_t *max_seqlen_q, int32_t *max_seqlen_k);

/*
 * Metadata of one decode step ("nano-vllm notes - Llama", prepare_decode),
 * host to host: sequence s feeds one token at position num_cached[s], whose
 * K/V goes to that position's slot; afterwards context_lens[s] =
 * num_cached[s] + 1 (the page's example: positions [5,3], context_lens [6,4]).
 *   positions, slot_mapping, context_lens   host int32 [num_seqs] (output)
 * Returns PA_ERR_INVALID for a negative num_cached, a block table row too
 * short for its position, or a needed entry that is negative or whose slots
 * pass INT32_MAX.  Nothing is written on error.
 */
int pa_prepare_decode(int num_seqs, const int32_t *num_cached, const int32_t *block_tables,
                      int max_blocks_per_seq, int block_size, int32_t *positions,
                      int32_t *slot_mapping, int32_t *context_lens);

/*
 * RoPE table ("Meta Llama source deep-dive", 3.3 precompute_freqs_cis):
 * rows m = 0 .. max_positions-1, columns i = 0 .. head_dim/2-1, each entry a
 * float pair {cos, sin} of the angle m * theta^(-2i/head_dim).  The angle,
 * cos and sin are computed in double precision on the host and each rounded
 * once to float.  device_table must hold pa_rope_table_bytes(...) bytes
 * (16-byte aligned).  Synchronises `stream` (the host staging buffer is
 * freed on return).
 */
size_t pa_rope_table_bytes(int max_positions, int head_dim);
int pa_rope_table_init(void *device_table, int max_positions, int head_dim, double theta,
                       pa_stream_t stream);

/*
 * Steps a1 + a2: rotate and append ("Meta Llama source deep-dive", 3.3
 * apply_rotary_emb and 3.5 step 2; "nano-vllm notes - Llama", slot_mapping).
 * For every new token t (num_tokens of them):
 *   - each adjacent pair (x_2i, x_2i+1) of every head of q[t] and k[t] is
 *     rotated by the table entry of row positions[t]:
 *       x' = fl32(fl32(x*c) - fl32(y*s)),  y' = fl32(fl32(x*s) + fl32(y*c)),
 *     then rounded to nearest-even fp16 and stored back in place (V is not
 *     rotated);
 *   - the rotated k[t] and the unchanged v[t] are copied bit for bit to slot
 *     slot_mapping[t] of `layer` (K plane and V plane).  slot < 0 means no
 *     write (a padding token).
 *   q     device fp16 [num_tokens][n_heads][head_dim], rotated in place
 *   k     device fp16 [num_tokens][n_kv_heads][head_dim], rotated in place
 *   v     device fp16 [num_tokens][n_kv_heads][head_dim]
 *   positions, slot_mapping   device int32 [num_tokens]
 *   rope_table   device, from pa_rope_table_init with max_positions rows
 * A position outside [0, max_positions) leaves that token untouched and sets
 * PA_DEV_BAD_POSITION; a slot past the pool sets PA_DEV_BAD_SLOT and skips
 * the write.  num_tokens == 0 is a no-op.
 */
int pa_rope_kv_write(void *q, void *k, const void *v, const int32_t *positions,
                     const int32_t *slot_mapping, int num_tokens, int n_heads, int n_kv_heads,
                     int head_dim, const void *rope_table, int max_positions,
                     const pa_cache_t *cache, int layer, int32_t *dev_status, pa_stream_t stream);

/*
 * Step a3: varlen causal prefill ("Meta Llama source deep-dive", 3.5 and 3.8;
 * "personal chatgpt 22 - llama2 generate", section 2; "nano-vllm notes -
 * Llama", prepare_prefill / flash_attn_varlen_func).  Sequence s owns query
 * rows cu_seqlens_q[s] .. cu_seqlens_q[s+1]-1 and
 * L_k = cu_seqlens_k[s+1] - cu_seqlens_k[s] keys, the first
 * p = L_k - L_q of them a cached prefix; query row i (absolute position
 * p + i) of head h attends to keys 0 .. p + i of KV head h / (n_heads /
 * n_kv_heads), all read from the cache through block_tables[s] (so the new
 * tokens' K/V must already have been written by pa_rope_kv_write):
 *     out = softmax(q k^T * scale) v,  scores and softmax in fp32, fp16 out.
 *   q            device fp16 [total_q][n_heads][head_dim] (rotated);
 *                total_q = cu_seqlens_q[num_seqs], the rows of q and out
 *   cu_seqlens_q, cu_seqlens_k   device int32 [num_seqs + 1]
 *   block_tables device int32 [num_seqs][max_blocks_per_seq]
 *                (max_blocks_per_seq * 16 must stay within INT32_MAX: the
 *                kernel bounds L_k by it in int32)
 *   max_seqlen_q host bound on any L_q (a longer sequence sets
 *                PA_DEV_BAD_LENGTH; its rows are still computed)
 *   out          device fp16 [total_q][n_heads][head_dim]
 *   scale        softmax scale; pass 0 for 1/sqrt(head_dim)
 * Built for head_dim 64 and 128, any n_heads divisible by n_kv_heads and
 * num_seqs <= 2048 (PA_ERR_UNSUPPORTED beyond); Q.K^T and P.V run on the
 * tcgen05 tensor cores with TMEM accumulators.
 */
int pa_prefill_varlen(const void *q, int total_q, const pa_cache_t *cache, int layer,
                      const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                      const int32_t *block_tables, int max_blocks_per_seq, int num_seqs,
                      int max_seqlen_q, int n_heads, int n_kv_heads, int head_dim, float scale,
                      void *out, int32_t *dev_status, pa_stream_t stream);

/*
 * Step a4: single-token GQA decode ("personal chatgpt 22 - llama2 generate",
 * section 3; "nano-vllm notes - Llama", prepare_decode /
 * flash_attn_with_kvcache).  Sequence s has context_lens[s] cached tokens
 * (its new token's K/V already appended); its query attends to all of them:
 *     out[s][h] = softmax(q[s][h] . K^T * scale) V   over KV head h / g,
 * scores and softmax in fp32, P rounded to fp16 for P.V, fp16 out.
 * The KV blocks of all (sequence, KV head) pairs are split into equal
 * contiguous ranges, one per CTA of a persistent grid; a pair cut between
 * ranges is finished by an online-softmax merge of its pieces.
 *   q             device fp16 [num_seqs][n_heads][head_dim] (rotated)
 *   block_tables  device int32 [num_seqs][max_blocks_per_seq]
 *                 (max_blocks_per_seq * 16 must stay within INT32_MAX)
 *   context_lens  device int32 [num_seqs], each in [1, max_blocks_per_seq*16]
 *                 (others set PA_DEV_BAD_LENGTH and their output is not written)
 *   workspace     device, pa_decode_workspace_bytes(...) bytes, 256-byte
 *                 aligned, ZEROED by the caller before its first use; every
 *                 call leaves it ready for the next.  A smaller workspace (at
 *                 least one CTA's records) only narrows the grid.  One call
 *                 at a time per workspace.
 *   out           device fp16 [num_seqs][n_heads][head_dim]
 *   scale         softmax scale; pass 0 for 1/sqrt(head_dim)
 * Built for head_dim 64 and 128, n_heads / n_kv_heads <= 8, num_seqs <= 4096.
 */
size_t pa_decode_workspace_bytes(int num_seqs, int n_heads, int n_kv_heads, int head_dim);
int pa_decode(const void *q, const pa_cache_t *cache, int layer, const int32_t *block_tables,
              int max_blocks_per_seq, const int32_t *context_lens, int num_seqs,
              int n_heads, int n_kv_heads, int head_dim, float scale, void *workspace,
              size_t workspace_bytes, void *out, int32_t *dev_status, pa_stream_t stream);

/*
 * pa_decode without a caller-supplied workspace.  The source pages have no
 * counterpart to this entry point: it exists for callers that cannot hand
 * the library device memory of their own, for example a plugin whose host
 * framework owns every device allocation and gives the plugin none, or a
 * caller that must not call cudaMalloc once it is running because of the
 * device-wide synchronisation and the failure modes an allocation brings.
 *
 * The scratch memory pa_decode needs (arrival counters and the per-CTA
 * partial records) lives instead in one fixed array of
 * PA_DECODE_NOALLOC_SCRATCH_BYTES bytes compiled into the library: every
 * GPU that loads libpa holds that array until the process exits.  This
 * entry point allocates nothing: no cudaMalloc, no cudaFree, no allocating
 * library call.  The first call on a device looks up the array's device
 * address for that device (with that device current) and remembers it
 * together with the device's current context; make that first call before
 * any stream capture starts.  A device reset (cudaDeviceReset) re-creates
 * the context and may move the array: the next call sees the new context
 * and looks the address up again, so it too must come before any capture.
 *
 * Arguments, results and device-side checks are those of pa_decode.  Each
 * call clears the arrival counters in the array on `stream` before the
 * kernel runs.  All calls in the process share the one array, so two calls
 * that run at the same time on the GPU (on different streams, or from
 * different threads) race and corrupt each other's results: serialise them.
 * Returns PA_ERR_WORKSPACE when the call needs more than the array holds
 * (pa_decode_workspace_bytes(...) > PA_DECODE_NOALLOC_SCRATCH_BYTES).  The
 * 8 MiB array holds the 608 per-CTA records (608 * 8448 B = 4.9 MiB at
 * head_dim 128, 2.5 MiB at 64) plus 4 bytes of counter per (sequence, KV
 * head), i.e. up to about 813 k (sequence, KV head) pairs at head_dim 128.
 * Up to 195 KV heads the bound that binds first is pa_decode's own
 * num_seqs <= 4096.
 */
#define PA_DECODE_NOALLOC_SCRATCH_BYTES (8u << 20)
int pa_decode_noalloc(const void *q, const pa_cache_t *cache, int layer,
                      const int32_t *block_tables, int max_blocks_per_seq,
                      const int32_t *context_lens, int num_seqs, int n_heads, int n_kv_heads,
                      int head_dim, float scale, void *out, int32_t *dev_status,
                      pa_stream_t stream);

/*
 * One decode step of a batch in one call: pa_rope_kv_write of the batch's
 * new tokens (one per sequence) followed by pa_decode, the two kernels
 * chained so that the decode kernel's set-up overlaps the RoPE/append
 * kernel (programmatic dependent launch; the decode kernel waits for the
 * append's writes before it reads Q or the cache).  The serving loop of
 * "nano-vllm notes - Llama" (prepare_decode, then the attention call with
 * context_lens) does these two things every step; the page captures such a
 * decode step in a CUDA graph, which pa_step_graph_create below does with
 * this call.
 *   q, k, v            device fp16 [num_seqs][n_heads | n_kv_heads][head_dim]
 *                      (q and k rotated in place)
 *   positions, slot_mapping, context_lens   device int32 [num_seqs]
 * Every other argument, the results and the device-side checks are those of
 * pa_rope_kv_write (num_tokens = num_seqs) and pa_decode; the first error
 * stops the call.  Allocates nothing and never synchronises.
 * Launch order: the RoPE/append kernel is launched as a programmatic
 * dependent of the work before it in the stream (it waits for it to finish
 * before touching memory), and lets the decode kernel start at once; the
 * decode kernel reads context_lens and block_tables in its set-up, before
 * its wait.  So the work that writes those two arrays must not let its
 * dependents launch early (griddepcontrol.launch_dependents): a copy, or a
 * kernel launched without that instruction, is what this library expects.
 */
int pa_decode_step(void *q, void *k, const void *v, const int32_t *positions,
                   const int32_t *slot_mapping, const void *rope_table, int max_positions,
                   const pa_cache_t *cache, int layer, const int32_t *block_tables,
                   int max_blocks_per_seq, const int32_t *context_lens, int num_seqs,
                   int n_heads, int n_kv_heads, int head_dim, float scale, void *workspace,
                   size_t workspace_bytes, void *out, int32_t *dev_status, pa_stream_t stream);

/*
 * One prefill step of a batch in one call: pa_rope_kv_write of the batch's
 * total_q new tokens followed by pa_prefill_varlen over them, chained as in
 * pa_decode_step (the prefill kernel's set-up overlaps the RoPE/append
 * kernel; it waits for the append's writes before it reads Q or the cache).
 * The prefill of "nano-vllm notes - Llama" (prepare_prefill: positions,
 * cu_seqlens, slot_mapping, then the varlen attention call) does these two
 * things for every batch of new prompts or prompt chunks.
 *   q, k, v            device fp16 [total_q][n_heads | n_kv_heads][head_dim]
 *                      (q and k rotated in place)
 *   positions, slot_mapping   device int32 [total_q]
 *   cu_seqlens_q, cu_seqlens_k   device int32 [num_seqs + 1]
 * Every other argument, the results and the device-side checks are those of
 * pa_rope_kv_write (num_tokens = total_q) and pa_prefill_varlen; the first
 * error stops the call.  Allocates nothing and never synchronises.
 */
int pa_prefill_step(void *q, void *k, const void *v, const int32_t *positions,
                    const int32_t *slot_mapping, const void *rope_table, int max_positions,
                    const pa_cache_t *cache, int layer, const int32_t *cu_seqlens_q,
                    const int32_t *cu_seqlens_k, const int32_t *block_tables,
                    int max_blocks_per_seq, int num_seqs, int total_q, int max_seqlen_q,
                    int n_heads, int n_kv_heads, int head_dim, float scale, void *out,
                    int32_t *dev_status, pa_stream_t stream);

/*
 * A decode step captured once into an executable CUDA graph and replayed
 * per step: pa_step_graph_create records pa_decode_step with the given
 * arguments (on a stream of its own, in relaxed capture mode) and
 * instantiates it; pa_step_graph_launch replays it on `stream`.  The replay
 * uses the same device buffers, batch size and shapes; what the buffers
 * hold (new tokens, positions, slots, context lengths, block tables) may
 * change between replays, as in a serving loop.  The caller keeps every
 * buffer alive and unchanged in size until pa_step_graph_destroy.  Errors: those of pa_decode_step found at capture (nothing is
 * created), PA_ERR_CUDA if capture or instantiation fails, PA_ERR_INVALID
 * for a NULL handle.
 */
typedef struct pa_step_graph *pa_step_graph_t;
int pa_step_graph_create(pa_step_graph_t *graph, void *q, void *k, const void *v,
                         const int32_t *positions, const int32_t *slot_mapping,
                         const void *rope_table, int max_positions, const pa_cache_t *cache,
                         int layer, const int32_t *block_tables, int max_blocks_per_seq,
                         const int32_t *context_lens, int num_seqs, int n_heads, int n_kv_heads,
                         int head_dim, float scale, void *workspace, size_t workspace_bytes,
                         void *out, int32_t *dev_status);
int pa_step_graph_launch(pa_step_graph_t graph, pa_stream_t stream);
int pa_step_graph_destroy(pa_step_graph_t graph);

/*
 * The same captured step with its host I/O inside the graph, so that one
 * replay moves a step's inputs in, runs it and brings its result back:
 *   first   in_bytes from host_in to dev_in (host to device), where dev_in
 *           is the device buffer that holds the step's inputs (q, k, v,
 *           positions, slot_mapping, block_tables, context_lens or any of
 *           them, laid out by the caller);
 *   then    pa_decode_step with the other arguments, as pa_step_graph_create;
 *   last    the output, num_seqs * n_heads * head_dim fp16, from `out` to
 *           host_out (device to host).
 * host_in and host_out must be page-locked host memory (cudaHostAlloc,
 * cudaMallocHost or registered) that stays alive until the graph is
 * destroyed; the caller fills host_in before a replay and reads host_out
 * after it has completed (e.g. after synchronising the replay's stream).
 * in_bytes = 0 leaves out the input copy, host_out = NULL the output copy.
 * Each copy is a small kernel that reads (or writes) the host buffer through
 * its device mapping (page-locked memory is mapped under unified addressing)
 * when the mapping exists and both addresses are 16-byte aligned, else a
 * cudaMemcpyAsync; the graph's kernels are chained by programmatic
 * dependent launch, each waiting for the one before it to finish.
 * Errors: those of pa_step_graph_create, and PA_ERR_INVALID for a missing
 * or pageable host buffer (nothing is created).
 */
int pa_step_graph_create_io(pa_step_graph_t *graph, void *q, void *k, const void *v,
                            const int32_t *positions, const int32_t *slot_mapping,
                            const void *rope_table, int max_positions, const pa_cache_t *cache,
                            int layer, const int32_t *block_tables, int max_blocks_per_seq,
                            const int32_t *context_lens, int num_seqs, int n_heads,
                            int n_kv_heads, int head_dim, float scale, void *workspace,
                            size_t workspace_bytes, void *out, int32_t *dev_status,
                            const void *host_in, void *dev_in, size_t in_bytes, void *host_out);

/*
 * Self-test of the kernels' failure detection; the pages have no
 * counterpart.  Every wait inside a libpa kernel (an mbarrier phase) is
 * bounded: after about a second it gives up, ORs PA_DEV_TIMEOUT into the
 * status word and lets the kernel finish, so the CUDA context stays usable.
 * This call launches one small kernel that waits, with that same bounded
 * wait, on a phase nothing completes: it takes about a second, then sets
 * PA_DEV_TIMEOUT in *dev_status (device int32).  Nothing faults or hangs.
 */
int pa_selftest_wait_timeout(int32_t *dev_status, pa_stream_t stream);

/*
 * NEXT-4: an int8 KV cache for decode.  "Meta Llama source deep-dive", 8.4,
 * lists a quantised (int8) KV cache among the production improvements; the
 * page gives no scheme, so this library fixes one: every (token, KV head)
 * row x of head_dim fp16 values (K after RoPE, V as given) is stored as
 *     scale = fl32(max_i |x_i| / 127)       (0 for an all-zero row)
 *     q_i   = clamp(rint(fl32(x_i / scale)), -127, 127)   (ties to even)
 * and stands for q_i * scale.  Layout (one allocation, codes then scales):
 *     codes  int8    [2][layers][num_blocks][block_size][n_kv_heads][head_dim]
 *     scales float32 [2][layers][num_blocks][n_kv_heads][block_size]
 * (a block's 16 scales of one KV head are contiguous: one 64-byte copy).
 * A decode step reads 2 * head_dim + 8 bytes per (token, KV head) instead of
 * 4 * head_dim.  Prefill against an int8 cache is not built.
 */
typedef struct {
    int8_t *codes;        /* device pointer to codes[0][0][0][0][0][0] */
    float *scales;        /* device pointer to scales[0][0][0][0][0] */
    int32_t layers;
    int32_t num_blocks;
    int32_t block_size;   /* 16 */
    int32_t n_kv_heads;
    int32_t head_dim;     /* 64 or 128 */
    int32_t owns;         /* 1 if pa_alloc_cache_i8 allocated it */
} pa_cache_i8_t;

/* Bytes of the pool: the codes rounded up to 256, then the scales. */
size_t pa_cache_i8_bytes(int layers, int num_blocks, int block_size, int n_kv_heads,
                         int head_dim);
/* As pa_alloc_cache, for the int8 pool (device_base 256-byte aligned, at
 * least pa_cache_i8_bytes(...) bytes, or NULL to allocate). */
int pa_alloc_cache_i8(pa_cache_i8_t *out, int layers, int num_blocks, int block_size,
                      int n_kv_heads, int head_dim, void *device_base);
int pa_free_cache_i8(pa_cache_i8_t *cache);

/* pa_rope_kv_write with the K/V rows quantised into the int8 pool (the
 * codes and scale of each row as above).  Q is rotated in place exactly as
 * by pa_rope_kv_write; arguments, results and checks are that call's. */
int pa_rope_kv_write_i8(void *q, void *k, const void *v, const int32_t *positions,
                        const int32_t *slot_mapping, int num_tokens, int n_heads,
                        int n_kv_heads, int head_dim, const void *rope_table,
                        int max_positions, const pa_cache_i8_t *cache, int layer,
                        int32_t *dev_status, pa_stream_t stream);

/* pa_decode against the int8 pool: scores use q . (codes * scale), P.V uses
 * (codes * scale); same arguments, workspace (pa_decode_workspace_bytes),
 * results and checks as pa_decode. */
int pa_decode_i8(const void *q, const pa_cache_i8_t *cache, int layer,
                 const int32_t *block_tables, int max_blocks_per_seq,
                 const int32_t *context_lens, int num_seqs, int n_heads, int n_kv_heads,
                 int head_dim, float scale, void *workspace, size_t workspace_bytes, void *out,
                 int32_t *dev_status, pa_stream_t stream);

/* Human-readable text of a pa_status code. */
const char *pa_strerror(int code);

/* PA_OK if the current CUDA device is an sm_103 part this library was built
 * for, PA_ERR_UNSUPPORTED for another device, PA_ERR_CUDA if there is none. */
int pa_check_device(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_H */
