/*
 * pkv.h -- paged KV-cache decode step with RoPE for one GPU (sm_103a), C ABI.
 *
 * The operation, in the words of the source pages (restated):
 *   For every sequence in a decode batch, rotate the new token's query and key
 *   with RoPE at the token's absolute position, store its key and value in a
 *   shared pool of BF16 pages (16 tokens per page, one block table per
 *   sequence and layer), then let every query head attend over its own
 *   sequence's cached pages with a softmax accumulated online in FP32, never
 *   gathering a contiguous prefix and never storing the scores.
 *   ("Hours of YouTube and 85 handtyped pages of notes on LLM Inference –
 *   Start here": the shared BF16 KV page pool item, the batched decode item
 *   and the direct paged decode attention item. The RoPE equations are those
 *   of "手写LLM推理引擎：Tokenizer、Transformer与Detokenizer三段式实现"
 *   section 3.2, read with rotate-half pairing.)
 *
 * Conventions shared by every entry point:
 *  - The return value is 0 on success or a negative errno value, as in the C
 *    engine of "llmc — 从零写一个大模型推理引擎（配套代码）" (introduction):
 *      -EINVAL  bad argument (null pointer, bad shape, misaligned storage,
 *               workspace too small, ...); nothing is launched.
 *      -ENOSPC  the storage given to kv_pool_create holds no page.
 *      -EIO     a CUDA runtime call failed; pkv_last_cuda_error() returns the
 *               cudaError_t value of the calling thread's last failure.
 *  - Tensor arguments are device pointers that the caller owns and keeps
 *    alive until the work queued on `stream` has finished. The library frees
 *    none of them and allocates no device memory except the pool's 4-byte
 *    error word (kv_pool_create).
 *  - `stream` is a cudaStream_t passed as void* (NULL: the legacy default
 *    stream). Every call only enqueues work on it; nothing synchronises except
 *    pkv_get_error.
 *  - Checks that need device data (lengths, page ids) are made by the
 *    kernels. A failed check skips the affected sequence or page and sets a
 *    bit (PKV_ERR_*) in the pool's error word; no kernel traps.
 *  - Fixed geometry: head_dim 64, page_size 16 tokens, bf16 cache.
 *
 * Pool layout (the contract between the append and the decode, and what the
 * test oracle indexes independently): physical page p is a contiguous block of
 * num_kv_heads * 2 * 16 * 64 bf16 values; the element for (page p, kv head h,
 * kind K=0 / V=1, slot s, dim d) is at bf16 offset
 *     (((p * num_kv_heads + h) * 2 + kind) * 16 + s) * 64 + d.
 * One kv head's keys and values for one page are one contiguous 4 KiB block.
 *
 * Sequence conventions: seq_lens[b] is the attention length AFTER the append
 * (cached tokens + the new one); the new token goes to cache index
 * seq_lens[b] - 1, i.e. slot (seq_lens[b]-1) % 16 of page
 * block_tables[b * max_blocks + (seq_lens[b]-1) / 16]; positions[b] is the
 * RoPE position it is rotated at. block_tables is the table of ONE layer,
 * row-major [batch][max_blocks]; entries past ceil(seq_lens[b]/16) are never
 * read. Query head i reads kv head i / (num_q_heads / num_kv_heads).
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PKV_HEAD_DIM 64
#define PKV_PAGE_SIZE 16
/* Largest query-head group (num_q_heads / num_kv_heads) the decode serves. */
#define PKV_MAX_GROUP 8

/* Bits of the pool's device error word. */
#define PKV_ERR_SEQ_LEN 0x1  /* seq_lens[b] < 1 or > max_blocks*16: sequence skipped, its output rows zeroed */
#define PKV_ERR_PAGE_ID 0x2  /* block-table entry outside [0, num_pages): that page skipped */
#define PKV_ERR_TIMEOUT 0x4  /* a bounded wait (a copy into shared memory, or another CTA's partial) gave up; results incomplete */
#define PKV_ERR_SPLITS  0x8  /* a row needed more than max_splits partial results: row skipped */
#define PKV_ERR_POSITION 0x10 /* a RoPE position outside the RoPE table's rows: token skipped, its rows zeroed */

typedef struct pkv_pool pkv_pool_t;

/*
 * Wrap caller-owned device storage as a page pool. ("Hours of YouTube …",
 * shared BF16 KV page pool item: one pool of physical pages, shared by all
 * sequences and layers, each page 16 tokens of K and V.)
 *   storage        device pointer, 16-byte aligned (-EINVAL otherwise)
 *   storage_bytes  size of storage; num_pages = storage_bytes / page bytes
 *                  (-ENOSPC if that is 0)
 *   num_kv_heads   1 .. 256
 *   head_dim       must be 64;  page_size  must be 16
 * On success *pool receives a handle; the storage is neither cleared nor
 * owned. Allocates the 4-byte device error word (zeroed) on the current
 * device, which must stay current for every call that uses the pool.
 */
int kv_pool_create(pkv_pool_t **pool, void *storage, size_t storage_bytes, int num_kv_heads,
                   int head_dim, int page_size);

/* Free the handle and its error word (not the storage). NULL is accepted. */
int kv_pool_destroy(pkv_pool_t *pool);

/* Number of physical pages, or -EINVAL for a NULL pool. */
int kv_pool_num_pages(const pkv_pool_t *pool);

/* Bytes of one physical page (0 for an unsupported geometry). Host only. */
size_t kv_pool_page_bytes(int num_kv_heads, int head_dim, int page_size);

/*
 * Bound of the one wait in the decode that depends on another CTA: the CTA
 * that merges a (sequence, kv head) segment split across CTAs looks at the
 * other CTAs' partial results, each look one round trip to L2, and after
 * `looks` looks without finding them all it gives up: PKV_ERR_TIMEOUT is set,
 * that segment's output rows are left unwritten and its workspace slots stay
 * written (zero the workspace again before the next call). The default,
 * 2^20 looks, is a second or more, where the partials arrive within
 * microseconds; 0 makes every such merger give up at once (a way to exercise
 * the timeout path without any wait). The setting belongs to the pool handle
 * and is read when a decode is launched (a captured CUDA graph keeps the
 * value it was captured with). *previous, if not NULL, receives the old value.
 * Host only; no device work. (Failure handling of this library, not on the
 * pages.)
 */
int kv_pool_set_merge_wait_limit(pkv_pool_t *pool, uint32_t looks, uint32_t *previous);

/*
 * RoPE + append for one layer. ("Hours of YouTube …", shared BF16 KV page pool
 * item: decode appends the new token at its absolute RoPE position;
 * "手写LLM推理引擎…" section 3.2: the rotation, inverse frequency
 * rope_theta^(-2j/64), pairs (j, j+32).)
 *   q             bf16 [batch][num_q_heads][64]
 *   k, v          bf16 [batch][num_kv_heads][64]
 *   q_rot         fp32 [batch][num_q_heads][64] out: the rotated query
 *   block_tables  int32 [batch][max_blocks], this layer
 *   seq_lens      int32 [batch], length after the append (>= 1)
 *   positions     int32 [batch], RoPE position of the new token
 *   rope_theta    RoPE base (> 0, finite)
 * The stored key is the bf16 rounding (nearest, ties to even) of the fp64
 * rotation by the correctly rounded fp64 cos and sin of the angle (as in
 * paged_rope_cos_sin): two rounded products and one rounded sum or
 * difference. v is copied bit for bit. q_rot is fp32, not rounded to bf16.
 * A sequence with a bad length or page id gets its q_rot written but nothing
 * stored in the pool (error bit set). batch == 0 is a no-op.
 * num_q_heads must be a multiple of the pool's num_kv_heads.
 */
int paged_kv_append_rope(pkv_pool_t *pool, const void *q, const void *k, const void *v,
                         float *q_rot, const int32_t *block_tables, int max_blocks,
                         const int32_t *seq_lens, const int32_t *positions, int batch,
                         int num_q_heads, double rope_theta, void *stream);

/*
 * Device bytes of workspace paged_gqa_decode needs for these sizes on the
 * current device (0 for invalid sizes). pages_per_split: as for
 * paged_gqa_decode (0 = automatic).
 */
size_t paged_gqa_decode_workspace_bytes(int batch, int num_q_heads, int num_kv_heads,
                                        int max_blocks, int pages_per_split);

/*
 * Paged GQA decode attention for one layer, split-KV with a log-sum-exp
 * merge, in one kernel launch on `stream`: the kernel merges the pieces of
 * the (sequence, kv head) segments it split, in shared memory where the
 * pieces ran in one CTA and through the workspace where they did not. ("Hours of YouTube …", direct paged decode attention
 * item: each query head streams its sequence's cached pages and accumulates
 * softmax-weighted values online in FP32, with no gathered prefix and no
 * stored scores. The split-KV form and its merge are flash-decoding, not on
 * the pages.)
 *   q_rot        fp32 [batch][num_q_heads][64], as written by paged_kv_append_rope
 *   out          fp32 [batch][num_q_heads][64]
 *   block_tables int32 [batch][max_blocks];  seq_lens int32 [batch] (>= 1)
 *   scale        softmax scale applied to q.k (typically 1/8)
 *   pages_per_split  0: balance all (sequence, kv head, page) work items
 *                evenly over the persistent grid; > 0: cut the work into
 *                ranges of this many pages (used to force splits in tests).
 *                Small values can give a CTA several rounds of ranges; a
 *                CTA that merges a split segment then waits for CTAs of an
 *                earlier round, so run such calls with the GPU to itself
 *                (otherwise the bounded wait may end in PKV_ERR_TIMEOUT).
 *   workspace    device memory of at least paged_gqa_decode_workspace_bytes(),
 *                256-byte aligned, ZERO-FILLED before its first use. It holds
 *                the partial results of segments split between CTAs, and a
 *                zero word means "not written in this call"; every call puts
 *                the words it wrote back to zero, so a workspace is zeroed
 *                once, when it is allocated. With pages_per_split = 0 it
 *                also holds the step's plan (paged_decode_plan), if any. (After a call that set
 *                PKV_ERR_TIMEOUT, zero it again: a CTA that gave up waiting
 *                for a neighbour's partial leaves its slots as they are; see
 *                kv_pool_set_merge_wait_limit.)
 *                Calls that share a workspace must not overlap on the GPU.
 * Constraints: num_q_heads = g * num_kv_heads with 1 <= g <= PKV_MAX_GROUP.
 * Rows of a sequence with a bad length are written as zeros.
 */
int paged_gqa_decode(const pkv_pool_t *pool, const float *q_rot, float *out,
                     const int32_t *block_tables, int max_blocks, const int32_t *seq_lens,
                     int batch, int num_q_heads, float scale, int pages_per_split,
                     void *workspace, size_t workspace_bytes, void *stream);

/*
 * The work plan of a decode step, written into the decode workspace. The
 * decode cuts the (sequence, kv head, page) work items of a launch into
 * ranges, one per warp, from the sequence lengths alone; the lengths are the
 * same in every layer of a step, so this call works the partition out once
 * (the page prefix sums and every range's first item) and each later
 * paged_decode_step (positions given) or paged_gqa_decode (positions NULL)
 * on the same workspace, with the same batch, lengths and shapes, reads it
 * instead of recomputing it in every CTA. A decode checks the plan against
 * its own lengths and launch shape and works the partition out itself when
 * they differ (a stale or missing plan costs time, never correctness).
 * Arguments as for paged_decode_step; pages_per_split is 0 (the automatic
 * partition). Batches above 2048 sequences are not planned (returns 0).
 * Launches one small kernel on `stream`, without programmatic dependent
 * launch, so a decode launched after it starts only once the plan is in
 * memory. (Not on the pages: a scheduling aid of this library.)
 */
int paged_decode_plan(const pkv_pool_t *pool, const int32_t *seq_lens, const int32_t *positions,
                      int rope_positions, int batch, int num_q_heads, int max_blocks,
                      void *workspace, size_t workspace_bytes, void *stream);

/* Bytes of a RoPE table of `rows` rows. */
#define PKV_ROPE_TABLE_BYTES(rows) ((size_t)(rows) * 1024u)

/*
 * RoPE cos/sin table: row r holds, for each frequency j < 32, the cos and sin
 * of the angle positions[r] * rope_theta^(-2j/64): the product rounded once
 * to fp64, then its cos and sin correctly rounded to fp64 (the fp64 values
 * nearest to the true ones, evaluated in double-double with a rounding test;
 * every angle of positions below 2^17 at bases 1e4, 5e5 and 1e6 is decided,
 * and elsewhere an undecided value, of probability about 2^-37, is within
 * half an ulp plus 2^-90 relative). Layout of the PKV_ROPE_TABLE_BYTES(rows)
 * bytes:
 *   float[rows][32][4]  {cos_hi, cos_lo, sin_hi, sin_lo}: cos_hi = cos
 *                       rounded to fp32, cos_lo = (cos - cos_hi) rounded to
 *                       fp32 (so cos_hi + cos_lo is within 2^-48 |cos|), the
 *                       same for sin; then
 *   double[rows][32][2] {cos, sin}.
 *   positions  int32 [rows];  table  out, 16-byte aligned
 * The evaluation is a chain of about 200 dependent fp64 operations per value,
 * which on this GPU takes about 13 us whatever the number of rows: the table
 * is meant to be built once (paged_rope_table_build), not per step.
 */
int paged_rope_cos_sin(const int32_t *positions, int rows, double rope_theta, void *table,
                       void *stream);

/*
 * The RoPE table of every position 0 .. num_positions - 1 (row p = position p),
 * as paged_rope_cos_sin builds it. ("手写LLM推理引擎…" section 3.2 precomputes
 * the cos/sin of every position up to the context length once, instead of
 * per use.) paged_decode_step and paged_prefill read the row of each token's
 * position from it. table: PKV_ROPE_TABLE_BYTES(num_positions) bytes,
 * 16-byte aligned. num_positions >= 1.
 */
int paged_rope_table_build(double rope_theta, int num_positions, void *table, void *stream);

/*
 * The whole decode step of one layer in one call: paged_kv_append_rope
 * followed by paged_gqa_decode, fused. ("Hours of YouTube …", batched decode
 * item: per layer, the new token of every sequence is rotated and appended,
 * then attention reads the sequence's pages; "手写LLM推理引擎…" section 4.2
 * proposes folding RoPE into the attention kernel to save launches.) The
 * decode warp that owns a sequence's last page rotates and stores the new
 * key and value (the same bytes paged_kv_append_rope stores: the rotation is
 * rounded to bf16 exactly as fp64 arithmetic on the same fp64 cos/sin rounds
 * it), and each warp rotates the query rows it uses (in fp32).
 *   q            bf16 [batch][num_q_heads][64];  k, v bf16 [batch][num_kv_heads][64]
 *   rope_table   a RoPE table of rope_positions rows, row p for position p
 *                (paged_rope_table_build), built once for the model's theta
 *   positions    int32 [batch], RoPE position of each new token; a position
 *                outside [0, rope_positions) skips the sequence (nothing
 *                appended, its rows zeroed) and sets PKV_ERR_POSITION
 *   q_rot        fp32 [batch][num_q_heads][64] out, or NULL: the rotated query
 *                (rows of sequences with a bad length or position are zeroed)
 *   out          fp32 [batch][num_q_heads][64]
 *   other arguments as for paged_gqa_decode; the workspace is sized by
 *   paged_gqa_decode_workspace_bytes().
 * A sequence whose new-token page id is bad gets no append and no attention
 * over that page (error bit set).
 * Launch order: the kernels are launched with programmatic dependent launch.
 * This call reads seq_lens, positions, block_tables and the pool's existing
 * pages before it waits for the kernel that precedes it in `stream`. That
 * kernel must therefore not write them if it lets its dependents start early
 * (griddepcontrol.launch_dependents / cudaTriggerProgrammaticLaunchCompletion).
 * A kernel that does not trigger early, a memcpy, or this library's own
 * kernels (which never write another layer's pages) are fine. q, k, v, the
 * RoPE table and all outputs are accessed only after that wait.
 */
int paged_decode_step(pkv_pool_t *pool, const void *q, const void *k, const void *v,
                      const void *rope_table, int rope_positions, const int32_t *positions,
                      float *q_rot, float *out, const int32_t *block_tables, int max_blocks,
                      const int32_t *seq_lens, int batch, int num_q_heads, float scale,
                      int pages_per_split, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Device bytes of workspace paged_prefill needs for total_tokens chunk tokens
 * over batch sequences with max_blocks-entry block tables (0 for invalid
 * sizes: a negative count, batch < 1 or max_blocks < 1).
 */
size_t paged_prefill_workspace_bytes(int total_tokens, int batch, int max_blocks);

/*
 * Chunked causal prefill into the pool. ("Hours of YouTube …": prefill fills
 * the prompt pages, the dense causal prefill item; RoPE per "手写LLM推理引擎…"
 * section 3.2.) Sequence b holds start_pos[b] cached tokens and brings the
 * chunk of tokens cu_tokens[b] .. cu_tokens[b+1]-1 (rows of q, k, v, q_rot and
 * out) at positions start_pos[b], start_pos[b]+1, ...:
 *   - every chunk token's k is rotated and stored, with its v, at its position
 *     in its sequence's pages, with the bytes paged_kv_append_rope would store
 *     for a decode token at that position;
 *   - q_rot is its rotated q;
 *   - out is the attention of each of its query heads over the sequence's
 *     first start_pos[b] + t + 1 tokens (causal: the cached ones, the chunk's
 *     earlier tokens and itself), as paged_gqa_decode computes it.
 *   q            bf16 [total_tokens][num_q_heads][64];  k, v bf16 [total_tokens][num_kv_heads][64]
 *   q_rot, out   fp32 [total_tokens][num_q_heads][64] out
 *                (q, v, q_rot, out and rope_table 16-byte aligned: -EINVAL otherwise)
 *   block_tables int32 [batch][max_blocks], the pages of every token up to
 *                start_pos[b] + chunk length assigned;  cu_tokens int32 [batch+1]
 *                (cu_tokens[0] = 0, non-decreasing, cu_tokens[batch] = total_tokens);
 *                start_pos int32 [batch] (>= 0)
 *   rope_table   a RoPE table of rope_positions rows, row p for position p
 *                (paged_rope_table_build), built once for the model's theta
 *   workspace    device memory of at least paged_prefill_workspace_bytes(),
 *                256-byte aligned, contents irrelevant
 * Launches three kernels on `stream`: a preparation (each chunk token's
 * sequence and position, and the tile plan), the append (every chunk token
 * stored as a decode token would be, with the same certified key rounding,
 * the cos and sin read from the table row of its position), and a
 * flash-attention kernel (launched to overlap the append's end, through
 * programmatic dependent launch; it lets no later kernel start early) on the tcgen05 tensor cores, one CTA per (sequence,
 * kv head, tile of up to 128 (token, query head) rows) that streams the
 * sequence's pages once per tile. Tokens of a malformed chunk (cu_tokens
 * decreasing, a negative start, or a position past max_blocks*16) are not
 * stored, their rows are zeroed and PKV_ERR_SEQ_LEN is set; tokens at a
 * position past the table's rows are treated the same way with
 * PKV_ERR_POSITION.
 */
int paged_prefill(pkv_pool_t *pool, const void *q, const void *k, const void *v, float *q_rot,
                  float *out, const int32_t *block_tables, int max_blocks,
                  const int32_t *cu_tokens, const int32_t *start_pos, int batch, int total_tokens,
                  int num_q_heads, const void *rope_table, int rope_positions, float scale,
                  void *workspace, size_t workspace_bytes, void *stream);

/* Bytes of the fixed device array paged_gqa_decode_no_alloc uses as workspace. */
#define PKV_NO_ALLOC_SCRATCH_BYTES (8u << 20)

/*
 * paged_gqa_decode for callers that cannot allocate device memory. The source
 * pages have no counterpart: this entry point exists because some callers may
 * not call cudaMalloc -- code running under a host framework whose memory
 * manager owns all device memory (a direct cudaMalloc there would synchronise
 * the device and escape the manager's accounting), or a plugin that a runtime
 * only hands its input and output buffers. It takes no workspace: the decode's
 * scratch lives in a fixed array of PKV_NO_ALLOC_SCRATCH_BYTES inside this
 * library, which every GPU that loads the library holds until the process
 * exits. It calls no allocation routine.
 *   Arguments, layouts and results are those of paged_gqa_decode.
 *   Returns -E2BIG when these sizes need more scratch than the array holds
 *   (paged_gqa_decode_workspace_bytes() > PKV_NO_ALLOC_SCRATCH_BYTES). With
 *   pages_per_split = 0 the need is two partial slots of (64 + 2) * group
 *   floats per warp of the persistent grid, 2 * SMs * CTAs per SM * warps
 *   per CTA * slot bytes, plus a plan area of about 8 bytes per sequence
 *   (22 KB at 2048); with groups of 8 on a 152-SM GPU (one CTA of 10 warps
 *   per SM) that is 6.2 MiB, so a GPU with 30% more SMs would get -E2BIG
 *   for groups of 8.
 *   The first call on each device looks up the array's device address (with
 *   that device current) and keeps it for the process; make that first call
 *   before any stream capture. The address does not survive a reset of the
 *   device's primary context (cudaDeviceReset): do not call this entry point
 *   after one.
 *   Each call first clears, on `stream`, the bytes of the array it will use
 *   (a cudaMemsetAsync, which allocates nothing), so the zero state the
 *   decode needs holds even after a call that ended with PKV_ERR_TIMEOUT.
 *   (This also clears any plan, so this entry point always works out its
 *   partition itself.)
 *   All calls share the one array: calls that overlap on the GPU (other
 *   streams, other threads) race and give wrong results; order them on one
 *   stream.
 */
int paged_gqa_decode_no_alloc(const pkv_pool_t *pool, const float *q_rot, float *out,
                              const int32_t *block_tables, int max_blocks,
                              const int32_t *seq_lens, int batch, int num_q_heads, float scale,
                              int pages_per_split, void *stream);

/*
 * The same decode, but every (sequence, query head) row leaves its split
 * results for paged_kv_split_combine instead of merging them:
 *   o_part     fp32 [batch*num_q_heads][max_splits][64]: split j's normalised output
 *   lse_part   fp32 [batch*num_q_heads][max_splits]: split j's log-sum-exp of the
 *              scaled scores (natural log)
 *   num_splits int32 [batch*num_q_heads]: number of splits of the row
 * pages_per_split must be > 0; max_splits must be at least
 * max_blocks / pages_per_split + 2 (integer division), else -EINVAL.
 */
int paged_gqa_decode_partials(const pkv_pool_t *pool, const float *q_rot,
                              const int32_t *block_tables, int max_blocks,
                              const int32_t *seq_lens, int batch, int num_q_heads, float scale,
                              int pages_per_split, float *o_part, float *lse_part,
                              int32_t *num_splits, int max_splits, void *stream);

/*
 * Log-sum-exp merge of split results (flash-decoding; not on the pages):
 * for each row r, with M = max_j lse[r][j] over j < num_splits[r] and
 * w_j = exp(lse[r][j] - M): out[r] = sum_j w_j o[r][j] / sum_j w_j.
 *   o_part [rows][max_splits][head_dim], lse_part [rows][max_splits],
 *   num_splits [rows] (rows with a count outside [1, max_splits], or whose
 *   every lse is -inf, are written as zeros), out [rows][head_dim] fp32.
 *   head_dim 1 .. 1024.
 */
int paged_kv_split_combine(const float *o_part, const float *lse_part, const int32_t *num_splits,
                           float *out, int rows, int max_splits, int head_dim, void *stream);

/*
 * Read the pool's device error word (PKV_ERR_* bits) into *bits; with reset
 * != 0 also clear it. Synchronises the device.
 */
int pkv_get_error(pkv_pool_t *pool, int *bits, int reset);

/* cudaError_t value of the calling thread's last CUDA failure (0 if none). */
int pkv_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
