/*
 * pkv.h — C ABI of the paged KV-cache attention library (libpagedkv.so).
 *
 * One engine step of PagedAttention over a block-table-indexed KV cache, as
 * the vLLM pages describe it: new K/V tokens are scattered into physical
 * cache slots given by slot_mapping, then every query token attends
 * causally over its own request's logical blocks, read through the
 * request's block table.
 *
 * Sources of the operations (page title, section):
 *  - "vLLM internals: managing the KV cache like an OS manages memory",
 *    section 2.1: the cache is cut into 16-token blocks, a per-request block
 *    table maps logical to physical blocks, and a fused cache-write op stores
 *    each new token's K/V in its physical slot.
 *  - "continuous batching and PagedAttention" tutorial (juhe.plus), section
 *    3.3 "Data structures" (logical token -> block, offset -> physical block)
 *    and section 3.6 "PagedAttention kernel" (loop over the request's
 *    blocks, look up the physical block, load K/V, accumulate softmax(QK^T)V).
 *  - "Inside vLLM: Anatomy of a High-Throughput LLM Inference System",
 *    "Executing the forward pass": slot_mapping is built when inputs are
 *    prepared, and all sequences are flattened into one super-sequence whose
 *    positions keep each sequence attending only to its own tokens.
 *  - "vLLM source reading", section 5.1: the kernel scatters new K/V by
 *    slot_mapping and gathers cached K/V by block table.
 *
 * Conventions shared by every call
 *  - All tensor pointers are DEVICE pointers owned by the caller.  The
 *    library allocates nothing, keeps no state between calls, and enqueues
 *    its kernels on `stream` (a cudaStream_t; NULL is the legacy default
 *    stream) in call order.  Calls return after enqueueing, not after the
 *    GPU has finished.
 *  - bf16 means IEEE bfloat16 (16-bit) values; int32/int64 are little-endian
 *    two's complement.
 *  - Host-side argument errors are returned BEFORE anything is enqueued.
 *    Errors the GPU finds (a slot or block id outside the cache, inconsistent
 *    lengths, a bounded wait that ran out) are written to a device status
 *    word (see each call); the host reads it after synchronising.
 *  - Block size is fixed at 16 tokens.  Head size is 64 or 128.
 *  - The attention calls launch their first kernel with programmatic
 *    dependent launch: it may start while the kernel just before it on the
 *    stream (normally pkv_kv_write) is still running, and it reads
 *    seq_lens, query_start_loc and block_tables at once.  Work of any
 *    ordinary kind before the call (copies, memsets, kernels launched
 *    without programmatic dependent launch) is complete by then.  A
 *    caller's own kernel that releases its dependents early
 *    (griddepcontrol.launch_dependents) must write that metadata first.
 *
 * KV cache layout (this library's own, not the one printed on the pages):
 *     bf16 kv_cache[num_blocks][num_kv_heads][2][16][head_size]
 *  index 0 of the third axis holds K, index 1 holds V.  A slot number is
 *  block * 16 + offset.  One block of one kv head is 2*16*head_size*2 bytes
 *  (8 KiB at head_size 128), contiguous; the whole cache is the pages'
 *  per-block formula 2 * block_size * num_kv_heads * head_size * 2 bytes
 *  times num_blocks.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PKV_BLOCK_SIZE 16

typedef enum pkv_status {
    PKV_OK = 0,
    PKV_ERR_NULL = 1,            /* a required pointer is NULL                        */
    PKV_ERR_SHAPE = 2,           /* sizes negative or inconsistent with each other    */
    PKV_ERR_UNSUPPORTED = 3,     /* head_size not 64/128, block_size not 16, ...      */
    PKV_ERR_ALIGNMENT = 4,       /* a pointer or stride breaks the stated alignment   */
    PKV_ERR_WORKSPACE = 5,       /* workspace missing or too small (size reported)    */
    PKV_ERR_CUDA = 6,            /* a CUDA runtime call or kernel launch failed       */
    /* written by the GPU into a device status word: */
    PKV_ERR_DEVICE_INDEX = 7,    /* a slot or block id outside the cache was skipped  */
    PKV_ERR_DEVICE_METADATA = 8, /* seq_len < query_len, query_start_loc not ordered, */
                                 /* a sequence longer than its table or the hints     */
    PKV_ERR_DEVICE_TIMEOUT = 9,  /* a bounded wait on an asynchronous copy ran out    */
    PKV_ERR_PROTOCOL = 10        /* combine given a workspace paged_attn did not fill */
                                 /* for the same num_tokens/num_q_heads/head_size     */
} pkv_status;

/*
 * pkv_kv_write — the cache write ("reshape_and_cache").
 *
 * For every token t in [0, num_tokens) with slot_mapping[t] >= 0:
 *     b = slot_mapping[t] / 16, o = slot_mapping[t] % 16, and for every kv head h
 *     kv_cache[b][h][0][o][:] = key  [t][h][:]   (bit copy)
 *     kv_cache[b][h][1][o][:] = value[t][h][:]
 * Tokens with a negative slot are padding and are skipped.  Nothing else in
 * the cache changes.  Two tokens with the same slot in one call leave that
 * slot holding one of them (which one is unspecified).
 *
 *  kv_cache            bf16, layout above; 16-byte aligned.
 *  num_blocks          blocks in the cache (>= 1).
 *  key, value          bf16; token t, head h starts at ptr + t*token_stride + h*head_size;
 *                      heads of one token are contiguous.  16-byte aligned.
 *  *_token_stride      elements between consecutive tokens (a multiple of 8,
 *                      >= num_kv_heads*head_size); lets K/V be views of a fused QKV.
 *  slot_mapping        int64 [num_tokens].
 *  device_status       optional int32 device word (may be NULL).  If a slot is
 *                      >= num_blocks*16, that token is skipped and
 *                      PKV_ERR_DEVICE_INDEX is stored there.  The library never
 *                      clears it: the caller zeroes it beforehand.
 * Returns PKV_OK or a host-side error code; num_tokens == 0 enqueues nothing.
 */
int pkv_kv_write(void *kv_cache, int64_t num_blocks, int32_t num_kv_heads,
                 int32_t head_size, int32_t block_size,
                 const void *key, int64_t key_token_stride,
                 const void *value, int64_t value_token_stride,
                 const int64_t *slot_mapping, int32_t num_tokens,
                 int32_t *device_status, void *stream);

/*
 * pkv_paged_attn — causal paged attention for one flattened batch.
 *
 * Request r owns query tokens [query_start_loc[r], query_start_loc[r+1]);
 * with q_r of them and seq_lens[r] = L_r, its context is c_r = L_r - q_r and
 * its i-th query token sits at position c_r + i.  That token's row for q
 * head h is
 *     out[t][h][:] = sum_j softmax_j(scale * <query[t][h], K_j>) * V_j,
 *     j = 0 .. c_r + i,
 * where K_j, V_j are read from block block_tables[r][j / 16], offset j % 16,
 * kv head h / (num_q_heads / num_kv_heads) (grouped-query attention).  The
 * request's new tokens must already be in the cache (call pkv_kv_write
 * first, on the same stream).  Scores and the softmax are fp32; out is bf16
 * rounded to nearest even.
 *
 * Long rows of short requests are split along their keys (split-K
 * flash-decoding): this call writes `out` directly for rows that were not
 * split and leaves per-split partial results in the workspace for the rest.
 * pkv_paged_attn_combine MUST follow on the same stream to finish those rows.
 *
 *  out               bf16 [num_tokens][num_q_heads][head_size], contiguous, 16-byte aligned.
 *  query             bf16; token t, head h at query + t*query_token_stride + h*head_size;
 *                    16-byte aligned, stride a multiple of 8.
 *  kv_cache          bf16, layout above, 16-byte aligned; num_blocks in [1, 2^31) and
 *                    num_blocks * num_kv_heads < 2^31 (PKV_ERR_SHAPE otherwise; such a
 *                    cache is terabytes).
 *  block_tables      int32 [num_seqs][max_blocks_per_seq]; entries past
 *                    ceil(L_r/16) are never read.
 *  seq_lens          int32 [num_seqs].
 *  query_start_loc   int32 [num_seqs+1], non-decreasing, [0] = 0, [num_seqs] <= num_tokens.
 *  max_query_len,
 *  max_seq_len       host-side upper bounds of q_r and L_r; they size the
 *                    workspace.  A device value above its bound is an error
 *                    (PKV_ERR_DEVICE_METADATA) and that request's rows are
 *                    left unwritten.
 *  scale             softmax scale, e.g. 1/sqrt(head_size).
 *  num_splits        0 = automatic; k > 0 splits each splittable row's keys
 *                    into min(k, 32, pages) parts (testing and tuning).
 *  workspace         device scratch of workspace_bytes (256-byte aligned).
 *                    Its first int32 is the device status word: this call
 *                    resets it to PKV_OK and the GPU stores an error code there.
 *  workspace_needed  if not NULL, receives the bytes this call needs.  With
 *                    workspace == NULL or too small, nothing is enqueued and
 *                    PKV_ERR_WORKSPACE is returned (the size query).
 * The workspace depends only on num_seqs, num_tokens, max_query_len,
 * max_seq_len, the head counts and head_size; one workspace serves any number
 * of calls in stream order.
 */
int pkv_paged_attn(void *out, const void *query, int64_t query_token_stride,
                   const void *kv_cache, int64_t num_blocks,
                   const int32_t *block_tables, int32_t max_blocks_per_seq,
                   const int32_t *seq_lens, const int32_t *query_start_loc,
                   int32_t num_seqs, int32_t num_tokens,
                   int32_t max_query_len, int32_t max_seq_len,
                   int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
                   int32_t block_size, float scale, int32_t num_splits,
                   void *workspace, size_t workspace_bytes, size_t *workspace_needed,
                   void *stream);

/*
 * pkv_paged_attn_shared_prefix — pkv_paged_attn for a batch whose requests
 * share a prefix of their block tables (cascade attention).
 *
 * Requests that share a prefix keep one physical copy of its blocks, each
 * block referenced from every sharer's table ("vLLM internals: managing the
 * KV cache like an OS manages memory", section 2.2: shared blocks with
 * reference counts; "continuous batching and PagedAttention" tutorial,
 * sections 3.5 and 5.2: parallel sampling, beam search and prefix caching
 * share the prompt's blocks).  This call computes exactly the result of
 * pkv_paged_attn (same arguments, same formula, same combine afterwards),
 * but reads the shared blocks once per kv head for all sharers: the keys of
 * the first `shared_prefix_blocks` table entries are attended by every
 * sharing row together on tensor-core tiles, cut into a few key ranges that
 * become splits of that row, and merged with the row's own keys by the
 * log-sum-exp combine (at most 32 splits per row in all).
 *
 * A request takes this path when its first shared_prefix_blocks table entries
 * equal request 0's, its query rows fit one decode tile (q_r * G <= 16) and
 * its context covers the prefix (L_r - q_r >= 16 * shared_prefix_blocks;
 * request 0's must too).  Other requests are computed as by pkv_paged_attn.
 * shared_prefix_blocks = 0 is pkv_paged_attn.  The workspace size also
 * depends on shared_prefix_blocks.
 */
int pkv_paged_attn_shared_prefix(void *out, const void *query, int64_t query_token_stride,
                                 const void *kv_cache, int64_t num_blocks,
                                 const int32_t *block_tables, int32_t max_blocks_per_seq,
                                 const int32_t *seq_lens, const int32_t *query_start_loc,
                                 int32_t num_seqs, int32_t num_tokens,
                                 int32_t max_query_len, int32_t max_seq_len,
                                 int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
                                 int32_t block_size, float scale, int32_t num_splits,
                                 int32_t shared_prefix_blocks,
                                 void *workspace, size_t workspace_bytes, size_t *workspace_needed,
                                 void *stream);

/*
 * FP8 KV cache ("vLLM internals: managing the KV cache like an OS manages
 * memory", section 7.2: the KV cache itself can be kept in FP8; "continuous
 * batching and PagedAttention" tutorial, sections 8.8 and 10.3 and the FAQ
 * of 10.8: an FP8 KV cache halves its memory at almost no loss).
 *
 * The cache has the bf16 layout with one byte per element:
 *     uint8 [num_blocks][num_kv_heads][2][16][head_size]
 * each byte an E4M3 code (OCP FP8: sign, 4 exponent bits with bias 7, 3
 * mantissa bits; exponent 0 subnormal; 0x7F and 0xFF NaN; largest finite
 * 448).  One fp32 scale covers all K (k_scale) and one all V (v_scale); a
 * stored code c stands for value(c) * scale.
 *
 * pkv_kv_write_fp8 — pkv_kv_write into an E4M3 cache.  Element x (bf16) of
 * a new K (V) row is stored as the E4M3 code nearest to the fp32 quotient
 * x / k_scale (x / v_scale), computed with IEEE division rounded to nearest;
 * ties go to the even code and magnitudes beyond 448 are held at 448, with
 * the sign kept (a result that rounds to zero keeps its sign).  Arguments
 * as pkv_kv_write; k_scale and v_scale must be positive and finite
 * (PKV_ERR_SHAPE otherwise).
 */
int pkv_kv_write_fp8(void *kv_cache, int64_t num_blocks, int32_t num_kv_heads,
                     int32_t head_size, int32_t block_size,
                     const void *key, int64_t key_token_stride,
                     const void *value, int64_t value_token_stride,
                     const int64_t *slot_mapping, int32_t num_tokens,
                     float k_scale, float v_scale,
                     int32_t *device_status, void *stream);

/*
 * pkv_paged_attn_fp8 — pkv_paged_attn over an E4M3 cache, with K_j and V_j
 * taken as value(code) * k_scale and value(code) * v_scale; arguments,
 * workspace and protocol (pkv_paged_attn_combine after it) as
 * pkv_paged_attn.  Decode rows run on the streaming decode kernel, long
 * chunks on the tensor-core kernel with K and V widened to f16 in shared
 * memory.  Scores, softmax and accumulation are fp32; the query enters the
 * products as f16 after a per-row power-of-two scaling (exact for every
 * query element not below 2^-24 of its row's largest).
 */
int pkv_paged_attn_fp8(void *out, const void *query, int64_t query_token_stride,
                       const void *kv_cache, int64_t num_blocks,
                       const int32_t *block_tables, int32_t max_blocks_per_seq,
                       const int32_t *seq_lens, const int32_t *query_start_loc,
                       int32_t num_seqs, int32_t num_tokens,
                       int32_t max_query_len, int32_t max_seq_len,
                       int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
                       int32_t block_size, float scale, float k_scale, float v_scale,
                       int32_t num_splits,
                       void *workspace, size_t workspace_bytes, size_t *workspace_needed,
                       void *stream);

/*
 * pkv_paged_attn_shared_prefix_fp8 — pkv_paged_attn_shared_prefix over an
 * E4M3 cache, with K_j and V_j taken as value(code) * k_scale and
 * value(code) * v_scale (as pkv_paged_attn_fp8): the shared prefix's keys are
 * read once per kv head for all sharers, widened to f16 in shared memory.
 * Arguments, workspace (sized as for pkv_paged_attn_shared_prefix) and
 * protocol (pkv_paged_attn_combine after it) as pkv_paged_attn_shared_prefix.
 */
int pkv_paged_attn_shared_prefix_fp8(void *out, const void *query, int64_t query_token_stride,
                                     const void *kv_cache, int64_t num_blocks,
                                     const int32_t *block_tables, int32_t max_blocks_per_seq,
                                     const int32_t *seq_lens, const int32_t *query_start_loc,
                                     int32_t num_seqs, int32_t num_tokens,
                                     int32_t max_query_len, int32_t max_seq_len,
                                     int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
                                     int32_t block_size, float scale, float k_scale, float v_scale,
                                     int32_t num_splits, int32_t shared_prefix_blocks,
                                     void *workspace, size_t workspace_bytes, size_t *workspace_needed,
                                     void *stream);

/*
 * pkv_paged_attn_combine — the log-sum-exp merge of split rows.
 *
 * For every row (t, h) that pkv_paged_attn split into n parts with partial
 * outputs o_s (each normalised over its own keys) and lse_s = log of the sum
 * of exp(score) over that part's keys:
 *     M = max_s lse_s,  w_s = exp(lse_s - M),
 *     out[t][h][:] = sum_s w_s o_s / sum_s w_s      (bf16, nearest even);
 * a part with no visible key has lse_s = -inf and weight 0.  Rows that were
 * not split are left untouched.
 *
 *  out, workspace    the same buffers given to the preceding pkv_paged_attn;
 *  num_tokens, num_q_heads, head_size
 *                    the same values; a mismatch with what that call recorded
 *                    in the workspace stores PKV_ERR_PROTOCOL in the status
 *                    word and writes nothing.
 */
int pkv_paged_attn_combine(void *out, const void *workspace, size_t workspace_bytes,
                           int32_t num_tokens, int32_t num_q_heads, int32_t head_size,
                           void *stream);

/*
 * pkv_copy_blocks — copy-on-write of shared blocks.
 *
 * "continuous batching and PagedAttention" tutorial, section 3.8 "COW and
 * reference counting" (and "vLLM internals: managing the KV cache like an OS
 * manages memory", section 2.2): a request about to write into a block that
 * other requests still share gets a fresh block holding a copy of the
 * shared one; its block table then points at the copy.  This call makes the
 * copies: for every pair p,
 *     kv_cache[block_mapping[2p+1]][h][k_or_v][:][:] =
 *         kv_cache[block_mapping[2p]][h][k_or_v][:][:]     for every kv head h,
 * a bit copy of all 2*16*head_size*2 bytes per kv head.  Pairs with a source
 * or destination outside [0, num_blocks) are skipped and PKV_ERR_DEVICE_INDEX
 * is stored in *device_status (when not NULL; never cleared by the library).
 * A block that is the destination of one pair and the source of another in
 * the same call has no defined result.
 *
 *  block_mapping   int64 [num_pairs][2]: {source block, destination block}.
 */
int pkv_copy_blocks(void *kv_cache, int64_t num_blocks, int32_t num_kv_heads,
                    int32_t head_size, int32_t block_size,
                    const int64_t *block_mapping, int32_t num_pairs,
                    int32_t *device_status, void *stream);

/*
 * pkv_paged_attn_noalloc — paged attention that allocates nothing.
 *
 * The pages have no counterpart to this call; it exists for callers that
 * cannot allocate GPU memory where they run attention (for example code
 * in a serving loop under a strict no-allocation policy, or a plugin whose
 * host engine owns all device memory and passes in only inputs and
 * outputs).  It computes exactly what pkv_paged_attn followed by
 * pkv_paged_attn_combine computes, with the same arguments except the
 * workspace: the scratch lives in a fixed array of this library's own device
 * memory, PKV_NOALLOC_SCRATCH_BYTES (256 MiB) on every GPU where the call's
 * code is loaded, held until the process exits.  It calls no cudaMalloc,
 * cudaFree or other allocating routine.
 *
 *  - Sizes whose scratch (the workspace size pkv_paged_attn would report)
 *    exceeds PKV_NOALLOC_SCRATCH_BYTES are refused with PKV_ERR_WORKSPACE
 *    before anything is enqueued; argument errors return the same codes as
 *    pkv_paged_attn.
 *  - Every call looks up the array's device address on the current device
 *    (a host-side query that enqueues nothing).  Under lazy module loading
 *    the first call on each device also loads this code onto the device;
 *    make that first call before any stream capture.
 *  - Every call on a device shares the one array and leaves its contents
 *    behind; each call rewrites all of the scratch it later reads, so nothing
 *    needs clearing between calls.  Calls that overlap on the GPU (other
 *    streams, other threads' streams) race on the array: keep them ordered,
 *    e.g. on one stream.
 *  - device_status: optional int32 device word.  After the call's kernels,
 *    an error the GPU found (a PKV_ERR_DEVICE_* code, or PKV_ERR_PROTOCOL)
 *    is stored there unless the word already holds an error: as for the
 *    other calls' status words, the first error stays and the library never
 *    clears the word, so the caller zeroes it beforehand.  A call that finds
 *    no error, or that has no requests (num_seqs == 0, nothing enqueued),
 *    leaves the word as it was.
 */
#define PKV_NOALLOC_SCRATCH_BYTES (256u << 20)

int pkv_paged_attn_noalloc(void *out, const void *query, int64_t query_token_stride,
                           const void *kv_cache, int64_t num_blocks,
                           const int32_t *block_tables, int32_t max_blocks_per_seq,
                           const int32_t *seq_lens, const int32_t *query_start_loc,
                           int32_t num_seqs, int32_t num_tokens,
                           int32_t max_query_len, int32_t max_seq_len,
                           int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
                           int32_t block_size, float scale, int32_t num_splits,
                           int32_t *device_status, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
