// Internal interface shared by the attention translation units: workspace
// layout, plan output, kernel parameter blocks and the prefill launcher.
#pragma once

#include "pkv_common.cuh"

namespace pkv {

constexpr int kMaxSplits = 32;        // key ranges per split row, at most
constexpr int kDecodeTileMaxRows = 64;  // longer requests go to the tensor-core prefill kernel
constexpr int kPrefillRows = 128;     // rows of one prefill tile (M of the MMA)
constexpr int kPrefillKeys = 128;     // keys of one prefill KV tile (N of S = Q K^T)
constexpr int32_t kMagic = 0x504B5633;  // "PKV3"

struct WsHeader {
    int32_t status;          // device status word (first 4 bytes)
    int32_t magic;
    int32_t n_chunks;        // decode-kernel chunks
    int32_t num_tokens;
    int32_t num_q_heads;
    int32_t head_size;
    int32_t num_seqs;
    int32_t pages_per_split;
    int32_t n_ptiles;        // prefill-kernel tiles
    int32_t n_crows;         // rows of the shared-prefix (cascade) pass, per kv head
    int32_t prefix_blocks;   // shared prefix in blocks (0: no cascade)
    int32_t prefix_parts;    // the prefix keys are cut into this many splits (KV-tile ranges)
    int32_t next_ptile_item;    // prefill kernel: next work item to claim, less its grid size
    int32_t next_prefix_item;   // shared-prefix pass: the same
    int32_t n_split_tokens;     // tokens whose rows the combine merges
    int32_t pad_;
    int64_t off_req;         // int4 [num_seqs]: {splits (0: refused), partial row base, first chunk, chunks}
    int64_t off_stoks;       // int4 [num_tokens]: split tokens {token, partial row of q head 0, splits, 0}
    int64_t off_chunks;      // int4 [max_chunks]: {request, split or tile, page begin, page end}
    int64_t off_ptiles;      // int4 [max_ptiles]: {request, q tile, kv tiles, 0}
    int64_t off_crows;       // int4 [max_crows]: {token, request, query index, q head in group}
    int64_t off_part_lse;    // float [max_prow]
    int64_t off_part_o;      // float [max_prow][head_size]
    int64_t max_chunks;
    int64_t max_ptiles;
    int64_t max_crows;
    int64_t max_prow;
    int64_t prow_used;
};
static_assert(sizeof(WsHeader) <= 256, "header must fit its 256-byte slot");

// After the header: int32 [2][kStatsCtas], the work items each CTA of the
// persistent prefill kernel (row 0) and of the shared-prefix pass (row 1)
// took, zeroed by the plan (a record of the dynamic schedule).
constexpr int64_t kStatsOffset = 256;
constexpr int kStatsCtas = 1024;

struct WsLayout {
    int64_t off_req, off_stoks, off_chunks, off_ptiles, off_crows, off_part_lse, off_part_o, total;
    int64_t max_chunks, max_ptiles, max_crows, max_prow;
    int32_t prefix_parts;     // splits of the shared prefix (0: no cascade)
};

// CTAs the shared-prefix pass aims for: one per SM of a 152-SM part (the
// kernel holds all of an SM's tensor memory).  Only the balance depends on it.
constexpr int kPrefixTargetCtas = 152;

struct PrefillParams {
    __nv_bfloat16 *out;
    const int32_t *block_tables;
    int32_t max_blocks_per_seq;
    const int32_t *seq_lens;
    const int32_t *qsl;
    int32_t num_q_heads, num_kv_heads, G;
    int64_t num_blocks;
    float scale_log2;
    int32_t lo_tiles;         // leading KV tiles whose P always enters P V as a bf16 pair
    float k_scale, v_scale;   // E4M3 cache: stored code * scale is the value
    uint8_t *ws;
};

// Parameters of the decode kernel (decode.cu).
struct AttnParams {
    __nv_bfloat16 *out;
    const __nv_bfloat16 *query;
    int64_t q_stride;         // elements per token
    const int32_t *block_tables;
    int32_t max_blocks_per_seq;
    const int32_t *seq_lens;
    const int32_t *qsl;
    int32_t num_q_heads, num_kv_heads, G;
    int64_t num_blocks;
    float scale_log2;         // scale * log2(e)
    float k_scale, v_scale;   // E4M3 cache: stored code * scale is the value (1 for bf16)
    uint8_t *ws;
};

// Decode grid: persistent CTAs of kDecodeWarps warps, decode_ctas_per_sm()
// per SM (set by the tiling of the head size and cache type).
constexpr int kDecodeWarps = 4;
int decode_ctas_per_sm(int32_t head_size, bool kv8);

// Tensor map of the cache for the decode kernel (bf16 or E4M3 pages).
int make_decode_map(CUtensorMap *map, const void *kv_cache, int64_t num_blocks, int32_t num_kv_heads,
                    int32_t head_size, bool kv8);
// Launch the decode kernel for this head size and cache type (programmatic
// dependent launch after the plan).
int launch_decode_path(const CUtensorMap &map, const AttnParams &ap, int32_t head_size, bool kv8, int grid, int dev,
                       cudaStream_t st);

// The shared-prefix (cascade) pass on the same kernel: rows of every request
// that shares the first `prefix_blocks` blocks of its table with request 0
// attend once to those blocks' keys, cut into `prefix_parts` ranges of KV
// tiles; range i is split i of each row.
int launch_prefix(const PrefillParams &p, const void *query, int64_t q_stride, const void *kv_cache,
                  int64_t num_blocks, int32_t head_size, int64_t grid, int dev, cudaStream_t stream,
                  bool kv8 = false);

// Is the tensor-core prefill kernel available for this head layout?
inline bool prefill_supported(int num_q_heads, int num_kv_heads, int head_size) {
    const int G = num_q_heads / num_kv_heads;
    return (head_size == 64 || head_size == 128) && G >= 1 && G <= kPrefillRows && (kPrefillRows % G) == 0;
}

// Host launcher of the prefill kernel (prefill_tc.cu).  `grid` CTAs; CTAs
// beyond the plan's tile count return at once.
int launch_prefill(const PrefillParams &p, const void *query, int64_t q_stride, int32_t num_tokens,
                   const void *kv_cache, int64_t num_blocks, int32_t head_size, int64_t grid, int dev,
                   cudaStream_t stream, bool kv8 = false);

}  // namespace pkv
