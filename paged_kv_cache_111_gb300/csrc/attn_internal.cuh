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
    int32_t epoch;              // decode kernel that plans itself: bumped once the header is written
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

// ---- splitting decode rows along their keys (the plan kernel, and the decode
// kernel when it plans a call itself, take the same decisions) ----

__host__ __device__ __forceinline__ int div_up(int a, int b) { return (a + b - 1) / b; }

// Pages per warp up to which a warp takes one chunk.
constexpr unsigned long long kOneChunkPages = 24;

// The automatic split size from the call's decode work (pages x kv heads)
// and the decode grid's warps.  Chunks of 4..64 pages.  Each chunk starts with
// a chain of dependent loads (its record, the request's lengths, the block
// table and Q), so a small batch (at most kOneChunkPages pages per warp) gets
// one chunk per warp; a larger one about three per warp, so that the warps
// finish together.
__device__ __forceinline__ int auto_pages_per_split(unsigned long long total_pages, int num_kv_heads,
                                                    int total_warps) {
    const unsigned long long work = total_pages * (unsigned long long)num_kv_heads;
    const unsigned long long warps = (unsigned long long)max(total_warps, 1);
    const unsigned long long per1 = (work + warps - 1) / warps;
    const unsigned long long per = per1 <= kOneChunkPages ? per1 : (work + 3 * warps - 1) / (3 * warps);
    return (int)min(64ull, max(4ull, per));
}

// {pages per split, splits} of a split row whose keys span `span` pages: at
// most `cap` splits; num_splits > 0 asks for that many, else splits of about
// pages_per_split pages; no split is empty.
__device__ __forceinline__ int2 split_geometry(int span, int pages_per_split, int num_splits, int cap) {
    int n;
    if (num_splits > 0) {
        n = min(min(num_splits, cap), span);
    } else {
        const int per = max(pages_per_split, div_up(span, cap));
        n = div_up(span, per);
    }
    const int per_split = div_up(span, n);
    return make_int2(per_split, div_up(span, per_split));
}

// Is request r's metadata consistent (query rows [q0, q1), L keys)?
__device__ __forceinline__ bool request_valid(int q0, int q1, int L, int num_tokens, int max_seq_len,
                                              int max_query_len, int max_blocks_per_seq) {
    const int q = q1 - q0;
    return !(q0 < 0 || q < 0 || q1 > num_tokens || L < q || L > max_seq_len || q > max_query_len ||
             div_up(L, kBlock) > max_blocks_per_seq);
}

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

// Log-sum-exp merge of one split row by one warp: the row's n partial
// outputs (part_o rows base .. base + n - 1, each normalised over its own
// keys) and their natural log-sum-exps (part_lse) give
//     M = max_s lse_s,  w_s = e^{lse_s - M},  out = sum_s w_s o_s / sum_s w_s
// (a part with lse = -inf weighs 0), written to dst as bf16.  The partials
// are read through L2 (ld.global.cg).  The log-sum-exps and a batch of partial rows (16 at head size
// 64, 8 at 128) are loaded together before any arithmetic: the merge is a
// short chain of dependent loads, bound by their latency.  n <= 32.
template <int HD>
__device__ __forceinline__ void merge_split_row(const float *part_o, const float *part_lse, int64_t base, int n,
                                                __nv_bfloat16 *dst, int lane) {
    const float NEG_INF = -__int_as_float(0x7f800000);
    constexpr int PER = HD / 32;              // dims per lane (2 or 4)
    constexpr int U = HD == 64 ? 16 : 8;
    auto load = [&](int64_t prow) -> float4 {
        const float *src = part_o + prow * HD + lane * PER;
        if constexpr (PER == 4) {
            return __ldcg(reinterpret_cast<const float4 *>(src));
        } else {
            const float2 v = __ldcg(reinterpret_cast<const float2 *>(src));
            return make_float4(v.x, v.y, 0.f, 0.f);
        }
    };
    const float lse = lane < n ? __ldcg(part_lse + base + lane) : NEG_INF;
    float4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) v[u] = u < n ? load(base + u) : make_float4(0.f, 0.f, 0.f, 0.f);
    float mx = lse;
#pragma unroll
    for (int s = 16; s; s >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, s));
    const float w = (lse == NEG_INF) ? 0.f : __expf(lse - mx);
    float wsum = w;
#pragma unroll
    for (int s = 16; s; s >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, s);
    float acc[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = 0.f;
    for (int s0 = 0;;) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const float wt = __shfl_sync(0xffffffffu, w, (s0 + u) & 31);   // 0 past the last split
            acc[0] += wt * v[u].x;
            acc[1] += wt * v[u].y;
            if constexpr (PER == 4) {
                acc[2] += wt * v[u].z;
                acc[3] += wt * v[u].w;
            }
        }
        s0 += U;
        if (s0 >= n) break;
#pragma unroll
        for (int u = 0; u < U; ++u) v[u] = s0 + u < n ? load(base + s0 + u) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    __nv_bfloat16 *d = dst + lane * PER;
    if constexpr (PER == 4) {
        *reinterpret_cast<uint2 *>(d) =
            make_uint2(pack_bf16x2(acc[0] * inv, acc[1] * inv), pack_bf16x2(acc[2] * inv, acc[3] * inv));
    } else {
        *reinterpret_cast<uint32_t *>(d) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    }
}

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
    // self_plan = 1: no plan kernel ran; the decode kernel plans the call
    // itself (see decode_self_plan_ok) and writes what the combine reads
    int32_t self_plan;
    int32_t num_seqs, num_tokens, head_size, max_query_len, max_seq_len;
    int32_t total_warps;      // warps of the decode grid
    WsLayout lay;
};

// Requests a decode kernel plans by itself at most (their lengths and plans
// sit in its shared memory before its rings are used).
constexpr int kSelfPlanSeqs = 1024;

// May the decode kernel plan this call itself?  Every request is a split row
// (max_query_len * G <= 16), nothing else runs (no prefill, no shared
// prefix), the split size is automatic, and the batch is small enough that
// every warp takes at most two chunks: num_seqs * kv heads <= warps, and the
// bound on the pages (num_seqs * ceil(max_seq_len / 16) * kv heads) is at
// most kOneChunkPages per warp.  (Then the plan's size order is moot: the
// chunks number at most the warps plus one per (request, kv head).)
inline bool decode_self_plan_ok(int64_t num_seqs, int64_t max_query_len, int64_t max_seq_len, int64_t G,
                                int64_t num_kv_heads, int64_t num_splits, int64_t prefix_blocks, int64_t warps) {
    if (num_seqs < 1 || num_seqs > kSelfPlanSeqs || num_splits != 0 || prefix_blocks != 0) return false;
    if (max_query_len * G > 16) return false;
    if (num_seqs * num_kv_heads > warps) return false;
    const int64_t pages = (max_seq_len + kBlock - 1) / kBlock;
    return num_seqs * pages * num_kv_heads <= static_cast<int64_t>(kOneChunkPages) * warps;
}

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

// The one-tile tensor-core kernel over an E4M3 cache (prefill_tc.cu): the
// shared-prefix (cascade) pass (rows of every request that shares the first
// `prefix_blocks` blocks of its table with request 0 attend once to those
// blocks' keys, cut into `prefix_parts` ranges of KV tiles; range i is split
// i of each row) and the chunks.  `grid` CTAs; CTAs beyond the plan's items
// return at once.
int launch_prefix_e4m3(const PrefillParams &p, const void *query, int64_t q_stride, const void *kv_cache,
                       int64_t num_blocks, int32_t head_size, int64_t grid, int dev, cudaStream_t stream);
int launch_prefill_e4m3(const PrefillParams &p, const void *query, int64_t q_stride, const void *kv_cache,
                        int64_t num_blocks, int32_t head_size, int64_t grid, int dev, cudaStream_t stream);

// Is the tensor-core prefill kernel available for this head layout?
inline bool prefill_supported(int num_q_heads, int num_kv_heads, int head_size) {
    const int G = num_q_heads / num_kv_heads;
    return (head_size == 64 || head_size == 128) && G >= 1 && G <= kPrefillRows && (kPrefillRows % G) == 0;
}

// Host launcher of the split-key prefill kernel over a bf16 cache
// (prefill_sk.cu): chunks (cascade = false) or the shared-prefix pass
// (cascade = true).  `grid` CTAs; CTAs beyond the plan's items return at once.
int launch_prefill_sk(const PrefillParams &p, const void *query, int64_t q_stride, int32_t num_tokens,
                      const void *kv_cache, int64_t num_blocks, int32_t head_size, bool cascade, int64_t grid, int dev,
                      cudaStream_t stream);

}  // namespace pkv
