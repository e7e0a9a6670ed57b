// Paged attention over a block-table-indexed KV cache, and its split-K merge.
//
// What is computed ("continuous batching and PagedAttention" tutorial,
// section 3.6 "PagedAttention kernel"; "vLLM source reading", sections 2.3
// and 5.1): every query row loops over its request's logical blocks, looks
// up the physical block in the block table, loads that block's K and V and
// folds softmax(scale * q.K^T) V into a running (max, sum, accumulator) state.
// Each request only sees its own tokens ("Inside vLLM: Anatomy of a
// High-Throughput LLM Inference System", "Executing the forward pass").
//
// How it runs on sm_103a (kernels enqueued by two calls, back to back with
// programmatic dependent launch; the decode kernel is in decode.cu, the
// tensor-core tile kernel in prefill_tc.cu):
//  1. plan_kernel (one CTA) reads seq_lens / query_start_loc, checks them,
//     and lists work chunks in the workspace, largest first.  A request whose
//     query rows for one kv head fit one 16-row tile (q_r * G <= 16: decode,
//     and short speculative-verify queries) has its keys split into up to 32
//     ranges of whole pages (split-K flash-decoding); a longer request is cut
//     into 16-row tiles that each stream every key they may see.
//  2. decode_kernel: persistent CTAs of NW warps.  Each warp takes chunks
//     (x kv heads) in a fixed order and streams the chunk's 16-token pages
//     through its own ring of DEPTH shared-memory stages.  A page of one kv
//     head (K then V, 2*16*head_size bf16, contiguous in the cache) arrives by
//     TMA tensor loads with 128-byte swizzle, so ldmatrix reads are free of
//     bank conflicts.  S = Q K^T and O += P V run on bf16 mma.sync tiles:
//     rows are the tile's (query token, q head of the group) pairs, so every
//     q head of a GQA group is served by one read of each KV page.
//  3. combine_kernel (second call): log-sum-exp merge of split rows.
//
// Masking never multiplies by zero: scores of keys a row may not see are
// replaced by -inf before the exponent, and V rows past the sequence end in
// its last page are zeroed in shared memory before P V, so NaN in unwritten
// cache slots cannot reach an output.
#include <mutex>

#include "attn_internal.cuh"

namespace pkv {

constexpr int kPlanThreads = 1024;
constexpr int kSizeBins = 256;      // counting-sort bins for chunk sizes (pages or KV tiles)

// ---- workspace layout ---------------------------------------------------------

static inline int64_t align256(int64_t x) { return (x + 255) & ~int64_t(255); }

static WsLayout ws_layout(int64_t num_seqs, int64_t num_tokens, int64_t max_query_len, int64_t max_seq_len,
                          int64_t num_q_heads, int64_t num_kv_heads, int64_t head_size, int64_t prefix_blocks) {
    const int64_t G = num_q_heads / num_kv_heads;
    WsLayout w;
    // split rows: requests with q_r * G <= 16, so q_r <= 16 / G
    const int64_t q_split = G <= 16 ? 16 / G : 0;
    int64_t split_tokens = num_seqs * q_split;
    if (split_tokens > num_tokens) split_tokens = num_tokens;
    const int64_t max_pages = (max_seq_len + kBlock - 1) / kBlock;
    const int64_t splits = max_pages < kMaxSplits ? (max_pages > 0 ? max_pages : 1) : kMaxSplits;
    // the shared prefix is cut into prefix_parts KV-tile ranges so that its
    // tiles (row tiles x kv heads x parts) about fill the GPU; every range is
    // non-empty
    w.max_crows = prefix_blocks > 0 ? split_tokens * G : 0;
    w.prefix_parts = 0;
    if (prefix_blocks > 0) {
        const int64_t kv_tiles = (prefix_blocks * kBlock + kPrefillKeys - 1) / kPrefillKeys;
        const int64_t row_tiles = (w.max_crows + kPrefillRows - 1) / kPrefillRows;
        int64_t parts = kPrefixTargetCtas / (row_tiles * num_kv_heads > 0 ? row_tiles * num_kv_heads : 1);
        parts = parts < 1 ? 1 : (parts > 8 ? 8 : parts);
        parts = parts > kv_tiles ? kv_tiles : parts;
        const int64_t per = (kv_tiles + parts - 1) / parts;
        w.prefix_parts = static_cast<int32_t>((kv_tiles + per - 1) / per);
    }
    // a cascade request's splits are its prefix ranges plus its own chunks
    w.max_prow = split_tokens * num_q_heads * (splits + w.prefix_parts);
    (void)max_query_len;
    // chunks: split requests give <= splits each; tiled ones ceil(q_r G / 16) <= q_r G / 16 + 1
    w.max_chunks = num_seqs * splits + (num_tokens * G + 15) / 16 + num_seqs;
    // prefill tiles: ceil(q_r G / 128) <= q_r G / 128 + 1
    w.max_ptiles = (num_tokens * G + kPrefillRows - 1) / kPrefillRows + num_seqs;
    int64_t off = kStatsOffset + 2 * kStatsCtas * 4;
    w.off_req = off;
    off = align256(off + 16 * num_seqs);
    w.off_stoks = off;
    off = align256(off + 16 * num_tokens);
    w.off_chunks = off;
    off = align256(off + 16 * w.max_chunks);
    w.off_ptiles = off;
    off = align256(off + 16 * w.max_ptiles);
    w.off_crows = off;
    off = align256(off + 16 * w.max_crows);
    w.off_part_lse = off;
    off = align256(off + 4 * w.max_prow);
    w.off_part_o = off;
    off = align256(off + 4 * w.max_prow * head_size);
    w.total = off;
    return w;
}

// ---- kernel parameters ----------------------------------------------------------

struct PlanParams {
    uint8_t *ws;
    const int32_t *seq_lens;
    const int32_t *qsl;
    int32_t num_seqs, num_tokens, num_q_heads, num_kv_heads, head_size;
    int32_t max_blocks_per_seq, max_query_len, max_seq_len;
    int32_t num_splits;       // 0 = auto
    int32_t total_warps;      // warps of the decode grid (for the automatic split size)
    int32_t prefill_ok;       // long requests go to the tensor-core prefill kernel
    int32_t prefix_blocks;    // shared prefix of the tables in blocks (0: no cascade)
    const int32_t *block_tables;
    WsLayout lay;
};


// ---- 1. planning ------------------------------------------------------------------

// Work of request r.  mode 0: rows split along key pages (q_r * G <= 16);
// mode 1: 16-row tiles on the decode kernel; mode 2: 128-row tiles on the
// tensor-core prefill kernel.
struct ReqPlan {
    int valid;        // metadata consistent
    int q, ctx;       // query tokens, context
    int rows;         // q_r * G
    int mode;
    int n_chunks;     // decode-kernel chunks (modes 0, 1) or prefill tiles (mode 2)
    int pages;        // key pages of the request (mode 0)
    int per_split;    // pages per split (mode 0)
    int first;        // first page of the decode chunks (mode 0): the shared prefix is split 0
};

// Mode 0 request r may take the cascade path: its table starts with request
// 0's first prefix_blocks blocks (`differs`: it does not), and every one of
// its rows sees all of them.
__device__ bool cascade_eligible(const PlanParams &p, const int *qsl, const int *lens, int r, bool differs) {
    const int K = p.prefix_blocks;
    if (K <= 0 || differs) return false;
    const int q = qsl[r + 1] - qsl[r];
    const int G = p.num_q_heads / p.num_kv_heads;
    if (q <= 0 || q * G > 16 || lens[0] - (qsl[1] - qsl[0]) < K * kBlock) return false;
    return lens[r] - q >= K * kBlock && K <= p.max_blocks_per_seq;
}

__device__ ReqPlan plan_request(const PlanParams &p, const int *qsl, const int *lens, int r, int pages_per_split,
                                bool cascade) {
    ReqPlan rp{0, 0, 0, 0, 0, 0, 0, 0, 0};
    const int G = p.num_q_heads / p.num_kv_heads;
    const int q0 = qsl[r], q1 = qsl[r + 1];
    const int q = q1 - q0;
    const int L = lens[r];
    if (!request_valid(q0, q1, L, p.num_tokens, p.max_seq_len, p.max_query_len, p.max_blocks_per_seq)) return rp;
    rp.valid = 1;
    rp.q = q;
    rp.ctx = L - q;
    rp.rows = q * G;
    if (rp.rows == 0) return rp;
    if (rp.rows <= 16) {
        rp.mode = 0;
        rp.pages = div_up(L, kBlock);
        rp.first = cascade ? p.prefix_blocks : 0;
        const int span = rp.pages - rp.first;            // >= 1: a cascade row sees a key past the prefix
        // at most kMaxSplits splits in all (the combine's limit), prefix ranges included
        const int cap = cascade ? kMaxSplits - p.lay.prefix_parts : kMaxSplits;
        const int2 sg = split_geometry(span, pages_per_split, p.num_splits, cap);
        rp.per_split = sg.x;
        rp.n_chunks = sg.y;
    } else if (p.prefill_ok && rp.rows > kDecodeTileMaxRows) {
        rp.mode = 2;
        rp.n_chunks = div_up(rp.rows, kPrefillRows);
    } else {
        rp.mode = 1;
        rp.n_chunks = div_up(rp.rows, 16);
    }
    return rp;
}

// What the chunks of a request need from its plan: {mode, first page (mode
// 0) or context, pages per split (mode 0) or rows, pages}.
__device__ __forceinline__ int4 chunk_geometry(const ReqPlan &rp) {
    return rp.mode == 0 ? make_int4(0, rp.first, rp.per_split, rp.pages) : make_int4(rp.mode, rp.ctx, rp.rows, rp.pages);
}

// Mode 0/1: page range of chunk k.  Mode 2: {0, KV tiles} of tile k.  A tile
// ending before request row `row_end` sees keys 0 .. ctx + last_row / G.
__device__ __forceinline__ int2 chunk_pages(const int4 &gm, int G, int k) {
    if (gm.x == 0) {
        const int b = gm.y + k * gm.z;
        return make_int2(b, min(gm.w, b + gm.z));
    }
    const int row_end = gm.x == 1 ? 16 * k + 16 : kPrefillRows * (k + 1);
    const int lim = gm.y + (min(gm.z, row_end) - 1) / G + 1;
    if (gm.x == 1) return make_int2(0, div_up(lim, kBlock));
    return make_int2(0, div_up(lim, kPrefillKeys));
}

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Exclusive scan of `count[b]` in descending bin order into `cursor[b]`, by
// one warp; returns the total.  Lane l holds the 8 bins 248 - 8l .. 255 - 8l
// (two 16-byte shared-memory accesses each way, free of bank conflicts), so
// lane 0 holds the largest sizes and its prefix is the warp scan's.
static_assert(kSizeBins == 32 * 8, "one warp scans the size bins, 8 per lane");
__device__ int scan_bins_desc(const int *count, int *cursor, int lane) {
    const int base = kSizeBins - 8 * (lane + 1);
    const int4 lo = *reinterpret_cast<const int4 *>(count + base);        // bins base .. base + 3
    const int4 hi = *reinterpret_cast<const int4 *>(count + base + 4);    // bins base + 4 .. base + 7
    const int sum = lo.x + lo.y + lo.z + lo.w + hi.x + hi.y + hi.z + hi.w;
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    int acc = incl - sum;                 // sizes above this lane's bins
    int4 chi, clo;                        // descending: base + 7 first
    chi.w = acc; acc += hi.w;
    chi.z = acc; acc += hi.z;
    chi.y = acc; acc += hi.y;
    chi.x = acc; acc += hi.x;
    clo.w = acc; acc += lo.w;
    clo.z = acc; acc += lo.z;
    clo.y = acc; acc += lo.y;
    clo.x = acc;
    *reinterpret_cast<int4 *>(cursor + base) = clo;
    *reinterpret_cast<int4 *>(cursor + base + 4) = chi;
    return __shfl_sync(0xffffffffu, incl, 31);
}

// Warp-aggregated shared-memory atomicAdd of 1 per lane on counter[bin]:
// returns this lane's slot (lanes sharing a bin get consecutive slots).
__device__ __forceinline__ int agg_inc(int *counter, int bin) {
    const unsigned active = __activemask();
    const unsigned peers = __match_any_sync(active, bin);
    const int leader = __ffs(peers) - 1;
    const int lane = threadIdx.x & 31;
    int base = 0;
    if (lane == leader) base = atomicAdd(&counter[bin], __popc(peers));
    base = __shfl_sync(peers, base, leader);
    return base + __popc(peers & ((1u << lane) - 1u));
}

// Block-wide exclusive scan of four non-negative counts (one set per
// thread); returns this thread's prefix and writes the totals to *total.
__device__ int4 block_scan4(int a, int b, int c, int d, int4 *warp_tot, int4 *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int4 in = make_int4(a, b, c, d);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int va = __shfl_up_sync(0xffffffffu, in.x, o);
        const int vb = __shfl_up_sync(0xffffffffu, in.y, o);
        const int vc = __shfl_up_sync(0xffffffffu, in.z, o);
        const int vd = __shfl_up_sync(0xffffffffu, in.w, o);
        if (lane >= o) {
            in.x += va;
            in.y += vb;
            in.z += vc;
            in.w += vd;
        }
    }
    if (lane == 31) warp_tot[warp] = in;
    __syncthreads();
    if (warp == 0) {
        const int nw = blockDim.x >> 5;
        const int4 w = lane < nw ? warp_tot[lane] : make_int4(0, 0, 0, 0);
        int4 x = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int va = __shfl_up_sync(0xffffffffu, x.x, o);
            const int vb = __shfl_up_sync(0xffffffffu, x.y, o);
            const int vc = __shfl_up_sync(0xffffffffu, x.z, o);
            const int vd = __shfl_up_sync(0xffffffffu, x.w, o);
            if (lane >= o) {
                x.x += va;
                x.y += vb;
                x.z += vc;
                x.w += vd;
            }
        }
        if (lane < nw) warp_tot[lane] = make_int4(x.x - w.x, x.y - w.y, x.z - w.z, x.w - w.w);   // exclusive
        if (lane == nw - 1) *total = x;
    }
    __syncthreads();
    const int4 wp = warp_tot[warp];
    return make_int4(wp.x + in.x - a, wp.y + in.y - b, wp.z + in.z - c, wp.w + in.w - d);
}

// One CTA plans the call: checks every request, splits decode rows along
// keys, cuts long requests into tiles, and lists the work largest first
// (counting sort by size) so the persistent decode kernel's fixed item order
// balances its warps.  Per-request and per-chunk passes run in parallel over
// requests and over chunks.  The requests' query starts, lengths and plans
// sit in shared memory when there are at most kPlanStagedSeqs of them (every
// pass then reads shared memory only); larger batches use the workspace.
constexpr int kPlanStagedSeqs = 1024;

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(PlanParams p) {
    __shared__ __align__(16) int bin_count[kSizeBins];
    __shared__ __align__(16) int bin_cursor[kSizeBins];
    __shared__ __align__(16) int pbin_count[kSizeBins];
    __shared__ __align__(16) int pbin_cursor[kSizeBins];
    __shared__ int bin_total[2];
    __shared__ int4 warp_tot[kPlanThreads / 32];
    __shared__ int4 totals;
    __shared__ unsigned long long total_pages;
    __shared__ int bad;
    __shared__ int pages_per_split;
    __shared__ int s_qsl[kPlanStagedSeqs + 1];
    __shared__ int s_len[kPlanStagedSeqs];
    __shared__ int4 s_req[kPlanStagedSeqs];
    __shared__ int4 s_geom[kPlanStagedSeqs];   // chunk geometry per request (staged batches)

    WsHeader *hdr = reinterpret_cast<WsHeader *>(p.ws);
    int4 *req_ws = reinterpret_cast<int4 *>(p.ws + p.lay.off_req);
    int4 *stoks = reinterpret_cast<int4 *>(p.ws + p.lay.off_stoks);
    int4 *chunks = reinterpret_cast<int4 *>(p.ws + p.lay.off_chunks);
    int4 *ptiles = reinterpret_cast<int4 *>(p.ws + p.lay.off_ptiles);
    int4 *crows = reinterpret_cast<int4 *>(p.ws + p.lay.off_crows);
    const int tid = threadIdx.x;
    const int nthr = blockDim.x;
    const int G = p.num_q_heads / p.num_kv_heads;
    pdl_trigger();
    // The kernel before this one on the stream (normally the cache write,
    // which touches neither the metadata nor the workspace) may still run.
    // A batch staged in shared memory is read and planned meanwhile; the
    // wait comes before the first workspace write.  A larger batch keeps
    // its per-request plans in the workspace and waits first.
    const bool staged = p.num_seqs <= kPlanStagedSeqs;
    if (!staged) pdl_wait();
    const int *qsl = staged ? s_qsl : p.qsl;
    const int *lens = staged ? s_len : p.seq_lens;
    // {splits (0: refused), partial row base, first chunk, chunks} per request;
    // .x is first the flag "table differs from request 0's in the prefix"
    int4 *req = staged ? s_req : req_ws;
    if (staged) {
        for (int r = tid; r <= p.num_seqs; r += nthr) s_qsl[r] = __ldg(p.qsl + r);
        for (int r = tid; r < p.num_seqs; r += nthr) s_len[r] = __ldg(p.seq_lens + r);
    }
    for (int i = tid; i < kSizeBins; i += nthr) {
        bin_count[i] = 0;
        pbin_count[i] = 0;
    }
    if (tid == 0) total_pages = 0;
    if (p.prefix_blocks > 0)
        for (int r = tid; r < p.num_seqs; r += nthr) req[r] = make_int4(0, 0, 0, 0);
    __syncthreads();
    if (tid == 0) bad = qsl[0] != 0;
    if (p.prefix_blocks > 0 && p.prefix_blocks <= p.max_blocks_per_seq) {
        // every (request, prefix block) pair at once, four loads in flight per thread
        const int K = p.prefix_blocks;
        const int64_t pairs = static_cast<int64_t>(p.num_seqs - 1) * K;
        for (int64_t i0 = tid; i0 < pairs; i0 += 4 * static_cast<int64_t>(nthr)) {
            int32_t a[4], b[4];
            int rr[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int64_t i = i0 + static_cast<int64_t>(u) * nthr;
                rr[u] = i < pairs ? 1 + static_cast<int>(i / K) : 0;
                const int blk = i < pairs ? static_cast<int>(i % K) : 0;
                a[u] = __ldg(p.block_tables + static_cast<int64_t>(rr[u]) * p.max_blocks_per_seq + blk);
                b[u] = __ldg(p.block_tables + blk);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (rr[u] > 0 && a[u] != b[u]) req[rr[u]].x = 1;
        }
        __syncthreads();                                 // uniform: prefix_blocks is a kernel parameter
    }

    // pass 1: total key pages of split requests (sets the automatic split size)
    unsigned long long mine = 0;
    for (int r = tid; r < p.num_seqs; r += nthr) {
        const int q = qsl[r + 1] - qsl[r];
        const int L = lens[r];
        if (q > 0 && q * G <= 16 && L >= q) {
            // a cascade request's prefix pages are not decode-kernel work
            const bool casc = cascade_eligible(p, qsl, lens, r, p.prefix_blocks > 0 && req[r].x != 0);
            mine += (unsigned long long)(div_up(L, kBlock) - (casc ? p.prefix_blocks : 0));
        }
    }
    mine = warp_sum_u64(mine);
    if ((tid & 31) == 0 && mine) atomicAdd(&total_pages, mine);
    __syncthreads();
    if (tid == 0) pages_per_split = auto_pages_per_split(total_pages, p.num_kv_heads, p.total_warps);
    __syncthreads();
    const int pps = pages_per_split;

    // pass 2: per request, its chunk count and partial rows; each thread owns
    // a contiguous range of requests so one block scan gives every base
    const int per_thr = div_up(max(p.num_seqs, 1), nthr);
    const int r_begin = min(p.num_seqs, tid * per_thr), r_end = min(p.num_seqs, r_begin + per_thr);
    // (a cascade request's splits are its suffix chunks plus the shared prefix)
    int my_chunks = 0, my_prows = 0, my_crows = 0, my_stoks = 0;
    unsigned my_casc = 0;                            // bit k: request r_begin + k takes the cascade path
    for (int r = r_begin; r < r_end; ++r) {
        const bool casc = cascade_eligible(p, qsl, lens, r, p.prefix_blocks > 0 && req[r].x != 0);
        if (casc && r - r_begin < 32) my_casc |= 1u << (r - r_begin);
        const ReqPlan rp = plan_request(p, qsl, lens, r, pps, casc && r - r_begin < 32);
        if (!rp.valid) {
            bad = 1;
            continue;
        }
        my_chunks += rp.n_chunks;
        const int nsplit = rp.n_chunks + (rp.first > 0 ? p.lay.prefix_parts : 0);
        if (rp.mode == 0 && nsplit > 1) {
            my_prows += rp.q * p.num_q_heads * nsplit;
            my_stoks += rp.q;
        }
        if (rp.first > 0) my_crows += rp.rows;
    }
    const int4 pre = block_scan4(my_chunks, my_prows, my_crows, my_stoks, warp_tot, &totals);
    if (staged) pdl_wait();       // the previous kernel on the stream may still read this workspace
    for (int i = tid; i < 2 * kStatsCtas; i += nthr) reinterpret_cast<int32_t *>(p.ws + kStatsOffset)[i] = 0;
    const int n_total = totals.x;
    // (split tokens too: with inconsistent query starts the requests' rows may
    // overlap and number more than the tokens)
    const bool fits = n_total <= p.lay.max_chunks + p.lay.max_ptiles && totals.y <= p.lay.max_prow &&
                      totals.z <= p.lay.max_crows && totals.w <= p.num_tokens;
    {
        int cb = pre.x, pbase = pre.y, crow = pre.z, sbase = pre.w;
        for (int r = r_begin; r < r_end; ++r) {
            const bool casc = (my_casc >> (r - r_begin)) & 1u;
            const ReqPlan rp = plan_request(p, qsl, lens, r, pps, casc);
            const int n = (rp.valid && fits) ? rp.n_chunks : 0;
            const int nsplit = rp.n_chunks + (rp.first > 0 ? p.lay.prefix_parts : 0);
            const bool split = rp.valid && fits && rp.mode == 0 && nsplit > 1;
            // a cascade request has splits = chunks + prefix_parts (>= 1), which
            // no other request has
            req[r] = make_int4(rp.valid && fits ? (split ? nsplit : 1) : 0, split ? pbase : 0, cb, n);
            if (staged) s_geom[r] = chunk_geometry(rp);
            if (rp.valid && fits && rp.first > 0) {
                const int q0 = qsl[r];
                for (int row = 0; row < rp.rows; ++row) crows[crow + row] = make_int4(q0 + row / G, r, row / G, row % G);
                crow += rp.rows;
            }
            cb += n;
            if (split) {
                // the request's tokens, whose rows the combine merges
                const int q0 = qsl[r];
                for (int i = 0; i < rp.q; ++i)
                    stoks[sbase + i] = make_int4(q0 + i, pbase + i * p.num_q_heads * nsplit, nsplit, 0);
                pbase += rp.q * p.num_q_heads * nsplit;
                sbase += rp.q;
            }
        }
    }
    __syncthreads();

    auto is_cascade = [&](const int4 &ri) { return p.lay.prefix_parts > 0 && ri.x == ri.w + p.lay.prefix_parts; };

    // pass 3: per chunk, its size bin (request found by binary search on the bases)
    auto owner = [&](int c) {
        int lo = 0, hi = p.num_seqs - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (req[mid].z <= c) lo = mid;
            else hi = mid - 1;
        }
        while (lo < p.num_seqs - 1 && req[lo].w == 0) ++lo;   // skip requests with no chunks
        return lo;
    };
    const int n_emit = fits ? n_total : 0;
    // (a staged batch keeps each request's chunk geometry in shared memory;
    // a larger one plans the request again)
    auto geometry = [&](int r, const int4 &ri) {
        return staged ? s_geom[r] : chunk_geometry(plan_request(p, qsl, lens, r, pps, is_cascade(ri)));
    };
    for (int c = tid; c < n_emit; c += nthr) {
        const int r = owner(c);
        const int4 ri = req[r];
        const int4 gm = geometry(r, ri);
        const int2 pg = chunk_pages(gm, G, c - ri.z);
        if (gm.x == 2) agg_inc(pbin_count, min(pg.y, kSizeBins - 1));
        else agg_inc(bin_count, min(pg.y - pg.x, kSizeBins - 1));
    }
    __syncthreads();
    if (tid < 64) {                                   // largest first; warp 0 decode chunks, warp 1 tiles
        const bool tiles = tid >= 32;
        const int acc = scan_bins_desc(tiles ? pbin_count : bin_count, tiles ? pbin_cursor : bin_cursor, tid & 31);
        if ((tid & 31) == 0) bin_total[tiles ? 1 : 0] = acc;
    }
    __syncthreads();
    if (tid == 0) {
        const bool ok = fits && bin_total[0] <= p.lay.max_chunks && bin_total[1] <= p.lay.max_ptiles;
        hdr->n_chunks = ok ? bin_total[0] : 0;
        hdr->n_ptiles = ok ? bin_total[1] : 0;
        if (!fits) bad = 1;
    }

    // pass 4: emit every chunk at its sorted position
    for (int c = tid; c < n_emit; c += nthr) {
        const int r = owner(c);
        const int4 ri = req[r];
        const bool casc = is_cascade(ri);
        const int4 gm = geometry(r, ri);
        const int k = c - ri.z;
        const int2 pg = chunk_pages(gm, G, k);
        if (gm.x == 2) {
            const int pos = agg_inc(pbin_cursor, min(pg.y, kSizeBins - 1));
            if (pos < p.lay.max_ptiles) ptiles[pos] = make_int4(r, k, pg.y, 0);
        } else {
            // chunk {request, split index (cascade: after the prefix ranges), pages}
            const int pos = agg_inc(bin_cursor, min(pg.y - pg.x, kSizeBins - 1));
            if (pos < p.lay.max_chunks) chunks[pos] = make_int4(r, k + (casc ? p.lay.prefix_parts : 0), pg.x, pg.y);
        }
    }
    if (staged)
        for (int r = tid; r < p.num_seqs; r += nthr) req_ws[r] = s_req[r];
    __syncthreads();
    if (tid == 0) {
        hdr->status = bad ? PKV_ERR_DEVICE_METADATA : PKV_OK;
        hdr->magic = kMagic;
        hdr->num_tokens = p.num_tokens;
        hdr->num_q_heads = p.num_q_heads;
        hdr->head_size = p.head_size;
        hdr->num_seqs = p.num_seqs;
        hdr->pages_per_split = pps;
        hdr->off_req = p.lay.off_req;
        hdr->off_stoks = p.lay.off_stoks;
        hdr->n_split_tokens = fits ? totals.w : 0;
        hdr->off_chunks = p.lay.off_chunks;
        hdr->off_ptiles = p.lay.off_ptiles;
        hdr->off_part_lse = p.lay.off_part_lse;
        hdr->off_part_o = p.lay.off_part_o;
        hdr->off_crows = p.lay.off_crows;
        hdr->n_crows = fits ? totals.z : 0;
        hdr->prefix_blocks = p.prefix_blocks;
        hdr->prefix_parts = p.lay.prefix_parts;
        hdr->next_ptile_item = 0;
        hdr->next_prefix_item = 0;
        hdr->max_chunks = p.lay.max_chunks;
        hdr->max_ptiles = p.lay.max_ptiles;
        hdr->max_crows = p.lay.max_crows;
        hdr->max_prow = p.lay.max_prow;
        hdr->prow_used = totals.y;
    }
}

// ---- 3. combine -------------------------------------------------------------------------

template <int HD>
__global__ void __launch_bounds__(256) combine_kernel(__nv_bfloat16 *out, const uint8_t *ws, int32_t num_tokens,
                                                      int32_t num_q_heads) {
    pdl_wait();       // every partial of the attention kernels is written
    const WsHeader *hdr = reinterpret_cast<const WsHeader *>(ws);
    // every header field this kernel uses, loaded at once (one round trip)
    const int magic = hdr->magic, h_tokens = hdr->num_tokens, h_heads = hdr->num_q_heads, h_hd = hdr->head_size;
    const int n_split = hdr->n_split_tokens;
    const int64_t off_stoks = hdr->off_stoks, off_lse = hdr->off_part_lse, off_o = hdr->off_part_o;
    if ((magic != kMagic) | (h_tokens != num_tokens) | (h_heads != num_q_heads) | (h_hd != HD)) {
        if (blockIdx.x == 0 && threadIdx.x == 0)
            set_status(reinterpret_cast<int32_t *>(const_cast<uint8_t *>(ws)), PKV_ERR_PROTOCOL);
        return;
    }
    const int4 *stoks = reinterpret_cast<const int4 *>(ws + off_stoks);
    const float *part_lse = reinterpret_cast<const float *>(ws + off_lse);
    const float *part_o = reinterpret_cast<const float *>(ws + off_o);
    const int lane = threadIdx.x & 31;
    // one warp per row (split token, q head), grid-strided over the rows
    const int64_t n_rows = static_cast<int64_t>(n_split) * num_q_heads;
    for (int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5); row < n_rows;
         row += static_cast<int64_t>(gridDim.x) * 8) {
        const int4 st = __ldg(stoks + row / num_q_heads);   // {token, partial row of q head 0, splits, 0}
        const int h = static_cast<int>(row % num_q_heads);
        merge_split_row<HD>(part_o, part_lse, st.y + static_cast<int64_t>(h) * st.z, st.z,
                            out + (static_cast<int64_t>(st.x) * num_q_heads + h) * HD, lane);
    }
}

static int paged_attn_impl(void *out, const void *query, int64_t query_token_stride, const void *kv_cache,
                           int64_t num_blocks, const int32_t *block_tables, int32_t max_blocks_per_seq,
                           const int32_t *seq_lens, const int32_t *query_start_loc, int32_t num_seqs,
                           int32_t num_tokens, int32_t max_query_len, int32_t max_seq_len, int32_t num_q_heads,
                           int32_t num_kv_heads, int32_t head_size, int32_t block_size, float scale,
                           int32_t num_splits, int32_t prefix_blocks, void *workspace, size_t workspace_bytes,
                           size_t *workspace_needed, void *stream, bool kv8 = false, float k_scale = 1.f,
                           float v_scale = 1.f) {
    // ---- host-side validation: nothing is enqueued on error ----
    if (num_seqs < 0 || num_tokens < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || max_query_len < 0 ||
        max_seq_len < 0 || max_blocks_per_seq < 0 || num_splits < 0 || prefix_blocks < 0)
        return PKV_ERR_SHAPE;
    if (prefix_blocks > max_blocks_per_seq) return PKV_ERR_SHAPE;
    if (block_size != kBlock || (head_size != 64 && head_size != 128)) return PKV_ERR_UNSUPPORTED;
    if (num_q_heads % num_kv_heads) return PKV_ERR_SHAPE;
    if (num_tokens > 0 && num_seqs == 0) return PKV_ERR_SHAPE;
    if (max_query_len > max_seq_len) return PKV_ERR_SHAPE;
    if (static_cast<int64_t>(max_blocks_per_seq) * kBlock < max_seq_len) return PKV_ERR_SHAPE;
    if (num_blocks < 1 || num_blocks > INT32_MAX) return PKV_ERR_SHAPE;
    // the tile kernels address a page of one kv head as block id x kv heads + head in 32 bits
    if (num_blocks * static_cast<int64_t>(num_kv_heads) > INT32_MAX) return PKV_ERR_SHAPE;
    if (!(scale == scale) || scale > 3.0e38f || scale < -3.0e38f) return PKV_ERR_SHAPE;
    if (!(k_scale > 0.f) || !(v_scale > 0.f) || k_scale > 3.0e38f || v_scale > 3.0e38f) return PKV_ERR_SHAPE;

    // long chunks and the shared-prefix pass go to the tensor-core tile kernel
    // (which widens an E4M3 cache's pages to f16 itself)
    const bool prefill_ok = prefill_supported(num_q_heads, num_kv_heads, head_size);
    if (!prefill_ok) prefix_blocks = 0;
    const WsLayout lay = ws_layout(num_seqs, num_tokens, max_query_len, max_seq_len, num_q_heads, num_kv_heads,
                                   head_size, prefix_blocks);
    if (workspace_needed) *workspace_needed = static_cast<size_t>(lay.total);
    if (num_seqs == 0) return PKV_OK;
    if (!out || !query || !kv_cache || !block_tables || !seq_lens || !query_start_loc) return PKV_ERR_NULL;
    if (!workspace || workspace_bytes < static_cast<size_t>(lay.total)) return PKV_ERR_WORKSPACE;
    if (query_token_stride < static_cast<int64_t>(num_q_heads) * head_size) return PKV_ERR_SHAPE;
    if (query_token_stride % 8) return PKV_ERR_ALIGNMENT;
    if ((reinterpret_cast<uintptr_t>(out) | reinterpret_cast<uintptr_t>(query) |
         reinterpret_cast<uintptr_t>(kv_cache)) & 15u)
        return PKV_ERR_ALIGNMENT;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return PKV_ERR_ALIGNMENT;
    if ((reinterpret_cast<uintptr_t>(block_tables) | reinterpret_cast<uintptr_t>(seq_lens) |
         reinterpret_cast<uintptr_t>(query_start_loc)) & 3u)
        return PKV_ERR_ALIGNMENT;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return PKV_ERR_CUDA;

    CUtensorMap map;
    int rc = make_decode_map(&map, kv_cache, num_blocks, num_kv_heads, head_size, kv8);
    if (rc) return rc;

    const int nw = kDecodeWarps;
    const int per_sm = decode_ctas_per_sm(head_size, kv8);
    const int64_t resident = static_cast<int64_t>(sms) * per_sm;
    const int64_t max_items = lay.max_chunks * num_kv_heads;
    int64_t grid = std::max<int64_t>(1, std::min(resident, (max_items + nw - 1) / nw));
    const int G = num_q_heads / num_kv_heads;
    const bool may_prefill = prefill_ok && static_cast<int64_t>(max_query_len) * G > kDecodeTileMaxRows;
    // a small decode-only batch is planned by the decode kernel itself: its
    // last CTA writes the header, the others (still one wave) take the chunks
    const int64_t sp_ctas = std::max<int64_t>(1, std::min(resident - 1, (max_items + nw - 1) / nw));
    const bool self_plan = !may_prefill && resident >= 2 &&
                           decode_self_plan_ok(num_seqs, max_query_len, max_seq_len, G, num_kv_heads, num_splits,
                                               prefix_blocks, sp_ctas * nw);
    if (self_plan) grid = sp_ctas + 1;
    const int64_t chunk_warps = (self_plan ? sp_ctas : grid) * nw;

    PlanParams pp;
    pp.ws = static_cast<uint8_t *>(workspace);
    pp.seq_lens = seq_lens;
    pp.qsl = query_start_loc;
    pp.num_seqs = num_seqs;
    pp.num_tokens = num_tokens;
    pp.num_q_heads = num_q_heads;
    pp.num_kv_heads = num_kv_heads;
    pp.head_size = head_size;
    pp.max_blocks_per_seq = max_blocks_per_seq;
    pp.max_query_len = max_query_len;
    pp.max_seq_len = max_seq_len;
    pp.num_splits = num_splits;
    pp.total_warps = static_cast<int32_t>(chunk_warps);
    pp.prefill_ok = prefill_ok ? 1 : 0;
    pp.prefix_blocks = prefix_blocks;
    pp.block_tables = block_tables;
    pp.lay = lay;
    // the plan's phases are chains of barriers and short loads: a batch of at
    // most 256 requests without a shared prefix plans faster on 256 threads
    // (the prefix comparison of every table with request 0's wants all of them)
    const int plan_threads = (prefix_blocks == 0 && num_seqs <= 256) ? 256 : kPlanThreads;
    if (!self_plan && launch_pdl(plan_kernel, dim3(1), dim3(plan_threads), 0, st, pp) != cudaSuccess)
        return PKV_ERR_CUDA;

    AttnParams ap;
    ap.out = static_cast<__nv_bfloat16 *>(out);
    ap.query = static_cast<const __nv_bfloat16 *>(query);
    ap.q_stride = query_token_stride;
    ap.block_tables = block_tables;
    ap.max_blocks_per_seq = max_blocks_per_seq;
    ap.seq_lens = seq_lens;
    ap.qsl = query_start_loc;
    ap.num_q_heads = num_q_heads;
    ap.num_kv_heads = num_kv_heads;
    ap.G = num_q_heads / num_kv_heads;
    ap.num_blocks = num_blocks;
    ap.scale_log2 = scale * 1.4426950408889634f;
    ap.k_scale = k_scale;
    ap.v_scale = v_scale;
    ap.ws = static_cast<uint8_t *>(workspace);
    ap.self_plan = self_plan ? 1 : 0;
    ap.num_seqs = num_seqs;
    ap.num_tokens = num_tokens;
    ap.head_size = head_size;
    ap.max_query_len = max_query_len;
    ap.max_seq_len = max_seq_len;
    ap.total_warps = static_cast<int32_t>(chunk_warps);
    ap.lay = lay;
    rc = launch_decode_path(map, ap, head_size, kv8, static_cast<int>(grid), dev, st);
    if (rc || (!may_prefill && prefix_blocks == 0)) return rc;
    PrefillParams fp;
    fp.out = ap.out;
    fp.block_tables = block_tables;
    fp.max_blocks_per_seq = max_blocks_per_seq;
    fp.seq_lens = seq_lens;
    fp.qsl = query_start_loc;
    fp.num_q_heads = num_q_heads;
    fp.num_kv_heads = num_kv_heads;
    fp.G = G;
    fp.num_blocks = num_blocks;
    fp.scale_log2 = ap.scale_log2;
    fp.lo_tiles = 0;
    fp.k_scale = k_scale;
    fp.v_scale = v_scale;
    fp.ws = ap.ws;
    // persistent kernels: one CTA per SM at most, and no more than their items
    const int64_t max_ctas = std::min(sms, kStatsCtas);
    if (prefix_blocks > 0) {
        const int64_t items = (lay.max_crows + kPrefillRows - 1) / kPrefillRows * num_kv_heads * lay.prefix_parts;
        rc = kv8 ? launch_prefix_e4m3(fp, query, query_token_stride, kv_cache, num_blocks, head_size,
                                      std::min(max_ctas, items), dev, st)
                 : launch_prefill_sk(fp, query, query_token_stride, num_tokens, kv_cache, num_blocks, head_size,
                                     true, std::min(max_ctas, items), dev, st);
        if (rc) return rc;
    }
    if (!may_prefill) return PKV_OK;
    const int64_t items = lay.max_ptiles * num_kv_heads;
    return kv8 ? launch_prefill_e4m3(fp, query, query_token_stride, kv_cache, num_blocks, head_size,
                                     std::min(max_ctas, items), dev, st)
               : launch_prefill_sk(fp, query, query_token_stride, num_tokens, kv_cache, num_blocks, head_size,
                                   false, std::min(max_ctas, items), dev, st);
}

}  // namespace pkv

extern "C" int pkv_paged_attn(void *out, const void *query, int64_t query_token_stride, const void *kv_cache,
                              int64_t num_blocks, const int32_t *block_tables, int32_t max_blocks_per_seq,
                              const int32_t *seq_lens, const int32_t *query_start_loc, int32_t num_seqs,
                              int32_t num_tokens, int32_t max_query_len, int32_t max_seq_len, int32_t num_q_heads,
                              int32_t num_kv_heads, int32_t head_size, int32_t block_size, float scale,
                              int32_t num_splits, void *workspace, size_t workspace_bytes, size_t *workspace_needed,
                              void *stream) {
    return pkv::paged_attn_impl(out, query, query_token_stride, kv_cache, num_blocks, block_tables,
                                max_blocks_per_seq, seq_lens, query_start_loc, num_seqs, num_tokens, max_query_len,
                                max_seq_len, num_q_heads, num_kv_heads, head_size, block_size, scale, num_splits, 0,
                                workspace, workspace_bytes, workspace_needed, stream);
}

extern "C" int pkv_paged_attn_shared_prefix(void *out, const void *query, int64_t query_token_stride,
                                            const void *kv_cache, int64_t num_blocks, const int32_t *block_tables,
                                            int32_t max_blocks_per_seq, const int32_t *seq_lens,
                                            const int32_t *query_start_loc, int32_t num_seqs, int32_t num_tokens,
                                            int32_t max_query_len, int32_t max_seq_len, int32_t num_q_heads,
                                            int32_t num_kv_heads, int32_t head_size, int32_t block_size,
                                            float scale, int32_t num_splits, int32_t shared_prefix_blocks,
                                            void *workspace, size_t workspace_bytes, size_t *workspace_needed,
                                            void *stream) {
    return pkv::paged_attn_impl(out, query, query_token_stride, kv_cache, num_blocks, block_tables,
                                max_blocks_per_seq, seq_lens, query_start_loc, num_seqs, num_tokens, max_query_len,
                                max_seq_len, num_q_heads, num_kv_heads, head_size, block_size, scale, num_splits,
                                shared_prefix_blocks, workspace, workspace_bytes, workspace_needed, stream);
}

extern "C" int pkv_paged_attn_shared_prefix_fp8(void *out, const void *query, int64_t query_token_stride,
                                                const void *kv_cache, int64_t num_blocks,
                                                const int32_t *block_tables, int32_t max_blocks_per_seq,
                                                const int32_t *seq_lens, const int32_t *query_start_loc,
                                                int32_t num_seqs, int32_t num_tokens, int32_t max_query_len,
                                                int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads,
                                                int32_t head_size, int32_t block_size, float scale, float k_scale,
                                                float v_scale, int32_t num_splits, int32_t shared_prefix_blocks,
                                                void *workspace, size_t workspace_bytes, size_t *workspace_needed,
                                                void *stream) {
    return pkv::paged_attn_impl(out, query, query_token_stride, kv_cache, num_blocks, block_tables,
                                max_blocks_per_seq, seq_lens, query_start_loc, num_seqs, num_tokens, max_query_len,
                                max_seq_len, num_q_heads, num_kv_heads, head_size, block_size, scale, num_splits,
                                shared_prefix_blocks, workspace, workspace_bytes, workspace_needed, stream, true,
                                k_scale, v_scale);
}

extern "C" int pkv_paged_attn_combine(void *out, const void *workspace, size_t workspace_bytes, int32_t num_tokens,
                                      int32_t num_q_heads, int32_t head_size, void *stream) {
    using namespace pkv;
    if (num_tokens < 0 || num_q_heads <= 0) return PKV_ERR_SHAPE;
    if (head_size != 64 && head_size != 128) return PKV_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PKV_OK;
    if (!out || !workspace) return PKV_ERR_NULL;
    if (workspace_bytes < 256) return PKV_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(out) & 15u) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return PKV_ERR_ALIGNMENT;
    // the rows to merge are known on the device only: a grid of at most 8
    // CTAs per SM strides over them
    const int64_t rows = static_cast<int64_t>(num_tokens) * num_q_heads;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return PKV_ERR_CUDA;
    const int64_t grid = std::min<int64_t>((rows + 7) / 8, static_cast<int64_t>(sms) * 8);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(out);
    const uint8_t *w = static_cast<const uint8_t *>(workspace);
    const cudaError_t e =
        head_size == 64 ? launch_pdl(combine_kernel<64>, dim3(static_cast<unsigned>(grid)), dim3(256), 0, st, o, w,
                                     num_tokens, num_q_heads)
                        : launch_pdl(combine_kernel<128>, dim3(static_cast<unsigned>(grid)), dim3(256), 0, st, o, w,
                                     num_tokens, num_q_heads);
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

extern "C" int pkv_paged_attn_fp8(void *out, const void *query, int64_t query_token_stride, const void *kv_cache,
                                  int64_t num_blocks, const int32_t *block_tables, int32_t max_blocks_per_seq,
                                  const int32_t *seq_lens, const int32_t *query_start_loc, int32_t num_seqs,
                                  int32_t num_tokens, int32_t max_query_len, int32_t max_seq_len,
                                  int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size, int32_t block_size,
                                  float scale, float k_scale, float v_scale, int32_t num_splits, void *workspace,
                                  size_t workspace_bytes, size_t *workspace_needed, void *stream) {
    return pkv::paged_attn_impl(out, query, query_token_stride, kv_cache, num_blocks, block_tables,
                                max_blocks_per_seq, seq_lens, query_start_loc, num_seqs, num_tokens, max_query_len,
                                max_seq_len, num_q_heads, num_kv_heads, head_size, block_size, scale, num_splits, 0,
                                workspace, workspace_bytes, workspace_needed, stream, true, k_scale, v_scale);
}
