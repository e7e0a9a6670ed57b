// Decode kernel of the paged-attention path: split-K and 16-row tiles over
// a block-table-indexed KV cache (see paged_attn.cu for the plan that lists
// its chunks and the combine that merges split rows).
//
// What is computed ("continuous batching and PagedAttention" tutorial,
// section 3.6 "PagedAttention kernel"; "vLLM source reading", sections 2.3
// and 5.1): every query row loops over its request's logical blocks, looks
// up the physical block in the block table, loads that block's K and V and
// folds softmax(scale * q.K^T) V into a running (max, sum, accumulator) state.
//
// Persistent CTAs of NW warps.  Each warp takes chunks (x kv heads) in a
// fixed order and streams the chunk's 16-token pages through its own ring of
// DEPTH shared-memory stages.  A page of one kv head (K then V,
// 2*16*head_size bf16, contiguous in the cache) arrives by TMA tensor loads
// with 128-byte swizzle, so ldmatrix reads are free of bank conflicts.
// S = Q K^T and O += P V run on bf16 mma.sync tiles: rows are the tile's
// (query token, q head of the group) pairs, so every q head of a GQA group is
// served by one read of each KV page.
#include <mutex>

#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "attn_internal.cuh"

namespace pkv {

// Shared-memory address of (row, 16-byte chunk) inside one TMA box of
// 32 rows x 128 bytes written with the 128-byte swizzle: chunk c of row R is
// stored at chunk position c ^ (R & 7).
__device__ __forceinline__ uint32_t swz(uint32_t box_base, int row, int chunk) {
    return box_base + row * 128 + ((chunk ^ (row & 7)) << 4);
}

// KV8 = false: bf16 cache; ring stages hold pages in the 16-bit layout the
// MMA loads read (128-byte swizzled 64-column boxes of 32 rows, K rows 0..15
// and V rows 16..31).  KV8 = true: E4M3 cache; ring stages hold the raw 8-bit
// page, whose V rows the warp widens to f16 into a private staging area
// before the MMAs (K is read from the raw page): the V halves of the 16-bit
// boxes only, kVBoxBytes apart.
template <int HD, int NW, int DEPTH, bool KV8>
struct DecodeCfg {
    static constexpr int kBoxes = HD / 64;                 // 64-element boxes per row
    static constexpr int kBoxBytes = 2 * kBlock * 128;     // K and V rows of one box: 4 KiB
    static constexpr int kPageBytes = kBoxes * kBoxBytes;  // one 16-bit page of one kv head
    static constexpr int kStageBytes = KV8 ? 2 * kBlock * HD : kPageBytes;
    static constexpr int kVBoxBytes = kBlock * 128;        // V rows of one box: 2 KiB
    static constexpr int kWarpBytes = DEPTH * kStageBytes + (KV8 ? kBoxes * kVBoxBytes : 0);
    static constexpr int kSmem = NW * kWarpBytes + NW * DEPTH * 8 + 1024;
};

// MMA element type of the decode kernel: bf16 for a bf16 cache; f16 for an
// E4M3 cache (E4M3 widens to f16 exactly in one instruction per pair).
template <bool F16> struct DecodeMath;
template <> struct DecodeMath<false> {
    static __device__ __forceinline__ void mma(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
        mma_bf16_16816(d, a, b0, b1);
    }
    static __device__ __forceinline__ void split(float x, float y, uint32_t &big, uint32_t &rest) {
        split_bf16x2(x, y, big, rest);
    }
};
template <> struct DecodeMath<true> {
    static __device__ __forceinline__ void mma(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
            "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    }
    // (x, y) -> one f16x2 pair
    static __device__ __forceinline__ void round(float x, float y, uint32_t &h) {
        const __half2 b = __floats2half2_rn(x, y);
        h = *reinterpret_cast<const uint32_t *>(&b);
    }
};

// Four E4M3 values (one 32-bit word, element 0 in the low byte) -> two f16x2
// words (elements 0,1 and 2,3; the lower element in the low half).
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t w, uint32_t &h01, uint32_t &h23) {
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "mov.b32 {lo, hi}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, lo;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, hi;\n\t}"
        : "=r"(h01), "=r"(h23)
        : "r"(w));
}

// Widen the V rows of one raw E4M3 page (linear [2][16][HD] bytes) into the
// 16-bit staging area: f16 values, 128-byte swizzled 64-column boxes of the
// V rows only (rows 16..31 of the 16-bit page's boxes, 2 KiB per box; `dst`
// is the address row 0 of box 0 would have, 2 KiB before the area).  Every lane
// converts 16-byte pieces, loading all of its pieces before converting any.
// At HD = 128 a quarter-warp takes two rows, half a row each, in alternating
// halves, so that both its 8-bit reads and its 16-bit stores hit eight
// distinct bank groups.
template <int HD>
__device__ __forceinline__ void widen_e4m3_values(uint32_t src, uint32_t dst, int lane) {
    constexpr int kChunks = 2 * kBlock * HD / 16;          // pieces of the page (K and V)
    constexpr int kFirst = kChunks / 2;                    // the V rows' pieces
    constexpr int kPerLane = (kChunks - kFirst) / 32;      // 2 or 4
    constexpr int kBoxBytes = kBlock * 128;                // V rows of one box
    static_assert(kChunks % 64 == 0, "whole V pieces per lane");
    auto piece = [&](int q, int &row, int &col) {
        if constexpr (HD == 128) {
            const int ph = q >> 3, k = q & 7, sub = k >> 2;
            row = 2 * (ph >> 1) + sub;
            col = 16 * (4 * (sub ^ (ph & 1)) + (k & 3));
        } else {
            row = (q * 16) / HD;
            col = (q * 16) % HD;
        }
    };
    uint32_t w[kPerLane][4];
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
        int row, col;
        piece(kFirst + lane + 32 * i, row, col);
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(w[i][0]), "=r"(w[i][1]), "=r"(w[i][2]), "=r"(w[i][3])
                     : "r"(src + row * HD + col));
    }
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
        int row, col;
        piece(kFirst + lane + 32 * i, row, col);
        uint32_t h[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) e4m3x4_to_f16x4(w[i][e], h[2 * e], h[2 * e + 1]);
        const uint32_t box = dst + (col / 64) * kBoxBytes;
        const int ch = (col % 64) / 8;
        const uint32_t a0 = box + row * 128 + ((ch ^ (row & 7)) << 4);
        const uint32_t a1 = box + row * 128 + (((ch + 1) ^ (row & 7)) << 4);
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a0), "r"(h[0]), "r"(h[1]), "r"(h[2]),
                     "r"(h[3])
                     : "memory");
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a1), "r"(h[4]), "r"(h[5]), "r"(h[6]),
                     "r"(h[7])
                     : "memory");
    }
}

// Decode tiling per head size and cache type: warps per CTA, ring stages per
// warp, resident CTAs per SM (the launch bound, so the registers fit).  At
// d = 64 a bf16 page is 4 KiB: four CTAs of three-stage rings (16 warps of
// independent page chains, 128 registers) keep more chunks in flight than
// two CTAs of six stages.
template <int HD, bool KV8 = false> struct DecodeTiling;
template <> struct DecodeTiling<64> { static constexpr int NW = 4, DEPTH = 3, CTAS_PER_SM = 4; };
template <> struct DecodeTiling<128> { static constexpr int NW = 4, DEPTH = 3, CTAS_PER_SM = 2; };
// E4M3 pages are half the bytes: more stages in flight, plus one staging page
// per warp (at d = 64, three CTAs of six-stage rings at 153 registers)
template <> struct DecodeTiling<64, true> { static constexpr int NW = 4, DEPTH = 6, CTAS_PER_SM = 3; };
template <> struct DecodeTiling<128, true> { static constexpr int NW = 4, DEPTH = 4, CTAS_PER_SM = 2; };

static_assert(DecodeTiling<64>::NW == kDecodeWarps && DecodeTiling<128>::NW == kDecodeWarps &&
                  DecodeTiling<64, true>::NW == kDecodeWarps && DecodeTiling<128, true>::NW == kDecodeWarps,
              "every decode tiling has kDecodeWarps warps per CTA");

// ---- the decode kernel's own plan ---------------------------------------------
//
// For a call that decode_self_plan_ok admits (every request a split row, a
// batch small enough that every warp takes at most two chunks) no plan kernel
// runs.  Every CTA plans the whole call in shared memory (the space its rings
// take later) with the plan kernel's decisions (request_valid, the automatic
// split size, split_geometry), lists chunks in request order, and takes its
// warps' chunks from that list.  The grid's last CTA takes no chunks: it
// writes what the combine and the caller read (header, status, split tokens),
// beside the other CTAs' work rather than before it.

// One chunk of a warp: request, split, page range, the request's splits and
// first partial row.
struct SelfChunk {
    int r, k, pb, npages, n_split, pbase;
};

struct SelfPlanShared {
    unsigned long long total_pages;
    int bad, fits;
    int4 warp_tot[kDecodeWarps];
    int4 tot;
};

// The plan of the call in `scr` (8 * num_seqs + 1 ints) and the chunks of
// this warp (round 0 and round 1 of the snake order); returns the number of
// items (chunks x kv heads), 0 when the metadata does not fit the workspace.
template <int NW>
__device__ int decode_self_plan(const AttnParams &p, int *scr, SelfPlanShared &sh, SelfChunk (&mine)[2]) {
    const int S = p.num_seqs, tid = threadIdx.x, nthr = NW * 32;
    const int lane = tid & 31, warp = tid >> 5;
    int *s_qsl = scr, *s_len = scr + S + 1, *s_cb = s_len + S, *s_nc = s_cb + S, *s_ps = s_nc + S;
    int *s_pg = s_ps + S, *s_pb = s_pg + S, *s_sb = s_pb + S;
    for (int r = tid; r <= S; r += nthr) s_qsl[r] = __ldg(p.qsl + r);
    for (int r = tid; r < S; r += nthr) s_len[r] = __ldg(p.seq_lens + r);
    if (tid == 0) {
        sh.total_pages = 0;
        sh.bad = 0;
    }
    __syncthreads();
    // total key pages (sets the automatic split size), and the metadata check
    unsigned long long pages = 0;
    int bad = tid == 0 && s_qsl[0] != 0;
    for (int r = tid; r < S; r += nthr) {
        const int q0 = s_qsl[r], q1 = s_qsl[r + 1], L = s_len[r];
        if (!request_valid(q0, q1, L, p.num_tokens, p.max_seq_len, p.max_query_len, p.max_blocks_per_seq)) bad = 1;
        else if (q1 > q0) pages += static_cast<unsigned long long>(div_up(L, kBlock));
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) pages += __shfl_xor_sync(0xffffffffu, pages, o);
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
        if (pages) atomicAdd(&sh.total_pages, pages);
        if (bad) sh.bad = 1;
    }
    __syncthreads();
    const int pps = auto_pages_per_split(sh.total_pages, p.num_kv_heads, p.total_warps);
    // per request: chunks, pages per split, partial rows and split tokens; each
    // thread a contiguous range of requests, one block scan for the bases
    const int per_thr = div_up(S, nthr);
    const int r_begin = min(S, tid * per_thr), r_end = min(S, r_begin + per_thr);
    int4 cnt = make_int4(0, 0, 0, 0);
    for (int r = r_begin; r < r_end; ++r) {
        const int q0 = s_qsl[r], q1 = s_qsl[r + 1], L = s_len[r];
        const int q = q1 - q0;
        int n = 0, ps = 0, span = 0;
        if (q > 0 && request_valid(q0, q1, L, p.num_tokens, p.max_seq_len, p.max_query_len, p.max_blocks_per_seq)) {
            span = div_up(L, kBlock);
            const int2 sg = split_geometry(span, pps, 0, kMaxSplits);
            ps = sg.x;
            n = sg.y;
        }
        s_nc[r] = n;
        s_ps[r] = ps;
        s_pg[r] = span;
        cnt.x += n;
        if (n > 1) {
            cnt.y += q * p.num_q_heads * n;
            cnt.z += q;
        }
    }
    int4 inc = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int a = __shfl_up_sync(0xffffffffu, inc.x, o), b = __shfl_up_sync(0xffffffffu, inc.y, o);
        const int c = __shfl_up_sync(0xffffffffu, inc.z, o);
        if (lane >= o) {
            inc.x += a;
            inc.y += b;
            inc.z += c;
        }
    }
    if (lane == 31) sh.warp_tot[warp] = inc;
    __syncthreads();
    if (tid == 0) {
        int4 acc = make_int4(0, 0, 0, 0);
        for (int w = 0; w < NW; ++w) {
            const int4 t = sh.warp_tot[w];
            sh.warp_tot[w] = acc;
            acc.x += t.x;
            acc.y += t.y;
            acc.z += t.z;
        }
        sh.tot = acc;
        sh.fits = acc.x <= p.lay.max_chunks && acc.y <= p.lay.max_prow && acc.z <= p.num_tokens;
        if (!sh.fits) sh.bad = 1;
    }
    __syncthreads();
    {
        const int4 wb = sh.warp_tot[warp];
        int cb = wb.x + inc.x - cnt.x, pb = wb.y + inc.y - cnt.y, sb = wb.z + inc.z - cnt.z;
        for (int r = r_begin; r < r_end; ++r) {
            const int n = s_nc[r];
            s_cb[r] = cb;
            s_pb[r] = pb;
            s_sb[r] = sb;
            cb += n;
            if (n > 1) {
                const int q = s_qsl[r + 1] - s_qsl[r];
                pb += q * p.num_q_heads * n;
                sb += q;
            }
        }
    }
    __syncthreads();
    const int n_items = sh.fits ? sh.tot.x * p.num_kv_heads : 0;
    // this warp's chunks: items wid and 2 W - 1 - wid (the snake order of the
    // loop), W the warps of every CTA but the last
    const int W = (gridDim.x - 1) * NW, wid = blockIdx.x * NW + warp;
#pragma unroll
    for (int round = 0; round < 2; ++round) {
        const int item = round ? 2 * W - 1 - wid : wid;
        SelfChunk c{-1, 0, 0, 0, 1, 0};
        if (wid < W && item < n_items) {
            const int ch = item / p.num_kv_heads;
            // the request of chunk ch: the last with chunk base <= ch, past any
            // request without chunks
            int lo = 0, hi = S - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (s_cb[mid] <= ch) lo = mid;
                else hi = mid - 1;
            }
            while (lo < S - 1 && s_nc[lo] == 0) ++lo;
            c.r = lo;
            c.k = ch - s_cb[lo];
            c.pb = c.k * s_ps[lo];
            c.npages = min(s_pg[lo], c.pb + s_ps[lo]) - c.pb;
            c.n_split = s_nc[lo] > 1 ? s_nc[lo] : 1;
            c.pbase = s_nc[lo] > 1 ? s_pb[lo] : 0;
        }
        mine[round] = c;
    }
    return n_items;
}

// The same plan made by one warp alone, in registers, for a batch of at most
// 32 x kWarpPlanPer requests: lane l holds requests [l per, (l + 1) per), the
// page total and the bases come from warp shuffles, and the owner of each of
// the warp's chunks is found by a ballot over the lanes' chunk ranges.  No
// block barrier and no shared memory: a chunk CTA's warps go from the
// metadata read to their first page loads on their own.  Decisions and
// bases are those of decode_self_plan (the grid's last CTA still makes that
// one, for the header and the split tokens).
constexpr int kWarpPlanPer = 2;

__device__ int decode_warp_plan(const AttnParams &p, SelfChunk (&mine)[2], int W, int wid) {
    const int S = p.num_seqs, lane = threadIdx.x & 31;
    const int per = div_up(S, 32);
    const int r0 = min(S, lane * per), r1 = min(S, r0 + per);
    int q0a[kWarpPlanPer], qa[kWarpPlanPer], La[kWarpPlanPer];
#pragma unroll
    for (int i = 0; i < kWarpPlanPer; ++i) {
        const int r = r0 + i;
        const bool in = i < per && r < r1;
        q0a[i] = in ? __ldg(p.qsl + r) : 0;
        qa[i] = in ? __ldg(p.qsl + r + 1) : 0;       // q1 for now
        La[i] = in ? __ldg(p.seq_lens + r) : 0;
    }
    // total key pages of the valid requests (the automatic split size)
    unsigned long long pages = 0;
    bool valid[kWarpPlanPer];
#pragma unroll
    for (int i = 0; i < kWarpPlanPer; ++i) {
        const bool in = i < per && r0 + i < r1;
        valid[i] = in && request_valid(q0a[i], qa[i], La[i], p.num_tokens, p.max_seq_len, p.max_query_len,
                                       p.max_blocks_per_seq);
        qa[i] -= q0a[i];                                 // query tokens
        if (valid[i] && qa[i] > 0) pages += static_cast<unsigned long long>(div_up(La[i], kBlock));
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) pages += __shfl_xor_sync(0xffffffffu, pages, o);
    const int pps = auto_pages_per_split(pages, p.num_kv_heads, p.total_warps);
    // per request: chunks, pages per split, page span; per lane: chunks,
    // partial rows, split tokens
    int na[kWarpPlanPer], psa[kWarpPlanPer], spa[kWarpPlanPer];
    int4 cnt = make_int4(0, 0, 0, 0);
#pragma unroll
    for (int i = 0; i < kWarpPlanPer; ++i) {
        int n = 0, ps = 0, span = 0;
        if (valid[i] && qa[i] > 0) {
            span = div_up(La[i], kBlock);
            const int2 sg = split_geometry(span, pps, 0, kMaxSplits);
            ps = sg.x;
            n = sg.y;
        }
        na[i] = n;
        psa[i] = ps;
        spa[i] = span;
        cnt.x += n;
        if (n > 1) {
            cnt.y += qa[i] * p.num_q_heads * n;
            cnt.z += qa[i];
        }
    }
    int4 inc = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int a = __shfl_up_sync(0xffffffffu, inc.x, o), b = __shfl_up_sync(0xffffffffu, inc.y, o);
        const int c = __shfl_up_sync(0xffffffffu, inc.z, o);
        if (lane >= o) {
            inc.x += a;
            inc.y += b;
            inc.z += c;
        }
    }
    const int tot_x = __shfl_sync(0xffffffffu, inc.x, 31), tot_y = __shfl_sync(0xffffffffu, inc.y, 31);
    const int tot_z = __shfl_sync(0xffffffffu, inc.z, 31);
    const bool fits = tot_x <= p.lay.max_chunks && tot_y <= p.lay.max_prow && tot_z <= p.num_tokens;
    const int n_items = fits ? tot_x * p.num_kv_heads : 0;
    const int cb0 = inc.x - cnt.x, pb0 = inc.y - cnt.y;      // this lane's first chunk and partial row
#pragma unroll
    for (int round = 0; round < 2; ++round) {
        const int item = round ? 2 * W - 1 - wid : wid;
        SelfChunk c{-1, 0, 0, 0, 1, 0};
        if (wid < W && item < n_items) {                     // uniform over the warp
            const int ch = item / p.num_kv_heads;
            const unsigned owners = __ballot_sync(0xffffffffu, cb0 <= ch && ch < cb0 + cnt.x);
            const int owner = __ffs(owners) - 1;
            int cb = cb0, pb = pb0;
            bool done = false;
#pragma unroll
            for (int i = 0; i < kWarpPlanPer; ++i) {
                if (!done && ch < cb + na[i]) {
                    done = true;
                    c.r = r0 + i;
                    c.k = ch - cb;
                    c.pb = c.k * psa[i];
                    c.npages = min(spa[i], c.pb + psa[i]) - c.pb;
                    c.n_split = na[i] > 1 ? na[i] : 1;
                    c.pbase = na[i] > 1 ? pb : 0;
                }
                cb += na[i];
                if (na[i] > 1) pb += qa[i] * p.num_q_heads * na[i];
            }
            c.r = __shfl_sync(0xffffffffu, c.r, owner);
            c.k = __shfl_sync(0xffffffffu, c.k, owner);
            c.pb = __shfl_sync(0xffffffffu, c.pb, owner);
            c.npages = __shfl_sync(0xffffffffu, c.npages, owner);
            c.n_split = __shfl_sync(0xffffffffu, c.n_split, owner);
            c.pbase = __shfl_sync(0xffffffffu, c.pbase, owner);
        }
        mine[round] = c;
    }
    return n_items;
}

// The last CTA of a self-planned call: the header, status and split tokens
// the plan kernel would have written (after every earlier kernel on the
// stream is complete), then the header's epoch is bumped.  (The request table
// is the plan kernel's record for its own decode launches; a self-planned
// call does not read it.)
template <int NW>
__device__ void decode_self_plan_publish(const AttnParams &p, const int *scr, const SelfPlanShared &sh) {
    const int S = p.num_seqs, tid = threadIdx.x, nthr = NW * 32;
    const int *s_qsl = scr, *s_len = scr + S + 1, *s_cb = s_len + S, *s_nc = s_cb + S;
    const int *s_pb = s_nc + 2 * S + S, *s_sb = s_pb + S;
    WsHeader *hdr = reinterpret_cast<WsHeader *>(p.ws);
    int4 *stoks = reinterpret_cast<int4 *>(p.ws + p.lay.off_stoks);
    const bool fits = sh.fits != 0;
    for (int i = tid; i < 2 * kStatsCtas; i += nthr) reinterpret_cast<int32_t *>(p.ws + kStatsOffset)[i] = 0;
    (void)s_len;
    (void)s_cb;
    for (int r = tid; r < S; r += nthr) {
        const int n = fits ? s_nc[r] : 0;
        const int q0 = s_qsl[r];
        const int q = s_qsl[r + 1] - q0;
        if (n > 1)
            for (int i = 0; i < q; ++i)
                stoks[s_sb[r] + i] = make_int4(q0 + i, s_pb[r] + i * p.num_q_heads * n, n, 0);
    }
    if (tid == 0) {
        hdr->status = sh.bad ? PKV_ERR_DEVICE_METADATA : PKV_OK;
        hdr->magic = kMagic;
        hdr->n_chunks = fits ? sh.tot.x : 0;
        hdr->num_tokens = p.num_tokens;
        hdr->num_q_heads = p.num_q_heads;
        hdr->head_size = p.head_size;
        hdr->num_seqs = S;
        hdr->pages_per_split = auto_pages_per_split(sh.total_pages, p.num_kv_heads, p.total_warps);
        hdr->n_ptiles = 0;
        hdr->n_crows = 0;
        hdr->prefix_blocks = 0;
        hdr->prefix_parts = 0;
        hdr->next_ptile_item = 0;
        hdr->next_prefix_item = 0;
        hdr->n_split_tokens = fits ? sh.tot.z : 0;
        hdr->off_req = p.lay.off_req;
        hdr->off_stoks = p.lay.off_stoks;
        hdr->off_chunks = p.lay.off_chunks;
        hdr->off_ptiles = p.lay.off_ptiles;
        hdr->off_crows = p.lay.off_crows;
        hdr->off_part_lse = p.lay.off_part_lse;
        hdr->off_part_o = p.lay.off_part_o;
        hdr->max_chunks = p.lay.max_chunks;
        hdr->max_ptiles = p.lay.max_ptiles;
        hdr->max_crows = p.lay.max_crows;
        hdr->max_prow = p.lay.max_prow;
        hdr->prow_used = sh.tot.y;
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) atomicAdd(&hdr->epoch, 1);
}

template <int HD, int NW, int DEPTH, bool KV8>
__global__ void __launch_bounds__(NW * 32, DecodeTiling<HD, KV8>::CTAS_PER_SM)
    decode_kernel(const __grid_constant__ CUtensorMap kv_map, const AttnParams p) {
    using Cfg = DecodeCfg<HD, NW, DEPTH, KV8>;
    using Math = DecodeMath<KV8>;
    constexpr int KSTEPS = HD / 16;       // k-steps of S = Q K^T
    constexpr int NTILES = HD / 8;        // n-tiles of O
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    uint8_t *ring = smem + warp * Cfg::kWarpBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + NW * Cfg::kWarpBytes) + warp * DEPTH;
    const uint32_t ring_u32 = smem_u32(ring);
    // E4M3: the staging area's V boxes, addressed as rows 16..31 of boxes kVBox apart
    const uint32_t vbase_kv8 = ring_u32 + DEPTH * Cfg::kStageBytes - Cfg::kVBoxBytes;
    constexpr uint32_t kVBox = KV8 ? Cfg::kVBoxBytes : Cfg::kBoxBytes;

    if (lane == 0) {
        for (int s = 0; s < DEPTH; ++s) mbar_init(&bars[s], 1);
        if (warp == 0) tma_prefetch_desc(&kv_map);
    }
    fence_barrier_init();
    __syncwarp();
    WsHeader *hdr = reinterpret_cast<WsHeader *>(p.ws);
    int32_t *status = reinterpret_cast<int32_t *>(p.ws);
    // a self-planned call: the plan in shared memory (the rings' space), read
    // and made while the kernel before this one may still run (it reads only
    // the call's metadata)
    __shared__ SelfPlanShared sp_shared;
    SelfChunk self_chunks[2];
    int n_items = 0;
    if (p.self_plan) {
        // (uniform over the CTA) a chunk CTA of a batch of at most 32 x
        // kWarpPlanPer requests plans per warp; the last CTA, and every CTA of a
        // larger batch, in shared memory
        const bool warp_plan = p.num_seqs <= 32 * kWarpPlanPer && blockIdx.x != gridDim.x - 1;
        if (warp_plan)
            n_items = decode_warp_plan(p, self_chunks, (gridDim.x - 1) * NW, blockIdx.x * NW + warp);
        else
            n_items = decode_self_plan<NW>(p, reinterpret_cast<int *>(smem), sp_shared, self_chunks);
        // the cache write before this kernel (and everything before it) is complete
        pdl_wait();
        if (blockIdx.x == gridDim.x - 1) {
            decode_self_plan_publish<NW>(p, reinterpret_cast<const int *>(smem), sp_shared);
            pdl_trigger();
            return;                              // (no chunks of its own)
        }
        if (!warp_plan) __syncthreads();         // the plan's shared memory is the rings' from here on
    } else {
        pdl_wait();       // the plan (and the cache write before it) are complete
    }
    pdl_trigger();
    // an error of a self-planned call is stored once the last CTA has reset the
    // status (the header's epoch moved on), so that the reset never overwrites it
    const int epoch0 = p.self_plan ? *reinterpret_cast<volatile int32_t *>(&hdr->epoch) : 0;
    auto report = [&](int32_t code) {
        if (p.self_plan) {
            const uint64_t t0 = global_ns();
            while (*reinterpret_cast<volatile int32_t *>(&hdr->epoch) == epoch0 && global_ns() - t0 < kWaitLimitNs) {
            }
        }
        set_status(status, code);
    };
    // the plan's lists, read through L2 (the plan wrote them; the offsets are the
    // layout the plan was given)
    const int4 *req = reinterpret_cast<const int4 *>(p.ws + p.lay.off_req);
    const int4 *chunks = reinterpret_cast<const int4 *>(p.ws + p.lay.off_chunks);
    float *part_lse = reinterpret_cast<float *>(p.ws + p.lay.off_part_lse);
    float *part_o = reinterpret_cast<float *>(p.ws + p.lay.off_part_o);
    if (!p.self_plan) n_items = __ldcg(&hdr->n_chunks) * p.num_kv_heads;

    const int W = (p.self_plan ? gridDim.x - 1 : gridDim.x) * NW;   // (a self-planned call: not the last CTA)
    const int wid = blockIdx.x * NW + warp;
    uint32_t seq = 0;              // pages consumed so far by this warp (ring position)
    const int g4 = lane >> 2;      // fragment row within 8
    const int t4 = lane & 3;       // fragment column pair
    const float NEG_INF = -__int_as_float(0x7f800000);

    for (int round = 0; round * W < n_items; ++round) {
        const int item = (round & 1) ? round * W + (W - 1 - wid) : round * W + wid;   // snake order
        if (item >= n_items) continue;
        // (a self-planned call has at most two rounds)
        const SelfChunk sc = (round & 1) ? self_chunks[1] : self_chunks[0];
        const int4 ch = p.self_plan ? make_int4(sc.r, sc.k, sc.pb, sc.pb + sc.npages) : __ldcg(chunks + item / p.num_kv_heads);
        const int g = item % p.num_kv_heads;
        const int r = ch.x;
        const int pb = ch.z;
        const int npages = ch.w - ch.z;
        const int L = p.seq_lens[r];
        const int qs = p.qsl[r];
        const int qlen = p.qsl[r + 1] - qs;
        const int ctx = L - qlen;
        const int rows_total = qlen * p.G;
        const bool split_mode = rows_total <= 16;
        const int tile = split_mode ? 0 : ch.y;
        const int split = split_mode ? ch.y : 0;
        const int4 info = p.self_plan ? make_int4(sc.n_split, sc.pbase, 0, 0) : __ldcg(req + r);
        const int n_split = split_mode ? info.x : 1;
        const int rows = min(16, rows_total - 16 * tile);

        // this thread's two fragment rows
        const int R0 = g4, R1 = g4 + 8;
        const int i0 = (16 * tile + R0) / p.G, hh0 = (16 * tile + R0) % p.G;
        const int i1 = (16 * tile + R1) / p.G, hh1 = (16 * tile + R1) % p.G;
        const int lim0 = R0 < rows ? ctx + i0 + 1 : 0;      // keys [0, lim) visible
        const int lim1 = R1 < rows ? ctx + i1 + 1 : 0;

        // block-table window: lane l holds the block of page (wbase + l)
        const int32_t *bt = p.block_tables + static_cast<int64_t>(r) * p.max_blocks_per_seq + pb;
        int wbase = 0;
        int win = lane < npages ? __ldg(bt + lane) : -1;

        auto issue = [&](int k) {            // page k of this chunk -> its ring stage
            const int blk = __shfl_sync(0xffffffffu, win, k - wbase);
            if (lane == 0) {
                if (blk < 0 || blk >= p.num_blocks) report(PKV_ERR_DEVICE_INDEX);
                const uint32_t st = (seq + k) % DEPTH;
                uint8_t *dst = ring + st * Cfg::kStageBytes;
                mbar_arrive_expect_tx(&bars[st], Cfg::kStageBytes);
                if constexpr (KV8) {
                    tma_load_5d(dst, &kv_map, &bars[st], 0, 0, 0, g, blk);       // the whole 8-bit page
                } else {
#pragma unroll
                    for (int bx = 0; bx < Cfg::kBoxes; ++bx)
                        tma_load_5d(dst + bx * Cfg::kBoxBytes, &kv_map, &bars[st], bx * 64, 0, 0, g, blk);
                }
            }
        };
        int issued = min(DEPTH, npages);
        for (int k = 0; k < issued; ++k) issue(k);

        // Q fragments (A operand, rows = (query token, q head) pairs)
        uint32_t qf[KSTEPS][4];
        {
            const __nv_bfloat16 *q0p = p.query + static_cast<int64_t>(qs + i0) * p.q_stride +
                                       static_cast<int64_t>(g * p.G + hh0) * HD;
            const __nv_bfloat16 *q1p = p.query + static_cast<int64_t>(qs + i1) * p.q_stride +
                                       static_cast<int64_t>(g * p.G + hh1) * HD;
            // E4M3 cache: the head dimension is permuted, the same way for Q and
            // K (a dot product does not depend on the order of its terms): in
            // k-step kk, lane column t4 takes dims t4 * HD/4 + 4 kk + 0..3 into
            // its k slots (2 t4, 2 t4 + 1, 2 t4 + 8, 2 t4 + 9), so that its K
            // values for one key are HD/4 contiguous bytes of the raw page
#pragma unroll
            for (int kk = 0; kk < KSTEPS; ++kk) {
                const int c = KV8 ? t4 * (HD / 4) + 4 * kk : kk * 16 + 2 * t4;
                const int c2 = KV8 ? c + 2 : c + 8;
                qf[kk][0] = R0 < rows ? __ldg(reinterpret_cast<const uint32_t *>(q0p + c)) : 0u;
                qf[kk][1] = R1 < rows ? __ldg(reinterpret_cast<const uint32_t *>(q1p + c)) : 0u;
                qf[kk][2] = R0 < rows ? __ldg(reinterpret_cast<const uint32_t *>(q0p + c2)) : 0u;
                qf[kk][3] = R1 < rows ? __ldg(reinterpret_cast<const uint32_t *>(q1p + c2)) : 0u;
            }
        }
        // score factors of the two rows (log2 domain); for an E4M3 cache each
        // Q row is scaled by a power of two 2^e into [2^14, 2^15) before it is
        // rounded to f16 (exact but for parts below 2^-24 of the row's
        // largest), and 2^-e and k_scale go into the factor
        float sf0 = p.scale_log2, sf1 = p.scale_log2;
        if constexpr (KV8) {
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int kk = 0; kk < KSTEPS; ++kk) {
                a0 = fmaxf(a0, fmaxf(fmaxf(fabsf(__uint_as_float(qf[kk][0] << 16)),
                                           fabsf(__uint_as_float(qf[kk][0] & 0xFFFF0000u))),
                                     fmaxf(fabsf(__uint_as_float(qf[kk][2] << 16)),
                                           fabsf(__uint_as_float(qf[kk][2] & 0xFFFF0000u)))));
                a1 = fmaxf(a1, fmaxf(fmaxf(fabsf(__uint_as_float(qf[kk][1] << 16)),
                                           fabsf(__uint_as_float(qf[kk][1] & 0xFFFF0000u))),
                                     fmaxf(fabsf(__uint_as_float(qf[kk][3] << 16)),
                                           fabsf(__uint_as_float(qf[kk][3] & 0xFFFF0000u)))));
            }
            a0 = fmaxf(a0, __shfl_xor_sync(0xffffffffu, a0, 1));
            a0 = fmaxf(a0, __shfl_xor_sync(0xffffffffu, a0, 2));
            a1 = fmaxf(a1, __shfl_xor_sync(0xffffffffu, a1, 1));
            a1 = fmaxf(a1, __shfl_xor_sync(0xffffffffu, a1, 2));
            // e = 14 - floor(log2 a), held in [-114, 126] so 2^e and 2^-e are normal
            const int e0 = a0 > 0.f ? min(126, max(-114, 14 - ilogbf(a0))) : 0;
            const int e1 = a1 > 0.f ? min(126, max(-114, 14 - ilogbf(a1))) : 0;
            const float u0 = __int_as_float((e0 + 127) << 23), u1 = __int_as_float((e1 + 127) << 23);
            auto to_f16 = [](uint32_t bf2, float u) {
                const __half2 h = __floats2half2_rn(__uint_as_float(bf2 << 16) * u,
                                                    __uint_as_float(bf2 & 0xFFFF0000u) * u);
                return *reinterpret_cast<const uint32_t *>(&h);
            };
#pragma unroll
            for (int kk = 0; kk < KSTEPS; ++kk) {
                qf[kk][0] = to_f16(qf[kk][0], u0);
                qf[kk][1] = to_f16(qf[kk][1], u1);
                qf[kk][2] = to_f16(qf[kk][2], u0);
                qf[kk][3] = to_f16(qf[kk][3], u1);
            }
            sf0 = p.scale_log2 * p.k_scale * __int_as_float((127 - e0) << 23);
            sf1 = p.scale_log2 * p.k_scale * __int_as_float((127 - e1) << 23);
        }

        float o[NTILES][4];
#pragma unroll
        for (int n = 0; n < NTILES; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
        float m0 = NEG_INF, m1 = NEG_INF, l0 = 0.f, l1 = 0.f;
        int failed_at = -1;

        for (int k = 0; k < npages; ++k) {
            const uint32_t st = (seq + k) % DEPTH;
            const uint32_t par = ((seq + k) / DEPTH) & 1u;
            const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars[st], par));
            if (!ok) {
                failed_at = k;
                break;
            }
            const uint32_t page = ring_u32 + st * Cfg::kStageBytes;
            // V rows 16..31 of box bx at swz(vbase + bx * kVBox, row, chunk): the ring
            // stage's own boxes (bf16), or the staging area's V-only boxes (E4M3)
            const uint32_t vbase = KV8 ? vbase_kv8 : page;
            const int j0 = (pb + k) * kBlock;       // first key of this page
            // E4M3: this lane's K bytes of keys g4 and 8 + g4 (HD/4 each, see the Q
            // fragments), straight from the raw page
            uint32_t kraw[2][KV8 ? KSTEPS : 1];
            if constexpr (KV8) {
#pragma unroll
                for (int n = 0; n < 2; ++n)
#pragma unroll
                    for (int v = 0; v < KSTEPS / 4; ++v)
                        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                                     : "=r"(kraw[n][4 * v]), "=r"(kraw[n][4 * v + 1]), "=r"(kraw[n][4 * v + 2]),
                                       "=r"(kraw[n][4 * v + 3])
                                     : "r"(page + (8 * n + g4) * HD + t4 * (HD / 4) + 16 * v));
                // widen the V rows, then hand the stage back to the copy engine
                widen_e4m3_values<HD>(page, vbase_kv8, lane);
                fence_proxy_async_smem();
                __syncwarp();
                const int nk = k + DEPTH;
                if (nk < npages) {
                    if (nk - wbase >= 32) {
                        wbase += 32;
                        win = wbase + lane < npages ? __ldg(bt + wbase + lane) : -1;
                    }
                    issue(nk);
                    ++issued;
                }
            }

            // zero V rows past the end of the sequence (last page only)
            if (j0 + kBlock > L) {
                const int vfirst = L - j0;
                const int nrows = kBlock - vfirst;
                for (int e = lane; e < Cfg::kBoxes * nrows * 8; e += 32) {
                    const int bx = e / (nrows * 8);
                    const int rem = e % (nrows * 8);
                    const int row = kBlock + vfirst + rem / 8;
                    const int chunk = rem % 8;
                    const uint32_t a = swz(vbase + bx * kVBox, row, chunk);
                    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0u) : "memory");
                }
                __syncwarp();
            }

            // S = Q K^T for the page's 16 tokens (two n-tiles)
            float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kk = 0; kk < KSTEPS; ++kk) {
                uint32_t b0, b1, b2, b3;
                if constexpr (KV8) {
                    e4m3x4_to_f16x4(kraw[0][kk], b0, b1);
                    e4m3x4_to_f16x4(kraw[1][kk], b2, b3);
                } else {
                    const int bx = kk / 4;
                    const int tok = ((lane >> 4) << 3) + (lane & 7);
                    const int chunk = (kk % 4) * 2 + ((lane >> 3) & 1);
                    ldsm_x4(swz(page + bx * Cfg::kBoxBytes, tok, chunk), b0, b1, b2, b3);
                }
                Math::mma(s0, qf[kk], b0, b1);
                Math::mma(s1, qf[kk], b2, b3);
            }

            // online softmax in the log2 domain; keys a row may not see get -inf
            const int c0 = j0 + 2 * t4, c1 = c0 + 1, c8 = c0 + 8, c9 = c0 + 9;
            float x[8];
            x[0] = c0 < lim0 ? s0[0] * sf0 : NEG_INF;
            x[1] = c1 < lim0 ? s0[1] * sf0 : NEG_INF;
            x[2] = c0 < lim1 ? s0[2] * sf1 : NEG_INF;
            x[3] = c1 < lim1 ? s0[3] * sf1 : NEG_INF;
            x[4] = c8 < lim0 ? s1[0] * sf0 : NEG_INF;
            x[5] = c9 < lim0 ? s1[1] * sf0 : NEG_INF;
            x[6] = c8 < lim1 ? s1[2] * sf1 : NEG_INF;
            x[7] = c9 < lim1 ? s1[3] * sf1 : NEG_INF;
            float mx0 = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[4], x[5]));
            float mx1 = fmaxf(fmaxf(x[2], x[3]), fmaxf(x[6], x[7]));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
            // a row's reference maximum moves only on its first visible key or
            // when the page's maximum exceeds it by more than 2^8, so weights
            // stay below 2^8 and O is rescaled (warp-uniformly) only then
            const bool up0 = mx0 > m0 + 8.f, up1 = mx1 > m1 + 8.f;
            if (__any_sync(0xffffffffu, up0 || up1)) {
                const float a0 = up0 ? fast_exp2(m0 - mx0) : 1.f;   // 0 when m = -inf
                const float a1 = up1 ? fast_exp2(m1 - mx1) : 1.f;
                m0 = up0 ? mx0 : m0;
                m1 = up1 ? mx1 : m1;
                l0 *= a0;
                l1 *= a1;
#pragma unroll
                for (int n = 0; n < NTILES; ++n) {
                    o[n][0] *= a0;
                    o[n][1] *= a0;
                    o[n][2] *= a1;
                    o[n][3] *= a1;
                }
            }
            const float ref0 = m0 == NEG_INF ? 0.f : m0;
            const float ref1 = m1 == NEG_INF ? 0.f : m1;
            float pr[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) pr[e] = fast_exp2(x[e] - (((e >> 1) & 1) ? ref1 : ref0));
            l0 += (pr[0] + pr[1] + pr[4] + pr[5]);
            l1 += (pr[2] + pr[3] + pr[6] + pr[7]);
            // P for P V.  bf16 cache: a bf16 pair (hi + remainder), about 16 bits of
            // each weight (one bf16 round, 8 bits, broke the tolerance on short rows).
            // E4M3 cache: one f16 per weight, 11 bits (a relative error below 2^-11
            // per weight, several times inside the tolerance), so one product per tile
            uint32_t pa[4], pl[4];
            if constexpr (KV8) {
                Math::round(pr[0], pr[1], pa[0]);
                Math::round(pr[2], pr[3], pa[1]);
                Math::round(pr[4], pr[5], pa[2]);
                Math::round(pr[6], pr[7], pa[3]);
            } else {
                Math::split(pr[0], pr[1], pa[0], pl[0]);
                Math::split(pr[2], pr[3], pa[1], pl[1]);
                Math::split(pr[4], pr[5], pa[2], pl[2]);
                Math::split(pr[6], pr[7], pa[3], pl[3]);
            }

            // O += P V (V rows are the page's tokens, read transposed)
#pragma unroll
            for (int n = 0; n < NTILES; n += 2) {
                const int bx = n / 8;
                const int tok = ((lane >> 3) & 1) * 8 + (lane & 7);
                const int chunk = (n % 8) + (lane >> 4);
                uint32_t b0, b1, b2, b3;
                ldsm_x4_trans(swz(vbase + bx * kVBox, kBlock + tok, chunk), b0, b1, b2, b3);
                Math::mma(o[n], pa, b0, b1);
                Math::mma(o[n + 1], pa, b2, b3);
                if constexpr (!KV8) {
                    Math::mma(o[n], pl, b0, b1);
                    Math::mma(o[n + 1], pl, b2, b3);
                }
            }

            if constexpr (!KV8) {
                // refill this stage with page k + DEPTH of the chunk
                fence_proxy_async_smem();
                __syncwarp();
                const int nk = k + DEPTH;
                if (nk < npages) {
                    if (nk - wbase >= 32) {
                        wbase += 32;
                        win = wbase + lane < npages ? __ldg(bt + wbase + lane) : -1;
                    }
                    issue(nk);
                    ++issued;
                }
            } else {
                __syncwarp();                    // the staging page is rewritten by the next page
            }
        }

        if (failed_at >= 0) {
            report(PKV_ERR_DEVICE_TIMEOUT);
            // let copies already in flight land before the CTA's memory is released
            for (int k = failed_at; k < issued; ++k) {
                const uint32_t st = (seq + k) % DEPTH;
                mbar_wait_bounded(&bars[st], ((seq + k) / DEPTH) & 1u);
            }
            return;
        }
        seq += npages;

        // finish the rows: quad sums of l, then normalise
        l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
        l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
        // (an E4M3 cache's V values are code * v_scale: the scale is applied once here)
        const float inv0 = l0 > 0.f ? (KV8 ? p.v_scale / l0 : 1.f / l0) : 0.f;
        const float inv1 = l1 > 0.f ? (KV8 ? p.v_scale / l1 : 1.f / l1) : 0.f;
        const int h0 = g * p.G + hh0, h1 = g * p.G + hh1;
        if (n_split <= 1) {
            if (R0 < rows) {
                __nv_bfloat16 *dst = p.out + (static_cast<int64_t>(qs + i0) * p.num_q_heads + h0) * HD;
#pragma unroll
                for (int n = 0; n < NTILES; ++n)
                    *reinterpret_cast<uint32_t *>(dst + n * 8 + 2 * t4) = pack_bf16x2(o[n][0] * inv0, o[n][1] * inv0);
            }
            if (R1 < rows) {
                __nv_bfloat16 *dst = p.out + (static_cast<int64_t>(qs + i1) * p.num_q_heads + h1) * HD;
#pragma unroll
                for (int n = 0; n < NTILES; ++n)
                    *reinterpret_cast<uint32_t *>(dst + n * 8 + 2 * t4) = pack_bf16x2(o[n][2] * inv1, o[n][3] * inv1);
            }
        } else {
            const float LN2 = 0.69314718055994531f;
            if (R0 < rows) {
                const int64_t prow = info.y + (static_cast<int64_t>(i0) * p.num_q_heads + h0) * n_split + split;
                float *dst = part_o + prow * HD;
#pragma unroll
                for (int n = 0; n < NTILES; ++n)
                    *reinterpret_cast<float2 *>(dst + n * 8 + 2 * t4) = make_float2(o[n][0] * inv0, o[n][1] * inv0);
                if (t4 == 0) part_lse[prow] = l0 > 0.f ? (m0 + __log2f(l0)) * LN2 : NEG_INF;
            }
            if (R1 < rows) {
                const int64_t prow = info.y + (static_cast<int64_t>(i1) * p.num_q_heads + h1) * n_split + split;
                float *dst = part_o + prow * HD;
#pragma unroll
                for (int n = 0; n < NTILES; ++n)
                    *reinterpret_cast<float2 *>(dst + n * 8 + 2 * t4) = make_float2(o[n][2] * inv1, o[n][3] * inv1);
                if (t4 == 0) part_lse[prow] = l1 > 0.f ? (m1 + __log2f(l1)) * LN2 : NEG_INF;
            }
        }
    }
}

// ---- host side --------------------------------------------------------------------

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// Tensor map of the cache as a 5-D bf16 tensor {head_size, 16, 2, Hkv, num_blocks}
// (innermost first), loaded in boxes of {64, 16, 2, 1, 1} with 128-byte swizzle.
static int make_kv_map(CUtensorMap *map, const void *kv_cache, int64_t num_blocks, int32_t num_kv_heads,
                       int32_t head_size) {
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return PKV_ERR_CUDA;
    const cuuint64_t dims[5] = {static_cast<cuuint64_t>(head_size), kBlock, 2,
                                static_cast<cuuint64_t>(num_kv_heads), static_cast<cuuint64_t>(num_blocks)};
    const cuuint64_t row = static_cast<cuuint64_t>(head_size) * 2;
    const cuuint64_t strides[4] = {row, row * kBlock, row * kBlock * 2, row * kBlock * 2 * num_kv_heads};
    const cuuint32_t box[5] = {64, kBlock, 2, 1, 1};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    const CUresult rc = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(kv_cache), dims, strides,
                            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return rc == CUDA_SUCCESS ? PKV_OK : PKV_ERR_CUDA;
}

// Tensor map of an E4M3 cache as a 5-D byte tensor {head_size, 16, 2, Hkv,
// num_blocks}; one box is a whole page of one kv head (K and V rows, 2*16*d
// bytes), unswizzled: the kernel widens it to f16 itself.
static int make_kv_map_e4m3(CUtensorMap *map, const void *kv_cache, int64_t num_blocks, int32_t num_kv_heads,
                            int32_t head_size) {
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return PKV_ERR_CUDA;
    const cuuint64_t dims[5] = {static_cast<cuuint64_t>(head_size), kBlock, 2,
                                static_cast<cuuint64_t>(num_kv_heads), static_cast<cuuint64_t>(num_blocks)};
    const cuuint64_t row = static_cast<cuuint64_t>(head_size);
    const cuuint64_t strides[4] = {row, row * kBlock, row * kBlock * 2, row * kBlock * 2 * num_kv_heads};
    const cuuint32_t box[5] = {static_cast<cuuint32_t>(head_size), kBlock, 2, 1, 1};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    const CUresult rc = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, const_cast<void *>(kv_cache), dims, strides, box,
                            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return rc == CUDA_SUCCESS ? PKV_OK : PKV_ERR_CUDA;
}

template <int HD, int NW, int DEPTH, bool KV8>
static int launch_decode(const CUtensorMap &map, const AttnParams &p, int grid, int dev, cudaStream_t stream) {
    using Cfg = DecodeCfg<HD, NW, DEPTH, KV8>;
    // 228 KiB of shared memory per SM, 1 KiB of it reserved per resident CTA
    static_assert((Cfg::kSmem + 1024) * DecodeTiling<HD, KV8>::CTAS_PER_SM <= 228 * 1024,
                  "the tiling's CTAs fit one SM's shared memory");
    static std::mutex mu;
    static uint64_t done_mask = 0;       // devices whose shared-memory limit is already raised
    {
        std::lock_guard<std::mutex> lock(mu);
        const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
        if (!bit || !(done_mask & bit)) {
            if (cudaFuncSetAttribute(decode_kernel<HD, NW, DEPTH, KV8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     Cfg::kSmem) != cudaSuccess)
                return PKV_ERR_CUDA;
            done_mask |= bit;
        }
    }
    if (launch_pdl(decode_kernel<HD, NW, DEPTH, KV8>, dim3(grid), dim3(NW * 32), Cfg::kSmem, stream, map, p) !=
        cudaSuccess)
        return PKV_ERR_CUDA;
    return PKV_OK;
}


int make_decode_map(CUtensorMap *map, const void *kv_cache, int64_t num_blocks, int32_t num_kv_heads,
                    int32_t head_size, bool kv8) {
    return kv8 ? make_kv_map_e4m3(map, kv_cache, num_blocks, num_kv_heads, head_size)
               : make_kv_map(map, kv_cache, num_blocks, num_kv_heads, head_size);
}

int decode_ctas_per_sm(int32_t head_size, bool kv8) {
    if (kv8) return head_size == 64 ? DecodeTiling<64, true>::CTAS_PER_SM : DecodeTiling<128, true>::CTAS_PER_SM;
    return head_size == 64 ? DecodeTiling<64>::CTAS_PER_SM : DecodeTiling<128>::CTAS_PER_SM;
}

int launch_decode_path(const CUtensorMap &map, const AttnParams &ap, int32_t head_size, bool kv8, int grid, int dev,
                       cudaStream_t st) {
    if (kv8) {
        using T64 = DecodeTiling<64, true>;
        using T128 = DecodeTiling<128, true>;
        return head_size == 64 ? launch_decode<64, T64::NW, T64::DEPTH, true>(map, ap, grid, dev, st)
                               : launch_decode<128, T128::NW, T128::DEPTH, true>(map, ap, grid, dev, st);
    }
    using T64 = DecodeTiling<64>;
    using T128 = DecodeTiling<128>;
    return head_size == 64 ? launch_decode<64, T64::NW, T64::DEPTH, false>(map, ap, grid, dev, st)
                           : launch_decode<128, T128::NW, T128::DEPTH, false>(map, ap, grid, dev, st);
}

}  // namespace pkv
