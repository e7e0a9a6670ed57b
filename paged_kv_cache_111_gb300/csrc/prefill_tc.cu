// Prefill-chunk paged attention on the 5th-generation tensor cores (tcgen05).
//
// The same computation as the decode path ("continuous batching and
// PagedAttention" tutorial, section 3.6: loop over the request's blocks
// through its block table, accumulate softmax(QK^T)V), for requests whose
// rows are many: a chunk of a chunked prefill ("Inside vLLM: Anatomy of a
// High-Throughput LLM Inference System", chunked prefill; "vLLM internals:
// managing the KV cache like an OS manages memory", section 3.2) attends
// causally, query i of the chunk seeing keys 0 .. context + i.
//
// One CTA computes one 128-row tile for one kv head.  Rows are
// (query token, q head of the GQA group) pairs, so one K/V tile in shared
// memory serves every q head of the group.  Per 128-key KV tile:
//   S = Q K^T      tcgen05.mma, A = Q from tensor memory, B = K from shared
//                  memory (K-major, 128-byte swizzle), D in tensor memory
//                  (two S buffers)
//   softmax        two threads per row, each with half of the tile's keys,
//                  read S from tensor memory, mask, share their row maxima
//                  through shared memory, keep a running max (rescaling
//                  their half of O only when the max grows by more than 2^8)
//                  and write P (bf16) over S
//   O += P V       tcgen05.mma, A = P from tensor memory, B = V (MN-major)
//                  from shared memory, D = O in tensor memory
// Every product reads A from tensor memory: on this part a change between
// shared-memory and tensor-memory A operands from one group of MMAs to the
// next costs about a third of the tensor pipe's rate.
// Warp roles: warp 0 loads (TMA: K and V pages through the block table into
// a three-stage ring), warp 1 issues the MMAs, warp 2 owns the
// tensor-memory allocation, warps 4-11 do softmax and the epilogue.
//
// When any row of the tile puts a large share of its weight on few keys of
// a KV tile (rows with few visible keys, or a peaked softmax), that tile's P
// also enters P V as its bf16 remainder (a second MMA), keeping ~16 bits per
// weight; other tiles' weights are each small and bf16 P is enough.  V rows past the sequence end in
// its last page are zeroed before P V, so NaN in unwritten cache slots never
// meets a zero weight.  Every wait is bounded.
#include <mutex>

#include "attn_internal.cuh"
#include "tc_common.cuh"

namespace pkv {

template <int HD>
struct PrefillCfg {
    static constexpr int kHalves = HD / 64;
    static constexpr int kStages = 3;                        // K and V ring depth
    static constexpr int kKVBytes = kHalves * kPrefillKeys * 128;   // one K (or V) tile
    static constexpr int kOffK = 0;
    static constexpr int kOffV = kOffK + kStages * kKVBytes;
    static constexpr int kOffBar = kOffV + kStages * kKVBytes;
    static constexpr int kOffXchg = kOffBar + 512;            // softmax halves' maxima and sums (3 KiB)
    static constexpr int kSmem = kOffXchg + 3072 + 1024;    // + alignment slack
    // tensor memory: two S buffers (each later holding that tile's P and its
    // bf16 remainder), O, and Q as the A operand of S = Q K^T
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256, kColQ = 384;
};

enum PrefillBar { kQFull = 0, kKFull0, kKFull1, kKFull2, kVFull0, kVFull1, kVFull2, kKEmpty0, kKEmpty1, kKEmpty2,
                  kVEmpty0, kVEmpty1, kVEmpty2, kSFull0, kSFull1, kPFull0, kPFull1, kODone0, kODone1, kVFix,
                  kXchg0, kXchg1, kXchg2, kXchg3,      // the two softmax warps of a lane quadrant
                  kNumBars };
static_assert(kNumBars * 8 + 16 + 64 <= 512, "barriers, the TMEM address slot and the votes fit their 512 bytes");
// P of tile j is announced on kPFull0 + (j & 1): with one barrier per parity a
// barrier never runs two phases ahead of the MMA thread's wait on it (the
// softmax warps can finish tile j + 1 before the MMA thread looks at tile j).

// A row whose weights in a KV tile are concentrated (sum of squared weights
// of the tile above this fraction of the squared running sum) needs P's bf16
// remainder in P V: bf16 rounding of a few large weights would otherwise
// exceed the output tolerance.
constexpr float kLoConcentration = 0.01f;

// ---- softmax arithmetic on fp32 pairs (Blackwell f32x2 instructions) ----------------

__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float &a, float &b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Bounded wait shared by every role; on timeout records the error and
// reports it so the role can stop.
__device__ __forceinline__ bool pf_wait(uint64_t *bar, uint32_t parity, int32_t *status) {
    if (mbar_wait_bounded(bar, parity)) return true;
    set_status(status, PKV_ERR_DEVICE_TIMEOUT);
    return false;
}

// CASCADE = false: one 128-row tile of one long request (a prefill chunk),
// causal, written to `out`.  CASCADE = true: 128 rows taken from every
// request that shares the first prefix_blocks blocks of its table with
// request 0, against one range of those blocks' KV tiles (every key of the
// prefix is visible to every such row); the result for range i is split i of
// each row (normalised partial output and its log-sum-exp), merged with the
// row's other splits by the combine.
template <int HD, bool CASCADE>
__global__ void __launch_bounds__(384, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap kv_map, const __nv_bfloat16 *__restrict__ query,
                   const int64_t q_stride, const PrefillParams p) {
    using Cfg = PrefillCfg<HD>;
    constexpr int S = Cfg::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg::kOffBar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + kNumBars);
    volatile uint32_t *votes = tmem_slot + 4;          // [2 tiles in flight][8 softmax warps]
    const uint32_t sK = smem_u32(smem + Cfg::kOffK);
    const uint32_t sV = smem_u32(smem + Cfg::kOffV);

    pdl_wait();       // the plan, the cache write and the decode kernel are complete
    pdl_trigger();
    const WsHeader *hdr = reinterpret_cast<const WsHeader *>(p.ws);
    int32_t *status = reinterpret_cast<int32_t *>(p.ws);
    const int n_parts = CASCADE ? hdr->prefix_parts : 1;
    const int n_tiles = CASCADE ? (hdr->n_crows + kPrefillRows - 1) / kPrefillRows : hdr->n_ptiles;
    const int n_items = n_tiles * p.num_kv_heads * n_parts;
    const int item = blockIdx.x;
    if (item >= n_items) return;                       // uniform over the CTA
    const int g = item % p.num_kv_heads;
    const int G = p.G;
    // t0: first KV tile of this CTA's key range (cascade part; 0 otherwise)
    int r, n_kv, L, qs, ctx, rows_total, row0, n_pages, part = 0, t0 = 0;
    if constexpr (CASCADE) {
        r = 0;                                         // the prefix blocks are read through request 0's table
        L = hdr->prefix_blocks * kBlock;               // every row sees keys 0 .. L-1
        const int kv_all = (L + kPrefillKeys - 1) / kPrefillKeys;
        const int per = (kv_all + n_parts - 1) / n_parts;   // the plan makes every range non-empty
        part = (item / p.num_kv_heads) % n_parts;
        t0 = part * per;
        n_kv = min(kv_all, t0 + per) - t0;
        n_pages = hdr->prefix_blocks;
        qs = ctx = 0;
        rows_total = hdr->n_crows;
        row0 = (item / (p.num_kv_heads * n_parts)) * kPrefillRows;
    } else {
        const int4 tile = reinterpret_cast<const int4 *>(p.ws + hdr->off_ptiles)[item / p.num_kv_heads];
        r = tile.x;
        n_kv = tile.z;
        L = p.seq_lens[r];
        qs = p.qsl[r];
        const int qlen = p.qsl[r + 1] - qs;
        ctx = L - qlen;
        rows_total = qlen * G;
        row0 = tile.y * kPrefillRows;                  // first request row of the tile
        n_pages = (L + kBlock - 1) / kBlock;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int b = 0; b < kNumBars; ++b)
            mbar_init(&bars[b], (b == kPFull0 || b == kPFull1 || b == kQFull) ? 8 : (b >= kXchg0 ? 2 : 1));
        tma_prefetch_desc(&kv_map);
    }
    if (warp == 2) {
        tmem_alloc(tmem_slot, Cfg::kTmemCols);
        tmem_relinquish();
    }
    fence_barrier_init();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // the KV tile holding the sequence's last key, when that page is partial
    const int end_tile = (!CASCADE && (L % kBlock)) ? (L - 1) / kPrefillKeys : -1;

    if (warp == 0) {
        // ---------------- producer: K and V pages through the block table ----------------
        bool ok = true;
        const int32_t *bt = p.block_tables + static_cast<int64_t>(r) * p.max_blocks_per_seq;
        // block ids in windows of 32 pages (4 KV tiles), one lane per page; the
        // next window is loaded a window ahead.  Pages past the sequence are -1
        // and load as zeros (outside the tensor map).
        constexpr int kPagesPerTile = kPrefillKeys / kBlock;
        auto load_window = [&](int w) -> int {
            const int page = t0 * kPagesPerTile + w * 32 + lane;
            const int b = page < n_pages ? __ldg(bt + page) : -1;
            if (page < n_pages && (b < 0 || b >= p.num_blocks))
                set_status(status, PKV_ERR_DEVICE_INDEX);   // loaded as zeros by the bounded TMA, reported
            return b;
        };
        int win_cur = load_window(0);
        int win_next = load_window(1);
        for (int j = 0; j < n_kv && ok; ++j) {
            const int st = j % S;
            if (j > 0 && (j * kPagesPerTile) % 32 == 0) {
                win_cur = win_next;
                win_next = load_window(j * kPagesPerTile / 32 + 1);
            }
            const int wofs = (j * kPagesPerTile) % 32;
            int pb[kPagesPerTile];
#pragma unroll
            for (int pg = 0; pg < kPagesPerTile; ++pg) pb[pg] = __shfl_sync(0xffffffffu, win_cur, wofs + pg);
            // K of tile j once S of tile j-S has read its stage
            if (j >= S) ok = __all_sync(0xffffffffu, pf_wait(&bars[kKEmpty0 + st], ((j - S) / S) & 1, status));
            if (!ok) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(&bars[kKFull0 + st], Cfg::kKVBytes);
#pragma unroll
                for (int pg = 0; pg < kPagesPerTile; ++pg)
                    for (int h = 0; h < Cfg::kHalves; ++h)
                        tma_load_5d(smem + Cfg::kOffK + st * Cfg::kKVBytes + h * (kPrefillKeys * 128) + pg * 2048,
                                    &kv_map, &bars[kKFull0 + st], h * 64, 0, 0, g, pb[pg]);
            }
            // V of tile j once P V of tile j-S has read its stage
            if (j >= S) ok = __all_sync(0xffffffffu, pf_wait(&bars[kVEmpty0 + st], ((j - S) / S) & 1, status));
            if (!ok) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(&bars[kVFull0 + st], Cfg::kKVBytes);
#pragma unroll
                for (int pg = 0; pg < kPagesPerTile; ++pg)
                    for (int h = 0; h < Cfg::kHalves; ++h)
                        tma_load_5d(smem + Cfg::kOffV + st * Cfg::kKVBytes + h * (kPrefillKeys * 128) + pg * 2048,
                                    &kv_map, &bars[kVFull0 + st], h * 64, 0, 1, g, pb[pg]);
            }
            if (j == end_tile) {
                // zero V rows past the sequence end in its last (partial) page
                ok = __all_sync(0xffffffffu, pf_wait(&bars[kVFull0 + st], (j / S) & 1, status));
                if (!ok) break;
                const int lp = (L - 1) / kBlock - j * kPagesPerTile;   // page within the tile
                const int first = L % kBlock;
                const int nrows = kBlock - first;
                for (int e = lane; e < Cfg::kHalves * nrows * 8; e += 32) {
                    const int h = e / (nrows * 8);
                    const int rem = e % (nrows * 8);
                    const int row = lp * kBlock + first + rem / 8;
                    const uint32_t a = sV + st * Cfg::kKVBytes + h * (kPrefillKeys * 128) + row * 128 + (rem % 8) * 16;
                    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0u) : "memory");
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[kVFix]);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t kIdescS = idesc_bf16_f32(kPrefillRows, kPrefillKeys, 0, 0);
            constexpr uint32_t kIdescO = idesc_bf16_f32(kPrefillRows, HD, 0, 1);
            bool ok = pf_wait(&bars[kQFull], 0, status);
            // S(j) = Q K^T into S buffer j & 1; A = Q in tensor memory
            auto issue_s = [&](int j) {
                const int st = j % S;
                const uint32_t d = tmem + ((j & 1) ? Cfg::kColS1 : Cfg::kColS0);
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const uint64_t b = smem_desc_sw128(sK + st * Cfg::kKVBytes + (kk >> 2) * (kPrefillKeys * 128) +
                                                           (kk & 3) * 32,
                                                       16, 1024);
                    umma_bf16_ts(d, tmem + Cfg::kColQ + kk * 8, b, kIdescS, kk > 0);
                }
                umma_commit(&bars[kSFull0 + (j & 1)]);
                umma_commit(&bars[kKEmpty0 + st]);
            };
            // O (+)= P V; A = P (or its remainder) in S buffer j & 1: keys
            // 64 h .. 64 h + 63 sit at columns 64 h + [0, 32) (P) and
            // 64 h + [32, 64) (remainder), each half within its own S columns
            auto issue_pv = [&](int j, uint32_t pcol, uint32_t accumulate) {
                const int st = j % S;
#pragma unroll
                for (int kk = 0; kk < kPrefillKeys / 16; ++kk) {
                    const uint64_t b = smem_desc_sw128(sV + st * Cfg::kKVBytes + kk * 2048, kPrefillKeys * 128, 1024);
                    umma_bf16_ts(tmem + Cfg::kColO, pcol + kk * 8 + (kk >> 2) * 32, b, kIdescO,
                                 (accumulate || kk > 0) ? 1u : 0u);
                }
            };
            for (int j0 = 0; j0 < 2 && j0 < n_kv && ok; ++j0) {
                ok = pf_wait(&bars[kKFull0 + j0], 0, status);
                if (!ok) break;
                tc_fence_after();
                issue_s(j0);
            }
            for (int j = 0; j < n_kv && ok; ++j) {
                const int st = j % S;
                ok = pf_wait(&bars[kPFull0 + (j & 1)], (j >> 1) & 1, status);
                if (ok) ok = pf_wait(&bars[kVFull0 + st], (j / S) & 1, status);
                if (ok && j == end_tile) ok = pf_wait(&bars[kVFix], 0, status);
                if (!ok) break;
                tc_fence_after();
                const uint32_t pbuf = tmem + ((j & 1) ? Cfg::kColS1 : Cfg::kColS0);
                uint32_t vote = 0;
#pragma unroll
                for (int w = 0; w < 8; ++w) vote |= votes[(j & 1) * 8 + w];
                const bool lo = vote != 0u;
                issue_pv(j, pbuf, j > 0);
                if (lo) issue_pv(j, pbuf + 32, 1);
                umma_commit(&bars[kODone0 + (j & 1)]);
                umma_commit(&bars[kVEmpty0 + st]);
                // S of tile j+2 overwrites S buffer j & 1, where P V of tile j reads
                // P: it is issued only once that product has completed (no
                // overlap of a tensor-memory operand read with a later write)
                if (j + 2 < n_kv) {
                    ok = pf_wait(&bars[kODone0 + (j & 1)], (j >> 1) & 1, status);
                    if (ok) ok = pf_wait(&bars[kKFull0 + (j + 2) % S], ((j + 2) / S) & 1, status);
                    if (!ok) break;
                    tc_fence_after();
                    issue_s(j + 2);
                }
            }
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ---------------- softmax + epilogue: two threads per row ----------------
        // warps 4-7 take keys (and output columns) of the first half of the tile,
        // warps 8-11 the second half; warp w reads tensor-memory lanes of quadrant
        // w % 4, so warps w and w + 4 share their 32 rows
        const int quad = warp & 3;
        const int half = (warp - 4) >> 2;
        const int row = quad * 32 + lane;
        const int rrow = row0 + row;                       // request row (cascade: row of the prefix pass)
        const bool valid = rrow < rows_total;
        // the row's query token and q head within the group; keys [0, lim) visible
        int tok = 0, hh = 0, lim = 0;
        int4 crow = make_int4(0, 0, 0, 0);
        if (valid) {
            if constexpr (CASCADE) {
                crow = reinterpret_cast<const int4 *>(p.ws + hdr->off_crows)[rrow];   // {token, request, index, head}
                tok = crow.x;
                hh = crow.w;
                lim = L;
            } else {
                tok = qs + rrow / G;
                hh = rrow % G;
                lim = ctx + rrow / G + 1;
            }
        }
        const float NEG_INF = -__int_as_float(0x7f800000);
        const uint32_t trow = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        constexpr int kHalfKeys = kPrefillKeys / 2;        // keys of a tile per thread
        constexpr int kHalfDims = HD / 2;                   // output columns per thread
        // exchange of the two halves' row maxima (by tile parity) and final sums
        float *xmax = reinterpret_cast<float *>(smem + Cfg::kOffXchg);          // [2][2][128]
        float *xsum = xmax + 2 * 2 * kPrefillRows;                               // [2][128]
        // the two warps of this quadrant meet on an mbarrier, one phase per
        // tile plus one for the final sums (bounded waits, like every other)
        uint64_t *xbar = &bars[kXchg0 + quad];
        auto post = [&]() {
            __syncwarp();
            if (lane == 0) mbar_arrive(xbar);
        };
        auto meet = [&](int phase) -> bool { return __all_sync(0xffffffffu, pf_wait(xbar, phase & 1, status)); };
        auto exchange = [&](int phase) -> bool {
            post();
            return meet(phase);
        };
        bool ok = true;

        // this half of the Q row -> tensor memory (A operand of S = Q K^T), zeros past the request
        {
            uint32_t qv[kHalfDims / 2];
            const __nv_bfloat16 *qp = query + static_cast<int64_t>(tok) * q_stride +
                                      static_cast<int64_t>(g * G + hh) * HD + half * kHalfDims;
#pragma unroll
            for (int c = 0; c < kHalfDims / 8; ++c) {
                const uint4 w = valid ? __ldg(reinterpret_cast<const uint4 *>(qp) + c) : make_uint4(0, 0, 0, 0);
                qv[4 * c + 0] = w.x;
                qv[4 * c + 1] = w.y;
                qv[4 * c + 2] = w.z;
                qv[4 * c + 3] = w.w;
            }
            if constexpr (kHalfDims / 2 == 32) {
                tmem_st32(trow + Cfg::kColQ + half * 32, qv);
            } else {
                tmem_st16(trow + Cfg::kColQ + half * 16, qv);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[kQFull]);
        }

        float m_ref = NEG_INF, l = 0.f;                    // l: this half's sum
        for (int j = 0; j < n_kv && ok; ++j) {
            const int sb = j & 1;
            const uint32_t sbuf = trow + (sb ? Cfg::kColS1 : Cfg::kColS0);
            ok = __all_sync(0xffffffffu, pf_wait(&bars[kSFull0 + sb], (j >> 1) & 1, status));
            if (!ok) break;
            tc_fence_after();
            // this half's scores (keys key0 .. key0 + 63); keys a row may not see
            // become -inf, tested only in tiles reaching some row's limit
            const int key0 = (t0 + j) * kPrefillKeys + half * kHalfKeys;
            float x[kHalfKeys];
            auto load_scores = [&]() {
                uint32_t v[2][32];
#pragma unroll
                for (int c = 0; c < 2; ++c) tmem_ld32(sbuf + half * kHalfKeys + c * 32, v[c]);
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < 2; ++c)
#pragma unroll
                    for (int e = 0; e < 32; ++e) x[c * 32 + e] = __uint_as_float(v[c][e]);
                if (__any_sync(0xffffffffu, key0 + kHalfKeys > lim)) {
#pragma unroll
                    for (int c = 0; c < kHalfKeys; ++c) x[c] = (key0 + c < lim) ? x[c] : NEG_INF;
                }
            };
            // weights p = 2^(x scale - ref) on pairs in place, with their sum
            // and sum of squares (the special-function unit has room for every
            // exponential of the tile)
            float psum = 0.f, psq = 0.f;
            auto weights = [&](float ref) {
                const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2), nref2 = f2_pack(-ref, -ref);
                uint64_t ps2[4] = {0, 0, 0, 0}, pq2[4] = {0, 0, 0, 0};
#pragma unroll
                for (int c = 0; c < kHalfKeys; c += 2) {
                    const uint64_t y2 = f2_fma(f2_pack(x[c], x[c + 1]), sc2, nref2);
                    float y0, y1;
                    f2_unpack(y2, y0, y1);
                    const uint64_t p2 = f2_pack(fast_exp2(y0), fast_exp2(y1));
                    ps2[(c >> 1) & 3] = f2_add(ps2[(c >> 1) & 3], p2);
                    pq2[(c >> 1) & 3] = f2_fma(p2, p2, pq2[(c >> 1) & 3]);
                    f2_unpack(p2, x[c], x[c + 1]);
                }
                float a0, a1, b0, b1;
                f2_unpack(f2_add(f2_add(ps2[0], ps2[1]), f2_add(ps2[2], ps2[3])), a0, a1);
                f2_unpack(f2_add(f2_add(pq2[0], pq2[1]), f2_add(pq2[2], pq2[3])), b0, b1);
                psum = a0 + a1;
                psq = b0 + b1;
            };
            load_scores();
            // this half's max (four chains of three-input maxima)
            float mx4[4] = {fmaxf(x[0], x[1]), fmaxf(x[2], x[3]), fmaxf(x[4], x[5]), fmaxf(x[6], x[7])};
#pragma unroll
            for (int c = 8; c < kHalfKeys; c += 8) {
                mx4[0] = fmax3(mx4[0], x[c], x[c + 1]);
                mx4[1] = fmax3(mx4[1], x[c + 2], x[c + 3]);
                mx4[2] = fmax3(mx4[2], x[c + 4], x[c + 5]);
                mx4[3] = fmax3(mx4[3], x[c + 6], x[c + 7]);
            }
            float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
            // post this half's max; while the other half's arrives, the weights
            // are computed against the current reference when it holds for
            // every row of this warp (the usual case after the first tile).
            // Rows past the request never see a key and keep a -inf reference;
            // a half that sees no key of a row has zero weights whatever the
            // reference becomes.  Every lane takes part in the vote.
            xmax[(sb * 2 + half) * kPrefillRows + row] = mx;
            post();
            const bool first = m_ref == NEG_INF;           // O holds nothing yet for this row
            const bool ready = first ? mx == NEG_INF : mx * p.scale_log2 <= m_ref + 8.f;
            const bool early = __all_sync(0xffffffffu, ready);
            if (early) weights(first ? 0.f : m_ref);
            ok = meet(j);
            if (!ok) break;
            mx = fmaxf(mx, xmax[(sb * 2 + (half ^ 1)) * kPrefillRows + row]);
            // log2-domain max (scale > 0 keeps the order of scores); both halves
            // take the same decisions from the same values
            const float m_new = fmaxf(m_ref, mx * p.scale_log2);
            const bool grow = !first && m_new > m_ref + 8.f;
            const float alpha = grow ? fast_exp2(m_ref - m_new) : 1.f;
            if (first || grow) m_ref = m_new;
            if (!early || __any_sync(0xffffffffu, grow)) {
                // the reference moved for some row of this warp: weights again
                // from this half's own S columns (no other warp writes them)
                tc_fence_after();
                load_scores();
                weights((m_ref == NEG_INF) ? 0.f : m_ref);
            }
            l = l * alpha + psum;
            // this warp's vote: does any of its rows need the remainder of P?
            // (half sums: if neither half's weights are concentrated, the row's
            // are not either)
            const bool need = j < p.lo_tiles || psq > kLoConcentration * l * l;
            const bool wneed = __any_sync(0xffffffffu, need);
            // P V of tile j-1 must be done before O is rescaled; the barrier of
            // tile j-2 (same parity) is waited every tile, which keeps each
            // barrier at most one phase ahead of this thread
            if (j >= 2) {
                ok = __all_sync(0xffffffffu, pf_wait(&bars[kODone0 + sb], ((j - 2) >> 1) & 1, status));
                if (!ok) break;
            }
            if (__any_sync(0xffffffffu, grow)) {              // rare: this half of O rescaled
                if (j >= 1) {
                    ok = __all_sync(0xffffffffu, pf_wait(&bars[kODone0 + (sb ^ 1)], ((j - 1) >> 1) & 1, status));
                    if (!ok) break;
                }
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < kHalfDims / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld32(trow + Cfg::kColO + half * kHalfDims + c * 32, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
                    tmem_st32(trow + Cfg::kColO + half * kHalfDims + c * 32, v);
                }
            }
            // P (bf16 pairs) of this half's keys into the tile's S buffer; the
            // remainder too when this warp asks for it, zeros otherwise
            {
                uint32_t w[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) w[e] = pack_bf16x2(x[2 * e], x[2 * e + 1]);
                tmem_st32(sbuf + half * 64, w);
                if (wneed) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const float a0 = x[2 * e], a1 = x[2 * e + 1];
                        const float2 hb = __bfloat1622float2(__floats2bfloat162_rn(a0, a1));
                        w[e] = pack_bf16x2(a0 - hb.x, a1 - hb.y);
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) w[e] = 0u;
                }
                tmem_st32(sbuf + half * 64 + 32, w);
            }
            tmem_st_wait();
            if (lane == 0) votes[(j & 1) * 8 + (warp - 4)] = wneed ? 1u : 0u;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[kPFull0 + (j & 1)]);
        }
        if (ok) {
            // epilogue: the last two P V, then O / l to bf16
            if (n_kv >= 2) ok = __all_sync(0xffffffffu, pf_wait(&bars[kODone0 + (n_kv & 1)], ((n_kv - 2) >> 1) & 1,
                                                                status));
            if (ok) ok = __all_sync(0xffffffffu, pf_wait(&bars[kODone0 + ((n_kv - 1) & 1)], ((n_kv - 1) >> 1) & 1,
                                                         status));
        }
        // the row's sum: this half's plus the other's
        if (ok) {
            xsum[half * kPrefillRows + row] = l;
            ok = exchange(n_kv);
            l += xsum[(half ^ 1) * kPrefillRows + row];
        }
        if (ok) {
            tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            uint32_t v[kHalfDims / 32][32];
#pragma unroll
            for (int c = 0; c < kHalfDims / 32; ++c) tmem_ld32(trow + Cfg::kColO + half * kHalfDims + c * 32, v[c]);
            tmem_ld_wait();
            if constexpr (CASCADE) {
                if (valid) {
                    // split `part` of the row: normalised partial output and natural log-sum-exp
                    const int4 ri = reinterpret_cast<const int4 *>(p.ws + hdr->off_req)[crow.y];
                    const int64_t prow =
                        ri.y + (static_cast<int64_t>(crow.z) * p.num_q_heads + g * G + hh) * ri.x + part;
                    float *po = reinterpret_cast<float *>(p.ws + hdr->off_part_o) + prow * HD + half * kHalfDims;
#pragma unroll
                    for (int c = 0; c < kHalfDims / 32; ++c)
#pragma unroll
                        for (int e = 0; e < 32; e += 4)
                            *reinterpret_cast<float4 *>(po + c * 32 + e) =
                                make_float4(__uint_as_float(v[c][e]) * inv, __uint_as_float(v[c][e + 1]) * inv,
                                            __uint_as_float(v[c][e + 2]) * inv, __uint_as_float(v[c][e + 3]) * inv);
                    if (half == 0)
                        reinterpret_cast<float *>(p.ws + hdr->off_part_lse)[prow] =
                            l > 0.f ? (m_ref + __log2f(l)) * 0.69314718055994531f : NEG_INF;
                }
            } else if (valid) {
                __nv_bfloat16 *dst =
                    p.out + (static_cast<int64_t>(tok) * p.num_q_heads + g * G + hh) * HD + half * kHalfDims;
#pragma unroll
                for (int c = 0; c < kHalfDims / 32; ++c)
#pragma unroll
                    for (int e = 0; e < 32; e += 8) {
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(v[c][e + 0]) * inv, __uint_as_float(v[c][e + 1]) * inv);
                        w.y = pack_bf16x2(__uint_as_float(v[c][e + 2]) * inv, __uint_as_float(v[c][e + 3]) * inv);
                        w.z = pack_bf16x2(__uint_as_float(v[c][e + 4]) * inv, __uint_as_float(v[c][e + 5]) * inv);
                        w.w = pack_bf16x2(__uint_as_float(v[c][e + 6]) * inv, __uint_as_float(v[c][e + 7]) * inv);
                        *reinterpret_cast<uint4 *>(dst + c * 32 + e) = w;
                    }
            }
        }
    }

    // teardown: every role is done with tensor memory
    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, Cfg::kTmemCols);
    }
}

// ---- host side --------------------------------------------------------------------

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
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

template <int HD, bool CASCADE>
static int launch_prefill_hd(const PrefillParams &p, const CUtensorMap &kvm, const void *query, int64_t q_stride,
                             int64_t grid, int dev, cudaStream_t stream) {
    using Cfg = PrefillCfg<HD>;
    static std::mutex mu;
    static uint64_t done_mask = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
        if (!bit || !(done_mask & bit)) {
            if (cudaFuncSetAttribute(prefill_kernel<HD, CASCADE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     Cfg::kSmem) != cudaSuccess)
                return PKV_ERR_CUDA;
            done_mask |= bit;
        }
    }
    if (launch_pdl(prefill_kernel<HD, CASCADE>, dim3(static_cast<unsigned>(grid)), dim3(384), Cfg::kSmem, stream,
                   kvm, static_cast<const __nv_bfloat16 *>(query), q_stride, p) != cudaSuccess)
        return PKV_ERR_CUDA;
    return PKV_OK;
}

static int make_page_map(CUtensorMap *kvm, const void *kv_cache, int64_t num_blocks, int32_t num_kv_heads,
                         int32_t head_size);

int launch_prefix(const PrefillParams &p, const void *query, int64_t q_stride, const void *kv_cache,
                  int64_t num_blocks, int32_t head_size, int64_t grid, int dev, cudaStream_t stream) {
    if (grid <= 0) return PKV_OK;
    CUtensorMap kvm;
    const int rc = make_page_map(&kvm, kv_cache, num_blocks, p.num_kv_heads, head_size);
    if (rc) return rc;
    if (head_size == 64) return launch_prefill_hd<64, true>(p, kvm, query, q_stride, grid, dev, stream);
    return launch_prefill_hd<128, true>(p, kvm, query, q_stride, grid, dev, stream);
}

int launch_prefill(const PrefillParams &p, const void *query, int64_t q_stride, int32_t num_tokens,
                   const void *kv_cache, int64_t num_blocks, int32_t head_size, int64_t grid, int dev,
                   cudaStream_t stream) {
    (void)num_tokens;
    if (grid <= 0) return PKV_OK;
    CUtensorMap kvm;
    const int rc = make_page_map(&kvm, kv_cache, num_blocks, p.num_kv_heads, head_size);
    if (rc) return rc;
    if (head_size == 64) return launch_prefill_hd<64, false>(p, kvm, query, q_stride, grid, dev, stream);
    return launch_prefill_hd<128, false>(p, kvm, query, q_stride, grid, dev, stream);
}

// Tensor map of the cache as {head_size, 16, 2, kv heads, blocks}; a box is
// the K (or V) rows of one page, 64 columns, 128-byte swizzle.
static int make_page_map(CUtensorMap *kvm, const void *kv_cache, int64_t num_blocks, int32_t num_kv_heads,
                         int32_t head_size) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return PKV_ERR_CUDA;
    const cuuint64_t dims[5] = {static_cast<cuuint64_t>(head_size), kBlock, 2, static_cast<cuuint64_t>(num_kv_heads),
                                static_cast<cuuint64_t>(num_blocks)};
    const cuuint64_t row = static_cast<cuuint64_t>(head_size) * 2;
    const cuuint64_t strides[4] = {row, row * kBlock, row * kBlock * 2, row * kBlock * 2 * num_kv_heads};
    const cuuint32_t box[5] = {64, kBlock, 1, 1, 1};
    const cuuint32_t es[5] = {1, 1, 1, 1, 1};
    if (enc(kvm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(kv_cache), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return PKV_ERR_CUDA;
    return PKV_OK;
}

}  // namespace pkv
