// Prefill-chunk paged attention over an E4M3 (8-bit) KV cache, on the
// 5th-generation tensor cores (tcgen05).  (The 16-bit cache has its own
// kernel, in prefill_sk.cu.)
//
// The same computation as the decode path ("continuous batching and
// PagedAttention" tutorial, section 3.6: loop over the request's blocks
// through its block table, accumulate softmax(QK^T)V), for requests whose
// rows are many: a chunk of a chunked prefill ("Inside vLLM: Anatomy of a
// High-Throughput LLM Inference System", chunked prefill; "vLLM internals:
// managing the KV cache like an OS manages memory", section 3.2) attends
// causally, query i of the chunk seeing keys 0 .. context + i.
//
// Work item: one 128-row tile for one kv head; a persistent CTA per SM
// takes items largest first from a shared counter.  Rows are
// (query token, q head of the GQA group) pairs, so one K/V tile in shared
// memory serves every q head of the group.  Per 128-key KV tile:
//   widen          the tile's raw E4M3 pages (TMA, one box per page and
//                  lane) are widened to f16 (exactly) by warps 2, 3, 12 and
//                  13 into a 16-bit ring, 128-byte swizzled
//   S = Q K^T      tcgen05.mma kind::f16, A = Q from tensor memory, B = K
//                  from shared memory (K-major), D in tensor memory (two S
//                  buffers)
//   softmax        two threads per row, each with half of the tile's keys,
//                  read S from tensor memory, mask, share their row maxima
//                  through shared memory, keep a running max (rescaling
//                  their half of O only when the max grows by more than 2^8)
//                  and write P (f16) over S
//   O += P V       tcgen05.mma, A = P from tensor memory, B = V (MN-major)
//                  from shared memory, D = O in tensor memory
// Both operands of a kind::f16 product share their type, so Q rows are
// scaled by a power of two into f16 and P is f16; k_scale enters the score
// factor and v_scale the epilogue.
// Warp roles: warp 0 loads, warp 1 issues the MMAs, warp 2 owns the
// tensor-memory allocation, warps 2, 3, 12 and 13 widen, warps 4-11 do
// softmax and the epilogue.
//
// When any row of the tile puts a large share of its weight on few keys of
// a KV tile (rows with few visible keys, or a peaked softmax), that tile's P
// also enters P V as its 16-bit remainder (a second MMA), keeping ~16 bits
// per weight; other tiles' weights are each small and one 16-bit P is
// enough.  V rows past the sequence end in its last page are zeroed before
// P V, so NaN in unwritten cache slots never meets a zero weight.  Every
// wait is bounded.
#include <mutex>

#include "prefill_common.cuh"

namespace pkv {

// Shared memory: the 16-bit K and V rings the MMAs read, the raw E4M3 ring
// the pages land in, barriers, the softmax exchange and the work items.
template <int HD>
struct PrefillCfg {
    static constexpr int kHalves = HD / 64;
    static constexpr int kStages = HD == 128 ? 2 : 3;          // 16-bit K and V ring depth
    static constexpr int kKVBytes = kHalves * kPrefillKeys * 128;   // one K (or V) tile
    static constexpr int kRawStages = 2;                     // raw E4M3 ring depth
    static constexpr int kRawBytes = kPrefillKeys * HD;      // one raw K (or V) tile
    static constexpr int kOffK = 0;
    static constexpr int kOffV = kOffK + kStages * kKVBytes;
    static constexpr int kOffRaw = kOffV + kStages * kKVBytes;
    static constexpr int kOffBar = kOffRaw + kRawStages * 2 * kRawBytes;
    static constexpr int kOffXchg = kOffBar + 512;            // softmax halves' maxima, sums, Q maxima (4 KiB)
    static constexpr int kOffItems = kOffXchg + 4096;         // ring of work items (256 bytes)
    static constexpr int kSmem = kOffItems + 256 + 1024;      // + alignment slack
    // tensor memory: two S buffers (each later holding that tile's P and its
    // f16 remainder), O, and Q as the A operand of S = Q K^T
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256, kColQ = 384;
};

enum PrefillBar { kQFull = 0, kKFull0, kKFull1, kKFull2, kVFull0, kVFull1, kVFull2, kKEmpty0, kKEmpty1, kKEmpty2,
                  kVEmpty0, kVEmpty1, kVEmpty2, kSFull0, kSFull1, kPFull0, kPFull1, kODone0, kODone1,
                  kVFix0, kVFix1, kVFix2,              // V rows past the sequence end zeroed, per stage
                  kXchg0, kXchg1, kXchg2, kXchg3,      // the two softmax warps of a lane quadrant
                  kItemFull0, kItemFull1, kItemFull2, kItemFull3,      // work-item ring
                  kItemEmpty0, kItemEmpty1, kItemEmpty2, kItemEmpty3,
                  kOFree,                              // O read out by the epilogue
                  kRFull0, kRFull1, kREmpty0, kREmpty1,  // raw E4M3 tiles
                  kNumBars };
static_assert(kNumBars * 8 + 16 + 64 <= 512, "barriers, the TMEM address slot and the votes fit their 512 bytes");
// P of tile j is announced on kPFull0 + (j & 1): with one barrier per parity a
// barrier never runs two phases ahead of the MMA thread's wait on it (the
// softmax warps can finish tile j + 1 before the MMA thread looks at tile j).


// Persistent: one CTA per SM.  The CTA's first item is its index; each later
// one is claimed from a counter the plan zeroes, in the plan's order
// (largest first).  The producer warp claims and decodes items and publishes
// them through a ring in shared memory; tiles and their barriers are counted
// across items, so the loads, the first products and the Q of the next item
// overlap the epilogue of the current one.
template <int HD, bool CASCADE>
__global__ void __launch_bounds__(448, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap kv_map, const __nv_bfloat16 *__restrict__ query,
                   const int64_t q_stride, const PrefillParams p) {
    using Cfg = PrefillCfg<HD>;
    constexpr int S = Cfg::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg::kOffBar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + kNumBars);
    volatile uint32_t *votes = tmem_slot + 4;          // [2 tiles in flight][8 softmax warps]
    volatile PfItem *items = reinterpret_cast<volatile PfItem *>(smem + Cfg::kOffItems);
    const uint32_t sK = smem_u32(smem + Cfg::kOffK);
    const uint32_t sV = smem_u32(smem + Cfg::kOffV);

    // The kernel launched just before this one (the decode kernel, or the
    // shared-prefix pass) may still be running: it writes other rows and other
    // splits than this kernel, and it started only after the plan (and the
    // cache write before the plan) had completed.  So the plan's lists are read
    // at once, through L2 (ws_ld), and the wait on that kernel comes at the
    // end, so that this grid completes after it and the combine sees both.
    pdl_trigger();
    const WsHeader *hdr = reinterpret_cast<const WsHeader *>(p.ws);
    int32_t *status = reinterpret_cast<int32_t *>(p.ws);
    const int n_parts = CASCADE ? ws_ld(&hdr->prefix_parts) : 1;
    const int n_tiles = CASCADE ? (ws_ld(&hdr->n_crows) + kPrefillRows - 1) / kPrefillRows : ws_ld(&hdr->n_ptiles);
    const int n_items = n_tiles * p.num_kv_heads * n_parts;
    if (static_cast<int>(blockIdx.x) >= n_items) {            // uniform over the CTA
        pdl_wait();
        return;
    }
    const int G = p.G;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // one barrier per thread: an mbarrier.init takes over a hundred cycles, and
    // one thread initialising all of them in turn held every CTA several us
    if (threadIdx.x < kNumBars) {
        const int b = threadIdx.x;
        int count = 1;
        if (b == kPFull0 || b == kPFull1 || b == kQFull || b == kOFree) count = 8;
        else if (b >= kXchg0 && b <= kXchg3) count = 2;
        else if (b >= kItemEmpty0 && b < kItemEmpty0 + kItemSlots) count = 13;   // MMA, softmax, converters
        else if (b == kREmpty0 || b == kREmpty1) count = 4;      // every converter warp
        else if ((b == kKFull0 || b == kKFull1 || b == kKFull2 || b == kVFull0 || b == kVFull1 ||
                         b == kVFull2 || b == kVFix0 || b == kVFix1 || b == kVFix2))
            count = 2;                                           // the two converters of K (of V)
        mbar_init(&bars[b], count);
    }
    if (threadIdx.x == 0) tma_prefetch_desc(&kv_map);
    if (warp == 2) {
        tmem_alloc(tmem_slot, Cfg::kTmemCols);
        tmem_relinquish();
    }
    fence_barrier_init();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // the item's KV tile holding the sequence's last key, when that page is partial
    auto end_tile_of = [](int L) { return (!CASCADE && (L % kBlock)) ? (L - 1) / kPrefillKeys : -1; };

    if (warp == 0) {
        // ---------------- producer: items, then K and V pages through the block table ----------------
        bool ok = true;
        int item = blockIdx.x;
        int gj = 0;                                    // KV tiles of this CTA so far (ring position)
        int taken = 0;                                 // items of this CTA
        int *next_item = reinterpret_cast<int *>(p.ws + (CASCADE ? offsetof(WsHeader, next_prefix_item)
                                                                  : offsetof(WsHeader, next_ptile_item)));
        for (int k = 0; ok; ++k) {
            const int slot = k % kItemSlots;
            // the slot's previous item has been read by the MMA thread and every softmax warp
            if (k >= kItemSlots)
                ok = __all_sync(0xffffffffu, pf_wait(&bars[kItemEmpty0 + slot], (k / kItemSlots - 1) & 1, status));
            if (!ok) break;
            PfItem it{};
            if (item < n_items) {
                it.valid = 1;
                it.g = item % p.num_kv_heads;
                if constexpr (CASCADE) {
                    it.r = 0;                          // the prefix blocks are read through request 0's table
                    it.L = ws_ld(&hdr->prefix_blocks) * kBlock;
                    const int kv_all = (it.L + kPrefillKeys - 1) / kPrefillKeys;
                    const int per = (kv_all + n_parts - 1) / n_parts;   // the plan makes every range non-empty
                    it.part = (item / p.num_kv_heads) % n_parts;
                    it.t0 = it.part * per;
                    it.n_kv = min(kv_all, it.t0 + per) - it.t0;
                    it.n_pages = ws_ld(&hdr->prefix_blocks);
                    it.rows_total = ws_ld(&hdr->n_crows);
                    it.row0 = (item / (p.num_kv_heads * n_parts)) * kPrefillRows;
                } else {
                    const int4 tile =
                        ws_ld(reinterpret_cast<const int4 *>(p.ws + ws_ld(&hdr->off_ptiles)) + item / p.num_kv_heads);
                    it.r = tile.x;
                    it.n_kv = tile.z;
                    it.L = p.seq_lens[it.r];
                    it.qs = p.qsl[it.r];
                    const int qlen = p.qsl[it.r + 1] - it.qs;
                    it.ctx = it.L - qlen;
                    it.rows_total = qlen * G;
                    it.row0 = tile.y * kPrefillRows;
                    it.n_pages = (it.L + kBlock - 1) / kBlock;
                }
            }
            if (lane == 0) {
                volatile int32_t *dst = reinterpret_cast<volatile int32_t *>(items + slot);
                const int32_t *src = reinterpret_cast<const int32_t *>(&it);
#pragma unroll
                for (int e = 0; e < static_cast<int>(sizeof(PfItem) / 4); ++e) dst[e] = src[e];
                mbar_arrive(&bars[kItemFull0 + slot]);
            }
            if (!it.valid) break;
            ++taken;

            const int32_t *bt = p.block_tables + static_cast<int64_t>(it.r) * p.max_blocks_per_seq;
            // block ids in windows of 32 pages (4 KV tiles), one lane per page; the
            // next window is loaded a window ahead.  Pages past the sequence are -1
            // and load as zeros (outside the tensor map).
            constexpr int kPagesPerTile = kPrefillKeys / kBlock;
            auto load_window = [&](int w) -> int {
                const int page = it.t0 * kPagesPerTile + w * 32 + lane;
                const int b = page < it.n_pages ? __ldg(bt + page) : -1;
                if (page < it.n_pages && (b < 0 || b >= p.num_blocks))
                    set_status(status, PKV_ERR_DEVICE_INDEX);   // loaded as zeros by the bounded TMA, reported
                return b;
            };
            int win_cur = load_window(0);
            int win_next = load_window(1);
            for (int j = 0; j < it.n_kv && ok; ++j) {
                const int gt = gj + j;
                if (j > 0 && (j * kPagesPerTile) % 32 == 0) {
                    win_cur = win_next;
                    win_next = load_window(j * kPagesPerTile / 32 + 1);
                }
                const int wofs = (j * kPagesPerTile) % 32;
                // the raw K and V pages of tile gt, once the converters are done
                // with tile gt - 2 (zeroing past the sequence end is theirs)
                const int rs = gt % Cfg::kRawStages;
                if (gt >= Cfg::kRawStages)
                    ok = __all_sync(0xffffffffu, pf_wait(&bars[kREmpty0 + rs],
                                                         ((gt - Cfg::kRawStages) / Cfg::kRawStages) & 1, status));
                if (!ok) break;
                // one box per lane (lanes 0-7 the K rows of page lane, 8-15 the V
                // rows of page lane - 8): the copy engine takes small boxes faster
                // from many issuing lanes than from one
                uint8_t *raw = smem + Cfg::kOffRaw + rs * 2 * Cfg::kRawBytes;
                if (lane == 0) mbar_arrive_expect_tx(&bars[kRFull0 + rs], 2 * Cfg::kRawBytes);
                __syncwarp();
                const int my_blk = __shfl_sync(0xffffffffu, win_cur, wofs + (lane % kPagesPerTile));
                if (lane < 2 * kPagesPerTile) {
                    const int kv = lane / kPagesPerTile, pg = lane % kPagesPerTile;
                    tma_load_5d(raw + kv * Cfg::kRawBytes + pg * kBlock * HD, &kv_map, &bars[kRFull0 + rs], 0, 0, kv,
                                it.g, my_blk);
                }
            }
            gj += it.n_kv;
            int nxt = 0;
            if (lane == 0) nxt = static_cast<int>(gridDim.x) + atomicAdd(next_item, 1);
            item = __shfl_sync(0xffffffffu, nxt, 0);
        }
        // this CTA's share of the schedule
        if (lane == 0)
            reinterpret_cast<int32_t *>(p.ws + kStatsOffset)[(CASCADE ? kStatsCtas : 0) + blockIdx.x] = taken;
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t kIdescS = idesc_f16_f32(kPrefillRows, kPrefillKeys, 0, 0);
            constexpr uint32_t kIdescO = idesc_f16_f32(kPrefillRows, HD, 0, 1);
            // S(gt) = Q K^T into S buffer gt & 1; A = Q in tensor memory
            auto issue_s = [&](int gt) {
                const int st = gt % S;
                const uint32_t d = tmem + ((gt & 1) ? Cfg::kColS1 : Cfg::kColS0);
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const uint64_t b = smem_desc_sw128(sK + st * Cfg::kKVBytes + (kk >> 2) * (kPrefillKeys * 128) +
                                                           (kk & 3) * 32,
                                                       16, 1024);
                    umma_f16_ts(d, tmem + Cfg::kColQ + kk * 8, b, kIdescS, kk > 0);
                }
                umma_commit(&bars[kSFull0 + (gt & 1)]);
                umma_commit(&bars[kKEmpty0 + st]);
            };
            // O (+)= P V; A = P (or its remainder) in S buffer gt & 1: keys
            // 64 h .. 64 h + 63 sit at columns 64 h + [0, 32) (P) and
            // 64 h + [32, 64) (remainder), each half within its own S columns
            auto issue_pv = [&](int gt, uint32_t pcol, uint32_t accumulate) {
                const int st = gt % S;
#pragma unroll
                for (int kk = 0; kk < kPrefillKeys / 16; ++kk) {
                    const uint64_t b = smem_desc_sw128(sV + st * Cfg::kKVBytes + kk * 2048, kPrefillKeys * 128, 1024);
                    umma_f16_ts(tmem + Cfg::kColO, pcol + kk * 8 + (kk >> 2) * 32, b, kIdescO,
                                 (accumulate || kk > 0) ? 1u : 0u);
                }
            };
            bool ok = true;
            int gj = 0;
            uint32_t vfix_par = 0;                     // phase parity of each stage's fix barrier
            for (int k = 0; ok; ++k) {
                const int slot = k % kItemSlots;
                ok = pf_wait(&bars[kItemFull0 + slot], (k / kItemSlots) & 1, status);
                if (!ok) break;
                const bool valid = items[slot].valid != 0;
                const int n_kv = items[slot].n_kv;
                const int end_tile = end_tile_of(items[slot].L);
                mbar_arrive(&bars[kItemEmpty0 + slot]);
                if (!valid) break;
                // Q of this item in tensor memory (written by the softmax warps)
                ok = pf_wait(&bars[kQFull], k & 1, status);
                for (int j0 = 0; j0 < 2 && j0 < n_kv && ok; ++j0) {
                    const int gt = gj + j0;
                    // S buffer gt & 1 is free once P V of tile gt-2 has read its P
                    if (gt >= 2) ok = pf_wait(&bars[kODone0 + (gt & 1)], ((gt - 2) >> 1) & 1, status);
                    if (ok) ok = pf_wait(&bars[kKFull0 + gt % S], (gt / S) & 1, status);
                    if (!ok) break;
                    tc_fence_after();
                    issue_s(gt);
                }
                for (int j = 0; j < n_kv && ok; ++j) {
                    const int gt = gj + j;
                    const int st = gt % S;
                    ok = pf_wait(&bars[kPFull0 + (gt & 1)], (gt >> 1) & 1, status);
                    if (ok) ok = pf_wait(&bars[kVFull0 + st], (gt / S) & 1, status);
                    if (ok && j == end_tile) {
                        ok = pf_wait(&bars[kVFix0 + st], (vfix_par >> st) & 1u, status);
                        vfix_par ^= 1u << st;
                    }
                    // the previous item's O has been read out by its epilogue
                    if (ok && j == 0 && k > 0) ok = pf_wait(&bars[kOFree], (k - 1) & 1, status);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t pbuf = tmem + ((gt & 1) ? Cfg::kColS1 : Cfg::kColS0);
                    uint32_t vote = 0;
#pragma unroll
                    for (int w = 0; w < 8; ++w) vote |= votes[(gt & 1) * 8 + w];
                    const bool lo = vote != 0u;
                    issue_pv(gt, pbuf, j > 0);
                    if (lo) issue_pv(gt, pbuf + 32, 1);
                    umma_commit(&bars[kODone0 + (gt & 1)]);
                    umma_commit(&bars[kVEmpty0 + st]);
                    // S of tile gt+2 overwrites S buffer gt & 1, where P V of tile gt
                    // reads P: it is issued only once that product has completed (no
                    // overlap of a tensor-memory operand read with a later write)
                    if (j + 2 < n_kv) {
                        ok = pf_wait(&bars[kODone0 + (gt & 1)], (gt >> 1) & 1, status);
                        if (ok) ok = pf_wait(&bars[kKFull0 + (gt + 2) % S], ((gt + 2) / S) & 1, status);
                        if (!ok) break;
                        tc_fence_after();
                        issue_s(gt + 2);
                    }
                }
                gj += n_kv;
            }
        }
        __syncwarp();
    } else if (warp == 2 || warp == 3 || warp >= 12) {
        // ---------------- converters (E4M3 cache): raw tiles -> f16 tiles ----------------
        // warps 2 and 12 widen K, 3 and 13 widen V (and zero V rows past the
        // sequence end: their scores are masked, but NaN times a zero weight
        // is NaN); warps 2 and 3 take the tile's first 64 keys, 12 and 13 the
        // rest.  They sit on four different schedulers.
        const bool isv = (warp & 1) != 0;
        const int row0 = warp >= 12 ? kPrefillKeys / 2 : 0;
        bool ok = true;
        int gj = 0;
        for (int k = 0; ok; ++k) {
            const int slot = k % kItemSlots;
            ok = __all_sync(0xffffffffu, pf_wait(&bars[kItemFull0 + slot], (k / kItemSlots) & 1, status));
            if (!ok) break;
            const bool valid = items[slot].valid != 0;
            const int n_kv = items[slot].n_kv;
            const int L = items[slot].L;
            const int t0 = items[slot].t0;
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[kItemEmpty0 + slot]);
            if (!valid) break;
            const int end_tile = end_tile_of(L);
            for (int j = 0; j < n_kv && ok; ++j) {
                const int gt = gj + j;
                const int st = gt % S, rs = gt % Cfg::kRawStages;
                ok = __all_sync(0xffffffffu, pf_wait(&bars[kRFull0 + rs], (gt / Cfg::kRawStages) & 1, status));
                if (ok && gt >= S)
                    ok = __all_sync(0xffffffffu,
                                    pf_wait(&bars[(isv ? kVEmpty0 : kKEmpty0) + st], ((gt - S) / S) & 1, status));
                if (!ok) break;
                const uint32_t src =
                    smem_u32(smem + Cfg::kOffRaw + rs * 2 * Cfg::kRawBytes + (isv ? Cfg::kRawBytes : 0));
                const uint32_t dst = (isv ? sV : sK) + st * Cfg::kKVBytes;
                const int zero_from = (isv && j == end_tile) ? L - (t0 + j) * kPrefillKeys : kPrefillKeys;
                // 16-element pieces: raw row r bytes 16c .. 16c + 15 -> 16-bit tile row r,
                // 64-column box c / 4, 16-byte chunks 2c % 8 and 2c % 8 + 1 at their
                // 128-byte-swizzle places
                constexpr int kPieces = kPrefillKeys / 2 * HD / 16;      // this warp's half of the rows
#pragma unroll 4
                for (int u = lane; u < kPieces; u += 32) {
                    const int r = row0 + u / (HD / 16), c = u % (HD / 16);
                    uint32_t w[4];
                    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                                 : "r"(src + r * HD + c * 16));
                    uint32_t h[8];
#pragma unroll
                    for (int e = 0; e < 4; ++e) e4m3x4_to_f16x4(w[e], h[2 * e], h[2 * e + 1]);
                    if (r >= zero_from) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) h[e] = 0u;
                    }
                    const uint32_t row = dst + (c >> 2) * (kPrefillKeys * 128) + r * 128;
                    const int c0 = (2 * c) & 7;
                    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(row + ((c0 ^ (r & 7)) << 4)),
                                 "r"(h[0]), "r"(h[1]), "r"(h[2]), "r"(h[3])
                                 : "memory");
                    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(row + (((c0 + 1) ^ (r & 7)) << 4)),
                                 "r"(h[4]), "r"(h[5]), "r"(h[6]), "r"(h[7])
                                 : "memory");
                }
                fence_proxy_async_smem();              // for the tensor core, and before the raw stage refills
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&bars[(isv ? kVFull0 : kKFull0) + st]);
                    if (isv && j == end_tile) mbar_arrive(&bars[kVFix0 + st]);
                    mbar_arrive(&bars[kREmpty0 + rs]);
                }
            }
            gj += n_kv;
        }
    } else if (warp >= 4 && warp < 12) {
        // ---------------- softmax + epilogue: two threads per row ----------------
        // warps 4-7 take keys (and output columns) of the first half of the tile,
        // warps 8-11 the second half; warp w reads tensor-memory lanes of quadrant
        // w % 4, so warps w and w + 4 share their 32 rows
        const int quad = warp & 3;
        const int half = (warp - 4) >> 2;
        const int row = quad * 32 + lane;
        const float NEG_INF = -__int_as_float(0x7f800000);
        const uint32_t trow = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        constexpr int kHalfKeys = kPrefillKeys / 2;        // keys of a tile per thread
        constexpr int kHalfDims = HD / 2;                   // output columns per thread
        // exchange of the two halves' row maxima (by tile parity) and final sums
        float *xmax = reinterpret_cast<float *>(smem + Cfg::kOffXchg);          // [2][2][128]
        float *xsum = xmax + 2 * 2 * kPrefillRows;                               // [2][128]
        float *xq = xsum + 2 * kPrefillRows;                                     // [2][128] (E4M3: Q maxima)
        // the two warps of this quadrant meet on an mbarrier, one phase per
        // tile plus one per item for the final sums (bounded waits, like every other)
        uint64_t *xbar = &bars[kXchg0 + quad];
        int xph = 0;
        auto post = [&]() {
            __syncwarp();
            if (lane == 0) mbar_arrive(xbar);
        };
        auto meet = [&]() -> bool {
            const bool done = __all_sync(0xffffffffu, pf_wait(xbar, xph & 1, status));
            ++xph;
            return done;
        };
        bool ok = true;

        // this thread's row of an item (read from the item's ring slot): query
        // token, q head within the group, keys [0, lim) visible; cascade rows
        // {token, request, index, head}
        struct RowInfo {
            int tok, hh, lim;
            bool valid;
            int4 crow;
        };
        auto row_info = [&](const volatile PfItem *it) -> RowInfo {
            RowInfo ri{0, 0, 0, false, make_int4(0, 0, 0, 0)};
            const int rrow = it->row0 + row;
            ri.valid = rrow < it->rows_total;
            if (ri.valid) {
                if constexpr (CASCADE) {
                    ri.crow = ws_ld(reinterpret_cast<const int4 *>(p.ws + ws_ld(&hdr->off_crows)) + rrow);
                    ri.tok = ri.crow.x;
                    ri.hh = ri.crow.w;
                    ri.lim = it->L;
                } else {
                    ri.tok = it->qs + rrow / G;
                    ri.hh = rrow % G;
                    ri.lim = it->ctx + rrow / G + 1;
                }
            }
            return ri;
        };
        // item k of this CTA: its ring slot once published; the slot is
        // released after the item's epilogue (every lane reads it meanwhile)
        auto wait_item = [&](int k) -> bool {
            return __all_sync(0xffffffffu,
                              pf_wait(&bars[kItemFull0 + k % kItemSlots], (k / kItemSlots) & 1, status));
        };
        auto release_item = [&](int k) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[kItemEmpty0 + k % kItemSlots]);
        };
        // score factor of this thread's row (log2 domain): the scale; over an
        // E4M3 cache also k_scale and the power of two that brought Q into f16
        float sl2 = p.scale_log2;
        // this half of the item's Q row -> tensor memory (A operand of S = Q K^T),
        // zeros past the request
        auto load_q = [&](const volatile PfItem *it) {
            const RowInfo ri = row_info(it);
            uint32_t qv[kHalfDims / 2];
            const __nv_bfloat16 *qp = query + static_cast<int64_t>(ri.tok) * q_stride +
                                      static_cast<int64_t>(it->g * G + ri.hh) * HD + half * kHalfDims;
#pragma unroll
            for (int c = 0; c < kHalfDims / 8; ++c) {
                const uint4 w = ri.valid ? __ldg(reinterpret_cast<const uint4 *>(qp) + c) : make_uint4(0, 0, 0, 0);
                qv[4 * c + 0] = w.x;
                qv[4 * c + 1] = w.y;
                qv[4 * c + 2] = w.z;
                qv[4 * c + 3] = w.w;
            }
            // the row scaled by 2^e into [2^14, 2^15) before rounding to f16 (exact
            // but for parts below 2^-24 of its largest); the two halves agree on e
            float a = 0.f;
#pragma unroll
            for (int e = 0; e < kHalfDims / 2; ++e)
                a = fmaxf(a, fmaxf(fabsf(__uint_as_float(qv[e] << 16)), fabsf(__uint_as_float(qv[e] & 0xFFFF0000u))));
            xq[half * kPrefillRows + row] = a;
            post();
            if (!meet()) a = 0.f;                  // timed out: the status says so
            a = fmaxf(a, xq[(half ^ 1) * kPrefillRows + row]);
            const int ex = a > 0.f ? min(126, max(-114, 14 - ilogbf(a))) : 0;
            const float u = __int_as_float((ex + 127) << 23);
#pragma unroll
            for (int e = 0; e < kHalfDims / 2; ++e) {
                const __half2 h = __floats2half2_rn(__uint_as_float(qv[e] << 16) * u,
                                                    __uint_as_float(qv[e] & 0xFFFF0000u) * u);
                qv[e] = *reinterpret_cast<const uint32_t *>(&h);
            }
            sl2 = p.scale_log2 * p.k_scale * __int_as_float((127 - ex) << 23);
            if constexpr (kHalfDims / 2 == 32) {
                tmem_st32(trow + Cfg::kColQ + half * 32, qv);
            } else {
                tmem_st16(trow + Cfg::kColQ + half * 16, qv);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[kQFull]);
        };

        ok = wait_item(0);
        if (ok && items[0].valid) load_q(items);
        int gj = 0;                                        // KV tiles of this CTA so far
        int k = 0;
        for (; ok && items[k % kItemSlots].valid; ++k) {
            const volatile PfItem *cur = items + k % kItemSlots;
            const int n_kv = cur->n_kv;
            const int kbase = cur->t0 * kPrefillKeys + half * kHalfKeys;
            // where this row's result goes (-1: nowhere): element offset in out,
            // or the partial row of split `part` (cascade)
            int64_t dst = -1;
            int lim = 0;
            {
                const RowInfo ri = row_info(cur);
                lim = ri.lim;
                if (ri.valid) {
                    if constexpr (CASCADE) {
                        const int4 rq = ws_ld(reinterpret_cast<const int4 *>(p.ws + ws_ld(&hdr->off_req)) + ri.crow.y);
                        dst = rq.y + (static_cast<int64_t>(ri.crow.z) * p.num_q_heads + cur->g * G + ri.hh) * rq.x +
                              cur->part;
                    } else {
                        dst = (static_cast<int64_t>(ri.tok) * p.num_q_heads + cur->g * G + ri.hh) * HD +
                              half * kHalfDims;
                    }
                }
            }
            float m_ref = NEG_INF, l = 0.f;                // l: this half's sum
            for (int j = 0; j < n_kv && ok; ++j) {
                const int gt = gj + j;
                const int sb = gt & 1;
                const uint32_t sbuf = trow + (sb ? Cfg::kColS1 : Cfg::kColS0);
                ok = __all_sync(0xffffffffu, pf_wait(&bars[kSFull0 + sb], (gt >> 1) & 1, status));
                if (!ok) break;
                tc_fence_after();
                // this half's scores (keys key0 .. key0 + 63); keys a row may not see
                // become -inf, tested only in tiles reaching some row's limit
                const int key0 = kbase + j * kPrefillKeys;
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
                    const uint64_t sc2 = f2_pack(sl2, sl2), nref2 = f2_pack(-ref, -ref);
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
                const bool first = m_ref == NEG_INF;       // O holds nothing yet for this row
                const bool ready = first ? mx == NEG_INF : mx * sl2 <= m_ref + 8.f;
                const bool early = __all_sync(0xffffffffu, ready);
                if (early) weights(first ? 0.f : m_ref);
                ok = meet();
                if (!ok) break;
                mx = fmaxf(mx, xmax[(sb * 2 + (half ^ 1)) * kPrefillRows + row]);
                // log2-domain max (scale > 0 keeps the order of scores); both halves
                // take the same decisions from the same values
                const float m_new = fmaxf(m_ref, mx * sl2);
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
                // P V of tile gt-1 must be done before O is rescaled; the barrier of
                // tile gt-2 (same parity) is waited every tile, which keeps each
                // barrier at most one phase ahead of this thread
                if (gt >= 2) {
                    ok = __all_sync(0xffffffffu, pf_wait(&bars[kODone0 + sb], ((gt - 2) >> 1) & 1, status));
                    if (!ok) break;
                }
                if (__any_sync(0xffffffffu, grow)) {          // rare: this half of O rescaled
                    // grow needs an earlier tile of this item, so j >= 1
                    ok = __all_sync(0xffffffffu, pf_wait(&bars[kODone0 + (sb ^ 1)], ((gt - 1) >> 1) & 1, status));
                    if (!ok) break;
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
                // P (f16 pairs) of this half's keys into the tile's S buffer; the
                // remainder too when this warp asks for it, zeros otherwise
                // (16 columns at a time: fewer registers live)
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t w[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) w[e] = pack_p<true>(x[32 * c + 2 * e], x[32 * c + 2 * e + 1]);
                    tmem_st16(sbuf + half * 64 + 16 * c, w);
                    if (wneed) {
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            w[e] = pack_p_rest<true>(x[32 * c + 2 * e], x[32 * c + 2 * e + 1]);
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 16; ++e) w[e] = 0u;
                    }
                    tmem_st16(sbuf + half * 64 + 32 + 16 * c, w);
                }
                tmem_st_wait();
                if (lane == 0) votes[sb * 8 + (warp - 4)] = wneed ? 1u : 0u;
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[kPFull0 + sb]);
            }
            gj += n_kv;
            // the next item's Q right away: every S of this item has completed
            if (ok) ok = wait_item(k + 1);
            if (ok && items[(k + 1) % kItemSlots].valid) load_q(items + (k + 1) % kItemSlots);
            if (ok) {
                // epilogue: the last two P V, then O / l
                if (n_kv >= 2)
                    ok = __all_sync(0xffffffffu, pf_wait(&bars[kODone0 + (gj & 1)], ((gj - 2) >> 1) & 1, status));
                if (ok)
                    ok = __all_sync(0xffffffffu, pf_wait(&bars[kODone0 + ((gj - 1) & 1)], ((gj - 1) >> 1) & 1, status));
            }
            // the row's sum: this half's plus the other's
            if (ok) {
                xsum[half * kPrefillRows + row] = l;
                post();
                ok = meet();
                l += xsum[(half ^ 1) * kPrefillRows + row];
            }
            if (ok) {
                tc_fence_after();
                const float inv = l > 0.f ? p.v_scale / l : 0.f;   // E4M3: V is code * v_scale
                uint32_t v[kHalfDims / 32][32];
#pragma unroll
                for (int c = 0; c < kHalfDims / 32; ++c) tmem_ld32(trow + Cfg::kColO + half * kHalfDims + c * 32, v[c]);
                tmem_ld_wait();
                // O is in registers: the next item's first P V may overwrite it
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[kOFree]);
                if (dst >= 0) {
                    if constexpr (CASCADE) {
                        // split `part` of the row: normalised partial output and natural log-sum-exp
                        float *po = reinterpret_cast<float *>(p.ws + ws_ld(&hdr->off_part_o)) + dst * HD + half * kHalfDims;
#pragma unroll
                        for (int c = 0; c < kHalfDims / 32; ++c)
#pragma unroll
                            for (int e = 0; e < 32; e += 4)
                                *reinterpret_cast<float4 *>(po + c * 32 + e) =
                                    make_float4(__uint_as_float(v[c][e]) * inv, __uint_as_float(v[c][e + 1]) * inv,
                                                __uint_as_float(v[c][e + 2]) * inv, __uint_as_float(v[c][e + 3]) * inv);
                        if (half == 0)
                            reinterpret_cast<float *>(p.ws + ws_ld(&hdr->off_part_lse))[dst] =
                                l > 0.f ? (m_ref + __log2f(l)) * 0.69314718055994531f : NEG_INF;
                    } else {
                        __nv_bfloat16 *o = p.out + dst;
#pragma unroll
                        for (int c = 0; c < kHalfDims / 32; ++c)
#pragma unroll
                            for (int e = 0; e < 32; e += 8) {
                                uint4 w;
                                w.x = pack_bf16x2(__uint_as_float(v[c][e + 0]) * inv, __uint_as_float(v[c][e + 1]) * inv);
                                w.y = pack_bf16x2(__uint_as_float(v[c][e + 2]) * inv, __uint_as_float(v[c][e + 3]) * inv);
                                w.z = pack_bf16x2(__uint_as_float(v[c][e + 4]) * inv, __uint_as_float(v[c][e + 5]) * inv);
                                w.w = pack_bf16x2(__uint_as_float(v[c][e + 6]) * inv, __uint_as_float(v[c][e + 7]) * inv);
                                *reinterpret_cast<uint4 *>(o + c * 32 + e) = w;
                            }
                    }
                }
            }
            release_item(k);
        }
        if (ok) release_item(k);                           // the closing (empty) item
    }

    // teardown: every role is done with tensor memory
    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, Cfg::kTmemCols);
    }
    pdl_wait();       // complete only after the kernel launched before this one
}

// ---- host side --------------------------------------------------------------------

EncodeTiledFn encode_fn() {
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
    if (launch_pdl(prefill_kernel<HD, CASCADE>, dim3(static_cast<unsigned>(grid)), dim3(448), Cfg::kSmem, stream,
                   kvm, static_cast<const __nv_bfloat16 *>(query), q_stride, p) != cudaSuccess)
        return PKV_ERR_CUDA;
    return PKV_OK;
}


int launch_prefix_e4m3(const PrefillParams &p, const void *query, int64_t q_stride, const void *kv_cache,
                       int64_t num_blocks, int32_t head_size, int64_t grid, int dev, cudaStream_t stream) {
    if (grid <= 0) return PKV_OK;
    CUtensorMap kvm;
    const int rc = make_page_map_e4m3(&kvm, kv_cache, num_blocks, p.num_kv_heads, head_size);
    if (rc) return rc;
    return head_size == 64 ? launch_prefill_hd<64, true>(p, kvm, query, q_stride, grid, dev, stream)
                           : launch_prefill_hd<128, true>(p, kvm, query, q_stride, grid, dev, stream);
}

int launch_prefill_e4m3(const PrefillParams &p, const void *query, int64_t q_stride, const void *kv_cache,
                        int64_t num_blocks, int32_t head_size, int64_t grid, int dev, cudaStream_t stream) {
    if (grid <= 0) return PKV_OK;
    CUtensorMap kvm;
    const int rc = make_page_map_e4m3(&kvm, kv_cache, num_blocks, p.num_kv_heads, head_size);
    if (rc) return rc;
    return head_size == 64 ? launch_prefill_hd<64, false>(p, kvm, query, q_stride, grid, dev, stream)
                           : launch_prefill_hd<128, false>(p, kvm, query, q_stride, grid, dev, stream);
}

// Tensor map of an E4M3 cache as bytes {head_size, 16, 2, kv heads, blocks};
// a box is the K (or V) rows of one page, unswizzled (the converter warps
// widen them).
int make_page_map_e4m3(CUtensorMap *kvm, const void *kv_cache, int64_t num_blocks, int32_t num_kv_heads,
                       int32_t head_size) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return PKV_ERR_CUDA;
    const cuuint64_t dims[5] = {static_cast<cuuint64_t>(head_size), kBlock, 2, static_cast<cuuint64_t>(num_kv_heads),
                                static_cast<cuuint64_t>(num_blocks)};
    const cuuint64_t row = static_cast<cuuint64_t>(head_size);
    const cuuint64_t strides[4] = {row, row * kBlock, row * kBlock * 2, row * kBlock * 2 * num_kv_heads};
    const cuuint32_t box[5] = {static_cast<cuuint32_t>(head_size), kBlock, 1, 1, 1};
    const cuuint32_t es[5] = {1, 1, 1, 1, 1};
    if (enc(kvm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, const_cast<void *>(kv_cache), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return PKV_ERR_CUDA;
    return PKV_OK;
}

}  // namespace pkv
