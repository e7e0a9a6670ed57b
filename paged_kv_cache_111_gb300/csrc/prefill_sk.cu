// Prefill-chunk paged attention on the 5th-generation tensor cores (bf16
// cache), with the keys of every tile split between two independent softmax
// streams.
//
// The same computation as the decode path ("continuous batching and
// PagedAttention" tutorial, section 3.6: loop over the request's blocks
// through its block table, accumulate softmax(QK^T)V), for requests whose
// rows are many: a chunk of a chunked prefill ("Inside vLLM: Anatomy of a
// High-Throughput LLM Inference System", chunked prefill; "vLLM internals:
// managing the KV cache like an OS manages memory", section 3.2) attends
// causally, query i of the chunk seeing keys 0 .. context + i.
//
// Work item: one 128-row tile of one request for one kv head; rows are
// (query token, q head of the GQA group) pairs, so one K/V tile in shared
// memory serves every q head of the group.  A persistent CTA per SM takes
// items largest first from a shared counter.  Per 128-key KV tile j:
//   S = Q K_j^T        tcgen05.mma, A = Q and B = K_j from shared memory
//                      (K-major, 128-byte swizzle), D in one of two S buffers
//                      in tensor memory, so S of tile j + 1 is computed while
//                      the softmax works on tile j
//   softmax            two threads per row: thread h takes keys 64 h .. 64 h + 63
//                      of every tile and keeps its own running max and sum (an
//                      online softmax over its half of the keys), so the two
//                      never wait for each other within the item
//   O_h += P_h V_j     tcgen05.mma, A = P_h from tensor memory (written over
//                      S), B = rows 64 h .. 64 h + 63 of V_j (MN-major) from
//                      shared memory, D = O_h in tensor memory
// At the end of the item the two halves of each row are merged (the
// log-sum-exp combination of two softmax states over disjoint keys) and
// written.  Tensor memory: S0, S1, O_0, O_1 (512 columns at head size 128).
// Q arrives by TMA (at head size 64 into the second of two buffers while the
// current item runs; at 128 into the one buffer once the item's last S has
// read it, about two tiles before the item ends).  K and V of a tile arrive
// together, one 4 KiB box per (page, 64-column half), into a ring stage that
// both products read in place (K's rows at one stride for S, each page's V
// rows for P V).
// Warp roles (384 threads): warp 0 claims items and loads Q (TMA, for a
// chunk) and the tiles' pages through the block table (TMA); warps 1 and 2
// issue the MMAs of key halves 0 and 1 (each its half's S and P V), each
// product as soon as its operands are ready; warp 2 also owns the
// tensor-memory allocation; for the shared-prefix pass, whose rows come from
// many requests, warp 3 gathers Q rows with asynchronous copies instead;
// warps 4-7 take keys 0-63 of every tile, warps 8-11 keys 64-127 (warp w
// reads the tensor-memory lanes of quadrant w % 4).
//
// When any row of a warp puts a large share of its weight on few keys of a
// tile (rows with few visible keys, or a peaked softmax), P's bf16 remainder
// also enters that half's P V (a second set of MMAs), keeping ~16 bits per
// weight.  V rows past the sequence end in its last page are zeroed before
// P V, so NaN in unwritten cache slots never meets a zero weight.  Every wait
// is bounded.
//
// What bounds it: the MMA threads' issue.  A tile takes 24 products (per key
// half 8 of 128 x 64 x 16 for S and 4 of 128 x 128 x 16 for P V), about 1,300
// cycles of tensor pipe, but an issuing thread shares its sub-partition's
// scheduler with two softmax warps (a warp reads only its tensor-memory lane
// quadrant, and the quadrant is the sub-partition), and their tensor-memory
// loads and stores and exponentials slow each issue from about 90 to
// 130-240 cycles.  Hence two issuing threads, and a softmax that reads S
// once and stores P with its remainder in one instruction per 32 keys.
#include <mutex>

#include "prefill_common.cuh"

namespace pkv {

template <int HD>
struct SKCfg {
    static constexpr int kHalves = HD / 64;
    static constexpr int kTileBytes = kHalves * 128 * 128;   // 128 rows x HD bf16 (a Q tile, or K or V of 128 keys)
    // A ring stage holds K and V of one 128-key tile as they land: one box per
    // (page, 64-column half of the head) of 4 KiB, laid out
    //   [token half th][K, V][token t % 8][64 columns]    (128-byte rows, 128-byte swizzle)
    // at half * kHalfBytes + page * kBoxBytes.  K's rows of the tile then sit at
    // one stride (8-row groups 2 KiB apart, in key order) for the S product, and
    // each page's V rows likewise for P V, so both products read the stage in
    // place: 16 boxes per tile at head size 128 instead of 32 separate K and V
    // boxes of 2 KiB, and the copy engine takes a box in about the same time
    // whatever its size up to 4 KiB.
    static constexpr int kBoxBytes = 4096;
    static constexpr int kHalfBytes = (kPrefillKeys / kBlock) * kBoxBytes;
    static constexpr int kStageBytes = kHalves * kHalfBytes;    // = 2 kTileBytes
    // Q buffers and ring depth.  A stage is refilled once both P V products of
    // its tile have read it, so the copies of tile j + 3 start when tile j's
    // products complete.  At head size 128 three stages (192 KiB) leave room for
    // one Q buffer, loaded once the item's last S product has read the previous
    // Q (about two tiles before the item ends), and for no alignment slack: the
    // dynamic shared memory must start 1 KiB-aligned (checked at entry).
    static constexpr int kQBufs = HD == 128 ? 1 : 2;
    static constexpr int kStages = HD == 128 ? 3 : 4;
    static constexpr int kOffQ = 0;
    static constexpr int kOffKV = kOffQ + kQBufs * kTileBytes;
    static constexpr int kOffBar = kOffKV + kStages * kStageBytes;
    static constexpr int kOffXchg = kOffBar + 448;            // the halves' final maxima and sums
    static constexpr int kOffItems = kOffXchg + 2 * 2 * kPrefillRows * 4;
    static constexpr int kSlack = HD == 128 ? 0 : 1024;       // alignment slack
    static constexpr int kSmem = kOffItems + 256 + kSlack;
    static constexpr uint32_t kTmemCols = 512;
    // S buffer b at columns 128 b (P and its remainder are written over it);
    // O of key half h at 256 + HD h
    static __device__ __forceinline__ uint32_t col_s(int b) { return 128u * b; }
    static __device__ __forceinline__ uint32_t col_o(int h) { return 256u + HD * h; }
};

enum SKBar {
    kSKQFull = 0,                 // Q buffer b loaded (+ b, up to two buffers)
    kSKQEmpty = 2,                // both MMA threads' last S of the item have read Q buffer b (+ b)
    kSKSFull = 4,                 // key half h of S buffer b written (+ 2 b + h)
    kSKPFull = 8,                 // P of key half h in S buffer b written (+ 2 b + h)
    kSKODone = 12,                // O_h += P_h V completed (+ h)
    kSKOReady = 14,               // the item's last O_h += P_h V completed (+ h)
    kSKOFree = 16,                // O_0 and O_1 read out by the epilogue
    kSKXchg = 17,                 // the two threads of a row meet (+ quadrant)
    kSKKVFull = 21,               // K and V of ring stage s landed (+ s, up to four)
    kSKKVEmpty = 25,              // both key halves' P V products of stage s's tile completed (+ s)
    kSKVFix = 29,                 // V rows past the sequence end zeroed in stage s (+ s)
    kSKItemFull = 33, kSKItemEmpty = 37,
    kSKNumBars = 41
};
static_assert(kSKNumBars * 8 + 16 + 64 <= 448, "barriers, the TMEM address slot and the votes fit 448 bytes");

constexpr int kSKThreads = 384;

// 16-byte asynchronous copy global -> shared (L2 only), and the wait for all
// of this thread's copies.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Persistent: one CTA per SM.  The CTA's first item is its index; each later
// one is claimed from a counter the plan zeroes, in the plan's order (largest
// first).  Tiles and barrier phases are counted across items, so the next
// item's loads, Q and first S products overlap the current item's last tiles
// and epilogue.
template <int HD, bool CASCADE>
__global__ void __launch_bounds__(kSKThreads, 1)
    prefill_sk_kernel(const __grid_constant__ CUtensorMap kv_map, const __grid_constant__ CUtensorMap q_map,
                      const __nv_bfloat16 *__restrict__ query, const int64_t q_stride, const PrefillParams p) {
    using Cfg = SKCfg<HD>;
    constexpr int R = Cfg::kStages, NQ = Cfg::kQBufs;
    static_assert(R <= 4 && NQ <= 2, "barriers of the ring and Q buffers");
    constexpr int kPagesPerTile = kPrefillKeys / kBlock;
    constexpr int kBoxesPerTile = kPagesPerTile * Cfg::kHalves;     // TMA boxes of a K and V tile
    static_assert(Cfg::kStageBytes == 2 * Cfg::kTileBytes, "a stage holds K and V of a tile");
    static_assert(kBoxesPerTile <= 32, "one box per lane");
    constexpr int kHalfKeys = kPrefillKeys / 2;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (Cfg::kSlack == 0 && (smem_u32(smem_raw) & 1023u)) {     // uniform over the grid
        // the kernel would not fit: no work, reported as a failed asynchronous step
        if (threadIdx.x == 0) set_status(reinterpret_cast<int32_t *>(p.ws), PKV_ERR_DEVICE_TIMEOUT);
        pdl_wait();
        return;
    }
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg::kOffBar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + kSKNumBars);
    // the softmax warps' votes for the remainder of P, one byte each,
    // [S buffer][key half][quadrant]: an MMA thread reads its half's four at once
    volatile uint8_t *votes = reinterpret_cast<volatile uint8_t *>(tmem_slot + 4);
    volatile PfItem *items = reinterpret_cast<volatile PfItem *>(smem + Cfg::kOffItems);
    const uint32_t sQ = smem_u32(smem + Cfg::kOffQ);
    const uint32_t sKV = smem_u32(smem + Cfg::kOffKV);

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
    // one thread initialising all of them in turn held every CTA ~2.5 us
    if (threadIdx.x < kSKNumBars) {
        const int b = threadIdx.x;
        int count = 1;
        if (b >= kSKPFull && b < kSKPFull + 4) count = 4;            // the key half's softmax warps
        else if (b == kSKOFree) count = 8;                            // every softmax warp
        else if (b >= kSKXchg && b < kSKXchg + 4) count = 2;         // the two warps of a quadrant
        else if (b >= kSKQEmpty && b < kSKQEmpty + 2) count = 2;     // both MMA threads
        else if (b >= kSKKVEmpty && b < kSKKVEmpty + 4) count = 2;   // both MMA threads
        else if (b >= kSKItemEmpty && b < kSKItemEmpty + kItemSlots)
            count = CASCADE ? 11 : 10;             // 2 MMA threads, 8 softmax warps (+ the Q gatherer)
        mbar_init(&bars[b], count);
    }
    if (threadIdx.x == 0) {
        tma_prefetch_desc(&kv_map);
        if (!CASCADE) tma_prefetch_desc(&q_map);
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

    // the item's KV tile holding the sequence's last key, when that page is partial
    auto end_tile_of = [](int L) { return (!CASCADE && (L % kBlock)) ? (L - 1) / kPrefillKeys : -1; };

    if (warp == 0) {
        // ---------------- producer: items, Q, then K and V pages through the block table ----------------
        bool ok = true;
        int item = blockIdx.x;
        int gj = 0;                                    // KV tiles of this CTA so far (ring position)
        int taken = 0;                                 // items of this CTA
        int *next_item = reinterpret_cast<int *>(p.ws + (CASCADE ? offsetof(WsHeader, next_prefix_item)
                                                                  : offsetof(WsHeader, next_ptile_item)));
        for (int k = 0; ok; ++k) {
            const int slot = k % kItemSlots;
            // the slot's previous item has been read by every consumer
            if (k >= kItemSlots)
                ok = __all_sync(0xffffffffu,
                                pf_wait(&bars[kSKItemEmpty + slot], (k / kItemSlots - 1) & 1, status));
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
                mbar_arrive(&bars[kSKItemFull + slot]);
            }
            if (!it.valid) break;
            ++taken;
            if constexpr (!CASCADE) {
                // Q of the item into buffer k % NQ, once the item NQ back has read it:
                // rows (token, q head) of the tile are the box {64 dims, G heads,
                // 128 / G tokens}; tokens past the batch load as zeros, rows past the
                // request are masked by the softmax
                const int qb = k % NQ;
                if (k >= NQ) ok = __all_sync(0xffffffffu, pf_wait(&bars[kSKQEmpty + qb], (k / NQ - 1) & 1, status));
                if (!ok) break;
                if (lane == 0) {
                    const int tok0 = it.qs + it.row0 / G;
                    mbar_arrive_expect_tx(&bars[kSKQFull + qb], Cfg::kTileBytes);
                    for (int h = 0; h < Cfg::kHalves; ++h)
                        tma_load_3d(smem + Cfg::kOffQ + qb * Cfg::kTileBytes + h * (kPrefillRows * 128), &q_map,
                                    &bars[kSKQFull + qb], h * 64, it.g * G, tok0);
                }
            }

            const int end_tile = end_tile_of(it.L);
            const int32_t *bt = p.block_tables + static_cast<int64_t>(it.r) * p.max_blocks_per_seq;
            // the pages' coordinates in the tensor map (block id x kv heads + head) in
            // windows of 32 pages (4 KV tiles), one lane per page; the next window is
            // loaded a window ahead.  Pages past the sequence, and block ids outside
            // the cache (reported), get -1 and load as zeros (outside the tensor map).
            auto load_window = [&](int w) -> int {
                const int page = it.t0 * kPagesPerTile + w * 32 + lane;
                const int b = page < it.n_pages ? __ldg(bt + page) : -1;
                if (page >= it.n_pages) return -1;
                if (b < 0 || b >= p.num_blocks) {
                    set_status(status, PKV_ERR_DEVICE_INDEX);
                    return -1;
                }
                return b * p.num_kv_heads + it.g;
            };
            int win_cur = load_window(0);
            int win_next = load_window(1);
            for (int j = 0; j < it.n_kv && ok; ++j) {
                const int gt = gj + j;
                const int st = gt % R;
                if (j > 0 && (j * kPagesPerTile) % 32 == 0) {
                    win_cur = win_next;
                    win_next = load_window(j * kPagesPerTile / 32 + 1);
                }
                const int wofs = (j * kPagesPerTile) % 32;
                // this lane's box: page lane / kHalves of the tile, columns 64 (lane % kHalves)
                const int my_pg = __shfl_sync(0xffffffffu, win_cur, wofs + (lane / Cfg::kHalves) % kPagesPerTile);
                // K and V of tile gt once both P V products of tile gt - R have read the stage
                if (gt >= R) ok = __all_sync(0xffffffffu, pf_wait(&bars[kSKKVEmpty + st], ((gt - R) / R) & 1, status));
                if (!ok) break;
                // one box per lane: the copy engine takes boxes faster from several
                // issuing lanes than from one
                if (lane == 0) mbar_arrive_expect_tx(&bars[kSKKVFull + st], Cfg::kStageBytes);
                __syncwarp();
                if (lane < kBoxesPerTile)
                    tma_load_5d(smem + Cfg::kOffKV + st * Cfg::kStageBytes + (lane % Cfg::kHalves) * Cfg::kHalfBytes +
                                    (lane / Cfg::kHalves) * Cfg::kBoxBytes,
                                &kv_map, &bars[kSKKVFull + st], (lane % Cfg::kHalves) * 64, 0, 0, 0, my_pg);
                if (j == end_tile) {
                    // zero V rows past the sequence end in its last (partial) page;
                    // one fix barrier per stage, so none runs two phases ahead
                    ok = __all_sync(0xffffffffu, pf_wait(&bars[kSKKVFull + st], (gt / R) & 1, status));
                    if (!ok) break;
                    const int lp = (it.L - 1) / kBlock - j * kPagesPerTile;   // page within the tile
                    const int first = it.L % kBlock;
                    const int nrows = kBlock - first;
                    for (int e = lane; e < Cfg::kHalves * nrows * 8; e += 32) {
                        const int c = e / (nrows * 8);
                        const int rem = e % (nrows * 8);
                        const int t = first + rem / 8;                       // token within the page
                        const uint32_t a = sKV + st * Cfg::kStageBytes + c * Cfg::kHalfBytes + lp * Cfg::kBoxBytes +
                                           (t >> 3) * 2048 + 1024 + (t & 7) * 128 + (rem % 8) * 16;
                        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0u) : "memory");
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars[kSKVFix + st]);
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
    } else if (warp == 1 || warp == 2) {
        // ---------------- MMA issuers: warp 1 key half 0, warp 2 key half 1 ----------------
        // Each thread issues its key half's S (N = 64, into its half of the S
        // buffer) and P V (into its O_h): the softmax warps of a sub-partition
        // slow the issue of an MMA thread beside them, and two threads on two
        // sub-partitions issue twice as many products at once.  A thread owns
        // its S columns and its O_h, so issue order within the thread covers
        // every hazard between its products.
        const int hh = warp - 1;
        if (lane == 0) {
            constexpr uint32_t kIdescS = idesc_bf16_f32(kPrefillRows, kHalfKeys, 0, 0);
            constexpr uint32_t kIdescO = idesc_bf16_f32(kPrefillRows, HD, 0, 1);
            // S_h(gt) = Q K_h^T into columns 64 hh of S buffer gt & 1: both operands
            // K-major in shared memory, Q's 8-row groups 1 KiB apart, K's 2 KiB apart
            // in the stage (keys 64 hh .. 64 hh + 63: pages 4 hh .. 4 hh + 3)
            auto issue_s = [&](int qb, int gt) {
                const int st = gt % R;
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const uint64_t a = smem_desc_sw128(
                        sQ + qb * Cfg::kTileBytes + (kk >> 2) * (kPrefillRows * 128) + (kk & 3) * 32, 16, 1024);
                    const uint64_t b = smem_desc_sw128(sKV + st * Cfg::kStageBytes + (kk >> 2) * Cfg::kHalfBytes +
                                                           hh * (kHalfKeys / kBlock) * Cfg::kBoxBytes + (kk & 3) * 32,
                                                       16, 2048);
                    umma_f16_ss(tmem + Cfg::col_s(gt & 1) + hh * kHalfKeys, a, b, kIdescS, kk > 0 ? 1u : 0u);
                }
                umma_commit(&bars[kSKSFull + 2 * (gt & 1) + hh]);
            };
            // O_hh (+)= P_hh V: A = P of key half hh in S buffer gt & 1, keys 64 hh +
            // 32 c .. 64 hh + 32 c + 31 at columns 64 hh + 32 c + [0, 16) (their bf16
            // remainder at + [16, 32)); B = V rows of page 4 hh + kk of the stage
            // (MN-major: the two 8-row groups 2 KiB apart, the column halves
            // kHalfBytes apart)
            auto issue_pv = [&](int gt, uint32_t lo, uint32_t accumulate) {
                const int st = gt % R;
#pragma unroll
                for (int kk = 0; kk < kHalfKeys / 16; ++kk) {
                    const uint64_t b = smem_desc_sw128(
                        sKV + st * Cfg::kStageBytes + (4 * hh + kk) * Cfg::kBoxBytes + 1024, Cfg::kHalfBytes, 2048);
                    const uint32_t a = tmem + Cfg::col_s(gt & 1) + 64 * hh + (kk >> 1) * 32 + (kk & 1) * 8 + lo;
                    umma_f16_ts(tmem + Cfg::col_o(hh), a, b, kIdescO, (accumulate || kk > 0) ? 1u : 0u);
                }
            };
            bool ok = true;
            int gj = 0;
            uint32_t vfix_par = 0;                     // phase parity of each stage's fix barrier
            for (int k = 0; ok; ++k) {
                const int slot = k % kItemSlots;
                ok = pf_wait(&bars[kSKItemFull + slot], (k / kItemSlots) & 1, status);
                if (!ok) break;
                const bool valid = items[slot].valid != 0;
                const int n_kv = items[slot].n_kv;
                const int end_tile = end_tile_of(items[slot].L);
                mbar_arrive(&bars[kSKItemEmpty + slot]);
                if (!valid) break;
                const int qb = k % NQ;
                ok = pf_wait(&bars[kSKQFull + qb], (k / NQ) & 1, status);
                // the item's S and P V products in dependency order, each as soon as
                // it may go: S(j) once its stage has landed and P V(j - 2) has been
                // issued (S buffer j & 1 last held P of tile j - 2, and the tcgen05.mma
                // operations of one thread execute in issue order, so that product has
                // read P before S is written); P V(j) once this half's P of tile j is
                // written, V has been fixed (end tile) and, for the item's first tile,
                // O has been read out by the previous item's epilogue.  S goes first
                // when both may: the softmax waits on it.
                int js = 0, jp = 0;
                uint64_t t_idle = 0;                   // start of the current wait (0: none)
                while (ok && jp < n_kv) {
                    const bool s_can = js < n_kv && js <= jp + 1;
                    const bool p_can = jp < js;
                    if (s_can && mbar_test_wait(&bars[kSKKVFull + (gj + js) % R], ((gj + js) / R) & 1)) {
                        tc_fence_after();
                        issue_s(qb, gj + js);
                        if (++js == n_kv) umma_commit(&bars[kSKQEmpty + qb]);
                        t_idle = 0;
                        continue;
                    }
                    if (p_can) {
                        const int gt = gj + jp;
                        const int st = gt % R, sb = gt & 1;
                        bool ready = mbar_test_wait(&bars[kSKPFull + 2 * sb + hh], (gt >> 1) & 1);
                        if (ready && jp == end_tile) ready = mbar_test_wait(&bars[kSKVFix + st], (vfix_par >> st) & 1u);
                        if (ready && jp == 0 && k > 0) ready = mbar_test_wait(&bars[kSKOFree], (k - 1) & 1);
                        if (ready) {
                            if (jp == end_tile) vfix_par ^= 1u << st;
                            tc_fence_after();
                            const uint32_t vote = *reinterpret_cast<volatile const uint32_t *>(votes + 8 * sb + 4 * hh);
                            issue_pv(gt, 0, jp > 0 ? 1u : 0u);
                            if (vote) issue_pv(gt, 16, 1u);
                            umma_commit(&bars[kSKODone + hh]);
                            umma_commit(&bars[kSKKVEmpty + st]);
                            if (++jp == n_kv) umma_commit(&bars[kSKOReady + hh]);
                            t_idle = 0;
                            continue;
                        }
                    }
                    // nothing may go yet: sleep on the likelier next event (the
                    // softmax's P while a P V may go, with a short hint so that a stage
                    // landing meanwhile is seen soon; else the stage S waits for),
                    // bounded like every other wait
                    if (p_can)
                        mbar_try_wait_for(&bars[kSKPFull + 2 * ((gj + jp) & 1) + hh], ((gj + jp) >> 1) & 1, 200);
                    else
                        mbar_try_wait(&bars[kSKKVFull + (gj + js) % R], ((gj + js) / R) & 1);
                    const uint64_t now = global_ns();
                    if (t_idle == 0) {
                        t_idle = now;
                    } else if (now - t_idle > kWaitLimitNs) {
                        set_status(status, PKV_ERR_DEVICE_TIMEOUT);
                        ok = false;
                    }
                }
                gj += n_kv;
            }
        }
        __syncwarp();
    } else if (warp == 3) {
        // ---------------- shared-prefix pass: Q gatherer, four rows per thread ----------------
        if constexpr (CASCADE) {
            bool ok = true;
            for (int k = 0; ok; ++k) {
                const int slot = k % kItemSlots;
                ok = __all_sync(0xffffffffu, pf_wait(&bars[kSKItemFull + slot], (k / kItemSlots) & 1, status));
                if (!ok) break;
                const bool valid = items[slot].valid != 0;
                const int row0 = items[slot].row0, rows_total = items[slot].rows_total, g = items[slot].g;
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[kSKItemEmpty + slot]);
                if (!valid) break;
                // rows {token, request, query index, q head in group}, all four of this
                // lane's looked up at once, before the wait for the buffer; zeros past
                // the rows
                const int4 *crows = reinterpret_cast<const int4 *>(p.ws + ws_ld(&hdr->off_crows));
                int4 crow4[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int rr = row0 + i * 32 + lane;
                    crow4[i] = rr < rows_total ? ws_ld(crows + rr) : make_int4(0, 0, 0, 0);
                }
                // Q buffer k % NQ, once the item NQ back has read it
                const int qb = k % NQ;
                if (k >= NQ) ok = __all_sync(0xffffffffu, pf_wait(&bars[kSKQEmpty + qb], (k / NQ - 1) & 1, status));
                if (!ok) break;
                const uint32_t qbase = sQ + qb * Cfg::kTileBytes;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int r = i * 32 + lane;                     // row within the tile
                    const bool vrow = row0 + r < rows_total;
                    const int4 crow = crow4[i];
                    const __nv_bfloat16 *src =
                        query + static_cast<int64_t>(crow.x) * q_stride + static_cast<int64_t>(g * G + crow.w) * HD;
#pragma unroll
                    for (int c = 0; c < HD / 8; ++c) {
                        const uint32_t dst =
                            qbase + (c >> 3) * (kPrefillRows * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4);
                        if (vrow) {
                            cp_async16(dst, src + c * 8);
                        } else {
                            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(dst), "r"(0u) : "memory");
                        }
                    }
                }
                cp_async_wait_all();
                fence_proxy_async_smem();          // visible to the tensor core's reads
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[kSKQFull + qb]);
            }
        }
    } else {
        // ---------------- softmax (one key half of a row per thread) and epilogue ----------------
        const int h = (warp - 4) >> 2;                  // key half
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const float NEG_INF = -__int_as_float(0x7f800000);
        const uint32_t trow = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        const uint32_t tOh = trow + Cfg::col_o(h);
        const float sl2 = p.scale_log2;
        // the halves' final maxima and sums, [half][row]; written once every
        // softmax warp has read the previous item's (its arrival on O-free)
        float *xm = reinterpret_cast<float *>(smem + Cfg::kOffXchg);
        float *xl = xm + 2 * kPrefillRows;
        uint64_t *xbar = &bars[kSKXchg + quad];
        bool ok = true;
        int gj = 0;                                     // KV tiles of this CTA so far
        int k = 0;
        for (;; ++k) {
            const int slot = k % kItemSlots;
            ok = __all_sync(0xffffffffu, pf_wait(&bars[kSKItemFull + slot], (k / kItemSlots) & 1, status));
            if (!ok) break;
            const volatile PfItem *cur = items + slot;
            if (!cur->valid) break;
            const int n_kv = cur->n_kv;
            const int kbase = cur->t0 * kPrefillKeys + h * kHalfKeys;
            const int g = cur->g;
            // this thread's row: keys [0, lim) visible; where its result goes
            // (-1: nowhere): element offset in out, or the partial row of split
            // `part` (cascade)
            const int rr = cur->row0 + row;
            int lim = 0;
            int64_t dst = -1;
            if (rr < cur->rows_total) {
                if constexpr (CASCADE) {
                    const int4 crow = ws_ld(reinterpret_cast<const int4 *>(p.ws + ws_ld(&hdr->off_crows)) + rr);
                    lim = cur->L;
                    const int4 rq = ws_ld(reinterpret_cast<const int4 *>(p.ws + ws_ld(&hdr->off_req)) + crow.y);
                    dst = rq.y + (static_cast<int64_t>(crow.z) * p.num_q_heads + g * G + crow.w) * rq.x + cur->part;
                } else {
                    lim = cur->ctx + rr / G + 1;
                    dst = (static_cast<int64_t>(cur->qs + rr / G) * p.num_q_heads + g * G + rr % G) * HD;
                }
            }
            float m_ref = NEG_INF, l = 0.f;                // this half's running max (log2 domain) and sum
            for (int j = 0; j < n_kv && ok; ++j) {
                const int gt = gj + j;
                const int sb = gt & 1;
                ok = __all_sync(0xffffffffu, pf_wait(&bars[kSKSFull + 2 * sb + h], (gt >> 1) & 1, status));
                if (!ok) break;
                tc_fence_after();
                const uint32_t tS = trow + Cfg::col_s(sb) + h * kHalfKeys;
                // keys a row may not see become -inf (tested only in tiles reaching
                // some row's limit)
                const int key0 = kbase + j * kPrefillKeys;
                const bool masked = __any_sync(0xffffffffu, key0 + kHalfKeys > lim);
                // this half's 64 scores, read once (the tensor-memory instructions of
                // the softmax warps delay the MMA thread's on the same sub-partition)
                float s[kHalfKeys];
                tmem_ld32f(tS, s);
                tmem_ld32f(tS + 32, s + 32);
                tmem_ld_wait();
                if (masked) {
#pragma unroll
                    for (int c = 0; c < kHalfKeys; ++c) s[c] = (key0 + c < lim) ? s[c] : NEG_INF;
                }
                // pass 1: their max (four chains of three-input maxima)
                float mx;
                {
                    float mx4[4] = {fmaxf(s[0], s[1]), fmaxf(s[2], s[3]), fmaxf(s[4], s[5]), fmaxf(s[6], s[7])};
#pragma unroll
                    for (int c = 8; c < kHalfKeys; c += 8) {
                        mx4[0] = fmax3(mx4[0], s[c], s[c + 1]);
                        mx4[1] = fmax3(mx4[1], s[c + 2], s[c + 3]);
                        mx4[2] = fmax3(mx4[2], s[c + 4], s[c + 5]);
                        mx4[3] = fmax3(mx4[3], s[c + 6], s[c + 7]);
                    }
                    mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
                }
                // log2-domain reference: moves on this half's first visible key, and
                // afterwards only when the tile's max exceeds it by more than 2^8
                // (scale > 0 keeps the order of scores)
                const bool first = m_ref == NEG_INF;
                const float m_new = fmaxf(m_ref, mx * sl2);
                const bool grow = !first && m_new > m_ref + 8.f;
                const float alpha = grow ? fast_exp2(m_ref - m_new) : 1.f;
                if (first || grow) m_ref = m_new;
                // pass 2, one 32-key piece at a time: weights p = 2^(s scale - ref)
                // with their sum and sum of squares; P as bf16 pairs and its bf16
                // remainder written over the piece's own 32 columns (32 c + [0, 16)
                // and 32 c + [16, 32) of this half) in one store.  The remainder
                // enters P V only when some warp of this half votes for it.
                const float ref = m_ref == NEG_INF ? 0.f : m_ref;
                const uint64_t sc2 = f2_pack(sl2, sl2), nref2 = f2_pack(-ref, -ref);
                uint64_t ps2[2] = {0, 0}, pq2[2] = {0, 0};
#pragma unroll
                for (int c = 0; c < kHalfKeys / 32; ++c) {
                    uint32_t wr[32];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const uint64_t y2 = f2_fma(f2_pack(s[32 * c + 2 * e], s[32 * c + 2 * e + 1]), sc2, nref2);
                        float y0, y1;
                        f2_unpack(y2, y0, y1);
                        const float p0 = fast_exp2(y0), p1 = fast_exp2(y1);
                        const uint64_t p2 = f2_pack(p0, p1);
                        ps2[e & 1] = f2_add(ps2[e & 1], p2);
                        pq2[e & 1] = f2_fma(p2, p2, pq2[e & 1]);
                        split_bf16x2(p0, p1, wr[e], wr[16 + e]);
                    }
                    tmem_st32(tS + 32 * c, wr);
                }
                if (__any_sync(0xffffffffu, grow)) {
                    // rare: O_h rescaled before this tile's P V is issued, once O_h +=
                    // P_h V of the previous tile has completed (grow needs an earlier
                    // tile of this item, so gt >= 1; that product's barrier cannot be
                    // two phases behind: S of this tile was committed after the
                    // products of tile gt - 2)
                    ok = __all_sync(0xffffffffu, pf_wait(&bars[kSKODone + h], (gt - 1) & 1, status));
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll 1
                    for (int c = 0; c < HD / 32; ++c) {
                        uint32_t v[32];
                        tmem_ld32(tOh + c * 32, v);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
                        tmem_st32(tOh + c * 32, v);
                    }
                }
                float a0, a1, b0, b1;
                f2_unpack(f2_add(ps2[0], ps2[1]), a0, a1);
                f2_unpack(f2_add(pq2[0], pq2[1]), b0, b1);
                const float psum = a0 + a1, psq = b0 + b1;
                l = l * alpha + psum;
                // this warp's vote: does any of its rows need the remainder of P?  (On
                // this half's own sums: the half's output part is accurate by itself,
                // and so is their merge.)
                const bool wneed = __any_sync(0xffffffffu, psq > kLoConcentration * l * l);
                tmem_st_wait();
                if (lane == 0) votes[8 * sb + 4 * h + quad] = wneed ? 1 : 0;
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[kSKPFull + 2 * sb + h]);
            }
            gj += n_kv;
            // epilogue: the two halves' states merged by log-sum-exp; this thread
            // writes output dims 64 h .. 64 h + 63 of its row
            if (ok && k > 0) ok = __all_sync(0xffffffffu, pf_wait(&bars[kSKOFree], (k - 1) & 1, status));
            if (ok) {
                xm[h * kPrefillRows + row] = m_ref;
                xl[h * kPrefillRows + row] = l;
                __syncwarp();
                if (lane == 0) mbar_arrive(xbar);
                ok = __all_sync(0xffffffffu, pf_wait(xbar, k & 1, status));
            }
            if (ok) ok = __all_sync(0xffffffffu, pf_wait(&bars[kSKOReady], k & 1, status));
            if (ok) ok = __all_sync(0xffffffffu, pf_wait(&bars[kSKOReady + 1], k & 1, status));
            if (ok) {
                const float m0 = xm[row], m1 = xm[kPrefillRows + row];
                const float l0 = xl[row], l1 = xl[kPrefillRows + row];
                const float M = fmaxf(m0, m1);
                // a half that saw no key has m = -inf and weight 0 (and O_h = 0)
                const float w0 = M == NEG_INF ? 0.f : fast_exp2(m0 - M);
                const float w1 = M == NEG_INF ? 0.f : fast_exp2(m1 - M);
                const float L = l0 * w0 + l1 * w1;
                const float inv = L > 0.f ? 1.f / L : 0.f;
                const float c0 = w0 * inv, c1 = w1 * inv;
                tc_fence_after();
                constexpr int kOutDims = HD / 2;                 // this thread's output dims
                uint32_t a[kOutDims / 32][32], b[kOutDims / 32][32];
#pragma unroll
                for (int c = 0; c < kOutDims / 32; ++c) {
                    tmem_ld32(trow + Cfg::col_o(0) + h * kOutDims + c * 32, a[c]);
                    tmem_ld32(trow + Cfg::col_o(1) + h * kOutDims + c * 32, b[c]);
                }
                tmem_ld_wait();
                // O_0 and O_1 are in registers: the next item's first P V may overwrite them
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[kSKOFree]);
                if (dst >= 0) {
                    if constexpr (CASCADE) {
                        // split `part` of the row: normalised partial output and natural log-sum-exp
                        float *po = reinterpret_cast<float *>(p.ws + ws_ld(&hdr->off_part_o)) + dst * HD + h * kOutDims;
#pragma unroll
                        for (int c = 0; c < kOutDims / 32; ++c)
#pragma unroll
                            for (int e = 0; e < 32; e += 4) {
                                float4 o4;
                                o4.x = __uint_as_float(a[c][e]) * c0 + __uint_as_float(b[c][e]) * c1;
                                o4.y = __uint_as_float(a[c][e + 1]) * c0 + __uint_as_float(b[c][e + 1]) * c1;
                                o4.z = __uint_as_float(a[c][e + 2]) * c0 + __uint_as_float(b[c][e + 2]) * c1;
                                o4.w = __uint_as_float(a[c][e + 3]) * c0 + __uint_as_float(b[c][e + 3]) * c1;
                                *reinterpret_cast<float4 *>(po + c * 32 + e) = o4;
                            }
                        if (h == 0)
                            reinterpret_cast<float *>(p.ws + ws_ld(&hdr->off_part_lse))[dst] =
                                L > 0.f ? (M + __log2f(L)) * 0.69314718055994531f : NEG_INF;
                    } else {
                        __nv_bfloat16 *o = p.out + dst + h * kOutDims;
#pragma unroll
                        for (int c = 0; c < kOutDims / 32; ++c)
#pragma unroll
                            for (int e = 0; e < 32; e += 8) {
                                uint4 w;
                                auto mix = [&](int i) {
                                    return __uint_as_float(a[c][e + i]) * c0 + __uint_as_float(b[c][e + i]) * c1;
                                };
                                w.x = pack_bf16x2(mix(0), mix(1));
                                w.y = pack_bf16x2(mix(2), mix(3));
                                w.z = pack_bf16x2(mix(4), mix(5));
                                w.w = pack_bf16x2(mix(6), mix(7));
                                *reinterpret_cast<uint4 *>(o + c * 32 + e) = w;
                            }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[kSKItemEmpty + slot]);
            if (!ok) break;
        }
        if (ok) {                                       // the closing (empty) item
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[kSKItemEmpty + k % kItemSlots]);
        }
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

template <int HD, bool CASCADE>
static int launch_sk_hd(const PrefillParams &p, const CUtensorMap &kvm, const CUtensorMap &qm, const void *query,
                        int64_t q_stride, int64_t grid, int dev, cudaStream_t stream) {
    using Cfg = SKCfg<HD>;
    static_assert(Cfg::kSmem <= 227 * 1024, "shared memory of one CTA");
    static std::mutex mu;
    static uint64_t done_mask = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
        if (!bit || !(done_mask & bit)) {
            if (cudaFuncSetAttribute(prefill_sk_kernel<HD, CASCADE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     Cfg::kSmem) != cudaSuccess)
                return PKV_ERR_CUDA;
            done_mask |= bit;
        }
    }
    if (launch_pdl(prefill_sk_kernel<HD, CASCADE>, dim3(static_cast<unsigned>(grid)), dim3(kSKThreads), Cfg::kSmem,
                   stream, kvm, qm, static_cast<const __nv_bfloat16 *>(query), q_stride, p) != cudaSuccess)
        return PKV_ERR_CUDA;
    return PKV_OK;
}

// Tensor map of the query as {head_size, q heads, tokens}: a box is 64 dims of
// G consecutive q heads of 128 / G consecutive tokens, 128-byte swizzle (one
// 128-row Q tile of a kv head's group, half or all of its head dimension).
static int make_query_map(CUtensorMap *qm, const void *query, int64_t q_stride, int32_t num_tokens,
                          int32_t num_q_heads, int32_t G, int32_t head_size) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return PKV_ERR_CUDA;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(head_size), static_cast<cuuint64_t>(num_q_heads),
                                static_cast<cuuint64_t>(num_tokens)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(head_size) * 2, static_cast<cuuint64_t>(q_stride) * 2};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(kPrefillRows / G)};
    const cuuint32_t es[3] = {1, 1, 1};
    if (enc(qm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(query), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return PKV_ERR_CUDA;
    return PKV_OK;
}

// Tensor map of the cache as {head_size, 8 tokens, K/V, 2 token halves, pages
// of every kv head (block id x kv heads + head)}: a box {64, 8, 2, 2, 1} is
// the K and V rows of one page, 64 columns, landing as [token half][K, V]
// [token % 8][64 columns] with 128-byte swizzle (4 KiB).
static int make_kv_tile_map(CUtensorMap *kvm, const void *kv_cache, int64_t num_blocks, int32_t num_kv_heads,
                            int32_t head_size) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return PKV_ERR_CUDA;
    const cuuint64_t row = static_cast<cuuint64_t>(head_size) * 2;
    const cuuint64_t dims[5] = {static_cast<cuuint64_t>(head_size), 8, 2, 2,
                                static_cast<cuuint64_t>(num_blocks) * static_cast<cuuint64_t>(num_kv_heads)};
    const cuuint64_t strides[4] = {row, row * kBlock, row * 8, row * kBlock * 2};
    const cuuint32_t box[5] = {64, 8, 2, 2, 1};
    const cuuint32_t es[5] = {1, 1, 1, 1, 1};
    if (enc(kvm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(kv_cache), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return PKV_ERR_CUDA;
    return PKV_OK;
}

int launch_prefill_sk(const PrefillParams &p, const void *query, int64_t q_stride, int32_t num_tokens,
                      const void *kv_cache, int64_t num_blocks, int32_t head_size, bool cascade, int64_t grid, int dev,
                      cudaStream_t stream) {
    if (grid <= 0) return PKV_OK;
    // (the kernel forms a page's coordinate block id x kv heads + head in 32 bits:
    // the call's argument checks hold num_blocks x kv heads below 2^31)
    CUtensorMap kvm, qm;
    int rc = make_kv_tile_map(&kvm, kv_cache, num_blocks, p.num_kv_heads, head_size);
    if (rc) return rc;
    if (cascade) {
        qm = kvm;                                  // not read: the pass gathers its query rows itself
        return head_size == 64 ? launch_sk_hd<64, true>(p, kvm, qm, query, q_stride, grid, dev, stream)
                               : launch_sk_hd<128, true>(p, kvm, qm, query, q_stride, grid, dev, stream);
    }
    rc = make_query_map(&qm, query, q_stride, num_tokens, p.num_q_heads, p.G, head_size);
    if (rc) return rc;
    return head_size == 64 ? launch_sk_hd<64, false>(p, kvm, qm, query, q_stride, grid, dev, stream)
                           : launch_sk_hd<128, false>(p, kvm, qm, query, q_stride, grid, dev, stream);
}

}  // namespace pkv
