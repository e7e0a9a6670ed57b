// Pieces shared by the tensor-core prefill kernels (prefill_sk.cu over a bf16
// cache, prefill_tc.cu over an E4M3 cache): softmax arithmetic on fp32 pairs,
// P packing, bounded waits, the work-item record and the plan loads through
// L2.
#pragma once

#include <cuda_fp16.h>

#include "attn_internal.cuh"
#include "tc_common.cuh"

namespace pkv {

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

// Four E4M3 values (one 32-bit word, element 0 in the low byte) -> two f16x2
// words (elements 0,1 and 2,3), exactly.
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t w, uint32_t &h01, uint32_t &h23) {
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "mov.b32 {lo, hi}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, lo;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, hi;\n\t}"
        : "=r"(h01), "=r"(h23)
        : "r"(w));
}

// P of a pair of keys as the 16-bit type of the products (bf16, or f16 over
// an E4M3 cache), and the remainder that the rounding left.
template <bool F16> __device__ __forceinline__ uint32_t pack_p(float a, float b) {
    if constexpr (F16) {
        const __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<const uint32_t *>(&h);
    } else {
        return pack_bf16x2(a, b);
    }
}
template <bool F16> __device__ __forceinline__ uint32_t pack_p_rest(float a, float b) {
    if constexpr (F16) {
        const float2 hb = __half22float2(__floats2half2_rn(a, b));
        const __half2 r = __floats2half2_rn(a - hb.x, b - hb.y);
        return *reinterpret_cast<const uint32_t *>(&r);
    } else {
        const float2 hb = __bfloat1622float2(__floats2bfloat162_rn(a, b));
        return pack_bf16x2(a - hb.x, b - hb.y);
    }
}

// Bounded wait shared by every role; on timeout records the error and
// reports it so the role can stop.
__device__ __forceinline__ bool pf_wait(uint64_t *bar, uint32_t parity, int32_t *status) {
    if (mbar_wait_bounded(bar, parity)) return true;
    set_status(status, PKV_ERR_DEVICE_TIMEOUT);
    return false;
}

// One work item: one 128-row tile for one kv head.  CASCADE = false: rows of
// one long request (a prefill chunk), causal, written to `out`.
// CASCADE = true: 128 rows taken from every request that shares the first
// prefix_blocks blocks of its table with request 0, against one range of
// those blocks' KV tiles (every key of the prefix is visible to every such
// row); the result for range i is split i of each row (normalised partial
// output and its log-sum-exp), merged with the row's other splits by the
// combine.
struct PfItem {
    int32_t valid;        // 0: no further item for this CTA
    int32_t r;            // request whose block table is read
    int32_t n_kv;         // KV tiles of the item
    int32_t L;            // keys of the request (cascade: of the prefix)
    int32_t qs, ctx;      // first query token, keys before the chunk
    int32_t rows_total;   // rows of the request (cascade: of the pass)
    int32_t row0;         // first row of the tile
    int32_t n_pages;      // pages of the key range's sequence
    int32_t part, t0;     // cascade split and its first KV tile (0 otherwise)
    int32_t g;            // kv head
};
constexpr int kItemSlots = 4;

// A workspace field written by the plan, loaded through L2 (not L1): the
// prefill kernel reads the plan before its programmatic-launch wait.
__device__ __forceinline__ int32_t ws_ld(const int32_t *a) { return __ldcg(a); }
__device__ __forceinline__ int64_t ws_ld(const int64_t *a) {
    return static_cast<int64_t>(__ldcg(reinterpret_cast<const long long *>(a)));
}
__device__ __forceinline__ int4 ws_ld(const int4 *a) { return __ldcg(a); }
static_assert(kItemSlots * sizeof(PfItem) <= 256, "item ring fits its 256 bytes");

// cuTensorMapEncodeTiled from the driver (looked up once); nullptr if missing.
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_fn();

// Tensor map of an E4M3 cache for its tile kernels: {head_size, 16, 2, kv
// heads, blocks}; a box is the K (or V) rows of one page as unswizzled bytes.
int make_page_map_e4m3(CUtensorMap *kvm, const void *kv_cache, int64_t num_blocks, int32_t num_kv_heads,
                       int32_t head_size);

}  // namespace pkv
