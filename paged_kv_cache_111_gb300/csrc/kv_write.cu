// Cache write ("reshape_and_cache"): scatter new K/V tokens into their slots;
// and the copy-on-write block copy.
//
// "vLLM internals: managing the KV cache like an OS manages memory", section
// 2.1 (the fused write op puts each new token's K/V into its physical block);
// "continuous batching and PagedAttention" tutorial, section 3.3 (token ->
// block slot / 16, offset slot % 16); "vLLM source reading", section 5.1
// (slot_mapping drives the scatter).
//
// A pure bit copy, HBM-bound: each thread moves one 16-byte vector of one
// token's K or V row; consecutive threads cover consecutive 16-byte pieces of
// a head's row, so reads and writes are coalesced 128-byte+ runs.
#include <cuda_fp8.h>

#include "pkv_common.cuh"

namespace pkv {

struct KvWriteParams {
    uint4 *cache;            // viewed as 16-byte vectors
    int64_t num_slots;       // num_blocks * 16
    const uint4 *key;
    const uint4 *value;
    int64_t key_stride_v;    // token stride in 16-byte vectors
    int64_t value_stride_v;
    const int64_t *slots;
    int32_t num_tokens;
    int32_t num_kv_heads;
    int32_t vec_shift;       // log2(head_size / 8)
    int32_t *status;
};

// One token per CTA iteration; the CTA's threads cover that token's K and V
// rows of every kv head, 16 bytes each.
__global__ void __launch_bounds__(256) kv_write_kernel(KvWriteParams p) {
    pdl_trigger();                                         // the attention plan may start (it reads no cache)
    const int vpr = 1 << p.vec_shift;                      // vectors per head row
    const int per_kv = p.num_kv_heads * vpr;               // vectors of K (or V) per token
    const int per_tok = 2 * per_kv;
    for (int64_t t = blockIdx.x; t < p.num_tokens; t += gridDim.x) {
        const int64_t slot = __ldg(p.slots + t);
        if (slot < 0) continue;                             // padding token
        if (slot >= p.num_slots) {
            if (threadIdx.x == 0) set_status(p.status, PKV_ERR_DEVICE_INDEX);
            continue;
        }
        const int64_t blk = slot / kBlock;
        const int64_t off = slot - blk * kBlock;
        const uint4 *ksrc = p.key + t * p.key_stride_v;
        const uint4 *vsrc = p.value + t * p.value_stride_v;
        for (int v = threadIdx.x; v < per_tok; v += blockDim.x) {
            const int which = v >= per_kv;                  // 0 = K, 1 = V
            const int rr = v - which * per_kv;
            const int h = rr >> p.vec_shift;
            const int c = rr & (vpr - 1);
            const uint4 val = __ldg((which ? vsrc : ksrc) + rr);
            const int64_t dst = (((blk * p.num_kv_heads + h) * 2 + which) * kBlock + off) * vpr + c;
            p.cache[dst] = val;
        }
    }
}

// The same scatter into an E4M3 cache: element x is stored as the E4M3 code
// nearest to the fp32 quotient x / scale (ties to even, held at +-448).
// Each thread turns one 16-byte vector of 8 bf16 into 8 bytes.
__global__ void __launch_bounds__(256) kv_write_fp8_kernel(KvWriteParams p, float k_scale, float v_scale) {
    pdl_trigger();
    const int vpr = 1 << p.vec_shift;                      // 16-byte input vectors per head row
    const int per_kv = p.num_kv_heads * vpr;
    const int per_tok = 2 * per_kv;
    uint2 *cache8 = reinterpret_cast<uint2 *>(p.cache);    // 8-byte output vectors
    for (int64_t t = blockIdx.x; t < p.num_tokens; t += gridDim.x) {
        const int64_t slot = __ldg(p.slots + t);
        if (slot < 0) continue;
        if (slot >= p.num_slots) {
            if (threadIdx.x == 0) set_status(p.status, PKV_ERR_DEVICE_INDEX);
            continue;
        }
        const int64_t blk = slot / kBlock;
        const int64_t off = slot - blk * kBlock;
        const uint4 *ksrc = p.key + t * p.key_stride_v;
        const uint4 *vsrc = p.value + t * p.value_stride_v;
        for (int v = threadIdx.x; v < per_tok; v += blockDim.x) {
            const int which = v >= per_kv;
            const int rr = v - which * per_kv;
            const int h = rr >> p.vec_shift;
            const int c = rr & (vpr - 1);
            const uint4 val = __ldg((which ? vsrc : ksrc) + rr);
            const float s = which ? v_scale : k_scale;
            const uint32_t w[4] = {val.x, val.y, val.z, val.w};
            uint32_t packed[2];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                uint32_t out = 0;
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const uint32_t pair = w[2 * i + j];
                    float2 f;
                    f.x = __fdiv_rn(__uint_as_float(pair << 16), s);
                    f.y = __fdiv_rn(__uint_as_float(pair & 0xFFFF0000u), s);
                    const __nv_fp8x2_storage_t q = __nv_cvt_float2_to_fp8x2(f, __NV_SATFINITE, __NV_E4M3);
                    out |= static_cast<uint32_t>(q) << (16 * j);
                }
                packed[i] = out;
            }
            const int64_t dst = (((blk * p.num_kv_heads + h) * 2 + which) * kBlock + off) * vpr + c;
            cache8[dst] = make_uint2(packed[0], packed[1]);
        }
    }
}

// Copy-on-write block copies: one CTA per (pair, kv head); the K and V pages
// of one kv head are one contiguous run of 2*16*head_size bf16.
__global__ void __launch_bounds__(256) copy_blocks_kernel(uint4 *cache, int64_t num_blocks, int32_t num_kv_heads,
                                                          int32_t vec_per_page, const int64_t *mapping,
                                                          int32_t num_pairs, int32_t *status) {
    const int64_t unit = blockIdx.x;
    const int64_t pair = unit / num_kv_heads;
    const int64_t h = unit - pair * num_kv_heads;
    if (pair >= num_pairs) return;
    const int64_t src = __ldg(mapping + 2 * pair), dst = __ldg(mapping + 2 * pair + 1);
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
        if (threadIdx.x == 0 && h == 0) set_status(status, PKV_ERR_DEVICE_INDEX);
        return;
    }
    if (src == dst) return;
    const uint4 *s = cache + (src * num_kv_heads + h) * vec_per_page;
    uint4 *d = cache + (dst * num_kv_heads + h) * vec_per_page;
    for (int v = threadIdx.x; v < vec_per_page; v += blockDim.x) d[v] = __ldg(s + v);
}

}  // namespace pkv

extern "C" int pkv_copy_blocks(void *kv_cache, int64_t num_blocks, int32_t num_kv_heads, int32_t head_size,
                               int32_t block_size, const int64_t *block_mapping, int32_t num_pairs,
                               int32_t *device_status, void *stream) {
    using namespace pkv;
    if (num_pairs < 0 || num_kv_heads <= 0 || num_blocks <= 0) return PKV_ERR_SHAPE;
    if (block_size != kBlock || (head_size != 64 && head_size != 128)) return PKV_ERR_UNSUPPORTED;
    if (num_pairs == 0) return PKV_OK;
    if (!kv_cache || !block_mapping) return PKV_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(kv_cache) & 15u) || (reinterpret_cast<uintptr_t>(block_mapping) & 7u))
        return PKV_ERR_ALIGNMENT;
    const int64_t units = static_cast<int64_t>(num_pairs) * num_kv_heads;
    if (units > 0x7fffffffLL) return PKV_ERR_SHAPE;
    const int32_t vec_per_page = 2 * kBlock * head_size / 8;
    copy_blocks_kernel<<<static_cast<unsigned>(units), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<uint4 *>(kv_cache), num_blocks, num_kv_heads, vec_per_page, block_mapping, num_pairs,
        device_status);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

extern "C" int pkv_kv_write(void *kv_cache, int64_t num_blocks, int32_t num_kv_heads, int32_t head_size,
                            int32_t block_size, const void *key, int64_t key_token_stride, const void *value,
                            int64_t value_token_stride, const int64_t *slot_mapping, int32_t num_tokens,
                            int32_t *device_status, void *stream) {
    using namespace pkv;
    if (num_tokens < 0 || num_kv_heads <= 0 || num_blocks <= 0) return PKV_ERR_SHAPE;
    if (block_size != kBlock || (head_size != 64 && head_size != 128)) return PKV_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PKV_OK;
    if (!kv_cache || !key || !value || !slot_mapping) return PKV_ERR_NULL;
    const int64_t row = static_cast<int64_t>(num_kv_heads) * head_size;
    if (key_token_stride < row || value_token_stride < row) return PKV_ERR_SHAPE;
    if ((key_token_stride % 8) || (value_token_stride % 8)) return PKV_ERR_ALIGNMENT;
    if ((reinterpret_cast<uintptr_t>(kv_cache) | reinterpret_cast<uintptr_t>(key) |
         reinterpret_cast<uintptr_t>(value)) & 15u)
        return PKV_ERR_ALIGNMENT;
    if (reinterpret_cast<uintptr_t>(slot_mapping) & 7u) return PKV_ERR_ALIGNMENT;
    if (num_blocks > (INT64_MAX / kBlock)) return PKV_ERR_SHAPE;

    KvWriteParams p;
    p.cache = static_cast<uint4 *>(kv_cache);
    p.num_slots = num_blocks * kBlock;
    p.key = static_cast<const uint4 *>(key);
    p.value = static_cast<const uint4 *>(value);
    p.key_stride_v = key_token_stride / 8;
    p.value_stride_v = value_token_stride / 8;
    p.slots = slot_mapping;
    p.num_tokens = num_tokens;
    p.num_kv_heads = num_kv_heads;
    p.vec_shift = head_size == 128 ? 4 : 3;
    p.status = device_status;

    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return PKV_ERR_CUDA;
    const int threads = 256;
    int64_t blocks = num_tokens;
    const int64_t cap = static_cast<int64_t>(sms) * 8;      // 8 resident 256-thread CTAs per SM
    if (blocks > cap) blocks = cap;
    kv_write_kernel<<<static_cast<unsigned>(blocks), threads, 0, static_cast<cudaStream_t>(stream)>>>(p);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

extern "C" int pkv_kv_write_fp8(void *kv_cache, int64_t num_blocks, int32_t num_kv_heads, int32_t head_size,
                                int32_t block_size, const void *key, int64_t key_token_stride, const void *value,
                                int64_t value_token_stride, const int64_t *slot_mapping, int32_t num_tokens,
                                float k_scale, float v_scale, int32_t *device_status, void *stream) {
    using namespace pkv;
    if (num_tokens < 0 || num_kv_heads <= 0 || num_blocks <= 0) return PKV_ERR_SHAPE;
    if (block_size != kBlock || (head_size != 64 && head_size != 128)) return PKV_ERR_UNSUPPORTED;
    if (!(k_scale > 0.f) || !(v_scale > 0.f) || k_scale > 3.0e38f || v_scale > 3.0e38f) return PKV_ERR_SHAPE;
    if (num_tokens == 0) return PKV_OK;
    if (!kv_cache || !key || !value || !slot_mapping) return PKV_ERR_NULL;
    const int64_t row = static_cast<int64_t>(num_kv_heads) * head_size;
    if (key_token_stride < row || value_token_stride < row) return PKV_ERR_SHAPE;
    if ((key_token_stride % 8) || (value_token_stride % 8)) return PKV_ERR_ALIGNMENT;
    if ((reinterpret_cast<uintptr_t>(kv_cache) | reinterpret_cast<uintptr_t>(key) |
         reinterpret_cast<uintptr_t>(value)) & 15u)
        return PKV_ERR_ALIGNMENT;
    if (reinterpret_cast<uintptr_t>(slot_mapping) & 7u) return PKV_ERR_ALIGNMENT;
    if (num_blocks > (INT64_MAX / kBlock)) return PKV_ERR_SHAPE;

    KvWriteParams p;
    p.cache = static_cast<uint4 *>(kv_cache);
    p.num_slots = num_blocks * kBlock;
    p.key = static_cast<const uint4 *>(key);
    p.value = static_cast<const uint4 *>(value);
    p.key_stride_v = key_token_stride / 8;
    p.value_stride_v = value_token_stride / 8;
    p.slots = slot_mapping;
    p.num_tokens = num_tokens;
    p.num_kv_heads = num_kv_heads;
    p.vec_shift = head_size == 128 ? 4 : 3;
    p.status = device_status;

    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return PKV_ERR_CUDA;
    int64_t blocks = num_tokens;
    const int64_t cap = static_cast<int64_t>(sms) * 8;
    if (blocks > cap) blocks = cap;
    kv_write_fp8_kernel<<<static_cast<unsigned>(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(p, k_scale,
                                                                                                         v_scale);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
