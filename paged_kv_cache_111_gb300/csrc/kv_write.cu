// Cache write ("reshape_and_cache"): scatter new K/V tokens into their slots;
// and the copy-on-write block copy.
//
// "vLLM internals: managing the KV cache like an OS manages memory", section
// 2.1 (the fused write op puts each new token's K/V into its physical block);
// "continuous batching and PagedAttention" tutorial, section 3.3 (token ->
// block slot / 16, offset slot % 16); "vLLM source reading", section 5.1
// (slot_mapping drives the scatter).
//
// A pure bit copy, HBM-bound: each thread moves 16-byte vectors of tokens' K
// or V rows; consecutive threads cover consecutive 16-byte pieces of a head's
// row, so reads and writes are coalesced 128-byte+ runs.
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

// The scatter is a flat loop over (token, 16-byte vector of the token's K
// then V row) pairs.  Each thread takes kWriteUnroll of them a grid stride
// apart and issues every load (slot and data) before any store: the write is
// a short chain of dependent memory operations, so its time is their latency
// unless many are in flight.
constexpr int kWriteUnroll = 4;

// Vector i of the flat loop: token t, K (0) or V (1), and the vector's index
// rr within that token's K or V row of all kv heads.
struct KvVec {
    int64_t t;
    int which, rr;
};
__device__ __forceinline__ KvVec kv_vec(int64_t i, bool narrow, int per_tok, int per_kv) {
    KvVec v;
    v.t = narrow ? static_cast<int64_t>(static_cast<uint32_t>(i) / static_cast<uint32_t>(per_tok)) : i / per_tok;
    const int e = static_cast<int>(i - v.t * per_tok);
    v.which = e >= per_kv;
    v.rr = e - v.which * per_kv;
    return v;
}

// Cache index, in units of one vector per 8 elements (16 bytes of bf16, 8
// bytes of E4M3), of vector rr of K or V of a token written to `slot`.
__device__ __forceinline__ int64_t kv_dst(const KvWriteParams &p, int64_t slot, int which, int rr) {
    const int vpr = 1 << p.vec_shift;
    const int64_t blk = slot / kBlock;
    const int64_t off = slot - blk * kBlock;
    return (((blk * p.num_kv_heads + (rr >> p.vec_shift)) * 2 + which) * kBlock + off) * vpr + (rr & (vpr - 1));
}

__global__ void __launch_bounds__(256) kv_write_kernel(KvWriteParams p) {
    pdl_trigger();                                         // the attention plan may start (it reads no cache)
    const int per_kv = p.num_kv_heads << p.vec_shift;      // vectors of K (or V) per token
    const int per_tok = 2 * per_kv;
    const int64_t total = static_cast<int64_t>(p.num_tokens) * per_tok;
    const bool narrow = total <= INT32_MAX;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i0 < total;
         i0 += kWriteUnroll * stride) {
        int64_t slot[kWriteUnroll];
        uint4 val[kWriteUnroll];
        int which[kWriteUnroll], rr[kWriteUnroll];
#pragma unroll
        for (int u = 0; u < kWriteUnroll; ++u) {
            const int64_t i = i0 + u * stride;
            slot[u] = -1;                                  // nothing to store
            if (i < total) {
                const KvVec v = kv_vec(i, narrow, per_tok, per_kv);
                which[u] = v.which;
                rr[u] = v.rr;
                slot[u] = __ldg(p.slots + v.t);
                val[u] = __ldg((v.which ? p.value + v.t * p.value_stride_v : p.key + v.t * p.key_stride_v) + v.rr);
            }
        }
#pragma unroll
        for (int u = 0; u < kWriteUnroll; ++u) {
            if (slot[u] < 0) continue;                     // padding token (or past the end)
            if (slot[u] >= p.num_slots) {
                set_status(p.status, PKV_ERR_DEVICE_INDEX);
                continue;
            }
            p.cache[kv_dst(p, slot[u], which[u], rr[u])] = val[u];
        }
    }
}

// The same scatter into an E4M3 cache: element x is stored as the E4M3 code
// nearest to the fp32 quotient x / scale (ties to even, held at +-448).
// Each vector of 8 bf16 becomes 8 bytes.
__device__ __forceinline__ uint2 bf16x8_to_e4m3(const uint4 &val, float s) {
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
    return make_uint2(packed[0], packed[1]);
}

__global__ void __launch_bounds__(256) kv_write_fp8_kernel(KvWriteParams p, float k_scale, float v_scale) {
    pdl_trigger();
    const int per_kv = p.num_kv_heads << p.vec_shift;      // 16-byte input vectors of K (or V) per token
    const int per_tok = 2 * per_kv;
    const int64_t total = static_cast<int64_t>(p.num_tokens) * per_tok;
    const bool narrow = total <= INT32_MAX;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    uint2 *cache8 = reinterpret_cast<uint2 *>(p.cache);    // 8-byte output vectors
    for (int64_t i0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i0 < total;
         i0 += kWriteUnroll * stride) {
        int64_t slot[kWriteUnroll];
        uint4 val[kWriteUnroll];
        int which[kWriteUnroll], rr[kWriteUnroll];
#pragma unroll
        for (int u = 0; u < kWriteUnroll; ++u) {
            const int64_t i = i0 + u * stride;
            slot[u] = -1;
            if (i < total) {
                const KvVec v = kv_vec(i, narrow, per_tok, per_kv);
                which[u] = v.which;
                rr[u] = v.rr;
                slot[u] = __ldg(p.slots + v.t);
                val[u] = __ldg((v.which ? p.value + v.t * p.value_stride_v : p.key + v.t * p.key_stride_v) + v.rr);
            }
        }
#pragma unroll
        for (int u = 0; u < kWriteUnroll; ++u) {
            if (slot[u] < 0) continue;
            if (slot[u] >= p.num_slots) {
                set_status(p.status, PKV_ERR_DEVICE_INDEX);
                continue;
            }
            cache8[kv_dst(p, slot[u], which[u], rr[u])] = bf16x8_to_e4m3(val[u], which[u] ? v_scale : k_scale);
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

namespace pkv {
// CTAs of the flat cache-write loop: one vector per thread where that takes
// at most 8 resident 256-thread CTAs per SM, else that many (grid-strided).
static int64_t write_grid(int64_t num_tokens, int32_t num_kv_heads, int32_t head_size, int sms, int threads) {
    const int64_t vectors = num_tokens * 2 * num_kv_heads * (head_size / 8);
    int64_t blocks = (vectors + threads - 1) / threads;
    const int64_t cap = static_cast<int64_t>(sms) * 8;
    return blocks > cap ? cap : (blocks < 1 ? 1 : blocks);
}
}  // namespace pkv

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
    const int64_t blocks = write_grid(num_tokens, num_kv_heads, head_size, sms, threads);
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
    const int64_t blocks = write_grid(num_tokens, num_kv_heads, head_size, sms, 256);
    kv_write_fp8_kernel<<<static_cast<unsigned>(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(p, k_scale,
                                                                                                         v_scale);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
