// Paged attention for callers that cannot allocate GPU memory.
//
// Some callers cannot call cudaMalloc (or any allocator) at the point where
// they run attention: code in a serving loop under a strict no-allocation
// policy, plugins of a host engine that owns all device memory and hands
// out only inputs and outputs, or embedded runtimes that forbid allocation
// after start-up.  For them this
// file offers one entry point that needs no workspace from the caller: the
// scratch that pkv_paged_attn keeps in its workspace lives instead in a
// fixed-size array of this library's own device memory.
//
// The array is a file-scope __device__ variable, so every GPU on which this
// file's device code is loaded holds PKV_NOALLOC_SCRATCH_BYTES of it until
// the process exits.  With CUDA's default lazy module loading that happens
// the first time this entry point runs on a device; with eager loading it
// happens when the library is loaded.  Host code cannot use the array's name
// as a device address: every call looks the address up with
// cudaGetSymbolAddress, with the call's device current, and passes it to the
// kernels.  The lookup is a host-side query that enqueues nothing; doing it
// on every call (instead of caching it) keeps the address right after the
// device's context has been torn down and the module loaded again.
#include "pkv_common.cuh"

namespace pkv {

static __device__ __align__(256) uint8_t g_noalloc_scratch[PKV_NOALLOC_SCRATCH_BYTES];

// The call's device status (the scratch's first word) into the caller's
// word, by the rule of every other status word of this library: the first
// error stored there stays, and the word is never cleared.
__global__ void forward_status_kernel(const int32_t *scratch_status, int32_t *device_status) {
    pdl_wait();       // the combine (and everything before it) has completed
    const int32_t s = *reinterpret_cast<const volatile int32_t *>(scratch_status);
    if (s != PKV_OK) atomicCAS(device_status, 0, s);
}

}  // namespace pkv

extern "C" int pkv_paged_attn_noalloc(void *out, const void *query, int64_t query_token_stride, const void *kv_cache,
                                      int64_t num_blocks, const int32_t *block_tables, int32_t max_blocks_per_seq,
                                      const int32_t *seq_lens, const int32_t *query_start_loc, int32_t num_seqs,
                                      int32_t num_tokens, int32_t max_query_len, int32_t max_seq_len,
                                      int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
                                      int32_t block_size, float scale, int32_t num_splits, int32_t *device_status,
                                      void *stream) {
    using namespace pkv;
    // size query: validates every argument and reports the scratch needed,
    // enqueueing nothing
    size_t need = 0;
    int rc = pkv_paged_attn(out, query, query_token_stride, kv_cache, num_blocks, block_tables,
                            max_blocks_per_seq, seq_lens, query_start_loc, num_seqs, num_tokens, max_query_len,
                            max_seq_len, num_q_heads, num_kv_heads, head_size, block_size, scale, num_splits,
                            nullptr, 0, &need, stream);
    if (rc == PKV_OK) return PKV_OK;              // nothing to do (no requests)
    if (rc != PKV_ERR_WORKSPACE) return rc;       // an argument error
    if (need > static_cast<size_t>(PKV_NOALLOC_SCRATCH_BYTES)) return PKV_ERR_WORKSPACE;

    // the array's address on the current device (the host-side name is only
    // a stand-in, never a device address)
    void *scratch = nullptr;
    if (cudaGetSymbolAddress(&scratch, g_noalloc_scratch) != cudaSuccess || !scratch) return PKV_ERR_CUDA;

    rc = pkv_paged_attn(out, query, query_token_stride, kv_cache, num_blocks, block_tables, max_blocks_per_seq,
                        seq_lens, query_start_loc, num_seqs, num_tokens, max_query_len, max_seq_len, num_q_heads,
                        num_kv_heads, head_size, block_size, scale, num_splits, scratch,
                        PKV_NOALLOC_SCRATCH_BYTES, &need, stream);
    if (rc) return rc;
    rc = pkv_paged_attn_combine(out, scratch, PKV_NOALLOC_SCRATCH_BYTES, num_tokens, num_q_heads, head_size,
                                stream);
    if (rc) return rc;
    if (device_status &&
        launch_pdl(forward_status_kernel, dim3(1), dim3(1), 0, static_cast<cudaStream_t>(stream),
                   static_cast<const int32_t *>(scratch), device_status) != cudaSuccess)
        return PKV_ERR_CUDA;
    return PKV_OK;
}
