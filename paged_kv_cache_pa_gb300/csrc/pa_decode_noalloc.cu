// pa_decode_noalloc.cu -- pa_decode_attention_noalloc: paged decode attention
// for callers that cannot allocate device memory.
//
// Some callers of this library cannot call cudaMalloc (or any allocator) at
// the point where they run attention: code executing inside another engine's
// execution phase (inference-engine plugins whose enqueue step must not
// allocate, because all memory is planned when the engine is built), and C
// callers whose device allocator belongs to a host framework they cannot
// reach.  They still own their inputs and outputs, but have no way to provide
// the decode workspace.  This entry point supplies it from a fixed array that
// lives inside the library.
//
// The array is PA_NOALLOC_WORKSPACE_BYTES of device memory.  Every GPU on
// which this library's device code is loaded holds that memory until the
// process exits.  All calls on a device share it, and it keeps whatever the
// last call left there.  The decode path needs nothing in it to start at
// zero: each call rewrites the part it reads (the claim counter and the work
// list) before use.  Two calls whose work overlaps on the GPU (for example
// on two streams without ordering between them) race on the array and give
// wrong results; order them on one stream.
#include <cuda_runtime.h>

#include "pa.h"
#include "pa_nvtx.cuh"

namespace {

// Device-side scratch for pa_decode_attention_noalloc.  In host code this name
// is only a stand-in for the symbol: its device address comes from
// cudaGetSymbolAddress, with the caller's device (and context) current.
static __device__ __align__(256) unsigned char g_noalloc_workspace[PA_NOALLOC_WORKSPACE_BYTES];

}  // namespace

extern "C" pa_status_t pa_decode_attention_noalloc(
    void *out, pa_dtype_t out_dtype, const void *query, const void *k_cache, const void *v_cache,
    const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens,
    int max_context_len, int num_seqs, int num_heads, int num_kv_heads, int head_dim,
    int num_blocks, float scale, pa_dtype_t dtype, unsigned int *dev_error_word,
    pa_stream_t stream) {
    PA_NVTX_RANGE("pa_decode_attention_noalloc");
    // The array's address is looked up on every call, in the context current
    // now: after a device reset, or under another context, the library's
    // device code is loaded again and the array can move.  The first lookup
    // in a context loads the library's device code there; later ones are a
    // host-side table lookup.
    void *ws = nullptr;
    if (cudaGetSymbolAddress(&ws, g_noalloc_workspace) != cudaSuccess || !ws) return PA_ERR_CUDA;
    // pa_decode_attention checks every argument first, in its own order, and
    // returns PA_ERR_WORKSPACE only for otherwise valid sizes whose workspace
    // exceeds the array.
    return pa_decode_attention(out, out_dtype, query, k_cache, v_cache, block_tables,
                               max_blocks_per_seq, context_lens, max_context_len, num_seqs,
                               num_heads, num_kv_heads, head_dim, num_blocks, scale, dtype, ws,
                               (size_t)PA_NOALLOC_WORKSPACE_BYTES, dev_error_word, stream);
}
