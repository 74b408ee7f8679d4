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
// zero: the plan kernel of each call rewrites the part it reads (the claim
// counter and the work list) before use.  Two calls whose work overlaps on
// the GPU (for example on two streams without ordering between them) race on
// the array and give wrong results; order them on one stream.
#include <cuda_runtime.h>

#include <mutex>

#include "pa.h"

namespace {

// Device-side scratch for pa_decode_attention_noalloc.  In host code this name
// is only a stand-in for the symbol: its device address comes from
// cudaGetSymbolAddress, done once per device below.
static __device__ __align__(256) unsigned char g_noalloc_workspace[PA_NOALLOC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_workspace_addr[kMaxDevices];  // device address of the array, per device

}  // namespace

extern "C" pa_status_t pa_decode_attention_noalloc(
    void *out, pa_dtype_t out_dtype, const void *query, const void *k_cache, const void *v_cache,
    const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens,
    int max_context_len, int num_seqs, int num_heads, int num_kv_heads, int head_dim,
    int num_blocks, float scale, pa_dtype_t dtype, unsigned int *dev_error_word,
    pa_stream_t stream) {
    const size_t need = pa_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim,
                                                 max_context_len);
    if (need > (size_t)PA_NOALLOC_WORKSPACE_BYTES) return PA_ERR_WORKSPACE;

    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return PA_ERR_UNSUPPORTED;
    void *ws = nullptr;
    {
        // First call on this device, with the device current: look up the
        // array's device address (this may load the library's device code).
        std::lock_guard<std::mutex> lock(g_mu);
        if (!g_workspace_addr[dev]) {
            void *addr = nullptr;
            if (cudaGetSymbolAddress(&addr, g_noalloc_workspace) != cudaSuccess || !addr)
                return PA_ERR_CUDA;
            g_workspace_addr[dev] = addr;
        }
        ws = g_workspace_addr[dev];
    }
    return pa_decode_attention(out, out_dtype, query, k_cache, v_cache, block_tables,
                               max_blocks_per_seq, context_lens, max_context_len, num_seqs,
                               num_heads, num_kv_heads, head_dim, num_blocks, scale, dtype, ws,
                               (size_t)PA_NOALLOC_WORKSPACE_BYTES, dev_error_word, stream);
}
