// pa_small_ops.cu -- pa_cache_write, pa_copy_blocks, pa_status_string.
//
// Both kernels move bytes unchanged with 16-byte vector loads and stores:
//   - cache write: a grid over (new token, 16-byte chunk group); the token's
//     Hkv rows of K and of V (Hkv * head_dim * 2 bytes each) go to block
//     slot/B, offset slot%B for block size B
//     [Efficient Memory Management for Large Language Model Serving with
//     PagedAttention, "Kernel-Level Optimizations", 1. fused reshape and
//     block write].
//   - block copy: a grid over (pair, layer x {K, V}, chunk); every CTA copies
//     one contiguous chunk of one block, so all pairs and layers go in a
//     single launch [same section, 3. fused block copy].
//   - swap: the same kernel between two pools, the GPU pool and a CPU swap
//     space in pinned host memory, either way.  On this machine the GPU
//     reaches host memory coherently over NVLink-C2C, so the kernel loads and
//     stores it directly: one launch moves every block of every layer, where
//     a copy engine would need one transfer per block and layer
//     [Efficient Memory Management ..., "Scheduling and Preemption":
//     swapping evicted blocks to CPU RAM and back].
#include <cuda_runtime.h>

#include <cstdint>

#include "pa.h"
#include "pa_launch.cuh"
#include "pa_nvtx.cuh"
#include "pa_ptx.cuh"

namespace {

constexpr int kWriteThreads = 256;

// grid (token, chunk group): every thread moves one 16-byte chunk of the
// token's K rows and the same chunk of its V rows.
__global__ void __launch_bounds__(kWriteThreads) cache_write_kernel(
    const uint4 *__restrict__ key, const uint4 *__restrict__ value, uint4 *__restrict__ k_cache,
    uint4 *__restrict__ v_cache, const int64_t *__restrict__ slot_mapping, long long num_slots,
    int block_shift, int num_kv_heads, int chunks_per_row, unsigned int *err) {
    pa::pdl_trigger();
    pa::pdl_wait();  // earlier kernels on the stream may still read or write the pools
    const int t = blockIdx.x;
    const int i = blockIdx.y * kWriteThreads + threadIdx.x;
    const int total = num_kv_heads * chunks_per_row;
    const int64_t slot = slot_mapping[t];
    if (slot < 0) return;                                  // padding token
    if (slot >= num_slots) {
        if (i == 0 && err) atomicOr(err, PA_ERRBIT_SLOT_OOB);
        return;
    }
    if (i >= total) return;
    const int64_t blk = slot >> block_shift, off = slot & ((1 << block_shift) - 1);
    const int h = i / chunks_per_row, c = i - h * chunks_per_row;
    const size_t src = (size_t)t * total + i;
    const size_t dst =
        ((((size_t)blk * num_kv_heads + h) << block_shift) + off) * chunks_per_row + c;
    const uint4 kv = __ldcs(key + src);
    const uint4 vv = __ldcs(value + src);
    k_cache[dst] = kv;
    v_cache[dst] = vv;
}

// Source and destination pools of every layer (the same arrays for a copy
// within one pool).
struct LayerPools {
    const uint4 *src_k[PA_MAX_LAYERS];
    const uint4 *src_v[PA_MAX_LAYERS];
    uint4 *dst_k[PA_MAX_LAYERS];
    uint4 *dst_v[PA_MAX_LAYERS];
};

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;

__global__ void __launch_bounds__(kCopyThreads) copy_blocks_kernel(
    const LayerPools pools, const int64_t *__restrict__ pairs, int num_src_blocks,
    int num_dst_blocks, int same_pool, long long chunks_per_block, long long chunks_per_cta,
    unsigned int *err) {
    pa::pdl_trigger();
    pa::pdl_wait();  // earlier kernels on the stream may still read or write the pools
    const int pair = blockIdx.x;
    const int layer = blockIdx.y >> 1;
    const int which = blockIdx.y & 1;
    const int64_t src = pairs[2 * pair], dst = pairs[2 * pair + 1];
    if (src < 0 || src >= num_src_blocks || dst < 0 || dst >= num_dst_blocks) {
        if (threadIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && err)
            atomicOr(err, PA_ERRBIT_BLOCK_OOB);
        return;
    }
    if (same_pool && src == dst) return;
    const uint4 *s = (which ? pools.src_v[layer] : pools.src_k[layer]) +
                     (size_t)src * chunks_per_block;
    uint4 *d = (which ? pools.dst_v[layer] : pools.dst_k[layer]) + (size_t)dst * chunks_per_block;
    const long long c0 = (long long)blockIdx.z * chunks_per_cta;
    long long c1 = c0 + chunks_per_cta;
    if (c1 > chunks_per_block) c1 = chunks_per_block;
    long long i = c0 + threadIdx.x;
    for (; i + (kCopyUnroll - 1) * kCopyThreads < c1; i += kCopyUnroll * kCopyThreads) {
        uint4 r[kCopyUnroll];
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) r[u] = __ldcs(s + i + u * kCopyThreads);
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) __stcs(d + i + u * kCopyThreads, r[u]);
    }
    for (; i < c1; i += kCopyThreads) __stcs(d + i, __ldcs(s + i));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool head_dim_ok(int d) { return d == 64 || d == 128 || d == 256; }

// One launch of copy_blocks_kernel over every pair and layer.
pa_status_t launch_move(const LayerPools &pools, int num_layers, const int64_t *block_pairs,
                        int num_pairs, int num_src_blocks, int num_dst_blocks, int same_pool,
                        int block_size, int num_kv_heads, int head_dim,
                        unsigned int *dev_error_word, pa_stream_t stream) {
    const long long chunks_per_block = (long long)num_kv_heads * block_size * head_dim * 2 / 16;
    // about 32 KiB per CTA: enough bytes in flight per CTA, enough CTAs per copy
    const long long chunks_per_cta = 2048;
    const long long splits = (chunks_per_block + chunks_per_cta - 1) / chunks_per_cta;
    if (splits > 65535) return PA_ERR_UNSUPPORTED;
    const dim3 grid((unsigned)num_pairs, (unsigned)(2 * num_layers), (unsigned)splits);
    const cudaError_t e =
        pa::launch_pdl(copy_blocks_kernel, grid, dim3(kCopyThreads), 0, (cudaStream_t)stream,
                       pools, block_pairs, num_src_blocks, num_dst_blocks, same_pool,
                       chunks_per_block, chunks_per_cta, dev_error_word);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

// The address kernels on the current device use for a pool pointer: device
// and managed memory as given, pinned host memory through its mapping; null
// for memory the device cannot reach (pageable host memory, another device).
const void *device_view(const void *p, int dev) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        (void)cudaGetLastError();  // not a CUDA pointer: clear the error
        return nullptr;
    }
    if (a.type == cudaMemoryTypeDevice) return a.device == dev ? p : nullptr;
    if (a.type == cudaMemoryTypeManaged) return p;
    if (a.type == cudaMemoryTypeHost) return a.devicePointer;
    return nullptr;
}

// log2 of a supported block size, or -1
int block_shift_of(int b) {
    for (int sh = 3; sh <= 8; ++sh)
        if (b == (1 << sh)) return sh;
    return -1;
}

}  // namespace

extern "C" pa_status_t pa_cache_write_ex(const void *key, const void *value, void *k_cache,
                                         void *v_cache, const int64_t *slot_mapping,
                                         int num_tokens, int num_blocks, int block_size,
                                         int num_kv_heads, int head_dim, pa_dtype_t dtype,
                                         unsigned int *dev_error_word, pa_stream_t stream) {
    PA_NVTX_RANGE("pa_cache_write_ex");
    if (num_tokens < 0 || num_blocks <= 0 || num_kv_heads <= 0) return PA_ERR_INVALID_ARG;
    const int shift = block_shift_of(block_size);
    if (shift < 0) return PA_ERR_UNSUPPORTED;
    if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_INVALID_ARG;
    if (!head_dim_ok(head_dim)) return PA_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PA_OK;
    if (!key || !value || !k_cache || !v_cache || !slot_mapping) return PA_ERR_INVALID_ARG;
    if (!aligned16(key) || !aligned16(value) || !aligned16(k_cache) || !aligned16(v_cache))
        return PA_ERR_INVALID_ARG;
    const int chunks_per_row = head_dim * 2 / 16;
    const int groups = (num_kv_heads * chunks_per_row + kWriteThreads - 1) / kWriteThreads;
    if (groups > 65535) return PA_ERR_UNSUPPORTED;
    const cudaError_t e = pa::launch_pdl(
        cache_write_kernel, dim3((unsigned)num_tokens, (unsigned)groups), dim3(kWriteThreads), 0,
        (cudaStream_t)stream, (const uint4 *)key, (const uint4 *)value, (uint4 *)k_cache,
        (uint4 *)v_cache, slot_mapping, (long long)num_blocks << shift, shift, num_kv_heads,
        chunks_per_row, dev_error_word);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

extern "C" pa_status_t pa_cache_write(const void *key, const void *value, void *k_cache,
                                      void *v_cache, const int64_t *slot_mapping, int num_tokens,
                                      int num_blocks, int num_kv_heads, int head_dim,
                                      pa_dtype_t dtype, unsigned int *dev_error_word,
                                      pa_stream_t stream) {
    PA_NVTX_RANGE("pa_cache_write");
    return pa_cache_write_ex(key, value, k_cache, v_cache, slot_mapping, num_tokens, num_blocks,
                             PA_BLOCK_SIZE, num_kv_heads, head_dim, dtype, dev_error_word,
                             stream);
}

extern "C" pa_status_t pa_copy_blocks_ex(void *const *k_caches, void *const *v_caches,
                                         int num_layers, const int64_t *block_pairs,
                                         int num_pairs, int num_blocks, int block_size,
                                         int num_kv_heads, int head_dim, pa_dtype_t dtype,
                                         unsigned int *dev_error_word, pa_stream_t stream) {
    PA_NVTX_RANGE("pa_copy_blocks_ex");
    if (num_layers <= 0 || num_pairs < 0 || num_blocks <= 0 || num_kv_heads <= 0)
        return PA_ERR_INVALID_ARG;
    if (block_shift_of(block_size) < 0) return PA_ERR_UNSUPPORTED;
    if (num_layers > PA_MAX_LAYERS) return PA_ERR_UNSUPPORTED;
    if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_INVALID_ARG;
    if (!head_dim_ok(head_dim)) return PA_ERR_UNSUPPORTED;
    if (num_pairs == 0) return PA_OK;
    if (!k_caches || !v_caches || !block_pairs) return PA_ERR_INVALID_ARG;
    LayerPools pools = {};
    for (int l = 0; l < num_layers; ++l) {
        if (!k_caches[l] || !v_caches[l] || !aligned16(k_caches[l]) || !aligned16(v_caches[l]))
            return PA_ERR_INVALID_ARG;
        pools.src_k[l] = pools.dst_k[l] = (uint4 *)k_caches[l];
        pools.src_v[l] = pools.dst_v[l] = (uint4 *)v_caches[l];
    }
    return launch_move(pools, num_layers, block_pairs, num_pairs, num_blocks, num_blocks, 1,
                       block_size, num_kv_heads, head_dim, dev_error_word, stream);
}

extern "C" pa_status_t pa_copy_blocks(void *const *k_caches, void *const *v_caches,
                                      int num_layers, const int64_t *block_pairs, int num_pairs,
                                      int num_blocks, int num_kv_heads, int head_dim,
                                      pa_dtype_t dtype, unsigned int *dev_error_word,
                                      pa_stream_t stream) {
    PA_NVTX_RANGE("pa_copy_blocks");
    return pa_copy_blocks_ex(k_caches, v_caches, num_layers, block_pairs, num_pairs, num_blocks,
                             PA_BLOCK_SIZE, num_kv_heads, head_dim, dtype, dev_error_word,
                             stream);
}

extern "C" pa_status_t pa_swap_blocks(void *const *dst_k_caches, void *const *dst_v_caches,
                                      const void *const *src_k_caches,
                                      const void *const *src_v_caches, int num_layers,
                                      const int64_t *block_pairs, int num_pairs,
                                      int num_dst_blocks, int num_src_blocks, int block_size,
                                      int num_kv_heads, int head_dim, pa_dtype_t dtype,
                                      unsigned int *dev_error_word, pa_stream_t stream) {
    PA_NVTX_RANGE("pa_swap_blocks");
    if (num_layers <= 0 || num_pairs < 0 || num_dst_blocks <= 0 || num_src_blocks <= 0 ||
        num_kv_heads <= 0)
        return PA_ERR_INVALID_ARG;
    if (num_layers > PA_MAX_LAYERS) return PA_ERR_UNSUPPORTED;
    if (block_shift_of(block_size) < 0) return PA_ERR_UNSUPPORTED;
    if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_INVALID_ARG;
    if (!head_dim_ok(head_dim)) return PA_ERR_UNSUPPORTED;
    if (num_pairs == 0) return PA_OK;
    if (!dst_k_caches || !dst_v_caches || !src_k_caches || !src_v_caches || !block_pairs)
        return PA_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
    const int64_t *pairs = static_cast<const int64_t *>(device_view(block_pairs, dev));
    if (!pairs) return PA_ERR_INVALID_ARG;
    LayerPools pools = {};
    for (int l = 0; l < num_layers; ++l) {
        const void *sk = src_k_caches[l], *sv = src_v_caches[l];
        const void *dk = dst_k_caches[l], *dv = dst_v_caches[l];
        if (!sk || !sv || !dk || !dv) return PA_ERR_INVALID_ARG;
        sk = device_view(sk, dev);
        sv = device_view(sv, dev);
        dk = device_view(dk, dev);
        dv = device_view(dv, dev);
        if (!sk || !sv || !dk || !dv) return PA_ERR_INVALID_ARG;
        if (!aligned16(sk) || !aligned16(sv) || !aligned16(dk) || !aligned16(dv))
            return PA_ERR_INVALID_ARG;
        pools.src_k[l] = (const uint4 *)sk;
        pools.src_v[l] = (const uint4 *)sv;
        pools.dst_k[l] = (uint4 *)dk;
        pools.dst_v[l] = (uint4 *)dv;
    }
    return launch_move(pools, num_layers, pairs, num_pairs, num_src_blocks, num_dst_blocks, 0, block_size, num_kv_heads, head_dim, dev_error_word,
                       stream);
}

extern "C" const char *pa_status_string(pa_status_t s) {
    switch (s) {
        case PA_OK: return "PA_OK";
        case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
        case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
        case PA_ERR_CUDA: return "PA_ERR_CUDA";
        case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE";
        case PA_ERR_TIMEOUT: return "PA_ERR_TIMEOUT";
        case PA_ERR_NO_BLOCKS: return "PA_ERR_NO_BLOCKS";
    }
    return "PA_ERR_UNKNOWN";
}
