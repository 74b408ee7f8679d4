// pa_decode_api.cu -- pa_decode_attention / pa_decode_workspace_size /
// pa_decode_partition_tokens: the plan kernel, the partition merge kernel and
// the host-side checks and launches.
//
// Context split: a sequence longer than part_tokens is cut into partitions of
// part_tokens tokens; every (sequence, partition, KV head) is an independent
// work item whose partial softmax state (max m, sum l, weighted values acc)
// is merged exactly afterwards by the merge kernel:
//     M = max_p m_p,  L = sum_p l_p 2^(m_p - M),  o = sum_p acc_p 2^(m_p - M) / L
// [vLLM Internals ..., "The kernel pays for the indirection": a grid axis over
// partitions; Paged Attention: Managing the KV Cache Like Virtual Memory,
// "Attention over scattered blocks": slices and a merge kernel; Efficient
// Memory Management ..., "PagedAttention Algorithm": blocks may be processed
// in any order and combined].
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cstring>

#include "pa_decode.cuh"
#include "pa_launch.cuh"
#include "pa_tmap.cuh"

namespace pa {

namespace {

constexpr int kMinPartTokens = 64;
constexpr long long kTargetItems = 2048;  // ~ 152 SMs x resident CTAs x a few items each

int choose_part_tokens(int num_seqs, int num_kv_heads, int max_context_len) {
    int p = kMaxPartTokens;
    const long long units = (long long)num_seqs * num_kv_heads;
    while (p > kMinPartTokens) {
        const long long items = units * ((max_context_len + p - 1) / p);
        if (items >= kTargetItems) break;
        p /= 2;
    }
    return p;
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

struct WsLayout {
    int part_tokens, max_parts;
    size_t items_off, m_off, l_off, acc_off, bytes;
};

WsLayout ws_layout(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                   int max_context_len) {
    WsLayout w;
    w.part_tokens = choose_part_tokens(num_seqs, num_kv_heads, max_context_len);
    w.max_parts = max_context_len > 0 ? (max_context_len + w.part_tokens - 1) / w.part_tokens : 1;
    size_t off = align256(sizeof(WsHeader));
    w.items_off = off;
    off = align256(off + (size_t)num_seqs * w.max_parts * sizeof(int4));
    if (w.max_parts > 1) {
        const size_t n = (size_t)num_seqs * num_heads * w.max_parts;
        w.m_off = off;
        off = align256(off + n * 4);
        w.l_off = off;
        off = align256(off + n * 4);
        w.acc_off = off;
        off = align256(off + n * head_dim * 4);
    } else {
        w.m_off = w.l_off = w.acc_off = off;
    }
    w.bytes = off;
    return w;
}

// One CTA: count (sequence, partition) pairs by size, lay them out longest
// first (a counting sort on the number of blocks), reset the claim counter,
// and zero the output rows of empty sequences.  Sequences are taken 1024 at
// a time, one per thread; shared-memory counters are bumped once per warp
// and size (warp-aggregated), so threads do not queue on one address.
//
// The work list is built before the programmatic-dependent-launch wait, so
// it overlaps the kernel before this call on the stream (typically the cache
// write); only the output rows wait for it.  Reading context_lens that early
// is safe because it is an input: a kernel that wrote it has completed before
// this grid starts, unless that kernel let dependents launch before writing
// it.  Writing the work list that early is safe because the attention
// kernels of earlier calls that share the workspace have finished with it:
// their producers read it, and release the claim counter with a fence,
// before they allow dependents to launch.
constexpr int kPlanThreads = 1024;

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(
    const int32_t *__restrict__ lens, int num_seqs, int max_context_len, int part_tokens,
    int num_kv_heads, int num_heads, int head_dim, int4 *__restrict__ items, WsHeader *hdr,
    void *out, int out_dtype, unsigned int *err) {
    pdl_trigger();  // the attention CTAs may start their set-up now
    constexpr int kKeys = kMaxPartTokens / kBlock + 1;
    __shared__ int hist[kKeys];
    __shared__ int offs[kKeys];
    const int PB = part_tokens / kBlock;
    const int tid = threadIdx.x, lane = tid & 31;
    const unsigned lt_mask = (1u << lane) - 1u;
    if (tid < kKeys) hist[tid] = 0;
    __syncthreads();
    // pass 1: histogram of partition sizes (in blocks)
    for (int s0 = 0; s0 < num_seqs; s0 += kPlanThreads) {
        const int s = s0 + tid;
        int L = s < num_seqs ? lens[s] : 1;
        const bool bad = L < 0 || L > max_context_len;
        if (bad && s < num_seqs && err) atomicOr(err, PA_ERRBIT_CONTEXT_LEN);
        if (bad) L = 0;
        const bool live = s < num_seqs && L > 0;
        const int np = live ? (L + part_tokens - 1) / part_tokens : 0;
        // full partitions: one add per warp
        int full = np > 1 ? np - 1 : 0;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) full += __shfl_xor_sync(0xffffffffu, full, off);
        if (lane == 0 && full) atomicAdd(&hist[PB], full);
        // last partitions: one add per distinct size in the warp
        const int key = live ? (L - (np - 1) * part_tokens + kBlock - 1) / kBlock : 0;
        const unsigned same = __match_any_sync(0xffffffffu, key);
        if (live && (same & lt_mask) == 0) atomicAdd(&hist[key], __popc(same));
    }
    __syncthreads();
    if (tid < 32) {  // exclusive scan over sizes, largest first
        const int key = PB - tid;
        const int v = (tid < PB) ? hist[key] : 0;
        int incl = v;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, incl, off);
            if (tid >= off) incl += u;
        }
        if (tid < PB) offs[key] = incl - v;
        if (tid == 31) {
            hdr->counter = 0u;
            hdr->n_items = (unsigned)incl * (unsigned)num_kv_heads;
        }
    }
    __syncthreads();
    // pass 2: place every (sequence, partition)
    for (int s0 = 0; s0 < num_seqs; s0 += kPlanThreads) {
        const int s = s0 + tid;
        const int L0 = s < num_seqs ? lens[s] : 0;
        const bool live = s < num_seqs && L0 > 0 && L0 <= max_context_len;
        const int L = live ? L0 : 0;
        const int np = live ? (L + part_tokens - 1) / part_tokens : 0;
        // full partitions of the warp: contiguous range from one add
        const int full = np > 1 ? np - 1 : 0;
        int incl = full;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += u;
        }
        const int total = __shfl_sync(0xffffffffu, incl, 31);
        int base = 0;
        if (lane == 31 && total) base = atomicAdd(&offs[PB], total);
        base = __shfl_sync(0xffffffffu, base, 31) + incl - full;
        for (int p = 0; p < full; ++p)
            items[base + p] = make_int4(s, p, part_tokens, np);
        // last partition: rank among the warp's lanes with the same size
        const int ntok = live ? L - (np - 1) * part_tokens : 0;
        const int key = live ? (ntok + kBlock - 1) / kBlock : 0;
        const unsigned same = __match_any_sync(0xffffffffu, key);
        const int leader = __ffs(same) - 1;
        int slot = 0;
        if (live && lane == leader) slot = atomicAdd(&offs[key], __popc(same));
        slot = __shfl_sync(0xffffffffu, slot, leader) + __popc(same & lt_mask);
        if (live) items[slot] = make_int4(s, np - 1, ntok, np);
    }
    pdl_wait();  // earlier work on the stream may still read out
    // the warp zeroes the output rows of its empty sequences together
    for (int s0 = 0; s0 < num_seqs; s0 += kPlanThreads) {
        const int s = s0 + tid;
        const int L = s < num_seqs ? lens[s] : 1;
        unsigned empty = __ballot_sync(0xffffffffu, s < num_seqs && (L <= 0 || L > max_context_len));
        while (empty) {
            const int src = __ffs(empty) - 1;
            empty &= empty - 1;
            const size_t base = (size_t)(s0 + (tid & ~31) + src) * num_heads * head_dim;
            for (int i = lane; i < num_heads * head_dim; i += 32)
                store_out(out, out_dtype, base + i, 0.f);
        }
    }
}

// One CTA per (sequence, query head) of a multi-partition sequence:
//   M = max_p m_p,  c_p = 2^(m_p - M),  L = sum_p l_p c_p,
//   o = sum_p acc_p c_p / L.
// One pass over the partials: the threads form partition groups of head_dim/4
// float4 columns each; group g folds partitions g, g + NG, ... into a running
// (M, L, o), rescaling it whenever the maximum grows, so a partition's m, l
// and acc are loaded together instead of in three dependent rounds.  The
// groups' states are then folded the same way through shared memory.
constexpr int kMergeThreads = 128;
constexpr int kMergeBatch = 4;  // partitions a thread loads before folding them

// (M, L, o) <- the merge of (M, L, o) and (mp, lp, a); an empty state has
// M = -inf (ex2(-inf) = 0 drops it).
__device__ __forceinline__ void fold_state(float &M, float &L, float4 &o, float mp, float lp,
                                           float4 a) {
    const float Mn = fmaxf(M, mp);
    if (Mn == -INFINITY) return;  // both empty
    const float c0 = ex2(M - Mn), c1 = ex2(mp - Mn);
    L = fmaf(L, c0, lp * c1);
    o.x = fmaf(o.x, c0, a.x * c1);
    o.y = fmaf(o.y, c0, a.y * c1);
    o.z = fmaf(o.z, c0, a.z * c1);
    o.w = fmaf(o.w, c0, a.w * c1);
    M = Mn;
}

template <int D>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const __grid_constant__ DecodeParams P) {
    constexpr int C = D / 4;                   // float4 columns
    constexpr int NG = kMergeThreads / C;      // partition groups
    __shared__ float s_m[NG], s_l[NG];
    __shared__ float4 s_acc[NG][C];
    const int s = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
    const int L = P.context_lens[s];  // an input: complete before this grid launched
    if (L <= P.part_tokens || L > P.max_context_len) return;  // one partition, or invalid
    const int np = (L + P.part_tokens - 1) / P.part_tokens;
    pdl_wait();  // partials from the attention kernel
    const size_t base = ((size_t)s * P.num_heads + h) * P.max_parts;
    const int col = tid % C, grp = tid / C;
    const float4 *acc = reinterpret_cast<const float4 *>(P.part_acc + base * D) + col;

    float M = -INFINITY, Lsum = 0.f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int p0 = grp; p0 < np; p0 += kMergeBatch * NG) {
        float mp[kMergeBatch], lp[kMergeBatch];
        float4 a[kMergeBatch];
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u) {
            const int p = p0 + u * NG;
            const bool in = p < np;
            mp[u] = in ? P.part_m[base + p] : -INFINITY;
            lp[u] = in ? P.part_l[base + p] : 0.f;
            a[u] = in ? acc[(size_t)p * C] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u) fold_state(M, Lsum, o, mp[u], lp[u], a[u]);
    }
    if (col == 0) {
        s_m[grp] = M;
        s_l[grp] = Lsum;
    }
    s_acc[grp][col] = o;
    __syncthreads();
    if (grp == 0) {
#pragma unroll
        for (int g = 1; g < NG; ++g) fold_state(M, Lsum, o, s_m[g], s_l[g], s_acc[g][col]);
        const size_t ob = ((size_t)s * P.num_heads + h) * D + col * 4;
        store_out(P.out, P.out_dtype, ob + 0, Lsum > 0.f ? o.x / Lsum : 0.f);
        store_out(P.out, P.out_dtype, ob + 1, Lsum > 0.f ? o.y / Lsum : 0.f);
        store_out(P.out, P.out_dtype, ob + 2, Lsum > 0.f ? o.z / Lsum : 0.f);
        store_out(P.out, P.out_dtype, ob + 3, Lsum > 0.f ? o.w / Lsum : 0.f);
    }
}

std::atomic<int> g_sm_count[64];

// 3-D view [head_dim / 64][rows][64] of a row-major [rows][head_dim] 16-bit
// tensor (strides: a row is head_dim * 2 bytes, a 64-element half 128 bytes);
// one box is box_rows rows of box_halves halves (all halves, or one),
// 128-byte swizzle; reads past the last row return zeros.
bool encode_rows(CUtensorMap *map, const void *base, pa_dtype_t dtype, unsigned long long rows,
                 int head_dim, int box_rows, int box_halves) {
    const cuuint64_t dims[3] = {64u, (cuuint64_t)rows, (cuuint64_t)(head_dim / 64)};
    const cuuint64_t strides[2] = {(cuuint64_t)head_dim * 2, 128u};
    const cuuint32_t box[3] = {64u, (cuuint32_t)box_rows, (cuuint32_t)box_halves};
    return encode_tiled(map, base, dtype, 3, dims, strides, box);
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// log2 of a supported pool block size (8 .. 256 tokens, a power of two), or -1
int block_shift_of(int b) {
    for (int sh = 3; sh <= 8; ++sh)
        if (b == (1 << sh)) return sh;
    return -1;
}

}  // namespace

int current_sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    int n = g_sm_count[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
            n = 1;
        g_sm_count[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

}  // namespace pa

using namespace pa;

extern "C" size_t pa_decode_workspace_size(int num_seqs, int num_heads, int num_kv_heads,
                                           int head_dim, int max_context_len) {
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || max_context_len < 0)
        return 0;
    return ws_layout(num_seqs, num_heads, num_kv_heads, head_dim, max_context_len).bytes;
}

extern "C" int pa_decode_partition_tokens(int num_seqs, int num_kv_heads, int max_context_len) {
    if (num_seqs < 0 || num_kv_heads <= 0 || max_context_len < 0) return 0;
    return choose_part_tokens(num_seqs, num_kv_heads, max_context_len);
}

namespace {

// Shared implementation of the paged (contig_rows == 0) and contiguous
// (contig_rows > 0) entry points.
pa_status_t decode_impl(void *out, pa_dtype_t out_dtype, const void *query, const void *k_cache,
                        const void *v_cache, const int32_t *block_tables, int max_blocks_per_seq,
                        int contig_rows, const int32_t *context_lens, int max_context_len,
                        int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                        int num_blocks, int block_size, float scale, pa_dtype_t dtype,
                        void *workspace, size_t workspace_bytes, unsigned int *dev_error_word,
                        pa_stream_t stream) {
    const int block_shift = block_shift_of(block_size);
    if (block_shift < 0) return PA_ERR_UNSUPPORTED;
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || max_context_len < 0)
        return PA_ERR_INVALID_ARG;
    if (num_heads % num_kv_heads != 0) return PA_ERR_INVALID_ARG;
    if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_INVALID_ARG;
    if (out_dtype != PA_F32 && out_dtype != dtype) return PA_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128 && head_dim != 256) return PA_ERR_UNSUPPORTED;
    if (num_heads / num_kv_heads > 8) return PA_ERR_UNSUPPORTED;
    // rows of the pool viewed as [rows][head_dim] (row coordinates are 32-bit)
    unsigned long long pool_rows;
    if (contig_rows == 0) {
        if (num_blocks <= 0 || max_blocks_per_seq <= 0) return PA_ERR_INVALID_ARG;
        if ((long long)max_context_len > (long long)block_size * max_blocks_per_seq)
            return PA_ERR_INVALID_ARG;
        pool_rows = (unsigned long long)num_blocks * num_kv_heads * block_size;
    } else {
        if (contig_rows < 0 || contig_rows % kBlock != 0 || max_context_len > contig_rows)
            return PA_ERR_INVALID_ARG;
        pool_rows = (unsigned long long)num_seqs * num_kv_heads * contig_rows;
    }
    if (pool_rows >= (1ull << 31)) return PA_ERR_UNSUPPORTED;
    if (num_seqs == 0) return PA_OK;
    if (!out || !query || !k_cache || !v_cache || !context_lens || !workspace)
        return PA_ERR_INVALID_ARG;
    if (contig_rows == 0 && !block_tables) return PA_ERR_INVALID_ARG;
    if (!aligned(out, 16) || !aligned(query, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
        return PA_ERR_INVALID_ARG;
    if (!aligned(workspace, 256)) return PA_ERR_WORKSPACE;
    const WsLayout w = ws_layout(num_seqs, num_heads, num_kv_heads, head_dim, max_context_len);
    if (workspace_bytes < w.bytes) return PA_ERR_WORKSPACE;

    unsigned char *ws = static_cast<unsigned char *>(workspace);
    DecodeParams P;
    memset(&P, 0, sizeof(P));
    if (uses_tensor_cores(num_heads / num_kv_heads, head_dim)) {
        // a 16-token chunk per box (all halves), or for 8-token blocks one
        // block's 8 rows of one 64-element half
        const bool eight = contig_rows == 0 && block_size < kBlock;
        const int box_rows = eight ? block_size : kBlock;
        const int box_halves = eight ? 1 : head_dim / 64;
        if (!encode_rows(&P.tmap_q, query, dtype, (unsigned long long)num_seqs * num_heads,
                         head_dim, 8, head_dim / 64) ||
            !encode_rows(&P.tmap_k, k_cache, dtype, pool_rows, head_dim, box_rows, box_halves) ||
            !encode_rows(&P.tmap_v, v_cache, dtype, pool_rows, head_dim, box_rows, box_halves))
            return PA_ERR_CUDA;
    }
    P.out = out;
    P.out_dtype = (int)out_dtype;
    P.q = query;
    P.k_cache = k_cache;
    P.v_cache = v_cache;
    P.block_tables = block_tables;
    P.max_blocks_per_seq = max_blocks_per_seq;
    P.block_size = block_size;
    P.block_shift = block_shift;
    P.contig_rows = contig_rows;
    P.context_lens = context_lens;
    P.max_context_len = max_context_len;
    P.num_seqs = num_seqs;
    P.num_heads = num_heads;
    P.num_kv_heads = num_kv_heads;
    P.G = num_heads / num_kv_heads;
    P.head_dim = head_dim;
    P.num_blocks = num_blocks;
    P.scale_log2 = scale * 1.4426950408889634f;
    P.part_tokens = w.part_tokens;
    P.max_parts = w.max_parts;
    P.hdr = reinterpret_cast<WsHeader *>(ws);
    P.items = reinterpret_cast<int4 *>(ws + w.items_off);
    P.part_m = reinterpret_cast<float *>(ws + w.m_off);
    P.part_l = reinterpret_cast<float *>(ws + w.l_off);
    P.part_acc = reinterpret_cast<float *>(ws + w.acc_off);
    P.err = dev_error_word;
    cudaStream_t st = (cudaStream_t)stream;

    if (launch_pdl(plan_kernel, dim3(1), dim3(kPlanThreads), 0, st, (const int32_t *)context_lens,
                   num_seqs, max_context_len, w.part_tokens, num_kv_heads, num_heads, head_dim,
                   P.items, P.hdr, out, (int)out_dtype, dev_error_word) != cudaSuccess)
        return PA_ERR_CUDA;

    long long cap = (long long)num_seqs * w.max_parts * num_kv_heads;
    if (cap > INT_MAX) cap = INT_MAX;
    pa_status_t st_launch;
    if (head_dim == 64)
        st_launch = launch_decode_d64(P, dtype, (int)cap, st);
    else if (head_dim == 128)
        st_launch = launch_decode_d128(P, dtype, (int)cap, st);
    else
        st_launch = launch_decode_d256(P, dtype, (int)cap, st);
    if (st_launch != PA_OK) return st_launch;

    if (w.max_parts > 1) {
        if (num_heads > 65535) return PA_ERR_UNSUPPORTED;
        const dim3 grid((unsigned)num_seqs, (unsigned)num_heads);
        cudaError_t e;
        if (head_dim == 64)
            e = launch_pdl(merge_kernel<64>, grid, dim3(kMergeThreads), 0, st, P);
        else if (head_dim == 128)
            e = launch_pdl(merge_kernel<128>, grid, dim3(kMergeThreads), 0, st, P);
        else
            e = launch_pdl(merge_kernel<256>, grid, dim3(kMergeThreads), 0, st, P);
        if (e != cudaSuccess) return PA_ERR_CUDA;
    }
    return PA_OK;
}

}  // namespace

extern "C" pa_status_t pa_decode_attention_ex(
    void *out, pa_dtype_t out_dtype, const void *query, const void *k_cache, const void *v_cache,
    const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens,
    int max_context_len, int num_seqs, int num_heads, int num_kv_heads, int head_dim,
    int num_blocks, int block_size, float scale, pa_dtype_t dtype, void *workspace,
    size_t workspace_bytes, unsigned int *dev_error_word, pa_stream_t stream) {
    return decode_impl(out, out_dtype, query, k_cache, v_cache, block_tables, max_blocks_per_seq,
                       0, context_lens, max_context_len, num_seqs, num_heads, num_kv_heads,
                       head_dim, num_blocks, block_size, scale, dtype, workspace,
                       workspace_bytes, dev_error_word, stream);
}

extern "C" pa_status_t pa_decode_attention(void *out, pa_dtype_t out_dtype, const void *query,
                                           const void *k_cache, const void *v_cache,
                                           const int32_t *block_tables, int max_blocks_per_seq,
                                           const int32_t *context_lens, int max_context_len,
                                           int num_seqs, int num_heads, int num_kv_heads,
                                           int head_dim, int num_blocks, float scale,
                                           pa_dtype_t dtype, void *workspace,
                                           size_t workspace_bytes, unsigned int *dev_error_word,
                                           pa_stream_t stream) {
    return decode_impl(out, out_dtype, query, k_cache, v_cache, block_tables, max_blocks_per_seq,
                       0, context_lens, max_context_len, num_seqs, num_heads, num_kv_heads,
                       head_dim, num_blocks, PA_BLOCK_SIZE, scale, dtype, workspace,
                       workspace_bytes, dev_error_word, stream);
}

extern "C" pa_status_t pa_decode_attention_contiguous(
    void *out, pa_dtype_t out_dtype, const void *query, const void *k_cache, const void *v_cache,
    int max_rows, const int32_t *context_lens, int max_context_len, int num_seqs, int num_heads,
    int num_kv_heads, int head_dim, float scale, pa_dtype_t dtype, void *workspace,
    size_t workspace_bytes, unsigned int *dev_error_word, pa_stream_t stream) {
    if (max_rows <= 0) return PA_ERR_INVALID_ARG;
    return decode_impl(out, out_dtype, query, k_cache, v_cache, nullptr, 0, max_rows,
                       context_lens, max_context_len, num_seqs, num_heads, num_kv_heads,
                       head_dim, 0, PA_BLOCK_SIZE, scale, dtype, workspace, workspace_bytes,
                       dev_error_word, stream);
}
