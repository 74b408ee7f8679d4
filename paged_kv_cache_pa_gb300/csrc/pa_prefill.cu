// pa_prefill.cu -- chunked-prefill attention over the paged KV cache, on the
// tensor cores (m16n8k16 MMAs, fp32 accumulation).
//
// What it computes: sequence s has n = query_start_loc[s+1] - query_start_loc[s]
// new tokens whose K/V are already in the cache as its last n positions, so
// its i-th new token sits at position p = context_lens[s] - n + i and attends
// causally over positions 0 .. p, read through block_tables[s]
// [Efficient Memory Management for Large Language Model Serving with
// PagedAttention, "End-to-End Decoding" (the prompt phase stores every prompt
// token's KV and attends over it in one pass) and "PagedAttention
// Algorithm"; vLLM Internals ..., chunked prefill in the scheduler (a prompt
// processed a token budget at a time)].
//
// How: one CTA per (query head h, sequence s, tile of 64 new tokens).  The
// grid runs the tiles of one (sequence, head) next to each other, heaviest
// first, and the heads of one KV head side by side, so the K/V tiles they
// all read come from L2 rather than HBM.  Warp 0 loads the Q tile with one
// tiled bulk copy (TMA, a 4-D view [head_dim/64][tokens][heads][64] of the
// query) and then streams 64-token K and V tiles of the sequence -- four
// 16-row chunks each, every chunk a TMA box of one pool block (two boxes per
// half for 8-token blocks) -- into an R-stage ring of mbarrier-guarded
// stages.  Warps 1..4 each own 16 query rows: S = Q K^T with ldmatrix
// fragments of the 128-byte-swizzled tiles, a causal and length mask, an
// online softmax in base 2, and O += P V with P split into two parts of the
// operand type for bf16 (so the weights keep ~16 bits), then O / l to the
// output.  Keys past a tile's last query position are masked, and their V
// rows are zeroed in shared memory before use (stale or poisoned data never
// reaches the output); every consumer warp zeroes them itself, writing the
// same zeros.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cstdint>
#include <cstring>
#include <type_traits>

#include "pa.h"
#include "pa_decode_mma.cuh"
#include "pa_launch.cuh"
#include "pa_ptx.cuh"
#include "pa_tmap.cuh"

namespace pa {
namespace {

constexpr int kPQ = 64;          // query tokens per CTA (4 warps x 16 rows)
constexpr int kPN = 64;          // keys per K/V tile (4 chunks of 16)
constexpr int kPChunks = kPN / 16;
constexpr int kPConsumers = 4;
constexpr int kPThreads = 32 * (kPConsumers + 1);
constexpr int kPMaxDevices = 64;

struct PrefillParams {
    CUtensorMap tmap_q, tmap_k, tmap_v;
    void *out;
    int out_dtype;
    const int32_t *block_tables;
    int max_blocks_per_seq;
    int block_size, block_shift;
    const int32_t *query_start_loc;
    const int32_t *context_lens;
    int max_query_len, max_context_len;
    int num_seqs, num_tokens, num_heads, num_kv_heads, G, head_dim, num_blocks;
    float scale_log2;
    unsigned int *err;
};

template <int D>
struct PLayout {
    static constexpr int KB = D / 64;
    static constexpr int R = D == 64 ? 4 : 2;                        // ring stages
    static constexpr size_t q_bytes = (size_t)KB * kPQ * 128;          // [half][64][64]
    static constexpr size_t chunk_bytes = (size_t)KB * kBoxBytes;      // [half][16][64]
    static constexpr size_t tile_bytes = kPChunks * chunk_bytes;
    static constexpr size_t q_off = 0;
    static constexpr size_t k_off = q_off + q_bytes;
    static constexpr size_t v_off = k_off + (size_t)R * tile_bytes;
    static constexpr size_t bad_off = v_off + (size_t)R * tile_bytes;  // uint32 [R]
    static constexpr size_t bar_off = (bad_off + 4 * R + 7) / 8 * 8;   // q_full, full[R], empty[R]
    static constexpr size_t flag_off = bar_off + (size_t)(1 + 2 * R) * 8;
    static constexpr size_t used = flag_off + 16;
    static constexpr size_t bytes = used + 1024;                       // base alignment slack
    static_assert(2 * (bytes + 1024) <= 233472, "two CTAs per SM");
};

__device__ __forceinline__ void tma_load_4d(void *dst, const void *tmap, int x, int y, int z,
                                            int w, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
        "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar))
        : "memory");
}

template <typename T>
__device__ __forceinline__ uint32_t pack2(float lo, float hi);
template <>
__device__ __forceinline__ uint32_t pack2<__half>(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}
template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// The work of one CTA, the same in every thread.
struct PItem {
    int s, h, hk, m;
    int n, L, c;         // new tokens, context length after the chunk, cached before it
    int q0, rows;        // first new token of the tile, rows in use (<= 64)
    int kv_end;          // keys 0 .. kv_end-1 are seen by some row of the tile
    int ntiles;
    int tok0;            // query row of the tile's first token
    bool ok, run;
};

__device__ __forceinline__ PItem make_item(const PrefillParams &P) {
    PItem it;
    it.m = (int)gridDim.x - 1 - (int)blockIdx.x;  // heaviest tiles first
    it.h = blockIdx.y;
    it.s = blockIdx.z;
    it.hk = it.h / P.G;
    const int a = P.query_start_loc[it.s], b = P.query_start_loc[it.s + 1];
    it.L = P.context_lens[it.s];
    it.n = b - a;
    it.tok0 = a;
    it.ok = a >= 0 && b <= P.num_tokens && it.n >= 0 && it.n <= P.max_query_len &&
            it.L >= it.n && it.L <= P.max_context_len;
    it.c = it.L - it.n;
    it.q0 = it.m * kPQ;
    it.rows = min(kPQ, it.n - it.q0);
    it.run = it.ok && it.rows > 0;
    it.kv_end = it.c + it.q0 + it.rows;
    it.ntiles = (it.kv_end + kPN - 1) / kPN;
    return it;
}

// ---------------------------------------------------------------------------
// producer warp
// ---------------------------------------------------------------------------
template <int D, typename T>
__device__ __forceinline__ void prefill_producer(const PrefillParams &P, const PItem &it,
                                                 unsigned char *sq, unsigned char *sk,
                                                 unsigned char *sv, uint32_t *stage_bad,
                                                 uint64_t *q_full, uint64_t *full,
                                                 uint64_t *empty, volatile int *abort_flag,
                                                 int lane) {
    using L = PLayout<D>;
    constexpr int KB = L::KB, R = L::R;
    const uint64_t policy = l2_evict_first_policy();
    const bool split = P.block_size < 16;  // 8-token blocks: a chunk spans two blocks
    const int32_t *row = P.block_tables + (size_t)it.s * P.max_blocks_per_seq;
    if (lane == 0) {
        mbar_arrive_expect_tx(q_full, (uint32_t)L::q_bytes);
        tma_load_4d(sq, &P.tmap_q, 0, it.h, it.tok0 + it.q0, 0, q_full);
    }
    // lane c < 4 holds chunk c's block ids for the tile in hand (x: the block
    // of its first token; y: the next block, for 8-token blocks)
    auto entries = [&](int j) -> int2 {
        int2 e = make_int2(-1, -1);
        const int tok = j * kPN + lane * 16;
        if (lane < kPChunks && tok < it.kv_end) {
            e.x = __ldg(&row[tok >> P.block_shift]);
            if (split && tok + 8 < it.kv_end) e.y = __ldg(&row[(tok >> P.block_shift) + 1]);
        }
        return e;
    };
    int2 cur = entries(0);
    int slot = 0;
    uint32_t phase = 0;
    int j = 0;
    bool aborted = false;
    for (; j < it.ntiles; ++j) {
        const int2 nxt = j + 1 < it.ntiles ? entries(j + 1) : make_int2(-1, -1);
        // this tile's chunks: which are in use, which name a bad block
        const int tok = j * kPN + lane * 16;
        const bool use = lane < kPChunks && tok < it.kv_end;
        const bool second = use && split && tok + 8 < it.kv_end;
        const bool bad_l = use && (cur.x < 0 || cur.x >= P.num_blocks ||
                                   (second && (cur.y < 0 || cur.y >= P.num_blocks)));
        const unsigned usemask = __ballot_sync(0xffffffffu, use);
        const unsigned bad = __ballot_sync(0xffffffffu, bad_l);
        const unsigned two = __ballot_sync(0xffffffffu, second);
        const unsigned good = usemask & ~bad;
        const uint32_t tx = split ? (uint32_t)(2 * KB * kHalfBoxBytes) *
                                        (uint32_t)(__popc(good) + __popc(two & good))
                                  : (uint32_t)(2 * KB * kBoxBytes) * (uint32_t)__popc(good);
        if (lane == 0 && bad && P.err) atomicOr(P.err, PA_ERRBIT_BLOCK_OOB);
        // this lane's copy
        bool issue;
        int y, z = 0, is_v;
        size_t off;
        if (!split) {  // lane 2c + kv: chunk c, K or V, both halves in one box
            const int c = min(lane >> 1, kPChunks - 1);
            const int pb = __shfl_sync(0xffffffffu, cur.x, c);
            issue = lane < 2 * kPChunks && ((good >> c) & 1u);
            const int t = j * kPN + c * 16;
            y = ((pb * P.num_kv_heads + it.hk) << P.block_shift) + (t & (P.block_size - 1));
            off = (size_t)c * L::chunk_bytes;
            is_v = lane & 1;
        } else {  // lane ((c * 2 + u) * KB + hf) * 2 + kv: half hf of block u of chunk c
            static_assert(kPChunks * 2 * KB * 2 <= 32, "one copy per lane");
            const int hf = (lane >> 1) % KB, u = (lane >> 1) / KB % 2,
                      c = min((lane >> 1) / (2 * KB), kPChunks - 1);
            const int p0 = __shfl_sync(0xffffffffu, cur.x, c);
            const int p1 = __shfl_sync(0xffffffffu, cur.y, c);
            issue = lane < kPChunks * 2 * KB * 2 && ((good >> c) & 1u) &&
                    (u == 0 || ((two >> c) & 1u));
            y = ((u ? p1 : p0) * P.num_kv_heads + it.hk) << P.block_shift;
            z = hf;
            off = (size_t)c * L::chunk_bytes + hf * kBoxBytes + u * kHalfBoxBytes;
            is_v = lane & 1;
        }
        bool ok = true;
        if (lane == 0) ok = mbar_wait(&empty[slot], phase ^ 1u, abort_flag);
        if (!__shfl_sync(0xffffffffu, (int)ok, 0)) {
            aborted = true;
            break;
        }
        if (lane == 0) {
            stage_bad[slot] = bad;
            mbar_arrive_expect_tx(&full[slot], tx);
        }
        __syncwarp();
        if (issue) {
            const size_t o = (size_t)slot * L::tile_bytes + off;
            if (is_v)
                tma_load_3d(sv + o, &P.tmap_v, 0, y, z, &full[slot], policy);
            else
                tma_load_3d(sk + o, &P.tmap_k, 0, y, z, &full[slot], policy);
        }
        __syncwarp();
        cur = nxt;
        if (++slot == R) {
            slot = 0;
            phase ^= 1u;
        }
    }
    if (aborted) {
        if (lane == 0) {
            *abort_flag = 1;
            if (P.err) atomicOr(P.err, PA_ERRBIT_TIMEOUT);
            // let the copies already issued land before the CTA can exit
            volatile int never = 0;
            mbar_wait(q_full, 0, &never);
            const int first = j > R ? j - R : 0;
            for (int k = first; k < j; ++k) mbar_wait(&full[k % R], (k / R) & 1u, &never);
        }
        __syncwarp();
    }
}

// ---------------------------------------------------------------------------
// consumer warps
// ---------------------------------------------------------------------------
template <int D, typename T>
__device__ __forceinline__ void prefill_consumer(const PrefillParams &P, const PItem &it,
                                                 unsigned char *sq, unsigned char *sk,
                                                 unsigned char *sv, const uint32_t *stage_bad,
                                                 uint64_t *q_full, uint64_t *full,
                                                 uint64_t *empty, volatile int *abort_flag,
                                                 int w, int lane) {
    using L = PLayout<D>;
    constexpr int KB = L::KB, R = L::R;
    constexpr int NK = D / 16;  // k-steps of Q K^T
    constexpr int NT = D / 8;   // n-tiles of P V
    constexpr bool kSplitP = sizeof(T) == 2 && !std::is_same<T, __half>::value;  // bf16
    const int g = lane >> 2, t = lane & 3;
    const float sc = P.scale_log2;
    auto fail = [&]() {
        if (lane == 0) {
            *abort_flag = 1;
            if (P.err) atomicOr(P.err, PA_ERRBIT_TIMEOUT);
        }
    };
    if (!__all_sync(0xffffffffu, mbar_wait(q_full, 0, abort_flag))) {
        fail();
        return;
    }
    // Q fragments of rows 16 w .. 16 w + 15
    uint32_t qa[NK][4];
    {
        const uint32_t qbase = smem_u32(sq);
        const int mi = lane >> 3;
        const int r = 16 * w + (mi & 1) * 8 + (lane & 7);
#pragma unroll
        for (int kk = 0; kk < NK; ++kk)
            ldsm_x4(qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3],
                    qbase + swz(2 * kk + (mi >> 1), r, (size_t)kPQ * 128));
    }
    // query positions of this thread's two rows (padding rows see every key)
    const int i0 = it.q0 + 16 * w + g, i1 = i0 + 8;
    const int qp0 = i0 < it.n ? it.c + i0 : it.L - 1;
    const int qp1 = i1 < it.n ? it.c + i1 : it.L - 1;
    const int wmin = it.c + it.q0 + 16 * w;  // the warp's smallest query position

    float o[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    int slot = 0;
    uint32_t phase = 0;
    for (int j = 0; j < it.ntiles; ++j) {
        if (!__all_sync(0xffffffffu, mbar_wait(&full[slot], phase, abort_flag))) {
            fail();
            return;
        }
        const uint32_t bad = stage_bad[slot];
        const int kbase_tok = j * kPN;
        unsigned char *kt = sk + (size_t)slot * L::tile_bytes;
        unsigned char *vt = sv + (size_t)slot * L::tile_bytes;
        // V rows no row of the tile may weigh: past kv_end, or in a skipped chunk
        const bool zero = bad || kbase_tok + kPN > it.kv_end;
        if (zero) {
            for (int i = lane; i < kPN * KB * 8; i += 32) {
                const int r = i / (KB * 8), rest = i % (KB * 8);  // row, 16-byte piece
                const int c = r >> 4;
                if (kbase_tok + r >= it.kv_end || ((bad >> c) & 1u))
                    *reinterpret_cast<uint4 *>(vt + (size_t)c * L::chunk_bytes +
                                               (rest >> 3) * kBoxBytes + (r & 15) * 128 +
                                               (rest & 7) * 16) = make_uint4(0, 0, 0, 0);
            }
            __syncwarp();
        }
        // S = Q K^T: 8 n-tiles of 8 keys
        float s[8][4];
#pragma unroll
        for (int n = 0; n < 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < NK; ++kk) {
            const int mi = lane >> 3;
            const int tok = 8 * (mi >> 1) + (lane & 7), chunk = 2 * kk + (mi & 1);
#pragma unroll
            for (int c = 0; c < kPChunks; ++c) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4(b0, b1, b2, b3,
                        smem_u32(kt + (size_t)c * L::chunk_bytes) + swz(chunk, tok, kBoxBytes));
                mma16816<T>(s[2 * c], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
                mma16816<T>(s[2 * c + 1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b2, b3);
            }
        }
        // scale to base 2; mask keys past each row's position and skipped chunks
        const bool mask = zero || kbase_tok + kPN - 1 > wmin;
#pragma unroll
        for (int n = 0; n < 8; ++n) {
#pragma unroll
            for (int e = 0; e < 4; ++e) s[n][e] *= sc;
            if (mask) {
                const int k0 = kbase_tok + 8 * n + 2 * t;
                const bool cb = (bad >> (n >> 1)) & 1u;
                if (cb || k0 > qp0) s[n][0] = -INFINITY;
                if (cb || k0 + 1 > qp0) s[n][1] = -INFINITY;
                if (cb || k0 > qp1) s[n][2] = -INFINITY;
                if (cb || k0 + 1 > qp1) s[n][3] = -INFINITY;
            }
        }
        // online softmax, rows g (0) and g + 8 (1); the quad t = 0..3 shares a row
        float mx0 = m0, mx1 = m1;
#pragma unroll
        for (int n = 0; n < 8; ++n) {
            mx0 = fmaxf(mx0, fmaxf(s[n][0], s[n][1]));
            mx1 = fmaxf(mx1, fmaxf(s[n][2], s[n][3]));
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float ms0 = mx0 == -INFINITY ? 0.f : mx0, ms1 = mx1 == -INFINITY ? 0.f : mx1;
        const float a0 = ex2(m0 - ms0), a1 = ex2(m1 - ms1);
        m0 = mx0;
        m1 = mx1;
        l0 *= a0;
        l1 *= a1;
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            o[n][0] *= a0;
            o[n][1] *= a0;
            o[n][2] *= a1;
            o[n][3] *= a1;
        }
#pragma unroll
        for (int n = 0; n < 8; ++n) {
            s[n][0] = ex2(s[n][0] - ms0);
            s[n][1] = ex2(s[n][1] - ms0);
            s[n][2] = ex2(s[n][2] - ms1);
            s[n][3] = ex2(s[n][3] - ms1);
            l0 += s[n][0] + s[n][1];
            l1 += s[n][2] + s[n][3];
        }
        // O += P V, one k-step per 16-key chunk
#pragma unroll
        for (int c = 0; c < kPChunks; ++c) {
            uint32_t ph[4], pl[4];
            if constexpr (kSplitP) {
                float r[8];
                ph[0] = pack_split<T>(s[2 * c][0], s[2 * c][1], r[0], r[1]);
                ph[1] = pack_split<T>(s[2 * c][2], s[2 * c][3], r[2], r[3]);
                ph[2] = pack_split<T>(s[2 * c + 1][0], s[2 * c + 1][1], r[4], r[5]);
                ph[3] = pack_split<T>(s[2 * c + 1][2], s[2 * c + 1][3], r[6], r[7]);
                pl[0] = pack2<T>(r[0], r[1]);
                pl[1] = pack2<T>(r[2], r[3]);
                pl[2] = pack2<T>(r[4], r[5]);
                pl[3] = pack2<T>(r[6], r[7]);
            } else {
                ph[0] = pack2<T>(s[2 * c][0], s[2 * c][1]);
                ph[1] = pack2<T>(s[2 * c][2], s[2 * c][3]);
                ph[2] = pack2<T>(s[2 * c + 1][0], s[2 * c + 1][1]);
                ph[3] = pack2<T>(s[2 * c + 1][2], s[2 * c + 1][3]);
            }
            const uint32_t vbase = smem_u32(vt + (size_t)c * L::chunk_bytes);
            const int mi = lane >> 3;
            const int tok = 8 * (mi & 1) + (lane & 7);
#pragma unroll
            for (int np = 0; np < NT / 2; ++np) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4_trans(b0, b1, b2, b3, vbase + swz(2 * np + (mi >> 1), tok, kBoxBytes));
                mma16816<T>(o[2 * np], ph[0], ph[1], ph[2], ph[3], b0, b1);
                mma16816<T>(o[2 * np + 1], ph[0], ph[1], ph[2], ph[3], b2, b3);
                if constexpr (kSplitP) {
                    mma16816<T>(o[2 * np], pl[0], pl[1], pl[2], pl[3], b0, b1);
                    mma16816<T>(o[2 * np + 1], pl[0], pl[1], pl[2], pl[3], b2, b3);
                }
            }
        }
        if (zero) fence_proxy_async_smem();  // zeroed rows before the next TMA here
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
        if (++slot == R) {
            slot = 0;
            phase ^= 1u;
        }
    }
    // O / l for the rows of this tile's sequence
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
    const size_t H = (size_t)P.num_heads;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const int i = half ? i1 : i0;
        if (i >= it.n) continue;
        const float inv = half ? inv1 : inv0;
        const size_t base = (((size_t)it.tok0 + i) * H + it.h) * D + 2 * t;
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            const float x = o[n][2 * half] * inv, y = o[n][2 * half + 1] * inv;
            if (P.out_dtype == PA_F32) {
                *reinterpret_cast<float2 *>(static_cast<float *>(P.out) + base + 8 * n) =
                    make_float2(x, y);
            } else {
                *reinterpret_cast<uint32_t *>(static_cast<T *>(P.out) + base + 8 * n) =
                    pack2<T>(x, y);
            }
        }
    }
}

template <int D, typename T>
__global__ void __launch_bounds__(kPThreads, 2) paged_prefill_kernel(const __grid_constant__ PrefillParams P) {
    using L = PLayout<D>;
    constexpr int R = L::R;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char *sq = smem + L::q_off;
    unsigned char *sk = smem + L::k_off;
    unsigned char *sv = smem + L::v_off;
    uint32_t *stage_bad = reinterpret_cast<uint32_t *>(smem + L::bad_off);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::bar_off);
    uint64_t *q_full = bars;
    uint64_t *full = bars + 1;
    uint64_t *empty = bars + 1 + R;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::flag_off);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        prefetch_tmap(&P.tmap_q);
        prefetch_tmap(&P.tmap_k);
        prefetch_tmap(&P.tmap_v);
        mbar_init(q_full, 1);
        for (int r = 0; r < R; ++r) {
            mbar_init(&full[r], 1);
            mbar_init(&empty[r], kPConsumers);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    pdl_trigger();
    pdl_wait();  // the cache write of the chunk (earlier on the stream) is complete
    const PItem it = make_item(P);
    if (!it.ok) {  // a length or offset out of range: flag it, zero the tile's rows
        if (threadIdx.x == 0 && P.err) atomicOr(P.err, PA_ERRBIT_CONTEXT_LEN);
        const int a = P.query_start_loc[it.s], b = P.query_start_loc[it.s + 1];
        if (a >= 0 && b <= P.num_tokens && b > a) {
            const int r0 = a + it.q0, r1 = min(b, r0 + kPQ);
            for (int r = r0; r < r1; ++r)
                for (int d = threadIdx.x; d < D; d += kPThreads)
                    store_out(P.out, P.out_dtype, ((size_t)r * P.num_heads + it.h) * D + d, 0.f);
        }
        return;
    }
    if (!it.run) return;
    if (warp == 0)
        prefill_producer<D, T>(P, it, sq, sk, sv, stage_bad, q_full, full, empty, abort_flag,
                               lane);
    else
        prefill_consumer<D, T>(P, it, sq, sk, sv, stage_bad, q_full, full, empty, abort_flag,
                               warp - 1, lane);
}

template <int D, typename T>
pa_status_t launch_prefill(const PrefillParams &P, dim3 grid, cudaStream_t stream) {
    using L = PLayout<D>;
    auto kern = paged_prefill_kernel<D, T>;
    static std::atomic<bool> attr_set[kPMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kPMaxDevices) return PA_ERR_CUDA;
    if (!attr_set[dev].load(std::memory_order_relaxed)) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)L::bytes) != cudaSuccess)
            return PA_ERR_CUDA;
        attr_set[dev].store(true, std::memory_order_relaxed);
    }
    return launch_pdl(kern, grid, dim3(kPThreads), L::bytes, stream, P) == cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

int shift_of(int b) {
    for (int sh = 3; sh <= 8; ++sh)
        if (b == (1 << sh)) return sh;
    return -1;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" pa_status_t pa_prefill_attention(
    void *out, pa_dtype_t out_dtype, const void *query, const void *k_cache, const void *v_cache,
    const int32_t *block_tables, int max_blocks_per_seq, const int32_t *query_start_loc,
    const int32_t *context_lens, int max_query_len, int max_context_len, int num_seqs,
    int num_tokens, int num_heads, int num_kv_heads, int head_dim, int num_blocks,
    int block_size, float scale, pa_dtype_t dtype, unsigned int *dev_error_word,
    pa_stream_t stream) {
    const int shift = shift_of(block_size);
    if (shift < 0) return PA_ERR_UNSUPPORTED;
    if (num_seqs < 0 || num_tokens < 0 || num_heads <= 0 || num_kv_heads <= 0 ||
        max_query_len < 0 || max_context_len < 0 || num_blocks <= 0 || max_blocks_per_seq <= 0)
        return PA_ERR_INVALID_ARG;
    if (num_heads % num_kv_heads != 0) return PA_ERR_INVALID_ARG;
    if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_INVALID_ARG;
    if (out_dtype != PA_F32 && out_dtype != dtype) return PA_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
    if ((long long)max_context_len > (long long)block_size * max_blocks_per_seq)
        return PA_ERR_INVALID_ARG;
    const unsigned long long pool_rows = (unsigned long long)num_blocks * num_kv_heads * block_size;
    if (pool_rows >= (1ull << 31) || (long long)num_tokens * num_heads >= (1ll << 31))
        return PA_ERR_UNSUPPORTED;
    if (num_seqs == 0 || num_tokens == 0 || max_query_len == 0) return PA_OK;
    if (!out || !query || !k_cache || !v_cache || !block_tables || !query_start_loc ||
        !context_lens)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(query) || !aligned16(k_cache) || !aligned16(v_cache))
        return PA_ERR_INVALID_ARG;
    const long long mtiles = (max_query_len + kPQ - 1) / kPQ;
    if (num_heads > 65535 || num_seqs > 65535 || mtiles > INT_MAX) return PA_ERR_UNSUPPORTED;

    PrefillParams P;
    memset(&P, 0, sizeof(P));
    const cuuint64_t KB = (cuuint64_t)head_dim / 64;
    {  // query [tokens][heads][head_dim] as [head_dim/64][tokens][heads][64]
        const cuuint64_t dims[4] = {64u, (cuuint64_t)num_heads, (cuuint64_t)num_tokens, KB};
        const cuuint64_t strides[3] = {(cuuint64_t)head_dim * 2,
                                       (cuuint64_t)num_heads * head_dim * 2, 128u};
        const cuuint32_t box[4] = {64u, 1u, (cuuint32_t)kPQ, (cuuint32_t)KB};
        if (!encode_tiled(&P.tmap_q, query, dtype, 4, dims, strides, box)) return PA_ERR_CUDA;
    }
    {  // pools [rows][head_dim] as [head_dim/64][rows][64]; a 16-row chunk per box,
       // or one 8-token block's rows of one half
        const bool eight = block_size < 16;
        const cuuint64_t dims[3] = {64u, (cuuint64_t)pool_rows, KB};
        const cuuint64_t strides[2] = {(cuuint64_t)head_dim * 2, 128u};
        const cuuint32_t box[3] = {64u, eight ? 8u : 16u, eight ? 1u : (cuuint32_t)KB};
        if (!encode_tiled(&P.tmap_k, k_cache, dtype, 3, dims, strides, box) ||
            !encode_tiled(&P.tmap_v, v_cache, dtype, 3, dims, strides, box))
            return PA_ERR_CUDA;
    }
    P.out = out;
    P.out_dtype = (int)out_dtype;
    P.block_tables = block_tables;
    P.max_blocks_per_seq = max_blocks_per_seq;
    P.block_size = block_size;
    P.block_shift = shift;
    P.query_start_loc = query_start_loc;
    P.context_lens = context_lens;
    P.max_query_len = max_query_len;
    P.max_context_len = max_context_len;
    P.num_seqs = num_seqs;
    P.num_tokens = num_tokens;
    P.num_heads = num_heads;
    P.num_kv_heads = num_kv_heads;
    P.G = num_heads / num_kv_heads;
    P.head_dim = head_dim;
    P.num_blocks = num_blocks;
    P.scale_log2 = scale * 1.4426950408889634f;
    P.err = dev_error_word;
    const dim3 grid((unsigned)mtiles, (unsigned)num_heads, (unsigned)num_seqs);
    cudaStream_t st = (cudaStream_t)stream;
    if (head_dim == 64)
        return dtype == PA_F16 ? launch_prefill<64, __half>(P, grid, st)
                               : launch_prefill<64, __nv_bfloat16>(P, grid, st);
    return dtype == PA_F16 ? launch_prefill<128, __half>(P, grid, st)
                           : launch_prefill<128, __nv_bfloat16>(P, grid, st);
}
