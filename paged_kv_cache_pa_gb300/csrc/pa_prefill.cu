// pa_prefill.cu -- chunked-prefill attention over the paged KV cache on the
// 5th-generation tensor cores (tcgen05: operands in shared memory,
// accumulators in tensor memory).
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
// How: one CTA per (tile of 128 new tokens, query head, sequence); the grid
// runs the tiles of one (sequence, head) next to each other, heaviest first,
// and the heads of one KV head side by side, so the K/V tiles they all read
// come from L2.  Six warps:
//   * warp 0 (producer): the Q tile with one tiled bulk copy (TMA, a 4-D view
//     [head_dim/64][tokens][heads][64] of the query), then the sequence's
//     64-key K and V tiles into an R-stage ring laid out [slice][key][64] --
//     one TMA box per block's share of a tile and slice, or one box for all
//     slices when a block holds the whole tile;
//   * warp 1: allocates tensor memory; one thread issues S_j = Q K_j^T
//     (M = 128 queries, N = 64 keys, K = head_dim; both operands K-major)
//     into one of two S buffers, and O += P_j V_j (M = 128, N = head_dim,
//     K = 64 keys; V MN-major) into the O accumulator, S_{j+1} while the
//     softmax works on S_j;
//   * warps 2..5 (softmax): one query row per thread.  Each loads its row of
//     S_j from tensor memory, masks keys past its position (by assignment),
//     keeps a running maximum and sum in base 2, writes P_j to a swizzled
//     shared tile -- one of two, so P V_j runs while P_{j+1} is written --
//     (in two parts of the operand type for bf16, so the weights
//     keep ~16 bits), and rescales its row of O in tensor memory only when
//     its maximum grew by more than 2^8 since the last rescale (the sum and O
//     share that reference, so the result is exact); at the end it loads O,
//     divides by the sum and stores the row.
// V rows no query of a tile may weigh (past its last position, or in a chunk
// with a bad block id) are zeroed in shared memory before P V reads them.
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
#include "pa_launch.cuh"
#include "pa_ptx.cuh"
#include "pa_tmap.cuh"
#include "pa_umma.cuh"

namespace pa {
namespace {

constexpr int kQM = 128;             // query rows per CTA (tensor-memory lanes)
constexpr int kKN = 64;              // keys per K/V tile
constexpr int kThreadsP = 192;       // producer, MMA, 4 softmax warps
constexpr int kSoftmaxThreads = 128;
constexpr uint32_t kTmemCols = 256;  // S0, S1 (64 columns each), O (head_dim)
constexpr float kRescaleLog2 = 8.f;  // lazy rescale threshold (base-2 units)
constexpr int kMaxDevicesP = 64;

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

// A K/V tile is laid out [slice][64 keys][64] (rows of 128 bytes, 128-byte
// swizzle) whatever the block size: S = Q K^T then runs as N = 64 MMAs and
// P V reads 16-key steps one slice apart.  The TMA copies follow the
// blocks: a unit is one block's share of the tile, tbr = min(block size,
// 64) keys; a 64-key unit is one copy of every slice, a shorter one one
// copy per slice.  Fewer, larger copies keep the producer ahead.
constexpr uint32_t kSliceBytes = (uint32_t)kKN * 128u;  // one slice of a tile

template <int D, bool kSplit>
struct PLayout {
    static constexpr int KB = D / 64;                                  // 64-element slices
    static constexpr int R = D == 64 ? 6 : (kSplit ? 3 : 4);           // ring stages
    static constexpr size_t q_bytes = (size_t)KB * kQM * 128;          // [slice][128][64]
    static constexpr size_t tile_bytes = (size_t)KB * kSliceBytes;     // [slice][64 keys][64]
    static constexpr size_t p_bytes = (size_t)kQM * 128;               // [128 rows][64 keys]
    static constexpr size_t q_off = 0;
    static constexpr size_t k_off = q_off + q_bytes;
    static constexpr size_t v_off = k_off + (size_t)R * tile_bytes;
    // two P buffers [2][128][64], each followed by its low part for bf16
    static constexpr size_t pbuf_bytes = p_bytes * (kSplit ? 2 : 1);
    static constexpr size_t p_off = v_off + (size_t)R * tile_bytes;
    static constexpr size_t bad_off = p_off + 2 * pbuf_bytes;          // uint32 [R]
    static constexpr size_t bar_off = (bad_off + 4 * R + 7) / 8 * 8;
    // q_full, kv_full[R], kv_empty[R], s_full[2], s_free[2], p_full[2], p_free[2], o_done
    static constexpr int kBars = 1 + 2 * R + 4 + 4 + 1;
    static constexpr size_t tmem_off = bar_off + (size_t)kBars * 8;
    static constexpr size_t flag_off = tmem_off + 8;
    static constexpr size_t used = flag_off + 8;
    static constexpr size_t bytes = used + 1024;                       // base alignment slack
    static_assert(bytes + 1024 <= 233472, "one CTA per SM");
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
template <typename T>
__device__ __forceinline__ float2 unpack2(uint32_t u);
template <>
__device__ __forceinline__ float2 unpack2<__nv_bfloat16>(uint32_t u) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u));
}

__device__ __forceinline__ void store_elem(void *out, int dtype, size_t idx, float v) {
    if (dtype == PA_F32)
        static_cast<float *>(out)[idx] = v;
    else if (dtype == PA_F16)
        static_cast<__half *>(out)[idx] = __float2half_rn(v);
    else
        static_cast<__nv_bfloat16 *>(out)[idx] = __float2bfloat16_rn(v);
}

// The work of one CTA, the same in every thread.
struct PItem {
    int s, h, hk, m;
    int n, L, c;   // new tokens, context length after the chunk, cached before it
    int q0, rows;  // first new token of the tile, rows in use (<= 128)
    int kv_end;    // keys 0 .. kv_end-1 are seen by some row of the tile
    int ntiles;
    int tok0;      // query row of the sequence's first new token
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
    it.q0 = it.m * kQM;
    it.rows = min(kQM, it.n - it.q0);
    it.run = it.ok && it.rows > 0;
    it.kv_end = it.c + it.q0 + it.rows;
    it.ntiles = (it.kv_end + kKN - 1) / kKN;
    return it;
}

struct Bars {
    uint64_t *q_full, *kv_full, *kv_empty, *s_full, *s_free, *p_full, *p_free, *o_done;
    // p_full[b] / p_free[b]: P buffer b written by the softmax / read by P V
};

// ---------------------------------------------------------------------------
// warp 0: TMA producer
// ---------------------------------------------------------------------------
template <int D, bool kSplit>
__device__ __forceinline__ void run_producer_p(const PrefillParams &P, const PItem &it,
                                               unsigned char *sq, unsigned char *sk,
                                               unsigned char *sv, uint32_t *stage_bad,
                                               const Bars &B, volatile int *abort_flag,
                                               int lane) {
    using L = PLayout<D, kSplit>;
    constexpr int KB = L::KB, R = L::R;
    const uint64_t policy = l2_evict_first_policy();
    const int32_t *row = P.block_tables + (size_t)it.s * P.max_blocks_per_seq;
    if (lane == 0) {
        mbar_arrive_expect_tx(B.q_full, (uint32_t)L::q_bytes);
        tma_load_4d(sq, &P.tmap_q, 0, it.h, it.tok0 + it.q0, 0, B.q_full);
    }
    // Block ids come in batches of 32 units: lane l holds the block of unit
    // 32 t + l of batch t; the next batch is loaded a whole batch ahead, so
    // no table load waits on the per-tile path.
    // unit sizes are powers of two: shifts and masks, no divisions
    const int lg_tbr = min(P.block_shift, 6);   // keys per unit: min(block size, 64)
    const int tbr = 1 << lg_tbr;
    const int lg_upt = 6 - lg_tbr;              // units per tile (1 .. 8)
    const int upt = 1 << lg_upt;
    const int lg_tpb = 5 - lg_upt;              // tiles per batch of 32 units
    const bool whole = lg_tbr == 6;             // one copy covers every slice
    const int lg_cpu = whole ? 1 : 1 + (KB == 2 ? 1 : 0);  // copies per unit (K and V)
    auto batch = [&](int t) -> int {
        const int tok = ((t << 5) + lane) << lg_tbr;
        return tok < it.kv_end ? __ldg(&row[tok >> P.block_shift]) : -1;
    };
    int cur = batch(0);
    int nxt = batch(1);
    int slot = 0;
    uint32_t phase = 0;
    int j = 0;
    bool aborted = false;
    for (; j < it.ntiles; ++j) {
        if (j > 0 && (j & ((1 << lg_tpb) - 1)) == 0) {
            cur = nxt;
            nxt = batch((j >> lg_tpb) + 1);
        }
        const int lb = (j & ((1 << lg_tpb) - 1)) << lg_upt;  // lane of the tile's unit 0
        // lane u < upt checks unit u of the tile
        const int e = __shfl_sync(0xffffffffu, cur, lb + min(lane, upt - 1));
        const bool use = lane < upt && j * kKN + (lane << lg_tbr) < it.kv_end;
        const bool bad_l = use && (e < 0 || e >= P.num_blocks);
        const unsigned usemask = __ballot_sync(0xffffffffu, use);
        const unsigned bad_u = __ballot_sync(0xffffffffu, bad_l);
        const unsigned good = usemask & ~bad_u;
        // skipped 16-token chunks, for the softmax's mask
        unsigned bad = 0;
        if (bad_u) {
            for (int u = 0; u < upt; ++u)
                if ((bad_u >> u) & 1u)
                    bad |= tbr >= 16 ? ((1u << (tbr >> 4)) - 1u) << ((u * tbr) >> 4)
                                     : 1u << ((u * tbr) >> 4);
            if (lane == 0 && P.err) atomicOr(P.err, PA_ERRBIT_BLOCK_OOB);
        }
        const uint32_t tx = (2u * KB * 128u << lg_tbr) * (uint32_t)__popc(good);
        // this lane's copy: lane = u * copies + c, c = 2 sl + kv (a 64-key
        // unit: c = kv, every slice at once)
        const int u = min(lane >> lg_cpu, upt - 1), cc = lane & ((1 << lg_cpu) - 1);
        const int is_v = cc & 1, sl = whole ? 0 : cc >> 1;
        const int pb = __shfl_sync(0xffffffffu, cur, lb + u);
        const bool issue = lane < (upt << lg_cpu) && ((good >> u) & 1u);
        const int t = j * kKN + (u << lg_tbr);
        const int y = ((pb * P.num_kv_heads + it.hk) << P.block_shift) + (t & (P.block_size - 1));
        const int z = sl;
        const size_t off = (size_t)sl * kSliceBytes + ((size_t)u << lg_tbr) * 128;

        bool ok = true;
        if (lane == 0) ok = mbar_wait(&B.kv_empty[slot], phase ^ 1u, abort_flag);
        if (!__shfl_sync(0xffffffffu, (int)ok, 0)) {
            aborted = true;
            break;
        }
        if (lane == 0) {
            stage_bad[slot] = bad;
            mbar_arrive_expect_tx(&B.kv_full[slot], tx);
        }
        __syncwarp();
        if (issue) {
            const size_t o = (size_t)slot * L::tile_bytes + off;
            if (is_v)
                tma_load_3d(sv + o, &P.tmap_v, 0, y, z, &B.kv_full[slot], policy);
            else
                tma_load_3d(sk + o, &P.tmap_k, 0, y, z, &B.kv_full[slot], policy);
        }
        __syncwarp();
        if (++slot == R) {
            slot = 0;
            phase ^= 1u;
        }
    }
    if (aborted && lane == 0) {
        *abort_flag = 1;
        if (P.err) atomicOr(P.err, PA_ERRBIT_TIMEOUT);
    }
    // every copy issued lands before the CTA can exit
    if (lane == 0) {
        volatile int never = 0;
        mbar_wait(B.q_full, 0, &never);
        const int first = j > R ? j - R : 0;
        for (int k = first; k < j; ++k) mbar_wait(&B.kv_full[k % R], (k / R) & 1u, &never);
    }
    __syncwarp();
}

// ---------------------------------------------------------------------------
// warp 1, one thread: MMA issue
// ---------------------------------------------------------------------------
template <int D, bool kSplit>
__device__ __forceinline__ void run_mma_p(const PItem &it, unsigned char *sq, unsigned char *sk,
                                          unsigned char *sv, unsigned char *sp, uint32_t tmem,
                                          const Bars &B, uint32_t fmt,
                                          volatile int *abort_flag) {
    using L = PLayout<D, kSplit>;
    constexpr int R = L::R;
    const uint32_t idesc_s = umma_idesc_f16(fmt, 0, 0, kQM, kKN);
    const uint32_t idesc_o = umma_idesc_f16(fmt, 0, 1, kQM, D);
    const uint32_t tm_o = tmem + 2 * kKN;
    const uint32_t aq = smem_u32(sq), ak = smem_u32(sk), av = smem_u32(sv), ap0 = smem_u32(sp);
    bool ok = mbar_wait(B.q_full, 0, abort_flag);
    tc_fence_after();
    // S_j = Q K_j^T into buffer j % 2; a K step of 16 is 32 bytes inside a
    // 64-element slice, and the slices are whole tiles apart
    auto issue_s = [&](int j, int slot) -> bool {
        const int b = j & 1;
        if (!mbar_wait(&B.kv_full[slot], (uint32_t)(j / R) & 1u, abort_flag)) return false;
        if (!mbar_wait(&B.s_free[b], (((uint32_t)j >> 1) & 1u) ^ 1u, abort_flag)) return false;
        tc_fence_after();
        const uint32_t kt = ak + (uint32_t)(slot * L::tile_bytes);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t in_slice = (uint32_t)((kk & 3) * 32);
            const uint64_t da =
                umma_desc_sw128(aq + (uint32_t)((kk >> 2) * kQM * 128) + in_slice, 16, 1024);
            const uint64_t db =
                umma_desc_sw128(kt + (uint32_t)(kk >> 2) * kSliceBytes + in_slice, 16, 1024);
            umma_f16(tmem + (uint32_t)(b * kKN), da, db, idesc_s, kk > 0 ? 1u : 0u);
        }
        umma_commit(&B.s_full[b]);
        return true;
    };
    // O += P_i V_i (V MN-major: 16 keys = 2048 bytes per K step, slices of
    // head_dim a tile slice apart), then free the P tile and the K/V stage
    auto issue_pv = [&](int i, int slot) -> bool {
        const int pb = i & 1;
        if (!mbar_wait(&B.p_full[pb], ((uint32_t)i >> 1) & 1u, abort_flag)) return false;
        tc_fence_after();
        const uint32_t vt = av + (uint32_t)(slot * L::tile_bytes);
        const uint32_t ap = ap0 + (uint32_t)(pb * L::pbuf_bytes);
        const uint32_t apl = ap + (uint32_t)L::p_bytes;
#pragma unroll
        for (int kk = 0; kk < kKN / 16; ++kk) {
            // keys 16 kk .. 16 kk + 15; slices of head_dim a tile slice apart
            const uint64_t db = umma_desc_sw128(vt + (uint32_t)(kk * 16 * 128), kSliceBytes, 1024);
            const uint64_t da = umma_desc_sw128(ap + (uint32_t)(kk * 32), 16, 1024);
            umma_f16(tm_o, da, db, idesc_o, (i > 0 || kk > 0) ? 1u : 0u);
            if constexpr (kSplit) {
                const uint64_t dl = umma_desc_sw128(apl + (uint32_t)(kk * 32), 16, 1024);
                umma_f16(tm_o, dl, db, idesc_o, 1u);
            }
        }
        umma_commit(&B.p_free[pb]);
        umma_commit(&B.kv_empty[slot]);
        return true;
    };
    if (ok) ok = issue_s(0, 0);
    for (int j = 1; ok && j <= it.ntiles; ++j) {
        if (j < it.ntiles) ok = issue_s(j, j % R);
        if (ok) ok = issue_pv(j - 1, (j - 1) % R);
    }
    if (!ok) *abort_flag = 1;
    umma_commit(B.o_done);  // after every MMA issued: the epilogue and the teardown
}

// ---------------------------------------------------------------------------
// warps 2..5: softmax, one query row per thread, and the output
// ---------------------------------------------------------------------------
template <int D, typename T, bool kSplit>
__device__ __forceinline__ void run_softmax_p(const PrefillParams &P, const PItem &it,
                                              unsigned char *sv, unsigned char *sp,
                                              const uint32_t *stage_bad,
                                              uint32_t tmem, const Bars &B,
                                              volatile int *abort_flag, int warp, int lane) {
    using L = PLayout<D, kSplit>;
    constexpr int KB = L::KB, R = L::R;
    const int wq = warp & 3;                 // tensor-memory lanes 32 wq .. 32 wq + 31
    const int r = 32 * wq + lane;            // this thread's query row
    const uint32_t lane_addr = (uint32_t)(32 * wq) << 16;
    const uint32_t tm_o = tmem + 2 * kKN;
    const int i = it.q0 + r;                 // new-token index of the row
    const int qpos = i < it.n ? it.c + i : it.L - 1;  // padding rows see every key
    const int tid = (warp - 2) * 32 + lane;  // 0 .. 127
    const float sc = P.scale_log2;
    float m_ref = -INFINITY, lsum = 0.f;
    bool ok = true;
    for (int j = 0; j < it.ntiles; ++j) {
        const int b = j & 1, slot = j % R;
        // the stage's data and its bad-chunk mask (written before the stage
        // was armed), then S_j
        if (!__all_sync(0xffffffffu,
                        mbar_wait(&B.kv_full[slot], ((uint32_t)j / R) & 1u, abort_flag) &&
                            mbar_wait(&B.s_full[b], ((uint32_t)j >> 1) & 1u, abort_flag))) {
            ok = false;
            break;
        }
        tc_fence_after();
        uint32_t su[kKN];
#pragma unroll
        for (int c = 0; c < kKN; c += 16)
            tmem_ld16(tmem + lane_addr + (uint32_t)(b * kKN + c),
                      *reinterpret_cast<uint32_t(*)[16]>(&su[c]));
        tmem_wait_ld();
        float s[kKN];
#pragma unroll
        for (int e = 0; e < kKN; ++e) s[e] = __uint_as_float(su[e]);
        tc_fence_before();
        mbar_arrive(&B.s_free[b]);  // S buffer b may take S_{j+2}
        const uint32_t bad = stage_bad[slot];
        const int kb = j * kKN;
        // scale to base 2; keys past the row's position or in a skipped chunk
        // one warp per scheduler runs this code, so the reductions keep eight
        // independent chains
        constexpr int kAcc = 8;
        float mxa[kAcc];
#pragma unroll
        for (int q = 0; q < kAcc; ++q) mxa[q] = m_ref;
        if (!bad && kb + kKN - 1 <= qpos) {  // every key of the tile is visible
#pragma unroll
            for (int e = 0; e < kKN; ++e) {
                s[e] *= sc;
                mxa[e % kAcc] = fmaxf(mxa[e % kAcc], s[e]);
            }
        } else {
#pragma unroll
            for (int e = 0; e < kKN; ++e) {
                const bool masked = kb + e > qpos || ((bad >> (e >> 4)) & 1u);
                s[e] = masked ? -INFINITY : s[e] * sc;
                mxa[e % kAcc] = fmaxf(mxa[e % kAcc], s[e]);
            }
        }
#pragma unroll
        for (int q = 1; q < kAcc; ++q) mxa[0] = fmaxf(mxa[0], mxa[q]);
        const float mx = mxa[0];
        // lazy rescale: only when the maximum grew by more than 2^8; O must
        // then be stable (P V_{j-1} finished)
        const bool grow = mx > m_ref + kRescaleLog2;
        if (__any_sync(0xffffffffu, grow)) {
            const float alpha = grow && m_ref != -INFINITY ? ex2(m_ref - mx) : 1.f;
            if (j > 0) {
                const int q = (j - 1) & 1;
                if (!__all_sync(0xffffffffu, mbar_wait(&B.p_free[q],
                                                       ((uint32_t)(j - 1) >> 1) & 1u,
                                                       abort_flag))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < D; c += 16) {
                    uint32_t u[16];
                    tmem_ld16(tm_o + lane_addr + (uint32_t)c, u);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        u[e] = __float_as_uint(__uint_as_float(u[e]) * alpha);
                    tmem_st16(tm_o + lane_addr + (uint32_t)c, u);
                }
                tmem_wait_st();
            }
            if (grow) {
                lsum *= alpha;
                m_ref = mx;
            }
        }
        const float ms = m_ref == -INFINITY ? 0.f : m_ref;
        // P buffer j % 2 is free once P V_{j-2} has finished
        const int pb = j & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(&B.p_free[pb], (((uint32_t)j >> 1) & 1u) ^ 1u,
                                               abort_flag))) {
            ok = false;
            break;
        }
        // P row: 64 keys = 8 chunks of 16 bytes, 128-byte swizzle
        unsigned char *prow = sp + (size_t)pb * L::pbuf_bytes + (size_t)r * 128;
        unsigned char *plrow = prow + L::p_bytes;
        float lsa[kAcc];
#pragma unroll
        for (int q = 0; q < kAcc; ++q) lsa[q] = 0.f;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float p0 = ex2(s[8 * c + 2 * e] - ms), p1 = ex2(s[8 * c + 2 * e + 1] - ms);
                lsa[(2 * e) % kAcc] += p0;
                lsa[(2 * e + 1) % kAcc] += p1;
                hi[e] = pack2<T>(p0, p1);
                if constexpr (kSplit) {
                    const float2 h = unpack2<T>(hi[e]);
                    lo[e] = pack2<T>(p0 - h.x, p1 - h.y);
                }
            }
            const int sw = (c ^ (r & 7)) << 4;
            *reinterpret_cast<uint4 *>(prow + sw) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            if constexpr (kSplit)
                *reinterpret_cast<uint4 *>(plrow + sw) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
#pragma unroll
        for (int q = 0; q < kAcc; ++q) lsum += lsa[q];
        // V rows no row may weigh: past kv_end, or in a skipped chunk
        if (bad || kb + kKN > it.kv_end) {
            unsigned char *vt = sv + (size_t)slot * L::tile_bytes;
            for (int q = tid; q < kKN * KB * 8; q += kSoftmaxThreads) {
                const int key = q / (KB * 8), rest = q % (KB * 8);  // 16-byte piece
                if (kb + key >= it.kv_end || ((bad >> (key >> 4)) & 1u))
                    *reinterpret_cast<uint4 *>(vt + (size_t)(rest >> 3) * kSliceBytes + key * 128 +
                                               (rest & 7) * 16) = make_uint4(0, 0, 0, 0);
            }
        }
        fence_proxy_async_smem();  // P (and zeroed V) before the tensor core reads them
        tc_fence_before();
        mbar_arrive(&B.p_full[pb]);
    }
    if (!ok) {
        *abort_flag = 1;
        if (P.err) atomicOr(P.err, PA_ERRBIT_TIMEOUT);
    }
    // epilogue: O / sum for the rows of this tile's sequence
    const bool done = mbar_wait(B.o_done, 0, abort_flag);
    tc_fence_after();
    if (!__all_sync(0xffffffffu, done && ok && !*abort_flag)) return;
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
    const size_t base = (((size_t)it.tok0 + i) * P.num_heads + it.h) * D;
#pragma unroll
    for (int c = 0; c < D; c += 16) {
        uint32_t u[16];
        tmem_ld16(tm_o + lane_addr + (uint32_t)c, u);
        tmem_wait_ld();
        if (i < it.n) {
            if (P.out_dtype == PA_F32) {
                float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(P.out) + base + c);
#pragma unroll
                for (int e = 0; e < 16; e += 4)
                    dst[e / 4] = make_float4(
                        __uint_as_float(u[e]) * inv, __uint_as_float(u[e + 1]) * inv,
                        __uint_as_float(u[e + 2]) * inv, __uint_as_float(u[e + 3]) * inv);
            } else {
                uint4 *dst = reinterpret_cast<uint4 *>(static_cast<T *>(P.out) + base + c);
#pragma unroll
                for (int e = 0; e < 16; e += 8)
                    dst[e / 8] = make_uint4(
                        pack2<T>(__uint_as_float(u[e]) * inv, __uint_as_float(u[e + 1]) * inv),
                        pack2<T>(__uint_as_float(u[e + 2]) * inv, __uint_as_float(u[e + 3]) * inv),
                        pack2<T>(__uint_as_float(u[e + 4]) * inv, __uint_as_float(u[e + 5]) * inv),
                        pack2<T>(__uint_as_float(u[e + 6]) * inv, __uint_as_float(u[e + 7]) * inv));
            }
        }
    }
}

template <int D, typename T>
__global__ void __launch_bounds__(kThreadsP, 1)
    paged_prefill_kernel(const __grid_constant__ PrefillParams P) {
    constexpr bool kSplit = std::is_same<T, __nv_bfloat16>::value;
    using L = PLayout<D, kSplit>;
    constexpr int R = L::R;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char *sq = smem + L::q_off;
    unsigned char *sk = smem + L::k_off;
    unsigned char *sv = smem + L::v_off;
    unsigned char *sp = smem + L::p_off;
    uint32_t *stage_bad = reinterpret_cast<uint32_t *>(smem + L::bad_off);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::bar_off);
    Bars B;
    B.q_full = bars;
    B.kv_full = bars + 1;
    B.kv_empty = bars + 1 + R;
    B.s_full = bars + 1 + 2 * R;
    B.s_free = bars + 3 + 2 * R;
    B.p_full = bars + 5 + 2 * R;
    B.p_free = bars + 7 + 2 * R;
    B.o_done = bars + 9 + 2 * R;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::tmem_off);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::flag_off);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    pdl_trigger();
    pdl_wait();  // the cache write of the chunk (earlier on the stream) is complete
    const PItem it = make_item(P);
    if (!it.ok) {  // a length or offset out of range: flag it, zero the tile's rows
        if (threadIdx.x == 0 && P.err) atomicOr(P.err, PA_ERRBIT_CONTEXT_LEN);
        const int a = P.query_start_loc[it.s], b = P.query_start_loc[it.s + 1];
        if (a >= 0 && b <= P.num_tokens && b > a) {
            const int r0 = a + it.q0, r1 = min(b, r0 + kQM);
            for (int r = r0; r < r1; ++r)
                for (int d = threadIdx.x; d < D; d += kThreadsP)
                    store_elem(P.out, P.out_dtype, ((size_t)r * P.num_heads + it.h) * D + d, 0.f);
        }
        return;
    }
    if (!it.run) return;

    if (threadIdx.x == 0) {
        prefetch_tmap(&P.tmap_q);
        prefetch_tmap(&P.tmap_k);
        prefetch_tmap(&P.tmap_v);
        for (int b = 0; b < L::kBars; ++b) mbar_init(&bars[b], 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&B.s_free[b], kSoftmaxThreads);
            mbar_init(&B.p_full[b], kSoftmaxThreads);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        run_producer_p<D, kSplit>(P, it, sq, sk, sv, stage_bad, B, abort_flag, lane);
    } else if (warp == 1) {
        if (lane == 0)
            run_mma_p<D, kSplit>(it, sq, sk, sv, sp, tmem, B, kSplit ? 1u : 0u, abort_flag);
        __syncwarp();
    } else {
        run_softmax_p<D, T, kSplit>(P, it, sv, sp, stage_bad, tmem, B, abort_flag, warp, lane);
    }
    // every MMA has completed before tensor memory is released
    if (warp == 1 && lane == 0) {
        volatile int never = 0;
        mbar_wait(B.o_done, 0, &never);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

template <int D, typename T>
pa_status_t launch_prefill(const PrefillParams &P, dim3 grid, cudaStream_t stream) {
    using L = PLayout<D, std::is_same<T, __nv_bfloat16>::value>;
    auto kern = paged_prefill_kernel<D, T>;
    static std::atomic<bool> attr_set[kMaxDevicesP];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevicesP) return PA_ERR_CUDA;
    if (!attr_set[dev].load(std::memory_order_relaxed)) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)L::bytes) != cudaSuccess)
            return PA_ERR_CUDA;
        attr_set[dev].store(true, std::memory_order_relaxed);
    }
    return launch_pdl(kern, grid, dim3(kThreadsP), L::bytes, stream, P) == cudaSuccess
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
    const long long mtiles = (max_query_len + kQM - 1) / kQM;
    if (num_heads > 65535 || num_seqs > 65535 || mtiles > INT_MAX) return PA_ERR_UNSUPPORTED;

    PrefillParams P;
    memset(&P, 0, sizeof(P));
    const cuuint64_t KB = (cuuint64_t)head_dim / 64;
    {  // query [tokens][heads][head_dim] as [head_dim/64][tokens][heads][64]
        const cuuint64_t dims[4] = {64u, (cuuint64_t)num_heads, (cuuint64_t)num_tokens, KB};
        const cuuint64_t strides[3] = {(cuuint64_t)head_dim * 2,
                                       (cuuint64_t)num_heads * head_dim * 2, 128u};
        const cuuint32_t box[4] = {64u, 1u, (cuuint32_t)kQM, (cuuint32_t)KB};
        if (!encode_tiled(&P.tmap_q, query, dtype, 4, dims, strides, box)) return PA_ERR_CUDA;
    }
    {  // pools [rows][head_dim] as [head_dim/64][rows][64]; a box is one
       // block's share of a 64-key tile: 64 rows of every slice, or
       // min(block size, 64) rows of one slice
        const cuuint64_t dims[3] = {64u, (cuuint64_t)pool_rows, KB};
        const cuuint64_t strides[2] = {(cuuint64_t)head_dim * 2, 128u};
        const cuuint32_t tbr = (cuuint32_t)(block_size < kKN ? block_size : kKN);
        const cuuint32_t box[3] = {64u, tbr, tbr == (cuuint32_t)kKN ? (cuuint32_t)KB : 1u};
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
