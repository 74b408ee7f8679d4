// pa_decode.cuh -- paged decode attention kernel for sm_103a.
//
// What it computes: for sequence s, query head h (KV head hk = h / G), the
// softmax(scale * q . k_t) weighted sum of v_t over the L = context_lens[s]
// tokens reached through block_tables[s], evaluated block by block with a
// running (online) softmax and merged exactly across blocks, warps and
// context partitions [Efficient Memory Management for Large Language Model
// Serving with PagedAttention, "PagedAttention Algorithm": block-wise
// reformulation of the attention equation; Paged Attention: Managing the KV
// Cache Like Virtual Memory, "Attention over scattered blocks": running
// softmax per query head sharing a KV head].
//
// How (one persistent CTA family per SM, warp-specialised):
//   * A work item is (piece of a sequence's context of <= part_tokens
//     tokens, KV head).  A plan kernel cuts every sequence's context into
//     pieces and lists them longest first; CTAs take their first three
//     items in a fixed order and claim the rest with one atomic each, so the
//     tail is short.  Each item names its sequence, its first token, its
//     token count and the partial-result slot (partition) it fills.
//   * A small batch (at most 256 (sequence, KV head) pairs, each context
//     within one partition, no shared prefixes) runs without the plan: the
//     kernels' DIRECT form takes each pair as one item, CTA b the pairs b,
//     b + grid, ...
//   * Runs of consecutive sequences whose block tables start with the same
//     full blocks share that prefix: the plan makes the shared prefix one
//     item whose query rows are all the run's queries (the tensor-core
//     kernel in pa_decode_mma.cuh takes those), and each sequence's own
//     remainder a plain item.  This kernel takes plain items only.
//   * Warp 0 (producer) resolves the item's block-table slice once (one
//     coalesced load, one entry per 16-token chunk; two for 8-token blocks)
//     and streams each chunk's K and V rows -- 16 rows x head_dim, only the
//     valid rows, contiguous within a block -- with 1-D bulk async copies
//     (TMA) into an R-stage shared-memory ring guarded by mbarriers (full:
//     transaction bytes; empty: one arrival per consumer warp).  The item's
//     G query rows ride with its first chunk.
//   * Block size B (tokens per block) is 8..256, a power of two, and only
//     changes where a chunk's rows come from: token t of a sequence is row
//     t % B of block block_tables[s][t / B]; a chunk lies in one block for
//     B >= 16 and spans two for B = 8.
//   * Warps 1..4 (consumers) each own 4 of a tile's 16 rows.  A row is split
//     over head_dim/8 lanes (16-byte chunks), so a warp reads 512 contiguous
//     bytes per instruction (no bank conflicts).  Scores: per-lane partial
//     dots, reduced with xor shuffles over the row's lanes.  Every lane keeps
//     its own running (max, sum, acc[8]) per query head over the rows it saw;
//     states are merged (shuffles, then shared memory) when the item ends.
//     Each K/V byte is read from HBM once and serves all G query heads.
//   * Output: the only item of a sequence writes the normalised row (fp32 or
//     the input type, round to nearest even); otherwise (max, sum, acc) go to
//     the workspace and the merge kernel combines the sequence's partitions.
// Scores are kept in base-2 units (q is pre-scaled by scale * log2 e) so the
// exponentials are single ex2 instructions.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "pa.h"
#include "pa_ptx.cuh"

namespace pa {

constexpr int kBlock = 16;             // tokens per ring stage (a chunk; one MMA n-extent)
constexpr int kNCW = 4;                // consumer warps
constexpr int kThreads = 32 * (kNCW + 1);
constexpr int kRowsPerWarp = kBlock / kNCW;
constexpr int kMaxPartTokens = 32 * kBlock;  // one producer lane per chunk of an item
constexpr int kEndFlag = 1;

struct alignas(16) StageMeta {
    int s, hk, p, nparts;
    int j, nblk, nvalid, flags;
};

// The plan writes up to two work lists: list 0 for the launch that takes
// shared-prefix items (or every item), list 1 for the CUDA-core kernel's
// plain items when a call runs both kernels.
struct WsHeader {
    unsigned int counter[2];  // items claimed beyond the first three rounds, per list
    unsigned int n_items[2];  // (piece, KV head) items in each list
};

// One entry per piece of a context, shared by its KV heads (item c of a list
// is entry c / num_kv_heads, KV head c % num_kv_heads):
//   x  the sequence (a shared-prefix item: the first sequence of its run)
//   y  the piece's first token, z its tokens (> 0)
//   w  bits 0..14: the partition (partial-result slot) the piece fills;
//      bits 16..30: the sequence's number of partitions, or for a
//      shared-prefix item the number of sequences in its run; bit 31: set
//      for a shared-prefix item
constexpr unsigned kGroupBit = 0x80000000u;
constexpr int kMaxParts = 0x7fff;
__host__ __device__ __forceinline__ int item_part(int w) { return w & 0x7fff; }
__host__ __device__ __forceinline__ int item_count(int w) { return (w >> 16) & 0x7fff; }
__host__ __device__ __forceinline__ bool item_is_group(int w) {
    return ((unsigned)w & kGroupBit) != 0u;
}
__host__ __device__ __forceinline__ int make_item_w(int part, int count, bool group) {
    return (int)((unsigned)part | ((unsigned)count << 16) | (group ? kGroupBit : 0u));
}

// Query rows of a shared-prefix item: the tmap_qs box holds Gb heads (G
// rounded up to a power of two, so every box has 8 rows) of 8 / Gb
// sequences; row r is head r / (8 / Gb) of the KV head's group and sequence
// r % (8 / Gb) of the run.  Rows of heads >= G belong to no item row.
__host__ __device__ __forceinline__ int group_box_heads(int G) {
    return G <= 1 ? 1 : (G <= 2 ? 2 : 4);
}
__host__ __device__ __forceinline__ int group_seqs_per_box(int G) {
    return 8 / group_box_heads(G);
}

struct DecodeParams {
    // Tensor maps of the query and the pools (tensor-core kernel only):
    // 3-D views [head_dim/64][rows][64], whole-row boxes, 128-byte swizzle.
    // tmap_qs views the query as [head_dim/64][heads][sequences][64] with a
    // box of G heads x 8/G sequences: the query rows of a shared-prefix item.
    CUtensorMap tmap_q, tmap_k, tmap_v, tmap_qs;
    void *out;
    int out_dtype;  // PA_F16, PA_BF16 or PA_F32
    const void *q;
    const void *k_cache;
    const void *v_cache;
    const int32_t *block_tables;
    int max_blocks_per_seq;
    int block_size, block_shift;  // tokens per pool block (8..256) and its log2
    // 0: paged pools reached through block_tables.  > 0: contiguous caches
    // [num_seqs][num_kv_heads][contig_rows][head_dim], no table.
    int contig_rows;
    const int32_t *context_lens;
    int max_context_len;
    int num_seqs, num_heads, num_kv_heads, G, head_dim, num_blocks;
    float scale_log2;  // scale * log2(e)
    int part_tokens, max_parts;
    int list;          // the work list this launch takes (0 or 1)
    int grouping;      // 1: the plan may form shared-prefix items
    int early_trigger; // 1: let the next kernel launch once the plan has completed
    // after_sibling = 1: the CUDA-core launch of a call that runs both
    // attention kernels.  It launches only once every CTA of the tensor-core
    // launch before it has seen the plan complete (early_trigger), so it
    // reads the plan's lists at once instead of waiting for that launch, and
    // waits for it only before it ends: whatever waits for this grid (the
    // merge) then sees both.
    int after_sibling;
    // direct = 1: no plan ran, and the host launches the kernels' DIRECT
    // form.  Item c is the whole context of (sequence c / Hkv, KV head
    // c % Hkv) and CTA b takes items b, b + grid, ... (for small batches whose
    // contexts fit one partition, with no shared prefixes); hdr, items and
    // nparts are then unused.
    int direct;
    WsHeader *hdr;
    int4 *items;       // the list this launch takes (entries as above)
    int *nparts;       // per sequence: its partitions (0: empty or invalid)
    float *part_m, *part_l, *part_acc;
    unsigned int *err;
};

template <typename T>
struct Cvt;
template <>
struct Cvt<__half> {
    static __device__ __forceinline__ void to_f32(const uint4 &u, float *f) {
        const __half2 *h = reinterpret_cast<const __half2 *>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 x = __half22float2(h[i]);
            f[2 * i] = x.x;
            f[2 * i + 1] = x.y;
        }
    }
};
template <>
struct Cvt<__nv_bfloat16> {
    static __device__ __forceinline__ void to_f32(const uint4 &u, float *f) {
        const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 x = __bfloat1622float2(h[i]);
            f[2 * i] = x.x;
            f[2 * i + 1] = x.y;
        }
    }
};

__device__ __forceinline__ void store_out(void *out, int dtype, size_t idx, float v) {
    if (dtype == PA_F32)
        static_cast<float *>(out)[idx] = v;
    else if (dtype == PA_F16)
        static_cast<__half *>(out)[idx] = __float2half_rn(v);
    else
        static_cast<__nv_bfloat16 *>(out)[idx] = __float2bfloat16_rn(v);
}

// Shared-memory layout of one CTA.
template <int D, int GM, int R>
struct Layout {
    static constexpr size_t kTileElems = (size_t)kBlock * D;
    static constexpr size_t k_off = 0;
    static constexpr size_t v_off = k_off + (size_t)R * kTileElems * 2;
    static constexpr size_t q_off = v_off + (size_t)R * kTileElems * 2;
    static constexpr size_t acc_off = q_off + (size_t)R * GM * D * 2;       // f32 [NCW][GM][D]
    static constexpr size_t m_off = acc_off + (size_t)kNCW * GM * D * 4;    // f32 [NCW][GM]
    static constexpr size_t l_off = m_off + (size_t)kNCW * GM * 4;          // f32 [NCW][GM]
    static constexpr size_t meta_off = (l_off + (size_t)kNCW * GM * 4 + 15) / 16 * 16;
    static constexpr size_t bar_off = meta_off + (size_t)R * sizeof(StageMeta);  // full[R], empty[R]
    static constexpr size_t cbar_off = bar_off + (size_t)2 * R * 8;  // consumer item barriers [2]
    static constexpr size_t flag_off = cbar_off + 2 * 8;       // abort flag
    static constexpr size_t bytes = flag_off + 16;
};

// Ring depth and CTAs per SM for a (head_dim, group) instantiation: as many
// 16-token K+V stages as fit the shared-memory share of one CTA.
template <int D, int GM>
struct Tuning {
    static constexpr int kMinBlocks = GM <= 2 ? 4 : 2;
    static constexpr size_t kBudget = 233472 / kMinBlocks - 1024 - 512;
    static constexpr size_t kStage = (size_t)2 * kBlock * D * 2 + (size_t)GM * D * 2 + 32 + 16;
    static constexpr size_t kFixed = (size_t)kNCW * GM * (D + 2) * 4 + 64;
    static constexpr int kRaw = (int)((kBudget - kFixed) / kStage);
    static constexpr int kStages = kRaw > 16 ? 16 : kRaw;
    static_assert(kStages >= 2, "ring too shallow");
};

// ---------------------------------------------------------------------------
// Item pipeline of one producer warp.  Rounds 0..2 are assigned statically
// (CTA b takes items b, b + grid, b + 2 grid), later items are claimed with
// one atomic each.  Four items are in flight: X (issuing), Y (block-table
// slice loaded), Z (entry loaded, slice loading), and the claim of the item
// after Z; every load is issued at least one item before its value is used,
// so only the very first item waits for two dependent loads.
// ---------------------------------------------------------------------------
// PA_DEBUG builds check every work item the producers take: a real
// sequence, a token range inside its context (inside every member's context
// for a shared-prefix item), and a partition slot that exists.  An item that
// fails is reported (PA_ERRBIT_INTERNAL) and skipped.
#ifdef PA_DEBUG
constexpr bool kDebugChecks = true;
#else
constexpr bool kDebugChecks = false;
#endif
template <bool DIRECT>
__device__ __forceinline__ bool item_ok(const DecodeParams &P, const int4 &e) {
    const int s = e.x, part = item_part(e.w), count = item_count(e.w);
    if (DIRECT && e.z == 0) return s >= 0 && s < P.num_seqs;  // an empty unit
    if (s < 0 || s >= P.num_seqs || e.y < 0 || e.z <= 0 || e.z > kMaxPartTokens) return false;
    if (part >= P.max_parts) return false;
    if (item_is_group(e.w)) {
        if (count < 2 || count > 8 || s + count > P.num_seqs) return false;
        for (int i = 0; i < count; ++i)
            if (e.y + e.z > P.context_lens[s + i]) return false;
        return true;
    }
    if (count < 1 || count > P.max_parts || part >= count) return false;
    return e.y + e.z <= P.context_lens[s];
}

// Without a plan, the producer of an empty or invalid unit (s, hk) writes its
// G output rows as zeros, and flags an invalid length once per sequence.
__device__ __forceinline__ void zero_unit_rows(const DecodeParams &P, int s, int hk, int lane) {
    const int L = P.context_lens[s];
    if (lane == 0 && hk == 0 && (L < 0 || L > P.max_context_len) && P.err)
        atomicOr(P.err, PA_ERRBIT_CONTEXT_LEN);
    const size_t base = ((size_t)s * P.num_heads + (size_t)hk * P.G) * P.head_dim;
    for (int i = lane; i < P.G * P.head_dim; i += 32) store_out(P.out, P.out_dtype, base + i, 0.f);
}

template <bool DIRECT>
struct ItemPipe {
    const DecodeParams *P;
    unsigned n_items, Hkv;
    int lane;
    unsigned cX, cY, cZ, raw;  // item indices; raw: lane 0's pending claim
    int4 eX, eY, eZ;           // entries (s, first token, tokens, w)
    int2 tX, tY;               // block-table entries of this lane's chunk of X and Y

    __device__ __forceinline__ int4 entry(unsigned c) const {
        if (c >= n_items) return make_int4(0, 0, 0, 0);
        if constexpr (DIRECT) {  // the unit's whole context; an empty or invalid one has no tokens
            const int seq = (int)(c / Hkv);
            const int L = P->context_lens[seq];
            const int Lv = (L < 0 || L > P->max_context_len) ? 0 : L;
            return make_int4(seq, 0, Lv, make_item_w(0, 1, false));
        }
        return __ldcg(&P->items[c / Hkv]);  // at L2: written by the plan in this call
    }
    // Lane j's chunk (tokens 16 j .. 16 j + 15 of the item): x = the block
    // holding its first token; y = the next block, read only for 8-token
    // blocks when the chunk has more than 8 tokens.
    __device__ __forceinline__ int2 table(unsigned c, int4 e) const {
        if (P->contig_rows) return make_int2(0, 0);  // contiguous cache: no table
        const int nchunk = (e.z + kBlock - 1) / kBlock;
        int2 r = make_int2(-1, -1);
        if (c < n_items && lane < nchunk) {
            const int32_t *row = P->block_tables + (size_t)e.x * P->max_blocks_per_seq;
            const int i = (e.y + lane * kBlock) >> P->block_shift;
            r.x = __ldg(&row[i]);
            if (P->block_size < kBlock && e.z - lane * kBlock > P->block_size)
                r.y = __ldg(&row[i + 1]);
        }
        return r;
    }
    // Lane 0 claims the next item beyond the three fixed rounds; no claim
    // (the answer is past the end) once the list is known to be exhausted,
    // so CTAs with nothing left do not queue on the counter.  Without a plan
    // the next item is simply the one a grid after `prev`.
    __device__ __forceinline__ unsigned claim(bool live, unsigned prev) const {
        if (lane != 0) return 0u;
        if constexpr (DIRECT) return prev + gridDim.x;
        if (!live) return n_items;
        return 3u * gridDim.x + atomicAdd(&P->hdr->counter[P->list], 1u);
    }
    __device__ __forceinline__ void init(const DecodeParams &params, unsigned n, int lane_) {
        P = &params;
        n_items = n;
        Hkv = (unsigned)params.num_kv_heads;
        lane = lane_;
        cX = blockIdx.x;
        cY = blockIdx.x + gridDim.x;
        cZ = blockIdx.x + 2u * gridDim.x;
        eX = entry(cX);
        eY = entry(cY);
        eZ = entry(cZ);
        raw = claim(3u * gridDim.x < n_items, cZ);
        tX = table(cX, eX);
        tY = table(cY, eY);
    }
    __device__ __forceinline__ bool valid() const { return cX < n_items; }
    // Move to the next item; called after the current item's copies are issued.
    __device__ __forceinline__ void advance() {
        const int2 tZ = table(cZ, eZ);
        const unsigned cW = __shfl_sync(0xffffffffu, raw, 0);
        const int4 eW = entry(cW);
        raw = claim(cW < n_items, cW);
        cX = cY; eX = eY; tX = tY;
        cY = cZ; eY = eZ; tY = tZ;
        cZ = cW; eZ = eW;
    }
};

// ---------------------------------------------------------------------------
// producer warp
// ---------------------------------------------------------------------------
template <int D, int GM, typename T, int R, bool DIRECT>
__device__ __forceinline__ void run_producer(const DecodeParams &P, T *sk, T *sv, T *sq,
                                             StageMeta *meta, uint64_t *full, uint64_t *empty,
                                             volatile int *abort_flag, int lane) {
    // The plan kernel's lists and counter (without a plan: whatever the
    // kernels before wrote, such as the cache write) are ready after this
    // wait.  A launch after the tensor-core one (after_sibling) only starts
    // once they are, and waits at its end instead.
    if (!P.after_sibling) pdl_wait();
    const unsigned n_items = DIRECT ? (unsigned)(P.num_seqs * P.num_kv_heads)
                                    : __ldcg(&P.hdr->n_items[P.list]);
    const unsigned Hkv = (unsigned)P.num_kv_heads;
    const int G = P.G;
    const uint64_t policy = l2_evict_first_policy();
    const T *kc = static_cast<const T *>(P.k_cache);
    const T *vc = static_cast<const T *>(P.v_cache);
    const T *qg = static_cast<const T *>(P.q);
    constexpr size_t kTile = (size_t)kBlock * D;

    ItemPipe<DIRECT> items;
    items.init(P, n_items, lane);

    uint32_t k = 0;      // stages issued so far
    int slot = 0;        // k % R
    uint32_t phase = 0;  // (k / R) & 1
    bool aborted = false;
    const bool split = !P.contig_rows && P.block_size < kBlock;  // 8-token blocks
    const uint32_t q_bytes = (uint32_t)(G * D * sizeof(T));
    while (items.valid()) {
        const unsigned cA = items.cX;
        const int4 eA = items.eX;
        const int2 tA = items.tX;

        if constexpr (kDebugChecks) {
            if (!item_ok<DIRECT>(P, eA)) {
                if (lane == 0 && P.err) atomicOr(P.err, PA_ERRBIT_INTERNAL);
                items.advance();
                continue;
            }
        }
        const int s = eA.x, t_item = eA.y, ntok = eA.z;
        const int part = item_part(eA.w), nparts = item_count(eA.w);
        const int hk = (int)(cA % Hkv);
        if constexpr (DIRECT) {
            if (ntok == 0) {  // an empty or invalid unit
                zero_unit_rows(P, s, hk, lane);
                items.advance();
                continue;
            }
        }
        const int nblk = (ntok + kBlock - 1) / kBlock;
        // Lane j prepares chunk j's copies once per item (all chunks at once),
        // so the per-chunk loop below only waits, arms the barrier and issues.
        const int nv = lane < nblk ? min(kBlock, ntok - lane * kBlock) : 0;
        // rows from the chunk's first block and (8-token blocks) its second
        const int n0 = split ? min(nv, P.block_size) : nv, n1 = nv - n0;
        const bool bad = nv > 0 && !P.contig_rows &&
                         (tA.x < 0 || tA.x >= P.num_blocks ||
                          (n1 > 0 && (tA.y < 0 || tA.y >= P.num_blocks)));
        const unsigned badmask = __ballot_sync(0xffffffffu, bad);  // skipped chunks
        if (lane == 0 && badmask && P.err) atomicOr(P.err, PA_ERRBIT_BLOCK_OOB);
        size_t off0 = 0, off1 = 0;  // element offsets of the rows in either pool
        if (nv > 0 && !bad) {
            const int t0 = t_item + lane * kBlock;  // the chunk's first token
            if (P.contig_rows) {
                off0 = (((size_t)s * Hkv + hk) * P.contig_rows + (size_t)t0) * D;
            } else {
                off0 = ((((size_t)tA.x * Hkv + hk) << P.block_shift) +
                        (size_t)(t0 & (P.block_size - 1))) * D;
                off1 = (((size_t)tA.y * Hkv + hk) << P.block_shift) * D;
            }
        }
        const uint32_t bytes0 = (uint32_t)n0 * D * (uint32_t)sizeof(T);
        const uint32_t bytes1 = (uint32_t)n1 * D * (uint32_t)sizeof(T);
        const T *qsrc = qg + ((size_t)s * P.num_heads + (size_t)hk * G) * D;

        for (int j = 0; j < nblk; ++j, ++k) {
            bool ok = true;
            if (lane == 0) ok = mbar_wait(&empty[slot], phase ^ 1u, abort_flag);
            if (!__shfl_sync(0xffffffffu, (int)ok, 0)) {  // warp-uniform outcome
                aborted = true;
                break;
            }
            if (lane == 0) {
                const int nvalid = ((badmask >> j) & 1u) ? 0 : min(kBlock, ntok - j * kBlock);
                StageMeta m;
                m.s = s; m.hk = hk; m.p = part; m.nparts = nparts;
                m.j = j; m.nblk = nblk; m.nvalid = nvalid; m.flags = 0;
                meta[slot] = m;
                mbar_arrive_expect_tx(&full[slot],
                                      2u * (uint32_t)nvalid * D * (uint32_t)sizeof(T) +
                                          (j == 0 ? q_bytes : 0u));
                if (j == 0) bulk_g2s_nohint(sq + (size_t)slot * GM * D, qsrc, q_bytes, &full[slot]);
            }
            __syncwarp();
            if (lane == j && nv > 0 && !bad) {
                T *dk = sk + slot * kTile, *dv = sv + slot * kTile;
                bulk_g2s(dk, kc + off0, bytes0, &full[slot], policy);
                bulk_g2s(dv, vc + off0, bytes0, &full[slot], policy);
                if (bytes1) {
                    bulk_g2s(dk + (size_t)n0 * D, kc + off1, bytes1, &full[slot], policy);
                    bulk_g2s(dv + (size_t)n0 * D, vc + off1, bytes1, &full[slot], policy);
                }
            }
            __syncwarp();
            if (++slot == R) {
                slot = 0;
                phase ^= 1u;
            }
        }
        if (aborted) break;
        items.advance();
    }
    if (!aborted) {  // end-of-work marker for the consumers
        const int slot = (int)(k % R);
        bool ok = true;
        if (lane == 0) ok = mbar_wait(&empty[slot], ((k / R) & 1u) ^ 1u, abort_flag);
        if (__shfl_sync(0xffffffffu, (int)ok, 0)) {
            if (lane == 0) {
                StageMeta m = {};
                m.flags = kEndFlag;
                meta[slot] = m;
                mbar_arrive(&full[slot]);
            }
        } else {
            aborted = true;
        }
    }
    if (aborted) {
        if (lane == 0) {
            *abort_flag = 1;
            if (P.err) atomicOr(P.err, PA_ERRBIT_TIMEOUT);
        }
        // let the copies already issued land before the CTA can exit
        if (lane == 0) {
            volatile int never = 0;
            const uint32_t first = k > (uint32_t)R ? k - R : 0u;
            for (uint32_t kk = first; kk < k; ++kk)
                mbar_drain_wait(&full[kk % R], (kk / R) & 1u, &never);
        }
        __syncwarp();
    }
    // The claim issued last is never used.  The fence waits until it (and
    // every claim before it) has been performed, so the counter is final
    // before the next call's plan kernel, which may start once this trigger
    // has fired in every CTA, resets it.
    __threadfence();
    pdl_trigger();
    if (P.after_sibling) pdl_wait();  // this grid ends after the tensor-core launch
}

// ---------------------------------------------------------------------------
// consumer warps
// ---------------------------------------------------------------------------
template <int D, int GM, typename T, int R>
__device__ __forceinline__ void run_consumer(const DecodeParams &P, const T *sk, const T *sv,
                                             const T *sq, const StageMeta *meta, uint64_t *full,
                                             uint64_t *empty, uint64_t *cbar, float *s_acc,
                                             float *s_m, float *s_l, volatile int *abort_flag,
                                             int cw, int lane) {
    constexpr int LPR = D / 8;           // lanes per row (16-byte chunks per row)
    constexpr int RPI = 32 / LPR;        // rows per warp instruction
    constexpr int NI = kRowsPerWarp / RPI;  // rows per lane per tile
    static_assert(NI >= 1, "head_dim too large");
    constexpr size_t kTile = (size_t)kBlock * D;
    const int c = lane % LPR, rg = lane / LPR;
    const int G = P.G;
    const int tid = cw * 32 + lane;
    uint32_t bar_par[2] = {0u, 0u};  // phase parity of the two consumer barriers
    // Bounded barrier over the 128 consumer threads; false if it gave up.
    auto consumer_sync = [&](int b) -> bool {
        mbar_arrive(&cbar[b]);
        const bool ok = mbar_wait(&cbar[b], bar_par[b], abort_flag);
        bar_par[b] ^= 1u;
        if (__all_sync(0xffffffffu, ok)) return true;
        if (lane == 0) {
            *abort_flag = 1;
            if (P.err) atomicOr(P.err, PA_ERRBIT_TIMEOUT);
        }
        return false;
    };

    float q[GM][8], acc[GM][8], m[GM], l[GM];
#pragma unroll
    for (int g = 0; g < GM; ++g) {
        m[g] = -INFINITY;
        l[g] = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) q[g][e] = acc[g][e] = 0.f;
    }

    int slot = -1;       // ring stage of this iteration
    uint32_t phase = 1;  // its phase parity
    for (;;) {
        if (++slot == R) slot = 0;
        if (slot == 0) phase ^= 1u;
        const bool ok = mbar_wait(&full[slot], phase, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) {  // warp-uniform outcome
            if (lane == 0) {
                *abort_flag = 1;
                if (P.err) atomicOr(P.err, PA_ERRBIT_TIMEOUT);
            }
            return;
        }
        const StageMeta mt = meta[slot];
        if (mt.flags & kEndFlag) return;
        const T *tk = sk + slot * kTile;
        const T *tv = sv + slot * kTile;

        if (mt.j == 0) {  // new item: load its query rows, reset the running state
            const T *tq = sq + (size_t)slot * GM * D;
#pragma unroll
            for (int g = 0; g < GM; ++g) {
                if (g < G) {
                    float f[8];
                    Cvt<T>::to_f32(*reinterpret_cast<const uint4 *>(tq + g * D + c * 8), f);
#pragma unroll
                    for (int e = 0; e < 8; ++e) q[g][e] = f[e] * P.scale_log2;
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) q[g][e] = 0.f;
                }
                m[g] = -INFINITY;
                l[g] = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[g][e] = 0.f;
            }
        }

        // scores for this lane's rows
        float sc[NI][GM];
        bool valid[NI];
#pragma unroll
        for (int i = 0; i < NI; ++i) {
            const int r = cw * kRowsPerWarp + i * RPI + rg;
            valid[i] = r < mt.nvalid;
            float kf[8];
            if (valid[i]) {
                Cvt<T>::to_f32(*reinterpret_cast<const uint4 *>(tk + r * D + c * 8), kf);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) kf[e] = 0.f;
            }
#pragma unroll
            for (int g = 0; g < GM; ++g) {
                float a = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) a = fmaf(q[g][e], kf[e], a);
                sc[i][g] = a;
            }
        }
#pragma unroll
        for (int i = 0; i < NI; ++i)
#pragma unroll
            for (int g = 0; g < GM; ++g)
#pragma unroll
                for (int off = LPR / 2; off > 0; off >>= 1)
                    sc[i][g] += __shfl_xor_sync(0xffffffffu, sc[i][g], off);

        // running softmax over the rows this lane has seen
        float pr[NI][GM];
#pragma unroll
        for (int g = 0; g < GM; ++g) {
            float mx = m[g];
#pragma unroll
            for (int i = 0; i < NI; ++i)
                if (valid[i]) mx = fmaxf(mx, sc[i][g]);
            const float ms = mx == -INFINITY ? 0.f : mx;
            const float alpha = ex2(m[g] - ms);
            l[g] *= alpha;
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[g][e] *= alpha;
#pragma unroll
            for (int i = 0; i < NI; ++i) {
                pr[i][g] = valid[i] ? ex2(sc[i][g] - ms) : 0.f;
                l[g] += pr[i][g];
            }
            m[g] = mx;
        }
#pragma unroll
        for (int i = 0; i < NI; ++i) {
            if (valid[i]) {
                const int r = cw * kRowsPerWarp + i * RPI + rg;
                float vf[8];
                Cvt<T>::to_f32(*reinterpret_cast<const uint4 *>(tv + r * D + c * 8), vf);
#pragma unroll
                for (int g = 0; g < GM; ++g)
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[g][e] = fmaf(pr[i][g], vf[e], acc[g][e]);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);  // tile consumed

        if (mt.j != mt.nblk - 1) continue;

        // ---- item complete: merge lane states, then warp states ----
#pragma unroll
        for (int off = LPR; off < 32; off <<= 1) {
#pragma unroll
            for (int g = 0; g < GM; ++g) {
                const float mo = __shfl_xor_sync(0xffffffffu, m[g], off);
                const float lo = __shfl_xor_sync(0xffffffffu, l[g], off);
                const float M = fmaxf(m[g], mo);
                const float Ms = M == -INFINITY ? 0.f : M;
                const float a = ex2(m[g] - Ms), b = ex2(mo - Ms);
                l[g] = l[g] * a + lo * b;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float ao = __shfl_xor_sync(0xffffffffu, acc[g][e], off);
                    acc[g][e] = acc[g][e] * a + ao * b;
                }
                m[g] = M;
            }
        }
        if (rg == 0) {
#pragma unroll
            for (int g = 0; g < GM; ++g) {
                float *dst = s_acc + ((size_t)cw * GM + g) * D + c * 8;
                *reinterpret_cast<float4 *>(dst) = make_float4(acc[g][0], acc[g][1], acc[g][2], acc[g][3]);
                *reinterpret_cast<float4 *>(dst + 4) = make_float4(acc[g][4], acc[g][5], acc[g][6], acc[g][7]);
                if (lane == 0) {
                    s_m[cw * GM + g] = m[g];
                    s_l[cw * GM + g] = l[g];
                }
            }
        }
        if (!consumer_sync(0)) return;
        const int H = P.num_heads;
        for (int idx = tid; idx < G * D; idx += kNCW * 32) {
            const int g = idx / D, d = idx - g * D;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kNCW; ++w) M = fmaxf(M, s_m[w * GM + g]);
            const float Ms = M == -INFINITY ? 0.f : M;
            float Lsum = 0.f, o = 0.f;
#pragma unroll
            for (int w = 0; w < kNCW; ++w) {
                const float cf = ex2(s_m[w * GM + g] - Ms);
                Lsum += s_l[w * GM + g] * cf;
                o += s_acc[((size_t)w * GM + g) * D + d] * cf;
            }
            const int h = mt.hk * G + g;
            if (mt.nparts == 1) {
                store_out(P.out, P.out_dtype, ((size_t)mt.s * H + h) * D + d,
                          Lsum > 0.f ? o / Lsum : 0.f);
            } else {
                const size_t pi = ((size_t)mt.s * H + h) * P.max_parts + mt.p;
                P.part_acc[pi * D + d] = o;
                if (d == 0) {
                    P.part_m[pi] = M;
                    P.part_l[pi] = Lsum;
                }
            }
        }
        if (!consumer_sync(1)) return;  // merge buffers free for the next item
    }
}

template <int D, int GM, typename T, int R, int MINB, bool DIRECT>
__global__ void __launch_bounds__(kThreads, MINB) paged_decode_kernel(const __grid_constant__ DecodeParams P) {
    extern __shared__ __align__(128) unsigned char smem[];
    using L = Layout<D, GM, R>;
    T *sk = reinterpret_cast<T *>(smem + L::k_off);
    T *sv = reinterpret_cast<T *>(smem + L::v_off);
    T *sq = reinterpret_cast<T *>(smem + L::q_off);
    float *s_acc = reinterpret_cast<float *>(smem + L::acc_off);
    float *s_m = reinterpret_cast<float *>(smem + L::m_off);
    float *s_l = reinterpret_cast<float *>(smem + L::l_off);
    StageMeta *meta = reinterpret_cast<StageMeta *>(smem + L::meta_off);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::bar_off);
    uint64_t *empty = full + R;
    uint64_t *cbar = reinterpret_cast<uint64_t *>(smem + L::cbar_off);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::flag_off);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        for (int r = 0; r < R; ++r) {
            mbar_init(&full[r], 1);
            mbar_init(&empty[r], kNCW);
        }
        mbar_init(&cbar[0], kNCW * 32);
        mbar_init(&cbar[1], kNCW * 32);
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (warp == 0)
        run_producer<D, GM, T, R, DIRECT>(P, sk, sv, sq, meta, full, empty, abort_flag, lane);
    else
        run_consumer<D, GM, T, R>(P, sk, sv, sq, meta, full, empty, cbar, s_acc, s_m, s_l,
                                  abort_flag, warp - 1, lane);
}

// Query groups of 2..8 heads with head_dim <= 128 run on the tensor cores
// (pa_decode_mma.cuh); single-head groups and head_dim 256 on the CUDA cores.
inline bool uses_tensor_cores(int G, int head_dim) { return G >= 2 && head_dim <= 128; }

// Which attention kernel a launch uses: the one the query group selects
// (tensor cores for G = 2..8 at head_dim <= 128, else CUDA cores), or the
// tensor-core kernel whatever G is (shared-prefix items of a G = 1 call).
constexpr int kKernelByGroup = 0;
constexpr int kKernelTensorCore = 1;

// Host-side launcher for one head_dim (defined in pa_decode_d{64,128,256}.cu).
pa_status_t launch_decode_d64(const DecodeParams &P, pa_dtype_t dtype, int grid_cap,
                              cudaStream_t stream, int kernel);
pa_status_t launch_decode_d128(const DecodeParams &P, pa_dtype_t dtype, int grid_cap,
                               cudaStream_t stream, int kernel);
pa_status_t launch_decode_d256(const DecodeParams &P, pa_dtype_t dtype, int grid_cap,
                               cudaStream_t stream, int kernel);

// Number of streaming multiprocessors of the current device (cached).
int current_sm_count();

}  // namespace pa
