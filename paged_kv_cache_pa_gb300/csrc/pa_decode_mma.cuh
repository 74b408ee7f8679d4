// pa_decode_mma.cuh -- paged decode attention on the tensor cores, for query
// groups of 2..8 heads per KV head (grouped-query attention), head_dim 64 or
// 128.
//
// With G query heads sharing a KV head, each 16-token block is a small dense
// contraction: S = Q K^T is [G x D] x [D x 16] and O += P V is
// [G x 16] x [16 x D].  Both run as m16n8k16 MMAs (fp16 or bf16 operands,
// fp32 accumulation) with the G query rows padded to 16
// [Paged Attention: Managing the KV Cache Like Virtual Memory, "Attention
// over scattered blocks": the query heads that share a KV head all use each
// K/V read; Efficient Memory Management for Large Language Model Serving with
// PagedAttention, "PagedAttention Algorithm": block-wise attention].
//
// Data movement: the producer warp fetches up to W blocks per stage (one
// per consumer warp) with tiled bulk copies (TMA) through 3-D tensor maps of
// the pools viewed as [head_dim / 64 halves][blocks * KV heads * 16 rows][64],
// with the 128-byte swizzle: one copy brings a 16-token chunk's whole K (or V)
// tile as [half][token][64], and the ldmatrix reads of the consumers are free
// of bank conflicts.  The copies of a stage are issued by separate lanes in
// one warp instruction.  The item's query rows (8-row box) ride with its
// first stage.  A chunk's box always has 16 rows, all inside one pool block
// for block sizes >= 16; with 8-token blocks the maps' boxes are 8 rows of
// one 64-element half, and a chunk takes two blocks x head_dim/64 halves,
// each landing at its place in the same [half][token][64] tile (8 rows of
// 128 bytes are one whole swizzle pattern).  Rows past the sequence's
// length are masked out of the scores and zeroed in the V tile before P V,
// so stale or poisoned data never reaches the output.
//
// Shared-prefix items: the plan turns the blocks that a run of consecutive
// sequences shares at the start of their tables into one item whose query
// rows are the run's queries for the KV head's G query heads (8 / G
// sequences at most, 2 for G = 3, G <= 4), loaded through a second tensor map that views
// the query as [head_dim / 64][heads][sequences][64].  Each shared K/V tile
// is then read once for the whole run; every sequence's own remainder is a
// plain item, and the partitions are merged exactly afterwards
// [Efficient Memory Management ..., "Shared prefix" and "Beam search": one
// physical copy of the shared blocks serves every sequence that maps them].
//
// Item ends: each consumer warp hands its running state for the item to a
// dedicated epilogue warp through one of two shared-memory buffers and goes
// straight on to the next stage; the epilogue warp merges the four states and
// writes each query row's output or partition's partial state.
//
// Precision: P is rounded to the operand type in two parts, P = P_hi + P_lo,
// and both are multiplied with V, so the weights carry ~16 significant bits
// (bf16 alone would carry 8).  Scores, the running softmax and the output
// accumulate in fp32.
#pragma once

#include "pa_decode.cuh"

namespace pa {

constexpr size_t kBoxBytes = 16 * 128;  // one chunk's 64-element box: 16 rows x 128 B
constexpr size_t kHalfBoxBytes = 8 * 128;  // an 8-token block's box: 8 rows x 128 B
constexpr size_t kQBoxBytes = 8 * 128;  // the query box: 8 rows x 128 B

// Per-item hand-off from the consumer warps to the epilogue warp.  count:
// the sequence's partitions (plain item) or the run's sequences (group).
struct alignas(16) ItemInfo {
    int s, hk, p, count;
    int flags, pad0, pad1, pad2;
};

constexpr int kGroupFlag = 2;  // StageMeta / ItemInfo flags: a shared-prefix item



// threads of a CTA with W consumer warps: producer, W consumers, epilogue
template <int W>
constexpr int threads_mma() { return 32 * (W + 2); }

template <int D, int R, int W>
struct LayoutMma {
    static constexpr int kBoxes = D / 64;
    static constexpr size_t k_off = 0;  // [R][BPS][boxes] boxes, 1 KiB aligned
    static constexpr size_t v_off = k_off + (size_t)R * W * kBoxes * kBoxBytes;
    static constexpr size_t q_off = v_off + (size_t)R * W * kBoxes * kBoxBytes;
    // two hand-off buffers: f32 acc [2][NCW][8][D], m and l [2][NCW][8]
    static constexpr size_t acc_off = q_off + (size_t)R * kBoxes * kQBoxBytes;
    static constexpr size_t m_off = acc_off + (size_t)2 * W * 8 * D * 4;
    static constexpr size_t l_off = m_off + (size_t)2 * W * 8 * 4;
    static constexpr size_t info_off = (l_off + (size_t)2 * W * 8 * 4 + 15) / 16 * 16;
    static constexpr size_t meta_off = info_off + 2 * sizeof(ItemInfo);
    static constexpr size_t bar_off = meta_off + (size_t)R * sizeof(StageMeta);
    // full[R], empty[R], acc_full[2], acc_empty[2]
    static constexpr size_t flag_off = bar_off + (size_t)(2 * R + 4) * 8;
    static constexpr size_t used = flag_off + 16;
    static constexpr size_t bytes = used + 1024;  // slack to align the base to 1 KiB
};

template <int D, int W>
struct TuningMma {
    static constexpr int kMinBlocks = W >= 4 ? 2 : (W == 2 ? 3 : 4);
    static constexpr size_t kBudget = 233472 / kMinBlocks - 1024 - 512;
    static constexpr size_t kStage =
        (size_t)2 * W * (D / 64) * kBoxBytes + (D / 64) * kQBoxBytes + 32 + 16;
    static constexpr size_t kFixed = (size_t)2 * W * 8 * (D + 2) * 4 + 2 * 32 + 96 + 1024;
    static constexpr int kRaw = (int)((kBudget - kFixed) / kStage);
    static constexpr int kStages = kRaw > 8 ? 8 : kRaw;
    static_assert(kStages >= 2, "ring too shallow");
};

template <typename T>
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1);
template <>
__device__ __forceinline__ void mma16816<__half>(float (&d)[4], uint32_t a0, uint32_t a1,
                                                 uint32_t a2, uint32_t a3, uint32_t b0,
                                                 uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
template <>
__device__ __forceinline__ void mma16816<__nv_bfloat16>(float (&d)[4], uint32_t a0, uint32_t a1,
                                                        uint32_t a2, uint32_t a3, uint32_t b0,
                                                        uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// (lo, hi) fp32 -> packed pair of T (lo in the low half); also returns the
// rounding residuals.
template <typename T>
__device__ __forceinline__ uint32_t pack_split(float lo, float hi, float &rlo, float &rhi);
template <>
__device__ __forceinline__ uint32_t pack_split<__half>(float lo, float hi, float &rlo, float &rhi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    const float2 b = __half22float2(h);
    rlo = lo - b.x;
    rhi = hi - b.y;
    return *reinterpret_cast<const uint32_t *>(&h);
}
template <>
__device__ __forceinline__ uint32_t pack_split<__nv_bfloat16>(float lo, float hi, float &rlo,
                                                              float &rhi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    const float2 b = __bfloat1622float2(h);
    rlo = lo - b.x;
    rhi = hi - b.y;
    return *reinterpret_cast<const uint32_t *>(&h);
}

// Byte offset of 16-byte chunk `chunk` (of the full head_dim row) of row
// `row` inside a block's [boxes] of 128-byte-swizzled rows.
__device__ __forceinline__ uint32_t swz(int chunk, int row, size_t box_bytes) {
    return (uint32_t)((chunk >> 3) * box_bytes + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
}

// ---------------------------------------------------------------------------
// producer warp: same item pipeline as the CUDA-core kernel, four blocks per
// stage, tiled TMA
// ---------------------------------------------------------------------------
template <int D, typename T, int R, int W, bool DIRECT>
__device__ __forceinline__ void run_producer_mma(const DecodeParams &P, unsigned char *sk,
                                                 unsigned char *sv, unsigned char *sq,
                                                 StageMeta *meta, uint64_t *full, uint64_t *empty,
                                                 volatile int *abort_flag, int lane) {
    constexpr int KB = D / 64;
    if (lane == 0) {
        prefetch_tmap(&P.tmap_k);
        prefetch_tmap(&P.tmap_v);
        prefetch_tmap(&P.tmap_q);
        if (P.grouping) prefetch_tmap(&P.tmap_qs);
    }
    pdl_wait();  // the plan's lists and counter (without a plan: the kernels before) are ready
    // The shared-prefix launch of a G = 1 call lets the CUDA-core kernel
    // after it launch once every CTA here has seen the plan complete: that
    // kernel reads the plan's lists at once, its CTAs start work as soon as
    // they fit, and it waits for this grid only before it ends.  (The next
    // call's plan still runs after this grid completes: it waits for the
    // kernels in between, which wait for this one.)
    if (P.early_trigger) pdl_trigger();
    const unsigned n_items = DIRECT ? (unsigned)(P.num_seqs * P.num_kv_heads)
                                    : __ldcg(&P.hdr->n_items[P.list]);
    const unsigned Hkv = (unsigned)P.num_kv_heads;
    const int G = P.G;
    const uint64_t policy = l2_evict_first_policy();

    ItemPipe<DIRECT> items;
    items.init(P, n_items, lane);

    uint32_t k = 0;
    bool aborted = false;
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
        const int part = item_part(eA.w), count = item_count(eA.w);
        const bool group = item_is_group(eA.w);
        const int hk = (int)(cA % Hkv);
        if constexpr (DIRECT) {
            if (ntok == 0) {  // an empty or invalid unit
                zero_unit_rows(P, s, hk, lane);
                items.advance();
                continue;
            }
        }
        const int nblk = (ntok + kBlock - 1) / kBlock;
        const int nst = (nblk + W - 1) / W;
        const bool split = !P.contig_rows && P.block_size < kBlock;  // 8-token blocks
        // query bytes: 8 rows either way (G heads of s and the rows after
        // them, or the run's box of heads x sequences)
        const uint32_t q_tx = (uint32_t)(KB * kQBoxBytes);
        for (int st = 0; st < nst; ++st, ++k) {
            // Everything that does not depend on the ring is worked out before
            // waiting for the slot, so a freed slot is refilled at once.
            const int j0 = st * W;
            const int nb = min(W, nblk - j0);
            // lane b < nb checks chunk b's block ids
            const int lb = min(j0 + min(lane, W - 1), 31);
            const int pc0 = __shfl_sync(0xffffffffu, tA.x, lb);
            const int pc1 = __shfl_sync(0xffffffffu, tA.y, lb);
            const bool second = split && lane < nb && ntok - (j0 + lane) * kBlock > P.block_size;
            const bool bad_l = lane < nb && !P.contig_rows &&
                               (pc0 < 0 || pc0 >= P.num_blocks ||
                                (second && (pc1 < 0 || pc1 >= P.num_blocks)));
            // chunks with an out-of-range block id are skipped
            const unsigned bad = __ballot_sync(0xffffffffu, bad_l);
            // 8-token blocks: chunks that need their second block
            const unsigned two = __ballot_sync(0xffffffffu, second);
            const uint32_t kv = split ? (uint32_t)(2 * KB * kHalfBoxBytes) *
                                            (uint32_t)(nb - __popc(bad) + __popc(two & ~bad))
                                      : (uint32_t)(2 * (nb - __popc(bad)) * KB * kBoxBytes);
            const uint32_t tx = kv + (st == 0 ? q_tx : 0u);
            // this lane's copy: its place in the stage, its row and half, K or V
            bool issue;
            int y, z = 0, is_v;
            size_t off;
            if (!split) {
                // lane 2b fetches chunk b's K tile, lane 2b+1 its V tile (both
                // 64-element halves in one 3-D box)
                const int b = min(lane >> 1, W - 1);
                const int pb = __shfl_sync(0xffffffffu, tA.x, min(j0 + b, 31));
                issue = lane < 2 * nb && !((bad >> b) & 1u);
                off = (size_t)b * KB * kBoxBytes;
                const int t0 = t_item + (j0 + b) * kBlock;  // the chunk's first token
                y = P.contig_rows ? (s * P.num_kv_heads + hk) * P.contig_rows + t0
                                  : ((pb * P.num_kv_heads + hk) << P.block_shift) +
                                        (t0 & (P.block_size - 1));
                is_v = lane & 1;
            } else {
                // 8-token blocks: lane = ((b * 2 + u) * KB + h) * 2 + kv fetches
                // half h of block u (0: first, 1: second) of chunk b, K or V
                static_assert(W * 2 * KB * 2 <= 32, "one copy per lane");
                const int h = (lane >> 1) % KB, u = (lane >> 1) / KB % 2,
                          b = min((lane >> 1) / (2 * KB), W - 1);
                const int p0 = __shfl_sync(0xffffffffu, tA.x, min(j0 + b, 31));
                const int p1 = __shfl_sync(0xffffffffu, tA.y, min(j0 + b, 31));
                issue = lane < W * 2 * KB * 2 && b < nb && !((bad >> b) & 1u) &&
                        (u == 0 || ((two >> b) & 1u));
                off = (size_t)b * KB * kBoxBytes + h * kBoxBytes + u * kHalfBoxBytes;
                y = ((u ? p1 : p0) * P.num_kv_heads + hk) << P.block_shift;
                z = h;
                is_v = lane & 1;
            }
            if (lane == 0 && bad && P.err) atomicOr(P.err, PA_ERRBIT_BLOCK_OOB);

            const int slot = (int)(k % R);
            bool ok = true;
            if (lane == 0) ok = mbar_wait(&empty[slot], ((k / R) & 1u) ^ 1u, abort_flag);
            if (!__shfl_sync(0xffffffffu, (int)ok, 0)) {
                aborted = true;
                break;
            }
            if (lane == 0) {
                StageMeta m;
                m.s = s; m.hk = hk; m.p = part; m.nparts = count;
                m.j = st; m.nblk = nst; m.nvalid = ntok - j0 * kBlock;
                m.flags = (int)(bad << 8) | (group ? kGroupFlag : 0);
                meta[slot] = m;
                mbar_arrive_expect_tx(&full[slot], tx);
            }
            __syncwarp();
            if (issue) {
                const size_t o = (size_t)slot * W * KB * kBoxBytes + off;
                if (is_v)
                    tma_load_3d(sv + o, &P.tmap_v, 0, y, z, &full[slot], policy);
                else
                    tma_load_3d(sk + o, &P.tmap_k, 0, y, z, &full[slot], policy);
            }
            if (st == 0 && lane == 0) {
                if (group)
                    tma_load_4d(sq + (size_t)slot * KB * kQBoxBytes, &P.tmap_qs, 0, s, hk * G, 0,
                                &full[slot], policy);
                else
                    tma_load_3d(sq + (size_t)slot * KB * kQBoxBytes, &P.tmap_q, 0,
                                s * P.num_heads + hk * G, 0, &full[slot], policy);
            }
            __syncwarp();
        }
        if (aborted) break;
        items.advance();
    }
    if (!aborted) {
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
}

// ---------------------------------------------------------------------------
// consumer warps: warp w takes block w of every stage
// ---------------------------------------------------------------------------
template <int D, typename T, int R, int W>
__device__ __forceinline__ void run_consumer_mma(const DecodeParams &P, unsigned char *sk,
                                                 unsigned char *sv, const unsigned char *sq,
                                                 const StageMeta *meta, uint64_t *full,
                                                 uint64_t *empty, uint64_t *acc_full,
                                                 uint64_t *acc_empty, float *s_acc, float *s_m,
                                                 float *s_l, ItemInfo *info,
                                                 volatile int *abort_flag, int cw, int lane) {
    constexpr int KB = D / 64;
    constexpr int NK = D / 16;  // k-steps of Q K^T
    constexpr int NT = D / 8;   // n-tiles of P V
    const int g = lane >> 2, t = lane & 3;
    const int G = P.G;
    const float sc = P.scale_log2;
    uint32_t handoffs = 0;  // items handed to the epilogue warp so far
    auto fail = [&]() {
        if (lane == 0) {
            *abort_flag = 1;
            if (P.err) atomicOr(P.err, PA_ERRBIT_TIMEOUT);
        }
    };
    // Take the next hand-off buffer (waits only if the epilogue is two items behind).
    auto take_buffer = [&](int &buf) -> bool {
        buf = (int)(handoffs & 1u);
        const bool ok = mbar_wait(&acc_empty[buf], ((handoffs >> 1) & 1u) ^ 1u, abort_flag);
        if (__all_sync(0xffffffffu, ok)) return true;
        fail();
        return false;
    };

    uint32_t qa[NK][2];
    float o[NT][4];
    float m_run = -INFINITY, l_run = 0.f;
#pragma unroll
    for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < NK; ++kk) qa[kk][0] = qa[kk][1] = 0u;

    for (uint32_t k = 0;; ++k) {
        const int slot = (int)(k % R);
        const bool okw = mbar_wait(&full[slot], (k / R) & 1u, abort_flag);
        if (!__all_sync(0xffffffffu, okw)) {
            fail();
            return;
        }
        const StageMeta mt = meta[slot];
        if (mt.flags & kEndFlag) {  // tell the epilogue warp there is no more work
            int buf;
            if (!take_buffer(buf)) return;
            if (cw == 0 && lane == 0) info[buf].flags = kEndFlag;
            mbar_arrive(&acc_full[buf]);
            return;
        }

        if (mt.j == 0) {  // new item: query fragments (rows 0..7; rows 8..15 are zero)
            const uint32_t qbase = smem_u32(sq + (size_t)slot * KB * kQBoxBytes);
#pragma unroll
            for (int kk = 0; kk < NK; kk += 2) {
                const int r = lane & 7, chunk = 2 * kk + (lane >> 3);
                ldsm_x4(qa[kk][0], qa[kk][1], qa[kk + 1][0], qa[kk + 1][1],
                        qbase + swz(chunk, r, kQBoxBytes));
            }
            m_run = -INFINITY;
            l_run = 0.f;
#pragma unroll
            for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
        }

        const int vb = min(kBlock, max(0, mt.nvalid - cw * kBlock));  // my block's tokens
        const bool mine = vb > 0 && !(((unsigned)mt.flags >> (8 + cw)) & 1u);
        if (mine) {
            unsigned char *kt = sk + (size_t)(slot * W + cw) * KB * kBoxBytes;
            unsigned char *vt = sv + (size_t)(slot * W + cw) * KB * kBoxBytes;
            if (vb < kBlock) {  // zero the V rows past the sequence's end
                for (int i = lane; i < (kBlock - vb) * KB * 8; i += 32) {
                    const int row = vb + i / (KB * 8), rest = i % (KB * 8);
                    *reinterpret_cast<uint4 *>(vt + (rest >> 3) * kBoxBytes + row * 128 +
                                               (rest & 7) * 16) = make_uint4(0, 0, 0, 0);
                }
                __syncwarp();
            }
            const uint32_t kbase = smem_u32(kt), vbase = smem_u32(vt);
            // S = Q K^T for the block's 16 tokens (two n-tiles of 8)
            float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kk = 0; kk < NK; ++kk) {
                const int mi = lane >> 3;
                const int tok = 8 * (mi >> 1) + (lane & 7), chunk = 2 * kk + (mi & 1);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(b0, b1, b2, b3, kbase + swz(chunk, tok, kBoxBytes));
                mma16816<T>(s0, qa[kk][0], 0u, qa[kk][1], 0u, b0, b1);
                mma16816<T>(s1, qa[kk][0], 0u, qa[kk][1], 0u, b2, b3);
            }
            // running softmax for row g (query head g); the quad t = 0..3 shares it
            float x[4] = {s0[0] * sc, s0[1] * sc, s1[0] * sc, s1[1] * sc};
            if (2 * t >= vb) x[0] = -INFINITY;
            if (2 * t + 1 >= vb) x[1] = -INFINITY;
            if (8 + 2 * t >= vb) x[2] = -INFINITY;
            if (9 + 2 * t >= vb) x[3] = -INFINITY;
            float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float mnew = fmaxf(m_run, mx);
            const float ms = mnew == -INFINITY ? 0.f : mnew;
            const float alpha = ex2(m_run - ms);
            float p[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) p[i] = ex2(x[i] - ms);
            l_run = l_run * alpha + (p[0] + p[1]) + (p[2] + p[3]);
            m_run = mnew;
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                o[n][0] *= alpha;
                o[n][1] *= alpha;
            }
            // O += P V with P = P_hi + P_lo (rows 8..15 of P are zero)
            float r0, r1, r2, r3;
            const uint32_t ph01 = pack_split<T>(p[0], p[1], r0, r1);
            const uint32_t ph23 = pack_split<T>(p[2], p[3], r2, r3);
            float d0, d1, d2, d3;
            const uint32_t pl01 = pack_split<T>(r0, r1, d0, d1);
            const uint32_t pl23 = pack_split<T>(r2, r3, d2, d3);
#pragma unroll
            for (int np = 0; np < NT / 2; ++np) {
                const int mi = lane >> 3;
                const int tok = 8 * (mi & 1) + (lane & 7), chunk = 2 * np + (mi >> 1);
                uint32_t b0, b1, b2, b3;
                ldsm_x4_trans(b0, b1, b2, b3, vbase + swz(chunk, tok, kBoxBytes));
                mma16816<T>(o[2 * np], ph01, 0u, ph23, 0u, b0, b1);
                mma16816<T>(o[2 * np], pl01, 0u, pl23, 0u, b0, b1);
                mma16816<T>(o[2 * np + 1], ph01, 0u, ph23, 0u, b2, b3);
                mma16816<T>(o[2 * np + 1], pl01, 0u, pl23, 0u, b2, b3);
            }
            if (vb < kBlock) fence_proxy_async_smem();  // zeroed rows before the next TMA here
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);  // stage consumed by this warp

        if (mt.j != mt.nblk - 1) continue;

        // ---- item complete: hand the warp's state to the epilogue warp ----
        float lq = l_run + __shfl_xor_sync(0xffffffffu, l_run, 1);
        lq += __shfl_xor_sync(0xffffffffu, lq, 2);
        int buf;
        if (!take_buffer(buf)) return;
        float *acc_b = s_acc + (size_t)buf * W * 8 * D;
        if (g < G || (mt.flags & kGroupFlag)) {  // a group item uses all 8 rows
            float *dst = acc_b + ((size_t)cw * 8 + g) * D + 2 * t;
#pragma unroll
            for (int n = 0; n < NT; ++n)
                *reinterpret_cast<float2 *>(dst + 8 * n) = make_float2(o[n][0], o[n][1]);
            if (t == 0) {
                s_m[(buf * W + cw) * 8 + g] = m_run;
                s_l[(buf * W + cw) * 8 + g] = lq;
            }
        }
        if (cw == 0 && lane == 0) {
            ItemInfo it;
            it.s = mt.s; it.hk = mt.hk; it.p = mt.p; it.count = mt.nparts;
            it.flags = mt.flags & kGroupFlag; it.pad0 = it.pad1 = it.pad2 = 0;
            info[buf] = it;
        }
        mbar_arrive(&acc_full[buf]);  // every consumer thread: its writes are released
        ++handoffs;
    }
}

// ---------------------------------------------------------------------------
// epilogue warp: merge the four consumer warps' states of each item and write
// the output row (one partition) or the partition's partial state
// ---------------------------------------------------------------------------
template <int D, int W>
__device__ __forceinline__ void run_epilogue_mma(const DecodeParams &P, uint64_t *acc_full,
                                                 uint64_t *acc_empty, const float *s_acc,
                                                 const float *s_m, const float *s_l,
                                                 const ItemInfo *info, volatile int *abort_flag,
                                                 int lane) {
    const int G = P.G, H = P.num_heads;
    for (uint32_t n = 0;; ++n) {
        const int buf = (int)(n & 1u);
        const bool ok = mbar_wait(&acc_full[buf], (n >> 1) & 1u, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) {
            if (lane == 0) {
                *abort_flag = 1;
                if (P.err) atomicOr(P.err, PA_ERRBIT_TIMEOUT);
            }
            return;
        }
        const ItemInfo it = info[buf];
        if (it.flags & kEndFlag) return;
        const float *acc_b = s_acc + (size_t)buf * W * 8 * D;
        const float *m_b = s_m + buf * W * 8, *l_b = s_l + buf * W * 8;
        // row r's merge of the W consumer warps' states, then its output
        // (one partition) or its partial state
        auto emit = [&](int r, int s_row, int h, int nparts) {
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < W; ++w) M = fmaxf(M, m_b[w * 8 + r]);
            const float Ms = M == -INFINITY ? 0.f : M;
            float cf[W], Lsum = 0.f;
#pragma unroll
            for (int w = 0; w < W; ++w) {
                cf[w] = ex2(m_b[w * 8 + r] - Ms);
                Lsum += l_b[w * 8 + r] * cf[w];
            }
            const size_t pi = ((size_t)s_row * H + h) * P.max_parts + it.p;
            for (int d = lane; d < D; d += 32) {
                float ov = 0.f;
#pragma unroll
                for (int w = 0; w < W; ++w) ov += acc_b[((size_t)w * 8 + r) * D + d] * cf[w];
                if (nparts == 1)
                    store_out(P.out, P.out_dtype, ((size_t)s_row * H + h) * D + d,
                              Lsum > 0.f ? ov / Lsum : 0.f);
                else
                    P.part_acc[pi * D + d] = ov;
            }
            if (nparts > 1 && lane == 0) {
                P.part_m[pi] = M;
                P.part_l[pi] = Lsum;
            }
        };
        if (!(it.flags & kGroupFlag)) {
            // the G heads of one sequence, all with the item's partition count
            for (int r = 0; r < G; ++r) emit(r, it.s, it.hk * G + r, it.count);
        } else {
            // a run's rows belong to different sequences: each row's own
            // partition count decides between the output and a partial
            const int nS = group_seqs_per_box(G);
            int np_lane = 0;
            if (lane < 8 && lane % nS < it.count) np_lane = P.nparts[it.s + lane % nS];
            for (int r = 0; r < 8; ++r) {
                const int gl = r / nS, sl = r % nS;
                const int np_row = __shfl_sync(0xffffffffu, np_lane, r);
                if (gl >= G || sl >= it.count) continue;  // no such row
                emit(r, it.s + sl, it.hk * G + gl, np_row);
            }
        }
        __syncwarp();
        mbar_arrive(&acc_empty[buf]);  // every lane: buffer free
    }
}

template <int D, typename T, int R, int MINB, int W, bool DIRECT>
__global__ void __launch_bounds__(threads_mma<W>(), MINB)
    paged_decode_mma_kernel(const __grid_constant__ DecodeParams P) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    using L = LayoutMma<D, R, W>;
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    unsigned char *sk = smem + L::k_off;
    unsigned char *sv = smem + L::v_off;
    unsigned char *sq = smem + L::q_off;
    float *s_acc = reinterpret_cast<float *>(smem + L::acc_off);
    float *s_m = reinterpret_cast<float *>(smem + L::m_off);
    float *s_l = reinterpret_cast<float *>(smem + L::l_off);
    ItemInfo *info = reinterpret_cast<ItemInfo *>(smem + L::info_off);
    StageMeta *meta = reinterpret_cast<StageMeta *>(smem + L::meta_off);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::bar_off);
    uint64_t *empty = full + R;
    uint64_t *acc_full = empty + R;
    uint64_t *acc_empty = acc_full + 2;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::flag_off);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        for (int r = 0; r < R; ++r) {
            mbar_init(&full[r], 1);
            mbar_init(&empty[r], W);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], W * 32);
            mbar_init(&acc_empty[b], 32);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (warp == 0)
        run_producer_mma<D, T, R, W, DIRECT>(P, sk, sv, sq, meta, full, empty, abort_flag, lane);
    else if (warp <= W)
        run_consumer_mma<D, T, R, W>(P, sk, sv, sq, meta, full, empty, acc_full, acc_empty, s_acc,
                                  s_m, s_l, info, abort_flag, warp - 1, lane);
    else
        run_epilogue_mma<D, W>(P, acc_full, acc_empty, s_acc, s_m, s_l, info, abort_flag, lane);
}

}  // namespace pa
