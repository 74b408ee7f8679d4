// pa_prefill.cu -- chunked-prefill attention over the paged KV cache on the
// 5th-generation tensor cores (tcgen05: operands in shared and tensor memory,
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
// How.  A work item is two 128-row query tiles of one sequence that read the
// same keys -- two query heads of one KV group over the same tokens when the
// group size is even, else two neighbouring token tiles of one head -- so each
// K/V tile loaded feeds two tiles of work.  A plan kernel lists the items that
// have work, heaviest (most K/V tiles) first.  The attention kernel is
// persistent, one CTA per SM; a CTA claims the next item of the list with an
// atomic counter, so long items start first and short ones fill the gaps.
// Every pipeline below runs on from one item to the next: the next item's Q,
// K/V and first S products are under way while the current one finishes.
// Sixteen warps; the two softmax warpgroups take 200 registers a thread from
// the other two, which keep 56:
//   * warp 8 (K producer): claims items and hands them to the other warps;
//     loads both Q tiles (tiled bulk copies, TMA, of a 4-D view
//     [head_dim/64][tokens][heads][64] of the query) once the previous item's
//     S products have stopped reading them, then the sequence's 64-key K
//     tiles into an RK-stage ring laid out [slice][key][64] -- one TMA box per
//     block's share of a tile and slice, or one box for all slices when a
//     block holds the whole tile;
//   * warp 9 (V producer): the V tiles into an RV-stage ring of the same
//     layout; it zeroes the V rows no query may weigh (a skipped block, keys
//     past the last one) before the tensor core reads them;
//   * warps 10, 11 (S issue of query tile 0, 1) and 12, 13 (P V issue): one
//     thread each issues, per K/V tile j, S = Q_t K_j^T (M = 128 queries,
//     N = 64 keys, K = head_dim; both operands K-major in shared memory) into
//     the tile's S buffer, or O_t += P V_j (M = 128, N = head_dim, K = 64
//     keys) with P read from a P buffer in tensor memory and V from shared
//     memory (MN-major).  One issuer per product and tile, so a wait of one
//     holds up only its own products; warp 14 allocates tensor memory, warp
//     15 is idle (register reallocation works by warpgroups);
//   * warps 0..3 and 4..7 (softmax of query tile 0 and 1): one query row per
//     thread.  Each loads its row of S_j from tensor memory (which frees the
//     S buffer for S_{j+1}), masks keys past its position (by assignment) and
//     keys of skipped blocks, keeps a running maximum and sum in base 2, and
//     writes P_j to a P buffer as packed 16-bit pairs (in two parts of the
//     operand type for bf16, so the weights keep ~16 bits).  It rescales its
//     row of O in tensor memory only when its maximum grew by more than 2^8
//     since the last rescale (the sum and O share that reference, so the
//     result is exact).  At the end of an item it loads O (which frees it for
//     the next item's P V), divides by the sum and writes the rows through a
//     staging buffer in shared memory, whole rows per store.
// A K stage is released when the S products that read it complete and a V
// stage when the P V products do.
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
#include "pa_nvtx.cuh"
#include "pa_ptx.cuh"
#include "pa_tmap.cuh"
#include "pa_umma.cuh"

namespace pa {
namespace {

constexpr int kQM = 128;             // query rows per tile (tensor-memory lanes)
constexpr int kKN = 64;              // keys per K/V tile
constexpr int kSoftmaxWarps = 8;     // two query tiles x four warps
constexpr int kWarpK = 8, kWarpV = 9;
constexpr int kWarpS = 10, kWarpPV = 12;  // + query tile
constexpr int kWarpAlloc = 14;
constexpr int kThreadsP = 32 * 16;
// registers a thread: 128 at launch (65536 / 512), then 200 for the softmax
// warpgroups and 56 for the other two -- the same total
constexpr int kRegsLaunch = 128, kRegsSoftmax = 200, kRegsOther = 56;
static_assert(2 * 128 * kRegsSoftmax + 2 * 128 * kRegsOther <= kThreadsP * kRegsLaunch,
              "register reallocation within the launch's registers");
constexpr int kTileThreads = 128;    // softmax threads of one query tile
constexpr int kItemReaders = 13;     // warps that take each item: 8 softmax, V, 4 issuers
constexpr int kStageWarpBytes = 4096;  // output staging of one softmax warp
// Tensor memory, 128 columns per query tile t at 128 t: S (64 columns of
// fp32), then P (64 columns: two buffers of 32 for fp16, one buffer of a
// high and a low 32-column part for bf16); O of tile t at 256 + t head_dim.
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleLog2 = 8.f;  // lazy rescale threshold (base-2 units)
constexpr int kMaxDevicesP = 64;
constexpr int kPlanThreads = 1024;
constexpr int kPlanBuckets = 2048;   // item costs (K/V tiles), the last bucket open-ended
// Workspace: a header of 4 words (claim counter, entries listed, items split),
// the entries (uint2: item id, part code) heaviest first, then for each split
// item a pair of finish counters and its two parts' partial results.
constexpr int kWorkHeader = 4;
constexpr int kMaxSplits = 160;      // items that may be split in two, at most

struct PrefillParams {
    CUtensorMap tmap_q, tmap_k, tmap_v;
    CUtensorMap tmap_out;  // out [tokens][heads][head_dim] as {head_dim, heads, tokens}
    void *out;
    int out_dtype;
    const int32_t *block_tables;
    int max_blocks_per_seq;
    int block_size, block_shift;
    const int32_t *query_start_loc;
    const int32_t *context_lens;
    int max_query_len, max_context_len;
    int num_seqs, num_tokens, num_heads, num_kv_heads, G, head_dim, num_blocks;
    int pair_heads;  // 1: an item's two tiles are heads 2y, 2y+1; 0: token tiles 2x, 2x+1
    int items_x, items_y;    // items of a sequence: x (token tiles or pairs) by y (heads or pairs)
    unsigned int num_items;  // num_seqs * items_x * items_y
    unsigned int grid;       // persistent CTAs
    int max_splits;          // split items the workspace has room for
    unsigned int *work;      // header: claim counter, entries listed, items split
    uint2 *entries;          // item id, part code (0: whole; 1 | part << 1 | slot << 2)
    unsigned int *split_cnt; // [max_splits][2 tiles]: parts finished
    float *part_m, *part_l;  // [max_splits][2 parts][2 tiles][128]: base-2 max and sum
    float *part_o;           // [max_splits][2 parts][2 tiles][128][head_dim]: unnormalised O
    float scale_log2;
    unsigned int *err;
};

// A K/V tile is laid out [slice][64 keys][64] (rows of 128 bytes, 128-byte
// swizzle) whatever the block size.  The TMA copies follow the blocks: a
// unit is one block's share of the tile, tbr = min(block size, 64) keys.
constexpr uint32_t kSliceBytes = (uint32_t)kKN * 128u;

// One query tile of an item.
struct PTile {
    int h;       // query head
    int q0;      // first new token of the tile
    int rows;    // rows in use (<= 128)
    int kv_end;  // keys 0 .. kv_end-1 are seen by some row of the tile
    int nt;      // 64-key tiles it reads
    bool act;
};

// One work item (or one part of a split item), the same in every thread that
// reads it.
struct PItem {
    int s, hk;
    int n, L, c;  // new tokens, context length after the chunk, cached before it
    int tok0;     // query row of the sequence's first new token
    int kv_end, ntiles;  // over both tiles
    int kt0, kt1;        // K/V tiles kt0 .. kt1-1 of 0 .. ntiles-1 (a part of a split item)
    int slot, part;      // split item: its partial-result slot and this part; slot -1: whole
    bool ok, run, stop;  // stop: no items left
    PTile t[2];
};

template <int D>
struct PLayout {
    static constexpr int KB = D / 64;                                  // 64-element slices
    static constexpr int RK = D == 64 ? 8 : 3;                         // K ring stages
    static constexpr int RV = D == 64 ? 8 : 5;                         // V ring stages
    static constexpr size_t qt_bytes = (size_t)KB * kQM * 128;         // [slice][128][64]
    static constexpr size_t tile_bytes = (size_t)KB * kSliceBytes;     // [slice][64 keys][64]
    static constexpr size_t q_off = 0;                                 // two Q tiles
    static constexpr size_t stage_off = q_off + 2 * qt_bytes;          // output staging
    static constexpr size_t k_off = stage_off + (size_t)kSoftmaxWarps * kStageWarpBytes;
    static constexpr size_t v_off = k_off + (size_t)RK * tile_bytes;
    static constexpr size_t item_off = v_off + (size_t)RV * tile_bytes;   // two PItem slots
    static constexpr size_t tag_off = item_off + 2 * sizeof(PItem);        // int [RK + RV]
    static constexpr size_t bar_off = (tag_off + 4 * (RK + RV) + 7) / 8 * 8;
    // q_full[2], q_free[2], k_full[RK], k_empty[RK], v_full[RV], v_empty[RV],
    // v_land, item_full[2], item_empty[2], s_full[2], s_free[2], p_full[2][2],
    // pv_done[2][2], o_free[2], o_done[2][2]
    static constexpr int kBars = 2 + 2 + 2 * RK + 2 * RV + 1 + 2 + 2 + 2 + 2 + 4 + 4 + 2 + 4;
    static constexpr size_t tmem_off = bar_off + (size_t)kBars * 8;
    static constexpr size_t flag_off = tmem_off + 8;
    static constexpr size_t split_off = flag_off + 8;                  // unsigned [2 tiles]
    static constexpr size_t used = split_off + 8;
    static constexpr size_t bytes = used + 1024;                       // base alignment slack
    static_assert(bytes <= 232448, "dynamic shared memory of one CTA");
};

struct Bars {
    // k_tag[s] / v_tag[s]: the K/V tile (counted from the CTA's first) the
    // producer last armed stage s with, written before the arming arrival
    volatile int *k_tag, *v_tag;
    uint64_t *q_full, *q_free;                // [2 tiles]
    uint64_t *k_full, *k_empty, *v_full, *v_empty, *v_land;
    uint64_t *item_full, *item_empty;         // [2 slots]
    uint64_t *s_full, *s_free;                // [2 tiles]
    uint64_t *p_full, *pv_done;               // [2 tiles][2 P buffers]
    uint64_t *o_free;                         // [2 tiles]
    uint64_t *o_done;                         // [2 tiles][S issuer, P V issuer]
};

// Tiled bulk store (TMA) of a shared-memory box to out, tracked as a bulk
// group of the issuing thread.
__device__ __forceinline__ void tma_store_3d(const void *tmap, int x, int y, int z,
                                             const void *src) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
            tmap),
        "r"(x), "r"(y), "r"(z), "r"(smem_u32(src))
        : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until this thread's bulk stores have read their shared-memory source
// (reads = true) or have completed.
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

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

// Item id -> (sequence, x, y) and its two tiles.
__device__ __forceinline__ PItem make_item(const PrefillParams &P, unsigned id) {
    PItem it;
    const int x = (int)(id % (unsigned)P.items_x);
    const unsigned rest = id / (unsigned)P.items_x;
    const int y = (int)(rest % (unsigned)P.items_y);
    it.s = (int)(rest / (unsigned)P.items_y);
    const int a = __ldg(&P.query_start_loc[it.s]), b = __ldg(&P.query_start_loc[it.s + 1]);
    it.L = __ldg(&P.context_lens[it.s]);
    it.n = b - a;
    it.tok0 = a;
    it.ok = a >= 0 && b <= P.num_tokens && it.n >= 0 && it.n <= P.max_query_len &&
            it.L >= it.n && it.L <= P.max_context_len;
    it.c = it.L - it.n;
    it.kv_end = 0;
    it.stop = false;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        PTile &tl = it.t[t];
        tl.h = P.pair_heads ? 2 * y + t : y;
        tl.q0 = (P.pair_heads ? x : 2 * x + t) * kQM;
        tl.rows = min(kQM, it.n - tl.q0);
        tl.act = it.ok && tl.rows > 0;
        tl.kv_end = it.c + tl.q0 + tl.rows;
        tl.nt = tl.act ? (tl.kv_end + kKN - 1) / kKN : 0;
        if (tl.act) it.kv_end = max(it.kv_end, tl.kv_end);
    }
    it.hk = it.t[0].h / P.G;  // both tiles read the same KV head
    it.ntiles = (it.kv_end + kKN - 1) / kKN;
    it.run = it.t[0].act || it.t[1].act;
    it.kt0 = 0;
    it.kt1 = it.ntiles;
    it.slot = -1;
    it.part = 0;
    return it;
}

// A part of a split item: the first part takes K/V tiles 0 .. ceil(n/2)-1,
// the second the rest.
__device__ __forceinline__ void apply_part(PItem &it, unsigned code) {
    if (!(code & 1u)) return;
    it.part = (int)((code >> 1) & 1u);
    it.slot = (int)(code >> 2);
    const int half = (it.ntiles + 1) / 2;
    it.kt0 = it.part ? half : 0;
    it.kt1 = it.part ? it.ntiles : half;
}

// -1: nothing to do (both tiles past the sequence's new tokens); else the K/V
// tiles the item reads (0 for a sequence whose lengths are out of range: its
// rows are zeroed and flagged).
__device__ __forceinline__ int item_cost(const PrefillParams &P, unsigned id) {
    const PItem it = make_item(P, id);
    if (!it.ok) return 0;
    return it.run ? it.ntiles : -1;
}

// Units of a tile and their block ids: a unit is tbr = 2^lg_tbr keys; lane l
// of a warp holds the block id of unit 32 t + l of batch t, so a batch
// covers 2^lg_tpb tiles.  Sizes are powers of two: shifts and masks only.
struct UnitGeo {
    int lg_tbr, lg_upt, upt, lg_tpb;
};

__device__ __forceinline__ UnitGeo unit_geo(int block_shift) {
    UnitGeo g;
    g.lg_tbr = min(block_shift, 6);
    g.lg_upt = 6 - g.lg_tbr;
    g.upt = 1 << g.lg_upt;
    g.lg_tpb = 5 - g.lg_upt;
    return g;
}

// Block id of this lane's unit of batch t; units from key `kv_end` on read as -1.
__device__ __forceinline__ int unit_entry(const PrefillParams &P, const int32_t *row,
                                          const UnitGeo &g, int t, int kv_end, int lane) {
    const int tok = ((t << 5) + lane) << g.lg_tbr;
    return tok < kv_end ? __ldg(&row[tok >> P.block_shift]) : -1;
}

// Every warp but the K producer takes item n from slot n % 2 (nullptr: the
// wait gave up), reads the fields it needs and gives the slot back.  `mask`:
// the lanes taking part (the whole warp, or lane 0 alone).
__device__ __forceinline__ const PItem *take_item(const PItem *items, const Bars &B, int n,
                                                  volatile int *abort_flag, int lane,
                                                  unsigned mask) {
    const int k = n & 1;
    bool ok = true;
    if (lane == 0) ok = mbar_wait(&B.item_full[k], (uint32_t)(n >> 1) & 1u, abort_flag);
    if (!__shfl_sync(mask, (int)ok, 0)) return nullptr;
    return &items[k];
}

__device__ __forceinline__ void give_item_back(const Bars &B, int n, int lane, unsigned mask) {
    __syncwarp(mask);
    if (lane == 0) mbar_arrive(&B.item_empty[n & 1]);
}

// Wait until K/V tile q (counted from the CTA's first) has landed in stage
// q % R.  A consumer that skips stages (its query tile needs fewer K/V tiles
// than the item's other one) can be a whole ring ahead of the producer, and
// then the parity of the phase it waits for is also the parity of the phase
// before; the stage's tag tells the two apart.
__device__ __forceinline__ bool wait_tile(uint64_t *full, volatile int *tag, int q, int R,
                                          volatile int *abort_flag) {
    const int st = q % R;
    const uint32_t parity = (uint32_t)(q / R) & 1u;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t polls = 0; polls < kWaitLimitPolls; ++polls) {
        if (mbar_try_wait(&full[st], parity) && tag[st] == q) return true;
        if ((polls & 31u) == 31u) {
            if (*abort_flag) return false;
            if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
        }
    }
    return false;
}

// What the softmax needs of an item's sequence.
struct SeqRows {
    int s, n, c, L, tok0;
};

// What the producers need of an item.
struct KVItem {
    int s, hk, kv_end, ntiles, kt0, kt1;
};

// ---------------------------------------------------------------------------
// plan: the items with work, heaviest first (a counting sort on the number of
// K/V tiles), as entries in the workspace.  An item whose K/V tiles exceed
// twice an SM's even share of the whole (2 total / grid) is split in two parts
// over its K/V tiles, the costliest first and at most max_splits of them; the
// two parts are separate entries and share a partial-result slot.
// ---------------------------------------------------------------------------
// exclusive start of each bucket in descending order of cost, in place; the
// total is returned (every thread)
__device__ __forceinline__ unsigned plan_scan_desc(unsigned *cnt, unsigned *warp_sum) {
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    constexpr int kPer = kPlanBuckets / kPlanThreads;
    static_assert(kPer * kPlanThreads == kPlanBuckets, "buckets per thread");
    unsigned v[kPer], local = 0;
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
        v[q] = cnt[kPlanBuckets - 1 - (kPer * tid + q)];
        local += v[q];
    }
    unsigned incl = local;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const unsigned o = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += o;
    }
    if (lane == 31) warp_sum[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        unsigned w = warp_sum[lane];
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const unsigned o = __shfl_up_sync(0xffffffffu, w, d);
            if (lane >= d) w += o;
        }
        warp_sum[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    unsigned start = incl - local + (wid > 0 ? warp_sum[wid - 1] : 0u);
    const unsigned total = warp_sum[kPlanThreads / 32 - 1];
    __syncthreads();  // every thread has read its counts
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
        cnt[kPlanBuckets - 1 - (kPer * tid + q)] = start;
        start += v[q];
    }
    __syncthreads();
    return total;
}

__global__ void __launch_bounds__(kPlanThreads, 1)
    prefill_plan_kernel(const __grid_constant__ PrefillParams P) {
    __shared__ unsigned int cnt[kPlanBuckets];
    __shared__ unsigned int warp_sum[kPlanThreads / 32];
    __shared__ unsigned long long s_total;
    __shared__ int s_split_cost;  // items of at least this cost are split
    __shared__ unsigned int s_slots;
    __shared__ int s_max_cost;
    pdl_trigger();
    const int tid = threadIdx.x;
    for (int b = tid; b < kPlanBuckets; b += kPlanThreads) cnt[b] = 0;
    if (tid == 0) {
        s_total = 0;
        s_slots = 0;
        s_max_cost = 0;
    }
    __syncthreads();
    // items per cost, and the total
    unsigned long long mine = 0;
    int my_max = 0;
    for (unsigned id = tid; id < P.num_items; id += kPlanThreads) {
        const int c = item_cost(P, id);
        if (c >= 0) {
            atomicAdd(&cnt[min(c, kPlanBuckets - 1)], 1u);
            mine += (unsigned long long)c;
            my_max = max(my_max, min(c, kPlanBuckets - 1));
        }
    }
    atomicAdd(&s_total, mine);
    atomicMax(&s_max_cost, my_max);
    __syncthreads();
    // the split threshold: above an even share, and no more items than slots
    if (tid == 0) {
        // twice an SM's even share: a part's own costs (partial results,
        // the merge) outweigh the balance gained below that
        const unsigned long long share = (2 * s_total + P.grid - 1) / max(1u, P.grid);
        int c = s_max_cost + 1;
        unsigned above = 0;
        while (c > 2 && (unsigned long long)(c - 1) > share &&
               above + cnt[c - 1] <= (unsigned)P.max_splits) {
            above += cnt[c - 1];
            --c;
        }
        s_split_cost = c;  // costs >= c are split (max cost + 1: none)
    }
    __syncthreads();
    const int split_cost = s_split_cost;
    // entries per cost: a split item gives two parts of ceil(c/2) and floor(c/2)
    for (int b = tid; b < kPlanBuckets; b += kPlanThreads) cnt[b] = 0;
    __syncthreads();
    for (unsigned id = tid; id < P.num_items; id += kPlanThreads) {
        const int c = item_cost(P, id);
        if (c < 0) continue;
        if (c >= split_cost) {
            atomicAdd(&cnt[min((c + 1) / 2, kPlanBuckets - 1)], 1u);
            atomicAdd(&cnt[min(c / 2, kPlanBuckets - 1)], 1u);
        } else {
            atomicAdd(&cnt[min(c, kPlanBuckets - 1)], 1u);
        }
    }
    __syncthreads();
    const unsigned total = plan_scan_desc(cnt, warp_sum);
    // Everything above only read the inputs.  The work list is written once
    // the kernel before this one has completed: the attention kernel depends
    // on it as well (the cache write of the chunk), and an earlier attention
    // call on this stream may still be taking entries from this workspace.
    pdl_wait();
    for (unsigned id = tid; id < P.num_items; id += kPlanThreads) {
        const int c = item_cost(P, id);
        if (c < 0) continue;
        if (c >= split_cost) {
            const unsigned slot = atomicAdd(&s_slots, 1u);
            const unsigned p0 = atomicAdd(&cnt[min((c + 1) / 2, kPlanBuckets - 1)], 1u);
            const unsigned p1 = atomicAdd(&cnt[min(c / 2, kPlanBuckets - 1)], 1u);
            P.entries[p0] = make_uint2(id, 1u | (0u << 1) | (slot << 2));
            P.entries[p1] = make_uint2(id, 1u | (1u << 1) | (slot << 2));
        } else {
            const unsigned pos = atomicAdd(&cnt[min(c, kPlanBuckets - 1)], 1u);
            P.entries[pos] = make_uint2(id, 0u);
        }
    }
    __syncthreads();
    for (unsigned i = tid; i < 2 * s_slots; i += kPlanThreads) P.split_cnt[i] = 0u;
    if (tid == 0) {
        P.work[0] = 0u;
        P.work[1] = total;
        P.work[2] = s_slots;
    }
}

// ---------------------------------------------------------------------------
// warps 8 and 9: TMA producers of K (and Q) and of V, one item
// ---------------------------------------------------------------------------
template <int D, bool kIsV>
__device__ __forceinline__ bool produce_item(const PrefillParams &P, const KVItem &it,
                                             unsigned char *skv, const Bars &B,
                                             volatile int *abort_flag, int lane, int &rc,
                                             int &land, bool &land_pending) {
    using L = PLayout<D>;
    constexpr int KB = L::KB, R = kIsV ? L::RV : L::RK;
    uint64_t *full = kIsV ? B.v_full : B.k_full;
    uint64_t *empty = kIsV ? B.v_empty : B.k_empty;
    const CUtensorMap *tmap = kIsV ? &P.tmap_v : &P.tmap_k;
    const uint64_t policy = l2_evict_first_policy();
    const int32_t *row = P.block_tables + (size_t)it.s * P.max_blocks_per_seq;
    const UnitGeo g = unit_geo(P.block_shift);
    const int tpb_mask = (1 << g.lg_tpb) - 1;
    const bool whole = g.lg_tbr == 6;                     // one copy covers every slice
    const int lg_cpu = whole ? 0 : (KB == 2 ? 1 : 0);     // copies per unit
    const uint32_t unit_bytes = (uint32_t)KB * 128u << g.lg_tbr;
    // rows from this key on are cleared in the last V tile
    const int tail_row = it.kv_end & (kKN - 1);
    const int b0 = it.kt0 >> g.lg_tpb;  // table batch of the first tile
    int cur = unit_entry(P, row, g, b0, it.kv_end, lane);
    int nxt = unit_entry(P, row, g, b0 + 1, it.kv_end, lane);
    for (int j = it.kt0; j < it.kt1; ++j, ++rc) {
        if (j > it.kt0 && (j & tpb_mask) == 0) {
            cur = nxt;
            nxt = unit_entry(P, row, g, (j >> g.lg_tpb) + 1, it.kv_end, lane);
        }
        const int lb = (j & tpb_mask) << g.lg_upt;  // lane of the tile's unit 0
        // lane u < upt checks unit u of the tile
        const int e = __shfl_sync(0xffffffffu, cur, lb + min(lane, g.upt - 1));
        const bool use = lane < g.upt && j * kKN + (lane << g.lg_tbr) < it.kv_end;
        const bool bad_l = use && (e < 0 || e >= P.num_blocks);
        const unsigned good = __ballot_sync(0xffffffffu, use && !bad_l);
        const unsigned bad_u = __ballot_sync(0xffffffffu, bad_l);
        if (!kIsV && bad_u && lane == 0 && P.err) atomicOr(P.err, PA_ERRBIT_BLOCK_OOB);
        const uint32_t tx = unit_bytes * (uint32_t)__popc(good);
        // this lane's copy: lane = u * copies + slice
        const int u = min(lane >> lg_cpu, g.upt - 1), sl = lane & ((1 << lg_cpu) - 1);
        const int pb = __shfl_sync(0xffffffffu, cur, lb + u);
        const bool issue = lane < (g.upt << lg_cpu) && ((good >> u) & 1u);
        const int tk = j * kKN + (u << g.lg_tbr);
        const int y = (((issue ? pb : 0) * P.num_kv_heads + it.hk) << P.block_shift) +
                      (tk & (P.block_size - 1));
        const size_t off = (size_t)sl * kSliceBytes + ((size_t)u << g.lg_tbr) * 128;
        const bool tail = kIsV && j == it.ntiles - 1 && tail_row != 0;
        const int slot = rc % R;

        bool ok = true;
        if (lane == 0) ok = mbar_wait(&empty[slot], (uint32_t)((rc / R) & 1) ^ 1u, abort_flag);
        if (!__shfl_sync(0xffffffffu, (int)ok, 0)) return false;
        unsigned char *st = skv + (size_t)slot * L::tile_bytes;
        if (kIsV && bad_u) {  // rows of skipped blocks: zeros, so 0-weight keys add nothing
            for (unsigned m = bad_u; m; m &= m - 1) {
                const int r0 = (__ffs(m) - 1) << g.lg_tbr;
                for (int q = lane; q < (KB * 8) << g.lg_tbr; q += 32) {
                    const int rr = r0 + q / (KB * 8), rest = q % (KB * 8);
                    *reinterpret_cast<uint4 *>(st + (size_t)(rest >> 3) * kSliceBytes +
                                               rr * 128 + (rest & 7) * 16) = make_uint4(0, 0, 0, 0);
                }
            }
            fence_proxy_async_smem();
        }
        uint64_t *bar = tail ? B.v_land : &full[slot];
        __syncwarp();
        if (lane == 0) {
            (kIsV ? B.v_tag : B.k_tag)[slot] = rc;  // before the arrival that arms the stage
            mbar_arrive_expect_tx(bar, tx);
        }
        __syncwarp();
        if (issue) tma_load_3d(st + off, tmap, 0, y, sl, bar, policy);
        __syncwarp();
        if (tail) {
            // the last tile: once it has landed, clear the rows past the last key
            land_pending = true;
            bool landed = true;
            if (lane == 0) landed = mbar_wait(B.v_land, (uint32_t)land & 1u, abort_flag);
            if (!__shfl_sync(0xffffffffu, (int)landed, 0)) return false;
            land_pending = false;
            ++land;
            for (int q = lane; q < (kKN - tail_row) * KB * 8; q += 32) {
                const int rr = tail_row + q / (KB * 8), rest = q % (KB * 8);
                *reinterpret_cast<uint4 *>(st + (size_t)(rest >> 3) * kSliceBytes + rr * 128 +
                                           (rest & 7) * 16) = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&full[slot]);
        }
    }
    return true;
}

// Rows of both tiles of an item whose sequence has lengths out of range: zeros.
__device__ __forceinline__ void zero_item_rows(const PrefillParams &P, const PItem &it,
                                               int lane) {
    if (lane == 0 && P.err) atomicOr(P.err, PA_ERRBIT_CONTEXT_LEN);
    const int a = P.query_start_loc[it.s], b = P.query_start_loc[it.s + 1];
    if (a < 0 || b > P.num_tokens || b <= a) return;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const int r0 = a + it.t[t].q0, r1 = min(b, r0 + kQM);
        for (int r = r0; r < r1; ++r)
            for (int d = lane; d < P.head_dim; d += 32)
                store_elem(P.out, P.out_dtype,
                           ((size_t)r * P.num_heads + it.t[t].h) * P.head_dim + d, 0.f);
    }
}

// warp 8: claims items, hands them out, loads Q and K
template <int D>
__device__ __forceinline__ void run_k_producer(const PrefillParams &P, unsigned char *sq,
                                               unsigned char *sk, PItem *items, const Bars &B,
                                               volatile int *abort_flag, int lane) {
    using L = PLayout<D>;
    const unsigned n_items = P.work[1];
    int n = 0, rc = 0, land = 0, qa[2] = {0, 0};
    bool land_pending = false, aborted = false;
    for (;;) {
        const int k = n & 1;
        bool ok = true;
        // slot k is free once every reader has taken item n - 2
        if (lane == 0 && n >= 2)
            ok = mbar_wait(&B.item_empty[k], (uint32_t)((n - 2) >> 1) & 1u, abort_flag);
        if (!__shfl_sync(0xffffffffu, (int)ok, 0)) {
            aborted = true;
            break;
        }
        unsigned id = 0xffffffffu, code = 0u;
        if (lane == 0) {
            const unsigned v = atomicAdd(&P.work[0], 1u);
            if (v < n_items) {
                const uint2 e = P.entries[v];
                id = e.x;
                code = e.y;
            }
        }
        id = __shfl_sync(0xffffffffu, id, 0);
        code = __shfl_sync(0xffffffffu, code, 0);
        PItem it;
        if (id != 0xffffffffu) {
            it = make_item(P, id);
            apply_part(it, code);
        } else {
            memset(&it, 0, sizeof(it));
            it.stop = true;
        }
        if (lane == 0) {
            items[k] = it;
            mbar_arrive(&B.item_full[k]);  // release: the item before the arrival
        }
        ++n;
        if (it.stop) break;
        if (!it.ok) {
            zero_item_rows(P, it, lane);
            continue;
        }
        // both Q tiles, each once the previous item's S products are done with it
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            if (!it.t[t].act) continue;
            if (lane == 0) {
                if (qa[t] > 0)
                    ok = ok && mbar_wait(&B.q_free[t], (uint32_t)(qa[t] - 1) & 1u, abort_flag);
                if (ok) {
                    mbar_arrive_expect_tx(&B.q_full[t], (uint32_t)L::qt_bytes);
                    tma_load_4d(sq + t * L::qt_bytes, &P.tmap_q, 0, it.t[t].h,
                                it.tok0 + it.t[t].q0, 0, &B.q_full[t]);
                    ++qa[t];
                }
            }
        }
        const KVItem kv{it.s, it.hk, it.kv_end, it.ntiles, it.kt0, it.kt1};
        if (!__shfl_sync(0xffffffffu, (int)ok, 0) ||
            !produce_item<D, false>(P, kv, sk, B, abort_flag, lane, rc, land, land_pending)) {
            aborted = true;
            break;
        }
    }
    if (aborted && lane == 0) {
        *abort_flag = 1;
        if (P.err) atomicOr(P.err, PA_ERRBIT_TIMEOUT);
    }
    // every copy issued lands before the CTA can exit
    if (lane == 0) {
        volatile int never = 0;
        for (int t = 0; t < 2; ++t)
            if (qa[t] > 0) mbar_drain_wait(&B.q_full[t], (uint32_t)(qa[t] - 1) & 1u, &never);
        const int first = rc > L::RK ? rc - L::RK : 0;
        for (int q = first; q < rc; ++q)
            mbar_drain_wait(&B.k_full[q % L::RK], (q / L::RK) & 1u, &never);
    }
    __syncwarp();
}

// warp 9: V
template <int D>
__device__ __forceinline__ void run_v_producer(const PrefillParams &P, unsigned char *sv,
                                               const PItem *items, const Bars &B,
                                               volatile int *abort_flag, int lane) {
    using L = PLayout<D>;
    int n = 0, rc = 0, land = 0;
    bool land_pending = false, aborted = false;
    for (;;) {
        const PItem *ip = take_item(items, B, n, abort_flag, lane, 0xffffffffu);
        if (!ip) {
            aborted = true;
            break;
        }
        const bool stop = ip->stop, iok = ip->ok;
        const KVItem kv{ip->s, ip->hk, ip->kv_end, ip->ntiles, ip->kt0, ip->kt1};
        give_item_back(B, n, lane, 0xffffffffu);
        ++n;
        if (stop) break;
        if (!iok) continue;
        if (!produce_item<D, true>(P, kv, sv, B, abort_flag, lane, rc, land, land_pending)) {
            aborted = true;
            break;
        }
    }
    if (aborted && lane == 0) {
        *abort_flag = 1;
        if (P.err) atomicOr(P.err, PA_ERRBIT_TIMEOUT);
    }
    // every copy issued lands before the CTA can exit; a tile abandoned while
    // its copies went to v_land waits there, not on its stage
    if (lane == 0) {
        volatile int never = 0;
        if (land_pending) mbar_drain_wait(B.v_land, (uint32_t)land & 1u, &never);
        // rc counts the tiles whose stage was armed (or, last of an item,
        // handed over after v_land)
        const int first = rc > L::RV ? rc - L::RV : 0;
        for (int q = first; q < rc; ++q)
            mbar_drain_wait(&B.v_full[q % L::RV], (q / L::RV) & 1u, &never);
    }
    __syncwarp();
}

// ---------------------------------------------------------------------------
// warps 10..13, one thread each: S (pv = 0) or P V (pv = 1) issue for query
// tile t, item after item
// ---------------------------------------------------------------------------
template <int D, bool kSplit>
__device__ __forceinline__ void run_mma_p(const PrefillParams &P, int t, int pv,
                                          const PItem *items, unsigned char *sq,
                                          unsigned char *sk, unsigned char *sv, uint32_t tmem,
                                          const Bars &B, volatile int *abort_flag) {
    using L = PLayout<D>;
    constexpr int RK = L::RK, RV = L::RV;
    constexpr int kNP = kSplit ? 1 : 2;                     // P buffers
    constexpr uint32_t fmt = kSplit ? 1u : 0u;
    const uint32_t idesc_s = umma_idesc_f16(fmt, 0, 0, kQM, kKN);
    const uint32_t idesc_o = umma_idesc_f16(fmt, 0, 1, kQM, D);
    const uint32_t aq = smem_u32(sq) + (uint32_t)(t * L::qt_bytes);
    const uint32_t ak = smem_u32(sk), av = smem_u32(sv);
    const uint32_t ts = tmem + (uint32_t)(t * 128);         // S, then P, of the tile
    const uint32_t to = tmem + 256u + (uint32_t)(t * D);    // O of the tile
    int n = 0, rc = 0, qa = 0, sc = 0, pc = 0, oa = 0;
    bool ok = true;
    for (;;) {
        const PItem *ip = take_item(items, B, n, abort_flag, 0, 1u);
        if (!ip) {
            ok = false;
            break;
        }
        const bool stop = ip->stop, iok = ip->ok;
        const int nt = t ? ip->t[1].nt : ip->t[0].nt;
        const int nt_other = t ? ip->t[0].nt : ip->t[1].nt;
        const int kt0 = ip->kt0, kt1 = ip->kt1;
        const int end = min(kt1, nt);  // this tile's K/V tiles in the entry: kt0 .. end-1
        give_item_back(B, n, 0, 1u);
        ++n;
        if (stop) break;
        if (!iok) continue;
        // A K/V stage is released by two arrivals, one per tile; past the
        // other tile's last K/V tile this issuer gives both.  An issuer never
        // arrives for a stage before it has seen that stage's tile land
        // (wait_tile), so its arrival cannot fall into an earlier phase.
        auto release = [&](uint64_t *bar, int j) {
            umma_commit(bar);
            if (j >= nt_other) umma_commit(bar);
        };
        if (!pv) {
            if (end > kt0) {
                ok = mbar_wait(&B.q_full[t], (uint32_t)qa & 1u, abort_flag);
                tc_fence_after();
            }
            // S_j into the tile's S buffer once the softmax has loaded the
            // previous S.  A K step of 16 is 32 bytes inside a 64-element
            // slice; slices are whole tiles apart.
            for (int j = kt0; ok && j < end; ++j, ++sc) {
                const int q = rc + (j - kt0), ks = q % RK;
                ok = wait_tile(B.k_full, B.k_tag, q, RK, abort_flag) &&
                     (sc == 0 || mbar_wait(&B.s_free[t], (uint32_t)(sc - 1) & 1u, abort_flag));
                if (!ok) break;
                tc_fence_after();
                const uint32_t kt = ak + (uint32_t)(ks * L::tile_bytes);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t in_slice = (uint32_t)((kk & 3) * 32);
                    const uint64_t da = umma_desc_sw128(
                        aq + (uint32_t)((kk >> 2) * kQM * 128) + in_slice, 16, 1024);
                    const uint64_t db =
                        umma_desc_sw128(kt + (uint32_t)(kk >> 2) * kSliceBytes + in_slice, 16, 1024);
                    umma_f16(ts, da, db, idesc_s, kk > 0 ? 1u : 0u);
                }
                umma_commit(&B.s_full[t]);
                release(&B.k_empty[ks], j);
            }
            if (end > kt0) {
                umma_commit(&B.q_free[t]);  // Q_t is not read once these have completed
                ++qa;
            }
        } else {
            // O += P_j V_j: P from its buffer (hi, then lo for bf16 32 columns
            // on), V MN-major (16 keys = 2048 bytes per K step, slices of
            // head_dim a tile slice apart); the item's first product starts
            // O afresh once the softmax has read out the previous item's O
            for (int j = kt0; ok && j < end; ++j, ++pc) {
                const int q = rc + (j - kt0), vs = q % RV, pb = pc % kNP;
                ok = wait_tile(B.v_full, B.v_tag, q, RV, abort_flag) &&
                     mbar_wait(&B.p_full[2 * t + pb], (uint32_t)(pc / kNP) & 1u, abort_flag) &&
                     (j > kt0 || oa == 0 ||
                      mbar_wait(&B.o_free[t], (uint32_t)(oa - 1) & 1u, abort_flag));
                if (!ok) break;
                tc_fence_after();
                const uint32_t vt = av + (uint32_t)(vs * L::tile_bytes);
                const uint32_t tp = ts + 64u + (uint32_t)(pb * 32);
#pragma unroll
                for (int kk = 0; kk < kKN / 16; ++kk) {
                    const uint64_t db =
                        umma_desc_sw128(vt + (uint32_t)(kk * 16 * 128), kSliceBytes, 1024);
                    umma_f16_tmem_a(to, tp + (uint32_t)(kk * 8), db, idesc_o,
                                    (j > kt0 || kk > 0) ? 1u : 0u);
                    if constexpr (kSplit)
                        umma_f16_tmem_a(to, tp + 32u + (uint32_t)(kk * 8), db, idesc_o, 1u);
                }
                umma_commit(&B.pv_done[2 * t + pb]);
                release(&B.v_empty[vs], j);
            }
            if (end > kt0) ++oa;
        }
        if (!ok) break;
        rc += kt1 - kt0;
    }
    if (!ok) {
        *abort_flag = 1;
        if (P.err) atomicOr(P.err, PA_ERRBIT_TIMEOUT);
    }
    umma_commit(&B.o_done[2 * t + pv]);  // after every MMA issued: the teardown
}

// ---------------------------------------------------------------------------
// output of one warp's 32 rows (O / sum), staged through shared memory in
// rounds of CR columns (128 bytes a row): the row of lane r in stage row r
// with its 16-byte chunks swizzled by r % 8 -- the layout of a TMA box of 32
// rows with the 128-byte swizzle.  When all 32 rows belong to the sequence a
// round leaves as one tiled bulk store (the warp waits only for the copy
// engine to read the stage); otherwise four rows per store instruction, rows
// past the sequence skipped.  O is released (o_free) once the last round has
// been loaded.
// ---------------------------------------------------------------------------
template <typename OutT>
__device__ __forceinline__ uint4 pack_out(const float *v);
template <>
__device__ __forceinline__ uint4 pack_out<float>(const float *v) {
    return make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]),
                      __float_as_uint(v[3]));
}
template <>
__device__ __forceinline__ uint4 pack_out<__half>(const float *v) {
    return make_uint4(pack2<__half>(v[0], v[1]), pack2<__half>(v[2], v[3]),
                      pack2<__half>(v[4], v[5]), pack2<__half>(v[6], v[7]));
}
template <>
__device__ __forceinline__ uint4 pack_out<__nv_bfloat16>(const float *v) {
    return make_uint4(pack2<__nv_bfloat16>(v[0], v[1]), pack2<__nv_bfloat16>(v[2], v[3]),
                      pack2<__nv_bfloat16>(v[4], v[5]), pack2<__nv_bfloat16>(v[6], v[7]));
}

template <int D, typename OutT>
__device__ __forceinline__ void store_rows(const PrefillParams &P, const SeqRows &it,
                                           const PTile &tl, uint32_t tm_o, float inv,
                                           unsigned char *stage, uint64_t *o_free, int wq,
                                           int lane) {
    constexpr int ES = (int)sizeof(OutT);
    constexpr int CR = kStageWarpBytes / (32 * ES);            // columns a round
    constexpr int NCH = CR * ES / 16;                           // 16-byte chunks a row
    constexpr int PER = 16 / ES;                                // elements a chunk
    static_assert(D % CR == 0 && NCH == 8, "staging shape");
    const int row0 = tl.q0 + 32 * wq;                           // tile row of lane 0
    const bool whole = row0 + 32 <= it.n;                       // every row in the sequence
#pragma unroll
    for (int q = 0; q < D / CR; ++q) {
        if (lane == 0) bulk_wait_read();  // the stage's previous store has read it
        __syncwarp();
        uint32_t u[CR];
#pragma unroll
        for (int c = 0; c < CR; c += 16)
            tmem_ld16(tm_o + (uint32_t)(q * CR + c), *reinterpret_cast<uint32_t(*)[16]>(&u[c]));
        tmem_wait_ld();
        if (q == D / CR - 1) {  // all of O has been read: the next item may start it afresh
            tc_fence_before();
            mbar_arrive(o_free);
        }
#pragma unroll
        for (int k = 0; k < NCH; ++k) {
            float v[PER];
#pragma unroll
            for (int e = 0; e < PER; ++e) v[e] = __uint_as_float(u[k * PER + e]) * inv;
            const int pos = k ^ (lane & 7);
            *reinterpret_cast<uint4 *>(stage + lane * (CR * ES) + pos * 16) = pack_out<OutT>(v);
        }
        if (whole) {
            fence_proxy_async_smem();  // the stage, before the copy engine reads it
            __syncwarp();
            if (lane == 0) tma_store_3d(&P.tmap_out, q * CR, tl.h, it.tok0 + row0, stage);
            continue;
        }
        __syncwarp();
#pragma unroll
        for (int it2 = 0; it2 < NCH; ++it2) {
            const int rr = it2 * (32 / NCH) + lane / NCH, k = lane % NCH;
            const int pos = k ^ (rr & 7);
            const uint4 w = *reinterpret_cast<const uint4 *>(stage + rr * (CR * ES) + pos * 16);
            if (row0 + rr < it.n) {
                const size_t tok = (size_t)it.tok0 + row0 + rr;
                unsigned char *dst = static_cast<unsigned char *>(P.out) +
                                     ((tok * P.num_heads + tl.h) * D + q * CR) * ES + k * 16;
                *reinterpret_cast<uint4 *>(dst) = w;
            }
        }
        __syncwarp();
    }
}

// ---------------------------------------------------------------------------
// split items.  Each part leaves its tile's unnormalised O (relative to its
// base-2 maximum m) with m and the sum l in the workspace; the part that
// finishes second combines them exactly:
//     M = max(m_0, m_1),  c_p = 2^(m_p - M),  o = (c_0 O_0 + c_1 O_1) / (c_0 l_0 + c_1 l_1)
// (a part that saw no key of a row has m = -inf and weighs nothing)
// [Efficient Memory Management ..., "PagedAttention Algorithm": blocks may be
// processed in any order and combined; vLLM Internals ..., partitions of a
// long sequence merged afterwards].
// ---------------------------------------------------------------------------
__device__ __forceinline__ size_t part_row(int slot, int part, int t) {
    return (((size_t)slot * 2 + part) * 2 + t) * kQM;
}

// The tile's O rows (raw, fp32), m and l of part `part` to the workspace,
// staged through shared memory so that stores write whole 128-byte rows.
template <int D>
__device__ __forceinline__ void store_partial(const PrefillParams &P, int slot, int part, int t,
                                              uint32_t tm_o, float m, float l,
                                              unsigned char *stage, uint64_t *o_free, int wq,
                                              int lane) {
    constexpr int CR = kStageWarpBytes / (32 * 4);  // 32 fp32 columns a round
    const int r0 = 32 * wq;
    const size_t prow = part_row(slot, part, t);
    P.part_m[prow + r0 + lane] = m;
    P.part_l[prow + r0 + lane] = l;
    float *base = P.part_o + (prow + r0) * D;
#pragma unroll
    for (int q = 0; q < D / CR; ++q) {
        if (lane == 0) bulk_wait_read();  // the stage's last tiled store has read it
        __syncwarp();
        uint32_t u[CR];
#pragma unroll
        for (int c = 0; c < CR; c += 16)
            tmem_ld16(tm_o + (uint32_t)(q * CR + c), *reinterpret_cast<uint32_t(*)[16]>(&u[c]));
        tmem_wait_ld();
        if (q == D / CR - 1) {  // all of O has been read: the next item may start it afresh
            tc_fence_before();
            mbar_arrive(o_free);
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int pos = k ^ (lane & 7);
            *reinterpret_cast<uint4 *>(stage + lane * 128 + pos * 16) =
                make_uint4(u[4 * k], u[4 * k + 1], u[4 * k + 2], u[4 * k + 3]);
        }
        __syncwarp();
#pragma unroll
        for (int it2 = 0; it2 < 8; ++it2) {
            const int rr = it2 * 4 + lane / 8, k = lane % 8;
            const uint4 w = *reinterpret_cast<const uint4 *>(stage + rr * 128 + ((k ^ (rr & 7)) * 16));
            *reinterpret_cast<uint4 *>(base + (size_t)rr * D + q * CR + k * 4) = w;
        }
        __syncwarp();
    }
}

// After a part's results are in the workspace: count the part finished for
// tile t of split slot `slot`; true in the 128 threads of the part that
// finished second.
__device__ __forceinline__ bool split_last(const PrefillParams &P, int slot, int t,
                                           volatile unsigned *split_old, int lane) {
    __threadfence();  // this part's results, before the count
    asm volatile("bar.sync %0, %1;" ::"r"(1 + t), "n"(kTileThreads) : "memory");
    if (threadIdx.x % kTileThreads == 0) split_old[t] = atomicAdd(&P.split_cnt[slot * 2 + t], 1u);
    asm volatile("bar.sync %0, %1;" ::"r"(1 + t), "n"(kTileThreads) : "memory");
    const bool last = split_old[t] == 1u;
    asm volatile("bar.sync %0, %1;" ::"r"(1 + t), "n"(kTileThreads) : "memory");
    if (last) __threadfence();  // the other part's results, after the count
    return last;
}

template <typename OutT>
__device__ __forceinline__ void store4(void *out, size_t idx, float4 v);
template <>
__device__ __forceinline__ void store4<float>(void *out, size_t idx, float4 v) {
    *reinterpret_cast<float4 *>(static_cast<float *>(out) + idx) = v;
}
template <>
__device__ __forceinline__ void store4<__half>(void *out, size_t idx, float4 v) {
    *reinterpret_cast<uint2 *>(static_cast<__half *>(out) + idx) =
        make_uint2(pack2<__half>(v.x, v.y), pack2<__half>(v.z, v.w));
}
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(void *out, size_t idx, float4 v) {
    *reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(out) + idx) =
        make_uint2(pack2<__nv_bfloat16>(v.x, v.y), pack2<__nv_bfloat16>(v.z, v.w));
}

// The merge of both parts for the warp's 32 rows: lane r holds row r's
// weights; rows are read and written four at a time, 32 columns (128 bytes
// of fp32) a row per instruction.
template <int D, typename OutT>
__device__ __forceinline__ void merge_rows(const PrefillParams &P, const SeqRows &sr,
                                           const PTile &tl, int slot, int t, int wq, int lane) {
    const int r0 = 32 * wq;
    const size_t p0 = part_row(slot, 0, t) + r0, p1 = part_row(slot, 1, t) + r0;
    const float m0 = P.part_m[p0 + lane], m1 = P.part_m[p1 + lane];
    const float l0 = P.part_l[p0 + lane], l1 = P.part_l[p1 + lane];
    const float M = fmaxf(m0, m1);
    const float c0 = m0 == -INFINITY ? 0.f : ex2(m0 - M);
    const float c1 = m1 == -INFINITY ? 0.f : ex2(m1 - M);
    const float lt = c0 * l0 + c1 * l1;
    const float inv = lt > 0.f ? 1.f / lt : 0.f;
    const float w0 = c0 * inv, w1 = c1 * inv;
    const float *o0 = P.part_o + p0 * D, *o1 = P.part_o + p1 * D;
#pragma unroll 2
    for (int g4 = 0; g4 < 8; ++g4) {
        const int rr = g4 * 4 + lane / 8;          // the row this lane works on
        const float a0 = __shfl_sync(0xffffffffu, w0, rr);
        const float a1 = __shfl_sync(0xffffffffu, w1, rr);
        const int row = tl.q0 + r0 + rr;
        const bool live = row < sr.n;
#pragma unroll
        for (int cb = 0; cb < D; cb += 32) {
            const int col = cb + (lane % 8) * 4;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (a0 != 0.f) {
                const float4 x = *reinterpret_cast<const float4 *>(o0 + (size_t)rr * D + col);
                v = make_float4(a0 * x.x, a0 * x.y, a0 * x.z, a0 * x.w);
            }
            if (a1 != 0.f) {
                const float4 x = *reinterpret_cast<const float4 *>(o1 + (size_t)rr * D + col);
                v = make_float4(fmaf(a1, x.x, v.x), fmaf(a1, x.y, v.y), fmaf(a1, x.z, v.z),
                                fmaf(a1, x.w, v.w));
            }
            if (live)
                store4<OutT>(P.out, (((size_t)sr.tok0 + row) * P.num_heads + tl.h) * D + col, v);
        }
    }
}

template <int D, typename T>
__device__ __forceinline__ void merge_parts(const PrefillParams &P, const SeqRows &sr,
                                            const PTile &tl, int slot, int t, int wq, int lane) {
    if (P.out_dtype == PA_F32)
        merge_rows<D, float>(P, sr, tl, slot, t, wq, lane);
    else
        merge_rows<D, T>(P, sr, tl, slot, t, wq, lane);
}

// Out-of-line copies of the split-item paths.  The bf16 kernel (P in two
// parts) calls these: kept out of its softmax branch they leave that branch
// smaller, which measured faster (GQA heads 430 against 414 TFLOP/s); the
// fp16 kernel measured faster with them inline (705 against 648).
template <int D>
__device__ __noinline__ void store_partial_call(const PrefillParams &P, int slot, int part,
                                                int t, uint32_t tm_o, float m, float l,
                                                unsigned char *stage, uint64_t *o_free, int wq,
                                                int lane) {
    store_partial<D>(P, slot, part, t, tm_o, m, l, stage, o_free, wq, lane);
}

template <int D, typename T>
__device__ __noinline__ void merge_parts_call(const PrefillParams &P, const SeqRows &sr,
                                              const PTile &tl, int slot, int t, int wq,
                                              int lane) {
    merge_parts<D, T>(P, sr, tl, slot, t, wq, lane);
}

// ---------------------------------------------------------------------------
// warps 0..7: softmax of query tile t = warp / 4, one row per thread, and the
// output, item after item
// ---------------------------------------------------------------------------
template <int D, typename T, bool kSplit>
__device__ __forceinline__ void run_softmax_p(const PrefillParams &P, int t, const PItem *items,
                                              unsigned char *stage, uint32_t tmem,
                                              const Bars &B, volatile int *abort_flag,
                                              volatile unsigned *split_old, int wq, int lane) {
    constexpr int kNP = kSplit ? 1 : 2;      // P buffers
    const int r = 32 * wq + lane;            // this thread's query row
    const uint32_t lane_addr = (uint32_t)(32 * wq) << 16;
    const uint32_t tm_s = tmem + (uint32_t)(t * 128) + lane_addr;
    const uint32_t tm_o = tmem + 256u + (uint32_t)(t * D) + lane_addr;
    const float sc = P.scale_log2;
    const bool fold = sc > 0.f;             // the same in every thread
    const float psc = fold ? sc : 1.f;      // scale applied in the exponent
    const float msc = fold ? 1.f : sc;      // scale applied before the maximum
    const UnitGeo g = unit_geo(P.block_shift);
    const int tpb_mask = (1 << g.lg_tpb) - 1;
    const unsigned unit_mask = (1u << g.upt) - 1u;
    int n = 0, scount = 0, pc = 0;
    bool ok = true;
    for (;;) {
        const PItem *ip = take_item(items, B, n, abort_flag, lane, 0xffffffffu);
        if (!ip) {
            ok = false;
            break;
        }
        const bool stop = ip->stop;
        const PTile tl = t ? ip->t[1] : ip->t[0];
        const SeqRows sr{ip->s, ip->n, ip->c, ip->L, ip->tok0};
        const int kt0 = ip->kt0, end = min(ip->kt1, tl.nt);  // this tile's K/V tiles
        const int slot = ip->slot, part = ip->part;
        give_item_back(B, n, lane, 0xffffffffu);
        ++n;
        if (stop) break;
        if (!tl.act) continue;
        if (end <= kt0) {  // a part of a split item with no keys for this tile
            const size_t mi = (((size_t)slot * 2 + part) * 2 + t) * kQM + r;
            P.part_m[mi] = -INFINITY;
            P.part_l[mi] = 0.f;
            if (split_last(P, slot, t, split_old, lane)) {
                if constexpr (kSplit) merge_parts_call<D, T>(P, sr, tl, slot, t, wq, lane);
                else merge_parts<D, T>(P, sr, tl, slot, t, wq, lane);
            }
            continue;
        }
        const int i = tl.q0 + r;                 // new-token index of the row
        const int qpos = i < sr.n ? sr.c + i : sr.L - 1;  // padding rows see every key
        // skipped blocks, from the table: bit u of a tile's mask = unit u
        // (the same test as the producers': a unit below kv_end with an id out
        // of range)
        const int32_t *row = P.block_tables + (size_t)sr.s * P.max_blocks_per_seq;
        auto bad_of = [&](int e, int bt) {
            const int tok = ((bt << 5) + lane) << g.lg_tbr;
            return __ballot_sync(0xffffffffu, tok < tl.kv_end && (e < 0 || e >= P.num_blocks));
        };
        const int b0 = kt0 >> g.lg_tpb;  // table batch of the first tile
        unsigned bb = bad_of(unit_entry(P, row, g, b0, tl.kv_end, lane), b0);
        int e_nxt = unit_entry(P, row, g, b0 + 1, tl.kv_end, lane);
        float m_ref = -INFINITY, lsum = 0.f;
        for (int j = kt0; j < end; ++j, ++scount, ++pc) {
            if (j > kt0 && (j & tpb_mask) == 0) {
                const int bt = j >> g.lg_tpb;
                bb = bad_of(e_nxt, bt);
                e_nxt = unit_entry(P, row, g, bt + 1, tl.kv_end, lane);
            }
            const unsigned bits = (bb >> ((j & tpb_mask) << g.lg_upt)) & unit_mask;
            if (!__all_sync(0xffffffffu,
                            mbar_wait(&B.s_full[t], (uint32_t)scount & 1u, abort_flag))) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t su[kKN];
#pragma unroll
            for (int c = 0; c < kKN; c += 16)
                tmem_ld16(tm_s + (uint32_t)c, *reinterpret_cast<uint32_t(*)[16]>(&su[c]));
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(&B.s_free[t]);  // the S buffer may take the next S
            float s[kKN];
#pragma unroll
            for (int e = 0; e < kKN; ++e) s[e] = __uint_as_float(su[e]);
            const int kb = j * kKN;
            // Keys past the row's position or in a skipped block read -inf.
            // With a positive scale the maximum is taken over the raw scores
            // and the scale goes into the exponent's FMA below (one multiply
            // a key less); otherwise the scores are scaled first.  In both
            // forms s ends up in units with p = 2^(s * psc - m).  One warp per
            // scheduler runs this code, so the reductions keep eight
            // independent chains.
            constexpr int kAcc = 8;
            float mxa[kAcc];
#pragma unroll
            for (int q = 0; q < kAcc; ++q) mxa[q] = -INFINITY;
            // the masked form is taken by the whole warp or not at all (a
            // warp on the diagonal would otherwise run both)
            if (__all_sync(0xffffffffu, !bits && kb + kKN - 1 <= qpos)) {  // all keys visible
                if (fold) {
#pragma unroll
                    for (int e = 0; e < kKN; ++e) mxa[e % kAcc] = fmaxf(mxa[e % kAcc], s[e]);
                } else {
#pragma unroll
                    for (int e = 0; e < kKN; ++e) {
                        s[e] *= sc;
                        mxa[e % kAcc] = fmaxf(mxa[e % kAcc], s[e]);
                    }
                }
            } else {
                // keys kb .. kb + nvis - 1 are at or before the row's position
                const int nvis = max(0, min(kKN, qpos - kb + 1));
                if (!bits) {  // (bits is the same in every lane)
#pragma unroll
                    for (int e = 0; e < kKN; ++e) {
                        s[e] = e >= nvis ? -INFINITY : s[e] * msc;
                        mxa[e % kAcc] = fmaxf(mxa[e % kAcc], s[e]);
                    }
                } else {  // and the keys of skipped blocks
#pragma unroll
                    for (int e = 0; e < kKN; ++e) {
                        const bool masked = e >= nvis || ((bits >> (e >> g.lg_tbr)) & 1u);
                        s[e] = masked ? -INFINITY : s[e] * msc;
                        mxa[e % kAcc] = fmaxf(mxa[e % kAcc], s[e]);
                    }
                }
            }
#pragma unroll
            for (int q = 1; q < kAcc; ++q) mxa[0] = fmaxf(mxa[0], mxa[q]);
            const float mx = fmaxf(m_ref, mxa[0] * psc);  // base-2 units
            // lazy rescale: only when the maximum grew by more than 2^8; O
            // must then be stable (the item's previous P V finished)
            const bool grow = mx > m_ref + kRescaleLog2;
            if (__any_sync(0xffffffffu, grow)) {
                const float alpha = grow && m_ref != -INFINITY ? ex2(m_ref - mx) : 1.f;
                if (j > kt0) {
                    const int pq = pc - 1;
                    if (!__all_sync(0xffffffffu,
                                    mbar_wait(&B.pv_done[2 * t + pq % kNP],
                                              (uint32_t)(pq / kNP) & 1u, abort_flag))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < D; c += 16) {
                        uint32_t u[16];
                        tmem_ld16(tm_o + (uint32_t)c, u);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            u[e] = __float_as_uint(__uint_as_float(u[e]) * alpha);
                        tmem_st16(tm_o + (uint32_t)c, u);
                    }
                }
                if (grow) {
                    lsum *= alpha;
                    m_ref = mx;
                }
            }
            const float ms = m_ref == -INFINITY ? 0.f : m_ref;
            // the P buffer is free once the P V that read it kNP products ago
            // has completed
            const int pb = pc % kNP;
            if (pc >= kNP && !__all_sync(0xffffffffu,
                                         mbar_wait(&B.pv_done[2 * t + pb],
                                                   (uint32_t)((pc - kNP) / kNP) & 1u,
                                                   abort_flag))) {
                ok = false;
                break;
            }
            // P: column c of the buffer holds keys 2c, 2c+1
            uint32_t ph[kKN / 2], pl[kKN / 2];
            float lsa[kAcc];
#pragma unroll
            for (int q = 0; q < kAcc; ++q) lsa[q] = 0.f;
#pragma unroll
            for (int c = 0; c < kKN / 2; ++c) {
                const float p0 = ex2(fmaf(s[2 * c], psc, -ms)), p1 = ex2(fmaf(s[2 * c + 1], psc, -ms));
                lsa[(2 * c) % kAcc] += p0;
                lsa[(2 * c + 1) % kAcc] += p1;
                ph[c] = pack2<T>(p0, p1);
                if constexpr (kSplit) {
                    const float2 h = unpack2<T>(ph[c]);
                    pl[c] = pack2<T>(p0 - h.x, p1 - h.y);
                }
            }
#pragma unroll
            for (int q = 0; q < kAcc; ++q) lsum += lsa[q];
            const uint32_t pcol = tm_s + 64u + (uint32_t)(pb * 32);
            tmem_st16(pcol, *reinterpret_cast<const uint32_t(*)[16]>(&ph[0]));
            tmem_st16(pcol + 16u, *reinterpret_cast<const uint32_t(*)[16]>(&ph[16]));
            if constexpr (kSplit) {
                tmem_st16(pcol + 32u, *reinterpret_cast<const uint32_t(*)[16]>(&pl[0]));
                tmem_st16(pcol + 48u, *reinterpret_cast<const uint32_t(*)[16]>(&pl[16]));
            }
            tmem_wait_st();  // P (and a rescaled O) before the tensor core reads them
            tc_fence_before();
            mbar_arrive(&B.p_full[2 * t + pb]);
        }
        if (!ok) break;
        // epilogue: O / sum once the tile's last P V has completed
        const int last = pc - 1;
        if (!__all_sync(0xffffffffu, mbar_wait(&B.pv_done[2 * t + last % kNP],
                                               (uint32_t)(last / kNP) & 1u, abort_flag))) {
            ok = false;
            break;
        }
        tc_fence_after();
        if (slot < 0) {
            const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
            if (P.out_dtype == PA_F32)
                store_rows<D, float>(P, sr, tl, tm_o, inv, stage, &B.o_free[t], wq, lane);
            else
                store_rows<D, T>(P, sr, tl, tm_o, inv, stage, &B.o_free[t], wq, lane);
        } else {
            // a part of a split item: its O, maximum and sum to the workspace;
            // the part that finishes second merges both
            if constexpr (kSplit)
                store_partial_call<D>(P, slot, part, t, tm_o, m_ref, lsum, stage, &B.o_free[t], wq,
                                      lane);
            else
                store_partial<D>(P, slot, part, t, tm_o, m_ref, lsum, stage, &B.o_free[t], wq, lane);
            if (split_last(P, slot, t, split_old, lane)) {
                if constexpr (kSplit) merge_parts_call<D, T>(P, sr, tl, slot, t, wq, lane);
                else merge_parts<D, T>(P, sr, tl, slot, t, wq, lane);
            }
        }
    }
    if (!ok) {
        *abort_flag = 1;
        if (P.err) atomicOr(P.err, PA_ERRBIT_TIMEOUT);
    }
    if (lane == 0) bulk_wait_all();  // the output has left shared memory and landed
    __syncwarp();
}

template <int D, typename T>
__global__ void __launch_bounds__(kThreadsP, 1)
    paged_prefill_kernel(const __grid_constant__ PrefillParams P) {
    constexpr bool kSplit = std::is_same<T, __nv_bfloat16>::value;
    using L = PLayout<D>;
    constexpr int RK = L::RK, RV = L::RV;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char *sq = smem + L::q_off;
    unsigned char *sk = smem + L::k_off;
    unsigned char *sv = smem + L::v_off;
    PItem *items = reinterpret_cast<PItem *>(smem + L::item_off);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::bar_off);
    Bars B;
    B.k_tag = reinterpret_cast<volatile int *>(smem + L::tag_off);
    B.v_tag = B.k_tag + RK;
    B.q_full = bars;
    B.q_free = B.q_full + 2;
    B.k_full = B.q_free + 2;
    B.k_empty = B.k_full + RK;
    B.v_full = B.k_empty + RK;
    B.v_empty = B.v_full + RV;
    B.v_land = B.v_empty + RV;
    B.item_full = B.v_land + 1;
    B.item_empty = B.item_full + 2;
    B.s_full = B.item_empty + 2;
    B.s_free = B.s_full + 2;
    B.p_full = B.s_free + 2;
    B.pv_done = B.p_full + 4;
    B.o_free = B.pv_done + 4;
    B.o_done = B.o_free + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::tmem_off);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::flag_off);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    pdl_trigger();
    if (threadIdx.x == 0) {
        prefetch_tmap(&P.tmap_q);
        prefetch_tmap(&P.tmap_k);
        prefetch_tmap(&P.tmap_v);
        prefetch_tmap(&P.tmap_out);
        for (int b = 0; b < L::kBars; ++b) mbar_init(&bars[b], 1);
        for (int b = 0; b < 4; ++b) mbar_init(&B.p_full[b], kTileThreads);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&B.s_free[b], kTileThreads);
            mbar_init(&B.o_free[b], kTileThreads);
            mbar_init(&B.item_empty[b], kItemReaders);
        }
        for (int b = 0; b < RK; ++b) mbar_init(&B.k_empty[b], 2);  // one arrival per tile
        for (int b = 0; b < RV; ++b) mbar_init(&B.v_empty[b], 2);
        for (int b = 0; b < RK + RV; ++b) B.k_tag[b] = -1;
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kWarpAlloc) tmem_alloc(tmem_slot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // each role's code follows its own register reallocation (code after a
    // join of the two would be held to the smaller count)
    if (warp < kSoftmaxWarps) {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
        pdl_wait();  // the plan, and through it the cache write of the chunk, is complete
        run_softmax_p<D, T, kSplit>(
            P, warp >> 2, items, smem + L::stage_off + (size_t)warp * kStageWarpBytes, tmem, B,
            abort_flag, reinterpret_cast<volatile unsigned *>(smem + L::split_off), warp & 3, lane);
    } else {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsOther));
        pdl_wait();
        if (warp == kWarpK) {
            run_k_producer<D>(P, sq, sk, items, B, abort_flag, lane);
        } else if (warp == kWarpV) {
            run_v_producer<D>(P, sv, items, B, abort_flag, lane);
        } else if (warp >= kWarpS && warp < kWarpPV + 2) {
            const int pv = warp >= kWarpPV ? 1 : 0, t = warp - (pv ? kWarpPV : kWarpS);
            if (lane == 0) {
                run_mma_p<D, kSplit>(P, t, pv, items, sq, sk, sv, tmem, B, abort_flag);
                // every MMA it issued has completed before tensor memory is released
                volatile int never = 0;
                mbar_drain_wait(&B.o_done[2 * t + pv], 0, &never);
            }
            __syncwarp();
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kWarpAlloc) tmem_dealloc(tmem, kTmemCols);
}

template <int D, typename T>
pa_status_t launch_prefill(const PrefillParams &P, unsigned grid, cudaStream_t stream) {
    using L = PLayout<D>;
    auto kern = paged_prefill_kernel<D, T>;
    static std::atomic<bool> attr_set[kMaxDevicesP];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevicesP) return PA_ERR_CUDA;
    if (!attr_set[dev].load(std::memory_order_relaxed)) {
        // the register reallocation inside the kernel assumes exactly
        // kRegsLaunch registers a thread at launch; anything else is refused
        cudaFuncAttributes fa;
        if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return PA_ERR_CUDA;
        if (fa.numRegs != kRegsLaunch) return PA_ERR_UNSUPPORTED;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)L::bytes) != cudaSuccess)
            return PA_ERR_CUDA;
        attr_set[dev].store(true, std::memory_order_relaxed);
    }
    if (launch_pdl(prefill_plan_kernel, dim3(1), dim3(kPlanThreads), 0, stream, P) != cudaSuccess)
        return PA_ERR_CUDA;
    return launch_pdl(kern, dim3(grid), dim3(kThreadsP), L::bytes, stream, P) == cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

int shift_of(int b) {
    for (int sh = 3; sh <= 8; ++sh)
        if (b == (1 << sh)) return sh;
    return -1;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Items of a batch: (num_seqs, items_x, items_y); false if out of range.
bool item_grid(int num_seqs, int num_heads, int num_kv_heads, int max_query_len, int *ix,
               int *iy, unsigned long long *count) {
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || max_query_len < 0 ||
        num_heads % num_kv_heads != 0)
        return false;
    const long long mtiles = ((long long)max_query_len + kQM - 1) / kQM;
    const bool pair_heads = (num_heads / num_kv_heads) % 2 == 0;
    *ix = (int)(pair_heads ? mtiles : (mtiles + 1) / 2);
    *iy = pair_heads ? num_heads / 2 : num_heads;
    *count = (unsigned long long)num_seqs * (unsigned long long)*ix * (unsigned long long)*iy;
    return true;
}

// Workspace layout for a batch (byte offsets, 256-byte aligned).
struct PWork {
    int max_splits;
    size_t entries, split_cnt, part_m, part_l, part_o, bytes;
};

size_t align256p(size_t x) { return (x + 255) / 256 * 256; }

PWork work_layout(unsigned long long n_items, int head_dim) {
    PWork w;
    w.max_splits = (int)(n_items < (unsigned long long)kMaxSplits ? n_items : kMaxSplits);
    const size_t ms = (size_t)w.max_splits;
    size_t off = align256p(kWorkHeader * sizeof(uint32_t));
    w.entries = off;
    off = align256p(off + 2 * (size_t)n_items * sizeof(uint2));
    w.split_cnt = off;
    off = align256p(off + ms * 2 * sizeof(uint32_t));
    w.part_m = off;
    off = align256p(off + ms * 4 * kQM * sizeof(float));
    w.part_l = off;
    off = align256p(off + ms * 4 * kQM * sizeof(float));
    w.part_o = off;
    off = align256p(off + ms * 4 * kQM * (size_t)head_dim * sizeof(float));
    w.bytes = off;
    return w;
}

int sm_count() {
    static std::atomic<int> cached[kMaxDevicesP];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevicesP) return 0;
    int v = cached[dev].load(std::memory_order_relaxed);
    if (v == 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return 0;
        cached[dev].store(v, std::memory_order_relaxed);
    }
    return v;
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" size_t pa_prefill_workspace_size(int num_seqs, int num_heads, int num_kv_heads,
                                            int head_dim, int max_query_len) {
    int ix = 0, iy = 0;
    unsigned long long count = 0;
    if (head_dim != 64 && head_dim != 128) return 0;
    if (!item_grid(num_seqs, num_heads, num_kv_heads, max_query_len, &ix, &iy, &count))
        return 0;
    if (count >= (1ull << 31)) return 0;
    return work_layout(count, head_dim).bytes;
}

extern "C" pa_status_t pa_prefill_attention(
    void *out, pa_dtype_t out_dtype, const void *query, const void *k_cache, const void *v_cache,
    const int32_t *block_tables, int max_blocks_per_seq, const int32_t *query_start_loc,
    const int32_t *context_lens, int max_query_len, int max_context_len, int num_seqs,
    int num_tokens, int num_heads, int num_kv_heads, int head_dim, int num_blocks,
    int block_size, float scale, pa_dtype_t dtype, void *workspace, size_t workspace_bytes,
    unsigned int *dev_error_word, pa_stream_t stream) {
    PA_NVTX_RANGE("pa_prefill_attention");
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
    int ix = 0, iy = 0;
    unsigned long long n_items = 0;
    if (!item_grid(num_seqs, num_heads, num_kv_heads, max_query_len, &ix, &iy, &n_items))
        return PA_ERR_INVALID_ARG;
    if (n_items >= (1ull << 31)) return PA_ERR_UNSUPPORTED;
    if (num_seqs == 0 || num_tokens == 0 || max_query_len == 0) return PA_OK;
    if (!out || !query || !k_cache || !v_cache || !block_tables || !query_start_loc ||
        !context_lens || !workspace)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(query) || !aligned16(k_cache) || !aligned16(v_cache))
        return PA_ERR_INVALID_ARG;
    const PWork wl = work_layout(n_items, head_dim);
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < wl.bytes)
        return PA_ERR_WORKSPACE;
    const int sms = sm_count();
    if (sms <= 0) return PA_ERR_CUDA;

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
    {  // out [tokens][heads][head_dim]; a box is 32 rows of 128 bytes
        const cuuint64_t es = out_dtype == PA_F32 ? 4u : 2u;
        const cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)num_heads,
                                    (cuuint64_t)num_tokens};
        const cuuint64_t strides[2] = {(cuuint64_t)head_dim * es,
                                       (cuuint64_t)num_heads * head_dim * es};
        const cuuint32_t box[3] = {(cuuint32_t)(128u / es), 1u, 32u};
        if (!encode_tiled(&P.tmap_out, out, out_dtype, 3, dims, strides, box)) return PA_ERR_CUDA;
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
    P.pair_heads = P.G % 2 == 0 ? 1 : 0;
    P.items_x = ix;
    P.items_y = iy;
    P.num_items = (unsigned)n_items;
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    P.work = reinterpret_cast<unsigned int *>(ws);
    P.entries = reinterpret_cast<uint2 *>(ws + wl.entries);
    P.split_cnt = reinterpret_cast<unsigned int *>(ws + wl.split_cnt);
    P.part_m = reinterpret_cast<float *>(ws + wl.part_m);
    P.part_l = reinterpret_cast<float *>(ws + wl.part_l);
    P.part_o = reinterpret_cast<float *>(ws + wl.part_o);
    P.max_splits = wl.max_splits;
    P.head_dim = head_dim;
    P.num_blocks = num_blocks;
    P.scale_log2 = scale * 1.4426950408889634f;
    P.err = dev_error_word;
    // persistent: one CTA per SM, never more CTAs than entries (items and parts)
    const unsigned long long n_entries = n_items + (unsigned long long)wl.max_splits;
    const unsigned grid = (unsigned)(n_entries < (unsigned long long)sms ? n_entries : sms);
    P.grid = grid;
    cudaStream_t st = (cudaStream_t)stream;
    if (head_dim == 64)
        return dtype == PA_F16 ? launch_prefill<64, __half>(P, grid, st)
                               : launch_prefill<64, __nv_bfloat16>(P, grid, st);
    return dtype == PA_F16 ? launch_prefill<128, __half>(P, grid, st)
                           : launch_prefill<128, __nv_bfloat16>(P, grid, st);
}
