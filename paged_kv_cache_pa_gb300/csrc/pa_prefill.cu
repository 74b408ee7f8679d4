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
// How: a CTA takes two 128-row query tiles of one sequence that read the same
// keys -- two query heads of one KV group over the same tokens when the group
// size is even, else two neighbouring token tiles of one head -- so each K/V
// tile it loads feeds two tiles of work.  The grid runs the heaviest tiles
// first.  Sixteen warps; the two softmax warpgroups take 200 registers a
// thread from the other two, which keep 56:
//   * warp 8 (K producer): both Q tiles (tiled bulk copies, TMA, of a 4-D view
//     [head_dim/64][tokens][heads][64] of the query), then the sequence's
//     64-key K tiles into an RK-stage ring laid out [slice][key][64] -- one
//     TMA box per block's share of a tile and slice, or one box for all
//     slices when a block holds the whole tile;
//   * warp 9 (V producer): the V tiles into an RV-stage ring of the same
//     layout; it zeroes the V rows no query may weigh (a skipped block, keys
//     past the last one) before the tensor core reads them;
//   * warps 10, 11 (S issue of query tile 0, 1) and 12, 13 (P V issue): one
//     thread each issues, per K/V tile j, S = Q_t K_j^T (M = 128 queries,
//     N = 64 keys, K = head_dim; both operands K-major in shared memory) into
//     the tile's S buffer, or O_t += P V_j (M = 128, N = head_dim, K = 64
//     keys) with P read from a P buffer in tensor memory and V from shared
//     memory (MN-major).  A thread gets one MMA into the tensor pipe every
//     70-90 ns whatever its size, so four issuers keep the pipe fed, and a
//     wait of one holds up only its own products; warp 14 allocates tensor
//     memory, warp 15 is idle (register reallocation works by warpgroups);
//   * warps 0..3 and 4..7 (softmax of query tile 0 and 1): one query row per
//     thread.  Each loads its row of S_j from tensor memory, masks keys past
//     its position (by assignment) and keys of skipped blocks, keeps a
//     running maximum and sum in base 2, and writes P_j to a P buffer as
//     packed 16-bit pairs (in two parts of the operand type for bf16, so the
//     weights keep ~16 bits).  S is released as soon as it has been loaded,
//     so S_{j+1} is computed while the softmax works on S_j.  It rescales its row of O in tensor memory only
//     when its maximum grew by more than 2^8 since the last rescale (the sum
//     and O share that reference, so the result is exact); at the end it
//     loads O, divides by the sum and stores the row.
// A K stage is released when the S products that read it complete and a V
// stage when the P V products do, so the copies run well ahead of the
// tensor core.
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
// Tensor memory, 128 columns per query tile t at 128 t: S (64 columns of
// fp32), then P (64 columns: two buffers of 32 for fp16, one buffer of a
// high and a low 32-column part for bf16); O of tile t at 256 + t head_dim.
constexpr uint32_t kTmemCols = 512;
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
    int pair_heads;  // 1: a CTA's two tiles are heads 2y, 2y+1; 0: token tiles 2x, 2x+1
    float scale_log2;
    unsigned int *err;
};

// A K/V tile is laid out [slice][64 keys][64] (rows of 128 bytes, 128-byte
// swizzle) whatever the block size.  The TMA copies follow the blocks: a
// unit is one block's share of the tile, tbr = min(block size, 64) keys.
constexpr uint32_t kSliceBytes = (uint32_t)kKN * 128u;

template <int D>
struct PLayout {
    static constexpr int KB = D / 64;                                  // 64-element slices
    static constexpr int RK = D == 64 ? 8 : 4;                         // K ring stages
    static constexpr int RV = D == 64 ? 8 : 6;                         // V ring stages
    static constexpr size_t qt_bytes = (size_t)KB * kQM * 128;         // [slice][128][64]
    static constexpr size_t tile_bytes = (size_t)KB * kSliceBytes;     // [slice][64 keys][64]
    static constexpr size_t q_off = 0;                                 // two Q tiles
    static constexpr size_t k_off = q_off + 2 * qt_bytes;
    static constexpr size_t v_off = k_off + (size_t)RK * tile_bytes;
    static constexpr size_t bar_off = v_off + (size_t)RV * tile_bytes;
    // q_full, k_full[RK], k_empty[RK], v_full[RV], v_empty[RV], v_land,
    // s_full[2], s_free[2], p_full[2][2], pv_done[2][2], o_done[2][2] (per
    // tile; o_done per issuer)
    static constexpr int kBars = 1 + 2 * RK + 2 * RV + 1 + 2 + 2 + 4 + 4 + 4;
    static constexpr size_t tmem_off = bar_off + (size_t)kBars * 8;
    static constexpr size_t flag_off = tmem_off + 8;
    static constexpr size_t used = flag_off + 8;
    static constexpr size_t bytes = used + 1024;                       // base alignment slack
    static_assert(bytes <= 232448, "dynamic shared memory of one CTA");
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

// One query tile of a CTA.
struct PTile {
    int h;       // query head
    int q0;      // first new token of the tile
    int rows;    // rows in use (<= 128)
    int kv_end;  // keys 0 .. kv_end-1 are seen by some row of the tile
    int nt;      // 64-key tiles it reads
    bool act;
};

// The work of one CTA, the same in every thread.
struct PItem {
    int s, hk;
    int n, L, c;  // new tokens, context length after the chunk, cached before it
    int tok0;     // query row of the sequence's first new token
    int kv_end, ntiles;  // over both tiles
    bool ok, run;
    PTile t[2];
};

__device__ __forceinline__ PItem make_item(const PrefillParams &P) {
    PItem it;
    it.s = blockIdx.z;
    const int a = P.query_start_loc[it.s], b = P.query_start_loc[it.s + 1];
    it.L = P.context_lens[it.s];
    it.n = b - a;
    it.tok0 = a;
    it.ok = a >= 0 && b <= P.num_tokens && it.n >= 0 && it.n <= P.max_query_len &&
            it.L >= it.n && it.L <= P.max_context_len;
    it.c = it.L - it.n;
    const int x = (int)gridDim.x - 1 - (int)blockIdx.x;  // heaviest tiles first
    it.kv_end = 0;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        PTile &tl = it.t[t];
        tl.h = P.pair_heads ? 2 * (int)blockIdx.y + t : (int)blockIdx.y;
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
    return it;
}

struct Bars {
    uint64_t *q_full, *k_full, *k_empty, *v_full, *v_empty, *v_land;
    uint64_t *s_full, *s_free;            // [2 tiles]
    uint64_t *p_full, *pv_done;           // [2 tiles][2 P buffers]
    uint64_t *o_done;  // [2 tiles][S issuer, P V issuer]
};

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

// ---------------------------------------------------------------------------
// warps 8 and 9: TMA producers of K (and Q) and of V
// ---------------------------------------------------------------------------
template <int D, bool kIsV>
__device__ __forceinline__ void run_producer_p(const PrefillParams &P, const PItem &it,
                                               unsigned char *sq, unsigned char *skv,
                                               const Bars &B, volatile int *abort_flag,
                                               int lane) {
    using L = PLayout<D>;
    constexpr int KB = L::KB, R = kIsV ? L::RV : L::RK;
    uint64_t *full = kIsV ? B.v_full : B.k_full;
    uint64_t *empty = kIsV ? B.v_empty : B.k_empty;
    const CUtensorMap *tmap = kIsV ? &P.tmap_v : &P.tmap_k;
    const uint64_t policy = l2_evict_first_policy();
    const int32_t *row = P.block_tables + (size_t)it.s * P.max_blocks_per_seq;
    if (!kIsV && lane == 0) {
        const uint32_t nq = (it.t[0].act ? 1u : 0u) + (it.t[1].act ? 1u : 0u);
        mbar_arrive_expect_tx(B.q_full, (uint32_t)L::qt_bytes * nq);
#pragma unroll
        for (int t = 0; t < 2; ++t)
            if (it.t[t].act)
                tma_load_4d(sq + t * L::qt_bytes, &P.tmap_q, 0, it.t[t].h,
                            it.tok0 + it.t[t].q0, 0, B.q_full);
    }
    const UnitGeo g = unit_geo(P.block_shift);
    const int tpb_mask = (1 << g.lg_tpb) - 1;
    const bool whole = g.lg_tbr == 6;                     // one copy covers every slice
    const int lg_cpu = whole ? 0 : (KB == 2 ? 1 : 0);     // copies per unit
    const uint32_t unit_bytes = (uint32_t)KB * 128u << g.lg_tbr;
    // rows from this key on are cleared in the last V tile
    const int tail_row = it.kv_end & (kKN - 1);
    int cur = unit_entry(P, row, g, 0, it.kv_end, lane);
    int nxt = unit_entry(P, row, g, 1, it.kv_end, lane);
    int slot = 0;
    uint32_t phase = 0;
    int j = 0;
    bool aborted = false, land_armed = false;
    for (; j < it.ntiles; ++j) {
        if (j > 0 && (j & tpb_mask) == 0) {
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

        bool ok = true;
        if (lane == 0) ok = mbar_wait(&empty[slot], phase ^ 1u, abort_flag);
        if (!__shfl_sync(0xffffffffu, (int)ok, 0)) {
            aborted = true;
            break;
        }
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
        if (lane == 0) mbar_arrive_expect_tx(bar, tx);
        __syncwarp();
        if (issue) tma_load_3d(st + off, tmap, 0, y, sl, bar, policy);
        __syncwarp();
        if (tail) {
            // the last tile: once it has landed, clear the rows past the last key
            land_armed = true;
            bool landed = true;
            if (lane == 0) landed = mbar_wait(B.v_land, 0, abort_flag);
            if (!__shfl_sync(0xffffffffu, (int)landed, 0)) {
                aborted = true;
                break;
            }
            for (int q = lane; q < (kKN - tail_row) * KB * 8; q += 32) {
                const int rr = tail_row + q / (KB * 8), rest = q % (KB * 8);
                *reinterpret_cast<uint4 *>(st + (size_t)(rest >> 3) * kSliceBytes + rr * 128 +
                                           (rest & 7) * 16) = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&full[slot]);
        }
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
        if (!kIsV) mbar_wait(B.q_full, 0, &never);
        if (land_armed) mbar_wait(B.v_land, 0, &never);
        const int first = j > R ? j - R : 0;
        for (int k = first; k < j; ++k) mbar_wait(&full[k % R], (k / R) & 1u, &never);
    }
    __syncwarp();
}

// ---------------------------------------------------------------------------
// warps 10..13, one thread each: S (pv = 0) or P V (pv = 1) issue for query
// tile t
// ---------------------------------------------------------------------------
template <int D, bool kSplit>
__device__ __forceinline__ void run_mma_p(const PItem &it, int t, int pv, unsigned char *sq,
                                          unsigned char *sk, unsigned char *sv, uint32_t tmem,
                                          const Bars &B, uint32_t fmt,
                                          volatile int *abort_flag) {
    using L = PLayout<D>;
    constexpr int RK = L::RK, RV = L::RV;
    const uint32_t idesc_s = umma_idesc_f16(fmt, 0, 0, kQM, kKN);
    const uint32_t idesc_o = umma_idesc_f16(fmt, 0, 1, kQM, D);
    const uint32_t aq = smem_u32(sq) + (uint32_t)(t * L::qt_bytes);
    const uint32_t ak = smem_u32(sk), av = smem_u32(sv);
    constexpr int kNP = kSplit ? 1 : 2;                     // P buffers
    const uint32_t ts = tmem + (uint32_t)(t * 128);         // S, then P, of the tile
    const uint32_t to = tmem + 256u + (uint32_t)(t * D);    // O of the tile
    const int nt = t ? it.t[1].nt : it.t[0].nt;
    const int nt_other = t ? it.t[0].nt : it.t[1].nt;
    // A K/V stage is released by two arrivals, one per tile; past the other
    // tile's last K/V tile this issuer gives both.
    auto release = [&](uint64_t *bar, int j) {
        umma_commit(bar);
        if (j >= nt_other) umma_commit(bar);
    };
    // S_j into the tile's S buffer once the softmax has loaded S_{j-1}.  A K
    // step of 16 is 32 bytes inside a 64-element slice; slices are whole
    // tiles apart.
    auto issue_s = [&](int j) -> bool {
        const int ks = j % RK;
        if (!mbar_wait(&B.k_full[ks], (uint32_t)(j / RK) & 1u, abort_flag)) return false;
        if (j >= 1 && !mbar_wait(&B.s_free[t], (uint32_t)(j - 1) & 1u, abort_flag)) return false;
        tc_fence_after();
        const uint32_t kt = ak + (uint32_t)(ks * L::tile_bytes);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t in_slice = (uint32_t)((kk & 3) * 32);
            const uint64_t da =
                umma_desc_sw128(aq + (uint32_t)((kk >> 2) * kQM * 128) + in_slice, 16, 1024);
            const uint64_t db =
                umma_desc_sw128(kt + (uint32_t)(kk >> 2) * kSliceBytes + in_slice, 16, 1024);
            umma_f16(ts, da, db, idesc_s, kk > 0 ? 1u : 0u);
        }
        umma_commit(&B.s_full[t]);
        release(&B.k_empty[ks], j);
        return true;
    };
    // O += P_j V_j: P from its buffer (hi, then lo for bf16 32 columns on),
    // V MN-major (16 keys = 2048 bytes per K step, slices of head_dim a tile
    // slice apart)
    auto issue_pv = [&](int j) -> bool {
        const int vs = j % RV, pb = kNP == 2 ? (j & 1) : 0;
        if (!mbar_wait(&B.v_full[vs], (uint32_t)(j / RV) & 1u, abort_flag)) return false;
        if (!mbar_wait(&B.p_full[2 * t + pb], (uint32_t)(j / kNP) & 1u, abort_flag)) return false;
        tc_fence_after();
        const uint32_t vt = av + (uint32_t)(vs * L::tile_bytes);
        const uint32_t tp = ts + 64u + (uint32_t)(pb * 32);
#pragma unroll
        for (int kk = 0; kk < kKN / 16; ++kk) {
            const uint64_t db = umma_desc_sw128(vt + (uint32_t)(kk * 16 * 128), kSliceBytes, 1024);
            umma_f16_tmem_a(to, tp + (uint32_t)(kk * 8), db, idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
            if constexpr (kSplit)
                umma_f16_tmem_a(to, tp + 32u + (uint32_t)(kk * 8), db, idesc_o, 1u);
        }
        umma_commit(&B.pv_done[2 * t + pb]);
        release(&B.v_empty[vs], j);
        return true;
    };
    bool ok = true;
    if (!pv) {
        ok = mbar_wait(B.q_full, 0, abort_flag);
        tc_fence_after();
        for (int j = 0; ok && j < nt; ++j) ok = issue_s(j);
    } else {
        for (int j = 0; ok && j < nt; ++j) ok = issue_pv(j);
    }
    if (!ok) *abort_flag = 1;
    umma_commit(&B.o_done[2 * t + pv]);  // after every MMA issued: the teardown
}

// ---------------------------------------------------------------------------
// output of one warp's 32 rows (O / sum), staged through shared memory so that
// each store instruction writes whole rows: rounds of CR columns, the row of
// lane r in stage row r with its 16-byte chunks swizzled by r % 8 (no bank
// conflicts either way), then 32 / NCH rows per store instruction
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
__device__ __forceinline__ void store_rows(const PrefillParams &P, const PItem &it,
                                           const PTile &tl, uint32_t tm_o, float inv,
                                           unsigned char *stage, int wq, int lane) {
    constexpr int kStage = (int)(PLayout<D>::qt_bytes / 4);    // bytes of this warp
    constexpr int ES = (int)sizeof(OutT);
    constexpr int CR = kStage / (32 * ES);                      // columns a round
    constexpr int NCH = CR * ES / 16;                           // 16-byte chunks a row
    constexpr int PER = 16 / ES;                                // elements a chunk
    static_assert(D % CR == 0 && NCH >= 8 && NCH <= 32 && 32 % NCH == 0, "staging shape");
    const int row0 = tl.q0 + 32 * wq;                           // tile row of lane 0
#pragma unroll
    for (int q = 0; q < D / CR; ++q) {
#pragma unroll
        for (int c = 0; c < CR; c += 16) {
            uint32_t u[16];
            tmem_ld16(tm_o + (uint32_t)(q * CR + c), u);
            tmem_wait_ld();
            float v[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] = __uint_as_float(u[e]) * inv;
#pragma unroll
            for (int k0 = 0; k0 < 16 / PER; ++k0) {
                const int k = c / PER + k0;                     // chunk of the row
                const int pos = (k & ~7) | ((k & 7) ^ (lane & 7));
                *reinterpret_cast<uint4 *>(stage + lane * (CR * ES) + pos * 16) =
                    pack_out<OutT>(&v[k0 * PER]);
            }
        }
        __syncwarp();
#pragma unroll
        for (int it2 = 0; it2 < NCH; ++it2) {
            const int rr = it2 * (32 / NCH) + lane / NCH, k = lane % NCH;
            const int pos = (k & ~7) | ((k & 7) ^ (rr & 7));
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
// warps 0..7: softmax of query tile t = warp / 4, one row per thread, and the
// output
// ---------------------------------------------------------------------------
template <int D, typename T, bool kSplit>
__device__ __forceinline__ void run_softmax_p(const PrefillParams &P, const PItem &it, int t,
                                              unsigned char *sq, uint32_t tmem, const Bars &B,
                                              volatile int *abort_flag, int wq, int lane) {
    constexpr int kNP = kSplit ? 1 : 2;      // P buffers
    const PTile tl = t ? it.t[1] : it.t[0];
    const int r = 32 * wq + lane;            // this thread's query row
    const uint32_t lane_addr = (uint32_t)(32 * wq) << 16;
    const uint32_t tm_s = tmem + (uint32_t)(t * 128) + lane_addr;
    const uint32_t tm_o = tmem + 256u + (uint32_t)(t * D) + lane_addr;
    const int i = tl.q0 + r;                 // new-token index of the row
    const int qpos = i < it.n ? it.c + i : it.L - 1;  // padding rows see every key
    const float sc = P.scale_log2;
    // skipped blocks, from the table: bit u of a tile's mask = unit u
    const int32_t *row = P.block_tables + (size_t)it.s * P.max_blocks_per_seq;
    const UnitGeo g = unit_geo(P.block_shift);
    const int tpb_mask = (1 << g.lg_tpb) - 1;
    const unsigned unit_mask = (1u << g.upt) - 1u;
    // (the same test as the producers': a unit below kv_end with an id out of range)
    auto bad_of = [&](int e, int bt) {
        const int tok = ((bt << 5) + lane) << g.lg_tbr;
        return __ballot_sync(0xffffffffu, tok < tl.kv_end && (e < 0 || e >= P.num_blocks));
    };
    unsigned bb = bad_of(unit_entry(P, row, g, 0, tl.kv_end, lane), 0);
    int e_nxt = unit_entry(P, row, g, 1, tl.kv_end, lane);
    float m_ref = -INFINITY, lsum = 0.f;
    bool ok = true;
    for (int j = 0; j < tl.nt; ++j) {
        if (j > 0 && (j & tpb_mask) == 0) {
            const int bt = j >> g.lg_tpb;
            bb = bad_of(e_nxt, bt);
            e_nxt = unit_entry(P, row, g, bt + 1, tl.kv_end, lane);
        }
        const unsigned bits = (bb >> ((j & tpb_mask) << g.lg_upt)) & unit_mask;
        if (!__all_sync(0xffffffffu,
                        mbar_wait(&B.s_full[t], (uint32_t)j & 1u, abort_flag))) {
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
        mbar_arrive(&B.s_free[t]);  // the S buffer may take S_{j+1}
        float s[kKN];
#pragma unroll
        for (int e = 0; e < kKN; ++e) s[e] = __uint_as_float(su[e]);
        const int kb = j * kKN;
        // scale to base 2; keys past the row's position or in a skipped block
        // one warp per scheduler runs this code, so the reductions keep eight
        // independent chains
        constexpr int kAcc = 8;
        float mxa[kAcc];
#pragma unroll
        for (int q = 0; q < kAcc; ++q) mxa[q] = m_ref;
        if (!bits && kb + kKN - 1 <= qpos) {  // every key of the tile is visible
#pragma unroll
            for (int e = 0; e < kKN; ++e) {
                s[e] *= sc;
                mxa[e % kAcc] = fmaxf(mxa[e % kAcc], s[e]);
            }
        } else {
#pragma unroll
            for (int e = 0; e < kKN; ++e) {
                const bool masked = kb + e > qpos || ((bits >> (e >> g.lg_tbr)) & 1u);
                s[e] = masked ? -INFINITY : s[e] * sc;
                mxa[e % kAcc] = fmaxf(mxa[e % kAcc], s[e]);
            }
        }
#pragma unroll
        for (int q = 1; q < kAcc; ++q) mxa[0] = fmaxf(mxa[0], mxa[q]);
        const float mx = mxa[0];
        // lazy rescale: only when the maximum grew by more than 2^8; O must
        // then be stable (P V_{j-1} of this tile finished)
        const bool grow = mx > m_ref + kRescaleLog2;
        if (__any_sync(0xffffffffu, grow)) {
            const float alpha = grow && m_ref != -INFINITY ? ex2(m_ref - mx) : 1.f;
            if (j > 0) {
                const int q = kNP == 2 ? ((j - 1) & 1) : 0;
                if (!__all_sync(0xffffffffu,
                                mbar_wait(&B.pv_done[2 * t + q],
                                          (uint32_t)((j - 1) / kNP) & 1u, abort_flag))) {
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
        // the P buffer is free once P V_{j - kNP} has completed
        const int pb = kNP == 2 ? (j & 1) : 0;
        if (j >= kNP && !__all_sync(0xffffffffu,
                                    mbar_wait(&B.pv_done[2 * t + pb],
                                              (uint32_t)((j - kNP) / kNP) & 1u, abort_flag))) {
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
            const float p0 = ex2(s[2 * c] - ms), p1 = ex2(s[2 * c + 1] - ms);
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
    if (!ok) {
        *abort_flag = 1;
        if (P.err) atomicOr(P.err, PA_ERRBIT_TIMEOUT);
    }
    // epilogue: O / sum once the tile's last P V has completed
    const int last = tl.nt - 1;
    const bool done = ok && mbar_wait(&B.pv_done[2 * t + (kNP == 2 ? (last & 1) : 0)],
                                      (uint32_t)(last / kNP) & 1u, abort_flag);
    tc_fence_after();
    if (!__all_sync(0xffffffffu, done && !*abort_flag)) return;
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
    unsigned char *stage = sq + (size_t)wq * (PLayout<D>::qt_bytes / 4);
    if (P.out_dtype == PA_F32)
        store_rows<D, float>(P, it, tl, tm_o, inv, stage, wq, lane);
    else
        store_rows<D, T>(P, it, tl, tm_o, inv, stage, wq, lane);
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
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::bar_off);
    Bars B;
    B.q_full = bars;
    B.k_full = bars + 1;
    B.k_empty = B.k_full + RK;
    B.v_full = B.k_empty + RK;
    B.v_empty = B.v_full + RV;
    B.v_land = B.v_empty + RV;
    B.s_full = B.v_land + 1;
    B.s_free = B.s_full + 2;
    B.p_full = B.s_free + 2;
    B.pv_done = B.p_full + 4;
    B.o_done = B.pv_done + 4;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::tmem_off);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::flag_off);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    pdl_trigger();
    pdl_wait();  // the cache write of the chunk (earlier on the stream) is complete
    const PItem it = make_item(P);
    if (!it.ok) {  // a length or offset out of range: flag it, zero the tiles' rows
        if (threadIdx.x == 0 && P.err) atomicOr(P.err, PA_ERRBIT_CONTEXT_LEN);
        const int a = P.query_start_loc[it.s], b = P.query_start_loc[it.s + 1];
        if (a >= 0 && b <= P.num_tokens && b > a) {
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                const int r0 = a + it.t[t].q0, r1 = min(b, r0 + kQM);
                for (int r = r0; r < r1; ++r)
                    for (int d = threadIdx.x; d < D; d += kThreadsP)
                        store_elem(P.out, P.out_dtype,
                                   ((size_t)r * P.num_heads + it.t[t].h) * D + d, 0.f);
            }
        }
        return;
    }
    if (!it.run) return;

    if (threadIdx.x == 0) {
        prefetch_tmap(&P.tmap_q);
        prefetch_tmap(&P.tmap_k);
        prefetch_tmap(&P.tmap_v);
        for (int b = 0; b < L::kBars; ++b) mbar_init(&bars[b], 1);
        for (int b = 0; b < 4; ++b) mbar_init(&B.p_full[b], kTileThreads);
        for (int b = 0; b < 2; ++b) mbar_init(&B.s_free[b], kTileThreads);
        for (int b = 0; b < RK; ++b) mbar_init(&B.k_empty[b], 2);  // one arrival per tile
        for (int b = 0; b < RV; ++b) mbar_init(&B.v_empty[b], 2);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kWarpAlloc) tmem_alloc(tmem_slot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp < kSoftmaxWarps)
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax));
    else
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsOther));
    if (warp < kSoftmaxWarps) {
        const int t = warp >> 2;
        if (t ? it.t[1].act : it.t[0].act)
            run_softmax_p<D, T, kSplit>(P, it, t, sq + t * L::qt_bytes, tmem, B, abort_flag,
                                        warp & 3, lane);
    } else if (warp == kWarpK) {
        run_producer_p<D, false>(P, it, sq, sk, B, abort_flag, lane);
    } else if (warp == kWarpV) {
        run_producer_p<D, true>(P, it, sq, sv, B, abort_flag, lane);
    } else if (warp >= kWarpS && warp < kWarpPV + 2) {
        const int pv = warp >= kWarpPV ? 1 : 0, t = warp - (pv ? kWarpPV : kWarpS);
        if (lane == 0 && (t ? it.t[1].act : it.t[0].act)) {
            run_mma_p<D, kSplit>(it, t, pv, sq, sk, sv, tmem, B, kSplit ? 1u : 0u, abort_flag);
            // every MMA it issued has completed before tensor memory is released
            volatile int never = 0;
            mbar_wait(&B.o_done[2 * t + pv], 0, &never);
        }
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kWarpAlloc) tmem_dealloc(tmem, kTmemCols);
}

template <int D, typename T>
pa_status_t launch_prefill(const PrefillParams &P, dim3 grid, cudaStream_t stream) {
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
    // a CTA's two query tiles: two heads of one KV group when the group size
    // is even, else two neighbouring token tiles of one head
    const int G = num_heads / num_kv_heads;
    const bool pair_heads = G % 2 == 0;

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
    P.G = G;
    P.pair_heads = pair_heads ? 1 : 0;
    P.head_dim = head_dim;
    P.num_blocks = num_blocks;
    P.scale_log2 = scale * 1.4426950408889634f;
    P.err = dev_error_word;
    const dim3 grid(pair_heads ? (unsigned)mtiles : (unsigned)((mtiles + 1) / 2),
                    pair_heads ? (unsigned)(num_heads / 2) : (unsigned)num_heads,
                    (unsigned)num_seqs);
    cudaStream_t st = (cudaStream_t)stream;
    if (head_dim == 64)
        return dtype == PA_F16 ? launch_prefill<64, __half>(P, grid, st)
                               : launch_prefill<64, __nv_bfloat16>(P, grid, st);
    return dtype == PA_F16 ? launch_prefill<128, __half>(P, grid, st)
                           : launch_prefill<128, __nv_bfloat16>(P, grid, st);
}
