// pa_decode_api.cu -- pa_decode_attention / pa_decode_workspace_size /
// pa_decode_partition_tokens: the plan kernel, the partition merge kernel and
// the host-side checks and launches.
//
// Context split: a sequence longer than part_tokens is cut into partitions of
// part_tokens tokens, and a prefix that a run of sequences shares is a
// partition of its own; every (piece, KV head) is an independent work item
// whose partial softmax state (max m, sum l, weighted values acc) is merged
// exactly afterwards by the merge kernel:
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
#include "pa_nvtx.cuh"
#include "pa_tmap.cuh"

namespace pa {

namespace {

// Below 256 tokens a piece is too short for its split to pay: the merge
// launch costs more than the shorter longest item saves.
constexpr int kMinPartTokens = 256;
constexpr long long kTargetItems = 2048;  // ~ 152 SMs x resident CTAs x a few items each
// Shared prefixes: runs of at most 8 / G consecutive sequences (G <= 4) whose
// tables start with the same blocks, at least kMinSharedTokens of them full,
// among at most kMaxGroupSeqs sequences (the plan keeps per-sequence state in
// shared memory).
constexpr int kMinSharedTokens = 64;
constexpr int kMaxGroupSeqs = 4096;
// Below this longest context the tokens a shared prefix could save do not
// pay for the work of finding it (and, for G = 1, a second kernel).
constexpr int kMinGroupContext = 256;
// A batch of at most this many (sequence, KV head) units, whose contexts
// each fit one partition and which forms no shared-prefix items, runs
// without the plan: each unit is one item, and CTA b takes units b,
// b + grid, ...  (right for any grid; at this size one item a CTA or less
// on a GB300).  The plan kernel and its dependent launch would cost more
// than such a batch's attention.
constexpr long long kDirectMaxUnits = 256;

bool plan_free(int num_seqs, int num_kv_heads, int max_parts, int grouping) {
    return !grouping && max_parts == 1 && (long long)num_seqs * num_kv_heads <= kDirectMaxUnits;
}

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

// Sequences per shared-prefix run for these sizes (0: no shared-prefix
// items): the tensor-core kernel's 8 query rows hold G heads (rounded up to
// a power of two) of 8 / that many sequences.
int group_seqs(int num_seqs, int G, int head_dim, int max_context_len) {
    if (head_dim > 128 || G > 4 || num_seqs < 2 || num_seqs > kMaxGroupSeqs) return 0;
    if (max_context_len < kMinGroupContext) return 0;
    return group_seqs_per_box(G);
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

struct WsLayout {
    int part_tokens, max_parts, group_seqs;
    long long list_cap;  // entries per list
    size_t items0_off, items1_off, nparts_off, m_off, l_off, acc_off, bytes;
};

WsLayout ws_layout(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                   int max_context_len) {
    WsLayout w;
    w.part_tokens = choose_part_tokens(num_seqs, num_kv_heads, max_context_len);
    w.group_seqs = group_seqs(num_seqs, num_heads / num_kv_heads, head_dim, max_context_len);
    const int np = max_context_len > 0 ? (max_context_len + w.part_tokens - 1) / w.part_tokens : 1;
    // a sequence in a run has the shared prefix's pieces and its own: at most
    // one partition more than its length alone needs
    w.max_parts = np + (w.group_seqs ? 1 : 0);
    // own pieces: <= np per sequence; shared-prefix pieces: <= np per run
    w.list_cap = (long long)num_seqs * np + (w.group_seqs ? (long long)(num_seqs / 2 + 1) * np : 0);
    size_t off = align256(sizeof(WsHeader));
    w.items0_off = off;
    off = align256(off + (size_t)w.list_cap * sizeof(int4));
    w.items1_off = off;
    off = align256(off + (size_t)(w.group_seqs ? w.list_cap : 1) * sizeof(int4));
    w.nparts_off = off;
    off = align256(off + (size_t)num_seqs * sizeof(int));
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

// ---------------------------------------------------------------------------
// Plan kernel (one CTA of 1024 threads).
//
//  1. Shared prefixes (when enabled): for each sequence s >= 1, the number of
//     leading blocks that are full in both s and s - 1 and hold the same
//     block ids in both tables.  Equal ids at equal positions hold the same
//     tokens, so those tokens' attention terms differ only in the query.
//     Sequence s joins s - 1's run when they share >= kMinSharedTokens; runs
//     are cut into groups of at most group_seqs sequences, and a group's
//     shared length is the smallest of its consecutive pairs' (a multiple of
//     16 tokens).
//  2. Every sequence's context is cut into pieces: a group's shared prefix
//     [0, T) once for the group (a shared-prefix item), and each sequence's
//     own range [T, L) (T = 0 outside groups), each into part_tokens pieces
//     and a shorter last piece.  A sequence's partitions are numbered prefix
//     pieces first.
//  3. The pieces are laid out longest first (a counting sort on their size
//     in 16-token chunks): shared-prefix pieces in list 0, the others in
//     list 0 or, when the call runs the CUDA-core kernel beside the
//     tensor-core one, in list 1.
//  4. After the programmatic-dependent-launch wait: the per-sequence counts
//     of partitions, and zero output rows for empty sequences.
//
// Steps 1-3 run before the wait, so they overlap the kernel before this call
// on the stream (the cache write of a decode step): context_lens and
// block_tables are inputs, complete before the call (a kernel that wrote
// them has finished, unless it let dependents launch before writing), and
// the work lists are free -- the attention kernels of earlier calls that
// share the workspace read them in their producers, which release the claim
// counters with a fence before they allow dependents to launch.  The
// partition counts are written after the wait because the epilogue and the
// merge of an earlier call may still read them until that call completes.
// ---------------------------------------------------------------------------
// The plan's block: one thread per sequence up to 1024 (at least 128), so a
// small batch's barriers involve few warps; with shared prefixes each
// thread keeps up to kSeqPerThread sequences' state (num_seqs <= 4096).
constexpr int kPlanThreads = 1024;
constexpr int kSeqPerThread = kMaxGroupSeqs / kPlanThreads;
int plan_threads(int num_seqs) {
    const int t = (num_seqs + 31) / 32 * 32;
    return t < 128 ? 128 : (t > kPlanThreads ? kPlanThreads : t);
}

struct PlanParams {
    const int32_t *lens;
    const int32_t *tables;
    int max_blocks_per_seq, block_shift;
    int num_seqs, max_context_len, part_tokens;
    int num_kv_heads, num_heads, head_dim;
    int group_seqs;  // 0: no shared-prefix items
    int split;       // 1: plain pieces go to list 1
    int4 *items0, *items1;
    int *nparts;
    WsHeader *hdr;
    void *out;
    int out_dtype;
    unsigned int *err;
};

// Shared memory of the plan: the fixed part, then (shared prefixes only) the
// per-sequence arrays, sized by the host for the call's num_seqs.
struct PlanShared {
    int hist[2][kMaxPartTokens / kBlock + 1];
    int offs[2][kMaxPartTokens / kBlock + 1];
    int red[32];
    int *shared_tok;   // [num_seqs] tokens s shares with s - 1 (0: none)
    short *run_start;  // [num_seqs] first sequence of s's run
};
constexpr size_t plan_smem_bytes(int num_seqs, bool grouping) {
    return sizeof(PlanShared) + (grouping ? (size_t)num_seqs * (4 + 2) + 16 : 0);
}

__device__ __forceinline__ int valid_len(const PlanParams &A, int s) {
    const int L = A.lens[s];
    return (L < 0 || L > A.max_context_len) ? 0 : L;
}

// Group of sequence s: (first sequence, sequences, shared tokens); n = 1 and
// T = 0 outside a group.
struct Group {
    int first, n, T;
};
__device__ __forceinline__ Group group_of(const PlanParams &A, const PlanShared &sh, int s,
                                          bool grouped) {
    Group g = {s, 1, 0};
    if (!grouped) return g;
    const int rs = sh.run_start[s];
    const int first = rs + (s - rs) / A.group_seqs * A.group_seqs;
    int n = 1, T = INT_MAX;
    while (n < A.group_seqs && first + n < A.num_seqs && sh.shared_tok[first + n] > 0) {
        T = min(T, sh.shared_tok[first + n]);
        ++n;
    }
    if (n >= 2) {
        g.first = first;
        g.n = n;
        g.T = T;
    }
    return g;
}

// Pieces of a range of len tokens: full part_tokens pieces and a shorter last one.
__device__ __forceinline__ int pieces_of(int len, int PT) { return (len + PT - 1) / PT; }

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const __grid_constant__ PlanParams A) {
    pdl_trigger();  // the attention CTAs may start their set-up now
    extern __shared__ __align__(16) unsigned char plan_smem[];
    PlanShared &sh = *reinterpret_cast<PlanShared *>(plan_smem);
    if (threadIdx.x == 0) {
        int *p = reinterpret_cast<int *>(plan_smem + sizeof(PlanShared));
        sh.shared_tok = p;
        sh.run_start = reinterpret_cast<short *>(p + A.num_seqs);
    }
    constexpr int kKeys = kMaxPartTokens / kBlock + 1;
    const int PT = A.part_tokens, PB = PT / kBlock;
    const int tid = threadIdx.x, lane = tid & 31;
    const int S = A.num_seqs;
    if (tid < 2 * kKeys) (&sh.hist[0][0])[tid] = 0;
    __syncthreads();

    // ---- 1. shared prefixes ------------------------------------------------
    bool grouped = false;  // the same in every thread: some run may form
    if (A.group_seqs) {
        const int min_blocks = kMinSharedTokens >> A.block_shift;
        // lengths and first block ids of s and s - 1, in one round of loads
        int len1[kSeqPerThread], len0[kSeqPerThread], id1[kSeqPerThread], id0[kSeqPerThread];
#pragma unroll
        for (int i = 0; i < kSeqPerThread; ++i) {
            const int s = tid * kSeqPerThread + i;
            len1[i] = len0[i] = 0;
            id1[i] = id0[i] = 0;
            if (s >= 1 && s < S) {
                const int32_t *r1 = A.tables + (size_t)s * A.max_blocks_per_seq;
                len1[i] = A.lens[s];
                len0[i] = A.lens[s - 1];
                id1[i] = __ldg(r1);
                id0[i] = __ldg(r1 - A.max_blocks_per_seq);
            }
        }
        // 0 where the first ids differ
        bool any = false;
#pragma unroll
        for (int i = 0; i < kSeqPerThread; ++i) {
            const bool ok1 = len1[i] >= 0 && len1[i] <= A.max_context_len;
            const bool ok0 = len0[i] >= 0 && len0[i] <= A.max_context_len;
            int j = (ok1 && ok0) ? min(len1[i], len0[i]) >> A.block_shift : 0;
            if (j < max(min_blocks, 1) || id1[i] != id0[i]) j = 0;
            if (j > A.max_blocks_per_seq) j = A.max_blocks_per_seq;
            const int s = tid * kSeqPerThread + i;
            if (s < S) sh.shared_tok[s] = j;  // blocks worth comparing, until compared
            any |= j > 0;
        }
        // nothing to compare anywhere (the usual batch): no runs, done
        grouped = __syncthreads_or(any) != 0;
    }
    if (grouped) {
        // Each thread compares the rows of sequences tid, tid + blockDim.x, ...
        // with the rows before them (every thread has a sequence before any
        // has a second), 16 blocks a round with every load of the round in
        // flight together (16-byte loads when the rows are 16-byte aligned),
        // and keeps the leading equal blocks as tokens: whole 16-token
        // chunks, none below the minimum.
        constexpr int kRound = 16;
        const bool vec = (reinterpret_cast<uintptr_t>(A.tables) & 15u) == 0 &&
                         (A.max_blocks_per_seq & 3) == 0;
        for (int s = tid; s < S; s += (int)blockDim.x) {
            const int c = sh.shared_tok[s];
            int first = c;  // blocks 0 .. first-1 are equal
            const int32_t *r1 = A.tables + (size_t)s * A.max_blocks_per_seq;
            const int32_t *r0 = r1 - A.max_blocks_per_seq;
            for (int j0 = 0; j0 < c && first == c; j0 += kRound) {
                int a[kRound], b[kRound];
                if (vec) {
#pragma unroll
                    for (int u = 0; u < kRound / 4; ++u) {
                        const bool in = j0 + 4 * u < c;  // a whole int4 inside the row
                        const int4 x = in ? __ldg(reinterpret_cast<const int4 *>(r1 + j0) + u)
                                          : make_int4(0, 0, 0, 0);
                        const int4 y = in ? __ldg(reinterpret_cast<const int4 *>(r0 + j0) + u)
                                          : make_int4(0, 0, 0, 0);
                        a[4 * u] = x.x; a[4 * u + 1] = x.y; a[4 * u + 2] = x.z; a[4 * u + 3] = x.w;
                        b[4 * u] = y.x; b[4 * u + 1] = y.y; b[4 * u + 2] = y.z; b[4 * u + 3] = y.w;
                    }
                } else {
#pragma unroll
                    for (int u = 0; u < kRound; ++u) {
                        const bool in = j0 + u < c;
                        a[u] = in ? __ldg(r1 + j0 + u) : 0;
                        b[u] = in ? __ldg(r0 + j0 + u) : 0;
                    }
                }
#pragma unroll
                for (int u = kRound - 1; u >= 0; --u)
                    if (j0 + u < c && a[u] != b[u]) first = j0 + u;
            }
            const int t = (first << A.block_shift) & ~(kBlock - 1);
            sh.shared_tok[s] = t >= kMinSharedTokens ? t : 0;
        }
        __syncthreads();
        // run starts: the last s' <= s that does not share with s' - 1 (an
        // inclusive max-scan)
        int last = -1;
#pragma unroll
        for (int i = 0; i < kSeqPerThread; ++i) {
            const int s = tid * kSeqPerThread + i;
            if (s < S && sh.shared_tok[s] == 0) last = s;
        }
        int incl = last;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl = max(incl, u);
        }
        if (lane == 31) sh.red[tid >> 5] = incl;
        __syncthreads();
        int carry = -1;
        for (int w = 0; w < (tid >> 5); ++w) carry = max(carry, sh.red[w]);
        int prev = __shfl_up_sync(0xffffffffu, incl, 1);
        if (lane == 0) prev = -1;
        int rs = max(carry, prev);
#pragma unroll
        for (int i = 0; i < kSeqPerThread; ++i) {
            const int s = tid * kSeqPerThread + i;
            if (s < S) {
                if (sh.shared_tok[s] == 0) rs = s;
                sh.run_start[s] = (short)rs;
            }
        }
        __syncthreads();
    }

    // ---- 2, 3. pieces, counted then placed longest first ------------------
    // One pass counts (place = false), the other writes (place = true).
    // Thread-strided over sequences, 1024 at a time; each thread handles its
    // sequence's own range and, for a group's first sequence, the prefix.
    // A range of len tokens is len / PT full pieces and one of len % PT.
    const int own_list = A.split ? 1 : 0;
    const int L_first = tid < S ? valid_len(A, tid) : 0;  // this thread's first sequence
    for (int pass = 0; pass < 2; ++pass) {
        const bool place = pass == 1;
        for (int s0 = 0; s0 < S; s0 += (int)blockDim.x) {
            const int s = s0 + tid;
            const int L = s0 == 0 ? L_first : (s < S ? valid_len(A, s) : 0);
            Group g = {s, 1, 0};
            if (grouped && L > 0) g = group_of(A, sh, s, grouped);
            // segment 0: the group's shared prefix (its first sequence only);
            // segment 1: the sequence's own range
            for (int seg = grouped ? 0 : 1; seg < 2; ++seg) {
                int len, t0, pbase, list, cnt;
                bool grp;
                if (seg == 0) {
                    grp = true;
                    len = (L > 0 && g.n >= 2 && g.first == s) ? g.T : 0;
                    t0 = 0;
                    pbase = 0;
                    list = 0;
                    cnt = g.n;
                } else {
                    grp = false;
                    len = L > 0 ? L - g.T : 0;
                    t0 = g.T;
                    pbase = pieces_of(g.T, PT);
                    list = own_list;
                    cnt = pbase + pieces_of(len, PT);
                }
                const int nf = len / PT, rem = len - nf * PT;
                const int key = (rem + kBlock - 1) / kBlock;  // 0: no short piece
                if (!place) {
                    // full pieces: one add per warp; the short piece: one add
                    int full = nf;
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1)
                        full += __shfl_xor_sync(0xffffffffu, full, off);
                    if (lane == 0 && full) atomicAdd(&sh.hist[list][PB], full);
                    if (key) atomicAdd(&sh.hist[list][key], 1);
                } else {
                    // full pieces of the warp: a contiguous range from one add
                    int incl = nf;
#pragma unroll
                    for (int off = 1; off < 32; off <<= 1) {
                        const int u = __shfl_up_sync(0xffffffffu, incl, off);
                        if (lane >= off) incl += u;
                    }
                    int base = 0;
                    if (lane == 31 && incl) base = atomicAdd(&sh.offs[list][PB], incl);
                    base = __shfl_sync(0xffffffffu, base, 31) + incl - nf;
                    int4 *items = list ? A.items1 : A.items0;
                    const int first = grp ? g.first : s;
                    for (int k = 0; k < nf; ++k)
                        items[base + k] = make_int4(first, t0 + k * PT, PT,
                                                    make_item_w(pbase + k, cnt, grp));
                    if (key) {
                        const int slot = atomicAdd(&sh.offs[list][key], 1);
                        items[slot] = make_int4(first, t0 + nf * PT, rem,
                                                make_item_w(pbase + nf, cnt, grp));
                    }
                }
            }
        }
        if (place) break;  // the placing pass is the last: nothing to order after it
        __syncthreads();
        if (tid < (A.split ? 64 : 32)) {  // exclusive scans over sizes, largest first
            const int list = tid >> 5;
            const int key = PB - lane;
            const int v = (lane < PB) ? sh.hist[list][key] : 0;
            int incl = v;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += u;
            }
            if (lane < PB) sh.offs[list][key] = incl - v;
            if (lane == 31) {
                A.hdr->counter[list] = 0u;
                A.hdr->n_items[list] = (unsigned)incl * (unsigned)A.num_kv_heads;
            }
        }
        if (tid == 32 && !A.split) {
            A.hdr->counter[1] = 0u;
            A.hdr->n_items[1] = 0u;
        }
        __syncthreads();
    }

    pdl_wait();  // earlier work on the stream may still read nparts and out
    for (int s0 = 0; s0 < S; s0 += (int)blockDim.x) {
        const int s = s0 + tid;
        const int L0 = s >= S ? 1 : (s0 == 0 ? (L_first > 0 ? L_first : A.lens[s]) : A.lens[s]);
        const bool bad = L0 < 0 || L0 > A.max_context_len;
        if (s < S) {
            if (bad && A.err) atomicOr(A.err, PA_ERRBIT_CONTEXT_LEN);
            const int L = bad ? 0 : L0;
            int np = 0;
            if (L > 0) {
                const Group g = group_of(A, sh, s, grouped);
                np = pieces_of(g.T, A.part_tokens) + pieces_of(L - g.T, A.part_tokens);
            }
            A.nparts[s] = np;
        }
        // the warp zeroes the output rows of its empty sequences together
        unsigned empty = __ballot_sync(0xffffffffu, s < S && (L0 <= 0 || bad));
        while (empty) {
            const int src = __ffs(empty) - 1;
            empty &= empty - 1;
            const size_t base = (size_t)(s0 + (tid & ~31) + src) * A.num_heads * A.head_dim;
            for (int i = lane; i < A.num_heads * A.head_dim; i += 32)
                store_out(A.out, A.out_dtype, base + i, 0.f);
        }
    }
}

// One CTA per (sequence, HPC query heads) of a multi-partition sequence:
//   M = max_p m_p,  c_p = 2^(m_p - M),  L = sum_p l_p c_p,
//   o = sum_p acc_p c_p / L.
// One pass over the partials: the TPH = 128 / HPC threads of a head cover its
// head_dim / 4 float4 columns (CPT columns a thread) and, when there are more
// threads than columns, form NG partition groups; group g folds partitions
// g, g + NG, ... into a running (M, L, o), rescaling it whenever the maximum
// grows, so a partition's m, l and acc are loaded together instead of in
// three dependent rounds.  The groups' states are then folded the same way
// through shared memory.  Several heads a CTA (HPC > 1) keep the grid small
// when most sequences need no merge: those CTAs only read a length and leave,
// and it is their launches, not the merges, that would cost the time.
constexpr int kMergeThreads = 128;
constexpr int kMergeBatch = 4;  // partitions a thread loads before folding them
constexpr int kMergeMaxCtas = 3072;  // heads per CTA grow until the grid is no larger

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

template <int D, int HPC>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const __grid_constant__ DecodeParams P) {
    constexpr int C = D / 4;                       // float4 columns of a head
    constexpr int TPH = kMergeThreads / HPC;       // threads of a head
    constexpr int CPT = C > TPH ? C / TPH : 1;     // columns a thread
    constexpr int NG = TPH > C ? TPH / C : 1;      // partition groups of a head
    static_assert(CPT * TPH == C * NG && (NG == 1 || CPT == 1), "merge shape");
    __shared__ float s_m[HPC][NG], s_l[HPC][NG];
    __shared__ float4 s_acc[HPC][NG][C];
    const int s = blockIdx.x, tid = threadIdx.x;
    const int hl = tid / TPH, th = tid % TPH;        // head within the CTA, thread within the head
    const int h = blockIdx.y * HPC + hl;
    const int grp = th / (C / CPT), c0 = (th % (C / CPT)) * CPT;  // partition group, first column
    const int L = P.context_lens[s];  // an input: complete before this grid launched
    if (L <= 0 || L > P.max_context_len) return;  // empty or invalid: a zero row
    // One partition for sure: no split, and no shared prefix.  A sequence can
    // share a prefix only with a neighbour whose first block id equals its
    // own (tables are inputs too, complete before this grid launched).
    if (L <= P.part_tokens) {
        if (!P.grouping || L <= kMinSharedTokens) return;
        const int32_t *row = P.block_tables + (size_t)s * P.max_blocks_per_seq;
        const int b0 = __ldg(row);
        const bool prev = s > 0 && __ldg(row - P.max_blocks_per_seq) == b0;
        const bool next = s + 1 < P.num_seqs && __ldg(row + P.max_blocks_per_seq) == b0;
        if (!prev && !next) return;
    }
    pdl_wait();  // partials from the attention kernels; the plan's counts
    const int np = P.grouping ? P.nparts[s] : (L + P.part_tokens - 1) / P.part_tokens;
    if constexpr (kDebugChecks) {
        if (np > P.max_parts) {
            if (tid == 0 && blockIdx.y == 0 && P.err) atomicOr(P.err, PA_ERRBIT_INTERNAL);
            return;
        }
    }
    if (np <= 1) return;
    const bool live = h < P.num_heads;  // the last CTA of a row may hold fewer heads
    const size_t base = ((size_t)s * P.num_heads + (live ? h : 0)) * P.max_parts;
    const float4 *acc = reinterpret_cast<const float4 *>(P.part_acc + base * D) + c0;

    float M = -INFINITY, Lsum = 0.f;
    float4 o[CPT];
#pragma unroll
    for (int c = 0; c < CPT; ++c) o[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    float Mc[CPT], Lc[CPT];
#pragma unroll
    for (int c = 0; c < CPT; ++c) {
        Mc[c] = -INFINITY;
        Lc[c] = 0.f;
    }
    for (int p0 = grp; live && p0 < np; p0 += kMergeBatch * NG) {
        float mp[kMergeBatch], lp[kMergeBatch];
        float4 a[kMergeBatch][CPT];
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u) {
            const int p = p0 + u * NG;
            const bool in = p < np;
            mp[u] = in ? P.part_m[base + p] : -INFINITY;
            lp[u] = in ? P.part_l[base + p] : 0.f;
#pragma unroll
            for (int c = 0; c < CPT; ++c)
                a[u][c] = in ? acc[(size_t)p * C + c] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u)
#pragma unroll
            for (int c = 0; c < CPT; ++c) fold_state(Mc[c], Lc[c], o[c], mp[u], lp[u], a[u][c]);
    }
    M = Mc[0];
    Lsum = Lc[0];  // every column folds the same (m, l): the same M and L
    if constexpr (NG > 1) {  // (then CPT == 1)
        if (c0 == 0) {
            s_m[hl][grp] = M;
            s_l[hl][grp] = Lsum;
        }
        s_acc[hl][grp][c0] = o[0];
        __syncthreads();
        if (grp != 0) return;
#pragma unroll
        for (int g = 1; g < NG; ++g) fold_state(M, Lsum, o[0], s_m[hl][g], s_l[hl][g], s_acc[hl][g][c0]);
    }
    if (!live) return;
#pragma unroll
    for (int c = 0; c < CPT; ++c) {
        const size_t ob = ((size_t)s * P.num_heads + h) * D + (size_t)(c0 + c) * 4;
        store_out(P.out, P.out_dtype, ob + 0, Lsum > 0.f ? o[c].x / Lsum : 0.f);
        store_out(P.out, P.out_dtype, ob + 1, Lsum > 0.f ? o[c].y / Lsum : 0.f);
        store_out(P.out, P.out_dtype, ob + 2, Lsum > 0.f ? o[c].z / Lsum : 0.f);
        store_out(P.out, P.out_dtype, ob + 3, Lsum > 0.f ? o[c].w / Lsum : 0.f);
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

// 4-D view [head_dim / 64][heads][sequences][64] of the query
// [sequences][heads][head_dim]; one box is group_box_heads(G) heads of
// group_seqs_per_box(G) consecutive sequences (8 rows), all halves: the
// query rows of a shared-prefix item.
bool encode_group_query(CUtensorMap *map, const void *q, pa_dtype_t dtype, int num_seqs,
                        int num_heads, int head_dim, int G) {
    const cuuint64_t dims[4] = {64u, (cuuint64_t)num_seqs, (cuuint64_t)num_heads,
                                (cuuint64_t)(head_dim / 64)};
    const cuuint64_t strides[3] = {(cuuint64_t)num_heads * head_dim * 2,
                                   (cuuint64_t)head_dim * 2, 128u};
    const cuuint32_t box[4] = {64u, (cuuint32_t)group_seqs_per_box(G),
                               (cuuint32_t)group_box_heads(G), (cuuint32_t)(head_dim / 64)};
    return encode_tiled(map, q, dtype, 4, dims, strides, box);
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

extern "C" int pa_decode_kernel_launches(int num_seqs, int num_heads, int num_kv_heads,
                                         int head_dim, int max_context_len) {
    if (num_seqs <= 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        max_context_len < 0 || num_heads % num_kv_heads != 0)
        return 0;
    const WsLayout w = ws_layout(num_seqs, num_heads, num_kv_heads, head_dim, max_context_len);
    const bool tc = uses_tensor_cores(num_heads / num_kv_heads, head_dim);
    const bool merge = w.max_parts > 1 && (max_context_len > w.part_tokens || w.group_seqs);
    if (plan_free(num_seqs, num_kv_heads, w.max_parts, w.group_seqs)) return 1;
    return 1 + ((w.group_seqs && !tc) ? 2 : 1) + (merge ? 1 : 0);
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

    if (w.max_parts > kMaxParts) return PA_ERR_UNSUPPORTED;
    const int G = num_heads / num_kv_heads;
    // shared-prefix items need block tables; with G = 1 they run on the
    // tensor-core kernel and the plain items on the CUDA-core kernel
    const int grouping = contig_rows == 0 ? w.group_seqs : 0;
    const bool tc = uses_tensor_cores(G, head_dim);
    const bool split = grouping && !tc;
    const bool merge = w.max_parts > 1 && (max_context_len > w.part_tokens || grouping);

    unsigned char *ws = static_cast<unsigned char *>(workspace);
    DecodeParams P;
    memset(&P, 0, sizeof(P));
    if (tc || grouping) {
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
        if (grouping &&
            !encode_group_query(&P.tmap_qs, query, dtype, num_seqs, num_heads, head_dim, G))
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
    P.G = G;
    P.head_dim = head_dim;
    P.num_blocks = num_blocks;
    P.scale_log2 = scale * 1.4426950408889634f;
    P.part_tokens = w.part_tokens;
    P.max_parts = w.max_parts;
    P.grouping = grouping ? 1 : 0;
    P.hdr = reinterpret_cast<WsHeader *>(ws);
    P.nparts = reinterpret_cast<int *>(ws + w.nparts_off);
    P.part_m = reinterpret_cast<float *>(ws + w.m_off);
    P.part_l = reinterpret_cast<float *>(ws + w.l_off);
    P.part_acc = reinterpret_cast<float *>(ws + w.acc_off);
    P.err = dev_error_word;
    cudaStream_t st = (cudaStream_t)stream;

    PlanParams A;
    memset(&A, 0, sizeof(A));
    A.lens = context_lens;
    A.tables = block_tables;
    A.max_blocks_per_seq = max_blocks_per_seq;
    A.block_shift = block_shift;
    A.num_seqs = num_seqs;
    A.max_context_len = max_context_len;
    A.part_tokens = w.part_tokens;
    A.num_kv_heads = num_kv_heads;
    A.num_heads = num_heads;
    A.head_dim = head_dim;
    A.group_seqs = grouping;
    A.split = split ? 1 : 0;
    A.items0 = reinterpret_cast<int4 *>(ws + w.items0_off);
    A.items1 = reinterpret_cast<int4 *>(ws + w.items1_off);
    A.nparts = P.nparts;
    A.hdr = P.hdr;
    A.out = out;
    A.out_dtype = (int)out_dtype;
    A.err = dev_error_word;
    const bool direct = plan_free(num_seqs, num_kv_heads, w.max_parts, grouping);
    P.direct = direct ? 1 : 0;
    if (!direct) {
        const size_t plan_smem = plan_smem_bytes(num_seqs, grouping != 0);
        if (plan_smem > 48 * 1024) return PA_ERR_UNSUPPORTED;  // never: grouping caps num_seqs
        if (launch_pdl(plan_kernel, dim3(1), dim3(plan_threads(num_seqs)), plan_smem, st, A) !=
            cudaSuccess)
            return PA_ERR_CUDA;
    }

    long long cap = direct ? (long long)num_seqs * num_kv_heads : w.list_cap * num_kv_heads;
    if (cap > INT_MAX) cap = INT_MAX;
    auto launch = [&](int kernel) -> pa_status_t {
        if (head_dim == 64) return launch_decode_d64(P, dtype, (int)cap, st, kernel);
        if (head_dim == 128) return launch_decode_d128(P, dtype, (int)cap, st, kernel);
        return launch_decode_d256(P, dtype, (int)cap, st, kernel);
    };
    pa_status_t st_launch;
    if (split) {
        // list 0: the shared-prefix items on the tensor-core kernel, which
        // lets the next kernel launch once the plan has completed; then list
        // 1: the plain items on the CUDA-core kernel, whose CTAs start work
        // as soon as they fit and wait for the tensor-core grid only at the
        // end
        P.list = 0;
        P.items = A.items0;
        P.early_trigger = 1;
        st_launch = launch(kKernelTensorCore);
        if (st_launch != PA_OK) return st_launch;
        P.early_trigger = 0;
        P.after_sibling = 1;
        P.list = 1;
        P.items = A.items1;
        st_launch = launch(kKernelByGroup);
    } else {
        P.list = 0;
        P.items = A.items0;
        st_launch = launch(kKernelByGroup);
    }
    if (st_launch != PA_OK) return st_launch;

    if (merge) {
        if (num_heads > 65535) return PA_ERR_UNSUPPORTED;
        // heads a CTA: 1, 2, 4 or 8, the fewest that keep the grid within
        // kMergeMaxCtas CTAs
        int hpc = 1;
        while (hpc < 8 && (long long)num_seqs * ((num_heads + hpc - 1) / hpc) > kMergeMaxCtas)
            hpc *= 2;
        const dim3 grid((unsigned)num_seqs, (unsigned)((num_heads + hpc - 1) / hpc));
        cudaError_t e = cudaErrorInvalidValue;
        auto go = [&](auto kern) { e = launch_pdl(kern, grid, dim3(kMergeThreads), 0, st, P); };
        if (head_dim == 64) {
            if (hpc == 1) go(merge_kernel<64, 1>); else if (hpc == 2) go(merge_kernel<64, 2>);
            else if (hpc == 4) go(merge_kernel<64, 4>); else go(merge_kernel<64, 8>);
        } else if (head_dim == 128) {
            if (hpc == 1) go(merge_kernel<128, 1>); else if (hpc == 2) go(merge_kernel<128, 2>);
            else if (hpc == 4) go(merge_kernel<128, 4>); else go(merge_kernel<128, 8>);
        } else {
            if (hpc == 1) go(merge_kernel<256, 1>); else if (hpc == 2) go(merge_kernel<256, 2>);
            else if (hpc == 4) go(merge_kernel<256, 4>); else go(merge_kernel<256, 8>);
        }
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
    PA_NVTX_RANGE("pa_decode_attention_ex");
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
    PA_NVTX_RANGE("pa_decode_attention");
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
    PA_NVTX_RANGE("pa_decode_attention_contiguous");
    if (max_rows <= 0) return PA_ERR_INVALID_ARG;
    return decode_impl(out, out_dtype, query, k_cache, v_cache, nullptr, 0, max_rows,
                       context_lens, max_context_len, num_seqs, num_heads, num_kv_heads,
                       head_dim, 0, PA_BLOCK_SIZE, scale, dtype, workspace, workspace_bytes,
                       dev_error_word, stream);
}
