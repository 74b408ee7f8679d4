// pa_block_manager.cpp -- host-side KV block manager behind include/pa_bm.h.
//
// Two pools of block ids (the GPU pool and the CPU swap space), each with a
// reference count per block and a free list that hands out a caller-given
// order first and then the lowest free id; sequences with a block table and
// a stored-token count.  Every entry point checks everything it needs before
// it changes anything, so a failed call leaves the manager as it was.
// [Efficient Memory Management for Large Language Model Serving with
// PagedAttention, "KV Cache Manager: Block Table Mapping", "The three
// primitive operations", "Copy-on-write mechanism", "Scheduling and
// Preemption"; vLLM Internals ..., "PagedAttention: page tables, for KV";
// Paged Attention: Managing the KV Cache Like Virtual Memory, "A paged KV
// cache, in code"]
#include "pa_bm.h"

#include <algorithm>
#include <cstdint>
#include <deque>
#include <functional>
#include <mutex>
#include <new>
#include <queue>
#include <unordered_map>
#include <utility>
#include <vector>

namespace {

// Block ids 0..n-1 with reference counts.
class Pool {
   public:
    explicit Pool(int n) : refs_(n, 0) {
        for (int b = 0; b < n; ++b) heap_.push(b);
    }
    int size() const { return (int)refs_.size(); }
    int num_free() const { return (int)(given_.size() + heap_.size()); }
    bool valid(int b) const { return b >= 0 && b < size(); }
    int refs(int b) const { return refs_[b]; }
    bool unused() const {
        return std::all_of(refs_.begin(), refs_.end(), [](int r) { return r == 0; });
    }
    // Hand out `order` first (ids must be distinct, valid and free).
    bool set_order(const int32_t *order, int n) {
        std::vector<char> seen(refs_.size(), 0);
        for (int i = 0; i < n; ++i) {
            if (!valid(order[i]) || seen[order[i]] || refs_[order[i]]) return false;
            seen[order[i]] = 1;
        }
        given_.assign(order, order + n);
        std::priority_queue<int, std::vector<int>, std::greater<int>> rest;
        for (int b = 0; b < size(); ++b)
            if (!seen[b] && !refs_[b]) rest.push(b);
        heap_.swap(rest);
        return true;
    }
    // Callers check num_free() first.
    int alloc() {
        int b;
        if (!given_.empty()) {
            b = given_.front();
            given_.pop_front();
        } else {
            b = heap_.top();
            heap_.pop();
        }
        refs_[b] = 1;
        return b;
    }
    void retain(int b) { ++refs_[b]; }
    void set_refs(int b, int r) { refs_[b] = r; }
    void release(int b) {
        if (--refs_[b] == 0) heap_.push(b);
    }

   private:
    std::vector<int> refs_;
    std::deque<int> given_;
    std::priority_queue<int, std::vector<int>, std::greater<int>> heap_;
};

struct Seq {
    std::vector<int> table;  // block ids, in the pool named by on_cpu
    int n = 0;               // stored tokens
    bool on_cpu = false;
};

}  // namespace

struct pa_block_manager {
    pa_block_manager(int g, int c, int b) : gpu(g), cpu(c), block_size(b) {}
    Pool gpu, cpu;
    int block_size;
    std::unordered_map<int64_t, Seq> seqs;
    int64_t next_id = 0;
    std::deque<std::pair<int64_t, int64_t>> copies;
    mutable std::mutex mu;

    Seq *find(int64_t id) {
        auto it = seqs.find(id);
        return it == seqs.end() ? nullptr : &it->second;
    }
    const Seq *find(int64_t id) const {
        auto it = seqs.find(id);
        return it == seqs.end() ? nullptr : &it->second;
    }
    // Blocks an append of `num` tokens allocates: a copy of a shared,
    // partially filled last block, plus the blocks the tokens spill into.
    int needed(const Seq &s, int num) const {
        const long long want = ((long long)s.n + num + block_size - 1) / block_size;
        const int cow = (s.n % block_size) && gpu.refs(s.table.back()) > 1 ? 1 : 0;
        return cow + (int)std::max(0LL, want - (long long)s.table.size());
    }
    pa_status_t swap(const int64_t *ids, int n, int64_t *pairs_out, int cap, int *num_pairs,
                     bool out);
};

pa_status_t pa_block_manager::swap(const int64_t *ids, int n, int64_t *pairs_out, int cap,
                                   int *num_pairs, bool out) {
    if (n < 0 || (n > 0 && !ids) || cap < 0 || (cap > 0 && !pairs_out) || !num_pairs)
        return PA_ERR_INVALID_ARG;
    Pool &from = out ? gpu : cpu;
    Pool &to = out ? cpu : gpu;
    std::vector<Seq *> group;
    for (int i = 0; i < n; ++i) {
        Seq *s = find(ids[i]);
        if (!s || s->on_cpu != !out) return PA_ERR_INVALID_ARG;
        if (std::find(group.begin(), group.end(), s) != group.end()) return PA_ERR_INVALID_ARG;
        group.push_back(s);
    }
    // distinct blocks in order of first use, and the group's references to each
    std::vector<int> blocks;
    std::unordered_map<int, int> uses;
    for (Seq *s : group)
        for (int b : s->table)
            if (uses[b]++ == 0) blocks.push_back(b);
    for (int b : blocks)
        if (from.refs(b) != uses[b]) return PA_ERR_INVALID_ARG;  // shared outside the group
    if ((int)blocks.size() > cap) return PA_ERR_INVALID_ARG;
    if ((int)blocks.size() > to.num_free()) return PA_ERR_NO_BLOCKS;
    std::unordered_map<int, int> moved;
    for (size_t i = 0; i < blocks.size(); ++i) {
        const int b = blocks[i];
        const int nb = to.alloc();
        to.set_refs(nb, from.refs(b));
        from.set_refs(b, 1);
        from.release(b);
        moved[b] = nb;
        pairs_out[2 * i] = b;
        pairs_out[2 * i + 1] = nb;
    }
    for (Seq *s : group) {
        for (int &b : s->table) b = moved[b];
        s->on_cpu = out;
    }
    *num_pairs = (int)blocks.size();
    return PA_OK;
}

extern "C" {

pa_status_t pa_bm_create(int num_gpu_blocks, int num_cpu_blocks, int block_size,
                         pa_block_manager_t **out) {
    if (!out || num_gpu_blocks <= 0 || num_cpu_blocks < 0 || block_size <= 0)
        return PA_ERR_INVALID_ARG;
    *out = new (std::nothrow) pa_block_manager(num_gpu_blocks, num_cpu_blocks, block_size);
    return *out ? PA_OK : PA_ERR_INVALID_ARG;
}

void pa_bm_destroy(pa_block_manager_t *bm) { delete bm; }

pa_status_t pa_bm_set_free_order(pa_block_manager_t *bm, const int32_t *order, int n) {
    if (!bm || n < 0 || (n > 0 && !order)) return PA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> g(bm->mu);
    if (!bm->gpu.unused()) return PA_ERR_INVALID_ARG;
    return bm->gpu.set_order(order, n) ? PA_OK : PA_ERR_INVALID_ARG;
}

int pa_bm_num_free_gpu(const pa_block_manager_t *bm) {
    if (!bm) return -1;
    std::lock_guard<std::mutex> g(bm->mu);
    return bm->gpu.num_free();
}

int pa_bm_num_free_cpu(const pa_block_manager_t *bm) {
    if (!bm) return -1;
    std::lock_guard<std::mutex> g(bm->mu);
    return bm->cpu.num_free();
}

int pa_bm_block_size(const pa_block_manager_t *bm) { return bm ? bm->block_size : -1; }

int pa_bm_refcount(const pa_block_manager_t *bm, int on_cpu, int block) {
    if (!bm) return -1;
    std::lock_guard<std::mutex> g(bm->mu);
    const Pool &p = on_cpu ? bm->cpu : bm->gpu;
    return p.valid(block) ? p.refs(block) : -1;
}

pa_status_t pa_bm_seq_create(pa_block_manager_t *bm, int64_t *seq_out) {
    if (!bm || !seq_out) return PA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> g(bm->mu);
    const int64_t id = bm->next_id++;
    bm->seqs.emplace(id, Seq());
    *seq_out = id;
    return PA_OK;
}

pa_status_t pa_bm_seq_fork(pa_block_manager_t *bm, int64_t parent, int64_t *child_out) {
    if (!bm || !child_out) return PA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> g(bm->mu);
    const Seq *p = bm->find(parent);
    if (!p) return PA_ERR_INVALID_ARG;
    Seq child = *p;
    Pool &pool = child.on_cpu ? bm->cpu : bm->gpu;
    for (int b : child.table) pool.retain(b);
    const int64_t id = bm->next_id++;
    bm->seqs.emplace(id, std::move(child));
    *child_out = id;
    return PA_OK;
}

pa_status_t pa_bm_seq_free(pa_block_manager_t *bm, int64_t seq) {
    if (!bm) return PA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> g(bm->mu);
    Seq *s = bm->find(seq);
    if (!s) return PA_ERR_INVALID_ARG;
    Pool &pool = s->on_cpu ? bm->cpu : bm->gpu;
    for (int b : s->table) pool.release(b);
    bm->seqs.erase(seq);
    return PA_OK;
}

pa_status_t pa_bm_seq_append(pa_block_manager_t *bm, int64_t seq, int num_tokens,
                             int64_t *slots_out) {
    if (!bm || num_tokens < 0) return PA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> g(bm->mu);
    Seq *s = bm->find(seq);
    if (!s || s->on_cpu) return PA_ERR_INVALID_ARG;
    if ((long long)s->n + num_tokens > INT32_MAX) return PA_ERR_INVALID_ARG;
    if (bm->needed(*s, num_tokens) > bm->gpu.num_free()) return PA_ERR_NO_BLOCKS;
    const int B = bm->block_size;
    if (s->n % B && bm->gpu.refs(s->table.back()) > 1) {  // copy-on-write of the last block
        const int old = s->table.back();
        const int nb = bm->gpu.alloc();
        bm->copies.emplace_back(old, nb);
        bm->gpu.release(old);
        s->table.back() = nb;
    }
    while ((long long)s->table.size() * B < (long long)s->n + num_tokens)
        s->table.push_back(bm->gpu.alloc());
    if (slots_out)
        for (int i = 0; i < num_tokens; ++i) {
            const int t = s->n + i;
            slots_out[i] = (int64_t)s->table[t / B] * B + t % B;
        }
    s->n += num_tokens;
    return PA_OK;
}

int pa_bm_blocks_needed(const pa_block_manager_t *bm, int64_t seq, int num_tokens) {
    if (!bm || num_tokens < 0) return -1;
    std::lock_guard<std::mutex> g(bm->mu);
    const Seq *s = bm->find(seq);
    if (!s || s->on_cpu) return -1;
    return bm->needed(*s, num_tokens);
}

int pa_bm_seq_len(const pa_block_manager_t *bm, int64_t seq) {
    if (!bm) return -1;
    std::lock_guard<std::mutex> g(bm->mu);
    const Seq *s = bm->find(seq);
    return s ? s->n : -1;
}

int pa_bm_seq_on_cpu(const pa_block_manager_t *bm, int64_t seq) {
    if (!bm) return -1;
    std::lock_guard<std::mutex> g(bm->mu);
    const Seq *s = bm->find(seq);
    return s ? (s->on_cpu ? 1 : 0) : -1;
}

int pa_bm_seq_table(const pa_block_manager_t *bm, int64_t seq, int32_t *out, int cap) {
    if (!bm || cap < 0 || (cap > 0 && !out)) return -1;
    std::lock_guard<std::mutex> g(bm->mu);
    const Seq *s = bm->find(seq);
    if (!s) return -1;
    const int nb = (int)s->table.size();
    for (int i = 0; i < std::min(cap, nb); ++i) out[i] = s->table[i];
    return nb;
}

pa_status_t pa_bm_build_batch(const pa_block_manager_t *bm, const int64_t *seqs, int n,
                              int32_t *block_tables, int max_blocks_per_seq,
                              int32_t *context_lens) {
    if (!bm || n < 0 || max_blocks_per_seq <= 0) return PA_ERR_INVALID_ARG;
    if (n > 0 && (!seqs || !block_tables || !context_lens)) return PA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> g(bm->mu);
    for (int i = 0; i < n; ++i) {
        const Seq *s = bm->find(seqs[i]);
        if (!s || s->on_cpu || (int)s->table.size() > max_blocks_per_seq)
            return PA_ERR_INVALID_ARG;
    }
    for (int i = 0; i < n; ++i) {
        const Seq *s = bm->find(seqs[i]);
        int32_t *row = block_tables + (size_t)i * max_blocks_per_seq;
        const int nb = (int)s->table.size();
        for (int j = 0; j < max_blocks_per_seq; ++j) row[j] = j < nb ? s->table[j] : -1;
        context_lens[i] = s->n;
    }
    return PA_OK;
}

int pa_bm_take_copies(pa_block_manager_t *bm, int64_t *pairs_out, int cap) {
    if (!bm || cap < 0 || (cap > 0 && !pairs_out)) return -1;
    std::lock_guard<std::mutex> g(bm->mu);
    int k = 0;
    while (k < cap && !bm->copies.empty()) {
        pairs_out[2 * k] = bm->copies.front().first;
        pairs_out[2 * k + 1] = bm->copies.front().second;
        bm->copies.pop_front();
        ++k;
    }
    return k;
}

int pa_bm_num_copies(const pa_block_manager_t *bm) {
    if (!bm) return -1;
    std::lock_guard<std::mutex> g(bm->mu);
    return (int)bm->copies.size();
}

pa_status_t pa_bm_swap_out(pa_block_manager_t *bm, const int64_t *seqs, int n,
                           int64_t *pairs_out, int cap, int *num_pairs) {
    if (!bm) return PA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> g(bm->mu);
    return bm->swap(seqs, n, pairs_out, cap, num_pairs, true);
}

pa_status_t pa_bm_swap_in(pa_block_manager_t *bm, const int64_t *seqs, int n,
                          int64_t *pairs_out, int cap, int *num_pairs) {
    if (!bm) return PA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> g(bm->mu);
    return bm->swap(seqs, n, pairs_out, cap, num_pairs, false);
}

}  // extern "C"
