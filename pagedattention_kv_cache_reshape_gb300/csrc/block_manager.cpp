// block_manager.cpp -- host-side physical block allocator that produces the
// block tables the kernels read.
//
// "vLLM изнутри: как устроен движок для быстрого инференса LLM", allocate_slots
// paragraph: the KV-cache manager keeps a pool of free blocks; allocate_slots
// computes how many new blocks a request needs (16 tokens per block, so 17 new
// tokens need ceil(17/16) = 2), checks that the pool holds that many, and
// otherwise leaves the decision to preempt or skip to the scheduler.
// "vLLM：颠覆大模型推理的高效API服务引擎深度解析" §2.2: blocks of a finished
// request go straight back to the free pool; §1.3: blocks may be referenced
// read-only by several block tables (shared prefixes), so a block returns to
// the pool only when its last reference goes.
#include <cstdint>
#include <cstring>
#include <deque>
#include <mutex>
#include <unordered_map>
#include <vector>

#include "pa.h"

struct pa_block_manager {
    int num_blocks;
    int block_size;
    int max_blocks_per_seq;
    std::deque<int32_t> free_queue;    // allocation takes from the front, frees go to the back
    std::vector<int32_t> refcount;
    struct Seq {
        std::vector<int32_t> blocks;
        int64_t num_tokens = 0;
    };
    std::unordered_map<int64_t, Seq> seqs;
    std::mutex mu;
};

namespace {
int64_t blocks_for(int64_t tokens, int block_size) {
    return tokens / block_size + (tokens % block_size != 0 ? 1 : 0);
}
}  // namespace

extern "C" {

pa_block_manager *pa_block_manager_create(int num_blocks, int block_size, int max_blocks_per_seq) {
    if (num_blocks <= 0 || block_size <= 0 || max_blocks_per_seq <= 0) return nullptr;
    pa_block_manager *m = new (std::nothrow) pa_block_manager();
    if (!m) return nullptr;
    m->num_blocks = num_blocks;
    m->block_size = block_size;
    m->max_blocks_per_seq = max_blocks_per_seq;
    m->refcount.assign(num_blocks, 0);
    for (int32_t b = 0; b < num_blocks; ++b) m->free_queue.push_back(b);
    return m;
}

void pa_block_manager_destroy(pa_block_manager *m) { delete m; }

int pa_block_manager_num_free(pa_block_manager *m) {
    if (!m) return -1;
    std::lock_guard<std::mutex> lock(m->mu);
    return (int)m->free_queue.size();
}

// allocate_slots with the manager's lock held
static pa_status allocate_locked(pa_block_manager *m, int64_t seq_id, int num_new_tokens) {
    if (num_new_tokens < 0) return PA_ERR_INVALID_ARG;
    pa_block_manager::Seq &s = m->seqs[seq_id];
    const int64_t total = s.num_tokens + num_new_tokens;
    const int64_t need = blocks_for(total, m->block_size) - (int64_t)s.blocks.size();
    if (blocks_for(total, m->block_size) > m->max_blocks_per_seq) {
        if (s.blocks.empty() && s.num_tokens == 0) m->seqs.erase(seq_id);
        return PA_ERR_INVALID_ARG;
    }
    // appending into a block another table also references would write a
    // shared block: not allowed (shared prefixes are whole blocks)
    if (num_new_tokens > 0 && s.num_tokens % m->block_size != 0 && !s.blocks.empty() &&
        m->refcount[s.blocks.back()] > 1)
        return PA_ERR_UNSUPPORTED;
    if (need > (int64_t)m->free_queue.size()) {   // not enough: nothing is taken
        if (s.blocks.empty() && s.num_tokens == 0) m->seqs.erase(seq_id);
        return PA_ERR_OUT_OF_RANGE;
    }
    for (int64_t i = 0; i < need; ++i) {
        const int32_t b = m->free_queue.front();
        m->free_queue.pop_front();
        m->refcount[b] = 1;
        s.blocks.push_back(b);
    }
    s.num_tokens = total;
    return PA_OK;
}

pa_status pa_allocate_slots(pa_block_manager *m, int64_t seq_id, int num_new_tokens) {
    if (!m) return PA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(m->mu);
    return allocate_locked(m, seq_id, num_new_tokens);
}

pa_status pa_allocate_slots_batch(pa_block_manager *m, const int64_t *seq_ids, const int32_t *num_new_tokens,
                                  int n, int32_t *statuses) {
    if (!m || n < 0 || (n > 0 && (!seq_ids || !num_new_tokens))) return PA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(m->mu);
    pa_status first = PA_OK;
    for (int i = 0; i < n; ++i) {
        const pa_status st = allocate_locked(m, seq_ids[i], num_new_tokens[i]);
        if (statuses) statuses[i] = st;
        if (st != PA_OK && first == PA_OK) first = st;
    }
    return first;
}

pa_status pa_free_sequence(pa_block_manager *m, int64_t seq_id) {
    if (!m) return PA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(m->mu);
    auto it = m->seqs.find(seq_id);
    if (it == m->seqs.end()) return PA_ERR_INVALID_ARG;
    for (int32_t b : it->second.blocks)
        if (--m->refcount[b] == 0) m->free_queue.push_back(b);
    m->seqs.erase(it);
    return PA_OK;
}

pa_status pa_share_prefix(pa_block_manager *m, int64_t parent_id, int64_t child_id, int num_tokens) {
    if (!m || num_tokens < 0) return PA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(m->mu);
    if (num_tokens % m->block_size != 0) return PA_ERR_UNSUPPORTED;   // whole blocks only
    auto pit = m->seqs.find(parent_id);
    if (pit == m->seqs.end() || m->seqs.count(child_id)) return PA_ERR_INVALID_ARG;
    const int64_t nb = num_tokens / m->block_size;
    if (nb > (int64_t)pit->second.blocks.size() || num_tokens > pit->second.num_tokens)
        return PA_ERR_INVALID_ARG;
    pa_block_manager::Seq child;
    child.blocks.assign(pit->second.blocks.begin(), pit->second.blocks.begin() + nb);
    child.num_tokens = num_tokens;
    for (int32_t b : child.blocks) ++m->refcount[b];
    m->seqs.emplace(child_id, std::move(child));
    return PA_OK;
}

pa_status pa_block_manager_tables(pa_block_manager *m, const int64_t *seq_ids, int n,
                                  int32_t *block_tables, int max_blocks, int32_t *num_tokens) {
    if (!m || n < 0 || (n > 0 && (!seq_ids || !block_tables || !num_tokens)) || max_blocks <= 0)
        return PA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(m->mu);
    for (int i = 0; i < n; ++i) {
        auto it = m->seqs.find(seq_ids[i]);
        if (it == m->seqs.end()) return PA_ERR_INVALID_ARG;
        const std::vector<int32_t> &bl = it->second.blocks;
        if ((int)bl.size() > max_blocks) return PA_ERR_INVALID_ARG;
        for (int j = 0; j < max_blocks; ++j)
            block_tables[(int64_t)i * max_blocks + j] = j < (int)bl.size() ? bl[j] : -1;
        num_tokens[i] = (int32_t)it->second.num_tokens;
    }
    return PA_OK;
}

int pa_block_manager_refcount(pa_block_manager *m, int block) {
    if (!m || block < 0 || block >= m->num_blocks) return -1;
    std::lock_guard<std::mutex> lock(m->mu);
    return m->refcount[block];
}

}  // extern "C"
