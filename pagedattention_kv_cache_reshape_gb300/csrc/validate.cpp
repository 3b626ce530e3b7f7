// validate.cpp -- pa_validate_inputs: host-side check of the preconditions the
// kernels rely on but do not test (ranges of lengths, table entries and
// slots; no slot written twice; no write into a block shared by several
// tables).  "vLLM：颠覆大模型推理的高效API服务引擎深度解析" §1.2-1.3: block
// tables map a sequence's logical blocks to physical ones, and shared blocks
// are only read.
#include <stdint.h>

#include <unordered_set>
#include <vector>

#include "pa.h"

namespace {

struct Report {
    int *check;
    int64_t *index;
    pa_status fail(int c, int64_t i, pa_status st) const {
        if (check) *check = c;
        if (index) *index = i;
        return st;
    }
};

}  // namespace

extern "C" pa_status pa_validate_inputs(const int32_t *block_tables, int num_seqs, int max_blocks,
                                        const int32_t *context_lens, const int64_t *slot_mapping,
                                        int num_slots, int block_size, int num_blocks,
                                        int *failed_check, int64_t *bad_index) {
    const Report rep{failed_check, bad_index};
    if (failed_check) *failed_check = 0;
    if (bad_index) *bad_index = -1;
    if (num_seqs < 0 || max_blocks < 0 || num_slots < 0 || block_size <= 0 || num_blocks < 0)
        return PA_ERR_INVALID_ARG;
    if ((context_lens && num_seqs > 0 && !block_tables) || (num_slots > 0 && !slot_mapping))
        return PA_ERR_INVALID_ARG;

    // references to each physical block from the used entries of all tables
    std::vector<int32_t> refs;
    if (context_lens) {
        refs.assign((size_t)num_blocks, 0);
        const int64_t max_tokens = (int64_t)max_blocks * block_size;
        for (int s = 0; s < num_seqs; ++s) {                              // check 1
            const int64_t ctx = context_lens[s];
            if (ctx < 1 || ctx > max_tokens) return rep.fail(1, s, PA_ERR_OUT_OF_RANGE);
        }
        for (int s = 0; s < num_seqs; ++s) {                              // check 2
            const int64_t used = ((int64_t)context_lens[s] + block_size - 1) / block_size;
            const int32_t *row = block_tables + (int64_t)s * max_blocks;
            for (int64_t j = 0; j < used; ++j) {
                const int32_t b = row[j];
                if (b < 0 || b >= num_blocks) return rep.fail(2, s, PA_ERR_OUT_OF_RANGE);
                ++refs[(size_t)b];
            }
        }
    }
    const int64_t pool_slots = (int64_t)num_blocks * block_size;
    for (int i = 0; i < num_slots; ++i)                                   // check 3
        if (slot_mapping[i] >= pool_slots) return rep.fail(3, i, PA_ERR_OUT_OF_RANGE);

    // check 4: a dense mark per pool slot when the pool is moderate, else a set
    if (pool_slots <= ((int64_t)1 << 28)) {
        std::vector<uint8_t> seen((size_t)pool_slots, 0);
        for (int i = 0; i < num_slots; ++i) {
            const int64_t sl = slot_mapping[i];
            if (sl < 0) continue;
            if (seen[(size_t)sl]) return rep.fail(4, i, PA_ERR_INVALID_ARG);
            seen[(size_t)sl] = 1;
        }
    } else {
        std::unordered_set<int64_t> seen;
        for (int i = 0; i < num_slots; ++i) {
            const int64_t sl = slot_mapping[i];
            if (sl < 0) continue;
            if (!seen.insert(sl).second) return rep.fail(4, i, PA_ERR_INVALID_ARG);
        }
    }
    if (context_lens) {                                                   // check 5
        for (int i = 0; i < num_slots; ++i) {
            const int64_t sl = slot_mapping[i];
            if (sl >= 0 && refs[(size_t)(sl / block_size)] >= 2) return rep.fail(5, i, PA_ERR_INVALID_ARG);
        }
    }
    return PA_OK;
}
