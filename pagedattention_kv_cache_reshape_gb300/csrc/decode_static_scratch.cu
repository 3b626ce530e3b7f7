// decode_static_scratch.cu -- pa_decode_static_scratch: the decode entry
// point for callers that cannot allocate device memory (a plugin interface
// that only passes tensor pointers, a serving process whose memory pool has
// claimed the free device memory).  Its scratch is a fixed array in this
// file instead of a caller workspace; the kernels are pa_decode's.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <vector>

#include "pa.h"

namespace {

// Held by every GPU that loads the library, until the process exits.
static __device__ __align__(256) uint8_t g_static_scratch[PA_STATIC_SCRATCH_BYTES];

// In host code g_static_scratch names a host-side stand-in, not device
// memory: a kernel given it would fault or read the wrong memory.  The
// device address is looked up once per device, with that device current.
cudaError_t static_scratch_address(void **out) {
    static std::mutex mu;
    static std::vector<void *> addr;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    if ((int)addr.size() <= dev) addr.resize(dev + 1, nullptr);
    if (addr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess) return e;
        addr[dev] = p;
    }
    *out = addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" pa_status pa_decode_static_scratch(void *out, const void *q, const void *k_cache,
                                              const void *v_cache, const int32_t *block_tables,
                                              const int32_t *context_lens, int num_seqs,
                                              int num_heads, int num_kv_heads, int head_dim,
                                              int block_size, int max_blocks, int num_blocks,
                                              float scale, pa_dtype dtype, int32_t *dev_status,
                                              pa_stream_t stream) {
    // reject what does not fit before touching the device
    const size_t need = pa_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim,
                                                 block_size, max_blocks);
    if (need > PA_STATIC_SCRATCH_BYTES) return PA_ERR_WORKSPACE;
    if (num_seqs == 0) return PA_OK;
    void *scratch = nullptr;
    if (static_scratch_address(&scratch) != cudaSuccess) return PA_ERR_CUDA;
    return pa_decode(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs, num_heads,
                     num_kv_heads, head_dim, block_size, max_blocks, num_blocks, scale, dtype,
                     scratch, PA_STATIC_SCRATCH_BYTES, dev_status, stream);
}
