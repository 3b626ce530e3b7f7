// decode_static_scratch.cu -- pa_decode_static_scratch: the decode entry
// point for callers that cannot allocate device memory (a plugin interface
// that only passes tensor pointers, a serving process whose memory pool has
// claimed the free device memory).  Its scratch is a fixed array in this
// file instead of a caller workspace; the kernels are pa_decode's.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <vector>

#include "pa.h"
#include "pa_internal.h"

namespace {

// Held by every GPU that loads the library, until the process exits.
static __device__ __align__(256) uint8_t g_static_scratch[PA_STATIC_SCRATCH_BYTES];

// Unique id of the calling thread's current CUDA context (stable for the
// context's life, never reused by a later context, so a cudaDeviceReset shows
// up as a new id); 0 when the driver entry points are unavailable or no
// context is current.
unsigned long long current_context_id() {
    typedef CUresult (*GetCurrentFn)(CUcontext *);
    typedef CUresult (*GetIdFn)(CUcontext, unsigned long long *);
    static GetCurrentFn get_current = nullptr;
    static GetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetIdFn>(p);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
    if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// In host code g_static_scratch names a host-side stand-in, not device
// memory: a kernel given it would fault or read the wrong memory.  The
// device address is looked up with the device current, once per device and
// context: a context created after a cudaDeviceReset gets a fresh lookup.
cudaError_t static_scratch_address(void **out) {
    struct Entry {
        void *addr = nullptr;
        unsigned long long ctx_id = 0;
    };
    static std::mutex mu;
    static std::vector<Entry> cache;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long id = current_context_id();
    std::lock_guard<std::mutex> lock(mu);
    if ((int)cache.size() <= dev) cache.resize(dev + 1);
    Entry &c = cache[dev];
    if (c.addr == nullptr || id == 0 || c.ctx_id != id) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess) return e;
        c.addr = p;
        c.ctx_id = current_context_id();   // the lookup made the context current
    }
    *out = c.addr;
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
    // pa_decode's own checks first, so both entry points return the same
    // codes; then the size limit, which only the split decode (the path that
    // uses scratch) is subject to; all before touching the device
    size_t need = 0;
    const pa_status st = pa::decode_requirements(out, q, k_cache, v_cache, block_tables, context_lens,
                                                 num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                                                 max_blocks, num_blocks, scale, dtype, &need);
    if (st != PA_OK) return st;
    if (need > PA_STATIC_SCRATCH_BYTES) return PA_ERR_WORKSPACE;
    if (num_seqs == 0) return PA_OK;
    void *scratch = nullptr;
    if (need > 0 && static_scratch_address(&scratch) != cudaSuccess) return PA_ERR_CUDA;
    return pa_decode(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs, num_heads,
                     num_kv_heads, head_dim, block_size, max_blocks, num_blocks, scale, dtype,
                     scratch, need > 0 ? PA_STATIC_SCRATCH_BYTES : 0, dev_status, stream);
}
