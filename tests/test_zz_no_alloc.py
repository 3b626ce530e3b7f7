"""pa_decode_static_scratch: decode for callers that cannot allocate device
memory (a plugin interface that only passes tensor pointers, a serving
process whose memory pool has claimed the free device memory).  Its scratch
is a fixed array inside the library; its results must match pa_decode's,
call after call, although every call reuses the same array.

This file is collected last so that a failure here never hides the others.
"""
import ctypes

import pytest
import torch

from pagedattention_kv_cache_reshape_gb300 import pa
from pagedattention_kv_cache_reshape_gb300 import workloads as W

from helpers import compare, gpu_step, oracle_blocks, to_f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from pagedattention_kv_cache_reshape_gb300 import build
    build.build()
    pa.load()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _call_c_abi(w, out):
    """The new entry point, called through the C ABI directly (ctypes)."""
    L = pa.load()
    rc = L.pa_decode_static_scratch(
        out.data_ptr(), w.q.data_ptr(), w.k_cache.data_ptr(), w.v_cache.data_ptr(),
        w.block_tables.data_ptr(), w.context_lens.data_ptr(), w.num_seqs, w.num_heads,
        w.num_kv_heads, w.head_dim, w.block_size, w.max_blocks, w.num_blocks,
        ctypes.c_float(w.scale), pa.DTYPE_BF16, None, torch.cuda.current_stream().cuda_stream)
    assert rc == pa.OK, pa.status_string(rc)


def test_static_scratch_decode_matches_workspace_decode_on_consecutive_calls():
    a = W.gqa(21, oracle_blocks, num_seqs=40, ctx_hi=900, shared_seqs=8, prefix_tokens=128, device=DEV)
    b = W.long(22, oracle_blocks, num_seqs=3, ctx=5000, num_blocks=1000, device=DEV)
    _, ref_a = gpu_step(a)            # writes the new tokens, then decodes with a workspace
    _, ref_b = gpu_step(b)
    torch.cuda.synchronize()
    for w, ref in ((a, ref_a), (b, ref_b), (a, ref_a)):   # consecutive calls share the array
        out = torch.full_like(w.q, float("nan"))
        _call_c_abi(w, out)
        torch.cuda.synchronize()
        compare(to_f64(out), to_f64(ref), torch.bfloat16, w.name)


def test_static_scratch_rejects_problems_beyond_its_size():
    need = pa.decode_workspace_size(16384, 32, 8, 128, 16, 512)
    assert need > pa.STATIC_SCRATCH_BYTES
    L = pa.load()
    rc = L.pa_decode_static_scratch(16, 16, 16, 16, 16, 16, 16384, 32, 8, 128, 16, 512, 1 << 20,
                                    ctypes.c_float(0.1), pa.DTYPE_BF16, None, None)
    assert rc == pa.ERR_WORKSPACE
