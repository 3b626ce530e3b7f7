"""pa_decode_static_scratch: decode for callers that cannot allocate device
memory (a plugin interface that only passes tensor pointers, a serving
process whose memory pool has claimed the free device memory).  Its scratch
is a fixed array inside the library; every call reuses that array, so its
results must equal pa_decode's bit for bit, call after call, and match the
oracle within the stated tolerance.

This file is collected last so that a failure here never hides the others.
"""
import ctypes

import pytest
import torch

from pagedattention_kv_cache_reshape_gb300 import pa
from pagedattention_kv_cache_reshape_gb300 import workloads as W

from helpers import compare, gpu_step, oracle_attention, oracle_blocks, oracle_write, to_f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from pagedattention_kv_cache_reshape_gb300 import build
    build.build()
    pa.load()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _call_c_abi(w, out, status, dtype_code=None):
    """The entry point called through the C ABI directly (ctypes)."""
    L = pa.load()
    return L.pa_decode_static_scratch(
        out.data_ptr(), w.q.data_ptr(), w.k_cache.data_ptr(), w.v_cache.data_ptr(),
        w.block_tables.data_ptr(), w.context_lens.data_ptr(), w.num_seqs, w.num_heads,
        w.num_kv_heads, w.head_dim, w.block_size, w.max_blocks, w.num_blocks,
        ctypes.c_float(w.scale), pa.DTYPE_BF16 if dtype_code is None else dtype_code,
        None if status is None else status.data_ptr(), torch.cuda.current_stream().cuda_stream)


def _prepared(w):
    """Writes the step's new tokens (GPU and oracle sides), decodes once through
    pa_decode with a caller workspace, and returns (pa_decode's output, the oracle's)."""
    wc = w.to("cpu")
    _, ref_gpu = gpu_step(w)
    oracle_write(wc)
    torch.cuda.synchronize()
    return ref_gpu.clone(), oracle_attention(wc)


def test_static_scratch_decode_matches_workspace_decode_on_consecutive_calls():
    a = W.gqa(21, oracle_blocks, num_seqs=40, ctx_hi=900, shared_seqs=8, prefix_tokens=128, device=DEV)
    b = W.long(22, oracle_blocks, num_seqs=3, ctx=5000, num_blocks=1000, device=DEV)
    ref_a, orc_a = _prepared(a)
    ref_b, orc_b = _prepared(b)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    # consecutive calls share the array; the third finds the second's contents there
    for w, ref, orc in ((a, ref_a, orc_a), (b, ref_b, orc_b), (a, ref_a, orc_a)):
        out = torch.full_like(w.q, float("nan"))
        assert _call_c_abi(w, out, status) == pa.OK
        torch.cuda.synchronize()
        assert pa.get_device_status(status) == 0, "device status set"
        # same kernels, same partition: bitwise equal to pa_decode
        assert torch.equal(out, ref), f"{w.name}: differs from pa_decode"
        compare(to_f64(out), orc, torch.bfloat16, w.name + " vs oracle")


def test_static_scratch_fp32_takes_the_cuda_core_kernel():
    """fp32 decode runs the CUDA-core kernel, which uses no scratch."""
    w = W.tiny(5, oracle_blocks, device=DEV)
    ref, orc = _prepared(w)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    for _ in range(2):
        out = torch.full_like(w.q, float("nan"))
        assert _call_c_abi(w, out, status, pa.DTYPE_F32) == pa.OK
        torch.cuda.synchronize()
        assert pa.get_device_status(status) == 0
        assert torch.equal(out, ref)
        compare(to_f64(out), orc, torch.float32, "tiny_fp32 vs oracle")


def test_static_scratch_rejects_problems_beyond_its_size():
    need = pa.decode_workspace_size(16384, 32, 8, 128, 16, 512)
    assert need > pa.STATIC_SCRATCH_BYTES
    L = pa.load()
    rc = L.pa_decode_static_scratch(16, 16, 16, 16, 16, 16, 16384, 32, 8, 128, 16, 512, 1 << 20,
                                    ctypes.c_float(0.1), pa.DTYPE_BF16, None, None)
    assert rc == pa.ERR_WORKSPACE


def test_static_scratch_status_codes_match_pa_decode():
    L = pa.load()
    f = ctypes.c_float(0.1)
    # a head mapping that does not divide: pa_decode's INVALID_ARG, also for an empty batch
    for n in (0, 16384):
        assert L.pa_decode_static_scratch(16, 16, 16, 16, 16, 16, n, 30, 8, 128, 16, 512, 1 << 20, f,
                                          pa.DTYPE_BF16, None, None) == pa.ERR_INVALID_ARG
    # an unknown dtype
    assert L.pa_decode_static_scratch(16, 16, 16, 16, 16, 16, 0, 32, 8, 128, 16, 512, 1 << 20, f,
                                      7, None, None) == pa.ERR_INVALID_ARG
    # an empty batch of a valid shape does nothing
    assert L.pa_decode_static_scratch(None, None, None, None, None, None, 0, 32, 8, 128, 16, 512, 64, f,
                                      pa.DTYPE_BF16, None, None) == pa.OK
