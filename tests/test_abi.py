"""The C-ABI library without a GPU: it loads, exports every symbol include/pa.h
declares, and its host-only logic (block count, status strings, argument
validation that returns before any CUDA call) behaves as documented."""
import ctypes
import os
import re

import pytest

import oracle
from pagedattention_kv_cache_reshape_gb300 import build as B
from pagedattention_kv_cache_reshape_gb300 import pa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return pa.load()


def _declared():
    src = open(os.path.join(ROOT, "include", "pa.h")).read()
    return re.findall(r"PA_API[^;(]*?\b(pa_\w+)\s*\(", src)


def test_header_declares_the_binding_exports():
    assert sorted(_declared()) == sorted(pa.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_no_cuda_runtime_dependency_at_load():
    # the runtime is linked statically: the library loads without libcudart
    import subprocess
    out = subprocess.run(["ldd", B.LIB], capture_output=True, text=True).stdout
    assert "libcudart" not in out and "libcuda.so" not in out


def test_num_blocks_needed_matches_oracle(lib):
    for bs in (1, 7, 16, 32):
        for n in range(0, 400):
            assert pa.num_blocks_needed(n, bs) == oracle.num_blocks_needed(n, bs)
    assert pa.num_blocks_needed(17, 16) == 2
    assert pa.num_blocks_needed(-1, 16) == -1 and pa.num_blocks_needed(3, 0) == -1


def test_status_strings(lib):
    assert pa.status_string(0) == "PA_OK"
    assert pa.status_string(3) == "PA_ERR_OUT_OF_RANGE"
    assert pa.status_string(99) == "PA_ERR_UNKNOWN"
    assert pa.version() >= 100


def test_host_validation_rejects_before_launch(lib):
    L = lib
    nul = None
    # slot mapping: tokens but no sequences
    assert L.pa_compute_slot_mapping(nul, 0, 4, nul, nul, 5, 16, 8, nul, nul, nul) == pa.ERR_INVALID_ARG
    # slot mapping: null pointers
    assert L.pa_compute_slot_mapping(nul, 1, 4, nul, nul, 5, 16, 8, nul, nul, nul) == pa.ERR_INVALID_ARG
    # zero tokens is a no-op
    assert L.pa_compute_slot_mapping(nul, 1, 4, nul, nul, 0, 16, 8, nul, nul, nul) == pa.OK
    # cache write: token stride shorter than a row
    assert L.pa_reshape_and_cache(1, 1, 10, 64, 1, 1, 1, 3, 2, 32, 16, 8, 0, nul, nul) == pa.ERR_INVALID_ARG
    # cache write: a block size below 1 (any positive block size is written)
    assert L.pa_reshape_and_cache(16, 16, 64, 64, 16, 16, 16, 3, 2, 32, 0, 8, 0, nul, nul) == pa.ERR_INVALID_ARG
    # decode: heads not a multiple of kv-heads
    assert L.pa_decode(16, 16, 16, 16, 16, 16, 2, 6, 4, 128, 16, 4, 8, 0.1, 1, 16, 1 << 20, nul, nul) \
        == pa.ERR_INVALID_ARG
    # decode: unsupported head_dim / block size
    assert L.pa_decode(16, 16, 16, 16, 16, 16, 2, 8, 4, 96, 16, 4, 8, 0.1, 1, 16, 1 << 20, nul, nul) \
        == pa.ERR_UNSUPPORTED
    for bs in (4, 24, 64):   # attention takes block sizes 8, 16 and 32
        assert L.pa_decode(16, 16, 16, 16, 16, 16, 2, 8, 4, 128, bs, 4, 8, 0.1, 1, 16, 1 << 20, nul, nul) \
            == pa.ERR_UNSUPPORTED
    # decode: bad dtype code, NaN scale, null pointer
    assert L.pa_decode(16, 16, 16, 16, 16, 16, 2, 8, 4, 128, 16, 4, 8, 0.1, 7, 16, 1 << 20, nul, nul) \
        == pa.ERR_INVALID_ARG
    assert L.pa_decode(16, 16, 16, 16, 16, 16, 2, 8, 4, 128, 16, 4, 8, float("nan"), 1, 16, 1 << 20, nul, nul) \
        == pa.ERR_INVALID_ARG
    assert L.pa_decode(nul, 16, 16, 16, 16, 16, 2, 8, 4, 128, 16, 4, 8, 0.1, 1, 16, 1 << 20, nul, nul) \
        == pa.ERR_INVALID_ARG
    # decode: nothing to do
    assert L.pa_decode(nul, nul, nul, nul, nul, nul, 0, 8, 4, 128, 16, 4, 8, 0.1, 1, nul, 0, nul, nul) == pa.OK
    # prefill: null cu_seqlens_q
    assert L.pa_varlen_prefill(16, 16, nul, 16, 16, 16, 16, 2, 9, 8, 8, 4, 128, 16, 4, 8, 0.1, 1, 16, 1 << 20,
                               nul, nul) == pa.ERR_INVALID_ARG
    # empty batches: nothing to do, nothing launched
    assert L.pa_varlen_prefill(nul, nul, nul, nul, nul, nul, nul, 0, 0, 0, 8, 4, 128, 16, 4, 8, 0.1, 1, nul, 0,
                               nul, nul) == pa.OK
    assert L.pa_varlen_prefill(nul, nul, nul, nul, nul, nul, nul, 3, 0, 0, 8, 4, 128, 16, 4, 8, 0.1, 1, nul, 0,
                               nul, nul) == pa.OK
    assert L.pa_varlen_encode(nul, nul, nul, nul, nul, nul, nul, 0, 0, 0, 8, 4, 128, 16, 4, 8, 0.1, 1, nul, 0,
                              nul, nul) == pa.OK
    assert L.pa_varlen_step(nul, nul, nul, nul, 512, 512, nul, nul, nul, nul, nul, nul, nul, 0, 0, 0, 8, 4, 128,
                            16, 4, 8, 0.1, 1, nul, 0, nul, nul) == pa.OK
    assert L.pa_decode_step(nul, nul, nul, nul, 512, 512, nul, nul, nul, nul, nul, nul, 0, nul, 0, 8, 4, 128, 16,
                            4, 8, 0.1, 1, nul, 0, nul, nul) == pa.OK
    # varlen step: tokens to write but no key rows
    assert L.pa_varlen_step(16, 16, nul, nul, 512, 512, 16, 16, 16, 16, 16, 16, 16, 2, 9, 8, 8, 4, 128, 16, 4,
                            8, 0.1, 1, 16, 1 << 20, nul, nul) == pa.ERR_INVALID_ARG
    # status helpers: null pointers
    assert L.pa_get_device_status(nul, nul, nul) == pa.ERR_INVALID_ARG
    assert L.pa_reset_device_status(nul, nul) == pa.ERR_INVALID_ARG


def test_workspace_size_grows_with_problem(lib):
    a = pa.decode_workspace_size(16, 32, 8, 128, 16, 64)
    b = pa.decode_workspace_size(256, 32, 8, 128, 16, 256)
    assert 0 < a < b
    assert a % 256 == 0 and b % 256 == 0
    assert pa.varlen_prefill_workspace_size(256, 4344, 32, 8, 128, 16, 256) >= b


def test_missing_library_fails_loudly(tmp_path):
    import importlib
    mod = importlib.import_module("pagedattention_kv_cache_reshape_gb300.pa")
    saved = mod._lib
    try:
        mod._lib = None
        with pytest.raises(ImportError):
            mod.load(str(tmp_path / "nope.so"))
    finally:
        mod._lib = saved


def test_wait_test_hook_checks_its_arguments(lib):
    # host-only: an unknown stall mode or a negative count is rejected; valid
    # settings are taken, and the defaults restore normal operation
    assert lib.pa_set_wait_test(0, 3, 0, None) == pa.ERR_INVALID_ARG
    assert lib.pa_set_wait_test(0, -1, 0, None) == pa.ERR_INVALID_ARG
    assert lib.pa_set_wait_test(0, pa.STALL_PRODUCER, -2, None) == pa.ERR_INVALID_ARG
    assert lib.pa_set_wait_test(5_000_000, pa.STALL_CONSUMER, 4, None) == pa.OK
    assert lib.pa_set_wait_test(0, pa.STALL_NONE, 0, None) == pa.OK
