"""Thin Python binding of the C ABI in include/pa.h (ctypes).

Argument marshalling only: torch tensors supply device pointers, the current
CUDA stream supplies the stream, and every step of the computation runs in the
library's CUDA kernels.  There is no CPU fallback: if ``libpa.so`` is missing
or a call fails, an exception is raised.

The functions keep the C names without the ``pa_`` prefix.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpa.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_OUT_OF_RANGE, ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT = range(7)
DTYPE_F32, DTYPE_BF16 = 0, 1

EXPORTS = (
    "pa_status_string", "pa_version", "pa_num_blocks_needed", "pa_compute_slot_mapping",
    "pa_reshape_and_cache", "pa_decode_workspace_size", "pa_decode",
    "pa_varlen_prefill_workspace_size", "pa_varlen_prefill", "pa_get_device_status",
    "pa_reset_device_status", "pa_set_timing_events", "pa_decode_static_scratch", "pa_decode_step",
    "pa_copy_blocks", "pa_varlen_encode", "pa_varlen_step",
    "pa_block_manager_create", "pa_block_manager_destroy", "pa_block_manager_num_free",
    "pa_block_manager_refcount", "pa_allocate_slots", "pa_free_sequence", "pa_share_prefix",
    "pa_block_manager_tables", "pa_validate_inputs", "pa_allocate_slots_batch", "pa_set_wait_test",
)
STATIC_SCRATCH_BYTES = 24 << 20
STALL_NONE, STALL_PRODUCER, STALL_CONSUMER = 0, 1, 2
WAIT_DECODE_PRODUCER, WAIT_DECODE_CONSUMER = 1, 2
WAIT_PREFILL_PRODUCER, WAIT_PREFILL_MMA, WAIT_PREFILL_SOFTMAX = 4, 8, 16


class PAError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libpa.so (built by __graft_entry__.build() or build.py)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise ImportError(f"{path} is missing: build the CUDA library first "
                              "(python -m pagedattention_kv_cache_reshape_gb300.build)")
        L = ctypes.CDLL(path)
        vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
        L.pa_status_string.restype = ctypes.c_char_p
        L.pa_status_string.argtypes = [i32]
        L.pa_version.restype = i32
        L.pa_num_blocks_needed.restype = i32
        L.pa_num_blocks_needed.argtypes = [i32, i32]
        L.pa_compute_slot_mapping.restype = i32
        L.pa_compute_slot_mapping.argtypes = [vp, i32, i32, vp, vp, i32, i32, i32, vp, vp, vp]
        L.pa_reshape_and_cache.restype = i32
        L.pa_reshape_and_cache.argtypes = [vp, vp, i64, i64, vp, vp, vp, i32, i32, i32, i32, i32, i32, vp, vp]
        L.pa_decode_workspace_size.restype = sz
        L.pa_decode_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32]
        L.pa_decode.restype = i32
        L.pa_decode.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, f32, i32,
                                vp, sz, vp, vp]
        L.pa_varlen_prefill_workspace_size.restype = sz
        L.pa_varlen_prefill_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, i32]
        L.pa_varlen_prefill.restype = i32
        L.pa_varlen_prefill.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32,
                                        i32, i32, f32, i32, vp, sz, vp, vp]
        L.pa_block_manager_create.restype = vp
        L.pa_block_manager_create.argtypes = [i32, i32, i32]
        L.pa_block_manager_destroy.restype = None
        L.pa_block_manager_destroy.argtypes = [vp]
        L.pa_block_manager_num_free.restype = i32
        L.pa_block_manager_num_free.argtypes = [vp]
        L.pa_block_manager_refcount.restype = i32
        L.pa_block_manager_refcount.argtypes = [vp, i32]
        L.pa_allocate_slots.restype = i32
        L.pa_allocate_slots.argtypes = [vp, i64, i32]
        L.pa_allocate_slots_batch.restype = i32
        L.pa_allocate_slots_batch.argtypes = [vp, vp, vp, i32, vp]
        L.pa_free_sequence.restype = i32
        L.pa_free_sequence.argtypes = [vp, i64]
        L.pa_share_prefix.restype = i32
        L.pa_share_prefix.argtypes = [vp, i64, i64, i32]
        L.pa_block_manager_tables.restype = i32
        L.pa_block_manager_tables.argtypes = [vp, vp, i32, vp, i32, vp]
        L.pa_varlen_encode.restype = i32
        L.pa_varlen_encode.argtypes = L.pa_varlen_prefill.argtypes
        L.pa_get_device_status.restype = i32
        L.pa_get_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_int32), vp]
        L.pa_reset_device_status.restype = i32
        L.pa_reset_device_status.argtypes = [vp, vp]
        L.pa_set_timing_events.restype = i32
        L.pa_set_timing_events.argtypes = [vp, vp]
        L.pa_set_wait_test.restype = i32
        L.pa_set_wait_test.argtypes = [ctypes.c_uint64, i32, i32, vp]
        L.pa_copy_blocks.restype = i32
        L.pa_copy_blocks.argtypes = [vp, vp, vp, vp, i64, i32, i32, vp, i32, vp, vp]
        L.pa_decode_step.restype = i32
        L.pa_decode_step.argtypes = [vp, vp, vp, vp, i64, i64, vp, vp, vp, vp, vp, vp, i32, vp, i32, i32, i32,
                                     i32, i32, i32, i32, f32, i32, vp, sz, vp, vp]
        L.pa_varlen_step.restype = i32
        L.pa_varlen_step.argtypes = [vp, vp, vp, vp, i64, i64, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32,
                                     i32, i32, i32, i32, i32, f32, i32, vp, sz, vp, vp]
        L.pa_decode_static_scratch.restype = i32
        L.pa_decode_static_scratch.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32,
                                               f32, i32, vp, vp]
        L.pa_validate_inputs.restype = i32
        L.pa_validate_inputs.argtypes = [vp, i32, i32, vp, vp, i32, i32, i32, ctypes.POINTER(ctypes.c_int),
                                         ctypes.POINTER(ctypes.c_int64)]
        _lib = L
        return L


def status_string(status: int) -> str:
    return load().pa_status_string(int(status)).decode()


def _check(rc: int, what: str) -> None:
    if rc != OK:
        raise PAError(rc, what)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dev(t: torch.Tensor, name: str, dtype=None) -> int:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _contig(t: torch.Tensor, name: str, dtype=None) -> int:
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return _dev(t, name, dtype)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return DTYPE_F32
    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    raise TypeError(f"unsupported dtype {t.dtype} (float32 or bfloat16)")


def _opt(t) -> int:
    return 0 if t is None else _dev(t, "dev_status", torch.int32)


# ------------------------------------------------------------------ calls

def version() -> int:
    return int(load().pa_version())


def num_blocks_needed(num_tokens: int, block_size: int) -> int:
    return int(load().pa_num_blocks_needed(int(num_tokens), int(block_size)))


def compute_slot_mapping(block_tables, seq_start, cu_seqlens_q, num_blocks: int, total_new: int,
                         block_size: int = 16, slot_mapping=None, dev_status=None, stream=None):
    """pa_compute_slot_mapping; returns the int64 slot_mapping tensor."""
    num_seqs, max_blocks = block_tables.shape
    if slot_mapping is None:
        slot_mapping = torch.empty(total_new, dtype=torch.int64, device=block_tables.device)
    rc = load().pa_compute_slot_mapping(
        _contig(block_tables, "block_tables", torch.int32), num_seqs, max_blocks,
        _contig(seq_start, "seq_start", torch.int32), _contig(cu_seqlens_q, "cu_seqlens_q", torch.int32),
        int(total_new), int(block_size), int(num_blocks),
        _contig(slot_mapping, "slot_mapping", torch.int64), _opt(dev_status), _stream(stream))
    _check(rc, "pa_compute_slot_mapping")
    return slot_mapping


def reshape_and_cache(key, value, k_cache, v_cache, slot_mapping, dev_status=None, stream=None):
    """pa_reshape_and_cache; key/value may be token-strided views (rows contiguous)."""
    num_blocks, block_size, hkv, d = k_cache.shape
    for name, t in (("key", key), ("value", value)):
        if t.dim() != 3 or t.shape[1:] != (hkv, d) or t.stride(2) != 1 or t.stride(1) != d:
            raise ValueError(f"{name} must be [tokens, {hkv}, {d}] with contiguous rows")
    if key.shape[0] != value.shape[0] or slot_mapping.numel() < key.shape[0]:
        raise ValueError("key, value and slot_mapping disagree on the token count")
    if not (key.dtype == value.dtype == k_cache.dtype == v_cache.dtype):
        raise TypeError("key, value and the pools must share one dtype")
    rc = load().pa_reshape_and_cache(
        _dev(key, "key"), _dev(value, "value"), key.stride(0), value.stride(0),
        _contig(k_cache, "k_cache"), _contig(v_cache, "v_cache"),
        _contig(slot_mapping, "slot_mapping", torch.int64), int(key.shape[0]), hkv, d,
        block_size, num_blocks, _dtype_code(k_cache), _opt(dev_status), _stream(stream))
    _check(rc, "pa_reshape_and_cache")


def decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_blocks) -> int:
    return int(load().pa_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim,
                                               block_size, max_blocks))


def varlen_prefill_workspace_size(num_seqs, total_q, num_heads, num_kv_heads, head_dim, block_size,
                                  max_blocks) -> int:
    return int(load().pa_varlen_prefill_workspace_size(num_seqs, total_q, num_heads, num_kv_heads,
                                                       head_dim, block_size, max_blocks))


def _ws(workspace, nbytes, device):
    if workspace is None:
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device)
    return workspace


def decode(q, k_cache, v_cache, block_tables, context_lens, scale: float, out=None,
           workspace=None, dev_status=None, stream=None):
    """pa_decode: q [num_seqs, H, D] -> out [num_seqs, H, D]."""
    num_seqs, H, D = q.shape
    num_blocks, block_size, hkv, d = k_cache.shape
    max_blocks = block_tables.shape[1]
    if out is None:
        out = torch.empty_like(q)
    need = decode_workspace_size(num_seqs, H, hkv, D, block_size, max_blocks)
    workspace = _ws(workspace, need, q.device)
    rc = load().pa_decode(
        _contig(out, "out"), _contig(q, "q"), _contig(k_cache, "k_cache"), _contig(v_cache, "v_cache"),
        _contig(block_tables, "block_tables", torch.int32), _contig(context_lens, "context_lens", torch.int32),
        num_seqs, H, hkv, D, block_size, max_blocks, num_blocks, float(scale), _dtype_code(q),
        _contig(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _opt(dev_status), _stream(stream))
    _check(rc, "pa_decode")
    return out


def decode_step(q, key, value, k_cache, v_cache, block_tables, context_lens, seq_start, cu_seqlens_new,
                scale: float, out=None, slot_mapping=None, workspace=None, dev_status=None, stream=None):
    """pa_decode_step: slot mapping + cache write of the new tokens + decode, in one call.
    Returns (slot_mapping, out)."""
    num_seqs, H, D = q.shape
    num_blocks, block_size, hkv, d = k_cache.shape
    max_blocks = block_tables.shape[1]
    total_new = int(key.shape[0])
    for name, t in (("key", key), ("value", value)):
        if t.dim() != 3 or t.shape[1:] != (hkv, d) or t.stride(2) != 1 or t.stride(1) != d:
            raise ValueError(f"{name} must be [tokens, {hkv}, {d}] with contiguous rows")
    if out is None:
        out = torch.empty_like(q)
    if slot_mapping is None:
        slot_mapping = torch.empty(total_new, dtype=torch.int64, device=q.device)
    need = decode_workspace_size(num_seqs, H, hkv, D, block_size, max_blocks)
    workspace = _ws(workspace, need, q.device)
    rc = load().pa_decode_step(
        _contig(out, "out"), _contig(q, "q"), _dev(key, "key"), _dev(value, "value"), key.stride(0),
        value.stride(0), _contig(k_cache, "k_cache"), _contig(v_cache, "v_cache"),
        _contig(block_tables, "block_tables", torch.int32), _contig(context_lens, "context_lens", torch.int32),
        _contig(seq_start, "seq_start", torch.int32), _contig(cu_seqlens_new, "cu_seqlens_new", torch.int32),
        total_new, _contig(slot_mapping, "slot_mapping", torch.int64), num_seqs, H, hkv, D, block_size,
        max_blocks, num_blocks, float(scale), _dtype_code(q), _contig(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _opt(dev_status), _stream(stream))
    _check(rc, "pa_decode_step")
    return slot_mapping, out


def copy_blocks(src_k, src_v, dst_k, dst_v, pairs, dev_status=None, stream=None):
    """pa_copy_blocks: whole blocks src -> dst between pools of equal block shape.
    Pools may be device tensors or pinned host tensors (reachable from the device);
    pairs is a device int32 tensor [n, 2]."""
    if src_k.shape[1:] != dst_k.shape[1:] or src_k.dtype != dst_k.dtype:
        raise ValueError("source and destination pools must share block shape and dtype")
    for name, t in (("src_k", src_k), ("src_v", src_v), ("dst_k", dst_k), ("dst_v", dst_v)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if not (t.is_cuda or t.is_pinned()):
            raise ValueError(f"{name} must be a CUDA tensor or pinned host memory")
    pairs = pairs.reshape(-1, 2)
    block_bytes = src_k[0].numel() * src_k.element_size()
    rc = load().pa_copy_blocks(src_k.data_ptr(), src_v.data_ptr(), dst_k.data_ptr(), dst_v.data_ptr(),
                               block_bytes, int(src_k.shape[0]), int(dst_k.shape[0]),
                               _contig(pairs, "pairs", torch.int32), int(pairs.shape[0]), _opt(dev_status),
                               _stream(stream))
    _check(rc, "pa_copy_blocks")


def varlen_prefill(q, cu_seqlens_q, k_cache, v_cache, block_tables, context_lens, scale: float,
                   max_q_len: int, out=None, workspace=None, dev_status=None, stream=None,
                   causal: bool = True):
    """pa_varlen_prefill (causal) or pa_varlen_encode (causal=False) over a
    concatenated super-sequence: q [total_q, H, D]."""
    total_q, H, D = q.shape
    num_blocks, block_size, hkv, d = k_cache.shape
    num_seqs, max_blocks = block_tables.shape
    if out is None:
        out = torch.empty_like(q)
    need = varlen_prefill_workspace_size(num_seqs, total_q, H, hkv, D, block_size, max_blocks)
    workspace = _ws(workspace, need, q.device)
    fn = load().pa_varlen_prefill if causal else load().pa_varlen_encode
    rc = fn(
        _contig(out, "out"), _contig(q, "q"), _contig(cu_seqlens_q, "cu_seqlens_q", torch.int32),
        _contig(k_cache, "k_cache"), _contig(v_cache, "v_cache"),
        _contig(block_tables, "block_tables", torch.int32), _contig(context_lens, "context_lens", torch.int32),
        num_seqs, total_q, int(max_q_len), H, hkv, D, block_size, max_blocks, num_blocks, float(scale),
        _dtype_code(q), _contig(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _opt(dev_status), _stream(stream))
    _check(rc, "pa_varlen_prefill" if causal else "pa_varlen_encode")
    return out


def varlen_step(q, key, value, k_cache, v_cache, cu_seqlens_q, block_tables, context_lens, seq_start,
                scale: float, max_q_len: int, out=None, slot_mapping=None, workspace=None, dev_status=None,
                stream=None):
    """pa_varlen_step: slot mapping + cache write of the step's query tokens + causal varlen
    attention over the super-sequence, in one call.  Returns (slot_mapping, out)."""
    total_q, H, D = q.shape
    num_blocks, block_size, hkv, d = k_cache.shape
    num_seqs, max_blocks = block_tables.shape
    for name, t in (("key", key), ("value", value)):
        if t.dim() != 3 or t.shape[0] != total_q or t.shape[1:] != (hkv, d) or t.stride(2) != 1 \
                or t.stride(1) != d:
            raise ValueError(f"{name} must be [{total_q}, {hkv}, {d}] with contiguous rows")
    if out is None:
        out = torch.empty_like(q)
    if slot_mapping is None:
        slot_mapping = torch.empty(total_q, dtype=torch.int64, device=q.device)
    need = varlen_prefill_workspace_size(num_seqs, total_q, H, hkv, D, block_size, max_blocks)
    workspace = _ws(workspace, need, q.device)
    rc = load().pa_varlen_step(
        _contig(out, "out"), _contig(q, "q"), _dev(key, "key"), _dev(value, "value"), key.stride(0),
        value.stride(0), _contig(k_cache, "k_cache"), _contig(v_cache, "v_cache"),
        _contig(cu_seqlens_q, "cu_seqlens_q", torch.int32), _contig(block_tables, "block_tables", torch.int32),
        _contig(context_lens, "context_lens", torch.int32), _contig(seq_start, "seq_start", torch.int32),
        _contig(slot_mapping, "slot_mapping", torch.int64), num_seqs, total_q, int(max_q_len), H, hkv, D,
        block_size, max_blocks, num_blocks, float(scale), _dtype_code(q), _contig(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _opt(dev_status), _stream(stream))
    _check(rc, "pa_varlen_step")
    return slot_mapping, out


def validate_inputs(block_tables, context_lens, slot_mapping, block_size: int, num_blocks: int):
    """pa_validate_inputs on host (CPU) tensors.  Returns (status, check, index):
    status PA_OK or the error code, check the failed check (1-5, 0 when OK) and
    index the offending row or slot index (-1 when OK).  context_lens and
    slot_mapping may be None."""
    def host(t, dtype, name):
        if t is None:
            return None, None
        t = torch.as_tensor(t)
        if t.device.type != "cpu" or t.dtype != dtype:
            raise TypeError(f"{name}: expected a CPU {dtype} tensor")
        t = t.contiguous()
        return t, t.data_ptr()
    bt, bt_p = host(block_tables, torch.int32, "block_tables")
    ctx, ctx_p = host(context_lens, torch.int32, "context_lens")
    sl, sl_p = host(slot_mapping, torch.int64, "slot_mapping")
    num_seqs, max_blocks = (bt.shape[0], bt.shape[1]) if bt is not None else (0, 0)
    check, index = ctypes.c_int(-1), ctypes.c_int64(-2)
    rc = load().pa_validate_inputs(bt_p, num_seqs, max_blocks, ctx_p, sl_p,
                                   0 if sl is None else sl.numel(), block_size, num_blocks,
                                   ctypes.byref(check), ctypes.byref(index))
    return int(rc), int(check.value), int(index.value)


def get_device_status(dev_status, stream=None) -> int:
    host = ctypes.c_int32(-1)
    rc = load().pa_get_device_status(_dev(dev_status, "dev_status", torch.int32), ctypes.byref(host),
                                     _stream(stream))
    _check(rc, "pa_get_device_status")
    return int(host.value)


def reset_device_status(dev_status, stream=None) -> None:
    _check(load().pa_reset_device_status(_dev(dev_status, "dev_status", torch.int32), _stream(stream)),
           "pa_reset_device_status")


def set_timing_events(ev_begin=None, ev_end=None) -> None:
    """pa_set_timing_events with torch.cuda.Event objects (or None, None)."""
    def handle(ev):
        if ev is None:
            return None
        if ev.cuda_event == 0:      # torch creates the CUDA event on first record
            ev.record()
        return ev.cuda_event
    _check(load().pa_set_timing_events(handle(ev_begin), handle(ev_end)), "pa_set_timing_events")


def set_wait_test(limit_ns: int = 0, stall: int = STALL_NONE, after: int = 0, sites=None) -> None:
    """pa_set_wait_test: the bounded in-kernel waits' limit (0 = one second) and
    the test stall for later calls from this thread; sites is an optional
    device int32 tensor that receives the WAIT_* bits of the waits that ran out."""
    _check(load().pa_set_wait_test(int(limit_ns), int(stall), int(after),
                                   None if sites is None else _dev(sites, "sites", torch.int32)),
           "pa_set_wait_test")


def decode_static_scratch(q, k_cache, v_cache, block_tables, context_lens, scale: float, out=None,
                          dev_status=None, stream=None):
    """pa_decode_static_scratch: pa_decode with the library's fixed scratch array
    (for callers that cannot allocate device memory)."""
    num_seqs, H, D = q.shape
    num_blocks, block_size, hkv, d = k_cache.shape
    max_blocks = block_tables.shape[1]
    if out is None:
        out = torch.empty_like(q)
    rc = load().pa_decode_static_scratch(
        _contig(out, "out"), _contig(q, "q"), _contig(k_cache, "k_cache"), _contig(v_cache, "v_cache"),
        _contig(block_tables, "block_tables", torch.int32), _contig(context_lens, "context_lens", torch.int32),
        num_seqs, H, hkv, D, block_size, max_blocks, num_blocks, float(scale), _dtype_code(q),
        _opt(dev_status), _stream(stream))
    _check(rc, "pa_decode_static_scratch")
    return out


class BlockManager:
    """Host block pool (pa_block_manager_*): allocate_slots, free, shared prefixes,
    and the int32 block tables / token counts the kernels consume."""

    def __init__(self, num_blocks: int, block_size: int = 16, max_blocks_per_seq: int = 4096):
        self._L = load()
        self._h = self._L.pa_block_manager_create(num_blocks, block_size, max_blocks_per_seq)
        if not self._h:
            raise ValueError("invalid block manager arguments")
        self.num_blocks, self.block_size, self.max_blocks_per_seq = num_blocks, block_size, max_blocks_per_seq

    def close(self):
        if self._h:
            self._L.pa_block_manager_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def num_free(self) -> int:
        return int(self._L.pa_block_manager_num_free(self._h))

    def refcount(self, block: int) -> int:
        return int(self._L.pa_block_manager_refcount(self._h, int(block)))

    def allocate_slots(self, seq_id: int, num_new_tokens: int) -> int:
        """Returns the status (OK, ERR_OUT_OF_RANGE when the pool is short, ...)."""
        return int(self._L.pa_allocate_slots(self._h, int(seq_id), int(num_new_tokens)))

    def allocate_slots_batch(self, seq_ids, num_new_tokens, statuses=None) -> int:
        """pa_allocate_slots_batch on host int64 seq_ids / int32 counts (numpy
        or CPU tensors); fills statuses (int32, same length) when given."""
        import numpy as np
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        cnt = np.ascontiguousarray(num_new_tokens, dtype=np.int32)
        if ids.shape != cnt.shape:
            raise ValueError("seq_ids and num_new_tokens must have the same length")
        st_ptr = None
        if statuses is not None:
            if not (isinstance(statuses, np.ndarray) and statuses.dtype == np.int32 and statuses.flags.c_contiguous
                    and statuses.shape == ids.shape):
                raise ValueError("statuses must be a contiguous int32 numpy array of the same length")
            st_ptr = statuses.ctypes.data
        return int(self._L.pa_allocate_slots_batch(self._h, ids.ctypes.data, cnt.ctypes.data, int(ids.size),
                                                   st_ptr))

    def free(self, seq_id: int) -> int:
        return int(self._L.pa_free_sequence(self._h, int(seq_id)))

    def share_prefix(self, parent_id: int, child_id: int, num_tokens: int) -> int:
        return int(self._L.pa_share_prefix(self._h, int(parent_id), int(child_id), int(num_tokens)))

    def tables(self, seq_ids, max_blocks: int):
        """(block_tables int32 [n, max_blocks], num_tokens int32 [n]) as CPU tensors."""
        ids = torch.tensor(list(seq_ids), dtype=torch.int64)
        bt = torch.empty((ids.numel(), max_blocks), dtype=torch.int32)
        nt = torch.empty(ids.numel(), dtype=torch.int32)
        rc = self._L.pa_block_manager_tables(self._h, ids.data_ptr(), ids.numel(), bt.data_ptr(),
                                             int(max_blocks), nt.data_ptr())
        _check(rc, "pa_block_manager_tables")
        return bt, nt
