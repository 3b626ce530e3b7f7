"""CPU fp64 oracle for the paged KV-cache hot path (ctypes wrapper over oracle.c).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package.  It shares
no code with the CUDA library and the CUDA library never calls it.

What each function computes, and the passage it follows, is documented in
``oracle.c``.  Inputs are CPU torch tensors (fp32 or bf16 for floating point,
int32 / int64 for indices); floating-point results come back as float64
numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

OK, ERR_ARG, ERR_RANGE = 0, 1, 3
F32, BF16 = 0, 1


class OracleError(ValueError):
    """The oracle rejected its inputs (bad argument or out-of-range index)."""


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (OpenMP when available).  Returns the .so path."""
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= newest:
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(tmp, _LIB)
    return _LIB


class _Problem(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p), ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
        ("block_tables", ctypes.c_void_p), ("context_lens", ctypes.c_void_p),
        ("cu_seqlens_q", ctypes.c_void_p),
        ("num_seqs", ctypes.c_int), ("num_heads", ctypes.c_int), ("num_kv_heads", ctypes.c_int),
        ("head_dim", ctypes.c_int), ("block_size", ctypes.c_int), ("max_blocks", ctypes.c_int),
        ("num_blocks", ctypes.c_int), ("dtype", ctypes.c_int), ("scale", ctypes.c_double),
        ("non_causal", ctypes.c_int),
    ]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            # ORACLE_LIB points the tests at a deliberately broken build (the
            # mutation tests check that the pins catch planted mistakes)
            L = ctypes.CDLL(os.environ.get("ORACLE_LIB") or build())
            vp, i32, i64, dp = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_void_p
            L.or_num_blocks_needed.restype = ctypes.c_longlong
            L.or_num_blocks_needed.argtypes = [ctypes.c_longlong, ctypes.c_longlong]
            L.or_slot_mapping.argtypes = [vp, i32, i32, vp, vp, i32, i32, vp]
            L.or_reshape_and_cache.argtypes = [vp, vp, i64, i64, vp, vp, vp, i32, i32, i32, i32, i32, i32]
            L.or_paged_attention.argtypes = [ctypes.POINTER(_Problem), dp, i32]
            L.or_paged_attention_rows.argtypes = [ctypes.POINTER(_Problem), vp, vp, i32, dp, i32]
            L.or_attention_partial.argtypes = [ctypes.POINTER(_Problem), i32, i32, i32,
                                               ctypes.c_longlong, ctypes.c_longlong, dp, dp, dp]
            L.or_merge_partials.argtypes = [dp, dp, dp, i32, i32, dp]
            L.or_copy_blocks.argtypes = [vp, vp, vp, vp, i64, i32, i32, vp, i32]
            L.or_max_threads.restype = i32
            _lib = L
    return _lib


def _check(rc: int, what: str) -> None:
    if rc != OK:
        kind = "out-of-range index" if rc == ERR_RANGE else "invalid argument"
        raise OracleError(f"oracle {what}: {kind} (code {rc})")


def _cpu(t: torch.Tensor, dtype=None) -> torch.Tensor:
    t = t.detach()
    if t.device.type != "cpu":
        t = t.cpu()
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {t.dtype}")
    return t.contiguous()


def _ptr(t: torch.Tensor) -> int:
    return t.data_ptr()


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"oracle supports float32 and bfloat16, got {t.dtype}")


def max_threads() -> int:
    return int(lib().or_max_threads())


# ---------------------------------------------------------------- a1
def num_blocks_needed(num_tokens: int, block_size: int) -> int:
    """ceil(num_tokens / block_size); -1 for invalid arguments."""
    return int(lib().or_num_blocks_needed(int(num_tokens), int(block_size)))


# ---------------------------------------------------------------- a2
def slot_mapping(block_tables, seq_start, cu_seqlens_q, block_size: int, num_blocks: int) -> np.ndarray:
    bt = _cpu(block_tables, torch.int32)
    ss = _cpu(seq_start, torch.int32)
    cu = _cpu(cu_seqlens_q, torch.int32)
    num_seqs, max_blocks = bt.shape
    total = int(cu[-1]) if cu.numel() else 0
    out = np.empty(total, dtype=np.int64)
    rc = lib().or_slot_mapping(_ptr(bt), num_seqs, max_blocks, _ptr(ss), _ptr(cu),
                               block_size, num_blocks, out.ctypes.data)
    _check(rc, "slot_mapping")
    return out


# ---------------------------------------------------------------- a3
def validate_slots(slots: np.ndarray) -> None:
    """Precondition of the cache write: live slots are pairwise distinct."""
    live = np.asarray(slots)[np.asarray(slots) >= 0]
    if np.unique(live).size != live.size:
        raise OracleError("duplicate slots in one cache write")


def reshape_and_cache(key, value, k_cache, v_cache, slots, block_size: int) -> None:
    """Writes key/value rows into the CPU pools in place (byte copies)."""
    for c in (k_cache, v_cache):
        if c.device.type != "cpu" or not c.is_contiguous():
            raise ValueError("pools must be contiguous CPU tensors (written in place)")
    slots = np.ascontiguousarray(np.asarray(slots, dtype=np.int64))
    validate_slots(slots)
    num_blocks, B, hkv, d = k_cache.shape
    if B != block_size:
        raise ValueError("pool block dimension differs from block_size")
    if key.stride(-1) != 1 or key.stride(-2) != d or value.stride(-1) != 1 or value.stride(-2) != d:
        raise ValueError("key/value rows must be [num_kv_heads, head_dim] contiguous")
    if key.device.type != "cpu" or value.device.type != "cpu":
        raise ValueError("key/value must be CPU tensors")
    rc = lib().or_reshape_and_cache(_ptr(key), _ptr(value), key.stride(0), value.stride(0),
                                    _ptr(k_cache), _ptr(v_cache), slots.ctypes.data,
                                    int(key.shape[0]), hkv, d, block_size, num_blocks,
                                    _dtype_code(k_cache))
    _check(rc, "reshape_and_cache")


# ---------------------------------------------------------------- a4 / a6
class Problem:
    """Keeps the CPU tensors alive while the C struct points into them."""

    def __init__(self, q, k_cache, v_cache, block_tables, context_lens, scale: float,
                 cu_seqlens_q=None, causal: bool = True):
        self.q = _cpu(q)
        self.k_cache = _cpu(k_cache)
        self.v_cache = _cpu(v_cache)
        if not (self.q.dtype == self.k_cache.dtype == self.v_cache.dtype):
            raise TypeError("q and pools must share one dtype")
        self.bt = _cpu(block_tables, torch.int32)
        self.ctx = _cpu(context_lens, torch.int32)
        self.cu = None if cu_seqlens_q is None else _cpu(cu_seqlens_q, torch.int32)
        num_blocks, B, hkv, d = self.k_cache.shape
        self.num_heads = int(self.q.shape[1])
        self.head_dim = d
        self.rows = int(self.q.shape[0])
        self.c = _Problem(
            q=_ptr(self.q), k_cache=_ptr(self.k_cache), v_cache=_ptr(self.v_cache),
            block_tables=_ptr(self.bt), context_lens=_ptr(self.ctx),
            cu_seqlens_q=None if self.cu is None else _ptr(self.cu),
            num_seqs=int(self.bt.shape[0]), num_heads=self.num_heads, num_kv_heads=hkv,
            head_dim=d, block_size=B, max_blocks=int(self.bt.shape[1]), num_blocks=num_blocks,
            dtype=_dtype_code(self.q), scale=float(scale), non_causal=0 if causal else 1)


def paged_attention(q, k_cache, v_cache, block_tables, context_lens, scale: float,
                    cu_seqlens_q=None, nthreads: int = 1, causal: bool = True) -> np.ndarray:
    """Full output [rows, num_heads, head_dim] in float64."""
    pr = Problem(q, k_cache, v_cache, block_tables, context_lens, scale, cu_seqlens_q, causal)
    out = np.zeros((pr.rows, pr.num_heads, pr.head_dim), dtype=np.float64)
    rc = lib().or_paged_attention(ctypes.byref(pr.c), out.ctypes.data, int(nthreads))
    _check(rc, "paged_attention")
    return out


def paged_attention_rows(q, k_cache, v_cache, block_tables, context_lens, scale: float,
                         rows, heads, cu_seqlens_q=None, nthreads: int = 1,
                         causal: bool = True) -> np.ndarray:
    """Output of selected (row, head) pairs: [nsel, head_dim] float64."""
    pr = Problem(q, k_cache, v_cache, block_tables, context_lens, scale, cu_seqlens_q, causal)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
    heads = np.ascontiguousarray(np.asarray(heads, dtype=np.int32))
    out = np.zeros((rows.size, pr.head_dim), dtype=np.float64)
    rc = lib().or_paged_attention_rows(ctypes.byref(pr.c), rows.ctypes.data, heads.ctypes.data,
                                       int(rows.size), out.ctypes.data, int(nthreads))
    _check(rc, "paged_attention_rows")
    return out


# ---------------------------------------------------------------- a5
def attention_partial(problem: Problem, s: int, i: int, h: int, j_begin: int, j_end: int):
    """(m, l, o) of one query row over keys [j_begin, j_end)."""
    m = np.zeros(1)
    l = np.zeros(1)
    o = np.zeros(problem.head_dim)
    rc = lib().or_attention_partial(ctypes.byref(problem.c), s, i, h, j_begin, j_end,
                                    m.ctypes.data, l.ctypes.data, o.ctypes.data)
    _check(rc, "attention_partial")
    return float(m[0]), float(l[0]), o


def merge_partials(m, l, o) -> np.ndarray:
    m = np.ascontiguousarray(np.asarray(m, dtype=np.float64))
    l = np.ascontiguousarray(np.asarray(l, dtype=np.float64))
    o = np.ascontiguousarray(np.asarray(o, dtype=np.float64))
    out = np.zeros(o.shape[-1])
    rc = lib().or_merge_partials(m.ctypes.data, l.ctypes.data, o.ctypes.data,
                                 int(m.size), int(o.shape[-1]), out.ctypes.data)
    _check(rc, "merge_partials")
    return out


# ---------------------------------------------------------------- block copy (swap, fork, pack)
def validate_block_pairs(pairs) -> None:
    """Precondition of one copy call: destinations distinct, and no block is
    both written and read in the same call."""
    p = np.asarray(pairs).reshape(-1, 2)
    live = p[(p[:, 0] >= 0) & (p[:, 1] >= 0)]
    if np.unique(live[:, 1]).size != live.shape[0]:
        raise OracleError("duplicate destination blocks in one copy")


def copy_blocks(src_k, src_v, dst_k, dst_v, pairs) -> None:
    """Copies whole blocks src -> dst (pairs [n, 2] int32), in place on CPU pools."""
    for t in (src_k, src_v, dst_k, dst_v):
        if t.device.type != "cpu" or not t.is_contiguous():
            raise ValueError("pools must be contiguous CPU tensors")
    pairs = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
    validate_block_pairs(pairs)
    block_bytes = src_k[0].numel() * src_k.element_size()
    if dst_k[0].numel() * dst_k.element_size() != block_bytes:
        raise ValueError("source and destination blocks differ in size")
    rc = lib().or_copy_blocks(_ptr(src_k), _ptr(src_v), _ptr(dst_k), _ptr(dst_v), block_bytes,
                              int(src_k.shape[0]), int(dst_k.shape[0]), pairs.ctypes.data,
                              int(pairs.shape[0]))
    _check(rc, "copy_blocks")
