"""Shared test helpers: run one hot-path step on the GPU through the C ABI, run
the same step in the oracle on CPU copies, and compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from pagedattention_kv_cache_reshape_gb300 import pa
from pagedattention_kv_cache_reshape_gb300 import workloads as W

# Tolerances stated for this path: fp32 inputs max |err| <= 1e-5; bf16 inputs
# max |err| <= 2e-2 and relative RMS <= 1e-2 (fp32 accumulation).
TOL = {torch.float32: dict(max_abs=1e-5, rel_rms=None),
       torch.bfloat16: dict(max_abs=2e-2, rel_rms=1e-2)}


def oracle_blocks(n, B):
    return oracle.num_blocks_needed(n, B)


def gpu_step(w: W.Workload, dev_status=None, out=None, workspace=None):
    """slot mapping -> cache write -> attention, all on the device.  Mutates the
    workload's device pools.  Returns (slots, out)."""
    slots = pa.compute_slot_mapping(w.block_tables, w.seq_start, w.cu_seqlens_q, w.num_blocks,
                                    w.total_q, block_size=w.block_size, dev_status=dev_status)
    pa.reshape_and_cache(w.key, w.value, w.k_cache, w.v_cache, slots, dev_status=dev_status)
    if w.decode_only:
        out = pa.decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale,
                        out=out, workspace=workspace, dev_status=dev_status)
    else:
        out = pa.varlen_prefill(w.q, w.cu_seqlens_q, w.k_cache, w.v_cache, w.block_tables,
                                w.context_lens, w.scale, int(w.q_lens.max()), out=out,
                                workspace=workspace, dev_status=dev_status)
    return slots, out


def oracle_write(w_cpu: W.Workload):
    """Oracle slot mapping + cache write on CPU copies (in place on w_cpu's pools)."""
    slots = oracle.slot_mapping(w_cpu.block_tables, w_cpu.seq_start, w_cpu.cu_seqlens_q,
                                w_cpu.block_size, w_cpu.num_blocks)
    oracle.reshape_and_cache(w_cpu.key, w_cpu.value, w_cpu.k_cache, w_cpu.v_cache, slots,
                             w_cpu.block_size)
    return slots


def oracle_attention(w_cpu: W.Workload, nthreads=None, causal=True):
    nthreads = nthreads or max(1, oracle.max_threads())
    return oracle.paged_attention(w_cpu.q, w_cpu.k_cache, w_cpu.v_cache, w_cpu.block_tables,
                                  w_cpu.context_lens, w_cpu.scale,
                                  cu_seqlens_q=None if w_cpu.decode_only else w_cpu.cu_seqlens_q,
                                  nthreads=nthreads, causal=causal)


def oracle_rows(w_cpu: W.Workload, rows, heads, nthreads=None):
    nthreads = nthreads or max(1, oracle.max_threads())
    return oracle.paged_attention_rows(w_cpu.q, w_cpu.k_cache, w_cpu.v_cache, w_cpu.block_tables,
                                       w_cpu.context_lens, w_cpu.scale, rows, heads,
                                       cu_seqlens_q=None if w_cpu.decode_only else w_cpu.cu_seqlens_q,
                                       nthreads=nthreads)


def compare(got: np.ndarray, ref: np.ndarray, dtype: torch.dtype, what: str = ""):
    tol = TOL[dtype]
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    max_abs = float(err.max()) if err.size else 0.0
    assert max_abs <= tol["max_abs"], f"{what}: max |err| {max_abs:.3e} > {tol['max_abs']}"
    if tol["rel_rms"] is not None and ref.size:
        rel = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))
        assert rel <= tol["rel_rms"], f"{what}: relative RMS {rel:.3e} > {tol['rel_rms']}"
    return max_abs


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().double().numpy()
