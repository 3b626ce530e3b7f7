"""Seeded synthetic inputs for the paged KV-cache hot path.

This module only draws inputs: sequence lengths, block tables over a shuffled
physical pool, and N(0, 1) values for queries, new keys/values and the cached
pool.  It holds none of the method's arithmetic (no slot computation, no cache
write, no attention).  The one host step it needs from the method -- how many
blocks a sequence of n tokens occupies -- is passed in by the caller as
``blocks_needed`` so that the CUDA side and the oracle side each use their own.

Workload shapes follow the pages' serving setup ("vLLM：颠覆大模型推理的高效API
服务引擎深度解析", §1.3 code and §3: LLaMA-2-7B heads, block size 16, up to 256
concurrent sequences, input 128 / output up to 256 tokens, power-law lengths)
and the five named configurations below.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Callable, Optional, Sequence

import numpy as np
import torch

BlocksNeeded = Callable[[int, int], int]


@dataclass
class Workload:
    name: str
    dtype: torch.dtype
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    max_blocks: int
    block_tables: torch.Tensor   # int32 [num_seqs, max_blocks], -1 = unused entry
    context_lens: torch.Tensor   # int32 [num_seqs]: tokens visible after this step's write
    seq_start: torch.Tensor      # int32 [num_seqs]: tokens already cached before this step
    cu_seqlens_q: torch.Tensor   # int32 [num_seqs + 1]: new-token (query) offsets
    q: torch.Tensor              # [total_q, num_heads, head_dim]
    key: torch.Tensor            # [total_q, num_kv_heads, head_dim] new keys
    value: torch.Tensor          # [total_q, num_kv_heads, head_dim] new values
    k_cache: torch.Tensor        # [num_blocks, block_size, num_kv_heads, head_dim]
    v_cache: torch.Tensor
    scale: float                 # fp32 value of 1/sqrt(head_dim)
    shared_prefix_seqs: int = 0
    shared_prefix_blocks: int = 0
    blocks_per_seq: list = field(default_factory=list)

    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.numel())

    @property
    def total_q(self) -> int:
        return int(self.q.shape[0])

    @property
    def q_lens(self) -> np.ndarray:
        cu = self.cu_seqlens_q.cpu().numpy()
        return cu[1:] - cu[:-1]

    @property
    def decode_only(self) -> bool:
        return bool(np.all(self.q_lens == 1))

    def to(self, device) -> "Workload":
        out = Workload(**{k: getattr(self, k) for k in self.__dataclass_fields__})
        for k in ("block_tables", "context_lens", "seq_start", "cu_seqlens_q", "q", "key",
                  "value", "k_cache", "v_cache"):
            setattr(out, k, getattr(self, k).to(device))
        return out


def fp32_scale(head_dim: int) -> float:
    """The fp32 value of 1/sqrt(head_dim), passed to both sides."""
    return float(np.float32(1.0) / np.sqrt(np.float32(head_dim)))


def _randn(shape, gen: torch.Generator, dtype: torch.dtype, device) -> torch.Tensor:
    """N(0, 1) drawn in fp32 chunk by chunk, rounded to `dtype` (RNE)."""
    n = int(np.prod(shape))
    out = torch.empty(n, dtype=dtype, device=device)
    chunk = 1 << 26
    for off in range(0, n, chunk):
        m = min(chunk, n - off)
        out[off:off + m] = torch.randn(m, generator=gen, device=device, dtype=torch.float32).to(dtype)
    return out.view(*shape)


def build(name: str, *, seed: int, blocks_needed: BlocksNeeded, dtype: torch.dtype,
          num_heads: int, num_kv_heads: int, head_dim: int, block_size: int,
          q_lens: Sequence[int], context_lens: Sequence[int],
          shared_prefix_seqs: int = 0, shared_prefix_tokens: int = 0,
          num_blocks: Optional[int] = None, pool_factor: float = 1.25,
          key_outlier_frac: float = 0.0, key_outlier_scale: float = 8.0,
          device="cpu") -> Workload:
    """Generic builder.  Sequences 0..shared_prefix_seqs-1 reference one set of
    physical prefix blocks read-only ("vLLM：颠覆…", §1.3 memory sharing)."""
    rng = np.random.default_rng(seed)
    q_lens = np.asarray(q_lens, dtype=np.int64)
    ctx = np.asarray(context_lens, dtype=np.int64)
    S = ctx.size
    assert q_lens.size == S and np.all(q_lens >= 0) and np.all(q_lens <= ctx) and np.all(ctx >= 1)
    nb = np.array([blocks_needed(int(c), block_size) for c in ctx], dtype=np.int64)
    pb = blocks_needed(shared_prefix_tokens, block_size) if shared_prefix_seqs else 0
    if shared_prefix_seqs:
        assert shared_prefix_tokens == pb * block_size, "shared prefix must be whole blocks"
        assert np.all(ctx[:shared_prefix_seqs] - q_lens[:shared_prefix_seqs] >= shared_prefix_tokens), \
            "new tokens must land after the shared prefix"
    private = nb.copy()
    private[:shared_prefix_seqs] -= pb
    used = int(pb + private.sum())
    if num_blocks is None:
        num_blocks = int(math.ceil(pool_factor * used))
    assert num_blocks >= used, "pool too small"
    perm = rng.permutation(num_blocks).astype(np.int32)
    max_blocks = int(nb.max())
    bt = np.full((S, max_blocks), -1, dtype=np.int32)
    prefix_ids = perm[:pb]
    cursor = pb
    for s in range(S):
        row = []
        if s < shared_prefix_seqs:
            row.extend(prefix_ids.tolist())
        row.extend(perm[cursor:cursor + private[s]].tolist())
        cursor += int(private[s])
        bt[s, :len(row)] = row
    cu = np.zeros(S + 1, dtype=np.int32)
    cu[1:] = np.cumsum(q_lens)
    total_q = int(cu[-1])

    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    q = _randn((total_q, num_heads, head_dim), gen, dtype, device)
    key = _randn((total_q, num_kv_heads, head_dim), gen, dtype, device)
    value = _randn((total_q, num_kv_heads, head_dim), gen, dtype, device)
    k_cache = _randn((num_blocks, block_size, num_kv_heads, head_dim), gen, dtype, device)
    v_cache = _randn((num_blocks, block_size, num_kv_heads, head_dim), gen, dtype, device)
    if key_outlier_frac > 0:
        # A fraction of cached token rows (every kv-head) and of new key rows is
        # scaled; x8 is exact in bf16.  The pool is a random permutation, so
        # picking physical rows is the same as picking logical positions.
        rows = k_cache.view(num_blocks * block_size, -1)
        mask = torch.rand(rows.shape[0], generator=gen, device=device) < key_outlier_frac
        rows[mask] = rows[mask] * key_outlier_scale
        krows = key.view(total_q, -1)
        kmask = torch.rand(total_q, generator=gen, device=device) < key_outlier_frac
        krows[kmask] = krows[kmask] * key_outlier_scale

    return Workload(
        name=name, dtype=dtype, num_heads=num_heads, num_kv_heads=num_kv_heads,
        head_dim=head_dim, block_size=block_size, num_blocks=num_blocks, max_blocks=max_blocks,
        block_tables=torch.from_numpy(bt).to(device),
        context_lens=torch.from_numpy(ctx.astype(np.int32)).to(device),
        seq_start=torch.from_numpy((ctx - q_lens).astype(np.int32)).to(device),
        cu_seqlens_q=torch.from_numpy(cu).to(device),
        q=q, key=key, value=value, k_cache=k_cache, v_cache=v_cache,
        scale=fp32_scale(head_dim), shared_prefix_seqs=int(shared_prefix_seqs),
        shared_prefix_blocks=int(pb), blocks_per_seq=nb.tolist())


def power_law_lengths(rng: np.random.Generator, n: int, exponent: float, lo: int, hi: int) -> np.ndarray:
    """Truncated continuous power law, pdf ~ x^-exponent on [lo, hi], by inverse CDF, floored."""
    a = 1.0 - exponent
    u = rng.random(n)
    x = (lo ** a + u * (hi ** a - lo ** a)) ** (1.0 / a)
    return np.clip(np.floor(x), lo, hi).astype(np.int64)


# ---------------------------------------------------------------- named configurations

def tiny(seed: int, blocks_needed: BlocksNeeded, device="cpu") -> Workload:
    """4 sequences, context {1, 16, 17, 50}, 4 heads / 4 kv-heads, head_dim 64, fp32,
    32-block pool, one decode token each."""
    return build("tiny_fp32", seed=seed, blocks_needed=blocks_needed, dtype=torch.float32,
                 num_heads=4, num_kv_heads=4, head_dim=64, block_size=16,
                 q_lens=[1, 1, 1, 1], context_lens=[1, 16, 17, 50], num_blocks=32, device=device)


def mha(seed: int, blocks_needed: BlocksNeeded, num_seqs: int = 64, ctx_lo: int = 128,
        ctx_hi: int = 384, block_size: int = 16, device="cpu") -> Workload:
    """LLaMA-2-7B-shaped MHA decode: 32 heads, head_dim 128, bf16, context U{lo..hi},
    pool 1.25x the used blocks."""
    rng = np.random.default_rng(seed + 1000)
    ctx = rng.integers(ctx_lo, ctx_hi + 1, size=num_seqs)
    name = "mha64_bf16" if num_seqs == 64 and ctx_hi == 384 else f"mha_{num_seqs}"
    return build(name if block_size == 16 else f"{name}_b{block_size}",
                 seed=seed, blocks_needed=blocks_needed, dtype=torch.bfloat16,
                 num_heads=32, num_kv_heads=32, head_dim=128, block_size=block_size,
                 q_lens=np.ones(num_seqs, dtype=np.int64), context_lens=ctx, device=device)


def gqa(seed: int, blocks_needed: BlocksNeeded, num_seqs: int = 256, ctx_lo: int = 16,
        ctx_hi: int = 4096, shared_seqs: int = 64, prefix_tokens: int = 1024,
        block_size: int = 16, device="cpu") -> Workload:
    """GQA decode at max_num_seqs: 32 q-heads / 8 kv-heads, head_dim 128, bf16, context
    power law x^-1.2 on [lo, hi]; sequences 0..shared_seqs-1 share a prefix_tokens
    system prompt (context = min(prefix + draw, hi))."""
    rng = np.random.default_rng(seed + 2000)
    ctx = power_law_lengths(rng, num_seqs, 1.2, ctx_lo, ctx_hi)
    ctx[:shared_seqs] = np.minimum(prefix_tokens + ctx[:shared_seqs], ctx_hi)
    name = "gqa256_bf16" if (num_seqs, ctx_hi, shared_seqs) == (256, 4096, 64) else f"gqa_{num_seqs}"
    return build(name if block_size == 16 else f"{name}_b{block_size}",
                 seed=seed, blocks_needed=blocks_needed, dtype=torch.bfloat16,
                 num_heads=32, num_kv_heads=8, head_dim=128, block_size=block_size,
                 q_lens=np.ones(num_seqs, dtype=np.int64), context_lens=ctx,
                 shared_prefix_seqs=shared_seqs, shared_prefix_tokens=prefix_tokens, device=device)


def mixed(seed: int, blocks_needed: BlocksNeeded, num_prefill: int = 8, chunk: int = 512,
          prefix_hi: int = 2048, num_decode: int = 248, dec_lo: int = 128, dec_hi: int = 2048,
          block_size: int = 16, device="cpu") -> Workload:
    """Mixed continuous-batching step: num_prefill chunks of `chunk` new tokens over
    U{0..prefix_hi} cached tokens plus num_decode decode rows with context U{lo..hi};
    the requests appear in a random order inside one super-sequence."""
    rng = np.random.default_rng(seed + 3000)
    prefixes = rng.integers(0, prefix_hi + 1, size=num_prefill)
    dec_ctx = rng.integers(dec_lo, dec_hi + 1, size=num_decode)
    q_lens = np.concatenate([np.full(num_prefill, chunk), np.ones(num_decode, dtype=np.int64)])
    ctx = np.concatenate([prefixes + chunk, dec_ctx])
    order = rng.permutation(q_lens.size)
    name = "mixed_bf16" if (num_prefill, chunk, num_decode) == (8, 512, 248) else f"mixed_{num_prefill}x{chunk}"
    return build(name if block_size == 16 else f"{name}_b{block_size}",
                 seed=seed, blocks_needed=blocks_needed, dtype=torch.bfloat16,
                 num_heads=32, num_kv_heads=8, head_dim=128, block_size=block_size,
                 q_lens=q_lens[order], context_lens=ctx[order], device=device)


def long(seed: int, blocks_needed: BlocksNeeded, num_seqs: int = 16, ctx: int = 32768,
         num_blocks: Optional[int] = None, block_size: int = 16, device="cpu") -> Workload:
    """Long-context split-KV decode: 16 x 32768 context, 32/8 heads, head_dim 128,
    bf16, 36,864-block pool (the same tokens at other block sizes), 1% of key
    rows scaled x8."""
    if num_blocks is None:
        num_blocks = 36864 * 16 // block_size
    name = "long_bf16" if (num_seqs, ctx) == (16, 32768) else f"long_{num_seqs}x{ctx}"
    return build(name if block_size == 16 else f"{name}_b{block_size}",
                 seed=seed, blocks_needed=blocks_needed, dtype=torch.bfloat16,
                 num_heads=32, num_kv_heads=8, head_dim=128, block_size=block_size,
                 q_lens=np.ones(num_seqs, dtype=np.int64), context_lens=np.full(num_seqs, ctx),
                 num_blocks=num_blocks, key_outlier_frac=0.01, device=device)


FULL_CONFIGS = {
    "tiny_fp32": tiny,
    "mha64_bf16": mha,
    "gqa256_bf16": gqa,
    "mixed_bf16": mixed,
    "long_bf16": long,
}


def long_single(seed: int, blocks_needed: BlocksNeeded, device="cpu") -> Workload:
    """One 131,072-token sequence (8,192 blocks; every decode CTA takes a slice
    of it), otherwise as the long-context configuration."""
    return long(seed, blocks_needed, num_seqs=1, ctx=131072, num_blocks=10240, device=device)


def prefill_chunks(seed: int, blocks_needed: BlocksNeeded, num_seqs: int = 8, chunk: int = 512,
                   cached: int = 2048, block_size: int = 16, device="cpu") -> Workload:
    """Prefill alone: num_seqs chunks of `chunk` new tokens, each over `cached`
    already-cached tokens (the mixed step's chunk shape at its longest prefix),
    32/8 heads, head_dim 128, bf16."""
    return build(f"prefill{num_seqs}x{chunk}_bf16", seed=seed, blocks_needed=blocks_needed,
                 dtype=torch.bfloat16, num_heads=32, num_kv_heads=8, head_dim=128, block_size=block_size,
                 q_lens=np.full(num_seqs, chunk), context_lens=np.full(num_seqs, cached + chunk),
                 device=device)


# shapes measured beside the five configurations above (not among them)
EXTRA_CONFIGS = {
    "long1x131k_bf16": long_single,
    "prefill8x512_bf16": prefill_chunks,
}


def make(name: str, seed: int, blocks_needed: BlocksNeeded, device="cpu") -> Workload:
    fn = FULL_CONFIGS.get(name) or EXTRA_CONFIGS[name]
    return fn(seed, blocks_needed, device=device)
