"""The seeded input generator: determinism, shapes and the structure of each workload."""
import numpy as np
import torch

import oracle
from pagedattention_kv_cache_reshape_gb300 import workloads as W

NB = oracle.num_blocks_needed


def test_deterministic_for_a_seed():
    a = W.gqa(3, NB, num_seqs=12, ctx_hi=300, shared_seqs=3, prefix_tokens=64)
    b = W.gqa(3, NB, num_seqs=12, ctx_hi=300, shared_seqs=3, prefix_tokens=64)
    for k in ("block_tables", "context_lens", "q", "key", "value", "k_cache", "v_cache"):
        assert torch.equal(getattr(a, k), getattr(b, k)), k
    c = W.gqa(4, NB, num_seqs=12, ctx_hi=300, shared_seqs=3, prefix_tokens=64)
    assert not torch.equal(a.q, c.q)


def test_tiny_config_shape():
    w = W.tiny(0, NB)
    assert w.context_lens.tolist() == [1, 16, 17, 50]
    assert w.num_blocks == 32 and w.dtype == torch.float32
    assert w.q.shape == (4, 4, 64) and w.key.shape == (4, 4, 64)
    assert w.k_cache.shape == (32, 16, 4, 64)
    assert w.blocks_per_seq == [1, 1, 2, 4]
    live = w.block_tables[w.block_tables >= 0]
    assert live.numel() == 8 and live.unique().numel() == 8
    assert w.seq_start.tolist() == [0, 15, 16, 49]
    assert abs(w.scale - 0.125) < 1e-9


def test_shared_prefix_structure():
    w = W.gqa(0, NB, num_seqs=20, ctx_hi=500, shared_seqs=5, prefix_tokens=128)
    bt = w.block_tables
    pb = 128 // 16
    for s in range(1, 5):
        assert torch.equal(bt[s, :pb], bt[0, :pb])
    # private blocks are never shared
    live = torch.cat([bt[s, (pb if s < 5 else 0):w.blocks_per_seq[s]] for s in range(20)])
    assert live.unique().numel() == live.numel()
    assert not set(live.tolist()) & set(bt[0, :pb].tolist())
    assert (w.context_lens[:5] >= 128 + 16).all()


def test_power_law_lengths_statistics():
    rng = np.random.default_rng(0)
    x = W.power_law_lengths(rng, 200000, 1.2, 16, 4096)
    assert x.min() >= 16 and x.max() <= 4096
    assert 110 <= np.median(x) <= 135         # analytic median ~123
    assert 460 <= x.mean() <= 540             # analytic mean ~498


def test_mixed_config_structure():
    w = W.mixed(0, NB, num_prefill=3, chunk=40, prefix_hi=70, num_decode=9, dec_lo=5, dec_hi=60)
    ql = w.q_lens
    assert sorted(ql.tolist()) == [1] * 9 + [40] * 3
    assert w.total_q == 3 * 40 + 9
    assert (w.seq_start.numpy() == w.context_lens.numpy() - ql).all()


def test_long_config_outliers_are_exact_multiples():
    w = W.long(0, NB, num_seqs=2, ctx=256, num_blocks=40)
    rows = w.k_cache.view(-1, w.num_kv_heads * w.head_dim).float()
    big = rows.abs().amax(1) > 7.0
    assert big.any()
    # scaled rows are x8 of an N(0,1) bf16 row: dividing by 8 is exact in bf16
    scaled = rows[big] / 8
    assert torch.equal(scaled.to(torch.bfloat16).float(), scaled)


def test_prefill_chunks_config_structure():
    # 3 chunks of 40 new tokens over 70 cached ones: every row a prefill row,
    # each sequence's new tokens at the end of its context
    w = W.prefill_chunks(0, NB, num_seqs=3, chunk=40, cached=70)
    assert w.q_lens.tolist() == [40, 40, 40]
    assert w.context_lens.tolist() == [110, 110, 110]
    assert not w.decode_only and w.total_q == 120
    assert (w.seq_start.numpy() == 70).all()
    assert w.num_heads == 32 and w.num_kv_heads == 8 and w.head_dim == 128 and w.dtype == torch.bfloat16
    assert w.blocks_per_seq == [NB(110, 16)] * 3
    assert "prefill8x512_bf16" in W.EXTRA_CONFIGS
