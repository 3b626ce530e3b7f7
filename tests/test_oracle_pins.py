"""Pins for the CPU fp64 oracle, against what the pages and the mathematics fix.

Nothing here retypes the oracle's formulas.  The pins are:
  * worked examples printed on the pages (tests/golden/*.txt, each cited);
  * the pool's own tensor indexing ([num_blocks, block_size, kv_heads, head_dim]);
  * closed forms of softmax attention;
  * torch's fp64 scaled_dot_product_attention on dense (unpaged) tensors;
  * invariants: block permutation, shared prefix, batch order, prefill/decode;
  * the algebraic split/merge identity;
  * input validation.
"""
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from pagedattention_kv_cache_reshape_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([int(x) for x in line.split()])
    return rows


def _nan_pool(num_blocks, B, hkv, d, dtype=torch.float64):
    return torch.full((num_blocks, B, hkv, d), float("nan"), dtype=dtype)


def _marker_rows(n, hkv, d, dtype=torch.float32):
    """Token t's row is filled with the value t + 1 (distinct, exact in fp32/bf16)."""
    return (torch.arange(1, n + 1, dtype=torch.float32).view(n, 1, 1).expand(n, hkv, d)
            .contiguous().to(dtype))


def _write_sequence(bt_row, seq_start, n_new, B, num_blocks, hkv=1, d=8, pool=None, dtype=torch.float32):
    """Write n_new marker tokens at positions seq_start.. via the oracle."""
    bt = torch.tensor([bt_row], dtype=torch.int32)
    slots = oracle.slot_mapping(bt, torch.tensor([seq_start], dtype=torch.int32),
                                torch.tensor([0, n_new], dtype=torch.int32), B, num_blocks)
    if pool is None:
        pool = torch.full((num_blocks, B, hkv, d), float("nan"), dtype=dtype)
    vpool = pool.clone()
    rows = _marker_rows(n_new, hkv, d, dtype) + seq_start
    oracle.reshape_and_cache(rows, rows, pool, vpool, slots, B)
    return slots, pool


# ------------------------------------------------------------------ a1

def test_block_count_golden():
    for n, B, expect in _golden("block_count.txt"):
        assert oracle.num_blocks_needed(n, B) == expect


def test_block_count_is_least_cover():
    # ceil(n/B) is the least k with k*B >= n.
    for B in range(1, 41):
        for n in range(0, 300):
            k = oracle.num_blocks_needed(n, B)
            assert k * B >= n and (k == 0 or (k - 1) * B < n)
    assert oracle.num_blocks_needed(5, 0) == -1
    assert oracle.num_blocks_needed(-1, 16) == -1


# ------------------------------------------------------------------ a2 / a3 against the pages

def test_17_token_prefill_spans_two_blocks():
    """17 new tokens at block size 16: 16 fill one physical block, the 17th opens
    the next one at offset 0 (allocate_slots example)."""
    (n, B, nblk), = _golden("block_count.txt")
    bt_row = [5, 2]  # any two physical blocks
    slots, pool = _write_sequence(bt_row, 0, n, B, num_blocks=8)
    assert len(set(slots.tolist())) == n
    # read back through the pool tensor's own indexing
    assert torch.equal(pool[5, :, 0, 0], torch.arange(1, 17, dtype=torch.float32))
    assert pool[2, 0, 0, 0].item() == 17.0
    assert torch.isnan(pool[2, 1:]).all()
    untouched = [b for b in range(8) if b not in bt_row]
    assert torch.isnan(pool[untouched]).all()


@pytest.mark.parametrize("B", [8, 32])
def test_prefill_lands_block_by_block_at_other_block_sizes(B):
    """The same 17-token prefill at block size B (a setting of the engine):
    token t lands at offset t % B of the table's block t // B, read back through
    the pool's own indexing, and ceil(17 / B) blocks are touched."""
    (n, _, _), = _golden("block_count.txt")
    nb = oracle.num_blocks_needed(n, B)
    assert nb == -(-n // B)
    bt_row = [7, 2, 5][:nb]
    slots, pool = _write_sequence(bt_row, 0, n, B, num_blocks=8)
    for t in range(n):
        assert pool[bt_row[t // B], t % B, 0, 0].item() == t + 1
    written = (~torch.isnan(pool[:, :, 0, 0])).sum().item()
    assert written == n
    untouched = [b for b in range(8) if b not in bt_row]
    assert torch.isnan(pool[untouched]).all()


@pytest.mark.parametrize("B", [8, 32])
def test_block_table_fill_at_other_block_sizes(B):
    """The 24 tokens of the fill example at block size B fill min(B, 24 - iB)
    tokens of logical block i, and the next token lands at logical block 24 // B,
    offset 24 % B."""
    n = sum(f for _, f in _golden("block_table_fill.txt"))
    nb = oracle.num_blocks_needed(n + 1, B)
    bt_row = [6, 1, 3, 4][:nb]
    slots, pool = _write_sequence(bt_row, 0, n, B, num_blocks=8)
    for logical, phys in enumerate(bt_row):
        written = (~torch.isnan(pool[phys, :, 0, 0])).sum().item()
        assert written == max(0, min(B, n - logical * B))
    _, pool = _write_sequence(bt_row, n, 1, B, num_blocks=8, pool=pool)
    assert pool[bt_row[n // B], n % B, 0, 0].item() == n + 1


def test_block_table_fill_example():
    """A request with 24 tokens over three blocks has fill counts 16 / 8 / 0, and
    its next token lands in logical block 1 at offset 8."""
    fills = [f for _, f in _golden("block_table_fill.txt")]
    B = 16
    n = sum(fills)
    bt_row = [6, 1, 3]
    slots, pool = _write_sequence(bt_row, 0, n, B, num_blocks=8)
    for logical, fill in enumerate(fills):
        phys = bt_row[logical]
        written = (~torch.isnan(pool[phys, :, 0, 0])).sum().item()
        assert written == fill
        if fill:
            assert not torch.isnan(pool[phys, :fill]).any()
    # decode the next token (position 24 = seq_start)
    slots2, pool = _write_sequence(bt_row, n, 1, B, num_blocks=8, pool=pool)
    assert pool[bt_row[1], 8, 0, 0].item() == n + 1
    assert torch.isnan(pool[bt_row[1], 9:]).all()
    assert torch.isnan(pool[bt_row[2]]).all()


@pytest.mark.parametrize("B", [8, 16, 32])
def test_slot_mapping_injective_and_in_pool(B):
    rng = np.random.default_rng(7)
    num_blocks = 64 * 16 // B + 8
    perm = rng.permutation(num_blocks).astype(np.int32)
    ctx = np.array([1, 15, 16, 17, 33, 100, 48])
    qlen = np.array([1, 15, 3, 17, 1, 36, 16])
    nb = [oracle.num_blocks_needed(int(c), B) for c in ctx]
    bt = np.full((len(ctx), max(nb)), -1, np.int32)
    cur = 0
    for s, k in enumerate(nb):
        bt[s, :k] = perm[cur:cur + k]
        cur += k
    cu = np.concatenate([[0], np.cumsum(qlen)]).astype(np.int32)
    slots = oracle.slot_mapping(torch.from_numpy(bt), torch.from_numpy((ctx - qlen).astype(np.int32)),
                                torch.from_numpy(cu), B, num_blocks)
    assert slots.size == qlen.sum()
    assert np.unique(slots).size == slots.size
    assert slots.min() >= 0 and slots.max() < num_blocks * B
    # each sequence's tokens land only in that sequence's blocks: write the
    # token index + 1 as a marker, then look it up through the pool's indexing
    pool = torch.full((num_blocks, B, 1, 1), float("nan"), dtype=torch.float32)
    marks = torch.arange(1, slots.size + 1, dtype=torch.float32).view(-1, 1, 1)
    oracle.reshape_and_cache(marks, marks, pool, pool.clone(), slots, B)
    where = {}
    for b, o in torch.nonzero(~torch.isnan(pool[:, :, 0, 0])).tolist():
        where[int(pool[b, o, 0, 0].item()) - 1] = b
    assert len(where) == slots.size
    for s in range(len(ctx)):
        blocks = {where[t] for t in range(cu[s], cu[s + 1])}
        assert blocks <= set(bt[s, :nb[s]].tolist())


def test_slot_mapping_rejects_out_of_range():
    bt = torch.tensor([[3, 99]], dtype=torch.int32)   # 99 is outside an 8-block pool
    with pytest.raises(oracle.OracleError):
        oracle.slot_mapping(bt, torch.tensor([10], dtype=torch.int32),
                            torch.tensor([0, 10], dtype=torch.int32), 16, 8)
    bt = torch.tensor([[3]], dtype=torch.int32)       # position 16 needs a 2nd table entry
    with pytest.raises(oracle.OracleError):
        oracle.slot_mapping(bt, torch.tensor([16], dtype=torch.int32),
                            torch.tensor([0, 1], dtype=torch.int32), 16, 8)


def test_cache_write_skips_negative_and_leaves_rest():
    B, nblk, hkv, d = 16, 4, 2, 8
    pool = torch.randn(nblk, B, hkv, d)
    before = pool.clone()
    vpool = torch.randn(nblk, B, hkv, d)
    vbefore = vpool.clone()
    key = torch.randn(3, hkv, d)
    val = torch.randn(3, hkv, d)
    slots = np.array([5, -1, 2 * B + 15], dtype=np.int64)
    oracle.reshape_and_cache(key, val, pool, vpool, slots, B)
    assert torch.equal(pool[0, 5], key[0]) and torch.equal(vpool[0, 5], val[0])
    assert torch.equal(pool[2, 15], key[2]) and torch.equal(vpool[2, 15], val[2])
    changed = (pool != before).flatten(2).any(-1)
    assert changed.sum().item() == 2
    assert (vpool != vbefore).flatten(2).any(-1).sum().item() == 2
    with pytest.raises(oracle.OracleError):
        oracle.reshape_and_cache(key, val, pool, vpool, np.array([1, 1, 2]), B)   # duplicates
    with pytest.raises(oracle.OracleError):
        oracle.reshape_and_cache(key, val, pool, vpool, np.array([1, 2, nblk * B]), B)


def test_cache_write_bf16_bit_copy_and_token_stride():
    B, nblk, hkv, d = 16, 4, 2, 8
    qkv = torch.randn(5, 3, hkv, d).to(torch.bfloat16)   # fused [tok, (q,k,v), hkv, d]
    key = qkv[:, 1]
    val = qkv[:, 2]
    pool = torch.zeros(nblk, B, hkv, d, dtype=torch.bfloat16)
    vpool = torch.zeros_like(pool)
    slots = np.array([0, 17, 34, 51, 63], dtype=np.int64)
    oracle.reshape_and_cache(key, val, pool, vpool, slots, B)
    for t, s in enumerate(slots):
        assert torch.equal(pool[s // B, s % B].view(torch.int16), key[t].view(torch.int16))
        assert torch.equal(vpool[s // B, s % B].view(torch.int16), val[t].view(torch.int16))


# ------------------------------------------------------------------ attention helpers

def _dense_problem(seed, ctx_list, q_lens, H, Hkv, D, B=16, dtype=torch.float64, extra_blocks=3):
    """Dense per-sequence K/V; paged into a NaN pool through the oracle's own
    slot mapping and cache write (prefill of the whole sequence)."""
    g = torch.Generator().manual_seed(seed)
    S = len(ctx_list)
    store = torch.float32 if dtype == torch.float64 else dtype
    Ks = [torch.randn(c, Hkv, D, generator=g).to(store) for c in ctx_list]
    Vs = [torch.randn(c, Hkv, D, generator=g).to(store) for c in ctx_list]
    nb = [oracle.num_blocks_needed(c, B) for c in ctx_list]
    num_blocks = sum(nb) + extra_blocks
    perm = torch.randperm(num_blocks, generator=g).to(torch.int32)
    bt = torch.full((S, max(nb)), -1, dtype=torch.int32)
    cur = 0
    for s, k in enumerate(nb):
        bt[s, :k] = perm[cur:cur + k]
        cur += k
    kpool = torch.full((num_blocks, B, Hkv, D), float("nan"), dtype=store)
    vpool = kpool.clone()
    ctx_t = torch.tensor(ctx_list, dtype=torch.int32)
    cu_all = torch.zeros(S + 1, dtype=torch.int32)
    cu_all[1:] = torch.cumsum(ctx_t, 0)
    slots = oracle.slot_mapping(bt, torch.zeros(S, dtype=torch.int32), cu_all, B, num_blocks)
    oracle.reshape_and_cache(torch.cat(Ks), torch.cat(Vs), kpool, vpool, slots, B)
    qlen_t = torch.tensor(q_lens, dtype=torch.int32)
    cu = torch.zeros(S + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(qlen_t, 0)
    q = torch.randn(int(cu[-1]), H, D, generator=g).to(store)
    return dict(q=q, kpool=kpool, vpool=vpool, bt=bt, ctx=ctx_t, cu=cu, Ks=Ks, Vs=Vs,
                scale=W.fp32_scale(D), H=H, Hkv=Hkv, D=D, B=B)


def _sdpa_reference(P, causal=True):
    """torch fp64 SDPA per sequence on the dense K/V, bottom-right causal, GQA by repeat."""
    H, Hkv = P["H"], P["Hkv"]
    outs = []
    for s in range(len(P["Ks"])):
        c = int(P["ctx"][s])
        a, b = int(P["cu"][s]), int(P["cu"][s + 1])
        ql = b - a
        q = P["q"][a:b].double().permute(1, 0, 2).unsqueeze(0)               # [1,H,ql,D]
        k = P["Ks"][s].double().repeat_interleave(H // Hkv, dim=1).permute(1, 0, 2).unsqueeze(0)
        v = P["Vs"][s].double().repeat_interleave(H // Hkv, dim=1).permute(1, 0, 2).unsqueeze(0)
        i = torch.arange(ql).view(-1, 1)
        j = torch.arange(c).view(1, -1)
        mask = j <= (c - ql + i)
        if causal:
            o = F.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=P["scale"])
        else:
            o = F.scaled_dot_product_attention(q, k, v, scale=P["scale"])
        outs.append(o[0].permute(1, 0, 2))
    return torch.cat(outs).numpy()


def _oracle_out(P, nthreads=2):
    return oracle.paged_attention(P["q"], P["kpool"], P["vpool"], P["bt"], P["ctx"], P["scale"],
                                  cu_seqlens_q=P["cu"], nthreads=nthreads)


# ------------------------------------------------------------------ a4 / a6 pins

@pytest.mark.parametrize("H,Hkv,D,B", [(4, 4, 64, 16), (8, 2, 32, 16), (6, 1, 16, 16), (32, 8, 128, 16),
                                       (8, 2, 32, 8), (8, 2, 32, 32), (32, 8, 128, 8), (32, 8, 128, 32)])
def test_decode_matches_fp64_sdpa(H, Hkv, D, B):
    ctx = [1, 16, 17, 50, 3, 64, 8, 9, 32, 33]
    P = _dense_problem(11, ctx, [1] * len(ctx), H, Hkv, D, B=B)
    np.testing.assert_allclose(_oracle_out(P), _sdpa_reference(P), rtol=0, atol=1e-12)


def test_decode_without_cu_seqlens_equals_one_row_each():
    ctx = [5, 40, 16]
    P = _dense_problem(3, ctx, [1, 1, 1], 4, 2, 32)
    a = _oracle_out(P)
    b = oracle.paged_attention(P["q"], P["kpool"], P["vpool"], P["bt"], P["ctx"], P["scale"])
    assert np.array_equal(a, b)


@pytest.mark.parametrize("B", [8, 16, 32])
def test_causal_prefill_matches_fp64_sdpa(B):
    # chunks over cached prefixes that do not start on a block boundary,
    # full prompts, and decode rows mixed in one super-sequence
    ctx = [40, 17, 1, 90, 33]
    qlen = [40, 5, 1, 37, 1]
    P = _dense_problem(5, ctx, qlen, 8, 2, 64, B=B)
    np.testing.assert_allclose(_oracle_out(P), _sdpa_reference(P), rtol=0, atol=1e-12)


def test_encode_only_matches_unmasked_fp64_sdpa():
    # whole prompts (the embedding workload) and chunks over a cached prefix
    ctx = [40, 17, 1, 90, 33]
    qlen = [40, 17, 1, 37, 2]
    P = _dense_problem(6, ctx, qlen, 8, 2, 64)
    out = oracle.paged_attention(P["q"], P["kpool"], P["vpool"], P["bt"], P["ctx"], P["scale"],
                                 cu_seqlens_q=P["cu"], causal=False)
    np.testing.assert_allclose(out, _sdpa_reference(P, causal=False), rtol=0, atol=1e-12)
    # every row of a sequence sees the same keys: equal queries give equal rows
    P["q"][1] = P["q"][0]
    out = oracle.paged_attention(P["q"], P["kpool"], P["vpool"], P["bt"], P["ctx"], P["scale"],
                                 cu_seqlens_q=P["cu"], causal=False)
    assert np.array_equal(out[0], out[1])
    # the last row of each sequence is the same in both modes
    causal = _oracle_out(P)
    for s in range(len(ctx)):
        r = int(P["cu"][s + 1]) - 1
        assert np.array_equal(out[r], causal[r])


@pytest.mark.parametrize("B", [8, 16, 32])
def test_closed_form_single_key_returns_value(B):
    P = _dense_problem(21, [1, 1], [1, 1], 4, 4, 16, B=B)
    o = _oracle_out(P)
    for s in range(2):
        assert np.array_equal(o[s], P["Vs"][s][0].double().numpy())


@pytest.mark.parametrize("B", [8, 16, 32])
def test_closed_form_equal_logits_give_mean_value(B):
    P = _dense_problem(22, [37, 5], [1, 1], 4, 2, 16, B=B)
    P["q"].zero_()                                   # every logit 0
    o = _oracle_out(P)
    for s in range(2):
        mean = P["Vs"][s].double().mean(0).repeat_interleave(2, dim=0).numpy()
        np.testing.assert_allclose(o[s], mean, rtol=0, atol=1e-13)


def test_closed_form_constant_value_rows():
    P = _dense_problem(23, [29], [1], 4, 1, 16)
    # every live value row becomes 0.75; dead slots stay NaN
    P["vpool"] = torch.where(torch.isnan(P["kpool"]), P["vpool"], torch.full_like(P["vpool"], 0.75))
    o = _oracle_out(P)
    np.testing.assert_allclose(o, 0.75, rtol=0, atol=1e-15)


def test_closed_form_dominant_key():
    P = _dense_problem(24, [30], [1], 2, 1, 16)
    # make key 7 align with both queries and be huge
    j = 7
    qdir = P["q"][0, 0].clone()
    P["q"][0, 1] = qdir
    # find key 7 in the pool: it holds the dense value Ks[0][7]
    target = P["Ks"][0][j]
    hits = (P["kpool"] == target).all(-1).all(-1)
    (b, o_), = torch.nonzero(hits).tolist()
    P["kpool"][b, o_, 0] = qdir * 50.0
    out = _oracle_out(P)
    v7 = P["Vs"][0][j][0].double().numpy()
    np.testing.assert_allclose(out[0, 0], v7, rtol=0, atol=1e-9)
    np.testing.assert_allclose(out[0, 1], v7, rtol=0, atol=1e-9)


@pytest.mark.parametrize("B", [8, 16, 32])
def test_block_permutation_invariance(B):
    P = _dense_problem(31, [50, 16, 77, 3], [1, 1, 4, 1], 8, 2, 32, B=B, extra_blocks=6)
    base = _oracle_out(P)
    nblk = P["kpool"].shape[0]
    perm = torch.randperm(nblk, generator=torch.Generator().manual_seed(9))
    kp = torch.empty_like(P["kpool"])
    vp = torch.empty_like(P["vpool"])
    kp[perm] = P["kpool"]
    vp[perm] = P["vpool"]
    bt = P["bt"].clone()
    live = bt >= 0
    bt[live] = perm[bt[live].long()].to(torch.int32)
    out = oracle.paged_attention(P["q"], kp, vp, bt, P["ctx"], P["scale"], cu_seqlens_q=P["cu"])
    assert np.array_equal(out, base)


def test_shared_prefix_blocks_read_only_identical_outputs():
    B, H, Hkv, D = 16, 4, 2, 16
    P = _dense_problem(41, [48, 48], [1, 1], H, Hkv, D)
    # sequence 1 references sequence 0's first two blocks (32-token shared prefix),
    # keeps a private third block whose contents equal sequence 0's third block
    bt = P["bt"].clone()
    bt[1, :2] = bt[0, :2]
    P["kpool"][bt[1, 2]] = P["kpool"][bt[0, 2]]
    P["vpool"][bt[1, 2]] = P["vpool"][bt[0, 2]]
    P["q"][1] = P["q"][0]
    P["bt"] = bt
    kbefore, vbefore = P["kpool"].clone(), P["vpool"].clone()
    out = _oracle_out(P)
    assert np.array_equal(out[0], out[1])
    assert torch.equal(kbefore.nan_to_num(7.0), P["kpool"].nan_to_num(7.0))
    assert torch.equal(vbefore.nan_to_num(7.0), P["vpool"].nan_to_num(7.0))


def test_batch_order_independence():
    P = _dense_problem(51, [20, 65, 9, 33], [3, 1, 9, 2], 4, 2, 16)
    base = _oracle_out(P)
    order = [2, 0, 3, 1]
    cu = P["cu"]
    rows = torch.cat([torch.arange(int(cu[s]), int(cu[s + 1])) for s in order])
    qlen = [int(cu[s + 1] - cu[s]) for s in order]
    ncu = torch.zeros(len(order) + 1, dtype=torch.int32)
    ncu[1:] = torch.cumsum(torch.tensor(qlen), 0)
    out = oracle.paged_attention(P["q"][rows], P["kpool"], P["vpool"], P["bt"][order],
                                 P["ctx"][order], P["scale"], cu_seqlens_q=ncu)
    assert np.array_equal(out, base[rows.numpy()])


@pytest.mark.parametrize("B", [8, 16, 32])
def test_prefill_row_equals_decode_at_that_position(B):
    n = 45
    P = _dense_problem(61, [n], [n], 4, 2, 32, B=B)
    pre = _oracle_out(P)
    for i in [0, 1, 15, 16, 17, 31, 44]:
        dec = oracle.paged_attention(P["q"][i:i + 1], P["kpool"], P["vpool"], P["bt"],
                                     torch.tensor([i + 1], dtype=torch.int32), P["scale"])
        assert np.array_equal(dec[0], pre[i])


def test_sampled_rows_equal_full_output():
    P = _dense_problem(71, [40, 9, 70], [4, 1, 6], 8, 4, 32)
    full = _oracle_out(P)
    rows = [0, 3, 4, 5, 10, 7]
    heads = [0, 7, 3, 5, 1, 2]
    sel = oracle.paged_attention_rows(P["q"], P["kpool"], P["vpool"], P["bt"], P["ctx"], P["scale"],
                                      rows, heads, cu_seqlens_q=P["cu"])
    for k, (r, h) in enumerate(zip(rows, heads)):
        assert np.array_equal(sel[k], full[r, h])


def test_bf16_inputs_widen_exactly():
    P = _dense_problem(81, [33, 7], [1, 1], 4, 2, 32, dtype=torch.bfloat16)
    out = _oracle_out(P)
    ref = _sdpa_reference(P)   # SDPA on the same bf16 values widened to fp64
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


def test_attention_rejects_bad_inputs():
    P = _dense_problem(91, [20], [1], 4, 2, 16)
    with pytest.raises(oracle.OracleError):
        oracle.paged_attention(P["q"], P["kpool"], P["vpool"], P["bt"],
                               torch.tensor([0], dtype=torch.int32), P["scale"])
    with pytest.raises(oracle.OracleError):   # context beyond the table's capacity
        oracle.paged_attention(P["q"], P["kpool"], P["vpool"], P["bt"],
                               torch.tensor([33], dtype=torch.int32), P["scale"])
    bt = P["bt"].clone()
    bt[0, 1] = P["kpool"].shape[0]
    with pytest.raises(oracle.OracleError):
        oracle.paged_attention(P["q"], P["kpool"], P["vpool"], bt, P["ctx"], P["scale"])


# ------------------------------------------------------------------ a5: split + merge

@pytest.mark.parametrize("nsplit", [1, 2, 3, 5, 8])
def test_split_merge_identity(nsplit):
    P = _dense_problem(101, [300, 77], [1, 1], 4, 2, 32)
    full = _oracle_out(P)
    prob = oracle.Problem(P["q"], P["kpool"], P["vpool"], P["bt"], P["ctx"], P["scale"], P["cu"])
    rng = np.random.default_rng(nsplit)
    for s, c in enumerate([300, 77]):
        cuts = np.sort(rng.choice(np.arange(1, c), size=nsplit - 1, replace=False)) if nsplit > 1 else []
        edges = [0, *cuts.tolist(), c] if nsplit > 1 else [0, c]
        for h in range(4):
            parts = [oracle.attention_partial(prob, s, 0, h, a, b) for a, b in zip(edges[:-1], edges[1:])]
            m = [p[0] for p in parts]
            l = [p[1] for p in parts]
            o = np.stack([p[2] for p in parts])
            merged = oracle.merge_partials(m, l, o)
            np.testing.assert_allclose(merged, full[s, h], rtol=0, atol=1e-13)


def test_merge_of_outlier_partials_is_stable():
    # partials whose maxima differ by hundreds must merge without overflow
    m = np.array([0.0, 400.0, -300.0])
    l = np.array([3.0, 2.0, 5.0])
    o = np.array([[3.0, 6.0], [2.0, -2.0], [5.0, 5.0]])
    out = oracle.merge_partials(m, l, o)
    np.testing.assert_allclose(out, [1.0, -1.0], rtol=0, atol=1e-15)


# ------------------------------------------------------------------ block copy (swap / fork / pack)

def test_copy_blocks_moves_whole_blocks_and_nothing_else():
    B, hkv, d = 16, 2, 8
    src_k = torch.randn(6, B, hkv, d).to(torch.bfloat16)
    src_v = torch.randn(6, B, hkv, d).to(torch.bfloat16)
    dst_k = torch.zeros(4, B, hkv, d, dtype=torch.bfloat16)
    dst_v = torch.zeros_like(dst_k)
    oracle.copy_blocks(src_k, src_v, dst_k, dst_v, [[5, 0], [2, 3], [-1, 1], [0, -1]])
    assert torch.equal(dst_k[0], src_k[5]) and torch.equal(dst_v[0], src_v[5])
    assert torch.equal(dst_k[3], src_k[2]) and torch.equal(dst_v[3], src_v[2])
    assert (dst_k[1:3] == 0).all() and (dst_v[1:3] == 0).all()


def test_copy_blocks_pack_then_unpack_restores_a_request():
    # pack a request's scattered blocks into a contiguous buffer, wipe them,
    # unpack into other physical blocks: attention through the new table is unchanged
    P = _dense_problem(111, [70], [1], 4, 2, 32, extra_blocks=8)
    base = _oracle_out(P)
    bt = P["bt"][0]
    nb = oracle.num_blocks_needed(70, 16)
    k_buf = torch.empty(nb, *P["kpool"].shape[1:], dtype=P["kpool"].dtype)
    v_buf = torch.empty_like(k_buf)
    pack = [[int(bt[i]), i] for i in range(nb)]
    oracle.copy_blocks(P["kpool"], P["vpool"], k_buf, v_buf, pack)
    free = sorted(set(range(P["kpool"].shape[0])) - set(bt[:nb].tolist()))
    new_ids = free[:nb]
    P["kpool"][bt[:nb].long()] = float("nan")
    P["vpool"][bt[:nb].long()] = float("nan")
    oracle.copy_blocks(k_buf, v_buf, P["kpool"], P["vpool"], [[i, new_ids[i]] for i in range(nb)])
    P["bt"] = P["bt"].clone()
    P["bt"][0, :nb] = torch.tensor(new_ids, dtype=torch.int32)
    assert np.array_equal(_oracle_out(P), base)


def test_copy_blocks_rejects_bad_pairs():
    k = torch.zeros(3, 16, 1, 8)
    with pytest.raises(oracle.OracleError):
        oracle.copy_blocks(k, k.clone(), k.clone(), k.clone(), [[0, 1], [2, 1]])   # same destination
    with pytest.raises(oracle.OracleError):
        oracle.copy_blocks(k, k.clone(), k.clone(), k.clone(), [[3, 0]])           # outside the source
