"""Host block manager (C++ in libpa): allocate_slots, free, shared prefixes.
CPU only -- these calls touch no GPU."""
import os

import numpy as np
import pytest
import torch

import oracle
from pagedattention_kv_cache_reshape_gb300 import build as B
from pagedattention_kv_cache_reshape_gb300 import pa

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    B.build()
    pa.load()


def _golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([int(x) for x in line.split()])
    return rows


def test_allocate_slots_takes_ceil_blocks_golden():
    (n, bs, nblk), = _golden("block_count.txt")
    m = pa.BlockManager(10, bs)
    assert m.allocate_slots(1, n) == pa.OK
    bt, nt = m.tables([1], 4)
    assert nt.tolist() == [n]
    assert (bt[0] >= 0).sum().item() == nblk
    assert m.num_free == 10 - nblk


def test_growth_fills_the_last_block_before_taking_another():
    fills = [f for _, f in _golden("block_table_fill.txt")]
    m = pa.BlockManager(8, 16)
    assert m.allocate_slots(7, sum(fills)) == pa.OK           # 24 tokens: blocks 16 + 8
    assert m.num_free == 6
    for _ in range(8):                                          # tokens 25..32 fill block 1
        assert m.allocate_slots(7, 1) == pa.OK
        assert m.num_free == 6
    assert m.allocate_slots(7, 1) == pa.OK                      # token 33 opens a third block
    assert m.num_free == 5
    # the next token after 24 landed in logical block 1, offset 8 (oracle slot map)
    m2 = pa.BlockManager(8, 16)
    m2.allocate_slots(0, 24)
    m2.allocate_slots(0, 1)
    bt, nt = m2.tables([0], 4)
    slots = oracle.slot_mapping(bt, torch.tensor([24], dtype=torch.int32),
                                torch.tensor([0, 1], dtype=torch.int32), 16, 8)
    assert slots[0] == int(bt[0, 1]) * 16 + 8


def test_pool_exhaustion_takes_nothing_and_reports():
    m = pa.BlockManager(5, 16)
    assert m.allocate_slots(1, 48) == pa.OK                     # 3 blocks
    assert m.allocate_slots(2, 40) == pa.ERR_OUT_OF_RANGE       # needs 3, 2 free
    assert m.num_free == 2
    assert m.allocate_slots(2, 32) == pa.OK                     # exactly 2
    assert m.num_free == 0
    assert m.allocate_slots(1, 1) == pa.ERR_OUT_OF_RANGE        # seq 1 must grow a block
    assert m.tables([1], 4)[1].tolist() == [48]                 # unchanged


def test_free_returns_blocks_and_they_are_reused():
    m = pa.BlockManager(6, 16)
    m.allocate_slots(1, 64)
    used = set(m.tables([1], 8)[0][0, :4].tolist())
    assert m.free(1) == pa.OK
    assert m.num_free == 6
    assert m.free(1) == pa.ERR_INVALID_ARG                      # unknown now
    m.allocate_slots(2, 96)
    assert set(m.tables([2], 8)[0][0, :6].tolist()) >= used


def test_shared_prefix_refcounts_and_release_order():
    m = pa.BlockManager(20, 16)
    m.allocate_slots(100, 64)                                   # parent: 4 blocks
    assert m.share_prefix(100, 101, 48) == pa.OK                # 3 shared blocks
    assert m.share_prefix(100, 102, 48) == pa.OK
    bt, nt = m.tables([100, 101, 102], 8)
    assert torch.equal(bt[1, :3], bt[0, :3]) and torch.equal(bt[2, :3], bt[0, :3])
    assert nt.tolist() == [64, 48, 48]
    for b in bt[0, :3].tolist():
        assert m.refcount(b) == 3
    assert m.refcount(int(bt[0, 3])) == 1
    m.allocate_slots(101, 16)                                   # private 4th block for 101
    bt, nt = m.tables([101], 8)
    assert m.refcount(int(bt[0, 3])) == 1
    free0 = m.num_free
    m.free(100)                                                 # parent leaves: shared blocks stay
    assert m.num_free == free0 + 1
    m.free(101)
    m.free(102)
    assert m.num_free == 20
    assert m.share_prefix(5, 6, 16) == pa.ERR_INVALID_ARG       # no parent


def test_partial_or_shared_writes_are_refused():
    m = pa.BlockManager(10, 16)
    m.allocate_slots(1, 40)
    assert m.share_prefix(1, 2, 20) == pa.ERR_UNSUPPORTED       # not whole blocks
    assert m.share_prefix(1, 2, 32) == pa.OK
    assert m.allocate_slots(2, 1) == pa.OK                      # 2's last block is full: new private block
    m3 = pa.BlockManager(10, 16, max_blocks_per_seq=2)
    assert m3.allocate_slots(9, 33) == pa.ERR_INVALID_ARG       # 3 blocks > the table width


def test_batch_from_the_manager_feeds_the_slot_mapping():
    rng = np.random.default_rng(3)
    m = pa.BlockManager(400, 16, max_blocks_per_seq=64)
    ids, qlen = list(range(12)), rng.integers(1, 90, 12)
    for s, n in zip(ids, qlen):
        assert m.allocate_slots(s, int(n)) == pa.OK
    bt, nt = m.tables(ids, 64)
    cu = torch.zeros(13, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(qlen, dtype=torch.int32), 0)
    slots = oracle.slot_mapping(bt, torch.zeros(12, dtype=torch.int32), cu, 16, 400)
    assert np.unique(slots).size == slots.size
    for s in ids:
        own = set(bt[s][bt[s] >= 0].tolist())
        assert {int(x) // 16 for x in slots[cu[s]:cu[s + 1]]} <= own


def test_batched_allocation_equals_one_call_per_sequence():
    """pa_allocate_slots_batch = pa_allocate_slots in order: the same statuses
    (including a pool running dry part-way and a shared last block) and the
    same block tables."""
    rng = np.random.default_rng(11)
    a = pa.BlockManager(40, 16, max_blocks_per_seq=32)
    b = pa.BlockManager(40, 16, max_blocks_per_seq=32)
    for m in (a, b):
        assert m.allocate_slots(0, 32) == pa.OK          # two whole blocks
        assert m.share_prefix(0, 1, 32) == pa.OK         # seq 1 shares them
        assert m.allocate_slots(2, 20) == pa.OK
        assert m.share_prefix(2, 3, 16) == pa.OK         # seq 3 shares block 0 of seq 2
    ids = np.array([5, 6, 0, 1, 2, 7, 3, 8, 9, 5], dtype=np.int64)
    cnt = rng.integers(0, 200, ids.size).astype(np.int32)
    cnt[4] = 3                                           # seq 2 appends into its own partial block
    want = [a.allocate_slots(int(s), int(n)) for s, n in zip(ids, cnt)]
    got = np.full(ids.size, -1, dtype=np.int32)
    first = b.allocate_slots_batch(ids, cnt, got)
    assert got.tolist() == want
    assert first == next((x for x in want if x != pa.OK), pa.OK)
    assert pa.ERR_OUT_OF_RANGE in want                   # the pool ran dry part-way
    # sequences that exist: the four set up, and those with an allocation that succeeded
    all_ids = sorted({int(s) for s, st in zip(ids, want) if st == pa.OK} | {0, 1, 2, 3})
    ta, na = a.tables(all_ids, 32)
    tb, nb = b.tables(all_ids, 32)
    assert np.array_equal(ta, tb) and np.array_equal(na, nb)
    assert a.num_free == b.num_free
    assert b.allocate_slots_batch(np.zeros(0, np.int64), np.zeros(0, np.int32)) == pa.OK
