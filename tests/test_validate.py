"""pa_validate_inputs: the host check of the preconditions the kernels rely on
but do not test (lengths and table entries in range, slots in the pool, no
slot written twice, no write into a block several tables share).  CPU only:
the call reads host memory and never touches a device."""
import numpy as np
import pytest
import torch

import oracle
from pagedattention_kv_cache_reshape_gb300 import build as B
from pagedattention_kv_cache_reshape_gb300 import pa
from pagedattention_kv_cache_reshape_gb300 import workloads as W


@pytest.fixture(scope="module", autouse=True)
def lib():
    B.build()
    return pa.load()


def _slots(w):
    """The step's slots, as the oracle computes them from the tables."""
    return torch.from_numpy(oracle.slot_mapping(w.block_tables, w.seq_start, w.cu_seqlens_q, w.block_size,
                                                w.num_blocks))


def _gqa(seed=0):
    # 12 sequences, 4 of them sharing a 128-token (8-block) prefix
    return W.gqa(seed, oracle.num_blocks_needed, num_seqs=12, ctx_hi=600, shared_seqs=4, prefix_tokens=128,
                 device="cpu")


@pytest.mark.parametrize("make", [lambda: _gqa(0), lambda: _gqa(1),
                                  lambda: W.tiny(0, oracle.num_blocks_needed, device="cpu"),
                                  lambda: W.mixed(0, oracle.num_blocks_needed, num_prefill=3, chunk=40,
                                                  prefix_hi=70, num_decode=9, dec_lo=5, dec_hi=300,
                                                  device="cpu")])
def test_generated_steps_pass(make):
    w = make()
    assert pa.validate_inputs(w.block_tables, w.context_lens, _slots(w), w.block_size, w.num_blocks) == (pa.OK, 0, -1)


def test_context_length_out_of_range():
    w = _gqa()
    for bad in (0, w.block_tables.shape[1] * w.block_size + 1):
        ctx = w.context_lens.clone()
        ctx[5] = bad
        assert pa.validate_inputs(w.block_tables, ctx, _slots(w), w.block_size, w.num_blocks) == \
            (pa.ERR_OUT_OF_RANGE, 1, 5)


def test_used_table_entry_out_of_range_and_unused_entries_ignored():
    w = _gqa()
    bt = w.block_tables.clone()
    s = 7
    used = -(-int(w.context_lens[s]) // w.block_size)
    if used < bt.shape[1]:
        bt[s, used:] = 10 ** 6            # entries past the context are not read
        assert pa.validate_inputs(bt, w.context_lens, None, w.block_size, w.num_blocks)[0] == pa.OK
    bt[s, used - 1] = w.num_blocks
    assert pa.validate_inputs(bt, w.context_lens, None, w.block_size, w.num_blocks) == (pa.ERR_OUT_OF_RANGE, 2, s)


def test_slot_beyond_pool_and_padding():
    w = _gqa()
    sl = _slots(w)
    sl[2] = -1                            # padding: skipped
    assert pa.validate_inputs(w.block_tables, w.context_lens, sl, w.block_size, w.num_blocks)[0] == pa.OK
    sl[4] = w.num_blocks * w.block_size
    assert pa.validate_inputs(w.block_tables, w.context_lens, sl, w.block_size, w.num_blocks) == \
        (pa.ERR_OUT_OF_RANGE, 3, 4)


def test_duplicate_slot_agrees_with_the_oracle_validator():
    w = _gqa()
    sl = _slots(w)
    sl[9] = sl[3]
    assert pa.validate_inputs(w.block_tables, w.context_lens, sl, w.block_size, w.num_blocks) == \
        (pa.ERR_INVALID_ARG, 4, 9)
    with pytest.raises(ValueError):
        oracle.validate_slots(sl.numpy())


def test_write_into_a_shared_prefix_block():
    w = _gqa()
    sl = _slots(w)
    shared_block = int(w.block_tables[0, 0])        # the first prefix block, in 4 tables
    assert int((w.block_tables[:4, 0] == shared_block).sum()) == 4
    sl[6] = shared_block * w.block_size + 3
    assert pa.validate_inputs(w.block_tables, w.context_lens, sl, w.block_size, w.num_blocks) == \
        (pa.ERR_INVALID_ARG, 5, 6)
    # without lengths the tables are not read, so only checks 3-4 apply
    assert pa.validate_inputs(w.block_tables, None, sl, w.block_size, w.num_blocks)[0] == pa.OK


def test_random_slot_sets_match_brute_force():
    rng = np.random.default_rng(3)
    for _ in range(200):
        nb, bs = int(rng.integers(1, 20)), int(rng.integers(1, 5))
        n = int(rng.integers(0, 30))
        sl = rng.integers(-2, nb * bs + 2, size=n).astype(np.int64)
        rc, check, idx = pa.validate_inputs(torch.zeros((0, 1), dtype=torch.int32), None, torch.from_numpy(sl),
                                            bs, nb)
        # brute force: first index that is out of the pool, else first repeat
        want = (pa.OK, 0, -1)
        over = [i for i, v in enumerate(sl) if v >= nb * bs]
        if over:
            want = (pa.ERR_OUT_OF_RANGE, 3, over[0])
        else:
            seen = set()
            for i, v in enumerate(sl):
                if v < 0:
                    continue
                if v in seen:
                    want = (pa.ERR_INVALID_ARG, 4, i)
                    break
                seen.add(v)
        assert (rc, check, idx) == want


def test_bad_sizes_rejected():
    assert pa.validate_inputs(torch.zeros((1, 1), dtype=torch.int32), torch.ones(1, dtype=torch.int32), None,
                              0, 4)[0] == pa.ERR_INVALID_ARG
