"""GPU parity of pa_copy_blocks (fork, swap to / from a pinned host pool, pack /
unpack) against the oracle's byte copy: bit-exact on every pool byte."""
import numpy as np
import pytest
import torch

import oracle
from pagedattention_kv_cache_reshape_gb300 import pa
from pagedattention_kv_cache_reshape_gb300 import workloads as W

from helpers import gpu_step, oracle_blocks

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from pagedattention_kv_cache_reshape_gb300 import build
    build.build()
    pa.load()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


@pytest.mark.parametrize("dtype,hkv,d", [(torch.bfloat16, 8, 128), (torch.float32, 4, 64), (torch.bfloat16, 1, 64)])
def test_fork_inside_one_pool_matches_oracle(dtype, hkv, d):
    g = torch.Generator().manual_seed(5)
    nblk = 300
    k = torch.randn(nblk, 16, hkv, d, generator=g).to(dtype)
    v = torch.randn(nblk, 16, hkv, d, generator=g).to(dtype)
    perm = torch.randperm(nblk, generator=g)
    src, dst = perm[:90], perm[90:180]            # disjoint: no destination is read
    pairs = torch.stack([src, dst], 1).to(torch.int32)
    pairs[7] = torch.tensor([-1, int(dst[7])])   # skipped pair
    kd, vd = k.to(DEV), v.to(DEV)
    pa.copy_blocks(kd, vd, kd, vd, pairs.to(DEV))
    oracle.copy_blocks(k, v, k, v, pairs.numpy())
    torch.cuda.synchronize()
    assert torch.equal(_bits(kd.cpu()), _bits(k)) and torch.equal(_bits(vd.cpu()), _bits(v))


def test_swap_out_to_pinned_host_and_back_keeps_attention_bitwise():
    w = W.gqa(17, oracle_blocks, num_seqs=16, ctx_hi=600, shared_seqs=0, prefix_tokens=0, device=DEV)
    _, before = gpu_step(w)
    s = 5                                            # swap sequence 5 out and back in elsewhere
    nb = w.blocks_per_seq[s]
    ids = w.block_tables[s, :nb].clone()
    host_k = torch.empty((nb,) + tuple(w.k_cache.shape[1:]), dtype=w.dtype).pin_memory()
    host_v = torch.empty_like(host_k).pin_memory()
    out_pairs = torch.stack([ids.cpu(), torch.arange(nb, dtype=torch.int32)], 1).to(torch.int32)
    pa.copy_blocks(w.k_cache, w.v_cache, host_k, host_v, out_pairs.to(DEV))          # swap out
    torch.cuda.synchronize()
    assert torch.equal(_bits(host_k), _bits(w.k_cache[ids.long()].cpu()))
    used = set(w.block_tables[w.block_tables >= 0].tolist())
    free = torch.tensor(sorted(set(range(w.num_blocks)) - used)[:nb], dtype=torch.int32)
    assert free.numel() == nb
    w.k_cache[ids.long()] = float("nan")             # the old blocks are reused by someone else
    w.v_cache[ids.long()] = float("nan")
    in_pairs = torch.stack([torch.arange(nb, dtype=torch.int32), free], 1).to(torch.int32)
    pa.copy_blocks(host_k, host_v, w.k_cache, w.v_cache, in_pairs.to(DEV))             # swap in
    bt = w.block_tables.clone()
    bt[s, :nb] = free.to(DEV)
    after = pa.decode(w.q, w.k_cache, w.v_cache, bt, w.context_lens, w.scale)
    torch.cuda.synchronize()
    assert torch.equal(after[s], before[s])


def test_pack_and_unpack_round_trip_matches_oracle():
    w = W.long(3, oracle_blocks, num_seqs=3, ctx=2000, num_blocks=500, device=DEV)
    nb = w.blocks_per_seq[1]
    ids = w.block_tables[1, :nb]
    buf_k = torch.empty((nb,) + tuple(w.k_cache.shape[1:]), dtype=w.dtype, device=DEV)
    buf_v = torch.empty_like(buf_k)
    pack = torch.stack([ids, torch.arange(nb, dtype=torch.int32, device=DEV)], 1).contiguous()
    pa.copy_blocks(w.k_cache, w.v_cache, buf_k, buf_v, pack)
    ck, cv = w.k_cache.cpu(), w.v_cache.cpu()
    rk = torch.empty_like(buf_k, device="cpu")
    rv = torch.empty_like(rk)
    oracle.copy_blocks(ck, cv, rk, rv, pack.cpu().numpy())
    torch.cuda.synchronize()
    assert torch.equal(_bits(buf_k.cpu()), _bits(rk)) and torch.equal(_bits(buf_v.cpu()), _bits(rv))
    # unpack into a fresh pool at reversed positions
    pool_k = torch.zeros_like(w.k_cache)
    pool_v = torch.zeros_like(w.v_cache)
    unpack = torch.stack([torch.arange(nb, dtype=torch.int32, device=DEV),
                          torch.arange(nb - 1, -1, -1, dtype=torch.int32, device=DEV)], 1).contiguous()
    pa.copy_blocks(buf_k, buf_v, pool_k, pool_v, unpack)
    torch.cuda.synchronize()
    assert torch.equal(_bits(pool_k[:nb].flip(0)), _bits(buf_k))


def test_out_of_range_pair_sets_status_and_skips():
    k = torch.randn(10, 16, 2, 64, device=DEV).to(torch.bfloat16)
    v = torch.randn_like(k)
    dk, dv = torch.zeros_like(k), torch.zeros_like(v)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    pairs = torch.tensor([[1, 2], [11, 3], [4, 99]], dtype=torch.int32, device=DEV)
    pa.copy_blocks(k, v, dk, dv, pairs, dev_status=status)
    assert pa.get_device_status(status) == pa.ERR_OUT_OF_RANGE
    assert torch.equal(dk[2], k[1])
    assert (dk[3] == 0).all() and (dk[[0, 1, 4, 5, 6, 7, 8, 9]] == 0).all()
