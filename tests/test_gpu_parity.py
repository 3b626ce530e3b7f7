"""GPU parity: the CUDA path through the C ABI against the CPU fp64 oracle on the
same seeded inputs.

Bit-exact: slot mapping and the whole cache pool after the write.  Floating
point: fp32 max |err| <= 1e-5; bf16 max |err| <= 2e-2 and relative RMS <= 1e-2.
Small versions of every workload are compared on every output; the full-size
workloads on every output where the oracle is quick and on a sample otherwise.
"""
import numpy as np
import pytest
import torch

import oracle
from pagedattention_kv_cache_reshape_gb300 import pa
from pagedattention_kv_cache_reshape_gb300 import workloads as W

from helpers import (compare, gpu_step, oracle_attention, oracle_blocks, oracle_rows,
                     oracle_write, to_f64)

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from pagedattention_kv_cache_reshape_gb300 import build
    build.build()
    pa.load()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


SMALL = {
    "tiny": lambda seed: W.tiny(seed, oracle_blocks, device=DEV),
    "mha_small": lambda seed: W.mha(seed, oracle_blocks, num_seqs=6, ctx_lo=100, ctx_hi=300, device=DEV),
    "gqa_small": lambda seed: W.gqa(seed, oracle_blocks, num_seqs=24, ctx_hi=700, shared_seqs=6,
                                    prefix_tokens=128, device=DEV),
    "long_small": lambda seed: W.long(seed, oracle_blocks, num_seqs=2, ctx=3000, num_blocks=420, device=DEV),
    "mixed_small": lambda seed: W.mixed(seed, oracle_blocks, num_prefill=3, chunk=40, prefix_hi=70,
                                        num_decode=9, dec_lo=5, dec_hi=300, device=DEV),
    "mqa_small": lambda seed: W.build("mqa", seed=seed, blocks_needed=oracle_blocks, dtype=torch.bfloat16,
                                      num_heads=8, num_kv_heads=1, head_dim=128, block_size=16,
                                      q_lens=[1] * 5, context_lens=[1, 17, 230, 64, 999], device=DEV),
    # 16 q-heads per kv-head: two warps of 8 heads share each kv-head's K/V tiles
    "g16_decode": lambda seed: W.build("g16d", seed=seed, blocks_needed=oracle_blocks, dtype=torch.bfloat16,
                                       num_heads=32, num_kv_heads=2, head_dim=128, block_size=16,
                                       q_lens=[1] * 6, context_lens=[3, 16, 161, 700, 48, 1200], device=DEV),
    # 32 q-heads on one kv-head: four warps share its K/V tiles
    "g32_decode": lambda seed: W.build("g32d", seed=seed, blocks_needed=oracle_blocks, dtype=torch.bfloat16,
                                       num_heads=32, num_kv_heads=1, head_dim=128, block_size=16,
                                       q_lens=[1] * 4, context_lens=[17, 300, 1, 520], device=DEV),
    # 12 q-heads per kv-head (not a power of two): two warps of 6 heads each
    "g12_decode": lambda seed: W.build("g12d", seed=seed, blocks_needed=oracle_blocks, dtype=torch.bfloat16,
                                       num_heads=48, num_kv_heads=4, head_dim=64, block_size=16,
                                       q_lens=[1] * 5, context_lens=[40, 16, 333, 2, 800], device=DEV),
    # 2 q-heads per kv-head, 16 kv-heads (two kv-head groups of 8)
    "g2_decode": lambda seed: W.build("g2d", seed=seed, blocks_needed=oracle_blocks, dtype=torch.bfloat16,
                                      num_heads=32, num_kv_heads=16, head_dim=128, block_size=16,
                                      q_lens=[1] * 5, context_lens=[1, 33, 250, 90, 640], device=DEV),
    # 12 kv-heads x 128 dims: a token row of 192 16-byte vectors, written by the step's
    # cache write as one full chunk of 128 and a ragged one of 64
    "row192_decode": lambda seed: W.build("r192", seed=seed, blocks_needed=oracle_blocks, dtype=torch.bfloat16,
                                          num_heads=24, num_kv_heads=12, head_dim=128, block_size=16,
                                          q_lens=[1] * 6, context_lens=[1, 16, 17, 300, 95, 700], device=DEV),
    # a single sequence: one token (one block for the whole grid), and a long one
    # (every CTA a slice of the same sequence, merged from 152 pieces)
    "one_token": lambda seed: W.build("one1", seed=seed, blocks_needed=oracle_blocks, dtype=torch.bfloat16,
                                      num_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                                      q_lens=[1], context_lens=[1], device=DEV),
    "one_long": lambda seed: W.build("oneL", seed=seed, blocks_needed=oracle_blocks, dtype=torch.bfloat16,
                                     num_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                                     q_lens=[1], context_lens=[9000], device=DEV),
    # one 131,072-token sequence: 8,192 blocks, every CTA a slice of it, one merge of all pieces
    "one_128k": lambda seed: W.build("one128k", seed=seed, blocks_needed=oracle_blocks, dtype=torch.bfloat16,
                                     num_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                                     q_lens=[1], context_lens=[131072], device=DEV),
    # one long MHA sequence: four kv-head groups, each cut over a quarter of the CTAs (tree merges)
    "one_long_mha": lambda seed: W.build("oneLm", seed=seed, blocks_needed=oracle_blocks, dtype=torch.bfloat16,
                                         num_heads=32, num_kv_heads=32, head_dim=128, block_size=16,
                                         q_lens=[1], context_lens=[20000], device=DEV),
    # one long sequence with 16 q-heads per kv-head: two warps per kv-head, each its own tree
    "one_long_g16": lambda seed: W.build("oneLg", seed=seed, blocks_needed=oracle_blocks, dtype=torch.bfloat16,
                                         num_heads=32, num_kv_heads=2, head_dim=64, block_size=16,
                                         q_lens=[1], context_lens=[40000], device=DEV),
    "d64_bf16": lambda seed: W.build("d64", seed=seed, blocks_needed=oracle_blocks, dtype=torch.bfloat16,
                                     num_heads=16, num_kv_heads=4, head_dim=64, block_size=16,
                                     q_lens=[1] * 7, context_lens=[5, 16, 33, 400, 2, 129, 1000], device=DEV),
    "fp32_gqa_prefill": lambda seed: W.build("f32p", seed=seed, blocks_needed=oracle_blocks,
                                             dtype=torch.float32, num_heads=8, num_kv_heads=2, head_dim=128,
                                             block_size=16, q_lens=[20, 1, 7, 1], context_lens=[20, 60, 40, 1],
                                             device=DEV),
}


def _cpu_copy(w):
    return w.to("cpu")


def _run_and_check_all(w, seeds_note=""):
    wc = _cpu_copy(w)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    slots, out = gpu_step(w, dev_status=status)
    torch.cuda.synchronize()
    assert pa.get_device_status(status) == 0
    ref_slots = oracle_write(wc)
    assert np.array_equal(slots.cpu().numpy(), ref_slots), "slot mapping differs"
    assert torch.equal(w.k_cache.cpu().view(torch.int16 if w.dtype == torch.bfloat16 else torch.int32),
                       wc.k_cache.view(torch.int16 if w.dtype == torch.bfloat16 else torch.int32))
    assert torch.equal(w.v_cache.cpu().view(torch.int16 if w.dtype == torch.bfloat16 else torch.int32),
                       wc.v_cache.view(torch.int16 if w.dtype == torch.bfloat16 else torch.int32))
    ref = oracle_attention(wc)
    return compare(to_f64(out), ref, w.dtype, w.name + seeds_note)


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("seed", [1, 2])
def test_small_workloads_every_output(name, seed):
    _run_and_check_all(SMALL[name](seed), f" seed {seed}")


PREFILL_CASES = {
    # name: (H, Hkv, D, q_lens, context_lens)
    "gqa4_mixed_lengths": (32, 8, 128, [300, 1, 7, 129, 2, 64], [300, 90, 1000, 129, 2, 2100]),
    "mha_g1": (8, 8, 128, [130, 17, 1], [400, 17, 33]),
    "g2": (8, 4, 128, [65, 3], [700, 50]),
    "g8": (16, 2, 128, [40, 16], [333, 16]),
    "g16": (16, 1, 128, [9, 25, 8], [9, 600, 300]),
    "d64_gqa": (16, 4, 64, [100, 33, 1], [517, 33, 260]),
    "long_prefix": (32, 8, 128, [48], [3000]),
}


@pytest.mark.parametrize("name", list(PREFILL_CASES))
def test_prefill_shapes_every_output(name):
    H, Hkv, D, ql, ctx = PREFILL_CASES[name]
    w = W.build(name, seed=13, blocks_needed=oracle_blocks, dtype=torch.bfloat16, num_heads=H,
                num_kv_heads=Hkv, head_dim=D, block_size=16, q_lens=ql, context_lens=ctx, device=DEV)
    _run_and_check_all(w)


@pytest.mark.parametrize("name", list(PREFILL_CASES) + ["fp32_encode"])
def test_encode_only_every_output(name):
    """pa_varlen_encode: no causal mask, each row sees its whole sequence."""
    if name == "fp32_encode":
        H, Hkv, D, ql, ctx, dt = 8, 2, 64, [20, 1, 7], [20, 33, 40], torch.float32
    else:
        (H, Hkv, D, ql, ctx), dt = PREFILL_CASES[name], torch.bfloat16
    w = W.build(name, seed=23, blocks_needed=oracle_blocks, dtype=dt, num_heads=H, num_kv_heads=Hkv,
                head_dim=D, block_size=16, q_lens=ql, context_lens=ctx, device=DEV)
    wc = w.to("cpu")
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    slots = pa.compute_slot_mapping(w.block_tables, w.seq_start, w.cu_seqlens_q, w.num_blocks, w.total_q)
    pa.reshape_and_cache(w.key, w.value, w.k_cache, w.v_cache, slots)
    out = pa.varlen_prefill(w.q, w.cu_seqlens_q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                            w.scale, int(w.q_lens.max()), dev_status=status, causal=False)
    torch.cuda.synchronize()
    assert pa.get_device_status(status) == 0
    oracle_write(wc)
    ref = oracle.paged_attention(wc.q, wc.k_cache, wc.v_cache, wc.block_tables, wc.context_lens, wc.scale,
                                 cu_seqlens_q=wc.cu_seqlens_q, nthreads=8, causal=False)
    compare(to_f64(out), ref, dt, name + " encode")


def test_tiny_config_full():
    # configuration: 4 sequences, context {1,16,17,50}, fp32, 32-block pool
    for seed in (0, 3, 4):
        _run_and_check_all(W.tiny(seed, oracle_blocks, device=DEV), f" seed {seed}")


@pytest.mark.parametrize("name", ["mha64_bf16", "gqa256_bf16", "long_bf16"])
def test_full_size_decode_every_output(name):
    w = W.make(name, 0, oracle_blocks, device=DEV)
    _run_and_check_all(w)


def test_many_sequences_decode_every_output():
    """1500 decode rows: the plan scans its prefix in several passes of its CTA,
    and most CTAs hold many whole sequences plus cut ones."""
    rng = np.random.default_rng(77)
    ctx = rng.integers(1, 200, size=1500)
    w = W.build("many", seed=77, blocks_needed=oracle_blocks, dtype=torch.bfloat16, num_heads=16,
                num_kv_heads=4, head_dim=128, block_size=16, q_lens=[1] * 1500, context_lens=ctx,
                device=DEV)
    _run_and_check_all(w)


def test_many_decode_rows_in_a_mixed_step_every_output():
    """2 prefill chunks among 1200 decode rows through pa_varlen_step: the
    shared plan launch with its write CTAs over several scan passes, and the SM
    split for a batch dominated by decode rows."""
    rng = np.random.default_rng(78)
    q_lens = np.ones(1202, dtype=np.int64)
    q_lens[[17, 900]] = [96, 150]
    ctx = rng.integers(1, 300, size=1202)
    ctx[17], ctx[900] = 96 + 40, 150 + 333
    w = W.build("many_mixed", seed=78, blocks_needed=oracle_blocks, dtype=torch.bfloat16, num_heads=32,
                num_kv_heads=8, head_dim=128, block_size=16, q_lens=q_lens, context_lens=ctx, device=DEV)
    wc = w.to("cpu")
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    slots, out = pa.varlen_step(w.q, w.key, w.value, w.k_cache, w.v_cache, w.cu_seqlens_q, w.block_tables,
                                w.context_lens, w.seq_start, w.scale, int(q_lens.max()), dev_status=status)
    torch.cuda.synchronize()
    assert pa.get_device_status(status) == 0
    assert np.array_equal(slots.cpu().numpy(), oracle_write(wc))
    assert torch.equal(w.k_cache.cpu().view(torch.int16), wc.k_cache.view(torch.int16))
    compare(to_f64(out), oracle_attention(wc), w.dtype, "many_mixed")


@pytest.mark.parametrize("num_seqs", [16384, 16385])
def test_largest_decode_batch_every_output(num_seqs):
    """16384 sequences, the most the persistent decode kernel takes (the plan
    keeps the whole prefix in 64 KB of shared memory); one more goes through
    the generic kernel.  Short contexts keep the oracle quick."""
    rng = np.random.default_rng(num_seqs)
    ctx = rng.integers(1, 40, size=num_seqs)
    w = W.build("largest", seed=num_seqs, blocks_needed=oracle_blocks, dtype=torch.bfloat16, num_heads=8,
                num_kv_heads=2, head_dim=64, block_size=16, q_lens=[1] * num_seqs, context_lens=ctx,
                device=DEV)
    _run_and_check_all(w)


def test_full_size_mixed_sampled():
    w = W.make("mixed_bf16", 0, oracle_blocks, device=DEV)
    wc = _cpu_copy(w)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    slots, out = gpu_step(w, dev_status=status)
    torch.cuda.synchronize()
    assert pa.get_device_status(status) == 0
    ref_slots = oracle_write(wc)
    assert np.array_equal(slots.cpu().numpy(), ref_slots)
    assert torch.equal(w.k_cache.cpu().view(torch.int16), wc.k_cache.view(torch.int16))
    assert torch.equal(w.v_cache.cpu().view(torch.int16), wc.v_cache.view(torch.int16))
    # every decode row, and the first, last and 14 random rows of every chunk, all heads
    cu = wc.cu_seqlens_q.numpy()
    ql = cu[1:] - cu[:-1]
    rng = np.random.default_rng(0)
    rows = []
    for s in range(len(ql)):
        if ql[s] == 1:
            rows.append(cu[s])
        else:
            rows.extend([cu[s], cu[s + 1] - 1, *rng.integers(cu[s], cu[s + 1], 14).tolist()])
    rows = np.unique(np.array(rows))
    H = w.num_heads
    rr = np.repeat(rows, H)
    hh = np.tile(np.arange(H), rows.size)
    ref = oracle_rows(wc, rr, hh)
    got = to_f64(out)[rr, hh]
    compare(got, ref, w.dtype, "mixed_bf16 sampled")


def test_prefill_plan_beyond_shared_memory_sampled():
    """A batch whose prefill work list exceeds what the planner stages in shared
    memory (more than 4096 CTA tiles of capacity) goes through its global
    scratch: 72 chunks of 480 rows over prefixes U{0..600} plus 40 decode rows,
    8 q-heads / 2 kv-heads, sampled rows against the oracle."""
    rng = np.random.default_rng(11)
    q_lens = np.concatenate([np.full(72, 480), np.ones(40, dtype=np.int64)])
    ctx = np.concatenate([480 + rng.integers(0, 601, 72), rng.integers(1, 900, 40)])
    order = rng.permutation(q_lens.size)
    w = W.build("big_plan", seed=11, blocks_needed=oracle_blocks, dtype=torch.bfloat16, num_heads=8,
                num_kv_heads=2, head_dim=128, block_size=16, q_lens=q_lens[order], context_lens=ctx[order],
                device=DEV)
    assert w.total_q // 8 + w.num_seqs + 1 > 4096
    wc = _cpu_copy(w)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    _, out = gpu_step(w, dev_status=status)
    torch.cuda.synchronize()
    assert pa.get_device_status(status) == 0
    oracle_write(wc)
    cu = wc.cu_seqlens_q.numpy()
    ql = cu[1:] - cu[:-1]
    rows = []
    for s_ in range(len(ql)):
        if ql[s_] == 1:
            rows.append(cu[s_])
        else:
            rows.extend([cu[s_], cu[s_ + 1] - 1, *rng.integers(cu[s_], cu[s_ + 1], 3).tolist()])
    rows = np.unique(np.array(rows))
    rr = np.repeat(rows, w.num_heads)
    hh = np.tile(np.arange(w.num_heads), rows.size)
    got = to_f64(out)
    assert np.all(np.isfinite(got))
    compare(got[rr, hh], oracle_rows(wc, rr, hh), w.dtype, "prefill plan in global scratch")


def _poison_unused(w):
    """NaN into every pool slot no sequence reads: unreferenced blocks and the
    tail of each sequence's last block (live slots found with the oracle)."""
    wc = _cpu_copy(w)
    slots = []
    for s in range(w.num_seqs):
        c = int(wc.context_lens[s])
        cu = torch.tensor([0, c], dtype=torch.int32)
        slots.append(oracle.slot_mapping(wc.block_tables[s:s + 1], torch.zeros(1, dtype=torch.int32),
                                         cu, w.block_size, w.num_blocks))
    live = np.unique(np.concatenate(slots))
    mask = torch.ones(w.num_blocks * w.block_size, dtype=torch.bool)
    mask[torch.from_numpy(live)] = False
    mask = mask.to(DEV)
    for pool in (w.k_cache, w.v_cache):
        pool.view(w.num_blocks * w.block_size, -1)[mask] = float("nan")


@pytest.mark.parametrize("name", ["gqa_small", "mixed_small", "tiny", "mha_small"])
def test_nan_poison_in_unused_slots_never_reaches_output(name):
    clean = SMALL[name](5)
    _, out_clean = gpu_step(clean)
    dirty = SMALL[name](5)
    _poison_unused(dirty)
    _, out_dirty = gpu_step(dirty)
    torch.cuda.synchronize()
    assert torch.isfinite(out_dirty.float()).all()
    assert torch.equal(out_clean, out_dirty)


@pytest.mark.parametrize("name", ["gqa_small", "long_small", "mixed_small"])
def test_block_permutation_bitwise_invariance(name):
    w = SMALL[name](7)
    _, base = gpu_step(w)          # writes the new tokens into w's pools
    out_before = base.clone()
    # move every block to a new physical id and renumber the tables
    perm = torch.randperm(w.num_blocks, generator=torch.Generator().manual_seed(3)).to(DEV)
    k2 = torch.empty_like(w.k_cache)
    v2 = torch.empty_like(w.v_cache)
    k2[perm] = w.k_cache
    v2[perm] = w.v_cache
    bt = w.block_tables.clone()
    live = bt >= 0
    bt[live] = perm[bt[live].long()].to(torch.int32)
    if w.decode_only:
        out = pa.decode(w.q, k2, v2, bt, w.context_lens, w.scale)
    else:
        out = pa.varlen_prefill(w.q, w.cu_seqlens_q, k2, v2, bt, w.context_lens, w.scale,
                                int(w.q_lens.max()))
    torch.cuda.synchronize()
    assert torch.equal(out, out_before)


def test_run_to_run_determinism():
    w = W.make("gqa256_bf16", 1, oracle_blocks, device=DEV)
    _, a = gpu_step(w)
    outs = [pa.decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale) for _ in range(3)]
    torch.cuda.synchronize()
    for o in outs:
        assert torch.equal(o, a)


@pytest.mark.parametrize("name", ["one_long", "one_128k", "one_long_mha", "one_long_g16"])
def test_many_piece_merge_is_deterministic(name):
    """One sequence over every CTA: its pieces merge up a fixed tree in whatever
    order they arrive; repeated calls and a stale workspace give the same bits."""
    w = SMALL[name](3)
    _, a = gpu_step(w)
    ws_bytes = pa.decode_workspace_size(w.num_seqs, w.num_heads, w.num_kv_heads, w.head_dim, 16, w.max_blocks)
    for fill in (0x00, 0xFF, 0x5A):
        ws = torch.full((ws_bytes,), fill, dtype=torch.uint8, device=DEV)
        o = pa.decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(o, a)


def _mixed_for_streams():
    w = W.mixed(4, oracle_blocks, num_prefill=4, chunk=300, prefix_hi=900, num_decode=60, dec_lo=20,
                dec_hi=1500, device=DEV)
    gpu_step(w)                                  # the cache write, then one eager call
    return w, int(w.q_lens.max())


def _varlen(w, out, max_q):
    return pa.varlen_prefill(w.q, w.cu_seqlens_q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                             w.scale, max_q, out=out)


def _capture(w, max_q, warm_up):
    out = torch.empty_like(w.q)
    if warm_up:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            _varlen(w, out, max_q)
        torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _varlen(w, out, max_q)
    for _ in range(3):
        out.fill_(float("nan"))
        g.replay()
    torch.cuda.synchronize()
    return out


def test_mixed_call_in_a_graph_matches_eager_and_oracle():
    """The decode rows and the prefill chunks of one call run at once (the
    prefill kernel on the SMs the decode kernel leaves); a CUDA graph of the
    call gives the eager output bitwise, and it matches the oracle."""
    w, max_q = _mixed_for_streams()
    eager = torch.empty_like(w.q)
    _varlen(w, eager, max_q)
    torch.cuda.synchronize()
    assert torch.equal(_capture(w, max_q, warm_up=True), eager)
    compare(to_f64(eager), oracle_attention(w.to("cpu")), w.dtype, "mixed, parts overlapped")


def test_first_call_of_a_thread_captured_matches_eager():
    """A thread whose very first call is captured into a CUDA graph (no eager
    warm-up on that thread) gives the eager output bitwise: the call keeps no
    per-thread state that a capture could not create."""
    import threading
    w, max_q = _mixed_for_streams()
    eager = torch.empty_like(w.q)
    _varlen(w, eager, max_q)
    torch.cuda.synchronize()
    got = {}

    def worker():
        try:
            torch.cuda.set_device(0)
            got["out"] = _capture(w, max_q, warm_up=False)
        except Exception as ex:  # surfaced below
            got["error"] = ex

    t = threading.Thread(target=worker)
    t.start()
    t.join()
    assert "error" not in got, got.get("error")
    assert torch.equal(got["out"], eager)


def test_shared_prefix_identical_outputs():
    """Sequences 0..3 reference the same 256-token prefix blocks read-only and
    hold identical private tails and queries: identical outputs, pool unchanged."""
    ctx = [300, 300, 300, 300, 57, 610, 16, 140]
    w = W.build("shared", seed=11, blocks_needed=oracle_blocks, dtype=torch.bfloat16, num_heads=32,
                num_kv_heads=8, head_dim=128, block_size=16, q_lens=[1] * 8, context_lens=ctx,
                shared_prefix_seqs=4, shared_prefix_tokens=256, device=DEV)
    pb = 256 // 16
    bt = w.block_tables
    assert torch.equal(bt[1, :pb], bt[0, :pb])
    for s in (1, 2, 3):
        for lb in range(pb, w.blocks_per_seq[0]):
            assert int(bt[s, lb]) != int(bt[0, lb])
            w.k_cache[bt[s, lb]] = w.k_cache[bt[0, lb]]
            w.v_cache[bt[s, lb]] = w.v_cache[bt[0, lb]]
    w.q[1:4] = w.q[0]
    kb, vb = w.k_cache.clone(), w.v_cache.clone()
    out = pa.decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale)
    torch.cuda.synchronize()
    for s in (1, 2, 3):
        assert torch.equal(out[s], out[0])
    assert torch.equal(kb.view(torch.int16), w.k_cache.view(torch.int16))
    assert torch.equal(vb.view(torch.int16), w.v_cache.view(torch.int16))
    wc = w.to("cpu")
    compare(to_f64(out), oracle_attention(wc), torch.bfloat16, "shared prefix")


def test_prefill_row_matches_decode_at_same_position():
    w = W.build("t6", seed=9, blocks_needed=oracle_blocks, dtype=torch.bfloat16, num_heads=32,
                num_kv_heads=8, head_dim=128, block_size=16, q_lens=[70], context_lens=[70], device=DEV)
    _, pre = gpu_step(w)
    for i in (0, 15, 16, 40, 69):
        dec = pa.decode(w.q[i:i + 1].contiguous(), w.k_cache, w.v_cache, w.block_tables,
                        torch.tensor([i + 1], dtype=torch.int32, device=DEV), w.scale)
        torch.cuda.synchronize()
        compare(to_f64(dec[0]), to_f64(pre[i]), torch.bfloat16, f"row {i}")


def test_token_strided_fused_qkv_write():
    w = SMALL["gqa_small"](4)
    T, hkv, d = w.key.shape
    fused = torch.empty(T, 3, hkv, d, dtype=w.dtype, device=DEV)
    fused[:, 0] = 0
    fused[:, 1] = w.key
    fused[:, 2] = w.value
    ref = SMALL["gqa_small"](4)
    slots = pa.compute_slot_mapping(w.block_tables, w.seq_start, w.cu_seqlens_q, w.num_blocks, w.total_q)
    pa.reshape_and_cache(fused[:, 1], fused[:, 2], w.k_cache, w.v_cache, slots)
    pa.reshape_and_cache(ref.key, ref.value, ref.k_cache, ref.v_cache, slots)
    torch.cuda.synchronize()
    assert torch.equal(w.k_cache.view(torch.int16), ref.k_cache.view(torch.int16))
    assert torch.equal(w.v_cache.view(torch.int16), ref.v_cache.view(torch.int16))


def test_negative_slot_is_skipped_and_out_of_range_slot_flagged():
    w = SMALL["mha_small"](2)
    before_k = w.k_cache.clone()
    slots = torch.full((w.total_q,), -1, dtype=torch.int64, device=DEV)
    slots[0] = 5
    slots[1] = w.num_blocks * 16            # outside the pool
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    pa.reshape_and_cache(w.key, w.value, w.k_cache, w.v_cache, slots, dev_status=status)
    assert pa.get_device_status(status) == pa.ERR_OUT_OF_RANGE
    changed = (w.k_cache != before_k).view(w.num_blocks * 16, -1).any(1)
    assert changed.nonzero().flatten().tolist() == [5]


def test_out_of_range_block_id_sets_status_without_fault():
    w = SMALL["gqa_small"](3)
    gpu_step(w)
    bt = w.block_tables.clone()
    bt[2, 0] = w.num_blocks + 100
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    pa.decode(w.q, w.k_cache, w.v_cache, bt, w.context_lens, w.scale, dev_status=status)
    assert pa.get_device_status(status) == pa.ERR_OUT_OF_RANGE
    # slot mapping over a bad entry: slot -1 and the status
    status.zero_()
    ss = torch.tensor([0], dtype=torch.int32, device=DEV)
    cu = torch.tensor([0, 3], dtype=torch.int32, device=DEV)
    s = pa.compute_slot_mapping(bt[2:3].contiguous(), ss, cu, w.num_blocks, 3, dev_status=status)
    assert pa.get_device_status(status) == pa.ERR_OUT_OF_RANGE
    assert s.tolist() == [-1, -1, -1]


def test_zero_context_flags_and_leaves_row_untouched():
    w = SMALL["gqa_small"](6)
    gpu_step(w)
    ctx = w.context_lens.clone()
    ctx[5] = 0
    out = torch.full_like(w.q, 7.0)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    pa.decode(w.q, w.k_cache, w.v_cache, w.block_tables, ctx, w.scale, out=out, dev_status=status)
    assert pa.get_device_status(status) == pa.ERR_OUT_OF_RANGE
    assert (out[5] == 7.0).all()
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("name", ["gqa_small", "mixed_small", "long_small", "mha_small"])
def test_stale_workspace_contents_do_not_matter(name):
    """The workspace may hold anything on entry (here: NaN bytes everywhere)."""
    w = SMALL[name](8)
    _, clean = gpu_step(w)
    ws_bytes = (pa.decode_workspace_size(w.num_seqs, w.num_heads, w.num_kv_heads, w.head_dim, 16, w.max_blocks)
                if w.decode_only else
                pa.varlen_prefill_workspace_size(w.num_seqs, w.total_q, w.num_heads, w.num_kv_heads,
                                                 w.head_dim, 16, w.max_blocks))
    ws = torch.full((ws_bytes,), 0xFF, dtype=torch.uint8, device=DEV)     # NaN patterns
    _, dirty = gpu_step(w, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(clean, dirty)


@pytest.mark.parametrize("name", ["gqa_small", "tiny", "long_small", "mha_small", "mqa_small", "d64_bf16",
                                  "g2_decode", "row192_decode", "one_token", "one_long"])
def test_fused_decode_step_equals_separate_calls(name):
    """pa_decode_step = slot mapping + cache write + decode, bit for bit."""
    a = SMALL[name](12)
    b = SMALL[name](12)
    slots_a, out_a = gpu_step(a)                   # three separate calls
    slots_b, out_b = pa.decode_step(b.q, b.key, b.value, b.k_cache, b.v_cache, b.block_tables,
                                    b.context_lens, b.seq_start, b.cu_seqlens_q, b.scale)
    torch.cuda.synchronize()
    assert torch.equal(slots_a, slots_b)
    bits = torch.int16 if a.dtype == torch.bfloat16 else torch.int32
    assert torch.equal(a.k_cache.view(bits), b.k_cache.view(bits))
    assert torch.equal(a.v_cache.view(bits), b.v_cache.view(bits))
    assert torch.equal(out_a, out_b)


def test_fused_decode_step_full_size_matches_oracle():
    w = W.make("gqa256_bf16", 2, oracle_blocks, device=DEV)
    wc = w.to("cpu")
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    slots, out = pa.decode_step(w.q, w.key, w.value, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                                w.seq_start, w.cu_seqlens_q, w.scale, dev_status=status)
    torch.cuda.synchronize()
    assert pa.get_device_status(status) == 0
    ref_slots = oracle_write(wc)
    assert np.array_equal(slots.cpu().numpy(), ref_slots)
    assert torch.equal(w.k_cache.cpu().view(torch.int16), wc.k_cache.view(torch.int16))
    compare(to_f64(out), oracle_attention(wc), torch.bfloat16, "decode step gqa256")


@pytest.mark.parametrize("name", ["gqa_small", "mha_small"])
def test_fused_decode_step_token_strided_and_bad_slot(name):
    w = SMALL[name](14)
    T, hkv, d = w.key.shape
    fused = torch.empty(T, 3, hkv, d, dtype=w.dtype, device=DEV)
    fused[:, 1] = w.key
    fused[:, 2] = w.value
    ref = SMALL[name](14)
    _, out_ref = gpu_step(ref)
    _, out = pa.decode_step(w.q, fused[:, 1], fused[:, 2], w.k_cache, w.v_cache, w.block_tables,
                            w.context_lens, w.seq_start, w.cu_seqlens_q, w.scale)
    torch.cuda.synchronize()
    assert torch.equal(out, out_ref)
    # an out-of-range table entry on a new token's block: status set, no fault
    bt = w.block_tables.clone()
    s = 3
    lb = int(w.seq_start[s]) // 16
    bt[s, lb] = w.num_blocks + 7
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    slots, _ = pa.decode_step(w.q, w.key, w.value, w.k_cache, w.v_cache, bt, w.context_lens, w.seq_start,
                              w.cu_seqlens_q, w.scale, dev_status=status)
    assert pa.get_device_status(status) == pa.ERR_OUT_OF_RANGE
    assert int(slots[s]) == -1


def _varlen_step(w, key=None, value=None, **kw):
    return pa.varlen_step(w.q, w.key if key is None else key, w.value if value is None else value,
                          w.k_cache, w.v_cache, w.cu_seqlens_q, w.block_tables, w.context_lens, w.seq_start,
                          w.scale, int(w.q_lens.max()), **kw)


@pytest.mark.parametrize("name", ["mixed_small", "fp32_gqa_prefill", "gqa_small", "g12_decode"])
def test_fused_varlen_step_equals_separate_calls(name):
    """pa_varlen_step = slot mapping + cache write + varlen attention, bit for bit
    (the write folded into the plan launch for mixed bf16 batches; separate
    kernels for fp32 and for decode-only batches)."""
    a = SMALL[name](13)
    b = SMALL[name](13)
    slots_a, out_a = gpu_step(a)
    slots_b, out_b = _varlen_step(b)
    torch.cuda.synchronize()
    assert torch.equal(slots_a, slots_b)
    bits = torch.int16 if a.dtype == torch.bfloat16 else torch.int32
    assert torch.equal(a.k_cache.view(bits), b.k_cache.view(bits))
    assert torch.equal(a.v_cache.view(bits), b.v_cache.view(bits))
    assert torch.equal(out_a, out_b)


def test_fused_varlen_step_full_size_mixed_and_strided():
    """The full mixed step through pa_varlen_step equals the three calls bit for
    bit, also with key / value as token-strided views of a fused QKV tensor."""
    a = W.make("mixed_bf16", 0, oracle_blocks, device=DEV)
    b = W.make("mixed_bf16", 0, oracle_blocks, device=DEV)
    slots_a, out_a = gpu_step(a)
    T, hkv, d = b.key.shape
    fused = torch.empty(T, 3, hkv, d, dtype=b.dtype, device=DEV)
    fused[:, 1] = b.key
    fused[:, 2] = b.value
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    slots_b, out_b = _varlen_step(b, key=fused[:, 1], value=fused[:, 2], dev_status=status)
    torch.cuda.synchronize()
    assert pa.get_device_status(status) == 0
    assert torch.equal(slots_a, slots_b)
    assert torch.equal(a.k_cache.view(torch.int16), b.k_cache.view(torch.int16))
    assert torch.equal(a.v_cache.view(torch.int16), b.v_cache.view(torch.int16))
    assert torch.equal(out_a, out_b)


def test_workspace_too_small_is_rejected():
    w = SMALL["gqa_small"](1)
    ws = torch.empty(64, dtype=torch.uint8, device=DEV)
    with pytest.raises(pa.PAError) as e:
        pa.decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale, workspace=ws)
    assert e.value.status == pa.ERR_WORKSPACE
