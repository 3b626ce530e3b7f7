"""The bounded in-kernel waits, made to run out on purpose.

Every wait of the pipelined kernels (the decode's TMA producer and attention
warps; the prefill's producer, MMA issuer and softmax warpgroups) gives up
after a time limit, records PA_ERR_TIMEOUT and lets the kernel return, so a
stuck pipeline cannot hang the GPU.  pa_set_wait_test shortens that limit and
makes one role of every CTA stop early without giving the signal the others
wait for: nothing ever sets it, so their waits run out.  Nothing faults:
every copy a CTA issued is waited for before it exits.

Each test checks that the status word reads PA_ERR_TIMEOUT, that the roles
expected to time out recorded it, and that the next normal call on the same
stream gives the result from before bit for bit.
"""
import pytest
import torch

from pagedattention_kv_cache_reshape_gb300 import pa
from pagedattention_kv_cache_reshape_gb300 import workloads as W

from helpers import gpu_step, oracle_blocks

pytestmark = pytest.mark.gpu
DEV = "cuda"
LIMIT_NS = 20_000_000   # 20 ms per wait that runs out


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from pagedattention_kv_cache_reshape_gb300 import build
    build.build()
    pa.load()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


@pytest.fixture(autouse=True)
def _normal_waits_after():
    yield
    pa.set_wait_test()      # whatever runs next waits normally


@pytest.fixture(scope="module")
def decode_case():
    # 64 sequences of up to 2000 tokens: every CTA streams a dozen blocks or more,
    # well past the stall point plus the three-stage ring
    w = W.gqa(7, oracle_blocks, num_seqs=64, ctx_hi=2000, shared_seqs=8, prefix_tokens=128, device=DEV)
    gpu_step(w)             # the step's new tokens are in the cache
    ref = pa.decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale)
    torch.cuda.synchronize()
    return w, ref.clone()


@pytest.fixture(scope="module")
def prefill_case():
    # prefill chunks only (no decode rows): 4 x 256 rows over up to 2048 cached
    # tokens, so the longest work items stream about 18 K/V tiles, past the stall
    # point plus the five-slot ring
    w = W.mixed(8, oracle_blocks, num_prefill=4, chunk=256, prefix_hi=2048, num_decode=0, device=DEV)
    gpu_step(w)
    ref = _prefill(w)
    torch.cuda.synchronize()
    return w, ref.clone()


def _decode(w, status=None):
    return pa.decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale,
                     out=torch.full_like(w.q, float("nan")), dev_status=status)


def _prefill(w, status=None):
    return pa.varlen_prefill(w.q, w.cu_seqlens_q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                             w.scale, int(w.q_lens.max()), out=torch.full_like(w.q, float("nan")),
                             dev_status=status)


def _stalled_then_normal(run, w, ref, stall, after, expect_sites):
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    sites = torch.zeros(1, dtype=torch.int32, device=DEV)
    pa.set_wait_test(LIMIT_NS, stall, after, sites)
    run(w, status)
    torch.cuda.synchronize()
    pa.set_wait_test()
    assert pa.get_device_status(status) == pa.ERR_TIMEOUT
    got = int(sites.item())
    for bit in expect_sites:
        assert got & bit, f"wait sites {got:#x}: bit {bit:#x} missing"
    # the context is intact: the next normal call on the same stream is exact
    status.zero_()
    out = run(w, status)
    torch.cuda.synchronize()
    assert pa.get_device_status(status) == pa.OK
    assert torch.equal(out, ref)
    return got


def test_short_limit_without_a_stall_changes_nothing(decode_case, prefill_case):
    for run, (w, ref) in ((_decode, decode_case), (_prefill, prefill_case)):
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        sites = torch.zeros(1, dtype=torch.int32, device=DEV)
        pa.set_wait_test(LIMIT_NS, pa.STALL_NONE, 0, sites)
        out = run(w, status)
        torch.cuda.synchronize()
        assert pa.get_device_status(status) == pa.OK and int(sites.item()) == 0
        assert torch.equal(out, ref)


def test_decode_consumers_time_out_when_the_producer_stops(decode_case):
    w, ref = decode_case
    got = _stalled_then_normal(_decode, w, ref, pa.STALL_PRODUCER, 2, [pa.WAIT_DECODE_CONSUMER])
    assert not got & pa.WAIT_DECODE_PRODUCER


def test_decode_producer_times_out_when_the_consumers_stop(decode_case):
    w, ref = decode_case
    got = _stalled_then_normal(_decode, w, ref, pa.STALL_CONSUMER, 2, [pa.WAIT_DECODE_PRODUCER])
    assert not got & pa.WAIT_DECODE_CONSUMER


def test_prefill_mma_and_softmax_time_out_when_the_producer_stops(prefill_case):
    w, ref = prefill_case
    got = _stalled_then_normal(_prefill, w, ref, pa.STALL_PRODUCER, 3,
                               [pa.WAIT_PREFILL_MMA, pa.WAIT_PREFILL_SOFTMAX])
    assert not got & pa.WAIT_PREFILL_PRODUCER


def test_prefill_producer_and_softmax_time_out_when_the_mma_issuer_stops(prefill_case):
    w, ref = prefill_case
    got = _stalled_then_normal(_prefill, w, ref, pa.STALL_CONSUMER, 3,
                               [pa.WAIT_PREFILL_PRODUCER, pa.WAIT_PREFILL_SOFTMAX])
    assert not got & pa.WAIT_PREFILL_MMA
