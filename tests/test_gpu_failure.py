"""Failure detection without a GPU fault.  Every wait inside the attention kernels is bounded:
when one runs out the kernel records PA_ETIMEOUT in the device status word (the tinyllm
interface's error classes, extended with a timeout), waits for its own copies (and, in the
tcgen05 kernel, MMAs) still in flight, writes nothing more and returns, so the context stays
usable.  PA_DEBUG_STALL_NS=<ns> makes the warp-MMA kernels' block waits and the tcgen05
kernel's softmax waits name a barrier that nothing signals, with every wait bounded at <ns>
(1 ms here; 20 ms for the tcgen05 kernel, whose other roles then give up in turn), so they run
out; the tests check the status, that the output is untouched, and that the next call on the
device gives the same bits as before."""
import contextlib
import os

import pytest
import torch

from paged_kv_cache_31_gb300 import workloads

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def pa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_31_gb300 import binding

    assert binding.pa_device_status() == binding.PA_OK
    return binding


@contextlib.contextmanager
def _stalled_waits(ns=1_000_000):
    old = os.environ.get("PA_DEBUG_STALL_NS")
    os.environ["PA_DEBUG_STALL_NS"] = str(ns)
    try:
        yield
    finally:
        if old is None:
            del os.environ["PA_DEBUG_STALL_NS"]
        else:
            os.environ["PA_DEBUG_STALL_NS"] = old


def _decode(pa, fp8):
    w = workloads.named(2, seed=12, device=DEV)
    kb, vb, kw = w.k_blocks, w.v_blocks, {}
    if fp8:
        kb, vb = workloads.fp8_pools(w)
        kw = dict(k_scale=0.125, v_scale=0.125)

    def call():
        out = torch.full_like(w.q, 7.0)
        pa.pa_varlen_forward(w.q, kb, vb, out, w.query_start_loc, w.seq_lens, w.positions,
                             w.block_tables, w.scale, **kw)
        return out
    return call


def _splitkv(pa):
    w = workloads.build("split", seq_lens=[700, 3000, 4100], q_lens=[1, 1, 1], num_heads=32,
                        num_kv_heads=8, head_dim=128, seed=13, device=DEV, partition_size=512)
    S, H, D, P = w.num_seqs, w.num_heads, w.head_dim, w.max_partitions()

    def call():
        out = torch.full_like(w.q, 7.0)
        ml = torch.empty((S, H, P), device=DEV)
        es = torch.empty_like(ml)
        to = torch.empty((S, H, P, D), device=DEV)
        pa.pa_decode_splitkv(w.q, w.k_blocks, w.v_blocks, out, ml, es, to, w.seq_lens,
                             w.block_tables, w.scale, partition_size=512)
        return out
    return call


@pytest.mark.parametrize("case", ["decode-bf16", "decode-fp8", "splitkv"])
def test_waits_that_run_out_report_timeout_and_the_device_stays_usable(pa, case):
    call = _splitkv(pa) if case == "splitkv" else _decode(pa, case == "decode-fp8")
    ref = call()
    assert pa.pa_device_status() == pa.PA_OK
    with _stalled_waits():
        call()
        assert pa.pa_device_status() == pa.PA_ETIMEOUT
        call()  # the status word was cleared by the read: it times out again
        assert pa.pa_device_status() == pa.PA_ETIMEOUT
    out = call()
    assert pa.pa_device_status() == pa.PA_OK
    assert torch.equal(out, ref)


def test_tcgen05_prefill_timeout_unwinds_and_the_device_stays_usable(pa):
    """The tcgen05 kernel's unwinding: the softmax warps' waits run out, every other role of
    both CTAs of each pair gives up at its next wait (the abort flag, or its own bounded
    wait), the producers wait for the copies they issued, the MMA issuers for their MMAs, and
    the pair meets before its tensor memory is freed.  No output row is written, and the next
    call gives the same bits as a call before the stall."""
    prior, chunk = [0, 300, 45, 700], [200, 129, 96, 257]
    w = workloads.build("stall", seq_lens=[p + c for p, c in zip(prior, chunk)], q_lens=chunk,
                        num_heads=32, num_kv_heads=8, head_dim=128, seed=14, device=DEV)

    def call():
        out = torch.full_like(w.q, 7.0)
        pa.pa_varlen_forward(w.q, w.k_blocks, w.v_blocks, out, w.query_start_loc, w.seq_lens,
                             w.positions, w.block_tables, w.scale)
        return out
    ref = call()
    assert pa.pa_device_status() == pa.PA_OK
    with _stalled_waits(20_000_000):
        out = call()
        assert pa.pa_device_status() == pa.PA_ETIMEOUT
        assert bool((out == 7.0).all()), "a timed-out prefill call wrote output"
    again = call()
    assert pa.pa_device_status() == pa.PA_OK
    assert torch.equal(again, ref)


def test_a_recorded_error_stops_later_kernels_until_it_is_read(pa):
    # the status word is sticky: after a timeout, kernels launched before the host reads it
    # write nothing (tinyllm 2.6: out untouched after an error)
    call = _decode(pa, False)
    with _stalled_waits():
        call()
    out = call()  # launched while the timeout is still recorded
    assert pa.pa_device_status() == pa.PA_ETIMEOUT
    assert bool((out == 7.0).all())
    assert pa.pa_device_status() == pa.PA_OK
