"""pa_varlen_forward_noalloc, the entry point for callers that cannot allocate device memory
(an op that is handed only its inputs and outputs, a runtime whose allocator it cannot reach,
a serving step that must not risk cudaMalloc's device synchronisation).  It keeps the
per-call plan in a fixed array inside the library instead of a caller workspace.

Checked through the C ABI against pa_varlen_forward on two different batches in a row (the
second call runs on whatever the first left in the shared array): both run the same kernels
on the same plan, so the outputs must agree bit for bit, and both must match the CPU oracle
within the attention tolerance.  Also checked: its size limit, and that a batch which
pa_varlen_forward rejects gets the same status here.
This file sorts last so that a stop-at-first-failure run has already run everything else.
"""
import ctypes

import pytest
import torch

from paged_kv_cache_31_gb300 import workloads
from tests.gpu_helpers import assert_attn_close, oracle_attention

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def pa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_31_gb300 import binding

    assert binding.pa_device_status() == binding.PA_OK
    return binding


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _raw_noalloc(pa, w, out, num_tokens=None, head_dim=None):
    """The entry point called directly through ctypes (no Python-side checks)."""
    T, H, D = w.q.shape
    NB, bs, Hkv, _ = w.k_blocks.shape
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    return pa._lib.pa_varlen_forward_noalloc(
        p(w.q), p(w.k_blocks), p(w.v_blocks), p(out), p(w.query_start_loc), p(w.seq_lens),
        p(w.positions), p(w.block_tables), w.num_seqs, T if num_tokens is None else num_tokens,
        H, Hkv, D if head_dim is None else head_dim, bs, NB, w.block_tables.shape[1],
        pa._DT[w.q.dtype], pa._DT[w.k_blocks.dtype], float(w.scale), int(w.causal),
        int(w.sliding_window), _stream())


def _raw_workspace(pa, w, out, ws, num_tokens=None, head_dim=None):
    """pa_varlen_forward through ctypes with the same arguments plus a workspace."""
    T, H, D = w.q.shape
    NB, bs, Hkv, _ = w.k_blocks.shape
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    return pa._lib.pa_varlen_forward(
        p(w.q), p(w.k_blocks), p(w.v_blocks), p(out), p(w.query_start_loc), p(w.seq_lens),
        p(w.positions), p(w.block_tables), w.num_seqs, T if num_tokens is None else num_tokens,
        H, Hkv, D if head_dim is None else head_dim, bs, NB, w.block_tables.shape[1],
        pa._DT[w.q.dtype], pa._DT[w.k_blocks.dtype], float(w.scale), int(w.causal),
        int(w.sliding_window), p(ws), ws.numel(), _stream())


def test_noalloc_matches_workspace_entry_on_two_calls_in_a_row(pa):
    # a mixed batch with prefill chunks (both attention kernels) and then a decode batch
    batches = [workloads.named(3, small=True, device=DEV, seed=4),
               workloads.named(2, small=True, device=DEV, seed=5)]
    for w in batches:
        ws = pa.workspace_for(w.q, w.k_blocks, w.query_start_loc, w.block_tables)
        ref = torch.full_like(w.q, float("nan"))
        assert _raw_workspace(pa, w, ref, ws) == pa.PA_OK
        got = torch.full_like(w.q, float("nan"))
        assert _raw_noalloc(pa, w, got) == pa.PA_OK
        assert pa.pa_device_status() == pa.PA_OK
        # same kernels, same plan layout: the same bits
        assert torch.equal(got, ref), f"noalloc differs from the workspace entry on {w.name}"
        assert_attn_close(got, oracle_attention(w, w.k_blocks.cpu(), w.v_blocks.cpu()),
                          f"noalloc vs oracle, {w.name}")


def test_noalloc_rejects_batches_beyond_its_fixed_array(pa):
    # a plan for 2^21 tokens needs well over the 4 MiB the library holds: rejected before any
    # launch, so the (deliberately tiny) tensors are never read
    w = workloads.build("huge", seq_lens=[8], q_lens=[1], num_heads=8, num_kv_heads=2,
                        head_dim=128, seed=1, device=DEV)
    out = torch.empty_like(w.q)
    assert _raw_noalloc(pa, w, out, num_tokens=1 << 21) == pa.PA_EINVAL
    assert pa.pa_device_status() == pa.PA_OK  # nothing was enqueued


@pytest.mark.parametrize("what", ["num_tokens", "head_dim"])
def test_noalloc_same_status_as_workspace_entry(pa, what):
    """A batch that pa_varlen_forward rejects as unsupported (more than INT32_MAX / 2 tokens, a
    head size above 256) gets the same status here, although its plan would also be larger
    than the fixed array; nothing is launched."""
    w = workloads.build("rej", seq_lens=[8], q_lens=[1], num_heads=8, num_kv_heads=2,
                        head_dim=128, seed=1, device=DEV)
    kw = {"num_tokens": (1 << 30) + 1} if what == "num_tokens" else {"head_dim": 512}
    ws = torch.empty(256, dtype=torch.uint8, device=DEV)
    out = torch.empty_like(w.q)
    a = _raw_workspace(pa, w, out, ws, **kw)
    b = _raw_noalloc(pa, w, out, **kw)
    assert a == pa.PA_EUNSUPPORTED and b == a, (a, b)
    assert pa.pa_device_status() == pa.PA_OK
