"""pa_varlen_forward_noalloc, the entry point for callers that cannot allocate device memory
(an op that is handed only its inputs and outputs, a runtime whose allocator it cannot reach,
a serving step that must not risk cudaMalloc's device synchronisation).  It keeps the
per-call plan in a fixed array inside the library instead of a caller workspace.

Checked through the C ABI against pa_varlen_forward on two different batches in a row (the
second call runs on whatever the first left in the shared array), and for its size limit.
This file sorts last so that a stop-at-first-failure run has already run everything else.
"""
import ctypes

import pytest
import torch

from paged_kv_cache_31_gb300 import workloads
from tests.gpu_helpers import assert_attn_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def pa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_31_gb300 import binding

    assert binding.pa_device_status() == binding.PA_OK
    return binding


def _raw_noalloc(pa, w, out):
    """The new entry point called directly through ctypes (no Python-side checks)."""
    T, H, D = w.q.shape
    NB, bs, Hkv, _ = w.k_blocks.shape
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    return pa._lib.pa_varlen_forward_noalloc(
        p(w.q), p(w.k_blocks), p(w.v_blocks), p(out), p(w.query_start_loc), p(w.seq_lens),
        p(w.positions), p(w.block_tables), w.num_seqs, T, H, Hkv, D, bs, NB,
        w.block_tables.shape[1], pa._DT[w.q.dtype], pa._DT[w.k_blocks.dtype], float(w.scale),
        int(w.causal), int(w.sliding_window),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_workspace_entry_on_two_calls_in_a_row(pa):
    batches = [workloads.named(3, small=True, device=DEV, seed=4),
               workloads.named(2, small=True, device=DEV, seed=5)]
    for w in batches:
        ref = torch.empty_like(w.q)
        pa.pa_varlen_forward(w.q, w.k_blocks, w.v_blocks, ref, w.query_start_loc, w.seq_lens,
                             w.positions, w.block_tables, w.scale, causal=w.causal,
                             sliding_window=w.sliding_window)
        got = torch.full_like(w.q, float("nan"))
        assert _raw_noalloc(pa, w, got) == pa.PA_OK
        assert pa.pa_device_status() == pa.PA_OK
        assert_attn_close(got, ref.float(), f"noalloc vs workspace entry, {w.name}")


def test_noalloc_rejects_batches_beyond_its_fixed_array(pa):
    # a plan for 2^21 tokens needs well over the 4 MiB the library holds: rejected before any
    # launch, so the (deliberately tiny) tensors are never read
    w = workloads.build("huge", seq_lens=[8], q_lens=[1], num_heads=8, num_kv_heads=2,
                        head_dim=128, seed=1, device=DEV)
    NB, bs, Hkv, D = w.k_blocks.shape
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    out = torch.empty_like(w.q)
    st = pa._lib.pa_varlen_forward_noalloc(
        p(w.q), p(w.k_blocks), p(w.v_blocks), p(out), p(w.query_start_loc), p(w.seq_lens),
        p(w.positions), p(w.block_tables), 1, 1 << 21, 8, Hkv, D, bs, NB, 1, pa.PA_BF16,
        pa.PA_BF16, 0.1, 1, 0, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == pa.PA_EINVAL
    assert pa.pa_device_status() == pa.PA_OK  # nothing was enqueued
