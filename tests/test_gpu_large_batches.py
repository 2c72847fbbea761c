"""Batches larger than the planner keeps in shared memory (more than 4096 sequences or 8192
tokens): the planner reads the metadata from global memory, checks the block tables itself and
waits for the kernels ahead of it before it starts.  Checked against the oracle on every row,
with e4m3 pools and per-block factors, and for the validation errors.
"""
import pytest
import torch

import oracle
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


def _many_seqs(seed=7):
    # 4200 decode sequences (past the planner's 4096), contexts 1..200
    g = torch.Generator().manual_seed(seed)
    lens = torch.randint(1, 201, (4200,), generator=g).tolist()
    return workloads.build("many-seqs", seq_lens=lens, q_lens=[1] * len(lens), num_heads=16,
                           num_kv_heads=4, head_dim=128, seed=seed, device=DEV)


def _oracle(w, kb, vb, **kw):
    st, ref, _ = oracle.varlen_attention(w.q.cpu(), kb.cpu(), vb.cpu(), w.query_start_loc,
                                         w.seq_lens, w.positions, w.block_tables, w.scale,
                                         causal=w.causal, sliding_window=w.sliding_window, **kw)
    assert st == oracle.OK
    return ref


def test_many_sequences(pa):
    w = _many_seqs()
    out = torch.full_like(w.q, float("nan"))
    pa.pa_varlen_forward(w.q, w.k_blocks, w.v_blocks, out, w.query_start_loc, w.seq_lens,
                         w.positions, w.block_tables, w.scale)
    assert pa.pa_device_status() == pa.PA_OK
    assert_attn_close(out, _oracle(w, w.k_blocks, w.v_blocks), "4200 sequences")


def test_many_tokens(pa):
    # 64 prefill chunks of 130 tokens (8320 tokens, past the planner's 8192): tcgen05 items
    # listed in global memory
    g = torch.Generator().manual_seed(8)
    prior = torch.randint(0, 300, (64,), generator=g).tolist()
    w = workloads.build("many-tokens", seq_lens=[p + 130 for p in prior], q_lens=[130] * 64,
                        num_heads=8, num_kv_heads=2, head_dim=128, seed=8, device=DEV,
                        sliding_window=200)
    out = torch.full_like(w.q, float("nan"))
    pa.pa_varlen_forward(w.q, w.k_blocks, w.v_blocks, out, w.query_start_loc, w.seq_lens,
                         w.positions, w.block_tables, w.scale, sliding_window=w.sliding_window)
    assert pa.pa_device_status() == pa.PA_OK
    assert_attn_close(out, _oracle(w, w.k_blocks, w.v_blocks), "8320 tokens")


def test_many_sequences_fp8_per_block(pa):
    w = _many_seqs(9)
    kb, vb = workloads.fp8_pools(w)
    NB, Hkv = kb.shape[0], w.num_kv_heads
    g = torch.Generator().manual_seed(10)
    ks = (2.0 ** (-5 + 3 * torch.rand((NB, Hkv), generator=g))).to(DEV)
    vs = (2.0 ** (-5 + 3 * torch.rand((NB, Hkv), generator=g))).to(DEV)
    out = torch.full_like(w.q, float("nan"))
    pa.pa_varlen_forward(w.q, kb, vb, out, w.query_start_loc, w.seq_lens, w.positions,
                         w.block_tables, w.scale, k_block_scales=ks, v_block_scales=vs)
    assert pa.pa_device_status() == pa.PA_OK
    ref = _oracle(w, kb, vb, k_block_scales=ks, v_block_scales=vs)
    assert_attn_close(out, ref, "4200 sequences, e4m3, per-block factors")
    # a bad factor of a block the last sequence reads: rejected, nothing written
    vs[int(w.block_tables[-1, 0]), 1] = float("nan")
    out = torch.full_like(w.q, 7.0)
    pa.pa_varlen_forward(w.q, kb, vb, out, w.query_start_loc, w.seq_lens, w.positions,
                         w.block_tables, w.scale, k_block_scales=ks, v_block_scales=vs)
    assert pa.pa_device_status() == pa.PA_EINVAL
    assert bool((out == 7.0).all())


def test_many_sequences_bad_table_entry(pa):
    w = _many_seqs(11)
    bt = w.block_tables.clone()
    bt[-1, 0] = w.k_blocks.shape[0]  # one past the pool, in the last sequence's table
    out = torch.full_like(w.q, 7.0)
    pa.pa_varlen_forward(w.q, w.k_blocks, w.v_blocks, out, w.query_start_loc, w.seq_lens,
                         w.positions, bt, w.scale)
    assert pa.pa_device_status() == pa.PA_EINVAL
    assert bool((out == 7.0).all())
