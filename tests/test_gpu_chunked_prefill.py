"""Chunked-context prefill from the library's pieces, as the vllm.cpp MLA-prefill page builds
it: for a chunk of n new tokens after c context positions,

  1. context attention: every new token attends to all c context positions (no causal mask),
     with its log-sum-exp (pa_varlen_forward_ex, causal = 0, seq_len = c);
  2. new-token attention: the chunk's own K/V rows, gathered out of the pool (pa_gather_kv) and
     scattered into a pool of their own (pa_slot_mapping, pa_reshape_and_cache), attended
     causally at positions 0 .. n-1, with its log-sum-exp;
  3. pa_merge_attn_states of the two (prefix = context, suffix = new tokens).

The merged result must equal direct causal attention over all c + n positions (the oracle),
and its lse the direct lse.  Tokens without context take the new-token part as is
(prefill_tokens_with_context counts the leading tokens that have context)."""
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


def _i32(x):
    return torch.tensor(x, dtype=torch.int32, device=DEV)


def _chunked(pa, w, ctx, new):
    """Steps 1-3 above for sequences with c >= 1 context positions."""
    T, H, D = w.q.shape
    Hkv, bs = w.num_kv_heads, w.block_size
    qsl = w.query_start_loc
    # 1. context attention: positions are only checked against seq_len = c here (no mask)
    out_c = torch.empty_like(w.q)
    lse_c = torch.empty((H, T), device=DEV)
    pos_c = _i32([c - 1 for c, n in zip(ctx, new) for _ in range(n)])
    pa.pa_varlen_forward(w.q, w.k_blocks, w.v_blocks, out_c, qsl, _i32(ctx), pos_c,
                         w.block_tables, w.scale, causal=False, lse=lse_c)
    # 2. the chunk's own K/V in a pool of its own, attended causally at 0 .. n-1
    kd = torch.empty((T, Hkv, D), dtype=w.k_blocks.dtype, device=DEV)
    vd = torch.empty_like(kd)
    pa.pa_gather_kv(w.k_blocks, w.v_blocks, kd, vd, qsl, w.block_tables, seq_starts=_i32(ctx))
    need = [(n + bs - 1) // bs for n in new]
    table = torch.zeros((len(new), max(need)), dtype=torch.int32)
    nxt = 0
    for s, k in enumerate(need):
        table[s, :k] = torch.arange(nxt, nxt + k)
        nxt += k
    table = table.to(DEV)
    k2 = torch.zeros((nxt, bs, Hkv, D), dtype=w.k_blocks.dtype, device=DEV)
    v2 = torch.zeros_like(k2)
    pos_n = _i32([j for n in new for j in range(n)])
    slots = pa.pa_slot_mapping(qsl, pos_n, table, bs, nxt)
    pa.pa_reshape_and_cache(kd, vd, k2, v2, slots)
    out_n = torch.empty_like(w.q)
    lse_n = torch.empty((H, T), device=DEV)
    pa.pa_varlen_forward(w.q, k2, v2, out_n, qsl, _i32(new), pos_n, table, w.scale, causal=True,
                         lse=lse_n)
    # 3. merge
    out = torch.empty_like(w.q)
    lse = torch.empty((H, T), device=DEV)
    pa.pa_merge_attn_states(out, lse, out_c, lse_c, out_n, lse_n)
    assert pa.pa_device_status() == pa.PA_OK
    return out, lse


@pytest.mark.parametrize("H,Hkv", [(32, 8), (8, 8)])
def test_chunked_context_prefill_equals_full_attention(pa, H, Hkv):
    # chunks on both attention kernels: long ones (tcgen05) and short ones (warp MMA)
    ctx = [1, 37, 300, 1024, 2000, 16]
    new = [200, 65, 512, 130, 9, 1]
    w = workloads.build("chunked", seq_lens=[c + n for c, n in zip(ctx, new)], q_lens=new,
                        num_heads=H, num_kv_heads=Hkv, head_dim=128, seed=H + 3, device=DEV)
    out, lse = _chunked(pa, w, ctx, new)
    st, ref, ref_lse = oracle.varlen_attention(w.q.cpu(), w.k_blocks.cpu(), w.v_blocks.cpu(),
                                               w.query_start_loc, w.seq_lens, w.positions,
                                               w.block_tables, w.scale, want_lse=True)
    assert st == oracle.OK
    assert_attn_close(out, ref, "chunked vs full")
    err = (lse.cpu() - ref_lse).abs()
    assert float(err.max()) < 1e-3 + 1e-4 * float(ref_lse.abs().max()), float(err.max())


def test_tokens_past_the_context_count_take_the_new_part(pa):
    # in a batch whose later tokens have no context, only the leading
    # prefill_tokens_with_context tokens are merged; the others copy the new-token attention
    T, H, D = 103, 16, 128
    g = torch.Generator(device=DEV).manual_seed(9)
    prefix = torch.randn((T, H, D), generator=g, device=DEV).to(torch.bfloat16)
    suffix = torch.randn((T, H, D), generator=g, device=DEV).to(torch.bfloat16)
    lse_p = torch.randn((H, T), generator=g, device=DEV)
    lse_s = torch.randn((H, T), generator=g, device=DEV)
    merged = torch.empty_like(prefix)
    lse = torch.empty((H, T), device=DEV)
    P = 70
    pa.pa_merge_attn_states(merged, lse, prefix, lse_p, suffix, lse_s,
                            prefill_tokens_with_context=P)
    assert pa.pa_device_status() == pa.PA_OK
    assert torch.equal(merged[P:], suffix[P:]) and torch.equal(lse[:, P:], lse_s[:, P:])
    assert not torch.equal(merged[:P], suffix[:P])
