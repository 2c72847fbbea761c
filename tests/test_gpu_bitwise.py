"""Decode equals prefill, bit for bit (tinyllm "Paged attention for decode in C", 2.4 and the
test equals_flash_attention_bitwise: blocks are tiles aligned to absolute positions, so a
token computed by the decode path and by the prefill path gets the same bits).

A prefill batch is run with PA_FLAG_BITWISE (every row on the 16-row warp-MMA kernel), then
every one of its tokens again as a decode token of its own (q_len 1, seq_len = position + 1,
the same table row and pool): out rows and lse must be identical.  The same holds without the
flag for sequences of at most 64 query rows per kv head, and for a token alone vs in a batch
(2.5, batch invariance).  The prefill results are also checked against the oracle.
"""
import math

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


def _run(pa, q, kb, vb, qsl, seq_lens, pos, table, w, bitwise, **kw):
    out = torch.full_like(q, float("nan"))
    lse = torch.full((q.shape[1], q.shape[0]), float("nan"), device=DEV)
    pa.pa_varlen_forward(q, kb, vb, out, qsl, seq_lens, pos, table, w.scale, causal=True,
                         sliding_window=w.sliding_window, lse=lse, bitwise=bitwise, **kw)
    assert pa.pa_device_status() == pa.PA_OK
    return out, lse


def _as_decode(w):
    """Every token of w as a decode token of its own: seq_len = position + 1, its sequence's
    table row, its query row."""
    qsl = w.query_start_loc.cpu().tolist()
    pos = w.positions.cpu()
    seq_of = torch.repeat_interleave(torch.arange(w.num_seqs),
                                     torch.tensor(w.q_lens_list))
    T = w.num_tokens
    return dict(qsl=torch.arange(T + 1, dtype=torch.int32, device=DEV),
                seq_lens=(pos + 1).to(torch.int32).to(DEV), pos=pos.to(DEV),
                table=w.block_tables[seq_of.to(DEV)].contiguous())


CASES = {
    # chunks of 17..300 tokens (68..1200 rows per kv head: prefill-class), GQA 4
    "gqa4": dict(seq_lens=[300, 777, 1500, 64, 2100], q_lens=[300, 100, 200, 64, 17],
                 num_heads=32, num_kv_heads=8, head_dim=128),
    # GQA 8 with a sliding window that cuts into the chunks
    "gqa8-window": dict(seq_lens=[900, 1700, 333], q_lens=[150, 40, 333], num_heads=64,
                        num_kv_heads=8, head_dim=128, sliding_window=200),
    # head size 64, MHA
    "d64": dict(seq_lens=[129, 520], q_lens=[129, 33], num_heads=8, num_kv_heads=8,
                head_dim=64),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_decode_equals_prefill_bitwise(pa, case):
    w = workloads.build(case, seed=sorted(CASES).index(case) + 81, device=DEV, **CASES[case])
    out_p, lse_p = _run(pa, w.q, w.k_blocks, w.v_blocks, w.query_start_loc, w.seq_lens,
                        w.positions, w.block_tables, w, bitwise=True)
    d = _as_decode(w)
    out_d, lse_d = _run(pa, w.q, w.k_blocks, w.v_blocks, d["qsl"], d["seq_lens"], d["pos"],
                        d["table"], w, bitwise=False)
    assert torch.equal(out_p, out_d), f"{case}: {int((out_p != out_d).sum())} elements differ"
    assert torch.equal(lse_p, lse_d)
    # and both are right
    st, ref, _ = oracle.varlen_attention(w.q.cpu(), w.k_blocks.cpu(), w.v_blocks.cpu(),
                                         w.query_start_loc, w.seq_lens, w.positions,
                                         w.block_tables, w.scale,
                                         sliding_window=w.sliding_window)
    assert st == oracle.OK
    assert_attn_close(out_p, ref, case)


def test_decode_equals_prefill_bitwise_fp8(pa):
    w = workloads.build("fp8", seed=91, device=DEV, **CASES["gqa8-window"])
    kb8, vb8 = workloads.fp8_pools(w)
    kw = dict(k_scale=0.125, v_scale=0.125)
    out_p, lse_p = _run(pa, w.q, kb8, vb8, w.query_start_loc, w.seq_lens, w.positions,
                        w.block_tables, w, bitwise=True, **kw)
    d = _as_decode(w)
    out_d, lse_d = _run(pa, w.q, kb8, vb8, d["qsl"], d["seq_lens"], d["pos"], d["table"], w,
                        bitwise=False, **kw)
    assert torch.equal(out_p, out_d) and torch.equal(lse_p, lse_d)


def test_decode_equals_prefill_bitwise_fp8_per_head_scales(pa):
    # one dequantisation scale per kv head: constant over a (sequence, kv head) unit, so the
    # decode and prefill rows still see the same arithmetic
    w = workloads.build("fp8-heads", seed=94, device=DEV, **CASES["gqa4"])
    sp = [2.0 + 4.0 * g for g in range(w.num_kv_heads)]
    kb8, vb8 = workloads.fp8_pools_per_head(w, sp)
    ks = torch.tensor([1.0 / x for x in sp], device=DEV)
    kw = dict(k_scales=ks, v_scales=ks * 0.7)
    out_p, lse_p = _run(pa, w.q, kb8, vb8, w.query_start_loc, w.seq_lens, w.positions,
                        w.block_tables, w, bitwise=True, **kw)
    d = _as_decode(w)
    out_d, lse_d = _run(pa, w.q, kb8, vb8, d["qsl"], d["seq_lens"], d["pos"], d["table"], w,
                        bitwise=False, **kw)
    assert torch.equal(out_p, out_d) and torch.equal(lse_p, lse_d)


def test_short_chunks_agree_without_the_flag(pa):
    # sequences of at most 64 rows per kv head stay on the warp-MMA kernel by default
    w = workloads.build("short", seq_lens=[40, 700, 1025, 16], q_lens=[16, 9, 16, 1],
                        num_heads=32, num_kv_heads=8, head_dim=128, seed=92, device=DEV,
                        sliding_window=500)
    out_p, lse_p = _run(pa, w.q, w.k_blocks, w.v_blocks, w.query_start_loc, w.seq_lens,
                        w.positions, w.block_tables, w, bitwise=False)
    d = _as_decode(w)
    out_d, lse_d = _run(pa, w.q, w.k_blocks, w.v_blocks, d["qsl"], d["seq_lens"], d["pos"],
                        d["table"], w, bitwise=False)
    assert torch.equal(out_p, out_d) and torch.equal(lse_p, lse_d)


def test_long_chunks_without_the_flag_are_close(pa):
    # prefill-class chunks take the tcgen05 kernel: within the tolerance of decode, not bitwise
    w = workloads.build("long", seed=93, device=DEV, **CASES["gqa4"])
    out_p, _ = _run(pa, w.q, w.k_blocks, w.v_blocks, w.query_start_loc, w.seq_lens,
                    w.positions, w.block_tables, w, bitwise=False)
    d = _as_decode(w)
    out_d, _ = _run(pa, w.q, w.k_blocks, w.v_blocks, d["qsl"], d["seq_lens"], d["pos"],
                    d["table"], w, bitwise=False)
    assert_attn_close(out_p, out_d.float(), "tcgen05 prefill vs decode")


def test_decode_token_alone_equals_in_batch(pa):
    # a windowed decode token alone and among 63 others (different lengths, tiles, units)
    w = workloads.named(2, seed=3, device=DEV)
    w.sliding_window = 300
    out_b, lse_b = _run(pa, w.q, w.k_blocks, w.v_blocks, w.query_start_loc, w.seq_lens,
                        w.positions, w.block_tables, w, bitwise=False)
    for s in (0, 17, 63):
        sub = workloads.subset(w, [s])
        out_s, lse_s = _run(pa, sub.q, w.k_blocks, w.v_blocks, sub.query_start_loc,
                            sub.seq_lens, sub.positions, sub.block_tables, w, bitwise=False)
        assert torch.equal(out_s[0], out_b[s]) and torch.equal(lse_s[:, 0], lse_b[:, s])


def test_unknown_flags_are_rejected(pa):
    import ctypes

    w = workloads.build("flags", seq_lens=[5], q_lens=[1], num_heads=4, num_kv_heads=2,
                        head_dim=64, seed=1, device=DEV)
    out = torch.empty_like(w.q)
    ws = pa.workspace_for(w.q, w.k_blocks, w.query_start_loc, w.block_tables)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = pa._lib.pa_varlen_forward_ex(
        p(w.q), p(w.k_blocks), p(w.v_blocks), p(out), p(w.query_start_loc), p(w.seq_lens),
        p(w.positions), p(w.block_tables), 1, 1, 4, 2, 64, 16, w.num_blocks,
        w.block_tables.shape[1], pa.PA_BF16, pa.PA_BF16, w.scale, 1, 0, None, None, 1.0, 1.0,
        2, p(ws), ws.numel(), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == pa.PA_EINVAL
    assert pa.pa_device_status() == pa.PA_OK
