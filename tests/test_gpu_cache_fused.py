"""pa_slot_mapping_and_cache: the slot mapping (TensorSharp class summary, "slot = blockId *
blockSize + offsetInBlock"; tinyllm 2.1) and the scatter (TensorSharp WriteKvToPagedPool) in
one launch for decode-sized batches.  Against the oracle's slot mapping and scatter (slots and
pools bit-exact), against the two separate calls, on the invalid cases (nothing written,
PA_EINVAL), on batches past the one-launch limits and on odd row sizes."""
import pytest
import torch

import oracle
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


def _oracle(w, kb, vb):
    st, slots = oracle.slot_mapping(w.query_start_loc, w.positions, w.block_tables,
                                    w.block_size, w.num_blocks)
    assert st == oracle.OK
    okb, ovb = kb.cpu().clone(), vb.cpu().clone()
    assert oracle.reshape_and_cache(w.k_new.cpu(), w.v_new.cpu(), okb, ovb, slots,
                                    w.block_size) == oracle.OK
    return slots, okb, ovb


def _bits(t):
    return t.cpu().view(torch.uint8) if t.dtype == torch.float8_e4m3fn else t.cpu()


CASES = {
    "decode-64": dict(cfg=2),
    "mixed-small": dict(seq_lens=[1, 17, 33, 50, 300], q_lens=[1, 17, 8, 1, 40], num_heads=8,
                        num_kv_heads=2, head_dim=64),
    "empty-seqs": dict(seq_lens=[5, 9, 40, 12], q_lens=[0, 3, 0, 12], num_heads=4,
                       num_kv_heads=4, head_dim=32),
    "big-3000": dict(seq_lens=[1500, 2000], q_lens=[1500, 1500], num_heads=8, num_kv_heads=8,
                     head_dim=64),  # 3000 tokens: past the one-launch limit
    "odd-rows-f32": dict(seq_lens=[7, 30], q_lens=[7, 2], num_heads=3, num_kv_heads=3,
                         head_dim=7, dtype=torch.float32),
    "odd-rows-bf16": dict(seq_lens=[7, 30], q_lens=[7, 2], num_heads=3, num_kv_heads=3,
                          head_dim=7),
}


def _build(name):
    kw = dict(CASES[name])
    if "cfg" in kw:
        return workloads.named(kw["cfg"], seed=4, device=DEV)
    return workloads.build(name, seed=sorted(CASES).index(name) + 5, device=DEV, **kw)


@pytest.mark.parametrize("case", sorted(CASES))
def test_fused_equals_oracle_and_separate_calls(pa, case):
    w = _build(case)
    kb0, vb0 = w.k_blocks.clone(), w.v_blocks.clone()
    slots = pa.pa_slot_mapping_and_cache(w.k_new, w.v_new, w.k_blocks, w.v_blocks,
                                         w.query_start_loc, w.positions, w.block_tables)
    assert pa.pa_device_status() == pa.PA_OK
    oslots, okb, ovb = _oracle(w, kb0, vb0)
    assert torch.equal(slots.cpu(), oslots)
    assert torch.equal(w.k_blocks.cpu(), okb) and torch.equal(w.v_blocks.cpu(), ovb)
    # the two separate calls give the same bits
    kb1, vb1 = kb0.clone(), vb0.clone()
    s1 = pa.pa_slot_mapping(w.query_start_loc, w.positions, w.block_tables, w.block_size,
                            w.num_blocks)
    pa.pa_reshape_and_cache(w.k_new, w.v_new, kb1, vb1, s1)
    assert pa.pa_device_status() == pa.PA_OK
    assert torch.equal(s1, slots) and torch.equal(kb1, w.k_blocks) and torch.equal(vb1, w.v_blocks)


@pytest.mark.parametrize("S,q", [(1024, 2), (683, 3), (2047, 1), (2048, 1)])
def test_fused_at_its_limits(pa, S, q):
    # 2048 tokens and 2047 sequences take the one-launch kernel; 2049 tokens (683 x 3) or 2048
    # sequences take the two launches
    lens = [q + (7 * i) % 60 for i in range(S)]
    w = workloads.build("limits", seq_lens=lens, q_lens=[q] * S, num_heads=4, num_kv_heads=2,
                        head_dim=32, seed=S + q, device=DEV)
    kb0, vb0 = w.k_blocks.clone(), w.v_blocks.clone()
    slots = pa.pa_slot_mapping_and_cache(w.k_new, w.v_new, w.k_blocks, w.v_blocks,
                                         w.query_start_loc, w.positions, w.block_tables)
    assert pa.pa_device_status() == pa.PA_OK
    oslots, okb, ovb = _oracle(w, kb0, vb0)
    assert torch.equal(slots.cpu(), oslots)
    assert torch.equal(w.k_blocks.cpu(), okb) and torch.equal(w.v_blocks.cpu(), ovb)


def test_fused_fp8_rows(pa):
    w = workloads.build("fp8", seq_lens=[9, 40], q_lens=[9, 3], num_heads=3, num_kv_heads=3,
                        head_dim=7, seed=8, device=DEV)
    k8 = w.k_new.float().to(torch.float8_e4m3fn)
    v8 = w.v_new.float().to(torch.float8_e4m3fn)
    kb = torch.zeros(w.k_blocks.shape, dtype=torch.float8_e4m3fn, device=DEV)
    vb = torch.zeros_like(kb)
    slots = pa.pa_slot_mapping_and_cache(k8, v8, kb, vb, w.query_start_loc, w.positions,
                                         w.block_tables)
    assert pa.pa_device_status() == pa.PA_OK
    st, oslots = oracle.slot_mapping(w.query_start_loc, w.positions, w.block_tables,
                                     w.block_size, w.num_blocks)
    okb, ovb = kb.cpu().clone(), vb.cpu().clone()
    assert oracle.reshape_and_cache(k8.cpu(), v8.cpu(), okb, ovb, oslots, w.block_size) == 0
    assert torch.equal(slots.cpu(), oslots)
    assert torch.equal(_bits(kb), _bits(okb)) and torch.equal(_bits(vb), _bits(ovb))


def _bad(pa, w, what):
    kb0, vb0 = w.k_blocks.clone(), w.v_blocks.clone()
    slots = pa.pa_slot_mapping_and_cache(w.k_new, w.v_new, w.k_blocks, w.v_blocks,
                                         w.query_start_loc, w.positions, w.block_tables)
    assert pa.pa_device_status() == pa.PA_EINVAL, what
    assert torch.equal(w.k_blocks, kb0) and torch.equal(w.v_blocks, vb0), what
    return slots


def test_invalid_tokens_write_nothing(pa):
    mk = lambda: workloads.build("bad", seq_lens=[20, 40, 7], q_lens=[4, 1, 7], num_heads=4,
                                 num_kv_heads=2, head_dim=32, seed=11, device=DEV)
    w = mk()  # a position past the table row
    w.positions[2] = w.block_tables.shape[1] * w.block_size + 3
    s = _bad(pa, w, "position past the table")
    assert int(s[2]) == -1 and int(s[0]) >= 0
    w = mk()  # a block id outside the pool
    w.block_tables[1, 2] = w.num_blocks + 5
    _bad(pa, w, "block id outside the pool")
    w = mk()  # a negative position
    w.positions[5] = -1
    _bad(pa, w, "negative position")
    w = mk()  # decreasing query_start_loc
    w.query_start_loc[1] = 6
    w.query_start_loc[2] = 5
    _bad(pa, w, "decreasing query_start_loc")
    w = mk()  # the last token belongs to no sequence
    w.query_start_loc[3] = w.num_tokens - 1
    _bad(pa, w, "uncovered token")
    assert pa.pa_device_status() == pa.PA_OK


# ------------------------------------------------------------------- pa_cache_and_attend

STEP_CASES = {
    "decode-64": dict(cfg=2),
    # prefill chunks (tcgen05 kernel) and decode tokens, windowed
    "mixed": dict(seq_lens=[600, 1300, 90, 2000, 4000], q_lens=[512, 130, 1, 1, 1],
                  num_heads=32, num_kv_heads=8, head_dim=128, sliding_window=1000),
    # past the one-launch limits: the calls run one after the other
    "big-3000": dict(seq_lens=[1500, 2000], q_lens=[1500, 1500], num_heads=8, num_kv_heads=8,
                     head_dim=64),
}


def _step_build(name):
    kw = dict(STEP_CASES[name])
    if "cfg" in kw:
        return workloads.named(kw["cfg"], seed=6, device=DEV)
    return workloads.build(name, seed=sorted(STEP_CASES).index(name) + 21, device=DEV, **kw)


def _two_calls(pa, w, kb, vb):
    s = pa.pa_slot_mapping_and_cache(w.k_new, w.v_new, kb, vb, w.query_start_loc, w.positions,
                                     w.block_tables)
    out = torch.full_like(w.q, float("nan"))
    pa.pa_varlen_forward(w.q, kb, vb, out, w.query_start_loc, w.seq_lens, w.positions,
                         w.block_tables, w.scale, causal=w.causal,
                         sliding_window=w.sliding_window)
    return s, out


@pytest.mark.parametrize("case", sorted(STEP_CASES))
def test_cache_and_attend_equals_the_two_calls(pa, case):
    w = _step_build(case)
    kb1, vb1 = w.k_blocks.clone(), w.v_blocks.clone()
    s1, out1 = _two_calls(pa, w, kb1, vb1)
    assert pa.pa_device_status() == pa.PA_OK
    out = torch.full_like(w.q, float("nan"))
    s = pa.pa_cache_and_attend(w.k_new, w.v_new, w.q, w.k_blocks, w.v_blocks, out,
                               w.query_start_loc, w.seq_lens, w.positions, w.block_tables,
                               w.scale, causal=w.causal, sliding_window=w.sliding_window)
    assert pa.pa_device_status() == pa.PA_OK
    assert torch.equal(s, s1)
    assert torch.equal(w.k_blocks, kb1) and torch.equal(w.v_blocks, vb1)
    assert torch.equal(out, out1)


def test_cache_and_attend_failures_leave_out_untouched(pa):
    w = _step_build("decode-64")
    w.block_tables[3, 0] = w.num_blocks + 1  # a bad block id: the scatter and the plan fail
    out = torch.full_like(w.q, 7.0)
    kb0, vb0 = w.k_blocks.clone(), w.v_blocks.clone()
    pa.pa_cache_and_attend(w.k_new, w.v_new, w.q, w.k_blocks, w.v_blocks, out,
                           w.query_start_loc, w.seq_lens, w.positions, w.block_tables, w.scale)
    assert pa.pa_device_status() == pa.PA_EINVAL
    assert bool((out == 7.0).all())
    w = _step_build("decode-64")
    w.seq_lens[5] = 0  # a context the plan rejects (the slots are fine: the rows are written)
    out = torch.full_like(w.q, 7.0)
    pa.pa_cache_and_attend(w.k_new, w.v_new, w.q, w.k_blocks, w.v_blocks, out,
                           w.query_start_loc, w.seq_lens, w.positions, w.block_tables, w.scale)
    assert pa.pa_device_status() == pa.PA_EINVAL
    assert bool((out == 7.0).all())
    assert pa.pa_device_status() == pa.PA_OK
