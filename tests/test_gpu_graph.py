"""A serving step captured in a CUDA graph: pa_cache_and_attend (slot mapping, scatter, plan
and attention) issues only stream-ordered launches, allocates nothing and never synchronises,
so the step can be captured once and replayed.  Replays must give the same slots, pool and
output bits as eager calls, for the decode batch and for a mixed batch whose prefill chunks
take the tcgen05 kernel, and a replay after the metadata changed (the next decode step,
every context one longer) must match an eager call on the new metadata."""
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


def _step(pa, w, kb, vb, out, ws, slots, stream):
    pa.pa_cache_and_attend(w.k_new, w.v_new, w.q, kb, vb, out, w.query_start_loc, w.seq_lens,
                           w.positions, w.block_tables, w.scale, causal=w.causal,
                           sliding_window=w.sliding_window, workspace=ws, slot_mapping=slots,
                           stream=stream)


@pytest.mark.parametrize("case", ["decode", "mixed"])
def test_captured_step_replays_bitwise(pa, case):
    if case == "decode":  # the decode batch's shape, one spare table column for the next step
        g0 = torch.Generator().manual_seed(31)
        lens = torch.randint(512, 4097, (64,), generator=g0).tolist()
        need = sum((n + 15) // 16 for n in lens)
        w = workloads.build("graph-decode", seq_lens=lens, q_lens=[1] * 64, num_heads=32,
                            num_kv_heads=8, head_dim=128, seed=31, device=DEV,
                            num_blocks=need + 64,
                            extra_table_cols=1)
    else:
        w = workloads.build("graph-mixed", seq_lens=[600, 1300, 90, 2000], q_lens=[512, 130, 1, 1],
                            num_heads=32, num_kv_heads=8, head_dim=128, seed=32, device=DEV)
    ws = pa.workspace_for(w.q, w.k_blocks, w.query_start_loc, w.block_tables)
    # eager reference on a copy of the pool
    kb_e, vb_e = w.k_blocks.clone(), w.v_blocks.clone()
    out_e = torch.empty_like(w.q)
    slots_e = torch.empty(w.num_tokens, dtype=torch.int32, device=DEV)
    _step(pa, w, kb_e, vb_e, out_e, ws, slots_e, None)
    assert pa.pa_device_status() == pa.PA_OK
    # capture on a side stream, then replay twice
    kb_g, vb_g = w.k_blocks.clone(), w.v_blocks.clone()
    out_g = torch.full_like(w.q, float("nan"))
    slots_g = torch.full((w.num_tokens,), -7, dtype=torch.int32, device=DEV)
    ws_g = torch.empty_like(ws)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # one eager run on the capture stream first (lazy set-up)
        _step(pa, w, kb_g, vb_g, out_g, ws_g, slots_g, s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        _step(pa, w, kb_g, vb_g, out_g, ws_g, slots_g, s)
    for _ in range(2):
        out_g.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert pa.pa_device_status() == pa.PA_OK
        assert torch.equal(out_g, out_e) and torch.equal(slots_g, slots_e)
        assert torch.equal(kb_g, kb_e) and torch.equal(vb_g, vb_e)
    if case != "decode":
        return
    # the next decode step: the metadata buffers the graph reads are updated in place.  A
    # sequence whose new token opens a block gets a block of its own in the spare table column
    # (unused entries hold 0, a block another sequence owns: two new tokens would then share
    # a slot, and the pool would depend on the order of their writes)
    lens_now = w.seq_lens.tolist()
    tables = w.block_tables.cpu()
    used = {int(tables[s_, b_]) for s_, n in enumerate(lens_now) for b_ in range((n + 15) // 16)}
    free = [i for i in range(w.num_blocks) if i not in used]
    opening = [s_ for s_, n in enumerate(lens_now) if n % 16 == 0]
    assert len(free) >= len(opening)
    for s_, blk in zip(opening, free):
        tables[s_, lens_now[s_] // 16] = blk
    w.block_tables.copy_(tables)
    w.seq_lens.add_(1)
    w.positions.add_(1)
    kb_e2, vb_e2 = kb_e.clone(), vb_e.clone()
    out_e2 = torch.empty_like(w.q)
    slots_e2 = torch.empty_like(slots_e)
    _step(pa, w, kb_e2, vb_e2, out_e2, ws, slots_e2, None)
    g.replay()
    torch.cuda.synchronize()
    assert pa.pa_device_status() == pa.PA_OK
    assert torch.equal(slots_g, slots_e2) and torch.equal(out_g, out_e2)
