"""GPU parity: the CUDA path through the C ABI against the CPU oracle, on the same seeded
inputs.  Indexing work (slot mapping, scatter, gather) must be bit-exact; attention within
|gpu - oracle| <= 2e-3 + 1e-2 |oracle| elementwise."""
import math

import pytest
import torch

import oracle
from paged_kv_cache_31_gb300 import workloads
from tests.gpu_helpers import assert_attn_close, oracle_attention

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_31_gb300 import binding

    assert binding.pa_device_status() == binding.PA_OK
    return binding


DEV = "cuda"


def _step(pa, w, kb=None, vb=None):
    """Slot mapping -> scatter of the new tokens -> varlen attention.  Returns
    (slots, kb, vb, out) on the device."""
    slots = pa.pa_slot_mapping(w.query_start_loc, w.positions, w.block_tables, w.block_size,
                               w.num_blocks)
    kb = w.k_blocks.clone() if kb is None else kb
    vb = w.v_blocks.clone() if vb is None else vb
    pa.pa_reshape_and_cache(w.k_new, w.v_new, kb, vb, slots)
    out = torch.full_like(w.q, float("nan"))
    pa.pa_varlen_forward(w.q, kb, vb, out, w.query_start_loc, w.seq_lens, w.positions,
                         w.block_tables, w.scale, causal=w.causal,
                         sliding_window=w.sliding_window)
    assert pa.pa_device_status() == pa.PA_OK
    return slots, kb, vb, out


def _oracle_cache(w, slots_gpu):
    st, oslots = oracle.slot_mapping(w.query_start_loc, w.positions, w.block_tables,
                                     w.block_size, w.num_blocks)
    assert st == oracle.OK
    assert torch.equal(slots_gpu.cpu(), oslots), "slot mapping differs"
    okb, ovb = w.k_blocks.cpu().clone(), w.v_blocks.cpu().clone()
    assert oracle.reshape_and_cache(w.k_new.cpu(), w.v_new.cpu(), okb, ovb, oslots,
                                    w.block_size) == oracle.OK
    return okb, ovb


# ------------------------------------------------------------------------------------------
# the five workloads, at sizes the oracle finishes in seconds


@pytest.mark.parametrize("cfg", [1, 2, 3, 5])
def test_varlen_small_workloads(pa, cfg):
    w = workloads.named(cfg, small=True, device=DEV)
    slots, kb, vb, out = _step(pa, w)
    okb, ovb = _oracle_cache(w, slots)
    assert torch.equal(kb.cpu(), okb) and torch.equal(vb.cpu(), ovb), "scatter differs"
    ref = oracle_attention(w, okb, ovb)
    assert_attn_close(out, ref, w.name)


def test_tiny_mixed_fp32_full(pa):
    w = workloads.named(1, device=DEV)
    slots, kb, vb, out = _step(pa, w)
    okb, ovb = _oracle_cache(w, slots)
    assert torch.equal(kb.cpu(), okb) and torch.equal(vb.cpu(), ovb)
    assert_attn_close(out, oracle_attention(w, okb, ovb), w.name)


@pytest.mark.parametrize("kw", [
    dict(head_dim=64, num_heads=8, num_kv_heads=2),                      # tensor-core path, D 64
    dict(head_dim=128, num_heads=32, num_kv_heads=1),                    # G = 32: 2 tiles per token
    dict(head_dim=128, num_heads=16, num_kv_heads=16),                   # G = 1 (MHA)
    dict(head_dim=96, num_heads=8, num_kv_heads=2),                      # general kernel: D 96
    dict(head_dim=128, num_heads=8, num_kv_heads=2, block_size=32),      # general kernel: b 32
    dict(head_dim=128, num_heads=8, num_kv_heads=2, causal=False, sliding_window=50),
    dict(head_dim=128, num_heads=8, num_kv_heads=4, sliding_window=33),
])
def test_varlen_shapes(pa, kw):
    lens, qlens = [1, 16, 17, 100, 257, 31], [1, 16, 5, 40, 3, 0]
    w = workloads.build("shape", seq_lens=lens, q_lens=qlens, seed=5, device=DEV, **kw)
    slots, kb, vb, out = _step(pa, w)
    okb, ovb = _oracle_cache(w, slots)
    assert_attn_close(out, oracle_attention(w, okb, ovb), str(kw))


@pytest.mark.parametrize("kw", [
    dict(head_dim=256, num_heads=4, num_kv_heads=2),                     # largest head size
    dict(head_dim=32, num_heads=8, num_kv_heads=2),                      # small head size
    dict(head_dim=128, num_heads=8, num_kv_heads=2, block_size=8),       # small blocks
    dict(head_dim=64, num_heads=4, num_kv_heads=2, block_size=64),       # large blocks
    dict(head_dim=128, num_heads=64, num_kv_heads=1),                    # G = 64: 2 tokens per
])                                                                       # tcgen05 query tile
def test_varlen_extreme_shapes(pa, kw):
    lens, qlens = [1, 64, 65, 300, 129], [1, 64, 40, 70, 1]
    w = workloads.build("extreme", seq_lens=lens, q_lens=qlens, seed=7, device=DEV, **kw)
    slots, kb, vb, out = _step(pa, w)
    okb, ovb = _oracle_cache(w, slots)
    assert_attn_close(out, oracle_attention(w, okb, ovb), str(kw))


def test_varlen_fp32_query_bf16_pool(pa):
    w = workloads.build("mix", seq_lens=[40, 90], q_lens=[3, 1], num_heads=4, num_kv_heads=2,
                        head_dim=64, seed=9, device=DEV)
    q32 = w.q.float()
    out = torch.empty_like(q32)
    pa.pa_varlen_forward(q32, w.k_blocks, w.v_blocks, out, w.query_start_loc, w.seq_lens,
                         w.positions, w.block_tables, w.scale)
    assert pa.pa_device_status() == pa.PA_OK
    st, ref, _ = oracle.varlen_attention(q32.cpu(), w.k_blocks.cpu(), w.v_blocks.cpu(),
                                         w.query_start_loc, w.seq_lens, w.positions,
                                         w.block_tables, w.scale)
    assert_attn_close(out, ref, "fp32 q / bf16 pool")


def test_unwritten_tail_slots_are_never_read(pa):
    """Slots past seq_len in a sequence's last block may hold anything (here NaN): no output
    may depend on them."""
    w = workloads.build("nan", seq_lens=[17, 33, 250], q_lens=[1, 5, 1], num_heads=8,
                        num_kv_heads=2, head_dim=128, seed=13, device=DEV)
    kb, vb = w.k_blocks.clone(), w.v_blocks.clone()
    for s, n in enumerate(w.seq_lens_list):
        last = int(w.block_tables[s, (n - 1) // 16])
        kb[last, n % 16 or 16:] = float("nan")
        vb[last, n % 16 or 16:] = float("nan")
    slots, kb, vb, out = _step(pa, w, kb, vb)
    assert torch.isfinite(out.float()).all()
    okb, ovb = kb.cpu(), vb.cpu()
    assert_attn_close(out, oracle_attention(w, okb, ovb), "nan tail")


# ------------------------------------------------------------------------------------------
# full-size workloads: every output of the decode, mixed and shared-prefix batches


def test_decode_batch_full(pa):
    w = workloads.named(2, device=DEV)
    slots, kb, vb, out = _step(pa, w)
    okb, ovb = _oracle_cache(w, slots)
    assert torch.equal(kb.cpu(), okb) and torch.equal(vb.cpu(), ovb)
    assert_attn_close(out, oracle_attention(w, okb, ovb), w.name)


def test_mixed_window_batch_full(pa):
    """All 4344 rows of the mixed batch (248 decode tokens and the 8 prefill chunks of 512
    tokens, window 4096), as one call runs them: the decode tiles on the warp-MMA kernel and
    the chunks on the tcgen05 kernel, both in their persistent longest-first orders."""
    w = workloads.named(3, device=DEV)
    slots, kb, vb, out = _step(pa, w)
    okb, ovb = _oracle_cache(w, slots)
    assert torch.equal(kb.cpu(), okb) and torch.equal(vb.cpu(), ovb)
    ref = oracle_attention(w, okb, ovb)
    assert_attn_close(out, ref, w.name)


def test_shared_prefix_full(pa):
    """All 256 fork sequences (128 shared physical blocks, private tails) against the oracle."""
    w = workloads.named(5, device=DEV)
    slots, kb, vb, out = _step(pa, w)
    okb, ovb = _oracle_cache(w, slots)
    assert torch.equal(kb.cpu(), okb) and torch.equal(vb.cpu(), ovb)
    assert_attn_close(out, oracle_attention(w, okb, ovb), w.name)


def test_shared_prefix_each_sequence_alone_equals_batch(pa):
    """The shared-prefix workload's own check: each of the 256 sequences, run alone through
    pa_varlen_forward on the same pool (the 128 shared blocks included), gives its row of the
    256-sequence batch bit for bit."""
    w = workloads.named(5, device=DEV)
    slots, kb, vb, batch = _step(pa, w)
    qsl = w.query_start_loc.cpu().tolist()
    assert (w.block_tables[:, :128] == w.block_tables[0, :128]).all(), "prefix not shared"
    ws = pa.workspace_for(w.q, kb, w.query_start_loc, w.block_tables)
    for s in range(w.num_seqs):
        a, b = qsl[s], qsl[s + 1]
        one = torch.full_like(w.q[a:b], 7.25)
        pa.pa_varlen_forward(w.q[a:b], kb, vb, one,
                             torch.tensor([0, b - a], dtype=torch.int32, device=DEV),
                             w.seq_lens[s:s + 1], w.positions[a:b],
                             w.block_tables[s:s + 1].contiguous(), w.scale, causal=w.causal,
                             sliding_window=w.sliding_window, workspace=ws)
        assert torch.equal(one, batch[a:b]), f"sequence {s} differs alone vs in the batch"
    assert pa.pa_device_status() == pa.PA_OK


# ------------------------------------------------------------------------------------------
# split-KV decode


def _split_buffers(w, dev=DEV):
    S, H, D, P = w.num_seqs, w.num_heads, w.head_dim, w.max_partitions()
    ml = torch.full((S, H, P), float("nan"), device=dev)
    es = torch.full((S, H, P), float("nan"), device=dev)
    to = torch.full((S, H, P, D), float("nan"), device=dev)
    return ml, es, to


def _mask_partitions(w, ml, es):
    for s, p in enumerate(w.masked_partition):
        ml[s, :, p] = -math.inf if s % 2 == 0 else math.inf
        es[s, :, p] = 0.0


@pytest.mark.parametrize("window", [0, 700])
def test_splitkv_small(pa, window):
    w = workloads.named(4, small=True, device=DEV)
    P = w.partition_size
    ml, es, to = _split_buffers(w)
    pa.pa_decode_splitkv_partials(w.q, w.k_blocks, w.v_blocks, ml, es, to, w.seq_lens,
                                  w.block_tables, w.scale, P, sliding_window=window)
    assert pa.pa_device_status() == pa.PA_OK
    st, oml, oes, oto = oracle.splitkv_partials(w.q, w.k_blocks, w.v_blocks, w.seq_lens,
                                                w.block_tables, w.scale, P, w.max_partitions(),
                                                window)
    assert st == oracle.OK
    empty = oes == 0
    assert torch.equal(es.cpu() == 0, empty), "empty partitions differ"
    assert torch.all(ml.cpu()[empty] == -math.inf) and torch.all(to.cpu()[empty] == 0)
    assert_attn_close(ml.cpu()[~empty], oml[~empty], "max_logits")
    assert_attn_close(es.cpu()[~empty], oes[~empty], "exp_sums")
    assert_attn_close(to, oto, "tmp_out")
    # reduce, unmasked and with one masked partition per sequence (the -inf merge case)
    for masked in (False, True):
        ml2, es2 = ml.clone(), es.clone()
        oml2, oes2 = oml.clone(), oes.clone()
        if masked:
            _mask_partitions(w, ml2, es2)
            _mask_partitions(w, oml2, oes2)
        out = torch.empty_like(w.q)
        pa.pa_decode_splitkv_reduce(out, ml2, es2, to, w.seq_lens, P)
        assert pa.pa_device_status() == pa.PA_OK
        st, ref = oracle.splitkv_reduce(oml2, oes2, oto, w.seq_lens, P)
        assert st == oracle.OK
        assert_attn_close(out, ref, f"reduce masked={masked}")
    # the one-call form equals partials + reduce
    out1 = torch.empty_like(w.q)
    pa.pa_decode_splitkv(w.q, w.k_blocks, w.v_blocks, out1, ml, es, to, w.seq_lens,
                         w.block_tables, w.scale, P, sliding_window=window)
    assert pa.pa_device_status() == pa.PA_OK
    st, ref = oracle.splitkv_reduce(oml, oes, oto, w.seq_lens, P)
    assert_attn_close(out1, ref, "pa_decode_splitkv")


def test_splitkv_all_partitions_masked(pa):
    w = workloads.named(4, small=True, device=DEV)
    ml, es, to = _split_buffers(w)
    pa.pa_decode_splitkv_partials(w.q, w.k_blocks, w.v_blocks, ml, es, to, w.seq_lens,
                                  w.block_tables, w.scale, w.partition_size)
    ml[:] = -math.inf
    ml[:, :, 1::2] = math.inf
    es[:] = 0
    out = torch.empty_like(w.q, dtype=torch.float32)
    pa.pa_decode_splitkv_reduce(out, ml, es, to, w.seq_lens, w.partition_size)
    assert pa.pa_device_status() == pa.PA_OK
    assert torch.equal(out, to[:, :, 0]), "all masked must pass partition 0 through"


def test_splitkv_long_context_full_sampled(pa):
    """8 x 131072 positions, H 64 / Hkv 8: GPU partials of two sequences against the oracle's,
    and every sequence's reduced output (one masked partition each) against the oracle's
    reduce of the GPU partials' oracle counterparts for those sequences."""
    w = workloads.named(4, device=DEV)
    P, MP = w.partition_size, w.max_partitions()
    ml, es, to = _split_buffers(w)
    pa.pa_decode_splitkv_partials(w.q, w.k_blocks, w.v_blocks, ml, es, to, w.seq_lens,
                                  w.block_tables, w.scale, P)
    _mask_partitions(w, ml, es)
    out = torch.empty_like(w.q)
    pa.pa_decode_splitkv_reduce(out, ml, es, to, w.seq_lens, P)
    assert pa.pa_device_status() == pa.PA_OK
    kb, vb = w.k_blocks.cpu(), w.v_blocks.cpu()
    for s in (1, 6):
        st, oml, oes, oto = oracle.splitkv_partials(w.q[s:s + 1].cpu(), kb, vb,
                                                    w.seq_lens[s:s + 1].cpu(),
                                                    w.block_tables[s:s + 1].cpu(), w.scale, P, MP)
        assert st == oracle.OK
        assert_attn_close(to[s:s + 1].cpu(), oto, f"tmp_out seq {s}")
        mp = w.masked_partition[s]
        ok = torch.ones_like(oes, dtype=torch.bool)
        ok[0, :, mp] = False
        assert_attn_close(es[s:s + 1].cpu()[ok], oes[ok], f"exp_sums seq {s}")
        oml[0, :, mp] = -math.inf if s % 2 == 0 else math.inf  # as _mask_partitions did on the GPU
        oes[0, :, mp] = 0.0
        st, ref = oracle.splitkv_reduce(oml, oes, oto, w.seq_lens[s:s + 1].cpu(), P)
        assert_attn_close(out[s:s + 1], ref, f"reduce seq {s}")


# ------------------------------------------------------------------------------------------
# merge_attn_states


# head sizes whose rows are a power of two of 16-byte chunks take the vectorised kernel (64,
# 128, 256); 80 (and an output 2 bytes off a 16-byte boundary) the one with a warp per row
@pytest.mark.parametrize("D,misaligned", [(128, False), (64, False), (256, False), (80, False),
                                          (128, True)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_merge_attn_states(pa, dtype, D, misaligned):
    g = torch.Generator().manual_seed(77)
    T, H = 300, 8
    po = torch.randn((T, H, D), generator=g).to(dtype)
    so = torch.randn((T, H, D), generator=g).to(dtype)
    pl = torch.randn((H, T), generator=g) * 3
    sl = torch.randn((H, T), generator=g) * 3
    inf = math.inf
    specials = [(inf, 0.5), (0.5, inf), (-inf, -inf), (inf, inf), (-inf, 1.0), (2.0, -inf),
                (inf, -inf)]
    for i, (a, b) in enumerate(specials):
        pl[i % H, i], sl[i % H, i] = a, b
    for ptc in (-1, 250):
        if misaligned:  # a view one element into a larger buffer
            out = torch.empty(T * H * D + 1, dtype=dtype, device=DEV)[1:].view(T, H, D)
        else:
            out = torch.empty_like(po, device=DEV)
        olse = torch.empty((H, T), device=DEV)
        pa.pa_merge_attn_states(out, olse, po.to(DEV), pl.to(DEV), so.to(DEV), sl.to(DEV), ptc)
        assert pa.pa_device_status() == pa.PA_OK
        st, ref, rlse = oracle.merge_attn_states(po, pl, so, sl, ptc)
        assert st == oracle.OK
        assert_attn_close(out, ref, f"merge out {dtype}")
        finite = torch.isfinite(rlse)
        assert torch.equal(torch.isfinite(olse.cpu()), finite)
        assert torch.equal(olse.cpu()[~finite], rlse[~finite])
        assert (olse.cpu()[finite] - rlse[finite]).abs().max() < 1e-5
        # the special cases pass one input through bit-exactly
        for i, (a, b) in enumerate(specials):
            h, t = i % H, i
            a2 = -inf if math.isinf(a) else a
            b2 = -inf if math.isinf(b) else b
            if a2 == -inf or b2 == -inf:
                assert torch.equal(out[t, h].cpu(), ref[t, h]), (a, b)


# ------------------------------------------------------------------------------------------
# gather


def test_gather_roundtrip_bitexact(pa):
    w = workloads.named(3, small=True, device=DEV)
    slots, kb, vb, _ = _step(pa, w)
    qsl = w.query_start_loc
    ko = torch.empty((w.num_tokens, w.num_kv_heads, w.head_dim), dtype=w.dtype, device=DEV)
    vo = torch.empty_like(ko)
    starts = (w.seq_lens - (qsl[1:] - qsl[:-1])).to(torch.int32)  # each chunk's first position
    pa.pa_gather_kv(kb, vb, ko, vo, qsl, w.block_tables, seq_starts=starts)
    assert pa.pa_device_status() == pa.PA_OK
    assert torch.equal(ko, w.k_new) and torch.equal(vo, w.v_new)
    st, oko, ovo = oracle.gather_kv(kb.cpu(), vb.cpu(), qsl, w.block_tables, seq_starts=starts)
    assert st == oracle.OK and torch.equal(ko.cpu(), oko) and torch.equal(vo.cpu(), ovo)
    # a whole-context gather (no starts) equals the oracle's
    cu = torch.cat([torch.zeros(1, dtype=torch.int64), w.seq_lens.cpu().cumsum(0)]).to(torch.int32)
    kf = torch.empty((int(cu[-1]), w.num_kv_heads, w.head_dim), dtype=w.dtype, device=DEV)
    pa.pa_gather_kv(kb, None, kf, None, cu.to(DEV), w.block_tables)
    assert pa.pa_device_status() == pa.PA_OK
    st, okf, _ = oracle.gather_kv(kb.cpu(), None, cu, w.block_tables)
    assert st == oracle.OK and torch.equal(kf.cpu(), okf)
