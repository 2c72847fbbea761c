"""GPU parity of prefill chunks, the sequences with more than 64 query rows per kv head that
run on the tcgen05 / tensor-memory kernel: every GQA group that divides the 128-row tile,
ragged chunk lengths, prior contexts that leave the first key tile partial, sliding windows,
non-causal chunks, NaN in never-written slots, and batches mixing them with decode tokens."""
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


def _run(pa, w):
    out = torch.full_like(w.q, float("nan"))
    pa.pa_varlen_forward(w.q, w.k_blocks, w.v_blocks, out, w.query_start_loc, w.seq_lens,
                         w.positions, w.block_tables, w.scale, causal=w.causal,
                         sliding_window=w.sliding_window)
    assert pa.pa_device_status() == pa.PA_OK
    return out


@pytest.mark.parametrize("H,Hkv", [(8, 8), (16, 8), (32, 8), (64, 8), (32, 2), (64, 2)])
def test_prefill_gqa_groups(pa, H, Hkv):
    # chunks after prior contexts of 0, 5, 16, 200 and 1000 positions, lengths not multiples
    # of the tile, plus two decode tokens
    prior = [0, 5, 16, 200, 1000, 3000, 40]
    chunk = [70, 130, 33, 256, 97, 1, 1]
    w = workloads.build("pre", seq_lens=[p + c for p, c in zip(prior, chunk)], q_lens=chunk,
                        num_heads=H, num_kv_heads=Hkv, head_dim=128, seed=H + Hkv, device=DEV)
    out = _run(pa, w)
    assert_attn_close(out, oracle_attention(w, w.k_blocks.cpu(), w.v_blocks.cpu()),
                      f"H {H} Hkv {Hkv}")


@pytest.mark.parametrize("window,causal", [(64, True), (300, True), (1, True), (0, False),
                                           (150, False)])
def test_prefill_windows_and_noncausal(pa, window, causal):
    prior = [0, 100, 700, 33]
    chunk = [200, 150, 300, 129]
    w = workloads.build("prewin", seq_lens=[p + c for p, c in zip(prior, chunk)], q_lens=chunk,
                        num_heads=32, num_kv_heads=8, head_dim=128, seed=window + 3,
                        sliding_window=window, causal=causal, device=DEV)
    out = _run(pa, w)
    assert_attn_close(out, oracle_attention(w, w.k_blocks.cpu(), w.v_blocks.cpu()),
                      f"window {window} causal {causal}")


def test_prefill_nan_in_unwritten_slots(pa):
    prior = [3, 250, 40]
    chunk = [90, 100, 300]
    w = workloads.build("prenan", seq_lens=[p + c for p, c in zip(prior, chunk)], q_lens=chunk,
                        num_heads=32, num_kv_heads=8, head_dim=128, seed=77, device=DEV,
                        extra_table_cols=2)
    kb, vb = w.k_blocks.clone(), w.v_blocks.clone()
    used = set()
    for s, n in enumerate(w.seq_lens_list):
        for i in range((n + 15) // 16):
            used.add(int(w.block_tables[s, i]))
        last = int(w.block_tables[s, (n - 1) // 16])
        if n % 16:
            kb[last, n % 16:] = float("nan")
            vb[last, n % 16:] = float("inf")
    for b in range(w.num_blocks):  # blocks no table uses
        if b not in used:
            kb[b] = float("nan")
            vb[b] = float("nan")
    w.k_blocks, w.v_blocks = kb, vb
    out = _run(pa, w)
    assert torch.isfinite(out.float()).all()
    assert_attn_close(out, oracle_attention(w, kb.cpu(), vb.cpu()), "nan tails")


def test_prefill_many_chunks_and_decodes(pa):
    g = torch.Generator().manual_seed(5)
    prior = [int(x) for x in torch.randint(0, 1500, (12,), generator=g)]
    chunk = [int(x) for x in torch.randint(17, 400, (12,), generator=g)]
    dec = [int(x) for x in torch.randint(1, 3000, (20,), generator=g)]
    w = workloads.build("premix", seq_lens=dec + [p + c for p, c in zip(prior, chunk)],
                        q_lens=[1] * 20 + chunk, num_heads=32, num_kv_heads=8, head_dim=128,
                        seed=6, sliding_window=1024, device=DEV)
    out = _run(pa, w)
    assert_attn_close(out, oracle_attention(w, w.k_blocks.cpu(), w.v_blocks.cpu()), "mixed")
    again = _run(pa, w)
    assert torch.equal(out, again), "prefill path not deterministic"


def test_prefill_output_only_16_byte_aligned(pa):
    # the tcgen05 kernel writes 32-byte stores when the output is 32-byte aligned and 16-byte
    # stores otherwise: an output that starts 16 bytes into its allocation must give the same
    # bits as an aligned one
    prior = [0, 300, 45]
    chunk = [200, 129, 96]
    w = workloads.build("pre16", seq_lens=[p + c for p, c in zip(prior, chunk)], q_lens=chunk,
                        num_heads=32, num_kv_heads=8, head_dim=128, seed=16, device=DEV)
    aligned = _run(pa, w)
    assert aligned.data_ptr() % 32 == 0
    buf = torch.full((w.q.numel() + 8,), float("nan"), dtype=w.q.dtype, device=DEV)
    out = buf[8:].view_as(w.q)
    assert out.data_ptr() % 32 == 16
    pa.pa_varlen_forward(w.q, w.k_blocks, w.v_blocks, out, w.query_start_loc, w.seq_lens,
                         w.positions, w.block_tables, w.scale, causal=w.causal)
    assert pa.pa_device_status() == pa.PA_OK
    assert torch.equal(out, aligned)
    assert torch.isnan(buf[:8].float()).all()


@pytest.mark.parametrize("big", [5.99e4, -6.5e4, 1.0e6, -1.0e30])
def test_prefill_v_beyond_f16_range(pa, big):
    """The tcgen05 kernel multiplies f16 weights with V widened to f16.  A V magnitude that f16
    holds (below 65520) is widened exactly; a larger one marks its 256-row item, which the
    warp-MMA kernel recomputes from the bf16 pool after the tcgen05 kernel.  Either way the
    output matches the oracle.  The large values sit at random visible positions, including
    keys that the causal mask hides from some rows of the same item (where an f16 infinity
    times a zero weight would be NaN), next to decode tokens that run alongside."""
    prior = [0, 300, 45, 1000, 17]
    chunk = [200, 129, 96, 1, 1]
    H, Hkv = 32, 8
    w = workloads.build("prebig", seq_lens=[p + c for p, c in zip(prior, chunk)], q_lens=chunk,
                        num_heads=H, num_kv_heads=Hkv, head_dim=128, seed=21, device=DEV)
    vb = w.v_blocks.clone()
    g = torch.Generator().manual_seed(abs(int(big)) % 1000 + 3)
    for s in range(3):  # the prefill chunks
        n = w.seq_lens_list[s]
        for _ in range(4):
            pos = int(torch.randint(0, n, (1,), generator=g))
            kvh = int(torch.randint(0, Hkv, (1,), generator=g))
            d = int(torch.randint(0, 128, (1,), generator=g))
            vb[int(w.block_tables[s, pos // 16]), pos % 16, kvh, d] = big
    w.v_blocks = vb
    out = _run(pa, w)
    assert torch.isfinite(out.float()).all()
    assert_attn_close(out, oracle_attention(w, w.k_blocks.cpu(), vb.cpu()), f"V with {big}")
    assert torch.equal(_run(pa, w), out), "not deterministic"


def test_mixed_batch_equals_its_parts_bitwise(pa):
    """In a mixed call the decode tiles run on the warp-MMA kernel beside the tcgen05 kernel,
    which the plan gives only part of the SMs; a prefill-only call gives it all of them and a
    decode-only call does not launch it.  Each item's arithmetic does not depend on where it
    runs, so the mixed batch gives, bit for bit, what its prefill chunks and its decode tokens
    give as two separate calls."""
    from tests.gpu_helpers import sub_batch
    w = workloads.named(3, device=DEV)
    mixed = _run(pa, w)
    for part in ([s for s, q in enumerate(w.q_lens_list) if q == 1],
                 [s for s, q in enumerate(w.q_lens_list) if q > 1]):
        sb = sub_batch(w, part)
        rows = sb["rows"].to(DEV)
        out = torch.full_like(w.q[rows], float("nan"))
        pa.pa_varlen_forward(w.q[rows].contiguous(), w.k_blocks, w.v_blocks, out,
                             sb["query_start_loc"].to(DEV), sb["seq_lens"].to(DEV),
                             sb["positions"].to(DEV), sb["block_tables"].to(DEV), w.scale,
                             causal=w.causal, sliding_window=w.sliding_window)
        assert pa.pa_device_status() == pa.PA_OK
        assert torch.equal(out, mixed[rows]), f"{len(part)} sequences differ from the mixed call"


@pytest.mark.parametrize("H,Hkv,window,causal", [(32, 8, 0, True), (8, 8, 0, True),
                                                 (64, 8, 300, True), (32, 2, 0, False),
                                                 (16, 8, 64, True)])
def test_prefill_fp8_pools(pa, H, Hkv, window, causal):
    """Prefill chunks over e4m3 pools on the tcgen05 kernel: the codes are staged by TMA and
    widened to f16 in shared memory by the converter warps (K into the dim-half layout, V
    into the MN-major one, rows past seq_len zeroed), q widened to f16 once per item; against
    the oracle over the same codes and scales, with NaN codes in the never-written rows."""
    import oracle
    prior = [0, 5, 200, 1000, 40, 3000]
    chunk = [150, 130, 256, 97, 1, 1]
    w = workloads.build("pre8", seq_lens=[p + c for p, c in zip(prior, chunk)], q_lens=chunk,
                        num_heads=H, num_kv_heads=Hkv, head_dim=128, seed=H + Hkv + window,
                        sliding_window=window, causal=causal, device=DEV)
    kb8, vb8 = workloads.fp8_pools(w)
    tab = w.block_tables.cpu()
    for s, n in enumerate(w.seq_lens_list):
        if n % 16:
            blk = int(tab[s, (n - 1) // 16])
            kb8.view(torch.uint8)[blk, n % 16:] = 0x7F
            vb8.view(torch.uint8)[blk, n % 16:] = 0xFF
    ks, vs = 0.125, 0.0625
    out = torch.full_like(w.q, float("nan"))
    pa.pa_varlen_forward(w.q, kb8, vb8, out, w.query_start_loc, w.seq_lens, w.positions,
                         w.block_tables, w.scale, causal=causal, sliding_window=window,
                         k_scale=ks, v_scale=vs)
    assert pa.pa_device_status() == pa.PA_OK
    st, ref, _ = oracle.varlen_attention(w.q.cpu(), kb8.cpu(), vb8.cpu(), w.query_start_loc,
                                         w.seq_lens, w.positions, w.block_tables, w.scale,
                                         causal=causal, sliding_window=window, k_scale=ks,
                                         v_scale=vs)
    assert st == oracle.OK
    assert_attn_close(out, ref, f"fp8 prefill H {H} Hkv {Hkv} window {window}")
    again = torch.empty_like(out)
    pa.pa_varlen_forward(w.q, kb8, vb8, again, w.query_start_loc, w.seq_lens, w.positions,
                         w.block_tables, w.scale, causal=causal, sliding_window=window,
                         k_scale=ks, v_scale=vs)
    assert torch.equal(out, again), "not deterministic"
