"""GPU parity of one dequantisation factor per (pool block, kv head) (tinyllm "Going further":
fp8 KV caches with scales per block) against the oracle's per-block functions:

  - pa_reshape_and_cache_per_block stores head g of a row written to slot s as
    x / factors[s // b, g], bit for bit, into fp8 and f32 pools (one launch and, above 2048
    tokens, the separate slot check);
  - pa_varlen_forward_per_block: decode tokens on the e4m3 warp-MMA kernel, prefill chunks on
    the tcgen05 kernel (K factors on the scores, V factors where the codes are widened), with
    sinks and lse; a
    factor far from its item's reference sends the item to the warp-MMA kernel; factors of
    any magnitude (2^-23 .. 2^20) keep the kernels' f16 values in range;
  - pa_decode_splitkv_partials_per_block, and partials + reduce against full attention;
  - a factor of a block that is read (or written) and is not a finite positive normal float
    (0, negative, inf, nan, the subnormal 1e-39) is rejected on the device (PA_EINVAL) with
    nothing written; a bad factor of a block nothing touches is ignored; pools that are not
    e4m3 are PA_EUNSUPPORTED;
  - with PA_FLAG_BITWISE a decode token gives the same bits as the same token inside a
    prefill chunk.
"""
import math

import pytest
import torch

import oracle
from paged_kv_cache_31_gb300 import workloads
from tests.gpu_helpers import assert_attn_close, assert_attn_close_scaled

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def pa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_31_gb300 import binding

    assert binding.pa_device_status() == binding.PA_OK
    return binding


def _factors(NB, Hkv, seed, lo=-5.0, hi=-2.0):
    # 2^U(lo, hi): the factors of neighbouring blocks differ by up to 8x
    g = torch.Generator().manual_seed(seed)
    return (2.0 ** (lo + (hi - lo) * torch.rand((NB, Hkv), generator=g))).to(DEV)


def _bits(t):
    return t.view(torch.uint8).cpu() if t.dtype == torch.float8_e4m3fn else t.cpu()


# ------------------------------------------------------------------------------------ scatter

@pytest.mark.parametrize("dst", [torch.float8_e4m3fn, torch.float32])
@pytest.mark.parametrize("T,Hkv,D", [(1, 4, 128), (37, 3, 7), (3000, 8, 128)])
def test_per_block_scatter_is_bit_exact(pa, dst, T, Hkv, D):
    b = 16
    NB = (T + b - 1) // b + 8
    g = torch.Generator().manual_seed(T + D + 5)
    k = torch.randn((T, Hkv, D), generator=g).to(torch.bfloat16)
    v = (torch.randn((T, Hkv, D), generator=g) * 3).to(torch.bfloat16)
    ks, vs = _factors(NB, Hkv, T + 1), _factors(NB, Hkv, T + 2)
    slots = torch.randperm(NB * b, generator=g)[:T].to(torch.int32)
    kb = torch.zeros((NB, b, Hkv, D), dtype=dst)
    vb = torch.zeros_like(kb)
    assert oracle.reshape_and_cache_per_block(k, v, kb, vb, slots, b, ks, vs) == oracle.OK
    gkb, gvb = torch.zeros_like(kb, device=DEV), torch.zeros_like(vb, device=DEV)
    pa.pa_reshape_and_cache(k.to(DEV), v.to(DEV), gkb, gvb, slots.to(DEV), k_block_scales=ks,
                            v_block_scales=vs)
    assert pa.pa_device_status() == pa.PA_OK
    assert torch.equal(_bits(gkb), _bits(kb)) and torch.equal(_bits(gvb), _bits(vb))


@pytest.mark.parametrize("T", [9, 3000])
def test_per_block_scatter_checks_the_written_blocks(pa, T):
    Hkv, D, b = 4, 128, 16
    NB = (T + b - 1) // b + 2  # the last two blocks are never written
    k = torch.randn((T, Hkv, D), device=DEV)
    slots = torch.arange(T, dtype=torch.int32, device=DEV)
    for bad in (0.0, -1.0, float("inf"), float("nan"), 1e-39):
        kb = torch.zeros((NB, b, Hkv, D), dtype=torch.float8_e4m3fn, device=DEV)
        vb = torch.zeros_like(kb)
        ks, vs = _factors(NB, Hkv, 3), _factors(NB, Hkv, 4)
        vs[0, 2] = bad  # block 0 receives rows
        pa.pa_reshape_and_cache(k, k, kb, vb, slots, k_block_scales=ks, v_block_scales=vs)
        assert pa.pa_device_status() == pa.PA_EINVAL
        assert int(kb.view(torch.uint8).count_nonzero()) == 0
        assert int(vb.view(torch.uint8).count_nonzero()) == 0
        vs[0, 2] = 0.25
        ks[NB - 1, 1] = bad  # no row goes there
        pa.pa_reshape_and_cache(k, k, kb, vb, slots, k_block_scales=ks, v_block_scales=vs)
        assert pa.pa_device_status() == pa.PA_OK


# ---------------------------------------------------------------------------------- attention

CASES = {
    # decode tokens, GQA 4
    "decode": dict(seq_lens=[1, 17, 300, 1000, 4096], q_lens=[1] * 5, num_heads=32,
                   num_kv_heads=8, head_dim=128),
    # prefill chunks (tcgen05) and decode tokens (warp-MMA), windowed
    "mixed": dict(seq_lens=[512, 700, 1300, 90, 2000], q_lens=[512, 200, 1, 1, 1],
                  num_heads=32, num_kv_heads=8, head_dim=128, sliding_window=600),
}


def _case(name):
    seed = sorted(CASES).index(name) + 211
    w = workloads.build(name, seed=seed, device=DEV, **CASES[name])
    kb, vb = workloads.fp8_pools(w)
    NB = kb.shape[0]
    return w, kb, vb, _factors(NB, w.num_kv_heads, seed), _factors(NB, w.num_kv_heads, seed + 1), seed


@pytest.mark.parametrize("case", sorted(CASES))
def test_per_block_attention_matches_oracle(pa, case):
    w, kb, vb, ks, vs, seed = _case(case)
    g = torch.Generator().manual_seed(seed)
    sinks = torch.randn((w.num_heads,), generator=g) + 1.0
    sinks[::3] = -math.inf
    out = torch.full_like(w.q, float("nan"))
    lse = torch.full((w.num_heads, w.num_tokens), float("nan"), device=DEV)
    pa.pa_varlen_forward(w.q, kb, vb, out, w.query_start_loc, w.seq_lens, w.positions,
                         w.block_tables, w.scale, causal=w.causal,
                         sliding_window=w.sliding_window, sinks=sinks.to(DEV), lse=lse,
                         k_block_scales=ks, v_block_scales=vs)
    assert pa.pa_device_status() == pa.PA_OK
    st, ref, ref_lse = oracle.varlen_attention(w.q.cpu(), kb.cpu(), vb.cpu(), w.query_start_loc,
                                               w.seq_lens, w.positions, w.block_tables, w.scale,
                                               causal=w.causal, sliding_window=w.sliding_window,
                                               want_lse=True, sinks=sinks, k_block_scales=ks,
                                               v_block_scales=vs)
    assert st == oracle.OK
    assert_attn_close(out, ref, f"per-block {case}")
    fin = torch.isfinite(ref_lse)
    assert torch.equal(torch.isinf(lse.cpu()), torch.isinf(ref_lse))
    err = (lse.cpu() - ref_lse).abs()
    assert float(err[fin].max()) < 1e-3 + 1e-4 * float(ref_lse[fin].abs().max())


def test_per_block_attention_checks_the_read_blocks(pa):
    w, kb, vb, ks, vs, _ = _case("decode")
    read = {int(w.block_tables[s, j]) for s in range(w.num_seqs)
            for j in range((int(w.seq_lens[s]) + 15) // 16)}
    unread = [i for i in range(kb.shape[0]) if i not in read]
    victim = int(w.block_tables[3, 5])
    for bad in (0.0, -0.5, float("inf"), float("nan"), 1e-39):
        v2 = vs.clone()
        v2[victim, 6] = bad
        out = torch.full_like(w.q, 7.0)
        pa.pa_varlen_forward(w.q, kb, vb, out, w.query_start_loc, w.seq_lens, w.positions,
                             w.block_tables, w.scale, k_block_scales=ks, v_block_scales=v2)
        assert pa.pa_device_status() == pa.PA_EINVAL
        assert bool((out == 7.0).all())
    assert unread, "the pool has blocks no table reads"
    k2 = ks.clone()
    k2[unread[0], 0] = float("nan")
    out = torch.full_like(w.q, 7.0)
    pa.pa_varlen_forward(w.q, kb, vb, out, w.query_start_loc, w.seq_lens, w.positions,
                         w.block_tables, w.scale, k_block_scales=k2, v_block_scales=vs)
    assert pa.pa_device_status() == pa.PA_OK
    assert bool(torch.isfinite(out.float()).all())


def test_per_block_needs_e4m3_pools(pa):
    w = workloads.build("bf16", seq_lens=[40], q_lens=[1], num_heads=8, num_kv_heads=2,
                        head_dim=128, seed=5, device=DEV)
    NB = w.k_blocks.shape[0]
    with pytest.raises(pa.PaError) as e:
        pa.pa_varlen_forward(w.q, w.k_blocks, w.v_blocks, torch.empty_like(w.q),
                             w.query_start_loc, w.seq_lens, w.positions, w.block_tables, w.scale,
                             k_block_scales=_factors(NB, 2, 1), v_block_scales=_factors(NB, 2, 2))
    assert e.value.status == pa.PA_EUNSUPPORTED
    assert pa.pa_device_status() == pa.PA_OK


@pytest.mark.parametrize("spread", ["large", "small"])
def test_per_block_factor_spread_is_recomputed(pa, spread):
    # a few V factors of the first prefill chunk far from its first block's (ratio 200 / 2^-5
    # or 10^-6 / 2^-2): in the tcgen05 kernel the products would leave f16's range or keep few
    # bits, so the item is recomputed by the warp-MMA kernel
    w, kb, vb, ks, vs, seed = _case("mixed")
    vs = vs.clone()
    for j in (1, 5, 9):
        vs[int(w.block_tables[0, j]), j % w.num_kv_heads] = 200.0 if spread == "large" else 1e-6
    out = torch.full_like(w.q, float("nan"))
    pa.pa_varlen_forward(w.q, kb, vb, out, w.query_start_loc, w.seq_lens, w.positions,
                         w.block_tables, w.scale, sliding_window=w.sliding_window,
                         k_block_scales=ks, v_block_scales=vs)
    assert pa.pa_device_status() == pa.PA_OK
    ref = _oracle_of(w, kb, vb, ks, vs)
    assert_attn_close_scaled(out, ref, _oracle_of(w, kb, _abs_codes(vb), ks, vs),
                             f"per-block factor spread {spread}")


@pytest.mark.parametrize("case", sorted(CASES))
@pytest.mark.parametrize("mag", ["tiny", "huge"])
def test_per_block_factor_magnitudes(pa, case, mag):
    # every factor near 2^-22 (V) and 2^-20 (K), or near 2^18 (V) and 2^2 (K): f16 products
    # and weights would underflow or overflow at these magnitudes taken as they are; the
    # kernels keep V in units of a reference factor.  The bound scales with V.
    w, kb, vb, _, _, seed = _case(case)
    NB, Hkv = kb.shape[0], w.num_kv_heads
    kexp, vexp = (-20.0, -22.0) if mag == "tiny" else (2.0, 18.0)
    ks = _factors(NB, Hkv, seed + 5, kexp - 1.5, kexp + 1.5)
    vs = _factors(NB, Hkv, seed + 6, vexp - 1.5, vexp + 1.5)
    out = torch.full_like(w.q, float("nan"))
    lse = torch.full((w.num_heads, w.num_tokens), float("nan"), device=DEV)
    pa.pa_varlen_forward(w.q, kb, vb, out, w.query_start_loc, w.seq_lens, w.positions,
                         w.block_tables, w.scale, causal=w.causal,
                         sliding_window=w.sliding_window, lse=lse, k_block_scales=ks,
                         v_block_scales=vs)
    assert pa.pa_device_status() == pa.PA_OK
    st, ref, ref_lse = oracle.varlen_attention(w.q.cpu(), kb.cpu(), vb.cpu(), w.query_start_loc,
                                               w.seq_lens, w.positions, w.block_tables, w.scale,
                                               causal=w.causal, sliding_window=w.sliding_window,
                                               want_lse=True, k_block_scales=ks,
                                               v_block_scales=vs)
    assert st == oracle.OK
    assert_attn_close_scaled(out, ref, _oracle_of(w, kb, _abs_codes(vb), ks, vs),
                             f"per-block {case}, {mag} factors")
    err = (lse.cpu() - ref_lse).abs()
    assert float(err.max()) < 1e-3 + 1e-4 * float(ref_lse.abs().max())


def _abs_codes(vb):
    # |code| of every e4m3 value (exact): the oracle over them gives each output's scale
    return vb.float().abs().to(torch.float8_e4m3fn)


def _oracle_of(w, kb, vb, ks, vs):
    st, ref, _ = oracle.varlen_attention(w.q.cpu(), kb.cpu(), vb.cpu(), w.query_start_loc,
                                         w.seq_lens, w.positions, w.block_tables, w.scale,
                                         causal=w.causal, sliding_window=w.sliding_window,
                                         k_block_scales=ks, v_block_scales=vs)
    assert st == oracle.OK
    return ref


def test_per_block_decode_equals_prefill_bitwise(pa):
    # the tokens of a 64-token chunk at positions 100..163, and each of them as a decode token
    # of its own (seq_len = position + 1, the same table): the same bits (PA_FLAG_BITWISE keeps
    # the chunk on the warp-MMA kernel)
    H, Hkv, D = 32, 8, 128
    chunk = workloads.build("chunk", seq_lens=[164], q_lens=[64], num_heads=H, num_kv_heads=Hkv,
                            head_dim=D, seed=17, device=DEV)
    kb, vb = workloads.fp8_pools(chunk)
    NB = kb.shape[0]
    ks, vs = _factors(NB, Hkv, 18), _factors(NB, Hkv, 19)
    out = torch.empty_like(chunk.q)
    pa.pa_varlen_forward(chunk.q, kb, vb, out, chunk.query_start_loc, chunk.seq_lens,
                         chunk.positions, chunk.block_tables, chunk.scale, k_block_scales=ks,
                         v_block_scales=vs, bitwise=True)
    T = 64
    qsl = torch.arange(T + 1, dtype=torch.int32, device=DEV)
    pos = chunk.positions.clone()
    sl = (pos + 1).to(torch.int32)
    bt = chunk.block_tables.repeat(T, 1).contiguous()
    dec = torch.empty_like(chunk.q)
    pa.pa_varlen_forward(chunk.q, kb, vb, dec, qsl, sl, pos, bt, chunk.scale, k_block_scales=ks,
                         v_block_scales=vs, bitwise=True)
    assert pa.pa_device_status() == pa.PA_OK
    assert torch.equal(dec, out)


def test_per_block_splitkv(pa):
    H, Hkv, D = 32, 8, 128
    lens = [1, 511, 512, 513, 1500, 4100]
    w = workloads.build("split-per-block", seq_lens=lens, q_lens=[1] * len(lens), num_heads=H,
                        num_kv_heads=Hkv, head_dim=D, seed=91, device=DEV, sliding_window=1700,
                        partition_size=512)
    kb, vb = workloads.fp8_pools(w)
    NB = kb.shape[0]
    ks, vs = _factors(NB, Hkv, 92), _factors(NB, Hkv, 93)
    P, MP, S = 512, w.max_partitions(), len(lens)
    ml = torch.full((S, H, MP), float("nan"), device=DEV)
    es = torch.full_like(ml, float("nan"))
    to = torch.full((S, H, MP, D), float("nan"), device=DEV)
    pa.pa_decode_splitkv_partials(w.q, kb, vb, ml, es, to, w.seq_lens, w.block_tables, w.scale,
                                  partition_size=P, sliding_window=1700, k_block_scales=ks,
                                  v_block_scales=vs)
    assert pa.pa_device_status() == pa.PA_OK
    st, rml, res, rto = oracle.splitkv_partials(w.q.cpu(), kb.cpu(), vb.cpu(), w.seq_lens,
                                                w.block_tables, w.scale, P, MP, 1700,
                                                k_block_scales=ks, v_block_scales=vs)
    assert st == oracle.OK
    assert torch.equal(torch.isinf(ml.cpu()), torch.isinf(rml))
    fin = torch.isfinite(rml)
    assert float((ml.cpu()[fin] - rml[fin]).abs().max()) < 1e-3
    assert float(((es.cpu() - res).abs() / res.clamp_min(1e-30))[res > 0].max()) < 2e-3
    assert_attn_close(to, rto, "per-block split tmp_out")
    out = torch.empty_like(w.q)
    pa.pa_decode_splitkv_reduce(out, ml, es, to, w.seq_lens, partition_size=P)
    assert pa.pa_device_status() == pa.PA_OK
    pos = torch.tensor([n - 1 for n in lens], dtype=torch.int32)
    qsl = torch.arange(S + 1, dtype=torch.int32)
    st, full, _ = oracle.varlen_attention(w.q.cpu(), kb.cpu(), vb.cpu(), qsl, w.seq_lens, pos,
                                          w.block_tables, w.scale, sliding_window=1700,
                                          k_block_scales=ks, v_block_scales=vs)
    assert st == oracle.OK
    assert_attn_close(out, full, "per-block split + reduce vs full")
