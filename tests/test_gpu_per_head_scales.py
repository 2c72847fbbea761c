"""GPU parity of one dequantisation scale per kv head (tinyllm "Going further": fp8 KV caches
with scales per head; "paged_attention_v2_pytorch.py": K = k_scale * pool, V = v_scale * pool)
against the oracle's per-head functions:

  - pa_reshape_and_cache_per_head stores head g of a row as x / k_scales[g], bit for bit, into
    fp8, bf16 and f32 pools;
  - pa_varlen_forward_per_head on the warp-MMA kernel (fp8 and bf16 pools), the tcgen05
    prefill kernel (bf16 pools) and the generic kernel, with sinks and lse;
  - pa_decode_splitkv_partials_per_head, and partials + reduce against full attention;
  - scales that are not finite and positive are rejected on the device (PA_EINVAL), with
    nothing written.
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


def _spreads(Hkv):
    # per-head spreads of the fp8 codes: 2 .. 64, so one pool scale would fit no head well
    return [2.0 * 2.0 ** (5.0 * g / max(Hkv - 1, 1)) for g in range(Hkv)]


def _bits(t):
    return t.view(torch.uint8).cpu() if t.dtype == torch.float8_e4m3fn else t.cpu()


# ------------------------------------------------------------------------------------ scatter

@pytest.mark.parametrize("dst", [torch.float8_e4m3fn, torch.bfloat16, torch.float32])
@pytest.mark.parametrize("T,Hkv,D", [(1, 4, 128), (37, 3, 7), (3000, 8, 128)])
def test_per_head_scatter_is_bit_exact(pa, dst, T, Hkv, D):
    b = 16
    NB = (T + b - 1) // b + 8
    g = torch.Generator().manual_seed(T + D)
    sp = torch.tensor(_spreads(Hkv)).view(1, Hkv, 1)
    k = (torch.randn((T, Hkv, D), generator=g) * sp).to(torch.bfloat16)
    v = (torch.randn((T, Hkv, D), generator=g) * sp * 3).to(torch.bfloat16)
    ks = (1.0 / sp.view(-1)).contiguous()
    vs = (0.7 / sp.view(-1)).contiguous()
    slots = torch.randperm(NB * b, generator=g)[:T].to(torch.int32)
    kb = torch.zeros((NB, b, Hkv, D), dtype=dst)
    vb = torch.zeros_like(kb)
    assert oracle.reshape_and_cache_per_head(k, v, kb, vb, slots, b, ks, vs) == oracle.OK
    gkb, gvb = torch.zeros_like(kb, device=DEV), torch.zeros_like(vb, device=DEV)
    pa.pa_reshape_and_cache(k.to(DEV), v.to(DEV), gkb, gvb, slots.to(DEV), k_scales=ks.to(DEV),
                            v_scales=vs.to(DEV))
    assert pa.pa_device_status() == pa.PA_OK
    assert torch.equal(_bits(gkb), _bits(kb)) and torch.equal(_bits(gvb), _bits(vb))


def test_per_head_scatter_rejects_bad_scales(pa):
    Hkv, D, b, NB, T = 4, 128, 16, 4, 9
    k = torch.randn((T, Hkv, D), device=DEV)
    kb = torch.zeros((NB, b, Hkv, D), dtype=torch.float8_e4m3fn, device=DEV)
    vb = torch.zeros_like(kb)
    slots = torch.arange(T, dtype=torch.int32, device=DEV)
    for bad in (0.0, -1.0, float("inf"), float("nan")):
        ks = torch.full((Hkv,), 0.5, device=DEV)
        ks[2] = bad
        pa.pa_reshape_and_cache(k, k, kb, vb, slots, k_scales=ks, v_scales=None)
        assert pa.pa_device_status() == pa.PA_EINVAL
        assert int(kb.view(torch.uint8).count_nonzero()) == 0
        assert int(vb.view(torch.uint8).count_nonzero()) == 0
    assert pa.pa_device_status() == pa.PA_OK


# ---------------------------------------------------------------------------------- attention

CASES = {
    # decode tokens on the fp8 warp-MMA kernel, GQA 4
    "decode-fp8": dict(pool="fp8", seq_lens=[1, 17, 300, 1000, 4096], q_lens=[1] * 5,
                       num_heads=32, num_kv_heads=8, head_dim=128),
    # prefill chunks and decode tokens on fp8 pools (all on the warp-MMA kernel), windowed
    "mixed-fp8": dict(pool="fp8", seq_lens=[512, 700, 1300, 90, 2000], q_lens=[512, 200, 1, 1, 1],
                      num_heads=32, num_kv_heads=8, head_dim=128, sliding_window=600),
    # bf16 pools: prefill chunks on the tcgen05 kernel, decode tokens on the warp-MMA kernel
    "mixed-bf16": dict(pool="bf16", seq_lens=[600, 1300, 90, 2000, 4000],
                       q_lens=[512, 130, 1, 1, 1], num_heads=32, num_kv_heads=8, head_dim=128),
    # the generic kernel: fp32 q and pools, head size 64, GQA 2
    "simt-f32": dict(pool="f32", seq_lens=[1, 40, 77, 300], q_lens=[1, 40, 2, 1], num_heads=8,
                     num_kv_heads=4, head_dim=64, dtype=torch.float32),
}


def _case(name):
    kw = dict(CASES[name])
    pool = kw.pop("pool")
    seed = sorted(CASES).index(name) + 111
    w = workloads.build(name, seed=seed, device=DEV, **kw)
    Hkv = w.num_kv_heads
    if pool == "fp8":
        sp = _spreads(Hkv)
        kb, vb = workloads.fp8_pools_per_head(w, sp)
        ks = torch.tensor([1.0 / x for x in sp], device=DEV)
        vs = torch.tensor([0.8 / x for x in sp], device=DEV)
    else:
        kb, vb = w.k_blocks, w.v_blocks
        ks = torch.linspace(0.6, 1.4, Hkv, device=DEV)
        vs = torch.linspace(1.5, 0.5, Hkv, device=DEV)
    return w, kb, vb, ks, vs, seed


@pytest.mark.parametrize("case", sorted(CASES))
def test_per_head_attention_matches_oracle(pa, case):
    w, kb, vb, ks, vs, seed = _case(case)
    g = torch.Generator().manual_seed(seed)
    sinks = torch.randn((w.num_heads,), generator=g) + 1.0
    sinks[::3] = -math.inf
    out = torch.full_like(w.q, float("nan"))
    lse = torch.full((w.num_heads, w.num_tokens), float("nan"), device=DEV)
    pa.pa_varlen_forward(w.q, kb, vb, out, w.query_start_loc, w.seq_lens, w.positions,
                         w.block_tables, w.scale, causal=w.causal,
                         sliding_window=w.sliding_window, sinks=sinks.to(DEV), lse=lse,
                         k_scales=ks, v_scales=vs)
    assert pa.pa_device_status() == pa.PA_OK
    st, ref, ref_lse = oracle.varlen_attention(w.q.cpu(), kb.cpu(), vb.cpu(), w.query_start_loc,
                                               w.seq_lens, w.positions, w.block_tables, w.scale,
                                               causal=w.causal, sliding_window=w.sliding_window,
                                               want_lse=True, sinks=sinks, k_scales=ks,
                                               v_scales=vs)
    assert st == oracle.OK
    assert_attn_close(out, ref, f"per-head {case}")
    fin = torch.isfinite(ref_lse)
    assert torch.equal(torch.isinf(lse.cpu()), torch.isinf(ref_lse))
    err = (lse.cpu() - ref_lse).abs()
    assert float(err[fin].max()) < 1e-3 + 1e-4 * float(ref_lse[fin].abs().max())


def test_equal_per_head_scales_match_the_pool_scale(pa):
    # every head at c is the per-pool scale c (to rounding: c is folded in a different order)
    w, kb, vb, _, _, _ = _case("mixed-bf16")
    Hkv = w.num_kv_heads
    run = lambda **kw: pa.pa_varlen_forward(
        w.q, kb, vb, torch.empty_like(w.q), w.query_start_loc, w.seq_lens, w.positions,
        w.block_tables, w.scale, **kw).float()
    a = run(k_scale=0.7, v_scale=1.3)
    b = run(k_scales=torch.full((Hkv,), 0.7, device=DEV),
            v_scales=torch.full((Hkv,), 1.3, device=DEV))
    assert_attn_close(b, a, "per-head c vs pool c")
    assert pa.pa_device_status() == pa.PA_OK


def test_per_head_attention_rejects_bad_scales(pa):
    w, kb, vb, ks, vs, _ = _case("decode-fp8")
    for bad in (0.0, -0.5, float("inf"), float("nan")):
        v2 = vs.clone()
        v2[5] = bad
        out = torch.full_like(w.q, 7.0)
        pa.pa_varlen_forward(w.q, kb, vb, out, w.query_start_loc, w.seq_lens, w.positions,
                             w.block_tables, w.scale, k_scales=ks, v_scales=v2)
        assert pa.pa_device_status() == pa.PA_EINVAL
        assert bool((out == 7.0).all())
    assert pa.pa_device_status() == pa.PA_OK


@pytest.mark.parametrize("pool,H,Hkv,D", [("fp8", 32, 8, 128), ("bf16", 32, 8, 128),
                                          ("fp8", 8, 2, 64)])
def test_per_head_splitkv(pa, pool, H, Hkv, D):
    lens = [1, 511, 512, 513, 1500, 4100]
    w = workloads.build("split-per-head", seq_lens=lens, q_lens=[1] * len(lens), num_heads=H,
                        num_kv_heads=Hkv, head_dim=D, seed=H + D + Hkv, device=DEV,
                        sliding_window=1700, partition_size=512)
    if pool == "fp8":
        sp = _spreads(Hkv)
        kb, vb = workloads.fp8_pools_per_head(w, sp)
        ks = torch.tensor([1.0 / x for x in sp], device=DEV)
        vs = torch.tensor([0.8 / x for x in sp], device=DEV)
    else:
        kb, vb = w.k_blocks, w.v_blocks
        ks = torch.linspace(0.6, 1.4, Hkv, device=DEV)
        vs = torch.linspace(1.5, 0.5, Hkv, device=DEV)
    P, MP, S = 512, w.max_partitions(), len(lens)
    ml = torch.full((S, H, MP), float("nan"), device=DEV)
    es = torch.full_like(ml, float("nan"))
    to = torch.full((S, H, MP, D), float("nan"), device=DEV)
    pa.pa_decode_splitkv_partials(w.q, kb, vb, ml, es, to, w.seq_lens, w.block_tables, w.scale,
                                  partition_size=P, sliding_window=1700, k_scales=ks,
                                  v_scales=vs)
    assert pa.pa_device_status() == pa.PA_OK
    st, rml, res, rto = oracle.splitkv_partials(w.q.cpu(), kb.cpu(), vb.cpu(), w.seq_lens,
                                                w.block_tables, w.scale, P, MP, 1700,
                                                k_scales=ks, v_scales=vs)
    assert st == oracle.OK
    assert torch.equal(torch.isinf(ml.cpu()), torch.isinf(rml))
    fin = torch.isfinite(rml)
    assert float((ml.cpu()[fin] - rml[fin]).abs().max()) < 1e-3
    assert float(((es.cpu() - res).abs() / res.clamp_min(1e-30))[res > 0].max()) < 2e-3
    assert_attn_close(to, rto, f"per-head split tmp_out {pool}")
    out = torch.empty_like(w.q)
    pa.pa_decode_splitkv_reduce(out, ml, es, to, w.seq_lens, partition_size=P)
    assert pa.pa_device_status() == pa.PA_OK
    pos = torch.tensor([n - 1 for n in lens], dtype=torch.int32)
    qsl = torch.arange(S + 1, dtype=torch.int32)
    st, full, _ = oracle.varlen_attention(w.q.cpu(), kb.cpu(), vb.cpu(), qsl, w.seq_lens, pos,
                                          w.block_tables, w.scale, sliding_window=1700,
                                          k_scales=ks, v_scales=vs)
    assert st == oracle.OK
    assert_attn_close(out, full, f"per-head split + reduce vs full {pool}")
