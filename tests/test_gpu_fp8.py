"""GPU parity of fp8 (e4m3) K/V pools ("paged_attention_v2_pytorch.py": kv_cache_dtype "fp8"
with k_scale / v_scale, K = k_scale * pool and V = v_scale * pool; tinyllm "Going further":
fp8 KV caches) against the oracle:

  - pa_reshape_and_cache_ex quantises new rows into the pool bit-exactly (the e4m3 code of
    x / scale, saturated, nearest-even), and into bf16 / f32 pools with a scale;
  - pa_reshape_and_cache and pa_gather_kv copy fp8 rows bit-exactly;
  - pa_varlen_forward_ex over fp8 pools (warp-MMA kernel for bf16 q and head size 128, the
    generic kernel otherwise) with scales, sinks and lse;
  - split-KV partials over fp8 pools, and partials + reduce against full attention.
"""
import math

import pytest
import torch

import oracle
from paged_kv_cache_31_gb300 import workloads
from tests.gpu_helpers import assert_attn_close

pytestmark = pytest.mark.gpu
DEV = "cuda"
KS, VS = 1.0 / 8, 0.11  # pools drawn with spread 8: K about N(0, 1), V about N(0, 0.88^2)


@pytest.fixture(scope="module")
def pa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_31_gb300 import binding

    assert binding.pa_device_status() == binding.PA_OK
    return binding


def _codes(t):
    return t.view(torch.uint8).cpu()


# ------------------------------------------------------------------------------------ scatter

def _special_values():
    """Values whose e4m3 rounding is decided at the edges: ties between neighbouring codes
    (normal and subnormal), just either side of a tie, saturation, zeros, infinities."""
    vals = [0.0, -0.0, 1.0625, 1.1875, -1.0625, 3 * 2.0 ** -10, 2.0 ** -10, 5 * 2.0 ** -10,
            2.0 ** -11, -(2.0 ** -11), 0.015625, 0.01953125, 448.0, 464.0, 465.0, 479.0, 1e6,
            -1e6, float("inf"), float("-inf"), 240.0, 232.0, 248.0, 0.001953125, 0.0029296875]
    x = torch.tensor(vals, dtype=torch.float32)
    up = torch.nextafter(x, torch.full_like(x, math.inf))
    dn = torch.nextafter(x, torch.full_like(x, -math.inf))
    return torch.cat([x, up, dn])


@pytest.mark.parametrize("src", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("T", [1, 37, 3000])  # the checked one-kernel path and the two-kernel one
def test_quantising_scatter_is_bit_exact(pa, src, T):
    Hkv, D, b, NB = 4, 128, 16, (3000 + 15) // 16 + 8
    g = torch.Generator().manual_seed(T + (src == torch.bfloat16))
    k = torch.randn((T, Hkv, D), generator=g) * 3
    v = torch.randn((T, Hkv, D), generator=g) * 120  # many saturate at v_scale 0.11
    sp = _special_values()
    n = min(sp.numel(), k.numel())
    k.view(-1)[:n] = sp[:n]
    v.view(-1)[-n:] = sp[:n] * 0.11
    k, v = k.to(src), v.to(src)
    slots = torch.randperm(NB * b, generator=g)[:T].to(torch.int32)
    kb = torch.zeros((NB, b, Hkv, D), dtype=torch.float8_e4m3fn)
    vb = torch.zeros_like(kb)
    st = oracle.reshape_and_cache_ex(k, v, kb, vb, slots, b, k_scale=0.25, v_scale=0.11)
    assert st == oracle.OK
    gkb = torch.zeros_like(kb, device=DEV)
    gvb = torch.zeros_like(vb, device=DEV)
    pa.pa_reshape_and_cache(k.to(DEV), v.to(DEV), gkb, gvb, slots.to(DEV), k_scale=0.25,
                            v_scale=0.11)
    assert pa.pa_device_status() == pa.PA_OK
    assert torch.equal(_codes(gkb), _codes(kb))
    assert torch.equal(_codes(gvb), _codes(vb))


@pytest.mark.parametrize("dst", [torch.bfloat16, torch.float32])
def test_scaled_scatter_into_wide_pools(pa, dst):
    Hkv, D, b, NB, T = 2, 64, 16, 8, 50
    g = torch.Generator().manual_seed(5)
    k = torch.randn((T, Hkv, D), generator=g)
    v = torch.randn((T, Hkv, D), generator=g)
    slots = torch.randperm(NB * b, generator=g)[:T].to(torch.int32)
    kb = torch.zeros((NB, b, Hkv, D), dtype=dst)
    vb = torch.zeros_like(kb)
    assert oracle.reshape_and_cache_ex(k, v, kb, vb, slots, b, k_scale=0.3,
                                       v_scale=1.7) == oracle.OK
    gkb, gvb = torch.zeros_like(kb, device=DEV), torch.zeros_like(vb, device=DEV)
    pa.pa_reshape_and_cache(k.to(DEV), v.to(DEV), gkb, gvb, slots.to(DEV), k_scale=0.3,
                            v_scale=1.7)
    assert pa.pa_device_status() == pa.PA_OK
    assert torch.equal(gkb.cpu(), kb) and torch.equal(gvb.cpu(), vb)


def test_quantising_scatter_checks_slots_and_scales(pa):
    Hkv, D, b, NB, T = 2, 128, 16, 4, 9
    k = torch.randn((T, Hkv, D), device=DEV)
    kb = torch.zeros((NB, b, Hkv, D), dtype=torch.float8_e4m3fn, device=DEV)
    vb = torch.zeros_like(kb)
    bad = torch.arange(T, dtype=torch.int32, device=DEV)
    bad[4] = NB * b  # one slot past the pool: nothing is written
    pa.pa_reshape_and_cache(k, k, kb, vb, bad, k_scale=0.5, v_scale=0.5)
    assert pa.pa_device_status() == pa.PA_EINVAL
    assert int(_codes(kb).count_nonzero()) == 0
    ok = torch.arange(T, dtype=torch.int32, device=DEV)
    for ks in (0.0, -1.0, float("inf"), float("nan")):
        with pytest.raises(pa.PaError) as e:
            pa.pa_reshape_and_cache(k, k, kb, vb, ok, k_scale=ks, v_scale=0.5)
        assert e.value.status == pa.PA_EINVAL
    assert pa.pa_device_status() == pa.PA_OK


@pytest.mark.parametrize("Hkv,D", [(2, 128), (3, 7)])  # 16-byte rows and odd-byte rows
def test_fp8_copy_scatter_and_gather_are_bit_exact(pa, Hkv, D):
    b, NB, T = 16, 12, 40
    g = torch.Generator().manual_seed(D)
    rows = torch.randint(0, 256, (T, Hkv, D), generator=g, dtype=torch.uint8)
    rows[rows == 0x7F] = 0  # NaN codes aside, any byte is a code
    rows[rows == 0xFF] = 0
    k = rows.view(torch.float8_e4m3fn)
    v = rows.flip(0).contiguous().view(torch.float8_e4m3fn)
    slots = torch.randperm(NB * b, generator=g)[:T].to(torch.int32)
    kb = torch.zeros((NB, b, Hkv, D), dtype=torch.float8_e4m3fn)
    vb = torch.zeros_like(kb)
    assert oracle.reshape_and_cache(k, v, kb, vb, slots, b) == oracle.OK
    gkb, gvb = torch.zeros_like(kb, device=DEV), torch.zeros_like(vb, device=DEV)
    pa.pa_reshape_and_cache(k.to(DEV), v.to(DEV), gkb, gvb, slots.to(DEV))
    assert pa.pa_device_status() == pa.PA_OK
    assert torch.equal(_codes(gkb), _codes(kb)) and torch.equal(_codes(gvb), _codes(vb))
    # gather two sequences back out through a table
    table = torch.randperm(NB, generator=g)[:10].to(torch.int32).view(2, 5)
    cu = torch.tensor([0, 33, 70], dtype=torch.int32)
    st, ko, vo = oracle.gather_kv(kb, vb, cu, table)
    assert st == oracle.OK
    gko = torch.empty((70, Hkv, D), dtype=torch.float8_e4m3fn, device=DEV)
    gvo = torch.empty_like(gko)
    pa.pa_gather_kv(gkb, gvb, gko, gvo, cu.to(DEV), table.to(DEV))
    assert pa.pa_device_status() == pa.PA_OK
    assert torch.equal(_codes(gko), _codes(ko)) and torch.equal(_codes(gvo), _codes(vo))


# ---------------------------------------------------------------------------------- attention

CASES = {
    # decode tokens on the fp8 warp-MMA kernel, GQA 4
    "decode": dict(seq_lens=[1, 17, 300, 1000, 4096], q_lens=[1] * 5, num_heads=32,
                   num_kv_heads=8, head_dim=128),
    # prefill chunks too: the tcgen05 kernel widens the codes to f16 in shared memory
    "prefill": dict(seq_lens=[512, 700, 1300, 90, 2000], q_lens=[512, 200, 130, 1, 1],
                    num_heads=32, num_kv_heads=8, head_dim=128),
    # sliding window, GQA 2
    "window": dict(seq_lens=[900, 2500, 3000], q_lens=[300, 1, 1], num_heads=16, num_kv_heads=8,
                   head_dim=128, sliding_window=256),
    # one kv head for 16 query heads
    "mqa": dict(seq_lens=[33, 1025, 64], q_lens=[1, 3, 64], num_heads=16, num_kv_heads=1,
                head_dim=128),
    # the generic kernel: head size 64, and fp32 q
    "simt-d64": dict(seq_lens=[1, 40, 77], q_lens=[1, 40, 2], num_heads=8, num_kv_heads=2,
                     head_dim=64),
    "simt-fp32q": dict(seq_lens=[5, 130], q_lens=[5, 1], num_heads=4, num_kv_heads=2,
                       head_dim=128, dtype=torch.float32),
}


def _case(name, seed):
    w = workloads.build(name, seed=seed, device=DEV, **CASES[name])
    kb8, vb8 = workloads.fp8_pools(w)
    return w, kb8, vb8


def _nan_tail(w, kb8, vb8):
    """NaN codes in the never-written rows of each sequence's last block: they must not reach
    the output (the attention never reads them as values)."""
    bs = w.block_size
    tab = w.block_tables.cpu()
    for s, n in enumerate(w.seq_lens_list):
        if n % bs:
            blk = int(tab[s, (n - 1) // bs])
            kb8.view(torch.uint8)[blk, n % bs:] = 0x7F
            vb8.view(torch.uint8)[blk, n % bs:] = 0xFF


@pytest.mark.parametrize("case", sorted(CASES))
def test_fp8_attention_matches_oracle(pa, case):
    seed = sorted(CASES).index(case) + 51
    w, kb8, vb8 = _case(case, seed)
    _nan_tail(w, kb8, vb8)
    g = torch.Generator().manual_seed(seed)
    sinks = torch.randn((w.num_heads,), generator=g) + 1.0
    sinks[::3] = -math.inf
    out = torch.full_like(w.q, float("nan"))
    lse = torch.full((w.num_heads, w.num_tokens), float("nan"), device=DEV)
    pa.pa_varlen_forward(w.q, kb8, vb8, out, w.query_start_loc, w.seq_lens, w.positions,
                         w.block_tables, w.scale, causal=w.causal,
                         sliding_window=w.sliding_window, sinks=sinks.to(DEV), lse=lse,
                         k_scale=KS, v_scale=VS)
    assert pa.pa_device_status() == pa.PA_OK
    st, ref, ref_lse = oracle.varlen_attention(w.q.cpu(), kb8.cpu(), vb8.cpu(), w.query_start_loc,
                                               w.seq_lens, w.positions, w.block_tables, w.scale,
                                               causal=w.causal, sliding_window=w.sliding_window,
                                               want_lse=True, sinks=sinks, k_scale=KS,
                                               v_scale=VS)
    assert st == oracle.OK
    assert_attn_close(out, ref, f"fp8 {case}")
    err = (lse.cpu() - ref_lse).abs()
    fin = torch.isfinite(ref_lse)
    assert torch.equal(torch.isinf(lse.cpu()), torch.isinf(ref_lse))
    assert float(err[fin].max()) < 1e-3 + 1e-4 * float(ref_lse[fin].abs().max())
    # deterministic
    out2 = torch.empty_like(out)
    pa.pa_varlen_forward(w.q, kb8, vb8, out2, w.query_start_loc, w.seq_lens, w.positions,
                         w.block_tables, w.scale, causal=w.causal,
                         sliding_window=w.sliding_window, sinks=sinks.to(DEV), lse=lse,
                         k_scale=KS, v_scale=VS)
    assert torch.equal(out, out2)


def test_fp8_scales_fold_exactly(pa):
    # k_scale enters the scores like the softmax scale; v_scale multiplies the output
    w, kb8, vb8 = _case("decode", 61)
    run = lambda scale, ks, vs: pa.pa_varlen_forward(
        w.q, kb8, vb8, torch.empty_like(w.q), w.query_start_loc, w.seq_lens, w.positions,
        w.block_tables, scale, k_scale=ks, v_scale=vs).float()
    a = run(w.scale * 0.25, 1.0, 1.0)
    b = run(w.scale, 0.25, 1.0)
    assert_attn_close(b, a, "k_scale as softmax scale")
    c = run(w.scale, 0.25, 2.0)
    assert_attn_close(c, 2.0 * a, "v_scale doubles")
    assert pa.pa_device_status() == pa.PA_OK


def test_fp8_rejects_bad_scales(pa):
    w, kb8, vb8 = _case("decode", 62)
    for ks in (0.0, -0.5, float("inf"), float("nan")):
        with pytest.raises(pa.PaError) as e:
            pa.pa_varlen_forward(w.q, kb8, vb8, torch.empty_like(w.q), w.query_start_loc,
                                 w.seq_lens, w.positions, w.block_tables, w.scale, k_scale=ks)
        assert e.value.status == pa.PA_EINVAL
    assert pa.pa_device_status() == pa.PA_OK


@pytest.mark.parametrize("H,Hkv,D", [(32, 8, 128), (8, 2, 64)])  # warp-MMA kernel, generic one
def test_fp8_splitkv(pa, H, Hkv, D):
    lens = [1, 511, 512, 513, 1500, 4100]
    w = workloads.build("split-fp8", seq_lens=lens, q_lens=[1] * len(lens), num_heads=H,
                        num_kv_heads=Hkv, head_dim=D, seed=H + D, device=DEV,
                        sliding_window=1700, partition_size=512)
    kb8, vb8 = workloads.fp8_pools(w)
    _nan_tail(w, kb8, vb8)
    P, MP, S = 512, w.max_partitions(), len(lens)
    ml = torch.full((S, H, MP), float("nan"), device=DEV)
    es = torch.full_like(ml, float("nan"))
    to = torch.full((S, H, MP, D), float("nan"), device=DEV)
    pa.pa_decode_splitkv_partials(w.q, kb8, vb8, ml, es, to, w.seq_lens, w.block_tables,
                                  w.scale, partition_size=P, sliding_window=1700, k_scale=KS,
                                  v_scale=VS)
    assert pa.pa_device_status() == pa.PA_OK
    st, rml, res, rto = oracle.splitkv_partials(w.q.cpu(), kb8.cpu(), vb8.cpu(), w.seq_lens,
                                                w.block_tables, w.scale, P, MP, 1700,
                                                k_scale=KS, v_scale=VS)
    assert st == oracle.OK
    assert torch.equal(torch.isinf(ml.cpu()), torch.isinf(rml))
    fin = torch.isfinite(rml)
    assert float((ml.cpu()[fin] - rml[fin]).abs().max()) < 1e-3
    assert float(((es.cpu() - res).abs() / res.clamp_min(1e-30))[res > 0].max()) < 2e-3
    assert_attn_close(to, rto, "fp8 split tmp_out")
    out = torch.empty_like(w.q)
    pa.pa_decode_splitkv_reduce(out, ml, es, to, w.seq_lens, partition_size=P)
    assert pa.pa_device_status() == pa.PA_OK
    pos = torch.tensor([n - 1 for n in lens], dtype=torch.int32)
    qsl = torch.arange(S + 1, dtype=torch.int32)
    st, full, _ = oracle.varlen_attention(w.q.cpu(), kb8.cpu(), vb8.cpu(), qsl, w.seq_lens, pos,
                                          w.block_tables, w.scale, sliding_window=1700,
                                          k_scale=KS, v_scale=VS)
    assert st == oracle.OK
    assert_attn_close(out, full, "fp8 split + reduce vs full")
