"""A seeded random sweep of varlen attention against the oracle: 24 batches drawn over GQA
ratios (1 to 16 query heads per kv head), head sizes 64 and 128, f32 and bf16 queries and
pools and fp8 pools with per-pool or per-kv-head scales, causal and non-causal masks,
sliding windows, attention sinks, and mixes of decode tokens, short chunks and
prefill-class chunks (so every kernel of the varlen call is reached).  Output within the
stated tolerance (tinyllm "Paged attention for decode in C", the naive-attention match) and
lse within 1e-3."""
import math
import random

import pytest
import torch

import oracle
from paged_kv_cache_31_gb300 import workloads
from tests.gpu_helpers import assert_attn_close

pytestmark = pytest.mark.gpu
DEV = "cuda"
HEADS = [(8, 8), (8, 2), (32, 8), (16, 1), (64, 8), (6, 2), (12, 4)]


@pytest.fixture(scope="module")
def pa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_31_gb300 import binding

    assert binding.pa_device_status() == binding.PA_OK
    return binding


def _draw(i):
    """Batch i of the sweep: every choice from a generator seeded with i."""
    rng = random.Random(1000 + i)
    H, Hkv = rng.choice(HEADS)
    D = rng.choice([64, 128, 128])
    pool = rng.choice(["bf16", "bf16", "f32", "fp8", "fp8-heads"])
    qdt = torch.float32 if pool == "f32" else torch.bfloat16
    causal = rng.random() < 0.85
    S = rng.randint(1, 10)
    seq_lens, q_lens = [], []
    for _ in range(S):
        n = rng.choice([rng.randint(1, 64), rng.randint(65, 1200), rng.randint(1201, 3000)])
        kind = rng.random()
        if kind < 0.5:
            q = 1
        elif kind < 0.8:
            q = rng.randint(1, min(n, 24))
        else:
            q = rng.randint(1, min(n, 400))
        seq_lens.append(n)
        q_lens.append(q)
    if not causal:  # keep the oracle's work bounded: short contexts without a mask
        seq_lens = [min(n, 700) for n in seq_lens]
        q_lens = [min(q, n) for q, n in zip(q_lens, seq_lens)]
    window = rng.choice([0, 0, rng.randint(1, 1500)])
    sinks = rng.random() < 0.3
    return dict(H=H, Hkv=Hkv, D=D, pool=pool, qdt=qdt, causal=causal, seq_lens=seq_lens,
                q_lens=q_lens, window=window, sinks=sinks, seed=2000 + i)


@pytest.mark.parametrize("i", range(24))
def test_random_batch_matches_oracle(pa, i):
    c = _draw(i)
    w = workloads.build(f"sweep-{i}", seq_lens=c["seq_lens"], q_lens=c["q_lens"],
                        num_heads=c["H"], num_kv_heads=c["Hkv"], head_dim=c["D"],
                        dtype=c["qdt"], causal=c["causal"], sliding_window=c["window"],
                        seed=c["seed"], device=DEV)
    kb, vb, kw, okw = w.k_blocks, w.v_blocks, {}, {}
    if c["pool"] == "fp8":
        kb, vb = workloads.fp8_pools(w)
        kw = okw = dict(k_scale=0.125, v_scale=0.125)
    elif c["pool"] == "fp8-heads":
        sp = [2.0 + 6.0 * g for g in range(c["Hkv"])]
        kb, vb = workloads.fp8_pools_per_head(w, sp)
        ks = torch.tensor([1.0 / x for x in sp], device=DEV)
        kw = okw = dict(k_scales=ks, v_scales=ks * 0.9)
    sinks = None
    if c["sinks"]:
        g = torch.Generator().manual_seed(c["seed"])
        sinks = torch.randn((w.num_heads,), generator=g) + 1.0
    out = torch.full_like(w.q, float("nan"))
    lse = torch.full((w.num_heads, w.num_tokens), float("nan"), device=DEV)
    pa.pa_varlen_forward(w.q, kb, vb, out, w.query_start_loc, w.seq_lens, w.positions,
                         w.block_tables, w.scale, causal=w.causal,
                         sliding_window=w.sliding_window, lse=lse,
                         sinks=None if sinks is None else sinks.to(DEV), **kw)
    assert pa.pa_device_status() == pa.PA_OK, c
    st, ref, ref_lse = oracle.varlen_attention(w.q.cpu(), kb.cpu(), vb.cpu(), w.query_start_loc,
                                               w.seq_lens, w.positions, w.block_tables, w.scale,
                                               causal=w.causal, sliding_window=w.sliding_window,
                                               want_lse=True, sinks=sinks, **okw)
    assert st == oracle.OK
    assert_attn_close(out, ref, f"sweep {i}: {c}")
    fin = torch.isfinite(ref_lse)
    assert torch.equal(torch.isinf(lse.cpu()), torch.isinf(ref_lse)), c
    if bool(fin.any()):
        err = (lse.cpu() - ref_lse).abs()
        assert float(err[fin].max()) < 1e-3 + 1e-4 * float(ref_lse[fin].abs().max()), c
