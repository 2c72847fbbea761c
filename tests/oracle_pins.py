"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each ``pin_*`` function raises AssertionError when the oracle disagrees with a
value, identity or special case that does not come from the oracle itself:

* the tinyllm page's worked example (section 3, golden/hand_example.json);
* brute-force dense attention in float64 over the *dense* per-sequence keys and
  values, from which the paged pool is built (tinyllm section 4,
  matches_naive_over_the_gathered_cache: GQA 6:2, D = 32, lengths 1 / 37 / 70,
  windows 0 and 20);
* closed forms (one visible key, a zero query, constant values), with and without
  attention sinks (TensorSharp ForwardWithSinks);
* invariances (permuted physical block ids, a sequence alone vs in a batch,
  shared prefix blocks vs private copies, thread count);
* the log-sum-exp identities behind split-KV and merge_attn_states, and the
  merge's infinite-lse special cases (vllm.cpp cpu_mla_prefill.cpp,
  MergeAttnStatesKernel);
* the validation contract (tinyllm section 2.6 / bad_tables_and_shapes);
* bfloat16 rounding against torch's own conversion, and the fp8 (e4m3) codes of every value
  against torch's float8_e4m3fn (with the pools' dequantisation scales).

The mutant test (test_oracle_mutants.py) plants known mistakes in the oracle
and checks that each is caught by at least one of these pins.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

import oracle
from paged_kv_cache_31_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _t(x, dtype=torch.int32):
    return torch.tensor(x, dtype=dtype)


# --------------------------------------------------------------------------------------------
# worked example (tinyllm section 3)


def _hand():
    with open(os.path.join(GOLDEN, "hand_example.json")) as f:
        g = json.load(f)
    NB, b, D = g["num_blocks"], g["block_size"], g["head_dim"]
    kb = torch.zeros((NB, b, 1, D), dtype=torch.float32)
    vb = torch.zeros((NB, b, 1, D), dtype=torch.float32)
    for j in range(g["context_len"]):
        kb[g["block_of_position"][j], g["slot_of_position"][j], 0] = torch.tensor(g["keys"][j])
        vb[g["block_of_position"][j], g["slot_of_position"][j], 0] = torch.tensor(g["values"][j])
    return g, kb, vb


def pin_hand_example():
    g, kb, vb = _hand()
    q = torch.tensor([[g["q"]]], dtype=torch.float32)
    meta = dict(query_start_loc=_t([0, 1]), seq_lens=_t([g["context_len"]]),
                positions=_t([g["query_position"]]), block_tables=_t([g["block_table"]]))
    for scale in (1.0, 0.37, 2.5, -0.8):
        st, out, lse = oracle.varlen_attention(q, kb, vb, scale=scale, want_lse=True, **meta)
        assert st == oracle.OK
        np.testing.assert_allclose(out[0, 0].numpy(), g["output"], rtol=0, atol=2e-6)
    # scale 1: running max 1 and denominator 2.3678794 -> lse = 1 + ln(2.3678794)
    st, out, lse = oracle.varlen_attention(q, kb, vb, scale=g["scale_for_intermediates"],
                                           want_lse=True, **meta)
    want = g["running_max"] + math.log(g["ell_final"])
    assert abs(float(lse[0, 0]) - want) < 1e-6, (float(lse[0, 0]), want)


def pin_hand_example_via_cache():
    """The same example written through slot mapping + scatter (tinyllm section 4,
    second hand_example row: the cache and the kernel share one layout)."""
    g, _, _ = _hand()
    NB, b, D = g["num_blocks"], g["block_size"], g["head_dim"]
    n = g["context_len"]
    qsl, pos, bt = _t([0, n]), _t(list(range(n))), _t([g["block_table"]])
    st, slots = oracle.slot_mapping(qsl, pos, bt, b, NB)
    assert st == oracle.OK
    want_slots = [g["block_of_position"][j] * b + g["slot_of_position"][j] for j in range(n)]
    assert slots.tolist() == want_slots, (slots.tolist(), want_slots)
    kb = torch.zeros((NB, b, 1, D))
    vb = torch.zeros((NB, b, 1, D))
    k = torch.tensor(g["keys"], dtype=torch.float32).view(n, 1, D)
    v = torch.tensor(g["values"], dtype=torch.float32).view(n, 1, D)
    assert oracle.reshape_and_cache(k, v, kb, vb, slots, b) == oracle.OK
    q = torch.tensor([[g["q"]]], dtype=torch.float32)
    st, out, _ = oracle.varlen_attention(q, kb, vb, _t([0, 1]), _t([n]),
                                         _t([g["query_position"]]), bt, scale=1.0)
    assert st == oracle.OK
    np.testing.assert_allclose(out[0, 0].numpy(), g["output"], rtol=0, atol=2e-6)


# --------------------------------------------------------------------------------------------
# brute force over the dense per-sequence cache


def _paged_from_dense(dense_k, dense_v, block_size, seed, extra_blocks=3):
    """Place each sequence's dense rows [n, Hkv, D] into a pool under a shuffled table:
    position j of sequence s goes to row j mod b of block table[s][j // b]."""
    gen = torch.Generator().manual_seed(seed)
    need = [(k.shape[0] + block_size - 1) // block_size for k in dense_k]
    NB = sum(need) + extra_blocks
    Hkv, D = dense_k[0].shape[1], dense_k[0].shape[2]
    perm = torch.randperm(NB, generator=gen).to(torch.int32)
    kb = torch.randn((NB, block_size, Hkv, D), generator=gen)
    vb = torch.randn((NB, block_size, Hkv, D), generator=gen)
    MB = max(need)
    table = torch.zeros((len(dense_k), MB), dtype=torch.int32)
    c = 0
    for s, (k, v) in enumerate(zip(dense_k, dense_v)):
        table[s, :need[s]] = perm[c:c + need[s]]
        c += need[s]
        for j in range(k.shape[0]):
            kb[table[s, j // block_size], j % block_size] = k[j]
            vb[table[s, j // block_size], j % block_size] = v[j]
    return kb, vb, table


def _dense_attention_f64(q, k, v, pos, n, scale, causal, window):
    """Plain softmax attention of queries q [Tq, H, D] at positions pos over the dense
    keys/values k, v [n, Hkv, D], with an explicit boolean mask, in float64.
    GQA expands each kv head to H / Hkv consecutive query heads (np.repeat)."""
    H, Hkv = q.shape[1], k.shape[1]
    kk = np.repeat(k.astype(np.float64), H // Hkv, axis=1)  # [n, H, D]
    vv = np.repeat(v.astype(np.float64), H // Hkv, axis=1)
    j = np.arange(n)[None, :]
    p = np.asarray(pos)[:, None]
    end = p + 1 if causal else np.full_like(p, n)
    vis = j < end
    if window > 0:
        vis &= j >= end - window
    out = np.zeros(q.shape, dtype=np.float64)
    for h in range(H):
        s = (q[:, h, :].astype(np.float64) @ kk[:, h, :].T) * scale  # [Tq, n]
        s = np.where(vis, s, -np.inf)
        s = s - s.max(axis=1, keepdims=True)
        e = np.exp(s)
        out[:, h, :] = (e / e.sum(axis=1, keepdims=True)) @ vv[:, h, :]
    return out


def pin_brute_force(window=0, causal=True, mixed=False, seed=3):
    H, Hkv, D, b = 6, 2, 32, 16
    lens = [1, 37, 70]
    qlens = [1, 5, 70] if mixed else [1, 1, 1]
    gen = torch.Generator().manual_seed(seed)
    dk = [torch.randn((n, Hkv, D), generator=gen) for n in lens]
    dv = [torch.randn((n, Hkv, D), generator=gen) for n in lens]
    kb, vb, table = _paged_from_dense(dk, dv, b, seed + 1)
    T = sum(qlens)
    q = torch.randn((T, H, D), generator=gen)
    qsl = np.cumsum([0] + qlens).tolist()
    pos = [p for n, ql in zip(lens, qlens) for p in range(n - ql, n)]
    scale = 1.0 / math.sqrt(D)
    st, out, _ = oracle.varlen_attention(q, kb, vb, _t(qsl), _t(lens), _t(pos), table,
                                         scale=scale, causal=causal, sliding_window=window)
    assert st == oracle.OK
    for s, n in enumerate(lens):
        a, z = qsl[s], qsl[s + 1]
        want = _dense_attention_f64(q[a:z].numpy(), dk[s].numpy(), dv[s].numpy(), pos[a:z], n,
                                    scale, causal, window)
        np.testing.assert_allclose(out[a:z].numpy(), want, rtol=1e-5, atol=2e-5)


def pin_brute_force_all():
    for window in (0, 20):
        pin_brute_force(window=window)
        pin_brute_force(window=window, mixed=True)
    pin_brute_force(window=0, causal=False, mixed=True)
    pin_brute_force(window=20, causal=False, mixed=True)


# --------------------------------------------------------------------------------------------
# closed forms


def pin_closed_forms():
    w = workloads.build("closed", seq_lens=[1, 40, 70], q_lens=[1, 3, 2], num_heads=4,
                        num_kv_heads=2, head_dim=16, dtype=torch.float32, seed=11)
    meta = dict(query_start_loc=w.query_start_loc, seq_lens=w.seq_lens, positions=w.positions,
                block_tables=w.block_tables)
    G = w.group
    # (a) window of one position: each query sees only itself -> o = v at its own position
    st, out, _ = oracle.varlen_attention(w.q, w.k_blocks, w.v_blocks, scale=w.scale,
                                         sliding_window=1, **meta)
    assert st == oracle.OK
    for t in range(w.num_tokens):
        s = int(np.searchsorted(w.query_start_loc.numpy(), t, side="right") - 1)
        p = int(w.positions[t])
        blk = int(w.block_tables[s, p // w.block_size])
        for h in range(w.num_heads):
            assert torch.equal(out[t, h], w.v_blocks[blk, p % w.block_size, h // G]), (t, h)
    # (b) a zero query: uniform weights -> the mean of the visible values
    qz = torch.zeros_like(w.q)
    st, out, _ = oracle.varlen_attention(qz, w.k_blocks, w.v_blocks, scale=w.scale, **meta)
    assert st == oracle.OK
    for t in range(w.num_tokens):
        s = int(np.searchsorted(w.query_start_loc.numpy(), t, side="right") - 1)
        p = int(w.positions[t])
        rows = [w.v_blocks[int(w.block_tables[s, j // 16]), j % 16].double() for j in range(p + 1)]
        mean = torch.stack(rows).mean(0)  # [Hkv, D]
        for h in range(w.num_heads):
            np.testing.assert_allclose(out[t, h].numpy(), mean[h // G].numpy(), rtol=1e-5,
                                       atol=1e-6)
    # (c) constant values -> that constant, whatever the scores
    vc = torch.full_like(w.v_blocks, 0.625)
    st, out, _ = oracle.varlen_attention(w.q, w.k_blocks, vc, scale=w.scale, **meta)
    assert st == oracle.OK
    np.testing.assert_allclose(out.numpy(), 0.625, rtol=1e-6, atol=0)


# --------------------------------------------------------------------------------------------
# attention sinks (TensorSharp ForwardWithSinks): a virtual position per head whose score is
# the sink logit and whose value is zero


def _sink_case(seed=41):
    w = workloads.build("sinks", seq_lens=[3, 40, 70], q_lens=[1, 3, 2], num_heads=4,
                        num_kv_heads=2, head_dim=16, dtype=torch.float32, seed=seed)
    meta = dict(query_start_loc=w.query_start_loc, seq_lens=w.seq_lens, positions=w.positions,
                block_tables=w.block_tables)
    return w, meta, torch.tensor([-1.5, 0.7, 2.0, -0.3], dtype=torch.float32)


def pin_sinks_closed_forms():
    w, meta, sinks = _sink_case()
    G = w.group
    # (a) -inf sinks are no sinks: the same bits for o and lse
    st, o0, l0 = oracle.varlen_attention(w.q, w.k_blocks, w.v_blocks, scale=w.scale,
                                         want_lse=True, **meta)
    st1, o1, l1 = oracle.varlen_attention(w.q, w.k_blocks, w.v_blocks, scale=w.scale,
                                          want_lse=True, sinks=torch.full((4,), -math.inf),
                                          **meta)
    assert st == oracle.OK and st1 == oracle.OK
    assert torch.equal(o0, o1) and torch.equal(l0, l1)
    # (b) a zero query: every visible score is 0, so each of the n visible values gets weight
    # 1 / (n + e^sink) and lse = log(n + e^sink)
    qz = torch.zeros_like(w.q)
    st, out, lse = oracle.varlen_attention(qz, w.k_blocks, w.v_blocks, scale=w.scale,
                                           want_lse=True, sinks=sinks, **meta)
    assert st == oracle.OK
    for t in range(w.num_tokens):
        s = int(np.searchsorted(w.query_start_loc.numpy(), t, side="right") - 1)
        p = int(w.positions[t])
        rows = [w.v_blocks[int(w.block_tables[s, j // 16]), j % 16].double() for j in range(p + 1)]
        total = torch.stack(rows).sum(0)  # [Hkv, D]
        n = p + 1
        for h in range(w.num_heads):
            den = n + math.exp(float(sinks[h]))
            np.testing.assert_allclose(out[t, h].numpy(), (total[h // G] / den).numpy(),
                                       rtol=1e-5, atol=1e-6)
            assert abs(float(lse[h, t]) - math.log(den)) < 1e-5, (t, h)


def pin_sinks_brute_force(seed=43):
    """Float64 softmax over [visible scores..., sink] with values [visible v..., 0]."""
    H, Hkv, D, b = 6, 2, 32, 16
    lens, qlens = [1, 37, 70], [1, 5, 70]
    gen = torch.Generator().manual_seed(seed)
    dk = [torch.randn((n, Hkv, D), generator=gen) for n in lens]
    dv = [torch.randn((n, Hkv, D), generator=gen) for n in lens]
    kb, vb, table = _paged_from_dense(dk, dv, b, seed + 1)
    T = sum(qlens)
    q = torch.randn((T, H, D), generator=gen)
    sinks = torch.randn((H,), generator=gen) * 2.0
    qsl = np.cumsum([0] + qlens).tolist()
    pos = [p for n, ql in zip(lens, qlens) for p in range(n - ql, n)]
    scale = 1.0 / math.sqrt(D)
    for window in (0, 20):
        st, out, lse = oracle.varlen_attention(q, kb, vb, _t(qsl), _t(lens), _t(pos), table,
                                               scale=scale, sliding_window=window,
                                               want_lse=True, sinks=sinks)
        assert st == oracle.OK
        for s, n in enumerate(lens):
            a, z = qsl[s], qsl[s + 1]
            kk = np.repeat(dk[s].numpy().astype(np.float64), H // Hkv, axis=1)
            vv = np.repeat(dv[s].numpy().astype(np.float64), H // Hkv, axis=1)
            j = np.arange(n)[None, :]
            end = np.asarray(pos[a:z])[:, None] + 1
            vis = j < end
            if window > 0:
                vis &= j >= end - window
            for h in range(H):
                sc = (q[a:z, h, :].numpy().astype(np.float64) @ kk[:, h, :].T) * scale
                sc = np.where(vis, sc, -np.inf)
                sc = np.concatenate([sc, np.full((z - a, 1), float(sinks[h]))], axis=1)
                mx = sc.max(axis=1, keepdims=True)
                e = np.exp(sc - mx)
                want = (e[:, :n] @ vv[:, h, :]) / e.sum(axis=1, keepdims=True)
                np.testing.assert_allclose(out[a:z, h].numpy(), want, rtol=1e-5, atol=2e-5)
                want_lse = (mx[:, 0] + np.log(e.sum(axis=1)))
                np.testing.assert_allclose(lse[h, a:z].numpy(), want_lse, rtol=1e-5, atol=2e-5)


# --------------------------------------------------------------------------------------------
# fp8 (e4m3) K/V pools with dequantisation scales (the V2 page's kv_cache_dtype "fp8",
# k_scale / v_scale: attention uses K = k_scale * pool, V = v_scale * pool)


def pin_fp8_codec():
    # decoding: every code, against torch's float8_e4m3fn
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).float()
    got = torch.tensor([oracle.fp8_to_f32(int(c)) for c in codes])
    assert bool(((ref == got) | (ref.isnan() & got.isnan())).all())
    # encoding: saturate to +-448, then round to nearest even -- torch's cast after a clamp
    # (values: every midpoint between neighbouring codes, their neighbours, and a sweep)
    fin = ref[(codes < 127)]  # non-negative finite codes, increasing
    mids = (fin[:-1] + fin[1:]) / 2
    g = torch.Generator().manual_seed(71)
    sweep = torch.randn(4000, generator=g) * torch.exp(torch.randn(4000, generator=g) * 3)
    xs = torch.cat([mids, torch.nextafter(mids, torch.zeros_like(mids)),
                    torch.nextafter(mids, torch.full_like(mids, 1e4)), sweep, -sweep,
                    torch.tensor([0.0, -0.0, 448.0, 449.0, 1e6, -1e6, 2.0 ** -10])])
    want = torch.clamp(xs, -448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
    got = torch.tensor([oracle.f32_to_fp8(float(x)) for x in xs], dtype=torch.uint8)
    assert torch.equal(got, want)


def pin_fp8_scatter():
    # the pool receives the e4m3 code of x / scale, exactly as torch quantises it
    g = torch.Generator().manual_seed(72)
    T, Hkv, D, b, NB = 20, 2, 32, 16, 4
    k = (torch.randn((T, Hkv, D), generator=g) * 3).to(torch.bfloat16)
    v = (torch.randn((T, Hkv, D), generator=g) * 100).to(torch.bfloat16)
    kb = torch.zeros((NB, b, Hkv, D), dtype=torch.float8_e4m3fn)
    vb = torch.zeros_like(kb)
    slots = torch.randperm(NB * b, generator=g)[:T].to(torch.int32)
    ks, vs = 0.0625, 0.37
    st = oracle.reshape_and_cache_ex(k, v, kb, vb, slots, b, k_scale=ks, v_scale=vs)
    assert st == oracle.OK
    q = lambda x, sc: torch.clamp(x.float() / sc, -448, 448).to(torch.float8_e4m3fn)
    for t in range(T):
        sl = int(slots[t])
        assert torch.equal(kb[sl // b, sl % b].view(torch.uint8), q(k[t], ks).view(torch.uint8))
        assert torch.equal(vb[sl // b, sl % b].view(torch.uint8), q(v[t], vs).view(torch.uint8))


def _fp8_case(seed=73):
    H, Hkv, D, b = 6, 2, 32, 16
    lens, qlens = [1, 37, 70], [1, 5, 70]
    gen = torch.Generator().manual_seed(seed)
    dk = [torch.randn((n, Hkv, D), generator=gen) for n in lens]
    dv = [torch.randn((n, Hkv, D), generator=gen) for n in lens]
    kb, vb, table = _paged_from_dense(dk, dv, b, seed + 1)
    kb8, vb8 = (kb * 4).to(torch.float8_e4m3fn), (vb * 4).to(torch.float8_e4m3fn)
    T = sum(qlens)
    q = torch.randn((T, H, D), generator=gen)
    qsl = np.cumsum([0] + qlens).tolist()
    pos = [p for n, ql in zip(lens, qlens) for p in range(n - ql, n)]
    return H, Hkv, D, lens, qsl, pos, q, kb8, vb8, table


def pin_fp8_attention_brute_force():
    H, Hkv, D, lens, qsl, pos, q, kb8, vb8, table = _fp8_case()
    ks, vs = 0.25, 0.37
    scale = 1.0 / math.sqrt(D)
    for window in (0, 20):
        st, out, _ = oracle.varlen_attention(q, kb8, vb8, _t(qsl), _t(lens), _t(pos), table,
                                             scale=scale, sliding_window=window, k_scale=ks,
                                             v_scale=vs)
        assert st == oracle.OK
        for s, n in enumerate(lens):
            rows = [table[s, j // 16] for j in range(n)]
            dk = torch.stack([kb8[int(rows[j]), j % 16].float() for j in range(n)]) * ks
            dv = torch.stack([vb8[int(rows[j]), j % 16].float() for j in range(n)]) * vs
            a, z = qsl[s], qsl[s + 1]
            want = _dense_attention_f64(q[a:z].numpy(), dk.numpy(), dv.numpy(), pos[a:z], n,
                                        scale, True, window)
            np.testing.assert_allclose(out[a:z].numpy(), want, rtol=1e-5, atol=2e-5)


def pin_dequant_scales():
    # k_scale multiplies every score exactly as the softmax scale does; v_scale multiplies the
    # output (a bf16 pool here: the scales are general dequantisation factors)
    w = workloads.build("scales", seq_lens=[5, 40, 70], q_lens=[1, 3, 2], num_heads=4,
                        num_kv_heads=2, head_dim=16, dtype=torch.float32, seed=74)
    meta = dict(query_start_loc=w.query_start_loc, seq_lens=w.seq_lens, positions=w.positions,
                block_tables=w.block_tables)
    st, o1, l1 = oracle.varlen_attention(w.q, w.k_blocks, w.v_blocks, scale=w.scale * 2.5,
                                         want_lse=True, **meta)
    st2, o2, l2 = oracle.varlen_attention(w.q, w.k_blocks, w.v_blocks, scale=w.scale,
                                          want_lse=True, k_scale=2.5, v_scale=3.0, **meta)
    assert st == oracle.OK and st2 == oracle.OK
    np.testing.assert_allclose(o2.numpy(), 3.0 * o1.numpy(), rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(l2.numpy(), l1.numpy(), rtol=1e-5, atol=1e-6)


# --------------------------------------------------------------------------------------------
# invariances


def _run(w, **kw):
    st, out, lse = oracle.varlen_attention(w.q, w.k_blocks, w.v_blocks, w.query_start_loc,
                                           w.seq_lens, w.positions, w.block_tables, w.scale,
                                           causal=w.causal, sliding_window=w.sliding_window,
                                           want_lse=True, **kw)
    assert st == oracle.OK
    return out, lse


def pin_block_permutation_invariance():
    w = workloads.build("perm", seq_lens=[5, 33, 64, 90], q_lens=[1, 4, 64, 1], num_heads=8,
                        num_kv_heads=2, head_dim=32, dtype=torch.bfloat16, seed=5,
                        sliding_window=40)
    out0, lse0 = _run(w)
    perm = torch.randperm(w.num_blocks, generator=torch.Generator().manual_seed(9))
    kb = torch.empty_like(w.k_blocks)
    vb = torch.empty_like(w.v_blocks)
    kb[perm] = w.k_blocks  # physical block b moves to id perm[b]
    vb[perm] = w.v_blocks
    w.k_blocks, w.v_blocks = kb, vb
    w.block_tables = perm[w.block_tables.long()].to(torch.int32)
    out1, lse1 = _run(w)
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)


def pin_batch_invariance_and_shared_prefix():
    """16 sequences sharing two prefix blocks (tinyllm shared_blocks_and_batch_invariance):
    each alone gives the same bits as in the batch, and the shared blocks read the same
    as private copies of them."""
    gen = torch.Generator().manual_seed(21)
    lens = [int(x) for x in torch.randint(33, 80, (16,), generator=gen)]
    w = workloads.build("fork", seq_lens=lens, q_lens=[1] * 16, num_heads=8, num_kv_heads=4,
                        head_dim=32, dtype=torch.bfloat16, seed=21, shared_prefix_blocks=2,
                        extra_table_cols=2)
    out_b, _ = _run(w)
    for s in range(16):
        st, out_1, _ = oracle.varlen_attention(
            w.q[s:s + 1], w.k_blocks, w.v_blocks, _t([0, 1]), w.seq_lens[s:s + 1],
            w.positions[s:s + 1], w.block_tables[s:s + 1].contiguous(), w.scale)
        assert st == oracle.OK and torch.equal(out_1[0], out_b[s]), s
    # private copies of the two prefix blocks for every sequence
    NB = w.num_blocks
    kb = torch.cat([w.k_blocks] + [w.k_blocks[w.block_tables[0, :2].long()]] * 16)
    vb = torch.cat([w.v_blocks] + [w.v_blocks[w.block_tables[0, :2].long()]] * 16)
    bt = w.block_tables.clone()
    for s in range(16):
        bt[s, 0], bt[s, 1] = NB + 2 * s, NB + 2 * s + 1
    w.k_blocks, w.v_blocks, w.block_tables, w.num_blocks = kb, vb, bt, kb.shape[0]
    out_p, _ = _run(w)
    assert torch.equal(out_b, out_p)


def pin_thread_invariance():
    w = workloads.named(3, small=True)
    n = oracle.num_threads()
    try:
        oracle.set_num_threads(1)
        out1, lse1 = _run(w)
        oracle.set_num_threads(max(2, n))
        outn, lsen = _run(w)
    finally:
        oracle.set_num_threads(n)
    assert torch.equal(out1, outn) and torch.equal(lse1, lsen)


# --------------------------------------------------------------------------------------------
# split-KV (PagedAttention V2 partitions and log-sum-exp reduction)


def _split_case(window=0, seed=31):
    lens = [1, 511, 512, 513, 1500, 2100]
    return workloads.build("split", seq_lens=lens, q_lens=[1] * len(lens), num_heads=8,
                           num_kv_heads=2, head_dim=32, dtype=torch.bfloat16, seed=seed,
                           sliding_window=window, partition_size=512)


def pin_splitkv_matches_full():
    for window in (0, 700):
        w = _split_case(window)
        P, MP = 512, w.max_partitions()
        st, ml, es, to = oracle.splitkv_partials(w.q, w.k_blocks, w.v_blocks, w.seq_lens,
                                                 w.block_tables, w.scale, P, MP, window)
        assert st == oracle.OK
        st, out = oracle.splitkv_reduce(ml, es, to, w.seq_lens, P)
        assert st == oracle.OK
        full, _ = _run(w)
        np.testing.assert_allclose(out.numpy(), full.numpy(), rtol=1e-5, atol=2e-6)
        # unused partitions carry (-inf, 0, 0)
        for s, n in enumerate(w.seq_lens_list):
            for p in range((n + P - 1) // P, MP):
                assert torch.all(ml[s, :, p] == -math.inf) and torch.all(es[s, :, p] == 0)
                assert torch.all(to[s, :, p] == 0)


def pin_splitkv_fp8_scaled():
    # split-KV partials over an fp8 pool with scales (the V2 page: kv_cache_dtype "fp8",
    # k_scale, v_scale) equal, bit for bit, the partials over the fp32 pool holding
    # k_scale * value(code) and v_scale * value(code) (torch's e4m3 decoding, one fp32 product)
    w = _split_case(window=700, seed=35)
    g = torch.Generator().manual_seed(36)
    kb8 = (torch.randn(w.k_blocks.shape, generator=g) * 8).to(torch.float8_e4m3fn)
    vb8 = (torch.randn(w.v_blocks.shape, generator=g) * 8).to(torch.float8_e4m3fn)
    ks, vs = 0.15, 0.11
    P, MP = 512, w.max_partitions()
    a = oracle.splitkv_partials(w.q, kb8, vb8, w.seq_lens, w.block_tables, w.scale, P, MP, 700,
                                k_scale=ks, v_scale=vs)
    b = oracle.splitkv_partials(w.q, kb8.float() * ks, vb8.float() * vs, w.seq_lens,
                                w.block_tables, w.scale, P, MP, 700)
    assert a[0] == oracle.OK and b[0] == oracle.OK
    for x, y in zip(a[1:], b[1:]):
        assert torch.equal(x, y)


def pin_splitkv_single_partition_passthrough():
    w = _split_case()
    st, ml, es, to = oracle.splitkv_partials(w.q, w.k_blocks, w.v_blocks, w.seq_lens,
                                             w.block_tables, w.scale, 512, w.max_partitions())
    st, out = oracle.splitkv_reduce(ml, es, to, w.seq_lens, 512)
    for s, n in enumerate(w.seq_lens_list):
        if n <= 512:
            assert torch.equal(out[s], to[s, :, 0]), s


def pin_splitkv_masked_partition():
    """Masking one partition's (max_logit, exp_sum) to (+/-inf, 0) removes exactly its keys:
    the result is dense attention over the context minus that partition (float64)."""
    w = _split_case()
    P, MP = 512, w.max_partitions()
    st, ml, es, to = oracle.splitkv_partials(w.q, w.k_blocks, w.v_blocks, w.seq_lens,
                                             w.block_tables, w.scale, P, MP)
    s = 5  # 2100 positions -> 5 partitions
    n = w.seq_lens_list[s]
    for masked, sign in ((1, -1.0), (3, 1.0)):
        ml2, es2 = ml.clone(), es.clone()
        ml2[s, :, masked] = sign * math.inf
        es2[s, :, masked] = 0.0
        st, out = oracle.splitkv_reduce(ml2, es2, to, w.seq_lens, P)
        assert st == oracle.OK
        rows = [j for j in range(n) if not (masked * P <= j < (masked + 1) * P)]
        k = torch.stack([w.k_blocks[int(w.block_tables[s, j // 16]), j % 16] for j in rows])
        v = torch.stack([w.v_blocks[int(w.block_tables[s, j // 16]), j % 16] for j in rows])
        want = _dense_attention_f64(w.q[s:s + 1].float().numpy(), k.float().numpy(),
                                    v.float().numpy(), [len(rows) - 1], len(rows), w.scale,
                                    True, 0)
        np.testing.assert_allclose(out[s:s + 1].numpy(), want, rtol=1e-5, atol=2e-6)


def pin_splitkv_all_masked():
    """Every partition masked: the reduction emits partition 0's output unchanged."""
    w = _split_case()
    P, MP = 512, w.max_partitions()
    st, ml, es, to = oracle.splitkv_partials(w.q, w.k_blocks, w.v_blocks, w.seq_lens,
                                             w.block_tables, w.scale, P, MP)
    ml[:] = -math.inf
    ml[:, :, 1::2] = math.inf
    es[:] = 0.0
    st, out = oracle.splitkv_reduce(ml, es, to, w.seq_lens, P)
    assert st == oracle.OK
    assert torch.equal(out, to[:, :, 0])


# --------------------------------------------------------------------------------------------
# merge_attn_states


def pin_merge_identity():
    """Attention over positions [0, n) equals the log-sum-exp merge of attention over
    [0, k) (prefix, no causal mask) and over [k, n) (suffix), and the merged lse is the
    full lse (chunked-context prefill, vllm.cpp cpu_mla_prefill.cpp)."""
    w = workloads.build("merge", seq_lens=[90, 47, 200], q_lens=[1, 1, 1], num_heads=4,
                        num_kv_heads=4, head_dim=32, dtype=torch.float32, seed=41)
    ks = [37, 16, 1]  # prefix lengths
    full, full_lse = _run(w)
    pre = []
    suf = []
    for s, (n, k) in enumerate(zip(w.seq_lens_list, ks)):
        one = dict(query_start_loc=_t([0, 1]), block_tables=w.block_tables[s:s + 1].contiguous(),
                   want_lse=True)
        # prefix: no causal mask over a context of k positions (the query's position only
        # has to lie inside that context)
        st, po, pl = oracle.varlen_attention(w.q[s:s + 1], w.k_blocks, w.v_blocks,
                                             seq_lens=_t([k]), positions=_t([k - 1]),
                                             scale=w.scale, causal=False, **one)
        assert st == oracle.OK
        # suffix: the query at n - 1 with a window of n - k positions sees exactly [k, n)
        st, so, sl = oracle.varlen_attention(w.q[s:s + 1], w.k_blocks, w.v_blocks,
                                             seq_lens=_t([n]), positions=_t([n - 1]),
                                             scale=w.scale, causal=True, sliding_window=n - k,
                                             **one)
        assert st == oracle.OK
        pre.append((po, pl))
        suf.append((so, sl))
    po = torch.cat([p[0] for p in pre])
    pl = torch.cat([p[1] for p in pre], dim=1).contiguous()
    so = torch.cat([p[0] for p in suf])
    sl = torch.cat([p[1] for p in suf], dim=1).contiguous()
    st, out, lse = oracle.merge_attn_states(po, pl, so, sl)
    assert st == oracle.OK
    np.testing.assert_allclose(out.numpy(), full.numpy(), rtol=1e-5, atol=2e-6)
    np.testing.assert_allclose(lse.numpy(), full_lse.numpy(), rtol=1e-6, atol=1e-6)
    # merging a state with itself keeps the output and adds ln 2 to the lse
    st, out2, lse2 = oracle.merge_attn_states(po, pl, po, pl)
    assert torch.equal(out2, po)
    np.testing.assert_allclose(lse2.numpy(), (pl + math.log(2.0)).numpy(), rtol=0, atol=1e-6)


def pin_merge_edge_cases():
    gen = torch.Generator().manual_seed(51)
    T, H, D = 6, 2, 8
    po = torch.randn((T, H, D), generator=gen)
    so = torch.randn((T, H, D), generator=gen)
    inf = math.inf
    pl = torch.tensor([[inf, -inf, -inf, inf, 0.5, 1.0], [0.3, inf, -inf, 2.0, -inf, 1.0]])
    sl = torch.tensor([[0.7, -inf, 1.5, inf, -inf, 2.0], [inf, inf, 0.2, -inf, 0.4, 1.0]])
    st, out, lse = oracle.merge_attn_states(po, pl, so, sl, prefill_tokens_with_context=5)
    assert st == oracle.OK
    for t in range(T):
        for h in range(H):
            p, s = float(pl[h, t]), float(sl[h, t])
            if t >= 5:  # past the with-context prefix: the suffix verbatim
                assert torch.equal(out[t, h], so[t, h]) and float(lse[h, t]) == s
                continue
            p = -inf if math.isinf(p) else p
            s = -inf if math.isinf(s) else s
            if p == -inf and s == -inf:  # both empty: the prefix output, lse -inf
                assert torch.equal(out[t, h], po[t, h]) and float(lse[h, t]) == -inf, (t, h)
            elif p == -inf:  # only the suffix has mass: it passes through exactly
                assert torch.equal(out[t, h], so[t, h]) and float(lse[h, t]) == s, (t, h)
            elif s == -inf:
                assert torch.equal(out[t, h], po[t, h]) and float(lse[h, t]) == p, (t, h)
            else:
                m = max(p, s)
                wp, ws = math.exp(p - m), math.exp(s - m)
                want = (po[t, h].double() * wp + so[t, h].double() * ws) / (wp + ws)
                np.testing.assert_allclose(out[t, h].numpy(), want.numpy(), rtol=1e-6, atol=1e-6)
                assert abs(float(lse[h, t]) - (m + math.log(wp + ws))) < 1e-6


# --------------------------------------------------------------------------------------------
# scatter / gather / slot mapping


def pin_scatter_gather_roundtrip():
    """Writing every position of a full prefill through slot mapping + scatter and reading
    it back through gather returns the written rows bit for bit."""
    for dtype in (torch.bfloat16, torch.float32):
        w = workloads.build("sg", seq_lens=[3, 16, 17, 50], q_lens=[3, 16, 17, 50], num_heads=4,
                            num_kv_heads=2, head_dim=8, dtype=dtype, seed=61, extra_table_cols=1)
        st, slots = oracle.slot_mapping(w.query_start_loc, w.positions, w.block_tables,
                                        w.block_size, w.num_blocks)
        assert st == oracle.OK and len(set(slots.tolist())) == w.num_tokens
        kb, vb = w.k_blocks.clone(), w.v_blocks.clone()
        assert oracle.reshape_and_cache(w.k_new, w.v_new, kb, vb, slots, 16) == oracle.OK
        st, ko, vo = oracle.gather_kv(kb, vb, w.query_start_loc, w.block_tables)
        assert st == oracle.OK
        assert torch.equal(ko, w.k_new) and torch.equal(vo, w.v_new)
        # the rest of the pool is untouched
        touched = torch.zeros(w.num_blocks * 16, dtype=torch.bool)
        touched[slots.long()] = True
        flat_k = kb.view(-1, *kb.shape[2:])
        assert torch.equal(flat_k[~touched], w.k_blocks.view(-1, *kb.shape[2:])[~touched])
        # gather with per-sequence start offsets (a context chunk)
        starts = _t([1, 0, 16, 20])
        cu = _t([0, 2, 18, 19, 49])
        st, ko2, _ = oracle.gather_kv(kb, None, cu, w.block_tables, seq_starts=starts)
        assert st == oracle.OK
        qsl = w.query_start_loc.tolist()
        for s in range(4):
            a, n = int(cu[s]), int(cu[s + 1] - cu[s])
            src = qsl[s] + int(starts[s])
            assert torch.equal(ko2[a:a + n], w.k_new[src:src + n]), s


def pin_scatter_gather_validation():
    w = workloads.build("sgv", seq_lens=[20], q_lens=[20], num_heads=2, num_kv_heads=1,
                        head_dim=8, dtype=torch.float32, seed=62)
    kb, vb = w.k_blocks.clone(), w.v_blocks.clone()
    bad = torch.arange(20, dtype=torch.int32)
    bad[7] = w.num_blocks * 16  # one slot past the pool
    assert oracle.reshape_and_cache(w.k_new, w.v_new, kb, vb, bad, 16) == oracle.EINVAL
    assert torch.equal(kb, w.k_blocks) and torch.equal(vb, w.v_blocks)
    st, _, _ = oracle.gather_kv(kb, vb, _t([0, 40]), w.block_tables)  # past the table row
    assert st == oracle.EINVAL


# --------------------------------------------------------------------------------------------
# validation (tinyllm bad_tables_and_shapes)


def pin_validation():
    D, b = 8, 16
    kb = torch.randn((16, b, 1, D))  # 16 physical blocks; some cases declare fewer
    vb = torch.randn((16, b, 1, D))
    q = torch.randn((2, 2, D))

    def call(seq_lens, positions, tables, H=2, Hkv=1, nb=None):
        out = torch.full((2, H, D), 7.25)
        st, out, _ = oracle.varlen_attention(
            q[:, :H].contiguous(), kb[:nb] if nb else kb, vb[:nb] if nb else vb, _t([0, 1, 2]),
            _t(seq_lens), _t(positions), _t(tables), scale=0.5, num_kv_heads=Hkv, out=out)
        return st, out

    st, out = call([5, 30], [4, 29], [[2, 0], [3, 4]])
    assert st == oracle.OK
    cases = [
        ("empty context", dict(seq_lens=[0, 30], positions=[0, 29], tables=[[2, 0], [3, 4]]),
         oracle.EINVAL),
        ("table too short", dict(seq_lens=[40, 30], positions=[39, 29], tables=[[2, 0], [3, 4]]),
         oracle.EINVAL),
        ("block id past the pool", dict(seq_lens=[5, 30], positions=[4, 29],
                                         tables=[[9, 0], [3, 1]], nb=4), oracle.EINVAL),
        ("position past the context", dict(seq_lens=[5, 30], positions=[5, 29],
                                            tables=[[2, 0], [3, 4]]), oracle.EINVAL),
        ("heads not a multiple of kv heads", dict(seq_lens=[5, 30], positions=[4, 29],
                                                   tables=[[2, 0], [3, 4]], H=2, Hkv=3),
         oracle.ESHAPE),
    ]
    for name, kw, want in cases:
        st, out = call(**kw)
        assert st == want, (name, st)
        assert torch.all(out == 7.25), name  # out untouched on error


# --------------------------------------------------------------------------------------------
# bfloat16 rounding


def pin_bf16_codec():
    vals = [0.0, -0.0, 1.0, -1.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -8 + 2.0 ** -20,
            3.0e38, 3.4e38, -3.4e38, 1e-40, -1e-41, 2.0 ** -133, math.inf, -math.inf, 0.1, 1.0 / 3,
            65504.0, 123456.789, -7.77e-20]
    gen = torch.Generator().manual_seed(71)
    vals += (torch.randn(2000, generator=gen) * 10.0 ** torch.randint(-30, 30, (2000,),
                                                                        generator=gen)).tolist()
    x = torch.tensor(vals, dtype=torch.float32)
    want = x.to(torch.bfloat16).view(torch.int16).to(torch.int32) & 0xFFFF
    got = torch.tensor([oracle.f32_to_bf16(float(v)) for v in x], dtype=torch.int32)
    assert torch.equal(got, want)
    assert oracle.f32_to_bf16(float("nan")) & 0x7F80 == 0x7F80
    for bits in (0x3F80, 0xBF80, 0x0001, 0x7F7F, 0x7F80, 0x8000, 0x4049):
        got = oracle.bf16_to_f32(bits)
        ref = torch.tensor([bits], dtype=torch.int32).to(torch.int16).view(torch.bfloat16).float()
        assert got == float(ref), hex(bits)


# --------------------------------------------------------------------------------------------
# one dequantisation scale per kv head (tinyllm "Going further": fp8 KV caches with scales per
# head or per block)


def pin_per_head_scatter():
    # head g of every new row holds x / k_scales[g]: torch's e4m3 code of the IEEE quotient
    # (clamped to +-448) in an fp8 pool, the quotient itself in an fp32 pool
    g = torch.Generator().manual_seed(75)
    T, Hkv, D, b, NB = 20, 3, 16, 16, 4
    k = (torch.randn((T, Hkv, D), generator=g) * 3).to(torch.bfloat16)
    v = (torch.randn((T, Hkv, D), generator=g) * 50).to(torch.bfloat16)
    ks = torch.tensor([0.0625, 0.5, 2.0])
    vs = torch.tensor([0.37, 0.11, 1.3])
    slots = torch.randperm(NB * b, generator=g)[:T].to(torch.int32)
    for dt in (torch.float8_e4m3fn, torch.float32):
        kb = torch.zeros((NB, b, Hkv, D), dtype=dt)
        vb = torch.zeros_like(kb)
        assert oracle.reshape_and_cache_per_head(k, v, kb, vb, slots, b, ks, vs) == oracle.OK
        for t in range(T):
            sl = int(slots[t])
            wk, wv = k[t].float() / ks[:, None], v[t].float() / vs[:, None]
            if dt == torch.float8_e4m3fn:
                wk = torch.clamp(wk, -448, 448).to(dt).view(torch.uint8)
                wv = torch.clamp(wv, -448, 448).to(dt).view(torch.uint8)
                gk, gv = kb[sl // b, sl % b].view(torch.uint8), vb[sl // b, sl % b].view(torch.uint8)
            else:
                gk, gv = kb[sl // b, sl % b], vb[sl // b, sl % b]
            assert torch.equal(gk, wk) and torch.equal(gv, wv)
    # a scale that is not finite and positive: EINVAL, nothing written
    for bad in (0.0, -1.0, float("inf"), float("nan")):
        ks2 = ks.clone()
        ks2[1] = bad
        kb = torch.zeros((NB, b, Hkv, D), dtype=torch.float32)
        vb = torch.zeros_like(kb)
        assert oracle.reshape_and_cache_per_head(k, v, kb, vb, slots, b, ks2, vs) == oracle.EINVAL
        assert not kb.any() and not vb.any()


def pin_per_head_attention():
    # per kv head scales on an fp8 pool equal, bit for bit, the unscaled attention over the fp32
    # pool holding k_scales[g] * value(code) (torch's e4m3 decoding, one fp32 product), with
    # GQA 3 so that query head h reads kv head h // 3; the same for the split-KV partials
    H, Hkv, D, lens, qsl, pos, q, kb8, vb8, table = _fp8_case(seed=76)
    ks, vs = torch.tensor([0.25, 0.6]), torch.tensor([0.37, 1.7])
    kbf = kb8.float() * ks.view(1, 1, Hkv, 1)
    vbf = vb8.float() * vs.view(1, 1, Hkv, 1)
    meta = dict(query_start_loc=_t(qsl), seq_lens=_t(lens), positions=_t(pos),
                block_tables=table, scale=1.0 / math.sqrt(D), want_lse=True)
    for window in (0, 20):
        st, o1, l1 = oracle.varlen_attention(q, kb8, vb8, sliding_window=window, k_scales=ks,
                                             v_scales=vs, **meta)
        st2, o2, l2 = oracle.varlen_attention(q, kbf, vbf, sliding_window=window, **meta)
        assert st == oracle.OK and st2 == oracle.OK
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
    # one decode query per sequence for the partials
    qd = torch.stack([q[qsl[s + 1] - 1] for s in range(len(lens))])
    # (float64 scales: the wrapper's fp32 copies must outlive the call)
    a = oracle.splitkv_partials(qd, kb8, vb8, _t(lens), table, 1.0 / math.sqrt(D), 16, 8,
                                k_scales=ks.double(), v_scales=vs.double())
    b = oracle.splitkv_partials(qd, kbf, vbf, _t(lens), table, 1.0 / math.sqrt(D), 16, 8)
    assert a[0] == oracle.OK and b[0] == oracle.OK
    for x, y in zip(a[1:], b[1:]):
        assert torch.equal(x, y)
    # an invalid scale is EINVAL
    for bad in (0.0, float("nan")):
        ks2 = ks.clone()
        ks2[0] = bad
        st, _, _ = oracle.varlen_attention(q, kb8, vb8, k_scales=ks2, v_scales=vs, **meta)
        assert st == oracle.EINVAL


def _block_scales(NB, Hkv, seed, lo=0.2, hi=2.0):
    g = torch.Generator().manual_seed(seed)
    return lo + (hi - lo) * torch.rand((NB, Hkv), generator=g)


def pin_per_block_scatter():
    # head g of a new row written to slot s holds x / scales[s // b, g]: torch's e4m3 code of
    # the IEEE quotient (clamped to +-448) in an fp8 pool, the quotient itself in an fp32 pool
    g = torch.Generator().manual_seed(77)
    T, Hkv, D, b, NB = 20, 3, 16, 16, 4
    k = (torch.randn((T, Hkv, D), generator=g) * 3).to(torch.bfloat16)
    v = (torch.randn((T, Hkv, D), generator=g) * 50).to(torch.bfloat16)
    ks, vs = _block_scales(NB, Hkv, 78, 0.05, 2.0), _block_scales(NB, Hkv, 79, 0.1, 1.5)
    slots = torch.randperm(NB * b, generator=g)[:T].to(torch.int32)
    for dt in (torch.float8_e4m3fn, torch.float32):
        kb = torch.zeros((NB, b, Hkv, D), dtype=dt)
        vb = torch.zeros_like(kb)
        assert oracle.reshape_and_cache_per_block(k, v, kb, vb, slots, b, ks, vs) == oracle.OK
        for t in range(T):
            sl = int(slots[t])
            wk = k[t].float() / ks[sl // b][:, None]
            wv = v[t].float() / vs[sl // b][:, None]
            if dt == torch.float8_e4m3fn:
                wk = torch.clamp(wk, -448, 448).to(dt).view(torch.uint8)
                wv = torch.clamp(wv, -448, 448).to(dt).view(torch.uint8)
                gk, gv = kb[sl // b, sl % b].view(torch.uint8), vb[sl // b, sl % b].view(torch.uint8)
            else:
                gk, gv = kb[sl // b, sl % b], vb[sl // b, sl % b]
            assert torch.equal(gk, wk) and torch.equal(gv, wv)
    # a bad factor of a block that is written to: EINVAL, nothing written; of a block no token
    # writes to: ignored
    written = {int(x) // b for x in slots}
    unwritten = [i for i in range(NB) if i not in written]
    for bad in (0.0, -1.0, float("inf"), float("nan"), 1e-39):
        ks2 = ks.clone()
        ks2[int(slots[0]) // b, 1] = bad
        kb = torch.zeros((NB, b, Hkv, D), dtype=torch.float32)
        vb = torch.zeros_like(kb)
        assert oracle.reshape_and_cache_per_block(k, v, kb, vb, slots, b, ks2, vs) == oracle.EINVAL
        assert not kb.any() and not vb.any()
        if unwritten:
            ks3 = ks.clone()
            ks3[unwritten[0], 0] = bad
            assert oracle.reshape_and_cache_per_block(k, v, kb, vb, slots, b, ks3, vs) == oracle.OK


def pin_per_block_attention():
    # per (pool block, kv head) scales on an fp8 pool equal, bit for bit, the unscaled attention
    # over the fp32 pool holding scales[block, g] * value(code) (one fp32 product), where block
    # is the physical id the table names (the tables are permutations of the pool); GQA 3; the
    # same for the split-KV partials
    H, Hkv, D, lens, qsl, pos, q, kb8, vb8, table = _fp8_case(seed=80)
    NB = kb8.shape[0]
    ks, vs = _block_scales(NB, Hkv, 81), _block_scales(NB, Hkv, 82)
    kbf = kb8.float() * ks.view(NB, 1, Hkv, 1)
    vbf = vb8.float() * vs.view(NB, 1, Hkv, 1)
    meta = dict(query_start_loc=_t(qsl), seq_lens=_t(lens), positions=_t(pos),
                block_tables=table, scale=1.0 / math.sqrt(D), want_lse=True)
    for window in (0, 20):
        st, o1, l1 = oracle.varlen_attention(q, kb8, vb8, sliding_window=window,
                                             k_block_scales=ks, v_block_scales=vs, **meta)
        st2, o2, l2 = oracle.varlen_attention(q, kbf, vbf, sliding_window=window, **meta)
        assert st == oracle.OK and st2 == oracle.OK
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
    qd = torch.stack([q[qsl[s + 1] - 1] for s in range(len(lens))])
    a = oracle.splitkv_partials(qd, kb8, vb8, _t(lens), table, 1.0 / math.sqrt(D), 16, 8,
                                k_block_scales=ks, v_block_scales=vs)
    b = oracle.splitkv_partials(qd, kbf, vbf, _t(lens), table, 1.0 / math.sqrt(D), 16, 8)
    assert a[0] == oracle.OK and b[0] == oracle.OK
    for x, y in zip(a[1:], b[1:]):
        assert torch.equal(x, y)
    # a bad factor of a block some sequence reads: EINVAL; of a block no table names: ignored
    used = {int(table[s, j]) for s, n in enumerate(lens) for j in range((n + 15) // 16)}
    unused = [i for i in range(NB) if i not in used]
    for bad in (0.0, float("nan"), 1e-39):
        vs2 = vs.clone()
        vs2[int(table[1, 0]), 1] = bad
        st, _, _ = oracle.varlen_attention(q, kb8, vb8, k_block_scales=ks, v_block_scales=vs2,
                                           **meta)
        assert st == oracle.EINVAL
        if unused:
            vs3 = vs.clone()
            vs3[unused[0], 0] = bad
            st, _, _ = oracle.varlen_attention(q, kb8, vb8, k_block_scales=ks,
                                               v_block_scales=vs3, **meta)
            assert st == oracle.OK


ALL_PINS = {
    "per_block_scatter": pin_per_block_scatter,
    "per_block_attention": pin_per_block_attention,
    "per_head_scatter": pin_per_head_scatter,
    "per_head_attention": pin_per_head_attention,
    "fp8_codec": pin_fp8_codec,
    "fp8_scatter": pin_fp8_scatter,
    "fp8_attention_brute_force": pin_fp8_attention_brute_force,
    "dequant_scales": pin_dequant_scales,
    "sinks_closed_forms": pin_sinks_closed_forms,
    "sinks_brute_force": pin_sinks_brute_force,
    "hand_example": pin_hand_example,
    "hand_example_via_cache": pin_hand_example_via_cache,
    "brute_force": pin_brute_force_all,
    "closed_forms": pin_closed_forms,
    "block_permutation": pin_block_permutation_invariance,
    "batch_and_shared_prefix": pin_batch_invariance_and_shared_prefix,
    "threads": pin_thread_invariance,
    "splitkv_matches_full": pin_splitkv_matches_full,
    "splitkv_fp8_scaled": pin_splitkv_fp8_scaled,
    "splitkv_single_partition": pin_splitkv_single_partition_passthrough,
    "splitkv_masked_partition": pin_splitkv_masked_partition,
    "splitkv_all_masked": pin_splitkv_all_masked,
    "merge_identity": pin_merge_identity,
    "merge_edge_cases": pin_merge_edge_cases,
    "scatter_gather_roundtrip": pin_scatter_gather_roundtrip,
    "scatter_gather_validation": pin_scatter_gather_validation,
    "validation": pin_validation,
    "bf16_codec": pin_bf16_codec,
}
