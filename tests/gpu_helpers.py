"""Shared helpers of the GPU parity tests: running the CPU oracle on a workload (or on a
subset of its sequences) and the attention tolerance of the comparisons."""
from __future__ import annotations

import torch

import oracle

# Attention outputs: |gpu - oracle| <= ATOL + RTOL * |oracle| elementwise (bf16 K/V, fp32
# accumulation on both sides, the oracle in fp32 on the same bf16 values).
ATOL = 2e-3
RTOL = 1e-2


def assert_attn_close(got, ref, what=""):
    got = got.detach().float().cpu()
    ref = ref.detach().float().cpu()
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert torch.isfinite(got).all(), f"{what}: non-finite GPU output"
    err = (got - ref).abs()
    bad = err > ATOL + RTOL * ref.abs()
    if bad.any():
        i = int(bad.flatten().nonzero()[0])
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {got.numel()} outside tolerance; max abs err "
            f"{float(err.max()):.3e}; first at flat {i}: gpu {float(got.flatten()[i]):.6f} "
            f"oracle {float(ref.flatten()[i]):.6f}")
    return float(err.max())


def assert_attn_close_scaled(got, ref, ref_abs, what=""):
    """assert_attn_close with the absolute part scaled to the size of the values each output row
    averages: ref_abs is the oracle's output over |V|, and a row's scale is its mean over the
    head dimension (about 0.8 for N(0, 1) values, where the fixed ATOL applies).  The bound
    then holds at any scale of V, and for rows that average values of very different sizes,
    where an output near 0 comes from the cancellation of large terms."""
    got = got.detach().float().cpu()
    ref = ref.detach().float().cpu()
    ref_abs = ref_abs.detach().float().cpu()
    assert got.shape == ref.shape == ref_abs.shape, (what, got.shape, ref.shape)
    assert torch.isfinite(got).all(), f"{what}: non-finite GPU output"
    scale = ref_abs.mean(dim=-1, keepdim=True).expand_as(ref)
    err = (got - ref).abs()
    bad = err > ATOL * scale + RTOL * ref.abs()
    if bad.any():
        i = int(bad.flatten().nonzero()[0])
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {got.numel()} outside tolerance; max err / scale "
            f"{float((err / scale.clamp_min(1e-30)).max()):.3e}; first at flat {i}: gpu "
            f"{float(got.flatten()[i]):.6g} oracle {float(ref.flatten()[i]):.6g} row scale "
            f"{float(scale.flatten()[i]):.6g}")
    return float(err.max())


def sub_batch(w, seqs):
    """Metadata of the sequences `seqs` of workload w as a batch of their own (same pool)."""
    qsl = w.query_start_loc.cpu().tolist()
    rows, new_qsl = [], [0]
    for s in seqs:
        rows.extend(range(qsl[s], qsl[s + 1]))
        new_qsl.append(new_qsl[-1] + qsl[s + 1] - qsl[s])
    idx = torch.tensor(rows, dtype=torch.long)
    sel = torch.tensor(seqs, dtype=torch.long)
    return dict(rows=idx, query_start_loc=torch.tensor(new_qsl, dtype=torch.int32),
                seq_lens=w.seq_lens.cpu()[sel].contiguous(),
                positions=w.positions.cpu()[idx].contiguous(),
                block_tables=w.block_tables.cpu()[sel].contiguous())


def oracle_attention(w, kb_cpu, vb_cpu, seqs=None, q=None):
    """Oracle output (fp32) for all sequences of w, or for `seqs` only (rows in order)."""
    q = (w.q if q is None else q).cpu()
    if seqs is None:
        st, out, _ = oracle.varlen_attention(q, kb_cpu, vb_cpu, w.query_start_loc, w.seq_lens,
                                             w.positions, w.block_tables, w.scale,
                                             causal=w.causal, sliding_window=w.sliding_window)
        assert st == oracle.OK, st
        return out
    sb = sub_batch(w, seqs)
    st, out, _ = oracle.varlen_attention(q[sb["rows"]].contiguous(), kb_cpu, vb_cpu,
                                         sb["query_start_loc"], sb["seq_lens"], sb["positions"],
                                         sb["block_tables"], w.scale, causal=w.causal,
                                         sliding_window=w.sliding_window)
    assert st == oracle.OK, st
    return out
