"""GPU parity of pa_varlen_forward_ex: per-head attention sinks (TensorSharp ForwardWithSinks:
a virtual position with the sink logit as its score and a zero value) and the log-sum-exp
output, on every kernel of the varlen path (decode tiles on the warp-MMA kernel, prefill
chunks on the tcgen05 kernel, fp32 batches on the SIMT kernel), against the oracle."""
import math

import pytest
import torch

import oracle
from paged_kv_cache_31_gb300 import workloads
from tests.gpu_helpers import assert_attn_close

pytestmark = pytest.mark.gpu
DEV = "cuda"
LSE_ATOL, LSE_RTOL = 1e-3, 1e-4


@pytest.fixture(scope="module")
def pa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_31_gb300 import binding

    assert binding.pa_device_status() == binding.PA_OK
    return binding


def _sinks(H, seed):
    g = torch.Generator().manual_seed(seed)
    s = torch.randn((H,), generator=g) * 2.0 + 1.0
    s[::5] = -math.inf  # some heads without a sink
    return s


def _gpu(pa, w, sinks=None, want_lse=True):
    out = torch.full_like(w.q, float("nan"))
    lse = None
    if want_lse:
        lse = torch.full((w.num_heads, w.num_tokens), float("nan"), device=DEV)
    pa.pa_varlen_forward(w.q, w.k_blocks, w.v_blocks, out, w.query_start_loc, w.seq_lens,
                         w.positions, w.block_tables, w.scale, causal=w.causal,
                         sliding_window=w.sliding_window,
                         sinks=None if sinks is None else sinks.to(DEV), lse=lse)
    assert pa.pa_device_status() == pa.PA_OK
    return out, lse


def _oracle(w, sinks=None):
    st, out, lse = oracle.varlen_attention(w.q.cpu(), w.k_blocks.cpu(), w.v_blocks.cpu(),
                                           w.query_start_loc, w.seq_lens, w.positions,
                                           w.block_tables, w.scale, causal=w.causal,
                                           sliding_window=w.sliding_window, want_lse=True,
                                           sinks=sinks)
    assert st == oracle.OK
    return out, lse


def _assert_lse_close(got, ref, what):
    got, ref = got.float().cpu(), ref.float().cpu()
    assert torch.equal(torch.isinf(got), torch.isinf(ref)), what
    fin = torch.isfinite(ref)
    err = (got[fin] - ref[fin]).abs()
    bad = err > LSE_ATOL + LSE_RTOL * ref[fin].abs()
    assert not bad.any(), (f"{what}: {int(bad.sum())} lse values off, "
                           f"max err {float(err.max()):.3e}")


CASES = {
    # decode tokens only: the warp-MMA kernel
    "decode": dict(seq_lens=[1, 17, 300, 1000, 4096], q_lens=[1] * 5, num_heads=32,
                   num_kv_heads=8, head_dim=128),
    # prefill chunks (more than 64 rows per kv head): the tcgen05 kernel, plus decode tokens
    "prefill": dict(seq_lens=[512, 700, 1300, 90, 2000], q_lens=[512, 200, 130, 1, 1],
                    num_heads=32, num_kv_heads=8, head_dim=128),
    # a sliding window on both kernels
    "window": dict(seq_lens=[900, 2500, 3000], q_lens=[300, 1, 1], num_heads=16, num_kv_heads=8,
                   head_dim=128, sliding_window=256),
    # fp32: the SIMT kernel
    "fp32": dict(seq_lens=[1, 17, 33, 50], q_lens=[1, 17, 8, 1], num_heads=4, num_kv_heads=2,
                 head_dim=64, dtype=torch.float32),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_sinks_and_lse_match_oracle(pa, case):
    kw = dict(CASES[case])
    w = workloads.build(case, seed=sorted(CASES).index(case) + 11, device=DEV, **kw)
    sinks = _sinks(w.num_heads, 7)
    out, lse = _gpu(pa, w, sinks)
    ref_out, ref_lse = _oracle(w, sinks)
    assert_attn_close(out, ref_out, f"{case} out")
    _assert_lse_close(lse, ref_lse, f"{case} lse")
    # deterministic
    out2, lse2 = _gpu(pa, w, sinks)
    assert torch.equal(out, out2) and torch.equal(lse, lse2), case


@pytest.mark.parametrize("case", sorted(CASES))
def test_lse_without_sinks(pa, case):
    w = workloads.build(case, seed=sorted(CASES).index(case) + 31, device=DEV, **CASES[case])
    out, lse = _gpu(pa, w)
    ref_out, ref_lse = _oracle(w)
    assert_attn_close(out, ref_out, f"{case} out")
    _assert_lse_close(lse, ref_lse, f"{case} lse")
    # the extended call computes exactly what pa_varlen_forward computes
    plain = torch.full_like(w.q, float("nan"))
    pa.pa_varlen_forward(w.q, w.k_blocks, w.v_blocks, plain, w.query_start_loc, w.seq_lens,
                         w.positions, w.block_tables, w.scale, causal=w.causal,
                         sliding_window=w.sliding_window)
    assert torch.equal(out, plain), case


def test_minus_inf_sinks_are_no_sinks(pa):
    w = workloads.build("prefill", seed=5, device=DEV, **CASES["prefill"])
    out0, lse0 = _gpu(pa, w)
    out1, lse1 = _gpu(pa, w, torch.full((w.num_heads,), -math.inf))
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)


def test_huge_sink_drains_the_output(pa):
    # a sink far above every score takes (almost) all the mass: out -> 0, lse -> the sink
    w = workloads.build("prefill", seed=6, device=DEV, **CASES["prefill"])
    sinks = torch.full((w.num_heads,), 60.0)
    out, lse = _gpu(pa, w, sinks)
    assert out.float().abs().max().item() < 1e-6
    assert torch.allclose(lse.cpu(), torch.full_like(lse.cpu(), 60.0), atol=1e-4)


@pytest.mark.parametrize("case", sorted(CASES))
def test_scaled_wide_pools_match_oracle(pa, case):
    # k_scale / v_scale on bf16 and f32 pools (every kernel folds k_scale into the softmax scale
    # and v_scale into the output), with sinks and lse, against the oracle
    kw = dict(CASES[case])
    w = workloads.build(case, seed=sorted(CASES).index(case) + 71, device=DEV, **kw)
    sinks = _sinks(w.num_heads, 9)
    out = torch.full_like(w.q, float("nan"))
    lse = torch.full((w.num_heads, w.num_tokens), float("nan"), device=DEV)
    pa.pa_varlen_forward(w.q, w.k_blocks, w.v_blocks, out, w.query_start_loc, w.seq_lens,
                         w.positions, w.block_tables, w.scale, causal=w.causal,
                         sliding_window=w.sliding_window, sinks=sinks.to(DEV), lse=lse,
                         k_scale=0.7, v_scale=1.9)
    assert pa.pa_device_status() == pa.PA_OK
    st, ref, ref_lse = oracle.varlen_attention(w.q.cpu(), w.k_blocks.cpu(), w.v_blocks.cpu(),
                                               w.query_start_loc, w.seq_lens, w.positions,
                                               w.block_tables, w.scale, causal=w.causal,
                                               sliding_window=w.sliding_window, want_lse=True,
                                               sinks=sinks, k_scale=0.7, v_scale=1.9)
    assert st == oracle.OK
    assert_attn_close(out, ref, f"{case} scaled out")
    _assert_lse_close(lse, ref_lse, f"{case} scaled lse")
