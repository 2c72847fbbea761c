"""Stream order of consecutive calls.

The varlen planner reads a call's metadata and plans before the kernels ahead of it on the
stream have finished, and the scatter of pa_cache_and_attend runs beside it: both must still
write nothing before the previous call's kernels are done.  A serving loop reuses freed
blocks, so the next step's scatter may write into a block the previous step's attention is
still reading.  Here call 1 (the 64-sequence decode batch) reads block X as the last block of
its shortest sequence, which the persistent kernel takes last; call 2, issued right behind it
on the same stream, scatters a new token into row r of block X, a row call 1 attends to.
Call 1's output must equal, bit for bit, the same call run alone on the untouched pool.
"""
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


def test_next_scatter_waits_for_previous_attention(pa):
    w = workloads.named(2, device=DEV, seed=3)
    kb0, vb0 = w.k_blocks.clone(), w.v_blocks.clone()
    ws1 = pa.workspace_for(w.q, w.k_blocks, w.query_start_loc, w.block_tables)
    out1 = torch.empty_like(w.q)

    def call1():
        pa.pa_varlen_forward(w.q, w.k_blocks, w.v_blocks, out1, w.query_start_loc, w.seq_lens,
                             w.positions, w.block_tables, w.scale, workspace=ws1)

    call1()
    torch.cuda.synchronize()
    ref = out1.clone()

    # the shortest sequence (taken last): its last block X, the row of its last position
    a = int(torch.argmin(w.seq_lens).item())
    n_a = int(w.seq_lens[a].item())
    x = int(w.block_tables[a, (n_a - 1) // w.block_size].item())
    r = (n_a - 1) % w.block_size
    # call 2: one sequence whose new token lands in row r of block X
    g = torch.Generator(device=DEV).manual_seed(11)
    H, Hkv, D = w.num_heads, w.num_kv_heads, w.head_dim
    q2 = torch.randn((1, H, D), generator=g, device=DEV).to(torch.bfloat16)
    k2 = torch.randn((1, Hkv, D), generator=g, device=DEV).to(torch.bfloat16)
    v2 = torch.randn((1, Hkv, D), generator=g, device=DEV).to(torch.bfloat16)
    qsl2 = torch.tensor([0, 1], dtype=torch.int32, device=DEV)
    sl2 = torch.tensor([r + 1], dtype=torch.int32, device=DEV)
    pos2 = torch.tensor([r], dtype=torch.int32, device=DEV)
    bt2 = torch.tensor([[x]], dtype=torch.int32, device=DEV)
    ws2 = pa.workspace_for(q2, w.k_blocks, qsl2, bt2)
    out2 = torch.empty_like(q2)

    for _ in range(8):
        w.k_blocks.copy_(kb0)
        w.v_blocks.copy_(vb0)
        out1.zero_()
        torch.cuda.synchronize()
        call1()
        pa.pa_cache_and_attend(k2, v2, q2, w.k_blocks, w.v_blocks, out2, qsl2, sl2, pos2, bt2,
                               w.scale, workspace=ws2)
        torch.cuda.synchronize()
        assert pa.pa_device_status() == pa.PA_OK
        assert torch.equal(w.k_blocks[x, r], k2[0]) and torch.equal(w.v_blocks[x, r], v2[0])
        assert torch.equal(out1, ref), "call 1 read a row that call 2 wrote after it"
