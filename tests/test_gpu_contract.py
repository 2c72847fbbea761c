"""GPU contract tests: validation before any write (tinyllm bad_tables_and_shapes), the
sticky device status word, bitwise determinism, batch invariance, shared prefix blocks, and
invariance to the physical block ids (tinyllm sections 2.5 and 4)."""
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


def _fwd(pa, w, q=None, kb=None, vb=None, tables=None, seq_lens=None, positions=None, out=None):
    q = w.q if q is None else q
    out = torch.full_like(q, 7.25) if out is None else out
    pa.pa_varlen_forward(q, w.k_blocks if kb is None else kb, w.v_blocks if vb is None else vb,
                         out, w.query_start_loc, w.seq_lens if seq_lens is None else seq_lens,
                         w.positions if positions is None else positions,
                         w.block_tables if tables is None else tables, w.scale, causal=w.causal,
                         sliding_window=w.sliding_window)
    return out


@pytest.mark.parametrize("case", ["block id past the pool", "negative block id", "empty context",
                                  "table too short", "position past the context",
                                  "decreasing query_start_loc"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_bad_metadata_writes_nothing(pa, case, dtype):
    w = workloads.build("bad", seq_lens=[20, 70, 5], q_lens=[1, 3, 1], num_heads=8,
                        num_kv_heads=2, head_dim=128, dtype=dtype, seed=17, device=DEV)
    tables, seq_lens, positions = w.block_tables.clone(), w.seq_lens.clone(), w.positions.clone()
    qsl = w.query_start_loc.clone()
    if case == "block id past the pool":
        tables[1, 3] = w.num_blocks + 5
    elif case == "negative block id":
        tables[0, 1] = -1
    elif case == "empty context":
        seq_lens[2] = 0
        positions[-1] = 0
    elif case == "table too short":
        seq_lens[1] = 16 * w.max_blocks_per_seq + 1
    elif case == "position past the context":
        positions[1] = 70
    elif case == "decreasing query_start_loc":
        qsl[2] = 0
    out = torch.full_like(w.q, 7.25)
    pa.pa_varlen_forward(w.q, w.k_blocks, w.v_blocks, out, qsl, seq_lens, positions, tables,
                         w.scale)
    assert pa.pa_device_status() == pa.PA_EINVAL
    assert torch.all(out == 7.25), "out written despite invalid metadata"
    # cleared: the same call with good metadata works again
    _fwd(pa, w, out=out)
    assert pa.pa_device_status() == pa.PA_OK
    assert not torch.all(out == 7.25)


def test_error_is_sticky_until_read(pa):
    w = workloads.build("sticky", seq_lens=[40], q_lens=[1], num_heads=4, num_kv_heads=2,
                        head_dim=128, seed=18, device=DEV)
    bad = w.block_tables.clone()
    bad[0, 0] = 10 ** 6
    _fwd(pa, w, tables=bad)
    out = _fwd(pa, w)  # valid, but the recorded error is still there
    torch.cuda.synchronize()
    assert torch.all(out == 7.25)
    assert pa.pa_device_status() == pa.PA_EINVAL
    assert pa.pa_device_status() == pa.PA_OK


def test_bad_slot_writes_nothing(pa):
    w = workloads.build("slot", seq_lens=[40, 9], q_lens=[40, 9], num_heads=4, num_kv_heads=2,
                        head_dim=128, seed=19, device=DEV)
    slots = pa.pa_slot_mapping(w.query_start_loc, w.positions, w.block_tables, 16, w.num_blocks)
    assert pa.pa_device_status() == pa.PA_OK
    slots[17] = w.num_blocks * 16  # one past the pool
    kb, vb = w.k_blocks.clone(), w.v_blocks.clone()
    pa.pa_reshape_and_cache(w.k_new, w.v_new, kb, vb, slots)
    assert pa.pa_device_status() == pa.PA_EINVAL
    assert torch.equal(kb, w.k_blocks) and torch.equal(vb, w.v_blocks)


def test_slot_mapping_flags_positions_outside_the_table(pa):
    w = workloads.build("slot2", seq_lens=[40], q_lens=[2], num_heads=4, num_kv_heads=2,
                        head_dim=128, seed=20, device=DEV)
    pos = w.positions.clone()
    pos[1] = 16 * w.max_blocks_per_seq  # past the table row
    slots = pa.pa_slot_mapping(w.query_start_loc, pos, w.block_tables, 16, w.num_blocks)
    assert pa.pa_device_status() == pa.PA_EINVAL
    assert int(slots[1]) == -1


def test_splitkv_rejects_too_few_partitions(pa):
    w = workloads.named(4, small=True, device=DEV)
    S, H, D = w.num_seqs, w.num_heads, w.head_dim
    P = w.max_partitions() - 1  # one partition short
    ml = torch.full((S, H, P), 5.0, device=DEV)
    es = torch.full((S, H, P), 5.0, device=DEV)
    to = torch.full((S, H, P, D), 5.0, device=DEV)
    pa.pa_decode_splitkv_partials(w.q, w.k_blocks, w.v_blocks, ml, es, to, w.seq_lens,
                                  w.block_tables, w.scale, w.partition_size)
    assert pa.pa_device_status() == pa.PA_EINVAL
    assert torch.all(ml == 5.0) and torch.all(to == 5.0)


@pytest.mark.parametrize("cfg", [2, 3])
def test_bitwise_deterministic(pa, cfg):
    w = workloads.named(cfg, small=True, device=DEV)
    outs = [_fwd(pa, w) for _ in range(3)]
    assert pa.pa_device_status() == pa.PA_OK
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])


def test_alone_vs_batch_of_16_and_shared_prefix(pa):
    """16 sequences share two prefix blocks: each gives the same bits alone and in the batch,
    and the same bits as with private copies of the prefix blocks."""
    g = torch.Generator().manual_seed(23)
    lens = [int(x) for x in torch.randint(33, 900, (16,), generator=g)]
    qlens = [1] * 12 + [3, 1, 7, 1]
    w = workloads.build("fork", seq_lens=lens, q_lens=qlens, num_heads=32, num_kv_heads=8,
                        head_dim=128, seed=23, shared_prefix_blocks=2, device=DEV)
    batch = _fwd(pa, w)
    qsl = w.query_start_loc.cpu().tolist()
    for s in range(16):
        a, b = qsl[s], qsl[s + 1]
        one = torch.full_like(w.q[a:b], 7.25)
        pa.pa_varlen_forward(w.q[a:b], w.k_blocks, w.v_blocks, one,
                             torch.tensor([0, b - a], dtype=torch.int32, device=DEV),
                             w.seq_lens[s:s + 1], w.positions[a:b],
                             w.block_tables[s:s + 1].contiguous(), w.scale)
        assert torch.equal(one, batch[a:b]), f"sequence {s} differs alone vs in the batch"
    NB = w.num_blocks
    prefix = w.block_tables[0, :2].long()
    kb = torch.cat([w.k_blocks] + [w.k_blocks[prefix]] * 16)
    vb = torch.cat([w.v_blocks] + [w.v_blocks[prefix]] * 16)
    bt = w.block_tables.clone()
    for s in range(16):
        bt[s, 0], bt[s, 1] = NB + 2 * s, NB + 2 * s + 1
    private = _fwd(pa, w, kb=kb, vb=vb, tables=bt)
    assert pa.pa_device_status() == pa.PA_OK
    assert torch.equal(private, batch)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_block_permutation_invariance(pa, dtype):
    w = workloads.build("perm", seq_lens=[5, 33, 64, 900, 300], q_lens=[1, 4, 64, 1, 20],
                        num_heads=16, num_kv_heads=4, head_dim=128, dtype=dtype, seed=29,
                        sliding_window=200, device=DEV)
    out0 = _fwd(pa, w)
    perm = torch.randperm(w.num_blocks, generator=torch.Generator().manual_seed(31)).to(DEV)
    kb = torch.empty_like(w.k_blocks)
    vb = torch.empty_like(w.v_blocks)
    kb[perm] = w.k_blocks
    vb[perm] = w.v_blocks
    out1 = _fwd(pa, w, kb=kb, vb=vb, tables=perm[w.block_tables.long()].to(torch.int32))
    assert pa.pa_device_status() == pa.PA_OK
    assert torch.equal(out0, out1)
