"""Seeded synthetic workloads for batched paged attention.

This module only *draws inputs*: sequence and chunk lengths, query positions,
block tables (a seeded permutation of the pool's block ids, consumed in order),
and N(0, 1) query / key / value data rounded to the compute dtype.  It holds no
attention, indexing or merge arithmetic, so the CUDA library and the CPU oracle
can both be fed from it without sharing any of the method.

The five named workloads follow the benchmark statement of the batched
paged-attention pages (TensorSharp ManagedPagedAttention layouts; tinyllm
"Paged attention for decode in C" tables and windows; the PagedAttention-V2
partitioning).  ``small=True`` variants keep the same structure (mix, GQA ratio,
head size, block size, window, masked partition, shared prefix) at sizes a CPU
reference finishes in seconds.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import torch

__all__ = ["Workload", "build", "named", "subset", "fp8_pools", "NAMES"]


@dataclasses.dataclass
class Workload:
    name: str
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    max_blocks_per_seq: int
    dtype: torch.dtype
    scale: float
    causal: bool
    sliding_window: int
    seq_lens_list: List[int]
    q_lens_list: List[int]
    query_start_loc: torch.Tensor  # int32 [S+1]
    seq_lens: torch.Tensor  # int32 [S]
    positions: torch.Tensor  # int32 [T]
    block_tables: torch.Tensor  # int32 [S, max_blocks_per_seq]
    q: torch.Tensor  # [T, H, D]
    k_new: torch.Tensor  # [T, Hkv, D]  the new tokens' keys (to be scattered)
    v_new: torch.Tensor  # [T, Hkv, D]
    k_blocks: torch.Tensor  # [NB, b, Hkv, D]  pool, prior context already present
    v_blocks: torch.Tensor
    partition_size: int = 0
    masked_partition: Optional[List[int]] = None  # split-KV: one masked partition per sequence
    shared_prefix_blocks: int = 0
    seed: int = 0

    @property
    def num_seqs(self) -> int:
        return len(self.seq_lens_list)

    @property
    def num_tokens(self) -> int:
        return int(sum(self.q_lens_list))

    @property
    def group(self) -> int:
        return self.num_heads // self.num_kv_heads

    def max_partitions(self) -> int:
        p = self.partition_size
        return max(1, max((n + p - 1) // p for n in self.seq_lens_list)) if p else 0

    def to(self, device) -> "Workload":
        fields = {}
        for f in dataclasses.fields(self):
            v = getattr(self, f.name)
            fields[f.name] = v.to(device) if isinstance(v, torch.Tensor) else v
        return Workload(**fields)


def _randn(shape, gen, device, dtype):
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    return x.to(dtype)


def build(name: str, seq_lens: List[int], q_lens: List[int], num_heads: int, num_kv_heads: int,
          head_dim: int, block_size: int = 16, dtype: torch.dtype = torch.bfloat16,
          causal: bool = True, sliding_window: int = 0, seed: int = 0, device="cpu",
          shared_prefix_blocks: int = 0, num_blocks: Optional[int] = None,
          scale: Optional[float] = None, partition_size: int = 0,
          masked_partition: Optional[List[int]] = None,
          positions: Optional[List[List[int]]] = None,
          extra_table_cols: int = 0) -> Workload:
    """Draw one batch.

    Sequence s holds ``seq_lens[s]`` cached positions (its new tokens included);
    its ``q_lens[s]`` new tokens sit at the last positions
    ``seq_len - q_len .. seq_len - 1`` unless ``positions`` gives them.  Block ids
    come from ``torch.randperm(num_blocks)`` on a CPU generator seeded with
    ``seed``: the first ``shared_prefix_blocks`` ids are common to every
    sequence's table, the rest are handed out in order.  ``num_blocks`` defaults
    to the blocks in use rounded up to a multiple of 16.  Unused table entries are
    0.  q, the new K/V rows and the whole pool are i.i.d. N(0, 1) drawn in fp32
    from a generator on ``device`` and rounded to ``dtype``."""
    assert len(seq_lens) == len(q_lens)
    S = len(seq_lens)
    cpu_gen = torch.Generator(device="cpu").manual_seed(seed)
    need = [(n + block_size - 1) // block_size for n in seq_lens]
    private = [max(0, nb - shared_prefix_blocks) for nb in need]
    if shared_prefix_blocks:
        assert all(nb >= shared_prefix_blocks for nb in need), "prefix longer than a sequence"
    used = shared_prefix_blocks + sum(private)
    if num_blocks is None:
        num_blocks = max(16, ((used + 15) // 16) * 16)
    assert num_blocks >= used
    perm = torch.randperm(num_blocks, generator=cpu_gen).to(torch.int32)
    max_blocks = max(need + [1]) + extra_table_cols
    tables = torch.zeros((S, max_blocks), dtype=torch.int32)
    cursor = shared_prefix_blocks
    for s in range(S):
        if shared_prefix_blocks:
            tables[s, :shared_prefix_blocks] = perm[:shared_prefix_blocks]
        k = private[s]
        tables[s, shared_prefix_blocks:shared_prefix_blocks + k] = perm[cursor:cursor + k]
        cursor += k

    pos: List[int] = []
    for s in range(S):
        if positions is not None:
            assert len(positions[s]) == q_lens[s]
            pos.extend(int(p) for p in positions[s])
        else:
            pos.extend(range(seq_lens[s] - q_lens[s], seq_lens[s]))
    qsl = [0]
    for ql in q_lens:
        qsl.append(qsl[-1] + ql)
    T = qsl[-1]

    dev_gen = torch.Generator(device=device).manual_seed(seed + 1)
    q = _randn((T, num_heads, head_dim), dev_gen, device, dtype)
    k_new = _randn((T, num_kv_heads, head_dim), dev_gen, device, dtype)
    v_new = _randn((T, num_kv_heads, head_dim), dev_gen, device, dtype)
    pool_shape = (num_blocks, block_size, num_kv_heads, head_dim)
    k_blocks = _randn(pool_shape, dev_gen, device, dtype)
    v_blocks = _randn(pool_shape, dev_gen, device, dtype)

    return Workload(
        name=name, num_heads=num_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
        block_size=block_size, num_blocks=num_blocks, max_blocks_per_seq=max_blocks,
        dtype=dtype, scale=(1.0 / math.sqrt(head_dim)) if scale is None else scale,
        causal=causal, sliding_window=sliding_window, seq_lens_list=list(seq_lens),
        q_lens_list=list(q_lens),
        query_start_loc=torch.tensor(qsl, dtype=torch.int32, device=device),
        seq_lens=torch.tensor(seq_lens, dtype=torch.int32, device=device),
        positions=torch.tensor(pos, dtype=torch.int32, device=device),
        block_tables=tables.to(device), q=q, k_new=k_new, v_new=v_new,
        k_blocks=k_blocks, v_blocks=v_blocks, partition_size=partition_size,
        masked_partition=masked_partition, shared_prefix_blocks=shared_prefix_blocks, seed=seed)


def fp8_pools(w: Workload, spread: float = 8.0, seed: Optional[int] = None):
    """e4m3 K and V pools of w's shape: i.i.d. N(0, spread^2) values drawn in fp32 (seeded) and
    cast with torch's float8_e4m3fn conversion, so the codes span the format's normal range and
    some subnormals.  With k_scale = v_scale = 1 / spread the dequantised pools are about
    N(0, 1), like the bf16 pools.  Only draws inputs: the attention over them is what is
    tested."""
    dev = w.k_blocks.device
    gen = torch.Generator(device=dev).manual_seed(w.seed + 7 if seed is None else seed)
    shape = tuple(w.k_blocks.shape)
    kb = (torch.randn(shape, generator=gen, device=dev) * spread).to(torch.float8_e4m3fn)
    vb = (torch.randn(shape, generator=gen, device=dev) * spread).to(torch.float8_e4m3fn)
    return kb, vb


def fp8_pools_per_head(w: Workload, spreads, seed: Optional[int] = None):
    """e4m3 K and V pools of w's shape whose kv head g is drawn i.i.d. N(0, spreads[g]^2) in
    fp32 (seeded) and cast with torch's float8_e4m3fn conversion: with per-head scales
    1 / spreads[g] every head dequantises to about N(0, 1).  Only draws inputs."""
    dev = w.k_blocks.device
    gen = torch.Generator(device=dev).manual_seed(w.seed + 9 if seed is None else seed)
    shape = tuple(w.k_blocks.shape)
    sp = torch.tensor(list(spreads), dtype=torch.float32, device=dev).view(1, 1, -1, 1)
    kb = (torch.randn(shape, generator=gen, device=dev) * sp).to(torch.float8_e4m3fn)
    vb = (torch.randn(shape, generator=gen, device=dev) * sp).to(torch.float8_e4m3fn)
    return kb, vb


def subset(w: Workload, seqs: List[int], name: Optional[str] = None) -> Workload:
    """The sequences `seqs` of w as a batch of their own, over the same pool (its query rows,
    new K/V rows and metadata, re-indexed)."""
    qsl = w.query_start_loc.cpu().tolist()
    rows = [t for s in seqs for t in range(qsl[s], qsl[s + 1])]
    dev = w.q.device
    idx = torch.tensor(rows, dtype=torch.long, device=dev)
    sel = torch.tensor(seqs, dtype=torch.long, device=dev)
    new_qsl = [0]
    for s in seqs:
        new_qsl.append(new_qsl[-1] + qsl[s + 1] - qsl[s])
    fields = {f.name: getattr(w, f.name) for f in dataclasses.fields(w)}
    fields.update(
        name=name or f"{w.name}-subset", seq_lens_list=[w.seq_lens_list[s] for s in seqs],
        q_lens_list=[w.q_lens_list[s] for s in seqs],
        query_start_loc=torch.tensor(new_qsl, dtype=torch.int32, device=dev),
        seq_lens=w.seq_lens[sel].contiguous(), positions=w.positions[idx].contiguous(),
        block_tables=w.block_tables[sel].contiguous(), q=w.q[idx].contiguous(),
        k_new=w.k_new[idx].contiguous(), v_new=w.v_new[idx].contiguous(),
        masked_partition=[w.masked_partition[s] for s in seqs] if w.masked_partition else None)
    return Workload(**fields)


def _uniform(gen, lo, hi, n):
    """n integers uniform in [lo, hi] (both ends included)."""
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=gen)]


NAMES = {
    1: "tiny-mixed-fp32",
    2: "decode-llama3-8b-64seq",
    3: "mixed-prefill-decode-window4096",
    4: "splitkv-decode-131072ctx",
    5: "shared-prefix-fork-decode-256seq",
}


def prefill_chunks(seed: int = 0, device="cpu") -> Workload:
    """The prefill chunks of workload 3 on their own: 8 chunks of 512 tokens after the same
    prior contexts U{0..2048}, with a pool holding only their blocks (a small case of the
    tcgen05 prefill kernel for profiling)."""
    g = torch.Generator(device="cpu").manual_seed(1000 + seed * 7 + 3)
    _uniform(g, 1024, 8192, 248)  # the decode contexts of workload 3, drawn first there
    prior = _uniform(g, 0, 2048, 8)
    return build("prefill-chunks", seq_lens=[c + 512 for c in prior], q_lens=[512] * 8,
                 num_heads=32, num_kv_heads=8, head_dim=128, sliding_window=4096, seed=seed,
                 device=device)


def named(cfg: int, seed: int = 0, device="cpu", small: bool = False) -> Workload:
    """The five benchmark workloads.

    1  tiny mixed fp32 batch: seq_lens {1, 17, 33, 50}, new tokens {1 decode,
       17-token prefill, 8-token chunk at positions 25..32, 1 decode}; H=4,
       Hkv=2, D=64, b=16, pool of 32 blocks, scale 1/8, causal, no window.
    2  decode batch, Llama-3-8B attention shape: 64 sequences x 1 token,
       contexts U{512..4096}; H=32, Hkv=8, D=128, bf16.
    3  mixed continuous batch: 248 decode tokens (contexts U{1024..8192}) and 8
       prefill chunks of 512 tokens after prior contexts U{0..2048}; H=32,
       Hkv=8, D=128, bf16, window 4096, causal.
    4  long-context split-KV decode: 8 sequences x 131072 context; H=64, Hkv=8,
       D=128, bf16, partitions of 512, one seeded masked partition per sequence.
    5  shared-prefix fork decode: 256 sequences sharing 128 physical blocks (a
       2048-token prefix), private tails U{0..512} tokens, then the decode token
       (seq_len = 2048 + tail + 1, so the new token always lands in a private
       block); H=32, Hkv=8, D=128, bf16.
    """
    g = torch.Generator(device="cpu").manual_seed(1000 + seed * 7 + cfg)
    name = NAMES[cfg] + ("-small" if small else "")
    if cfg == 1:
        return build(name, seq_lens=[1, 17, 33, 50], q_lens=[1, 17, 8, 1], num_heads=4,
                     num_kv_heads=2, head_dim=64, block_size=16, dtype=torch.float32,
                     causal=True, sliding_window=0, seed=seed, device=device, num_blocks=32,
                     scale=1.0 / 8.0)
    if cfg == 2:
        S = 8 if small else 64
        lens = _uniform(g, 512, 4096, S)
        return build(name, seq_lens=lens, q_lens=[1] * S, num_heads=32, num_kv_heads=8,
                     head_dim=128, seed=seed, device=device)
    if cfg == 3:
        n_dec, n_pre, chunk = (12, 2, 96) if small else (248, 8, 512)
        dec_lens = _uniform(g, 300, 1500, n_dec) if small else _uniform(g, 1024, 8192, n_dec)
        prior = _uniform(g, 0, 400, n_pre) if small else _uniform(g, 0, 2048, n_pre)
        window = 512 if small else 4096
        seq_lens = dec_lens + [c + chunk for c in prior]
        q_lens = [1] * n_dec + [chunk] * n_pre
        return build(name, seq_lens=seq_lens, q_lens=q_lens, num_heads=32, num_kv_heads=8,
                     head_dim=128, sliding_window=window, seed=seed, device=device)
    if cfg == 4:
        S, ctx = (2, 4096 + 300) if small else (8, 131072)
        P = 512
        nparts = (ctx + P - 1) // P
        masked = _uniform(g, 0, nparts - 1, S)
        return build(name, seq_lens=[ctx] * S, q_lens=[1] * S, num_heads=64, num_kv_heads=8,
                     head_dim=128, seed=seed, device=device, partition_size=P,
                     masked_partition=masked)
    if cfg == 5:
        S, prefix_blocks, tail_max = (16, 8, 64) if small else (256, 128, 512)
        tails = _uniform(g, 0, tail_max, S)
        seq_lens = [prefix_blocks * 16 + t + 1 for t in tails]
        return build(name, seq_lens=seq_lens, q_lens=[1] * S, num_heads=32, num_kv_heads=8,
                     head_dim=128, seed=seed, device=device,
                     shared_prefix_blocks=prefix_blocks)
    raise ValueError(f"unknown workload {cfg}")
