"""CPU oracle for batched paged attention -- TEST INFRASTRUCTURE ONLY.

Thin ctypes wrappers over ``pa_oracle.c`` (plain C, fp32, two-pass softmax).
Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline /
reference leg may import this package; the library under
``paged_kv_cache_31_gb300`` never does.  Every function takes CPU tensors
(contiguous; bf16 data is passed as its raw bits) and returns the oracle's status
code together with freshly allocated outputs.

Status codes: 0 OK, 1 EINVAL, 2 ESHAPE, 3 EUNSUPPORTED (the tinyllm decode
interface's error classes).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
# PA_ORACLE_SANITIZE=1: an AddressSanitizer + UndefinedBehaviorSanitizer build (the process
# must preload the ASan runtime; tests/test_oracle_sanitizers.py runs the pins that way)
_SANITIZE = os.environ.get("PA_ORACLE_SANITIZE") == "1"
_LIB = os.path.join(_HERE, "libpa_oracle_san.so" if _SANITIZE else "libpa_oracle.so")
_lock = threading.Lock()
_lib = None

OK, EINVAL, ESHAPE, EUNSUPPORTED = 0, 1, 2, 3
_DT = {torch.float32: 0, torch.bfloat16: 1, torch.float8_e4m3fn: 2}


def build(force: bool = False) -> str:
    """Compile pa_oracle.c with gcc (-O2, OpenMP, no fast-math) next to itself."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-std=c11", "-O2", "-fopenmp", "-fPIC", "-shared", "-Wall", "-Wextra",
               "-fno-fast-math", "-ffp-contract=off", "-o", tmp, _SRC, "-lm"]
        if _SANITIZE:
            cmd[2:3] = ["-O1", "-g", "-fsanitize=address,undefined", "-fno-sanitize-recover=all",
                        "-fno-omit-frame-pointer"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            i32, i64, f32, vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p
            L.oracle_set_mutant.argtypes = [ctypes.c_int]
            L.oracle_get_mutant.restype = ctypes.c_int
            L.oracle_num_threads.restype = ctypes.c_int
            L.oracle_set_num_threads.argtypes = [ctypes.c_int]
            L.oracle_slot_mapping.argtypes = [vp, vp, vp, i32, i32, i32, i64, vp]
            L.oracle_reshape_and_cache.argtypes = [vp, vp, vp, vp, vp, i64, i32, i32, i32, i64, i32]
            L.oracle_reshape_and_cache_ex.argtypes = [vp, vp, vp, vp, vp, i64, i32, i32, i32, i64,
                                                      i32, i32, f32, f32]
            L.oracle_gather_kv.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i64, i32, i32]
            L.oracle_varlen_attention.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i64, i32,
                                                  i32, i32, i32, i64, i32, i32, i32, i32, f32, i32,
                                                  i32]
            L.oracle_varlen_attention_ex.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i64,
                                                     i32, i32, i32, i32, i64, i32, i32, i32, i32,
                                                     f32, i32, i32, vp, f32, f32]
            L.oracle_splitkv_partials.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32,
                                                  i32, i64, i32, i32, i32, i32, i32, f32, i32]
            L.oracle_splitkv_partials_ex.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32,
                                                     i32, i32, i64, i32, i32, i32, i32, i32, f32,
                                                     i32, f32, f32]
            L.oracle_reshape_and_cache_per_head.argtypes = [vp, vp, vp, vp, vp, i64, i32, i32,
                                                            i32, i64, i32, i32, vp, vp]
            L.oracle_varlen_attention_per_head.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32,
                                                           i64, i32, i32, i32, i32, i64, i32, i32,
                                                           i32, i32, f32, i32, i32, vp, vp, vp]
            L.oracle_splitkv_partials_per_head.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32,
                                                           i32, i32, i32, i32, i64, i32, i32, i32,
                                                           i32, i32, f32, i32, vp, vp]
            # the per-block variants take the same arguments as the per-head ones
            L.oracle_reshape_and_cache_per_block.argtypes = L.oracle_reshape_and_cache_per_head.argtypes
            L.oracle_varlen_attention_per_block.argtypes = L.oracle_varlen_attention_per_head.argtypes
            L.oracle_splitkv_partials_per_block.argtypes = L.oracle_splitkv_partials_per_head.argtypes
            L.oracle_splitkv_reduce.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32]
            L.oracle_merge_attn_states.argtypes = [vp, vp, vp, vp, vp, vp, i64, i32, i32, i64, i32]
            L.oracle_fp8_to_f32.argtypes = [ctypes.c_uint8]
            L.oracle_fp8_to_f32.restype = f32
            L.oracle_f32_to_fp8.argtypes = [f32]
            L.oracle_f32_to_fp8.restype = ctypes.c_uint8
            L.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
            L.oracle_bf16_to_f32.restype = f32
            L.oracle_f32_to_bf16.argtypes = [f32]
            L.oracle_f32_to_bf16.restype = ctypes.c_uint16
            for name in ("oracle_slot_mapping", "oracle_reshape_and_cache", "oracle_gather_kv",
                         "oracle_varlen_attention", "oracle_varlen_attention_ex",
                         "oracle_reshape_and_cache_ex", "oracle_reshape_and_cache_per_head",
                         "oracle_varlen_attention_per_head", "oracle_splitkv_partials_per_head",
                         "oracle_splitkv_partials", "oracle_splitkv_partials_ex",
                         "oracle_splitkv_reduce",
                         "oracle_merge_attn_states"):
                getattr(L, name).restype = ctypes.c_int
            _lib = L
    return _lib


def _p(t):
    if t is None:
        return None
    assert t.device.type == "cpu" and t.is_contiguous(), "oracle takes contiguous CPU tensors"
    return ctypes.c_void_p(t.data_ptr())


def _cpu(t):
    return None if t is None else t.detach().to("cpu").contiguous()


def set_mutant(n: int) -> None:
    lib().oracle_set_mutant(int(n))


def num_threads() -> int:
    return lib().oracle_num_threads()


def set_num_threads(n: int) -> None:
    lib().oracle_set_num_threads(int(n))


def bf16_to_f32(bits: int) -> float:
    return lib().oracle_bf16_to_f32(bits)


def f32_to_bf16(x: float) -> int:
    return lib().oracle_f32_to_bf16(x)


def slot_mapping(query_start_loc, positions, block_tables, block_size, num_blocks):
    qsl, pos, bt = _cpu(query_start_loc), _cpu(positions), _cpu(block_tables)
    out = torch.full((pos.numel(),), -7, dtype=torch.int32)
    st = lib().oracle_slot_mapping(_p(qsl), _p(pos), _p(bt), qsl.numel() - 1, bt.shape[1],
                                   block_size, num_blocks, _p(out))
    return st, out


def fp8_to_f32(code: int) -> float:
    return lib().oracle_fp8_to_f32(code)


def f32_to_fp8(x: float) -> int:
    return lib().oracle_f32_to_fp8(x)


def reshape_and_cache_ex(k, v, k_blocks, v_blocks, slot_mapping_, block_size, k_scale=1.0,
                         v_scale=1.0):
    """Scatter with conversion: the pool (possibly fp8) receives k / k_scale, v / v_scale."""
    k, v, sm = _cpu(k), _cpu(v), _cpu(slot_mapping_)
    assert k_blocks.is_contiguous() and v_blocks.is_contiguous()
    T, Hkv, D = k.shape
    return lib().oracle_reshape_and_cache_ex(_p(k), _p(v), _p(k_blocks), _p(v_blocks), _p(sm),
                                             T, Hkv, D, block_size, k_blocks.shape[0],
                                             _DT[k.dtype], _DT[k_blocks.dtype], float(k_scale),
                                             float(v_scale))


def reshape_and_cache_per_head(k, v, k_blocks, v_blocks, slot_mapping_, block_size, k_scales,
                               v_scales):
    """Scatter with conversion and one scale per kv head: head g of a row is stored as
    k / k_scales[g], v / v_scales[g] (None: 1 for every head)."""
    k, v, sm = _cpu(k), _cpu(v), _cpu(slot_mapping_)
    ksc, vsc = _scales(k_scales), _scales(v_scales)
    assert k_blocks.is_contiguous() and v_blocks.is_contiguous()
    T, Hkv, D = k.shape
    return lib().oracle_reshape_and_cache_per_head(_p(k), _p(v), _p(k_blocks), _p(v_blocks),
                                                   _p(sm), T, Hkv, D, block_size,
                                                   k_blocks.shape[0], _DT[k.dtype],
                                                   _DT[k_blocks.dtype], _p(ksc), _p(vsc))


def reshape_and_cache_per_block(k, v, k_blocks, v_blocks, slot_mapping_, block_size,
                                k_block_scales, v_block_scales):
    """Scatter with conversion and one scale per (pool block, kv head): head g of a row written
    to slot s is stored as k / k_block_scales[s // block_size, g] (None: 1)."""
    k, v, sm = _cpu(k), _cpu(v), _cpu(slot_mapping_)
    ksc, vsc = _scales(k_block_scales), _scales(v_block_scales)
    assert k_blocks.is_contiguous() and v_blocks.is_contiguous()
    T, Hkv, D = k.shape
    return lib().oracle_reshape_and_cache_per_block(_p(k), _p(v), _p(k_blocks), _p(v_blocks),
                                                    _p(sm), T, Hkv, D, block_size,
                                                    k_blocks.shape[0], _DT[k.dtype],
                                                    _DT[k_blocks.dtype], _p(ksc), _p(vsc))


def _scales(x):
    return None if x is None else _cpu(x).to(torch.float32).contiguous()


def reshape_and_cache(k, v, k_blocks, v_blocks, slot_mapping_, block_size):
    """Scatter in place into (CPU) k_blocks / v_blocks."""
    k, v, sm = _cpu(k), _cpu(v), _cpu(slot_mapping_)
    assert k_blocks.is_contiguous() and v_blocks.is_contiguous()
    T, Hkv, D = k.shape
    return lib().oracle_reshape_and_cache(_p(k), _p(v), _p(k_blocks), _p(v_blocks), _p(sm), T,
                                          Hkv, D, block_size, k_blocks.shape[0], _DT[k.dtype])


def gather_kv(k_blocks, v_blocks, cu_seq_lens, block_tables, seq_starts=None):
    kb, vb = _cpu(k_blocks), _cpu(v_blocks)
    cu, bt, ss = _cpu(cu_seq_lens), _cpu(block_tables), _cpu(seq_starts)
    NB, bs, Hkv, D = kb.shape
    rows = int(cu[-1])
    ko = torch.zeros((rows, Hkv, D), dtype=kb.dtype)
    vo = torch.zeros((rows, Hkv, D), dtype=kb.dtype) if vb is not None else None
    st = lib().oracle_gather_kv(_p(kb), _p(vb), _p(ko), _p(vo), _p(cu), _p(ss), _p(bt),
                                cu.numel() - 1, Hkv, D, bs, NB, bt.shape[1], _DT[kb.dtype])
    return st, ko, vo


def varlen_attention(q, k_blocks, v_blocks, query_start_loc, seq_lens, positions, block_tables,
                     scale, causal=True, sliding_window=0, out_dtype=torch.float32,
                     want_lse=False, num_kv_heads=None, out=None, sinks=None, k_scale=1.0,
                     v_scale=1.0, k_scales=None, v_scales=None, k_block_scales=None,
                     v_block_scales=None):
    """Two-pass attention of every (token, head).  Returns (status, out [T,H,D], lse [H,T]).
    sinks: optional [H] fp32 sink logits (a virtual zero-valued position per head);
    k_scale / v_scale: dequantisation scales of the pool (K = k_scale * pool);
    k_scales / v_scales: one scale per kv head instead (K = k_scales[g] * pool);
    k_block_scales / v_block_scales: [NB, Hkv], one per (pool block, kv head) instead."""
    q, kb, vb = _cpu(q), _cpu(k_blocks), _cpu(v_blocks)
    qsl, sl, pos, bt = _cpu(query_start_loc), _cpu(seq_lens), _cpu(positions), _cpu(block_tables)
    T, H, D = q.shape
    NB, bs, Hkv, Dk = kb.shape
    if num_kv_heads is not None:
        Hkv = num_kv_heads
    if out is None:
        out = torch.zeros((T, H, D), dtype=out_dtype)
    lse = torch.full((H, T), float("nan"), dtype=torch.float32) if want_lse else None
    sk = None if sinks is None else _cpu(sinks).to(torch.float32).contiguous()
    args = (_p(q), _p(kb), _p(vb), _p(out), _p(lse), _p(qsl), _p(sl), _p(pos), _p(bt),
            qsl.numel() - 1, T, H, Hkv, D, bs, NB, bt.shape[1], _DT[q.dtype], _DT[kb.dtype],
            _DT[out.dtype], float(scale), int(bool(causal)), int(sliding_window), _p(sk))
    if k_block_scales is not None or v_block_scales is not None:
        ksc, vsc = _scales(k_block_scales), _scales(v_block_scales)
        st = lib().oracle_varlen_attention_per_block(*args, _p(ksc), _p(vsc))
    elif k_scales is not None or v_scales is not None:
        ksc, vsc = _scales(k_scales), _scales(v_scales)
        st = lib().oracle_varlen_attention_per_head(*args, _p(ksc), _p(vsc))
    else:
        st = lib().oracle_varlen_attention_ex(*args, float(k_scale), float(v_scale))
    return st, out, lse


def splitkv_partials(q, k_blocks, v_blocks, seq_lens, block_tables, scale, partition_size,
                     max_parts, sliding_window=0, k_scale=1.0, v_scale=1.0, k_scales=None,
                     v_scales=None, k_block_scales=None, v_block_scales=None):
    """Phase 1 of split-KV decode: (status, max_logits, exp_sums, tmp_out).  k_scale / v_scale:
    dequantisation scales of the pool (K = k_scale * pool); k_scales / v_scales: one per kv
    head instead."""
    q, kb, vb, sl, bt = _cpu(q), _cpu(k_blocks), _cpu(v_blocks), _cpu(seq_lens), _cpu(block_tables)
    S, H, D = q.shape
    NB, bs, Hkv, _ = kb.shape
    ml = torch.full((S, H, max_parts), float("nan"), dtype=torch.float32)
    es = torch.full((S, H, max_parts), float("nan"), dtype=torch.float32)
    to = torch.full((S, H, max_parts, D), float("nan"), dtype=torch.float32)
    args = (_p(q), _p(kb), _p(vb), _p(ml), _p(es), _p(to), _p(sl), _p(bt), S, H, Hkv, D, bs, NB,
            bt.shape[1], partition_size, max_parts, _DT[q.dtype], _DT[kb.dtype], float(scale),
            int(sliding_window))
    if k_block_scales is not None or v_block_scales is not None:
        ksc, vsc = _scales(k_block_scales), _scales(v_block_scales)
        st = lib().oracle_splitkv_partials_per_block(*args, _p(ksc), _p(vsc))
    elif k_scales is not None or v_scales is not None:
        ksc, vsc = _scales(k_scales), _scales(v_scales)  # kept alive across the call
        st = lib().oracle_splitkv_partials_per_head(*args, _p(ksc), _p(vsc))
    else:
        st = lib().oracle_splitkv_partials_ex(*args, float(k_scale), float(v_scale))
    return st, ml, es, to


def splitkv_reduce(max_logits, exp_sums, tmp_out, seq_lens, partition_size,
                   out_dtype=torch.float32):
    ml, es, to, sl = _cpu(max_logits), _cpu(exp_sums), _cpu(tmp_out), _cpu(seq_lens)
    S, H, P, D = to.shape
    out = torch.zeros((S, H, D), dtype=out_dtype)
    st = lib().oracle_splitkv_reduce(_p(out), _p(ml), _p(es), _p(to), _p(sl), S, H, D,
                                     partition_size, P, _DT[out_dtype])
    return st, out


def merge_attn_states(prefix_out, prefix_lse, suffix_out, suffix_lse,
                      prefill_tokens_with_context=-1, want_lse=True):
    po, pl, so, sl = _cpu(prefix_out), _cpu(prefix_lse), _cpu(suffix_out), _cpu(suffix_lse)
    T, H, D = po.shape
    out = torch.zeros_like(po)
    out_lse = torch.full((H, T), float("nan"), dtype=torch.float32) if want_lse else None
    st = lib().oracle_merge_attn_states(_p(out), _p(out_lse), _p(po), _p(pl), _p(so), _p(sl), T,
                                        H, D, int(prefill_tokens_with_context), _DT[po.dtype])
    return st, out, out_lse
