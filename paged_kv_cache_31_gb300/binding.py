"""ctypes binding of libpa.so: the C ABI of include/pa.h, call for call.

Each ``pa_*`` function takes torch tensors that live on the current CUDA device,
checks their shapes / dtypes / contiguity, passes raw pointers and the current
stream to the library, and raises ``PaError`` on a non-OK status.  It does no
arithmetic of its own: every step of the path runs in the library's kernels.
Importing this module loads the library and raises if it has not been built
(``python -c "import __graft_entry__ as g; g.build()"``); there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpa.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"libpa.so is not built ({LIB_PATH}); run __graft_entry__.build() first")

_lib = ctypes.CDLL(LIB_PATH)

PA_OK, PA_EINVAL, PA_ESHAPE, PA_EUNSUPPORTED, PA_ECUDA, PA_ETIMEOUT = range(6)
PA_F32, PA_BF16, PA_FP8_E4M3 = 0, 1, 2
PA_FLAG_BITWISE = 1
_DT = {torch.float32: PA_F32, torch.bfloat16: PA_BF16, torch.float8_e4m3fn: PA_FP8_E4M3}

_vp, _i32, _i64, _f32, _sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                              ctypes.c_size_t)
_SIGS = {
    "pa_version": ([], ctypes.c_int),
    "pa_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "pa_device_status": ([_vp], ctypes.c_int),
    "pa_slot_mapping": ([_vp, _vp, _vp, _i32, _i64, _i32, _i32, _i64, _vp, _vp], ctypes.c_int),
    "pa_reshape_and_cache": ([_vp, _vp, _vp, _vp, _vp, _i64, _i32, _i32, _i32, _i64, ctypes.c_int,
                              _vp], ctypes.c_int),
    "pa_slot_mapping_and_cache": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64, _i32, _i32,
                                   _i32, _i32, _i64, ctypes.c_int, _vp, _vp], ctypes.c_int),
    "pa_reshape_and_cache_ex": ([_vp, _vp, _vp, _vp, _vp, _i64, _i32, _i32, _i32, _i64,
                                 ctypes.c_int, ctypes.c_int, _f32, _f32, _vp], ctypes.c_int),
    "pa_reshape_and_cache_per_head": ([_vp, _vp, _vp, _vp, _vp, _i64, _i32, _i32, _i32, _i64,
                                       ctypes.c_int, ctypes.c_int, _vp, _vp, _vp], ctypes.c_int),
    "pa_reshape_and_cache_per_block": ([_vp, _vp, _vp, _vp, _vp, _i64, _i32, _i32, _i32, _i64,
                                        ctypes.c_int, ctypes.c_int, _vp, _vp, _vp], ctypes.c_int),
    "pa_varlen_forward_workspace_size": ([_i32, _i64, _i32, _i32, _i32, _i32, _i32], _sz),
    "pa_varlen_forward": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64, _i32, _i32, _i32,
                           _i32, _i64, _i32, ctypes.c_int, ctypes.c_int, _f32, _i32, _i32, _vp,
                           _sz, _vp], ctypes.c_int),
    "pa_varlen_forward_ex": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64, _i32, _i32,
                              _i32, _i32, _i64, _i32, ctypes.c_int, ctypes.c_int, _f32, _i32,
                              _i32, _vp, _vp, _f32, _f32, ctypes.c_uint32, _vp, _sz, _vp],
                             ctypes.c_int),
    "pa_varlen_forward_per_head": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64, _i32,
                                    _i32, _i32, _i32, _i64, _i32, ctypes.c_int, ctypes.c_int,
                                    _f32, _i32, _i32, _vp, _vp, _vp, _vp, ctypes.c_uint32, _vp,
                                    _sz, _vp], ctypes.c_int),
    "pa_varlen_forward_per_block": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64, _i32,
                                     _i32, _i32, _i32, _i64, _i32, ctypes.c_int, ctypes.c_int,
                                     _f32, _i32, _i32, _vp, _vp, _vp, _vp, ctypes.c_uint32, _vp,
                                     _sz, _vp], ctypes.c_int),
    "pa_cache_and_attend": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64, _i32,
                             _i32, _i32, _i32, _i64, _i32, ctypes.c_int, ctypes.c_int, _f32,
                             _i32, _i32, _vp, _vp, _sz, _vp], ctypes.c_int),
    "pa_varlen_forward_noalloc": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64, _i32, _i32,
                                   _i32, _i32, _i64, _i32, ctypes.c_int, ctypes.c_int, _f32, _i32,
                                   _i32, _vp], ctypes.c_int),
    "pa_decode_splitkv_partials": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32,
                                    _i32, _i64, _i32, _i32, _i32, ctypes.c_int, ctypes.c_int, _f32,
                                    _i32, _vp], ctypes.c_int),
    "pa_decode_splitkv_partials_ex": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32,
                                       _i32, _i32, _i64, _i32, _i32, _i32, ctypes.c_int,
                                       ctypes.c_int, _f32, _i32, _f32, _f32, _vp], ctypes.c_int),
    "pa_decode_splitkv_partials_per_head": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32,
                                             _i32, _i32, _i32, _i64, _i32, _i32, _i32,
                                             ctypes.c_int, ctypes.c_int, _f32, _i32, _vp, _vp,
                                             _vp], ctypes.c_int),
    "pa_decode_splitkv_partials_per_block": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32,
                                              _i32, _i32, _i32, _i32, _i64, _i32, _i32, _i32,
                                              ctypes.c_int, ctypes.c_int, _f32, _i32, _vp, _vp,
                                              _vp], ctypes.c_int),
    "pa_decode_splitkv_reduce": ([_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32,
                                  ctypes.c_int, _vp], ctypes.c_int),
    "pa_decode_splitkv": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32,
                           _i64, _i32, _i32, _i32, ctypes.c_int, ctypes.c_int, _f32, _i32, _vp],
                          ctypes.c_int),
    "pa_merge_attn_states": ([_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i32, _i32, _i64, ctypes.c_int,
                              _vp], ctypes.c_int),
    "pa_gather_kv": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64, _i32, _i32, _i32, _i64, _i32,
                      ctypes.c_int, _vp], ctypes.c_int),
}
for _name, (_args, _res) in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.argtypes = _args
    _f.restype = _res

EXPORTED = tuple(_SIGS)


class PaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


def status_string(status: int) -> str:
    return _lib.pa_status_string(int(status)).decode()


def version() -> int:
    return _lib.pa_version()


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(st: int, where: str):
    if st != PA_OK:
        raise PaError(st, where)


def _dev(*ts):
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("tensors must live on the CUDA device")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


def _i32t(*ts):
    for t in ts:
        if t is not None and t.dtype != torch.int32:
            raise ValueError("metadata tensors must be int32")


def pa_device_status(stream=None) -> int:
    """Synchronise the stream; return and clear the device's sticky status word."""
    return _lib.pa_device_status(_stream(stream))


def pa_slot_mapping(query_start_loc, positions, block_tables, block_size, num_blocks, out=None,
                    stream=None):
    _dev(query_start_loc, positions, block_tables)
    _i32t(query_start_loc, positions, block_tables)
    T = positions.numel()
    if out is None:
        out = torch.empty(T, dtype=torch.int32, device=positions.device)
    _check(_lib.pa_slot_mapping(_p(query_start_loc), _p(positions), _p(block_tables),
                                query_start_loc.numel() - 1, T, block_tables.shape[1], block_size,
                                num_blocks, _p(out), _stream(stream)), "pa_slot_mapping")
    return out


def pa_slot_mapping_and_cache(k, v, k_blocks, v_blocks, query_start_loc, positions,
                              block_tables, out=None, stream=None):
    """pa_slot_mapping followed by pa_reshape_and_cache, one launch for decode-sized batches;
    returns the slot mapping."""
    _dev(k, v, k_blocks, v_blocks, query_start_loc, positions, block_tables, out)
    _i32t(query_start_loc, positions, block_tables, out)
    if k.shape != v.shape or k.dim() != 3 or k_blocks.shape != v_blocks.shape:
        raise ValueError("k, v must be [T, Hkv, D]; pools [NB, b, Hkv, D]")
    if k.dtype != k_blocks.dtype or v.dtype != v_blocks.dtype or k.dtype != v.dtype:
        raise ValueError("new rows and pools must share one dtype")
    T, Hkv, D = k.shape
    NB, bs, Hkv2, D2 = k_blocks.shape
    if (Hkv, D) != (Hkv2, D2) or positions.numel() != T:
        raise ValueError("kv heads / head size / token count differ between rows and pool")
    if out is None:
        out = torch.empty(T, dtype=torch.int32, device=k.device)
    _check(_lib.pa_slot_mapping_and_cache(_p(k), _p(v), _p(k_blocks), _p(v_blocks),
                                          _p(query_start_loc), _p(positions), _p(block_tables),
                                          query_start_loc.numel() - 1, T, block_tables.shape[1],
                                          Hkv, D, bs, NB, _DT[k.dtype], _p(out),
                                          _stream(stream)), "pa_slot_mapping_and_cache")
    return out


def pa_reshape_and_cache(k, v, k_blocks, v_blocks, slot_mapping, stream=None, k_scale=None,
                         v_scale=None, k_scales=None, v_scales=None, k_block_scales=None,
                         v_block_scales=None):
    """pa_reshape_and_cache (rows and pools of one dtype, a copy), or pa_reshape_and_cache_ex
    when the pools' dtype differs from the rows' or a scale is given (pool = rows / scale,
    rounded to the pool's dtype, e.g. torch.float8_e4m3fn), or
    pa_reshape_and_cache_per_head when k_scales / v_scales (device fp32 [num_kv_heads]) are
    given, or pa_reshape_and_cache_per_block with k_block_scales / v_block_scales (device fp32
    [num_blocks, num_kv_heads], both)."""
    _dev(k, v, k_blocks, v_blocks, slot_mapping)
    _i32t(slot_mapping)
    if k.shape != v.shape or k.dim() != 3 or k_blocks.shape != v_blocks.shape:
        raise ValueError("k, v must be [T, Hkv, D]; pools [NB, b, Hkv, D]")
    if k.dtype != v.dtype or k_blocks.dtype != v_blocks.dtype:
        raise ValueError("k and v (and the two pools) must share one dtype")
    T, Hkv, D = k.shape
    NB, bs, Hkv2, D2 = k_blocks.shape
    if (Hkv, D) != (Hkv2, D2):
        raise ValueError("kv heads / head size differ between rows and pool")
    if k_block_scales is not None or v_block_scales is not None:
        _block_scales(NB, Hkv, k_block_scales, v_block_scales)
        _check(_lib.pa_reshape_and_cache_per_block(_p(k), _p(v), _p(k_blocks), _p(v_blocks),
                                                   _p(slot_mapping), T, Hkv, D, bs, NB,
                                                   _DT[k.dtype], _DT[k_blocks.dtype],
                                                   _p(k_block_scales), _p(v_block_scales),
                                                   _stream(stream)),
               "pa_reshape_and_cache_per_block")
        return
    if k_scales is not None or v_scales is not None:
        _head_scales(Hkv, k_scales, v_scales)
        _check(_lib.pa_reshape_and_cache_per_head(_p(k), _p(v), _p(k_blocks), _p(v_blocks),
                                                  _p(slot_mapping), T, Hkv, D, bs, NB,
                                                  _DT[k.dtype], _DT[k_blocks.dtype],
                                                  _p(k_scales), _p(v_scales), _stream(stream)),
               "pa_reshape_and_cache_per_head")
        return
    if k.dtype == k_blocks.dtype and k_scale is None and v_scale is None:
        _check(_lib.pa_reshape_and_cache(_p(k), _p(v), _p(k_blocks), _p(v_blocks),
                                         _p(slot_mapping), T, Hkv, D, bs, NB, _DT[k.dtype],
                                         _stream(stream)), "pa_reshape_and_cache")
        return
    _check(_lib.pa_reshape_and_cache_ex(_p(k), _p(v), _p(k_blocks), _p(v_blocks),
                                        _p(slot_mapping), T, Hkv, D, bs, NB, _DT[k.dtype],
                                        _DT[k_blocks.dtype],
                                        1.0 if k_scale is None else float(k_scale),
                                        1.0 if v_scale is None else float(v_scale),
                                        _stream(stream)), "pa_reshape_and_cache_ex")


def _head_scales(Hkv, *arrays):
    for a in arrays:
        if a is None:
            continue
        _dev(a)
        if a.dtype != torch.float32 or a.shape != (Hkv,) or not a.is_contiguous():
            raise ValueError("per-head scales must be contiguous fp32 [num_kv_heads] tensors")


def _block_scales(NB, Hkv, ks, vs):
    if ks is None or vs is None:
        raise ValueError("per-block scales need both k_block_scales and v_block_scales")
    for a in (ks, vs):
        _dev(a)
        if a.dtype != torch.float32 or a.shape != (NB, Hkv) or not a.is_contiguous():
            raise ValueError("per-block scales must be contiguous fp32 [num_blocks, num_kv_heads]")


def pa_varlen_forward_workspace_size(num_seqs, num_tokens, num_heads, num_kv_heads, head_dim,
                                     max_blocks_per_seq, block_size) -> int:
    return int(_lib.pa_varlen_forward_workspace_size(num_seqs, num_tokens, num_heads, num_kv_heads,
                                                     head_dim, max_blocks_per_seq, block_size))


def workspace_for(q, k_blocks, query_start_loc, block_tables):
    T, H, D = q.shape
    NB, bs, Hkv, _ = k_blocks.shape
    n = pa_varlen_forward_workspace_size(query_start_loc.numel() - 1, T, H, Hkv, D,
                                         block_tables.shape[1], bs)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=q.device)


def pa_varlen_forward(q, k_blocks, v_blocks, out, query_start_loc, seq_lens, positions,
                      block_tables, scale, causal=True, sliding_window=0, workspace=None,
                      stream=None, sinks=None, lse=None, k_scale=1.0, v_scale=1.0,
                      bitwise=False, k_scales=None, v_scales=None, k_block_scales=None,
                      v_block_scales=None):
    """pa_varlen_forward, or pa_varlen_forward_ex when sinks ([H] fp32 sink logits), lse
    (a [H, T] fp32 output), a dequantisation scale other than 1 or bitwise=True
    (PA_FLAG_BITWISE: decode and prefill rows give the same bits) is given, or
    pa_varlen_forward_per_head with k_scales / v_scales (device fp32 [num_kv_heads]), or
    pa_varlen_forward_per_block with k_block_scales / v_block_scales (device fp32
    [num_blocks, num_kv_heads], both; e4m3 pools)."""
    _dev(q, k_blocks, v_blocks, out, query_start_loc, seq_lens, positions, block_tables, workspace,
         sinks, lse)
    _i32t(query_start_loc, seq_lens, positions, block_tables)
    if q.dim() != 3 or out.shape != q.shape or out.dtype != q.dtype:
        raise ValueError("q and out must be [T, H, D] of one dtype")
    if k_blocks.shape != v_blocks.shape or k_blocks.dtype != v_blocks.dtype:
        raise ValueError("k_blocks and v_blocks must match")
    T, H, D = q.shape
    NB, bs, Hkv, D2 = k_blocks.shape
    if D2 != D:
        raise ValueError("head size differs between q and the pool")
    if workspace is None:
        workspace = workspace_for(q, k_blocks, query_start_loc, block_tables)
    per_head = k_scales is not None or v_scales is not None
    per_block = k_block_scales is not None or v_block_scales is not None
    if (per_head or per_block) and (k_scale != 1.0 or v_scale != 1.0):
        raise ValueError("give either per-pool, per-head or per-block scales")
    if per_head and per_block:
        raise ValueError("give either per-head or per-block scales")
    if (sinks is None and lse is None and k_scale == 1.0 and v_scale == 1.0 and not bitwise
            and not per_head and not per_block):
        _check(_lib.pa_varlen_forward(_p(q), _p(k_blocks), _p(v_blocks), _p(out),
                                      _p(query_start_loc), _p(seq_lens), _p(positions),
                                      _p(block_tables), query_start_loc.numel() - 1, T, H, Hkv, D,
                                      bs, NB, block_tables.shape[1], _DT[q.dtype],
                                      _DT[k_blocks.dtype], float(scale), int(bool(causal)),
                                      int(sliding_window), _p(workspace), workspace.numel(),
                                      _stream(stream)),
               "pa_varlen_forward")
        return out
    if sinks is not None and (sinks.dtype != torch.float32 or sinks.shape != (H,)
                              or not sinks.is_contiguous()):
        raise ValueError("sinks must be a contiguous fp32 [num_heads] tensor")
    if lse is not None and (lse.dtype != torch.float32 or lse.shape != (H, T)
                            or not lse.is_contiguous()):
        raise ValueError("lse must be a contiguous fp32 [num_heads, num_tokens] tensor")
    head = (_p(q), _p(k_blocks), _p(v_blocks), _p(out), _p(query_start_loc), _p(seq_lens),
            _p(positions), _p(block_tables), query_start_loc.numel() - 1, T, H, Hkv, D, bs, NB,
            block_tables.shape[1], _DT[q.dtype], _DT[k_blocks.dtype], float(scale),
            int(bool(causal)), int(sliding_window), _p(sinks), _p(lse))
    tail = (PA_FLAG_BITWISE if bitwise else 0, _p(workspace), workspace.numel(), _stream(stream))
    if per_head:
        _head_scales(Hkv, k_scales, v_scales)
        _check(_lib.pa_varlen_forward_per_head(*head, _p(k_scales), _p(v_scales), *tail),
               "pa_varlen_forward_per_head")
        return out
    if per_block:
        _block_scales(NB, Hkv, k_block_scales, v_block_scales)
        _check(_lib.pa_varlen_forward_per_block(*head, _p(k_block_scales), _p(v_block_scales),
                                                *tail), "pa_varlen_forward_per_block")
        return out
    _check(_lib.pa_varlen_forward_ex(*head, float(k_scale), float(v_scale), *tail),
           "pa_varlen_forward_ex")
    return out


def pa_cache_and_attend(k_new, v_new, q, k_blocks, v_blocks, out, query_start_loc, seq_lens,
                        positions, block_tables, scale, causal=True, sliding_window=0,
                        workspace=None, slot_mapping=None, stream=None):
    """pa_slot_mapping_and_cache of the new rows, then pa_varlen_forward of q (one call; the
    scatter overlaps the attention's planning kernel).  Returns the slot mapping."""
    _dev(k_new, v_new, q, k_blocks, v_blocks, out, query_start_loc, seq_lens, positions,
         block_tables, workspace, slot_mapping)
    _i32t(query_start_loc, seq_lens, positions, block_tables, slot_mapping)
    if q.dim() != 3 or out.shape != q.shape or out.dtype != q.dtype:
        raise ValueError("q and out must be [T, H, D] of one dtype")
    if k_blocks.shape != v_blocks.shape or k_blocks.dtype != v_blocks.dtype:
        raise ValueError("k_blocks and v_blocks must match")
    if k_new.shape != v_new.shape or k_new.dtype != k_blocks.dtype or v_new.dtype != v_blocks.dtype:
        raise ValueError("new rows must be [T, Hkv, D] of the pool dtype")
    T, H, D = q.shape
    NB, bs, Hkv, D2 = k_blocks.shape
    if D2 != D or k_new.shape != (T, Hkv, D):
        raise ValueError("shapes of q, the new rows and the pool differ")
    if workspace is None:
        workspace = workspace_for(q, k_blocks, query_start_loc, block_tables)
    if slot_mapping is None:
        slot_mapping = torch.empty(T, dtype=torch.int32, device=q.device)
    _check(_lib.pa_cache_and_attend(_p(k_new), _p(v_new), _p(q), _p(k_blocks), _p(v_blocks),
                                    _p(out), _p(query_start_loc), _p(seq_lens), _p(positions),
                                    _p(block_tables), query_start_loc.numel() - 1, T, H, Hkv, D,
                                    bs, NB, block_tables.shape[1], _DT[q.dtype],
                                    _DT[k_blocks.dtype], float(scale), int(bool(causal)),
                                    int(sliding_window), _p(slot_mapping), _p(workspace),
                                    workspace.numel(), _stream(stream)), "pa_cache_and_attend")
    return slot_mapping


def pa_varlen_forward_noalloc(q, k_blocks, v_blocks, out, query_start_loc, seq_lens, positions,
                              block_tables, scale, causal=True, sliding_window=0, stream=None):
    """pa_varlen_forward for callers that cannot allocate: the plan lives in a fixed 4 MiB
    array inside the library (one per device), so no workspace is passed or allocated.
    Calls that may overlap on the GPU share that array and must not be issued."""
    _dev(q, k_blocks, v_blocks, out, query_start_loc, seq_lens, positions, block_tables)
    _i32t(query_start_loc, seq_lens, positions, block_tables)
    if q.dim() != 3 or out.shape != q.shape or out.dtype != q.dtype:
        raise ValueError("q and out must be [T, H, D] of one dtype")
    if k_blocks.shape != v_blocks.shape or k_blocks.dtype != v_blocks.dtype:
        raise ValueError("k_blocks and v_blocks must match")
    T, H, D = q.shape
    NB, bs, Hkv, D2 = k_blocks.shape
    if D2 != D:
        raise ValueError("head size differs between q and the pool")
    _check(_lib.pa_varlen_forward_noalloc(_p(q), _p(k_blocks), _p(v_blocks), _p(out),
                                          _p(query_start_loc), _p(seq_lens), _p(positions),
                                          _p(block_tables), query_start_loc.numel() - 1, T, H,
                                          Hkv, D, bs, NB, block_tables.shape[1], _DT[q.dtype],
                                          _DT[k_blocks.dtype], float(scale), int(bool(causal)),
                                          int(sliding_window), _stream(stream)),
           "pa_varlen_forward_noalloc")
    return out


def _split_shapes(q, k_blocks, max_logits, tmp_out):
    S, H, D = q.shape
    NB, bs, Hkv, D2 = k_blocks.shape
    if D2 != D or tmp_out.shape[:2] != (S, H) or tmp_out.shape[3] != D:
        raise ValueError("split-KV shapes disagree")
    if max_logits.shape != tmp_out.shape[:3]:
        raise ValueError("max_logits / exp_sums must be [S, H, P]")
    return S, H, D, NB, bs, Hkv, tmp_out.shape[2]


def pa_decode_splitkv_partials(q, k_blocks, v_blocks, max_logits, exp_sums, tmp_out, seq_lens,
                               block_tables, scale, partition_size=512, sliding_window=0,
                               stream=None, k_scale=1.0, v_scale=1.0, k_scales=None,
                               v_scales=None, k_block_scales=None, v_block_scales=None):
    """pa_decode_splitkv_partials, or pa_decode_splitkv_partials_ex when a dequantisation scale
    other than 1 is given, or pa_decode_splitkv_partials_per_head with k_scales / v_scales
    (device fp32 [num_kv_heads]), or pa_decode_splitkv_partials_per_block with k_block_scales /
    v_block_scales (device fp32 [num_blocks, num_kv_heads], both; e4m3 pools)."""
    _dev(q, k_blocks, v_blocks, max_logits, exp_sums, tmp_out, seq_lens, block_tables)
    _i32t(seq_lens, block_tables)
    S, H, D, NB, bs, Hkv, P = _split_shapes(q, k_blocks, max_logits, tmp_out)
    if k_block_scales is not None or v_block_scales is not None:
        _block_scales(NB, Hkv, k_block_scales, v_block_scales)
        _check(_lib.pa_decode_splitkv_partials_per_block(
            _p(q), _p(k_blocks), _p(v_blocks), _p(max_logits), _p(exp_sums), _p(tmp_out),
            _p(seq_lens), _p(block_tables), S, H, Hkv, D, bs, NB, block_tables.shape[1],
            partition_size, P, _DT[q.dtype], _DT[k_blocks.dtype], float(scale),
            int(sliding_window), _p(k_block_scales), _p(v_block_scales), _stream(stream)),
            "pa_decode_splitkv_partials_per_block")
        return
    if k_scales is not None or v_scales is not None:
        _head_scales(Hkv, k_scales, v_scales)
        _check(_lib.pa_decode_splitkv_partials_per_head(
            _p(q), _p(k_blocks), _p(v_blocks), _p(max_logits), _p(exp_sums), _p(tmp_out),
            _p(seq_lens), _p(block_tables), S, H, Hkv, D, bs, NB, block_tables.shape[1],
            partition_size, P, _DT[q.dtype], _DT[k_blocks.dtype], float(scale),
            int(sliding_window), _p(k_scales), _p(v_scales), _stream(stream)),
            "pa_decode_splitkv_partials_per_head")
        return
    if k_scale != 1.0 or v_scale != 1.0:
        _check(_lib.pa_decode_splitkv_partials_ex(
            _p(q), _p(k_blocks), _p(v_blocks), _p(max_logits), _p(exp_sums), _p(tmp_out),
            _p(seq_lens), _p(block_tables), S, H, Hkv, D, bs, NB, block_tables.shape[1],
            partition_size, P, _DT[q.dtype], _DT[k_blocks.dtype], float(scale),
            int(sliding_window), float(k_scale), float(v_scale), _stream(stream)),
            "pa_decode_splitkv_partials_ex")
        return
    _check(_lib.pa_decode_splitkv_partials(_p(q), _p(k_blocks), _p(v_blocks), _p(max_logits),
                                           _p(exp_sums), _p(tmp_out), _p(seq_lens),
                                           _p(block_tables), S, H, Hkv, D, bs, NB,
                                           block_tables.shape[1], partition_size, P,
                                           _DT[q.dtype], _DT[k_blocks.dtype], float(scale),
                                           int(sliding_window), _stream(stream)),
           "pa_decode_splitkv_partials")


def pa_decode_splitkv_reduce(out, max_logits, exp_sums, tmp_out, seq_lens, partition_size=512,
                             stream=None):
    _dev(out, max_logits, exp_sums, tmp_out, seq_lens)
    _i32t(seq_lens)
    S, H, P, D = tmp_out.shape
    if out.shape != (S, H, D):
        raise ValueError("out must be [S, H, D]")
    _check(_lib.pa_decode_splitkv_reduce(_p(out), _p(max_logits), _p(exp_sums), _p(tmp_out),
                                         _p(seq_lens), S, H, D, partition_size, P,
                                         _DT[out.dtype], _stream(stream)),
           "pa_decode_splitkv_reduce")
    return out


def pa_decode_splitkv(q, k_blocks, v_blocks, out, max_logits, exp_sums, tmp_out, seq_lens,
                      block_tables, scale, partition_size=512, sliding_window=0, stream=None):
    _dev(q, k_blocks, v_blocks, out, max_logits, exp_sums, tmp_out, seq_lens, block_tables)
    _i32t(seq_lens, block_tables)
    S, H, D, NB, bs, Hkv, P = _split_shapes(q, k_blocks, max_logits, tmp_out)
    if out.shape != q.shape or out.dtype != q.dtype:
        raise ValueError("out must match q")
    _check(_lib.pa_decode_splitkv(_p(q), _p(k_blocks), _p(v_blocks), _p(out), _p(max_logits),
                                  _p(exp_sums), _p(tmp_out), _p(seq_lens), _p(block_tables), S, H,
                                  Hkv, D, bs, NB, block_tables.shape[1], partition_size, P,
                                  _DT[q.dtype], _DT[k_blocks.dtype], float(scale),
                                  int(sliding_window), _stream(stream)), "pa_decode_splitkv")
    return out


def pa_merge_attn_states(out, out_lse, prefix_out, prefix_lse, suffix_out, suffix_lse,
                         prefill_tokens_with_context=-1, stream=None):
    _dev(out, out_lse, prefix_out, prefix_lse, suffix_out, suffix_lse)
    T, H, D = prefix_out.shape
    if out.shape != prefix_out.shape or suffix_out.shape != prefix_out.shape:
        raise ValueError("outputs must be [T, H, D]")
    if out.dtype != prefix_out.dtype or suffix_out.dtype != prefix_out.dtype:
        raise ValueError("outputs must share one dtype")
    for lse in (prefix_lse, suffix_lse, out_lse):
        if lse is not None and (lse.shape != (H, T) or lse.dtype != torch.float32):
            raise ValueError("lse must be fp32 [H, T]")
    _check(_lib.pa_merge_attn_states(_p(out), _p(out_lse), _p(prefix_out), _p(prefix_lse),
                                     _p(suffix_out), _p(suffix_lse), T, H, D,
                                     int(prefill_tokens_with_context), _DT[out.dtype],
                                     _stream(stream)), "pa_merge_attn_states")
    return out


def pa_gather_kv(k_blocks, v_blocks, k_out, v_out, cu_seq_lens, block_tables, seq_starts=None,
                 stream=None):
    _dev(k_blocks, v_blocks, k_out, v_out, cu_seq_lens, block_tables, seq_starts)
    _i32t(cu_seq_lens, block_tables, seq_starts)
    NB, bs, Hkv, D = k_blocks.shape
    if k_out.dim() != 3 or k_out.shape[1:] != (Hkv, D) or k_out.dtype != k_blocks.dtype:
        raise ValueError("k_out must be [rows, Hkv, D] of the pool dtype")
    _check(_lib.pa_gather_kv(_p(k_blocks), _p(v_blocks), _p(k_out), _p(v_out), _p(cu_seq_lens),
                             _p(seq_starts), _p(block_tables), cu_seq_lens.numel() - 1,
                             k_out.shape[0], Hkv, D, bs, NB, block_tables.shape[1],
                             _DT[k_blocks.dtype], _stream(stream)), "pa_gather_kv")
