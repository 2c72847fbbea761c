"""The C-ABI library builds, loads on a machine without a GPU, and exports every call that
include/pa.h declares.  No compute call is made here."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    with open(os.path.join(ROOT, "include", "pa.h")) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z_0-9]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_31_gb300 import _build

    path = _build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_boundary():
    names = _declared()
    for want in ("pa_reshape_and_cache", "pa_varlen_forward", "pa_decode_splitkv",
                 "pa_decode_splitkv_partials", "pa_decode_splitkv_reduce",
                 "pa_merge_attn_states", "pa_gather_kv", "pa_slot_mapping", "pa_device_status"):
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_binding_covers_the_header(lib):
    from paged_kv_cache_31_gb300 import binding

    assert sorted(binding.EXPORTED) == _declared()
    assert binding.version() >= 100
    assert binding.status_string(binding.PA_EINVAL) == "PA_EINVAL"


def test_host_side_argument_errors_need_no_gpu(lib):
    """Shape and argument errors are returned before anything touches the device."""
    from paged_kv_cache_31_gb300 import binding as b

    L = b._lib
    # heads not a multiple of kv heads
    st = L.pa_varlen_forward(None, None, None, None, None, None, None, None, 1, 1, 6, 4, 128, 16,
                             8, 1, b.PA_BF16, b.PA_BF16, 1.0, 1, 0, None, 0, None)
    assert st == b.PA_ESHAPE
    # unsupported dtype
    st = L.pa_varlen_forward(None, None, None, None, None, None, None, None, 1, 1, 8, 4, 128, 16,
                             8, 1, 7, b.PA_BF16, 1.0, 1, 0, None, 0, None)
    assert st == b.PA_EUNSUPPORTED
    # missing pointers
    st = L.pa_varlen_forward(None, None, None, None, None, None, None, None, 1, 1, 8, 4, 128, 16,
                             8, 1, b.PA_BF16, b.PA_BF16, 1.0, 1, 0, None, 0, None)
    assert st == b.PA_EINVAL
    st = L.pa_reshape_and_cache(None, None, None, None, None, 4, 0, 128, 16, 8, b.PA_BF16, None)
    assert st == b.PA_ESHAPE
    st = L.pa_merge_attn_states(None, None, None, None, None, None, 4, 8, 128, -1, b.PA_F32, None)
    assert st == b.PA_EINVAL
    st = L.pa_decode_splitkv_partials(None, None, None, None, None, None, None, None, 2, 8, 2, 128,
                                      16, 64, 8, 500, 4, b.PA_BF16, b.PA_BF16, 1.0, 0, None)
    assert st == b.PA_EUNSUPPORTED  # partition not a multiple of the block size
    # empty batches are a no-op
    assert L.pa_varlen_forward(None, None, None, None, None, None, None, None, 0, 0, 8, 4, 128, 16,
                               8, 1, b.PA_BF16, b.PA_BF16, 1.0, 1, 0, None, 0, None) == b.PA_OK
    # workspace size grows with the batch and is 256-byte granular
    a = b.pa_varlen_forward_workspace_size(4, 27, 4, 2, 64, 4, 16)
    c = b.pa_varlen_forward_workspace_size(256, 4344, 32, 8, 128, 512, 16)
    assert a % 256 == 0 and c % 256 == 0 and c > a > 0


def test_host_side_errors_of_the_extended_calls(lib):
    """The extended entry points' argument errors, also returned before any device work."""
    from paged_kv_cache_31_gb300 import binding as b

    L = b._lib
    fake = ctypes.c_void_p(16)  # never dereferenced: every case below returns first
    # pa_varlen_forward_ex: unknown flag bits, non-positive / non-finite scales
    for ks, vs, flags in ((1.0, 1.0, 2), (0.0, 1.0, 0), (1.0, -1.0, 0), (float("inf"), 1.0, 0),
                          (float("nan"), 1.0, 0)):
        st = L.pa_varlen_forward_ex(None, None, None, None, None, None, None, None, 0, 0, 8, 4,
                                    128, 16, 8, 1, b.PA_BF16, b.PA_BF16, 1.0, 1, 0, None, None,
                                    ks, vs, flags, None, 0, None)
        assert st == b.PA_EINVAL, (ks, vs, flags)
    # fp8 is a pool type only
    st = L.pa_varlen_forward_ex(None, None, None, None, None, None, None, None, 0, 0, 8, 4, 128,
                                16, 8, 1, b.PA_FP8_E4M3, b.PA_FP8_E4M3, 1.0, 1, 0, None, None,
                                1.0, 1.0, 0, None, 0, None)
    assert st == b.PA_EUNSUPPORTED
    # pa_reshape_and_cache_ex: fp8 new rows are not a source type; bad scales
    st = L.pa_reshape_and_cache_ex(None, None, None, None, None, 0, 2, 128, 16, 8, b.PA_FP8_E4M3,
                                   b.PA_FP8_E4M3, 1.0, 1.0, None)
    assert st == b.PA_EUNSUPPORTED
    st = L.pa_reshape_and_cache_ex(None, None, None, None, None, 0, 2, 128, 16, 8, b.PA_BF16,
                                   b.PA_FP8_E4M3, 0.0, 1.0, None)
    assert st == b.PA_EINVAL
    # slots are int32: a pool of more than 2^31 - 1 slots is refused
    big_nb = (1 << 31) // 16 + 1
    st = L.pa_slot_mapping(fake, fake, fake, 1, 1, 1, 16, big_nb, fake, None)
    assert st == b.PA_EUNSUPPORTED
    st = L.pa_slot_mapping_and_cache(fake, fake, fake, fake, fake, fake, fake, 1, 1, 1, 2, 128,
                                     16, big_nb, b.PA_BF16, fake, None)
    assert st == b.PA_EUNSUPPORTED
    st = L.pa_cache_and_attend(fake, fake, fake, fake, fake, fake, fake, fake, fake, fake, 1, 1, 8,
                               2, 128, 16, big_nb, 1, b.PA_BF16, b.PA_BF16, 1.0, 1, 0, fake, fake,
                               1 << 20, None)
    assert st == b.PA_EUNSUPPORTED
    # missing new rows
    st = L.pa_cache_and_attend(None, None, fake, fake, fake, fake, fake, fake, fake, fake, 1, 1, 8,
                               2, 128, 16, 8, 1, b.PA_BF16, b.PA_BF16, 1.0, 1, 0, None, fake,
                               1 << 20, None)
    assert st == b.PA_EINVAL
    # empty steps are a no-op
    assert L.pa_slot_mapping_and_cache(None, None, None, None, None, None, None, 0, 0, 0, 2, 128,
                                       16, 8, b.PA_BF16, None, None) == b.PA_OK


def test_host_side_errors_of_the_per_head_calls(lib):
    """The per kv head scale calls check shapes, dtypes and pointers on the host like the
    per-pool ones (the scales themselves are device arrays, validated on the device)."""
    from paged_kv_cache_31_gb300 import binding as b

    L = b._lib
    fake = ctypes.c_void_p(16)  # never dereferenced: every case below returns first
    # scatter: fp8 is not a source type; a negative kv head count; missing rows
    assert L.pa_reshape_and_cache_per_head(None, None, None, None, None, 1, 2, 128, 16, 8,
                                           b.PA_FP8_E4M3, b.PA_FP8_E4M3, fake, fake,
                                           None) == b.PA_EUNSUPPORTED
    assert L.pa_reshape_and_cache_per_head(fake, fake, fake, fake, fake, 1, -2, 128, 16, 8,
                                           b.PA_BF16, b.PA_FP8_E4M3, fake, fake,
                                           None) == b.PA_ESHAPE
    assert L.pa_reshape_and_cache_per_head(None, None, fake, fake, fake, 1, 2, 128, 16, 8,
                                           b.PA_BF16, b.PA_FP8_E4M3, fake, fake,
                                           None) == b.PA_EINVAL
    assert L.pa_reshape_and_cache_per_head(None, None, None, None, None, 0, 2, 128, 16, 8,
                                           b.PA_BF16, b.PA_FP8_E4M3, fake, fake,
                                           None) == b.PA_OK  # nothing to write
    # varlen: unknown flag bits; a GQA group that does not divide; fp8 queries
    st = L.pa_varlen_forward_per_head(None, None, None, None, None, None, None, None, 0, 0, 8, 4,
                                      128, 16, 8, 1, b.PA_BF16, b.PA_BF16, 1.0, 1, 0, None, None,
                                      fake, fake, 2, None, 0, None)
    assert st == b.PA_EINVAL
    st = L.pa_varlen_forward_per_head(None, None, None, None, None, None, None, None, 0, 0, 8, 3,
                                      128, 16, 8, 1, b.PA_BF16, b.PA_BF16, 1.0, 1, 0, None, None,
                                      fake, fake, 0, None, 0, None)
    assert st == b.PA_ESHAPE
    st = L.pa_varlen_forward_per_head(None, None, None, None, None, None, None, None, 0, 0, 8, 4,
                                      128, 16, 8, 1, b.PA_FP8_E4M3, b.PA_FP8_E4M3, 1.0, 1, 0,
                                      None, None, fake, fake, 0, None, 0, None)
    assert st == b.PA_EUNSUPPORTED
    # split-KV partials: a partition size that is not a multiple of the block size
    st = L.pa_decode_splitkv_partials_per_head(fake, fake, fake, fake, fake, fake, fake, fake, 1,
                                               8, 4, 128, 16, 8, 1, 500, 4, b.PA_BF16,
                                               b.PA_BF16, 1.0, 0, fake, fake, None)
    assert st == b.PA_EUNSUPPORTED
