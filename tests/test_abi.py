"""The C-ABI library loads, exports every entry point include/tq.h declares, and
rejects bad arguments on the host before touching a device (no GPU needed)."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tq.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tq_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    path = __graft_entry__.build_library()
    return C.CDLL(path)


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("tq_codec_create", "tq_codec_destroy", "tq_encode", "tq_encode_append", "tq_decode_attend",
              "tq_decode_attend_workspace_bytes", "tq_dequant", "tq_get_device_error"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing


def test_host_side_argument_checks(lib):
    lib.tq_codec_create.argtypes = [C.c_int, C.c_int, C.c_uint64, C.POINTER(C.c_void_p)]
    h = C.c_void_p()
    for dim, bits in [(100, 4), (16, 4), (544, 4), (128, 5), (128, 1), (128, 0)]:
        assert lib.tq_codec_create(dim, bits, 42, C.byref(h)) == 1     # TQ_ERR_INVALID_ARG
    assert lib.tq_codec_create(128, 4, 42, None) == 1
    lib.tq_encode.argtypes = [C.c_void_p, C.c_void_p, C.c_int64, C.c_int64, C.c_void_p, C.c_int64, C.c_void_p,
                              C.c_void_p]
    assert lib.tq_encode(None, None, 10, 128, None, 64, None, None) == 1
    lib.tq_status_string.restype = C.c_char_p
    assert lib.tq_status_string(5) == b"workspace too small"
    assert lib.tq_version() >= 10000


def test_package_binding_loads_and_parses_schemes():
    import quantized_kv_cache_10_gb300 as tq
    assert tq.parse_scheme("turbo4") == (4, 4)
    assert tq.parse_scheme("turbo4v2") == (4, 2)
    assert tq.parse_scheme("turbo0v4") == (16, 4)
    assert tq.parse_scheme("turbo3") == (3, 3)
    with pytest.raises(ValueError):
        tq.parse_scheme("kivi4")
    assert tq.bytes_per_vec(128, 3) == 48 and tq.bytes_per_vec(96, 3) == 36 and tq.bytes_per_vec(128, 16) == 256


def test_host_side_checks_of_the_newer_entry_points(lib):
    vp, i32, i64, u64, sz = C.c_void_p, C.c_int, C.c_int64, C.c_uint64, C.c_size_t
    h = C.c_void_p()
    # QJL codecs: power-of-two dims and 2-4 MSE bits only (checked before any device work)
    lib.tq_codec_create_qjl.argtypes = [i32, i32, u64, C.POINTER(vp)]
    for dim, bits in [(96, 3), (160, 3), (128, 8), (128, 16), (128, 1)]:
        assert lib.tq_codec_create_qjl(dim, bits, 42, C.byref(h)) == 1
    assert lib.tq_codec_create_qjl(128, 3, 42, None) == 1
    lib.tq_codec_export_sketch.argtypes = [vp, vp]
    assert lib.tq_codec_export_sketch(None, None) == 1
    lib.tq_encode_qjl.argtypes = [vp, vp, i64, i64, vp, i64, vp, vp, i64, vp, vp]
    assert lib.tq_encode_qjl(None, None, 4, 128, None, 48, None, None, 16, None, None) == 1
    lib.tq_decode_attend_qjl.argtypes = [vp] * 10 + [i32, i32, i32, i64, C.c_float, vp, vp, sz, vp]
    assert lib.tq_decode_attend_qjl(*([None] * 10), 1, 8, 1, 64, 0.1, None, None, 0, None) == 1
    # several query positions: L outside [1, 4096] is refused by the workspace query and the call
    lib.tq_decode_attend_multi_workspace_bytes.argtypes = [i32, i32, i32, i32, i64, i32]
    lib.tq_decode_attend_multi_workspace_bytes.restype = sz
    for L in (0, -1, 4097):
        assert lib.tq_decode_attend_multi_workspace_bytes(1, 8, 1, L, 64, 128) == 0
    lib.tq_decode_attend_multi.argtypes = [vp, vp, vp, i32] + [vp] * 5 + [i32, i32, i32, i64, vp, vp, vp, i32,
                                                                        C.c_float, vp, vp, sz, vp]
    assert lib.tq_decode_attend_multi(None, None, None, 0, *([None] * 5), 1, 8, 1, 64, None, None, None, 0,
                                      0.1, None, None, 0, None) == 1
    # the K+V pending-batch encode refuses missing codecs before touching a device
    lib.tq_encode_append_kv.argtypes = [vp, vp, vp, vp, i32, i32, i32, vp, i64, vp, vp, vp, vp, vp, vp]
    assert lib.tq_encode_append_kv(None, None, None, None, 1, 8, 64, None, 128, None, None, None, None, None,
                                   None) == 1
    # the cache refuses missing codecs
    lib.tq_cache_create.argtypes = [vp, vp, i32, i32, i32, i64, i32, C.POINTER(vp)]
    assert lib.tq_cache_create(None, None, 1, 8, 1, 64, 0, C.byref(h)) == 1
