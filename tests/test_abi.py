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
