"""Python binding of libtq, the GB300 TurboQuant KV-cache hot path.

The functions here carry the names of the C ABI in ``include/tq.h`` and only
marshal arguments: every step of encode, decode attention and dequant runs in
the library's CUDA kernels.  PyTorch supplies device memory and streams.
Importing this package fails loudly when ``libtq.so`` has not been built;
there is no CPU fallback.
"""
from __future__ import annotations

import ctypes as C
import os
import re

import torch

__all__ = [
    "TQError", "Codec", "tq_version", "tq_codec_create", "tq_codec_destroy", "tq_codec_info",
    "tq_codec_export", "tq_codec_export_rotation", "tq_codebook_gaussian", "tq_encode", "tq_encode_append",
    "tq_encode_append_kv", "tq_dequant",
    "tq_decode_attend_workspace_bytes", "tq_workspace_init", "tq_decode_attend",
    "tq_get_device_error", "tq_decode_attend_noalloc", "tq_decode_attend_tail",
    "tq_decode_attend_multi", "tq_decode_attend_multi_workspace_bytes", "tq_codec_create_qjl",
    "tq_codec_export_sketch", "tq_encode_qjl", "tq_decode_attend_qjl", "parse_scheme", "bytes_per_vec",
    "LIB_PATH", "KVCache", "TQ_DEVERR_SEQ_LEN", "TQ_DEVERR_POSITION", "TQ_DEVERR_TIMEOUT", "TQ_DEVERR_LAYOUT",
]

# TQ_LIB_VARIANT=timeline loads the profiling build (libtq_timeline.so, see timeline.py)
_LIBNAME = "libtq_timeline.so" if os.environ.get("TQ_LIB_VARIANT") == "timeline" else "libtq.so"
LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), _LIBNAME)
if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'` "
                      "(the CUDA library is required; there is no CPU fallback)")
_lib = C.CDLL(LIB_PATH)

TQ_DEVERR_SEQ_LEN = 1
TQ_DEVERR_POSITION = 2
TQ_DEVERR_TIMEOUT = 4
TQ_DEVERR_LAYOUT = 8

_vp, _i32, _i64, _u64, _sz = C.c_void_p, C.c_int, C.c_int64, C.c_uint64, C.c_size_t
_sig = {
    "tq_version": (_i32, []),
    "tq_status_string": (C.c_char_p, [_i32]),
    "tq_codec_create": (_i32, [_i32, _i32, _u64, C.POINTER(_vp)]),
    "tq_codec_destroy": (None, [_vp]),
    "tq_codec_info": (_i32, [_vp, C.POINTER(_i32), C.POINTER(_i32), C.POINTER(_i32), C.POINTER(_i32),
                             C.POINTER(C.POINTER(C.c_float))]),
    "tq_codec_export": (_i32, [_vp, _vp, _vp, _vp, _vp]),
    "tq_codec_export_rotation": (_i32, [_vp, _vp, _vp]),
    "tq_codebook_gaussian": (_i32, [_i32, _vp, _vp]),
    "tq_encode": (_i32, [_vp, _vp, _i64, _i64, _vp, _i64, _vp, _vp]),
    "tq_encode_append": (_i32, [_vp, _vp, _i32, _i32, _i32, _vp, _i64, _vp, _vp, _vp, _vp]),
    "tq_debug_set_timeline": (_i32, [_vp, _sz]),
    "tq_encode_append_kv": (_i32, [_vp, _vp, _vp, _vp, _i32, _i32, _i32, _vp, _i64, _vp, _vp, _vp, _vp, _vp, _vp]),
    "tq_dequant": (_i32, [_vp, _vp, _vp, _i64, _vp, _vp]),
    "tq_decode_attend_workspace_bytes": (_sz, [_i32, _i32, _i32, _i64, _i32]),
    "tq_workspace_init": (_i32, [_vp, _sz, _vp]),
    "tq_decode_attend": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i64, C.c_float,
                                _vp, _vp, _sz, _vp]),
    "tq_get_device_error": (_i32, [_vp, _vp, C.POINTER(_i32)]),
    "tq_decode_attend_tail": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i64, _vp, _vp, _vp,
                                     _i32, C.c_float, _vp, _vp, C.c_size_t, _vp]),
    "tq_decode_attend_multi_workspace_bytes": (_sz, [_i32, _i32, _i32, _i32, _i64, _i32]),
    "tq_decode_attend_multi": (_i32, [_vp, _vp, _vp, _i32, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i64, _vp, _vp,
                                      _vp, _i32, C.c_float, _vp, _vp, C.c_size_t, _vp]),
    "tq_codec_create_qjl": (_i32, [_i32, _i32, _u64, C.POINTER(_vp)]),
    "tq_codec_export_sketch": (_i32, [_vp, _vp]),
    "tq_encode_qjl": (_i32, [_vp, _vp, _i64, _i64, _vp, _i64, _vp, _vp, _i64, _vp, _vp]),
    "tq_decode_attend_qjl": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i64,
                                    C.c_float, _vp, _vp, _sz, _vp]),
    "tq_cache_create": (_i32, [_vp, _vp, _i32, _i32, _i32, _i64, _i32, C.POINTER(_vp)]),
    "tq_cache_destroy": (None, [_vp]),
    "tq_cache_prefill": (_i32, [_vp, _vp, _vp, _i32, _vp]),
    "tq_cache_decode": (_i32, [_vp, _vp, _vp, _vp, C.c_float, _vp, _vp]),
    "tq_cache_info": (_i32, [_vp, C.POINTER(_i64), C.POINTER(_i64), C.POINTER(_i32), C.POINTER(_sz)]),
    "tq_cache_device_error": (_i32, [_vp, _vp, C.POINTER(_i32)]),
    "tq_decode_attend_noalloc": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i64, C.c_float,
                                        _vp, _vp]),
}
for _name, (_res, _args) in _sig.items():
    _f = getattr(_lib, _name)
    _f.restype = _res
    _f.argtypes = _args


class TQError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = _lib.tq_status_string(status).decode()
        super().__init__(f"{what}: {msg} (status {status})")


def _check(status: int, what: str):
    if status != 0:
        raise TQError(status, what)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dev(t: torch.Tensor, dtype, name: str) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _contig(t: torch.Tensor, name: str):
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def parse_scheme(scheme: str) -> tuple[int, int]:
    """'turbo4' -> (4, 4); 'turbo4v2' -> (4, 2); 'turbo0v4' -> (16, 4): key bits 0 means raw fp16 keys
    ("add TurboQuant KV cache compression", Schemes)."""
    m = re.fullmatch(r"turbo(\d+)(?:v(\d+))?", scheme)
    if not m:
        raise ValueError(f"unknown scheme {scheme!r}")
    kb = int(m.group(1))
    vb = int(m.group(2)) if m.group(2) else kb
    return (16 if kb == 0 else kb), vb


def bytes_per_vec(dim: int, bits: int) -> int:
    return dim * 2 if bits == 16 else dim * bits // 8


def tq_version() -> int:
    return _lib.tq_version()


class Codec:
    """Handle of a tq_codec (rotation + codebook for one (dim, bits, seed))."""

    def __init__(self, handle: int):
        self._h = handle
        d, b, bpv, w = _i32(), _i32(), _i32(), _i32()
        _check(_lib.tq_codec_info(handle, C.byref(d), C.byref(b), C.byref(bpv), C.byref(w), None), "tq_codec_info")
        self.dim, self.bits, self.bytes_per_vec, self.is_wht = d.value, b.value, bpv.value, bool(w.value)

    @property
    def handle(self) -> int:
        return self._h

    def close(self):
        if self._h:
            _lib.tq_codec_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def tq_codec_create(dim: int, bits: int, seed: int) -> Codec:
    h = _vp()
    _check(_lib.tq_codec_create(dim, bits, C.c_uint64(seed), C.byref(h)), "tq_codec_create")
    return Codec(h.value)


def tq_codec_create_qjl(dim: int, bits: int, seed: int) -> Codec:
    """Key codec of the QJL-residual variant: `bits`-bit MSE codes + a dim-row sign sketch."""
    h = _vp()
    _check(_lib.tq_codec_create_qjl(dim, bits, C.c_uint64(seed), C.byref(h)), "tq_codec_create_qjl")
    c = Codec(h.value)
    c.qjl = True
    return c


def tq_codec_export_sketch(codec: Codec):
    import numpy as np
    S = np.zeros((codec.dim, codec.dim), dtype=np.float32)
    _check(_lib.tq_codec_export_sketch(codec.handle, S.ctypes.data), "tq_codec_export_sketch")
    return S


def tq_codec_destroy(codec: Codec):
    codec.close()


def tq_codec_info(codec: Codec) -> dict:
    """dim, bits, bytes_per_vec, is_wht and the centroids (a numpy copy of the codec's host table)."""
    import numpy as np
    ptr = C.POINTER(C.c_float)()
    _check(_lib.tq_codec_info(codec.handle, None, None, None, None, C.byref(ptr)), "tq_codec_info")
    cent = np.ctypeslib.as_array(ptr, shape=(1 << codec.bits,)).copy() if ptr else None
    return dict(dim=codec.dim, bits=codec.bits, bytes_per_vec=codec.bytes_per_vec, is_wht=codec.is_wht,
                centroids=cent)


def tq_codec_export_rotation(codec: Codec) -> dict:
    """The codec's rotation: signs (Walsh-Hadamard) or dense Q, as numpy arrays."""
    import numpy as np
    d = codec.dim
    s = np.zeros(d, dtype=np.int8)
    q = np.zeros((d, d), dtype=np.float32)
    _check(_lib.tq_codec_export_rotation(codec.handle, s.ctypes.data, q.ctypes.data), "tq_codec_export_rotation")
    return dict(signs=s if codec.is_wht else None, dense_q=None if codec.is_wht else q)


def tq_codebook_gaussian(bits: int) -> dict:
    """The Lloyd-Max codebook of N(0,1) with 2^bits levels as the library builds it (host only)."""
    import numpy as np
    n = 1 << min(max(bits, 0), 8)  # buffers for the valid range; the library checks bits
    c = np.zeros(n, dtype=np.float32)
    m = np.zeros(max(n - 1, 1), dtype=np.float64)
    _check(_lib.tq_codebook_gaussian(bits, c.ctypes.data, m.ctypes.data), "tq_codebook_gaussian")
    return dict(centroids=c, midpoints=m[: n - 1])


def tq_codec_export(codec: Codec) -> dict:
    """Host tables of the codec as numpy arrays (signs, dense_q, centroids, midpoints)."""
    import numpy as np
    d = codec.dim
    s = np.zeros(d, dtype=np.int8)
    q = np.zeros((d, d), dtype=np.float32)
    n = 1 << codec.bits if codec.bits != 16 else 1
    c = np.zeros(n, dtype=np.float32)
    m = np.zeros(max(n - 1, 1), dtype=np.float64)
    _check(_lib.tq_codec_export(codec.handle, s.ctypes.data, q.ctypes.data, c.ctypes.data, m.ctypes.data),
           "tq_codec_export")
    return dict(signs=s if codec.is_wht else None, dense_q=None if codec.is_wht else q,
                centroids=c if codec.bits != 16 else None, midpoints=m[: n - 1] if codec.bits != 16 else None)


def tq_encode(codec: Codec, x: torch.Tensor, codes: torch.Tensor, norms: torch.Tensor, stream=None):
    """x [n, dim] fp16 (rows may be strided) -> codes [n, >=bytes_per_vec] uint8, norms [n] fp16."""
    n = x.shape[0]
    if x.dim() != 2 or x.shape[1] != codec.dim or x.stride(1) != 1:
        raise ValueError("x must be [n, dim] with unit inner stride")
    if codes.dim() != 2 or codes.shape[0] != n or codes.stride(1) != 1:
        raise ValueError("codes must be [n, bytes] with unit inner stride")
    if norms.numel() != n:
        raise ValueError("norms must have n elements")
    _check(_lib.tq_encode(codec.handle, _dev(x, torch.float16, "x"), n, x.stride(0),
                          _dev(codes, torch.uint8, "codes"), codes.stride(0), _dev(norms, torch.float16, "norms"),
                          _stream(stream)), "tq_encode")


def tq_encode_qjl(codec: Codec, x: torch.Tensor, codes: torch.Tensor, norms: torch.Tensor, signs: torch.Tensor,
                  rnorms: torch.Tensor, stream=None):
    """tq_encode plus the QJL residual sketch: signs [n, >=dim/8] uint8 (row stride a multiple
    of 4), rnorms [n] fp16."""
    n = x.shape[0]
    if x.dim() != 2 or x.shape[1] != codec.dim or x.stride(1) != 1:
        raise ValueError("x must be [n, dim] with unit inner stride")
    for t, nm in ((codes, "codes"), (signs, "signs")):
        if t.dim() != 2 or t.shape[0] != n or t.stride(1) != 1:
            raise ValueError(f"{nm} must be [n, bytes] with unit inner stride")
    if norms.numel() != n or rnorms.numel() != n:
        raise ValueError("norms / rnorms must have n elements")
    _check(_lib.tq_encode_qjl(codec.handle, _dev(x, torch.float16, "x"), n, x.stride(0),
                              _dev(codes, torch.uint8, "codes"), codes.stride(0), _dev(norms, torch.float16, "norms"),
                              _dev(signs, torch.uint8, "signs"), signs.stride(0),
                              _dev(rnorms, torch.float16, "rnorms"), _stream(stream)), "tq_encode_qjl")


def tq_encode_append(codec: Codec, x: torch.Tensor, start_pos: torch.Tensor, codes: torch.Tensor,
                     norms: torch.Tensor, dev_error: torch.Tensor | None = None, stream=None):
    """x [B, Hkv, T, dim] fp16 -> cache codes [B, Hkv, max_seq, bpv] / norms [B, Hkv, max_seq] at
    positions start_pos[b] + t."""
    B, H, T, d = x.shape
    if d != codec.dim:
        raise ValueError("x last dim must equal codec dim")
    for t, nm in ((x, "x"), (codes, "codes"), (norms, "norms"), (start_pos, "start_pos")):
        _contig(t, nm)
    max_seq = codes.shape[2]
    if tuple(codes.shape) != (B, H, max_seq, codec.bytes_per_vec) or tuple(norms.shape) != (B, H, max_seq):
        raise ValueError("cache shapes do not match")
    err = _dev(dev_error, torch.int32, "dev_error") if dev_error is not None else None
    _check(_lib.tq_encode_append(codec.handle, _dev(x, torch.float16, "x"), B, H, T,
                                 _dev(start_pos, torch.int32, "start_pos"), max_seq,
                                 _dev(codes, torch.uint8, "codes"), _dev(norms, torch.float16, "norms"), err,
                                 _stream(stream)), "tq_encode_append")


def tq_encode_append_kv(ck: Codec, cv: Codec, k: torch.Tensor, v: torch.Tensor, start_pos: torch.Tensor,
                        k_codes: torch.Tensor, k_norms: torch.Tensor, v_codes: torch.Tensor, v_norms: torch.Tensor,
                        dev_error: torch.Tensor | None = None, stream=None):
    """The K and V pending batches [B, Hkv, T, dim] fp16 into their caches in one launch (codes
    [B, Hkv, max_seq, bpv], norms [B, Hkv, max_seq]) at positions start_pos[b] + t."""
    B, H, T, d = k.shape
    if tuple(v.shape) != (B, H, T, d) or d != ck.dim or d != cv.dim:
        raise ValueError("k and v must be [B, Hkv, T, dim] with the codecs' dim")
    for t, nm in ((k, "k"), (v, "v"), (k_codes, "k_codes"), (k_norms, "k_norms"), (v_codes, "v_codes"),
                  (v_norms, "v_norms"), (start_pos, "start_pos")):
        _contig(t, nm)
    max_seq = k_codes.shape[2]
    if (tuple(k_codes.shape) != (B, H, max_seq, ck.bytes_per_vec) or tuple(k_norms.shape) != (B, H, max_seq) or
            tuple(v_codes.shape) != (B, H, max_seq, cv.bytes_per_vec) or tuple(v_norms.shape) != (B, H, max_seq)):
        raise ValueError("cache shapes do not match")
    err = _dev(dev_error, torch.int32, "dev_error") if dev_error is not None else None
    _check(_lib.tq_encode_append_kv(ck.handle, cv.handle, _dev(k, torch.float16, "k"), _dev(v, torch.float16, "v"),
                                    B, H, T, _dev(start_pos, torch.int32, "start_pos"), max_seq,
                                    _dev(k_codes, torch.uint8, "k_codes"), _dev(k_norms, torch.float16, "k_norms"),
                                    _dev(v_codes, torch.uint8, "v_codes"), _dev(v_norms, torch.float16, "v_norms"),
                                    err, _stream(stream)), "tq_encode_append_kv")


def tq_dequant(codec: Codec, codes: torch.Tensor, norms: torch.Tensor, out: torch.Tensor, stream=None):
    """codes [n, bpv] uint8 + norms [n] fp16 -> out [n, dim] fp32."""
    for t, nm in ((codes, "codes"), (norms, "norms"), (out, "out")):
        _contig(t, nm)
    n = norms.numel()
    if codes.numel() != n * codec.bytes_per_vec or out.numel() != n * codec.dim:
        raise ValueError("shape mismatch")
    _check(_lib.tq_dequant(codec.handle, _dev(codes, torch.uint8, "codes"), _dev(norms, torch.float16, "norms"), n,
                           _dev(out, torch.float32, "out"), _stream(stream)), "tq_dequant")


def tq_decode_attend_workspace_bytes(B: int, n_q_heads: int, n_kv_heads: int, max_seq: int, dim: int) -> int:
    return int(_lib.tq_decode_attend_workspace_bytes(B, n_q_heads, n_kv_heads, max_seq, dim))


def tq_workspace_init(workspace: torch.Tensor, stream=None):
    _check(_lib.tq_workspace_init(_dev(workspace, torch.uint8, "workspace"), workspace.numel(), _stream(stream)),
           "tq_workspace_init")


def tq_decode_attend(ck: Codec, cv: Codec, q: torch.Tensor, k: torch.Tensor, k_norms: torch.Tensor | None,
                     v_codes: torch.Tensor, v_norms: torch.Tensor, seq_lens: torch.Tensor, out: torch.Tensor,
                     workspace: torch.Tensor, scale: float | None = None, stream=None):
    """Fused decode attention.  q/out [B, Hq, dim] fp16; k [B, Hkv, S, bpv] uint8 (or [B, Hkv, S, dim] fp16
    for a raw-K codec); norms [B, Hkv, S] fp16; v_codes [B, Hkv, S, bpv] uint8; seq_lens [B] int32."""
    B, Hq, d = q.shape
    Hkv, S = v_codes.shape[1], v_codes.shape[2]
    for t, nm in ((q, "q"), (k, "k"), (v_codes, "v_codes"), (v_norms, "v_norms"), (seq_lens, "seq_lens"),
                  (out, "out"), (workspace, "workspace")):
        _contig(t, nm)
    if ck.bits == 16:
        kp = _dev(k, torch.float16, "k")
        kn = None
    else:
        kp = _dev(k, torch.uint8, "k")
        _contig(k_norms, "k_norms")
        kn = _dev(k_norms, torch.float16, "k_norms")
    if scale is None:
        scale = d ** -0.5
    _check(_lib.tq_decode_attend(ck.handle, cv.handle, _dev(q, torch.float16, "q"), kp, kn,
                                 _dev(v_codes, torch.uint8, "v_codes"), _dev(v_norms, torch.float16, "v_norms"),
                                 _dev(seq_lens, torch.int32, "seq_lens"), B, Hq, Hkv, S, float(scale),
                                 _dev(out, torch.float16, "out"), _dev(workspace, torch.uint8, "workspace"),
                                 workspace.numel(), _stream(stream)), "tq_decode_attend")


def tq_decode_attend_tail(ck: Codec, cv: Codec, q: torch.Tensor, k: torch.Tensor, k_norms: torch.Tensor | None,
                          v_codes: torch.Tensor, v_norms: torch.Tensor, seq_lens: torch.Tensor, k_tail: torch.Tensor,
                          v_tail: torch.Tensor, tail_lens: torch.Tensor, out: torch.Tensor, workspace: torch.Tensor,
                          scale: float | None = None, stream=None):
    """tq_decode_attend plus unencoded fp16 tail tokens in the same softmax: k_tail / v_tail
    [B, Hkv, max_tail, dim] fp16, tail_lens [B] int32 (tokens of the tail used per sequence)."""
    B, Hq, d = q.shape
    Hkv, S = v_codes.shape[1], v_codes.shape[2]
    max_tail = k_tail.shape[2]
    for t, nm in ((q, "q"), (k, "k"), (v_codes, "v_codes"), (v_norms, "v_norms"), (seq_lens, "seq_lens"),
                  (k_tail, "k_tail"), (v_tail, "v_tail"), (tail_lens, "tail_lens"), (out, "out"),
                  (workspace, "workspace")):
        _contig(t, nm)
    if tuple(k_tail.shape) != (B, Hkv, max_tail, d) or tuple(v_tail.shape) != (B, Hkv, max_tail, d):
        raise ValueError("k_tail / v_tail must be [B, Hkv, max_tail, dim]")
    if ck.bits == 16:
        kp = _dev(k, torch.float16, "k")
        kn = None
    else:
        kp = _dev(k, torch.uint8, "k")
        _contig(k_norms, "k_norms")
        kn = _dev(k_norms, torch.float16, "k_norms")
    if scale is None:
        scale = d ** -0.5
    _check(_lib.tq_decode_attend_tail(ck.handle, cv.handle, _dev(q, torch.float16, "q"), kp, kn,
                                      _dev(v_codes, torch.uint8, "v_codes"), _dev(v_norms, torch.float16, "v_norms"),
                                      _dev(seq_lens, torch.int32, "seq_lens"), B, Hq, Hkv, S,
                                      _dev(k_tail, torch.float16, "k_tail"), _dev(v_tail, torch.float16, "v_tail"),
                                      _dev(tail_lens, torch.int32, "tail_lens"), max_tail, float(scale),
                                      _dev(out, torch.float16, "out"), _dev(workspace, torch.uint8, "workspace"),
                                      workspace.numel(), _stream(stream)), "tq_decode_attend_tail")


def tq_decode_attend_multi_workspace_bytes(B: int, n_q_heads: int, n_kv_heads: int, L: int, max_seq: int,
                                           dim: int) -> int:
    return int(_lib.tq_decode_attend_multi_workspace_bytes(B, n_q_heads, n_kv_heads, L, max_seq, dim))


def tq_decode_attend_multi(ck: Codec, cv: Codec, q: torch.Tensor, k: torch.Tensor, k_norms: torch.Tensor | None,
                           v_codes: torch.Tensor, v_norms: torch.Tensor, seq_lens: torch.Tensor, out: torch.Tensor,
                           workspace: torch.Tensor, k_tail: torch.Tensor | None = None,
                           v_tail: torch.Tensor | None = None, tail_lens: torch.Tensor | None = None,
                           scale: float | None = None, stream=None):
    """Causal attention of the last L positions of every sequence: q, out [B, Hq, L, dim] fp16;
    the sequence is its packed tokens then (optionally) its fp16 tail tokens k_tail / v_tail
    [B, Hkv, max_tail, dim] with tail_lens [B] int32 of them in use."""
    B, Hq, L, d = q.shape
    Hkv, S = v_codes.shape[1], v_codes.shape[2]
    for t, nm in ((q, "q"), (k, "k"), (v_codes, "v_codes"), (v_norms, "v_norms"), (seq_lens, "seq_lens"),
                  (out, "out"), (workspace, "workspace")):
        _contig(t, nm)
    if tuple(out.shape) != (B, Hq, L, d):
        raise ValueError("out must be [B, Hq, L, dim]")
    if tail_lens is None:
        if k_tail is not None or v_tail is not None:
            raise ValueError("k_tail / v_tail need tail_lens")
        kt = vt = tl = None
        max_tail = 0
    else:
        for t, nm in ((k_tail, "k_tail"), (v_tail, "v_tail"), (tail_lens, "tail_lens")):
            _contig(t, nm)
        max_tail = k_tail.shape[2]
        if tuple(k_tail.shape) != (B, Hkv, max_tail, d) or tuple(v_tail.shape) != (B, Hkv, max_tail, d):
            raise ValueError("k_tail / v_tail must be [B, Hkv, max_tail, dim]")
        kt, vt = _dev(k_tail, torch.float16, "k_tail"), _dev(v_tail, torch.float16, "v_tail")
        tl = _dev(tail_lens, torch.int32, "tail_lens")
    if ck.bits == 16:
        kp = _dev(k, torch.float16, "k")
        kn = None
    else:
        kp = _dev(k, torch.uint8, "k")
        _contig(k_norms, "k_norms")
        kn = _dev(k_norms, torch.float16, "k_norms")
    if scale is None:
        scale = d ** -0.5
    _check(_lib.tq_decode_attend_multi(ck.handle, cv.handle, _dev(q, torch.float16, "q"), L, kp, kn,
                                       _dev(v_codes, torch.uint8, "v_codes"), _dev(v_norms, torch.float16, "v_norms"),
                                       _dev(seq_lens, torch.int32, "seq_lens"), B, Hq, Hkv, S, kt, vt, tl, max_tail,
                                       float(scale), _dev(out, torch.float16, "out"),
                                       _dev(workspace, torch.uint8, "workspace"), workspace.numel(),
                                       _stream(stream)), "tq_decode_attend_multi")


def tq_decode_attend_qjl(ck: Codec, cv: Codec, q: torch.Tensor, k_codes: torch.Tensor, k_norms: torch.Tensor,
                         k_signs: torch.Tensor, k_rnorms: torch.Tensor, v_codes: torch.Tensor,
                         v_norms: torch.Tensor, seq_lens: torch.Tensor, out: torch.Tensor, workspace: torch.Tensor,
                         scale: float | None = None, stream=None):
    """tq_decode_attend with QJL-sketched keys: k_signs [B, Hkv, S, dim/8] uint8 and
    k_rnorms [B, Hkv, S] fp16 beside the MSE codes and norms."""
    B, Hq, d = q.shape
    Hkv, S = v_codes.shape[1], v_codes.shape[2]
    for t, nm in ((q, "q"), (k_codes, "k_codes"), (k_norms, "k_norms"), (k_signs, "k_signs"),
                  (k_rnorms, "k_rnorms"), (v_codes, "v_codes"), (v_norms, "v_norms"), (seq_lens, "seq_lens"),
                  (out, "out"), (workspace, "workspace")):
        _contig(t, nm)
    if tuple(k_signs.shape) != (B, Hkv, S, d // 8):
        raise ValueError("k_signs must be [B, Hkv, max_seq, dim/8]")
    if scale is None:
        scale = d ** -0.5
    _check(_lib.tq_decode_attend_qjl(ck.handle, cv.handle, _dev(q, torch.float16, "q"),
                                     _dev(k_codes, torch.uint8, "k_codes"), _dev(k_norms, torch.float16, "k_norms"),
                                     _dev(k_signs, torch.uint8, "k_signs"), _dev(k_rnorms, torch.float16, "k_rnorms"),
                                     _dev(v_codes, torch.uint8, "v_codes"), _dev(v_norms, torch.float16, "v_norms"),
                                     _dev(seq_lens, torch.int32, "seq_lens"), B, Hq, Hkv, S, float(scale),
                                     _dev(out, torch.float16, "out"), _dev(workspace, torch.uint8, "workspace"),
                                     workspace.numel(), _stream(stream)), "tq_decode_attend_qjl")


class KVCache:
    """The two-phase KV cache of one layer (tq_cache_*): raw fp16 prefill compressed on the
    first decode step, then per step attend + append with pending tokens kept in fp16 and
    encoded 64 at a time; the first min_tokens tokens of every sequence stay fp16 (sink
    tokens).  Owns its device memory."""

    def __init__(self, ck: Codec, cv: Codec, B: int, n_q_heads: int, n_kv_heads: int, max_seq: int,
                 min_tokens: int = 0):
        h = _vp()
        _check(_lib.tq_cache_create(ck.handle, cv.handle, B, n_q_heads, n_kv_heads, max_seq, min_tokens,
                                    C.byref(h)), "tq_cache_create")
        self._h, self._codecs = h.value, (ck, cv)   # the codecs must outlive the cache
        self.B, self.Hq, self.Hkv, self.dim = B, n_q_heads, n_kv_heads, cv.dim

    def prefill(self, k: torch.Tensor, v: torch.Tensor, stream=None):
        """k, v: fp16 [B, Hkv, T, dim] on the device."""
        T = k.shape[2]
        for t, nm in ((k, "k"), (v, "v")):
            _contig(t, nm)
            if tuple(t.shape) != (self.B, self.Hkv, T, self.dim):
                raise ValueError(f"{nm} must be [B, Hkv, T, dim]")
        _check(_lib.tq_cache_prefill(self._h, _dev(k, torch.float16, "k"), _dev(v, torch.float16, "v"), T,
                                     _stream(stream)), "tq_cache_prefill")

    def decode(self, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, out: torch.Tensor,
               scale: float | None = None, stream=None):
        """q, out: fp16 [B, Hq, dim]; k_new, v_new: fp16 [B, Hkv, dim]."""
        for t, nm in ((q, "q"), (k_new, "k_new"), (v_new, "v_new"), (out, "out")):
            _contig(t, nm)
        if scale is None:
            scale = self.dim ** -0.5
        _check(_lib.tq_cache_decode(self._h, _dev(q, torch.float16, "q"), _dev(k_new, torch.float16, "k_new"),
                                    _dev(v_new, torch.float16, "v_new"), float(scale),
                                    _dev(out, torch.float16, "out"), _stream(stream)), "tq_cache_decode")

    def info(self):
        """(tokens held, packed tokens, pending fp16 tokens, bytes in use)."""
        t, e, p, b = _i64(), _i64(), _i32(), _sz()
        _check(_lib.tq_cache_info(self._h, C.byref(t), C.byref(e), C.byref(p), C.byref(b)), "tq_cache_info")
        return t.value, e.value, p.value, b.value

    def device_error(self, stream=None) -> int:
        code = _i32()
        st = _lib.tq_cache_device_error(self._h, _stream(stream), C.byref(code))
        if st not in (0, 6):
            raise TQError(st, "tq_cache_device_error")
        return code.value

    def close(self):
        if self._h:
            _lib.tq_cache_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def tq_get_device_error(error_word: torch.Tensor, stream=None) -> int:
    """Reads and clears a device error word (a decode workspace or an int32 flag tensor)."""
    code = _i32()
    st = _lib.tq_get_device_error(error_word.data_ptr(), _stream(stream), C.byref(code))
    if st not in (0, 6):
        raise TQError(st, "tq_get_device_error")
    return code.value


def tq_decode_attend_noalloc(ck: Codec, cv: Codec, q: torch.Tensor, k: torch.Tensor, k_norms: torch.Tensor | None,
                             v_codes: torch.Tensor, v_norms: torch.Tensor, seq_lens: torch.Tensor, out: torch.Tensor,
                             scale: float | None = None, stream=None):
    """tq_decode_attend without a workspace, for callers that cannot allocate device memory: the
    split-K scratch is a fixed 8 MiB array inside the library (see include/tq.h)."""
    B, Hq, d = q.shape
    Hkv, S = v_codes.shape[1], v_codes.shape[2]
    for t, nm in ((q, "q"), (k, "k"), (v_codes, "v_codes"), (v_norms, "v_norms"), (seq_lens, "seq_lens"),
                  (out, "out")):
        _contig(t, nm)
    if ck.bits == 16:
        kp, kn = _dev(k, torch.float16, "k"), None
    else:
        kp, kn = _dev(k, torch.uint8, "k"), _dev(k_norms, torch.float16, "k_norms")
    if scale is None:
        scale = d ** -0.5
    _check(_lib.tq_decode_attend_noalloc(ck.handle, cv.handle, _dev(q, torch.float16, "q"), kp, kn,
                                         _dev(v_codes, torch.uint8, "v_codes"), _dev(v_norms, torch.float16, "v_norms"),
                                         _dev(seq_lens, torch.int32, "seq_lens"), B, Hq, Hkv, S, float(scale),
                                         _dev(out, torch.float16, "out"), _stream(stream)), "tq_decode_attend_noalloc")
