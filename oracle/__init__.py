"""CPU oracle for the TurboQuant KV-cache hot path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never links,
loads or calls it, and it shares no code with the CUDA path: the C source
``tq_oracle.c`` builds every table it needs (signs, dense rotation, Lloyd-Max
codebook) itself from (dim, bits, seed).

What it computes, and from which pages (titles and sections):
  * encode (norm, rotation, boundary-count quantisation, LSB-first packing):
    "add TurboQuant KV cache compression" (mlx-swift-lm PR #232), Design;
    VeloxQuant-MLX "How I built VeloxQuant-MLX", Stage 1 / Stage 2 /
    The Bit-Packing Problem; VeloxQuant-MLX RVQ post, The Throughput Problem.
  * Lloyd-Max codebook by numerical integration: "How I built VeloxQuant-MLX",
    The Core Idea.
  * dequant-then-naive-softmax attention: the fused-decode post
    ("anyone still talking about mlx-swift-lm?") fixes what the fused kernel
    must equal.

Parity status: every function is pinned by tests in tests/test_oracle_*.py and
tests/test_codebook.py.  The dense (non-power-of-two) rotation is pinned to
numpy's Householder QR of the same seeded Gaussian (sign-fixed, orthogonal) and,
as applied in encode, to an independent fp64 product z = Q k, the exact norm and
the threshold scale D / sqrt(d).  Which orthogonal matrix (the Gaussian stream,
the QR sign convention) is a reading of ours: the pages print no worked example
of it.
"""
from __future__ import annotations

import ctypes as C
import functools
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tq_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile tq_oracle.c into liboracle.so (plain gcc, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = C.CDLL(build())
            vp, i64, i32, u64, dp = C.c_void_p, C.c_int64, C.c_int, C.c_uint64, C.c_double
            L.orc_splitmix64.argtypes = [u64, i64, vp]
            L.orc_signs.argtypes = [i32, u64, vp]
            L.orc_gaussian.argtypes = [i64, u64, vp]
            L.orc_hadamard.argtypes = [i32, vp]
            L.orc_dense_q.argtypes = [i32, u64, vp]
            L.orc_dense_q.restype = i32
            L.orc_lloyd_max.argtypes = [i32, vp, vp, vp, vp]
            L.orc_lloyd_max.restype = i32
            L.orc_f16_to_f64.argtypes = [C.c_uint16]
            L.orc_f16_to_f64.restype = dp
            L.orc_f64_to_f16.argtypes = [dp]
            L.orc_f64_to_f16.restype = C.c_uint16
            L.orc_pack.argtypes = [vp, i32, i32, vp]
            L.orc_unpack.argtypes = [vp, i32, i32, vp]
            L.orc_codec_new.argtypes = [i32, i32, u64]
            L.orc_codec_new.restype = vp
            L.orc_codec_free.argtypes = [vp]
            L.orc_codec_tables.argtypes = [vp, vp, vp, vp, vp]
            L.orc_encode.argtypes = [vp, vp, i64, i64, vp, i64, vp, vp, vp]
            L.orc_encode.restype = i32
            L.orc_encode_codes.argtypes = [vp, vp, vp, vp, vp]
            L.orc_encode_codes.restype = i32
            L.orc_dequant.argtypes = [vp, vp, i64, vp, i64, vp]
            L.orc_dequant.restype = i32
            L.orc_attention_unit.argtypes = [vp, vp, vp, i32, vp, vp, vp, vp, i64, dp, vp]
            L.orc_attention_unit.restype = i32
            L.orc_attention_unit_tail.argtypes = [vp, vp, vp, i32, vp, vp, vp, vp, i64, vp, vp, i64, dp, vp, vp]
            L.orc_attention_unit_tail.restype = i32
            L.orc_attention_multi_unit.argtypes = [vp, vp, vp, i32, i32, vp, vp, vp, vp, i64, vp, vp, i64,
                                                   dp, vp]
            L.orc_attention_multi_unit.restype = i32
            L.orc_qjl_sketch_copy.argtypes = [i32, u64, vp]
            L.orc_encode_qjl.argtypes = [vp, u64, vp, i64, i64, vp, i64, vp, vp, i64, vp]
            L.orc_encode_qjl.restype = i32
            L.orc_qjl_scores.argtypes = [vp, u64, vp, i32, vp, vp, vp, vp, i64, vp]
            L.orc_qjl_scores.restype = i32
            L.orc_attention_qjl_unit.argtypes = [vp, u64, vp, vp, i32, vp, vp, vp, vp, vp, vp, i64, dp, vp]
            L.orc_attention_qjl_unit.restype = i32
            _lib = L
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"] or a.ndim == 0
    return a.ctypes.data_as(C.c_void_p)


# ---------------------------------------------------------------------------
# Building blocks
# ---------------------------------------------------------------------------
def splitmix64(seed: int, n: int) -> np.ndarray:
    out = np.zeros(n, dtype=np.uint64)
    lib().orc_splitmix64(C.c_uint64(seed), n, _p(out))
    return out


def signs(d: int, seed: int) -> np.ndarray:
    out = np.zeros(d, dtype=np.int8)
    lib().orc_signs(d, C.c_uint64(seed), _p(out))
    return out


def gaussian(n: int, seed: int) -> np.ndarray:
    out = np.zeros(n, dtype=np.float64)
    lib().orc_gaussian(n, C.c_uint64(seed), _p(out))
    return out


def hadamard(d: int) -> np.ndarray:
    out = np.zeros((d, d), dtype=np.int32)
    lib().orc_hadamard(d, _p(out))
    return out


def dense_q(d: int, seed: int) -> np.ndarray:
    out = np.zeros((d, d), dtype=np.float32)
    if lib().orc_dense_q(d, C.c_uint64(seed), _p(out)) != 0:
        raise RuntimeError("dense rotation failed")
    return out


@functools.lru_cache(maxsize=None)
def lloyd_max(bits: int):
    """(c64, c32, midpoints, residual, steps) for N(0,1) with 2**bits levels."""
    n = 1 << bits
    c64 = np.zeros(n, dtype=np.float64)
    c32 = np.zeros(n, dtype=np.float32)
    mid = np.zeros(max(n - 1, 1), dtype=np.float64)
    res = np.zeros(1, dtype=np.float64)
    steps = lib().orc_lloyd_max(bits, _p(c64), _p(c32), _p(mid), _p(res))
    for a in (c64, c32, mid):
        a.setflags(write=False)
    return c64, c32, mid[: n - 1], float(res[0]), int(steps)


def f16_to_f64(bits16: int) -> float:
    return lib().orc_f16_to_f64(C.c_uint16(bits16))


def f64_to_f16(x: float) -> int:
    return int(lib().orc_f64_to_f16(C.c_double(x)))


def pack(codes, d: int, bits: int) -> np.ndarray:
    c = np.ascontiguousarray(codes, dtype=np.int32)
    out = np.zeros((d * bits + 7) // 8, dtype=np.uint8)
    lib().orc_pack(_p(c), d, bits, _p(out))
    return out


def unpack(packed, d: int, bits: int) -> np.ndarray:
    p = np.ascontiguousarray(packed, dtype=np.uint8)
    out = np.zeros(d, dtype=np.int32)
    lib().orc_unpack(_p(p), d, bits, _p(out))
    return out


# ---------------------------------------------------------------------------
# Codec-level oracle
# ---------------------------------------------------------------------------
class Codec:
    """The oracle's own codec for one (dim, bits, seed); bits == 16 is raw fp16."""

    def __init__(self, dim: int, bits: int, seed: int):
        self.dim, self.bits, self.seed = dim, bits, seed
        self.is_wht = dim > 0 and (dim & (dim - 1)) == 0
        self._h = lib().orc_codec_new(dim, bits, C.c_uint64(seed))
        if not self._h:
            raise RuntimeError("oracle codec creation failed")
        self.bytes_per_vec = dim * bits // 8

    def __del__(self):
        h = getattr(self, "_h", None)
        if h and _lib is not None:
            _lib.orc_codec_free(h)
            self._h = None

    def tables(self):
        d = self.dim
        s = np.zeros(d, dtype=np.int8)
        Q = np.zeros((d, d), dtype=np.float32)
        n = 1 << self.bits if self.bits != 16 else 1
        c32 = np.zeros(n, dtype=np.float32)
        mid = np.zeros(max(n - 1, 1), dtype=np.float64)
        lib().orc_codec_tables(self._h, _p(s), _p(Q), _p(c32), _p(mid))
        return dict(signs=s if self.is_wht else None, Q=None if self.is_wht else Q,
                    centroids=c32 if self.bits != 16 else None,
                    midpoints=mid[: n - 1] if self.bits != 16 else None)

    def encode(self, x_f16: np.ndarray):
        """x: [n, d] float16 -> (codes [n, bpv] uint8, norms [n] float16, near_ties, mismatches)."""
        x = np.ascontiguousarray(x_f16, dtype=np.float16).reshape(-1, self.dim)
        n = x.shape[0]
        codes = np.zeros((n, self.bytes_per_vec), dtype=np.uint8)
        norms = np.zeros(n, dtype=np.uint16)
        ties = np.zeros(1, dtype=np.int64)
        mism = np.zeros(1, dtype=np.int64)
        xv = x.view(np.uint16)
        rc = lib().orc_encode(self._h, _p(xv), n, self.dim, _p(codes), self.bytes_per_vec,
                              _p(norms), _p(ties), _p(mism))
        if rc != 0:
            raise RuntimeError("oracle encode failed")
        return codes, norms.view(np.float16), int(ties[0]), int(mism[0])

    def encode_codes(self, x_f16: np.ndarray):
        """One vector -> (integer codes [d], rotated coordinates w [d] (fp64), D)."""
        x = np.ascontiguousarray(x_f16, dtype=np.float16).reshape(self.dim).view(np.uint16)
        codes = np.zeros(self.dim, dtype=np.int32)
        w = np.zeros(self.dim, dtype=np.float64)
        D = np.zeros(1, dtype=np.float64)
        lib().orc_encode_codes(self._h, _p(x), _p(codes), _p(w), _p(D))
        return codes, w, float(D[0])

    # ---- QJL residual sketch (TurboQuantProd): this codec's MSE codes + sign bits ----
    def qjl_sketch(self) -> np.ndarray:
        """The fp32 sketch matrix S [d, d] (rows j) of this codec's seed."""
        S = np.zeros((self.dim, self.dim), dtype=np.float32)
        lib().orc_qjl_sketch_copy(self.dim, C.c_uint64(self.seed), _p(S))
        return S

    def encode_qjl(self, x_f16: np.ndarray):
        """x [n, d] fp16 -> (codes, norms fp16, signs [n, d/8] uint8, residual norms fp16)."""
        x = np.ascontiguousarray(x_f16, dtype=np.float16).reshape(-1, self.dim)
        n, d = x.shape[0], self.dim
        codes = np.zeros((n, self.bytes_per_vec), dtype=np.uint8)
        norms = np.zeros(n, dtype=np.uint16)
        signs = np.zeros((n, d // 8), dtype=np.uint8)
        rn = np.zeros(n, dtype=np.uint16)
        rc = lib().orc_encode_qjl(self._h, C.c_uint64(self.seed), _p(x.view(np.uint16)), n, d, _p(codes),
                                  self.bytes_per_vec, _p(norms), _p(signs), d // 8, _p(rn))
        if rc != 0:
            raise RuntimeError("oracle QJL encode failed")
        return codes, norms.view(np.float16), signs, rn.view(np.float16)

    def qjl_scores(self, q_f16, codes, norms, signs, rnorms) -> np.ndarray:
        """Estimated <q_g, k_n> [G, n] (unscaled) from the stored MSE + QJL fields."""
        q = np.ascontiguousarray(q_f16, dtype=np.float16).reshape(-1, self.dim)
        G, n = q.shape[0], np.asarray(codes).reshape(-1, self.bytes_per_vec).shape[0]
        out = np.zeros((G, n), dtype=np.float64)
        rc = lib().orc_qjl_scores(self._h, C.c_uint64(self.seed), _p(q.view(np.uint16)), G,
                                  _p(np.ascontiguousarray(codes, dtype=np.uint8)),
                                  _p(np.ascontiguousarray(norms, dtype=np.float16).view(np.uint16)),
                                  _p(np.ascontiguousarray(signs, dtype=np.uint8)),
                                  _p(np.ascontiguousarray(rnorms, dtype=np.float16).view(np.uint16)), n, _p(out))
        if rc != 0:
            raise RuntimeError("oracle QJL scores failed")
        return out

    def dequant(self, codes: np.ndarray, norms_f16: np.ndarray) -> np.ndarray:
        c = np.ascontiguousarray(codes, dtype=np.uint8).reshape(-1, self.bytes_per_vec)
        nr = np.ascontiguousarray(norms_f16, dtype=np.float16).reshape(-1).view(np.uint16)
        n = c.shape[0]
        out = np.zeros((n, self.dim), dtype=np.float64)
        if lib().orc_dequant(self._h, _p(c), self.bytes_per_vec, _p(nr), n, _p(out)) != 0:
            raise RuntimeError("oracle dequant failed")
        return out


def attention_unit(ck: Codec, cv: Codec, q_f16: np.ndarray, k, k_norms, v_codes, v_norms,
                   length: int, scale: float, k_tail=None, v_tail=None, return_lse: bool = False):
    """Attention of G query heads [G, d] over one KV head's first `length` tokens,
    followed by the raw fp16 tail tokens k_tail / v_tail [n_tail, d] when given.

    k is packed K codes [>=length, bpv] (with k_norms) or raw fp16 K [>=length, d]
    when ck.bits == 16.  Returns [G, d] float64 (and the [G] log-sum-exp of the
    scaled scores when return_lse).
    """
    q = np.ascontiguousarray(q_f16, dtype=np.float16)
    G = q.shape[0]
    d = cv.dim
    out = np.zeros((G, d), dtype=np.float64)
    if ck.bits == 16:
        kk = np.ascontiguousarray(k, dtype=np.float16).view(np.uint16)
        kn = np.zeros(1, dtype=np.uint16)
    else:
        kk = np.ascontiguousarray(k, dtype=np.uint8)
        kn = np.ascontiguousarray(k_norms, dtype=np.float16).view(np.uint16)
    vc = np.ascontiguousarray(v_codes, dtype=np.uint8)
    vn = np.ascontiguousarray(v_norms, dtype=np.float16).view(np.uint16)
    if k_tail is None:
        kt = vt = np.zeros((1, d), dtype=np.uint16)
        nt = 0
    else:
        kt = np.ascontiguousarray(k_tail, dtype=np.float16).reshape(-1, d).view(np.uint16)
        vt = np.ascontiguousarray(v_tail, dtype=np.float16).reshape(-1, d).view(np.uint16)
        nt = kt.shape[0]
        assert vt.shape[0] == nt
    lse = np.zeros(G, dtype=np.float64)
    rc = lib().orc_attention_unit_tail(ck._h, cv._h, _p(q.view(np.uint16)), G, _p(kk), _p(kn), _p(vc),
                                       _p(vn), int(length), _p(kt), _p(vt), int(nt), float(scale),
                                       _p(out), _p(lse))
    if rc != 0:
        raise RuntimeError("oracle attention failed")
    return (out, lse) if return_lse else out


def attention_multi_unit(ck: Codec, cv: Codec, q_f16: np.ndarray, k, k_norms, v_codes, v_norms,
                         length: int, scale: float, k_tail=None, v_tail=None):
    """Causal attention of the last L positions of one (batch, KV head) unit.

    q_f16 [G, L, d]: the L query rows of each of the G query heads sharing the
    KV head.  The sequence is the first `length` cached tokens followed by the
    raw fp16 tail tokens k_tail / v_tail [n_tail, d]; query l sits at position
    length + n_tail - L + l and sees the tokens up to it.  Returns [G, L, d]
    float64.
    """
    q = np.ascontiguousarray(q_f16, dtype=np.float16)
    G, L, d = q.shape
    assert d == cv.dim
    out = np.zeros((G, L, d), dtype=np.float64)
    if ck.bits == 16:
        kk = np.ascontiguousarray(k, dtype=np.float16).view(np.uint16)
        kn = np.zeros(1, dtype=np.uint16)
    else:
        kk = np.ascontiguousarray(k, dtype=np.uint8)
        kn = np.ascontiguousarray(k_norms, dtype=np.float16).view(np.uint16)
    vc = np.ascontiguousarray(v_codes, dtype=np.uint8)
    vn = np.ascontiguousarray(v_norms, dtype=np.float16).view(np.uint16)
    if k_tail is None:
        kt = vt = np.zeros((1, d), dtype=np.uint16)
        nt = 0
    else:
        kt = np.ascontiguousarray(k_tail, dtype=np.float16).reshape(-1, d).view(np.uint16)
        vt = np.ascontiguousarray(v_tail, dtype=np.float16).reshape(-1, d).view(np.uint16)
        nt = kt.shape[0]
        assert vt.shape[0] == nt
    rc = lib().orc_attention_multi_unit(ck._h, cv._h, _p(q.view(np.uint16)), G, L, _p(kk), _p(kn), _p(vc),
                                        _p(vn), int(length), _p(kt), _p(vt), int(nt), float(scale), _p(out))
    if rc != 0:
        raise RuntimeError("oracle multi-query attention failed")
    return out


def attention_qjl_unit(ck: Codec, cv: Codec, q_f16, k_codes, k_norms, k_signs, k_rnorms, v_codes, v_norms,
                       length: int, scale: float) -> np.ndarray:
    """Decode attention of G query heads [G, d] over `length` keys stored as MSE codes
    + QJL sign sketch + residual norms (scores by the QJL estimator) and MSE-coded
    values.  Returns [G, d] float64."""
    q = np.ascontiguousarray(q_f16, dtype=np.float16)
    G, d = q.shape
    out = np.zeros((G, d), dtype=np.float64)
    rc = lib().orc_attention_qjl_unit(
        ck._h, C.c_uint64(ck.seed), cv._h, _p(q.view(np.uint16)), G,
        _p(np.ascontiguousarray(k_codes, dtype=np.uint8)),
        _p(np.ascontiguousarray(k_norms, dtype=np.float16).view(np.uint16)),
        _p(np.ascontiguousarray(k_signs, dtype=np.uint8)),
        _p(np.ascontiguousarray(k_rnorms, dtype=np.float16).view(np.uint16)),
        _p(np.ascontiguousarray(v_codes, dtype=np.uint8)),
        _p(np.ascontiguousarray(v_norms, dtype=np.float16).view(np.uint16)), int(length), float(scale), _p(out))
    if rc != 0:
        raise RuntimeError("oracle QJL attention failed")
    return out


def attention(ck: Codec, cv: Codec, q, k, k_norms, v_codes, v_norms, seq_lens, scale,
              units=None, threads: int = 1) -> np.ndarray:
    """Whole-batch decode attention.  q [B, Hq, d]; cache tensors [B, Hkv, S, ...].

    Query head h uses KV head h // (Hq // Hkv).  `units` restricts the work to a
    list of (b, kvh) pairs (other outputs stay NaN).  `threads` > 1 runs units on
    a thread pool (ctypes releases the GIL during each call).
    """
    B, Hq, d = q.shape
    Hkv = v_codes.shape[1]
    G = Hq // Hkv
    out = np.full((B, Hq, d), np.nan, dtype=np.float64)
    if units is None:
        units = [(b, h) for b in range(B) for h in range(Hkv)]

    def run(u):
        b, h = u
        L = int(seq_lens[b])
        kk = k[b, h, :max(L, 1)]
        kn = None if ck.bits == 16 else k_norms[b, h, :max(L, 1)]
        out[b, h * G:(h + 1) * G] = attention_unit(ck, cv, q[b, h * G:(h + 1) * G], kk, kn,
                                                   v_codes[b, h, :max(L, 1)],
                                                   v_norms[b, h, :max(L, 1)], L, scale)

    if threads <= 1:
        for u in units:
            run(u)
    else:
        from concurrent.futures import ThreadPoolExecutor
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(run, units))
    return out
