"""Seeded synthetic inputs for the TurboQuant hot path (tests and bench).

This module holds none of the method's arithmetic: it only draws the fp16
K/V/q tensors, the outlier channels and the ragged lengths that stand in for
the pages' model workloads (Llama-3.2-3B / Qwen3-8B / Mistral-7B style
attention layers: 24/8 or 32/8 or 64/8 heads, head_dim 128).

Generator: SplitMix64 (Steele, Lea, Flood 2014) in counter form, output i of
a stream with seed s is mix(s + (i + 1) * 0x9E3779B97F4A7C15); standard
normals by Box-Muller on consecutive output pairs (u1 = (x0 >> 11 + 1) 2^-53,
u2 = (x1 >> 11) 2^-53).  Every (tensor, batch, kv-head) slice has its own
stream so any slice can be regenerated alone.  Values are drawn in fp64,
rounded to fp32, outlier channels scaled by 8 in fp32, then rounded to fp16.
"""
from __future__ import annotations

import dataclasses
import math
from concurrent.futures import ThreadPoolExecutor

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def splitmix64(seed: int, n: int, start: int = 0) -> np.ndarray:
    """Outputs start .. start+n-1 of the SplitMix64 stream with the given seed."""
    with np.errstate(over="ignore"):
        i = np.arange(start + 1, start + n + 1, dtype=np.uint64)
        return _mix(np.uint64(seed & (2**64 - 1)) + i * GAMMA)


def stream_seed(seed: int, *ids: int) -> int:
    """Seed of a sub-stream: fold the ids into the seed with the SplitMix64 finaliser."""
    h = np.array([seed & (2**64 - 1)], dtype=np.uint64)
    with np.errstate(over="ignore"):
        for v in ids:
            h = _mix(h ^ np.uint64((v + 0x632BE59BD9B4E019) & (2**64 - 1)))
    return int(h[0])


def normal(seed: int, n: int) -> np.ndarray:
    """n standard normals (fp64) by Box-Muller from one SplitMix64 stream."""
    m = (n + 1) // 2
    x = splitmix64(seed, 2 * m)
    u1 = ((x[0::2] >> np.uint64(11)) + np.uint64(1)).astype(np.float64) * 2.0**-53
    u2 = (x[1::2] >> np.uint64(11)).astype(np.float64) * 2.0**-53
    r = np.sqrt(-2.0 * np.log(u1))
    out = np.empty(2 * m, dtype=np.float64)
    out[0::2] = r * np.cos(2.0 * math.pi * u2)
    out[1::2] = r * np.sin(2.0 * math.pi * u2)
    return out[:n]


def permutation(seed: int, n: int) -> np.ndarray:
    """Fisher-Yates shuffle of range(n) driven by SplitMix64(seed)."""
    p = np.arange(n)
    x = splitmix64(seed, n)
    for i in range(n - 1, 0, -1):
        j = int(x[n - 1 - i] % np.uint64(i + 1))
        p[i], p[j] = p[j], p[i]
    return p


def outlier_channels(d: int, seed: int = 0) -> np.ndarray:
    """d/32 channels (4 at d=128, 3 at d=96) picked by a seeded permutation."""
    return np.sort(permutation(seed + 1, d)[: d // 32])


def fp16_normal(seed: int, shape, outliers=None, scale: float = 8.0) -> np.ndarray:
    z = normal(seed, int(np.prod(shape))).astype(np.float32).reshape(shape)
    if outliers is not None and len(outliers):
        z[..., outliers] *= np.float32(scale)
    return z.astype(np.float16)


# Tensor ids for stream_seed.
Q_ID, K_ID, V_ID, LEN_ID, NEWK_ID, NEWV_ID, ENC_ID = 1, 2, 3, 4, 5, 6, 7


@dataclasses.dataclass(frozen=True)
class Workload:
    """One decode-attention layer workload."""
    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    S: int                 # max_seq (cache capacity per sequence)
    k_bits: int            # 16 = raw fp16 keys
    v_bits: int
    k_outliers: bool
    ragged: tuple | None = None   # (lo, hi) inclusive length range, else every length = S
    seed: int = 0
    rot_seed: int = 42
    len_seed: int = 1

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    def lengths(self) -> np.ndarray:
        if self.ragged is None:
            return np.full(self.B, self.S, dtype=np.int32)
        lo, hi = self.ragged
        x = splitmix64(self.len_seed, self.B)
        return (lo + (x % np.uint64(hi - lo + 1)).astype(np.int64)).astype(np.int32)

    def outliers(self):
        return outlier_channels(self.d, self.seed) if self.k_outliers else None

    def q(self) -> np.ndarray:
        return fp16_normal(stream_seed(self.seed, Q_ID), (self.B, self.Hq, self.d))

    def k_slice(self, b: int, h: int, n: int | None = None) -> np.ndarray:
        n = self.S if n is None else n
        return fp16_normal(stream_seed(self.seed, K_ID, b, h), (n, self.d), self.outliers())

    def v_slice(self, b: int, h: int, n: int | None = None) -> np.ndarray:
        n = self.S if n is None else n
        return fp16_normal(stream_seed(self.seed, V_ID, b, h), (n, self.d))

    def kv(self, which: str, threads: int = 8) -> np.ndarray:
        """Full [B, Hkv, S, d] fp16 K or V (slices generated on a thread pool)."""
        out = np.empty((self.B, self.Hkv, self.S, self.d), dtype=np.float16)
        f = self.k_slice if which == "k" else self.v_slice

        def run(bh):
            b, h = bh
            out[b, h] = f(b, h)

        units = [(b, h) for b in range(self.B) for h in range(self.Hkv)]
        if threads <= 1:
            for u in units:
                run(u)
        else:
            with ThreadPoolExecutor(threads) as ex:
                list(ex.map(run, units))
        return out

    def packed_kv_bytes(self) -> int:
        """Bytes of packed cache the decode reads: sum_b len_b * Hkv * (bytes_K + bytes_V), norms included."""
        kb = self.d * 2 if self.k_bits == 16 else self.d * self.k_bits // 8 + 2
        vb = self.d * self.v_bits // 8 + 2
        return int(self.lengths().astype(np.int64).sum()) * self.Hkv * (kb + vb)


# The five workloads (tiny; Llama-3.2-3B-shaped; asymmetric ragged; 32K long
# context; head_dim 256 at batch 32) and the head_dim-96 variant of the 32K one.
WORKLOADS = {
    "c1_tiny": Workload("c1_tiny", 1, 1, 1, 64, 256, 4, 4, False),
    "c2_llama3b": Workload("c2_llama3b", 1, 24, 8, 128, 4096, 4, 4, True),
    "c3_turbo4v2_ragged": Workload("c3_turbo4v2_ragged", 8, 32, 8, 128, 8192, 4, 2, True, ragged=(1024, 8192)),
    "c4_long_k8v3": Workload("c4_long_k8v3", 1, 64, 8, 128, 32768, 8, 3, True),
    "c4_long_k8v3_d96": Workload("c4_long_k8v3_d96", 1, 64, 8, 96, 32768, 8, 3, True),
    "c5_turbo0v4_d256": Workload("c5_turbo0v4_d256", 32, 32, 8, 256, 16384, 16, 4, False),
    "c5_turbo3_d256": Workload("c5_turbo3_d256", 32, 32, 8, 256, 16384, 3, 3, False),
}

# Encode-throughput sweep of the head_dim-256 workload: 1 .. 2^20 vectors.
ENCODE_SWEEP = [4**i for i in range(11)]
