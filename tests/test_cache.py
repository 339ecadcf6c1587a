"""The two-phase KV cache (tq_cache_*): raw fp16 prefill compressed on the first
decode step, then per step attend + append with the pending tokens in fp16,
encoded 64 at a time.  Each checked step is compared with the CPU oracle's
attention over the packed tokens followed by the fp16 ones (pending + new)."""
import math

import numpy as np
import pytest

import oracle
import tq_inputs
from tq_helpers import check_close, codecs, oracle_codecs, torch_mods

pytestmark = pytest.mark.gpu

PB = 64  # pending batch


@pytest.mark.parametrize("kb,vb,G", [(4, 4, 4), (8, 3, 8), (16, 4, 2)])
def test_cache_prefill_then_decode_steps(kb, vb, G):
    torch, tq = torch_mods()
    dev = torch.device("cuda")
    T0, steps = 100, 140
    w = tq_inputs.Workload("t", B=2, Hq=2 * G, Hkv=2, d=128, S=T0 + steps, k_bits=kb, v_bits=vb, k_outliers=True)
    ck, cv = codecs(w)
    ok_k, ok_v = oracle_codecs(w)
    K, V = w.kv("k", 1), w.kv("v", 1)
    cache = tq.KVCache(ck, cv, w.B, w.Hq, w.Hkv, max_seq=512)
    cache.prefill(torch.from_numpy(np.ascontiguousarray(K[:, :, :T0])).to(dev),
                  torch.from_numpy(np.ascontiguousarray(V[:, :, :T0])).to(dev))
    assert cache.info()[:3] == (T0, 0, 0)
    # the oracle's codes of every token (encoding is per vector)
    codes = {}
    for b in range(w.B):
        for h in range(w.Hkv):
            kk = K[b, h] if kb == 16 else ok_k.encode(K[b, h])[:2]
            codes[b, h] = (kk, ok_v.encode(V[b, h])[:2])
    out = torch.empty((w.B, w.Hq, w.d), dtype=torch.float16, device=dev)
    check = {1, 2, 63, 64, 65, 129, 140}
    for s in range(1, steps + 1):
        q = tq_inputs.fp16_normal(1000 + s, (w.B, w.Hq, w.d))
        t_new = T0 + s - 1
        cache.decode(torch.from_numpy(q).to(dev), torch.from_numpy(np.ascontiguousarray(K[:, :, t_new])).to(dev),
                     torch.from_numpy(np.ascontiguousarray(V[:, :, t_new])).to(dev), out)
        E = T0 + PB * ((s - 1) // PB)       # packed tokens seen by this step
        P = (s - 1) % PB                     # pending fp16 tokens before the new one
        if s in check:
            torch.cuda.synchronize()
            got = out.float().cpu().numpy().astype(np.float64)
            ref = np.zeros_like(got)
            for b in range(w.B):
                for h in range(w.Hkv):
                    kk, (vc, vn) = codes[b, h]
                    kc, kn = (kk[:E], None) if kb == 16 else (kk[0][:E], kk[1][:E])
                    ref[b, h * G:(h + 1) * G] = oracle.attention_unit(
                        ok_k, ok_v, q[b, h * G:(h + 1) * G], kc, kn, vc[:E], vn[:E], E, 1 / math.sqrt(w.d),
                        K[b, h, E:E + P + 1], V[b, h, E:E + P + 1])
            check_close(got, ref, f"cache K{kb}V{vb} step {s}")
        tokens, enc, pend, nbytes = cache.info()
        assert tokens == T0 + s
        assert enc == T0 + PB * (s // PB) and pend == s % PB
    assert cache.device_error() == 0
    per_tok = (w.d * kb // 8 + (0 if kb == 16 else 2)) + (w.d * vb // 8 + 2)
    assert nbytes == w.B * w.Hkv * (enc * per_tok + pend * w.d * 4)


def test_cache_refuses_overflow_and_late_prefill():
    torch, tq = torch_mods()
    dev = torch.device("cuda")
    w = tq_inputs.Workload("t", B=1, Hq=4, Hkv=1, d=64, S=16, k_bits=4, v_bits=4, k_outliers=False)
    ck, cv = codecs(w)
    cache = tq.KVCache(ck, cv, 1, 4, 1, max_seq=16)
    kv = torch.from_numpy(w.kv("k", 1)).to(dev)
    cache.prefill(kv[:, :, :10].contiguous(), kv[:, :, :10].contiguous())
    q = torch.zeros((1, 4, 64), dtype=torch.float16, device=dev)
    new = torch.zeros((1, 1, 64), dtype=torch.float16, device=dev)
    out = torch.empty_like(q)
    for _ in range(6):
        cache.decode(q, new, new, out)
    with pytest.raises(tq.TQError):
        cache.decode(q, new, new, out)          # 16 tokens held: full
    with pytest.raises(tq.TQError):
        cache.prefill(kv[:, :, :2].contiguous(), kv[:, :, :2].contiguous())


@pytest.mark.parametrize("kb,vb,G,T0,N", [(8, 3, 4, 40, 16), (4, 2, 2, 5, 16), (16, 4, 2, 30, 8)])
def test_cache_sink_tokens_stay_fp16(kb, vb, G, T0, N):
    # The first N tokens of every sequence stay fp16 for good (turboquant-mlx guide "KV
    # cache compression", --kv-min-tokens); the rest follow the two-phase scheme.  Each
    # checked step is compared with the oracle's attention over the packed tokens and the
    # fp16 ones (sinks, pending, the new token).  T0 < N: decode tokens fill the sinks first.
    torch, tq = torch_mods()
    dev = torch.device("cuda")
    steps = 150
    w = tq_inputs.Workload("t", B=2, Hq=2 * G, Hkv=2, d=128, S=T0 + steps, k_bits=kb, v_bits=vb, k_outliers=True)
    ck, cv = codecs(w)
    ok_k, ok_v = oracle_codecs(w)
    K, V = w.kv("k", 1), w.kv("v", 1)
    cache = tq.KVCache(ck, cv, w.B, w.Hq, w.Hkv, max_seq=512, min_tokens=N)
    cache.prefill(torch.from_numpy(np.ascontiguousarray(K[:, :, :T0])).to(dev),
                  torch.from_numpy(np.ascontiguousarray(V[:, :, :T0])).to(dev))
    codes = {}
    for b in range(w.B):
        for h in range(w.Hkv):
            kk = K[b, h] if kb == 16 else ok_k.encode(K[b, h])[:2]
            codes[b, h] = (kk, ok_v.encode(V[b, h])[:2])
    sinks, enc, pend = min(N, T0), T0 - min(N, T0), 0      # the cache's own counters, step by step
    out = torch.empty((w.B, w.Hq, w.d), dtype=torch.float16, device=dev)
    check = {1, 2, 11, 12, 13, 64, 65, 66, 76, 77, 129, 150}
    for s in range(1, steps + 1):
        q = tq_inputs.fp16_normal(2000 + s, (w.B, w.Hq, w.d))
        n = T0 + s - 1
        assert n == sinks + enc + pend
        cache.decode(torch.from_numpy(q).to(dev), torch.from_numpy(np.ascontiguousarray(K[:, :, n])).to(dev),
                     torch.from_numpy(np.ascontiguousarray(V[:, :, n])).to(dev), out)
        if s in check:
            torch.cuda.synchronize()
            got = out.float().cpu().numpy().astype(np.float64)
            ref = np.zeros_like(got)
            pk = slice(sinks, sinks + enc)                     # packed token positions
            for b in range(w.B):
                for h in range(w.Hkv):
                    kk, (vc, vn) = codes[b, h]
                    if enc == 0:                                # no packed token: a dummy row, length 0
                        pk0 = slice(0, 1)
                    else:
                        pk0 = pk
                    kc, kn = (kk[pk0], None) if kb == 16 else (kk[0][pk0], kk[1][pk0])
                    tail = np.r_[0:sinks, sinks + enc:n + 1]     # sinks, pending, the new token
                    ref[b, h * G:(h + 1) * G] = oracle.attention_unit(
                        ok_k, ok_v, q[b, h * G:(h + 1) * G], kc, kn, vc[pk0], vn[pk0], enc, 1 / math.sqrt(w.d),
                        K[b, h, tail], V[b, h, tail])
            check_close(got, ref, f"cache sinks N={N} T0={T0} K{kb}V{vb} step {s}")
        if sinks < N:
            sinks += 1
        else:
            pend += 1
            if pend == PB:
                enc, pend = enc + PB, 0
        tokens, e, p, nbytes = cache.info()
        assert (tokens, e, p) == (sinks + enc + pend, enc, pend)
    assert cache.device_error() == 0
    per_tok = (w.d * kb // 8 + (0 if kb == 16 else 2)) + (w.d * vb // 8 + 2)
    assert nbytes == w.B * w.Hkv * (enc * per_tok + (sinks + pend) * w.d * 4)
