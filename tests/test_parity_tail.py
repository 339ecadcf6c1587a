"""Decode attention with unencoded fp16 tail tokens in the same softmax
(tq_decode_attend_tail) against the CPU oracle's attention over the
dequantised cache followed by the raw tail: max-abs <= 2e-3, rel-L2 <= 1e-3."""
import math

import numpy as np
import pytest

import oracle
import tq_inputs
from tq_helpers import check_close, codecs, encode_cache, oracle_codecs, torch_mods

pytestmark = pytest.mark.gpu


def _run(w, lens, tail_lens, max_tail, seed=900):
    torch, tq = torch_mods()
    dev = torch.device("cuda")
    ck, cv = codecs(w)
    ok_k, ok_v = oracle_codecs(w)
    K, V, q = w.kv("k", 1), w.kv("v", 1), w.q()
    kc, kn, vc, vn = encode_cache(w, ck, cv, K, V)
    kt = tq_inputs.fp16_normal(seed, (w.B, w.Hkv, max_tail, w.d))
    vt = tq_inputs.fp16_normal(seed + 1, (w.B, w.Hkv, max_tail, w.d))
    out = torch.empty((w.B, w.Hq, w.d), dtype=torch.float16, device=dev)
    ws = torch.empty(tq.tq_decode_attend_workspace_bytes(w.B, w.Hq, w.Hkv, w.S, w.d), dtype=torch.uint8, device=dev)
    tq.tq_workspace_init(ws)
    tq.tq_decode_attend_tail(ck, cv, torch.from_numpy(q).to(dev), kc, kn, vc, vn,
                             torch.tensor(lens, dtype=torch.int32, device=dev), torch.from_numpy(kt).to(dev),
                             torch.from_numpy(vt).to(dev), torch.tensor(tail_lens, dtype=torch.int32, device=dev),
                             out, ws)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().astype(np.float64)
    ref = np.zeros_like(got)
    G = w.G
    for b in range(w.B):
        L = int(min(max(lens[b], 0), w.S))
        T = int(min(max(tail_lens[b], 0), max_tail))
        for h in range(w.Hkv):
            n = max(L, 1)
            if w.k_bits == 16:
                kk, kkn = K[b, h, :n], None
            else:
                kk, kkn, _, _ = ok_k.encode(K[b, h, :n])
            vcc, vnn, _, _ = ok_v.encode(V[b, h, :n])
            ref[b, h * G:(h + 1) * G] = oracle.attention_unit(
                ok_k, ok_v, q[b, h * G:(h + 1) * G], kk, kkn, vcc, vnn, L, 1 / math.sqrt(w.d),
                kt[b, h, :T], vt[b, h, :T])
    return got, ref, ws


@pytest.mark.parametrize("G", [1, 4, 8])
@pytest.mark.parametrize("kb,vb", [(8, 3), (4, 4), (16, 4), (3, 2)])
def test_tail_small_all_outputs(G, kb, vb):
    w = tq_inputs.Workload("t", B=3, Hq=2 * G, Hkv=2, d=128, S=520, k_bits=kb, v_bits=vb, k_outliers=True)
    got, ref, _ = _run(w, lens=[517, 0, 64], tail_lens=[5, 64, 0], max_tail=64)
    check_close(got, ref, f"tail G={G} K{kb}V{vb}")


@pytest.mark.parametrize("d", [64, 96, 256])
def test_tail_head_dims(d):
    w = tq_inputs.Workload("t", B=2, Hq=8, Hkv=2, d=d, S=384, k_bits=4, v_bits=3, k_outliers=True)
    got, ref, _ = _run(w, lens=[383, 100], tail_lens=[17, 1], max_tail=32)
    check_close(got, ref, f"tail d={d}")


def test_tail_lengths_are_clamped_and_flagged():
    torch, tq = torch_mods()
    w = tq_inputs.Workload("t", B=2, Hq=4, Hkv=2, d=128, S=256, k_bits=4, v_bits=4, k_outliers=False)
    got, ref, ws = _run(w, lens=[200, 50], tail_lens=[-3, 99], max_tail=16)
    assert tq.tq_get_device_error(ws) == tq.TQ_DEVERR_SEQ_LEN
    check_close(got, ref, "tail clamped")


def test_tail_full_size_long_context_sampled():
    # the 32K-token 8-bit K / 3-bit V workload with a 37-token pending tail, units sampled
    torch, tq = torch_mods()
    dev = torch.device("cuda")
    w = tq_inputs.WORKLOADS["c4_long_k8v3"]
    ck, cv = codecs(w)
    ok_k, ok_v = oracle_codecs(w)
    K, V, q = w.kv("k", 8), w.kv("v", 8), w.q()
    kc, kn, vc, vn = encode_cache(w, ck, cv, K, V)
    max_tail, T = 64, 37
    kt = tq_inputs.fp16_normal(31, (w.B, w.Hkv, max_tail, w.d))
    vt = tq_inputs.fp16_normal(32, (w.B, w.Hkv, max_tail, w.d))
    out = torch.empty((w.B, w.Hq, w.d), dtype=torch.float16, device=dev)
    ws = torch.empty(tq.tq_decode_attend_workspace_bytes(w.B, w.Hq, w.Hkv, w.S, w.d), dtype=torch.uint8, device=dev)
    tq.tq_workspace_init(ws)
    lens = w.lengths()
    tq.tq_decode_attend_tail(ck, cv, torch.from_numpy(q).to(dev), kc, kn, vc, vn, torch.from_numpy(lens).to(dev),
                             torch.from_numpy(kt).to(dev), torch.from_numpy(vt).to(dev),
                             torch.full((w.B,), T, dtype=torch.int32, device=dev), out, ws)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().astype(np.float64)
    kcc, knn, vcc, vnn = kc.cpu().numpy(), kn.cpu().numpy(), vc.cpu().numpy(), vn.cpu().numpy()
    G = w.G
    for b, h in [(0, 0), (0, 5)]:
        L = int(lens[b])
        # the GPU-written codes and norms of this unit are the oracle's encoding, bit for bit
        # (so the comparison below is against the oracle's attention over its own cache)
        rkc, rkn, _, mk = ok_k.encode(K[b, h, :L])
        rvc, rvn, _, mv = ok_v.encode(V[b, h, :L])
        assert mk == 0 and mv == 0
        assert np.array_equal(kcc[b, h, :L], rkc) and np.array_equal(vcc[b, h, :L], rvc)
        assert np.array_equal(knn[b, h, :L].view(np.uint16), rkn.view(np.uint16))
        assert np.array_equal(vnn[b, h, :L].view(np.uint16), rvn.view(np.uint16))
        ref = oracle.attention_unit(ok_k, ok_v, q[b, h * G:(h + 1) * G], kcc[b, h, :L], knn[b, h, :L],
                                    vcc[b, h, :L], vnn[b, h, :L], L, 1 / math.sqrt(w.d), kt[b, h, :T], vt[b, h, :T])
        check_close(got[b, h * G:(h + 1) * G], ref, f"c4 tail unit {b},{h}")
