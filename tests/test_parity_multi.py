"""Attention of several query positions per head (tq_decode_attend_multi:
chunked prefill, speculative verification) against the CPU oracle's causal
attention over the dequantised cache followed by the raw fp16 tail:
max-abs <= 2e-3, rel-L2 <= 1e-3."""
import math

import numpy as np
import pytest

import oracle
import tq_inputs
from tq_helpers import ATOL, check_close, codecs, encode_cache, oracle_codecs, torch_mods

pytestmark = pytest.mark.gpu

# The first rows of a chunk attend to one or a few tokens, so their outputs are
# dequantised values (up to ~4 in magnitude) whose fp16 store alone is off by up to
# ~1e-3; the kernel's own error (beyond that rounding) keeps a 2x margin to the bound.
MARGIN = ATOL / 2


def _run(w, L, lens, tail_lens=None, max_tail=0, seed=700):
    torch, tq = torch_mods()
    dev = torch.device("cuda")
    ck, cv = codecs(w)
    ok_k, ok_v = oracle_codecs(w)
    K, V = w.kv("k", 1), w.kv("v", 1)
    q = tq_inputs.fp16_normal(seed, (w.B, w.Hq, L, w.d))
    kc, kn, vc, vn = encode_cache(w, ck, cv, K, V)
    kt = vt = None
    tail = {}
    if tail_lens is not None:
        kt = tq_inputs.fp16_normal(seed + 1, (w.B, w.Hkv, max_tail, w.d))
        vt = tq_inputs.fp16_normal(seed + 2, (w.B, w.Hkv, max_tail, w.d))
        tail = dict(k_tail=torch.from_numpy(kt).to(dev), v_tail=torch.from_numpy(vt).to(dev),
                    tail_lens=torch.tensor(tail_lens, dtype=torch.int32, device=dev))
    out = torch.empty((w.B, w.Hq, L, w.d), dtype=torch.float16, device=dev)
    ws = torch.empty(tq.tq_decode_attend_multi_workspace_bytes(w.B, w.Hq, w.Hkv, L, w.S, w.d), dtype=torch.uint8,
                     device=dev)
    tq.tq_workspace_init(ws)
    tq.tq_decode_attend_multi(ck, cv, torch.from_numpy(q).to(dev), kc, kn, vc, vn,
                              torch.tensor(lens, dtype=torch.int32, device=dev), out, ws, **tail)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().astype(np.float64)
    ref = np.zeros_like(got)
    G = w.G
    for b in range(w.B):
        n_b = int(min(max(lens[b], 0), w.S))
        T = 0 if tail_lens is None else int(min(max(tail_lens[b], 0), max_tail))
        for h in range(w.Hkv):
            n = max(n_b, 1)
            if w.k_bits == 16:
                kk, kkn = K[b, h, :n], None
            else:
                kk, kkn, _, _ = ok_k.encode(K[b, h, :n])
            vcc, vnn, _, _ = ok_v.encode(V[b, h, :n])
            ref[b, h * G:(h + 1) * G] = oracle.attention_multi_unit(
                ok_k, ok_v, q[b, h * G:(h + 1) * G], kk, kkn, vcc, vnn, n_b, 1 / math.sqrt(w.d),
                kt[b, h, :T] if T else None, vt[b, h, :T] if T else None)
    return got, ref, ws


@pytest.mark.parametrize("G,L", [(1, 2), (4, 2), (8, 4), (2, 7), (8, 5), (3, 10)])
@pytest.mark.parametrize("kb,vb", [(8, 3), (4, 4), (16, 4), (3, 2)])
def test_multi_small_all_outputs(G, L, kb, vb):
    # lengths: a long sequence, an empty one, one shorter than L, one ending inside a tile
    w = tq_inputs.Workload("m", B=4, Hq=2 * G, Hkv=2, d=128, S=520, k_bits=kb, v_bits=vb, k_outliers=True)
    got, ref, ws = _run(w, L, lens=[517, 0, 3, 64], tail_lens=[1, 4, 0, 20], max_tail=32)
    check_close(got, ref, f"multi G={G} L={L} K{kb}V{vb}", beyond_store_max=MARGIN)
    _, tq = torch_mods()
    assert tq.tq_get_device_error(ws) == 0


@pytest.mark.parametrize("L", [1, 3, 16])
def test_multi_without_tail_masks_inside_the_cache(L):
    # no tail: the causal mask falls on the last L packed tokens
    w = tq_inputs.Workload("m", B=2, Hq=8, Hkv=2, d=128, S=384, k_bits=8, v_bits=3, k_outliers=True)
    got, ref, _ = _run(w, L, lens=[384, 130])
    check_close(got, ref, f"multi no tail L={L}", beyond_store_max=MARGIN)


@pytest.mark.parametrize("d,kb", [(64, 4), (96, 8), (256, 3), (256, 16), (160, 4)])
def test_multi_head_dims(d, kb):
    # d 160 has no tensor-core instantiation: the SIMT kernel runs
    w = tq_inputs.Workload("m", B=2, Hq=8, Hkv=2, d=d, S=256, k_bits=kb, v_bits=3, k_outliers=True)
    got, ref, _ = _run(w, 3, lens=[255, 77], tail_lens=[1, 9], max_tail=16)
    check_close(got, ref, f"multi d={d} K{kb}", beyond_store_max=MARGIN)


def test_multi_l1_is_the_decode_call():
    # L == 1 through the multi entry point runs the same kernels as tq_decode_attend_tail
    torch, tq = torch_mods()
    dev = torch.device("cuda")
    w = tq_inputs.Workload("m", B=2, Hq=16, Hkv=2, d=128, S=512, k_bits=8, v_bits=3, k_outliers=True)
    ck, cv = codecs(w)
    kc, kn, vc, vn = encode_cache(w, ck, cv, w.kv("k", 1), w.kv("v", 1))
    q = torch.from_numpy(tq_inputs.fp16_normal(5, (w.B, w.Hq, w.d))).to(dev)
    kt = torch.from_numpy(tq_inputs.fp16_normal(6, (w.B, w.Hkv, 8, w.d))).to(dev)
    vt = torch.from_numpy(tq_inputs.fp16_normal(7, (w.B, w.Hkv, 8, w.d))).to(dev)
    lens = torch.tensor([500, 17], dtype=torch.int32, device=dev)
    tl = torch.tensor([8, 2], dtype=torch.int32, device=dev)
    ws = torch.empty(tq.tq_decode_attend_multi_workspace_bytes(w.B, w.Hq, w.Hkv, 1, w.S, w.d), dtype=torch.uint8,
                     device=dev)
    assert ws.numel() == tq.tq_decode_attend_workspace_bytes(w.B, w.Hq, w.Hkv, w.S, w.d)
    tq.tq_workspace_init(ws)
    a = torch.empty((w.B, w.Hq, 1, w.d), dtype=torch.float16, device=dev)
    b = torch.empty((w.B, w.Hq, w.d), dtype=torch.float16, device=dev)
    tq.tq_decode_attend_multi(ck, cv, q.view(w.B, w.Hq, 1, w.d), kc, kn, vc, vn, lens, a, ws, k_tail=kt, v_tail=vt,
                              tail_lens=tl)
    tq.tq_decode_attend_tail(ck, cv, q, kc, kn, vc, vn, lens, kt, vt, tl, b, ws)
    torch.cuda.synchronize()
    assert torch.equal(a.view(w.B, w.Hq, w.d), b)


def test_multi_full_size_long_context_sampled():
    # the 32K-token 8-bit K / 3-bit V workload verifying 4 drafted tokens (the last 4 of a
    # 37-token fp16 tail), units sampled
    torch, tq = torch_mods()
    dev = torch.device("cuda")
    w = tq_inputs.WORKLOADS["c4_long_k8v3"]
    ck, cv = codecs(w)
    ok_k, ok_v = oracle_codecs(w)
    K, V = w.kv("k", 8), w.kv("v", 8)
    kc, kn, vc, vn = encode_cache(w, ck, cv, K, V)
    L, max_tail, T = 4, 64, 37
    q = tq_inputs.fp16_normal(41, (w.B, w.Hq, L, w.d))
    kt = tq_inputs.fp16_normal(42, (w.B, w.Hkv, max_tail, w.d))
    vt = tq_inputs.fp16_normal(43, (w.B, w.Hkv, max_tail, w.d))
    out = torch.empty((w.B, w.Hq, L, w.d), dtype=torch.float16, device=dev)
    ws = torch.empty(tq.tq_decode_attend_multi_workspace_bytes(w.B, w.Hq, w.Hkv, L, w.S, w.d), dtype=torch.uint8,
                     device=dev)
    tq.tq_workspace_init(ws)
    lens = w.lengths()
    tq.tq_decode_attend_multi(ck, cv, torch.from_numpy(q).to(dev), kc, kn, vc, vn, torch.from_numpy(lens).to(dev),
                              out, ws, k_tail=torch.from_numpy(kt).to(dev), v_tail=torch.from_numpy(vt).to(dev),
                              tail_lens=torch.full((w.B,), T, dtype=torch.int32, device=dev))
    torch.cuda.synchronize()
    assert tq.tq_get_device_error(ws) == 0
    got = out.float().cpu().numpy().astype(np.float64)
    kcc, knn, vcc, vnn = kc.cpu().numpy(), kn.cpu().numpy(), vc.cpu().numpy(), vn.cpu().numpy()
    G = w.G
    for b, h in [(0, 2), (0, 7)]:
        n = int(lens[b])
        # the GPU-written codes and norms of this unit are the oracle's encoding, bit for bit
        rkc, rkn, _, mk = ok_k.encode(K[b, h, :n])
        rvc, rvn, _, mv = ok_v.encode(V[b, h, :n])
        assert mk == 0 and mv == 0
        assert np.array_equal(kcc[b, h, :n], rkc) and np.array_equal(vcc[b, h, :n], rvc)
        assert np.array_equal(knn[b, h, :n].view(np.uint16), rkn.view(np.uint16))
        assert np.array_equal(vnn[b, h, :n].view(np.uint16), rvn.view(np.uint16))
        ref = oracle.attention_multi_unit(ok_k, ok_v, q[b, h * G:(h + 1) * G], kcc[b, h, :n], knn[b, h, :n],
                                          vcc[b, h, :n], vnn[b, h, :n], n, 1 / math.sqrt(w.d), kt[b, h, :T],
                                          vt[b, h, :T])
        check_close(got[b, h * G:(h + 1) * G], ref, f"c4 multi unit {b},{h}", beyond_store_max=MARGIN)
