"""Keys with the QJL residual sketch (the TurboQuantProd variant): GPU encode
against the oracle bit for bit (codes, norms, sign bits, residual norms), and
decode attention with the QJL estimator against the oracle's attention
(max-abs <= 2e-3, rel-L2 <= 1e-3)."""
import math

import numpy as np
import pytest

import oracle
import tq_inputs
from tq_helpers import check_close, torch_mods

pytestmark = pytest.mark.gpu


def _gpu_encode_qjl(codec, x):
    torch, tq = torch_mods()
    dev = torch.device("cuda")
    n, d = x.shape
    codes = torch.full((n, codec.bytes_per_vec), 0xAB, dtype=torch.uint8, device=dev)
    norms = torch.empty(n, dtype=torch.float16, device=dev)
    signs = torch.full((n, d // 8), 0xCD, dtype=torch.uint8, device=dev)
    rn = torch.empty(n, dtype=torch.float16, device=dev)
    tq.tq_encode_qjl(codec, torch.from_numpy(x).to(dev), codes, norms, signs, rn)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), norms.cpu().numpy(), signs.cpu().numpy(), rn.cpu().numpy()


def _assert_same(got, ref):
    for g, r in zip(got, ref):
        np.testing.assert_array_equal(np.asarray(g).view(np.uint8), np.asarray(r).view(np.uint8))


@pytest.mark.parametrize("d", [64, 128, 256])
def test_qjl_sketch_matches_oracle(d):
    _, tq = torch_mods()
    c = tq.tq_codec_create_qjl(d, 3, 42)
    np.testing.assert_array_equal(tq.tq_codec_export_sketch(c), oracle.Codec(d, 3, 42).qjl_sketch())


@pytest.mark.parametrize("d,bits", [(64, 2), (128, 2), (128, 3), (128, 4), (256, 3), (32, 4), (512, 2)])
def test_qjl_encode_bit_exact(d, bits):
    _, tq = torch_mods()
    c = tq.tq_codec_create_qjl(d, bits, 42)
    oc = oracle.Codec(d, bits, 42)
    x = tq_inputs.fp16_normal(tq_inputs.stream_seed(0, tq_inputs.ENC_ID, d, bits, 1), (777, d),
                              tq_inputs.outlier_channels(d))
    _assert_same(_gpu_encode_qjl(c, x), oc.encode_qjl(x))


def test_qjl_encode_edge_rows():
    # zero, tiny, one-hot, integer-valued and large (finite-norm) rows
    _, tq = torch_mods()
    d = 128
    rng = np.random.default_rng(9)
    rows = [np.zeros(d), np.full(d, 2.0 ** -24), np.where(np.arange(d) == 5, 1.0, 0.0),
            np.where(np.arange(d) % 2 == 0, 2.0 ** -24, -3.0), rng.integers(-3, 4, d).astype(np.float64),
            np.full(d, 4000.0)]
    x = np.concatenate([np.array(rows).astype(np.float16), tq_inputs.fp16_normal(81, (30, d)) * np.float16(1e-3),
                        tq_inputs.fp16_normal(82, (30, d)) * np.float16(300)]).astype(np.float16)
    for bits in (2, 3, 4):
        c = tq.tq_codec_create_qjl(d, bits, 7)
        oc = oracle.Codec(d, bits, 7)
        ref = oc.encode_qjl(x)
        _assert_same(_gpu_encode_qjl(c, x), ref)
        assert np.all(ref[2][0] == 0) and ref[3][0] == 0          # zero row: no residual


def _decode_case(G, lens, d=128, kbits=3, vbits=3, S=520, B=None, seed=0):
    torch, tq = torch_mods()
    dev = torch.device("cuda")
    B = len(lens) if B is None else B
    Hkv = 2
    w = tq_inputs.Workload("qjl", B=B, Hq=G * Hkv, Hkv=Hkv, d=d, S=S, k_bits=kbits, v_bits=vbits, k_outliers=True,
                           seed=seed)
    ck, cv = tq.tq_codec_create_qjl(d, kbits, 42), tq.tq_codec_create(d, vbits, 42)
    ok, ov = oracle.Codec(d, kbits, 42), oracle.Codec(d, vbits, 42)
    K, V, q = w.kv("k", 1), w.kv("v", 1), w.q()
    n = B * Hkv * S
    kc = torch.empty((B, Hkv, S, ck.bytes_per_vec), dtype=torch.uint8, device=dev)
    kn = torch.empty((B, Hkv, S), dtype=torch.float16, device=dev)
    ks = torch.empty((B, Hkv, S, d // 8), dtype=torch.uint8, device=dev)
    kr = torch.empty((B, Hkv, S), dtype=torch.float16, device=dev)
    vc = torch.empty((B, Hkv, S, cv.bytes_per_vec), dtype=torch.uint8, device=dev)
    vn = torch.empty((B, Hkv, S), dtype=torch.float16, device=dev)
    tq.tq_encode_qjl(ck, torch.from_numpy(K).to(dev).view(n, d), kc.view(n, -1), kn.view(-1), ks.view(n, -1),
                     kr.view(-1))
    tq.tq_encode(cv, torch.from_numpy(V).to(dev).view(n, d), vc.view(n, -1), vn.view(-1))
    out = torch.empty((B, w.Hq, d), dtype=torch.float16, device=dev)
    ws = torch.empty(tq.tq_decode_attend_workspace_bytes(B, w.Hq, Hkv, S, d), dtype=torch.uint8, device=dev)
    tq.tq_workspace_init(ws)
    tq.tq_decode_attend_qjl(ck, cv, torch.from_numpy(q).to(dev), kc, kn, ks, kr, vc, vn,
                            torch.tensor(lens, dtype=torch.int32, device=dev), out, ws)
    torch.cuda.synchronize()
    assert tq.tq_get_device_error(ws) == 0
    got = out.float().cpu().numpy().astype(np.float64)
    # the oracle attends over its own encode of the same keys (bit-identical to the GPU's)
    ref = np.zeros_like(got)
    for b in range(B):
        L = int(lens[b])
        for h in range(Hkv):
            m = max(L, 1)
            c_, n_, s_, r_ = ok.encode_qjl(K[b, h, :m])
            vc_, vn_, _, _ = ov.encode(V[b, h, :m])
            ref[b, h * G:(h + 1) * G] = oracle.attention_qjl_unit(ok, ov, q[b, h * G:(h + 1) * G], c_, n_, s_, r_,
                                                                  vc_, vn_, L, 1 / math.sqrt(d))
    return got, ref


@pytest.mark.parametrize("G", [1, 4, 8, 16])
@pytest.mark.parametrize("kbits", [2, 3])
def test_qjl_decode_parity(G, kbits):
    # G <= 8: tensor-core kernel; G = 16 (two row groups per KV head): the SIMT kernel
    got, ref = _decode_case(G, lens=[517, 0, 64], kbits=kbits)
    check_close(got, ref, f"qjl G={G} K{kbits}+1")


@pytest.mark.parametrize("d", [64, 256])
def test_qjl_decode_head_dims(d):
    got, ref = _decode_case(4, lens=[255, 31], d=d, S=256)
    check_close(got, ref, f"qjl d={d}")


def test_qjl_codecs_are_refused_where_keys_carry_no_sketch():
    torch, tq = torch_mods()
    dev = torch.device("cuda")
    ck, cv = tq.tq_codec_create_qjl(128, 3, 1), tq.tq_codec_create(128, 3, 1)
    B, H, S, d = 1, 1, 64, 128
    kc = torch.zeros((B, H, S, ck.bytes_per_vec), dtype=torch.uint8, device=dev)
    kn = torch.zeros((B, H, S), dtype=torch.float16, device=dev)
    vc = torch.zeros((B, H, S, cv.bytes_per_vec), dtype=torch.uint8, device=dev)
    q = torch.zeros((B, H, d), dtype=torch.float16, device=dev)
    out = torch.empty_like(q)
    ws = torch.zeros(tq.tq_decode_attend_workspace_bytes(B, H, H, S, d), dtype=torch.uint8, device=dev)
    lens = torch.full((B,), S, dtype=torch.int32, device=dev)
    with pytest.raises(tq.TQError):
        tq.tq_decode_attend(ck, cv, q, kc, kn, vc, kn, lens, out, ws)
    with pytest.raises(tq.TQError):
        tq.KVCache(ck, cv, B, H, H, S)
    with pytest.raises(tq.TQError):                 # an MSE codec has no sketch
        x = torch.zeros((4, d), dtype=torch.float16, device=dev)
        tq.tq_encode_qjl(cv, x, torch.zeros((4, 48), dtype=torch.uint8, device=dev),
                         torch.zeros(4, dtype=torch.float16, device=dev),
                         torch.zeros((4, 16), dtype=torch.uint8, device=dev),
                         torch.zeros(4, dtype=torch.float16, device=dev))


def test_qjl_full_size_long_context_sampled():
    # the 32K-token shape (64/8 heads, d 128) with 3-bit MSE + QJL keys and 3-bit values,
    # the bench's launch configuration; two (batch, KV head) units compared
    torch, tq = torch_mods()
    dev = torch.device("cuda")
    w = tq_inputs.WORKLOADS["c4_long_k8v3"]
    d, S, Hkv = w.d, w.S, w.Hkv
    ck, cv = tq.tq_codec_create_qjl(d, 3, w.rot_seed), tq.tq_codec_create(d, 3, w.rot_seed)
    ok, ov = oracle.Codec(d, 3, w.rot_seed), oracle.Codec(d, 3, w.rot_seed)
    K, V, q = w.kv("k", 8), w.kv("v", 8), w.q()
    n = w.B * Hkv * S
    kc = torch.empty((w.B, Hkv, S, ck.bytes_per_vec), dtype=torch.uint8, device=dev)
    kn = torch.empty((w.B, Hkv, S), dtype=torch.float16, device=dev)
    ks = torch.empty((w.B, Hkv, S, d // 8), dtype=torch.uint8, device=dev)
    kr = torch.empty((w.B, Hkv, S), dtype=torch.float16, device=dev)
    vc = torch.empty((w.B, Hkv, S, cv.bytes_per_vec), dtype=torch.uint8, device=dev)
    vn = torch.empty((w.B, Hkv, S), dtype=torch.float16, device=dev)
    tq.tq_encode_qjl(ck, torch.from_numpy(K).to(dev).view(n, d), kc.view(n, -1), kn.view(-1), ks.view(n, -1),
                     kr.view(-1))
    tq.tq_encode(cv, torch.from_numpy(V).to(dev).view(n, d), vc.view(n, -1), vn.view(-1))
    out = torch.empty((w.B, w.Hq, d), dtype=torch.float16, device=dev)
    ws = torch.empty(tq.tq_decode_attend_workspace_bytes(w.B, w.Hq, Hkv, S, d), dtype=torch.uint8, device=dev)
    tq.tq_workspace_init(ws)
    lens = w.lengths()
    tq.tq_decode_attend_qjl(ck, cv, torch.from_numpy(q).to(dev), kc, kn, ks, kr, vc, vn,
                            torch.from_numpy(lens).to(dev), out, ws)
    torch.cuda.synchronize()
    assert tq.tq_get_device_error(ws) == 0
    got = out.float().cpu().numpy().astype(np.float64)
    kcc, knn, kss, krr = kc.cpu().numpy(), kn.cpu().numpy(), ks.cpu().numpy(), kr.cpu().numpy()
    vcc, vnn = vc.cpu().numpy(), vn.cpu().numpy()
    G = w.G
    for b, h in [(0, 1), (0, 6)]:
        L = int(lens[b])
        # the GPU's sketch fields of this unit are the oracle's, bit for bit
        c_, n_, s_, r_ = ok.encode_qjl(K[b, h, :L])
        assert np.array_equal(kss[b, h, :L], s_) and np.array_equal(krr[b, h, :L].view(np.uint16), r_.view(np.uint16))
        ref = oracle.attention_qjl_unit(ok, ov, q[b, h * G:(h + 1) * G], kcc[b, h, :L], knn[b, h, :L], kss[b, h, :L],
                                        krr[b, h, :L], vcc[b, h, :L], vnn[b, h, :L], L, 1 / math.sqrt(d))
        check_close(got[b, h * G:(h + 1) * G], ref, f"c4-shape qjl unit {b},{h}")
