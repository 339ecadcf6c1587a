"""GPU encode (through the C ABI) against the CPU oracle: codes, packed bytes and
fp16 norms must match bit for bit."""
import numpy as np
import pytest

import oracle
import tq_inputs
from tq_helpers import torch_mods

pytestmark = pytest.mark.gpu


def _gpu_encode(codec, x, stride=None):
    torch, tq = torch_mods()
    dev = torch.device("cuda")
    n, d = x.shape
    xt = torch.from_numpy(x).to(dev)
    if stride is not None:       # rows embedded in a wider buffer
        buf = torch.zeros((n, stride), dtype=torch.float16, device=dev)
        buf[:, :d] = xt
        xt = buf[:, :d]
    codes = torch.full((n, codec.bytes_per_vec), 0xAB, dtype=torch.uint8, device=dev)
    norms = torch.empty(n, dtype=torch.float16, device=dev)
    tq.tq_encode(codec, xt, codes, norms)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), norms.cpu().numpy()


def test_codec_tables_match_oracle():
    torch, tq = torch_mods()
    for d in (64, 96, 128, 160, 256):
        for bits in (2, 3, 4, 8):
            c = tq.tq_codec_create(d, bits, 42)
            t = tq.tq_codec_export(c)
            o = oracle.Codec(d, bits, 42).tables()
            np.testing.assert_array_equal(t["centroids"], o["centroids"])
            np.testing.assert_array_equal(t["midpoints"], o["midpoints"])
            if c.is_wht:
                np.testing.assert_array_equal(t["signs"], o["signs"])
            else:
                np.testing.assert_array_equal(t["dense_q"], o["Q"])
            # the same tables through tq_codec_info (host centroids) and tq_codec_export_rotation
            np.testing.assert_array_equal(tq.tq_codec_info(c)["centroids"], t["centroids"])
            r = tq.tq_codec_export_rotation(c)
            if c.is_wht:
                np.testing.assert_array_equal(r["signs"], t["signs"])
            else:
                np.testing.assert_array_equal(r["dense_q"], t["dense_q"])


@pytest.mark.parametrize("d,bits", [(64, 4), (128, 2), (128, 3), (128, 4), (128, 8), (96, 3), (96, 8),
                                    (256, 3), (256, 4), (32, 4), (512, 2), (160, 4)])
def test_encode_bit_exact(d, bits):
    torch, tq = torch_mods()
    c = tq.tq_codec_create(d, bits, 42)
    oc = oracle.Codec(d, bits, 42)
    x = tq_inputs.fp16_normal(tq_inputs.stream_seed(0, tq_inputs.ENC_ID, d, bits), (1037, d),
                              tq_inputs.outlier_channels(d))
    codes, norms = _gpu_encode(c, x)
    rc, rn, ties, mism = oc.encode(x)
    assert mism == 0
    np.testing.assert_array_equal(codes, rc)
    np.testing.assert_array_equal(norms.view(np.uint16), rn.view(np.uint16))


def test_encode_edge_values_and_strided_rows():
    torch, tq = torch_mods()
    d = 128
    rng = np.random.default_rng(5)
    rows = [np.zeros(d), np.full(d, 65504.0), np.full(d, -65504.0), np.full(d, 2.0**-24),
            np.where(np.arange(d) == 7, 1.0, 0.0), np.where(np.arange(d) % 2 == 0, 2.0**-24, -3.0),
            (rng.integers(-3, 4, d)).astype(np.float64)]
    x = np.array(rows).astype(np.float16)
    x = np.concatenate([x, tq_inputs.fp16_normal(77, (25, d)) * np.float16(1e-3),
                        tq_inputs.fp16_normal(78, (25, d)) * np.float16(300)]).astype(np.float16)
    for bits in (2, 3, 4, 8):
        c = tq.tq_codec_create(d, bits, 7)
        oc = oracle.Codec(d, bits, 7)
        rc, rn, _, _ = oc.encode(x)
        for stride in (None, 136):
            codes, norms = _gpu_encode(c, x, stride)
            np.testing.assert_array_equal(codes, rc)
            np.testing.assert_array_equal(norms.view(np.uint16), rn.view(np.uint16))
    assert np.all(rc[0] == 0) and np.isinf(rn[1]) and np.isinf(rn[2])


@pytest.mark.parametrize("n", [0, 1, 7, 8, 9, 1000])
def test_encode_ragged_counts(n):
    torch, tq = torch_mods()
    d, bits = 256, 3
    c = tq.tq_codec_create(d, bits, 42)
    x = tq_inputs.fp16_normal(123, (max(n, 1), d))[:n]
    if n == 0:
        dev = torch.device("cuda")
        tq.tq_encode(c, torch.empty((0, d), dtype=torch.float16, device=dev),
                     torch.empty((0, c.bytes_per_vec), dtype=torch.uint8, device=dev),
                     torch.empty(0, dtype=torch.float16, device=dev))
        return
    codes, norms = _gpu_encode(c, x)
    rc, rn, _, _ = oracle.Codec(d, bits, 42).encode(x)
    np.testing.assert_array_equal(codes, rc)
    np.testing.assert_array_equal(norms.view(np.uint16), rn.view(np.uint16))


def test_encode_append_pending_batch_and_bad_positions():
    # Pending-token batches of 64 written into a cache ("add TurboQuant KV cache
    # compression", Design: batch recompression).
    torch, tq = torch_mods()
    dev = torch.device("cuda")
    B, H, T, S, d, bits = 3, 2, 64, 256, 128, 4
    c = tq.tq_codec_create(d, bits, 42)
    x = tq_inputs.fp16_normal(99, (B, H, T, d), tq_inputs.outlier_channels(d))
    start = np.array([0, 100, 250], dtype=np.int32)        # the last one overflows max_seq
    codes = torch.zeros((B, H, S, c.bytes_per_vec), dtype=torch.uint8, device=dev)
    norms = torch.zeros((B, H, S), dtype=torch.float16, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    tq.tq_encode_append(c, torch.from_numpy(x).to(dev), torch.from_numpy(start).to(dev), codes, norms, err)
    torch.cuda.synchronize()
    assert tq.tq_get_device_error(err) == tq.TQ_DEVERR_POSITION
    assert tq.tq_get_device_error(err) == 0          # read clears it
    cc, nn = codes.cpu().numpy(), norms.cpu().numpy()
    oc = oracle.Codec(d, bits, 42)
    for b in range(B):
        for h in range(H):
            rc, rn, _, _ = oc.encode(x[b, h])
            for t in range(T):
                p = start[b] + t
                if p < S:
                    np.testing.assert_array_equal(cc[b, h, p], rc[t])
                    assert nn[b, h, p].view(np.uint16) == rn[t].view(np.uint16)
            untouched = np.ones(S, bool)
            untouched[start[b]:min(S, start[b] + T)] = False
            assert np.all(cc[b, h, untouched] == 0)


@pytest.mark.parametrize("d,kb,vb", [(128, 8, 3), (128, 4, 2), (96, 8, 3), (256, 3, 3)])
def test_encode_append_kv_is_two_appends_in_one_launch(d, kb, vb):
    # The K and V pending batches encoded in one launch ("add TurboQuant KV cache
    # compression", Design: batch recompression): bit for bit the two single-codec
    # appends, and the oracle's encoding of every written row.
    torch, tq = torch_mods()
    dev = torch.device("cuda")
    B, H, T, S = 2, 3, 64, 320
    ck, cv = tq.tq_codec_create(d, kb, 42), tq.tq_codec_create(d, vb, 42)
    k = tq_inputs.fp16_normal(51, (B, H, T, d), tq_inputs.outlier_channels(d))
    v = tq_inputs.fp16_normal(52, (B, H, T, d))
    start = torch.tensor([7, 256], dtype=torch.int32, device=dev)
    kd, vd = torch.from_numpy(k).to(dev), torch.from_numpy(v).to(dev)

    def caches():
        return (torch.zeros((B, H, S, ck.bytes_per_vec), dtype=torch.uint8, device=dev),
                torch.zeros((B, H, S), dtype=torch.float16, device=dev),
                torch.zeros((B, H, S, cv.bytes_per_vec), dtype=torch.uint8, device=dev),
                torch.zeros((B, H, S), dtype=torch.float16, device=dev))
    a = caches()
    tq.tq_encode_append_kv(ck, cv, kd, vd, start, *a)
    b = caches()
    tq.tq_encode_append(ck, kd, start, b[0], b[1])
    tq.tq_encode_append(cv, vd, start, b[2], b[3])
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.uint8), y.view(torch.uint8))
    ok, ov = oracle.Codec(d, kb, 42), oracle.Codec(d, vb, 42)
    kc, kn, vc, vn = (t.cpu().numpy() for t in a)
    st = start.cpu().numpy()
    for bb in range(B):
        for h in range(H):
            rkc, rkn, _, m1 = ok.encode(k[bb, h])
            rvc, rvn, _, m2 = ov.encode(v[bb, h])
            assert m1 == 0 and m2 == 0
            sl = slice(st[bb], st[bb] + T)
            np.testing.assert_array_equal(kc[bb, h, sl], rkc)
            np.testing.assert_array_equal(vc[bb, h, sl], rvc)
            np.testing.assert_array_equal(kn[bb, h, sl].view(np.uint16), rkn.view(np.uint16))
            np.testing.assert_array_equal(vn[bb, h, sl].view(np.uint16), rvn.view(np.uint16))


def test_encode_append_kv_argument_checks():
    torch, tq = torch_mods()
    dev = torch.device("cuda")
    c128, c96 = tq.tq_codec_create(128, 4, 42), tq.tq_codec_create(96, 4, 42)
    raw = tq.tq_codec_create(128, 16, 42)
    x = torch.zeros((1, 1, 4, 128), dtype=torch.float16, device=dev)
    pos = torch.zeros(1, dtype=torch.int32, device=dev)
    kc = torch.zeros((1, 1, 8, 64), dtype=torch.uint8, device=dev)
    kn = torch.zeros((1, 1, 8), dtype=torch.float16, device=dev)
    lib = tq._lib
    st = torch.cuda.current_stream().cuda_stream
    args = (x.data_ptr(), x.data_ptr(), 1, 1, 4, pos.data_ptr(), 8, kc.data_ptr(), kn.data_ptr(), kc.data_ptr(),
            kn.data_ptr(), None, st)
    assert lib.tq_encode_append_kv(c128.handle, c96.handle, *args) == 1      # different dims
    assert lib.tq_encode_append_kv(raw.handle, c128.handle, *args) == 1      # raw keys are not encoded
    assert lib.tq_encode_append_kv(c128.handle, c128.handle, *args[:7], None, *args[8:]) == 1
    assert lib.tq_encode_append_kv(c128.handle, c128.handle, *args) == 0
    torch.cuda.synchronize()


@pytest.mark.parametrize("name", ["c2_llama3b", "c4_long_k8v3", "c4_long_k8v3_d96"])
def test_encode_full_size_sampled(name):
    # Full-size K/V of the workload encoded in one launch each; a sample of rows
    # is re-encoded by the oracle.
    torch, tq = torch_mods()
    w = tq_inputs.WORKLOADS[name]
    dev = torch.device("cuda")
    ck = tq.tq_codec_create(w.d, w.k_bits, w.rot_seed)
    oc = oracle.Codec(w.d, w.k_bits, w.rot_seed)
    K = w.kv("k")
    n = w.B * w.Hkv * w.S
    codes = torch.empty((n, ck.bytes_per_vec), dtype=torch.uint8, device=dev)
    norms = torch.empty(n, dtype=torch.float16, device=dev)
    tq.tq_encode(ck, torch.from_numpy(K).to(dev).view(n, w.d), codes, norms)
    cc, nn = codes.cpu().numpy(), norms.cpu().numpy()
    idx = np.unique(np.concatenate([np.arange(64), n - 1 - np.arange(64),
                                    np.random.default_rng(0).integers(0, n, 1500)]))
    rc, rn, _, mism = oc.encode(K.reshape(n, w.d)[idx])
    assert mism == 0
    np.testing.assert_array_equal(cc[idx], rc)
    np.testing.assert_array_equal(nn[idx].view(np.uint16), rn.view(np.uint16))
