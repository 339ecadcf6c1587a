"""GPU dequant against the oracle (relative L2 <= 1e-5) and the C-ABI error paths
that need a device (every failure is made on the host; nothing faults a GPU)."""
import numpy as np
import pytest

import oracle
import tq_inputs
from tq_helpers import torch_mods

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d,bits", [(64, 4), (128, 2), (128, 3), (128, 8), (96, 3), (256, 4), (160, 8)])
def test_dequant_matches_oracle(d, bits):
    torch, tq = torch_mods()
    dev = torch.device("cuda")
    c = tq.tq_codec_create(d, bits, 42)
    oc = oracle.Codec(d, bits, 42)
    x = tq_inputs.fp16_normal(31, (500, d), tq_inputs.outlier_channels(d))
    rc, rn, _, _ = oc.encode(x)
    out = torch.empty((500, d), dtype=torch.float32, device=dev)
    tq.tq_dequant(c, torch.from_numpy(rc).to(dev), torch.from_numpy(rn).to(dev), out)
    got = out.cpu().numpy().astype(np.float64)
    ref = oc.dequant(rc, rn)
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) <= 1e-5


def test_error_statuses():
    torch, tq = torch_mods()
    import ctypes as C
    lib = tq._lib
    dev = torch.device("cuda")
    ck = tq.tq_codec_create(128, 4, 1)
    cv = tq.tq_codec_create(128, 4, 2)
    c96 = tq.tq_codec_create(96, 4, 2)
    raw = tq.tq_codec_create(128, 16, 0)
    B, Hq, Hkv, S = 1, 8, 2, 64
    q = torch.zeros((B, Hq, 128), dtype=torch.float16, device=dev)
    kc = torch.zeros((B, Hkv, S, 64), dtype=torch.uint8, device=dev)
    kn = torch.zeros((B, Hkv, S), dtype=torch.float16, device=dev)
    lens = torch.full((B,), S, dtype=torch.int32, device=dev)
    out = torch.empty_like(q)
    need = tq.tq_decode_attend_workspace_bytes(B, Hq, Hkv, S, 128)
    assert need > 0
    ws = torch.zeros(need, dtype=torch.uint8, device=dev)

    def call(ckh, cvh, Hq_=Hq, Hkv_=Hkv, S_=S, ws_bytes=need, knp=kn.data_ptr(), kp=kc.data_ptr(), wsp=ws.data_ptr()):
        st = torch.cuda.current_stream().cuda_stream
        return lib.tq_decode_attend(ckh, cvh, q.data_ptr(), kp, knp, kc.data_ptr(), kn.data_ptr(), lens.data_ptr(),
                                    B, Hq_, Hkv_, S_, C.c_float(0.1), out.data_ptr(), wsp, ws_bytes, st)

    assert call(ck.handle, cv.handle) == 0
    assert call(ck.handle, c96.handle) == 1            # dims differ
    assert call(ck.handle, raw.handle) == 1            # raw fp16 V is not supported
    assert call(ck.handle, cv.handle, Hq_=7) == 1      # Hq % Hkv != 0
    assert call(ck.handle, cv.handle, S_=60) == 1      # max_seq % 8 != 0
    assert call(ck.handle, cv.handle, ws_bytes=need - 1) == 5
    assert call(ck.handle, cv.handle, knp=None) == 1   # quantised K needs norms
    assert call(raw.handle, cv.handle) == 1            # raw K must not pass norms
    assert call(ck.handle, cv.handle, kp=kc.data_ptr() + 4) == 1   # misaligned cache
    assert call(ck.handle, cv.handle, wsp=ws.data_ptr() + 16) == 5  # misaligned workspace
    assert tq.tq_decode_attend_workspace_bytes(1, 7, 2, 64, 128) == 0
    # encode argument checks
    x = torch.zeros((4, 128), dtype=torch.float16, device=dev)
    codes = torch.zeros((4, 64), dtype=torch.uint8, device=dev)
    norms = torch.zeros(4, dtype=torch.float16, device=dev)
    st = torch.cuda.current_stream().cuda_stream
    assert lib.tq_encode(ck.handle, x.data_ptr(), 4, 128, codes.data_ptr(), 64, norms.data_ptr(), st) == 0
    assert lib.tq_encode(ck.handle, x.data_ptr() + 2, 4, 128, codes.data_ptr(), 64, norms.data_ptr(), st) == 1
    assert lib.tq_encode(ck.handle, x.data_ptr(), 4, 128, codes.data_ptr(), 62, norms.data_ptr(), st) == 1
    assert lib.tq_encode(raw.handle, x.data_ptr(), 4, 128, codes.data_ptr(), 64, norms.data_ptr(), st) == 1
    with pytest.raises(tq.TQError):
        tq.tq_codec_create(100, 4, 0)
    torch.cuda.synchronize()
