"""tq_decode_attend_noalloc: decode attention for callers that cannot allocate device
memory (they cannot hand over a workspace), running on the library's fixed scratch.

Checked through the C ABI against tq_decode_attend with a caller workspace, on two
calls in a row.  Both run the same split plan and the same kernels, whose merges
are in a fixed order, so the outputs must be identical bit for bit.  This file is
collected last so a stop-at-first-failure run has already run every other test."""
import ctypes as C

import numpy as np
import pytest

import tq_inputs
from tq_helpers import codecs, encode_cache, torch_mods

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["c2_llama3b", "c4_long_k8v3"])
def test_noalloc_matches_workspace_entry_point(name):
    torch, tq = torch_mods()
    lib = tq._lib
    dev = torch.device("cuda")
    w = tq_inputs.WORKLOADS[name]
    ck, cv = codecs(w)
    K, V, q = w.kv("k", 8), w.kv("v", 8), w.q()
    kc, kn, vc, vn = encode_cache(w, ck, cv, K, V)
    qd = torch.from_numpy(q).to(dev)
    lens = torch.from_numpy(w.lengths()).to(dev)
    scale = w.d ** -0.5
    st = torch.cuda.current_stream().cuda_stream
    # reference: the existing entry point with a caller-provided workspace
    ref = torch.empty((w.B, w.Hq, w.d), dtype=torch.float16, device=dev)
    ws = torch.empty(tq.tq_decode_attend_workspace_bytes(w.B, w.Hq, w.Hkv, w.S, w.d), dtype=torch.uint8, device=dev)
    tq.tq_workspace_init(ws)
    tq.tq_decode_attend(ck, cv, qd, kc, kn, vc, vn, lens, ref, ws, scale=scale)
    for _ in range(2):
        out = torch.full((w.B, w.Hq, w.d), float("nan"), dtype=torch.float16, device=dev)
        rc = lib.tq_decode_attend_noalloc(ck.handle, cv.handle, qd.data_ptr(), kc.data_ptr(), kn.data_ptr(),
                                          vc.data_ptr(), vn.data_ptr(), lens.data_ptr(), w.B, w.Hq, w.Hkv, w.S,
                                          C.c_float(scale), out.data_ptr(), st)
        assert rc == 0
        torch.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy().view(np.uint16), ref.cpu().numpy().view(np.uint16))


def test_noalloc_rejects_shapes_beyond_its_scratch():
    torch, tq = torch_mods()
    lib = tq._lib
    dev = torch.device("cuda")
    ck, cv = tq.tq_codec_create(128, 4, 42), tq.tq_codec_create(128, 4, 42)
    small = torch.zeros(4096, dtype=torch.uint8, device=dev)
    B, Hq, Hkv, S = 2048, 64, 8, 64          # 16384 units: workspace far above 8 MiB
    assert tq.tq_decode_attend_workspace_bytes(B, Hq, Hkv, S, 128) > 8 << 20
    p = small.data_ptr()
    st = torch.cuda.current_stream().cuda_stream
    rc = lib.tq_decode_attend_noalloc(ck.handle, cv.handle, p, p, p, p, p, p, B, Hq, Hkv, S, C.c_float(0.1), p, st)
    assert rc == 5                            # TQ_ERR_WORKSPACE, nothing enqueued
    torch.cuda.synchronize()


def test_noalloc_rejects_sketched_keys_before_enqueueing():
    # keys with the QJL sketch need tq_decode_attend_qjl: refused by the argument checks,
    # before the scratch's error word is cleared on the stream
    torch, tq = torch_mods()
    lib = tq._lib
    dev = torch.device("cuda")
    ck, cv = tq.tq_codec_create_qjl(128, 3, 42), tq.tq_codec_create(128, 3, 42)
    buf = torch.zeros(1 << 16, dtype=torch.uint8, device=dev)
    p = buf.data_ptr()
    st = torch.cuda.current_stream().cuda_stream
    rc = lib.tq_decode_attend_noalloc(ck.handle, cv.handle, p, p, p, p, p, p, 1, 8, 8, 64, C.c_float(0.1), p, st)
    assert rc == 1                            # TQ_ERR_INVALID_ARG
    torch.cuda.synchronize()
