"""Shared helpers of the GPU parity tests (CUDA path through the C ABI vs the CPU oracle)."""
from __future__ import annotations

import math
import os

import numpy as np

import oracle
import tq_inputs

ATOL = 2e-3      # max-abs bound on attention outputs
RTOL_L2 = 1e-3   # relative L2 bound on attention outputs


def torch_mods():
    import torch
    import quantized_kv_cache_10_gb300 as tq
    return torch, tq


def codecs(w):
    torch, tq = torch_mods()
    return tq.tq_codec_create(w.d, w.k_bits, w.rot_seed), tq.tq_codec_create(w.d, w.v_bits, w.rot_seed)


def oracle_codecs(w):
    return oracle.Codec(w.d, w.k_bits, w.rot_seed), oracle.Codec(w.d, w.v_bits, w.rot_seed)


def encode_cache(w, ck, cv, K, V):
    """Encode host fp16 K/V [B, Hkv, S, d] on the GPU into a packed cache."""
    torch, tq = torch_mods()
    dev = torch.device("cuda")
    n = w.B * w.Hkv * w.S
    if w.k_bits == 16:
        kc = torch.from_numpy(K).to(dev)
        kn = None
    else:
        kc = torch.empty((w.B, w.Hkv, w.S, ck.bytes_per_vec), dtype=torch.uint8, device=dev)
        kn = torch.empty((w.B, w.Hkv, w.S), dtype=torch.float16, device=dev)
        tq.tq_encode(ck, torch.from_numpy(K).to(dev).view(n, w.d), kc.view(n, -1), kn.view(-1))
    vc = torch.empty((w.B, w.Hkv, w.S, cv.bytes_per_vec), dtype=torch.uint8, device=dev)
    vn = torch.empty((w.B, w.Hkv, w.S), dtype=torch.float16, device=dev)
    tq.tq_encode(cv, torch.from_numpy(V).to(dev).view(n, w.d), vc.view(n, -1), vn.view(-1))
    return kc, kn, vc, vn


def decode(w, ck, cv, q, kc, kn, vc, vn, lens=None, scale=None):
    torch, tq = torch_mods()
    dev = torch.device("cuda")
    lens = w.lengths() if lens is None else lens
    out = torch.empty((w.B, w.Hq, w.d), dtype=torch.float16, device=dev)
    ws = torch.empty(tq.tq_decode_attend_workspace_bytes(w.B, w.Hq, w.Hkv, w.S, w.d), dtype=torch.uint8, device=dev)
    tq.tq_workspace_init(ws)
    tq.tq_decode_attend(ck, cv, torch.from_numpy(np.ascontiguousarray(q)).to(dev), kc, kn, vc, vn,
                        torch.from_numpy(np.asarray(lens, dtype=np.int32)).to(dev), out, ws,
                        scale=scale)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64), ws


def check_close(got, ref, what="", beyond_store_max=None):
    """got: the CUDA path's fp16 attention output (as float64); ref: the oracle's fp64 value.

    Asserts the raw max-abs error <= ATOL and the relative L2 error <= RTOL_L2.  Beside
    the raw error it reports the error beyond the fp16 output store's own rounding
    (half an fp16 ulp of the reference value: the part an exactly computed result
    would still show), which isolates the kernel's arithmetic; beyond_store_max, when
    given, bounds that part too.  Returns (raw max-abs, beyond-store max, rel-L2)."""
    err = got - ref
    half_ulp = np.spacing(np.abs(ref).astype(np.float16)).astype(np.float64) / 2
    raw = float(np.abs(err).max()) if err.size else 0.0
    beyond = float(np.maximum(np.abs(err) - half_ulp, 0.0).max()) if err.size else 0.0
    nrm = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(err) / nrm) if nrm > 0 else float(np.linalg.norm(err))
    log = os.environ.get("TQ_PARITY_LOG")      # optional record of the measured errors
    if log:
        with open(log, "a") as f:
            f.write(f"{what}\tmax_abs {raw:.3e}\tbeyond_fp16_store {beyond:.3e}\trel_l2 {rel:.3e}\n")
    msg = f"{what}: max-abs {raw:.3e} (<= {ATOL}), {beyond:.3e} beyond the fp16 store, rel-L2 {rel:.3e} (<= {RTOL_L2})"
    assert raw <= ATOL and rel <= RTOL_L2, msg
    if beyond_store_max is not None:
        assert beyond <= beyond_store_max, msg + f"; beyond-store bound {beyond_store_max}"
    return raw, beyond, rel


def oracle_unit_reference(w, ok_k, ok_v, q, K, V, b, h, lens):
    """Oracle encode of one (b, kvh) unit and its attention output [G, d]."""
    L = int(lens[b])
    n = max(L, 1)
    if w.k_bits == 16:
        kk, kn = K[b, h, :n], None
    else:
        kk, kn, _, mism = ok_k.encode(K[b, h, :n])
        assert mism == 0
    vc, vn, _, mism = ok_v.encode(V[b, h, :n])
    assert mism == 0
    G = w.G
    return oracle.attention_unit(ok_k, ok_v, q[b, h * G:(h + 1) * G], kk, kn, vc, vn, L,
                                 1.0 / math.sqrt(w.d)), (kk, kn, vc, vn)
