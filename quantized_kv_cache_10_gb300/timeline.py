"""Phase timeline of the fused decode attention (profiling build).

Builds libtq_timeline.so (the library compiled with -DTQ_TIMELINE), runs decode-attention
calls of a workload and prints, per phase, the min / median / max over the CTAs of
globaltimer stamps (microseconds):

  back-to-back  64 calls replayed from a CUDA graph over cycled cache replicas (the
                bench's launch configuration); times relative to the end of the
                previous call (its last combine CTA's store)
  isolated      one call after an L2 flush; times relative to the first decode CTA's
                entry

Decode CTA phases: entry, codec tables landed, dependency wait passed, first tile
consumed, own loop done (consumer warp 0), all warps' loops done, partial written,
and the rotated query block ready (after the prologue's barrier).
Combine CTA phases: entry, dependency wait passed, output stored.

  python -m quantized_kv_cache_10_gb300.timeline [--workload c4_long_k8v3]
  (or python quantized_kv_cache_10_gb300/timeline.py ...)
"""
from __future__ import annotations

import argparse
import importlib.util
import math
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SLOTS, STAMPS = 4096, 8
DEC = ["entry", "sm", "wait", "first_tile", "loop_w0", "loops_all", "partial", "q_ready"]
COMB = ["entry", "wait", "stored", "sm"]


def _build_timeline_lib():
    spec = importlib.util.spec_from_file_location("_tq_build", os.path.join(HERE, "_build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod.build(variant="timeline")


def _records(buf, half):
    base = half * 2 * SLOTS * STAMPS
    dec = buf[base:base + SLOTS * STAMPS].reshape(SLOTS, STAMPS)
    comb = buf[base + SLOTS * STAMPS:base + 2 * SLOTS * STAMPS].reshape(SLOTS, STAMPS)
    return dec[dec[:, 0] > 0], comb[comb[:, 0] > 0]


def _report(title, dec, comb, origin):
    print(title)
    print(f"  decode CTAs {len(dec)}, combine CTAs {len(comb)} (us from the origin: min / median / max)")
    for i, name in enumerate(DEC):
        if name == "sm":
            continue
        x = (dec[:, i].astype(np.int64) - origin) / 1e3
        print(f"  decode  {name:11s} {x.min():8.2f} {np.median(x):8.2f} {x.max():8.2f}")
    for i, name in enumerate(COMB):
        if name == "sm":
            continue
        x = (comb[:, i].astype(np.int64) - origin) / 1e3
        print(f"  combine {name:11s} {x.min():8.2f} {np.median(x):8.2f} {x.max():8.2f}")
    # the latest decode CTAs: entry, first tile, partial (us) and the SM each ran on
    late = np.argsort(dec[:, 6])[-4:]
    for j in late:
        e, f, pt = ((int(dec[j, k]) - origin) / 1e3 for k in (0, 3, 6))
        print(f"  late decode CTA: SM {int(dec[j, 1]) & 0xffffffff}  entry {e:.2f}  first tile {f:.2f}  "
              f"partial {pt:.2f}")
    # token-balanced schedule: segments per CTA (counted above the SM id) and the CTA span
    # (entry to partial) by segment count
    nseg = (dec[:, 1].astype(np.uint64) >> np.uint64(32)).astype(np.int64)
    if nseg.max() > 0:
        span = (dec[:, 6].astype(np.int64) - dec[:, 0].astype(np.int64)) / 1e3
        for k in np.unique(nseg):
            sel = nseg == k
            print(f"  CTAs with {k} segment(s): {int(sel.sum()):4d}, entry-to-partial median "
                  f"{np.median(span[sel]):.2f} us, max {span[sel].max():.2f} us")
    sms = np.bincount(comb[:, 3].astype(np.int64) & 0xffffffff) if len(comb) else np.zeros(1)
    print(f"  combine CTAs per SM: at most {sms.max()}; SMs with more than one: {int((sms > 1).sum())}")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="c4_long_k8v3")
    args = ap.parse_args()
    if os.environ.get("TQ_LIB_VARIANT") != "timeline":
        # the package loads its library at import (and `-m` imports it first): start
        # again as a script with the profiling build selected
        _build_timeline_lib()
        env = dict(os.environ, TQ_LIB_VARIANT="timeline")
        os.execve(sys.executable, [sys.executable, os.path.abspath(__file__), *sys.argv[1:]], env)
    sys.path.insert(0, ROOT)
    import torch
    import quantized_kv_cache_10_gb300 as tq
    import tq_inputs

    dev = torch.device("cuda")
    w = tq_inputs.WORKLOADS[args.workload]
    ck, cv = tq.tq_codec_create(w.d, w.k_bits, w.rot_seed), tq.tq_codec_create(w.d, w.v_bits, w.rot_seed)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    R = 1 << (max(2, math.ceil(4 * l2 / w.packed_kv_bytes())) - 1).bit_length()
    R = min(R, 64)
    n = w.B * w.Hkv * w.S
    K, V = torch.from_numpy(w.kv("k", 16)).to(dev), torch.from_numpy(w.kv("v", 16)).to(dev)
    vc = torch.empty((R, w.B, w.Hkv, w.S, cv.bytes_per_vec), dtype=torch.uint8, device=dev)
    vn = torch.empty((R, w.B, w.Hkv, w.S), dtype=torch.float16, device=dev)
    if w.k_bits == 16:
        kc = K.unsqueeze(0).repeat(R, 1, 1, 1, 1)
        kn = None
    else:
        kc = torch.empty((R, w.B, w.Hkv, w.S, ck.bytes_per_vec), dtype=torch.uint8, device=dev)
        kn = torch.empty((R, w.B, w.Hkv, w.S), dtype=torch.float16, device=dev)
        tq.tq_encode(ck, K.view(n, w.d), kc[0].view(n, -1), kn[0].view(-1))
    tq.tq_encode(cv, V.view(n, w.d), vc[0].view(n, -1), vn[0].view(-1))
    for r in range(1, R):
        vc[r].copy_(vc[0])
        vn[r].copy_(vn[0])
        if kn is not None:
            kc[r].copy_(kc[0])
            kn[r].copy_(kn[0])
    del K, V
    q = torch.from_numpy(w.q()).to(dev)
    lens = torch.from_numpy(w.lengths()).to(dev)
    out = torch.empty((w.B, w.Hq, w.d), dtype=torch.float16, device=dev)
    ws = torch.empty(tq.tq_decode_attend_workspace_bytes(w.B, w.Hq, w.Hkv, w.S, w.d), dtype=torch.uint8, device=dev)
    tq.tq_workspace_init(ws)
    buf = torch.zeros(4 * SLOTS * STAMPS, dtype=torch.int64, device=dev)
    if tq._lib.tq_debug_set_timeline(buf.data_ptr(), buf.numel() * 8) != 0:
        raise RuntimeError("the timeline build did not load")

    def attend(i):
        r = i % R
        tq.tq_decode_attend(ck, cv, q, kc[r], None if kn is None else kn[r], vc[r], vn[r], lens, out, ws)

    # calls are numbered from the registration: 8 eager ones, then the 64 of the graph
    # (a replay reuses the numbers baked in at capture), so the graph's last call has
    # index 71 (odd half) and the one before it index 70 (even half)
    for i in range(8):
        attend(i)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(64):
            attend(i)
    for _ in range(4):
        g.replay()
    torch.cuda.synchronize()
    h = buf.cpu().numpy().view(np.uint64)
    dec, comb = _records(h, 71 & 1)
    pdec, pcomb = _records(h, 70 & 1)
    origin = int(pcomb[:, 2].max())
    print(f"workload {w.name}: B{w.B} Hq{w.Hq} Hkv{w.Hkv} d{w.d} S{w.S} K{w.k_bits}/V{w.v_bits}, "
          f"{w.packed_kv_bytes()} packed bytes per call")
    _report("back-to-back (origin: end of the previous call)", dec, comb, origin)
    print(f"  call period {(int(comb[:, 2].max()) - origin) / 1e3:.2f} us")

    flush = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
    flush.zero_()
    torch.cuda._sleep(100000)
    attend(0)
    torch.cuda.synchronize()
    h = buf.cpu().numpy().view(np.uint64)
    dec, comb = _records(h, 72 & 1)                  # the 73rd call since the registration
    origin = int(dec[:, 0].min())
    _report("isolated after an L2 flush (origin: first decode CTA's entry)", dec, comb, origin)
    print(f"  call span {(int(comb[:, 2].max()) - origin) / 1e3:.2f} us")
    tq._lib.tq_debug_set_timeline(None, 0)


if __name__ == "__main__":
    main()
