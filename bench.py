"""Benchmark of the TurboQuant KV-cache hot path on GB300.

One step = one decode step of the 32K long-context workload (batch 1, 64 query
heads / 8 KV heads, head_dim 128, 8-bit K / 3-bit V, 32768 cached tokens):
fused split-K decode attention over the whole packed cache; every 64th step
also encodes the pending batch of 64 tokens (K and V of every KV head) into
the cache first ("add TurboQuant KV cache compression", Design: pending tokens
are encoded in batches of 64).  value = packed-KV bytes attended per second
(GB/s) over all timed steps.

Inputs larger than L2: the packed cache exists in R replicas (R >= 4 x L2 /
cache bytes, a power of two) and step i reads replica i mod R, so every read
comes from HBM.  The steps run back to back, replayed from CUDA graphs of 64
steps (launch overhead off the host), bracketed by one pair of CUDA events.
Caches so small that this needs more than 64 replicas are instead timed one
call at a time after an L2 flush.  The roofline object is the decode-attention
call alone (decode kernel + combine kernel), timed the same way; `e2e` runs
the steps eagerly through the public API with the host->device copy of the
step's inputs (q, lengths, and the new K/V on encode steps) from pinned memory
and the device->host read of the output in every step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl tq|reference]

--impl reference times the CPU oracle (the plain, slow implementation the tests
compare against) on the host cores over a bounded sample of the same workload.
Under torchrun (N > 1) every rank runs an independent replica (the method has
no exchange step); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import glob
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import tq_inputs  # noqa: E402

WORKLOAD = "c4_long_k8v3"
METRIC = "fused decode-attend GB/s of packed KV (% of HBM peak); encode Mvec/s"


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value, device="cpu"):
    """The largest of every rank's value (the slowest rank's time); the value itself when
    no process group of more than one rank is running.  device: where the reduction's
    tensor lives (the rank's GPU for NCCL, the host for gloo)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank, world_size, slowest_seconds):
    """Whole-job throughput: the units every rank processed (replicas: the same count on each)
    over the slowest rank's time."""
    return world_size * units_per_rank / slowest_seconds


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def _source_sha():
    """Hash of the sources that define the decode kernels (the ncu counters' validity key)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "quantized_kv_cache_10_gb300", "csrc")
    for f in sorted(glob.glob(os.path.join(csrc, "tq_decode_*")) + [os.path.join(csrc, "tq_internal.h")]):
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _traffic(kernel_name):
    """DRAM bytes per launch from a committed ncu summary, if taken on the current source."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel_name)
    if not e or e.get("source_sha") != _source_sha():
        return None
    return e.get("dram_bytes_per_launch")


def _lead(us=30.0):
    """Keeps the GPU busy for ~us microseconds on the current stream before a start event,
    so that the timed launches are already queued when the event fires: device time
    without the host's submission latency."""
    import torch
    torch.cuda._sleep(int(us * _sm_mhz()))


def _sm_mhz():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return float(json.load(f).get("sm_max_mhz", 2070.0))
    return 2070.0


class Clocks:
    """Samples SM clocks and throttle reasons with nvidia-smi while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- CPU oracle (baseline arm)
class OracleSample:
    """The oracle's decode attention over a token prefix of every (b, kvh) unit of a
    workload, on a thread pool (ctypes releases the GIL during each oracle call)."""

    def __init__(self, w, seconds_target=12.0, threads=None):
        import oracle
        self.oracle = oracle
        self.w = w
        self.threads = threads or len(os.sched_getaffinity(0))
        self.ok_k = oracle.Codec(w.d, w.k_bits, w.rot_seed)
        self.ok_v = oracle.Codec(w.d, w.v_bits, w.rot_seed)
        self.units = [(b, h) for b in range(w.B) for h in range(w.Hkv)]
        self.q = w.q()
        self.n = 256
        self._prep()
        dt = self.run()
        n = int(min(w.S, max(256, self.n * seconds_target / max(dt, 1e-3))))
        self.n = max(256, n // 8 * 8)
        self._prep()
        self.used = min(self.threads, len(self.units))

    def _prep(self):
        w, n = self.w, self.n
        self.data = []
        for b, h in self.units:
            K, V = w.k_slice(b, h, n), w.v_slice(b, h, n)
            kc, kn = (K, None) if w.k_bits == 16 else self.ok_k.encode(K)[:2]
            vc, vn = self.ok_v.encode(V)[:2]
            self.data.append((b, h, kc, kn, vc, vn))

    def run(self):
        from concurrent.futures import ThreadPoolExecutor
        w, n = self.w, self.n

        def one(t):
            b, h, kc, kn, vc, vn = t
            self.oracle.attention_unit(self.ok_k, self.ok_v, self.q[b, h * w.G:(h + 1) * w.G], kc, kn, vc, vn, n,
                                       1 / math.sqrt(w.d))

        t0 = time.perf_counter()
        with ThreadPoolExecutor(min(self.threads, len(self.data))) as ex:
            list(ex.map(one, self.data))
        return time.perf_counter() - t0

    def bytes(self):
        w = self.w
        kb = w.d * 2 if w.k_bits == 16 else w.d * w.k_bits // 8 + 2
        vb = w.d * w.v_bits // 8 + 2
        return self.n * len(self.units) * (kb + vb)

    def describe(self):
        w = self.w
        return (f"oracle decode attention over the first {self.n} of {w.S} tokens of all {len(self.units)} "
                f"(batch, kv-head) units of {w.name} on {self.used} threads")


def reference_arm(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    w = tq_inputs.WORKLOADS[args.workload]
    per_step = min(args.ref_seconds, 150.0 / (args.steps + args.warmup))
    smp = OracleSample(w, seconds_target=per_step)
    per = []
    for i in range(args.warmup + args.steps):
        dt = smp.run()
        if i >= args.warmup:
            per.append(smp.bytes() / dt / 1e9)
    v = statistics.median(per)
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{w.name}: B{w.B} Hq{w.Hq} Hkv{w.Hkv} d{w.d} S{w.S} K{w.k_bits}/V{w.v_bits}"},
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": smp.used, "kind": "oracle",
                             "sample": smp.describe()},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- GPU arm
# integer-equivalent instructions per encoded vector (lane operations), the bound the
# exact encode is held to: the int64 butterfly (d log2 d add/subs, two 32-bit
# operations each), the exact 128-bit square sum (~5 per element), the b-step
# binary search (compare + select per step) and the packing (~3 per element)
def encode_lane_ops(d, bits):
    return 2 * d * int(math.log2(d)) + 5 * d + (2 * bits + 3) * d


def encode_sweep(tq, dev, stream, peak_gbs, sm_mhz, sizes=None, d=256, bits_list=(3, 4), seed=0, rot_seed=42):
    """Encode throughput over batch sizes (the head-dim-256 workload's codecs: 3-bit K/V and
    the 4-bit V of the raw-key scheme).  Each size runs back-to-back calls replayed from a
    CUDA graph; call r reads vectors [(r N) mod 2^20, +N) of a 2^20-vector input (512 MB),
    so sizes >= 2^18 stream from HBM and smaller ones are latency-bound and L2-resident."""
    import torch
    sizes = sizes or tq_inputs.ENCODE_SWEEP
    NMAX = max(sizes)
    base = 1 << 16
    blk = torch.from_numpy(tq_inputs.fp16_normal(tq_inputs.stream_seed(seed, 7, 0), (base, d))).to(dev)
    x = blk.repeat((NMAX + base - 1) // base, 1)[:NMAX].contiguous()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    lane_rate = sms * 128 * sm_mhz * 1e6                     # 32-bit lane operations per second
    out = []
    for bits in bits_list:
        c = tq.tq_codec_create(d, bits, rot_seed)
        codes = torch.empty((NMAX, c.bytes_per_vec), dtype=torch.uint8, device=dev)
        norms = torch.empty(NMAX, dtype=torch.float16, device=dev)
        for N in sizes:
            calls = max(4, min(256, (1 << 22) // N))
            offs = [(r * N) % NMAX for r in range(calls)]

            def run():
                for o in offs:
                    tq.tq_encode(c, x[o:o + N], codes[o:o + N], norms[o:o + N])
            run()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                run()
            g.replay()
            torch.cuda.synchronize()
            ts = []
            for _ in range(3):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                _lead()
                e0.record(stream)
                g.replay()
                e1.record(stream)
                torch.cuda.synchronize()
                ts.append(e0.elapsed_time(e1) * 1e-3 / calls)
            t = statistics.median(ts)
            bpv = 2 * d + c.bytes_per_vec + 2
            out.append({"n_vec": N, "dim": d, "bits": bits, "us_per_call": t * 1e6, "Mvec_s": N / t / 1e6,
                        "hbm_frac": N * bpv / t / 1e9 / peak_gbs,
                        "intop_frac": N * encode_lane_ops(d, bits) / t / lane_rate})
        del codes, norms
    return {"points": out, "bytes_per_vec": "2d + d*b/8 + 2",
            "intop_bound": f"lane ops per vector 2 d log2 d + 5 d + (2 b + 3) d at {sms} SMs x 128 lanes x "
                           f"{sm_mhz:.0f} MHz"}


def e2e_from_c(tq, ck, cv, w, K, V, q, lens, pos, k_new, v_new, out, kc, kn, vc, vn, R, wsb, stream, steps,
               warmup, PB, bytes_step, world, graph_steps=0):
    """The same steps driven from a C loop over the C ABI (libtq_e2e.so): per step the
    host->device copy of q and the lengths from pinned memory on a copy stream (every 64th
    step also the pending K/V batch and its positions, then tq_encode_append_kv), one
    tq_decode_attend, and the device->host copy of the output; CUDA events on the stream."""
    import ctypes
    import torch
    path = os.path.join(ROOT, "quantized_kv_cache_10_gb300", "libtq_e2e.so")
    if not os.path.exists(path):
        return None
    lib = ctypes.CDLL(path)
    f = lib.tq_e2e_decode_steps
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    f.argtypes = [vp, vp, i32, i32, i32, i64, i32, vp, sz, sz] + [vp] * 4 + [vp, vp, vp, vp, i32, vp, sz] + \
        [vp] * 5 + \
        [i32, i32, i32, vp] + [ctypes.POINTER(ctypes.c_double)] * 4
    f.restype = i32
    # the step's inputs in one staging buffer: the query block, then the lengths (16-byte aligned)
    qb = w.B * w.Hq * w.d * 2
    off = (qb + 15) // 16 * 16
    h_in = torch.zeros(off + 4 * w.B, dtype=torch.uint8).pin_memory()
    h_in[:qb].copy_(torch.from_numpy(w.q()).view(torch.uint8).reshape(-1))
    h_in[off:].copy_(torch.from_numpy(w.lengths()).view(torch.uint8))
    stride = (h_in.numel() + 255) // 256 * 256                 # two device input buffers (ping-pong)
    d_in = torch.empty(2 * stride, dtype=torch.uint8, device=q.device)
    h_pos = torch.from_numpy(w.lengths() - PB).pin_memory()
    h_k = torch.from_numpy(np.ascontiguousarray(K[:, :, -PB:])).pin_memory()
    h_v = torch.from_numpy(np.ascontiguousarray(V[:, :, -PB:])).pin_memory()
    h_out = torch.empty((2, w.B, w.Hq, w.d), dtype=torch.float16).pin_memory()
    d_out2 = torch.empty((2, w.B, w.Hq, w.d), dtype=torch.float16, device=q.device)
    sec, hsec, h2d, d2h = ctypes.c_double(), ctypes.c_double(), ctypes.c_double(), ctypes.c_double()
    if graph_steps:                       # a stream that can be captured (not the legacy default stream)
        torch.cuda.synchronize()
        stream = torch.cuda.Stream()
    rc = f(ck.handle, cv.handle, w.B, w.Hq, w.Hkv, w.S, PB, d_in.data_ptr(), off, stride, pos.data_ptr(),
           k_new.data_ptr(), v_new.data_ptr(), d_out2.data_ptr(), kc.data_ptr(), kn.data_ptr(), vc.data_ptr(),
           vn.data_ptr(), R, wsb.data_ptr(), wsb.numel(), h_in.data_ptr(), h_pos.data_ptr(),
           h_k.data_ptr(), h_v.data_ptr(), h_out.data_ptr(), warmup, steps, graph_steps, stream.cuda_stream,
           ctypes.byref(sec), ctypes.byref(hsec), ctypes.byref(h2d), ctypes.byref(d2h))
    if rc != 0:
        raise RuntimeError(f"end-to-end C loop failed with code {rc}")
    v = job_throughput(bytes_step * steps, world, max_over_ranks(sec.value, q.device)) / 1e9
    if graph_steps:
        return {"value": v, "unit": "GB/s", "h2d_bytes_per_step": h2d.value, "d2h_bytes_per_step": d2h.value,
                "host_us_per_step": hsec.value * 1e6,
                "driver": f"the same C loop's steps captured once as CUDA graphs of {graph_steps} steps (copies, "
                          "encode and decode-attention calls as recorded) and replayed"}
    return {"value": v, "unit": "GB/s", "h2d_bytes_per_step": h2d.value, "d2h_bytes_per_step": d2h.value,
            "host_us_per_step": hsec.value * 1e6,
            "driver": "C loop over the C ABI (libtq_e2e.so): per step one cudaMemcpyAsync of the query block and "
                      "lengths (pinned, double-buffered, on an input copy stream overlapping the previous step), one "
                      "tq_decode_attend, one cudaMemcpyAsync of the output back (double-buffered, own stream); every 64th "
                      "step the K/V batch "
                      "copies and tq_encode_append_kv"}


def gpu_arm(args):
    import torch
    ws_, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws_ > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    import quantized_kv_cache_10_gb300 as tq

    w = tq_inputs.WORKLOADS[args.workload]
    ck = tq.tq_codec_create(w.d, w.k_bits, w.rot_seed)
    cv = tq.tq_codec_create(w.d, w.v_bits, w.rot_seed)
    bytes_step = w.packed_kv_bytes()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    # Inputs larger than L2: R replicas of the packed cache, cycled, so a replica
    # is evicted (>= 4x L2 of other traffic) before it is read again.  Caches too
    # small for that (R > 64) are measured one call at a time after an L2 flush.
    need = max(2, math.ceil(4 * l2 / bytes_step))
    R = 1 << (need - 1).bit_length()
    replica_mode = R <= 64
    if not replica_mode:
        R = 1
    # prefill: generate K/V on the host, encode the whole cache on the GPU (replica 0)
    K, V = w.kv("k", 16), w.kv("v", 16)
    n = w.B * w.Hkv * w.S
    vc = torch.empty((R, w.B, w.Hkv, w.S, cv.bytes_per_vec), dtype=torch.uint8, device=dev)
    vn = torch.empty((R, w.B, w.Hkv, w.S), dtype=torch.float16, device=dev)
    Kd, Vd = torch.from_numpy(K).to(dev), torch.from_numpy(V).to(dev)
    if w.k_bits == 16:                                       # raw fp16 keys (turbo0v*): stored as they are
        kc = torch.empty((R, w.B, w.Hkv, w.S, w.d), dtype=torch.float16, device=dev)
        kc[0].copy_(Kd)
        kn = None
    else:
        kc = torch.empty((R, w.B, w.Hkv, w.S, ck.bytes_per_vec), dtype=torch.uint8, device=dev)
        kn = torch.empty((R, w.B, w.Hkv, w.S), dtype=torch.float16, device=dev)
    # encode throughput of the prefill (one launch per tensor), events on this stream
    enc_times = []
    n_enc = n if w.k_bits == 16 else 2 * n
    for i in range(4):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        if w.k_bits != 16:
            tq.tq_encode(ck, Kd.view(n, w.d), kc[0].view(n, -1), kn[0].view(-1))
        tq.tq_encode(cv, Vd.view(n, w.d), vc[0].view(n, -1), vn[0].view(-1))
        e1.record()
        torch.cuda.synchronize()
        if i > 0:
            enc_times.append(e0.elapsed_time(e1) * 1e-3)
    enc_mvec = n_enc / statistics.median(enc_times) / 1e6
    del Kd, Vd
    for r in range(1, R):
        kc[r].copy_(kc[0])
        vc[r].copy_(vc[0])
        vn[r].copy_(vn[0])
        if kn is not None:
            kn[r].copy_(kn[0])
    q = torch.from_numpy(w.q()).to(dev)
    lens = torch.from_numpy(w.lengths()).to(dev)
    PB = 64                                                  # pending-token batch
    pos = (lens - PB).to(torch.int32)                        # the batch is the last 64 cached tokens
    k_new = torch.from_numpy(np.ascontiguousarray(K[:, :, -PB:])).to(dev)
    v_new = torch.from_numpy(np.ascontiguousarray(V[:, :, -PB:])).to(dev)
    out = torch.empty((w.B, w.Hq, w.d), dtype=torch.float16, device=dev)
    wsb = torch.empty(tq.tq_decode_attend_workspace_bytes(w.B, w.Hq, w.Hkv, w.S, w.d), dtype=torch.uint8, device=dev)
    tq.tq_workspace_init(wsb)
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def encode_batch(r):
        if w.k_bits == 16:
            kc[r, :, :, -PB:].copy_(k_new)                   # raw fp16 keys are stored as they are
            tq.tq_encode_append(cv, v_new, pos, vc[r], vn[r])
        else:
            tq.tq_encode_append_kv(ck, cv, k_new, v_new, pos, kc[r], kn[r], vc[r], vn[r])   # one launch

    def attend(r):
        tq.tq_decode_attend(ck, cv, q, kc[r], None if kn is None else kn[r], vc[r], vn[r], lens, out, wsb)

    def step(i):
        if i % PB == 0:
            encode_batch(i % R)
        attend(i % R)

    enc_launches = 1                                         # our kernels per pending-batch encode
    launches = 2 * args.steps + enc_launches * ((args.steps + PB - 1) // PB)

    def capture(fn, count):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(count):
                fn(i)
        return g

    for i in range(args.warmup):
        if not replica_mode:
            flush.zero_()
        step(i)
    torch.cuda.synchronize()
    graphs = None
    if replica_mode:
        try:
            tail = args.steps % PB
            graphs = (capture(step, PB), capture(step, tail) if tail else None,
                      capture(lambda i: attend(i % R), PB))
            for g in graphs:
                if g is not None:
                    g.replay()
            torch.cuda.synchronize()
        except Exception as exc:                             # capture unsupported: eager launches
            print(f"# CUDA graph capture failed ({exc}); timing eager launches", file=sys.stderr)
            graphs = None
    if ws_ > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with Clocks(local) as clk:
        if replica_mode:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            _lead()
            e0.record(stream)
            if graphs:
                for _ in range(args.steps // PB):
                    graphs[0].replay()
                if graphs[1] is not None:
                    graphs[1].replay()
            else:
                for i in range(args.steps):
                    step(i)
            e1.record(stream)
            torch.cuda.synchronize()
            tot = e0.elapsed_time(e1) * 1e-3
            # the decode-attention call alone (no pending-batch encodes), same replicas
            reps = max(8, args.steps // PB)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            _lead()
            e0.record(stream)
            for j in range(reps):
                if graphs:
                    graphs[2].replay()
                else:
                    for i in range(PB):
                        attend(i % R)
            e1.record(stream)
            torch.cuda.synchronize()
            dec_mean = e0.elapsed_time(e1) * 1e-3 / (reps * PB)
        else:
            step_t, dec_t = [], []
            for i in range(args.steps):
                flush.zero_()
                e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
                _lead()
                e0.record(stream)
                if i % PB == 0:
                    encode_batch(0)
                e1.record(stream)
                attend(0)
                e2.record(stream)
                torch.cuda.synchronize()
                step_t.append(e0.elapsed_time(e2) * 1e-3)
                dec_t.append(e1.elapsed_time(e2) * 1e-3)
            tot = sum(step_t)
            dec_mean = statistics.mean(dec_t)
    torch.cuda.synchronize()
    assert tq.tq_get_device_error(wsb) == 0
    tot = max_over_ranks(tot, dev)
    if ws_ > 1:
        torch.distributed.barrier()
    value = job_throughput(bytes_step * args.steps, ws_, tot) / 1e9
    peak, peak_kind = _peaks()
    achieved = bytes_step / dec_mean / 1e9

    # the same decode-attention call with a 63-token unencoded fp16 tail (the most a
    # pending batch holds before it is encoded), read in the same softmax
    tail_us = None
    if replica_mode and graphs:
        TT = 63
        k_tail = torch.from_numpy(np.ascontiguousarray(K[:, :, :PB])).to(dev)
        v_tail = torch.from_numpy(np.ascontiguousarray(V[:, :, :PB])).to(dev)
        tlens = torch.full((w.B,), TT, dtype=torch.int32, device=dev)

        def attend_tail(i):
            r = i % R
            tq.tq_decode_attend_tail(ck, cv, q, kc[r], None if kn is None else kn[r], vc[r], vn[r], lens, k_tail,
                                     v_tail, tlens, out, wsb)

        gt = capture(attend_tail, PB)
        gt.replay()
        torch.cuda.synchronize()
        reps = max(8, args.steps // PB)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        _lead()
        e0.record(stream)
        for j in range(reps):
            gt.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        tail_us = e0.elapsed_time(e1) * 1e3 / (reps * PB)

    # speculative verification: the same cache attended by L = 4 query positions per head
    # (4 drafted tokens held as the fp16 tail), causal, one decode + combine launch pair
    multi = None
    if replica_mode and graphs:
        LQ = 4
        mq = torch.from_numpy(tq_inputs.fp16_normal(tq_inputs.stream_seed(w.seed, tq_inputs.Q_ID, 1),
                                                    (w.B, w.Hq, LQ, w.d))).to(dev)
        mout = torch.empty((w.B, w.Hq, LQ, w.d), dtype=torch.float16, device=dev)
        mws = torch.empty(tq.tq_decode_attend_multi_workspace_bytes(w.B, w.Hq, w.Hkv, LQ, w.S, w.d),
                          dtype=torch.uint8, device=dev)
        tq.tq_workspace_init(mws)
        mk = torch.from_numpy(np.ascontiguousarray(K[:, :, :LQ])).to(dev)
        mv = torch.from_numpy(np.ascontiguousarray(V[:, :, :LQ])).to(dev)
        mlens = torch.full((w.B,), LQ, dtype=torch.int32, device=dev)

        def attend_multi(i):
            r = i % R
            tq.tq_decode_attend_multi(ck, cv, mq, kc[r], None if kn is None else kn[r], vc[r], vn[r], lens, mout,
                                      mws, k_tail=mk, v_tail=mv, tail_lens=mlens)

        gm = capture(attend_multi, PB)
        gm.replay()
        torch.cuda.synchronize()
        reps = max(8, args.steps // PB)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        _lead()
        e0.record(stream)
        for j in range(reps):
            gm.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        m_us = e0.elapsed_time(e1) * 1e3 / (reps * PB)
        multi = {"query_positions": LQ, "fp16_tail_tokens": LQ, "call_us": m_us,
                 "packed_GBps": bytes_step / (m_us * 1e-6) / 1e9}

    # keys with the QJL residual sketch (TurboQuantProd: 3-bit MSE codes + 1 sign bit per
    # sketch row + residual norm) on the same shape, values as above
    qjl = None
    if replica_mode and graphs and (w.d & (w.d - 1)) == 0:
        qb = 3
        cq = tq.tq_codec_create_qjl(w.d, qb, w.rot_seed)
        qkc = torch.empty((R, w.B, w.Hkv, w.S, cq.bytes_per_vec), dtype=torch.uint8, device=dev)
        qkn = torch.empty((R, w.B, w.Hkv, w.S), dtype=torch.float16, device=dev)
        qks = torch.empty((R, w.B, w.Hkv, w.S, w.d // 8), dtype=torch.uint8, device=dev)
        qkr = torch.empty((R, w.B, w.Hkv, w.S), dtype=torch.float16, device=dev)
        Kd = torch.from_numpy(K).to(dev)
        qenc = []
        for i in range(3):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            _lead()
            e0.record(stream)
            tq.tq_encode_qjl(cq, Kd.view(n, w.d), qkc[0].view(n, -1), qkn[0].view(-1), qks[0].view(n, -1),
                             qkr[0].view(-1))
            e1.record(stream)
            torch.cuda.synchronize()
            if i > 0:
                qenc.append(e0.elapsed_time(e1) * 1e-3)
        del Kd
        for r in range(1, R):
            qkc[r].copy_(qkc[0])
            qkn[r].copy_(qkn[0])
            qks[r].copy_(qks[0])
            qkr[r].copy_(qkr[0])

        def attend_qjl(i):
            r = i % R
            tq.tq_decode_attend_qjl(cq, cv, q, qkc[r], qkn[r], qks[r], qkr[r], vc[r], vn[r], lens, out, wsb)

        gq = capture(attend_qjl, PB)
        gq.replay()
        torch.cuda.synchronize()
        reps = max(4, args.steps // (4 * PB))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        _lead()
        e0.record(stream)
        for j in range(reps):
            gq.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        q_us = e0.elapsed_time(e1) * 1e3 / (reps * PB)
        qbytes = int(w.lengths().astype(np.int64).sum()) * w.Hkv * (
            cq.bytes_per_vec + 2 + w.d // 8 + 2 + cv.bytes_per_vec + 2)
        qjl = {"k_mse_bits": qb, "sketch_rows": w.d, "packed_bytes": qbytes, "call_us": q_us,
               "GBps": qbytes / (q_us * 1e-6) / 1e9, "kernel": "tensor-core (mma.sync)",
               "encode_Mvec_s": n / statistics.median(qenc) / 1e6}
        del qkc, qkn, qks, qkr

    # one call on its own after an L2 flush (latency of an isolated decode step)
    iso = []
    for i in range(16):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        _lead()
        e0.record(stream)
        attend(0)
        e1.record(stream)
        torch.cuda.synchronize()
        iso.append(e0.elapsed_time(e1) * 1e3)

    # encode throughput sweep over batch sizes (1 .. 2^20 vectors, head dim 256, 3 and 4 bits)
    sweep = None
    if not args.no_encode_sweep:
        sweep = encode_sweep(tq, dev, stream, peak, _sm_mhz())

    # ---- end to end through the C ABI, driven from C: pinned host inputs in, output back ----
    e2e_c = e2e_g = None
    if w.k_bits != 16 and replica_mode:
        e2e_c = e2e_from_c(tq, ck, cv, w, K, V, q, lens, pos, k_new, v_new, out, kc, kn, vc, vn, R, wsb, stream,
                           args.steps, args.warmup, PB, bytes_step, ws_)
        e2e_g = e2e_from_c(tq, ck, cv, w, K, V, q, lens, pos, k_new, v_new, out, kc, kn, vc, vn, R, wsb, stream,
                           max(args.steps, PB), args.warmup, PB, bytes_step, ws_, graph_steps=PB)

    # ---- end to end through the Python binding: pinned host inputs in, output back ----
    h_q = torch.from_numpy(w.q()).pin_memory()
    h_k = torch.from_numpy(np.ascontiguousarray(K[:, :, -PB:])).pin_memory()
    h_v = torch.from_numpy(np.ascontiguousarray(V[:, :, -PB:])).pin_memory()
    h_len = torch.from_numpy(w.lengths()).pin_memory()
    h_out = torch.empty((w.B, w.Hq, w.d), dtype=torch.float16).pin_memory()

    def e2e_step(i):
        q.copy_(h_q, non_blocking=True)
        lens.copy_(h_len, non_blocking=True)
        h2d = h_q.numel() * 2 + h_len.numel() * 4
        if i % PB == 0:
            k_new.copy_(h_k, non_blocking=True)
            v_new.copy_(h_v, non_blocking=True)
            torch.sub(lens, PB, out=pos)
            encode_batch(i % R)
            h2d += h_k.numel() * 2 + h_v.numel() * 2
        attend(i % R)
        h_out.copy_(out, non_blocking=True)
        return h2d

    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize()
    h2d_tot = 0
    if replica_mode:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(args.steps):
            h2d_tot += e2e_step(i)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_tot = e0.elapsed_time(e1) * 1e-3
    else:
        e2e_tot = 0.0
        for i in range(args.steps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            h2d_tot += e2e_step(i)
            e1.record(stream)
            torch.cuda.synchronize()
            e2e_tot += e0.elapsed_time(e1) * 1e-3
    h2d = h2d_tot / args.steps
    d2h = h_out.numel() * 2
    e2e_v = job_throughput(bytes_step * args.steps, ws_, max_over_ranks(e2e_tot, dev)) / 1e9

    if rank != 0:
        if ws_ > 1:
            torch.distributed.destroy_process_group()
        return
    cpu = None
    if ws_ == 1 and not args.no_cpu_baseline:
        smp = OracleSample(w, seconds_target=args.ref_seconds)
        dt = smp.run()
        cpu = {"value": smp.bytes() / dt / 1e9, "unit": "GB/s", "cores": smp.used, "kind": "oracle",
               "sample": smp.describe()}
    kname = "decode_attend"
    if replica_mode:
        l2note = (f"inputs larger than L2: {R} replicas of the packed cache "
                  f"({R * bytes_step / 1e6:.0f} MB, >= 4x the {l2 / 1e6:.0f} MB L2) cycled, no flush; "
                  f"steps replayed from CUDA graphs of {PB} steps" if graphs else
                  f"inputs larger than L2: {R} replicas of the packed cache cycled, no flush; eager launches")
    else:
        l2note = "flushed before every step (write of 2x L2), the flush outside the timed events"
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws_, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": tot / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"{w.name}: B{w.B} Hq{w.Hq} Hkv{w.Hkv} d{w.d} S{w.S} K{w.k_bits}/V{w.v_bits}",
                   "step": "fused decode attention; every 64th step first encodes the 64-token pending batch (K,V)",
                   "packed_kv_bytes": bytes_step, "l2": l2note, "parallelism": f"replicas x{ws_}"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": _traffic(kname), "peak_kind": peak_kind,
                     "kernel": kname, "decode_us": dec_mean * 1e6,
                     "note": "one decode-attention call (decode kernel + split-K combine kernel) per launch"},
        "isolated_call_us": statistics.median(iso),
        "with_fp16_tail": {"tail_tokens": 63, "call_us": tail_us},
        "multi_query": multi,
        "qjl": qjl,
        "encode": {"value": enc_mvec, "unit": "Mvec/s", "n_vec": n_enc, "dim": w.d},
        "encode_sweep": sweep,
        "e2e": e2e_c if e2e_c else {"value": e2e_v, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                                    "d2h_bytes_per_step": d2h, "driver": "Python binding"},
        "e2e_graph": e2e_g,
        "e2e_python": {"value": e2e_v, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                       "driver": "Python binding (ctypes) per call"},
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    if ws_ > 1:
        torch.distributed.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=16384)
    ap.add_argument("--warmup", type=int, default=64)
    ap.add_argument("--impl", default="tq", choices=["tq", "reference"])
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(tq_inputs.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-seconds", type=float, default=12.0)
    ap.add_argument("--no-encode-sweep", action="store_true")
    args = ap.parse_args()
    if args.impl == "reference":
        reference_arm(args)
    else:
        gpu_arm(args)


if __name__ == "__main__":
    main()
