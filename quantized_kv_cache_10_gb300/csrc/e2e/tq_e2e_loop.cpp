// tq_e2e_loop.cpp -- end-to-end decode steps driven from C through the public C ABI
// (include/tq.h), for the benchmark's end-to-end figure.  Built as its own library
// (libtq_e2e.so, linked against libtq.so); nothing of the hot path lives here.
//
// One step, as a serving loop issues it: the step's inputs (the query block followed
// by the sequence lengths, one pinned staging buffer) go host->device on an input copy
// stream into one of two device input buffers while the previous step computes; the
// compute stream waits for that copy, runs (every 64th step) tq_encode_append_kv of
// the pending K / V batch copied the same way, then one tq_decode_attend into one of
// two output buffers; an output copy stream waits for it and reads the output back
// into one of two pinned host buffers.  Every
// step's copies are inside the timed region.  Step i uses cache replica i mod R
// (replicas laid out back to back), so reads come from HBM.  Timed with CUDA events
// recorded on the compute stream after joining the copy stream; the host's own
// enqueue time per step is returned beside it.  With graph_steps > 0 the same steps
// are captured once as CUDA graphs of graph_steps steps and replayed.
#include <chrono>
#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "tq.h"

namespace {

struct Rep {
    uint8_t* kc;
    uint16_t* kn;
    uint8_t* vc;
    uint16_t* vn;
};

}  // namespace

extern "C" {

// Returns 0 on success, a tq_status of a failed call, or 100 + a CUDA error code.
int tq_e2e_decode_steps(const tq_codec* ck, const tq_codec* cv, int B, int n_q_heads, int n_kv_heads,
                        int64_t max_seq, int pending_batch,
                        // two device input buffers (query block, then the lengths at byte offset
                        // lens_offset) back to back, each in_stride bytes; positions, pending K / V
                        // batch, and two output blocks back to back
                        uint8_t* d_in, size_t lens_offset, size_t in_stride, int32_t* d_pos, uint16_t* d_knew,
                        uint16_t* d_vnew, uint16_t* d_out,
                        // cache replicas: R back-to-back copies of codes and norms
                        uint8_t* kc, uint16_t* kn, uint8_t* vc, uint16_t* vn, int R, void* ws, size_t ws_bytes,
                        // pinned host buffers: the staged inputs, positions, K / V batch, two outputs
                        const uint8_t* h_in, const int32_t* h_pos, const uint16_t* h_knew, const uint16_t* h_vnew,
                        uint16_t* h_out, int warmup, int steps, int graph_steps, void* stream, double* seconds,
                        double* host_seconds, double* h2d_bytes_per_step, double* d2h_bytes_per_step) {
    if (!ck || !cv || R <= 0 || steps <= 0 || pending_batch <= 0) return TQ_ERR_INVALID_ARG;
    int dim = 0, kbits = 0, vbits = 0, kbpv = 0, vbpv = 0, wht = 0;
    tq_codec_info(ck, &dim, &kbits, &kbpv, &wht, nullptr);
    tq_codec_info(cv, &dim, &vbits, &vbpv, &wht, nullptr);
    if (kbits == 16) return TQ_ERR_UNSUPPORTED;  // raw keys are copied, not encoded: not driven here
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t units = static_cast<size_t>(B) * n_kv_heads;
    const size_t rows = units * static_cast<size_t>(max_seq);
    const size_t q_bytes = static_cast<size_t>(B) * n_q_heads * dim * 2;
    const size_t len_bytes = static_cast<size_t>(B) * 4;
    const size_t new_bytes = units * pending_batch * dim * 2;
    if (lens_offset < q_bytes || lens_offset % 16 || in_stride < lens_offset + len_bytes || in_stride % 256)
        return TQ_ERR_INVALID_ARG;
    const size_t in_bytes = lens_offset + len_bytes;
    // input copies and output copies on streams of their own, so that the next step's input
    // copy does not queue behind this step's output read (which waits for this step's compute)
    cudaStream_t cp = nullptr, co = nullptr;
    cudaEvent_t in_ready[2], in_free[2], out_ready[2], e0, e1, joined;
    cudaError_t e = cudaStreamCreateWithFlags(&cp, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&co, cudaStreamNonBlocking);
    if (e != cudaSuccess) return 100 + e;
    for (int i = 0; i < 2; ++i) {
        cudaEventCreateWithFlags(&in_ready[i], cudaEventDisableTiming);
        cudaEventCreateWithFlags(&in_free[i], cudaEventDisableTiming);
        cudaEventCreateWithFlags(&out_ready[i], cudaEventDisableTiming);
    }
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    cudaEventCreateWithFlags(&joined, cudaEventDisableTiming);
    auto rep = [&](int r) {
        return Rep{kc + static_cast<size_t>(r) * rows * kbpv, kn + static_cast<size_t>(r) * rows,
                   vc + static_cast<size_t>(r) * rows * vbpv, vn + static_cast<size_t>(r) * rows};
    };
    double h2d = 0.0;
    bool first[2] = {true, true};
    auto step = [&](int i) -> int {
        const int j = i & 1;
        uint8_t* din = d_in + j * in_stride;
        const Rep c = rep(i % R);
        // inputs of step i: copy stream, once buffer j is no longer read by step i - 2
        if (!first[j] && (e = cudaStreamWaitEvent(cp, in_free[j], 0)) != cudaSuccess) return 100 + e;
        if ((e = cudaMemcpyAsync(din, h_in, in_bytes, cudaMemcpyHostToDevice, cp)) != cudaSuccess) return 100 + e;
        h2d += static_cast<double>(in_bytes);
        if (i % pending_batch == 0) {
            if ((e = cudaMemcpyAsync(d_knew, h_knew, new_bytes, cudaMemcpyHostToDevice, cp)) != cudaSuccess) return 100 + e;
            if ((e = cudaMemcpyAsync(d_vnew, h_vnew, new_bytes, cudaMemcpyHostToDevice, cp)) != cudaSuccess) return 100 + e;
            if ((e = cudaMemcpyAsync(d_pos, h_pos, len_bytes, cudaMemcpyHostToDevice, cp)) != cudaSuccess) return 100 + e;
            h2d += 2.0 * new_bytes + len_bytes;
        }
        cudaEventRecord(in_ready[j], cp);
        // compute: the pending-batch encode every 64th step, then the decode attention into
        // output buffer j, once step i - 2's read of it is done
        if ((e = cudaStreamWaitEvent(st, in_ready[j], 0)) != cudaSuccess) return 100 + e;
        if (!first[j] && (e = cudaStreamWaitEvent(st, out_ready[j], 0)) != cudaSuccess) return 100 + e;
        uint16_t* dout = d_out + j * (q_bytes / 2);
        if (i % pending_batch == 0) {
            const tq_status s = tq_encode_append_kv(ck, cv, d_knew, d_vnew, B, n_kv_heads, pending_batch, d_pos,
                                                    max_seq, c.kc, c.kn, c.vc, c.vn, nullptr, stream);
            if (s != TQ_OK) return s;
        }
        const tq_status s = tq_decode_attend(ck, cv, reinterpret_cast<const uint16_t*>(din), c.kc, c.kn, c.vc, c.vn,
                                             reinterpret_cast<const int32_t*>(din + lens_offset), B, n_q_heads,
                                             n_kv_heads, max_seq, 1.0f / __builtin_sqrtf(static_cast<float>(dim)),
                                             dout, ws, ws_bytes, stream);
        if (s != TQ_OK) return s;
        cudaEventRecord(in_free[j], st);
        first[j] = false;
        // the output back to the host on the output copy stream (after the step's compute)
        if ((e = cudaStreamWaitEvent(co, in_free[j], 0)) != cudaSuccess) return 100 + e;
        if ((e = cudaMemcpyAsync(h_out + j * (q_bytes / 2), dout, q_bytes, cudaMemcpyDeviceToHost, co)) !=
            cudaSuccess)
            return 100 + e;
        cudaEventRecord(out_ready[j], co);
        return 0;
    };
    // the compute stream waits for both copy streams' work so far
    auto join = [&]() {
        cudaEventRecord(joined, cp);
        cudaStreamWaitEvent(st, joined, 0);
        cudaEventRecord(joined, co);
        cudaStreamWaitEvent(st, joined, 0);
    };
    // graph_steps > 0: the steps are captured once as CUDA graphs of graph_steps steps (the
    // copies, the encode and the decode-attention calls as recorded) and replayed
    cudaGraphExec_t gexec = nullptr;
    auto capture = [&](int count) -> int {
        cudaGraph_t g = nullptr;
        cudaError_t ce = cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal);
        if (ce != cudaSuccess) return 100 + ce;
        cudaEventRecord(joined, st);                // the copy streams join the capture
        cudaStreamWaitEvent(cp, joined, 0);
        cudaStreamWaitEvent(co, joined, 0);
        first[0] = first[1] = true;
        int r2 = 0;
        for (int i = 0; i < count && r2 == 0; ++i) r2 = step(i);
        join();
        ce = cudaStreamEndCapture(st, &g);
        if (r2) return r2;
        if (ce != cudaSuccess) return 100 + ce;
        ce = cudaGraphInstantiate(&gexec, g, 0);
        cudaGraphDestroy(g);
        return ce == cudaSuccess ? 0 : 100 + ce;
    };
    int rc = 0;
    for (int i = 0; i < warmup && rc == 0; ++i) rc = step(i);
    double graph_h2d = 0.0;  // bytes copied to the device by one captured graph
    if (rc == 0 && graph_steps > 0) {
        const double before = h2d;
        rc = capture(graph_steps);
        graph_h2d = h2d - before;
        if (rc == 0) rc = cudaGraphLaunch(gexec, st) == cudaSuccess ? 0 : 100;  // one warm replay
    }
    if (rc == 0) {
        join();
        e = cudaStreamSynchronize(st);
        if (e != cudaSuccess) rc = 100 + e;
    }
    h2d = 0.0;
    float ms = 0.0f;
    int done = steps;
    if (rc == 0) {
        const auto h0 = std::chrono::steady_clock::now();
        cudaEventRecord(e0, st);
        if (gexec) {
            done = (steps / graph_steps) * graph_steps;
            for (int i = 0; i < steps / graph_steps && rc == 0; ++i)
                if (cudaGraphLaunch(gexec, st) != cudaSuccess) rc = 100;
        } else {
            for (int i = 0; i < steps && rc == 0; ++i) rc = step(i);
        }
        join();                          // the last output read is part of the timed region
        cudaEventRecord(e1, st);
        *host_seconds = std::chrono::duration<double>(std::chrono::steady_clock::now() - h0).count() / done;
        e = cudaEventSynchronize(e1);
        if (rc == 0 && e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
        if (rc == 0 && e != cudaSuccess) rc = 100 + e;
    }
    cudaStreamSynchronize(cp);
    cudaStreamSynchronize(co);
    const bool graphed = gexec != nullptr;
    if (gexec) cudaGraphExecDestroy(gexec);
    for (int i = 0; i < 2; ++i) {
        cudaEventDestroy(in_ready[i]);
        cudaEventDestroy(in_free[i]);
        cudaEventDestroy(out_ready[i]);
    }
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    cudaEventDestroy(joined);
    cudaStreamDestroy(cp);
    cudaStreamDestroy(co);
    if (rc) return rc;
    *seconds = ms * 1e-3 * steps / done;          // per `steps` steps
    if (graphed) h2d = graph_h2d * done / graph_steps;  // the captured copies, replayed
    *h2d_bytes_per_step = h2d / done;
    *d2h_bytes_per_step = static_cast<double>(q_bytes);
    return 0;
}

}  // extern "C"
