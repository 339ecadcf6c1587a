// tq_api.cpp -- argument checking and dispatch for the C ABI in include/tq.h.
// Every check happens before anything is enqueued; a failed check returns a
// status and leaves the stream untouched.
#include <atomic>
#include <cstdint>

#include "tq_internal.h"

namespace {

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

tq_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return TQ_OK;
    if (e == cudaErrorNotSupported) return TQ_ERR_UNSUPPORTED;
    return TQ_ERR_CUDA;
}

constexpr int kMaxQueryPositions = 4096;  // tq_decode_attend_multi: L

bool on_codec_device(const tq_codec* c) {
    int d = -1;
    return cudaGetDevice(&d) == cudaSuccess && d == c->device;
}

}  // namespace

namespace {

#ifdef TQ_TIMELINE
std::atomic<unsigned long long*> g_timeline{nullptr};
std::atomic<unsigned int> g_timeline_calls{0};  // decode-attention calls since registration
#endif

}  // namespace

unsigned long long* tq::timeline_buffer() {
#ifdef TQ_TIMELINE
    return g_timeline.load();
#else
    return nullptr;
#endif
}

namespace {

tq_status decode_attend_impl(const tq_codec* ck, const tq_codec* cv, const uint16_t* q, const void* k,
                             const uint16_t* k_norms, const uint8_t* v_codes, const uint16_t* v_norms,
                             const int32_t* seq_lens, int B, int n_q_heads, int n_kv_heads, int L,
                             int64_t max_seq, const uint16_t* k_tail, const uint16_t* v_tail,
                             const int32_t* tail_lens, int max_tail, float scale, uint16_t* out, void* workspace,
                             size_t ws_bytes, void* stream, const uint8_t* k_signs = nullptr,
                             const uint16_t* k_rnorms = nullptr) {
    if (!ck || !cv || cv->bits == 16 || ck->dim != cv->dim || cv->qjl) return TQ_ERR_INVALID_ARG;
    // keys with the QJL sketch come with their sign bits and residual norms, others without
    if (bool(ck->qjl) != (k_signs != nullptr) || bool(ck->qjl) != (k_rnorms != nullptr)) return TQ_ERR_INVALID_ARG;
    if (k_signs && (!aligned(k_signs, 4) || !aligned(k_rnorms, 2))) return TQ_ERR_INVALID_ARG;
    if (!q || !k || !v_codes || !v_norms || !seq_lens || !out) return TQ_ERR_INVALID_ARG;
    if ((ck->bits == 16) != (k_norms == nullptr)) return TQ_ERR_INVALID_ARG;
    if (B <= 0 || n_q_heads <= 0 || n_kv_heads <= 0 || n_q_heads % n_kv_heads != 0) return TQ_ERR_INVALID_ARG;
    if (max_seq <= 0 || max_seq % 8 != 0 || L <= 0 || L > kMaxQueryPositions) return TQ_ERR_INVALID_ARG;
    if (!aligned(k, 16) || !aligned(v_codes, 16) || !aligned(v_norms, 16) || (k_norms && !aligned(k_norms, 16)))
        return TQ_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(out, 4) || !aligned(seq_lens, 4)) return TQ_ERR_INVALID_ARG;
    if (tail_lens) {
        if (!k_tail || !v_tail || max_tail <= 0 || !aligned(tail_lens, 4) || !aligned(k_tail, 16) ||
            !aligned(v_tail, 16))
            return TQ_ERR_INVALID_ARG;
    }
    if (!on_codec_device(ck) || !on_codec_device(cv)) return TQ_ERR_INVALID_ARG;
    tq::DecodePlan p;
    if (!tq::make_decode_plan(cv->dim, cv->device, B, n_q_heads, n_kv_heads, L, max_seq, p))
        return TQ_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, 256) || ws_bytes < p.ws_bytes) return TQ_ERR_WORKSPACE;
    tq::DecodeArgs a{tq::dev_view(ck), tq::dev_view(cv), q, k, k_norms, v_codes, v_norms, seq_lens,
                     B, n_q_heads, n_kv_heads, max_seq, scale, out, workspace,
                     tail_lens ? k_tail : nullptr, tail_lens ? v_tail : nullptr, tail_lens,
                     tail_lens ? max_tail : 0, 0, nullptr, nullptr, k_signs, k_rnorms, L};
    a.tl = tq::timeline_buffer();
#ifdef TQ_TIMELINE
    a.tl_seq = g_timeline_calls.fetch_add(1);
#endif
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaErrorNotSupported;
    if (tq::decode_mma_supported(ck, cv)) {
        p.kernel = 1;
        e = tq::launch_decode_mma(a, p, st);  // may shrink the split plan
    }
    if (e == cudaErrorNotSupported) {
        p.kernel = 0;
        e = tq::launch_decode_simt(a, p, st);
    }
    if (e != cudaSuccess) return from_cuda(e);
    return from_cuda(tq::launch_decode_combine(a, p, st));
}

}  // namespace

extern "C" {

tq_status tq_encode(const tq_codec* c, const uint16_t* x, int64_t n_vec, int64_t x_row_stride, uint8_t* codes,
                    int64_t code_row_stride, uint16_t* norms, void* stream) {
    if (!c || c->bits == 16 || n_vec < 0) return TQ_ERR_INVALID_ARG;
    if (n_vec == 0) return TQ_OK;
    if (!x || !codes || !norms) return TQ_ERR_INVALID_ARG;
    if (!aligned(x, 4) || (x_row_stride & 1) || x_row_stride < c->dim) return TQ_ERR_INVALID_ARG;
    if (!aligned(codes, 4) || (code_row_stride & 3) || code_row_stride < c->bytes_per_vec)
        return TQ_ERR_INVALID_ARG;
    if (!aligned(norms, 2) || !on_codec_device(c)) return TQ_ERR_INVALID_ARG;
    return from_cuda(tq::launch_encode(c, x, n_vec, x_row_stride, codes, code_row_stride, norms, 0, 0, 0, nullptr,
                                       0, nullptr, static_cast<cudaStream_t>(stream)));
}

tq_status tq_encode_qjl(const tq_codec* c, const uint16_t* x, int64_t n_vec, int64_t x_row_stride, uint8_t* codes,
                        int64_t code_row_stride, uint16_t* norms, uint8_t* signs, int64_t sign_row_stride,
                        uint16_t* rnorms, void* stream) {
    if (!c || !c->qjl || n_vec < 0) return TQ_ERR_INVALID_ARG;
    if (n_vec == 0) return TQ_OK;
    if (!signs || !rnorms || !aligned(signs, 4) || (sign_row_stride & 3) || sign_row_stride < c->dim / 8 ||
        !aligned(rnorms, 2))
        return TQ_ERR_INVALID_ARG;
    tq_status s = tq_encode(c, x, n_vec, x_row_stride, codes, code_row_stride, norms, stream);
    if (s != TQ_OK) return s;
    return from_cuda(tq::launch_qjl_sketch(c, x, n_vec, x_row_stride, codes, code_row_stride, norms, signs,
                                           sign_row_stride, rnorms, static_cast<cudaStream_t>(stream)));
}

tq_status tq_encode_append(const tq_codec* c, const uint16_t* x, int B, int n_kv_heads, int T,
                           const int32_t* start_pos, int64_t max_seq, uint8_t* codes, uint16_t* norms,
                           int32_t* dev_error, void* stream) {
    if (!c || c->bits == 16 || B < 0 || n_kv_heads < 0 || T < 0 || max_seq <= 0) return TQ_ERR_INVALID_ARG;
    if (B == 0 || n_kv_heads == 0 || T == 0) return TQ_OK;
    if (!x || !start_pos || !codes || !norms) return TQ_ERR_INVALID_ARG;
    if (!aligned(x, 4) || !aligned(codes, 4) || !aligned(norms, 2) || !aligned(start_pos, 4))
        return TQ_ERR_INVALID_ARG;
    if (dev_error && !aligned(dev_error, 4)) return TQ_ERR_INVALID_ARG;
    if (!on_codec_device(c)) return TQ_ERR_INVALID_ARG;
    return from_cuda(tq::launch_encode(c, x, 0, c->dim, codes, c->bytes_per_vec, norms, B, n_kv_heads, T,
                                       start_pos, max_seq, dev_error, static_cast<cudaStream_t>(stream)));
}

tq_status tq_encode_append_kv(const tq_codec* ck, const tq_codec* cv, const uint16_t* k, const uint16_t* v, int B,
                              int n_kv_heads, int T, const int32_t* start_pos, int64_t max_seq, uint8_t* k_codes,
                              uint16_t* k_norms, uint8_t* v_codes, uint16_t* v_norms, int32_t* dev_error,
                              void* stream) {
    if (!ck || !cv || ck->bits == 16 || cv->bits == 16 || ck->qjl || cv->qjl || ck->dim != cv->dim)
        return TQ_ERR_INVALID_ARG;
    if (B < 0 || n_kv_heads < 0 || T < 0 || max_seq <= 0) return TQ_ERR_INVALID_ARG;
    if (B == 0 || n_kv_heads == 0 || T == 0) return TQ_OK;
    if (!k || !v || !start_pos || !k_codes || !k_norms || !v_codes || !v_norms) return TQ_ERR_INVALID_ARG;
    if (!aligned(k, 4) || !aligned(v, 4) || !aligned(k_codes, 4) || !aligned(v_codes, 4) || !aligned(k_norms, 2) ||
        !aligned(v_norms, 2) || !aligned(start_pos, 4))
        return TQ_ERR_INVALID_ARG;
    if (dev_error && !aligned(dev_error, 4)) return TQ_ERR_INVALID_ARG;
    if (!on_codec_device(ck) || !on_codec_device(cv)) return TQ_ERR_INVALID_ARG;
    const tq::EncodeJob jobs[2] = {
        {ck, k, 0, ck->dim, k_codes, ck->bytes_per_vec, k_norms, B, n_kv_heads, T, start_pos, max_seq, dev_error, T},
        {cv, v, 0, cv->dim, v_codes, cv->bytes_per_vec, v_norms, B, n_kv_heads, T, start_pos, max_seq, dev_error, T}};
    return from_cuda(tq::launch_encode_jobs(jobs, 2, static_cast<cudaStream_t>(stream)));
}

tq_status tq_dequant(const tq_codec* c, const uint8_t* codes, const uint16_t* norms, int64_t n_vec, float* out,
                     void* stream) {
    if (!c || c->bits == 16 || n_vec < 0) return TQ_ERR_INVALID_ARG;
    if (n_vec == 0) return TQ_OK;
    if (!codes || !norms || !out || !aligned(codes, 4) || !aligned(norms, 2) || !aligned(out, 4))
        return TQ_ERR_INVALID_ARG;
    if (!on_codec_device(c)) return TQ_ERR_INVALID_ARG;
    return from_cuda(tq::launch_dequant(c, codes, norms, n_vec, out, static_cast<cudaStream_t>(stream)));
}

size_t tq_decode_attend_workspace_bytes(int B, int n_q_heads, int n_kv_heads, int64_t max_seq, int dim) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dim < 32 || dim > 512 || dim % 32) return 0;
    tq::DecodePlan p;
    if (!tq::make_decode_plan(dim, dev, B, n_q_heads, n_kv_heads, 1, max_seq, p)) return 0;
    return p.ws_bytes;
}

size_t tq_decode_attend_multi_workspace_bytes(int B, int n_q_heads, int n_kv_heads, int L, int64_t max_seq,
                                              int dim) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dim < 32 || dim > 512 || dim % 32 || L <= 0 || L > kMaxQueryPositions) return 0;
    tq::DecodePlan p;
    if (!tq::make_decode_plan(dim, dev, B, n_q_heads, n_kv_heads, L, max_seq, p)) return 0;
    return p.ws_bytes;
}

tq_status tq_workspace_init(void* ws, size_t bytes, void* stream) {
    if (!ws || bytes == 0) return TQ_ERR_INVALID_ARG;
    return from_cuda(cudaMemsetAsync(ws, 0, bytes, static_cast<cudaStream_t>(stream)));
}

tq_status tq_decode_attend(const tq_codec* ck, const tq_codec* cv, const uint16_t* q, const void* k,
                           const uint16_t* k_norms, const uint8_t* v_codes, const uint16_t* v_norms,
                           const int32_t* seq_lens, int B, int n_q_heads, int n_kv_heads, int64_t max_seq,
                           float scale, uint16_t* out, void* workspace, size_t ws_bytes, void* stream) {
    return decode_attend_impl(ck, cv, q, k, k_norms, v_codes, v_norms, seq_lens, B, n_q_heads, n_kv_heads, 1,
                              max_seq, nullptr, nullptr, nullptr, 0, scale, out, workspace, ws_bytes, stream);
}

tq_status tq_decode_attend_tail(const tq_codec* ck, const tq_codec* cv, const uint16_t* q, const void* k,
                                const uint16_t* k_norms, const uint8_t* v_codes, const uint16_t* v_norms,
                                const int32_t* seq_lens, int B, int n_q_heads, int n_kv_heads, int64_t max_seq,
                                const uint16_t* k_tail, const uint16_t* v_tail, const int32_t* tail_lens,
                                int max_tail, float scale, uint16_t* out, void* workspace, size_t ws_bytes,
                                void* stream) {
    if (!tail_lens) return TQ_ERR_INVALID_ARG;
    return decode_attend_impl(ck, cv, q, k, k_norms, v_codes, v_norms, seq_lens, B, n_q_heads, n_kv_heads, 1,
                              max_seq, k_tail, v_tail, tail_lens, max_tail, scale, out, workspace, ws_bytes,
                              stream);
}

tq_status tq_decode_attend_multi(const tq_codec* ck, const tq_codec* cv, const uint16_t* q, int L, const void* k,
                                 const uint16_t* k_norms, const uint8_t* v_codes, const uint16_t* v_norms,
                                 const int32_t* seq_lens, int B, int n_q_heads, int n_kv_heads, int64_t max_seq,
                                 const uint16_t* k_tail, const uint16_t* v_tail, const int32_t* tail_lens,
                                 int max_tail, float scale, uint16_t* out, void* workspace, size_t ws_bytes,
                                 void* stream) {
    return decode_attend_impl(ck, cv, q, k, k_norms, v_codes, v_norms, seq_lens, B, n_q_heads, n_kv_heads, L,
                              max_seq, k_tail, v_tail, tail_lens, max_tail, scale, out, workspace, ws_bytes,
                              stream);
}

tq_status tq_decode_attend_qjl(const tq_codec* ck, const tq_codec* cv, const uint16_t* q, const uint8_t* k_codes,
                               const uint16_t* k_norms, const uint8_t* k_signs, const uint16_t* k_rnorms,
                               const uint8_t* v_codes, const uint16_t* v_norms, const int32_t* seq_lens, int B,
                               int n_q_heads, int n_kv_heads, int64_t max_seq, float scale, uint16_t* out,
                               void* workspace, size_t ws_bytes, void* stream) {
    if (!ck || !ck->qjl || !k_signs || !k_rnorms) return TQ_ERR_INVALID_ARG;
    return decode_attend_impl(ck, cv, q, k_codes, k_norms, v_codes, v_norms, seq_lens, B, n_q_heads, n_kv_heads, 1,
                              max_seq, nullptr, nullptr, nullptr, 0, scale, out, workspace, ws_bytes, stream,
                              k_signs, k_rnorms);
}

tq_status tq_debug_set_timeline(void* buffer, size_t bytes) {
#ifdef TQ_TIMELINE
    const size_t need = (2ull * 2 * tq::kTlSlotsHost * tq::kTlStampsHost) * sizeof(unsigned long long);
    if (buffer && (bytes < need || !aligned(buffer, 8))) return TQ_ERR_INVALID_ARG;
    g_timeline.store(static_cast<unsigned long long*>(buffer));
    g_timeline_calls.store(0);
    return TQ_OK;
#else
    (void)buffer;
    (void)bytes;
    return TQ_ERR_UNSUPPORTED;
#endif
}

tq_status tq_get_device_error(void* error_word, void* stream, int* code) {
    if (!error_word || !code) return TQ_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, error_word, sizeof(v), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return TQ_ERR_CUDA;
    *code = v;
    if (v != 0) {
        e = cudaMemsetAsync(error_word, 0, sizeof(v), st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
        if (e != cudaSuccess) return TQ_ERR_CUDA;
        return TQ_ERR_DEVICE_CHECK;
    }
    return TQ_OK;
}

}  // extern "C"
