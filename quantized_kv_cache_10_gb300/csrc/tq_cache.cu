// tq_cache.cu -- the two-phase KV cache around the hot path ("add TurboQuant KV
// cache compression", Design: raw fp16 during prefill, batch-compress on the
// first decode token; pending tokens encoded in batches of 64; the cache
// interface update / attend / memory of "How I built VeloxQuant-MLX").
//
// Optionally the first min_tokens tokens of every sequence stay fp16 for good
// (sink tokens; turboquant-mlx guide "KV cache compression", --kv-min-tokens:
// "keeps the first N tokens in FP16"): they sit in front of the pending tokens in
// the fp16 tail buffer, which the combine kernel scores in the same softmax.
//
// Device state of one cache (B sequences of equal length, one layer):
//   packed K / V codes + fp16 norms  [B, Hkv, max_seq, ...]   (raw K: fp16 rows)
//   fp16 tail K / V                  [B, Hkv, min_tokens + 64, d]: the sink tokens,
//                                    then the pending tokens (not yet encoded)
//   prefill staging K / V fp16       [B, Hkv, T, d]           (phase 1 only)
//   encoded-token count per sequence (int32 [B], for the decode and encode calls)
//   the decode workspace.
// A decode step is two launches (decode kernel, combine kernel) and, every 64th
// step, the encode of the full pending batch: the combine kernel attends the
// new token after the pending ones and appends it to the pending buffer.
#include <cstring>
#include <new>

#include "tq_internal.h"

struct tq_cache {
    const tq_codec* ck = nullptr;
    const tq_codec* cv = nullptr;
    int B = 0, Hq = 0, Hkv = 0, dim = 0, device = 0;
    int64_t max_seq = 0;
    uint8_t* kc = nullptr;      // packed K codes, or raw fp16 K rows (bits 16)
    uint16_t* kn = nullptr;     // K norms (null for raw K)
    uint8_t* vc = nullptr;
    uint16_t* vn = nullptr;
    uint16_t* pk = nullptr;     // pending fp16 [B, Hkv, kPending, d]
    uint16_t* pv = nullptr;
    uint16_t* rk = nullptr;     // prefill staging (phase 1)
    uint16_t* rv = nullptr;
    int raw_T = 0;
    int n_sink = 0;             // tokens kept fp16 at the start of every sequence (min_tokens)
    int sinks = 0;              // of them held so far (sequences shorter than min_tokens)
    int32_t* d_count = nullptr; // [B] encoded tokens per sequence
    int32_t* d_err = nullptr;   // device error word of the encode calls
    void* ws = nullptr;
    size_t ws_bytes = 0;
    int64_t encoded = 0;        // tokens in the packed cache (per sequence)
    int pending = 0;            // tokens in the pending buffer (per sequence)
    bool count_stale = true;    // d_count holds an encode start position, not `encoded`
};

namespace {

constexpr int kPending = 64;    // pending tokens encoded as one batch
constexpr int kMaxSinks = 4096;  // fp16 sink tokens per sequence at most

__global__ void fill_i32(int32_t* p, int n, int32_t v) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) p[i] = v;
}

cudaError_t set_count(tq_cache* c, int64_t v, cudaStream_t st) {
    fill_i32<<<(c->B + 127) / 128, 128, 0, st>>>(c->d_count, c->B, static_cast<int32_t>(v));
    return cudaGetLastError();
}

void release(tq_cache* c) {
    cudaFree(c->kc);
    cudaFree(c->kn);
    cudaFree(c->vc);
    cudaFree(c->vn);
    cudaFree(c->pk);
    cudaFree(c->pv);
    cudaFree(c->rk);
    cudaFree(c->rv);
    cudaFree(c->d_count);
    cudaFree(c->d_err);
    cudaFree(c->ws);
}

tq_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return TQ_OK;
    if (e == cudaErrorMemoryAllocation) return TQ_ERR_OOM;
    if (e == cudaErrorNotSupported) return TQ_ERR_UNSUPPORTED;
    return TQ_ERR_CUDA;
}

size_t row_bytes(const tq_codec* c) { return static_cast<size_t>(c->bytes_per_vec); }

int tail_rows(const tq_cache* c) { return c->n_sink + kPending; }

// Appends T fp16 tokens at position `pos` of every sequence's packed cache: token t of
// the (sequence, KV head) plane p is k[(p * plane + t) * d] (plane >= T rows per plane).
tq_status encode_tokens(tq_cache* c, const uint16_t* k, const uint16_t* v, int T, int64_t plane, int64_t pos,
                        cudaStream_t st) {
    if (T <= 0) return TQ_OK;
    c->count_stale = true;
    cudaError_t e = set_count(c, pos, st);
    if (e != cudaSuccess) return from_cuda(e);
    const int planes = c->B * c->Hkv;
    if (c->ck->bits == 16) {
        // raw K rows are stored as they are: one strided copy per (sequence, KV head) plane
        const size_t rb = static_cast<size_t>(c->dim) * 2;
        e = cudaMemcpy2DAsync(c->kc + pos * rb, static_cast<size_t>(c->max_seq) * rb, k, static_cast<size_t>(plane) * rb,
                              static_cast<size_t>(T) * rb, static_cast<size_t>(planes), cudaMemcpyDeviceToDevice, st);
        if (e != cudaSuccess) return from_cuda(e);
        const tq::EncodeJob jv{c->cv, v, 0, c->dim, c->vc, c->cv->bytes_per_vec, c->vn, c->B, c->Hkv, T,
                               c->d_count, c->max_seq, c->d_err, plane};
        return from_cuda(tq::launch_encode_jobs(&jv, 1, st));
    }
    // K and V in one launch
    const tq::EncodeJob jobs[2] = {
        {c->ck, k, 0, c->dim, c->kc, c->ck->bytes_per_vec, c->kn, c->B, c->Hkv, T, c->d_count, c->max_seq, c->d_err,
         plane},
        {c->cv, v, 0, c->dim, c->vc, c->cv->bytes_per_vec, c->vn, c->B, c->Hkv, T, c->d_count, c->max_seq, c->d_err,
         plane}};
    return from_cuda(tq::launch_encode_jobs(jobs, 2, st));
}

}  // namespace

extern "C" {

tq_status tq_cache_create(const tq_codec* ck, const tq_codec* cv, int B, int n_q_heads, int n_kv_heads,
                          int64_t max_seq, int min_tokens, tq_cache** out) {
    if (!out) return TQ_ERR_INVALID_ARG;
    *out = nullptr;
    if (!ck || !cv || cv->bits == 16 || ck->dim != cv->dim) return TQ_ERR_INVALID_ARG;
    if (ck->qjl || cv->qjl) return TQ_ERR_UNSUPPORTED;  // the cache keeps MSE-coded keys only
    if (B <= 0 || n_q_heads <= 0 || n_kv_heads <= 0 || n_q_heads % n_kv_heads != 0) return TQ_ERR_INVALID_ARG;
    if (max_seq <= 0 || max_seq % 8 != 0 || max_seq > (int64_t(1) << 30)) return TQ_ERR_INVALID_ARG;
    if (min_tokens < 0 || min_tokens > kMaxSinks) return TQ_ERR_INVALID_ARG;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != ck->device || dev != cv->device) return TQ_ERR_INVALID_ARG;
    tq_cache* c = new (std::nothrow) tq_cache();
    if (!c) return TQ_ERR_OOM;
    c->ck = ck;
    c->cv = cv;
    c->B = B;
    c->Hq = n_q_heads;
    c->Hkv = n_kv_heads;
    c->dim = cv->dim;
    c->device = dev;
    c->max_seq = max_seq;
    c->n_sink = min_tokens;
    const size_t rows = static_cast<size_t>(B) * n_kv_heads * static_cast<size_t>(max_seq);
    const size_t prow = static_cast<size_t>(B) * n_kv_heads * tail_rows(c) * c->dim;
    c->ws_bytes = tq_decode_attend_workspace_bytes(B, n_q_heads, n_kv_heads, max_seq, c->dim);
    cudaError_t e = c->ws_bytes ? cudaSuccess : cudaErrorInvalidValue;
    if (e == cudaSuccess) e = cudaMalloc(&c->kc, rows * row_bytes(ck));
    if (e == cudaSuccess && ck->bits != 16) e = cudaMalloc(&c->kn, rows * 2);
    if (e == cudaSuccess) e = cudaMalloc(&c->vc, rows * row_bytes(cv));
    if (e == cudaSuccess) e = cudaMalloc(&c->vn, rows * 2);
    if (e == cudaSuccess) e = cudaMalloc(&c->pk, prow * 2);
    if (e == cudaSuccess) e = cudaMalloc(&c->pv, prow * 2);
    if (e == cudaSuccess) e = cudaMalloc(&c->d_count, static_cast<size_t>(B) * 4);
    if (e == cudaSuccess) e = cudaMalloc(&c->d_err, 4);
    if (e == cudaSuccess) e = cudaMalloc(&c->ws, c->ws_bytes);
    if (e == cudaSuccess) e = cudaMemset(c->d_err, 0, 4);
    if (e == cudaSuccess) e = cudaMemset(c->ws, 0, c->ws_bytes);
    if (e != cudaSuccess) {
        release(c);
        delete c;
        return from_cuda(e);
    }
    *out = c;
    return TQ_OK;
}

void tq_cache_destroy(tq_cache* c) {
    if (!c) return;
    release(c);
    delete c;
}

tq_status tq_cache_prefill(tq_cache* c, const uint16_t* k, const uint16_t* v, int T, void* stream) {
    if (!c || !k || !v || T <= 0) return TQ_ERR_INVALID_ARG;
    if (c->encoded != 0 || c->pending != 0 || c->raw_T != 0) return TQ_ERR_INVALID_ARG;  // prefill once, first
    if (T > c->max_seq) return TQ_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t n = static_cast<size_t>(c->B) * c->Hkv * static_cast<size_t>(T) * c->dim;
    cudaError_t e = cudaMallocAsync(&c->rk, n * 2, st);
    if (e == cudaSuccess) e = cudaMallocAsync(&c->rv, n * 2, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(c->rk, k, n * 2, cudaMemcpyDeviceToDevice, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(c->rv, v, n * 2, cudaMemcpyDeviceToDevice, st);
    if (e != cudaSuccess) return from_cuda(e);
    c->raw_T = T;
    return TQ_OK;
}

tq_status tq_cache_decode(tq_cache* c, const uint16_t* q, const uint16_t* k_new, const uint16_t* v_new,
                          float scale, uint16_t* out, void* stream) {
    if (!c || !q || !k_new || !v_new || !out) return TQ_ERR_INVALID_ARG;
    if (c->sinks + c->encoded + c->raw_T + c->pending + 1 > c->max_seq) return TQ_ERR_INVALID_ARG;  // full
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    tq_status s = TQ_OK;
    if (c->raw_T > 0) {
        // phase 2 begins: the first min_tokens prefill tokens become the fp16 sink tokens,
        // the rest are batch-compressed
        const int s0 = c->raw_T < c->n_sink ? c->raw_T : c->n_sink;
        const size_t rb = static_cast<size_t>(c->dim) * 2;
        const size_t planes = static_cast<size_t>(c->B) * c->Hkv;
        cudaError_t e0 = cudaSuccess;
        if (s0 > 0) {
            e0 = cudaMemcpy2DAsync(c->pk, tail_rows(c) * rb, c->rk, c->raw_T * rb, s0 * rb, planes,
                                   cudaMemcpyDeviceToDevice, st);
            if (e0 == cudaSuccess)
                e0 = cudaMemcpy2DAsync(c->pv, tail_rows(c) * rb, c->rv, c->raw_T * rb, s0 * rb, planes,
                                       cudaMemcpyDeviceToDevice, st);
            if (e0 != cudaSuccess) return from_cuda(e0);
        }
        s = encode_tokens(c, c->rk + static_cast<size_t>(s0) * c->dim, c->rv + static_cast<size_t>(s0) * c->dim,
                          c->raw_T - s0, c->raw_T, 0, st);
        if (s != TQ_OK) return s;
        cudaFreeAsync(c->rk, st);
        cudaFreeAsync(c->rv, st);
        c->rk = c->rv = nullptr;
        c->sinks = s0;
        c->encoded = c->raw_T - s0;
        c->raw_T = 0;
    }
    cudaError_t e = cudaSuccess;
    if (c->count_stale) {  // the lengths the decode reads: the packed-token count
        e = set_count(c, c->encoded, st);
        if (e != cudaSuccess) return from_cuda(e);
        c->count_stale = false;
    }
    // attend over the packed tokens, the pending ones and the new one; append the new one
    tq::DecodePlan p;
    if (!tq::make_decode_plan(c->dim, c->device, c->B, c->Hq, c->Hkv, 1, c->max_seq, p)) return TQ_ERR_INVALID_ARG;
    if (c->ws_bytes < p.ws_bytes) return TQ_ERR_WORKSPACE;
    // the fp16 tail: the sink tokens, then the pending ones; the new token goes after them
    tq::DecodeArgs a{tq::dev_view(c->ck), tq::dev_view(c->cv), q, c->kc, c->kn, c->vc, c->vn, c->d_count,
                     c->B, c->Hq, c->Hkv, c->max_seq, scale, out, c->ws,
                     c->pk, c->pv, nullptr, tail_rows(c), c->sinks + c->pending, k_new, v_new, nullptr, nullptr, 1};
    e = cudaErrorNotSupported;
    if (tq::decode_mma_supported(c->ck, c->cv)) {
        p.kernel = 1;
        e = tq::launch_decode_mma(a, p, st);
    }
    if (e == cudaErrorNotSupported) {
        p.kernel = 0;
        e = tq::launch_decode_simt(a, p, st);
    }
    if (e == cudaSuccess) e = tq::launch_decode_combine(a, p, st);
    if (e != cudaSuccess) return from_cuda(e);
    if (c->sinks < c->n_sink) {  // the sequence is still shorter than min_tokens: one more sink
        ++c->sinks;
        return TQ_OK;
    }
    if (++c->pending == kPending) {
        const size_t off = static_cast<size_t>(c->n_sink) * c->dim;  // the pending rows follow the sinks
        s = encode_tokens(c, c->pk + off, c->pv + off, kPending, tail_rows(c), c->encoded, st);
        if (s != TQ_OK) return s;
        c->encoded += kPending;
        c->pending = 0;
    }
    return TQ_OK;
}

tq_status tq_cache_info(const tq_cache* c, int64_t* tokens, int64_t* encoded, int* pending,
                        size_t* bytes_in_use) {
    if (!c) return TQ_ERR_INVALID_ARG;
    const int64_t units = static_cast<int64_t>(c->B) * c->Hkv;
    if (tokens) *tokens = c->sinks + c->encoded + c->pending + c->raw_T;
    if (encoded) *encoded = c->encoded;
    if (pending) *pending = c->pending;
    if (bytes_in_use) {
        const size_t packed = row_bytes(c->ck) + (c->ck->bits == 16 ? 0 : 2) + row_bytes(c->cv) + 2;
        const size_t raw = static_cast<size_t>(c->dim) * 2 * 2;
        *bytes_in_use = static_cast<size_t>(units) * (static_cast<size_t>(c->encoded) * packed +
                                                      static_cast<size_t>(c->sinks + c->pending + c->raw_T) * raw);
    }
    return TQ_OK;
}

tq_status tq_cache_device_error(tq_cache* c, void* stream, int* code) {
    if (!c || !code) return TQ_ERR_INVALID_ARG;
    int a = 0, b = 0;
    tq_status s1 = tq_get_device_error(c->d_err, stream, &a);
    tq_status s2 = tq_get_device_error(c->ws, stream, &b);
    *code = a | b;
    if (s1 == TQ_ERR_CUDA || s2 == TQ_ERR_CUDA) return TQ_ERR_CUDA;
    return (*code != 0) ? TQ_ERR_DEVICE_CHECK : TQ_OK;
}

}  // extern "C"
