// tq_noalloc.cu -- decode attention for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they attend: code
// running inside a CUDA-graph capture they do not control, plugins hosted by
// an engine that owns every allocation, or real-time loops where allocation is
// forbidden.  tq_decode_attend_noalloc serves them by running the ordinary
// decode attention on a scratch area that lives in this library's own device
// memory: a file-scope __device__ array, reserved when the library's module is
// loaded on a device and held until the process exits.
//
// In host code the array's name is only a host-side stand-in, not a device
// address, so the address is fetched once per device with
// cudaGetSymbolAddress (with that device current) and cached; kernels are
// given that address.
#include <cstdint>
#include <mutex>

#include "tq_internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(8) << 20;  // 8 MiB per device
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_decode_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set-up on the first call).
cudaError_t scratch_address(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" {

tq_status tq_decode_attend_noalloc(const tq_codec* ck, const tq_codec* cv, const uint16_t* q, const void* k,
                                   const uint16_t* k_norms, const uint8_t* v_codes, const uint16_t* v_norms,
                                   const int32_t* seq_lens, int B, int n_q_heads, int n_kv_heads, int64_t max_seq,
                                   float scale, uint16_t* out, void* stream) {
    // The same argument checks as tq_decode_attend, made before anything is enqueued.
    if (!ck || !cv || cv->bits == 16 || ck->dim != cv->dim) return TQ_ERR_INVALID_ARG;
    if (ck->qjl || cv->qjl) return TQ_ERR_INVALID_ARG;  // sketched keys have their own entry point
    if (!q || !k || !v_codes || !v_norms || !seq_lens || !out) return TQ_ERR_INVALID_ARG;
    if ((ck->bits == 16) != (k_norms == nullptr)) return TQ_ERR_INVALID_ARG;
    if (B <= 0 || n_q_heads <= 0 || n_kv_heads <= 0 || n_q_heads % n_kv_heads != 0) return TQ_ERR_INVALID_ARG;
    if (max_seq <= 0 || max_seq % 8 != 0) return TQ_ERR_INVALID_ARG;
    if (!aligned(k, 16) || !aligned(v_codes, 16) || !aligned(v_norms, 16) || (k_norms && !aligned(k_norms, 16)))
        return TQ_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(out, 4) || !aligned(seq_lens, 4)) return TQ_ERR_INVALID_ARG;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != ck->device || dev != cv->device) return TQ_ERR_INVALID_ARG;
    tq::DecodePlan p;
    if (!tq::make_decode_plan(cv->dim, cv->device, B, n_q_heads, n_kv_heads, 1, max_seq, p)) return TQ_ERR_INVALID_ARG;
    if (p.ws_bytes > kScratchBytes) return TQ_ERR_WORKSPACE;  // shape too large for the fixed scratch
    void* ws = nullptr;
    if (scratch_address(&ws) != cudaSuccess) return TQ_ERR_CUDA;
    // The scratch keeps whatever the previous call left: clear the error word,
    // which must start at zero.
    if (cudaMemsetAsync(ws, 0, p.part_offset, static_cast<cudaStream_t>(stream)) != cudaSuccess) return TQ_ERR_CUDA;
    return tq_decode_attend(ck, cv, q, k, k_norms, v_codes, v_norms, seq_lens, B, n_q_heads, n_kv_heads, max_seq,
                            scale, out, ws, kScratchBytes, stream);
}

}  // extern "C"
