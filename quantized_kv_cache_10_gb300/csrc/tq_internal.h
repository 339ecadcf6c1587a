// tq_internal.h -- declarations shared by the libtq translation units.
// Not part of the public ABI (include/tq.h is).
#pragma once

#include <cstddef>
#include <cstdint>
#include <vector>

#include <cuda_runtime.h>

#include "tq.h"

// Codec: host tables (fp64 construction, see tq_codec.cpp) and their device
// copies.  Immutable after tq_codec_create.
struct tq_codec {
    int dim = 0;
    int bits = 0;          // 2, 3, 4, 8, or 16 (raw fp16 keys)
    int is_wht = 0;
    int bytes_per_vec = 0;
    int device = 0;
    uint64_t seed = 0;

    std::vector<int8_t> signs;        // [dim] (WHT)
    std::vector<float> dense_q;       // [dim*dim] row-major, z = Q k (dense)
    std::vector<float> centroids;     // [2^bits]
    std::vector<double> midpoints;    // [2^bits - 1]

    // Device copies (owned).
    float* d_centroids = nullptr;     // [2^bits] fp32
    double* d_midpoints = nullptr;    // [2^bits - 1] fp64
    uint32_t* d_sign_bits = nullptr;  // [dim/32] bit j%32 of word j/32 set <=> s_j = -1
    float* d_q = nullptr;             // [dim*dim] Q row-major (dense)
    float* d_qt = nullptr;            // [dim*dim] Q^T row-major (dense)
    // Decode tables in compact form (see tq_decode_mma.cu):
    //  d_ktab: K-role entries for fp16 hi/lo split of centroid values;
    //  d_vtab: V-role entries (fp16 hi).
    uint32_t* d_ktab = nullptr;
    uint32_t* d_vtab = nullptr;
    int ktab_words = 0;
    int vtab_words = 0;
    float k_alpha = 1.0f;   // d_ktab holds fp16(k_alpha * c): the kernel scales q' by 1 / k_alpha
    float v_alpha = 1.0f;   // d_vtab holds fp16(v_alpha * c): the kernel scales its output by 1 / v_alpha
    // QJL residual sketch (keys of the TurboQuantProd variant, power-of-two dim): m = dim
    // rows of iid N(0,1) from the Gaussian stream of seed + 2, rounded to fp32
    int qjl = 0;
    std::vector<float> sketch;        // [dim*dim] S row-major, S[j][i]
    float* d_sketch = nullptr;        // S
    float* d_sketch_t = nullptr;      // S^T row-major: S^T[i][j] = S[j][i]
};

namespace tq {

// Host-side codebook / rotation construction (tq_codec.cpp).
void lloyd_max_gaussian(int bits, std::vector<double>& c64);
int dense_rotation(int dim, uint64_t seed, std::vector<float>& q);
void gaussian_stream(size_t n, uint64_t seed, std::vector<double>& out);
void rademacher_signs(int dim, uint64_t seed, std::vector<int8_t>& s);

int num_sms(int device);

// Launchers (tq_encode.cu / tq_dequant.cu / tq_decode_*.cu).  All return
// cudaGetLastError() of the launch.
cudaError_t launch_encode(const tq_codec* c, const uint16_t* x, int64_t n, int64_t xstride,
                          uint8_t* codes, int64_t cstride, uint16_t* norms,
                          // append mode (B > 0): x is [B, H, T, d], destination rows from start_pos
                          int B, int H, int T, const int32_t* start_pos, int64_t max_seq,
                          int32_t* dev_error, cudaStream_t st);

// One encode job: n vectors of x (row stride xstride) into codes / norms, or, in
// append mode (B > 0), x [B, H, T, dim] into cache rows from start_pos[b].
struct EncodeJob {
    const tq_codec* c;
    const uint16_t* x;
    int64_t n, xstride;
    uint8_t* codes;
    int64_t cstride;
    uint16_t* norms;
    int B, H, T;
    const int32_t* start_pos;
    int64_t max_seq;
    int32_t* dev_error;
    int64_t xplane;  // append mode: rows of x per (sequence, head) plane (>= T; 0: T, contiguous)
};
// One or two jobs (same dim and rotation kind, e.g. the K and the V pending batch)
// in one launch.
cudaError_t launch_encode_jobs(const EncodeJob* jobs, int njobs, cudaStream_t st);

cudaError_t launch_dequant(const tq_codec* c, const uint8_t* codes, const uint16_t* norms,
                           int64_t n, float* out, cudaStream_t st);

// QJL residual sketch of n vectors already encoded (codes, norms) with the codec's
// MSE part: sign bits [n][sign_stride bytes] and residual norms [n] (tq_qjl.cu).
cudaError_t launch_qjl_sketch(const tq_codec* c, const uint16_t* x, int64_t n, int64_t xstride,
                              const uint8_t* codes, int64_t cstride, const uint16_t* norms, uint8_t* signs,
                              int64_t sstride, uint16_t* rnorms, cudaStream_t st);

// Split-K plan for decode attention, shared by the workspace-size query and
// the launcher so both agree for a given device and shape.
struct DecodePlan {
    int kernel;          // 0 = SIMT (general), 1 = tensor-core (mma.sync) kernel
    int n_units;         // B * n_kv_heads
    int G;               // query heads per KV head
    int L;               // query positions per query head (1 for decode)
    int S;               // query rows per unit: G * L, head-major (row = head * L + position)
    int q_chunks;        // CTAs per (unit, split) along the rows: groups of at most 8 rows
    int n_split;         // CTAs per unit along the sequence
    int64_t chunk;       // tokens per split (multiple of 8 / tile)
    size_t ws_bytes;     // total workspace bytes
    size_t part_offset;  // byte offset of the split-K partial records
    int decode_smem;     // dynamic shared memory of the decode kernel launched (0: unknown)
    // Token-balanced schedule (tensor-core kernel, one query position, several sequences):
    // the units' tokens laid end to end, unit u = b * Hkv + h spanning stream_ovh positions
    // without tokens (the fixed cost of starting a unit) and len_b rounded up to 8, and CTA
    // c of n_cta takes an equal share of the positions.  Its records are at slots c + u
    // (the combine finds a unit's CTAs from the same lengths).
    int stream;          // 1: token-balanced schedule, 0: n_split splits of chunk tokens per unit
    int n_cta;           // CTAs of the token-balanced schedule
    int stream_ovh;      // positions without tokens per unit (a multiple of 8)
    int n_rec;           // partial records the workspace holds
};

// Split-K plan (independent of the kernel chosen, so the workspace size only
// depends on the shape and the device).  plan.kernel is set by the caller.
bool make_decode_plan(int dim, int device, int B, int Hq, int Hkv, int L, int64_t max_seq, DecodePlan& plan);

// By-value view of a codec for kernels (host structs are not visible on the
// device).
struct DevCodec {
    int dim, bits, is_wht, bpv;
    const float* centroids;
    const uint32_t* sign_bits;
    const float* q;    // Q row-major (dense)
    const float* qt;   // Q^T row-major (dense)
    const uint32_t* ktab;
    const uint32_t* vtab;
    float k_alpha, v_alpha;
    const float* sketch;    // QJL sketch S [dim][dim] (keys of the TurboQuantProd variant), else null
    const float* sketch_t;  // its transpose S^T [dim][dim]
};

inline DevCodec dev_view(const tq_codec* c) {
    return DevCodec{c->dim, c->bits, c->is_wht, c->bytes_per_vec, c->d_centroids, c->d_sign_bits, c->d_q,
                    c->d_qt, c->d_ktab, c->d_vtab, c->k_alpha, c->v_alpha, c->qjl ? c->d_sketch : nullptr,
                    c->qjl ? c->d_sketch_t : nullptr};
}

struct DecodeArgs {
    DevCodec ck;
    DevCodec cv;
    const uint16_t* q;
    const void* k;
    const uint16_t* k_norms;
    const uint8_t* v_codes;
    const uint16_t* v_norms;
    const int32_t* seq_lens;
    int B, Hq, Hkv;
    int64_t max_seq;
    float scale;
    uint16_t* out;
    void* ws;
    // unencoded fp16 tail tokens read in the same softmax: tail_lens[b] of them, or
    // tail_n for every sequence when tail_lens is null (no tail when tail_n <= 0)
    const uint16_t* k_tail;
    const uint16_t* v_tail;
    const int32_t* tail_lens;
    int max_tail;
    int tail_n;
    // optional new token [B, Hkv, dim] fp16: attended after the tail and appended to it
    // (written at tail index tail_n into k_tail / v_tail) in the same launch
    const uint16_t* k_new;
    const uint16_t* v_new;
    // keys of the TurboQuantProd variant (ck.sketch set): sign bits of the residual's
    // sketch [B, Hkv, max_seq, dim/8] and residual norms [B, Hkv, max_seq] fp16
    const uint8_t* k_signs;
    const uint16_t* k_rnorms;
    // query positions per query head: q and out are [B, Hq, L, dim]; the queries are the
    // last L positions of each sequence (packed tokens, then tail tokens) and each attends
    // to the tokens up to its own position (L == 1: every token)
    int L;
    // phase-timeline buffer of a profiling build (tq_debug_set_timeline), else null, and
    // the call's index (its parity selects the half of the buffer the call writes)
    unsigned long long* tl;
    unsigned int tl_seq;
};

// The timeline buffer registered with tq_debug_set_timeline (profiling builds), else null;
// its layout (tq_decode_common.cuh): 2 + 2 * 2 * kTlSlotsHost * kTlStampsHost words.
unsigned long long* timeline_buffer();
constexpr int kTlSlotsHost = 4096, kTlStampsHost = 8;

cudaError_t launch_decode_simt(const DecodeArgs& a, const DecodePlan& p, cudaStream_t st);
// Returns cudaErrorNotSupported when no tensor-core instantiation matches.
// May lower p.n_split / raise p.chunk (one CTA per SM); p is then the plan the
// kernel ran with, which the combine kernel needs.
cudaError_t launch_decode_mma(const DecodeArgs& a, DecodePlan& p, cudaStream_t st);
bool decode_mma_supported(const tq_codec* ck, const tq_codec* cv);
// Combine of the split-K partials, inverse V rotation and fp16 store
// (tq_decode_combine.cu).  Launched right after a decode kernel on the same
// stream; p must be the plan that kernel ran with.
cudaError_t launch_decode_combine(const DecodeArgs& a, const DecodePlan& p, cudaStream_t st);

}  // namespace tq
