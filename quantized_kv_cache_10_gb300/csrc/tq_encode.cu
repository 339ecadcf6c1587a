// tq_encode.cu -- bit-exact TurboQuant encode on sm_103a.
//
// Per vector ("How I built VeloxQuant-MLX", Stage 1 + Stage 2; RVQ post,
// "The Throughput Problem"; "add TurboQuant KV cache compression", Design):
//   k_i = x_i * 2^24 (exact int64), S = sum k_i^2 (exact 128-bit),
//   D = RN64(sqrt(RN64(S))), norm = RN16(D * 2^-24);
//   WHT dims: w = H (s . k) by an exact int64 butterfly (registers, then
//   warp shuffles), code_j = #{ i : w_j > RN64(m_i * D) };
//   other dims: z_j = fp64 fma chain of Q[j][i] k_i over ascending i,
//   code_j = #{ i : z_j > RN64(m_i * RN64(D / RN64(sqrt(d)))) };
//   codes packed LSB-first into 32-bit words.
// One warp per vector at a time: lane l owns elements [l*E, (l+1)*E), E = d / 32.
// The 2^b - 1 thresholds of a vector are computed once per warp (spread over
// its lanes) into shared memory and each coordinate finds its code by a b-step
// binary search over them ("number of boundaries exceeded").
#include <cuda_fp16.h>
#include <math_constants.h>

#include "tq_internal.h"

namespace tq {
namespace {

constexpr unsigned kFull = 0xffffffffu;

struct EncParams {
    const uint16_t* x;
    int64_t n;
    int64_t xstride;
    uint8_t* codes;
    int64_t cstride;
    uint16_t* norms;
    // append mode when B > 0: x is planes of xplane >= T rows per (sequence, head)
    int B, H, T;
    int64_t xplane;
    const int32_t* start_pos;
    int64_t max_seq;
    int32_t* dev_error;
    // codec
    const double* mid;
    const uint32_t* sign_bits;
    const float* qt;  // Q^T row-major (dense)
    int bits;
    int dim;
    int vb;           // vectors per warp batch (power-of-two dims), 1..32
};

__device__ __forceinline__ int64_t f16_exact(uint32_t h) {
    const int e = (h >> 10) & 31;
    const int64_t m = h & 1023;
    const int64_t k = (e == 0) ? m : ((m | 1024) << (e - 1));
    return (h & 0x8000u) ? -k : k;
}

// Correctly rounded conversion of the unsigned 128-bit integer hi:lo.
__device__ __forceinline__ double u128_to_f64_rn(uint64_t hi, uint64_t lo) {
    if (hi == 0) return __ull2double_rn(lo);
    const int nz = __clzll(static_cast<long long>(hi));
    uint64_t top, rest;
    if (nz == 0) {
        top = hi;
        rest = lo;
    } else {
        top = (hi << nz) | (lo >> (64 - nz));
        rest = lo << nz;
    }
    top |= (rest != 0) ? 1ull : 0ull;  // sticky bit below the rounding position
    return ldexp(__ull2double_rn(top), 64 - nz);
}

// Exact 128-bit sum of squares of the warp's values (hi:lo on all lanes).
template <int E>
__device__ __forceinline__ void warp_sumsq(const int64_t (&k)[E], int E_rt, uint64_t& hi_out, uint64_t& lo_out) {
    uint64_t lo = 0, hi = 0;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        if (e < E_rt) {
            const uint64_t a = static_cast<uint64_t>(k[e] < 0 ? -k[e] : k[e]);
            const uint64_t plo = a * a, phi = __umul64hi(a, a);
            const uint64_t nlo = lo + plo;
            hi += phi + (nlo < lo ? 1ull : 0ull);
            lo = nlo;
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const uint64_t olo = __shfl_xor_sync(kFull, lo, off);
        const uint64_t ohi = __shfl_xor_sync(kFull, hi, off);
        const uint64_t nlo = lo + olo;
        hi += ohi + (nlo < lo ? 1ull : 0ull);
        lo = nlo;
    }
    hi_out = hi;
    lo_out = lo;
}

// Exact sum of squares of the warp's values, returned as RN64 on all lanes.
template <int E>
__device__ __forceinline__ double warp_sumsq_rn(const int64_t (&k)[E], int E_rt) {
    uint64_t lo = 0, hi = 0;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        if (e < E_rt) {
            const uint64_t a = static_cast<uint64_t>(k[e] < 0 ? -k[e] : k[e]);
            const uint64_t plo = a * a, phi = __umul64hi(a, a);
            const uint64_t nlo = lo + plo;
            hi += phi + (nlo < lo ? 1ull : 0ull);
            lo = nlo;
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const uint64_t olo = __shfl_xor_sync(kFull, lo, off);
        const uint64_t ohi = __shfl_xor_sync(kFull, hi, off);
        const uint64_t nlo = lo + olo;
        hi += ohi + (nlo < lo ? 1ull : 0ull);
        lo = nlo;
    }
    return u128_to_f64_rn(hi, lo);
}

// Source row, destination row, and whether the row is written.
__device__ __forceinline__ bool map_row(const EncParams& p, int64_t v, const uint16_t*& src,
                                        int64_t& dst) {
    if (p.B <= 0) {
        src = p.x + v * p.xstride;
        dst = v;
        return true;
    }
    const int64_t per_b = static_cast<int64_t>(p.H) * p.T;
    const int64_t b = v / per_b;
    const int64_t rem = v - b * per_b;
    const int64_t h = rem / p.T;
    const int64_t t = rem - h * p.T;
    src = p.x + ((b * p.H + h) * p.xplane + t) * p.dim;
    const int64_t pos = static_cast<int64_t>(__ldg(p.start_pos + b)) + t;
    if (pos < 0 || pos >= p.max_seq) return false;
    dst = (b * p.H + h) * p.max_seq + pos;
    return true;
}

template <int E>
__device__ __forceinline__ void load_row(const uint16_t* src, int lane, int E_rt, uint32_t (&hv)[E]) {
    const uint16_t* s = src + lane * E_rt;
    if ((E_rt & 1) == 0) {
        const uint32_t* s32 = reinterpret_cast<const uint32_t*>(s);
#pragma unroll
        for (int e = 0; e < E; e += 2) {
            if (e < E_rt) {
                const uint32_t u = __ldg(s32 + e / 2);
                hv[e] = u & 0xffffu;
                if (e + 1 < E) hv[e + 1] = u >> 16;
            }
        }
    } else {
#pragma unroll
        for (int e = 0; e < E; ++e)
            if (e < E_rt) hv[e] = __ldg(s + e);
    }
}

// Packs the lane's E codes into the warp's shared word buffer and writes the
// row (d*b/32 words) with coalesced 32-bit stores.
template <int E>
__device__ __forceinline__ void pack_store(const int (&code)[E], int E_rt, int lane, int bits, int dim,
                                           uint32_t* buf, uint8_t* dst_row) {
    const int W = dim * bits / 32;
    for (int i = lane; i < W; i += 32) buf[i] = 0u;
    __syncwarp();
#pragma unroll
    for (int e = 0; e < E; ++e) {
        if (e < E_rt) {
            const int p = (lane * E_rt + e) * bits;
            const int word = p >> 5, sh = p & 31;
            const uint32_t c = static_cast<uint32_t>(code[e]);
            atomicOr(buf + word, c << sh);
            if (sh + bits > 32) atomicOr(buf + word + 1, c >> (32 - sh));
        }
    }
    __syncwarp();
    uint32_t* d32 = reinterpret_cast<uint32_t*>(dst_row);
    for (int i = lane; i < W; i += 32) d32[i] = buf[i];
    __syncwarp();
}

// Launched with programmatic stream serialization: the kernel may start while
// the previous kernel on the stream still runs.  Its inputs (the vectors, the
// positions) and its outputs are touched only after this wait, which returns
// once everything stream-ordered before it has completed; right after it the
// next kernel (e.g. the decode attention that reads the cache) may begin its
// own set-up.
__device__ __forceinline__ void grid_dependency_sync() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

constexpr int kWarps = 8;
constexpr float kNearTie = 2e-6f;  // relative margin of the fp32 boundary test (see below)

// |w| rounded to fp32 from its two 32-bit halves (relative error <= 2^-23).
__device__ __forceinline__ float abs_to_f32(int64_t w) {
    const uint64_t a = static_cast<uint64_t>(w < 0 ? -w : w);
    return fmaf(static_cast<float>(static_cast<uint32_t>(a >> 32)), 4294967296.0f,
                static_cast<float>(static_cast<uint32_t>(a)));
}

// Exact code of an integer coordinate: #{ i : w > RN64(m_i * D) }, by a
// binary search with the thresholds computed in fp64 on the fly.
__device__ __noinline__ int exact_code(int64_t w, double D, const double* mid, int L) {
    int pos = 0;
    for (int s = L >> 1; s > 0; s >>= 1)
        if (__double2ll_rd(__dmul_rn(__ldg(mid + pos + s - 1), D)) < w) pos += s;
    return pos;
}

// Power-of-two dims: E = dim / 32 in {1, 2, 4, 8, 16}.
//
// A warp takes 32 vectors at a time.  Pass 1 forms each vector's exact 128-bit
// sum of squares (all lanes), lane j keeping vector j's; the fp64 work of the
// norm (rounding S, the square root, the fp16 norm) then runs once for all 32
// vectors, one per lane -- the GPU's fp64 rate is a small fraction of its
// fp32 and integer rates.  For 2-4 bit codes the 2^b - 1 exact integer
// thresholds floor(RN64(m_i D)) (w > RN64(m_i D) <=> w > floor(...), w an
// integer) of the 32 vectors are formed in the same lane-parallel step.  Pass
// 2 re-reads each vector, applies the exact int64 butterfly and finds each
// code by a binary search: over those integer thresholds for 2-4 bits; for 8
// bits (255 thresholds per vector) over fp32 thresholds m_i * D, a coordinate
// within 2e-6 (relative) of its fp32 boundaries -- further than the fp32
// rounding of w, m_i, D and the product can move it -- being decided exactly
// instead (exact_code).  Outside that margin the fp32 comparison agrees with
// w > RN64(m_i D), so the codes are bit-exact either way.
//
// Two jobs (e.g. the K and the V pending batch, each with its own codec) may
// share one launch: blocks [0, grid0) take job 0, the rest job 1.
template <int E>
__device__ __forceinline__ void encode_wht_body(const EncParams& p, int64_t blk, int64_t nblk) {
    __shared__ float s_thr[kWarps][256];         // 8-bit codes: fp32 thresholds of one vector
    __shared__ int64_t s_ithr[kWarps][32 * 15];  // 2-4 bit codes: integer thresholds of 32 vectors
    __shared__ uint32_t s_pack[kWarps][128];
    __shared__ float s_mid[256];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int L = 1 << p.bits;
    // codec data (written by no kernel) before the dependency wait
    for (int i = threadIdx.x; i < L - 1; i += blockDim.x) s_mid[i] = __double2float_rn(__ldg(p.mid + i));
    grid_dependency_sync();
    __syncthreads();
    float* thr = s_thr[warp];
    int64_t* ithr = s_ithr[warp];
    uint32_t* pk = s_pack[warp];
    const bool small_book = p.bits <= 4;
    // signs of this lane's elements as a bit mask
    uint32_t smask = 0;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const int j = lane * E + e;
        smask |= ((__ldg(p.sign_bits + (j >> 5)) >> (j & 31)) & 1u) << e;
    }
    const int64_t total = (p.B > 0) ? static_cast<int64_t>(p.B) * p.H * p.T : p.n;
    const int64_t nbatch = (total + p.vb - 1) / p.vb;
    for (int64_t bt = blk * kWarps + warp; bt < nbatch; bt += nblk * kWarps) {
        const int64_t v0 = bt * p.vb;
        const int nb = static_cast<int>(min(static_cast<int64_t>(p.vb), total - v0));
        // ---- pass 1: exact sums of squares; lane j keeps vector j's
        uint64_t my_hi = 0, my_lo = 0;
        for (int jv = 0; jv < nb; ++jv) {
            const uint16_t* src;
            int64_t dst;
            if (!map_row(p, v0 + jv, src, dst)) continue;
            uint32_t hv[E];
            load_row<E>(src, lane, E, hv);
            int64_t k[E];
#pragma unroll
            for (int e = 0; e < E; ++e) k[e] = f16_exact(hv[e]);
            uint64_t hi, lo;
            warp_sumsq<E>(k, E, hi, lo);
            if (lane == jv) {
                my_hi = hi;
                my_lo = lo;
            }
        }
        // ---- fp64 per vector, one vector per lane: D = RN64(sqrt(RN64(S))), the norm
        double myD = 0.0;
        float myDf = 0.0f;
        int64_t mydst = -1;
        if (lane < nb) {
            const uint16_t* src;
            if (map_row(p, v0 + lane, src, mydst)) {
                myD = __dsqrt_rn(u128_to_f64_rn(my_hi, my_lo));
                myDf = __double2float_rn(myD);
                p.norms[mydst] = __half_as_ushort(__double2half(ldexp(myD, -24)));
                if (small_book)
                    for (int i = 0; i < L - 1; ++i) ithr[lane * 15 + i] = __double2ll_rd(__dmul_rn(__ldg(p.mid + i), myD));
            } else {
                mydst = -1;
                if (p.dev_error) atomicOr(p.dev_error, TQ_DEVERR_POSITION);
            }
        }
        __syncwarp();  // the batch's integer thresholds are visible to the warp
        // ---- pass 2: rotate and quantise
        for (int jv = 0; jv < nb; ++jv) {
            const int64_t dst = __shfl_sync(kFull, mydst, jv);
            if (dst < 0) continue;
            const double D = __shfl_sync(kFull, myD, jv);
            const float Df = __shfl_sync(kFull, myDf, jv);
            const uint16_t* src;
            int64_t dst_unused;
            map_row(p, v0 + jv, src, dst_unused);
            uint32_t hv[E];
            load_row<E>(src, lane, E, hv);
            int64_t k[E];
#pragma unroll
            for (int e = 0; e < E; ++e) k[e] = f16_exact(hv[e]);
            if (!small_book)
                for (int i = lane; i < L - 1; i += 32) thr[i] = s_mid[i] * Df;
            // w = H (s . k): in-lane stages, then cross-lane stages
#pragma unroll
            for (int e = 0; e < E; ++e)
                if ((smask >> e) & 1u) k[e] = -k[e];
#pragma unroll
            for (int h = 1; h < E; h <<= 1) {
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    if ((e & h) == 0) {
                        const int64_t a = k[e], b = k[e + h];
                        k[e] = a + b;
                        k[e + h] = a - b;
                    }
                }
            }
#pragma unroll
            for (int m = 1; m < 32; m <<= 1) {
                const bool upper = (lane & m) != 0;
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const int64_t o = __shfl_xor_sync(kFull, k[e], m);
                    k[e] = upper ? (o - k[e]) : (k[e] + o);
                }
            }
            __syncwarp();
            int code[E];
            if (small_book) {
                const int64_t* it = ithr + jv * 15;
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    int pos = 0;
                    for (int st = L >> 1; st > 0; st >>= 1)
                        if (it[pos + st - 1] < k[e]) pos += st;
                    code[e] = pos;
                }
            } else {
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const float af = abs_to_f32(k[e]);
                const float wf = k[e] < 0 ? -af : af;
                int pos = 0;
                for (int st = L >> 1; st > 0; st >>= 1)
                    if (thr[pos + st - 1] < wf) pos += st;
                // the boundaries next to the fp32 result decide it; any within the margin -> exact
                bool near = false;
                if (pos > 0) {
                    const float t = thr[pos - 1];
                    near |= fabsf(wf - t) <= kNearTie * fabsf(t);
                }
                if (pos < L - 1) {
                    const float t = thr[pos];
                    near |= fabsf(wf - t) <= kNearTie * fabsf(t);
                }
                if (near) pos = exact_code(k[e], D, p.mid, L);
                code[e] = pos;
            }
            }
            pack_store<E>(code, E, lane, p.bits, p.dim, pk, p.codes + dst * p.cstride);
        }
    }
}

template <int E>
__global__ void __launch_bounds__(kWarps * 32) encode_wht_kernel(const __grid_constant__ EncParams p0,
                                                                 const __grid_constant__ EncParams p1, int grid0) {
    if (static_cast<int>(blockIdx.x) < grid0)
        encode_wht_body<E>(p0, blockIdx.x, grid0);
    else
        encode_wht_body<E>(p1, blockIdx.x - grid0, gridDim.x - grid0);
}

constexpr int kDenseWarps = 4;
constexpr int kDenseMaxE = 15;

// Other dims (multiple of 32, not a power of two): E = dim / 32 at run time.
__device__ __forceinline__ void encode_dense_body(const EncParams& p, int64_t blk, int64_t nblk) {
    __shared__ double s_thr[kDenseWarps][256];
    __shared__ uint32_t s_pack[kDenseWarps][128];
    __shared__ double s_k[kDenseWarps][kDenseMaxE * 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int L = 1 << p.bits;
    const int E = p.dim >> 5;
    double* thr = s_thr[warp];
    uint32_t* pk = s_pack[warp];
    double* kk = s_k[warp];
    const double sqrt_d = __dsqrt_rn(static_cast<double>(p.dim));
    const int64_t total = (p.B > 0) ? static_cast<int64_t>(p.B) * p.H * p.T : p.n;
    grid_dependency_sync();
    for (int64_t v = blk * kDenseWarps + warp; v < total; v += nblk * kDenseWarps) {
        const uint16_t* src;
        int64_t dst;
        if (!map_row(p, v, src, dst)) {
            if (lane == 0 && p.dev_error) atomicOr(p.dev_error, TQ_DEVERR_POSITION);
            continue;
        }
        uint32_t hv[kDenseMaxE];
        load_row<kDenseMaxE>(src, lane, E, hv);
        int64_t k[kDenseMaxE];
#pragma unroll
        for (int e = 0; e < kDenseMaxE; ++e) {
            k[e] = (e < E) ? f16_exact(hv[e]) : 0;
            if (e < E) kk[lane * E + e] = static_cast<double>(k[e]);  // exact: |k| < 2^40
        }
        const double D = __dsqrt_rn(warp_sumsq_rn<kDenseMaxE>(k, E));
        const double sc = __ddiv_rn(D, sqrt_d);
        for (int i = lane; i < L; i += 32)
            thr[i] = (i < L - 1) ? __dmul_rn(__ldg(p.mid + i), sc) : CUDART_INF;
        __syncwarp();
        int code[kDenseMaxE];
#pragma unroll
        for (int e = 0; e < kDenseMaxE; ++e) {
            code[e] = 0;
            if (e < E) {
                const int j = lane * E + e;
                double acc = 0.0;
                for (int i = 0; i < p.dim; ++i)
                    acc = __fma_rn(static_cast<double>(__ldg(p.qt + static_cast<int64_t>(i) * p.dim + j)),
                                   kk[i], acc);
                int pos = 0;
                for (int s = L >> 1; s > 0; s >>= 1)
                    if (thr[pos + s - 1] < acc) pos += s;
                code[e] = pos;
            }
        }
        pack_store<kDenseMaxE>(code, E, lane, p.bits, p.dim, pk, p.codes + dst * p.cstride);
        if (lane == 0) p.norms[dst] = __half_as_ushort(__double2half(ldexp(D, -24)));
        __syncwarp();
    }
}

__global__ void __launch_bounds__(kDenseWarps * 32) encode_dense_kernel(const __grid_constant__ EncParams p0,
                                                                         const __grid_constant__ EncParams p1,
                                                                         int grid0) {
    if (static_cast<int>(blockIdx.x) < grid0)
        encode_dense_body(p0, blockIdx.x, grid0);
    else
        encode_dense_body(p1, blockIdx.x - grid0, gridDim.x - grid0);
}

// Parameters and grid of one encode job (vb and the grid depend on the vector count).
static EncParams make_params(const EncodeJob& j, int sms, int& grid) {
    const tq_codec* c = j.c;
    EncParams p{};
    p.x = j.x;
    p.n = j.n;
    p.xstride = j.xstride;
    p.codes = j.codes;
    p.cstride = j.cstride;
    p.norms = j.norms;
    p.B = j.B;
    p.H = j.H;
    p.T = j.T;
    p.xplane = j.xplane > 0 ? j.xplane : j.T;
    p.start_pos = j.start_pos;
    p.max_seq = j.max_seq;
    p.dev_error = j.dev_error;
    p.mid = c->d_midpoints;
    p.sign_bits = c->d_sign_bits;
    p.qt = c->d_qt;
    p.bits = c->bits;
    p.dim = c->dim;
    const int64_t total = (j.B > 0) ? static_cast<int64_t>(j.B) * j.H * j.T : j.n;
    if (c->is_wht) {
        // batches of up to 32 vectors per warp, smaller when there are too few vectors to
        // give every warp of the GPU one (pending-batch encodes of a few thousand vectors)
        const int64_t per_warp = total / (static_cast<int64_t>(sms) * kWarps * 4);
        p.vb = static_cast<int>(per_warp < 1 ? 1 : (per_warp > 32 ? 32 : per_warp));
        const int64_t want = ((total + p.vb - 1) / p.vb + kWarps - 1) / kWarps;
        grid = static_cast<int>(want < int64_t(sms) * 16 ? want : int64_t(sms) * 16);
    } else {
        const int64_t want = (total + kDenseWarps - 1) / kDenseWarps;
        grid = static_cast<int>(want < int64_t(sms) * 16 ? want : int64_t(sms) * 16);
    }
    return p;
}

template <typename K>
static cudaError_t launch_pdl(K kernel, int grid, int threads, cudaStream_t st, const EncParams& p0,
                              const EncParams& p1, int grid0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, p0, p1, grid0);
}

}  // namespace

cudaError_t launch_encode_jobs(const EncodeJob* jobs, int njobs, cudaStream_t st) {
    if (njobs < 1 || njobs > 2) return cudaErrorInvalidValue;
    const tq_codec* c = jobs[0].c;
    if (njobs == 2 && (jobs[1].c->dim != c->dim || jobs[1].c->is_wht != c->is_wht)) return cudaErrorInvalidValue;
    const int sms = num_sms(c->device);
    int g[2] = {0, 0};
    EncParams p[2];
    for (int i = 0; i < njobs; ++i) p[i] = make_params(jobs[i], sms, g[i]);
    if (njobs == 1) p[1] = p[0];
    const int grid = g[0] + g[1];
    if (grid <= 0) return cudaSuccess;   // nothing to encode
    if (c->is_wht) {
        switch (c->dim / 32) {
            case 1: return launch_pdl(encode_wht_kernel<1>, grid, kWarps * 32, st, p[0], p[1], g[0]);
            case 2: return launch_pdl(encode_wht_kernel<2>, grid, kWarps * 32, st, p[0], p[1], g[0]);
            case 4: return launch_pdl(encode_wht_kernel<4>, grid, kWarps * 32, st, p[0], p[1], g[0]);
            case 8: return launch_pdl(encode_wht_kernel<8>, grid, kWarps * 32, st, p[0], p[1], g[0]);
            case 16: return launch_pdl(encode_wht_kernel<16>, grid, kWarps * 32, st, p[0], p[1], g[0]);
            default: return cudaErrorInvalidValue;
        }
    }
    if (c->dim / 32 > kDenseMaxE) return cudaErrorInvalidValue;
    return launch_pdl(encode_dense_kernel, grid, kDenseWarps * 32, st, p[0], p[1], g[0]);
}

cudaError_t launch_encode(const tq_codec* c, const uint16_t* x, int64_t n, int64_t xstride,
                          uint8_t* codes, int64_t cstride, uint16_t* norms, int B, int H, int T,
                          const int32_t* start_pos, int64_t max_seq, int32_t* dev_error,
                          cudaStream_t st) {
    const EncodeJob j{c, x, n, xstride, codes, cstride, norms, B, H, T, start_pos, max_seq, dev_error, T};
    return launch_encode_jobs(&j, 1, st);
}

}  // namespace tq
