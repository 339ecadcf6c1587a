// tq_qjl.cu -- QJL residual sketch of encoded keys (the TurboQuantProd variant,
// "How I built VeloxQuant-MLX", Stage 3: QJL Residual Correction).
//
// A key keeps its MSE codes and norm (tq_encode with the codec's bits) plus
// the sign bits of a Gaussian sketch of its quantisation residual and the
// residual's norm.  Arithmetic, fixed so that the sign decisions and the norm
// are reproducible bit for bit:
//   w     = H (s . k), k_i = x_i 2^24: exact int64 (the encode's rotation);
//   rho_i = RN64(w_i 2^-24 - n16 c[code_i]) (one fma), rounded to fp32:
//           sqrt(d) times the residual in the rotated basis;
//   gamma = RN16(sqrt(G2 / d)), G2 = fp64 chain over i ascending of rho_i^2;
//   t_j   = fp32 fma chain over i ascending of S[j][i] rho_i, sign bit j set
//           when t_j < 0 (packed LSB-first, dim / 8 bytes per key).
#include <cuda_fp16.h>

#include "tq_internal.h"

namespace tq {
namespace {

constexpr unsigned kFull = 0xffffffffu;

// x * 2^24 as an exact integer (every finite fp16 value is a multiple of 2^-24).
__device__ __forceinline__ long long f16_fixed(uint16_t h) {
    const int e = (h >> 10) & 31, m = h & 1023;
    const long long mag = e == 0 ? static_cast<long long>(m) : static_cast<long long>(1024 + m) << (e - 1);
    return (h & 0x8000u) ? -mag : mag;
}

__device__ __forceinline__ int code_at(const uint8_t* row, int i, int bits) {
    const int p = i * bits, byte = p >> 3, sh = p & 7;
    uint32_t w = row[byte];
    if (sh + bits > 8) w |= static_cast<uint32_t>(row[byte + 1]) << 8;
    return static_cast<int>((w >> sh) & ((1u << bits) - 1u));
}

// Keys in batches of KB per warp (grid-stride over batches); E = dim / 32.  Per key the
// warp forms the exact rotation and the fp32 residual (kept for the batch in shared
// memory); then lane k runs key k's fp64 norm chain (so that one fp64 instruction serves
// KB keys), and the sketch chains of all KB keys run together, each S^T load feeding KB
// of them.  Every chain keeps its order (i ascending), so the results are the same bits.
template <int E>
struct QjlShape {
    static constexpr int D = 32 * E;
    static constexpr int WARPS = E >= 16 ? 2 : 4;                 // warps per CTA
    static constexpr int KB = E >= 16 ? 4 : (E >= 8 ? 8 : 16);    // keys per batch
    static constexpr int RS = D + 1;                              // residual row stride (floats)
};

template <int E>
__global__ void __launch_bounds__(QjlShape<E>::WARPS * 32)
    qjl_sketch_kernel(const uint16_t* x, int64_t n, int64_t xstride, const uint8_t* codes, int64_t cstride,
                      const uint16_t* norms, const float* centroids, const uint32_t* sign_bits, const float* st,
                      int bits, uint8_t* signs, int64_t sstride, uint16_t* rnorms) {
    using Q = QjlShape<E>;
    constexpr int D = Q::D, KB = Q::KB, RS = Q::RS;
    __shared__ long long s_w[Q::WARPS][D];
    __shared__ float s_rho[Q::WARPS][KB * RS];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    long long* w = s_w[warp];
    float* rho = s_rho[warp];
    const int64_t nbatch = (n + KB - 1) / KB;
    for (int64_t bt = static_cast<int64_t>(blockIdx.x) * Q::WARPS + warp; bt < nbatch;
         bt += static_cast<int64_t>(gridDim.x) * Q::WARPS) {
        const int64_t v0 = bt * KB;
        const int nk = static_cast<int>(n - v0 < KB ? n - v0 : KB);
        for (int k = 0; k < KB; ++k) {
            float* rk = rho + k * RS;
            if (k >= nk) {  // rows past the last key: zeros (their sums are not stored)
                for (int i = lane; i < D; i += 32) rk[i] = 0.0f;
                continue;
            }
            const int64_t v = v0 + k;
            const uint16_t* xr = x + v * xstride;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const int i = lane + 32 * e;
                const long long kx = f16_fixed(xr[i]);
                w[i] = ((__ldg(sign_bits + (i >> 5)) >> (i & 31)) & 1u) ? -kx : kx;
            }
            __syncwarp();
            // Sylvester butterfly in natural order, exact in int64 (|w| < 2^48)
            for (int hh = 1; hh < D; hh <<= 1) {
                for (int i = lane; i < D / 2; i += 32) {
                    const int lo = (i / hh) * (2 * hh) + (i % hh);
                    const long long a = w[lo], b = w[lo + hh];
                    w[lo] = a + b;
                    w[lo + hh] = a - b;
                }
                __syncwarp();
            }
            const double n16 = static_cast<double>(__half2float(__ushort_as_half(norms[v])));
            const uint8_t* cr = codes + v * cstride;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const int i = lane + 32 * e;
                const double c = static_cast<double>(__ldg(centroids + code_at(cr, i, bits)));
                rk[i] = __double2float_rn(__fma_rn(-n16, c, static_cast<double>(w[i]) * 0x1.0p-24));
            }
            __syncwarp();  // w is rewritten by the next key
        }
        // residual norms: lane k, key k's fp64 chain over i ascending (rows RS apart:
        // the lanes read distinct banks)
        if (lane < nk) {
            const float* rk = rho + lane * RS;
            double g2 = 0.0;
            for (int i = 0; i < D; ++i) {
                const double r = static_cast<double>(rk[i]);
                g2 = __fma_rn(r, r, g2);
            }
            rnorms[v0 + lane] = __half_as_ushort(__double2half(sqrt(g2 / static_cast<double>(D))));
        }
        // t_j of every key of the batch, j = lane + 32 kk, each an fp32 fma chain over i
        // ascending; S^T rows are read across the lanes (coalesced), each load feeding KB keys
        float t[KB][E];
#pragma unroll
        for (int k = 0; k < KB; ++k)
#pragma unroll
            for (int kk = 0; kk < E; ++kk) t[k][kk] = 0.0f;
#pragma unroll 2
        for (int i = 0; i < D; ++i) {
            const float* row = st + static_cast<int64_t>(i) * D + lane;
            float sv[E];
#pragma unroll
            for (int kk = 0; kk < E; ++kk) sv[kk] = __ldg(row + 32 * kk);
#pragma unroll
            for (int k = 0; k < KB; ++k) {
                const float r = rho[k * RS + i];
#pragma unroll
                for (int kk = 0; kk < E; ++kk) t[k][kk] = __fmaf_rn(sv[kk], r, t[k][kk]);
            }
        }
#pragma unroll
        for (int k = 0; k < KB; ++k) {
            if (k >= nk) break;
            uint32_t* sw = reinterpret_cast<uint32_t*>(signs + (v0 + k) * sstride);
#pragma unroll
            for (int kk = 0; kk < E; ++kk) {
                const uint32_t word = __ballot_sync(kFull, t[k][kk] < 0.0f);
                if (lane == 0) sw[kk] = word;
            }
        }
        __syncwarp();  // the residual rows are rewritten by the next batch
    }
}

template <int E>
cudaError_t launch_e(const tq_codec* c, const uint16_t* x, int64_t n, int64_t xstride, const uint8_t* codes,
                     int64_t cstride, const uint16_t* norms, uint8_t* signs, int64_t sstride, uint16_t* rnorms,
                     cudaStream_t st) {
    using Q = QjlShape<E>;
    const int64_t nbatch = (n + Q::KB - 1) / Q::KB;
    const int64_t want = (nbatch + Q::WARPS - 1) / Q::WARPS;
    const int64_t cap = int64_t(num_sms(c->device)) * 16;
    const int grid = static_cast<int>(want < cap ? want : cap);
    qjl_sketch_kernel<E><<<grid, Q::WARPS * 32, 0, st>>>(x, n, xstride, codes, cstride, norms, c->d_centroids,
                                                          c->d_sign_bits, c->d_sketch_t, c->bits, signs, sstride,
                                                          rnorms);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_qjl_sketch(const tq_codec* c, const uint16_t* x, int64_t n, int64_t xstride,
                              const uint8_t* codes, int64_t cstride, const uint16_t* norms, uint8_t* signs,
                              int64_t sstride, uint16_t* rnorms, cudaStream_t st) {
    if (n <= 0) return cudaSuccess;
    switch (c->dim / 32) {
        case 1: return launch_e<1>(c, x, n, xstride, codes, cstride, norms, signs, sstride, rnorms, st);
        case 2: return launch_e<2>(c, x, n, xstride, codes, cstride, norms, signs, sstride, rnorms, st);
        case 4: return launch_e<4>(c, x, n, xstride, codes, cstride, norms, signs, sstride, rnorms, st);
        case 8: return launch_e<8>(c, x, n, xstride, codes, cstride, norms, signs, sstride, rnorms, st);
        case 16: return launch_e<16>(c, x, n, xstride, codes, cstride, norms, signs, sstride, rnorms, st);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace tq
