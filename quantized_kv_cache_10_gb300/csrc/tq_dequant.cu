// tq_dequant.cu -- debugging dequantiser: x^ = n16 * R^T (c[codes] / sqrt(d)).
//
// R = H diag(s) / sqrt(d) ("How I built VeloxQuant-MLX", Stage 1), so
// R^T y = diag(s) H y / sqrt(d) and x^ = (n16 / d) * s . (H c[codes]); the
// dense rotation gives x^ = (n16 / sqrt(d)) * Q^T c[codes].  fp32 throughout,
// one warp per vector, the butterfly in registers and warp shuffles.
#include <cuda_fp16.h>

#include "tq_internal.h"

namespace tq {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kWarps = 8;

struct DqParams {
    const uint8_t* codes;
    const uint16_t* norms;
    int64_t n;
    float* out;
    const float* centroids;
    const uint32_t* sign_bits;
    const float* q;  // Q row-major (dense)
    int bits, dim, bpv;
};

// Code j of a packed row (LSB-first bit stream).
__device__ __forceinline__ int code_at(const uint8_t* row, int j, int bits) {
    const int p = j * bits;
    const int byte = p >> 3, sh = p & 7;
    uint32_t w = row[byte];
    if (sh + bits > 8) w |= static_cast<uint32_t>(row[byte + 1]) << 8;
    return static_cast<int>((w >> sh) & ((1u << bits) - 1u));
}

template <int E>
__global__ void __launch_bounds__(kWarps * 32) dequant_wht_kernel(const DqParams p) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t smask = 0;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const int j = lane * E + e;
        smask |= ((__ldg(p.sign_bits + (j >> 5)) >> (j & 31)) & 1u) << e;
    }
    const float inv_d = 1.0f / static_cast<float>(p.dim);
    for (int64_t v = static_cast<int64_t>(blockIdx.x) * kWarps + warp; v < p.n;
         v += static_cast<int64_t>(gridDim.x) * kWarps) {
        const uint8_t* row = p.codes + v * p.bpv;
        float y[E];
#pragma unroll
        for (int e = 0; e < E; ++e) y[e] = __ldg(p.centroids + code_at(row, lane * E + e, p.bits));
#pragma unroll
        for (int h = 1; h < E; h <<= 1) {
#pragma unroll
            for (int e = 0; e < E; ++e) {
                if ((e & h) == 0) {
                    const float a = y[e], b = y[e + h];
                    y[e] = a + b;
                    y[e + h] = a - b;
                }
            }
        }
#pragma unroll
        for (int m = 1; m < 32; m <<= 1) {
            const bool upper = (lane & m) != 0;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const float o = __shfl_xor_sync(kFull, y[e], m);
                y[e] = upper ? (o - y[e]) : (y[e] + o);
            }
        }
        const float sc = __half2float(__ushort_as_half(p.norms[v])) * inv_d;
        float* o = p.out + v * p.dim + lane * E;
#pragma unroll
        for (int e = 0; e < E; ++e) o[e] = ((smask >> e) & 1u) ? -(y[e] * sc) : (y[e] * sc);
    }
}

__global__ void __launch_bounds__(kWarps * 32) dequant_dense_kernel(const DqParams p) {
    extern __shared__ float s_y[];  // [kWarps][dim]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float* y = s_y + warp * p.dim;
    const float rsd = 1.0f / sqrtf(static_cast<float>(p.dim));
    for (int64_t v = static_cast<int64_t>(blockIdx.x) * kWarps + warp; v < p.n;
         v += static_cast<int64_t>(gridDim.x) * kWarps) {
        const uint8_t* row = p.codes + v * p.bpv;
        for (int j = lane; j < p.dim; j += 32) y[j] = __ldg(p.centroids + code_at(row, j, p.bits));
        __syncwarp();
        const float sc = __half2float(__ushort_as_half(p.norms[v])) * rsd;
        for (int i = lane; i < p.dim; i += 32) {
            float acc = 0.0f;
            for (int j = 0; j < p.dim; ++j) acc = fmaf(__ldg(p.q + static_cast<int64_t>(j) * p.dim + i), y[j], acc);
            p.out[v * p.dim + i] = acc * sc;
        }
        __syncwarp();
    }
}

}  // namespace

cudaError_t launch_dequant(const tq_codec* c, const uint8_t* codes, const uint16_t* norms, int64_t n,
                           float* out, cudaStream_t st) {
    if (n <= 0) return cudaSuccess;
    DqParams p{codes, norms, n, out, c->d_centroids, c->d_sign_bits, c->d_q, c->bits, c->dim,
               c->bytes_per_vec};
    const int sms = num_sms(c->device);
    const int64_t want = (n + kWarps - 1) / kWarps;
    const int grid = static_cast<int>(want < int64_t(sms) * 16 ? want : int64_t(sms) * 16);
    if (c->is_wht) {
        switch (c->dim / 32) {
            case 1: dequant_wht_kernel<1><<<grid, kWarps * 32, 0, st>>>(p); break;
            case 2: dequant_wht_kernel<2><<<grid, kWarps * 32, 0, st>>>(p); break;
            case 4: dequant_wht_kernel<4><<<grid, kWarps * 32, 0, st>>>(p); break;
            case 8: dequant_wht_kernel<8><<<grid, kWarps * 32, 0, st>>>(p); break;
            case 16: dequant_wht_kernel<16><<<grid, kWarps * 32, 0, st>>>(p); break;
            default: return cudaErrorInvalidValue;
        }
    } else {
        dequant_dense_kernel<<<grid, kWarps * 32, sizeof(float) * kWarps * c->dim, st>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace tq
