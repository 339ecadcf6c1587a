// tq_decode_common.cuh -- pieces shared by the decode-attention kernels:
// workspace layout, query rotation, split-K partial publication and the
// last-arriving-CTA combine with the single inverse rotation.
//
// Scores are kept in log2 units: with q' = R q * (log2(e) * scale / sqrt(d)),
// s2_n = n16_K[n] * sum_j q'_j c_K[code_nj] equals log2(e) * scale * <q, K^_n>
// ("anyone still talking about mlx-swift-lm?": scores against K in its
// rotated basis).  V is accumulated in the rotated basis as
// acc_j = sum_n p_n n16_V[n] c_V[code_nj], and the output is
// o = R^T acc / (l sqrt(d)), i.e. diag(s) H acc / (l d) for the WHT rotation
// and Q^T acc / (l sqrt(d)) for the dense one.
#pragma once

#include <cuda_fp16.h>
#include <math_constants.h>

#include "tq_internal.h"

namespace tq {

constexpr unsigned kFullMask = 0xffffffffu;
constexpr int kGP = 8;                       // query slots per partial record
constexpr float kLog2e = 1.4426950408889634f;

// Partial record of one (virtual unit, split): o[kGP][d], m[kGP], l[kGP].
__device__ __forceinline__ float* partial_ptr(void* ws, const DecodePlan& p, int vu, int split, int d) {
    float* base = reinterpret_cast<float*>(static_cast<char*>(ws) + p.part_offset);
    return base + (static_cast<int64_t>(vu) * p.n_split + split) * (kGP * (d + 2));
}

__device__ __forceinline__ uint32_t* ticket_ptr(void* ws, const DecodePlan& p, int vu) {
    return reinterpret_cast<uint32_t*>(static_cast<char*>(ws) + p.ticket_offset) + vu;
}

__device__ __forceinline__ int32_t* error_ptr(void* ws) { return static_cast<int32_t*>(ws); }

// Clamped sequence length of batch b (flags out-of-range values).
__device__ __forceinline__ int64_t clamped_len(const DecodeArgs& a, int b) {
    int64_t L = __ldg(a.seq_lens + b);
    if (L < 0 || L > a.max_seq) {
        if (threadIdx.x == 0) atomicOr(error_ptr(a.ws), TQ_DEVERR_SEQ_LEN);
        L = L < 0 ? 0 : a.max_seq;
    }
    return L;
}

// q' for query head h into dst[0..d): the K rotation applied to q, scaled by
// log2(e) * scale / sqrt(d) (raw K: q * log2(e) * scale, no rotation).
// Executed by one full warp.
__device__ inline void rotate_query_warp(const DecodeArgs& a, int b, int h, float* dst) {
    const int lane = threadIdx.x & 31;
    const int d = a.cv.dim;
    const uint16_t* q = a.q + (static_cast<int64_t>(b) * a.Hq + h) * d;
    const DevCodec& ck = a.ck;
    if (ck.bits == 16) {
        const float f = kLog2e * a.scale;
        for (int j = lane; j < d; j += 32) dst[j] = __half2float(__ushort_as_half(q[j])) * f;
        __syncwarp();
        return;
    }
    if (ck.is_wht) {
        // dst <- s . q, then an in-place shared-memory butterfly (natural order).
        const uint32_t* sb = ck.sign_bits;
        for (int j = lane; j < d; j += 32) {
            const float v = __half2float(__ushort_as_half(q[j]));
            dst[j] = ((__ldg(sb + (j >> 5)) >> (j & 31)) & 1u) ? -v : v;
        }
        __syncwarp();
        for (int hh = 1; hh < d; hh <<= 1) {
            for (int i = lane; i < d / 2; i += 32) {
                const int lo = (i / hh) * (2 * hh) + (i % hh);
                const float x = dst[lo], y = dst[lo + hh];
                dst[lo] = x + y;
                dst[lo + hh] = x - y;
            }
            __syncwarp();
        }
        const float f = kLog2e * a.scale / static_cast<float>(d);
        for (int j = lane; j < d; j += 32) dst[j] *= f;
        __syncwarp();
    } else {
        const float* qt = ck.qt;  // Q^T row-major: (Q q)_j = sum_i Q^T[i][j] q_i
        const float f = kLog2e * a.scale * rsqrtf(static_cast<float>(d));
        for (int j = lane; j < d; j += 32) {
            float acc = 0.0f;
            for (int i = 0; i < d; ++i)
                acc = fmaf(__ldg(qt + static_cast<int64_t>(i) * d + j), __half2float(__ushort_as_half(q[i])), acc);
            dst[j] = acc * f;
        }
        __syncwarp();
    }
}

// Inverse V rotation and fp16 store of the normalised rotated outputs x[g][0..d)
// of query heads h0 + g, g < Gc (x in shared memory, overwritten).  `signs` are
// the V codec's sign words, in shared memory when the caller has them there.
__device__ inline void write_outputs(const DecodeArgs& a, int b, int h0, int Gc, float* x_all,
                                     const uint32_t* signs) {
    const int d = a.cv.dim;
    const int tid = threadIdx.x, nth = blockDim.x;
    const DevCodec& cv = a.cv;
    const int warp = tid >> 5, lane = tid & 31, nw = nth >> 5;
    if (cv.is_wht) {
        for (int g = warp; g < Gc; g += nw) {
            float* x = x_all + g * d;
            for (int hh = 1; hh < d; hh <<= 1) {
                for (int i = lane; i < d / 2; i += 32) {
                    const int lo = ((i & ~(hh - 1)) << 1) | (i & (hh - 1));
                    const float u = x[lo], v = x[lo + hh];
                    x[lo] = u + v;
                    x[lo + hh] = u - v;
                }
                __syncwarp();
            }
            const float f = 1.0f / static_cast<float>(d);
            uint16_t* o = a.out + (static_cast<int64_t>(b) * a.Hq + h0 + g) * d;
            for (int j = lane; j < d; j += 32) {
                const float v = x[j] * f;
                const bool neg = (signs[j >> 5] >> (j & 31)) & 1u;
                o[j] = __half_as_ushort(__float2half_rn(neg ? -v : v));
            }
        }
    } else {
        const float f = rsqrtf(static_cast<float>(d));
        for (int i = tid; i < Gc * d; i += nth) {
            const int g = i / d, col = i - g * d;
            const float* x = x_all + g * d;
            float acc = 0.0f;
#pragma unroll 8
            for (int j = 0; j < d; ++j) acc = fmaf(__ldg(cv.q + static_cast<int64_t>(j) * d + col), x[j], acc);
            a.out[(static_cast<int64_t>(b) * a.Hq + h0 + g) * d + col] = __half_as_ushort(__float2half_rn(acc * f));
        }
    }
}

// Publishes this CTA's partial (already in smem: so[kGP][d], sm[kGP], sl[kGP])
// and, if it is the last CTA of the virtual unit, combines all partials,
// applies the inverse V rotation and writes the fp16 outputs.
// The last CTA's path is a chain of L2 round trips, so it is kept short: one
// release atomic for the ticket, every partial of a group of outputs requested
// in one batch (CH splits at a time) together with the (m, l) pairs, and the
// sign words taken from shared memory (`signs`) when the caller has them.
// Must be called by all threads of the block.  scratch: >= kGP*(d + 2*n_split + 1) floats.
template <int CH>
__device__ inline void publish_and_combine(const DecodeArgs& a, const DecodePlan& p, int vu, int split,
                                           int b, int h0, int Gc, const float* so, const float* sm,
                                           const float* sl, float* scratch, int* s_flag,
                                           const uint32_t* signs) {
    const int d = a.cv.dim;
    const int tid = threadIdx.x, nth = blockDim.x;
    float* part = partial_ptr(a.ws, p, vu, split, d);
    for (int i = tid; i < kGP * d; i += nth) part[i] = so[i];
    for (int g = tid; g < kGP; g += nth) {
        part[kGP * d + g] = sm[g];
        part[kGP * d + kGP + g] = sl[g];
    }
    __syncthreads();
    if (tid == 0) {
        // the barrier orders the block's partial stores before this release atomic
        uint32_t prev;
        asm volatile("atom.add.release.gpu.global.u32 %0, [%1], 1;"
                     : "=r"(prev)
                     : "l"(ticket_ptr(a.ws, p, vu))
                     : "memory");
        const int last = (prev == static_cast<uint32_t>(p.n_split - 1)) ? 1 : 0;
        if (last) asm volatile("fence.acq_rel.gpu;" ::: "memory");  // acquire the other CTAs' partials
        *s_flag = last;
    }
    __syncthreads();
    if (*s_flag == 0) return;
    // ---- last CTA of this unit: merge partials ----
    const int ns = p.n_split;
    float* pm = scratch + kGP * d;   // [ns][kGP]: m, then the weights
    float* pl = pm + ns * kGP;       // [ns][kGP]: l
    float* inv = pl + ns * kGP;      // [kGP]: 1 / L
    const float* base = partial_ptr(a.ws, p, vu, 0, d);
    const int rec = kGP * (d + 2);
    const int nout = kGP * d;
    constexpr int OPT = 4;           // outputs per thread per group
    for (int i = tid; i < ns * kGP; i += nth) {
        const int sp = i / kGP, g = i - sp * kGP;
        pm[i] = __ldcg(base + sp * rec + kGP * d + g);
        pl[i] = __ldcg(base + sp * rec + kGP * d + kGP + g);
    }
    float ov[OPT][CH];
#pragma unroll
    for (int k = 0; k < OPT; ++k)
#pragma unroll
        for (int j = 0; j < CH; ++j) {
            const int i = tid + nth * k;
            ov[k][j] = (i < nout && j < ns) ? __ldcg(base + j * rec + i) : 0.0f;
        }
    __syncthreads();
    if (tid < kGP) {
        const int g = tid;
        float M = -CUDART_INF_F;
        for (int sp = 0; sp < ns; ++sp) M = fmaxf(M, pm[sp * kGP + g]);
        float L = 0.0f;
        for (int sp = 0; sp < ns; ++sp) {
            const float ms = pm[sp * kGP + g];
            const float w = (ms == -CUDART_INF_F) ? 0.0f : exp2f(ms - M);
            pm[sp * kGP + g] = w;
            L += w * pl[sp * kGP + g];
        }
        inv[g] = (L > 0.0f) ? 1.0f / L : 0.0f;
    }
    __syncthreads();
    int grp = 0;
    for (int i0 = tid; i0 < nout; i0 += nth * OPT, ++grp) {
        float acc[OPT];
#pragma unroll
        for (int k = 0; k < OPT; ++k) acc[k] = 0.0f;
        for (int c0 = 0; c0 < ns; c0 += CH) {
            if (grp > 0 || c0 > 0) {
#pragma unroll
                for (int k = 0; k < OPT; ++k)
#pragma unroll
                    for (int j = 0; j < CH; ++j) {
                        const int i = i0 + nth * k;
                        ov[k][j] = (i < nout && c0 + j < ns) ? __ldcg(base + (c0 + j) * rec + i) : 0.0f;
                    }
            }
#pragma unroll
            for (int k = 0; k < OPT; ++k) {
                const int i = i0 + nth * k;
                if (i < nout) {
                    const int g = i / d;
#pragma unroll
                    for (int j = 0; j < CH; ++j)
                        if (c0 + j < ns) acc[k] = fmaf(pm[(c0 + j) * kGP + g], ov[k][j], acc[k]);
                }
            }
        }
#pragma unroll
        for (int k = 0; k < OPT; ++k) {
            const int i = i0 + nth * k;
            if (i < nout) scratch[i] = acc[k] * inv[i / d];
        }
    }
    __syncthreads();
    write_outputs(a, b, h0, Gc, scratch, signs ? signs : a.cv.sign_bits);
    if (tid == 0) *ticket_ptr(a.ws, p, vu) = 0u;  // every CTA of this unit has arrived
}

}  // namespace tq
