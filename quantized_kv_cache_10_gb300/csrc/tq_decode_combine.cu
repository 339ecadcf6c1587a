// tq_decode_combine.cu -- split-K (flash-decoding) combine of the decode
// partials, the single inverse V rotation and the fp16 store.
//
// The decode kernels leave one record per (virtual unit, sequence split):
// o[kGP][d] relative to the split's running max m, with m and the weight sum l
// ("anyone still talking about mlx-swift-lm?": online softmax, P . V in the
// rotated basis).  This kernel merges them exactly as the online softmax
// would have: M = max_s m_s, w_s = 2^(m_s - M), L = sum_s w_s l_s,
// acc = sum_s w_s o_s / L, and returns acc to the original basis once
// ("add TurboQuant KV cache compression": R^T applied to the output, not to
// every cached vector): diag(s) H acc / d for the Walsh-Hadamard rotation,
// Q^T acc / sqrt(d) for the dense one.
//
// One CTA per (batch, query head).  It is launched with programmatic stream
// serialization: its CTAs may be resident before the decode grid finishes,
// and griddepcontrol.wait holds them until that grid has completed and its
// partial records are visible.  Every head is merged in parallel, each in one
// round of loads, instead of all heads of a unit by one last-arriving CTA.
#include "tq_decode_common.cuh"

namespace tq {
namespace {

constexpr int kCombineWarps = 4;

template <int N>
__device__ __forceinline__ void load_vec(const float* p, float (&v)[N]) {
    if constexpr (N % 4 == 0) {
#pragma unroll
        for (int i = 0; i < N / 4; ++i) {
            const float4 x = __ldcg(reinterpret_cast<const float4*>(p) + i);
            v[4 * i] = x.x;
            v[4 * i + 1] = x.y;
            v[4 * i + 2] = x.z;
            v[4 * i + 3] = x.w;
        }
    } else if constexpr (N % 2 == 0) {
#pragma unroll
        for (int i = 0; i < N / 2; ++i) {
            const float2 x = __ldcg(reinterpret_cast<const float2*>(p) + i);
            v[2 * i] = x.x;
            v[2 * i + 1] = x.y;
        }
    } else {
#pragma unroll
        for (int i = 0; i < N; ++i) v[i] = __ldcg(p + i);
    }
}

// Online merge of one more partial (m_s, l_s, o_s) into (m, l, acc).
template <int VPL>
__device__ __forceinline__ void merge_state(float& m, float& l, float (&acc)[VPL], float ms, float ls,
                                            const float (&os)[VPL]) {
    if (ms == -CUDART_INF_F) return;  // empty split
    const float mn = fmaxf(m, ms);
    const float a = exp2f(m - mn);    // 0 while m is -inf
    const float w = exp2f(ms - mn);
    l = fmaf(l, a, ls * w);
#pragma unroll
    for (int v = 0; v < VPL; ++v) acc[v] = fmaf(acc[v], a, os[v] * w);
    m = mn;
}

// One CTA per (batch, query head); VPL = d / 32 dims per lane: lane owns dims
// [VPL lane, VPL (lane + 1)).  Warp w merges splits w, w + 4, ... in one pass
// (every load of a batch in flight at once, no separate max pass), then warp 0
// merges the four warp states in a fixed order and writes the head's output.
template <int VPL>
__global__ void __launch_bounds__(kCombineWarps * 32) decode_combine_kernel(const DecodeArgs a, const DecodePlan p) {
    constexpr int D = 32 * VPL;
    __shared__ __align__(16) float s_o[kCombineWarps][D];
    __shared__ float s_m[kCombineWarps], s_l[kCombineWarps];
    __shared__ __align__(16) float s_ot[kCombineWarps][D];     // raw fp16 tail, original basis
    __shared__ float s_mt[kCombineWarps], s_lt[kCombineWarps];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // the V codec's sign word of this lane's dims (codec data, written by no kernel)
    uint32_t sw = 0;
    if ((VPL & (VPL - 1)) == 0 && a.cv.is_wht) sw = __ldg(a.cv.sign_bits + ((lane * VPL) >> 5));
    // let the next decode kernel on the stream start its table set-up, then
    // wait for this call's decode grid (and the visibility of its records)
    allow_dependent_launch();
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int pair = blockIdx.x;
    const int u = pair / p.G, hl = pair - (pair / p.G) * p.G;  // unit, head within its group
    const int qc = hl / kGP, g = hl - qc * kGP;
    const int vu = u * p.q_chunks + qc;
    const int b = u / a.Hkv;
    const int h = (u - b * a.Hkv) * p.G + hl;
    const int ns = p.n_split;
    const int rec = kGP * (D + 2);
    const float* base = partial_ptr(a.ws, p, vu, 0, D);
    const float* ob = base + g * D + lane * VPL;

    constexpr int CH = VPL <= 4 ? 8 : (VPL <= 8 ? 4 : 2);
    float m = -CUDART_INF_F, l = 0.0f, acc[VPL];
#pragma unroll
    for (int v = 0; v < VPL; ++v) acc[v] = 0.0f;
    for (int s0 = warp; s0 < ns; s0 += kCombineWarps * CH) {
        float ov[CH][VPL], mv[CH], lv[CH];
#pragma unroll
        for (int j = 0; j < CH; ++j) {
            const int sp = s0 + j * kCombineWarps;
            mv[j] = -CUDART_INF_F;
            lv[j] = 0.0f;
            if (sp < ns) {
                const float* r = base + static_cast<int64_t>(sp) * rec;
                mv[j] = __ldcg(r + kGP * D + g);
                lv[j] = __ldcg(r + kGP * D + kGP + g);
                load_vec<VPL>(ob + static_cast<int64_t>(sp) * rec, ov[j]);
            }
        }
#pragma unroll
        for (int j = 0; j < CH; ++j) merge_state<VPL>(m, l, acc, mv[j], lv[j], ov[j]);
    }
#pragma unroll
    for (int v = 0; v < VPL; ++v) s_o[warp][lane * VPL + v] = acc[v];
    if (lane == 0) {
        s_m[warp] = m;
        s_l[warp] = l;
    }
    // Unencoded fp16 tail tokens of the sequence (pending tokens, sink tokens) in the
    // same softmax: warp w scores tokens w, w + 4, ... against the unrotated query in
    // the original basis (log2 units, like the cache) and keeps its own online state.
    int nt = 0;
    if (a.tail_lens) {
        nt = __ldg(a.tail_lens + b);
        if (nt < 0 || nt > a.max_tail) {
            if (threadIdx.x == 0) atomicOr(error_ptr(a.ws), TQ_DEVERR_SEQ_LEN);
            nt = nt < 0 ? 0 : a.max_tail;
        }
    }
    if (nt > 0) {
        float qv[VPL], mt = -CUDART_INF_F, lt = 0.0f, ot[VPL];
        const float f = kLog2e * a.scale;
        const uint16_t* qh = a.q + (static_cast<int64_t>(b) * a.Hq + h) * D + lane * VPL;
#pragma unroll
        for (int v = 0; v < VPL; ++v) {
            qv[v] = __half2float(__ushort_as_half(qh[v])) * f;
            ot[v] = 0.0f;
        }
        const int64_t row0 = (static_cast<int64_t>(b) * a.Hkv + (h / p.G)) * a.max_tail;
        for (int n = warp; n < nt; n += kCombineWarps) {
            const uint16_t* kr = a.k_tail + (row0 + n) * D + lane * VPL;
            const uint16_t* vr = a.v_tail + (row0 + n) * D + lane * VPL;
            float part = 0.0f, vv[VPL];
#pragma unroll
            for (int v = 0; v < VPL; ++v) {
                part = fmaf(qv[v], __half2float(__ushort_as_half(kr[v])), part);
                vv[v] = __half2float(__ushort_as_half(vr[v]));
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(kFullMask, part, off);
            const float mn = fmaxf(mt, part);
            const float al = exp2f(mt - mn);  // 0 while mt is -inf
            const float pw = exp2f(part - mn);
            lt = fmaf(lt, al, pw);
#pragma unroll
            for (int v = 0; v < VPL; ++v) ot[v] = fmaf(ot[v], al, pw * vv[v]);
            mt = mn;
        }
#pragma unroll
        for (int v = 0; v < VPL; ++v) s_ot[warp][lane * VPL + v] = ot[v];
        if (lane == 0) {
            s_mt[warp] = mt;
            s_lt[warp] = lt;
        }
    }
    __syncthreads();
    if (warp != 0) return;
    m = -CUDART_INF_F;
    l = 0.0f;
#pragma unroll
    for (int v = 0; v < VPL; ++v) acc[v] = 0.0f;
#pragma unroll
    for (int w = 0; w < kCombineWarps; ++w) {
        float os[VPL];
#pragma unroll
        for (int v = 0; v < VPL; ++v) os[v] = s_o[w][lane * VPL + v];
        merge_state<VPL>(m, l, acc, s_m[w], s_l[w], os);
    }
    const float inv = (l > 0.0f) ? 1.0f / l : 0.0f;  // seq_len 0: zero output
#pragma unroll
    for (int v = 0; v < VPL; ++v) acc[v] *= inv;

    float res[VPL];
    bool done = false;
    if constexpr ((VPL & (VPL - 1)) == 0) {
        if (a.cv.is_wht) {
            // H acc: butterflies of stride < VPL inside the lane, the rest across lanes
#pragma unroll
            for (int hh = 1; hh < VPL; hh <<= 1)
#pragma unroll
                for (int v = 0; v < VPL; ++v)
                    if (!(v & hh)) {
                        const float x = acc[v], y = acc[v + hh];
                        acc[v] = x + y;
                        acc[v + hh] = x - y;
                    }
#pragma unroll
            for (int lm = 1; lm < 32; lm <<= 1) {
                const bool upper = (lane & lm) != 0;
#pragma unroll
                for (int v = 0; v < VPL; ++v) {
                    const float y = __shfl_xor_sync(kFullMask, acc[v], lm);
                    acc[v] = upper ? (y - acc[v]) : (acc[v] + y);
                }
            }
            const float f = 1.0f / static_cast<float>(D);
            const int sb = (lane * VPL) & 31;
#pragma unroll
            for (int v = 0; v < VPL; ++v) {
                const float x = acc[v] * f;
                res[v] = ((sw >> (sb + v)) & 1u) ? -x : x;
            }
            done = true;
        }
    }
    if (!done) {
        // Q^T acc / sqrt(d): column c of the output is sum_j Q[j][c] acc[j], j ascending
        const float f = rsqrtf(static_cast<float>(D));
#pragma unroll
        for (int v = 0; v < VPL; ++v) res[v] = 0.0f;
        const float* qcol = a.cv.q + lane * VPL;
        for (int src = 0; src < 32; ++src) {
#pragma unroll
            for (int w = 0; w < VPL; ++w) {
                const float xj = __shfl_sync(kFullMask, acc[w], src);
                const float* qrow = qcol + static_cast<int64_t>(src * VPL + w) * D;
#pragma unroll
                for (int v = 0; v < VPL; ++v) res[v] = fmaf(__ldg(qrow + v), xj, res[v]);
            }
        }
#pragma unroll
        for (int v = 0; v < VPL; ++v) res[v] *= f;
    }
    if (nt > 0) {
        // merge the tail's state (original basis) with the cache's normalised output res:
        // out = (W_c res + W_t o_t / l_t) / (W_c + W_t), W = sum of weights relative to one max
        float mt = -CUDART_INF_F, lt = 0.0f, ot[VPL];
#pragma unroll
        for (int v = 0; v < VPL; ++v) ot[v] = 0.0f;
#pragma unroll
        for (int w = 0; w < kCombineWarps; ++w) {
            if (w < nt) {  // warps beyond the tail length hold no state
                float os[VPL];
#pragma unroll
                for (int v = 0; v < VPL; ++v) os[v] = s_ot[w][lane * VPL + v];
                merge_state<VPL>(mt, lt, ot, s_mt[w], s_lt[w], os);
            }
        }
        const float mm = fmaxf(m, mt);
        const float wc = (m == -CUDART_INF_F) ? 0.0f : l * exp2f(m - mm);
        const float wt = lt * exp2f(mt - mm);
        const float den = wc + wt;
        const float ic = den > 0.0f ? wc / den : 0.0f, it = den > 0.0f ? exp2f(mt - mm) / den : 0.0f;
#pragma unroll
        for (int v = 0; v < VPL; ++v) res[v] = fmaf(res[v], ic, ot[v] * it);
    }
    uint16_t* o = a.out + (static_cast<int64_t>(b) * a.Hq + h) * D + lane * VPL;
    if constexpr (VPL % 2 == 0) {
        // out is 4-byte aligned and VPL lane offsets are even: 32-bit stores
        uint32_t* o32 = reinterpret_cast<uint32_t*>(o);
#pragma unroll
        for (int v = 0; v < VPL; v += 2)
            o32[v / 2] = uint32_t(__half_as_ushort(__float2half_rn(res[v]))) |
                         (uint32_t(__half_as_ushort(__float2half_rn(res[v + 1]))) << 16);
    } else {
#pragma unroll
        for (int v = 0; v < VPL; ++v) o[v] = __half_as_ushort(__float2half_rn(res[v]));
    }
}

template <int VPL>
cudaError_t launch_vpl(const DecodeArgs& a, const DecodePlan& p, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.n_units * p.G);
    cfg.blockDim = dim3(kCombineWarps * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_combine_kernel<VPL>, a, p);
}

}  // namespace

cudaError_t launch_decode_combine(const DecodeArgs& a, const DecodePlan& p, cudaStream_t st) {
    switch (a.cv.dim / 32) {
        case 1: return launch_vpl<1>(a, p, st);
        case 2: return launch_vpl<2>(a, p, st);
        case 3: return launch_vpl<3>(a, p, st);
        case 4: return launch_vpl<4>(a, p, st);
        case 5: return launch_vpl<5>(a, p, st);
        case 6: return launch_vpl<6>(a, p, st);
        case 7: return launch_vpl<7>(a, p, st);
        case 8: return launch_vpl<8>(a, p, st);
        case 16: return launch_vpl<16>(a, p, st);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace tq
