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
// One CTA per query row (batch, query head, query position).  It is launched
// with programmatic stream serialization: its CTAs may be resident before the
// decode grid finishes, and griddepcontrol.wait holds them until that grid has
// completed and its partial records are visible.  Every row is merged in
// parallel, each in one round of loads, instead of all rows of a unit by one
// last-arriving CTA.
#include <atomic>

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

// VPL consecutive fp16 values (a lane's dims of one row) as packed pairs, bypassing L1:
// one 4-, 8- or 16-byte load where VPL allows (the rows are 16-byte aligned).
template <int VPL>
__device__ __forceinline__ void load_halves(const uint16_t* p, uint32_t (&h)[(VPL + 1) / 2]) {
    if constexpr (VPL % 8 == 0) {
#pragma unroll
        for (int i = 0; i < VPL / 8; ++i) {
            const uint4 x = __ldcg(reinterpret_cast<const uint4*>(p) + i);
            h[4 * i] = x.x;
            h[4 * i + 1] = x.y;
            h[4 * i + 2] = x.z;
            h[4 * i + 3] = x.w;
        }
    } else if constexpr (VPL == 4) {
        const uint2 x = __ldcg(reinterpret_cast<const uint2*>(p));
        h[0] = x.x;
        h[1] = x.y;
    } else if constexpr (VPL == 2) {
        h[0] = __ldcg(reinterpret_cast<const unsigned int*>(p));
    } else {
#pragma unroll
        for (int i = 0; i < (VPL + 1) / 2; ++i) {
            const uint32_t lo = __ldcg(p + 2 * i);
            const uint32_t hi = (2 * i + 1 < VPL) ? __ldcg(p + 2 * i + 1) : 0u;
            h[i] = lo | (hi << 16);
        }
    }
}

__device__ __forceinline__ float half_at(const uint32_t* h, int v) {
    return __half2float(__ushort_as_half(static_cast<uint16_t>(h[v >> 1] >> (16 * (v & 1)))));
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

// x (lane owns dims [VPL lane, VPL (lane + 1)), original basis) -> sqrt(d) R x, the units
// of the decode kernels' rotated accumulators: H (s . x) for the Walsh-Hadamard
// rotation R = H diag(s) / sqrt(d), sqrt(d) Q x for the dense one.
template <int VPL>
__device__ __forceinline__ void to_rotated_units(const DecodeArgs& a, float (&x)[VPL], int lane) {
    constexpr int D = 32 * VPL;
    if constexpr ((VPL & (VPL - 1)) == 0) {
        if (a.cv.is_wht) {
            const uint32_t sw = __ldg(a.cv.sign_bits + ((lane * VPL) >> 5));
            const int sb = (lane * VPL) & 31;
#pragma unroll
            for (int v = 0; v < VPL; ++v)
                if ((sw >> (sb + v)) & 1u) x[v] = -x[v];
#pragma unroll
            for (int hh = 1; hh < VPL; hh <<= 1)
#pragma unroll
                for (int v = 0; v < VPL; ++v)
                    if (!(v & hh)) {
                        const float p = x[v], q = x[v + hh];
                        x[v] = p + q;
                        x[v + hh] = p - q;
                    }
#pragma unroll
            for (int lm = 1; lm < 32; lm <<= 1) {
                const bool upper = (lane & lm) != 0;
#pragma unroll
                for (int v = 0; v < VPL; ++v) {
                    const float y = __shfl_xor_sync(kFullMask, x[v], lm);
                    x[v] = upper ? (y - x[v]) : (x[v] + y);
                }
            }
            return;
        }
    }
    // (Q x)_i = sum_j Q^T[j][i] x_j, j ascending
    float r[VPL];
#pragma unroll
    for (int v = 0; v < VPL; ++v) r[v] = 0.0f;
    const float* qcol = a.cv.qt + lane * VPL;
    for (int src = 0; src < 32; ++src) {
#pragma unroll
        for (int w = 0; w < VPL; ++w) {
            const float xj = __shfl_sync(kFullMask, x[w], src);
            const float* qrow = qcol + static_cast<int64_t>(src * VPL + w) * D;
#pragma unroll
            for (int v = 0; v < VPL; ++v) r[v] = fmaf(__ldg(qrow + v), xj, r[v]);
        }
    }
    const float sd = sqrtf(static_cast<float>(D));
#pragma unroll
    for (int v = 0; v < VPL; ++v) x[v] = r[v] * sd;
}

// One CTA per query row (batch, query head, query position); VPL = d / 32 dims per
// lane: lane owns dims
// [VPL lane, VPL (lane + 1)).  Warp w merges splits w, w + 4, ... in one pass
// (every load of a batch in flight at once, no separate max pass), then warp 0
// merges the four warp states in a fixed order and writes the head's output.
//
// Residence beside the decode kernel: the combine grid becomes eligible while every
// decode CTA is resident, and only if a combine CTA fits beside one does it start there
// (scoring the tail during the decode); otherwise its CTAs wait for the first SMs the
// decode grid frees and pile up there, several per SM, keeping the next call's decode
// CTAs off those SMs.  So it uses at most 64 registers per thread up to d = 160 (one
// warp per SM sub-partition fits beside three 144-register decode warps), the same
// shared-memory split as the decode kernel, and a shared-memory pad sized at launch
// so that exactly one combine CTA fits beside a decode CTA.
// WIDE: the instantiation for decode kernels that fill their SMs (the token-balanced
// schedule), beside which no combine CTA runs anyway: eight tail tokens per warp and round
// instead of two, for four times fewer round trips to memory (up to 128 registers).
template <int VPL, bool WIDE>
__global__ void __launch_bounds__(kCombineWarps * 32, (WIDE ? 4 : (VPL <= 5 ? 8 : 4)))
    decode_combine_kernel(const DecodeArgs a, const DecodePlan p) {
    constexpr int D = 32 * VPL;
    __shared__ __align__(16) float s_o[kCombineWarps][D];
    __shared__ float s_m[kCombineWarps], s_l[kCombineWarps];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#ifdef TQ_TIMELINE
    unsigned long long tl_t[kTlStamps] = {};  // entry, dependency wait passed, output stored, SM id
#endif
    TQ_TL(tl_t, 0);
    // the V codec's sign word of this lane's dims (codec data, written by no kernel)
    uint32_t sw = 0;
    if ((VPL & (VPL - 1)) == 0 && a.cv.is_wht) sw = __ldg(a.cv.sign_bits + ((lane * VPL) >> 5));
    const int pair = blockIdx.x;
    const int u = pair / p.S, hl = pair - (pair / p.S) * p.S;  // unit, row within the unit
    const int qc = hl / kGP, g = hl - qc * kGP;
    const int vu = u * p.q_chunks + qc;
    const int b = u / a.Hkv;
    const int kvh = u - b * a.Hkv;
    const int ell = hl % p.L;  // query position (the unit's rows are head-major)
    const int64_t qrow = (static_cast<int64_t>(b) * a.Hq + static_cast<int64_t>(kvh) * p.G) * p.L + hl;
    // let the next decode kernel on the stream start its table set-up
    allow_dependent_launch();
    // Unencoded fp16 tail tokens of the sequence (pending tokens, sink tokens) in the
    // same softmax: warp w scores tokens w, w + 4, ... against the unrotated query in
    // the original basis (log2 units, like the cache) and keeps its own online state.
    // The decode kernel triggers this grid only after its own dependency wait, so the
    // call's inputs (q, the tail, the new token) are complete here, before this
    // grid's wait: the tail overlaps the decode kernel.  (Loads bypass L1.)
    float tail_m = -CUDART_INF_F, tail_l = 0.0f, tail_o[VPL];
#pragma unroll
    for (int v = 0; v < VPL; ++v) tail_o[v] = 0.0f;
    const int nt = tail_count(a, b);  // tail tokens in the buffer
    const int nvis = p.L > 1 ? tail_visible(nt, p.L, ell) : nt;  // of them before this row's position
    const int64_t tail_row0 = (static_cast<int64_t>(b) * a.Hkv + kvh) * a.max_tail;
    const int64_t new_row = static_cast<int64_t>(b) * a.Hkv + kvh;
    const int ntot = nvis + (a.k_new ? 1 : 0);  // the new token is scored after the buffer's
    if (a.k_new && hl == 0 && warp == 0) {
        // append the new token to the tail buffer (one CTA per KV head writes it; the
        // other CTAs of the head read only tokens below nt)
        if (nt < a.max_tail) {
            const uint16_t* ks = a.k_new + new_row * D;
            const uint16_t* vs = a.v_new + new_row * D;
            uint16_t* kd = const_cast<uint16_t*>(a.k_tail) + (tail_row0 + nt) * D;
            uint16_t* vd = const_cast<uint16_t*>(a.v_tail) + (tail_row0 + nt) * D;
            for (int i = lane; i < D; i += 32) {
                kd[i] = __ldcg(ks + i);
                vd[i] = __ldcg(vs + i);
            }
        } else if (lane == 0) {
            atomicOr(error_ptr(a.ws), TQ_DEVERR_SEQ_LEN);
        }
    }
    if (ntot > 0) {
        float qv[VPL], mt = -CUDART_INF_F, lt = 0.0f, ot[VPL];
        const float f = kLog2e * a.scale;
        const uint16_t* qh = a.q + qrow * D + lane * VPL;
#pragma unroll
        for (int v = 0; v < VPL; ++v) {
            qv[v] = __half2float(__ushort_as_half(__ldcg(qh + v))) * f;
            ot[v] = 0.0f;
        }
        // TCH tokens per round with all their loads in flight (one memory latency per round)
        constexpr int TCH = WIDE ? (VPL >= 16 ? 4 : 8) : (VPL <= 2 ? 4 : 2);
        constexpr int HW = (VPL + 1) / 2;  // packed fp16 pairs per row slice
        for (int n0 = warp; n0 < ntot; n0 += kCombineWarps * TCH) {
            uint32_t kh[TCH][HW], vh[TCH][HW];
#pragma unroll
            for (int j = 0; j < TCH; ++j) {
                const int n = n0 + j * kCombineWarps;
                if (n < ntot) {
                    const int64_t row = (n < nvis) ? (tail_row0 + n) : new_row;
                    load_halves<VPL>(((n < nvis) ? a.k_tail : a.k_new) + row * D + lane * VPL, kh[j]);
                    load_halves<VPL>(((n < nvis) ? a.v_tail : a.v_new) + row * D + lane * VPL, vh[j]);
                }
            }
#pragma unroll
            for (int j = 0; j < TCH; ++j) {
                if (n0 + j * kCombineWarps < ntot) {
                    float part = 0.0f;
#pragma unroll
                    for (int v = 0; v < VPL; ++v) part = fmaf(qv[v], half_at(kh[j], v), part);
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(kFullMask, part, off);
                    const float mn = fmaxf(mt, part);
                    const float al = exp2f(mt - mn);  // 0 while mt is -inf
                    const float pw = exp2f(part - mn);
                    lt = fmaf(lt, al, pw);
#pragma unroll
                    for (int v = 0; v < VPL; ++v) ot[v] = fmaf(ot[v], al, pw * half_at(vh[j], v));
                    mt = mn;
                }
            }
        }
        // into the units of the cache's accumulator, sqrt(d) R o_t (= H (s . o_t) for the
        // Walsh-Hadamard rotation, sqrt(d) Q o_t for the dense one), so that the tail merges
        // with the cache partials like one more partial
        to_rotated_units<VPL>(a, ot, lane);
        tail_m = mt;
        tail_l = lt;
#pragma unroll
        for (int v = 0; v < VPL; ++v) tail_o[v] = ot[v];
    }
    // This row's records: n_split of them, or, on the token-balanced schedule, those of the
    // CTAs whose positions cover the unit (none while the sequence is empty), found from
    // the lengths here, before the wait, while the decode kernel runs.
    int ns = p.n_split;
    int64_t rec0 = static_cast<int64_t>(vu) * p.n_split;
    if (p.stream) {
        int64_t first;
        stream_unit_ctas(a, p.n_cta, p.stream_ovh, b, kvh, lane, first, ns);
        rec0 = first + u;
    }
    // wait for this call's decode grid (and the visibility of its records)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    TQ_TL(tl_t, 1);
    const int rec = kGP * (D + 2);
    const float* base = partial_slot_ptr(a.ws, p, rec0, D);
    const float* ob = base + g * D + lane * VPL;

    constexpr int CH = VPL <= 4 ? 5 : (VPL <= 8 ? 4 : 2);
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
    merge_state<VPL>(m, l, acc, tail_m, tail_l, tail_o);  // (a no-op without tail tokens)
#pragma unroll
    for (int v = 0; v < VPL; ++v) s_o[warp][lane * VPL + v] = acc[v];
    if (lane == 0) {
        s_m[warp] = m;
        s_l[warp] = l;
    }
    __syncthreads();
    // the dense inverse rotation is shared by the four warps; the Walsh-Hadamard one is
    // warp 0's alone
    const bool dense = !((VPL & (VPL - 1)) == 0 && a.cv.is_wht);
    if (!dense && warp != 0) return;
    if (warp == 0) {
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
        if (dense) {  // the merged row for every warp (warp 0 has read the states)
#pragma unroll
            for (int v = 0; v < VPL; ++v) s_o[0][lane * VPL + v] = acc[v];
        }
    }

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
        // Q^T acc / sqrt(d): column c of the output is sum_j Q[j][c] acc[j]; warp w sums the
        // quarter j in [w D/4, (w + 1) D/4) ascending (Q rows across the lanes, acc[j] a
        // broadcast from shared memory), and warp 0 adds the four in a fixed order
        __syncthreads();
        const float f = rsqrtf(static_cast<float>(D));
        constexpr int JW = (D + kCombineWarps - 1) / kCombineWarps;
#pragma unroll
        for (int v = 0; v < VPL; ++v) res[v] = 0.0f;
        const float* qcol = a.cv.q + lane * VPL;
#pragma unroll
        for (int jj = 0; jj < JW; ++jj) {  // (unrolled: every load of the quarter in flight at once)
            const int j = warp * JW + jj;
            if (j < D) {
                const float xj = s_o[0][j];
                const float* qrow = qcol + static_cast<int64_t>(j) * D;
#pragma unroll
                for (int v = 0; v < VPL; ++v) res[v] = fmaf(__ldg(qrow + v), xj, res[v]);
            }
        }
        __syncthreads();  // every warp has read the merged row
        if (warp != 0) {
#pragma unroll
            for (int v = 0; v < VPL; ++v) s_o[warp][lane * VPL + v] = res[v];
        }
        __syncthreads();
        if (warp != 0) return;
#pragma unroll
        for (int w = 1; w < kCombineWarps; ++w)
#pragma unroll
            for (int v = 0; v < VPL; ++v) res[v] += s_o[w][lane * VPL + v];
#pragma unroll
        for (int v = 0; v < VPL; ++v) res[v] *= f;
    }
    uint16_t* o = a.out + qrow * D + lane * VPL;
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
#ifdef TQ_TIMELINE
    TQ_TL(tl_t, 2);
    if (threadIdx.x == 0 && a.tl) {
        unsigned sm;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
        tl_t[3] = sm;  // the SM this CTA ran on
        unsigned long long* r = tl_record(a, true, blockIdx.x);
        if (r)
            for (int i = 0; i < kTlStamps; ++i) r[i] = tl_t[i];
    }
#endif
}

// Shared memory per SM and reserved per CTA on the current device (cached per device).
void smem_limits(int& per_sm, int& reserved) {
    static std::atomic<int> cache_sm[64], cache_res[64];
    int dev = 0;
    cudaGetDevice(&dev);
    const int i = dev & 63;
    per_sm = cache_sm[i].load();
    reserved = cache_res[i].load();
    if (per_sm == 0) {
        if (cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess) per_sm = 0;
        if (cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess) reserved = 0;
        cache_res[i].store(reserved);
        cache_sm[i].store(per_sm);
    }
}

// Dynamic shared memory that pads a combine CTA so that exactly one fits beside a
// decode CTA of the kernel just launched (0 when that is not in reach).  The combine
// grid becomes eligible while every decode CTA is resident; padded this way its CTAs
// spread one per SM instead of several on the SMs that free up first, where they
// would keep out the next call's decode CTA (a second one does not fit there either).
int combine_pad_bytes(int decode_smem, int static_bytes) {
    if (decode_smem <= 0) return 0;
    int per_sm = 0, reserved = 0;
    smem_limits(per_sm, reserved);
    const int free_bytes = per_sm - (decode_smem + reserved);  // beside one decode CTA
    const int own = static_bytes + reserved;                   // one combine CTA, unpadded
    if (free_bytes < own || free_bytes > 96 * 1024) return 0;
    // one padded CTA: own + pad <= free_bytes - 256; two: 2 (own + pad) > free_bytes
    const int pad = free_bytes / 2 + 256 - own;
    if (pad <= 0 || own + pad > free_bytes - 256 || pad > 48 * 1024) return 0;
    return (pad + 127) / 128 * 128;
}

template <int VPL, bool WIDE>
cudaError_t launch_vpl(const DecodeArgs& a, const DecodePlan& p, cudaStream_t st) {
    // The L1 / shared-memory split of an SM is set for the CTAs it holds, and a CTA whose
    // kernel prefers another split waits for an idle SM: the combine asks for the same
    // all-shared-memory split as the decode kernel, so that it can run beside it.
    static std::atomic<uint64_t> configured{0};  // one bit per device
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t bit = 1ull << (dev & 63);
    if (!(configured.load() & bit)) {
        const cudaError_t e = cudaFuncSetAttribute(decode_combine_kernel<VPL, WIDE>,
                                                   cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.n_units * p.S);
    cfg.blockDim = dim3(kCombineWarps * 32);
    constexpr int kStatic = kCombineWarps * 32 * VPL * 4 + 2 * kCombineWarps * 4;  // s_o, s_m, s_l
    cfg.dynamicSmemBytes = combine_pad_bytes(p.decode_smem, kStatic);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_combine_kernel<VPL, WIDE>, a, p);
}

template <bool WIDE>
cudaError_t launch_wide(const DecodeArgs& a, const DecodePlan& p, cudaStream_t st) {
    switch (a.cv.dim / 32) {
        case 1: return launch_vpl<1, WIDE>(a, p, st);
        case 2: return launch_vpl<2, WIDE>(a, p, st);
        case 3: return launch_vpl<3, WIDE>(a, p, st);
        case 4: return launch_vpl<4, WIDE>(a, p, st);
        case 5: return launch_vpl<5, WIDE>(a, p, st);
        case 6: return launch_vpl<6, WIDE>(a, p, st);
        case 7: return launch_vpl<7, WIDE>(a, p, st);
        case 8: return launch_vpl<8, WIDE>(a, p, st);
        case 16: return launch_vpl<16, WIDE>(a, p, st);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace

cudaError_t launch_decode_combine(const DecodeArgs& a, const DecodePlan& p, cudaStream_t st) {
    return p.stream ? launch_wide<true>(a, p, st) : launch_wide<false>(a, p, st);
}

}  // namespace tq
