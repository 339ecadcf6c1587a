// tq_decode_simt.cu -- general fused decode attention (any supported dim,
// bit width and GQA ratio) on the fp32 SIMT pipes.
//
// One CTA per (batch, KV head, group of <= 8 query rows, sequence split); the
// rows of a KV head are its G query heads times the L query positions of each,
// head-major.  Each warp walks every 8th token of the split: it unpacks the
// token's K codes, looks the centroids up in shared memory, scores all query
// rows of the group at once (GQA without expanding K/V: "add TurboQuant KV
// cache compression", review of the NR0 head mapping: a row's KV head follows
// from its query head), masks the tokens after each row's position, updates an
// online softmax
// and accumulates P . dequant(V) in the rotated basis ("anyone still talking
// about mlx-swift-lm?").  Warp states merge in shared memory and the CTA
// writes its split-K partial; the combine kernel (tq_decode_combine.cu)
// merges the splits and applies the single inverse V rotation.
//
// This path is the correctness baseline and the fallback for shapes the
// tensor-core kernel does not instantiate.
#include <atomic>
#include <algorithm>

#include "tq_decode_common.cuh"

namespace tq {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ int code_at(const uint8_t* row, int j, int bits) {
    const int p = j * bits;
    const int byte = p >> 3, sh = p & 7;
    uint32_t w = row[byte];
    if (sh + bits > 8) w |= static_cast<uint32_t>(row[byte + 1]) << 8;
    return static_cast<int>((w >> sh) & ((1u << bits) - 1u));
}

template <int E>
__global__ void __launch_bounds__(kThreads) decode_simt_kernel(const DecodeArgs a, const DecodePlan p) {
    extern __shared__ float smem[];
    constexpr int d = 32 * E;
    float* qs = smem;                    // [kGP][d]
    float* ctk = qs + kGP * d;           // [256]
    float* ctv = ctk + 256;              // [256]
    float* so = ctv + 256;               // [kGP][d]
    float* wm = so + kGP * d;            // [kWarps][kGP]
    float* wl = wm + kWarps * kGP;       // [kWarps][kGP]
    float* cm = wl + kWarps * kGP;       // [kGP]
    float* cl = cm + kGP;                // [kGP]
    float* uq = cl + kGP;                // [kGP][d] S q' (keys with the QJL sketch)

    allow_dependent_launch();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int vu = blockIdx.y, split = blockIdx.x;
    const int u = vu / p.q_chunks, qc = vu - (vu / p.q_chunks) * p.q_chunks;
    const int b = u / a.Hkv;
    const int kvh = u - b * a.Hkv;
    const int s0 = qc * kGP;                      // first row of this group within the unit
    const int Gc = min(kGP, p.S - s0);
    const int64_t row0q = (static_cast<int64_t>(b) * a.Hq + static_cast<int64_t>(kvh) * p.G) * p.L + s0;
    const int64_t len = clamped_len(a, b);
    const int64_t t0 = static_cast<int64_t>(split) * p.chunk;
    const int64_t t1 = min(len, t0 + p.chunk);
    // end of the packed tokens each row sees (causal; every token when L == 1)
    int64_t vis[kGP];
    {
        const int tail = p.L > 1 ? tail_count(a, b) : 0;
#pragma unroll
        for (int g = 0; g < kGP; ++g) vis[g] = packed_visible(len, tail, p.L, (s0 + g) % p.L);
    }

    if (warp < Gc) rotate_query_warp(a, row0q + warp, qs + warp * d);
    const bool rawk = a.ck.bits == 16;
    if (!rawk)
        for (int i = tid; i < (1 << a.ck.bits); i += kThreads) ctk[i] = __ldg(a.ck.centroids + i);
    for (int i = tid; i < (1 << a.cv.bits); i += kThreads) ctv[i] = __ldg(a.cv.centroids + i);
    for (int i = tid; i < kGP * d; i += kThreads) so[i] = 0.0f;
    __syncthreads();
    const bool qjl = a.ck.sketch != nullptr;
    if (qjl) {
        // u = S q' per query row: the sketch of the rotated, scaled query ("How I built
        // VeloxQuant-MLX", Stage 3: the correction reads <S_j, q> for every sketch row j)
        for (int idx = tid; idx < Gc * d; idx += kThreads) {
            const int g = idx / d, j = idx - (idx / d) * d;
            const float* srow = a.ck.sketch + static_cast<int64_t>(j) * d;
            float acc = 0.0f;
            for (int i = 0; i < d; ++i) acc = fmaf(__ldg(srow + i), qs[g * d + i], acc);
            uq[idx] = acc;
        }
        __syncthreads();
    }
    // QJL correction in score units: gamma sqrt(pi/2) / m * sqrt(d) with m = d sketch rows
    // (q' carries 1 / sqrt(d) of the rotation's scale)
    const float qjl_coef = 1.2533141373155003f * rsqrtf(static_cast<float>(d));

    float m[kGP], l[kGP], o[kGP][E];
#pragma unroll
    for (int g = 0; g < kGP; ++g) {
        m[g] = -CUDART_INF_F;
        l[g] = 0.0f;
#pragma unroll
        for (int e = 0; e < E; ++e) o[g][e] = 0.0f;
    }
    const int64_t row0 = static_cast<int64_t>(u) * a.max_seq;
    const int kb = a.ck.bits, vb = a.cv.bits;
    for (int64_t t = t0 + warp; t < t1; t += kWarps) {
        float kv[E];
        float nk = 1.0f;
        if (rawk) {
            const uint16_t* kr = static_cast<const uint16_t*>(a.k) + (row0 + t) * d + lane * E;
#pragma unroll
            for (int e = 0; e < E; ++e) kv[e] = __half2float(__ushort_as_half(kr[e]));
        } else {
            const uint8_t* kr = static_cast<const uint8_t*>(a.k) + (row0 + t) * a.ck.bpv;
#pragma unroll
            for (int e = 0; e < E; ++e) kv[e] = ctk[code_at(kr, lane * E + e, kb)];
            nk = __half2float(__ushort_as_half(a.k_norms[row0 + t]));
        }
        float s[kGP];
        if (qjl) {
            // <q, k^_MSE> + gamma sqrt(pi/2) / m sum_j z_j <S_j, R q>, this lane's E dims
            const uint32_t zb = static_cast<uint32_t>(code_at(a.k_signs + (row0 + t) * (d / 8), lane, E));
            const float gk = __half2float(__ushort_as_half(a.k_rnorms[row0 + t])) * qjl_coef;
#pragma unroll
            for (int g = 0; g < kGP; ++g) {
                float part = 0.0f, zq = 0.0f;
                if (g < Gc) {
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        part = fmaf(qs[g * d + lane * E + e], kv[e], part);
                        const float u = uq[g * d + lane * E + e];
                        zq += ((zb >> e) & 1u) ? -u : u;
                    }
                    part = fmaf(gk, zq, part * nk);
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(kFullMask, part, off);
                }
                s[g] = part;
            }
        } else {
#pragma unroll
            for (int g = 0; g < kGP; ++g) {
                float part = 0.0f;
                if (g < Gc) {
#pragma unroll
                    for (int e = 0; e < E; ++e) part = fmaf(qs[g * d + lane * E + e], kv[e], part);
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(kFullMask, part, off);
                }
                s[g] = part * nk;
            }
        }
        bool seen[kGP];
#pragma unroll
        for (int g = 0; g < kGP; ++g) seen[g] = g < Gc && t < vis[g];
        const uint8_t* vr = a.v_codes + (row0 + t) * a.cv.bpv;
        float vv[E];
#pragma unroll
        for (int e = 0; e < E; ++e) vv[e] = ctv[code_at(vr, lane * E + e, vb)];
        const float nv = __half2float(__ushort_as_half(a.v_norms[row0 + t]));
#pragma unroll
        for (int g = 0; g < kGP; ++g) {
            if (seen[g]) {
                const float mn = fmaxf(m[g], s[g]);
                const float alpha = exp2f(m[g] - mn);
                const float pp = exp2f(s[g] - mn);
                l[g] = fmaf(l[g], alpha, pp);
                const float pv = pp * nv;
#pragma unroll
                for (int e = 0; e < E; ++e) o[g][e] = fmaf(o[g][e], alpha, pv * vv[e]);
                m[g] = mn;
            }
        }
    }
    // ---- merge the warps of this CTA ----
    if (lane == 0)
#pragma unroll
        for (int g = 0; g < kGP; ++g) {
            wm[warp * kGP + g] = m[g];
            wl[warp * kGP + g] = l[g];
        }
    __syncthreads();
    // fixed warp order, so repeated calls give identical bits
    for (int w = 0; w < kWarps; ++w) {
        if (warp == w) {
#pragma unroll
            for (int g = 0; g < kGP; ++g) {
                if (g < Gc) {
                    float M = -CUDART_INF_F;
                    for (int w2 = 0; w2 < kWarps; ++w2) M = fmaxf(M, wm[w2 * kGP + g]);
                    const float f = (m[g] == -CUDART_INF_F) ? 0.0f : exp2f(m[g] - M);
#pragma unroll
                    for (int e = 0; e < E; ++e) so[g * d + lane * E + e] += o[g][e] * f;
                }
            }
        }
        __syncthreads();
    }
    if (tid < kGP) {
        const int g = tid;
        float M = -CUDART_INF_F;
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wm[w * kGP + g]);
        float L = 0.0f;
        for (int w = 0; w < kWarps; ++w) {
            const float mw = wm[w * kGP + g];
            if (mw != -CUDART_INF_F) L += wl[w * kGP + g] * exp2f(mw - M);
        }
        cm[g] = (g < Gc) ? M : -CUDART_INF_F;
        cl[g] = (g < Gc) ? L : 0.0f;
    }
    __syncthreads();
    write_partial(a, p, vu, split, so, cm, cl, tid, kThreads);
}

size_t simt_smem_bytes(int d) { return sizeof(float) * (size_t(kGP) * d * 3 + 512 + 2 * kWarps * kGP + 2 * kGP); }

template <int E>
cudaError_t launch_simt_e(const DecodeArgs& a, const DecodePlan& p, cudaStream_t st) {
    const size_t smem = simt_smem_bytes(32 * E);
    static std::atomic<uint64_t> configured{0};  // one bit per device
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t bit = 1ull << (dev & 63);
    if (!(configured.load() & bit)) {
        cudaError_t e = cudaFuncSetAttribute(decode_simt_kernel<E>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             200 * 1024);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit);
    }
    dim3 grid(p.n_split, p.n_units * p.q_chunks);
    decode_simt_kernel<E><<<grid, kThreads, smem, st>>>(a, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_simt(const DecodeArgs& a, const DecodePlan& p, cudaStream_t st) {
    switch (a.cv.dim / 32) {
        case 1: return launch_simt_e<1>(a, p, st);
        case 2: return launch_simt_e<2>(a, p, st);
        case 3: return launch_simt_e<3>(a, p, st);
        case 4: return launch_simt_e<4>(a, p, st);
        case 5: return launch_simt_e<5>(a, p, st);
        case 6: return launch_simt_e<6>(a, p, st);
        case 7: return launch_simt_e<7>(a, p, st);
        case 8: return launch_simt_e<8>(a, p, st);
        case 16: return launch_simt_e<16>(a, p, st);
        default: return cudaErrorNotSupported;
    }
}

bool make_decode_plan(int d, int device, int B, int Hq, int Hkv, int L, int64_t max_seq, DecodePlan& plan) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || max_seq <= 0 || d <= 0 || L <= 0) return false;
    plan = DecodePlan{};
    plan.G = Hq / Hkv;
    plan.L = L;
    if (int64_t(plan.G) * L > (1 << 20)) return false;
    plan.S = plan.G * L;
    plan.kernel = 0;
    plan.q_chunks = (plan.S + kGP - 1) / kGP;
    if (int64_t(B) * Hkv * plan.q_chunks > 65535) return false;  // grid y
    plan.n_units = B * Hkv;
    const int64_t vunits = int64_t(plan.n_units) * plan.q_chunks;
    const int64_t target = 2 * int64_t(num_sms(device));
    int64_t ns = (target + vunits - 1) / vunits;
    const int64_t cap = (max_seq + 255) / 256;
    if (ns > cap) ns = cap;
    if (ns < 1) ns = 1;
    int64_t chunk = (max_seq + ns - 1) / ns;
    chunk = (chunk + 63) / 64 * 64;
    plan.chunk = chunk;
    plan.n_split = int((max_seq + chunk - 1) / chunk);
    plan.part_offset = 256;  // after the device error word
    plan.decode_smem = 0;    // set by the tensor-core launcher
    // records: n_split per virtual unit, or, for the token-balanced schedule (one query
    // position, one row group per unit), one per CTA plus one per unit
    int64_t nrec = vunits * plan.n_split;
    if (L == 1 && plan.q_chunks == 1) nrec = std::max<int64_t>(nrec, num_sms(device) + int64_t(plan.n_units));
    plan.n_rec = int(nrec);
    plan.stream = 0;
    plan.n_cta = 0;
    plan.stream_ovh = 0;
    plan.ws_bytes = plan.part_offset + size_t(nrec) * kGP * (d + 2) * sizeof(float);
    return true;
}

}  // namespace tq
