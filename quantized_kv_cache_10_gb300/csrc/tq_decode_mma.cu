// tq_decode_mma.cu -- host side of the tensor-core fused decode attention for GQA groups of up
// to 8 query heads ("anyone still talking about mlx-swift-lm?": one dispatch,
// K read once in its rotated basis, inline dequant; "add TurboQuant KV cache
// compression", review of the NR0 path: every query head of a KV head's group
// served from one read of that head's cache).
//
// Per CTA: one (batch, KV head, sequence split).  One producer warp streams
// tiles of TS tokens (packed K codes, packed V codes, both norm vectors) into
// an NSTAGE-deep shared-memory ring with 1-D TMA bulk copies
// (cp.async.bulk ... mbarrier::complete_tx); eight consumer warps each take
// 16*MT tokens of a tile:
//   scores  S[16 tok x 8 col] += Khat[16 x 16 dims] * Q'[16 dims x 8 col]
//           (mma.sync m16n8k16, fp16 in, fp32 accumulate), Khat built in
//           registers from the codes through replicated shared-memory tables
//           holding each centroid as fp16 hi + fp16 lo, and q' split the same
//           way into separate columns, so the product keeps ~fp32 accuracy;
//   softmax online in fp32 (exp2 of log2-scaled scores);
//   P.V     O^T[16 dims x 8 col] += Vhat^T[16 dims x 16 tok] * P[16 tok x 8]
//           with P moved from the score layout by movmatrix.trans and Vhat
//           looked up two tokens at a time from a pair table.
// Warps merge in shared memory in a fixed order and the CTA writes its split-K
// partial; the combine kernel (tq_decode_combine.cu) merges the splits and
// applies the single inverse V rotation.
//
// Register/shared layouts (thread = 4*g + t in its warp):
//   K role (A of the score mma, rows = tokens): thread t owns dims
//     [(D/4) t, (D/4)(t+1)); k-tile kt uses dims (D/4) t + 4 kt + {0,1,2,3}
//     for the k columns {2t, 2t+1, 2t+8, 2t+9}.  The q' B fragment uses the
//     same map.
//   V role (A of the P.V mma, rows = dims): thread g owns dims
//     [(D/8) g, (D/8)(g+1)); m-tile dm rows g / g+8 are dims (D/8) g + 2 dm + 0/1.
//   Query columns: NT == 2 (5..8 heads): column j of n-tile 0 / 1 = q_hi / q_lo
//     of head j; NT == 1 (<= 4 heads): column 2j / 2j+1 = q_hi / q_lo of head j,
//     and in P.V head j sits in column 2j.
#include <cuda_fp16.h>

#include <algorithm>
#include <cmath>

#include "tq_decode_mma.cuh"

namespace tq {

// Positions without tokens per unit on the token-balanced schedule, at d <= 128 (scaled by
// 128 / d) and at d 256.
constexpr int kStreamOvhD128 = 768;
constexpr int kStreamOvhD256 = 320;

// ---------------------------------------------------------------------------
// Host: compact decode tables, built once per codec.
// The tensor cores take fp16 operands, and a centroid rounded to fp16 is off
// by up to 2^-11 of itself -- a fixed error per code that does not average
// out.  Every codebook value is therefore stored scaled by a factor alpha in
// [1, 2) chosen so that the fp16 roundings of alpha * |c_i| are as close to
// exact as possible (for 2/3/4-bit codebooks the worst relative error drops
// from ~2^-12 to ~2^-21 / 2^-15.5 / 2^-13.5); the kernel divides alpha out
// of q' (K) or of the output (V).
//   ktab: K role.  bits <= 4: per pair index p = c0 | c1 << bits one word
//         h(c0) | h(c1) << 16 with h(c) = fp16(alpha c);  bits == 8 (alpha 1):
//         one word per code hi | lo << 16, hi = fp16(c), lo = fp16(c - hi).
//   vtab: V role.  bits <= 4: per pair index one word h(c0) | h(c1) << 16;
//         bits == 8: one word per code h | h << 16.
// ---------------------------------------------------------------------------
namespace {

uint16_t f16_bits(float x) {
    __half h = __float2half_rn(x);
    return __half_as_ushort(h);
}

float f16_val(uint16_t b) { return __half2float(__ushort_as_half(b)); }

// Relative error of rounding x > 0 to the nearest fp16 (normal range, ties
// to even do not matter for the maximum), in double arithmetic.
double f16_rel_err(double x) {
    int e = 0;
    std::frexp(x, &e);                         // x = m 2^e, m in [0.5, 1)
    const double ulp = std::ldexp(1.0, e - 11);
    return std::fabs(x - std::nearbyint(x / ulp) * ulp) / x;
}

// alpha = 1 + i / steps minimising the worst relative fp16 rounding error of
// alpha * |c| over the codebook (first such i on ties).
float table_alpha(const std::vector<float>& cent, int steps) {
    std::vector<double> mags;
    for (float v : cent) {
        const double m = std::fabs(double(v));
        if (m > 0.0 && std::find(mags.begin(), mags.end(), m) == mags.end()) mags.push_back(m);
    }
    double best = 1e300;
    int best_i = 0;
    for (int i = 0; i < steps; ++i) {
        const double a = 1.0 + double(i) / steps;
        double worst = 0.0;
        for (double m : mags) {
            worst = std::max(worst, f16_rel_err(a * m));
            if (worst >= best) break;
        }
        if (worst < best) {
            best = worst;
            best_i = i;
        }
    }
    return float(1.0 + double(best_i) / steps);
}

}  // namespace

void build_decode_tables(tq_codec& c, std::vector<uint32_t>& ktab, std::vector<uint32_t>& vtab) {
    ktab.clear();
    vtab.clear();
    c.k_alpha = 1.0f;
    c.v_alpha = 1.0f;
    if (c.bits == 16) return;
    const int L = 1 << c.bits;
    const float alpha = table_alpha(c.centroids, c.bits <= 4 ? (1 << 18) : (1 << 12));
    c.v_alpha = alpha;
    c.k_alpha = c.bits <= 4 ? alpha : 1.0f;
    std::vector<uint16_t> hk(L), lk(L), hv(L);
    for (int i = 0; i < L; ++i) {
        const float x = c.centroids[i];
        hk[i] = f16_bits(c.k_alpha * x);
        lk[i] = f16_bits(x - f16_val(hk[i]));  // used for 8-bit codes only (k_alpha = 1)
        hv[i] = f16_bits(c.v_alpha * x);
    }
    if (c.bits <= 4) {
        for (int p = 0; p < L * L; ++p) {
            const int c0 = p & (L - 1), c1 = p >> c.bits;
            ktab.push_back(uint32_t(hk[c0]) | (uint32_t(hk[c1]) << 16));
            vtab.push_back(uint32_t(hv[c0]) | (uint32_t(hv[c1]) << 16));
        }
    } else {
        for (int i = 0; i < L; ++i) {
            ktab.push_back(uint32_t(hk[i]) | (uint32_t(lk[i]) << 16));
            vtab.push_back(uint32_t(hv[i]) | (uint32_t(hv[i]) << 16));
        }
    }
}


namespace mma_detail {

cudaError_t encode_raw_k_map(CUtensorMap* map, const void* k, int dim, int64_t rows, int box_rows) {
    using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
    static std::atomic<EncodeFn> fn{nullptr};
    EncodeFn f = fn.load();
    if (!f) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        const cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !ptr) return cudaErrorNotSupported;
        f = reinterpret_cast<EncodeFn>(ptr);
        fn.store(f);
    }
    const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(dim), static_cast<cuuint64_t>(rows)};
    const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(dim) * 2};
    const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estride[2] = {1, 1};
    const CUresult r = f(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(k), gdim, gstride, box, estride,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace mma_detail

bool decode_mma_supported(const tq_codec* ck, const tq_codec* cv) {
    if (cv->bits == 16 || ck->dim != cv->dim) return false;
    const int d = cv->dim;
    if (d != 64 && d != 96 && d != 128 && d != 256) return false;
    for (const auto& s : mma_detail::kSchemes)
        if (s[0] == ck->bits && s[1] == cv->bits) return mma_detail::mma_fits(d, ck->bits, cv->bits);
    return false;
}

template <int D>
cudaError_t launch_mma_d_extern(const DecodeArgs& a, DecodePlan& p, int kb, int vb, int nt, cudaStream_t st);
// defined in tq_decode_mma_d{64,96,128,256}.cu
template <>
cudaError_t launch_mma_d_extern<64>(const DecodeArgs&, DecodePlan&, int, int, int, cudaStream_t);
template <>
cudaError_t launch_mma_d_extern<96>(const DecodeArgs&, DecodePlan&, int, int, int, cudaStream_t);
template <>
cudaError_t launch_mma_d_extern<128>(const DecodeArgs&, DecodePlan&, int, int, int, cudaStream_t);
template <>
cudaError_t launch_mma_d_extern<256>(const DecodeArgs&, DecodePlan&, int, int, int, cudaStream_t);
template <int D>
cudaError_t launch_mma_d_stream_extern(const DecodeArgs& a, DecodePlan& p, int kb, int vb, int nt, cudaStream_t st);
// defined in tq_decode_mma_d{64,128,256}_stream.cu
template <>
cudaError_t launch_mma_d_stream_extern<64>(const DecodeArgs&, DecodePlan&, int, int, int, cudaStream_t);
template <>
cudaError_t launch_mma_d_stream_extern<128>(const DecodeArgs&, DecodePlan&, int, int, int, cudaStream_t);
template <>
cudaError_t launch_mma_d_stream_extern<256>(const DecodeArgs&, DecodePlan&, int, int, int, cudaStream_t);

cudaError_t launch_decode_mma(const DecodeArgs& a, DecodePlan& p, cudaStream_t st) {
    // query rows per CTA, min(S, 8): up to 4 (one n-tile, hi/lo columns of q) or 5..8;
    // codes 3 and 4 are the same for the instantiation with several query positions or
    // row groups per unit (causal masks, fp16 hi/lo split of P), 5 and 6 for keys with
    // the QJL sketch (one row group, one query position, 16-byte aligned sketch fields)
    const bool multi = p.L > 1 || p.q_chunks > 1;
    int nt = (p.S > 4 ? 2 : 1) + (multi ? 2 : 0);
    // several query positions with 8-bit keys at d <= 128 and an even number of row groups:
    // two groups per CTA, one dequantised tile feeding both groups' contractions
    int rg = 1;
    if (multi && a.ck.bits == 8 && a.cv.dim <= 128 && (a.cv.dim & (a.cv.dim - 1)) == 0 && p.q_chunks % 2 == 0 &&
        !a.k_signs) {
        nt = 7;
        rg = 2;
    }
    if (a.k_signs) {
        const auto al16 = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; };
        if (multi || !al16(a.k_signs) || !al16(a.k_rnorms)) return cudaErrorNotSupported;  // SIMT
        nt = (p.S > 4 ? 2 : 1) + 4;
    }
    // one CTA per SM: as many splits per (batch, KV head) as fill the SMs once
    const DecodePlan p0 = p;
    int dev = 0;
    cudaGetDevice(&dev);
    const int64_t sms = num_sms(dev);
    const int64_t ctas = int64_t(p.n_units) * (p.q_chunks / rg);  // CTAs per split
    int64_t ns = (sms + ctas - 1) / ctas;
    // several row groups per unit (each re-reads the unit's tiles, mostly from L2):
    // keep the grid to one wave
    if (p.q_chunks > 1 && ns * ctas > sms) ns = sms / ctas;
    const int64_t cap = (a.max_seq + 255) / 256;
    if (ns > cap) ns = cap;
    if (ns < 1) ns = 1;
    int64_t chunk = (a.max_seq + ns - 1) / ns;
    chunk = (chunk + 63) / 64 * 64;
    ns = (a.max_seq + chunk - 1) / chunk;
    if (ns <= p0.n_split) {  // the workspace was sized for p0.n_split splits
        p.n_split = static_cast<int>(ns);
        p.chunk = chunk;
    }
    cudaError_t e = cudaErrorNotSupported;
    // Several sequences, one query position: the token-balanced schedule, one CTA per SM
    // over all units' tokens (ragged lengths and unit counts that do not fill whole waves
    // leave no SM idle).  It needs the power-of-two (Walsh-Hadamard) dims and coded keys.
    const int d = a.cv.dim;
    if (a.B > 1 && !multi && !a.k_signs && a.ck.bits != 16 && (d & (d - 1)) == 0 &&
        sms + int64_t(p.n_units) <= p0.n_rec) {
        p.stream = 1;
        p.n_cta = static_cast<int>(sms);
        // the fixed cost of starting a unit (its queries, the segment's merge and record),
        // in tokens of the loop at this head dim
        p.stream_ovh = (d <= 128 ? kStreamOvhD128 * (128 / d) : kStreamOvhD256) & ~7;
        switch (d) {
            case 64: e = launch_mma_d_stream_extern<64>(a, p, a.ck.bits, a.cv.bits, nt, st); break;
            case 128: e = launch_mma_d_stream_extern<128>(a, p, a.ck.bits, a.cv.bits, nt, st); break;
            case 256: e = launch_mma_d_stream_extern<256>(a, p, a.ck.bits, a.cv.bits, nt, st); break;
            default: break;
        }
        if (e != cudaErrorNotSupported) return e;
        p.stream = 0;
        p.n_cta = 0;
        p.stream_ovh = 0;
    }
    switch (a.cv.dim) {
        case 64: e = launch_mma_d_extern<64>(a, p, a.ck.bits, a.cv.bits, nt, st); break;
        case 96: e = launch_mma_d_extern<96>(a, p, a.ck.bits, a.cv.bits, nt, st); break;
        case 128: e = launch_mma_d_extern<128>(a, p, a.ck.bits, a.cv.bits, nt, st); break;
        case 256: e = launch_mma_d_extern<256>(a, p, a.ck.bits, a.cv.bits, nt, st); break;
        default: break;
    }
    if (e == cudaErrorNotSupported) p = p0;  // the caller falls back with its own plan
    return e;
}

}  // namespace tq
