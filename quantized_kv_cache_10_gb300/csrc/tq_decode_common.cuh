// tq_decode_common.cuh -- pieces shared by the decode-attention kernels:
// workspace layout, query rotation and the split-K partial records that the
// combine kernel (tq_decode_combine.cu) merges before the single inverse
// rotation.
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

// Partial record at slot `slot` of the token-balanced schedule (CTA c, unit u: slot c + u).
__device__ __forceinline__ float* partial_slot_ptr(void* ws, const DecodePlan& p, int64_t slot, int d) {
    float* base = reinterpret_cast<float*>(static_cast<char*>(ws) + p.part_offset);
    return base + slot * (kGP * (d + 2));
}

__device__ __forceinline__ int32_t* error_ptr(void* ws) { return static_cast<int32_t*>(ws); }

// Token-balanced schedule (several sequences, one query position, tensor-core kernel)
// The units' tokens are laid end to end in unit order (u = b * Hkv + h), unit u
// spanning ovh positions that hold no token and then len_b rounded up to a
// multiple of 8 (an empty sequence spans nothing), and CTA c takes positions
// [c W, (c + 1) W), W = the total over the CTAs rounded up to 8 (at least kStreamMinW).
// The positions without tokens stand for the fixed cost of starting a unit (its queries,
// a partial record), so a CTA that starts more units gets fewer tokens (ovh, a multiple
// of 8, is the plan's: that cost is a time, so its size in tokens follows the loop's
// rate).  Every boundary
// is a multiple of 8, so each segment of a unit starts on an 8-token boundary (16-byte
// aligned copies) and holds at least one real token.  Every warp that needs the
// segments walks them itself (warp-collective, same result in each).
constexpr int64_t kStreamMinW = 256;

// Positions of one unit of a sequence of len tokens (ovh: the positions without tokens
// at a unit's start, the plan's stream_ovh).
__device__ __forceinline__ int64_t stream_unit_ext(int64_t ovh, int64_t len) {
    return len > 0 ? ovh + ((len + 7) & ~int64_t(7)) : 0;
}

__device__ __forceinline__ int64_t stream_len(const DecodeArgs& a, int b, bool flag) {
    int64_t L = __ldg(a.seq_lens + b);
    if (L < 0 || L > a.max_seq) {
        if (flag) atomicOr(error_ptr(a.ws), TQ_DEVERR_SEQ_LEN);
        L = L < 0 ? 0 : a.max_seq;
    }
    return L;
}

// Total positions (all units) and the positions per CTA, W (warp-collective).
__device__ __forceinline__ void stream_extent(const DecodeArgs& a, int n_cta, int64_t ovh, int lane, bool flag,
                                              int64_t& tot, int64_t& W) {
    tot = 0;
    for (int b0 = 0; b0 < a.B; b0 += 32) {
        const int bb = b0 + lane;
        int64_t sp = bb < a.B ? stream_unit_ext(ovh, stream_len(a, bb, flag)) : 0;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sp += __shfl_xor_sync(kFullMask, sp, o);
        tot += sp;
    }
    tot *= a.Hkv;
    W = (tot + n_cta - 1) / n_cta;
    W = max((W + 7) & ~int64_t(7), kStreamMinW);
}

// The CTAs whose positions cover unit (b, h): the first and their count (0 when the
// sequence is empty) -- its records are slots first + u .. first + u + count - 1
// (warp-collective).
__device__ __forceinline__ void stream_unit_ctas(const DecodeArgs& a, int n_cta, int64_t ovh, int b, int h,
                                                 int lane, int64_t& first, int& count) {
    int64_t tot, W;
    stream_extent(a, n_cta, ovh, lane, false, tot, W);
    // positions before sequence b: its units start there
    int64_t before = 0;
    for (int b0 = 0; b0 < b; b0 += 32) {
        const int bb = b0 + lane;
        int64_t sp = bb < b ? stream_unit_ext(ovh, stream_len(a, bb, false)) : 0;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sp += __shfl_xor_sync(kFullMask, sp, o);
        before += sp;
    }
    const int64_t ext = stream_unit_ext(ovh, stream_len(a, b, false));
    const int64_t us = before * a.Hkv + static_cast<int64_t>(h) * ext;  // the unit's first position
    first = (us + ovh) / W;                                             // ... holding a token
    count = ext > 0 ? static_cast<int>((us + ext - 1) / W - first + 1) : 0;
}

struct StreamWalk {
    int b, h;          // current unit: sequence b, KV head h
    int64_t len;       // len_b (clamped)
    int64_t ext;       // positions of the unit (ovh + len_b rounded up to 8)
    int64_t us;        // first position of the unit (its tokens start at us + ovh)
    int64_t ovh;       // positions without tokens at a unit's start
    int64_t a0;        // first token of this CTA's segment in the unit
    int64_t end;       // the CTA's positions end here
    int64_t W;         // positions per CTA
    bool valid;        // a segment is current

    // Segment [a0, a1) of unit (b, h), a1 <= len.
    __device__ __forceinline__ int64_t a1() const { return min(len, end - (us + ovh)); }

    // Walk start for CTA c of n_cta (lengths flagged by warp 0's lanes only).
    __device__ __forceinline__ void init(const DecodeArgs& a, int c, int n_cta, int64_t ovh_, int lane, bool flag) {
        int64_t tot;
        ovh = ovh_;
        stream_extent(a, n_cta, ovh, lane, flag, tot, W);
        const int64_t P = static_cast<int64_t>(c) * W;
        valid = P < tot;
        end = min(P + W, tot);
        b = 0;
        h = 0;
        len = ext = us = a0 = 0;
        if (!valid) return;
        // the sequence whose units hold position P
        int64_t base = 0;
        for (int b0 = 0; b0 < a.B; b0 += 32) {
            const int bb = b0 + lane;
            const int64_t L = bb < a.B ? stream_len(a, bb, false) : 0;
            const int64_t sp = stream_unit_ext(ovh, L) * a.Hkv;
            int64_t inc = sp;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int64_t y = __shfl_up_sync(kFullMask, inc, o);
                if (lane >= o) inc += y;
            }
            const unsigned hit = __ballot_sync(kFullMask, bb < a.B && base + inc > P);
            if (hit) {
                const int l = __ffs(hit) - 1;
                b = b0 + l;
                const int64_t sb = base + __shfl_sync(kFullMask, inc - sp, l);
                len = __shfl_sync(kFullMask, L, l);
                ext = stream_unit_ext(ovh, len);
                h = static_cast<int>((P - sb) / ext);
                us = sb + static_cast<int64_t>(h) * ext;
                const int64_t r0 = us + ovh;  // the unit's first token
                a0 = P > r0 ? P - r0 : 0;
                valid = end > r0;  // else the CTA's positions end before any token
                return;
            }
            base += __shfl_sync(kFullMask, inc, 31);
        }
        valid = false;  // not reached: P < tot
    }

    // Next segment (the next unit with tokens), if the CTA's positions reach its tokens.
    __device__ __forceinline__ void next(const DecodeArgs& a) {
        const int64_t ue = us + ext;
        if (end <= ue) {
            valid = false;
            return;
        }
        us = ue;
        a0 = 0;
        if (++h == a.Hkv) {
            h = 0;
            do {
                ++b;
                len = b < a.B ? stream_len(a, b, false) : 0;
            } while (len == 0 && b < a.B);
            ext = stream_unit_ext(ovh, len);
            if (b >= a.B) {  // not reached: end <= total
                valid = false;
                return;
            }
        }
        valid = end > us + ovh;
    }
};

// Clamped sequence length of batch b (flags out-of-range values).
__device__ __forceinline__ int64_t clamped_len(const DecodeArgs& a, int b) {
    int64_t L = __ldg(a.seq_lens + b);
    if (L < 0 || L > a.max_seq) {
        if (threadIdx.x == 0) atomicOr(error_ptr(a.ws), TQ_DEVERR_SEQ_LEN);
        L = L < 0 ? 0 : a.max_seq;
    }
    return L;
}

// Unencoded tail tokens of sequence b: tail_lens[b] (clamped to [0, max_tail],
// out-of-range values flagged), else tail_n for every sequence, else 0.  The
// new token of the cache manager is not counted.
__device__ __forceinline__ int tail_count(const DecodeArgs& a, int b) {
    if (a.tail_lens) {
        int nt = __ldcg(a.tail_lens + b);
        if (nt < 0 || nt > a.max_tail) {
            if (threadIdx.x == 0) atomicOr(error_ptr(a.ws), TQ_DEVERR_SEQ_LEN);
            nt = nt < 0 ? 0 : a.max_tail;
        }
        return nt;
    }
    return (a.k_tail && a.tail_n > 0) ? a.tail_n : 0;
}

// Causal visibility for query position ell of L: the queries are the last L of
// the sequence's len + tail tokens (packed first, then tail), and each attends
// to the tokens up to its own position.  Packed tokens visible: all of them
// unless the query sits before the end of the packed part.
__device__ __forceinline__ int64_t packed_visible(int64_t len, int tail, int L, int ell) {
    const int64_t hidden = static_cast<int64_t>(L - 1 - ell) - tail;  // packed tokens after the query
    return hidden > 0 ? (len > hidden ? len - hidden : 0) : len;
}
// ... and tail tokens visible to it.
__device__ __forceinline__ int tail_visible(int tail, int L, int ell) {
    const int v = tail - (L - 1 - ell);
    return v > 0 ? v : 0;
}

// q' for query row `row` of q ([B, Hq, L, d] as rows of d) into dst[0..d): the K
// rotation applied to q, scaled by log2(e) * scale / sqrt(d) (raw K:
// q * log2(e) * scale, no rotation).  Executed by one full warp.
__device__ inline void rotate_query_warp(const DecodeArgs& a, int64_t row, float* dst) {
    const int lane = threadIdx.x & 31;
    const int d = a.cv.dim;
    const uint16_t* q = a.q + row * d;
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

// Phase timeline of the decode and combine kernels, for profiling builds only
// (compiled with -DTQ_TIMELINE into libtq_timeline.so; the library built by
// default contains none of it).  Buffer of 64-bit words: two halves (the calls
// of even / odd index since the buffer was registered) of kTlSlots decode-CTA
// records and kTlSlots combine-CTA records of kTlStamps globaltimer stamps (ns).
#ifdef TQ_TIMELINE
constexpr int kTlSlots = kTlSlotsHost, kTlStamps = kTlStampsHost;
#define TQ_TL(arr, i) \
    if (threadIdx.x == 0) (arr)[i] = tl_now()
__device__ __forceinline__ unsigned long long tl_now() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ unsigned long long* tl_record(const DecodeArgs& a, bool combine, int slot) {
    if (slot >= kTlSlots) return nullptr;
    return a.tl + (a.tl_seq & 1u) * (2ull * kTlSlots * kTlStamps) + ((combine ? kTlSlots : 0) + slot) * kTlStamps;
}
#else
#define TQ_TL(arr, i)
#endif

// Lets the kernel that follows on the stream (launched with programmatic
// stream serialization) be scheduled while this grid still runs.  A CTA counts
// as triggered at the first execution by any of its threads, and the combine
// kernel reads the call's inputs before its own dependency wait, so a decode
// kernel executes this only in threads that have passed griddepcontrol.wait
// (or, launched without programmatic serialization, anywhere: everything
// before it on the stream has then completed before it starts).
__device__ __forceinline__ void allow_dependent_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Writes this CTA's split-K partial: so[kGP][d] (unnormalised, relative to the
// CTA's max), sm[kGP] (max, log2 units), sl[kGP] (sum of weights).  Every CTA
// writes its record, also when its split is empty (sm = -inf), so the combine
// reads n_split complete records.  Must be called by `nth` threads tid < nth.
__device__ inline void write_partial(const DecodeArgs& a, const DecodePlan& p, int vu, int split, const float* so,
                                     const float* sm, const float* sl, int tid, int nth) {
    const int d = a.cv.dim;
    float* part = partial_ptr(a.ws, p, vu, split, d);
    // d is a multiple of 32 and records are 16-byte aligned: float4 copies
    const float4* s4 = reinterpret_cast<const float4*>(so);
    float4* p4 = reinterpret_cast<float4*>(part);
    for (int i = tid; i < kGP * d / 4; i += nth) p4[i] = s4[i];
    for (int g = tid; g < kGP; g += nth) {
        part[kGP * d + g] = sm[g];
        part[kGP * d + kGP + g] = sl[g];
    }
}

}  // namespace tq
