// tq_decode_mma.cuh -- the tensor-core fused decode-attention kernel template
// (instantiated per head dim in tq_decode_mma_d*.cu).
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
// applies the single inverse V rotation.  Every wait is bounded: a wait that
// gives up records TQ_DEVERR_TIMEOUT and the CTA drains its copies and exits.
//
// Register/shared layouts (thread = 4*g + t in its warp):
//   K role (A of the score mma, rows = tokens): thread t owns dims
//     [(D/4) t, (D/4)(t+1)); k-tile kt uses dims (D/4) t + 4 kt + {0,1,2,3}
//     for the k columns {2t, 2t+1, 2t+8, 2t+9}.  The q' B fragment uses the
//     same map.
//   V role (A of the P.V mma, rows = dims): thread g owns dims
//     [(D/8) g, (D/8)(g+1)); m-tile dm rows g / g+8 are dims (D/8) g + 2 dm + 0/1.
//   Query columns: NT == 2 (5..8 heads): column j of n-tile 0 / 1 = q_hi / q_lo
//     of head j (8-bit K: n-tile 0 only); NT == 1 (<= 4 heads): column 2j / 2j+1
//     = q_hi / q_lo of head j, and in P.V head j sits in column 2j.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>

#include <atomic>

#include "tq_decode_common.cuh"

namespace tq {
namespace mma_detail {
// ---------------------------------------------------------------------------
// PTX helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait (about a second of SM clock); false on timeout.
constexpr long long kWaitCycles = 2000000000LL;
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > kWaitCycles) return false;
    return true;
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// 2-D tensor copy (TMA) of one box at column x, row y of the tensor map into shared memory.
__device__ __forceinline__ void tma_g2s_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

// L2 prefetch of a byte range (16-byte aligned, size a multiple of 16); a hint
// with no effect on what any load returns.
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void prefetch_l2_2d(const CUtensorMap* map, int x, int y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y)
                 : "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// fp16 (hi, lo) split of two fp32 values: hi = fp16(x), lo = fp16(x - hi), so hi + lo
// carries x to ~2^-22 relative (packed pairs: a in the low half).
__device__ __forceinline__ void split_f16x2(float a, float b, uint32_t& hi, uint32_t& lo) {
    const __half2 h = __floats2half2_rn(a, b);
    const float2 f = __half22float2(h);
    const __half2 l = __floats2half2_rn(a - f.x, b - f.y);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = *reinterpret_cast<const uint32_t*>(&l);
}

// 2^x by the hardware's approximate base-2 exponential (PTX ex2.approx.ftz: relative
// error ~2^-22, subnormal results flushed to zero, 2^-inf = 0).  The softmax weights it
// forms are rounded to fp16 for the P.V contraction, and the flushed ones are below
// 2^-126 of the running maximum.
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ void lds64(uint32_t addr, uint32_t& a, uint32_t& b) {
    asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(a), "=r"(b) : "r"(addr));
}

__device__ __forceinline__ void sts32(uint32_t addr, uint32_t a) {
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(a) : "memory");
}

__device__ __forceinline__ void sts64(uint32_t addr, uint32_t a, uint32_t b) {
    asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(addr), "r"(a), "r"(b) : "memory");
}

// 32 bits of the little-endian word array w starting at bit s (compile-time s).
template <int NW>
__device__ __forceinline__ uint32_t bits_at(const uint32_t (&w)[NW], int s) {
    const int i = s >> 5, sh = s & 31;
    const uint32_t lo = (i < NW) ? w[i] : 0u;
    const uint32_t hi = (i + 1 < NW) ? w[i + 1] : 0u;
    return sh ? __funnelshift_r(lo, hi, sh) : lo;
}

// 32 bits of w starting at bit s, where s may be negative (low bits then zero).
template <int NW>
__device__ __forceinline__ uint32_t bits_from(const uint32_t (&w)[NW], int s) {
    return (s >= 0) ? bits_at<NW>(w, s) : (w[0] << (-s));
}

// ((field of `width` bits at bit s) << dst) | lane_off, in two instructions.
template <int NW>
__device__ __forceinline__ uint32_t field_addr(const uint32_t (&w)[NW], int s, int width, int dst, uint32_t lane_off) {
    const uint32_t m = ((1u << width) - 1u) << dst;
    return (bits_from<NW>(w, s - dst) & m) | lane_off;
}

// ---------------------------------------------------------------------------
// Configuration
// ---------------------------------------------------------------------------
constexpr int kSmemLimit = 227 * 1024;

constexpr int al16(int x) { return (x + 15) / 16 * 16; }
constexpr int al128(int x) { return (x + 127) / 128 * 128; }
constexpr int al1024(int x) { return (x + 1023) / 1024 * 1024; }

// Consumer warps per CTA (+ one TMA producer warp), measured per kind:
//   raw fp16 K: 4, whose stages are 4x larger per token, so that four stages
//     of 64 tokens fit;
//   8-bit K, d <= 128: 8 with two m-tiles per warp per stage (more independent
//     work per warp beats more warps here: 18.7 vs 19.9 us on the 32K workload);
//   other coded K: 11 with one m-tile, three warps per SM sub-partition at the
//     168-register budget.
constexpr int nwc_for(int D, int KB) { return KB == 16 ? 4 : (KB == 8 && D <= 128) ? 8 : 11; }

// Bytes of one stage of ts tokens: K codes (raw K: D/64 swizzled column blocks
// of ts rows x 128 B, each 1024-byte aligned), V codes, K norms, V norms, and
// for keys with the QJL sketch their sign bits and residual norms.
constexpr int stage_bytes(int D, int KB, int VB, int ts, bool qjl = false) {
    return KB == 16 ? al1024((D / 64) * al1024(ts * 128) + al128(ts * D * VB / 8 + 16) + 2 * al128(ts * 2))
                    : al128(ts * D * KB / 8 + 16) + al128(ts * D * VB / 8 + 16) + 2 * al128(ts * 2) +
                          (qjl ? al128(ts * D / 8) + al128(ts * 2) : 0);
}

// Shared-memory layout of one (D, K bits, V bits) instantiation; the same
// function serves the kernel (constexpr) and the host's support test.
struct Layout {
    int nwc, krows, vrows, ktab, vtab, kw, vw, pro, bqb, ubq, fixed, mt, ts, stage, nstage, smem;
    // 8-bit K and pairs of 4-bit K ("table block"): both lookup tables share one
    // 64 KB block at the fixed shared address kTBlock -- K in the first 128 B of
    // each 256-B row, V in the second -- so that a byte permute forms a whole K
    // address and one mask-or a whole V address.  The small regions and `g` stages sit below
    // the block, the other `na` stages above it.
    bool tblock;
    int small, g, na;
    // 2-4 bit K ("based" tables): the K and V pair tables (128-B rows) at the same fixed
    // address kTBlock, the larger first and the other at kTBlock + its size, so that each
    // table's base bits ride in the lane offset and an address is a mask-or (no add).
    // Small regions and `g` stages below, `na` stages above kTBlock + tt.
    bool based;
    int kbase, vbase, tt;
};

// Shared address where the dynamic shared memory starts on this GPU (the
// first 1 KB of a CTA's window is reserved by the system); the table-block
// layout is sized for it and every kernel checks it at run time.
constexpr int kSmemBase = 1024;
constexpr int kTBlock = 65536;

constexpr Layout make_layout(int D, int KB, int VB, bool qjl = false, bool multi = false, int rg = 1);

constexpr Layout make_tblock_layout(int D, int KB, int VB, int mt, bool multi, int rg = 1) {
    Layout L{};
    L.tblock = true;
    L.based = false;
    L.nwc = nwc_for(D, KB);
    L.krows = 256;
    L.vrows = (VB <= 4) ? (1 << (2 * VB)) : 256;
    L.ktab = 0;
    L.vtab = 0;
    L.kw = L.krows;
    L.vw = L.vrows;
    L.pro = al128(L.kw * 4) + al128(L.vw * 4) + al128(kGP * D * 2) + 128;
    // q' B fragments in shared memory: D > 128, or several query positions (q_hi and q_lo
    // n-tiles, which registers would not hold beside the rest)
    L.bqb = (D > 128 || multi) ? (D / 8) * 2 * 256 * rg : 0;
    L.small = kGP * D * 4 * rg + 1024 + L.pro + L.bqb;
    L.fixed = L.small;
    L.mt = mt;
    L.ts = L.nwc * 16 * mt;
    L.stage = stage_bytes(D, KB, VB, L.ts);
    const int below = kTBlock - kSmemBase - L.small;
    L.g = below > 0 ? below / L.stage : 0;
    L.na = (kSmemBase + kSmemLimit - 2 * kTBlock) / L.stage;
    if (L.g > 4) L.g = 4;
    if (L.g + L.na > 4) L.na = 4 - L.g;
    // the warp merge uses the stages above the block as one contiguous area
    while (L.na * L.stage < L.nwc * kGP * D * 4 && L.g > 0 && L.na < (kSmemBase + kSmemLimit - 2 * kTBlock) / L.stage) {
        --L.g;
        ++L.na;
    }
    L.nstage = (L.na * L.stage >= L.nwc * kGP * D * 4) ? L.g + L.na : 0;
    L.smem = 2 * kTBlock + L.na * L.stage - kSmemBase;
    return L;
}

constexpr Layout make_based_layout(const Layout& lin, int D, int KB, int VB, bool qjl, int mt, int rg) {
    Layout L = lin;
    L.based = true;
    L.tblock = false;
    // the larger table first: the other's base (the larger's size, a power of two) and
    // its offsets (below its own, smaller, size) never share a bit
    L.kbase = (L.ktab >= L.vtab) ? 0 : L.vtab;
    L.vbase = (L.ktab >= L.vtab) ? L.ktab : 0;
    L.tt = L.ktab + L.vtab;
    L.small = kGP * D * 4 * rg + 1024 + L.pro + L.bqb + L.ubq;
    L.fixed = L.small;
    L.mt = mt;
    L.ts = L.nwc * 16 * mt;
    L.stage = stage_bytes(D, KB, VB, L.ts, qjl);
    const int below = kTBlock - kSmemBase - L.small;
    const int above_max = (kSmemBase + kSmemLimit - kTBlock - L.tt) / L.stage;
    L.g = below > 0 ? below / L.stage : 0;
    L.na = above_max;
    if (L.g > 4) L.g = 4;
    if (L.g + L.na > 4) L.na = 4 - L.g;
    // the warp merge uses the stages above the tables as one contiguous area
    while (L.na * L.stage < L.nwc * kGP * D * 4 && L.g > 0 && L.na < above_max) {
        --L.g;
        ++L.na;
    }
    L.nstage = (L.na * L.stage >= L.nwc * kGP * D * 4) ? L.g + L.na : 0;
    L.smem = kTBlock + L.tt + L.na * L.stage - kSmemBase;
    return L;
}

constexpr Layout make_layout(int D, int KB, int VB, bool qjl, bool multi, int rg) {
    if (KB == 8 || (KB == 4 && !qjl && !multi)) {
        // the table block, when it holds at least as many stages as the linear layout would
        // (4-bit keys: a pair of codes is one byte, so the same byte permute forms the address)
        const Layout t2 = make_tblock_layout(D, KB, VB, 2, multi, rg), t1 = make_tblock_layout(D, KB, VB, 1, multi, rg);
        const Layout t = (D <= 128 && t2.nstage >= 3) ? t2 : t1;
        if (t.nstage >= 3) return t;
    }
    Layout L{};
    L.nwc = nwc_for(D, KB);
    L.krows = (KB == 16) ? 0 : (KB <= 4) ? (1 << (2 * KB)) : 256;
    L.vrows = (VB <= 4) ? (1 << (2 * VB)) : 256;
    // 32 lanes x 4 B: 128-B rows for pair entries, 256-B rows for 8-bit codes
    // (so the code byte becomes the row with one byte permute)
    L.ktab = L.krows * ((KB <= 4) ? 128 : 256);
    L.vtab = L.vrows * 128;   // 32 lanes x 4 B
    // TMA landing area for the prologue: compact K / V tables, the query block, sign words
    L.kw = L.krows;                                              // compact K table words
    L.vw = L.vrows;                                              // compact V table words
    L.pro = al128(L.kw * 4) + al128(L.vw * 4) + al128(kGP * D * 2) + 128;
    // D > 128: the q' B fragments live in shared memory (one copy, 8 B per lane
    // per (k-tile, n-tile)) instead of registers
    // (also with the QJL sketch, whose own fragments and per-row values need the registers)
    // (and for 8-bit K with several query positions: q_hi and q_lo n-tiles)
    L.bqb = (D > 128 || qjl || (multi && KB == 8)) ? ((KB == 8) ? D / 8 : D / 16) * 2 * 256 * rg : 0;
    // keys with the QJL sketch: the B fragments of u = S q' (D / 16 k-tiles, up to two n-tiles)
    L.ubq = qjl ? (D / 16) * 2 * 256 : 0;
    // (+1024 for raw K: the ring is aligned to 1024 B at run time)
    L.fixed = L.ktab + L.vtab + kGP * D * 4 * rg + 1024 + L.pro + L.bqb + L.ubq + (KB == 16 ? 1024 : 0);
    // two m-tiles per warp per stage when three such stages fit (so two are in
    // flight while one is consumed), else one
    L.mt = (KB != 16 && D <= 128 && L.fixed + 3 * stage_bytes(D, KB, VB, L.nwc * 32, qjl) <= kSmemLimit) ? 2 : 1;
    L.ts = L.nwc * 16 * L.mt;
    L.stage = stage_bytes(D, KB, VB, L.ts, qjl);
    const int cap = (KB == 16) ? 6 : 4;
    const int ns = (kSmemLimit - L.fixed) / L.stage;
    L.nstage = ns > cap ? cap : ns;
    L.smem = L.fixed + L.nstage * L.stage;
    L.tblock = false;
    L.based = false;
    L.kbase = L.vbase = L.tt = 0;
    L.small = 0;
    L.g = 0;
    L.na = L.nstage;
    if (KB <= 4) {
        // the based tables when they keep as many stages of the same size
        const Layout b = make_based_layout(L, D, KB, VB, qjl, L.mt, rg);
        if (b.nstage >= L.nstage) return b;
    }
    return L;
}

// Whether an instantiation fits (two stages at least); host and device.
constexpr bool mma_fits(int D, int KB, int VB, bool qjl = false, bool multi = false) {
    return (KB != 16 || D % 64 == 0) && (!qjl || KB <= 4) && make_layout(D, KB, VB, qjl, multi).nstage >= 2;
}
// ... and the instantiation with two row groups per CTA (several query positions, 8-bit K)
constexpr bool mma_fits_rg2(int D, int KB, int VB) {
    return KB == 8 && D <= 128 && make_layout(D, KB, VB, false, true, 2).nstage >= 3;
}

// RG: groups of kGP query rows a CTA serves at once (2: one dequantised tile feeds both
// groups' contractions; the instantiation with several query positions and 8-bit keys)
template <int D, int KB, int VB, int NT, bool QJL = false, bool MULTI = false, int RG = 1>
struct Cfg {
    static constexpr Layout L = make_layout(D, KB, VB, QJL, MULTI, RG);
    static constexpr int NWC = L.nwc;               // consumer warps
    static constexpr int NTHREADS = (NWC + 1) * 32;
    // register budget per thread: 8-bit K at d <= 128 measured fastest at 144 (17.3 vs 18.3 us
    // per call at 168 on the 32K workload; 128: 19.4, 136: 17.6, 152: 18.5, 160: 18.5); others
    // take what three warps per SM sub-partition allow (raw K: two warps)
    // (the instantiation for several query positions, whose 8-bit K scores keep q_lo, takes 168)
    static constexpr int MAXREG = (KB == 16) ? 232 : (KB == 8 && D <= 128 && !MULTI) ? 144 : 168;
    static constexpr int MT = L.mt;                 // m-tiles of 16 tokens per warp per stage
    static constexpr int TS = L.ts;                 // tokens per stage
    static constexpr bool KRAW = (KB == 16);        // raw fp16 K rows (no codebook)
    static constexpr int BPK = D * KB / 8;
    static constexpr int BPV = D * VB / 8;
    static constexpr int KT = D / 16;               // P.V dim m-tiles
    // 8-bit K: each dim contributes two k elements (K_hi, K_lo) against (q, q), so the
    // table word is the mma operand as it stands; other widths pair neighbouring dims.
    static constexpr bool KEXP = (KB == 8);
    static constexpr int KTS = KEXP ? D / 8 : D / 16;  // score k-tiles
    // score n-tiles: 8-bit K with 5..8 query heads scores against q_hi only --
    // (K_hi, K_lo) x q_hi keeps K exact to ~2^-22 and leaves only q's fp16
    // rounding (~2^-12 relative), for 1.5 instead of 2.5 mma per token.  With
    // several query positions the first rows of a chunk see one or a few tokens,
    // where a score's rounding is not averaged over many tokens but moves the
    // output directly: they keep q_lo too.
    static constexpr int NTS = (KEXP && NT == 2 && !MULTI) ? 1 : NT;
    static constexpr int BQB = L.bqb;
    static constexpr bool BQ_SMEM = BQB > 0;
    static constexpr bool KPAIR = KB <= 4;
    static constexpr bool VPAIR = VB <= 4;
    static constexpr int KROWS = L.krows;
    static constexpr int KTAB = L.ktab;
    static constexpr int VROWS = L.vrows;
    static constexpr int VTAB = L.vtab;
    // per-thread chunk of one row, in bits and 32-bit words
    static constexpr int KCB = (D / 4) * (KRAW ? 8 : KB);  // K role: thread t, dims (D/4) t ...
    static constexpr int KCW = (KCB + 31) / 32;
    static constexpr int VCB = (D / 8) * VB;        // V role: thread g, dims (D/8) g ...
    static constexpr int VCW = (VCB + 31) / 32;
    // stage buffers (+16 B slack: chunk loads may read one word past a row)
    static constexpr int KREG = al1024(TS * 128);   // raw K: one swizzled 64-column block
    static constexpr int KBUF = KRAW ? (D / 64) * KREG : al128(TS * BPK + 16);
    static constexpr int VBUF = al128(TS * BPV + 16);
    static constexpr int NBUF = al128(TS * 2);
    // keys with the QJL sketch: sign bits (D / 8 bytes per token) and residual norms
    static constexpr int SBUF = QJL ? al128(TS * D / 8) : 0;
    static constexpr int RBUF = QJL ? al128(TS * 2) : 0;
    static constexpr int UBQ = L.ubq;
    static constexpr int STAGE = L.stage;
    static constexpr int QBYTES = kGP * D * 4 * RG;  // q' fp32 of every row group
    static constexpr int RGS = RG;                   // row groups (q' fragment stride)
    static constexpr int KW = L.kw, VW = L.vw;
    static constexpr int PRO = L.pro;
    static constexpr int PRO_K = 0;                              // offsets inside the prologue area
    static constexpr int PRO_V = al128(KW * 4);
    static constexpr int PRO_Q = PRO_V + al128(VW * 4);
    static constexpr int PRO_S = PRO_Q + al128(kGP * D * 2);
    static constexpr int MISC = 1024;               // barriers, m/l exchange
    static constexpr int FIXED = L.fixed;
    static constexpr int NSTAGE = L.nstage;
    static constexpr int SMEM = L.smem;
    static constexpr bool TBLOCK = L.tblock;
    static constexpr bool BASED = L.based;
    static constexpr int KBASE = L.kbase, VBASE = L.vbase, TT = L.tt;
    static constexpr int VMODE = TBLOCK ? 1 : BASED ? 2 : 0;  // V table addressing (v_role)
    // K lookups addressed by one byte permute of the code word: 8-bit codes, or pairs of
    // 4-bit codes (one byte) in the table block
    static constexpr bool KPERM = KEXP || (KB == 4 && TBLOCK);
    static constexpr int SMALL = L.small, G_BELOW = L.g, N_ABOVE = L.na;
    static_assert(STAGE >= KBUF + VBUF + 2 * NBUF + SBUF + RBUF, "stage size");
    static_assert(!QJL || (KB <= 4 && D % 32 == 0), "the QJL sketch rides on 2-4 bit keys");
    static_assert(NSTAGE >= 2 && NSTAGE <= 8, "stage count");
    static_assert(!KRAW || D % 64 == 0, "raw K needs 64-column blocks");
    // epilogue scratch (per-warp O slices, combine weights) lives in the stage ring
    static_assert(N_ABOVE * STAGE >= NWC * kGP * D * 4, "stage ring too small for the warp merge");
};

// ---------------------------------------------------------------------------
// Dequant: K role (pairs of neighbouring dims of one token)
// ---------------------------------------------------------------------------
// For k-tile kt of one token row whose chunk words are w (2-4 bit codes): A
// registers for dims base+0,1 (hi01) and base+2,3 (hi23) from the pair table
// (index = 2*KB bits at bit 4*KB*kt and 4*KB*kt + 2*KB; rows of 128 B).
template <int KB, int KCW>
__device__ __forceinline__ void k_role(const uint32_t (&w)[KCW], int kt, uint32_t tab, uint32_t lane_off,
                                       uint32_t& hi01, uint32_t& hi23) {
    const int s0 = 4 * KB * kt;
    hi01 = lds32(tab + field_addr<KCW>(w, s0, 2 * KB, 7, lane_off));
    hi23 = lds32(tab + field_addr<KCW>(w, s0 + 2 * KB, 2 * KB, 7, lane_off));
}

// ---------------------------------------------------------------------------
// Dequant: V role (one dim of two tokens a, b)
// ---------------------------------------------------------------------------
// MODE: where the V table sits.  0: anywhere (the table address is added), 1: the table
// block (256-B rows), 2: the based tables (128-B rows); in 1 and 2 lane4 already holds
// the table's address bits and the lane offset, so an address is one shift and one or.
template <int VB, int VCW, int MODE>
__device__ __forceinline__ uint32_t v_role(const uint32_t (&wa)[VCW], const uint32_t (&wb)[VCW], int j,
                                           uint32_t tab, uint32_t lane4) {
    const int s = VB * j;
    const uint32_t m = (1u << VB) - 1u;
    constexpr int RS = (MODE == 1) ? 8 : 7;
    const uint32_t t = (MODE == 0) ? tab : 0u;
    if constexpr (VB <= 4) {
        const uint32_t ca = bits_at<VCW>(wa, s) & m;
        const uint32_t cb = bits_at<VCW>(wb, s) & m;
        return lds32(t + (((ca | (cb << VB)) << RS) | lane4));
    } else {
        const uint32_t ca = bits_at<VCW>(wa, s) & m;
        const uint32_t cb = bits_at<VCW>(wb, s) & m;
        const uint32_t va = lds32(t + ((ca << RS) | lane4));
        const uint32_t vb = lds32(t + ((cb << RS) | lane4));
        return __byte_perm(va, vb, 0x7610);
    }
}

// V role for 2-4 bit codes.  Two tokens' chunks of up to 16 dims (a, b as
// 64-bit values) are interleaved once into z_even / z_odd whose field i
// (2*VB bits) is code_a | code_b << VB of dim 2i / 2i+1; each pair is then one
// shift and one mask.
template <int VB, int MODE>
struct VPairs {
    static constexpr uint64_t even_mask() {
        uint64_t m = 0;
        for (int i = 0; i < 16; i += 2) m |= ((1ull << VB) - 1ull) << (i * VB);
        return m;
    }
    uint64_t ze, zo;
    __device__ __forceinline__ VPairs(uint64_t a, uint64_t b) {
        constexpr uint64_t me = even_mask();
        ze = (a & me) | ((b << VB) & ~me);
        zo = ((a >> VB) & me) | (b & ~me);
    }
    // shared-memory address of the pair-table slot for dim j (0..15) of the chunk
    // (MODE 1 / 2: lane4 carrying the table address, so no add; v_role's modes)
    __device__ __forceinline__ uint32_t addr(int j, uint32_t tab, uint32_t lane4) const {
        constexpr int RS = (MODE == 1) ? 8 : 7;
        const uint64_t z = (j & 1) ? zo : ze;
        const int s = VB * (j & ~1);
        const uint32_t x = (s >= RS) ? static_cast<uint32_t>(z >> (s - RS)) : static_cast<uint32_t>(z << (RS - s));
        const uint32_t f = (x & (((1u << (2 * VB)) - 1u) << RS)) | lane4;
        return (MODE != 0) ? f : tab + f;
    }
};

// Bits [bit, bit + 32 NW - (bit & 31)) of a row (4-byte aligned) in the low bits of the
// result: NW words, the fewest that hold the field the caller uses (at most 64 bits).
template <int NW>
__device__ __forceinline__ uint64_t load_bits_w(const uint8_t* row, int bit) {
    static_assert(NW >= 1 && NW <= 3, "words");
    const uint32_t* p = reinterpret_cast<const uint32_t*>(row) + (bit >> 5);
    const int sh = bit & 31;
    const uint32_t w0 = p[0];
    const uint32_t w1 = (NW > 1) ? p[1] : 0u;
    const uint32_t w2 = (NW > 2) ? p[2] : 0u;
    const uint32_t lo = __funnelshift_r(w0, w1, sh);
    const uint32_t hi = __funnelshift_r(w1, w2, sh);
    return (static_cast<uint64_t>(hi) << 32) | lo;
}

// Words a thread's V-role field spans at most: min(16, D/8) dims of VB bits at bit
// g * (D/8) VB + 16 VB sub of the row, over the eight g and the NSUB chunks.
constexpr int v_field_words(int D, int VB) {
    const int nsub = (D / 8 + 15) / 16;
    const int nb = (D / 8 < 16 ? D / 8 : 16) * VB;
    int m = 1;
    for (int g = 0; g < 8; ++g)
        for (int sub = 0; sub < nsub; ++sub) {
            const int sh = (g * (D / 8) * VB + 16 * VB * sub) % 32;
            const int w = (sh + nb + 31) / 32;
            m = w > m ? w : m;
        }
    return m;
}

// Loads NW 32-bit words of a row chunk starting at bit `bit` of the row (row
// 4-byte aligned).  One word past the chunk may be read (stage slack).
template <int NW>
__device__ __forceinline__ void load_chunk(const uint8_t* row, int bit, uint32_t (&w)[NW]) {
    const uint32_t* p = reinterpret_cast<const uint32_t*>(row) + (bit >> 5);
    const int sh = bit & 31;
    if (sh == 0) {
#pragma unroll
        for (int i = 0; i < NW; ++i) w[i] = p[i];
    } else {
        uint32_t prev = p[0];
#pragma unroll
        for (int i = 0; i < NW; ++i) {
            const uint32_t nxt = p[i + 1];
            w[i] = __funnelshift_r(prev, nxt, sh);
            prev = nxt;
        }
    }
}

// K row chunk: thread t's dims of token row `row`.  For 32 B chunks at D=128,
// odd rows load their two 16-byte halves in the opposite order so a quarter
// warp never hits the same banks twice.
template <int D, int KB, int KCW>
__device__ __forceinline__ void load_k_chunk(const uint8_t* kbuf, int row, int t, uint32_t (&w)[KCW]) {
    constexpr int BPK = D * KB / 8;
    constexpr int KCB = (D / 4) * KB;
    if constexpr (KCB % 128 == 0) {
        const uint4* p = reinterpret_cast<const uint4*>(kbuf + row * BPK + t * (KCB / 8));
        constexpr int NV = KCW / 4;
        const int rot = row & 1;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int ii = (i + rot) % NV;
            const uint4 v = p[ii];
            // select by compile-time index to keep w in registers
#pragma unroll
            for (int jj = 0; jj < NV; ++jj)
                if (jj == ii) {
                    w[4 * jj] = v.x;
                    w[4 * jj + 1] = v.y;
                    w[4 * jj + 2] = v.z;
                    w[4 * jj + 3] = v.w;
                }
        }
    } else {
        load_chunk<KCW>(kbuf + row * BPK, t * KCB, w);
    }
}

// ---------------------------------------------------------------------------
// Prologue helpers (consumer threads)
// ---------------------------------------------------------------------------
// Replicates the compact decode tables into one slot per lane: slot s of the
// ROWS * 32 slots is row s / 32, lane s % 32.  A warp writes whole rows (the
// thread count is a multiple of 32), so its loads of the compact entry are
// broadcasts and its stores cover all banks.
template <typename C, int ROWS, int ENTRY_WORDS, int ROW_BYTES>
__device__ __forceinline__ void replicate_one(const uint32_t* src, uint8_t* dst, int ctid) {
    constexpr int NTH = C::NWC * 32;
#pragma unroll 4
    for (int s = ctid; s < ROWS * 32; s += NTH) {
        const int r = s >> 5, l = s & 31;
        if constexpr (ENTRY_WORDS == 2)
            *reinterpret_cast<uint2*>(dst + r * ROW_BYTES + l * 8) = *reinterpret_cast<const uint2*>(src + 2 * r);
        else
            *reinterpret_cast<uint32_t*>(dst + r * ROW_BYTES + l * 4) = src[r];
    }
}

template <typename C>
__device__ __forceinline__ void replicate_tables(const uint32_t* kcompact, const uint32_t* vcompact, uint8_t* ktab_s,
                                                 uint8_t* vtab_s, int ctid) {
    if constexpr (C::KROWS > 0)
        replicate_one<C, C::KROWS, 1, (C::KPAIR && !C::TBLOCK) ? 128 : 256>(kcompact, ktab_s, ctid);
    replicate_one<C, C::VROWS, 1, C::TBLOCK ? 256 : 128>(vcompact, vtab_s, ctid);
}

// q' = R q * log2(e) * scale / sqrt(D) for the G query heads of the unit into
// qs[kGP][D] (rows >= G zero), with every global load in flight at once.
template <int D, int NWC, bool RAW, int ROWS = kGP>
__device__ __forceinline__ void rotate_queries(const DecodeArgs& a, const uint16_t* qg, const uint16_t* qglob,
                                               const uint32_t* signs, int G, float* qs, int warp, int lane, int ctid) {
    constexpr int NTH = NWC * 32;
    if constexpr (RAW) {
        // raw fp16 K is scored in the original basis: q' = q * log2(e) * scale
        const float f = kLog2e * a.scale;
        for (int i = ctid; i < ROWS * D; i += NTH)
            qs[i] = (i < G * D) ? __half2float(__ushort_as_half(qg[i])) * f : 0.0f;
    } else if constexpr ((D & (D - 1)) == 0) {
        // Power-of-two dims always carry the Walsh-Hadamard rotation, the others the dense
        // one.  Warp w rotates query rows w, w + NWC, ... < G in registers, straight from global memory
        // (lane l holds dims [VPL l, VPL (l + 1))): H (s . q) by butterflies of stride < VPL
        // inside the lane and the rest across lanes, natural (Sylvester) order.
        constexpr int VPL = D / 32;
        for (int row = warp; row < G; row += NWC) {
            const uint16_t* src = qglob + row * D + lane * VPL;
            float x[VPL];
            if constexpr (VPL == 8) {
                const uint4 u = *reinterpret_cast<const uint4*>(src);
                const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int v = 0; v < 8; ++v)
                    x[v] = __half2float(__ushort_as_half(static_cast<uint16_t>(w4[v / 2] >> (16 * (v & 1)))));
            } else if constexpr (VPL == 4) {
                const uint2 u = *reinterpret_cast<const uint2*>(src);
                const uint32_t w2[2] = {u.x, u.y};
#pragma unroll
                for (int v = 0; v < 4; ++v)
                    x[v] = __half2float(__ushort_as_half(static_cast<uint16_t>(w2[v / 2] >> (16 * (v & 1)))));
            } else {
#pragma unroll
                for (int v = 0; v < VPL; ++v) x[v] = __half2float(__ushort_as_half(src[v]));
            }
            const uint32_t sw = signs[(lane * VPL) >> 5] >> ((lane * VPL) & 31);
#pragma unroll
            for (int v = 0; v < VPL; ++v)
                if ((sw >> v) & 1u) x[v] = -x[v];
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
            const float f = kLog2e * a.scale / (static_cast<float>(D) * a.ck.k_alpha);
            float* dst = qs + row * D + lane * VPL;
#pragma unroll
            for (int v = 0; v < VPL; ++v) dst[v] = x[v] * f;
        }
        for (int i = G * D + ctid; i < ROWS * D; i += NTH) qs[i] = 0.0f;
    } else {
        // dense: stage q in qs, then each thread forms whole columns j of Q q
        for (int i = ctid; i < kGP * D; i += NTH)
            qs[i] = (i < G * D) ? __half2float(__ushort_as_half(qg[i])) : 0.0f;
        asm volatile("bar.sync 1, %0;" ::"n"(NWC * 32) : "memory");
        // (when D divides the threads twice or more, each column's rows are split between
        // RS threads: each loads the column, then forms kGP / RS of its rows)
        constexpr int RS = (NTH >= 4 * D) ? 4 : (NTH >= 2 * D) ? 2 : 1;
        constexpr int RPT = kGP / RS;             // rows per thread
        constexpr int CPT = (D * RS + NTH - 1) / NTH;  // (column, row slice) items per thread
        float acc[CPT][RPT];
#pragma unroll
        for (int c = 0; c < CPT; ++c) {
            const int item = ctid + NTH * c;
            const int j = item % D, g0 = (item / D) * RPT;
#pragma unroll
            for (int g = 0; g < RPT; ++g) acc[c][g] = 0.0f;
            if (item < D * RS) {
                float col[D];
#pragma unroll
                for (int i = 0; i < D; ++i) col[i] = __ldg(a.ck.qt + static_cast<int64_t>(i) * D + j);
#pragma unroll
                for (int g = 0; g < RPT; ++g)
                    if (g0 + g < G)
#pragma unroll
                        for (int i = 0; i < D; ++i) acc[c][g] = fmaf(col[i], qs[(g0 + g) * D + i], acc[c][g]);
            }
        }
        asm volatile("bar.sync 1, %0;" ::"n"(NWC * 32) : "memory");
        const float f = kLog2e * a.scale * rsqrtf(static_cast<float>(D)) / a.ck.k_alpha;
#pragma unroll
        for (int c = 0; c < CPT; ++c) {
            const int item = ctid + NTH * c;
            const int j = item % D, g0 = (item / D) * RPT;
            if (item < D * RS)
#pragma unroll
                for (int g = 0; g < RPT; ++g) qs[(g0 + g) * D + j] = acc[c][g] * f;
        }
    }
}

// q' B fragments of k-tile kt (n-tiles 0 and, when C::NTS == 2, 1): from
// registers, or from the shared-memory copy when C::BQ_SMEM.
template <typename C, typename BQ>
__device__ __forceinline__ void q_frag(const BQ& Bq, uint32_t bq_a, int kt, int lane, uint32_t& q00, uint32_t& q01,
                                       uint32_t& q10, uint32_t& q11, int rg = 0) {
    if constexpr (C::BQ_SMEM) {
        // (row group rg's fragments follow group 0's within each k-tile)
        const int f0 = (kt * C::RGS + rg) * C::NTS;
        lds64(bq_a + (f0 * 32 + lane) * 8, q00, q01);
        if constexpr (C::NTS == 2) lds64(bq_a + ((f0 + 1) * 32 + lane) * 8, q10, q11);
    } else {
        q00 = Bq[kt][0][0];
        q01 = Bq[kt][0][1];
        if constexpr (C::NTS == 2) {
            q10 = Bq[kt][1][0];
            q11 = Bq[kt][1][1];
        }
    }
}

// float2 slot of (row, dims 2c and 2c + 1) in a warp's merge slice of kGP rows x D/2
// units: row-major, with bits 0-1 of c XOR-ed by a Gray code of the row and, where the
// lane's g does not already vary them, bits 2-3 by bits of c above bit 3.  In the
// epilogue's stores (lane g, t: c = (D/16) g + dm, rows 2t / 2t + 1 or t) the 16 lanes
// of a half-warp then hit 16 distinct 8-byte bank pairs.  Only bits 0-3 of c change and
// the XOR depends on the row and on bits of c above bit 3 only: an involution per row.
template <int D>
__device__ __forceinline__ int merge_slot(int row, int c) {
    const int fold = (D >= 256) ? ((c >> 4) & 3) << 2 : (D >= 128) ? ((c >> 4) & 1) << 2 : 0;
    return row * (D / 2) + (c ^ (((row ^ (row >> 1)) & 3) | fold));
}

// Warp-merge area of the token-balanced schedule: beside the ring when it fits, so that
// the producer keeps filling the ring with the next segment's tiles while the consumers
// merge a segment (rows 4..7 of a warp's slice are zero with up to four query heads and
// are not stored).  0: the merge reuses the ring, and the producer waits for it.
template <int D, int KB, int VB, int NT, bool QJL, bool MULTI, bool STREAM>
constexpr int stream_merge_bytes() {
    using C = Cfg<D, KB, VB, NT, QJL, MULTI>;
    const int bytes = C::NWC * ((NT == 2) ? kGP : 4) * D * 4;
    return (STREAM && C::SMEM + bytes <= kSmemLimit) ? bytes : 0;
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
// (the token-balanced schedule's walk state does not fit the 144-register budget of the
// 8-bit-key decode: those instantiations take 168, one CTA of 9 warps per SM either way)
template <int D, int KB, int VB, int NT, bool MULTI, bool QJL, bool STREAM, int RG>
__global__ void __maxnreg__(((STREAM && KB == 8) ? 168 : Cfg<D, KB, VB, NT, QJL, MULTI, RG>::MAXREG))
    decode_mma_kernel(const DecodeArgs a, const DecodePlan p, const __grid_constant__ CUtensorMap kmap) {
    using C = Cfg<D, KB, VB, NT, QJL, MULTI, RG>;
    // two row groups per CTA: several query positions, 8-bit keys (their byte-permute
    // lookups and q' fragments in shared memory), one schedule per unit
    static_assert(RG == 1 || (RG == 2 && MULTI && C::KEXP && C::BQ_SMEM && !STREAM && !QJL &&
                              (D & (D - 1)) == 0), "row groups");
    // q is staged in shared memory by the producer for raw K and the dense rotation; with
    // the Walsh-Hadamard rotation each consumer warp reads its query row itself
    constexpr bool Q_STAGED = C::KRAW || (D & (D - 1)) != 0;
    // the token-balanced schedule (STREAM) serves one query position, one row group, coded
    // keys without the sketch and the Walsh-Hadamard rotation
    static_assert(!STREAM || (!MULTI && !QJL && !Q_STAGED), "token-balanced schedule");
    constexpr bool SEP = stream_merge_bytes<D, KB, VB, NT, QJL, MULTI, STREAM>() > 0;
    constexpr int SROWS = (SEP && NT == 1) ? 4 : kGP;  // rows of a warp's merge slice
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sbase = smem_addr(smem);
    // table block (8-bit K): the tables at shared address kTBlock, the rest around them
    // (based tables: at kTBlock + KBASE / VBASE)
    uint8_t* ktab_s = C::TBLOCK  ? smem + (static_cast<uint32_t>(kTBlock) - sbase)
                      : C::BASED ? smem + (static_cast<uint32_t>(kTBlock + C::KBASE) - sbase)
                                 : smem;
    uint8_t* vtab_s = C::TBLOCK  ? ktab_s + 128
                      : C::BASED ? smem + (static_cast<uint32_t>(kTBlock + C::VBASE) - sbase)
                                 : ktab_s + C::KTAB;
    float* qs = reinterpret_cast<float*>((C::TBLOCK || C::BASED) ? smem : vtab_s + C::VTAB);  // [kGP][D]
    uint8_t* misc = reinterpret_cast<uint8_t*>(qs) + C::QBYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(misc);                  // [NSTAGE <= 8]
    uint64_t* empty = full + 8;                                          // [NSTAGE <= 8]
    uint64_t* setup = full + 16;                                         // codec tables, sign words
    uint64_t* setup_q = full + 17;                                       // the query block
    int* s_erel = reinterpret_cast<int*>(misc + 160);                    // [kGP] causal ends
    int* s_erel1 = reinterpret_cast<int*>(misc + 976);                   // [kGP] the second row group's
    float* wm = reinterpret_cast<float*>(misc + 256);                    // [C::NWC][kGP]
    float* wl = wm + C::NWC * kGP;                                         // [C::NWC][kGP]
    int* s_abort = reinterpret_cast<int*>(wl + C::NWC * kGP);
    static_assert(256 + 2 * C::NWC * kGP * 4 + 4 <= 976, "misc area: the second group's causal ends");
    uint8_t* pro = misc + C::MISC;                                       // prologue landing area
    uint8_t* bq_s = pro + C::PRO;                                    // q' fragments (D > 128)
    uint8_t* ubq_s = bq_s + C::BQB;                                      // u = S q' fragments (QJL)
    uint8_t* below = ubq_s + C::UBQ;                                     // stages 0 .. G_BELOW-1
    if constexpr (C::KRAW)  // the swizzled K blocks need 1024-byte aligned shared addresses
        below += (1024u - (smem_addr(below) & 1023u)) & 1023u;
    // stages G_BELOW .. NSTAGE-1, contiguous (also the warp-merge area)
    constexpr uint32_t kAbove = C::TBLOCK ? 2u * kTBlock : static_cast<uint32_t>(kTBlock + C::TT);
    uint8_t* ring = (C::TBLOCK || C::BASED) ? smem + (kAbove - sbase) : below;
    auto stage_ptr = [&](int s) -> uint8_t* {
        return ((C::TBLOCK || C::BASED) && s < C::G_BELOW) ? below + s * C::STAGE
                                                             : ring + (s - C::G_BELOW) * C::STAGE;
    };
    if constexpr (C::TBLOCK || C::BASED) {
        // the layout was sized for the dynamic shared memory starting at kSmemBase
        if (sbase + C::SMALL + C::G_BELOW * C::STAGE > static_cast<uint32_t>(kTBlock) ||
            kAbove + C::N_ABOVE * C::STAGE > sbase + C::SMEM) {
            if (threadIdx.x == 0) atomicOr(error_ptr(a.ws), TQ_DEVERR_LAYOUT);
            return;
        }
    }

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
#ifdef TQ_TIMELINE
    // stamps of consumer thread 0 (in spare bytes of the barrier area, not registers):
    // entry, [the SM id], dependency wait passed, first tile consumed, own loop done, all
    // warps' loops done, partial written, query ready
    // (misc: barriers at 0..143, causal ends at 160..191, free 192..255, warp maxima from 256)
    unsigned long long* tl_t = reinterpret_cast<unsigned long long*>(misc + 192);
    static_assert(kTlStamps * 8 <= 64, "timeline stamps");
#endif
    TQ_TL(tl_t, 0);
    // blockIdx.y: (unit, group of <= kGP query rows); the unit's rows are its G query
    // heads times L query positions, head-major, contiguous in q and out
    // (the MULTI instantiation serves several query positions or more than kGP rows per
    // unit; the other one is the decode case: one CTA per unit along y, rows = heads)
    // (the token-balanced schedule sets u, b, kvh, qrow0, row0 and t0 per segment)
    // (with RG row groups a CTA serves chunks c0 .. c0 + RG - 1 of its unit: records vu + rg)
    const int split = blockIdx.x;
    int u = MULTI ? static_cast<int>(blockIdx.y) / (p.q_chunks / RG) : static_cast<int>(blockIdx.y);
    int vu = MULTI ? u * p.q_chunks + (static_cast<int>(blockIdx.y) - u * (p.q_chunks / RG)) * RG
                   : static_cast<int>(blockIdx.y);
    const int s0 = MULTI ? (vu - u * p.q_chunks) * kGP : 0;
    int b = u / a.Hkv, kvh = u - (u / a.Hkv) * a.Hkv;
    const int G = MULTI ? min(kGP, p.S - s0) : p.G;  // query rows of this CTA (its first group)
    const int G1 = (RG == 2) ? min(kGP, p.S - s0 - kGP) : 0;  // the second group's rows
    int64_t qrow0 = MULTI ? (static_cast<int64_t>(b) * a.Hq + static_cast<int64_t>(kvh) * p.G) * p.L + s0
                          : static_cast<int64_t>(b) * a.Hq + kvh * G;
    int64_t row0 = static_cast<int64_t>(u) * a.max_seq;
    int64_t t0 = STREAM ? 0 : static_cast<int64_t>(split) * p.chunk;
    // This kernel is launched with programmatic stream serialization: it may
    // start while the previous kernel on the stream (e.g. the combine of the
    // previous call, which reads this workspace) still runs.  Until
    // griddepcontrol.wait it touches only the codec's tables and sign words,
    // which no kernel writes; q, the cache, the lengths and the workspace come
    // after the wait.
    //
    // The dependent combine launch counts a CTA as triggered at the first
    // griddepcontrol.launch_dependents any of its threads executes, so no
    // thread executes it before it has itself passed griddepcontrol.wait: the
    // combine reads the call's inputs (q, the tail, the new token) and writes
    // the tail buffer before its own wait, which is only safe once everything
    // stream-ordered before this kernel has completed.
    int64_t t1 = t0;
    int ntiles = 0;

    if (tid == 0) {
        for (int s = 0; s < C::NSTAGE; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, C::NWC);
        }
        mbar_init(setup, 1);
        mbar_init(setup_q, 1);
        *s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    int issued = 0;  // tiles whose copies the producer has started (producer lane 0)
    // tiles the producer issues before it reads the length: a ring-full, within max_seq
    auto pre_tiles = [](int64_t t0_, int64_t chunk, int64_t max_seq) -> int {
        const int64_t e = min(t0_ + chunk, max_seq);
        const int64_t n = e > t0_ ? (e - t0_ + C::TS - 1) / C::TS : 0;
        return static_cast<int>(min(n, static_cast<int64_t>(C::NSTAGE)));
    };
    if (warp == C::NWC) {
        // ------------------------------------------------------------ producer
        // (lanes 1-31 issue nothing and never trigger the dependent launch: the
        // CTA's trigger must follow a dependency wait)
        const uint8_t* kg = static_cast<const uint8_t*>(a.k);
        // Tile li of the token range [t0, tend): its copies into stage gi % NSTAGE.
        // (gi: the tile's place in the ring sequence, li: its place in the token range)
        auto issue = [&](int gi, int li, int64_t tend) {
            const int s = gi % C::NSTAGE;
            const int64_t ts = t0 + static_cast<int64_t>(li) * C::TS;
            const int64_t nv = min(static_cast<int64_t>(C::TS), tend - ts);
            const uint32_t n8 = static_cast<uint32_t>((nv + 7) & ~int64_t(7));
            uint8_t* st = stage_ptr(s);
            const uint32_t vbytes = n8 * C::BPV, nbytes = n8 * 2;
            if constexpr (C::KRAW) {
                // whole boxes of TS rows per 64-column block (rows past the tensor read as zero)
                mbar_arrive_expect_tx(full + s, (D / 64) * C::TS * 128 + vbytes + nbytes);
#pragma unroll
                for (int cb = 0; cb < D / 64; ++cb)
                    tma_g2s_2d(st + cb * C::KREG, &kmap, 64 * cb, static_cast<int>(row0 + ts), full + s);
            } else {
                const uint32_t kbytes = n8 * C::BPK;
                const uint32_t sgbytes = QJL ? n8 * (D / 8) : 0u;
                mbar_arrive_expect_tx(full + s, kbytes + vbytes + 2 * nbytes + (QJL ? sgbytes + nbytes : 0u));
                bulk_g2s(st, kg + (row0 + ts) * C::BPK, kbytes, full + s);
                bulk_g2s(st + C::KBUF + C::VBUF, a.k_norms + row0 + ts, nbytes, full + s);
                if constexpr (QJL) {
                    bulk_g2s(st + C::KBUF + C::VBUF + 2 * C::NBUF, a.k_signs + (row0 + ts) * (D / 8), sgbytes,
                             full + s);
                    bulk_g2s(st + C::KBUF + C::VBUF + 2 * C::NBUF + C::SBUF, a.k_rnorms + row0 + ts, nbytes,
                             full + s);
                }
            }
            bulk_g2s(st + C::KBUF, a.v_codes + (row0 + ts) * C::BPV, vbytes, full + s);
            bulk_g2s(st + C::KBUF + C::VBUF + C::NBUF, a.v_norms + row0 + ts, nbytes, full + s);
        };
        if (lane == 0) {
            // prologue data first: compact tables, this unit's query block, sign words
            const uint32_t qbytes = static_cast<uint32_t>((G + G1) * D * 2);
            // sign words: K codec's at PRO_S, V codec's at PRO_S + 64 (<= 64 B each, D <= 512)
            const uint32_t sbytes = (a.ck.is_wht && !C::KRAW) ? 16u * ((D / 32 * 4 + 15) / 16) : 0u;
            const uint32_t vsbytes = a.cv.is_wht ? 16u * ((D / 32 * 4 + 15) / 16) : 0u;
            mbar_arrive_expect_tx(setup, C::KW * 4 + C::VW * 4 + sbytes + vsbytes);
            if constexpr (C::KW > 0) bulk_g2s(pro + C::PRO_K, a.ck.ktab, C::KW * 4, setup);
            bulk_g2s(pro + C::PRO_V, a.cv.vtab, C::VW * 4, setup);
            if (sbytes) bulk_g2s(pro + C::PRO_S, a.ck.sign_bits, sbytes, setup);
            if (vsbytes) bulk_g2s(pro + C::PRO_S + 64, a.cv.sign_bits, vsbytes, setup);
            if constexpr (STREAM) {
                // the segments come from every sequence's length: pull the lengths into L2
                // (whole 16-byte granules of the caller's 256-byte aligned buffer)
                const uintptr_t l0 = reinterpret_cast<uintptr_t>(a.seq_lens) & ~uintptr_t(15);
                const uintptr_t l1 = (reinterpret_cast<uintptr_t>(a.seq_lens + a.B) + 15) & ~uintptr_t(15);
                prefetch_l2(reinterpret_cast<const void*>(l0), static_cast<uint32_t>(l1 - l0 < 4096 ? l1 - l0 : 4096));
            } else {
                {
                    // While the previous kernel finishes, pull the first tile of this split
                    // (by max_seq: the lengths are not read yet) into L2 -- only the first:
                    // all CTAs' first tiles then arrive within the overlap, and the next ones
                    // stream once the copies start.  A prefetch changes no value any load
                    // returns, so it may precede the wait; the copies into shared memory
                    // come after it.
                    const int64_t pf_end = min(min(t0 + p.chunk, a.max_seq), t0 + static_cast<int64_t>(C::TS));
                    if (pf_end > t0) {
                        const uint32_t ntok = static_cast<uint32_t>(pf_end - t0);  // a multiple of 8
                        if constexpr (C::KRAW) {
                            for (int it = 0; it * C::TS < static_cast<int>(ntok); ++it)
#pragma unroll
                                for (int cb = 0; cb < D / 64; ++cb)
                                    prefetch_l2_2d(&kmap, 64 * cb, static_cast<int>(row0 + t0 + it * C::TS));
                        } else {
                            prefetch_l2(static_cast<const uint8_t*>(a.k) + (row0 + t0) * C::BPK, ntok * C::BPK);
                            prefetch_l2(a.k_norms + row0 + t0, ntok * 2);
                        }
                        prefetch_l2(a.v_codes + (row0 + t0) * C::BPV, ntok * C::BPV);
                        prefetch_l2(a.v_norms + row0 + t0, ntok * 2);
                    }
                    // the query block and the 16-byte granule holding seq_lens[b] (allocations
                    // are 256-byte aligned, so the granule lies inside the caller's buffer)
                    prefetch_l2(a.q + qrow0 * D, qbytes);
                    prefetch_l2(reinterpret_cast<const void*>(reinterpret_cast<uintptr_t>(a.seq_lens + b) & ~uintptr_t(15)), 16);
                }
                asm volatile("griddepcontrol.wait;" ::: "memory");
                allow_dependent_launch();
                if constexpr (Q_STAGED) {
                    mbar_arrive_expect_tx(setup_q, qbytes);
                    bulk_g2s(pro + C::PRO_Q, a.q + qrow0 * D, qbytes, setup_q);
                }
                // The first ring-full of tiles goes out before the sequence length is known, sized
                // by max_seq (every copy stays inside the caller's cache); the consumers mask the
                // tokens past the length, and tiles past it are drained unconsumed.
                const int pre = pre_tiles(t0, p.chunk, a.max_seq);
                for (int it = 0; it < pre; ++it) issue(it, it, min(t0 + p.chunk, a.max_seq));
                t1 = min(clamped_len(a, b), t0 + p.chunk);
                ntiles = (t1 > t0) ? static_cast<int>((t1 - t0 + C::TS - 1) / C::TS) : 0;
                issued = pre;
                for (int it = pre; it < ntiles; ++it) {
                    const int s = it % C::NSTAGE;
                    if (it >= C::NSTAGE && !mbar_wait(empty + s, ((it / C::NSTAGE) - 1) & 1)) {
                        atomicOr(error_ptr(a.ws), TQ_DEVERR_TIMEOUT);
                        *s_abort = 1;
                        break;
                    }
                    issue(it, it, t1);
                    issued = it + 1;
                }
                // Tiles issued before the length was known that lie past it are never consumed:
                // their copies land before the consumers reuse the ring for the merge.
                for (int it = ntiles; it < pre; ++it) {
                    if (!mbar_wait(full + (it % C::NSTAGE), (it / C::NSTAGE) & 1)) {
                        atomicOr(error_ptr(a.ws), TQ_DEVERR_TIMEOUT);
                        *s_abort = 1;
                        break;
                    }
                }
            }
        }
        if constexpr (STREAM) {
            // Segment by segment: the copies of the segment's tiles (continuing around the
            // ring); where the merge reuses the ring, then the arrival on barrier 2 (all
            // copies issued) and, before the next segment's copies, barrier 3: the
            // consumers' merge of this segment is done.
            __syncwarp();
            asm volatile("griddepcontrol.wait;" ::: "memory");
            if (lane == 0) allow_dependent_launch();
            StreamWalk sw;
            sw.init(a, blockIdx.x, p.n_cta, p.stream_ovh, lane, false);
            int itg = 0;
            bool stop = false;
            while (sw.valid) {
                u = sw.b * a.Hkv + sw.h;
                row0 = static_cast<int64_t>(u) * a.max_seq;
                t0 = sw.a0;
                const int64_t te = sw.a1();
                const int nt = static_cast<int>((te - t0 + C::TS - 1) / C::TS);
                if (lane == 0 && !stop) {
                    for (int it = 0; it < nt; ++it) {
                        const int gi = itg + it;
                        if (gi >= C::NSTAGE && !mbar_wait(empty + (gi % C::NSTAGE), ((gi / C::NSTAGE) - 1) & 1)) {
                            atomicOr(error_ptr(a.ws), TQ_DEVERR_TIMEOUT);
                            *s_abort = 1;
                            stop = true;
                            break;
                        }
                        issue(gi, it, te);
                        issued = gi + 1;
                    }
                }
                itg += nt;
                __syncwarp();
                if constexpr (!SEP) asm volatile("bar.arrive 2, %0;" ::"n"((C::NWC + 1) * 32) : "memory");
                sw.next(a);
                if (!SEP && sw.valid) asm volatile("bar.sync 3, %0;" ::"n"((C::NWC + 1) * 32) : "memory");
            }
        } else {
            __syncwarp();  // reconverge the producer warp before the block-wide barriers
            asm volatile("bar.arrive 2, %0;" ::"n"((C::NWC + 1) * 32) : "memory");
        }
    } else {
        // ------------------------------------------------------------ consumers: prologue
        const int ctid = tid;  // 0 .. C::NWC * 32 - 1
        int64_t len = 0;
        // Every prologue read of global memory is issued at once (one memory
        // latency for the CTA, not one per loop iteration).
        bool ok = __all_sync(kFullMask, mbar_wait(setup, 0));
#ifdef TQ_TIMELINE
        if (threadIdx.x == 0) {  // slot 1: the SM this CTA runs on
            unsigned sm;
            asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
            tl_t[1] = sm;
        }
#endif
        replicate_tables<C>(reinterpret_cast<const uint32_t*>(pro + C::PRO_K),
                            reinterpret_cast<const uint32_t*>(pro + C::PRO_V), ktab_s, vtab_s, ctid);
        asm volatile("griddepcontrol.wait;" ::: "memory");
        TQ_TL(tl_t, 2);
        // Past the wait, everything stream-ordered before this kernel is complete: the
        // combine kernel that follows may start (and read the call's inputs) once every
        // CTA has triggered, which each CTA does only after one of its threads has
        // passed this wait.
        allow_dependent_launch();
        StreamWalk sw;
        if constexpr (STREAM) sw.init(a, blockIdx.x, p.n_cta, p.stream_ovh, lane, warp == 0);
        int itg = 0;  // ring position of the segment's first tile
        // One pass per segment of a unit's tokens: this CTA's split of its unit, or, on the
        // token-balanced schedule, each unit its positions cover (barrier 3 tells the
        // producer that the segment's merge no longer reads the ring).
        for (;;) {
            if constexpr (STREAM) {
                if (!sw.valid) break;
                b = sw.b;
                kvh = sw.h;
                u = vu = b * a.Hkv + kvh;
                qrow0 = static_cast<int64_t>(b) * a.Hq + kvh * G;
                row0 = static_cast<int64_t>(u) * a.max_seq;
                t0 = sw.a0;
                len = sw.len;
                t1 = sw.a1();
            } else {
                len = clamped_len(a, b);
                t1 = min(len, t0 + p.chunk);
            }
            ntiles = (t1 > t0) ? static_cast<int>((t1 - t0 + C::TS - 1) / C::TS) : 0;
            {
                if constexpr (Q_STAGED) ok = __all_sync(kFullMask, ok && mbar_wait(setup_q, 0));
                if (!ok && lane == 0) {
                    atomicOr(error_ptr(a.ws), TQ_DEVERR_TIMEOUT);
                    *s_abort = 1;
                }
                rotate_queries<D, C::NWC, C::KRAW, kGP * RG>(a, reinterpret_cast<const uint16_t*>(pro + C::PRO_Q),
                                                             a.q + qrow0 * D,
                                                             reinterpret_cast<const uint32_t*>(pro + C::PRO_S), G + G1,
                                                             qs, warp, lane, ctid);
                if (MULTI && ctid < kGP * RG) {
                    // Causal end of each query row, as tokens past t0: the rows' positions are the
                    // last L of the sequence (packed tokens, then tail), so every packed token is
                    // visible when L == 1 or the tail is long enough.  Clamped to t1, it also marks
                    // the split's end.  (The second row group's ends sit at s_erel1.)
                    const int tail = p.L > 1 ? tail_count(a, b) : 0;
                    const int64_t e = min(packed_visible(len, tail, p.L, (s0 + ctid) % p.L), t1);
                    (ctid < kGP ? s_erel : s_erel1)[ctid % kGP] = e > t0 ? static_cast<int>(e - t0) : 0;
                }
            }
            asm volatile("bar.sync 1, %0;" ::"n"(C::NWC * 32) : "memory");
            TQ_TL(tl_t, 7);

            const int g = lane >> 2, t = lane & 3;
            // q' B fragments: Bq[kt][nt][2] (in shared memory for D > 128)
            uint32_t Bq[C::BQ_SMEM ? 1 : C::KTS][C::NTS][2];
            const uint32_t bq_a = smem_addr(bq_s);
#pragma unroll
            for (int rg = 0; rg < RG; ++rg) {
#pragma unroll
            for (int kt = 0; kt < C::KTS; ++kt) {
#pragma unroll
                for (int nt = 0; nt < C::NTS; ++nt) {
                    const int qh = rg * kGP + ((NT == 2) ? g : (g >> 1));
                    const bool lo_part = (NT == 2) ? (nt == 1) : ((g & 1) != 0);
                    uint32_t b0, b1;
                    if constexpr (C::KEXP) {
                        // dims d0, d1 = (D/4) t + 2 kt + {0, 1}; k pair = (K_hi, K_lo) of one dim
                        const int d0 = (D / 4) * t + 2 * kt;
                        float v[2];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const float x = qs[qh * D + d0 + e];
                            const float hi = __half2float(__float2half_rn(x));
                            v[e] = lo_part ? (x - hi) : x;
                        }
                        if (NT == 2 && lo_part) {  // q_lo multiplies K_hi only
                            b0 = pack_f16(v[0], 0.0f);
                            b1 = pack_f16(v[1], 0.0f);
                        } else {
                            b0 = pack_f16(v[0], v[0]);
                            b1 = pack_f16(v[1], v[1]);
                        }
                    } else {
                        // coded K: dims (D/4) t + 4 kt + {0..3} (the K-role map); raw K:
                        // the ldmatrix layout, dims 16 kt + 2 t + {0, 1, 8, 9}
                        const int base = C::KRAW ? 16 * kt + 2 * t : (D / 4) * t + 4 * kt;
                        float v[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float x = qs[qh * D + base + (C::KRAW ? (e & 1) + 8 * (e >> 1) : e)];
                            const float hi = __half2float(__float2half_rn(x));
                            v[e] = lo_part ? (x - hi) : x;
                        }
                        b0 = pack_f16(v[0], v[1]);
                        b1 = pack_f16(v[2], v[3]);
                    }
                    if constexpr (C::BQ_SMEM) {
                        // (row group rg's fragments after group 0's in each k-tile; warp rg writes them)
                        if (warp == rg) sts64(bq_a + (((kt * RG + rg) * C::NTS + nt) * 32 + lane) * 8, b0, b1);
                    } else {
                        Bq[kt][nt][0] = b0;
                        Bq[kt][nt][1] = b1;
                    }
                }
            }
            }
            if constexpr (QJL) {
                // u = S q' for this CTA's query rows, as B fragments of the sketch k-tiles ("How I
                // built VeloxQuant-MLX", Stage 3: the correction reads <S_j, q> for every sketch
                // row j).  Sketch k-tile kk, thread (g, t): k = 2t, 2t+1, 2t+8, 2t+9 are sketch rows
                // 32 (kk / 2) + b, b = 4t + 2 (kk % 2) + 0, 16, 1, 17 -- bits b of the keys' sign
                // word kk / 2, so that the two bits of an A register sit 16 apart and one shift puts
                // them on its fp16 sign bits.  q' is split into fp16 hi and lo as for the scores.
                // Warp w takes sketch rows j = 32 w + lane for all rows of q' (S^T rows read
                // across the lanes, coalesced; q' broadcast from shared memory), then forms the
                // fragments of k-tiles 2w and 2w + 1 from its lanes by shuffles.
                const uint32_t ubq_a = smem_addr(ubq_s);
                // With enough warps each block of 32 sketch rows is summed by two warps over the
                // two halves of i (16 loads of S^T in flight per batch, from L2); the second
                // warp's partial sums pass through the block's own fragment area, which the
                // first warp reads before it writes the fragments there.
                constexpr int NB = D / 32;
                constexpr bool HALVES = 2 * NB <= C::NWC;
                constexpr int RQ = (NT == 2) ? kGP : 4;                   // rows that hold a query
                constexpr uint32_t PBYTES = (NT == 2) ? 1024u : 512u;     // a block's fragment area
                const int part = HALVES ? warp / NB : 0;
                for (int w = (HALVES ? warp % NB : warp); w < NB && part < 2; w += (HALVES ? NB : C::NWC)) {
                    float uq[kGP];
#pragma unroll
                    for (int g2 = 0; g2 < kGP; ++g2) uq[g2] = 0.0f;
                    const float* col = a.ck.sketch_t + 32 * w + lane;
                    const int i_beg = HALVES ? part * (D / 2) : 0, i_end = HALVES ? i_beg + D / 2 : D;
                    for (int i0 = i_beg; i0 < i_end; i0 += 16) {
                        float sv[16];
#pragma unroll
                        for (int k = 0; k < 16; ++k) sv[k] = __ldg(col + static_cast<int64_t>(i0 + k) * D);
#pragma unroll
                        for (int k = 0; k < 16; ++k)
#pragma unroll
                            for (int g2 = 0; g2 < kGP; ++g2) uq[g2] = fmaf(sv[k], qs[g2 * D + i0 + k], uq[g2]);
                    }
                    if (HALVES) {
                        const uint32_t pa = ubq_a + static_cast<uint32_t>(w) * PBYTES;
                        if (part == 1) {
#pragma unroll
                            for (int g2 = 0; g2 < RQ; ++g2) sts32(pa + (g2 * 32 + lane) * 4, __float_as_uint(uq[g2]));
                        }
                        asm volatile("bar.sync 1, %0;" ::"n"(C::NWC * 32) : "memory");
                        if (part == 1) break;
#pragma unroll
                        for (int g2 = 0; g2 < RQ; ++g2) uq[g2] += __uint_as_float(lds32(pa + (g2 * 32 + lane) * 4));
                        __syncwarp();
                    }
                    const int gg = lane >> 2, tt = lane & 3;
                    const int qh = (NT == 2) ? gg : (gg >> 1);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int kk = 2 * w + h;
                        float hi[4], lo[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            // sketch row 32 w + b of query row qh, from lane b = 4 tt + 2 h + (e / 2) + 16 (e % 2)
                            float x = 0.0f;
#pragma unroll
                            for (int g2 = 0; g2 < kGP; ++g2) {
                                const float y = __shfl_sync(kFullMask, uq[g2], 4 * tt + 2 * h + (e >> 1) + 16 * (e & 1));
                                if (g2 == qh) x = y;
                            }
                            hi[e] = __half2float(__float2half_rn(x));
                            lo[e] = x - hi[e];
                        }
                        if constexpr (NT == 2) {
                            sts64(ubq_a + ((kk * 2) * 32 + lane) * 8, pack_f16(hi[0], hi[1]), pack_f16(hi[2], hi[3]));
                            sts64(ubq_a + ((kk * 2 + 1) * 32 + lane) * 8, pack_f16(lo[0], lo[1]), pack_f16(lo[2], lo[3]));
                        } else {
                            const float* v = (gg & 1) ? lo : hi;  // interleaved hi / lo columns
                            sts64(ubq_a + (kk * 32 + lane) * 8, pack_f16(v[0], v[1]), pack_f16(v[2], v[3]));
                        }
                    }
                    if (HALVES) break;
                }
                // the warps without a block meet the halves' barrier too
                if (HALVES && warp >= 2 * NB) asm volatile("bar.sync 1, %0;" ::"n"(C::NWC * 32) : "memory");
            }
            if constexpr (C::BQ_SMEM || QJL) asm volatile("bar.sync 1, %0;" ::"n"(C::NWC * 32) : "memory");

            float O[RG][C::KT][4];  // per row group
            float m_run[RG][NT], l_run[RG][NT];
#pragma unroll
            for (int rg = 0; rg < RG; ++rg) {
#pragma unroll
                for (int i = 0; i < C::KT; ++i) O[rg][i][0] = O[rg][i][1] = O[rg][i][2] = O[rg][i][3] = 0.0f;
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    m_run[rg][j] = -CUDART_INF_F;
                    l_run[rg][j] = 0.0f;
                }
            }
            const uint32_t ktab_a = smem_addr(ktab_s), vtab_a = smem_addr(vtab_s);
            // table block: the table address bits ride in the lane offsets (kTBlock is
            // 64 KB aligned, the V half of a row starts at +128)
            const uint32_t koff = uint32_t(lane * 4) | (C::TBLOCK  ? uint32_t(kTBlock)
                                                        : C::BASED ? uint32_t(kTBlock + C::KBASE)
                                                                   : 0u);
            const uint32_t lane4 = uint32_t(lane * 4) | (C::TBLOCK  ? uint32_t(kTBlock) + 128u
                                                         : C::BASED ? uint32_t(kTBlock + C::VBASE)
                                                                    : 0u);

            // ------------------------------------------------------------ main loop
            // (after a wait gave up, the token-balanced schedule's later segments skip their tiles)
            const int nloop = (STREAM && *reinterpret_cast<volatile int*>(s_abort)) ? 0 : ntiles;
            for (int it = 0; it < nloop; ++it) {
                const int gi = itg + it;  // the tile's place in the ring sequence
                const int s = gi % C::NSTAGE;
                // the warp decides together so every later barrier is reached convergently
                const bool ok = __all_sync(kFullMask, mbar_wait(full + s, (gi / C::NSTAGE) & 1));
                if (!ok) {
                    if (lane == 0) {
                        atomicOr(error_ptr(a.ws), TQ_DEVERR_TIMEOUT);
                        *s_abort = 1;
                    }
                    break;
                }
#ifdef TQ_TIMELINE
                if (it == 0) TQ_TL(tl_t, 3);
#endif
                const uint8_t* st = stage_ptr(s);
                const uint8_t* kbuf = st;
                const uint8_t* vbuf = st + C::KBUF;
                const __half* knrm = reinterpret_cast<const __half*>(st + C::KBUF + C::VBUF);
                const __half* vnrm = reinterpret_cast<const __half*>(st + C::KBUF + C::VBUF + C::NBUF);
                const int64_t ts = t0 + static_cast<int64_t>(it) * C::TS;
                const int nvalid = static_cast<int>(min(static_cast<int64_t>(C::TS), t1 - ts));
                const int r0 = warp * 16 * C::MT;
                if (r0 < nvalid) {
                    // ---- scores for MT m-tiles ----
                    float sc[RG][C::MT][C::NTS][4];
#pragma unroll
                    for (int mt = 0; mt < C::MT; ++mt) {
#pragma unroll
                        for (int rg = 0; rg < RG; ++rg)
#pragma unroll
                            for (int nt = 0; nt < C::NTS; ++nt)
                                sc[rg][mt][nt][0] = sc[rg][mt][nt][1] = sc[rg][mt][nt][2] = sc[rg][mt][nt][3] = 0.0f;
                        const int ra = r0 + 16 * mt + g, rb = ra + 8;
                        if constexpr (C::KRAW) {
                            // rows r0 + 16 mt + 0..15 of the swizzled 64-column blocks: lanes 0-7 /
                            // 8-15 / 16-23 / 24-31 address rows 0-7 / 8-15 / 0-7 / 8-15 at 16-byte
                            // chunk 2 kl / 2 kl / 2 kl + 1 / 2 kl + 1 of the block, chunk c of
                            // row r sitting at chunk c ^ (r & 7)
                            const uint32_t rowa = smem_addr(kbuf) +
                                                  static_cast<uint32_t>((r0 + 16 * mt + (lane & 15)) * 128);
#pragma unroll
                            for (int kt = 0; kt < C::KTS; ++kt) {
                                const int cb = kt >> 2, kl = kt & 3;
                                const uint32_t chunk = static_cast<uint32_t>(2 * kl) + static_cast<uint32_t>(lane >> 4);
                                uint32_t a0, a1, a2, a3;
                                ldmatrix_x4(rowa + cb * C::KREG + ((chunk ^ static_cast<uint32_t>(lane & 7)) << 4), a0, a1,
                                            a2, a3);
                                uint32_t q00, q01, q10 = 0u, q11 = 0u;
                                q_frag<C>(Bq, bq_a, kt, lane, q00, q01, q10, q11);
                                mma16816(sc[0][mt][0], a0, a1, a2, a3, q00, q01);
                                if constexpr (C::NTS == 2) mma16816(sc[0][mt][1], a0, a1, a2, a3, q10, q11);
                            }
                        } else {
                        uint32_t wa[C::KCW], wb[C::KCW];
                        load_k_chunk<D, KB, C::KCW>(kbuf, ra, t, wa);
                        load_k_chunk<D, KB, C::KCW>(kbuf, rb, t, wb);
                        if constexpr (C::KPERM) {
#pragma unroll
                            for (int kt = 0; kt < C::KTS; ++kt) {
                                // bytes 2(kt&1), 2(kt&1)+1 of word kt/2 are dims d0, d1 of this k-tile
                                // (4-bit keys: the pairs of dims d0, d0 + 1 and d0 + 2, d0 + 3)
                                const uint32_t wA = wa[kt >> 1], wB = wb[kt >> 1];
                                // address = [koff byte 3][koff byte 2 / 0][code][koff byte 0]: with the
                                // table block the permute alone forms it, else it is added to ktab_a
                                const uint32_t sel0 = (C::TBLOCK ? 0x7604u : 0x5504u) + ((2u * (kt & 1)) << 4);
                                const uint32_t sel1 = sel0 + 0x10u;
                                const uint32_t kb = C::TBLOCK ? 0u : ktab_a;
                                const uint32_t r0v = lds32(kb + __byte_perm(wA, koff, sel0));
                                const uint32_t r1v = lds32(kb + __byte_perm(wB, koff, sel0));
                                const uint32_t r2v = lds32(kb + __byte_perm(wA, koff, sel1));
                                const uint32_t r3v = lds32(kb + __byte_perm(wB, koff, sel1));
                                // (every row group's contraction takes the same dequantised operand)
#pragma unroll
                                for (int rg = 0; rg < RG; ++rg) {
                                    uint32_t q00, q01, q10 = 0u, q11 = 0u;
                                    q_frag<C>(Bq, bq_a, kt, lane, q00, q01, q10, q11, rg);
                                    mma16816(sc[rg][mt][0], r0v, r1v, r2v, r3v, q00, q01);
                                    if constexpr (C::NTS == 2) mma16816(sc[rg][mt][1], r0v, r1v, r2v, r3v, q10, q11);
                                }
                            }
                        } else {
#pragma unroll
                            for (int kt = 0; kt < C::KTS; ++kt) {
                                uint32_t ah01, ah23, bh01, bh23;
                                // (based tables: the table's address bits are in koff)
                                k_role<KB, C::KCW>(wa, kt, C::BASED ? 0u : ktab_a, koff, ah01, ah23);
                                k_role<KB, C::KCW>(wb, kt, C::BASED ? 0u : ktab_a, koff, bh01, bh23);
                                // A regs: {row g: k 2t,2t+1}, {row g+8: k 2t,2t+1}, {row g: k 2t+8,2t+9}, {row g+8: ...}
                                uint32_t q00, q01, q10 = 0u, q11 = 0u;
                                q_frag<C>(Bq, bq_a, kt, lane, q00, q01, q10, q11);
                                mma16816(sc[0][mt][0], ah01, bh01, ah23, bh23, q00, q01);
                                if constexpr (C::NTS == 2) mma16816(sc[0][mt][1], ah01, bh01, ah23, bh23, q10, q11);
                            }
                            if constexpr (QJL) {
                                // QJL correction into the same accumulators: row r's A entries are
                                // +-v_r, v_r = gamma_r sqrt(pi/2) k_alpha / (sqrt(D) n16_K[r]) (the
                                // accumulator is scaled by n16_K[r] afterwards), sign from bit j
                                const uint8_t* sg = st + C::KBUF + C::VBUF + 2 * C::NBUF;
                                const __half* rnm = reinterpret_cast<const __half*>(sg + C::SBUF);
                                const float kap = 1.2533141373155003f * a.ck.k_alpha * rsqrtf(static_cast<float>(D));
                                const float nka = __half2float(knrm[ra]), nkb = __half2float(knrm[rb]);
                                const float fva = nka > 0.0f ? __half2float(rnm[ra]) * kap / nka : 0.0f;
                                const float fvb = nkb > 0.0f ? __half2float(rnm[rb]) * kap / nkb : 0.0f;
                                const uint32_t hva = pack_f16(fva, fva), hvb = pack_f16(fvb, fvb);
                                const uint32_t sga = smem_addr(sg) + static_cast<uint32_t>(ra * (D / 8));
                                const uint32_t sgb = smem_addr(sg) + static_cast<uint32_t>(rb * (D / 8));
                                const uint32_t ubq_a = smem_addr(ubq_s);
                                const int sh0 = 15 - 4 * t;  // bit 4t of a sign word -> bit 15
#pragma unroll
                                for (int w4 = 0; w4 < D / 32; ++w4) {
                                    const uint32_t wsa = lds32(sga + 4 * w4), wsb = lds32(sgb + 4 * w4);
#pragma unroll
                                    for (int h = 0; h < 2; ++h) {
                                        const int kk = 2 * w4 + h;
                                        // bits b, b + 16 (b = 4t + 2h) -> the sign bits of k = 2t, 2t + 1;
                                        // bits b + 1, b + 17 -> those of k = 2t + 8, 2t + 9
                                        const int s0 = sh0 - 2 * h;
                                        const uint32_t a0 = hva ^ ((wsa << s0) & 0x80008000u);
                                        const uint32_t a2 = hva ^ ((wsa << (s0 - 1)) & 0x80008000u);
                                        const uint32_t a1 = hvb ^ ((wsb << s0) & 0x80008000u);
                                        const uint32_t a3 = hvb ^ ((wsb << (s0 - 1)) & 0x80008000u);
                                        uint32_t u00, u01;
                                        lds64(ubq_a + ((kk * C::NTS) * 32 + lane) * 8, u00, u01);
                                        mma16816(sc[0][mt][0], a0, a1, a2, a3, u00, u01);
                                        if constexpr (C::NTS == 2) {
                                            uint32_t u10, u11;
                                            lds64(ubq_a + ((kk * C::NTS + 1) * 32 + lane) * 8, u10, u11);
                                            mma16816(sc[0][mt][1], a0, a1, a2, a3, u10, u11);
                                        }
                                    }
                                }
                            }
                        }
                        }
                    }
                    // ---- scale by K norms, mask (tile end, causal limit), tile max ----
                    // (per row group: each has its own rows, causal ends and running state)
                    float sv[RG][C::MT][2][NT];  // [group][m-tile][row g / g+8][query slot]
                    float muse[RG][NT];
#pragma unroll
                    for (int rg = 0; rg < RG; ++rg) {
                    const int* erel = (rg == 0) ? s_erel : s_erel1;
                    float tmax[NT];
#pragma unroll
                    for (int j = 0; j < NT; ++j) tmax[j] = -CUDART_INF_F;
                    // this thread's query rows (2t + j, or t when NT == 1): causal ends in the tile
                    // (decode: the tile's end)
                    int lim[NT];
#pragma unroll
                    for (int j = 0; j < NT; ++j) lim[j] = MULTI ? erel[(NT == 2) ? 2 * t + j : t] - it * C::TS : nvalid;
#pragma unroll
                    for (int mt = 0; mt < C::MT; ++mt) {
#pragma unroll
                        for (int hr = 0; hr < 2; ++hr) {
                            const int r = r0 + 16 * mt + g + 8 * hr;
                            const float nk = C::KRAW ? 1.0f : __half2float(knrm[r]);
#pragma unroll
                            for (int j = 0; j < NT; ++j) {
                                float x;
                                if constexpr (C::NTS == 2)
                                    x = sc[rg][mt][0][2 * hr + j] + sc[rg][mt][1][2 * hr + j];
                                else if constexpr (NT == 2)
                                    x = sc[rg][mt][0][2 * hr + j];
                                else
                                    x = sc[rg][mt][0][2 * hr] + sc[rg][mt][0][2 * hr + 1];
                                // lim <= t1 - ts, so this also masks the rows past the tile's end
                                x = (r < lim[j]) ? x * nk : -CUDART_INF_F;
                                sv[rg][mt][hr][j] = x;
                                tmax[j] = fmaxf(tmax[j], x);
                            }
                        }
                    }
#pragma unroll
                    for (int j = 0; j < NT; ++j) {
                        tmax[j] = fmaxf(tmax[j], __shfl_xor_sync(kFullMask, tmax[j], 4));
                        tmax[j] = fmaxf(tmax[j], __shfl_xor_sync(kFullMask, tmax[j], 8));
                        tmax[j] = fmaxf(tmax[j], __shfl_xor_sync(kFullMask, tmax[j], 16));
                    }
                    float alpha[NT];
                    bool rescale = false;
#pragma unroll
                    for (int j = 0; j < NT; ++j) {
                        const float mn = fmaxf(m_run[rg][j], tmax[j]);
                        muse[rg][j] = (mn == -CUDART_INF_F) ? 0.0f : mn;
                        alpha[j] = ex2_approx(m_run[rg][j] - muse[rg][j]);
                        rescale |= (alpha[j] != 1.0f);
                        m_run[rg][j] = mn;
                        l_run[rg][j] *= alpha[j];
                    }
                    if (__any_sync(kFullMask, rescale)) {
                        // (MULTI, NT == 1: columns 2t and 2t + 1 both hold row t, hi and lo of P)
                        const float a1 = (NT == 2 || MULTI) ? alpha[NT - 1] : 1.0f;
#pragma unroll
                        for (int i = 0; i < C::KT; ++i) {
                            O[rg][i][0] *= alpha[0];
                            O[rg][i][1] *= a1;
                            O[rg][i][2] *= alpha[0];
                            O[rg][i][3] *= a1;
                        }
                    }
                    }
                    // ---- probabilities, P' = p * n16_V, P.V ----
#pragma unroll
                    for (int mt = 0; mt < C::MT; ++mt) {
                        const int rbase = r0 + 16 * mt;
                        if (rbase >= nvalid) break;
                        uint32_t pb0[RG], pb1[RG], pl0[RG], pl1[RG];  // P fragments per row group
#pragma unroll
                        for (int rg = 0; rg < RG; ++rg) {
                        float pv[2][NT];
#pragma unroll
                        for (int hr = 0; hr < 2; ++hr) {
                            const int r = rbase + g + 8 * hr;
                            const bool ok = r < nvalid;
                            const float nvv = __half2float(vnrm[r]);
#pragma unroll
                            for (int j = 0; j < NT; ++j) {
                                const float pp = ex2_approx(sv[rg][mt][hr][j] - muse[rg][j]);
                                l_run[rg][j] += pp;
                                pv[hr][j] = ok ? pp * nvv : 0.0f;
                            }
                        }
                        // With several query positions (MULTI), P' is fp16 hi + lo, so the weights
                        // keep ~2^-22 of their precision: the first rows of a chunk see only a few
                        // tokens, and one fp16 P would carry their weights' 2^-11 rounding into
                        // the output.  NT == 1 puts the lo part in the free column 2t + 1, NT == 2
                        // multiplies V by it in a second mma.  Decode keeps one fp16 P, as fp16
                        // attention does.
                        uint32_t x0, x1;
                        pl0[rg] = 0u;
                        pl1[rg] = 0u;
                        if constexpr (NT == 2) {
                            if constexpr (MULTI) {
                                uint32_t y0, y1;
                                split_f16x2(pv[0][0], pv[0][1], x0, y0);
                                split_f16x2(pv[1][0], pv[1][1], x1, y1);
                                pl0[rg] = movmatrix_t(y0);
                                pl1[rg] = movmatrix_t(y1);
                            } else {
                                x0 = pack_f16(pv[0][0], pv[0][1]);
                                x1 = pack_f16(pv[1][0], pv[1][1]);
                            }
                        } else if constexpr (MULTI) {
                            uint32_t h0, l0;  // (row g, row g + 8) pairs
                            split_f16x2(pv[0][0], pv[1][0], h0, l0);
                            x0 = (h0 & 0xffffu) | (l0 << 16);
                            x1 = (h0 >> 16) | (l0 & 0xffff0000u);
                        } else {
                            x0 = pack_f16(pv[0][0], 0.0f);
                            x1 = pack_f16(pv[1][0], 0.0f);
                        }
                        pb0[rg] = movmatrix_t(x0);
                        pb1[rg] = movmatrix_t(x1);
                        }
                        // V of tokens 2t, 2t+1, 2t+8, 2t+9 of this m-tile, thread g's dims
                        constexpr bool SPLIT = MULTI && NT == 2;
                        if constexpr (C::VPAIR) {
                            constexpr int NSUB = (D / 8 + 15) / 16;  // chunks of up to 16 dims
#pragma unroll
                            for (int sub = 0; sub < NSUB; ++sub) {
                                const int vbit = g * C::VCB + 16 * VB * sub;
                                constexpr int VW = v_field_words(D, VB);  // words per field (2 at D 128, 3 bits)
                                const VPairs<VB, C::VMODE> p01(load_bits_w<VW>(vbuf + (rbase + 2 * t) * C::BPV, vbit),
                                                     load_bits_w<VW>(vbuf + (rbase + 2 * t + 1) * C::BPV, vbit));
                                const VPairs<VB, C::VMODE> p89(load_bits_w<VW>(vbuf + (rbase + 2 * t + 8) * C::BPV, vbit),
                                                     load_bits_w<VW>(vbuf + (rbase + 2 * t + 9) * C::BPV, vbit));
                                constexpr int DM_PER_SUB = 8;  // 16 dims = 8 m-tiles of two rows
#pragma unroll
                                for (int k = 0; k < DM_PER_SUB; ++k) {
                                    const int dm = sub * DM_PER_SUB + k;
                                    if (dm < C::KT) {
                                        const uint32_t a0 = lds32(p01.addr(2 * k, vtab_a, lane4));
                                        const uint32_t a1 = lds32(p01.addr(2 * k + 1, vtab_a, lane4));
                                        const uint32_t a2 = lds32(p89.addr(2 * k, vtab_a, lane4));
                                        const uint32_t a3 = lds32(p89.addr(2 * k + 1, vtab_a, lane4));
#pragma unroll
                                        for (int rg = 0; rg < RG; ++rg) {
                                            mma16816(O[rg][dm], a0, a1, a2, a3, pb0[rg], pb1[rg]);
                                            if constexpr (SPLIT) mma16816(O[rg][dm], a0, a1, a2, a3, pl0[rg], pl1[rg]);
                                        }
                                    }
                                }
                            }
                        } else {
                            uint32_t v0[C::VCW], v1[C::VCW], v2[C::VCW], v3[C::VCW];
                            const int vb = g * C::VCB;
                            load_chunk<C::VCW>(vbuf + (rbase + 2 * t) * C::BPV, vb, v0);
                            load_chunk<C::VCW>(vbuf + (rbase + 2 * t + 1) * C::BPV, vb, v1);
                            load_chunk<C::VCW>(vbuf + (rbase + 2 * t + 8) * C::BPV, vb, v2);
                            load_chunk<C::VCW>(vbuf + (rbase + 2 * t + 9) * C::BPV, vb, v3);
#pragma unroll
                            for (int dm = 0; dm < C::KT; ++dm) {
                                const uint32_t a0 = v_role<VB, C::VCW, C::VMODE>(v0, v1, 2 * dm, vtab_a, lane4);
                                const uint32_t a1 = v_role<VB, C::VCW, C::VMODE>(v0, v1, 2 * dm + 1, vtab_a, lane4);
                                const uint32_t a2 = v_role<VB, C::VCW, C::VMODE>(v2, v3, 2 * dm, vtab_a, lane4);
                                const uint32_t a3 = v_role<VB, C::VCW, C::VMODE>(v2, v3, 2 * dm + 1, vtab_a, lane4);
#pragma unroll
                                for (int rg = 0; rg < RG; ++rg) {
                                    mma16816(O[rg][dm], a0, a1, a2, a3, pb0[rg], pb1[rg]);
                                    if constexpr (SPLIT) mma16816(O[rg][dm], a0, a1, a2, a3, pl0[rg], pl1[rg]);
                                }
                            }
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(empty + s);
            }
            // (row group by row group: one partial record each)
#pragma unroll
            for (int rg = 0; rg < RG; ++rg) {
                // ------------------------------------------------------------ warp totals
                TQ_TL(tl_t, 4);
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    l_run[rg][j] += __shfl_xor_sync(kFullMask, l_run[rg][j], 4);
                    l_run[rg][j] += __shfl_xor_sync(kFullMask, l_run[rg][j], 8);
                    l_run[rg][j] += __shfl_xor_sync(kFullMask, l_run[rg][j], 16);
                }
                if (g == 0) {
#pragma unroll
                    for (int j = 0; j < NT; ++j) {
                        const int q = (NT == 2) ? 2 * t + j : t;
                        wm[warp * kGP + q] = m_run[rg][j];
                        wl[warp * kGP + q] = l_run[rg][j];
                    }
                    if constexpr (NT == 1) {
                        wm[warp * kGP + 4 + t] = -CUDART_INF_F;
                        wl[warp * kGP + 4 + t] = 0.0f;
                    }
                }
                // every consumer is done with the ring, wm / wl are visible, and the producer has no
                // copy in flight (barrier 2 counts the producer warp's arrival); with a merge area of
                // its own the producer goes on, and the consumers alone meet
                // (a second row group: the consumers alone, the producer arrived once)
                if (SEP || rg > 0)
                    asm volatile("bar.sync 1, %0;" ::"n"(C::NWC * 32) : "memory");
                else
                    asm volatile("bar.sync 2, %0;" ::"n"((C::NWC + 1) * 32) : "memory");
                TQ_TL(tl_t, 5);
                float f[NT];
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    const int q = (NT == 2) ? 2 * t + j : t;
                    float M = -CUDART_INF_F;
                    for (int w = 0; w < C::NWC; ++w) M = fmaxf(M, wm[w * kGP + q]);
                    // the V table holds v_alpha * c: divide it out here, once per output
                    f[j] = (m_run[rg][j] == -CUDART_INF_F) ? 0.0f : exp2f(m_run[rg][j] - M) / a.cv.v_alpha;
                }
                // Each warp's O slice goes to shared memory as float2 units (dims 2c, 2c + 1 of one
                // row) at merge_slot(): row-major with the low bits of c XOR-ed, so that the 16 lanes
                // of a half-warp store to 16 distinct bank pairs (row-major without it put every lane
                // of a row parity on the same two banks).
                float2* const merge_base = reinterpret_cast<float2*>(SEP ? smem + C::SMEM : ring);
                float2* slice = merge_base + warp * (SROWS * D / 2);
#pragma unroll
                for (int dm = 0; dm < C::KT; ++dm) {
                    const int c = (D / 16) * g + dm;  // dims (D/8) g + 2 dm + {0, 1}
                    if constexpr (NT == 2) {
                        slice[merge_slot<D>(2 * t, c)] = make_float2(f[0] * O[rg][dm][0], f[0] * O[rg][dm][2]);
                        slice[merge_slot<D>(2 * t + 1, c)] = make_float2(f[1] * O[rg][dm][1], f[1] * O[rg][dm][3]);
                    } else if constexpr (MULTI) {  // columns 2t, 2t + 1: the hi and lo parts of row t's P
                        slice[merge_slot<D>(t, c)] = make_float2(f[0] * (O[rg][dm][0] + O[rg][dm][1]), f[0] * (O[rg][dm][2] + O[rg][dm][3]));
                        slice[merge_slot<D>(4 + t, c)] = make_float2(0.0f, 0.0f);
                    } else {
                        slice[merge_slot<D>(t, c)] = make_float2(f[0] * O[rg][dm][0], f[0] * O[rg][dm][2]);
                        if constexpr (SROWS == kGP) slice[merge_slot<D>(4 + t, c)] = make_float2(0.0f, 0.0f);
                    }
                }
                asm volatile("bar.sync 1, %0;" ::"n"(C::NWC * 32) : "memory");
                // fixed-order sum of the warp slices, straight into this CTA's partial record: thread i
                // sums the float4 at physical units 2i, 2i + 1 of every slice (the same swizzled place
                // in each) and stores it at its logical place (units c0 and c0 ^ 1 of the row)
                float* part = STREAM ? partial_slot_ptr(a.ws, p, static_cast<int64_t>(blockIdx.x) + u, D)
                                     : partial_ptr(a.ws, p, vu + rg, split, D);
                const float4* all4 = reinterpret_cast<const float4*>(merge_base);
                float4* part4 = reinterpret_cast<float4*>(part);
                for (int i = tid; i < kGP * D / 4; i += C::NWC * 32) {
                    const int row = (2 * i) / (D / 2), cp = (2 * i) % (D / 2);
                    if (SROWS < kGP && row >= SROWS) {  // rows with no query head
                        part4[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                        continue;
                    }
                    float4 acc = all4[i];
#pragma unroll
                    for (int w = 1; w < C::NWC; ++w) {
                        const float4 x = all4[w * (SROWS * D / 4) + i];
                        acc.x += x.x;
                        acc.y += x.y;
                        acc.z += x.z;
                        acc.w += x.w;
                    }
                    const int c0 = merge_slot<D>(row, cp) - row * (D / 2);  // the swizzle is an involution
                    part4[row * (D / 4) + (c0 >> 1)] = (c0 & 1) ? make_float4(acc.z, acc.w, acc.x, acc.y) : acc;
                }
                if (tid < kGP) {
                    const int q = tid;
                    float M = -CUDART_INF_F;
                    for (int w = 0; w < C::NWC; ++w) M = fmaxf(M, wm[w * kGP + q]);
                    float L = 0.0f;
                    for (int w = 0; w < C::NWC; ++w) {
                        const float mw = wm[w * kGP + q];
                        if (mw != -CUDART_INF_F) L += wl[w * kGP + q] * exp2f(mw - M);
                    }
                    const int Gg = (rg == 0) ? G : G1;  // rows of this group
                    part[kGP * D + q] = (q < Gg) ? M : -CUDART_INF_F;
                    part[kGP * D + kGP + q] = (q < Gg) ? L : 0.0f;
                }
                // the next group rewrites wm / wl and the slices once every thread is done with them
                if (RG > 1 && rg + 1 < RG) asm volatile("bar.sync 1, %0;" ::"n"(C::NWC * 32) : "memory");
            }
            if constexpr (STREAM) {
                itg += ntiles;
#ifdef TQ_TIMELINE
                if (threadIdx.x == 0) tl_t[1] += 1ull << 32;  // segments, above the SM id
#endif
                sw.next(a);
                if (!sw.valid) break;
                if constexpr (SEP) {
                    // the slices are read: the next segment's merge may overwrite them
                    asm volatile("bar.sync 1, %0;" ::"n"(C::NWC * 32) : "memory");
                } else {
                    asm volatile("bar.arrive 3, %0;" ::"n"((C::NWC + 1) * 32) : "memory");
                }
            } else {
                break;
            }
        }  // segments
    }
    __syncthreads();
#ifdef TQ_TIMELINE
    TQ_TL(tl_t, 6);
    if (tid == 0 && a.tl) {
        unsigned long long* r = tl_record(a, false, blockIdx.y * gridDim.x + blockIdx.x);
        if (r)
            for (int i = 0; i < kTlStamps; ++i) r[i] = tl_t[i];
    }
#endif
    if (warp == C::NWC && lane == 0 && *s_abort) {
        // a wait gave up: let every copy this CTA issued land before shared memory is released
        for (int it = (issued > C::NSTAGE ? issued - C::NSTAGE : 0); it < issued; ++it) {
            const long long c0 = clock64();
            while (!mbar_try_wait(full + (it % C::NSTAGE), (it / C::NSTAGE) & 1) && clock64() - c0 < kWaitCycles) {
            }
        }
    }
}


// Tensor map of raw fp16 K for the 2-D TMA copies (host; tq_decode_mma.cu).
cudaError_t encode_raw_k_map(CUtensorMap* map, const void* k, int dim, int64_t rows, int box_rows);

// Launch of one instantiation; split plan for one CTA per SM.
template <int D, int KB, int VB, int NT, bool MULTI, bool QJL = false, bool STREAM = false, int RG = 1>
cudaError_t launch_inst(const DecodeArgs& a, DecodePlan& p, cudaStream_t st) {
    using C = Cfg<D, KB, VB, NT, QJL, MULTI, RG>;
    static std::atomic<uint64_t> configured{0};  // one bit per device
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t bit = 1ull << (dev & 63);
    constexpr int SMEM = C::SMEM + stream_merge_bytes<D, KB, VB, NT, QJL, MULTI, STREAM>();
    if (!(configured.load() & bit)) {
        cudaError_t e = cudaFuncSetAttribute(decode_mma_kernel<D, KB, VB, NT, MULTI, QJL, STREAM, RG>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit);
    }
    CUtensorMap kmap{};
    if constexpr (C::KRAW) {
        // raw K [B * Hkv * max_seq rows, D] fp16 in boxes of TS rows x 64 columns, 128-byte swizzle
        const cudaError_t e = encode_raw_k_map(&kmap, a.k, D, static_cast<int64_t>(a.B) * a.Hkv * a.max_seq, C::TS);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = STREAM ? dim3(p.n_cta, 1) : dim3(p.n_split, p.n_units * (p.q_chunks / RG));
    cfg.blockDim = dim3(C::NTHREADS);
    cfg.dynamicSmemBytes = SMEM;
    p.decode_smem = SMEM;  // the combine kernel sizes its footprint against it
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_mma_kernel<D, KB, VB, NT, MULTI, QJL, STREAM, RG>, a, p, kmap);
}

#define TQ_MMA_CASE(KB_, VB_)                                                                 \
    if constexpr (mma_fits(D, KB_, VB_)) {                                                    \
        if (kb == KB_ && vb == VB_)                                                           \
            switch (nt) {                                                                     \
                case 1: return launch_inst<D, KB_, VB_, 1, false>(a, p, st);                      \
                case 2: return launch_inst<D, KB_, VB_, 2, false>(a, p, st);                      \
                case 3:                                                                       \
                case 4:                                                                       \
                    if constexpr (mma_fits(D, KB_, VB_, false, true))                         \
                        return nt == 3 ? launch_inst<D, KB_, VB_, 1, true>(a, p, st)              \
                                       : launch_inst<D, KB_, VB_, 2, true>(a, p, st);             \
                    return cudaErrorNotSupported;                                             \
                case 7:                                                                       \
                    if constexpr (KB_ == 8 && (D & (D - 1)) == 0 && mma_fits_rg2(D, KB_, VB_)) \
                        return launch_inst<D, KB_, VB_, 2, true, false, false, 2>(a, p, st);  \
                    return cudaErrorNotSupported;                                             \
                default:                                                                      \
                    if constexpr (KB_ <= 4 && (D & (D - 1)) == 0 && mma_fits(D, KB_, VB_, true)) \
                        return nt == 5 ? launch_inst<D, KB_, VB_, 1, false, true>(a, p, st)       \
                                       : launch_inst<D, KB_, VB_, 2, false, true>(a, p, st);      \
                    return cudaErrorNotSupported;                                             \
            }                                                                                 \
    }

// The token-balanced schedule's instantiations: one query position, one row group, coded
// keys, Walsh-Hadamard rotation (power-of-two dims).
#define TQ_MMA_STREAM_CASE(KB_, VB_)                                                          \
    if constexpr (mma_fits(D, KB_, VB_) && KB_ != 16 && (D & (D - 1)) == 0) {                 \
        if (kb == KB_ && vb == VB_) {                                                         \
            if (nt == 1) return launch_inst<D, KB_, VB_, 1, false, false, true>(a, p, st);    \
            if (nt == 2) return launch_inst<D, KB_, VB_, 2, false, false, true>(a, p, st);    \
            return cudaErrorNotSupported;                                                     \
        }                                                                                     \
    }

// The (K bits, V bits) schemes with a tensor-core instantiation.
constexpr int kSchemes[][2] = {{4, 4}, {3, 3}, {2, 2}, {4, 2}, {4, 3}, {8, 3}, {8, 4}, {8, 8}, {8, 2}, {3, 2},
                               {16, 4}, {16, 2}, {16, 3}};

template <int D>
cudaError_t launch_mma_d_stream(const DecodeArgs& a, DecodePlan& p, int kb, int vb, int nt, cudaStream_t st) {
    TQ_MMA_STREAM_CASE(4, 4)
    TQ_MMA_STREAM_CASE(3, 3)
    TQ_MMA_STREAM_CASE(2, 2)
    TQ_MMA_STREAM_CASE(4, 2)
    TQ_MMA_STREAM_CASE(4, 3)
    TQ_MMA_STREAM_CASE(8, 3)
    TQ_MMA_STREAM_CASE(8, 4)
    TQ_MMA_STREAM_CASE(8, 8)
    TQ_MMA_STREAM_CASE(8, 2)
    TQ_MMA_STREAM_CASE(3, 2)
    return cudaErrorNotSupported;
}

template <int D>
cudaError_t launch_mma_d(const DecodeArgs& a, DecodePlan& p, int kb, int vb, int nt, cudaStream_t st) {
    TQ_MMA_CASE(4, 4)
    TQ_MMA_CASE(3, 3)
    TQ_MMA_CASE(2, 2)
    TQ_MMA_CASE(4, 2)
    TQ_MMA_CASE(4, 3)
    TQ_MMA_CASE(8, 3)
    TQ_MMA_CASE(8, 4)
    TQ_MMA_CASE(8, 8)
    TQ_MMA_CASE(8, 2)
    TQ_MMA_CASE(3, 2)
    TQ_MMA_CASE(16, 4)
    TQ_MMA_CASE(16, 2)
    TQ_MMA_CASE(16, 3)
    return cudaErrorNotSupported;
}

#undef TQ_MMA_CASE
#undef TQ_MMA_STREAM_CASE

}  // namespace mma_detail
}  // namespace tq
