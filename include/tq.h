/*
 * tq.h -- C ABI of libtq, the GB300 (sm_103a) TurboQuant KV-cache hot path.
 *
 * What the library computes follows these pages (titles and sections):
 *  [PR]  "add TurboQuant KV cache compression" (mlx-swift-lm pull request #232):
 *        "Schemes" (asymmetric K/V bit widths, raw-fp16 keys) and "Design"
 *        (WHT for power-of-two head dims, dense fallback otherwise, one
 *        rotation and codebook shared per (dim, bits, seed), pending tokens
 *        encoded in batches).
 *  [VQ]  VeloxQuant-MLX, "How I built VeloxQuant-MLX": "Stage 1: Random
 *        Rotation", "Stage 2: Lloyd-Max Scalar Quantization" (norm kept as
 *        fp16), "The Core Idea" (Lloyd-Max conditions), "The Bit-Packing
 *        Problem" (LSB-first packing).
 *  [RVQ] VeloxQuant-MLX RVQ post, "The Throughput Problem": O(d log d)
 *        Hadamard rotation; quantisation by counting the midpoints a value
 *        exceeds.
 *  [TW]  "anyone still talking about mlx-swift-lm?": fused single-dispatch
 *        decode -- score, softmax and inline dequant in one kernel, K read
 *        once in its rotated basis, GQA served without expanding K/V.
 *
 * Conventions for every entry point:
 *  - Pointers named as device memory must point to memory of the device that
 *    is current when the call is made; host pointers are plain host memory.
 *  - fp16 values are passed as uint16_t bit patterns (IEEE binary16).
 *  - `stream` is a cudaStream_t cast to void* (NULL = the legacy default
 *    stream).  Every compute call only enqueues work on that stream and
 *    returns; nothing allocates device memory except tq_codec_create.
 *  - Arguments are checked before any launch; a failed check returns a
 *    status and enqueues nothing.  Violations that can only be seen on the
 *    device (lengths or positions read from device memory) are clamped and
 *    recorded in a device error word (see tq_get_device_error); kernels never
 *    trap and never wait on other blocks.
 *  - Inputs holding Inf/NaN are outside the contract.
 */
#ifndef TQ_H_
#define TQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TQ_OK = 0,
    TQ_ERR_INVALID_ARG = 1,   /* a pointer, size, stride or alignment is invalid */
    TQ_ERR_UNSUPPORTED = 2,   /* a valid request this build has no kernel for */
    TQ_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed */
    TQ_ERR_OOM = 4,           /* tq_codec_create could not allocate */
    TQ_ERR_WORKSPACE = 5,     /* workspace missing or smaller than required */
    TQ_ERR_DEVICE_CHECK = 6   /* a device-side check fired (tq_get_device_error) */
} tq_status;

/* Device error codes (bit flags) recorded by kernels. */
#define TQ_DEVERR_SEQ_LEN   1   /* seq_lens[b] < 0 or > max_seq: clamped */
#define TQ_DEVERR_POSITION  2   /* encode_append position outside [0, max_seq): row skipped */
#define TQ_DEVERR_TIMEOUT   4   /* a bounded wait inside a kernel gave up; its outputs are invalid */
#define TQ_DEVERR_LAYOUT    8   /* the GPU's shared-memory window does not match the layout the
                                   decode kernel was built for; its outputs are invalid */

typedef struct tq_codec tq_codec;   /* opaque; immutable after creation */

/* Library version as 10000*major + 100*minor + patch. */
int tq_version(void);

/* Short English text for a status code (static storage). */
const char *tq_status_string(tq_status s);

/*
 * Codec: the rotation and codebook shared by every layer that uses the same
 * (dim, bits, seed) ([PR] Design, "Shared codecs").
 *   dim   head dimension, a multiple of 32 in [32, 512].  Powers of two use
 *         the randomised Walsh-Hadamard rotation R = H diag(s) / sqrt(dim)
 *         with Rademacher signs s drawn from SplitMix64(seed) ([VQ] Stage 1,
 *         [RVQ]); other sizes use a dense orthogonal Q, the QR factor of a
 *         seeded Gaussian matrix ([PR] Design; [VQ] Stage 1).
 *   bits  2, 3, 4 or 8: Lloyd-Max codebook of N(0,1) with 2^bits levels
 *         ([VQ] The Core Idea); 16: raw fp16 keys, no codebook ([PR] Schemes,
 *         turbo0v*; such a codec may only be passed as the K codec of
 *         tq_decode_attend).
 *   seed  selects the signs / the dense matrix.
 * The codec is built on the host (fp64) and its tables are copied to the
 * current device, which the codec then belongs to.  *out receives a handle
 * owned by the caller (free with tq_codec_destroy).  Thread-safe to use from
 * several threads once created.
 * Errors: TQ_ERR_INVALID_ARG (dim/bits/out), TQ_ERR_OOM, TQ_ERR_CUDA.
 */
tq_status tq_codec_create(int dim, int bits, uint64_t seed, tq_codec **out);

/* Frees the codec and its device tables (NULL is ignored).  The caller must
 * ensure no enqueued work still uses it. */
void tq_codec_destroy(tq_codec *codec);

/* Codec parameters; any output pointer may be NULL.  bytes_per_vec is the
 * packed row size dim*bits/8 (dim*2 for bits == 16); is_wht is 1 for the
 * Hadamard rotation, 0 for the dense one; *centroids_host points at the
 * codec's own host copy of its 2^bits fp32 centroids, ascending (NULL for
 * bits == 16), valid until tq_codec_destroy. */
tq_status tq_codec_info(const tq_codec *codec, int *dim, int *bits, int *bytes_per_vec,
                        int *is_wht, const float **centroids_host);

/* The rotation of the codec (host copies; either pointer may be NULL):
 * signs [dim] int8 (+1/-1) for the Walsh-Hadamard rotation, dense_q
 * [dim*dim] fp32 row-major Q (z = Q k) for the dense one; the pointer of the
 * other kind is left untouched.  ("How I built VeloxQuant-MLX", Stage 1.) */
tq_status tq_codec_export_rotation(const tq_codec *codec, int8_t *signs, float *dense_q);

/* The Lloyd-Max codebook of N(0,1) with 2^bits levels, built on the host as
 * tq_codec_create builds it ("How I built VeloxQuant-MLX", Stage 2: cell
 * boundaries at the midpoints of neighbouring centroids, each centroid the
 * conditional mean of its cell), without a device:
 *   centroids  [2^bits] fp32 ascending, RN of the fp64 solution
 *   midpoints  [2^bits - 1] fp64 (c_i + c_{i+1}) / 2 of the fp32 centroids, or NULL
 * bits in 1..8.  Errors: TQ_ERR_INVALID_ARG. */
tq_status tq_codebook_gaussian(int bits, float *centroids, double *midpoints);

/* Copies the codec's host tables out (any pointer may be NULL):
 *   signs      [dim] int8 (+1/-1), WHT codecs only (left untouched otherwise)
 *   dense_q    [dim*dim] fp32 row-major Q (z = Q k), dense codecs only
 *   centroids  [2^bits] fp32 ascending (not for bits == 16)
 *   midpoints  [2^bits - 1] fp64, (c_i + c_{i+1}) / 2
 * These are the tables the kernels use; tests compare them with tables an
 * independent implementation builds from the same (dim, bits, seed). */
tq_status tq_codec_export(const tq_codec *codec, int8_t *signs, float *dense_q, float *centroids,
                          double *midpoints);

/*
 * Encode n_vec fp16 vectors ([VQ] Stage 1 + Stage 2; [RVQ] boundary-count
 * quantisation; [VQ] The Bit-Packing Problem), bit-exactly:
 *   k_i = x_i * 2^24 exactly; S = sum k_i^2 exactly; D = RN64(sqrt(RN64(S)));
 *   WHT: w = H (s . k) exactly, code_j = #{ i : w_j > RN64(m_i * D) };
 *   dense: z_j = fp64 fma chain of Q[j][i] * k_i over ascending i,
 *          code_j = #{ i : z_j > RN64(m_i * RN64(D / RN64(sqrt(dim)))) };
 *   codes packed LSB-first (bit j*bits + t of the row = bit t of code_j);
 *   norms[v] = RN16(D * 2^-24) (the L2 norm of the fp16 vector).
 *   x       device, fp16, row v at x + v * x_row_stride (elements)
 *   codes   device, row v at codes + v * code_row_stride (bytes), each row
 *           bytes_per_vec long, written completely
 *   norms   device, fp16 [n_vec]
 * Requirements: x 4-byte aligned and x_row_stride even; codes 4-byte aligned
 * and code_row_stride a multiple of 4; bits != 16.  n_vec == 0 is a no-op.
 */
tq_status tq_encode(const tq_codec *codec, const uint16_t *x, int64_t n_vec, int64_t x_row_stride,
                    uint8_t *codes, int64_t code_row_stride, uint16_t *norms, void *stream);

/*
 * Encode a pending-token batch straight into a cache ([PR] Design, "Batch
 * recompression": pending tokens encoded together).
 *   x          device fp16 [B, n_kv_heads, T, dim] contiguous
 *   start_pos  device int32 [B]: token t of sequence b goes to position
 *              start_pos[b] + t
 *   codes      device cache [B, n_kv_heads, max_seq, bytes_per_vec]
 *   norms      device cache [B, n_kv_heads, max_seq] fp16
 *   dev_error  optional device int32 word; positions outside [0, max_seq)
 *              are skipped and TQ_DEVERR_POSITION is OR-ed into it.
 * Same arithmetic and alignment rules as tq_encode.
 */
tq_status tq_encode_append(const tq_codec *codec, const uint16_t *x, int B, int n_kv_heads, int T,
                           const int32_t *start_pos, int64_t max_seq, uint8_t *codes,
                           uint16_t *norms, int32_t *dev_error, void *stream);

/*
 * The K and the V pending-token batch of one layer encoded in one launch
 * ([PR] Design, "Batch recompression": the pending K and V tokens are
 * recompressed together), each with its own codec; otherwise exactly two
 * tq_encode_append calls (same arguments, same results, bit for bit).
 *   ck, cv           coded codecs of the same dim (bits != 16, no QJL sketch)
 *   k, v             device fp16 [B, n_kv_heads, T, dim] contiguous
 *   start_pos        device int32 [B], shared by K and V
 *   k_codes, k_norms K cache [B, n_kv_heads, max_seq, ck bytes_per_vec] / [.., max_seq] fp16
 *   v_codes, v_norms V cache, likewise with cv
 *   dev_error        optional, as for tq_encode_append
 * Errors: TQ_ERR_INVALID_ARG on a null pointer, misalignment, different dims,
 * raw or sketched codecs, or codecs of another device; nothing is enqueued then.
 */
tq_status tq_encode_append_kv(const tq_codec *ck, const tq_codec *cv, const uint16_t *k, const uint16_t *v,
                              int B, int n_kv_heads, int T, const int32_t *start_pos, int64_t max_seq,
                              uint8_t *k_codes, uint16_t *k_norms, uint8_t *v_codes, uint16_t *v_norms,
                              int32_t *dev_error, void *stream);

/*
 * Dequantise (debugging aid): out[v] = n16_v * R^T (c[codes_v] / sqrt(dim)),
 * fp32, computed with a fp32 butterfly (WHT) or fp32 Q^T product (dense).
 *   codes device [n_vec, bytes_per_vec] contiguous; norms device fp16
 *   [n_vec]; out device fp32 [n_vec, dim].  Requires codes 4-byte aligned.
 */
tq_status tq_dequant(const tq_codec *codec, const uint8_t *codes, const uint16_t *norms,
                     int64_t n_vec, float *out, void *stream);

/*
 * Bytes of device workspace tq_decode_attend needs for this shape on the
 * current device (0 on invalid arguments).  The workspace holds a device
 * error word and the split-K partial results.
 */
size_t tq_decode_attend_workspace_bytes(int B, int n_q_heads, int n_kv_heads, int64_t max_seq,
                                        int dim);

/* Zeroes a workspace on `stream`.  Required once before the first
 * tq_decode_attend that uses it (the device error word must start at zero). */
tq_status tq_workspace_init(void *workspace, size_t ws_bytes, void *stream);

/*
 * Fused single-dispatch decode attention over the packed cache ([TW]; [PR]
 * Design): one query per sequence,
 *   out[b,h] = sum_n softmax_n(scale * <q[b,h], K^[b,kvh,n]>) V^[b,kvh,n],
 *   n < seq_lens[b], kvh = h / (n_q_heads / n_kv_heads) (each KV head serves
 *   its contiguous group of query heads without expanding K/V),
 * where K^ and V^ are the dequantised cache (K^ = raw fp16 when the K codec
 * has bits == 16).  The query is rotated once, scores and P.V are computed
 * in the rotated basis against codebook values, the softmax is online and
 * split over the sequence (flash-decoding), and one inverse V rotation is
 * applied to each output head.  seq_lens[b] == 0 gives a zero output.
 * Two kernels are enqueued: the decode kernel, which writes one partial per
 * sequence split, and the combine kernel, launched with programmatic stream
 * serialization so it is resident before the decode kernel ends, which merges
 * the splits and writes `out`.
 *   ck, cv     K and V codecs: same dim; cv->bits != 16
 *   q          device fp16 [B, n_q_heads, dim]
 *   k          device: packed K codes [B, n_kv_heads, max_seq, ck bytes_per_vec]
 *              or raw fp16 K [B, n_kv_heads, max_seq, dim] (ck bits == 16)
 *   k_norms    device fp16 [B, n_kv_heads, max_seq] (NULL for raw K)
 *   v_codes    device [B, n_kv_heads, max_seq, cv bytes_per_vec]
 *   v_norms    device fp16 [B, n_kv_heads, max_seq]
 *   seq_lens   device int32 [B]; values outside [0, max_seq] are clamped and
 *              flagged with TQ_DEVERR_SEQ_LEN
 *   scale      softmax scale (1/sqrt(dim) in the usual model)
 *   out        device fp16 [B, n_q_heads, dim]
 *   workspace  device, >= tq_decode_attend_workspace_bytes(...) bytes,
 *              256-byte aligned, zeroed once by tq_workspace_init; one
 *              workspace must not be used by two calls that can overlap.
 * Requirements: n_q_heads % n_kv_heads == 0; max_seq % 8 == 0; q and every
 * cache pointer 16-byte aligned.  Errors: TQ_ERR_INVALID_ARG, TQ_ERR_UNSUPPORTED,
 * TQ_ERR_WORKSPACE, TQ_ERR_CUDA.
 */
tq_status tq_decode_attend(const tq_codec *ck, const tq_codec *cv, const uint16_t *q,
                           const void *k, const uint16_t *k_norms, const uint8_t *v_codes,
                           const uint16_t *v_norms, const int32_t *seq_lens, int B, int n_q_heads,
                           int n_kv_heads, int64_t max_seq, float scale, uint16_t *out,
                           void *workspace, size_t ws_bytes, void *stream);

/*
 * tq_decode_attend with unencoded fp16 tail tokens read in the same softmax:
 * for sequence b the attention runs over its seq_lens[b] packed tokens and then
 * tail_lens[b] raw tokens of k_tail / v_tail -- the pending tokens that wait
 * in fp16 until a batch of 64 is encoded ("add TurboQuant KV cache
 * compression", Design) or fp16 sink tokens (turboquant-mlx guide "KV cache
 * compression") -- with no separate pass over them.  The tail is scored
 * against the unrotated query and merged with the cache's softmax state in
 * the original basis (the combine kernel does it).
 *   k_tail, v_tail  device fp16 [B, n_kv_heads, max_tail, dim], 16-byte aligned
 *   tail_lens       device int32 [B]; values outside [0, max_tail] are clamped
 *                   and flagged with TQ_DEVERR_SEQ_LEN; 0 = no tail token
 *   max_tail        > 0
 * Every other argument, the workspace and the errors as tq_decode_attend.
 */
tq_status tq_decode_attend_tail(const tq_codec *ck, const tq_codec *cv, const uint16_t *q,
                                const void *k, const uint16_t *k_norms, const uint8_t *v_codes,
                                const uint16_t *v_norms, const int32_t *seq_lens, int B, int n_q_heads,
                                int n_kv_heads, int64_t max_seq, const uint16_t *k_tail,
                                const uint16_t *v_tail, const int32_t *tail_lens, int max_tail,
                                float scale, uint16_t *out, void *workspace, size_t ws_bytes,
                                void *stream);

/*
 * Attention of several query positions per sequence over the packed cache
 * (and optional fp16 tail), for chunked prefill and speculative verification
 * ("add TurboQuant KV cache compression", review of the NR0 path: a query chunk
 * holds L rows per query head, and every row reads the KV head of its query
 * head).  The sequence b is its seq_lens[b] packed tokens followed by its
 * tail_lens[b] tail tokens (none when tail_lens is NULL); the L queries of a
 * head are its last L positions, query l at position
 * seq_lens[b] + tail_lens[b] - L + l, and each attends to the tokens at
 * positions up to its own (causal).  A query before the first token gives a
 * zero row.  L == 1 is tq_decode_attend / tq_decode_attend_tail.
 * Every KV tile is dequantised once per group of up to 8 query rows (rows are
 * head-major: the G heads of a KV head times L positions).
 *   q, out    device fp16 [B, n_q_heads, L, dim] (q 16-byte aligned)
 *   L         1 .. 4096
 *   k_tail, v_tail, tail_lens, max_tail   as tq_decode_attend_tail, or all
 *             NULL / 0 for no tail
 *   workspace device, >= tq_decode_attend_multi_workspace_bytes(...) bytes,
 *             otherwise as tq_decode_attend
 * Every other argument and the errors as tq_decode_attend.
 */
size_t tq_decode_attend_multi_workspace_bytes(int B, int n_q_heads, int n_kv_heads, int L, int64_t max_seq,
                                              int dim);
tq_status tq_decode_attend_multi(const tq_codec *ck, const tq_codec *cv, const uint16_t *q, int L,
                                 const void *k, const uint16_t *k_norms, const uint8_t *v_codes,
                                 const uint16_t *v_norms, const int32_t *seq_lens, int B, int n_q_heads,
                                 int n_kv_heads, int64_t max_seq, const uint16_t *k_tail,
                                 const uint16_t *v_tail, const int32_t *tail_lens, int max_tail,
                                 float scale, uint16_t *out, void *workspace, size_t ws_bytes,
                                 void *stream);

/*
 * Keys with a QJL residual sketch (the TurboQuantProd variant, "How I built
 * VeloxQuant-MLX", Stage 3: QJL Residual Correction): a key keeps its
 * `bits`-bit MSE codes and norm, plus the sign bits of a Gaussian sketch of
 * its quantisation residual (m = dim sketch rows, 1 bit each) and the
 * residual's norm, and attention estimates <q, k> as
 *   <q, k^_MSE> + |r| sqrt(pi/2) / m * sum_j z_j <S_j, R q>
 * (unbiased; z_j = +1 / -1 for sign bit 0 / 1, R the codec's rotation).
 *
 * tq_codec_create_qjl: as tq_codec_create with bits in {2, 3, 4} (the MSE part)
 *   and a power-of-two dim; S is the Gaussian stream of seed + 2 (Box-Muller on
 *   SplitMix64, the dense rotation's generator) rounded to fp32, S[j][i].
 *   tq_codec_export_sketch copies S (host, dim * dim floats).
 * tq_encode_qjl: tq_encode of the MSE part, then per vector
 *   rho_i = RN64(w_i 2^-24 - n16 c[code_i]) rounded to fp32 (w = H (s . k),
 *   k = x 2^24 exact), sign bit j = [fp32 fma chain over i ascending of
 *   S[j][i] rho_i < 0] (LSB-first, dim / 8 bytes per vector), and
 *   rnorms = RN16(sqrt(G2 / dim)), G2 = fp64 chain over i ascending of rho_i^2.
 *     signs   device [n_vec] rows of sign_row_stride bytes (a multiple of 4,
 *             >= dim / 8), 4-byte aligned
 *     rnorms  device fp16 [n_vec]
 *   Other arguments and rules as tq_encode.
 * tq_decode_attend_qjl: tq_decode_attend with the QJL estimator for the scores;
 *   k_signs [B, n_kv_heads, max_seq, dim / 8], k_rnorms [B, n_kv_heads,
 *   max_seq] fp16 beside the MSE codes and norms (16-byte aligned for the
 *   tensor-core kernel; other alignments, and more than 8 query heads per KV
 *   head, run on the SIMT kernel).
 * A QJL codec passed to the other decode calls or to tq_cache_create is
 * rejected (their keys carry no sketch); tq_encode / tq_encode_append with it
 * write the MSE part only.
 */
tq_status tq_codec_create_qjl(int dim, int bits, uint64_t seed, tq_codec **out);
tq_status tq_codec_export_sketch(const tq_codec *codec, float *sketch);
tq_status tq_encode_qjl(const tq_codec *codec, const uint16_t *x, int64_t n_vec, int64_t x_row_stride,
                        uint8_t *codes, int64_t code_row_stride, uint16_t *norms, uint8_t *signs,
                        int64_t sign_row_stride, uint16_t *rnorms, void *stream);
tq_status tq_decode_attend_qjl(const tq_codec *ck, const tq_codec *cv, const uint16_t *q,
                               const uint8_t *k_codes, const uint16_t *k_norms, const uint8_t *k_signs,
                               const uint16_t *k_rnorms, const uint8_t *v_codes, const uint16_t *v_norms,
                               const int32_t *seq_lens, int B, int n_q_heads, int n_kv_heads,
                               int64_t max_seq, float scale, uint16_t *out, void *workspace,
                               size_t ws_bytes, void *stream);

/*
 * Two-phase KV cache of one layer for B sequences of equal length ("add
 * TurboQuant KV cache compression", Design; the update / attend / memory
 * interface of "How I built VeloxQuant-MLX"): prefill tokens are kept as raw
 * fp16 and compressed in one batch on the first decode step; after that every
 * decode step attends over the packed tokens, the pending fp16 tokens and the
 * step's new token, and appends the new token to the pending buffer in the same
 * launch; when 64 tokens are pending they are encoded into the packed cache.
 * The cache owns its device memory (allocated by tq_cache_create and
 * tq_cache_prefill, released by tq_cache_destroy); it keeps host-side counters,
 * so calls on one cache must come from one host thread in order, on one stream
 * (or streams the caller orders).  Codecs must outlive the cache.
 *   tq_cache_create   ck, cv as for tq_decode_attend; max_seq % 8 == 0 (tokens per
 *                     sequence the cache holds); min_tokens in [0, 4096]: the first
 *                     min_tokens tokens of every sequence stay fp16 for good (sink
 *                     tokens, turboquant-mlx guide "KV cache compression",
 *                     --kv-min-tokens), scored exactly in the same softmax; the
 *                     rest are packed as above.
 *   tq_cache_prefill  k, v: device fp16 [B, n_kv_heads, T, dim]; only before the
 *                     first decode step, once.
 *   tq_cache_decode   q: device fp16 [B, n_q_heads, dim]; k_new, v_new: device
 *                     fp16 [B, n_kv_heads, dim]; out: device fp16 [B, n_q_heads,
 *                     dim].  TQ_ERR_INVALID_ARG once max_seq tokens are held.
 *   tq_cache_info     tokens held (sinks included), packed, pending; bytes in use
 *                     (packed bytes of the packed tokens, 4*dim bytes per fp16
 *                     token -- sink, pending or prefill -- per KV head).
 *   tq_cache_device_error  reads and clears the device error words (syncs).
 */
typedef struct tq_cache tq_cache;
tq_status tq_cache_create(const tq_codec *ck, const tq_codec *cv, int B, int n_q_heads, int n_kv_heads,
                          int64_t max_seq, int min_tokens, tq_cache **out);
void tq_cache_destroy(tq_cache *cache);
tq_status tq_cache_prefill(tq_cache *cache, const uint16_t *k, const uint16_t *v, int T, void *stream);
tq_status tq_cache_decode(tq_cache *cache, const uint16_t *q, const uint16_t *k_new, const uint16_t *v_new,
                          float scale, uint16_t *out, void *stream);
tq_status tq_cache_info(const tq_cache *cache, int64_t *tokens, int64_t *encoded, int *pending,
                        size_t *bytes_in_use);
tq_status tq_cache_device_error(tq_cache *cache, void *stream, int *code);

/*
 * Decode attention for callers that cannot allocate device memory.  The
 * pages have no counterpart of this entry point; it exists for code that must
 * not call cudaMalloc where it attends -- work recorded into a CUDA graph it
 * does not own, plugins whose host engine owns every allocation, loops where
 * allocating is forbidden -- and so cannot provide the workspace
 * tq_decode_attend needs.
 *
 * Same arguments, arithmetic and results as tq_decode_attend, without the
 * workspace.  The split-K scratch is instead a fixed 8 MiB array in the
 * library's own device memory, one per GPU that loads the library, held until
 * the process exits.  Shapes whose workspace
 * (tq_decode_attend_workspace_bytes) would exceed 8 MiB are rejected with
 * TQ_ERR_WORKSPACE before anything is enqueued.  Nothing is allocated: no
 * cudaMalloc/cudaFree, no allocating library call; each call enqueues one
 * cudaMemsetAsync that clears the scratch's error word (the scratch keeps the
 * previous call's contents otherwise), then the decode-attention kernels.
 * The first call on a device looks up the scratch's device address
 * (cudaGetSymbolAddress, with that device current) and caches it; make that
 * first call before any stream capture.  Every call on a device shares the
 * same scratch, so calls that can overlap on the GPU (different streams
 * without ordering) race and must not be issued.  Device-side length errors
 * are clamped as in tq_decode_attend but are not reported by this entry point.
 */
tq_status tq_decode_attend_noalloc(const tq_codec *ck, const tq_codec *cv, const uint16_t *q,
                                   const void *k, const uint16_t *k_norms, const uint8_t *v_codes,
                                   const uint16_t *v_norms, const int32_t *seq_lens, int B,
                                   int n_q_heads, int n_kv_heads, int64_t max_seq, float scale,
                                   uint16_t *out, void *stream);

/*
 * Profiling builds only (libtq_timeline.so, compiled with -DTQ_TIMELINE): registers
 * a zeroed device buffer of at least 4 * 4096 * 8 * 8 bytes, 8-byte aligned, into
 * which every later decode-attention call records globaltimer stamps of its decode
 * and combine CTAs' phases, calls of even and odd index since the registration in
 * alternate halves (NULL unregisters).  The default library
 * returns TQ_ERR_UNSUPPORTED and records nothing.  No counterpart on the pages: a
 * measurement aid.
 */
tq_status tq_debug_set_timeline(void *buffer, size_t bytes);

/*
 * Reads and clears the device error word of a decode workspace (or of any
 * int32 word passed as dev_error to tq_encode_append).  Synchronises
 * `stream`.  *code receives the OR of TQ_DEVERR_* flags seen since the last
 * read; returns TQ_ERR_DEVICE_CHECK when it is non-zero.
 */
tq_status tq_get_device_error(void *error_word, void *stream, int *code);

#ifdef __cplusplus
}
#endif

#endif /* TQ_H_ */
