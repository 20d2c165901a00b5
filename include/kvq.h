/*
 * kvq.h -- C ABI of the streamed QKV projection with rotated, group-scaled,
 * packed low-bit K/V, and of the attention that reads that packed K/V.
 *
 * The operations follow the comfy-kitchen feature request "Streamed QKV
 * Projection and Packed Low-Bit K/V Support for Extreme Long-Sequence
 * Attention" (section "Proposed backend capability": a streamed/tiled QKV
 * GEMM keeps Q in BF16/FP16 and sends K and V through rotate -> quantise ->
 * packed 4-bit storage; attention consumes Q and the packed K/V and decodes
 * K/V tile by tile; section "Dense fallback is important": no full BF16
 * expansion of K/V; section "Mixed precision for conditioning": chosen token
 * ranges at INT8).  The rotation, scaling and rounding conventions follow
 * vram_lab.py ("VRAM Lab"): `_hadamard` (Sylvester Hadamard / sqrt(n)),
 * `_fq_int4` (group absmax / 7, round half to even), `_Int8KV` (rotated INT8,
 * absmax / 127; rotated-basis identities q.k = (qH).(kH), P.V = (P.(VH)).H^T).
 *
 * Conventions shared by every call
 *  - head_dim is 128; hidden = heads * 128.
 *  - H is the 128x128 Sylvester Hadamard matrix divided by sqrt(128); "rotate"
 *    means x -> x.H computed as the fast Walsh-Hadamard transform with
 *    butterfly strides 1, 2, ..., 64 in fp32, then one multiply by
 *    fp32(1/sqrt(128)).  H is symmetric, so un-rotating is the same operation.
 *  - Quantiser (per head, per group of `group` in {32, 64, 128} elements of
 *    the rotated vector y): amax = max|y|; s = fp16_rn(amax / Q) with Q = 7
 *    (bits 4) or 127 (bits 8); code = clamp(rint(y / float(s)), -Q, Q) (ties
 *    to even, IEEE division), or 0 when s == 0.
 *  - Packed store ("store"), one per K and one per V, HEAD-MAJOR:
 *      codes  uint8 [heads][cap][128*bits/8]  (bits 4: element 2i in the low
 *             nibble of byte i, 2i+1 in the high nibble, two's complement;
 *             bits 8: one int8 per element)
 *      scales fp16  [heads][cap][128/group]
 *    For the single-precision calls cap = kvq_padded_rows(n) (n rounded up to
 *    a multiple of 128); rows n..cap-1 are written as zero codes and scales.
 *  - Q and attention outputs are token-major [n][hidden] with head h at
 *    columns h*128 .. h*128+127; BF16 unless stated.
 *  - All device pointers are caller-owned and must be 16-byte aligned, except
 *    the scales pointers of a range table (kvq_range), which need only the
 *    alignment of one scales row (2 * 128 / group bytes), so that a range may
 *    be a window starting at any row of a store.  The library allocates no
 *    device memory and keeps no workspace.
 *  - Calls are asynchronous on `stream` (NULL = the legacy default stream)
 *    and never synchronise.  Argument errors are reported before any launch;
 *    launch failures return KVQ_ERR_CUDA.  Every device-side wait is bounded:
 *    a wait that runs out sets a device error word that kvq_device_status()
 *    reads, and the kernel returns early (its outputs are then undefined).
 *  - Inputs must be finite, and rotated Q, K and V values must lie within the
 *    fp16 range (|v| < 65504): the attention computes on fp16 operands.
 *  - Score range of the attention: the dequantised K^ operand is rounded to
 *    fp16 (11 significant bits), which moves a score s = sm_scale q.k^ by
 *    about |s| 2^-12 and an output by that much of |v|.  The parity bar
 *    (max-abs 1e-2, relative L2 5e-3 against the exact attention on the same
 *    packed K/V) is met for row maxima |s| up to about 35 (measured; Q and K
 *    RMS-normalised per head reach about 14); at |s| ~ 70 the max-abs error
 *    reaches about 1.2e-2 while the relative L2 error stays near 1e-3.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define KVQ_API __attribute__((visibility("default")))
#else
#define KVQ_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream handle (the same object as cudaStream_t / CUstream). */
typedef struct CUstream_st *kvq_stream_t;

enum kvq_status {
    KVQ_OK = 0,
    KVQ_ERR_ARG = 1,         /* a size, count or pointer argument is invalid */
    KVQ_ERR_ALIGN = 2,       /* a pointer or leading dimension is not 16-byte aligned */
    KVQ_ERR_UNSUPPORTED = 3, /* a valid but unsupported combination (a RoPE width other than 64 or 128) */
    KVQ_ERR_CUDA = 4,        /* a CUDA runtime or driver call failed */
    KVQ_ERR_TIMEOUT = 5,     /* a device-side wait ran out (see kvq_device_status) */
    KVQ_ERR_TOO_LARGE = 6    /* the request needs more than the library's fixed state area */
};

#define KVQ_HEAD_DIM 128
#define KVQ_ROW_TILE 128
#define KVQ_MAX_RANGES 16

/* Human-readable name of a status code (static storage). */
KVQ_API const char *kvq_status_str(int status);

/* Library version string (static storage). */
KVQ_API const char *kvq_version(void);

/* ---------------------------------------------------------------- sizes
 * Byte sizes of the packed store ("Potential reduction": Q BF16 plus 4-bit
 * K and V, plus quantisation metadata).  Pure host functions. */

/* n rounded up to a multiple of KVQ_ROW_TILE (the row capacity `cap`). */
KVQ_API int64_t kvq_padded_rows(int64_t n);
/* Bytes of ONE codes array (K or V): heads * cap * 128 * bits / 8. */
KVQ_API size_t kvq_codes_bytes(int64_t cap, int hidden, int bits);
/* Bytes of ONE scales array (K or V): heads * cap * (128 / group) * 2. */
KVQ_API size_t kvq_scales_bytes(int64_t cap, int hidden, int group);

/* ---------------------------------------------------------------- a1: rotate + quantise + pack
 * ("Quality-oriented low-bit format": Hadamard rotation, per-group scaling.)
 * kv: BF16 [n][ld_kv] device; K = columns [0, hidden), V = [hidden, 2*hidden).
 * Writes the K and V stores (cap = kvq_padded_rows(n), pad rows zeroed).
 * group in {32, 64, 128}; bits in {4, 8}.  ld_kv >= 2*hidden, a multiple of 8.
 * Codes and scales are bit-exact with the conventions above.  Rows and code
 * arrays on 32-byte boundaries (kv, ld_kv * 2, k_codes, v_codes) take 32-byte
 * loads and stores, which run faster; other valid layouts give the same bytes. */
KVQ_API int kv_rotate_quant_pack(const void *kv, int64_t n, int hidden, int64_t ld_kv, int group, int bits, void *k_codes,
                         void *v_codes, void *k_scales, void *v_scales, kvq_stream_t stream);

/* ---------------------------------------------------------------- a1b: unpack (diagnostic)
 * Inverse of a1: dequantise (code * float(s)), un-rotate, round to BF16 into
 * kv_out [n][ld_out] (K then V, as a1's input).  This materialises BF16 K/V
 * by design; the attention never calls it.  An output on 32-byte boundaries
 * (kv_out, ld_out * 2) takes 32-byte stores, which run faster; other valid
 * layouts give the same bytes. */
KVQ_API int kv_unpack(const void *k_codes, const void *v_codes, const void *k_scales, const void *v_scales, int64_t n,
              int hidden, int group, int bits, void *kv_out, int64_t ld_out, kvq_stream_t stream);

/* ---------------------------------------------------------------- a2: streamed fused QKV projection
 * ("Proposed backend capability": streamed/tiled QKV GEMM; Q -> BF16,
 * K and V -> rotate + quantise -> packed 4-bit.)
 * x: BF16 [n][hidden]; w_qkv: BF16 [3*hidden][hidden] (rows [0,C) produce Q,
 * [C,2C) K, [2C,3C) V; head h = 128 consecutive rows within each block).
 * For each token: acc = x . w_qkv^T in fp32 on the tensor cores, then per head
 *   Q: [RMSNorm with q_norm_w] -> rotate -> BF16 (round to nearest even) into q_out [n][hidden]
 *   K: [RMSNorm with k_norm_w] -> rotate -> quantise/pack (bits 4) into the K store
 *   V: rotate -> quantise/pack (bits 4) into the V store
 * RMSNorm is v * (1/sqrt(mean(v^2) + eps)) * w over the head's 128 values,
 * w a [128] fp32 device vector (NULL = no normalisation).  The rotation takes
 * the fp32 accumulator directly.  Tokens are processed chunk by chunk in
 * chunk_tokens-row chunks (0 = one chunk); results do not depend on the
 * chunk size.  No [n][3*hidden] tensor and no BF16 K/V exist at any time.
 * The stores' pad rows n .. kvq_padded_rows(n)-1 are set to zero.
 * q_out must not alias x. */
KVQ_API int streamed_qkv_proj(const void *x, const void *w_qkv, int64_t n, int hidden, int group, int64_t chunk_tokens,
                      const float *q_norm_w, const float *k_norm_w, float eps, void *q_out, void *k_codes,
                      void *v_codes, void *k_scales, void *v_scales, kvq_stream_t stream);

/* ---------------------------------------------------------------- a4: packed-K/V attention
 * ("Proposed backend capability": attention reads Q BF16 and packed INT4
 * K/V, decoding K/V tile by tile; "Dense fallback is important".)
 * q: BF16 [n_q][hidden], ROTATED basis (as written by streamed_qkv_proj).
 * K/V stores: bits 4, cap = kvq_padded_rows(n_kv).  Non-causal softmax over
 * all n_kv keys with scale sm_scale (<= 0 selects 1/sqrt(128)), then the
 * output is un-rotated: out[i] = (sum_j p_ij v^_j / sum_j p_ij) . H, head by head.
 * out: [n_q][hidden], BF16 (out_fp32 = 0) or fp32 (out_fp32 = 1).  With BF16
 * output, out may equal q (each output row depends only on its own query
 * row and every row is read before it is written by the same CTA).  */
KVQ_API int packed_kv_attention(const void *q, int64_t n_q, const void *k_codes, const void *v_codes, const void *k_scales,
                        const void *v_scales, int64_t n_kv, int hidden, int group, float sm_scale, int out_fp32,
                        void *out, kvq_stream_t stream);

/* Causal form of packed_kv_attention.  The pages name a general packed-K/V
 * attention primitive ("Proposed backend capability"); the causal form is
 * the usual prefix mask.  Query row i sits at key position q_pos0 + i and
 * attends keys j <= q_pos0 + i (j < n_kv); q_pos0 >= 0, so every row sees key
 * 0.  A query chunk [a, a + m) of a sequence attends with q pointing at row a
 * and q_pos0 = a, and gives the rows of the one-call result.  Arguments,
 * layouts, aliasing and errors as packed_kv_attention, plus KVQ_ERR_ARG for
 * q_pos0 < 0.  Work is about half of the unmasked call when q_pos0 = 0 and
 * n_q = n_kv (key tiles past a CTA pair's last row are skipped). */
KVQ_API int packed_kv_attention_causal(const void *q, int64_t n_q, int64_t q_pos0, const void *k_codes,
                               const void *v_codes, const void *k_scales, const void *v_scales, int64_t n_kv,
                               int hidden, int group, float sm_scale, int out_fp32, void *out,
                               kvq_stream_t stream);

/* ---------------------------------------------------------------- a6: mixed precision by token range
 * ("Mixed precision for conditioning": text / reference / audio ranges at
 * INT8, generated video at rotated INT4.)  Every range holds its own K and V
 * stores of `bits` (4 or 8) with row capacity `cap` (>= len, the head stride
 * of its arrays); token t of the sequence is row t - start of the range that
 * holds it.  Ranges must be given in order and tile [0, n) exactly, at most
 * KVQ_MAX_RANGES of them.  INT8 ranges use the same rotation, so Q and the
 * output need no per-range handling.  The projection writes rows 0 .. len-1
 * of every range and nothing past them (the attention never reads rows past
 * len as keys), so a range may be a window into a larger store: pointers
 * advanced by the window's first row, cap the store's head stride. */
typedef struct kvq_range {
    int64_t start;
    int64_t len;
    int64_t cap;
    int32_t bits;
    int32_t reserved;
    void *k_codes;
    void *v_codes;
    void *k_scales;
    void *v_scales;
} kvq_range;

KVQ_API int streamed_qkv_proj_mixed(const void *x, const void *w_qkv, int64_t n, int hidden, int group,
                            int64_t chunk_tokens, const float *q_norm_w, const float *k_norm_w, float eps,
                            void *q_out, const kvq_range *ranges, int n_ranges, kvq_stream_t stream);

/* ---------------------------------------------------------------- next rows f2, f3: RoPE, sections
 * streamed_qkv_proj_mixed with two additions.
 *
 * RoPE (vram_lab.py `_norm_rope`: "fused RMSNorm + split-half RoPE"): a
 * split-half rotary position embedding of Q and K, applied after the RMSNorm
 * and before the Hadamard rotation.  rope_cs: fp32, rot_dim floats per token
 * row of x, row t at rope_cs + t*rot_dim, holding the pairs (cos_i, sin_i),
 * i < rot_dim/2; with H = rot_dim/2, dims i and i+H of each head become
 * x_i cos_i - x_{i+H} sin_i and x_{i+H} cos_i + x_i sin_i, dims past rot_dim
 * stay.  The table is the caller's (positions and frequencies are not the
 * library's business), read only, 16-byte aligned.  rot_dim 64 or 128, else
 * KVQ_ERR_UNSUPPORTED; rope_cs == NULL means no RoPE.
 *
 * Sections (vram_lab.py's two phases: K/V of every token first, then Q
 * recomputed per query chunk): KVQ_SECTION_Q computes and writes Q only (the
 * GEMM walks W's first hidden rows; ranges may be NULL), KVQ_SECTION_KV the K/V
 * stores only (W's last 2*hidden rows; q_out may be NULL), both = the full
 * projection.  Each section's bytes are those of the full call.
 *
 * Other arguments and errors as streamed_qkv_proj_mixed; KVQ_ERR_ARG for
 * sections outside 1..3. */
#define KVQ_SECTION_Q 1
#define KVQ_SECTION_KV 2
KVQ_API int streamed_qkv_proj_ex(const void *x, const void *w_qkv, int64_t n, int hidden, int group,
                         int64_t chunk_tokens, const float *q_norm_w, const float *k_norm_w, float eps,
                         const float *rope_cs, int rot_dim, int sections, void *q_out, const kvq_range *ranges,
                         int n_ranges, kvq_stream_t stream);

KVQ_API int packed_kv_attention_mixed(const void *q, int64_t n_q, const kvq_range *ranges, int n_ranges, int hidden,
                              int group, float sm_scale, int out_fp32, void *out, kvq_stream_t stream);

/* ---------------------------------------------------------------- next row f3: attention over key chunks
 * vram_lab.py ("VRAM Lab"), `_blockwise_attention_q` and `_online_combine`:
 * attention of a query chunk against K/V blocks, each block's normalised
 * output and log-sum-exp merged into an fp32 accumulator, the output
 * un-rotated once at the end; and the module notes on the streamed block,
 * which plan K/V staged in host memory and streamed to the device block by
 * block.  This call attends ONE key chunk of a packed store and carries the
 * state between calls, so the store never needs to be on the device whole.
 *
 * q, n_q, hidden, group, sm_scale: as packed_kv_attention.  ranges /
 * n_ranges: the key chunk as a range table (as packed_kv_attention_mixed; a
 * window of a larger store is a range whose pointers start at the window's
 * first row and whose cap is the store's head stride; starts tile [0, chunk)).
 * The carried state, caller-owned, fp32, 16-byte aligned, not aliasing q or out:
 *   o_acc   [n_q][hidden]  normalised output over the keys seen so far, in the
 *                          rotated basis (not un-rotated)
 *   lse_acc [n_q][heads]   natural log of sum_j exp(s_j) over those keys,
 *                          s_j = sm_scale * q . k^_j
 * flags:
 *   0                  start: the state becomes this chunk's (o, lse)
 *   KVQ_PARTIAL_MERGE  merge this chunk into the state:
 *                        new = log(exp(lse_acc) + exp(lse)),
 *                        o_acc = o_acc exp(lse_acc - new) + o exp(lse - new)
 *   | KVQ_PARTIAL_FINAL  write the (merged) result, un-rotated, to out
 *                      ([n_q][hidden], BF16 or fp32 by out_fp32); out may
 *                      equal q for BF16 output.  Without FINAL, out is unused.
 * FINAL | MERGE merges through o_acc, whose contents are unspecified after
 * the call (lse_acc is left as it was).  FINAL alone touches no state, so
 * o_acc / lse_acc may be NULL then (it is packed_kv_attention_mixed).
 * Each row's result depends only on its own query row and on the order of
 * the chunks, never on how the queries are chunked.
 * Errors: as packed_kv_attention_mixed, plus KVQ_ERR_ARG for flags outside
 * 0..3, a state pointer the flags need that is NULL or aliases q / out, and
 * out NULL with FINAL; KVQ_ERR_ALIGN for a state pointer not 16-byte aligned. */
#define KVQ_PARTIAL_MERGE 1
#define KVQ_PARTIAL_FINAL 2
KVQ_API int packed_kv_attention_partial(const void *q, int64_t n_q, const kvq_range *ranges, int n_ranges,
                                        int hidden, int group, float sm_scale, int flags, float *o_acc,
                                        float *lse_acc, int out_fp32, void *out, kvq_stream_t stream);

/* ---------------------------------------------------------------- the key-chunk attention without caller memory
 * This call has no counterpart on the pages; it serves callers that cannot
 * allocate device memory.  Code that runs inside a host owning all device
 * memory (a server's or framework's pool, a plugin with a fixed budget) and
 * given no workspace, or on a path where cudaMalloc is not allowed because it
 * may synchronise the device, cannot provide the o_acc / lse_acc buffers of
 * packed_kv_attention_partial.  This variant keeps that state in a fixed area
 * of device memory owned by the library: KVQ_STATIC_STATE_BYTES (16 MiB),
 * reserved on every device that loads the library and held until the process
 * exits.  It calls no cudaMalloc, cudaFree or other allocating routine.
 *
 * Arguments, flags and results are those of packed_kv_attention_partial
 * without o_acc / lse_acc; the caller still passes Q, the key chunk (ranges)
 * and, with KVQ_PARTIAL_FINAL, the output.  A query set of n_q rows needs
 * n_q * (hidden + hidden / 128) * 4 bytes of state; larger requests return
 * KVQ_ERR_TOO_LARGE (at hidden 7168: at most 580 query rows).
 *
 * The state area is one per device and shared by every call: a call without
 * KVQ_PARTIAL_MERGE overwrites it (nothing needs clearing), and a later call
 * with KVQ_PARTIAL_MERGE continues from whatever the last call left.  So one
 * sequence of calls (start, merges, final) runs at a time per device: calls
 * that overlap on the GPU (two sequences on different streams) race on the
 * area.  The first call on a device looks up the area's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  Errors as packed_kv_attention_partial, plus
 * KVQ_ERR_TOO_LARGE. */
#define KVQ_STATIC_STATE_BYTES (16u << 20)
KVQ_API int packed_kv_attention_partial_static(const void *q, int64_t n_q, const kvq_range *ranges, int n_ranges,
                                               int hidden, int group, float sm_scale, int flags, int out_fp32,
                                               void *out, kvq_stream_t stream);

/* ---------------------------------------------------------------- device status
 * Waits for `stream`, then returns KVQ_OK, or KVQ_ERR_TIMEOUT if a bounded
 * device wait of any kernel of this library ran out since the last call
 * (and clears the record), or KVQ_ERR_CUDA if the stream reports an error. */
KVQ_API int kvq_device_status(kvq_stream_t stream);

/* Self-test of the bounded wait: launches one block that waits on an
 * mbarrier nothing ever arrives at, bounded by `ns` nanoseconds (at most
 * 1e9); the wait runs out, the block records KVQ_ERR_TIMEOUT and returns.
 * A following kvq_device_status() reports it.  Used by the test suite to
 * show that a wait which cannot complete ends with a status, not a hang. */
KVQ_API int kvq_selftest_wait_timeout(uint64_t ns, kvq_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* KVQ_H */
