// api.cu -- the C ABI (include/kvq.h): argument validation, tensor-map
// encoding and kernel launches.  Nothing here allocates device memory.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "internal.h"

namespace kvq {

namespace {
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;
int g_sm_count[64] = {0};

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool valid_group(int g) { return g == 32 || g == 64 || g == 128; }
bool valid_hidden(int hidden) { return hidden >= 128 && hidden % 128 == 0 && hidden <= (1 << 20); }
}  // namespace

int encode_tmap_2d(void *map, const void *base, int dtype_bf16, uint64_t inner, uint64_t outer,
                   uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer) {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    });
    if (!g_encode) return 1;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_stride_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(static_cast<CUtensorMap *>(map),
                          dtype_bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                          const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? 0 : 1;
}

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    if (g_sm_count[dev] == 0) {
        int c = 0;
        if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || c <= 0) c = 1;
        g_sm_count[dev] = c;
    }
    return g_sm_count[dev];
}

int report_cuda(cudaError_t e, const char *what) {
    if (e == cudaSuccess) return KVQ_OK;
    const char *dbg = std::getenv("KVQ_DEBUG");
    if (dbg && dbg[0] == '1') std::fprintf(stderr, "kvq: %s: %s\n", what, cudaGetErrorString(e));
    return KVQ_ERR_CUDA;
}

namespace {
int check_range_table(const kvq_range *ranges, int n_ranges, int64_t n, int hidden, int group, bool need_ptrs,
                      RangeTable *out) {
    if (!ranges || n_ranges < 1 || n_ranges > KVQ_MAX_RANGES || !valid_group(group)) return KVQ_ERR_ARG;
    int64_t next = 0;
    std::memset(out, 0, sizeof(*out));
    out->n = n_ranges;
    for (int i = 0; i < n_ranges; ++i) {
        const kvq_range &r = ranges[i];
        if (r.start != next || r.len < 1 || r.cap < r.len || r.cap % KVQ_ROW_TILE) return KVQ_ERR_ARG;
        if (r.bits != 4 && r.bits != 8) return KVQ_ERR_ARG;
        if (need_ptrs && (!r.k_codes || !r.v_codes || !r.k_scales || !r.v_scales)) return KVQ_ERR_ARG;
        // codes rows are 64 or 128 bytes and move by bulk copies: 16-byte aligned; scales
        // are read and written one row (2 * 128 / group bytes) at a time, so a window
        // starting at any row of an aligned store is aligned enough
        const uintptr_t srow = 2u * static_cast<uintptr_t>(128 / group);
        if (!aligned16(r.k_codes) || !aligned16(r.v_codes) || (reinterpret_cast<uintptr_t>(r.k_scales) % srow) ||
            (reinterpret_cast<uintptr_t>(r.v_scales) % srow))
            return KVQ_ERR_ALIGN;
        next += r.len;
        RangeDev &d = out->r[i];
        d.start = r.start;
        d.len = r.len;
        d.cap = r.cap;
        d.bits = r.bits;
        d.k_codes = static_cast<uint8_t *>(r.k_codes);
        d.v_codes = static_cast<uint8_t *>(r.v_codes);
        d.k_scales = static_cast<uint16_t *>(r.k_scales);
        d.v_scales = static_cast<uint16_t *>(r.v_scales);
    }
    if (next != n) return KVQ_ERR_ARG;
    (void)hidden;
    return KVQ_OK;
}

int cuda_status(cudaError_t e) { return report_cuda(e, "launch"); }
}  // namespace

}  // namespace kvq

using namespace kvq;

namespace {
int attention_common(const void *q, int64_t n_q, const kvq_range *ranges, int n_ranges, int hidden, int group,
                     float sm_scale, int out_fp32, void *out, kvq_stream_t stream, int causal, int64_t q_pos0) {
    if (!q || !out) return KVQ_ERR_ARG;
    if (n_q < 1 || n_q > (int64_t(1) << 31) - 256 || !valid_hidden(hidden) || !valid_group(group)) return KVQ_ERR_ARG;
    if (out_fp32 != 0 && out_fp32 != 1) return KVQ_ERR_ARG;
    if (out_fp32 && out == q) return KVQ_ERR_ARG;
    if (!aligned16(q) || !aligned16(out)) return KVQ_ERR_ALIGN;
    int64_t n_kv = 0;
    if (ranges && n_ranges >= 1 && n_ranges <= KVQ_MAX_RANGES)
        for (int i = 0; i < n_ranges; ++i) n_kv += ranges[i].len;
    RangeTable t;
    int st = check_range_table(ranges, n_ranges, n_kv, hidden, group, true, &t);
    if (st) return st;
    if (causal && q_pos0 < 0) return KVQ_ERR_ARG;
    if (!(sm_scale > 0.0f)) sm_scale = 0.08838834764831845f;
    return launch_attention(q, n_q, t, hidden, group, sm_scale, out_fp32, out, reinterpret_cast<cudaStream_t>(stream),
                            causal, q_pos0);
}

int single_range(const void *k_codes, const void *v_codes, const void *k_scales, const void *v_scales, int64_t n_kv,
                 kvq_range *r) {
    if (n_kv < 1) return KVQ_ERR_ARG;
    std::memset(r, 0, sizeof(*r));
    r->start = 0;
    r->len = n_kv;
    r->cap = kvq_padded_rows(n_kv);
    r->bits = 4;
    r->k_codes = const_cast<void *>(k_codes);
    r->v_codes = const_cast<void *>(v_codes);
    r->k_scales = const_cast<void *>(k_scales);
    r->v_scales = const_cast<void *>(v_scales);
    return KVQ_OK;
}
}  // namespace

extern "C" {

const char *kvq_status_str(int status) {
    switch (status) {
        case KVQ_OK: return "ok";
        case KVQ_ERR_ARG: return "invalid argument";
        case KVQ_ERR_ALIGN: return "pointer or leading dimension not 16-byte aligned";
        case KVQ_ERR_UNSUPPORTED: return "unsupported combination";
        case KVQ_ERR_CUDA: return "CUDA error";
        case KVQ_ERR_TIMEOUT: return "device wait timed out";
        case KVQ_ERR_TOO_LARGE: return "request exceeds the library's fixed state area (KVQ_STATIC_STATE_BYTES)";
        default: return "unknown status";
    }
}

const char *kvq_version(void) { return "kvq 0.1 (sm_103a)"; }

int64_t kvq_padded_rows(int64_t n) {
    if (n <= 0) return 0;
    return (n + KVQ_ROW_TILE - 1) / KVQ_ROW_TILE * KVQ_ROW_TILE;
}

size_t kvq_codes_bytes(int64_t cap, int hidden, int bits) {
    if (cap <= 0 || !valid_hidden(hidden) || (bits != 4 && bits != 8)) return 0;
    return static_cast<size_t>(hidden / 128) * static_cast<size_t>(cap) * (128u * bits / 8u);
}

size_t kvq_scales_bytes(int64_t cap, int hidden, int group) {
    if (cap <= 0 || !valid_hidden(hidden) || !valid_group(group)) return 0;
    return static_cast<size_t>(hidden / 128) * static_cast<size_t>(cap) * static_cast<size_t>(128 / group) * 2u;
}

int kv_rotate_quant_pack(const void *kv, int64_t n, int hidden, int64_t ld_kv, int group, int bits, void *k_codes,
                         void *v_codes, void *k_scales, void *v_scales, kvq_stream_t stream) {
    if (!kv || !k_codes || !v_codes || !k_scales || !v_scales) return KVQ_ERR_ARG;
    if (n < 1 || n > (int64_t(1) << 31) || !valid_hidden(hidden) || !valid_group(group) || (bits != 4 && bits != 8))
        return KVQ_ERR_ARG;
    if (ld_kv < 2 * static_cast<int64_t>(hidden)) return KVQ_ERR_ARG;
    if (!aligned16(kv) || ld_kv % 8 || !aligned16(k_codes) || !aligned16(v_codes) || !aligned16(k_scales) ||
        !aligned16(v_scales))
        return KVQ_ERR_ALIGN;
    return cuda_status(launch_kv_rotate_quant_pack(kv, n, hidden, ld_kv, group, bits, k_codes, v_codes, k_scales,
                                                   v_scales, reinterpret_cast<cudaStream_t>(stream)));
}

int kv_unpack(const void *k_codes, const void *v_codes, const void *k_scales, const void *v_scales, int64_t n,
              int hidden, int group, int bits, void *kv_out, int64_t ld_out, kvq_stream_t stream) {
    if (!kv_out || !k_codes || !v_codes || !k_scales || !v_scales) return KVQ_ERR_ARG;
    if (n < 1 || n > (int64_t(1) << 31) || !valid_hidden(hidden) || !valid_group(group) || (bits != 4 && bits != 8))
        return KVQ_ERR_ARG;
    if (ld_out < 2 * static_cast<int64_t>(hidden)) return KVQ_ERR_ARG;
    if (!aligned16(kv_out) || ld_out % 8 || !aligned16(k_codes) || !aligned16(v_codes) || !aligned16(k_scales) ||
        !aligned16(v_scales))
        return KVQ_ERR_ALIGN;
    return cuda_status(launch_kv_unpack(k_codes, v_codes, k_scales, v_scales, n, hidden, group, bits, kv_out, ld_out,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

int streamed_qkv_proj_mixed(const void *x, const void *w_qkv, int64_t n, int hidden, int group,
                            int64_t chunk_tokens, const float *q_norm_w, const float *k_norm_w, float eps,
                            void *q_out, const kvq_range *ranges, int n_ranges, kvq_stream_t stream) {
    return streamed_qkv_proj_ex(x, w_qkv, n, hidden, group, chunk_tokens, q_norm_w, k_norm_w, eps, nullptr, 0,
                                KVQ_SECTION_Q | KVQ_SECTION_KV, q_out, ranges, n_ranges, stream);
}

int streamed_qkv_proj_ex(const void *x, const void *w_qkv, int64_t n, int hidden, int group, int64_t chunk_tokens,
                         const float *q_norm_w, const float *k_norm_w, float eps, const float *rope_cs, int rot_dim,
                         int sections, void *q_out, const kvq_range *ranges, int n_ranges, kvq_stream_t stream) {
    if (sections < 1 || sections > 3) return KVQ_ERR_ARG;
    const bool want_q = sections & KVQ_SECTION_Q, want_kv = sections & KVQ_SECTION_KV;
    if (rope_cs && rot_dim != 64 && rot_dim != 128) return KVQ_ERR_UNSUPPORTED;
    if (rope_cs && !aligned16(rope_cs)) return KVQ_ERR_ALIGN;
    if (!x || !w_qkv || (want_q && !q_out)) return KVQ_ERR_ARG;
    if (n < 1 || n > (int64_t(1) << 31) - 256 || !valid_hidden(hidden) || !valid_group(group) || chunk_tokens < 0)
        return KVQ_ERR_ARG;
    if (!(eps >= 0.0f)) return KVQ_ERR_ARG;
    if (want_q && x == q_out) return KVQ_ERR_ARG;
    if (!aligned16(x) || !aligned16(w_qkv) || (want_q && !aligned16(q_out))) return KVQ_ERR_ALIGN;
    if ((q_norm_w && (reinterpret_cast<uintptr_t>(q_norm_w) & 3u)) ||
        (k_norm_w && (reinterpret_cast<uintptr_t>(k_norm_w) & 3u)))
        return KVQ_ERR_ALIGN;
    RangeTable t;
    std::memset(&t, 0, sizeof(t));
    if (want_kv) {
        const int st = check_range_table(ranges, n_ranges, n, hidden, group, true, &t);
        if (st) return st;
    }
    return launch_qkv_proj(x, w_qkv, n, hidden, group, chunk_tokens, q_norm_w, k_norm_w, eps,
                           want_q ? q_out : nullptr, t, reinterpret_cast<cudaStream_t>(stream), rope_cs, rot_dim,
                           sections);
}

int streamed_qkv_proj(const void *x, const void *w_qkv, int64_t n, int hidden, int group, int64_t chunk_tokens,
                      const float *q_norm_w, const float *k_norm_w, float eps, void *q_out, void *k_codes,
                      void *v_codes, void *k_scales, void *v_scales, kvq_stream_t stream) {
    kvq_range r;
    std::memset(&r, 0, sizeof(r));
    r.start = 0;
    r.len = n;
    r.cap = kvq_padded_rows(n);
    r.bits = 4;
    r.k_codes = k_codes;
    r.v_codes = v_codes;
    r.k_scales = k_scales;
    r.v_scales = v_scales;
    int st = streamed_qkv_proj_mixed(x, w_qkv, n, hidden, group, chunk_tokens, q_norm_w, k_norm_w, eps, q_out, &r, 1,
                                     stream);
    if (st || r.cap == n) return st;
    // the whole store is the caller's: its pad rows n .. cap-1 of every head become zero
    const size_t heads = static_cast<size_t>(hidden / 128), pad = static_cast<size_t>(r.cap - n);
    const size_t cb = 64, sb = 2 * static_cast<size_t>(128 / group);  // bytes per row: codes, scales
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    for (void *base : {k_codes, v_codes})
        if (e == cudaSuccess)
            e = cudaMemset2DAsync(static_cast<uint8_t *>(base) + n * cb, r.cap * cb, 0, pad * cb, heads, s);
    for (void *base : {k_scales, v_scales})
        if (e == cudaSuccess)
            e = cudaMemset2DAsync(static_cast<uint8_t *>(base) + n * sb, r.cap * sb, 0, pad * sb, heads, s);
    return cuda_status(e);
}


int packed_kv_attention_mixed(const void *q, int64_t n_q, const kvq_range *ranges, int n_ranges, int hidden,
                              int group, float sm_scale, int out_fp32, void *out, kvq_stream_t stream) {
    return attention_common(q, n_q, ranges, n_ranges, hidden, group, sm_scale, out_fp32, out, stream, 0, 0);
}

int packed_kv_attention(const void *q, int64_t n_q, const void *k_codes, const void *v_codes, const void *k_scales,
                        const void *v_scales, int64_t n_kv, int hidden, int group, float sm_scale, int out_fp32,
                        void *out, kvq_stream_t stream) {
    kvq_range r;
    const int st = single_range(k_codes, v_codes, k_scales, v_scales, n_kv, &r);
    if (st) return st;
    return attention_common(q, n_q, &r, 1, hidden, group, sm_scale, out_fp32, out, stream, 0, 0);
}

int packed_kv_attention_causal(const void *q, int64_t n_q, int64_t q_pos0, const void *k_codes, const void *v_codes,
                               const void *k_scales, const void *v_scales, int64_t n_kv, int hidden, int group,
                               float sm_scale, int out_fp32, void *out, kvq_stream_t stream) {
    kvq_range r;
    const int st = single_range(k_codes, v_codes, k_scales, v_scales, n_kv, &r);
    if (st) return st;
    return attention_common(q, n_q, &r, 1, hidden, group, sm_scale, out_fp32, out, stream, 1, q_pos0);
}

int packed_kv_attention_partial(const void *q, int64_t n_q, const kvq_range *ranges, int n_ranges, int hidden,
                                int group, float sm_scale, int flags, float *o_acc, float *lse_acc, int out_fp32,
                                void *out, kvq_stream_t stream) {
    if (flags < 0 || flags > (KVQ_PARTIAL_MERGE | KVQ_PARTIAL_FINAL)) return KVQ_ERR_ARG;
    const bool merge = flags & KVQ_PARTIAL_MERGE, final = flags & KVQ_PARTIAL_FINAL;
    if (!q || (final && !out)) return KVQ_ERR_ARG;
    if (merge || !final) {  // the state is read (merge) or written (not final)
        if (!o_acc || !lse_acc) return KVQ_ERR_ARG;
        const void *st[2] = {o_acc, lse_acc};
        for (const void *a : st)
            if (a == q || (final && a == out)) return KVQ_ERR_ARG;
        if (!aligned16(o_acc) || !aligned16(lse_acc)) return KVQ_ERR_ALIGN;
    }
    if (n_q < 1 || n_q > (int64_t(1) << 31) - 256 || !valid_hidden(hidden) || !valid_group(group)) return KVQ_ERR_ARG;
    if (out_fp32 != 0 && out_fp32 != 1) return KVQ_ERR_ARG;
    if (final && out_fp32 && out == q) return KVQ_ERR_ARG;
    if (!aligned16(q) || (final && !aligned16(out))) return KVQ_ERR_ALIGN;
    int64_t n_kv = 0;
    if (ranges && n_ranges >= 1 && n_ranges <= KVQ_MAX_RANGES)
        for (int i = 0; i < n_ranges; ++i) n_kv += ranges[i].len;
    RangeTable t;
    const int st = check_range_table(ranges, n_ranges, n_kv, hidden, group, true, &t);
    if (st) return st;
    if (!(sm_scale > 0.0f)) sm_scale = 0.08838834764831845f;
    return launch_attention(q, n_q, t, hidden, group, sm_scale, out_fp32, final ? out : nullptr,
                            reinterpret_cast<cudaStream_t>(stream), 0, 0, flags, o_acc, lse_acc);
}

int kvq_device_status(kvq_stream_t stream) {
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return KVQ_ERR_CUDA;
    unsigned int a = 0, b = 0, c = 0;
    if (read_clear_err_quant(&a) != cudaSuccess || read_clear_err_proj(&b) != cudaSuccess ||
        read_clear_err_attn(&c) != cudaSuccess)
        return KVQ_ERR_CUDA;
    return (a | b | c) ? KVQ_ERR_TIMEOUT : KVQ_OK;
}

int kvq_selftest_wait_timeout(uint64_t ns, kvq_stream_t stream) {
    if (ns == 0 || ns > 1000000000ull) return KVQ_ERR_ARG;
    return cuda_status(launch_selftest_wait(ns, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
