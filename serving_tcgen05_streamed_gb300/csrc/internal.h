// internal.h -- declarations shared by the library's translation units
// (kernel launchers, the device error words, the range table).
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "kvq.h"

namespace kvq {

// One token range of a packed store, as the kernels see it.
struct RangeDev {
    int64_t start, len, cap;
    int bits, pad_;
    uint8_t *k_codes, *v_codes;
    uint16_t *k_scales, *v_scales;
};

struct RangeTable {
    int n;
    int pad_;
    RangeDev r[KVQ_MAX_RANGES];
};

// Launchers (return a cudaError_t from the launch).
cudaError_t launch_kv_rotate_quant_pack(const void *kv, int64_t n, int hidden, int64_t ld, int group, int bits,
                                        void *k_codes, void *v_codes, void *k_scales, void *v_scales,
                                        cudaStream_t s);
cudaError_t launch_kv_unpack(const void *k_codes, const void *v_codes, const void *k_scales, const void *v_scales,
                             int64_t n, int hidden, int group, int bits, void *kv_out, int64_t ld_out,
                             cudaStream_t s);
// Returns 0 on success, a kvq_status otherwise.
int launch_qkv_proj(const void *x, const void *w, int64_t n, int hidden, int group, int64_t chunk_tokens,
                    const float *q_norm_w, const float *k_norm_w, float eps, void *q_out, const RangeTable &ranges,
                    cudaStream_t s, const float *rope_cs = nullptr, int rot_dim = 0, int sections = 3);
// partial_flags < 0: the one-call attention; otherwise a key-chunk call with
// KVQ_PARTIAL_* flags and the carried state (o_acc, lse_acc).
int launch_attention(const void *q, int64_t n_q, const RangeTable &ranges, int hidden, int group, float sm_scale,
                     int out_fp32, void *out, cudaStream_t s, int causal = 0, int64_t q_pos0 = 0,
                     int partial_flags = -1, float *o_acc = nullptr, float *lse_acc = nullptr);
cudaError_t launch_selftest_wait(uint64_t ns, cudaStream_t s);

// Device error words, one per translation unit: read-and-clear (synchronous).
cudaError_t read_clear_err_quant(unsigned int *v);
cudaError_t read_clear_err_proj(unsigned int *v);
cudaError_t read_clear_err_attn(unsigned int *v);

// Driver entry point for tensor-map encoding (resolved once through the runtime).
int encode_tmap_2d(void *map, const void *base, int dtype_bf16_or_f16, uint64_t inner, uint64_t outer,
                   uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer);

int sm_count();

// Maps a CUDA error to a kvq status; with KVQ_DEBUG=1 in the environment the
// error string is printed to stderr.
int report_cuda(cudaError_t e, const char *what);

}  // namespace kvq
