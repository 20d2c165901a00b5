// kv_quant.cu -- standalone rotate + quantise + pack of BF16 K/V into the
// head-major packed store, and its inverse (unpack, a diagnostic).
//
// The comfy-kitchen feature request ("Quality-oriented low-bit format")
// asks for fixed-width rotated INT4 with per-group scaling; vram_lab.py's
// `_hadamard`, `_fq_int4` and `_Int8KV` fix the rotation and rounding rules
// implemented in quant.cuh.
//
// Both kernels are HBM-bound: per token they move 2*hidden*2 bytes of BF16
// and 2*hidden*(bits/8 + 2/group) bytes of codes and scales.  One warp owns
// one 128-wide head vector (4 consecutive elements per lane); a block of 8
// warps covers 8 head slots x 32 tokens, loading 8 tokens per warp before
// computing so that enough bytes are in flight.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"
#include "quant.cuh"

namespace kvq {
namespace {

__device__ unsigned int g_err_quant;

constexpr int kWarps = 8;
constexpr int kTokensPerBlock = 32;
constexpr int kBatch = 8;

__device__ __forceinline__ uint2 ld_nc_u2(const void *p) {
    uint2 v;
    asm volatile("ld.global.nc.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

template <int GROUP, int BITS>
__global__ void __launch_bounds__(kWarps * 32) rotate_quant_pack_kernel(const __nv_bfloat16 *__restrict__ kv,
                                                                         int64_t n, int64_t cap, int heads,
                                                                         int64_t ld, uint8_t *__restrict__ k_codes,
                                                                         uint8_t *__restrict__ v_codes,
                                                                         uint16_t *__restrict__ k_scales,
                                                                         uint16_t *__restrict__ v_scales) {
    constexpr int CB = 128 * BITS / 8;  // code bytes per head row
    constexpr int SG = 128 / GROUP;     // scales per head row
    constexpr int LANES_PER_GROUP = GROUP / 4;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hs = blockIdx.y * kWarps + warp;  // head slot: K heads then V heads
    if (hs >= 2 * heads) return;
    const int kvi = hs >= heads ? 1 : 0;
    const int h = hs - kvi * heads;
    uint8_t *codes = (kvi ? v_codes : k_codes) + static_cast<int64_t>(h) * cap * CB;
    uint16_t *scales = (kvi ? v_scales : k_scales) + static_cast<int64_t>(h) * cap * SG;
    const __nv_bfloat16 *src = kv + static_cast<int64_t>(hs) * 128 + lane * 4;
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kTokensPerBlock;

#pragma unroll 1
    for (int tb = 0; tb < kTokensPerBlock; tb += kBatch) {
        uint2 raw[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int64_t t = t0 + tb + u;
            raw[u] = (t < n) ? ld_nc_u2(src + t * ld) : make_uint2(0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int64_t t = t0 + tb + u;
            float v[4];
            v[0] = __uint_as_float(raw[u].x << 16);
            v[1] = __uint_as_float(raw[u].x & 0xFFFF0000u);
            v[2] = __uint_as_float(raw[u].y << 16);
            v[3] = __uint_as_float(raw[u].y & 0xFFFF0000u);
            rotate128_warp(v, lane);
            uint16_t sbits;
            const uint32_t packed = quant128_warp<GROUP, BITS>(v, sbits);
            if (t < cap) {
                if constexpr (BITS == 4) {
                    reinterpret_cast<uint16_t *>(codes + t * CB)[lane] = static_cast<uint16_t>(packed);
                } else {
                    reinterpret_cast<uint32_t *>(codes + t * CB)[lane] = packed;
                }
                if ((lane % LANES_PER_GROUP) == 0) scales[t * SG + lane / LANES_PER_GROUP] = sbits;
            }
        }
    }
}

template <int GROUP, int BITS>
__global__ void __launch_bounds__(kWarps * 32) unpack_kernel(const uint8_t *__restrict__ k_codes,
                                                              const uint8_t *__restrict__ v_codes,
                                                              const uint16_t *__restrict__ k_scales,
                                                              const uint16_t *__restrict__ v_scales, int64_t n,
                                                              int64_t cap, int heads, __nv_bfloat16 *__restrict__ out,
                                                              int64_t ld_out) {
    constexpr int CB = 128 * BITS / 8;
    constexpr int SG = 128 / GROUP;
    constexpr int LANES_PER_GROUP = GROUP / 4;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hs = blockIdx.y * kWarps + warp;
    if (hs >= 2 * heads) return;
    const int kvi = hs >= heads ? 1 : 0;
    const int h = hs - kvi * heads;
    const uint8_t *codes = (kvi ? v_codes : k_codes) + static_cast<int64_t>(h) * cap * CB;
    const uint16_t *scales = (kvi ? v_scales : k_scales) + static_cast<int64_t>(h) * cap * SG;
    __nv_bfloat16 *dst = out + static_cast<int64_t>(hs) * 128 + lane * 4;
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kTokensPerBlock;
#pragma unroll 1
    for (int u = 0; u < kTokensPerBlock; ++u) {
        const int64_t t = t0 + u;
        if (t >= n) break;
        uint32_t packed;
        if constexpr (BITS == 4) {
            packed = reinterpret_cast<const uint16_t *>(codes + t * CB)[lane];
        } else {
            packed = reinterpret_cast<const uint32_t *>(codes + t * CB)[lane];
        }
        const float s = __half2float(__ushort_as_half(scales[t * SG + lane / LANES_PER_GROUP]));
        float v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            int c;
            if constexpr (BITS == 4) {
                c = static_cast<int>((packed >> (4 * j)) & 0xFu);
                c = (c ^ 8) - 8;
            } else {
                c = static_cast<int>(static_cast<int8_t>((packed >> (8 * j)) & 0xFFu));
            }
            v[j] = static_cast<float>(c) * s;
        }
        rotate128_warp(v, lane);
        const __nv_bfloat162 lo = __floats2bfloat162_rn(v[0], v[1]);
        const __nv_bfloat162 hi = __floats2bfloat162_rn(v[2], v[3]);
        uint2 w;
        w.x = *reinterpret_cast<const uint32_t *>(&lo);
        w.y = *reinterpret_cast<const uint32_t *>(&hi);
        *reinterpret_cast<uint2 *>(dst + t * ld_out) = w;
    }
}

}  // namespace

cudaError_t launch_kv_rotate_quant_pack(const void *kv, int64_t n, int hidden, int64_t ld, int group, int bits,
                                        void *k_codes, void *v_codes, void *k_scales, void *v_scales,
                                        cudaStream_t s) {
    const int heads = hidden / 128;
    const int64_t cap = kvq_padded_rows(n);
    dim3 grid(static_cast<unsigned>(cap / kTokensPerBlock), static_cast<unsigned>((2 * heads + kWarps - 1) / kWarps));
    dim3 block(kWarps * 32);
    auto *kvp = static_cast<const __nv_bfloat16 *>(kv);
    auto *kc = static_cast<uint8_t *>(k_codes);
    auto *vc = static_cast<uint8_t *>(v_codes);
    auto *ks = static_cast<uint16_t *>(k_scales);
    auto *vs = static_cast<uint16_t *>(v_scales);
#define KVQ_LAUNCH_PACK(G, B) \
    rotate_quant_pack_kernel<G, B><<<grid, block, 0, s>>>(kvp, n, cap, heads, ld, kc, vc, ks, vs)
    if (bits == 4) {
        if (group == 32) KVQ_LAUNCH_PACK(32, 4);
        else if (group == 64) KVQ_LAUNCH_PACK(64, 4);
        else KVQ_LAUNCH_PACK(128, 4);
    } else {
        if (group == 32) KVQ_LAUNCH_PACK(32, 8);
        else if (group == 64) KVQ_LAUNCH_PACK(64, 8);
        else KVQ_LAUNCH_PACK(128, 8);
    }
#undef KVQ_LAUNCH_PACK
    return cudaGetLastError();
}

cudaError_t launch_kv_unpack(const void *k_codes, const void *v_codes, const void *k_scales, const void *v_scales,
                             int64_t n, int hidden, int group, int bits, void *kv_out, int64_t ld_out,
                             cudaStream_t s) {
    const int heads = hidden / 128;
    const int64_t cap = kvq_padded_rows(n);
    dim3 grid(static_cast<unsigned>(cap / kTokensPerBlock), static_cast<unsigned>((2 * heads + kWarps - 1) / kWarps));
    dim3 block(kWarps * 32);
    auto *kc = static_cast<const uint8_t *>(k_codes);
    auto *vc = static_cast<const uint8_t *>(v_codes);
    auto *ks = static_cast<const uint16_t *>(k_scales);
    auto *vs = static_cast<const uint16_t *>(v_scales);
    auto *o = static_cast<__nv_bfloat16 *>(kv_out);
#define KVQ_LAUNCH_UNPACK(G, B) unpack_kernel<G, B><<<grid, block, 0, s>>>(kc, vc, ks, vs, n, cap, heads, o, ld_out)
    if (bits == 4) {
        if (group == 32) KVQ_LAUNCH_UNPACK(32, 4);
        else if (group == 64) KVQ_LAUNCH_UNPACK(64, 4);
        else KVQ_LAUNCH_UNPACK(128, 4);
    } else {
        if (group == 32) KVQ_LAUNCH_UNPACK(32, 8);
        else if (group == 64) KVQ_LAUNCH_UNPACK(64, 8);
        else KVQ_LAUNCH_UNPACK(128, 8);
    }
#undef KVQ_LAUNCH_UNPACK
    return cudaGetLastError();
}

// ------------------------------------------------------------------ bounded-wait self-test
namespace {
__global__ void selftest_wait_kernel(uint64_t ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);  // nothing ever arrives
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait(&bar, 0, &abort_flag, &g_err_quant, ns);
    __syncthreads();
}
}  // namespace

cudaError_t launch_selftest_wait(uint64_t ns, cudaStream_t s) {
    selftest_wait_kernel<<<1, 32, 0, s>>>(ns);
    return cudaGetLastError();
}

cudaError_t read_clear_err_quant(unsigned int *v) {
    cudaError_t e = cudaMemcpyFromSymbol(v, g_err_quant, sizeof(unsigned int));
    if (e != cudaSuccess) return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_err_quant, &zero, sizeof(unsigned int));
}

}  // namespace kvq
