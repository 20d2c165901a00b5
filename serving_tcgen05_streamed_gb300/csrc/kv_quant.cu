// kv_quant.cu -- standalone rotate + quantise + pack of BF16 K/V into the
// head-major packed store, and its inverse (unpack, a diagnostic).
//
// The comfy-kitchen feature request ("Quality-oriented low-bit format")
// asks for fixed-width rotated INT4 with per-group scaling; vram_lab.py's
// `_hadamard`, `_fq_int4` and `_Int8KV` fix the rotation and rounding rules
// implemented in quant.cuh.
//
// Both kernels are HBM-bound: per token they move 2*hidden*2 bytes of BF16
// and 2*hidden*(bits/8 + 2/group) bytes of codes and scales.  Four lanes own
// one 128-wide head vector, 32 consecutive elements each, so five of the
// seven butterfly stages and (for groups of 32) the whole group absmax stay
// inside a lane, and a lane's codes leave in one 16-byte store (the unpack
// has an interleaved form for unaligned outputs, see there).  A warp works on
// 8 tokens of one head slot at a time (K heads, then V heads); a block of 8
// warps covers 8 head slots x 128 tokens in 16 passes.
//
// The pack kernel is held to 64 registers, so four blocks (32 warps) share an
// SM: one pass of 8 tokens at a time fits (ptxas reports one 8-byte spill
// store in the INT8 forms), and this measured 1.5-4 % faster than two passes
// loaded ahead at 80 registers, 3 blocks / SM.  Instead of registers, each pass asks L2 for the
// next pass's rows (prefetch.global.L2, one instruction per warp, no register
// held), so the next pass's loads find their lines on chip: +10 % for the
// pack kernel, +3 % for unpack (N = 262,144, same codes).  Blocks of 32 tokens
// left a quarter of the passes without a prefetch; blocks longer than 128
// tokens measured slower.  The stride-1 butterfly reads the BF16 halves
// directly (+1 %).  Global accesses move whole 32-byte sectors where the
// alignment allows (32-byte loads and stores, sm_100 and later).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"
#include "quant.cuh"

namespace kvq {
namespace {

__device__ unsigned int g_err_quant;

constexpr int kWarps = 8;
constexpr int kTokensPerBlock = 128;  // divides the padded row count, a multiple of 128
constexpr int kPass = 8;              // tokens per warp pass (4 lanes per token)
constexpr int kPasses = kTokensPerBlock / kPass;

// Asks L2 to fetch the 128-byte line holding p; no register receives data.
__device__ __forceinline__ void prefetch_l2(const void *p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<uint64_t>(p)));
}

// 32-byte global accesses (sm_100 and later): one instruction moves a whole
// sector.  The address must be 32-byte aligned.
__device__ __forceinline__ void ld_global_nc_v8(const void *p, uint32_t (&r)[8]) {
    asm volatile("ld.global.nc.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "l"(p));
}
__device__ __forceinline__ void st_global_v8(void *p, const uint32_t (&r)[8]) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(r[0]), "r"(r[1]),
                 "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}

// WIDE: the K/V rows and the code stores are 32-byte aligned, so a lane's 64
// bytes of BF16 arrive in two 32-byte loads (each a whole sector; four 16-byte
// loads each touch half of four sectors) and an INT8 lane's 32 code bytes
// leave in one store: +5 % (INT4, G = 32) and +9 % (INT8, G = 128) at
// N = 262,144, same codes.  Otherwise the 16-byte form runs.
template <int GROUP, int BITS, bool WIDE>
__global__ void __launch_bounds__(kWarps * 32, 4) rotate_quant_pack_kernel(const __nv_bfloat16 *__restrict__ kv,
                                                                         int64_t n, int64_t cap, int heads,
                                                                         int64_t ld, uint8_t *__restrict__ k_codes,
                                                                         uint8_t *__restrict__ v_codes,
                                                                         uint16_t *__restrict__ k_scales,
                                                                         uint16_t *__restrict__ v_scales) {
    constexpr int CB = 128 * BITS / 8;  // code bytes per head row
    constexpr int SG = 128 / GROUP;     // scales per head row
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hs = blockIdx.y * kWarps + warp;  // head slot: K heads then V heads
    if (hs >= 2 * heads) return;
    const int kvi = hs >= heads ? 1 : 0;
    const int h = hs - kvi * heads;
    const int q = lane & 3;
    uint8_t *codes = (kvi ? v_codes : k_codes) + static_cast<int64_t>(h) * cap * CB;
    uint16_t *scales = (kvi ? v_scales : k_scales) + static_cast<int64_t>(h) * cap * SG;
    const __nv_bfloat16 *src = kv + static_cast<int64_t>(hs) * 128 + q * 32;
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kTokensPerBlock + (lane >> 2);

#pragma unroll 1
    for (int p = 0; p < kPasses; ++p) {
        const int64_t t = t0 + p * kPass;
        // the next pass's rows: lanes 0 and 2 of each quad cover the head row's two 128-byte lines
        if ((q & 1) == 0 && p + 1 < kPasses && t + kPass < n) prefetch_l2(src + (t + kPass) * ld);
        uint32_t w[16];
        if constexpr (WIDE) {
            uint32_t a[8], b[8];
            if (t < n) {
                ld_global_nc_v8(src + t * ld, a);
                ld_global_nc_v8(src + t * ld + 16, b);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) a[i] = b[i] = 0u;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                w[i] = a[i];
                w[8 + i] = b[i];
            }
        } else {
            uint4 raw[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                raw[i] = (t < n) ? ld_global_nc_v4(src + t * ld + 8 * i) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                w[4 * i] = raw[i].x;
                w[4 * i + 1] = raw[i].y;
                w[4 * i + 2] = raw[i].z;
                w[4 * i + 3] = raw[i].w;
            }
        }
        float v[32];
        rotate128_quad_bf16(w, v, lane);
        uint32_t words[BITS];
        uint16_t sbits;
        quant128_quad<GROUP, BITS>(v, words, sbits);
        uint4 *dst = reinterpret_cast<uint4 *>(codes + t * CB + q * (CB / 4));
        if constexpr (WIDE && BITS == 8) {
            st_global_v8(dst, words);
        } else {
#pragma unroll
            for (int i = 0; i < BITS / 4; ++i)
                st_global_v4(dst + i, make_uint4(words[4 * i], words[4 * i + 1], words[4 * i + 2], words[4 * i + 3]));
        }
        if ((q % (GROUP / 32)) == 0) scales[t * SG + q / (GROUP / 32)] = sbits;
    }
}

// The unpack writes 28 KB of BF16 per token against 8 KB of codes read, so its
// stores decide its rate; they must write whole 32-byte sectors.  With the
// output 32-byte aligned, a lane keeps 32 consecutive elements and stores its
// 64 bytes as two 32-byte stores (unpack_kernel); otherwise lane q of a quad
// holds elements 32i + 8q .. 32i + 8q + 7 (the interleaved quad layout) and each
// of its four 16-byte stores joins the quad's to 64 consecutive bytes
// (unpack_interleaved_kernel).  The contiguous layout with 16-byte stores wrote
// half sectors: 4.89 TB/s against 5.82 (interleaved) and 6.29 (32-byte
// stores) at N = 262,144, G = 32, INT4, same output bits.
template <int GROUP, int BITS>
__global__ void __launch_bounds__(kWarps * 32) unpack_kernel(const uint8_t *__restrict__ k_codes,
                                                              const uint8_t *__restrict__ v_codes,
                                                              const uint16_t *__restrict__ k_scales,
                                                              const uint16_t *__restrict__ v_scales, int64_t n,
                                                              int64_t cap, int heads, __nv_bfloat16 *__restrict__ out,
                                                              int64_t ld_out) {
    constexpr int CB = 128 * BITS / 8;
    constexpr int SG = 128 / GROUP;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hs = blockIdx.y * kWarps + warp;
    if (hs >= 2 * heads) return;
    const int kvi = hs >= heads ? 1 : 0;
    const int h = hs - kvi * heads;
    const int q = lane & 3;
    const uint8_t *codes = (kvi ? v_codes : k_codes) + static_cast<int64_t>(h) * cap * CB;
    const uint16_t *scales = (kvi ? v_scales : k_scales) + static_cast<int64_t>(h) * cap * SG;
    __nv_bfloat16 *dst = out + static_cast<int64_t>(hs) * 128 + q * 32;
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kTokensPerBlock + (lane >> 2);
#pragma unroll 1
    for (int p = 0; p < kPasses; ++p) {
        const int64_t t = t0 + p * kPass;
        // the next pass's code rows (CB bytes each, consecutive in the head-major store)
        // and its scale rows (8 x SG fp16, one line)
        if (q == 0 && p + 1 < kPasses && t + kPass < n) prefetch_l2(codes + (t + kPass) * CB);
        if (lane == 0 && p + 1 < kPasses && t + kPass < n) prefetch_l2(scales + (t + kPass) * SG);
        // every lane of the quad takes part in the shuffles; rows past n are not stored
        const bool live = t < n;
        uint4 cw[BITS / 4];
        float s = 0.0f;
        if (live) {
#pragma unroll
            for (int i = 0; i < BITS / 4; ++i) cw[i] = ld_global_nc_v4(codes + t * CB + q * (CB / 4) + 16 * i);
            s = __half2float(__ushort_as_half(scales[t * SG + q / (GROUP / 32)]));
        } else {
#pragma unroll
            for (int i = 0; i < BITS / 4; ++i) cw[i] = make_uint4(0u, 0u, 0u, 0u);
        }
        float v[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            const uint32_t word = (&cw[e / (32 / BITS) / 4].x)[(e / (32 / BITS)) % 4];
            int c;
            if constexpr (BITS == 4) {
                c = static_cast<int>((word >> (4 * (e % 8))) & 0xFu);
                c = (c ^ 8) - 8;
            } else {
                c = static_cast<int>(static_cast<int8_t>((word >> (8 * (e % 4))) & 0xFFu));
            }
            v[e] = static_cast<float>(c) * s;
        }
        rotate128_quad(v, lane);
        if (live) {
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                uint32_t w8[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const __nv_bfloat162 b2 = __floats2bfloat162_rn(v[16 * i + 2 * k], v[16 * i + 2 * k + 1]);
                    w8[k] = *reinterpret_cast<const uint32_t *>(&b2);
                }
                st_global_v8(dst + t * ld_out + 16 * i, w8);
            }
        }
    }
}

template <int GROUP, int BITS>
__global__ void __launch_bounds__(kWarps * 32) unpack_interleaved_kernel(
    const uint8_t *__restrict__ k_codes, const uint8_t *__restrict__ v_codes, const uint16_t *__restrict__ k_scales,
    const uint16_t *__restrict__ v_scales, int64_t n, int64_t cap, int heads, __nv_bfloat16 *__restrict__ out,
    int64_t ld_out) {
    constexpr int CB = 128 * BITS / 8;
    constexpr int SG = 128 / GROUP;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hs = blockIdx.y * kWarps + warp;
    if (hs >= 2 * heads) return;
    const int kvi = hs >= heads ? 1 : 0;
    const int h = hs - kvi * heads;
    const int q = lane & 3;
    const uint8_t *codes = (kvi ? v_codes : k_codes) + static_cast<int64_t>(h) * cap * CB;
    const uint16_t *scales = (kvi ? v_scales : k_scales) + static_cast<int64_t>(h) * cap * SG;
    __nv_bfloat16 *dst = out + static_cast<int64_t>(hs) * 128 + q * 8;
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kTokensPerBlock + (lane >> 2);
#pragma unroll 1
    for (int p = 0; p < kPasses; ++p) {
        const int64_t t = t0 + p * kPass;
        // the next pass's code rows (CB bytes each, consecutive in the head-major store)
        // and its scale rows (8 x SG fp16, one line)
        if (q == 0 && p + 1 < kPasses && t + kPass < n) prefetch_l2(codes + (t + kPass) * CB);
        if (lane == 0 && p + 1 < kPasses && t + kPass < n) prefetch_l2(scales + (t + kPass) * SG);
        // every lane of the quad takes part in the shuffles; rows past n are not stored
        const bool live = t < n;
        uint16_t srow[SG];  // the token's scales, one load
        if constexpr (SG == 4) {
            const uint2 x = live ? __ldg(reinterpret_cast<const uint2 *>(scales + t * SG)) : make_uint2(0u, 0u);
            srow[0] = static_cast<uint16_t>(x.x);
            srow[1] = static_cast<uint16_t>(x.x >> 16);
            srow[2] = static_cast<uint16_t>(x.y);
            srow[3] = static_cast<uint16_t>(x.y >> 16);
        } else if constexpr (SG == 2) {
            const unsigned int x = live ? __ldg(reinterpret_cast<const unsigned int *>(scales + t * SG)) : 0u;
            srow[0] = static_cast<uint16_t>(x);
            srow[1] = static_cast<uint16_t>(x >> 16);
        } else {
            srow[0] = live ? scales[t * SG] : static_cast<uint16_t>(0);
        }
        float v[32];
#pragma unroll
        for (int i = 0; i < 4; ++i) {  // elements 32i + 8q .. +7: 4 code bytes (INT4) or 8 (INT8)
            const float s = __half2float(__ushort_as_half(srow[(32 * i) / GROUP]));
            uint32_t w0 = 0u, w1 = 0u;
            if (live) {
                const uint8_t *c = codes + t * CB + (32 * i + 8 * q) * BITS / 8;
                if constexpr (BITS == 4) {
                    w0 = __ldg(reinterpret_cast<const unsigned int *>(c));
                } else {
                    const uint2 x = __ldg(reinterpret_cast<const uint2 *>(c));
                    w0 = x.x;
                    w1 = x.y;
                }
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                int c;
                if constexpr (BITS == 4) {
                    c = static_cast<int>((w0 >> (4 * k)) & 0xFu);
                    c = (c ^ 8) - 8;
                } else {
                    c = static_cast<int>(static_cast<int8_t>(((k < 4 ? w0 : w1) >> (8 * (k & 3))) & 0xFFu));
                }
                v[8 * i + k] = static_cast<float>(c) * s;
            }
        }
        rotate128_quad_interleaved(v, lane);
        if (live) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint32_t w4[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const __nv_bfloat162 b2 = __floats2bfloat162_rn(v[8 * i + 2 * k], v[8 * i + 2 * k + 1]);
                    w4[k] = *reinterpret_cast<const uint32_t *>(&b2);
                }
                *reinterpret_cast<uint4 *>(dst + t * ld_out + 32 * i) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
            }
        }
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
    const bool wide = reinterpret_cast<uintptr_t>(kv) % 32 == 0 && (ld * 2) % 32 == 0 &&
                      reinterpret_cast<uintptr_t>(k_codes) % 32 == 0 && reinterpret_cast<uintptr_t>(v_codes) % 32 == 0;
#define KVQ_LAUNCH_PACK(G, B)                                                                                  \
    do {                                                                                                       \
        if (wide)                                                                                              \
            rotate_quant_pack_kernel<G, B, true><<<grid, block, 0, s>>>(kvp, n, cap, heads, ld, kc, vc, ks, vs);  \
        else                                                                                                   \
            rotate_quant_pack_kernel<G, B, false><<<grid, block, 0, s>>>(kvp, n, cap, heads, ld, kc, vc, ks, vs); \
    } while (0)
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
    const bool wide = reinterpret_cast<uintptr_t>(kv_out) % 32 == 0 && (ld_out * 2) % 32 == 0;
#define KVQ_LAUNCH_UNPACK(G, B)                                                                        \
    do {                                                                                               \
        if (wide)                                                                                      \
            unpack_kernel<G, B><<<grid, block, 0, s>>>(kc, vc, ks, vs, n, cap, heads, o, ld_out);             \
        else                                                                                           \
            unpack_interleaved_kernel<G, B><<<grid, block, 0, s>>>(kc, vc, ks, vs, n, cap, heads, o, ld_out); \
    } while (0)
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
