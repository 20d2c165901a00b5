// attention.cu -- dense attention over a packed rotated low-bit K/V store.
//
// The comfy-kitchen feature request ("Proposed backend capability", "Dense
// fallback is important") asks for attention that reads Q in BF16 and K/V as
// packed 4-bit codes and decodes K/V tile by tile inside the kernel, never
// expanding the whole K/V to BF16.  vram_lab.py's kvi8r store shows the
// algebra used here: with an orthonormal H, q.k = (qH).(kH) and
// P.V = (P.(VH)).H^T, so attention runs entirely in the rotated basis and the
// output is un-rotated once; `_online_combine` is the log-sum-exp merge that
// the running softmax below performs tile by tile.
//
// One CTA = one head x 256 query rows, as two 128-row tiles A and B that
// take turns on the tensor core (ping-pong): while the softmax of tile A
// works on its scores, the tensor core runs tile B's P.V and next Q.K^T, and
// the other way round.  16 warps in four warpgroups:
//   WG0, WG1   softmax of tile A / B: one thread per query row; reads the S
//              row from TMEM, keeps a running max in the log2 domain and
//              rescales the output accumulator only when the row max grew by
//              more than 2^8 (the stale max is used consistently for P and the
//              row sum, so the result is exact); writes P as FP16 back into
//              the first 64 TMEM columns of its own S, and at the end divides
//              by the row sum, un-rotates the row with the 128-point fast
//              Walsh-Hadamard transform in registers and stores it.
//   WG2        dequantisers: per 128-key tile, load the INT4 / INT8 codes and
//              fp16 scales straight from global memory (issued one tile
//              ahead), decode them with integer bit tricks into FP16
//              (code * scale) and store K^ [key][dim] and V^T [dim][key] in
//              the 128-byte-swizzled K-major layout the tensor core reads.
//              K^'s dims are permuted inside each 8-dim chunk (the order
//              e0 e4 e1 e5 e2 e6 e3 e7 falls out of the nibble decode); Q is
//              permuted the same way when it is converted, so Q.K^T is
//              unchanged.  They also convert the BF16 Q tiles to FP16 once.
//   WG3        warp 12: TMA of the Q tiles, TMEM allocation and the single
//              MMA thread; warps 13-15 idle.
// Registers are redistributed with setmaxnreg: 176 per softmax thread, 104
// per dequantiser, 56 for WG3 (512 threads x 128 at launch).
// TMEM (512 columns): S_A, S_B, O_A, O_B, 128 columns each; P_t aliases the
// first 64 columns of S_t.  tcgen05.mma instructions from one thread execute
// in issue order, so S_t(j+1), issued after P_t(j).V^(j), overwrites P_t(j)
// only after that MMA has read it; and the commit that signals S_t(j+1) also
// covers P_t(j).V^(j), so O_t is final for tile j when the softmax sees S_t(j+1).
// Scores, the softmax and O are fp32; the MMA operands are FP16 (11-bit
// significand: the rotation spreads values evenly, where BF16's 8 bits would
// cost a noticeably higher error floor).  No split over keys: every query
// row is computed by one CTA in one fixed order, so results do not depend on
// how the queries are tiled or chunked.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdlib>
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"
#include "quant.cuh"

namespace kvq {
namespace {

__device__ unsigned int g_err_attn;

constexpr int BQT = 128;       // query rows per tile
constexpr int NQT = 2;         // query tiles per CTA
constexpr int BQ = BQT * NQT;  // query rows per CTA
constexpr int BKV = 128;       // keys per tile
constexpr int KV_STAGES = 2;   // K^ / V^T shared-memory stages
constexpr int NUM_DQ_THREADS = 128;
constexpr int NUM_SM_THREADS = 128;  // per query tile
constexpr int NUM_THREADS = 512;
constexpr int WARP_MMA = 12;
constexpr int REG_SOFTMAX = 176, REG_DEQUANT = 104, REG_MMA = 56;
static_assert(2 * 128 * REG_SOFTMAX + 128 * REG_DEQUANT + 128 * REG_MMA <= NUM_THREADS * 128,
              "register split exceeds the launch budget");
constexpr int TILE_BYTES = 128 * 128 * 2;  // one 128x128 fp16 operand tile
constexpr int HALF_BYTES = TILE_BYTES / 2;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

__host__ __device__ constexpr uint32_t tm_s(int t) { return static_cast<uint32_t>(t * 128); }
__host__ __device__ constexpr uint32_t tm_o(int t) { return static_cast<uint32_t>(256 + t * 128); }

struct AttnParams {
    int64_t n_q;
    int hidden;
    int total_tiles;
    float scale_log2;  // sm_scale * log2(e)
    int out_fp32;
    void *out;
    RangeTable ranges;
    int tiles_before[KVQ_MAX_RANGES + 1];
};

struct SmemLayout {
    static constexpr int Q = 0;                           // NQT tiles
    static constexpr int K = Q + NQT * TILE_BYTES;        // KV_STAGES tiles
    static constexpr int V = K + KV_STAGES * TILE_BYTES;  // KV_STAGES tiles
    static constexpr int BAR = V + KV_STAGES * TILE_BYTES;
    static constexpr int BYTES = BAR + 256 + 1024;
};

// Physical byte offset of 16-byte chunk `c` (0..15 along K) of row `r` in a
// 128-row K-major tile stored as two 64-element halves, 128-byte swizzle.
__device__ __forceinline__ uint32_t sw128_off(int r, int c) {
    return static_cast<uint32_t>((c >> 3) * HALF_BYTES + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}
__device__ __forceinline__ uint32_t lop_and_xor(uint32_t a, uint32_t mask, uint32_t x) {
    // (a & mask) ^ x in one LOP3
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(r) : "r"(a), "r"(mask), "r"(x));
    return r;
}
__device__ __forceinline__ uint32_t h2_add(uint32_t a, uint32_t b) {
    __half2 r = __hadd2(*reinterpret_cast<__half2 *>(&a), *reinterpret_cast<__half2 *>(&b));
    return *reinterpret_cast<uint32_t *>(&r);
}
__device__ __forceinline__ uint32_t h2_fma(uint32_t a, uint32_t b, uint32_t c) {
    __half2 r = __hfma2(*reinterpret_cast<__half2 *>(&a), *reinterpret_cast<__half2 *>(&b),
                        *reinterpret_cast<__half2 *>(&c));
    return *reinterpret_cast<uint32_t *>(&r);
}
__device__ __forceinline__ uint32_t h2_mul(uint32_t a, uint32_t b) {
    __half2 r = __hmul2(*reinterpret_cast<__half2 *>(&a), *reinterpret_cast<__half2 *>(&b));
    return *reinterpret_cast<uint32_t *>(&r);
}

// fp16 bit patterns used by the decode
constexpr uint32_t H2_NEG1032 = 0xE408E408u;  // (-1032, -1032)
constexpr uint32_t H2_NEG72 = 0xD480D480u;    // (-72, -72)
constexpr uint32_t H2_1_16 = 0x2C002C00u;     // (1/16, 1/16)
constexpr uint32_t H2_NEG1152 = 0xE480E480u;  // (-1152, -1152)

// Eight INT4 codes (one 32-bit word, element e in bits 4e..4e+3) -> four
// FP16 pairs (e0,e4) (e1,e5) (e2,e6) (e3,e7), each times the scale pair s2.
__device__ __forceinline__ void dq_int4_word(uint32_t w, uint32_t s2, uint32_t (&o)[4]) {
    const uint32_t w8 = w >> 8;
    const uint32_t t0 = lop_and_xor(w, 0x000F000Fu, 0x64086408u);  // 1024 + (c0 + 8)
    const uint32_t t1 = lop_and_xor(w, 0x00F000F0u, 0x64806480u);  // 1024 + 16 (c1 + 8)
    const uint32_t t2 = lop_and_xor(w8, 0x000F000Fu, 0x64086408u);
    const uint32_t t3 = lop_and_xor(w8, 0x00F000F0u, 0x64806480u);
    o[0] = h2_mul(h2_add(t0, H2_NEG1032), s2);
    o[1] = h2_mul(h2_fma(t1, H2_1_16, H2_NEG72), s2);
    o[2] = h2_mul(h2_add(t2, H2_NEG1032), s2);
    o[3] = h2_mul(h2_fma(t3, H2_1_16, H2_NEG72), s2);
}
// Two bytes (int8 codes) at byte positions picked by `sel` into an FP16 pair times s2.
__device__ __forceinline__ uint32_t dq_int8_pair(uint32_t a, uint32_t b, uint32_t sel, uint32_t s2) {
    const uint32_t x = prmt(a, b, sel);
    const uint32_t t = lop_and_xor(x, 0x00FF00FFu, 0x64806480u);  // 1024 + (c + 128)
    return h2_mul(h2_add(t, H2_NEG1152), s2);
}
__device__ __forceinline__ uint32_t h2_dup(uint16_t s) { return static_cast<uint32_t>(s) * 0x10001u; }
__device__ __forceinline__ uint32_t h2_pack(uint16_t lo, uint16_t hi) {
    return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

// Packed fp32 pair arithmetic (one instruction for two lanes of work).
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float &a, float &b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// The tile sequence walks the ranges in order; tile j of the sequence is
// local tile j - tiles_before[g] of range g.
struct TileRef {
    int g;
    int64_t key0;  // first key (row) of the tile inside range g
    int valid;     // keys of the tile that exist (1..128)
};
__device__ __forceinline__ TileRef tile_ref(const AttnParams &p, int j) {
    int g = 0;
    while (g + 1 < p.ranges.n && j >= p.tiles_before[g + 1]) ++g;
    TileRef t;
    t.g = g;
    t.key0 = static_cast<int64_t>(j - p.tiles_before[g]) * BKV;
    const int64_t rem = p.ranges.r[g].len - t.key0;
    t.valid = rem < BKV ? static_cast<int>(rem) : BKV;
    return t;
}

// Raw codes a dequantiser thread holds for one tile (MIXED = INT8 possible).
template <bool MIXED>
struct RawTile {
    uint4 k[MIXED ? 8 : 4];                                     // one key row: 64 (INT4) or 128 (INT8) bytes
    typename std::conditional<MIXED, uint4, uint2>::type v[8];  // 8 keys x 16 dims (8 B INT4, 16 B INT8)
    uint16_t ks[4];                                             // scales of the key row (128/GROUP used)
    uint16_t vs[8];                                             // scale of each of the 8 keys, 16-dim block
    int bits;
};

template <int GROUP, bool MIXED>
__device__ __forceinline__ void load_raw(const AttnParams &p, int head, int j, int tid, RawTile<MIXED> &R) {
    const TileRef t = tile_ref(p, j);
    const RangeDev &rg = p.ranges.r[t.g];
    const int bits = MIXED ? rg.bits : 4;
    R.bits = bits;
    const int cb = bits == 4 ? 64 : 128;
    constexpr int SG = 128 / GROUP;
    {  // K unit: key row tid
        const int r = tid;
        if (r < t.valid) {
            const int64_t row = static_cast<int64_t>(head) * rg.cap + t.key0 + r;
            const uint4 *src = reinterpret_cast<const uint4 *>(rg.k_codes + row * cb);
#pragma unroll
            for (int i = 0; i < (MIXED ? 8 : 4); ++i)
                if (i < cb / 16) R.k[i] = ld_global_nc_v4(src + i);
            const uint16_t *ss = rg.k_scales + row * SG;
#pragma unroll
            for (int g = 0; g < SG; ++g) R.ks[g] = __ldg(ss + g);
        } else {
#pragma unroll
            for (int i = 0; i < (MIXED ? 8 : 4); ++i) R.k[i] = make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int g = 0; g < SG; ++g) R.ks[g] = 0;
        }
    }
    {  // V unit: keys 8*kb .. 8*kb+7, dims 16*db .. 16*db+15
        const int kb = tid & 15, db = tid >> 4;
        const int g = (16 * db) / GROUP;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int r = 8 * kb + k;
            if (r < t.valid) {
                const int64_t row = static_cast<int64_t>(head) * rg.cap + t.key0 + r;
                if constexpr (MIXED) {
                    if (bits == 4) {
                        const uint2 x = *reinterpret_cast<const uint2 *>(rg.v_codes + row * 64 + db * 8);
                        R.v[k] = make_uint4(x.x, x.y, 0, 0);
                    } else {
                        R.v[k] = ld_global_nc_v4(rg.v_codes + row * 128 + db * 16);
                    }
                } else {
                    R.v[k] = *reinterpret_cast<const uint2 *>(rg.v_codes + row * 64 + db * 8);
                }
                R.vs[k] = __ldg(rg.v_scales + row * SG + g);
            } else {
                R.v[k] = {};
                R.vs[k] = 0;
            }
        }
    }
}

template <int GROUP, bool MIXED>
__device__ __forceinline__ void store_tile(const RawTile<MIXED> &R, uint8_t *k_tile, uint8_t *v_tile, int tid) {
    {  // K^ row tid: 16 chunks of 8 dims (permuted e0 e4 e1 e5 e2 e6 e3 e7)
        const int r = tid;
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            const uint32_t s2 = h2_dup(R.ks[(c * 8) / GROUP]);
            uint32_t o[4];
            if (!MIXED || R.bits == 4) {
                const uint32_t w = (&R.k[c >> 2].x)[c & 3];
                dq_int4_word(w, s2, o);
            } else {
                const uint32_t a = (&R.k[c >> 1].x)[(c & 1) * 2];
                const uint32_t b = (&R.k[c >> 1].x)[(c & 1) * 2 + 1];
                o[0] = dq_int8_pair(a, b, 0x0400u, s2);
                o[1] = dq_int8_pair(a, b, 0x0501u, s2);
                o[2] = dq_int8_pair(a, b, 0x0602u, s2);
                o[3] = dq_int8_pair(a, b, 0x0703u, s2);
            }
            *reinterpret_cast<uint4 *>(k_tile + sw128_off(r, c)) = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
    {  // V^T rows 16*db .. 16*db+15, chunk kb (keys 8kb .. 8kb+7, natural order)
        const int kb = tid & 15, db = tid >> 4;
        uint32_t s2[4];
#pragma unroll
        for (int kp = 0; kp < 4; ++kp) s2[kp] = h2_pack(R.vs[2 * kp], R.vs[2 * kp + 1]);
        if (!MIXED || R.bits == 4) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {  // dims 4q .. 4q+3 of the 16-dim block
                uint32_t out[4][4];         // [dim][key pair]
#pragma unroll
                for (int kp = 0; kp < 4; ++kp) {
                    const uint32_t aw = reinterpret_cast<const uint32_t *>(&R.v[2 * kp])[q >> 1];
                    const uint32_t bw = reinterpret_cast<const uint32_t *>(&R.v[2 * kp + 1])[q >> 1];
                    // low half: 4 dims of key a, high half: the same 4 dims of key a+1
                    const uint32_t x = prmt(aw, bw, (q & 1) ? 0x7632u : 0x5410u);
                    uint32_t o[4];
                    dq_int4_word(x, s2[kp], o);
#pragma unroll
                    for (int d = 0; d < 4; ++d) out[d][kp] = o[d];
                }
#pragma unroll
                for (int d = 0; d < 4; ++d)
                    *reinterpret_cast<uint4 *>(v_tile + sw128_off(16 * db + 4 * q + d, kb)) =
                        make_uint4(out[d][0], out[d][1], out[d][2], out[d][3]);
            }
        } else {
#pragma unroll
            for (int d = 0; d < 16; ++d) {
                uint32_t w4[4];
#pragma unroll
                for (int kp = 0; kp < 4; ++kp) {
                    const uint32_t aw = reinterpret_cast<const uint32_t *>(&R.v[2 * kp])[d >> 2];
                    const uint32_t bw = reinterpret_cast<const uint32_t *>(&R.v[2 * kp + 1])[d >> 2];
                    const uint32_t bi = static_cast<uint32_t>(d & 3);
                    w4[kp] = dq_int8_pair(aw, bw, bi | ((4u + bi) << 8), s2[kp]);
                }
                *reinterpret_cast<uint4 *>(v_tile + sw128_off(16 * db + d, kb)) =
                    make_uint4(w4[0], w4[1], w4[2], w4[3]);
            }
        }
    }
}

__device__ __forceinline__ void tmem_ld128(uint32_t taddr, uint32_t (&r)[128]) {
    tmem_ld32(taddr + 0, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
    tmem_ld32(taddr + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
    tmem_ld32(taddr + 64, *reinterpret_cast<uint32_t(*)[32]>(&r[64]));
    tmem_ld32(taddr + 96, *reinterpret_cast<uint32_t(*)[32]>(&r[96]));
    tmem_ld_wait();
}

template <int GROUP, bool MIXED>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    attention_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ AttnParams p) {
    using L = SmemLayout;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sQ = smem + L::Q;
    uint8_t *sK = smem + L::K;
    uint8_t *sV = smem + L::V;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::BAR);
    uint64_t *q_tma = bars + 0;
    uint64_t *q_ready = bars + 1;
    uint64_t *kv_full = bars + 2;   // [KV_STAGES]
    uint64_t *kv_empty = bars + 4;  // [KV_STAGES]
    uint64_t *s_full = bars + 6;    // [NQT]
    uint64_t *p_full = bars + 8;    // [NQT]
    uint64_t *pv_done = bars + 10;  // [NQT]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 12);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int head = blockIdx.y;
    const int64_t q0 = static_cast<int64_t>(blockIdx.x) * BQ;
    const int T = p.total_tiles;

    if (threadIdx.x == 0) {
        mbar_init(q_tma, 1);
        mbar_init(q_ready, NUM_DQ_THREADS);
        for (int i = 0; i < KV_STAGES; ++i) {
            mbar_init(&kv_full[i], NUM_DQ_THREADS);
            mbar_init(&kv_empty[i], 1);
        }
        for (int i = 0; i < NQT; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], NUM_SM_THREADS);
            mbar_init(&pv_done[i], 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == WARP_MMA) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp >= 12) {
        setmaxnreg_dec<REG_MMA>();
        // ------------------------------------------------------------ WG3: Q load + MMA issue
        if (warp == WARP_MMA) {
            if (elect_one()) {
                prefetch_tmap(&tm_q);
                mbar_arrive_expect_tx(q_tma, NQT * TILE_BYTES);
#pragma unroll
                for (int t = 0; t < NQT; ++t) {
                    const int y = static_cast<int>(q0) + t * BQT;
                    tma_load_2d(sQ + t * TILE_BYTES, &tm_q, q_tma, head * 128, y);
                    tma_load_2d(sQ + t * TILE_BYTES + HALF_BYTES, &tm_q, q_tma, head * 128 + 64, y);
                }
                constexpr uint32_t idesc = make_idesc_f16(128, 128, 0);
                const uint32_t qa = smem_u32(sQ);
                bool ok = mbar_wait(q_ready, 0, abort_flag, &g_err_attn);
                tc_fence_after();
                auto issue_s = [&](int j, int t) {  // S_t(j) = Q_t . K^_j^T
                    const uint32_t kb = smem_u32(sK + (j % KV_STAGES) * TILE_BYTES);
                    const uint32_t d = tmem + tm_s(t);
                    const uint32_t q = qa + t * TILE_BYTES;
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const uint32_t off = (k >> 2) * HALF_BYTES + (k & 3) * 32;
                        mma_f16_ss(d, make_sdesc_sw128(q + off), make_sdesc_sw128(kb + off), idesc, k > 0);
                    }
                    mma_commit(&s_full[t]);
                };
                if (ok && T > 0) {
                    ok = mbar_wait(&kv_full[0], 0, abort_flag, &g_err_attn);
                    if (ok) {
                        tc_fence_after();
                        issue_s(0, 0);
                        issue_s(0, 1);
                    }
                }
                for (int j = 0; ok && j < T; ++j) {
                    const int st = j % KV_STAGES;
                    const uint32_t vb = smem_u32(sV + st * TILE_BYTES);
                    for (int t = 0; t < NQT && ok; ++t) {
                        // O_t += P_t(j) . V^_j, P_t read from TMEM (the first 64 columns of S_t)
                        ok = mbar_wait(&p_full[t], j & 1, abort_flag, &g_err_attn);
                        if (!ok) break;
                        tc_fence_after();
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const uint32_t off = (k >> 2) * HALF_BYTES + (k & 3) * 32;
                            mma_f16_ts(tmem + tm_o(t), tmem + tm_s(t) + k * 8, make_sdesc_sw128(vb + off), idesc,
                                       (j > 0 || k > 0) ? 1u : 0u);
                        }
                        mma_commit(&pv_done[t]);
                        if (t == NQT - 1) mma_commit(&kv_empty[st]);
                        if (j + 1 < T) {
                            if (t == 0) {
                                ok = mbar_wait(&kv_full[(j + 1) % KV_STAGES], ((j + 1) / KV_STAGES) & 1, abort_flag,
                                               &g_err_attn);
                                if (!ok) break;
                                tc_fence_after();
                            }
                            issue_s(j + 1, t);
                        }
                    }
                }
                // drain: nothing this thread issued is still running when the CTA exits
                volatile int no_abort = 0;
                if (*abort_flag) {
                    mma_commit(&pv_done[0]);
                    mbar_wait(&pv_done[0], 0, &no_abort, nullptr, 1000000000ull);
                }
                mbar_wait(q_tma, 0, &no_abort, nullptr);
            }
            __syncwarp();
        }
    } else if (warp >= 8) {
        setmaxnreg_dec<REG_DEQUANT>();
        // ------------------------------------------------------------ WG2: dequantisers
        const int tid = threadIdx.x - 256;  // 0..127
        // Q: BF16 -> FP16 in place, dims permuted e0 e4 e1 e5 e2 e6 e3 e7 within each 8-chunk
        const bool ok = mbar_wait(q_tma, 0, abort_flag, &g_err_attn);
        if (ok) {
#pragma unroll 4
            for (int i = tid; i < NQT * TILE_BYTES / 16; i += NUM_DQ_THREADS) {
                uint4 *c = reinterpret_cast<uint4 *>(sQ + i * 16);
                const uint4 v = *c;
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
                float f[8];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    f[2 * e] = __uint_as_float(w[e] << 16);
                    f[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
                }
                uint32_t o[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const __half2 h = __floats2half2_rn(f[e], f[e + 4]);
                    o[e] = *reinterpret_cast<const uint32_t *>(&h);
                }
                *c = make_uint4(o[0], o[1], o[2], o[3]);
            }
            fence_proxy_async_smem();
        }
        mbar_arrive(q_ready);
        RawTile<MIXED> raw;
        if (ok && T > 0) load_raw<GROUP, MIXED>(p, head, 0, tid, raw);
        for (int j = 0; ok && j < T && !*abort_flag; ++j) {
            const int st = j % KV_STAGES;
            if (!mbar_wait(&kv_empty[st], ((j / KV_STAGES) & 1) ^ 1, abort_flag, &g_err_attn)) break;
            store_tile<GROUP, MIXED>(raw, sK + st * TILE_BYTES, sV + st * TILE_BYTES, tid);
            fence_proxy_async_smem();
            mbar_arrive(&kv_full[st]);
            if (j + 1 < T) load_raw<GROUP, MIXED>(p, head, j + 1, tid, raw);
        }
    } else {
        setmaxnreg_inc<REG_SOFTMAX>();
        // ------------------------------------------------------------ WG0 / WG1: softmax + epilogue
        const int t = warp >> 2;  // query tile
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;  // query row inside the tile
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t sa = tmem + lane_base + tm_s(t);
        const uint32_t oa = tmem + lane_base + tm_o(t);
        float m = -INFINITY;  // running max (log2 units, possibly stale)
        float l = 0.0f;       // running sum of p
        const float sl = p.scale_log2;
        bool ok = true;
        for (int j = 0; j < T; ++j) {
            // the wait result is made warp-uniform before any warp-collective TMEM access
            if (!__all_sync(0xffffffffu, mbar_wait(&s_full[t], j & 1, abort_flag, &g_err_attn))) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sr[128];
            tmem_ld128(sa, sr);
            const int valid = tile_ref(p, j).valid;
            if (valid < BKV) {
#pragma unroll
                for (int c = 0; c < 128; ++c)
                    if (c >= valid) sr[c] = __float_as_uint(-INFINITY);
            }
            float mx0 = __uint_as_float(sr[0]), mx1 = __uint_as_float(sr[1]);
#pragma unroll
            for (int c = 2; c < 126; c += 4) {
                mx0 = fmax3(mx0, __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
                mx1 = fmax3(mx1, __uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3]));
            }
            const float mx = fmax3(mx0, mx1, fmaxf(__uint_as_float(sr[126]), __uint_as_float(sr[127])));
            // Lazy rescaling: a row moves its max only when it grew by more than the
            // threshold, a decision that depends on that row's scores alone.  The
            // O rescale uses warp-collective TMEM loads and stores, so it runs for
            // the whole warp when any row needs it; the other rows multiply by 1.
            const float cand = mx * sl;
            float alpha = 1.0f;
            const bool grow = cand > m + kRescaleThreshold;
            if (grow) {
                alpha = ex2_approx(m - cand);  // 0 on the first tile
                m = cand;
            }
            const bool rescale = __any_sync(0xffffffffu, grow);
            // p = 2^(s*sl - m) as FP16 pairs, packed over S's first 64 columns
            const uint64_t sl2 = f2_pack(sl, sl), nm2 = f2_pack(-m, -m);
            uint64_t acc0 = f2_pack(0.0f, 0.0f), acc1 = acc0;
            uint32_t pk[64];
#pragma unroll
            for (int c = 0; c < 128; c += 4) {
                const uint64_t a0 = f2_fma(f2_pack(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), sl2, nm2);
                const uint64_t a1 =
                    f2_fma(f2_pack(__uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3])), sl2, nm2);
                float x0, x1, x2, x3;
                f2_unpack(a0, x0, x1);
                f2_unpack(a1, x2, x3);
                const __half2 h0 = __floats2half2_rn(ex2_approx(x0), ex2_approx(x1));
                const __half2 h1 = __floats2half2_rn(ex2_approx(x2), ex2_approx(x3));
                pk[c >> 1] = *reinterpret_cast<const uint32_t *>(&h0);
                pk[(c >> 1) + 1] = *reinterpret_cast<const uint32_t *>(&h1);
                // the row sum uses the same FP16-rounded weights the MMA sees
                const float2 f0 = __half22float2(h0), f1 = __half22float2(h1);
                acc0 = f2_add(acc0, f2_pack(f0.x, f0.y));
                acc1 = f2_add(acc1, f2_pack(f1.x, f1.y));
            }
            float u0, u1, u2, u3;
            f2_unpack(acc0, u0, u1);
            f2_unpack(acc1, u2, u3);
            l = l * alpha + ((u0 + u1) + (u2 + u3));
            // S_t(j) completing implies P_t(j-1).V^(j-1) completed: O_t is final for j-1
            if (rescale && j > 0) {
#pragma unroll 1
                for (int c0 = 0; c0 < 128; c0 += 32) {
                    uint32_t o32[32];
                    tmem_ld32(oa + c0, o32);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) o32[i] = __float_as_uint(__uint_as_float(o32[i]) * alpha);
                    tmem_st16(oa + c0, *reinterpret_cast<const uint32_t(*)[16]>(&o32[0]));
                    tmem_st16(oa + c0 + 16, *reinterpret_cast<const uint32_t(*)[16]>(&o32[16]));
                }
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_st16(sa + c * 16, *reinterpret_cast<const uint32_t(*)[16]>(&pk[c * 16]));
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&p_full[t]);
        }
        // epilogue: O / l, un-rotate, store
        if (ok && T > 0 && __all_sync(0xffffffffu, mbar_wait(&pv_done[t], (T - 1) & 1, abort_flag, &g_err_attn))) {
            tc_fence_after();
            uint32_t oraw[128];
            tmem_ld128(oa, oraw);
            const float inv_l = 1.0f / l;
            float o[128];
#pragma unroll
            for (int c = 0; c < 128; ++c) o[c] = __uint_as_float(oraw[c]) * inv_l;
            rotate128_thread(o);
            const int64_t row = q0 + t * BQT + r;
            if (row < p.n_q) {
                if (p.out_fp32) {
                    float4 *dst =
                        reinterpret_cast<float4 *>(static_cast<float *>(p.out) + row * p.hidden + head * 128);
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        dst[i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
                } else {
                    uint4 *dst =
                        reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.out) + row * p.hidden + head * 128);
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        uint32_t w4[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const __nv_bfloat162 b2 = __floats2bfloat162_rn(o[8 * i + 2 * k], o[8 * i + 2 * k + 1]);
                            w4[k] = *reinterpret_cast<const uint32_t *>(&b2);
                        }
                        dst[i] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == WARP_MMA) tmem_dealloc(tmem, 512);
}

template <int GROUP, bool MIXED>
int launch_one(const CUtensorMap &tm, const AttnParams &p, dim3 grid, cudaStream_t s) {
    constexpr int smem = SmemLayout::BYTES;
    auto fn = attention_kernel<GROUP, MIXED>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess) {
        fn<<<grid, NUM_THREADS, smem, s>>>(tm, p);
        e = cudaGetLastError();
    }
    return report_cuda(e, "attention launch");
}

template <int GROUP>
int launch_group(const CUtensorMap &tm, const AttnParams &p, dim3 grid, bool mixed, cudaStream_t s) {
    return mixed ? launch_one<GROUP, true>(tm, p, grid, s) : launch_one<GROUP, false>(tm, p, grid, s);
}

}  // namespace

int launch_attention(const void *q, int64_t n_q, const RangeTable &ranges, int hidden, int group, float sm_scale,
                     int out_fp32, void *out, cudaStream_t s) {
    alignas(64) CUtensorMap tm_q;
    if (encode_tmap_2d(&tm_q, q, 1, static_cast<uint64_t>(hidden), static_cast<uint64_t>(n_q),
                       static_cast<uint64_t>(hidden) * 2, 64, BQT))
        return KVQ_ERR_CUDA;
    AttnParams p{};
    p.n_q = n_q;
    p.hidden = hidden;
    p.scale_log2 = sm_scale * 1.4426950408889634f;
    p.out_fp32 = out_fp32;
    p.out = out;
    p.ranges = ranges;
    int tiles = 0;
    bool mixed = false;
    for (int g = 0; g < ranges.n; ++g) {
        p.tiles_before[g] = tiles;
        tiles += static_cast<int>((ranges.r[g].len + BKV - 1) / BKV);
        if (ranges.r[g].bits != 4) mixed = true;
    }
    p.tiles_before[ranges.n] = tiles;
    p.total_tiles = tiles;
    dim3 grid(static_cast<unsigned>((n_q + BQ - 1) / BQ), static_cast<unsigned>(hidden / 128));
    if (group == 32) return launch_group<32>(tm_q, p, grid, mixed, s);
    if (group == 64) return launch_group<64>(tm_q, p, grid, mixed, s);
    return launch_group<128>(tm_q, p, grid, mixed, s);
}

cudaError_t read_clear_err_attn(unsigned int *v) {
    cudaError_t e = cudaMemcpyFromSymbol(v, g_err_attn, sizeof(unsigned int));
    if (e != cudaSuccess) return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_err_attn, &zero, sizeof(unsigned int));
}

}  // namespace kvq
