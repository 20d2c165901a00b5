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
// A cluster of two CTAs (a CTA pair on two SMs) works on one head and 512
// query rows; each CTA owns 256 of them as two 128-row tiles A and B.  The
// tensor core runs 256-row MMAs over the pair (tcgen05 cta_group::2): rows
// 0-127 from the even CTA, 128-255 from the odd one, while the B operand is
// split along N between the two SMs.  So each CTA decodes only half of every
// K/V tile: keys 64r .. 64r+63 of K^ (all 128 dims) and dims 64r .. 64r+63 of
// V^ (all 128 keys), r = the CTA's rank in the pair.  Tiles A and B take
// turns on the tensor core (ping-pong): while the softmax of tile A works on
// its scores, the tensor core runs tile B's P.V and next Q.K^T, and the other
// way round.  16 warps per CTA in four warpgroups:
//   WG0, WG1   softmax of tile A / B: one thread per query row; reads the S
//              row from TMEM, keeps a running max in the log2 domain and
//              rescales the output accumulator only when the row max grew by
//              more than 2^8 (the stale max is used consistently for P and the
//              row sum, so the result is exact); writes P as FP16 back into
//              the first 64 TMEM columns of its own S, and at the end divides
//              by the row sum, un-rotates the row with the 128-point fast
//              Walsh-Hadamard transform in registers and stores it.
//   WG2 + warps 14-15   dequantisers (192 threads): per 128-key tile, read
//              the INT4 / INT8 codes of the CTA's halves from a shared-memory
//              staging buffer and the fp16 scales from global memory (a tile
//              ahead), decode them with integer bit tricks into FP16
//              (code * scale) and store K^ and V^, both [key][dim], in the
//              128-byte-swizzled layout the tensor core reads (K^ as the
//              K-major B operand of Q.K^T, V^ as the MN-major B operand of
//              P.V^).  K^ is decoded as soon as the last Q.K^T of its stage
//              has run, V^ once the last P.V^ has.  The dims are permuted
//              inside each 8-dim chunk (the order e0 e4 e1 e5 e2 e6 e3 e7
//              falls out of the nibble decode): Q is permuted the same way
//              when it is converted, so Q.K^T is unchanged, and the output
//              columns come out in the same order and are put back in the
//              epilogue.  They also convert the CTA's BF16 Q tiles to FP16 once.
//   warp 12    TMA of the CTA's Q tiles, TMEM allocation (jointly with the
//              peer CTA) and, in the even CTA, the single MMA thread.
//   warp 13    bulk copies (TMA engine) of each tile's codes into the staging
//              ring, as far ahead as its three stages allow (three INT4
//              tiles, or one INT8 tile and part of the next).
// K^ and V^ have three shared-memory stages each, so the dequantisers can
// work up to two tiles ahead of the tensor core.
// The MMA thread waits on barriers of the even CTA that the threads of both
// CTAs arrive on; its commits arrive on the same barriers of both CTAs.
// Registers are redistributed with setmaxnreg: 168 per softmax thread, 88
// for the rest (512 threads x 128 at launch).
// TMEM (512 columns per CTA): S_A, S_B, O_A, O_B, 128 columns each; P_t
// aliases the first 64 columns of S_t.  tcgen05.mma instructions from one
// thread execute in issue order, so S_t(j+1), issued after P_t(j).V^(j),
// overwrites P_t(j) only after that MMA has read it; and the commit that
// signals S_t(j+1) also covers P_t(j).V^(j), so O_t is final for tile j when
// the softmax sees S_t(j+1).
// Scores, the softmax and O are fp32; the MMA operands are FP16 (11-bit
// significand: the rotation spreads values evenly, where BF16's 8 bits would
// cost a noticeably higher error floor).  No split over keys: every query
// row is computed by one CTA pair in one fixed order, so results do not
// depend on how the queries are tiled or chunked.
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
constexpr int KV_STAGES = 3;   // K^ / V^ shared-memory stages
constexpr int NUM_DQ_THREADS = 192;  // warps 8-11 and 14-15
constexpr int NUM_DQ_WARPS = NUM_DQ_THREADS / 32;
constexpr int NUM_SM_WARPS = 4;  // per query tile
constexpr int NUM_THREADS = 512;
constexpr int WARP_MMA = 12, WARP_LOAD = 13;
constexpr int REG_SOFTMAX = 168, REG_OTHER = 88;
static_assert(2 * 128 * REG_SOFTMAX + 2 * 128 * REG_OTHER <= NUM_THREADS * 128,
              "register split exceeds the launch budget");
constexpr int Q_TILE_BYTES = 128 * 128 * 2;  // 128 rows x 128 dims, as two 64-dim halves
constexpr int Q_HALF_BYTES = Q_TILE_BYTES / 2;
constexpr int K_TILE_BYTES = 64 * 128 * 2;  // the CTA's 64 keys x 128 dims, as two 64-dim halves
constexpr int K_HALF_BYTES = K_TILE_BYTES / 2;
constexpr int V_TILE_BYTES = 128 * 64 * 2;  // 128 keys x the CTA's 64 dims
constexpr uint16_t kPairMask = 0x3;
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
    int causal;      // 1: query row i (at key position q_pos0 + i) sees keys j <= q_pos0 + i
    int64_t q_pos0;  // single store only
    // Attention over one key chunk with a carried state (vram_lab.py's blockwise
    // attention and `_online_combine`): 0 for the one-call attention; otherwise
    // KVQ_PARTIAL_MERGE / KVQ_PARTIAL_FINAL bits, plus kPartial.
    int partial;
    float *o_acc;    // [n_q][hidden] fp32: normalised output so far, rotated basis
    float *lse_acc;  // [n_q][heads] fp32: log sum exp(s) over the keys so far
};
constexpr int kPartial = 4;  // set in AttnParams::partial for every key-chunk call

// Staging buffers of packed codes, filled by bulk copies: three 16 KB stages.
// An INT4 tile takes one stage: the CTA's 64 K rows (4 KB) at offset 0 and
// all 128 V rows (8 KB, of which the CTA decodes its half of each row) at
// offset 4096.  An INT8 tile takes two consecutive stages (in ring order):
// 64 K rows (8 KB) in the first, 128 V rows (16 KB) in the second.  The
// loader and the dequantisers walk the same running stage counter.
struct Staging {
    static constexpr int STAGES = 3;
    static constexpr int STAGE_BYTES = 16384;
    static constexpr int BYTES = STAGES * STAGE_BYTES;
    static constexpr int INT4_V_OFFSET = 4096;
};
__host__ __device__ constexpr int stages_of(int bits) { return bits == 8 ? 2 : 1; }

// Dynamic shared memory, 1024-byte aligned (checked at run time).
struct SmemLayout {
    static constexpr int Q = 0;                             // NQT tiles
    static constexpr int K = Q + NQT * Q_TILE_BYTES;        // KV_STAGES tiles
    static constexpr int V = K + KV_STAGES * K_TILE_BYTES;  // KV_STAGES tiles
    static constexpr int STG = V + KV_STAGES * V_TILE_BYTES;
    static constexpr int BAR = STG + Staging::BYTES;
    static constexpr int BYTES = BAR + 256;
};
static_assert((11 + 2 * Staging::STAGES + 3 * KV_STAGES) * 8 + 8 <= 256,
              "barriers and the TMEM slot overflow their area");
static_assert(SmemLayout::BYTES <= 227 * 1024, "dynamic shared memory above the per-CTA limit");

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
__device__ __forceinline__ float lg2_approx(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
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

// The tile sequence walks the ranges in order: tile j of the sequence is
// local tile j - tiles_before[g] of range g.  Every role walks it with its own
// cursor, one step per tile.
struct TileRef {
    int g;         // range
    int lt;        // tile inside the range
    int64_t key0;  // first key (row) of the tile inside range g
    int valid;     // keys of the tile that exist (1..128)
};
struct TileCursor {
    int g = 0, lt = 0;
    __device__ __forceinline__ TileRef ref(const AttnParams &p) const {
        TileRef t;
        t.g = g;
        t.lt = lt;
        t.key0 = static_cast<int64_t>(lt) * BKV;
        const int64_t rem = p.ranges.r[g].len - t.key0;
        t.valid = rem < BKV ? static_cast<int>(rem) : BKV;
        return t;
    }
    __device__ __forceinline__ void next(const AttnParams &p) {
        if (++lt == p.tiles_before[g + 1] - p.tiles_before[g]) {
            lt = 0;
            ++g;
        }
    }
};

// A tile's decode work in one CTA is split into units of 16 staged code
// bytes: UK units of the CTA's 64 K rows (all 128 dims: cpr = 4 columns of
// 16 bytes per row for INT4, 8 for INT8), then UV units of the CTA's half of
// the 128 V rows (cpr / 2 columns per row).  Dequantiser d takes units d,
// d + 192, d + 384, ...; a warp's 32 consecutive units are all K or all V.
//
// 16-byte shared-memory accesses are served eight lanes at a time, and each
// group of eight takes one pass when it touches eight different 16-byte bank
// positions.  K units are dealt to lanes so that both the code loads (row
// stride 64 or 128 bytes) and the swizzled operand stores (position
// ((dims / 8) mod 8) xor (row mod 8)) of every group of eight lanes fall on
// eight distinct positions:
//   INT4: lanes 8p..8p+7 take rows {2a, 2a+1} x columns {0, 1} and rows
//         {2b, 2b+1} x columns {2, 3}, {a, b} = {0, 1} xor (p & 1), in row
//         block 4 (p >> 1);
//   INT8: lanes 8p..8p+7 take columns 0..3 of one row and 4..7 of the other
//         row of the pair 2 (p >> 1), {0, 1} in the order p & 1.
// V units go row-major (four rows x two columns, or two rows x four columns,
// per group of eight): conflict-free stores, two-way conflicting loads, as
// only half of each staged V row is read.
template <int BITS>
struct UnitPlan {
    static constexpr int LG = BITS == 8 ? 3 : 2;  // log2 of 16-byte code columns per key row
    static constexpr int UK = 64 << LG;           // K units
    static constexpr int UV = 128 << (LG - 1);    // V units
    static constexpr int MAX_UNITS = (UK + UV + NUM_DQ_THREADS - 1) / NUM_DQ_THREADS;
    static constexpr int CPC = BITS == 8 ? 2 : 4;  // 8-dim chunks per 16-byte column
    // key row r (0..63) and code column cc of K unit rem
    static __device__ __forceinline__ void k_rc(int rem, int &r, int &cc) {
        const int x = rem & 31, swap = ((x >> 2) ^ (x >> 3)) & 1;
        if constexpr (BITS == 4) {
            r = ((rem >> 5) << 3) + ((x >> 4) << 2) + (swap << 1) + (x & 1);
            cc = ((x >> 1) & 1) | (((x >> 2) & 1) << 1);
        } else {
            r = ((rem >> 5) << 2) + ((x >> 4) << 1) + swap;
            cc = x & 7;
        }
    }
    // key row r (0..127) and code column c2 (0 .. cpr/2 - 1, inside the CTA's half) of V unit rem
    static __device__ __forceinline__ void v_rc(int rem, int &r, int &c2) {
        r = rem >> (LG - 1);
        c2 = rem & ((1 << (LG - 1)) - 1);
    }
};
constexpr int kMaxUnits = UnitPlan<8>::MAX_UNITS;

// fp16 scale of each unit of dequantiser d for tile t (0 for rows past the
// tile's valid keys), loaded straight from global memory one tile ahead.
template <int GROUP, int BITS>
__device__ __forceinline__ void load_scales(const AttnParams &p, int head, uint32_t rank, const TileRef &t, int d,
                                            uint32_t (&sc)[kMaxUnits]) {
    using U = UnitPlan<BITS>;
    constexpr int SG = 128 / GROUP;
    const RangeDev &rg = p.ranges.r[t.g];
    const int64_t row0 = static_cast<int64_t>(head) * rg.cap + t.key0;
#pragma unroll
    for (int i = 0; i < U::MAX_UNITS; ++i) {
        const int u = d + NUM_DQ_THREADS * i;
        int key, cc;
        const uint16_t *base;
        if (u < U::UK) {
            U::k_rc(u, key, cc);
            key += 64 * static_cast<int>(rank);
            base = rg.k_scales;
        } else {
            int c2;
            U::v_rc(u - U::UK, key, c2);
            cc = (static_cast<int>(rank) << (U::LG - 1)) + c2;
            base = rg.v_scales;
        }
        const int g = (cc << (7 - U::LG)) / GROUP;  // column x dims per column / GROUP
        sc[i] = (u < U::UK + U::UV && key < t.valid) ? static_cast<uint32_t>(__ldg(base + (row0 + key) * SG + g))
                                                      : 0u;
    }
}

// Decodes unit u of a staged tile into the CTA's K^ half ([64 keys][128
// dims] as two 64-dim halves) or V^ half ([128 keys][64 dims]), 128-byte
// swizzle, dims permuted inside each 8-dim chunk; rows past `valid` become zeros.
template <int BITS>
__device__ __forceinline__ void decode_unit(const uint8_t *stg_k, const uint8_t *stg_v, int u, int valid,
                                            uint32_t rank, uint32_t scale, uint8_t *k_tile, uint8_t *v_tile) {
    using U = UnitPlan<BITS>;
    constexpr int ROW_BYTES = 16 << U::LG;
    const uint8_t *src;
    uint8_t *dst;
    uint32_t c0, r7;  // first 8-dim chunk of the unit inside its 128-byte row, row swizzle
    bool live;
    if (u < U::UK) {
        int r, cc;
        U::k_rc(u, r, cc);
        src = stg_k + r * ROW_BYTES + cc * 16;
        const int c = cc * U::CPC;  // 0..15 over the 128 dims
        dst = k_tile + (c >> 3) * K_HALF_BYTES + r * 128;
        c0 = static_cast<uint32_t>(c & 7);
        r7 = static_cast<uint32_t>(r & 7);
        live = 64 * static_cast<int>(rank) + r < valid;
    } else {
        int r, c2;
        U::v_rc(u - U::UK, r, c2);
        src = stg_v + r * ROW_BYTES + ((static_cast<int>(rank) << (U::LG - 1)) + c2) * 16;
        dst = v_tile + r * 128;
        c0 = static_cast<uint32_t>(c2 * U::CPC);  // 0..7 over the CTA's 64 dims
        r7 = static_cast<uint32_t>(r & 7);
        live = r < valid;
    }
    const uint4 w = *reinterpret_cast<const uint4 *>(src);
    const uint32_t s2 = h2_dup(static_cast<uint16_t>(scale));
    if constexpr (BITS == 4) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {  // dims 32cc + 8k .. +7
            uint32_t o[4] = {0u, 0u, 0u, 0u};
            if (live) dq_int4_word((&w.x)[k], s2, o);
            *reinterpret_cast<uint4 *>(dst + (((c0 + k) ^ r7) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
        }
    } else {
#pragma unroll
        for (int k = 0; k < 2; ++k) {  // dims 16cc + 8k .. +7
            const uint32_t a = (&w.x)[2 * k], b = (&w.x)[2 * k + 1];
            uint32_t o[4] = {0u, 0u, 0u, 0u};
            if (live) {
                o[0] = dq_int8_pair(a, b, 0x0400u, s2);
                o[1] = dq_int8_pair(a, b, 0x0501u, s2);
                o[2] = dq_int8_pair(a, b, 0x0602u, s2);
                o[3] = dq_int8_pair(a, b, 0x0703u, s2);
            }
            *reinterpret_cast<uint4 *>(dst + (((c0 + k) ^ r7) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
}

// Decodes the dequantiser's units of one tile: K units first (once the K^
// stage is free), then V units (once the V^ stage is free).  Every wait result
// is made warp-uniform, so a warp leaves together.
template <int BITS>
__device__ __forceinline__ bool decode_tile(const uint8_t *stg_k, const uint8_t *stg_v, int d, int valid,
                                            uint32_t rank, const uint32_t (&sc)[kMaxUnits], uint8_t *kt,
                                            uint8_t *vt, uint64_t *k_empty, uint64_t *v_empty, uint32_t ph,
                                            volatile int *abort_flag) {
    using U = UnitPlan<BITS>;
    if (!__all_sync(0xffffffffu, mbar_wait(k_empty, ph, abort_flag, &g_err_attn))) return false;
    bool v_free = false;
#pragma unroll
    for (int i = 0; i < U::MAX_UNITS; ++i) {
        const int u = d + NUM_DQ_THREADS * i;
        if (u >= U::UK + U::UV) break;
        if (u >= U::UK && !v_free) {
            if (!__all_sync(0xffffffffu, mbar_wait(v_empty, ph, abort_flag, &g_err_attn))) return false;
            v_free = true;
        }
        decode_unit<BITS>(stg_k, stg_v, u, valid, rank, sc[i], kt, vt);
    }
    return v_free || __all_sync(0xffffffffu, mbar_wait(v_empty, ph, abort_flag, &g_err_attn));
}

// First query row of this CTA, recomputed where needed (from a special
// register) rather than kept live.  Causal pairs go in row order too: running
// them longest first (reversed) measured 0.7 % slower at N = 152,263, with
// every head's pairs dispatched one head after another either way.
template <bool CAUSAL>
__device__ __forceinline__ int64_t cta_row0() {
    return static_cast<int64_t>(blockIdx.x) * BQ;
}
// Key tiles this CTA pair walks: all of them, or (causal) those up to the
// position of the pair's last query row; both CTAs of a pair get the same count.
template <bool CAUSAL>
__device__ __forceinline__ int cta_tiles(const AttnParams &p) {
    if (!CAUSAL) return p.total_tiles;
    const int64_t first = cta_row0<true>() & ~int64_t(2 * BQ - 1);  // the pair's first row
    const int64_t end = p.n_q < first + 2 * BQ ? p.n_q : first + 2 * BQ;
    const int64_t need = (p.q_pos0 + end - 1) / BKV + 1;
    return need < p.total_tiles ? static_cast<int>(need) : p.total_tiles;
}

// A shared-memory matrix descriptor moved by `bytes`: the start address is
// the low 14-bit field (address / 16), and shared-memory addresses stay below
// 2^18 bytes, so the sum never carries out of it.  Descriptors are built once
// and moved with one 32-bit add per MMA.
__device__ __forceinline__ uint64_t desc_add(uint64_t d, uint32_t bytes) {
    return (d & 0xFFFFFFFF00000000ull) | static_cast<uint32_t>(static_cast<uint32_t>(d) + (bytes >> 4));
}

__device__ __forceinline__ void tmem_ld128(uint32_t taddr, uint32_t (&r)[128]) {
    tmem_ld32(taddr + 0, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
    tmem_ld32(taddr + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
    tmem_ld32(taddr + 64, *reinterpret_cast<uint32_t(*)[32]>(&r[64]));
    tmem_ld32(taddr + 96, *reinterpret_cast<uint32_t(*)[32]>(&r[96]));
    tmem_ld_wait();
}

template <int GROUP, bool MIXED, bool CAUSAL>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    attention_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ AttnParams p) {
    using L = SmemLayout;
    using SL = Staging;
    extern __shared__ __align__(1024) uint8_t smem[];
    // Both CTAs of a pair see the same offsets, so both leave here or neither does.
    if (smem_u32(smem) & 1023u) {  // the layout below assumes a 1024-byte aligned base
        if (threadIdx.x == 0) atomicOr(&g_err_attn, 2u);
        return;
    }
    uint8_t *sQ = smem + L::Q;
    uint8_t *sK = smem + L::K;
    uint8_t *sV = smem + L::V;
    uint8_t *sStg = smem + L::STG;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::BAR);
    uint64_t *q_tma = bars + 0;
    uint64_t *q_ready = bars + 1;             // even CTA: Q of both CTAs converted
    uint64_t *s_full = bars + 2;              // [NQT]
    uint64_t *p_full = bars + 4;              // [NQT], even CTA: P of both CTAs in TMEM
    uint64_t *p_half = bars + 6;              // [NQT], even CTA: P of keys 0-63 of both CTAs in TMEM
    uint64_t *pv_done = bars + 8;             // [NQT]
    uint64_t *stg_full = bars + 10;              // [SL::STAGES]
    uint64_t *stg_empty = stg_full + SL::STAGES;  // [SL::STAGES]
    uint64_t *drain = stg_empty + SL::STAGES;    // even CTA: every MMA has completed
    uint64_t *kv_full = drain + 1;               // [KV_STAGES], even CTA: both CTAs' halves decoded
    uint64_t *k_empty = kv_full + KV_STAGES;  // [KV_STAGES]: K^ stage read by its last Q.K^T
    uint64_t *v_empty = k_empty + KV_STAGES;  // [KV_STAGES]: V^ stage read by its last P.V^
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(v_empty + KV_STAGES);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int head = blockIdx.y;
    const int T = cta_tiles<CAUSAL>(p);

    if (threadIdx.x == 0) {
        mbar_init(q_tma, 1);
        mbar_init(q_ready, 2 * NUM_DQ_WARPS);
        for (int i = 0; i < KV_STAGES; ++i) {
            mbar_init(&kv_full[i], 2 * NUM_DQ_WARPS);
            mbar_init(&k_empty[i], 1);
            mbar_init(&v_empty[i], 1);
        }
        for (int i = 0; i < NQT; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], 2 * NUM_SM_WARPS);
            mbar_init(&p_half[i], 2 * NUM_SM_WARPS);
            mbar_init(&pv_done[i], 1);
        }
        for (int i = 0; i < SL::STAGES; ++i) {
            mbar_init(&stg_full[i], 1);
            mbar_init(&stg_empty[i], NUM_DQ_THREADS);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == WARP_MMA) {
        tmem_alloc_pair(tmem_slot, 512);
        tmem_relinquish_pair();
    }
    // the peer may arrive on this CTA's barriers only once they are initialised
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp >= 8) {
    setmaxnreg_dec<REG_OTHER>();  // WG2 and WG3, one instruction for both warpgroups
    if (warp == WARP_MMA || warp == WARP_LOAD) {
        // ------------------------------------------------------------ warp 12: Q load + MMA issue
        if (warp == WARP_MMA) {
            if (elect_one()) {
                prefetch_tmap(&tm_q);
                mbar_arrive_expect_tx(q_tma, NQT * Q_TILE_BYTES);
#pragma unroll
                for (int t = 0; t < NQT; ++t) {
                    const int y = static_cast<int>(cta_row0<CAUSAL>()) + t * BQT;
                    tma_load_2d(sQ + t * Q_TILE_BYTES, &tm_q, q_tma, head * 128, y);
                    tma_load_2d(sQ + t * Q_TILE_BYTES + Q_HALF_BYTES, &tm_q, q_tma, head * 128 + 64, y);
                }
                if (rank == 0) {
                    constexpr uint32_t idesc = make_idesc_f16(256, 128, 0);
                    constexpr uint32_t idesc_pv = make_idesc_f16(256, 128, 0, 1);  // V^ [key][dim]: MN-major B
                    const uint32_t qa = smem_u32(sQ);
                    bool ok = mbar_wait_cluster(q_ready, 0, abort_flag, &g_err_attn);
                    tc_fence_after();
                    const uint64_t dq = make_sdesc_sw128(qa);
                    const uint64_t dk = make_sdesc_sw128(smem_u32(sK));
                    const uint64_t dv = make_sdesc_sw128_mn(smem_u32(sV), V_TILE_BYTES);
                    auto issue_s = [&](int j, int t) {  // S_t(j) = Q_t . K^_j^T over the pair
                        const uint64_t kd = desc_add(dk, (j % KV_STAGES) * K_TILE_BYTES);
                        const uint32_t d = tmem + tm_s(t);
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const uint32_t kin = (k >> 2) * Q_HALF_BYTES + (k & 3) * 32;
                            mma_f16_ss_pair(d, desc_add(dq, t * Q_TILE_BYTES + kin),
                                            desc_add(kd, (k >> 2) * K_HALF_BYTES + (k & 3) * 32), idesc, k > 0);
                        }
                        mma_commit_pair(&s_full[t], kPairMask);
                    };
                    if (ok && T > 0) {
                        ok = mbar_wait_cluster(&kv_full[0], 0, abort_flag, &g_err_attn);
                        if (ok) {
                            tc_fence_after();
                            issue_s(0, 0);
                            issue_s(0, 1);
                            mma_commit_pair(&k_empty[0], kPairMask);
                        }
                    }
                    for (int j = 0; ok && j < T; ++j) {
                        const int st = j % KV_STAGES;
                        const uint64_t vd = desc_add(dv, st * V_TILE_BYTES);
                        for (int t = 0; t < NQT && ok; ++t) {
                            // O_t += P_t(j) . V^_j, P_t read from TMEM (the first 64 columns of S_t);
                            // keys 0-63 go as soon as their P is written, keys 64-127 after
#pragma unroll
                            for (int hf = 0; hf < 2; ++hf) {
                                ok = mbar_wait_cluster(hf == 0 ? &p_half[t] : &p_full[t], j & 1, abort_flag,
                                                       &g_err_attn);
                                if (!ok) break;
                                tc_fence_after();
#pragma unroll
                                for (int k = 4 * hf; k < 4 * hf + 4; ++k) {  // keys 16k .. 16k+15: 16 rows of V^
                                    mma_f16_ts_pair(tmem + tm_o(t), tmem + tm_s(t) + k * 8,
                                                    desc_add(vd, k * 2048), idesc_pv,
                                                    (j > 0 || k > 0) ? 1u : 0u);
                                }
                            }
                            if (!ok) break;
                            mma_commit_pair(&pv_done[t], kPairMask);
                            if (t == NQT - 1) mma_commit_pair(&v_empty[st], kPairMask);
                            if (j + 1 < T) {
                                if (t == 0) {
                                    ok = mbar_wait_cluster(&kv_full[(j + 1) % KV_STAGES], ((j + 1) / KV_STAGES) & 1,
                                                           abort_flag, &g_err_attn);
                                    if (!ok) break;
                                    tc_fence_after();
                                }
                                issue_s(j + 1, t);
                                if (t == NQT - 1) mma_commit_pair(&k_empty[(j + 1) % KV_STAGES], kPairMask);
                            }
                        }
                    }
                    // drain: every MMA this thread issued has completed before the pair tears down
                    volatile int no_abort = 0;
                    mma_commit_pair(drain, 0x1);
                    mbar_wait(drain, 0, &no_abort, nullptr, 1000000000ull);
                }
                volatile int no_abort = 0;
                mbar_wait(q_tma, 0, &no_abort, nullptr);
            }
            __syncwarp();
        } else {
            // ------------------------------------------------------------ bulk copies of the codes
            if (elect_one()) {
                uint32_t armed = 0, armed_parity = 0;
                int k = 0;  // running stage counter
                TileCursor cur;
                for (int j = 0; j < T && !*abort_flag; ++j, cur.next(p)) {
                    const TileRef tr = cur.ref(p);
                    const RangeDev &rg = p.ranges.r[tr.g];
                    const int bits = MIXED ? rg.bits : 4;
                    const uint32_t cb = bits == 8 ? 128u : 64u;  // code bytes per key row
                    const int64_t row0 = static_cast<int64_t>(head) * rg.cap + tr.key0;
                    const uint8_t *ksrc = rg.k_codes + (row0 + 64 * static_cast<int64_t>(rank)) * cb;
                    const uint8_t *vsrc = rg.v_codes + row0 * cb;
                    bool fine = true;
                    for (int c = 0; c < stages_of(bits) && fine; ++c) {
                        const int s = (k + c) % SL::STAGES;
                        const uint32_t ph = static_cast<uint32_t>(((k + c) / SL::STAGES) & 1);
                        fine = mbar_wait(&stg_empty[s], ph ^ 1u, abort_flag, &g_err_attn);
                        if (!fine) break;
                        uint8_t *dst = sStg + s * SL::STAGE_BYTES;
                        if (bits == 4) {  // K and V codes share the stage
                            mbar_arrive_expect_tx(&stg_full[s], 64u * cb + 128u * cb);
                            bulk_load(dst, ksrc, 64u * cb, &stg_full[s]);
                            bulk_load(dst + SL::INT4_V_OFFSET, vsrc, 128u * cb, &stg_full[s]);
                        } else if (c == 0) {  // K codes in the first stage
                            mbar_arrive_expect_tx(&stg_full[s], 64u * cb);
                            bulk_load(dst, ksrc, 64u * cb, &stg_full[s]);
                        } else {  // V codes in the second
                            mbar_arrive_expect_tx(&stg_full[s], 128u * cb);
                            bulk_load(dst, vsrc, 128u * cb, &stg_full[s]);
                        }
                        armed |= 1u << s;
                        armed_parity = (armed_parity & ~(1u << s)) | (ph << s);
                    }
                    if (!fine) break;
                    k += stages_of(bits);
                }
                // drain: the last copies have landed before the CTA exits
                volatile int no_abort = 0;
                for (int s = 0; s < SL::STAGES; ++s)
                    if (armed & (1u << s)) mbar_wait(&stg_full[s], (armed_parity >> s) & 1u, &no_abort, nullptr);
            }
            __syncwarp();
        }
    } else {
        // ------------------------------------------------------------ dequantisers (warps 8-11, 14-15)
        const int d = warp < 12 ? static_cast<int>(threadIdx.x) - 256 : static_cast<int>(threadIdx.x) - 448 + 128;
        // Q: BF16 -> FP16 in place, dims permuted e0 e4 e1 e5 e2 e6 e3 e7 within each 8-chunk
        const bool ok = __all_sync(0xffffffffu, mbar_wait(q_tma, 0, abort_flag, &g_err_attn));
        if (ok) {
#pragma unroll 2
            for (int i = d; i < NQT * Q_TILE_BYTES / 16; i += NUM_DQ_THREADS) {
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
            __syncwarp();
            // the even CTA's barrier, in the cluster window
            if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(q_ready), 0));
        }
        uint32_t sc[kMaxUnits];
        TileCursor cur, ahead;  // tile j, and tile j + 1 for the scale loads
        auto prefetch_scales = [&]() {
            const TileRef ta = ahead.ref(p);
            if (!MIXED || p.ranges.r[ta.g].bits == 4) load_scales<GROUP, 4>(p, head, rank, ta, d, sc);
            else load_scales<GROUP, 8>(p, head, rank, ta, d, sc);
            ahead.next(p);
        };
        if (ok && T > 0) prefetch_scales();
        int k = 0;  // running stage counter, as the loader's
        int j = 0;
        bool going = ok;
        // Tiles go in stretches of one precision, each through a loop compiled for it,
        // so an INT4 stretch runs the same code as the INT4-only kernel.
        auto stretch = [&](auto bits_c) {
            constexpr int BITS = decltype(bits_c)::value;
            const int g0 = cur.g;
            for (; j < T && (!MIXED || cur.g == g0); ++j, cur.next(p)) {
                const int st = j % KV_STAGES;
                const uint32_t ph = ((j / KV_STAGES) & 1) ^ 1;
                const TileRef tr = cur.ref(p);
                const int s0 = k % SL::STAGES, s1 = (k + stages_of(BITS) - 1) % SL::STAGES;
                if (*abort_flag ||
                    !__all_sync(0xffffffffu, mbar_wait(&stg_full[s0], (k / SL::STAGES) & 1, abort_flag, &g_err_attn)) ||
                    (BITS == 8 && !__all_sync(0xffffffffu, mbar_wait(&stg_full[s1], ((k + 1) / SL::STAGES) & 1,
                                                                     abort_flag, &g_err_attn)))) {
                    going = false;
                    return;
                }
                const uint8_t *stg_k = sStg + s0 * SL::STAGE_BYTES;
                const uint8_t *stg_v = BITS == 8 ? sStg + s1 * SL::STAGE_BYTES : stg_k + SL::INT4_V_OFFSET;
                uint8_t *kt = sK + st * K_TILE_BYTES;
                uint8_t *vt = sV + st * V_TILE_BYTES;
                if (!decode_tile<BITS>(stg_k, stg_v, d, tr.valid, rank, sc, kt, vt, &k_empty[st], &v_empty[st], ph,
                                       abort_flag)) {
                    going = false;
                    return;
                }
                mbar_arrive(&stg_empty[s0]);  // every staged byte of this tile has been read
                if (BITS == 8) mbar_arrive(&stg_empty[s1]);
                k += stages_of(BITS);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&kv_full[st]), 0));
                if (j + 1 < T) prefetch_scales();
            }
        };
        while (going && j < T) {
            if (!MIXED || p.ranges.r[cur.g].bits == 4) stretch(std::integral_constant<int, 4>{});
            else stretch(std::integral_constant<int, 8>{});
        }
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
        TileCursor cur;
        for (int j = 0; j < T; ++j, cur.next(p)) {
            // the wait result is made warp-uniform before any warp-collective TMEM access
            if (!__all_sync(0xffffffffu, mbar_wait(&s_full[t], j & 1, abort_flag, &g_err_attn))) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sr[128];
            tmem_ld128(sa, sr);
            int nvis = cur.ref(p).valid;  // keys of this tile the row sees
            if constexpr (CAUSAL) {
                const int64_t lim = p.q_pos0 + cta_row0<true>() + t * BQT + r - static_cast<int64_t>(j) * BKV + 1;
                if (lim < nvis) nvis = lim < 0 ? 0 : static_cast<int>(lim);
            }
            if (nvis < BKV) {
#pragma unroll
                for (int c = 0; c < 128; ++c)
                    if (c >= nvis) sr[c] = __float_as_uint(-INFINITY);
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
            // p = 2^(s*sl - m) as FP16 pairs, packed over S's first 64 columns, in two
            // halves of 64 keys: the MMA starts on keys 0-63 while keys 64-127 are computed
            const uint64_t sl2 = f2_pack(sl, sl), nm2 = f2_pack(-m, -m);
            uint64_t acc0 = f2_pack(0.0f, 0.0f), acc1 = acc0;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                uint32_t pk[32];
#pragma unroll
                for (int c = 64 * hf; c < 64 * hf + 64; c += 4) {
                    const uint64_t a0 =
                        f2_fma(f2_pack(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), sl2, nm2);
                    const uint64_t a1 =
                        f2_fma(f2_pack(__uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3])), sl2, nm2);
                    float x0, x1, x2, x3;
                    f2_unpack(a0, x0, x1);
                    f2_unpack(a1, x2, x3);
                    x0 = ex2_approx(x0);
                    x1 = ex2_approx(x1);
                    x2 = ex2_approx(x2);
                    x3 = ex2_approx(x3);
                    const __half2 h0 = __floats2half2_rn(x0, x1);
                    const __half2 h1 = __floats2half2_rn(x2, x3);
                    pk[(c - 64 * hf) >> 1] = *reinterpret_cast<const uint32_t *>(&h0);
                    pk[((c - 64 * hf) >> 1) + 1] = *reinterpret_cast<const uint32_t *>(&h1);
                    // the row sum takes the fp32 weights (the MMA sees them rounded to FP16,
                    // a relative 2^-12 per weight that averages out in the sum)
                    acc0 = f2_add(acc0, f2_pack(x0, x1));
                    acc1 = f2_add(acc1, f2_pack(x2, x3));
                }
                // S_t(j) completing implies P_t(j-1).V^(j-1) completed: O_t is final for
                // j-1 and is rescaled before the first P_t(j).V^(j) is issued
                if (hf == 0 && rescale && j > 0) {
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
                tmem_st16(sa + 32 * hf, *reinterpret_cast<const uint32_t(*)[16]>(&pk[0]));
                tmem_st16(sa + 32 * hf + 16, *reinterpret_cast<const uint32_t(*)[16]>(&pk[16]));
                tmem_st_wait();  // also covers the O rescale above
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(hf == 0 ? &p_half[t] : &p_full[t]), 0));
            }
            float u0, u1, u2, u3;
            f2_unpack(acc0, u0, u1);
            f2_unpack(acc1, u2, u3);
            l = l * alpha + ((u0 + u1) + (u2 + u3));
        }
        // epilogue: O / l, un-rotate, store
        if (ok && T > 0 && __all_sync(0xffffffffu, mbar_wait(&pv_done[t], (T - 1) & 1, abort_flag, &g_err_attn))) {
            tc_fence_after();
            const int64_t row = cta_row0<CAUSAL>() + t * BQT + r;
            const float inv_l = 1.0f / l;
            // Key-chunk calls that carry a state: this chunk's o = O / l and its
            // log-sum-exp ln sum_j e^(s_j tau) = (m + log2 l) ln 2 (the weights are
            // 2^(s_j tau log2 e - m)), merged into the state as `_online_combine`
            // does: new = ln(e^lse_acc + e^lse), o = o_acc e^(lse_acc - new) + o e^(lse - new).
            // O leaves TMEM 32 columns at a time straight into the state, so no more
            // than 32 columns are live during the merge.  A final call then reads
            // the merged row back for the un-rotation.  The weights use the hardware
            // exp2 / log2 approximations (relative error about 1e-7).
            const int partial = CAUSAL ? 0 : p.partial;  // key-chunk calls are never causal
            const bool merge = partial & KVQ_PARTIAL_MERGE, final = partial & KVQ_PARTIAL_FINAL;
            const bool via_state = partial && (merge || !final);
            if (via_state) {
                constexpr float kLn2 = 0.69314718055994531f, kLog2e = 1.4426950408889634f;
                const bool live = row < p.n_q;
                float *acc = p.o_acc + (live ? row : 0) * p.hidden + head * 128;
                float *lacc = p.lse_acc + (live ? row : 0) * (p.hidden >> 7) + head;
                const float lc2 = m + lg2_approx(l);
                float nw = lc2, wa = 0.0f, wc = inv_l;
                if (merge && live) {
                    const float la2 = *lacc * kLog2e;
                    const float hi = fmaxf(la2, lc2), lo = fminf(la2, lc2);
                    nw = hi + lg2_approx(1.0f + ex2_approx(lo - hi));
                    wa = ex2_approx(la2 - nw);
                    wc = ex2_approx(lc2 - nw) * inv_l;
                }
#pragma unroll 1
                for (int c0 = 0; c0 < 128; c0 += 32) {
                    uint32_t oc[32];
                    tmem_ld32(oa + c0, oc);  // warp-wide: every lane loads, live or not
                    tmem_ld_wait();
                    if (live) {
                        float4 *dst = reinterpret_cast<float4 *>(acc + c0);
#pragma unroll
                        for (int c = 0; c < 32; c += 8) {  // columns e0 e4 e1 e5 e2 e6 e3 e7 -> dims e0..e7
                            float v[8];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                v[e] = __fmul_rn(__uint_as_float(oc[c + 2 * e]), wc);
                                v[4 + e] = __fmul_rn(__uint_as_float(oc[c + 2 * e + 1]), wc);
                            }
                            if (merge) {
                                const float4 a0 = dst[c / 4], a1 = dst[c / 4 + 1];
                                v[0] = fmaf(a0.x, wa, v[0]);
                                v[1] = fmaf(a0.y, wa, v[1]);
                                v[2] = fmaf(a0.z, wa, v[2]);
                                v[3] = fmaf(a0.w, wa, v[3]);
                                v[4] = fmaf(a1.x, wa, v[4]);
                                v[5] = fmaf(a1.y, wa, v[5]);
                                v[6] = fmaf(a1.z, wa, v[6]);
                                v[7] = fmaf(a1.w, wa, v[7]);
                            }
                            dst[c / 4] = make_float4(v[0], v[1], v[2], v[3]);
                            dst[c / 4 + 1] = make_float4(v[4], v[5], v[6], v[7]);
                        }
                    }
                }
                if (live && !final) *lacc = nw * kLn2;
            }
            if (!via_state || final) {
                float o[128];
                if (via_state) {  // the merged row, back from the state (this thread's own writes)
                    const float4 *src = reinterpret_cast<const float4 *>(
                        p.o_acc + (row < p.n_q ? row : 0) * p.hidden + head * 128);
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float4 a = row < p.n_q ? src[i] : make_float4(0.f, 0.f, 0.f, 0.f);
                        o[4 * i] = a.x;
                        o[4 * i + 1] = a.y;
                        o[4 * i + 2] = a.z;
                        o[4 * i + 3] = a.w;
                    }
                } else {
                    uint32_t oraw[128];
                    tmem_ld128(oa, oraw);
                    // V^'s dims, hence O's columns, are in the order e0 e4 e1 e5 e2 e6 e3 e7 per 8-dim chunk.
                    // The products are rounded on their own (never contracted into the first
                    // butterfly), so every instantiation of the kernel gives the same bits.
#pragma unroll
                    for (int c = 0; c < 128; c += 8) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            o[c + e] = __fmul_rn(__uint_as_float(oraw[c + 2 * e]), inv_l);
                            o[c + 4 + e] = __fmul_rn(__uint_as_float(oraw[c + 2 * e + 1]), inv_l);
                        }
                    }
                }
                rotate128_thread(o);
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
    }

    // neither CTA of the pair leaves (or frees TMEM) while the other may still
    // arrive on its barriers or the MMAs may still touch its memory
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    if (warp == WARP_MMA) tmem_dealloc_pair(tmem, 512);
}

template <int GROUP, bool MIXED, bool CAUSAL>
int launch_one(const CUtensorMap &tm, const AttnParams &p, dim3 grid, cudaStream_t s) {
    constexpr int smem = SmemLayout::BYTES;
    auto fn = attention_kernel<GROUP, MIXED, CAUSAL>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess) {
        fn<<<grid, NUM_THREADS, smem, s>>>(tm, p);
        e = cudaGetLastError();
    }
    return report_cuda(e, "attention launch");
}

template <int GROUP>
int launch_group(const CUtensorMap &tm, const AttnParams &p, dim3 grid, bool mixed, cudaStream_t s) {
    if (p.causal) return launch_one<GROUP, false, true>(tm, p, grid, s);  // single INT4 store
    return mixed ? launch_one<GROUP, true, false>(tm, p, grid, s) : launch_one<GROUP, false, false>(tm, p, grid, s);
}

}  // namespace

int launch_attention(const void *q, int64_t n_q, const RangeTable &ranges, int hidden, int group, float sm_scale,
                     int out_fp32, void *out, cudaStream_t s, int causal, int64_t q_pos0, int partial_flags,
                     float *o_acc, float *lse_acc) {
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
    p.causal = causal;
    p.q_pos0 = q_pos0;
    p.partial = partial_flags < 0 ? 0 : (partial_flags | kPartial);
    p.o_acc = o_acc;
    p.lse_acc = lse_acc;
    // CTA pairs: an even number of CTAs of BQ query rows each
    const int64_t pairs = (n_q + 2 * BQ - 1) / (2 * BQ);
    dim3 grid(static_cast<unsigned>(2 * pairs), static_cast<unsigned>(hidden / 128));
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
