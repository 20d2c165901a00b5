// qkv_proj.cu -- streamed fused QKV projection on the 5th-generation tensor
// cores, with the Q / K / V epilogue fused in.
//
// The comfy-kitchen feature request ("Proposed backend capability") asks for
// a streamed/tiled QKV GEMM that never materialises the full high-precision
// [N, 3*hidden] output: Q is kept in BF16, K and V go through rotate ->
// quantise -> packed 4-bit storage inside the projection.  vram_lab.py's
// `_phase1_kv` fixes the fused row layout ([q | k | v], heads of 128
// contiguous columns) and `_norm_rope` the per-head RMSNorm of Q and K.
//
// Design (CTA pairs on two SMs, persistent, one pair per two SMs):
//   tile       256 tokens x 256 output columns (two heads) per pair, K-step 64;
//              each CTA owns 128 of the tokens
//   warp 0     TMA producer of each CTA: its 128 rows of x and its half (128
//              rows) of the tile's W rows per stage, 128-byte swizzle,
//              6-stage shared-memory ring.  The copies of both CTAs complete
//              on the even CTA's barrier of the stage (the CTA-pair form of
//              the TMA load), which the even producer arms for both CTAs' bytes.
//   warp 1     TMEM allocation (jointly with the peer).  In the even CTA the
//              MMA issuer: tcgen05.mma.cta_group::2 kind::f16 M=256 N=256
//              K=16 (rows 0-127 from the even CTA, 128-255 from the odd one;
//              B split along N between the two SMs), fp32 accumulators in each
//              CTA's TMEM, two 256-column accumulators so the epilogue of one
//              tile overlaps the main loop of the next.
//   warps 2-5  epilogue of each CTA on its own 128 rows: one thread per token
//              row reads a head's 128 fp32 values from TMEM (tcgen05.ld
//              32x32b), applies RMSNorm (Q, K, optional), the 128-point
//              rotation, and writes Q as BF16 or K / V as group-scaled INT4 /
//              INT8 codes into the head-major store.  The accumulator never
//              leaves the SM in fp32 or BF16.
// Tiles are walked chunk by chunk (chunk_tokens rows at a time, rounded up
// to whole 256-row pair tiles).  Inside a chunk they go in groups of
// RASTER_M pair tiles (2048 rows of x, 29 MB), each group sweeping every W
// column block before the next starts: the group's x stays in L2 while W
// streams past, and a W block is used by all the group's tiles at once.
// Every output element depends only on its token row, so the results do not
// depend on the chunk size or the walk.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"
#include "quant.cuh"

namespace kvq {
namespace {

__device__ unsigned int g_err_proj;

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 6;
constexpr int BNH = BN / 2;          // W rows (output columns) each CTA of the pair loads
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BNH * BK * 2;
constexpr uint16_t kPairMask = 0x3;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int NUM_THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /* align slack */ + 256 /* barriers */;
#ifndef KVQ_RASTER_M
#define KVQ_RASTER_M 8
#endif
constexpr int RASTER_M = KVQ_RASTER_M;  // pair tiles of x per group of the tile walk

struct ProjParams {
    int64_t n;
    int hidden;
    int m_tiles, n_tiles, k_blocks;
    int col_tile0;  // first 256-column tile of W walked (tiles col_tile0 .. col_tile0 + n_tiles - 1)
    int sections;   // bit 0: write Q, bit 1: write K and V (128-column halves of other sections are skipped)
    int chunk_m_tiles;
    int64_t total_tiles;
    const float *q_norm_w;
    const float *k_norm_w;
    float eps;
    const float *rope_cs;  // split-half RoPE table, rot_dim floats ((cos, sin) pairs) per token row, or null
    __nv_bfloat16 *q_out;
    RangeTable ranges;
};

// m_idx counts pair tiles of 2 * BM rows (p.m_tiles, p.chunk_m_tiles are in pair tiles)
__device__ __forceinline__ void tile_coords(int64_t T, const ProjParams &p, int &m_idx, int &n_idx) {
    const int64_t per_chunk = static_cast<int64_t>(p.chunk_m_tiles) * p.n_tiles;
    const int64_t c = T / per_chunk;
    const int64_t local = T - c * per_chunk;
    const int m0 = static_cast<int>(c) * p.chunk_m_tiles;
    const int mc = min(p.chunk_m_tiles, p.m_tiles - m0);  // pair tiles in this chunk
    const int G = min(RASTER_M, mc);
    const int64_t per_group = static_cast<int64_t>(G) * p.n_tiles;
    const int gi = static_cast<int>(local / per_group);   // group inside the chunk (the last may be short)
    const int64_t lg = local - gi * per_group;
    const int gm0 = gi * G;
    const int gmc = min(G, mc - gm0);
    n_idx = p.col_tile0 + static_cast<int>(lg / gmc);
    m_idx = m0 + gm0 + static_cast<int>(lg % gmc);
}

__device__ __forceinline__ void rmsnorm128(float (&v)[128], const float *__restrict__ w, float eps) {
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
    for (int i = 0; i < 128; i += 4) {
        s0 = fmaf(v[i], v[i], s0);
        s1 = fmaf(v[i + 1], v[i + 1], s1);
        s2 = fmaf(v[i + 2], v[i + 2], s2);
        s3 = fmaf(v[i + 3], v[i + 3], s3);
    }
    const float ms = ((s0 + s1) + (s2 + s3)) * (1.0f / 128.0f);
    const float r = 1.0f / sqrtf(ms + eps);
#pragma unroll
    for (int i = 0; i < 128; ++i) v[i] = __fmul_rn(__fmul_rn(v[i], r), __ldg(w + i));
}

// Split-half rotary position embedding of one head row in registers (the
// `_norm_rope` step of vram_lab.py: after the RMSNorm, before the Hadamard
// rotation): with H = ROT/2 and (c_i, s_i) from the row's table,
// y_i = x_i c_i - x_{i+H} s_i and y_{i+H} = x_{i+H} c_i + x_i s_i for i < H;
// fp32 products, then one fp32 sum.
template <int ROT>
__device__ __forceinline__ void rope_split_half(float (&v)[128], const float *__restrict__ cs) {
    constexpr int H = ROT / 2;
    const float4 *t4 = reinterpret_cast<const float4 *>(cs);
#pragma unroll
    for (int i = 0; i < H; i += 2) {
        const float4 t = __ldg(t4 + i / 2);  // c_i, s_i, c_{i+1}, s_{i+1}
        const float a0 = v[i], b0 = v[i + H], a1 = v[i + 1], b1 = v[i + 1 + H];
        v[i] = __fsub_rn(__fmul_rn(a0, t.x), __fmul_rn(b0, t.y));
        v[i + H] = __fadd_rn(__fmul_rn(b0, t.x), __fmul_rn(a0, t.y));
        v[i + 1] = __fsub_rn(__fmul_rn(a1, t.z), __fmul_rn(b1, t.w));
        v[i + 1 + H] = __fadd_rn(__fmul_rn(b1, t.z), __fmul_rn(a1, t.w));
    }
}

template <int GROUP, int BITS>
__device__ __forceinline__ void store_codes(const float (&v)[128], uint8_t *codes_row, uint16_t *scales_row) {
    uint32_t words[128 * BITS / 32];
    uint16_t sb[128 / GROUP];
    quant128_thread<GROUP, BITS>(v, words, sb);
    uint4 *dst = reinterpret_cast<uint4 *>(codes_row);
#pragma unroll
    for (int i = 0; i < 128 * BITS / 128; ++i)
        dst[i] = make_uint4(words[4 * i], words[4 * i + 1], words[4 * i + 2], words[4 * i + 3]);
    if constexpr (GROUP == 32) {
        *reinterpret_cast<uint2 *>(scales_row) =
            make_uint2(sb[0] | (static_cast<uint32_t>(sb[1]) << 16), sb[2] | (static_cast<uint32_t>(sb[3]) << 16));
    } else if constexpr (GROUP == 64) {
        *reinterpret_cast<uint32_t *>(scales_row) = sb[0] | (static_cast<uint32_t>(sb[1]) << 16);
    } else {
        *scales_row = sb[0];
    }
}

template <int GROUP, int ROT>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    qkv_proj_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                    const __grid_constant__ ProjParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *smem_a = smem;
    uint8_t *smem_b = smem + STAGES * A_BYTES;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + STAGES * STAGE_BYTES);  // even CTA: both CTAs' copies landed
    uint64_t *empty = full + STAGES;       // both CTAs: the stage's MMAs completed
    uint64_t *tfull = empty + STAGES;      // both CTAs: an accumulator is complete
    uint64_t *tempty = tfull + 2;          // even CTA: both CTAs' epilogues have read an accumulator
    uint64_t *drain = tempty + 2;          // even CTA: every MMA issued has completed (abort path only)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int64_t cluster = blockIdx.x >> 1, clusters = gridDim.x >> 1;
    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], 2 * 4);  // one arrive per epilogue warp of both CTAs
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tm_x);
        prefetch_tmap(&tm_w);
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, TMEM_COLS);
        tmem_relinquish_pair();
    }
    // the peer may arrive on this CTA's barriers only once they are initialised
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ---------------------------------------------------------- TMA producer (both CTAs)
        // its 128 rows of x and its half (128 rows) of the tile's W rows, into its own ring;
        // both CTAs' copies complete on the even CTA's full barrier of the stage
        if (elect_one()) {
            const uint32_t full_leader = mapa_shared(smem_u32(full), 0);
            int stage = 0;
            uint32_t phase = 0;
            uint32_t armed = 0;  // bit s: stage s has been armed at least once
            uint32_t armed_parity = 0;
            bool issued = false;
            for (int64_t T = cluster; T < p.total_tiles && !*abort_flag; T += clusters) {
                int m_idx, n_idx;
                tile_coords(T, p, m_idx, n_idx);
                const int y = (2 * m_idx + static_cast<int>(rank)) * BM;
                bool ok = true;
                for (int kb = 0; kb < p.k_blocks; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, &g_err_proj)) {
                        ok = false;
                        break;
                    }
                    if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * STAGE_BYTES);
                    const uint32_t bar = full_leader + stage * 8;
                    tma_load_2d_pair(smem_a + stage * A_BYTES, &tm_x, bar, kb * BK, y);
                    tma_load_2d_pair(smem_b + stage * B_BYTES, &tm_w, bar, kb * BK,
                                     n_idx * BN + static_cast<int>(rank) * BNH);
                    issued = true;
                    armed |= 1u << stage;
                    armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
            }
            // drain: every copy this thread started has landed before the CTA exits.  The even
            // CTA waits on its barriers, which count both CTAs' bytes; it reaches the final
            // cluster barrier, and with it lets the odd CTA leave, only after that.  An odd CTA
            // that gave up (a wait ran out) cannot see the even CTA's barriers: it gives its
            // copies in flight a bounded grace period instead.
            volatile int no_abort = 0;
            if (rank == 0) {
                for (int s = 0; s < STAGES; ++s)
                    if (armed & (1u << s)) mbar_wait(&full[s], (armed_parity >> s) & 1u, &no_abort, nullptr);
            } else if (issued && *abort_flag) {
                const uint64_t t0 = globaltimer_ns();
                while (globaltimer_ns() - t0 < 100000ull) {
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (rank == 1) {
            // the odd CTA's MMA warp has nothing to issue: the even CTA's MMAs read its stages
        } else if (elect_one()) {
            // ------------------------------------------------------ even CTA: MMA issuer for the pair
            constexpr uint32_t idesc = make_idesc_f16(2 * BM, BN, 1);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool issued = false;
            for (int64_t T = cluster; T < p.total_tiles && !*abort_flag; T += clusters) {
                if (!mbar_wait_cluster(&tempty[acc], acc_phase ^ 1u, abort_flag, &g_err_proj)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                bool ok = true;
                for (int kb = 0; kb < p.k_blocks; ++kb) {
                    if (!mbar_wait(&full[stage], phase, abort_flag, &g_err_proj)) {  // both CTAs' bytes
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(smem_a + stage * A_BYTES);
                    const uint32_t b_addr = smem_u32(smem_b + stage * B_BYTES);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k) {
                        mma_f16_ss_pair(d_tmem, make_sdesc_sw128(a_addr + k * 32), make_sdesc_sw128(b_addr + k * 32),
                                        idesc, (kb | k) != 0 ? 1u : 0u);
                    }
                    issued = true;
                    mma_commit_pair(&empty[stage], kPairMask);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit_pair(&tfull[acc], kPairMask);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            if (issued && *abort_flag) {
                // drain: every MMA issued so far has completed before the pair tears down;
                // on a barrier of its own, so no epilogue takes a partial accumulator as complete
                volatile int no_abort = 0;
                mma_commit_pair(drain, 0x1);
                mbar_wait(drain, 0, &no_abort, nullptr, 1000000000ull);
            }
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------- epilogue
        const int quarter = warp & 3;
        const int C = p.hidden;
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        int acc = 0;
        uint32_t acc_phase = 0;
        const uint32_t tempty_leader = mapa_shared(smem_u32(tempty), 0);
        for (int64_t T = cluster; T < p.total_tiles && !*abort_flag; T += clusters) {
            int m_idx, n_idx;
            tile_coords(T, p, m_idx, n_idx);
            m_idx = 2 * m_idx + static_cast<int>(rank);  // this CTA's 128-row tile of the pair's 256
            // warp-uniform before the warp-collective TMEM loads
            if (!__all_sync(0xffffffffu, mbar_wait(&tfull[acc], acc_phase, abort_flag, &g_err_proj))) break;
            if (__any_sync(0xffffffffu, *abort_flag)) break;  // a wait elsewhere ran out: store nothing more
            tc_fence_after();
            const int64_t row = static_cast<int64_t>(m_idx) * BM + quarter * 32 + lane;
#pragma unroll 1
            for (int j = 0; j < 2; ++j) {
                uint32_t raw[128];
                const uint32_t taddr = tmem_base + lane_base + static_cast<uint32_t>(acc * BN + j * 128);
                tmem_ld32(taddr + 0, *reinterpret_cast<uint32_t(*)[32]>(&raw[0]));
                tmem_ld32(taddr + 32, *reinterpret_cast<uint32_t(*)[32]>(&raw[32]));
                tmem_ld32(taddr + 64, *reinterpret_cast<uint32_t(*)[32]>(&raw[64]));
                tmem_ld32(taddr + 96, *reinterpret_cast<uint32_t(*)[32]>(&raw[96]));
                tmem_ld_wait();
                const int gcol = n_idx * BN + j * 128;
                if (gcol >= 3 * C) continue;
                float v[128];
#pragma unroll
                for (int i = 0; i < 128; ++i) v[i] = __uint_as_float(raw[i]);
                const int sect = gcol / C;
                if (!((p.sections >> (sect == 0 ? 0 : 1)) & 1)) continue;
                const int head = (gcol - sect * C) >> 7;
                if (sect == 0) {
                    if (p.q_norm_w) rmsnorm128(v, p.q_norm_w, p.eps);
                    if constexpr (ROT > 0) {
                        if (row < p.n) rope_split_half<ROT>(v, p.rope_cs + row * ROT);
                    }
                    rotate128_thread(v);
                    if (row < p.n) {
                        uint4 *dst = reinterpret_cast<uint4 *>(p.q_out + row * C + head * 128);
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            uint32_t w4[4];
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                const __nv_bfloat162 b2 = __floats2bfloat162_rn(v[8 * i + 2 * k], v[8 * i + 2 * k + 1]);
                                w4[k] = *reinterpret_cast<const uint32_t *>(&b2);
                            }
                            dst[i] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                        }
                    }
                } else {
                    if (sect == 1 && p.k_norm_w) rmsnorm128(v, p.k_norm_w, p.eps);
                    if constexpr (ROT > 0) {
                        if (sect == 1 && row < p.n) rope_split_half<ROT>(v, p.rope_cs + row * ROT);
                    }
                    rotate128_thread(v);
                    // the range holding this token; rows past a range's len are never
                    // written (a range may be a window into a larger store)
                    int g = 0;
                    for (int i = 1; i < p.ranges.n; ++i)
                        if (row >= p.ranges.r[i].start) g = i;
                    const RangeDev &R = p.ranges.r[g];
                    const int64_t rr = row - R.start;
                    if (row < p.n && rr < R.len) {
                        const bool is_k = (sect == 1);
                        if (R.bits == 4) {
                            uint8_t *cr = (is_k ? R.k_codes : R.v_codes) + (head * R.cap + rr) * 64;
                            uint16_t *sr = (is_k ? R.k_scales : R.v_scales) + (head * R.cap + rr) * (128 / GROUP);
                            store_codes<GROUP, 4>(v, cr, sr);
                        } else {
                            uint8_t *cr = (is_k ? R.k_codes : R.v_codes) + (head * R.cap + rr) * 128;
                            uint16_t *sr = (is_k ? R.k_scales : R.v_scales) + (head * R.cap + rr) * (128 / GROUP);
                            store_codes<GROUP, 8>(v, cr, sr);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(tempty_leader + acc * 8);
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
    }

    // neither CTA of the pair frees TMEM or leaves while the other may still touch its memory
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem_base, TMEM_COLS);
}

}  // namespace

namespace {
template <int GROUP, int ROT>
cudaError_t launch_proj(const CUtensorMap &tm_x, const CUtensorMap &tm_w, const ProjParams &p, int grid,
                        cudaStream_t s) {
    auto fn = qkv_proj_kernel<GROUP, ROT>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e == cudaSuccess) fn<<<grid, NUM_THREADS, SMEM_BYTES, s>>>(tm_x, tm_w, p);
    return e;
}
template <int GROUP>
cudaError_t launch_rot(const CUtensorMap &tm_x, const CUtensorMap &tm_w, const ProjParams &p, int rot, int grid,
                       cudaStream_t s) {
    if (rot == 64) return launch_proj<GROUP, 64>(tm_x, tm_w, p, grid, s);
    if (rot == 128) return launch_proj<GROUP, 128>(tm_x, tm_w, p, grid, s);
    return launch_proj<GROUP, 0>(tm_x, tm_w, p, grid, s);
}
}  // namespace

int launch_qkv_proj(const void *x, const void *w, int64_t n, int hidden, int group, int64_t chunk_tokens,
                    const float *q_norm_w, const float *k_norm_w, float eps, void *q_out, const RangeTable &ranges,
                    cudaStream_t s, const float *rope_cs, int rot_dim, int sections) {
    alignas(64) CUtensorMap tm_x, tm_w;
    if (encode_tmap_2d(&tm_x, x, 1, static_cast<uint64_t>(hidden), static_cast<uint64_t>(n),
                       static_cast<uint64_t>(hidden) * 2, BK, BM))
        return KVQ_ERR_CUDA;
    if (encode_tmap_2d(&tm_w, w, 1, static_cast<uint64_t>(hidden), static_cast<uint64_t>(3) * hidden,
                       static_cast<uint64_t>(hidden) * 2, BK, BNH))
        return KVQ_ERR_CUDA;
    ProjParams p{};
    p.n = n;
    p.hidden = hidden;
    p.m_tiles = static_cast<int>((n + 2 * BM - 1) / (2 * BM));  // pair tiles of 256 rows
    // the W rows (output columns) of the requested sections: Q = [0, C), K and V = [C, 3C)
    const int c0 = (sections & 1) ? 0 : hidden, c1 = (sections & 2) ? 3 * hidden : hidden;
    p.col_tile0 = c0 / BN;
    p.n_tiles = (c1 + BN - 1) / BN - p.col_tile0;
    p.sections = sections;
    p.k_blocks = hidden / BK;
    int64_t cm = chunk_tokens <= 0 ? p.m_tiles : (chunk_tokens + 2 * BM - 1) / (2 * BM);
    if (cm > p.m_tiles) cm = p.m_tiles;
    p.chunk_m_tiles = static_cast<int>(cm);
    p.total_tiles = static_cast<int64_t>(p.m_tiles) * p.n_tiles;
    p.q_norm_w = q_norm_w;
    p.k_norm_w = k_norm_w;
    p.eps = eps;
    p.q_out = static_cast<__nv_bfloat16 *>(q_out);
    p.ranges = ranges;
    p.rope_cs = rope_cs;
    const int rot = rope_cs ? rot_dim : 0;
    const int64_t pairs = sm_count() / 2;  // one CTA pair per two SMs, persistent
    const int grid = 2 * static_cast<int>(p.total_tiles < pairs ? p.total_tiles : pairs);
    cudaError_t e;
    if (group == 32) e = launch_rot<32>(tm_x, tm_w, p, rot, grid, s);
    else if (group == 64) e = launch_rot<64>(tm_x, tm_w, p, rot, grid, s);
    else e = launch_rot<128>(tm_x, tm_w, p, rot, grid, s);
    if (e == cudaSuccess) e = cudaGetLastError();
    return report_cuda(e, "projection launch");
}

cudaError_t read_clear_err_proj(unsigned int *v) {
    cudaError_t e = cudaMemcpyFromSymbol(v, g_err_proj, sizeof(unsigned int));
    if (e != cudaSuccess) return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_err_proj, &zero, sizeof(unsigned int));
}

}  // namespace kvq
