// KDA chunked prefill forward with 16-token chunks and no exponent centering: the
// chunk-size ablation of the tcgen05 kernel in kda_fwd_tc.cu.
//
// With 16 tokens the prefix G of a chunk lies in [16 b, 0], so 2^G and 2^-G stay in the
// bf16 normal range for the same lower_bound range that the 32-token kernel reaches only
// with the fixed anchor C = 16 b ("FlashInfer PR #4262" notes, section 2).  Without the
// anchor the operands simplify: Q_d = Q_c = scale q 2^G, K_d = K_c = k 2^G,
// K_i = k 2^-G and K_r = K_i diag(a) with a = 2^G_T.  Everything else is the 32-token
// design at half the chunk: the same warp roles, TMEM residency of the fp32 state, a
// two-slot ring, and per chunk
//   GEMM1  [O_0 | P] = S_bf16 [Q_d | K_d]^T      M128 N32  K128  (A = bf16 S from TMEM)
//          P -= V^T                              M128 N16  K16   (A = V from SMEM, B = -I)
//   GEMM2  U = (-R) (-B2)                        M128 N16  K16   (B2 = diag(beta) INV^T)
//   GEMM3  S += U K_r,  O += U Mqk^T             M128 N128 + N16, K16
// The 16 x 16 inverse is one forward substitution in one warp.
#include <cuda.h>

#include "kda_device.cuh"
#include "kda_kernels.h"
#include "kda_sm100.cuh"

namespace kda {
namespace {

constexpr int C16 = 16;   // tokens per chunk
constexpr int TC_THREADS = 384;
constexpr int W_PREP0 = 4, PREP_WARPS = 8;
constexpr int T_MMA = 32, T_TMA = 64, W_BETA = 2, T_STORE = 96;
constexpr int PREP_THREADS = PREP_WARPS * 32;
constexpr int NSLOT = 2;
constexpr long long WAIT_LIMIT = 2000000000LL;  // SM cycles (~1 s) before a wait gives up

// Slot layout (bytes); raw q/k/g land where derived operands are later written.
constexpr uint32_t SL_QDKD = 0;       // [Q_d | K_d]: 32 rows x 128, K-major, 128-B swizzle (raw q at 0, k at 4096)
constexpr uint32_t SL_RAWQ = 0, SL_RAWK = 4096;
constexpr uint32_t SL_KR = 8192;      // K_r [16 tokens][128], two 64-channel blocks, 128-B swizzle (raw g here)
constexpr uint32_t SL_RAWG = 8192;
constexpr uint32_t SL_V = 12288;      // raw v, two [16][64] swizzled blocks; then the output tile [16][128]
constexpr uint32_t SL_MQT = 16384;    // Mqk [16][16], K-major core layout
constexpr uint32_t SL_INV = 16896;    // -B2 [16][16], K-major core layout
constexpr uint32_t SL_A = 17408;      // fp32 [128]: 2^G_T
constexpr uint32_t SL_BETA = 17920;   // fp32 [16]
constexpr uint32_t SLOT_BYTES = 18432;

constexpr uint32_t OFF_KI = NSLOT * SLOT_BYTES;   // K_i [16][128], XOR-swizzled 16-byte chunks
constexpr uint32_t OFF_MISC = OFF_KI + 4096;      // tot[8][128], rq[16], rk[16], then L
constexpr int LC = 20;                            // fp32 row stride of L (column-major)
constexpr uint32_t OFF_XT = OFF_MISC + 8 * 128 * 4 + 128;   // X = INV, fp32 [16][17]
constexpr uint32_t OFF_NEGI = OFF_XT + 16 * 17 * 4 + 64;    // -I (bf16 16 x 16, K-major core layout)
constexpr uint32_t OFF_BAR = OFF_NEGI + 512;
enum { B_FULLTMA = 0, B_FULLV = 2, B_AREADY = 4, B_FULL = 6, B_G1 = 8, B_G2, B_G3, B_COUNT };
constexpr uint32_t OFF_TMEMADDR = OFF_BAR + B_COUNT * 8;
constexpr uint32_t SMEM_USED = OFF_TMEMADDR + 16;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;
static_assert(SLOT_BYTES % 1024 == 0 && OFF_KI % 256 == 0, "slot / tile alignment");
static_assert(16 * LC * 4 <= 8 * 128 * 4 + 128, "L fits over the prefix partials");
static_assert(2 * (SMEM_BYTES + 1024) <= 233472, "two CTAs must fit one SM");

// TMEM columns: S (fp32), O [128,144), P then U [144,160), and the bf16 copy of S whose
// first 8 columns carry -R and then U between the GEMMs.
constexpr uint32_t TM_S = 0, TM_O = 128, TM_P = 144, TM_SB = 192, TM_COLS = 256;

struct TmaMaps {
    CUtensorMap q, k, v, g, out;   // boxes of 16 tokens; v: 64 channels with the 128-byte swizzle
};

struct Unit {
    uint32_t base;
    unsigned char* gbase;
    int64_t bos, eos;
    int nchunks, n, h;
    uint32_t tmem;
};

__device__ __forceinline__ uint32_t bar_addr(const Unit& u, int b) { return u.base + OFF_BAR + 8u * b; }
__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }
__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }
__device__ __forceinline__ float2 bf2_to_f2(uint32_t w) { return make_float2(bf16_lo(w), bf16_hi(w)); }
__device__ __forceinline__ uint32_t f2_to_bf2(float2 x) { return pack_bf16x2(x.x, x.y); }

// byte offset of (row, col) in a 16 x 128 bf16 scratch tile (chunk ^= row % 8)
__device__ __forceinline__ uint32_t sc128(int row, int col) {
    return (uint32_t)(row * 256 + ((((col >> 3) ^ (row & 7))) << 4) + ((col & 7) << 1));
}

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, uint32_t* status,
                                          uint32_t max_sleep_ns = 0) {
    const bool ok = mbar_wait_bounded(bar, parity, status, KDA_DEVERR_TIMEOUT, WAIT_LIMIT, max_sleep_ns);
    return __all_sync(0xffffffffu, ok);
}

// Wind-down after an expired wait: the warp keeps meeting its group at every named barrier
// the group still has ahead (plain bar.sync, no waits, no work) until the sequence ends, so
// no sibling is ever left at a barrier and the fast path keeps its code.  Chain group:
// barrier k of chunk c (0: before chunk 0; 1: after GEMM1; 2: after U; 3: after the output
// staging; 4: after the next decay, for every chunk but the last).
__device__ __noinline__ void chain_wind_down(int c, int k, int nchunks) {
    if (k == 0) {
        named_bar_sync(2, 128);
        k = 1;
    }
    for (; c < nchunks; ++c, k = 1)
        for (; k <= (c + 1 < nchunks ? 4 : 3); ++k) named_bar_sync(2, 128);
}
// Prep group: barrier k (0-3) of chunk c, the last one after the wait for the next boxes.
__device__ __noinline__ void prep_wind_down(int c, int k, int nchunks) {
    for (; c < nchunks; ++c, k = 0)
        for (; k < 4; ++k) named_bar_sync(1, PREP_THREADS);
}

__device__ __forceinline__ void load_state16(const FwdParams& p, size_t off, uint32_t (&r)[16]) {
    if (!p.init_state) {
#pragma unroll
        for (int j = 0; j < 16; ++j) r[j] = 0u;
    } else if (p.init_f32) {
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const float*>(p.init_state) + off);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint4 x = src[j];
            r[4 * j] = x.x; r[4 * j + 1] = x.y; r[4 * j + 2] = x.z; r[4 * j + 3] = x.w;
        }
    } else {
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.init_state) + off);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const uint4 x = src[j];
            const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                r[8 * j + 2 * m] = w[m] << 16;
                r[8 * j + 2 * m + 1] = w[m] & 0xffff0000u;
            }
        }
    }
}

__device__ __forceinline__ void store_state16(const FwdParams& p, size_t off, const uint32_t (&r)[16]) {
    if (!p.final_state) return;
    if (p.final_f32) {
        uint4* dst = reinterpret_cast<uint4*>(static_cast<float*>(p.final_state) + off);
#pragma unroll
        for (int j = 0; j < 4; ++j) dst[j] = make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
    } else {
        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.final_state) + off);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            dst[j] = make_uint4(pack_bf16x2(u2f(r[8 * j]), u2f(r[8 * j + 1])),
                                pack_bf16x2(u2f(r[8 * j + 2]), u2f(r[8 * j + 3])),
                                pack_bf16x2(u2f(r[8 * j + 4]), u2f(r[8 * j + 5])),
                                pack_bf16x2(u2f(r[8 * j + 6]), u2f(r[8 * j + 7])));
        }
    }
}

// The 16 fp32 P columns of this lane -> bf16 -> the first 8 columns of the bf16 copy of S.
__device__ __forceinline__ void p_cols_to_bf16(uint32_t lane_addr) {
    uint32_t pr[16], rp[8];
    tmem_ld16(lane_addr + TM_P, pr);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 8; ++i) rp[i] = pack_bf16x2(u2f(pr[2 * i]), u2f(pr[2 * i + 1]));
    tmem_st8(lane_addr + TM_SB, rp);
    tmem_wait_st();
}

// One pass over S: its bf16 copy (the next GEMM1 operand), then S = S diag(a) in place.
__device__ __forceinline__ void copy_and_decay(uint32_t lane_addr, const float* a_s) {
#pragma unroll 1
    for (int piece = 0; piece < 8; ++piece) {
        uint32_t r[16];
        tmem_ld16(lane_addr + TM_S + piece * 16, r);
        tmem_wait_ld();
        uint32_t b[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) b[j] = pack_bf16x2(u2f(r[2 * j]), u2f(r[2 * j + 1]));
        tmem_st8(lane_addr + TM_SB + piece * 8, b);
        const float4* a4 = reinterpret_cast<const float4*>(a_s + piece * 16);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float4 a = a4[j];
            const float2 x0 = __fmul2_rn(make_float2(u2f(r[4 * j]), u2f(r[4 * j + 1])), make_float2(a.x, a.y));
            const float2 x1 = __fmul2_rn(make_float2(u2f(r[4 * j + 2]), u2f(r[4 * j + 3])), make_float2(a.z, a.w));
            r[4 * j] = f2u(x0.x); r[4 * j + 1] = f2u(x0.y);
            r[4 * j + 2] = f2u(x1.x); r[4 * j + 3] = f2u(x1.y);
        }
        tmem_st16(lane_addr + TM_S + piece * 16, r);
    }
}

__device__ __forceinline__ int chunk_valid(const Unit& u, int c) {
    const int64_t t0 = u.bos + (int64_t)c * C16;
    return (int)((u.eos - t0) < C16 ? (u.eos - t0) : C16);
}

__device__ __forceinline__ void load_qkg(const TmaMaps& maps, const Unit& u, int c) {
    const int s = c & 1;
    const int t0 = (int)(u.bos + (int64_t)c * C16);
    const uint32_t slot = u.base + s * SLOT_BYTES, full = bar_addr(u, B_FULLTMA + s);
    mbar_arrive_expect_tx(full, 3u * C16 * HD * 2u);
    tma_load_3d(slot + SL_RAWQ, &maps.q, 0, u.h, t0, full);
    tma_load_3d(slot + SL_RAWK, &maps.k, 0, u.h, t0, full);
    tma_load_3d(slot + SL_RAWG, &maps.g, 0, u.h, t0, full);
}

__device__ __forceinline__ void load_v(const TmaMaps& maps, const Unit& u, int c) {
    const int s = c & 1;
    const int t0 = (int)(u.bos + (int64_t)c * C16);
    const uint32_t slot = u.base + s * SLOT_BYTES, full = bar_addr(u, B_FULLV + s);
    mbar_arrive_expect_tx(full, C16 * HD * 2u);
    tma_load_3d(slot + SL_V, &maps.v, 0, u.h, t0, full);
    tma_load_3d(slot + SL_V + 2048, &maps.v, 64, u.h, t0, full);
}

__device__ __forceinline__ void prefetch_chunk(const TmaMaps& maps, const Unit& u, int c) {
    const int t0 = (int)(u.bos + (int64_t)c * C16);
    tma_prefetch_l2_3d(&maps.q, 0, u.h, t0);
    tma_prefetch_l2_3d(&maps.k, 0, u.h, t0);
    tma_prefetch_l2_3d(&maps.g, 0, u.h, t0);
    tma_prefetch_l2_3d(&maps.v, 0, u.h, t0);
    tma_prefetch_l2_3d(&maps.v, 64, u.h, t0);
}

__device__ __forceinline__ float load_beta(const FwdParams& p, const Unit& u, int c, int lane) {
    const int64_t t0 = u.bos + (int64_t)c * C16;
    return lane < chunk_valid(u, c)
               ? bf16_bits_to_f32(reinterpret_cast<const uint16_t*>(p.beta)[(t0 + lane) * p.H + u.h])
               : 0.f;
}

// beta of a chunk by the 32 lanes of one warp (lanes >= 16 only arrive)
__device__ __forceinline__ void put_beta(const Unit& u, int c, int lane, float b) {
    if (lane < C16) reinterpret_cast<float*>(u.gbase + (c & 1) * SLOT_BYTES + SL_BETA)[lane] = b;
    mbar_arrive(bar_addr(u, B_FULLTMA + (c & 1)));
}

// ------------------------------------------------------------------------------
// Chain group: state row v = TMEM lane v.
// ------------------------------------------------------------------------------
__device__ void chain_group(const FwdParams& p, const TmaMaps& maps, const Unit& u, int pt) {
    constexpr uint32_t idesc1 = make_idesc_bf16_f32(128, 32);
    constexpr uint32_t idescv = make_idesc_bf16_f32(128, 16, false, true);
    constexpr uint32_t idesc2 = make_idesc_bf16_f32(128, 16);
    constexpr uint32_t idesc3 = make_idesc_bf16_f32(128, 128, true);
    const int w = pt >> 5, lane = pt & 31;
    const uint32_t lane_addr = u.tmem + ((uint32_t)(w * 32) << 16);
    const int v = pt;
    const size_t srow = (((size_t)u.n * p.H + u.h) * HD + v) * HD;

#pragma unroll 1
    for (int piece = 0; piece < 8; ++piece) {
        uint32_t r[16];
        load_state16(p, srow + piece * 16, r);
        if (u.nchunks == 0) store_state16(p, srow + piece * 16, r);
        else tmem_st16(lane_addr + TM_S + piece * 16, r);
    }
    if (u.nchunks == 0) return;
    const int first = u.nchunks < NSLOT ? u.nchunks : NSLOT;
    if (pt == T_TMA)
        for (int c = 0; c < first; ++c) load_qkg(maps, u, c);
    if (pt == T_STORE)
        for (int c = 0; c < first; ++c) load_v(maps, u, c);
    if (w == W_BETA)
        for (int c = 0; c < first; ++c) put_beta(u, c, lane, load_beta(p, u, c, lane));
    int issued = first;
    if (pt < 32) {   // -I (16 x 16): thread = (row n, 8-column block)
        const int n = pt >> 1, kb = pt & 1;
        const uint32_t m1 = ((n >> 3) == kb) ? ((n & 1) ? 0xBF800000u : 0x0000BF80u) : 0u;
        const int wi = (n & 7) >> 1;
        *reinterpret_cast<uint4*>(u.gbase + OFF_NEGI + core_offset(n, 8 * kb, 16)) =
            make_uint4(wi == 0 ? m1 : 0u, wi == 1 ? m1 : 0u, wi == 2 ? m1 : 0u, wi == 3 ? m1 : 0u);
        fence_proxy_async_smem();
    }
    tmem_wait_st();
    bool ok = warp_wait(bar_addr(u, B_AREADY), 0, p.status, 256);
    if (ok) {
        copy_and_decay(lane_addr, reinterpret_cast<const float*>(u.gbase + SL_A));
        tmem_wait_st();
        tc_fence_before();
        named_bar_sync(2, 128);
    } else {
        chain_wind_down(0, 0, u.nchunks);
    }

#pragma unroll 1
    for (int c = 0; ok && c < u.nchunks; ++c) {
        const int s = c & 1;
        const uint32_t cpar = c & 1, kpar = (c >> 1) & 1;
        const uint32_t slot = u.base + s * SLOT_BYTES;
        const bool refill = c + NSLOT < u.nchunks;
        if (pt == T_TMA && refill) prefetch_chunk(maps, u, c + NSLOT);
        if (!warp_wait(bar_addr(u, B_FULL + s), kpar, p.status, 256)) { chain_wind_down(c, 1, u.nchunks); break; }
        float beta_next = 0.f;
        if (refill && w == W_BETA) beta_next = load_beta(p, u, c + NSLOT, lane);
        if (w == 1) {
            if (!warp_wait(bar_addr(u, B_FULLV + s), kpar, p.status, 256)) { chain_wind_down(c, 1, u.nchunks); break; }
            tc_fence_after();
            if (pt == T_MMA) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    tc_mma_ts(u.tmem + TM_O, u.tmem + TM_SB + kk * 8,
                              make_sdesc_kmajor_sw128(slot + SL_QDKD + (kk >> 2) * 4096 + (kk & 3) * 32), idesc1, kk > 0);
                tc_mma_ss(u.tmem + TM_P, make_sdesc_mnmajor_sw128(slot + SL_V, 2048, 1024),
                          make_sdesc_kmajor_noswizzle(u.base + OFF_NEGI, 128, 256), idescv, 1u);   // P -= V^T
                tc_commit(bar_addr(u, B_G1));
            }
        }

        if (!warp_wait(bar_addr(u, B_G1), cpar, p.status)) { chain_wind_down(c, 1, u.nchunks); break; }
        tc_fence_after();
        if (refill && w == W_BETA) put_beta(u, c + NSLOT, lane, beta_next);
        p_cols_to_bf16(lane_addr);   // -R = P - V^T
        tc_fence_before();
        named_bar_sync(2, 128);
        if (pt == T_MMA) {   // GEMM2 U = (-R) (-B2)
            tc_fence_after();
            tc_mma_ts(u.tmem + TM_P, u.tmem + TM_SB, make_sdesc_kmajor_noswizzle(slot + SL_INV, 128, 256), idesc2, 0u);
            tc_commit(bar_addr(u, B_G2));
        }
        if (!warp_wait(bar_addr(u, B_G2), cpar, p.status)) { chain_wind_down(c, 2, u.nchunks); break; }
        tc_fence_after();
        p_cols_to_bf16(lane_addr);   // U
        tc_fence_before();
        named_bar_sync(2, 128);
        if (pt == T_MMA) {   // GEMM3: S += U K_r, O += U Mqk^T
            tc_fence_after();
            tc_mma_ts(u.tmem + TM_S, u.tmem + TM_SB, make_sdesc_mnmajor_sw128(slot + SL_KR, 2048, 1024), idesc3, 1u);
            tc_mma_ts(u.tmem + TM_O, u.tmem + TM_SB, make_sdesc_kmajor_noswizzle(slot + SL_MQT, 128, 256), idesc2, 1u);
            tc_commit(bar_addr(u, B_G3));
        }
        if (!warp_wait(bar_addr(u, B_G3), cpar, p.status)) { chain_wind_down(c, 3, u.nchunks); break; }
        tc_fence_after();
        if (refill) {
            if (pt == T_TMA) load_qkg(maps, u, c + NSLOT);
            issued = c + NSLOT + 1;
        }

        {   // O of this chunk -> staging tile [token][v] in the slot's v region
            unsigned char* ost = u.gbase + s * SLOT_BYTES + SL_V + 2 * v;
            uint32_t o[16];
            tmem_ld16(lane_addr + TM_O, o);
            tmem_wait_ld();
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const uint32_t pr = pack_bf16x2(u2f(o[2 * m]), u2f(o[2 * m + 1]));
                *reinterpret_cast<uint16_t*>(ost + (2 * m) * 256) = (uint16_t)(pr & 0xffffu);
                *reinterpret_cast<uint16_t*>(ost + (2 * m + 1) * 256) = (uint16_t)(pr >> 16);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        named_bar_sync(2, 128);
        if (pt == T_STORE) {
            const int64_t t0 = u.bos + (int64_t)c * C16;
            const int nvalid = chunk_valid(u, c);
            const uint32_t ost = slot + SL_V;
            if (nvalid == C16) {
                tma_store_3d(&maps.out, ost, 0, u.h, (int)t0);
            } else {
                for (int i = 0; i < nvalid; ++i)
                    bulk_store(p.out + ((t0 + i) * p.H + u.h) * HD, ost + i * 256, 256);
            }
            bulk_commit();
            if (refill) {
                bulk_wait_read_all();
                load_v(maps, u, c + NSLOT);
            }
        }

        if (c + 1 < u.nchunks) {
            if (!warp_wait(bar_addr(u, B_AREADY + (s ^ 1)), ((c + 1) >> 1) & 1, p.status, 256)) { chain_wind_down(c, 4, u.nchunks); break; }
            copy_and_decay(lane_addr, reinterpret_cast<const float*>(u.gbase + (s ^ 1) * SLOT_BYTES + SL_A));
            tmem_wait_st();
            tc_fence_before();
            named_bar_sync(2, 128);
        } else {
#pragma unroll 1
            for (int piece = 0; piece < 8; ++piece) {
                uint32_t r[16];
                tmem_ld16(lane_addr + TM_S + piece * 16, r);
                tmem_wait_ld();
                store_state16(p, srow + piece * 16, r);
            }
        }
    }
    if (pt == T_STORE) bulk_wait_all();
    if (pt == T_TMA || pt == T_STORE) {
        const int b0 = pt == T_TMA ? B_FULLTMA : B_FULLV;
        for (int c = issued - NSLOT < 0 ? 0 : issued - NSLOT; c < issued; ++c)
            mbar_wait_bounded(bar_addr(u, b0 + (c & 1)), (c >> 1) & 1, p.status, KDA_DEVERR_TIMEOUT, WAIT_LIMIT);
    }
}

// ------------------------------------------------------------------------------
// Prep group (256 threads).  Elementwise phases: thread = (channel quad 4 lane .. 4 lane
// + 3, tokens 2 pw and 2 pw + 1).
// ------------------------------------------------------------------------------
__device__ void prep_group(const FwdParams& p, const Unit& u, int pt) {
    const int lane = pt & 31, pw = pt >> 5, gq = lane >> 2, tq = lane & 3;
    const int c0 = 4 * lane;
    const float eA = expf(p.A_log[u.h]);
    const float gm = -eA * LOG2E;                       // sigmoid(x) = 1 / (1 + 2^(gm (g + dt)))
    const float4 dt = *reinterpret_cast<const float4*>(p.dt_bias + u.h * HD + c0);
    const float2 gmv = make_float2(gm, gm);
    const float2 gb01 = make_float2(gm * dt.x, gm * dt.y), gb23 = make_float2(gm * dt.z, gm * dt.w);
    const float bcoef = p.lower_bound * LOG2E;          // b
    // store offsets of token 2 pw; token 2 pw + r differs by one XOR (row bit, chunk bit 0)
    const uint32_t oq = sw128_offset(2 * pw, c0, 32);   // Q_d = Q_c rows 0-15, K_d = K_c rows 16-31
    const uint32_t okr = sw128_offset(2 * pw, c0, 16);
    const uint32_t oki = sc128(2 * pw, c0);

    unsigned char* kis = u.gbase + OFF_KI;
    float* tot = reinterpret_cast<float*>(u.gbase + OFF_MISC);   // [8][128]
    float* rq = tot + PREP_WARPS * HD;
    float* rk = rq + C16;
    float* Lc = tot;                                             // after the prefix and norms are used
    float* X = reinterpret_cast<float*>(u.gbase + OFF_XT);       // [16][17]

#pragma unroll 1
    for (int c = 0; c < u.nchunks; ++c) {
        const int s = c & 1;
        const uint32_t kpar = (c >> 1) & 1;
        unsigned char* gslot = u.gbase + s * SLOT_BYTES;
        if (c == 0 && !warp_wait(bar_addr(u, B_FULLTMA + s), kpar, p.status, 128)) { prep_wind_down(0, 0, u.nchunks); return; }
        const int64_t t0 = u.bos + (int64_t)c * C16;
        const int nvalid = (int)((u.eos - t0) < C16 ? (u.eos - t0) : C16);
        const float* bs = reinterpret_cast<const float*>(gslot + SL_BETA);

        // ---- A: q/k row norms (8 threads per row of 128), gate and local prefix
        uint2 qv[2], kv[2];
        float2 G01[2], G23[2];
        {
            const int row = pt >> 3, part = pt & 7;   // rows 0-15 q, 16-31 k; 16 elements per thread
            const unsigned char* rp = gslot + (row < C16 ? SL_RAWQ + row * 256 : SL_RAWK + (row - C16) * 256);
            const uint4 wa = *reinterpret_cast<const uint4*>(rp + part * 16);
            const uint4 wb = *reinterpret_cast<const uint4*>(rp + (part + 8) * 16);
            uint2 gw[2];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const uint32_t off = (2 * pw + r) * 256 + c0 * 2;
                qv[r] = *reinterpret_cast<const uint2*>(gslot + SL_RAWQ + off);
                kv[r] = *reinterpret_cast<const uint2*>(gslot + SL_RAWK + off);
                gw[r] = *reinterpret_cast<const uint2*>(gslot + SL_RAWG + off);
            }
            float2 acc01 = make_float2(0.f, 0.f), acc23 = make_float2(0.f, 0.f);
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int i = 2 * pw + r;
                const float2 x01 = __ffma2_rn(gmv, bf2_to_f2(gw[r].x), gb01);
                const float2 x23 = __ffma2_rn(gmv, bf2_to_f2(gw[r].y), gb23);
                const float bl = i < nvalid ? bcoef : 0.f;
                const float2 blv = make_float2(bl, bl);
                acc01 = __ffma2_rn(blv, make_float2(rcp_approx(1.f + ex2_approx(x01.x)), rcp_approx(1.f + ex2_approx(x01.y))),
                                   acc01);
                acc23 = __ffma2_rn(blv, make_float2(rcp_approx(1.f + ex2_approx(x23.x)), rcp_approx(1.f + ex2_approx(x23.y))),
                                   acc23);
                G01[r] = acc01;
                G23[r] = acc23;
            }
            *reinterpret_cast<float4*>(tot + pw * HD + c0) = make_float4(acc01.x, acc01.y, acc23.x, acc23.y);

            float2 ss0 = make_float2(0.f, 0.f), ss1 = make_float2(0.f, 0.f);
            const uint32_t ws[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
                const float2 x0 = bf2_to_f2(ws[e]), x1 = bf2_to_f2(ws[e + 1]);
                ss0 = __ffma2_rn(x0, x0, ss0);
                ss1 = __ffma2_rn(x1, x1, ss1);
            }
            const float2 ss = __fadd2_rn(ss0, ss1);
            float sum = ss.x + ss.y;
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            sum += __shfl_xor_sync(0xffffffffu, sum, 2);
            sum += __shfl_xor_sync(0xffffffffu, sum, 4);
            const int tok = row & (C16 - 1);
            const float rn = tok < nvalid ? rsqrtf(sum + NORM_EPS) : 0.f;
            if (part == 0) {
                if (row < C16) rq[tok] = rn; else rk[tok] = rn;
            }
        }
        named_bar_sync(1, PREP_THREADS);   // raw q/k/g are no longer read after this point

        // ---- B: prefix combine, operands (no anchor: 2^G and 2^-G stay normal)
        {
            float2 T01 = make_float2(0.f, 0.f), T23 = make_float2(0.f, 0.f);
            {
                float2 off01 = make_float2(0.f, 0.f), off23 = make_float2(0.f, 0.f);
#pragma unroll
                for (int qq = 0; qq < PREP_WARPS; ++qq) {
                    const float4 t4 = *reinterpret_cast<const float4*>(tot + qq * HD + c0);
                    const float2 a01 = make_float2(t4.x, t4.y), a23 = make_float2(t4.z, t4.w);
                    if (qq < pw) { off01 = __fadd2_rn(off01, a01); off23 = __fadd2_rn(off23, a23); }
                    T01 = __fadd2_rn(T01, a01);
                    T23 = __fadd2_rn(T23, a23);
                }
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    G01[r] = __fadd2_rn(G01[r], off01);
                    G23[r] = __fadd2_rn(G23[r], off23);
                }
            }
            const float2 a01 = make_float2(ex2_approx(T01.x), ex2_approx(T01.y));
            const float2 a23 = make_float2(ex2_approx(T23.x), ex2_approx(T23.y));
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int i = 2 * pw + r;
                const uint32_t x7 = (uint32_t)((r << 4) | (r << 7)), x8 = (uint32_t)((r << 4) | (r << 8));
                const float qs = rq[i] * p.scale, ks = rk[i];
                const float2 k01 = __fmul2_rn(bf2_to_f2(kv[r].x), make_float2(ks, ks));
                const float2 k23 = __fmul2_rn(bf2_to_f2(kv[r].y), make_float2(ks, ks));
                const float2 ep01 = make_float2(ex2_approx(G01[r].x), ex2_approx(G01[r].y));
                const float2 ep23 = make_float2(ex2_approx(G23[r].x), ex2_approx(G23[r].y));
                const float2 qc01 = __fmul2_rn(__fmul2_rn(bf2_to_f2(qv[r].x), make_float2(qs, qs)), ep01);
                const float2 qc23 = __fmul2_rn(__fmul2_rn(bf2_to_f2(qv[r].y), make_float2(qs, qs)), ep23);
                *reinterpret_cast<uint2*>(gslot + SL_QDKD + (oq ^ x7)) = make_uint2(f2_to_bf2(qc01), f2_to_bf2(qc23));
                const float2 kc01 = __fmul2_rn(k01, ep01), kc23 = __fmul2_rn(k23, ep23);
                *reinterpret_cast<uint2*>(gslot + SL_QDKD + ((oq ^ x7) + C16 * 128)) =
                    make_uint2(f2_to_bf2(kc01), f2_to_bf2(kc23));
                const float2 em01 = make_float2(ex2_approx(-G01[r].x), ex2_approx(-G01[r].y));
                const float2 em23 = make_float2(ex2_approx(-G23[r].x), ex2_approx(-G23[r].y));
                const float2 ki01 = __fmul2_rn(k01, em01), ki23 = __fmul2_rn(k23, em23);
                *reinterpret_cast<uint2*>(kis + (oki ^ x8)) = make_uint2(f2_to_bf2(ki01), f2_to_bf2(ki23));
                *reinterpret_cast<uint2*>(gslot + SL_KR + (okr ^ x7)) =
                    make_uint2(f2_to_bf2(__fmul2_rn(ki01, a01)), f2_to_bf2(__fmul2_rn(ki23, a23)));   // K_r
            }
            if (pw == 4)
                *reinterpret_cast<float4*>(gslot + SL_A + c0 * 4) = make_float4(a01.x, a01.y, a23.x, a23.y);
        }
        // (C reads Q_c, K_c from the slot through the generic proxy; the tensor core reads
        // the slot only after FULL, ordered by the proxy fence before the last barrier)
        named_bar_sync(1, PREP_THREADS);
        if (pt == 0) mbar_arrive(bar_addr(u, B_AREADY + s));

        // ---- C: K_c K_i^T (warps 0, 1) and Q_c K_i^T (warps 2, 3), one 16 x 8 tile each
        if (pw < 4) {
            const int mat = pw >> 1, nt = pw & 1;   // mat 0: A = K_c (slot rows 16-31), 1: A = Q_c (rows 0-15)
            const int arow = (mat ? 0 : C16) + (lane & 7) + ((lane >> 3) & 1) * 8;
            float acc[4] = {0.f, 0.f, 0.f, 0.f}, acc2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kk = 0; kk < 8; kk += 2) {
                uint32_t a[4], a2[4], b[4];
                ldmatrix_x4_s(a, u.base + s * SLOT_BYTES + SL_QDKD + sw128_offset(arow, kk * 16 + (lane >> 4) * 8, 32));
                ldmatrix_x4_s(a2, u.base + s * SLOT_BYTES + SL_QDKD + sw128_offset(arow, kk * 16 + 16 + (lane >> 4) * 8, 32));
                // K_i rows 8 nt .. 8 nt + 7, k steps kk and kk + 1
                ldmatrix_x4_s(b, smem_u32(kis + sc128(8 * nt + (lane & 7), kk * 16 + (lane >> 3) * 8)));
                mma_bf16_16816(acc, a, b[0], b[1]);
                mma_bf16_16816(acc2, a2, b[2], b[3]);
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[e] += acc2[e];
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int i = gq + hf * 8, j = 8 * nt + 2 * tq;
                const float v0 = acc[2 * hf], v1 = acc[2 * hf + 1];
                if (mat == 0) {   // L = strictLower(beta_i Akk), column-major; select, never multiply
                    Lc[j * LC + i] = (j < i) ? bs[i] * v0 : 0.f;
                    Lc[(j + 1) * LC + i] = (j + 1 < i) ? bs[i] * v1 : 0.f;
                } else {
                    *reinterpret_cast<uint32_t*>(gslot + SL_MQT + core_offset(i, j, C16)) =
                        pack_bf16x2((j <= i) ? v0 : 0.f, (j + 1 <= i) ? v1 : 0.f);   // Mqk
                }
            }
        }
        named_bar_sync(1, PREP_THREADS);

        // ---- D: INV = (I + L)^-1 (16 x 16) by forward substitution in warp 0 (lane = column),
        //      then -B2[i][j] = -beta_j X[i][j] into the slot, one row per lane
        if (pw == 0) {
            const int cc = lane & 15;
            float x[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) x[r] = (r == cc) ? 1.f : 0.f;
#pragma unroll
            for (int k = 0; k < 15; ++k) {
                const float xk = x[k];
                const float* col = Lc + k * LC;
#pragma unroll
                for (int r4 = (k + 1) >> 2; r4 < 4; ++r4) {
                    const float4 l4 = *reinterpret_cast<const float4*>(col + 4 * r4);
                    const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (4 * r4 + e > k) x[4 * r4 + e] = fmaf(-lv[e], xk, x[4 * r4 + e]);
                }
            }
            if (lane < 16) {
#pragma unroll
                for (int r = 0; r < 16; ++r) X[r * 17 + cc] = x[r];
            }
            __syncwarp();
            if (lane < 16) {
                const float* xr = X + cc * 17;
                uint32_t wv[8];
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    wv[j] = pack_bf16x2(-bs[2 * j] * xr[2 * j], -bs[2 * j + 1] * xr[2 * j + 1]);
                *reinterpret_cast<uint4*>(gslot + SL_INV + core_offset(cc, 0, C16)) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                *reinterpret_cast<uint4*>(gslot + SL_INV + core_offset(cc, 8, C16)) = make_uint4(wv[4], wv[5], wv[6], wv[7]);
            }
        }
        fence_proxy_async_smem();
        if (c + 1 < u.nchunks && !warp_wait(bar_addr(u, B_FULLTMA + (s ^ 1)), ((c + 1) >> 1) & 1, p.status, 128)) {
            prep_wind_down(c, 3, u.nchunks);
            return;
        }
        named_bar_sync(1, PREP_THREADS);
        if (pt == 0) mbar_arrive(bar_addr(u, B_FULL + s));
    }
}

__global__ void __launch_bounds__(TC_THREADS, 2) kda_fwd_tc16_kernel(const FwdParams p, const __grid_constant__ TmaMaps maps) {
    extern __shared__ unsigned char smem_raw[];
    if (*reinterpret_cast<volatile uint32_t*>(p.status) & KDA_DEVERR_CU_SEQLENS) return;

    const int tid = threadIdx.x, warp = tid >> 5;
    Unit u;
    {
        const uint32_t raw = smem_u32(smem_raw);
        u.base = (raw + 1023u) & ~1023u;
        u.gbase = smem_raw + (u.base - raw);
        u.h = blockIdx.x % p.H;
        const int r = blockIdx.x / p.H;
        u.n = p.order ? p.order[r] : r;
        seq_range(p, u.n, u.bos, u.eos);
        u.nchunks = (int)((u.eos - u.bos + C16 - 1) / C16);
    }
    if (tid == 0) {
        for (int s = 0; s < NSLOT; ++s) {
            mbar_init(bar_addr(u, B_FULLTMA + s), 33);
            mbar_init(bar_addr(u, B_FULLV + s), 1);
            mbar_init(bar_addr(u, B_AREADY + s), 1);
            mbar_init(bar_addr(u, B_FULL + s), 1);
        }
        for (int b = B_G1; b < B_COUNT; ++b) mbar_init(bar_addr(u, b), 1);
        mbar_fence_init();
    }
    if (tid == 32) {
        tma_prefetch_desc(&maps.q);
        tma_prefetch_desc(&maps.k);
        tma_prefetch_desc(&maps.v);
        tma_prefetch_desc(&maps.g);
        tma_prefetch_desc(&maps.out);
    }
    if (warp == 0) {
        tmem_alloc(u.base + OFF_TMEMADDR, TM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    u.tmem = *reinterpret_cast<volatile uint32_t*>(u.gbase + OFF_TMEMADDR);

    if (warp < W_PREP0) chain_group(p, maps, u, tid);
    else prep_group(p, u, tid - W_PREP0 * 32);

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(u.tmem, TM_COLS);
    }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = []() -> EncodeTiledFn {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess || q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<EncodeTiledFn>(f);
    }();
    return fn;
}

// [T_total, H, 128] bf16 as a 3-D tensor (d, h, t); boxes of (64 or 128) x 1 x 16.
bool encode_map16(CUtensorMap* m, const void* ptr, int64_t T_total, int H, bool sw128) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)HD, (cuuint64_t)H, (cuuint64_t)(T_total > 0 ? T_total : 1)};
    const cuuint64_t strides[2] = {(cuuint64_t)HD * 2, (cuuint64_t)H * HD * 2};
    const cuuint32_t box[3] = {(cuuint32_t)(sw128 ? 64 : HD), 1, (cuuint32_t)C16};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_fwd_tc16(const FwdParams& p, cudaStream_t stream) {
    const int units = p.nseq * p.H;
    if (units == 0) return cudaSuccess;
    TmaMaps maps;
    if (!encode_map16(&maps.q, p.q, p.T_total, p.H, false) || !encode_map16(&maps.k, p.k, p.T_total, p.H, false) ||
        !encode_map16(&maps.v, p.v, p.T_total, p.H, true) || !encode_map16(&maps.g, p.g, p.T_total, p.H, false) ||
        !encode_map16(&maps.out, p.out, p.T_total, p.H, false))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(kda_fwd_tc16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    kda_fwd_tc16_kernel<<<units, TC_THREADS, SMEM_BYTES, stream>>>(p, maps);
    return cudaGetLastError();
}

}  // namespace kda
