// KDA chunked prefill forward on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// One CTA per (sequence, head) unit, two CTAs per SM.  The fp32 V x K state stays
// resident in Tensor Memory for the whole sequence ("FlashInfer PR #4262" notes,
// section 6); the recurrent GEMMs run as tcgen05.mma with fp32 TMEM accumulators,
// and the small intra-chunk products as warp-level mma.sync (section 7).
//
// Warp roles (320 threads):
//   warps 0-3  TMEM group: thread v owns state row v (TMEM lane v).  Decays S,
//              turns P into R = (V^T - P) diag(beta), converts U to bf16, drains the
//              chunk output O, refreshes the bf16 copy of S, loads/stores the state.
//   warp 4     MMA issuer (one thread) and TMEM allocator.
//   warp 5     TMA producer: q, k, v, g boxes of 32 tokens per chunk, plus beta.
//   warps 6-9  prep group: gate, prefix, q/k norms, centered operands (section 2),
//              K_c K_i^T and Q_c K_i^T with mma.sync, the 32x32 inverse (section 3).
// A two-slot SMEM ring carries prepared chunks from the prep group to the recurrent
// consumer, which takes chunks strictly in order (section 4); mbarriers give
// backpressure both ways, and every wait is bounded (timeout -> status bit).
//
// TMEM columns (256 per CTA): [0,128) fp32 S; [128,160) O; [160,192) P, then U;
// [192,256) bf16 copy of S (A operand of GEMM1, two values per column).
// Per chunk c (GEMM shapes M x N x K):
//   GEMM1  [O_0 | P] = S_bf16 [Q_d | K_d]^T           128 x 64 x 128   (A from TMEM)
//          S *= diag(a)                               (CUDA cores, TMEM ld/st)
//          R = (V^T - P) diag(beta)                   (CUDA cores -> SMEM, bf16)
//   GEMM2  U = R INV^T                                128 x 32 x 32
//   GEMM3  [S | O] += U [K_r | Mqk^T]                 128 x 160 x 32   (section 8)
#include <cuda.h>

#include "kda_device.cuh"
#include "kda_kernels.h"
#include "kda_sm100.cuh"

namespace kda {
namespace {

constexpr int TC_THREADS = 320;
constexpr int W_MMA = 4, W_TMA = 5, W_PREP0 = 6;
constexpr int NSLOT = 2;
constexpr long long WAIT_LIMIT = 2000000000LL;  // SM cycles (~1 s) before a wait gives up

// Slot layout (bytes).  Raw q/k/g land where their derived operands are written.
constexpr uint32_t SL_QDKD = 0;       // [Q_d | K_d] 64 x 128 K-major (raw q at 0, raw k at 8192)
constexpr uint32_t SL_RAWQ = 0, SL_RAWK = 8192;
constexpr uint32_t SL_KRMQ = 16384;   // [K_r^T (128 rows) | Mqk (32 rows)] x 32 K-major (raw g at 16384)
constexpr uint32_t SL_RAWG = 16384;
constexpr uint32_t SL_INV = 26624;    // INV 32 x 32 K-major (row j, column i)
constexpr uint32_t SL_V = 28672;      // raw v [32][128]
constexpr uint32_t SL_BETA = 36864;   // fp32 [32]
constexpr uint32_t SL_A = 36992;      // fp32 [128]: 2^G_T
constexpr uint32_t SLOT_BYTES = 37888;

constexpr int PROW = 136;                              // padded bf16 row of the prep tiles
constexpr uint32_t PTILE = 32 * PROW * 2;              // 8704 B
constexpr uint32_t OFF_PREP = NSLOT * SLOT_BYTES;      // Q_c, K_c, K_i; later L, X (fp32) over Q_c
constexpr uint32_t OFF_MISC = OFF_PREP + 3 * PTILE;    // tot[2][128], rq[32], rk[32]
constexpr uint32_t OFF_RU = 103424;                    // R, then U: 128 x 32 K-major (8 KB)
constexpr uint32_t OFF_BAR = OFF_RU + 8192;
enum { B_FULLTMA = 0, B_FULL = 2, B_EMPTY = 4, B_G1 = 6, B_G2, B_G3, B_RREADY, B_UREADY, B_SREADY, B_DRAIN,
       B_COUNT };
constexpr uint32_t OFF_TMEMADDR = OFF_BAR + B_COUNT * 8;
constexpr uint32_t SMEM_USED = OFF_TMEMADDR + 16;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;      // slack to align the base to 1 KB
static_assert(OFF_MISC + 1280 <= OFF_RU, "prep scratch overlaps R/U");
static_assert(2 * (SMEM_BYTES + 1024) <= 233472, "two CTAs must fit one SM");

constexpr uint32_t TM_S = 0, TM_O = 128, TM_PU = 160, TM_SB = 192, TM_COLS = 256;

struct TmaMaps {
    CUtensorMap q, k, v, g;
};

struct Unit {
    uint32_t base;        // shared-window address of the 1 KB-aligned smem base
    unsigned char* gbase; // generic pointer to the same place
    int64_t bos, eos;
    int nchunks, n, h;
    uint32_t tmem;
};

__device__ __forceinline__ uint32_t bar_addr(const Unit& u, int b) { return u.base + OFF_BAR + 8u * b; }
__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }
__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }

// Bounded wait, with the verdict made uniform over the warp.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, uint32_t* status) {
    const bool ok = mbar_wait_bounded(bar, parity, status, KDA_DEVERR_TIMEOUT, WAIT_LIMIT);
    return __all_sync(0xffffffffu, ok);
}

// 32 consecutive state values of row `row_off` (element offset), as fp32 bits.
__device__ __forceinline__ void load_state_piece(const FwdParams& p, size_t off, uint32_t (&r)[32]) {
    if (!p.init_state) {
#pragma unroll
        for (int j = 0; j < 32; ++j) r[j] = 0u;
    } else if (p.init_f32) {
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const float*>(p.init_state) + off);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint4 x = src[j];
            r[4 * j] = x.x; r[4 * j + 1] = x.y; r[4 * j + 2] = x.z; r[4 * j + 3] = x.w;
        }
    } else {
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.init_state) + off);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
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

__device__ __forceinline__ void store_state_piece(const FwdParams& p, size_t off, const uint32_t (&r)[32]) {
    if (!p.final_state) return;
    if (p.final_f32) {
        uint4* dst = reinterpret_cast<uint4*>(static_cast<float*>(p.final_state) + off);
#pragma unroll
        for (int j = 0; j < 8; ++j) dst[j] = make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
    } else {
        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.final_state) + off);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            dst[j] = make_uint4(pack_bf16x2(u2f(r[8 * j]), u2f(r[8 * j + 1])),
                                pack_bf16x2(u2f(r[8 * j + 2]), u2f(r[8 * j + 3])),
                                pack_bf16x2(u2f(r[8 * j + 4]), u2f(r[8 * j + 5])),
                                pack_bf16x2(u2f(r[8 * j + 6]), u2f(r[8 * j + 7])));
        }
    }
}

// ------------------------------------------------------------------------------
// TMEM group: state row v = TMEM lane v.
// ------------------------------------------------------------------------------
__device__ void tmem_group(const FwdParams& p, const Unit& u, int pt) {
    const int w = pt >> 5;
    const uint32_t lane_addr = u.tmem + ((uint32_t)(w * 32) << 16);
    const int v = pt;
    const size_t srow = (((size_t)u.n * p.H + u.h) * HD + v) * HD;

    // initial state -> TMEM (fp32 and its bf16 copy); an empty sequence copies it through
#pragma unroll 1
    for (int piece = 0; piece < 4; ++piece) {
        uint32_t r[32];
        load_state_piece(p, srow + piece * 32, r);
        if (u.nchunks == 0) {
            store_state_piece(p, srow + piece * 32, r);
            continue;
        }
        tmem_st32(lane_addr + TM_S + piece * 32, r);
        uint32_t b[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) b[j] = pack_bf16x2(u2f(r[2 * j]), u2f(r[2 * j + 1]));
        tmem_st16(lane_addr + TM_SB + piece * 16, b);
    }
    if (u.nchunks == 0) return;
    tmem_wait_st();
    tc_fence_before();
    named_bar_sync(2, 128);
    if (pt == 0) mbar_arrive(bar_addr(u, B_SREADY));

    unsigned char* ru = u.gbase + OFF_RU;
#pragma unroll 1
    for (int c = 0; c < u.nchunks; ++c) {
        const int s = c & 1;
        const uint32_t kpar = (c >> 1) & 1, cpar = c & 1;
        const unsigned char* gslot = u.gbase + s * SLOT_BYTES;
        if (!warp_wait(bar_addr(u, B_FULL + s), kpar, p.status)) return;

        // S_d = S diag(a): off the critical path, overlapping GEMM1 (which reads the bf16 copy)
        const float* a_s = reinterpret_cast<const float*>(gslot + SL_A);
#pragma unroll 1
        for (int piece = 0; piece < 4; ++piece) {
            uint32_t r[32];
            tmem_ld32(lane_addr + TM_S + piece * 32, r);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] = f2u(u2f(r[j]) * a_s[piece * 32 + j]);
            tmem_st32(lane_addr + TM_S + piece * 32, r);
        }
        tmem_wait_st();

        // R = (V^T - P) diag(beta) -> SMEM (bf16, K-major row v)
        if (!warp_wait(bar_addr(u, B_G1), cpar, p.status)) return;
        tc_fence_after();
        uint32_t pr[32];
        tmem_ld32(lane_addr + TM_PU, pr);
        tmem_wait_ld();
        {
            const uint16_t* vs = reinterpret_cast<const uint16_t*>(gslot + SL_V);
            const float* bs = reinterpret_cast<const float*>(gslot + SL_BETA);
            uint32_t rp[16];
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
                const float r0 = (bf16_bits_to_f32(vs[i * HD + v]) - u2f(pr[i])) * bs[i];
                const float r1 = (bf16_bits_to_f32(vs[(i + 1) * HD + v]) - u2f(pr[i + 1])) * bs[i + 1];
                rp[i >> 1] = pack_bf16x2(r0, r1);
            }
#pragma unroll
            for (int kg = 0; kg < 4; ++kg)
                *reinterpret_cast<uint4*>(ru + core_offset(v, 8 * kg, 32)) =
                    make_uint4(rp[4 * kg], rp[4 * kg + 1], rp[4 * kg + 2], rp[4 * kg + 3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        named_bar_sync(2, 128);
        if (pt == 0) mbar_arrive(bar_addr(u, B_RREADY));

        // U -> bf16 -> SMEM (GEMM2 has finished reading R)
        if (!warp_wait(bar_addr(u, B_G2), cpar, p.status)) return;
        tc_fence_after();
        tmem_ld32(lane_addr + TM_PU, pr);
        tmem_wait_ld();
        {
            uint32_t up[16];
#pragma unroll
            for (int i = 0; i < 32; i += 2) up[i >> 1] = pack_bf16x2(u2f(pr[i]), u2f(pr[i + 1]));
#pragma unroll
            for (int kg = 0; kg < 4; ++kg)
                *reinterpret_cast<uint4*>(ru + core_offset(v, 8 * kg, 32)) =
                    make_uint4(up[4 * kg], up[4 * kg + 1], up[4 * kg + 2], up[4 * kg + 3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        named_bar_sync(2, 128);
        if (pt == 0) mbar_arrive(bar_addr(u, B_UREADY));

        // O -> out rows of this chunk; bf16 copy of S for the next chunk (or the final state)
        if (!warp_wait(bar_addr(u, B_G3), cpar, p.status)) return;
        tc_fence_after();
        tmem_ld32(lane_addr + TM_O, pr);
        tmem_wait_ld();
        {
            const int64_t t0 = u.bos + (int64_t)c * CH;
            const int nvalid = (int)((u.eos - t0) < CH ? (u.eos - t0) : CH);
            __nv_bfloat16* orow = p.out + (t0 * p.H + u.h) * HD + v;
            const int64_t tstride = (int64_t)p.H * HD;
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (i < nvalid) orow[i * tstride] = __float2bfloat16_rn(u2f(pr[i]));
        }
        if (c + 1 < u.nchunks) {
#pragma unroll 1
            for (int piece = 0; piece < 4; ++piece) {
                uint32_t r[32];
                tmem_ld32(lane_addr + TM_S + piece * 32, r);
                tmem_wait_ld();
                uint32_t b[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) b[j] = pack_bf16x2(u2f(r[2 * j]), u2f(r[2 * j + 1]));
                tmem_st16(lane_addr + TM_SB + piece * 16, b);
            }
            tmem_wait_st();
            tc_fence_before();
            named_bar_sync(2, 128);
            if (pt == 0) mbar_arrive(bar_addr(u, B_SREADY));
        } else {
#pragma unroll 1
            for (int piece = 0; piece < 4; ++piece) {
                uint32_t r[32];
                tmem_ld32(lane_addr + TM_S + piece * 32, r);
                tmem_wait_ld();
                store_state_piece(p, srow + piece * 32, r);
            }
        }
    }
}

// ------------------------------------------------------------------------------
// MMA issuer (one thread).
// ------------------------------------------------------------------------------
__device__ void mma_issuer(const FwdParams& p, const Unit& u) {
    constexpr uint32_t idesc1 = make_idesc_bf16_f32(128, 64);
    constexpr uint32_t idesc2 = make_idesc_bf16_f32(128, 32);
    constexpr uint32_t idesc3 = make_idesc_bf16_f32(128, 160);
    const uint32_t ru = u.base + OFF_RU;
    bool issued = false;
#pragma unroll 1
    for (int c = 0; c < u.nchunks; ++c) {
        const int s = c & 1;
        const uint32_t kpar = (c >> 1) & 1, cpar = c & 1;
        const uint32_t slot = u.base + s * SLOT_BYTES;
        if (!mbar_wait_bounded(bar_addr(u, B_FULL + s), kpar, p.status, KDA_DEVERR_TIMEOUT, WAIT_LIMIT)) break;
        if (!mbar_wait_bounded(bar_addr(u, B_SREADY), cpar, p.status, KDA_DEVERR_TIMEOUT, WAIT_LIMIT)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
            tc_mma_ts(u.tmem + TM_O, u.tmem + TM_SB + kk * 8,
                      make_sdesc_kmajor_noswizzle(slot + SL_QDKD + kk * 256, 128, 2048), idesc1, kk > 0);
        tc_commit(bar_addr(u, B_G1));
        issued = true;
        if (!mbar_wait_bounded(bar_addr(u, B_RREADY), cpar, p.status, KDA_DEVERR_TIMEOUT, WAIT_LIMIT)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 2; ++kk)
            tc_mma_ss(u.tmem + TM_PU, make_sdesc_kmajor_noswizzle(ru + kk * 256, 128, 512),
                      make_sdesc_kmajor_noswizzle(slot + SL_INV + kk * 256, 128, 512), idesc2, kk > 0);
        tc_commit(bar_addr(u, B_G2));
        if (!mbar_wait_bounded(bar_addr(u, B_UREADY), cpar, p.status, KDA_DEVERR_TIMEOUT, WAIT_LIMIT)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 2; ++kk)
            tc_mma_ss(u.tmem + TM_S, make_sdesc_kmajor_noswizzle(ru + kk * 256, 128, 512),
                      make_sdesc_kmajor_noswizzle(slot + SL_KRMQ + kk * 256, 128, 512), idesc3, 1u);
        tc_commit(bar_addr(u, B_G3));
        tc_commit(bar_addr(u, B_EMPTY + s));
    }
    if (issued) {  // nothing of ours may still run on the tensor core when TMEM is freed
        tc_commit(bar_addr(u, B_DRAIN));
        mbar_wait_bounded(bar_addr(u, B_DRAIN), 0, p.status, KDA_DEVERR_TIMEOUT, WAIT_LIMIT);
    }
}

// ------------------------------------------------------------------------------
// TMA producer (one warp).
// ------------------------------------------------------------------------------
__device__ void tma_producer(const FwdParams& p, const TmaMaps& maps, const Unit& u, int lane) {
    int issued = 0;
#pragma unroll 1
    for (int c = 0; c < u.nchunks; ++c) {
        const int s = c & 1;
        const int k = c >> 1;
        if (c >= NSLOT && !warp_wait(bar_addr(u, B_EMPTY + s), (k - 1) & 1, p.status)) break;
        const int64_t t0 = u.bos + (int64_t)c * CH;
        const int nvalid = (int)((u.eos - t0) < CH ? (u.eos - t0) : CH);
        unsigned char* gslot = u.gbase + s * SLOT_BYTES;
        float bval = 0.f;
        if (lane < nvalid)
            bval = bf16_bits_to_f32(reinterpret_cast<const uint16_t*>(p.beta)[(t0 + lane) * p.H + u.h]);
        reinterpret_cast<float*>(gslot + SL_BETA)[lane] = bval;
        const uint32_t full = bar_addr(u, B_FULLTMA + s);
        mbar_arrive(full);
        if (lane == 0) {
            const uint32_t slot = u.base + s * SLOT_BYTES;
            mbar_arrive_expect_tx(full, 4u * CH * HD * 2u);
            tma_load_3d(slot + SL_RAWQ, &maps.q, 0, u.h, (int)t0, full);
            tma_load_3d(slot + SL_RAWK, &maps.k, 0, u.h, (int)t0, full);
            tma_load_3d(slot + SL_RAWG, &maps.g, 0, u.h, (int)t0, full);
            tma_load_3d(slot + SL_V, &maps.v, 0, u.h, (int)t0, full);
        }
        __syncwarp();
        issued = c + 1;
    }
    // copies still in flight must land before the CTA exits
    if (lane == 0) {
        for (int c = issued - NSLOT < 0 ? 0 : issued - NSLOT; c < issued; ++c)
            mbar_wait_bounded(bar_addr(u, B_FULLTMA + (c & 1)), (c >> 1) & 1, p.status, KDA_DEVERR_TIMEOUT,
                              WAIT_LIMIT);
    }
    __syncwarp();
}

// ------------------------------------------------------------------------------
// Prep group (128 threads): everything of a chunk that does not need the state.
// ------------------------------------------------------------------------------
__device__ void prep_group(const FwdParams& p, const Unit& u, int pt) {
    const int lane = pt & 31, pw = pt >> 5, gq = lane >> 2, tq = lane & 3;
    const int pp = pt & 63, half = pt >> 6, ch0 = 2 * pp;
    const float eA = expf(p.A_log[u.h]);
    const float gm = -eA * LOG2E;
    const float gb0 = gm * p.dt_bias[u.h * HD + ch0];
    const float gb1 = gm * p.dt_bias[u.h * HD + ch0 + 1];
    const float bcoef = p.lower_bound * LOG2E;   // b
    const float Cst = 16.f * bcoef;              // fixed anchor C = 16 b
    const float twoC = ex2_approx(Cst);

    __nv_bfloat16* Qc = reinterpret_cast<__nv_bfloat16*>(u.gbase + OFF_PREP);
    __nv_bfloat16* Kc = Qc + 32 * PROW;
    __nv_bfloat16* Ki = Kc + 32 * PROW;
    float* Lf = reinterpret_cast<float*>(u.gbase + OFF_PREP);   // over Q_c once it is consumed
    float* Xf = Lf + 32 * 33;
    float* tot = reinterpret_cast<float*>(u.gbase + OFF_MISC);
    float* rq = tot + 256;
    float* rk = rq + 32;

#pragma unroll 1
    for (int c = 0; c < u.nchunks; ++c) {
        const int s = c & 1;
        const uint32_t kpar = (c >> 1) & 1;
        unsigned char* gslot = u.gbase + s * SLOT_BYTES;
        if (!warp_wait(bar_addr(u, B_FULLTMA + s), kpar, p.status)) return;
        const int64_t t0 = u.bos + (int64_t)c * CH;
        const int nvalid = (int)((u.eos - t0) < CH ? (u.eos - t0) : CH);
        const unsigned char* rawq = gslot + SL_RAWQ;
        const unsigned char* rawk = gslot + SL_RAWK;
        const unsigned char* rawg = gslot + SL_RAWG;

        // ---- A: gate, local prefix over 16 tokens x 2 channels; q/k row norms
        uint32_t qw[16], kw[16];
        float G0[16], G1[16];
        {
            float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int i = 16 * half + j;
                const bool valid = i < nvalid;
                const uint32_t gw = lds32(rawg + i * 256 + ch0 * 2);
                qw[j] = valid ? lds32(rawq + i * 256 + ch0 * 2) : 0u;
                kw[j] = valid ? lds32(rawk + i * 256 + ch0 * 2) : 0u;
                float l0 = bcoef * rcp_approx(1.f + ex2_approx(fmaf(gm, bf16_lo(gw), gb0)));
                float l1 = bcoef * rcp_approx(1.f + ex2_approx(fmaf(gm, bf16_hi(gw), gb1)));
                if (!valid) l0 = l1 = 0.f;
                acc0 += l0;
                acc1 += l1;
                G0[j] = acc0;
                G1[j] = acc1;
            }
            tot[half * HD + ch0] = acc0;
            tot[half * HD + ch0 + 1] = acc1;
        }
        {
            const int r = pt >> 1, part = pt & 1;
            const unsigned char* rowp = (r < 32 ? rawq + r * 256 : rawk + (r - 32) * 256) + part * 128;
            float ss = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int ee = (e + pt) & 7;   // rotate so a quarter-warp hits distinct banks
                const uint4 w4 = *reinterpret_cast<const uint4*>(rowp + ee * 16);
                const uint32_t ws[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const float lo = bf16_lo(ws[m]), hi = bf16_hi(ws[m]);
                    ss = fmaf(lo, lo, ss);
                    ss = fmaf(hi, hi, ss);
                }
            }
            ss += __shfl_xor_sync(0xffffffffu, ss, 1);
            if (part == 0) {
                const int tok = r & 31;
                const float rn = tok < nvalid ? rsqrtf(ss + NORM_EPS) : 0.f;
                if (r < 32) rq[tok] = rn; else rk[tok] = rn;
            }
        }
        named_bar_sync(1, 128);   // raw q/k/g are no longer read after this point

        // ---- B: prefix combine, centered operands
        {
            float off0 = 0.f, off1 = 0.f, tot0 = 0.f, tot1 = 0.f;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const float a0 = tot[hh * HD + ch0], a1 = tot[hh * HD + ch0 + 1];
                if (hh < half) { off0 += a0; off1 += a1; }
                tot0 += a0;
                tot1 += a1;
            }
            const float rho0 = ex2_approx(tot0 - Cst), rho1 = ex2_approx(tot1 - Cst);
            if (half == 0) {
                float* a_s = reinterpret_cast<float*>(gslot + SL_A);
                a_s[ch0] = ex2_approx(tot0);
                a_s[ch0 + 1] = ex2_approx(tot1);
            }
            uint32_t kr0[8], kr1[8];
            float pend0 = 0.f, pend1 = 0.f;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int i = 16 * half + j;
                const float Ga = G0[j] + off0, Gb = G1[j] + off1;
                const float ep0 = ex2_approx(Ga - Cst), ep1 = ex2_approx(Gb - Cst);
                const float em0 = ex2_approx(Cst - Ga), em1 = ex2_approx(Cst - Gb);
                const float qs = rq[i] * p.scale, ks = rk[i];
                const float q0 = bf16_lo(qw[j]) * qs, q1 = bf16_hi(qw[j]) * qs;
                const float k0 = bf16_lo(kw[j]) * ks, k1 = bf16_hi(kw[j]) * ks;
                const float qc0 = q0 * ep0, qc1 = q1 * ep1;
                const float kc0 = k0 * ep0, kc1 = k1 * ep1;
                const float ki0 = k0 * em0, ki1 = k1 * em1;
                const int o = i * PROW + ch0;
                *reinterpret_cast<uint32_t*>(&Qc[o]) = pack_bf16x2(qc0, qc1);
                *reinterpret_cast<uint32_t*>(&Kc[o]) = pack_bf16x2(kc0, kc1);
                *reinterpret_cast<uint32_t*>(&Ki[o]) = pack_bf16x2(ki0, ki1);
                *reinterpret_cast<uint32_t*>(gslot + SL_QDKD + core_offset(i, ch0, HD)) =
                    pack_bf16x2(qc0 * twoC, qc1 * twoC);                       // Q_d
                *reinterpret_cast<uint32_t*>(gslot + SL_QDKD + core_offset(32 + i, ch0, HD)) =
                    pack_bf16x2(kc0 * twoC, kc1 * twoC);                       // K_d
                const float r0 = ki0 * rho0, r1 = ki1 * rho1;                  // K_r
                if (j & 1) {
                    kr0[j >> 1] = pack_bf16x2(pend0, r0);
                    kr1[j >> 1] = pack_bf16x2(pend1, r1);
                } else {
                    pend0 = r0;
                    pend1 = r1;
                }
            }
#pragma unroll
            for (int g8 = 0; g8 < 2; ++g8) {   // K_r^T rows ch0, ch0+1; tokens 16 half + 8 g8 .. +7
                const int kk = 16 * half + 8 * g8;
                *reinterpret_cast<uint4*>(gslot + SL_KRMQ + core_offset(ch0, kk, 32)) =
                    make_uint4(kr0[4 * g8], kr0[4 * g8 + 1], kr0[4 * g8 + 2], kr0[4 * g8 + 3]);
                *reinterpret_cast<uint4*>(gslot + SL_KRMQ + core_offset(ch0 + 1, kk, 32)) =
                    make_uint4(kr1[4 * g8], kr1[4 * g8 + 1], kr1[4 * g8 + 2], kr1[4 * g8 + 3]);
            }
        }
        fence_proxy_async_smem();
        named_bar_sync(1, 128);

        // ---- C: K_c K_i^T (warps 0-1) and Q_c K_i^T (warps 2-3), 16 rows x 32 columns each
        {
            const int mat = pw >> 1, mt = pw & 1;
            const __nv_bfloat16* Ab = mat ? Qc : Kc;
            float acc[4][4];
#pragma unroll
            for (int t = 0; t < 4; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                uint32_t a[4];
                ldmatrix_x4(a, Ab + (mt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * PROW + kk * 16 + (lane >> 4) * 8);
#pragma unroll
                for (int nb = 0; nb < 2; ++nb) {
                    uint32_t b[4];
                    ldmatrix_x4(b, Ki + (nb * 16 + (lane & 7) + (lane >> 4) * 8) * PROW + kk * 16 + ((lane >> 3) & 1) * 8);
                    mma_bf16_16816(acc[2 * nb], a, b[0], b[1]);
                    mma_bf16_16816(acc[2 * nb + 1], a, b[2], b[3]);
                }
            }
            named_bar_sync(1, 128);   // Q_c / K_c / K_i fully read: L and X may overwrite them
            const float* bs = reinterpret_cast<const float*>(gslot + SL_BETA);
#pragma unroll
            for (int t = 0; t < 4; ++t) {
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const int i = mt * 16 + gq + hf * 8;
                    const int j = t * 8 + 2 * tq;
                    const float v0 = acc[t][2 * hf], v1 = acc[t][2 * hf + 1];
                    // select, never multiply: the masked upper triangle may hold inf/NaN
                    if (mat == 0) {
                        Lf[i * 33 + j] = (j < i) ? bs[i] * v0 : 0.f;
                        Lf[i * 33 + j + 1] = (j + 1 < i) ? bs[i] * v1 : 0.f;
                    } else {
                        *reinterpret_cast<uint32_t*>(gslot + SL_KRMQ + core_offset(128 + i, j, 32)) =
                            pack_bf16x2((j <= i) ? v0 : 0.f, (j + 1 <= i) ? v1 : 0.f);   // Mqk
                    }
                }
            }
        }
        named_bar_sync(1, 128);

        // ---- D: INV = (I + L)^-1: diagonal 16x16 blocks by forward substitution
        if (pw == 0) {
            const int o = (lane >> 4) * 16, col = lane & 15;
            float x[16];
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) x[rr] = (rr == col) ? 1.f : 0.f;
#pragma unroll
            for (int kk = 0; kk < 16; ++kk) {
                const float xk = x[kk];
#pragma unroll
                for (int rr = kk + 1; rr < 16; ++rr) x[rr] = fmaf(-Lf[(o + rr) * 33 + o + kk], xk, x[rr]);
            }
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) Xf[(o + rr) * 33 + o + col] = x[rr];
        }
        named_bar_sync(1, 128);
#pragma unroll
        for (int it = 0; it < 2; ++it) {   // T1 = L21 A^-1 (upper-right block of X as scratch)
            const int e = it * 128 + pt, rr = e >> 4, cc = e & 15;
            float acc = 0.f;
            for (int m = cc; m < 16; ++m) acc = fmaf(Lf[(16 + rr) * 33 + m], Xf[m * 33 + cc], acc);
            Xf[rr * 33 + 16 + cc] = acc;
        }
        named_bar_sync(1, 128);
#pragma unroll
        for (int it = 0; it < 2; ++it) {   // X21 = -D^-1 T1
            const int e = it * 128 + pt, rr = e >> 4, cc = e & 15;
            float acc = 0.f;
            for (int m = 0; m <= rr; ++m) acc = fmaf(Xf[(16 + rr) * 33 + 16 + m], Xf[m * 33 + 16 + cc], acc);
            Xf[(16 + rr) * 33 + cc] = -acc;
        }
        named_bar_sync(1, 128);
#pragma unroll
        for (int it = 0; it < 4; ++it) {   // INV rows j, column pairs i (upper triangle = 0)
            const int e = it * 128 + pt, j = e >> 4, i2 = (e & 15) * 2;
            const float v0 = (i2 <= j) ? Xf[j * 33 + i2] : 0.f;
            const float v1 = (i2 + 1 <= j) ? Xf[j * 33 + i2 + 1] : 0.f;
            *reinterpret_cast<uint32_t*>(gslot + SL_INV + core_offset(j, i2, 32)) = pack_bf16x2(v0, v1);
        }
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        if (pt == 0) mbar_arrive(bar_addr(u, B_FULL + s));
    }
}

__global__ void __launch_bounds__(TC_THREADS, 2) kda_fwd_tc_kernel(const FwdParams p, const __grid_constant__ TmaMaps maps) {
    extern __shared__ unsigned char smem_raw[];
    if (*reinterpret_cast<volatile uint32_t*>(p.status) & KDA_DEVERR_CU_SEQLENS) return;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    Unit u;
    {
        const uint32_t raw = smem_u32(smem_raw);
        u.base = (raw + 1023u) & ~1023u;
        u.gbase = smem_raw + (u.base - raw);
        u.h = blockIdx.x % p.H;
        const int r = blockIdx.x / p.H;
        u.n = p.order ? p.order[r] : r;
        seq_range(p, u.n, u.bos, u.eos);
        u.nchunks = (int)((u.eos - u.bos + CH - 1) / CH);
    }
    if (tid == 0) {
        for (int s = 0; s < NSLOT; ++s) {
            mbar_init(bar_addr(u, B_FULLTMA + s), 33);
            mbar_init(bar_addr(u, B_FULL + s), 1);
            mbar_init(bar_addr(u, B_EMPTY + s), 1);
        }
        for (int b = B_G1; b < B_COUNT; ++b) mbar_init(bar_addr(u, b), 1);
        mbar_fence_init();
    }
    if (warp == W_TMA && lane == 0) {
        tma_prefetch_desc(&maps.q);
        tma_prefetch_desc(&maps.k);
        tma_prefetch_desc(&maps.v);
        tma_prefetch_desc(&maps.g);
    }
    if (warp == W_MMA) {
        tmem_alloc(u.base + OFF_TMEMADDR, TM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    u.tmem = *reinterpret_cast<volatile uint32_t*>(u.gbase + OFF_TMEMADDR);

    if (warp < 4) {
        tmem_group(p, u, tid);
    } else if (warp == W_MMA) {
        if (lane == 0) mma_issuer(p, u);
    } else if (warp == W_TMA) {
        tma_producer(p, maps, u, lane);
    } else {
        prep_group(p, u, tid - W_PREP0 * 32);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == W_MMA) {
        tc_fence_after();
        tmem_dealloc(u.tmem, TM_COLS);
    }
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
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

// [T_total, H, 128] bf16 viewed as a 3-D tensor (d, h, t); boxes of 128 x 1 x 32.
bool encode_tokens_map(CUtensorMap* m, const void* ptr, int64_t T_total, int H) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)HD, (cuuint64_t)H, (cuuint64_t)(T_total > 0 ? T_total : 1)};
    const cuuint64_t strides[2] = {(cuuint64_t)HD * 2, (cuuint64_t)H * HD * 2};
    const cuuint32_t box[3] = {(cuuint32_t)HD, 1, (cuuint32_t)CH};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

size_t fwd_tc_smem_bytes() { return SMEM_BYTES; }

cudaError_t launch_fwd_tc(const FwdParams& p, cudaStream_t stream) {
    const int units = p.nseq * p.H;
    if (units == 0) return cudaSuccess;
    TmaMaps maps;
    if (!encode_tokens_map(&maps.q, p.q, p.T_total, p.H) || !encode_tokens_map(&maps.k, p.k, p.T_total, p.H) ||
        !encode_tokens_map(&maps.v, p.v, p.T_total, p.H) || !encode_tokens_map(&maps.g, p.g, p.T_total, p.H))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(kda_fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    kda_fwd_tc_kernel<<<units, TC_THREADS, SMEM_BYTES, stream>>>(p, maps);
    return cudaGetLastError();
}

}  // namespace kda
