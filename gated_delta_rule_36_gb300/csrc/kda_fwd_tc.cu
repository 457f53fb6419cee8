// KDA chunked prefill forward on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// One CTA per (sequence, head) unit, two CTAs per SM; with no more units than SMs, one CTA
// per SM (a second instantiation); with at most a quarter as many, a cluster of four CTAs
// per unit, three of which prepare chunks for the fourth's chain, and with at most half as
// many a cluster of two, one CTA preparing for the other (the cluster schedules, below).  The fp32 V x K state stays resident in Tensor Memory for the whole sequence
// ("FlashInfer PR #4262" notes, section 6); the recurrent GEMMs run as tcgen05.mma with
// fp32 TMEM accumulators, and the small intra-chunk products as warp-level mma.sync
// (section 7).
//
// Per chunk (section 3 notation; R = V^T - P, B2 = diag(beta) INV^T):
//   GEMM1  [O_0 | P] = S_bf16 [Q_d | K_d]^T           M128 N64  K128  (A = bf16 S from TMEM)
//          P -= V^T                                   M128 N32  K32   (A = V from SMEM, B = -I)
//          S = S diag(a)                              CUDA cores, before GEMM3 (its bf16 copy, taken
//                                                     first, is GEMM1's A operand)
//   GEMM2  U = (-R) (-B2)                             M128 N32  K32   (A = -R in bf16 from TMEM)
//   GEMM3  S += U K_r,  O += U Mqk^T                  M128 N128 + N32, K32 (A = U in bf16 from TMEM)
// The prep warps build Q_d, K_d, K_r, Mqk and L for a chunk (mma.sync for the 32 x 32
// products) and the inverse warp turns L into -B2, while the chain runs the previous one.
//
// Warp roles (448 threads, up to 72 registers each, with two CTAs per SM):
//   warps 0-3   chain group: thread v owns state row v (TMEM lane v): initial/final
//               state I/O, the bf16 copy of S, the decay, R' and the chunk output O.
//               Single threads of its warps issue the TMA loads of q, k, g and beta
//               (warp 2) and the output store and v loads (warp 3); warp 0 owns the
//               TMEM allocation.
//   warps 4-11  prep group: gate, prefix, q/k norms, centered operands (section 2),
//               K_c K_i^T and Q_c K_i^T with mma.sync (three of its warps, one block pair each).
//   warp 12     inverse warp: (I + L)^-1 and -B2 of chunk c while the prep group
//               builds chunk c + 1.
//   warp 13     MMA warp: issues the chain's tensor-core MMAs as the chain hands each A
//               operand over (named barriers, arrive / sync), GEMM1's first half of k while
//               the chain still converts the second half of S.
//   warps 14-17 (one CTA per SM only, 576 threads) epilogue warps: read each chunk's O out of
//               a double-buffered pair of TMEM column groups, stage and store it, and refill
//               the slot's v, so that the output leaves the chain's path (as in the cluster home).
// A two-slot SMEM ring (three slots with one CTA per SM, whose shared memory has room)
// carries prepared chunks to the strictly ordered recurrent consumer (section 4): the
// chain refills a slot as soon as GEMM3 has read it, and
// every mbarrier wait is bounded (on expiry: KDA_DEVERR_TIMEOUT and the CTA winds down).
//
// TMEM columns (256 per CTA): [0,128) fp32 S; [128,160) O; [160,192) P;
// [192,256) bf16 copy of S (two values per column), whose first 16 columns hold R'
// between GEMM1 and GEMM3.
#include <cuda.h>

#include <atomic>

#include "kda_device.cuh"
#include "kda_kernels.h"
#include "kda_sm100.cuh"

namespace kda {
namespace {

constexpr int TC_THREADS = 448;
constexpr int W_PREP0 = 4, PREP_WARPS = 8;
constexpr int W_INV = W_PREP0 + PREP_WARPS;   // the inverse warp: (I + L)^-1 of chunk c while the prep warps take c + 1
constexpr int W_ISSUE = W_INV + 1;            // the MMA warp
constexpr int TC_THREADS_LE = 576;            // one CTA per SM: warps 14-17 read the output out
// Duties of the chain group, spread over its warps (one per SM sub-partition): warp 2
// refills q, k, g and beta, warp 3 stores each output tile and then refills v, whose slot
// region held the tile.  (With two CTAs on an SM lane 0 of the MMA warp issues alone; with
// one CTA per SM the whole warp issues through elect.sync.)
constexpr int T_TMA = 64, W_BETA = 2, T_STORE = 96;
constexpr int PREP_THREADS = PREP_WARPS * 32;
constexpr int NSLOT = 2;     // the ring of a CTA with its own chain (two CTAs per SM)
constexpr int NSL1 = 3;      // the ring of one CTA per SM: chunk c in slot c % 3
constexpr int MAX_RING = 4;  // the ring of a cluster-of-two helper
#ifdef KDA_WAIT_TEST
// The test-only build of the timeout path: waits give up after ~2 ms, and the inverse warp
// skips its FULLD arrival for local chunk p.test_skip_chunk (chosen by the host), so that a
// wait of the chain runs out and the kernel has to wind down and return KDA_DEVERR_TIMEOUT.
constexpr long long WAIT_LIMIT = 4000000LL;
#else
constexpr long long WAIT_LIMIT = 2000000000LL;  // SM cycles (~1 s) before a wait gives up
#endif

// Slot layout (bytes).  Raw q/k/g land where derived operands are later written.
constexpr uint32_t SL_QDKD = 0;       // [Q_d | K_d]: 64 rows x 128, K-major, 128-B swizzle (raw q at 0, k at 8192)
constexpr uint32_t SL_RAWQ = 0, SL_RAWK = 8192;
constexpr uint32_t SL_KR = 16384;     // K_r [32 tokens][128]: two 64-channel blocks, 128-B swizzle (MN-major B of GEMM3)
constexpr uint32_t SL_RAWG = 16384;
constexpr uint32_t SL_V = 24576;      // raw v, two [32][64] 128-B swizzled blocks (MN-major A of P -= V^T);
                                      // after GEMM1 the chunk output staging tile [32 tokens][128]
constexpr uint32_t SL_MQT = 32768;    // Mqk [32 i][32 j], K-major core layout (B of O += U Mqk^T)
constexpr uint32_t SL_INV = 34816;    // -B2 [32 i][32 j] = -beta_j INV[i][j], K-major core layout (B of GEMM2)
constexpr uint32_t SL_A = 36864;      // fp32 [128]: 2^G_T
constexpr uint32_t SL_BETA = 37376;   // fp32 [32]
constexpr uint32_t SLOT_BYTES = 37888;

// Prep scratch (per CTA).  32 x 128 bf16 tiles with 16-byte chunks XOR-swizzled by
// (row % 8), so that both the row-wise stores and ldmatrix reads are conflict-free.
constexpr uint32_t OFF_QC = NSLOT * SLOT_BYTES;   // Q_c
constexpr uint32_t OFF_KC = OFF_QC + 8192;        // K_c
constexpr uint32_t OFF_KI = OFF_KC + 8192;        // K_i
constexpr uint32_t OFF_MISC = OFF_KI + 8192;      // tot[8][128], rq[32], rk[32]
constexpr uint32_t MISC_BYTES = (8 * 128 + 64 + 128) * 4;
// L = strictLower(diag(beta) K_c K_i^T) in fp32, its three nonzero 16 x 16 blocks, each
// column-major with a column stride of LB floats: L11 at 0, L22 at 336 (16 floats past its
// 320-float block, so that the two half-warps of the substitution read different banks), L21 at 672.
constexpr int LB = 20;
constexpr int LB_11 = 0, LB_22 = 336, LB_21 = 672;
constexpr uint32_t OFF_L = OFF_MISC + MISC_BYTES;
constexpr uint32_t L_BYTES = (LB_21 + 16 * LB) * 4;
// X = INV's two diagonal blocks (fp32, row-major, row stride XB floats): X11 at 0, X22 at
// XB_22 (16 floats past its block for the same reason).  Private to the inverse warp.
constexpr int XB = 24;
constexpr int XB_22 = 16 * XB + 16;
constexpr uint32_t OFF_X = OFF_L + L_BYTES;
constexpr uint32_t X_BYTES = (XB_22 + 16 * XB) * 4;
constexpr uint32_t OFF_NEGI = OFF_X + X_BYTES;   // -I (bf16 32 x 32, K-major core layout)
constexpr uint32_t OFF_BAR = OFF_NEGI + 2048;
// Per slot: FULLTMA (q, k, g boxes and beta landed), FULLV (v box landed; three slots in a
// cluster's home CTA), AREADY (the prep warps wrote a), FULLP (the prep warps finished the
// chunk's operands and L), FULLD (the inverse warp wrote -B2).  LFREE: the inverse warp has
// read L.  Chain: G1, G2, G3 (MMA commits).  Cluster schedule (below): FULLOP (home slot s
// holds a pushed chunk: the arming arrival and the copies' bytes), HSLOT (on a helper: its home
// slot is free for its next chunk), COPIED (on a helper: the push of the chunk in its slot b
// has landed and been consumed).  OREADY b / OFREE b (cluster home): the chain has finished
// chunk c (its O in buffer b = c % 2) / the epilogue warps have read the O out.
enum {
    B_FULLTMA = 0, B_FULLV = 4, B_AREADY = 7, B_FULLP = 11, B_FULLD = 15, B_LFREE = 19, B_G1, B_G2, B_G3,
    B_FULLOP = 23, B_HSLOT = 26, B_COPIED = 29, B_OREADY = 33, B_OFREE = 35, B_COUNT = 37
};
constexpr uint32_t OFF_TMEMADDR = OFF_BAR + B_COUNT * 8;
constexpr uint32_t OFF_PUSHED = OFF_TMEMADDR + 4;   // (cluster home) pushes issued by helper h, at + 4 h
constexpr uint32_t SMEM_USED = OFF_TMEMADDR + 16;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;      // slack to align the base to 1 KB
static_assert(SLOT_BYTES % 1024 == 0, "slots must keep the 128-B swizzle atoms 1 KB aligned");
static_assert(2 * (SMEM_BYTES + 1024) <= 233472, "two CTAs must fit one SM");
static_assert(OFF_QC % 256 == 0 && OFF_KC % 256 == 0 && OFF_KI % 256 == 0, "scratch tiles must be 256-B aligned");
static_assert(OFF_L % 16 == 0 && OFF_X % 16 == 0 && OFF_NEGI % 16 == 0, "float4 / descriptor alignment");

// Cluster schedules, for few units: a cluster of 1 + kNH CTAs per unit.  The home CTA (rank
// 0) runs the chain over NSH slots; helper h (rank h + 1) prepares the chunks c = h (mod kNH)
// in its own ring of slots with the prep and inverse warps (two slots with three helpers,
// four with one) and pushes each finished chunk into home slot c % NSH with a shared ->
// distributed shared memory bulk copy.
constexpr int NSH = 3;
__host__ __device__ constexpr int cl_ring(int nh) { return nh == 1 ? 4 : 2; }
constexpr uint32_t OFF_SLOT2 = (SMEM_USED + 1023) & ~1023u;   // the third and fourth slots
__host__ __device__ constexpr uint32_t smem_bytes_cl(int nh) { return OFF_SLOT2 + (nh == 1 ? 2 : 1) * SLOT_BYTES + 1024; }
static_assert(smem_bytes_cl(1) <= 232448 && smem_bytes_cl(3) <= 232448, "the cluster layouts must fit one CTA's shared memory");
// One CTA per SM with its own prep: the same three slots (slot 2 past the scratch).
constexpr uint32_t SMEM_BYTES_LE = smem_bytes_cl(3);

// bf16 state resident in shared memory (a design alternative, one CTA per SM): the 128 x 128
// state as GEMM1's A operand, K-major with the 128-byte swizzle, two 64-column blocks of 16 KB.
constexpr uint32_t OFF_STATE = (SMEM_USED + 1023) & ~1023u;
constexpr uint32_t STATE_BLOCK = 128 * 128;
constexpr uint32_t SMEM_BYTES_SS = OFF_STATE + 2 * STATE_BLOCK + 1024;
static_assert(SMEM_BYTES_SS <= 232448, "the shared-memory state layout must fit one CTA's shared memory");
// The pushed part of a slot: [Q_d | K_d] and K_r (bytes [0, SL_V)), then Mqk, -B2 and a
// (bytes [SL_MQT, SL_BETA)); v is the home CTA's own.
constexpr uint32_t PUSH_A = SL_V, PUSH_B = SL_BETA - SL_MQT, PUSH_BYTES = PUSH_A + PUSH_B;
static_assert(PUSH_A % 16 == 0 && PUSH_B % 16 == 0 && SL_MQT % 16 == 0, "bulk copies move 16-byte units");
static_assert(OFF_PUSHED + 4 * 3 <= SMEM_USED, "the push counts live beside the TMEM address");
__host__ __device__ constexpr uint32_t slot_off(int s) { return s < 2 ? (uint32_t)s * SLOT_BYTES : OFF_SLOT2 + (uint32_t)(s - 2) * SLOT_BYTES; }

// Shared -> distributed shared memory bulk copy: `bytes` (a multiple of 16) from this CTA's
// `src` to `dst` in a peer CTA, completing its transaction bytes on the peer's mbarrier `mbar`
// (dst and mbar are shared::cluster addresses, 16- and 8-byte aligned).
__device__ __forceinline__ void bulk_copy_to_peer(uint32_t dst, uint32_t src, uint32_t bytes, uint32_t mbar) {
    asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
                 "r"(src), "r"(bytes), "r"(mbar)
                 : "memory");
}
// A 32-bit store into a peer CTA's shared memory.
__device__ __forceinline__ void st_dsmem_u32(uint32_t cluster_addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;\n" ::"r"(cluster_addr), "r"(v) : "memory");
}

// Index of element (i, j), j < 16 or i, j >= 16, of L in its block layout.
__host__ __device__ constexpr int l_index(int i, int j) {
    return (i < 16 ? LB_11 : (j < 16 ? LB_21 : LB_22)) + (j & 15) * LB + (i & 15);
}

// TMEM columns: S (fp32), O, P then U (fp32), and the bf16 copy of S whose first 16
// columns carry -R and then U between the GEMMs.
constexpr uint32_t TM_S = 0, TM_O = 128, TM_P = 160, TM_SB = 192, TM_COLS = 256;
// The cluster schedule's home CTA has its SM to itself and takes all 512 columns: [O | P] is
// double-buffered by chunk parity (chunk c uses columns TM_O + 128 (c % 2)), so that the
// epilogue warps read chunk c's O while the chain runs chunk c + 1.
constexpr uint32_t TM_OP_STRIDE = 128, TM_COLS_CL = 512;

struct TmaMaps {
    CUtensorMap q, k, v, g, out;   // v, out: boxes of 64 channels with the 128-byte swizzle
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
__device__ __forceinline__ float2 bf2_to_f2(uint32_t w) { return make_float2(bf16_lo(w), bf16_hi(w)); }
__device__ __forceinline__ uint32_t f2_to_bf2(float2 x) { return pack_bf16x2(x.x, x.y); }

// byte offset of (row, col) in a 32 x 128 bf16 scratch tile (chunk ^= row % 8)
__device__ __forceinline__ uint32_t sc128(int row, int col) {
    return (uint32_t)(row * 256 + ((((col >> 3) ^ (row & 7))) << 4) + ((col & 7) << 1));
}

// Range checks of the KDA_CHECKED build (a second library for the tests; the product build
// compiles them away).  The shared-memory and Tensor-Memory layouts are compile-time constants
// checked by the static_asserts above; what depends on the data or the thread is checked here:
// global state rows, beta and output rows, token coordinates of the tensor copies, and the
// row / column arguments of the tile index functions.  A failed check sets
// KDA_DEVERR_INTERNAL in the status word and clamps the index into range, so the access stays
// in bounds and the kernel runs to its end: the build never faults on a bad index.
#ifdef KDA_CHECKED
static __shared__ uint32_t* s_chk_status;
__device__ __forceinline__ int64_t chk_range(int64_t x, int64_t lo, int64_t hi) {
    if (x >= lo && x < hi) return x;
    atomicOr(s_chk_status, KDA_DEVERR_INTERNAL);
    return lo;
}
#define KDA_CHK(x, lo, hi) chk_range((int64_t)(x), (int64_t)(lo), (int64_t)(hi))
#else
#define KDA_CHK(x, lo, hi) (x)
#endif
// tile index functions with their arguments checked
__device__ __forceinline__ uint32_t sw128_at(int r, int k, int rows) {
    return sw128_offset((int)KDA_CHK(r, 0, rows), (int)KDA_CHK(k, 0, HD), rows);
}
__device__ __forceinline__ uint32_t core_at(int r, int k, int kt) {
    return core_offset((int)KDA_CHK(r, 0, CH), (int)KDA_CHK(k, 0, kt), kt);
}
__device__ __forceinline__ int l_at(int i, int j) {
    i = (int)KDA_CHK(i, 0, CH);
    j = (int)KDA_CHK(j, 0, (i < 16 ? 16 : CH));   // L keeps no upper-right block
    return l_index(i, j);
}
__device__ __forceinline__ uint32_t sc_at(int row, int col) { return sc128((int)KDA_CHK(row, 0, CH), (int)KDA_CHK(col, 0, HD)); }

// Bounded wait, with the verdict made uniform over the warp.  `max_sleep_ns` > 0 backs
// off between polls (long waits off the critical path).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, uint32_t* status,
                                          uint32_t max_sleep_ns = 0) {
    const bool ok = mbar_wait_bounded(bar, parity, status, KDA_DEVERR_TIMEOUT, WAIT_LIMIT, max_sleep_ns);
    return __all_sync(0xffffffffu, ok);
}

// Wind-down after an expired wait.  A group's named barriers are not bounded, so a warp
// whose wait expired keeps meeting its group at every barrier the group still has ahead
// (plain bar.sync, no waits and no work) until the sequence ends.  Its siblings either finish
// normally or see a wait of their own expire (whatever the wound-down warp would have
// produced never comes) and join it, so no warp is ever left at a barrier, and the fast path
// keeps its code as it is.
__device__ __noinline__ void epilogue_wind_down(int c, int nchunks) {
    for (; c < nchunks; ++c) named_bar_sync(3, 128);
}
// Prep group: barrier k of its local chunk j (0: after phase A, 1: after the prefix scan,
// 2: after phase B, 3: after phase C).
__device__ __noinline__ void prep_wind_down(int j, int k, int nloc) {
    for (; j < nloc; ++j, k = 0)
        for (; k < 4; ++k) named_bar_sync(1, PREP_THREADS);
}

// 16 state values of row `off` (element offset) as fp32 bits (zeros without an initial state).
__device__ __forceinline__ void load_state16(const FwdParams& p, size_t off, uint32_t (&r)[16]) {
    off = (size_t)KDA_CHK(off, 0, (int64_t)p.nseq * p.H * HD * HD - 15);
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
    off = (size_t)KDA_CHK(off, 0, (int64_t)p.nseq * p.H * HD * HD - 15);
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

// The 32 fp32 P columns of this lane (-R after GEMM1, U after GEMM2) -> bf16 -> the
// first 16 columns of the bf16 copy of S (the A operand of the next GEMM).
__device__ __forceinline__ void p_cols_to_bf16(uint32_t lane_addr, uint32_t tm_p = TM_P) {
    uint32_t rp[16];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        uint32_t pr[16];
        tmem_ld16(lane_addr + tm_p + hh * 16, pr);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 8; ++i) rp[hh * 8 + i] = pack_bf16x2(u2f(pr[2 * i]), u2f(pr[2 * i + 1]));
    }
    tmem_st16(lane_addr + TM_SB, rp);
    tmem_wait_st();
}

// The chain's hand-offs to the MMA warp: named barriers that the chain warps arrive on
// (bar.arrive, no wait) and the MMA warp syncs on, 160 threads each.  G1A / G1B: the first /
// second half of the bf16 copy of S is in place (GEMM1's k blocks 0-3 / 4-7); G2: -R is in
// place and -B2 has been written; G3: U is in place.  Each one is used once per chunk, and
// the next use of an id waits for an MMA commit that follows the MMA warp's sync on it.
constexpr int NB_G1A = 4, NB_G1B = 5, NB_G2 = 6, NB_G3 = 7, NB_HAND = 160;

// A finished half of the state pass: this thread's TMEM (or shared-memory) stores are
// complete and ordered before the MMA warp's GEMM1 issue.
template <bool kSmem>
__device__ __forceinline__ void hand_off_half(int id) {
    tmem_wait_st();
    if constexpr (kSmem) fence_proxy_async_smem();   // GEMM1 reads the tile
    tc_fence_before();
    named_bar_arrive(id, NB_HAND);
}

// One pass over S: its bf16 copy (the next GEMM1 operand, taken before the decay), then
// S = S diag(a) in place with the next chunk's a (its GEMM3 adds to the decayed S).
// Once the first half of the copy is in place it is handed to the MMA warp (G1A).
// kBf16State (the state-precision ablation) decays the bf16 copy instead, i.e. rounds the
// carried state to bf16 at every chunk boundary, as a bf16 state store would.
// kSmem (the shared-memory state alternative): the bf16 copy goes to row `v` of the state tile
// in shared memory (GEMM1's A operand) instead of Tensor Memory; with kBf16State it is also the
// state that is decayed and updated.
template <bool kBf16State, bool kSmem = false>
__device__ __forceinline__ void copy_and_decay(uint32_t lane_addr, const float* a_s, unsigned char* st = nullptr,
                                               int v = 0) {
#pragma unroll 1
    for (int piece = 0; piece < 8; ++piece) {
        uint32_t r[16];
        tmem_ld16(lane_addr + TM_S + piece * 16, r);
        tmem_wait_ld();
        uint32_t b[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) b[j] = pack_bf16x2(u2f(r[2 * j]), u2f(r[2 * j + 1]));
        if constexpr (kSmem) {
            *reinterpret_cast<uint4*>(st + sw128_at(v, 16 * piece, 128)) = make_uint4(b[0], b[1], b[2], b[3]);
            *reinterpret_cast<uint4*>(st + sw128_at(v, 16 * piece + 8, 128)) = make_uint4(b[4], b[5], b[6], b[7]);
        } else {
            tmem_st8(lane_addr + TM_SB + piece * 8, b);
        }
        if (kBf16State) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                r[2 * j] = b[j] << 16;
                r[2 * j + 1] = b[j] & 0xffff0000u;
            }
        }
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
        if (piece == 3) hand_off_half<kSmem>(NB_G1A);
    }
}

// The same pass software-pipelined: piece p + 1 is loaded while piece p is converted,
// decayed and stored.  It shortens the chain of a CTA that has its SM to itself (3.9 % on a
// 32-unit workload) and costs throughput when two CTAs share an SM, so only the one-CTA-
// per-SM instantiation uses it.
template <bool kBf16State>
__device__ __forceinline__ void copy_and_decay_pipelined(uint32_t lane_addr, const float* a_s) {
    uint32_t r[2][16];
    tmem_ld16(lane_addr + TM_S, r[0]);
    tmem_wait_ld_regs(r[0]);
#pragma unroll
    for (int piece = 0; piece < 8; ++piece) {
        uint32_t (&c)[16] = r[piece & 1];
        if (piece + 1 < 8) tmem_ld16(lane_addr + TM_S + (piece + 1) * 16, r[(piece + 1) & 1]);
        uint32_t b[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) b[j] = pack_bf16x2(u2f(c[2 * j]), u2f(c[2 * j + 1]));
        tmem_st8(lane_addr + TM_SB + piece * 8, b);
        if (kBf16State) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                c[2 * j] = b[j] << 16;
                c[2 * j + 1] = b[j] & 0xffff0000u;
            }
        }
        const float4* a4 = reinterpret_cast<const float4*>(a_s + piece * 16);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float4 a = a4[j];
            const float2 x0 = __fmul2_rn(make_float2(u2f(c[4 * j]), u2f(c[4 * j + 1])), make_float2(a.x, a.y));
            const float2 x1 = __fmul2_rn(make_float2(u2f(c[4 * j + 2]), u2f(c[4 * j + 3])), make_float2(a.z, a.w));
            c[4 * j] = f2u(x0.x); c[4 * j + 1] = f2u(x0.y);
            c[4 * j + 2] = f2u(x1.x); c[4 * j + 3] = f2u(x1.y);
        }
        tmem_st16(lane_addr + TM_S + piece * 16, c);
        if (piece == 3) hand_off_half<false>(NB_G1A);
        if (piece + 1 < 8) tmem_wait_ld_regs(r[(piece + 1) & 1]);
    }
}

// ------------------------------------------------------------------------------
// Chain group: state row v = TMEM lane v; single threads issue the TMA copies.
// ------------------------------------------------------------------------------
__device__ __forceinline__ int chunk_valid(const Unit& u, int c) {
    const int64_t t0 = u.bos + (int64_t)c * CH;
    return (int)((u.eos - t0) < CH ? (u.eos - t0) : CH);
}

// q, k, g boxes of chunk c into slot s (on FULLTMA, which beta completes).
__device__ __forceinline__ void load_qkg(const TmaMaps& maps, const Unit& u, int c, int s) {
    const int t0 = (int)KDA_CHK(u.bos + (int64_t)c * CH, u.bos, u.eos);
    const uint32_t slot = u.base + slot_off(s), full = bar_addr(u, B_FULLTMA + s);
    mbar_arrive_expect_tx(full, 3u * CH * HD * 2u);
    tma_load_3d(slot + SL_RAWQ, &maps.q, 0, u.h, t0, full);
    tma_load_3d(slot + SL_RAWK, &maps.k, 0, u.h, t0, full);
    tma_load_3d(slot + SL_RAWG, &maps.g, 0, u.h, t0, full);
}

// the v box of chunk c (two 64-channel halves, 128-byte swizzle) into slot s, on FULLV.
__device__ __forceinline__ void load_v(const TmaMaps& maps, const Unit& u, int c, int s) {
    const int t0 = (int)KDA_CHK(u.bos + (int64_t)c * CH, u.bos, u.eos);
    const uint32_t slot = u.base + slot_off(s), full = bar_addr(u, B_FULLV + s);
    mbar_arrive_expect_tx(full, CH * HD * 2u);
    tma_load_3d(slot + SL_V, &maps.v, 0, u.h, t0, full);
    tma_load_3d(slot + SL_V + 4096, &maps.v, 64, u.h, t0, full);
}

// Pull chunk c's q, k, g, v boxes into L2 ahead of the loads that refill its slot.
__device__ __forceinline__ void prefetch_chunk(const TmaMaps& maps, const Unit& u, int c) {
    const int t0 = (int)(u.bos + (int64_t)c * CH);
    tma_prefetch_l2_3d(&maps.q, 0, u.h, t0);
    tma_prefetch_l2_3d(&maps.k, 0, u.h, t0);
    tma_prefetch_l2_3d(&maps.g, 0, u.h, t0);
    tma_prefetch_l2_3d(&maps.v, 0, u.h, t0);
    tma_prefetch_l2_3d(&maps.v, 64, u.h, t0);
}

// beta of token `lane` of chunk c, by a plain load: its token stride is 2H bytes, too narrow
// for a tensor box when H is small.  The load is predicated and its bits are kept as they are
// (BETA_NONE past the end), so a warp that loads beta ahead does not wait for the load until
// it uses the value (beta_of).  kBetaLogit (KDA_FLAG_BETA_LOGIT): the stored value is a logit
// and beta = sigmoid(logit).
constexpr uint32_t BETA_NONE = 0x10000u;   // no token: beta = 0 (not a 16-bit pattern)
__device__ __forceinline__ uint32_t load_beta_bits(const FwdParams& p, const Unit& u, int c, int lane) {
    const int64_t t0 = u.bos + (int64_t)c * CH;
    uint32_t raw = BETA_NONE;
    if (lane < chunk_valid(u, c))
        raw = reinterpret_cast<const uint16_t*>(p.beta)[KDA_CHK((t0 + lane) * p.H + u.h, 0, p.T_total * p.H)];
    return raw;
}
template <bool kBetaLogit>
__device__ __forceinline__ float beta_of(uint32_t raw) {
    if (raw == BETA_NONE) return 0.f;
    const float b = bf16_bits_to_f32((uint16_t)raw);
    if constexpr (kBetaLogit) return rcp_approx(1.f + ex2_approx(-b * LOG2E));
    return b;
}
template <bool kBetaLogit>
__device__ __forceinline__ float load_beta(const FwdParams& p, const Unit& u, int c, int lane) {
    return beta_of<kBetaLogit>(load_beta_bits(p, u, c, lane));
}

__device__ __forceinline__ void put_beta(const Unit& u, int s, int lane, float b) {
    reinterpret_cast<float*>(u.gbase + slot_off(s) + SL_BETA)[lane] = b;
    mbar_arrive(bar_addr(u, B_FULLTMA + s));
}

// Wind-down of the chain warps (see above).  Step k of chunk c: 0 the state pass before it
// (hand-offs G1A, G1B), 1 the hand-off G2, 2 the hand-off G3, 3 the barrier after the output
// staging (not in the cluster home, whose epilogue warps stage the output).  A wound-down
// warp syncs on the hand-offs instead of arriving: with no waits in between, plain arrivals
// could reach the next generation of a barrier before the MMA warp has met the current one.
template <bool kEpi = false>
__device__ __noinline__ void chain_wind_down(int c, int k, int nchunks) {
    for (; c < nchunks; ++c, k = 0)
        for (; k < 4; ++k) {
            if (k == 0) {
                named_bar_sync(NB_G1A, NB_HAND);
                named_bar_sync(NB_G1B, NB_HAND);
            } else if (k == 1) {
                named_bar_sync(NB_G2, NB_HAND);
            } else if (k == 2) {
                named_bar_sync(NB_G3, NB_HAND);
            } else if (!kEpi) {
                named_bar_sync(2, 128);
            }
        }
}
// Wind-down of the MMA warp from the start of chunk c: it meets every hand-off still ahead.
__device__ __noinline__ void mma_wind_down(int c, int nchunks) {
    for (; c < nchunks; ++c) {
        named_bar_sync(NB_G1A, NB_HAND);
        named_bar_sync(NB_G1B, NB_HAND);
        named_bar_sync(NB_G2, NB_HAND);
        named_bar_sync(NB_G3, NB_HAND);
    }
}

// kCl: the chain of a cluster's home CTA.  Its NSH slots receive pushed chunks (FULLOP
// stands for AREADY, FULLP and FULLD at once), it loads v alone, and once GEMM3 has read a slot
// it signals OREADY, on which the epilogue warps also hand the slot back to its helper.
// kSmemState: the bf16 state resident in shared memory (with kBf16State and kWarpIssue).
// kEpi: epilogue warps of the CTA read the output out (the cluster home, or one CTA per SM
// with epilogue warps): O is double-buffered and the chain only signals OREADY.
// kR3: one CTA per SM with its own prep: a ring of three slots, chunk c in slot c % 3.
template <bool kBf16State, bool kWarpIssue, bool kBetaLogit, bool kCl, bool kSmemState = false, bool kEpi = kCl,
          bool kR3 = false>
__device__ void chain_group(const FwdParams& p, const TmaMaps& maps, const Unit& u, int pt) {
    static_assert(!kSmemState || (kBf16State && kWarpIssue && !kCl), "the shared-memory state runs one CTA per SM");
    static_assert(!kR3 || (kEpi && !kCl), "the three-slot ring has epilogue warps");
    unsigned char* st_smem = u.gbase + OFF_STATE;
    constexpr int NS = kCl ? NSH : (kR3 ? NSL1 : NSLOT);   // slots in the ring
    constexpr bool kCtr = kCl || kR3;                        // slot and round kept as counters
    const int w = pt >> 5, lane = pt & 31;
    const uint32_t lane_addr = u.tmem + ((uint32_t)(w * 32) << 16);
    const int v = pt;
    const size_t srow = (((size_t)u.n * p.H + u.h) * HD + v) * HD;

    // initial state -> TMEM; an empty sequence copies it straight through
#pragma unroll 1
    for (int piece = 0; piece < 8; ++piece) {
        uint32_t r[16];
        load_state16(p, srow + piece * 16, r);
        if (u.nchunks == 0) store_state16(p, srow + piece * 16, r);
        else tmem_st16(lane_addr + TM_S + piece * 16, r);
    }
    if (u.nchunks == 0) return;
    const int first = u.nchunks < NS ? u.nchunks : NS;
    if constexpr (!kCl) {
        if (pt == T_TMA)
            for (int c = 0; c < first; ++c) load_qkg(maps, u, c, c);
        if (w == W_BETA)
            for (int c = 0; c < first; ++c) put_beta(u, c, lane, load_beta<kBetaLogit>(p, u, c, lane));
    }
    if (pt == T_STORE)
        for (int c = 0; c < first; ++c) load_v(maps, u, c, c);
    // beta of chunk c + 2 goes into the slot during iteration c; it is loaded an iteration
    // ahead (its 2-byte loads, 2H bytes apart, miss the caches)
    uint32_t beta_ahead = (!kCl && w == W_BETA && NS < u.nchunks) ? load_beta_bits(p, u, NS, lane) : BETA_NONE;
    int issued = first;    // chunks whose boxes were requested
    int vissued = first;   // chunks whose v boxes were requested
    {   // -I: B operand of P -= V^T; thread = (row n, 8-column block)
        const int n = pt >> 2, kb = pt & 3;
        const uint32_t m1 = ((n >> 3) == kb) ? ((n & 1) ? 0xBF800000u : 0x0000BF80u) : 0u;   // bf16 -1 at column n
        const int wi = (n & 7) >> 1;
        *reinterpret_cast<uint4*>(u.gbase + OFF_NEGI + core_at(n, 8 * kb, 32)) =
            make_uint4(wi == 0 ? m1 : 0u, wi == 1 ? m1 : 0u, wi == 2 ? m1 : 0u, wi == 3 ? m1 : 0u);
        fence_proxy_async_smem();
    }
    tmem_wait_st();
    // the state pass before chunk c: the bf16 copy of S (GEMM1's A operand) handed to the MMA
    // warp in two halves, and the decay by chunk c's a
    auto state_pass = [&](const float* a_s) {
        if constexpr (kSmemState)
            copy_and_decay<kBf16State, true>(lane_addr, a_s, st_smem, pt);
        else if constexpr (kWarpIssue)
            copy_and_decay_pipelined<kBf16State>(lane_addr, a_s);
        else
            copy_and_decay<kBf16State>(lane_addr, a_s);
        hand_off_half<kSmemState>(NB_G1B);
    };
    bool ok = warp_wait(bar_addr(u, kCl ? B_FULLOP : B_AREADY), 0, p.status, 256);   // a of chunk 0
    if (ok) state_pass(reinterpret_cast<const float*>(u.gbase + SL_A));
    else chain_wind_down<kEpi>(0, 0, u.nchunks);

    int sc = 0, kq = 0;   // (cluster home) slot c % NS and round c / NS
    // chain trace (cluster schedule): SM clock at KDA_TRACE_POINTS steps of each chunk of one unit
    const bool trace_me = kCl && p.trace != nullptr && (int64_t)u.n * p.H + u.h == p.trace_unit;
    auto stamp = [&](int c, int i) {
        if (trace_me && c < p.trace_chunks) p.trace[(size_t)c * KDA_TRACE_POINTS + i] = (unsigned long long)clock64();
    };
#pragma unroll 1
    for (int c = 0; ok && c < u.nchunks; ++c) {
        const int s = kCtr ? sc : (c & 1);
        if (kCl && pt == 0) stamp(c, 0);
        const uint32_t cpar = c & 1, kpar = kCtr ? (kq & 1) : ((c >> 1) & 1);
        const uint32_t soff = kCtr ? slot_off(s) : s * SLOT_BYTES;
        const uint32_t slot = u.base + soff;
        const uint32_t tO = TM_O + (kEpi ? TM_OP_STRIDE * (uint32_t)(c & 1) : 0u), tP = tO + 32;
        const bool refill = c + NS < u.nchunks;
        uint32_t beta_next = BETA_NONE;
        if constexpr (!kCl) {
            if (pt == T_TMA && refill) prefetch_chunk(maps, u, c + NS);
            // chunk c + 2's beta goes into the slot once the inverse warp is done with this one's
            beta_next = beta_ahead;
            if (w == W_BETA && c + NS + 1 < u.nchunks) beta_ahead = load_beta_bits(p, u, c + NS + 1, lane);
        }

        // -R = P - V^T -> bf16 -> TMEM: A operand of GEMM2, which also waits for -B2
        // (the wait spans GEMM1, and the prep of the chunk when that runs late)
        if (!warp_wait(bar_addr(u, B_G1), cpar, p.status, 64)) { chain_wind_down<kEpi>(c, 1, u.nchunks); break; }
        tc_fence_after();
        if (kCl && pt == 0) stamp(c, 4);
        p_cols_to_bf16(lane_addr, tP);
        if (kCl && pt == 0) stamp(c, 5);
        if constexpr (!kCl) {
            if (!warp_wait(bar_addr(u, B_FULLD + s), kpar, p.status, 64)) { chain_wind_down<kEpi>(c, 1, u.nchunks); break; }
            if (refill && w == W_BETA) put_beta(u, s, lane, beta_of<kBetaLogit>(beta_next));
        }
        tc_fence_before();
        named_bar_arrive(NB_G2, NB_HAND);
        if (kCl && pt == 0) stamp(c, 6);

        // U -> bf16 -> TMEM: A operand of GEMM3
        if (!warp_wait(bar_addr(u, B_G2), cpar, p.status)) { chain_wind_down<kEpi>(c, 2, u.nchunks); break; }
        tc_fence_after();
        p_cols_to_bf16(lane_addr, tP);
        tc_fence_before();
        named_bar_arrive(NB_G3, NB_HAND);
        if (!warp_wait(bar_addr(u, B_G3), cpar, p.status)) { chain_wind_down<kEpi>(c, 3, u.nchunks); break; }
        tc_fence_after();

        if constexpr (kEpi) {
            // this chunk's O is final (and a cluster home's pushed operands have been read for
            // the last time): the epilogue warps take it from here
            if (pt == 0) {
                tc_fence_before();
                mbar_arrive(bar_addr(u, B_OREADY + (c & 1)));
            }
        }
        if constexpr (!kCl) {
            // The slot's q, k, g regions have been read for the last time: refill them with
            // chunk c + 2 (its boxes were prefetched into L2 at the top of the iteration)
            if (refill) {
                if (pt == T_TMA) load_qkg(maps, u, c + NS, s);
                issued = c + NS + 1;
            }
        }
        // O of this chunk -> staging tile [token][v] in the slot's v region (GEMM1 has read
        // v) -> tensor stores (row copies for a tail chunk); once the stores have read the
        // tile, the region takes chunk c + 2's v.  A full chunk's tile has the v boxes'
        // layout (two [32][64] blocks, 128-byte swizzle): the 16x256b TMEM load gives each
        // thread two adjacent tokens of one state row, and stmatrix.trans writes 8 tokens x
        // 8 rows per matrix as 16-byte rows, conflict-free under the swizzle.
        if constexpr (!kEpi) {   // (epilogue warps, where the CTA has them, do this part for it)
        const bool full = chunk_valid(u, c) == CH;
        if (full) {
            const uint32_t tile = slot + SL_V;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {   // lanes 32 w + 16 hf .. + 15
                const int base = 32 * w + 16 * hf;
                uint32_t o[16];
                tmem_ld_16x256b_x4(u.tmem + ((uint32_t)base << 16) + TM_O, o);
                tmem_wait_ld();
                // matrix j of a store: (row block lb, token block tb) = (j & 1, 2 st + (j >> 1));
                // its register: rows base + 8 lb + t / 4, tokens 8 tb + 2 (t % 4) + {0, 1}
                const int j = lane >> 3, k = lane & 7;
                const int v0 = base + 8 * (j & 1);
#pragma unroll
                for (int st = 0; st < 2; ++st) {
                    const int tok = 8 * (2 * st + (j >> 1)) + k;
                    const uint32_t r0 = pack_bf16x2(u2f(o[8 * st + 0]), u2f(o[8 * st + 1]));
                    const uint32_t r1 = pack_bf16x2(u2f(o[8 * st + 2]), u2f(o[8 * st + 3]));
                    const uint32_t r2 = pack_bf16x2(u2f(o[8 * st + 4]), u2f(o[8 * st + 5]));
                    const uint32_t r3 = pack_bf16x2(u2f(o[8 * st + 6]), u2f(o[8 * st + 7]));
                    stmatrix_x4_trans_s(tile + sw128_at(tok, v0, 32), r0, r1, r2, r3);
                }
            }
        } else {
            unsigned char* ost = u.gbase + soff + SL_V + 2 * v;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                uint32_t o[16];
                tmem_ld16(lane_addr + TM_O + hh * 16, o);
                tmem_wait_ld();
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    const uint32_t pr = pack_bf16x2(u2f(o[2 * m]), u2f(o[2 * m + 1]));
                    const int i = hh * 16 + 2 * m;
                    *reinterpret_cast<uint16_t*>(ost + i * 256) = (uint16_t)(pr & 0xffffu);
                    *reinterpret_cast<uint16_t*>(ost + (i + 1) * 256) = (uint16_t)(pr >> 16);
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        named_bar_sync(2, 128);
        if (pt == T_STORE) {
            const int64_t t0 = u.bos + (int64_t)c * CH;
            const int nvalid = chunk_valid(u, c);
            const uint32_t ost = slot + SL_V;
            if (nvalid == CH) {
                const int tc = (int)KDA_CHK(t0, u.bos, u.eos - CH + 1);   // a full chunk inside its sequence
                tma_store_3d(&maps.out, ost, 0, u.h, tc);
                tma_store_3d(&maps.out, ost + 4096, 64, u.h, tc);
            } else {
                for (int i = 0; i < nvalid; ++i)
                    bulk_store(p.out + (KDA_CHK(t0 + i, u.bos, u.eos) * p.H + u.h) * HD, ost + i * 256, 256);
            }
            bulk_commit();
        }
        }

        const int s1 = kCtr ? (s + 1 == NS ? 0 : s + 1) : (s ^ 1);
        if (c + 1 < u.nchunks) {
            // the bf16 copy of S for the next GEMM1 and the decay by the next chunk's a
            if constexpr (kCl) {
                if (!warp_wait(bar_addr(u, B_FULLOP + s1), (s1 == 0 ? kq + 1 : kq) & 1, p.status, 256)) { chain_wind_down<kEpi>(c + 1, 0, u.nchunks); break; }
            } else {
                const uint32_t apar = kCtr ? ((s1 == 0 ? kq + 1 : kq) & 1) : (((c + 1) >> 1) & 1);
                if (!warp_wait(bar_addr(u, B_AREADY + s1), apar, p.status, 256)) { chain_wind_down<kEpi>(c + 1, 0, u.nchunks); break; }
            }
            state_pass(reinterpret_cast<const float*>(u.gbase + (kCtr ? slot_off(s1) : s1 * SLOT_BYTES) + SL_A));
            // the output store has had the state pass to read the staging tile: the region
            // takes chunk c + 2's v
            if (!kEpi && pt == T_STORE && refill) {
                bulk_wait_read_all();
                load_v(maps, u, c + NS, s);
                vissued = c + NS + 1;
            }
        } else {
#pragma unroll 1
            for (int piece = 0; piece < 8; ++piece) {
                uint32_t r[16];
                tmem_ld16(lane_addr + TM_S + piece * 16, r);
                tmem_wait_ld();
                store_state16(p, srow + piece * 16, r);
            }
        }
        if constexpr (kCtr) {
            sc = s1;
            if (s1 == 0) ++kq;
        }
    }
    if (pt == T_STORE) bulk_wait_all();   // the output must be in global memory before the kernel ends
    (void)vissued;
    if (!kCl && pt == T_TMA) {
        // boxes still in flight must land before the CTA exits (only after a timeout can
        // one be unconsumed)
        for (int c = issued - NS < 0 ? 0 : issued - NS; c < issued; ++c)
            mbar_wait_bounded(bar_addr(u, B_FULLTMA + c % NS), (c / NS) & 1, p.status, KDA_DEVERR_TIMEOUT, WAIT_LIMIT);
    }
    if (!kEpi && pt == T_STORE) {
        // likewise the v boxes: the last NS requested (phases before them have completed)
        for (int c = vissued - NS < 0 ? 0 : vissued - NS; c < vissued; ++c)
            mbar_wait_bounded(bar_addr(u, B_FULLV + c % NS), (c / NS) & 1, p.status, KDA_DEVERR_TIMEOUT, WAIT_LIMIT);
    }
}

// ------------------------------------------------------------------------------
// MMA warp: issues every tensor-core MMA of the chain (kWarpIssue: the whole warp through
// elect.sync; else lane 0 alone), each once the chain has handed its A operand over, and
// commits each GEMM to its mbarrier (G1, G2, G3).  GEMM1's k blocks 0-3 go out while the chain
// still converts and decays the second half of S.
// ------------------------------------------------------------------------------
template <bool kWarpIssue, bool kCl, bool kSmemState, bool kEpi = kCl, bool kR3 = false>
__device__ void mma_warp(const FwdParams& p, const Unit& u, int lane) {
    constexpr int NS = kCl ? NSH : (kR3 ? NSL1 : NSLOT);
    constexpr bool kCtr = kCl || kR3;
    constexpr uint32_t idesc1 = make_idesc_bf16_f32(128, 64);
    constexpr uint32_t idescv = make_idesc_bf16_f32(128, 32, false, true);   // A = V^T, MN-major
    constexpr uint32_t idesc2 = make_idesc_bf16_f32(128, 32);                // GEMM2, and O += U Mqk^T
    constexpr uint32_t idesc3 = make_idesc_bf16_f32(128, 128, true);         // S += U K_r, B MN-major
    auto mma_ts = [&](uint32_t d, uint32_t a, uint64_t b, uint32_t id, uint32_t acc) {
        if constexpr (kWarpIssue) tc_mma_ts_warp(d, a, b, id, acc);
        else if (lane == 0) tc_mma_ts(d, a, b, id, acc);
    };
    auto mma_ss = [&](uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
        if constexpr (kWarpIssue) tc_mma_ss_warp(d, a, b, id, acc);
        else if (lane == 0) tc_mma_ss(d, a, b, id, acc);
    };
    auto commit = [&](uint32_t bar) {
        if constexpr (kWarpIssue) tc_commit_warp(bar);
        else if (lane == 0) tc_commit(bar);
    };
    int committed = 0;   // chunks whose GEMM3 was committed
    int sc = 0, kq = 0;
    const bool trace_me = kCl && lane == 0 && p.trace != nullptr && (int64_t)u.n * p.H + u.h == p.trace_unit;
    auto stamp = [&](int c, int i) {
        if (trace_me && c < p.trace_chunks) p.trace[(size_t)c * KDA_TRACE_POINTS + i] = (unsigned long long)clock64();
    };
#pragma unroll 1
    for (int c = 0; c < u.nchunks; ++c) {
        const int s = kCtr ? sc : (c & 1);
        const uint32_t kpar = kCtr ? (kq & 1) : ((c >> 1) & 1);
        const uint32_t slot = u.base + (kCtr ? slot_off(s) : s * SLOT_BYTES);
        const uint32_t tO = TM_O + (kEpi ? TM_OP_STRIDE * (uint32_t)(c & 1) : 0u), tP = tO + 32;
        // the chunk's operands (the cluster home's chain waited for the pushed chunk before its
        // state pass) and its v box; (cluster home) the epilogue warps have read out chunk c - 2's
        // O from this buffer
        stamp(c, 1);
        bool ok = kCl || warp_wait(bar_addr(u, B_FULLP + s), kpar, p.status, 256);
        ok = ok && warp_wait(bar_addr(u, B_FULLV + s), kpar, p.status, 256);
        if (kEpi && c >= 2) ok = ok && warp_wait(bar_addr(u, B_OFREE + (c & 1)), (uint32_t)(((c >> 1) + 1) & 1), p.status, 256);
        if (!ok) {
            mma_wind_down(c, u.nchunks);
            break;
        }
        stamp(c, 2);
        auto b1 = [&](int kk) { return make_sdesc_kmajor_sw128(slot + SL_QDKD + (kk >> 2) * 8192 + (kk & 3) * 32); };
        auto gemm1 = [&](int kk) {
            if constexpr (kSmemState)
                mma_ss(u.tmem + tO, make_sdesc_kmajor_sw128(u.base + OFF_STATE + (kk >> 2) * STATE_BLOCK + (kk & 3) * 32),
                       b1(kk), idesc1, kk > 0);
            else
                mma_ts(u.tmem + tO, u.tmem + TM_SB + kk * 8, b1(kk), idesc1, kk > 0);
        };
        // GEMM1 [O_0 | P] = S_bf16 [Q_d | K_d]^T, in two halves of k, then P -= V^T
        named_bar_sync(NB_G1A, NB_HAND);
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) gemm1(kk);
        named_bar_sync(NB_G1B, NB_HAND);
        tc_fence_after();
#pragma unroll
        for (int kk = 4; kk < 8; ++kk) gemm1(kk);
#pragma unroll
        for (int kk = 0; kk < 2; ++kk)
            mma_ss(u.tmem + tP, make_sdesc_mnmajor_sw128(slot + SL_V + kk * 2048, 4096, 1024),
                   make_sdesc_kmajor_noswizzle(u.base + OFF_NEGI + kk * 256, 128, 512), idescv, 1u);   // P -= V^T
        commit(bar_addr(u, B_G1));
        stamp(c, 3);
        // GEMM2 U = (-R) (-B2), into the P columns
        named_bar_sync(NB_G2, NB_HAND);
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 2; ++kk)
            mma_ts(u.tmem + tP, u.tmem + TM_SB + kk * 8, make_sdesc_kmajor_noswizzle(slot + SL_INV + kk * 256, 128, 512), idesc2,
                   kk > 0);
        commit(bar_addr(u, B_G2));
        stamp(c, 7);
        // GEMM3: S += U K_r, O += U Mqk^T
        named_bar_sync(NB_G3, NB_HAND);
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
            mma_ts(u.tmem + TM_S, u.tmem + TM_SB + kk * 8, make_sdesc_mnmajor_sw128(slot + SL_KR + kk * 2048, 4096, 1024),
                   idesc3, 1u);
            mma_ts(u.tmem + tO, u.tmem + TM_SB + kk * 8, make_sdesc_kmajor_noswizzle(slot + SL_MQT + kk * 256, 128, 512),
                   idesc2, 1u);
        }
        commit(bar_addr(u, B_G3));
        committed = c + 1;
        if constexpr (kCtr) {
            sc = s + 1 == NS ? 0 : s + 1;
            if (sc == 0) ++kq;
        }
    }
    // the MMAs must be complete before the CTA frees its Tensor Memory (after a wind-down the
    // chain may not have waited for the last ones); MMAs complete in order
    if (committed > 0)
        mbar_wait_bounded(bar_addr(u, B_G3), (uint32_t)((committed - 1) & 1), p.status, KDA_DEVERR_TIMEOUT, WAIT_LIMIT);
}

// ------------------------------------------------------------------------------
// Prep group (256 threads): everything of a chunk that does not need the state.
// Elementwise phases: thread = (channel quad: channels 4 lane .. 4 lane + 3,
// token quad: tokens 4 pw .. 4 pw + 3), pw = warp index within the group.
// ------------------------------------------------------------------------------
// The group prepares the chunks c = c_first + kStride j, j < nloc, in its slots j % 2 (all
// of them, or one helper's share in the cluster schedule).
template <bool kSoftplus, int kStride, int kRing = NSLOT>
__device__ void prep_group(const FwdParams& p, const Unit& u, int pt, int c_first, int nloc) {
    const int lane = pt & 31, pw = pt >> 5, gq = lane >> 2, tq = lane & 3;
    const int c0 = 4 * lane;
    // phase B store offsets of token 4 pw (channels c0 .. c0 + 3); token 4 pw + r differs by one XOR:
    // its row adds r to bits 8-9 (scratch tiles, 256-byte rows) or 7-8 (swizzled slot, 128-byte rows),
    // and its 16-byte chunk index is XORed with r
    const uint32_t oB_sc = sc_at(4 * pw, c0);
    const uint32_t oB_sw = sw128_at(4 * pw, c0, 64);
    const uint32_t oB_kr = sw128_at(4 * pw, c0, 32);
    const float eA = expf(p.A_log[u.h]);
    const float gm = -eA * LOG2E;                       // sigmoid(x) = 1 / (1 + 2^(gm (g + dt)))
    const float4 dt = *reinterpret_cast<const float4*>(p.dt_bias + u.h * HD + c0);
    const float2 gmv = make_float2(gm, gm);
    const float2 gb01 = make_float2(gm * dt.x, gm * dt.y), gb23 = make_float2(gm * dt.z, gm * dt.w);
    const float bcoef = p.lower_bound * LOG2E;          // b
    // fixed anchor C = rint(16 b): an integer, so 2^C is exact in bf16 and Q_d = Q_c 2^C,
    // K_d = K_c 2^C are exact rescalings of the bf16 Q_c, K_c (one packed bf16 multiply);
    // |G - C| and |C - G| stay <= 126 for every lower_bound >= -5.4585 (G lies in [32 b, 0])
    const float Cst = rintf(16.f * bcoef);
    const float twoC = ex2_approx(Cst);
    const float2 bcv = make_float2(bcoef, bcoef);

    unsigned char* qcs = u.gbase + OFF_QC;
    unsigned char* kcs = u.gbase + OFF_KC;
    unsigned char* kis = u.gbase + OFF_KI;
    float* Lb = reinterpret_cast<float*>(u.gbase + OFF_L);
    float* tot = reinterpret_cast<float*>(u.gbase + OFF_MISC);            // [8][128]
    float* totg = tot + PREP_WARPS * HD + 64;                              // [128]
    // partial rows 4-7 hold their channels rotated by 16, so that the scan's two half-warps
    // (rows 0-3 and 4-7 of the same channels) use disjoint banks
    auto trot = [](int qq, int ch) { return (ch + ((qq >> 2) << 4)) & (HD - 1); };
    float* rq = tot + PREP_WARPS * HD;
    float* rk = rq + 32;

#pragma unroll 1
    for (int j = 0; j < nloc; ++j) {
        const int c = c_first + kStride * j;
        const int s = j % kRing;
        const uint32_t kpar = (j / kRing) & 1;
        unsigned char* gslot = u.gbase + slot_off(s);
        if (!warp_wait(bar_addr(u, B_FULLTMA + s), kpar, p.status, 128)) { prep_wind_down(j, 0, nloc); return; }
        const int64_t t0 = u.bos + (int64_t)c * CH;
        const int nvalid = (int)((u.eos - t0) < CH ? (u.eos - t0) : CH);
        const float* bs = reinterpret_cast<const float*>(gslot + SL_BETA);

        // ---- A: q/k row norms (row pass: 4 threads per row), gate and local prefix over
        //      4 tokens x 4 channels; the two are independent and written so that they overlap
        uint2 qv[4], kv[4];
        float2 G01[4], G23[4];
        {
            const int row = pt >> 2, part = pt & 3;   // rows 0-31 q, 32-63 k; 32 elements per thread
            const unsigned char* rp = gslot + (row < 32 ? SL_RAWQ + row * 256 : SL_RAWK + (row - 32) * 256);
            uint4 w4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
                w4[e] = *reinterpret_cast<const uint4*>(rp + ((4 * e + part + 4 * (row & 1)) & 15) * 16);
            uint2 gw[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const uint32_t off = (4 * pw + r) * 256 + c0 * 2;
                qv[r] = *reinterpret_cast<const uint2*>(gslot + SL_RAWQ + off);
                kv[r] = *reinterpret_cast<const uint2*>(gslot + SL_RAWK + off);
                gw[r] = *reinterpret_cast<const uint2*>(gslot + SL_RAWG + off);
            }

            float2 acc01 = make_float2(0.f, 0.f), acc23 = make_float2(0.f, 0.f);
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int i = 4 * pw + r;
                if constexpr (kSoftplus) {
                    // lambda2 = max(-e^A softplus(z) log2 e, b), z = g + dt_bias, with
                    // softplus(z) log2 e = max(z, 0) log2 e + log2(1 + 2^(-|z| log2 e)); tokens past
                    // the end: lambda = 0
                    const float2 z01 = __fadd2_rn(bf2_to_f2(gw[r].x), make_float2(dt.x, dt.y));
                    const float2 z23 = __fadd2_rn(bf2_to_f2(gw[r].y), make_float2(dt.z, dt.w));
                    const float zs[4] = {z01.x, z01.y, z23.x, z23.y};
                    float lam[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float sp2 = fmaf(fmaxf(zs[e], 0.f), LOG2E, lg2_approx(1.f + ex2_approx(-fabsf(zs[e]) * LOG2E)));
                        lam[e] = i < nvalid ? fmaxf(-eA * sp2, bcoef) : 0.f;
                    }
                    acc01 = __fadd2_rn(acc01, make_float2(lam[0], lam[1]));
                    acc23 = __fadd2_rn(acc23, make_float2(lam[2], lam[3]));
                } else {
                    const float2 x01 = __ffma2_rn(gmv, bf2_to_f2(gw[r].x), gb01);
                    const float2 x23 = __ffma2_rn(gmv, bf2_to_f2(gw[r].y), gb23);
                    const float bl = i < nvalid ? bcoef : 0.f;   // tokens past the end: lambda = 0
                    const float2 blv = make_float2(bl, bl);
                    acc01 = __ffma2_rn(blv, make_float2(rcp_approx(1.f + ex2_approx(x01.x)), rcp_approx(1.f + ex2_approx(x01.y))),
                                       acc01);
                    acc23 = __ffma2_rn(blv, make_float2(rcp_approx(1.f + ex2_approx(x23.x)), rcp_approx(1.f + ex2_approx(x23.y))),
                                       acc23);
                }
                G01[r] = acc01;
                G23[r] = acc23;
            }
            *reinterpret_cast<float4*>(tot + pw * HD + trot(pw, c0)) = make_float4(acc01.x, acc01.y, acc23.x, acc23.y);

            float2 ss0 = make_float2(0.f, 0.f), ss1 = make_float2(0.f, 0.f);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 x0 = bf2_to_f2(w4[e].x), x1 = bf2_to_f2(w4[e].y), x2 = bf2_to_f2(w4[e].z), x3 = bf2_to_f2(w4[e].w);
                ss0 = __ffma2_rn(x0, x0, ss0);
                ss1 = __ffma2_rn(x1, x1, ss1);
                ss0 = __ffma2_rn(x2, x2, ss0);
                ss1 = __ffma2_rn(x3, x3, ss1);
            }
            const float2 ss = __fadd2_rn(ss0, ss1);
            float sum = ss.x + ss.y;
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            sum += __shfl_xor_sync(0xffffffffu, sum, 2);
            const int tok = row & 31;
            const float rn = tok < nvalid ? rsqrtf(sum + NORM_EPS) : 0.f;
            if (part == 0) {
                if (row < 32) rq[tok] = rn; else rk[tok] = rn;
            }
        }
        named_bar_sync(1, PREP_THREADS);   // raw q/k/g are no longer read after this point

        // ---- prefix across the warps: thread (pw, lane) scans the 4 partials of warps 4 h .. 4 h + 3
        //      (h = lane / 16) of channel 16 pw + lane % 16, in place: tot[qq] becomes the exclusive
        //      prefix of warp qq, and totg the chunk total
        {
            const int ch = 16 * pw + (lane & 15), h = lane >> 4;
            float* col = tot + 4 * h * HD + trot(4 * h, ch);
            const float x0 = col[0], x1 = col[HD], x2 = col[2 * HD], x3 = col[3 * HD];
            const float s2 = x0 + x1, s3 = s2 + x2, s4 = s3 + x3;
            const float other = __shfl_xor_sync(0xffffffffu, s4, 16);
            const float base = h ? other : 0.f;
            col[0] = base;
            col[HD] = base + x0;
            col[2 * HD] = base + s2;
            col[3 * HD] = base + s3;
            if (h == 0) totg[ch] = s4 + other;
        }
        named_bar_sync(1, PREP_THREADS);
        // ---- B: centered operands
        {
            float2 T01, T23;
            {
                const float4 o4 = *reinterpret_cast<const float4*>(tot + pw * HD + trot(pw, c0));
                const float4 t4 = *reinterpret_cast<const float4*>(totg + c0);
                float2 off01 = make_float2(o4.x, o4.y), off23 = make_float2(o4.z, o4.w);
                T01 = make_float2(t4.x, t4.y);
                T23 = make_float2(t4.z, t4.w);
                const float2 mC = make_float2(-Cst, -Cst);
                off01 = __fadd2_rn(off01, mC);
                off23 = __fadd2_rn(off23, mC);
#pragma unroll
                for (int r = 0; r < 4; ++r) {   // G - C
                    G01[r] = __fadd2_rn(G01[r], off01);
                    G23[r] = __fadd2_rn(G23[r], off23);
                }
            }
            const __nv_bfloat162 twoC2 = __float2bfloat162_rn(twoC);   // exact: C is an integer
            // rho = 2^(G_T - C) of this thread's channels: K_r = K_i diag(rho) = k 2^(G_T - G)
            const float2 rho01 = make_float2(ex2_approx(T01.x - Cst), ex2_approx(T01.y - Cst));
            const float2 rho23 = make_float2(ex2_approx(T23.x - Cst), ex2_approx(T23.y - Cst));
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int i = 4 * pw + r;
                const uint32_t o = oB_sc ^ (uint32_t)((r << 4) | (r << 8));        // sc128(i, c0)
                const uint32_t od = oB_sw ^ (uint32_t)((r << 4) | (r << 7));       // sw128_offset(i, c0, 64)
                const float qs = rq[i] * p.scale, ks = rk[i];
                const float2 k01 = __fmul2_rn(bf2_to_f2(kv[r].x), make_float2(ks, ks));
                const float2 k23 = __fmul2_rn(bf2_to_f2(kv[r].y), make_float2(ks, ks));
                {   // 2^(G - C): Q_c, K_c and the recurrent-domain Q_d, K_d
                    const float2 ep01 = make_float2(ex2_approx(G01[r].x), ex2_approx(G01[r].y));
                    const float2 ep23 = make_float2(ex2_approx(G23[r].x), ex2_approx(G23[r].y));
                    const float2 qc01 = __fmul2_rn(__fmul2_rn(bf2_to_f2(qv[r].x), make_float2(qs, qs)), ep01);
                    const float2 qc23 = __fmul2_rn(__fmul2_rn(bf2_to_f2(qv[r].y), make_float2(qs, qs)), ep23);
                    uint2 w = make_uint2(f2_to_bf2(qc01), f2_to_bf2(qc23));
                    *reinterpret_cast<uint2*>(qcs + o) = w;
                    __nv_bfloat162* hw = reinterpret_cast<__nv_bfloat162*>(&w);
                    hw[0] = __hmul2(hw[0], twoC2);
                    hw[1] = __hmul2(hw[1], twoC2);
                    *reinterpret_cast<uint2*>(gslot + SL_QDKD + od) = w;   // Q_d
                    const float2 kc01 = __fmul2_rn(k01, ep01), kc23 = __fmul2_rn(k23, ep23);
                    w = make_uint2(f2_to_bf2(kc01), f2_to_bf2(kc23));
                    *reinterpret_cast<uint2*>(kcs + o) = w;
                    hw[0] = __hmul2(hw[0], twoC2);
                    hw[1] = __hmul2(hw[1], twoC2);
                    *reinterpret_cast<uint2*>(gslot + SL_QDKD + (od + 32 * 128)) = w;   // K_d
                }
                {   // 2^(C - G): K_i and K_r = K_i 2^(G_T - C)
                    const float2 em01 = make_float2(ex2_approx(-G01[r].x), ex2_approx(-G01[r].y));
                    const float2 em23 = make_float2(ex2_approx(-G23[r].x), ex2_approx(-G23[r].y));
                    const float2 ki01 = __fmul2_rn(k01, em01), ki23 = __fmul2_rn(k23, em23);
                    *reinterpret_cast<uint2*>(kis + o) = make_uint2(f2_to_bf2(ki01), f2_to_bf2(ki23));
                    *reinterpret_cast<uint2*>(gslot + SL_KR + (oB_kr ^ (uint32_t)((r << 4) | (r << 7)))) =
                        make_uint2(f2_to_bf2(__fmul2_rn(ki01, rho01)), f2_to_bf2(__fmul2_rn(ki23, rho23)));   // K_r
                }
            }
            if (pw == 4)   // a = 2^G_T: the chain's decay of S
                *reinterpret_cast<float4*>(gslot + SL_A + c0 * 4) =
                    make_float4(ex2_approx(T01.x), ex2_approx(T01.y), ex2_approx(T23.x), ex2_approx(T23.y));
        }
        // (the slot operands written here are read by the tensor core only after FULLP, and
        // the proxy fence before the end-of-chunk barrier orders them)
        named_bar_sync(1, PREP_THREADS);
        if (pt == 0) mbar_arrive(bar_addr(u, B_AREADY + s));   // the chain may decay S by a

        // ---- C: K_c K_i^T and Q_c K_i^T, the three nonzero 16 x 16 blocks (mt, nb) = (1,0), (1,1),
        //      (0,0) of each, on warps 1-3; a warp computes the same block of both products, so
        //      the K_i fragments it loads serve both.  Warp 0 writes the zero upper-right block of
        //      Mqk (L keeps no such block); warps 4-7 have no part in this phase.
        if (pw == 0) {   // rows 0-15, columns 16-31: 4 core matrices of 8 rows x 16 bytes, one row a lane
            const int cm = lane >> 3;
            *reinterpret_cast<uint4*>(gslot + SL_MQT + core_at(8 * (cm >> 1) + (lane & 7), 16 + 8 * (cm & 1), 32)) =
                make_uint4(0u, 0u, 0u, 0u);
        } else if (pw < 4) {
            const int mt = pw == 3 ? 0 : 1, nb = pw == 2 ? 1 : 0;
            float acck[2][4], accq[2][4];
#pragma unroll
            for (int t = 0; t < 2; ++t)
#pragma unroll
                for (int e = 0; e < 4; ++e) acck[t][e] = accq[t][e] = 0.f;
            // 16-byte chunk 2 kk + h of row r sits at chunk (2 kk + h) ^ (r % 8) = (h ^ (r % 8)) ^ 2 kk:
            // k step kk is one XOR of the k-step-0 address with kk << 5 (the tiles are 256-byte aligned)
            const uint32_t aoff = sc_at(mt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8, (lane >> 4) * 8);
            const uint32_t ak0 = smem_u32(kcs + aoff), aq0 = smem_u32(qcs + aoff);
            const uint32_t b0 = smem_u32(kis + sc_at(nb * 16 + (lane & 7) + (lane >> 4) * 8, ((lane >> 3) & 1) * 8));
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                uint32_t ak[4], aq[4], b[4];
                ldmatrix_x4_s(b, b0 ^ (kk << 5));
                ldmatrix_x4_s(ak, ak0 ^ (kk << 5));
                ldmatrix_x4_s(aq, aq0 ^ (kk << 5));
                mma_bf16_16816(acck[0], ak, b[0], b[1]);
                mma_bf16_16816(acck[1], ak, b[2], b[3]);
                mma_bf16_16816(accq[0], aq, b[0], b[1]);
                mma_bf16_16816(accq[1], aq, b[2], b[3]);
            }
            // L is rewritten only once the inverse warp has read the previous chunk's
            if (j > 0 && !warp_wait(bar_addr(u, B_LFREE), (j - 1) & 1, p.status)) { prep_wind_down(j, 3, nloc); return; }
#pragma unroll
            for (int t = 0; t < 2; ++t) {
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const int i = mt * 16 + gq + hf * 8;
                    const int jj = nb * 16 + t * 8 + 2 * tq;
                    // select, never multiply: the masked upper triangle may hold inf/NaN
                    Lb[l_at(i, jj)] = (jj < i) ? bs[i] * acck[t][2 * hf] : 0.f;
                    Lb[l_at(i, jj + 1)] = (jj + 1 < i) ? bs[i] * acck[t][2 * hf + 1] : 0.f;
                    *reinterpret_cast<uint32_t*>(gslot + SL_MQT + core_at(i, jj, 32)) =
                        pack_bf16x2((jj <= i) ? accq[t][2 * hf] : 0.f, (jj + 1 <= i) ? accq[t][2 * hf + 1] : 0.f);   // Mqk
                }
            }
        }
        fence_proxy_async_smem();   // Q_d, K_d, K_r, Mqk are read by the tensor core
        named_bar_sync(1, PREP_THREADS);
        if (pt == 0) mbar_arrive(bar_addr(u, B_FULLP + s));
    }
}

// ------------------------------------------------------------------------------
// Inverse warp: INV = X = (I + L)^-1 of chunk c, in fp32, while the prep warps take chunk
// c + 1.  The two diagonal 16 x 16 blocks by forward substitution (lane = column; lanes
// 0-15 block 1, lanes 16-31 block 2), then X21 = -X22 L21 X11, computed transposed with tf32
// mma.sync (fp32 operands passed as they are: the tensor core uses their top 19 bits):
// T2^T = X11^T L21^T, then X21^T = -T2^T X22^T, whose A operand is the first product's
// accumulator with its k index permuted (k slot t <-> column 2t, slot t + 4 <-> column
// 2t + 1, and the B operand rows permuted alike).
// -B2[i][j] = -beta_j X[i][j] goes to the slot in the K-major core layout (the B operand
// of GEMM2); its upper-right block is zero and written once.
// ------------------------------------------------------------------------------
__device__ __forceinline__ uint16_t bf16_bits(float x) { return (uint16_t)(pack_bf16x2(x, 0.f) & 0xffffu); }

template <int kRing = NSLOT>
__device__ void inverse_warp(const FwdParams& p, const Unit& u, int lane, int nloc) {   // nloc: as the prep group's
    const int gq = lane >> 2, tq = lane & 3;
    const int b = lane >> 4, cc = lane & 15;   // substitution: block b, column cc
    const float* Lb = reinterpret_cast<const float*>(u.gbase + OFF_L);
    float* Xb = reinterpret_cast<float*>(u.gbase + OFF_X);
#pragma unroll
    for (int s = 0; s < kRing; ++s)   // -B2[i][j] = 0 for i < 16 <= j (nothing else writes there)
        *reinterpret_cast<uint4*>(u.gbase + slot_off(s) + SL_INV + core_at(lane >> 1, 16 + 8 * (lane & 1), 32)) =
            make_uint4(0, 0, 0, 0);

#pragma unroll 1
    for (int j = 0; j < nloc; ++j) {
        const int s = j % kRing;
        const uint32_t kpar = (j / kRing) & 1;
        unsigned char* b2s = u.gbase + slot_off(s) + SL_INV;
        const float* bs = reinterpret_cast<const float*>(u.gbase + slot_off(s) + SL_BETA);
        if (!warp_wait(bar_addr(u, B_FULLP + s), kpar, p.status, 128)) return;

        // ---- diagonal blocks: x[r] = X_bb[r][cc]
        {
            const float* Ld = Lb + (b ? LB_22 : LB_11);
            float x[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) x[r] = (r == cc) ? 1.f : 0.f;
#pragma unroll
            for (int k = 0; k < 15; ++k) {
                const float2 mxk = make_float2(-x[k], -x[k]);
                const float* col = Ld + k * LB;
#pragma unroll
                for (int r4 = (k + 1) >> 2; r4 < 4; ++r4) {
                    const float4 l4 = *reinterpret_cast<const float4*>(col + 4 * r4);
#pragma unroll
                    for (int pr = 0; pr < 2; ++pr) {   // rows 4 r4 + 2 pr and 4 r4 + 2 pr + 1 below row k
                        const int r = 4 * r4 + 2 * pr;
                        const float la = pr ? l4.z : l4.x, lb = pr ? l4.w : l4.y;
                        if (r > k) {
                            const float2 y = __ffma2_rn(make_float2(la, lb), mxk, make_float2(x[r], x[r + 1]));
                            x[r] = y.x;
                            x[r + 1] = y.y;
                        } else if (r + 1 > k) {
                            x[r + 1] = fmaf(lb, mxk.x, x[r + 1]);
                        }
                    }
                }
            }
            // X_bb to shared memory, for the block product and the -B2 rows below
            float* xc = Xb + (b ? XB_22 : 0) + cc;
#pragma unroll
            for (int r = 0; r < 16; ++r) xc[r * XB] = x[r];
        }
        __syncwarp();

        // ---- T2^T = X11^T L21^T: t[nt][e] = T2^T[gq + 8 (e >> 1)][8 nt + 2 tq + (e & 1)]
        float t[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) t[nt][0] = t[nt][1] = t[nt][2] = t[nt][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
            const int k0 = ks * 8 + tq;
            const uint32_t a[4] = {__float_as_uint(Xb[k0 * XB + gq]), __float_as_uint(Xb[k0 * XB + gq + 8]),
                                   __float_as_uint(Xb[(k0 + 4) * XB + gq]), __float_as_uint(Xb[(k0 + 4) * XB + gq + 8])};
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {   // B[k][n] = L21[8 nt + n][k]
                const float* l21 = Lb + LB_21 + nt * 8 + gq;
                mma_tf32_1688(t[nt], a, __float_as_uint(l21[k0 * LB]), __float_as_uint(l21[(k0 + 4) * LB]));
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_addr(u, B_LFREE));   // L has been read: the prep warps may rewrite it

        // -B2 rows of the diagonal blocks: lane n reads row n of its block of X and writes the
        // row's 16 values as two 16-byte stores (a lane per row keeps the core-matrix layout's
        // stores free of bank conflicts; a lane per column would put every lane on four banks)
        {
            const int n = lane, o = n & 16;
            const float* xr = Xb + (o ? XB_22 : 0) + (n & 15) * XB;
            uint32_t wv[8];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                const float4 xv = *reinterpret_cast<const float4*>(xr + 4 * q4);
                const float4 bv = *reinterpret_cast<const float4*>(bs + o + 4 * q4);
                wv[2 * q4] = pack_bf16x2(-bv.x * xv.x, -bv.y * xv.y);
                wv[2 * q4 + 1] = pack_bf16x2(-bv.z * xv.z, -bv.w * xv.w);
            }
            *reinterpret_cast<uint4*>(b2s + core_at(n, o, 32)) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
            *reinterpret_cast<uint4*>(b2s + core_at(n, o + 8, 32)) = make_uint4(wv[4], wv[5], wv[6], wv[7]);
        }

        // ---- y = T2^T X22^T = (X22 T2)^T = -X21^T: y[nt][e] = y[gq + 8 (e >> 1)][8 nt + 2 tq + (e & 1)]
        float y[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) y[nt][0] = y[nt][1] = y[nt][2] = y[nt][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
            const uint32_t a[4] = {__float_as_uint(t[ks][0]), __float_as_uint(t[ks][2]), __float_as_uint(t[ks][1]),
                                   __float_as_uint(t[ks][3])};
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {   // B[slot][n]: X22[8 nt + n][8 ks + 2 tq] and [.. + 1]
                const float2 x2 = *reinterpret_cast<const float2*>(Xb + XB_22 + (nt * 8 + gq) * XB + ks * 8 + 2 * tq);
                mma_tf32_1688(y[nt], a, __float_as_uint(x2.x), __float_as_uint(x2.y));
            }
        }
        // -B2[16 + rr][cc] = -beta_cc X21[rr][cc] = beta_cc y[cc][rr]
        const float bl = bs[gq], bh = bs[gq + 8];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int ci = gq + 8 * (e >> 1), rr = 8 * nt + 2 * tq + (e & 1);
                *reinterpret_cast<uint16_t*>(b2s + core_at(16 + rr, ci, 32)) = bf16_bits((e >> 1 ? bh : bl) * y[nt][e]);
            }
        fence_proxy_async_smem();   // -B2 is read by the tensor core
        __syncwarp();
#ifdef KDA_WAIT_TEST
        if (j == p.test_skip_chunk) continue;   // the arrival a chain warp then waits for in vain
#endif
        if (lane == 0) mbar_arrive(bar_addr(u, B_FULLD + s));
    }
}

// ------------------------------------------------------------------------------
// Cluster schedules.  Chunk c is prepared by helper h = c % kNH as its chunk j = c / kNH, in
// its slot j % ring (ring = 2 slots with three helpers, 4 with one), and pushed into home slot
// c % NSH.  Every barrier that one side completes for the other has one instance per slot
// (HSLOT: per home slot the helper pushes into), so no wait can see a phase two ahead of its
// own.
// ------------------------------------------------------------------------------

// Once every CTA of the cluster has published its push count: wait until every push issued
// has landed, so that no copy is in flight when a CTA of the cluster exits.  seen[h] chunks of
// home slot h were finished by the chain (their pushes landed); a push is only issued into an
// armed slot, and a slot is armed for its next chunk only once the chain has finished the
// one before, so at most one push a slot is left to wait for.
template <int kNH>
__device__ void home_drain(const FwdParams& p, const Unit& u, const int (&seen)[NSH]) {
#pragma unroll 1
    for (int hs = 0; hs < NSH; ++hs) {
        // pushes into home slot hs: those of helper hs (three helpers), or every third of the
        // one helper's, from its chunk hs on
        const int n = *reinterpret_cast<volatile int*>(u.gbase + OFF_PUSHED + 4 * (kNH == 1 ? 0 : hs));
        const int pushed = kNH == 1 ? (n > hs ? (n - hs + NSH - 1) / NSH : 0) : n;
        for (int j = seen[hs]; j < pushed; ++j)
            mbar_wait_bounded(bar_addr(u, B_FULLOP + hs), (uint32_t)(j & 1), p.status, KDA_DEVERR_TIMEOUT, WAIT_LIMIT);
    }
}

// Home CTA, warps 8-11 (TMEM lanes 32 (w % 4) ..): once the chain has finished chunk c
// (OREADY, its O in buffer c % 2), read the O out, stage it in the slot's v region (GEMM1 has
// read v) and store it (tensor stores, row copies for a tail chunk), release the buffer
// (OFREE), then refill the region with chunk c + 3's v once the stores have read it.  This
// takes the output off the chain's critical path.  The helpers hear from two single threads
// meanwhile: lane 0 of warp 9 arms home slot hs = c % NSH for chunk c + NSH (an arrival and
// the bytes to come) and tells that chunk's helper it may push it (HSLOT); lane 0 of warp 10
// tells chunk c's helper that the slot which held it may be refilled (COPIED).  seen[hs]
// (lane 0 of warp 9) counts the chunks of home slot hs the chain has finished.
template <int kNH>
__device__ void home_epilogue(const FwdParams& p, const TmaMaps& maps, const Unit& u, int et, int (&seen)[NSH]) {
    // kNH == 0: a CTA with its own prep (one per SM) and a ring of three slots, no helpers to signal
    constexpr int NS = kNH ? NSH : NSL1, RING = cl_ring(kNH);
    const int w = et >> 5, lane = et & 31, v = et;
    const uint32_t lane_addr = u.tmem + ((uint32_t)(w * 32) << 16);
    // chunks whose v boxes have been requested: the chain loads the first NS, this thread the rest
    int vissued = u.nchunks < NS ? u.nchunks : NS;
#pragma unroll 1
    for (int c = 0; c < u.nchunks; ++c) {
        const int b = c & 1, s = c % NS;
        const uint32_t soff = slot_off(s), slot = u.base + soff;
        const uint32_t tO = TM_O + TM_OP_STRIDE * (uint32_t)b;
        if (!warp_wait(bar_addr(u, B_OREADY + b), (uint32_t)((c >> 1) & 1), p.status, 256)) {
            epilogue_wind_down(c, u.nchunks);
            break;
        }
        tc_fence_after();
        if constexpr (kNH > 0) {
            const int hs = c % NS;
            if (et == 32) {   // home slot hs takes chunk c + NS next, from helper (c + NS) % kNH
                ++seen[hs];
                if (c + NS < u.nchunks) {
                    mbar_arrive_expect_tx(bar_addr(u, B_FULLOP + hs), PUSH_BYTES);
                    mbar_arrive_remote(mapa_shared(bar_addr(u, B_HSLOT + hs / kNH), (uint32_t)((c + NS) % kNH + 1)));
                }
            } else if (et == 64) {   // the helper slot that held chunk c
                mbar_arrive_remote(mapa_shared(bar_addr(u, B_COPIED + (c / kNH) % RING), (uint32_t)(c % kNH + 1)));
            }
        }
        const int nvalid = chunk_valid(u, c);
        if (nvalid == CH) {   // the tile in the v boxes' layout (see the chain's staging)
            const uint32_t tile = slot + SL_V;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int base = 32 * w + 16 * hf;
                uint32_t o[16];
                tmem_ld_16x256b_x4(u.tmem + ((uint32_t)base << 16) + tO, o);
                tmem_wait_ld();
                const int j = lane >> 3, k = lane & 7;
                const int v0 = base + 8 * (j & 1);
#pragma unroll
                for (int st = 0; st < 2; ++st) {
                    const int tok = 8 * (2 * st + (j >> 1)) + k;
                    const uint32_t r0 = pack_bf16x2(u2f(o[8 * st + 0]), u2f(o[8 * st + 1]));
                    const uint32_t r1 = pack_bf16x2(u2f(o[8 * st + 2]), u2f(o[8 * st + 3]));
                    const uint32_t r2 = pack_bf16x2(u2f(o[8 * st + 4]), u2f(o[8 * st + 5]));
                    const uint32_t r3 = pack_bf16x2(u2f(o[8 * st + 6]), u2f(o[8 * st + 7]));
                    stmatrix_x4_trans_s(tile + sw128_at(tok, v0, 32), r0, r1, r2, r3);
                }
            }
        } else {
            unsigned char* ost = u.gbase + soff + SL_V + 2 * v;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                uint32_t o[16];
                tmem_ld16(lane_addr + tO + hh * 16, o);
                tmem_wait_ld();
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    const uint32_t pr = pack_bf16x2(u2f(o[2 * m]), u2f(o[2 * m + 1]));
                    const int i = hh * 16 + 2 * m;
                    *reinterpret_cast<uint16_t*>(ost + i * 256) = (uint16_t)(pr & 0xffffu);
                    *reinterpret_cast<uint16_t*>(ost + (i + 1) * 256) = (uint16_t)(pr >> 16);
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        named_bar_sync(3, 128);
        if (et == 0) {
            mbar_arrive(bar_addr(u, B_OFREE + b));   // the buffer's columns have been read
            const int64_t t0 = u.bos + (int64_t)c * CH;
            const uint32_t ost = slot + SL_V;
            if (nvalid == CH) {
                const int tc = (int)KDA_CHK(t0, u.bos, u.eos - CH + 1);
                tma_store_3d(&maps.out, ost, 0, u.h, tc);
                tma_store_3d(&maps.out, ost + 4096, 64, u.h, tc);
            } else {
                for (int i = 0; i < nvalid; ++i)
                    bulk_store(p.out + (KDA_CHK(t0 + i, u.bos, u.eos) * p.H + u.h) * HD, ost + i * 256, 256);
            }
            bulk_commit();
            if (c + NS < u.nchunks) {
                bulk_wait_read_all();
                load_v(maps, u, c + NS, s);
                vissued = c + NS + 1;
            }
        }
    }
    if (et == 0) {
        bulk_wait_all();   // the output must be in global memory before the kernel ends
        // the last v boxes requested, by either thread, must have landed (only after a timeout
        // can one be unconsumed); earlier phases of the same barriers completed before these
        for (int c = vissued - NS < 0 ? 0 : vissued - NS; c < vissued; ++c)
            mbar_wait_bounded(bar_addr(u, B_FULLV + c % NS), (c / NS) & 1, p.status, KDA_DEVERR_TIMEOUT, WAIT_LIMIT);
    }
}

// Helper CTA, warps 0-3: warp 2 loads the q, k, g boxes (lane 0) and beta of the helper's
// chunks into its ring of kRing slots, the slot of local chunk j once chunk j - kRing, pushed
// from it, has been consumed; lane 0 of warp 3 pushes each chunk the prep and inverse warps
// have finished into home slot c % NSH, once that is free, and at the end publishes how many
// pushes it issued.
template <bool kBetaLogit, int kNH>
__device__ void helper_io(const FwdParams& p, const TmaMaps& maps, const Unit& u, int pt, int h, int nloc) {
    constexpr int kRing = cl_ring(kNH);
    const int w = pt >> 5, lane = pt & 31;
    if (w == W_BETA) {
        int loaded = 0;
#pragma unroll 1
        for (int j = 0; j < nloc; ++j) {
            const int c = h + kNH * j, b = j % kRing;
            if (j >= kRing && !__all_sync(0xffffffffu, mbar_wait_bounded<true>(bar_addr(u, B_COPIED + b), (uint32_t)((j / kRing - 1) & 1),
                                                                                p.status, KDA_DEVERR_TIMEOUT, WAIT_LIMIT, 256)))
                break;
            if (lane == 0) load_qkg(maps, u, c, b);
            put_beta(u, b, lane, load_beta<kBetaLogit>(p, u, c, lane));
            loaded = j + 1;
        }
        // boxes still in flight must land before the CTA exits (only after a timeout can one
        // be unconsumed)
        if (lane == 0)
            for (int j = loaded - kRing < 0 ? 0 : loaded - kRing; j < loaded; ++j)
                mbar_wait_bounded(bar_addr(u, B_FULLTMA + j % kRing), (uint32_t)((j / kRing) & 1), p.status, KDA_DEVERR_TIMEOUT,
                                  WAIT_LIMIT);
    } else if (pt == T_STORE) {
        int pushed = 0;
#pragma unroll 1
        for (int j = 0; j < nloc; ++j) {
            const int c = h + kNH * j, b = j % kRing, hs = c % NSH;
            const uint32_t par = (j / kRing) & 1;
            if (!mbar_wait_bounded(bar_addr(u, B_FULLP + b), par, p.status, KDA_DEVERR_TIMEOUT, WAIT_LIMIT, 256)) break;
            if (!mbar_wait_bounded(bar_addr(u, B_FULLD + b), par, p.status, KDA_DEVERR_TIMEOUT, WAIT_LIMIT, 256)) break;
            // home slot hs is free (and armed for this push) once the chain has finished chunk
            // c - NSH: one barrier per home slot the helper pushes into
            if (c >= NSH && !mbar_wait_bounded<true>(bar_addr(u, B_HSLOT + hs / kNH), (uint32_t)((c / NSH - 1) & 1), p.status,
                                                      KDA_DEVERR_TIMEOUT, WAIT_LIMIT, 256))
                break;
            const uint32_t dst = mapa_shared(u.base + slot_off(hs), 0u), full = mapa_shared(bar_addr(u, B_FULLOP + hs), 0u);
            const uint32_t src = u.base + slot_off(b);
            bulk_copy_to_peer(dst, src, PUSH_A, full);
            bulk_copy_to_peer(dst + SL_MQT, src + SL_MQT, PUSH_B, full);
            pushed = j + 1;
        }
        st_dsmem_u32(mapa_shared(u.base + OFF_PUSHED + 4 * h, 0u), (uint32_t)pushed);
    }
}

// kWarpIssue: the instantiation for one CTA per SM (warp-wide MMA issue, pipelined state
// pass, and the register file to itself: up to 128 registers a thread instead of 72).
// kCl: the cluster schedule (one CTA per SM too).
// kSmemState: the bf16 state resident in shared memory (one CTA per SM).
// kNH: (cluster schedules) helpers per cluster, 3 or 1.
template <bool kBf16State, bool kWarpIssue, bool kSoftplus, bool kBetaLogit, bool kCl = false, bool kSmemState = false,
          int kNH = 3>
__global__ void __launch_bounds__((kWarpIssue && !kCl && !kSmemState) ? TC_THREADS_LE : TC_THREADS, kWarpIssue ? 1 : 2)
    kda_fwd_tc_kernel(const FwdParams p, const __grid_constant__ TmaMaps maps) {
    constexpr int CL_SIZE = kNH + 1;
    // one CTA per SM: four more warps (14-17) read the output out
    constexpr bool kLoneEpi = kWarpIssue && !kCl && !kSmemState;
    extern __shared__ unsigned char smem_raw[];
    if (*reinterpret_cast<volatile uint32_t*>(p.status) & KDA_DEVERR_CU_SEQLENS) return;

    const int tid = threadIdx.x, warp = tid >> 5;
#ifdef KDA_CHECKED
    if (tid == 0) s_chk_status = p.status;   // published by the __syncthreads below
#endif
    const int rank = kCl ? (int)cluster_ctarank() : 0;   // 0: the home CTA
    const bool home = rank == 0;
    int seen[NSH] = {0, 0, 0};   // (cluster home, lane 0 of warp 9) chunks finished per home slot
    Unit u;
    {
        const uint32_t raw = smem_u32(smem_raw);
        u.base = (raw + 1023u) & ~1023u;
        u.gbase = smem_raw + (u.base - raw);
        const int unit = kCl ? (int)(blockIdx.x / CL_SIZE) : (int)blockIdx.x;
        u.h = unit % p.H;
        const int r = unit / p.H;
        u.n = p.order ? p.order[r] : r;
        seq_range(p, u.n, u.bos, u.eos);
        u.nchunks = (int)((u.eos - u.bos + CH - 1) / CH);
    }
    if (tid == 0) {
        for (int s = 0; s < MAX_RING; ++s) mbar_init(bar_addr(u, B_FULLTMA + s), 33);
        for (int b = B_FULLV; b < B_COUNT; ++b) mbar_init(bar_addr(u, b), 1);
        mbar_fence_init();
        if (kCl && home) {   // the first NSH home slots await their pushes
            for (int h = 0; h < NSH && h < u.nchunks; ++h) mbar_arrive_expect_tx(bar_addr(u, B_FULLOP + h), PUSH_BYTES);
            for (int h = 0; h < 3; ++h) *reinterpret_cast<int*>(u.gbase + OFF_PUSHED + 4 * h) = 0;
        }
    }
    if (tid == 32) {
        tma_prefetch_desc(&maps.q);
        tma_prefetch_desc(&maps.k);
        tma_prefetch_desc(&maps.v);
        tma_prefetch_desc(&maps.g);
        tma_prefetch_desc(&maps.out);
    }
    if (warp == 0 && home) {
        tmem_alloc(u.base + OFF_TMEMADDR, (kCl || kLoneEpi) ? TM_COLS_CL : TM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if constexpr (kCl) cluster_sync_all();   // every CTA's barriers are initialised before a peer arrives on one
    u.tmem = home ? *reinterpret_cast<volatile uint32_t*>(u.gbase + OFF_TMEMADDR) : 0u;

    if constexpr (!kCl) {
        // one CTA per SM (kLoneEpi): a ring of three slots
        constexpr int kRing = kLoneEpi ? NSL1 : NSLOT;
        if (warp < W_PREP0) {
            chain_group<kBf16State, kWarpIssue, kBetaLogit, false, kSmemState, kLoneEpi, kLoneEpi>(p, maps, u, tid);
        } else if (warp < W_INV) {
            prep_group<kSoftplus, 1, kRing>(p, u, tid - W_PREP0 * 32, 0, u.nchunks);
        } else if (warp == W_INV) {
            inverse_warp<kRing>(p, u, tid & 31, u.nchunks);
        } else if (warp == W_ISSUE) {
            mma_warp<kWarpIssue, false, kSmemState, kLoneEpi, kLoneEpi>(p, u, tid & 31);
        } else if (kLoneEpi) {
            home_epilogue<0>(p, maps, u, tid & 127, seen);   // warps 14-17: TMEM lanes 32 (warp % 4) ..
        }
    } else if (home) {
        if (warp < W_PREP0) chain_group<false, true, kBetaLogit, true>(p, maps, u, tid);
        else if (warp < W_PREP0 + 4) {}   // warps 4-7 have no part in the home CTA
        else if (warp < W_INV) home_epilogue<kNH>(p, maps, u, tid - (W_PREP0 + 4) * 32, seen);
        else if (warp == W_ISSUE) mma_warp<true, true, false>(p, u, tid & 31);
    } else {
        const int h = rank - 1;
        const int nloc = u.nchunks > h ? (u.nchunks - h + kNH - 1) / kNH : 0;
        if (warp < W_PREP0) helper_io<kBetaLogit, kNH>(p, maps, u, tid, h, nloc);
        else if (warp < W_INV) prep_group<kSoftplus, kNH, cl_ring(kNH)>(p, u, tid - W_PREP0 * 32, h, nloc);
        else if (warp == W_INV) inverse_warp<cl_ring(kNH)>(p, u, tid & 31, nloc);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0 && home) {
        tc_fence_after();
        tmem_dealloc(u.tmem, (kCl || kLoneEpi) ? TM_COLS_CL : TM_COLS);
    }
    // no CTA leaves while a peer may still read its shared memory, write it or arrive on its
    // barriers: every CTA has published its push count; the home waits for the pushes in flight
    if constexpr (kCl) {
        cluster_sync_all();
        if (home && warp == W_PREP0 + 5) {
            if ((tid & 31) == 0) home_drain<kNH>(p, u, seen);
            __syncwarp();   // converged at the aligned cluster barrier
        }
        cluster_sync_all();
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

// [T_total, H, 128] bf16 viewed as a 3-D tensor (d, h, t); boxes of `box_d` x 1 x 32
// (box_d = 64 with the 128-byte swizzle, 128 without).
bool encode_tokens_map(CUtensorMap* m, const void* ptr, int64_t T_total, int H, bool sw128 = false) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)HD, (cuuint64_t)H, (cuuint64_t)(T_total > 0 ? T_total : 1)};
    const cuuint64_t strides[2] = {(cuuint64_t)HD * 2, (cuuint64_t)H * HD * 2};
    const cuuint32_t box[3] = {(cuuint32_t)(sw128 ? 64 : HD), 1, (cuuint32_t)CH};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

using Kernel = void (*)(const FwdParams, const TmaMaps);

// The cluster instantiation for the flags and helper count (3: clusters of four CTAs, 1:
// clusters of two), with its launch configuration (the attribute array must outlive the
// configuration's use).
Kernel cluster_config(uint32_t flags, int nh, long long units, cudaStream_t stream, cudaLaunchAttribute* attr,
                      cudaLaunchConfig_t* cfg) {
    static constexpr Kernel table_cl[2][2][2] = {   // [one helper][softplus][beta logit]
        {{kda_fwd_tc_kernel<false, true, false, false, true>, kda_fwd_tc_kernel<false, true, false, true, true>},
         {kda_fwd_tc_kernel<false, true, true, false, true>, kda_fwd_tc_kernel<false, true, true, true, true>}},
        {{kda_fwd_tc_kernel<false, true, false, false, true, false, 1>, kda_fwd_tc_kernel<false, true, false, true, true, false, 1>},
         {kda_fwd_tc_kernel<false, true, true, false, true, false, 1>, kda_fwd_tc_kernel<false, true, true, true, true, false, 1>}}};
    const Kernel ck = table_cl[nh == 1][(flags & KDA_FLAG_GATE_SOFTPLUS) != 0][(flags & KDA_FLAG_BETA_LOGIT) != 0];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)(nh + 1);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    *cfg = cudaLaunchConfig_t{};
    cfg->gridDim = dim3((unsigned)(units * (nh + 1)));
    cfg->blockDim = dim3(TC_THREADS);
    cfg->dynamicSmemBytes = smem_bytes_cl(nh);
    cfg->stream = stream;
    cfg->attrs = attr;
    cfg->numAttrs = 1;
    return ck;
}

// Whether every cluster of (nh + 1) CTAs for `units` units can be resident at once.  The count
// is a property of the device and the instantiation: ask the runtime once (the query costs
// more host time than a whole launch) and keep the answer.
cudaError_t clusters_fit(int dev, uint32_t flags, int nh, long long units, bool* fit) {
    constexpr int kMaxDev = 64;
    static std::atomic<int> resident_cache[kMaxDev][2][4];   // zero-initialised: 0 = not asked yet
    const int fi = (int)(flags & 3u);
    std::atomic<int>* slot = dev < kMaxDev ? &resident_cache[dev][nh == 1][fi] : nullptr;
    int resident = slot ? slot->load(std::memory_order_relaxed) - 1 : -1;
    if (resident < 0) {
        cudaLaunchAttribute attr[1];
        cudaLaunchConfig_t cfg;
        const Kernel ck = cluster_config(flags, nh, units, nullptr, attr, &cfg);
        cudaError_t e = cudaFuncSetAttribute(ck, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes_cl(nh));
        if (e != cudaSuccess) return e;
        if (cudaOccupancyMaxActiveClusters(&resident, ck, &cfg) != cudaSuccess) {
            (void)cudaGetLastError();   // no cluster schedule on this device
            resident = 0;
        }
        if (slot) slot->store(resident + 1, std::memory_order_relaxed);
    }
    *fit = resident >= units;
    return cudaSuccess;
}

}  // namespace

size_t fwd_tc_smem_bytes() { return SMEM_BYTES; }

// One CTA per unit, two on an SM, when the units outnumber the SMs; with at most a quarter
// as many units as SMs, a cluster of four CTAs per unit, and with at most 7/25 as many a
// cluster of two, if every cluster can be resident at once (clusters must fit the GPCs);
// else one CTA per unit with an SM to itself.  (Clusters of two are paced by their one
// helper: on GB300, at 8,192 tokens a unit, they take 0.478 ms up to 42 units against 0.520
// for one CTA per SM, and 0.534 from 43 units on, a step measured at every count from 37 to
// 46; 7/25 of the 152 SMs is 42.6.)  The bf16-state ablation keeps its one instantiation.
cudaError_t fwd_tc_schedule(long long units, uint32_t flags, bool bf16_state, int* sched) {
    *sched = KDA_SCHEDULE_TWO_PER_SM;
    if (bf16_state || units <= 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (units > sms) return cudaSuccess;
    *sched = KDA_SCHEDULE_ONE_PER_SM;
    for (int nh : {3, 1}) {
        if (units * (nh + 1) > sms || (nh == 1 && units * 25 > 7LL * sms)) continue;
        bool fit = false;
        e = clusters_fit(dev, flags, nh, units, &fit);
        if (e != cudaSuccess) return e;
        if (fit) {
            *sched = nh == 3 ? KDA_SCHEDULE_CLUSTER : KDA_SCHEDULE_CLUSTER2;
            break;
        }
    }
    return cudaSuccess;
}

cudaError_t launch_fwd_tc(const FwdParams& p, cudaStream_t stream, bool bf16_state, bool smem_state) {
    const int units = p.nseq * p.H;
    if (units == 0) return cudaSuccess;
    TmaMaps maps;
    if (!encode_tokens_map(&maps.q, p.q, p.T_total, p.H) || !encode_tokens_map(&maps.k, p.k, p.T_total, p.H) ||
        !encode_tokens_map(&maps.v, p.v, p.T_total, p.H, true) || !encode_tokens_map(&maps.g, p.g, p.T_total, p.H) ||
        !encode_tokens_map(&maps.out, p.out, p.T_total, p.H, true))
        return cudaErrorInvalidValue;
    if (smem_state) {   // the shared-memory state alternative: one CTA per unit, one per SM
        auto ks = kda_fwd_tc_kernel<true, true, false, false, false, true>;
        cudaError_t e = cudaFuncSetAttribute(ks, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES_SS);
        if (e != cudaSuccess) return e;
        ks<<<units, TC_THREADS, SMEM_BYTES_SS, stream>>>(p, maps);
        return cudaGetLastError();
    }
    int sched = KDA_SCHEDULE_TWO_PER_SM;
    cudaError_t e = fwd_tc_schedule(units, p.flags, bf16_state, &sched);
    if (e != cudaSuccess) return e;
    if (sched == KDA_SCHEDULE_CLUSTER || sched == KDA_SCHEDULE_CLUSTER2) {
        const int nh = sched == KDA_SCHEDULE_CLUSTER ? 3 : 1;
        cudaLaunchAttribute attr[1];
        cudaLaunchConfig_t cfg;
        const Kernel ck = cluster_config(p.flags, nh, units, stream, attr, &cfg);
        e = cudaFuncSetAttribute(ck, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes_cl(nh));
        if (e != cudaSuccess) return e;
        e = cudaLaunchKernelEx(&cfg, ck, p, maps);
        return e != cudaSuccess ? e : cudaGetLastError();
    }
    // one CTA per SM: the MMA warp issues warp-wide (the interface variants are
    // separate instantiations, so the default one is unchanged)
    const bool lone = sched == KDA_SCHEDULE_ONE_PER_SM, sp = (p.flags & KDA_FLAG_GATE_SOFTPLUS) != 0;
    const bool lg = (p.flags & KDA_FLAG_BETA_LOGIT) != 0;
    static constexpr Kernel table[2][2][2] = {   // [lone][softplus][beta logit]
        {{kda_fwd_tc_kernel<false, false, false, false>, kda_fwd_tc_kernel<false, false, false, true>},
         {kda_fwd_tc_kernel<false, false, true, false>, kda_fwd_tc_kernel<false, false, true, true>}},
        {{kda_fwd_tc_kernel<false, true, false, false>, kda_fwd_tc_kernel<false, true, false, true>},
         {kda_fwd_tc_kernel<false, true, true, false>, kda_fwd_tc_kernel<false, true, true, true>}}};
    auto kernel = bf16_state ? kda_fwd_tc_kernel<true, false, false, false> : table[lone][sp][lg];
    const bool le = lone && !bf16_state;   // one CTA per SM: epilogue warps and a ring of three slots
    const uint32_t smem = le ? SMEM_BYTES_LE : SMEM_BYTES;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kernel<<<units, le ? TC_THREADS_LE : TC_THREADS, smem, stream>>>(p, maps);
    return cudaGetLastError();
}

}  // namespace kda
