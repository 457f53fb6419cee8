// KDA chunked prefill forward, register-resident variant.
//
// One CTA (8 warps) per (sequence, head) unit.  The fp32 V x K state lives in the
// mma.sync accumulator registers of the 8 warps (warp w owns value rows
// 16w..16w+15) for the whole sequence, so it never leaves the SM between chunks.
// Every GEMM of a chunk runs on warp-level mma.sync (bf16 in, fp32 accumulate).
//
// Per 32-token chunk (FlashInfer PR #4262 notes, sections 1-3):
//   gate -> base-2 log-decay lambda2 in [b, 0], b = lower_bound*log2(e)
//   G = inclusive prefix of lambda2 over the chunk; G_T = G at the chunk end
//   q, k L2-normalised; fixed anchor C = 16 b (section 2)
//   Q_c = scale qh 2^(G-C), K_c = kh 2^(G-C), K_i = kh 2^(C-G)
//   L = strictLower(diag(beta) K_c K_i^T), Mqk = lowerTri(Q_c K_i^T), INV = (I+L)^-1
//   Q_d = Q_c 2^C, K_d = K_c 2^C, K_r = K_i 2^(G_T - C), a = 2^G_T
//   [O_0 | P] = S [Q_d | K_d]^T, R = (V^T - P) diag(beta), U = R INV^T
//   [S | O] = [S diag(a) | O_0] + U [K_r | Mqk^T]
// Tokens past the sequence end are zero-filled with lambda = beta = 0, which makes
// them inert in every product; their output rows are not stored.
#include "kda_device.cuh"
#include "kda_kernels.h"

namespace kda {
namespace {

constexpr int THREADS = 256;
constexpr int SROW = 136;  // bf16 stride of a 32 x 128 tile (272 B: ldmatrix rows hit distinct banks)
constexpr int TROW = 40;   // bf16 stride of a 32 x 32 tile
constexpr int FROW = 33;   // fp32 stride of a 32 x 32 tile

struct Smem {
    __nv_bfloat16 q[CH * SROW];    // raw q, then Q_d
    __nv_bfloat16 k[CH * SROW];    // raw k, then K_d
    __nv_bfloat16 v[CH * SROW];    // raw v
    __nv_bfloat16 g[CH * SROW];    // raw g, then K_r
    __nv_bfloat16 qc[CH * SROW];   // Q_c
    __nv_bfloat16 kc[CH * SROW];   // K_c
    __nv_bfloat16 ki[CH * SROW];   // K_i
    __nv_bfloat16 ost[CH * SROW];  // output staging [token][value row]
    __nv_bfloat16 mqk[CH * TROW];  // Mqk [i][j]
    __nv_bfloat16 inv[CH * TROW];  // INV [j][i]
    float L[CH * FROW];            // strictLower(diag(beta) K_c K_i^T)
    float X[CH * FROW];            // INV in fp32 (+ scratch in its upper-right block)
    float beta[CH];
    float rq[CH];
    float rk[CH];
    float tot[4][HD];              // per-quarter gate sums
    float a[HD];                   // 2^G_T
};

__device__ __forceinline__ void load_state(const FwdParams& p, size_t base, int w, int gq, int tq,
                                           float (&s)[16][4]) {
    if (!p.init_state) {
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
        return;
    }
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            const size_t off = base + (size_t)(16 * w + gq + 8 * hf) * HD + 8 * nt + 2 * tq;
            if (p.init_f32) {
                const float2 x = *reinterpret_cast<const float2*>(static_cast<const float*>(p.init_state) + off);
                s[nt][2 * hf] = x.x;
                s[nt][2 * hf + 1] = x.y;
            } else {
                const uint32_t x = *reinterpret_cast<const uint32_t*>(
                    static_cast<const __nv_bfloat16*>(p.init_state) + off);
                s[nt][2 * hf] = bf16_lo(x);
                s[nt][2 * hf + 1] = bf16_hi(x);
            }
        }
    }
}

__device__ __forceinline__ void store_state(const FwdParams& p, size_t base, int w, int gq, int tq,
                                            const float (&s)[16][4]) {
    if (!p.final_state) return;
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            const size_t off = base + (size_t)(16 * w + gq + 8 * hf) * HD + 8 * nt + 2 * tq;
            if (p.final_f32) {
                *reinterpret_cast<float2*>(static_cast<float*>(p.final_state) + off) =
                    make_float2(s[nt][2 * hf], s[nt][2 * hf + 1]);
            } else {
                *reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(p.final_state) + off) =
                    pack_bf16x2(s[nt][2 * hf], s[nt][2 * hf + 1]);
            }
        }
    }
}

__global__ void __launch_bounds__(THREADS, 1) kda_fwd_mma_kernel(const FwdParams p) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    Smem& sm = *reinterpret_cast<Smem*>(smem_raw);

    if (*reinterpret_cast<volatile uint32_t*>(p.status) & KDA_DEVERR_CU_SEQLENS) return;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gq = lane >> 2, tq = lane & 3;
    const int h = blockIdx.x % p.H;
    const int r = blockIdx.x / p.H;
    const int n = p.order ? p.order[r] : r;
    int64_t bos, eos;
    seq_range(p, n, bos, eos);
    const int nchunks = (int)((eos - bos + CH - 1) / CH);

    // Gate constants: lambda2 = b * sigmoid(eA (g + dt)), sigmoid(x) = 1 / (1 + 2^(-x log2 e)).
    const int pp = tid & 63, quarter = tid >> 6, ch0 = 2 * pp;
    const float eA = expf(p.A_log[h]);
    const float gm = -eA * LOG2E;
    const float gb0 = gm * p.dt_bias[h * HD + ch0];
    const float gb1 = gm * p.dt_bias[h * HD + ch0 + 1];
    const float bcoef = p.lower_bound * LOG2E;
    const float Cst = 16.f * bcoef;          // fixed anchor
    const float twoC = ex2_approx(Cst);

    const size_t sbase = ((size_t)n * p.H + h) * HD * HD;
    float s[16][4];
    load_state(p, sbase, warp, gq, tq, s);

    for (int c = 0; c < nchunks; ++c) {
        const int64_t t0 = bos + (int64_t)c * CH;
        const int nvalid = (int)((eos - t0) < CH ? (eos - t0) : CH);

        // ---- stage q, k, v, g rows of this chunk (zero-filled past the sequence end)
#pragma unroll
        for (int it = 0; it < 8; ++it) {
            const int idx = it * THREADS + tid;
            const int tsel = idx >> 9, row = (idx >> 4) & 31, seg = idx & 15;
            const __nv_bfloat16* base = tsel == 0 ? p.q : tsel == 1 ? p.k : tsel == 2 ? p.v : p.g;
            __nv_bfloat16* dst = (tsel == 0 ? sm.q : tsel == 1 ? sm.k : tsel == 2 ? sm.v : sm.g) +
                                 row * SROW + seg * 8;
            const bool valid = row < nvalid;
            const int64_t tok = valid ? t0 + row : bos;
            cp_async16(dst, base + (tok * p.H + h) * HD + seg * 8, valid ? 16 : 0);
        }
        cp_async_commit();
        if (tid < CH) {
            sm.beta[tid] = tid < nvalid
                ? bf16_bits_to_f32(reinterpret_cast<const uint16_t*>(p.beta)[(t0 + tid) * p.H + h])
                : 0.f;
        }
        cp_async_wait_all();
        __syncthreads();

        // ---- gate and local prefix (8 tokens x 2 channels per thread); row norms
        float G0[8], G1[8];
        {
            float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int i = quarter * 8 + j;
                const uint32_t gw = lds32(&sm.g[i * SROW + ch0]);
                float l0 = bcoef * rcp_approx(1.f + ex2_approx(fmaf(gm, bf16_lo(gw), gb0)));
                float l1 = bcoef * rcp_approx(1.f + ex2_approx(fmaf(gm, bf16_hi(gw), gb1)));
                if (i >= nvalid) l0 = l1 = 0.f;
                acc0 += l0;
                acc1 += l1;
                G0[j] = acc0;
                G1[j] = acc1;
            }
            sm.tot[quarter][ch0] = acc0;
            sm.tot[quarter][ch0 + 1] = acc1;
        }
        {
            const int rr = tid >> 2, part = tid & 3;
            const __nv_bfloat16* rowp = (rr < CH ? sm.q + rr * SROW : sm.k + (rr - CH) * SROW) + part * 32;
            float ss = 0.f;
#pragma unroll
            for (int e = 0; e < 32; e += 8) {
                const uint4 w4 = *reinterpret_cast<const uint4*>(rowp + e);
                const uint32_t ws[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const float lo = bf16_lo(ws[m]), hi = bf16_hi(ws[m]);
                    ss = fmaf(lo, lo, ss);
                    ss = fmaf(hi, hi, ss);
                }
            }
            ss += __shfl_xor_sync(0xffffffffu, ss, 1);
            ss += __shfl_xor_sync(0xffffffffu, ss, 2);
            if (part == 0) {
                const float rn = rsqrtf(ss + NORM_EPS);
                if (rr < CH) sm.rq[rr] = rn; else sm.rk[rr - CH] = rn;
            }
        }
        __syncthreads();

        // ---- prefix combine and centered operands
        {
            float off0 = 0.f, off1 = 0.f, tot0 = 0.f, tot1 = 0.f;
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
                const float a0 = sm.tot[qq][ch0], a1 = sm.tot[qq][ch0 + 1];
                if (qq < quarter) { off0 += a0; off1 += a1; }
                tot0 += a0;
                tot1 += a1;
            }
            const float rho0 = ex2_approx(tot0 - Cst), rho1 = ex2_approx(tot1 - Cst);
            if (quarter == 0) {
                sm.a[ch0] = ex2_approx(tot0);
                sm.a[ch0 + 1] = ex2_approx(tot1);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int i = quarter * 8 + j;
                const float Ga = G0[j] + off0, Gb = G1[j] + off1;
                const float ep0 = ex2_approx(Ga - Cst), ep1 = ex2_approx(Gb - Cst);
                const float em0 = ex2_approx(Cst - Ga), em1 = ex2_approx(Cst - Gb);
                const uint32_t qw = lds32(&sm.q[i * SROW + ch0]);
                const uint32_t kw = lds32(&sm.k[i * SROW + ch0]);
                const float qs = sm.rq[i] * p.scale, ks = sm.rk[i];
                const float q0 = bf16_lo(qw) * qs, q1 = bf16_hi(qw) * qs;
                const float k0 = bf16_lo(kw) * ks, k1 = bf16_hi(kw) * ks;
                const float qc0 = q0 * ep0, qc1 = q1 * ep1;
                const float kc0 = k0 * ep0, kc1 = k1 * ep1;
                const float ki0 = k0 * em0, ki1 = k1 * em1;
                const int o = i * SROW + ch0;
                *reinterpret_cast<uint32_t*>(&sm.qc[o]) = pack_bf16x2(qc0, qc1);
                *reinterpret_cast<uint32_t*>(&sm.kc[o]) = pack_bf16x2(kc0, kc1);
                *reinterpret_cast<uint32_t*>(&sm.ki[o]) = pack_bf16x2(ki0, ki1);
                *reinterpret_cast<uint32_t*>(&sm.q[o]) = pack_bf16x2(qc0 * twoC, qc1 * twoC);  // Q_d
                *reinterpret_cast<uint32_t*>(&sm.k[o]) = pack_bf16x2(kc0 * twoC, kc1 * twoC);  // K_d
                *reinterpret_cast<uint32_t*>(&sm.g[o]) = pack_bf16x2(ki0 * rho0, ki1 * rho1);  // K_r
            }
        }
        __syncthreads();

        // ---- intra-chunk products: warps 0-3 K_c K_i^T, warps 4-7 Q_c K_i^T (16x16 block each)
        {
            const int mat = warp >> 2, mt = (warp >> 1) & 1, nb = warp & 1;
            const __nv_bfloat16* Ab = mat ? sm.qc : sm.kc;
            float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                uint32_t a[4], b[4];
                ldmatrix_x4(a, Ab + (mt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * SROW + kk * 16 + (lane >> 4) * 8);
                ldmatrix_x4(b, sm.ki + (nb * 16 + (lane & 7) + (lane >> 4) * 8) * SROW + kk * 16 + ((lane >> 3) & 1) * 8);
                mma_bf16_16816(acc[0], a, b[0], b[1]);
                mma_bf16_16816(acc[1], a, b[2], b[3]);
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int i = mt * 16 + gq + (e >> 1) * 8;
                    const int j = nb * 16 + nt * 8 + 2 * tq + (e & 1);
                    const float val = acc[nt][e];
                    // select, never multiply: the masked upper triangle may hold inf/NaN
                    if (mat == 0) sm.L[i * FROW + j] = (j < i) ? sm.beta[i] * val : 0.f;
                    else sm.mqk[i * TROW + j] = __float2bfloat16_rn((j <= i) ? val : 0.f);
                }
            }
        }
        __syncthreads();

        // ---- INV = (I + L)^-1: two 16x16 diagonal blocks by forward substitution
        if (warp == 0) {
            const int o = (lane >> 4) * 16, col = lane & 15;
            float x[16];
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) x[rr] = (rr == col) ? 1.f : 0.f;
#pragma unroll
            for (int kk = 0; kk < 16; ++kk) {
                const float xk = x[kk];
#pragma unroll
                for (int rr = kk + 1; rr < 16; ++rr) x[rr] = fmaf(-sm.L[(o + rr) * FROW + o + kk], xk, x[rr]);
            }
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) sm.X[(o + rr) * FROW + o + col] = x[rr];
        }
        __syncthreads();
        {   // T1 = L21 A^-1 (kept in the unused upper-right block of X)
            const int rr = tid >> 4, cc = tid & 15;
            float acc = 0.f;
            for (int m = cc; m < 16; ++m) acc = fmaf(sm.L[(16 + rr) * FROW + m], sm.X[m * FROW + cc], acc);
            sm.X[rr * FROW + 16 + cc] = acc;
        }
        __syncthreads();
        {   // X21 = -D^-1 T1
            const int rr = tid >> 4, cc = tid & 15;
            float acc = 0.f;
            for (int m = 0; m <= rr; ++m) acc = fmaf(sm.X[(16 + rr) * FROW + 16 + m], sm.X[m * FROW + 16 + cc], acc);
            sm.X[(16 + rr) * FROW + cc] = -acc;
        }
        __syncthreads();
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int e = it * THREADS + tid, j = e >> 5, i = e & 31;
            sm.inv[j * TROW + i] = __float2bfloat16_rn(i <= j ? sm.X[j * FROW + i] : 0.f);
        }
        __syncthreads();

        // ---- recurrence for this warp's 16 value rows
        {
            float o[4][4], pm[4][4];
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) o[nt][e] = pm[nt][e] = 0.f;
            // [O_0 | P] = S [Q_d | K_d]^T
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t a[4] = {pack_bf16x2(s[2 * kk][0], s[2 * kk][1]),
                                       pack_bf16x2(s[2 * kk][2], s[2 * kk][3]),
                                       pack_bf16x2(s[2 * kk + 1][0], s[2 * kk + 1][1]),
                                       pack_bf16x2(s[2 * kk + 1][2], s[2 * kk + 1][3])};
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    const __nv_bfloat16* bq = sm.q + (nt * 8 + gq) * SROW + kk * 16 + 2 * tq;
                    mma_bf16_16816(o[nt], a, lds32(bq), lds32(bq + 8));
                    const __nv_bfloat16* bk = sm.k + (nt * 8 + gq) * SROW + kk * 16 + 2 * tq;
                    mma_bf16_16816(pm[nt], a, lds32(bk), lds32(bk + 8));
                }
            }
            // S_d = S diag(a)
#pragma unroll
            for (int nt = 0; nt < 16; ++nt) {
                const float a0 = sm.a[nt * 8 + 2 * tq], a1 = sm.a[nt * 8 + 2 * tq + 1];
                s[nt][0] *= a0; s[nt][1] *= a1; s[nt][2] *= a0; s[nt][3] *= a1;
            }
            // R = (V^T - P) diag(beta)
            const uint16_t* vs = reinterpret_cast<const uint16_t*>(sm.v);
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int i = nt * 8 + 2 * tq + (e & 1);
                    const int vr = 16 * warp + gq + (e >> 1) * 8;
                    pm[nt][e] = (bf16_bits_to_f32(vs[i * SROW + vr]) - pm[nt][e]) * sm.beta[i];
                }
            }
            // U = R INV^T
            float u[4][4];
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) u[nt][e] = 0.f;
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                const uint32_t a[4] = {pack_bf16x2(pm[2 * kk][0], pm[2 * kk][1]),
                                       pack_bf16x2(pm[2 * kk][2], pm[2 * kk][3]),
                                       pack_bf16x2(pm[2 * kk + 1][0], pm[2 * kk + 1][1]),
                                       pack_bf16x2(pm[2 * kk + 1][2], pm[2 * kk + 1][3])};
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    const __nv_bfloat16* bp = sm.inv + (nt * 8 + gq) * TROW + kk * 16 + 2 * tq;
                    mma_bf16_16816(u[nt], a, lds32(bp), lds32(bp + 8));
                }
            }
            // [S | O] += U [K_r | Mqk^T]
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                const uint32_t a[4] = {pack_bf16x2(u[2 * kk][0], u[2 * kk][1]),
                                       pack_bf16x2(u[2 * kk][2], u[2 * kk][3]),
                                       pack_bf16x2(u[2 * kk + 1][0], u[2 * kk + 1][1]),
                                       pack_bf16x2(u[2 * kk + 1][2], u[2 * kk + 1][3])};
#pragma unroll
                for (int np = 0; np < 8; ++np) {
                    uint32_t b[4];
                    ldmatrix_x4_trans(b, sm.g + (kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * SROW +
                                             np * 16 + (lane >> 4) * 8);
                    mma_bf16_16816(s[2 * np], a, b[0], b[1]);
                    mma_bf16_16816(s[2 * np + 1], a, b[2], b[3]);
                }
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    const __nv_bfloat16* bp = sm.mqk + (nt * 8 + gq) * TROW + kk * 16 + 2 * tq;
                    mma_bf16_16816(o[nt], a, lds32(bp), lds32(bp + 8));
                }
            }
            // O -> staging [token][value row]
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int i = nt * 8 + 2 * tq + (e & 1);
                    const int vr = 16 * warp + gq + (e >> 1) * 8;
                    sm.ost[i * SROW + vr] = __float2bfloat16_rn(o[nt][e]);
                }
            }
        }
        __syncthreads();
#pragma unroll
        for (int it = 0; it < 2; ++it) {
            const int idx = it * THREADS + tid, row = idx >> 4, seg = idx & 15;
            if (row < nvalid) {
                *reinterpret_cast<uint4*>(p.out + ((t0 + row) * p.H + h) * HD + seg * 8) =
                    *reinterpret_cast<const uint4*>(sm.ost + row * SROW + seg * 8);
            }
        }
        // The next chunk's staging writes only buffers whose last readers finished
        // before the barrier above; ost is rewritten only after several barriers.
    }
    store_state(p, sbase, warp, gq, tq, s);
}

}  // namespace

size_t fwd_mma_smem_bytes() { return sizeof(Smem); }

cudaError_t launch_fwd_mma(const FwdParams& p, cudaStream_t stream) {
    const int units = p.nseq * p.H;
    if (units == 0) return cudaSuccess;
    const size_t smem = sizeof(Smem);
    cudaError_t e = cudaFuncSetAttribute(kda_fwd_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kda_fwd_mma_kernel<<<units, THREADS, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace kda
