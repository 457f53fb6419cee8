// Single-token decode step: for every (sequence, head) one token decays, corrects and
// reads out the V x K state ("FlashInfer PR #4262: Core Optimization Summary", section 3,
// with a chunk of one token: the diagonal decay S D with D = diag(exp(lambda)), the
// delta-rule correction beta (v - S D k^) k^T, and the read-out of the written state).
//
// The state rows (V index) evolve independently, so one pass over each row does all of
// it: a = (S D k^)_r and b = (S D q^)_r come from one read of row r, then
//   u_r = beta (v_r - a),   S_r <- S_r D + u_r k^T,   out_r = scale (b + u_r (k^ . q^)),
// since (S D + u k^T) q^ = S D q^ + u (k^ . q^).  Each row is read once and written once:
// the step is bound by HBM (128 x 128 x 4 bytes each way per unit for an fp32 state).
//
// Grid: one CTA of 4 warps per (unit, block of 32 rows); a warp takes 8 rows, lane l the
// key channels 4 l .. 4 l + 3, and holds all 8 rows' loads in flight before it computes.
#include "kda_device.cuh"
#include "kda_kernels.h"

namespace kda {
namespace {

constexpr int DEC_THREADS = 128;
constexpr int DEC_ROWS_PER_WARP = 8;
constexpr int DEC_ROWS_PER_CTA = 32;
constexpr int DEC_BLOCKS_PER_UNIT = HD / DEC_ROWS_PER_CTA;

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

__device__ __forceinline__ float4 bf16x4_to_f4(uint2 w) {
    return make_float4(bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y));
}

template <bool kBetaLogit, bool kSoftplus>
__global__ void __launch_bounds__(DEC_THREADS) kda_decode_kernel(const FwdParams p) {
    const int unit = blockIdx.x / DEC_BLOCKS_PER_UNIT, rb = blockIdx.x % DEC_BLOCKS_PER_UNIT;
    const int h = unit % p.H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c0 = 4 * lane;
    const size_t tok = (size_t)unit * HD;   // the (sequence, head) row of q, k, v, g, out
    const int r0 = rb * DEC_ROWS_PER_CTA + warp * DEC_ROWS_PER_WARP;

    // per key channel (this lane's four): k^, q^, D = exp(lambda)
    const float4 q4 = bf16x4_to_f4(*reinterpret_cast<const uint2*>(p.q + tok + c0));
    const float4 k4 = bf16x4_to_f4(*reinterpret_cast<const uint2*>(p.k + tok + c0));
    const float4 g4 = bf16x4_to_f4(*reinterpret_cast<const uint2*>(p.g + tok + c0));
    const float4 dt = *reinterpret_cast<const float4*>(p.dt_bias + (size_t)h * HD + c0);
    const float rq = rsqrtf(warp_sum(q4.x * q4.x + q4.y * q4.y + q4.z * q4.z + q4.w * q4.w) + NORM_EPS);
    const float rk = rsqrtf(warp_sum(k4.x * k4.x + k4.y * k4.y + k4.z * k4.z + k4.w * k4.w) + NORM_EPS);
    const float kh[4] = {k4.x * rk, k4.y * rk, k4.z * rk, k4.w * rk};
    const float qh[4] = {q4.x * rq, q4.y * rq, q4.z * rq, q4.w * rq};
    const float kq = warp_sum(kh[0] * qh[0] + kh[1] * qh[1] + kh[2] * qh[2] + kh[3] * qh[3]);
    // lambda = lower_bound sigmoid(exp(A_log) (g + dt_bias)), or with KDA_FLAG_GATE_SOFTPLUS
    // max(-exp(A_log) softplus(g + dt_bias), lower_bound); base 2: D = 2^(lambda log2 e)
    const float eA = expf(p.A_log[h]);
    const float gm = -eA * LOG2E;
    const float bcoef = p.lower_bound * LOG2E;
    const float gx[4] = {g4.x + dt.x, g4.y + dt.y, g4.z + dt.z, g4.w + dt.w};
    float D[4], dk[4], dq[4];
    if constexpr (kSoftplus) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
            D[j] = ex2_approx(fmaxf(-eA * fmaf(fmaxf(gx[j], 0.f), LOG2E, lg2_approx(1.f + ex2_approx(-fabsf(gx[j]) * LOG2E))),
                                    bcoef));
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) D[j] = ex2_approx(bcoef * rcp_approx(1.f + ex2_approx(gm * gx[j])));
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        dk[j] = D[j] * kh[j];
        dq[j] = D[j] * qh[j];
    }
    float beta = bf16_bits_to_f32(reinterpret_cast<const uint16_t*>(p.beta)[unit]);
    if constexpr (kBetaLogit) beta = rcp_approx(1.f + ex2_approx(-beta * LOG2E));
    // the warp's 8 state rows, all loads in flight at once
    const size_t srow0 = ((size_t)unit * HD + r0) * HD + c0;
    float4 s[DEC_ROWS_PER_WARP];
#pragma unroll
    for (int i = 0; i < DEC_ROWS_PER_WARP; ++i) {
        const size_t off = srow0 + (size_t)i * HD;
        if (p.init_state == nullptr) s[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        else if (p.init_f32) s[i] = *reinterpret_cast<const float4*>(static_cast<const float*>(p.init_state) + off);
        else s[i] = bf16x4_to_f4(*reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(p.init_state) + off));
    }

    const float vr = bf16_bits_to_f32(reinterpret_cast<const uint16_t*>(p.v)[tok + r0 + (lane & 7)]);

    float my_out = 0.f;
#pragma unroll
    for (int i = 0; i < DEC_ROWS_PER_WARP; ++i) {
        const float sv[4] = {s[i].x, s[i].y, s[i].z, s[i].w};
        float a = 0.f, b = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            a = fmaf(sv[j], dk[j], a);
            b = fmaf(sv[j], dq[j], b);
        }
        a = warp_sum(a);
        b = warp_sum(b);
        const float u = beta * (__shfl_sync(0xffffffffu, vr, i) - a);
        if (lane == i) my_out = p.scale * fmaf(u, kq, b);
        float nv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) nv[j] = fmaf(sv[j], D[j], u * kh[j]);
        if (p.final_state != nullptr) {
            const size_t off = srow0 + (size_t)i * HD;
            if (p.final_f32)
                *reinterpret_cast<float4*>(static_cast<float*>(p.final_state) + off) = make_float4(nv[0], nv[1], nv[2], nv[3]);
            else
                *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.final_state) + off) =
                    make_uint2(pack_bf16x2(nv[0], nv[1]), pack_bf16x2(nv[2], nv[3]));
        }
    }
    if (lane < DEC_ROWS_PER_WARP)
        reinterpret_cast<uint16_t*>(p.out)[tok + r0 + lane] = (uint16_t)(pack_bf16x2(my_out, 0.f) & 0xffffu);
}

}  // namespace

cudaError_t launch_decode(const FwdParams& p, cudaStream_t stream) {
    const long long units = (long long)p.nseq * p.H;
    if (units == 0) return cudaSuccess;
    if (units * DEC_BLOCKS_PER_UNIT > 0x7fffffffLL) return cudaErrorInvalidValue;
    const bool logit = (p.flags & KDA_FLAG_BETA_LOGIT) != 0, sp = (p.flags & KDA_FLAG_GATE_SOFTPLUS) != 0;
    auto kernel = logit ? (sp ? kda_decode_kernel<true, true> : kda_decode_kernel<true, false>)
                        : (sp ? kda_decode_kernel<false, true> : kda_decode_kernel<false, false>);
    kernel<<<(unsigned)(units * DEC_BLOCKS_PER_UNIT), DEC_THREADS, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace kda
