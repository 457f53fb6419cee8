// C ABI of the KDA prefill forward: argument validation, workspace layout and
// stream-ordered launches.  Nothing here allocates device memory or synchronises
// (except kda_read_device_status, which exists to read the device status word).
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "kda.h"
#include "kda_kernels.h"

namespace {

thread_local char g_last_error[512] = "";
// kda_fwd_set_trace settings of this host thread
thread_local unsigned long long* g_trace = nullptr;
thread_local int64_t g_trace_chunks = 0, g_trace_unit = 0;

kda_status fail(kda_status s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    return s;
}

// Workspace layout (offsets in bytes):
//   [0, 256)         header: uint32 status word at 0, the rest reserved
//   [256, 256 + 4N)  int32 longest-first sequence order (packed mode)
constexpr size_t kHeaderBytes = 256;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

size_t elem_size(int32_t dt) { return dt == KDA_F32 ? 4 : dt == KDA_I64 ? 8 : 2; }

bool present(const kda_tensor* t) { return t != nullptr && t->data != nullptr; }

size_t numel(const kda_tensor* t) {
    size_t n = 1;
    for (int i = 0; i < t->ndim; ++i) n *= (size_t)t->shape[i];
    return n;
}

kda_status check_tensor(const char* name, const kda_tensor* t, int32_t dtype, int ndim,
                        const int64_t* shape, size_t align) {
    if (!present(t)) return fail(KDA_ERR_INVALID_ARG, "%s: missing", name);
    if (t->dtype != dtype) return fail(KDA_ERR_INVALID_ARG, "%s: dtype %d, expected %d", name, t->dtype, dtype);
    if (t->ndim != ndim) return fail(KDA_ERR_INVALID_ARG, "%s: ndim %d, expected %d", name, t->ndim, ndim);
    for (int i = 0; i < ndim; ++i) {
        if (t->shape[i] != shape[i]) {
            return fail(KDA_ERR_INVALID_ARG, "%s: dim %d is %lld, expected %lld", name, i,
                        (long long)t->shape[i], (long long)shape[i]);
        }
    }
    if (((uintptr_t)t->data) % align != 0)
        return fail(KDA_ERR_INVALID_ARG, "%s: data pointer not %zu-byte aligned", name, align);
    return KDA_OK;
}

kda_status check_state(const char* name, const kda_tensor* t, int64_t nseq, int64_t H) {
    if (!present(t)) return KDA_OK;
    if (t->dtype != KDA_BF16 && t->dtype != KDA_F32)
        return fail(KDA_ERR_INVALID_ARG, "%s: dtype must be bf16 or fp32", name);
    const int64_t shape[4] = {nseq, H, KDA_HEAD_DIM, KDA_HEAD_DIM};
    return check_tensor(name, t, t->dtype, 4, shape, 16);
}

}  // namespace

namespace kda {
// Record a message for kda_last_error() from another translation unit of the library.
void set_last_error(const char* msg) { snprintf(g_last_error, sizeof(g_last_error), "%s", msg); }
}  // namespace kda

extern "C" {

size_t kda_workspace_size(int64_t T_total, int H, int N) {
    if (T_total < 0 || H < 0 || N < 0) return 0;
    const size_t order_bytes = align_up((size_t)(N > 0 ? N : 1) * sizeof(int32_t), 256);
    return kHeaderBytes + order_bytes;
}

const char* kda_status_string(kda_status s) {
    switch (s) {
        case KDA_OK: return "ok";
        case KDA_ERR_INVALID_ARG: return "invalid argument";
        case KDA_ERR_UNSUPPORTED: return "unsupported configuration";
        case KDA_ERR_ALIAS: return "initial_state/final_state overlap without being an exact alias";
        case KDA_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
        case KDA_ERR_CUDA: return "CUDA error";
    }
    return "unknown status";
}

const char* kda_last_error(void) { return g_last_error; }

kda_status kda_fwd(const kda_tensor* q, const kda_tensor* k, const kda_tensor* v,
                   const kda_tensor* g, const kda_tensor* beta, float scale,
                   const kda_tensor* out, const kda_tensor* A_log, const kda_tensor* dt_bias,
                   float lower_bound, const kda_tensor* initial_state,
                   const kda_tensor* final_state, const kda_tensor* cu_seqlens,
                   void* workspace, size_t workspace_bytes, kda_stream_t stream) {
    g_last_error[0] = '\0';
    return kda::fwd_device(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state, final_state,
                           cu_seqlens, workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream), true, true,
                           0u);
}

kda_status kda_fwd_ex(const kda_tensor* q, const kda_tensor* k, const kda_tensor* v,
                      const kda_tensor* g, const kda_tensor* beta, float scale,
                      const kda_tensor* out, const kda_tensor* A_log, const kda_tensor* dt_bias,
                      float lower_bound, const kda_tensor* initial_state,
                      const kda_tensor* final_state, const kda_tensor* cu_seqlens,
                      void* workspace, size_t workspace_bytes, uint32_t flags, kda_stream_t stream) {
    g_last_error[0] = '\0';
    return kda::fwd_device(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state, final_state,
                           cu_seqlens, workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream), true, true,
                           flags);
}

}  // extern "C"

// The body of kda_fwd: every host-side check, then (with `enqueue`) the status reset
// (with `reset_status`), the schedule and the forward on `s`.
kda_status kda::fwd_device(const kda_tensor* q, const kda_tensor* k, const kda_tensor* v, const kda_tensor* g,
                           const kda_tensor* beta, float scale, const kda_tensor* out, const kda_tensor* A_log,
                           const kda_tensor* dt_bias, float lower_bound, const kda_tensor* initial_state,
                           const kda_tensor* final_state, const kda_tensor* cu_seqlens, void* workspace,
                           size_t workspace_bytes, cudaStream_t s, bool reset_status, bool enqueue,
                           uint32_t flags) {
    const uint32_t kernel = flags & KDA_FLAG_KERNEL_MASK;
    const uint32_t iface = flags & ~KDA_FLAG_KERNEL_MASK;
    if (iface & ~(KDA_FLAG_BETA_LOGIT | KDA_FLAG_GATE_SOFTPLUS))
        return fail(KDA_ERR_INVALID_ARG, "flags: unknown bits 0x%x", iface & ~(KDA_FLAG_BETA_LOGIT | KDA_FLAG_GATE_SOFTPLUS));
    if (kernel > KDA_KERNEL_SMEM_STATE) return fail(KDA_ERR_INVALID_ARG, "flags: unknown kernel 0x%x", kernel);
    if (kernel != KDA_KERNEL_DEFAULT && iface != 0)
        return fail(KDA_ERR_UNSUPPORTED, "the interface flags are built into the default kernel only");
    if (!present(q)) return fail(KDA_ERR_INVALID_ARG, "q: missing");
    if (q->ndim != 4) return fail(KDA_ERR_INVALID_ARG, "q: ndim %d, expected 4 [B,T,H,128]", q->ndim);
    const int64_t B = q->shape[0], T = q->shape[1], H = q->shape[2];
    if (q->shape[3] != KDA_HEAD_DIM)
        return fail(KDA_ERR_UNSUPPORTED, "head dim %lld: only %d is built", (long long)q->shape[3], KDA_HEAD_DIM);
    if (B < 1 || T < 0 || H < 1) return fail(KDA_ERR_INVALID_ARG, "bad q shape [%lld,%lld,%lld,128]",
                                             (long long)B, (long long)T, (long long)H);
    if (B * T > (int64_t)INT32_MAX || H > 65535)
        return fail(KDA_ERR_UNSUPPORTED, "B*T must be < 2^31 and H <= 65535");
    const int64_t qshape[4] = {B, T, H, KDA_HEAD_DIM};
    kda_status st;
    if ((st = check_tensor("q", q, KDA_BF16, 4, qshape, 16)) != KDA_OK) return st;
    if ((st = check_tensor("k", k, KDA_BF16, 4, qshape, 16)) != KDA_OK) return st;
    if ((st = check_tensor("v", v, KDA_BF16, 4, qshape, 16)) != KDA_OK) return st;
    if ((st = check_tensor("g", g, KDA_BF16, 4, qshape, 16)) != KDA_OK) return st;
    if ((st = check_tensor("out", out, KDA_BF16, 4, qshape, 16)) != KDA_OK) return st;
    const int64_t bshape[3] = {B, T, H};
    if ((st = check_tensor("beta", beta, KDA_BF16, 3, bshape, 2)) != KDA_OK) return st;
    const int64_t ashape[1] = {H};
    if ((st = check_tensor("A_log", A_log, KDA_F32, 1, ashape, 4)) != KDA_OK) return st;
    const int64_t dshape[2] = {H, KDA_HEAD_DIM};
    if ((st = check_tensor("dt_bias", dt_bias, KDA_F32, 2, dshape, 16)) != KDA_OK) return st;
    if (!isfinite(scale)) return fail(KDA_ERR_INVALID_ARG, "scale must be finite");
    if (!isfinite(lower_bound) || lower_bound > 0.f)
        return fail(KDA_ERR_INVALID_ARG, "lower_bound must be finite and <= 0");
    if (lower_bound < KDA_MIN_LOWER_BOUND)
        return fail(KDA_ERR_UNSUPPORTED,
                    "lower_bound %g < %g: chunk-32 centered operands would leave the bf16 normal range",
                    (double)lower_bound, (double)KDA_MIN_LOWER_BOUND);

    int64_t nseq = B;
    const bool packed = present(cu_seqlens);
    if (packed) {
        if (cu_seqlens->dtype != KDA_I64 || cu_seqlens->ndim != 1 || cu_seqlens->shape[0] < 1)
            return fail(KDA_ERR_INVALID_ARG, "cu_seqlens: expected int64 [N+1]");
        if (B != 1) return fail(KDA_ERR_INVALID_ARG, "packed mode (cu_seqlens) requires B == 1");
        if (((uintptr_t)cu_seqlens->data) % 8 != 0)
            return fail(KDA_ERR_INVALID_ARG, "cu_seqlens: data pointer not 8-byte aligned");
        nseq = cu_seqlens->shape[0] - 1;
        if (nseq > (int64_t)INT32_MAX / 65536) return fail(KDA_ERR_UNSUPPORTED, "too many sequences");
    }
    if ((st = check_state("initial_state", initial_state, nseq, H)) != KDA_OK) return st;
    if ((st = check_state("final_state", final_state, nseq, H)) != KDA_OK) return st;
    if (present(initial_state) && present(final_state)) {
        const uintptr_t a0 = (uintptr_t)initial_state->data;
        const uintptr_t a1 = a0 + numel(initial_state) * elem_size(initial_state->dtype);
        const uintptr_t b0 = (uintptr_t)final_state->data;
        const uintptr_t b1 = b0 + numel(final_state) * elem_size(final_state->dtype);
        const bool overlap = a0 < b1 && b0 < a1;
        if (overlap && !(a0 == b0 && initial_state->dtype == final_state->dtype))
            return fail(KDA_ERR_ALIAS, "initial_state and final_state overlap but are not the same buffer and dtype");
    }
    const size_t need = kda_workspace_size(B * T, (int)H, (int)nseq);
    if (workspace == nullptr || ((uintptr_t)workspace) % 256 != 0)
        return fail(KDA_ERR_WORKSPACE, "workspace must be a 256-byte aligned device pointer");
    if (workspace_bytes < need)
        return fail(KDA_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", workspace_bytes, need);

    if (!enqueue) return KDA_OK;
    uint32_t* status = static_cast<uint32_t*>(workspace);
    int32_t* order = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + kHeaderBytes);

    cudaError_t e = reset_status ? cudaMemsetAsync(status, 0, sizeof(uint32_t), s) : cudaSuccess;
    if (e != cudaSuccess) return fail(KDA_ERR_CUDA, "status reset: %s", cudaGetErrorString(e));
    if (packed) {
        e = kda::launch_schedule(static_cast<const int64_t*>(cu_seqlens->data), (int)nseq, B * T, order, status, s);
        if (e != cudaSuccess) return fail(KDA_ERR_CUDA, "schedule launch: %s", cudaGetErrorString(e));
    }

    kda::FwdParams p;
    memset(&p, 0, sizeof(p));
    p.q = static_cast<const __nv_bfloat16*>(q->data);
    p.k = static_cast<const __nv_bfloat16*>(k->data);
    p.v = static_cast<const __nv_bfloat16*>(v->data);
    p.g = static_cast<const __nv_bfloat16*>(g->data);
    p.beta = static_cast<const __nv_bfloat16*>(beta->data);
    p.out = static_cast<__nv_bfloat16*>(out->data);
    p.A_log = static_cast<const float*>(A_log->data);
    p.dt_bias = static_cast<const float*>(dt_bias->data);
    p.init_state = present(initial_state) ? initial_state->data : nullptr;
    p.init_f32 = present(initial_state) && initial_state->dtype == KDA_F32;
    p.final_state = present(final_state) ? final_state->data : nullptr;
    p.final_f32 = present(final_state) && final_state->dtype == KDA_F32;
    p.cu_seqlens = packed ? static_cast<const int64_t*>(cu_seqlens->data) : nullptr;
    p.order = packed ? order : nullptr;
    p.status = status;
    p.T = T;
    p.T_total = B * T;
    p.H = (int)H;
    p.nseq = (int)nseq;
    p.scale = scale;
    p.lower_bound = lower_bound;
    p.flags = iface;
    p.trace = g_trace;
    p.trace_chunks = g_trace_chunks;
    p.trace_unit = g_trace_unit;
    p.test_skip_chunk = -1;
#ifdef KDA_WAIT_TEST
    if (const char* sk = getenv("KDA_TEST_SKIP_FULLD")) p.test_skip_chunk = atoll(sk);
#endif

    // the kernel field selects a design alternative (include/kda.h); the default is the
    // tcgen05 kernel with 32-token chunks and the fp32 state resident in TMEM
    switch (kernel) {
        case KDA_KERNEL_CHUNK16: e = kda::launch_fwd_tc16(p, s); break;
        case KDA_KERNEL_REGISTER_STATE: e = kda::launch_fwd_mma(p, s); break;
        case KDA_KERNEL_BF16_STATE: e = kda::launch_fwd_tc(p, s, true); break;
        case KDA_KERNEL_SMEM_STATE: e = kda::launch_fwd_tc(p, s, true, true); break;
        default: e = kda::launch_fwd_tc(p, s, false); break;
    }
    if (e != cudaSuccess) return fail(KDA_ERR_CUDA, "forward launch: %s", cudaGetErrorString(e));
    return KDA_OK;
}

extern "C" {

kda_status kda_decode(const kda_tensor* q, const kda_tensor* k, const kda_tensor* v, const kda_tensor* g,
                      const kda_tensor* beta, float scale, const kda_tensor* out, const kda_tensor* A_log,
                      const kda_tensor* dt_bias, float lower_bound, const kda_tensor* initial_state,
                      const kda_tensor* final_state, kda_stream_t stream) {
    return kda_decode_ex(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state, final_state, 0u,
                         stream);
}

kda_status kda_decode_ex(const kda_tensor* q, const kda_tensor* k, const kda_tensor* v, const kda_tensor* g,
                         const kda_tensor* beta, float scale, const kda_tensor* out, const kda_tensor* A_log,
                         const kda_tensor* dt_bias, float lower_bound, const kda_tensor* initial_state,
                         const kda_tensor* final_state, uint32_t flags, kda_stream_t stream) {
    g_last_error[0] = '\0';
    if (flags & ~(KDA_FLAG_BETA_LOGIT | KDA_FLAG_GATE_SOFTPLUS))
        return fail(KDA_ERR_INVALID_ARG, "flags: unknown bits");
    if (!present(q)) return fail(KDA_ERR_INVALID_ARG, "q: missing");
    if (q->ndim != 3) return fail(KDA_ERR_INVALID_ARG, "q: ndim %d, expected 3 [B,H,128]", q->ndim);
    const int64_t B = q->shape[0], H = q->shape[1];
    if (q->shape[2] != KDA_HEAD_DIM)
        return fail(KDA_ERR_UNSUPPORTED, "head dim %lld: only %d is built", (long long)q->shape[2], KDA_HEAD_DIM);
    if (B < 0 || H < 1) return fail(KDA_ERR_INVALID_ARG, "bad q shape [%lld,%lld,128]", (long long)B, (long long)H);
    if (B * H > (int64_t)INT32_MAX / 4) return fail(KDA_ERR_UNSUPPORTED, "B*H too large");
    const int64_t tshape[3] = {B, H, KDA_HEAD_DIM};
    kda_status st;
    if ((st = check_tensor("q", q, KDA_BF16, 3, tshape, 16)) != KDA_OK) return st;
    if ((st = check_tensor("k", k, KDA_BF16, 3, tshape, 16)) != KDA_OK) return st;
    if ((st = check_tensor("v", v, KDA_BF16, 3, tshape, 16)) != KDA_OK) return st;
    if ((st = check_tensor("g", g, KDA_BF16, 3, tshape, 16)) != KDA_OK) return st;
    if ((st = check_tensor("out", out, KDA_BF16, 3, tshape, 16)) != KDA_OK) return st;
    const int64_t bshape[2] = {B, H};
    if ((st = check_tensor("beta", beta, KDA_BF16, 2, bshape, 2)) != KDA_OK) return st;
    const int64_t ashape[1] = {H};
    if ((st = check_tensor("A_log", A_log, KDA_F32, 1, ashape, 4)) != KDA_OK) return st;
    const int64_t dshape[2] = {H, KDA_HEAD_DIM};
    if ((st = check_tensor("dt_bias", dt_bias, KDA_F32, 2, dshape, 16)) != KDA_OK) return st;
    if (!isfinite(scale)) return fail(KDA_ERR_INVALID_ARG, "scale must be finite");
    if (!isfinite(lower_bound) || lower_bound > 0.f)
        return fail(KDA_ERR_INVALID_ARG, "lower_bound must be finite and <= 0");
    if ((st = check_state("initial_state", initial_state, B, H)) != KDA_OK) return st;
    if ((st = check_state("final_state", final_state, B, H)) != KDA_OK) return st;
    if (present(initial_state) && present(final_state)) {
        const uintptr_t a0 = (uintptr_t)initial_state->data;
        const uintptr_t a1 = a0 + numel(initial_state) * elem_size(initial_state->dtype);
        const uintptr_t b0 = (uintptr_t)final_state->data;
        const uintptr_t b1 = b0 + numel(final_state) * elem_size(final_state->dtype);
        if (a0 < b1 && b0 < a1 && !(a0 == b0 && initial_state->dtype == final_state->dtype))
            return fail(KDA_ERR_ALIAS, "initial_state and final_state overlap but are not the same buffer and dtype");
    }
    kda::FwdParams p;
    memset(&p, 0, sizeof(p));
    p.q = static_cast<const __nv_bfloat16*>(q->data);
    p.k = static_cast<const __nv_bfloat16*>(k->data);
    p.v = static_cast<const __nv_bfloat16*>(v->data);
    p.g = static_cast<const __nv_bfloat16*>(g->data);
    p.beta = static_cast<const __nv_bfloat16*>(beta->data);
    p.out = static_cast<__nv_bfloat16*>(out->data);
    p.A_log = static_cast<const float*>(A_log->data);
    p.dt_bias = static_cast<const float*>(dt_bias->data);
    p.init_state = present(initial_state) ? initial_state->data : nullptr;
    p.init_f32 = present(initial_state) && initial_state->dtype == KDA_F32;
    p.final_state = present(final_state) ? final_state->data : nullptr;
    p.final_f32 = present(final_state) && final_state->dtype == KDA_F32;
    p.flags = flags;
    p.T = 1;
    p.T_total = B;
    p.H = (int)H;
    p.nseq = (int)B;
    p.scale = scale;
    p.lower_bound = lower_bound;
    const cudaError_t e = kda::launch_decode(p, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(KDA_ERR_CUDA, "decode launch: %s", cudaGetErrorString(e));
    return KDA_OK;
}

kda_status kda_fwd_set_trace(void* device_buffer, size_t bytes, int64_t unit) {
    if (device_buffer == nullptr) {
        g_trace = nullptr;
        g_trace_chunks = 0;
        return KDA_OK;
    }
    const size_t per_chunk = 8u * KDA_TRACE_POINTS;
    if (((uintptr_t)device_buffer) % 8 != 0 || bytes < per_chunk || unit < 0)
        return fail(KDA_ERR_INVALID_ARG, "trace buffer must be 8-byte aligned and hold a chunk; unit >= 0");
    g_trace = static_cast<unsigned long long*>(device_buffer);
    g_trace_chunks = (int64_t)(bytes / per_chunk);
    g_trace_unit = unit;
    return KDA_OK;
}

kda_status kda_fwd_schedule(int64_t units, uint32_t flags, int32_t* schedule) {
    if (schedule == nullptr) return fail(KDA_ERR_INVALID_ARG, "null schedule");
    if (units < 0) return fail(KDA_ERR_INVALID_ARG, "units must be >= 0");
    if (flags & ~(KDA_FLAG_BETA_LOGIT | KDA_FLAG_GATE_SOFTPLUS))
        return fail(KDA_ERR_INVALID_ARG, "flags: unknown bits 0x%x (interface flags of the default kernel only)",
                    flags & ~(KDA_FLAG_BETA_LOGIT | KDA_FLAG_GATE_SOFTPLUS));
    int sched = KDA_SCHEDULE_TWO_PER_SM;
    const cudaError_t e = kda::fwd_tc_schedule(units, flags, false, &sched);
    if (e != cudaSuccess) return fail(KDA_ERR_CUDA, "schedule query: %s", cudaGetErrorString(e));
    *schedule = sched;
    return KDA_OK;
}

kda_status kda_read_device_status(const void* workspace, kda_stream_t stream, uint32_t* bits) {
    if (workspace == nullptr || bits == nullptr) return fail(KDA_ERR_INVALID_ARG, "null argument");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e == cudaSuccess) e = cudaMemcpy(bits, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail(KDA_ERR_CUDA, "status read: %s", cudaGetErrorString(e));
    return KDA_OK;
}

}  // extern "C"
