// kda_fwd_host: the forward on host buffers.  The caller hands in host tensors and one
// device buffer; the call copies the inputs in, runs the forward and copies the results
// out, pipelined over groups of sequences so that a group's host-to-device copies overlap
// the previous groups' forward and device-to-host copies (the link carries both
// directions at once).  Nothing here allocates memory; everything is stream-ordered after
// the work already on the caller's stream, and the call returns before the copies finish.
#include <string.h>

#include <algorithm>
#include <vector>

#include "kda.h"
#include "kda_kernels.h"

namespace {

constexpr size_t kAlign = 256;
constexpr int kMaxGroups = 64;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool present(const kda_tensor* t) { return t != nullptr && t->data != nullptr; }

size_t state_elem_bytes(int dtype) { return dtype == KDA_F32 ? 4 : dtype == KDA_BF16 ? 2 : 0; }

// Offsets of every device copy inside the caller's device buffer.
struct Layout {
    size_t q, k, v, g, out, beta, a_log, dt_bias, init, fin, cu, ws, ws_bytes, total;
};

Layout layout(int64_t B, int64_t T, int64_t H, int64_t nseq, int64_t ncu, int init_dtype, int final_dtype) {
    Layout L;
    const size_t tok = (size_t)(B * T) * (size_t)H * KDA_HEAD_DIM * 2;
    const size_t st = (size_t)nseq * (size_t)H * KDA_HEAD_DIM * KDA_HEAD_DIM;
    size_t o = 0;
    L.q = o; o = align_up(o + tok);
    L.k = o; o = align_up(o + tok);
    L.v = o; o = align_up(o + tok);
    L.g = o; o = align_up(o + tok);
    L.out = o; o = align_up(o + tok);
    L.beta = o; o = align_up(o + (size_t)(B * T) * (size_t)H * 2);
    L.a_log = o; o = align_up(o + (size_t)H * 4);
    L.dt_bias = o; o = align_up(o + (size_t)H * KDA_HEAD_DIM * 4);
    L.init = o; o = align_up(o + st * state_elem_bytes(init_dtype));
    L.fin = o; o = align_up(o + st * state_elem_bytes(final_dtype));
    L.cu = o; o = align_up(o + (size_t)(ncu > 0 ? ncu + kMaxGroups : 1) * sizeof(int64_t));
    L.ws = o;
    L.ws_bytes = kda_workspace_size(B * T, (int)H, (int)nseq);
    o = align_up(o + L.ws_bytes);
    L.total = o;
    return L;
}

kda_status fail(kda_status s, const char* msg) {
    kda::set_last_error(msg);
    return s;
}

kda_tensor dev_tensor(const kda_tensor* host, void* data) {
    kda_tensor t = *host;
    t.data = data;
    return t;
}

// The copy streams and events of one host thread on one device, created by the thread's
// first call there and reused by its later calls (streams and events are not allocated on
// the hot path).  Reusing an event is safe: cudaStreamWaitEvent waits for the record that is
// current when it is called, and every wait on an event is enqueued before the event is
// recorded again.
struct Resources {
    cudaStream_t s_in = nullptr, s_out = nullptr;
    cudaEvent_t ev[2 + 2 * kMaxGroups] = {};
    int used = 0;   // events handed out by the current call
    ~Resources() {   // at thread exit; errors (a runtime already unloaded) are ignored
        for (cudaEvent_t e : ev)
            if (e) cudaEventDestroy(e);
        if (s_in) cudaStreamDestroy(s_in);
        if (s_out) cudaStreamDestroy(s_out);
    }
    cudaError_t begin() {   // the streams (first call only) and a fresh run of events
        used = 0;
        cudaError_t r = cudaSuccess;
        if (!s_in) r = cudaStreamCreateWithFlags(&s_in, cudaStreamNonBlocking);
        if (r == cudaSuccess && !s_out) r = cudaStreamCreateWithFlags(&s_out, cudaStreamNonBlocking);
        return r;
    }
    cudaError_t event(cudaEvent_t* e) {
        if (used >= (int)(sizeof(ev) / sizeof(ev[0]))) return cudaErrorInvalidValue;
        cudaError_t r = cudaSuccess;
        if (!ev[used]) r = cudaEventCreateWithFlags(&ev[used], cudaEventDisableTiming);
        if (r == cudaSuccess) *e = ev[used++];
        return r;
    }
};

constexpr int kMaxDevices = 64;
thread_local Resources t_res[kMaxDevices];

}  // namespace

extern "C" {

size_t kda_fwd_host_device_bytes(int64_t B, int64_t T, int H, int64_t N, int init_dtype, int final_dtype) {
    if (B < 1 || T < 0 || H < 1 || N < 0) return 0;
    const int64_t nseq = N > 0 ? N : B;
    return layout(B, T, H, nseq, N > 0 ? N + 1 : 0, init_dtype, final_dtype).total;
}

size_t kda_fwd_host_workspace_offset(int64_t B, int64_t T, int H, int64_t N, int init_dtype, int final_dtype) {
    if (B < 1 || T < 0 || H < 1 || N < 0) return 0;
    const int64_t nseq = N > 0 ? N : B;
    return layout(B, T, H, nseq, N > 0 ? N + 1 : 0, init_dtype, final_dtype).ws;
}

kda_status kda_fwd_host(const kda_tensor* q, const kda_tensor* k, const kda_tensor* v, const kda_tensor* g,
                        const kda_tensor* beta, float scale, const kda_tensor* out, const kda_tensor* A_log,
                        const kda_tensor* dt_bias, float lower_bound, const kda_tensor* initial_state,
                        const kda_tensor* final_state, const kda_tensor* cu_seqlens, void* device_buffer,
                        size_t device_bytes, int groups, kda_stream_t stream) {
    kda::set_last_error("");
    if (!present(q) || q->ndim != 4) return fail(KDA_ERR_INVALID_ARG, "q: expected a 4-D [B,T,H,128] tensor");
    const int64_t B = q->shape[0], T = q->shape[1], H = q->shape[2];
    if (B < 1 || T < 0 || H < 1) return fail(KDA_ERR_INVALID_ARG, "bad q shape");
    if (!present(k) || !present(v) || !present(g) || !present(out) || !present(beta) || !present(A_log) ||
        !present(dt_bias))
        return fail(KDA_ERR_INVALID_ARG, "q, k, v, g, beta, out, A_log and dt_bias are required");
    const bool packed = present(cu_seqlens);
    if (packed && (cu_seqlens->dtype != KDA_I64 || cu_seqlens->ndim != 1 || cu_seqlens->shape[0] < 1))
        return fail(KDA_ERR_INVALID_ARG, "cu_seqlens: expected int64 [N+1]");
    const int64_t ncu = packed ? cu_seqlens->shape[0] : 0;
    const int64_t nseq = packed ? ncu - 1 : B;
    const int init_dtype = present(initial_state) ? initial_state->dtype : -1;
    const int final_dtype = present(final_state) ? final_state->dtype : -1;
    if (device_buffer == nullptr || ((uintptr_t)device_buffer) % kAlign != 0)
        return fail(KDA_ERR_WORKSPACE, "device_buffer must be a 256-byte aligned device pointer");
    const Layout L = layout(B, T, H, nseq, packed ? ncu : 0, init_dtype, final_dtype);
    if (device_bytes < L.total) return fail(KDA_ERR_WORKSPACE, "device_buffer too small (see kda_fwd_host_device_bytes)");
    char* dbuf = static_cast<char*>(device_buffer);

    // the device-side request: the same checks as kda_fwd, on the full-size copies
    kda_tensor dq = dev_tensor(q, dbuf + L.q), dk = dev_tensor(k, dbuf + L.k), dv = dev_tensor(v, dbuf + L.v);
    kda_tensor dg = dev_tensor(g, dbuf + L.g), dout = dev_tensor(out, dbuf + L.out);
    kda_tensor db = dev_tensor(beta, dbuf + L.beta), da = dev_tensor(A_log, dbuf + L.a_log);
    kda_tensor dd = dev_tensor(dt_bias, dbuf + L.dt_bias);
    kda_tensor di{}, df{}, dc{};
    if (present(initial_state)) di = dev_tensor(initial_state, dbuf + L.init);
    if (present(final_state)) df = dev_tensor(final_state, dbuf + L.fin);
    if (packed) dc = dev_tensor(cu_seqlens, dbuf + L.cu);
    kda_status st = kda::fwd_device(&dq, &dk, &dv, &dg, &db, scale, &dout, &da, &dd, lower_bound,
                                    present(initial_state) ? &di : nullptr, present(final_state) ? &df : nullptr,
                                    packed ? &dc : nullptr, dbuf + L.ws, L.ws_bytes, nullptr, false, false, 0u);
    if (st != KDA_OK) return st;
    // host states: in place (the same buffer) or disjoint, as for kda_fwd
    if (present(initial_state) && present(final_state)) {
        const size_t sb = (size_t)nseq * H * KDA_HEAD_DIM * KDA_HEAD_DIM;
        const uintptr_t a0 = (uintptr_t)initial_state->data, a1 = a0 + sb * state_elem_bytes(init_dtype);
        const uintptr_t b0 = (uintptr_t)final_state->data, b1 = b0 + sb * state_elem_bytes(final_dtype);
        if (a0 < b1 && b0 < a1 && !(a0 == b0 && init_dtype == final_dtype))
            return fail(KDA_ERR_ALIAS, "initial_state and final_state overlap but are not the same buffer and dtype");
    }

    // sequences of each group: consecutive, with token counts falling linearly from the
    // first group to the last (proportional to want, want - 1, ..., 1): the last group's
    // forward and copies back are the part of the call nothing overlaps, so it is the smallest
    const int64_t* cu = packed ? static_cast<const int64_t*>(cu_seqlens->data) : nullptr;
    if (packed) {
        if (cu[0] != 0) return fail(KDA_ERR_INVALID_ARG, "cu_seqlens[0] must be 0");
        for (int64_t n = 0; n < nseq; ++n)
            if (cu[n + 1] < cu[n]) return fail(KDA_ERR_INVALID_ARG, "cu_seqlens must be non-decreasing");
        if (cu[nseq] > B * T) return fail(KDA_ERR_INVALID_ARG, "cu_seqlens[N] exceeds the token count");
    }
    const int want = std::max(1, std::min(groups > 0 ? groups : 8, kMaxGroups));
    auto tok_of = [&](int64_t n) { return packed ? cu[n] : n * T; };   // first token of sequence n
    const int64_t tok_total = tok_of(nseq);
    std::vector<int64_t> cut{0};   // group j: sequences [cut[j], cut[j+1])
    const int64_t wsum = (int64_t)want * (want + 1) / 2;
    int64_t wacc = 0;
    for (int j = 1; j < want; ++j) {
        wacc += want - (j - 1);   // weight of group j - 1
        const int64_t target = tok_total * wacc / wsum;
        int64_t n = cut.back();
        while (n < nseq && tok_of(n) < target) ++n;
        if (n > cut.back() && n < nseq) cut.push_back(n);
    }
    cut.push_back(nseq);
    const int ng = (int)cut.size() - 1;

    // rebased cu_seqlens of every group, one copy (staged from pageable memory)
    std::vector<int64_t> cu_groups;
    std::vector<size_t> cu_off(ng, 0);
    if (packed) {
        for (int j = 0; j < ng; ++j) {
            cu_off[j] = cu_groups.size();
            for (int64_t n = cut[j]; n <= cut[j + 1]; ++n) cu_groups.push_back(cu[n] - cu[cut[j]]);
        }
    }

    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        kda::set_last_error(e != cudaSuccess ? cudaGetErrorString(e) : "device index out of range");
        return KDA_ERR_CUDA;
    }
    Resources& r = t_res[dev];
    cudaStream_t s_user = reinterpret_cast<cudaStream_t>(stream);
    cudaEvent_t ev_start, ev_done;
    e = r.begin();
    if (e == cudaSuccess) e = r.event(&ev_start);
    if (e == cudaSuccess) e = r.event(&ev_done);
    if (e == cudaSuccess) e = cudaEventRecord(ev_start, s_user);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(r.s_in, ev_start, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(r.s_out, ev_start, 0);
    auto h2d = [&](size_t doff, const void* src, size_t bytes) {
        if (e == cudaSuccess && bytes > 0) e = cudaMemcpyAsync(dbuf + doff, src, bytes, cudaMemcpyHostToDevice, r.s_in);
    };
    auto d2h = [&](void* dst, size_t doff, size_t bytes) {
        if (e == cudaSuccess && bytes > 0) e = cudaMemcpyAsync(dst, dbuf + doff, bytes, cudaMemcpyDeviceToHost, r.s_out);
    };
    if (packed) h2d(L.cu, cu_groups.data(), cu_groups.size() * sizeof(int64_t));
    h2d(L.a_log, A_log->data, (size_t)H * 4);
    h2d(L.dt_bias, dt_bias->data, (size_t)H * KDA_HEAD_DIM * 4);

    const size_t row = (size_t)H * KDA_HEAD_DIM * 2;                        // one token of q, k, v, g, out
    const size_t srow = (size_t)H * KDA_HEAD_DIM * KDA_HEAD_DIM;            // one sequence of the state
    for (int j = 0; j < ng && e == cudaSuccess; ++j) {
        const int64_t n0 = cut[j], n1 = cut[j + 1];
        const int64_t t0 = tok_of(n0), t1 = tok_of(n1);
        const size_t ntok = (size_t)(t1 - t0);
        h2d(L.q + t0 * row, static_cast<const char*>(q->data) + t0 * row, ntok * row);
        h2d(L.k + t0 * row, static_cast<const char*>(k->data) + t0 * row, ntok * row);
        h2d(L.v + t0 * row, static_cast<const char*>(v->data) + t0 * row, ntok * row);
        h2d(L.g + t0 * row, static_cast<const char*>(g->data) + t0 * row, ntok * row);
        h2d(L.beta + t0 * H * 2, static_cast<const char*>(beta->data) + t0 * H * 2, ntok * H * 2);
        if (present(initial_state)) {
            const size_t es = state_elem_bytes(init_dtype);
            h2d(L.init + n0 * srow * es, static_cast<const char*>(initial_state->data) + n0 * srow * es,
                (size_t)(n1 - n0) * srow * es);
        }
        cudaEvent_t ev_in, ev_fwd;
        if (e == cudaSuccess) e = r.event(&ev_in);
        if (e == cudaSuccess) e = r.event(&ev_fwd);
        if (e == cudaSuccess) e = cudaEventRecord(ev_in, r.s_in);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s_user, ev_in, 0);
        if (e != cudaSuccess) break;

        // the group's forward on the caller's stream: its tokens and states, offset
        const int64_t gB = packed ? 1 : n1 - n0, gT = packed ? (t1 - t0) : T;
        const int64_t tshape[4] = {gB, gT, H, KDA_HEAD_DIM};
        auto tok_tensor = [&](size_t base) {
            kda_tensor t{};
            t.data = dbuf + base + t0 * row;
            t.dtype = KDA_BF16;
            t.ndim = 4;
            memcpy(t.shape, tshape, sizeof(tshape));
            return t;
        };
        kda_tensor gq = tok_tensor(L.q), gk = tok_tensor(L.k), gv = tok_tensor(L.v), gg = tok_tensor(L.g);
        kda_tensor gout = tok_tensor(L.out);
        kda_tensor gb{};
        gb.data = dbuf + L.beta + t0 * H * 2;
        gb.dtype = KDA_BF16;
        gb.ndim = 3;
        gb.shape[0] = gB; gb.shape[1] = gT; gb.shape[2] = H;
        kda_tensor gi{}, gf{}, gc{};
        const int64_t sshape[4] = {n1 - n0, H, KDA_HEAD_DIM, KDA_HEAD_DIM};
        if (present(initial_state)) {
            gi.data = dbuf + L.init + n0 * srow * state_elem_bytes(init_dtype);
            gi.dtype = init_dtype; gi.ndim = 4; memcpy(gi.shape, sshape, sizeof(sshape));
        }
        if (present(final_state)) {
            gf.data = dbuf + L.fin + n0 * srow * state_elem_bytes(final_dtype);
            gf.dtype = final_dtype; gf.ndim = 4; memcpy(gf.shape, sshape, sizeof(sshape));
        }
        if (packed) {
            gc.data = dbuf + L.cu + cu_off[j] * sizeof(int64_t);
            gc.dtype = KDA_I64; gc.ndim = 1; gc.shape[0] = n1 - n0 + 1;
        }
        st = kda::fwd_device(&gq, &gk, &gv, &gg, &gb, scale, &gout, &da, &dd, lower_bound,
                             present(initial_state) ? &gi : nullptr, present(final_state) ? &gf : nullptr,
                             packed ? &gc : nullptr, dbuf + L.ws, L.ws_bytes, s_user, j == 0, true, 0u);
        if (st != KDA_OK) return st;
        if ((e = cudaEventRecord(ev_fwd, s_user)) == cudaSuccess) e = cudaStreamWaitEvent(r.s_out, ev_fwd, 0);

        // the group's results back to the host
        d2h(static_cast<char*>(out->data) + t0 * row, L.out + t0 * row, ntok * row);
        if (present(final_state)) {
            const size_t es = state_elem_bytes(final_dtype);
            d2h(static_cast<char*>(final_state->data) + n0 * srow * es, L.fin + n0 * srow * es,
                (size_t)(n1 - n0) * srow * es);
        }
    }
    if (e == cudaSuccess) e = cudaEventRecord(ev_done, r.s_out);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s_user, ev_done, 0);
    if (e != cudaSuccess) {
        kda::set_last_error(cudaGetErrorString(e));
        return KDA_ERR_CUDA;
    }
    return KDA_OK;
}

}  // extern "C"
