/*
 * kda.h -- C ABI of the GB300 (sm_103a) Kimi Delta Attention prefill forward.
 *
 * One call runs the whole chunked recurrent prefill of a batch on one GPU:
 * per (sequence, head) unit and per token it applies the in-kernel gate
 * (per-key-channel log-decay in [lower_bound, 0] from g, A_log, dt_bias),
 * L2-normalises q and k, decays the V x K state per key channel, applies the
 * beta-weighted delta-rule correction S += beta (v - S k) k^T and emits
 * out = scale * S q.  Inside, tokens are processed in 32-token chunks through the
 * centered intra-chunk matrices (Mqk, the inverse of the unit lower-triangular
 * system) and state/output GEMMs.
 *
 * Sources (web pages that describe the method; the library shares no code with them):
 *  - "FlashInfer PR #4262: Core Optimization Summary": section 1 (the fused
 *    per-chunk pipeline), section 2 (fixed-anchor exponent centering), section 3
 *    (chunk decomposition), sections 10 and 12 (exact in-place state alias and the
 *    supported contract: bf16 q/k/v/g/beta, head dim 128, fp32 A_log/dt_bias,
 *    finite negative lower_bound).
 *  - "How FlashKDA Manages Recurrent State Across Sequences and Batch Modes":
 *    the fwd(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound,
 *    initial_state, final_state, cu_seqlens) call, batched vs packed modes and the
 *    workspace sized from (T_total, H, N).
 *  - "How FlashKDA Stores On-Chip Recurrent State in BF16": bf16 or fp32 state I/O.
 *
 * Ownership: the caller owns every buffer, including the workspace.  The library
 * never allocates, frees or synchronises a stream inside kda_fwd; all work is
 * enqueued on `stream` in order.  All data pointers are DEVICE pointers.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream; NULL means the legacy default stream. */
typedef struct CUstream_st* kda_stream_t;

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1,   /* dtype, shape, contiguity, alignment or value check failed  */
    KDA_ERR_UNSUPPORTED = 2,   /* valid request outside the built kernel's contract            */
    KDA_ERR_ALIAS = 3,         /* initial/final state overlap other than an exact alias         */
    KDA_ERR_WORKSPACE = 4,     /* workspace missing, too small or misaligned                    */
    KDA_ERR_CUDA = 5           /* a CUDA runtime/driver call or kernel launch failed            */
} kda_status;

typedef enum { KDA_BF16 = 0, KDA_F32 = 1, KDA_I64 = 2 } kda_dtype;

/* A dense, contiguous (row-major) device tensor.  data == NULL marks an absent
 * optional tensor; the descriptor pointer itself may also be NULL for those. */
typedef struct {
    void* data;
    int32_t dtype;     /* kda_dtype */
    int32_t ndim;
    int64_t shape[4];
} kda_tensor;

/* Head dimension handled by the kernel: K = V = 128. */
#define KDA_HEAD_DIM 128
/* Most negative lower_bound the chunk-32 centered operands support:
 * 16 |lower_bound| log2(e) <= 126 keeps 2^(G - C) and 2^(C - G) normal in bf16
 * (FlashInfer PR #4262 notes, sections 2 and 14). */
#define KDA_MIN_LOWER_BOUND (-5.4585f)

/* Interface variants (the flags of kda_fwd_ex and kda_decode_ex; 0 = kda_fwd / kda_decode):
 * KDA_FLAG_BETA_LOGIT     beta holds logits; the step uses sigmoid(beta)
 * KDA_FLAG_GATE_SOFTPLUS  lambda = max(-exp(A_log) softplus(g + dt_bias), lower_bound)
 *                         instead of lower_bound sigmoid(exp(A_log) (g + dt_bias)); both lie in
 *                         [lower_bound, 0] (FlashInfer PR #4262 notes, sections 2 and 12) */
#define KDA_FLAG_BETA_LOGIT    0x1u
#define KDA_FLAG_GATE_SOFTPLUS 0x2u

/* Kernel selection (a 4-bit field of the flags of kda_fwd_ex, one value at a time): the
 * design alternatives the pages weigh, built beside the default kernel so that each can
 * be measured and checked against the oracle.  Each computes the same forward; none takes
 * an interface flag (KDA_ERR_UNSUPPORTED), and values not listed are KDA_ERR_INVALID_ARG.
 *   KDA_KERNEL_DEFAULT           32-token chunks, fixed exponent anchor, fp32 state resident
 *                                in Tensor Memory (FlashInfer PR #4262 notes, sections 2 and 6)
 *   KDA_KERNEL_CHUNK16           16-token chunks without the exponent anchor (same notes,
 *                                sections 2 and 14: the chunk-size alternative)
 *   KDA_KERNEL_REGISTER_STATE    fp32 state in mma.sync accumulator registers, every product
 *                                on mma.sync (the pre-tcgen05 placement of the state)
 *   KDA_KERNEL_BF16_STATE        the default kernel with the carried state rounded to bf16 at
 *                                every chunk boundary ("How FlashKDA Stores On-Chip Recurrent
 *                                State in BF16": the precision of a bf16 state store)
 *   KDA_KERNEL_SMEM_STATE        that bf16 state resident in shared memory (GEMM1 reads it through
 *                                a shared-memory descriptor; decay and update in fp32 in Tensor
 *                                Memory, rounded to bf16 once per chunk, as the same page and
 *                                "FlashKDA State Update Numerical Precision" describe); the extra
 *                                32 KB of shared memory leaves room for one CTA per SM */
#define KDA_FLAG_KERNEL_MASK        0xF00u
#define KDA_KERNEL_DEFAULT          0x000u
#define KDA_KERNEL_CHUNK16          0x100u
#define KDA_KERNEL_REGISTER_STATE   0x200u
#define KDA_KERNEL_BF16_STATE       0x300u
#define KDA_KERNEL_SMEM_STATE       0x400u

/* Device-side status bits, in the first 32-bit word of the workspace. */
#define KDA_DEVERR_CU_SEQLENS 0x1u  /* cu_seqlens[0] != 0, decreasing, or cu_seqlens[N] > T */
#define KDA_DEVERR_TIMEOUT    0x2u  /* a bounded on-chip wait expired; outputs are invalid  */
#define KDA_DEVERR_INTERNAL   0x4u  /* an internal consistency check failed                 */

/*
 * Bytes of workspace kda_fwd needs for T_total = B*T tokens, H heads and
 * N sequences (N = B in batched mode, the number of cu_seqlens intervals in
 * packed mode).  Mirrors get_workspace_size(T_total, H, N) of the FlashKDA API
 * page.  The workspace holds the device status word and the longest-first
 * sequence order; its contents need no initialisation.  Returns 0 for negative
 * arguments.
 */
size_t kda_workspace_size(int64_t T_total, int H, int N);

/*
 * Run the KDA chunked prefill forward.
 *
 *   q, k, g, out   bf16 [B, T, H, 128]         (out is written; rows of tokens that
 *   v              bf16 [B, T, H, 128]          belong to no sequence are NOT written)
 *   beta           bf16 [B, T, H]               used as given (no sigmoid)
 *   scale          finite float, applied to the normalised q
 *   A_log          fp32 [H];   dt_bias  fp32 [H, 128]
 *   lower_bound    finite, in [KDA_MIN_LOWER_BOUND, 0]
 *   initial_state  NULL/absent (= zero state) or bf16/fp32 [Nseq, H, 128 (V), 128 (K)]
 *   final_state    NULL/absent (not stored) or bf16/fp32 [Nseq, H, 128, 128]; may be the
 *                  exact same allocation (same pointer, dtype and shape) as initial_state
 *                  for an in-place update; any other overlap is KDA_ERR_ALIAS
 *   cu_seqlens     NULL/absent = batched mode (Nseq = B, one chain per batch row);
 *                  else int64 [N+1] with B == 1 (packed mode, Nseq = N): sequence n is
 *                  tokens [cu_seqlens[n], cu_seqlens[n+1]) and starts from
 *                  initial_state[n] (or zero); no state crosses a boundary
 *   workspace      >= kda_workspace_size(B*T, H, Nseq) bytes, 256-byte aligned
 *   stream         stream the work is enqueued on
 *
 * All tensors must be contiguous with 16-byte aligned data (beta: 2-byte).
 * Host-detectable problems return a status before anything is enqueued.  Problems
 * only the device can see (cu_seqlens contents, an expired bounded wait) set
 * KDA_DEVERR_* bits in the workspace; read them with kda_read_device_status.
 * A call whose cu_seqlens fail the device check writes neither out nor final_state.
 */
kda_status kda_fwd(const kda_tensor* q, const kda_tensor* k, const kda_tensor* v,
                   const kda_tensor* g, const kda_tensor* beta, float scale,
                   const kda_tensor* out, const kda_tensor* A_log, const kda_tensor* dt_bias,
                   float lower_bound, const kda_tensor* initial_state,
                   const kda_tensor* final_state, const kda_tensor* cu_seqlens,
                   void* workspace, size_t workspace_bytes, kda_stream_t stream);

/*
 * kda_fwd with interface variants and kernel selection: `flags` is a combination of
 * KDA_FLAG_* bits plus at most one KDA_KERNEL_* value in the KDA_FLAG_KERNEL_MASK field
 * (other bits or values: KDA_ERR_INVALID_ARG; an interface flag with a kernel other than
 * the default: KDA_ERR_UNSUPPORTED).  Everything else is as for kda_fwd.
 */
kda_status kda_fwd_ex(const kda_tensor* q, const kda_tensor* k, const kda_tensor* v,
                      const kda_tensor* g, const kda_tensor* beta, float scale,
                      const kda_tensor* out, const kda_tensor* A_log, const kda_tensor* dt_bias,
                      float lower_bound, const kda_tensor* initial_state,
                      const kda_tensor* final_state, const kda_tensor* cu_seqlens,
                      void* workspace, size_t workspace_bytes, uint32_t flags, kda_stream_t stream);

/*
 * The launch schedule the default (tensor-core) kernel of kda_fwd / kda_fwd_ex takes on the
 * current device for `units`
 * (sequence, head) units (sequences x H) with `flags`, written to *schedule:
 *   KDA_SCHEDULE_TWO_PER_SM  one CTA per unit, two CTAs sharing each SM (more units than SMs)
 *   KDA_SCHEDULE_ONE_PER_SM  one CTA per unit with an SM to itself (up to one unit per SM)
 *   KDA_SCHEDULE_CLUSTER     a cluster of four CTAs per unit: one runs the recurrence, three
 *                            prepare its chunks (up to a quarter as many units as SMs, when
 *                            every cluster can be resident at once)
 *   KDA_SCHEDULE_CLUSTER2    a cluster of two CTAs per unit: one runs the recurrence, one
 *                            prepares its chunks (up to 7/25 as many units as SMs, when the
 *                            clusters of four do not apply and every cluster of two can be
 *                            resident at once)
 * A unit's arithmetic is the same in every schedule: outputs and states do not depend on it.
 * Returns KDA_ERR_INVALID_ARG for units < 0, unknown flag bits, a kernel other than the
 * default or a null `schedule`, and
 * KDA_ERR_CUDA when the device cannot be queried.  An addition of this library: the
 * FlashInfer notes (section 9) choose instead between their M128 and M64 variants.
 */
#define KDA_SCHEDULE_TWO_PER_SM 0
#define KDA_SCHEDULE_ONE_PER_SM 1
#define KDA_SCHEDULE_CLUSTER    2
#define KDA_SCHEDULE_CLUSTER2   3
kda_status kda_fwd_schedule(int64_t units, uint32_t flags, int32_t* schedule);

/*
 * Chain trace, for profiling the recurrence of one unit (a profiling aid; off by default).
 * After kda_fwd_set_trace(buf, bytes, unit) with a device buffer, the forward launches of
 * this host thread that take a cluster schedule (KDA_SCHEDULE_CLUSTER or KDA_SCHEDULE_CLUSTER2)
 * record, for (sequence, head) unit `unit`
 * (sequence * H + head), KDA_TRACE_POINTS SM clock readings (uint64, one SM's clock) per
 * chunk c < bytes / (8 * KDA_TRACE_POINTS), at buf[c * KDA_TRACE_POINTS + i]:
 *   0 the chunk's iteration starts            4 GEMM1 has completed
 *   1 the MMA warp waits for the chunk's v    5 -R is in bf16 in Tensor Memory
 *   2 v has landed                            6 GEMM2's operands are ready
 *   3 GEMM1 is issued                         7 GEMM2 is issued
 * (points 0 and 4-6 are read by thread 0 of the chain, 1-3 and 7 by the MMA warp; point 6
 * is read after thread 0's non-blocking hand-off, so it can come a few cycles after 7.)
 * Other launches and entries leave the buffer untouched; outputs do not depend on tracing.
 * The caller owns the buffer, which the traced launches write on their streams: it must
 * stay allocated until they complete.  kda_fwd_set_trace(NULL, 0, 0) turns it off.  A
 * profiling aid of this library; the pages describe no counterpart.  Returns KDA_ERR_INVALID_ARG for a buffer
 * that is not 8-byte aligned or holds less than one chunk, or a negative unit.
 */
#define KDA_TRACE_POINTS 8
kda_status kda_fwd_set_trace(void* device_buffer, size_t bytes, int64_t unit);

/* Static description of a status code. */
const char* kda_status_string(kda_status s);

/* Human-readable detail of the last non-OK status returned on this host thread. */
const char* kda_last_error(void);

/*
 * Wait for `stream`, then copy the device status word of the last kda_fwd that
 * used `workspace` into *bits (0 = no device-side error).  Synchronises the
 * stream: meant for tests and debugging, not for the hot path.
 */
kda_status kda_read_device_status(const void* workspace, kda_stream_t stream, uint32_t* bits);

/* Largest number of sequences (N in packed mode, B in batched mode) that
 * kda_fwd_no_alloc accepts: its built-in workspace is 256 + 4 * this many bytes. */
#define KDA_NO_ALLOC_MAX_SEQS 16384

/*
 * The same forward as kda_fwd, for callers that cannot allocate device memory and
 * so cannot pass a workspace: for example a plugin inside a host framework that owns
 * the whole device memory pool and gives its plugins no allocator, or a serving loop
 * that must never allocate at run time.  The pages describe no counterpart of this
 * call; it is an addition of this library.
 *
 * Arguments, results and errors are those of kda_fwd, minus the workspace.  The
 * workspace is instead a fixed array in the library's own device memory
 * (256 + 4 * KDA_NO_ALLOC_MAX_SEQS bytes), which every GPU that loads the library
 * holds until the process exits.  Nothing in this call allocates or frees memory.
 *  - More than KDA_NO_ALLOC_MAX_SEQS sequences: KDA_ERR_UNSUPPORTED, nothing enqueued.
 *  - `stream` must belong to the current device (KDA_ERR_INVALID_ARG otherwise): the
 *    launches go to the current device, as for kda_fwd.
 *  - The first call on a device looks up the array's device address on that device;
 *    make that first call before any stream capture.  The address is kept for the
 *    rest of the process: it does not survive a cudaDeviceReset of that device.
 *  - Every call on a device shares the one array, and the array keeps what the last
 *    call left in it (kda_fwd clears the status word at the start of each call).
 *    Calls whose work overlaps on the GPU (for example on two streams at once) race
 *    on it: order them on one stream or with events.
 *  - If workspace_used is not NULL it receives the array's device address, so the
 *    status word can be read with kda_read_device_status.
 */
kda_status kda_fwd_no_alloc(const kda_tensor* q, const kda_tensor* k, const kda_tensor* v,
                            const kda_tensor* g, const kda_tensor* beta, float scale,
                            const kda_tensor* out, const kda_tensor* A_log, const kda_tensor* dt_bias,
                            float lower_bound, const kda_tensor* initial_state,
                            const kda_tensor* final_state, const kda_tensor* cu_seqlens,
                            kda_stream_t stream, const void** workspace_used);

/*
 * One decode step: every sequence takes one token, in the order of the recurrence of
 * kda_fwd (decay the state by exp(lambda) per key channel, delta-rule correction with the
 * normalised key, read-out of the written state with the normalised, scaled query).
 * The result equals kda_fwd with T = 1 in batched mode; the kernel is a separate one, a
 * single pass over each state row (the step is bound by the state's HBM traffic).
 *
 *   q, k, g, v, out  bf16 [B, H, 128]     one token per sequence
 *   beta             bf16 [B, H]          used as given
 *   scale, A_log, dt_bias, lower_bound    as for kda_fwd (lower_bound only needs to be
 *                                         finite and <= 0: no chunk operands to keep in range)
 *   initial_state    NULL/absent (zero) or bf16/fp32 [B, H, 128, 128]
 *   final_state      NULL/absent or bf16/fp32 [B, H, 128, 128]; may be exactly the same
 *                    allocation as initial_state (the usual in-place decode update)
 *   stream           stream the work is enqueued on
 *
 * No workspace and no device-side error: every check is made on the host before the
 * launch (KDA_ERR_INVALID_ARG / UNSUPPORTED / ALIAS / CUDA as for kda_fwd).
 */
kda_status kda_decode(const kda_tensor* q, const kda_tensor* k, const kda_tensor* v,
                      const kda_tensor* g, const kda_tensor* beta, float scale,
                      const kda_tensor* out, const kda_tensor* A_log, const kda_tensor* dt_bias,
                      float lower_bound, const kda_tensor* initial_state,
                      const kda_tensor* final_state, kda_stream_t stream);

/* kda_decode with interface variants (`flags` as for kda_fwd_ex). */
kda_status kda_decode_ex(const kda_tensor* q, const kda_tensor* k, const kda_tensor* v,
                         const kda_tensor* g, const kda_tensor* beta, float scale,
                         const kda_tensor* out, const kda_tensor* A_log, const kda_tensor* dt_bias,
                         float lower_bound, const kda_tensor* initial_state,
                         const kda_tensor* final_state, uint32_t flags, kda_stream_t stream);

/*
 * Device bytes kda_fwd_host needs for a request: q/k/v/g/out [B, T, H, 128], beta, A_log,
 * dt_bias, the states (init_dtype / final_dtype: KDA_BF16, KDA_F32, or -1 when absent),
 * N = number of cu_seqlens intervals (0 for batched mode), and the workspace.  Returns
 * 0 for invalid arguments.
 */
size_t kda_fwd_host_device_bytes(int64_t B, int64_t T, int H, int64_t N, int init_dtype, int final_dtype);

/*
 * kda_fwd on HOST buffers: every tensor descriptor (q ... cu_seqlens) points to host
 * memory, with the shapes, dtypes and meaning of kda_fwd.  The call copies the inputs to
 * `device_buffer` (>= kda_fwd_host_device_bytes bytes, 256-byte aligned, owned by the
 * caller and holding nothing the caller needs), runs the forward, and copies `out` and
 * `final_state` back.  It splits the sequences into up to `groups` consecutive groups whose
 * token counts fall from the first to the last (groups <= 0: 8; the last group's work is
 * the only part nothing overlaps) and pipelines them over three streams: the
 * host-to-device copies of group j + 1 run while group j computes and its results are
 * copied back.  The two copy streams and the events are the library's: created by a host
 * thread's first call on a device and reused by that thread's later calls there.  The work is ordered after everything already on `stream` and `stream`
 * is ordered after all of it; the call itself returns once the work is enqueued, so the
 * host buffers must stay untouched until `stream` reaches that point.  Host buffers should
 * be page-locked (cudaHostAlloc / pinned): pageable ones work but are copied synchronously.
 * Output rows of tokens that belong to no sequence are not written, as with kda_fwd.
 * initial_state and final_state may be the same host buffer (in place).
 *
 * Errors: the checks of kda_fwd, plus cu_seqlens validated on the host (cu[0] == 0,
 * non-decreasing, cu[N] <= B*T: KDA_ERR_INVALID_ARG) and a missing or too small
 * device_buffer (KDA_ERR_WORKSPACE); all before anything is enqueued.  Device-side status
 * bits go to the workspace inside device_buffer: read them with kda_read_device_status on
 * (char*)device_buffer + kda_fwd_host_workspace_offset(...).  Not capturable in a CUDA
 * graph (the per-group cu_seqlens are staged from pageable memory).
 */
kda_status kda_fwd_host(const kda_tensor* q, const kda_tensor* k, const kda_tensor* v,
                        const kda_tensor* g, const kda_tensor* beta, float scale,
                        const kda_tensor* out, const kda_tensor* A_log, const kda_tensor* dt_bias,
                        float lower_bound, const kda_tensor* initial_state,
                        const kda_tensor* final_state, const kda_tensor* cu_seqlens,
                        void* device_buffer, size_t device_bytes, int groups, kda_stream_t stream);

/* Byte offset of the workspace (and so of the device status word) inside the
 * device_buffer of a kda_fwd_host call with these arguments; 0 for invalid ones. */
size_t kda_fwd_host_workspace_offset(int64_t B, int64_t T, int H, int64_t N, int init_dtype, int final_dtype);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
