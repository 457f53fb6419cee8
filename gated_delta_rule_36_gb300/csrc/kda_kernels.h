// Internal launch entry points of the KDA kernels (host side, not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

#include "kda_device.cuh"
#include "kda.h"

namespace kda {

// Sequences are sorted longest-first only up to this count; beyond it the
// identity order is used (the sort is a quadratic rank count).
constexpr int kMaxSortedSeqs = 8192;

// Packed mode: validate cu_seqlens on the device (sets KDA_DEVERR_CU_SEQLENS) and
// write the longest-first sequence order to `order`.
cudaError_t launch_schedule(const int64_t* cu_seqlens, int nseq, int64_t T_total, int32_t* order,
                            uint32_t* status, cudaStream_t stream);

// Register-resident mma.sync forward (one CTA per unit): the ablation variant that
// keeps the state in mma.sync accumulator registers.
cudaError_t launch_fwd_mma(const FwdParams& p, cudaStream_t stream);
size_t fwd_mma_smem_bytes();

// tcgen05 forward (one CTA per unit, two per SM, state resident in TMEM).  bf16_state
// rounds the carried state to bf16 at every chunk boundary: the state-precision ablation;
// smem_state (with bf16_state) keeps that bf16 state resident in shared memory, one CTA per SM:
// the state-placement ablation.
cudaError_t launch_fwd_tc(const FwdParams& p, cudaStream_t stream, bool bf16_state = false, bool smem_state = false);
size_t fwd_tc_smem_bytes();
// The KDA_SCHEDULE_* a launch of the tensor-core kernel over `units` units takes on the
// current device.
cudaError_t fwd_tc_schedule(long long units, uint32_t flags, bool bf16_state, int* sched);

// The same with 16-token chunks and no exponent anchor: the chunk-size ablation.
cudaError_t launch_fwd_tc16(const FwdParams& p, cudaStream_t stream);

// Single-token decode step (T = 1 per sequence, batched layout [B, H, 128]).
cudaError_t launch_decode(const FwdParams& p, cudaStream_t stream);

}  // namespace kda

namespace kda {
// Set the text kda_last_error() returns on this host thread.
void set_last_error(const char* msg);

// The body of kda_fwd (include/kda.h): every host-side check of the request and, with
// `enqueue`, its launches on `stream`; `reset_status` clears the device status word first;
// `flags` are the KDA_FLAG_* interface variants.
// With enqueue == false nothing touches the device: the call only validates.
kda_status fwd_device(const kda_tensor* q, const kda_tensor* k, const kda_tensor* v, const kda_tensor* g,
                      const kda_tensor* beta, float scale, const kda_tensor* out, const kda_tensor* A_log,
                      const kda_tensor* dt_bias, float lower_bound, const kda_tensor* initial_state,
                      const kda_tensor* final_state, const kda_tensor* cu_seqlens, void* workspace,
                      size_t workspace_bytes, cudaStream_t stream, bool reset_status, bool enqueue,
                      uint32_t flags);
}  // namespace kda
