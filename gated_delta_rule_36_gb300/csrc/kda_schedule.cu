// Unit scheduling for packed (cu_seqlens) mode: device-side validation of the
// boundaries and a longest-first sequence order, so that the long chains start
// first and the grid's tail is made of short sequences (FlashInfer PR #4262 notes,
// section 9: packed seq_order for tail utilisation; the result does not change).
#include "kda_kernels.h"

namespace kda {
namespace {

__global__ void kda_schedule_kernel(const int64_t* __restrict__ cu, int nseq, int64_t T_total,
                                    int32_t* __restrict__ order, uint32_t* __restrict__ status) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i == 0 && (cu[0] != 0 || cu[nseq] > T_total)) atomicOr(status, KDA_DEVERR_CU_SEQLENS);
    if (i >= nseq) return;
    const int64_t li = cu[i + 1] - cu[i];
    if (li < 0) atomicOr(status, KDA_DEVERR_CU_SEQLENS);
    if (nseq > kMaxSortedSeqs) {
        order[i] = i;
        return;
    }
    // rank in the order (length descending, index ascending): a permutation of 0..nseq-1
    int rank = 0;
    for (int j = 0; j < nseq; ++j) {
        const int64_t lj = cu[j + 1] - cu[j];
        rank += (lj > li) || (lj == li && j < i);
    }
    order[rank] = i;
}

}  // namespace

cudaError_t launch_schedule(const int64_t* cu_seqlens, int nseq, int64_t T_total, int32_t* order,
                            uint32_t* status, cudaStream_t stream) {
    const int threads = 256;
    const int blocks = nseq > 0 ? (nseq + threads - 1) / threads : 1;
    kda_schedule_kernel<<<blocks, threads, 0, stream>>>(cu_seqlens, nseq, T_total, order, status);
    return cudaGetLastError();
}

}  // namespace kda
