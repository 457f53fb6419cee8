// kda_fwd_no_alloc: the same forward as kda_fwd for callers that cannot hand the
// library a workspace buffer, because they have no way to allocate device memory
// themselves -- for example a plugin running inside a host framework that owns the
// whole device memory pool and gives its plugins no allocator, or a serving loop
// that must not allocate (an allocation can block, fragment the pool or fail at run
// time).
//
// The workspace lives in a fixed-size array in this library's own device memory
// (`g_no_alloc_workspace`, below).  Every GPU that loads the library holds that array
// until the process exits.  Nothing here calls cudaMalloc, cudaFree or any other
// allocating routine.
#include <mutex>

#include "kda.h"
#include "kda_kernels.h"

namespace {

// Largest number of sequences (N in packed mode, B in batched mode) a call may use.
constexpr int kNoAllocMaxSeqs = KDA_NO_ALLOC_MAX_SEQS;
// Same layout as a caller workspace: 256-byte header + int32 order per sequence.
constexpr size_t kNoAllocBytes = 256 + (size_t)kNoAllocMaxSeqs * sizeof(int32_t);

// Device-resident workspace shared by every kda_fwd_no_alloc call on a device.
// In host code this name is only a stand-in for the symbol: its device address comes
// from cudaGetSymbolAddress, looked up once per device.
static __device__ __align__(256) unsigned char g_no_alloc_workspace[kNoAllocBytes];

constexpr int kMaxDevices = 256;
std::mutex g_mu;
void* g_workspace_addr[kMaxDevices] = {};

// Device address of g_no_alloc_workspace on `dev`, resolved once with `dev` current.  The
// cached address does not survive cudaDeviceReset on that device.
cudaError_t workspace_address(int dev, void** addr) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_workspace_addr[dev] == nullptr) {
        int prev = -1;
        cudaError_t e = cudaGetDevice(&prev);
        if (e != cudaSuccess) return e;
        if (prev != dev && (e = cudaSetDevice(dev)) != cudaSuccess) return e;
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_no_alloc_workspace);
        if (prev != dev) {
            const cudaError_t e2 = cudaSetDevice(prev);
            if (e == cudaSuccess) e = e2;
        }
        if (e != cudaSuccess) return e;
        g_workspace_addr[dev] = p;
    }
    *addr = g_workspace_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" kda_status kda_fwd_no_alloc(const kda_tensor* q, const kda_tensor* k, const kda_tensor* v,
                                       const kda_tensor* g, const kda_tensor* beta, float scale,
                                       const kda_tensor* out, const kda_tensor* A_log,
                                       const kda_tensor* dt_bias, float lower_bound,
                                       const kda_tensor* initial_state, const kda_tensor* final_state,
                                       const kda_tensor* cu_seqlens, kda_stream_t stream,
                                       const void** workspace_used) {
    if (workspace_used) *workspace_used = nullptr;
    // Refuse, before touching the device, a batch that needs more than the array holds.
    if (q != nullptr && q->data != nullptr && q->ndim == 4) {
        const int64_t nseq = (cu_seqlens != nullptr && cu_seqlens->data != nullptr && cu_seqlens->ndim == 1)
                                 ? cu_seqlens->shape[0] - 1
                                 : q->shape[0];
        if (nseq > kNoAllocMaxSeqs) {
            kda::set_last_error("kda_fwd_no_alloc: more sequences than the built-in workspace holds "
                                "(KDA_NO_ALLOC_MAX_SEQS); use kda_fwd with a caller workspace");
            return KDA_ERR_UNSUPPORTED;
        }
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int dev = -1, cur = -1;
    cudaError_t e = cudaStreamGetDevice(s, &dev);
    if (e == cudaSuccess) e = cudaGetDevice(&cur);
    if (e == cudaSuccess && dev != cur) {
        // kda_fwd launches on the current device and picks its schedule from it
        kda::set_last_error("kda_fwd_no_alloc: the stream belongs to another device than the current one");
        return KDA_ERR_INVALID_ARG;
    }
    if (e == cudaSuccess && (dev < 0 || dev >= kMaxDevices)) e = cudaErrorInvalidDevice;
    void* ws = nullptr;
    if (e == cudaSuccess) e = workspace_address(dev, &ws);
    if (e != cudaSuccess) {
        kda::set_last_error("kda_fwd_no_alloc: could not resolve the built-in workspace on the stream's device");
        return KDA_ERR_CUDA;
    }
    if (workspace_used) *workspace_used = ws;
    return kda_fwd(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state, final_state,
                   cu_seqlens, ws, kNoAllocBytes, stream);
}
