// csa_topk_select_noalloc: the top-k selection of csa_topk_select for callers
// that cannot allocate device memory -- for example a plugin running inside
// another runtime that owns all of the device's memory and hands this library
// only its input and output buffers, or a latency-critical path where a
// cudaMalloc, which can synchronise the device, is not acceptable.
//
// Instead of a caller-provided workspace, the candidate buffer of the
// two-phase selection lives in a fixed file-scope device array.  Every GPU
// that loads this library holds that array until the process exits.
#include <mutex>

#include "../../include/csa.h"
#include "common.cuh"
#include "kernels.h"

namespace {

// Scratch shared by every call on a device: for rows longer than one CTA's
// capacity, a threshold, a counter and an entry list per row (64 KB a row at
// k = 1024, so 63 rows of the 1M-context decode shape fit in 4 MiB).
static __device__ __align__(256) uint8_t g_topk_scratch[CSA_TOPK_NOALLOC_SCRATCH_BYTES];

constexpr int MAX_DEVICES = 64;
std::mutex g_mu;
void* g_scratch_ptr[MAX_DEVICES] = {};

// Device address of the scratch array on the current device.  In host code
// the symbol g_topk_scratch is only a host-side stand-in, never a device
// address, so it is looked up here once per device, with that device current.
csa_status_t scratch_address(void** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return csa::report(CSA_ERR_CUDA, "cudaGetDevice failed");
    if (dev < 0 || dev >= MAX_DEVICES) return csa::report(CSA_ERR_UNSUPPORTED, "device index out of range");
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_topk_scratch);
        if (e != cudaSuccess || !p)
            return csa::report(CSA_ERR_CUDA, "cudaGetSymbolAddress of the top-k scratch array failed");
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return CSA_OK;
}

}  // namespace

extern "C" csa_status_t csa_topk_select_noalloc(int B, int n_q, int64_t q_pos0, int m, int N_c, int k,
                                                const float* scores, int32_t* topk, csa_stream_t stream)
{
    if (B < 0 || n_q < 0 || m < 1 || N_c < 0 || q_pos0 < 0) return csa::report(CSA_ERR_INVALID_ARG, "bad sizes");
    if (!csa::topk_supported(N_c, k)) return csa::report(CSA_ERR_UNSUPPORTED, "top-k needs 1 <= k <= 4096, N_c <= 524288");
    const long long rows = (long long)B * n_q;
    if (rows == 0) return CSA_OK;
    if (!csa::topk_rows_ok(rows, N_c, k)) return csa::report(CSA_ERR_UNSUPPORTED, "top-k row count exceeds the grid limit");
    if (!topk || (reinterpret_cast<uintptr_t>(topk) & 15u) ||
        (N_c > 0 && (!scores || (reinterpret_cast<uintptr_t>(scores) & 15u))))
        return csa::report(CSA_ERR_ALIGNMENT, "scores/topk NULL or not 16-byte aligned");
    const size_t need = csa::topk_workspace_bytes(rows, N_c, k);
    if (need > (size_t)CSA_TOPK_NOALLOC_SCRATCH_BYTES)
        return csa::report(CSA_ERR_WORKSPACE,
                           "selection needs more scratch than the built-in 4 MiB array "
                           "(CSA_TOPK_NOALLOC_SCRATCH_BYTES); use csa_topk_select with a workspace");
    void* scratch = nullptr;
    if (need > 0) {
        const csa_status_t st = scratch_address(&scratch);
        if (st != CSA_OK) return st;
    }
    // The per-row counters must start at zero: launch_topk clears them on
    // the stream (one memset) before the long-row kernels use them.
    const cudaError_t e = csa::launch_topk(scores, false, N_c, B, n_q, q_pos0, m, N_c, k, topk, n_q, scratch,
                                           reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return csa::report(CSA_ERR_CUDA, cudaGetErrorString(e));
    return CSA_OK;
}
