// Greedy acceptance for callers that cannot allocate device memory.
//
// sd_accept_greedy needs a caller-provided workspace.  Some hosts cannot give
// one: they hand every byte of device memory to their own pool allocator and
// forbid extensions from calling cudaMalloc (it synchronises the device and
// goes around the pool), or they only have the input and output buffers at
// hand when the call is made.  This entry point serves them from scratch
// memory the library itself owns: a file-scope __device__ array of fixed size,
// which every GPU that loads the library holds until the process exits.
//
// The array is a host-side symbol here, not a device address, so host code
// asks the runtime for its device address once per device (the first call on
// that device does this, under a lock) and passes that address down.  Nothing
// on this path allocates: no cudaMalloc, no cudaFree, no allocating library
// routine.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = 1u << 20;  // 1 MiB
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_greedy_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kNoAllocMaxDevices] = {};

}  // namespace

extern "C" sd_status sd_accept_greedy_noalloc(const int32_t *draft_ids, const void *target_logits, int B, int T,
                                              int V, sd_dtype dtype, int32_t *n_accepted, int32_t *correction_id,
                                              void *stream) {
    const size_t need = sd_accept_greedy_workspace_size(B, T, V, dtype);
    if (need == 0) return sdv::report_error(SD_ERR_INVALID_ARG, "need B >= 1, T in [1, 16], V >= 1");
    if (need > kNoAllocScratchBytes)
        return sdv::report_error(SD_ERR_WORKSPACE,
                                 "this shape needs more scratch than the 1 MiB the no-allocation entry point owns; "
                                 "use sd_accept_greedy with a caller workspace");
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return sdv::report_error(SD_ERR_CUDA, "cudaGetDevice failed");
    if (dev < 0 || dev >= kNoAllocMaxDevices) return sdv::report_error(SD_ERR_UNSUPPORTED, "device index out of range");
    void *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_noalloc_mu);
        if (!g_noalloc_ptr[dev]) {
            void *p = nullptr;
            e = cudaGetSymbolAddress(&p, g_noalloc_greedy_scratch);
            if (e != cudaSuccess || !p)
                return sdv::report_error(SD_ERR_CUDA, "cudaGetSymbolAddress of the no-allocation scratch failed");
            g_noalloc_ptr[dev] = p;
        }
        scratch = g_noalloc_ptr[dev];
    }
    // the scratch keeps whatever the previous call left; its ticket counters
    // must start at zero, so the part this call uses is cleared first, in order
    // on the caller's stream
    e = cudaMemsetAsync(scratch, 0, need, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return sdv::report_error(SD_ERR_CUDA, "clearing the no-allocation scratch failed");
    return sd_accept_greedy(draft_ids, target_logits, B, T, V, dtype, n_accepted, correction_id, scratch,
                            kNoAllocScratchBytes, stream);
}
