// sptp_ffn_forward_noalloc: the SP-TP FFN boundary for callers that cannot
// allocate device memory.  Such callers hold only device pointers to their
// inputs and outputs: a plugin running inside a host framework that owns every
// device allocation, or a serving loop that must not call cudaMalloc (it can
// synchronise the device and stall other streams).  Instead of a caller
// workspace, this entry point uses one scratch array that the library
// declares itself and that every GPU loading the library holds until exit.
#include <mutex>

#include "sptp.h"
#include "sptp_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = static_cast<size_t>(SPTP_NOALLOC_SCRATCH_BYTES);

// Scratch of the no-allocation entry point (status words, normed activations
// and SwiGLU output).  Every call shares it and it keeps the last call's
// contents; the forward clears its status words itself when it starts.
__device__ __align__(256) unsigned char g_noalloc_scratch[kStaticScratchBytes];

// Device address of g_noalloc_scratch on each device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device, with that device current.
int scratch_address(void** out) {
    static std::mutex mu;
    static void* addr[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SPTP_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return SPTP_ERR_CUDA;
        addr[dev] = p;
    }
    *out = addr[dev];
    return SPTP_OK;
}

}  // namespace

extern "C" int sptp_ffn_forward_noalloc(const void* x, const void* partials, const void* gamma, const void* W1g,
                                        const void* W1u, const void* W2, int M, int d, int F, int P, int chunks,
                                        float eps, int dtype, void* out, void* resid_out, void* cuda_stream) {
    const size_t need = sptp_ffn_workspace_size(M, d, F, P, chunks, dtype);
    if (need == 0) {
        // Invalid sizes: let the workspace entry point report the same error
        // code.  It rejects these arguments before it touches the workspace
        // or makes any CUDA call, so a host placeholder stands in for it.
        alignas(256) static unsigned char placeholder[256];
        return sptp_ffn_forward(x, partials, gamma, W1g, W1u, W2, M, d, F, P, chunks, eps, dtype, out, resid_out,
                                placeholder, 0, cuda_stream);
    }
    if (need > kStaticScratchBytes) return SPTP_ERR_TOO_LARGE;
    void* scratch = nullptr;
    const int rc = scratch_address(&scratch);
    if (rc != SPTP_OK) return rc;
    return sptp_ffn_forward(x, partials, gamma, W1g, W1u, W2, M, d, F, P, chunks, eps, dtype, out, resid_out,
                            scratch, kStaticScratchBytes, cuda_stream);
}
