// sptp_ffn_forward_noalloc: the SP-TP FFN boundary for callers that cannot
// allocate device memory.  Such callers hold only device pointers to their
// inputs and outputs: a plugin running inside a host framework that owns every
// device allocation, or a serving loop that must not call cudaMalloc (it can
// synchronise the device and stall other streams).  Instead of a caller
// workspace, this entry point uses one scratch array that the library
// declares itself and that every GPU loading the library holds until exit.
#include <cudaTypedefs.h>

#include <mutex>

#include "sptp.h"
#include "sptp_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = static_cast<size_t>(SPTP_NOALLOC_SCRATCH_BYTES);

// Scratch of the no-allocation entry point (status words, normed activations
// and SwiGLU output).  Every call shares it and it keeps the last call's
// contents; the forward clears its status words itself when it starts.
__device__ __align__(256) unsigned char g_noalloc_scratch[kStaticScratchBytes];

// Identity of the current context: the device address of a __device__
// variable belongs to the context that loaded the module, and a reset device
// gets a new context (with a new id) in which the module is loaded again.
bool current_context_id(unsigned long long* id) {
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
    });
    CUcontext ctx = nullptr;
    if (get_current == nullptr || get_id == nullptr || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr)
        return false;
    return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of g_noalloc_scratch in the current context.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// with cudaGetSymbolAddress, once per device and context, with that device
// current (the runtime makes the device's context current on first use).
int scratch_address(void** out) {
    static std::mutex mu;
    static void* addr[64] = {};
    static unsigned long long ctx_of[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return SPTP_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(mu);
    unsigned long long ctx = 0;
    const bool have_ctx = current_context_id(&ctx);
    if (addr[dev] == nullptr || !have_ctx || ctx_of[dev] != ctx) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();  // leave no error pending for the caller's next runtime call
            addr[dev] = nullptr;
            return SPTP_ERR_CUDA;
        }
        // the context exists now (the lookup created it if it had not)
        if (!have_ctx && !current_context_id(&ctx)) ctx = 0;
        addr[dev] = p;
        ctx_of[dev] = ctx;
    }
    *out = addr[dev];
    return SPTP_OK;
}

// Any 256-byte aligned non-null address that is neither a device pointer nor
// dereferenced: it stands for the scratch array while the arguments are
// checked (the checks make no CUDA call and touch no memory).
alignas(256) unsigned char g_placeholder[256];

}  // namespace

extern "C" int sptp_ffn_forward_noalloc(const void* x, const void* partials, const void* gamma, const void* W1g,
                                        const void* W1u, const void* W2, int M, int d, int F, int P, int chunks,
                                        float eps, sptp_dtype dtype, void* out, void* resid_out,
                                        void* cuda_stream) {
    // 1. the arguments, checked as sptp_ffn_forward checks them, before the
    //    size limit and before any CUDA call (so the codes are the same)
    const size_t need = sptp_ffn_workspace_size(M, d, F, P, chunks, dtype);
    int rc = sptp::check_ffn_forward_args(x, partials, gamma, W1g, W1u, W2, M, d, F, P, chunks, eps, dtype, out,
                                          resid_out, g_placeholder, need, SPTP_VARIANT_AUTO);
    if (rc != SPTP_OK) return rc;
    // 2. the static array's limit
    if (need > kStaticScratchBytes) return SPTP_ERR_TOO_LARGE;
    if (M == 0) return SPTP_OK;
    // 3. the device, then the array's address on it
    if ((rc = sptp::current_device_ok()) != SPTP_OK) return rc;
    void* scratch = nullptr;
    if ((rc = scratch_address(&scratch)) != SPTP_OK) return rc;
    return sptp_ffn_forward(x, partials, gamma, W1g, W1u, W2, M, d, F, P, chunks, eps, dtype, out, resid_out,
                            scratch, kStaticScratchBytes, cuda_stream);
}

extern "C" int sptp_noalloc_read_device_status(void* cuda_stream) {
    int rc = sptp::current_device_ok();
    if (rc != SPTP_OK) return rc;
    void* scratch = nullptr;
    if ((rc = scratch_address(&scratch)) != SPTP_OK) return rc;
    return sptp_read_device_status(scratch, cuda_stream);
}

extern "C" int sptp_noalloc_wait_selftest(unsigned long long limit_ns, int preset_flag, void* cuda_stream) {
    int rc = sptp::current_device_ok();
    if (rc != SPTP_OK) return rc;
    void* scratch = nullptr;
    if ((rc = scratch_address(&scratch)) != SPTP_OK) return rc;
    return sptp_wait_selftest(scratch, kStaticScratchBytes, limit_ns, preset_flag, cuda_stream);
}
