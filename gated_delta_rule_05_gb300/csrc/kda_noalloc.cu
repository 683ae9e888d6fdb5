// kda_noalloc.cu -- kda_prefill_noalloc: the prefill entry point for callers
// that cannot allocate device memory.
//
// kda_prefill needs a small device workspace (the varlen work list and its
// status words) that the caller allocates.  Some callers cannot do that: an
// inference engine that plans all of its device memory once at start-up and
// forbids allocation afterwards, or a plugin host that hands a library only
// the input and output buffers of an operation.  For them this entry point
// takes the same arguments minus the workspace and uses a fixed scratch array
// that lives in the library's own device image instead.
//
// Facts a caller must know:
//   * The scratch is a file-scope __device__ array of kNoAllocScratchBytes
//     (about 16 KiB), enough for kNoAllocMaxSeqs sequences.  Every GPU that
//     loads the library holds one copy of it until the process exits.
//   * Host code cannot use the array's name as a device address.  The first
//     call on each device, with that device current, looks its address up
//     with cudaGetSymbolAddress (which may load the library's device code),
//     so make that first call before any stream capture starts.  Later calls
//     on the same device reuse the address while the device's current
//     context is the one it was looked up in; a new context (after
//     cudaDeviceReset, for example) has its own copy of the array, and its
//     address is looked up again.
//   * The status words kda_prefill leaves in its workspace (an invalid
//     cu_seqlens, a wait that gave up) stay in this private array, where
//     the caller cannot read them.
//   * The array has room for the work list only, so the producer / consumer
//     kernel (whose operand ring needs tens of MB) is never selected.
//   * Every call on a device shares the same array.  Calls that may overlap
//     on the GPU (on different streams, or from different host threads
//     without ordering) race on it and must not be issued that way.
//   * The array keeps the last call's contents.  Nothing in it has to start
//     at zero: each call that passes cu_seqlens rewrites the sequence order,
//     work counter and error word before any kernel reads them, and a call
//     without cu_seqlens reads none of it.
//   * Nothing here calls cudaMalloc, cudaFree or any allocating routine.
#include <cuda.h>

#include <mutex>

#include "kda_internal.cuh"

namespace {

constexpr int32_t kNoAllocMaxSeqs = 4096;
constexpr size_t kNoAllocScratchBytes =
    kda::kWsHeaderBytes + (size_t)kNoAllocMaxSeqs * sizeof(int32_t);
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_prefill_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
// Per device: the context the address was looked up in, and the address.
CUcontext g_scratch_ctx[kMaxDevices] = {};
void* g_scratch_addr[kMaxDevices] = {};

// The driver's cuCtxGetCurrent, looked up once through the runtime (the
// library does not link the driver library itself).
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
CtxGetCurrentFn ctx_get_current_fn()
{
    static CtxGetCurrentFn fn = nullptr;
    static bool looked = false;
    if (!looked) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(p);
        looked = true;
    }
    return fn;
}

// Device address of the scratch array in the current device's current
// context; nullptr if the lookup fails.
void* scratch_on_current_device()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    CtxGetCurrentFn get_ctx = ctx_get_current_fn();
    if (get_ctx == nullptr) return nullptr;
    // Before the runtime's first use of the device no context is current yet
    // (ctx stays null); cudaGetSymbolAddress then makes it current.
    CUcontext ctx = nullptr;
    if (get_ctx(&ctx) != CUDA_SUCCESS) return nullptr;
    if (ctx == nullptr || g_scratch_addr[dev] == nullptr || g_scratch_ctx[dev] != ctx) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_prefill_scratch) != cudaSuccess) return nullptr;
        if (get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr) return nullptr;
        g_scratch_addr[dev] = p;
        g_scratch_ctx[dev] = ctx;
    }
    return g_scratch_addr[dev];
}

}  // namespace

extern "C" kda_status_t kda_prefill_noalloc(const void* q, const void* k, const void* v,
                                            const float* log_alpha, const float* beta,
                                            const float* S0, const int32_t* cu_seqlens,
                                            int32_t num_seqs, int64_t total_tokens, int32_t H,
                                            int32_t d_k, int32_t d_v, kda_dtype_t dtype, void* o,
                                            float* S_final, cudaStream_t stream)
{
    if (num_seqs > kNoAllocMaxSeqs) return KDA_ERR_WORKSPACE;   // beyond the fixed scratch
    if (num_seqs < 1) return KDA_ERR_INVALID_ARG;
    void* scratch = scratch_on_current_device();
    if (scratch == nullptr) return KDA_ERR_CUDA;
    return kda_prefill(q, k, v, log_alpha, beta, S0, cu_seqlens, num_seqs, total_tokens, H, d_k,
                       d_v, dtype, o, S_final, scratch, kNoAllocScratchBytes, stream);
}
