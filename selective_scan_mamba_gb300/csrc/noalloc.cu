// noalloc.cu -- ssd_chunk_scan_fwd_noalloc: the chunked SSD scan with its scratch held
// in a fixed device array owned by the library, for callers that cannot allocate
// device memory themselves.
//
// The scratch lives in one file-scope __device__ array of kSsdNoallocScratchBytes.
// Every GPU that loads the library holds that array until the process exits.  Host
// code must not pass the array's symbol to a kernel (on the host it only names a
// stand-in, not device memory); instead, the first call on each device looks up the
// array's device address with cudaGetSymbolAddress while that device is current, and
// later calls on the same device reuse it.  That first call should therefore come
// before any stream capture.  The address belongs to the CUDA context it was looked up
// in: the cache remembers that context, and a call made under another one (after
// cudaDeviceReset, say, which destroys the primary context and unloads the module) looks
// the address up again instead of writing through a stale pointer.
//
// All calls share the one array: calls whose GPU work overlaps (several streams, or
// several host threads) race on it and must be ordered by the caller.  The array keeps
// whatever the last call left there; nothing in it needs to start at zero, because the
// chunk-state pass writes every element it later reads.
#include <cuda.h>
#include <cuda_runtime.h>
#include <mutex>
#include <stdio.h>

#include "launch.h"
#include "ssmscan.h"

namespace {

constexpr size_t kSsdNoallocScratchBytes = SSM_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_ssd_scratch[kSsdNoallocScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {nullptr};
CUcontext g_scratch_ctx[kMaxDevices] = {nullptr};  // context each cached address belongs to

thread_local char g_noalloc_err[320] = "";

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

// The current CUDA context, through the runtime's driver entry point (the library has no
// link-time dependency on libcuda).
cudaError_t current_context(CUcontext* ctx) {
    static CtxGetCurrentFn fn = nullptr;  // guarded by g_mu
    if (fn == nullptr) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000,
                                                         cudaEnableDefault, &q);
        if (e != cudaSuccess) return e;
        if (q != cudaDriverEntryPointSuccess || f == nullptr) return cudaErrorNotSupported;
        fn = reinterpret_cast<CtxGetCurrentFn>(f);
    }
    return fn(ctx) == CUDA_SUCCESS ? cudaSuccess : cudaErrorDeviceUninitialized;
}

// Device address of the scratch array on the current device, looked up once per device
// and context.
cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    CUcontext ctx = nullptr;
    if (g_scratch_addr[dev] != nullptr) {
        e = current_context(&ctx);
        if (e != cudaSuccess) return e;
    }
    if (g_scratch_addr[dev] == nullptr || ctx != g_scratch_ctx[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_ssd_scratch);  // initialises the context if needed
        if (e != cudaSuccess) return e;
        if ((e = current_context(&ctx)) != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
        g_scratch_ctx[dev] = ctx;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" {

size_t ssd_noalloc_scratch_capacity(void) { return kSsdNoallocScratchBytes; }

ssm_status ssd_chunk_scan_fwd_noalloc(const ssd_params* p, void* stream) {
    // Shapes and pointers are checked by the regular entry point's size query first.
    const size_t need = ssd_chunk_scan_workspace_size(p);
    if (p == nullptr) return ssd_chunk_scan_fwd(p, nullptr, 0, stream);  // reports the error
    if (need == 0 && p->seqlen > 0) return ssd_chunk_scan_fwd(p, nullptr, 0, stream);
    if (need > kSsdNoallocScratchBytes) {
        snprintf(g_noalloc_err, sizeof(g_noalloc_err),
                 "ssd_chunk_scan_fwd_noalloc: this problem needs %zu bytes of scratch, more than "
                 "the library's fixed %zu-byte array; use ssd_chunk_scan_fwd with a caller "
                 "workspace",
                 need, kSsdNoallocScratchBytes);
        return ssm::set_error(SSM_ERR_INVALID_ARG, g_noalloc_err);
    }
    // the scratch size above was computed for the current device: the stream must be one
    // of its streams
    int cur = 0, sdev = 0;
    cudaError_t e = cudaGetDevice(&cur);
    if (e == cudaSuccess) e = cudaStreamGetDevice(static_cast<cudaStream_t>(stream), &sdev);
    if (e != cudaSuccess) {
        snprintf(g_noalloc_err, sizeof(g_noalloc_err),
                 "ssd_chunk_scan_fwd_noalloc: cannot query the stream's device: %s",
                 cudaGetErrorString(e));
        return ssm::set_error(SSM_ERR_CUDA, g_noalloc_err);
    }
    if (sdev != cur) {
        snprintf(g_noalloc_err, sizeof(g_noalloc_err),
                 "ssd_chunk_scan_fwd_noalloc: the stream belongs to device %d, but device %d is "
                 "current (make the stream's device current first)",
                 sdev, cur);
        return ssm::set_error(SSM_ERR_INVALID_ARG, g_noalloc_err);
    }
    void* ws = nullptr;
    e = scratch_address(&ws);
    if (e != cudaSuccess) {
        snprintf(g_noalloc_err, sizeof(g_noalloc_err),
                 "ssd_chunk_scan_fwd_noalloc: cudaGetSymbolAddress failed: %s",
                 cudaGetErrorString(e));
        return ssm::set_error(SSM_ERR_CUDA, g_noalloc_err);
    }
    return ssd_chunk_scan_fwd(p, ws, kSsdNoallocScratchBytes, stream);
}

}  // extern "C"
