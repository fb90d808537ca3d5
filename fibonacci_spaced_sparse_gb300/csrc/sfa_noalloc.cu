// sfa_noalloc.cu -- sfa_forward_noalloc: the forward for callers that must not
// allocate device memory themselves.
//
// Some callers cannot hand the library a workspace: code that runs where no
// allocator is reachable (a plugin inside a host application that owns all
// device memory, a fixed-footprint real-time service, a tool that may only use
// memory reserved up front).  For them this entry point keeps the forward's
// scratch -- the rotated keys of the bf16 path -- in a fixed array that is part
// of the library image, so the call itself allocates nothing.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds its 8 MiB until the process exits.  In host code its name is
// only a host-side handle.  Its device address belongs to one CUDA context:
// it is looked up with cudaGetSymbolAddress in the context current at the
// call and cached under that context's key (sfa::context_key), so a caller
// that switches to a context of its own (cuCtxCreate) gets the address that
// is valid in the context it calls from.
#include <mutex>

#include "sfa.h"
#include "sfa_internal.cuh"

namespace {

constexpr size_t kScratchBytes = size_t(8) << 20;  // 8 MiB

__device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
struct ScratchAddr {
    unsigned long long key;  // context the address was looked up in (0: none yet)
    void* addr;
};
ScratchAddr g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of g_scratch in the context current on this thread.
sfa_status scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return SFA_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return SFA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    ScratchAddr& slot = g_scratch_addr[dev];
    const unsigned long long key = sfa::context_key();
    if (key == 0 || slot.key != key) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) {
            (void)cudaGetLastError();
            return SFA_ERR_CUDA;
        }
        // the lookup makes the runtime's context current if none was
        slot.key = sfa::context_key();
        slot.addr = p;
    }
    *out = slot.addr;
    return SFA_OK;
}

}  // namespace

extern "C" {

SFA_API size_t sfa_forward_noalloc_scratch_bytes(void) { return kScratchBytes; }

SFA_API sfa_status sfa_forward_noalloc(const sfa_params* p, const void* Q, const void* K, const void* V,
                                       const float* rope_table, void* O, float* lse,
                                       unsigned int* status, cudaStream_t stream) {
    const size_t need = sfa_forward_workspace_size(p);  // 0 also for invalid arguments
    if (need > kScratchBytes) return SFA_ERR_UNSUPPORTED;
    void* ws = nullptr;
    size_t ws_bytes = 0;
    if (need > 0) {
        const sfa_status st = scratch_address(&ws);
        if (st != SFA_OK) return st;
        ws_bytes = kScratchBytes;
    }
    return sfa_forward(p, Q, K, V, rope_table, O, lse, ws, ws_bytes, status, stream);
}

}  // extern "C"
