// fa_noalloc.cu -- fa_fwd_noalloc: the forward for callers that cannot
// allocate device memory.
//
// fa_fwd takes a caller-allocated workspace (status words that the kernel
// flags when one of its bounded waits runs out of time, and the counters of
// its work queue).  Some callers cannot provide one: code running inside a
// memory allocator's own hooks, code in a process whose device memory is all
// handed out by a framework that forbids side allocations, or a path that
// must not call cudaMalloc because it may synchronise the device.  For them
// this file keeps that scratch in a file-scope __device__ array, which every
// GPU that loads the library holds until the process exits, and hands its
// device address to the same kernels.
#include <cstdio>
#include <mutex>

#include <cudaTypedefs.h>

#include "fa_internal.h"
#include "ptx.cuh"

namespace {

// Stated maximum of the static scratch: 4 KiB per device.
constexpr size_t kNoAllocScratchBytes = 4096;
static __device__ __align__(256) uint32_t g_noalloc_scratch[kNoAllocScratchBytes / sizeof(uint32_t)];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
struct ScratchSlot {
    void* ptr;                 // device address of g_noalloc_scratch in that context
    unsigned long long ctx;    // the context it was looked up in (cuCtxGetId)
};
ScratchSlot g_slot[kMaxDevices] = {};

// The unique id of the calling thread's current context, through the
// runtime's driver entry points (no link against libcuda).  0 if the driver
// does not offer it; the address is then looked up on every call.
unsigned long long current_context_id() {
    static PFN_cuCtxGetCurrent_v4000 get_cur = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_cur = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    });
    if (!get_cur || !get_id) return 0;
    CUcontext c = nullptr;
    unsigned long long id = 0;
    if (get_cur(&c) != CUDA_SUCCESS || !c || get_id(c, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// The device address of g_noalloc_scratch on the current device.  In host
// code the array's name is only a host-side stand-in, so the address is
// looked up with the device current: once per device and context (a
// cudaDeviceReset gives the device a new context, and the array a new
// address, so the lookup is repeated then).
fa_status scratch_for_current_device(void** out) {
    char msg[256];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        snprintf(msg, sizeof(msg), "cudaGetDevice: %s", cudaGetErrorString(e));
        return fa::report(FA_ERR_CUDA, msg);
    }
    if (dev < 0 || dev >= kMaxDevices) {
        snprintf(msg, sizeof(msg), "device %d is beyond the %d devices the static scratch serves", dev, kMaxDevices);
        return fa::report(FA_ERR_UNSUPPORTED, msg);
    }
    std::lock_guard<std::mutex> lock(g_mu);
    // cudaGetDevice does not create the context; the symbol lookup does, so
    // the context id is read after it when the slot is empty.
    const unsigned long long ctx = current_context_id();
    ScratchSlot& s = g_slot[dev];
    if (!s.ptr || ctx == 0 || s.ctx != ctx) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            snprintf(msg, sizeof(msg), "cudaGetSymbolAddress of the static scratch: %s", cudaGetErrorString(e));
            return fa::report(FA_ERR_CUDA, msg);
        }
        s.ptr = p;
        s.ctx = current_context_id();
    }
    *out = s.ptr;
    return FA_OK;
}

}  // namespace

extern "C" fa_status fa_fwd_noalloc(const fa_fwd_args* a, const fa_block_mask* bm, const fa_score_desc* sc,
                                    void* stream) {
    const size_t need = fa_workspace_bytes();
    if (need > kNoAllocScratchBytes) {
        char msg[160];
        snprintf(msg, sizeof(msg), "the forward needs %zu bytes of scratch, more than the %zu-byte static maximum",
                 need, kNoAllocScratchBytes);
        return fa::report(FA_ERR_UNSUPPORTED, msg);
    }
    void* scratch = nullptr;
    fa_status st = scratch_for_current_device(&scratch);
    if (st != FA_OK) return st;
    // A rejected call must touch nothing: the arguments are checked before
    // the shared array is cleared (a clear could reset the work queue of a
    // call still running on another stream).
    st = fa::fwd_validate(a, bm, sc, scratch);
    if (st != FA_OK) return st;
    // Every call shares the array and it keeps the last call's contents: the
    // status words and the queue counters must start at zero, so clear them
    // on this call's stream.
    cudaError_t e = cudaMemsetAsync(scratch, 0, need, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        char msg[160];
        snprintf(msg, sizeof(msg), "clearing the static scratch: %s", cudaGetErrorString(e));
        return fa::report(FA_ERR_CUDA, msg);
    }
    return fa_fwd(a, bm, sc, scratch, stream);
}
