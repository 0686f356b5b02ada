// fa_fwd_splitkv_noalloc: the split-KV forward with its workspace in a fixed
// device array of this library instead of caller memory, for callers that
// must not allocate device memory during a call.
//
// The array is a file-scope __device__ variable of this translation unit, so
// it is part of the library's device image: it takes device memory in every
// CUDA context that loads that image (under lazy module loading, the default,
// the first time this entry point runs in the context; with
// CUDA_MODULE_LOADING=EAGER, when the context is created) and keeps it until
// the context is destroyed.  Host code cannot use the name of a __device__
// variable as a device address (on the host it names a stand-in object), so
// the address is asked of the runtime with the device current, on the first
// call in each CUDA context, and passed to the kernels as an ordinary
// pointer.  A context that cudaDeviceReset destroyed and the runtime created
// again has a new ID and gets a fresh lookup; a failed lookup is not
// remembered.
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <mutex>

#include "fa.h"
#include "fa_launch.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

struct ScratchSlot {
    std::mutex mu;
    uint64_t ctx = 0;    // context the address was looked up in
    void* ptr = nullptr;
};
ScratchSlot g_slots[kMaxDevices];

// Device address of the array in the current context of device `dev` (the
// caller has made `dev` current).
cudaError_t scratch_address(int dev, void** out) {
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    ScratchSlot& s = g_slots[dev];
    std::lock_guard<std::mutex> lock(s.mu);
    const uint64_t ctx = fa::current_context_id();
    if (ctx == 0 || ctx != s.ctx || s.ptr == nullptr) {
        void* p = nullptr;
        const cudaError_t err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (err != cudaSuccess) return err;  // not remembered: the next call tries again
        s.ptr = p;
        s.ctx = fa::current_context_id();    // the lookup may have created the context
    }
    *out = s.ptr;
    return cudaSuccess;
}

}  // namespace

extern "C" fa_status fa_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int Z,
                                            int Hq, int Hkv, int Nq, int Nkv, int D, const fa_strides* sq,
                                            const fa_strides* sk, const fa_strides* sv, const fa_strides* so,
                                            float scale, int causal, fa_dtype dtype, cudaStream_t stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
    void* scratch = nullptr;
    if (scratch_address(dev, &scratch) != cudaSuccess || scratch == nullptr) return FA_ERR_CUDA;
    // fa_fwd_splitkv rejects, with FA_ERR_WORKSPACE, a device that needs more
    // than the array holds; nothing in the array has to start at zero, since
    // every partial result the merge reads is written earlier in the same call
    return fa_fwd_splitkv(q, k, v, o, lse, Z, Hq, Hkv, Nq, Nkv, D, sq, sk, sv, so, scale, causal, dtype, scratch,
                          (size_t)FA_NOALLOC_SCRATCH_BYTES, stream);
}
