// Specialisations of the attention forward kernel for head dim 128.
#include <atomic>
#include <cstdint>

#include "fa_fwd_kernel.cuh"
#include "fa_launch.h"

namespace fa {

template <bool CAUSAL, bool BF16, int VAR>
static cudaError_t launch_one(const LaunchArgs& a) {
    auto kernel = fa_fwd_kernel<128, CAUSAL, BF16, VAR>;
    constexpr int smem = Traits<128>::SMEM_BYTES;
    // the opt-in shared memory size is set once per device
    static std::atomic<uint64_t> configured{0};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(configured.load() & bit)) {
        err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (err != cudaSuccess) return err;
        configured.fetch_or(bit);
    }
    // programmatic dependent launch: the kernel's set-up may overlap the tail
    // of the previous kernel on the stream (it waits for it before any
    // global memory access)
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.grid);
    cfg.blockDim = dim3(Traits<128>::THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = a.stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    err = cudaLaunchKernelEx(&cfg, kernel, *a.tmQ, *a.tmK, *a.tmV, *a.tmO, a.params);
    // split schedule: one merge block per cut between CTA ranges, same stream
    if constexpr (VAR == 0) {
        if (err == cudaSuccess && a.params.split && a.grid > 1) {
            cudaLaunchConfig_t mcfg = {};
            mcfg.gridDim = dim3(a.grid - 1);
            mcfg.blockDim = dim3(MERGE_THREADS);
            mcfg.stream = a.stream;
            mcfg.attrs = attr;
            mcfg.numAttrs = 1;
            err = cudaLaunchKernelEx(&mcfg, fa_split_merge_kernel<128, CAUSAL, BF16>, a.params, a.grid);
        }
    }
    return err;
}

// variant 0: fa_fwd; 1: window / variable length; 2: the same with ALiBi;
// 4: fa_fwd with alternating causal rounds (tile mode)
cudaError_t launch_d128(const LaunchArgs& a, bool causal, bool bf16, int variant) {
    if (variant == 2) {
        if (causal) return bf16 ? launch_one<true, true, 2>(a) : launch_one<true, false, 2>(a);
        return bf16 ? launch_one<false, true, 2>(a) : launch_one<false, false, 2>(a);
    }
    if (variant == 1) {
        if (causal) return bf16 ? launch_one<true, true, 1>(a) : launch_one<true, false, 1>(a);
        return bf16 ? launch_one<false, true, 1>(a) : launch_one<false, false, 1>(a);
    }
    if (variant == 4 && causal) return bf16 ? launch_one<true, true, 4>(a) : launch_one<true, false, 4>(a);
    if (causal) return bf16 ? launch_one<true, true, 0>(a) : launch_one<true, false, 0>(a);
    return bf16 ? launch_one<false, true, 0>(a) : launch_one<false, false, 0>(a);
}

}  // namespace fa
