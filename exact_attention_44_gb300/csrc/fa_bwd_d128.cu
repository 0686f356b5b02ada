// Specialisations of the attention backward for head dim 128.
#include <atomic>
#include <cstdint>

#include "fa_bwd_kernel.cuh"
#include "fa_launch.h"

namespace fa {

template <typename K>
static cudaError_t set_smem_once(K kernel, int smem, std::atomic<uint64_t>& configured) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(configured.load() & bit)) {
        err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (err != cudaSuccess) return err;
        configured.fetch_or(bit);
    }
    return cudaSuccess;
}

template <bool CAUSAL, bool BF16>
static cudaError_t launch_one(const BwdLaunchArgs& a) {
    using T = BwdTraits<128>;
    auto bwd = fa_bwd_kernel<128, CAUSAL, BF16>;
    static std::atomic<uint64_t> configured{0};
    cudaError_t err;
    if ((err = set_smem_once(bwd, T::FUSED_SMEM_BYTES, configured)) != cudaSuccess) return err;
    // Δ and lse2 per query row; then dK, dV and dQ in one launch.  Each
    // launch is a programmatic dependent of the one before it on the stream:
    // its set-up overlaps that kernel's tail, and it waits for it
    // (griddepcontrol.wait) before touching global memory.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.stream = a.stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(a.pre_grid);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    if ((err = cudaLaunchKernelEx(&cfg, fa_bwd_pre_kernel<128, BF16>, a.params)) != cudaSuccess) return err;
    cfg.gridDim = dim3(a.grid);
    cfg.blockDim = dim3(BWD_THREADS);
    cfg.dynamicSmemBytes = T::FUSED_SMEM_BYTES;
    return cudaLaunchKernelEx(&cfg, bwd, *a.tmK, *a.tmV, *a.tmQ, *a.tmDO, *a.tmDK, *a.tmDV, *a.tmDQ, a.params);
}

cudaError_t launch_bwd_d128(const BwdLaunchArgs& a, bool causal, bool bf16) {
    if (causal) return bf16 ? launch_one<true, true>(a) : launch_one<true, false>(a);
    return bf16 ? launch_one<false, true>(a) : launch_one<false, false>(a);
}

}  // namespace fa
