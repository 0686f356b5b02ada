// Specialisations of the attention backward for head dim 16.
#include <atomic>
#include <cstdint>

#include "fa_bwd_kernel.cuh"
#include "fa_launch.h"

namespace fa {

template <bool CAUSAL, bool BF16>
static cudaError_t launch_one(const BwdLaunchArgs& a) {
    auto kernel = fa_bwd_kernel<16, CAUSAL, BF16>;
    constexpr int smem = BwdTraits<16>::SMEM_BYTES;
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
    // Δ and lse2 per query row, zeroed dQ accumulator; then the gradients; then dQ
    fa_bwd_pre_kernel<16, BF16><<<a.pre_grid, 256, 0, a.stream>>>(a.params);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    kernel<<<a.grid, BWD_THREADS, smem, a.stream>>>(*a.tmK, *a.tmV, *a.tmQ, *a.tmDO, a.params);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    fa_bwd_dq_kernel<16, BF16><<<a.post_grid, 256, 0, a.stream>>>(a.params);
    return cudaGetLastError();
}

cudaError_t launch_bwd_d16(const BwdLaunchArgs& a, bool causal, bool bf16) {
    if (causal) return bf16 ? launch_one<true, true>(a) : launch_one<true, false>(a);
    return bf16 ? launch_one<false, true>(a) : launch_one<false, false>(a);
}

}  // namespace fa
