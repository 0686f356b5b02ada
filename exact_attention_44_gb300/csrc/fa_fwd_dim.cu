// Specialisations of the attention forward kernel for one head dim, D =
// FA_HEAD_DIM (the build compiles this file once per supported D, in parallel:
// "把 FlashAttention 搬上昇腾：Triton-Ascend CV Pipeline 优化实战", section 七,
// specialises the kernel per head dim the same way).
#ifndef FA_HEAD_DIM
#error "compile with -DFA_HEAD_DIM=<16|32|64|128|256>"
#endif
#include <cstdint>

#include "fa_fwd_kernel.cuh"
#include "fa_fwd_chain_kernel.cuh"
#if FA_HEAD_DIM == 128
#include "fa_fwd_pair_kernel.cuh"
#endif
#include "fa_launch.h"

namespace fa {

template <bool CAUSAL, bool BF16, int VAR>
static cudaError_t launch_one(const LaunchArgs& a) {
    constexpr int D = FA_HEAD_DIM;
    auto kernel = fa_fwd_kernel<D, CAUSAL, BF16, VAR>;
    constexpr int smem = Traits<D>::SMEM_BYTES;
    static std::atomic<uint64_t> configured{0};  // context the opt-in shared memory size was set in
    cudaError_t err = set_smem_for_context(kernel, smem, configured);
    if (err != cudaSuccess) return err;
    // programmatic dependent launch: the kernel's set-up may overlap the tail
    // of the previous kernel on the stream (it waits for it before any
    // global memory access)
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.grid);
    cfg.blockDim = dim3(Traits<D>::THREADS);
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
            err = cudaLaunchKernelEx(&mcfg, fa_split_merge_kernel<D, CAUSAL, BF16>, a.params, a.grid);
        }
    }
    return err;
}

// variant 0: fa_fwd; 1: window / variable length; 2: the same with ALiBi;
// 4: fa_fwd with alternating causal rounds (tile mode)
#define FA_CAT2(a, b) a##b
#define FA_CAT(a, b) FA_CAT2(a, b)
cudaError_t FA_CAT(launch_d, FA_HEAD_DIM)(const LaunchArgs& a, bool causal, bool bf16, int variant) {
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


#if FA_HEAD_DIM <= 128
// The two-softmax-chain kernel (fa_fwd, whole tiles, head dims up to 128).
template <bool CAUSAL, bool BF16, bool ALT>
static cudaError_t launch_chain_one(const LaunchArgs& a) {
    constexpr int D = FA_HEAD_DIM;
    auto kernel = fa_fwd_chain_kernel<D, CAUSAL, BF16, ALT>;
    constexpr int smem = Traits<D>::SMEM_BYTES;
    static std::atomic<uint64_t> configured{0};  // context the opt-in shared memory size was set in
    cudaError_t err = set_smem_for_context(kernel, smem, configured);
    if (err != cudaSuccess) return err;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.grid);
    cfg.blockDim = dim3(CHAIN_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = a.stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, *a.tmQ, *a.tmK, *a.tmV, *a.tmO, a.params);
}

cudaError_t FA_CAT(launch_chain_d, FA_HEAD_DIM)(const LaunchArgs& a, bool causal, bool bf16, bool alt) {
    if (causal) {
        if (alt) return bf16 ? launch_chain_one<true, true, true>(a) : launch_chain_one<true, false, true>(a);
        return bf16 ? launch_chain_one<true, true, false>(a) : launch_chain_one<true, false, false>(a);
    }
    return bf16 ? launch_chain_one<false, true, false>(a) : launch_chain_one<false, false, false>(a);
}
#endif

#if FA_HEAD_DIM == 128
// The CTA-pair kernel (fa_fwd, whole tiles, D = 128): clusters of two CTAs,
// a.grid = 2 x clusters.
template <bool CAUSAL, bool BF16, bool ALT>
static cudaError_t launch_pair_one(const LaunchArgs& a) {
    constexpr int D = FA_HEAD_DIM;
    auto kernel = fa_fwd_pair_kernel<D, CAUSAL, BF16, ALT>;
    constexpr int smem = PairTraits<D>::SMEM_BYTES;
    static std::atomic<uint64_t> configured{0};
    cudaError_t err = set_smem_for_context(kernel, smem, configured);
    if (err != cudaSuccess) return err;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.grid);
    cfg.blockDim = dim3(CHAIN_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = a.stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, *a.tmQ, *a.tmK, *a.tmV, *a.tmO, a.params);
}

cudaError_t launch_pair_d128(const LaunchArgs& a, bool causal, bool bf16, bool alt) {
    if (causal) {
        if (alt) return bf16 ? launch_pair_one<true, true, true>(a) : launch_pair_one<true, false, true>(a);
        return bf16 ? launch_pair_one<true, true, false>(a) : launch_pair_one<true, false, false>(a);
    }
    return bf16 ? launch_pair_one<false, true, false>(a) : launch_pair_one<false, false, false>(a);
}

// Clusters of the pair kernel that can be resident at once on the current
// device (pairs of SMs in one GPC); every instantiation has the same
// resources.  Asked once per context; 0 when the query fails.
int pair_cluster_limit_d128() {
    static std::atomic<uint64_t> ctx{0};
    static std::atomic<int> limit{0};
    const uint64_t id = current_context_id();
    if (id != 0 && ctx.load() == id) return limit.load();
    auto kernel = fa_fwd_pair_kernel<FA_HEAD_DIM, false, true, false>;
    constexpr int smem = PairTraits<FA_HEAD_DIM>::SMEM_BYTES;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(CHAIN_THREADS);
    cfg.dynamicSmemBytes = smem;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) return 0;
    limit.store(n);
    if (id != 0) ctx.store(id);
    return n;
}
#endif

}  // namespace fa
