// Specialisations of the attention backward for one head dim, D =
// FA_HEAD_DIM (compiled once per supported D, in parallel).
#ifndef FA_HEAD_DIM
#error "compile with -DFA_HEAD_DIM=<16|32|64|128|256>"
#endif
#include <cstdint>

#if FA_HEAD_DIM == 256
#include "fa_bwd_wide_kernel.cuh"
#else
#include "fa_bwd_kernel.cuh"
#endif
#include "fa_launch.h"

namespace fa {

template <bool CAUSAL, bool BF16, int VAR>
static cudaError_t launch_one(const BwdLaunchArgs& a) {
    constexpr int D = FA_HEAD_DIM;
#if FA_HEAD_DIM == 256
    auto bwd = fa_bwd_wide_kernel<CAUSAL, BF16, VAR>;
    constexpr int SMEM = WideTraits::SMEM_BYTES, THREADS = WIDE_THREADS;
#else
    auto bwd = fa_bwd_kernel<D, CAUSAL, BF16, VAR>;
    constexpr int SMEM = BwdTraits<D>::FUSED_SMEM_BYTES, THREADS = BwdWarps<D>::THREADS;
#endif
    static std::atomic<uint64_t> configured{0};  // context the opt-in shared memory size was set in
    cudaError_t err;
    if ((err = set_smem_for_context(bwd, SMEM, configured)) != cudaSuccess) return err;
#if FA_HEAD_DIM != 256
    if constexpr (BwdWarps<D>::SPLIT_REGS) {
        // the warpgroups' setmaxnreg budgets add up only at this launch size
        static std::atomic<int> regs{0};
        if (regs.load() == 0) {
            cudaFuncAttributes attr;
            if ((err = cudaFuncGetAttributes(&attr, bwd)) != cudaSuccess) return err;
            regs.store(attr.numRegs);
        }
        if (regs.load() != (int)BwdWarps<D>::REG_LAUNCH) return cudaErrorInvalidConfiguration;
    }
#endif
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
    if ((err = cudaLaunchKernelEx(&cfg, fa_bwd_pre_kernel<D, BF16>, a.params)) != cudaSuccess) return err;
    cfg.gridDim = dim3(a.grid);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = SMEM;
    return cudaLaunchKernelEx(&cfg, bwd, *a.tmK, *a.tmV, *a.tmQ, *a.tmDO, *a.tmDK, *a.tmDV, *a.tmDQ, a.params);
}

#define FA_CAT2(a, b) a##b
#define FA_CAT(a, b) FA_CAT2(a, b)
// variant 0: fa_bwd; 1: window (fa_bwd_ex); 2: window and ALiBi; 3: packed
// variable-length sequences with a window and ALiBi; 4: packed sequences with
// a window
cudaError_t FA_CAT(launch_bwd_d, FA_HEAD_DIM)(const BwdLaunchArgs& a, bool causal, bool bf16, int variant) {
    if (variant == 4) {
        if (causal) return bf16 ? launch_one<true, true, 4>(a) : launch_one<true, false, 4>(a);
        return bf16 ? launch_one<false, true, 4>(a) : launch_one<false, false, 4>(a);
    }
    if (variant == 3) {
        if (causal) return bf16 ? launch_one<true, true, 3>(a) : launch_one<true, false, 3>(a);
        return bf16 ? launch_one<false, true, 3>(a) : launch_one<false, false, 3>(a);
    }
    if (variant == 2) {
        if (causal) return bf16 ? launch_one<true, true, 2>(a) : launch_one<true, false, 2>(a);
        return bf16 ? launch_one<false, true, 2>(a) : launch_one<false, false, 2>(a);
    }
    if (variant == 1) {
        if (causal) return bf16 ? launch_one<true, true, 1>(a) : launch_one<true, false, 1>(a);
        return bf16 ? launch_one<false, true, 1>(a) : launch_one<false, false, 1>(a);
    }
    if (causal) return bf16 ? launch_one<true, true, 0>(a) : launch_one<true, false, 0>(a);
    return bf16 ? launch_one<false, true, 0>(a) : launch_one<false, false, 0>(a);
}

}  // namespace fa
