// Per-head-dim launchers: fa_fwd_dim.cu and fa_bwd_dim.cu, each compiled once
// per head dim (-DFA_HEAD_DIM=D), in parallel.
#pragma once

#include <cuda.h>
#include <cuda_runtime_api.h>

#include <atomic>
#include <cstdint>

#include "fa_params.h"

namespace fa {

// ID of the calling thread's current CUDA context (cuCtxGetId), or 0 when
// there is none or the driver cannot say.  Per-context state of this library
// (a kernel's shared-memory attribute, the device address of a __device__
// variable) is remembered under this ID: a context destroyed by
// cudaDeviceReset and created again gets a new ID, so that state is set up
// anew instead of reused.
uint64_t current_context_id();

// Set `kernel`'s opt-in dynamic shared memory size, once per CUDA context:
// `ctx` holds the ID of the context it was last set in.  A failed call is not
// remembered (the next launch tries again).
template <typename K>
inline cudaError_t set_smem_for_context(K kernel, int smem, std::atomic<uint64_t>& ctx) {
    const uint64_t id = current_context_id();
    if (id != 0 && ctx.load() == id) return cudaSuccess;
    const cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err == cudaSuccess && id != 0) ctx.store(id);
    return err;
}

struct LaunchArgs {
    const CUtensorMap* tmQ;
    const CUtensorMap* tmK;
    const CUtensorMap* tmV;
    const CUtensorMap* tmO;  // O in 32-row boxes, for the epilogue's tensor stores
    FwdParams params;
    int grid;
    cudaStream_t stream;
};

// Launch fa_fwd_kernel<D, causal, bf16, variant> (variant 0: fa_fwd, 1:
// window / variable length, 2: with ALiBi, 4: fa_fwd with alternating causal
// rounds; and the split merge when the parameters ask for the split
// schedule); returns the launches' error code.
cudaError_t launch_d16(const LaunchArgs& a, bool causal, bool bf16, int variant);
cudaError_t launch_d32(const LaunchArgs& a, bool causal, bool bf16, int variant);
cudaError_t launch_d64(const LaunchArgs& a, bool causal, bool bf16, int variant);
cudaError_t launch_d128(const LaunchArgs& a, bool causal, bool bf16, int variant);
cudaError_t launch_d256(const LaunchArgs& a, bool causal, bool bf16, int variant);

// Launch fa_fwd_chain_kernel<D, causal, bf16, alt>: whole tiles (fa_fwd,
// D <= 128) with two softmax chains taking the key blocks in turn; the same
// grid and tile order as the one-tile kernel's tile mode.
cudaError_t launch_chain_d16(const LaunchArgs& a, bool causal, bool bf16, bool alt);
cudaError_t launch_chain_d32(const LaunchArgs& a, bool causal, bool bf16, bool alt);
cudaError_t launch_chain_d64(const LaunchArgs& a, bool causal, bool bf16, bool alt);
cudaError_t launch_chain_d128(const LaunchArgs& a, bool causal, bool bf16, bool alt);

// Launch fa_fwd_pair_kernel<128, causal, bf16, alt>: whole tiles (fa_fwd,
// D = 128) in units of two tiles per cluster of two CTAs (params.pair*);
// a.grid = 2 x clusters, at most 2 x pair_cluster_limit_d128(), and tmK in
// 64-row boxes (each CTA loads half of every key block).
cudaError_t launch_pair_d128(const LaunchArgs& a, bool causal, bool bf16, bool alt);
int pair_cluster_limit_d128();

// fa_lse_merge: parts share one layout; rows = Z * H * N
constexpr int MERGE_MAX_PARTS = 16;
struct MergeArgs {
    const void* o[MERGE_MAX_PARTS];
    const float* lse[MERGE_MAX_PARTS];
    int nparts, H, N, D;
    int64_t rows;
    int64_t sp_b, sp_h, sp_n;  // part strides (elements)
    int64_t so_b, so_h, so_n;  // output strides (elements)
    void* out;
    float* out_lse;
};
cudaError_t launch_lse_merge(const MergeArgs& a, bool bf16, int grid, cudaStream_t stream);

// Backward: the pre kernel, then the fused dK/dV + dQ kernel, on one stream
struct BwdLaunchArgs {
    const CUtensorMap* tmK;
    const CUtensorMap* tmV;
    const CUtensorMap* tmQ;
    const CUtensorMap* tmDO;
    const CUtensorMap* tmDQ;  // gradients in 32-row boxes, for the epilogues' tensor stores
    const CUtensorMap* tmDK;
    const CUtensorMap* tmDV;
    BwdParams params;
    int grid, pre_grid;  // the fused dK/dV + dQ kernel, the pre kernel
    cudaStream_t stream;
};
cudaError_t launch_bwd_d16(const BwdLaunchArgs& a, bool causal, bool bf16, int variant);
cudaError_t launch_bwd_d32(const BwdLaunchArgs& a, bool causal, bool bf16, int variant);
cudaError_t launch_bwd_d64(const BwdLaunchArgs& a, bool causal, bool bf16, int variant);
cudaError_t launch_bwd_d128(const BwdLaunchArgs& a, bool causal, bool bf16, int variant);
cudaError_t launch_bwd_d256(const BwdLaunchArgs& a, bool causal, bool bf16, int variant);

// Host-side shape facts of each specialisation.
int block_n_for(int D);      // keys per block
int smem_bytes_for(int D);   // dynamic shared memory per CTA
int swizzle_elems_for(int D);  // elements per swizzled row chunk (TMA box inner extent)

}  // namespace fa
