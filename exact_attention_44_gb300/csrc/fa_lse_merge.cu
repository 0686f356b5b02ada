// Combination of attention results over disjoint key sets by their
// log-sum-exps (the fa_lse_merge entry point).  One thread per 8 columns of
// a row; memory-bound: it reads every part once and writes the result once.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "fa_launch.h"

namespace fa {

template <bool BF16>
__device__ __forceinline__ float2 unpack2(uint32_t w) {
    if constexpr (BF16) return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
    else return __half22float2(*reinterpret_cast<const __half2*>(&w));
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2f(float lo, float hi) {
    if constexpr (BF16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    } else {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    }
}

// With λ_s = lse_s[r] (natural log) and μ = max_s λ_s:
//   lse[r] = μ + log Σ_s e^(λ_s − μ),   o[r] = Σ_s e^(λ_s − μ) o_s[r] / Σ_s e^(λ_s − μ)
template <bool BF16>
__global__ void __launch_bounds__(256) fa_lse_merge_kernel(const MergeArgs a) {
    const int C = a.D / 8;  // 16-byte chunks per row
    const int64_t total = a.rows * C;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = idx / C;
        const int c = (int)(idx - r * C);
        const int64_t n = r % a.N, zh = r / a.N;
        const int64_t h = zh % a.H, z = zh / a.H;
        const int64_t off_p = z * a.sp_b + h * a.sp_h + n * a.sp_n + 8 * c;
        float mx = -INFINITY;
#pragma unroll
        for (int s = 0; s < MERGE_MAX_PARTS; ++s)
            if (s < a.nparts) mx = fmaxf(mx, a.lse[s][r]);
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        float den = 0.f;
        if (mx != -INFINITY) {
#pragma unroll
            for (int s = 0; s < MERGE_MAX_PARTS; ++s) {
                if (s < a.nparts) {
                    const float w = expf(a.lse[s][r] - mx);
                    den += w;
                    const uint4 v = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.o[s]) + off_p);
                    const uint32_t words[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float2 f = unpack2<BF16>(words[i]);
                        acc[2 * i] += w * f.x;
                        acc[2 * i + 1] += w * f.y;
                    }
                }
            }
        }
        const float inv = den > 0.f ? 1.f / den : 0.f;
        uint4 out;
        out.x = pack2f<BF16>(acc[0] * inv, acc[1] * inv);
        out.y = pack2f<BF16>(acc[2] * inv, acc[3] * inv);
        out.z = pack2f<BF16>(acc[4] * inv, acc[5] * inv);
        out.w = pack2f<BF16>(acc[6] * inv, acc[7] * inv);
        *reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) + z * a.so_b + h * a.so_h + n * a.so_n + 8 * c) = out;
        if (c == 0 && a.out_lse != nullptr) a.out_lse[r] = den > 0.f ? mx + logf(den) : -INFINITY;
    }
}

cudaError_t launch_lse_merge(const MergeArgs& a, bool bf16, int grid, cudaStream_t stream) {
    if (bf16) fa_lse_merge_kernel<true><<<grid, 256, 0, stream>>>(a);
    else fa_lse_merge_kernel<false><<<grid, 256, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace fa
