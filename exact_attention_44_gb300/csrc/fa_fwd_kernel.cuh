// Fused attention forward, O = softmax(Q Kᵀ · scale) V with the per-row
// log-sum-exp, for sm_103a: TMA tile loads through mbarrier rings, tcgen05
// MMAs accumulating in tensor memory, online softmax in registers.
//
// The method is the tiled online-softmax forward of the pages
//   "Build Triton-Ascend Fused Attention" (Workflow, Implementation Pattern),
//   "Write Triton Attention Kernel" (Required reasoning process, steps 1-9;
//     Kernel design rules; Correctness requirements),
//   "把 FlashAttention 搬上昇腾：Triton-Ascend CV Pipeline 优化实战" (section 一:
//     exp2 with scale·log2(e), fp32 state, P cast to the input type;
//     section 八: causal loop bound at the diagonal).
// Its GB300 form:
//   * one persistent CTA per SM walks a static list of 128-row query tiles;
//   * warp 0 (one lane) streams Q once per tile and K_j, V_j per key block by
//     TMA into swizzled shared-memory rings guarded by full/empty mbarriers;
//   * warp 1 (one lane) issues S_j = Q K_jᵀ into a double-buffered S in TMEM
//     and O += P_j V_j with P_j read from TMEM (double-buffered), committing
//     each to mbarriers; S_{j+1} runs on the tensor cores while the softmax
//     works on S_j;
//   * warps 2-5 (128 threads, thread = query row = TMEM lane) run the online
//     softmax: mask (diagonal and tail blocks only), row max, exp2, row sum,
//     P -> fp16/bf16 into TMEM; O is rescaled in TMEM only when a row maximum
//     grows by more than 2^RESCALE_LOG2 (below that the stale maximum keeps
//     every p <= 2^RESCALE_LOG2, and O / l and lse are unchanged);
//   * warps 6-9 run the epilogue of the previous tile while the softmax warps
//     start the next one: read O out of TMEM, release it to the MMA warp, then
//     O / l -> global and lse = (m + log2 l)·ln 2.
// Every mbarrier wait is bounded; on expiry the CTA records the site in the
// status word, stops every role, lets its copies and MMAs land and frees TMEM.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fa_params.h"
#include "fa_ptx.cuh"

namespace fa {

// A row maximum (in log2 units of the scaled score) may run ahead of the one
// the probabilities are referenced to by at most this much before O and l
// are rescaled: probabilities stay <= 2^8 = 256, exact in fp16/bf16 range.
constexpr float RESCALE_LOG2 = 8.0f;

template <int D_>
struct Traits {
    static constexpr int D = D_;
    static constexpr int BN = D == 256 ? 64 : 128;            // keys per block
    static constexpr int SW = D * 2 >= 128 ? 128 : D * 2;      // bytes per swizzled row chunk
    static constexpr int SWE = SW / 2;                         // elements per row chunk
    static constexpr int NCHUNK = D / SWE;                     // row chunks per tile row
    static constexpr uint32_t SWIZZLE_CODE = SW == 128 ? 2u : SW == 64 ? 4u : 6u;  // UMMA descriptor code
    static constexpr int Q_BYTES = BM * D * 2;
    static constexpr int KV_BYTES = BN * D * 2;
    static constexpr int Q_STAGES = D == 256 ? 1 : 2;
    // K and V rings are two deep, like S and P: K slot s is free once S of
    // that block is complete, V slot s once its P·V is; those two commits
    // release the slots, so no separate "empty" barriers exist.
    static constexpr int KV_STAGES = 2;
    // tensor memory columns (lane = query row): a ring of SR score blocks,
    // each holding S_g (BN fp32 columns) and then, in its first BN/2
    // columns, P_g (two 16-bit values per column); then O (D fp32 columns)
    static constexpr int SR = 3;
    static constexpr uint32_t TM_S = 0;                        // S/P ring slot r at TM_S + r * BN
    static constexpr uint32_t TM_O = SR * BN;                  // O
    static constexpr uint32_t TMEM_COLS = 512;
    static_assert(TM_O + D <= TMEM_COLS, "tensor memory budget");
    // shared memory (offsets from a 1024-byte aligned base)
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + Q_STAGES * Q_BYTES;
    static constexpr int OFF_V = OFF_K + KV_STAGES * KV_BYTES;
    // softmax -> epilogue hand-over, 2 slots of {m, l of half 0, l of half 1} per row
    static constexpr int OFF_HAND = OFF_V + KV_STAGES * KV_BYTES;
    // partial row maxima of the two column halves, 2 slots (by block parity)
    static constexpr int OFF_RED = OFF_HAND + 2 * 3 * BM * 4;
    static constexpr int OFF_BAR = OFF_RED + 2 * 2 * BM * 4;
    // barrier indices
    static constexpr int B_QFULL = 0;
    static constexpr int B_QEMPTY = B_QFULL + Q_STAGES;
    static constexpr int B_KFULL = B_QEMPTY + Q_STAGES;        // [2] K tile landed (TMA)
    static constexpr int B_VFULL = B_KFULL + KV_STAGES;        // [2] V tile landed (TMA)
    static constexpr int B_SFULL = B_VFULL + KV_STAGES;        // [SR] S_g ready; K slot free (commit)
    static constexpr int B_PFULL = B_SFULL + SR;               // [SR] P_g written (256 softmax threads)
    static constexpr int B_PVDONE = B_PFULL + SR;              // [SR] O += P_g V_g complete; slot and V slot free (commit)
    static constexpr int B_EPIFULL = B_PVDONE + SR;            // [2] m, l of a tile handed over (256)
    static constexpr int B_EPIEMPTY = B_EPIFULL + 2;           // [2] hand-over slot read (128)
    static constexpr int B_OFREE = B_EPIEMPTY + 2;             // O read out of TMEM (128)
    static constexpr int B_RED = B_OFREE + 1;                  // [2] both halves' partial maxima written (256)
    static constexpr int B_DRAIN = B_RED + 2;                  // [2] teardown of the two MMA issuers
    static constexpr int NUM_BARS = B_DRAIN + 2;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;    // tmem base, abort flag
    static constexpr int SMEM_USED = OFF_MISC + 16;
    // >= 120 KB keeps one CTA per SM, so no CTA ever waits on another's TMEM
    static constexpr int SMEM_BYTES = (SMEM_USED + 1024) > 120 * 1024 ? SMEM_USED + 1024 : 120 * 1024;
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");

    static __device__ __forceinline__ uint32_t bar_count(int i) {
        if (i >= B_PFULL && i < B_PFULL + SR) return 256;
        if (i >= B_EPIFULL && i < B_EPIFULL + 2) return 256;
        if (i >= B_EPIEMPTY && i < B_OFREE + 1) return 128;
        if (i >= B_RED && i < B_RED + 2) return 256;
        return 1;
    }
};

struct Ctl {
    volatile int* abort_flag;
    uint32_t* status;
    uint64_t limit_ns;
};

__device__ __forceinline__ void record_timeout(const Ctl& c, uint32_t site) {
    *c.abort_flag = 1;
    atomicCAS(c.status, 0u, 5u /* FA_ERR_DEVICE_TIMEOUT */ | (site << 8) | ((blockIdx.x & 0xFFFFu) << 16));
}

// Wait for the phase of `bar` with parity `parity`.  Gives up (false) when
// another role has aborted or after limit_ns, recording the site.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, const Ctl& c, uint32_t site) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    for (;;) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if (*c.abort_flag) return false;
        if (ptx::globaltimer_ns() - t0 > c.limit_ns) {
            record_timeout(c, site);
            return false;
        }
    }
}

// The same wait taken by a whole warp: every lane leaves with the same answer,
// so no lane can run ahead into a warp-collective tcgen05 access alone.
__device__ __forceinline__ bool warp_wait_phase(uint32_t bar, uint32_t parity, const Ctl& c, uint32_t site) {
    return __all_sync(0xffffffffu, wait_phase(bar, parity, c, site));
}

// Teardown wait after an abort: ignores the abort flag, bounded by limit_ns.
__device__ __forceinline__ bool drain_phase(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    const uint64_t t0 = ptx::globaltimer_ns();
    while (!ptx::mbar_try_wait(bar, parity))
        if (ptx::globaltimer_ns() - t0 > limit_ns) return false;
    return true;
}

struct TileInfo {
    int z, hq, hk, q_start, nkv;
};

// Barrier slot and phase parity of key block g (global count) in a ring of R.
template <int R>
__device__ __forceinline__ uint32_t rslot(uint32_t g) { return g % R; }
template <int R>
__device__ __forceinline__ uint32_t rphase(uint32_t g) { return (g / R) & 1u; }

// Tile t of the static schedule.  Non-causal: head-major, so the CTAs running
// at the same time share a head's K/V in L2.  Causal: query blocks from the
// last (most key blocks) to the first, heads innermost, so the heavy tiles go
// first and the light ones fill the tail.  A causal tile stops at the key
// block holding its last row ("Write Triton Attention Kernel", step 9).
template <bool CAUSAL, int BN>
__device__ __forceinline__ TileInfo tile_info(int t, const FwdParams& p) {
    TileInfo ti;
    const int heads = p.Z * p.Hq;
    int head, mb;
    if (CAUSAL) {
        mb = p.Tq - 1 - t / heads;
        head = t % heads;
    } else {
        head = t / p.Tq;
        mb = t % p.Tq;
    }
    ti.z = head / p.Hq;
    ti.hq = head % p.Hq;
    ti.hk = ti.hq / p.group;  // GQA: kv head = q head // (Hq / Hkv)
    ti.q_start = mb * BM;
    if (CAUSAL) {
        const int last_row = min(ti.q_start + BM, p.Nq) - 1;
        ti.nkv = min(p.Tk, last_row / BN + 1);
    } else {
        ti.nkv = p.Tk;
    }
    return ti;
}

// ------------------------------------------------------------ TMA producers -
// Two threads load: one Q and K (the S stream's operands), one V (the P·V
// stream's), so a K load never queues behind a V slot that is still in use.
// With two Q slots the next tile's Q is requested right after the current
// tile's first K: its slot held the tile before, whose last S is complete by
// the time the second K's slot frees anyway.

template <int D, bool CAUSAL>
__device__ void run_producer_qk(const CUtensorMap* tmQ, const CUtensorMap* tmK, const FwdParams& p, uint32_t sbase,
                                uint32_t bar0, const Ctl& ctl) {
    using T = Traits<D>;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    const uint64_t pol_q = ptx::policy_evict_first();
    const uint64_t pol_kv = ptx::policy_evict_last();
    uint32_t qi = 0, ki = 0;  // loads issued into each ring
    bool ok = true;
    bool withheld = false;
    auto load_q = [&](const TileInfo& ti) -> bool {
        const uint32_t s = qi % T::Q_STAGES, ph = (qi / T::Q_STAGES) & 1u;
        if (!wait_phase(bar(T::B_QEMPTY + s), ph ^ 1u, ctl, SITE_Q_EMPTY)) return false;
        ptx::mbar_arrive_expect_tx(bar(T::B_QFULL + s), T::Q_BYTES);
        const uint32_t dst = sbase + T::OFF_Q + s * T::Q_BYTES;
        for (int c = 0; c < T::NCHUNK; ++c)
            ptx::tma_load_4d(dst + c * (BM * T::SW), tmQ, bar(T::B_QFULL + s), c * T::SWE, ti.q_start, ti.hq, ti.z,
                             pol_q);
        ++qi;
        return true;
    };
    int t = blockIdx.x;
    if (t < p.ntiles) ok = load_q(tile_info<CAUSAL, T::BN>(t, p));
    for (; ok && t < p.ntiles; t += gridDim.x) {
        const TileInfo ti = tile_info<CAUSAL, T::BN>(t, p);
        for (int j = 0; j < ti.nkv; ++j) {
            // slot ki & 1 held block ki - 2, free once S of that block is complete
            const uint32_t s = ki & 1u;
            if (ki >= 2 && !wait_phase(bar(T::B_SFULL + rslot<T::SR>(ki - 2)), rphase<T::SR>(ki - 2), ctl,
                                       SITE_K_EMPTY)) { ok = false; break; }
            if (p.inject_stall && blockIdx.x == 0 && !withheld) {
                withheld = true;  // never issued: the S issuer's wait for this block must time out
            } else {
                ptx::mbar_arrive_expect_tx(bar(T::B_KFULL + s), T::KV_BYTES);
                const uint32_t dst = sbase + T::OFF_K + s * T::KV_BYTES;
                for (int c = 0; c < T::NCHUNK; ++c)
                    ptx::tma_load_4d(dst + c * (T::BN * T::SW), tmK, bar(T::B_KFULL + s), c * T::SWE, j * T::BN,
                                     ti.hk, ti.z, pol_kv);
            }
            ++ki;
            // with two Q slots the next tile's Q can go right after the first
            // K; with one, only after the last K (its slot frees at this
            // tile's last S, which needs that K)
            const int q_at = T::Q_STAGES >= 2 ? 0 : ti.nkv - 1;
            if (j == q_at && t + (int)gridDim.x < p.ntiles && !load_q(tile_info<CAUSAL, T::BN>(t + gridDim.x, p))) {
                ok = false;
                break;
            }
        }
    }
    if (!ok) {
        // Let every copy still in flight land before shared memory is released.
        // The withheld load never completes; its wait simply runs out.
        const uint64_t lim = ctl.limit_ns;
        for (uint32_t i = qi > (uint32_t)T::Q_STAGES ? qi - T::Q_STAGES : 0; i < qi; ++i)
            drain_phase(bar(T::B_QFULL + i % T::Q_STAGES), (i / T::Q_STAGES) & 1u, lim);
        for (uint32_t i = ki > 2u ? ki - 2u : 0u; i < ki; ++i)
            drain_phase(bar(T::B_KFULL + (i & 1u)), (i >> 1) & 1u, withheld ? lim / 64 : lim);
    }
}

template <int D, bool CAUSAL>
__device__ void run_producer_v(const CUtensorMap* tmV, const FwdParams& p, uint32_t sbase, uint32_t bar0,
                               const Ctl& ctl) {
    using T = Traits<D>;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    const uint64_t pol_kv = ptx::policy_evict_last();
    uint32_t vi = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < p.ntiles; t += gridDim.x) {
        const TileInfo ti = tile_info<CAUSAL, T::BN>(t, p);
        for (int j = 0; j < ti.nkv; ++j) {
            // slot vi & 1 held block vi - 2, free once its P·V is complete
            const uint32_t s = vi & 1u;
            if (vi >= 2 && !wait_phase(bar(T::B_PVDONE + rslot<T::SR>(vi - 2)), rphase<T::SR>(vi - 2), ctl,
                                       SITE_V_EMPTY)) { ok = false; break; }
            ptx::mbar_arrive_expect_tx(bar(T::B_VFULL + s), T::KV_BYTES);
            const uint32_t dst = sbase + T::OFF_V + s * T::KV_BYTES;
            for (int c = 0; c < T::NCHUNK; ++c)
                ptx::tma_load_4d(dst + c * (T::BN * T::SW), tmV, bar(T::B_VFULL + s), c * T::SWE, j * T::BN, ti.hk,
                                 ti.z, pol_kv);
            ++vi;
        }
    }
    if (!ok)
        for (uint32_t i = vi > 2u ? vi - 2u : 0u; i < vi; ++i)
            drain_phase(bar(T::B_VFULL + (i & 1u)), (i >> 1) & 1u, ctl.limit_ns);
}

// ------------------------------------------------------------ MMA issuers ---
// Issuing a tcgen05.mma stalls the issuing thread until the tensor core takes
// it, and the tensor core queues little, so a single issuer leaves it idle
// whenever that thread waits on a barrier.  Two threads issue instead: one
// the S = Q Kᵀ stream, one the O += P V stream; each waits while the other
// feeds the tensor core.  The streams touch disjoint TMEM (S vs P and O) and
// shared memory (Q, K vs V) and are ordered only through mbarriers.
// Descriptors are a per-stage base word plus a compile-time offset.

// S_g = Q K_gᵀ ("Write Triton Attention Kernel", step 5b) into S[g & 1]
template <int D, bool CAUSAL, bool BF16>
__device__ void run_mma_qk(const FwdParams& p, uint32_t sbase, uint32_t bar0, uint32_t tmem, const Ctl& ctl) {
    using T = Traits<D>;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    constexpr uint32_t IDESC = ptx::idesc_f16(BM, T::BN, BF16, false, false);  // Q, K both K-major
    constexpr uint32_t HI = ptx::smem_desc_hi(8 * T::SW, T::SWIZZLE_CODE);     // 8-row swizzle atoms
    const uint32_t q_lo0 = ptx::smem_desc_lo(sbase + T::OFF_Q, 16);
    const uint32_t k_lo0 = ptx::smem_desc_lo(sbase + T::OFF_K, 16);
    uint32_t qi = 0, g = 0;  // Q tiles and S blocks issued
    bool ok = true;
    for (int t = blockIdx.x; ok && t < p.ntiles; t += gridDim.x) {
        const TileInfo ti = tile_info<CAUSAL, T::BN>(t, p);
        const uint32_t qs = qi % T::Q_STAGES;
        if (!wait_phase(bar(T::B_QFULL + qs), (qi / T::Q_STAGES) & 1u, ctl, SITE_Q_FULL)) { ok = false; break; }
        const uint32_t q_lo = q_lo0 + qs * (T::Q_BYTES >> 4);
        for (int j = 0; j < ti.nkv; ++j, ++g) {
            const uint32_t kb = g & 1u, r = rslot<T::SR>(g);
            if (!wait_phase(bar(T::B_KFULL + kb), (g >> 1) & 1u, ctl, SITE_K_FULL)) { ok = false; break; }
            // ring slot r held block g - SR (S, then P) until O += P V of that
            // block completed; the softmax, seeing S_g, may then overwrite it
            if (g >= (uint32_t)T::SR && !wait_phase(bar(T::B_PVDONE + r), rphase<T::SR>(g - T::SR), ctl, SITE_S_FREE)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            const uint32_t k_lo = k_lo0 + kb * (T::KV_BYTES >> 4);
            const uint32_t d_tmem = tmem + T::TM_S + r * T::BN;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t a_off = (((kk * 16) / T::SWE) * (BM * T::SW) + ((kk * 16) % T::SWE) * 2) >> 4;
                const uint32_t b_off = (((kk * 16) / T::SWE) * (T::BN * T::SW) + ((kk * 16) % T::SWE) * 2) >> 4;
                ptx::mma_ss(d_tmem, ptx::desc64(q_lo + a_off, HI), ptx::desc64(k_lo + b_off, HI), IDESC,
                            kk > 0 ? 1u : 0u);
            }
            ptx::tc_commit(bar(T::B_SFULL + r));  // S ready, K slot kb free
            if (j == ti.nkv - 1) {
                ptx::tc_commit(bar(T::B_QEMPTY + qs));  // last use of this Q tile
                ++qi;
            }
        }
    }
    if (!ok) {
        // every MMA this thread issued must finish before TMEM and shared memory go away
        ptx::tc_commit(bar(T::B_DRAIN));
        drain_phase(bar(T::B_DRAIN), 0u, ctl.limit_ns);
    }
}

// O += P_g V_g (step 5h); the first block of a tile overwrites O, once the
// epilogue has read the previous tile's O out of TMEM
template <int D, bool CAUSAL, bool BF16>
__device__ void run_mma_pv(const FwdParams& p, uint32_t sbase, uint32_t bar0, uint32_t tmem, const Ctl& ctl) {
    using T = Traits<D>;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    constexpr uint32_t IDESC = ptx::idesc_f16(BM, D, BF16, false, true);      // V is MN-major (D contiguous)
    constexpr uint32_t HI = ptx::smem_desc_hi(8 * T::SW, T::SWIZZLE_CODE);
    const uint32_t v_lo0 = ptx::smem_desc_lo(sbase + T::OFF_V, T::BN * T::SW);  // LBO: next column chunk of V
    uint32_t g = 0, ntile = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < p.ntiles; t += gridDim.x, ++ntile) {
        const TileInfo ti = tile_info<CAUSAL, T::BN>(t, p);
        for (int j = 0; j < ti.nkv; ++j, ++g) {
            const uint32_t vb = g & 1u, r = rslot<T::SR>(g);
            if (j == 0 && ntile > 0 &&
                !wait_phase(bar(T::B_OFREE), (ntile - 1) & 1u, ctl, SITE_O_FREE)) { ok = false; break; }
            if (!wait_phase(bar(T::B_PFULL + r), rphase<T::SR>(g), ctl, SITE_P_FULL)) { ok = false; break; }
            if (!wait_phase(bar(T::B_VFULL + vb), (g >> 1) & 1u, ctl, SITE_V_FULL)) { ok = false; break; }
            ptx::tc_fence_after();
            const uint32_t v_lo = v_lo0 + vb * (T::KV_BYTES >> 4);
            const uint32_t a_tmem = tmem + T::TM_S + r * T::BN;  // P_g over the first BN/2 columns of the slot
            const uint32_t acc0 = j > 0 ? 1u : 0u;
#pragma unroll
            for (int kk = 0; kk < T::BN / 16; ++kk)
                ptx::mma_ts(tmem + T::TM_O, a_tmem + kk * 8, ptx::desc64(v_lo + ((kk * 16 * T::SW) >> 4), HI), IDESC,
                            kk > 0 ? 1u : acc0);
            ptx::tc_commit(bar(T::B_PVDONE + r));  // O updated, ring slot r and V slot vb free
        }
    }
    if (!ok) {
        ptx::tc_commit(bar(T::B_DRAIN + 1));
        drain_phase(bar(T::B_DRAIN + 1), 0u, ctl.limit_ns);
    }
}

// ------------------------------------------------------------ softmax -------
template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    if constexpr (BF16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    } else {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    }
}

// O[row, c0 : c0 + NCOL] *= alpha for the rows of this warp's lane quadrant
template <int NCOL>
__device__ __forceinline__ void rescale_o(uint32_t taddr, float alpha) {
    if constexpr (NCOL >= 32) {
        const uint64_t a2 = ptx::pack_f32x2(alpha, alpha);
#pragma unroll
        for (int i = 0; i < NCOL / 32; ++i) {
            uint32_t r[32];
            ptx::tmem_ld32(taddr + 32 * i, r);
#pragma unroll
            for (int x = 0; x < 16; ++x) {
                float lo, hi;
                ptx::unpack_f32x2(ptx::fmul2(ptx::pack_f32x2(__uint_as_float(r[2 * x]), __uint_as_float(r[2 * x + 1])),
                                             a2),
                                  lo, hi);
                r[2 * x] = __float_as_uint(lo);
                r[2 * x + 1] = __float_as_uint(hi);
            }
            ptx::tmem_st32(taddr + 32 * i, r);
        }
    } else if constexpr (NCOL == 16) {
        uint32_t r[16];
        ptx::tmem_ld16(taddr, r);
#pragma unroll
        for (int x = 0; x < 16; ++x) r[x] = __float_as_uint(__uint_as_float(r[x]) * alpha);
        ptx::tmem_st16(taddr, r);
    } else {
        uint32_t r[8];
        ptx::tmem_ld8(taddr, r);
#pragma unroll
        for (int x = 0; x < 8; ++x) r[x] = __float_as_uint(__uint_as_float(r[x]) * alpha);
        ptx::tmem_st8(taddr, r);
    }
}

// Online softmax for one column half of every key block: 128 threads, thread
// = query row = TMEM lane; the two halves swap partial row maxima through
// shared memory, so both reference the same maximum m, and each keeps its
// own partial denominator (the epilogue adds them).
template <int D, bool CAUSAL, bool BF16>
__device__ void run_softmax(const FwdParams& p, uint32_t bar0, uint32_t tmem, float* hand, float* red, int h,
                            const Ctl& ctl) {
    using T = Traits<D>;
    constexpr int BN = T::BN;
    constexpr int HC = BN / 2;                 // score columns per thread
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    const int quad = (threadIdx.x / 32) % 4;  // TMEM lane quadrant this warp may access
    const int row = quad * 32 + threadIdx.x % 32;
    const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
    const float c = p.scale_log2;
    const uint64_t c2 = ptx::pack_f32x2(c, c);
    uint32_t step = 0, ntile = 0;

    for (int t = blockIdx.x; t < p.ntiles; t += gridDim.x, ++ntile) {
        const TileInfo ti = tile_info<CAUSAL, BN>(t, p);
        const int q_row = ti.q_start + row;
        // running max (log2 units of the scaled score) and denominator, fp32
        // ("Write Triton Attention Kernel", step 4; the initial l is 0)
        float m = -INFINITY, l = 0.f;
        for (int j = 0; j < ti.nkv; ++j) {
            const uint32_t r = rslot<T::SR>(step);      // ring slot of S_j / P_j
            const uint32_t b = step & 1u, ph = (step >> 1) & 1u;  // max-exchange slot
            if (!warp_wait_phase(bar(T::B_SFULL + r), rphase<T::SR>(step), ctl, SITE_S_FULL)) return;
            ptx::tc_fence_after();
            const uint32_t s_addr = tmem + lane_addr + T::TM_S + r * BN;
            float s[HC];
#pragma unroll
            for (int i = 0; i < HC / 32; ++i) {
                uint32_t rr[32];
                ptx::tmem_ld32(s_addr + h * HC + 32 * i, rr);
#pragma unroll
                for (int x = 0; x < 32; ++x) s[32 * i + x] = __uint_as_float(rr[x]);
            }
            // the mask goes on the scores before the row max (Correctness
            // requirements); only the diagonal block and the key tail need it
            const int k0 = j * BN + h * HC;
            const bool need_mask = (CAUSAL && j * BN + BN - 1 > ti.q_start) || (j * BN + BN > p.Nkv);
            if (need_mask) {
                const int kmax = CAUSAL ? min(p.Nkv - 1, q_row) : p.Nkv - 1;  // last kept key for this row
#pragma unroll
                for (int x = 0; x < HC; ++x)
                    if (k0 + x > kmax) s[x] = -INFINITY;
            }
            float mx0 = fmaxf(s[0], s[1]), mx1 = fmaxf(s[2], s[3]);
#pragma unroll
            for (int x = 4; x < HC; x += 4) {  // HC is a multiple of 4
                mx0 = ptx::fmax3(mx0, s[x], s[x + 1]);
                mx1 = ptx::fmax3(mx1, s[x + 2], s[x + 3]);
            }
            // Swap partial maxima with the other half.  Arriving also says this
            // thread's S is in registers: P is written over the slot's first
            // columns only once both halves have arrived.  (Exchange slot b is
            // free: every thread read it two blocks ago before arriving last block.)
            const float pmax = fmaxf(mx0, mx1);
            red[(b * 2 + h) * BM + row] = pmax;
            ptx::mbar_arrive(bar(T::B_RED + b));
            if (j == 0) {
                // the first block sets the reference maximum m
                if (!warp_wait_phase(bar(T::B_RED + b), ph, ctl, SITE_MAX_XCHG)) return;
                m = fmaxf(pmax, red[(b * 2 + (h ^ 1)) * BM + row]) * c;  // scale > 0
            }
            // p = 2^(s·scale·log2e − m) against the current reference m; l sums
            // the fp32 p, P V uses p cast to the input type
            constexpr int NP = HC / 2;  // packed P columns of this half
            uint32_t pk[NP];
            auto exps = [&](float ref) -> uint64_t {
                const uint64_t negm2 = ptx::pack_f32x2(-ref, -ref);
                uint64_t sum2 = ptx::pack_f32x2(0.f, 0.f);
#pragma unroll
                for (int x = 0; x < NP; ++x) {
                    float a0, a1;
                    ptx::unpack_f32x2(ptx::ffma2(ptx::pack_f32x2(s[2 * x], s[2 * x + 1]), c2, negm2), a0, a1);
                    const float p0 = ptx::ex2(a0), p1 = ptx::ex2(a1);
                    sum2 = ptx::fadd2(sum2, ptx::pack_f32x2(p0, p1));
                    pk[x] = pack2<BF16>(p0, p1);
                }
                return sum2;
            };
            uint64_t sum2 = exps(m);
            float alpha = 1.f;
            if (j > 0) {
                // the block maximum arrives while the exponentials run; only
                // when it exceeds m by more than 2^RESCALE_LOG2 are P redone
                // against the new maximum, and O and l rescaled by alpha before
                // this block is added to them (Kernel design rules).  Both
                // halves see the same values, so both take the same branch.
                if (!warp_wait_phase(bar(T::B_RED + b), ph, ctl, SITE_MAX_XCHG)) return;
                const float m_tile = fmaxf(pmax, red[(b * 2 + (h ^ 1)) * BM + row]) * c;
                if (__any_sync(0xffffffffu, m_tile > m + RESCALE_LOG2)) {
                    const float m_new = fmaxf(m, m_tile);
                    alpha = ptx::ex2(m - m_new);
                    m = m_new;
                    sum2 = exps(m);
                    const uint32_t g = step - 1;
                    if (!warp_wait_phase(bar(T::B_PVDONE + rslot<T::SR>(g)), rphase<T::SR>(g), ctl, SITE_PV_DONE))
                        return;
                    ptx::tc_fence_after();
                    rescale_o<D / 2>(tmem + lane_addr + T::TM_O + h * (D / 2), alpha);
                }
            }
            // P_j over the first BN/2 columns of its slot: keys h*HC.. at packed column h*HC/2
            if constexpr (NP == 32) ptx::tmem_st32(s_addr + h * NP, pk);
            else ptx::tmem_st16(s_addr + h * NP, pk);
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(T::B_PFULL + r));
            float sl, sh;
            ptx::unpack_f32x2(sum2, sl, sh);
            l = l * alpha + (sl + sh);
            ++step;
        }
        // hand m and this half's l to the epilogue warps
        const uint32_t slot = ntile & 1u;
        if (!warp_wait_phase(bar(T::B_EPIEMPTY + slot), ((ntile >> 1) & 1u) ^ 1u, ctl, SITE_EPI_EMPTY)) return;
        if (h == 0) hand[slot * 3 * BM + row] = m;
        hand[slot * 3 * BM + (1 + h) * BM + row] = l;
        ptx::mbar_arrive(bar(T::B_EPIFULL + slot));
    }
}

// ------------------------------------------------------------ epilogue ------
// O = acc / l in the input type, lse = m + log(l) in natural-log units
// ("Write Triton Attention Kernel", steps 6-8).  O is read out of TMEM and
// converted first, TMEM is handed back to the MMA warp, then rows are stored.
template <int D, bool CAUSAL, bool BF16>
__device__ void run_epilogue(const FwdParams& p, uint32_t bar0, uint32_t tmem, const float* hand, const Ctl& ctl) {
    using T = Traits<D>;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    const int quad = (threadIdx.x / 32) % 4;
    const int row = quad * 32 + threadIdx.x % 32;
    const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
    uint32_t step = 0, ntile = 0;
    constexpr int CH = D >= 32 ? 32 : 16;               // columns per TMEM load
    constexpr int HELD = D <= 128 ? D / CH : 64 / CH;    // chunks converted before their stores
    for (int t = blockIdx.x; t < p.ntiles; t += gridDim.x, ++ntile) {
        const TileInfo ti = tile_info<CAUSAL, T::BN>(t, p);
        step += ti.nkv;
        const uint32_t slot = ntile & 1u;
        if (!warp_wait_phase(bar(T::B_EPIFULL + slot), (ntile >> 1) & 1u, ctl, SITE_EPI_FULL)) return;
        const float m = hand[slot * 3 * BM + row];
        const float l = hand[slot * 3 * BM + BM + row] + hand[slot * 3 * BM + 2 * BM + row];
        ptx::mbar_arrive(bar(T::B_EPIEMPTY + slot));
        const uint32_t g = step - 1;  // the tile's last P·V
        if (!warp_wait_phase(bar(T::B_PVDONE + rslot<T::SR>(g)), rphase<T::SR>(g), ctl, SITE_PV_DONE)) return;
        ptx::tc_fence_after();

        const int q_row = ti.q_start + row;
        const bool store = q_row < p.Nq;
        const float inv_l = 1.f / l;
        uint8_t* orow = reinterpret_cast<uint8_t*>(p.o) +
                        2 * ((int64_t)ti.z * p.so_z + (int64_t)ti.hq * p.so_h + (int64_t)q_row * p.so_n);
#pragma unroll
        for (int base = 0; base < D / CH; base += HELD) {
            uint32_t o2[HELD][CH / 2];
#pragma unroll
            for (int i = 0; i < HELD; ++i) {
                uint32_t r[CH];
                if constexpr (CH == 32) ptx::tmem_ld32(tmem + lane_addr + T::TM_O + (base + i) * CH, r);
                else ptx::tmem_ld16(tmem + lane_addr + T::TM_O + (base + i) * CH, r);
#pragma unroll
                for (int x = 0; x < CH / 2; ++x)
                    o2[i][x] = pack2<BF16>(__uint_as_float(r[2 * x]) * inv_l, __uint_as_float(r[2 * x + 1]) * inv_l);
            }
            if (base + HELD == D / CH) {
                // all of O has been read: the MMA warp may overwrite it with the next tile
                ptx::tc_fence_before();
                ptx::mbar_arrive(bar(T::B_OFREE));
            }
            if (store) {
#pragma unroll
                for (int i = 0; i < HELD; ++i) {
                    uint4* dst = reinterpret_cast<uint4*>(orow + 2 * (base + i) * CH);
#pragma unroll
                    for (int x = 0; x < CH / 8; ++x)
                        dst[x] = make_uint4(o2[i][4 * x], o2[i][4 * x + 1], o2[i][4 * x + 2], o2[i][4 * x + 3]);
                }
            }
        }
        if (store && p.lse != nullptr)
            p.lse[((int64_t)ti.z * p.Hq + ti.hq) * p.Nq + q_row] = (m + log2f(l)) * 0.6931471805599453f;
    }
}

// ------------------------------------------------------------ kernel --------
template <int D, bool CAUSAL, bool BF16>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
    using T = Traits<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = ptx::smem_addr(smem);
    const uint32_t bar0 = sbase + T::OFF_BAR;
    float* hand = reinterpret_cast<float*>(smem + T::OFF_HAND);
    float* red = reinterpret_cast<float*>(smem + T::OFF_RED);
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + T::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + T::OFF_MISC + 4);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        for (int i = 0; i < T::NUM_BARS; ++i) ptx::mbar_init(bar0 + 8u * i, T::bar_count(i));
        *abort_flag = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tmQ);
        ptx::prefetch_tmap(&tmK);
        ptx::prefetch_tmap(&tmV);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_addr(const_cast<uint32_t*>(tmem_slot)), T::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const Ctl ctl{abort_flag, p.status, p.wait_limit_ns};

    if (warp == 0) {
        if (lane == 0) run_producer_qk<D, CAUSAL>(&tmQ, &tmK, p, sbase, bar0, ctl);
    } else if (warp == 15) {
        if (lane == 0) run_producer_v<D, CAUSAL>(&tmV, p, sbase, bar0, ctl);
    } else if (warp == 1) {
        if (lane == 0) run_mma_qk<D, CAUSAL, BF16>(p, sbase, bar0, tmem, ctl);
    } else if (warp == 2) {
        if (lane == 0) run_mma_pv<D, CAUSAL, BF16>(p, sbase, bar0, tmem, ctl);
    } else if (warp < 11) {
        run_softmax<D, CAUSAL, BF16>(p, bar0, tmem, hand, red, (warp - 3) / 4, ctl);
    } else if (warp < 15) {
        run_epilogue<D, CAUSAL, BF16>(p, bar0, tmem, hand, ctl);
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, T::TMEM_COLS);
    }
}

}  // namespace fa
