// Attention backward for head dim 256 on sm_103a: gradients dQ, dK, dV of
// the fused forward from the saved log-sum-exp (blog "把 FlashAttention 搬上昇腾：
// Triton-Ascend CV Pipeline 优化实战", section 二: recompute P from the lse,
// then dP, dS and the three gradients; section 七 treats D = 256 in pieces
// of D = 128 for the same reason this kernel does: one pass does not fit).
//
// At D = 256 the layout of the smaller head dims (fa_bwd_kernel.cuh) fits
// neither budget: its dK/dV phase would need Sᵀ, dPᵀ, dV and dK in tensor
// memory (128 + 128 + 256 + 256 of 512 columns) and 64 KB tiles of K, V, Q and
// dO in shared memory (256 of 227 KB).  So:
//   dK/dV phase   per unit (128-key block, kv head), K and V resident, query
//                 steps of 64 rows (Q, dO: 32 KB each), and two passes over
//                 the steps, each with one 256-column accumulator in TMEM:
//                   dV pass   Sᵀ = K Qᵢᵀ, Pᵀ = 2^(Sᵀ·scale·log2e − lse2ᵢ),
//                             dV += Pᵀ dOᵢ
//                   dK pass   Sᵀ, Pᵀ as above, dPᵀ = V dOᵢᵀ,
//                             dSᵀ = Pᵀ ∘ (dPᵀ − Δᵢ), dK += dSᵀ Qᵢ
//                 (five products a step instead of four: Sᵀ is computed twice);
//   dQ phase      per unit (128-row query block, query head), Q and dO
//                 resident, key steps of 64 keys:
//                   S = Qᵢ Kⱼᵀ, dP = dOᵢ Vⱼᵀ, dS = P ∘ (dP − Δ), dQ += dS Kⱼ.
// The dV pass does not need V: its 64 KB hold a second slot of Q, dO (and a
// second Sᵀ block in TMEM), so that pass issues step t + 1's Sᵀ before step
// t's accumulation while step t + 2's copies are in flight, and V loads once
// the pass is done.  The dK pass and the dQ phase are single-buffered (no
// room for a second slot; measured on GB300 at Z8 H16 N2048 with one slot
// everywhere: ~2.2 us a step in the dV pass against ~0.7 us of tensor work);
// in the dK pass a step's dO, read only by its dPᵀ, is loaded as soon as the
// previous step's dPᵀ is done, so only Q waits for the accumulation.
// dK, dV and dQ are each summed inside one CTA: no atomics, bitwise
// reproducible.
// Variant instantiations (VAR 1-4: window, ALiBi, packed sequences; the
// forward's options, "Write Triton Attention Kernel", Inputs) take the
// shared unit decoders' window ranges and sequence tables: loads start at the
// sequence's rows and the window's first key block, pairs are masked only in
// steps not wholly kept, ALiBi subtracts slope·log2e·|i − j| in both phases, and a
// 32-row box that crosses a sequence end is stored row by row.
// The pre kernel (Δ, base-2 lse), the unit orders and the tile stores are the
// smaller head dims' (fa_bwd_kernel.cuh).
//
// Warps: 0-7 softmax, two column groups of 32 of each 64-column step (thread
// = TMEM lane: a key in the dK/dV phase, a query in the dQ phase), 8-11
// epilogue, 12 TMA producer, 13 MMA issuer.  Every wait is bounded as in the
// forward kernel.
#pragma once

#include "fa_bwd_kernel.cuh"

namespace fa {

// Softmax column groups of a 64-column step (4 warps each).  Measured on
// GB300 at Z8 H16 N2048: two groups of 32 columns +1.1 % non-causal, +3.3 %
// causal against one group of 64 (the steps are bound by their serial
// load -> Sᵀ -> softmax -> accumulation chain more than by the softmax).
constexpr int WIDE_NG = 2;
constexpr int WIDE_CW = 64 / WIDE_NG;
constexpr int WIDE_SOFTMAX_WARPS = 4 * WIDE_NG;
constexpr int WIDE_THREADS = (WIDE_SOFTMAX_WARPS + 6) * 32;

struct WideTraits {
    static constexpr int D = 256;
    static constexpr int SW = 128;                 // bytes per swizzled row chunk
    static constexpr int SWE = 64;                 // elements per row chunk
    static constexpr int NCHUNK = D / SWE;         // 4
    static constexpr uint32_t SWIZZLE_CODE = 2u;   // 128-byte swizzle
    static constexpr int STEP = 64;                // query rows (dK/dV) or keys (dQ) per step
    static constexpr int TILE128 = 128 * D * 2;    // 64 KB: a resident 128-row tile
    static constexpr int TILE64 = STEP * D * 2;    // 32 KB: a step's 64-row tile
    // ---- dK / dV phase ----
    static constexpr int KV_OFF_K = 0;
    static constexpr int KV_OFF_V = KV_OFF_K + TILE128;       // V (dK pass), or slot 1's Q and dO (dV pass)
    static constexpr int KV_OFF_Q = KV_OFF_V + TILE128;       // slot 0's Q
    static constexpr int KV_OFF_DO = KV_OFF_Q + TILE64;       // slot 0's dO
    static constexpr int KV_OFF_LSE = KV_OFF_DO + TILE64;     // [2] x 64 floats
    static constexpr int KV_OFF_DELTA = KV_OFF_LSE + 512;     // [2] x 64 floats
    static constexpr int KV_OFF_OST = (KV_OFF_DELTA + 512 + 1023) / 1024 * 1024;  // epilogue staging
    static constexpr int KV_OFF_BAR = KV_OFF_OST + 128 * SW;
    static constexpr int KB_K_FULL = 0;       // K of a unit landed (TMA)
    static constexpr int KB_KV_EMPTY = 1;     // the unit's last Sᵀ and dPᵀ are done (commit)
    static constexpr int KB_QD_FULL = 2;      // [2] Q, dO, lse2, Δ of a step landed in slot b
    static constexpr int KB_QD_EMPTY = 4;     // [2] that step's products are done (commit)
    static constexpr int KB_S_FULL = 6;       // [2] Sᵀ (and dPᵀ in the dK pass) in TMEM (commit)
    static constexpr int KB_P_FULL = 8;       // [2] Pᵀ (dV pass) or dSᵀ (dK pass) written (every softmax thread)
    static constexpr int KB_ACC_FULL = 10;    // dV or dK of a unit complete (commit)
    static constexpr int KB_ACC_FREE = 11;    // that accumulator read out (128)
    static constexpr int KB_DRAIN = 12;
    static constexpr int KB_V_FULL = 13;      // V of a unit landed, after the dV pass (TMA)
    static constexpr int KB_DO_FULL = 14;     // dK pass: a step's dO landed (TMA)
    static constexpr int KB_DO_EMPTY = 15;    // dK pass: that step's dPᵀ is done (commit)
    static constexpr int KV_NUM_BARS = 16;
    // a step slot's Q and dO tiles (slot 1 lives where V goes)
    static __host__ __device__ constexpr uint32_t kv_q(uint32_t b) { return b ? KV_OFF_V : KV_OFF_Q; }
    static __host__ __device__ constexpr uint32_t kv_do(uint32_t b) { return b ? KV_OFF_V + TILE64 : KV_OFF_DO; }
    static constexpr int KV_SMEM_USED = KV_OFF_BAR + KV_NUM_BARS * 8;
    // ---- dQ phase ----
    static constexpr int Q_OFF_Q = 0;
    static constexpr int Q_OFF_DO = Q_OFF_Q + TILE128;
    static constexpr int Q_OFF_K = Q_OFF_DO + TILE128;
    static constexpr int Q_OFF_V = Q_OFF_K + TILE64;
    static constexpr int Q_OFF_OST = Q_OFF_V + TILE64;
    static constexpr int Q_OFF_BAR = Q_OFF_OST + 128 * SW;
    static constexpr int QB_QD_FULL = 0;      // Q, dO of a unit landed
    static constexpr int QB_QD_EMPTY = 1;     // the unit's last S and dP are done (commit)
    static constexpr int QB_KV_FULL = 2;      // K of a step landed
    static constexpr int QB_KV_EMPTY = 3;     // that step's products are done (commit)
    static constexpr int QB_S_FULL = 4;       // S and dP in TMEM (commit)
    static constexpr int QB_DS_FULL = 5;      // dS written (every softmax thread)
    static constexpr int QB_DQ_FULL = 6;      // dQ of a unit complete (commit)
    static constexpr int QB_DQ_FREE = 7;      // dQ read out (128)
    static constexpr int QB_DRAIN = 8;
    static constexpr int QB_V_FULL = 9;       // V of a step landed
    static constexpr int QB_V_EMPTY = 10;     // that step's dP is done (commit)
    static constexpr int Q_NUM_BARS = 11;
    static constexpr int Q_SMEM_USED = Q_OFF_BAR + Q_NUM_BARS * 8;
    static constexpr int OFF_MISC = ((KV_SMEM_USED > Q_SMEM_USED ? KV_SMEM_USED : Q_SMEM_USED) + 15) & ~15;
    static constexpr int SMEM_USED = OFF_MISC + 16;
    static constexpr int SMEM_BYTES = SMEM_USED + 1024;
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
    // tensor memory: two 64-column fp32 blocks (S / Sᵀ, dP / dPᵀ; P, dS packed
    // by each column group over the first half of its own columns) and one
    // 256-column accumulator
    static constexpr uint32_t TM_S = 0;
    static constexpr uint32_t TM_DP = 64;
    // dV pass: Sᵀ of slot b (slot 1 takes the dPᵀ block, unused in that pass)
    static __host__ __device__ constexpr uint32_t tm_slot(uint32_t b) { return b ? TM_DP : TM_S; }
    static constexpr uint32_t TM_ACC = 256;
    static constexpr uint32_t TMEM_COLS = 512;
    static_assert(TM_ACC + D <= TMEM_COLS, "tensor memory budget");

    static __device__ __forceinline__ uint32_t kv_bar_count(int i) {
        if (i >= KB_P_FULL && i < KB_P_FULL + 2) return 32 * WIDE_SOFTMAX_WARPS;
        return i == KB_ACC_FREE ? 128 : 1;
    }
    static __device__ __forceinline__ uint32_t q_bar_count(int i) {
        if (i == QB_DS_FULL) return 32 * WIDE_SOFTMAX_WARPS;
        return i == QB_DQ_FREE ? 128 : 1;
    }
};

// K-major operand of `rows` rows in 64-element (128-byte) swizzled chunks:
// descriptor start offset (16-byte units) of the 16-element K step kk
__device__ __forceinline__ uint32_t wide_kmaj(int kk, int rows) {
    return (uint32_t)(((kk / 4) * (rows * 128) + (kk % 4) * 32) >> 4);
}

// A 64-row step tile (rows r0 .. r0 + 63 of the 256-wide tensor) into shared
// memory: four 64-element column chunks of one 64-row box each.
__device__ __forceinline__ void wide_load64(uint32_t dst, const CUtensorMap* map, uint32_t bar, int r0, int h, int z,
                                            uint64_t pol) {
#pragma unroll
    for (int c = 0; c < 4; ++c) ptx::tma_load_4d(dst + c * (64 * 128), map, bar, c * 64, r0, h, z, pol);
}
// A resident 128-row tile: four column chunks of two 64-row boxes each.
__device__ __forceinline__ void wide_load128(uint32_t dst, const CUtensorMap* map, uint32_t bar, int r0, int h, int z,
                                             uint64_t pol) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        ptx::tma_load_4d(dst + c * (128 * 128), map, bar, c * 64, r0, h, z, pol);
        ptx::tma_load_4d(dst + c * (128 * 128) + 64 * 128, map, bar, c * 64, r0 + 64, h, z, pol);
    }
}

// ================================================================ dK / dV ===
// A unit's steps: per query head of the group, the 64-row halves of the
// query blocks from i0 on (causal: block j's keys are seen from block j on).
__device__ __forceinline__ void wide_step(const BwdUnit& w, int s, const BwdParams& p, int& hq, int& r0) {
    const int per_head = 2 * w.per_head;
    hq = w.hk * p.group + s / per_head;
    r0 = (w.i0 + (s % per_head) / 2) * 128 + (s % 2) * 64;
}

// Step slots: the dV pass alternates slots 0 and 1 (step s in slot s & 1),
// the dK pass uses slot 0.  Every role counts the fills of each slot;
// fill n of a slot completes phase n & 1 of its barriers.
template <bool CAUSAL, int VAR>
__device__ void wide_kv_producer(const CUtensorMap* tmK, const CUtensorMap* tmV, const CUtensorMap* tmQ,
                                 const CUtensorMap* tmDO, const BwdParams& p, uint32_t sbase, uint32_t bar0,
                                 const Ctl& ctl) {
    using T = WideTraits;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    const uint64_t pol_kv = ptx::policy_evict_first();
    const uint64_t pol_q = ptx::policy_evict_last();
    uint32_t uc = 0, vc = 0, n0 = 0, n1 = 0;  // fills of slots 0 and 1
    uint32_t nd = 0;                          // dO fills of the dK passes
    bool ok = true;
    bool withheld = false;
    // Q, dO, lse2, Δ of step s into slot b, once that slot's previous step is done
    auto fill = [&](const BwdUnit& w, int s, uint32_t b) -> bool {
        const uint32_t nb = b ? n1 : n0;
        if (nb >= 1 && !wait_phase(bar(T::KB_QD_EMPTY + b), (nb - 1) & 1u, ctl, SITE_B_QD_EMPTY)) return false;
        int hq, r0;
        wide_step(w, s, p, hq, r0);
        const uint32_t full = bar(T::KB_QD_FULL + b);
        ptx::mbar_arrive_expect_tx(full, 2 * T::TILE64 + 512);
        wide_load64(sbase + T::kv_q(b), tmQ, full, w.qrow0 + r0, hq, w.zc, pol_q);
        wide_load64(sbase + T::kv_do(b), tmDO, full, w.qrow0 + r0, hq, w.zc, pol_q);
        const int64_t row0 = ((int64_t)w.z * p.Hq + hq) * p.Tq * 128 + r0;
        ptx::bulk_load(sbase + T::KV_OFF_LSE + b * 256u, p.lse2 + row0, 256, full);
        ptx::bulk_load(sbase + T::KV_OFF_DELTA + b * 256u, p.delta + row0, 256, full);
        if (b) ++n1;
        else ++n0;
        return true;
    };
    // dK pass step s in slot 0: dO (read only by the step's dPᵀ) as soon as
    // the previous step's dPᵀ is done, then Q, lse2, Δ once the previous
    // step's accumulation is (it reads Q); the first step's dO waits for the
    // dV pass's last slot-0 accumulation, which read the dO buffer
    auto fill_dk = [&](const BwdUnit& w, int s) -> bool {
        int hq, r0;
        wide_step(w, s, p, hq, r0);
        if (s == 0) {
            if (n0 >= 1 && !wait_phase(bar(T::KB_QD_EMPTY), (n0 - 1) & 1u, ctl, SITE_B_QD_EMPTY)) return false;
        } else if (!wait_phase(bar(T::KB_DO_EMPTY), (nd - 1) & 1u, ctl, SITE_B_QD_EMPTY)) {
            return false;
        }
        ptx::mbar_arrive_expect_tx(bar(T::KB_DO_FULL), T::TILE64);
        wide_load64(sbase + T::kv_do(0), tmDO, bar(T::KB_DO_FULL), w.qrow0 + r0, hq, w.zc, pol_q);
        ++nd;
        if (n0 >= 1 && !wait_phase(bar(T::KB_QD_EMPTY), (n0 - 1) & 1u, ctl, SITE_B_QD_EMPTY)) return false;
        const uint32_t full = bar(T::KB_QD_FULL);
        ptx::mbar_arrive_expect_tx(full, T::TILE64 + 512);
        wide_load64(sbase + T::kv_q(0), tmQ, full, w.qrow0 + r0, hq, w.zc, pol_q);
        const int64_t row0 = ((int64_t)w.z * p.Hq + hq) * p.Tq * 128 + r0;
        ptx::bulk_load(sbase + T::KV_OFF_LSE, p.lse2 + row0, 256, full);
        ptx::bulk_load(sbase + T::KV_OFF_DELTA, p.delta + row0, 256, full);
        ++n0;
        return true;
    };
    for (int pos = blockIdx.x; ok && unit_at<CAUSAL>(pos) < p.nunits; pos += gridDim.x) {
        const BwdUnit w = bwd_unit<CAUSAL, VAR>(unit_at<CAUSAL>(pos), p);
        if (!unit_checked(w, p, ctl, SITE_CHECK_BWD_LOAD)) { ok = false; break; }
        if (w.nsteps == 0) continue;
        // K and the V region (slot 1, then V) are free once the previous
        // unit's last Sᵀ and dPᵀ are done
        if (uc > 0 && !wait_phase(bar(T::KB_KV_EMPTY), (uc - 1) & 1u, ctl, SITE_B_KV_EMPTY)) { ok = false; break; }
        if (p.inject_stall && blockIdx.x == 0 && uc == 0) {
            withheld = true;  // never issued: the issuer's wait for K must time out
        } else {
            ptx::mbar_arrive_expect_tx(bar(T::KB_K_FULL), T::TILE128);
            wide_load128(sbase + T::KV_OFF_K, tmK, bar(T::KB_K_FULL), w.krow0 + w.j * 128, w.hk, w.zc, pol_kv);
        }
        ++uc;
        const int steps = 2 * w.nsteps;  // >= 2: slot 1 is filled at least once
        for (int s = 0; ok && s < steps; ++s) ok = fill(w, s, (uint32_t)s & 1u);
        if (!ok) break;
        // V over slot 1, once its last dV step is done
        if (!wait_phase(bar(T::KB_QD_EMPTY + 1), (n1 - 1) & 1u, ctl, SITE_B_QD_EMPTY)) { ok = false; break; }
        ptx::mbar_arrive_expect_tx(bar(T::KB_V_FULL), T::TILE128);
        wide_load128(sbase + T::KV_OFF_V, tmV, bar(T::KB_V_FULL), w.krow0 + w.j * 128, w.hk, w.zc, pol_kv);
        ++vc;
        for (int s = 0; ok && s < steps; ++s) ok = fill_dk(w, s);
    }
    if (!ok) {
        // (the withheld copy never completes; its wait simply runs out)
        if (uc > 0) drain_phase(bar(T::KB_K_FULL), (uc - 1) & 1u, withheld && uc == 1 ? ctl.limit_ns / 64 : ctl.limit_ns);
        if (vc > 0) drain_phase(bar(T::KB_V_FULL), (vc - 1) & 1u, ctl.limit_ns);
        if (n0 > 0) drain_phase(bar(T::KB_QD_FULL), (n0 - 1) & 1u, ctl.limit_ns);
        if (nd > 0) drain_phase(bar(T::KB_DO_FULL), (nd - 1) & 1u, ctl.limit_ns);
        if (n1 > 0) drain_phase(bar(T::KB_QD_FULL + 1), (n1 - 1) & 1u, ctl.limit_ns);
    }
}

template <bool CAUSAL, bool BF16, int VAR>
__device__ void wide_kv_issuer(const BwdParams& p, uint32_t sbase, uint32_t bar0, uint32_t tmem, const Ctl& ctl) {
    using T = WideTraits;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    constexpr uint32_t ID_S = ptx::idesc_f16(128, 64, BF16, false, false);   // Sᵀ = K Qᵀ, dPᵀ = V dOᵀ (N = 64)
    constexpr uint32_t ID_ACC = ptx::idesc_f16(128, 256, BF16, false, true); // dV, dK: B MN-major (N = 256)
    constexpr uint32_t HI = ptx::smem_desc_hi(8 * T::SW, T::SWIZZLE_CODE);
    const uint32_t k_lo = ptx::smem_desc_lo(sbase + T::KV_OFF_K, 16);
    const uint32_t v_lo = ptx::smem_desc_lo(sbase + T::KV_OFF_V, 16);
    auto q_lo = [&](uint32_t b) { return ptx::smem_desc_lo(sbase + T::kv_q(b), 16); };
    auto do_lo = [&](uint32_t b) { return ptx::smem_desc_lo(sbase + T::kv_do(b), 16); };
    // MN-major views (LBO: the next 64-column chunk, 64 rows on)
    auto qmn_lo = [&](uint32_t b) { return ptx::smem_desc_lo(sbase + T::kv_q(b), 64 * T::SW); };
    auto domn_lo = [&](uint32_t b) { return ptx::smem_desc_lo(sbase + T::kv_do(b), 64 * T::SW); };
    uint32_t uc = 0, acc = 0, n0 = 0, n1 = 0;  // fills of slots 0 and 1 consumed
    uint32_t nd = 0;                           // dO fills of the dK passes consumed
    bool ok = true;
    // Sᵀ = K Qᵀ of the step in slot b into TMEM block tm, K = 256 in 16 steps
    auto issue_s = [&](uint32_t b, uint32_t tm) {
#pragma unroll
        for (int kk = 0; kk < 16; ++kk)
            ptx::mma_ss(tmem + tm, ptx::desc64(k_lo + wide_kmaj(kk, 128), HI),
                        ptx::desc64(q_lo(b) + wide_kmaj(kk, 64), HI), ID_S, kk > 0 ? 1u : 0u);
    };
    // acc += (Pᵀ or dSᵀ in TMEM block a) times (dO or Q of slot b); its
    // commit frees the slot and the block.  s: the step's place in its pass.
    auto accumulate = [&](uint32_t a, uint32_t b_lo, uint32_t b, int s, int steps) -> bool {
        if (s == 0 && acc > 0 && !wait_phase(bar(T::KB_ACC_FREE), (acc - 1) & 1u, ctl, SITE_B_ACC_FREE)) return false;
        ptx::tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
            ptx::mma_ts(tmem + T::TM_ACC, tmem + a + packed_col<WIDE_CW>(kk), ptx::desc64(b_lo + ((kk * 16 * T::SW) >> 4), HI), ID_ACC,
                        (s > 0 || kk > 0) ? 1u : 0u);
        ptx::tc_commit(bar(T::KB_QD_EMPTY + b));  // the step's Q, dO and TMEM block free
        if (s == steps - 1) {
            ptx::tc_commit(bar(T::KB_ACC_FULL));  // dV (dV pass) or dK (dK pass) of the unit complete
            ++acc;
        }
        return true;
    };
    for (int pos = blockIdx.x; ok && unit_at<CAUSAL>(pos) < p.nunits; pos += gridDim.x) {
        const BwdUnit w = bwd_unit<CAUSAL, VAR>(unit_at<CAUSAL>(pos), p);
        if (!unit_checked(w, p, ctl, SITE_CHECK_BWD_MMA)) { ok = false; break; }
        if (w.nsteps == 0) continue;
        if (!wait_phase(bar(T::KB_K_FULL), uc & 1u, ctl, SITE_B_KV_FULL)) { ok = false; break; }
        const int steps = 2 * w.nsteps;
        // dV pass: step s + 1's Sᵀ goes to the tensor core before step s's
        // accumulation (which waits for the softmax).  Its slot and TMEM
        // block were freed by step s - 1's accumulation, which the copies of
        // step s + 1 (QD_FULL) already waited for.
        int pend = -1;          // the step whose accumulation is still to issue
        uint32_t pend_n = 0;    // its fill count
        for (int s = 0; s <= steps && ok; ++s) {
            if (s < steps) {
                const uint32_t b = (uint32_t)s & 1u, nb = b ? n1++ : n0++;
                if (!wait_phase(bar(T::KB_QD_FULL + b), nb & 1u, ctl, SITE_B_QD_FULL)) { ok = false; break; }
                ptx::tc_fence_after();
                issue_s(b, T::tm_slot(b));
                ptx::tc_commit(bar(T::KB_S_FULL + b));
            }
            if (pend >= 0) {
                const uint32_t b = (uint32_t)pend & 1u;
                if (!wait_phase(bar(T::KB_P_FULL + b), pend_n & 1u, ctl, SITE_B_P_FULL) ||
                    !accumulate(T::tm_slot(b), domn_lo(b), b, pend, steps)) {
                    ok = false;
                    break;
                }
            }
            pend = s;
            pend_n = s < steps ? (((uint32_t)s & 1u) ? n1 : n0) - 1 : 0;
        }
        if (!ok) break;
        // dK pass in slot 0: needs V, loaded over slot 1 after the dV pass
        if (!wait_phase(bar(T::KB_V_FULL), uc & 1u, ctl, SITE_B_KV_FULL)) { ok = false; break; }
        for (int s = 0; s < steps; ++s) {
            const uint32_t nb = n0++;
            if (!wait_phase(bar(T::KB_QD_FULL), nb & 1u, ctl, SITE_B_QD_FULL)) { ok = false; break; }
            ptx::tc_fence_after();
            issue_s(0, T::TM_S);
            if (!wait_phase(bar(T::KB_DO_FULL), nd & 1u, ctl, SITE_B_QD_FULL)) { ok = false; break; }
            ++nd;
            ptx::tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 16; ++kk)
                ptx::mma_ss(tmem + T::TM_DP, ptx::desc64(v_lo + wide_kmaj(kk, 128), HI),
                            ptx::desc64(do_lo(0) + wide_kmaj(kk, 64), HI), ID_S, kk > 0 ? 1u : 0u);
            ptx::tc_commit(bar(T::KB_S_FULL));
            ptx::tc_commit(bar(T::KB_DO_EMPTY));  // the step's dO is free once its dPᵀ is done
            // the unit's last Sᵀ and dPᵀ were its last reads of K and V: the
            // next unit's K (and slot 1, over V) may land during the last dK step
            if (s + 1 == steps) ptx::tc_commit(bar(T::KB_KV_EMPTY));
            if (!wait_phase(bar(T::KB_P_FULL), nb & 1u, ctl, SITE_B_P_FULL) ||
                !accumulate(T::TM_DP, qmn_lo(0), 0, s, steps)) {
                ok = false;
                break;
            }
        }
        if (!ok) break;
        ++uc;
    }
    // every MMA of this phase completes before the dQ phase reuses shared memory
    ptx::tc_commit(bar(T::KB_DRAIN));
    drain_phase(bar(T::KB_DRAIN), 0u, ctl.limit_ns);
}

// Thread = key (TMEM lane); column group h takes the step's queries h*CW ..
// h*CW + CW - 1.  dV pass: Pᵀ over the first half of the group's columns of
// the step's Sᵀ block; dK pass: Pᵀ in registers, dSᵀ = Pᵀ ∘ (dPᵀ − Δ) over the
// first half of the group's columns of dPᵀ.  P and dS are rounded to the
// input type (the products' operands).
template <bool CAUSAL, bool BF16, int VAR>
__device__ void wide_kv_softmax(const BwdParams& p, uint32_t sbase, uint32_t bar0, uint32_t tmem, int h,
                                const Ctl& ctl) {
    static_assert(WIDE_CW == 32, "one 32-column TMEM load per group");
    using T = WideTraits;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    const int quad = (threadIdx.x / 32) % 4;
    const int row = quad * 32 + threadIdx.x % 32;  // key within the block
    const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
    const float c = p.scale_log2;
    uint32_t n0 = 0, n1 = 0;  // fills of slots 0 and 1 consumed
    for (int pos = blockIdx.x; unit_at<CAUSAL>(pos) < p.nunits; pos += gridDim.x) {
        const BwdUnit w = bwd_unit<CAUSAL, VAR>(unit_at<CAUSAL>(pos), p);
        if (!unit_checked(w, p, ctl, SITE_CHECK_BWD_SOFTMAX)) return;
        const int key = w.j * 128 + row;
        const int steps = 2 * w.nsteps;
        for (int pass = 0; pass < 2; ++pass) {
            for (int s = 0; s < steps; ++s) {
                const uint32_t b = pass == 0 ? (uint32_t)s & 1u : 0u, ph = (b ? n1++ : n0++) & 1u;
                int hq, r0;
                wide_step(w, s, p, hq, r0);
                // lse2 and Δ of the step's queries arrive with Qᵢ (TMA); the
                // slot is refilled only after this step's P_FULL
                if (!warp_wait_phase(bar(T::KB_QD_FULL + b), ph, ctl, SITE_B_QD_FULL)) return;
                if (!warp_wait_phase(bar(T::KB_S_FULL + b), ph, ctl, SITE_B_S_FULL)) return;
                ptx::tc_fence_after();
                const uint32_t lse_a = sbase + T::KV_OFF_LSE + b * 256u + 4u * (h * WIDE_CW);
                const uint32_t del_a = sbase + T::KV_OFF_DELTA + b * 256u + 4u * (h * WIDE_CW);
                const uint32_t tm_s = (pass == 0 ? T::tm_slot(b) : T::TM_S) + h * WIDE_CW;
                // causal: only the diagonal block has keys after queries (key > query -> P = 0)
                const bool diag = CAUSAL && r0 / 128 == w.j;
                const int q0 = r0 + h * WIDE_CW;  // the group's first query
                // variants: d = query − key, masked per pair only in a step not
                // wholly kept (window sides, causal rule, keys past the
                // sequence's); ALiBi adds slope2·|d| (log2 units)
                const bool full = VAR == 0 || var_block_kept<CAUSAL>(r0 - (w.j * 128 + 127), r0 + 63 - w.j * 128,
                                                                     w.j * 128 + 128, w.nk, p);
                const float slope2 = bwd_alibi(VAR) ? -__ldg(p.alibi + hq) * 1.4426950408889634f : 0.f;
                uint32_t pk[WIDE_CW / 2];
                {
                    uint32_t a[32];
                    ptx::tmem_ld32(tmem + lane_addr + tm_s, a);
#pragma unroll
                    for (int x = 0; x < 32; x += 2) {
                        float l0, l1;
                        asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(l0), "=f"(l1) : "r"(lse_a + 4u * x));
                        float e0 = fmaf(__uint_as_float(a[x]), c, -l0);
                        float e1 = fmaf(__uint_as_float(a[x + 1]), c, -l1);
                        if constexpr (VAR == 0) {
                            if (diag && key > q0 + x) e0 = -INFINITY;
                            if (diag && key > q0 + x + 1) e1 = -INFINITY;
                        } else {
                            const int d0 = q0 + x - key;
                            if constexpr (bwd_alibi(VAR)) {
                                e0 = fmaf(slope2, fabsf((float)d0), e0);
                                e1 = fmaf(slope2, fabsf((float)(d0 + 1)), e1);
                            }
                            if (!full) {
                                if (var_dropped<CAUSAL>(d0, key, w.nk, p)) e0 = -INFINITY;
                                if (var_dropped<CAUSAL>(d0 + 1, key, w.nk, p)) e1 = -INFINITY;
                            }
                        }
                        pk[x / 2] = pack2<BF16>(ptx::ex2(e0), ptx::ex2(e1));
                    }
                }
                if (pass == 0) {
                    ptx::tmem_st16(tmem + lane_addr + tm_s, pk);
                } else {
                    const uint32_t tm_dp = T::TM_DP + h * WIDE_CW;
                    uint32_t a[32];
                    ptx::tmem_ld32(tmem + lane_addr + tm_dp, a);
                    uint32_t ds[16];
#pragma unroll
                    for (int x = 0; x < 16; ++x) {
                        float d0, d1;
                        asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(d0), "=f"(d1) : "r"(del_a + 8u * x));
                        const float2 pp = unpack2<BF16>(pk[x]);  // dS uses the rounded P
                        ds[x] = pack2<BF16>(pp.x * (__uint_as_float(a[2 * x]) - d0),
                                            pp.y * (__uint_as_float(a[2 * x + 1]) - d1));
                    }
                    ptx::tmem_st16(tmem + lane_addr + tm_dp, ds);
                }
                ptx::tmem_wait_st();
                ptx::tc_fence_before();
                ptx::mbar_arrive(bar(T::KB_P_FULL + b));
            }
        }
    }
}

// Thread = key: dV, then dK (times scale), read out, released, stored; a
// unit no query sees gets zeros.
template <bool CAUSAL, bool BF16, int VAR>
__device__ void wide_kv_epilogue(const CUtensorMap* tmDK, const CUtensorMap* tmDV, const BwdParams& p, uint32_t sbase,
                                 uint32_t bar0, uint32_t tmem, const Ctl& ctl) {
    using T = WideTraits;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    const int quad = (threadIdx.x / 32) % 4;
    const int row = quad * 32 + threadIdx.x % 32;
    const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
    const uint32_t stage = sbase + T::KV_OFF_OST + (uint32_t)quad * 32u * T::SW;
    auto drain = [&]() {
        if (threadIdx.x % 32 == 0) ptx::bulk_wait_all();
    };
    uint32_t acc = 0;
    for (int pos = blockIdx.x; unit_at<CAUSAL>(pos) < p.nunits; pos += gridDim.x) {
        const BwdUnit w = bwd_unit<CAUSAL, VAR>(unit_at<CAUSAL>(pos), p);
        if (!unit_checked(w, p, ctl, SITE_CHECK_BWD_EPILOGUE)) {
            drain();
            return;
        }
        const int key = w.j * 128 + row;  // within the unit's sequence
        uint8_t* dk_row = reinterpret_cast<uint8_t*>(p.dk) +
                          2 * ((int64_t)w.zc * p.sdk_z + (int64_t)w.hk * p.sdk_h + (int64_t)(w.krow0 + key) * p.sdk_n);
        uint8_t* dv_row = reinterpret_cast<uint8_t*>(p.dv) +
                          2 * ((int64_t)w.zc * p.sdv_z + (int64_t)w.hk * p.sdv_h + (int64_t)(w.krow0 + key) * p.sdv_n);
        if (w.nsteps == 0) {
            if (key < w.nk) {
#pragma unroll
                for (int x = 0; x < 256 / 8; ++x) {
                    reinterpret_cast<uint4*>(dk_row)[x] = make_uint4(0, 0, 0, 0);
                    reinterpret_cast<uint4*>(dv_row)[x] = make_uint4(0, 0, 0, 0);
                }
            }
            continue;
        }
        const int key0 = w.j * 128 + 32 * quad;
        for (int pass = 0; pass < 2; ++pass, ++acc) {
            if (!warp_wait_phase(bar(T::KB_ACC_FULL), acc & 1u, ctl, SITE_B_ACC_FULL)) {
                drain();
                return;
            }
            ptx::tc_fence_after();
            const auto release = [&]() {
                ptx::tc_fence_before();
                ptx::mbar_arrive(bar(T::KB_ACC_FREE));
            };
            // a 32-row box past the end of a packed sequence goes row by row
            if (!bwd_varlen(VAR) || p.cu_k == nullptr || key0 + 32 <= w.nk) {
                tma_store_rows<256, T::SW, BF16>(tmem + lane_addr + T::TM_ACC, pass == 0 ? 1.f : p.scale, stage,
                                                 pass == 0 ? tmDV : tmDK, w.krow0 + key0, w.hk, w.zc, key0 < w.nk,
                                                 release);
            } else {
                direct_store_row<256, BF16>(tmem + lane_addr + T::TM_ACC, pass == 0 ? 1.f : p.scale,
                                            pass == 0 ? dv_row : dk_row, key < w.nk, release);
            }
        }
    }
    drain();
}

// ===================================================================== dQ ===
template <bool CAUSAL, int VAR>
__device__ void wide_q_producer(const CUtensorMap* tmK, const CUtensorMap* tmV, const CUtensorMap* tmQ,
                                const CUtensorMap* tmDO, const BwdParams& p, uint32_t sbase, uint32_t bar0,
                                const Ctl& ctl, int first) {
    using T = WideTraits;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    const uint64_t pol_q = ptx::policy_evict_first();
    const uint64_t pol_kv = ptx::policy_evict_last();
    uint32_t uc = 0, g = 0, gv = 0;  // fills of Q/dO, K and V
    bool ok = true;
    for (int pos = first; ok && unit_at<CAUSAL>(pos) < p.nunits_q; pos += gridDim.x) {
        const DqUnit w = dq_unit<CAUSAL, VAR>(unit_at<CAUSAL>(pos), p);
        if (!unit_checked(w, p, ctl, SITE_CHECK_BWD_LOAD)) { ok = false; break; }
        if (w.skip) continue;
        if (uc > 0 && !wait_phase(bar(T::QB_QD_EMPTY), (uc - 1) & 1u, ctl, SITE_B_QD_EMPTY)) { ok = false; break; }
        ptx::mbar_arrive_expect_tx(bar(T::QB_QD_FULL), 2 * T::TILE128);
        wide_load128(sbase + T::Q_OFF_Q, tmQ, bar(T::QB_QD_FULL), w.qrow0 + w.i * 128, w.hq, w.zc, pol_q);
        wide_load128(sbase + T::Q_OFF_DO, tmDO, bar(T::QB_QD_FULL), w.qrow0 + w.i * 128, w.hq, w.zc, pol_q);
        ++uc;
        const int steps = 2 * w.nkv;  // 64-key steps
        for (int s = 0; s < steps; ++s, ++g) {
            // V (read only by the step's dP) once the previous step's dP is
            // done, then K once the previous step's dQ product (it reads K) is
            if (gv >= 1 && !wait_phase(bar(T::QB_V_EMPTY), (gv - 1) & 1u, ctl, SITE_B_KV_EMPTY)) { ok = false; break; }
            ptx::mbar_arrive_expect_tx(bar(T::QB_V_FULL), T::TILE64);
            wide_load64(sbase + T::Q_OFF_V, tmV, bar(T::QB_V_FULL), w.krow0 + w.j0 * 128 + s * 64, w.hk, w.zc, pol_kv);
            ++gv;
            if (g >= 1 && !wait_phase(bar(T::QB_KV_EMPTY), (g - 1) & 1u, ctl, SITE_B_KV_EMPTY)) { ok = false; break; }
            ptx::mbar_arrive_expect_tx(bar(T::QB_KV_FULL), T::TILE64);
            wide_load64(sbase + T::Q_OFF_K, tmK, bar(T::QB_KV_FULL), w.krow0 + w.j0 * 128 + s * 64, w.hk, w.zc, pol_kv);
        }
    }
    if (!ok) {
        if (uc > 0) drain_phase(bar(T::QB_QD_FULL), (uc - 1) & 1u, ctl.limit_ns);
        if (g > 0) drain_phase(bar(T::QB_KV_FULL), (g - 1) & 1u, ctl.limit_ns);
        if (gv > 0) drain_phase(bar(T::QB_V_FULL), (gv - 1) & 1u, ctl.limit_ns);
    }
}

template <bool CAUSAL, bool BF16, int VAR>
__device__ void wide_q_issuer(const BwdParams& p, uint32_t sbase, uint32_t bar0, uint32_t tmem, const Ctl& ctl,
                              int first) {
    using T = WideTraits;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    constexpr uint32_t ID_S = ptx::idesc_f16(128, 64, BF16, false, false);    // S = Q Kᵀ, dP = dO Vᵀ (N = 64)
    constexpr uint32_t ID_DQ = ptx::idesc_f16(128, 256, BF16, false, true);   // dQ += dS K (K MN-major)
    constexpr uint32_t HI = ptx::smem_desc_hi(8 * T::SW, T::SWIZZLE_CODE);
    const uint32_t q_lo = ptx::smem_desc_lo(sbase + T::Q_OFF_Q, 16);
    const uint32_t do_lo = ptx::smem_desc_lo(sbase + T::Q_OFF_DO, 16);
    const uint32_t k_lo = ptx::smem_desc_lo(sbase + T::Q_OFF_K, 16);
    const uint32_t v_lo = ptx::smem_desc_lo(sbase + T::Q_OFF_V, 16);
    const uint32_t kmn_lo = ptx::smem_desc_lo(sbase + T::Q_OFF_K, 64 * T::SW);
    uint32_t uc = 0, g = 0;
    bool ok = true;
    for (int pos = first; ok && unit_at<CAUSAL>(pos) < p.nunits_q; pos += gridDim.x) {
        const DqUnit w = dq_unit<CAUSAL, VAR>(unit_at<CAUSAL>(pos), p);
        if (!unit_checked(w, p, ctl, SITE_CHECK_BWD_MMA)) { ok = false; break; }
        if (w.skip) continue;
        if (!wait_phase(bar(T::QB_QD_FULL), uc & 1u, ctl, SITE_B_QD_FULL)) { ok = false; break; }
        const int steps = 2 * w.nkv;
        for (int s = 0; s < steps; ++s, ++g) {
            if (!wait_phase(bar(T::QB_KV_FULL), g & 1u, ctl, SITE_B_KV_FULL)) { ok = false; break; }
            ptx::tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 16; ++kk)
                ptx::mma_ss(tmem + T::TM_S, ptx::desc64(q_lo + wide_kmaj(kk, 128), HI),
                            ptx::desc64(k_lo + wide_kmaj(kk, 64), HI), ID_S, kk > 0 ? 1u : 0u);
            if (!wait_phase(bar(T::QB_V_FULL), g & 1u, ctl, SITE_B_KV_FULL)) { ok = false; break; }
            ptx::tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 16; ++kk)
                ptx::mma_ss(tmem + T::TM_DP, ptx::desc64(do_lo + wide_kmaj(kk, 128), HI),
                            ptx::desc64(v_lo + wide_kmaj(kk, 64), HI), ID_S, kk > 0 ? 1u : 0u);
            ptx::tc_commit(bar(T::QB_S_FULL));
            ptx::tc_commit(bar(T::QB_V_EMPTY));  // the step's V is free once its dP is done
            // the unit's last S and dP were its last reads of Q and dO
            if (s + 1 == steps) ptx::tc_commit(bar(T::QB_QD_EMPTY));
            if (!wait_phase(bar(T::QB_DS_FULL), g & 1u, ctl, SITE_B_DS_FULL)) { ok = false; break; }
            if (s == 0 && uc > 0 && !wait_phase(bar(T::QB_DQ_FREE), (uc - 1) & 1u, ctl, SITE_B_DQ_FREE)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                ptx::mma_ts(tmem + T::TM_ACC, tmem + T::TM_S + packed_col<WIDE_CW>(kk), ptx::desc64(kmn_lo + ((kk * 16 * T::SW) >> 4), HI),
                            ID_DQ, (s > 0 || kk > 0) ? 1u : 0u);
            ptx::tc_commit(bar(T::QB_KV_EMPTY));  // K of the step free
        }
        if (!ok) break;
        ptx::tc_commit(bar(T::QB_DQ_FULL));
        ++uc;
    }
    if (!ok) {
        ptx::tc_commit(bar(T::QB_DRAIN));
        drain_phase(bar(T::QB_DRAIN), 0u, ctl.limit_ns);
    }
}

// Thread = query (TMEM lane); column group h takes the step's keys h*CW ..
// h*CW + CW - 1: P = 2^(S·c − lse2), dS = P ∘ (dP − Δ) over the first half of
// the group's columns of S.
template <bool CAUSAL, bool BF16, int VAR>
__device__ void wide_q_softmax(const BwdParams& p, uint32_t bar0, uint32_t tmem, int h, const Ctl& ctl, int first) {
    using T = WideTraits;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    const int quad = (threadIdx.x / 32) % 4;
    const int row = quad * 32 + threadIdx.x % 32;
    const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
    const float c = p.scale_log2;
    uint32_t g = 0;
    for (int pos = first; unit_at<CAUSAL>(pos) < p.nunits_q; pos += gridDim.x) {
        const DqUnit w = dq_unit<CAUSAL, VAR>(unit_at<CAUSAL>(pos), p);
        if (!unit_checked(w, p, ctl, SITE_CHECK_BWD_SOFTMAX)) return;
        if (w.skip) continue;
        const int64_t r = ((int64_t)w.z * p.Hq + w.hq) * p.Tq * 128 + (int64_t)w.i * 128 + row;
        const float l2 = __ldg(p.lse2 + r), dl = __ldg(p.delta + r);
        const float slope2 = bwd_alibi(VAR) ? -__ldg(p.alibi + w.hq) * 1.4426950408889634f : 0.f;
        const int q = w.i * 128 + row;
        const int steps = 2 * w.nkv;
        for (int s = 0; s < steps; ++s, ++g) {
            if (!warp_wait_phase(bar(T::QB_S_FULL), g & 1u, ctl, SITE_B_S_FULL)) return;
            ptx::tc_fence_after();
            const int kb = w.j0 * 128 + s * 64;         // the step's first key
            const bool diag = CAUSAL && kb / 128 == w.i;  // keys after the query only on the diagonal block
            const int k0 = kb + h * WIDE_CW;              // the group's first key
            // variants: d = query − key, masked per pair only in a step not wholly kept
            const bool full = VAR == 0 || var_block_kept<CAUSAL>(w.i * 128 - (kb + 63), w.i * 128 + 127 - kb, kb + 64,
                                                                 w.nk, p);
            uint32_t sa[32], da[32];
            ptx::tmem_ld32_issue(tmem + lane_addr + T::TM_S + h * WIDE_CW, sa);
            ptx::tmem_ld32_issue(tmem + lane_addr + T::TM_DP + h * WIDE_CW, da);
            ptx::tmem_wait_ld();
            ptx::reg_fence32(sa);
            ptx::reg_fence32(da);
            uint32_t ds[16];
#pragma unroll
            for (int x = 0; x < 16; ++x) {
                const int k = 2 * x;
                float e0 = fmaf(__uint_as_float(sa[k]), c, -l2);
                float e1 = fmaf(__uint_as_float(sa[k + 1]), c, -l2);
                if constexpr (VAR == 0) {
                    if (diag && k0 + k > q) e0 = -INFINITY;
                    if (diag && k0 + k + 1 > q) e1 = -INFINITY;
                } else {
                    const int d0 = q - (k0 + k);
                    if constexpr (bwd_alibi(VAR)) {
                        e0 = fmaf(slope2, fabsf((float)d0), e0);
                        e1 = fmaf(slope2, fabsf((float)(d0 - 1)), e1);
                    }
                    if (!full) {
                        if (var_dropped<CAUSAL>(d0, k0 + k, w.nk, p)) e0 = -INFINITY;
                        if (var_dropped<CAUSAL>(d0 - 1, k0 + k + 1, w.nk, p)) e1 = -INFINITY;
                    }
                }
                const float2 pp = unpack2<BF16>(pack2<BF16>(ptx::ex2(e0), ptx::ex2(e1)));  // P rounded as in dV
                ds[x] = pack2<BF16>(pp.x * (__uint_as_float(da[k]) - dl), pp.y * (__uint_as_float(da[k + 1]) - dl));
            }
            ptx::tmem_st16(tmem + lane_addr + T::TM_S + h * WIDE_CW, ds);
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(T::QB_DS_FULL));
        }
    }
}

// Thread = query: dQ (times scale) read out, released, stored.
template <bool CAUSAL, bool BF16, int VAR>
__device__ void wide_q_epilogue(const CUtensorMap* tmDQ, const BwdParams& p, uint32_t sbase, uint32_t bar0,
                                uint32_t tmem, const Ctl& ctl, int first) {
    using T = WideTraits;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    const int quad = (threadIdx.x / 32) % 4;
    const int row = quad * 32 + threadIdx.x % 32;  // query within the block
    const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
    const uint32_t stage = sbase + T::Q_OFF_OST + (uint32_t)quad * 32u * T::SW;
    auto drain = [&]() {
        if (threadIdx.x % 32 == 0) ptx::bulk_wait_all();
    };
    uint32_t uc = 0;
    for (int pos = first; unit_at<CAUSAL>(pos) < p.nunits_q; pos += gridDim.x) {
        const DqUnit w = dq_unit<CAUSAL, VAR>(unit_at<CAUSAL>(pos), p);
        if (!unit_checked(w, p, ctl, SITE_CHECK_BWD_EPILOGUE)) {
            drain();
            return;
        }
        if (w.skip) continue;
        if (!warp_wait_phase(bar(T::QB_DQ_FULL), uc & 1u, ctl, SITE_B_DQ_FULL)) {
            drain();
            return;
        }
        ptx::tc_fence_after();
        const int q0 = w.i * 128 + 32 * quad;
        const auto release = [&]() {
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(T::QB_DQ_FREE));
        };
        if (!bwd_varlen(VAR) || p.cu_q == nullptr || q0 + 32 <= w.nq) {
            tma_store_rows<256, T::SW, BF16>(tmem + lane_addr + T::TM_ACC, p.scale, stage, tmDQ, w.qrow0 + q0, w.hq,
                                             w.zc, q0 < w.nq, release);
        } else {
            const int qr = w.i * 128 + row;
            uint8_t* dq_row = reinterpret_cast<uint8_t*>(p.dq) +
                              2 * ((int64_t)w.zc * p.sdq_z + (int64_t)w.hq * p.sdq_h + (int64_t)(w.qrow0 + qr) * p.sdq_n);
            direct_store_row<256, BF16>(tmem + lane_addr + T::TM_ACC, p.scale, dq_row, qr < w.nq, release);
        }
        ++uc;
    }
    drain();
}

// ================================================================ fused ======
// dK/dV units (positions c, c + grid, ...) then dQ units from position
// grid - 1 - c on, in the same shared memory and TMEM, as for the smaller
// head dims.
template <bool CAUSAL, bool BF16, int VAR = 0>
__global__ void __launch_bounds__(WIDE_THREADS, 1)
    fa_bwd_wide_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
                       const __grid_constant__ CUtensorMap tmDK, const __grid_constant__ CUtensorMap tmDV,
                       const __grid_constant__ CUtensorMap tmDQ, const BwdParams p) {
    using T = WideTraits;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = nullptr;
    if (!bwd_smem_base(smem_raw, T::SMEM_USED, T::SMEM_BYTES, p, smem)) return;
    const uint32_t sbase = ptx::smem_addr(smem);
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + T::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + T::OFF_MISC + 4);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    const uint32_t kbar0 = sbase + T::KV_OFF_BAR;
    if (threadIdx.x == 0) {
        for (int i = 0; i < T::KV_NUM_BARS; ++i) ptx::mbar_init(kbar0 + 8u * i, T::kv_bar_count(i));
        *abort_flag = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tmK);
        ptx::prefetch_tmap(&tmV);
        ptx::prefetch_tmap(&tmQ);
        ptx::prefetch_tmap(&tmDO);
        ptx::prefetch_tmap(&tmDK);
        ptx::prefetch_tmap(&tmDV);
        ptx::prefetch_tmap(&tmDQ);
    }
    constexpr int W_EPI = WIDE_SOFTMAX_WARPS, W_PRODUCER = W_EPI + 4, W_ISSUER = W_EPI + 5;
    if (warp == W_ISSUER) {
        ptx::tmem_alloc(ptx::smem_addr(const_cast<uint32_t*>(tmem_slot)), T::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const Ctl ctl{abort_flag, p.status, p.wait_limit_ns};
    ptx::grid_dependency_wait();
    ptx::grid_launch_dependents();
    if (warp < W_EPI) {
        wide_kv_softmax<CAUSAL, BF16, VAR>(p, sbase, kbar0, tmem, warp / 4, ctl);
    } else if (warp < W_PRODUCER) {
        wide_kv_epilogue<CAUSAL, BF16, VAR>(&tmDK, &tmDV, p, sbase, kbar0, tmem, ctl);
    } else if (warp == W_PRODUCER) {
        if (lane == 0) wide_kv_producer<CAUSAL, VAR>(&tmK, &tmV, &tmQ, &tmDO, p, sbase, kbar0, ctl);
    } else {
        if (lane == 0) wide_kv_issuer<CAUSAL, BF16, VAR>(p, sbase, kbar0, tmem, ctl);
    }
    ptx::tc_fence_before();
    __syncthreads();

    if (*abort_flag == 0) {
        const uint32_t qbar0 = sbase + T::Q_OFF_BAR;
        if (threadIdx.x == 0) {
            for (int i = 0; i < T::Q_NUM_BARS; ++i) ptx::mbar_init(qbar0 + 8u * i, T::q_bar_count(i));
            ptx::fence_mbar_init();
        }
        __syncthreads();
        ptx::tc_fence_after();
        const int first = (int)gridDim.x - 1 - (int)blockIdx.x;
        if (warp < W_EPI) {
            wide_q_softmax<CAUSAL, BF16, VAR>(p, qbar0, tmem, warp / 4, ctl, first);
        } else if (warp < W_PRODUCER) {
            wide_q_epilogue<CAUSAL, BF16, VAR>(&tmDQ, p, sbase, qbar0, tmem, ctl, first);
        } else if (warp == W_PRODUCER) {
            if (lane == 0) wide_q_producer<CAUSAL, VAR>(&tmK, &tmV, &tmQ, &tmDO, p, sbase, qbar0, ctl, first);
        } else {
            if (lane == 0) wide_q_issuer<CAUSAL, BF16, VAR>(p, sbase, qbar0, tmem, ctl, first);
        }
        ptx::tc_fence_before();
        __syncthreads();
    }
    if (warp == W_ISSUER) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, T::TMEM_COLS);
    }
}

}  // namespace fa
