// Attention backward for sm_103a: gradients dQ, dK, dV of the fused forward
// from the saved log-sum-exp, with the score and probability blocks rebuilt
// on chip (blog "把 FlashAttention 搬上昇腾：Triton-Ascend CV Pipeline 优化实战",
// section 二: recompute P from the lse, dP, dS, then dQ / dK / dV; "Write
// Triton Attention Kernel", step 8 and Correctness requirements: the backward
// needs lse = m + log l).
//
// One unit of work is one block of 128 keys of one key/value head; a
// persistent CTA walks units, and for each loops over every query block of
// every query head of the GQA group (from the diagonal block on, when
// causal).  Per step (query block i of head hq), with keys as TMEM lanes:
//     Sᵀ  = K Qᵢᵀ                       (tcgen05, both from shared memory)
//     Pᵀ  = 2^(Sᵀ·scale·log2e − lse2ᵢ)   (softmax warps; -> TMEM as fp16/bf16)
//     dPᵀ = V dOᵢᵀ
//     dV += Pᵀ dOᵢ                       (A = Pᵀ from TMEM)
//     dSᵀ = Pᵀ ∘ (dPᵀ − Δᵢ)               (softmax warps; -> shared memory)
//     dK += dSᵀ Qᵢ                       (A = dSᵀ, K-major)
//     dQᵢ = dS K                         (A = dSᵀ read MN-major; -> fp32 adds
//                                         into the dQ accumulator in global)
// dK and dV stay in TMEM for the whole unit and are written once (dK times
// scale); dQ = scale · accumulator is converted by a last kernel.  Δ =
// rowsum(dO ∘ O) and the base-2 lse come from a first kernel.
//
// Warps: 0-3 and 4-7 the two column halves of each 128x128 block (thread =
// key = TMEM lane), 8-11 the epilogue (dQ adds, dK and dV stores; thread =
// TMEM lane), 12 the TMA producer, 13 the MMA issuer.  Every wait is bounded
// as in the forward kernel.  Head dims 16 to 128 (TMEM holds Sᵀ/Pᵀ, dPᵀ/dQ,
// dV and dK: 256 + 2D columns).
#pragma once

#include "fa_fwd_kernel.cuh"

namespace fa {

constexpr int BWD_THREADS = 14 * 32;

// two fp16 / bf16 values -> float2 (exact)
template <bool BF16>
__device__ __forceinline__ float2 unpack2(uint32_t w) {
    if constexpr (BF16) return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
    else return __half22float2(*reinterpret_cast<const __half2*>(&w));
}

template <int D_>
struct BwdTraits {
    static constexpr int D = D_;
    static_assert(D <= 128, "the backward keeps dK and dV in TMEM: D <= 128");
    static constexpr int BN = 128;                            // keys per unit
    static constexpr int SW = D * 2 >= 128 ? 128 : D * 2;      // bytes per swizzled row chunk of Q, K, V, dO
    static constexpr int SWE = SW / 2;
    static constexpr int NCHUNK = D / SWE;
    static constexpr uint32_t SWIZZLE_CODE = SW == 128 ? 2u : SW == 64 ? 4u : 6u;
    static constexpr int TILE = 128 * D * 2;                  // one 128-row tile of Q, K, V or dO
    static constexpr int DS_BYTES = 128 * 128 * 2;            // dSᵀ: 128 keys x 128 queries, 128-B swizzle
    // shared memory
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = OFF_K + TILE;
    static constexpr int OFF_Q = OFF_V + TILE;                // [2]
    static constexpr int OFF_DO = OFF_Q + 2 * TILE;           // [2]
    static constexpr int OFF_DS = OFF_DO + 2 * TILE;
    static constexpr int OFF_LSE = OFF_DS + DS_BYTES;         // [2] x 128 floats
    static constexpr int OFF_DELTA = OFF_LSE + 2 * 512;       // [2] x 128 floats
    static constexpr int OFF_BAR = OFF_DELTA + 2 * 512;
    // barriers
    static constexpr int B_KV_FULL = 0;       // K, V of a unit landed (TMA)
    static constexpr int B_KV_EMPTY = 1;      // the unit's MMAs are done (commit)
    static constexpr int B_QD_FULL = 2;       // [2] Q, dO, lse2, Δ of a step landed (TMA)
    static constexpr int B_QD_EMPTY = 4;      // [2] that step's MMAs are done (commit)
    static constexpr int B_S_FULL = 6;        // Sᵀ in TMEM (commit)
    static constexpr int B_DP_FULL = 7;       // dPᵀ in TMEM (commit)
    static constexpr int B_P_FULL = 8;        // Pᵀ written to TMEM (256)
    static constexpr int B_DS_FULL = 9;       // dSᵀ written to shared memory (256)
    static constexpr int B_DQ_FULL = 10;      // dQ partial in TMEM; dSᵀ buffer free (commit)
    static constexpr int B_DQ_FREE = 11;      // dQ partial read out of TMEM (128)
    static constexpr int B_ACC_FULL = 12;     // dK, dV of a unit complete (commit)
    static constexpr int B_ACC_FREE = 13;     // dK, dV read out of TMEM (128)
    static constexpr int B_DRAIN = 14;        // issuer teardown
    static constexpr int NUM_BARS = 15;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
    static constexpr int SMEM_USED = OFF_MISC + 16;
    // + slack to align the base to 1024 bytes where it fits (D = 128 fills
    // the 227 KB; there the base must already be aligned, which the kernel checks)
    static constexpr int SMEM_BYTES = SMEM_USED + 1024 <= 227 * 1024 ? SMEM_USED + 1024 : SMEM_USED;
    static_assert(SMEM_USED <= 227 * 1024, "shared memory budget");
    // TMEM columns
    static constexpr uint32_t TM_S = 0;                       // Sᵀ (fp32); Pᵀ over columns 0-31 and 64-95
    static constexpr uint32_t TM_DP = 128;                    // dPᵀ (fp32), then the dQ partial (D columns)
    static constexpr uint32_t TM_DV = 256;
    static constexpr uint32_t TM_DK = 256 + D;
    static constexpr uint32_t TMEM_COLS = 512;

    static __device__ __forceinline__ uint32_t bar_count(int i) {
        if (i == B_P_FULL || i == B_DS_FULL) return 256;
        if (i == B_DQ_FREE || i == B_ACC_FREE) return 128;
        return 1;
    }
};

// Unit u: key block j (ascending: with a causal mask the first key blocks
// have the most query blocks), then z, kv head.  Its steps run over the
// group's query heads and, per head, the query blocks from i0 on.
struct BwdUnit {
    int z, hk, j, i0, per_head, nsteps;
};

template <bool CAUSAL>
__device__ __forceinline__ BwdUnit bwd_unit(int u, const BwdParams& p) {
    BwdUnit w;
    const int zh = p.Z * p.Hkv;
    w.j = u / zh;
    w.z = (u % zh) / p.Hkv;
    w.hk = (u % zh) % p.Hkv;
    // causal (top-left): query row r sees keys <= r, so query blocks before
    // the key block's own index see none of its keys
    w.i0 = CAUSAL ? w.j : 0;
    w.per_head = p.Tq > w.i0 ? p.Tq - w.i0 : 0;
    w.nsteps = w.per_head * p.group;
    return w;
}

// step s of a unit: query head and query block
__device__ __forceinline__ void bwd_step(const BwdUnit& w, int s, const BwdParams& p, int& hq, int& i) {
    hq = w.hk * p.group + s / w.per_head;
    i = w.i0 + s % w.per_head;
}

// ------------------------------------------------------------ producer ------
template <int D, bool CAUSAL>
__device__ void bwd_producer(const CUtensorMap* tmK, const CUtensorMap* tmV, const CUtensorMap* tmQ,
                             const CUtensorMap* tmDO, const BwdParams& p, uint32_t sbase, uint32_t bar0,
                             const Ctl& ctl) {
    using T = BwdTraits<D>;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    const uint64_t pol_kv = ptx::policy_evict_first();  // read once per unit
    const uint64_t pol_q = ptx::policy_evict_last();    // read by every key block
    uint32_t uc = 0, t = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < p.nunits; u += gridDim.x) {
        const BwdUnit w = bwd_unit<CAUSAL>(u, p);
        if (w.nsteps == 0) continue;
        if (uc > 0 && !wait_phase(bar(T::B_KV_EMPTY), (uc - 1) & 1u, ctl, SITE_B_KV_EMPTY)) { ok = false; break; }
        ptx::mbar_arrive_expect_tx(bar(T::B_KV_FULL), 2 * T::TILE);
        for (int c = 0; c < T::NCHUNK; ++c) {
            ptx::tma_load_4d(sbase + T::OFF_K + c * (128 * T::SW), tmK, bar(T::B_KV_FULL), c * T::SWE, w.j * 128,
                             w.hk, w.z, pol_kv);
            ptx::tma_load_4d(sbase + T::OFF_V + c * (128 * T::SW), tmV, bar(T::B_KV_FULL), c * T::SWE, w.j * 128,
                             w.hk, w.z, pol_kv);
        }
        ++uc;
        for (int s = 0; s < w.nsteps; ++s, ++t) {
            const uint32_t st = t & 1u;
            if (t >= 2 && !wait_phase(bar(T::B_QD_EMPTY + st), ((t - 2) >> 1) & 1u, ctl, SITE_B_QD_EMPTY)) {
                ok = false;
                break;
            }
            int hq, i;
            bwd_step(w, s, p, hq, i);
            const uint32_t full = bar(T::B_QD_FULL + st);
            ptx::mbar_arrive_expect_tx(full, 2 * T::TILE + 1024);
            for (int c = 0; c < T::NCHUNK; ++c) {
                ptx::tma_load_4d(sbase + T::OFF_Q + st * T::TILE + c * (128 * T::SW), tmQ, full, c * T::SWE, i * 128,
                                 hq, w.z, pol_q);
                ptx::tma_load_4d(sbase + T::OFF_DO + st * T::TILE + c * (128 * T::SW), tmDO, full, c * T::SWE,
                                 i * 128, hq, w.z, pol_q);
            }
            const int64_t row0 = ((int64_t)w.z * p.Hq + hq) * p.Tq * 128 + (int64_t)i * 128;
            ptx::bulk_load(sbase + T::OFF_LSE + st * 512, p.lse2 + row0, 512, full);
            ptx::bulk_load(sbase + T::OFF_DELTA + st * 512, p.delta + row0, 512, full);
        }
    }
    if (!ok) {
        // let the copies in flight land before shared memory goes away
        if (uc > 0) drain_phase(bar(T::B_KV_FULL), (uc - 1) & 1u, ctl.limit_ns);
        for (uint32_t x = t > 2u ? t - 2u : 0u; x < t; ++x)
            drain_phase(bar(T::B_QD_FULL + (x & 1u)), (x >> 1) & 1u, ctl.limit_ns);
    }
}

// ------------------------------------------------------------ MMA issuer ----
template <int D, bool CAUSAL, bool BF16>
__device__ void bwd_issuer(const BwdParams& p, uint32_t sbase, uint32_t bar0, uint32_t tmem, const Ctl& ctl) {
    using T = BwdTraits<D>;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    // Sᵀ = K Qᵀ and dPᵀ = V dOᵀ: A and B K-major (rows of 128 keys / queries, D contiguous)
    constexpr uint32_t ID_SQ = ptx::idesc_f16(128, 128, BF16, false, false);
    // dV += Pᵀ dO and dK += dSᵀ Q: N = D, B MN-major (D contiguous along N)
    constexpr uint32_t ID_ND = ptx::idesc_f16(128, D, BF16, false, true);
    // dQ = dS K: A = dSᵀ read MN-major (queries contiguous), B = K MN-major
    constexpr uint32_t ID_DQ = ptx::idesc_f16(128, D, BF16, true, true);
    constexpr uint32_t HI = ptx::smem_desc_hi(8 * T::SW, T::SWIZZLE_CODE);  // Q, K, V, dO tiles
    constexpr uint32_t HI_DS = ptx::smem_desc_hi(8 * 128, 2u);              // dSᵀ: 128-B swizzle
    const uint32_t k_lo = ptx::smem_desc_lo(sbase + T::OFF_K, 16);
    const uint32_t v_lo = ptx::smem_desc_lo(sbase + T::OFF_V, 16);
    const uint32_t kmn_lo = ptx::smem_desc_lo(sbase + T::OFF_K, 128 * T::SW);     // K as MN-major B
    const uint32_t ds_lo = ptx::smem_desc_lo(sbase + T::OFF_DS, 16);             // dSᵀ as K-major A
    const uint32_t dsmn_lo = ptx::smem_desc_lo(sbase + T::OFF_DS, 128 * 128);    // dSᵀ as MN-major A
    // K-major operand of 128 rows: 16-element step kk inside swizzled chunks
    auto kmaj = [&](int kk, int swe, int sw) -> uint32_t {
        return (uint32_t)((((kk * 16) / swe) * (128 * sw) + ((kk * 16) % swe) * 2) >> 4);
    };
    // Sᵀ of step t into TMEM; its operands are stage t & 1
    auto issue_s = [&](uint32_t t) -> bool {
        const uint32_t st = t & 1u;
        if (!wait_phase(bar(T::B_QD_FULL + st), (t >> 1) & 1u, ctl, SITE_B_QD_FULL)) return false;
        ptx::tc_fence_after();
        const uint32_t q_lo = ptx::smem_desc_lo(sbase + T::OFF_Q + st * T::TILE, 16);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
            ptx::mma_ss(tmem + T::TM_S, ptx::desc64(k_lo + kmaj(kk, T::SWE, T::SW), HI),
                        ptx::desc64(q_lo + kmaj(kk, T::SWE, T::SW), HI), ID_SQ, kk > 0 ? 1u : 0u);
        ptx::tc_commit(bar(T::B_S_FULL));
        return true;
    };
    // Order per step t: dPᵀ_t, dV_t, then Sᵀ_{t+1} (its columns were last read
    // by dV_t, issued before it; the softmax warps keep Pᵀ_t in registers), then
    // dK_t and dQ_t -- so the softmax warps build Pᵀ_{t+1} while the tensor core
    // runs dK_t and dQ_t.
    uint32_t uc = 0, t = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < p.nunits; u += gridDim.x) {
        const BwdUnit w = bwd_unit<CAUSAL>(u, p);
        if (w.nsteps == 0) continue;
        if (!wait_phase(bar(T::B_KV_FULL), uc & 1u, ctl, SITE_B_KV_FULL)) { ok = false; break; }
        if (!issue_s(t)) { ok = false; break; }
        for (int s = 0; s < w.nsteps; ++s, ++t) {
            const uint32_t st = t & 1u;
            const uint32_t qmn_lo = ptx::smem_desc_lo(sbase + T::OFF_Q + st * T::TILE, 128 * T::SW);
            const uint32_t do_lo = ptx::smem_desc_lo(sbase + T::OFF_DO + st * T::TILE, 16);
            const uint32_t domn_lo = ptx::smem_desc_lo(sbase + T::OFF_DO + st * T::TILE, 128 * T::SW);
            // dPᵀ = V dOᵢᵀ, once the previous dQ partial (same columns) is read out
            if (t > 0 && !wait_phase(bar(T::B_DQ_FREE), (t - 1) & 1u, ctl, SITE_B_DQ_FREE)) { ok = false; break; }
            ptx::tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
                ptx::mma_ss(tmem + T::TM_DP, ptx::desc64(v_lo + kmaj(kk, T::SWE, T::SW), HI),
                            ptx::desc64(do_lo + kmaj(kk, T::SWE, T::SW), HI), ID_SQ, kk > 0 ? 1u : 0u);
            ptx::tc_commit(bar(T::B_DP_FULL));
            // dV += Pᵀ dOᵢ; the first step of a unit waits for the last unit's dK, dV to be read
            if (!wait_phase(bar(T::B_P_FULL), t & 1u, ctl, SITE_B_P_FULL)) { ok = false; break; }
            if (s == 0 && uc > 0 && !wait_phase(bar(T::B_ACC_FREE), (uc - 1) & 1u, ctl, SITE_B_ACC_FREE)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            // Pᵀ of queries 0-63 sits in packed columns 0-31, of queries 64-127 in 64-95
#pragma unroll
            for (int kk = 0; kk < 128 / 16; ++kk)
                ptx::mma_ts(tmem + T::TM_DV, tmem + T::TM_S + (kk < 4 ? kk * 8 : 64 + (kk - 4) * 8),
                            ptx::desc64(domn_lo + ((kk * 16 * T::SW) >> 4), HI), ID_ND, (s > 0 || kk > 0) ? 1u : 0u);
            if (s + 1 < w.nsteps && !issue_s(t + 1)) { ok = false; break; }
            // dK += dSᵀ Qᵢ and dQᵢ = dS K, once dSᵀ is in shared memory
            if (!wait_phase(bar(T::B_DS_FULL), t & 1u, ctl, SITE_B_DS_FULL)) { ok = false; break; }
            ptx::tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 128 / 16; ++kk)
                ptx::mma_ss(tmem + T::TM_DK, ptx::desc64(ds_lo + kmaj(kk, 64, 128), HI_DS),
                            ptx::desc64(qmn_lo + ((kk * 16 * T::SW) >> 4), HI), ID_ND, (s > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
            for (int kk = 0; kk < 128 / 16; ++kk)
                ptx::mma_ss(tmem + T::TM_DP, ptx::desc64(dsmn_lo + ((kk * 16 * 128) >> 4), HI_DS),
                            ptx::desc64(kmn_lo + ((kk * 16 * T::SW) >> 4), HI), ID_DQ, kk > 0 ? 1u : 0u);
            ptx::tc_commit(bar(T::B_DQ_FULL));       // dQ partial ready, dSᵀ buffer free
            ptx::tc_commit(bar(T::B_QD_EMPTY + st));  // Qᵢ, dOᵢ slot free
        }
        if (!ok) break;
        ptx::tc_commit(bar(T::B_ACC_FULL));  // dK, dV of the unit complete
        ptx::tc_commit(bar(T::B_KV_EMPTY));  // K, V free
        ++uc;
    }
    if (!ok) {
        ptx::tc_commit(bar(T::B_DRAIN));
        drain_phase(bar(T::B_DRAIN), 0u, ctl.limit_ns);
    }
}

// ------------------------------------------------------------ Pᵀ and dSᵀ ----
// Thread = key (TMEM lane); half h takes queries h*64 .. h*64 + 63.  Each
// half writes its Pᵀ over its own Sᵀ columns (packed columns h*64 ..), so no
// half overwrites scores the other has not read.
template <int D, bool CAUSAL, bool BF16>
__device__ void bwd_softmax(const BwdParams& p, uint32_t sbase, uint32_t bar0, uint32_t tmem, int h,
                            const Ctl& ctl) {
    using T = BwdTraits<D>;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    const int quad = (threadIdx.x / 32) % 4;
    const int row = quad * 32 + threadIdx.x % 32;  // key within the block
    const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
    const float c = p.scale_log2;
    uint32_t t = 0;
    for (int u = blockIdx.x; u < p.nunits; u += gridDim.x) {
        const BwdUnit w = bwd_unit<CAUSAL>(u, p);
        for (int s = 0; s < w.nsteps; ++s, ++t) {
            const uint32_t st = t & 1u;
            int hq, i;
            bwd_step(w, s, p, hq, i);
            // lse2 and Δ of the step's queries arrive with Qᵢ (TMA)
            if (!warp_wait_phase(bar(T::B_QD_FULL + st), (t >> 1) & 1u, ctl, SITE_B_QD_FULL)) return;
            const uint32_t lse_a = sbase + T::OFF_LSE + st * 512 + h * 256;
            const uint32_t del_a = sbase + T::OFF_DELTA + st * 512 + h * 256;
            if (!warp_wait_phase(bar(T::B_S_FULL), t & 1u, ctl, SITE_B_S_FULL)) return;
            ptx::tc_fence_after();
            // causal: only the diagonal block has keys after queries (key > query -> 0)
            const bool diag = CAUSAL && i == w.j;
            // Pᵀ in the input type (it is the tensor-core operand of dV, and
            // dS below uses the same rounded values)
            uint32_t pk[32];
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                uint32_t r[32];
                ptx::tmem_ld32(tmem + lane_addr + T::TM_S + h * 64 + 32 * cc, r);
#pragma unroll
                for (int x = 0; x < 16; ++x) {
                    const int col = h * 64 + 32 * cc + 2 * x;
                    float l0, l1;
                    asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(l0), "=f"(l1) : "r"(lse_a + 4u * (32 * cc + 2 * x)));
                    float e0 = fmaf(__uint_as_float(r[2 * x]), c, -l0);
                    float e1 = fmaf(__uint_as_float(r[2 * x + 1]), c, -l1);
                    if (diag && row > col) e0 = -INFINITY;
                    if (diag && row > col + 1) e1 = -INFINITY;
                    pk[16 * cc + x] = pack2<BF16>(ptx::ex2(e0), ptx::ex2(e1));
                }
            }
            ptx::tmem_st32(tmem + lane_addr + T::TM_S + h * 64, pk);
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(T::B_P_FULL));

            if (!warp_wait_phase(bar(T::B_DP_FULL), t & 1u, ctl, SITE_B_DP_FULL)) return;
            // the dSᵀ buffer is free once the previous step's dK and dQ MMAs completed
            if (t > 0 && !warp_wait_phase(bar(T::B_DQ_FULL), (t - 1) & 1u, ctl, SITE_B_DS_FREE)) return;
            ptx::tc_fence_after();
            const uint32_t ds_row = sbase + T::OFF_DS + h * (128 * 128) + row * 128;
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                uint32_t r[32];
                ptx::tmem_ld32(tmem + lane_addr + T::TM_DP + h * 64 + 32 * cc, r);
                uint32_t ds[16];
#pragma unroll
                for (int x = 0; x < 16; ++x) {
                    float d0, d1;
                    asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(d0), "=f"(d1) : "r"(del_a + 4u * (32 * cc + 2 * x)));
                    const float2 pp = unpack2<BF16>(pk[16 * cc + x]);
                    ds[x] = pack2<BF16>(pp.x * (__uint_as_float(r[2 * x]) - d0), pp.y * (__uint_as_float(r[2 * x + 1]) - d1));
                }
                // 16-byte units 4cc .. 4cc + 3 of this row of the chunk, 128-B swizzle
#pragma unroll
                for (int uu = 0; uu < 4; ++uu) {
                    const uint32_t unit = (uint32_t)(4 * cc + uu) ^ (uint32_t)(row & 7);
                    ptx::st_shared_v4(ds_row + unit * 16, ds[4 * uu], ds[4 * uu + 1], ds[4 * uu + 2], ds[4 * uu + 3]);
                }
            }
            ptx::fence_proxy_async_smem();
            ptx::mbar_arrive(bar(T::B_DS_FULL));
        }
    }
}

// ------------------------------------------------------------ epilogue ------
// Thread = TMEM lane.  Per step: the dQ partial (lane = query) is read out,
// released, and added into the fp32 accumulator.  Per unit: dK (times scale)
// and dV (lane = key) are read out, released and stored in the input type.
template <int D, bool CAUSAL, bool BF16>
__device__ void bwd_epilogue(const BwdParams& p, uint32_t bar0, uint32_t tmem, const Ctl& ctl) {
    using T = BwdTraits<D>;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    const int quad = (threadIdx.x / 32) % 4;
    const int row = quad * 32 + threadIdx.x % 32;
    const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
    constexpr int CH = D >= 32 ? 32 : 16;
    uint32_t t = 0, uc = 0;
    for (int u = blockIdx.x; u < p.nunits; u += gridDim.x) {
        const BwdUnit w = bwd_unit<CAUSAL>(u, p);
        const int key = w.j * 128 + row;
        uint8_t* dk_row = reinterpret_cast<uint8_t*>(p.dk) +
                          2 * ((int64_t)w.z * p.sdk_z + (int64_t)w.hk * p.sdk_h + (int64_t)key * p.sdk_n);
        uint8_t* dv_row = reinterpret_cast<uint8_t*>(p.dv) +
                          2 * ((int64_t)w.z * p.sdv_z + (int64_t)w.hk * p.sdv_h + (int64_t)key * p.sdv_n);
        if (w.nsteps == 0) {
            // no query sees these keys: zero gradients
            if (key < p.Nkv) {
#pragma unroll
                for (int x = 0; x < D / 8; ++x) {
                    reinterpret_cast<uint4*>(dk_row)[x] = make_uint4(0, 0, 0, 0);
                    reinterpret_cast<uint4*>(dv_row)[x] = make_uint4(0, 0, 0, 0);
                }
            }
            continue;
        }
        for (int s = 0; s < w.nsteps; ++s, ++t) {
            int hq, i;
            bwd_step(w, s, p, hq, i);
            if (!warp_wait_phase(bar(T::B_DQ_FULL), t & 1u, ctl, SITE_B_DQ_FULL)) return;
            ptx::tc_fence_after();
            const int q = i * 128 + row;
            float* acc = p.dq_acc + (((int64_t)w.z * p.Hq + hq) * p.Nq + q) * D;
#pragma unroll
            for (int cc = 0; cc < D / CH; ++cc) {
                uint32_t r[CH];
                if constexpr (CH == 32) ptx::tmem_ld32(tmem + lane_addr + T::TM_DP + cc * CH, r);
                else ptx::tmem_ld16(tmem + lane_addr + T::TM_DP + cc * CH, r);
                if (cc == D / CH - 1) {
                    ptx::tc_fence_before();
                    ptx::mbar_arrive(bar(T::B_DQ_FREE));
                }
                if (q < p.Nq) {
#pragma unroll
                    for (int x = 0; x < CH / 4; ++x)
                        ptx::red_add_v4(acc + cc * CH + 4 * x, __uint_as_float(r[4 * x]), __uint_as_float(r[4 * x + 1]),
                                        __uint_as_float(r[4 * x + 2]), __uint_as_float(r[4 * x + 3]));
                }
            }
        }
        if (!warp_wait_phase(bar(T::B_ACC_FULL), uc & 1u, ctl, SITE_B_ACC_FULL)) return;
        ptx::tc_fence_after();
#pragma unroll
        for (int which = 0; which < 2; ++which) {
            const uint32_t col0 = which == 0 ? T::TM_DV : T::TM_DK;
            const float mul = which == 0 ? 1.f : p.scale;
            uint8_t* dst = which == 0 ? dv_row : dk_row;
#pragma unroll
            for (int cc = 0; cc < D / CH; ++cc) {
                uint32_t r[CH];
                if constexpr (CH == 32) ptx::tmem_ld32(tmem + lane_addr + col0 + cc * CH, r);
                else ptx::tmem_ld16(tmem + lane_addr + col0 + cc * CH, r);
                if (which == 1 && cc == D / CH - 1) {
                    ptx::tc_fence_before();
                    ptx::mbar_arrive(bar(T::B_ACC_FREE));
                }
                if (key < p.Nkv) {
#pragma unroll
                    for (int x = 0; x < CH / 8; ++x)
                        reinterpret_cast<uint4*>(dst + 2 * cc * CH)[x] = make_uint4(
                            pack2<BF16>(__uint_as_float(r[8 * x]) * mul, __uint_as_float(r[8 * x + 1]) * mul),
                            pack2<BF16>(__uint_as_float(r[8 * x + 2]) * mul, __uint_as_float(r[8 * x + 3]) * mul),
                            pack2<BF16>(__uint_as_float(r[8 * x + 4]) * mul, __uint_as_float(r[8 * x + 5]) * mul),
                            pack2<BF16>(__uint_as_float(r[8 * x + 6]) * mul, __uint_as_float(r[8 * x + 7]) * mul));
                }
            }
        }
        ++uc;
    }
}

// ------------------------------------------------------------ kernel --------
template <int D, bool CAUSAL, bool BF16>
__global__ void __launch_bounds__(BWD_THREADS, 1)
    fa_bwd_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
                  const BwdParams p) {
    using T = BwdTraits<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    if (pad + T::SMEM_USED > T::SMEM_BYTES) {
        // no room to align the swizzled tiles: report and leave (uniform for the CTA)
        if (threadIdx.x == 0) atomicCAS(p.status, 0u, 4u /* FA_ERR_CUDA */ | (0xFFu << 8) | ((blockIdx.x & 0xFFFFu) << 16));
        return;
    }
    uint8_t* smem = smem_raw + pad;
    const uint32_t sbase = raw + pad;
    const uint32_t bar0 = sbase + T::OFF_BAR;
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + T::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + T::OFF_MISC + 4);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        for (int i = 0; i < T::NUM_BARS; ++i) ptx::mbar_init(bar0 + 8u * i, T::bar_count(i));
        *abort_flag = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tmK);
        ptx::prefetch_tmap(&tmV);
        ptx::prefetch_tmap(&tmQ);
        ptx::prefetch_tmap(&tmDO);
    }
    if (warp == 13) {
        ptx::tmem_alloc(ptx::smem_addr(const_cast<uint32_t*>(tmem_slot)), T::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const Ctl ctl{abort_flag, p.status, p.wait_limit_ns};
    if (warp < 8) {
        bwd_softmax<D, CAUSAL, BF16>(p, sbase, bar0, tmem, warp / 4, ctl);
    } else if (warp < 12) {
        bwd_epilogue<D, CAUSAL, BF16>(p, bar0, tmem, ctl);
    } else if (warp == 12) {
        if (lane == 0) bwd_producer<D, CAUSAL>(&tmK, &tmV, &tmQ, &tmDO, p, sbase, bar0, ctl);
    } else {
        if (lane == 0) bwd_issuer<D, CAUSAL, BF16>(p, sbase, bar0, tmem, ctl);
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 13) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, T::TMEM_COLS);
    }
}

// ------------------------------------------------------------ pre / post ----
// Per query row, padded to whole 128-row blocks: Δ = rowsum(dO ∘ O) in fp32
// from the input-type values, the lse in base 2 (+inf past Nq, so those
// columns get P = 0), and a zeroed row of the dQ accumulator.
template <int D, bool BF16>
__global__ void __launch_bounds__(256) fa_bwd_pre_kernel(const BwdParams p) {
    constexpr int TPR = D / 8;  // threads per row, 16 bytes of O and of dO each
    const int64_t rows = (int64_t)p.Z * p.Hq * p.Tq * 128;
    const int sub = threadIdx.x % TPR;
    for (int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / TPR; r < rows;
         r += (int64_t)gridDim.x * blockDim.x / TPR) {
        const int64_t head = r / ((int64_t)p.Tq * 128);
        const int i = (int)(r - head * p.Tq * 128);
        const int z = (int)(head / p.Hq), hq = (int)(head % p.Hq);
        float delta = 0.f;
        if (i < p.Nq) {
            const uint4 a = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.o) + (int64_t)z * p.so_z +
                                                           (int64_t)hq * p.so_h + (int64_t)i * p.so_n)[sub];
            const uint4 b = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.dO) + (int64_t)z * p.sdo_z +
                                                           (int64_t)hq * p.sdo_h + (int64_t)i * p.sdo_n)[sub];
            const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int y = 0; y < 4; ++y) {
                const float2 fa = unpack2<BF16>(aw[y]), fb = unpack2<BF16>(bw[y]);
                delta = fmaf(fa.x, fb.x, delta);
                delta = fmaf(fa.y, fb.y, delta);
            }
            float4* acc = reinterpret_cast<float4*>(p.dq_acc + (head * p.Nq + i) * D) + 2 * sub;
            acc[0] = make_float4(0.f, 0.f, 0.f, 0.f);
            acc[1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        // the row's TPR lanes are consecutive lanes of one warp
#pragma unroll
        for (int m = TPR / 2; m > 0; m /= 2) delta += __shfl_xor_sync(0xffffffffu, delta, m);
        if (sub == 0) {
            p.delta[r] = delta;
            p.lse2[r] = i < p.Nq ? p.lse[head * p.Nq + i] * 1.4426950408889634f : INFINITY;
        }
    }
}

// dQ = scale · accumulator, in the input type; one thread per 8 columns
template <int D, bool BF16>
__global__ void __launch_bounds__(256) fa_bwd_dq_kernel(const BwdParams p) {
    constexpr int C = D / 8;
    const int64_t items = (int64_t)p.Z * p.Hq * p.Nq * C;
    for (int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; x < items; x += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = x / C;
        const int c = (int)(x - r * C);
        const int64_t head = r / p.Nq;
        const int i = (int)(r - head * p.Nq);
        const int z = (int)(head / p.Hq), hq = (int)(head % p.Hq);
        const float4* a = reinterpret_cast<const float4*>(p.dq_acc + r * D + 8 * c);
        const float4 a0 = a[0], a1 = a[1];
        const float m = p.scale;
        uint4 out = make_uint4(pack2<BF16>(a0.x * m, a0.y * m), pack2<BF16>(a0.z * m, a0.w * m),
                               pack2<BF16>(a1.x * m, a1.y * m), pack2<BF16>(a1.z * m, a1.w * m));
        *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.dq) + (int64_t)z * p.sdq_z + (int64_t)hq * p.sdq_h +
                                  (int64_t)i * p.sdq_n + 8 * c) = out;
    }
}

}  // namespace fa
