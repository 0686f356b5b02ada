// Fused attention forward at head dim 128 on CTA pairs: O = softmax(Q Kᵀ ·
// scale) V and the per-row log-sum-exp, whole query tiles, the two-softmax-
// chain kernel's arithmetic (fa_fwd_chain_kernel.cuh) with its matrix products
// spread over two SMs.
//
// The method is the tiled online-softmax forward of the pages ("Write Triton
// Attention Kernel", Required reasoning process steps 1-9; "把 FlashAttention
// 搬上昇腾：Triton-Ascend CV Pipeline 优化实战", sections 一 and 八).  What this
// kernel changes is where the operands of the products live.  On one SM a
// 128 x 128 key block moves ~160 KB through shared memory at D = 128 (the
// products read Q and K, 64 KB, and V, 32 KB; TMA writes K and V, 64 KB):
// ~1250 cycles at 128 B/clk against 1024 cycles of tensor-core work.  Here a
// cluster of two CTAs takes two query tiles that see the same key blocks
// (two query heads of one GQA group, or query blocks 2m and 2m + 1 of one
// head), and each key block is multiplied once for both as an M = 256
// product (tcgen05 cta_group::2): each CTA holds its own 128 query rows and
// HALF of every K and V block (keys 64r .. 64r + 63 of K, columns 64r ..
// 64r + 63 of V for CTA r), the tensor cores of the two SMs exchange the
// halves, and each SM moves ~96 KB a block.
//
// Roles, per CTA (512 threads):
//   warp 0         TMA: this CTA's Q tile and K half of each block
//   warp 3         TMA: this CTA's V half of each block
//   warp 1         even CTA: issues S_g = Q K_gᵀ (M = 256) for both CTAs;
//                  odd CTA: forwards "my Q tile / K half landed" to the even CTA
//   warp 2         even CTA: issues O += P_g V_g (M = 256, P from each CTA's
//                  TMEM); odd CTA: forwards "my V half landed"
//   warpgroups 1-2 the two softmax chains over this CTA's rows (unchanged)
//   warpgroup 3    the epilogue of this CTA's rows (unchanged)
// The even CTA's commits arrive on the barriers of both CTAs (multicast), so
// each CTA's softmax, epilogue and producers wait on their own barriers; the
// odd CTA's "P written" and "O read" go to the even CTA's barriers, one
// arrival per warp.  Every wait is bounded; both CTAs end with a cluster
// barrier before their TMEM is freed, so neither leaves while the other may
// still reach its shared memory or tensor memory.
#pragma once

#include "fa_fwd_chain_kernel.cuh"

namespace fa {

// Shared memory, TMEM and barriers of one CTA of a pair (D = 128).
//
// Rings.  A score slot holds S_g only until the softmax chain has loaded it
// (then released, arrive_sfree); P_g goes to a P slot of its own, released
// when O += P_g V_g is complete.  So a score slot's round trip is "S issued
// -> scores loaded", not a block's whole path through softmax and P·V (which
// with three shared S/P slots measured ~735 ns a block against ~512 ns of
// tensor work).  K and V slots have their own release barriers, committed
// by the issuer that last read them.
template <int D>
struct PairTraits {
    static_assert(D == 128, "CTA-pair kernel: head dim 128");
    static constexpr int BN = 128;                      // keys per block (both halves)
    static constexpr int SW = 128;                      // 128-byte swizzle rows
    static constexpr int SWE = 64;
    static constexpr int NCHUNK = D / SWE;              // 2
    static constexpr uint32_t SWIZZLE_CODE = 2u;
    static constexpr int Q_BYTES = BM * D * 2;          // 32 KB: this CTA's query tile
    static constexpr int KH_BYTES = (BN / 2) * D * 2;   // 16 KB: 64 keys x 128 columns
    static constexpr int VH_BYTES = BN * (D / 2) * 2;   // 16 KB: 128 keys x 64 columns
    static constexpr int Q_STAGES = 2;
    static constexpr int KV_STAGES = 4;
    static constexpr int SR = 2;                        // score slots (fp32, BN columns)
    static constexpr int PR = 2;                        // P slots (16-bit pairs, BN / 2 columns)
    static constexpr uint32_t TM_S = 0;
    static constexpr uint32_t TM_P = SR * BN;
    static constexpr uint32_t TM_O = TM_P + PR * (BN / 2);
    static constexpr uint32_t TMEM_COLS = 512;
    static_assert(TM_O + D <= TMEM_COLS, "tensor memory budget");
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + Q_STAGES * Q_BYTES;
    static constexpr int OFF_V = OFF_K + KV_STAGES * KH_BYTES;
    static constexpr int OFF_HAND = OFF_V + KV_STAGES * VH_BYTES;  // 2 slots x {m0, l0, m1, l1} x BM
    static constexpr int OFF_RED = OFF_HAND + 2 * 4 * BM * 4;      // m hand-off, 2 slots x BM
    static constexpr int OFF_OST = (OFF_RED + 2 * BM * 4 + 1023) / 1024 * 1024;
    static constexpr int OFF_BAR = OFF_OST + BM * SW;
    static constexpr int B_QFULL = 0;                      // [2] this CTA's Q tile landed (TMA)
    static constexpr int B_QEMPTY = B_QFULL + Q_STAGES;    // [2] last S of the tile done (commit, both CTAs)
    static constexpr int B_KFULL = B_QEMPTY + Q_STAGES;    // [KV] this CTA's K half landed (TMA)
    static constexpr int B_KEMPTY = B_KFULL + KV_STAGES;   // [KV] S of that block done (commit, both)
    static constexpr int B_VFULL = B_KEMPTY + KV_STAGES;   // [KV] this CTA's V half landed (TMA)
    static constexpr int B_VEMPTY = B_VFULL + KV_STAGES;   // [KV] P·V of that block done (commit, both)
    static constexpr int B_SFULL = B_VEMPTY + KV_STAGES;   // [SR] S_g in TMEM (commit, both)
    static constexpr int B_SFREE = B_SFULL + SR;           // [SR] even CTA: S_g loaded by both CTAs
    static constexpr int B_PFULL = B_SFREE + SR;           // [PR] even CTA: P_g written by both CTAs
    static constexpr int B_PVDONE = B_PFULL + PR;          // [PR] O += P_g V_g done (commit, both)
    static constexpr int B_EPIFULL = B_PVDONE + PR;        // [2] (m, l) of a tile handed over (both chains)
    static constexpr int B_EPIEMPTY = B_EPIFULL + 2;       // [2] hand-over read (epilogue)
    static constexpr int B_OFREE = B_EPIEMPTY + 2;         // even CTA: O read out by both CTAs
    static constexpr int B_RED = B_OFREE + 1;              // [2] m hand-off between the chains
    static constexpr int B_DRAIN = B_RED + 2;              // [2] the even CTA's issuers' teardown
    static constexpr int B_PEER_Q = B_DRAIN + 2;           // [2] even CTA: the odd CTA's Q tile landed
    static constexpr int B_PEER_K = B_PEER_Q + 2;          // [KV] even CTA: the odd CTA's K half landed
    static constexpr int B_PEER_V = B_PEER_K + KV_STAGES;  // [KV] even CTA: the odd CTA's V half landed
    static constexpr int NUM_BARS = B_PEER_V + KV_STAGES;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
    static constexpr int SMEM_USED = OFF_MISC + 16;
    static constexpr int SMEM_BYTES = SMEM_USED + 1024;
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
    // S_g loaded / P_g written / O read: the 4 warps of the chain (or
    // epilogue) of each CTA arrive once each
    static constexpr uint32_t PAIR_ARRIVALS = 4 + 4;

    static __host__ __device__ __forceinline__ uint32_t kv_slot(uint32_t g) { return g % KV_STAGES; }
    static __host__ __device__ __forceinline__ uint32_t kv_phase(uint32_t g) { return (g / KV_STAGES) & 1u; }
    static __device__ __forceinline__ uint32_t bar_count(int i) {
        if (i >= B_SFREE && i < B_SFREE + SR) return PAIR_ARRIVALS;
        if (i >= B_PFULL && i < B_PFULL + PR) return PAIR_ARRIVALS;
        if (i == B_OFREE) return PAIR_ARRIVALS;
        if (i >= B_EPIFULL && i < B_EPIFULL + 2) return 8;   // both chains' warps
        if (i >= B_EPIEMPTY && i < B_EPIEMPTY + 2) return 4;
        if (i >= B_RED && i < B_RED + 2) return 4;
        return 1;
    }
};

// The schedule of a CTA pair: cluster c takes units c, c + clusters, ...
// (alternating direction by round when ALT), each unit a tile of a virtual
// head (p.pair_heads of them, p.pair_tq virtual query blocks each) in the
// whole-tile order: non-causal head-major, causal in groups of
// p.pair_head_group virtual heads from the heaviest block down.  A CTA's Seg
// is its own query tile of the unit; both CTAs of a unit visit the same key
// blocks (for query blocks 2m, 2m + 1 under a causal mask: those of 2m + 1,
// the last of which is masked whole for the rows of 2m).
template <bool CAUSAL, bool ALT>
struct PairSched {
    uint32_t rank;
    __device__ explicit PairSched(const FwdParams&) : rank(ptx::cluster_ctarank()) {}
    static __device__ __forceinline__ int64_t unit_at(int64_t pos) {
        if (!CAUSAL || !ALT) return pos;
        const uint32_t x = (uint32_t)pos, g = ptx::cluster_count_x(), round = x / g;
        return (round & 1u) ? (int64_t)(2u * round * g + g - 1u - x) : pos;
    }
    __device__ __forceinline__ int64_t first(const FwdParams&) const { return (int64_t)ptx::cluster_id_x(); }
    __device__ __forceinline__ bool valid(int64_t pos, const FwdParams& p) const {
        return unit_at(pos) < p.pair_units;
    }
    __device__ __forceinline__ int64_t next(int64_t pos, const Seg&, const FwdParams&) const {
        return pos + ptx::cluster_count_x();
    }
    __device__ __forceinline__ Seg seg(int64_t pos, const FwdParams& p) const {
        using S1 = Sched<CAUSAL, 128>;
        const uint32_t t = (uint32_t)unit_at(pos), tq = (uint32_t)p.pair_tq;
        uint32_t vh, vmb;
        if (CAUSAL) {
            const uint32_t heads = (uint32_t)p.pair_heads, G = (uint32_t)p.pair_head_group;
            const uint32_t g0 = t / (G * tq) * G;
            const uint32_t gc = heads - g0 < G ? heads - g0 : G;
            const uint32_t w = t - g0 * tq;
            const uint32_t r = w / gc;
            vmb = tq - 1 - r;
            vh = g0 + (w - r * gc);
        } else {
            vh = t / tq;
            vmb = t - vh * tq;
        }
        Seg s;
        int mb;
        if (p.pair == 1) {
            const uint32_t hp = (uint32_t)p.Hq / 2u, z = vh / hp;
            s.z = (int)z;
            s.hq = (int)(2u * (vh - z * hp) + rank);
            mb = (int)vmb;
            s.nkv = S1::tile_nkv(mb, p);
        } else {
            const uint32_t z = vh / (uint32_t)p.Hq;
            s.z = (int)z;
            s.hq = (int)(vh - z * (uint32_t)p.Hq);
            mb = (int)(2u * vmb + rank);
            const int upper = 2 * (int)vmb + 1 < p.Tq ? 2 * (int)vmb + 1 : p.Tq - 1;
            s.nkv = S1::tile_nkv(upper, p);
        }
        s.hk = s.hq / p.group;
        s.q_start = mb * BM;
        s.nq = p.Nq;
        s.nk = p.Nkv;
        s.qrow0 = 0;
        s.krow0 = 0;
        s.zc = s.z;
        s.lse0 = ((int64_t)s.z * p.Hq + s.hq) * p.Nq;
        s.jb = 0;
        s.je = s.nkv;
        s.slot = -1;
        return s;
    }
};

// The softmax chains' and epilogue's view of a pair (see ChainSolo).
template <int D, bool CAUSAL, bool ALT>
struct ChainPair {
    using L = PairTraits<D>;
    using S = PairSched<CAUSAL, ALT>;
    static constexpr bool kCluster = false;  // see the note on waits below
    static constexpr bool kSplitP = true;
    static constexpr int kCheckVar = 0;
    uint32_t bar0;       // this CTA's barriers
    uint32_t lead_bar0;  // the even CTA's barriers, as a cluster address
    bool lead;
    __device__ __forceinline__ void arrive(int i) const {
        // the warp's TMEM writes / reads are complete (each lane waited for
        // them and fenced before this call): one arrival for the warp
        if (lead) {
            ptx::mbar_arrive_warp(bar0 + 8u * (uint32_t)i);
        } else {
            __syncwarp();
            if (threadIdx.x % 32 == 0) ptx::mbar_arrive_remote_relaxed(lead_bar0 + 8u * (uint32_t)i);
        }
    }
    __device__ __forceinline__ void arrive_p(uint32_t r) const { arrive(L::B_PFULL + (int)r); }
    __device__ __forceinline__ void arrive_sfree(uint32_t r) const { arrive(L::B_SFREE + (int)r); }
    __device__ __forceinline__ void arrive_ofree() const { arrive(L::B_OFREE); }
};

// ------------------------------------------------------------ TMA producers -
template <int D, bool CAUSAL, bool ALT>
__device__ void pair_producer_qk(const CUtensorMap* tmQ, const CUtensorMap* tmK, const FwdParams& p, uint32_t sbase,
                                 uint32_t bar0, uint32_t rank, const Ctl& ctl) {
    using T = PairTraits<D>;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    const uint64_t pol_q = ptx::policy_evict_first();
    const uint64_t pol_kv = ptx::policy_evict_last();
    uint32_t qi = 0, ki = 0;
    bool ok = true;
    bool withheld = false;
    auto load_q = [&](const Seg& sg) -> bool {
        if (!seg_checked<0, T::BN>(sg, p, ctl, SITE_CHECK_LOAD_QK)) return false;
        const uint32_t s = qi % T::Q_STAGES, ph = (qi / T::Q_STAGES) & 1u;
        if (!wait_phase(bar(T::B_QEMPTY + s), ph ^ 1u, ctl, SITE_Q_EMPTY)) return false;
        ptx::mbar_arrive_expect_tx(bar(T::B_QFULL + s), T::Q_BYTES);
        const uint32_t dst = sbase + T::OFF_Q + s * T::Q_BYTES;
        for (int c = 0; c < T::NCHUNK; ++c)
            ptx::tma_load_4d(dst + c * (BM * T::SW), tmQ, bar(T::B_QFULL + s), c * T::SWE, sg.q_start, sg.hq, sg.zc,
                             pol_q);
        ++qi;
        return true;
    };
    const PairSched<CAUSAL, ALT> sc(p);
    int64_t pos = sc.first(p);
    if (sc.valid(pos, p)) ok = load_q(sc.seg(pos, p));
    while (ok && sc.valid(pos, p)) {
        const Seg sg = sc.seg(pos, p);
        const int64_t nxt = sc.next(pos, sg, p);
        for (int j = sg.jb; j < sg.je; ++j) {
            // the slot held block ki - KV_STAGES, free once S of that block is complete
            constexpr uint32_t KV = T::KV_STAGES;
            const uint32_t s = T::kv_slot(ki);
            if (ki >= KV && !wait_phase(bar(T::B_KEMPTY + s), T::kv_phase(ki) ^ 1u, ctl, SITE_K_EMPTY)) {
                ok = false;
                break;
            }
            if (p.inject_stall && blockIdx.x == 0 && !withheld) {
                withheld = true;  // never issued: the S issuer's wait for this half must time out
            } else {
                ptx::mbar_arrive_expect_tx(bar(T::B_KFULL + s), T::KH_BYTES);
                const uint32_t dst = sbase + T::OFF_K + s * T::KH_BYTES;
                for (int c = 0; c < T::NCHUNK; ++c)
                    ptx::tma_load_4d(dst + c * ((T::BN / 2) * T::SW), tmK, bar(T::B_KFULL + s), c * T::SWE,
                                     j * T::BN + (int)rank * (T::BN / 2), sg.hk, sg.zc, pol_kv);
            }
            ++ki;
            if (j == sg.jb && sc.valid(nxt, p) && !load_q(sc.seg(nxt, p))) { ok = false; break; }
        }
        pos = nxt;
    }
    if (!ok) {
        const uint64_t lim = ctl.limit_ns;
        for (uint32_t i = qi > (uint32_t)T::Q_STAGES ? qi - T::Q_STAGES : 0; i < qi; ++i)
            drain_phase(bar(T::B_QFULL + i % T::Q_STAGES), (i / T::Q_STAGES) & 1u, lim);
        for (uint32_t i = ki > (uint32_t)T::KV_STAGES ? ki - T::KV_STAGES : 0u; i < ki; ++i)
            drain_phase(bar(T::B_KFULL + T::kv_slot(i)), T::kv_phase(i), withheld ? lim / 64 : lim);
    }
}

template <int D, bool CAUSAL, bool ALT>
__device__ void pair_producer_v(const CUtensorMap* tmV, const FwdParams& p, uint32_t sbase, uint32_t bar0,
                                uint32_t rank, const Ctl& ctl) {
    using T = PairTraits<D>;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    const uint64_t pol_kv = ptx::policy_evict_last();
    uint32_t vi = 0;
    bool ok = true;
    const PairSched<CAUSAL, ALT> sc(p);
    for (int64_t pos = sc.first(p); ok && sc.valid(pos, p);) {
        const Seg sg = sc.seg(pos, p);
        if (!seg_checked<0, T::BN>(sg, p, ctl, SITE_CHECK_LOAD_V)) { ok = false; break; }
        for (int j = sg.jb; j < sg.je; ++j) {
            constexpr uint32_t KV = T::KV_STAGES;
            const uint32_t s = T::kv_slot(vi);
            if (vi >= KV && !wait_phase(bar(T::B_VEMPTY + s), T::kv_phase(vi) ^ 1u, ctl, SITE_V_EMPTY)) {
                ok = false;
                break;
            }
            ptx::mbar_arrive_expect_tx(bar(T::B_VFULL + s), T::VH_BYTES);
            // columns 64 rank .. 64 rank + 63 of the block's 128 keys: one swizzle chunk
            ptx::tma_load_4d(sbase + T::OFF_V + s * T::VH_BYTES, tmV, bar(T::B_VFULL + s), (int)rank * T::SWE,
                             j * T::BN, sg.hk, sg.zc, pol_kv);
            ++vi;
        }
        pos = sc.next(pos, sg, p);
    }
    if (!ok)
        for (uint32_t i = vi > (uint32_t)T::KV_STAGES ? vi - T::KV_STAGES : 0u; i < vi; ++i)
            drain_phase(bar(T::B_VFULL + T::kv_slot(i)), T::kv_phase(i), ctl.limit_ns);
}

// ------------------------------------------------------------ odd CTA: forwarders
// The even CTA's issuers must know that the odd CTA's halves have landed
// before they multiply them: these threads wait for each of the odd CTA's
// copies to complete and then arrive on the even CTA's barrier.
template <int D, bool CAUSAL, bool ALT>
__device__ void pair_forward_qk(const FwdParams& p, uint32_t bar0, uint32_t lead_bar0, const Ctl& ctl) {
    using T = PairTraits<D>;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    auto lead = [&](int i) { return lead_bar0 + 8u * (uint32_t)i; };
    uint32_t qi = 0, g = 0;
    const PairSched<CAUSAL, ALT> sc(p);
    for (int64_t pos = sc.first(p); sc.valid(pos, p);) {
        const Seg sg = sc.seg(pos, p);
        pos = sc.next(pos, sg, p);
        const uint32_t qs = qi % T::Q_STAGES;
        if (!wait_phase(bar(T::B_QFULL + qs), (qi / T::Q_STAGES) & 1u, ctl, SITE_Q_FULL)) return;
        ptx::mbar_arrive_remote_relaxed(lead(T::B_PEER_Q + (int)qs));
        ++qi;
        for (int j = sg.jb; j < sg.je; ++j, ++g) {
            if (!wait_phase(bar(T::B_KFULL + T::kv_slot(g)), T::kv_phase(g), ctl, SITE_K_FULL)) return;
            ptx::mbar_arrive_remote_relaxed(lead(T::B_PEER_K + (int)T::kv_slot(g)));
        }
    }
}

template <int D, bool CAUSAL, bool ALT>
__device__ void pair_forward_v(const FwdParams& p, uint32_t bar0, uint32_t lead_bar0, const Ctl& ctl) {
    using T = PairTraits<D>;
    uint32_t g = 0;
    const PairSched<CAUSAL, ALT> sc(p);
    for (int64_t pos = sc.first(p); sc.valid(pos, p);) {
        const Seg sg = sc.seg(pos, p);
        pos = sc.next(pos, sg, p);
        for (int j = sg.jb; j < sg.je; ++j, ++g) {
            if (!wait_phase(bar0 + 8u * (T::B_VFULL + T::kv_slot(g)), T::kv_phase(g), ctl, SITE_V_FULL)) return;
            ptx::mbar_arrive_remote_relaxed(lead_bar0 + 8u * (T::B_PEER_V + T::kv_slot(g)));
        }
    }
}

// ------------------------------------------------------------ even CTA: issuers
// S_g = Q K_gᵀ for both CTAs' tiles: M = 256 (each CTA's 128 query rows),
// N = 128 keys (64 from each CTA's K half), K = D.
template <int D, bool CAUSAL, bool BF16, bool ALT>
__device__ void pair_mma_qk(const FwdParams& p, uint32_t sbase, uint32_t bar0, uint32_t tmem, const Ctl& ctl) {
    using T = PairTraits<D>;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    const uint32_t IDESC = ptx::idesc_f16(2 * BM, T::BN, BF16, false, false) | (p.negate_s ? ptx::IDESC_NEGATE_A : 0u);
    constexpr uint32_t HI = ptx::smem_desc_hi(8 * T::SW, T::SWIZZLE_CODE);
    const uint32_t q_lo0 = ptx::smem_desc_lo(sbase + T::OFF_Q, 16);
    const uint32_t k_lo0 = ptx::smem_desc_lo(sbase + T::OFF_K, 16);
    uint32_t qi = 0, g = 0;
    bool ok = true;
    const PairSched<CAUSAL, ALT> sc(p);
    for (int64_t pos = sc.first(p); ok && sc.valid(pos, p);) {
        const Seg sg = sc.seg(pos, p);
        if (!seg_checked<0, T::BN>(sg, p, ctl, SITE_CHECK_MMA_S)) { ok = false; break; }
        pos = sc.next(pos, sg, p);
        const uint32_t qs = qi % T::Q_STAGES, qph = (qi / T::Q_STAGES) & 1u;
        if (!wait_phase(bar(T::B_QFULL + qs), qph, ctl, SITE_Q_FULL) ||
            !wait_phase(bar(T::B_PEER_Q + qs), qph, ctl, SITE_PEER_Q)) { ok = false; break; }
        const uint32_t q_lo = q_lo0 + qs * (T::Q_BYTES >> 4);
        for (int j = sg.jb; j < sg.je; ++j, ++g) {
            const uint32_t kb = T::kv_slot(g), r = rslot<T::SR>(g);
            if (!wait_phase(bar(T::B_KFULL + kb), T::kv_phase(g), ctl, SITE_K_FULL) ||
                !wait_phase(bar(T::B_PEER_K + kb), T::kv_phase(g), ctl, SITE_PEER_K)) { ok = false; break; }
            // the score slot held S_{g - SR}: free once both CTAs have loaded it
            if (g >= (uint32_t)T::SR &&
                !wait_phase(bar(T::B_SFREE + r), rphase<T::SR>(g - T::SR), ctl, SITE_S_FREE)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            const uint32_t k_lo = k_lo0 + kb * (T::KH_BYTES >> 4);
            const uint32_t d_tmem = tmem + T::TM_S + r * T::BN;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t a_off = (((kk * 16) / T::SWE) * (BM * T::SW) + ((kk * 16) % T::SWE) * 2) >> 4;
                const uint32_t b_off = (((kk * 16) / T::SWE) * ((T::BN / 2) * T::SW) + ((kk * 16) % T::SWE) * 2) >> 4;
                ptx::mma2_ss(d_tmem, ptx::desc64(q_lo + a_off, HI), ptx::desc64(k_lo + b_off, HI), IDESC,
                             kk > 0 ? 1u : 0u);
            }
            ptx::tc_commit2(bar(T::B_SFULL + r), 3);   // S ready in both CTAs
            ptx::tc_commit2(bar(T::B_KEMPTY + kb), 3);  // their K slots free
            if (j == sg.je - 1) {
                ptx::tc_commit2(bar(T::B_QEMPTY + qs), 3);
                ++qi;
            }
        }
    }
    // every product this thread issued completes (and its arrivals land)
    // before the CTAs may leave
    ptx::tc_commit2(bar(T::B_DRAIN), 1);
    if (!drain_phase(bar(T::B_DRAIN), 0u, ctl.limit_ns)) record_timeout(ctl, SITE_DRAIN);
}

// O += P_g V_g for both CTAs: M = 256 (P from each CTA's TMEM), N = D
// (columns 0-63 from the even CTA's V half, 64-127 from the odd CTA's),
// K = 128 keys.
template <int D, bool CAUSAL, bool BF16, bool ALT>
__device__ void pair_mma_pv(const FwdParams& p, uint32_t sbase, uint32_t bar0, uint32_t tmem, const Ctl& ctl) {
    using T = PairTraits<D>;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    constexpr uint32_t IDESC = ptx::idesc_f16(2 * BM, D, BF16, false, true);   // V is MN-major
    constexpr uint32_t HI = ptx::smem_desc_hi(8 * T::SW, T::SWIZZLE_CODE);
    const uint32_t v_lo0 = ptx::smem_desc_lo(sbase + T::OFF_V, T::VH_BYTES);
    uint32_t g = 0, ntile = 0;
    bool ok = true;
    const PairSched<CAUSAL, ALT> sc(p);
    for (int64_t pos = sc.first(p); ok && sc.valid(pos, p); ++ntile) {
        const Seg sg = sc.seg(pos, p);
        if (!seg_checked<0, T::BN>(sg, p, ctl, SITE_CHECK_MMA_PV)) { ok = false; break; }
        pos = sc.next(pos, sg, p);
        for (int j = sg.jb; j < sg.je; ++j, ++g) {
            const uint32_t vb = T::kv_slot(g), r = rslot<T::PR>(g);
            if (j == sg.jb && ntile > 0 &&
                !wait_phase(bar(T::B_OFREE), (ntile - 1) & 1u, ctl, SITE_O_FREE)) { ok = false; break; }
            if (!wait_phase(bar(T::B_PFULL + r), rphase<T::PR>(g), ctl, SITE_P_FULL)) { ok = false; break; }
            if (!wait_phase(bar(T::B_VFULL + vb), T::kv_phase(g), ctl, SITE_V_FULL) ||
                !wait_phase(bar(T::B_PEER_V + vb), T::kv_phase(g), ctl, SITE_PEER_V)) { ok = false; break; }
            ptx::tc_fence_after();
            const uint32_t v_lo = v_lo0 + vb * (T::VH_BYTES >> 4);
            const uint32_t a_tmem = tmem + T::TM_P + r * (T::BN / 2);  // P_g in its own slot
            const uint32_t acc0 = j > sg.jb ? 1u : 0u;
#pragma unroll
            for (int kk = 0; kk < T::BN / 16; ++kk)
                ptx::mma2_ts(tmem + T::TM_O, a_tmem + kk * 8, ptx::desc64(v_lo + ((kk * 16 * T::SW) >> 4), HI), IDESC,
                             kk > 0 ? 1u : acc0);
            ptx::tc_commit2(bar(T::B_PVDONE + r), 3);   // O updated, P slot free
            ptx::tc_commit2(bar(T::B_VEMPTY + vb), 3);  // V slots free
        }
    }
    ptx::tc_commit2(bar(T::B_DRAIN + 1), 1);
    if (!drain_phase(bar(T::B_DRAIN + 1), 0u, ctl.limit_ns)) record_timeout(ctl, SITE_DRAIN);
}

// ------------------------------------------------------------ kernel --------
// Launched in clusters of two (one CTA per SM); the grid is twice the number
// of co-resident clusters or of units, whichever is smaller.
template <int D, bool CAUSAL, bool BF16, bool ALT>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(CHAIN_THREADS, 1)
    fa_fwd_pair_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                       const FwdParams p) {
    using T = PairTraits<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = ptx::smem_addr(smem);
    const uint32_t bar0 = sbase + T::OFF_BAR;
    float* hand = reinterpret_cast<float*>(smem + T::OFF_HAND);
    float* mx = reinterpret_cast<float*>(smem + T::OFF_RED);
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + T::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + T::OFF_MISC + 4);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t rank = ptx::cluster_ctarank();
    const bool lead = rank == 0;
    const uint32_t lead_bar0 = ptx::mapa_shared(bar0, 0);

    if (threadIdx.x == 0) {
        for (int i = 0; i < T::NUM_BARS; ++i) ptx::mbar_init(bar0 + 8u * i, T::bar_count(i));
        *abort_flag = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tmQ);
        ptx::prefetch_tmap(&tmK);
        ptx::prefetch_tmap(&tmV);
        ptx::prefetch_tmap(&tmO);
    }
    if (warp == 1) {
        ptx::tmem_alloc2(ptx::smem_addr(const_cast<uint32_t*>(tmem_slot)), T::TMEM_COLS);
        ptx::tmem_relinquish2();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const Ctl ctl{abort_flag, p.status, p.wait_limit_ns};
    // both CTAs' barriers are initialised before either CTA arrives on the other's
    ptx::cluster_sync();
    ptx::grid_dependency_wait();
    ptx::grid_launch_dependents();

    const int wg = warp / 4;
    const ChainPair<D, CAUSAL, ALT> cp{bar0, lead_bar0, lead};
    if (wg == 0) {
        ptx::setmaxnreg_dec<CHAIN_REG_CTRL>();
        if (lane == 0) {
            if (warp == 0) {
                pair_producer_qk<D, CAUSAL, ALT>(&tmQ, &tmK, p, sbase, bar0, rank, ctl);
            } else if (warp == 1) {
                if (lead) pair_mma_qk<D, CAUSAL, BF16, ALT>(p, sbase, bar0, tmem, ctl);
                else pair_forward_qk<D, CAUSAL, ALT>(p, bar0, lead_bar0, ctl);
            } else if (warp == 2) {
                if (lead) pair_mma_pv<D, CAUSAL, BF16, ALT>(p, sbase, bar0, tmem, ctl);
                else pair_forward_v<D, CAUSAL, ALT>(p, bar0, lead_bar0, ctl);
            } else {
                pair_producer_v<D, CAUSAL, ALT>(&tmV, p, sbase, bar0, rank, ctl);
            }
        }
    } else if (wg < 3) {
        ptx::setmaxnreg_inc<CHAIN_REG_SOFTMAX>();
        chain_softmax<D, CAUSAL, BF16>(p, cp, tmem, hand, mx, wg - 1, ctl);
    } else {
        ptx::setmaxnreg_dec<CHAIN_REG_EPI>();
        chain_epilogue<D, CAUSAL, BF16>(&tmO, p, cp, sbase, tmem, hand, ctl);
    }

    ptx::tc_fence_before();
    __syncthreads();
    // neither CTA frees its TMEM or leaves while the other may still reach it
    ptx::cluster_sync();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc2(tmem, T::TMEM_COLS);
    }
}

}  // namespace fa
