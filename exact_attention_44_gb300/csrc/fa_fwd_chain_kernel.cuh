// Fused attention forward for head dims up to 128 with two softmax chains:
// O = softmax(Q Kᵀ · scale) V and the per-row log-sum-exp, whole query tiles.
//
// The method is the tiled online-softmax forward of the pages ("Write Triton
// Attention Kernel", Required reasoning process steps 1-9 and Kernel design
// rules; "Build Triton-Ascend Fused Attention", Implementation Pattern;
// "把 FlashAttention 搬上昇腾：Triton-Ascend CV Pipeline 优化实战", section 一: exp2
// with scale·log2(e), fp32 state, P cast to the input type; section 八: the
// causal loop bound).  That blog keeps the matrix unit busy by letting the
// vector unit's softmax of one block overlap the matrix products of others
// (sections 三, 四).  Here the tensor-core side is the one-tile kernel's:
// warp 0 loads Q and K, warp 3 V, warp 1 issues S_g = Q K_gᵀ into a ring of
// three TMEM score slots, warp 2 issues O += P_g V_g (fa_fwd_kernel.cuh).
// What changes is the softmax: one chain of warps working through the key
// blocks one after another cannot keep up with the tensor core (per 128 x 128
// block it waits for the scores, loads them, takes the row maximum, runs 16384
// exponentials through the MUFU unit and stores P, and only then starts the
// next block), so two chains take the blocks in turn:
//
//   warpgroup 1 (chain 0): blocks g = 0, 2, 4, ...   thread = query row,
//   warpgroup 2 (chain 1): blocks g = 1, 3, 5, ...   all 128 scores in registers
//
// and each has two blocks' worth of tensor-core time for one block.  The
// online softmax is sequential in its running maximum m; the chains keep it
// consistent through a per-row hand-off: after taking the maximum of block g
// the chain publishes the m that blocks 0..g settled on, and the chain of
// block g+1 reads it before its exponentials.  As in the one-tile kernel, m
// moves only when a block maximum exceeds it by more than 2^RESCALE_LOG2;
// the chain that moves it rescales O in TMEM (after the P·V of block g-1 has
// completed, before its own P is released).  Each chain keeps its own part
// of the row sum l, referenced to the m it last saw (rescaled when it learns
// of a larger one), and the epilogue combines them:
//     m = max(m_0, m_1),   l = l_0 · 2^(m_0 − m) + l_1 · 2^(m_1 − m).
// Warpgroup 3 is the epilogue (O / l -> input type -> TMA tensor stores,
// lse = (m + log2 l)·ln 2).  setmaxnreg moves registers from warpgroups 0
// and 3 to the softmax chains.  Every mbarrier wait is bounded; on expiry
// the CTA records the site in the status word, stops every role, lets its
// copies and MMAs land and frees TMEM.
#pragma once

#include <type_traits>

#include "fa_fwd_kernel.cuh"

namespace fa {

constexpr int CHAIN_THREADS = 512;  // four warpgroups
// registers per thread of each warpgroup after setmaxnreg; launched with 128
// each (512 threads, one CTA per SM), the budgets add up to the same total
constexpr uint32_t CHAIN_REG_CTRL = 72;      // warpgroup 0: loads and MMA issue
constexpr uint32_t CHAIN_REG_SOFTMAX = 176;  // warpgroups 1, 2: the softmax chains
constexpr uint32_t CHAIN_REG_EPI = 88;       // warpgroup 3: epilogue
static_assert(128 * (CHAIN_REG_CTRL + 2 * CHAIN_REG_SOFTMAX + CHAIN_REG_EPI) == CHAIN_THREADS * 128,
              "register budgets of the warpgroups");

// Key pairs (of every 16) whose exponentials the chain softmax computes on the
// FMA pipe (ptx::exp2_poly2) instead of the MUFU unit, in blocks without a
// masked key.  None: measured on GB300 (Z8 H16 N2048, D 16/32/64, fp16, both
// masks), giving 2, 4, 6 or 8 pairs of every 16 to the polynomial made every
// shape slower, by 10-15 % at 2 and 30-40 % at 8 -- a packed FMA pair costs two
// pipe cycles and the polynomial needs ~8 of them plus integer work, against
// 8 XU cycles for two MUFU ex2, so it only trades one busy pipe for another
// and adds issue slots; the softmax here is bound by its latency chain.
constexpr int chain_emu_pairs(int D) { return D < 0 ? 1 : 0; }

// The one-tile kernel's shared memory, TMEM and barrier layout (so that its
// producers and MMA issuers run unchanged), with the softmax regions and
// arrival counts of two chains of 128 threads:
//   hand-over to the epilogue, per tile slot: m_0, l_0, m_1, l_1 per row
//     (in the region of the one-tile kernel's hand-over);
//   hand-off of m between the chains, two slots by block parity (in the
//     region of its partial-maximum exchange), completion on B_RED.
template <int D>
struct ChainTraits : Traits<D> {
    using T = Traits<D>;
    static_assert(D <= 128 && T::BN == 128, "two-chain kernel: head dims up to 128");
    static_assert(4 * BM * 4 * 2 <= 2 * T::HAND_ROWS * BM * 4, "epilogue hand-over fits");
    static_assert(2 * BM * 4 <= 2 * T::NG * BM * 4, "m hand-off fits");
    // arrivals are one per warp (ptx::mbar_arrive_warp)
    static __device__ __forceinline__ uint32_t bar_count(int i) {
        if (i >= T::B_PFULL && i < T::B_PFULL + T::SR) return 4;        // one chain writes P_g
        if (i >= T::B_EPIFULL && i < T::B_EPIFULL + 2) return 8;        // both chains hand over
        if (i >= T::B_EPIEMPTY && i < T::B_OFREE + 1) return 4;         // epilogue
        if (i >= T::B_RED && i < T::B_RED + 2) return 4;                // one chain publishes m
        return 1;
    }
};

// What the softmax chains and the epilogue need from their kernel: the
// TMEM and barrier layout (L), the tile schedule (S), the scope of their
// waits, and how "P_g written" and "O read" reach the P·V issuer.  One CTA:
// every thread arrives on the CTA's own barrier.
// kSplitP: P_g goes to a ring of its own (L::PR slots of BN / 2 columns at
// L::TM_P) instead of over the first columns of S_g, so that the score slot
// is released (arrive_sfree) as soon as the scores are loaded, and the P slot
// once O += P V of the block that used it last is complete.
template <int D, bool CAUSAL, bool ALT>
struct ChainSolo {
    using L = Traits<D>;
    using S = Sched<CAUSAL, L::BN, false, ALT>;
    static constexpr bool kCluster = false;
    static constexpr bool kSplitP = false;
    static constexpr int kCheckVar = ALT ? 4 : 0;  // the schedule seg_checked validates
    uint32_t bar0;
    __device__ __forceinline__ void arrive_p(uint32_t r) const { ptx::mbar_arrive_warp(bar0 + 8u * (L::B_PFULL + r)); }
    __device__ __forceinline__ void arrive_sfree(uint32_t) const {}
    __device__ __forceinline__ void arrive_ofree() const { ptx::mbar_arrive_warp(bar0 + 8u * L::B_OFREE); }
};

// ------------------------------------------------------------ softmax chain -
// Chain `ch` (0 or 1) of the online softmax: the key blocks g with g % 2 ==
// ch, counting every block of every tile this CTA runs.  Thread = query row
// = TMEM lane; the block's 128 scores sit in the thread's registers.
template <int D, bool CAUSAL, bool BF16, class C>
__device__ void chain_softmax(const FwdParams& p, const C& cp, uint32_t tmem, float* hand, float* mx, int ch,
                              const Ctl& ctl) {
    using T = typename C::L;
    constexpr int BN = T::BN;
    constexpr bool CL = C::kCluster;
    const uint32_t bar0 = cp.bar0;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    const int quad = (threadIdx.x / 32) % 4;  // TMEM lane quadrant this warp may access
    const int row = quad * 32 + threadIdx.x % 32;
    const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
    const uint32_t o_addr = tmem + lane_addr + T::TM_O;
    const float c = p.scale_log2;  // > 0: a negative scale negates S instead
    const uint64_t c2 = ptx::pack_f32x2(c, c);
    uint32_t g = 0, ntile = 0;
    const typename C::S sc(p);
    for (int64_t pos = sc.first(p); sc.valid(pos, p); ++ntile) {
        const Seg ti = sc.seg(pos, p);
        if (!seg_checked<C::kCheckVar, BN>(ti, p, ctl, SITE_CHECK_SOFTMAX)) return;
        pos = sc.next(pos, ti, p);
        const int q_row = ti.q_start + row;
        float m = -INFINITY, l = 0.f;  // this chain's view of the running max, its part of the row sum
        bool have = false;             // a block of this tile went through this chain
        for (int j = ti.jb; j < ti.je; ++j, ++g) {
            if ((g & 1u) != (uint32_t)ch) continue;
            const uint32_t r = rslot<T::SR>(g);
            if (!warp_wait_phase<CL>(bar(T::B_SFULL + r), rphase<T::SR>(g), ctl, SITE_S_FULL)) return;
            ptx::tc_fence_after();
            const uint32_t s_addr = tmem + lane_addr + T::TM_S + r * BN;
            const uint32_t pr = rslot<T::PR>(g);
            uint32_t p_addr = s_addr;  // P over the first BN / 2 columns of the score slot
            if constexpr (C::kSplitP) p_addr = tmem + lane_addr + T::TM_P + pr * (BN / 2);
            float s[BN];
            {
                uint32_t r0[32], r1[32], r2[32], r3[32];
                ptx::tmem_ld32_issue(s_addr, r0);
                ptx::tmem_ld32_issue(s_addr + 32, r1);
                ptx::tmem_ld32_issue(s_addr + 64, r2);
                ptx::tmem_ld32_issue(s_addr + 96, r3);
                ptx::tmem_wait_ld();
                if constexpr (C::kSplitP) {
                    // the scores are in registers: S_{g + SR} may overwrite the slot
                    ptx::tc_fence_before();
                    cp.arrive_sfree(r);
                }
                ptx::reg_fence32(r0);
                ptx::reg_fence32(r1);
                ptx::reg_fence32(r2);
                ptx::reg_fence32(r3);
#pragma unroll
                for (int x = 0; x < 32; ++x) {
                    s[x] = __uint_as_float(r0[x]);
                    s[32 + x] = __uint_as_float(r1[x]);
                    s[64 + x] = __uint_as_float(r2[x]);
                    s[96 + x] = __uint_as_float(r3[x]);
                }
            }
            // the mask goes on the scores before the row max (Correctness
            // requirements); only the diagonal block and the key tail need it
            const int k0 = j * BN;
            const bool masked = (CAUSAL && k0 + BN - 1 > ti.q_start) || (k0 + BN > p.Nkv);
            if (masked) {
                const int kmax = (CAUSAL ? min(p.Nkv - 1, q_row) : p.Nkv - 1) - k0;  // last kept key of this row
#pragma unroll
                for (int x = 0; x < BN; ++x)
                    if (x > kmax) s[x] = -INFINITY;
            }
            float mx0 = fmaxf(s[0], s[1]), mx1 = fmaxf(s[2], s[3]), mx2 = fmaxf(s[4], s[5]), mx3 = fmaxf(s[6], s[7]);
#pragma unroll
            for (int x = 8; x < BN; x += 8) {
                mx0 = ptx::fmax3(mx0, s[x], s[x + 1]);
                mx1 = ptx::fmax3(mx1, s[x + 2], s[x + 3]);
                mx2 = ptx::fmax3(mx2, s[x + 4], s[x + 5]);
                mx3 = ptx::fmax3(mx3, s[x + 6], s[x + 7]);
            }
            // Every processed block of a whole tile holds a kept key of every
            // row (a causal tile stops at its diagonal block, the key tail
            // block starts below Nkv), so the block maximum is finite.
            const float m_blk = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * c;
            // The running maximum after block g - 1 (the other chain's block),
            // published once that chain had taken its decision.  Every block
            // waits for it, also at a tile's first block (where it belongs to
            // the previous tile and is not used): so each hand-off slot is read
            // before the chain that wrote it writes it again.
            float m_prev = -INFINITY;
            if (g > 0) {
                const uint32_t h = (g - 1u) & 1u;
                if (!warp_wait_phase<CL>(bar(T::B_RED + h), ((g - 1u) >> 1) & 1u, ctl, SITE_MAX_XCHG)) return;
                m_prev = mx[h * BM + row];
            }
            float alpha = 1.f;
            bool rescale = false;
            if (j == ti.jb) {
                m = m_blk;  // the tile's first block sets the reference maximum
                l = 0.f;
            } else {
                if (!have) {
                    m = m_prev;  // this chain's first block of the tile
                    l = 0.f;
                } else if (m_prev > m) {
                    l *= ptx::ex2(m - m_prev);  // the other chain moved m (and rescaled O)
                    m = m_prev;
                }
                // m moves only when a row maximum runs more than 2^RESCALE_LOG2
                // ahead of it; then O and l are rescaled by alpha before this
                // block is added to them ("Write Triton Attention Kernel",
                // Kernel design rules).  A warp decides as one (TMEM access).
                if (__any_sync(0xffffffffu, m_blk > m + RESCALE_LOG2)) {
                    const float m_new = fmaxf(m, m_blk);
                    alpha = ptx::ex2(m - m_new);
                    m = m_new;
                    l *= alpha;
                    rescale = true;
                }
            }
            have = true;
            // publish the maximum blocks 0..g settled on for the chain of block g + 1
            mx[(g & 1u) * BM + row] = m;
            ptx::mbar_arrive_warp(bar(T::B_RED + (g & 1u)));
            // p = 2^(s·c − m): l sums the fp32 p, the P·V product takes p cast
            // to the input type, over the first BN/2 columns of the slot.  In
            // a block with no masked key, EMU of every 16 key pairs take the
            // polynomial exponential on the FMA pipe and the others the MUFU
            // unit's ex2, whose throughput otherwise bounds this loop.
            if constexpr (C::kSplitP) {
                // the P slot held P_{g - PR}: free once that block's P·V is complete
                if (g >= (uint32_t)T::PR &&
                    !warp_wait_phase<CL>(bar(T::B_PVDONE + pr), rphase<T::PR>(g - T::PR), ctl, SITE_P_FREE))
                    return;
                ptx::tc_fence_after();
            }
            const uint64_t negm2 = ptx::pack_f32x2(-m, -m);
            uint64_t sum_a = ptx::pack_f32x2(0.f, 0.f), sum_b = sum_a;
            auto exps = [&](auto emu) {
                constexpr int EMU = decltype(emu)::value;
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                    uint32_t pk[16];
#pragma unroll
                    for (int x = 0; x < 16; ++x) {
                        const int k = c4 * 32 + 2 * x;
                        const uint64_t a2 = ptx::ffma2(ptx::pack_f32x2(s[k], s[k + 1]), c2, negm2);
                        float p0, p1;
                        if (x < EMU) {
                            ptx::unpack_f32x2(ptx::exp2_poly2(a2), p0, p1);
                        } else {
                            float a0, a1;
                            ptx::unpack_f32x2(a2, a0, a1);
                            p0 = ptx::ex2(a0);
                            p1 = ptx::ex2(a1);
                        }
                        if (x & 1) sum_b = ptx::fadd2(sum_b, ptx::pack_f32x2(p0, p1));
                        else sum_a = ptx::fadd2(sum_a, ptx::pack_f32x2(p0, p1));
                        pk[x] = pack2<BF16>(p0, p1);
                    }
                    // keys 32·c4 .. at packed columns 16·c4 .. (of the score slot:
                    // scores this thread has read)
                    ptx::tmem_st16(p_addr + 16 * c4, pk);
                }
            };
            constexpr int EMU = chain_emu_pairs(D);
            if (EMU > 0 && !masked) exps(std::integral_constant<int, EMU>{});
            else exps(std::integral_constant<int, 0>{});
            if (rescale) {
                // O holds every block up to g - 1 once that block's P·V is complete
                if (!warp_wait_phase<CL>(bar(T::B_PVDONE + rslot<T::PR>(g - 1u)), rphase<T::PR>(g - 1u), ctl,
                                         SITE_PV_DONE))
                    return;
                ptx::tc_fence_after();
                rescale_o<D>(o_addr, alpha);
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            cp.arrive_p(pr);
            float sa, sb, sc2, sd;
            ptx::unpack_f32x2(sum_a, sa, sb);
            ptx::unpack_f32x2(sum_b, sc2, sd);
            l += (sa + sb) + (sc2 + sd);
        }
        // hand this chain's (m, l) of the tile to the epilogue (-inf, 0 if
        // no block of the tile went through this chain)
        const uint32_t slot = ntile & 1u;
        if (!warp_wait_phase<CL>(bar(T::B_EPIEMPTY + slot), ((ntile >> 1) & 1u) ^ 1u, ctl, SITE_EPI_EMPTY)) return;
        hand[(slot * 4 + 2 * ch) * BM + row] = have ? m : -INFINITY;
        hand[(slot * 4 + 2 * ch + 1) * BM + row] = l;
        ptx::mbar_arrive_warp(bar(T::B_EPIFULL + slot));
    }
}

// ------------------------------------------------------------ epilogue ------
// O = acc / l in the input type through shared memory and TMA tensor stores
// (one 32-row box per warp and swizzle chunk), lse = (m + log2 l)·ln 2
// ("Write Triton Attention Kernel", steps 6-8), with m and l combined from
// the two chains; O is released to the P·V issuer as soon as it is read.
template <int D, bool CAUSAL, bool BF16, class C>
__device__ void chain_epilogue(const CUtensorMap* tmO, const FwdParams& p, const C& cp, uint32_t sbase,
                               uint32_t tmem, const float* hand, const Ctl& ctl) {
    using T = typename C::L;
    constexpr bool CL = C::kCluster;
    const uint32_t bar0 = cp.bar0;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    const int quad = (threadIdx.x / 32) % 4;
    const int row = quad * 32 + threadIdx.x % 32;
    const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
    const int lane = threadIdx.x % 32;
    const uint32_t stage = sbase + T::OFF_OST + (uint32_t)quad * 32u * T::SW;  // this warp's staging rows
    uint32_t step = 0, ntile = 0;
    auto drain = [&]() {
        if (lane == 0) ptx::bulk_wait_all();
    };
    const typename C::S sc(p);
    for (int64_t pos = sc.first(p); sc.valid(pos, p); ++ntile) {
        const Seg ti = sc.seg(pos, p);
        if (!seg_checked<C::kCheckVar, T::BN>(ti, p, ctl, SITE_CHECK_EPILOGUE)) {
            drain();
            return;
        }
        pos = sc.next(pos, ti, p);
        step += ti.je - ti.jb;
        const uint32_t slot = ntile & 1u;
        if (!warp_wait_phase<CL>(bar(T::B_EPIFULL + slot), (ntile >> 1) & 1u, ctl, SITE_EPI_FULL)) {
            drain();
            return;
        }
        const float m0 = hand[(slot * 4 + 0) * BM + row], l0 = hand[(slot * 4 + 1) * BM + row];
        const float m1 = hand[(slot * 4 + 2) * BM + row], l1 = hand[(slot * 4 + 3) * BM + row];
        ptx::mbar_arrive_warp(bar(T::B_EPIEMPTY + slot));
        // O is referenced to the larger maximum (m only grows from block to
        // block); a chain without a block of the tile has m = -inf, l = 0
        const float m = fmaxf(m0, m1);
        const float l = l0 * ptx::ex2(m0 - m) + l1 * ptx::ex2(m1 - m);
        const uint32_t g = step - 1;  // the tile's last P·V
        if (!warp_wait_phase<CL>(bar(T::B_PVDONE + rslot<T::PR>(g)), rphase<T::PR>(g), ctl, SITE_PV_DONE)) {
            drain();
            return;
        }
        ptx::tc_fence_after();
        const int q_row = ti.q_start + row;
        tma_store_rows<D, T::SW, BF16>(tmem + lane_addr + T::TM_O, 1.f / l, stage, tmO, ti.q_start + 32 * quad,
                                       ti.hq, ti.z, ti.q_start + 32 * quad < p.Nq, [&]() {
                                           // all of O has been read: the next tile's P·V may overwrite it
                                           ptx::tc_fence_before();
                                           cp.arrive_ofree();
                                       });
        if (q_row < p.Nq && p.lse != nullptr) p.lse[ti.lse0 + q_row] = (m + log2f(l)) * 0.6931471805599453f;
    }
    drain();
}

// ------------------------------------------------------------ kernel --------
template <int D, bool CAUSAL, bool BF16, bool ALT>
__global__ void __launch_bounds__(CHAIN_THREADS, 1)
    fa_fwd_chain_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                        const FwdParams p) {
    using T = Traits<D>;
    using CT = ChainTraits<D>;
    constexpr int VAR = ALT ? 4 : 0;  // the producers' and issuers' schedule: whole tiles
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = ptx::smem_addr(smem);
    const uint32_t bar0 = sbase + T::OFF_BAR;
    float* hand = reinterpret_cast<float*>(smem + T::OFF_HAND);
    float* mx = reinterpret_cast<float*>(smem + T::OFF_RED);
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + T::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + T::OFF_MISC + 4);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        for (int i = 0; i < T::NUM_BARS; ++i) ptx::mbar_init(bar0 + 8u * i, CT::bar_count(i));
        *abort_flag = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tmQ);
        ptx::prefetch_tmap(&tmK);
        ptx::prefetch_tmap(&tmV);
        ptx::prefetch_tmap(&tmO);
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
    // launched as a programmatic dependent of the previous kernel on the
    // stream: the set-up above overlaps its tail, nothing below touches
    // global memory before it has completed
    ptx::grid_dependency_wait();
    ptx::grid_launch_dependents();

    const int wg = warp / 4;
    if (wg == 0) {
        ptx::setmaxnreg_dec<CHAIN_REG_CTRL>();
        if (lane == 0) {
            if (warp == 0) run_producer_qk<D, CAUSAL, VAR>(&tmQ, &tmK, p, sbase, bar0, ctl);
            else if (warp == 1) run_mma_qk<D, CAUSAL, BF16, VAR>(p, sbase, bar0, tmem, ctl);
            else if (warp == 2) run_mma_pv<D, CAUSAL, BF16, VAR>(p, sbase, bar0, tmem, ctl);
            else run_producer_v<D, CAUSAL, VAR>(&tmV, p, sbase, bar0, ctl);
        }
    } else if (wg < 3) {
        ptx::setmaxnreg_inc<CHAIN_REG_SOFTMAX>();
        chain_softmax<D, CAUSAL, BF16>(p, ChainSolo<D, CAUSAL, ALT>{bar0}, tmem, hand, mx, wg - 1, ctl);
    } else {
        ptx::setmaxnreg_dec<CHAIN_REG_EPI>();
        chain_epilogue<D, CAUSAL, BF16>(&tmO, p, ChainSolo<D, CAUSAL, ALT>{bar0}, sbase, tmem, hand, ctl);
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, T::TMEM_COLS);
    }
}

}  // namespace fa
