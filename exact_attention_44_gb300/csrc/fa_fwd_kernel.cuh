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
//   * one persistent CTA per SM walks a static schedule (Sched): whole
//     128-row query tiles, or, in split mode, one equal range of
//     (tile, key block) pairs per CTA whose cut tiles a second kernel merges;
//   * warp 0 (one lane) streams Q once per segment and K_j per key block, warp
//     3 (one lane) V_j, by TMA into swizzled shared-memory rings guarded by
//     mbarriers;
//   * warp 1 (one lane) issues S_g = Q K_gᵀ into a three-slot ring in TMEM,
//     warp 2 (one lane) O += P_g V_g with P_g read from the same slot; each
//     commits to mbarriers, so S of later blocks runs while the softmax works;
//   * warps 4 .. 4 + 4 NG - 1 (NG column groups x 128 threads, thread = query
//     row = TMEM lane) run the online softmax: mask (diagonal and tail blocks
//     only), row max swapped between the groups, exp2, row sum, P -> fp16/bf16
//     into TMEM;
//     O is rescaled in TMEM only when a row maximum grows by more than
//     2^RESCALE_LOG2 (below that the stale maximum keeps every
//     p <= 2^RESCALE_LOG2, and O / l and lse are unchanged);
//   * the last 4 warps run the epilogue of the previous segment while the softmax
//     warps start the next: read O out of TMEM, release it to the P·V issuer,
//     then O / l -> global and lse = (m + log2 l)·ln 2 (or the part's O / l
//     and base-2 lse -> workspace).
// Every mbarrier wait is bounded; on expiry the CTA records the site in the
// status word, stops every role, lets its copies and MMAs land and frees TMEM.
#pragma once

#include <climits>

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
    static constexpr int PR = SR;                              // P_g lives in its score slot
    static constexpr uint32_t TM_S = 0;                        // S/P ring slot r at TM_S + r * BN
    static constexpr uint32_t TM_O = SR * BN;                  // O
    static constexpr uint32_t TMEM_COLS = 512;
    static_assert(TM_O + D <= TMEM_COLS, "tensor memory budget");
    // shared memory (offsets from a 1024-byte aligned base)
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + Q_STAGES * Q_BYTES;
    static constexpr int OFF_V = OFF_K + KV_STAGES * KV_BYTES;
    // softmax -> epilogue hand-over, 2 slots of {m, l of each column group} per row
    // softmax column groups: four keep each thread's chain per key block
    // short; at D = 256 two (the 64-key blocks are narrow, and four groups
    // of 768 threads leave too few registers for the 256-column epilogue)
    static constexpr int NG = D == 256 ? 2 : 4;
    static constexpr int THREADS = fwd_threads(NG);
    static constexpr int HAND_ROWS = 1 + NG;
    static constexpr int OFF_HAND = OFF_V + KV_STAGES * KV_BYTES;
    // partial row maxima of the column groups, 2 slots (by block parity)
    static constexpr int OFF_RED = OFF_HAND + 2 * HAND_ROWS * BM * 4;
    // O staging for the tensor stores: 32 rows x one swizzle chunk per
    // epilogue warp, aligned to the swizzle pattern's 1024-byte period
    static constexpr int OFF_OST = (OFF_RED + 2 * NG * BM * 4 + 1023) / 1024 * 1024;
    static constexpr int OFF_BAR = OFF_OST + BM * SW;
    // barrier indices
    static constexpr int B_QFULL = 0;
    static constexpr int B_QEMPTY = B_QFULL + Q_STAGES;
    static constexpr int B_KFULL = B_QEMPTY + Q_STAGES;        // [2] K tile landed (TMA)
    static constexpr int B_VFULL = B_KFULL + KV_STAGES;        // [2] V tile landed (TMA)
    static constexpr int B_SFULL = B_VFULL + KV_STAGES;        // [SR] S_g ready; K slot free (commit)
    static constexpr int B_PFULL = B_SFULL + SR;               // [SR] P_g written (all softmax threads)
    static constexpr int B_PVDONE = B_PFULL + SR;              // [SR] O += P_g V_g complete; slot and V slot free (commit)
    static constexpr int B_EPIFULL = B_PVDONE + SR;            // [2] m, l of a tile handed over (softmax threads)
    static constexpr int B_EPIEMPTY = B_EPIFULL + 2;           // [2] hand-over slot read (128)
    static constexpr int B_OFREE = B_EPIEMPTY + 2;             // O read out of TMEM (128)
    static constexpr int B_RED = B_OFREE + 1;                  // [2] every group's partial maxima written
    static constexpr int B_DRAIN = B_RED + 2;                  // [2] teardown of the two MMA issuers
    static constexpr int NUM_BARS = B_DRAIN + 2;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;    // tmem base, abort flag
    static constexpr int SMEM_USED = OFF_MISC + 16;
    // >= 120 KB keeps one CTA per SM, so no CTA ever waits on another's TMEM
    static constexpr int SMEM_BYTES = (SMEM_USED + 1024) > 120 * 1024 ? SMEM_USED + 1024 : 120 * 1024;
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");

    static __device__ __forceinline__ uint32_t bar_count(int i) {
        if (i >= B_PFULL && i < B_PFULL + SR) return 128 * NG;
        if (i >= B_EPIFULL && i < B_EPIFULL + 2) return 128 * NG;
        if (i >= B_EPIEMPTY && i < B_OFREE + 1) return 128;
        if (i >= B_RED && i < B_RED + 2) return 128 * NG;
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
// another role has aborted or after limit_ns, recording the site.  CLUSTER:
// the phase may complete through arrivals from the other CTA of a pair, whose
// writes the wait then acquires (cluster scope).
template <bool CLUSTER = false>
__device__ __forceinline__ bool try_phase(uint32_t bar, uint32_t parity) {
    if constexpr (CLUSTER) return ptx::mbar_try_wait_cluster(bar, parity);
    else return ptx::mbar_try_wait(bar, parity);
}
template <bool CLUSTER = false>
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, const Ctl& c, uint32_t site) {
    if (try_phase<CLUSTER>(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    for (;;) {
        if (try_phase<CLUSTER>(bar, parity)) return true;
        if (*c.abort_flag) return false;
        if (ptx::globaltimer_ns() - t0 > c.limit_ns) {
            record_timeout(c, site);
            return false;
        }
    }
}

// The same wait taken by a whole warp: every lane leaves with the same answer,
// so no lane can run ahead into a warp-collective tcgen05 access alone.
template <bool CLUSTER = false>
__device__ __forceinline__ bool warp_wait_phase(uint32_t bar, uint32_t parity, const Ctl& c, uint32_t site) {
    return __all_sync(0xffffffffu, wait_phase<CLUSTER>(bar, parity, c, site));
}

// Teardown wait after an abort: ignores the abort flag, bounded by limit_ns.
template <bool CLUSTER = false>
__device__ __forceinline__ bool drain_phase(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    const uint64_t t0 = ptx::globaltimer_ns();
    while (!try_phase<CLUSTER>(bar, parity))
        if (ptx::globaltimer_ns() - t0 > limit_ns) return false;
    return true;
}

// The kernel's VAR argument: kind 0 plain (fa_fwd), 1 window / variable
// length, 2 the same with ALiBi; bit 4 set: plain with alternating causal
// rounds (see the schedule).
__host__ __device__ constexpr int var_kind(int var) { return var & 3; }
__host__ __device__ constexpr bool var_alt(int var) { return (var & 4) != 0; }

// One unit of a CTA's work: key blocks [jb, je) of the query tile
// (z, hq, q_start), whose whole key range is [0, nkv).
struct Seg {
    int z, hq, hk, q_start;
    int nkv;     // key blocks the whole tile visits
    int jb, je;  // the key blocks of this segment
    int slot;    // -1: the whole tile, finished into O and lse; else the partial-result slot
    // the tile's sequence: query and key lengths, first packed rows, the
    // batch coordinate of the tensor maps, and where its lse rows start
    int nq, nk, qrow0, krow0, zc;
    int64_t lse0;
};

// The key block visited at step j (jb <= j < je) of a segment.  With an
// ALiBi bias (kind 2) the block holding the tile's diagonal goes first: it
// holds every row's largest bias (0 at the row's own key), so the running
// maximum it sets is not exceeded by more than the rescale threshold later
// and the other blocks, in order after it, redo no exponentials and leave O
// unscaled.  (In plain order a causal tile meets ever larger biases, and
// with a slope of 1/2 each 128-key block raised the maximum by 64.)  The
// online softmax gives the same result in any order.  Otherwise block j.
template <int VAR, int BN>
__device__ __forceinline__ int key_block(const Seg& sg, int j) {
    if constexpr (var_kind(VAR) != 2) {
        return j;
    } else {
        int d = (sg.q_start + BM / 2) / BN;  // the block of the tile's middle row's own key
        d = d < sg.jb ? sg.jb : (d > sg.je - 1 ? sg.je - 1 : d);
        if (j == sg.jb) return d;
        return j - 1 >= d ? j : j - 1;  // the others in order, d skipped
    }
}

// Debug builds (compiled with FA_DEBUG_CHECKS=1; `python -m
// exact_attention_44_gb300.build --debug-checks`) check every unit a role
// decodes against the launch's sizes before the role touches memory for it:
// batch, query head, key/value head (and its GQA relation), first query row,
// key-block range and partial-result slot.  A unit outside them records
// STATUS_DEVICE_CHECK with the role's site in the status word and raises the
// CTA's abort flag, so every role stops at its next wait and the kernel ends
// as after a timed-out wait (copies and products land, TMEM is freed).  No
// trap or device assert is used.  Release builds compile the checks away.
#ifndef FA_DEBUG_CHECKS
#define FA_DEBUG_CHECKS 0
#endif

template <int VAR, int BN>
__device__ __forceinline__ bool seg_checked(const Seg& s, const FwdParams& p, const Ctl& c, uint32_t site) {
    if constexpr (!FA_DEBUG_CHECKS) {
        return true;
    } else {
        const bool packed = var_kind(VAR) != 0 && p.cu_q != nullptr;
        const int nb = packed ? 1 : p.Z;  // batch extent of the tensor maps
        const int tk = (s.nk + BN - 1) / BN;
        bool ok = s.z >= 0 && s.z < p.Z && s.zc >= 0 && s.zc < nb && s.hq >= 0 && s.hq < p.Hq && s.hk >= 0 &&
                  s.hk < p.Hkv && s.hk == s.hq / p.group && s.q_start >= 0 && s.q_start % BM == 0 &&
                  s.qrow0 >= 0 && s.krow0 >= 0 && s.nq >= 0 && s.nk >= 0 && s.qrow0 + s.nq <= p.Nq &&
                  s.krow0 + s.nk <= p.Nkv && s.jb >= 0 && s.jb < s.je && s.je <= s.nkv && s.lse0 >= 0 &&
                  s.lse0 + (packed ? 0 : s.nq) <= (int64_t)p.Z * p.Hq * p.Nq &&
                  s.slot >= -1 && s.slot < 2 * (int)gridDim.x;
        // a key block past the keys: allowed only as a variant tile's single
        // block whose rows keep no key (it is masked whole)
        // (a CTA pair of query blocks 2m, 2m + 1 may hold a tile past the rows)
        if (var_kind(VAR) == 0) ok = ok && s.je <= tk && (s.q_start < s.nq || p.pair == 2);
        else ok = ok && (s.je <= tk || s.je == s.jb + 1);
        if (!ok) {
            *c.abort_flag = 1;
            atomicCAS(c.status, 0u, STATUS_DEVICE_CHECK | (site << 8) | ((blockIdx.x & 0xFFFFu) << 16));
        }
        return ok;
    }
}

// Barrier slot and phase parity of key block g (global count) in a ring of R.
template <int R>
__device__ __forceinline__ uint32_t rslot(uint32_t g) { return g % R; }
template <int R>
__device__ __forceinline__ uint32_t rphase(uint32_t g) { return (g / R) & 1u; }

// The static schedule, in one of two modes.
//
// Tile mode (split == 0): CTA c takes one whole tile per round of `grid`
// tiles.  Non-causal tiles go head-major, CTA c taking tiles c, c + grid, ...,
// so the CTAs running at the same time share a head's K/V in L2.  Causal
// ones go in groups of p.head_group heads, sized on the host so that a
// group's K/V fits in a third of L2; within a group
// from the last query block (most key blocks) to the first with the group's
// heads innermost, so the heavy tiles go first and the light ones fill the
// tail, and the tiles of a head run close together in time.  (With every
// head in one group, 1024 heads of N = 1024 re-read each head's K/V from
// DRAM for each of its query blocks.)  With ALT (its own kernel
// instantiation, so that the plain order compiles as if it did not exist)
// the causal rounds alternate direction (CTA c takes tile c of round 0, tile
// grid - 1 - c of round 1, ...), so a CTA that drew a heavier tile in one
// round draws a lighter one in the next; the host picks it only for long
// tiles, where it was measured faster (causal_alternates in the host code).
//
// Split mode (split != 0): the (tile, key block) pairs of all tiles, tiles
// head-major and query blocks ascending, are laid end to end and cut into
// `grid` equal ranges, one per CTA.  A tile that a cut crosses leaves a
// partial result (O / l in fp32 and the base-2 log-sum-exp of the part) in a
// slot of the workspace: slot 2c holds the part CTA c starts with, slot 2c + 1
// the part it ends with; a second kernel merges the parts of each cut tile.
//
// A causal tile stops at the key block holding its last row ("Write Triton
// Attention Kernel", step 9).  Positions are tiles in tile mode and
// (tile, key block) pairs in split mode.
template <bool CAUSAL, int BN, bool VAR = false, bool ALT = false>
struct Sched {
    int64_t hi;  // split mode: end of this CTA's range

    static __host__ __device__ __forceinline__ int tile_nkv(int mb, const FwdParams& p) {
        if (!CAUSAL) return p.Tk;
        const int end = mb * BM + BM < p.Nq ? mb * BM + BM : p.Nq;
        const int n = (end - 1) / BN + 1;
        return n < p.Tk ? n : p.Tk;
    }
    // key blocks visited by query blocks 0 .. mb-1 of one head: for a causal
    // block m below the last, tile_nkv(m) = min(Tk, r (m + 1)) with r = BM / BN
    static __host__ __device__ __forceinline__ int64_t head_prefix(int mb, const FwdParams& p) {
        if (!CAUSAL) return (int64_t)mb * p.Tk;
        constexpr int64_t r = BM / BN;
        const int64_t full = p.Tk / r;  // blocks m with r (m + 1) <= Tk
        const int64_t m = mb < full ? mb : full;
        return r * m * (m + 1) / 2 + (mb - m) * (int64_t)p.Tk;
    }
    // tile mode: the tile at position pos = round * grid + c (CTA c), in 32 bits
    static __host__ __device__ __forceinline__ int64_t tile_at(int64_t pos, int grid) {
        if (!CAUSAL || !ALT) return pos;
        const uint32_t x = (uint32_t)pos, g = (uint32_t)grid, round = x / g;
        return (round & 1u) ? (int64_t)(2u * round * g + g - 1u - x) : pos;
    }
    // tile mode, causal: tile t of the order above.  Tile indices fit in 32
    // bits (the host checks Z * Hq * Tq), and 32-bit divisions keep this
    // short: every role runs it at the start of every tile.
    static __host__ __device__ __forceinline__ void causal_tile(int64_t t64, const FwdParams& p, int64_t& head,
                                                                int& mb) {
        const uint32_t t = (uint32_t)t64, heads = (uint32_t)(p.Z * p.Hq), G = (uint32_t)p.head_group;
        const uint32_t tq = (uint32_t)p.Tq;
        const uint32_t g0 = t / (G * tq) * G;             // first head of t's group
        const uint32_t gc = heads - g0 < G ? heads - g0 : G;  // heads in the group
        const uint32_t w = t - g0 * tq;                   // t's place in the group
        const uint32_t r = w / gc;
        mb = (int)(tq - 1 - r);
        head = g0 + (w - r * gc);
    }
    // split mode: first position of tile (head, mb), and the tile holding position x
    static __host__ __device__ __forceinline__ int64_t tile_pos(int64_t head, int mb, const FwdParams& p) {
        return head * p.head_blocks + head_prefix(mb, p);
    }
    static __host__ __device__ __forceinline__ void tile_of(int64_t x, const FwdParams& p, int64_t& head, int& mb) {
        head = x / p.head_blocks;
        const int64_t rem = x - head * p.head_blocks;
        if (!CAUSAL) {
            mb = (int)(rem / p.Tk);
        } else {  // largest mb with head_prefix(mb) <= rem
            int lo = 0, up = p.Tq - 1;
            while (lo < up) {
                const int mid = (lo + up + 1) / 2;
                if (head_prefix(mid, p) <= rem) lo = mid;
                else up = mid - 1;
            }
            mb = lo;
        }
    }
    // split mode: range of CTA c is [range_lo(c), range_lo(c + 1)); cta_of(x)
    // is the CTA whose range holds x (every range is non-empty: grid <= total)
    static __host__ __device__ __forceinline__ int64_t range_lo(int64_t c, int64_t grid, const FwdParams& p) {
        return p.total_blocks * c / grid;
    }
    static __host__ __device__ __forceinline__ int64_t cta_of(int64_t x, int64_t grid, const FwdParams& p) {
        return ((x + 1) * grid + p.total_blocks - 1) / p.total_blocks - 1;
    }

    __device__ explicit Sched(const FwdParams& p) : hi(p.split ? range_lo(blockIdx.x + 1, gridDim.x, p) : 0) {}
    // the variant schedule skips tiles past the end of their sequence
    __device__ __forceinline__ int64_t skip_empty(int64_t pos, const FwdParams& p) const {
        if constexpr (VAR) {
            for (; tile_at(pos, gridDim.x) < p.ntiles; pos += gridDim.x) {
                const Seg t = var_seg(pos, p);
                if (t.q_start < t.nq) break;
            }
        }
        return pos;
    }
    __device__ __forceinline__ int64_t first(const FwdParams& p) const {
        if constexpr (VAR) return skip_empty(blockIdx.x, p);
        return p.split ? range_lo(blockIdx.x, gridDim.x, p) : (int64_t)blockIdx.x;
    }
    __device__ __forceinline__ bool valid(int64_t pos, const FwdParams& p) const {
        if (VAR || !p.split) return tile_at(pos, gridDim.x) < p.ntiles;
        return pos < hi;
    }
    __device__ __forceinline__ int64_t next(int64_t pos, const Seg& sg, const FwdParams& p) const {
        if constexpr (VAR) return skip_empty(pos + gridDim.x, p);
        return p.split ? pos + (sg.je - sg.jb) : pos + gridDim.x;
    }
    __device__ __forceinline__ Seg seg(int64_t pos, const FwdParams& p) const {
        if constexpr (VAR) return var_seg(pos, p);
        Seg s;
        int64_t head;
        int mb;
        if (p.split) {
            tile_of(pos, p, head, mb);
        } else if (CAUSAL) {
            causal_tile(tile_at(pos, gridDim.x), p, head, mb);
        } else {
            const uint32_t t = (uint32_t)pos, h = t / (uint32_t)p.Tq;
            head = h;
            mb = (int)(t - h * (uint32_t)p.Tq);
        }
        {
            const uint32_t hz = (uint32_t)head / (uint32_t)p.Hq;  // head < Z * Hq < 2^31
            s.z = (int)hz;
            s.hq = (int)((uint32_t)head - hz * (uint32_t)p.Hq);
        }
        s.hk = s.hq / p.group;  // GQA: kv head = q head // (Hq / Hkv)
        s.q_start = mb * BM;
        s.nkv = tile_nkv(mb, p);
        s.nq = p.Nq;
        s.nk = p.Nkv;
        s.qrow0 = 0;
        s.krow0 = 0;
        s.zc = s.z;
        s.lse0 = head * p.Nq;
        if (p.split) {
            const int64_t t0 = tile_pos(head, mb, p);
            s.jb = (int)(pos - t0);
            s.je = hi - t0 < s.nkv ? (int)(hi - t0) : s.nkv;
            s.slot = (s.jb == 0 && s.je == s.nkv) ? -1 : 2 * (int)blockIdx.x + (s.jb > 0 ? 0 : 1);
        } else {
            s.jb = 0;
            s.je = s.nkv;
            s.slot = -1;
        }
        return s;
    }

    // Variant tiles (whole tiles only): the sequence's lengths and packed
    // offsets, and the key blocks that hold a kept key for some row of the
    // tile -- at least one block, so that a tile whose rows keep no key at
    // all still finishes them (as O = 0, lse = -inf).
    __device__ __forceinline__ Seg var_seg(int64_t pos, const FwdParams& p) const {
        Seg s;
        int head, mb;
        if (CAUSAL) {
            int64_t h64;
            causal_tile(tile_at(pos, gridDim.x), p, h64, mb);
            head = (int)h64;
        } else {
            const uint32_t t = (uint32_t)pos, h = t / (uint32_t)p.Tq;
            head = (int)h;
            mb = (int)(t - h * (uint32_t)p.Tq);
        }
        s.z = head / p.Hq;
        s.hq = head - s.z * p.Hq;
        s.hk = s.hq / p.group;
        s.q_start = mb * BM;
        if (p.cu_q != nullptr) {
            const int q0 = __ldg(p.cu_q + s.z), q1 = __ldg(p.cu_q + s.z + 1);
            const int k0 = __ldg(p.cu_k + s.z), k1 = __ldg(p.cu_k + s.z + 1);
            // clamp to the packed extents so that no store leaves the tensors
            s.qrow0 = q0 < 0 ? 0 : (q0 > p.Nq ? p.Nq : q0);
            s.krow0 = k0 < 0 ? 0 : (k0 > p.Nkv ? p.Nkv : k0);
            const int nq = q1 - s.qrow0, nk = k1 - s.krow0;
            s.nq = nq < 0 ? 0 : (nq > p.Nq - s.qrow0 ? p.Nq - s.qrow0 : nq);
            s.nk = nk < 0 ? 0 : (nk > p.Nkv - s.krow0 ? p.Nkv - s.krow0 : nk);
            s.zc = 0;
            s.lse0 = (int64_t)s.hq * p.Nq + s.qrow0;
        } else {
            s.nq = p.Nq;
            s.nk = p.Nkv;
            s.qrow0 = 0;
            s.krow0 = 0;
            s.zc = s.z;
            s.lse0 = (int64_t)head * p.Nq;
        }
        const int q_last = (s.q_start + BM < s.nq ? s.q_start + BM : s.nq) - 1;
        int hi_key = s.nk - 1;
        if (CAUSAL && q_last < hi_key) hi_key = q_last;
        if (p.win_right >= 0 && q_last + p.win_right < hi_key) hi_key = q_last + p.win_right;
        const int lo_key = (p.win_left >= 0 && s.q_start - p.win_left > 0) ? s.q_start - p.win_left : 0;
        const int tk = (s.nk + BN - 1) / BN;
        int jb = lo_key / BN;
        if (jb > tk - 1) jb = tk > 0 ? tk - 1 : 0;
        const int je = hi_key >= lo_key ? hi_key / BN + 1 : jb + 1;
        s.jb = jb;
        s.je = je > jb ? je : jb + 1;
        s.nkv = s.je;
        s.slot = -1;
        return s;
    }
};

// ------------------------------------------------------------ TMA producers -
// Two threads load: one Q and K (the S stream's operands), one V (the P·V
// stream's), so a K load never queues behind a V slot that is still in use.
// With two Q slots the next tile's Q is requested right after the current
// tile's first K: its slot held the tile before, whose last S is complete by
// the time the second K's slot frees anyway.

template <int D, bool CAUSAL, int VAR>
__device__ void run_producer_qk(const CUtensorMap* tmQ, const CUtensorMap* tmK, const FwdParams& p, uint32_t sbase,
                                uint32_t bar0, const Ctl& ctl) {
    using T = Traits<D>;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    const uint64_t pol_q = ptx::policy_evict_first();
    const uint64_t pol_kv = ptx::policy_evict_last();
    uint32_t qi = 0, ki = 0;  // loads issued into each ring
    bool ok = true;
    bool withheld = false;
    auto load_q = [&](const Seg& sg) -> bool {
        if (!seg_checked<VAR, T::BN>(sg, p, ctl, SITE_CHECK_LOAD_QK)) return false;
        const uint32_t s = qi % T::Q_STAGES, ph = (qi / T::Q_STAGES) & 1u;
        if (!wait_phase(bar(T::B_QEMPTY + s), ph ^ 1u, ctl, SITE_Q_EMPTY)) return false;
        ptx::mbar_arrive_expect_tx(bar(T::B_QFULL + s), T::Q_BYTES);
        const uint32_t dst = sbase + T::OFF_Q + s * T::Q_BYTES;
        for (int c = 0; c < T::NCHUNK; ++c)
            ptx::tma_load_4d(dst + c * (BM * T::SW), tmQ, bar(T::B_QFULL + s), c * T::SWE, sg.qrow0 + sg.q_start,
                             sg.hq, sg.zc, pol_q);
        ++qi;
        return true;
    };
    const Sched<CAUSAL, T::BN, (var_kind(VAR) != 0), var_alt(VAR)> sc(p);
    int64_t pos = sc.first(p);
    if (sc.valid(pos, p)) ok = load_q(sc.seg(pos, p));
    while (ok && sc.valid(pos, p)) {
        const Seg sg = sc.seg(pos, p);
        if (!seg_checked<VAR, T::BN>(sg, p, ctl, SITE_CHECK_LOAD_QK)) { ok = false; break; }
        const int64_t nxt = sc.next(pos, sg, p);
        for (int j = sg.jb; j < sg.je; ++j) {
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
                    ptx::tma_load_4d(dst + c * (T::BN * T::SW), tmK, bar(T::B_KFULL + s), c * T::SWE,
                                     sg.krow0 + key_block<VAR, T::BN>(sg, j) * T::BN, sg.hk, sg.zc, pol_kv);
            }
            ++ki;
            // with two Q slots the next segment's Q can go right after the
            // first K; with one, only after the last K (its slot frees at this
            // segment's last S, which needs that K)
            const int q_at = T::Q_STAGES >= 2 ? sg.jb : sg.je - 1;
            if (j == q_at && sc.valid(nxt, p) && !load_q(sc.seg(nxt, p))) {
                ok = false;
                break;
            }
        }
        pos = nxt;
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

template <int D, bool CAUSAL, int VAR>
__device__ void run_producer_v(const CUtensorMap* tmV, const FwdParams& p, uint32_t sbase, uint32_t bar0,
                               const Ctl& ctl) {
    using T = Traits<D>;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    const uint64_t pol_kv = ptx::policy_evict_last();
    uint32_t vi = 0;
    bool ok = true;
    const Sched<CAUSAL, T::BN, (var_kind(VAR) != 0), var_alt(VAR)> sc(p);
    for (int64_t pos = sc.first(p); ok && sc.valid(pos, p);) {
        const Seg sg = sc.seg(pos, p);
        if (!seg_checked<VAR, T::BN>(sg, p, ctl, SITE_CHECK_LOAD_V)) { ok = false; break; }
        for (int j = sg.jb; j < sg.je; ++j) {
            // slot vi & 1 held block vi - 2, free once its P·V is complete
            const uint32_t s = vi & 1u;
            if (vi >= 2 && !wait_phase(bar(T::B_PVDONE + rslot<T::SR>(vi - 2)), rphase<T::SR>(vi - 2), ctl,
                                       SITE_V_EMPTY)) { ok = false; break; }
            ptx::mbar_arrive_expect_tx(bar(T::B_VFULL + s), T::KV_BYTES);
            const uint32_t dst = sbase + T::OFF_V + s * T::KV_BYTES;
            for (int c = 0; c < T::NCHUNK; ++c)
                ptx::tma_load_4d(dst + c * (T::BN * T::SW), tmV, bar(T::B_VFULL + s), c * T::SWE,
                                 sg.krow0 + key_block<VAR, T::BN>(sg, j) * T::BN, sg.hk, sg.zc, pol_kv);
            ++vi;
        }
        pos = sc.next(pos, sg, p);
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
template <int D, bool CAUSAL, bool BF16, int VAR>
__device__ void run_mma_qk(const FwdParams& p, uint32_t sbase, uint32_t bar0, uint32_t tmem, const Ctl& ctl) {
    using T = Traits<D>;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    // Q, K both K-major; with a negative scale Q is negated (the kernel's c is |scale|·log2e)
    const uint32_t IDESC = ptx::idesc_f16(BM, T::BN, BF16, false, false) | (p.negate_s ? ptx::IDESC_NEGATE_A : 0u);
    constexpr uint32_t HI = ptx::smem_desc_hi(8 * T::SW, T::SWIZZLE_CODE);     // 8-row swizzle atoms
    const uint32_t q_lo0 = ptx::smem_desc_lo(sbase + T::OFF_Q, 16);
    const uint32_t k_lo0 = ptx::smem_desc_lo(sbase + T::OFF_K, 16);
    uint32_t qi = 0, g = 0;  // Q tiles and S blocks issued
    bool ok = true;
    const Sched<CAUSAL, T::BN, (var_kind(VAR) != 0), var_alt(VAR)> sc(p);
    for (int64_t pos = sc.first(p); ok && sc.valid(pos, p);) {
        const Seg sg = sc.seg(pos, p);
        if (!seg_checked<VAR, T::BN>(sg, p, ctl, SITE_CHECK_MMA_S)) { ok = false; break; }
        pos = sc.next(pos, sg, p);
        const uint32_t qs = qi % T::Q_STAGES;
        if (!wait_phase(bar(T::B_QFULL + qs), (qi / T::Q_STAGES) & 1u, ctl, SITE_Q_FULL)) { ok = false; break; }
        const uint32_t q_lo = q_lo0 + qs * (T::Q_BYTES >> 4);
        for (int j = sg.jb; j < sg.je; ++j, ++g) {
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
            if (j == sg.je - 1) {
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

// O += P_g V_g (step 5h); the first block of a segment overwrites O, once
// the epilogue has read the previous segment's O out of TMEM
template <int D, bool CAUSAL, bool BF16, int VAR>
__device__ void run_mma_pv(const FwdParams& p, uint32_t sbase, uint32_t bar0, uint32_t tmem, const Ctl& ctl) {
    using T = Traits<D>;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    constexpr uint32_t IDESC = ptx::idesc_f16(BM, D, BF16, false, true);      // V is MN-major (D contiguous)
    constexpr uint32_t HI = ptx::smem_desc_hi(8 * T::SW, T::SWIZZLE_CODE);
    const uint32_t v_lo0 = ptx::smem_desc_lo(sbase + T::OFF_V, T::BN * T::SW);  // LBO: next column chunk of V
    uint32_t g = 0, ntile = 0;
    bool ok = true;
    const Sched<CAUSAL, T::BN, (var_kind(VAR) != 0), var_alt(VAR)> sc(p);
    for (int64_t pos = sc.first(p); ok && sc.valid(pos, p); ++ntile) {
        const Seg sg = sc.seg(pos, p);
        if (!seg_checked<VAR, T::BN>(sg, p, ctl, SITE_CHECK_MMA_PV)) { ok = false; break; }
        pos = sc.next(pos, sg, p);
        for (int j = sg.jb; j < sg.je; ++j, ++g) {
            const uint32_t vb = g & 1u, r = rslot<T::SR>(g);
            if (j == sg.jb && ntile > 0 &&
                !wait_phase(bar(T::B_OFREE), (ntile - 1) & 1u, ctl, SITE_O_FREE)) { ok = false; break; }
            if (!wait_phase(bar(T::B_PFULL + r), rphase<T::SR>(g), ctl, SITE_P_FULL)) { ok = false; break; }
            if (!wait_phase(bar(T::B_VFULL + vb), (g >> 1) & 1u, ctl, SITE_V_FULL)) { ok = false; break; }
            ptx::tc_fence_after();
            const uint32_t v_lo = v_lo0 + vb * (T::KV_BYTES >> 4);
            const uint32_t a_tmem = tmem + T::TM_S + r * T::BN;  // P_g over the first BN/2 columns of the slot
            const uint32_t acc0 = j > sg.jb ? 1u : 0u;
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
    } else if constexpr (NCOL == 8) {
        uint32_t r[8];
        ptx::tmem_ld8(taddr, r);
#pragma unroll
        for (int x = 0; x < 8; ++x) r[x] = __float_as_uint(__uint_as_float(r[x]) * alpha);
        ptx::tmem_st8(taddr, r);
    } else {
        uint32_t r[4];
        ptx::tmem_ld4(taddr, r);
#pragma unroll
        for (int x = 0; x < 4; ++x) r[x] = __float_as_uint(__uint_as_float(r[x]) * alpha);
        ptx::tmem_st4(taddr, r);
    }
}

// Online softmax for one column group of every key block: 128 threads, thread
// = query row = TMEM lane; the groups swap partial row maxima through shared
// memory, so all reference the same maximum m, and each keeps its own
// partial denominator (the epilogue adds them).
template <int D, bool CAUSAL, bool BF16, int VAR>
__device__ void run_softmax(const FwdParams& p, uint32_t bar0, uint32_t tmem, float* hand, float* red, int h,
                            const Ctl& ctl) {
    using T = Traits<D>;
    constexpr int BN = T::BN;
    constexpr int NG = T::NG;                  // column groups; h is this thread's
    constexpr int HC = BN / NG;                // score columns per thread
    static_assert(HC == 16 || HC == 32, "column group width");
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    const int quad = (threadIdx.x / 32) % 4;  // TMEM lane quadrant this warp may access
    const int row = quad * 32 + threadIdx.x % 32;
    const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
    const float c = p.scale_log2;
    // with an ALiBi bias (the kind 2 instantiation) the scores are scaled
    // and biased in place (units of log2), so the maximum and the
    // exponentials take them as they are
    constexpr bool bias = var_kind(VAR) == 2;
    const float cm = bias ? 1.f : c;
    const uint64_t c2 = ptx::pack_f32x2(cm, cm);
    uint32_t step = 0, ntile = 0;

    const Sched<CAUSAL, BN, (var_kind(VAR) != 0), var_alt(VAR)> sc(p);
    for (int64_t pos = sc.first(p); sc.valid(pos, p); ++ntile) {
        const Seg ti = sc.seg(pos, p);
        if (!seg_checked<VAR, BN>(ti, p, ctl, SITE_CHECK_SOFTMAX)) return;
        pos = sc.next(pos, ti, p);
        const int q_row = ti.q_start + row;
        float slope2 = 0.f;
        if constexpr (bias) slope2 = -__ldg(p.alibi + ti.hq) * 1.4426950408889634f;
        // running max (log2 units of the scaled score) and denominator, fp32
        // ("Write Triton Attention Kernel", step 4; the initial l is 0)
        float m = -INFINITY, l = 0.f;
        for (int j = ti.jb; j < ti.je; ++j) {
            const uint32_t r = rslot<T::SR>(step);      // ring slot of S_j / P_j
            const uint32_t b = step & 1u, ph = (step >> 1) & 1u;  // max-exchange slot
            if (!warp_wait_phase(bar(T::B_SFULL + r), rphase<T::SR>(step), ctl, SITE_S_FULL)) return;
            ptx::tc_fence_after();
            const uint32_t s_addr = tmem + lane_addr + T::TM_S + r * BN;
            float s[HC];
            {
                uint32_t rr[HC];
                if constexpr (HC == 32) ptx::tmem_ld32(s_addr + h * HC, rr);
                else ptx::tmem_ld16(s_addr + h * HC, rr);
#pragma unroll
                for (int x = 0; x < HC; ++x) s[x] = __uint_as_float(rr[x]);
            }
            // the mask goes on the scores before the row max (Correctness
            // requirements); only the diagonal block and the key tail need it
            const int kj = key_block<VAR, BN>(ti, j);  // the key block of this step
            const int k0 = kj * BN + h * HC;
            if constexpr (var_kind(VAR) == 0) {
                const bool need_mask = (CAUSAL && kj * BN + BN - 1 > ti.q_start) || (kj * BN + BN > p.Nkv);
                if (need_mask) {
                    const int kmax = CAUSAL ? min(p.Nkv - 1, q_row) : p.Nkv - 1;  // last kept key for this row
#pragma unroll
                    for (int x = 0; x < HC; ++x)
                        if (k0 + x > kmax) s[x] = -INFINITY;
                }
            } else {
                // kept keys of this row: kmin .. kmax (sequence end, causal
                // diagonal, window sides); the mask is applied only when some
                // row of the tile loses a key of this block
                const int blast = kj * BN + BN - 1;
                bool full = blast < ti.nk;
                if (CAUSAL) full = full && blast <= ti.q_start;
                if (p.win_right >= 0) full = full && blast <= ti.q_start + p.win_right;
                if (p.win_left >= 0) full = full && kj * BN >= ti.q_start + BM - 1 - p.win_left;
                if (!full) {
                    int kmax = ti.nk - 1;
                    if (CAUSAL) kmax = min(kmax, q_row);
                    if (p.win_right >= 0) kmax = min(kmax, q_row + p.win_right);
                    const int kmin = p.win_left >= 0 ? q_row - p.win_left : INT_MIN;
#pragma unroll
                    for (int x = 0; x < HC; ++x)
                        if (k0 + x > kmax || k0 + x < kmin) s[x] = -INFINITY;
                }
                if constexpr (bias) {
                    // scaled score plus -slope |i - j|, in log2 units.  When the
                    // whole block lies on one side of every row of the tile,
                    // |i - j| is linear in the key: the bias of a pair of keys
                    // advances by one packed add and joins the scaled scores in
                    // one packed FMA.  (The repeated adds round at most ~8 ulp
                    // of the largest bias of the 32 keys, which matters only
                    // where that bias is small: a key far from its row's
                    // maximum has p = 0 either way.)
                    const float d0 = (float)(q_row - k0);  // i - j at x = 0
                    if (blast <= ti.q_start || kj * BN >= ti.q_start + BM - 1) {
                        const float sgn = blast <= ti.q_start ? 1.f : -1.f;
                        const float b0 = slope2 * sgn * d0, step = -slope2 * sgn;
                        const uint64_t cs2 = ptx::pack_f32x2(c, c), inc2 = ptx::pack_f32x2(2.f * step, 2.f * step);
                        uint64_t b2 = ptx::pack_f32x2(b0, b0 + step);
#pragma unroll
                        for (int x = 0; x < HC; x += 2) {
                            ptx::unpack_f32x2(ptx::ffma2(ptx::pack_f32x2(s[x], s[x + 1]), cs2, b2), s[x], s[x + 1]);
                            b2 = ptx::fadd2(b2, inc2);
                        }
                    } else {
#pragma unroll
                        for (int x = 0; x < HC; ++x) s[x] = fmaf(s[x], c, slope2 * fabsf(d0 - (float)x));
                    }
                }
            }
            float mx0 = fmaxf(s[0], s[1]), mx1 = fmaxf(s[2], s[3]);
#pragma unroll
            for (int x = 4; x < HC; x += 4) {  // HC is a multiple of 4
                mx0 = ptx::fmax3(mx0, s[x], s[x + 1]);
                mx1 = ptx::fmax3(mx1, s[x + 2], s[x + 3]);
            }
            // Swap partial maxima with the other groups.  Arriving also says
            // this thread's S is in registers: P is written over the slot's
            // first columns only once every group has arrived.  (Exchange slot
            // b is free: every thread read it two blocks ago before arriving
            // last block.)
            const float pmax = fmaxf(mx0, mx1);
            red[(b * NG + h) * BM + row] = pmax;
            ptx::mbar_arrive(bar(T::B_RED + b));
            auto block_max = [&]() {
                float mm = pmax;
#pragma unroll
                for (int g2 = 0; g2 < NG; ++g2) mm = fmaxf(mm, red[(b * NG + g2) * BM + row]);
                return mm * cm;  // cm > 0 (a negative scale negates S instead)
            };
            if (j == ti.jb) {
                // the first block sets the reference maximum m
                if (!warp_wait_phase(bar(T::B_RED + b), ph, ctl, SITE_MAX_XCHG)) return;
                m = block_max();
            }
            // p = 2^(s·scale·log2e − m) against the current reference m; l sums
            // the fp32 p, P V uses p cast to the input type
            constexpr int NP = HC / 2;  // packed P columns of this group
            uint32_t pk[NP];
            auto exps = [&](float ref) -> uint64_t {
                // a row with no kept key so far (only in a segment that starts
                // past the diagonal of a causal tile) has p = 0, not 2^(-inf + inf)
                ref = ref == -INFINITY ? 0.f : ref;
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
            if (j > ti.jb) {
                // the block maximum arrives while the exponentials run; only
                // when it exceeds m by more than 2^RESCALE_LOG2 are P redone
                // against the new maximum, and O and l rescaled by alpha before
                // this block is added to them (Kernel design rules).  Both
                // halves see the same values, so both take the same branch.
                if (!warp_wait_phase(bar(T::B_RED + b), ph, ctl, SITE_MAX_XCHG)) return;
                const float m_tile = block_max();
                if (__any_sync(0xffffffffu, m_tile > m + RESCALE_LOG2)) {
                    const float m_new = fmaxf(m, m_tile);
                    // a row that has kept no key yet (m = -inf) has l = 0 and
                    // O = 0: alpha 0, not 2^(-inf + inf)
                    alpha = m == -INFINITY ? 0.f : ptx::ex2(m - m_new);
                    m = m_new;
                    sum2 = exps(m);
                    const uint32_t g = step - 1;
                    if (!warp_wait_phase(bar(T::B_PVDONE + rslot<T::SR>(g)), rphase<T::SR>(g), ctl, SITE_PV_DONE))
                        return;
                    ptx::tc_fence_after();
                    rescale_o<D / NG>(tmem + lane_addr + T::TM_O + h * (D / NG), alpha);
                }
            }
            // P_j over the first BN/2 columns of its slot: keys h*HC.. at packed column h*HC/2
            if constexpr (NP == 16) ptx::tmem_st16(s_addr + h * NP, pk);
            else ptx::tmem_st8(s_addr + h * NP, pk);
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(T::B_PFULL + r));
            float sl, sh;
            ptx::unpack_f32x2(sum2, sl, sh);
            l = l * alpha + (sl + sh);
            ++step;
        }
        // hand m and this column group's l to the epilogue warps
        const uint32_t slot = ntile & 1u;
        if (!warp_wait_phase(bar(T::B_EPIEMPTY + slot), ((ntile >> 1) & 1u) ^ 1u, ctl, SITE_EPI_EMPTY)) return;
        if (h == 0) hand[slot * T::HAND_ROWS * BM + row] = m;
        hand[slot * T::HAND_ROWS * BM + (1 + h) * BM + row] = l;
        ptx::mbar_arrive(bar(T::B_EPIFULL + slot));
    }
}

// One warp's 32 rows of a 128-lane TMEM block out to global memory through
// shared memory and TMA tensor stores.  The warp reads its TMEM lanes at
// columns taddr .. taddr + D - 1, multiplies by `mul` and converts to the
// input type; for each swizzle chunk (SW bytes of a row) it fills its 32-row
// staging area `stage` (1024-byte aligned, 32 * SW bytes) in the tensor map's
// swizzled layout -- 16-byte piece c of row `lane` at piece c ^ swz, bank
// conflict free -- and lane 0 stores the box at (chunk, row0, h, z) unless
// `store` is false.  Before refilling the area lane 0 waits until the previous
// box has been read out of it.  `after_read` runs in every lane once the last
// TMEM load is complete.  The caller's lane 0 must finish with
// bulk_wait_all() before the CTA exits.
template <int D, int SW, bool BF16, typename AfterRead>
__device__ __forceinline__ void tma_store_rows(uint32_t taddr, float mul, uint32_t stage, const CUtensorMap* map,
                                               int row0, int h, int z, bool store, AfterRead&& after_read) {
    constexpr int SWE = SW / 2;                 // elements per chunk row
    constexpr int CH = SWE >= 32 ? 32 : 16;     // columns per TMEM load
    const int lane = threadIdx.x % 32;
    const uint32_t swz = ((uint32_t)lane * SW >> 7) & (SW / 16 - 1);
#pragma unroll 1
    for (int k = 0; k < D / SWE; ++k) {
        uint32_t pk[SWE / 2];
#pragma unroll
        for (int i = 0; i < SWE / CH; ++i) {
            uint32_t r[CH];
            if constexpr (CH == 32) ptx::tmem_ld32(taddr + k * SWE + i * CH, r);
            else ptx::tmem_ld16(taddr + k * SWE + i * CH, r);
#pragma unroll
            for (int x = 0; x < CH / 2; ++x)
                pk[i * (CH / 2) + x] =
                    pack2<BF16>(__uint_as_float(r[2 * x]) * mul, __uint_as_float(r[2 * x + 1]) * mul);
        }
        if (k == D / SWE - 1) after_read();
        if (lane == 0) ptx::bulk_wait_read_all();
        __syncwarp();
#pragma unroll
        for (int c = 0; c < SW / 16; ++c)
            ptx::st_shared_v4(stage + (uint32_t)lane * SW + ((c ^ swz) << 4), pk[4 * c], pk[4 * c + 1], pk[4 * c + 2],
                              pk[4 * c + 3]);
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && store) {
            ptx::tma_store_4d(map, stage, k * SWE, row0, h, z);
            ptx::bulk_commit();
        }
    }
}

// ------------------------------------------------------------ epilogue ------
// O = acc / l in the input type, lse = m + log(l) in natural-log units
// ("Write Triton Attention Kernel", steps 6-8).  O is read out of TMEM and
// converted, TMEM is handed back to the MMA warp once all of it is read, and
// the rows go out through shared memory and TMA tensor stores: each warp
// stages its 32 rows one swizzle chunk at a time in its own quarter of the
// staging buffer, and its lane 0 stores the 32-row box.  (Stores of one row
// per thread put 32 rows into every warp instruction; measured on GB300 they
// slowed the softmax warps' shared-memory traffic by about 10 % at N = 1024.)
template <int D, bool CAUSAL, bool BF16, int VAR>
__device__ void run_epilogue(const CUtensorMap* tmO, const FwdParams& p, uint32_t sbase, uint32_t bar0, uint32_t tmem,
                             const float* hand, const Ctl& ctl) {
    using T = Traits<D>;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    const int quad = (threadIdx.x / 32) % 4;
    const int row = quad * 32 + threadIdx.x % 32;
    const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
    const int lane = threadIdx.x % 32;
    uint32_t step = 0, ntile = 0;
    constexpr int CH = D >= 32 ? 32 : 16;               // columns per TMEM load
    constexpr int HELD = D / CH < 2 ? D / CH : 2;        // chunks converted before their stores
    const uint32_t stage = sbase + T::OFF_OST + (uint32_t)quad * 32u * T::SW;  // this warp's staging rows
    // lane 0's stores must have read shared memory before the CTA exits
    auto drain = [&]() {
        if (lane == 0) ptx::bulk_wait_all();
    };
    const Sched<CAUSAL, T::BN, (var_kind(VAR) != 0), var_alt(VAR)> sc(p);
    for (int64_t pos = sc.first(p); sc.valid(pos, p); ++ntile) {
        const Seg ti = sc.seg(pos, p);
        if (!seg_checked<VAR, T::BN>(ti, p, ctl, SITE_CHECK_EPILOGUE)) {
            drain();
            return;
        }
        pos = sc.next(pos, ti, p);
        step += ti.je - ti.jb;
        const uint32_t slot = ntile & 1u;
        if (!warp_wait_phase(bar(T::B_EPIFULL + slot), (ntile >> 1) & 1u, ctl, SITE_EPI_FULL)) {
            drain();
            return;
        }
        const float m = hand[slot * T::HAND_ROWS * BM + row];
        float l = 0.f;
#pragma unroll
        for (int g2 = 0; g2 < T::NG; ++g2) l += hand[slot * T::HAND_ROWS * BM + (1 + g2) * BM + row];
        ptx::mbar_arrive(bar(T::B_EPIEMPTY + slot));
        const uint32_t g = step - 1;  // the tile's last P·V
        if (!warp_wait_phase(bar(T::B_PVDONE + rslot<T::SR>(g)), rphase<T::SR>(g), ctl, SITE_PV_DONE)) {
            drain();
            return;
        }
        ptx::tc_fence_after();

        if (ti.slot >= 0) {
            // part of a tile cut by the split schedule: O / l in fp32 and the
            // base-2 log-sum-exp of this part, for the merge kernel.  Slot
            // layout: float4 column group c4 of row r at [c4][r], then the
            // BM log-sum-exps, so a warp's 32 rows store 512 contiguous
            // bytes.  Rows past Nq are not stored (the merge skips them too).
            // A row with no kept key in the part (l = 0) gets O = 0 and -inf.
            const bool keep = ti.q_start + row < p.Nq;
            float* part = p.scratch + (int64_t)ti.slot * p.slot_floats;
            float4* pcol = reinterpret_cast<float4*>(part) + row;
            const float inv_l = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
            for (int i = 0; i < D / CH; ++i) {
                uint32_t r[CH];
                if constexpr (CH == 32) ptx::tmem_ld32(tmem + lane_addr + T::TM_O + i * CH, r);
                else ptx::tmem_ld16(tmem + lane_addr + T::TM_O + i * CH, r);
                if (keep) {
#pragma unroll
                    for (int x = 0; x < CH / 4; ++x)
                        pcol[(i * (CH / 4) + x) * BM] =
                            make_float4(__uint_as_float(r[4 * x]) * inv_l, __uint_as_float(r[4 * x + 1]) * inv_l,
                                        __uint_as_float(r[4 * x + 2]) * inv_l, __uint_as_float(r[4 * x + 3]) * inv_l);
                }
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(T::B_OFREE));
            if (keep) part[(int64_t)BM * D + row] = l > 0.f ? m + log2f(l) : -INFINITY;
            continue;
        }
        const int q_row = ti.q_start + row;
        const bool store = q_row < ti.nq;
        // a variant row with no kept key (l = 0) is finished as O = 0, lse = -inf
        const float inv_l = (var_kind(VAR) != 0 && !(l > 0.f)) ? 0.f : 1.f / l;
        // The tensor map clips rows past the tensor's end.  A warp whose rows
        // run past the end of a packed sequence (the next sequence's rows
        // follow) stores its rows one by one instead.
        if (var_kind(VAR) == 0 || p.cu_q == nullptr || ti.q_start + 32 * quad + 32 <= ti.nq) {
            // (a box that starts past the last row has nothing to store)
            tma_store_rows<D, T::SW, BF16>(tmem + lane_addr + T::TM_O, inv_l, stage, tmO,
                                           ti.qrow0 + ti.q_start + 32 * quad, ti.hq, ti.zc,
                                           ti.q_start + 32 * quad < ti.nq, [&]() {
                                               // all of O has been read: the MMA warp may overwrite it
                                               ptx::tc_fence_before();
                                               ptx::mbar_arrive(bar(T::B_OFREE));
                                           });
            if (store && p.lse != nullptr)
                p.lse[ti.lse0 + q_row] = (var_kind(VAR) != 0 && !(l > 0.f)) ? -INFINITY : (m + log2f(l)) * 0.6931471805599453f;
            continue;
        }
        uint8_t* orow = reinterpret_cast<uint8_t*>(p.o) +
                        2 * ((int64_t)ti.zc * p.so_z + (int64_t)ti.hq * p.so_h + (int64_t)(ti.qrow0 + q_row) * p.so_n);
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
            p.lse[ti.lse0 + q_row] = (var_kind(VAR) != 0 && !(l > 0.f)) ? -INFINITY : (m + log2f(l)) * 0.6931471805599453f;
    }
    drain();
}

// ------------------------------------------------------------ kernel --------
template <int D, bool CAUSAL, bool BF16, int VAR>
__global__ void __launch_bounds__(Traits<D>::THREADS, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                  const FwdParams p) {
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

    constexpr int SOFTMAX_END = 4 + 4 * T::NG;  // warps 4 .. SOFTMAX_END - 1: softmax; then 4 epilogue warps
    if (warp == 0) {
        if (lane == 0) run_producer_qk<D, CAUSAL, VAR>(&tmQ, &tmK, p, sbase, bar0, ctl);
    } else if (warp == 3) {
        if (lane == 0) run_producer_v<D, CAUSAL, VAR>(&tmV, p, sbase, bar0, ctl);
    } else if (warp == 1) {
        if (lane == 0) run_mma_qk<D, CAUSAL, BF16, VAR>(p, sbase, bar0, tmem, ctl);
    } else if (warp == 2) {
        if (lane == 0) run_mma_pv<D, CAUSAL, BF16, VAR>(p, sbase, bar0, tmem, ctl);
    } else if (warp < SOFTMAX_END) {
        run_softmax<D, CAUSAL, BF16, VAR>(p, bar0, tmem, hand, red, (warp - 4) / 4, ctl);
    } else {
        run_epilogue<D, CAUSAL, BF16, VAR>(&tmO, p, sbase, bar0, tmem, hand, ctl);
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, T::TMEM_COLS);
    }
}

// ------------------------------------------------------------ split merge ---
// Finishes every tile that the split schedule cut.  Block b - 1 looks at the
// cut between the ranges of CTAs b - 1 and b; the cuts inside a tile share
// its rows, each merging a slice from the part CTA c0 (which holds the
// tile's first block) ends with (slot 2 c0 + 1) and the parts CTAs
// c0 + 1 .. c1 start with (slots 2c).  With λ_s the base-2
// log-sum-exp of part s (over its keys) and O_s = its O / l,
//     λ = log2 Σ_s 2^λ_s,      O = Σ_s 2^(λ_s − λ) O_s,
// the same rescaling by the change of maximum that the online softmax applies
// between key blocks ("Write Triton Attention Kernel", Kernel design rules).
// A thread takes a row and 32 of its columns, and loads a part's columns
// together so their latencies overlap; when the tile has few rows, up to 32
// lanes share a (row, columns) item and split the parts between them.
// Measured on GB300 for a decode step (Z1 Hq32 Hkv8 Nq1 Nkv32768 D128: 8
// tiles of 4 rows, about 19 parts each): one lane per item took 26 us.
constexpr int MERGE_THREADS = 4 * BM;

template <int D, bool CAUSAL, bool BF16>
__global__ void __launch_bounds__(MERGE_THREADS) fa_split_merge_kernel(const FwdParams p, int grid) {
    using S = Sched<CAUSAL, Traits<D>::BN>;
    ptx::grid_dependency_wait();  // the parts are written by the launch before
    const int64_t b = (int64_t)blockIdx.x + 1;
    const int64_t xb = S::range_lo(b, grid, p);
    int64_t head;
    int mb;
    S::tile_of(xb, p, head, mb);
    const int64_t t0 = S::tile_pos(head, mb, p);
    if (xb == t0) return;  // the cut falls between tiles
    // The tile's parts come from CTAs c0 (the one holding its first block)
    // .. c1, so the cuts inside it are c0 + 1 .. c1: each of those blocks
    // merges one slice of the tile's rows.
    const int64_t c0 = S::cta_of(t0, grid, p);
    const int64_t c1 = S::cta_of(t0 + S::tile_nkv(mb, p) - 1, grid, p);
    const int tile_rows = p.Nq - mb * BM < BM ? p.Nq - mb * BM : BM;  // rows the parts stored
    const int slices = (int)(c1 - c0), slice = (int)(b - 1 - c0);
    const int per = (tile_rows + slices - 1) / slices;
    const int row0 = slice * per;
    const int rows = tile_rows - row0 < per ? tile_rows - row0 : per;  // rows of this block
    if (rows <= 0) return;
    auto part = [&](int64_t c) -> const float* {
        return p.scratch + (c == c0 ? 2 * c + 1 : 2 * c) * p.slot_floats;
    };
    // A work item is (row, CH float4 column groups).  With few rows (a
    // decode step stores 4) there are fewer items than threads: then SPL
    // consecutive lanes share an item, each taking every SPL-th part, so
    // the parts' loads overlap instead of following one another, and the
    // lanes combine max, normaliser and O by shuffles.  Every thread runs
    // the same number of rounds, so the shuffles always see whole warps.
    constexpr int W = D / 4;                      // float4 column groups of a row
    constexpr int CH = W < 8 ? W : 8;             // groups per item
    const int items = rows * (W / CH);
    int spl = 1;
    while (spl < 32 && items * spl * 2 <= MERGE_THREADS) spl *= 2;
    const int lane_s = threadIdx.x % spl;
    const int z = (int)(head / p.Hq), hq = (int)(head % p.Hq);
    for (int it0 = 0; it0 < items; it0 += MERGE_THREADS / spl) {
        const int it = it0 + (int)threadIdx.x / spl;
        const bool ok = it < items;
        // consecutive items are consecutive rows, so that a warp's loads of one
        // column group ([group][row] in a part) are contiguous
        const int r = ok ? row0 + it % rows : 0, g0 = ok ? (it / rows) * CH : 0;
        // the parts' log-sum-exps of this row, PB loads at a time so that they overlap
        constexpr int PB = 8;
        float mx = -INFINITY;
        if (ok) {
            for (int64_t c = c0 + lane_s; c <= c1; c += PB * spl) {
                float x[PB];
#pragma unroll
                for (int i = 0; i < PB; ++i)
                    x[i] = c + i * spl <= c1 ? __ldg(part(c + i * spl) + BM * D + r) : -INFINITY;
#pragma unroll
                for (int i = 0; i < PB; ++i) mx = fmaxf(mx, x[i]);
            }
        }
        for (int m = spl / 2; m > 0; m /= 2) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
        float den = 0.f;
        float4 acc[CH];
#pragma unroll
        for (int i = 0; i < CH; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (ok) {
#pragma unroll 2
            for (int64_t c = c0 + lane_s; c <= c1; c += spl) {
                const float* pc = part(c);
                const float w = exp2f(__ldg(pc + BM * D + r) - mx);
                den += w;
                const float4* col = reinterpret_cast<const float4*>(pc) + r;
                float4 v[CH];
#pragma unroll
                for (int i = 0; i < CH; ++i) v[i] = __ldg(col + (g0 + i) * BM);
#pragma unroll
                for (int i = 0; i < CH; ++i) {
                    acc[i].x += w * v[i].x;
                    acc[i].y += w * v[i].y;
                    acc[i].z += w * v[i].z;
                    acc[i].w += w * v[i].w;
                }
            }
        }
        for (int m = spl / 2; m > 0; m /= 2) {
            den += __shfl_xor_sync(0xffffffffu, den, m);
#pragma unroll
            for (int i = 0; i < CH; ++i) {
                acc[i].x += __shfl_xor_sync(0xffffffffu, acc[i].x, m);
                acc[i].y += __shfl_xor_sync(0xffffffffu, acc[i].y, m);
                acc[i].z += __shfl_xor_sync(0xffffffffu, acc[i].z, m);
                acc[i].w += __shfl_xor_sync(0xffffffffu, acc[i].w, m);
            }
        }
        if (!ok || lane_s != 0) continue;
        const int q_row = mb * BM + r;
        const float inv = 1.f / den;
        if (g0 == 0 && p.lse != nullptr) p.lse[head * p.Nq + q_row] = (mx + log2f(den)) * 0.6931471805599453f;
        uint8_t* orow = reinterpret_cast<uint8_t*>(p.o) +
                        2 * ((int64_t)z * p.so_z + (int64_t)hq * p.so_h + (int64_t)q_row * p.so_n);
#pragma unroll
        for (int i = 0; i < CH; ++i) {
            uint2 out;
            out.x = pack2<BF16>(acc[i].x * inv, acc[i].y * inv);
            out.y = pack2<BF16>(acc[i].z * inv, acc[i].w * inv);
            reinterpret_cast<uint2*>(orow)[g0 + i] = out;
        }
    }
}

}  // namespace fa
