// Attention backward for sm_103a: gradients dQ, dK, dV of the fused forward
// from the saved log-sum-exp, with the score and probability blocks rebuilt
// on chip (blog "把 FlashAttention 搬上昇腾：Triton-Ascend CV Pipeline 优化实战",
// section 二: recompute P from the lse, dP, dS, then dQ / dK / dV; "Write
// Triton Attention Kernel", step 8 and Correctness requirements: the backward
// needs lse = m + log l).
//
// Two kernels on one stream: fa_bwd_pre_kernel, then fa_bwd_kernel, which
// runs a dK/dV phase and then a dQ phase in each CTA:
//   pre kernel         per query row: Δ = rowsum(dO ∘ O) and the base-2 lse;
//   dK/dV phase        one unit per (128-key block, kv head): loops over every
//                      query block of every query head of the GQA group (from
//                      the diagonal on when causal), keys as TMEM lanes:
//                          Sᵀ  = K Qᵢᵀ,  Pᵀ = 2^(Sᵀ·scale·log2e − lse2ᵢ)
//                          dPᵀ = V dOᵢᵀ, dSᵀ = Pᵀ ∘ (dPᵀ − Δᵢ)
//                          dV += Pᵀ dOᵢ,  dK += dSᵀ Qᵢ   (Pᵀ, dSᵀ from TMEM)
//                      dK (times scale) and dV stay in TMEM and are stored once;
//   dQ phase           one unit per (128-row query block, query head): loops
//                      over the key blocks it sees, queries as TMEM lanes:
//                          S = Qᵢ Kⱼᵀ, dP = dOᵢ Vⱼᵀ, dS = P ∘ (dP − Δ),
//                          dQ += dS Kⱼ   (dS from TMEM)
//                      dQ (times scale) stays in TMEM and is stored once.
// dQ is summed over key blocks inside one CTA, so no atomics are needed and
// the result is bitwise reproducible; the price is recomputing S and dP in
// the dQ phase (7 tensor-core products per block pair instead of 5).
//
// Warps (both phases): column groups of each 128x128 block (thread = TMEM
// lane; four groups of 32 columns, warps 0-15, at D = 128, else two of 64,
// warps 0-7), then the 4 epilogue warps, the TMA producer and the MMA issuer
// (at D = 128 two idle warps complete the last warpgroup).  Every wait is bounded as in the forward kernel.  Head
// dims 16 to 128 (the dK/dV phase's TMEM holds Sᵀ/Pᵀ, dPᵀ/dSᵀ, dV and dK:
// 256 + 2D columns).
#pragma once

#include "fa_fwd_kernel.cuh"

namespace fa {

// The softmax warps of both phases split the 128 columns of a block into NG
// groups of CW (4 warps each, one per TMEM lane quarter); then 4 epilogue
// warps, the TMA producer and the MMA issuer.  Four groups at D = 128, two
// below (measured on GB300: four groups +4 % at Z1 Hq32 Hkv8 N8192 D128,
// level at N1024; at D = 64 3-4 % slower than two, and still 1-2 % slower
// with the register split below).
template <int D>
struct BwdWarps {
    static constexpr int NG = D == 128 ? 4 : 2;
    static constexpr int CW = 128 / NG;
    static constexpr int CH = CW == 32 ? 16 : 32;  // columns per softmax TMEM load
    static constexpr int SOFTMAX_WARPS = 4 * NG;
    // D = 128: whole warpgroups (the last one: producer, issuer and two idle
    // warps), launched at 80 registers a thread; setmaxnreg then gives the
    // softmax warpgroups 88 and splits the rest between the epilogue and the
    // last warpgroup.
    // The host launches this kernel only after checking that it was built
    // with exactly REG_LAUNCH registers, so the budgets always add up.
    static constexpr bool SPLIT_REGS = D == 128;
    static constexpr int WARPS = SPLIT_REGS ? (SOFTMAX_WARPS + 6 + 3) / 4 * 4 : SOFTMAX_WARPS + 6;
    static constexpr int THREADS = WARPS * 32;
    static constexpr uint32_t REG_LAUNCH = 65536 / THREADS / 8 * 8;
    // Causal (short units, the epilogue's read-out often on the critical
    // path): epilogue 72, producer/issuer 56.  Non-causal: epilogue 56 with
    // the leaner store (bwd_store_rows), producer/issuer 72, whose MMA issue
    // then spills less (measured on GB300: +3.0 % at Z1 Hq32 Hkv8 N8192,
    // +1.2 % at Z4 H16 N1024 non-causal, -1.4 % if used when causal).
    static constexpr uint32_t REG_SOFTMAX = 88;
    static constexpr uint32_t reg_epi(bool causal) { return causal ? 72 : 56; }
    static constexpr uint32_t reg_ctrl(bool causal) { return causal ? 56 : 72; }
    static constexpr bool lean_store(bool causal) { return SPLIT_REGS && !causal; }
    static_assert(!SPLIT_REGS || 128 * (NG * REG_SOFTMAX + reg_epi(true) + reg_ctrl(true)) == THREADS * REG_LAUNCH,
                  "register budgets of the warpgroups");
    static_assert(!SPLIT_REGS || 128 * (NG * REG_SOFTMAX + reg_epi(false) + reg_ctrl(false)) == THREADS * REG_LAUNCH,
                  "register budgets of the warpgroups");
};

// TMEM loads and stores of a width fixed at compile time
template <int N>
__device__ __forceinline__ void tmem_ld_n(uint32_t taddr, uint32_t (&r)[N]) {
    static_assert(N == 16 || N == 32, "16 or 32 columns");
    if constexpr (N == 32) ptx::tmem_ld32(taddr, r);
    else ptx::tmem_ld16(taddr, r);
}
template <int N>
__device__ __forceinline__ void tmem_st_n(uint32_t taddr, const uint32_t (&r)[N]) {
    static_assert(N == 8 || N == 16 || N == 32, "8, 16 or 32 columns");
    if constexpr (N == 32) ptx::tmem_st32(taddr, r);
    else if constexpr (N == 16) ptx::tmem_st16(taddr, r);
    else ptx::tmem_st8(taddr, r);
}

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
    static constexpr int SW = D * 2 >= 128 ? 128 : D * 2;      // bytes per swizzled row chunk of Q, K, V, dO
    static constexpr int SWE = SW / 2;
    static constexpr int NCHUNK = D / SWE;
    static constexpr uint32_t SWIZZLE_CODE = SW == 128 ? 2u : SW == 64 ? 4u : 6u;
    static constexpr int TILE = 128 * D * 2;                  // one 128-row tile of Q, K, V or dO

    // ---- dK / dV phase ----
    // shared memory: K, V of the unit; Q, dO, lse2, Δ of two steps
    static constexpr int KV_OFF_K = 0;
    static constexpr int KV_OFF_V = KV_OFF_K + TILE;
    static constexpr int KV_OFF_Q = KV_OFF_V + TILE;          // [2]
    static constexpr int KV_OFF_DO = KV_OFF_Q + 2 * TILE;     // [2]
    static constexpr int KV_OFF_LSE = KV_OFF_DO + 2 * TILE;   // [2] x 128 floats
    static constexpr int KV_OFF_DELTA = KV_OFF_LSE + 2 * 512; // [2] x 128 floats
    // dK / dV staging for the tensor stores: 32 rows x one swizzle chunk per
    // epilogue warp, aligned to the swizzle pattern's 1024-byte period
    static constexpr int KV_OFF_OST = (KV_OFF_DELTA + 2 * 512 + 1023) / 1024 * 1024;
    static constexpr int KV_OFF_BAR = KV_OFF_OST + 128 * SW;
    static constexpr int KB_KV_FULL = 0;      // K, V of a unit landed (TMA)
    static constexpr int KB_KV_EMPTY = 1;     // the unit's last Sᵀ and dPᵀ are done (commit)
    static constexpr int KB_QD_FULL = 2;      // [2] Q, dO, lse2, Δ of a step landed (TMA)
    static constexpr int KB_QD_EMPTY = 4;     // [2] that step's products are done (commit)
    static constexpr int KB_S_FULL = 6;       // Sᵀ in TMEM (commit)
    static constexpr int KB_DP_FULL = 7;      // dPᵀ in TMEM (commit)
    static constexpr int KB_P_FULL = 8;       // Pᵀ written over Sᵀ (every softmax thread)
    static constexpr int KB_DS_FULL = 9;      // dSᵀ written over dPᵀ (every softmax thread)
    static constexpr int KB_ACC_FULL = 10;    // dK, dV of a unit complete (commit)
    static constexpr int KB_ACC_FREE = 11;    // dK, dV read out of TMEM (128)
    static constexpr int KB_DRAIN = 12;
    static constexpr int KV_NUM_BARS = 13;
    static constexpr int KV_OFF_MISC = KV_OFF_BAR + KV_NUM_BARS * 8;
    static constexpr int KV_SMEM_USED = KV_OFF_MISC + 16;
    static constexpr int KV_SMEM_BYTES = KV_SMEM_USED + 1024;  // + slack to align the base to 1024 bytes
    static_assert(KV_SMEM_BYTES <= 227 * 1024, "shared memory budget");
    static constexpr uint32_t TM_S = 0;       // Sᵀ (fp32); Pᵀ packed over columns 0-31 and 64-95
    static constexpr uint32_t TM_DP = 128;    // dPᵀ (fp32); dSᵀ packed over columns 128-159 and 192-223
    static constexpr uint32_t TM_DV = 256;
    static constexpr uint32_t TM_DK = 256 + D;

    // ---- dQ phase ----
    // shared memory: Q, dO of the unit; K, V of two key blocks
    static constexpr int Q_OFF_Q = 0;
    static constexpr int Q_OFF_DO = Q_OFF_Q + TILE;
    static constexpr int Q_OFF_K = Q_OFF_DO + TILE;           // [2]
    static constexpr int Q_OFF_V = Q_OFF_K + 2 * TILE;        // [2]
    static constexpr int Q_OFF_OST = Q_OFF_V + 2 * TILE;       // dQ staging (as KV_OFF_OST)
    static constexpr int Q_OFF_BAR = Q_OFF_OST + 128 * SW;
    static constexpr int QB_QD_FULL = 0;      // Q, dO of a unit landed (TMA)
    static constexpr int QB_QD_EMPTY = 1;     // the unit's last S and dP are done (commit)
    static constexpr int QB_KV_FULL = 2;      // [2] K, V of a key block landed (TMA)
    static constexpr int QB_KV_EMPTY = 4;     // [2] that block's products are done (commit)
    static constexpr int QB_S_FULL = 6;       // [2] S in its TMEM slot (commit)
    static constexpr int QB_DP_FULL = 8;      // dP in TMEM (commit)
    static constexpr int QB_DS_FULL = 9;      // [2] dS written over S in its slot (every softmax thread)
    static constexpr int QB_DQ_FULL = 11;     // dQ of a unit complete (commit)
    static constexpr int QB_DQ_FREE = 12;     // dQ read out of TMEM (128)
    static constexpr int QB_DRAIN = 13;
    static constexpr int Q_NUM_BARS = 14;
    static constexpr int Q_OFF_MISC = Q_OFF_BAR + Q_NUM_BARS * 8;
    static constexpr int Q_SMEM_USED = Q_OFF_MISC + 16;
    static constexpr int Q_SMEM_BYTES = Q_SMEM_USED + 1024;
    static_assert(Q_SMEM_BYTES <= 227 * 1024, "shared memory budget");
    // ---- the fused kernel: dK/dV phase, then dQ phase, in the same shared
    // memory; the TMEM address and the abort flag sit past both layouts ----
    static constexpr int FUSED_OFF_MISC = (KV_SMEM_USED > Q_SMEM_USED ? KV_SMEM_USED : Q_SMEM_USED) + 15 & ~15;
    static constexpr int FUSED_SMEM_USED = FUSED_OFF_MISC + 16;
    static constexpr int FUSED_SMEM_BYTES = FUSED_SMEM_USED + 1024;
    static_assert(FUSED_SMEM_BYTES <= 227 * 1024, "shared memory budget");
    static constexpr uint32_t TM_QS = 0;      // [2] S (fp32); dS packed over columns s*128 + 0-31 and 64-95
    static constexpr uint32_t TM_QDP = 256;   // dP (fp32)
    static constexpr uint32_t TM_DQ = 384;

    static constexpr uint32_t TMEM_COLS = 512;
    static_assert(256 + 2 * D <= 512 && 384 + D <= 512, "tensor memory budget");

    static __device__ __forceinline__ uint32_t kv_bar_count(int i) {
        if (i == KB_P_FULL || i == KB_DS_FULL) return 32 * BwdWarps<D_>::SOFTMAX_WARPS;
        if (i == KB_ACC_FREE) return 128;
        return 1;
    }
    static __device__ __forceinline__ uint32_t q_bar_count(int i) {
        if (i == QB_DS_FULL || i == QB_DS_FULL + 1) return 32 * BwdWarps<D_>::SOFTMAX_WARPS;
        if (i == QB_DQ_FREE) return 128;
        return 1;
    }
};

// K-major operand of 128 rows in swizzled chunks of swe elements: descriptor
// start offset (16-byte units) of the 16-element K step kk
__host__ __device__ constexpr uint32_t kmaj_off(int kk, int swe, int sw) {
    return (uint32_t)((((kk * 16) / swe) * (128 * sw) + ((kk * 16) % swe) * 2) >> 4);
}

// Packed 16-bit columns of a 128-wide block written by column groups of CW
// over the first halves of their own fp32 columns: K step kk (16 elements)
template <int CW>
__device__ __forceinline__ uint32_t packed_col(int kk) {
    return (uint32_t)((16 * kk / CW) * CW + (16 * kk % CW) / 2);
}

// ---------------------------------------------------------------- schedules --
// CTA c takes one unit per round of `grid` units.  Causal units are ordered
// heaviest first; the rounds alternate direction (unit c of round 0, unit
// grid - 1 - c of round 1, ...), so a CTA that drew a heavier unit in one
// round draws a lighter one in the next.
template <bool CAUSAL>
__device__ __forceinline__ int unit_at(int pos) {
    if (!CAUSAL) return pos;
    const int grid = (int)gridDim.x, round = pos / grid;
    return (round & 1) ? 2 * round * grid + grid - 1 - pos : pos;
}

// dK/dV unit u: key block j (ascending: with a causal mask the first key
// blocks have the most query blocks) of kv head (z, hk).  The kv heads go in
// groups of p.kv_head_group, sized on the host so that the query rows a
// group reads (Q, dO) fit in a third of L2; within a group key blocks are
// outermost and heads innermost.  A unit's steps run over the group's query
// heads and, per head, the query blocks from i0 on.
// Variant kernels: VAR 0 plain; 1 window; 2 window and ALiBi; 3 packed
// sequences with a window and ALiBi; 4 packed sequences with a window.
__host__ __device__ constexpr bool bwd_alibi(int VAR) { return VAR == 2 || VAR == 3; }
__host__ __device__ constexpr bool bwd_varlen(int VAR) { return VAR >= 3; }

// zc, qrow0, krow0: the batch coordinate and first query / key row of the
// unit's sequence in the tensor maps; nq, nk: its query and key counts (the
// whole tensors but for packed variable-length batches).
struct BwdUnit {
    int z, hk, j, i0, per_head, nsteps;
    int zc, qrow0, krow0, nq, nk;
};

// Sequence z's rows and counts (packed variants with a sequence table), else
// the dense batch z's.  Offsets are clamped to the packed extents.
template <int VAR, typename U>
__device__ __forceinline__ void unit_sequence(U& w, const BwdParams& p) {
    w.zc = w.z;
    w.qrow0 = 0;
    w.krow0 = 0;
    w.nq = p.Nq;
    w.nk = p.Nkv;
    if constexpr (bwd_varlen(VAR)) {
        if (p.cu_q != nullptr) {
            auto clampi = [](int x, int hi) { return x < 0 ? 0 : (x > hi ? hi : x); };
            const int q0 = clampi(__ldg(p.cu_q + w.z), p.Nq), q1 = clampi(__ldg(p.cu_q + w.z + 1), p.Nq);
            const int k0 = clampi(__ldg(p.cu_k + w.z), p.Nkv), k1 = clampi(__ldg(p.cu_k + w.z + 1), p.Nkv);
            w.zc = 0;
            w.qrow0 = q0;
            w.krow0 = k0;
            w.nq = q1 > q0 ? q1 - q0 : 0;
            w.nk = k1 > k0 ? k1 - k0 : 0;
        }
    }
}

// Variant kernels (window, ALiBi, packed sequences) visit only the query blocks holding a row that keeps a
// key of block j: rows j·128 − win_right .. j·128 + 127 + win_left (of the
// unit's sequence).
template <bool CAUSAL, int VAR = 0>
__device__ __forceinline__ BwdUnit bwd_unit(int u, const BwdParams& p) {
    BwdUnit w;
    const int zh = p.Z * p.Hkv, G = p.kv_head_group;
    const int g0 = u / (G * p.Tk) * G;           // first head of u's group
    const int gc = zh - g0 < G ? zh - g0 : G;    // heads in the group
    const int x = u - g0 * p.Tk;                 // u's place in the group
    w.j = x / gc;
    const int zhk = g0 + x % gc;
    w.z = zhk / p.Hkv;
    w.hk = zhk % p.Hkv;
    unit_sequence<VAR>(w, p);
    // causal (top-left): query row r sees keys <= r, so query blocks before
    // the key block's own index see none of its keys
    w.i0 = CAUSAL ? w.j : 0;
    int i_end = p.Tq;
    if constexpr (bwd_varlen(VAR)) {
        // the sequence's query blocks; a key block past its keys has none
        i_end = (w.nq + 127) / 128 < p.Tq ? (w.nq + 127) / 128 : p.Tq;
        if (w.j * 128 >= w.nk) i_end = 0;
    }
    if constexpr (VAR != 0) {
        if (p.win_right >= 0) {
            const int lo_row = w.j * 128 - p.win_right;
            if (lo_row > 0 && lo_row / 128 > w.i0) w.i0 = lo_row / 128;
        }
        if (p.win_left >= 0) {
            const int64_t hi_block = ((int64_t)w.j * 128 + 127 + p.win_left) / 128 + 1;
            if (hi_block < i_end) i_end = (int)hi_block;
        }
    }
    w.per_head = i_end > w.i0 ? i_end - w.i0 : 0;
    w.nsteps = w.per_head * p.group;
    return w;
}

__device__ __forceinline__ void bwd_step(const BwdUnit& w, int s, const BwdParams& p, int& hq, int& i) {
    hq = w.hk * p.group + s / w.per_head;
    i = w.i0 + s % w.per_head;
}

// dQ unit u: query block i of head (z, hq).  Non-causal: head-major, so the
// CTAs running together share a head's K/V.  Causal: heads in groups of
// p.q_head_group (the group's K/V within a third of L2), and within a group
// the last query block (most key blocks) first, heads innermost.  It sees
// key blocks j0 .. j0 + nkv - 1 (j0 = 0 but in the variant kernels, whose
// window bounds the blocks: keys i·128 − win_left .. i·128 + 127 +
// win_right; a block whose rows keep no key at all still takes one key
// block, every pair of it masked, and ends with dQ = 0).
struct DqUnit {
    int z, hq, hk, i, j0, nkv;
    int zc, qrow0, krow0, nq, nk;
    bool skip;  // packed sequences: a query block past the sequence's rows (no work, nothing stored)
};

template <bool CAUSAL, int VAR = 0>
__device__ __forceinline__ DqUnit dq_unit(int u, const BwdParams& p) {
    DqUnit w;
    const int heads = p.Z * p.Hq;
    int head;
    if (CAUSAL) {
        const int G = p.q_head_group;
        const int g0 = u / (G * p.Tq) * G;
        const int gc = heads - g0 < G ? heads - g0 : G;
        const int x = u - g0 * p.Tq;
        w.i = p.Tq - 1 - x / gc;
        head = g0 + x % gc;
    } else {
        head = u / p.Tq;
        w.i = u % p.Tq;
    }
    w.z = head / p.Hq;
    w.hq = head % p.Hq;
    w.hk = w.hq / p.group;
    unit_sequence<VAR>(w, p);
    w.skip = bwd_varlen(VAR) && w.i * 128 >= w.nq;
    int tk = p.Tk;
    if constexpr (bwd_varlen(VAR)) {
        // the sequence's key blocks (a sequence without keys: one, masked)
        tk = (w.nk + 127) / 128 < p.Tk ? (w.nk + 127) / 128 : p.Tk;
        tk = tk > 0 ? tk : 1;
    }
    w.j0 = 0;
    w.nkv = CAUSAL ? (w.i + 1 < tk ? w.i + 1 : tk) : tk;
    if constexpr (VAR != 0) {
        int jlo = 0, jhi = w.nkv;
        if (p.win_left >= 0) {
            const int lo_key = w.i * 128 - p.win_left;
            jlo = lo_key > 0 ? lo_key / 128 : 0;
        }
        if (p.win_right >= 0) {
            const int64_t hi_block = ((int64_t)w.i * 128 + 127 + p.win_right) / 128 + 1;
            if (hi_block < jhi) jhi = (int)hi_block;
        }
        if (jlo >= jhi) {
            jlo = jlo < tk - 1 ? jlo : tk - 1;
            jhi = jlo + 1;
        }
        w.j0 = jlo;
        w.nkv = jhi - jlo;
    }
    return w;
}

// Variant kernels: whether query q drops key k, for d = q − k (the top-left
// causal rule and the window sides of fa_fwd_ex; a key past the keys is
// dropped too: with a window a row may keep none of the real keys, and its
// lse is then −inf), and whether a whole 128 × 128 block of differences
// d_min .. d_max with keys below k_end is kept.
template <bool CAUSAL>
__device__ __forceinline__ bool var_dropped(int d, int k, int nk, const BwdParams& p) {
    return k >= nk || (CAUSAL && d < 0) || (p.win_left >= 0 && d > p.win_left) ||
           (p.win_right >= 0 && -d > p.win_right);
}
template <bool CAUSAL>
__device__ __forceinline__ bool var_block_kept(int d_min, int d_max, int k_end, int nk, const BwdParams& p) {
    return k_end <= nk && (!CAUSAL || d_min >= 0) && (p.win_left < 0 || d_max <= p.win_left) &&
           (p.win_right < 0 || -d_min <= p.win_right);
}

// Debug builds (FA_DEBUG_CHECKS=1): every role checks each unit it decodes
// against the launch's sizes before touching memory for it, as the forward's
// roles do; a unit outside them records FA_ERR_DEVICE_CHECK with the role's
// site and raises the CTA's abort flag, so the kernel ends through the same
// path as a timed-out wait.  Other builds compile the checks away.
__device__ __forceinline__ bool bwd_check_failed(const Ctl& c, uint32_t site) {
    *c.abort_flag = 1;
    atomicCAS(c.status, 0u, STATUS_DEVICE_CHECK | (site << 8) | ((blockIdx.x & 0xFFFFu) << 16));
    return false;
}
__device__ __forceinline__ bool unit_checked(const BwdUnit& w, const BwdParams& p, const Ctl& c, uint32_t site) {
    if constexpr (!FA_DEBUG_CHECKS) {
        return true;
    } else {
        // the unit's query blocks are i0 .. Tq - 1 of each query head of the group
        const bool ok = w.z >= 0 && w.z < p.Z && w.hk >= 0 && w.hk < p.Hkv && w.j >= 0 && w.j < p.Tk &&
                        w.i0 >= 0 && w.per_head >= 0 && (w.per_head == 0 || w.i0 + w.per_head <= p.Tq) &&
                        w.nsteps == w.per_head * p.group;
        return ok || bwd_check_failed(c, site);
    }
}
__device__ __forceinline__ bool unit_checked(const DqUnit& w, const BwdParams& p, const Ctl& c, uint32_t site) {
    if constexpr (!FA_DEBUG_CHECKS) {
        return true;
    } else {
        const bool ok = w.z >= 0 && w.z < p.Z && w.hq >= 0 && w.hq < p.Hq && w.hk == w.hq / p.group &&
                        w.hk < p.Hkv && w.i >= 0 && w.i < p.Tq && w.j0 >= 0 && w.nkv >= 1 && w.j0 + w.nkv <= p.Tk;
        return ok || bwd_check_failed(c, site);
    }
}

// ================================================================ dK / dV ===

template <int D, bool CAUSAL, int VAR>
__device__ void kv_producer(const CUtensorMap* tmK, const CUtensorMap* tmV, const CUtensorMap* tmQ,
                            const CUtensorMap* tmDO, const BwdParams& p, uint32_t sbase, uint32_t bar0,
                            const Ctl& ctl) {
    using T = BwdTraits<D>;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    const uint64_t pol_kv = ptx::policy_evict_first();  // read once per unit
    const uint64_t pol_q = ptx::policy_evict_last();    // read by every key block
    uint32_t uc = 0, t = 0;
    bool ok = true;
    bool withheld = false;
    for (int pos = blockIdx.x; ok && unit_at<CAUSAL>(pos) < p.nunits; pos += gridDim.x) {
        const BwdUnit w = bwd_unit<CAUSAL, VAR>(unit_at<CAUSAL>(pos), p);
        if (!unit_checked(w, p, ctl, SITE_CHECK_BWD_LOAD)) { ok = false; break; }
        if (w.nsteps == 0) continue;
        if (uc > 0 && !wait_phase(bar(T::KB_KV_EMPTY), (uc - 1) & 1u, ctl, SITE_B_KV_EMPTY)) { ok = false; break; }
        if (p.inject_stall && blockIdx.x == 0 && uc == 0) {
            withheld = true;  // never issued: the issuer's wait for K, V must time out
        } else {
            ptx::mbar_arrive_expect_tx(bar(T::KB_KV_FULL), 2 * T::TILE);
            for (int c = 0; c < T::NCHUNK; ++c) {
                ptx::tma_load_4d(sbase + T::KV_OFF_K + c * (128 * T::SW), tmK, bar(T::KB_KV_FULL), c * T::SWE,
                                 w.krow0 + w.j * 128, w.hk, w.zc, pol_kv);
                ptx::tma_load_4d(sbase + T::KV_OFF_V + c * (128 * T::SW), tmV, bar(T::KB_KV_FULL), c * T::SWE,
                                 w.krow0 + w.j * 128, w.hk, w.zc, pol_kv);
            }
        }
        ++uc;
        for (int s = 0; s < w.nsteps; ++s, ++t) {
            const uint32_t st = t & 1u;
            if (t >= 2 && !wait_phase(bar(T::KB_QD_EMPTY + st), ((t - 2) >> 1) & 1u, ctl, SITE_B_QD_EMPTY)) {
                ok = false;
                break;
            }
            int hq, i;
            bwd_step(w, s, p, hq, i);
            const uint32_t full = bar(T::KB_QD_FULL + st);
            ptx::mbar_arrive_expect_tx(full, 2 * T::TILE + 1024);
            for (int c = 0; c < T::NCHUNK; ++c) {
                ptx::tma_load_4d(sbase + T::KV_OFF_Q + st * T::TILE + c * (128 * T::SW), tmQ, full, c * T::SWE,
                                 w.qrow0 + i * 128, hq, w.zc, pol_q);
                ptx::tma_load_4d(sbase + T::KV_OFF_DO + st * T::TILE + c * (128 * T::SW), tmDO, full, c * T::SWE,
                                 w.qrow0 + i * 128, hq, w.zc, pol_q);
            }
            const int64_t row0 = ((int64_t)w.z * p.Hq + hq) * p.Tq * 128 + (int64_t)i * 128;
            ptx::bulk_load(sbase + T::KV_OFF_LSE + st * 512, p.lse2 + row0, 512, full);
            ptx::bulk_load(sbase + T::KV_OFF_DELTA + st * 512, p.delta + row0, 512, full);
        }
    }
    if (!ok) {
        // let the copies in flight land before shared memory goes away (the
        // withheld copy never completes; its wait simply runs out)
        if (uc > 0) drain_phase(bar(T::KB_KV_FULL), (uc - 1) & 1u, withheld && uc == 1 ? ctl.limit_ns / 64 : ctl.limit_ns);
        for (uint32_t x = t > 2u ? t - 2u : 0u; x < t; ++x)
            drain_phase(bar(T::KB_QD_FULL + (x & 1u)), (x >> 1) & 1u, ctl.limit_ns);
    }
}

// Per step t: dPᵀ_t, dV_t, then Sᵀ_{t+1} (its columns were last read by dV_t,
// issued before it), then dK_t -- so the softmax warps build Pᵀ_{t+1} while
// the tensor core runs dK_t and dPᵀ_{t+1}.  Products issued by one thread
// run in order, so a product never overwrites TMEM an earlier one still reads.
template <int D, bool CAUSAL, bool BF16, int VAR>
__device__ void kv_issuer(const BwdParams& p, uint32_t sbase, uint32_t bar0, uint32_t tmem, const Ctl& ctl) {
    using T = BwdTraits<D>;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    constexpr uint32_t ID_SQ = ptx::idesc_f16(128, 128, BF16, false, false);  // Sᵀ = K Qᵀ, dPᵀ = V dOᵀ
    constexpr uint32_t ID_ND = ptx::idesc_f16(128, D, BF16, false, true);     // dV, dK: B MN-major (N = D)
    constexpr uint32_t HI = ptx::smem_desc_hi(8 * T::SW, T::SWIZZLE_CODE);
    const uint32_t k_lo = ptx::smem_desc_lo(sbase + T::KV_OFF_K, 16);
    const uint32_t v_lo = ptx::smem_desc_lo(sbase + T::KV_OFF_V, 16);
    auto issue_s = [&](uint32_t t) -> bool {
        const uint32_t st = t & 1u;
        if (!wait_phase(bar(T::KB_QD_FULL + st), (t >> 1) & 1u, ctl, SITE_B_QD_FULL)) return false;
        ptx::tc_fence_after();
        const uint32_t q_lo = ptx::smem_desc_lo(sbase + T::KV_OFF_Q + st * T::TILE, 16);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
            ptx::mma_ss(tmem + T::TM_S, ptx::desc64(k_lo + kmaj_off(kk, T::SWE, T::SW), HI),
                        ptx::desc64(q_lo + kmaj_off(kk, T::SWE, T::SW), HI), ID_SQ, kk > 0 ? 1u : 0u);
        ptx::tc_commit(bar(T::KB_S_FULL));
        return true;
    };
    uint32_t uc = 0, t = 0;
    bool ok = true;
    for (int pos = blockIdx.x; ok && unit_at<CAUSAL>(pos) < p.nunits; pos += gridDim.x) {
        const BwdUnit w = bwd_unit<CAUSAL, VAR>(unit_at<CAUSAL>(pos), p);
        if (!unit_checked(w, p, ctl, SITE_CHECK_BWD_MMA)) { ok = false; break; }
        if (w.nsteps == 0) continue;
        if (!wait_phase(bar(T::KB_KV_FULL), uc & 1u, ctl, SITE_B_KV_FULL)) { ok = false; break; }
        if (!issue_s(t)) { ok = false; break; }
        for (int s = 0; s < w.nsteps; ++s, ++t) {
            const uint32_t st = t & 1u;
            const uint32_t do_lo = ptx::smem_desc_lo(sbase + T::KV_OFF_DO + st * T::TILE, 16);
            const uint32_t domn_lo = ptx::smem_desc_lo(sbase + T::KV_OFF_DO + st * T::TILE, 128 * T::SW);
            const uint32_t qmn_lo = ptx::smem_desc_lo(sbase + T::KV_OFF_Q + st * T::TILE, 128 * T::SW);
            // dPᵀ = V dOᵢᵀ
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
                ptx::mma_ss(tmem + T::TM_DP, ptx::desc64(v_lo + kmaj_off(kk, T::SWE, T::SW), HI),
                            ptx::desc64(do_lo + kmaj_off(kk, T::SWE, T::SW), HI), ID_SQ, kk > 0 ? 1u : 0u);
            ptx::tc_commit(bar(T::KB_DP_FULL));
            // the unit's last Sᵀ and dPᵀ were its last reads of K and V: the
            // next unit's K, V may land while its last dV, dK run
            if (s + 1 == w.nsteps) ptx::tc_commit(bar(T::KB_KV_EMPTY));
            // dV += Pᵀ dOᵢ; a unit's first step waits for the last unit's dK, dV to be read
            if (!wait_phase(bar(T::KB_P_FULL), t & 1u, ctl, SITE_B_P_FULL)) { ok = false; break; }
            if (s == 0 && uc > 0 && !wait_phase(bar(T::KB_ACC_FREE), (uc - 1) & 1u, ctl, SITE_B_ACC_FREE)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 128 / 16; ++kk)
                ptx::mma_ts(tmem + T::TM_DV, tmem + T::TM_S + packed_col<BwdWarps<D>::CW>(kk),
                            ptx::desc64(domn_lo + ((kk * 16 * T::SW) >> 4), HI), ID_ND, (s > 0 || kk > 0) ? 1u : 0u);
            if (s + 1 < w.nsteps && !issue_s(t + 1)) { ok = false; break; }
            // dK += dSᵀ Qᵢ
            if (!wait_phase(bar(T::KB_DS_FULL), t & 1u, ctl, SITE_B_DS_FULL)) { ok = false; break; }
            ptx::tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 128 / 16; ++kk)
                ptx::mma_ts(tmem + T::TM_DK, tmem + T::TM_DP + packed_col<BwdWarps<D>::CW>(kk),
                            ptx::desc64(qmn_lo + ((kk * 16 * T::SW) >> 4), HI), ID_ND, (s > 0 || kk > 0) ? 1u : 0u);
            ptx::tc_commit(bar(T::KB_QD_EMPTY + st));  // Qᵢ, dOᵢ slot free
        }
        if (!ok) break;
        ptx::tc_commit(bar(T::KB_ACC_FULL));  // dK, dV of the unit complete
        ++uc;
    }
    // every MMA of this phase completes before the dQ phase reuses shared memory
    ptx::tc_commit(bar(T::KB_DRAIN));
    drain_phase(bar(T::KB_DRAIN), 0u, ctl.limit_ns);
}

// Thread = key (TMEM lane); column group h takes queries h*CW .. h*CW + CW - 1
// and writes its Pᵀ and dSᵀ (input type, two per column) over its own fp32
// columns, so no group overwrites values another has not read.
template <int D, bool CAUSAL, bool BF16, int VAR>
__device__ void kv_softmax(const BwdParams& p, uint32_t sbase, uint32_t bar0, uint32_t tmem, int h, const Ctl& ctl) {
    using T = BwdTraits<D>;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    const int quad = (threadIdx.x / 32) % 4;
    const int row = quad * 32 + threadIdx.x % 32;  // key within the block
    const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
    const float c = p.scale_log2;
    constexpr int CW = BwdWarps<D>::CW, CH = BwdWarps<D>::CH;
    uint32_t t = 0;
    for (int pos = blockIdx.x; unit_at<CAUSAL>(pos) < p.nunits; pos += gridDim.x) {
        const BwdUnit w = bwd_unit<CAUSAL, VAR>(unit_at<CAUSAL>(pos), p);
        if (!unit_checked(w, p, ctl, SITE_CHECK_BWD_SOFTMAX)) return;
        for (int s = 0; s < w.nsteps; ++s, ++t) {
            const uint32_t st = t & 1u;
            int hq, i;
            bwd_step(w, s, p, hq, i);
            // lse2 and Δ of the step's queries arrive with Qᵢ (TMA)
            if (!warp_wait_phase(bar(T::KB_QD_FULL + st), (t >> 1) & 1u, ctl, SITE_B_QD_FULL)) return;
            const uint32_t lse_a = sbase + T::KV_OFF_LSE + st * 512 + h * CW * 4;
            const uint32_t del_a = sbase + T::KV_OFF_DELTA + st * 512 + h * CW * 4;
            if (!warp_wait_phase(bar(T::KB_S_FULL), t & 1u, ctl, SITE_B_S_FULL)) return;
            ptx::tc_fence_after();
            // causal: only the diagonal block has keys after queries (key > query -> 0)
            const bool diag = CAUSAL && i == w.j;
            // variants: d = query − key = dbase + col; the window and causal
            // rule drop pairs unless the whole block is kept; ALiBi adds
            // slope2·|d| (log2 units)
            const int dbase = (i - w.j) * 128 - row;
            const bool full =
                VAR == 0 || var_block_kept<CAUSAL>((i - w.j) * 128 - 127, (i - w.j) * 128 + 127, w.j * 128 + 128, w.nk, p);
            const int key = w.j * 128 + row;
            const float slope2 =
                bwd_alibi(VAR) ? -__ldg(p.alibi + hq) * 1.4426950408889634f : 0.f;
            const float dbf = (float)(dbase + h * CW);  // d of this group's first column (exact: |d| < 2^24)
            uint32_t pk[CW / 2];  // Pᵀ in the input type: the dV operand, and what dS uses
#pragma unroll
            for (int cc = 0; cc < CW / CH; ++cc) {
                uint32_t r[CH];
                tmem_ld_n<CH>(tmem + lane_addr + T::TM_S + h * CW + CH * cc, r);
#pragma unroll
                for (int x = 0; x < CH / 2; ++x) {
                    const int col = h * CW + CH * cc + 2 * x;
                    float l0, l1;
                    asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(l0), "=f"(l1) : "r"(lse_a + 4u * (CH * cc + 2 * x)));
                    float e0 = fmaf(__uint_as_float(r[2 * x]), c, -l0);
                    float e1 = fmaf(__uint_as_float(r[2 * x + 1]), c, -l1);
                    if constexpr (VAR == 0) {
                        if (diag && row > col) e0 = -INFINITY;
                        if (diag && row > col + 1) e1 = -INFINITY;
                    } else {
                        const int d0 = dbase + col;
                        if constexpr (bwd_alibi(VAR)) {
                            const float df = dbf + (float)(CH * cc + 2 * x);
                            e0 = fmaf(slope2, fabsf(df), e0);
                            e1 = fmaf(slope2, fabsf(df + 1.f), e1);
                        }
                        if (!full) {
                            if (var_dropped<CAUSAL>(d0, key, w.nk, p)) e0 = -INFINITY;
                            if (var_dropped<CAUSAL>(d0 + 1, key, w.nk, p)) e1 = -INFINITY;
                        }
                    }
                    pk[(CH / 2) * cc + x] = pack2<BF16>(ptx::ex2(e0), ptx::ex2(e1));
                }
            }
            tmem_st_n<CW / 2>(tmem + lane_addr + T::TM_S + h * CW, pk);
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(T::KB_P_FULL));

            if (!warp_wait_phase(bar(T::KB_DP_FULL), t & 1u, ctl, SITE_B_DP_FULL)) return;
            ptx::tc_fence_after();
#pragma unroll
            for (int cc = 0; cc < CW / CH; ++cc) {
                uint32_t r[CH];
                tmem_ld_n<CH>(tmem + lane_addr + T::TM_DP + h * CW + CH * cc, r);
                uint32_t ds[CH / 2];
#pragma unroll
                for (int x = 0; x < CH / 2; ++x) {
                    float d0, d1;
                    asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(d0), "=f"(d1) : "r"(del_a + 4u * (CH * cc + 2 * x)));
                    const float2 pp = unpack2<BF16>(pk[(CH / 2) * cc + x]);
                    ds[x] = pack2<BF16>(pp.x * (__uint_as_float(r[2 * x]) - d0), pp.y * (__uint_as_float(r[2 * x + 1]) - d1));
                }
                // packed columns h*CW + (CH/2)cc .. : fp32 columns this thread has already read
                tmem_st_n<CH / 2>(tmem + lane_addr + T::TM_DP + h * CW + (CH / 2) * cc, ds);
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(T::KB_DS_FULL));
        }
    }
}

// The forward's tma_store_rows (one warp's 32 rows of a TMEM block out
// through its staging area and TMA tensor stores) with fewer registers: each
// swizzle chunk is converted and staged 32 columns at a time instead of
// whole, so the epilogue warpgroup fits in its setmaxnreg budget.
template <int D, int SW, bool BF16, typename AfterRead>
__device__ __forceinline__ void bwd_store_rows(uint32_t taddr, float mul, uint32_t stage, const CUtensorMap* map,
                                               int row0, int h, int z, bool store, AfterRead&& after_read) {
    constexpr int SWE = SW / 2;              // elements per chunk row
    constexpr int CH = SWE >= 32 ? 32 : 16;  // columns per TMEM load
    constexpr int UPC = CH / 8;              // 16-byte units a piece fills
    const int lane = threadIdx.x % 32;
    const uint32_t swz = ((uint32_t)lane * SW >> 7) & (SW / 16 - 1);
#pragma unroll 1
    for (int k = 0; k < D / SWE; ++k) {
#pragma unroll
        for (int i = 0; i < SWE / CH; ++i) {
            uint32_t r[CH];
            if constexpr (CH == 32) ptx::tmem_ld32(taddr + k * SWE + i * CH, r);
            else ptx::tmem_ld16(taddr + k * SWE + i * CH, r);
            uint32_t pk[CH / 2];
#pragma unroll
            for (int x = 0; x < CH / 2; ++x)
                pk[x] = pack2<BF16>(__uint_as_float(r[2 * x]) * mul, __uint_as_float(r[2 * x + 1]) * mul);
            if (k == D / SWE - 1 && i == SWE / CH - 1) after_read();
            if (i == 0) {
                // the previous box must have been read out of the staging
                // area (waited for after this chunk's first TMEM load)
                if (lane == 0) ptx::bulk_wait_read_all();
                __syncwarp();
            }
#pragma unroll
            for (int c = 0; c < UPC; ++c)
                ptx::st_shared_v4(stage + (uint32_t)lane * SW + ((((uint32_t)(i * UPC + c)) ^ swz) << 4), pk[4 * c],
                                  pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        }
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && store) {
            ptx::tma_store_4d(map, stage, k * SWE, row0, h, z);
            ptx::bulk_commit();
        }
    }
}

// The store the epilogue warps use (bwd_store_rows where their register
// budget is the smaller one, else the forward's tma_store_rows)
template <int D, int SW, bool BF16, bool LEAN, typename AfterRead>
__device__ __forceinline__ void epi_store_rows(uint32_t taddr, float mul, uint32_t stage, const CUtensorMap* map,
                                               int row0, int h, int z, bool store, AfterRead&& after_read) {
    if constexpr (LEAN) bwd_store_rows<D, SW, BF16>(taddr, mul, stage, map, row0, h, z, store, after_read);
    else tma_store_rows<D, SW, BF16>(taddr, mul, stage, map, row0, h, z, store, after_read);
}

// One row per thread, straight to global memory, for a 32-row box that runs
// past the end of a packed sequence: the next sequence's rows follow, so the
// tensor store's clipping at the tensor's end does not guard them.  Every lane
// takes part in the TMEM loads; only lanes with `store` write.  `after_read`
// runs once the last TMEM load is complete.
template <int D, bool BF16, typename AfterRead>
__device__ __forceinline__ void direct_store_row(uint32_t taddr, float mul, uint8_t* dst_row, bool store,
                                                 AfterRead&& after_read) {
    constexpr int CH = D >= 32 ? 32 : 16;  // columns per TMEM load
#pragma unroll 1
    for (int k = 0; k < D / CH; ++k) {
        uint32_t r[CH];
        if constexpr (CH == 32) ptx::tmem_ld32(taddr + k * CH, r);
        else ptx::tmem_ld16(taddr + k * CH, r);
        uint32_t pk[CH / 2];
#pragma unroll
        for (int x = 0; x < CH / 2; ++x)
            pk[x] = pack2<BF16>(__uint_as_float(r[2 * x]) * mul, __uint_as_float(r[2 * x + 1]) * mul);
        if (k == D / CH - 1) after_read();
        if (store) {
            uint4* dst = reinterpret_cast<uint4*>(dst_row + 2 * k * CH);
#pragma unroll
            for (int x = 0; x < CH / 8; ++x) dst[x] = make_uint4(pk[4 * x], pk[4 * x + 1], pk[4 * x + 2], pk[4 * x + 3]);
        }
    }
}

// Thread = TMEM lane = key: per unit, dK (times scale) and dV are read out,
// released and stored in the input type; a unit no query sees gets zeros.
template <int D, bool CAUSAL, bool BF16, int VAR>
__device__ void kv_epilogue(const CUtensorMap* tmDK, const CUtensorMap* tmDV, const BwdParams& p, uint32_t sbase,
                            uint32_t bar0, uint32_t tmem, const Ctl& ctl) {
    using T = BwdTraits<D>;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    const int quad = (threadIdx.x / 32) % 4;
    const int row = quad * 32 + threadIdx.x % 32;
    const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
    const uint32_t stage = sbase + T::KV_OFF_OST + (uint32_t)quad * 32u * T::SW;  // this warp's staging rows
    // lane 0's stores must have read shared memory before the CTA exits
    auto drain = [&]() {
        if (threadIdx.x % 32 == 0) ptx::bulk_wait_all();
    };
    uint32_t uc = 0;
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
                for (int x = 0; x < D / 8; ++x) {
                    reinterpret_cast<uint4*>(dk_row)[x] = make_uint4(0, 0, 0, 0);
                    reinterpret_cast<uint4*>(dv_row)[x] = make_uint4(0, 0, 0, 0);
                }
            }
            continue;
        }
        if (!warp_wait_phase(bar(T::KB_ACC_FULL), uc & 1u, ctl, SITE_B_ACC_FULL)) {
            drain();
            return;
        }
        ptx::tc_fence_after();
        // dV, then dK (x scale), as 32-row boxes of this warp's keys; a box
        // that starts past the last key has nothing to store
        const int key0 = w.j * 128 + 32 * quad;
        // dK and dV read: the next unit may accumulate into them (a separate
        // signal for dV, letting the next unit's first dV start before dK is
        // read, measured 2 % slower at N = 8192 on GB300)
        const auto release = [&]() {
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(T::KB_ACC_FREE));
        };
        if (!bwd_varlen(VAR) || p.cu_k == nullptr || key0 + 32 <= w.nk) {
            epi_store_rows<D, T::SW, BF16, BwdWarps<D>::lean_store(CAUSAL)>(tmem + lane_addr + T::TM_DV, 1.f, stage, tmDV, w.krow0 + key0, w.hk, w.zc,
                                           key0 < w.nk, []() {});
            epi_store_rows<D, T::SW, BF16, BwdWarps<D>::lean_store(CAUSAL)>(tmem + lane_addr + T::TM_DK, p.scale, stage, tmDK, w.krow0 + key0, w.hk,
                                           w.zc, key0 < w.nk, release);
        } else {
            direct_store_row<D, BF16>(tmem + lane_addr + T::TM_DV, 1.f, dv_row, key < w.nk, []() {});
            direct_store_row<D, BF16>(tmem + lane_addr + T::TM_DK, p.scale, dk_row, key < w.nk, release);
        }
        ++uc;
    }
    drain();
}

// Aligned dynamic shared memory base (the swizzled tiles need 1024 bytes);
// false (and an error in the status word) when the launch left no room.
__device__ __forceinline__ bool bwd_smem_base(uint8_t* raw, int used, int bytes, const BwdParams& p, uint8_t*& smem) {
    const uint32_t a = ptx::smem_addr(raw);
    const uint32_t pad = (1024u - (a & 1023u)) & 1023u;
    if (pad + (uint32_t)used > (uint32_t)bytes) {
        if (threadIdx.x == 0) atomicCAS(p.status, 0u, 4u /* FA_ERR_CUDA */ | (0xFFu << 8) | ((blockIdx.x & 0xFFFFu) << 16));
        return false;
    }
    smem = raw + pad;
    return true;
}


// ===================================================================== dQ ===

template <int D, bool CAUSAL, int VAR>
__device__ void q_producer(const CUtensorMap* tmK, const CUtensorMap* tmV, const CUtensorMap* tmQ,
                           const CUtensorMap* tmDO, const BwdParams& p, uint32_t sbase, uint32_t bar0, const Ctl& ctl, int first) {
    using T = BwdTraits<D>;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    const uint64_t pol_q = ptx::policy_evict_first();  // read once per unit
    const uint64_t pol_kv = ptx::policy_evict_last();  // read by every query block of the group
    uint32_t uc = 0, g = 0;
    bool ok = true;
    for (int pos = first; ok && unit_at<CAUSAL>(pos) < p.nunits_q; pos += gridDim.x) {
        const DqUnit w = dq_unit<CAUSAL, VAR>(unit_at<CAUSAL>(pos), p);
        if (!unit_checked(w, p, ctl, SITE_CHECK_BWD_LOAD)) { ok = false; break; }
        if (w.skip) continue;
        if (uc > 0 && !wait_phase(bar(T::QB_QD_EMPTY), (uc - 1) & 1u, ctl, SITE_B_QD_EMPTY)) { ok = false; break; }
        ptx::mbar_arrive_expect_tx(bar(T::QB_QD_FULL), 2 * T::TILE);
        for (int c = 0; c < T::NCHUNK; ++c) {
            ptx::tma_load_4d(sbase + T::Q_OFF_Q + c * (128 * T::SW), tmQ, bar(T::QB_QD_FULL), c * T::SWE,
                             w.qrow0 + w.i * 128, w.hq, w.zc, pol_q);
            ptx::tma_load_4d(sbase + T::Q_OFF_DO + c * (128 * T::SW), tmDO, bar(T::QB_QD_FULL), c * T::SWE,
                             w.qrow0 + w.i * 128, w.hq, w.zc, pol_q);
        }
        ++uc;
        for (int j = 0; j < w.nkv; ++j, ++g) {
            const uint32_t st = g & 1u;
            if (g >= 2 && !wait_phase(bar(T::QB_KV_EMPTY + st), ((g - 2) >> 1) & 1u, ctl, SITE_B_KV_EMPTY)) {
                ok = false;
                break;
            }
            const uint32_t full = bar(T::QB_KV_FULL + st);
            ptx::mbar_arrive_expect_tx(full, 2 * T::TILE);
            for (int c = 0; c < T::NCHUNK; ++c) {
                ptx::tma_load_4d(sbase + T::Q_OFF_K + st * T::TILE + c * (128 * T::SW), tmK, full, c * T::SWE,
                                 w.krow0 + (w.j0 + j) * 128, w.hk, w.zc, pol_kv);
                ptx::tma_load_4d(sbase + T::Q_OFF_V + st * T::TILE + c * (128 * T::SW), tmV, full, c * T::SWE,
                                 w.krow0 + (w.j0 + j) * 128, w.hk, w.zc, pol_kv);
            }
        }
    }
    if (!ok) {
        if (uc > 0) drain_phase(bar(T::QB_QD_FULL), (uc - 1) & 1u, ctl.limit_ns);
        for (uint32_t x = g > 2u ? g - 2u : 0u; x < g; ++x)
            drain_phase(bar(T::QB_KV_FULL + (x & 1u)), (x >> 1) & 1u, ctl.limit_ns);
    }
}

// Per key block g: S_{g+1} goes to the other TMEM slot while the softmax
// warps turn S_g and dP_g into dS_g; then dQ += dS_g K_g and dP_{g+1}.
template <int D, bool CAUSAL, bool BF16, int VAR>
__device__ void q_issuer(const BwdParams& p, uint32_t sbase, uint32_t bar0, uint32_t tmem, const Ctl& ctl, int first) {
    using T = BwdTraits<D>;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    constexpr uint32_t ID_SQ = ptx::idesc_f16(128, 128, BF16, false, false);  // S = Q Kᵀ, dP = dO Vᵀ
    constexpr uint32_t ID_DQ = ptx::idesc_f16(128, D, BF16, false, true);     // dQ += dS K (K MN-major)
    constexpr uint32_t HI = ptx::smem_desc_hi(8 * T::SW, T::SWIZZLE_CODE);
    const uint32_t q_lo = ptx::smem_desc_lo(sbase + T::Q_OFF_Q, 16);
    const uint32_t do_lo = ptx::smem_desc_lo(sbase + T::Q_OFF_DO, 16);
    auto issue_s = [&](uint32_t g) -> bool {
        const uint32_t st = g & 1u;
        if (!wait_phase(bar(T::QB_KV_FULL + st), (g >> 1) & 1u, ctl, SITE_B_KV_FULL)) return false;
        ptx::tc_fence_after();
        const uint32_t k_lo = ptx::smem_desc_lo(sbase + T::Q_OFF_K + st * T::TILE, 16);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
            ptx::mma_ss(tmem + T::TM_QS + st * 128, ptx::desc64(q_lo + kmaj_off(kk, T::SWE, T::SW), HI),
                        ptx::desc64(k_lo + kmaj_off(kk, T::SWE, T::SW), HI), ID_SQ, kk > 0 ? 1u : 0u);
        ptx::tc_commit(bar(T::QB_S_FULL + st));
        return true;
    };
    auto issue_dp = [&](uint32_t g) {
        const uint32_t v_lo = ptx::smem_desc_lo(sbase + T::Q_OFF_V + (g & 1u) * T::TILE, 16);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
            ptx::mma_ss(tmem + T::TM_QDP, ptx::desc64(do_lo + kmaj_off(kk, T::SWE, T::SW), HI),
                        ptx::desc64(v_lo + kmaj_off(kk, T::SWE, T::SW), HI), ID_SQ, kk > 0 ? 1u : 0u);
        ptx::tc_commit(bar(T::QB_DP_FULL));
    };
    uint32_t uc = 0, g = 0;
    bool ok = true;
    for (int pos = first; ok && unit_at<CAUSAL>(pos) < p.nunits_q; pos += gridDim.x) {
        const DqUnit w = dq_unit<CAUSAL, VAR>(unit_at<CAUSAL>(pos), p);
        if (!unit_checked(w, p, ctl, SITE_CHECK_BWD_MMA)) { ok = false; break; }
        if (w.skip) continue;
        if (!wait_phase(bar(T::QB_QD_FULL), uc & 1u, ctl, SITE_B_QD_FULL)) { ok = false; break; }
        if (!issue_s(g)) { ok = false; break; }
        issue_dp(g);
        // the unit's last S and dP are its last reads of Q and dO: the next
        // unit's Q, dO may land while its last dQ products run
        if (w.nkv == 1) ptx::tc_commit(bar(T::QB_QD_EMPTY));
        for (int j = 0; j < w.nkv; ++j, ++g) {
            const uint32_t st = g & 1u;
            if (j + 1 < w.nkv && !issue_s(g + 1)) { ok = false; break; }
            if (!wait_phase(bar(T::QB_DS_FULL + st), (g >> 1) & 1u, ctl, SITE_B_DS_FULL)) { ok = false; break; }
            if (j == 0 && uc > 0 && !wait_phase(bar(T::QB_DQ_FREE), (uc - 1) & 1u, ctl, SITE_B_DQ_FREE)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            const uint32_t kmn_lo = ptx::smem_desc_lo(sbase + T::Q_OFF_K + st * T::TILE, 128 * T::SW);
#pragma unroll
            for (int kk = 0; kk < 128 / 16; ++kk)
                ptx::mma_ts(tmem + T::TM_DQ, tmem + T::TM_QS + st * 128 + packed_col<BwdWarps<D>::CW>(kk),
                            ptx::desc64(kmn_lo + ((kk * 16 * T::SW) >> 4), HI), ID_DQ, (j > 0 || kk > 0) ? 1u : 0u);
            ptx::tc_commit(bar(T::QB_KV_EMPTY + st));  // K_g, V_g free
            if (j + 1 < w.nkv) {
                issue_dp(g + 1);
                if (j + 2 == w.nkv) ptx::tc_commit(bar(T::QB_QD_EMPTY));  // Q, dO free
            }
        }
        if (!ok) break;
        ptx::tc_commit(bar(T::QB_DQ_FULL));   // dQ of the unit complete
        ++uc;
    }
    if (!ok) {
        ptx::tc_commit(bar(T::QB_DRAIN));
        drain_phase(bar(T::QB_DRAIN), 0u, ctl.limit_ns);
    }
}

// Thread = query (TMEM lane); column group h takes keys h*CW .. h*CW + CW - 1 of each
// block.  lse2 and Δ are per row, so they stay in registers for the unit.
template <int D, bool CAUSAL, bool BF16, int VAR>
__device__ void q_softmax(const BwdParams& p, uint32_t bar0, uint32_t tmem, int h, const Ctl& ctl, int first) {
    using T = BwdTraits<D>;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    const int quad = (threadIdx.x / 32) % 4;
    const int row = quad * 32 + threadIdx.x % 32;  // query within the block
    const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
    const float c = p.scale_log2;
    constexpr int CW = BwdWarps<D>::CW, CH = BwdWarps<D>::CH;
    uint32_t g = 0;
    for (int pos = first; unit_at<CAUSAL>(pos) < p.nunits_q; pos += gridDim.x) {
        const DqUnit w = dq_unit<CAUSAL, VAR>(unit_at<CAUSAL>(pos), p);
        if (!unit_checked(w, p, ctl, SITE_CHECK_BWD_SOFTMAX)) return;
        if (w.skip) continue;
        const int64_t r = ((int64_t)w.z * p.Hq + w.hq) * p.Tq * 128 + (int64_t)w.i * 128 + row;
        const float l2 = __ldg(p.lse2 + r), dl = __ldg(p.delta + r);
        const float slope2 =
            bwd_alibi(VAR) ? -__ldg(p.alibi + w.hq) * 1.4426950408889634f : 0.f;
        for (int j = 0; j < w.nkv; ++j, ++g) {
            const uint32_t st = g & 1u;
            const uint32_t slot = tmem + lane_addr + T::TM_QS + st * 128;
            if (!warp_wait_phase(bar(T::QB_S_FULL + st), (g >> 1) & 1u, ctl, SITE_B_S_FULL)) return;
            ptx::tc_fence_after();
            const int jj = w.j0 + j;                // the key block
            const bool diag = CAUSAL && jj == w.i;  // key > query only on the diagonal block
            // variants: d = query − key = dbase − col (as in the dK/dV phase)
            const int dbase = (w.i - jj) * 128 + row;
            const float dbf = (float)(dbase - h * CW);  // d of this group's first column (exact: |d| < 2^24)
            const bool full =
                VAR == 0 || var_block_kept<CAUSAL>((w.i - jj) * 128 - 127, (w.i - jj) * 128 + 127, jj * 128 + 128, w.nk, p);
            uint32_t pk[CW / 2];
#pragma unroll
            for (int cc = 0; cc < CW / CH; ++cc) {
                uint32_t rr[CH];
                tmem_ld_n<CH>(slot + h * CW + CH * cc, rr);
#pragma unroll
                for (int x = 0; x < CH / 2; ++x) {
                    const int col = h * CW + CH * cc + 2 * x;
                    float e0 = fmaf(__uint_as_float(rr[2 * x]), c, -l2);
                    float e1 = fmaf(__uint_as_float(rr[2 * x + 1]), c, -l2);
                    if constexpr (VAR == 0) {
                        if (diag && col > row) e0 = -INFINITY;
                        if (diag && col + 1 > row) e1 = -INFINITY;
                    } else {
                        const int d0 = dbase - col;
                        if constexpr (bwd_alibi(VAR)) {
                            const float df = dbf - (float)(CH * cc + 2 * x);
                            e0 = fmaf(slope2, fabsf(df), e0);
                            e1 = fmaf(slope2, fabsf(df - 1.f), e1);
                        }
                        if (!full) {
                            if (var_dropped<CAUSAL>(d0, jj * 128 + col, w.nk, p)) e0 = -INFINITY;
                            if (var_dropped<CAUSAL>(d0 - 1, jj * 128 + col + 1, w.nk, p)) e1 = -INFINITY;
                        }
                    }
                    pk[(CH / 2) * cc + x] = pack2<BF16>(ptx::ex2(e0), ptx::ex2(e1));
                }
            }
            if (!warp_wait_phase(bar(T::QB_DP_FULL), g & 1u, ctl, SITE_B_DP_FULL)) return;
            ptx::tc_fence_after();
#pragma unroll
            for (int cc = 0; cc < CW / CH; ++cc) {
                uint32_t rr[CH];
                tmem_ld_n<CH>(tmem + lane_addr + T::TM_QDP + h * CW + CH * cc, rr);
                uint32_t ds[CH / 2];
#pragma unroll
                for (int x = 0; x < CH / 2; ++x) {
                    const float2 pp = unpack2<BF16>(pk[(CH / 2) * cc + x]);
                    ds[x] = pack2<BF16>(pp.x * (__uint_as_float(rr[2 * x]) - dl), pp.y * (__uint_as_float(rr[2 * x + 1]) - dl));
                }
                // dS over the slot's packed columns h*64 + 16cc .. (S already read)
                tmem_st_n<CH / 2>(slot + h * CW + (CH / 2) * cc, ds);
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(T::QB_DS_FULL + st));
        }
    }
}

// Thread = TMEM lane = query: dQ (times scale) read out, released, stored.
template <int D, bool CAUSAL, bool BF16, int VAR>
__device__ void q_epilogue(const CUtensorMap* tmDQ, const BwdParams& p, uint32_t sbase, uint32_t bar0, uint32_t tmem,
                           const Ctl& ctl, int first) {
    using T = BwdTraits<D>;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    const int quad = (threadIdx.x / 32) % 4;
    const int row = quad * 32 + threadIdx.x % 32;  // query within the block
    const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
    const uint32_t stage = sbase + T::Q_OFF_OST + (uint32_t)quad * 32u * T::SW;  // this warp's staging rows
    // lane 0's stores must have read shared memory before the CTA exits
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
        // dQ (x scale) as 32-row boxes of this warp's queries
        const int q0 = w.i * 128 + 32 * quad;
        const auto release = [&]() {
            // dQ read: the next unit may accumulate into it
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(T::QB_DQ_FREE));
        };
        if (!bwd_varlen(VAR) || p.cu_q == nullptr || q0 + 32 <= w.nq) {
            epi_store_rows<D, T::SW, BF16, BwdWarps<D>::lean_store(CAUSAL)>(tmem + lane_addr + T::TM_DQ, p.scale, stage, tmDQ, w.qrow0 + q0, w.hq, w.zc,
                                           q0 < w.nq, release);
        } else {
            const int qr = w.i * 128 + row;
            uint8_t* dq_row = reinterpret_cast<uint8_t*>(p.dq) +
                              2 * ((int64_t)w.zc * p.sdq_z + (int64_t)w.hq * p.sdq_h + (int64_t)(w.qrow0 + qr) * p.sdq_n);
            direct_store_row<D, BF16>(tmem + lane_addr + T::TM_DQ, p.scale, dq_row, qr < w.nq, release);
        }
        ++uc;
    }
    drain();
}


// ================================================================ pre pass ==
// Per query row, padded to whole 128-row blocks: Δ = rowsum(dO ∘ O) in fp32
// from the input-type values, and the lse in base 2 (+inf past Nq, or past a
// packed sequence's length, so those rows and columns get P = 0: the rows of
// the next sequence that a block crossing the end reads contribute nothing).  D/8 threads per row, 16 bytes of O and dO each.
// ================================================================ fused ======
// One launch runs both gradient kernels' work: each CTA takes its dK/dV units
// (positions c, c + grid, ...), then, in the same shared memory and TMEM, its
// dQ units from position grid - 1 - c on, so a CTA that drew one more dK/dV
// unit than others draws one fewer dQ unit (Z4 H16 N1024: 512 + 512 units on
// 152 CTAs, at most 7 per CTA instead of 4 + 4).  The phases need nothing
// from each other (both read the pre kernel's lse2 and Delta), so no CTA
// waits for another.  The dQ phase's barriers lie in memory the dK/dV phase
// used for data; they are set up only after every role of that phase has
// finished: its MMAs drained, its tensor stores read out.
template <int D, bool CAUSAL, bool BF16, int VAR>
__global__ void __launch_bounds__(BwdWarps<D>::THREADS, 1)
    fa_bwd_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
                  const __grid_constant__ CUtensorMap tmDK, const __grid_constant__ CUtensorMap tmDV,
                  const __grid_constant__ CUtensorMap tmDQ, const BwdParams p) {
    using T = BwdTraits<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = nullptr;
    if (!bwd_smem_base(smem_raw, T::FUSED_SMEM_USED, T::FUSED_SMEM_BYTES, p, smem)) return;
    const uint32_t sbase = ptx::smem_addr(smem);
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + T::FUSED_OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + T::FUSED_OFF_MISC + 4);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    // ---- dK / dV ----
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
    constexpr int W_EPI = BwdWarps<D>::SOFTMAX_WARPS, W_PRODUCER = W_EPI + 4, W_ISSUER = W_EPI + 5;
    if (warp == W_ISSUER) {
        ptx::tmem_alloc(ptx::smem_addr(const_cast<uint32_t*>(tmem_slot)), T::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const Ctl ctl{abort_flag, p.status, p.wait_limit_ns};
    // launched as a programmatic dependent: the set-up above overlaps the
    // previous kernel's tail; nothing below touches global memory before it
    // has completed
    ptx::grid_dependency_wait();
    ptx::grid_launch_dependents();
    if constexpr (BwdWarps<D>::SPLIT_REGS) {
        if (warp < W_EPI) ptx::setmaxnreg_inc<BwdWarps<D>::REG_SOFTMAX>();
        else if (warp < W_PRODUCER) ptx::setmaxnreg_dec<BwdWarps<D>::reg_epi(CAUSAL)>();
        else ptx::setmaxnreg_dec<BwdWarps<D>::reg_ctrl(CAUSAL)>();
    }
    if (warp < W_EPI) {
        kv_softmax<D, CAUSAL, BF16, VAR>(p, sbase, kbar0, tmem, warp / 4, ctl);
    } else if (warp < W_PRODUCER) {
        kv_epilogue<D, CAUSAL, BF16, VAR>(&tmDK, &tmDV, p, sbase, kbar0, tmem, ctl);
    } else if (warp == W_PRODUCER) {
        if (lane == 0) kv_producer<D, CAUSAL, VAR>(&tmK, &tmV, &tmQ, &tmDO, p, sbase, kbar0, ctl);
    } else if (warp == W_ISSUER) {
        if (lane == 0) kv_issuer<D, CAUSAL, BF16, VAR>(p, sbase, kbar0, tmem, ctl);
    }
    ptx::tc_fence_before();
    __syncthreads();

    // ---- dQ (skipped after an abort: the status word already says why) ----
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
            q_softmax<D, CAUSAL, BF16, VAR>(p, qbar0, tmem, warp / 4, ctl, first);
        } else if (warp < W_PRODUCER) {
            q_epilogue<D, CAUSAL, BF16, VAR>(&tmDQ, p, sbase, qbar0, tmem, ctl, first);
        } else if (warp == W_PRODUCER) {
            if (lane == 0) q_producer<D, CAUSAL, VAR>(&tmK, &tmV, &tmQ, &tmDO, p, sbase, qbar0, ctl, first);
        } else if (warp == W_ISSUER) {
            if (lane == 0) q_issuer<D, CAUSAL, BF16, VAR>(p, sbase, qbar0, tmem, ctl, first);
        }
        ptx::tc_fence_before();
        __syncthreads();
    }
    if (warp == W_ISSUER) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, T::TMEM_COLS);
    }
}

template <int D, bool BF16>
__global__ void __launch_bounds__(256) fa_bwd_pre_kernel(const BwdParams p) {
    ptx::grid_dependency_wait();  // O, dO and lse come from earlier kernels on the stream
    ptx::grid_launch_dependents();
    constexpr int TPR = D / 8;
    const int64_t rows = (int64_t)p.Z * p.Hq * p.Tq * 128;
    const int sub = threadIdx.x % TPR;
    // the trip count is the same for the TPR lanes of a row (rows and the
    // stride are multiples of 32 / TPR), so the shuffles below see them all
    for (int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / TPR; r < rows;
         r += (int64_t)gridDim.x * blockDim.x / TPR) {
        const int64_t head = r / ((int64_t)p.Tq * 128);
        const int i = (int)(r - head * p.Tq * 128);
        const int z = (int)(head / p.Hq), hq = (int)(head % p.Hq);
        // the row's batch entry, packed row and lse index; packed sequences:
        // row i of sequence z, kept while i is below its length
        int zc = z, n = p.Nq;
        int64_t qr = i, li = head * p.Nq + i;
        if (p.cu_q != nullptr) {
            const int q0 = min(max(__ldg(p.cu_q + z), 0), p.Nq), q1 = min(max(__ldg(p.cu_q + z + 1), 0), p.Nq);
            zc = 0;
            n = q1 > q0 ? q1 - q0 : 0;
            qr = (int64_t)q0 + i;
            li = (int64_t)hq * p.Nq + q0 + i;
        }
        const bool kept = i < n;
        float delta = 0.f;
        if (kept) {
            const uint4 a = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.o) + (int64_t)zc * p.so_z +
                                                           (int64_t)hq * p.so_h + qr * p.so_n)[sub];
            const uint4 b = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.dO) + (int64_t)zc * p.sdo_z +
                                                           (int64_t)hq * p.sdo_h + qr * p.sdo_n)[sub];
            const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int y = 0; y < 4; ++y) {
                const float2 fa = unpack2<BF16>(aw[y]), fb = unpack2<BF16>(bw[y]);
                delta = fmaf(fa.x, fb.x, delta);
                delta = fmaf(fa.y, fb.y, delta);
            }
        }
#pragma unroll
        for (int m = TPR / 2; m > 0; m /= 2) delta += __shfl_xor_sync(0xffffffffu, delta, m);
        if (sub == 0) {
            p.delta[r] = delta;
            p.lse2[r] = kept ? p.lse[li] * 1.4426950408889634f : INFINITY;
        }
    }
}

}  // namespace fa
