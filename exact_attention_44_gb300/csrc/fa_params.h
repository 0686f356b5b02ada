// Kernel parameter block for the attention forward kernels (host and device).
#pragma once

#include <cstdint>

namespace fa {

constexpr int BM = 128;            // query rows per tile (one TMEM lane per row)
// Warp roles of the forward kernel: warp 0: Q/K loads, warp 1: S = Q Kᵀ
// issuer, warp 2: O += P V issuer, warp 3: V loads, then 4 warps per softmax
// column group (thread = query row = TMEM lane), then 4 epilogue warps.  The
// number of column groups depends on the head dim (Traits<D>::NG).
constexpr int fwd_threads(int groups) { return 32 * (4 + 4 * groups + 4); }

// Where a bounded wait gave up; recorded in bits 8-15 of the device status word.
enum WaitSite : uint32_t {
    SITE_Q_FULL = 1,
    SITE_K_FULL = 2,
    SITE_V_FULL = 3,
    SITE_Q_EMPTY = 4,
    SITE_K_EMPTY = 5,
    SITE_V_EMPTY = 6,
    SITE_S_FULL = 7,
    SITE_P_FULL = 8,
    SITE_PV_DONE = 9,
    SITE_EPI_FULL = 10,
    SITE_EPI_EMPTY = 11,
    SITE_O_FREE = 12,
    SITE_MAX_XCHG = 13,
    SITE_P_FREE = 14,
    SITE_S_FREE = 15,
    SITE_PEER_Q = 16,       // CTA pair: the other CTA's Q tile, K or V half landed
    SITE_PEER_K = 17,
    SITE_PEER_V = 18,
    SITE_DRAIN = 19,
    // backward
    SITE_B_KV_FULL = 20,
    SITE_B_KV_EMPTY = 21,
    SITE_B_QD_FULL = 22,
    SITE_B_QD_EMPTY = 23,
    SITE_B_S_FULL = 24,
    SITE_B_DP_FULL = 25,
    SITE_B_P_FULL = 26,
    SITE_B_DS_FULL = 27,
    SITE_B_DS_FREE = 28,
    SITE_B_DQ_FULL = 29,
    SITE_B_DQ_FREE = 30,
    SITE_B_ACC_FULL = 31,
    SITE_B_ACC_FREE = 32,
    // debug index checks (builds with FA_DEBUG_CHECKS=1): the role that found
    // a unit outside the launch's sizes
    SITE_CHECK_LOAD_QK = 40,
    SITE_CHECK_LOAD_V = 41,
    SITE_CHECK_MMA_S = 42,
    SITE_CHECK_MMA_PV = 43,
    SITE_CHECK_SOFTMAX = 44,
    SITE_CHECK_EPILOGUE = 45,
    SITE_CHECK_BWD_LOAD = 46,       // backward roles: TMA producer, MMA issuer, softmax, epilogue
    SITE_CHECK_BWD_MMA = 47,
    SITE_CHECK_BWD_SOFTMAX = 48,
    SITE_CHECK_BWD_EPILOGUE = 49,
};

// Status code of a failed debug index check (FA_ERR_DEVICE_CHECK in fa.h).
constexpr uint32_t STATUS_DEVICE_CHECK = 7;

struct FwdParams {
    void* o;                 // output, dtype of the inputs, d-stride 1
    float* lse;              // (Z, Hq, Nq) fp32 contiguous, or nullptr
    int64_t so_z, so_h, so_n;  // O strides in elements
    int Z, Hq, Hkv, Nq, Nkv;
    int group;               // Hq / Hkv
    int Tq, Tk;              // ceil(Nq / BM), ceil(Nkv / BN)
    int ntiles;              // Z * Hq * Tq
    int head_group;          // causal tile order: (z, hq) heads per group (>= 1)
    // |scale| * log2(e), > 0 (see fwd_scale in the host code); with
    // negate_s the S = Q Kᵀ products negate Q, so that the kernel's scores
    // times scale_log2 are the scaled scores of a negative scale
    float scale_log2;
    int negate_s;
    uint32_t* status;        // device status word (first error wins)
    uint64_t wait_limit_ns;  // bound on every mbarrier wait
    int inject_stall;        // test hook: 1 = withhold the first K tile of CTA 0 (waits must time out)
    // split-KV schedule (split != 0): (tile, key block) pairs cut into one range per CTA
    int split;
    int64_t head_blocks;     // key blocks visited by all query tiles of one (z, hq) head
    int64_t total_blocks;    // Z * Hq * head_blocks
    float* scratch;          // partial-result slots, 2 per CTA, each slot_floats floats
    int64_t slot_floats;     // BM * D floats of O / l, then BM floats of base-2 lse, padded
    // variants (the kernel instantiated with VAR): key j is kept for query i
    // iff i - win_left <= j <= i + win_right (-1: open side); ALiBi adds
    // -alibi[hq] * |i - j| to the scaled score; with cu_q / cu_k, Z counts
    // sequences of packed rows and Tq covers the longest query sequence
    int win_left, win_right;
    const float* alibi;      // (Hq) slopes, or nullptr
    const int* cu_q;         // (Z + 1) offsets into the packed query rows, or nullptr
    const int* cu_k;         // (Z + 1) offsets into the packed key rows
    // CTA-pair kernel (pair != 0): a cluster of two CTAs takes a unit of two
    // query tiles that see the same key blocks -- pair 1: query heads 2k and
    // 2k + 1 (one GQA group) at query block mb; pair 2: query blocks 2m and
    // 2m + 1 of one head -- one tile per CTA.  Units are tiles of "virtual
    // heads" of pair_tq virtual query blocks, ordered like whole tiles
    // (causal: groups of pair_head_group virtual heads, heaviest first).
    int pair;
    int pair_heads;          // Z * Hq / 2 (pair 1) or Z * Hq (pair 2)
    int pair_tq;             // Tq (pair 1) or ceil(Tq / 2) (pair 2)
    int pair_units;          // pair_heads * pair_tq
    int pair_head_group;
};

// Backward kernel parameters (fa_bwd).  Tensor strides are in elements; the
// workspace holds, per query row padded to whole 128-row blocks, the base-2
// lse (+inf past Nq) and Delta = rowsum(dO * O).
struct BwdParams {
    const void* o;           // forward output, dtype
    const float* lse;        // forward lse (Z, Hq, Nq), natural log
    const void* dO;          // upstream gradient, dtype
    void* dq;                // outputs, dtype
    void* dk;
    void* dv;
    int64_t so_z, so_h, so_n;
    int64_t sdo_z, sdo_h, sdo_n;
    int64_t sdq_z, sdq_h, sdq_n;
    int64_t sdk_z, sdk_h, sdk_n;
    int64_t sdv_z, sdv_h, sdv_n;
    int Z, Hq, Hkv, Nq, Nkv;
    int group;               // Hq / Hkv
    int Tq, Tk;              // query blocks of 128 rows, key blocks of 128 keys
    int nunits;              // dK/dV units: Z * Hkv * Tk (one key block of one kv head)
    int nunits_q;            // dQ units: Z * Hq * Tq (one query block of one query head)
    int kv_head_group;       // dK/dV unit order: (z, kv head) heads per group (>= 1)
    int q_head_group;        // causal dQ unit order: (z, q head) heads per group (>= 1)
    float scale;             // softmax scale (dQ and dK carry it)
    float scale_log2;        // scale * log2(e)
    float* lse2;             // (Z, Hq, Tq * 128) fp32
    float* delta;            // (Z, Hq, Tq * 128) fp32
    uint32_t* status;
    uint64_t wait_limit_ns;
    int inject_stall;        // test hook: 1 = withhold CTA 0's first K/V copy of the dK/dV phase
    // variants (the kernel instantiated with VAR, D <= 128): key j is kept
    // for query i iff i - win_left <= j <= i + win_right (-1: open side);
    // ALiBi adds -alibi[hq] * |i - j| to the scaled score
    int win_left, win_right;
    const float* alibi;      // (Hq) slopes, or nullptr
    // packed variable-length batches (VAR 3, 4): Z counts sequences, sequence
    // z owns query rows cu_q[z] .. cu_q[z+1]-1 and key rows cu_k[z] ..
    // cu_k[z+1]-1 of (1, H, total, D) tensors (Nq, Nkv: the totals; Tq, Tk:
    // blocks of the longest sequence); lse is (Hq, Nq)
    const int* cu_q;
    const int* cu_k;
};

}  // namespace fa
