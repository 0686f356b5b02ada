// C ABI of libfa: argument validation, TMA tensor maps, specialisation
// dispatch, launch, and the per-device status word.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cfloat>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <mutex>
#include <vector>
#include <algorithm>

#include "fa.h"
#include "fa_bwd_kernel.cuh"
#include "fa_fwd_kernel.cuh"
#include "fa_launch.h"

namespace {

__device__ uint32_t g_fa_status;  // first device-side error of any launch on this device

constexpr int kMaxDevices = 64;

// What a launch needs to know about device `dev` (the current device): its
// SM count and L2 size (fixed for the device), and the device address of the
// status word, which belongs to the current CUDA context: it is looked up
// again when the context changes (after cudaDeviceReset the module is loaded
// anew and the word may move).  Failures are not remembered.
struct DeviceInfo {
    std::mutex mu;
    bool have_attrs = false;
    int sms = 0;
    int l2_bytes = 0;
    uint64_t ctx = 0;  // context the status address was looked up in (0: none yet)
    uint32_t* status = nullptr;
};
DeviceInfo g_devices[kMaxDevices];

struct LaunchInfo {
    int sms;
    int l2_bytes;
    uint32_t* status;
};

cudaError_t device_info(int dev, LaunchInfo* out) {
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    DeviceInfo& d = g_devices[dev];
    std::lock_guard<std::mutex> lock(d.mu);
    cudaError_t err;
    if (!d.have_attrs) {
        int sms = 0, l2 = 0;
        if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return err;
        if ((err = cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev)) != cudaSuccess) return err;
        d.sms = sms;
        d.l2_bytes = l2;
        d.have_attrs = true;
    }
    // the status word's address in the current context, looked up on the
    // first call in a context (which should come before any stream capture)
    const uint64_t ctx = fa::current_context_id();
    if (ctx == 0 || ctx != d.ctx || d.status == nullptr) {
        void* status = nullptr;
        if ((err = cudaGetSymbolAddress(&status, g_fa_status)) != cudaSuccess) return err;
        d.status = static_cast<uint32_t*>(status);
        d.ctx = fa::current_context_id();  // the lookup may have created the context
    }
    *out = LaunchInfo{d.sms, d.l2_bytes, d.status};
    return cudaSuccess;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// cuCtxGetCurrent and cuCtxGetId through the runtime's driver entry points
// (no link against libcuda): the ID of the calling thread's current context.
struct CtxFns {
    PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    PFN_cuCtxGetId_v12000 get_id = nullptr;
};
const CtxFns& ctx_fns() {
    static const CtxFns fns = [] {
        CtxFns f;
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            f.get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            f.get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
        return f;
    }();
    return fns;
}

std::atomic<uint64_t> g_wait_limit_ns{0};
std::atomic<int> g_inject_stall{0};
std::atomic<int> g_force_split{0};  // 0: decide by shape, 1: always cut key ranges, 2: never
std::atomic<int> g_force_chains{0};  // 0: decide by shape, 1: two softmax chains wherever they apply, 2: never
std::atomic<int> g_force_pair{0};    // 0: decide by shape, 1: CTA pairs wherever they apply, 2: never

uint64_t wait_limit_ns() {
    uint64_t v = g_wait_limit_ns.load();
    if (v) return v;
    double ms = 2000.0;  // every wait in a healthy kernel takes microseconds
    if (const char* e = std::getenv("FA_WAIT_LIMIT_MS")) {
        double x = std::atof(e);
        if (x >= 1.0 && x <= 600000.0) ms = x;
    }
    v = (uint64_t)(ms * 1e6);
    g_wait_limit_ns.store(v);
    return v;
}

// With FA_DEBUG set in the environment, a failed CUDA call is described on
// stderr before FA_ERR_CUDA is returned.
fa_status cuda_fail(const char* what, int code, const char* text) {
    static const bool verbose = std::getenv("FA_DEBUG") != nullptr;
    if (verbose) std::fprintf(stderr, "libfa: %s failed: %d %s\n", what, code, text ? text : "");
    return FA_ERR_CUDA;
}
fa_status cuda_fail(const char* what, cudaError_t e) { return cuda_fail(what, (int)e, cudaGetErrorString(e)); }
fa_status cuda_fail(const char* what, CUresult r) { return cuda_fail(what, (int)r, "driver error"); }

bool supported_head_dim(int D) { return D == 16 || D == 32 || D == 64 || D == 128 || D == 256; }

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// The forward kernels take the softmax scale as c = |scale|·log2(e) > 0 and
// its sign separately.  They reference the probabilities of a row to the
// maximum of the raw scores times c and mask keys by setting raw scores to
// -inf, both of which need c > 0:
//   * scale < 0: the S = Q Kᵀ products negate Q (the tensor core's negate-A
//     bit, exact in fp16/bf16), so raw score times c is scale·s·log2(e);
//   * scale = 0 (every kept key weighs the same): c is the smallest normal
//     fp32 value 2^-126.  For a score |s| < 2^100, s·c has magnitude below
//     2^-25, where 2^x rounds to 1 in fp32, so every kept key gets p = 1 as
//     with scale 0, and masked keys (-inf) still get p = 0;
//   * a scale whose c overflows fp32 (|scale| > FLT_MAX / log2(e), about
//     2.4e38) is rejected: no scaled score would be representable.
// Returns false for a scale the kernels cannot take (non-finite, or c
// overflows).
bool fwd_scale(float scale, float* c, int* negate) {
    if (!std::isfinite(scale)) return false;
    const double x = std::fabs((double)scale) * 1.4426950408889634;  // exp(y) = 2^(y log2 e)
    if (!(x <= (double)FLT_MAX)) return false;
    float cf = (float)x;
    if (!(cf >= FLT_MIN)) cf = FLT_MIN;  // zero, or below the normal range
    *c = cf;
    *negate = scale < 0.f ? 1 : 0;
    return true;
}

fa_status check_shape(int Z, int Hq, int Hkv, int Nq, int Nkv, int D, int causal) {
    if (Z < 0 || Hq < 0 || Hkv < 1 || Nq < 0 || Nkv < 0) return FA_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return FA_ERR_INVALID_ARG;  // GQA group size Hq / Hkv must be whole
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    if (!supported_head_dim(D)) return FA_ERR_UNSUPPORTED;
    const int64_t rows = (int64_t)Z * Hq * Nq;
    if (rows > 0 && Nkv == 0) return FA_ERR_INVALID_ARG;  // softmax over no keys is undefined
    if ((int64_t)Z * Hq * cdiv(Nq, fa::BM) > INT32_MAX) return FA_ERR_UNSUPPORTED;
    return FA_OK;
}

// d-stride 1, 16-byte aligned base, non-negative strides that are multiples of
// 8 elements in every dimension of extent > 1 (TMA and 16-byte stores).
fa_status check_tensor(const void* ptr, const fa_strides* s, int64_t nb, int64_t nh, int64_t nn) {
    if (ptr == nullptr || s == nullptr) return FA_ERR_INVALID_ARG;
    if (s->d != 1) return FA_ERR_ALIGNMENT;
    if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0) return FA_ERR_ALIGNMENT;
    const int64_t st[3] = {s->b, s->h, s->n};
    const int64_t ext[3] = {nb, nh, nn};
    for (int i = 0; i < 3; ++i) {
        if (ext[i] <= 1) continue;
        if (st[i] < 0 || st[i] % 8 != 0 || st[i] >= (int64_t(1) << 38)) return FA_ERR_ALIGNMENT;
    }
    return FA_OK;
}

// 4-D tensor map (d, n, h, b) with a box of `box_rows` rows x one swizzle chunk.
CUresult make_map(CUtensorMap* map, const void* ptr, fa_dtype dt, int D, int N, int H, int B, const fa_strides* s,
                  int box_rows) {
    const int swe = fa::swizzle_elems_for(D);
    const CUtensorMapSwizzle sw = swe == 64   ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : swe == 32 ? CU_TENSOR_MAP_SWIZZLE_64B
                                              : CU_TENSOR_MAP_SWIZZLE_32B;
    // a dimension of extent 1 is never stepped along; give it a harmless stride
    const uint64_t filler = (uint64_t)D * 2 * (uint64_t)(N > 0 ? N : 1);
    auto bytes = [&](int64_t stride, int64_t extent) -> cuuint64_t {
        return extent > 1 ? (cuuint64_t)(stride * 2) : (cuuint64_t)filler;
    };
    cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)N, (cuuint64_t)H, (cuuint64_t)B};
    cuuint64_t strides[3] = {bytes(s->n, N), bytes(s->h, H), bytes(s->b, B)};
    cuuint32_t box[4] = {(cuuint32_t)swe, (cuuint32_t)box_rows, 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    auto fn = encode_fn();
    if (fn == nullptr) return CUDA_ERROR_NOT_SUPPORTED;
    return fn(map, dt == FA_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
              const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace

namespace fa {
uint64_t current_context_id() {
    const CtxFns& f = ctx_fns();
    if (f.get_current == nullptr || f.get_id == nullptr) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (f.get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
    if (f.get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return (uint64_t)id;
}

template <int D>
static void facts(int* bn, int* smem, int* swe) {
    *bn = Traits<D>::BN;
    *smem = Traits<D>::SMEM_BYTES;
    *swe = Traits<D>::SWE;
}
static void facts_for(int D, int* bn, int* smem, int* swe) {
    switch (D) {
        case 16: facts<16>(bn, smem, swe); break;
        case 32: facts<32>(bn, smem, swe); break;
        case 64: facts<64>(bn, smem, swe); break;
        case 128: facts<128>(bn, smem, swe); break;
        default: facts<256>(bn, smem, swe); break;
    }
}
int block_n_for(int D) { int a, b, c; facts_for(D, &a, &b, &c); return a; }
int smem_bytes_for(int D) { int a, b, c; facts_for(D, &a, &b, &c); return b; }
int swizzle_elems_for(int D) { int a, b, c; facts_for(D, &a, &b, &c); return c; }
}  // namespace fa

namespace {

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// Backward workspace: lse2 and Δ per query row padded to whole 128-row blocks.
size_t bwd_workspace_bytes(int Z, int Hq, int Nq, int D) {
    (void)D;
    const size_t tq = (size_t)cdiv(Nq, 128);
    return 2 * align256((size_t)Z * Hq * tq * 128 * 4);
}

// Floats per partial-result slot of the split schedule: O / l of BM rows
// (BM x D) and their base-2 log-sum-exps (BM), padded to 256 bytes.
int64_t split_slot_floats(int D) { return ((int64_t)fa::BM * D + fa::BM + 63) / 64 * 64; }
size_t split_workspace_bytes(int D, int grid) { return (size_t)2 * grid * split_slot_floats(D) * sizeof(float); }

// (tile, key block) pairs of one (z, hq) head under the kernel's schedule
template <bool CAUSAL, int BN>
int64_t head_blocks_t(const fa::FwdParams& p) {
    using S = fa::Sched<CAUSAL, BN>;
    return S::head_prefix(p.Tq - 1, p) + S::tile_nkv(p.Tq - 1, p);
}
int64_t head_blocks(const fa::FwdParams& p, bool causal, int bn) {
    if (bn == 64) return causal ? head_blocks_t<true, 64>(p) : head_blocks_t<false, 64>(p);
    return causal ? head_blocks_t<true, 128>(p) : head_blocks_t<false, 128>(p);
}

// Key blocks of the busiest CTA when whole tiles are dealt round-robin to
// `grid` CTAs in the kernel's tile order (causal: last query block first).
template <bool CAUSAL, int BN, bool ALT>
int64_t tile_mode_max_blocks_t(const fa::FwdParams& p, int grid) {
    using S = fa::Sched<CAUSAL, BN, false, ALT>;
    if (!CAUSAL) return cdiv(p.ntiles, grid) * p.Tk;
    int64_t worst = 0;
    for (int c = 0; c < grid; ++c) {
        int64_t sum = 0;
        for (int64_t pos = c; S::tile_at(pos, grid) < p.ntiles; pos += grid) {
            int64_t head;
            int mb;
            S::causal_tile(S::tile_at(pos, grid), p, head, mb);
            sum += S::tile_nkv(mb, p);
        }
        worst = std::max(worst, sum);
    }
    return worst;
}
int64_t tile_mode_max_blocks(const fa::FwdParams& p, bool causal, int bn, int grid, bool alt) {
    if (!causal) return bn == 64 ? tile_mode_max_blocks_t<false, 64, false>(p, grid)
                                 : tile_mode_max_blocks_t<false, 128, false>(p, grid);
    if (bn == 64) return alt ? tile_mode_max_blocks_t<true, 64, true>(p, grid)
                             : tile_mode_max_blocks_t<true, 64, false>(p, grid);
    return alt ? tile_mode_max_blocks_t<true, 128, true>(p, grid) : tile_mode_max_blocks_t<true, 128, false>(p, grid);
}

// Heads per group of a head-grouped work order: as many as keep the group's
// data (bytes_per_unit per key/value head, shared by `group` consecutive query
// heads) within a third of L2, but enough that a group holds at least four
// rounds of work (units_per_head units per head, `sms` CTAs), so that its
// heaviest-first order still balances the CTAs.
int causal_head_group(int heads, int group, int64_t kv_head_bytes, int l2_bytes, int64_t units_per_head, int sms) {
    const int64_t budget = std::max<int64_t>((int64_t)l2_bytes / 3, 1);
    const int64_t kv_heads = std::max<int64_t>(1, budget / std::max<int64_t>(kv_head_bytes, 1));
    const int64_t min_heads = cdiv(4 * (int64_t)sms, std::max<int64_t>(units_per_head, 1));
    return (int)std::min<int64_t>(std::max(kv_heads * group, min_heads), heads);
}

// Whether the causal tile rounds alternate direction.  On paper it always
// balances the CTAs at least as well, but measured on GB300 it was faster
// only with long tiles: +11 % at N = 2048 D = 256 (17 key blocks a tile on
// average), +5 % at N = 8192 D = 128 (32), flat at N = 2048 D = 128 (8.5),
// and 6-8 % slower at N = 1024 (4.5 blocks: 64 and 1024 heads, D 64 and 128).
bool causal_alternates(const fa::FwdParams& p, int bn) {
    const int64_t blocks = head_blocks(p, true, bn);  // key blocks of one head's tiles
    return blocks >= 16 * (int64_t)p.Tq;
}

// Cutting key ranges costs a partial write per cut tile, a merge launch and
// shorter pipelines, measured on GB300 at about the time of 2048 keys of one
// tile; it pays when whole tiles would leave the busiest CTA that much more
// work than an even cut.  Many tiles per CTA are balanced already.
constexpr int64_t kSplitGainKeys = 2048;
bool split_pays(const fa::FwdParams& p, bool causal, int bn, int sms, bool alt) {
    if ((int64_t)p.ntiles >= 16 * (int64_t)sms) return false;
    const int tile_grid = std::min(p.ntiles, sms);
    const int64_t tile_max = tile_mode_max_blocks(p, causal, bn, tile_grid, alt);
    const int64_t split_max = cdiv(p.total_blocks, std::min<int64_t>(p.total_blocks, sms));
    return (tile_max - split_max) * bn > kSplitGainKeys;
}

cudaError_t launch_for(int D, const fa::LaunchArgs& a, bool causal, bool bf16, int variant) {
    switch (D) {
        case 16: return fa::launch_d16(a, causal, bf16, variant);
        case 32: return fa::launch_d32(a, causal, bf16, variant);
        case 64: return fa::launch_d64(a, causal, bf16, variant);
        case 128: return fa::launch_d128(a, causal, bf16, variant);
        default: return fa::launch_d256(a, causal, bf16, variant);
    }
}

cudaError_t launch_chain_for(int D, const fa::LaunchArgs& a, bool causal, bool bf16, bool alt) {
    switch (D) {
        case 16: return fa::launch_chain_d16(a, causal, bf16, alt);
        case 32: return fa::launch_chain_d32(a, causal, bf16, alt);
        case 64: return fa::launch_chain_d64(a, causal, bf16, alt);
        default: return fa::launch_chain_d128(a, causal, bf16, alt);
    }
}

// Whole-tile launches may run the two-softmax-chain kernel
// (fa_fwd_chain_kernel: two warpgroups take the key blocks in turn, each with
// a whole row of scores per thread) for head dims up to 128; D = 256 (256
// score columns would not fit a thread's registers) and the split schedule
// run the one-chain kernel.  Measured on GB300 (same tiles, same order):
// where the softmax sets the pace -- head dims up to 64 -- with long tiles
// (at least 16 key blocks a tile on average) two chains were 9-17 % faster
// (Z8 H16 N2048 non-causal, D 16/32/64); with short tiles (N = 1024, or
// causal at N = 2048: 4.5-8.5 blocks) 1-25 % slower, since the blocks of a
// tile then pass through a chain of one warpgroup instead of four; and at
// D = 128, where the tensor core and its shared-memory operand traffic set
// the pace, 3-25 % slower.  fa_debug_force_chains overrides the choice.
bool chain_kernel_applies(const fa::FwdParams& p, int D, bool causal, bool split) {
    if (split || D > 128) return false;
    const int force = g_force_chains.load();
    if (force != 0) return force == 1;
    return D <= 64 && head_blocks(p, causal, 128) >= 16 * (int64_t)p.Tq;
}

// Whole-tile launches at D = 128 can run the CTA-pair kernel
// (fa_fwd_pair_kernel: a cluster of two CTAs takes two query tiles that see
// the same key blocks and multiplies each key block once for both, M = 256,
// each SM holding half of every K and V block), with the two softmax chains
// of fa_fwd_chain_kernel on each SM.  It cuts the shared-memory traffic of a
// key block per SM from ~160 KB to ~96 KB, which bounds the one-SM kernels
// at D = 128; measured on GB300 the bound then moves to the two chains'
// softmax (~1.36 us per chain and block), and the pair kernel runs level
// with the one-SM kernel on long tiles (the 32K causal GQA workload 1495 vs
// 1495 TFLOP/s, N = 8192 0.99x) and slower on short ones (Z8 H16 N2048
// causal 0.78x).  So it runs only when fa_debug_force_pair asks for it.
bool pair_kernel_applies(const fa::FwdParams& p, int D, bool causal, bool split) {
    (void)p;
    (void)causal;
    if (split || D != 128) return false;
    return g_force_pair.load() == 1;
}

// The pair kernel's units (fa::FwdParams::pair*): head pairs when the GQA
// group is even (both heads see the same K/V and key blocks), else pairs of
// adjacent query blocks of one head.
void set_pair_units(fa::FwdParams& p, int D, bool causal, int l2_bytes, int clusters) {
    p.pair = p.group % 2 == 0 ? 1 : 2;
    p.pair_heads = p.pair == 1 ? p.Z * p.Hq / 2 : p.Z * p.Hq;
    p.pair_tq = p.pair == 1 ? p.Tq : (p.Tq + 1) / 2;
    p.pair_units = (int)((int64_t)p.pair_heads * p.pair_tq);
    const int per_kv = p.pair == 1 ? p.group / 2 : p.group;  // virtual heads sharing a K/V head
    p.pair_head_group = causal ? causal_head_group(p.pair_heads, per_kv, (int64_t)p.Nkv * D * 4, l2_bytes,
                                                   p.pair_tq, std::max(clusters, 1))
                               : 1;
}

// Key blocks of the busiest cluster of the pair kernel with `clusters`
// clusters (host mirror of PairSched: unit order, alternating rounds, each
// unit's key blocks).
template <bool CAUSAL>
int64_t pair_max_blocks_t(const fa::FwdParams& p, bool alt, int clusters) {
    using S = fa::Sched<CAUSAL, 128>;
    int64_t worst = 0;
    for (int c = 0; c < clusters; ++c) {
        int64_t sum = 0;
        for (int64_t pos = c;; pos += clusters) {
            int64_t t = pos;
            if (CAUSAL && alt) {
                const int64_t round = pos / clusters;
                if (round & 1) t = 2 * round * clusters + clusters - 1 - pos;
            }
            if (t >= p.pair_units) break;
            int vmb;
            if (CAUSAL) {
                const int64_t G = p.pair_head_group, tq = p.pair_tq;
                const int64_t g0 = t / (G * tq) * G;
                const int64_t gc = std::min<int64_t>(G, p.pair_heads - g0);
                vmb = (int)(tq - 1 - (t - g0 * tq) / gc);
            } else {
                vmb = (int)(t % p.pair_tq);
            }
            sum += p.pair == 1 ? S::tile_nkv(vmb, p) : S::tile_nkv(std::min(2 * vmb + 1, p.Tq - 1), p);
        }
        worst = std::max(worst, sum);
    }
    return worst;
}

// The schedule of a forward launch whose sizes are in p (Z .. ntiles):
// causal head groups and alternating rounds for whole tiles, and whether key
// ranges are cut across CTAs (only where the caller allows it: the cut needs
// a workspace).  Shared by the launch and the host-only fa_fwd_schedule.
struct SchedChoice {
    int grid = 0;
    bool split = false;
    bool alt = false;
    bool chains = false;  // the two-softmax-chain kernel (same tiles and order as the one-chain kernel)
    bool pair = false;    // the CTA-pair kernel (grid and order set by set_pair_units at launch)
};
SchedChoice choose_schedule(fa::FwdParams& p, int D, bool causal, int bn, int sms, int l2_bytes, bool split_allowed) {
    SchedChoice c;
    p.head_group = causal_head_group(p.Z * p.Hq, p.group, (int64_t)p.Nkv * D * 4, l2_bytes, p.Tq, sms);
    // the order whole tiles would run in: causal rounds alternate for long tiles
    c.alt = causal && causal_alternates(p, bn);
    c.grid = std::min(p.ntiles, sms);
    if (split_allowed) {
        p.head_blocks = head_blocks(p, causal, bn);
        p.total_blocks = (int64_t)p.Z * p.Hq * p.head_blocks;
        const int force = g_force_split.load();
        if (force == 1 || (force == 0 && split_pays(p, causal, bn, sms, c.alt))) {
            c.split = true;
            c.grid = (int)std::min<int64_t>(p.total_blocks, sms);
        }
    }
    c.chains = chain_kernel_applies(p, D, causal, c.split);
    c.pair = pair_kernel_applies(p, D, causal, c.split);
    return c;
}

// GQA packing.  Without a causal mask a query row's result does not depend on
// its position, so the g query heads that share a key/value head can be run
// as one head of g * Nq rows against that K/V: each key block is then loaded
// and multiplied once per group instead of once per query head.  Done when
// the rows of a group are short (Nq < 128: decode-like and few-query shapes)
// and the layout allows the view: a query head's rows follow the previous
// head's (h-stride = Nq * n-stride), batches follow whole head sets, and K/V
// heads are evenly strided within a batch.  The lse layout (Z, Hq, Nq)
// contiguous is the same memory as (Z * Hkv, 1, g * Nq).
bool gqa_pack_view(int Z, int Hq, int Hkv, int Nq, int causal, const fa_strides* sq, const fa_strides* sk,
                   const fa_strides* sv, const fa_strides* so, fa_strides* pq, fa_strides* pk, fa_strides* pv,
                   fa_strides* po) {
    const int g = Hkv > 0 ? Hq / Hkv : 0;
    if (causal || g < 2 || Nq >= fa::BM || Nq < 1) return false;
    if (!sq || !sk || !sv || !so) return false;
    auto rows_follow = [&](const fa_strides* s) {
        return s->d == 1 && s->h == (int64_t)Nq * s->n && (Z <= 1 || s->b == (int64_t)Hq * s->h);
    };
    auto kv_even = [&](const fa_strides* s) { return s->d == 1 && (Z <= 1 || s->b == (int64_t)Hkv * s->h); };
    if (!rows_follow(sq) || !rows_follow(so) || !kv_even(sk) || !kv_even(sv)) return false;
    // batch index z * Hkv + hk; one head; rows gi * Nq + n
    *pq = fa_strides{(int64_t)g * sq->h, 0, sq->n, 1};
    *po = fa_strides{(int64_t)g * so->h, 0, so->n, 1};
    *pk = fa_strides{sk->h, 0, sk->n, 1};
    *pv = fa_strides{sv->h, 0, sv->n, 1};
    return true;
}

fa_status fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, int Z, int Hq, int Hkv, int Nq,
                   int Nkv, int D, const fa_strides* sq, const fa_strides* sk, const fa_strides* sv,
                   const fa_strides* so, float scale, int causal, fa_dtype dtype, cudaStream_t stream, bool split,
                   void* workspace, size_t workspace_bytes) {
    fa_status st = check_shape(Z, Hq, Hkv, Nq, Nkv, D, causal);
    if (st != FA_OK) return st;
    fa_strides pq, pk, pv, po;
    if ((int64_t)Z * Hq * Nq > 0 && gqa_pack_view(Z, Hq, Hkv, Nq, causal, sq, sk, sv, so, &pq, &pk, &pv, &po)) {
        // the same problem seen as Z * Hkv heads of g * Nq query rows (validated as such)
        return fwd_impl(q, k, v, o, lse, Z * Hkv, 1, 1, Nq * (Hq / Hkv), Nkv, D, &pq, &pk, &pv, &po, scale, causal,
                        dtype, stream, split, workspace, workspace_bytes);
    }
    if (dtype != FA_DTYPE_F16 && dtype != FA_DTYPE_BF16) return FA_ERR_UNSUPPORTED;
    float c = 0.f;
    int negate = 0;
    if (!fwd_scale(scale, &c, &negate)) return FA_ERR_INVALID_ARG;
    if ((int64_t)Z * Hq * Nq == 0) return FA_OK;
    if ((st = check_tensor(q, sq, Z, Hq, Nq)) != FA_OK) return st;
    if ((st = check_tensor(k, sk, Z, Hkv, Nkv)) != FA_OK) return st;
    if ((st = check_tensor(v, sv, Z, Hkv, Nkv)) != FA_OK) return st;
    if ((st = check_tensor(o, so, Z, Hq, Nq)) != FA_OK) return st;
    if (lse != nullptr && reinterpret_cast<uintptr_t>(lse) % 4 != 0) return FA_ERR_ALIGNMENT;
    if (split && (workspace == nullptr || reinterpret_cast<uintptr_t>(workspace) % 256 != 0))
        return FA_ERR_WORKSPACE;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
    LaunchInfo li;
    if (device_info(dev, &li) != cudaSuccess) return FA_ERR_CUDA;
    const LaunchInfo* info = &li;

    const int bn = fa::block_n_for(D);
    fa::LaunchArgs a;
    fa::FwdParams& p = a.params;
    p = fa::FwdParams{};
    p.o = o;
    p.lse = lse;
    p.so_z = so->b;
    p.so_h = so->h;
    p.so_n = so->n;
    p.Z = Z;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.Nq = Nq;
    p.Nkv = Nkv;
    p.group = Hq / Hkv;
    p.Tq = (int)cdiv(Nq, fa::BM);
    p.Tk = (int)cdiv(Nkv, bn);
    p.ntiles = (int)((int64_t)Z * Hq * p.Tq);
    p.scale_log2 = c;
    p.negate_s = negate;
    p.status = info->status;
    p.wait_limit_ns = wait_limit_ns();
    p.inject_stall = g_inject_stall.load();
    // split: one equal range of (tile, key block) pairs per SM (every range
    // non-empty), when that beats whole tiles for this shape
    if (split && workspace_bytes < split_workspace_bytes(D, info->sms)) return FA_ERR_WORKSPACE;
    const SchedChoice choice = choose_schedule(p, D, causal != 0, bn, info->sms, info->l2_bytes, split);
    const bool alt = choice.alt;
    a.grid = choice.grid;
    if (choice.split) {
        p.split = 1;
        p.slot_floats = split_slot_floats(D);
        p.scratch = static_cast<float*>(workspace);
    }

    CUtensorMap mq, mk, mv, mo;
    if (make_map(&mq, q, dtype, D, Nq, Hq, Z, sq, fa::BM) != CUDA_SUCCESS) return FA_ERR_CUDA;
    if (make_map(&mk, k, dtype, D, Nkv, Hkv, Z, sk, bn) != CUDA_SUCCESS) return FA_ERR_CUDA;
    if (make_map(&mv, v, dtype, D, Nkv, Hkv, Z, sv, bn) != CUDA_SUCCESS) return FA_ERR_CUDA;
    if (make_map(&mo, o, dtype, D, Nq, Hq, Z, so, 32) != CUDA_SUCCESS) return FA_ERR_CUDA;
    a.tmQ = &mq;
    a.tmK = &mk;
    a.tmV = &mv;
    a.tmO = &mo;
    a.stream = stream;

    if (choice.pair) {
        // clusters of two CTAs, as many as can be resident (pairs of SMs in
        // one GPC), each CTA loading half of every key block
        const int limit = fa::pair_cluster_limit_d128();
        if (limit > 0) {
            set_pair_units(p, D, causal != 0, info->l2_bytes, limit);
            a.grid = 2 * std::min(p.pair_units, limit);
            CUtensorMap mk_half;
            if (make_map(&mk_half, k, dtype, D, Nkv, Hkv, Z, sk, bn / 2) != CUDA_SUCCESS) return FA_ERR_CUDA;
            a.tmK = &mk_half;
            const cudaError_t err = fa::launch_pair_d128(a, causal != 0, dtype == FA_DTYPE_BF16, alt);
            return err == cudaSuccess ? FA_OK : cuda_fail("forward launch", err);
        }
        p.pair = 0;  // no cluster of two fits this device: the one-SM kernels
    }
    if (choice.chains) {
        const cudaError_t err = launch_chain_for(D, a, causal != 0, dtype == FA_DTYPE_BF16, alt);
        return err == cudaSuccess ? FA_OK : cuda_fail("forward launch", err);
    }
    // kernel variant 4: the plain kernel with alternating causal rounds (tile mode only)
    const cudaError_t err = launch_for(D, a, causal != 0, dtype == FA_DTYPE_BF16, alt && !p.split ? 4 : 0);
    return err == cudaSuccess ? FA_OK : cuda_fail("forward launch", err);
}

// The variant forward (fa_fwd_ex): window, ALiBi and packed variable-length
// batches, whole tiles only.
fa_status fwd_ex_impl(const void* q, const void* k, const void* v, void* o, float* lse, int Z, int Hq, int Hkv,
                      int Nq, int Nkv, int D, const fa_strides* sq, const fa_strides* sk, const fa_strides* sv,
                      const fa_strides* so, float scale, int causal, fa_dtype dtype, const fa_fwd_options* opt,
                      cudaStream_t stream) {
    fa_status st = check_shape(Z, Hq, Hkv, Nq, Nkv, D, causal);
    if (st != FA_OK) return st;
    if (dtype != FA_DTYPE_F16 && dtype != FA_DTYPE_BF16) return FA_ERR_UNSUPPORTED;
    float c = 0.f;
    int negate = 0;
    if (!fwd_scale(scale, &c, &negate)) return FA_ERR_INVALID_ARG;
    if (opt->window_left < -1 || opt->window_right < -1) return FA_ERR_INVALID_ARG;
    const bool varlen = opt->cu_seqlens_q != nullptr || opt->cu_seqlens_k != nullptr;
    if (varlen && (opt->cu_seqlens_q == nullptr || opt->cu_seqlens_k == nullptr || opt->max_seqlen_q < 0))
        return FA_ERR_INVALID_ARG;
    if (varlen && (reinterpret_cast<uintptr_t>(opt->cu_seqlens_q) % 4 != 0 ||
                   reinterpret_cast<uintptr_t>(opt->cu_seqlens_k) % 4 != 0))
        return FA_ERR_ALIGNMENT;
    if (opt->alibi_slopes != nullptr && reinterpret_cast<uintptr_t>(opt->alibi_slopes) % 4 != 0)
        return FA_ERR_ALIGNMENT;
    // Without a sequence table, a bias or a window side shorter than every
    // query-key distance, the call is fa_fwd: it takes the plain kernel (the
    // variant kernel's per-block window and sequence checks cost ~15 %).
    const int64_t reach_all = (int64_t)Nq + Nkv;
    const auto open = [&](int w) { return w < 0 || (int64_t)w > reach_all; };
    if (!varlen && opt->alibi_slopes == nullptr && open(opt->window_left) && open(opt->window_right))
        return fwd_impl(q, k, v, o, lse, Z, Hq, Hkv, Nq, Nkv, D, sq, sk, sv, so, scale, causal, dtype, stream, false,
                        nullptr, 0);
    const int tq = (int)cdiv(varlen ? opt->max_seqlen_q : Nq, fa::BM);
    if ((int64_t)Z * Hq * tq > INT32_MAX) return FA_ERR_UNSUPPORTED;
    if ((varlen ? (int64_t)Nq : (int64_t)Z * Hq * Nq) == 0 || (int64_t)Z * Hq * tq == 0) return FA_OK;
    // packed tensors of a variable-length batch have one batch entry
    const int nb = varlen ? 1 : Z;
    if ((st = check_tensor(q, sq, nb, Hq, Nq)) != FA_OK) return st;
    if ((st = check_tensor(k, sk, nb, Hkv, Nkv)) != FA_OK) return st;
    if ((st = check_tensor(v, sv, nb, Hkv, Nkv)) != FA_OK) return st;
    if ((st = check_tensor(o, so, nb, Hq, Nq)) != FA_OK) return st;
    if (lse != nullptr && reinterpret_cast<uintptr_t>(lse) % 4 != 0) return FA_ERR_ALIGNMENT;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
    LaunchInfo li;
    if (device_info(dev, &li) != cudaSuccess) return FA_ERR_CUDA;
    const LaunchInfo* info = &li;

    const int bn = fa::block_n_for(D);
    fa::LaunchArgs a;
    fa::FwdParams& p = a.params;
    p = fa::FwdParams{};
    p.o = o;
    p.lse = lse;
    p.so_z = so->b;
    p.so_h = so->h;
    p.so_n = so->n;
    p.Z = Z;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.Nq = Nq;
    p.Nkv = Nkv;
    p.group = Hq / Hkv;
    p.Tq = tq;
    p.Tk = (int)cdiv(Nkv, bn);
    p.ntiles = (int)((int64_t)Z * Hq * tq);
    // a packed sequence's keys: about Nkv / Z of the packed rows
    p.head_group = causal_head_group(Z * Hq, p.group, (int64_t)(varlen ? std::max(1, Nkv / Z) : Nkv) * D * 4,
                                     info->l2_bytes, p.Tq, info->sms);
    p.scale_log2 = c;
    p.negate_s = negate;
    p.status = info->status;
    p.wait_limit_ns = wait_limit_ns();
    p.inject_stall = g_inject_stall.load();
    // a side longer than every distance between a query and a key is open
    // (and i +- window can then not overflow on the device)
    const int64_t reach = (int64_t)Nq + Nkv;
    p.win_left = opt->window_left > reach ? -1 : opt->window_left;
    p.win_right = opt->window_right > reach ? -1 : opt->window_right;
    p.alibi = opt->alibi_slopes;
    p.cu_q = varlen ? opt->cu_seqlens_q : nullptr;
    p.cu_k = varlen ? opt->cu_seqlens_k : nullptr;
    a.grid = std::min(p.ntiles, info->sms);

    CUtensorMap mq, mk, mv, mo;
    if (make_map(&mq, q, dtype, D, Nq, Hq, nb, sq, fa::BM) != CUDA_SUCCESS) return FA_ERR_CUDA;
    if (make_map(&mk, k, dtype, D, Nkv, Hkv, nb, sk, bn) != CUDA_SUCCESS) return FA_ERR_CUDA;
    if (make_map(&mv, v, dtype, D, Nkv, Hkv, nb, sv, bn) != CUDA_SUCCESS) return FA_ERR_CUDA;
    if (make_map(&mo, o, dtype, D, Nq, Hq, nb, so, 32) != CUDA_SUCCESS) return FA_ERR_CUDA;
    a.tmQ = &mq;
    a.tmK = &mk;
    a.tmV = &mv;
    a.tmO = &mo;
    a.stream = stream;
    const cudaError_t err = launch_for(D, a, causal != 0, dtype == FA_DTYPE_BF16, p.alibi != nullptr ? 2 : 1);
    return err == cudaSuccess ? FA_OK : cuda_fail("variant forward launch", err);
}

}  // namespace

extern "C" {

const char* fa_status_string(fa_status s) {
    switch (s) {
        case FA_OK: return "FA_OK";
        case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
        case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
        case FA_ERR_ALIGNMENT: return "FA_ERR_ALIGNMENT";
        case FA_ERR_CUDA: return "FA_ERR_CUDA";
        case FA_ERR_DEVICE_TIMEOUT: return "FA_ERR_DEVICE_TIMEOUT";
        case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE";
        case FA_ERR_DEVICE_CHECK: return "FA_ERR_DEVICE_CHECK";
    }
    return "FA_ERR_UNKNOWN";
}

fa_status fa_fwd_plan(int Z, int Hq, int Hkv, int Nq, int Nkv, int D, int causal, int num_sms, int64_t* tiles,
                      int64_t* kv_blocks, int* block_n, int* grid, int* smem_bytes) {
    const fa_status st = check_shape(Z, Hq, Hkv, Nq, Nkv, D, causal);
    if (st != FA_OK) return st;
    const int bn = fa::block_n_for(D);
    const int64_t tq = cdiv(Nq, fa::BM), tk = cdiv(Nkv, bn);
    const int64_t nt = (int64_t)Z * Hq * tq;
    int64_t pairs = 0;
    if (causal) {
        for (int64_t mb = 0; mb < tq; ++mb) {  // same bound as the kernel's Sched::tile_nkv
            const int64_t last_row = std::min<int64_t>(mb * fa::BM + fa::BM, Nq) - 1;
            pairs += std::min<int64_t>(tk, last_row / bn + 1);
        }
        pairs *= (int64_t)Z * Hq;
    } else {
        pairs = nt * tk;
    }
    if (tiles) *tiles = nt;
    if (kv_blocks) *kv_blocks = pairs;
    if (block_n) *block_n = bn;
    if (grid) *grid = (int)(num_sms > 0 ? std::min<int64_t>(nt, num_sms) : nt);
    if (smem_bytes) *smem_bytes = fa::smem_bytes_for(D);
    return FA_OK;
}

fa_status fa_fwd_schedule(int Z, int Hq, int Hkv, int Nq, int Nkv, int D, int causal, int splitkv, int num_sms,
                          int64_t l2_bytes, fa_fwd_schedule_info* out) {
    if (out == nullptr || num_sms < 1 || l2_bytes < 1) return FA_ERR_INVALID_ARG;
    const fa_status st = check_shape(Z, Hq, Hkv, Nq, Nkv, D, causal);
    if (st != FA_OK) return st;
    *out = fa_fwd_schedule_info{};
    // contiguous BNSD tensors, seen as the launch sees them (GQA packing included)
    const fa_strides sq{(int64_t)Hq * Nq * D, (int64_t)Nq * D, D, 1}, sk{(int64_t)Hkv * Nkv * D, (int64_t)Nkv * D, D, 1};
    fa_strides pq, pk, pv, po;
    if ((int64_t)Z * Hq * Nq > 0 && gqa_pack_view(Z, Hq, Hkv, Nq, causal, &sq, &sk, &sk, &sq, &pq, &pk, &pv, &po)) {
        Nq *= Hq / Hkv;
        Z *= Hkv;
        Hq = Hkv = 1;
        out->gqa_packed = 1;
    }
    const int bn = fa::block_n_for(D);
    fa::FwdParams p{};
    p.Z = Z;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.Nq = Nq;
    p.Nkv = Nkv;
    p.group = Hq / Hkv;
    p.Tq = (int)cdiv(Nq, fa::BM);
    p.Tk = (int)cdiv(Nkv, bn);
    p.ntiles = (int)((int64_t)Z * Hq * p.Tq);
    if (p.ntiles == 0) return FA_OK;
    const int l2 = (int)std::min<int64_t>(l2_bytes, INT32_MAX);
    const SchedChoice c = choose_schedule(p, D, causal != 0, bn, num_sms, l2, splitkv != 0);
    out->grid = c.grid;
    out->split = c.split ? 1 : 0;
    out->head_group = p.head_group;
    out->alternate = c.alt && !c.split ? 1 : 0;
    out->tiles = p.ntiles;
    out->kv_blocks = (int64_t)Z * Hq * head_blocks(p, causal != 0, bn);
    out->softmax_chains = c.chains || c.pair ? 2 : 1;
    out->busiest_blocks = c.split ? cdiv(out->kv_blocks, c.grid)
                                  : tile_mode_max_blocks(p, causal != 0, bn, c.grid, c.alt);
    out->cta_pairs = c.pair ? 1 : 0;
    if (c.pair) {
        // clusters of two: as many as the SMs hold (at launch: as the device can hold at once)
        const int clusters = std::max(1, num_sms / 2);
        set_pair_units(p, D, causal != 0, l2, clusters);
        const int used = std::min(p.pair_units, clusters);
        out->grid = 2 * used;
        out->head_group = causal ? p.pair_head_group : p.head_group;
        out->busiest_blocks = causal ? pair_max_blocks_t<true>(p, c.alt, used) : pair_max_blocks_t<false>(p, false, used);
    }
    return FA_OK;
}

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int Z, int Hq, int Hkv, int Nq,
                 int Nkv, int D, const fa_strides* sq, const fa_strides* sk, const fa_strides* sv,
                 const fa_strides* so, float scale, int causal, fa_dtype dtype, cudaStream_t stream) {
    return fwd_impl(q, k, v, o, lse, Z, Hq, Hkv, Nq, Nkv, D, sq, sk, sv, so, scale, causal, dtype, stream, false,
                    nullptr, 0);
}

fa_status fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int Z, int Hq, int Hkv,
                         int Nq, int Nkv, int D, const fa_strides* sq, const fa_strides* sk, const fa_strides* sv,
                         const fa_strides* so, float scale, int causal, fa_dtype dtype, void* workspace,
                         size_t workspace_bytes, cudaStream_t stream) {
    return fwd_impl(q, k, v, o, lse, Z, Hq, Hkv, Nq, Nkv, D, sq, sk, sv, so, scale, causal, dtype, stream, true,
                    workspace, workspace_bytes);
}

fa_status fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int Z, int Hq, int Hkv, int Nq,
                    int Nkv, int D, const fa_strides* sq, const fa_strides* sk, const fa_strides* sv,
                    const fa_strides* so, float scale, int causal, fa_dtype dtype, const fa_fwd_options* options,
                    cudaStream_t stream) {
    static const fa_fwd_options none = {-1, -1, nullptr, nullptr, nullptr, 0, 0};
    return fwd_ex_impl(q, k, v, o, lse, Z, Hq, Hkv, Nq, Nkv, D, sq, sk, sv, so, scale, causal, dtype,
                       options ? options : &none, stream);
}

fa_status fa_bwd_workspace_size(int Z, int Hq, int Nq, int D, size_t* bytes) {
    if (bytes == nullptr || Z < 0 || Hq < 0 || Nq < 0) return FA_ERR_INVALID_ARG;
    if (!supported_head_dim(D)) return FA_ERR_UNSUPPORTED;
    *bytes = bwd_workspace_bytes(Z, Hq, Nq, D);
    return FA_OK;
}

// The backward, plain (variant 0) or with the options of fa_bwd_ex (variant
// 1: window; 2: window and ALiBi; 3: packed variable-length sequences with a
// window and ALiBi; 4: packed sequences with a window).  With a sequence table (cu_q, cu_k) Z
// counts sequences, the tensors have one batch entry, Nq / Nkv are the packed
// row totals, max_q / max_k bound the sequences' lengths and lse is (Hq, Nq).
static fa_status bwd_impl(const void* q, const void* k, const void* v, const void* o, const float* lse,
                          const void* dO, void* dq, void* dk, void* dv, int Z, int Hq, int Hkv, int Nq, int Nkv, int D,
                          const fa_strides* sq, const fa_strides* sk, const fa_strides* sv, const fa_strides* so,
                          const fa_strides* sdo, const fa_strides* sdq, const fa_strides* sdk,
                          const fa_strides* sdv, float scale, int causal, fa_dtype dtype, void* workspace,
                          size_t workspace_bytes, cudaStream_t stream, int variant, int win_left, int win_right,
                          const float* alibi, const int32_t* cu_q = nullptr, const int32_t* cu_k = nullptr,
                          int max_q = 0, int max_k = 0) {
    fa_status st = check_shape(Z, Hq, Hkv, Nq, Nkv, D, causal);
    if (st != FA_OK) return st;
    if (!supported_head_dim(D)) return FA_ERR_UNSUPPORTED;
    if (dtype != FA_DTYPE_F16 && dtype != FA_DTYPE_BF16) return FA_ERR_UNSUPPORTED;
    // any finite scale whose log2 factor is finite in fp32: the backward
    // builds P = 2^(s·scale·log2e − lse·log2e) from the saved lse (no row
    // maximum) and masks after scaling, so the sign and zero need no care
    if (!std::isfinite(scale) || !(std::fabs((double)scale) * 1.4426950408889634 <= (double)FLT_MAX))
        return FA_ERR_INVALID_ARG;
    if ((int64_t)Z * Hkv * Nkv == 0) return FA_OK;
    if (Nq == 0) return FA_ERR_INVALID_ARG;  // gradients of an empty query set: nothing to differentiate
    // packed tensors of a variable-length batch have one batch entry
    const bool varlen = cu_q != nullptr;
    const int nb = varlen ? 1 : Z;
    const int rows_q = varlen ? max_q : Nq;                    // query rows per (sequence, head) computed
    const int rows_k = varlen ? (max_k > 0 ? max_k : Nkv) : Nkv;  // key rows per (sequence, head)
    if ((st = check_tensor(q, sq, nb, Hq, Nq)) != FA_OK) return st;
    if ((st = check_tensor(k, sk, nb, Hkv, Nkv)) != FA_OK) return st;
    if ((st = check_tensor(v, sv, nb, Hkv, Nkv)) != FA_OK) return st;
    if ((st = check_tensor(o, so, nb, Hq, Nq)) != FA_OK) return st;
    if ((st = check_tensor(dO, sdo, nb, Hq, Nq)) != FA_OK) return st;
    if ((st = check_tensor(dq, sdq, nb, Hq, Nq)) != FA_OK) return st;
    if ((st = check_tensor(dk, sdk, nb, Hkv, Nkv)) != FA_OK) return st;
    if ((st = check_tensor(dv, sdv, nb, Hkv, Nkv)) != FA_OK) return st;
    if (lse == nullptr) return FA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(lse) % 4 != 0) return FA_ERR_ALIGNMENT;
    if (workspace == nullptr || reinterpret_cast<uintptr_t>(workspace) % 256 != 0 ||
        workspace_bytes < bwd_workspace_bytes(Z, Hq, rows_q, D))
        return FA_ERR_WORKSPACE;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
    LaunchInfo li;
    if (device_info(dev, &li) != cudaSuccess) return FA_ERR_CUDA;
    const LaunchInfo* info = &li;

    fa::BwdLaunchArgs a;
    fa::BwdParams& p = a.params;
    p = fa::BwdParams{};
    p.o = o;
    p.lse = lse;
    p.dO = dO;
    p.dq = dq;
    p.dk = dk;
    p.dv = dv;
    p.so_z = so->b; p.so_h = so->h; p.so_n = so->n;
    p.sdo_z = sdo->b; p.sdo_h = sdo->h; p.sdo_n = sdo->n;
    p.sdq_z = sdq->b; p.sdq_h = sdq->h; p.sdq_n = sdq->n;
    p.sdk_z = sdk->b; p.sdk_h = sdk->h; p.sdk_n = sdk->n;
    p.sdv_z = sdv->b; p.sdv_h = sdv->h; p.sdv_n = sdv->n;
    p.Z = Z;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.Nq = Nq;
    p.Nkv = Nkv;
    p.group = Hq / Hkv;
    p.Tq = (int)cdiv(rows_q, 128);
    p.Tk = (int)cdiv(rows_k, 128);
    const int64_t units = (int64_t)Z * Hkv * p.Tk, units_q = (int64_t)Z * Hq * p.Tq;
    if (units > INT32_MAX || units_q > INT32_MAX) return FA_ERR_UNSUPPORTED;
    p.nunits = (int)units;
    p.nunits_q = (int)units_q;
    // a dK/dV group reads the Q and dO rows of its kv heads' query heads; a
    // causal dQ group the K and V of its query heads (shared within a GQA
    // group); a packed sequence holds about a Z-th of the packed rows
    const int64_t seq_q = varlen ? std::max(1, Nq / std::max(1, Z)) : Nq;
    const int64_t seq_k = varlen ? std::max(1, Nkv / std::max(1, Z)) : Nkv;
    p.kv_head_group = causal_head_group(Z * Hkv, 1, (int64_t)p.group * seq_q * D * 4, info->l2_bytes, p.Tk, info->sms);
    // D = 256, non-causal: groups of about one round of CTAs, so every key
    // block of a head runs at once and its Q and dO (re-read by both passes
    // of every step) stay in L2.  Measured on GB300 (Z8 H16 N2048): +6.0 %;
    // causal -10 % (its heaviest-first order needs the larger groups), D = 64
    // -2 %, D = 128 level.
    if (!causal && D == 256)
        p.kv_head_group = (int)std::min<int64_t>(Z * Hkv, std::max<int64_t>(1, cdiv(info->sms, p.Tk)));
    p.q_head_group = causal_head_group(Z * Hq, p.group, seq_k * D * 4, info->l2_bytes, p.Tq, info->sms);
    p.scale = scale;
    p.scale_log2 = (float)((double)scale * 1.4426950408889634);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const size_t row_bytes = align256((size_t)Z * Hq * p.Tq * 128 * 4);
    p.lse2 = reinterpret_cast<float*>(ws);
    p.delta = reinterpret_cast<float*>(ws + row_bytes);
    p.status = info->status;
    p.wait_limit_ns = wait_limit_ns();
    p.inject_stall = g_inject_stall.load();
    p.win_left = win_left;
    p.win_right = win_right;
    p.alibi = alibi;
    p.cu_q = cu_q;
    p.cu_k = varlen ? cu_k : nullptr;

    // operand loads: 128-row boxes; at D = 256 the kernel moves 64-row steps
    // (and its resident 128-row tiles as two boxes)
    CUtensorMap mk, mv, mq, mdo;
    CUresult cr;
    const int box = D == 256 ? 64 : 128;
    if ((cr = make_map(&mk, k, dtype, D, Nkv, Hkv, nb, sk, box)) != CUDA_SUCCESS) return cuda_fail("K tensor map", cr);
    if ((cr = make_map(&mv, v, dtype, D, Nkv, Hkv, nb, sv, box)) != CUDA_SUCCESS) return cuda_fail("V tensor map", cr);
    if ((cr = make_map(&mq, q, dtype, D, Nq, Hq, nb, sq, box)) != CUDA_SUCCESS) return cuda_fail("Q tensor map", cr);
    if ((cr = make_map(&mdo, dO, dtype, D, Nq, Hq, nb, sdo, box)) != CUDA_SUCCESS)
        return cuda_fail("dO tensor map", cr);
    CUtensorMap mdq, mdk, mdv;
    if ((cr = make_map(&mdq, dq, dtype, D, Nq, Hq, nb, sdq, 32)) != CUDA_SUCCESS) return cuda_fail("dQ tensor map", cr);
    if ((cr = make_map(&mdk, dk, dtype, D, Nkv, Hkv, nb, sdk, 32)) != CUDA_SUCCESS) return cuda_fail("dK tensor map", cr);
    if ((cr = make_map(&mdv, dv, dtype, D, Nkv, Hkv, nb, sdv, 32)) != CUDA_SUCCESS) return cuda_fail("dV tensor map", cr);
    a.tmK = &mk;
    a.tmV = &mv;
    a.tmQ = &mq;
    a.tmDO = &mdo;
    a.tmDQ = &mdq;
    a.tmDK = &mdk;
    a.tmDV = &mdv;
    // one CTA per SM (or per unit): dK/dV units from position c, dQ units from grid - 1 - c
    a.grid = (int)std::min<int64_t>(std::max(units, units_q), info->sms);
    const int64_t pre_threads = (int64_t)Z * Hq * p.Tq * 128 * (D / 8);
    a.pre_grid = (int)std::max<int64_t>(1, std::min<int64_t>(cdiv(pre_threads, 256), (int64_t)info->sms * 16));
    a.stream = stream;
    const bool bf16 = dtype == FA_DTYPE_BF16;
    cudaError_t err;
    switch (D) {
        case 16: err = fa::launch_bwd_d16(a, causal != 0, bf16, variant); break;
        case 32: err = fa::launch_bwd_d32(a, causal != 0, bf16, variant); break;
        case 64: err = fa::launch_bwd_d64(a, causal != 0, bf16, variant); break;
        case 128: err = fa::launch_bwd_d128(a, causal != 0, bf16, variant); break;
        default: err = fa::launch_bwd_d256(a, causal != 0, bf16, variant); break;
    }
    return err == cudaSuccess ? FA_OK : cuda_fail("backward launch", err);
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                 void* dq, void* dk, void* dv, int Z, int Hq, int Hkv, int Nq, int Nkv, int D, const fa_strides* sq,
                 const fa_strides* sk, const fa_strides* sv, const fa_strides* so, const fa_strides* sdo,
                 const fa_strides* sdq, const fa_strides* sdk, const fa_strides* sdv, float scale, int causal,
                 fa_dtype dtype, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    return bwd_impl(q, k, v, o, lse, dO, dq, dk, dv, Z, Hq, Hkv, Nq, Nkv, D, sq, sk, sv, so, sdo, sdq, sdk, sdv, scale,
                    causal, dtype, workspace, workspace_bytes, stream, 0, -1, -1, nullptr);
}

fa_status fa_bwd_ex(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                    void* dq, void* dk, void* dv, int Z, int Hq, int Hkv, int Nq, int Nkv, int D,
                    const fa_strides* sq, const fa_strides* sk, const fa_strides* sv, const fa_strides* so,
                    const fa_strides* sdo, const fa_strides* sdq, const fa_strides* sdk, const fa_strides* sdv,
                    float scale, int causal, fa_dtype dtype, const fa_fwd_options* options, void* workspace,
                    size_t workspace_bytes, cudaStream_t stream) {
    const fa_fwd_options none = {-1, -1, nullptr, nullptr, nullptr, 0, 0};
    const fa_fwd_options* opt = options != nullptr ? options : &none;
    if (opt->window_left < -1 || opt->window_right < -1) return FA_ERR_INVALID_ARG;
    const bool varlen = opt->cu_seqlens_q != nullptr || opt->cu_seqlens_k != nullptr;
    if (varlen && (opt->cu_seqlens_q == nullptr || opt->cu_seqlens_k == nullptr || opt->max_seqlen_q < 0 ||
                   opt->max_seqlen_k < 0))
        return FA_ERR_INVALID_ARG;
    if (varlen && (reinterpret_cast<uintptr_t>(opt->cu_seqlens_q) % 4 != 0 ||
                   reinterpret_cast<uintptr_t>(opt->cu_seqlens_k) % 4 != 0))
        return FA_ERR_ALIGNMENT;
    if (opt->alibi_slopes != nullptr && reinterpret_cast<uintptr_t>(opt->alibi_slopes) % 4 != 0)
        return FA_ERR_ALIGNMENT;
    // a window side longer than every query-key distance is open
    const int64_t reach_all = (int64_t)Nq + Nkv;
    const auto open = [&](int w) { return w < 0 || (int64_t)w > reach_all; };
    const int wl = open(opt->window_left) ? -1 : opt->window_left;
    const int wr = open(opt->window_right) ? -1 : opt->window_right;
    const bool alibi = opt->alibi_slopes != nullptr;
    const int variant = varlen ? (alibi ? 3 : 4) : alibi ? 2 : (wl >= 0 || wr >= 0) ? 1 : 0;
    return bwd_impl(q, k, v, o, lse, dO, dq, dk, dv, Z, Hq, Hkv, Nq, Nkv, D, sq, sk, sv, so, sdo, sdq, sdk, sdv, scale,
                    causal, dtype, workspace, workspace_bytes, stream, variant, wl, wr, opt->alibi_slopes,
                    varlen ? opt->cu_seqlens_q : nullptr, varlen ? opt->cu_seqlens_k : nullptr, opt->max_seqlen_q,
                    opt->max_seqlen_k);
}

fa_status fa_fwd_splitkv_workspace_size_for(int D, int num_sms, size_t* bytes) {
    if (bytes == nullptr || num_sms < 1) return FA_ERR_INVALID_ARG;
    if (!supported_head_dim(D)) return FA_ERR_UNSUPPORTED;
    *bytes = split_workspace_bytes(D, num_sms);
    return FA_OK;
}

fa_status fa_fwd_splitkv_workspace_size(int D, size_t* bytes) {
    if (bytes == nullptr) return FA_ERR_INVALID_ARG;
    if (!supported_head_dim(D)) return FA_ERR_UNSUPPORTED;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
    LaunchInfo li;
    if (device_info(dev, &li) != cudaSuccess) return FA_ERR_CUDA;
    const LaunchInfo* info = &li;
    *bytes = split_workspace_bytes(D, info->sms);
    return FA_OK;
}

fa_status fa_lse_merge(int nparts, const void* const* o_parts, const float* const* lse_parts, int Z, int H, int N,
                       int D, const fa_strides* sp, void* o, float* lse, const fa_strides* so, fa_dtype dtype,
                       cudaStream_t stream) {
    if (nparts < 1 || nparts > FA_MERGE_MAX_PARTS || o_parts == nullptr || lse_parts == nullptr)
        return FA_ERR_INVALID_ARG;
    if (Z < 0 || H < 0 || N < 0) return FA_ERR_INVALID_ARG;
    if (!supported_head_dim(D) || (dtype != FA_DTYPE_F16 && dtype != FA_DTYPE_BF16)) return FA_ERR_UNSUPPORTED;
    const int64_t rows = (int64_t)Z * H * N;
    if (rows == 0) return FA_OK;
    fa_status st;
    fa::MergeArgs a{};
    for (int s = 0; s < nparts; ++s) {
        if ((st = check_tensor(o_parts[s], sp, Z, H, N)) != FA_OK) return st;
        if (lse_parts[s] == nullptr) return FA_ERR_INVALID_ARG;
        if (reinterpret_cast<uintptr_t>(lse_parts[s]) % 4 != 0) return FA_ERR_ALIGNMENT;
        a.o[s] = o_parts[s];
        a.lse[s] = lse_parts[s];
    }
    if ((st = check_tensor(o, so, Z, H, N)) != FA_OK) return st;
    if (lse != nullptr && reinterpret_cast<uintptr_t>(lse) % 4 != 0) return FA_ERR_ALIGNMENT;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
    LaunchInfo li;
    if (device_info(dev, &li) != cudaSuccess) return FA_ERR_CUDA;
    const LaunchInfo* info = &li;
    a.nparts = nparts;
    a.H = H;
    a.N = N;
    a.D = D;
    a.rows = rows;
    a.sp_b = sp->b;
    a.sp_h = sp->h;
    a.sp_n = sp->n;
    a.so_b = so->b;
    a.so_h = so->h;
    a.so_n = so->n;
    a.out = o;
    a.out_lse = lse;
    const int64_t items = rows * (D / 8);
    const int grid = (int)std::min<int64_t>(cdiv(items, 256), (int64_t)info->sms * 8);
    return fa::launch_lse_merge(a, dtype == FA_DTYPE_BF16, grid, stream) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_device_status(cudaStream_t stream, uint32_t* detail) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return FA_ERR_CUDA;
    uint32_t word = 0;
    if (cudaMemcpyFromSymbol(&word, g_fa_status, sizeof(word)) != cudaSuccess) return FA_ERR_CUDA;
    if (word != 0) {
        const uint32_t zero = 0;
        if (cudaMemcpyToSymbol(g_fa_status, &zero, sizeof(zero)) != cudaSuccess) return FA_ERR_CUDA;
    }
    if (detail) *detail = word;
    return word == 0 ? FA_OK : (fa_status)(word & 0xFFu);
}

// Test hook (declared in fa.h): the softmax kernels' polynomial exponential
// applied to an array, so that it can be checked against CUDA's exp2f.
namespace {
__global__ void exp2_poly_kernel(const float* __restrict__ x, float* __restrict__ y, int64_t n) {
    const int64_t i = 2 * ((int64_t)blockIdx.x * blockDim.x + threadIdx.x);
    if (i >= n) return;
    const float x1 = i + 1 < n ? x[i + 1] : 0.f;
    float y0, y1;
    fa::ptx::unpack_f32x2(fa::ptx::exp2_poly2(fa::ptx::pack_f32x2(x[i], x1)), y0, y1);
    y[i] = y0;
    if (i + 1 < n) y[i + 1] = y1;
}
}  // namespace

fa_status fa_debug_exp2(const float* x, float* y, int64_t n, cudaStream_t stream) {
    if (n < 0 || (n > 0 && (x == nullptr || y == nullptr))) return FA_ERR_INVALID_ARG;
    if (n == 0) return FA_OK;
    const int64_t pairs = (n + 1) / 2, blocks = (pairs + 255) / 256;
    if (blocks > INT32_MAX) return FA_ERR_UNSUPPORTED;
    exp2_poly_kernel<<<(unsigned)blocks, 256, 0, stream>>>(x, y, n);
    const cudaError_t err = cudaGetLastError();
    return err == cudaSuccess ? FA_OK : cuda_fail("exp2 test launch", err);
}

// Test hooks (declared in fa.h): the bound on every device-side wait, and a
// switch that makes CTA 0 withhold one K tile so that its waits run out.
void fa_debug_set_wait_limit_ms(double ms) {
    g_wait_limit_ns.store(ms > 0 ? (uint64_t)(ms * 1e6) : 0);
}
void fa_debug_inject_stall(int enable) { g_inject_stall.store(enable ? 1 : 0); }
void fa_debug_force_split(int mode) { g_force_split.store(mode == 1 || mode == 2 ? mode : 0); }
void fa_debug_force_chains(int mode) { g_force_chains.store(mode == 1 || mode == 2 ? mode : 0); }
void fa_debug_force_pair(int mode) { g_force_pair.store(mode == 1 || mode == 2 ? mode : 0); }

}  // extern "C"
