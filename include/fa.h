/*
 * libfa -- fused scaled-dot-product attention forward for GB300 (sm_103a).
 *
 * C ABI.  Plain pointers and sizes only; every tensor pointer is a DEVICE
 * pointer owned by the caller.  Link against libfa.so.
 *
 * The operation (pages "把 FlashAttention 搬上昇腾：Triton-Ascend CV Pipeline
 * 优化实战", section 一, and "Write Triton Attention Kernel", Required reasoning
 * process steps 1-9): for every batch z < Z, query head hq < Hq with key/value
 * head hk = hq / (Hq / Hkv), query row i < Nq,
 *
 *     s_ij       = scale * sum_d Q[z,hq,i,d] * K[z,hk,j,d]     for kept keys j
 *     O[z,hq,i,:] = sum_j softmax_j(s_i.) * V[z,hk,j,:]
 *     lse[z,hq,i] = log(sum_j exp(s_ij))                       (natural log)
 *
 * where the kept keys are j < Nkv, and with causal != 0 only j <= i (the
 * top-left convention: query row i sees keys 0..i, also when Nq != Nkv).
 * The N x N score matrix never reaches global memory: the kernel tiles over
 * keys with the online softmax ("Build Triton-Ascend Fused Attention",
 * Implementation Pattern), keeping the running max, denominator and output
 * accumulator in fp32 and casting the probabilities to the input type before
 * the P·V product.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes.  Host-side errors are returned before anything is enqueued. */
typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,     /* null pointer, negative size, Hq % Hkv != 0, Nkv == 0 with work, non-finite scale */
    FA_ERR_UNSUPPORTED = 2,     /* D not in {16, 32, 64, 128, 256}, dtype not fp16/bf16 */
    FA_ERR_ALIGNMENT = 3,       /* d-stride != 1, a base or stride not 16-byte aligned, negative stride */
    FA_ERR_CUDA = 4,            /* a CUDA runtime/driver call failed (launch, tensor map, device query) */
    FA_ERR_DEVICE_TIMEOUT = 5,  /* a bounded device-side wait ran out (see fa_device_status) */
    FA_ERR_WORKSPACE = 6,       /* workspace missing, not 256-byte aligned, or smaller than required */
    FA_ERR_DEVICE_CHECK = 7     /* debug-check builds only: a kernel role decoded a unit outside the
                                   launch's sizes (see fa_device_status) and stopped */
} fa_status;

typedef enum { FA_DTYPE_F16 = 0, FA_DTYPE_BF16 = 1 } fa_dtype;

/* Element strides of a BNSD tensor: batch, head, sequence, head-dim.  Every
 * tensor carries its own strides ("Build Triton-Ascend Fused Attention",
 * Ascend Guardrails; "Write Triton Attention Kernel", Kernel design rules), so
 * BNSD, BSND ("BNHD") and other permuted or padded layouts are all accepted as
 * long as d == 1 and the other strides are multiples of 8 elements. */
typedef struct {
    int64_t b, h, n, d;
} fa_strides;

/*
 * fa_fwd -- enqueue the attention forward on `stream` (asynchronous).
 *
 *   q    (Z, Hq,  Nq,  D)  dtype, strides *sq
 *   k    (Z, Hkv, Nkv, D)  dtype, strides *sk
 *   v    (Z, Hkv, Nkv, D)  dtype, strides *sv
 *   o    (Z, Hq,  Nq,  D)  dtype, strides *so   (written)
 *   lse  (Z, Hq,  Nq)      fp32, contiguous      (written; may be NULL to skip)
 *   scale   softmax scale (commonly 1/sqrt(D)): any finite value, zero and
 *           negative included ("Write Triton Attention Kernel", Inputs 4:
 *           1/sqrt(D) or a custom value), as long as |scale|·log2(e) is
 *           finite in fp32 (|scale| <= ~2.4e38).  Scale 0 weighs every kept
 *           key equally (O = mean of their V, lse = log of their count).
 *   causal  0 or 1
 *   dtype   FA_DTYPE_F16 or FA_DTYPE_BF16 for Q, K, V and O
 *   stream  CUDA stream (0 = legacy default stream)
 *
 * Requirements: D in {16, 32, 64, 128, 256}; Hq % Hkv == 0 (GQA/MQA when
 * Hkv < Hq); Nkv >= 1 whenever Z*Hq*Nq > 0; q, k, v, o 16-byte aligned with
 * d-stride 1 and the other strides multiples of 8 elements (16 bytes);
 * lse 4-byte aligned.  Any Nq, Nkv (ragged tails are masked).  Z*Hq*Nq == 0
 * is a no-op that returns FA_OK.
 *
 * Ownership: the caller owns every buffer and must keep them alive until the
 * stream reaches this work.  The library allocates no device memory per call;
 * it keeps one 4-byte status word per device for device-side errors.
 *
 * Errors: argument errors return FA_ERR_INVALID_ARG / FA_ERR_UNSUPPORTED /
 * FA_ERR_ALIGNMENT synchronously and enqueue nothing; a failed launch returns
 * FA_ERR_CUDA.  A device-side wait that runs out is reported later through
 * fa_device_status().  No CPU fallback exists.
 */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int Z, int Hq, int Hkv, int Nq,
                 int Nkv, int D, const fa_strides* sq, const fa_strides* sk, const fa_strides* sv,
                 const fa_strides* so, float scale, int causal, fa_dtype dtype, cudaStream_t stream);

/*
 * Options of fa_fwd_ex: the variants the page "Write Triton Attention Kernel"
 * names for such a kernel ("Use this when": windowed attention, ALiBi;
 * "Inputs", items 3 and 6, and "Correctness requirements": CSR-style
 * variable-length batches whose key loop ends at each sequence's length).
 * The pages give no formulas; with i the query row and j the key within one
 * sequence (both from 0, the top-left convention of the causal mask):
 *
 *   window_left, window_right   key j is kept iff j >= i - window_left and
 *                               j <= i + window_right; -1 leaves a side open
 *                               (and with causal, also j <= i)
 *   alibi_slopes                NULL, or a device array of Hq fp32 slopes:
 *                               the scaled score of (i, j) in head hq gets
 *                               -alibi_slopes[hq] * |i - j|
 *   cu_seqlens_q, cu_seqlens_k  NULL (padded batches), or device arrays of
 *                               Z + 1 int32 offsets: sequence z owns query
 *                               rows cu_seqlens_q[z] .. cu_seqlens_q[z+1]-1
 *                               and key rows cu_seqlens_k[z] .. [z+1]-1 of
 *                               packed tensors, and attends only to its own
 *                               keys; both start at 0 and never decrease
 *   max_seqlen_q                with cu_seqlens: at least the longest query
 *                               sequence (rows past it are not computed)
 *   max_seqlen_k                with cu_seqlens, read by fa_bwd_ex only: at
 *                               least the longest key sequence (keys past it
 *                               get no gradient), or 0 for the packed total
 *
 * A query row with no kept key gets O = 0 and lse = -inf.
 */
typedef struct {
    int window_left;
    int window_right;
    const float* alibi_slopes;
    const int32_t* cu_seqlens_q;
    const int32_t* cu_seqlens_k;
    int max_seqlen_q;
    int max_seqlen_k;
} fa_fwd_options;

/*
 * fa_fwd_ex -- fa_fwd with the options above.  With no sequence table, no
 * slopes and both window sides open (-1 or longer than Nq + Nkv; NULL options
 * included) the call is fa_fwd and runs fa_fwd's kernel.  Arguments are those
 * of fa_fwd, except
 * with cu_seqlens set: Z is the number of sequences, the tensors are packed
 * with a batch extent of one -- q and o (1, Hq, Nq, D), k and v (1, Hkv, Nkv,
 * D), any strides as for fa_fwd (the batch stride is ignored), Nq and Nkv the
 * packed row counts (total rows, Nkv >= 1) -- and lse is (Hq, Nq) fp32
 * contiguous.  Whole query tiles only (no split-KV schedule).
 *
 * Errors: those of fa_fwd, plus FA_ERR_INVALID_ARG for a window side below
 * -1, only one of the cu_seqlens arrays, or max_seqlen_q < 0, and
 * FA_ERR_ALIGNMENT for an option array not 4-byte aligned.  The contents of
 * the device arrays are not validated on the host; offsets outside the packed
 * extents are clamped to them on the device.
 */
fa_status fa_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int Z, int Hq, int Hkv, int Nq,
                    int Nkv, int D, const fa_strides* sq, const fa_strides* sk, const fa_strides* sv,
                    const fa_strides* so, float scale, int causal, fa_dtype dtype, const fa_fwd_options* options,
                    cudaStream_t stream);

/*
 * fa_fwd_splitkv -- the same attention forward as fa_fwd (same arguments,
 * same results up to rounding), scheduled for problems with few query tiles
 * and many keys: decode-like and cross-attention shapes, long causal heads.
 *
 * fa_fwd hands whole 128-row query tiles to the SMs, so with fewer tiles than
 * SMs (or a tile count just above a multiple of it) SMs idle.  When that
 * idle share is large (the busiest SM would get at least 2048 keys' worth of
 * key blocks more than an even cut gives it), the (query tile, key block)
 * pairs of all tiles are laid end to end and cut into one equal range per
 * SM; otherwise the call runs exactly as fa_fwd does.  A tile that a cut
 * crosses is computed in parts,
 * each over a contiguous range of key blocks; every part leaves its O / l in
 * fp32 and its log-sum-exp in `workspace`, and a second kernel on the same
 * stream combines the parts of each such tile by their log-sum-exps:
 *     lse = log(sum_s exp(lse_s)),   O = sum_s exp(lse_s - lse) * O_s,
 * the rescaling the online softmax applies between key blocks ("Write
 * Triton Attention Kernel", Kernel design rules), with the per-part lse of
 * step 8.  No CTA waits for another.
 *
 *   workspace        device memory, 256-byte aligned, at least the size
 *                    fa_fwd_splitkv_workspace_size() returns for D on this
 *                    device; its contents need no initialisation and are
 *                    overwritten.  Two calls that may run at the same time
 *                    (different streams) must not share one workspace.
 *   workspace_bytes  its size in bytes
 *
 * Errors: those of fa_fwd, plus FA_ERR_WORKSPACE for a missing, misaligned or
 * too small workspace.  Results are bitwise reproducible for a given shape
 * and device (the cut points depend only on the shape and the SM count).
 */
fa_status fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int Z, int Hq, int Hkv,
                         int Nq, int Nkv, int D, const fa_strides* sq, const fa_strides* sk, const fa_strides* sv,
                         const fa_strides* so, float scale, int causal, fa_dtype dtype, void* workspace,
                         size_t workspace_bytes, cudaStream_t stream);

/*
 * fa_fwd_splitkv_workspace_size -- bytes of workspace fa_fwd_splitkv needs
 * for head dim D on the current device, for any problem size: two partial
 * slots per SM, each 128 x D fp32 values plus 128 fp32 log-sum-exps (about
 * 20 MB for D = 128 and 40 MB for D = 256 on 152 SMs).  Returns
 * FA_ERR_UNSUPPORTED for an unsupported D, FA_ERR_CUDA without a device.
 */
fa_status fa_fwd_splitkv_workspace_size(int D, size_t* bytes);

/*
 * fa_fwd_splitkv_workspace_size_for -- host only, no CUDA call: the same size
 * for a device with num_sms SMs (two slots per SM, each 128 x D + 128 fp32
 * values padded to 256 bytes).  FA_ERR_INVALID_ARG for a NULL bytes or
 * num_sms < 1, FA_ERR_UNSUPPORTED for an unsupported D.
 */
fa_status fa_fwd_splitkv_workspace_size_for(int D, int num_sms, size_t* bytes);

/* Size in bytes of the device array fa_fwd_splitkv_noalloc works in (40 MiB). */
#define FA_NOALLOC_SCRATCH_BYTES (40u * 1024u * 1024u)

/*
 * fa_fwd_splitkv_noalloc -- fa_fwd_splitkv without a caller workspace and
 * without allocating anything: the partial results live in a fixed array of
 * FA_NOALLOC_SCRATCH_BYTES inside this library's device image.  (The pages
 * have no counterpart of this entry point.)
 *
 * For callers that cannot allocate device memory while they run: a
 * cudaMalloc synchronises the whole device and can take milliseconds, which
 * a latency-bound serving loop cannot afford; a plugin interface may hand
 * over only input and output buffers; another allocator may own all of the
 * device's memory.  Arguments, results and the other errors are those of
 * fa_fwd_splitkv; this call makes no cudaMalloc or cudaFree.
 *
 * The array is part of this library's device image, so it takes 40 MiB of
 * device memory in each CUDA context that loads the image, until that
 * context is destroyed.  Under lazy module loading (the CUDA default) that
 * happens on the first call of this entry point in the context, and the
 * call fails with FA_ERR_CUDA if 40 MiB of device memory are not free then;
 * with CUDA_MODULE_LOADING=EAGER every context the process creates reserves
 * the 40 MiB when it is created, whether or not it ever calls this entry
 * point.  The first call in each context also looks up the array's device
 * address (with the device current); make that first call before any stream
 * capture.  A context destroyed by cudaDeviceReset and created again gets a
 * new lookup on its next first call; a failed lookup is retried by the next
 * call.  40 MiB covers two partial slots per SM at D = 256 on GPUs of up to
 * 159 SMs (fa_fwd_splitkv_workspace_size_for gives the need for a given SM
 * count); a device that needs more is rejected with FA_ERR_WORKSPACE before
 * anything is enqueued.
 * Nothing in the array has to start at zero: each call writes every slot it
 * later reads.  All calls on a device share the one array, so two calls whose
 * work may overlap on the GPU (different streams without ordering between
 * them, or other host threads) corrupt each other's results; order them on
 * one stream or synchronise between them.
 */
fa_status fa_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int Z, int Hq,
                                 int Hkv, int Nq, int Nkv, int D, const fa_strides* sq, const fa_strides* sk,
                                 const fa_strides* sv, const fa_strides* so, float scale, int causal, fa_dtype dtype,
                                 cudaStream_t stream);

/* Most partial results fa_lse_merge combines in one call. */
#define FA_MERGE_MAX_PARTS 16

/*
 * fa_lse_merge -- combine attention results computed over disjoint key sets
 * (for instance a sequence split into shards, each run through fa_fwd
 * against its own keys, on one GPU or several) into the result over their
 * union:
 *     lse[r] = log(sum_s exp(lse_s[r])),
 *     o[r,:] = sum_s exp(lse_s[r] - lse[r]) * o_s[r,:]
 * for every row r = (z, h, n).  The parts are what fa_fwd writes: O
 * normalised by its own denominator, in dtype, and the natural-log lse
 * ("Write Triton Attention Kernel", step 8).  Arithmetic is fp32; O is
 * rounded once to dtype.  A row whose parts all have lse = -inf (no kept
 * key anywhere) gets o = 0 and lse = -inf.
 *
 *   nparts     1 .. FA_MERGE_MAX_PARTS
 *   o_parts    host array of nparts device pointers, each (Z, H, N, D) dtype
 *              with the element strides *sp (shared by all parts)
 *   lse_parts  host array of nparts device pointers, each (Z, H, N) fp32
 *              contiguous
 *   o          (Z, H, N, D) dtype, strides *so (written; may alias no part)
 *   lse        (Z, H, N) fp32 contiguous (written), or NULL to skip
 *
 * Requirements: D in {16, 32, 64, 128, 256}; every O pointer 16-byte aligned
 * with d-stride 1 and other strides multiples of 8 elements; lse pointers
 * 4-byte aligned.  Z*H*N == 0 is a no-op.  Asynchronous on `stream`;
 * argument errors return before anything is enqueued.
 */
fa_status fa_lse_merge(int nparts, const void* const* o_parts, const float* const* lse_parts, int Z, int H, int N,
                       int D, const fa_strides* sp, void* o, float* lse, const fa_strides* so, fa_dtype dtype,
                       cudaStream_t stream);

/*
 * fa_bwd -- gradients of the attention forward (blog "把 FlashAttention 搬上昇腾：
 * Triton-Ascend CV Pipeline 优化实战", section 二; "Write Triton Attention
 * Kernel", step 8: the backward rebuilds the probabilities from the saved
 * lse).  For a loss with upstream gradient dO = dLoss/dO:
 *
 *     P_ij  = exp(s_ij - lse_i)           s_ij = scale q_i . k_j (kept keys)
 *     dV_j  = sum_i P_ij dO_i             dP_ij = dO_i . v_j
 *     dS_ij = P_ij (dP_ij - Delta_i)      Delta_i = dO_i . O_i
 *     dQ_i  = scale sum_j dS_ij k_j       dK_j = scale sum_i dS_ij q_i
 *
 * with dK, dV of a key/value head summed over the query heads of its GQA
 * group, and the causal rule of fa_fwd.
 *
 *   q, k, v, o   the forward's inputs and output, layouts as for fa_fwd
 *   lse          the forward's lse (Z, Hq, Nq) fp32 contiguous (required)
 *   dO           (Z, Hq, Nq, D) dtype, strides *sdo
 *   dq           (Z, Hq, Nq, D) dtype, strides *sdq     (written)
 *   dk, dv       (Z, Hkv, Nkv, D) dtype, strides *sdk, *sdv (written)
 *   workspace    device memory, 256-byte aligned, at least
 *                fa_bwd_workspace_size(Z, Hq, Nq, D) bytes (per-row Delta
 *                and lse); no initialisation needed, overwritten; not shared
 *                by calls that may overlap
 *
 * Requirements: those of fa_fwd (D in {16, 32, 64, 128, 256}) and Nq >= 1
 * whenever Z*Hkv*Nkv > 0.  Two kernels on `stream`: Delta and lse per row;
 * then one persistent kernel whose CTAs first compute dK and dV (a unit per
 * key block and kv head, over every query of the group), then dQ (a unit per
 * query block and head, over its keys, recomputing the scores).  At D = 256
 * the dK/dV units take dV and dK in two passes over the queries (one
 * 256-column accumulator in tensor memory at a time) and both phases step
 * 64 rows at a time.  No atomics: results are bitwise reproducible.
 * Errors: those of fa_fwd, plus FA_ERR_WORKSPACE for a missing, misaligned
 * or small workspace.
 */
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                 void* dq, void* dk, void* dv, int Z, int Hq, int Hkv, int Nq, int Nkv, int D, const fa_strides* sq,
                 const fa_strides* sk, const fa_strides* sv, const fa_strides* so, const fa_strides* sdo,
                 const fa_strides* sdq, const fa_strides* sdk, const fa_strides* sdv, float scale, int causal,
                 fa_dtype dtype, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * fa_bwd_ex -- fa_bwd for fa_fwd_ex's options (fa_fwd_options above; the
 * variants of "Write Triton Attention Kernel", Inputs): the same formulas with
 * s_ij = scale q_i . k_j - alibi_slopes[hq] |i - j| over the kept keys of the
 * window (and the causal rule), within each packed sequence when cu_seqlens
 * are set.  Arguments are those of fa_bwd plus `options` (NULL: none); q, k,
 * v, o and lse come from fa_fwd_ex (or fa_fwd) with the same options.  With no
 * sequence table, both window sides open (-1 or longer than Nq + Nkv) and no
 * slopes the call is fa_bwd.  A dK/dV unit visits only the query blocks that
 * keep a key of its block, a dQ unit only the key blocks its rows keep; a
 * query row with no kept key gets dQ = 0, a key no row keeps dK = dV = 0.
 *
 * With cu_seqlens set, as for fa_fwd_ex: Z is the number of sequences, all
 * nine tensors are packed with a batch extent of one (q, o, dO, dq (1, Hq, Nq,
 * D); k, v, dk, dv (1, Hkv, Nkv, D); Nq and Nkv the packed row totals), lse is
 * (Hq, Nq) fp32 contiguous, and the workspace is fa_bwd_workspace_size(Z, Hq,
 * max_seqlen_q, D) bytes.  Rows of the packed tensors outside every sequence
 * are not written.
 *
 * Errors: those of fa_bwd, plus FA_ERR_INVALID_ARG for a window side below
 * -1, only one of the cu_seqlens arrays, or a negative max_seqlen_q or
 * max_seqlen_k, and FA_ERR_ALIGNMENT for an option array not 4-byte aligned.
 * Every head dim of fa_bwd takes every option.  The offsets are not validated
 * on the host; those outside the packed extents are clamped to them on the
 * device.
 */
fa_status fa_bwd_ex(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                    void* dq, void* dk, void* dv, int Z, int Hq, int Hkv, int Nq, int Nkv, int D,
                    const fa_strides* sq, const fa_strides* sk, const fa_strides* sv, const fa_strides* so,
                    const fa_strides* sdo, const fa_strides* sdq, const fa_strides* sdk, const fa_strides* sdv,
                    float scale, int causal, fa_dtype dtype, const fa_fwd_options* options, void* workspace,
                    size_t workspace_bytes, cudaStream_t stream);

/* Bytes of workspace fa_bwd (and fa_bwd_ex) needs (host only; FA_ERR_UNSUPPORTED for an unsupported D). */
fa_status fa_bwd_workspace_size(int Z, int Hq, int Nq, int D, size_t* bytes);

/* Human-readable name of a status code (static storage, never NULL). */
const char* fa_status_string(fa_status status);

/*
 * fa_device_status -- synchronise `stream`, then read and clear the current
 * device's status word.  Returns FA_OK, FA_ERR_DEVICE_TIMEOUT (a bounded
 * mbarrier wait inside a kernel gave up and the kernel exited cleanly),
 * FA_ERR_DEVICE_CHECK (only in a library built with debug index checks,
 * `python -m exact_attention_44_gb300.build --debug-checks`: a role of the
 * forward kernel found a unit outside the launch's sizes, recorded it and
 * stopped; the wait site field then names the role), or FA_ERR_CUDA if the
 * synchronisation itself failed.  When `detail` is not
 * NULL it receives the raw word: bits 0-7 the code, 8-15 the wait site,
 * 16-31 the CTA index that gave up first.
 */
fa_status fa_device_status(cudaStream_t stream, uint32_t* detail);

/*
 * fa_fwd_plan -- host-only description of the work fa_fwd would launch; no
 * CUDA call is made.  Pass num_sms > 0 to size the persistent grid for that
 * many SMs (0 leaves *grid at the tile count).  Outputs (each may be NULL):
 *   tiles      query tiles of 128 rows, Z * Hq * ceil(Nq / 128)
 *   kv_blocks  (query tile, key block) pairs the kernel visits; with causal
 *              set the loop stops at the diagonal block (page "把 FlashAttention
 *              搬上昇腾...", section 八: 8 x 8 tiles -> 36 visited)
 *   block_n    keys per block for this D (128, or 64 at D = 256)
 *   grid       CTAs launched: min(tiles, num_sms)
 *   smem_bytes dynamic shared memory per CTA
 * Returns the same argument errors as fa_fwd for bad shapes.
 */
fa_status fa_fwd_plan(int Z, int Hq, int Hkv, int Nq, int Nkv, int D, int causal, int num_sms, int64_t* tiles,
                      int64_t* kv_blocks, int* block_n, int* grid, int* smem_bytes);

/*
 * fa_fwd_schedule -- host-only: the schedule fa_fwd (splitkv = 0) or
 * fa_fwd_splitkv (splitkv = 1) picks for contiguous BNSD tensors of these
 * sizes on a device with num_sms SMs and l2_bytes of L2 (what the calls read
 * from the device); no CUDA call is made.  The page "把 FlashAttention 搬上昇腾..."
 * (sections 五, 八) schedules heavy causal tiles first over a persistent grid;
 * the grouping and alternation below are this library's refinements of that.
 *   grid            CTAs of the forward launch
 *   split           1: key ranges cut into one equal range per CTA and the
 *                   cut tiles merged (fa_fwd_splitkv only, where it pays)
 *   gqa_packed      1: the query heads of each GQA group run as one head of
 *                   g * Nq rows (non-causal, Nq < 128)
 *   head_group      causal whole-tile order: heads per group (all heads when
 *                   their K/V fit in a third of L2)
 *   alternate       causal whole-tile order: rounds alternate direction
 *                   (long tiles only)
 *   tiles           query tiles of the launch (after packing)
 *   kv_blocks       (tile, key block) pairs of the launch
 *   busiest_blocks  key blocks of the busiest CTA in the schedule that runs
 *   softmax_chains  2: whole tiles of head dims up to 128 run the kernel
 *                   whose softmax is two warpgroups taking the key blocks in
 *                   turn (the same tiles and order); 1: one chain
 *   cta_pairs       1: whole tiles at D = 128 run on clusters of two CTAs,
 *                   each cluster taking two query tiles that see the same key
 *                   blocks (two query heads of a GQA group, else query blocks
 *                   2m and 2m + 1 of one head) and multiplying each key block
 *                   once for both (M = 256 over two SMs, each holding half of
 *                   every K and V block), with two softmax chains per SM;
 *                   grid is then 2 x min(units, num_sms / 2) (at launch: the
 *                   clusters the device can hold at once) and busiest_blocks
 *                   the key blocks of the busiest cluster
 * Errors: those of fa_fwd_plan for bad shapes; FA_ERR_INVALID_ARG for a NULL
 * out, num_sms < 1 or l2_bytes < 1.  fa_debug_force_split applies here too.
 */
typedef struct {
    int grid;
    int split;
    int gqa_packed;
    int head_group;
    int alternate;
    int64_t tiles;
    int64_t kv_blocks;
    int64_t busiest_blocks;
    int softmax_chains;
    int cta_pairs;
} fa_fwd_schedule_info;

fa_status fa_fwd_schedule(int Z, int Hq, int Hkv, int Nq, int Nkv, int D, int causal, int splitkv, int num_sms,
                          int64_t l2_bytes, fa_fwd_schedule_info* out);

/*
 * Test hooks for the failure-detection path; not for production use.
 *
 * fa_debug_set_wait_limit_ms -- bound, in milliseconds, on every mbarrier wait
 *   inside later launches (default 2000, or FA_WAIT_LIMIT_MS from the
 *   environment; ms <= 0 restores that default).  A healthy kernel waits
 *   microseconds; the bound only matters when something is wrong.
 * fa_debug_force_split -- how fa_fwd_splitkv chooses between cutting key
 *   ranges and whole tiles: 0 by the shape (default), 1 always cut, 2 never.
 * fa_debug_force_chains -- which kernel runs whole tiles of head dims up to
 *   128: 0 by the shape (default: two softmax chains), 1 two chains, 2 one
 *   chain.  Both compute the same result (up to the order of rounding).
 * fa_debug_force_pair -- whether whole tiles at D = 128 run on CTA pairs
 *   (see fa_fwd_schedule's cta_pairs): 0 default (one-SM kernels: the pair
 *   kernel measured level with them on long tiles and slower on short ones),
 *   1 wherever the kernel applies, 2 never.  It takes precedence over
 *   fa_debug_force_chains.  The same result up to the order of rounding.
 * fa_debug_inject_stall -- when enabled, CTA 0 of later launches never issues
 *   the copy of its first K tile (forward kernels) or of its first unit's K
 *   and V (fa_bwd's dK/dV phase), so the wait for it runs out: the kernel
 *   records FA_ERR_DEVICE_TIMEOUT (read with fa_device_status), every role of
 *   that CTA stops, in-flight copies and MMAs land, TMEM is freed and the
 *   kernel returns.  The other CTAs finish their tiles.  Outputs of such a
 *   launch are incomplete.  No GPU fault, trap or hang is involved.
 */
void fa_debug_set_wait_limit_ms(double ms);

/*
 * fa_debug_exp2 -- test hook: y[i] = 2^x[i] computed by the polynomial
 *   exponential the softmax kernels use for part of their exponentials (the
 *   pages compute p = exp2(s·scale·log2e − m): "把 FlashAttention 搬上昇腾...",
 *   section 一): Cody-Waite reduction in base 2, a degree-4 minimax polynomial
 *   of 2^f on [-1/2, 1/2] (max relative error 2.6e-6), the integer part added
 *   to the exponent field.  Meant for arguments <= 8 (the softmax never
 *   exceeds its rescale threshold); x <= -126 gives ~1.2e-38.  x and y are
 *   device arrays of n floats; asynchronous on `stream`.
 */
fa_status fa_debug_exp2(const float* x, float* y, int64_t n, cudaStream_t stream);
void fa_debug_inject_stall(int enable);
void fa_debug_force_split(int mode);
void fa_debug_force_chains(int mode);
void fa_debug_force_pair(int mode);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
