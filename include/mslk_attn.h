/*
 * mslk_attn.h — C ABI of the GB300 (sm_103a) fused multi-head attention forward library.
 *
 * What the calls compute (MSLK kernel reference, "Attention - Core fMHA"):
 *
 *   out[b,i,h,:] = sum_{j in A_i} softmax_j(scale * q[b,i,h,:] . k[b,j,h,:]) * v[b,j,h,:]
 *   lse[b,h,i]   = ln sum_{j in A_i} exp(scale * q[b,i,h,:] . k[b,j,h,:])
 *
 * without materialising the score matrix.  A_i is the set of keys the mask allows
 * for query row i (MSLK kernel reference, "Attention - Biases & masks").  A row whose
 * allowed set is empty gets out = 0 and lse = -inf.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Tensors are [B, M, H, D] (q, out), [B, Mkv, Hkv, D] (k, v): batch, sequence, head,
 *    head dim.  Only the head dim must be contiguous (stride 1); the batch, sequence and
 *    head strides may be anything that meets the alignment rule below, and are given in
 *    ELEMENTS by mslk_strides (MSLK kernel reference > Attention - Core fMHA >
 *    memory_efficient_attention, constraints).  The output has the query layout with its
 *    last dimension replaced by the value head dim.
 *  - Grouped K/V heads (GQA / MQA): mslk_attn takes Hkv K/V heads for H query heads
 *    (Hkv divides H; query head h reads K/V head h / (H / Hkv)).  The other calls take
 *    Hkv = H, except that a k/v head stride of 0 (an expand() of one head) means one K/V
 *    head shared by every query head.  The pages' 5-D BMGHK layout with K/V expanded over
 *    the H axis is this with Hkv = G once the (G, H) axes are flattened group-major
 *    (bmghk2bmhk); the Python binding does that flattening on views.
 *  - q, k, v are bf16 (E4M3 for mslk_attn_fwd_fp8).  K == Kv and the head dim is 64, 96
 *    or 128 (96 runs on the 128-wide kernels with the missing columns read as zeros);
 *    other head dims, and K != Kv, return MSLK_ERR_UNSUPPORTED.
 *  - lse is fp32 [B, H, M], contiguous.  Packed variable-length batches (B = 1) use
 *    [1, H, total_q].
 *  - Every pointer is caller-owned DEVICE memory (except the mslk_seqlens struct and
 *    the mslk_strides structs, which live on the host and are read during the call).
 *    The library allocates no device memory and keeps no state between calls, apart
 *    from a per-device error word read by mslk_device_status() and the fixed workspace
 *    array of mslk_attn_split_kv_static.
 *  - Alignment: q, k, v, out base pointers 16-byte aligned; every free stride times the
 *    element size a multiple of 16 bytes (the tensor-memory-accelerator copy rule).
 *    Violations return MSLK_ERR_MISALIGNED.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy default
 *    stream).  Argument errors return before any launch and write nothing.  A failed
 *    launch returns MSLK_ERR_CUDA.  Kernels bound every internal wait; a wait that runs
 *    out sets the device error word, which mslk_device_status() reports as
 *    MSLK_ERR_DEVICE_TIMEOUT.
 *  - scale <= 0 or NaN selects the default 1/sqrt(K) (scale=None in the pages).
 *  - Results are deterministic: no atomics on the data path; the same inputs give the
 *    same bits.
 */
#ifndef MSLK_ATTN_H
#define MSLK_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MSLK_OK = 0,
  MSLK_ERR_INVALID_ARG = 1,     /* null pointer, bad size, bad mask/seqlens combination */
  MSLK_ERR_UNSUPPORTED = 2,     /* valid request this build does not implement (head dim) */
  MSLK_ERR_MISALIGNED = 3,      /* base pointer or stride breaks the 16-byte rule */
  MSLK_ERR_CUDA = 4,            /* a CUDA runtime/driver call failed */
  MSLK_ERR_DEVICE_TIMEOUT = 5   /* a bounded in-kernel wait ran out (mslk_device_status) */
} mslk_status;

/* Mask kinds (MSLK kernel reference, "Attention - Biases & masks"). */
typedef enum {
  MSLK_MASK_NONE = 0,              /* every key */
  MSLK_MASK_CAUSAL = 1,            /* LowerTriangularMask: top-left, key position <= query row */
  MSLK_MASK_BLOCKDIAG = 2,         /* BlockDiagonalMask: packed sequences, B = 1 */
  MSLK_MASK_BLOCKDIAG_CAUSAL = 3,  /* BlockDiagonalCausalMask: top-left causal inside each block */
  /* LowerTriangularFromBottomRightMask: query i pairs with key i + Mkv - M, keys after it are
   * masked (forward only; a split-KV chunk expresses this through kv_offset). */
  MSLK_MASK_CAUSAL_BOTTOM_RIGHT = 4,
  /* BlockDiagonalCausalFromBottomRightMask: the same inside every packed block (forward only). */
  MSLK_MASK_BLOCKDIAG_CAUSAL_BOTTOM_RIGHT = 5
} mslk_mask_kind;

/*
 * Alignment and local window of a mask (same page: LowerTriangularFromBottomRight-
 * LocalAttentionMask, LocalAttentionFromBottomRightMask, BlockDiagonalCausalLocal-
 * AttentionMask, BlockDiagonalCausalLocalAttentionFromBottomRightMask; the pages name
 * them without formulas, this is the reading the library implements).  Query row i of a
 * block of Lq rows and Lk keys (the whole tensor for dense kinds, one packed sequence for
 * block-diagonal kinds) is PAIRED with key position p = i + (bottom_right ? Lk - Lq : 0);
 * key position j (kv_offset + chunk index for partials) is allowed iff
 *     j <= p                       for causal kinds (window_right must be -1 or 0),
 *     j <= p + window_right        for other kinds when window_right >= 0,
 *     j >= p - window_left         when window_left >= 0,
 * on top of the kind's own rule (same block for block-diagonal kinds).  -1 leaves that side
 * open.  A causal local window of w keys (the pages' window_size) is window_left = w - 1.
 */
typedef struct {
  int32_t bottom_right;  /* 0 or 1; kinds 4 and 5 imply 1.  Forward only. */
  int32_t window_left;   /* >= 0, or -1: unbounded */
  int32_t window_right;  /* >= 0, or -1: unbounded */
} mslk_band;

typedef enum { MSLK_DTYPE_BF16 = 0, MSLK_DTYPE_FP32 = 1 } mslk_dtype;

/* Element strides of the batch, sequence and head dimensions (head dim stride is 1). */
typedef struct {
  int64_t b, m, h;
} mslk_strides;

/*
 * Sequence metadata of a packed batch (BlockDiagonalMask.from_seqlens; the standalone
 * Blackwell facade's cu_seqlens_q / cu_seqlens_k / max_seq_len_q / max_seq_len_k).
 * cu_seqlens_q/k are DEVICE int32 arrays of n_seqs + 1 non-decreasing offsets starting
 * at 0 and ending at M / Mkv.  max_seqlen_q must be >= every query length (rows of longer
 * sequences beyond it are not computed).  Offsets outside [0, M] / [0, Mkv] are clamped
 * by the kernels, never dereferenced.  Ignored (may be NULL) for the dense masks.
 */
typedef struct {
  const int32_t* cu_seqlens_q;
  const int32_t* cu_seqlens_k;
  int32_t n_seqs;
  int32_t max_seqlen_q;
  int32_t max_seqlen_k;
} mslk_seqlens;

/*
 * mslk_attn_fwd — fused attention forward returning out and (optionally) lse.
 * MSLK kernel reference, "Attention - Core fMHA" > memory_efficient_attention_forward
 * (out only, lse == NULL) and memory_efficient_attention_forward_requires_grad
 * (returns (output, lse)); raw op "Attention - Raw Blackwell torch ops" > fmha_fwd.
 *
 *   q [B,M,H,K] bf16 (strides sq), k [B,Mkv,H,K] bf16 (sk), v [B,Mkv,H,Kv] bf16 (sv).
 *   out [B,M,H,Kv] bf16 (strides so), written for every row.
 *   lse [B,H,M] fp32 contiguous, or NULL to skip it.
 *   mask_kind: mslk_mask_kind.  Block-diagonal kinds need B == 1 and `seqlens`.
 *   Dropout is not part of this API (the pages' forward-with-LSE call rejects it).
 * Sizes: B, M, H, Mkv >= 0 (B, M or H == 0: nothing to do; Mkv == 0: out = 0, lse = -inf).
 */
mslk_status mslk_attn_fwd(const void* q, const void* k, const void* v,
                          const mslk_strides* sq, const mslk_strides* sk,
                          const mslk_strides* sv, const mslk_strides* so,
                          int32_t B, int32_t M, int32_t Mkv, int32_t H, int32_t K, int32_t Kv,
                          float scale, int32_t mask_kind, const mslk_seqlens* seqlens,
                          void* out, float* lse, void* stream);

/*
 * mslk_attn_partial — attention over ONE disjoint key/value chunk, for exact split-KV.
 * MSLK kernel reference, "Attention - Core fMHA" > memory_efficient_attention_partial:
 * call it once per chunk with the same queries, then combine with mslk_merge_attentions.
 *
 * Arguments as mslk_attn_fwd, with k/v (and Mkv) describing the chunk only, plus:
 *   kv_offset  position of the chunk's first key in the full key sequence (inside each
 *              packed sequence for the block-diagonal kinds).  Causal kinds and windows
 *              read it: key j of the chunk is at position kv_offset + j (causal: allowed
 *              for row i iff kv_offset + j <= i).  Bottom-right kinds are forward only.
 *   out_dtype  MSLK_DTYPE_FP32 (recommended: keeps the merge exact to fp32) or
 *              MSLK_DTYPE_BF16.  out strides `so` are in elements of that type.
 *   lse        required, fp32 [B,H,M] contiguous.  Rows with no allowed key in this chunk
 *              get out = 0, lse = -inf, so the merge gives the chunk zero weight.
 */
mslk_status mslk_attn_partial(const void* q, const void* k, const void* v,
                              const mslk_strides* sq, const mslk_strides* sk,
                              const mslk_strides* sv, const mslk_strides* so,
                              int32_t B, int32_t M, int32_t Mkv, int32_t H, int32_t K,
                              int32_t Kv, float scale, int32_t mask_kind,
                              const mslk_seqlens* seqlens, int64_t kv_offset, void* out,
                              int32_t out_dtype, float* lse, void* stream);

/*
 * mslk_attn_fwd_band / mslk_attn_partial_band — as mslk_attn_fwd / mslk_attn_partial with a
 * mask alignment and local window (mslk_band, read during the call; NULL = no window,
 * top-left unless the kind says otherwise).  Windows work with every mask kind; for the
 * partial call bottom_right must be 0 (fold Lk_full - Lq into kv_offset instead).
 * Key tiles outside every row's window are skipped, so a window of W keys costs
 * O(M * W) instead of O(M * Mkv).
 */
mslk_status mslk_attn_fwd_band(const void* q, const void* k, const void* v,
                               const mslk_strides* sq, const mslk_strides* sk,
                               const mslk_strides* sv, const mslk_strides* so,
                               int32_t B, int32_t M, int32_t Mkv, int32_t H, int32_t K,
                               int32_t Kv, float scale, int32_t mask_kind,
                               const mslk_seqlens* seqlens, const mslk_band* band, void* out,
                               float* lse, void* stream);
mslk_status mslk_attn_partial_band(const void* q, const void* k, const void* v,
                                   const mslk_strides* sq, const mslk_strides* sk,
                                   const mslk_strides* sv, const mslk_strides* so,
                                   int32_t B, int32_t M, int32_t Mkv, int32_t H, int32_t K,
                                   int32_t Kv, float scale, int32_t mask_kind,
                                   const mslk_seqlens* seqlens, const mslk_band* band,
                                   int64_t kv_offset, void* out, int32_t out_dtype, float* lse,
                                   void* stream);

/*
 * Key lanes (same page: BlockDiagonalPaddedKeysMask, BlockDiagonalCausalWithOffsetPadded-
 * KeysMask, PagedBlockDiagonalPaddedKeysMask and their local variants; named without
 * formulas, this is the reading the library implements).  Queries are packed as for the
 * block-diagonal kinds (cu_seqlens_q); sequence s owns a key lane of seqlen_k[s] valid
 * keys.  Logical key p of lane s is K/V row seqstart_k[s] + p (padded lanes), or, when
 * block_table is given, row block_table[s * max_pages + p / page_size] * page_size +
 * p % page_size of a pool of pages.  All arrays are DEVICE int32.  Rows past a lane's
 * valid keys are never read; keys past max_pages * page_size are ignored; rows outside
 * [0, Mkv) read as zeros.  page_size: a multiple of 128, or of 64 when every sequence has
 * at most 8 queries (the decode kernel streams 32/64-key tiles).
 */
typedef struct {
  const int32_t* seqlen_k;     /* [n_seqs] valid keys of each lane */
  const int32_t* seqstart_k;   /* [n_seqs] first row of each lane (unused with block_table) */
  const int32_t* block_table;  /* [n_seqs * max_pages] physical page per logical page, or NULL */
  int32_t page_size;           /* rows per page (block_table only) */
  int32_t max_pages;           /* columns of block_table */
} mslk_kv_lanes;

/*
 * mslk_attn_fwd_lanes — forward over key lanes.  q [1, total_q, H, K] packed with
 * seqlens->cu_seqlens_q (n_seqs, max_seqlen_q; max_seqlen_k = the longest lane;
 * cu_seqlens_k is not read); k, v [1, Mkv, H, D] hold the lanes or the page pool.
 * mask_kind: MSLK_MASK_BLOCKDIAG, _BLOCKDIAG_CAUSAL or _BLOCKDIAG_CAUSAL_BOTTOM_RIGHT
 * (the pages' "causal with offset"); band: optional window (NULL: none).
 */
mslk_status mslk_attn_fwd_lanes(const void* q, const void* k, const void* v,
                                const mslk_strides* sq, const mslk_strides* sk,
                                const mslk_strides* sv, const mslk_strides* so, int32_t M,
                                int32_t Mkv, int32_t H, int32_t K, int32_t Kv, float scale,
                                int32_t mask_kind, const mslk_seqlens* seqlens,
                                const mslk_kv_lanes* lanes, const mslk_band* band, void* out,
                                float* lse, void* stream);

/*
 * FP8 E4M3 inputs ("Attention - Core fMHA": the Blackwell and FlashAttention-3 forward
 * backends list FP8 E4M3; pack_fp8_tensorwise_per_head carries tensorwise or per-head
 * scales; the raw flash3 op takes descale_q / descale_k / descale_v).  Element x of head
 * h stands for the real value e4m3(x) * descale[h]; with per_tensor = 1 every head uses
 * descale[0].  The descales are DEVICE fp32 arrays read by the kernels: descale_q [H],
 * descale_k and descale_v [H] (or [1] when k/v use a shared head, head stride 0).
 */
typedef struct {
  const float* descale_q;
  const float* descale_k;
  const float* descale_v;
  int32_t per_tensor;
} mslk_fp8_scales;

/*
 * mslk_attn_fwd_fp8 — forward on E4M3 q, k, v (one byte per element; strides in
 * elements, multiples of 16; bases 16-byte aligned), bf16 out, fp32 lse (or NULL).
 * Masks, windows and bottom-right alignment as mslk_attn_fwd_band (band may be NULL);
 * key lanes as mslk_attn_fwd_lanes when `lanes` is non-NULL (then B must be 1).
 * The result is attention on the dequantized values.  Query blocks of at most 8 rows (per
 * packed sequence) may run on the CUDA-core kernel (probabilities rounded to f16); larger
 * ones on the tensor cores (kind::f8f6f4; K = Kv = 64 runs zero-padded to 128), where the
 * probabilities are rounded to E4M3 before P.V (relative error <= 2^-4 per probability;
 * the row sum uses the unrounded values).  Paged lanes need page_size a multiple of 128
 * (of 8192 / K when every sequence has at most 8 queries).
 */
mslk_status mslk_attn_fwd_fp8(const void* q, const void* k, const void* v,
                              const mslk_strides* sq, const mslk_strides* sk,
                              const mslk_strides* sv, const mslk_strides* so, int32_t B,
                              int32_t M, int32_t Mkv, int32_t H, int32_t K, int32_t Kv,
                              float scale, int32_t mask_kind, const mslk_seqlens* seqlens,
                              const mslk_band* band, const mslk_kv_lanes* lanes,
                              const mslk_fp8_scales* scales, void* out, float* lse,
                              void* stream);

/*
 * Every option of the forward and partial calls in one argument struct (read during the
 * call), for callers that need a combination the calls above do not take — in particular
 * grouped-query attention (Hkv K/V heads for H query heads).
 *   Hkv        K/V heads: 0 means H; otherwise Hkv divides H and query head h reads K/V
 *              head h / (H / Hkv) (the pages' BMGHK layout flattened group-major,
 *              bmghk2bmhk).  A k/v head stride of 0 still means one shared head.
 *   seqlens, band, lanes, fp8   as in the calls above (each may be NULL).
 *   partial    0: forward (mslk_attn_fwd*); 1: one K/V chunk (mslk_attn_partial*): lse
 *              required, kv_offset read, no bottom-right alignment, no key lanes.
 *   out_dtype  MSLK_DTYPE_BF16 or MSLK_DTYPE_FP32 for either mode.
 * Few query rows with a group ratio r > 1 fold up to 8 / rows query heads of a K/V head
 * into one block of rows, so that head's keys and values are streamed once for them.
 */
typedef struct {
  const void* q;
  const void* k;
  const void* v;
  mslk_strides sq, sk, sv, so;
  int32_t B, M, Mkv, H, Hkv, K, Kv;
  float scale;
  int32_t mask_kind;
  const mslk_seqlens* seqlens;
  const mslk_band* band;
  const mslk_kv_lanes* lanes;
  const mslk_fp8_scales* fp8;
  int32_t partial;
  int64_t kv_offset;
  void* out;
  int32_t out_dtype;
  float* lse;
  uint32_t flags;  /* MSLK_FLAG_* */
} mslk_attn_args;

/*
 * MSLK_FLAG_INDEPENDENT: the call may start before earlier launches on the stream have
 * finished (programmatic dependent launch), so back-to-back partials of a split-KV loop
 * overlap their ramp and tail.  Every kernel of this library lets a dependent launch start
 * as soon as it begins, so a run of flagged calls may overlap one another and the last
 * launch made WITHOUT the flag before them.  The caller states that no launch in that
 * window writes this call's inputs (q, k, v, descales, sequence tables) or reads or
 * writes its outputs (out, lse); e.g. the chunks of one split, each with its own out and
 * lse slice.  Calls without the flag keep plain stream order: they start only after every
 * earlier launch on the stream has finished, so a merge that reads the partials' outputs
 * waits for all of them.
 */
#define MSLK_FLAG_INDEPENDENT 1u

mslk_status mslk_attn(const mslk_attn_args* args, void* stream);

/*
 * mslk_attn_plan — which kernel mslk_attn would launch for these arguments under the
 * current path policy, without launching anything or touching the device: the same
 * validation (and the same error statuses) as mslk_attn, then *plan (caller-owned, host)
 * receives MSLK_PLAN_NONE (nothing to compute), MSLK_PLAN_FILL (no keys: out = 0 and
 * lse = -inf are written by a fill kernel), MSLK_PLAN_CUDA_CORES (the few-row kernel), or
 * MSLK_PLAN_TENSOR_CORES with MSLK_PLAN_FOLDED_HEADS (a group's query heads as the rows
 * of one unit) and / or MSLK_PLAN_SPLIT_UNITS (rows fit one 128-row tile: both softmax
 * warpgroups share a unit's key tiles).  Thread-safe; the device pointers are not read.
 */
#define MSLK_PLAN_NONE 0
#define MSLK_PLAN_FILL 1
#define MSLK_PLAN_CUDA_CORES 2
#define MSLK_PLAN_TENSOR_CORES 4
#define MSLK_PLAN_FOLDED_HEADS 8
#define MSLK_PLAN_SPLIT_UNITS 16
mslk_status mslk_attn_plan(const mslk_attn_args* args, int32_t* plan);

/*
 * mslk_merge_attentions — exact log-sum-exp merge of n chunk results into preallocated
 * outputs.  MSLK kernel reference, "Attention - Core fMHA" > merge_attentions (exact
 * normalised output over the union of chunks, not an average; write_lse; output_dtype)
 * and "Attention - Merge & storage utilities" > triton_splitk.merge_attentions
 * (in-place into preallocated outputs) / fmha_merge_attentions_varargs.
 *
 *   out_split  fp32, chunk c at out_split + c*chunk_stride_out, each [B,M,H,Kv] with
 *              strides s_split (chunks stacked on a leading axis, or any equally spaced
 *              views).
 *   lse_split  fp32, chunk c at lse_split + c*chunk_stride_lse, each [B,H,M] contiguous.
 *   n_chunks   >= 1 (zero partials is an error, as merge_attentions_autograd raises).
 *   out        [B,M,H,Kv] of out_dtype (BF16 or FP32), strides so.
 *   lse        fp32 [B,H,M] contiguous, or NULL (write_lse = False).
 * Per row: LSE = M* + ln sum_c exp(lse_c - M*) with M* = max_c lse_c;
 * out = sum_c exp(lse_c - LSE) * out_c; a row whose chunks are all -inf gets out = 0 and
 * LSE = -inf.  Kv must be a multiple of 4; out_split, out and their strides 16-byte
 * aligned; lse_split, the lse chunk stride and lse 4-byte aligned (MSLK_ERR_MISALIGNED).
 */
mslk_status mslk_merge_attentions(const float* out_split, const float* lse_split,
                                  int32_t n_chunks, int64_t chunk_stride_out,
                                  int64_t chunk_stride_lse, int32_t B, int32_t M, int32_t H,
                                  int32_t Kv, const mslk_strides* s_split,
                                  const mslk_strides* so, void* out, int32_t out_dtype,
                                  float* lse, void* stream);

/*
 * mslk_merge_attentions_varargs — the same merge over chunks that are separate
 * allocations (MSLK kernel reference, "Attention - Merge & storage utilities" >
 * torch.ops.mslk.fmha_merge_attentions_varargs, which takes lists of chunk tensors).
 *
 *   out_chunks  HOST array of n_chunks DEVICE pointers, chunk c's fp32 [B,M,H,Kv] output,
 *               every chunk with the strides s_split; read during the call only.
 *   lse_chunks  HOST array of n_chunks DEVICE pointers, chunk c's fp32 [B,H,M] lse
 *               (contiguous).
 *   n_chunks    1 .. MSLK_MERGE_MAX_VARARGS.
 * Other arguments, the result and the alignment rules as mslk_merge_attentions; every
 * chunk pointer follows the rule of out_split / lse_split.  Nothing is copied or stacked:
 * the kernel reads each chunk where it lies.
 */
#define MSLK_MERGE_MAX_VARARGS 128
mslk_status mslk_merge_attentions_varargs(const float* const* out_chunks,
                                          const float* const* lse_chunks, int32_t n_chunks,
                                          int32_t B, int32_t M, int32_t H, int32_t Kv,
                                          const mslk_strides* s_split, const mslk_strides* so,
                                          void* out, int32_t out_dtype, float* lse,
                                          void* stream);

/*
 * mslk_splitk_size — keys per split for split-KV attention (MSLK kernel reference,
 * "Attention - Standalone Blackwell FMHA" > get_splitk_heuristic: a split size from the
 * batch, the key count, the K/V heads and the SM count; 0 when one split covers the keys).
 * This library's rule: enough splits that every (batch, K/V head) unit has one split per
 * SM share, splits = ceil(sm_count / (batch * kv_heads)); size = ceil(seqlen_kv / splits)
 * rounded up to a multiple of tile_n; 0 when that size reaches seqlen_kv.  tile_n <= 0
 * means 256; sm_count <= 0 reads the current device's SM count (148 without a device).
 * Host-only and thread-safe; non-positive sizes give 0.
 */
int32_t mslk_splitk_size(int32_t batch, int32_t seqlen_kv, int32_t kv_heads, int32_t tile_n,
                         int32_t sm_count);

/*
 * mslk_attn_split_kv — exact split-KV attention in one call: the keys of a forward
 * problem are cut into n_chunks equal contiguous chunks (chunk c holds keys
 * [c * Mkv / n, (c + 1) * Mkv / n)), mslk_attn's partial form runs on each (fp32 results
 * in `workspace`), and the merge writes args->out and args->lse.  The same result as the
 * forward call within the merge's rounding ("Attention - Core fMHA" >
 * memory_efficient_attention_partial then merge_attentions, which is exact).
 *   args       a FORWARD problem as for mslk_attn (partial = 0): bf16 inputs, dense masks
 *              (none, causal, bottom-right causal), windows, grouped K/V heads; key lanes,
 *              block-diagonal masks and E4M3 inputs return MSLK_ERR_UNSUPPORTED.  A bottom-right
 *              alignment is folded into each chunk's kv_offset.  args->out_dtype and
 *              args->lse (NULL: not written) apply to the merged result.
 *   n_chunks   >= 1, or 0 to take ceil(Mkv / mslk_splitk_size(B, Mkv, Hkv, 256, SMs))
 *              (one chunk when that is 0); more chunks than keys are cut to one per key.
 *   workspace  caller-owned DEVICE memory, 256-byte aligned, of at least the size that
 *              mslk_attn_split_kv_workspace returns: the chunks' outputs [n, B, M, H, Kv]
 *              then their lse [n, B, H, M], fp32.  It is overwritten; it may be reused
 *              once the call's work on `stream` is done.
 * Launch order on `stream`: chunk 0, chunks 1.. n-1 declared independent of the one before
 * (they read the same inputs and write separate workspace slices), then the merge in plain
 * stream order.  args->flags applies to chunk 0 only.  Every argument error is returned
 * before the first launch.
 */
mslk_status mslk_attn_split_kv(const mslk_attn_args* args, int32_t n_chunks, void* workspace,
                               size_t workspace_bytes, void* stream);
/*
 * mslk_attn_split_kv_static — mslk_attn_split_kv without a workspace argument, for callers
 * that cannot allocate device memory when they call: a plug-in run by a host that owns all
 * device memory and hands kernels only their inputs and outputs, or a latency-critical
 * loop that cannot take cudaMalloc's device-wide synchronisation.  (The pages have no
 * counterpart: their split-K calls allocate their partial outputs.)
 *
 * The workspace is a fixed array of MSLK_SPLIT_KV_STATIC_BYTES inside the library; every
 * GPU that loads the library holds it until the process exits.  The call allocates
 * nothing: no cudaMalloc, cudaFree or allocating library routine.
 *   args, n_chunks  as mslk_attn_split_kv.  A problem whose workspace (as
 *                   mslk_attn_split_kv_workspace reports it) is larger than the array is
 *                   refused with MSLK_ERR_UNSUPPORTED before anything is launched.
 * The array's device address is looked up the first time the call runs on a device, with
 * that device current; make that first call before any stream capture.  Every call shares
 * the array, which keeps the previous call's contents; nothing in it needs to start at zero
 * (each chunk's partial writes all it holds before the merge reads it).  Calls whose work
 * overlaps on the GPU (different streams, or threads without an order between them) race
 * on the array: order them on one stream, or give each its own workspace with
 * mslk_attn_split_kv.
 */
#define MSLK_SPLIT_KV_STATIC_BYTES (16u << 20)
mslk_status mslk_attn_split_kv_static(const mslk_attn_args* args, int32_t n_chunks, void* stream);
/* Bytes of workspace mslk_attn_split_kv needs for these arguments and chunk count; the
 * tensor pointers in args are not read and may be NULL (the other checks still apply). */
mslk_status mslk_attn_split_kv_workspace(const mslk_attn_args* args, int32_t n_chunks,
                                         size_t* bytes);

/*
 * Reason for the last non-OK status returned on the calling thread (like the pages'
 * not_supported_reasons).  Thread-local; valid until the thread's next library call.
 */
const char* mslk_last_error(void);

/*
 * Synchronises `stream`, then reads and clears the current device's error word.
 * Returns MSLK_ERR_DEVICE_TIMEOUT if any kernel since the last check gave up on a
 * bounded wait (the kernel then wrote nothing further and returned), MSLK_ERR_CUDA if
 * the synchronisation itself failed, else MSLK_OK.
 */
mslk_status mslk_device_status(void* stream);

/*
 * Sets the limit of every in-kernel wait, in nanoseconds (default 2e9; minimum 1e5).
 * Process-wide; read at launch time.
 */
void mslk_set_wait_timeout_ns(int64_t ns);

/*
 * Diagnostic: launches one CTA that waits on a barrier nothing ever completes, bounded by
 * the current wait limit, so callers can see the timeout path end cleanly.  Returns the
 * launch status; the timeout itself is reported by mslk_device_status().
 */
mslk_status mslk_diag_bounded_wait(void* stream);

/*
 * Kernel choice, process-wide: 0 automatic (default: for at most 8 query rows per batch
 * or packed sequence, the CUDA-core kernel unless a measured rate model says the
 * tensor-core kernel streams the keys faster — more rows, or E4M3 inputs, and enough
 * (batch, head) units; grouped heads with one query position go to the tensor cores with
 * enough units; paged lanes whose page size is not a multiple of 128 stay on the CUDA
 * cores; the tensor-core kernel otherwise), 1 always the tensor-core kernel, 2 the
 * CUDA-core kernel wherever it applies (at most 8 query rows).  All choices compute the
 * same function (E4M3 within the rounding stated at mslk_attn_fwd_fp8); tests use this
 * to run one problem through each kernel.
 */
void mslk_set_path_policy(int32_t policy);

/* Library version, major * 10000 + minor * 100 + patch. */
int32_t mslk_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MSLK_ATTN_H */
