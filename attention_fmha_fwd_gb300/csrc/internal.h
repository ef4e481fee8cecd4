// internal.h — launch descriptions shared by the C-ABI layer and the kernel files.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/mslk_attn.h"

namespace mslk {

// A validated attention problem (forward or partial), strides in elements.
struct AttnProblem {
  const void* q;
  const void* k;
  const void* v;
  mslk_strides sq, sk, sv, so;
  int B, M, Mkv, H, K, Kv;
  float scale;          // already defaulted (> 0)
  int mask_kind;
  const int32_t* cu_q;  // device, block-diagonal kinds only
  const int32_t* cu_k;
  int n_seqs, max_seqlen_q, max_seqlen_k;
  int64_t kv_offset;    // 0 for the forward call
  // Band of allowed keys: key position j (kv_offset added) is allowed for query row i
  // iff band_lo <= j - i <= band_hi (kBandOpen: that side open), plus, for block-diagonal
  // kinds with band_seq_shift, each sequence's Lk - Lq added to both bounds.
  int64_t band_lo, band_hi;
  bool band_seq_shift;
  // Key lanes (block-diagonal kinds only): per-sequence key count, first row (padded
  // lanes) or page table (paged lanes); lanes == false: keys come from cu_k.
  bool lanes;
  const int32_t* lane_len;
  const int32_t* lane_start;
  const int32_t* block_table;
  int page_size, max_pages;
  // E4M3 q/k/v: element x of head h stands for x * descale[h] (descale[0] when
  // descale_per_tensor); device fp32 arrays.
  bool fp8;
  const float* descale_q;
  const float* descale_k;
  const float* descale_v;
  bool descale_per_tensor;
  void* out;
  bool out_fp32;
  float* lse;           // may be null (forward without lse)
  // K/V heads: query head h reads K/V head h / kv_group (kv_group = H / Hkv).  A k/v head
  // stride of 0 is one shared head (Hkv = 1).
  int Hkv, kv_group;
  // > 1: one query position per batch / packed sequence, run on the tensor cores with the
  // kv_group query heads of a K/V head as the rows of one unit (set by the dispatcher).
  int fold;
  bool independent;  // MSLK_FLAG_INDEPENDENT: may overlap the preceding launch
};

// Most chunks one varargs merge takes (its pointer table travels as a kernel parameter).
constexpr int kMergeMaxVarargs = MSLK_MERGE_MAX_VARARGS;

struct MergeProblem {
  const float* out_split;
  const float* lse_split;
  // Varargs merge: chunk c's output and lse at chunk_out[c] / chunk_lse[c] (host arrays of
  // n_chunks device pointers); null for the stacked layout above.
  const float* const* chunk_out;
  const float* const* chunk_lse;
  int n_chunks;
  int64_t cs_out, cs_lse;
  int B, M, H, Kv;
  mslk_strides ss, so;
  void* out;
  bool out_fp32;
  float* lse;
};

// Where bounded in-kernel waits report, and how long they wait.
struct DeviceCtl {
  unsigned int* err;
  unsigned long long timeout_ns;
};

// Error-word bits.
constexpr unsigned int kErrWaitTimeout = 1u;

constexpr bool is_causal(int mask_kind) {
  return mask_kind == MSLK_MASK_CAUSAL || mask_kind == MSLK_MASK_BLOCKDIAG_CAUSAL ||
         mask_kind == MSLK_MASK_CAUSAL_BOTTOM_RIGHT || mask_kind == MSLK_MASK_BLOCKDIAG_CAUSAL_BOTTOM_RIGHT;
}
constexpr bool is_blockdiag(int mask_kind) {
  return mask_kind == MSLK_MASK_BLOCKDIAG || mask_kind == MSLK_MASK_BLOCKDIAG_CAUSAL ||
         mask_kind == MSLK_MASK_BLOCKDIAG_CAUSAL_BOTTOM_RIGHT;
}
constexpr bool is_bottom_right(int mask_kind) {
  return mask_kind == MSLK_MASK_CAUSAL_BOTTOM_RIGHT || mask_kind == MSLK_MASK_BLOCKDIAG_CAUSAL_BOTTOM_RIGHT;
}
// An open side of the key band (far beyond any int32 position difference).
constexpr int64_t kBandOpen = int64_t(1) << 40;

// Largest query-row count the CUDA-core decode kernel takes.
constexpr int kDecodeMaxRows = 8;
// Folded grouped heads on the tensor cores: at most one 256-row unit of heads, and at
// least this many (batch or sequence, K/V head) units (below it the CUDA-core kernel,
// which splits keys over thread-block clusters, fills the SMs better).
constexpr int kFoldMaxRows = 256;
constexpr long long kFoldMinUnits = 64;

// Tensor-core (tcgen05) forward/partial kernel.  `why` receives a reason on failure.
cudaError_t launch_fmha_tc(const AttnProblem& p, const DeviceCtl& ctl, cudaStream_t stream,
                           const char** why);
// CUDA-core streaming kernel for M <= kDecodeMaxRows with dense masks.
cudaError_t launch_fmha_decode(const AttnProblem& p, const DeviceCtl& ctl, cudaStream_t stream,
                               const char** why);
// out = 0, lse = -inf for every row (no keys at all).
cudaError_t launch_fill_empty(const AttnProblem& p, cudaStream_t stream);
// LSE merge.
cudaError_t launch_merge(const MergeProblem& p, const DeviceCtl& ctl, cudaStream_t stream);
// Diagnostic bounded wait on a barrier that never completes.
cudaError_t launch_bounded_wait_diag(const DeviceCtl& ctl, cudaStream_t stream);

}  // namespace mslk
