// mslk_attn.cu — the C ABI: argument validation with reasons, path selection, the
// per-device error word of the bounded in-kernel waits, and two small kernels
// (empty-key fill, bounded-wait diagnostic).
//
// Validation follows the pages' support checks (an operator's not_supported_reasons
// and check_lastdim_alignment_stride1): every rejection returns before any launch,
// writes nothing, and leaves its reason in mslk_last_error().

#include <cuda_bf16.h>

#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cmath>
#include <cstdio>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace mslk {
namespace {

thread_local char g_last_error[512] = "";
std::atomic<long long> g_timeout_ns{2000000000LL};

// 0 = automatic, 1 = always the tensor-core kernel, 2 = the decode kernel where it applies.
std::atomic<int> g_path_policy{0};

mslk_status fail(mslk_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
mslk_status fail(mslk_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return s;
}

mslk_status ok() {
  g_last_error[0] = '\0';
  return MSLK_OK;
}

__device__ unsigned int g_error_word;

// Device address of g_error_word for the current device (looked up once per device).
unsigned int* error_word_ptr() {
  constexpr int kMaxDevices = 64;
  static unsigned int* ptrs[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (ptrs[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<unsigned int*>(p);
  }
  return ptrs[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Stride rule for tensors read by TMA or written with 16-byte vectors: every stride of a
// dimension with extent > 1 is a positive multiple of `mult` elements.  A stride of 0 is
// allowed on the head dimension of k/v when `allow_zero_head`.
const char* check_strides(const mslk_strides& s, long long batch, long long rows, long long heads,
                          int mult, bool allow_zero_head) {
  if (s.b < 0 || s.m < 0 || s.h < 0) return "negative stride";
  if (batch > 1 && (s.b == 0 || s.b % mult)) return "batch stride";
  if (rows > 1 && (s.m == 0 || s.m % mult)) return "sequence stride";
  if (heads > 1) {
    if (s.h == 0 && !allow_zero_head) return "head stride";
    if (s.h % mult) return "head stride";
  }
  return nullptr;
}

mslk_status validate_attn(AttnProblem& p, const void* q, const void* k, const void* v,
                          const mslk_strides* sq, const mslk_strides* sk, const mslk_strides* sv,
                          const mslk_strides* so, int32_t B, int32_t M, int32_t Mkv, int32_t H,
                          int32_t K, int32_t Kv, float scale, int32_t mask_kind,
                          const mslk_seqlens* seqlens, const mslk_band* band, int64_t kv_offset,
                          void* out, int32_t out_dtype, float* lse, bool lse_required,
                          bool partial, const char* who, int in_bytes = 2, int32_t Hkv = 0) {
  if (B < 0 || M < 0 || Mkv < 0 || H < 0) return fail(MSLK_ERR_INVALID_ARG, "%s: negative size", who);
  if (mask_kind < MSLK_MASK_NONE || mask_kind > MSLK_MASK_BLOCKDIAG_CAUSAL_BOTTOM_RIGHT)
    return fail(MSLK_ERR_INVALID_ARG, "%s: unknown mask_kind %d", who, mask_kind);
  const int32_t wl = band ? band->window_left : -1;
  const int32_t wr = band ? band->window_right : -1;
  if (band && band->bottom_right != 0 && band->bottom_right != 1)
    return fail(MSLK_ERR_INVALID_ARG, "%s: band.bottom_right must be 0 or 1", who);
  if (wl < -1 || wr < -1)
    return fail(MSLK_ERR_INVALID_ARG, "%s: window sizes must be >= 0 (or -1 for unbounded)", who);
  if (is_causal(mask_kind) && wr > 0)
    return fail(MSLK_ERR_INVALID_ARG, "%s: causal masks have no right window (window_right %d)", who, wr);
  const bool bottom_right = is_bottom_right(mask_kind) || (band && band->bottom_right);
  if (partial && bottom_right)
    return fail(MSLK_ERR_INVALID_ARG,
                "%s: bottom-right alignment is forward only; fold Lk_full - M into kv_offset", who);
  if (out_dtype != MSLK_DTYPE_BF16 && out_dtype != MSLK_DTYPE_FP32)
    return fail(MSLK_ERR_INVALID_ARG, "%s: unknown out_dtype %d", who, out_dtype);
  if (sq == nullptr || sk == nullptr || sv == nullptr || so == nullptr)
    return fail(MSLK_ERR_INVALID_ARG, "%s: null strides", who);
  if (K != Kv)
    return fail(MSLK_ERR_UNSUPPORTED, "%s: K (%d) != Kv (%d) is not supported", who, K, Kv);
  if (K != 64 && K != 96 && K != 128)
    return fail(MSLK_ERR_UNSUPPORTED, "%s: head dim %d not supported (64, 96 or 128)", who, K);
  p = AttnProblem{};
  p.q = q;
  p.k = k;
  p.v = v;
  p.sq = *sq;
  p.sk = *sk;
  p.sv = *sv;
  p.so = *so;
  p.B = B;
  p.M = M;
  p.Mkv = Mkv;
  p.H = H;
  p.K = K;
  p.Kv = Kv;
  p.scale = (scale > 0.f && std::isfinite(scale)) ? scale : 1.0f / std::sqrt(static_cast<float>(K));
  p.mask_kind = mask_kind;
  p.kv_offset = kv_offset;
  p.Hkv = H;
  p.kv_group = 1;
  // Band on (key position - query row): causal kinds close it at 0, windows at -wl / +wr;
  // a dense bottom-right alignment shifts both bounds by Mkv - M, a block-diagonal one by
  // each sequence's Lk - Lq (added in the kernels).
  p.band_hi = is_causal(mask_kind) ? 0 : (wr >= 0 ? wr : kBandOpen);
  p.band_lo = wl >= 0 ? -static_cast<int64_t>(wl) : -kBandOpen;
  p.band_seq_shift = bottom_right && is_blockdiag(mask_kind);
  if (bottom_right && !is_blockdiag(mask_kind)) {
    const int64_t shift = static_cast<int64_t>(Mkv) - M;
    if (p.band_hi != kBandOpen) p.band_hi += shift;
    if (p.band_lo != -kBandOpen) p.band_lo += shift;
  }
  p.out = out;
  p.out_fp32 = out_dtype == MSLK_DTYPE_FP32;
  p.lse = lse;
  if (B == 0 || H == 0 || M == 0) return ok();  // nothing to compute
  if (out == nullptr) return fail(MSLK_ERR_INVALID_ARG, "%s: out is null", who);
  if (lse_required && lse == nullptr) return fail(MSLK_ERR_INVALID_ARG, "%s: lse is required", who);
  if (is_blockdiag(mask_kind)) {
    if (B != 1)
      return fail(MSLK_ERR_INVALID_ARG, "%s: block-diagonal masks take a packed batch (B = 1), got B = %d",
                  who, B);
    if (seqlens == nullptr || seqlens->cu_seqlens_q == nullptr || seqlens->cu_seqlens_k == nullptr)
      return fail(MSLK_ERR_INVALID_ARG, "%s: block-diagonal mask needs cu_seqlens_q/k", who);
    if (seqlens->n_seqs < 1 || seqlens->max_seqlen_q < 1 || seqlens->max_seqlen_q > M ||
        seqlens->max_seqlen_k < 0 || seqlens->max_seqlen_k > Mkv)
      return fail(MSLK_ERR_INVALID_ARG, "%s: bad seqlens (n_seqs %d, max_seqlen_q %d, max_seqlen_k %d)",
                  who, seqlens->n_seqs, seqlens->max_seqlen_q, seqlens->max_seqlen_k);
    p.cu_q = seqlens->cu_seqlens_q;
    p.cu_k = seqlens->cu_seqlens_k;
    p.n_seqs = seqlens->n_seqs;
    p.max_seqlen_q = seqlens->max_seqlen_q;
    p.max_seqlen_k = seqlens->max_seqlen_k;
  }
  if (Mkv == 0) return ok();  // every row empty; q/k/v are not read
  if (q == nullptr || k == nullptr || v == nullptr)
    return fail(MSLK_ERR_INVALID_ARG, "%s: q/k/v is null", who);
  if ((sk->h == 0) != (sv->h == 0) && H > 1)
    return fail(MSLK_ERR_INVALID_ARG, "%s: k and v must both or neither use a shared (stride 0) head", who);
  // K/V heads: Hkv (0: as many as H), or one shared head when the k/v head stride is 0.
  if (Hkv == 0) Hkv = H;
  if (H > 1 && sk->h == 0) Hkv = 1;
  if (Hkv < 1 || H % Hkv)
    return fail(MSLK_ERR_INVALID_ARG, "%s: K/V heads (%d) must divide the query heads (%d)", who, Hkv, H);
  p.Hkv = Hkv;
  p.kv_group = H / Hkv;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v))
    return fail(MSLK_ERR_MISALIGNED, "%s: q/k/v base must be 16-byte aligned", who);
  const int in_mult = 16 / in_bytes;  // elements per 16 bytes
  if (const char* w = check_strides(*sq, B, M, H, in_mult, false))
    return fail(MSLK_ERR_MISALIGNED, "%s: q %s must be a positive multiple of %d elements (16 bytes)", who, w, in_mult);
  if (const char* w = check_strides(*sk, B, Mkv, Hkv, in_mult, true))
    return fail(MSLK_ERR_MISALIGNED, "%s: k %s must be a positive multiple of %d elements (16 bytes)", who, w, in_mult);
  if (const char* w = check_strides(*sv, B, Mkv, Hkv, in_mult, true))
    return fail(MSLK_ERR_MISALIGNED, "%s: v %s must be a positive multiple of %d elements (16 bytes)", who, w, in_mult);
  if (!aligned16(out)) return fail(MSLK_ERR_MISALIGNED, "%s: out base must be 16-byte aligned", who);
  if (const char* w = check_strides(*so, B, M, H, p.out_fp32 ? 4 : 8, false))
    return fail(MSLK_ERR_MISALIGNED, "%s: out %s must be a positive multiple of 16 bytes", who, w);
  if ((reinterpret_cast<uintptr_t>(lse) & 3u) != 0)
    return fail(MSLK_ERR_MISALIGNED, "%s: lse must be 4-byte aligned", who);
  if (kv_offset < -(1LL << 31) || kv_offset > (1LL << 31))
    return fail(MSLK_ERR_INVALID_ARG, "%s: kv_offset out of range", who);
  return ok();
}

__global__ void fill_empty_kernel(void* out, int out_fp32, long long so_b, long long so_m,
                                  long long so_h, float* lse, int B, int M, int H, int D) {
  const long long n = static_cast<long long>(B) * M * H;
  for (long long r = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; r < n;
       r += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int h = static_cast<int>(r % H);
    const int m = static_cast<int>((r / H) % M);
    const int b = static_cast<int>(r / (static_cast<long long>(H) * M));
    for (int c = 0; c < D; ++c) {
      const long long off = b * so_b + m * so_m + h * so_h + c;
      if (out_fp32)
        static_cast<float*>(out)[off] = 0.f;
      else
        static_cast<__nv_bfloat16*>(out)[off] = __float2bfloat16(0.f);
    }
    if (lse != nullptr) lse[(static_cast<long long>(b) * H + h) * M + m] = -INFINITY;
  }
}

// One thread waits, bounded, on a barrier that nothing completes.
__global__ void bounded_wait_diag_kernel(unsigned int* err, unsigned long long timeout_ns) {
  __shared__ uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 1);
  fence_mbar_init();
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(b, 0)) {
    if (globaltimer_ns() - t0 > timeout_ns) {
      atomicOr(err, kErrWaitTimeout);
      break;
    }
  }
}

DeviceCtl device_ctl() {
  return DeviceCtl{error_word_ptr(), static_cast<unsigned long long>(g_timeout_ns.load())};
}

// Few query rows: the CUDA-core kernel splits each head's keys over a thread-block cluster
// but its work grows with the rows; the tensor-core kernel pays the same per key tile for 1
// to 128 rows but streams one (batch, head) unit per CTA (both softmax warpgroups on it).
// Rates measured on GB300 (keys per second): tensor cores min(memory rate, ~1.7e8 per
// unit); CUDA cores min(memory rate, ~1.9e10 / rows) — e.g. 16 x 8 heads x 32768 keys at 8
// rows: 351 vs 1817 us; at 1 row bf16 stays on the CUDA cores (323 vs 330 us) and E4M3
// goes to the tensor cores (202 vs 221 us).
bool few_rows_prefer_tensor_cores(int rows, long long units, int K, bool fp8) {
  const double bytes_per_key = (fp8 ? 2.0 : 4.0) * K;  // k + v
  // (a few rows fit one Q tile: the split units' two softmax warpgroups share the keys)
  const double tc = std::min(6.2e12 / bytes_per_key, static_cast<double>(units) * 1.7e8);
  const double cc = std::min(6.6e12 / bytes_per_key, 1.9e10 / rows);
  return tc > 1.05 * cc;
}

// Which kernel a validated problem runs on (MSLK_PLAN_* bits), from the problem and the
// path policy alone (no device access): run_attn launches what this returns.
int32_t choose_path(const AttnProblem& p, int policy) {
  if (p.B == 0 || p.H == 0 || p.M == 0) return MSLK_PLAN_NONE;
  if (p.Mkv == 0) return MSLK_PLAN_FILL;
  const int rows_q = is_blockdiag(p.mask_kind) ? p.max_seqlen_q : p.M;
  const long long units = static_cast<long long>(is_blockdiag(p.mask_kind) ? p.n_seqs : p.B) * p.H;
  // The tensor-core kernel reads 128-key tiles, each inside one page: pages of another
  // size (accepted for few rows, which the CUDA-core kernel reads) keep few rows there.
  const bool tc_pages_ok = p.block_table == nullptr || p.page_size % 128 == 0;
  const bool decode_ok = rows_q <= kDecodeMaxRows &&
                         (policy == 2 || !tc_pages_ok ||
                          !few_rows_prefer_tensor_cores(rows_q, units, p.K, p.fp8));
  // Grouped heads with one query position per batch / sequence: the tensor cores take the
  // group's query heads as the rows of one unit and stream each K/V head once at the
  // memory rate (the CUDA-core kernel's cost grows with the rows), when there are enough
  // (batch, K/V head) units to fill the SMs.
  const long long fold_units = static_cast<long long>(is_blockdiag(p.mask_kind) ? p.n_seqs : p.B) * p.Hkv;
  const bool fold = p.kv_group > 1 && rows_q == 1 && p.kv_group <= kFoldMaxRows &&
                    policy != 2 && tc_pages_ok &&
                    (policy == 1 || fold_units >= kFoldMinUnits);
  if (!fold && decode_ok && policy != 1) return MSLK_PLAN_CUDA_CORES;
  // tensor cores: split units when every unit's rows fit one 128-row Q tile
  const int rows = fold ? p.kv_group : rows_q;
  return MSLK_PLAN_TENSOR_CORES | (fold ? MSLK_PLAN_FOLDED_HEADS : 0) |
         (rows <= 128 ? MSLK_PLAN_SPLIT_UNITS : 0);
}

mslk_status run_attn(const AttnProblem& p, cudaStream_t stream, const char* who) {
  if (p.B == 0 || p.H == 0 || p.M == 0) return ok();
  if (p.Mkv == 0) {
    fill_empty_kernel<<<256, 256, 0, stream>>>(p.out, p.out_fp32 ? 1 : 0, p.so.b, p.so.m, p.so.h,
                                              p.lse, p.B, p.M, p.H, p.Kv);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(MSLK_ERR_CUDA, "%s: %s", who, cudaGetErrorString(e));
    return ok();
  }
  const DeviceCtl ctl = device_ctl();
  if (ctl.err == nullptr) return fail(MSLK_ERR_CUDA, "%s: no CUDA device / module", who);
  const int32_t plan = choose_path(p, g_path_policy.load());
  cudaError_t e;
  const char* why = "launch failed";
  if (plan & MSLK_PLAN_FOLDED_HEADS) {
    AttnProblem f = p;
    f.fold = p.kv_group;
    e = launch_fmha_tc(f, ctl, stream, &why);
  } else if (plan == MSLK_PLAN_CUDA_CORES) {
    e = launch_fmha_decode(p, ctl, stream, &why);
  } else {
    e = launch_fmha_tc(p, ctl, stream, &why);
  }
  if (e != cudaSuccess) return fail(MSLK_ERR_CUDA, "%s: %s (%s)", who, why, cudaGetErrorString(e));
  return ok();
}

}  // namespace
}  // namespace mslk

using namespace mslk;

namespace {

// The key-lane descriptor on its own (before the problem is validated).
mslk_status check_lanes(const mslk_kv_lanes* lanes, int32_t mask_kind, const char* who) {
  if (!is_blockdiag(mask_kind))
    return fail(MSLK_ERR_INVALID_ARG, "%s: key lanes need a block-diagonal mask kind (got %d)", who, mask_kind);
  if (lanes == nullptr || lanes->seqlen_k == nullptr)
    return fail(MSLK_ERR_INVALID_ARG, "%s: lanes->seqlen_k is required", who);
  if (lanes->block_table != nullptr) {
    if (lanes->page_size <= 0 || lanes->max_pages <= 0)
      return fail(MSLK_ERR_INVALID_ARG, "%s: paged lanes need page_size > 0 and max_pages > 0", who);
  } else if (lanes->seqstart_k == nullptr) {
    return fail(MSLK_ERR_INVALID_ARG, "%s: lanes need seqstart_k or block_table", who);
  }
  return ok();
}

// cu_seqlens_k is not read for lanes: validation only needs a non-null pointer there.
mslk_seqlens lanes_seqlens(const mslk_seqlens* seqlens, const mslk_kv_lanes* lanes) {
  mslk_seqlens sl{};
  if (seqlens != nullptr) {
    sl = *seqlens;
    if (sl.cu_seqlens_k == nullptr) sl.cu_seqlens_k = lanes->seqlen_k;
  }
  return sl;
}

// Lanes on a validated problem: a key tile never straddles a page (the decode kernel's
// tiles hold 8192 / (K * element bytes) keys, the tensor-core kernel's 128).
mslk_status apply_lanes(AttnProblem& p, const mslk_kv_lanes* lanes, const char* who) {
  if (lanes->block_table != nullptr) {
    const bool decode = p.max_seqlen_q <= kDecodeMaxRows && g_path_policy.load() != 1;
    const int width = p.K > 64 ? 128 : 64;  // the decode kernel's head-dim width
    const int multiple = decode ? (p.fp8 ? 8192 / width : 64) : 128;
    if (lanes->page_size % multiple)
      return fail(MSLK_ERR_UNSUPPORTED, "%s: page_size %d must be a multiple of %d", who,
                  lanes->page_size, multiple);
  }
  p.lanes = true;
  p.lane_len = lanes->seqlen_k;
  p.lane_start = lanes->seqstart_k;
  p.block_table = lanes->block_table;
  p.page_size = lanes->page_size;
  p.max_pages = lanes->max_pages;
  p.cu_k = nullptr;
  return ok();
}

mslk_attn_args make_args(const void* q, const void* k, const void* v, const mslk_strides& sq,
                         const mslk_strides& sk, const mslk_strides& sv, const mslk_strides& so,
                         int32_t B, int32_t M, int32_t Mkv, int32_t H, int32_t K, int32_t Kv,
                         float scale, int32_t mask_kind, const mslk_seqlens* seqlens,
                         const mslk_band* band, void* out, float* lse) {
  mslk_attn_args a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.sq = sq;
  a.sk = sk;
  a.sv = sv;
  a.so = so;
  a.B = B;
  a.M = M;
  a.Mkv = Mkv;
  a.H = H;
  a.Hkv = 0;
  a.K = K;
  a.Kv = Kv;
  a.scale = scale;
  a.mask_kind = mask_kind;
  a.seqlens = seqlens;
  a.band = band;
  a.out = out;
  a.out_dtype = MSLK_DTYPE_BF16;
  a.lse = lse;
  return a;
}

// Every option of the forward / partial call: validation, then the kernels.
mslk_status attn_general(const mslk_attn_args& a, cudaStream_t stream, const char* who,
                         int32_t* plan = nullptr) {
  const mslk_fp8_scales* f8 = a.fp8;
  if (f8 != nullptr) {
    if (f8->descale_q == nullptr || f8->descale_k == nullptr || f8->descale_v == nullptr)
      return fail(MSLK_ERR_INVALID_ARG, "%s: descale_q, descale_k and descale_v are required", who);
    if (f8->per_tensor != 0 && f8->per_tensor != 1)
      return fail(MSLK_ERR_INVALID_ARG, "%s: scales.per_tensor must be 0 or 1", who);
    if ((reinterpret_cast<uintptr_t>(f8->descale_q) | reinterpret_cast<uintptr_t>(f8->descale_k) |
         reinterpret_cast<uintptr_t>(f8->descale_v)) & 3u)
      return fail(MSLK_ERR_MISALIGNED, "%s: descales must be 4-byte aligned", who);
  }
  if (a.partial != 0 && a.partial != 1)
    return fail(MSLK_ERR_INVALID_ARG, "%s: partial must be 0 or 1", who);
  if (a.flags & ~MSLK_FLAG_INDEPENDENT)
    return fail(MSLK_ERR_INVALID_ARG, "%s: unknown flags %#x", who, a.flags);
  if (a.Hkv < 0) return fail(MSLK_ERR_INVALID_ARG, "%s: negative Hkv", who);
  mslk_status s = ok();
  mslk_seqlens sl{};
  const mslk_seqlens* slp = a.seqlens;
  if (a.lanes != nullptr) {
    if (a.partial) return fail(MSLK_ERR_UNSUPPORTED, "%s: key lanes are forward only", who);
    s = check_lanes(a.lanes, a.mask_kind, who);
    if (s != MSLK_OK) return s;
    if (a.B != 1)
      return fail(MSLK_ERR_INVALID_ARG, "%s: key lanes take packed queries (B = 1), got B = %d", who, a.B);
    sl = lanes_seqlens(a.seqlens, a.lanes);
    slp = a.seqlens ? &sl : nullptr;
  }
  AttnProblem p;
  s = validate_attn(p, a.q, a.k, a.v, &a.sq, &a.sk, &a.sv, &a.so, a.B, a.M, a.Mkv, a.H, a.K, a.Kv,
                    a.scale, a.mask_kind, slp, a.band, a.partial ? a.kv_offset : 0, a.out,
                    a.out_dtype, a.lse, a.partial == 1, a.partial == 1, who, f8 ? 1 : 2, a.Hkv);
  if (s != MSLK_OK) return s;
  p.independent = (a.flags & MSLK_FLAG_INDEPENDENT) != 0;
  if (f8 != nullptr) {
    p.fp8 = true;
    p.descale_q = f8->descale_q;
    p.descale_k = f8->descale_k;
    p.descale_v = f8->descale_v;
    p.descale_per_tensor = f8->per_tensor == 1;
  }
  if (a.lanes != nullptr) {
    s = apply_lanes(p, a.lanes, who);
    if (s != MSLK_OK) return s;
  }
  if (plan != nullptr) {
    *plan = choose_path(p, g_path_policy.load());
    return ok();
  }
  return run_attn(p, stream, who);
}

// The checks every merge entry shares (sizes, dtype, strides, out and lse); fills the
// problem's common fields.  B, M or H == 0 returns MSLK_OK with nothing to do.
mslk_status validate_merge(MergeProblem& p, int32_t n_chunks, int32_t B, int32_t M, int32_t H,
                           int32_t Kv, const mslk_strides* s_split, const mslk_strides* so,
                           void* out, int32_t out_dtype, float* lse, const char* who) {
  if (n_chunks < 1) return fail(MSLK_ERR_INVALID_ARG, "%s: n_chunks must be >= 1 (got %d)", who, n_chunks);
  if (B < 0 || M < 0 || H < 0 || Kv < 0) return fail(MSLK_ERR_INVALID_ARG, "%s: negative size", who);
  if (out_dtype != MSLK_DTYPE_BF16 && out_dtype != MSLK_DTYPE_FP32)
    return fail(MSLK_ERR_INVALID_ARG, "%s: unknown out_dtype %d", who, out_dtype);
  if (s_split == nullptr || so == nullptr) return fail(MSLK_ERR_INVALID_ARG, "%s: null strides", who);
  if (B == 0 || M == 0 || H == 0) return ok();
  if (Kv == 0 || Kv % 4) return fail(MSLK_ERR_UNSUPPORTED, "%s: Kv (%d) must be a positive multiple of 4", who, Kv);
  if (out == nullptr) return fail(MSLK_ERR_INVALID_ARG, "%s: null pointer", who);
  if (!aligned16(out)) return fail(MSLK_ERR_MISALIGNED, "%s: out_split/out must be 16-byte aligned", who);
  if ((reinterpret_cast<uintptr_t>(lse) & 3u) != 0)
    return fail(MSLK_ERR_MISALIGNED, "%s: lse_split/lse must be 4-byte aligned", who);
  if (const char* w = check_strides(*s_split, B, M, H, 4, false))
    return fail(MSLK_ERR_MISALIGNED, "%s: out_split %s must be a positive multiple of 4 elements", who, w);
  const bool out_fp32 = out_dtype == MSLK_DTYPE_FP32;
  if (const char* w = check_strides(*so, B, M, H, out_fp32 ? 4 : 8, false))
    return fail(MSLK_ERR_MISALIGNED, "%s: out %s must be a positive multiple of 16 bytes", who, w);
  p.n_chunks = n_chunks;
  p.B = B;
  p.M = M;
  p.H = H;
  p.Kv = Kv;
  p.ss = *s_split;
  p.so = *so;
  p.out = out;
  p.out_fp32 = out_fp32;
  p.lse = lse;
  return ok();
}

mslk_status run_merge(const MergeProblem& p, cudaStream_t stream, const char* who) {
  const DeviceCtl ctl = device_ctl();
  if (ctl.err == nullptr) return fail(MSLK_ERR_CUDA, "%s: no CUDA device / module", who);
  const cudaError_t e = launch_merge(p, ctl, stream);
  if (e != cudaSuccess) return fail(MSLK_ERR_CUDA, "%s: %s", who, cudaGetErrorString(e));
  return ok();
}

int current_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 148;
  return n;
}

// Keys per split (a multiple of tile_n) so that every (batch, K/V head) unit gets enough
// splits for one (unit, split) pair per SM; 0 when one split covers the keys.
int32_t splitk_size(int32_t batch, int32_t seqlen_kv, int32_t kv_heads, int32_t tile_n,
                    int32_t sm_count) {
  if (batch <= 0 || seqlen_kv <= 0 || kv_heads <= 0) return 0;
  if (tile_n <= 0) tile_n = 256;
  if (sm_count <= 0) sm_count = current_sm_count();
  const long long units = static_cast<long long>(batch) * kv_heads;
  const long long splits = std::max(1LL, (sm_count + units - 1) / units);
  long long size = (seqlen_kv + splits - 1) / splits;
  size = (size + tile_n - 1) / tile_n * tile_n;
  return size >= seqlen_kv ? 0 : static_cast<int32_t>(size);
}

// Chunk count of a split-KV call: the caller's, or from splitk_size; at most one per key.
int32_t split_chunks(const mslk_attn_args& a, int32_t n_chunks) {
  if (n_chunks <= 0) {
    const int32_t hkv = a.Hkv > 0 ? a.Hkv : ((a.H > 1 && a.sk.h == 0) ? 1 : a.H);
    const int32_t size = splitk_size(a.B, a.Mkv, hkv, 256, 0);
    n_chunks = size == 0 ? 1 : (a.Mkv + size - 1) / size;
  }
  return std::max(1, std::min(n_chunks, std::max(1, a.Mkv)));
}

// Workspace of a split-KV call: the chunks' fp32 outputs [n, B, M, H, Kv] (contiguous),
// then their lse [n, B, H, M]; the lse block starts on a 256-byte boundary.
struct SplitLayout {
  size_t out_chunk_elems, lse_chunk_elems, lse_offset, bytes;
};
SplitLayout split_layout(const mslk_attn_args& a, int32_t n) {
  SplitLayout l{};
  l.out_chunk_elems = static_cast<size_t>(a.B) * a.M * a.H * a.Kv;
  l.lse_chunk_elems = static_cast<size_t>(a.B) * a.H * a.M;
  l.lse_offset = (static_cast<size_t>(n) * l.out_chunk_elems * sizeof(float) + 255) / 256 * 256;
  l.bytes = l.lse_offset + static_cast<size_t>(n) * l.lse_chunk_elems * sizeof(float);
  return l;
}

// The arguments a split-KV call accepts, checked before anything is launched: those of the
// forward call (validated by planning it), dense masks only, no key lanes.
mslk_status check_split_args(const mslk_attn_args* a, int32_t n_chunks, const char* who) {
  if (a == nullptr) return fail(MSLK_ERR_INVALID_ARG, "%s: args is null", who);
  if (a->partial != 0) return fail(MSLK_ERR_INVALID_ARG, "%s: args must describe a forward (partial = 0)", who);
  if (a->lanes != nullptr) return fail(MSLK_ERR_UNSUPPORTED, "%s: key lanes are not split", who);
  if (is_blockdiag(a->mask_kind))
    return fail(MSLK_ERR_UNSUPPORTED, "%s: block-diagonal masks are not split (dense masks only)", who);
  if (a->fp8 != nullptr) return fail(MSLK_ERR_UNSUPPORTED, "%s: E4M3 inputs are not split (bf16 only)", who);
  if (n_chunks < 0) return fail(MSLK_ERR_INVALID_ARG, "%s: n_chunks must be >= 0 (got %d)", who, n_chunks);
  int32_t plan = 0;
  return attn_general(*a, nullptr, who, &plan);
}

// Partials over n equal contiguous key chunks into the workspace, then the merge into
// args.out / args.lse.  Chunk c > 0 is launched independent of chunk c - 1 (they read the
// same q, k, v and write separate workspace slices); the merge waits for all of them.
mslk_status run_split_kv(const mslk_attn_args& a, int32_t n, float* ws_out, float* ws_lse,
                         cudaStream_t stream, const char* who) {
  const SplitLayout l = split_layout(a, n);
  const int esz = 2;  // bf16 keys and values
  const bool br = is_bottom_right(a.mask_kind) || (a.band != nullptr && a.band->bottom_right);
  // A bottom-right alignment is a shift of the key positions: folded into kv_offset.
  const int64_t shift = br ? static_cast<int64_t>(a.Mkv) - a.M : 0;
  mslk_band band{0, -1, -1};
  if (a.band != nullptr) band = *a.band;
  band.bottom_right = 0;
  const mslk_strides s_ws{static_cast<int64_t>(a.M) * a.H * a.Kv, static_cast<int64_t>(a.H) * a.Kv, a.Kv};
  for (int32_t c = 0; c < n; ++c) {
    const int32_t k0 = static_cast<int32_t>(static_cast<int64_t>(c) * a.Mkv / n);
    const int32_t k1 = static_cast<int32_t>(static_cast<int64_t>(c + 1) * a.Mkv / n);
    mslk_attn_args ca = a;
    ca.k = static_cast<const uint8_t*>(a.k) + static_cast<int64_t>(k0) * a.sk.m * esz;
    ca.v = static_cast<const uint8_t*>(a.v) + static_cast<int64_t>(k0) * a.sv.m * esz;
    ca.Mkv = k1 - k0;
    ca.mask_kind = a.mask_kind == MSLK_MASK_CAUSAL_BOTTOM_RIGHT ? MSLK_MASK_CAUSAL : a.mask_kind;
    ca.band = &band;
    ca.partial = 1;
    ca.kv_offset = k0 - shift;
    ca.out = ws_out + c * l.out_chunk_elems;
    ca.so = s_ws;
    ca.out_dtype = MSLK_DTYPE_FP32;
    ca.lse = ws_lse + c * l.lse_chunk_elems;
    ca.flags = c > 0 ? MSLK_FLAG_INDEPENDENT : (a.flags & MSLK_FLAG_INDEPENDENT);
    const mslk_status s = attn_general(ca, stream, who);
    if (s != MSLK_OK) return s;
  }
  MergeProblem m{};
  mslk_status s = validate_merge(m, n, a.B, a.M, a.H, a.Kv, &s_ws, &a.so, a.out, a.out_dtype, a.lse, who);
  if (s != MSLK_OK) return s;
  m.out_split = ws_out;
  m.lse_split = ws_lse;
  m.cs_out = static_cast<int64_t>(l.out_chunk_elems);
  m.cs_lse = static_cast<int64_t>(l.lse_chunk_elems);
  return run_merge(m, stream, who);
}

// Workspace of mslk_attn_split_kv_static: a fixed array in every device that loads the
// library, held until the process exits.  Host code cannot use the array's name as a
// device address; split_static_workspace() looks the address up (cudaGetSymbolAddress)
// the first time it runs on each device, with that device current.
static __device__ __align__(256) unsigned char g_split_static[MSLK_SPLIT_KV_STATIC_BYTES];

float* split_static_workspace(cudaError_t* err) {
  constexpr int kMaxDevices = 64;
  static float* ptrs[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kMaxDevices) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (ptrs[dev] == nullptr) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_split_static);
    if (*err != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<float*>(p);
  }
  return ptrs[dev];
}

}  // namespace

extern "C" {

mslk_status mslk_attn_fwd(const void* q, const void* k, const void* v, const mslk_strides* sq,
                          const mslk_strides* sk, const mslk_strides* sv, const mslk_strides* so,
                          int32_t B, int32_t M, int32_t Mkv, int32_t H, int32_t K, int32_t Kv,
                          float scale, int32_t mask_kind, const mslk_seqlens* seqlens, void* out,
                          float* lse, void* stream) {
  AttnProblem p;
  const mslk_status s = validate_attn(p, q, k, v, sq, sk, sv, so, B, M, Mkv, H, K, Kv, scale,
                                      mask_kind, seqlens, nullptr, 0, out, MSLK_DTYPE_BF16, lse,
                                      false, false, "mslk_attn_fwd");
  if (s != MSLK_OK) return s;
  return run_attn(p, static_cast<cudaStream_t>(stream), "mslk_attn_fwd");
}

mslk_status mslk_attn_partial(const void* q, const void* k, const void* v, const mslk_strides* sq,
                              const mslk_strides* sk, const mslk_strides* sv, const mslk_strides* so,
                              int32_t B, int32_t M, int32_t Mkv, int32_t H, int32_t K, int32_t Kv,
                              float scale, int32_t mask_kind, const mslk_seqlens* seqlens,
                              int64_t kv_offset, void* out, int32_t out_dtype, float* lse,
                              void* stream) {
  AttnProblem p;
  const mslk_status s = validate_attn(p, q, k, v, sq, sk, sv, so, B, M, Mkv, H, K, Kv, scale,
                                      mask_kind, seqlens, nullptr, kv_offset, out, out_dtype, lse,
                                      true, true, "mslk_attn_partial");
  if (s != MSLK_OK) return s;
  return run_attn(p, static_cast<cudaStream_t>(stream), "mslk_attn_partial");
}

mslk_status mslk_attn_fwd_band(const void* q, const void* k, const void* v, const mslk_strides* sq,
                               const mslk_strides* sk, const mslk_strides* sv, const mslk_strides* so,
                               int32_t B, int32_t M, int32_t Mkv, int32_t H, int32_t K, int32_t Kv,
                               float scale, int32_t mask_kind, const mslk_seqlens* seqlens,
                               const mslk_band* band, void* out, float* lse, void* stream) {
  AttnProblem p;
  const mslk_status s = validate_attn(p, q, k, v, sq, sk, sv, so, B, M, Mkv, H, K, Kv, scale,
                                      mask_kind, seqlens, band, 0, out, MSLK_DTYPE_BF16, lse, false,
                                      false, "mslk_attn_fwd_band");
  if (s != MSLK_OK) return s;
  return run_attn(p, static_cast<cudaStream_t>(stream), "mslk_attn_fwd_band");
}

mslk_status mslk_attn_partial_band(const void* q, const void* k, const void* v,
                                   const mslk_strides* sq, const mslk_strides* sk,
                                   const mslk_strides* sv, const mslk_strides* so, int32_t B,
                                   int32_t M, int32_t Mkv, int32_t H, int32_t K, int32_t Kv,
                                   float scale, int32_t mask_kind, const mslk_seqlens* seqlens,
                                   const mslk_band* band, int64_t kv_offset, void* out,
                                   int32_t out_dtype, float* lse, void* stream) {
  AttnProblem p;
  const mslk_status s = validate_attn(p, q, k, v, sq, sk, sv, so, B, M, Mkv, H, K, Kv, scale,
                                      mask_kind, seqlens, band, kv_offset, out, out_dtype, lse,
                                      true, true, "mslk_attn_partial_band");
  if (s != MSLK_OK) return s;
  return run_attn(p, static_cast<cudaStream_t>(stream), "mslk_attn_partial_band");
}

mslk_status mslk_attn_plan(const mslk_attn_args* args, int32_t* plan) {
  const char* who = "mslk_attn_plan";
  if (args == nullptr || plan == nullptr) return fail(MSLK_ERR_INVALID_ARG, "%s: args and plan are required", who);
  return attn_general(*args, nullptr, who, plan);
}

mslk_status mslk_attn(const mslk_attn_args* args, void* stream) {
  const char* who = "mslk_attn";
  if (args == nullptr) return fail(MSLK_ERR_INVALID_ARG, "%s: args is null", who);
  return attn_general(*args, static_cast<cudaStream_t>(stream), who);
}

mslk_status mslk_attn_fwd_lanes(const void* q, const void* k, const void* v, const mslk_strides* sq,
                                const mslk_strides* sk, const mslk_strides* sv, const mslk_strides* so,
                                int32_t M, int32_t Mkv, int32_t H, int32_t K, int32_t Kv, float scale,
                                int32_t mask_kind, const mslk_seqlens* seqlens,
                                const mslk_kv_lanes* lanes, const mslk_band* band, void* out,
                                float* lse, void* stream) {
  const char* who = "mslk_attn_fwd_lanes";
  if (sq == nullptr || sk == nullptr || sv == nullptr || so == nullptr)
    return fail(MSLK_ERR_INVALID_ARG, "%s: null strides", who);
  if (lanes == nullptr) return fail(MSLK_ERR_INVALID_ARG, "%s: lanes->seqlen_k is required", who);
  mslk_attn_args a = make_args(q, k, v, *sq, *sk, *sv, *so, 1, M, Mkv, H, K, Kv, scale, mask_kind,
                               seqlens, band, out, lse);
  a.lanes = lanes;
  return attn_general(a, static_cast<cudaStream_t>(stream), who);
}

mslk_status mslk_attn_fwd_fp8(const void* q, const void* k, const void* v, const mslk_strides* sq,
                              const mslk_strides* sk, const mslk_strides* sv, const mslk_strides* so,
                              int32_t B, int32_t M, int32_t Mkv, int32_t H, int32_t K, int32_t Kv,
                              float scale, int32_t mask_kind, const mslk_seqlens* seqlens,
                              const mslk_band* band, const mslk_kv_lanes* lanes,
                              const mslk_fp8_scales* scales, void* out, float* lse, void* stream) {
  const char* who = "mslk_attn_fwd_fp8";
  if (scales == nullptr)
    return fail(MSLK_ERR_INVALID_ARG, "%s: descale_q, descale_k and descale_v are required", who);
  if (sq == nullptr || sk == nullptr || sv == nullptr || so == nullptr)
    return fail(MSLK_ERR_INVALID_ARG, "%s: null strides", who);
  mslk_attn_args a = make_args(q, k, v, *sq, *sk, *sv, *so, B, M, Mkv, H, K, Kv, scale, mask_kind,
                               seqlens, band, out, lse);
  a.lanes = lanes;
  a.fp8 = scales;
  return attn_general(a, static_cast<cudaStream_t>(stream), who);
}

mslk_status mslk_merge_attentions(const float* out_split, const float* lse_split, int32_t n_chunks,
                                  int64_t chunk_stride_out, int64_t chunk_stride_lse, int32_t B,
                                  int32_t M, int32_t H, int32_t Kv, const mslk_strides* s_split,
                                  const mslk_strides* so, void* out, int32_t out_dtype, float* lse,
                                  void* stream) {
  const char* who = "mslk_merge_attentions";
  MergeProblem p{};
  mslk_status s = validate_merge(p, n_chunks, B, M, H, Kv, s_split, so, out, out_dtype, lse, who);
  if (s != MSLK_OK || B == 0 || M == 0 || H == 0) return s;
  if (out_split == nullptr || lse_split == nullptr)
    return fail(MSLK_ERR_INVALID_ARG, "%s: null pointer", who);
  if (!aligned16(out_split))
    return fail(MSLK_ERR_MISALIGNED, "%s: out_split/out must be 16-byte aligned", who);
  if ((reinterpret_cast<uintptr_t>(lse_split) & 3u) != 0)
    return fail(MSLK_ERR_MISALIGNED, "%s: lse_split/lse must be 4-byte aligned", who);
  if (n_chunks > 1 && (chunk_stride_out <= 0 || chunk_stride_out % 4))
    return fail(MSLK_ERR_MISALIGNED, "%s: chunk_stride_out must be a positive multiple of 4", who);
  if (n_chunks > 1 && chunk_stride_lse <= 0)
    return fail(MSLK_ERR_INVALID_ARG, "%s: chunk_stride_lse must be positive", who);
  p.out_split = out_split;
  p.lse_split = lse_split;
  p.cs_out = chunk_stride_out;
  p.cs_lse = chunk_stride_lse;
  return run_merge(p, static_cast<cudaStream_t>(stream), who);
}

mslk_status mslk_merge_attentions_varargs(const float* const* out_chunks,
                                          const float* const* lse_chunks, int32_t n_chunks,
                                          int32_t B, int32_t M, int32_t H, int32_t Kv,
                                          const mslk_strides* s_split, const mslk_strides* so,
                                          void* out, int32_t out_dtype, float* lse, void* stream) {
  const char* who = "mslk_merge_attentions_varargs";
  if (n_chunks > kMergeMaxVarargs)
    return fail(MSLK_ERR_UNSUPPORTED, "%s: at most %d chunks (got %d)", who, kMergeMaxVarargs, n_chunks);
  MergeProblem p{};
  mslk_status s = validate_merge(p, n_chunks, B, M, H, Kv, s_split, so, out, out_dtype, lse, who);
  if (s != MSLK_OK || B == 0 || M == 0 || H == 0) return s;
  if (out_chunks == nullptr || lse_chunks == nullptr)
    return fail(MSLK_ERR_INVALID_ARG, "%s: null chunk array", who);
  for (int c = 0; c < n_chunks; ++c) {
    if (out_chunks[c] == nullptr || lse_chunks[c] == nullptr)
      return fail(MSLK_ERR_INVALID_ARG, "%s: chunk %d is null", who, c);
    if (!aligned16(out_chunks[c]))
      return fail(MSLK_ERR_MISALIGNED, "%s: chunk %d output must be 16-byte aligned", who, c);
    if ((reinterpret_cast<uintptr_t>(lse_chunks[c]) & 3u) != 0)
      return fail(MSLK_ERR_MISALIGNED, "%s: chunk %d lse must be 4-byte aligned", who, c);
  }
  p.chunk_out = out_chunks;
  p.chunk_lse = lse_chunks;
  return run_merge(p, static_cast<cudaStream_t>(stream), who);
}

int32_t mslk_splitk_size(int32_t batch, int32_t seqlen_kv, int32_t kv_heads, int32_t tile_n,
                         int32_t sm_count) {
  return splitk_size(batch, seqlen_kv, kv_heads, tile_n, sm_count);
}

mslk_status mslk_attn_split_kv_static(const mslk_attn_args* args, int32_t n_chunks, void* stream) {
  const char* who = "mslk_attn_split_kv_static";
  mslk_status s = check_split_args(args, n_chunks, who);
  if (s != MSLK_OK) return s;
  const mslk_attn_args& a = *args;
  if (a.B == 0 || a.M == 0 || a.H == 0 || a.Mkv == 0)  // nothing to split: the forward call
    return attn_general(a, static_cast<cudaStream_t>(stream), who);
  const int32_t n = split_chunks(a, n_chunks);
  const SplitLayout l = split_layout(a, n);
  if (l.bytes > static_cast<size_t>(MSLK_SPLIT_KV_STATIC_BYTES))
    return fail(MSLK_ERR_UNSUPPORTED,
                "%s: %d chunks of this problem need a %zu-byte workspace, above the library's "
                "fixed %zu bytes (fewer chunks, or mslk_attn_split_kv with a workspace)",
                who, n, l.bytes, static_cast<size_t>(MSLK_SPLIT_KV_STATIC_BYTES));
  cudaError_t e = cudaSuccess;
  float* ws = split_static_workspace(&e);
  if (ws == nullptr)
    return fail(MSLK_ERR_CUDA, "%s: no device address for the fixed workspace (%s)", who,
                cudaGetErrorString(e));
  return run_split_kv(a, n, ws, ws + l.lse_offset / sizeof(float), static_cast<cudaStream_t>(stream), who);
}

mslk_status mslk_attn_split_kv_workspace(const mslk_attn_args* args, int32_t n_chunks,
                                         size_t* bytes) {
  const char* who = "mslk_attn_split_kv_workspace";
  if (bytes == nullptr) return fail(MSLK_ERR_INVALID_ARG, "%s: bytes is null", who);
  if (args == nullptr) return fail(MSLK_ERR_INVALID_ARG, "%s: args is null", who);
  // Sizes only: the tensor pointers are not read (a stand-in passes the pointer checks,
  // nothing is launched).
  mslk_attn_args a = *args;
  const void* stand_in = reinterpret_cast<const void*>(static_cast<uintptr_t>(256));
  if (a.q == nullptr) a.q = stand_in;
  if (a.k == nullptr) a.k = stand_in;
  if (a.v == nullptr) a.v = stand_in;
  if (a.out == nullptr) a.out = const_cast<void*>(stand_in);
  const mslk_status s = check_split_args(&a, n_chunks, who);
  if (s != MSLK_OK) return s;
  *bytes = split_layout(a, split_chunks(a, n_chunks)).bytes;
  return ok();
}

mslk_status mslk_attn_split_kv(const mslk_attn_args* args, int32_t n_chunks, void* workspace,
                               size_t workspace_bytes, void* stream) {
  const char* who = "mslk_attn_split_kv";
  mslk_status s = check_split_args(args, n_chunks, who);
  if (s != MSLK_OK) return s;
  const mslk_attn_args& a = *args;
  if (a.B == 0 || a.M == 0 || a.H == 0 || a.Mkv == 0)  // nothing to split: the forward call
    return attn_general(a, static_cast<cudaStream_t>(stream), who);
  const int32_t n = split_chunks(a, n_chunks);
  const SplitLayout l = split_layout(a, n);
  if (workspace == nullptr) return fail(MSLK_ERR_INVALID_ARG, "%s: workspace is null", who);
  if (reinterpret_cast<uintptr_t>(workspace) & 255u)
    return fail(MSLK_ERR_MISALIGNED, "%s: workspace must be 256-byte aligned", who);
  if (workspace_bytes < l.bytes)
    return fail(MSLK_ERR_INVALID_ARG, "%s: workspace of %zu bytes is below the %zu needed", who,
                workspace_bytes, l.bytes);
  float* ws = static_cast<float*>(workspace);
  return run_split_kv(a, n, ws, ws + l.lse_offset / sizeof(float), static_cast<cudaStream_t>(stream), who);
}

const char* mslk_last_error(void) { return g_last_error; }

mslk_status mslk_device_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(MSLK_ERR_CUDA, "mslk_device_status: %s", cudaGetErrorString(e));
  unsigned int word = 0;
  e = cudaMemcpyFromSymbol(&word, g_error_word, sizeof(word));
  if (e != cudaSuccess) return fail(MSLK_ERR_CUDA, "mslk_device_status: %s", cudaGetErrorString(e));
  if (word != 0) {
    const unsigned int zero = 0;
    cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero));
    if (word & kErrWaitTimeout)
      return fail(MSLK_ERR_DEVICE_TIMEOUT, "a kernel gave up on a bounded wait");
  }
  return ok();
}

void mslk_set_wait_timeout_ns(int64_t ns) { g_timeout_ns.store(ns < 100000 ? 100000 : ns); }

mslk_status mslk_diag_bounded_wait(void* stream) {
  const DeviceCtl ctl = device_ctl();
  if (ctl.err == nullptr) return fail(MSLK_ERR_CUDA, "mslk_diag_bounded_wait: no CUDA device");
  bounded_wait_diag_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(ctl.err, ctl.timeout_ns);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(MSLK_ERR_CUDA, "mslk_diag_bounded_wait: %s", cudaGetErrorString(e));
  return ok();
}

void mslk_set_path_policy(int32_t policy) { g_path_policy.store(policy); }

int32_t mslk_version(void) { return 100; }

}  // extern "C"
