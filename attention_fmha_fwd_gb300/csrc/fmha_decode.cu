// fmha_decode.cu — attention forward / partial for a handful of query rows (at most 8 per
// batch or packed sequence), on the CUDA cores.
//
// With one query row per head each K/V element is used once, so the work is a stream
// of K and V from HBM (about 1 FLOP per byte); tensor-core tiles would be 128-fold
// padding.  The keys of one (batch, head) are split over a thread-block cluster of CS
// CTAs (CS = 1..16, above 8 only where the device schedules it, chosen from how many such
// clusters stay resident, to minimise waves x keys per CTA); inside a CTA one
// producer warp streams tiles of T keys (8 KiB of K plus 8 KiB of V: T = 4096 / D bf16 or
// 8192 / D E4M3 keys) through a ring of shared-memory stages with TMA, so up to 192 KiB per SM are in
// flight whatever the register budget.  Eight consumer warps take the tiles round robin.  Lane l holds
// head-dim elements [l*V, l*V+V) of every row (V = D/32) and reads them from shared
// memory (one 256/128-byte row per warp instruction); a halving butterfly leaves key l's
// full score on lane l, followed by the base-2 online softmax and one pass over the V
// rows for all query rows.  Warp states (max, sum, accumulator) merge through shared
// memory and the CTAs of a cluster merge through distributed shared memory, by the same
// LSE rule as the split-KV merge; no global scratch memory is used.
//
// Semantics follow MSLK's memory_efficient_attention / _partial ("Attention - Core
// fMHA"): out = softmax(scale q.k^T + mask) v over the allowed keys; lse = ln sum exp;
// rows without an allowed key get out = 0, lse = -inf.
//
// Modes: dense batches or packed sequences (grid row = sequence: its queries from
// cu_seqlens_q, its keys from cu_seqlens_k or a key lane, padded or paged through an
// incremental page cursor); every mask as a band on key - row with a per-sequence
// bottom-right shift; grouped K/V heads, with up to 8 / rows query heads of a K/V head
// folded into one CTA's rows (each row's query position in shared memory); E4M3 inputs
// (fmha_decode_fp8_kernel: 8 KiB tiles hold twice the keys, products by f32-accumulating
// mixed-precision FMAs on exact f16 values, probabilities rounded to f16 for P.V).
// Tiles of 64 or more keys are folded 32 + 32 keys per step.

#include <cuda_bf16.h>

#include <algorithm>
#include <atomic>
#include <cmath>

#include "internal.h"
#include "ptx.cuh"
#include "tmap.h"

namespace mslk {
namespace {

constexpr int kWarps = 8;                      // consumer warps
constexpr int kThreads = (kWarps + 1) * 32;    // + one producer warp
constexpr int kStages = 12;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// F8: K/V (and Q) are E4M3 bytes, so a tile holds twice the keys in the same 8 KiB.
template <int D, bool F8>
struct DecLayout {
  static constexpr int kEsz = F8 ? 1 : 2;          // bytes per element
  static constexpr int kT = 8192 / (D * kEsz);     // keys per tile: 32/64 (bf16), 64/128 (E4M3)
  static constexpr int kTileBytes = kT * D * kEsz; // one tensor's tile: 8 KiB
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr int kFullOff = kRingBytes;      // full[kStages] mbarriers
  static constexpr int kEmptyOff = kFullOff + 8 * kStages;
  static constexpr int kAbortOff = kEmptyOff + 8 * kStages;
  static constexpr int kIssuedOff = kAbortOff + 4;  // tiles issued so far (producer-written)
  static constexpr int kPosOff = kAbortOff + 16;    // query position of each row [8]
  static constexpr int kBytes = kPosOff + 32;
  static constexpr int kAlloc = kBytes + 1024;     // slack for 1024-byte alignment
};

struct DecArgs {
  const uint8_t* q;  // bf16 or E4M3 elements
  long long sq_b, sq_m, sq_h;
  int M, Mkv, H;
  // Query head h reads K/V head h / kv_group; each CTA takes `fold` query heads of one K/V
  // head (a divisor of kv_group) as extra rows, so that K/V head is streamed once for them.
  int kv_group, fold;
  // Head-dim elements that exist (head dim 96 runs on the 128-wide kernel: the tensor maps
  // zero-fill K/V columns 96..127, and lanes past them neither load q nor store out).
  int d_real;
  int independent;  // launched with programmatic stream serialization (see the host side)
  int cs;  // CTAs per (batch, head): the cluster size
  // Key j is allowed for query row m iff m + lo <= j <= m + hi (kv_offset folded in;
  // +-kBandOpen: open), plus each packed sequence's Lk - Lq when band_seq is set.
  long long lo, hi;
  int band_seq;
  // Sequence mode (block-diagonal kinds): grid row = packed sequence s, its queries
  // cu_q[s]..cu_q[s+1], its keys cu_k[s]..cu_k[s+1] or a key lane (lane_len[s] keys at
  // lane_start[s] + p, or paged at block_table[s * max_pages + p / page_size] *
  // page_size + p % page_size).
  int seq_mode, lanes;
  const int* cu_q;
  const int* cu_k;
  const int* lane_len;
  const int* lane_start;
  const int* block_table;
  int page_size, max_pages;
  float scale_log2;
  // E4M3 inputs: element x of head h stands for x * descale[h] (descale[0] when
  // desc_per_tensor); q and k descales fold into the score scale, v's into the output.
  const float* dq;
  const float* dk;
  const float* dv;
  int desc_per_tensor;
  void* out;
  int out_fp32;
  long long so_b, so_m, so_h;
  float* lse;
  unsigned int* err;
  unsigned long long timeout_ns;
};

// V consecutive head-dim elements of one row -> fp32 (bf16: widen; E4M3: exact convert).
template <int V, bool F8>
struct Vec;
template <>
struct Vec<4, false> {
  using T = uint2;
  MSLK_DEV static void to_float(T x, float* f) {
    f[0] = __uint_as_float(x.x << 16);
    f[1] = __uint_as_float(x.x & 0xFFFF0000u);
    f[2] = __uint_as_float(x.y << 16);
    f[3] = __uint_as_float(x.y & 0xFFFF0000u);
  }
};
template <>
struct Vec<2, false> {
  using T = uint32_t;
  MSLK_DEV static void to_float(T x, float* f) {
    f[0] = __uint_as_float(x << 16);
    f[1] = __uint_as_float(x & 0xFFFF0000u);
  }
};
template <>
struct Vec<4, true> {
  using T = uint32_t;
  MSLK_DEV static void to_float(T x, float* f) {
    const float2 a = e4m3x2_to_f2(static_cast<uint16_t>(x & 0xFFFFu));
    const float2 b = e4m3x2_to_f2(static_cast<uint16_t>(x >> 16));
    f[0] = a.x;
    f[1] = a.y;
    f[2] = b.x;
    f[3] = b.y;
  }
};
template <>
struct Vec<2, true> {
  using T = uint16_t;
  MSLK_DEV static void to_float(T x, float* f) {
    const float2 a = e4m3x2_to_f2(x);
    f[0] = a.x;
    f[1] = a.y;
  }
};

MSLK_DEV float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
MSLK_DEV float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// v[0..31] are one lane's partial sums for 32 keys.  Returns on lane l the full sum over
// all 32 lanes for key l.  Each halving step keeps the half of the values selected by one
// lane bit and adds the partner lane's other half.
MSLK_DEV float butterfly_reduce32(float (&v)[32], int lane) {
  int n = 32;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    n /= 2;
    const bool up = lane & o;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (i < n) {
        const float send = up ? v[i] : v[i + n];
        const float keep = up ? v[i + n] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
      }
    }
  }
  return v[0];
}

// Bounded mbarrier wait: false on timeout (recorded in the error word and the CTA's abort
// flag) or when another warp of the CTA has already given up.
MSLK_DEV bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag, const DecArgs& a) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > a.timeout_ns) {
      *abort_flag = 1;
      atomicOr(a.err, kErrWaitTimeout);
      return false;
    }
  }
}

// Bounded wait until the producer has issued more than `i` tiles.  Tile i is issued only
// after tile i - kStages (same stage, possibly another warp's) has been consumed, so the
// stage's previous full-barrier phase has completed and a parity wait on it cannot be
// satisfied by that older phase.
MSLK_DEV bool wait_issued(const volatile int* issued, int i, volatile int* abort_flag, const DecArgs& a) {
  if (*issued > i) {
    __threadfence_block();
    return true;
  }
  const uint64_t t0 = globaltimer_ns();
  while (*issued <= i) {
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > a.timeout_ns) {
      *abort_flag = 1;
      atomicOr(a.err, kErrWaitTimeout);
      return false;
    }
  }
  __threadfence_block();
  return true;
}

template <int D, int MQ>
struct DecodeState {
  float m_run[MQ], l_run[MQ], acc[MQ][D / 32];
};

// Folds one tile of keys (in shared memory, row-major [T][D]) into the warp's
// online-softmax state, 32 keys at a time.  bf16: qf holds the query rows pre-multiplied by
// the base-2 score scale.  E4M3: qh holds them as exact f16 pairs, the products are formed
// with mixed-precision FMAs (exact, added in fp32), the score is scaled by qscale after the
// reduction, and p is rounded to f16 (relative 2^-11) for P.V.
// Row m (m < nrows) holds the query at position pos[m] (folded query heads share positions).
template <int D, int MQ, bool F8>
MSLK_DEV void fold_tile(int nrows, const int* pos, long long lo, long long hi,
                        const float (&qf)[MQ][D / 32], const uint32_t (&qh)[MQ][D / 64],
                        const float (&qscale)[MQ], const uint8_t* sK, const uint8_t* sV, int key0,
                        int kb1, int lane, DecodeState<D, MQ>& st) {
  constexpr int VE = D / 32;
  constexpr int T = DecLayout<D, F8>::kT;
  constexpr int ES = DecLayout<D, F8>::kEsz;
  // Blocks of 32 keys folded per step: two when the tile holds 64 or more keys, so the
  // two score reductions interleave and one max / sum / rescale covers both.
  constexpr int NB = T >= 64 ? 2 : 1;
  // With few query rows each lane has only MQ * VE accumulator chains; the blocks of a
  // step then accumulate separately (twice the independent FMA chains) and are summed once.
  constexpr int NA = (NB == 2 && MQ <= 2) ? 2 : 1;
  using VT = typename Vec<VE, F8>::T;
#pragma unroll 1
  for (int sb = 0; sb < T; sb += 32 * NB) {
    const int n_valid = kb1 - (key0 + sb);  // keys of this step below kb1 (warp-uniform)
    if (n_valid <= 0) break;                // the rest of the tile is past the range
    const VT* kp = reinterpret_cast<const VT*>(sK + (sb * D + lane * VE) * ES);
    const VT* vp = reinterpret_cast<const VT*>(sV + (sb * D + lane * VE) * ES);
    float p[NB][MQ];
#pragma unroll
    for (int m = 0; m < MQ; ++m) {
#pragma unroll
      for (int b = 0; b < NB; ++b) p[b][m] = 0.f;
      if (m >= nrows) continue;
      float part[NB][32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          const VT kx = kp[(b * 32 + j) * (D / VE)];
          float d = 0.f;
          if constexpr (F8) {
            if constexpr (VE == 4) {
              d = dot2_f16_f32(d, qh[m][0], e4m3x2_to_f16x2(static_cast<uint16_t>(kx & 0xFFFFu)));
              d = dot2_f16_f32(d, qh[m][1], e4m3x2_to_f16x2(static_cast<uint16_t>(kx >> 16)));
            } else {
              d = dot2_f16_f32(d, qh[m][0], e4m3x2_to_f16x2(kx));
            }
          } else {
            float kf[VE];
            Vec<VE, F8>::to_float(kx, kf);
#pragma unroll
            for (int e = 0; e < VE; ++e) d = fmaf(qf[m][e], kf[e], d);
          }
          part[b][j] = d;
        }
      }
      float sc[NB];
      float mx = -INFINITY;
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        sc[b] = butterfly_reduce32(part[b], lane);
        if constexpr (F8) sc[b] *= qscale[m];
        const int my_key = key0 + sb + b * 32 + lane;
        const bool allowed = my_key < kb1 && my_key <= pos[m] + hi && my_key >= pos[m] + lo;
        sc[b] = allowed ? sc[b] : -INFINITY;
        mx = fmaxf(mx, sc[b]);
      }
      const float m_new = fmaxf(st.m_run[m], warp_max(mx));
      const float msub = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = ex2_approx(st.m_run[m] - msub);  // m_run = -inf -> 0
      float psum = 0.f;
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        p[b][m] = ex2_approx(sc[b] - msub);
        psum += p[b][m];
      }
      st.l_run[m] = st.l_run[m] * alpha + warp_sum(psum);
      st.m_run[m] = m_new;
#pragma unroll
      for (int e = 0; e < VE; ++e) st.acc[m][e] *= alpha;
    }
    // V rows at or past kb1 get p = 0, but they may hold anything (a key lane's
    // unwritten tail) and 0 * NaN is NaN: this warp owns the tile, so it clears them.
    if (n_valid < 32 * NB) {
      uint8_t* tail = const_cast<uint8_t*>(sV) + (sb + n_valid) * D * ES;
      for (int off = lane * 16; off < (32 * NB - n_valid) * D * ES; off += 32 * 16)
        *reinterpret_cast<uint4*>(tail + off) = make_uint4(0, 0, 0, 0);
      __syncwarp();
    }
    // One pass over the V rows for every query row.
    float acc2[NA][MQ][VE];
#pragma unroll
    for (int m = 0; m < MQ; ++m)
#pragma unroll
      for (int e = 0; e < VE; ++e) {
        acc2[0][m][e] = st.acc[m][e];
        if constexpr (NA == 2) acc2[NA - 1][m][e] = 0.f;
      }
    if constexpr (F8) {
      uint32_t ph[NB][MQ];
#pragma unroll
      for (int b = 0; b < NB; ++b)
#pragma unroll
        for (int m = 0; m < MQ; ++m) ph[b][m] = f32_to_f16_bits(p[b][m]);
#pragma unroll 2
      for (int j = 0; j < 32; ++j) {
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          const VT vx = vp[(b * 32 + j) * (D / VE)];
          uint32_t vh[VE / 2];
          if constexpr (VE == 4) {
            vh[0] = e4m3x2_to_f16x2(static_cast<uint16_t>(vx & 0xFFFFu));
            vh[1] = e4m3x2_to_f16x2(static_cast<uint16_t>(vx >> 16));
          } else {
            vh[0] = e4m3x2_to_f16x2(vx);
          }
#pragma unroll
          for (int m = 0; m < MQ; ++m) {
            if (m >= nrows) continue;
            const uint32_t pj = __shfl_sync(0xffffffffu, ph[b][m], j);
            float(&ac)[VE] = acc2[b % NA][m];
#pragma unroll
            for (int e = 0; e < VE / 2; ++e) axpy2_f16_f32(ac[2 * e], ac[2 * e + 1], pj, vh[e]);
          }
        }
      }
    } else {
#pragma unroll 4
      for (int j = 0; j < 32; ++j) {
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          float vf[VE];
          Vec<VE, F8>::to_float(vp[(b * 32 + j) * (D / VE)], vf);
#pragma unroll
          for (int m = 0; m < MQ; ++m) {
            if (m >= nrows) continue;
            const float pj = __shfl_sync(0xffffffffu, p[b][m], j);
            float(&ac)[VE] = acc2[b % NA][m];
#pragma unroll
            for (int e = 0; e < VE; ++e) ac[e] = fmaf(pj, vf[e], ac[e]);
          }
        }
      }
    }
#pragma unroll
    for (int m = 0; m < MQ; ++m)
#pragma unroll
      for (int e = 0; e < VE; ++e) st.acc[m][e] = NA == 2 ? acc2[0][m][e] + acc2[NA - 1][m][e] : acc2[0][m][e];
  }
}

template <int D, int MQ, bool F8>
MSLK_DEV void decode_body(const CUtensorMap& tm_k, const CUtensorMap& tm_v, const DecArgs& a) {
  using L = DecLayout<D, F8>;
  constexpr int VE = D / 32;  // head-dim elements per lane
  constexpr int T = L::kT;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned, derived from the shared array itself so accesses stay shared-space
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbortOff);
  volatile int* issued_ctr = reinterpret_cast<volatile int*>(smem + L::kIssuedOff);

  // A following launch that declared itself independent of this one may start now; a
  // launch without that declaration still waits for this grid to complete.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int rank = static_cast<int>(blockIdx.x) % a.cs;  // CTA rank inside the cluster
  const int hq0 = static_cast<int>(blockIdx.x) / a.cs * a.fold;  // first query head of the CTA
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int hk = hq0 / a.kv_group;
  // This CTA's query rows [qrow0, qrow0 + nq) and keys [0, nk) (row krow0 + key, or paged)
  // of batch coordinate bc: a batch (dense) or a packed sequence s (sequence mode).
  const int s_idx = blockIdx.y;
  int bc = s_idx, qrow0 = 0, nq = a.M, nk = a.Mkv, krow0 = 0;
  long long lo = a.lo, hi = a.hi;
  if (a.seq_mode) {
    bc = 0;
    qrow0 = min(max(a.cu_q[s_idx], 0), a.M);
    nq = min(min(max(a.cu_q[s_idx + 1], qrow0), a.M) - qrow0, MQ / a.fold);
    if (a.lanes) {
      nk = max(a.lane_len[s_idx], 0);
      if (a.block_table != nullptr)
        nk = static_cast<int>(min(static_cast<long long>(nk), static_cast<long long>(a.max_pages) * a.page_size));
      else
        krow0 = a.lane_start[s_idx];
    } else {
      krow0 = min(max(a.cu_k[s_idx], 0), a.Mkv);
      nk = min(max(a.cu_k[s_idx + 1], krow0), a.Mkv) - krow0;
    }
    if (a.band_seq) {
      const long long shift = static_cast<long long>(nk) - nq;
      if (lo > -kBandOpen) lo += shift;
      if (hi < kBandOpen) hi += shift;
    }
  }

  // Rows: query head hq0 + r / nq at position r % nq, for r < nrows = nq * fold (the
  // positions live in shared memory: warp-uniform, read by broadcast).
  const int nrows = nq * a.fold;
  int* pos = reinterpret_cast<int*>(smem + L::kPosOff);

  // Keys of this (batch or sequence, head) that some row may see: from row 0's lower band
  // edge to the last row's upper edge, split over the cluster's CTAs in whole tiles.
  const long long k_first = max(0LL, lo);
  const long long k_last = min(static_cast<long long>(nk) - 1, static_cast<long long>(nq - 1) + hi);
  const bool any = k_first <= k_last && nq > 0;
  const int tile_first = any ? static_cast<int>(k_first / T) : 0;
  const int tiles_all = any ? static_cast<int>(k_last / T) + 1 - tile_first : 0;
  const int per_cta = (tiles_all + a.cs - 1) / a.cs;
  const int t0 = min(tiles_all, rank * per_cta);
  const int n_tiles = max(0, min(tiles_all, t0 + per_cta) - t0);
  const int key_base = (tile_first + t0) * T;
  const int kb1 = static_cast<int>(min(k_last + 1, static_cast<long long>(tile_first + t0 + n_tiles) * T));

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(sbase + L::kFullOff + 8 * s, 1);
      mbar_init(sbase + L::kEmptyOff + 8 * s, 1);
    }
    *abort_flag = 0;
    *issued_ctr = 0;
    for (int r = 0; r < MQ; ++r) pos[r] = nq > 0 ? r % nq : 0;
    fence_mbar_init();
  }
  __syncthreads();

  DecodeState<D, MQ> st;
#pragma unroll
  for (int m = 0; m < MQ; ++m) {
    st.m_run[m] = -INFINITY;
    st.l_run[m] = 0.f;
#pragma unroll
    for (int e = 0; e < VE; ++e) st.acc[m][e] = 0.f;
  }

  if (warp == kWarps) {
    // Producer: tile i -> stage i % kStages, after the consumer of tile i - kStages has
    // released the stage; the issued count it publishes tells consumers when a stage's
    // barrier is on the phase of their tile.  Afterwards it waits (bounded) for every copy it issued, so no
    // copy is still writing shared memory when the stages are reused below.
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      int issued = 0;
      // Paged lane (T divides page_size): the page table entry of the next page is read
      // one page ahead, so its latency is off the issue path.
      const bool paged = a.seq_mode && a.block_table != nullptr;
      const int* table = paged ? a.block_table + static_cast<long long>(s_idx) * a.max_pages : nullptr;
      const int n_pages_lane = paged ? (nk + a.page_size - 1) / a.page_size : 0;
      int page = paged ? key_base / a.page_size : 0;
      int in_page = paged ? key_base - page * a.page_size : 0;  // key offset inside the page
      int phys = (paged && page < n_pages_lane) ? table[page] : 0;
      int phys_next = (paged && page + 1 < n_pages_lane) ? table[page + 1] : 0;
      for (int i = 0; i < n_tiles; ++i) {
        const int s = i % kStages;
        if (i >= kStages &&
            !wait_bounded(sbase + L::kEmptyOff + 8 * s, ((i / kStages) - 1) & 1, abort_flag, a))
          break;
        const uint32_t full = sbase + L::kFullOff + 8 * s;
        const uint32_t dst = sbase + s * L::kStageBytes;
        const int row = paged ? phys * a.page_size + in_page : krow0 + key_base + i * T;
        if (paged && (in_page += T) == a.page_size) {  // the next tile starts the next page
          in_page = 0;
          ++page;
          phys = phys_next;
          phys_next = page + 1 < n_pages_lane ? table[page + 1] : 0;
        }
        mbar_arrive_expect_tx(full, L::kStageBytes);
        tma_load_4d(dst, &tm_k, full, 0, row, hk, bc);
        tma_load_4d(dst + L::kTileBytes, &tm_v, full, 0, row, hk, bc);
        ++issued;
        __threadfence_block();
        *issued_ctr = issued;
      }
      const uint64_t t_start = globaltimer_ns();
      for (int i = max(0, issued - kStages); i < issued; ++i) {
        const uint32_t full = sbase + L::kFullOff + 8 * (i % kStages);
        while (!mbar_try_wait(full, (i / kStages) & 1)) {
          if (globaltimer_ns() - t_start > a.timeout_ns) {
            *abort_flag = 1;
            atomicOr(a.err, kErrWaitTimeout);
            break;
          }
        }
      }
    }
    __syncwarp();
  } else {
    // Query rows, pre-multiplied by scale * log2(e): scores come out in base 2.
    using VT = typename Vec<VE, F8>::T;
    float qscale[MQ];
    float qf[MQ][VE];
    uint32_t qh[MQ][VE / 2];  // E4M3 rows as exact f16 pairs
#pragma unroll
    for (int m = 0; m < MQ; ++m) {
#pragma unroll
      for (int e = 0; e < VE / 2; ++e) qh[m][e] = 0u;
      qscale[m] = a.scale_log2;
      const int hq = hq0 + (nq > 0 ? m / nq : 0);  // row m: query head hq, position pos[m]
      // (warp-uniform: after the reduction lane j holds key j's score, scaled by qscale)
      if constexpr (F8)
        if (m < nrows) qscale[m] *= a.dq[a.desc_per_tensor ? 0 : hq] * a.dk[a.desc_per_tensor ? 0 : hk];
      if (m < nrows && lane * VE < a.d_real) {
        const long long el = bc * a.sq_b + (qrow0 + m % nq) * a.sq_m + hq * a.sq_h + lane * VE;
        const VT x = *reinterpret_cast<const VT*>(a.q + el * L::kEsz);
        if constexpr (F8) {
          if constexpr (VE == 4) {
            qh[m][0] = e4m3x2_to_f16x2(static_cast<uint16_t>(x & 0xFFFFu));
            qh[m][1] = e4m3x2_to_f16x2(static_cast<uint16_t>(x >> 16));
          } else {
            qh[m][0] = e4m3x2_to_f16x2(x);
          }
        }
        Vec<VE, F8>::to_float(x, qf[m]);
#pragma unroll
        for (int e = 0; e < VE; ++e) qf[m][e] *= qscale[m];
      } else {
#pragma unroll
        for (int e = 0; e < VE; ++e) qf[m][e] = 0.f;
      }
    }
    for (int i = warp; i < n_tiles; i += kWarps) {
      const int s = i % kStages;
      const bool ok = __all_sync(0xffffffffu,
                                 wait_issued(issued_ctr, i, abort_flag, a) &&
                                     wait_bounded(sbase + L::kFullOff + 8 * s, (i / kStages) & 1, abort_flag, a));
      if (!ok) break;
      const uint8_t* sK = smem + s * L::kStageBytes;
      fold_tile<D, MQ, F8>(nrows, pos, lo, hi, qf, qh, qscale, sK, sK + L::kTileBytes, key_base + i * T, kb1, lane, st);
      __syncwarp();
      if (lane == 0) mbar_arrive(sbase + L::kEmptyOff + 8 * s);
    }
  }
  __syncthreads();  // every copy has landed and every tile has been read: the ring is free

  // Merge the warps' states: M* = max_w m_w; L = sum_w 2^(m_w - M*) l_w;
  // acc = sum_w 2^(m_w - M*) acc_w.  The CTA's merged state goes to c_* for the cluster.
  // These arrays reuse the ring's shared memory.
  float(*s_m)[MQ] = reinterpret_cast<float(*)[MQ]>(smem);
  float(*s_l)[MQ] = reinterpret_cast<float(*)[MQ]>(smem + kWarps * MQ * 4);
  float(*s_acc)[MQ][D] = reinterpret_cast<float(*)[MQ][D]>(smem + 2 * kWarps * MQ * 4);
  float* c_m = reinterpret_cast<float*>(smem + 2 * kWarps * MQ * 4 + kWarps * MQ * D * 4);
  float* c_l = c_m + MQ;
  float(*c_acc)[D] = reinterpret_cast<float(*)[D]>(c_l + MQ);
  if (warp < kWarps) {
#pragma unroll
    for (int m = 0; m < MQ; ++m) {
      if (lane == 0) {
        s_m[warp][m] = st.m_run[m];
        s_l[warp][m] = st.l_run[m];
      }
#pragma unroll
      for (int e = 0; e < VE; ++e) s_acc[warp][m][lane * VE + e] = st.acc[m][e];
    }
  }
  __syncthreads();
  // Warp w merges row w (MQ <= 8: at most one row per warp).
  for (int m = warp; m < nrows; m += kWarps + 1) {
    float mstar = -INFINITY;
    for (int w = 0; w < kWarps; ++w) mstar = fmaxf(mstar, s_m[w][m]);
    const float msub = (mstar == -INFINITY) ? 0.f : mstar;
    float Ls = 0.f;
    float o[VE];
#pragma unroll
    for (int e = 0; e < VE; ++e) o[e] = 0.f;
    for (int w = 0; w < kWarps; ++w) {
      const float c = ex2_approx(s_m[w][m] - msub);
      Ls = fmaf(c, s_l[w][m], Ls);
#pragma unroll
      for (int e = 0; e < VE; ++e) o[e] = fmaf(c, s_acc[w][m][lane * VE + e], o[e]);
    }
    if (lane == 0) {
      c_m[m] = mstar;
      c_l[m] = Ls;
    }
#pragma unroll
    for (int e = 0; e < VE; ++e) c_acc[m][lane * VE + e] = o[e];
  }

  // Cluster merge: rank 0 reads every rank's (c_m, c_l, c_acc) through distributed shared
  // memory and writes the row; the second barrier keeps the other CTAs (and their shared
  // memory) alive until rank 0 has read them.
  if (a.cs > 1) cluster_sync(); else __syncthreads();
  if (rank == 0) {
    for (int m = warp; m < nrows; m += kWarps + 1) {
      const int hq = hq0 + m / nq, qrow = qrow0 + m % nq;
      float mstar = -INFINITY;
      for (int r = 0; r < a.cs; ++r)
        mstar = fmaxf(mstar, a.cs > 1 ? ld_shared_cluster_f32(mapa_shared(smem_u32(&c_m[m]), r)) : c_m[m]);
      const float msub = (mstar == -INFINITY) ? 0.f : mstar;
      float Ls = 0.f;
      float o[VE];
#pragma unroll
      for (int e = 0; e < VE; ++e) o[e] = 0.f;
      for (int r = 0; r < a.cs; ++r) {
        const float mr = a.cs > 1 ? ld_shared_cluster_f32(mapa_shared(smem_u32(&c_m[m]), r)) : c_m[m];
        const float lr = a.cs > 1 ? ld_shared_cluster_f32(mapa_shared(smem_u32(&c_l[m]), r)) : c_l[m];
        const float c = ex2_approx(mr - msub);
        Ls = fmaf(c, lr, Ls);
#pragma unroll
        for (int e = 0; e < VE; ++e) {
          const float x = a.cs > 1 ? ld_shared_cluster_f32(mapa_shared(smem_u32(&c_acc[m][lane * VE + e]), r))
                                   : c_acc[m][lane * VE + e];
          o[e] = fmaf(c, x, o[e]);
        }
      }
      float inv = (Ls > 0.f) ? 1.f / Ls : 0.f;
      if constexpr (F8) inv *= a.dv[a.desc_per_tensor ? 0 : hk];
      if (lane * VE >= a.d_real) {
        // (padding lanes of a narrower head dim write nothing)
      } else if (a.out_fp32) {
        float* op = static_cast<float*>(a.out) + bc * a.so_b + qrow * a.so_m + hq * a.so_h + lane * VE;
#pragma unroll
        for (int e = 0; e < VE; ++e) op[e] = o[e] * inv;
      } else {
        __nv_bfloat16* op =
            static_cast<__nv_bfloat16*>(a.out) + bc * a.so_b + qrow * a.so_m + hq * a.so_h + lane * VE;
#pragma unroll
        for (int e = 0; e < VE; e += 2)
          *reinterpret_cast<uint32_t*>(op + e) = pack_bf16x2(o[e] * inv, o[e + 1] * inv);
      }
      if (lane == 0 && a.lse != nullptr)
        a.lse[(static_cast<long long>(bc) * a.H + hq) * a.M + qrow] =
            (Ls > 0.f) ? (mstar + lg2_approx(Ls)) * kLn2 : -INFINITY;
    }
  }
  if (a.cs > 1) cluster_sync();
}

template <int D, int MQ>
__global__ void __launch_bounds__(kThreads, 1)
    fmha_decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const DecArgs a) {
  decode_body<D, MQ, false>(tm_k, tm_v, a);
}

// E4M3 q, k, v with per-head or tensorwise descales.
template <int D, int MQ>
__global__ void __launch_bounds__(kThreads, 1)
    fmha_decode_fp8_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                           const DecArgs a) {
  decode_body<D, MQ, true>(tm_k, tm_v, a);
}

// B: grid rows (batches, or packed sequences in sequence mode); rows_q / rows_k: the
// longest query and key range of one grid row.
template <int D, int MQ, bool F8>
cudaError_t launch_dm(const CUtensorMap& tk, const CUtensorMap& tv, DecArgs a, int B, int H,
                      int rows_q, int rows_k, cudaStream_t stream) {
  using L = DecLayout<D, F8>;
  constexpr auto kernel = F8 ? fmha_decode_fp8_kernel<D, MQ> : fmha_decode_kernel<D, MQ>;
  static_assert(L::kAlloc <= 227 * 1024, "shared memory");
  static_assert(2 * kWarps * MQ * 4 + kWarps * MQ * D * 4 + 2 * MQ * 4 + MQ * D * 4 <= L::kRingBytes,
                "merge arrays must fit in the ring");
  // The shared-memory opt-in is per device; set it once on each.
  constexpr int kMaxDevices = 64;
  static std::atomic<int> opted_in[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  // Per cluster size c = 1..16: how many clusters the device keeps resident at once (0: c
  // not schedulable).  Sizes above 8 are non-portable and opted into explicitly.
  constexpr int kSizes = 16;
  static std::atomic<int> resident[kMaxDevices][kSizes];
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!opted_in[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             L::kAlloc);
    if (e != cudaSuccess) return e;
    const bool big_ok = cudaFuncSetAttribute(kernel,
                                             cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
    for (int si = 0; si < kSizes; ++si) {
      const int c = si + 1;
      int n = 0;
      if (c <= 8 || big_ok) {
        cudaLaunchConfig_t q{};
        q.gridDim = dim3(static_cast<unsigned>(c));
        q.blockDim = dim3(kThreads);
        q.dynamicSmemBytes = L::kAlloc;
        cudaLaunchAttribute qa[1];
        qa[0].id = cudaLaunchAttributeClusterDimension;
        qa[0].val.clusterDim.x = static_cast<unsigned>(c);
        qa[0].val.clusterDim.y = 1;
        qa[0].val.clusterDim.z = 1;
        q.attrs = qa;
        q.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, kernel, &q) != cudaSuccess) n = 0;
      }
      resident[dev][si].store(n, std::memory_order_relaxed);
    }
    (void)cudaGetLastError();  // a refused query only removes that size
    opted_in[dev].store(1, std::memory_order_release);
  }
  // Cluster size: fewest waves x keys per CTA, i.e. the smallest ceil(units / resident) / c,
  // with every CTA keeping at least two tiles per consumer warp (ties: the smaller c).
  {
    const long long units = static_cast<long long>(B) * H;
    // key tiles some row may see (the band's reach, as in the kernel; a per-sequence
    // shift is unknown here, so such bands count every key)
    const long long lo = a.band_seq ? -kBandOpen : a.lo, hi = a.band_seq ? kBandOpen : a.hi;
    const long long k_first = std::max(0LL, lo);
    const long long k_last = std::min(static_cast<long long>(rows_k) - 1, static_cast<long long>(rows_q - 1) + hi);
    const long long tiles = k_first <= k_last ? k_last / L::kT + 1 - k_first / L::kT : 0;
    int best = 1;
    double best_cost = 1e300;
    for (int si = 0; si < kSizes; ++si) {
      const int c = si + 1;
      const int n = resident[dev][si].load(std::memory_order_relaxed);
      if (n <= 0 || (c > 1 && tiles / c < 2 * kWarps)) continue;
      const double cost = static_cast<double>((units + n - 1) / n) / c;
      if (cost < best_cost * 0.999) {
        best_cost = cost;
        best = c;
      }
    }
    a.cs = best;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(H * a.cs), static_cast<unsigned>(B));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = L::kAlloc;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(a.cs);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (a.independent) {
    // the caller's inputs are not written by the previous launch: start while it finishes
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 2;
  }
  return cudaLaunchKernelEx(&cfg, kernel, tk, tv, a);
}

// H: CTAs per grid row (query heads / fold); rows: query rows per CTA (positions x fold).
template <int D, bool F8>
cudaError_t launch_d(const CUtensorMap& tk, const CUtensorMap& tv, const DecArgs& a, int B, int H,
                     int rows_q, int rows, int rows_k, cudaStream_t stream) {
  if (rows <= 1) return launch_dm<D, 1, F8>(tk, tv, a, B, H, rows_q, rows_k, stream);
  if (rows <= 2) return launch_dm<D, 2, F8>(tk, tv, a, B, H, rows_q, rows_k, stream);
  if (rows <= 4) return launch_dm<D, 4, F8>(tk, tv, a, B, H, rows_q, rows_k, stream);
  return launch_dm<D, 8, F8>(tk, tv, a, B, H, rows_q, rows_k, stream);
}


}  // namespace

cudaError_t launch_fmha_decode(const AttnProblem& p, const DeviceCtl& ctl, cudaStream_t stream,
                               const char** why) {
  EncodeTiledFn enc = tensor_map_encoder();
  if (enc == nullptr) {
    *why = "cuTensorMapEncodeTiled is not available from the driver";
    return cudaErrorNotSupported;
  }
  const int D = p.K > 64 ? 128 : 64;  // the kernel's width (96 runs zero-padded to 128)
  const int esz = p.fp8 ? 1 : 2;
  const int T = 8192 / (D * esz);
  const long long hk = p.Hkv;
  CUtensorMap tk, tv;
  if (!encode_rows_plain(enc, &tk, p.k, p.K, p.Mkv, hk, p.B, p.sk.m, p.sk.h, p.sk.b, D, T, p.fp8) ||
      !encode_rows_plain(enc, &tv, p.v, p.K, p.Mkv, hk, p.B, p.sv.m, p.sv.h, p.sv.b, D, T, p.fp8)) {
    *why = "cuTensorMapEncodeTiled rejected a k/v layout";
    return cudaErrorInvalidValue;
  }
  DecArgs a{};
  a.q = static_cast<const uint8_t*>(p.q);
  a.dq = p.descale_q;
  a.dk = p.descale_k;
  a.dv = p.descale_v;
  a.desc_per_tensor = p.descale_per_tensor ? 1 : 0;
  a.sq_b = p.sq.b;
  a.sq_m = p.sq.m;
  a.sq_h = p.sq.h;
  a.M = p.M;
  a.Mkv = p.Mkv;
  a.H = p.H;
  a.kv_group = p.kv_group;
  a.d_real = p.K;
  a.independent = p.independent ? 1 : 0;
  a.lo = p.band_lo <= -kBandOpen ? -kBandOpen : p.band_lo - p.kv_offset;
  a.hi = p.band_hi >= kBandOpen ? kBandOpen : p.band_hi - p.kv_offset;
  a.scale_log2 = p.scale * kLog2e;
  a.out = p.out;
  a.out_fp32 = p.out_fp32 ? 1 : 0;
  a.so_b = p.so.b;
  a.so_m = p.so.m;
  a.so_h = p.so.h;
  a.lse = p.lse;
  a.err = ctl.err;
  a.timeout_ns = ctl.timeout_ns;
  a.cs = 1;  // chosen per kernel instantiation from the device's cluster residency
  int grid_rows = p.B, rows_q = p.M, rows_k = p.Mkv;
  if (is_blockdiag(p.mask_kind)) {
    a.seq_mode = 1;
    a.cu_q = p.cu_q;
    a.cu_k = p.cu_k;
    a.band_seq = p.band_seq_shift ? 1 : 0;
    a.lanes = p.lanes ? 1 : 0;
    a.lane_len = p.lane_len;
    a.lane_start = p.lane_start;
    a.block_table = p.block_table;
    a.page_size = p.page_size;
    a.max_pages = p.max_pages;
    grid_rows = p.n_seqs;
    rows_q = p.max_seqlen_q;
    rows_k = p.max_seqlen_k;
  }
  if (grid_rows == 0 || rows_q == 0) return cudaSuccess;
  // Fold the most query heads of a K/V head into one CTA's rows that stay within the
  // kernel's row limit (a divisor of the group, so a CTA never spans two K/V heads).
  a.fold = 1;
  for (int d = p.kv_group; d >= 1; --d)
    if (p.kv_group % d == 0 && static_cast<long long>(rows_q) * d <= kDecodeMaxRows) {
      a.fold = d;
      break;
    }
  const int heads = p.H / a.fold, rows = rows_q * a.fold;
  *why = "decode kernel launch failed";
  if (p.fp8) {
    if (D == 128) return launch_d<128, true>(tk, tv, a, grid_rows, heads, rows_q, rows, rows_k, stream);
    return launch_d<64, true>(tk, tv, a, grid_rows, heads, rows_q, rows, rows_k, stream);
  }
  if (D == 128) return launch_d<128, false>(tk, tv, a, grid_rows, heads, rows_q, rows, rows_k, stream);
  return launch_d<64, false>(tk, tv, a, grid_rows, heads, rows_q, rows, rows_k, stream);
}

}  // namespace mslk
