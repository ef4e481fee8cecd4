// fmha_tc.cu — tensor-core attention forward / partial for sm_103a.
//
// Computes, for every query row i of a 256-row unit (two 128-row Q tiles) of one
// (batch or packed sequence, head):
//     out_i = sum_j softmax_j(scale * q_i . k_j) v_j      over the keys the mask allows
//     lse_i = ln sum_j exp(scale * q_i . k_j)
// as in MSLK's memory_efficient_attention ("Attention - Core fMHA"), streaming K/V in
// 128-key tiles so the score matrix never leaves the SM.
//
// Persistent: one CTA per SM walks a static list of units (heavy-first, snake-assigned);
// barrier phases carry across units, so the next unit's Q/K/V loads and first MMAs
// overlap the current unit's last tiles and its output.
// Per CTA (512 threads, four warpgroups):
//   warps 0-3   softmax for Q tile 0 (thread t owns row t = TMEM lane t)
//   warps 4-7   softmax for Q tile 1
//   warps 8-11  output: normalise O_t, store it (TMA), write lse; the softmax warpgroups
//               hand over their row max and sum and go straight on to the next unit
//   warp  12    tcgen05.mma issue (one elected thread) + TMEM allocation
//   warp  13    TMA producer (one elected thread); warps 14-15 idle
// Register budgets per warpgroup (setmaxnreg): softmax 176, output 96, MMA/TMA 64.
// Tensor memory (512 columns): S0 [0,128), S1 [128,256), O0 [256,256+D), O1 [384,384+D),
// fp32 accumulators, row r of a tile in lane r.  The bf16 probabilities P_t overwrite the
// first 64 columns of S_t (two values per column) and feed the PV MMA from tensor memory;
// they are published in two halves of 64 keys so the first half's PV runs while the
// second half is computed.
// Shared memory: Q0, Q1, a ring of K/V tiles (4 stages at D=128) and one output staging
// tile, in the 128-byte-swizzled K-major layout TMA writes (V is read MN-major by the PV
// MMA).  Each Q tile has its own full/empty barriers: the next unit's Q0 loads as soon as
// this unit's last S0 MMA has run, and the next unit's first S0 is issued as soon as Q
// tile 0 of this unit is done (one key tile before Q tile 1 under a causal mask).
// The MMA and TMA roles run as whole converged warps that issue through one elected lane:
// their operands stay warp-uniform, so they need few issue slots while the softmax
// warpgroups keep the SM's schedulers busy.
//
// MMA order (ping-pong: the tensor core works on one tile while the other tile's
// softmax runs):  S0_lo S1_lo | PV0_j S0_{j+1} PV1_j S1_{j+1} | ...  (each tile only over
// its own key tiles).  S_t(j+1) is committed after PV_t(j), so when a softmax warpgroup
// sees S_t(j+1) its O_t is stable (it may rescale it) and PV_t(j) has finished reading
// P_t; MMAs issued by one thread execute in order, so S_t(j+1) overwrites P_t(j) only
// after PV_t(j) read it.  Measured: issuing each tile's MMAs from its own warp instead
// was slower (the two streams interleave worse on the tensor core).
//
// Online softmax in base 2: m2 = running max of scale*log2(e)*s; p = 2^(scale*log2e*s - m2);
// l = running sum of p.  The running max used for p is only raised when the row max
// grows by more than 8 (a factor 256), which leaves the result exact (p, l and O all
// share the same reference) and makes O rescaling rare.  lse = (m2 + log2 l) * ln 2.
//
// Every mbarrier wait is bounded (globaltimer); a timeout sets the device error word,
// raises a CTA-wide abort flag, drains in-flight copies/MMAs and returns.
//
// Variants and modes:
//  * masks are one band lo <= key - row <= hi (causal, windows, bottom-right, kv_offset);
//    a unit only streams key tiles inside its rows' band; kLowerEdge compiles the lower
//    edge check in (windows);
//  * packed sequences (cu_seqlens) and key lanes (padded starts or a page table): a unit's
//    rows and keys come from its sequence; the V rows past a lane's end in its last tile
//    are zeroed in shared memory before the PV MMA (an unwritten cache tail may be NaN);
//  * grouped K/V heads: query head h reads K/V head h / kv_group;
//  * folded heads (fold = r): one query position per batch / sequence, the unit's rows are
//    the r query heads of one K/V head (q/out tensor maps are views), all at position 0;
//  * split units (the kSplit instantiation, launches with at most 128 rows per unit, e.g.
//    folded heads with r <= 128): both Q tiles hold the unit's rows and take alternate
//    key tiles, each with its own running max, sum and O, and the output warpgroup merges
//    the two by log-sum-exp (both tiles' max and sum through shared memory), so both
//    softmax warpgroups work on a decode unit;
//  * E4M3 inputs (fmha_tc_fp8_kernel, head dim 128): kind::f8f6f4 MMAs, one 128-byte
//    swizzle atom per row, E4M3 probabilities four per TMEM column, descales folded into
//    the exponent scale (q, k) and the output normalisation (v).

#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <mutex>
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace mslk {
namespace {

constexpr int kBlockM = 128;
constexpr int kBlockN = 128;
constexpr int kQTiles = 2;
constexpr int kUnitRows = kQTiles * kBlockM;
constexpr int kThreads = 512;
constexpr int kWarpOut = 8;   // warps 8-11: the output warpgroup
constexpr int kWarpMma = 12;
constexpr int kWarpLoad = 13;
// Registers per thread after the warpgroups rebalance (setmaxnreg).  Each scheduler
// partition holds one warp of every warpgroup, so the four shares add up to its 16384
// registers: 176 + 176 (softmax) + 96 (output) + 64 (MMA / TMA) = 512 per lane.
constexpr int kRegsSoftmax = 176;
constexpr int kRegsOut = 96;
constexpr int kRegsIssue = 64;
static_assert(2 * kRegsSoftmax + kRegsOut + kRegsIssue == 65536 / 4 / 32, "register split");
constexpr int kTmemCols = 512;
constexpr int kSwizzleAtom = 16384;  // one 64-column K-block of a 128-row tile (bytes)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 of the largest un-rescaled p (256)

// F8: q, k, v are E4M3 bytes; a 128-wide row is then one 128-byte swizzle atom.
template <int D, bool F8>
struct Layout {
  static constexpr int kEsz = F8 ? 1 : 2;             // bytes per input element
  static constexpr int kKBlocks = D * kEsz / 128;     // 128-byte swizzle atoms per row
  static constexpr int kTileBytes = kBlockM * D * kEsz;  // Q, K or V tile (128 rows)
  static constexpr int kStages = kTileBytes == 32768 ? 4 : 8;  // a 128 KiB K/V ring
  static constexpr int kQOff = 0;
  static constexpr int kKVOff = kQOff + kQTiles * kTileBytes;
  // Output staging: one 16 KiB buffer for the output warpgroup (128 rows x 128 bytes, the
  // 128-byte-swizzled layout of one TMA store box).
  static constexpr int kStageOutBytes = kBlockM * 128;
  static constexpr int kOutOff = kKVOff + kStages * kTileBytes;
  static constexpr int kBarOff = kOutOff + kStageOutBytes;
  // q_full[2], q_empty[2], kv_full[S], kv_empty[S], s_full[2], p_half[2], p_full[2],
  // o_done[2], o_free[2], st_full[2], st_empty[2], drain
  static constexpr int kNumBars = 4 + 2 * kStages + 14 + 1;
  static constexpr int kMiscOff = kBarOff + 8 * kNumBars;  // abort flag, tmem slot
  // Row statistics a softmax warpgroup hands to the output warpgroup at a unit's end:
  // [Q tile][row] (running max, running sum), fp32.
  static constexpr int kStatsOff = kMiscOff + 16;
  static constexpr int kBytes = kStatsOff + kQTiles * kBlockM * 8;
  static constexpr int kAlloc = kBytes + 1024;  // room to align the base to 1024
};

struct TcArgs {
  int M, Mkv, H;
  int Z;            // batches, or packed sequences
  int total_units;  // units_m * H * Z
  int kv_group;     // query heads per K/V head
  int varlen;
  int units_m;
  float scale_log2;
  // Key j of a sequence/chunk is allowed for its query row r iff r + lo <= j <= r + hi
  // (kv_offset already folded in; +-kBandOpen: open), plus Lk - Lq per packed sequence
  // when band_seq is set.
  long long lo, hi;
  int band_seq;
  // Key lanes (varlen only): lane_len[z] keys, at lane_start[z] + p or, paged, at
  // block_table[z * max_pages + p / page_size] * page_size + p % page_size.
  int lanes;
  const int* lane_len;
  const int* lane_start;
  const int* block_table;
  int page_size, max_pages;
  const int* cu_q;
  const int* cu_k;
  void* out;
  int out_fp32;
  long long so_b, so_m, so_h;
  float* lse;
  int tma_store;    // 1: write output tiles through shared memory with TMA stores
  // Folded query heads (fold = r > 1): one query position per batch / packed sequence, and
  // the unit's rows are the r query heads of K/V head h (q/out tensor maps are views of r
  // rows x H/r heads); every row sits at query position 0.
  int fold;
  long long lse_sb, lse_sh, lse_sm;
  // Output columns written: D, or the true head dim when a narrower one runs zero-padded
  // (head dim 96, or E4M3 head dim 64, on the 128-wide kernel: the tensor maps zero-fill
  // the missing columns).
  int d_out;  // lse element of (Q/O batch coordinate, head, row)
  // E4M3 inputs: element x of head h stands for x * descale[h] (descale[0] when
  // desc_per_tensor); q and k descales fold into the score scale, v's into the output.
  const float* dq;
  const float* dk;
  const float* dv;
  int desc_per_tensor;
  unsigned int* err;
  unsigned long long timeout_ns;
};

struct WaitCtl {
  volatile int* abort_flag;
  unsigned int* err;
  unsigned long long timeout_ns;
};

// Bounded wait: true when the phase completed; false on abort or timeout (which also
// raises the abort flag and records the timeout in the device error word).
MSLK_DEV bool wait_slow(uint32_t bar, uint32_t parity, const WaitCtl& w, bool honor_abort) {
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (honor_abort && *w.abort_flag) return false;
    if (globaltimer_ns() - t0 > w.timeout_ns) {
      *w.abort_flag = 1;
      atomicOr(w.err, kErrWaitTimeout);
      return false;
    }
  }
}
MSLK_DEV bool wait_bar(uint32_t bar, uint32_t parity, const WaitCtl& w, bool honor_abort = true) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_slow(bar, parity, w, honor_abort);
}

// Whole-warp wait with a warp-uniform result; the warp is converged afterwards.
MSLK_DEV bool wait_bar_warp(uint32_t bar, uint32_t parity, const WaitCtl& w, bool honor_abort = true) {
  const bool ok = __all_sync(0xffffffffu, wait_bar(bar, parity, w, honor_abort));
  __syncwarp();
  return ok;
}

MSLK_DEV float u2f(uint32_t x) { return __uint_as_float(x); }
MSLK_DEV uint32_t f2u(float x) { return __float_as_uint(x); }

// Shared-memory descriptors are built once per buffer; stepping to the next 16-element
// slice only adds a constant to the start-address field (16-byte units), so each MMA
// issue is two integer adds and the instruction itself.
MSLK_DEV uint64_t desc_kmajor(uint32_t saddr) { return smem_desc_sw128(saddr, 16, 1024); }
MSLK_DEV uint64_t desc_mnmajor(uint32_t saddr) { return smem_desc_sw128(saddr, kSwizzleAtom, 1024); }
// Start-address step (16-byte units) of K-slice kk in a K-major 128-byte-swizzled tile.
__host__ __device__ constexpr uint32_t kmajor_step(int kk) {
  return static_cast<uint32_t>(((kk / 4) * kSwizzleAtom + (kk % 4) * 32) >> 4);
}

// S_t = Q_t K^T over the head dim, 32 bytes of it per MMA (16 bf16 or 32 E4M3 columns).
template <int D, bool F8>
MSLK_DEV void issue_qk(uint32_t d_tmem, uint64_t q_desc, uint64_t k_desc) {
  if constexpr (F8) {
    constexpr uint32_t idesc = idesc_e4m3_f32(kBlockM, kBlockN, false);
#pragma unroll
    for (int kk = 0; kk < D / 32; ++kk)
      mma_f8_ss_elect(d_tmem, q_desc + kmajor_step(kk), k_desc + kmajor_step(kk), idesc, kk > 0 ? 1u : 0u);
  } else {
    constexpr uint32_t idesc = idesc_bf16_f32(kBlockM, kBlockN, false);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk)
      mma_f16_ss_elect(d_tmem, q_desc + kmajor_step(kk), k_desc + kmajor_step(kk), idesc, kk > 0 ? 1u : 0u);
  }
}

// O_t (+)= P_t V over the 128 keys of the tile.  P_t is read from tensor memory, 8 columns
// per MMA (16 bf16 keys, or 32 E4M3 keys); V is read MN-major: 8-key groups 1024 bytes
// apart (SBO), 128-byte column blocks of the head dim 16 KiB apart (LBO; bf16 has two);
// one MMA's keys span 2048 (bf16) or 4096 (E4M3) bytes.
// Half h of the tile's keys ([64 h, 64 h + 64)): the softmax publishes P in two halves so
// the first half's MMAs run while the second half's exponentials are computed.
template <int D, bool F8>
MSLK_DEV void issue_pv_half(uint32_t o_tmem, uint32_t p_tmem, uint64_t v_desc, uint32_t accumulate,
                            int h) {
  if constexpr (F8) {
    constexpr uint32_t idesc = idesc_e4m3_f32(kBlockM, D, true);
#pragma unroll
    for (int i = 0; i < kBlockN / 64; ++i) {
      const int kk = h * (kBlockN / 64) + i;
      mma_f8_ts_elect(o_tmem, p_tmem + kk * 8, v_desc + static_cast<uint32_t>(kk * 4096 / 16),
                      idesc, kk > 0 ? 1u : accumulate);
    }
  } else {
    constexpr uint32_t idesc = idesc_bf16_f32(kBlockM, D, true);
#pragma unroll
    for (int i = 0; i < kBlockN / 32; ++i) {
      const int kk = h * (kBlockN / 32) + i;
      mma_f16_ts_elect(o_tmem, p_tmem + kk * 8, v_desc + static_cast<uint32_t>(kk * 2048 / 16),
                       idesc, kk > 0 ? 1u : accumulate);
    }
  }
}

// Bits [0, n) set, n clamped to [0, 32].
MSLK_DEV uint32_t low_bits(int n) {
  return n >= 32 ? 0xffffffffu : (n <= 0 ? 0u : (1u << n) - 1u);
}

// One work unit: 256 query rows of one (batch or packed sequence, head).
struct Unit {
  int b, h, hk, z;
  int qb;  // batch coordinate of the unit's Q/O rows (a packed row when folded and varlen)
  int q_base, Lq, k_base, Lk;
  int r0;
  int lo, hi;  // the band of this unit's sequence (see TcArgs), clamped to +-2^30
  // Q tile t takes key tiles tlo[t], tlo[t] + step, ... below thi[t] (empty: tlo == thi);
  // the unit streams [jlo, jhi), their union, which has no gaps because the band's lower
  // edge never passes its upper edge.  step = 2 (split): the unit's rows fit one Q tile,
  // and both Q tiles hold those rows and take alternate key tiles, each with its own
  // running max, sum and O; the epilogue merges the two by their log-sum-exp.
  int tlo[2], thi[2];
  int jlo, jhi;
  int step;
  MSLK_DEV bool has(int t) const { return tlo[t] < thi[t]; }
  MSLK_DEV bool has(int t, int j) const {
    return tlo[t] <= j && j < thi[t] && (step == 1 || ((j - tlo[t]) & 1) == 0);
  }
  // (has(t)) step is 1 or 2: a shift, not a divide (a divide takes the special-function
  // unit, which the softmax warps keep busy with exponentials)
  MSLK_DEV int count(int t) const { return (thi[t] - tlo[t] + step - 1) >> (step - 1); }
  MSLK_DEV int last(int t) const { return tlo[t] + (count(t) - 1) * step; }         // (has(t))
  MSLK_DEV int row0(int t) const { return r0 + (step == 2 ? 0 : t * kBlockM); }  // first row
};

// Unit i of the heavy-first order: unit rows descend level by level (causal units late in
// the sequence see the most keys), heads vary fastest within a level.  Returns false if
// the unit has no rows (a packed sequence shorter than the unit's first row).
template <bool kSplit>
MSLK_DEV bool decode_unit(const TcArgs& a, int i, Unit& u) {
  const int per_level = a.H * a.Z;
  const int level = i / per_level;
  const int rem = i - level * per_level;
  const int unit_m = a.units_m - 1 - level;
  u.h = rem % a.H;
  const int z = rem / a.H;
  u.hk = u.h / a.kv_group;
  u.z = z;
  if (a.varlen) {
    u.b = 0;
    const int qs = min(max(a.cu_q[z], 0), a.M);
    const int qe = min(max(a.cu_q[z + 1], qs), a.M);
    u.q_base = qs;
    u.Lq = qe - qs;
    if (a.lanes) {
      // Rows outside [0, Mkv) are clipped by the tensor map (zero fill); a paged lane is
      // cut at the end of its page table.
      u.k_base = a.block_table != nullptr ? 0 : a.lane_start[z];
      int len = max(a.lane_len[z], 0);
      if (a.block_table != nullptr) len = static_cast<int>(min(static_cast<long long>(len),
                                                               static_cast<long long>(a.max_pages) * a.page_size));
      u.Lk = len;
    } else {
      const int ks = min(max(a.cu_k[z], 0), a.Mkv);
      const int ke = min(max(a.cu_k[z + 1], ks), a.Mkv);
      u.k_base = ks;
      u.Lk = ke - ks;
    }
  } else {
    u.b = z;
    u.q_base = 0;
    u.Lq = a.M;
    u.k_base = 0;
    u.Lk = a.Mkv;
  }
  u.qb = u.b;
  int lq_pos = u.Lq;  // query positions of the block (1 when heads are folded into rows)
  if (a.fold) {
    if (u.Lq <= 0) return false;  // a packed sequence without a query
    u.qb = a.varlen ? u.q_base : z;
    u.q_base = 0;
    u.Lq = a.fold;
    lq_pos = 1;
  }
  u.r0 = unit_m * kUnitRows;
  if (u.r0 < 0 || u.r0 >= u.Lq) return false;  // (a unit index past the unit space)
  {
    long long lo = a.lo, hi = a.hi;
    if (a.band_seq) {
      const long long shift = static_cast<long long>(u.Lk) - lq_pos;
      if (lo > -kBandOpen) lo += shift;
      if (hi < kBandOpen) hi += shift;
    }
    // Row and key positions are below 2^31, so bounds beyond +-2^30 of any difference
    // that matters act as open; clamping keeps the per-row arithmetic in 32 bits.
    constexpr long long kClamp = 1LL << 30;
    u.lo = static_cast<int>(max(-kClamp, min(kClamp, lo)));
    u.hi = static_cast<int>(max(-kClamp, min(kClamp, hi)));
  }
  for (int t = 0; t < kQTiles; ++t) {
    const long long row0 = u.r0 + t * kBlockM;
    u.tlo[t] = u.thi[t] = 0;
    if (row0 >= u.Lq) continue;  // rows past the sequence: nothing to compute
    const long long row1 = min(row0 + kBlockM, static_cast<long long>(u.Lq)) - 1;
    const long long p0 = a.fold ? 0 : row0, p1 = a.fold ? 0 : row1;  // query positions
    const long long k_first = max(0LL, p0 + u.lo);
    const long long k_last = min(static_cast<long long>(u.Lk) - 1, p1 + u.hi);
    if (k_first > k_last) continue;
    u.tlo[t] = static_cast<int>(k_first / kBlockN);
    u.thi[t] = static_cast<int>(k_last / kBlockN) + 1;
  }
  u.step = 1;
  if (kSplit && u.r0 + kBlockM >= u.Lq && u.thi[0] - u.tlo[0] >= 2) {
    // One Q tile of rows over two or more key tiles: split them between both Q tiles.
    u.step = 2;
    u.tlo[1] = u.tlo[0] + 1;
    u.thi[1] = u.thi[0];
  }
  if (u.has(0) && u.has(1)) {
    u.jlo = min(u.tlo[0], u.tlo[1]);
    u.jhi = max(u.thi[0], u.thi[1]);
  } else {
    u.jlo = u.has(0) ? u.tlo[0] : u.tlo[1];
    u.jhi = u.has(0) ? u.thi[0] : u.thi[1];
  }
  return true;
}

// Static schedule over the heavy-first order, in snake rounds: CTA c takes position c of
// even rounds and position G-1-c of odd rounds, which evens out the per-CTA work.
MSLK_DEV int unit_at(int round, int c, int G) {
  return round * G + ((round & 1) ? (G - 1 - c) : c);
}

// kLowerEdge: the band has a lower edge (a local window), so masked tiles test both
// edges; without it the per-row lower limit is compiled out of the softmax.
// F8: E4M3 q, k, v (kind::f8f6f4 MMAs; P is rounded to E4M3 for the PV MMA).
template <int D, bool kLowerEdge, bool F8, bool kSplit>
MSLK_DEV void tc_body(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                      const CUtensorMap& tm_o, const TcArgs& a) {
  using L = Layout<D, F8>;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned, derived from the shared array itself so accesses stay shared-space
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  // (broadcast from lane 0: the compiler then knows the role branches are warp-uniform,
  // which the per-role register budgets below rely on)
  const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x / 32), 0);
  const int lane = threadIdx.x % 32;
  const int G = gridDim.x;
  // A following launch declared independent of this one may start now (the others wait
  // for this grid to complete as usual).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int cta = blockIdx.x;
  const int n_rounds = (a.total_units + G - 1) / G;

  // ---------------------------------------------------------------- setup
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  const uint32_t bar0 = smem_u32(bars);
  auto q_full = [&](int t) { return bar0 + 8u * t; };        // Q tile t loaded
  auto q_empty = [&](int t) { return bar0 + 8u * (2 + t); };  // Q tile t's last S MMA done
  auto kv_full = [&](int s) { return bar0 + 8u * (4 + s); };
  auto kv_empty = [&](int s) { return bar0 + 8u * (4 + L::kStages + s); };
  auto s_full = [&](int t) { return bar0 + 8u * (4 + 2 * L::kStages + t); };
  // P_t's first 64 keys / all 128 are in tensor memory (the PV MMAs over them may start)
  auto p_half = [&](int t) { return bar0 + 8u * (6 + 2 * L::kStages + t); };
  auto p_full = [&](int t) { return bar0 + 8u * (8 + 2 * L::kStages + t); };
  auto o_done = [&](int t) { return bar0 + 8u * (10 + 2 * L::kStages + t); };  // O_t final
  auto o_free = [&](int t) { return bar0 + 8u * (12 + 2 * L::kStages + t); };  // O_t read out
  // softmax warpgroup t wrote its rows' max and sum / the output warpgroup read them
  auto st_full = [&](int t) { return bar0 + 8u * (14 + 2 * L::kStages + t); };
  auto st_empty = [&](int t) { return bar0 + 8u * (16 + 2 * L::kStages + t); };
  const uint32_t bar_drain = bar0 + 8u * (18 + 2 * L::kStages);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff + 8);
  const WaitCtl wc{abort_flag, a.err, a.timeout_ns};

  const uint32_t s_base = smem_u32(smem);
  auto q_addr = [&](int t) { return s_base + L::kQOff + t * L::kTileBytes; };
  auto kv_addr = [&](int s) { return s_base + L::kKVOff + s * L::kTileBytes; };

  if (threadIdx.x == 0) {
    for (int t = 0; t < kQTiles; ++t) {
      mbar_init(q_full(t), 1);
      mbar_init(q_empty(t), 1);
    }
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(kv_full(s), 1);
      mbar_init(kv_empty(s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(s_full(t), 1);
      mbar_init(p_full(t), kBlockM / 32);  // one arrival per softmax warp
      mbar_init(p_half(t), kBlockM / 32);
      mbar_init(o_done(t), 1);
      mbar_init(o_free(t), kBlockM / 32);  // one arrival per output warp
      mbar_init(st_full(t), kBlockM / 32);
      mbar_init(st_empty(t), kBlockM / 32);
    }
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpLoad && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    if (a.tma_store) tma_prefetch_desc(&tm_o);
  }
  if (warp == kWarpMma) {
    __syncwarp();
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= kWarpMma) {
    setmaxnreg_dec<kRegsIssue>();  // MMA, TMA and two idle warps
  if (warp == kWarpLoad) {
    // ------------------------------------------------------------ TMA producer (whole warp)
    // Order per unit: Q0, K_lo, Q1, V_lo, K_lo+1, V_lo+1, ...  Each Q tile waits only for its own
    // tile's last S MMA of the previous unit, so the next unit's Q0 (and K_0) arrive in
    // time for the MMA warp to start S0_0 before the current unit's last tile-1 step.
    int uc = 0, it = 0;
    int q_issued[kQTiles] = {0, 0};
    bool ok = true;
    auto load_q = [&](int t, const Unit& u) {
      if (!(ok = wait_bar_warp(q_empty(t), (uc & 1) ^ 1, wc))) return;
      mbar_arrive_expect_tx_elect(q_full(t), L::kTileBytes);
      for (int kb = 0; kb < L::kKBlocks; ++kb)
        tma_load_4d_elect(q_addr(t) + kb * kSwizzleAtom, &tm_q, q_full(t), kb * (128 / L::kEsz),
                          u.q_base + u.row0(t), u.h, u.qb);
      ++q_issued[t];
    };
    auto load_kv = [&](int j, int which, const Unit& u) {  // K_j (which = 0) or V_j
      const int s = it % L::kStages;
      if (!(ok = wait_bar_warp(kv_empty(s), ((it / L::kStages) & 1) ^ 1, wc))) return;
      mbar_arrive_expect_tx_elect(kv_full(s), L::kTileBytes);
      const CUtensorMap* tm = which ? &tm_v : &tm_k;
      int row = u.k_base + j * kBlockN;
      if (a.block_table != nullptr) {  // paged lane: the tile lies inside one page
        const int key = j * kBlockN;
        row = a.block_table[static_cast<long long>(u.z) * a.max_pages + key / a.page_size] * a.page_size +
              key % a.page_size;
      }
      for (int kb = 0; kb < L::kKBlocks; ++kb)
        tma_load_4d_elect(kv_addr(s) + kb * kSwizzleAtom, tm, kv_full(s), kb * (128 / L::kEsz), row, u.hk, u.b);
      ++it;
    };
    for (int k = 0; k < n_rounds && ok; ++k) {
      const int i = unit_at(k, cta, G);
      Unit u;
      if (i >= a.total_units || !decode_unit<kSplit>(a, i, u) || u.jhi <= u.jlo) continue;
      load_q(0, u);
      if (ok) load_kv(u.jlo, 0, u);
      if (ok) load_q(1, u);
      if (ok) load_kv(u.jlo, 1, u);
      for (int j = u.jlo + 1; j < u.jhi && ok; ++j) {
        load_kv(j, 0, u);
        if (ok) load_kv(j, 1, u);
      }
      if (ok) ++uc;
    }
    if (!ok) {  // let every copy this warp issued land before the CTA exits
      for (int t = 0; t < kQTiles; ++t)
        if (q_issued[t] > 0) wait_bar_warp(q_full(t), (q_issued[t] - 1) & 1, wc, false);
      for (int k = max(0, it - L::kStages); k < it; ++k)
        wait_bar_warp(kv_full(k % L::kStages), (k / L::kStages) & 1, wc, false);
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer (whole warp)
    const uint32_t tm_s[2] = {tmem + 0u, tmem + 128u};
    const uint32_t tm_o[2] = {tmem + 256u, tmem + 384u};
    const uint64_t q_desc[2] = {desc_kmajor(q_addr(0)), desc_kmajor(q_addr(1))};
    // Ring stages are kTileBytes apart: stage s adds s * kTileBytes / 16 to the address field.
    const uint64_t kdesc0 = desc_kmajor(kv_addr(0));
    const uint64_t vdesc0 = desc_mnmajor(kv_addr(0));
    auto kv_kdesc = [&](int st) { return kdesc0 + static_cast<uint32_t>(st * (L::kTileBytes >> 4)); };
    auto kv_vdesc = [&](int st) { return vdesc0 + static_cast<uint32_t>(st * (L::kTileBytes >> 4)); };
    // uc: units; uc_t: units in which Q tile t has keys (o_free phases); jg_t: its key tiles.
    int uc = 0, it = 0, uc0 = 0, uc1 = 0, jg0 = 0, jg1 = 0;
    bool ok = true;
    // Units are decoded 32 rounds at a time, one per lane (a decode costs ~1.5k cycles of
    // integer divides and parameter loads, which at every unit boundary sat between this
    // warp's last P.V and the next S); the MMA fields of round batch + l stay in lane l's
    // registers and are fetched with shuffles.
    int batch = -32;          // first round of the decoded batch
    uint32_t with_work = 0;   // lanes whose unit has key tiles
    int m_jlo = 0, m_jhi = 0, m_tlo0 = 0, m_thi0 = 0, m_tlo1 = 0, m_thi1 = 0, m_step = 1, m_lk = 0;
    auto decode_batch = [&](int first) {
      batch = first;
      const int k = first + lane;
      Unit uu;
      bool work = false;
      if (k < n_rounds) {
        const int i = unit_at(k, cta, G);
        work = i < a.total_units && decode_unit<kSplit>(a, i, uu) && uu.jhi > uu.jlo;
      }
      if (work) {
        m_jlo = uu.jlo; m_jhi = uu.jhi; m_tlo0 = uu.tlo[0]; m_thi0 = uu.thi[0];
        m_tlo1 = uu.tlo[1]; m_thi1 = uu.thi[1]; m_step = uu.step; m_lk = uu.Lk;
      }
      with_work = __ballot_sync(0xffffffffu, work);
    };
    // The next unit with work at or after round k (k_out = its round), false if none; only
    // the fields this warp reads are set in uo.
    auto next_unit = [&](int k, int& k_out, Unit& uo) {
      if constexpr (F8) {  // (measured: the E4M3 kernel runs better decoding in place)
        for (; k < n_rounds; ++k) {
          const int i = unit_at(k, cta, G);
          if (i < a.total_units && decode_unit<kSplit>(a, i, uo) && uo.jhi > uo.jlo) {
            k_out = k;
            return true;
          }
        }
        return false;
      } else {
        while (k < n_rounds) {
          if (k < batch || k >= batch + 32) decode_batch(k & ~31);
          const uint32_t m = with_work & (0xffffffffu << (k - batch));
          if (m != 0u) {
            const int l = __ffs(m) - 1;
            k_out = batch + l;
            uo.jlo = __shfl_sync(0xffffffffu, m_jlo, l);
            uo.jhi = __shfl_sync(0xffffffffu, m_jhi, l);
            uo.tlo[0] = __shfl_sync(0xffffffffu, m_tlo0, l);
            uo.thi[0] = __shfl_sync(0xffffffffu, m_thi0, l);
            uo.tlo[1] = __shfl_sync(0xffffffffu, m_tlo1, l);
            uo.thi[1] = __shfl_sync(0xffffffffu, m_thi1, l);
            uo.step = __shfl_sync(0xffffffffu, m_step, l);
            uo.Lk = __shfl_sync(0xffffffffu, m_lk, l);
            return true;
          }
          k = batch + 32;
        }
        return false;
      }
    };
    Unit u;
    int ku = 0;
    bool have = next_unit(0, ku, u);
    bool s0_issued = false;  // the unit's first S0 was issued during the previous unit
    bool v_ready = false;    // (E4M3) the key tile's V was waited for in the previous step
    // The next unit's first S0 (its Q0 was loaded after this unit's last S0 MMA; its first K
    // is ring entry ikn).  S0 is free: this unit's last PV0 precedes it in issue order.
    auto issue_next_s0 = [&](const Unit& un, int ikn) {
      if (!(ok = wait_bar_warp(q_full(0), (uc + 1) & 1, wc))) return;
      if (!(ok = wait_bar_warp(kv_full(ikn % L::kStages), (ikn / L::kStages) & 1, wc))) return;
      tc_fence_after();
      issue_qk<D, F8>(tm_s[0], q_desc[0], kv_kdesc(ikn % L::kStages));
      mma_commit_elect(s_full(0));
      if (un.last(0) == un.jlo) mma_commit_elect(q_empty(0));
      s0_issued = true;
    };
    while (have && ok) {
      Unit un;
      int kn = 0;
      const bool have_next = next_unit(ku + 1, kn, un);
      const int jlo = u.jlo;
      const int jhi = u.jhi;
      // Q tile t's first and last key tiles (last < first: none)
      const int lo0 = u.tlo[0], lo1 = u.tlo[1];
      const int last0 = u.has(0) ? u.last(0) : lo0 - 1, last1 = u.has(1) ? u.last(1) : lo1 - 1;
      const int ik0 = it++;  // K_jlo's ring position
      const int sk0 = ik0 % L::kStages;
      // S_t(jlo): S_t is free (its last P was consumed by the previous unit's PV_t, which
      // was issued before this and executes first).  Q tile 0 starts at jlo whenever it
      // has keys (its rows come first, so its key range starts first).
      if (!s0_issued) {
        if (!(ok = wait_bar_warp(q_full(0), uc & 1, wc))) break;
        if (!(ok = wait_bar_warp(kv_full(sk0), (ik0 / L::kStages) & 1, wc))) break;
        tc_fence_after();
        if (u.has(0, jlo)) {
          issue_qk<D, F8>(tm_s[0], q_desc[0], kv_kdesc(sk0));
          mma_commit_elect(s_full(0));
        }
        if (!u.has(0) || last0 == jlo) mma_commit_elect(q_empty(0));  // Q0's last S issued
      }
      s0_issued = false;
      if (!(ok = wait_bar_warp(q_full(1), uc & 1, wc))) break;
      if (!(ok = wait_bar_warp(kv_full(sk0), (ik0 / L::kStages) & 1, wc))) break;
      tc_fence_after();
      if (u.has(1, jlo)) {
        issue_qk<D, F8>(tm_s[1], q_desc[1], kv_kdesc(sk0));
        mma_commit_elect(s_full(1));
      }
      mma_commit_elect(kv_empty(sk0));
      if (!u.has(1) || last1 == jlo) mma_commit_elect(q_empty(1));
      for (int j = jlo; j < jhi && ok; ++j) {
        const bool more = j + 1 < jhi;
        const int iv = it;       // V_j's ring position
        const int ik = it + 1;   // K_{j+1}'s
        it += more ? 2 : 1;
        const int sv = iv % L::kStages;
        const int sk = ik % L::kStages;
        if (!v_ready && !(ok = wait_bar_warp(kv_full(sv), (iv / L::kStages) & 1, wc))) break;
        v_ready = false;
        if (a.lane_len != nullptr && (j + 1) * kBlockN > u.Lk) {
          // A key lane's last tile: the rows past its last key may hold anything (an
          // unwritten cache).  Their P is 0, but 0 * NaN is NaN in the PV MMA, so they are
          // cleared first (row r of each 64-column block: bytes [128 r, 128 r + 128)).
          const int r0 = max(0, u.Lk - j * kBlockN);
          uint8_t* vt = smem + L::kKVOff + sv * L::kTileBytes;
          for (int kb = 0; kb < L::kKBlocks; ++kb)
            for (int off = r0 * 128 + lane * 16; off < kBlockN * 128; off += 32 * 16)
              *reinterpret_cast<uint4*>(vt + kb * kSwizzleAtom + off) = make_uint4(0, 0, 0, 0);
          fence_proxy_async_smem();  // generic-proxy writes, read next by the tensor core
          __syncwarp();
        }
        if (u.step == 2) {
          // Split unit: key tile j belongs to Q tile tj, j + 1 to the other one (tn).
          // S_tn(j+1) goes first, so tn's softmax runs while tj's does; S_tn is free (its
          // last P was read by PV_tn(j-1), issued before).
          const int tj = (j - jlo) & 1, tn = tj ^ 1;
          if (more) {
            if (!(ok = wait_bar_warp(kv_full(sk), (ik / L::kStages) & 1, wc))) break;
            tc_fence_after();
            issue_qk<D, F8>(tm_s[tn], q_desc[tn], kv_kdesc(sk));
            mma_commit_elect(s_full(tn));
            if (j + 1 == (tn ? last1 : last0)) mma_commit_elect(q_empty(tn));
          }
          const int lo_j = tj ? lo1 : lo0;
          if (!(ok = wait_bar_warp(p_half(tj), (tj ? jg1 : jg0) & 1, wc))) break;
          if (j == lo_j && !(ok = wait_bar_warp(o_free(tj), ((tj ? uc1 : uc0) & 1) ^ 1, wc))) break;
          tc_fence_after();
          issue_pv_half<D, F8>(tm_o[tj], tm_s[tj], kv_vdesc(sv), j > lo_j ? 1u : 0u, 0);
          if (!(ok = wait_bar_warp(p_full(tj), (tj ? jg1 : jg0) & 1, wc))) break;
          tc_fence_after();
          issue_pv_half<D, F8>(tm_o[tj], tm_s[tj], kv_vdesc(sv), 1u, 1);
          // o_done(0) after the unit's last PV of either tile: O_0 and O_1 both final
          // (tile 0 merges them; o_done(1) has no phase in split units)
          if (!more) mma_commit_elect(o_done(0));
          if (tj) ++jg1; else ++jg0;
          mma_commit_elect(kv_empty(sv));
          if (more) mma_commit_elect(kv_empty(sk));
        } else {
          // Q tile 0 (when key tile j is one of its tiles): PV0_j, then S0_{j+1}
          if (u.has(0, j)) {
            if (!(ok = wait_bar_warp(p_half(0), jg0 & 1, wc))) break;
            if (j == lo0 && !(ok = wait_bar_warp(o_free(0), (uc0 & 1) ^ 1, wc))) break;
            tc_fence_after();
            issue_pv_half<D, F8>(tm_o[0], tm_s[0], kv_vdesc(sv), j > lo0 ? 1u : 0u, 0);
            if (!(ok = wait_bar_warp(p_full(0), jg0 & 1, wc))) break;
            tc_fence_after();
            issue_pv_half<D, F8>(tm_o[0], tm_s[0], kv_vdesc(sv), 1u, 1);
            if (j == last0) mma_commit_elect(o_done(0));
            ++jg0;
          }
          if (!more && j == last0 && have_next && un.has(0)) {
            // Both tiles end here: the next unit's S0 goes ahead of PV1, so softmax 0
            // starts the next unit while softmax 1 finishes this one.  (Its first K
            // follows V_j in the ring: entry it.)
            issue_next_s0(un, it);
            if (!ok) break;
          }
          if (more) {
            if (!(ok = wait_bar_warp(kv_full(sk), (ik / L::kStages) & 1, wc))) break;
            tc_fence_after();
            if (u.has(0, j + 1)) {
              issue_qk<D, F8>(tm_s[0], q_desc[0], kv_kdesc(sk));
              mma_commit_elect(s_full(0));
              if (j + 1 == last0) mma_commit_elect(q_empty(0));
            }
          }
          // Q tile 1: PV1_j, then S1_{j+1}
          if (u.has(1, j)) {
            if (!(ok = wait_bar_warp(p_half(1), jg1 & 1, wc))) break;
            if (j == lo1 && !(ok = wait_bar_warp(o_free(1), (uc1 & 1) ^ 1, wc))) break;
            tc_fence_after();
            issue_pv_half<D, F8>(tm_o[1], tm_s[1], kv_vdesc(sv), j > lo1 ? 1u : 0u, 0);
            if (!(ok = wait_bar_warp(p_full(1), jg1 & 1, wc))) break;
            tc_fence_after();
            issue_pv_half<D, F8>(tm_o[1], tm_s[1], kv_vdesc(sv), 1u, 1);
            if (j == last1) mma_commit_elect(o_done(1));
            ++jg1;
          }
          mma_commit_elect(kv_empty(sv));
          if (more) {
            if constexpr (F8) {
              // E4M3: V_{j+1} (ring entry it) is waited for here, ahead of S1_{j+1}, so the
              // step from S1_{j+1} to PV0_{j+1} has one wait less; measured 55.3-55.6 vs
              // 57.2 us causal.  (The bf16 kernel runs slower this way: with its 4-stage
              // ring V_{j+1} is not always in yet.)
              if (!(ok = wait_bar_warp(kv_full(it % L::kStages), (it / L::kStages) & 1, wc))) break;
              v_ready = true;
            }
            if (u.has(1, j + 1)) {
              issue_qk<D, F8>(tm_s[1], q_desc[1], kv_kdesc(sk));
              mma_commit_elect(s_full(1));
              if (j + 1 == last1) mma_commit_elect(q_empty(1));  // the unit's last S1 MMA was issued
            }
            mma_commit_elect(kv_empty(sk));
            if (j == last0 && j + 2 == jhi && have_next && un.has(0)) {
              // Q tile 0 is done one key tile before Q tile 1 (causal): the next unit's S0
              // runs while softmax 1 works on this unit's last tile.  Ring: V_{j+1} is entry
              // it, the next unit's first K entry it + 1 (within the ring: it - 3 was waited on).
              issue_next_s0(un, it + 1);
              if (!ok) break;
            }
          }
        }
        if (!more && have_next && un.has(0) && !s0_issued) {
          // Otherwise the next unit's first S0 right behind this unit's last PV, before this
          // warp decodes units and waits for Q1 (its first K follows V_{jhi-1}: entry it).
          issue_next_s0(un, it);
          if (!ok) break;
        }
      }
      if (!ok) break;
      ++uc;
      if (u.has(0)) ++uc0;
      if (u.has(1)) ++uc1;
      u = un;
      ku = kn;
      have = have_next;
    }
    if (!ok) {  // wait for every MMA this warp issued
      mma_commit_elect(bar_drain);
      wait_bar_warp(bar_drain, 0, wc, false);
    }
  }
  } else if (warp < kWarpOut) {
    setmaxnreg_inc<kRegsSoftmax>();
    // ------------------------------------------------------------ softmax warpgroups
    const int t = warp / 4;                   // Q tile
    const int row_in_tile = (warp % 4) * 32 + lane;
    const uint32_t lane_bits = static_cast<uint32_t>((warp % 4) * 32) << 16;
    const uint32_t ts = tmem + static_cast<uint32_t>(t * 128) + lane_bits;
    const uint32_t to = tmem + 256u + static_cast<uint32_t>(t * 128) + lane_bits;
    // Barrier phase parities, one register: bit 1 s_full(t) (this tile's key tiles), bit 2
    // st_empty(t) (units in which this tile handed row statistics over).
    uint32_t ph = 0;
    bool ok = true;
    for (int k = 0; k < n_rounds && ok; ++k) {
      const int i = unit_at(k, cta, G);
      Unit u;
      if (i >= a.total_units || !decode_unit<kSplit>(a, i, u)) continue;
      const int row_first = u.row0(t);  // first row of this Q tile (sequence coords)
      const int r = row_first + row_in_tile;
      // this Q tile's key tiles (selects, not a runtime index, keep u in registers)
      const int tlo_t = t == 0 ? u.tlo[0] : u.tlo[1];
      const int n_t = ((t == 0 ? u.thi[0] : u.thi[1]) - tlo_t + u.step - 1) >> (u.step - 1);
      float sl2 = a.scale_log2;
      if constexpr (F8) {
        const int hq = a.fold ? u.h * a.fold + min(r, a.fold - 1) : u.h;  // this row's query head
        sl2 *= a.dq[a.desc_per_tensor ? 0 : hq] * a.dk[a.desc_per_tensor ? 0 : u.hk];
      }
      if (n_t <= 0) continue;  // no allowed key for any row: the output warpgroup writes them
      float m_run = -INFINITY;
      float l_run = 0.f;
      for (int j = 0; j < n_t; ++j, ph ^= 2u) {
        // tcgen05.ld is warp-collective: take every wait decision warp-uniformly.
        ok = __all_sync(0xffffffffu, wait_bar(s_full(t), (ph >> 1) & 1u, wc));
        if (!ok) break;
        __syncwarp();
        tc_fence_after();
        const int key0 = (tlo_t + j * u.step) * kBlockN;
        // The tile is allowed whole for every row iff its last key is below Lk and within
        // the first row's upper band edge and its first key is within the last row's lower
        // edge; otherwise column c is allowed iff lim_lo <= c <= lim_c (this row's band
        // edges, and key < Lk).
        // (query positions: the row's own, or 0 for every row when heads are folded)
        const int pos_first = a.fold ? 0 : row_first;
        const int pos_last = a.fold ? 0 : row_first + kBlockM - 1;
        const int pos = a.fold ? 0 : r;
        const bool need_mask = (key0 + kBlockN > u.Lk) ||
                               (key0 + kBlockN - 1 > pos_first + u.hi) ||
                               (kLowerEdge && key0 < pos_last + u.lo);
        int lim_c = kBlockN - 1, lim_lo = 0;
        if (need_mask) {
          lim_c = max(-1, min(min(u.Lk - 1, pos + u.hi) - key0, kBlockN - 1));
          if constexpr (kLowerEdge) lim_lo = max(0, min(max(0, pos + u.lo) - key0, kBlockN));
        }
        // The whole S row comes out of tensor memory (two 64-column loads, one wait; 128
        // registers): mask it (only tiles crossing a mask limit), take the row max, then
        // form p = 2^(s*scale*log2e - m) and the row sum and write P as bf16 pairs over S's
        // first 64 columns, a quarter (16 columns) at a time.  P is published in two halves
        // of 64 keys: the MMA warp issues P.V over the first half while the second half's
        // exponentials run.
        uint32_t sr[128];
        tmem_ld_32x32b_x64_nowait(ts, sr);
        tmem_ld_32x32b_x64_nowait(ts + 64, sr + 64);
        tmem_ld_wait();
        if (need_mask) {
          // One allowed-column bit word per 32 columns, then a bit test per column:
          // -inf is excluded from the max and 2^-inf = 0.
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t w = low_bits(lim_c + 1 - 32 * q4);
            if constexpr (kLowerEdge) w &= ~low_bits(lim_lo - 32 * q4);
#pragma unroll
            for (int c = 0; c < 32; ++c)
              if (!((w >> c) & 1u)) sr[32 * q4 + c] = 0xFF800000u;
          }
        }
        float mx8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) mx8[e] = fmax3(u2f(sr[e]), u2f(sr[8 + e]), u2f(sr[16 + e]));
#pragma unroll
        for (int c = 24; c < 120; c += 16)
#pragma unroll
          for (int e = 0; e < 8; ++e) mx8[e] = fmax3(mx8[e], u2f(sr[c + e]), u2f(sr[c + 8 + e]));
#pragma unroll
        for (int e = 0; e < 8; ++e) mx8[e] = fmaxf(mx8[e], u2f(sr[120 + e]));
        const float mx = fmaxf(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], fmax3(mx8[5], mx8[6], mx8[7])));
        const float m_new = fmaxf(m_run, mx * sl2);
        const bool rescale = m_new > m_run + kRescaleThreshold;
        float alpha = 1.f;
        if (rescale) {
          alpha = ex2_approx(m_run - m_new);
          m_run = m_new;
        }
        l_run *= alpha;
        if (j > 0 && __any_sync(0xffffffffu, rescale)) {
          // O_t is stable here: PV_t(j-1) completed before S_t(j) was signalled, and
          // PV_t(j) is not issued before P's first half is published.  (8 columns at a
          // time: the S row still occupies 128 registers.)
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 8) {
            uint32_t o[8];
            tmem_ld_32x32b_x8(to + c0, o);
#pragma unroll
            for (int e = 0; e < 8; ++e) o[e] = f2u(u2f(o[e]) * alpha);
            tmem_st_32x32b_x8(to + c0, o);
          }
        }
        const float msub = (m_run == -INFINITY) ? 0.f : m_run;
        const uint64_t sl2x2 = pack_f2(sl2, sl2);
        const uint64_t nmx2 = pack_f2(-msub, -msub);
        uint64_t rs2[4] = {0ull, 0ull, 0ull, 0ull};  // 8 independent partial sums, in pairs
#pragma unroll
        for (int qtr = 0; qtr < 4; ++qtr) {
          if constexpr (F8) {
            // P as E4M3, four per column, over S's first 32 columns.  p <= 2^8 (the lazy
            // rescale bound) stays inside E4M3's range (448).
            uint32_t pk[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const int c = qtr * 32 + 4 * e;
              const float2 x = unpack_f2(ffma2(pack_f2(u2f(sr[c]), u2f(sr[c + 1])), sl2x2, nmx2));
              const float2 y = unpack_f2(ffma2(pack_f2(u2f(sr[c + 2]), u2f(sr[c + 3])), sl2x2, nmx2));
              const float p0 = ex2_approx(x.x), p1 = ex2_approx(x.y);
              const float p2 = ex2_approx(y.x), p3 = ex2_approx(y.y);
              rs2[(2 * e) % 4] = fadd2(rs2[(2 * e) % 4], pack_f2(p0, p1));
              rs2[(2 * e + 1) % 4] = fadd2(rs2[(2 * e + 1) % 4], pack_f2(p2, p3));
              pk[e] = pack_e4m3x4(p0, p1, p2, p3);
            }
            tmem_st_32x32b_x8(ts + qtr * 8, pk);
          } else {
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int c = qtr * 32 + 2 * e;
              const float2 x = unpack_f2(ffma2(pack_f2(u2f(sr[c]), u2f(sr[c + 1])), sl2x2, nmx2));
              const float p0 = ex2_approx(x.x);
              const float p1 = ex2_approx(x.y);
              rs2[e % 4] = fadd2(rs2[e % 4], pack_f2(p0, p1));
              pk[e] = pack_bf16x2(p0, p1);
            }
            tmem_st_32x32b_x16(ts + qtr * 16, pk);
          }
          if (qtr == 1) {  // keys [0, 64) of P_t are in tensor memory
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_half(t));
          }
        }
        {
          const float2 r0 = unpack_f2(fadd2(rs2[0], rs2[1]));
          const float2 r1 = unpack_f2(fadd2(rs2[2], rs2[3]));
          l_run += (r0.x + r0.y) + (r1.x + r1.y);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full(t));  // one arrival per warp
      }
      // Hand the row's max and sum to the output warpgroup (once it has read the previous
      // unit's) and go straight on to the next unit: the output warpgroup normalises and
      // stores O_t while this warpgroup's next tiles run.
      ok = ok && __all_sync(0xffffffffu, wait_bar(st_empty(t), ((ph >> 2) & 1u) ^ 1u, wc));
      if (!ok) break;
      reinterpret_cast<float2*>(smem + L::kStatsOff)[t * kBlockM + row_in_tile] = make_float2(m_run, l_run);
      __syncwarp();
      if (lane == 0) mbar_arrive(st_full(t));
      ph ^= 4u;
    }
  } else {
    setmaxnreg_dec<kRegsOut>();
    // ------------------------------------------------------------ output warpgroup
    // Per unit and Q tile: wait for O_t to be final and for the softmax warpgroup's row
    // statistics, read O_t out of tensor memory (then it may take the next unit's P.V),
    // normalise, and store through the staging buffer with TMA stores.  Split units merge
    // O_1 and Q tile 1's statistics into Q tile 0's rows by log-sum-exp.
    const int row_in_tile = (warp % 4) * 32 + lane;
    const uint32_t lane_bits = static_cast<uint32_t>((warp % 4) * 32) << 16;
    const float2* const stats = reinterpret_cast<const float2*>(smem + L::kStatsOff);
    const bool leader = warp == kWarpOut && lane == 0;
    uint8_t* stage = smem + L::kOutOff + row_in_tile * 128;
    const uint32_t stage_base = s_base + L::kOutOff;
    int od[2] = {0, 0};  // o_done(t) phases consumed
    int sc[2] = {0, 0};  // st_full(t) phases consumed
    bool ok = true;
    for (int k = 0; k < n_rounds && ok; ++k) {
      const int i = unit_at(k, cta, G);
      Unit u;
      if (i >= a.total_units || !decode_unit<kSplit>(a, i, u)) continue;
      const bool split = u.step == 2;
#pragma unroll 1
      for (int t = 0; t < (split ? 1 : kQTiles) && ok; ++t) {
        const int row_first = u.row0(t);
        const int r = row_first + row_in_tile;
        const bool valid = r < u.Lq;
        const long long row = static_cast<long long>(u.q_base) + r;
        const int n_t = ((t == 0 ? u.thi[0] : u.thi[1]) - (t == 0 ? u.tlo[0] : u.tlo[1]) + u.step - 1) >> (u.step - 1);
        if (n_t <= 0) {  // no allowed key for any row of this Q tile
          if (valid) {
            for (int c = 0; c < a.d_out; c += 4) {
              if (a.out_fp32) {
                float* o = static_cast<float*>(a.out) + u.qb * a.so_b + row * a.so_m + u.h * a.so_h + c;
                *reinterpret_cast<float4*>(o) = make_float4(0.f, 0.f, 0.f, 0.f);
              } else {
                __nv_bfloat16* o =
                    static_cast<__nv_bfloat16*>(a.out) + u.qb * a.so_b + row * a.so_m + u.h * a.so_h + c;
                *reinterpret_cast<uint2*>(o) = make_uint2(0u, 0u);
              }
            }
            if (a.lse != nullptr) a.lse[u.qb * a.lse_sb + u.h * a.lse_sh + row * a.lse_sm] = -INFINITY;
          }
          continue;
        }
        // O_t final (split units: after the unit's last P.V of either tile), then the stats
        ok = __all_sync(0xffffffffu, wait_bar(o_done(t), od[t] & 1, wc));
        ok = ok && __all_sync(0xffffffffu, wait_bar(st_full(t), sc[t] & 1, wc));
        if (split) ok = ok && __all_sync(0xffffffffu, wait_bar(st_full(1), sc[1] & 1, wc));
        if (!ok) break;
        ++od[t];
        const float2 ml0 = stats[t * kBlockM + row_in_tile];
        const float2 ml1 = split ? stats[kBlockM + row_in_tile] : make_float2(-INFINITY, 0.f);
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(st_empty(t));
          if (split) mbar_arrive(st_empty(1));
        }
        ++sc[t];
        if (split) ++sc[1];
        const float m_out = fmaxf(ml0.x, ml1.x);
        float c0 = (ml0.x == -INFINITY) ? 0.f : ex2_approx(ml0.x - m_out);
        float c1 = (ml1.x == -INFINITY) ? 0.f : ex2_approx(ml1.x - m_out);
        const float l_out = ml0.y * c0 + ml1.y * c1;
        tc_fence_after();
        float inv_l = (l_out > 0.f) ? 1.f / l_out : 0.f;
        if constexpr (F8) inv_l *= a.dv[a.desc_per_tensor ? 0 : u.hk];
        c0 *= inv_l;
        c1 *= inv_l;
        const uint32_t to = tmem + 256u + static_cast<uint32_t>(t * 128) + lane_bits;
        const uint32_t to1 = tmem + 384u + lane_bits;  // O_1 (split units)
        // Output tiles go through the staging buffer and one TMA store per 128-byte column
        // band, except the tail tile of a packed sequence (a whole 128-row box would spill
        // into the next sequence), which is stored row by row.
        // (folded rows: the view's row extent is r, so a 128-row box is clipped there)
        const bool use_tma = a.tma_store && (a.fold || !(a.varlen && row_first + kBlockM > u.Lq));
        if (a.out_fp32) {
          // 4-byte outputs: bands of 32 columns
          const int n_bands = (a.d_out + 31) / 32;
#pragma unroll 1
          for (int band = 0; band < n_bands; ++band) {
            uint32_t o[32];
            tmem_ld_32x32b_x32(to + band * 32, o);
            if (split) {
              uint32_t o1[32];
              tmem_ld_32x32b_x32(to1 + band * 32, o1);
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = f2u(u2f(o[e]) * c0 + u2f(o1[e]) * c1);
            } else {
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = f2u(u2f(o[e]) * c0);
            }
            if (band == n_bands - 1) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) {
                mbar_arrive(o_free(t));  // O_t may now take the next unit's PV
                if (split) mbar_arrive(o_free(1));
              }
            }
            if (use_tma) {
              if (leader) bulk_wait_read0();  // the previous band's store has read the buffer
              named_bar_sync(1, kBlockM);
#pragma unroll
              for (int c = 0; c < 32; c += 4) {
                const int chunk = (c / 4) ^ (row_in_tile & 7);  // 128-byte swizzle
                *reinterpret_cast<float4*>(stage + chunk * 16) =
                    make_float4(u2f(o[c]), u2f(o[c + 1]), u2f(o[c + 2]), u2f(o[c + 3]));
              }
              fence_proxy_async_smem();
              named_bar_sync(1, kBlockM);
              if (leader) {
                tma_store_4d(&tm_o, stage_base, band * 32, u.q_base + row_first, u.h, u.qb);
                bulk_commit();
              }
            } else if (valid) {
              float* op = static_cast<float*>(a.out) + u.qb * a.so_b + row * a.so_m + u.h * a.so_h + band * 32;
#pragma unroll
              for (int c = 0; c < 32; c += 4)
                *reinterpret_cast<float4*>(op + c) =
                    make_float4(u2f(o[c]), u2f(o[c + 1]), u2f(o[c + 2]), u2f(o[c + 3]));
            }
          }
        } else {
          // bf16 outputs: bands of 64 columns, read 32 at a time
          const int n_bands = (a.d_out + 63) / 64;  // a partial last band is clipped by the map
#pragma unroll 1
          for (int band = 0; band < n_bands; ++band) {
            uint4 w[8];
#pragma unroll
            for (int hb = 0; hb < 64; hb += 32) {
              uint32_t o[32];
              tmem_ld_32x32b_x32(to + band * 64 + hb, o);
              if (split) {
                uint32_t o1[32];
                tmem_ld_32x32b_x32(to1 + band * 64 + hb, o1);
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] = f2u(u2f(o[e]) * c0 + u2f(o1[e]) * c1);
              } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] = f2u(u2f(o[e]) * c0);
              }
#pragma unroll
              for (int c = 0; c < 32; c += 8) {
                uint4& x = w[(hb + c) / 8];
                x.x = pack_bf16x2(u2f(o[c]), u2f(o[c + 1]));
                x.y = pack_bf16x2(u2f(o[c + 2]), u2f(o[c + 3]));
                x.z = pack_bf16x2(u2f(o[c + 4]), u2f(o[c + 5]));
                x.w = pack_bf16x2(u2f(o[c + 6]), u2f(o[c + 7]));
              }
            }
            if (band == n_bands - 1) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) {
                mbar_arrive(o_free(t));  // O_t may now take the next unit's PV
                if (split) mbar_arrive(o_free(1));
              }
            }
            if (use_tma) {
              if (leader) bulk_wait_read0();  // the previous band's store has read the buffer
              named_bar_sync(1, kBlockM);
#pragma unroll
              for (int ch = 0; ch < 8; ++ch)
                *reinterpret_cast<uint4*>(stage + ((ch ^ (row_in_tile & 7)) * 16)) = w[ch];
              fence_proxy_async_smem();
              named_bar_sync(1, kBlockM);
              if (leader) {
                tma_store_4d(&tm_o, stage_base, band * 64, u.q_base + row_first, u.h, u.qb);
                bulk_commit();
              }
            } else if (valid) {
              __nv_bfloat16* op =
                  static_cast<__nv_bfloat16*>(a.out) + u.qb * a.so_b + row * a.so_m + u.h * a.so_h + band * 64;
#pragma unroll
              for (int ch = 0; ch < 8; ++ch)
                if (band * 64 + ch * 8 < a.d_out) *reinterpret_cast<uint4*>(op + ch * 8) = w[ch];
            }
          }
        }
        if (valid && a.lse != nullptr)
          a.lse[u.qb * a.lse_sb + u.h * a.lse_sh + row * a.lse_sm] =
              (l_out > 0.f) ? (m_out + lg2_approx(l_out)) * kLn2 : -INFINITY;
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  if (warp == kWarpOut && lane == 0) bulk_wait0();  // output stores complete
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// kSplit: units whose rows fit one Q tile split their key tiles between both Q tiles
// (launches with at most 128 rows per unit; a separate instantiation, so the others keep
// their code).
template <int D, bool kLowerEdge, bool kSplit>
__global__ void __launch_bounds__(kThreads, 1)
    fmha_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                   const TcArgs a) {
  tc_body<D, kLowerEdge, false, kSplit>(tm_q, tm_k, tm_v, tm_o, a);
}

// E4M3 q, k, v (head dim 128), bf16 or fp32 output.
template <bool kLowerEdge, bool kSplit>
__global__ void __launch_bounds__(kThreads, 1)
    fmha_tc_fp8_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                       const TcArgs a) {
  tc_body<128, kLowerEdge, true, kSplit>(tm_q, tm_k, tm_v, tm_o, a);
}

// ------------------------------------------------------------------ host side
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// [batch, rows, heads, D] bf16 (or, with u8, E4M3 bytes) tensor with free strides
// (elements) -> 4-D tiled map with a 128-byte x 128-row box (one 128-byte swizzle atom per
// row).  Dimensions of extent 1 get a dummy stride (never stepped over).
bool encode_bhmd(EncodeTiledFn enc, CUtensorMap* map, const void* base, int D, long long rows,
                 long long heads, long long batch, long long s_m, long long s_h, long long s_b,
                 bool u8) {
  const long long elt = u8 ? 1 : 2;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(batch)};
  long long st_m = s_m * elt;
  long long st_h = heads > 1 ? s_h * elt : st_m * rows;
  long long st_b = batch > 1 ? s_b * elt : st_h * heads;
  if (rows == 1) st_m = 16;
  if (st_h <= 0 || st_h % 16) st_h = 16;
  if (st_b <= 0 || st_b % 16) st_b = 16;
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(st_m), static_cast<cuuint64_t>(st_h),
                           static_cast<cuuint64_t>(st_b)};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(128 / elt), kBlockM, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(map, u8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
             const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int num_sms() {
  constexpr int kMaxDevices = 64;
  static int cache[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
  if (cache[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n > 0 ? n : 148;
  }
  return cache[dev];
}

// Output [batch, rows, heads, D] (bf16 or fp32) for TMA stores of 128-byte column bands.
bool encode_out(EncodeTiledFn enc, CUtensorMap* map, void* base, bool fp32, int D, long long rows,
                long long heads, long long batch, long long s_m, long long s_h, long long s_b) {
  const long long elt = fp32 ? 4 : 2;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(batch)};
  long long st_m = s_m * elt;
  long long st_h = heads > 1 ? s_h * elt : st_m * rows;
  long long st_b = batch > 1 ? s_b * elt : st_h * heads;
  if (rows == 1) st_m = 16;
  if (st_h <= 0 || st_h % 16) st_h = 16;
  if (st_b <= 0 || st_b % 16) st_b = 16;
  if (st_m <= 0 || st_m % 16) return false;
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(st_m), static_cast<cuuint64_t>(st_h),
                           static_cast<cuuint64_t>(st_b)};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(128 / elt), kBlockM, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(map, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims,
             strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, bool F8>
cudaError_t launch_d(const AttnProblem& p, const DeviceCtl& ctl, cudaStream_t stream,
                     const char** why) {
  using Lt = Layout<D, F8>;
  EncodeTiledFn enc = get_encode_fn();
  if (enc == nullptr) {
    *why = "cuTensorMapEncodeTiled is not available from the driver";
    return cudaErrorNotSupported;
  }
  const long long hk = p.Hkv;
  const bool varlen = is_blockdiag(p.mask_kind);
  // Folded heads: q and out as [batch or packed row][r rows (head stride)][H / r heads].
  const int R = p.fold;
  const long long q_rows = R ? R : p.M, q_heads = R ? p.Hkv : p.H;
  const long long q_batch = R ? (varlen ? p.M : p.B) : p.B;
  const long long sq_m = R ? p.sq.h : p.sq.m, sq_h = R ? R * p.sq.h : p.sq.h;
  const long long sq_b = R ? (varlen ? p.sq.m : p.sq.b) : p.sq.b;
  const long long so_m = R ? p.so.h : p.so.m, so_h = R ? R * p.so.h : p.so.h;
  const long long so_b = R ? (varlen ? p.so.m : p.so.b) : p.so.b;
  CUtensorMap tq, tk, tv;
  const int Dd = p.K;  // the tensors' head dim (below D: columns past it read as zeros)
  if (!encode_bhmd(enc, &tq, p.q, Dd, q_rows, q_heads, q_batch, sq_m, sq_h, sq_b, F8) ||
      !encode_bhmd(enc, &tk, p.k, Dd, p.Mkv, hk, p.B, p.sk.m, p.sk.h, p.sk.b, F8) ||
      !encode_bhmd(enc, &tv, p.v, Dd, p.Mkv, hk, p.B, p.sv.m, p.sv.h, p.sv.b, F8)) {
    *why = "cuTensorMapEncodeTiled rejected a q/k/v layout";
    return cudaErrorInvalidValue;
  }
  // Output tiles: bands of 128 bytes (64 bf16 / 32 fp32 columns) x 128 rows.
  CUtensorMap to{};
  const bool tma_store =
      encode_out(enc, &to, p.out, p.out_fp32, Dd, q_rows, q_heads, q_batch, so_m, so_h, so_b);
  TcArgs a{};
  a.fold = R;
  a.d_out = Dd;
  if (R) {
    // lse [B, H, 1] (dense) or [1, H, total_q] (packed): query head = K/V head * r + row
    a.lse_sb = varlen ? 1 : p.H;
    a.lse_sh = varlen ? static_cast<long long>(R) * p.M : R;
    a.lse_sm = varlen ? p.M : 1;
  } else {
    a.lse_sb = static_cast<long long>(p.H) * p.M;
    a.lse_sh = p.M;
    a.lse_sm = 1;
  }
  a.M = p.M;
  a.Mkv = p.Mkv;
  a.H = R ? p.Hkv : p.H;
  a.kv_group = R ? 1 : p.kv_group;
  a.lo = p.band_lo <= -kBandOpen ? -kBandOpen : p.band_lo - p.kv_offset;
  a.hi = p.band_hi >= kBandOpen ? kBandOpen : p.band_hi - p.kv_offset;
  a.band_seq = p.band_seq_shift ? 1 : 0;
  a.lanes = p.lanes ? 1 : 0;
  a.lane_len = p.lane_len;
  a.lane_start = p.lane_start;
  a.block_table = p.block_table;
  a.page_size = p.page_size;
  a.max_pages = p.max_pages;
  a.varlen = is_blockdiag(p.mask_kind) ? 1 : 0;
  const int rows = R ? R : (a.varlen ? p.max_seqlen_q : p.M);
  a.units_m = (rows + kUnitRows - 1) / kUnitRows;
  a.scale_log2 = p.scale * kLog2e;
  a.cu_q = p.cu_q;
  a.cu_k = p.cu_k;
  a.out = p.out;
  a.out_fp32 = p.out_fp32 ? 1 : 0;
  a.so_b = so_b;
  a.so_m = so_m;
  a.so_h = so_h;
  a.lse = p.lse;
  a.tma_store = tma_store ? 1 : 0;
  a.dq = p.descale_q;
  a.dk = p.descale_k;
  a.dv = p.descale_v;
  a.desc_per_tensor = p.descale_per_tensor ? 1 : 0;
  a.err = ctl.err;
  a.timeout_ns = ctl.timeout_ns;
  a.Z = a.varlen ? p.n_seqs : p.B;
  const long long total = static_cast<long long>(a.units_m) * a.H * a.Z;  // the kernel's head count
  if (total == 0) return cudaSuccess;
  if (total > 0x7fffffffLL) {
    *why = "too many work units";
    return cudaErrorInvalidValue;
  }
  a.total_units = static_cast<int>(total);
  // Persistent: one CTA per SM (or fewer when there are fewer units).
  const dim3 grid(static_cast<unsigned>(std::min<long long>(total, num_sms())));
  // Split units when every unit's rows fit one Q tile (decode-shaped units over many key
  // tiles: both softmax warpgroups work on them); launches with longer rows keep the
  // instantiation without them.
  const bool split = rows <= kBlockM;
  const bool edge = a.lo > -kBandOpen;
  auto kernel = edge ? (split ? fmha_tc_kernel<D, true, true> : fmha_tc_kernel<D, true, false>)
                     : (split ? fmha_tc_kernel<D, false, true> : fmha_tc_kernel<D, false, false>);
  if constexpr (F8)
    kernel = edge ? (split ? fmha_tc_fp8_kernel<true, true> : fmha_tc_fp8_kernel<true, false>)
                  : (split ? fmha_tc_fp8_kernel<false, true> : fmha_tc_fp8_kernel<false, false>);
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Lt::kAlloc);
  if (e != cudaSuccess) {
    *why = "cudaFuncSetAttribute(max dynamic shared memory) failed";
    return e;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Lt::kAlloc;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  if (p.independent) {
    // the caller's inputs are not written by the previous launch: start while it finishes
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  e = cudaLaunchKernelEx(&cfg, kernel, tq, tk, tv, to, a);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) {
    static thread_local char msg[160];
    cudaFuncAttributes fa{};
    cudaFuncGetAttributes(&fa, kernel);
    snprintf(msg, sizeof(msg),
             "fmha_tc_kernel launch failed (regs/thread %d, max threads/block %d, dyn smem %d)",
             fa.numRegs, fa.maxThreadsPerBlock, Lt::kAlloc);
    *why = msg;
  }
  return e;
}

}  // namespace

cudaError_t launch_fmha_tc(const AttnProblem& p, const DeviceCtl& ctl, cudaStream_t stream,
                           const char** why) {
  if (p.fp8) {
    // head dims 64 and 96 run on the 128-wide E4M3 kernel, zero-padded by the tensor maps
    if (p.K == 128 || p.K == 96 || p.K == 64) return launch_d<128, true>(p, ctl, stream, why);
    *why = "E4M3 inputs on the tensor-core path need head dim 64, 96 or 128";
    return cudaErrorInvalidValue;
  }
  if (p.K == 128 || p.K == 96) return launch_d<128, false>(p, ctl, stream, why);  // 96: zero-padded
  if (p.K == 64) return launch_d<64, false>(p, ctl, stream, why);
  *why = "head dim must be 64 or 128";
  return cudaErrorInvalidValue;
}

}  // namespace mslk
