// fmha_tc.cu — tensor-core attention forward / partial for sm_103a.
//
// Computes, for every query row i of a 256-row unit (two 128-row Q tiles) of one
// (batch or packed sequence, head):
//     out_i = sum_j softmax_j(scale * q_i . k_j) v_j      over the keys the mask allows
//     lse_i = ln sum_j exp(scale * q_i . k_j)
// as in MSLK's memory_efficient_attention ("Attention - Core fMHA"), streaming K/V in
// 128-key tiles so the score matrix never leaves the SM.
//
// Per CTA (320 threads, one CTA per SM):
//   warps 0-3   softmax for Q tile 0 (thread t owns row t = TMEM lane t)
//   warps 4-7   softmax for Q tile 1
//   warp  8     tcgen05.mma issue (one thread) + TMEM allocation
//   warp  9     TMA producer (one thread)
// Tensor memory (512 columns): S0 [0,128), S1 [128,256), O0 [256,256+D), O1 [384,384+D),
// fp32 accumulators, row r of a tile in lane r.  The bf16 probabilities P_t overwrite the
// first 64 columns of S_t (two values per column) and feed the PV MMA from tensor memory.
// Shared memory: Q0, Q1 and a 5-stage ring of K/V tiles, in the 128-byte-swizzled
// K-major layout TMA writes (V is read MN-major by the PV MMA).
// The MMA and TMA roles run as whole converged warps that issue through one elected lane:
// their operands stay warp-uniform, so they need few issue slots while the softmax
// warpgroups keep the SM's schedulers busy.
//
// MMA order (ping-pong: the tensor core works on one tile while the other tile's
// softmax runs):  S0_0 S1_0 | PV0_j S0_{j+1} PV1_j S1_{j+1} | ...
// S_t(j+1) is committed after PV_t(j), so when a softmax warpgroup sees S_t(j+1) its
// O_t is stable (it may rescale it) and PV_t(j) has finished reading P_t; MMAs issued by
// one thread execute in order, so S_t(j+1) overwrites P_t(j) only after PV_t(j) read it.
//
// Online softmax in base 2: m2 = running max of scale*log2(e)*s; p = 2^(scale*log2e*s - m2);
// l = running sum of p.  The running max used for p is only raised when the row max
// grows by more than 8 (a factor 256), which leaves the result exact (p, l and O all
// share the same reference) and makes O rescaling rare.  lse = (m2 + log2 l) * ln 2.
//
// Every mbarrier wait is bounded (globaltimer); a timeout sets the device error word,
// raises a CTA-wide abort flag, drains in-flight copies/MMAs and returns.

#include <cuda.h>
#include <cuda_bf16.h>

#include <cmath>
#include <cstdio>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace mslk {
namespace {

constexpr int kBlockM = 128;
constexpr int kBlockN = 128;
constexpr int kQTiles = 2;
constexpr int kUnitRows = kQTiles * kBlockM;
constexpr int kThreads = 320;
constexpr int kWarpMma = 8;
constexpr int kWarpLoad = 9;
constexpr int kTmemCols = 512;
constexpr int kSwizzleAtom = 16384;  // one 64-column K-block of a 128-row tile (bytes)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 of the largest un-rescaled p (256)

template <int D>
struct Layout {
  static constexpr int kKBlocks = D / 64;
  static constexpr int kTileBytes = kBlockM * D * 2;  // Q, K or V tile (128 rows)
  static constexpr int kStages = (D == 128) ? 5 : 8;
  static constexpr int kQOff = 0;
  static constexpr int kKVOff = kQOff + kQTiles * kTileBytes;
  static constexpr int kBarOff = kKVOff + kStages * kTileBytes;
  // q_full, kv_full[S], kv_empty[S], s_full[2], p_full[2], o_done[2], drain
  static constexpr int kNumBars = 1 + 2 * kStages + 6 + 1;
  static constexpr int kMiscOff = kBarOff + 8 * kNumBars;  // abort flag, tmem slot
  static constexpr int kBytes = kMiscOff + 16;
  static constexpr int kAlloc = kBytes + 1024;  // room to align the base to 1024
};

struct TcArgs {
  int M, Mkv, H;
  int hk_shared;
  int causal, varlen;
  int units_m;
  float scale_log2;
  long long kv_offset;
  const int* cu_q;
  const int* cu_k;
  void* out;
  int out_fp32;
  long long so_b, so_m, so_h;
  float* lse;
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

// S_t = Q_t K^T over the head dim, 16 columns per MMA.
template <int D>
MSLK_DEV void issue_qk(uint32_t d_tmem, uint64_t q_desc, uint64_t k_desc) {
  constexpr uint32_t idesc = idesc_bf16_f32(kBlockM, kBlockN, false);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk)
    mma_f16_ss_elect(d_tmem, q_desc + kmajor_step(kk), k_desc + kmajor_step(kk), idesc, kk > 0 ? 1u : 0u);
}

// O_t (+)= P_t V over the 128 keys of the tile, 16 keys per MMA.  P_t is read from tensor
// memory (16 bf16 keys = 8 columns per MMA); V is read MN-major: 8-key groups 1024 bytes
// apart (SBO), 64-column halves of the head dim 16 KiB apart (LBO); 16 keys are 2048 bytes.
template <int D>
MSLK_DEV void issue_pv(uint32_t o_tmem, uint32_t p_tmem, uint64_t v_desc, uint32_t accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32(kBlockM, D, true);
#pragma unroll
  for (int kk = 0; kk < kBlockN / 16; ++kk)
    mma_f16_ts_elect(o_tmem, p_tmem + kk * 8, v_desc + static_cast<uint32_t>(kk * 2048 / 16),
                     idesc, kk > 0 ? 1u : accumulate);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    fmha_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const TcArgs a) {
  using L = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  // ---------------------------------------------------------------- work unit
  const int unit = a.units_m - 1 - static_cast<int>(blockIdx.x);  // late (heavy) rows first
  const int h = blockIdx.y;
  const int z = blockIdx.z;
  int b, q_base, Lq, k_base, Lk;
  if (a.varlen) {
    b = 0;
    const int qs = min(max(a.cu_q[z], 0), a.M);
    const int qe = min(max(a.cu_q[z + 1], qs), a.M);
    const int ks = min(max(a.cu_k[z], 0), a.Mkv);
    const int ke = min(max(a.cu_k[z + 1], ks), a.Mkv);
    q_base = qs;
    Lq = qe - qs;
    k_base = ks;
    Lk = ke - ks;
  } else {
    b = z;
    q_base = 0;
    Lq = a.M;
    k_base = 0;
    Lk = a.Mkv;
  }
  const int r0 = unit * kUnitRows;
  if (r0 >= Lq) return;
  int n_tiles = (Lk + kBlockN - 1) / kBlockN;
  if (a.causal) {
    const long long last_row = min(r0 + kUnitRows - 1, Lq - 1);
    const long long kmax = last_row - a.kv_offset;  // last allowed key of the unit
    n_tiles = kmax < 0 ? 0 : static_cast<int>(min(static_cast<long long>(n_tiles), kmax / kBlockN + 1));
  }
  const int hk = a.hk_shared ? 0 : h;

  if (n_tiles == 0) {  // no allowed key for any row of the unit
    const int rows = min(kUnitRows, Lq - r0);
    for (int idx = threadIdx.x; idx < rows * (D / 4); idx += kThreads) {
      const long long row = q_base + r0 + idx / (D / 4);
      const int c = (idx % (D / 4)) * 4;
      if (a.out_fp32) {
        float* o = static_cast<float*>(a.out) + b * a.so_b + row * a.so_m + h * a.so_h + c;
        *reinterpret_cast<float4*>(o) = make_float4(0.f, 0.f, 0.f, 0.f);
      } else {
        __nv_bfloat16* o = static_cast<__nv_bfloat16*>(a.out) + b * a.so_b + row * a.so_m + h * a.so_h + c;
        *reinterpret_cast<uint2*>(o) = make_uint2(0u, 0u);
      }
    }
    if (a.lse != nullptr)
      for (int r = threadIdx.x; r < rows; r += kThreads)
        a.lse[(static_cast<long long>(b) * a.H + h) * a.M + q_base + r0 + r] = -INFINITY;
    return;
  }

  // ---------------------------------------------------------------- setup
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  const uint32_t bar0 = smem_u32(bars);
  const uint32_t bar_q = bar0;
  auto kv_full = [&](int s) { return bar0 + 8u * (1 + s); };
  auto kv_empty = [&](int s) { return bar0 + 8u * (1 + L::kStages + s); };
  auto s_full = [&](int t) { return bar0 + 8u * (1 + 2 * L::kStages + t); };
  auto p_full = [&](int t) { return bar0 + 8u * (3 + 2 * L::kStages + t); };
  auto o_done = [&](int t) { return bar0 + 8u * (5 + 2 * L::kStages + t); };
  const uint32_t bar_drain = bar0 + 8u * (7 + 2 * L::kStages);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff + 8);
  const WaitCtl wc{abort_flag, a.err, a.timeout_ns};

  const uint32_t s_base = smem_u32(smem);
  auto q_addr = [&](int t) { return s_base + L::kQOff + t * L::kTileBytes; };
  auto kv_addr = [&](int s) { return s_base + L::kKVOff + s * L::kTileBytes; };

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(kv_full(s), 1);
      mbar_init(kv_empty(s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(s_full(t), 1);
      mbar_init(p_full(t), kBlockM / 32);  // one arrival per softmax warp
      mbar_init(o_done(t), 1);
    }
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpLoad && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
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

  if (warp == kWarpLoad) {
    // ------------------------------------------------------------ TMA producer (whole warp)
    mbar_arrive_expect_tx_elect(bar_q, kQTiles * L::kTileBytes);
    for (int t = 0; t < kQTiles; ++t)
      for (int kb = 0; kb < L::kKBlocks; ++kb)
        tma_load_4d_elect(q_addr(t) + kb * kSwizzleAtom, &tm_q, bar_q, kb * 64,
                          q_base + r0 + t * kBlockM, h, b);
    int it = 0;
    bool ok = true;
    for (int j = 0; j < n_tiles && ok; ++j) {
      for (int which = 0; which < 2; ++which, ++it) {  // K_j then V_j
        const int s = it % L::kStages;
        if (!(ok = wait_bar_warp(kv_empty(s), ((it / L::kStages) & 1) ^ 1, wc))) break;
        mbar_arrive_expect_tx_elect(kv_full(s), L::kTileBytes);
        const CUtensorMap* tm = which ? &tm_v : &tm_k;
        for (int kb = 0; kb < L::kKBlocks; ++kb)
          tma_load_4d_elect(kv_addr(s) + kb * kSwizzleAtom, tm, kv_full(s), kb * 64,
                            k_base + j * kBlockN, hk, b);
      }
    }
    if (!ok) {  // let every copy this warp issued land before the CTA exits
      wait_bar_warp(bar_q, 0, wc, false);
      for (int k = max(0, it - L::kStages); k < it; ++k)
        wait_bar_warp(kv_full(k % L::kStages), (k / L::kStages) & 1, wc, false);
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer (whole warp)
    {
      const uint32_t tm_s[2] = {tmem + 0u, tmem + 128u};
      const uint32_t tm_o[2] = {tmem + 256u, tmem + 384u};
      const uint64_t q_desc[2] = {desc_kmajor(q_addr(0)), desc_kmajor(q_addr(1))};
      // Ring stages are kTileBytes apart: stage s adds s * kTileBytes / 16 to the address field.
      const uint64_t kdesc0 = desc_kmajor(kv_addr(0));
      const uint64_t vdesc0 = desc_mnmajor(kv_addr(0));
      auto kv_kdesc = [&](int st) { return kdesc0 + static_cast<uint32_t>(st * (L::kTileBytes >> 4)); };
      auto kv_vdesc = [&](int st) { return vdesc0 + static_cast<uint32_t>(st * (L::kTileBytes >> 4)); };
      bool ok = wait_bar_warp(bar_q, 0, wc);
      int it = 0;
      if (ok) ok = wait_bar_warp(kv_full(0), 0, wc);
      if (ok) {
        tc_fence_after();
        issue_qk<D>(tm_s[0], q_desc[0], kv_kdesc(0));
        mma_commit_elect(s_full(0));
        issue_qk<D>(tm_s[1], q_desc[1], kv_kdesc(0));
        mma_commit_elect(s_full(1));
        mma_commit_elect(kv_empty(0));
        it = 1;
      }
      for (int j = 0; j < n_tiles && ok; ++j) {
        const int sv = it % L::kStages;
        if (!(ok = wait_bar_warp(kv_full(sv), (it / L::kStages) & 1, wc))) break;
        ++it;
        const bool more = j + 1 < n_tiles;
        int sk = 0;
        // Q tile 0: PV0_j, then S0_{j+1}
        if (!(ok = wait_bar_warp(p_full(0), j & 1, wc))) break;
        tc_fence_after();
        issue_pv<D>(tm_o[0], tm_s[0], kv_vdesc(sv), j > 0 ? 1u : 0u);
        if (more) {
          sk = it % L::kStages;
          if (!(ok = wait_bar_warp(kv_full(sk), (it / L::kStages) & 1, wc))) break;
          ++it;
          tc_fence_after();
          issue_qk<D>(tm_s[0], q_desc[0], kv_kdesc(sk));
          mma_commit_elect(s_full(0));
        } else {
          mma_commit_elect(o_done(0));
        }
        // Q tile 1: PV1_j, then S1_{j+1}
        if (!(ok = wait_bar_warp(p_full(1), j & 1, wc))) break;
        tc_fence_after();
        issue_pv<D>(tm_o[1], tm_s[1], kv_vdesc(sv), j > 0 ? 1u : 0u);
        mma_commit_elect(kv_empty(sv));
        if (more) {
          issue_qk<D>(tm_s[1], q_desc[1], kv_kdesc(sk));
          mma_commit_elect(s_full(1));
          mma_commit_elect(kv_empty(sk));
        } else {
          mma_commit_elect(o_done(1));
        }
      }
      if (!ok) {  // wait for every MMA this thread issued
        mma_commit_elect(bar_drain);
        wait_bar_warp(bar_drain, 0, wc, false);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax warpgroups
    const int t = warp / 4;                   // Q tile
    const int row_in_tile = (warp % 4) * 32 + lane;
    const uint32_t lane_bits = static_cast<uint32_t>((warp % 4) * 32) << 16;
    const uint32_t ts = tmem + static_cast<uint32_t>(t * 128) + lane_bits;
    const uint32_t to = tmem + 256u + static_cast<uint32_t>(t * 128) + lane_bits;
    const int row_first = r0 + t * kBlockM;   // first row of this Q tile (sequence coords)
    const int r = row_first + row_in_tile;
    const float sl2 = a.scale_log2;
    float m_run = -INFINITY;
    float l_run = 0.f;
    bool ok = true;

    for (int j = 0; j < n_tiles; ++j) {
      // tcgen05.ld is warp-collective: take every wait decision warp-uniformly.
      ok = __all_sync(0xffffffffu, wait_bar(s_full(t), j & 1, wc));
      if (!ok) break;
      __syncwarp();
      tc_fence_after();
      uint32_t sr[kBlockN];
      tmem_ld_32x32b_x128(ts, sr);
      float s[kBlockN];
#pragma unroll
      for (int c = 0; c < kBlockN; ++c) s[c] = u2f(sr[c]);

      const int key0 = j * kBlockN;
      const bool need_mask =
          (key0 + kBlockN > Lk) || (a.causal && (a.kv_offset + key0 + kBlockN - 1 > row_first));
      if (need_mask) {
        // Column c of this tile is allowed iff c <= lim (key < Lk, and for causal masks
        // kv_offset + key <= r).
        long long lim = static_cast<long long>(Lk) - 1 - key0;
        if (a.causal) lim = min(lim, static_cast<long long>(r) - a.kv_offset - key0);
        const int lim_c = static_cast<int>(max(-1LL, min(lim, static_cast<long long>(kBlockN))));
#pragma unroll
        for (int c = 0; c < kBlockN; ++c) s[c] = (c <= lim_c) ? s[c] : -INFINITY;
      }
      // Row max as 8 independent chains (a single chain would serialise 127 maxes).
      float mx8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx8[i] = s[i];
#pragma unroll
      for (int c = 8; c < kBlockN; c += 8)
#pragma unroll
        for (int i = 0; i < 8; ++i) mx8[i] = fmaxf(mx8[i], s[c + i]);
      const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                             fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
      const float m_new = fmaxf(m_run, mx * sl2);
      const bool rescale = m_new > m_run + kRescaleThreshold;
      float alpha = 1.f;
      if (rescale) {
        alpha = ex2_approx(m_run - m_new);
        m_run = m_new;
      }
      l_run *= alpha;
      const float msub = (m_run == -INFINITY) ? 0.f : m_run;
      float rs8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};  // 8 independent partial sums
#pragma unroll
      for (int half = 0; half < 2; ++half) {  // P as packed bf16 pairs over S's first 64 columns
        uint32_t pk[32];
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          float p[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            p[e] = ex2_approx(fmaf(s[half * 64 + ch * 8 + e], sl2, -msub));
            rs8[e] += p[e];
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) pk[ch * 4 + e] = pack_bf16x2(p[2 * e], p[2 * e + 1]);
        }
        tmem_st_32x32b_x32(ts + half * 32, pk);
      }
      l_run += ((rs8[0] + rs8[1]) + (rs8[2] + rs8[3])) + ((rs8[4] + rs8[5]) + (rs8[6] + rs8[7]));
      if (j > 0 && __any_sync(0xffffffffu, rescale)) {
        // O_t is stable here: PV_t(j-1) completed before S_t(j) was signalled, and
        // PV_t(j) is not issued before this warpgroup arrives on p_full.
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t o[32];
          tmem_ld_32x32b_x32(to + c0, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = f2u(u2f(o[i]) * alpha);
          tmem_st_32x32b_x32(to + c0, o);
        }
        tmem_st_wait();
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full(t));  // one arrival per warp
    }

    if (ok) ok = __all_sync(0xffffffffu, wait_bar(o_done(t), 0, wc));
    if (ok) {
      __syncwarp();
      tc_fence_after();
      const bool valid = r < Lq;
      const float inv_l = (l_run > 0.f) ? 1.f / l_run : 0.f;
      const long long row = static_cast<long long>(q_base) + r;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t o[32];
        tmem_ld_32x32b_x32(to + c0, o);
        float x[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] = u2f(o[i]) * inv_l;
        if (valid) {
          if (a.out_fp32) {
            float* op = static_cast<float*>(a.out) + b * a.so_b + row * a.so_m + h * a.so_h + c0;
#pragma unroll
            for (int c = 0; c < 32; c += 4)
              *reinterpret_cast<float4*>(op + c) = make_float4(x[c], x[c + 1], x[c + 2], x[c + 3]);
          } else {
            __nv_bfloat16* op =
                static_cast<__nv_bfloat16*>(a.out) + b * a.so_b + row * a.so_m + h * a.so_h + c0;
#pragma unroll
            for (int c = 0; c < 32; c += 8) {
              uint4 w;
              w.x = pack_bf16x2(x[c], x[c + 1]);
              w.y = pack_bf16x2(x[c + 2], x[c + 3]);
              w.z = pack_bf16x2(x[c + 4], x[c + 5]);
              w.w = pack_bf16x2(x[c + 6], x[c + 7]);
              *reinterpret_cast<uint4*>(op + c) = w;
            }
          }
        }
      }
      if (valid && a.lse != nullptr)
        a.lse[(static_cast<long long>(b) * a.H + h) * a.M + row] =
            (l_run > 0.f) ? (m_run + lg2_approx(l_run)) * kLn2 : -INFINITY;
    }
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
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

// [batch, rows, heads, D] bf16 tensor with free strides (elements) -> 4-D tiled map with a
// 64 x 128 box (one 128-byte swizzle atom per row).  Dimensions of extent 1 get a dummy
// stride (never stepped over).
bool encode_bhmd(EncodeTiledFn enc, CUtensorMap* map, const void* base, int D, long long rows,
                 long long heads, long long batch, long long s_m, long long s_h, long long s_b) {
  const long long elt = 2;
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
  cuuint32_t box[4] = {64, kBlockM, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_d(const AttnProblem& p, const DeviceCtl& ctl, cudaStream_t stream,
                     const char** why) {
  using Lt = Layout<D>;
  EncodeTiledFn enc = get_encode_fn();
  if (enc == nullptr) {
    *why = "cuTensorMapEncodeTiled is not available from the driver";
    return cudaErrorNotSupported;
  }
  const long long hk = p.kv_head_shared ? 1 : p.H;
  CUtensorMap tq, tk, tv;
  if (!encode_bhmd(enc, &tq, p.q, D, p.M, p.H, p.B, p.sq.m, p.sq.h, p.sq.b) ||
      !encode_bhmd(enc, &tk, p.k, D, p.Mkv, hk, p.B, p.sk.m, p.sk.h, p.sk.b) ||
      !encode_bhmd(enc, &tv, p.v, D, p.Mkv, hk, p.B, p.sv.m, p.sv.h, p.sv.b)) {
    *why = "cuTensorMapEncodeTiled rejected a q/k/v layout";
    return cudaErrorInvalidValue;
  }
  TcArgs a{};
  a.M = p.M;
  a.Mkv = p.Mkv;
  a.H = p.H;
  a.hk_shared = p.kv_head_shared ? 1 : 0;
  a.causal = is_causal(p.mask_kind) ? 1 : 0;
  a.varlen = is_blockdiag(p.mask_kind) ? 1 : 0;
  const int rows = a.varlen ? p.max_seqlen_q : p.M;
  a.units_m = (rows + kUnitRows - 1) / kUnitRows;
  a.scale_log2 = p.scale * kLog2e;
  a.kv_offset = p.kv_offset;
  a.cu_q = p.cu_q;
  a.cu_k = p.cu_k;
  a.out = p.out;
  a.out_fp32 = p.out_fp32 ? 1 : 0;
  a.so_b = p.so.b;
  a.so_m = p.so.m;
  a.so_h = p.so.h;
  a.lse = p.lse;
  a.err = ctl.err;
  a.timeout_ns = ctl.timeout_ns;
  const dim3 grid(a.units_m, p.H, a.varlen ? p.n_seqs : p.B);
  if (grid.x == 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(fmha_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Lt::kAlloc);
  if (e != cudaSuccess) {
    *why = "cudaFuncSetAttribute(max dynamic shared memory) failed";
    return e;
  }
  fmha_tc_kernel<D><<<grid, kThreads, Lt::kAlloc, stream>>>(tq, tk, tv, a);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    static thread_local char msg[160];
    cudaFuncAttributes fa{};
    cudaFuncGetAttributes(&fa, fmha_tc_kernel<D>);
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
  if (p.K == 128) return launch_d<128>(p, ctl, stream, why);
  if (p.K == 64) return launch_d<64>(p, ctl, stream, why);
  *why = "head dim must be 64 or 128";
  return cudaErrorInvalidValue;
}

}  // namespace mslk
