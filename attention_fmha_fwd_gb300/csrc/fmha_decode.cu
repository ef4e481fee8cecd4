// fmha_decode.cu — attention forward / partial for a handful of query rows (M <= 8)
// with dense masks, on the CUDA cores.
//
// With one query row per head each K/V element is used once, so the work is a stream
// of K and V from HBM (about 1 FLOP per byte); tensor-core tiles would be 128-fold
// padding.  Each CTA owns one (batch, head) and streams all its keys: 8 warps take
// contiguous key ranges; lane l holds head-dim elements [l*V, l*V+V) of every row
// (V = D/32), loads 32 (or 16) keys of K and V per step with 8-byte (D=128) / 4-byte
// (D=64) coalesced loads (a 256/128-byte row per warp instruction), forms the scores
// with a halving butterfly (each lane ends up with one key's full score), and runs the
// base-2 online softmax.  The 8 warp states (max, sum, accumulator) are then merged through shared
// memory by the same LSE rule as the split-KV merge.
//
// Semantics follow MSLK's memory_efficient_attention / _partial ("Attention - Core
// fMHA"): out = softmax(scale q.k^T + mask) v over the allowed keys; lse = ln sum exp;
// rows without an allowed key get out = 0, lse = -inf.

#include <cuda_bf16.h>

#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace mslk {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct DecArgs {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  long long sq_b, sq_m, sq_h;
  long long sk_b, sk_m, sk_h;
  long long sv_b, sv_m, sv_h;
  int M, Mkv, H;
  int hk_shared, causal;
  long long kv_offset;
  float scale_log2;
  void* out;
  int out_fp32;
  long long so_b, so_m, so_h;
  float* lse;
};

template <int V>
struct Vec;
template <>
struct Vec<4> {
  using T = uint2;
  MSLK_DEV static void to_float(T x, float* f) {
    f[0] = __uint_as_float(x.x << 16);
    f[1] = __uint_as_float(x.x & 0xFFFF0000u);
    f[2] = __uint_as_float(x.y << 16);
    f[3] = __uint_as_float(x.y & 0xFFFF0000u);
  }
};
template <>
struct Vec<2> {
  using T = uint32_t;
  MSLK_DEV static void to_float(T x, float* f) {
    f[0] = __uint_as_float(x << 16);
    f[1] = __uint_as_float(x & 0xFFFF0000u);
  }
};

template <typename T>
MSLK_DEV T ldg_stream(const T* p) {
  return __ldg(p);
}

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

// v[0..N-1] (N = 16 or 32) are one lane's partial sums for N keys.  Returns on lane l
// the full sum over all 32 lanes for key l / (32 / N).  Each halving step keeps the half
// of the values selected by one lane bit and adds the partner lane's other half.
template <int N>
MSLK_DEV float butterfly_reduce(float (&v)[N], int lane) {
  int n = N;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    if (n > 1) {
      n /= 2;
#pragma unroll
      for (int i = 0; i < N / 2; ++i) {
        if (i < n) {
          const bool up = lane & o;
          const float send = up ? v[i] : v[i + n];
          const float keep = up ? v[i + n] : v[i];
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
      }
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
    }
  }
  return v[0];
}

template <int D, int MQ>
__global__ void __launch_bounds__(kThreads, 1) fmha_decode_kernel(const DecArgs a) {
  constexpr int VE = D / 32;  // head-dim elements per lane
  // Keys per step: 32 (a key per lane) unless the registers of several query rows
  // need the smaller step (16 keys, each score held by a lane pair).
  constexpr int KB = (D == 128 && MQ > 1) ? 16 : 32;
  constexpr int kDup = 32 / KB;
  using VT = typename Vec<VE>::T;
  const int h = blockIdx.x;
  const int b = blockIdx.y;
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int hk = a.hk_shared ? 0 : h;

  // Query rows, pre-multiplied by scale * log2(e): scores come out in base 2.
  float qf[MQ][VE];
#pragma unroll
  for (int m = 0; m < MQ; ++m) {
    if (m < a.M) {
      const VT x = *reinterpret_cast<const VT*>(a.q + b * a.sq_b + m * a.sq_m + h * a.sq_h + lane * VE);
      Vec<VE>::to_float(x, qf[m]);
#pragma unroll
      for (int e = 0; e < VE; ++e) qf[m][e] *= a.scale_log2;
    } else {
#pragma unroll
      for (int e = 0; e < VE; ++e) qf[m][e] = 0.f;
    }
  }

  // Keys this warp owns: contiguous, a multiple of 32 long.
  int n_keys = a.Mkv;
  if (a.causal) {  // key j allowed iff kv_offset + j <= row; the last row sees the most
    const long long kmax = static_cast<long long>(a.M - 1) - a.kv_offset;
    n_keys = kmax < 0 ? 0 : static_cast<int>(min(static_cast<long long>(n_keys), kmax + 1));
  }
  const int blocks = (n_keys + KB - 1) / KB;
  const int per_warp = (blocks + kWarps - 1) / kWarps;
  const int kb0 = warp * per_warp * KB;
  const int kb1 = min(n_keys, (warp + 1) * per_warp * KB);

  float m_run[MQ], l_run[MQ], acc[MQ][VE];
#pragma unroll
  for (int m = 0; m < MQ; ++m) {
    m_run[m] = -INFINITY;
    l_run[m] = 0.f;
#pragma unroll
    for (int e = 0; e < VE; ++e) acc[m][e] = 0.f;
  }

  const __nv_bfloat16* kbase = a.k + b * a.sk_b + hk * a.sk_h + lane * VE;
  const __nv_bfloat16* vbase = a.v + b * a.sv_b + hk * a.sv_h + lane * VE;
  for (int k0 = kb0; k0 < kb1; k0 += KB) {
    VT kr[KB], vr[KB];
#pragma unroll
    for (int j = 0; j < KB; ++j) {
      const int key = k0 + j;
      if (key < kb1) {
        kr[j] = ldg_stream(reinterpret_cast<const VT*>(kbase + static_cast<long long>(key) * a.sk_m));
        vr[j] = ldg_stream(reinterpret_cast<const VT*>(vbase + static_cast<long long>(key) * a.sv_m));
      } else {
        kr[j] = VT{};
        vr[j] = VT{};
      }
    }
    const int my_key = k0 + lane / kDup;
#pragma unroll
    for (int m = 0; m < MQ; ++m) {
      if (m >= a.M) break;
      float part[KB];
#pragma unroll
      for (int j = 0; j < KB; ++j) {
        float kf[VE];
        Vec<VE>::to_float(kr[j], kf);
        float d = 0.f;
#pragma unroll
        for (int e = 0; e < VE; ++e) d = fmaf(qf[m][e], kf[e], d);
        part[j] = d;
      }
      float sc = butterfly_reduce<KB>(part, lane);
      const bool allowed = my_key < kb1 && (!a.causal || a.kv_offset + my_key <= m);
      sc = allowed ? sc : -INFINITY;
      const float m_new = fmaxf(m_run[m], warp_max(sc));
      const float msub = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = ex2_approx(m_run[m] - msub);  // m_run = -inf -> 0
      const float p = ex2_approx(sc - msub);
      // With lane pairs holding the same key, count each key once in the sum.
      l_run[m] = l_run[m] * alpha + warp_sum((lane % kDup == 0) ? p : 0.f);
      m_run[m] = m_new;
#pragma unroll
      for (int e = 0; e < VE; ++e) acc[m][e] *= alpha;
#pragma unroll
      for (int j = 0; j < KB; ++j) {
        const float pj = __shfl_sync(0xffffffffu, p, j * kDup);
        float vf[VE];
        Vec<VE>::to_float(vr[j], vf);
#pragma unroll
        for (int e = 0; e < VE; ++e) acc[m][e] = fmaf(pj, vf[e], acc[m][e]);
      }
    }
  }

  // Merge the warps' states: M* = max_w m_w; L = sum_w 2^(m_w - M*) l_w;
  // out = sum_w 2^(m_w - M*) acc_w / L.
  __shared__ float s_m[kWarps][MQ];
  __shared__ float s_l[kWarps][MQ];
  __shared__ float s_acc[kWarps][MQ][D];
#pragma unroll
  for (int m = 0; m < MQ; ++m) {
    if (lane == 0) {
      s_m[warp][m] = m_run[m];
      s_l[warp][m] = l_run[m];
    }
#pragma unroll
    for (int e = 0; e < VE; ++e) s_acc[warp][m][lane * VE + e] = acc[m][e];
  }
  __syncthreads();
  // Warp w finalises rows w, w + 8, ... (MQ <= 8: one row per warp).
  for (int m = warp; m < a.M && m < MQ; m += kWarps) {
    float mstar = -INFINITY;
    for (int w = 0; w < kWarps; ++w) mstar = fmaxf(mstar, s_m[w][m]);
    const float msub = (mstar == -INFINITY) ? 0.f : mstar;
    float L = 0.f;
    float o[VE];
#pragma unroll
    for (int e = 0; e < VE; ++e) o[e] = 0.f;
    for (int w = 0; w < kWarps; ++w) {
      const float c = ex2_approx(s_m[w][m] - msub);
      L = fmaf(c, s_l[w][m], L);
#pragma unroll
      for (int e = 0; e < VE; ++e) o[e] = fmaf(c, s_acc[w][m][lane * VE + e], o[e]);
    }
    const float inv = (L > 0.f) ? 1.f / L : 0.f;
    if (a.out_fp32) {
      float* op = static_cast<float*>(a.out) + b * a.so_b + m * a.so_m + h * a.so_h + lane * VE;
#pragma unroll
      for (int e = 0; e < VE; ++e) op[e] = o[e] * inv;
    } else {
      __nv_bfloat16* op =
          static_cast<__nv_bfloat16*>(a.out) + b * a.so_b + m * a.so_m + h * a.so_h + lane * VE;
#pragma unroll
      for (int e = 0; e < VE; e += 2)
        *reinterpret_cast<uint32_t*>(op + e) = pack_bf16x2(o[e] * inv, o[e + 1] * inv);
    }
    if (lane == 0 && a.lse != nullptr)
      a.lse[(static_cast<long long>(b) * a.H + h) * a.M + m] =
          (L > 0.f) ? (mstar + lg2_approx(L)) * kLn2 : -INFINITY;
  }
}

template <int D, int MQ>
cudaError_t launch_dm(const DecArgs& a, int B, int H, cudaStream_t stream) {
  fmha_decode_kernel<D, MQ><<<dim3(H, B), kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const DecArgs& a, int B, int H, cudaStream_t stream) {
  if (a.M <= 1) return launch_dm<D, 1>(a, B, H, stream);
  if (a.M <= 2) return launch_dm<D, 2>(a, B, H, stream);
  if (a.M <= 4) return launch_dm<D, 4>(a, B, H, stream);
  return launch_dm<D, 8>(a, B, H, stream);
}

}  // namespace

cudaError_t launch_fmha_decode(const AttnProblem& p, const DeviceCtl& ctl, cudaStream_t stream) {
  (void)ctl;  // no waits in this kernel
  DecArgs a{};
  a.q = static_cast<const __nv_bfloat16*>(p.q);
  a.k = static_cast<const __nv_bfloat16*>(p.k);
  a.v = static_cast<const __nv_bfloat16*>(p.v);
  a.sq_b = p.sq.b;
  a.sq_m = p.sq.m;
  a.sq_h = p.sq.h;
  a.sk_b = p.sk.b;
  a.sk_m = p.sk.m;
  a.sk_h = p.sk.h;
  a.sv_b = p.sv.b;
  a.sv_m = p.sv.m;
  a.sv_h = p.sv.h;
  a.M = p.M;
  a.Mkv = p.Mkv;
  a.H = p.H;
  a.hk_shared = p.kv_head_shared ? 1 : 0;
  a.causal = is_causal(p.mask_kind) ? 1 : 0;
  a.kv_offset = p.kv_offset;
  a.scale_log2 = p.scale * kLog2e;
  a.out = p.out;
  a.out_fp32 = p.out_fp32 ? 1 : 0;
  a.so_b = p.so.b;
  a.so_m = p.so.m;
  a.so_h = p.so.h;
  a.lse = p.lse;
  if (p.K == 128) return launch_d<128>(a, p.B, p.H, stream);
  return launch_d<64>(a, p.B, p.H, stream);
}

}  // namespace mslk
