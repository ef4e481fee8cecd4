// merge.cu — exact LSE merge of split-KV chunk results (MSLK merge_attentions,
// "Attention - Core fMHA"; in-place variant in "Attention - Merge & storage utilities").
//
// Per output row (b, m, h):  M* = max_c lse_c,  LSE = M* + ln sum_c exp(lse_c - M*),
// out = sum_c exp(lse_c - LSE) out_c; every chunk -inf -> out = 0, LSE = -inf.
//
// HBM-bound: one warp per row, rows ordered (b, h, m) so a block's lse reads are
// contiguous; each lane reads 16-byte float4 pieces of every chunk row (a 512-byte row
// per warp instruction at Kv = 128) with up to 8 chunk loads in flight per lane.

#include <cuda_bf16.h>

#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace mslk {
namespace {

constexpr int kWarpsPerBlock = 8;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct MergeArgs {
  const float* out_split;
  const float* lse_split;
  int n;
  long long cs_out, cs_lse;
  int B, M, H, Kv;
  long long ss_b, ss_m, ss_h;
  void* out;
  int out_fp32;
  long long so_b, so_m, so_h;
  float* lse;
  long long rows;
};

MSLK_DEV float4 ldg_f4(const float* p) {
  float4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
               : "l"(p));
  return r;
}

__global__ void __launch_bounds__(kWarpsPerBlock * 32) merge_kernel(const MergeArgs a) {
  const int lane = threadIdx.x % 32;
  const long long row = static_cast<long long>(blockIdx.x) * kWarpsPerBlock + threadIdx.x / 32;
  if (row >= a.rows) return;
  const int m = static_cast<int>(row % a.M);
  const long long bh = row / a.M;
  const int h = static_cast<int>(bh % a.H);
  const int b = static_cast<int>(bh / a.H);
  const long long lse_idx = bh * a.M + m;  // [B, H, M]

  // Chunk weights, in base 2: w_c = 2^(log2e*lse_c - log2e*LSE).
  float mstar = -INFINITY;
  for (int c = lane; c < a.n; c += 32) mstar = fmaxf(mstar, a.lse_split[c * a.cs_lse + lse_idx]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mstar = fmaxf(mstar, __shfl_xor_sync(0xffffffffu, mstar, o));
  const float msub2 = (mstar == -INFINITY) ? 0.f : mstar * kLog2e;
  float sumw = 0.f;
  for (int c = lane; c < a.n; c += 32)
    sumw += ex2_approx(fmaf(a.lse_split[c * a.cs_lse + lse_idx], kLog2e, -msub2));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sumw += __shfl_xor_sync(0xffffffffu, sumw, o);
  const bool empty = !(sumw > 0.f);
  const float lse2 = msub2 + lg2_approx(sumw);  // log2e * LSE
  const float inv_sum = empty ? 0.f : 1.f / sumw;

  const float* src = a.out_split + b * a.ss_b + m * a.ss_m + h * a.ss_h;
  for (int d0 = lane * 4; d0 < a.Kv; d0 += 128) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c0 = 0; c0 < a.n; c0 += 8) {
      float4 x[8];
      float w[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int c = c0 + u;
        if (c < a.n) {
          x[u] = ldg_f4(src + c * a.cs_out + d0);
          // exp(lse_c - LSE) = 2^(log2e lse_c - msub2) / sumw
          w[u] = ex2_approx(fmaf(a.lse_split[c * a.cs_lse + lse_idx], kLog2e, -msub2)) * inv_sum;
        } else {
          x[u] = make_float4(0.f, 0.f, 0.f, 0.f);
          w[u] = 0.f;
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        acc.x = fmaf(w[u], x[u].x, acc.x);
        acc.y = fmaf(w[u], x[u].y, acc.y);
        acc.z = fmaf(w[u], x[u].z, acc.z);
        acc.w = fmaf(w[u], x[u].w, acc.w);
      }
    }
    if (a.out_fp32) {
      float* o = static_cast<float*>(a.out) + b * a.so_b + m * a.so_m + h * a.so_h + d0;
      *reinterpret_cast<float4*>(o) = acc;
    } else {
      __nv_bfloat16* o = static_cast<__nv_bfloat16*>(a.out) + b * a.so_b + m * a.so_m + h * a.so_h + d0;
      *reinterpret_cast<uint2*>(o) = make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
    }
  }
  if (lane == 0 && a.lse != nullptr) a.lse[lse_idx] = empty ? -INFINITY : lse2 * kLn2;
}

}  // namespace

cudaError_t launch_merge(const MergeProblem& p, cudaStream_t stream) {
  MergeArgs a{};
  a.out_split = p.out_split;
  a.lse_split = p.lse_split;
  a.n = p.n_chunks;
  a.cs_out = p.cs_out;
  a.cs_lse = p.cs_lse;
  a.B = p.B;
  a.M = p.M;
  a.H = p.H;
  a.Kv = p.Kv;
  a.ss_b = p.ss.b;
  a.ss_m = p.ss.m;
  a.ss_h = p.ss.h;
  a.out = p.out;
  a.out_fp32 = p.out_fp32 ? 1 : 0;
  a.so_b = p.so.b;
  a.so_m = p.so.m;
  a.so_h = p.so.h;
  a.lse = p.lse;
  a.rows = static_cast<long long>(p.B) * p.H * p.M;
  const long long blocks = (a.rows + kWarpsPerBlock - 1) / kWarpsPerBlock;
  if (blocks == 0) return cudaSuccess;
  merge_kernel<<<static_cast<unsigned>(blocks), kWarpsPerBlock * 32, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace mslk
