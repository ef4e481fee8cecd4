// merge.cu — exact LSE merge of split-KV chunk results (MSLK merge_attentions,
// "Attention - Core fMHA"; in-place variant in "Attention - Merge & storage utilities").
//
// Per output row (b, m, h):  M* = max_c lse_c,  LSE = M* + ln sum_c exp(lse_c - M*),
// out = sum_c exp(lse_c - LSE) out_c; every chunk -inf -> out = 0, LSE = -inf.
//
// HBM-bound: one warp per row, rows ordered (b, m, h) so neighbouring warps read
// neighbouring pieces of every chunk (sequential streams through each chunk); each lane
// reads 16-byte float4 pieces of every chunk row (a 512-byte row per warp instruction at
// Kv = 128), up to 8 chunks in flight per lane together with their lse, folded with a
// running maximum.

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

// Chunk c of a varargs merge: separately allocated [B, M, H, Kv] output and [B, H, M] lse
// arrays (kernel parameters, so no device-side table has to be written first).
struct ChunkTable {
  const float* out[kMergeMaxVarargs];
  const float* lse[kMergeMaxVarargs];
};

MSLK_DEV float4 ldg_f4(const float* p) {
  float4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
               : "l"(p));
  return r;
}

// Where chunk c's row and lse live: stacked (base + c * chunk stride: the group's G loads
// walk one pointer) or a pointer table.
struct StackedChunks {
  template <int G>
  MSLK_DEV void load(const MergeArgs& a, int c0, long long off, float4 (&x)[G]) const {
    const float* p = a.out_split + c0 * a.cs_out + off;
#pragma unroll
    for (int u = 0; u < G; ++u) {
      x[u] = (c0 + u < a.n) ? ldg_f4(p) : make_float4(0.f, 0.f, 0.f, 0.f);
      p += a.cs_out;
    }
  }
  MSLK_DEV const float* lse(const MergeArgs& a, int c, long long idx) const {
    return a.lse_split + c * a.cs_lse + idx;
  }
};
struct TableChunks {
  const ChunkTable* t;
  template <int G>
  MSLK_DEV void load(const MergeArgs& a, int c0, long long off, float4 (&x)[G]) const {
#pragma unroll
    for (int u = 0; u < G; ++u)
      x[u] = (c0 + u < a.n) ? ldg_f4(t->out[c0 + u] + off) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  MSLK_DEV const float* lse(const MergeArgs&, int c, long long idx) const { return t->lse[c] + idx; }
};

// G = chunks folded per memory round trip (2, 4 or 8): fewer for small n keeps the
// registers low and the number of rows in flight per SM high.
template <int G, class Chunks>
MSLK_DEV void merge_rows(const MergeArgs& a, const Chunks& ch) {
  const int lane = threadIdx.x % 32;
  const long long row = static_cast<long long>(blockIdx.x) * kWarpsPerBlock + threadIdx.x / 32;
  if (row >= a.rows) return;
  const int h = static_cast<int>(row % a.H);
  const long long bm_ = row / a.H;
  const int m = static_cast<int>(bm_ % a.M);
  const int b = static_cast<int>(bm_ / a.M);
  const long long lse_idx = (static_cast<long long>(b) * a.H + h) * a.M + m;  // [B, H, M]
  const long long src = b * a.ss_b + m * a.ss_m + h * a.ss_h;  // row offset inside a chunk

  for (int d0 = lane * 4; d0 < a.Kv; d0 += 128) {
    // Chunks are folded G at a time with a running maximum (all in base 2):
    //   mx = max lse seen so far, sw = sum_c 2^(l2e*lse_c - mx), acc = sum_c 2^(...) out_c.
    // A group's chunk rows and lse values are requested together (lane u fetches the lse
    // of chunk u and shares it), so each group costs one memory round trip.
    float mx = -INFINITY, sw = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c0 = 0; c0 < a.n; c0 += G) {
      float4 x[G];
      ch.template load<G>(a, c0, src + d0, x);
      const float mine = (lane < G && c0 + lane < a.n) ? __ldg(ch.lse(a, c0 + lane, lse_idx)) * kLog2e
                                                       : -INFINITY;
      float l2[G];
#pragma unroll
      for (int u = 0; u < G; ++u) l2[u] = __shfl_sync(0xffffffffu, mine, u);
      float bm = l2[0];
#pragma unroll
      for (int u = 1; u < G; ++u) bm = fmaxf(bm, l2[u]);
      const float nm = fmaxf(mx, bm);
      if (nm == -INFINITY) continue;  // every chunk so far is empty
      const float r = ex2_approx(mx - nm);  // mx = -inf -> 0
      sw *= r;
      acc.x *= r;
      acc.y *= r;
      acc.z *= r;
      acc.w *= r;
#pragma unroll
      for (int u = 0; u < G; ++u) {
        const float wgt = ex2_approx(l2[u] - nm);  // empty chunk -> 0
        sw += wgt;
        acc.x = fmaf(wgt, x[u].x, acc.x);
        acc.y = fmaf(wgt, x[u].y, acc.y);
        acc.z = fmaf(wgt, x[u].z, acc.z);
        acc.w = fmaf(wgt, x[u].w, acc.w);
      }
      mx = nm;
    }
    const bool empty = !(sw > 0.f);
    const float inv = empty ? 0.f : 1.f / sw;
    acc.x *= inv;
    acc.y *= inv;
    acc.z *= inv;
    acc.w *= inv;
    if (a.out_fp32) {
      float* o = static_cast<float*>(a.out) + b * a.so_b + m * a.so_m + h * a.so_h + d0;
      *reinterpret_cast<float4*>(o) = acc;
    } else {
      __nv_bfloat16* o = static_cast<__nv_bfloat16*>(a.out) + b * a.so_b + m * a.so_m + h * a.so_h + d0;
      *reinterpret_cast<uint2*>(o) = make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
    }
    if (d0 == 0 && a.lse != nullptr) a.lse[lse_idx] = empty ? -INFINITY : (mx + lg2_approx(sw)) * kLn2;
  }
}

template <int G>
__global__ void __launch_bounds__(kWarpsPerBlock * 32) merge_kernel(const MergeArgs a) {
  merge_rows<G>(a, StackedChunks{});
}

template <int G>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    merge_table_kernel(const MergeArgs a, const __grid_constant__ ChunkTable t) {
  merge_rows<G>(a, TableChunks{&t});
}

}  // namespace

cudaError_t launch_merge(const MergeProblem& p, const DeviceCtl& ctl, cudaStream_t stream) {
  (void)ctl;  // no waits in this kernel
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
  if (a.rows == 0) return cudaSuccess;
  const long long blocks = (a.rows + kWarpsPerBlock - 1) / kWarpsPerBlock;
  const dim3 grid(static_cast<unsigned>(blocks)), block(kWarpsPerBlock * 32);
  if (p.chunk_out != nullptr) {  // separately allocated chunks: pointer table as a parameter
    ChunkTable t{};
    for (int c = 0; c < p.n_chunks; ++c) {
      t.out[c] = p.chunk_out[c];
      t.lse[c] = p.chunk_lse[c];
    }
    if (a.n <= 2)
      merge_table_kernel<2><<<grid, block, 0, stream>>>(a, t);
    else if (a.n <= 4)
      merge_table_kernel<4><<<grid, block, 0, stream>>>(a, t);
    else
      merge_table_kernel<8><<<grid, block, 0, stream>>>(a, t);
    return cudaGetLastError();
  }
  if (a.n <= 2)
    merge_kernel<2><<<grid, block, 0, stream>>>(a);
  else if (a.n <= 4)
    merge_kernel<4><<<grid, block, 0, stream>>>(a);
  else
    merge_kernel<8><<<grid, block, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace mslk
