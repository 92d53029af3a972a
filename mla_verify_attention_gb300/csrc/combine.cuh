// Merge of the per-slice partial states of the key-range split.
//
// Page "The Decisive Microbench: When Theory Meets Silicon", section "The
// KV-Split Solution": a second kernel merges the slices' unnormalised
// accumulators with the online-softmax combine.  For one query row with
// slices s (running max m_s in log2-scaled units, running sum l_s, accumulator
// O_s): M = max m_s, w_s = 2^(m_s - M), L = sum w_s l_s, out = sum w_s O_s / L,
// lse = (M + log2 L) ln 2.  Slices with l_s = 0 are skipped (their O_s is 0).
//
// Memory-bound: one 128-thread block per query row, 16-byte loads and stores,
// fully coalesced over the 512-wide rows; up to kBatch slices' loads in flight.
// The batch follows the slice count (4, 8 or 16): a smaller batch takes fewer
// registers, so more blocks (rows) are resident per SM, and a call with many
// rows and few slices (many short streams) is not a train of short waves.
#pragma once
#include <cstdint>
#include <math_constants.h>

#include "ptx.cuh"

namespace mla {

struct CombineParams {
  const float* part_o;     // [nsplit][N][512]
  const float2* part_ml;   // [nsplit][N]
  const int32_t* seq_lens;
  float* out;              // [N][512]
  float* lse;              // [N]
  int N;                   // B * q * H rows
  int rows_per_stream;     // q * H
  int q, Smax, nsplit, chunk_keys;
  const int* plan;         // device-side {chunk_tiles, nsplit}, or null (the fields above)
};

// Launched as a programmatic dependent of the split kernel: the block may start
// while that grid still runs and waits here until its results are visible.
__device__ __forceinline__ void wait_for_split_grid() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// kBatch 16: four blocks per SM (<= 128 registers), all rows of a 64-head,
// 9-draft call in one wave; kBatch 8 and 4: 6 and 12 blocks per SM.
// kGroups > 1 (calls with few rows and many slices, e.g. 8 heads): each of
// kGroups groups of 128 threads merges every kGroups-th slice of the row, and
// the groups' states are merged through shared memory at the end.
template <int kBatch, int kGroups>
__global__ void __launch_bounds__(128 * kGroups, kGroups > 1 ? 1 : (kBatch == 16 ? 4 : (kBatch == 8 ? 6 : 12)))
    combine_kernel(const CombineParams p) {
  wait_for_split_grid();
  const int row = blockIdx.x;
  const int tid = threadIdx.x & 127;
  const int grp = threadIdx.x >> 7;
  const int b = row / p.rows_per_stream;
  const int S = p.seq_lens[b];
  if (S < p.q || S > p.Smax) return;   // reported by the split kernel
  const int chunk_keys = p.plan != nullptr ? p.plan[0] * 64 : p.chunk_keys;
  const int ns = min(p.plan != nullptr ? p.plan[1] : p.nsplit, (S + chunk_keys - 1) / chunk_keys);
  const float2* ml = p.part_ml + row;
  const float4* src = reinterpret_cast<const float4*>(p.part_o + static_cast<size_t>(row) * 512) + tid;
  const size_t step4 = static_cast<size_t>(p.N) * 128;   // float4s between slices
  // Every slice s < ns wrote its partial (an all-zero accumulator where no key
  // was visible).  A batch's (m, l) pairs and accumulators are all requested
  // before any is used; batches are merged online (running max M).
  float M = -CUDART_INF_F, L = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = grp; s0 < ns; s0 += kBatch * kGroups) {
    float2 v[kBatch];
    float4 o[kBatch];
#pragma unroll
    for (int e = 0; e < kBatch; ++e) {
      const int s = s0 + e * kGroups;
      if (s < ns) {
        v[e] = ml[static_cast<size_t>(s) * p.N];
        o[e] = src[s * step4];
      } else {
        v[e] = make_float2(-CUDART_INF_F, 0.f);
        o[e] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    float Mb = M;
#pragma unroll
    for (int e = 0; e < kBatch; ++e) Mb = v[e].y > 0.f ? fmaxf(Mb, v[e].x) : Mb;
    if (Mb == -CUDART_INF_F) continue;            // nothing visible so far
    const float c = ex2(M - Mb);                  // 0 while M = -inf (L, acc are 0 then)
    L *= c;
    acc.x *= c; acc.y *= c; acc.z *= c; acc.w *= c;
#pragma unroll
    for (int e = 0; e < kBatch; ++e) {
      const float w = v[e].y > 0.f ? ex2(v[e].x - Mb) : 0.f;
      L += w * v[e].y;
      acc.x += w * o[e].x;
      acc.y += w * o[e].y;
      acc.z += w * o[e].z;
      acc.w += w * o[e].w;
    }
    M = Mb;
  }
  if (kGroups > 1) {
    __shared__ float gm[kGroups], gl[kGroups];
    __shared__ float4 gacc[kGroups][128];
    if (tid == 0) {
      gm[grp] = M;
      gl[grp] = L;
    }
    gacc[grp][tid] = acc;
    __syncthreads();
    if (grp != 0) return;
    M = -CUDART_INF_F;
#pragma unroll
    for (int g = 0; g < kGroups; ++g) M = gl[g] > 0.f ? fmaxf(M, gm[g]) : M;
    L = 0.f;
    acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -CUDART_INF_F) {
#pragma unroll
      for (int g = 0; g < kGroups; ++g) {
        const float w = gl[g] > 0.f ? ex2(gm[g] - M) : 0.f;
        const float4 a = gacc[g][tid];
        L += w * gl[g];
        acc.x += w * a.x;
        acc.y += w * a.y;
        acc.z += w * a.z;
        acc.w += w * a.w;
      }
    }
  }
  float4* dst = reinterpret_cast<float4*>(p.out + static_cast<size_t>(row) * 512) + tid;
  if (M == -CUDART_INF_F) {
    *dst = make_float4(0.f, 0.f, 0.f, 0.f);
    if (tid == 0) p.lse[row] = -CUDART_INF_F;
    return;
  }
  const float inv = 1.f / L;
  *dst = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  if (tid == 0) p.lse[row] = (M + log2f(L)) * 0.6931471805599453f;
}

// Few rows and many slices (e.g. 8 or 16 heads over a long stream): each row is
// merged by kCols blocks of 512 / kCols columns, and in each block kGroups
// groups of 32 threads (4 columns a thread) merge every kGroups-th slice, so
// that up to kBatch * kGroups slices' loads are in flight per block at once;
// the groups' states are merged through shared memory.  Grid (rows, kCols).
template <int kBatch, int kGroups, int kCols>
__global__ void __launch_bounds__(32 * kGroups, 2) combine_cols_kernel(const CombineParams p) {
  static_assert(kCols * 32 * 4 == 512, "one float4 per thread of a 32-thread group");
  wait_for_split_grid();
  const int row = blockIdx.x;
  const int lane = threadIdx.x & 31;
  const int grp = threadIdx.x >> 5;
  const int b = row / p.rows_per_stream;
  const int S = p.seq_lens[b];
  if (S < p.q || S > p.Smax) return;   // reported by the split kernel
  const int chunk_keys = p.plan != nullptr ? p.plan[0] * 64 : p.chunk_keys;
  const int ns = min(p.plan != nullptr ? p.plan[1] : p.nsplit, (S + chunk_keys - 1) / chunk_keys);
  const float2* ml = p.part_ml + row;
  const int col4 = blockIdx.y * 32 + lane;                 // float4 column of this thread
  const float4* src = reinterpret_cast<const float4*>(p.part_o + static_cast<size_t>(row) * 512) + col4;
  const size_t step4 = static_cast<size_t>(p.N) * 128;   // float4s between slices
  float M = -CUDART_INF_F, L = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = grp; s0 < ns; s0 += kBatch * kGroups) {
    float2 v[kBatch];
    float4 o[kBatch];
#pragma unroll
    for (int e = 0; e < kBatch; ++e) {
      const int s = s0 + e * kGroups;
      if (s < ns) {
        v[e] = ml[static_cast<size_t>(s) * p.N];
        o[e] = src[s * step4];
      } else {
        v[e] = make_float2(-CUDART_INF_F, 0.f);
        o[e] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    float Mb = M;
#pragma unroll
    for (int e = 0; e < kBatch; ++e) Mb = v[e].y > 0.f ? fmaxf(Mb, v[e].x) : Mb;
    if (Mb == -CUDART_INF_F) continue;            // nothing visible so far
    const float c = ex2(M - Mb);                  // 0 while M = -inf (L, acc are 0 then)
    L *= c;
    acc.x *= c; acc.y *= c; acc.z *= c; acc.w *= c;
#pragma unroll
    for (int e = 0; e < kBatch; ++e) {
      const float w = v[e].y > 0.f ? ex2(v[e].x - Mb) : 0.f;
      L += w * v[e].y;
      acc.x += w * o[e].x;
      acc.y += w * o[e].y;
      acc.z += w * o[e].z;
      acc.w += w * o[e].w;
    }
    M = Mb;
  }
  __shared__ float gm[kGroups], gl[kGroups];
  __shared__ float4 gacc[kGroups][32];
  if (lane == 0) {
    gm[grp] = M;
    gl[grp] = L;
  }
  gacc[grp][lane] = acc;
  __syncthreads();
  if (grp != 0) return;
  M = -CUDART_INF_F;
#pragma unroll
  for (int g = 0; g < kGroups; ++g) M = gl[g] > 0.f ? fmaxf(M, gm[g]) : M;
  L = 0.f;
  acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (M != -CUDART_INF_F) {
#pragma unroll
    for (int g = 0; g < kGroups; ++g) {
      const float w = gl[g] > 0.f ? ex2(gm[g] - M) : 0.f;
      const float4 a = gacc[g][lane];
      L += w * gl[g];
      acc.x += w * a.x;
      acc.y += w * a.y;
      acc.z += w * a.z;
      acc.w += w * a.w;
    }
  }
  float4* dst = reinterpret_cast<float4*>(p.out + static_cast<size_t>(row) * 512) + col4;
  const bool lse_writer = blockIdx.y == 0 && lane == 0;
  if (M == -CUDART_INF_F) {
    *dst = make_float4(0.f, 0.f, 0.f, 0.f);
    if (lse_writer) p.lse[row] = -CUDART_INF_F;
    return;
  }
  const float inv = 1.f / L;
  *dst = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  if (lse_writer) p.lse[row] = (M + log2f(L)) * 0.6931471805599453f;
}

}  // namespace mla
