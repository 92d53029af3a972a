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
// fully coalesced over the 512-wide rows.
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
};

__global__ void __launch_bounds__(128) combine_kernel(const CombineParams p) {
  const int row = blockIdx.x;
  const int tid = threadIdx.x;
  const int b = row / p.rows_per_stream;
  const int S = p.seq_lens[b];
  if (S < p.q || S > p.Smax) return;   // reported by the split kernel
  const int ns = min(p.nsplit, (S + p.chunk_keys - 1) / p.chunk_keys);
  const float2* ml = p.part_ml + row;
  float M = -CUDART_INF_F;
#pragma unroll 8
  for (int s = 0; s < ns; ++s) {
    const float2 v = ml[static_cast<size_t>(s) * p.N];
    M = v.y > 0.f ? fmaxf(M, v.x) : M;
  }
  float4* dst = reinterpret_cast<float4*>(p.out + static_cast<size_t>(row) * 512) + tid;
  if (M == -CUDART_INF_F) {
    *dst = make_float4(0.f, 0.f, 0.f, 0.f);
    if (tid == 0) p.lse[row] = -CUDART_INF_F;
    return;
  }
  // Every slice s < ns wrote its partial (an all-zero accumulator where no key
  // was visible), so the loads are unconditional: eight independent 16-byte
  // loads are in flight per thread.
  float L = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const float4* src = reinterpret_cast<const float4*>(p.part_o + static_cast<size_t>(row) * 512) + tid;
  const size_t step4 = static_cast<size_t>(p.N) * 128;   // float4s between slices
  for (int s0 = 0; s0 < ns; s0 += 8) {
    float4 o[8];
    float w[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int s = min(s0 + e, ns - 1);
      o[e] = src[s * step4];
      const float2 v = ml[static_cast<size_t>(s) * p.N];
      w[e] = (s0 + e < ns && v.y > 0.f) ? ex2(v.x - M) : 0.f;
      L += w[e] * (s0 + e < ns ? v.y : 0.f);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      acc.x += w[e] * o[e].x;
      acc.y += w[e] * o[e].y;
      acc.z += w[e] * o[e].z;
      acc.w += w[e] * o[e].w;
    }
  }
  const float inv = 1.f / L;
  *dst = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  if (tid == 0) p.lse[row] = (M + log2f(L)) * 0.6931471805599453f;
}

}  // namespace mla
