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

// Running state of one row's merge: max M (log2 units), sum L and four
// accumulator columns.
struct MergeState {
  float M, L;
  float4 acc;
};

__device__ __forceinline__ MergeState empty_state() {
  MergeState st;
  st.M = -CUDART_INF_F;
  st.L = 0.f;
  st.acc = make_float4(0.f, 0.f, 0.f, 0.f);
  return st;
}

// The row's slice count, or -1 for a stream length the split kernel reported.
__device__ __forceinline__ int row_slices(const CombineParams& p, int row) {
  const int S = p.seq_lens[row / p.rows_per_stream];
  if (S < p.q || S > p.Smax) return -1;
  const int chunk_keys = p.plan != nullptr ? p.plan[0] * 64 : p.chunk_keys;
  return min(p.plan != nullptr ? p.plan[1] : p.nsplit, (S + chunk_keys - 1) / chunk_keys);
}

// Slices first, first + stride, ... (< ns) of one row into `st`.  Every slice
// wrote its partial (an all-zero accumulator where no key was visible).  A
// batch's (m, l) pairs and accumulators are all requested before any is used;
// batches are merged online.  `ml` and `src` point at slice 0 of the row.
template <int kBatch>
__device__ __forceinline__ void merge_slices(MergeState& st, const float2* ml, const float4* src,
                                             int N, int ns, int first, int stride) {
  const size_t step4 = static_cast<size_t>(N) * 128;   // float4s between slices
  for (int s0 = first; s0 < ns; s0 += kBatch * stride) {
    float2 v[kBatch];
    float4 o[kBatch];
#pragma unroll
    for (int e = 0; e < kBatch; ++e) {
      const int s = s0 + e * stride;
      if (s < ns) {
        v[e] = ml[static_cast<size_t>(s) * N];
        o[e] = src[s * step4];
      } else {
        v[e] = make_float2(-CUDART_INF_F, 0.f);
        o[e] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    float Mb = st.M;
#pragma unroll
    for (int e = 0; e < kBatch; ++e) Mb = v[e].y > 0.f ? fmaxf(Mb, v[e].x) : Mb;
    if (Mb == -CUDART_INF_F) continue;            // nothing visible so far
    const float c = ex2(st.M - Mb);               // 0 while M = -inf (L, acc are 0 then)
    st.L *= c;
    st.acc.x *= c; st.acc.y *= c; st.acc.z *= c; st.acc.w *= c;
#pragma unroll
    for (int e = 0; e < kBatch; ++e) {
      const float w = v[e].y > 0.f ? ex2(v[e].x - Mb) : 0.f;
      st.L += w * v[e].y;
      st.acc.x += w * o[e].x;
      st.acc.y += w * o[e].y;
      st.acc.z += w * o[e].z;
      st.acc.w += w * o[e].w;
    }
    st.M = Mb;
  }
}

// The states of kGroups groups of kLanes threads (thread t of group g holds
// columns t) merged through shared memory into group 0's threads; the other
// groups' threads get false and are done.  Every thread of the block calls it.
template <int kGroups, int kLanes>
__device__ __forceinline__ bool merge_groups(MergeState& st, int grp, int t) {
  __shared__ float gm[kGroups], gl[kGroups];
  __shared__ float4 gacc[kGroups][kLanes];
  if (t == 0) {
    gm[grp] = st.M;
    gl[grp] = st.L;
  }
  gacc[grp][t] = st.acc;
  __syncthreads();
  if (grp != 0) return false;
  st = empty_state();
#pragma unroll
  for (int g = 0; g < kGroups; ++g) st.M = gl[g] > 0.f ? fmaxf(st.M, gm[g]) : st.M;
  if (st.M != -CUDART_INF_F) {
#pragma unroll
    for (int g = 0; g < kGroups; ++g) {
      const float w = gl[g] > 0.f ? ex2(gm[g] - st.M) : 0.f;
      const float4 a = gacc[g][t];
      st.L += w * gl[g];
      st.acc.x += w * a.x;
      st.acc.y += w * a.y;
      st.acc.z += w * a.z;
      st.acc.w += w * a.w;
    }
  }
  return true;
}

// Four columns (float4 `col4`) of the normalised output row, and its lse when
// `lse_writer`; an empty row gives out = 0 and lse = -inf.
__device__ __forceinline__ void write_row(const CombineParams& p, int row, int col4,
                                          const MergeState& st, bool lse_writer) {
  float4* dst = reinterpret_cast<float4*>(p.out + static_cast<size_t>(row) * 512) + col4;
  if (st.M == -CUDART_INF_F) {
    *dst = make_float4(0.f, 0.f, 0.f, 0.f);
    if (lse_writer) p.lse[row] = -CUDART_INF_F;
    return;
  }
  const float inv = 1.f / st.L;
  *dst = make_float4(st.acc.x * inv, st.acc.y * inv, st.acc.z * inv, st.acc.w * inv);
  if (lse_writer) p.lse[row] = (st.M + log2f(st.L)) * 0.6931471805599453f;
}

// One block of 128 * kGroups threads per row.  kBatch 16: four blocks per SM
// (<= 128 registers), all rows of a 64-head, 9-draft call in one wave; kBatch
// 8 and 4: 6 and 12 blocks per SM.  kGroups > 1 (few rows, many slices): each
// of kGroups groups of 128 threads merges every kGroups-th slice of the row.
template <int kBatch, int kGroups>
__global__ void __launch_bounds__(128 * kGroups, kGroups > 1 ? 1 : (kBatch == 16 ? 4 : (kBatch == 8 ? 6 : 12)))
    combine_kernel(const CombineParams p) {
  wait_for_split_grid();
  const int row = blockIdx.x;
  const int tid = threadIdx.x & 127;
  const int grp = threadIdx.x >> 7;
  const int ns = row_slices(p, row);
  if (ns < 0) return;   // reported by the split kernel
  MergeState st = empty_state();
  merge_slices<kBatch>(st, p.part_ml + row,
                       reinterpret_cast<const float4*>(p.part_o + static_cast<size_t>(row) * 512) + tid,
                       p.N, ns, grp, kGroups);
  if (kGroups > 1 && !merge_groups<kGroups, 128>(st, grp, tid)) return;
  write_row(p, row, tid, st, tid == 0);
}

// Few rows and many slices (e.g. 8 heads over a long stream): each row is
// merged by kCols blocks of 512 / kCols columns, and in each block kGroups
// groups of 32 threads (4 columns a thread) merge every kGroups-th slice, so
// that up to kBatch * kGroups slices' loads are in flight per block at once.
// Grid (rows, kCols).
template <int kBatch, int kGroups, int kCols>
__global__ void __launch_bounds__(32 * kGroups, 2) combine_cols_kernel(const CombineParams p) {
  static_assert(kCols * 32 * 4 == 512, "one float4 per thread of a 32-thread group");
  wait_for_split_grid();
  const int row = blockIdx.x;
  const int lane = threadIdx.x & 31;
  const int grp = threadIdx.x >> 5;
  const int ns = row_slices(p, row);
  if (ns < 0) return;   // reported by the split kernel
  const int col4 = blockIdx.y * 32 + lane;                 // float4 column of this thread
  MergeState st = empty_state();
  merge_slices<kBatch>(st, p.part_ml + row,
                       reinterpret_cast<const float4*>(p.part_o + static_cast<size_t>(row) * 512) + col4,
                       p.N, ns, grp, kGroups);
  if (!merge_groups<kGroups, 32>(st, grp, lane)) return;
  write_row(p, row, col4, st, blockIdx.y == 0 && lane == 0);
}

}  // namespace mla
