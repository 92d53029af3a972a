// Device-side split plan for calls with several streams (2..32).
//
// The host sizes the grid and the workspace for up to `nsplit_max` slices per
// stream without seeing the stream lengths (they live on the device).  With
// ragged lengths the best slice count is often smaller: the 8-stream ragged
// batch's split kernel took 86 us at 6 slices per stream and 109 us at the
// host's 8.  This kernel (one block, one warp per candidate count) estimates
// the split kernel's makespan for each candidate: the slices in the split
// kernel's start order (full slices first, slice-major; then the streams'
// shorter last slices, longest first; ordered_slice), list-scheduled onto
// slots / n_rt groups of clusters (the n_rt units of a slice start together),
// each slice costing a fixed part plus a per-tile part, measured on GB300:
// ~15 us per unit (launch, Q load, pipeline fill and drain, epilogue) and per
// 64-key tile ~0.86 us with P in one bf16 term, ~1.3 us with two.  It writes
// {chunk_tiles, nsplit} for the split and merge kernels; the host's count stays
// unless another is over 3 % cheaper.  (Computed inside the split kernel
// instead, the same estimate cost every call ~1.2 us even where it did not run.)
#pragma once
#include <cstdint>

#include "ptx.cuh"

namespace mla {

constexpr int kPlanMaxCandidates = 12;   // the largest counts up to nsplit_max
constexpr int kPlanMaxGroups = 96;       // 3 per lane
constexpr float kPlanUnitUs = 15.0f;
constexpr float kPlanTileUs1 = 0.86f;
constexpr float kPlanTileUs2 = 1.3f;

struct PlanParams {
  const int32_t* seq_lens;
  int* plan;                  // out: {chunk_tiles, nsplit}
  int B, q, Smax;
  int n_rt;                   // row tiles per stream (units per slice)
  int nsplit_max;             // the host's count (grid and workspace size)
  int min_chunk;              // shortest slice in tiles
  int slots;                  // clusters resident at once
  int two_term_max_keys;
};

// Times in 1/16 us; a group's state is the key (finish << 7 | group), so one
// warp-wide unsigned minimum (redux.sync) finds the earliest-free group.
__device__ __forceinline__ unsigned plan_time(float us) { return static_cast<unsigned>(us * 16.f + 0.5f); }

// One block of 32 * min(nsplit_max, kPlanMaxCandidates) threads.
__global__ void __launch_bounds__(32 * kPlanMaxCandidates, 1) plan_kernel(const PlanParams p) {
  __shared__ unsigned cost[kPlanMaxCandidates];
  __shared__ int chunk_of[kPlanMaxCandidates];
  // This grid is itself a programmatic dependent of the grid before it: wait
  // for that grid before reading the stream lengths.  The split kernel is this
  // grid's programmatic dependent: it may be scheduled now and waits for this
  // grid's completion before reading the plan.
  grid_dependency_wait();
  if (threadIdx.x == 0) grid_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int ncand = blockDim.x >> 5;
  const int ns = p.nsplit_max - ncand + 1 + warp;   // this warp's candidate
  int tiles = 0;
  float tile_us = kPlanTileUs1;
  if (lane < p.B) {
    const int S = p.seq_lens[lane];
    tiles = (S < p.q || S > p.Smax) ? 0 : (S + 63) / 64;
    tile_us = S <= p.two_term_max_keys ? kPlanTileUs2 : kPlanTileUs1;
  }
  const int tiles_max = max(1, static_cast<int>(__reduce_max_sync(0xFFFFFFFFu, static_cast<unsigned>(tiles))));
  const int chunk = max(p.min_chunk, (tiles_max + ns - 1) / ns);
  const int full = tiles / chunk;
  const int rem = tiles - full * chunk;
  const unsigned full_cost = plan_time(kPlanUnitUs + chunk * tile_us);   // lane b: a full slice of stream b
  const int groups = min(kPlanMaxGroups, max(1, p.slots / p.n_rt));
  unsigned g0 = lane < groups ? static_cast<unsigned>(lane) : 0xFFFFFFFFu;
  unsigned g1 = lane + 32 < groups ? static_cast<unsigned>(lane + 32) : 0xFFFFFFFFu;
  unsigned g2 = lane + 64 < groups ? static_cast<unsigned>(lane + 64) : 0xFFFFFFFFu;
  unsigned end = 0;
  int placed = 0;
  // One slice of cost c (the first `groups` slices take groups 0, 1, ... at 0).
  auto place = [&](unsigned c) {
    const unsigned m = placed < groups ? static_cast<unsigned>(placed)
                                       : __reduce_min_sync(0xFFFFFFFFu, min(g0, min(g1, g2)));
    ++placed;
    const unsigned grp = m & 127u;
    const unsigned f = (m >> 7) + c;
    end = max(end, f);
    const unsigned key = (f << 7) | grp;
    if (grp == static_cast<unsigned>(lane)) g0 = key;
    else if (grp == static_cast<unsigned>(lane + 32)) g1 = key;
    else if (grp == static_cast<unsigned>(lane + 64)) g2 = key;
  };
  for (int s = 0; s < ns; ++s) {              // full slices, slice-major
    unsigned m = __ballot_sync(0xFFFFFFFFu, full > s);
    if (!m) break;
    while (m) {
      const int b = __ffs(m) - 1;
      m &= m - 1;
      place(__shfl_sync(0xFFFFFFFFu, full_cost, b));
    }
  }
  bool left = rem > 0;                        // last slices, longest first
  while (true) {
    const unsigned key = left ? (static_cast<unsigned>(rem) << 5) | static_cast<unsigned>(31 - lane) : 0u;
    const unsigned top = __reduce_max_sync(0xFFFFFFFFu, key);
    if (top == 0u) break;
    const int b = 31 - static_cast<int>(top & 31u);
    if (lane == b) left = false;
    place(plan_time(kPlanUnitUs + static_cast<int>(top >> 5) * __shfl_sync(0xFFFFFFFFu, tile_us, b)));
  }
  if (lane == 0) {
    cost[warp] = end;
    chunk_of[warp] = chunk;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned host = cost[ncand - 1];
    int best = ncand - 1;
    for (int c = 0; c < ncand; ++c)
      if (cost[c] < host - host / 32u && cost[c] < cost[best]) best = c;
    p.plan[0] = chunk_of[best];
    p.plan[1] = p.nsplit_max - ncand + 1 + best;
  }
}

}  // namespace mla
