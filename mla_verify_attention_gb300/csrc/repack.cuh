// Paged caches whose pages are not whole 64-key tiles (page size 1, the
// scattered-row layout the pages name for production, included).
//
// The split kernel streams 64-key tiles with TMA, which needs a tile's rows to
// be contiguous.  For such caches the rows of every stream are first copied,
// in key order, into a contiguous [B][Smax][576] scratch cache in the call's
// workspace; the split kernel then runs on that copy exactly as on a
// contiguous cache (so the results are those of the contiguous call, bit for
// bit).  The copy is a plain bandwidth kernel: the cache is read once from its
// pages and written once, and ten CTAs of the split kernel then read each row
// of the copy, mostly from L2.
//
// (Gathering the rows inside the split kernel instead, with cp.async into its
// shared-memory ring, measured 135 us per call at best against 97 us for copy
// + split on a 64k-key stream with 1-key pages: the gather code competed with
// the softmax and MMA warps for the instruction cache, and a tile's rows can
// only be fetched a tile ahead.  TMA tile::gather4 moved ~16 GB/s per SM.)
#pragma once
#include <cstdint>

namespace mla {

struct RepackParams {
  const uint8_t* pool;          // [pool_rows][576] bf16 page pool
  const int32_t* block_table;   // [B][max_blocks]
  const int32_t* seq_lens;      // [B]
  uint8_t* dst;                 // [B][Smax][576] bf16 contiguous copy
  unsigned int* status;         // device status word (kStatusPage)
  int B, max_blocks, page_size, pool_pages, Smax;
};

constexpr int kRepackThreads = 256;
constexpr int kRowPieces = (kDl + kDr) * 2 / 16;         // 72 16-byte pieces per cache row
constexpr int kRepackPieces = kKeys * kRowPieces;         // per 64-key tile
constexpr int kRepackBatch = 6;                           // loads in flight per thread
static_assert(kRepackPieces % (kRepackBatch * kRepackThreads) == 0, "repack batches");

// Grid: x = 64-key tile of a stream, y = stream (strided when B > gridDim.y).
// Keys at or past seq_lens[b] (clamped to [0, Smax]) are not copied: the split
// kernel gives them no weight whatever they hold.  A block-table entry outside
// the pool is reported (kStatusPage) and replaced by page 0, as on the TMA path.
__global__ void __launch_bounds__(kRepackThreads, 4) repack_kernel(const RepackParams p) {
  __shared__ int32_t rows[kKeys];
  const int t = threadIdx.x;
  // This grid is a programmatic dependent of the grid before it: wait for
  // that grid before reading anything.  The split kernel is this grid's
  // programmatic dependent: its CTAs may start (Q loads, tensor-memory setup)
  // while the last copies run; its cache loads wait for this grid's completion.
  grid_dependency_wait();
  if (t == 0) grid_launch_dependents();
  const int key0 = blockIdx.x * kKeys;
  for (int b = blockIdx.y; b < p.B; b += gridDim.y) {
    int S = p.seq_lens[b];
    S = S < 0 ? 0 : (S > p.Smax ? p.Smax : S);
    const int nk = min(kKeys, S - key0);
    if (nk <= 0) continue;   // uniform across the block
    __syncthreads();         // rows[] of the previous stream fully read
    if (t < nk) {
      const int key = key0 + t;
      const int blk = key / p.page_size;
      int page = p.block_table[static_cast<size_t>(b) * p.max_blocks + blk];
      if (page < 0 || page >= p.pool_pages) {
        atomicOr(p.status, kStatusPage);
        page = 0;
      }
      rows[t] = page * p.page_size + (key - blk * p.page_size);
    }
    __syncthreads();
    uint8_t* out = p.dst + (static_cast<size_t>(b) * p.Smax + key0) * (kRowPieces * 16);
#pragma unroll 1
    for (int base = 0; base < kRepackPieces; base += kRepackBatch * kRepackThreads) {
      uint4 v[kRepackBatch];
#pragma unroll
      for (int i = 0; i < kRepackBatch; ++i) {
        const int idx = base + i * kRepackThreads + t;
        const int r = idx / kRowPieces;
        const int c = idx - r * kRowPieces;
        if (r < nk)
          v[i] = __ldg(reinterpret_cast<const uint4*>(p.pool + static_cast<size_t>(rows[r]) * (kRowPieces * 16)) + c);
      }
#pragma unroll
      for (int i = 0; i < kRepackBatch; ++i) {
        const int idx = base + i * kRepackThreads + t;
        const int r = idx / kRowPieces;
        const int c = idx - r * kRowPieces;
        if (r < nk) reinterpret_cast<uint4*>(out + static_cast<size_t>(r) * (kRowPieces * 16))[c] = v[i];
      }
    }
  }
}

}  // namespace mla
