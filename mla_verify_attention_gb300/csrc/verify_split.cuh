// Split kernel of absorbed-MLA verify attention on sm_103a.
//
// What it computes (pages by title):
//   "The Flash Attention Kernel That Had to Be Built: Designing sm_120 MLA
//   Verify for Blackwell Consumer GPUs", section "What Input Knowledge Is
//   Required to Understand This Message": score = q_nope . kv_c + q_pe . k_pe
//   over a 576-wide cache row, tree-masked, softmax, output = weighted sum of
//   the 512-wide latent; online softmax over key tiles ("Flash Attention
//   Algorithm").  "The Decisive Microbench: When Theory Meets Silicon",
//   section "The KV-Split Solution": each block works on one slice of the key
//   range and leaves its unnormalised accumulator and statistics in scratch
//   for a second, merging kernel.
//
// How (GB300 design, not the pages' sm_120 one).  In absorbed MLA every head
// reads the same latent cache, so the 64 heads x q_len drafts of a stream are
// the M dimension of one dense contraction.  One work unit is 128 query rows
// (flattened (draft, head) rows of one stream) against one key slice, run by a
// cluster of two CTAs on two SMs:
//
//   S CTA (cluster rank 0): Q[128 x 576] bf16 lives in tensor memory and is
//     the A operand of S = Q K^T (tcgen05.mma, M=128, N=64 keys, K=576, fp32
//     scores in tensor memory, double-buffered).  Eight softmax warps, two
//     threads per row (32 keys each): scale, tree mask, running max with lazy
//     rescaling, exp2, running sum, and bf16 P, staged in shared memory with
//     the per-row rescale factors and moved into the O CTA by one bulk copy
//     per tile.
//   O CTA (cluster rank 1): owns the 128 x 512 fp32 accumulator, i.e. all 512
//     tensor-memory columns.  Its MMA warp runs O += P V with P (K-major) and
//     V (MN-major, the latent part of the same cache rows) from shared memory,
//     N=256 per instruction.  Eight helper warps rescale O rows when the S CTA
//     raised a row's max, zero cache rows past the slice end, and write the
//     result through shared memory and TMA tensor stores.
//
// Each CTA streams the cache slice it needs with TMA (128-byte swizzle), from
// a contiguous cache or from pages of a multiple of 64 keys (caches with other
// page sizes are first copied into a contiguous one, see repack.cuh).  P is
// rounded to bf16 because V is bf16 in the cache.  With the lazily kept row
// max even the dominant key's p carries that rounding, so streams up to
// two_term_max_keys keys (where a few keys carry most of the weight) send P as
// two bf16 terms hi + lo and the PV product is issued once per term.  The
// kCorrect instantiation sends one term for longer streams and removes the
// dominant key's rounding instead: each softmax thread tracks its largest
// score since its row's max last changed and keeps that half tile's scores,
// finds the key after the loop and recomputes the error p - bf16(p) of its P,
// and the O CTA adds error x that key's value row to the accumulator before
// the epilogue.
//
// Units start in index order.  For 2..32 streams the index order is a list
// schedule (ordered_slice), and the slice length may come from plan_kernel
// (planner.cuh), which chose it from the stream lengths.
#pragma once
#include <cstdint>
#include <cstdio>
#include <cuda.h>
#include <math_constants.h>

#include "ptx.cuh"

namespace mla {

constexpr int kDl = 512;
constexpr int kDr = 64;
constexpr int kRows = 128;                       // query rows per unit (MMA M)
constexpr int kKeys = 64;                        // keys per tile (QK N, PV K)
constexpr int kChunk = kKeys * 64 * 2;           // 8 KB: 64 keys x 64 dims bf16
constexpr int kQChunk = kRows * 64 * 2;          // 16 KB: 128 rows x 64 dims bf16
constexpr int kKChunks = 9;                      // 576 / 64
constexpr int kVChunks = 8;                      // 512 / 64
constexpr int kKSlots = 2;                       // S CTA key-tile ring: 2 x 72 KB
constexpr int kVSlots = 2;                       // O CTA value-tile ring: 2 x 64 KB
constexpr int kKTile = kKChunks * kChunk;        // 72 KB per key tile, loaded as two boxes:
constexpr int kKSplit = 5;                       //   part 0 = chunks 0..4 (40 KB),
constexpr int kKPart0 = kKSplit * kChunk;        //   part 1 = chunks 5..8 (32 KB), each with
constexpr int kKPart1 = kKTile - kKPart0;        //   its own full / empty barriers
constexpr int kVTile = kVChunks * kChunk;        // 64 KB: one TMA box per tile
constexpr int kPTerm = kRows * kKeys * 2;        // 16 KB per P term
// One P exchange buffer: [alpha: 128 f32 | flags: 4 u32 | pad][P hi][P lo].
// The S CTA fills its copy and moves it with one bulk copy into the same
// offset of the O CTA, where the PV MMA reads P from it.
constexpr int kPHead = 1024;
constexpr int kPBuf = kPHead + 2 * kPTerm;
constexpr int kPOffset = kKSlots * kKTile;       // after the K ring / V tiles (144 KB)
constexpr int kThreads = 384;                    // 12 warps: 4 control + 8 row warps
// Q rows are staged (by TMA, then moved to tensor memory by the softmax warps)
// behind key slot 0, so that key tile 0 can load at the same time as Q.
constexpr int kQStage = kKTile;
constexpr int kQBytes = kKChunks * kQChunk;     // 144 KB
constexpr int kRingBytes = (kPOffset + 2 * kPBuf > kQStage + kQBytes) ? kPOffset + 2 * kPBuf
                                                                      : kQStage + kQBytes;
constexpr uint32_t kSoftmaxBar = 1;              // named barrier of the 8 softmax warps
constexpr uint32_t kEpilogueBar = 2;             // O CTA: 2 and 3, one per half of the helpers
constexpr int kOutBlock = kRows * 32 * 4;        // 16 KB: [128 rows][32 fp32 columns]
constexpr int kOutBufs = 6;                      // staging blocks per helper half
static_assert(2 * kOutBufs * kOutBlock <= kRingBytes, "epilogue staging must fit the ring");
constexpr int kRowThreads = 256;                 // two threads per row (one per 32-key half)
constexpr uint32_t kQCols = 288;                 // Q in tensor memory: 576 bf16 = 288 cols
// Dominant-key correction (kCorrect): a row's correction is skipped when its
// error is not above 2^-kCorrSkipLog2 of the row sum; a skipped term moves the
// output by at most 2^-13 of a value entry.
constexpr float kCorrSkipLog2 = 13.0f;
// kCorrect, S CTA: the scores of the tile that holds each row half's largest
// score are kept (128 bytes per row half, 16-byte units XOR-swizzled by row)
// in the second P term's space of the two P buffers, unused with one term.
constexpr int kTopScoresOffset = kPOffset + kPHead + kPTerm;   // + half * kPBuf
// Per helper warp: 32 rows x 64 bytes of value rows, the transpose buffer of
// the correction's coalesced loads, after the epilogue's staging blocks.
constexpr int kCorrBufOffset = 2 * kOutBufs * kOutBlock;
constexpr int kCorrWarpBytes = 32 * 64;
static_assert(kCorrBufOffset + 8 * kCorrWarpBytes <= kRingBytes, "correction buffers must fit the ring");
constexpr float kLazyRescale = 8.0f;             // log2 units: keep the max unless it grows by 2^8
constexpr uint64_t kWaitNs = 2000000000ull;      // bounded waits: 2 s

constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 64, 0, 0);
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 256, 0, 1);

enum : uint32_t { kCmdDone = 0xFFFFFFFFu, kCmdZeroTail = 0x80000000u };

// Device status bits (first error wins in the host's report).
enum : uint32_t { kStatusSeqLen = 1u, kStatusTimeout = 2u, kStatusPage = 4u };

// Optional timeline of the split kernel (a build with -DMLA_TRACE; the
// library's normal build compiles every stamp away).  %globaltimer stamps, in
// ns: per tile j of the first kTraceUnits work units, the moments each role
// passed its pipeline waits (kTrace* below), and per CTA of every unit (up to
// kTraceSpanUnits) the moments it passed the prologue, loop and epilogue.
#ifdef MLA_TRACE
constexpr int kTraceUnits = 8, kTraceEvents = 10, kTraceTiles = 128, kTraceSpanUnits = 1024;
constexpr int kTraceSpans = 12;
__device__ unsigned long long g_trace_tiles[kTraceUnits][2][kTraceEvents][kTraceTiles];
__device__ unsigned long long g_trace_spans[kTraceSpanUnits][2][kTraceSpans];
#define MLA_TRACE_TILE(ev, j)                                                           \
  do {                                                                                  \
    const int u_ = static_cast<int>(blockIdx.x >> 1);                                   \
    if (u_ < kTraceUnits && (j) < kTraceTiles)                                          \
      g_trace_tiles[u_][blockIdx.x & 1][ev][j] = globaltimer_ns();                      \
  } while (0)
#define MLA_TRACE_SPAN(ev)                                                              \
  do {                                                                                  \
    const int u_ = static_cast<int>(blockIdx.x >> 1);                                   \
    if (u_ < kTraceSpanUnits) g_trace_spans[u_][blockIdx.x & 1][ev] = globaltimer_ns(); \
  } while (0)
#else
#define MLA_TRACE_TILE(ev, j) do {} while (0)
#define MLA_TRACE_SPAN(ev) do {} while (0)
#endif
// Tile events: S CTA (rank 0) / O CTA (rank 1).
enum {
  kTrQK0 = 0,      // S MMA warp: key tile part 0 landed, QK(j) starts
  kTrQK1 = 1,      //   part 1 landed
  kTrQKIssued = 2, //   QK(j) issued and committed
  kTrSoftIn = 3,   // S softmax (warp 4, lane 0): scores of tile j in registers
  kTrStaged = 4,   //   P(j) staged, before the per-tile barrier
  kTrBarrier = 5,  //   past the per-tile barrier
  kTrCopy = 6,     // S copy issuer: O's P buffer free, P(j) copy issued
  kTrKLoad0 = 7,   // S producer: part 0 of key tile j issued (slot free)
  kTrKLoad1 = 8,   //   part 1 issued
  kTrPFull = 0,    // O MMA warp: P(j) landed
  kTrVFull = 1,    //   value tile j landed
  kTrPVIssued = 2, //   PV(j) issued and committed
  kTrVLoad = 3,    // O producer: value slot free, tile j issued
};
// Spans (per CTA): entry, prologue done (after the cluster sync), Q landed (S)
// / -, Q in tensor memory (S) / -, main loop done, results ready for the
// epilogue (O), epilogue stores complete (O), exit; within the prologue: unit
// decoded, barriers initialised and first loads issued, tensor memory
// allocated, CTA barrier passed.
enum { kSpEntry = 0, kSpSynced = 1, kSpQLanded = 2, kSpQReady = 3, kSpLoopDone = 4,
       kSpEpiReady = 5, kSpEpiDone = 6, kSpExit = 7, kSpDecoded = 8, kSpIssued = 9,
       kSpAlloc = 10, kSpCtaSync = 11 };

struct SplitParams {
  const int32_t* seq_lens;
  const uint32_t* mask;
  float* lse;
  float2* part_ml;    // [nsplit][B*rows]; the outputs themselves go through the map_out tensor map
  unsigned int* status;
  int B, q, H, Smax;
  int n_rt, nsplit, chunk_tiles;
  int two_term_max_keys;
  float scale_log2;   // scale * log2(e)
  // Paged cache (null block_table: contiguous [B][Smax][576] cache).  Key k of
  // stream b is row block_table[b][k / page_size] * page_size + k % page_size of
  // the page pool, with page_size a multiple of 64 (no tile crosses a page).
  const int32_t* block_table;   // [B][max_blocks]
  int max_blocks, page_size, pool_pages;
  // Test control (mla_verify_attn_set_test_controls): unit 0 never loads the second part of
  // key tile 0, so its bounded waits run out and report MLA_ERR_DEVICE_TIMEOUT.
  int test_stall;
  // Calls with 2..kOrderedStreams streams: {chunk_tiles, nsplit} chosen by
  // plan_kernel from the stream lengths (null: the host's values hold).  nsplit
  // above stays the host's (grid, workspace, partials or direct output).
  const int* plan;
  // The cache the tensor maps describe, for the dominant-key correction's
  // row reads: [streams][kv_rows][576] bf16 (paged: one stream of pool rows).
  const uint8_t* kv;
  long long kv_rows;
};

struct __align__(1024) Smem {
  uint8_t ring[kRingBytes];
  float2 ml[kRows];
  float xmax[2][kRows];      // S CTA: per-half partial row max of the current tile
  float xl[kRows];           // S CTA: second half's running sum, combined at the end
  float2 xbest[2][kRows];    // S CTA, per half: {largest score, its key} (kCorrect)
  float2 corr[kRows];        // O CTA: {P error, key} of the row's dominant key (kCorrect)
  uint64_t kfull[2][kKSlots], kempty[2][kKSlots];   // [part][slot]
  uint64_t qfull, qready;
  uint64_t sfull[2], sempty[2];
  uint64_t pempty[2];
  uint64_t vfull[kVSlots], vempty[kVSlots];
  uint64_t pfull[2];
  uint64_t odone, corrgo, corrdone, mlfull, drain;
  uint32_t tmem_base;
  uint32_t abort_flag;
  uint32_t cmd;
};

struct Unit {
  int b, rt, sp;
  int S, prefix;
  int k0, k1, ntiles;
  int rows_total, row0, valid_rows;
  bool empty, two_term, zero_tail;
};

// Streams up to which slices are started longest first (one lane per stream).
constexpr int kOrderedStreams = 32;
// How the split kernel follows the preceding grid (template parameter kDep).
constexpr int kDepNone = 0, kDepCopy = 1, kDepPlan = 2;
constexpr int kMinSliceTiles = 2;   // shortest slice: a unit's fixed cost needs a few tiles

// Slice (stream b, index sp, stream length S_b) of the t-th slice in start
// order, for B <= kOrderedStreams; b = -1 for the empty slices at the end.  Clusters start in
// index order, so this is a list schedule: every stream's full-length slices
// first (slice-major), then the streams' shorter last slices, longest first
// (ties: lower stream first), so that the device does not end on a tail of
// long slices started late.  Computed by each warp with one lane per stream.
__device__ __forceinline__ void ordered_slice(const SplitParams& p, int chunk, int t, int& b, int& sp,
                                              int& S_b) {
  const int lane = threadIdx.x & 31;
  int tiles = 0, S = 0;
  if (lane < p.B) {
    S = p.seq_lens[lane];
    tiles = (S < p.q || S > p.Smax) ? 0 : (S + kKeys - 1) / kKeys;
  }
  const int full = tiles / chunk;
  const int rem = tiles - full * chunk;
  int base = 0;
  for (int s = 0; s < p.nsplit; ++s) {
    unsigned m = __ballot_sync(0xFFFFFFFFu, full > s);
    const int n = __popc(m);
    if (n == 0) break;
    if (t < base + n) {
      for (int i = 0; i < t - base; ++i) m &= m - 1;   // the (t - base)-th stream with a slice s
      b = __ffs(m) - 1;
      sp = s;
      S_b = __shfl_sync(0xFFFFFFFFu, S, b);
      return;
    }
    base += n;
  }
  t -= base;
  int rank = 0;   // among the shorter last slices
  for (int o = 0; o < 32; ++o) {
    const int ro = __shfl_sync(0xFFFFFFFFu, rem, o);
    rank += (ro > rem || (ro == rem && o < lane)) ? 1 : 0;
  }
  const unsigned hit = __ballot_sync(0xFFFFFFFFu, rem > 0 && rank == t);
  const int src = hit ? __ffs(hit) - 1 : 0;
  const int full_hit = __shfl_sync(0xFFFFFFFFu, full, src);
  S_b = __shfl_sync(0xFFFFFFFFu, S, src);
  b = hit ? src : -1;
  sp = hit ? full_hit : 0;
}

// Called by every thread of the CTA (full warps) at kernel start.
__device__ __forceinline__ Unit decode_unit(const SplitParams& p) {
  Unit u;
  // Each slice's n_rt row tiles are consecutive units (they read the same keys).
  // For 2 to kOrderedStreams streams, slices start longest first
  // (ordered_slice); otherwise slice-major (all streams' slice 0, then slice 1,
  // ...), which for one stream is the same order.
  const int unit = blockIdx.x >> 1;
  u.rt = unit % p.n_rt;
  const int t = unit / p.n_rt;
  int b, sp, S;
  int chunk = p.chunk_tiles;
  if (p.B > 1 && p.B <= kOrderedStreams) {
    if (p.plan != nullptr) chunk = p.plan[0];   // the slice length plan_kernel chose
    ordered_slice(p, chunk, t, b, sp, S);
  } else {
    b = t % p.B;
    sp = t / p.B;
    S = p.seq_lens[b];
  }
  const bool none = b < 0;   // an empty slice at the end of the order
  u.b = none ? 0 : b;
  u.sp = sp;
  u.S = none ? p.q : S;
  u.prefix = u.S - p.q;
  u.rows_total = p.q * p.H;
  u.row0 = u.rt * kRows;
  u.valid_rows = min(kRows, u.rows_total - u.row0);
  const bool bad = u.S < p.q || u.S > p.Smax;
  u.k0 = u.sp * chunk * kKeys;
  u.k1 = min(u.S, u.k0 + chunk * kKeys);
  u.empty = none || bad || u.k0 >= u.k1;
  u.ntiles = u.empty ? 0 : (u.k1 - u.k0 + kKeys - 1) / kKeys;
  u.two_term = u.S <= p.two_term_max_keys;
  u.zero_tail = !u.empty && ((u.k1 - u.k0) % kKeys) != 0;
  return u;
}

// TMA coordinates (row, stream) of the first key of a 64-key tile: the key
// within stream b of the contiguous cache, or the row of the page pool.  A
// block-table entry outside the pool is reported and replaced by page 0.
// (The cache layout is a template parameter of the producers: a per-tile
// runtime test in the MMA warps' loops had measurably slowed the MMA issue
// even when never taken.)
template <bool kPaged>
__device__ __forceinline__ int2 tile_origin(const SplitParams& p, const Unit& u, int key) {
  if (!kPaged) return make_int2(key, u.b);
  const int blk = key / p.page_size;
  int page = __ldg(p.block_table + static_cast<size_t>(u.b) * p.max_blocks + blk);
  if (page < 0 || page >= p.pool_pages) {
    atomicOr(p.status, kStatusPage);
    page = 0;
  }
  return make_int2(page * p.page_size + (key - blk * p.page_size), 0);
}

// Bounded wait that also gives up as soon as another warp of the CTA aborted.
// On a timeout the kernel records the error, prints which wait gave up (site
// number, cluster rank, warp, parity) and makes the other warps unwind.
template <bool kCluster = false>
__device__ __noinline__ bool wait_slow(Smem& sm, uint32_t bar, uint32_t parity,
                                       const SplitParams& p, int site) {
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
    if (*reinterpret_cast<volatile uint32_t*>(&sm.abort_flag)) return false;
    if (globaltimer_ns() - t0 > kWaitNs) {
      atomicOr(p.status, kStatusTimeout);
      *reinterpret_cast<volatile uint32_t*>(&sm.abort_flag) = 1u;
      printf("mla_verify_attn: wait timed out: site %d rank %u block %d warp %d parity %u\n", site,
             cluster_ctarank(), static_cast<int>(blockIdx.x), static_cast<int>(threadIdx.x >> 5),
             parity);
      return false;
    }
  }
}

template <bool kCluster = false>
__device__ __forceinline__ bool wait_or_abort(Smem& sm, uint32_t bar, uint32_t parity,
                                              const SplitParams& p, int site) {
  if (kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
  return wait_slow<kCluster>(sm, bar, parity, p, site);
}

// Wait by a whole converged warp; the result is made warp-uniform so that the
// warp can keep executing .sync.aligned / elect.sync instructions together.
template <bool kCluster = false>
__device__ __forceinline__ bool warp_wait(Smem& sm, uint32_t bar, uint32_t parity,
                                          const SplitParams& p, int site) {
  const bool ok = wait_or_abort<kCluster>(sm, bar, parity, p, site);
  return __all_sync(0xFFFFFFFFu, ok);
}

// Before a CTA exits, every TMA copy it issued must have landed: wait for the
// last phase each ring slot was armed for.  Consumed phases return at once.
__device__ __forceinline__ void drain_ring(const uint64_t* full, int nslots, int n_issued) {
  for (int n = n_issued - 1; n >= 0 && n >= n_issued - nslots; --n)
    mbar_wait(smem_u32(&full[n % nslots]), (n / nslots) & 1, kWaitNs / 2);
}

// ============================================================ S CTA roles

// Key tile j, part `part` (chunks 0..4 or 5..8) into its ring slot.
__device__ __forceinline__ void s_issue_part(Smem& sm, const CUtensorMap* map_kv0,
                                             const CUtensorMap* map_kv1, int2 org, int j, int part,
                                             int* n_issued) {
  const int slot = j % kKSlots;
  const uint32_t full = smem_u32(&sm.kfull[part][slot]);
  mbar_arrive_expect_tx(full, part ? kKPart1 : kKPart0);
  tma_load_4d(smem_u32(sm.ring) + slot * kKTile + part * kKPart0, part ? map_kv1 : map_kv0, 0,
              org.x, part ? kKSplit : 0, org.y, full);
  n_issued[part] = j + 1;
}

// Thread 0, right after the barriers are initialised and before the CTA and
// cluster syncs (~0.8 us): the Q rows of this unit (8 latent chunks + 1 rope
// chunk of [128 rows x 64 dims], as boxes [8][128][64] of q_nope and [128][64]
// of q_rope) and, unless the cache is a copy still being written by the
// preceding grid, key tile 0 (slot 0 lies outside the Q staging area).
template <bool kPaged, bool kAfterCopy>
__device__ __forceinline__ void s_producer_start(Smem& sm, const Unit& u, const SplitParams& p,
                                                 const CUtensorMap* map_qn, const CUtensorMap* map_qr,
                                                 const CUtensorMap* map_kv0, const CUtensorMap* map_kv1,
                                                 int* n_issued) {
  tma_prefetch_desc(map_qn);
  tma_prefetch_desc(map_qr);
  tma_prefetch_desc(map_kv0);
  tma_prefetch_desc(map_kv1);
  const uint32_t qst = smem_u32(sm.ring) + kQStage;
  const uint32_t qfull = smem_u32(&sm.qfull);
  const int y = u.b * u.rows_total + u.row0;
  mbar_arrive_expect_tx(qfull, kQBytes);
  tma_load_3d(qst, map_qn, 0, y, 0, qfull);
  tma_load_2d(qst + kVChunks * kQChunk, map_qr, 0, y, qfull);
  if constexpr (!kAfterCopy) {
    const int2 org = tile_origin<kPaged>(p, u, u.k0);
    s_issue_part(sm, map_kv0, map_kv1, org, 0, 0, n_issued);
    // Test hook: unit 0 never loads the second part of key tile 0.
    if (!(p.test_stall && blockIdx.x == 0)) s_issue_part(sm, map_kv0, map_kv1, org, 0, 1, n_issued);
  }
}

// The rest of the key tiles, after the syncs.  Two boxes per 64-key tile:
// [5 chunks][64 keys][64 dims] and [4 chunks][64][64].  A part's buffer is
// refilled as soon as the MMAs that read it are done, so the first chunks of
// tile j+2 load while the last ones of tile j are used.  Tile origins are
// looked up two tiles ahead (a block-table read for paged caches).
template <bool kPaged, bool kAfterCopy>
__device__ __forceinline__ void s_producer(Smem& sm, const Unit& u, const SplitParams& p,
                                           const CUtensorMap* map_kv0, const CUtensorMap* map_kv1,
                                           int* n_issued) {
  if (kAfterCopy) grid_dependency_wait();   // the cache is the preceding grid's copy
  const int j0 = kAfterCopy ? 0 : 1;
  // (Block-table entries are read only for tiles of the slice.)
  int2 org0 = j0 < u.ntiles ? tile_origin<kPaged>(p, u, u.k0 + j0 * kKeys) : make_int2(0, 0);
  int2 org1 = j0 + 1 < u.ntiles ? tile_origin<kPaged>(p, u, u.k0 + (j0 + 1) * kKeys) : org0;
  for (int j = j0; j < u.ntiles; ++j) {
    const int2 org = org0;
    org0 = org1;
    if (j + 2 < u.ntiles) org1 = tile_origin<kPaged>(p, u, u.k0 + (j + 2) * kKeys);
    if (j == 1) {
      // Slot 1 lies in the Q staging area: wait until the softmax warps have
      // moved Q into tensor memory.
      if (!wait_or_abort(sm, smem_u32(&sm.qready), 0, p, 1)) return;
      fence_proxy_async();
    }
    const int slot = j % kKSlots;
#pragma unroll
    for (int part = 0; part < 2; ++part) {
      if (p.test_stall && blockIdx.x == 0 && j == 0 && part == 1) continue;
      if (!wait_or_abort(sm, smem_u32(&sm.kempty[part][slot]), ((j / kKSlots) & 1) ^ 1, p, 2))
        return;
      s_issue_part(sm, map_kv0, map_kv1, org, j, part, n_issued);
      MLA_TRACE_TILE(kTrKLoad0 + part, j);
    }
  }
}

// The MMA warp runs converged; one elected lane issues (issue cost then stays
// negligible next to the 36 MMAs of a tile).
__device__ __forceinline__ void s_mma(Smem& sm, const Unit& u, const SplitParams& p,
                                      uint32_t tmem) {
  const uint32_t ring = smem_u32(sm.ring);
  if (!warp_wait(sm, smem_u32(&sm.qready), 0, p, 3)) return;
  tc_fence_after();
  for (int j = 0; j < u.ntiles; ++j) {
    const int buf = j & 1;
    if (!warp_wait(sm, smem_u32(&sm.sempty[buf]), ((j >> 1) & 1) ^ 1, p, 4)) return;
    tc_fence_after();
    const uint32_t d = tmem + kQCols + 64 * buf;
    const int slot = j % kKSlots;
    // Descriptor of chunk c = descriptor of chunk 0 + c * 8 KB (in 16-byte units).
    const uint64_t bdesc0 = sdesc_sw128(ring + slot * kKTile, 16, 1024);
    if (!warp_wait(sm, smem_u32(&sm.kfull[0][slot]), (j / kKSlots) & 1, p, 5)) return;
    if ((threadIdx.x & 31) == 0) MLA_TRACE_TILE(kTrQK0, j);
    tc_fence_after();
#pragma unroll
    for (int c = 0; c < kKSplit; ++c)
      mma_ts_chunk_elect(d, tmem + c * 32, bdesc0 + static_cast<uint64_t>(c * (kChunk >> 4)),
                         kIdescQK, c != 0);
    mma_commit_elect(smem_u32(&sm.kempty[0][slot]));
    if (!warp_wait(sm, smem_u32(&sm.kfull[1][slot]), (j / kKSlots) & 1, p, 5)) return;
    if ((threadIdx.x & 31) == 0) MLA_TRACE_TILE(kTrQK1, j);
    tc_fence_after();
#pragma unroll
    for (int c = kKSplit; c < kKChunks; ++c)
      mma_ts_chunk_elect(d, tmem + c * 32, bdesc0 + static_cast<uint64_t>(c * (kChunk >> 4)),
                         kIdescQK, 1u);
    mma_commit_elect(smem_u32(&sm.kempty[1][slot]));
    mma_commit_elect(smem_u32(&sm.sfull[buf]));
    if ((threadIdx.x & 31) == 0) MLA_TRACE_TILE(kTrQKIssued, j);
  }
}

// Eight softmax warps: warp 4+w and warp 8+w both own tensor-memory lanes
// 32w..32w+31 (one query row per lane); the first takes keys 0..31 of each
// tile, the second keys 32..63.  The two halves agree on the row max through
// shared memory once per tile; each keeps its own part of the running sum.
// kTwoTerm: P goes out as two bf16 terms hi + lo (short streams).
// kCorrect: one term, plus the row's top key and its P's rounding error for
// the O CTA.
template <bool kTwoTerm, bool kCorrect>
__device__ __forceinline__ void s_softmax(Smem& sm, const Unit& u, const SplitParams& p,
                                          uint32_t tmem, int wq, int half, int lane) {
  const int r = wq * 32 + lane;                     // row of the unit == tensor-memory lane
  const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
  const int R = u.row0 + r;
  const bool row_valid = r < u.valid_rows;
  uint64_t mask64 = 0;
  if (row_valid) {
    const int i = R / p.H;
    const int words = (p.q + 31) >> 5;
    const uint32_t* mrow = p.mask + (static_cast<size_t>(u.b) * p.q + i) * words;
    mask64 = mrow[0];
    if (words > 1) mask64 |= static_cast<uint64_t>(mrow[1]) << 32;
    if (p.q < 64) mask64 &= (1ull << p.q) - 1ull;
  }

  // ---- Q: staging shared memory -> registers -> tensor memory (each half
  // moves four or five of the nine 64-dim chunks of its row).  All exits of
  // the softmax warps are taken together (they share named barriers).
  const bool qok = warp_wait(sm, smem_u32(&sm.qfull), 0, p, 6);
  if (wq == 0 && half == 0 && lane == 0) MLA_TRACE_SPAN(kSpQLanded);
  if (named_bar_red_or(kSoftmaxBar, kRowThreads, !qok)) return;
  for (int c = half; c < kKChunks; c += 2) {
    const uint8_t* src = sm.ring + kQStage + c * kQChunk + r * 128;
    uint32_t v[32];
#pragma unroll
    for (int q4 = 0; q4 < 8; ++q4) {
      const uint4 x = *reinterpret_cast<const uint4*>(src + ((q4 ^ (r & 7)) << 4));
      v[4 * q4 + 0] = x.x;
      v[4 * q4 + 1] = x.y;
      v[4 * q4 + 2] = x.z;
      v[4 * q4 + 3] = x.w;
    }
    MLA_TMEM_ST_32x32b_X32(tmem + lane_base + c * 32, v);
  }
  tmem_st_wait();
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(smem_u32(&sm.qready));
  if (wq == 0 && half == 0 && lane == 0) MLA_TRACE_SPAN(kSpQReady);

  // ---- peer (O CTA) addresses: the exchange buffers sit at the same offsets
  const uint32_t peer = 1;
  const uint32_t xbuf0 = smem_u32(sm.ring + kPOffset);
  const uint32_t xbuf0_remote = mapa_shared(xbuf0, peer);
  const uint32_t pfull_remote0 = mapa_shared(smem_u32(&sm.pfull[0]), peer);
  const uint32_t pfull_remote1 = mapa_shared(smem_u32(&sm.pfull[1]), peer);
  const uint32_t xbytes = kPHead + (kTwoTerm ? 2u : 1u) * kPTerm;

  // With a positive scale the row max is taken on raw scores and the scale is
  // folded into the exp2 argument: p = 2^(s * a - m).  Otherwise the scores
  // are scaled first and a_eff = 1.
  const float a = p.scale_log2;
  const bool pos = a > 0.f;
  const float a_eff = pos ? a : 1.f;
  float m_used = -CUDART_INF_F;   // log2-scaled running max actually used for P
  float l = 0.f;                  // this half's running sum of P
  bool copy_failed = false;       // set by the copy-issuing thread only
  bool finished = true;
  // kCorrect: this half's largest score (before the scale) since its row's
  // max last changed, and its tile, whose scores the top-scores area keeps.
  // The key's P was staged with the final max, so its rounding error follows
  // from the score alone once the loop is done; tracking costs a compare per
  // tile and a store of 32 scores when a row half sees a new top score
  // (searching for the key in every such tile slowed the loop by ~8 %).
  float best_raw = -CUDART_INF_F;
  int best_j = 0;
  uint8_t* const top_scores = sm.ring + kTopScoresOffset + half * kPBuf + r * 128;

  // Stage P (and the row sums) for 8 keys at a time into exchange buffer `xb`
  // [alpha | flags | P hi | P lo] with exponent offset msub; returns the sum.
  auto stage_p = [&](const uint32_t* sr, uint8_t* xb, float msub) -> float {
    uint8_t* ph = xb + kPHead + r * 128;
    // Exponent arguments and running sums in packed fp32 pairs.
    const uint64_t a2 = f2pack(a_eff, a_eff);
    const uint64_t m2 = f2pack(-msub, -msub);
    uint64_t ls2[2] = {0ull, 0ull};                 // bit pattern 0 = (0.f, 0.f)
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      const int unit = 4 * half + q4;               // 16-byte unit = keys 8*unit .. 8*unit+7
      uint32_t h[4], lw[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int c = 4 * q4 + e;
        float x0, x1;
        f2unpack(ffma2(f2pack(__uint_as_float(sr[2 * c]), __uint_as_float(sr[2 * c + 1])), a2, m2),
                 x0, x1);
        const float p0 = ex2(x0);
        const float p1 = ex2(x1);
        ls2[e & 1] = fadd2(ls2[e & 1], f2pack(p0, p1));
        h[e] = pack_bf16x2(p0, p1);
        if (kTwoTerm) lw[e] = pack_bf16x2(p0 - bf16lo_to_f32(h[e]), p1 - bf16hi_to_f32(h[e]));
      }
      *reinterpret_cast<uint4*>(ph + ((unit ^ (r & 7)) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
      if (kTwoTerm)
        *reinterpret_cast<uint4*>(ph + kPTerm + ((unit ^ (r & 7)) << 4)) =
            make_uint4(lw[0], lw[1], lw[2], lw[3]);
    }
    float s0, s1, s2, s3;
    f2unpack(ls2[0], s0, s1);
    f2unpack(ls2[1], s2, s3);
    return (s0 + s1) + (s2 + s3);
  };

  for (int j = 0; j < u.ntiles; ++j) {
    const int buf = j & 1;
    const bool got = warp_wait(sm, smem_u32(&sm.sfull[buf]), (j >> 1) & 1, p, 7);
    if (wq == 0 && half == 0 && lane == 0) MLA_TRACE_TILE(kTrSoftIn, j);
    uint32_t sr[32];
    float mh = -CUDART_INF_F;   // this half's tile max (log2-scaled)
    float mraw = -CUDART_INF_F; // the same before the scale (kCorrect)
    if (got) {
      tc_fence_after();
      MLA_TMEM_LD_32x32b_X32(tmem + lane_base + kQCols + 64 * buf + 32 * half, sr);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.sempty[buf]));
      if (!pos) {
#pragma unroll
        for (int c = 0; c < 32; ++c) sr[c] = __float_as_uint(__uint_as_float(sr[c]) * a);
      }

      // Keys wholly inside the prefix are visible; otherwise bit c of `vis`
      // says whether key key0+c is visible to this row.
      const int key0 = u.k0 + j * kKeys + 32 * half;
      if (!row_valid) {
#pragma unroll
        for (int c = 0; c < 32; ++c) sr[c] = __float_as_uint(-CUDART_INF_F);
      } else if (key0 + 32 > u.prefix) {
        const int np = u.prefix - key0;             // prefix keys in this half tile (may be <= 0)
        uint32_t vis = np >= 32 ? ~0u : (np > 0 ? (1u << np) - 1u : 0u);
        const uint64_t drafts = np > 0 ? mask64 << np : (-np < 64 ? mask64 >> (-np) : 0ull);
        vis |= static_cast<uint32_t>(drafts);
        const int nk = u.S - key0;                  // keys of the stream in this half tile
        if (nk < 32) vis &= nk > 0 ? (1u << nk) - 1u : 0u;
#pragma unroll
        for (int c = 0; c < 32; ++c)
          if (!((vis >> c) & 1u)) sr[c] = __float_as_uint(-CUDART_INF_F);
      }
      float mx[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) mx[k] = __uint_as_float(sr[k]);
#pragma unroll
      for (int c = 4; c < 32; ++c) mx[c & 3] = fmaxf(mx[c & 3], __uint_as_float(sr[c]));
      mraw = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
      mh = mraw * a_eff;
    }
    // Lazy rescale: P may exceed 1 by up to 2^kLazyRescale; O and l only get
    // rescaled (here and in the O CTA) when the max grows beyond that.  Each
    // half first assumes that neither half of its row needs that (the usual
    // case once a few tiles are in) and stages P with the current max; the
    // one barrier per tile tells whether any row of the tile overflowed.
    const bool ovf = mh > m_used + kLazyRescale;
    uint8_t* xb = sm.ring + kPOffset + buf * kPBuf;
    // Buffer `buf` was last read by the copy of tile j-2, which its issuer
    // saw completed before the previous tile's barrier.
    float lsum = stage_p(sr, xb, m_used == -CUDART_INF_F ? 0.f : m_used);
    if (half == 0 && lane == 0) reinterpret_cast<uint32_t*>(xb + 512)[wq] = 0u;
    // The copy of tile j-1 must have read its buffer before anyone passes
    // this barrier: tile j+1 reuses that buffer.
    if (half == 0 && r == 0) bulk_wait_read<0>();
    fence_proxy_async_smem();
    // One barrier per tile: any overflowing row, or any failed wait.  Only
    // then (rarely) a second one tells the two apart.
    if (wq == 0 && half == 0 && lane == 0) MLA_TRACE_TILE(kTrStaged, j);
    const bool any_ovf = named_bar_red_or(kSoftmaxBar, kRowThreads, ovf || !got || copy_failed);
    if (wq == 0 && half == 0 && lane == 0) MLA_TRACE_TILE(kTrBarrier, j);
    if (any_ovf) {
      if (named_bar_red_or(kSoftmaxBar, kRowThreads, !got || copy_failed)) {
        finished = false;
        break;
      }
      // Some row's max grew beyond the lazy bound: agree on the row max
      // through shared memory, rescale, and stage P again.
      sm.xmax[half][r] = mh;
      named_bar_sync(kSoftmaxBar, kRowThreads);
      const float mt = fmaxf(sm.xmax[0][r], sm.xmax[1][r]);
      float alpha = 1.f;
      bool flag = false;
      if (mt > m_used + kLazyRescale) {
        alpha = ex2(m_used - mt);          // 0 when nothing was visible before
        flag = (m_used != -CUDART_INF_F);  // an all-zero O row needs no rescale
        m_used = mt;
        l *= alpha;
        if (kCorrect) best_raw = -CUDART_INF_F;   // restart under the new max (re-taken below)
      }
      lsum = stage_p(sr, xb, m_used == -CUDART_INF_F ? 0.f : m_used);
      if (half == 0) {
        reinterpret_cast<float*>(xb)[r] = alpha;
        const uint32_t fl = __any_sync(0xFFFFFFFFu, flag) ? 1u : 0u;
        if (lane == 0) reinterpret_cast<uint32_t*>(xb + 512)[wq] = fl;
      }
      fence_proxy_async_smem();
      named_bar_sync(kSoftmaxBar, kRowThreads);
    }
    l += lsum;
    if (half == 0 && r == 0) {
      // The O CTA's buffer `buf` is free once its PV product of tile j-2 is done.
      if (wait_or_abort<true>(sm, smem_u32(&sm.pempty[buf]), ((j >> 1) & 1) ^ 1, p, 8)) {
        MLA_TRACE_TILE(kTrCopy, j);
        bulk_copy_to_peer(xbuf0_remote + buf * kPBuf, xbuf0 + buf * kPBuf, xbytes,
                          buf ? pfull_remote1 : pfull_remote0);
        bulk_commit_group();
      } else {
        copy_failed = true;
      }
    }
    if (kCorrect && mraw > best_raw) {
      best_raw = mraw;
      best_j = j;
#pragma unroll
      for (int q4 = 0; q4 < 8; ++q4)
        *reinterpret_cast<uint4*>(top_scores + ((q4 ^ (r & 7)) << 4)) =
            make_uint4(sr[4 * q4], sr[4 * q4 + 1], sr[4 * q4 + 2], sr[4 * q4 + 3]);
    }
  }
  if (half == 0 && r == 0) bulk_wait_read<0>();
  if (wq == 0 && half == 0 && lane == 0) MLA_TRACE_SPAN(kSpLoopDone);
  if (!finished) return;
  if (half == 1) sm.xl[r] = l;
  if (kCorrect) {
    // This half's key: the first of its kept scores equal to its top score.
    int key = -1;
    if (best_raw != -CUDART_INF_F) {
      uint32_t v[32];
#pragma unroll
      for (int q4 = 0; q4 < 8; ++q4) {
        const uint4 x = *reinterpret_cast<const uint4*>(top_scores + ((q4 ^ (r & 7)) << 4));
        v[4 * q4] = x.x;
        v[4 * q4 + 1] = x.y;
        v[4 * q4 + 2] = x.z;
        v[4 * q4 + 3] = x.w;
      }
      int cb = -1;
#pragma unroll
      for (int c = 31; c >= 0; --c)
        if (__uint_as_float(v[c]) == best_raw) cb = c;
      if (cb >= 0) key = u.k0 + best_j * kKeys + 32 * half + cb;
    }
    sm.xbest[half][r] = make_float2(best_raw, __int_as_float(key));
  }
  if (named_bar_red_or(kSoftmaxBar, kRowThreads, copy_failed)) return;
  if (half == 0) {
    const uint32_t mlfull_remote = mapa_shared(smem_u32(&sm.mlfull), peer);
    st_async_v2(mapa_shared(smem_u32(&sm.ml[r]), peer), __float_as_uint(m_used),
                __float_as_uint(l + sm.xl[r]), mlfull_remote);
    if (kCorrect) {
      // The row's key: the larger of the halves' top scores (the first half on
      // ties), and the rounding error of its P, recomputed exactly as staged
      // (same fused multiply-add and exp2, with the final max).
      const float2 b0 = sm.xbest[0][r], b1 = sm.xbest[1][r];
      const bool h1 = b1.x > b0.x;
      const int key = __float_as_int(h1 ? b1.y : b0.y);
      float e = 0.f;
      if (key >= 0) {
        const float pc = ex2(fmaf(h1 ? b1.x : b0.x, a_eff, -m_used));
        e = pc - bf16lo_to_f32(pack_bf16x2(pc, pc));
      }
      st_async_v2(mapa_shared(smem_u32(&sm.corr[r]), peer), __float_as_uint(e),
                  static_cast<uint32_t>(key >= 0 ? key : 0), mlfull_remote);
    }
  }
}

// ============================================================ O CTA roles

// Value tile j into its ring slot.
__device__ __forceinline__ void o_issue(Smem& sm, const CUtensorMap* map_kv, int2 org, int j,
                                        int& n_issued) {
  const int slot = j & 1;
  const uint32_t full = smem_u32(&sm.vfull[slot]);
  mbar_arrive_expect_tx(full, kVTile);
  tma_load_4d(smem_u32(sm.ring) + slot * kVTile, map_kv, 0, org.x, 0, org.y, full);
  n_issued = j + 1;
}

// Thread 0 before the syncs: value tiles 0 and 1 (both slots start empty),
// unless the cache is a copy still being written by the preceding grid.
template <bool kPaged, bool kAfterCopy>
__device__ __forceinline__ void o_producer_start(Smem& sm, const Unit& u, const SplitParams& p,
                                                 const CUtensorMap* map_kv, int& n_issued) {
  tma_prefetch_desc(map_kv);
  if constexpr (!kAfterCopy) {
    for (int j = 0; j < 2 && j < u.ntiles; ++j)
      o_issue(sm, map_kv, tile_origin<kPaged>(p, u, u.k0 + j * kKeys), j, n_issued);
  }
}

template <bool kPaged, bool kAfterCopy>
__device__ __forceinline__ void o_producer(Smem& sm, const Unit& u, const SplitParams& p,
                                           const CUtensorMap* map_kv, int& n_issued) {
  if (kAfterCopy) grid_dependency_wait();   // the cache is the preceding grid's copy
  const int j0 = kAfterCopy ? 0 : 2;
  // (Block-table entries are read only for tiles of the slice.)
  int2 org0 = j0 < u.ntiles ? tile_origin<kPaged>(p, u, u.k0 + j0 * kKeys) : make_int2(0, 0);
  int2 org1 = j0 + 1 < u.ntiles ? tile_origin<kPaged>(p, u, u.k0 + (j0 + 1) * kKeys) : org0;
  for (int j = j0; j < u.ntiles; ++j) {
    const int2 org = org0;
    org0 = org1;
    if (j + 2 < u.ntiles) org1 = tile_origin<kPaged>(p, u, u.k0 + (j + 2) * kKeys);
    const int slot = j & 1;
    if (!wait_or_abort(sm, smem_u32(&sm.vempty[slot]), ((j >> 1) & 1) ^ 1, p, 9)) return;
    o_issue(sm, map_kv, org, j, n_issued);
    MLA_TRACE_TILE(kTrVLoad, j);
  }
}

__device__ __forceinline__ uint32_t p_tile_bytes(const Unit& u) {
  return kPHead + (u.two_term ? 2u : 1u) * kPTerm;
}

// Hand a command to the four O-CTA helper warps and wait until they are done.
// Called by the whole MMA warp.
__device__ __forceinline__ bool o_command(Smem& sm, uint32_t cmd, int& ncmd, const SplitParams& p,
                                          int lane) {
  if (lane == 0) {
    *reinterpret_cast<volatile uint32_t*>(&sm.cmd) = cmd;
    mbar_arrive(smem_u32(&sm.corrgo));
  }
  __syncwarp();
  const bool ok = warp_wait(sm, smem_u32(&sm.corrdone), ncmd & 1, p, 10);
  ++ncmd;
  return ok;
}

__device__ __forceinline__ void o_mma(Smem& sm, const Unit& u, const SplitParams& p,
                                      uint32_t tmem, int lane) {
  const uint32_t ring = smem_u32(sm.ring);
  const uint32_t pbytes = p_tile_bytes(u);
  int ncmd = 0;
  for (int j = 0; j < u.ntiles; ++j) {
    const int buf = j & 1;
    const int slot = j & 1;
    if (!warp_wait<true>(sm, smem_u32(&sm.pfull[buf]), (j >> 1) & 1, p, 11)) break;
    if (lane == 0) MLA_TRACE_TILE(kTrPFull, j);
    if (lane == 0 && j + 2 < u.ntiles) mbar_arrive_expect_tx(smem_u32(&sm.pfull[buf]), pbytes);
    fence_proxy_async_smem();
    if (!warp_wait(sm, smem_u32(&sm.vfull[slot]), (j >> 1) & 1, p, 12)) break;
    if (lane == 0) MLA_TRACE_TILE(kTrVFull, j);
    if (j == u.ntiles - 1 && u.zero_tail) {
      if (!o_command(sm, kCmdZeroTail | static_cast<uint32_t>(j), ncmd, p, lane)) break;
    }
    const uint8_t* xb = sm.ring + kPOffset + buf * kPBuf;
    const volatile uint32_t* fl = reinterpret_cast<const volatile uint32_t*>(xb + 512);
    const bool flagged = j > 0 && (fl[0] | fl[1] | fl[2] | fl[3]) != 0;
    if (flagged) {
      // Rows whose max grew: O must be scaled after PV(j-1) lands and before
      // PV(j) accumulates.  PV(j-2) is complete (its slot was refilled), so
      // the only pending phase of vempty[(j-1)&1] is PV(j-1)'s.
      if (!warp_wait(sm, smem_u32(&sm.vempty[(j - 1) & 1]), ((j - 1) >> 1) & 1, p, 13)) break;
      if (!o_command(sm, static_cast<uint32_t>(j), ncmd, p, lane)) break;
    }
    tc_fence_after();
    const uint32_t pb = ring + kPOffset + buf * kPBuf + kPHead;
    const uint32_t vb = ring + slot * kVTile;
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint64_t bdesc = sdesc_sw128(vb + 4 * h * kChunk + ks * 2048, kChunk, 1024);
        mma_ss_elect(tmem + 256 * h, sdesc_sw128(pb + ks * 32, 16, 1024), bdesc, kIdescPV,
                     (j > 0 || ks > 0) ? 1u : 0u);
        if (u.two_term)
          mma_ss_elect(tmem + 256 * h, sdesc_sw128(pb + kPTerm + ks * 32, 16, 1024), bdesc,
                       kIdescPV, 1u);
      }
    }
    mma_commit_elect(smem_u32(&sm.vempty[slot]));
    mma_commit_mc_elect(smem_u32(&sm.pempty[buf]), static_cast<uint16_t>(1u));  // rank 0 = S CTA
    if (lane == 0) MLA_TRACE_TILE(kTrPVIssued, j);
  }
  mma_commit_elect(smem_u32(&sm.odone));
  if (lane == 0) MLA_TRACE_SPAN(kSpLoopDone);
  if (lane == 0) {
    *reinterpret_cast<volatile uint32_t*>(&sm.cmd) = kCmdDone;
    mbar_arrive(smem_u32(&sm.corrgo));
  }
  __syncwarp();
}

// Cache row of key `key` of the unit's stream (576 bf16).
__device__ __forceinline__ const uint8_t* cache_row(const SplitParams& p, const Unit& u, int key) {
  const int2 o = p.block_table != nullptr ? tile_origin<true>(p, u, key) : tile_origin<false>(p, u, key);
  return p.kv + (static_cast<size_t>(o.y) * static_cast<size_t>(p.kv_rows) + static_cast<size_t>(o.x)) *
                    static_cast<size_t>((kDl + kDr) * 2);
}

// 8 value columns (one 16-byte load of bf16) times e, added to 8 fp32 bit patterns.
__device__ __forceinline__ void add_scaled_bf16x8(uint32_t* v, const uint4& x, float e) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    v[2 * k] = __float_as_uint(fmaf(e, __uint_as_float(w[k] << 16), __uint_as_float(v[2 * k])));
    v[2 * k + 1] =
        __float_as_uint(fmaf(e, __uint_as_float(w[k] & 0xFFFF0000u), __uint_as_float(v[2 * k + 1])));
  }
}

// Eight helper warps: warp 4+w and warp 8+w own tensor-memory lanes
// 32w..32w+31 (one output row per lane) and split the 512 accumulator columns.
// kCorrect (with `corr`): the epilogue adds the dominant key's P error times
// its value row to each row.  The value rows are read one 32-column block
// ahead, each warp's 32 rows together (four lanes per row, eight rows per
// load instruction, instead of 32 rows per instruction), and handed to the
// rows' threads through a per-warp shared-memory buffer.
template <bool kCorrect>
__device__ __forceinline__ void o_helpers(Smem& sm, const Unit& u, const SplitParams& p,
                                          const CUtensorMap* map_out, uint32_t tmem, int wq,
                                          int half, int lane, bool corr) {
  const int r = wq * 32 + lane;
  const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
  const uint32_t col0 = 256u * half;
  const int tid = half * 128 + wq * 32 + lane;
  int ncmd = 0;
  bool failed = false;   // kept instead of returning: the epilogue's barriers need every warp
  while (true) {
    if (!warp_wait(sm, smem_u32(&sm.corrgo), ncmd & 1, p, 14)) {
      failed = true;
      break;
    }
    ++ncmd;
    const uint32_t cmd = *reinterpret_cast<volatile uint32_t*>(&sm.cmd);
    if (cmd == kCmdDone) break;
    if (cmd & kCmdZeroTail) {
      // Cache rows at or beyond the slice end hold arbitrary values (even NaN);
      // P is 0 there but 0 * NaN would poison O, so clear them.
      const int j = static_cast<int>(cmd & 0xFFFF);
      const int z0 = u.k1 - (u.k0 + j * kKeys);
      const int nrow = kKeys - z0;
      uint8_t* tile = sm.ring + (j & 1) * kVTile;
      for (int it = tid; it < nrow * kVChunks * 8; it += kRowThreads) {
        const int q4 = it & 7;
        const int rr = z0 + ((it >> 3) % nrow);
        const int c = (it >> 3) / nrow;
        *reinterpret_cast<uint4*>(tile + c * kChunk + rr * 128 + q4 * 16) = make_uint4(0, 0, 0, 0);
      }
      fence_proxy_async_smem();
    } else {
      const int buf = static_cast<int>(cmd) & 1;
      const float alpha = reinterpret_cast<const float*>(sm.ring + kPOffset + buf * kPBuf)[r];
      tc_fence_after();
      if (__any_sync(0xFFFFFFFFu, alpha != 1.f)) {
        for (int cc = 0; cc < 8; ++cc) {
          uint32_t v[32];
          MLA_TMEM_LD_32x32b_X32(tmem + lane_base + col0 + 32 * cc, v);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
          MLA_TMEM_ST_32x32b_X32(tmem + lane_base + col0 + 32 * cc, v);
        }
        tmem_st_wait();
      }
      tc_fence_before();
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&sm.corrdone));
  }

  // ---- epilogue.  Each half of the helper warps owns 256 of the 512 output
  // columns: per 32-column block its 128 threads move their rows from tensor
  // memory into a 128-byte-swizzled [128 rows][32] staging block in the (now
  // idle) ring, and one thread writes the block with a TMA tensor store; rows
  // past this stream's q*H rows lie outside the tensor map and are not written.
  // The staging below uses named barriers: all 128 threads of a half decide
  // together whether the results are complete.
  const uint32_t bar = kEpilogueBar + static_cast<uint32_t>(half);
  bool ready;
  // kCorrect: this row's P error; rows of the warp that need a correction;
  // this lane's load slots: rows 8i + lane/4 (i = 0..3), 16 bytes at lane%4.
  float ce = 0.f;
  uint32_t need = 0u;
  const uint8_t* lrow[4] = {nullptr, nullptr, nullptr, nullptr};
  uint4 lx[4];
  if (kCorrect) {
    // (Waiting for the softmax results before the last PV, to start these
    // loads earlier, made the 33-draft, 16384-key call 2.2 us slower.)
    ready = !failed && warp_wait(sm, smem_u32(&sm.odone), 0, p, 15) &&
            warp_wait<true>(sm, smem_u32(&sm.mlfull), 0, p, 16);
    const uint8_t* vrow = nullptr;
    if (ready && corr) {
      const float2 cr = sm.corr[r];
      const float lrow_sum = sm.ml[r].y;
      if (r < u.valid_rows && fabsf(cr.x) > lrow_sum * exp2f(-kCorrSkipLog2)) {
        ce = cr.x;
        vrow = cache_row(p, u, static_cast<int>(__float_as_uint(cr.y))) + col0 * 2;
      }
    }
    need = __ballot_sync(0xFFFFFFFFu, ce != 0.f);
    if (need) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int rr = 8 * i + (lane >> 2);
        const uint64_t a = __shfl_sync(0xFFFFFFFFu, reinterpret_cast<uint64_t>(vrow), rr);
        lrow[i] = reinterpret_cast<const uint8_t*>(a) + 16 * (lane & 3);
        if ((need >> rr) & 1u) lx[i] = *reinterpret_cast<const uint4*>(lrow[i]);
      }
    }
  } else {
    ready = !failed && warp_wait(sm, smem_u32(&sm.odone), 0, p, 15) &&
            warp_wait<true>(sm, smem_u32(&sm.mlfull), 0, p, 16);
  }
  if (named_bar_red_or(bar, kRows, !ready)) return;
  if (tid == 0) MLA_TRACE_SPAN(kSpEpiReady);
  tc_fence_after();
  const float2 ml = sm.ml[r];
  const bool valid = r < u.valid_rows;
  const size_t grow = static_cast<size_t>(u.b) * u.rows_total + u.row0 + r;  // global row
  const bool direct = p.nsplit == 1;
  const float scale_out = direct ? (ml.y > 0.f ? 1.f / ml.y : 0.f) : 1.f;
  if (valid && half == 0) {
    if (direct)
      p.lse[grow] = ml.y > 0.f ? (ml.x + log2f(ml.y)) * 0.6931471805599453f : -CUDART_INF_F;
    else
      p.part_ml[static_cast<size_t>(u.sp) * p.B * u.rows_total + grow] = ml;
  }
  // Each warp stages and stores its own 32 rows (one [32 rows][32 columns]
  // TMA box per block), without waiting for the other warps; a warp whose rows
  // all lie past the stream's rows has nothing to store.
  if (32 * wq >= u.valid_rows) {
    tc_fence_before();
    return;
  }
  // Tensor-memory loads run one block ahead: block cc+1 is requested before
  // block cc is staged (tcgen05.wait::ld then waits for it at the next step).
  uint32_t va[32], vb[32];
  MLA_TMEM_LD_32x32b_X32(tmem + lane_base + col0, va);
  tmem_ld_wait();
#pragma unroll
  for (int cc = 0; cc < 8; ++cc) {
    const int slot = cc < kOutBufs ? cc : cc - kOutBufs;
    uint8_t* blk = sm.ring + (half * kOutBufs + slot) * kOutBlock;
    uint32_t* v = (cc & 1) ? vb : va;
    uint32_t* vn = (cc & 1) ? va : vb;
    if (cc + 1 < 8) MLA_TMEM_LD_32x32b_X32(tmem + lane_base + col0 + 32 * (cc + 1), vn);
    if (cc == kOutBufs) {
      // Blocks 0 and 1 reuse their staging buffers: this warp's stores must
      // have read them (at most kOutBufs - 2 of its groups still reading).
      if (lane == 0) bulk_wait_read<kOutBufs - 2>();
      __syncwarp();
    }
    if (kCorrect && need) {
      // Block cc of the warp's value rows: loaded lanes -> buffer (row-major,
      // 64 bytes a row, 16-byte units XOR-swizzled by (row >> 1) & 3, so that
      // neither side has bank conflicts) -> each row's own thread.
      uint8_t* wbuf = sm.ring + kCorrBufOffset + (half * 4 + wq) * kCorrWarpBytes;
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int rr = 8 * i + (lane >> 2);
        if ((need >> rr) & 1u)
          *reinterpret_cast<uint4*>(wbuf + rr * 64 + 16 * ((lane & 3) ^ ((rr >> 1) & 3))) = lx[i];
      }
      __syncwarp();
      uint4 c[4];
#pragma unroll
      for (int k = 0; k < 4; ++k)
        c[k] = *reinterpret_cast<const uint4*>(wbuf + lane * 64 + 16 * (k ^ ((lane >> 1) & 3)));
      if (cc + 1 < 8) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if ((need >> (8 * i + (lane >> 2))) & 1u)
            lx[i] = *reinterpret_cast<const uint4*>(lrow[i] + 64 * (cc + 1));
      }
      if (ce != 0.f) {
#pragma unroll
        for (int k = 0; k < 4; ++k) add_scaled_bf16x8(v + 8 * k, c[k], ce);
      }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e)
      *reinterpret_cast<float4*>(blk + r * 128 + ((e ^ (r & 7)) << 4)) =
          make_float4(__uint_as_float(v[4 * e]) * scale_out, __uint_as_float(v[4 * e + 1]) * scale_out,
                      __uint_as_float(v[4 * e + 2]) * scale_out, __uint_as_float(v[4 * e + 3]) * scale_out);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_4d(map_out, smem_u32(blk + wq * 32 * 128), static_cast<int>(col0) + 32 * cc,
                   u.row0 + 32 * wq, u.b, direct ? 0 : u.sp);
      bulk_commit_group();
    }
    if (cc + 1 < 8) tmem_ld_wait();
  }
  if (lane == 0) bulk_wait_all();
  if (wq == 0 && lane == 0 && half == 0) MLA_TRACE_SPAN(kSpEpiDone);
  tc_fence_before();
}

// ============================================================ kernel

// kDep: how the kernel follows the grid before it in the stream.
//   kDepNone: plain stream order.
//   kDepCopy: programmatic dependent of the grid that copied a paged cache into
//     a contiguous one; only the cache loads wait for that grid.
//   kDepPlan: programmatic dependent of the grid before it (plan_kernel, or
//     any other); every thread waits for that grid before reading anything.
//     (The plan is then ready; and a dependent launch starts sooner after the
//     grid before it ends than a plain one, with the same ordering.)
// (Separate instantiations: the wait instruction in the kernel cost ~0.7 us per
// call even when not executed.)  kCorrect: units that send one P term also
// remove their dominant keys' rounding (a separate instantiation too, so that
// the kernel for longer caches carries none of its code).
template <int kDep, bool kCorrect>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    verify_split_kernel(const __grid_constant__ CUtensorMap map_qn,
                        const __grid_constant__ CUtensorMap map_qr,
                        const __grid_constant__ CUtensorMap map_kvs0,
                        const __grid_constant__ CUtensorMap map_kvs1,
                        const __grid_constant__ CUtensorMap map_kvo,
                        const __grid_constant__ CUtensorMap map_out, const SplitParams p) {
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                      ~static_cast<uintptr_t>(1023));
  constexpr bool kAfterCopy = kDep == kDepCopy;
  if (kDep == kDepPlan) grid_dependency_wait();   // the preceding grid (the plan, if any) is done
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t role = cluster_ctarank();   // 0: scores + softmax, 1: PV accumulator
  if (tid == 0) MLA_TRACE_SPAN(kSpEntry);
  const Unit u = decode_unit(p);
  if (tid == 0) MLA_TRACE_SPAN(kSpDecoded);
  const bool corr = kCorrect && !u.two_term;   // one-term P plus the dominant-key correction
  // The slice merge is launched as a programmatic dependent of this grid; it
  // may be scheduled now and waits for this grid's completion itself.
  if (tid == 0) grid_launch_dependents();
  int n_issued[2] = {0, 0};   // thread 0: tiles issued per ring part (S) / value tiles (O)

  if (tid == 0) {
    // A stream length outside [q, Smax] is reported once: by the unit of its
    // slice 0 and row tile 0 (slice-major order), or by CTA 0 (ordered starts,
    // which give such a stream no slices).
    if (p.B > 1 && p.B <= kOrderedStreams) {
      if (blockIdx.x == 0)
        for (int b = 0; b < p.B; ++b)
          if (p.seq_lens[b] < p.q || p.seq_lens[b] > p.Smax) atomicOr(p.status, kStatusSeqLen);
    } else if ((u.S < p.q || u.S > p.Smax) && role == 0 && u.sp == 0 && u.rt == 0) {
      atomicOr(p.status, kStatusSeqLen);
    }
    for (int i = 0; i < kKSlots; ++i) {
      for (int part = 0; part < 2; ++part) {
        mbar_init(smem_u32(&sm.kfull[part][i]), 1);
        mbar_init(smem_u32(&sm.kempty[part][i]), 1);
      }
    }
    mbar_init(smem_u32(&sm.qfull), 1);
    mbar_init(smem_u32(&sm.qready), 8);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&sm.sfull[i]), 1);
      mbar_init(smem_u32(&sm.sempty[i]), 8);
      mbar_init(smem_u32(&sm.pempty[i]), 1);
      mbar_init(smem_u32(&sm.pfull[i]), 1);
      mbar_init(smem_u32(&sm.vfull[i]), 1);
      mbar_init(smem_u32(&sm.vempty[i]), 1);
    }
    mbar_init(smem_u32(&sm.odone), 1);
    mbar_init(smem_u32(&sm.corrgo), 1);
    mbar_init(smem_u32(&sm.corrdone), 8);
    mbar_init(smem_u32(&sm.mlfull), 1);
    mbar_init(smem_u32(&sm.drain), 1);

    sm.abort_flag = 0;
    sm.cmd = 0;
    if (role == 1 && !u.empty) {
      // P buffers 0 and 1 expect tiles 0 and 1; m/l expect one pair per row.
      mbar_arrive_expect_tx(smem_u32(&sm.pfull[0]), p_tile_bytes(u));
      if (u.ntiles > 1) mbar_arrive_expect_tx(smem_u32(&sm.pfull[1]), p_tile_bytes(u));
      mbar_arrive_expect_tx(smem_u32(&sm.mlfull), kRows * (corr ? 16 : 8));
    }
    fence_mbarrier_init_cluster();
    fence_proxy_async_smem();   // the initialised barriers, before TMA completes on them
  }
  // Arrive on the cluster barrier as soon as the barriers are initialised; the
  // wait below (before any access to the peer CTA) overlaps the first loads
  // and the tensor-memory allocation.
  cluster_arrive_relaxed();
  if (tid == 0) {
    if (!u.empty) {
      if (role == 0) {
        if (p.block_table != nullptr)
          s_producer_start<true, kAfterCopy>(sm, u, p, &map_qn, &map_qr, &map_kvs0, &map_kvs1, n_issued);
        else
          s_producer_start<false, kAfterCopy>(sm, u, p, &map_qn, &map_qr, &map_kvs0, &map_kvs1, n_issued);
      } else {
        tma_prefetch_desc(&map_out);
        if (p.block_table != nullptr)
          o_producer_start<true, kAfterCopy>(sm, u, p, &map_kvo, n_issued[0]);
        else
          o_producer_start<false, kAfterCopy>(sm, u, p, &map_kvo, n_issued[0]);
      }
    }
    MLA_TRACE_SPAN(kSpIssued);
  }
  if (!u.empty && warp == 2) {
    tmem_alloc(smem_u32(&sm.tmem_base), 512);
    tmem_relinquish();
    if (lane == 0) MLA_TRACE_SPAN(kSpAlloc);
  }
  tc_fence_before();
  __syncthreads();
  if (tid == 0) MLA_TRACE_SPAN(kSpCtaSync);
  cluster_wait();
  tc_fence_after();
  if (tid == 0) MLA_TRACE_SPAN(kSpSynced);
  const uint32_t tmem = sm.tmem_base;

  if (!u.empty) {
    if (role == 0) {
      if (warp == 0 && lane == 0) {
        if (p.block_table != nullptr)
          s_producer<true, kAfterCopy>(sm, u, p, &map_kvs0, &map_kvs1, n_issued);
        else
          s_producer<false, kAfterCopy>(sm, u, p, &map_kvs0, &map_kvs1, n_issued);
        mbar_wait(smem_u32(&sm.qfull), 0, kWaitNs / 2);
        drain_ring(sm.kfull[0], kKSlots, n_issued[0]);
        drain_ring(sm.kfull[1], kKSlots, n_issued[1]);
      } else if (warp == 1) {
        s_mma(sm, u, p, tmem);
        mma_commit_elect(smem_u32(&sm.drain));
        mbar_wait(smem_u32(&sm.drain), 0, kWaitNs);
        __syncwarp();
      } else if (warp >= 4) {
        if (u.two_term)
          s_softmax<true, false>(sm, u, p, tmem, warp & 3, (warp - 4) >> 2, lane);  // half = warp / 4 - 1
        else
          s_softmax<false, kCorrect>(sm, u, p, tmem, warp & 3, (warp - 4) >> 2, lane);
      }
    } else {
      if (warp == 0 && lane == 0) {
        if (p.block_table != nullptr)
          o_producer<true, kAfterCopy>(sm, u, p, &map_kvo, n_issued[0]);
        else
          o_producer<false, kAfterCopy>(sm, u, p, &map_kvo, n_issued[0]);
        drain_ring(sm.vfull, kVSlots, n_issued[0]);
      } else if (warp == 1) {
        o_mma(sm, u, p, tmem, lane);
        mma_commit_elect(smem_u32(&sm.drain));
        mbar_wait(smem_u32(&sm.drain), 0, kWaitNs);
        __syncwarp();
      } else if (warp >= 4) {
        o_helpers<kCorrect>(sm, u, p, &map_out, tmem, warp & 3, (warp - 4) >> 2, lane, corr);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (!u.empty && warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (tid == 0) MLA_TRACE_SPAN(kSpExit);
  cluster_sync_all();
}

}  // namespace mla
