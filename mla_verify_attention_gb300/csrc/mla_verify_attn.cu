// Host side of the C ABI declared in include/mla_verify_attn.h: argument
// checks, the split plan, TMA tensor maps and the two launches (split kernel,
// then the merge of slice partials when the key range is split).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "mla_verify_attn.h"
#include "combine.cuh"
#include "verify_split.cuh"
#include "repack.cuh"
#include "planner.cuh"

namespace {

// Per-device status word (bits of mla::kStatus*), read and cleared by
// mla_verify_attn_last_device_error().
__device__ unsigned int g_mla_status;

constexpr int kMaxDevices = 64;
// Shortest slice (mla::kMinSliceTiles): a slice of a short stream still pays
// the unit's fixed cost (Q load, epilogue) and adds a partial to merge.
// Measured on tree9/chain9 shapes: 2-tile slices beat longer ones while all
// units fit one wave.
constexpr int kMinTilesPerSlice = mla::kMinSliceTiles;
// P precision.  Rounding P to one bf16 term (with the lazily kept row max)
// put errors up to 4.8e-3 into outputs of streams of 4105..32760 keys, and up
// to ~3e-3 into longer streams where one key carries much of a row's weight.
// Streams up to kTwoTermMaxKeys keys send P as hi + lo (their slices are short,
// and the second PV product is cheap there); longer ones send one term plus
// the correction of each row's dominant key (the kCorrect kernel).  The limit
// can be moved with mla_verify_attn_set_two_term_max_keys.
constexpr int kTwoTermMaxKeys = 4096;
constexpr size_t kSmemBytes = sizeof(mla::Smem) + 1024;   // + manual 1 KB alignment

struct DeviceInfo {
  bool ready = false;
  int status = MLA_ERR_UNSUPPORTED_DEVICE;
  int sms = 0;
  int max_clusters = 0;
  unsigned int* status_word = nullptr;
  PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
};

std::mutex g_mutex;
DeviceInfo g_devices[kMaxDevices];

// Events recorded around the split kernel (mla_verify_attn_set_timing_events).
cudaEvent_t g_timing_before = nullptr;
cudaEvent_t g_timing_after = nullptr;

// Test controls (mla_verify_attn_set_test_controls): a forced slice count
// (0 = the plan's own) and the stall of one work unit; plain loads per call.
std::atomic<int> g_force_nsplit{0};
std::atomic<int> g_test_stall{0};
// Longest stream that sends P as two terms (mla_verify_attn_set_two_term_max_keys).
std::atomic<int> g_two_term_max_keys{kTwoTermMaxKeys};

int device_info(DeviceInfo** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return MLA_ERR_UNSUPPORTED_DEVICE;
  }
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceInfo& d = g_devices[dev];
  if (!d.ready) {
    d.ready = true;
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      d.status = MLA_ERR_UNSUPPORTED_DEVICE;
    } else if (major != 10 || minor != 3) {
      d.status = MLA_ERR_UNSUPPORTED_DEVICE;   // the kernels are built for sm_103a only
    } else {
      d.sms = sms;
      d.status = MLA_OK;
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                           cudaEnableDefault, &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr)
        d.status = MLA_ERR_UNSUPPORTED_DEVICE;
      d.encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
      using SplitFn = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap,
                               CUtensorMap, mla::SplitParams);
      const SplitFn fns[6] = {mla::verify_split_kernel<mla::kDepNone, false>,
                              mla::verify_split_kernel<mla::kDepCopy, false>,
                              mla::verify_split_kernel<mla::kDepPlan, false>,
                              mla::verify_split_kernel<mla::kDepNone, true>,
                              mla::verify_split_kernel<mla::kDepCopy, true>,
                              mla::verify_split_kernel<mla::kDepPlan, true>};
      for (const SplitFn fn : fns)
        if (d.status == MLA_OK && cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                       static_cast<int>(kSmemBytes)) != cudaSuccess)
          d.status = MLA_ERR_LAUNCH;
      if (d.status == MLA_OK) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * sms, 1, 1);
        cfg.blockDim = dim3(mla::kThreads, 1, 1);
        cfg.dynamicSmemBytes = kSmemBytes;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, mla::verify_split_kernel<mla::kDepNone, false>, &cfg) != cudaSuccess ||
            n < 1)
          n = sms / 2;
        d.max_clusters = n;
        void* sym = nullptr;
        if (cudaGetSymbolAddress(&sym, g_mla_status) != cudaSuccess) d.status = MLA_ERR_LAUNCH;
        d.status_word = static_cast<unsigned int*>(sym);
      }
      cudaGetLastError();
    }
  }
  *out = &d;
  return d.status;
}

bool shape_ok(int B, int q, int H, int Smax) {
  if (B < 0 || q < 1 || q > 64 || H < 1 || Smax < 1 || Smax >= (1 << 24)) return false;
  const long long rows = static_cast<long long>(B) * q * H;
  return rows < (1LL << 31);
}

int plan(int B, int q, int H, int Smax, int max_clusters, int* n_rt, int* nsplit, int* chunk) {
  if (!shape_ok(B, q, H, Smax) || max_clusters < 1) return MLA_ERR_SHAPE;
  const int rows = q * H;
  const int nrt = (rows + mla::kRows - 1) / mla::kRows;
  const int tiles = (Smax + mla::kKeys - 1) / mla::kKeys;
  const long long base = static_cast<long long>(B > 0 ? B : 1) * nrt;
  long long ns;
  const long long forced = g_force_nsplit.load(std::memory_order_relaxed);
  int ct;
  if (forced > 0) {
    ns = forced < tiles ? forced : tiles;
    ct = static_cast<int>((tiles + ns - 1) / ns);
  } else {
    if (B <= 1) {
      ns = base >= max_clusters ? 1 : max_clusters / base;   // one wave of clusters
    } else {
      // Several streams (of unknown, possibly ragged lengths): about four
      // waves' worth of slices, so that long streams are cut up even when the
      // streams alone fill a wave; the device refines the count (planner.cuh).
      ns = (4LL * max_clusters + base - 1) / base;
    }
    ct = static_cast<int>((tiles + ns - 1) / ns);
    if (ct < kMinTilesPerSlice) ct = kMinTilesPerSlice;
  }
  if (ct > tiles) ct = tiles;
  ns = (tiles + ct - 1) / ct;
  *n_rt = nrt;
  *nsplit = static_cast<int>(ns);
  *chunk = ct;
  return MLA_OK;
}

// Split calls: [nsplit][B*q*H][512] fp32 accumulators, [nsplit][B*q*H] (max, sum)
// pairs, then (at a 256-byte boundary) 256 bytes for the device-side plan.
size_t plan_offset(int B, int q, int H, int nsplit) {
  const size_t n = static_cast<size_t>(B) * q * H;
  const size_t end = static_cast<size_t>(nsplit) * n * (512 * sizeof(float) + sizeof(float2));
  return (end + 255) & ~static_cast<size_t>(255);
}
size_t workspace_bytes_for(int B, int q, int H, int nsplit) {
  if (nsplit <= 1) return 0;
  return plan_offset(B, q, H, nsplit) + 256;
}

bool nsplit_forced() { return g_force_nsplit.load(std::memory_order_relaxed) > 0; }

// Calls whose slice count plan_kernel chooses from the stream lengths: split
// calls with 2 to 32 streams, unless the count is forced.
bool device_planned(int B, int nsplit) {
  return B >= 2 && B <= mla::kOrderedStreams && nsplit > 1 && !nsplit_forced();
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// A paged call whose pages are not whole 64-key tiles keeps, after the split
// partials in its workspace (at a 256-byte boundary), a contiguous copy of the
// cache: [B][Smax][576] bf16.
bool needs_copy(int page_size) { return page_size % mla::kKeys != 0; }
size_t copy_offset(size_t partial_bytes) { return (partial_bytes + 255) & ~static_cast<size_t>(255); }
size_t copy_bytes(int B, int Smax) { return static_cast<size_t>(B) * Smax * (576 * 2); }
bool paged_args_ok(int max_blocks, int page_size) {
  return page_size >= 1 && max_blocks >= 1 &&
         static_cast<long long>(max_blocks) * page_size < (1LL << 24);
}

int encode(DeviceInfo* d, CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims,
           const cuuint64_t* strides, const cuuint32_t* box,
           CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  const cuuint32_t elem[4] = {1, 1, 1, 1};
  const CUresult r = d->encode(map, dtype, rank, const_cast<void*>(base),
                               dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MLA_OK : MLA_ERR_LAUNCH;
}

}  // namespace

extern "C" {

const char* mla_verify_attn_strerror(int status) {
  switch (status) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_NULLPTR: return "MLA_ERR_NULLPTR: a required pointer is NULL";
    case MLA_ERR_SHAPE: return "MLA_ERR_SHAPE: B, q_len, H or Smax outside the supported range";
    case MLA_ERR_ALIGN: return "MLA_ERR_ALIGN: a pointer misses its required alignment";
    case MLA_ERR_WORKSPACE: return "MLA_ERR_WORKSPACE: workspace smaller than required";
    case MLA_ERR_UNSUPPORTED_DEVICE: return "MLA_ERR_UNSUPPORTED_DEVICE: current device is not sm_103";
    case MLA_ERR_LAUNCH: return "MLA_ERR_LAUNCH: kernel launch or tensor-map creation failed";
    case MLA_ERR_PAGE: return "MLA_ERR_PAGE: a block-table entry outside the page pool";
    case MLA_ERR_DEVICE_TIMEOUT: return "MLA_ERR_DEVICE_TIMEOUT: a device pipeline wait gave up";
    case MLA_ERR_SEQLEN: return "MLA_ERR_SEQLEN: seq_lens[b] outside [q_len, Smax]";
    case MLA_ERR_ARG: return "MLA_ERR_ARG: invalid argument";
    default: return "unknown mla_verify_attn status";
  }
}

int mla_verify_attn_plan(int B, int q_len, int H, int Smax, int max_clusters, int* n_row_tiles,
                         int* nsplit, int* chunk_tiles) {
  if (!n_row_tiles || !nsplit || !chunk_tiles) return MLA_ERR_NULLPTR;
  if (!shape_ok(B, q_len, H, Smax)) return MLA_ERR_SHAPE;
  if (max_clusters <= 0) {
    DeviceInfo* d = nullptr;
    const int st = device_info(&d);
    if (st != MLA_OK) return st;
    max_clusters = d->max_clusters;
  }
  return plan(B, q_len, H, Smax, max_clusters, n_row_tiles, nsplit, chunk_tiles);
}

size_t mla_verify_attn_workspace_size(int B, int q_len, int H, int Smax) {
  if (!shape_ok(B, q_len, H, Smax)) return 0;
  DeviceInfo* d = nullptr;
  if (device_info(&d) != MLA_OK) return 0;
  int nrt, ns, ct;
  if (plan(B, q_len, H, Smax, d->max_clusters, &nrt, &ns, &ct) != MLA_OK) return 0;
  return workspace_bytes_for(B, q_len, H, ns);
}

size_t mla_verify_attn_paged_workspace_size(int B, int q_len, int H, int max_blocks, int page_size) {
  if (!paged_args_ok(max_blocks, page_size)) return 0;
  const int Smax = max_blocks * page_size;
  const size_t partials = mla_verify_attn_workspace_size(B, q_len, H, Smax);
  if (!needs_copy(page_size)) return partials;
  if (!shape_ok(B, q_len, H, Smax)) return 0;
  return copy_offset(partials) + copy_bytes(B, Smax);
}

}  // extern "C"

namespace {

// One verify call: a contiguous cache (block_table == nullptr) or a paged one.
struct Call {
  const void* q_nope_abs;
  const void* q_rope;
  const void* kv;                 // [B][Smax][576] or the page pool [pool_rows][576]
  const int32_t* seq_lens;
  const uint32_t* tree_mask;
  int B, q_len, H, Smax;
  float scale;
  float* out;
  float* lse;
  void* workspace;
  size_t workspace_bytes;
  cudaStream_t stream;
  const int32_t* block_table;     // paged: [B][max_blocks]
  int max_blocks, page_size;
  long long pool_rows;
};

int run(const Call& c) {
  const void* q_nope_abs = c.q_nope_abs;
  const void* q_rope = c.q_rope;
  const int32_t* seq_lens = c.seq_lens;
  const uint32_t* tree_mask = c.tree_mask;
  const int B = c.B, q_len = c.q_len, H = c.H, Smax = c.Smax;
  const float scale = c.scale;
  float* out = c.out;
  float* lse = c.lse;
  void* workspace = c.workspace;
  const size_t workspace_bytes = c.workspace_bytes;
  cudaStream_t stream = c.stream;
  // Paged caches: pages of a multiple of 64 keys are read in place (TMA tiles
  // through the block table); others are first copied into the workspace.
  const bool copy = c.block_table != nullptr && needs_copy(c.page_size);
  const bool paged = c.block_table != nullptr && !copy;
  if (!shape_ok(B, q_len, H, Smax)) return MLA_ERR_SHAPE;
  if (!std::isfinite(scale)) return MLA_ERR_ARG;
  if (B == 0) return MLA_OK;
  if (!q_nope_abs || !q_rope || !c.kv || !seq_lens || !tree_mask || !out || !lse)
    return MLA_ERR_NULLPTR;
  if (!aligned(q_nope_abs, 16) || !aligned(q_rope, 16) || !aligned(c.kv, 16) || !aligned(out, 16) ||
      !aligned(lse, 4) || !aligned(seq_lens, 4) || !aligned(tree_mask, 4) ||
      (workspace && !aligned(workspace, 256)))
    return MLA_ERR_ALIGN;

  DeviceInfo* d = nullptr;
  int st = device_info(&d);
  if (st != MLA_OK) return st;
  int nrt, ns, ct;
  st = plan(B, q_len, H, Smax, d->max_clusters, &nrt, &ns, &ct);
  if (st != MLA_OK) return st;
  const size_t partials = workspace_bytes_for(B, q_len, H, ns);
  const size_t need = copy ? copy_offset(partials) + copy_bytes(B, Smax) : partials;
  if (need > 0 && (!workspace || workspace_bytes < need)) return MLA_ERR_WORKSPACE;
  // The cache the split kernel reads: the caller's, or the contiguous copy.
  const void* kv = copy ? static_cast<const void*>(static_cast<char*>(workspace) + copy_offset(partials))
                        : c.kv;

  const long long rows = static_cast<long long>(B) * q_len * H;
  // Tensor maps.  Each cache (and q_nope) row of 576 (512) bf16 is viewed as
  // chunks of 64 dims; the chunk index is its own dimension (stride 128 B) so
  // that one TMA box brings [chunk][row][64 dims] into shared memory, i.e. a
  // whole 64-key tile per copy, in the 128-byte-swizzled layout the MMAs read.
  CUtensorMap map_qn, map_qr, map_kvs0, map_kvs1, map_kvo;
  {
    const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(rows), 8};
    const cuuint64_t strides[2] = {512 * 2, 64 * 2};
    const cuuint32_t box[3] = {64, mla::kRows, 8};
    if (encode(d, &map_qn, q_nope_abs, 3, dims, strides, box) != MLA_OK) return MLA_ERR_LAUNCH;
  }
  {
    const cuuint64_t dims[2] = {64, static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {64 * 2};
    const cuuint32_t box[2] = {64, mla::kRows};
    if (encode(d, &map_qr, q_rope, 2, dims, strides, box) != MLA_OK) return MLA_ERR_LAUNCH;
  }
  {
    // Rows of the cache: [B][Smax] (contiguous) or the page pool (paged, one "stream").
    const cuuint64_t nrow = paged ? static_cast<cuuint64_t>(c.pool_rows) : static_cast<cuuint64_t>(Smax);
    const cuuint64_t dims[4] = {64, nrow, 9, static_cast<cuuint64_t>(paged ? 1 : B)};
    const cuuint64_t strides[3] = {576 * 2, 64 * 2, nrow * 576 * 2};
    // S CTA: a key tile's chunks 0..4 and 5..8 as two boxes; O CTA: chunks 0..7.
    const cuuint32_t box_s0[4] = {64, mla::kKeys, mla::kKSplit, 1};
    const cuuint32_t box_s1[4] = {64, mla::kKeys, 9 - mla::kKSplit, 1};
    const cuuint32_t box_o[4] = {64, mla::kKeys, 8, 1};
    if (encode(d, &map_kvs0, kv, 4, dims, strides, box_s0) != MLA_OK) return MLA_ERR_LAUNCH;
    if (encode(d, &map_kvs1, kv, 4, dims, strides, box_s1) != MLA_OK) return MLA_ERR_LAUNCH;
    if (encode(d, &map_kvo, kv, 4, dims, strides, box_o) != MLA_OK) return MLA_ERR_LAUNCH;
  }
  // Results: fp32 [slice][stream][q*H rows][512] (the slice partials, or `out`
  // itself when the key range is not split), stored in [32 rows][32] boxes
  // (one per warp of the epilogue).
  float* const part_o = static_cast<float*>(workspace);
  CUtensorMap map_out;
  {
    const long long rps = static_cast<long long>(q_len) * H;   // rows per stream
    const cuuint64_t dims[4] = {512, static_cast<cuuint64_t>(rps), static_cast<cuuint64_t>(B),
                                static_cast<cuuint64_t>(ns)};
    const cuuint64_t strides[3] = {512 * 4, static_cast<cuuint64_t>(rps) * 512 * 4,
                                   static_cast<cuuint64_t>(rows) * 512 * 4};
    const cuuint32_t box[4] = {32, 32, 1, 1};
    if (encode(d, &map_out, ns > 1 ? static_cast<void*>(part_o) : static_cast<void*>(out), 4, dims,
               strides, box, CU_TENSOR_MAP_DATA_TYPE_FLOAT32) != MLA_OK)
      return MLA_ERR_LAUNCH;
  }

  mla::SplitParams p;
  p.seq_lens = seq_lens;
  p.mask = tree_mask;
  p.lse = lse;
  p.part_ml = ns > 1 ? reinterpret_cast<float2*>(static_cast<char*>(workspace) +
                                                 static_cast<size_t>(ns) * rows * 512 * 4)
                     : nullptr;
  p.status = d->status_word;
  p.B = B;
  p.q = q_len;
  p.H = H;
  p.Smax = Smax;
  p.n_rt = nrt;
  p.nsplit = ns;
  p.chunk_tiles = ct;
  const bool planned = device_planned(B, ns);
  int* const plan_dev = planned ? reinterpret_cast<int*>(static_cast<char*>(workspace) +
                                                         plan_offset(B, q_len, H, ns))
                                : nullptr;
  p.plan = plan_dev;
  const bool corrected = true;
  const int two_term_max_keys = g_two_term_max_keys.load(std::memory_order_relaxed);
  p.two_term_max_keys = two_term_max_keys;
  p.kv = static_cast<const uint8_t*>(kv);
  p.kv_rows = paged ? c.pool_rows : static_cast<long long>(Smax);
  p.test_stall = g_test_stall.load(std::memory_order_relaxed) != 0 ? 1 : 0;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.block_table = paged ? c.block_table : nullptr;
  p.max_blocks = paged ? c.max_blocks : 0;
  p.page_size = paged ? c.page_size : 0;
  p.pool_pages = paged ? static_cast<int>(c.pool_rows / c.page_size) : 0;
  const long long units = static_cast<long long>(B) * nrt * ns;
  if (2 * units >= (1LL << 31)) return MLA_ERR_SHAPE;
  if (copy) {
    mla::RepackParams rp;
    rp.pool = static_cast<const uint8_t*>(c.kv);
    rp.block_table = c.block_table;
    rp.seq_lens = seq_lens;
    rp.dst = static_cast<uint8_t*>(const_cast<void*>(kv));
    rp.status = d->status_word;
    rp.B = B;
    rp.max_blocks = c.max_blocks;
    rp.page_size = c.page_size;
    rp.pool_pages = static_cast<int>(c.pool_rows / c.page_size);
    rp.Smax = Smax;
    // A programmatic dependent of the grid before it (it waits for that grid first).
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((Smax + mla::kKeys - 1) / mla::kKeys, B < 65535 ? B : 65535, 1);
    cfg.blockDim = dim3(mla::kRepackThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, mla::repack_kernel, rp) != cudaSuccess) {
      cudaGetLastError();
      return MLA_ERR_LAUNCH;
    }
  }
  if (planned) {
    mla::PlanParams pp;
    pp.seq_lens = seq_lens;
    pp.plan = plan_dev;
    pp.B = B;
    pp.q = q_len;
    pp.Smax = Smax;
    pp.n_rt = nrt;
    pp.nsplit_max = ns;
    pp.min_chunk = kMinTilesPerSlice;
    pp.slots = d->max_clusters;
    pp.two_term_max_keys = two_term_max_keys;
    const int ncand = ns < mla::kPlanMaxCandidates ? ns : mla::kPlanMaxCandidates;
    // A programmatic dependent of the grid before it (it waits for that grid
    // first), so that its launch overlaps that grid's end.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(32 * ncand), 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, mla::plan_kernel, pp) != cudaSuccess) {
      cudaGetLastError();
      return MLA_ERR_LAUNCH;
    }
  }
  const bool timing = g_timing_before != nullptr;
  // The split kernel is a programmatic dependent of the grid before it: of
  // the cache copy (prologue overlapped, cache loads wait for the copy), or of
  // whatever grid precedes the call, the planner included (every thread waits
  // for that grid before reading anything, so the ordering is that of the
  // stream; launched this way the kernel starts ~2 us sooner after the grid
  // before it ends).  Not while the timing events are recorded between the
  // launches.
  // (With a plan, the planner runs after the copy and is the grid before.)
  const int dep = timing ? mla::kDepNone : (copy && !planned ? mla::kDepCopy : mla::kDepPlan);
  if (timing && cudaEventRecord(g_timing_before, stream) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_LAUNCH;
  }
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(2 * units), 1, 1);
    cfg.blockDim = dim3(mla::kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = dep != mla::kDepNone ? 1 : 0;
    using SplitFn = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap,
                             CUtensorMap, mla::SplitParams);
    const SplitFn fns[2][3] = {{mla::verify_split_kernel<mla::kDepNone, false>,
                                mla::verify_split_kernel<mla::kDepCopy, false>,
                                mla::verify_split_kernel<mla::kDepPlan, false>},
                               {mla::verify_split_kernel<mla::kDepNone, true>,
                                mla::verify_split_kernel<mla::kDepCopy, true>,
                                mla::verify_split_kernel<mla::kDepPlan, true>}};
    const SplitFn fn = fns[corrected ? 1 : 0][dep];
    if (cudaLaunchKernelEx(&cfg, fn, map_qn, map_qr, map_kvs0, map_kvs1, map_kvo, map_out, p) !=
        cudaSuccess) {
      cudaGetLastError();
      return MLA_ERR_LAUNCH;
    }
  }
  if (timing && cudaEventRecord(g_timing_after, stream) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_LAUNCH;
  }
  if (ns > 1) {
    mla::CombineParams c;
    c.part_o = part_o;
    c.part_ml = p.part_ml;
    c.seq_lens = seq_lens;
    c.out = out;
    c.lse = lse;
    c.N = static_cast<int>(rows);
    c.rows_per_stream = q_len * H;
    c.q = q_len;
    c.Smax = Smax;
    c.nsplit = ns;
    c.chunk_keys = ct * mla::kKeys;
    c.plan = plan_dev;
    // Programmatic dependent launch: the merge blocks may be scheduled while
    // the split kernel drains and wait (griddepcontrol.wait) for its results.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(rows), 1, 1);
    cfg.blockDim = dim3(128, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = timing ? 0 : 1;   // an event between the launches: plain ordering
    // Slices per load batch: 16 while all rows fit one wave at four blocks per
    // SM, else 8 (more resident rows; batches are merged online).
    const int nb = ns <= 4 ? 4 : ((ns <= 8 || rows > 4LL * d->sms) ? 8 : 16);
    // Few rows and many slices (e.g. 8 or 16 heads over a long stream): the
    // slices of a row are shared by groups of threads.  While four blocks of
    // 128 columns per row fit one wave (two per SM), sixteen groups per block
    // (one round of loads for up to 96 slices: H = 8 at 64k keys 33.7 -> 31.1
    // us/call); otherwise one block per row of four 128-thread groups (at 16
    // heads the column split took 2 waves and was 1.8 us slower).
    const bool grouped = ns > 16 && rows <= d->sms;
    const bool cols = grouped && 4 * rows <= 2LL * d->sms;
    if (cols) {
      cfg.gridDim = dim3(static_cast<unsigned>(rows), 4, 1);
      cfg.blockDim = dim3(16 * 32, 1, 1);
    } else if (grouped) {
      cfg.blockDim = dim3(4 * 128, 1, 1);
    }
    if (cudaLaunchKernelEx(&cfg, cols ? mla::combine_cols_kernel<6, 16, 4>
                                 : grouped ? mla::combine_kernel<16, 4>
                                 : (nb == 4 ? mla::combine_kernel<4, 1>
                                            : (nb == 8 ? mla::combine_kernel<8, 1> : mla::combine_kernel<16, 1>)),
                           c) != cudaSuccess) {
      cudaGetLastError();
      return MLA_ERR_LAUNCH;
    }
  }
  return MLA_OK;
}

}  // namespace

extern "C" {

int mla_verify_attn(const void* q_nope_abs, const void* q_rope, const void* kv,
                    const int32_t* seq_lens, const uint32_t* tree_mask, int B, int q_len, int H,
                    int Smax, float scale, float* out, float* lse, void* workspace,
                    size_t workspace_bytes, cudaStream_t stream) {
  Call c{q_nope_abs, q_rope, kv, seq_lens, tree_mask, B, q_len, H, Smax, scale, out, lse,
         workspace, workspace_bytes, stream, nullptr, 0, 0, 0};
  return run(c);
}

int mla_verify_attn_paged(const void* q_nope_abs, const void* q_rope, const void* kv_pool,
                          long long pool_rows, const int32_t* block_table, int max_blocks,
                          int page_size, const int32_t* seq_lens, const uint32_t* tree_mask, int B,
                          int q_len, int H, float scale, float* out, float* lse, void* workspace,
                          size_t workspace_bytes, cudaStream_t stream) {
  if (!paged_args_ok(max_blocks, page_size) || pool_rows < 1 || pool_rows % page_size != 0 ||
      pool_rows >= (1LL << 31))
    return MLA_ERR_SHAPE;
  if (B > 0 && (!block_table || !kv_pool)) return MLA_ERR_NULLPTR;
  if (block_table && !aligned(block_table, 4)) return MLA_ERR_ALIGN;
  Call c{q_nope_abs, q_rope, kv_pool, seq_lens, tree_mask, B, q_len, H, max_blocks * page_size,
         scale, out, lse, workspace, workspace_bytes, stream, block_table, max_blocks, page_size,
         pool_rows};
  return run(c);
}

int mla_verify_attn_set_timing_events(cudaEvent_t before_split, cudaEvent_t after_split) {
  if ((before_split == nullptr) != (after_split == nullptr)) return MLA_ERR_NULLPTR;
  g_timing_before = before_split;
  g_timing_after = after_split;
  return MLA_OK;
}

#ifdef MLA_TRACE
// Trace builds only (not part of the ABI): copies the split kernel's timeline
// buffers of the current device to the host and clears them.
int mla_verify_attn_trace_read(unsigned long long* tiles, unsigned long long* spans) {
  if (cudaDeviceSynchronize() != cudaSuccess) return MLA_ERR_LAUNCH;
  if (cudaMemcpyFromSymbol(tiles, mla::g_trace_tiles, sizeof(mla::g_trace_tiles)) != cudaSuccess ||
      cudaMemcpyFromSymbol(spans, mla::g_trace_spans, sizeof(mla::g_trace_spans)) != cudaSuccess)
    return MLA_ERR_LAUNCH;
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, mla::g_trace_tiles) != cudaSuccess ||
      cudaMemset(p, 0, sizeof(mla::g_trace_tiles)) != cudaSuccess ||
      cudaGetSymbolAddress(&p, mla::g_trace_spans) != cudaSuccess ||
      cudaMemset(p, 0, sizeof(mla::g_trace_spans)) != cudaSuccess)
    return MLA_ERR_LAUNCH;
  return MLA_OK;
}
#endif

int mla_verify_attn_set_two_term_max_keys(int max_keys) {
  if (max_keys < 0) return MLA_ERR_ARG;
  g_two_term_max_keys.store(max_keys, std::memory_order_relaxed);
  return MLA_OK;
}

int mla_verify_attn_set_test_controls(int force_nsplit, int stall) {
  if (force_nsplit < 0) return MLA_ERR_ARG;
  g_force_nsplit.store(force_nsplit, std::memory_order_relaxed);
  g_test_stall.store(stall != 0 ? 1 : 0, std::memory_order_relaxed);
  return MLA_OK;
}

int mla_verify_attn_last_device_error(cudaStream_t stream) {
  DeviceInfo* d = nullptr;
  const int st = device_info(&d);
  if (st != MLA_OK) return st;
  if (cudaStreamSynchronize(stream) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_LAUNCH;
  }
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_mla_status, sizeof v) != cudaSuccess) return MLA_ERR_LAUNCH;
  const unsigned int zero = 0;
  if (v != 0 && cudaMemcpyToSymbol(g_mla_status, &zero, sizeof zero) != cudaSuccess)
    return MLA_ERR_LAUNCH;
  if (v & mla::kStatusSeqLen) return MLA_ERR_SEQLEN;
  if (v & mla::kStatusTimeout) return MLA_ERR_DEVICE_TIMEOUT;
  if (v & mla::kStatusPage) return MLA_ERR_PAGE;
  return MLA_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Scratch-free variant (declared in mla_verify_attn.h): for callers that cannot
// allocate device memory, the key-split partials go to a fixed array compiled
// into this library instead of a caller-provided workspace.
namespace {

// One copy per device that loads the library, held until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[MLA_VERIFY_NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mutex;
void* g_noalloc_addr[kMaxDevices];   // device address of g_noalloc_scratch, per device

}  // namespace

extern "C" int mla_verify_attn_noalloc(const void* q_nope_abs, const void* q_rope, const void* kv,
                                       const int32_t* seq_lens, const uint32_t* tree_mask, int B,
                                       int q_len, int H, int Smax, float scale, float* out,
                                       float* lse, cudaStream_t stream) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return MLA_ERR_UNSUPPORTED_DEVICE;
  }
  void* scratch = nullptr;
  {
    // First call on this device (which must be current): look up the array's
    // device address once; host code cannot use the symbol itself.
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (g_noalloc_addr[dev] == nullptr) {
      void* addr = nullptr;
      if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || addr == nullptr) {
        cudaGetLastError();
        return MLA_ERR_UNSUPPORTED_DEVICE;
      }
      g_noalloc_addr[dev] = addr;
    }
    scratch = g_noalloc_addr[dev];
  }
  // Invalid shapes report 0 here and are rejected by mla_verify_attn below.
  if (mla_verify_attn_workspace_size(B, q_len, H, Smax) > MLA_VERIFY_NOALLOC_SCRATCH_BYTES)
    return MLA_ERR_WORKSPACE;
  return mla_verify_attn(q_nope_abs, q_rope, kv, seq_lens, tree_mask, B, q_len, H, Smax, scale,
                         out, lse, scratch, MLA_VERIFY_NOALLOC_SCRATCH_BYTES, stream);
}
