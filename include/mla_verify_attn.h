/*
 * mla_verify_attn.h -- C ABI of the GB300 (sm_103a) absorbed-MLA verify-attention library.
 *
 * The operation (pages by title):
 *   "The Flash Attention Kernel That Had to Be Built: Designing sm_120 MLA
 *   Verify for Blackwell Consumer GPUs", section "What Input Knowledge Is
 *   Required to Understand This Message": each cache row is a 512-wide latent
 *   kv_c followed by a 64-wide decoupled RoPE key k_pe; a query row is an
 *   absorbed q_nope (512) and q_pe (64); score = q_nope . kv_c + q_pe . k_pe;
 *   the latent kv_c is also the value; a draft query sees the keys its
 *   candidate tree allows (paragraph "Speculative Decoding with DFlash"), the
 *   others are set to -inf before a softmax ("Flash Attention Algorithm").
 *   "The Decisive Microbench: When Theory Meets Silicon", section "The
 *   KV-Split Solution": the key range is split across thread blocks whose
 *   unnormalised partial states are merged by a second kernel with the
 *   online-softmax combine.
 *
 * For stream b, draft i < q_len, head h < H, with prefix_b = seq_lens[b] - q_len:
 *   visible(t) = t < prefix_b  or  (t < seq_lens[b] and bit (t - prefix_b) of mask row i)
 *   s_t        = scale * (sum_d q_nope[b,i,h,d] kv[b,t,d] + sum_e q_rope[b,i,h,e] kv[b,t,512+e])
 *   out[b,i,h] = sum_{visible t} softmax(s)_t * kv[b,t,0:512]
 *   lse[b,i,h] = ln sum_{visible t} exp(s_t)          (-inf and out = 0 if nothing is visible)
 *
 * Conventions for every entry point:
 *   - Device pointers unless stated otherwise; the caller owns all memory.
 *     The library allocates no device memory.
 *   - Calls are asynchronous on `stream`.  Argument errors are detected on the
 *     host and returned before anything is launched.  Problems only the GPU can
 *     see (a seq_lens value out of range, an internal wait that timed out) are
 *     recorded in a per-device status word read by mla_verify_attn_last_device_error.
 *   - bf16 tensors are passed as `const void*` holding IEEE bfloat16 values.
 *   - Results are deterministic for fixed inputs, Smax and device.
 *   - Precision: scores, softmax statistics and the output accumulate in fp32;
 *     the softmax weights enter the weights-times-values product in bf16 (the
 *     cache is bf16).  Their rounding is compensated where it would show:
 *     streams of up to 4096 keys (mla_verify_attn_set_two_term_max_keys moves
 *     the limit) send the weights as two bf16 terms; longer ones send one and
 *     add back the rounding error of each row's largest-score key.  Measured
 *     against an fp64 evaluation of the formula above: max |out error| <= 5e-4
 *     on N(0,1) inputs of every length and <= 6.4e-4 with a planted dominant
 *     key; a row whose weight several strong keys share keeps the rounding of
 *     all but the largest (3.0e-3 with 20 planted keys in one 126-tile slice,
 *     removed by two terms).  The tests hold it to 2e-3 (lse: 1e-3).
 *   - Stream capture: no entry point reads device memory on the host or
 *     synchronises inside mla_verify_attn.  Grid, split plan and tensor maps
 *     depend only on (B, q_len, H, Smax), the pointers and the device, so after
 *     the first call on a device (one-time setup: kernel attributes, occupancy
 *     query) a call may be captured into a CUDA graph; each replay reads the
 *     inputs' contents at replay time (seq_lens may change, within Smax).
 */
#ifndef MLA_VERIFY_ATTN_H
#define MLA_VERIFY_ATTN_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes (returned by the entry points and by the device status). */
enum mla_status {
  MLA_OK = 0,
  MLA_ERR_NULLPTR = -1,            /* a required pointer is NULL */
  MLA_ERR_SHAPE = -2,              /* B, q_len, H or Smax outside the supported range */
  MLA_ERR_ALIGN = -3,              /* a pointer misses its required alignment */
  MLA_ERR_WORKSPACE = -4,          /* workspace smaller than mla_verify_attn_workspace_size() */
  MLA_ERR_UNSUPPORTED_DEVICE = -5, /* current device is not sm_103 (GB300) or has no CUDA context */
  MLA_ERR_LAUNCH = -6,             /* a kernel launch or tensor-map creation failed */
  MLA_ERR_DEVICE_TIMEOUT = -7,     /* (device status) an internal pipeline wait gave up */
  MLA_ERR_SEQLEN = -8,             /* (device status) some seq_lens[b] outside [q_len, Smax] */
  MLA_ERR_ARG = -9,                /* any other invalid argument (e.g. non-finite scale) */
  MLA_ERR_PAGE = -10               /* (device status) a block-table entry outside the page pool */
};

/*
 * Bytes of scratch memory mla_verify_attn needs for these sizes on the
 * current device (0 when the key range is not split).  The value depends only
 * on (B, q_len, H, Smax) and the device's SM count.  Host-only; launches
 * nothing.  Returns 0 as well for invalid sizes (mla_verify_attn then reports
 * MLA_ERR_SHAPE).
 * Scratch holds the per-split partial states of the key-range split (page
 * "The Decisive Microbench: When Theory Meets Silicon", section "The KV-Split
 * Solution"): [nsplit][B*q_len*H][512] fp32 accumulators followed by
 * [nsplit][B*q_len*H][2] fp32 (running max, running sum), then, at a
 * 256-byte boundary, 256 bytes where calls with 2 to 32 streams keep the
 * slice plan the device chose from seq_lens (a smaller slice count than the
 * host's nsplit when the streams are ragged).
 */
size_t mla_verify_attn_workspace_size(int B, int q_len, int H, int Smax);

/*
 * Verify attention for B streams of q_len draft queries over a latent cache.
 *
 *   q_nope_abs  [B, q_len, H, 512] bf16, contiguous; 16-byte aligned.
 *   q_rope      [B, q_len, H, 64]  bf16, contiguous; 16-byte aligned.
 *   kv          [B, Smax, 576]     bf16, contiguous; row = latent (512) | rope (64);
 *               16-byte aligned.  Rows t < seq_lens[b] must be finite; rows at or
 *               beyond seq_lens[b] may hold anything (NaN included) and are never used.
 *   seq_lens    [B] int32: prefix_b + q_len, with q_len <= seq_lens[b] <= Smax.  The
 *               drafts' own cache rows are rows prefix_b .. seq_lens[b]-1.
 *   tree_mask   [B, q_len, ceil(q_len/32)] uint32; bit j (LSB first, word j/32) of row
 *               i set <=> draft i sees draft j.  Bits >= q_len are ignored.
 *   B >= 0, 1 <= q_len <= 64, 1 <= H, q_len*H*B < 2^31, 1 <= Smax < 2^24.
 *   scale       finite float multiplying every score (e.g. 1/sqrt(192)).
 *   out         [B, q_len, H, 512] fp32, normalised output; 16-byte aligned.
 *   lse         [B, q_len, H] fp32, natural log-sum-exp of the scaled scores; 4-byte aligned.
 *   workspace   device scratch of at least mla_verify_attn_workspace_size(B, q_len, H,
 *               Smax) bytes, 256-byte aligned (may be NULL when that size is 0).  Its
 *               contents on entry do not matter; it is not read after the call.
 *   stream      CUDA stream (0 = legacy default stream).
 *
 * Returns MLA_OK after enqueuing the work, or a negative mla_status with nothing
 * enqueued.  Calls that share a workspace must not overlap on the GPU.
 */
int mla_verify_attn(const void* q_nope_abs, const void* q_rope, const void* kv,
                    const int32_t* seq_lens, const uint32_t* tree_mask, int B, int q_len, int H,
                    int Smax, float scale, float* out, float* lse, void* workspace,
                    size_t workspace_bytes, cudaStream_t stream);

/*
 * mla_verify_attn over a paged cache.  The pages have no paged interface; they
 * name a paged cache (page_size 1, scattered rows) as the production layout
 * (page "The Moment of Truth: Benchmarking a Custom sm_120 Flash Attention
 * Kernel", section "Output Knowledge Created").  Pages of a multiple of 64 keys
 * are read in place with whole-tile TMA loads; for any other page size (1
 * included) a first kernel copies each stream's rows, in key order, into a
 * contiguous cache in the workspace, which the split kernel then reads (the
 * results equal the contiguous call's bit for bit).  The computation is that
 * of mla_verify_attn with
 *   kv[b, t, :] = kv_pool[block_table[b, t / page_size] * page_size + t % page_size, :]
 * i.e. key t of stream b lives in page block_table[b][t / page_size] of the pool.
 *
 *   kv_pool      [pool_rows, 576] bf16, rows = pages x page_size, 16-byte aligned.
 *                Rows of pages no stream refers to, and rows past a stream's
 *                seq_len, may hold anything (NaN included).
 *   pool_rows    rows in the pool: a multiple of page_size, < 2^31.
 *   block_table  [B, max_blocks] int32, 4-byte aligned: the page of each
 *                page_size-key block; entries past ceil(seq_lens[b] / page_size)
 *                are not read.  An entry outside [0, pool_rows / page_size) is
 *                reported as MLA_ERR_PAGE through the device status (that
 *                stream's results are then undefined).
 *   max_blocks   blocks per stream in block_table; Smax = max_blocks * page_size
 *                (< 2^24) bounds seq_lens[b].
 *   workspace    at least mla_verify_attn_paged_workspace_size(B, q_len, H,
 *                max_blocks, page_size) bytes (MLA_ERR_WORKSPACE otherwise).
 *   page_size    keys per page, >= 1 (MLA_ERR_SHAPE otherwise).  Multiples of 64
 *                are the fast path: a 64-key tile then never crosses a page.
 * All other arguments, results and errors as for mla_verify_attn.
 */
/*
 * Workspace bytes mla_verify_attn_paged needs on the current device: that of
 * mla_verify_attn for Smax = max_blocks * page_size, plus, when page_size is
 * not a multiple of 64, a contiguous copy of the cache (B * Smax * 1152 bytes,
 * after the partials at a 256-byte boundary).  0 for arguments the call would
 * reject (and, like mla_verify_attn_workspace_size, without a usable device).
 * Host-only.
 */
size_t mla_verify_attn_paged_workspace_size(int B, int q_len, int H, int max_blocks, int page_size);

int mla_verify_attn_paged(const void* q_nope_abs, const void* q_rope, const void* kv_pool,
                          long long pool_rows, const int32_t* block_table, int max_blocks,
                          int page_size, const int32_t* seq_lens, const uint32_t* tree_mask, int B,
                          int q_len, int H, float scale, float* out, float* lse, void* workspace,
                          size_t workspace_bytes, cudaStream_t stream);

/*
 * Synchronises `stream`, then returns and clears the current device's status
 * word: MLA_OK, MLA_ERR_SEQLEN, MLA_ERR_DEVICE_TIMEOUT or MLA_ERR_PAGE (the first recorded),
 * or MLA_ERR_LAUNCH if the synchronisation itself failed.  The word is shared
 * by all calls on the device since it was last read.
 * Every internal pipeline wait gives up after 2 s; the call's kernels then
 * unwind (waiting, again bounded, for their own copies in flight) and leave
 * the context usable.  mla_verify_attn_set_test_controls can make one work
 * unit withhold a cache load, to exercise that path.
 */
int mla_verify_attn_last_device_error(cudaStream_t stream);

/* Human-readable name of a status code (static string; never NULL). */
const char* mla_verify_attn_strerror(int status);

/*
 * The split plan mla_verify_attn uses, for inspection and tests (host-only):
 *   n_row_tiles  = ceil(q_len*H / 128) query-row tiles per stream,
 *   nsplit       = number of key-range slices (1 = no split, no scratch),
 *   chunk_tiles  = 64-key tiles per slice.
 * `max_clusters` is the number of 2-CTA clusters that fit on the device at
 * once (pass <= 0 to query the current device).  Honours a slice count forced
 * with mla_verify_attn_set_test_controls.  For 2 to 32 streams (count not
 * forced) this is the largest plan: a one-block planning kernel of the call
 * may choose fewer slices from the device's seq_lens, and the slices then
 * start longest first.
 * Returns MLA_OK or a status.
 */
int mla_verify_attn_plan(int B, int q_len, int H, int Smax, int max_clusters, int* n_row_tiles,
                         int* nsplit, int* chunk_tiles);

/*
 * Measurement aid; the pages have no counterpart.  While both events are
 * non-NULL, every mla_verify_attn call records `before_split` on its stream
 * just before the split kernel is launched and `after_split` just after it, so
 * cudaEventElapsedTime(before_split, after_split) is the split kernel's own
 * duration.  While they are set, the slice merge is launched without overlapping
 * the split kernel's tail.  NULL, NULL switches recording off.  The events are
 * the caller's (cudaEventCreate); the library only records them.  Set this only
 * while no other thread is calling into the library.  Returns MLA_OK, or
 * MLA_ERR_NULLPTR when exactly one event is NULL.
 */
int mla_verify_attn_set_timing_events(cudaEvent_t before_split, cudaEvent_t after_split);

/*
 * Precision control; the pages have no counterpart (their kernels keep P in
 * fp32).  V is bf16 in the cache and the tensor-core product takes P and V in
 * one type, so P is rounded to bf16.  Streams of at most `max_keys` keys
 * (seq_lens[b] <= max_keys) send P as two bf16 terms, hi + lo, and run the
 * P.V product once per term: outputs then match fp32 P to ~1e-5.  Longer
 * streams send one term and remove the rounding of each row's largest-score
 * key; a row whose weight several strong keys share keeps the others'
 * rounding (up to ~2^-9 of a value entry), which two terms remove at the cost
 * of the second product (the 64k-key, 9-draft call takes ~36 % longer).
 * Default 4096; 0 sends one term for every stream; INT_MAX two terms for every
 * stream.  Process-wide, for calls enqueued after it returns.  Returns MLA_OK,
 * or MLA_ERR_ARG for a negative `max_keys`.  Host-only.
 */
int mla_verify_attn_set_two_term_max_keys(int max_keys);

/*
 * Test controls; the pages have no counterpart.  Process-wide settings that
 * every later call reads (a relaxed atomic load per call, no environment
 * lookup), meant for the library's own tests:
 *   force_nsplit > 0  forces the number of key-range slices (at most one per
 *                     64-key tile of Smax), so that small inputs exercise the
 *                     split and merge path; it also changes what
 *                     mla_verify_attn_plan and the workspace sizes report,
 *                     and switches the device-side slice plan off.  0 restores
 *                     the library's own plan.
 *   stall != 0        makes work unit 0 of every later call withhold one of its
 *                     cache loads: its bounded waits run out after 2 s, the
 *                     call's kernels unwind and the device status reports
 *                     MLA_ERR_DEVICE_TIMEOUT.  0 switches this off.
 * Set these only while no call is being made from another thread.  Returns
 * MLA_OK, or MLA_ERR_ARG for a negative force_nsplit (nothing changes then).
 */
int mla_verify_attn_set_test_controls(int force_nsplit, int stall);

/*
 * mla_verify_attn without a caller-provided workspace.  This entry point has no
 * counterpart on the pages; it exists for callers that cannot allocate device
 * memory for scratch: code whose device memory is entirely pre-planned by its
 * own arena allocator (no way to hand out an extra buffer), latency-critical
 * loops where cudaMalloc/cudaFree would synchronise the device, and plain C
 * callers that link only this library and have no allocator of their own.
 *
 * Arguments and results are those of mla_verify_attn minus workspace and
 * workspace_bytes.  The key-split partials live instead in one fixed scratch
 * array of MLA_VERIFY_NOALLOC_SCRATCH_BYTES (32 MiB) compiled into this library
 * (a file-scope __device__ array: every GPU that loads the library holds it
 * until the process exits).  Calls whose partials need more than that return
 * MLA_ERR_WORKSPACE and enqueue nothing; use mla_verify_attn with a workspace
 * for them.  Nothing here calls cudaMalloc, cudaFree or any allocating routine.
 *
 * The first call on a device looks up the scratch array's device address
 * (cudaGetSymbolAddress) and caches it; make that first call before any stream
 * capture.  All calls on a device share that device's array, and it keeps the
 * last call's contents; nothing in it needs to start at zero (each call writes
 * every partial it later reads).  Calls on the same device that overlap on the
 * GPU (e.g. issued to two streams without ordering between them) race on the
 * array and may corrupt each other's results: order them, e.g. on one stream.
 */
#define MLA_VERIFY_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
int mla_verify_attn_noalloc(const void* q_nope_abs, const void* q_rope, const void* kv,
                            const int32_t* seq_lens, const uint32_t* tree_mask, int B, int q_len,
                            int H, int Smax, float scale, float* out, float* lse,
                            cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MLA_VERIFY_ATTN_H */
