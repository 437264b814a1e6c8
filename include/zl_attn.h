/*
 * zl_attn.h -- C ABI of the coalesced varlen attention library (libzl_attn.so).
 *
 * The operation is the attention call of the Coalesced Attention Engine in
 * Zellige, "Moldable Sequence Placement for Mixed Image-Video DiT Training"
 * (arXiv 2608.01150v1), §IV-D: all whole sequences of one GPU are packed into
 * ONE block-diagonal softmax-attention call that keeps the sequences separate
 * and returns outputs in input order, and shards of split long sequences run
 * alongside them.  Per sequence s and head h (full bidirectional attention,
 * §II-A, no mask):
 *
 *     S   = Q_s K_s^T * scale
 *     O_s = softmax(S) V_s            (row-wise softmax)
 *     LSE = log(sum_j exp(S_ij))      (natural log, one value per query row)
 *
 * Conventions shared by every entry point
 *   - Packed token layout.  Q/O are [Tq, H, d] and K/V are [Tk, H, d],
 *     row-major, d contiguous.  Sequence s owns query rows
 *     [cu_seqlens_q[s], cu_seqlens_q[s+1]) and key rows
 *     [cu_seqlens_k[s], cu_seqlens_k[s+1]).  Tq = cu_seqlens_q[num_seqs].
 *   - LSE buffers are head-major: lse[h * Tq + row], float32.
 *   - cu_seqlens_* and tile tables are HOST arrays (int32, num_seqs + 1
 *     entries, cu[0] = 0, non-decreasing).  All other pointers are DEVICE
 *     pointers of the current CUDA device, 16-byte aligned.
 *   - Every device buffer must hold the size the batch implies (Tq or Tk
 *     rows of H * d elements, H * Tq LSE values, the queried workspace
 *     bytes).  The library sees pointers, not allocations, so it cannot
 *     check this: a shorter buffer is read or written past its end.  The
 *     Python binding checks it against the tensors' shapes before each call.
 *   - The caller owns every buffer.  The library never calls cudaMalloc and
 *     allocates no device memory per call: scratch comes from the caller's
 *     `workspace` (zl_varlen_attn_bwd_static alone uses a fixed 64 MiB
 *     array in the library's device image instead, reserved on each device
 *     the library is loaded on).  On the host, calls build small std::vector
 *     tables (the schedule, the tile grid) and, while zl_profile_begin is
 *     active, create two CUDA events per launch.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and return after enqueue.  Arguments are validated on the host
 *     before anything is enqueued; an invalid call returns an error and leaves
 *     every output untouched.  Device-side faults surface through
 *     zl_sync_check().
 *   - Every entry point returns a zl_status (0 = success, < 0 = error) and
 *     never aborts the process.
 *   - Thread-safe.  Global state: a per-device cache of device attributes
 *     (SM count, the merge kernels' resident blocks per SM), a process-wide
 *     launch counter, the optional profiling hook (zl_profile_*), one device
 *     error word per kernel family (set by a kernel that gave up a wait, read
 *     and cleared by zl_sync_check) and zl_varlen_attn_bwd_static's scratch
 *     array.
 */
#ifndef ZL_ATTN_H
#define ZL_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ZL_OK = 0,
  ZL_EINVAL = -1,        /* malformed arguments (sizes, cu_seqlens, tile table) */
  ZL_EUNSUPPORTED = -2,  /* valid but not implemented (head_dim, dtype, mode)   */
  ZL_EALIGN = -3,        /* a device pointer is not 16-byte aligned             */
  ZL_EWORKSPACE = -4,    /* workspace missing or smaller than required          */
  ZL_ECUDA = -5,         /* a CUDA runtime/driver call failed                   */
  ZL_ETIMEOUT = -6,      /* a kernel gave up a bounded wait (reported by
                            zl_sync_check)                                      */
  ZL_ENODEVICE = -7      /* no usable sm_103 device                             */
} zl_status;

typedef enum {
  ZL_BF16 = 0,           /* bf16 inputs/outputs, float32 accumulation, tensor cores */
  ZL_FP32 = 1            /* float32 inputs/outputs, float32 SIMT arithmetic         */
} zl_dtype;

/*
 * One (query-chunk x head-range x KV-chunk) tile of a split sequence.
 * Zellige §IV-A gives every sequence a parallelism configuration (q, h, k):
 * split factors along the query axis (all-gather), the head axis (Ulysses) and
 * the key/value axis (ring), composable, (1, 1, 1) meaning whole; §IV-D runs
 * the shards of split sequences alongside whole ones, and §II-B / Table II
 * describe how a key-split sequence's attention is accumulated exactly from
 * its K/V blocks.  A tile is one shard of such a configuration.  Offsets are
 * relative to the sequence's own query and key ranges; heads are absolute.
 *
 * The tiles of a sequence must form a full grid: n_h_chunks x n_q_chunks x
 * n_kv_chunks tiles, one per (h_chunk, q_chunk, kv_chunk), whose head ranges
 * partition [0, H), whose query ranges partition the sequence's queries and
 * whose key ranges partition its keys (every tile with the same h_chunk has
 * the same head range, every tile with the same q_chunk the same query range,
 * every tile with the same kv_chunk the same key range; chunk ranges
 * contiguous, in chunk order, none empty).  A sequence listed in the tile
 * table is not also run whole.  A sequence with n_kv_chunks = 1 (a (q, h, 1)
 * configuration) needs no merge: its tiles write o and lse directly.
 *
 * h_len = 0 selects all H heads (h_start and h_chunk must then be 0), so a
 * zero-initialised head range means "not split by heads".
 */
typedef struct {
  int32_t seq;          /* index into cu_seqlens_q / cu_seqlens_k             */
  int32_t q_start;      /* first query of the chunk, relative to the sequence */
  int32_t q_len;        /* >= 1                                               */
  int32_t k_start;      /* first key of the chunk, relative to the sequence   */
  int32_t k_len;        /* >= 1                                               */
  int32_t q_chunk;      /* 0 .. n_q_chunks-1                                  */
  int32_t kv_chunk;     /* 0 .. n_kv_chunks-1: the partial slot it writes     */
  int32_t n_kv_chunks;  /* same for every tile of the sequence, 1 .. 64       */
  int32_t h_start;      /* first head of the tile's head range                */
  int32_t h_len;        /* heads in the range, 0 = all H heads                */
  int32_t h_chunk;      /* 0 .. n_h_chunks-1                                  */
} zl_tile_t;

/* Human-readable name of a status code (static string, never NULL). */
const char* zl_status_string(int32_t status);

/* ABI version of this header: (major << 16) | minor.  2.0: head-sharded
 * tiles; 2.1 adds ZL_FWD_BF16_PARTIALS, zl_lse_merge_ex and the schedule
 * queries (no existing entry changed). */
int32_t zl_version(void);

/*
 * Workspace needed by zl_varlen_attn_fwd for this batch, in bytes (0 when no
 * sequence is split along its keys).  It holds the float32 shard partials:
 * for the sequences with n_kv_chunks > 1 (in sequence order, R = sum of their
 * query lengths, P = largest n_kv_chunks) an O partial [P][R][H][d] and an
 * LSE partial [P][H][R], then the fused-merge arrival counters.  Under
 * ZL_FWD_BF16_PARTIALS the O partial holds bf16 elements in the first half
 * of the same region; the size is the same.
 * Same argument rules as zl_varlen_attn_fwd.  Writes the size to *bytes.
 */
zl_status zl_varlen_attn_fwd_workspace_size(
    const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int32_t num_seqs,
    int32_t num_heads, int32_t head_dim, const zl_tile_t* tiles, int32_t num_tiles,
    size_t* bytes);

/* One work item of the forward, as zl_varlen_attn_fwd_schedule reports it. */
typedef struct {
  int32_t launch;   /* forward launch of the call that runs it (a call with more
                       segments than one launch's parameters hold makes several) */
  int32_t seq;      /* sequence index                                          */
  int32_t tile;     /* index into the caller's tile table; -1: the whole sequence */
  int32_t head;     /* head                                                     */
  int32_t q_start;  /* first query row, relative to the sequence                */
  int32_t q_len;    /* query rows (up to 256 for ZL_BF16, 128 for ZL_FP32)      */
  int32_t k_start;  /* first key of the rows' key range, relative to the sequence */
  int32_t k_len;    /* keys every row of the item attends to                    */
} zl_work_item_t;

/*
 * The forward's work items for this batch, host only (no device work): the
 * tile scheduler of the Coalesced Attention Engine (Zellige §IV-D orders the
 * call's segments stably; §IV-C fills in decreasing price) as this library
 * applies it on one GPU.  Segments -- whole sequences and tiles -- are stably
 * ordered by decreasing key count (ties in input order); each splits into
 * items head by head, query block fastest; items run in this order, every SM
 * taking the next one when it is ready.  Writes the first max_items items to
 * `items` (host; may be NULL when max_items is 0) and their total to
 * *n_items.  Same argument rules and errors as zl_varlen_attn_fwd; `dtype`
 * selects the item size (256 query rows for ZL_BF16, 128 for ZL_FP32).
 */
zl_status zl_varlen_attn_fwd_schedule(
    const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int32_t num_seqs,
    int32_t num_heads, int32_t head_dim, int32_t dtype,
    const zl_tile_t* tiles, int32_t num_tiles,
    zl_work_item_t* items, int64_t max_items, int64_t* n_items);

/*
 * Forward of the coalesced block-diagonal attention (Zellige §IV-D).
 *
 * q [Tq,H,d], k/v [Tk,H,d]     inputs, dtype `dtype`, device
 * cu_seqlens_q, cu_seqlens_k   host, num_seqs + 1 entries each
 * num_heads H >= 1, head_dim d in {64, 128}
 * softmax_scale                > 0; pass 1/sqrt(d) for the usual scaling
 * tiles, num_tiles             host tile table (may be NULL when 0)
 * o [Tq,H,d]                   output, same dtype as the inputs
 * lse [H,Tq]                   output, float32, natural log
 * workspace                    device, >= zl_varlen_attn_fwd_workspace_size
 *
 * Whole sequences and every tile run in one persistent launch whose work
 * items (sequence-or-tile x head of its range x query block) are ordered
 * longest first, ties in input order; each SM takes the next item of that
 * order when it is ready for one, so the launch balances itself.  It shares
 * the GPU safely with concurrent launches on other streams.  Tiles of key-split sequences write
 * float32 partials into the workspace, and a merge launch per such sequence
 * (zl_lse_merge's kernel) then combines each query row's partials into o and
 * lse exactly; tiles of sequences split only by queries and heads write o and
 * lse directly.  A sequence with queries but no keys is rejected (ZL_EINVAL);
 * zero-length sequences are skipped.
 */
zl_status zl_varlen_attn_fwd(
    const void* q, const void* k, const void* v,
    const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int32_t num_seqs,
    int32_t num_heads, int32_t head_dim, int32_t dtype, float softmax_scale,
    const zl_tile_t* tiles, int32_t num_tiles,
    void* o, float* lse,
    void* workspace, size_t workspace_bytes, void* stream);

/* Flags of zl_varlen_attn_fwd_ex. */
enum {
  /* Merge the tile partials inside the forward launch: each tile counts
   * itself per (128-query block, head) after writing its partial, and the
   * tile that completes the set merges the partials of those rows (exact, as
   * zl_lse_merge; no waiting).  Saves the merge launch; measured slower than
   * the separate merge on the long-video batches, because the merging CTA's
   * tensor pipeline idles meanwhile.  bf16 only (ignored for ZL_FP32). */
  ZL_FWD_FUSED_MERGE = 1,
  /* Tiles of key-split sequences write their partial O rows in bf16 instead
   * of float32 (partial LSEs stay float32), which halves the bytes the
   * partials move through HBM, and the merge (separate or fused) reads them
   * back in bf16 and accumulates in float32.  Each partial row is rounded to
   * bf16 once before the merge: an added error of at most 2^-9 of each
   * partial's magnitude, inside the bf16 output's own rounding budget.  The
   * workspace is the same (its float32 size is an upper bound).  bf16 only
   * (ignored for ZL_FP32). */
  ZL_FWD_BF16_PARTIALS = 2
};

/*
 * zl_varlen_attn_fwd with option flags (a bitwise OR of ZL_FWD_* values; 0
 * gives exactly zl_varlen_attn_fwd).  Same arguments, layouts and workspace
 * otherwise.
 */
zl_status zl_varlen_attn_fwd_ex(
    const void* q, const void* k, const void* v,
    const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int32_t num_seqs,
    int32_t num_heads, int32_t head_dim, int32_t dtype, float softmax_scale,
    const zl_tile_t* tiles, int32_t num_tiles,
    void* o, float* lse,
    void* workspace, size_t workspace_bytes, void* stream, uint32_t flags);

/*
 * Exact merge of partial attention results over disjoint key sets: the
 * accumulation step of block-wise (ring / all-gather) attention in Zellige
 * §II-B and Table II.  For every query row r and head h:
 *
 *     lse = log(sum_p exp(lse_p))
 *     o   = sum_p exp(lse_p - lse) * o_p
 *
 * A row whose partials all have lse_p = -inf gets o = 0, lse = -inf.
 *
 * o_partial    device float32, part p row r head h at
 *              ((p * part_stride_rows + r) * H + h) * d
 * lse_partial  device float32, at (p * H + h) * part_stride_rows + r
 * n_parts      1 .. 64;  rows >= 0;  part_stride_rows >= rows
 * o            device, [rows][H][d] in out_dtype (ZL_BF16: round to nearest
 *              even; ZL_FP32)
 * lse          device float32, at h * lse_head_stride + r; lse_head_stride
 *              >= rows
 * Memory-bound; one launch.
 */
zl_status zl_lse_merge(
    const float* o_partial, const float* lse_partial, int32_t n_parts,
    int64_t rows, int32_t num_heads, int32_t head_dim, int64_t part_stride_rows,
    void* o, int32_t out_dtype, float* lse, int64_t lse_head_stride, void* stream);

/*
 * zl_lse_merge with the partial O rows in part_dtype: ZL_FP32 (exactly
 * zl_lse_merge) or ZL_BF16 (the same layout in bf16 elements, as written by
 * the forward under ZL_FWD_BF16_PARTIALS).  lse_partial stays float32 and
 * the accumulation is float32 either way.  Other part_dtype values give
 * ZL_EUNSUPPORTED; the other arguments and errors are zl_lse_merge's.
 */
zl_status zl_lse_merge_ex(
    const void* o_partial, int32_t part_dtype, const float* lse_partial, int32_t n_parts,
    int64_t rows, int32_t num_heads, int32_t head_dim, int64_t part_stride_rows,
    void* o, int32_t out_dtype, float* lse, int64_t lse_head_stride, void* stream);

/*
 * Workspace needed by zl_varlen_attn_bwd, in bytes: a float32 dQ accumulator
 * [Tq][H][d] and the float32 row term D = rowsum(dO * O) [H][Tq].
 */
zl_status zl_varlen_attn_bwd_workspace_size(
    const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int32_t num_seqs,
    int32_t num_heads, int32_t head_dim, size_t* bytes);

/* One work item of the backward, as zl_varlen_attn_bwd_schedule reports it. */
typedef struct {
  int32_t launch;   /* backward launch of the call that runs it                */
  int32_t seq;      /* sequence index                                          */
  int32_t head;     /* head                                                     */
  int32_t k_start;  /* first key of the item's key block, relative to the sequence */
  int32_t k_len;    /* keys of the block (up to 128)                            */
  int32_t q_len;    /* query rows the block visits: all of the sequence's       */
} zl_bwd_work_item_t;

/*
 * The backward's work items for this batch, host only (no device work).
 * The backward of a split sequence is the sum over its tiles, i.e. the
 * backward of the whole sequence, so every sequence runs whole; sequences
 * are stably ordered by decreasing query count (the rows each of their key
 * blocks visits), each splits into 128-key blocks head by head, key block
 * fastest, and the items run in this order, every SM taking the next one
 * when it is ready.  Writes the first max_items items to `items` (host; may
 * be NULL when max_items is 0) and their total to *n_items.  Same argument
 * rules and errors as zl_varlen_attn_bwd's batch description (cu_seqlens,
 * heads, head_dim, tiles).
 */
zl_status zl_varlen_attn_bwd_schedule(
    const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int32_t num_seqs,
    int32_t num_heads, int32_t head_dim, const zl_tile_t* tiles, int32_t num_tiles,
    zl_bwd_work_item_t* items, int64_t max_items, int64_t* n_items);

/*
 * Backward of zl_varlen_attn_fwd: the analytic gradient of
 * O = softmax(Q K^T * scale) V per sequence and head (the paper trains with
 * exact backward, §V-A; the formula is plain calculus):
 *
 *     P  = exp(S - LSE)      (recomputed from the forward's LSE)
 *     D  = rowsum(dO * O)
 *     dV = P^T dO,   dS = P * (dO V^T - D),
 *     dQ = scale * dS K,   dK = scale * dS^T Q
 *
 * q, k, v, o, dout    device, dtype `dtype` (ZL_BF16 only), layouts as above
 * lse                 device float32 [H][Tq] from the forward
 * tiles               the forward's tile table: the backward of a split
 *                     sequence sums the contributions of all of its tiles,
 *                     which equals the backward of the whole sequence, so it
 *                     is computed that way (validated, then run whole)
 * dq [Tq,H,d], dk/dv [Tk,H,d]   outputs, dtype `dtype`
 * workspace           device, >= zl_varlen_attn_bwd_workspace_size
 */
zl_status zl_varlen_attn_bwd(
    const void* q, const void* k, const void* v, const void* o, const float* lse,
    const void* dout,
    const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int32_t num_seqs,
    int32_t num_heads, int32_t head_dim, int32_t dtype, float softmax_scale,
    const zl_tile_t* tiles, int32_t num_tiles,
    void* dq, void* dk, void* dv,
    void* workspace, size_t workspace_bytes, void* stream);

/*
 * Backward that needs no workspace.  The paper has no counterpart to this
 * entry point; it exists for callers that cannot allocate device memory at
 * the moment they need a gradient: a plugin inside an engine that owns all
 * device memory and forbids allocation while it executes, code between
 * stream-capture begin and end, where a new allocation would not be part of
 * the captured work, or a process whose memory a pooling allocator has
 * reserved and that may not call it.
 *
 * Same operation, arguments and layouts as zl_varlen_attn_bwd with
 * dtype = ZL_BF16, minus the tile table (tiles do not change a backward's
 * result) and the workspace.  Its scratch (float32 dQ accumulator and D) is a
 * 64 MiB array in the library's device image, reserved on every GPU the
 * library is loaded on until the process exits.  Limit: Tq * H * d (rounded
 * up to a multiple of 64) + Tq * H <= 16,777,216 float32 values, e.g.
 * Tq <= 3,250 tokens at H = 40, d = 128; a larger batch returns
 * ZL_EWORKSPACE before any GPU work.  The caller still owns and passes every
 * input and output.
 *
 * The first call on each device (with that device current) looks up the
 * array's device address; make that first call before any stream capture.
 * All calls on a device share the array: calls whose kernels may overlap on
 * the GPU (unordered streams) race on it and give undefined results; calls on
 * one stream are safe.  Each call clears the accumulator it uses, so results
 * do not depend on earlier calls.  Allocates no device memory and creates
 * no CUDA objects: its launches count in zl_launch_count but are not timed
 * by zl_profile_*, whose events it would have to create.  Batch rules and errors are
 * zl_varlen_attn_bwd's (token bounds included), checked before the scratch
 * limit.
 */
zl_status zl_varlen_attn_bwd_static(
    const void* q, const void* k, const void* v, const void* o, const float* lse,
    const void* dout,
    const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int32_t num_seqs,
    int32_t num_heads, int32_t head_dim, float softmax_scale,
    void* dq, void* dk, void* dv, void* stream);

/*
 * Synchronizes `stream`, then reports (and clears) any error a kernel of this
 * library flagged on the current device: ZL_ETIMEOUT when a bounded wait
 * inside a kernel ran out (the kernel stopped early and its outputs are
 * undefined), ZL_ECUDA for a CUDA error.  ZL_OK otherwise.
 */
zl_status zl_sync_check(void* stream);

/*
 * Self-test of failure detection.  The pages have no counterpart; what it
 * exercises is the rule every kernel here follows: no wait is unbounded, a
 * wait that runs out records an error and ends the CTA's other roles, and the
 * kernel returns so that the context stays usable.  It enqueues one small
 * kernel whose wait on an mbarrier that nothing arrives on gives up after
 * limit_ns nanoseconds (1 .. 1e9; else ZL_EINVAL), while a second warp of
 * the same CTA, waiting with the kernels' own limit, must leave as soon as the
 * first one has given up.  No copy or MMA is in flight and no memory is
 * touched.  The next zl_sync_check(stream) returns ZL_ETIMEOUT (and clears
 * the record); work enqueued afterwards runs normally.
 */
zl_status zl_selftest_wait_timeout(uint64_t limit_ns, void* stream);

/* Number of kernel launches this library has enqueued in this process. */
int64_t zl_launch_count(void);

/*
 * Per-kernel timing, the single-GPU counterpart of the paper's Hardware
 * Profiler, which measures execution time per configuration (Zellige §IV-B).
 * Between zl_profile_begin() and zl_profile_end() every kernel this library
 * launches is bracketed by two CUDA events on its stream.  zl_profile_end()
 * waits for those events, writes one entry per kernel name (launch count and
 * summed device time) into `entries` (up to max_entries; *n_entries gets the
 * number written), releases the events and stops recording.  Recording is
 * process-wide; begin while already recording returns ZL_EINVAL.
 */
typedef struct {
  char name[32];
  int64_t launches;
  double total_ms;
} zl_profile_entry_t;

zl_status zl_profile_begin(void);
zl_status zl_profile_end(zl_profile_entry_t* entries, int32_t max_entries, int32_t* n_entries);

#ifdef __cplusplus
}
#endif

#endif /* ZL_ATTN_H */
