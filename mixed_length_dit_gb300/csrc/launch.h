// Internal interface between the host library (zl_host.cpp) and the kernel
// translation units.  Not part of the public C ABI.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace zl {

// Query rows per work item and keys per inner block of the tensor-core
// kernels.  One 128-row query block maps onto the 128 TMEM lanes.
constexpr int kBlockM = 128;
constexpr int kBlockN = 128;

// Query rows per work item of the tensor-core forward: two 128-row tiles
// that share every K/V tile.
constexpr int kFwdRowsPerItem = 2 * kBlockM;

// Work segments passed by value in one launch (kernel parameter space).
constexpr int kMaxSegs = 640;

// One segment of forward work: a whole sequence or one shard tile.  Its work
// items are (head of [h0, h0 + nh), query block of rows_per_item rows) pairs,
// numbered from item0 with the query block fastest.
struct FwdSeg {
  int32_t q_row0;    // packed row of the segment's first query
  int32_t k_row0;    // packed row of the segment's first key
  int32_t q_len;     // >= 1
  int32_t k_len;     // >= 1
  int32_t out_row0;  // slot < 0: row in o/lse; else row in the partial slot
  int32_t slot;      // -1: writes o/lse directly, else the partial slot (kv chunk)
  int32_t item0;     // first work item of the segment
  int32_t counter0;  // tile: first arrival counter of its query chunk (+ qb * H + h)
  int32_t n_kv;      // tile: kv chunks of its sequence (partials to merge)
  int32_t h0;        // first head
  int32_t nh;        // heads, >= 1
};

struct FwdArgs {
  void* o;              // whole-sequence output [Tq][H][d] (bf16 or f32)
  float* lse;           // [H][lse_stride]
  float* o_part;        // partial O  [P][part_rows][H][d] f32 (bf16 elements when part_bf16)
  float* lse_part;      // partial LSE [P][H][part_rows] f32
  int32_t* counters;    // tile arrival counters, zero at launch (fused merge)
  int32_t fused_merge;  // tensor-core path: the last arriving tile merges the partials
  int32_t part_bf16;    // tensor-core path: partial O rows in bf16
  int64_t lse_stride;   // Tq
  int64_t part_rows;    // R
  int32_t num_heads;
  float scale;          // softmax scale
  float scale_log2;     // scale * log2(e)
  int32_t n_items;
  int32_t n_segs;
  int32_t rows_per_item;  // query rows per work item: 256 (tensor cores, two tiles) or 128 (float32)
  FwdSeg segs[kMaxSegs];
};
static_assert(sizeof(FwdArgs) <= 32764, "forward arguments exceed the kernel parameter space");

struct MergeArgs {
  const void* o_part;   // float32, or bf16 when part_bf16
  const float* lse_part;
  void* o;
  float* lse;
  int64_t rows;
  int64_t part_stride_rows;
  int64_t lse_head_stride;
  int32_t n_parts;
  int32_t num_heads;
  int32_t out_bf16;
  int32_t part_bf16;
};

// Backward work: one item per (sequence, head, 128-key block); the item loops
// over every 128-row query block of the sequence.
struct BwdSeg {
  int32_t q_row0;
  int32_t k_row0;
  int32_t q_len;
  int32_t k_len;
  int32_t item0;
};

struct BwdArgs {
  const float* lse;      // [H][Tq]
  const float* dsum;     // D [H][Tq]
  float* dq_acc;         // [Tq][H][d] f32, zeroed before the launch
  void* dk;              // [Tk][H][d] bf16
  void* dv;              // [Tk][H][d] bf16
  int64_t lse_stride;    // Tq
  int32_t num_heads;
  float scale;
  float scale_log2;
  int32_t n_items;
  int32_t n_segs;
  BwdSeg segs[kMaxSegs];
};

// ---------------------------------------------------------------- launchers
// Each returns the CUDA error of the launch (cudaSuccess when enqueued).
// The tensor-core kernels are launched with one CTA per work item
// (args.n_items): the CTAs resident at a time steal the unstarted ones.
// to: bf16 map of the output o with the same box shape as tq (the kernel
// stores full 128-row tiles of final rows through it).
cudaError_t launch_fwd_tc(int head_dim, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, const CUtensorMap& to, const FwdArgs& args,
                          cudaStream_t stream);
cudaError_t launch_fwd_f32(int head_dim, const float* q, const float* k, const float* v,
                           const FwdArgs& args, cudaStream_t stream);
cudaError_t launch_merge(int head_dim, const MergeArgs& args, int num_sms, cudaStream_t stream);
cudaError_t launch_bwd_preprocess(int head_dim, const void* o, const void* dout, float* dsum,
                                  float* dq_acc, int64_t tq, int32_t num_heads, int num_sms,
                                  cudaStream_t stream);
// Query rows per block of the backward kernel: the row count of the Q / dO
// tensor-map boxes and of the dQ accumulator boxes it is launched with.
int bwd_query_block();
// tq, tdo: bf16 maps with 64-column x bwd_query_block()-row boxes; tk, tv:
// 64 x 128 boxes; tdq: float32 view [Tq][H*d] of the dQ accumulator with
// 32-column x bwd_query_block()-row boxes, 128-byte swizzle (the kernel adds
// into it with TMA).  args.dq_acc must be zeroed before the launch.
cudaError_t launch_bwd_tc(int head_dim, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq,
                          const BwdArgs& args, cudaStream_t stream);
cudaError_t launch_dq_convert(int head_dim, const float* dq_acc, void* dq, int64_t tq,
                              int32_t num_heads, float scale, int num_sms, cudaStream_t stream);

// Counts one kernel launch in the process-wide launch counter.
void note_launch();

// Shared-memory bytes a CTA of the tensor-core forward / backward requests.
size_t fwd_tc_smem_bytes(int head_dim);
size_t bwd_tc_smem_bytes(int head_dim);

// Error words recorded by bounded waits in each kernel family (read and
// cleared; synchronous).
uint32_t fwd_take_error();
uint32_t bwd_take_error();
uint32_t selftest_take_error();

// One CTA whose wait on an mbarrier nobody arrives on runs out after
// limit_ns (the bounded-wait self-test; see zl_selftest_wait_timeout).
cudaError_t launch_wait_timeout_selftest(uint64_t limit_ns, cudaStream_t stream);

}  // namespace zl
