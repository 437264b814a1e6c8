// Host-side helpers shared by the library's entry points (zl_host.cpp and
// bwd_static.cu): the batch checks, the tensor maps the tensor-core kernels
// read and write, and the launch counter / profiling hook.  Internal; not part
// of the public C ABI.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "launch.h"
#include "zl_attn.h"

namespace zl {

// Largest packed token count (queries or keys) a call accepts: row indices of
// every block, including one block of padding past the end, stay in int32.
constexpr int64_t kMaxTokens = (int64_t(1) << 31) - 1 - 2 * kBlockM;

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The checks every entry point applies to a batch description before any
// CUDA call: num_seqs >= 0, 1 <= num_heads <= 4096, head_dim in {64, 128},
// both cu_seqlens arrays start at 0 and never decrease, both totals
// <= kMaxTokens, (T + one block) * H * d <= 2^40 for queries and keys, and no
// sequence with queries but no keys.  Writes Tq and Tk.
zl_status check_batch(const int32_t* cu_q, const int32_t* cu_k, int32_t num_seqs, int32_t num_heads,
                      int32_t head_dim, int64_t* tq, int64_t* tk);

// 2-D view [rows][H*d] of a packed bf16 tensor: boxes of 64 columns x
// box_rows rows with the 128-byte swizzle the UMMA descriptors expect; rows
// past the end read as zero.  False if the driver entry point is missing or
// the encoding fails.
bool make_map(CUtensorMap* map, const void* base, int64_t rows, int nh, int hd, int box_rows = 128);

// float32 view [rows][H*d] of the backward's dQ accumulator: boxes of 32
// columns x box_rows rows with the 128-byte swizzle, the shape the backward
// adds into with TMA.
bool make_map_acc(CUtensorMap* map, const float* base, int64_t rows, int nh, int hd, int box_rows);

// One launch, counted and (while zl_profile_begin is active) bracketed by two
// CUDA events on `stream`: prof_before creates and records the first event,
// prof_after records the second and files the pair under `name`.
struct ProfScope {
  cudaEvent_t start = nullptr;
  cudaEvent_t stop = nullptr;
  bool on = false;
};
zl_status prof_before(ProfScope* p, cudaStream_t stream);
zl_status prof_after(ProfScope* p, const char* name, cudaStream_t stream, cudaError_t launch_error);

template <typename F>
zl_status launch_counted(const char* name, cudaStream_t stream, F fn) {
  ProfScope p;
  const zl_status st = prof_before(&p, stream);
  if (st != ZL_OK) return st;
  return prof_after(&p, name, stream, fn());
}

}  // namespace zl
