// zl_varlen_attn_bwd_static: the backward without a caller workspace.
//
// Some callers cannot allocate device memory when they need a gradient: a
// plugin inside an engine that owns all device memory and forbids allocation
// during execution, code running between stream-capture begin and end where a
// fresh allocation would not be part of the graph, or a process whose memory
// is fully reserved by a pooling allocator it may not call.  This entry point
// serves them: its scratch (the float32 dQ accumulator and the row term D) is
// a fixed array in this library's device image instead of a workspace
// argument.  The caller still provides every input and output buffer.
//
// The array is reserved on each GPU the library is loaded on and kept until
// the process exits.  Every call on a device uses the same array, so calls
// whose kernels overlap on the GPU (different streams without ordering) race
// on it; calls on one stream, or otherwise ordered, are safe.  The preprocess
// kernel rewrites all of D and zeroes the part of the accumulator a call uses,
// so nothing left by an earlier call leaks into the next.
//
// Its launches are counted (zl_launch_count) but not timed by the profiling
// hook: bracketing them would create CUDA events, and this entry point
// allocates nothing at all.
#include <algorithm>
#include <cmath>
#include <mutex>

#include "host.h"
#include "launch.h"
#include "zl_attn.h"

namespace {

constexpr size_t kStaticScratchFloats = size_t(16) << 20;   // 64 MiB of float32

static __device__ __align__(256) float zl_bwd_static_scratch[kStaticScratchFloats];

struct StaticDevice {
  std::once_flag once;
  float* scratch = nullptr;   // device address of zl_bwd_static_scratch
  int sms = 0;
  zl_status status = ZL_OK;
};
StaticDevice g_static_dev[128];

// Once per device, with that device current: check it, and look up the device
// address of the scratch array (in host code the array's name is only a
// host-side stand-in, never a device address).
zl_status static_setup(float** scratch, int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return ZL_ENODEVICE;
  }
  if (dev < 0 || dev >= 128) return ZL_ENODEVICE;
  StaticDevice& d = g_static_dev[dev];
  std::call_once(d.once, [&d, dev] {
    int major = 0, minor = 0, n = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      d.status = ZL_ECUDA;
      return;
    }
    if (major != 10 || minor != 3) {
      d.status = ZL_ENODEVICE;
      return;
    }
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, zl_bwd_static_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      d.status = ZL_ECUDA;
      return;
    }
    d.scratch = static_cast<float*>(p);
    d.sms = n;
    d.status = ZL_OK;
  });
  *scratch = d.scratch;
  *sms = d.sms;
  return d.status;
}

}  // namespace

extern "C" zl_status zl_varlen_attn_bwd_static(
    const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
    const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int32_t num_seqs, int32_t num_heads,
    int32_t head_dim, float softmax_scale, void* dq, void* dk, void* dv, void* stream) {
  // ---- host-side checks, before any CUDA call: the batch rules of every
  // entry point (token bounds included), then the scratch limit
  int64_t tq = 0, tk = 0;
  const zl_status bst = zl::check_batch(cu_seqlens_q, cu_seqlens_k, num_seqs, num_heads, head_dim, &tq, &tk);
  if (bst != ZL_OK) return bst;
  if (!(softmax_scale > 0.f) || !std::isfinite(softmax_scale)) return ZL_EINVAL;
  if (tq == 0 && tk == 0) return ZL_OK;
  // scratch: dQ accumulator [Tq][H][d], then D [H][Tq] at a 256-byte boundary
  const size_t acc_floats = (static_cast<size_t>(tq) * num_heads * head_dim + 63) & ~size_t(63);
  const size_t need = acc_floats + static_cast<size_t>(tq) * num_heads;
  if (need > kStaticScratchFloats) return ZL_EWORKSPACE;
  if ((tq > 0 && (!q || !o || !lse || !dout || !dq)) || (tk > 0 && (!k || !v || !dk || !dv))) return ZL_EINVAL;
  const void* ptrs[] = {q, k, v, o, dout, dq, dk, dv, lse};
  for (const void* p : ptrs)
    if (p && !zl::aligned16(p)) return ZL_EALIGN;

  float* scratch = nullptr;
  int sms = 0;
  zl_status st = static_setup(&scratch, &sms);
  if (st != ZL_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t row_bytes = static_cast<size_t>(num_heads) * head_dim * 2;
  for (int32_t i = 0; i < num_seqs; ++i) {
    const int32_t lq = cu_seqlens_q[i + 1] - cu_seqlens_q[i];
    const int32_t lk = cu_seqlens_k[i + 1] - cu_seqlens_k[i];
    if (lq == 0 && lk > 0) {
      if (cudaMemsetAsync(static_cast<char*>(dk) + cu_seqlens_k[i] * row_bytes, 0, lk * row_bytes, s) !=
              cudaSuccess ||
          cudaMemsetAsync(static_cast<char*>(dv) + cu_seqlens_k[i] * row_bytes, 0, lk * row_bytes, s) !=
              cudaSuccess) {
        cudaGetLastError();
        return ZL_ECUDA;
      }
    }
  }
  if (tq == 0) return ZL_OK;
  float* dq_acc = scratch;
  float* dsum = scratch + acc_floats;
  if (zl::launch_bwd_preprocess(head_dim, o, dout, dsum, dq_acc, tq, num_heads, sms, s) != cudaSuccess) {
    cudaGetLastError();
    return ZL_ECUDA;
  }
  zl::note_launch();
  CUtensorMap mq, mk, mv, mdo, mdq;
  const int bq = zl::bwd_query_block();
  if (!zl::make_map(&mq, q, tq, num_heads, head_dim, bq) || !zl::make_map(&mk, k, tk, num_heads, head_dim) ||
      !zl::make_map(&mv, v, tk, num_heads, head_dim) || !zl::make_map(&mdo, dout, tq, num_heads, head_dim, bq) ||
      !zl::make_map_acc(&mdq, dq_acc, tq, num_heads, head_dim, bq))
    return ZL_ECUDA;
  static thread_local zl::BwdArgs args;
  args.lse = lse;
  args.dsum = dsum;
  args.dq_acc = dq_acc;
  args.dk = dk;
  args.dv = dv;
  args.lse_stride = tq;
  args.num_heads = num_heads;
  args.scale = softmax_scale;
  args.scale_log2 = softmax_scale * 1.4426950408889634f;
  // Sequences in input order, up to kMaxSegs per launch; within a launch the
  // longest query range first (ties by packed position, i.e. input order).
  int32_t next = 0;
  while (next < num_seqs) {
    int32_t n = 0;
    while (next < num_seqs && n < zl::kMaxSegs) {
      const int32_t lq = cu_seqlens_q[next + 1] - cu_seqlens_q[next];
      const int32_t lk = cu_seqlens_k[next + 1] - cu_seqlens_k[next];
      if (lq > 0 && lk > 0) args.segs[n++] = zl::BwdSeg{cu_seqlens_q[next], cu_seqlens_k[next], lq, lk, 0};
      ++next;
    }
    if (n == 0) continue;
    std::sort(args.segs, args.segs + n, [](const zl::BwdSeg& a, const zl::BwdSeg& b) {
      return a.q_len != b.q_len ? a.q_len > b.q_len : a.q_row0 < b.q_row0;
    });
    int64_t items = 0;
    for (int32_t i = 0; i < n; ++i) {
      args.segs[i].item0 = static_cast<int32_t>(items);
      items += int64_t(num_heads) * ((args.segs[i].k_len + zl::kBlockN - 1) / zl::kBlockN);
    }
    args.n_segs = n;
    if (items > INT32_MAX) return ZL_EINVAL;      // more items than a grid (and an int32 index) can hold
    args.n_items = static_cast<int32_t>(items);
    if (zl::launch_bwd_tc(head_dim, mq, mk, mv, mdo, mdq, args, s) != cudaSuccess) {
      cudaGetLastError();
      return ZL_ECUDA;
    }
    zl::note_launch();
  }
  if (zl::launch_dq_convert(head_dim, dq_acc, dq, tq, num_heads, softmax_scale, sms, s) != cudaSuccess) {
    cudaGetLastError();
    return ZL_ECUDA;
  }
  zl::note_launch();
  return ZL_OK;
}
