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
#include <algorithm>
#include <cmath>
#include <mutex>

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

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

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

EncodeTiledFn static_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    cudaGetLastError();
  });
  return fn;
}

bool static_map(CUtensorMap* map, const void* base, int64_t rows, int nh, int hd, int box_rows = 128) {
  EncodeTiledFn fn = static_encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(nh) * hd, static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(nh) * hd * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// float32 view [rows][H*d] of the dQ accumulator: boxes of 32 columns x
// box_rows rows with the 128-byte swizzle, the shape the backward adds with TMA.
bool static_map_acc(CUtensorMap* map, const float* base, int64_t rows, int nh, int hd, int box_rows) {
  EncodeTiledFn fn = static_encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(nh) * hd, static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(nh) * hd * 4};
  const cuuint32_t box[2] = {32, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" zl_status zl_varlen_attn_bwd_static(
    const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
    const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int32_t num_seqs, int32_t num_heads,
    int32_t head_dim, float softmax_scale, void* dq, void* dk, void* dv, void* stream) {
  // ---- host-side checks, before any CUDA call
  if (num_seqs < 0 || num_heads < 1 || num_heads > 4096 || !cu_seqlens_q || !cu_seqlens_k) return ZL_EINVAL;
  if (head_dim != 64 && head_dim != 128) return ZL_EUNSUPPORTED;
  if (!(softmax_scale > 0.f) || !std::isfinite(softmax_scale)) return ZL_EINVAL;
  if (cu_seqlens_q[0] != 0 || cu_seqlens_k[0] != 0) return ZL_EINVAL;
  for (int32_t s = 0; s < num_seqs; ++s) {
    if (cu_seqlens_q[s + 1] < cu_seqlens_q[s] || cu_seqlens_k[s + 1] < cu_seqlens_k[s]) return ZL_EINVAL;
    if (cu_seqlens_q[s + 1] > cu_seqlens_q[s] && cu_seqlens_k[s + 1] == cu_seqlens_k[s]) return ZL_EINVAL;
  }
  const int64_t tq = cu_seqlens_q[num_seqs];
  const int64_t tk = cu_seqlens_k[num_seqs];
  if (tq == 0 && tk == 0) return ZL_OK;
  // scratch: dQ accumulator [Tq][H][d], then D [H][Tq] at a 256-byte boundary
  const size_t acc_floats = (static_cast<size_t>(tq) * num_heads * head_dim + 63) & ~size_t(63);
  const size_t need = acc_floats + static_cast<size_t>(tq) * num_heads;
  if (need > kStaticScratchFloats) return ZL_EWORKSPACE;
  if ((tq > 0 && (!q || !o || !lse || !dout || !dq)) || (tk > 0 && (!k || !v || !dk || !dv))) return ZL_EINVAL;
  const void* ptrs[] = {q, k, v, o, dout, dq, dk, dv, lse};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return ZL_EALIGN;

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
  if (!static_map(&mq, q, tq, num_heads, head_dim, bq) || !static_map(&mk, k, tk, num_heads, head_dim) ||
      !static_map(&mv, v, tk, num_heads, head_dim) || !static_map(&mdo, dout, tq, num_heads, head_dim, bq) ||
      !static_map_acc(&mdq, dq_acc, tq, num_heads, head_dim, bq))
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
