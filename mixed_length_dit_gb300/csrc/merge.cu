// Exact merge of partial attention results over disjoint key sets (the
// accumulation step of block-wise ring / all-gather attention, Zellige
// arXiv 2608.01150v1 §II-B and Table II).  Per query row r and head h:
//     lse = log(sum_p exp(lse_p)),   o = sum_p exp(lse_p - lse) * o_p.
//
// Memory-bound.  A group of d/4 threads owns one (head, row) pair and reads
// 16 bytes of each partial O row per thread, so each group reads whole
// 256/512-byte rows; groups are numbered head-major so the LSE reads and
// writes of neighbouring groups are contiguous.  Grid-stride over all pairs
// with a grid of a few waves of the SMs.
#include "common.cuh"
#include "launch.h"

namespace zl {
namespace {

constexpr int kMergeThreads = 256;

template <int HD, bool OUT_BF16>
__global__ void __launch_bounds__(kMergeThreads)
merge_kernel(const __grid_constant__ MergeArgs a) {
  constexpr int G = HD / 4;
  const int li = threadIdx.x % G;
  const int64_t total = a.rows * a.num_heads;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * (kMergeThreads / G);
  const int64_t nh = a.num_heads;
  const int64_t ps = a.part_stride_rows;
  for (int64_t g = static_cast<int64_t>(blockIdx.x) * (kMergeThreads / G) + threadIdx.x / G; g < total;
       g += stride) {
    const int64_t h = g / a.rows;
    const int64_t r = g - h * a.rows;
    float m = -INFINITY;
    for (int p = 0; p < a.n_parts; ++p) m = fmaxf(m, a.lse_part[(p * nh + h) * ps + r]);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float lse_out = -INFINITY;
    if (m != -INFINITY) {
      float sum = 0.f;
#pragma unroll 4
      for (int p = 0; p < a.n_parts; ++p) {
        const float wgt = expf(a.lse_part[(p * nh + h) * ps + r] - m);
        const float4 x = *reinterpret_cast<const float4*>(a.o_part + ((p * ps + r) * nh + h) * HD + 4 * li);
        sum += wgt;
        acc.x = fmaf(wgt, x.x, acc.x);
        acc.y = fmaf(wgt, x.y, acc.y);
        acc.z = fmaf(wgt, x.z, acc.z);
        acc.w = fmaf(wgt, x.w, acc.w);
      }
      const float inv = 1.f / sum;
      acc.x *= inv;
      acc.y *= inv;
      acc.z *= inv;
      acc.w *= inv;
      lse_out = m + logf(sum);
    }
    const size_t o_off = (static_cast<size_t>(r) * nh + h) * HD + 4 * li;
    if (OUT_BF16) {
      uint2 pk;
      pk.x = pack_bf16x2(acc.x, acc.y);
      pk.y = pack_bf16x2(acc.z, acc.w);
      *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(a.o) + o_off) = pk;
    } else {
      *reinterpret_cast<float4*>(reinterpret_cast<float*>(a.o) + o_off) = acc;
    }
    if (li == 0) a.lse[h * a.lse_head_stride + r] = lse_out;
  }
}

template <int HD>
cudaError_t launch_hd(const MergeArgs& a, int num_sms, cudaStream_t stream) {
  constexpr int G = HD / 4;
  const int64_t groups = a.rows * a.num_heads;
  const int64_t blocks_needed = (groups + (kMergeThreads / G) - 1) / (kMergeThreads / G);
  const int grid = static_cast<int>(blocks_needed < int64_t(num_sms) * 8 ? blocks_needed : int64_t(num_sms) * 8);
  if (grid <= 0) return cudaSuccess;
  if (a.out_bf16)
    merge_kernel<HD, true><<<grid, kMergeThreads, 0, stream>>>(a);
  else
    merge_kernel<HD, false><<<grid, kMergeThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_merge(int head_dim, const MergeArgs& args, int num_sms, cudaStream_t stream) {
  if (head_dim == 64) return launch_hd<64>(args, num_sms, stream);
  if (head_dim == 128) return launch_hd<128>(args, num_sms, stream);
  return cudaErrorInvalidValue;
}

}  // namespace zl
