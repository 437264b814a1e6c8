// Exact merge of partial attention results over disjoint key sets (the
// accumulation step of block-wise ring / all-gather attention, Zellige
// arXiv 2608.01150v1 §II-B and Table II).  Per query row r and head h:
//     lse = log(sum_p exp(lse_p)),   o = sum_p exp(lse_p - lse) * o_p.
//
// Memory-bound.  A group of d/4 threads owns one (head, row) pair and reads
// 16 bytes of each partial O row per thread, so each group reads whole
// 256/512-byte rows; groups are numbered head-major so the LSE reads and
// writes of neighbouring groups are contiguous.  Grid-stride over all pairs
// with one full wave of resident blocks.
#include "common.cuh"
#include "launch.h"

namespace zl {
namespace {

constexpr int kMergeThreads = 256;

template <bool OUT_BF16>
__device__ __forceinline__ void store_row(const MergeArgs& a, size_t o_off, float4 v) {
  if (OUT_BF16) {
    uint2 pk;
    pk.x = pack_bf16x2(v.x, v.y);
    pk.y = pack_bf16x2(v.z, v.w);
    *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(a.o) + o_off) = pk;
  } else {
    *reinterpret_cast<float4*>(reinterpret_cast<float*>(a.o) + o_off) = v;
  }
}

// Merges the partials of one (head, row) pair; this thread owns 4 of its d
// columns.  NP > 0: the part count is known at compile time, so every LSE
// and O load of the row is issued before any arithmetic.  NP = 0: any count.
template <int HD, int NP, bool OUT_BF16>
__device__ __forceinline__ void merge_pair(const MergeArgs& a, int64_t h, int64_t r, int li) {
  const int64_t nh = a.num_heads;
  const int64_t ps = a.part_stride_rows;
  const int np = NP > 0 ? NP : a.n_parts;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float lse_out = -INFINITY;
  if (NP > 0) {
    float l[NP > 0 ? NP : 1];
    float4 x[NP > 0 ? NP : 1];
#pragma unroll
    for (int p = 0; p < NP; ++p) {
      l[p] = a.lse_part[(p * nh + h) * ps + r];
      x[p] = *reinterpret_cast<const float4*>(a.o_part + ((p * ps + r) * nh + h) * HD + 4 * li);
    }
    float m = l[0];
#pragma unroll
    for (int p = 1; p < NP; ++p) m = fmaxf(m, l[p]);
    if (m != -INFINITY) {
      float sum = 0.f;
#pragma unroll
      for (int p = 0; p < NP; ++p) {
        const float wgt = expf(l[p] - m);
        sum += wgt;
        acc.x = fmaf(wgt, x[p].x, acc.x);
        acc.y = fmaf(wgt, x[p].y, acc.y);
        acc.z = fmaf(wgt, x[p].z, acc.z);
        acc.w = fmaf(wgt, x[p].w, acc.w);
      }
      const float inv = 1.f / sum;
      acc = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
      lse_out = m + logf(sum);
    }
  } else {
    float m = -INFINITY;
    for (int p = 0; p < np; ++p) m = fmaxf(m, a.lse_part[(p * nh + h) * ps + r]);
    if (m != -INFINITY) {
      float sum = 0.f;
#pragma unroll 4
      for (int p = 0; p < np; ++p) {
        const float wgt = expf(a.lse_part[(p * nh + h) * ps + r] - m);
        const float4 x = *reinterpret_cast<const float4*>(a.o_part + ((p * ps + r) * nh + h) * HD + 4 * li);
        sum += wgt;
        acc.x = fmaf(wgt, x.x, acc.x);
        acc.y = fmaf(wgt, x.y, acc.y);
        acc.z = fmaf(wgt, x.z, acc.z);
        acc.w = fmaf(wgt, x.w, acc.w);
      }
      const float inv = 1.f / sum;
      acc = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
      lse_out = m + logf(sum);
    }
  }
  store_row<OUT_BF16>(a, (static_cast<size_t>(r) * nh + h) * HD + 4 * li, acc);
  if (li == 0) a.lse[h * a.lse_head_stride + r] = lse_out;
}

// A group of d/4 threads owns one (head, row) pair at a time; groups are
// numbered head-major so LSE reads and writes of neighbouring groups are
// contiguous.  Each group takes two pairs per pass (half a grid apart) so
// twice the loads are in flight.
template <int HD, int NP, bool OUT_BF16>
__global__ void __launch_bounds__(kMergeThreads)
merge_kernel(const __grid_constant__ MergeArgs a) {
  constexpr int G = HD / 4;
  constexpr int kGroups = kMergeThreads / G;
  const int li = threadIdx.x % G;
  const int64_t total = a.rows * a.num_heads;
  const int64_t n_groups = static_cast<int64_t>(gridDim.x) * kGroups;
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * kGroups + threadIdx.x / G;
  for (int64_t g = gid; g < total; g += 2 * n_groups) {
    const int64_t g2 = g + n_groups;
    const int64_t h = g / a.rows;
    const int64_t r = g - h * a.rows;
    if (g2 < total) {
      const int64_t h2 = g2 / a.rows;
      const int64_t r2 = g2 - h2 * a.rows;
      merge_pair<HD, NP, OUT_BF16>(a, h, r, li);
      merge_pair<HD, NP, OUT_BF16>(a, h2, r2, li);
    } else {
      merge_pair<HD, NP, OUT_BF16>(a, h, r, li);
    }
  }
}

template <int HD, bool OUT_BF16>
void launch_np(const MergeArgs& a, int grid, cudaStream_t stream) {
  switch (a.n_parts) {
    case 2: merge_kernel<HD, 2, OUT_BF16><<<grid, kMergeThreads, 0, stream>>>(a); break;
    case 4: merge_kernel<HD, 4, OUT_BF16><<<grid, kMergeThreads, 0, stream>>>(a); break;
    default: merge_kernel<HD, 0, OUT_BF16><<<grid, kMergeThreads, 0, stream>>>(a); break;
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
    launch_np<HD, true>(a, grid, stream);
  else
    launch_np<HD, false>(a, grid, stream);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_merge(int head_dim, const MergeArgs& args, int num_sms, cudaStream_t stream) {
  if (head_dim == 64) return launch_hd<64>(args, num_sms, stream);
  if (head_dim == 128) return launch_hd<128>(args, num_sms, stream);
  return cudaErrorInvalidValue;
}

}  // namespace zl
