// Exact merge of partial attention results over disjoint key sets (the
// accumulation step of block-wise ring / all-gather attention, Zellige
// arXiv 2608.01150v1 §II-B and Table II).  Per query row r and head h:
//     lse = log(sum_p exp(lse_p)),   o = sum_p exp(lse_p - lse) * o_p.
//
// Memory-bound.  A group of threads owns one (head, row) pair and reads 16
// bytes of each partial O row per thread (4 float32 or 8 bf16 columns), so
// each group reads whole rows; groups are numbered head-major so the LSE reads and
// writes of neighbouring groups are contiguous.  Grid-stride over all pairs
// with exactly one full wave of resident blocks.
#include "common.cuh"
#include "launch.h"

namespace zl {
namespace {

constexpr int kMergeThreads = 256;

// Each thread owns E consecutive columns of a row: 4 for float32 partials and
// 8 for bf16 ones, so every partial load is 16 bytes.
template <bool PART_BF16>
struct PartCols {
  static constexpr int E = PART_BF16 ? 8 : 4;
};

// E consecutive elements of a partial O row (bf16 widens exactly).
template <bool PART_BF16>
__device__ __forceinline__ void load_part(const MergeArgs& a, int64_t off, float (&x)[PartCols<PART_BF16>::E]) {
  if constexpr (PART_BF16) {
    const uint4 u = *reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(a.o_part) + off);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = bf16x2_to_float2(w[i]);
      x[2 * i] = f.x;
      x[2 * i + 1] = f.y;
    }
  } else {
    const float4 v = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(a.o_part) + off);
    x[0] = v.x;
    x[1] = v.y;
    x[2] = v.z;
    x[3] = v.w;
  }
}

template <bool OUT_BF16, int E>
__device__ __forceinline__ void store_row(const MergeArgs& a, size_t o_off, const float (&v)[E]) {
  if constexpr (OUT_BF16) {
    uint32_t pk[E / 2];
#pragma unroll
    for (int i = 0; i < E / 2; ++i) pk[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
    __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(a.o) + o_off;
    if constexpr (E == 8)
      *reinterpret_cast<uint4*>(dst) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    else
      *reinterpret_cast<uint2*>(dst) = make_uint2(pk[0], pk[1]);
  } else {
    float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(a.o) + o_off);
#pragma unroll
    for (int i = 0; i < E / 4; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
  }
}

// Merges the partials of one (head, row) pair; this thread owns E of its d
// columns.  NP > 0: the part count is known at compile time, so every LSE
// and O load of the row is issued before any arithmetic.  NP = 0: any count.
template <int HD, int NP, bool OUT_BF16, bool PART_BF16>
__device__ __forceinline__ void merge_pair(const MergeArgs& a, int64_t h, int64_t r, int li) {
  constexpr int E = PartCols<PART_BF16>::E;
  const int64_t nh = a.num_heads;
  const int64_t ps = a.part_stride_rows;
  const int np = NP > 0 ? NP : a.n_parts;
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  float lse_out = -INFINITY;
  if (NP > 0) {
    float l[NP > 0 ? NP : 1];
    float x[NP > 0 ? NP : 1][E];
#pragma unroll
    for (int p = 0; p < NP; ++p) {
      l[p] = a.lse_part[(p * nh + h) * ps + r];
      load_part<PART_BF16>(a, ((p * ps + r) * nh + h) * HD + E * li, x[p]);
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
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = fmaf(wgt, x[p][e], acc[e]);
      }
      const float inv = 1.f / sum;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] *= inv;
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
        float x[E];
        load_part<PART_BF16>(a, ((p * ps + r) * nh + h) * HD + E * li, x);
        sum += wgt;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = fmaf(wgt, x[e], acc[e]);
      }
      const float inv = 1.f / sum;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] *= inv;
      lse_out = m + logf(sum);
    }
  }
  store_row<OUT_BF16, E>(a, (static_cast<size_t>(r) * nh + h) * HD + E * li, acc);
  if (li == 0) a.lse[h * a.lse_head_stride + r] = lse_out;
}

// A group of d/E threads owns one (head, row) pair at a time; groups are
// numbered head-major so LSE reads and writes of neighbouring groups are
// contiguous.  Each group takes two pairs per pass (half a grid apart) so
// twice the loads are in flight.
template <int HD, int NP, bool OUT_BF16, bool PART_BF16>
__global__ void __launch_bounds__(kMergeThreads)
merge_kernel(const __grid_constant__ MergeArgs a) {
  constexpr int G = HD / PartCols<PART_BF16>::E;
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
      merge_pair<HD, NP, OUT_BF16, PART_BF16>(a, h, r, li);
      merge_pair<HD, NP, OUT_BF16, PART_BF16>(a, h2, r2, li);
    } else {
      merge_pair<HD, NP, OUT_BF16, PART_BF16>(a, h, r, li);
    }
  }
}

// Blocks of a kernel resident per SM at once (asked once per kernel): the
// grid is one full wave of them, so no partial second wave runs at low
// occupancy at the end.
template <typename K>
int resident_blocks(K kernel) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kMergeThreads, 0) != cudaSuccess || n < 1) {
    cudaGetLastError();
    n = 1;
  }
  return n;
}

template <int HD, int NP, bool OUT_BF16, bool PART_BF16>
void launch_one(const MergeArgs& a, int num_sms, cudaStream_t stream) {
  static const int per_sm = resident_blocks(merge_kernel<HD, NP, OUT_BF16, PART_BF16>);
  constexpr int kGroups = kMergeThreads / (HD / PartCols<PART_BF16>::E);
  const int64_t groups = a.rows * a.num_heads;
  const int64_t blocks_needed = (groups + kGroups - 1) / kGroups;
  const int64_t wave = int64_t(num_sms) * per_sm;
  const int grid = static_cast<int>(blocks_needed < wave ? blocks_needed : wave);
  if (grid <= 0) return;
  merge_kernel<HD, NP, OUT_BF16, PART_BF16><<<grid, kMergeThreads, 0, stream>>>(a);
}

template <int HD, bool OUT_BF16, bool PART_BF16>
void launch_np(const MergeArgs& a, int num_sms, cudaStream_t stream) {
  switch (a.n_parts) {
    case 2: launch_one<HD, 2, OUT_BF16, PART_BF16>(a, num_sms, stream); break;
    case 4: launch_one<HD, 4, OUT_BF16, PART_BF16>(a, num_sms, stream); break;
    default: launch_one<HD, 0, OUT_BF16, PART_BF16>(a, num_sms, stream); break;
  }
}

template <int HD>
cudaError_t launch_hd(const MergeArgs& a, int num_sms, cudaStream_t stream) {
  if (a.out_bf16 && a.part_bf16)
    launch_np<HD, true, true>(a, num_sms, stream);
  else if (a.out_bf16)
    launch_np<HD, true, false>(a, num_sms, stream);
  else if (a.part_bf16)
    launch_np<HD, false, true>(a, num_sms, stream);
  else
    launch_np<HD, false, false>(a, num_sms, stream);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_merge(int head_dim, const MergeArgs& args, int num_sms, cudaStream_t stream) {
  if (head_dim == 64) return launch_hd<64>(args, num_sms, stream);
  if (head_dim == 128) return launch_hd<128>(args, num_sms, stream);
  return cudaErrorInvalidValue;
}

}  // namespace zl
