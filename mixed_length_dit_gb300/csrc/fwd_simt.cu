// Forward in float32 without tensor cores, for callers that need float32
// inputs and ~1e-6 relative accuracy (ZL_FP32).  Same work items, segment
// table and outputs as the tensor-core kernel; the arithmetic is float32 FMA
// with an online softmax in natural-log units (expf).
//
// A block takes one work item (segment, head, 128-row query block): 128 query
// rows, HD/64 threads per row (each holds 64 of the row's query and output
// columns; the two halves of a score are combined with one shuffle).  Keys and
// values stream through shared memory 32 rows at a time.
#include "common.cuh"
#include "launch.h"
#include "work.cuh"

namespace zl {
namespace {

constexpr int kKeyChunk = 32;

template <int HD>
__global__ void __launch_bounds__(128 * (HD / 64))
fwd_f32_kernel(const float* __restrict__ q, const float* __restrict__ k,
               const float* __restrict__ v, const __grid_constant__ FwdArgs args) {
  constexpr int TPR = HD / 64;
  __shared__ float sK[kKeyChunk][HD];
  __shared__ float sV[kKeyChunk][HD];
  const int row = threadIdx.x / TPR;
  const int part = threadIdx.x % TPR;
  const int nh = args.num_heads;
  const float scale = args.scale;

  for (int it = blockIdx.x; it < args.n_items; it += gridDim.x) {
    const FwdWork w = decode_fwd(args, it);
    const FwdSeg& sg = args.segs[w.seg];
    const int q_local = w.qb * kBlockM + row;
    const bool row_ok = q_local < sg.q_len;
    float qv[64], acc[64];
    const float* qsrc = q + (static_cast<size_t>(sg.q_row0 + q_local) * nh + w.h) * HD + part * 64;
#pragma unroll
    for (int c = 0; c < 64; ++c) {
      qv[c] = row_ok ? qsrc[c] : 0.f;
      acc[c] = 0.f;
    }
    float m = -INFINITY, l = 0.f;
    for (int kc = 0; kc < sg.k_len; kc += kKeyChunk) {
      const int n = min(kKeyChunk, sg.k_len - kc);
      __syncthreads();
      for (int idx = threadIdx.x; idx < n * HD; idx += blockDim.x) {
        const int j = idx / HD, c = idx % HD;
        const size_t src = (static_cast<size_t>(sg.k_row0 + kc + j) * nh + w.h) * HD + c;
        sK[j][c] = k[src];
        sV[j][c] = v[src];
      }
      __syncthreads();
      for (int j = 0; j < n; ++j) {
        float dot = 0.f;
#pragma unroll
        for (int c = 0; c < 64; ++c) dot = fmaf(qv[c], sK[j][part * 64 + c], dot);
        if (TPR == 2) dot += __shfl_xor_sync(0xffffffffu, dot, 1);
        const float s = dot * scale;
        if (s > m) {
          const float corr = expf(m - s);   // 0 when m = -inf
          l *= corr;
#pragma unroll
          for (int c = 0; c < 64; ++c) acc[c] *= corr;
          m = s;
        }
        const float p = expf(s - m);
        l += p;
#pragma unroll
        for (int c = 0; c < 64; ++c) acc[c] = fmaf(p, sV[j][part * 64 + c], acc[c]);
      }
    }
    if (row_ok) {
      const float inv_l = 1.f / l;
      const float lse_val = m + logf(l);
      float* dst;
      if (sg.slot < 0) {
        dst = reinterpret_cast<float*>(args.o) +
              (static_cast<size_t>(sg.q_row0 + q_local) * nh + w.h) * HD + part * 64;
        if (part == 0) args.lse[static_cast<size_t>(w.h) * args.lse_stride + sg.q_row0 + q_local] = lse_val;
      } else {
        const size_t prow = static_cast<size_t>(sg.slot) * args.part_rows + sg.out_row0 + q_local;
        dst = args.o_part + (prow * nh + w.h) * HD + part * 64;
        if (part == 0)
          args.lse_part[(static_cast<size_t>(sg.slot) * nh + w.h) * args.part_rows + sg.out_row0 + q_local] =
              lse_val;
      }
#pragma unroll
      for (int c = 0; c < 64; c += 4)
        *reinterpret_cast<float4*>(dst + c) =
            make_float4(acc[c] * inv_l, acc[c + 1] * inv_l, acc[c + 2] * inv_l, acc[c + 3] * inv_l);
    }
  }
}

}  // namespace

cudaError_t launch_fwd_f32(int head_dim, const float* q, const float* k, const float* v,
                           const FwdArgs& args, cudaStream_t stream) {
  const int grid = args.n_items;
  if (grid <= 0) return cudaSuccess;
  if (head_dim == 64) {
    fwd_f32_kernel<64><<<grid, 128, 0, stream>>>(q, k, v, args);
  } else if (head_dim == 128) {
    fwd_f32_kernel<128><<<grid, 256, 0, stream>>>(q, k, v, args);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace zl
