// Memory-bound helpers of the backward pass.
//
// bwd_preprocess:  D[h][t] = sum_d dO[t][h][d] * O[t][h][d]  (float32 sum of
//                  bf16 products; the row term of dS = P * (dP - D)), and
//                  zeroes the float32 dQ accumulator row [t][h][:].
// dq_convert:      dq = bf16(scale * dq_acc).
//
// Both walk (head, token) pairs head-major with a group of d/8 threads per
// pair (16 bytes of each bf16 row per thread), grid-stride, so D is written
// contiguously and each O / dO row is read as one whole 128/256-byte run.
#include "common.cuh"
#include "launch.h"

namespace zl {
namespace {

constexpr int kAuxThreads = 256;

template <int HD>
__global__ void __launch_bounds__(kAuxThreads)
bwd_pre_kernel(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dout,
               float* __restrict__ dsum, float* __restrict__ dq_acc, int64_t tq, int32_t nh) {
  constexpr int G = HD / 8;
  const int li = threadIdx.x % G;
  const int64_t total = tq * nh;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * (kAuxThreads / G);
  // The loop bound is uniform over the block so every lane reaches the
  // shuffles below; pairs past the end only skip their loads and stores.
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * (kAuxThreads / G); base < total; base += stride) {
    const int64_t g = base + threadIdx.x / G;
    const bool valid = g < total;
    const int64_t h = valid ? g / tq : 0;
    const int64_t t = valid ? g - h * tq : 0;
    const size_t off = (static_cast<size_t>(t) * nh + h) * HD + 8 * li;
    const uint4 zero4 = make_uint4(0u, 0u, 0u, 0u);
    const uint4 a = valid ? *reinterpret_cast<const uint4*>(o + off) : zero4;
    const uint4 b = valid ? *reinterpret_cast<const uint4*>(dout + off) : zero4;
    float acc = 0.f;
    const uint32_t av[4] = {a.x, a.y, a.z, a.w};
    const uint32_t bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 x = bf16x2_to_float2(av[e]);
      const float2 y = bf16x2_to_float2(bv[e]);
      acc = fmaf(x.x, y.x, acc);
      acc = fmaf(x.y, y.y, acc);
    }
#pragma unroll
    for (int m = G / 2; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
    if (!valid) continue;
    if (li == 0) dsum[h * tq + t] = acc;
    float4* z = reinterpret_cast<float4*>(dq_acc + off);
    z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

__global__ void __launch_bounds__(kAuxThreads)
dq_convert_kernel(const float4* __restrict__ acc, uint4* __restrict__ out, int64_t n8, float scale) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kAuxThreads;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kAuxThreads + threadIdx.x; i < n8; i += stride) {
    const float4 x = acc[2 * i];
    const float4 y = acc[2 * i + 1];
    out[i] = make_uint4(pack_bf16x2(x.x * scale, x.y * scale), pack_bf16x2(x.z * scale, x.w * scale),
                        pack_bf16x2(y.x * scale, y.y * scale), pack_bf16x2(y.z * scale, y.w * scale));
  }
}

int grid_for(int64_t work_units, int per_block, int num_sms) {
  const int64_t need = (work_units + per_block - 1) / per_block;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  return static_cast<int>(need < cap ? need : cap);
}

}  // namespace

cudaError_t launch_bwd_preprocess(int head_dim, const void* o, const void* dout, float* dsum, float* dq_acc,
                                  int64_t tq, int32_t num_heads, int num_sms, cudaStream_t stream) {
  const int64_t pairs = tq * num_heads;
  if (pairs == 0) return cudaSuccess;
  const auto* ob = static_cast<const __nv_bfloat16*>(o);
  const auto* db = static_cast<const __nv_bfloat16*>(dout);
  if (head_dim == 64) {
    bwd_pre_kernel<64><<<grid_for(pairs, kAuxThreads / 8, num_sms), kAuxThreads, 0, stream>>>(
        ob, db, dsum, dq_acc, tq, num_heads);
  } else if (head_dim == 128) {
    bwd_pre_kernel<128><<<grid_for(pairs, kAuxThreads / 16, num_sms), kAuxThreads, 0, stream>>>(
        ob, db, dsum, dq_acc, tq, num_heads);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_dq_convert(int head_dim, const float* dq_acc, void* dq, int64_t tq, int32_t num_heads,
                              float scale, int num_sms, cudaStream_t stream) {
  const int64_t n8 = tq * num_heads * head_dim / 8;
  if (n8 == 0) return cudaSuccess;
  dq_convert_kernel<<<grid_for(n8, kAuxThreads, num_sms), kAuxThreads, 0, stream>>>(
      reinterpret_cast<const float4*>(dq_acc), static_cast<uint4*>(dq), n8, scale);
  return cudaGetLastError();
}

}  // namespace zl
