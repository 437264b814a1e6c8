// Backward of coalesced varlen attention on sm_103a tensor cores.
//
// The analytic gradient of O = softmax(Q K^T * scale) V per sequence and head
// (the Zellige paper trains with exact backward, arXiv 2608.01150v1 §V-A):
//     P = exp(S - LSE) (recomputed from the forward's LSE),  D = rowsum(dO * O)
//     dV = P^T dO,  dS = P * (dO V^T - D),  dK = scale dS^T Q,  dQ = scale dS K
//
// A work item is (sequence, head, 128-key block).  Its CTA keeps K_j and V_j
// in shared memory and the dV / dK accumulators in TMEM, and walks every
// 128-row query block i of the sequence (starting at a block that depends on
// j, so that CTAs working on one head spread their dQ additions over
// different rows).  Per query block, with key rows on the TMEM lanes:
//     S^T  = K_j Q_i^T          (SS MMA)         -> TMEM [0,128)
//     dP^T = V_j dO_i^T         (SS MMA)         -> TMEM [128,256)
//     compute warps: P^T = 2^(S^T*scale*log2e - LSE_i*log2e),
//                    dS^T = P^T * (dP^T - D_i)   (bf16, back into TMEM, and
//                    dS into shared memory as an MN-major operand)
//     dV  += P^T  dO_i          (TS MMA, A from TMEM)  -> TMEM [256,384)
//     dK  += dS^T Q_i           (TS MMA)               -> TMEM [384,512)
//     dQ_i = dS K_j             (SS MMA, both MN-major) -> TMEM [0,128)
//     compute warps add dQ_i into a float32 accumulator in global memory
//     (vector atomics); dq_convert later scales and rounds it.
// After the last query block the compute warps write dV and scale * dK.
//
// Roles (320 threads, one CTA per SM): warps 0-7 compute (warp w reads TMEM
// lanes 32*(w%4).. and query columns 64*(w/4)..), warp 8 TMA producer, warp 9
// MMA issuer.  Every wait is bounded.
#include "common.cuh"
#include "launch.h"

namespace zl {
namespace {

__device__ uint32_t g_bwd_err;

constexpr int kBwdThreads = 320;
constexpr int kComputeThreads = 256;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kBwdStages = 2;
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;

template <int HD>
struct BwdSmem {
  uint8_t k[kBlockN * HD * 2];                    // HD/64 boxes of [128 rows][128 B]
  uint8_t v[kBlockN * HD * 2];
  uint8_t q[kBwdStages][kBlockM * HD * 2];
  uint8_t dout[kBwdStages][kBlockM * HD * 2];
  uint8_t ds[kBlockN * kBlockM * 2];              // dS^T rows (two 64-query halves), then dQ staging
  float lse2[kBlockM];                            // LSE * log2(e) of the query block
  float dsum[kBlockM];                            // D of the query block
  uint64_t kv_full, kv_empty;
  uint64_t qd_full[kBwdStages], qd_empty[kBwdStages];
  uint64_t s_full, sg_done, stage_full, dq_full, dq_drained, dkdv_full, dkdv_drained;
  uint64_t dq_staged, dq_free;
  uint32_t tmem_base;
  int abort_flag;
};

struct BwdWork {
  int seg;
  int h;
  int kb;
};

__device__ __forceinline__ BwdWork decode_bwd(const BwdArgs& a, int it) {
  int lo = 0, hi = a.n_segs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (a.segs[mid].item0 <= it) lo = mid; else hi = mid - 1;
  }
  const BwdSeg& s = a.segs[lo];
  const int nkb = (s.k_len + kBlockN - 1) / kBlockN;
  const int local = it - s.item0;
  return {lo, local / nkb, local % nkb};
}

__device__ __forceinline__ void drain_delay(uint64_t ns) {
  const uint64_t t0 = globaltimer();
  while (globaltimer() - t0 < ns) {
  }
}

// TMEM column of the bf16 operand (P^T or dS^T) for query k-step ks: half h
// of the query block lives at [64h, 64h+32) of its region.
__device__ __forceinline__ uint32_t op_col(int ks) { return (ks >> 2) * 64 + (ks & 3) * 8; }

// The LSE*log2e (threads 0-127) or D (threads 128-255) value of query row t
// of query block i; padding rows give P = 0 (LSE = +inf) and D = 0.
__device__ __forceinline__ float staged_value(const BwdArgs& a, const BwdSeg& sg, int h, int i, int tid) {
  const int t = tid & 127;
  const int qg = i * kBlockM + t;
  if (qg >= sg.q_len) return tid < 128 ? INFINITY : 0.f;
  const size_t idx = static_cast<size_t>(h) * a.lse_stride + sg.q_row0 + qg;
  return tid < 128 ? a.lse[idx] * kLog2e : a.dsum[idx];
}

template <int HD>
__global__ void __launch_bounds__(kBwdThreads, 1)
bwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
              const __grid_constant__ CUtensorMap tmDQ, const __grid_constant__ BwdArgs args) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  auto* sm = reinterpret_cast<BwdSmem<HD>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* abort_flag = &sm->abort_flag;

  if (threadIdx.x == 0) {
    mbar_init(&sm->kv_full, 1);
    mbar_init(&sm->kv_empty, 1);
    for (int s = 0; s < kBwdStages; ++s) {
      mbar_init(&sm->qd_full[s], 1);
      mbar_init(&sm->qd_empty[s], 1);
    }
    mbar_init(&sm->s_full, 1);
    mbar_init(&sm->sg_done, kComputeThreads);
    mbar_init(&sm->stage_full, kComputeThreads);
    mbar_init(&sm->dq_full, 1);
    mbar_init(&sm->dq_drained, kComputeThreads);
    mbar_init(&sm->dkdv_full, 1);
    mbar_init(&sm->dkdv_drained, kComputeThreads);
    mbar_init(&sm->dq_staged, kComputeThreads);
    mbar_init(&sm->dq_free, 1);
    sm->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&sm->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm->tmem_base;
  const uint32_t tS = tmem;          // S^T f32, then P^T bf16 at [64h, 64h+32)
  const uint32_t tDP = tmem + 128;   // dP^T f32, then dS^T bf16 at 128 + [64h, 64h+32), then dQ_i f32
  const uint32_t tDV = tmem + 256;
  const uint32_t tDK = tmem + 384;
  const uint32_t tDQ = tDP;

  if (warp == kProducerWarp) {
    if (lane == 0) {
      tma_prefetch_map(&tmQ);
      tma_prefetch_map(&tmK);
      tma_prefetch_map(&tmV);
      tma_prefetch_map(&tmDO);
      uint32_t item_it = 0, qd_it = 0;
      bool ok = true;
      for (int it = blockIdx.x; it < args.n_items && ok; it += gridDim.x, ++item_it) {
        const BwdWork w = decode_bwd(args, it);
        const BwdSeg& sg = args.segs[w.seg];
        const int nqb = (sg.q_len + kBlockM - 1) / kBlockM;
        const int start = w.kb % nqb;
        const int x0 = w.h * HD;
        if (!mbar_wait(&sm->kv_empty, (item_it & 1u) ^ 1u, abort_flag, &g_bwd_err, ERR_TIMEOUT_PRODUCER)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&sm->kv_full, 2 * kBlockN * HD * 2);
#pragma unroll
        for (int c = 0; c < HD / 64; ++c) {
          tma_load_2d(sm->k + c * kBlockN * 128, &tmK, &sm->kv_full, x0 + c * 64, sg.k_row0 + w.kb * kBlockN);
          tma_load_2d(sm->v + c * kBlockN * 128, &tmV, &sm->kv_full, x0 + c * 64, sg.k_row0 + w.kb * kBlockN);
        }
        for (int ii = 0; ii < nqb; ++ii, ++qd_it) {
          const int i = (start + ii) % nqb;
          const uint32_t st = qd_it % kBwdStages;
          const uint32_t ph = (qd_it / kBwdStages) & 1u;
          if (!mbar_wait(&sm->qd_empty[st], ph ^ 1u, abort_flag, &g_bwd_err, ERR_TIMEOUT_PRODUCER)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&sm->qd_full[st], 2 * kBlockM * HD * 2);
#pragma unroll
          for (int c = 0; c < HD / 64; ++c) {
            tma_load_2d(sm->q[st] + c * kBlockM * 128, &tmQ, &sm->qd_full[st], x0 + c * 64,
                        sg.q_row0 + i * kBlockM);
            tma_load_2d(sm->dout[st] + c * kBlockM * 128, &tmDO, &sm->qd_full[st], x0 + c * 64,
                        sg.q_row0 + i * kBlockM);
          }
        }
      }
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16(kBlockN, kBlockM, false, false);   // S^T, dP^T
      constexpr uint32_t idesc_acc = idesc_bf16(kBlockN, HD, false, true);       // dV, dK
      constexpr uint32_t idesc_dq = idesc_bf16(kBlockM, HD, true, true);         // dQ
      const uint32_t k_addr = smem_u32(sm->k);
      const uint32_t v_addr = smem_u32(sm->v);
      const uint32_t ds_addr = smem_u32(sm->ds);
      uint32_t item_it = 0, qd_it = 0, blk = 0;
      bool ok = true;
      // S^T = K Q_i^T into TMEM [0,128)
      auto issue_s = [&](uint32_t st) {
        const uint32_t q_addr = smem_u32(sm->q[st]);
#pragma unroll
        for (int ks = 0; ks < HD / 16; ++ks) {
          const uint32_t off = (ks >> 2) * (kBlockM * 128) + (ks & 3) * 32;
          umma_ss(tS, sdesc_sw128(k_addr + off, 16, 1024), sdesc_sw128(q_addr + off, 16, 1024), idesc_s,
                  ks > 0 ? 1u : 0u);
        }
      };
      for (int it = blockIdx.x; it < args.n_items && ok; it += gridDim.x, ++item_it) {
        const BwdWork w = decode_bwd(args, it);
        const BwdSeg& sg = args.segs[w.seg];
        const int nqb = (sg.q_len + kBlockM - 1) / kBlockM;
        if (!mbar_wait(&sm->kv_full, item_it & 1u, abort_flag, &g_bwd_err, ERR_TIMEOUT_MMA) ||
            !mbar_wait(&sm->qd_full[qd_it % kBwdStages], (qd_it / kBwdStages) & 1u, abort_flag, &g_bwd_err,
                       ERR_TIMEOUT_MMA)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_s(qd_it % kBwdStages);
        for (int ii = 0; ii < nqb; ++ii, ++qd_it, ++blk) {
          const uint32_t st = qd_it % kBwdStages;
          // dP^T = V dO_i^T into [128,256) once the previous dQ has been read out
          if (!mbar_wait(&sm->dq_drained, (blk & 1u) ^ 1u, abort_flag, &g_bwd_err, ERR_TIMEOUT_MMA)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t q_addr = smem_u32(sm->q[st]);
          const uint32_t do_addr = smem_u32(sm->dout[st]);
#pragma unroll
          for (int ks = 0; ks < HD / 16; ++ks) {
            const uint32_t off = (ks >> 2) * (kBlockM * 128) + (ks & 3) * 32;
            umma_ss(tDP, sdesc_sw128(v_addr + off, 16, 1024), sdesc_sw128(do_addr + off, 16, 1024), idesc_s,
                    ks > 0 ? 1u : 0u);
          }
          umma_commit(&sm->s_full);
          if (!mbar_wait(&sm->sg_done, blk & 1u, abort_flag, &g_bwd_err, ERR_TIMEOUT_MMA) ||
              (ii == 0 &&
               !mbar_wait(&sm->dkdv_drained, (item_it & 1u) ^ 1u, abort_flag, &g_bwd_err, ERR_TIMEOUT_MMA))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t acc0 = ii > 0 ? 1u : 0u;
#pragma unroll
          for (int ks = 0; ks < kBlockM / 16; ++ks) {
            umma_ts(tDV, tS + op_col(ks), sdesc_sw128(do_addr + ks * 2048, kBlockM * 128, 1024), idesc_acc,
                    (acc0 | (ks > 0 ? 1u : 0u)));
          }
#pragma unroll
          for (int ks = 0; ks < kBlockM / 16; ++ks) {
            umma_ts(tDK, tDP + op_col(ks), sdesc_sw128(q_addr + ks * 2048, kBlockM * 128, 1024), idesc_acc,
                    (acc0 | (ks > 0 ? 1u : 0u)));
          }
          // dQ_i = dS K into [128, 128+HD), after dK has read dS^T there
#pragma unroll
          for (int ks = 0; ks < kBlockN / 16; ++ks) {
            umma_ss(tDQ, sdesc_sw128(ds_addr + ks * 2048, kBlockN * 128, 1024),
                    sdesc_sw128(k_addr + ks * 2048, kBlockN * 128, 1024), idesc_dq, ks > 0 ? 1u : 0u);
          }
          umma_commit(&sm->dq_full);
          umma_commit(&sm->qd_empty[st]);
          if (ii + 1 < nqb) {
            // next S^T overlaps the dQ drain (dV has read P^T out of [0,128))
            const uint32_t nq = qd_it + 1;
            if (!mbar_wait(&sm->qd_full[nq % kBwdStages], (nq / kBwdStages) & 1u, abort_flag, &g_bwd_err,
                           ERR_TIMEOUT_MMA)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_s(nq % kBwdStages);
          }
        }
        if (!ok) break;
        umma_commit(&sm->dkdv_full);
        umma_commit(&sm->kv_empty);
      }
    }
  } else {
    // ------------------------------------------------------------ compute
    const int w4 = warp & 3;
    const int half = warp >> 2;
    const uint32_t lane_off = static_cast<uint32_t>(w4 * 32) << 16;
    const int jrow = w4 * 32 + lane;        // key row of S^T / dP^T, query row of dQ
    const int nh = args.num_heads;
    const float sl2 = args.scale_log2;
    uint32_t item_it = 0, blk = 0, stg = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < args.n_items && ok; it += gridDim.x, ++item_it) {
      const BwdWork w = decode_bwd(args, it);
      const BwdSeg& sg = args.segs[w.seg];
      const int nqb = (sg.q_len + kBlockM - 1) / kBlockM;
      const int start = w.kb % nqb;
      const bool kv_ok = w.kb * kBlockN + jrow < sg.k_len;
      float pref = staged_value(args, sg, w.h, start, threadIdx.x);
      for (int ii = 0; ii < nqb; ++ii, ++blk) {
        const int i = (start + ii) % nqb;
        // Stage LSE*log2e and D of this query block once every compute
        // thread is done with the previous one; prefetch the next block's.
        if (!__all_sync(0xffffffffu,
                        blk == 0 || mbar_wait(&sm->sg_done, (blk - 1) & 1u, abort_flag, &g_bwd_err,
                                              ERR_TIMEOUT_SOFTMAX))) {
          ok = false;
          break;
        }
        if (threadIdx.x < 128) sm->lse2[threadIdx.x] = pref;
        else sm->dsum[threadIdx.x - 128] = pref;
        mbar_arrive(&sm->stage_full);
        if (ii + 1 < nqb) pref = staged_value(args, sg, w.h, (start + ii + 1) % nqb, threadIdx.x);
        if (!__all_sync(0xffffffffu,
                        mbar_wait(&sm->stage_full, blk & 1u, abort_flag, &g_bwd_err, ERR_TIMEOUT_SOFTMAX)) ||
            !__all_sync(0xffffffffu,
                        mbar_wait(&sm->s_full, blk & 1u, abort_flag, &g_bwd_err, ERR_TIMEOUT_SOFTMAX))) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint8_t* ds_row = sm->ds + half * (kBlockN * 128) + jrow * 128;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int col = 64 * half + 32 * cc;     // query column within the block
          uint32_t s[32], dp[32];
          tmem_ld32(tS + lane_off + col, s);
          tmem_ld32(tDP + lane_off + col, dp);
          tmem_wait_ld();
          reg_fence(s);
          reg_fence(dp);
          uint32_t pp[16], dd[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int c0 = col + 2 * e;
            float p0 = fast_exp2(fmaf(__uint_as_float(s[2 * e]), sl2, -sm->lse2[c0]));
            float p1 = fast_exp2(fmaf(__uint_as_float(s[2 * e + 1]), sl2, -sm->lse2[c0 + 1]));
            if (!kv_ok) {
              p0 = 0.f;
              p1 = 0.f;
            }
            const float d0 = p0 * (__uint_as_float(dp[2 * e]) - sm->dsum[c0]);
            const float d1 = p1 * (__uint_as_float(dp[2 * e + 1]) - sm->dsum[c0 + 1]);
            pp[e] = pack_bf16x2(p0, p1);
            dd[e] = pack_bf16x2(d0, d1);
          }
          tmem_st16(tS + lane_off + 64 * half + 16 * cc, pp);
          tmem_st16(tDP + lane_off + 64 * half + 16 * cc, dd);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int chunk = cc * 4 + c;
            *reinterpret_cast<uint4*>(ds_row + ((chunk ^ (jrow & 7)) << 4)) =
                make_uint4(dd[4 * c], dd[4 * c + 1], dd[4 * c + 2], dd[4 * c + 3]);
          }
        }
        fence_proxy_async_smem();
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&sm->sg_done);
        // ---------------------------------------------- drain dQ_i
        // Read this thread's HD/2 columns of its query row out of TMEM (which
        // frees the columns for the next dP^T), then push them through the
        // dS buffer (128-byte swizzled boxes of 32 columns) into the float32
        // accumulator with TMA reduce-add.  Padding rows carry exact zeros.
        if (!__all_sync(0xffffffffu,
                        mbar_wait(&sm->dq_full, blk & 1u, abort_flag, &g_bwd_err, ERR_TIMEOUT_SOFTMAX))) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t g[HD / 64][32];
#pragma unroll
        for (int c = 0; c < HD / 64; ++c) tmem_ld32(tDQ + lane_off + half * (HD / 2) + 32 * c, g[c]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < HD / 64; ++c) reg_fence(g[c]);
        tc_fence_before();
        mbar_arrive(&sm->dq_drained);
        uint8_t* box = sm->ds + half * (kBlockM * 128) + jrow * 128;
#pragma unroll
        for (int c = 0; c < HD / 64; ++c, ++stg) {
#pragma unroll
          for (int e = 0; e < 8; ++e)
            *reinterpret_cast<uint4*>(box + ((e ^ (jrow & 7)) << 4)) =
                make_uint4(g[c][4 * e], g[c][4 * e + 1], g[c][4 * e + 2], g[c][4 * e + 3]);
          fence_proxy_async_smem();
          mbar_arrive(&sm->dq_staged);
          if (threadIdx.x == 0) {
            const bool staged = mbar_wait(&sm->dq_staged, stg & 1u, abort_flag, &g_bwd_err, ERR_TIMEOUT_SOFTMAX);
            if (staged) {
              const int y = sg.q_row0 + i * kBlockM;
              tma_reduce_add_2d(&tmDQ, sm->ds, w.h * HD + 32 * c, y);
              tma_reduce_add_2d(&tmDQ, sm->ds + kBlockM * 128, w.h * HD + HD / 2 + 32 * c, y);
              bulk_commit_group();
              bulk_wait_group_read0();
            }
            mbar_arrive(&sm->dq_free);
          }
          if (!__all_sync(0xffffffffu,
                          mbar_wait(&sm->dq_free, stg & 1u, abort_flag, &g_bwd_err, ERR_TIMEOUT_SOFTMAX))) {
            ok = false;
            break;
          }
        }
        if (!ok) break;
      }
      if (!ok) break;
      // ------------------------------------------------ dV, dK of the key block
      if (!__all_sync(0xffffffffu,
                      mbar_wait(&sm->dkdv_full, item_it & 1u, abort_flag, &g_bwd_err, ERR_TIMEOUT_SOFTMAX)))
        break;
      tc_fence_after();
      const size_t krow = static_cast<size_t>(sg.k_row0 + w.kb * kBlockN + jrow);
      __nv_bfloat16* dv_dst = reinterpret_cast<__nv_bfloat16*>(args.dv) + (krow * nh + w.h) * HD + half * (HD / 2);
      __nv_bfloat16* dk_dst = reinterpret_cast<__nv_bfloat16*>(args.dk) + (krow * nh + w.h) * HD + half * (HD / 2);
#pragma unroll
      for (int c = 0; c < HD / 64; ++c) {
        uint32_t a[32], b[32];
        tmem_ld32(tDV + lane_off + half * (HD / 2) + 32 * c, a);
        tmem_ld32(tDK + lane_off + half * (HD / 2) + 32 * c, b);
        tmem_wait_ld();
        reg_fence(a);
        reg_fence(b);
        if (kv_ok) {
          uint4* dv4 = reinterpret_cast<uint4*>(dv_dst + 32 * c);
          uint4* dk4 = reinterpret_cast<uint4*>(dk_dst + 32 * c);
          const float sc = args.scale;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            dv4[e] = make_uint4(pack_bf16x2(__uint_as_float(a[8 * e + 0]), __uint_as_float(a[8 * e + 1])),
                                pack_bf16x2(__uint_as_float(a[8 * e + 2]), __uint_as_float(a[8 * e + 3])),
                                pack_bf16x2(__uint_as_float(a[8 * e + 4]), __uint_as_float(a[8 * e + 5])),
                                pack_bf16x2(__uint_as_float(a[8 * e + 6]), __uint_as_float(a[8 * e + 7])));
            dk4[e] = make_uint4(
                pack_bf16x2(__uint_as_float(b[8 * e + 0]) * sc, __uint_as_float(b[8 * e + 1]) * sc),
                pack_bf16x2(__uint_as_float(b[8 * e + 2]) * sc, __uint_as_float(b[8 * e + 3]) * sc),
                pack_bf16x2(__uint_as_float(b[8 * e + 4]) * sc, __uint_as_float(b[8 * e + 5]) * sc),
                pack_bf16x2(__uint_as_float(b[8 * e + 6]) * sc, __uint_as_float(b[8 * e + 7]) * sc));
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&sm->dkdv_drained);
    }
    // the accumulator additions must have landed before the CTA exits
    if (threadIdx.x == 0) bulk_wait_group0();
  }

  // ---------------------------------------------------------------- teardown
  __syncwarp();
  if (*abort_flag) drain_delay(2000000ull);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

template <int HD>
cudaError_t launch_hd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                      const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdArgs& args, int grid,
                      cudaStream_t stream) {
  const size_t smem = sizeof(BwdSmem<HD>) + 1024;
  cudaError_t e = cudaFuncSetAttribute(bwd_tc_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  bwd_tc_kernel<HD><<<grid, kBwdThreads, smem, stream>>>(tq, tk, tv, tdo, tdq, args);
  return cudaGetLastError();
}

}  // namespace

size_t bwd_tc_smem_bytes(int head_dim) {
  return head_dim == 64 ? sizeof(BwdSmem<64>) + 1024 : sizeof(BwdSmem<128>) + 1024;
}

cudaError_t launch_bwd_tc(int head_dim, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq,
                          const BwdArgs& args, int grid, cudaStream_t stream) {
  if (head_dim == 64) return launch_hd<64>(tq, tk, tv, tdo, tdq, args, grid, stream);
  if (head_dim == 128) return launch_hd<128>(tq, tk, tv, tdo, tdq, args, grid, stream);
  return cudaErrorInvalidValue;
}

uint32_t bwd_take_error() {
  uint32_t v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_bwd_err, sizeof(v)) != cudaSuccess) return 0xFFFFFFFFu;
  if (v != 0) cudaMemcpyToSymbol(g_bwd_err, &zero, sizeof(zero));
  return v;
}

}  // namespace zl
