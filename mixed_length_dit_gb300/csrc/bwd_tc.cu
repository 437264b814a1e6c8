// Backward of coalesced varlen attention on sm_103a tensor cores.
//
// The analytic gradient of O = softmax(Q K^T * scale) V per sequence and head
// (the Zellige paper trains with exact backward, arXiv 2608.01150v1 §V-A):
//     P = exp(S - LSE) (recomputed from the forward's LSE),  D = rowsum(dO * O)
//     dV = P^T dO,  dS = P * (dO V^T - D),  dK = scale dS^T Q,  dQ = scale dS K
//
// A work item is (sequence, head, 128-key block j).  Its CTA keeps K_j and V_j
// in shared memory and the dV / dK accumulators in TMEM, and walks every
// 64-row query block i of the sequence (starting at a block that depends on
// j, so CTAs working on one head spread their dQ additions over different
// rows).  Key rows sit on the 128 TMEM lanes.  Per query block g:
//     S^T  = K_j Q_i^T      (SS MMA, N = 64)           -> S[g % 2]
//     dP^T = V_j dO_i^T     (SS MMA)                   -> DP
//     softmax-grad warps load S^T and dP^T (DP is then free for the next
//       block), form P^T = 2^(S^T*scale*log2e - LSE*log2e) in bf16 over
//       S[g % 2] for the TS MMA, and dS^T = P^T (dP^T - D) in bf16 into shared
//       memory ([key][query], the operand layout both MMAs below read)
//     dV  += P^T dO_i       (TS MMA, A from TMEM)      -> TMEM
//     dK  += dS^T Q_i       (SS MMA, A = dS^T K-major) -> TMEM
//     dQ_i^T = K_j^T dS_i^T (SS MMA, both MN-major)    -> DQ (d on the lanes)
//     drain warps read dQ_i^T out of TMEM, stage it in 128-byte-swizzled
//       32-column boxes inside the Q_i/dO_i stage once dV and dK are done
//       with it, and add it into a float32 accumulator in global memory with
//       TMA reduce-add (a bulk copy holds no load/store slots while L2
//       performs the additions); the stage goes back to the producer once the
//       copy engine has read it.  dq_convert later scales and rounds it.
// dQ^T has a TMEM region of its own, so the chain dQ^T -> drain runs beside
// the main loop: S^T of block g+2 reuses S[g % 2] right after dV of block g
// (issued earlier by the same thread, and MMAs of one thread execute in
// order), and dP^T of block g+1 reuses DP once the softmax-grad warps have
// loaded dP^T of block g.
// Each query block's MMAs come from three issuing threads in different warps,
// one per chain of dependencies (S^T -> dV, dP^T -> dK, dS -> dQ^T), so each
// product goes out as soon as its own inputs are ready (M128 x N64 MMAs
// take ~54 cycles each of the shared tensor pipe, N = 128 ones 64): A issues
// S^T and dV, B issues dP^T and dK, C issues dQ^T.  A and B issue the
// S^T / dP^T of the next block before the accumulation of the current one.
//
// Roles (512 threads, one CTA per SM): warps 0-7 softmax-grad (warp w reads
// TMEM lanes 32*(w%4).. and query columns 32*(w/4)..), warps 8-11 dQ drain
// and, after a key block's last query block, its dV/dK epilogue (so the
// softmax-grad warps go straight on to the next item), warp 12 TMA producer
// (4-stage Q/dO ring; once it knows the next item it prefetches that item's
// K/V and first Q/dO tiles into L2), warps 13-15 MMA issuers.  Every wait is
// bounded.
// The grid holds one CTA per item, ordered longest-first by the host; the
// resident CTA of an SM takes its own item, then the producer steals the next
// unstarted one from the launch queue (cluster launch control) and hands its
// index to the other roles.
#include "common.cuh"
#include "launch.h"

namespace zl {
namespace {

__device__ uint32_t g_bwd_err;

constexpr int kBQ = 64;                     // query rows per block in the backward
constexpr int kBwdThreads = 512;
constexpr int kSgThreads = 256;
constexpr int kDrainThreads = 128;
constexpr int kDrainWarp0 = 8;
constexpr int kProducerWarp = 12;
constexpr int kMmaWarpA = 13;               // S^T (into S[b]), dV
constexpr int kMmaWarpB = 14;               // dP^T (into DP), dK
constexpr int kMmaWarpC = 15;               // dQ^T (into DQ)
constexpr int kQdStages = 4;
constexpr int kItemReaders = 15;             // issuers A, B, C + 4 drain warps + 8 softmax-grad warps
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;

template <int HD>
struct BwdSmem {
  uint8_t k[kBlockN * HD * 2];                    // HD/64 boxes of [128 rows][128 B]
  uint8_t v[kBlockN * HD * 2];
  uint8_t qd[kQdStages][2 * kBQ * HD * 2];        // Q_i then dO_i, HD/64 boxes of [64 rows][128 B] each
  uint8_t ds[2][kBlockN * kBQ * 2];               // dS as [128 key rows][64 queries], 128B-swizzled
  float lse2[2][kBQ];                             // LSE * log2(e) of the query block
  float dsum[2][kBQ];                             // D of the query block
  uint64_t kv_full, kv_empty;
  uint64_t qd_full[kQdStages], qd_empty[kQdStages];
  uint64_t qd_read[kQdStages];                    // dV and dK of the stage's block are done
  uint64_t s_full[2], sg_done[2], ds_free[2];
  uint64_t dp_free, dq_full, dq_drained;
  uint64_t stage_full, dkdv_full, dkdv_drained;
  ItemRing ring;                                  // work items, producer -> the other roles
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

// TMEM column (relative to S[b]) of the bf16 operand P^T for query k-step ks:
// queries 32h..32h+31 of the block live at [32h, 32h+16).
__device__ __forceinline__ uint32_t op_col(int ks) { return (ks >> 1) * 32 + (ks & 1) * 8; }

// LSE*log2e (threads 0-63) or D (threads 64-127) of query row t of block i;
// padding rows give P = 0 (LSE = +inf) and D = 0.  Other threads: unused.
__device__ __forceinline__ float staged_value(const BwdArgs& a, const BwdSeg& sg, int h, int i, int tid) {
  const int t = tid & (kBQ - 1);
  const int qg = i * kBQ + t;
  if (tid >= 2 * kBQ) return 0.f;
  if (qg >= sg.q_len) return tid < kBQ ? INFINITY : 0.f;
  const size_t idx = static_cast<size_t>(h) * a.lse_stride + sg.q_row0 + qg;
  return tid < kBQ ? a.lse[idx] * kLog2e : a.dsum[idx];
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
    mbar_init(&sm->kv_empty, 3);                   // A, B and C are done with K/V
    for (int s = 0; s < kQdStages; ++s) {
      mbar_init(&sm->qd_full[s], 1);
      mbar_init(&sm->qd_empty[s], kDrainThreads / 32);   // each drain warp, after its reduce read the stage
      mbar_init(&sm->qd_read[s], 2);                     // dV (A) and dK (B) commits
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm->s_full[b], 2);                // S^T from A, dP^T from B
      mbar_init(&sm->sg_done[b], kSgThreads);
      mbar_init(&sm->ds_free[b], 2);               // dK (B) and dQ^T (C) have read dS
    }
    mbar_init(&sm->dp_free, kSgThreads);
    mbar_init(&sm->dq_full, 1);
    mbar_init(&sm->dq_drained, kDrainThreads);
    mbar_init(&sm->stage_full, kSgThreads);
    mbar_init(&sm->dkdv_full, 2);
    mbar_init(&sm->dkdv_drained, kDrainThreads);
    ring_init(&sm->ring, kItemReaders);
    sm->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarpA) {
    tmem_alloc(&sm->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm->tmem_base;
  // S[b] = tmem + 64b, DP = tmem + 128, DQ = tmem + 192 (64 columns each), dV, dK.
  const uint32_t tDP = tmem + 128;
  const uint32_t tDQ = tmem + 192;
  const uint32_t tDV = tmem + 256;
  const uint32_t tDK = tmem + 384;

  if (warp == kProducerWarp) {
    if (lane == 0) {
      tma_prefetch_map(&tmQ);
      tma_prefetch_map(&tmK);
      tma_prefetch_map(&tmV);
      tma_prefetch_map(&tmDO);
      uint32_t item_it = 0, qd_it = 0, steal_ph = 0;
      // the CTA's own item comes first
      bool ok = ring_publish(&sm->ring, 0, static_cast<int>(blockIdx.x), abort_flag, &g_bwd_err,
                             ERR_TIMEOUT_PRODUCER);
      for (uint32_t n = 1, it = blockIdx.x; ok; ++n, ++item_it) {
        const BwdWork w = decode_bwd(args, static_cast<int>(it));
        const BwdSeg& sg = args.segs[w.seg];
        const int nqb = (sg.q_len + kBQ - 1) / kBQ;
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
        bool asked = false;
        for (int ii = 0; ii < nqb; ++ii, ++qd_it) {
          const int i = (start + ii) % nqb;
          const uint32_t st = qd_it % kQdStages;
          const uint32_t ph = (qd_it / kQdStages) & 1u;
          if (ii == nqb - 1) {
            // the item's last Q/dO block is next: ask for the following item
            // now, a few query blocks before the other roles need it
            ring_ask(&sm->ring);
            asked = true;
          }
          if (!mbar_wait(&sm->qd_empty[st], ph ^ 1u, abort_flag, &g_bwd_err, ERR_TIMEOUT_PRODUCER)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&sm->qd_full[st], 2 * kBQ * HD * 2);
#pragma unroll
          for (int c = 0; c < HD / 64; ++c) {
            tma_load_2d(sm->qd[st] + c * kBQ * 128, &tmQ, &sm->qd_full[st], x0 + c * 64, sg.q_row0 + i * kBQ);
            tma_load_2d(sm->qd[st] + kBQ * HD * 2 + c * kBQ * 128, &tmDO, &sm->qd_full[st], x0 + c * 64,
                        sg.q_row0 + i * kBQ);
          }
        }
        if (!ok) break;
        if (!asked) ring_ask(&sm->ring);       // a key block without queries
        const int next = ring_answer(&sm->ring, steal_ph, args.n_items, abort_flag, &g_bwd_err,
                                     ERR_TIMEOUT_PRODUCER);
        if (next >= 0) {
          // The next item's K/V tiles (loaded once the current item's MMAs
          // release K/V) and its first Q/dO block into L2 now, a few query
          // blocks early, so that those loads hit L2.
          const BwdWork nw = decode_bwd(args, next);
          const BwdSeg& ns = args.segs[nw.seg];
          const int nx0 = nw.h * HD;
          const int nqb_next = (ns.q_len + kBQ - 1) / kBQ;
          const int q_first = ns.q_row0 + (nw.kb % nqb_next) * kBQ;
#pragma unroll
          for (int c = 0; c < HD / 64; ++c) {
            tma_prefetch_l2_2d(&tmK, nx0 + c * 64, ns.k_row0 + nw.kb * kBlockN);
            tma_prefetch_l2_2d(&tmV, nx0 + c * 64, ns.k_row0 + nw.kb * kBlockN);
            tma_prefetch_l2_2d(&tmQ, nx0 + c * 64, q_first);
            tma_prefetch_l2_2d(&tmDO, nx0 + c * 64, q_first);
          }
        }
        if (next == -2 ||
            !ring_publish(&sm->ring, n, next, abort_flag, &g_bwd_err, ERR_TIMEOUT_PRODUCER) || next < 0)
          break;
        it = static_cast<uint32_t>(next);
      }
    }
  } else if (warp == kMmaWarpA || warp == kMmaWarpB) {
    // ------------------------------------------------------------ MMA issuers A and B
    // A: S^T_g = K Q_g^T -> S[g % 2], then dV += P^T dO_g (P^T read from S[g % 2]).
    // B: dP^T_g = V dO_g^T -> DP, then dK += dS^T Q_g (dS^T read from shared memory).
    // Each issues the S^T (or dP^T) of block g+1 before the accumulation of
    // block g, so the softmax-grad of g+1 can start while g accumulates.
    if (lane == 0) {
      const bool is_a = warp == kMmaWarpA;
      constexpr uint32_t idesc_s = idesc_bf16(kBlockN, kBQ, false, false);   // M128 N64
      constexpr uint32_t idesc_acc = idesc_bf16(kBlockN, HD, false, true);   // dV, dK
      const uint32_t a_op = smem_u32(is_a ? sm->k : sm->v);                   // K for S^T, V for dP^T
      const uint32_t err = ERR_TIMEOUT_MMA;
      uint32_t item_it = 0, g0 = 0;
      bool ok = true;
      // S^T (A) or dP^T (B) of block gg into S[gg % 2] or DP.
      auto issue_first = [&](uint32_t gg) -> bool {
        const uint32_t b = gg & 1u;
        const uint32_t st = gg % kQdStages;
        if (!mbar_wait(&sm->qd_full[st], (gg / kQdStages) & 1u, abort_flag, &g_bwd_err, err)) return false;
        // B: the softmax-grad warps must have loaded dP^T of block gg-1
        if (!is_a && gg > 0 && !mbar_wait(&sm->dp_free, (gg - 1) & 1u, abort_flag, &g_bwd_err, err)) return false;
        tc_fence_after();
        const uint32_t b_op = smem_u32(sm->qd[st]) + (is_a ? 0u : static_cast<uint32_t>(kBQ * HD * 2));
        const uint32_t t_out = is_a ? tmem + 64u * b : tDP;
#pragma unroll
        for (int ks = 0; ks < HD / 16; ++ks) {
          const uint32_t ka = (ks >> 2) * (kBlockN * 128) + (ks & 3) * 32;
          const uint32_t qa = (ks >> 2) * (kBQ * 128) + (ks & 3) * 32;
          umma_ss(t_out, sdesc_sw128(a_op + ka, 16, 1024), sdesc_sw128(b_op + qa, 16, 1024), idesc_s,
                  ks > 0 ? 1u : 0u);
        }
        umma_commit(&sm->s_full[b]);
        return true;
      };
      for (uint32_t n = 0; ok; ++n, ++item_it) {
        const int it = ring_take(&sm->ring, n, abort_flag, &g_bwd_err, err, false);
        if (it < 0) break;
        const BwdWork w = decode_bwd(args, it);
        const BwdSeg& sg = args.segs[w.seg];
        const uint32_t nqb = static_cast<uint32_t>((sg.q_len + kBQ - 1) / kBQ);
        if (!mbar_wait(&sm->kv_full, item_it & 1u, abort_flag, &g_bwd_err, err) || !issue_first(g0)) {
          ok = false;
          break;
        }
        for (uint32_t ii = 0; ii < nqb; ++ii) {
          const uint32_t gg = g0 + ii;
          const uint32_t b = gg & 1u;
          const uint32_t st = gg % kQdStages;
          if (ii + 1 < nqb && !issue_first(gg + 1)) {
            ok = false;
            break;
          }
          if (!mbar_wait(&sm->sg_done[b], (gg >> 1) & 1u, abort_flag, &g_bwd_err, err) ||
              (ii == 0 && !mbar_wait(&sm->dkdv_drained, (item_it & 1u) ^ 1u, abort_flag, &g_bwd_err, err))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t acc0 = ii > 0 ? 1u : 0u;
          if (is_a) {
            // dV: A = P^T in S[b] (TMEM), B = dO_g (MN-major)
            const uint32_t do_op = smem_u32(sm->qd[st]) + static_cast<uint32_t>(kBQ * HD * 2);
#pragma unroll
            for (int ks = 0; ks < kBQ / 16; ++ks) {
              umma_ts(tDV, tmem + 64u * b + op_col(ks), sdesc_sw128(do_op + ks * 2048, kBQ * 128, 1024),
                      idesc_acc, acc0 | (ks > 0 ? 1u : 0u));
            }
          } else {
            // dK: A = dS^T as [key][query] rows (K-major), B = Q_g (MN-major)
            const uint32_t ds_op = smem_u32(sm->ds[b]);
            const uint32_t q_op = smem_u32(sm->qd[st]);
#pragma unroll
            for (int ks = 0; ks < kBQ / 16; ++ks) {
              umma_ss(tDK, sdesc_sw128(ds_op + ks * 32, 16, 1024), sdesc_sw128(q_op + ks * 2048, kBQ * 128, 1024),
                      idesc_acc, acc0 | (ks > 0 ? 1u : 0u));
            }
            umma_commit(&sm->ds_free[b]);
          }
          umma_commit(&sm->qd_read[st]);
        }
        if (!ok) break;
        g0 += nqb;
        umma_commit(&sm->dkdv_full);
        umma_commit(&sm->kv_empty);
      }
    }
  } else if (warp == kMmaWarpC) {
    // ------------------------------------------------------------ MMA issuer C
    // dQ_g^T = K^T dS_g^T into DQ once the drain warps have read the previous
    // block's dQ^T out of it.  A = K as MN-major (d on M; for d = 64 the upper
    // 64 rows read the V tile and are never drained), B = dS MN-major.
    if (lane == 0) {
      constexpr uint32_t idesc_dq = idesc_bf16(128, kBQ, true, true);        // M128 N64
      const uint32_t k_addr = smem_u32(sm->k);
      uint32_t item_it = 0, g = 0;
      bool ok = true;
      for (uint32_t n = 0; ok; ++n, ++item_it) {
        const int it = ring_take(&sm->ring, n, abort_flag, &g_bwd_err, ERR_TIMEOUT_MMA, false);
        if (it < 0) break;
        const BwdWork w = decode_bwd(args, it);
        const BwdSeg& sg = args.segs[w.seg];
        const int nqb = (sg.q_len + kBQ - 1) / kBQ;
        if (!mbar_wait(&sm->kv_full, item_it & 1u, abort_flag, &g_bwd_err, ERR_TIMEOUT_MMA)) {
          ok = false;
          break;
        }
        for (int ii = 0; ii < nqb; ++ii, ++g) {
          const uint32_t b = g & 1u;
          if (!mbar_wait(&sm->sg_done[b], (g >> 1) & 1u, abort_flag, &g_bwd_err, ERR_TIMEOUT_MMA) ||
              (g > 0 && !mbar_wait(&sm->dq_drained, (g - 1) & 1u, abort_flag, &g_bwd_err, ERR_TIMEOUT_MMA))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t ds_addr = smem_u32(sm->ds[b]);
#pragma unroll
          for (int ks = 0; ks < kBlockN / 16; ++ks) {
            umma_ss(tDQ, sdesc_sw128(k_addr + ks * 2048, kBlockN * 128, 1024),
                    sdesc_sw128(ds_addr + ks * 2048, 16, 1024), idesc_dq, ks > 0 ? 1u : 0u);
          }
          umma_commit(&sm->dq_full);
          umma_commit(&sm->ds_free[b]);
        }
        if (!ok) break;
        umma_commit(&sm->kv_empty);
      }
    }
  } else if (warp >= kDrainWarp0) {
    // ------------------------------------------------------------ dQ drain
    // Lane l of drain warp dw holds dQ^T row d = 32 dw + l for the block's 64
    // queries.  Rows past the sequence carry exact zeros (P = 0 there).
    const int dw = warp - kDrainWarp0;                 // TMEM lane quadrant = d / 32
    const uint32_t lane_off = static_cast<uint32_t>(dw * 32) << 16;
    const bool active = dw * 32 < HD;
    const int nh = args.num_heads;
    uint32_t g = 0, item_it = 0;
    bool ok = true;
    for (uint32_t n = 0; ok; ++n, ++item_it) {
      const int it = ring_take(&sm->ring, n, abort_flag, &g_bwd_err, ERR_TIMEOUT_OTHER, true);
      if (it < 0) break;
      const BwdWork w = decode_bwd(args, it);
      const BwdSeg& sg = args.segs[w.seg];
      const int nqb = (sg.q_len + kBQ - 1) / kBQ;
      const int start = w.kb % nqb;
      for (int ii = 0; ii < nqb; ++ii, ++g) {
        const int i = (start + ii) % nqb;
        if (!__all_sync(0xffffffffu,
                        mbar_wait(&sm->dq_full, g & 1u, abort_flag, &g_bwd_err, ERR_TIMEOUT_OTHER))) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t v0[32], v1[32];
        tmem_ld32(tDQ + lane_off, v0);
        tmem_ld32(tDQ + lane_off + 32, v1);
        tmem_wait_ld();
        reg_fence(v0);
        reg_fence(v1);
        tc_fence_before();
        mbar_arrive(&sm->dq_drained);
        const uint32_t st = g % kQdStages;
        if (!active) {
          if (lane == 0) mbar_arrive(&sm->qd_empty[st]);
          continue;
        }
        // dV and dK (issuers A, B) may still be reading dO_i / Q_i out of this stage
        if (!__all_sync(0xffffffffu, mbar_wait(&sm->qd_read[st], (g / kQdStages) & 1u, abort_flag, &g_bwd_err,
                                               ERR_TIMEOUT_OTHER))) {
          ok = false;
          break;
        }
        // This warp's box in the dead Q_i/dO_i stage: [64 query rows][32 d
        // floats], 16-byte chunk c of row r at c ^ (r & 7).
        uint8_t* box = sm->qd[st] + dw * (kBQ * 128);
        const uint32_t cl = static_cast<uint32_t>(lane) >> 2;
        const uint32_t wl = (static_cast<uint32_t>(lane) & 3u) * 4;
#pragma unroll
        for (int r = 0; r < 32; ++r) {
          *reinterpret_cast<uint32_t*>(box + r * 128 + ((cl ^ (r & 7)) << 4) + wl) = v0[r];
          *reinterpret_cast<uint32_t*>(box + (r + 32) * 128 + ((cl ^ (r & 7)) << 4) + wl) = v1[r];
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_reduce_add_2d(&tmDQ, box, w.h * HD + 32 * dw, sg.q_row0 + i * kBQ);
          bulk_commit_group();
          bulk_wait_group_read0();           // box read: the stage may be refilled
          mbar_arrive(&sm->qd_empty[st]);
        }
      }
      if (!ok) break;
      // ------------------------------------------------ dV, dK of the key block
      // Lane l of drain warp dw holds key row 32 dw + l of both accumulators;
      // the next item's first dV / dK MMAs wait until all 128 rows are read.
      if (!__all_sync(0xffffffffu,
                      mbar_wait(&sm->dkdv_full, item_it & 1u, abort_flag, &g_bwd_err, ERR_TIMEOUT_OTHER))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int jrow = dw * 32 + lane;
      const bool kv_ok = w.kb * kBlockN + jrow < sg.k_len;
      const size_t krow = static_cast<size_t>(sg.k_row0) + static_cast<size_t>(w.kb * kBlockN + jrow);
      __nv_bfloat16* dv_dst = reinterpret_cast<__nv_bfloat16*>(args.dv) + (krow * nh + w.h) * HD;
      __nv_bfloat16* dk_dst = reinterpret_cast<__nv_bfloat16*>(args.dk) + (krow * nh + w.h) * HD;
      const float sc = args.scale;
#pragma unroll 1
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t a[32], bb[32];
        tmem_ld32(tDV + lane_off + 32 * c, a);
        tmem_ld32(tDK + lane_off + 32 * c, bb);
        tmem_wait_ld();
        reg_fence(a);
        reg_fence(bb);
        if (kv_ok) {
          uint4* dv4 = reinterpret_cast<uint4*>(dv_dst + 32 * c);
          uint4* dk4 = reinterpret_cast<uint4*>(dk_dst + 32 * c);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            dv4[e] = make_uint4(pack_bf16x2(__uint_as_float(a[8 * e + 0]), __uint_as_float(a[8 * e + 1])),
                                pack_bf16x2(__uint_as_float(a[8 * e + 2]), __uint_as_float(a[8 * e + 3])),
                                pack_bf16x2(__uint_as_float(a[8 * e + 4]), __uint_as_float(a[8 * e + 5])),
                                pack_bf16x2(__uint_as_float(a[8 * e + 6]), __uint_as_float(a[8 * e + 7])));
            dk4[e] = make_uint4(
                pack_bf16x2(__uint_as_float(bb[8 * e + 0]) * sc, __uint_as_float(bb[8 * e + 1]) * sc),
                pack_bf16x2(__uint_as_float(bb[8 * e + 2]) * sc, __uint_as_float(bb[8 * e + 3]) * sc),
                pack_bf16x2(__uint_as_float(bb[8 * e + 4]) * sc, __uint_as_float(bb[8 * e + 5]) * sc),
                pack_bf16x2(__uint_as_float(bb[8 * e + 6]) * sc, __uint_as_float(bb[8 * e + 7]) * sc));
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&sm->dkdv_drained);
    }
    if (lane == 0) bulk_wait_group0();        // the additions must land before exit
  } else {
    // ------------------------------------------------------------ softmax-grad
    const int w4 = warp & 3;
    const int half = warp >> 2;
    const uint32_t lane_off = static_cast<uint32_t>(w4 * 32) << 16;
    const int jrow = w4 * 32 + lane;        // key row within the block
    const float sl2 = args.scale_log2;
    uint32_t g = 0;
    bool ok = true;
    for (uint32_t n = 0; ok; ++n) {
      const int it = ring_take(&sm->ring, n, abort_flag, &g_bwd_err, ERR_TIMEOUT_SOFTMAX, true);
      if (it < 0) break;
      const BwdWork w = decode_bwd(args, it);
      const BwdSeg& sg = args.segs[w.seg];
      const int nqb = (sg.q_len + kBQ - 1) / kBQ;
      const int start = w.kb % nqb;
      const bool kv_ok = w.kb * kBlockN + jrow < sg.k_len;
      float pref = staged_value(args, sg, w.h, start, threadIdx.x);
      for (int ii = 0; ii < nqb; ++ii, ++g) {
        const uint32_t b = g & 1u;
        // stage LSE*log2e and D of this block; prefetch the next block's
        if (threadIdx.x < kBQ) sm->lse2[b][threadIdx.x] = pref;
        else if (threadIdx.x < 2 * kBQ) sm->dsum[b][threadIdx.x - kBQ] = pref;
        mbar_arrive(&sm->stage_full);
        if (ii + 1 < nqb) pref = staged_value(args, sg, w.h, (start + ii + 1) % nqb, threadIdx.x);
        if (!__all_sync(0xffffffffu,
                        mbar_wait(&sm->stage_full, g & 1u, abort_flag, &g_bwd_err, ERR_TIMEOUT_SOFTMAX)) ||
            !__all_sync(0xffffffffu,
                        mbar_wait(&sm->s_full[b], (g >> 1) & 1u, abort_flag, &g_bwd_err, ERR_TIMEOUT_SOFTMAX))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tS = tmem + 64 * b + lane_off + 32 * half;
        uint32_t s[32], dp[32];
        tmem_ld32(tS, s);
        tmem_ld32(tDP + lane_off + 32 * half, dp);
        tmem_wait_ld();
        reg_fence(s);
        reg_fence(dp);
        tc_fence_before();
        mbar_arrive(&sm->dp_free);             // dP^T of the next block may overwrite DP
        const float* l2 = sm->lse2[b] + 32 * half;
        const float* dsm = sm->dsum[b] + 32 * half;
        uint32_t pp[16], dd[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float2 lv = *reinterpret_cast<const float2*>(l2 + 2 * e);
          const float2 dv = *reinterpret_cast<const float2*>(dsm + 2 * e);
          float p0 = fast_exp2(fmaf(__uint_as_float(s[2 * e]), sl2, -lv.x));
          float p1 = fast_exp2(fmaf(__uint_as_float(s[2 * e + 1]), sl2, -lv.y));
          if (!kv_ok) {
            p0 = 0.f;
            p1 = 0.f;
          }
          const float d0 = p0 * (__uint_as_float(dp[2 * e]) - dv.x);
          const float d1 = p1 * (__uint_as_float(dp[2 * e + 1]) - dv.y);
          pp[e] = pack_bf16x2(p0, p1);
          dd[e] = pack_bf16x2(d0, d1);
        }
        tmem_st16(tS, pp);
        // dS of block g-2 must have been read by dK and dQ^T before it is overwritten
        if (!__all_sync(0xffffffffu, g < 2 || mbar_wait(&sm->ds_free[b], ((g - 2) >> 1) & 1u, abort_flag,
                                                         &g_bwd_err, ERR_TIMEOUT_SOFTMAX))) {
          ok = false;
          break;
        }
        uint8_t* ds_row = sm->ds[b] + jrow * 128;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int chunk = half * 4 + c;
          *reinterpret_cast<uint4*>(ds_row + ((chunk ^ (jrow & 7)) << 4)) =
              make_uint4(dd[4 * c], dd[4 * c + 1], dd[4 * c + 2], dd[4 * c + 3]);
        }
        fence_proxy_async_smem();
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&sm->sg_done[b]);
      }
      if (!ok) break;
    }
  }

  // ---------------------------------------------------------------- teardown
  __syncwarp();
  if (*abort_flag) drain_delay(2000000ull);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarpA) tmem_dealloc(tmem, kTmemCols);
}

template <int HD>
cudaError_t launch_hd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                      const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdArgs& args,
                      cudaStream_t stream) {
  const size_t smem = sizeof(BwdSmem<HD>) + 1024;
  cudaError_t e = cudaFuncSetAttribute(bwd_tc_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  bwd_tc_kernel<HD><<<args.n_items, kBwdThreads, smem, stream>>>(tq, tk, tv, tdo, tdq, args);
  return cudaGetLastError();
}

}  // namespace

int bwd_query_block() { return kBQ; }

size_t bwd_tc_smem_bytes(int head_dim) {
  return head_dim == 64 ? sizeof(BwdSmem<64>) + 1024 : sizeof(BwdSmem<128>) + 1024;
}

cudaError_t launch_bwd_tc(int head_dim, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdq,
                          const BwdArgs& args, cudaStream_t stream) {
  if (head_dim == 64) return launch_hd<64>(tq, tk, tv, tdo, tdq, args, stream);
  if (head_dim == 128) return launch_hd<128>(tq, tk, tv, tdo, tdq, args, stream);
  return cudaErrorInvalidValue;
}

uint32_t bwd_take_error() {
  uint32_t v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_bwd_err, sizeof(v)) != cudaSuccess) return 0xFFFFFFFFu;
  if (v != 0) cudaMemcpyToSymbol(g_bwd_err, &zero, sizeof(zero));
  return v;
}

}  // namespace zl
