// Forward of coalesced varlen attention on sm_103a tensor cores.
//
// One persistent launch runs every work item of the batch: a work item is
// (segment, head, pair of 128-row query tiles), where a segment is a whole
// sequence or one shard tile of a split sequence (Zellige, arXiv
// 2608.01150v1, §IV-D: whole sequences packed into one block-diagonal call,
// shards alongside them).  Items arrive ordered longest-first from the host
// scheduler.  The grid holds one CTA per item, of which one per SM is
// resident; a resident CTA takes its own item first and then steals the
// next unstarted one from the launch queue (cluster launch control), so an
// SM that finishes early picks up the next item in longest-first order.
//
// The two query tiles of an item share every K_j / V_j tile that the producer
// brings into shared memory.  Per CTA (352 threads):
//   warp 8      TMA producer: K_0, the two Q tiles once per item, then V_0
//               and the further K_j / V_j through a four-stage ring (128-byte
//               swizzle, 64-column boxes).
//               It also steals the next item and hands it to the other roles
//               through a two-slot ring in shared memory.
//   warps 9,10  MMA issuers, one thread each, one per query tile t:
//               S_t = Q_t K_j^T (SS, M=128 N=128) into TMEM, then
//               O_t += P_t V_j (TS: P read from TMEM, V from shared memory as
//               an MN-major operand) into TMEM.  One issuing thread per tile,
//               so each tile's MMAs go out as soon as its own softmax hands
//               over, whatever the other tile is doing.
//   warps 0-7   softmax, warpgroup t for tile t: thread r of the group owns
//               query row r = TMEM lane r.  Loads its S row, tracks the
//               running max m and sum l in base 2, writes
//               P = 2^(S*scale*log2e - m) as bf16 over the S columns, and
//               rescales the O row in TMEM when m grows by more than 2^8
//               (lazy rescale; exactness holds for any m used consistently).
//               After the last block it normalises O and writes O and LSE:
//               a full 128-row tile of final rows is staged in the tile's
//               own Q buffer (dead after the item's last S MMAs) and stored
//               with TMA, and the producer loads the next item's Q there once
//               the store has read it; partial tiles and shard partials are
//               stored per thread.
//   The two warpgroups take turns (an mbarrier per group, handed back and
//   forth): the exponentials of one tile run while the tensor cores work on
//   the other tile, instead of both groups competing for the SFU while the
//   tensor pipe idles.
// TMEM: tile t uses S/P in columns [256t, 256t+128) and O in
// [256t+128, 256t+128+d); 512 columns.
//
// Whole sequences write O in bf16 and LSE in natural log.  Tiles write their
// partial O (float32, or bf16 when args.part_bf16) and their own LSE into a
// partial slot for the merge kernel; with
// the fused merge they then count themselves in an arrival counter per
// (query block, head) of their query chunk, and the warpgroup that brings the
// count to the number of kv chunks merges all partials of those 128 rows into
// O and LSE exactly (no waiting: every other partial is complete and fenced).
// Waiting warps (softmax groups between turns, issuers between blocks) let
// the hardware suspend them for up to 10 us per try_wait instead of its
// default limit: fewer polls of the barriers, 1-2% faster on every workload.
#define ZL_TRY_WAIT_HINT_NS 10000
#include "common.cuh"
#include "launch.h"
#include "work.cuh"

namespace zl {
namespace {

__device__ uint32_t g_fwd_err;

constexpr int kFwdThreads = 352;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp0 = 9;                 // tile 0; tile 1 is kMmaWarp0 + 1
constexpr int kFwdStages = 4;
constexpr int kItemReaders = 10;             // 2 issuer threads + 8 softmax warps
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;   // in log2 units: P <= 2^8
constexpr float kLn2 = 0.6931471805599453f;

template <int HD>
struct FwdSmem {
  uint8_t q[2][kBlockM * HD * 2];              // per tile: HD/64 boxes of [128 rows][128 B]
  uint8_t kv[kFwdStages][kBlockN * HD * 2];    // K_j or V_j, same box layout
  uint64_t q_full[2], q_empty[2];
  uint64_t kv_full[kFwdStages], kv_empty[kFwdStages];
  uint64_t s_full[2], p_full[2], o_full[2];
  uint64_t turn[2];                            // softmax group t may run its next block
  uint64_t grp_sync[2];                        // barrier of softmax group t's 128 threads
  uint32_t grp_uses[2][128];                   // per thread: its earlier arrivals on grp_sync[t]
  ItemRing ring;                               // work items, producer -> the other roles
  uint32_t tmem_base;
  int abort_flag;
  int is_last[2];                              // group t completed a row block's partials
};

// Merges the n_kv float32 partials of one query row of a tile (all written
// and fenced by their CTAs) into the bf16 output and the LSE:
//     lse = log sum_j exp(lse_j),  o = sum_j exp(lse_j - lse) o_j.
template <int HD>
__device__ __forceinline__ void merge_tile_row(const FwdArgs& a, const FwdSeg& sg, int h, int q_local) {
  const int64_t nh = a.num_heads;
  const size_t prow = static_cast<size_t>(sg.out_row0 + q_local);
  float m = -INFINITY;
  for (int j = 0; j < sg.n_kv; ++j)
    m = fmaxf(m, __ldcg(a.lse_part + (static_cast<size_t>(j) * nh + h) * a.part_rows + prow));
  float sum = 0.f;
  for (int j = 0; j < sg.n_kv; ++j)
    sum += expf(__ldcg(a.lse_part + (static_cast<size_t>(j) * nh + h) * a.part_rows + prow) - m);
  const float inv = 1.f / sum;
  __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(a.o) + (static_cast<size_t>(sg.q_row0 + q_local) * nh + h) * HD;
#pragma unroll 1
  for (int c = 0; c < HD / 32; ++c) {
    float acc[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) acc[e] = 0.f;
    for (int j = 0; j < sg.n_kv; ++j) {
      const float wj = expf(__ldcg(a.lse_part + (static_cast<size_t>(j) * nh + h) * a.part_rows + prow) - m) * inv;
      const size_t off = ((static_cast<size_t>(j) * a.part_rows + prow) * nh + h) * HD + c * 32;
      if (a.part_bf16) {
        const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(a.o_part) + off);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const uint4 x = __ldcg(src + v);
          const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = bf16x2_to_float2(w4[e]);
            acc[8 * v + 2 * e] = fmaf(wj, f.x, acc[8 * v + 2 * e]);
            acc[8 * v + 2 * e + 1] = fmaf(wj, f.y, acc[8 * v + 2 * e + 1]);
          }
        }
      } else {
        const float4* src = reinterpret_cast<const float4*>(a.o_part + off);
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const float4 x = __ldcg(src + v);
          acc[4 * v + 0] = fmaf(wj, x.x, acc[4 * v + 0]);
          acc[4 * v + 1] = fmaf(wj, x.y, acc[4 * v + 1]);
          acc[4 * v + 2] = fmaf(wj, x.z, acc[4 * v + 2]);
          acc[4 * v + 3] = fmaf(wj, x.w, acc[4 * v + 3]);
        }
      }
    }
    uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
    for (int v = 0; v < 4; ++v)
      d4[v] = make_uint4(pack_bf16x2(acc[8 * v + 0], acc[8 * v + 1]), pack_bf16x2(acc[8 * v + 2], acc[8 * v + 3]),
                         pack_bf16x2(acc[8 * v + 4], acc[8 * v + 5]), pack_bf16x2(acc[8 * v + 6], acc[8 * v + 7]));
  }
  a.lse[static_cast<size_t>(h) * a.lse_stride + sg.q_row0 + q_local] = m + logf(sum);
}

// Spin for about `ns` nanoseconds: lets copies and MMAs already in flight land
// before an aborting CTA releases its shared memory and TMEM.
__device__ __forceinline__ void drain_delay(uint64_t ns) {
  const uint64_t t0 = globaltimer();
  while (globaltimer() - t0 < ns) {
  }
}

// Does query tile t (0 or 1) of this item hold any row of the segment?
__device__ __forceinline__ bool tile_present(const FwdSeg& sg, const FwdWork& w, int t) {
  return (2 * w.qb + t) * kBlockM < sg.q_len;
}

// Registers are granted per group of four warps, so 352 threads leave at
// most 168 registers per thread.
template <int HD>
__global__ void __launch_bounds__(kFwdThreads, 1)
fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
              const __grid_constant__ FwdArgs args) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  auto* sm = reinterpret_cast<FwdSmem<HD>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  volatile int* abort_flag = &sm->abort_flag;

  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(&sm->q_full[t], 1);
      mbar_init(&sm->q_empty[t], 2);           // the item's last S MMAs, and the epilogue done with q[t]
      mbar_init(&sm->s_full[t], 1);
      mbar_init(&sm->p_full[t], 128);
      mbar_init(&sm->o_full[t], 1);
      mbar_init(&sm->turn[t], 128);
      mbar_init(&sm->grp_sync[t], 128);
    }
    for (int s = 0; s < kFwdStages; ++s) {
      mbar_init(&sm->kv_full[s], 1);
      mbar_init(&sm->kv_empty[s], 2);          // both issuers are done with the stage
    }
    ring_init(&sm->ring, kItemReaders);
    sm->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp0) {
    tmem_alloc(&sm->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm->tmem_base;

  if (warp == kProducerWarp) {
    if (lane == 0) {
      tma_prefetch_map(&tmQ);
      tma_prefetch_map(&tmK);
      tma_prefetch_map(&tmV);
      uint32_t kv_it = 0;
      uint32_t q_it[2] = {0u, 0u};
      uint32_t steal_ph = 0;
      // the CTA's own item comes first
      bool ok = ring_publish(&sm->ring, 0, static_cast<int>(blockIdx.x), abort_flag, &g_fwd_err,
                             ERR_TIMEOUT_PRODUCER);
      for (uint32_t n = 1, it = blockIdx.x; ok; ++n) {
        const FwdWork w = decode_fwd(args, static_cast<int>(it));
        const FwdSeg& sg = args.segs[w.seg];
        const int nkb = (sg.k_len + kBlockN - 1) / kBlockN;
        const int x0 = w.h * HD;
        bool asked = false;
        // The item's Q tiles, each once the previous item's tile has released
        // its buffer (its last S MMAs and its output store).  Issued after
        // K_0, whose ring stage frees earlier: tile 0's first S then does not
        // wait for tile 1's epilogue of the previous item.
        auto load_q = [&]() {
          for (int t = 0; t < 2 && ok; ++t) {
            if (!tile_present(sg, w, t)) continue;
            if (!mbar_wait(&sm->q_empty[t], (q_it[t] & 1u) ^ 1u, abort_flag, &g_fwd_err, ERR_TIMEOUT_PRODUCER)) {
              ok = false;
              break;
            }
            ++q_it[t];
            mbar_arrive_expect_tx(&sm->q_full[t], kBlockM * HD * 2);
            const int q_row = sg.q_row0 + (2 * w.qb + t) * kBlockM;
#pragma unroll
            for (int c = 0; c < HD / 64; ++c)
              tma_load_2d(sm->q[t] + c * kBlockM * 128, &tmQ, &sm->q_full[t], x0 + c * 64, q_row);
          }
        };
        if (nkb == 0) load_q();
        for (int j = 0; j < nkb && ok; ++j) {
          if (j == nkb - 1) {
            // the item's last K/V tiles are next: ask for the following item
            // now, about two key blocks before the issuers need it
            ring_ask(&sm->ring);
            asked = true;
          }
#pragma unroll
          for (int kv = 0; kv < 2; ++kv) {
            const uint32_t st = kv_it % kFwdStages;
            const uint32_t ph = (kv_it / kFwdStages) & 1u;
            if (!mbar_wait(&sm->kv_empty[st], ph ^ 1u, abort_flag, &g_fwd_err, ERR_TIMEOUT_PRODUCER)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&sm->kv_full[st], kBlockN * HD * 2);
            const CUtensorMap* map = kv ? &tmV : &tmK;
#pragma unroll
            for (int c = 0; c < HD / 64; ++c)
              tma_load_2d(sm->kv[st] + c * kBlockN * 128, map, &sm->kv_full[st], x0 + c * 64,
                          sg.k_row0 + j * kBlockN);
            ++kv_it;
            if (j == 0 && kv == 0) {
              load_q();
              if (!ok) break;
            }
          }
        }
        if (!ok) break;
        if (!asked) ring_ask(&sm->ring);       // an item without keys
        const int next = ring_answer(&sm->ring, steal_ph, args.n_items, abort_flag, &g_fwd_err,
                                     ERR_TIMEOUT_PRODUCER);
        if (next >= 0) {
          // The next item's Q tiles and first K/V tiles into L2 now, about two
          // key blocks before they are loaded (Q once the current item's last
          // S MMAs are done, K/V as ring stages free up), so those loads hit L2.
          const FwdWork nw = decode_fwd(args, next);
          const FwdSeg& ns = args.segs[nw.seg];
          const int nx0 = nw.h * HD;
#pragma unroll
          for (int c = 0; c < HD / 64; ++c) {
            for (int t = 0; t < 2; ++t)
              if (tile_present(ns, nw, t))
                tma_prefetch_l2_2d(&tmQ, nx0 + c * 64, ns.q_row0 + (2 * nw.qb + t) * kBlockM);
            tma_prefetch_l2_2d(&tmK, nx0 + c * 64, ns.k_row0);
            tma_prefetch_l2_2d(&tmV, nx0 + c * 64, ns.k_row0);
          }
        }
        if (next == -2 ||
            !ring_publish(&sm->ring, n, next, abort_flag, &g_fwd_err, ERR_TIMEOUT_PRODUCER) || next < 0)
          break;
        it = static_cast<uint32_t>(next);
      }
    }
  } else if (warp == kMmaWarp0 || warp == kMmaWarp0 + 1) {
    // ------------------------------------------------------------ MMA issuer of tile t
    // Every K/V stage is released by both issuers, also by the issuer of an
    // absent tile 1 (which waits for each stage to fill, so it can never
    // release a stage twice within one fill).
    if (lane == 0) {
      const int t = warp - kMmaWarp0;
      constexpr uint32_t idesc_qk = idesc_bf16(kBlockM, kBlockN, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16(kBlockM, HD, false, true);
      // Operand descriptors: the start-address field holds (address >> 4), so
      // the descriptor of a k-step is the tile's base descriptor plus the
      // step's byte offset >> 4 (no carry: shared addresses stay below 256 KB).
      // Building them this way keeps the issuing thread's per-MMA work short.
      const uint64_t q_desc = sdesc_sw128(smem_u32(sm->q[t]), 16, 1024);
      const uint32_t tS = tmem + 256u * t;
      const uint32_t tO = tS + 128u;
      uint32_t kv_it = 0, q_it = 0, blk_it = 0;
      bool ok = true;
      for (uint32_t n = 0; ok; ++n) {
        const int it = ring_take(&sm->ring, n, abort_flag, &g_fwd_err, ERR_TIMEOUT_MMA, false);
        if (it < 0) break;
        const FwdWork w = decode_fwd(args, it);
        const FwdSeg& sg = args.segs[w.seg];
        const int nkb = (sg.k_len + kBlockN - 1) / kBlockN;
        const bool has = tile_present(sg, w, t);
        if (has && !mbar_wait(&sm->q_full[t], q_it & 1u, abort_flag, &g_fwd_err, ERR_TIMEOUT_MMA)) {
          ok = false;
          break;
        }
        for (int j = 0; j < nkb; ++j) {
          // S_t = Q_t K_j^T
          uint32_t st = kv_it % kFwdStages;
          uint32_t ph = (kv_it / kFwdStages) & 1u;
          if (!mbar_wait(&sm->kv_full[st], ph, abort_flag, &g_fwd_err, ERR_TIMEOUT_MMA)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (has) {
            const uint64_t k_desc = sdesc_sw128(smem_u32(sm->kv[st]), 16, 1024);
#pragma unroll
            for (int ks = 0; ks < HD / 16; ++ks) {
              const uint64_t off16 = ((ks >> 2) * (kBlockM * 128) + (ks & 3) * 32) >> 4;
              umma_ss(tS, q_desc + off16, k_desc + off16, idesc_qk, ks > 0 ? 1u : 0u);
            }
            umma_commit(&sm->s_full[t]);
            // Q_t is read by S MMAs only: after the item's last one the
            // producer may bring the next item's Q_t
            if (j == nkb - 1) umma_commit(&sm->q_empty[t]);
          }
          umma_commit(&sm->kv_empty[st]);
          ++kv_it;
          // O_t += P_t V_j once softmax group t has written P_t (and rescaled O_t)
          st = kv_it % kFwdStages;
          ph = (kv_it / kFwdStages) & 1u;
          if (!mbar_wait(&sm->kv_full[st], ph, abort_flag, &g_fwd_err, ERR_TIMEOUT_MMA) ||
              (has && !mbar_wait(&sm->p_full[t], blk_it & 1u, abort_flag, &g_fwd_err, ERR_TIMEOUT_MMA))) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (has) {
            const uint64_t v_desc = sdesc_sw128(smem_u32(sm->kv[st]), kBlockN * 128, 1024);
#pragma unroll
            for (int ks = 0; ks < kBlockN / 16; ++ks) {
              umma_ts(tO, tS + ks * 8, v_desc + static_cast<uint64_t>(ks * (2048 >> 4)), idesc_pv,
                      (j > 0 || ks > 0) ? 1u : 0u);
            }
            ++blk_it;
          }
          umma_commit(&sm->kv_empty[st]);
          ++kv_it;
        }
        if (!ok) break;
        if (has) {
          umma_commit(&sm->o_full[t]);
          ++q_it;
        }
      }
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ softmax group t
    const int t = warp >> 2;
    const int row = (warp & 3) * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + 256u * t;
    const uint32_t tO = tS + 128u;
    const float sl2 = args.scale_log2;
    const int nh = args.num_heads;
    uint32_t blk_it = 0, q_it = 0, turn_it = 0;
    // this thread's count of grp_sync[t] phases, kept in shared memory so it
    // takes no register across the block loop
    sm->grp_uses[t][row] = 0;
    // group 1 hands the first turn to group 0
    if (t == 1) mbar_arrive(&sm->turn[0]);
    for (uint32_t n = 0;; ++n) {
      const int it = ring_take(&sm->ring, n, abort_flag, &g_fwd_err, ERR_TIMEOUT_SOFTMAX, true);
      if (it < 0) break;
      const FwdWork w = decode_fwd(args, it);
      const FwdSeg& sg = args.segs[w.seg];
      const int nkb = (sg.k_len + kBlockN - 1) / kBlockN;
      const bool has = tile_present(sg, w, t);
      float m_run = -INFINITY;
      float l_run = 0.f;
      bool ok = true;
      for (int j = 0; j < nkb; ++j, ++turn_it) {
        // all lanes must agree before the warp-wide tcgen05.ld below
        if (!__all_sync(0xffffffffu,
                        (!has || mbar_wait(&sm->s_full[t], blk_it & 1u, abort_flag, &g_fwd_err,
                                           ERR_TIMEOUT_SOFTMAX)) &&
                            mbar_wait(&sm->turn[t], turn_it & 1u, abort_flag, &g_fwd_err, ERR_TIMEOUT_SOFTMAX))) {
          ok = false;
          break;
        }
        if (!has) {
          mbar_arrive(&sm->turn[t ^ 1]);
          continue;
        }
        tc_fence_after();
        uint32_t s[4][32];
        const int valid = sg.k_len - j * kBlockN;
        float m_raw;
        // Speculation on a full block after the first: the exponentials of
        // the first 32 columns are computed with the running max while the
        // other 96 columns load.  They stand if the block does not raise the
        // max past the lazy-rescale threshold (the running max is then kept,
        // exactly as without speculation); otherwise the block is redone from
        // TMEM, where S is still intact.
        bool spec_done = false;
        uint32_t p0[16];
        uint64_t acc[2] = {0ull, 0ull};
        if (valid >= kBlockN) {
          // full block: the reducing TMEM load returns each 32-column max
          float r[4];
          r[0] = tmem_ld32_max(tS + lane_off, s[0]);
          tmem_wait_ld();
          reg_fence(s[0]);
          reg_fence_f(r[0]);
#pragma unroll
          for (int c = 1; c < 4; ++c) r[c] = tmem_ld32_max(tS + lane_off + c * 32, s[c]);
          const bool spec = j > 0 && __all_sync(0xffffffffu, r[0] * sl2 <= m_run + kRescaleThreshold);
          if (spec) {
            const uint64_t sl2x2 = f2_pack(sl2, sl2);
            const uint64_t negm2 = f2_pack(-m_run, -m_run);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const uint64_t x = f2_fma(f2_pack(__uint_as_float(s[0][2 * i]), __uint_as_float(s[0][2 * i + 1])),
                                        sl2x2, negm2);
              float x0, x1;
              f2_unpack(x, x0, x1);
              const float a = fast_exp2(x0);
              const float b = fast_exp2(x1);
              acc[i & 1] = f2_add(acc[i & 1], f2_pack(a, b));
              p0[i] = pack_bf16x2(a, b);
            }
          }
          tmem_wait_ld();
#pragma unroll
          for (int c = 1; c < 4; ++c) {
            reg_fence(s[c]);
            reg_fence_f(r[c]);
          }
          m_raw = fmaxf(fmaxf(r[0], r[1]), fmaxf(r[2], r[3]));
          spec_done = spec && __all_sync(0xffffffffu, m_raw * sl2 <= m_run + kRescaleThreshold);
          if (!spec_done) {
            // (rare) the first 32 columns again, for the exact path below
            acc[0] = 0ull;
            acc[1] = 0ull;
            tmem_ld32(tS + lane_off, s[0]);
            tmem_wait_ld();
            reg_fence(s[0]);
          }
        } else {
          // last block of the segment: columns past its keys do not count
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld32(tS + lane_off + c * 32, s[c]);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 4; ++c) reg_fence(s[c]);
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (c * 32 + i >= valid) s[c][i] = __float_as_uint(-INFINITY);
          float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            mx0 = fmax3(mx0, __uint_as_float(s[0][i]), __uint_as_float(s[0][i + 1]));
            mx1 = fmax3(mx1, __uint_as_float(s[1][i]), __uint_as_float(s[1][i + 1]));
            mx2 = fmax3(mx2, __uint_as_float(s[2][i]), __uint_as_float(s[2][i + 1]));
            mx3 = fmax3(mx3, __uint_as_float(s[3][i]), __uint_as_float(s[3][i + 1]));
          }
          m_raw = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
        }
        const float m_blk = m_raw * sl2;
        const float m_new = fmaxf(m_run, m_blk);
        const bool need = m_new > m_run + kRescaleThreshold;
        float alpha = 1.f;
        if (need) {
          alpha = fast_exp2(m_run - m_new);   // 0 on the first block (m_run = -inf)
          m_run = m_new;
        }
        l_run *= alpha;
        const float neg_m = -m_run;
        // exponent arguments and row sums on float32 pairs; each quarter of P
        // goes to TMEM as soon as it is packed, freeing its S registers
        const uint64_t sl2x2 = f2_pack(sl2, sl2);
        const uint64_t negm2 = f2_pack(neg_m, neg_m);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if (c == 0 && spec_done) {
            tmem_st16(tS + lane_off, p0);
            continue;
          }
          uint32_t p[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const uint64_t x = f2_fma(f2_pack(__uint_as_float(s[c][2 * i]), __uint_as_float(s[c][2 * i + 1])),
                                      sl2x2, negm2);
            float x0, x1;
            f2_unpack(x, x0, x1);
            const float a = fast_exp2(x0);
            const float b = fast_exp2(x1);
            acc[i & 1] = f2_add(acc[i & 1], f2_pack(a, b));
            p[i] = pack_bf16x2(a, b);
          }
          tmem_st16(tS + lane_off + 16 * c, p);
        }
        float ls0, ls1;
        f2_unpack(f2_add(acc[0], acc[1]), ls0, ls1);
        // the exponentials are done: the other group may take its turn
        mbar_arrive(&sm->turn[t ^ 1]);
        if (j > 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll 1
          for (int c = 0; c < HD / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + lane_off + c * 32, o);
            tmem_wait_ld();
            reg_fence(o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(tO + lane_off + c * 32, o);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&sm->p_full[t]);
        ++blk_it;
        l_run += ls0 + ls1;
      }
      if (!ok) break;
      if (!has) continue;
      // ---------------------------------------------------------- epilogue
      if (!__all_sync(0xffffffffu,
                      mbar_wait(&sm->o_full[t], q_it & 1u, abort_flag, &g_fwd_err, ERR_TIMEOUT_SOFTMAX)))
        break;
      ++q_it;
      tc_fence_after();
      const int qb = 2 * w.qb + t;             // 128-row query block within the segment
      const int q_local = qb * kBlockM + row;
      const bool row_ok = q_local < sg.q_len;
      const float inv_l = 1.f / l_run;
      const float lse_val = (m_run + log2f(l_run)) * kLn2;
      const bool tma_tile = sg.slot < 0 && (qb + 1) * kBlockM <= sg.q_len;
      // q[t] is free once the item's last S MMAs are done (o_full implies
      // it); the epilogue of a full tile of final rows uses it as the staging
      // area of its TMA store and releases it after the store has read it,
      // any other epilogue releases it at once.
      if (!tma_tile && row == 0) mbar_arrive(&sm->q_empty[t]);
      if (tma_tile) {
        // Each thread packs its row into q[t] in the Q tile's own layout
        // (64-column boxes of [128 rows][128 B], 128-byte swizzle), and one
        // thread stores the boxes with TMA: the rows of a tile are H*d
        // elements apart, so per-thread stores would each touch their own
        // lines.
        const uint32_t r7 = static_cast<uint32_t>(row & 7);
#pragma unroll 1
        for (int c = 0; c < HD / 32; ++c) {
          uint32_t oa[32];
          tmem_ld32(tO + lane_off + c * 32, oa);
          tmem_wait_ld();
          reg_fence(oa);
          uint8_t* box_row = sm->q[t] + (c >> 1) * (kBlockM * 128) + row * 128;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t* src = oa + 8 * k;
            uint4 pk;
            pk.x = pack_bf16x2(__uint_as_float(src[0]) * inv_l, __uint_as_float(src[1]) * inv_l);
            pk.y = pack_bf16x2(__uint_as_float(src[2]) * inv_l, __uint_as_float(src[3]) * inv_l);
            pk.z = pack_bf16x2(__uint_as_float(src[4]) * inv_l, __uint_as_float(src[5]) * inv_l);
            pk.w = pack_bf16x2(__uint_as_float(src[6]) * inv_l, __uint_as_float(src[7]) * inv_l);
            const uint32_t chunk = static_cast<uint32_t>((c & 1) * 4 + k);
            *reinterpret_cast<uint4*>(box_row + ((chunk ^ r7) << 4)) = pk;
          }
        }
        fence_proxy_async_smem();
        // only the storing thread waits for the group's rows; the others
        // just arrive (and count the phase)
        mbar_arrive(&sm->grp_sync[t]);
        const uint32_t phase = sm->grp_uses[t][row]++;
        if (row == 0) {
          if (!mbar_wait(&sm->grp_sync[t], phase & 1u, abort_flag, &g_fwd_err, ERR_TIMEOUT_SOFTMAX)) break;
#pragma unroll
          for (int c2 = 0; c2 < HD / 64; ++c2)
            tma_store_2d(&tmO, sm->q[t] + c2 * (kBlockM * 128), w.h * HD + c2 * 64, sg.q_row0 + qb * kBlockM);
          bulk_commit_group();
          bulk_wait_group_read0();             // q[t] read: the next item's Q may land there
          mbar_arrive(&sm->q_empty[t]);
        }
        args.lse[static_cast<size_t>(w.h) * args.lse_stride + sg.q_row0 + q_local] = lse_val;
      } else if (sg.slot < 0) {
        __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(args.o) +
                             (static_cast<size_t>(sg.q_row0 + q_local) * nh + w.h) * HD;
#pragma unroll 1
        for (int c = 0; c < HD / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + lane_off + c * 32, o);
          tmem_wait_ld();
          reg_fence(o);
          if (row_ok) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint4 pk;
              pk.x = pack_bf16x2(__uint_as_float(o[8 * v + 0]) * inv_l, __uint_as_float(o[8 * v + 1]) * inv_l);
              pk.y = pack_bf16x2(__uint_as_float(o[8 * v + 2]) * inv_l, __uint_as_float(o[8 * v + 3]) * inv_l);
              pk.z = pack_bf16x2(__uint_as_float(o[8 * v + 4]) * inv_l, __uint_as_float(o[8 * v + 5]) * inv_l);
              pk.w = pack_bf16x2(__uint_as_float(o[8 * v + 6]) * inv_l, __uint_as_float(o[8 * v + 7]) * inv_l);
              d4[v] = pk;
            }
          }
        }
        if (row_ok) args.lse[static_cast<size_t>(w.h) * args.lse_stride + sg.q_row0 + q_local] = lse_val;
      } else {
        const size_t prow = static_cast<size_t>(sg.slot) * args.part_rows + sg.out_row0 + q_local;
        const size_t off = (prow * nh + w.h) * HD;
#pragma unroll 1
        for (int c = 0; c < HD / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + lane_off + c * 32, o);
          tmem_wait_ld();
          reg_fence(o);
          if (row_ok && args.part_bf16) {
            uint4* d4 = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(args.o_part) + off + c * 32);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint4 pk;
              pk.x = pack_bf16x2(__uint_as_float(o[8 * v + 0]) * inv_l, __uint_as_float(o[8 * v + 1]) * inv_l);
              pk.y = pack_bf16x2(__uint_as_float(o[8 * v + 2]) * inv_l, __uint_as_float(o[8 * v + 3]) * inv_l);
              pk.z = pack_bf16x2(__uint_as_float(o[8 * v + 4]) * inv_l, __uint_as_float(o[8 * v + 5]) * inv_l);
              pk.w = pack_bf16x2(__uint_as_float(o[8 * v + 6]) * inv_l, __uint_as_float(o[8 * v + 7]) * inv_l);
              d4[v] = pk;
            }
          } else if (row_ok) {
            float4* d4 = reinterpret_cast<float4*>(args.o_part + off + c * 32);
#pragma unroll
            for (int v = 0; v < 8; ++v)
              d4[v] = make_float4(__uint_as_float(o[4 * v + 0]) * inv_l, __uint_as_float(o[4 * v + 1]) * inv_l,
                                  __uint_as_float(o[4 * v + 2]) * inv_l, __uint_as_float(o[4 * v + 3]) * inv_l);
          }
        }
        if (row_ok)
          args.lse_part[(static_cast<size_t>(sg.slot) * nh + w.h) * args.part_rows + sg.out_row0 + q_local] =
              lse_val;
        // Fused merge: publish this partial; the group that completes the set
        // of kv chunks of this (query block, head) merges them into o / lse.
        if (!args.fused_merge) continue;
        __threadfence();
        uint32_t u = sm->grp_uses[t][row];
        if (!__all_sync(0xffffffffu, mbar_sync(&sm->grp_sync[t], u, abort_flag, &g_fwd_err, ERR_TIMEOUT_SOFTMAX)))
          break;
        if (row == 0)
          sm->is_last[t] = atomicAdd(args.counters + sg.counter0 + qb * nh + w.h, 1) == sg.n_kv - 1;
        const bool synced =
            __all_sync(0xffffffffu, mbar_sync(&sm->grp_sync[t], u, abort_flag, &g_fwd_err, ERR_TIMEOUT_SOFTMAX));
        sm->grp_uses[t][row] = u;
        if (!synced) break;
        if (sm->is_last[t]) {
          __threadfence();
          if (row_ok) merge_tile_row<HD>(args, sg, w.h, q_local);
        }
      }
    }
    // this group's output stores must have completed before the CTA exits
    if (row == 0) bulk_wait_group0();
  }

  // ---------------------------------------------------------------- teardown
  __syncwarp();
  if (*abort_flag) drain_delay(2000000ull);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp0) tmem_dealloc(tmem, kTmemCols);
}

template <int HD>
cudaError_t launch_tc(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                      const CUtensorMap& to, const FwdArgs& args, cudaStream_t stream) {
  const size_t smem = sizeof(FwdSmem<HD>) + 1024;
  cudaError_t e = cudaFuncSetAttribute(fwd_tc_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  fwd_tc_kernel<HD><<<args.n_items, kFwdThreads, smem, stream>>>(tq, tk, tv, to, args);
  return cudaGetLastError();
}

}  // namespace

size_t fwd_tc_smem_bytes(int head_dim) {
  return head_dim == 64 ? sizeof(FwdSmem<64>) + 1024 : sizeof(FwdSmem<128>) + 1024;
}

cudaError_t launch_fwd_tc(int head_dim, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, const CUtensorMap& to, const FwdArgs& args,
                          cudaStream_t stream) {
  if (head_dim == 64) return launch_tc<64>(tq, tk, tv, to, args, stream);
  if (head_dim == 128) return launch_tc<128>(tq, tk, tv, to, args, stream);
  return cudaErrorInvalidValue;
}

uint32_t fwd_take_error() {
  uint32_t v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_fwd_err, sizeof(v)) != cudaSuccess) return 0xFFFFFFFFu;
  if (v != 0) cudaMemcpyToSymbol(g_fwd_err, &zero, sizeof(zero));
  return v;
}

}  // namespace zl
