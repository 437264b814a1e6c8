// Host side of libzl_attn: argument validation, the longest-first tile
// scheduler, workspace layout, tensor-map setup and kernel launches behind
// the C ABI in include/zl_attn.h.
//
// Scheduling (Zellige, arXiv 2608.01150v1, §IV-D): the engine runs whole
// sequences and the shards of split sequences together and orders its
// segments stably, ties broken by placement order; the planner's filler stage
// (§IV-C, Eq. 8 and Alg. 1) takes sequences in decreasing price.  On one GPU
// the same largest-first idea becomes: every segment (whole sequence or tile)
// is costed by the keys each of its 128-row query blocks must visit, segments
// are stably sorted by decreasing cost (ties keep input order) and numbered
// into work items in that order.  The kernels launch one CTA per item; the
// resident CTA of each SM steals the next unstarted item when it needs one,
// so the long video blocks start first and the cheap image blocks fill the
// tail on whichever SMs come free.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>

#include "host.h"
#include "launch.h"
#include "zl_attn.h"

namespace {

using zl::FwdArgs;
using zl::FwdSeg;
using zl::kBlockM;
using zl::kBlockN;
using zl::kMaxSegs;
using zl::aligned16;
using zl::launch_counted;
using zl::make_map;
using zl::make_map_acc;

std::atomic<int64_t> g_launches{0};

// ------------------------------------------------------------------ profiling
struct ProfRecord {
  const char* name;
  cudaEvent_t start;
  cudaEvent_t stop;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<ProfRecord> g_prof;

// ------------------------------------------------------------------ device
struct DevInfo {
  int sms = 0;
  int status = 1;  // 1 = not queried yet, else a zl_status
};
std::mutex g_dev_mu;
DevInfo g_dev[128];

zl_status device_sms(int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return ZL_ENODEVICE;
  }
  if (dev < 0 || dev >= 128) return ZL_ENODEVICE;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DevInfo& d = g_dev[dev];
  if (d.status == 1) {
    int major = 0, minor = 0, n = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      d.status = ZL_ECUDA;
    } else if (major != 10 || minor != 3) {
      d.status = ZL_ENODEVICE;   // the kernels are built for sm_103a only
    } else {
      d.sms = n;
      d.status = ZL_OK;
    }
  }
  *sms = d.sms;
  return static_cast<zl_status>(d.status);
}

// ------------------------------------------------------------------ validation
struct SplitSeq {
  int seq = 0;
  int n_kv = 0;
  bool merged = false;   // n_kv > 1: tiles write partials, a merge combines them
  int64_t rbase = 0;     // merged: first row of this sequence in every partial slot
  int64_t len = 0;       // query length
  std::vector<int64_t> counter0;   // merged: first arrival counter of each query chunk
};

struct Plan {
  int64_t tq = 0, tk = 0;
  std::vector<int> split_index;     // per sequence: -1, or index into splits
  std::vector<SplitSeq> splits;
  std::vector<zl_tile_t> tiles;     // sorted by (seq, h_chunk, q_chunk, kv_chunk), h_len resolved
  std::vector<int32_t> tile_src;    // index of each sorted tile in the caller's table
  int64_t part_rows = 0;            // R
  int n_parts = 0;                  // P
  int64_t n_counters = 0;           // arrival counters: (query chunk, 128-row block) x head
};

zl_status check_cu(const int32_t* cu, int32_t b, int64_t* total) {
  if (!cu) return ZL_EINVAL;
  if (cu[0] != 0) return ZL_EINVAL;
  for (int32_t s = 0; s < b; ++s)
    if (cu[s + 1] < cu[s]) return ZL_EINVAL;
  *total = cu[b];
  if (*total > zl::kMaxTokens) return ZL_EINVAL;
  return ZL_OK;
}

zl_status make_plan(const int32_t* cu_q, const int32_t* cu_k, int32_t b, int32_t nh, int32_t hd,
                    const zl_tile_t* tiles, int32_t n_tiles, Plan* plan) {
  if (n_tiles < 0) return ZL_EINVAL;
  const zl_status st = zl::check_batch(cu_q, cu_k, b, nh, hd, &plan->tq, &plan->tk);
  if (st != ZL_OK) return st;
  plan->split_index.assign(static_cast<size_t>(b), -1);
  plan->splits.clear();
  plan->tiles.clear();
  if (n_tiles == 0) return ZL_OK;
  if (!tiles) return ZL_EINVAL;
  plan->tiles.assign(tiles, tiles + n_tiles);
  for (zl_tile_t& t : plan->tiles) {
    if (t.seq < 0 || t.seq >= b) return ZL_EINVAL;
    const int64_t lq = cu_q[t.seq + 1] - cu_q[t.seq];
    const int64_t lk = cu_k[t.seq + 1] - cu_k[t.seq];
    if (t.n_kv_chunks < 1 || t.n_kv_chunks > 64) return ZL_EINVAL;
    if (t.kv_chunk < 0 || t.kv_chunk >= t.n_kv_chunks || t.q_chunk < 0 || t.q_chunk >= 1 << 20)
      return ZL_EINVAL;
    if (t.q_len < 1 || t.k_len < 1 || t.q_start < 0 || t.k_start < 0) return ZL_EINVAL;
    if (int64_t(t.q_start) + t.q_len > lq || int64_t(t.k_start) + t.k_len > lk) return ZL_EINVAL;
    if (t.h_len == 0) {
      if (t.h_start != 0 || t.h_chunk != 0) return ZL_EINVAL;
      t.h_len = nh;
    }
    if (t.h_start < 0 || t.h_len < 1 || int64_t(t.h_start) + t.h_len > nh) return ZL_EINVAL;
    if (t.h_chunk < 0 || t.h_chunk >= nh) return ZL_EINVAL;
  }
  plan->tile_src.resize(plan->tiles.size());
  for (size_t x = 0; x < plan->tile_src.size(); ++x) plan->tile_src[x] = static_cast<int32_t>(x);
  std::stable_sort(plan->tile_src.begin(), plan->tile_src.end(), [&](int32_t ia, int32_t ic) {
    const zl_tile_t& a = plan->tiles[static_cast<size_t>(ia)];
    const zl_tile_t& c = plan->tiles[static_cast<size_t>(ic)];
    if (a.seq != c.seq) return a.seq < c.seq;
    if (a.h_chunk != c.h_chunk) return a.h_chunk < c.h_chunk;
    if (a.q_chunk != c.q_chunk) return a.q_chunk < c.q_chunk;
    return a.kv_chunk < c.kv_chunk;
  });
  {
    std::vector<zl_tile_t> sorted;
    sorted.reserve(plan->tiles.size());
    for (int32_t x : plan->tile_src) sorted.push_back(plan->tiles[static_cast<size_t>(x)]);
    plan->tiles.swap(sorted);
  }
  // Each split sequence: a full n_h x n_q x n_kv grid.  Head chunk 0's tiles
  // are an n_q x n_kv grid partitioning the query range and the key range
  // into contiguous chunks in chunk order; every further head chunk repeats
  // that grid exactly over the next contiguous head range.
  size_t i = 0;
  int64_t rbase = 0;
  while (i < plan->tiles.size()) {
    const int seq = plan->tiles[i].seq;
    size_t j = i;
    while (j < plan->tiles.size() && plan->tiles[j].seq == seq) ++j;
    size_t g = i;   // end of head chunk 0
    while (g < j && plan->tiles[g].h_chunk == plan->tiles[i].h_chunk) ++g;
    const size_t per_h = g - i;
    if ((j - i) % per_h != 0) return ZL_EINVAL;
    const int n_h = static_cast<int>((j - i) / per_h);
    const int n_kv = plan->tiles[i].n_kv_chunks;
    if (per_h % static_cast<size_t>(n_kv) != 0) return ZL_EINVAL;
    const int n_q = static_cast<int>(per_h / static_cast<size_t>(n_kv));
    const int64_t lq = cu_q[seq + 1] - cu_q[seq];
    const int64_t lk = cu_k[seq + 1] - cu_k[seq];
    int64_t q_expect = 0;
    for (int qc = 0; qc < n_q; ++qc) {
      int64_t k_expect = 0;
      const zl_tile_t& first = plan->tiles[i + static_cast<size_t>(qc) * n_kv];
      if (first.q_start != q_expect) return ZL_EINVAL;
      for (int kc = 0; kc < n_kv; ++kc) {
        const zl_tile_t& t = plan->tiles[i + static_cast<size_t>(qc) * n_kv + kc];
        if (t.n_kv_chunks != n_kv || t.q_chunk != qc || t.kv_chunk != kc) return ZL_EINVAL;
        if (t.q_start != first.q_start || t.q_len != first.q_len) return ZL_EINVAL;
        const zl_tile_t& col0 = plan->tiles[i + kc];   // same kv chunk, q chunk 0
        if (t.k_start != col0.k_start || t.k_len != col0.k_len) return ZL_EINVAL;
        if (t.k_start != k_expect) return ZL_EINVAL;
        k_expect += t.k_len;
      }
      if (k_expect != lk) return ZL_EINVAL;
      q_expect += first.q_len;
    }
    if (q_expect != lq) return ZL_EINVAL;
    int64_t h_expect = 0;
    for (int hc = 0; hc < n_h; ++hc) {
      const zl_tile_t& h_first = plan->tiles[i + static_cast<size_t>(hc) * per_h];
      if (h_first.h_start != h_expect) return ZL_EINVAL;
      for (size_t x = 0; x < per_h; ++x) {
        const zl_tile_t& t = plan->tiles[i + static_cast<size_t>(hc) * per_h + x];
        const zl_tile_t& ref = plan->tiles[i + x];   // same position in head chunk 0
        if (t.h_chunk != hc || t.h_start != h_first.h_start || t.h_len != h_first.h_len) return ZL_EINVAL;
        if (t.q_chunk != ref.q_chunk || t.kv_chunk != ref.kv_chunk || t.n_kv_chunks != n_kv ||
            t.q_start != ref.q_start || t.q_len != ref.q_len || t.k_start != ref.k_start || t.k_len != ref.k_len)
          return ZL_EINVAL;
      }
      h_expect += h_first.h_len;
    }
    if (h_expect != nh) return ZL_EINVAL;
    SplitSeq sp;
    sp.seq = seq;
    sp.n_kv = n_kv;
    sp.merged = n_kv > 1;
    sp.len = lq;
    if (sp.merged) {
      sp.rbase = rbase;
      rbase += lq;
      plan->n_parts = std::max(plan->n_parts, n_kv);
      for (int qc = 0; qc < n_q; ++qc) {
        const zl_tile_t& first = plan->tiles[i + static_cast<size_t>(qc) * n_kv];
        sp.counter0.push_back(plan->n_counters);
        plan->n_counters += int64_t((first.q_len + kBlockM - 1) / kBlockM) * nh;
      }
    }
    plan->split_index[static_cast<size_t>(seq)] = static_cast<int>(plan->splits.size());
    plan->splits.push_back(std::move(sp));
    i = j;
  }
  plan->part_rows = rbase;
  return ZL_OK;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

size_t fwd_workspace_bytes(const Plan& p, int nh, int hd) {
  if (p.part_rows == 0) return 0;
  const size_t o_bytes = static_cast<size_t>(p.n_parts) * p.part_rows * nh * hd * sizeof(float);
  const size_t l_bytes = static_cast<size_t>(p.n_parts) * nh * p.part_rows * sizeof(float);
  const size_t c_bytes = static_cast<size_t>(p.n_counters) * sizeof(int32_t);
  return align256(o_bytes) + align256(l_bytes) + align256(c_bytes);
}

// ------------------------------------------------------------------ scheduler
struct Segment {
  FwdSeg seg;
  int64_t cost;   // keys visited per query block
  int order;      // input order (sequence index, then tile order)
  int32_t seq;    // the segment's sequence
  int32_t tile;   // index in the caller's tile table, or -1: the whole sequence
};

// Whole sequences and tiles as segments, stably ordered by decreasing cost.
std::vector<Segment> schedule_fwd(const Plan& p, const int32_t* cu_q, const int32_t* cu_k, int32_t b, int nh) {
  std::vector<Segment> segs;
  segs.reserve(static_cast<size_t>(b) + p.tiles.size());
  size_t ti = 0;
  int order = 0;
  for (int32_t s = 0; s < b; ++s) {
    const int32_t lq = cu_q[s + 1] - cu_q[s];
    const int32_t lk = cu_k[s + 1] - cu_k[s];
    const int si = p.split_index[static_cast<size_t>(s)];
    if (si < 0) {
      if (lq == 0) continue;
      Segment g;
      g.seg = FwdSeg{cu_q[s], cu_k[s], lq, lk, cu_q[s], -1, 0, 0, 0, 0, nh};
      g.cost = lk;
      g.order = order++;
      g.seq = s;
      g.tile = -1;
      segs.push_back(g);
    } else {
      const SplitSeq& sp = p.splits[static_cast<size_t>(si)];
      while (ti < p.tiles.size() && p.tiles[ti].seq < s) ++ti;
      for (; ti < p.tiles.size() && p.tiles[ti].seq == s; ++ti) {
        const zl_tile_t& t = p.tiles[ti];
        Segment g;
        if (sp.merged) {
          g.seg = FwdSeg{cu_q[s] + t.q_start, cu_k[s] + t.k_start, t.q_len, t.k_len,
                         static_cast<int32_t>(sp.rbase + t.q_start), t.kv_chunk, 0,
                         static_cast<int32_t>(sp.counter0[static_cast<size_t>(t.q_chunk)]), sp.n_kv,
                         t.h_start, t.h_len};
        } else {   // one kv chunk: the tile's rows are final
          g.seg = FwdSeg{cu_q[s] + t.q_start, cu_k[s] + t.k_start, t.q_len, t.k_len,
                         cu_q[s] + t.q_start, -1, 0, 0, 0, t.h_start, t.h_len};
        }
        g.cost = t.k_len;
        g.order = order++;
        g.seq = s;
        g.tile = p.tile_src[ti];
        segs.push_back(g);
      }
    }
  }
  std::stable_sort(segs.begin(), segs.end(),
                   [](const Segment& a, const Segment& c) { return a.cost > c.cost; });
  return segs;
}

// Backward segments.  The backward of a split sequence is the sum over its
// tiles, which is the backward of the whole sequence: every sequence runs
// whole, costed by the query rows each of its key blocks visits, stably
// longest first.
struct BSeg {
  zl::BwdSeg seg;
  int64_t cost;
  int32_t seq;
};

std::vector<BSeg> schedule_bwd(const int32_t* cu_q, const int32_t* cu_k, int32_t b) {
  std::vector<BSeg> segs;
  for (int32_t i = 0; i < b; ++i) {
    const int32_t lq = cu_q[i + 1] - cu_q[i];
    const int32_t lk = cu_k[i + 1] - cu_k[i];
    if (lq == 0 || lk == 0) continue;
    segs.push_back(BSeg{zl::BwdSeg{cu_q[i], cu_k[i], lq, lk, 0}, lq, i});
  }
  std::stable_sort(segs.begin(), segs.end(), [](const BSeg& a, const BSeg& c) { return a.cost > c.cost; });
  return segs;
}

// Fills args.segs with segments [first, last) and numbers their items; false
// if the launch would hold more items than a grid (and an int32 index) can.
bool fill_args(FwdArgs* args, const std::vector<Segment>& segs, size_t first, size_t last, int rows_per_item) {
  int64_t items = 0;
  args->n_segs = static_cast<int32_t>(last - first);
  args->rows_per_item = rows_per_item;
  for (size_t i = first; i < last; ++i) {
    FwdSeg s = segs[i].seg;
    s.item0 = static_cast<int32_t>(items);
    args->segs[i - first] = s;
    items += int64_t(s.nh) * ((s.q_len + rows_per_item - 1) / rows_per_item);
    if (items > INT32_MAX) return false;
  }
  args->n_items = static_cast<int32_t>(items);
  return true;
}

zl_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return ZL_OK;
  cudaGetLastError();
  return ZL_ECUDA;
}

}  // namespace

namespace zl {

void note_launch() { g_launches.fetch_add(1); }

zl_status check_batch(const int32_t* cu_q, const int32_t* cu_k, int32_t num_seqs, int32_t num_heads,
                      int32_t head_dim, int64_t* tq, int64_t* tk) {
  if (num_seqs < 0 || num_heads < 1 || num_heads > 4096) return ZL_EINVAL;
  if (head_dim != 64 && head_dim != 128) return ZL_EUNSUPPORTED;
  zl_status st = check_cu(cu_q, num_seqs, tq);
  if (st != ZL_OK) return st;
  st = check_cu(cu_k, num_seqs, tk);
  if (st != ZL_OK) return st;
  if ((*tq + kBlockM) * int64_t(num_heads) * head_dim > (int64_t(1) << 40)) return ZL_EINVAL;
  if ((*tk + kBlockN) * int64_t(num_heads) * head_dim > (int64_t(1) << 40)) return ZL_EINVAL;
  for (int32_t s = 0; s < num_seqs; ++s)
    if (cu_q[s + 1] > cu_q[s] && cu_k[s + 1] == cu_k[s]) return ZL_EINVAL;  // queries without keys
  return ZL_OK;
}

namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
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
}  // namespace

bool make_map(CUtensorMap* map, const void* base, int64_t rows, int nh, int hd, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(nh) * hd, static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(nh) * hd * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_acc(CUtensorMap* map, const float* base, int64_t rows, int nh, int hd, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(nh) * hd, static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(nh) * hd * 4};
  const cuuint32_t box[2] = {32, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

zl_status prof_before(ProfScope* p, cudaStream_t stream) {
  {
    std::lock_guard<std::mutex> lock(g_prof_mu);
    p->on = g_prof_on;
  }
  if (!p->on) return ZL_OK;
  if (cudaEventCreate(&p->start) != cudaSuccess || cudaEventCreate(&p->stop) != cudaSuccess ||
      cudaEventRecord(p->start, stream) != cudaSuccess) {
    cudaGetLastError();
    if (p->start) cudaEventDestroy(p->start);
    if (p->stop) cudaEventDestroy(p->stop);
    return ZL_ECUDA;
  }
  return ZL_OK;
}

zl_status prof_after(ProfScope* p, const char* name, cudaStream_t stream, cudaError_t launch_error) {
  if (launch_error != cudaSuccess) {
    cudaGetLastError();
    if (p->on) {
      cudaEventDestroy(p->start);
      cudaEventDestroy(p->stop);
    }
    return ZL_ECUDA;
  }
  g_launches.fetch_add(1);
  if (!p->on) return ZL_OK;
  if (cudaEventRecord(p->stop, stream) != cudaSuccess) {
    cudaGetLastError();
    cudaEventDestroy(p->start);
    cudaEventDestroy(p->stop);
    return ZL_ECUDA;
  }
  std::lock_guard<std::mutex> lock(g_prof_mu);
  g_prof.push_back(ProfRecord{name, p->start, p->stop});
  return ZL_OK;
}

}  // namespace zl

// =================================================================== C ABI
extern "C" {

const char* zl_status_string(int32_t status) {
  switch (status) {
    case ZL_OK: return "ok";
    case ZL_EINVAL: return "invalid argument";
    case ZL_EUNSUPPORTED: return "unsupported configuration";
    case ZL_EALIGN: return "device pointer not 16-byte aligned";
    case ZL_EWORKSPACE: return "workspace missing or too small";
    case ZL_ECUDA: return "CUDA error";
    case ZL_ETIMEOUT: return "a kernel gave up a bounded wait";
    case ZL_ENODEVICE: return "no sm_103 CUDA device";
    default: return "unknown status";
  }
}

int32_t zl_version(void) { return (2 << 16) | 1; }

int64_t zl_launch_count(void) { return g_launches.load(); }

zl_status zl_varlen_attn_fwd_workspace_size(const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                            int32_t num_seqs, int32_t num_heads, int32_t head_dim,
                                            const zl_tile_t* tiles, int32_t num_tiles, size_t* bytes) {
  if (!bytes) return ZL_EINVAL;
  Plan plan;
  const zl_status st = make_plan(cu_seqlens_q, cu_seqlens_k, num_seqs, num_heads, head_dim, tiles,
                                 num_tiles, &plan);
  if (st != ZL_OK) return st;
  *bytes = fwd_workspace_bytes(plan, num_heads, head_dim);
  return ZL_OK;
}

zl_status zl_varlen_attn_fwd_schedule(const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int32_t num_seqs,
                                      int32_t num_heads, int32_t head_dim, int32_t dtype, const zl_tile_t* tiles,
                                      int32_t num_tiles, zl_work_item_t* items, int64_t max_items,
                                      int64_t* n_items) {
  if (!n_items || max_items < 0 || (max_items > 0 && !items)) return ZL_EINVAL;
  if (dtype != ZL_BF16 && dtype != ZL_FP32) return ZL_EUNSUPPORTED;
  Plan plan;
  const zl_status st = make_plan(cu_seqlens_q, cu_seqlens_k, num_seqs, num_heads, head_dim, tiles, num_tiles, &plan);
  if (st != ZL_OK) return st;
  const std::vector<Segment> segs = schedule_fwd(plan, cu_seqlens_q, cu_seqlens_k, num_seqs, num_heads);
  const int rows = dtype == ZL_BF16 ? zl::kFwdRowsPerItem : kBlockM;
  // the numbering of fill_args and the kernels' decode: launch by launch,
  // segment by segment, head-major, query block fastest
  int64_t n = 0;
  int32_t launch = 0;
  for (size_t first = 0; first < segs.size(); first += kMaxSegs, ++launch) {
    const size_t last = std::min(segs.size(), first + kMaxSegs);
    for (size_t i = first; i < last; ++i) {
      const Segment& g = segs[i];
      const FwdSeg& s = g.seg;
      const int32_t q0 = s.q_row0 - cu_seqlens_q[g.seq];
      const int32_t k0 = s.k_row0 - cu_seqlens_k[g.seq];
      const int32_t nqb = (s.q_len + rows - 1) / rows;
      for (int32_t h = s.h0; h < s.h0 + s.nh; ++h)
        for (int32_t qb = 0; qb < nqb; ++qb, ++n) {
          if (n >= max_items) continue;
          zl_work_item_t& w = items[n];
          w.launch = launch;
          w.seq = g.seq;
          w.tile = g.tile;
          w.head = h;
          w.q_start = q0 + qb * rows;
          w.q_len = std::min(rows, s.q_len - qb * rows);
          w.k_start = k0;
          w.k_len = s.k_len;
        }
    }
  }
  *n_items = n;
  return ZL_OK;
}

zl_status zl_lse_merge(const float* o_partial, const float* lse_partial, int32_t n_parts, int64_t rows,
                       int32_t num_heads, int32_t head_dim, int64_t part_stride_rows, void* o,
                       int32_t out_dtype, float* lse, int64_t lse_head_stride, void* stream) {
  return zl_lse_merge_ex(o_partial, ZL_FP32, lse_partial, n_parts, rows, num_heads, head_dim, part_stride_rows,
                         o, out_dtype, lse, lse_head_stride, stream);
}

zl_status zl_lse_merge_ex(const void* o_partial, int32_t part_dtype, const float* lse_partial, int32_t n_parts,
                          int64_t rows, int32_t num_heads, int32_t head_dim, int64_t part_stride_rows, void* o,
                          int32_t out_dtype, float* lse, int64_t lse_head_stride, void* stream) {
  if (n_parts < 1 || n_parts > 64 || rows < 0 || num_heads < 1 || part_stride_rows < rows ||
      lse_head_stride < rows)
    return ZL_EINVAL;
  if (head_dim != 64 && head_dim != 128) return ZL_EUNSUPPORTED;
  if (out_dtype != ZL_BF16 && out_dtype != ZL_FP32) return ZL_EUNSUPPORTED;
  if (part_dtype != ZL_BF16 && part_dtype != ZL_FP32) return ZL_EUNSUPPORTED;
  if (rows == 0) return ZL_OK;
  if (!o_partial || !lse_partial || !o || !lse) return ZL_EINVAL;
  if (!aligned16(o_partial) || !aligned16(o)) return ZL_EALIGN;
  if (rows * num_heads > (int64_t(1) << 40)) return ZL_EINVAL;
  int sms = 0;
  zl_status st = device_sms(&sms);
  if (st != ZL_OK) return st;
  zl::MergeArgs a;
  a.o_part = o_partial;
  a.lse_part = lse_partial;
  a.o = o;
  a.lse = lse;
  a.rows = rows;
  a.part_stride_rows = part_stride_rows;
  a.lse_head_stride = lse_head_stride;
  a.n_parts = n_parts;
  a.num_heads = num_heads;
  a.out_bf16 = out_dtype == ZL_BF16 ? 1 : 0;
  a.part_bf16 = part_dtype == ZL_BF16 ? 1 : 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return launch_counted("lse_merge", s, [&] { return zl::launch_merge(head_dim, a, sms, s); });
}

zl_status zl_varlen_attn_fwd(const void* q, const void* k, const void* v, const int32_t* cu_seqlens_q,
                             const int32_t* cu_seqlens_k, int32_t num_seqs, int32_t num_heads,
                             int32_t head_dim, int32_t dtype, float softmax_scale, const zl_tile_t* tiles,
                             int32_t num_tiles, void* o, float* lse, void* workspace,
                             size_t workspace_bytes, void* stream) {
  return zl_varlen_attn_fwd_ex(q, k, v, cu_seqlens_q, cu_seqlens_k, num_seqs, num_heads, head_dim, dtype,
                               softmax_scale, tiles, num_tiles, o, lse, workspace, workspace_bytes, stream, 0u);
}

zl_status zl_varlen_attn_fwd_ex(const void* q, const void* k, const void* v, const int32_t* cu_seqlens_q,
                                const int32_t* cu_seqlens_k, int32_t num_seqs, int32_t num_heads,
                                int32_t head_dim, int32_t dtype, float softmax_scale, const zl_tile_t* tiles,
                                int32_t num_tiles, void* o, float* lse, void* workspace,
                                size_t workspace_bytes, void* stream, uint32_t flags) {
  if ((flags & ~static_cast<uint32_t>(ZL_FWD_FUSED_MERGE | ZL_FWD_BF16_PARTIALS)) != 0) return ZL_EINVAL;
  const bool fused = (flags & ZL_FWD_FUSED_MERGE) != 0 && dtype == ZL_BF16;
  const bool part_bf16 = (flags & ZL_FWD_BF16_PARTIALS) != 0 && dtype == ZL_BF16;
  if (dtype != ZL_BF16 && dtype != ZL_FP32) return ZL_EUNSUPPORTED;
  if (!(softmax_scale > 0.f) || !std::isfinite(softmax_scale)) return ZL_EINVAL;
  Plan plan;
  zl_status st = make_plan(cu_seqlens_q, cu_seqlens_k, num_seqs, num_heads, head_dim, tiles, num_tiles, &plan);
  if (st != ZL_OK) return st;
  if (plan.tq == 0) return ZL_OK;
  if (!q || !k || !v || !o || !lse) return ZL_EINVAL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse)) return ZL_EALIGN;
  const size_t need = fwd_workspace_bytes(plan, num_heads, head_dim);
  if (need > 0 && (!workspace || workspace_bytes < need)) return ZL_EWORKSPACE;
  if (need > 0 && (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return ZL_EALIGN;
  int sms = 0;
  st = device_sms(&sms);
  if (st != ZL_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  const std::vector<Segment> segs = schedule_fwd(plan, cu_seqlens_q, cu_seqlens_k, num_seqs, num_heads);
  static thread_local FwdArgs args;   // ~27 KB: kept off the stack
  std::memset(&args, 0, sizeof(args));
  args.o = o;
  args.lse = lse;
  args.lse_stride = plan.tq;
  args.num_heads = num_heads;
  args.scale = softmax_scale;
  args.scale_log2 = softmax_scale * 1.4426950408889634f;
  if (need > 0) {
    char* ws = static_cast<char*>(workspace);
    args.o_part = reinterpret_cast<float*>(ws);
    const size_t o_bytes = align256(static_cast<size_t>(plan.n_parts) * plan.part_rows * num_heads * head_dim * sizeof(float));
    const size_t l_bytes = align256(static_cast<size_t>(plan.n_parts) * num_heads * plan.part_rows * sizeof(float));
    args.lse_part = reinterpret_cast<float*>(ws + o_bytes);
    args.counters = reinterpret_cast<int32_t*>(ws + o_bytes + l_bytes);
    args.part_rows = plan.part_rows;
    args.fused_merge = fused ? 1 : 0;
    args.part_bf16 = part_bf16 ? 1 : 0;
    if (fused) {
      st = cuda_status(cudaMemsetAsync(args.counters, 0, static_cast<size_t>(plan.n_counters) * sizeof(int32_t), s));
      if (st != ZL_OK) return st;
    }
  }
  CUtensorMap mq, mk, mv, mo;
  if (dtype == ZL_BF16) {
    if (!make_map(&mq, q, plan.tq, num_heads, head_dim) || !make_map(&mk, k, plan.tk, num_heads, head_dim) ||
        !make_map(&mv, v, plan.tk, num_heads, head_dim) || !make_map(&mo, o, plan.tq, num_heads, head_dim))
      return ZL_ECUDA;
  }
  for (size_t first = 0; first < segs.size(); first += kMaxSegs) {
    const size_t last = std::min(segs.size(), first + kMaxSegs);
    if (!fill_args(&args, segs, first, last, dtype == ZL_BF16 ? zl::kFwdRowsPerItem : kBlockM)) return ZL_EINVAL;
    if (args.n_items == 0) continue;
    if (dtype == ZL_BF16) {
      st = launch_counted("fwd_tc", s, [&] { return zl::launch_fwd_tc(head_dim, mq, mk, mv, mo, args, s); });
    } else {
      st = launch_counted("fwd_f32", s, [&] {
        return zl::launch_fwd_f32(head_dim, static_cast<const float*>(q), static_cast<const float*>(k),
                                  static_cast<const float*>(v), args, s);
      });
    }
    if (st != ZL_OK) return st;
  }
  // Combine each split sequence's partial slots into its rows of o and lse
  // (unless the forward kernel merged them in its last arriving tiles).
  const size_t esz = dtype == ZL_BF16 ? 2 : 4;
  for (const SplitSeq& sp : plan.splits) {
    if (fused) break;
    if (!sp.merged) continue;
    zl::MergeArgs m;
    m.o_part = static_cast<const char*>(static_cast<const void*>(args.o_part)) +
               static_cast<size_t>(sp.rbase) * num_heads * head_dim * (part_bf16 ? 2 : 4);
    m.part_bf16 = part_bf16 ? 1 : 0;
    m.lse_part = args.lse_part + sp.rbase;
    m.o = static_cast<char*>(o) + static_cast<size_t>(cu_seqlens_q[sp.seq]) * num_heads * head_dim * esz;
    m.lse = lse + cu_seqlens_q[sp.seq];
    m.rows = sp.len;
    m.part_stride_rows = plan.part_rows;
    m.lse_head_stride = plan.tq;
    m.n_parts = sp.n_kv;
    m.num_heads = num_heads;
    m.out_bf16 = dtype == ZL_BF16 ? 1 : 0;
    st = launch_counted("lse_merge", s, [&] { return zl::launch_merge(head_dim, m, sms, s); });
    if (st != ZL_OK) return st;
  }
  return ZL_OK;
}

zl_status zl_varlen_attn_bwd_workspace_size(const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                            int32_t num_seqs, int32_t num_heads, int32_t head_dim,
                                            size_t* bytes) {
  if (!bytes) return ZL_EINVAL;
  Plan plan;
  const zl_status st = make_plan(cu_seqlens_q, cu_seqlens_k, num_seqs, num_heads, head_dim, nullptr, 0, &plan);
  if (st != ZL_OK) return st;
  *bytes = align256(static_cast<size_t>(plan.tq) * num_heads * head_dim * sizeof(float)) +
           align256(static_cast<size_t>(plan.tq) * num_heads * sizeof(float));
  return ZL_OK;
}

zl_status zl_varlen_attn_bwd_schedule(const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int32_t num_seqs,
                                      int32_t num_heads, int32_t head_dim, const zl_tile_t* tiles, int32_t num_tiles,
                                      zl_bwd_work_item_t* items, int64_t max_items, int64_t* n_items) {
  if (!n_items || max_items < 0 || (max_items > 0 && !items)) return ZL_EINVAL;
  Plan plan;
  const zl_status st = make_plan(cu_seqlens_q, cu_seqlens_k, num_seqs, num_heads, head_dim, tiles, num_tiles, &plan);
  if (st != ZL_OK) return st;
  const std::vector<BSeg> segs = schedule_bwd(cu_seqlens_q, cu_seqlens_k, num_seqs);
  // the kernels' numbering: launch by launch, segment by segment, head-major,
  // key block fastest
  int64_t n = 0;
  int32_t launch = 0;
  for (size_t first = 0; first < segs.size(); first += kMaxSegs, ++launch) {
    const size_t last = std::min(segs.size(), first + kMaxSegs);
    for (size_t i = first; i < last; ++i) {
      const zl::BwdSeg& s = segs[i].seg;
      const int32_t nkb = (s.k_len + kBlockN - 1) / kBlockN;
      for (int32_t h = 0; h < num_heads; ++h)
        for (int32_t kb = 0; kb < nkb; ++kb, ++n) {
          if (n >= max_items) continue;
          zl_bwd_work_item_t& w = items[n];
          w.launch = launch;
          w.seq = segs[i].seq;
          w.head = h;
          w.k_start = kb * kBlockN;
          w.k_len = std::min(kBlockN, s.k_len - kb * kBlockN);
          w.q_len = s.q_len;
        }
    }
  }
  *n_items = n;
  return ZL_OK;
}

zl_status zl_varlen_attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                             const void* dout, const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                             int32_t num_seqs, int32_t num_heads, int32_t head_dim, int32_t dtype,
                             float softmax_scale, const zl_tile_t* tiles, int32_t num_tiles, void* dq,
                             void* dk, void* dv, void* workspace, size_t workspace_bytes, void* stream) {
  if (dtype != ZL_BF16) return ZL_EUNSUPPORTED;
  if (!(softmax_scale > 0.f) || !std::isfinite(softmax_scale)) return ZL_EINVAL;
  Plan plan;
  zl_status st = make_plan(cu_seqlens_q, cu_seqlens_k, num_seqs, num_heads, head_dim, tiles, num_tiles, &plan);
  if (st != ZL_OK) return st;
  if (plan.tq == 0 && plan.tk == 0) return ZL_OK;
  if ((plan.tq > 0 && (!q || !o || !lse || !dout || !dq)) || (plan.tk > 0 && (!k || !v || !dk || !dv)))
    return ZL_EINVAL;
  const void* ptrs[] = {q, k, v, o, dout, dq, dk, dv, lse};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return ZL_EALIGN;
  const size_t dq_bytes = align256(static_cast<size_t>(plan.tq) * num_heads * head_dim * sizeof(float));
  const size_t need = dq_bytes + align256(static_cast<size_t>(plan.tq) * num_heads * sizeof(float));
  if (plan.tq > 0 && (!workspace || workspace_bytes < need)) return ZL_EWORKSPACE;
  if (plan.tq > 0 && (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return ZL_EALIGN;
  int sms = 0;
  st = device_sms(&sms);
  if (st != ZL_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t row_bytes = static_cast<size_t>(num_heads) * head_dim * 2;

  // Keys of sequences without queries get zero gradients.
  for (int32_t i = 0; i < num_seqs; ++i) {
    const int32_t lq = cu_seqlens_q[i + 1] - cu_seqlens_q[i];
    const int32_t lk = cu_seqlens_k[i + 1] - cu_seqlens_k[i];
    if (lq == 0 && lk > 0) {
      st = cuda_status(cudaMemsetAsync(static_cast<char*>(dk) + cu_seqlens_k[i] * row_bytes, 0, lk * row_bytes, s));
      if (st == ZL_OK)
        st = cuda_status(cudaMemsetAsync(static_cast<char*>(dv) + cu_seqlens_k[i] * row_bytes, 0, lk * row_bytes, s));
      if (st != ZL_OK) return st;
    }
  }
  if (plan.tq == 0) return ZL_OK;

  float* dq_acc = static_cast<float*>(workspace);
  float* dsum = reinterpret_cast<float*>(static_cast<char*>(workspace) + dq_bytes);
  st = launch_counted("bwd_preprocess", s, [&] {
    return zl::launch_bwd_preprocess(head_dim, o, dout, dsum, dq_acc, plan.tq, num_heads, sms, s);
  });
  if (st != ZL_OK) return st;

  const std::vector<BSeg> segs = schedule_bwd(cu_seqlens_q, cu_seqlens_k, num_seqs);
  CUtensorMap mq, mk, mv, mdo, mdq;
  const int bq = zl::bwd_query_block();
  if (!make_map(&mq, q, plan.tq, num_heads, head_dim, bq) || !make_map(&mk, k, plan.tk, num_heads, head_dim) ||
      !make_map(&mv, v, plan.tk, num_heads, head_dim) || !make_map(&mdo, dout, plan.tq, num_heads, head_dim, bq) ||
      !make_map_acc(&mdq, dq_acc, plan.tq, num_heads, head_dim, bq))
    return ZL_ECUDA;
  static thread_local zl::BwdArgs args;
  std::memset(&args, 0, sizeof(args));
  args.lse = lse;
  args.dsum = dsum;
  args.dq_acc = dq_acc;
  args.dk = dk;
  args.dv = dv;
  args.lse_stride = plan.tq;
  args.num_heads = num_heads;
  args.scale = softmax_scale;
  args.scale_log2 = softmax_scale * 1.4426950408889634f;
  for (size_t first = 0; first < segs.size(); first += kMaxSegs) {
    const size_t last = std::min(segs.size(), first + kMaxSegs);
    int64_t items = 0;
    args.n_segs = static_cast<int32_t>(last - first);
    for (size_t i = first; i < last; ++i) {
      zl::BwdSeg b = segs[i].seg;
      b.item0 = static_cast<int32_t>(items);
      args.segs[i - first] = b;
      items += int64_t(num_heads) * ((b.k_len + kBlockN - 1) / kBlockN);
    }
    if (items > INT32_MAX) return ZL_EINVAL;      // more items than a grid (and an int32 index) can hold
    args.n_items = static_cast<int32_t>(items);
    if (items == 0) continue;
    st = launch_counted("bwd_tc", s, [&] { return zl::launch_bwd_tc(head_dim, mq, mk, mv, mdo, mdq, args, s); });
    if (st != ZL_OK) return st;
  }
  return launch_counted("dq_convert", s, [&] {
    return zl::launch_dq_convert(head_dim, dq_acc, dq, plan.tq, num_heads, softmax_scale, sms, s);
  });
}

zl_status zl_profile_begin(void) {
  std::lock_guard<std::mutex> lock(g_prof_mu);
  if (g_prof_on) return ZL_EINVAL;
  g_prof_on = true;
  g_prof.clear();
  return ZL_OK;
}

zl_status zl_profile_end(zl_profile_entry_t* entries, int32_t max_entries, int32_t* n_entries) {
  std::vector<ProfRecord> recs;
  {
    std::lock_guard<std::mutex> lock(g_prof_mu);
    if (!g_prof_on) return ZL_EINVAL;
    g_prof_on = false;
    recs.swap(g_prof);
  }
  std::vector<zl_profile_entry_t> agg;
  zl_status st = ZL_OK;
  for (const ProfRecord& r : recs) {
    float ms = 0.f;
    if (st == ZL_OK &&
        (cudaEventSynchronize(r.stop) != cudaSuccess || cudaEventElapsedTime(&ms, r.start, r.stop) != cudaSuccess)) {
      cudaGetLastError();
      st = ZL_ECUDA;
    }
    cudaEventDestroy(r.start);
    cudaEventDestroy(r.stop);
    size_t i = 0;
    while (i < agg.size() && std::strncmp(agg[i].name, r.name, sizeof(agg[i].name)) != 0) ++i;
    if (i == agg.size()) {
      zl_profile_entry_t e;
      std::memset(&e, 0, sizeof(e));
      std::strncpy(e.name, r.name, sizeof(e.name) - 1);
      agg.push_back(e);
    }
    agg[i].launches += 1;
    agg[i].total_ms += ms;
  }
  int32_t n = 0;
  for (size_t i = 0; i < agg.size() && entries && n < max_entries; ++i) entries[n++] = agg[i];
  if (n_entries) *n_entries = n;
  return st;
}

zl_status zl_sync_check(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return ZL_ECUDA;
  }
  const uint32_t ef = zl::fwd_take_error();
  const uint32_t eb = zl::bwd_take_error();
  const uint32_t es = zl::selftest_take_error();
  if (ef == 0xFFFFFFFFu || eb == 0xFFFFFFFFu || es == 0xFFFFFFFFu) return ZL_ECUDA;
  if (ef != 0 || eb != 0 || es != 0) return ZL_ETIMEOUT;
  return ZL_OK;
}

zl_status zl_selftest_wait_timeout(uint64_t limit_ns, void* stream) {
  if (limit_ns == 0 || limit_ns > 1000000000ull) return ZL_EINVAL;
  int sms = 0;
  const zl_status st = device_sms(&sms);
  if (st != ZL_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return launch_counted("selftest_wait", s, [&] { return zl::launch_wait_timeout_selftest(limit_ns, s); });
}

}  // extern "C"
