// Work-item decoding shared by the forward kernels: the host scheduler
// numbers items segment by segment (head-major over the segment's head range,
// query block of a.rows_per_item rows fastest).
#pragma once
#include "launch.h"

namespace zl {

struct FwdWork {
  int seg;
  int h;
  int qb;
};

__device__ __forceinline__ FwdWork decode_fwd(const FwdArgs& a, int it) {
  int lo = 0, hi = a.n_segs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (a.segs[mid].item0 <= it) lo = mid; else hi = mid - 1;
  }
  const FwdSeg& s = a.segs[lo];
  const int nqb = (s.q_len + a.rows_per_item - 1) / a.rows_per_item;
  const int local = it - s.item0;
  return {lo, s.h0 + local / nqb, local % nqb};
}

}  // namespace zl
