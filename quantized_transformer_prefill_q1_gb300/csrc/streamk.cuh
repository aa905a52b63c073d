// streamk.cuh — the stream-K partition shared by the quantised GEMMs: the k-blocks of all
// output tiles form one list cut into equal contiguous ranges, one per persistent CTA.
#pragma once
#include <algorithm>

namespace pf {
namespace sk {

// n_mt x n_nt tiles of kbt k-blocks each, `total` k-blocks in all, cut into `ctas` contiguous
// ranges. Units [late0, ctas) start later than the others (the scheduler places the CTAs
// launched last on SMs that the previous kernel still holds), so each of them takes dk
// k-blocks fewer: the ranges are equal on a virtual list in which every late unit's range is
// padded by dk k-blocks. dk = 0 gives CTA c [total c / ctas, total (c + 1) / ctas).
struct Plan {
  int n_mt, n_nt, kbt;
  long long total;
  int ctas;
  int late0, dk;  // dk <= total / ctas - 1 keeps every range non-empty
  __host__ __device__ __forceinline__ long long begin(int c) const {
    const long long vt = total + static_cast<long long>(ctas - late0) * dk;
    return vt * c / ctas - static_cast<long long>(dk) * (c > late0 ? c - late0 : 0);
  }
  // unit whose range holds k-block w (the unskewed guess is off by a few units at most)
  __host__ __device__ __forceinline__ int owner(long long w) const {
    int c = static_cast<int>(((w + 1) * ctas - 1) / total);
    while (c > 0 && begin(c) > w) --c;
    while (c + 1 < ctas && begin(c + 1) <= w) ++c;
    return c;
  }
  // scratch slot (0 or 1) of contributor c's partial for `tile`: 0 if c's range begins
  // inside the tile, 1 if it begins at or before the tile's start
  __host__ __device__ __forceinline__ int slot(int c, int tile) const {
    return begin(c) > static_cast<long long>(tile) * kbt ? 0 : 1;
  }
};

struct Segment {
  int tile, mt, nt, kb0, nkb;
  bool whole;
};

// The segments of one CTA's range in processing order: the partial first and last
// segments (if any) come first, the shorter of the two ahead (its epilogue then runs under
// the longer one's main loop), then the whole tiles in k order.
struct Range {
  long long b, e;
  int t0, n, first_part, last_part;
  bool swap;  // the partial last segment runs first
  __host__ __device__ __forceinline__ Range(const Plan& p, int c) {
    b = p.begin(c);
    e = p.begin(c + 1);
    t0 = static_cast<int>(b / p.kbt);
    const int t1 = static_cast<int>((e - 1) / p.kbt);
    n = t1 - t0 + 1;
    const long long s0_end = std::min<long long>(e, static_cast<long long>(t0 + 1) * p.kbt);
    first_part = (b == static_cast<long long>(t0) * p.kbt && s0_end - b == p.kbt) ? 0 : 1;
    last_part = (n > 1 && e != static_cast<long long>(t1 + 1) * p.kbt) ? 1 : 0;
    swap = first_part && last_part && e - static_cast<long long>(t1) * p.kbt < s0_end - b;
  }
  __host__ __device__ __forceinline__ Segment at(const Plan& p, int k) const {
    int i = k < first_part ? 0 : (k < first_part + last_part ? n - 1 : k - last_part);
    if (swap && k < 2) i = k == 0 ? n - 1 : 0;
    Segment s;
    s.tile = t0 + i;
    const long long ts = static_cast<long long>(s.tile) * p.kbt;
    const long long lo = std::max(b, ts), hi = std::min(e, ts + p.kbt);
    s.kb0 = static_cast<int>(lo - ts);
    s.nkb = static_cast<int>(hi - lo);
    s.whole = s.nkb == p.kbt;
    s.nt = s.tile / p.n_mt;
    s.mt = s.tile - s.nt * p.n_mt;  // token tiles fastest: neighbouring tiles share weights
    return s;
  }
};


}  // namespace sk
}  // namespace pf
