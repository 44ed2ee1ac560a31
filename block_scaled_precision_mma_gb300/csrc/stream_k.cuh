// stream_k.cuh -- work split of a persistent GEMM launch: whole output tiles round robin,
// and the last wave's tiles split along K over the workers that would otherwise idle
// (stream-K).  Shared by the dense SM-pair kernel (a worker: one SM pair) and the grouped
// BF16 kernel (a worker: one CTA).
//
// A split tile's K range is cut into granules of `gran` k-stages; each worker with a
// stream-K range takes a contiguous share of the granules of the split tiles, writes
// its partial sums of each tile it touches to its own slot, and the last worker to
// arrive at a tile adds every contributor's slot in K order (a fixed order, so results
// do not depend on which worker arrives last).
#pragma once
#include <cstdint>

namespace bsmma {

// Units [0, t_dp) whole and round robin; the P workers with a stream-K range share W
// granules of units [t_dp, units), gpu granules per unit.
struct DSched {
  int units, KS, gran, gpu, t_dp, P, W;
};

// cost_stages: the extra time of a split range (pipeline start, partial sums written and
// added) in k-stages of one unit's own time; min_granules: the shortest range worth a
// split.  The tail wave's `rem` units are split only when rem / workers of a unit plus
// that cost beats the wave's one whole unit, and only when the split puts more workers
// to work.
__device__ __forceinline__ DSched make_dsched(int units, int KS, int gran, int workers,
                                              bool can_split, int cost_stages, int min_granules) {
  DSched s;
  s.units = units;
  s.KS = KS;
  s.gran = gran;
  s.gpu = (KS + gran - 1) / gran;
  s.t_dp = units;
  s.P = 0;
  s.W = 0;
  const int rem = units % workers;
  if (can_split && rem != 0 &&
      static_cast<int64_t>(rem) * KS <= static_cast<int64_t>(workers) * (KS - cost_stages)) {
    const int64_t W = static_cast<int64_t>(rem) * s.gpu;
    int64_t P = W / min_granules;
    if (P > workers) P = workers;
    if (P > rem && W < INT32_MAX) {
      s.t_dp = units - rem;
      s.P = static_cast<int>(P);
      s.W = static_cast<int>(W);
    }
  }
  return s;
}
// First granule of worker c's stream-K range.
__device__ __forceinline__ int dsk_begin(const DSched& s, int c) {
  return static_cast<int>(static_cast<int64_t>(c) * s.W / s.P);
}
// Worker whose range holds granule `it`.
__device__ __forceinline__ int dsk_owner(const DSched& s, int it) {
  return static_cast<int>((static_cast<int64_t>(it + 1) * s.P - 1) / s.W);
}
// Work item of a warp: unit u, stages [ks0, ks1).  The position (next whole unit, next
// granule, end) lives in shared memory, one copy per warp, so it costs no registers.
__device__ __forceinline__ void dwork_init(const DSched& s, volatile int* st, int c) {
  st[0] = c;
  st[1] = c < s.P ? dsk_begin(s, c) : 0;
  st[2] = c < s.P ? dsk_begin(s, c + 1) : 0;
}
__device__ __forceinline__ bool dwork_next(const DSched& s, volatile int* st, int workers, int& u,
                                           int& ks0, int& ks1) {
  const int dp = st[0];
  if (dp < s.t_dp) {
    u = dp;
    ks0 = 0;
    ks1 = s.KS;
    st[0] = dp + workers;
    return true;
  }
  const int it = st[1], end = st[2];
  if (it >= end) return false;
  const int v = it / s.gpu;
  const int g0 = it - v * s.gpu;
  const int g1 = s.gpu - g0 <= end - it ? s.gpu : g0 + (end - it);
  st[1] = it + (g1 - g0);
  u = s.t_dp + v;
  ks0 = g0 * s.gran;
  ks1 = g1 * s.gran < s.KS ? g1 * s.gran : s.KS;
  return true;
}
// Workers contributing to split unit v (= u - t_dp): c_lo .. c_hi.
__device__ __forceinline__ int dsk_first_worker(const DSched& s, int v) {
  return dsk_owner(s, v * s.gpu);
}
__device__ __forceinline__ int dsk_last_worker(const DSched& s, int v) {
  return dsk_owner(s, (v + 1) * s.gpu - 1);
}
// Which of worker c's two partial-sum slots holds its part of split unit v: 0 when v is
// the first unit its range touches, else 1 (v is then the last one).  Units strictly
// inside a range are whole and need no slot, so two slots per worker suffice.
__device__ __forceinline__ int dsk_slot(const DSched& s, int c, int v) {
  return dsk_begin(s, c) / s.gpu == v ? 0 : 1;
}

}  // namespace bsmma
