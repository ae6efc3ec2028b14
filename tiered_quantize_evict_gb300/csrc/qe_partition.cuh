// qe_partition.cuh -- the integer arithmetic that cuts one layer's unit x tile sequence into the
// attention launch's cost-weighted ranges (stream-K).  Host and device: the host test builds it
// and checks every function against its definition.
//
// Every quotient is exact.  32-bit divisions are used wherever the operands fit, because a
// 64-bit integer division is a long software sequence at the start of every launch.
#pragma once
#include "qe_common.cuh"

namespace qe {

// floor(a / b), b > 0
QE_HD unsigned long long udiv_fit(unsigned long long a, unsigned b) {
  return a <= 0xFFFFFFFFull ? (unsigned long long)((unsigned)a / b) : a / b;
}

// Tile order inside a unit: the nbt bf16 sub-tiles and the nq 2-bit windows are interleaved
// evenly: tile i is a 2-bit window iff floor((i+1) nq / n) > floor(i nq / n), n = nbt + nq.
// The number of 2-bit windows among tiles [0, i):
QE_HD int tiles_q_before(int i, int nq, int n) {
  return (int)udiv_fit((unsigned long long)i * (unsigned)nq, (unsigned)n);
}
// cost position of tile i inside its unit (bf16 sub-tile cost cb, 2-bit window cost cq)
QE_HD long long tile_cost_start(int i, int nq, int n, int cb, int cq) {
  const int qb = tiles_q_before(i, nq, n);
  return (long long)(i - qb) * cb + (long long)qb * cq;
}

// End of the cost ranges before warp w (0 <= w <= NW) of a layer of `units` units of cost Cu:
// ceil(w C / NW) with C = units Cu, written as k Cu + c with k = floor(w units / NW) and
// 0 <= c = ceil(Cu (w units mod NW) / NW) <= Cu.
struct RangeEnd {
  long long x, c;
  int k;
};
QE_HD RangeEnd range_end(long long Cu, int NW, int units, int w) {
  const unsigned nw = (unsigned)NW;
  const unsigned long long a = (unsigned long long)w * (unsigned)units;
  const unsigned long long k = udiv_fit(a, nw);
  const unsigned long long rem = a - k * nw;
  RangeEnd e;
  e.c = (long long)udiv_fit((unsigned long long)Cu * rem + (nw - 1), nw);
  e.k = (int)k;
  e.x = (long long)k * Cu + e.c;
  return e;
}

// Index of bf16 tile number loc (bf16 order) in the interleaved order: tiles [0, j) hold
// j - floor(j nq / n) = ceil(j nbt / n) bf16 tiles, so the smallest j holding more than loc of
// them is floor(loc n / nbt) + 1 and the tile is j - 1.
QE_HD int bf16_tile_index(int loc, int n, int nbt) {
  return (int)udiv_fit((unsigned long long)loc * (unsigned)n, (unsigned)nbt);
}

// Where the first tile starting at or after cost position r (0 <= r < Cu) of a unit lies,
// roughly: tile i starts less than |cb - cq| from i Cu / n, so the answer is within
// |cb - cq| / min(cb, cq) + 1 tiles of floor(r n / Cu).
QE_HD long long first_tile_estimate(long long r, int n, long long Cu) {
  const unsigned long long rn = (unsigned long long)r * (unsigned)n;
  return Cu <= 0xFFFFFFFFll ? (long long)udiv_fit(rn, (unsigned)Cu) : (long long)(rn / (unsigned long long)Cu);
}

}  // namespace qe
