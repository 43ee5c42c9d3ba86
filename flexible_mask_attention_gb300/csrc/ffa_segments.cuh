// Tile classification of one slice against one q-tile (forward) or one k-tile
// (backward), in closed form.
//
// Inside slice s = ([qs,qe), [ks,ke), t) query row i sees keys [lo(i), hi(i))
// with lo(i) = ks + (t & 2 ? i - qs : 0) and hi(i) = ke - (t & 1 ? qe-1-i : 0)
// (MagiAttention, card "Calculate KV Interval Boundaries for Mask Types").
// Both bounds are non-decreasing in i, and the rows whose interval is
// non-empty are contiguous, so over a block of rows the union of the
// intervals is [lo(first), hi(last)) and their intersection is
// [lo(last), hi(first)).  Every tile of the union holds a visible entry; a
// tile is FULL (every entry visible) exactly when every row of the q-tile is
// a non-empty row of the slice and the k-tile lies inside the intersection.
// The backward view swaps the roles: key column c is seen by rows
// [qlo(c), qhi(c)) with qlo(c) = max(qs, t & 1 ? c + qe - ke : qs) and
// qhi(c) = min(qe, t & 2 ? c - ks + qs + 1 : qe).
#pragma once

namespace ffa {

struct TileRun {
  int b, fb, fe, e;  // tiles [b, e) are visited; [fb, fe) of them are FULL (fb == fe: none)
};

struct SliceDesc {
  int qs, qe, ks, ke, t;
};

__host__ __device__ inline int div_floor128(int x) { return x >> 7; }
__host__ __device__ inline int div_ceil128(int x) { return (x + 127) >> 7; }

// Tiles of k visited by q-tile `qt` under slice s.  Returns false when none.
__host__ __device__ inline bool fwd_tile_run(const SliceDesc& s, int qt, TileRun& run) {
  const int R0 = qt * 128, R1 = R0 + 128;
  const int qlen = s.qe - s.qs, klen = s.ke - s.ks;
  if (qlen <= 0 || klen <= 0) return false;
  const int r0 = s.qs > R0 ? s.qs : R0;
  const int r1 = s.qe < R1 ? s.qe : R1;
  if (r0 >= r1) return false;
  int v0 = r0, v1 = r1;  // rows of [r0, r1) whose interval is non-empty
  if (s.t == 1) {
    const int first = s.qe - klen;  // hi(i) > lo(i) = ks  <=>  i >= qe - klen
    if (first > v0) v0 = first;
  } else if (s.t == 2) {
    const int last = s.qs + klen;   // lo(i) < hi(i) = ke  <=>  i < qs + klen
    if (last < v1) v1 = last;
  } else if (s.t == 3) {
    if (klen < qlen) return false;  // band width klen - qlen + 1 <= 0
  }
  if (v0 >= v1) return false;
  const int lo_first = s.ks + ((s.t & 2) ? v0 - s.qs : 0);
  const int lo_last = s.ks + ((s.t & 2) ? (v1 - 1) - s.qs : 0);
  const int hi_first = s.ke - ((s.t & 1) ? s.qe - 1 - v0 : 0);
  const int hi_last = s.ke - ((s.t & 1) ? s.qe - 1 - (v1 - 1) : 0);
  run.b = div_floor128(lo_first);
  run.e = div_ceil128(hi_last);
  run.fb = run.fe = run.e;
  if (v0 == R0 && v1 == R1 && lo_last < hi_first) {
    const int a = div_ceil128(lo_last), z = div_floor128(hi_first);
    if (a < z) {
      run.fb = a;
      run.fe = z;
    }
  }
  return true;
}

// Tiles of q visited by k-tile `kt` under slice s.  Returns false when none.
__host__ __device__ inline bool bwd_tile_run(const SliceDesc& s, int kt, TileRun& run) {
  const int C0 = kt * 128, C1 = C0 + 128;
  const int qlen = s.qe - s.qs, klen = s.ke - s.ks;
  if (qlen <= 0 || klen <= 0) return false;
  const int c0 = s.ks > C0 ? s.ks : C0;
  const int c1 = s.ke < C1 ? s.ke : C1;
  if (c0 >= c1) return false;
  if (s.t == 3 && klen < qlen) return false;  // no row sees anything
  // Every column of the slice is seen by some row for types 0..2 and for a
  // non-empty band, so all of [c0, c1) counts.
  auto qlo = [&](int c) {
    const int a = (s.t & 1) ? c + s.qe - s.ke : s.qs;
    return a > s.qs ? a : s.qs;
  };
  auto qhi = [&](int c) {
    const int a = (s.t & 2) ? c - s.ks + s.qs + 1 : s.qe;
    return a < s.qe ? a : s.qe;
  };
  const int u_lo = qlo(c0), u_hi = qhi(c1 - 1);
  const int i_lo = qlo(c1 - 1), i_hi = qhi(c0);
  run.b = div_floor128(u_lo);
  run.e = div_ceil128(u_hi);
  run.fb = run.fe = run.e;
  if (c0 == C0 && c1 == C1 && i_lo < i_hi) {
    const int a = div_ceil128(i_lo), z = div_floor128(i_hi);
    if (a < z) {
      run.fb = a;
      run.fe = z;
    }
  }
  return true;
}

// Visible (q, k) pairs of one slice: sum over its rows of |[lo(i), hi(i))|.
__host__ __device__ inline long long slice_area(const SliceDesc& s) {
  const long long qlen = s.qe - s.qs, klen = s.ke - s.ks;
  if (qlen <= 0 || klen <= 0) return 0;
  switch (s.t) {
    case 0:
      return qlen * klen;
    case 1:
    case 2: {  // rows keep klen, klen-1, ... keys until they run out
      const long long n = qlen < klen ? qlen : klen;
      return n * klen - n * (n - 1) / 2;
    }
    default:
      return klen >= qlen ? qlen * (klen - qlen + 1) : 0;
  }
}

}  // namespace ffa
