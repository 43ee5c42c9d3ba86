// Slice planner and tile scheduler (device kernels) plus the host side of the
// C ABI declared in include/ffa.h.
//
// Work-list specification (all of it computed on the device):
//   * Forward visits of q-tile qt: one per k-tile kt that holds a visible
//     entry, in kt order; kind FULL when one slice makes all 128 x 128
//     entries visible, PARTIAL otherwise; a tile seen by several slices
//     carries the list of those slices (masked by the union of their windows).
//   * Forward units pair two 128-row halves that share K/V tiles:
//       - grouped-query heads (Hq / Hkv >= 2): one q-tile, two query heads of
//         the same kv head; the steps are the q-tile's visits;
//       - otherwise: q-tiles 2u and 2u+1 of one head; the steps merge the two
//         visit lists on kt (equal kt -> one shared step, in list order).
//   * Item cost = sum over its steps and busy halves of 4 (FULL) or 5
//     (PARTIAL).  Items are sorted by cost octave floor(log2(cost + 1))
//     (descending), then kv head, then cost (descending), then index; the
//     persistent kernels draw them in that order from a work queue.
//   * While fewer than `split_below` items have work, each such item is cut
//     into equal runs of steps whose partial results are merged by
//     logsumexp afterwards.
//   * Backward visits of k-tile kt: one per q-tile, merged the same way, in
//     qt order; one item per (kt, kv head), cost g * visit costs.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <vector>

#include "ffa_internal.cuh"

namespace ffa {
namespace {

constexpr int kFullCost = 4, kPartialCost = 5;
constexpr int kMaxLocalSegs = 64;

__global__ void k_pack_slices(const int* __restrict__ qr, const int* __restrict__ kr,
                              const int* __restrict__ ty, int S, Slice* out) {
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s < S) out[s] = Slice{qr[2 * s], qr[2 * s + 1], kr[2 * s], kr[2 * s + 1], ty[s]};
}

// flags[0]: bad range/type, flags[1]: overlap.  area: visible pairs per head.
__global__ void k_check_slices(const Slice* __restrict__ sl, int S, int Tq, int Tk, int* flags,
                               unsigned long long* area) {
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= S) return;
  const Slice x = sl[s];
  if (x.qs < 0 || x.qs > x.qe || x.qe > Tq || x.ks < 0 || x.ks > x.ke || x.ke > Tk || x.t < 0 ||
      x.t > 3) {
    atomicExch(&flags[0], 1);
    return;
  }
  atomicAdd(area, (unsigned long long)slice_area(x));
}

// ---- per-tile slice lists ---------------------------------------------------
// List of tile t: the non-empty slices whose q range (kQ) or k range meets
// rows/keys [128t, 128t+128), in slice order.  One block per tile walks the
// slices 256 at a time; a block scan of the hit flags places each hit, so the
// order never depends on scheduling.  Count mode (list == nullptr) writes the
// list lengths to cnt.
constexpr int kListThreads = 256;

template <bool kQ>
__global__ void __launch_bounds__(kListThreads)
    k_tile_slices(const Slice* __restrict__ sl, int S, const int* __restrict__ off,
                  int* __restrict__ cnt, int* __restrict__ list) {
  __shared__ int warp_tot[kListThreads / 32];
  const int t = blockIdx.x, lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int lo = t * 128, hi = lo + 128;
  int base = list ? off[t] : 0;
  for (int s0 = 0; s0 < S; s0 += kListThreads) {
    const int s = s0 + threadIdx.x;
    bool hit = false;
    if (s < S) {
      const Slice x = sl[s];
      if (x.qs < x.qe && x.ks < x.ke)
        hit = kQ ? (x.qs < hi && x.qe > lo) : (x.ks < hi && x.ke > lo);
    }
    const unsigned m = __ballot_sync(0xffffffffu, hit);
    if (lane == 0) warp_tot[w] = __popc(m);
    __syncthreads();
    int before = 0, total = 0;
    for (int i = 0; i < kListThreads / 32; ++i) {
      before += i < w ? warp_tot[i] : 0;
      total += warp_tot[i];
    }
    if (hit && list) list[base + before + __popc(m & ((1u << lane) - 1u))] = s;
    base += total;
    __syncthreads();
  }
  if (!list && threadIdx.x == 0) cnt[t] = base;
}

// Two non-empty slices overlap iff their rectangles meet; then they share a
// row, hence a q-tile, so only pairs within one q-tile's list are compared.
// Lists of up to kSweepMax slices are sorted by k start in shared memory and
// swept: slice i is compared only with the following slices that start
// before its k end (the only ones whose k range can meet it).  Longer lists
// compare every pair.
constexpr int kSweepMax = 4096;

__global__ void __launch_bounds__(kListThreads)
    k_check_overlap(const Slice* __restrict__ sl, const int* __restrict__ list,
                    const int* __restrict__ off, const int* __restrict__ cnt, int* flags) {
  __shared__ unsigned long long key[kSweepMax];  // (k start << 32) | list position
  const int* L = list + off[blockIdx.x];
  const int n = cnt[blockIdx.x];
  if (n > kSweepMax) {
    for (int i = threadIdx.x; i < n; i += kListThreads) {
      const Slice a = sl[L[i]];
      for (int j = i + 1; j < n; ++j) {
        const Slice b = sl[L[j]];
        if (a.qs < b.qe && b.qs < a.qe && a.ks < b.ke && b.ks < a.ke) {
          atomicExch(&flags[1], 1);
          return;
        }
      }
    }
    return;
  }
  int n2 = 1;
  while (n2 < n) n2 <<= 1;
  for (int i = threadIdx.x; i < n2; i += kListThreads)
    key[i] = i < n ? ((unsigned long long)(unsigned)sl[L[i]].ks << 32) | (unsigned)i : ~0ull;
  __syncthreads();
  for (int k = 2; k <= n2; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n2; i += kListThreads) {
        const int l = i ^ j;
        if (l > i) {
          const unsigned long long a = key[i], b = key[l];
          if ((a > b) == ((i & k) == 0)) {
            key[i] = b;
            key[l] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  for (int i = threadIdx.x; i < n; i += kListThreads) {
    const Slice a = sl[L[key[i] & 0xffffffffu]];
    for (int j = i + 1; j < n && (int)(key[j] >> 32) < a.ke; ++j) {
      const Slice b = sl[L[key[j] & 0xffffffffu]];
      if (a.qs < b.qe && b.qs < a.qe) {  // k ranges meet: b.ks in [a.ks, a.ke)
        atomicExch(&flags[1], 1);
        return;
      }
    }
  }
}

// Single-block exclusive scan of n int32 counts; total in *total.
__device__ __forceinline__ int warp_sum(int v) {
  for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
  return v;
}

__global__ void k_scan(const int* __restrict__ in, int n, int* __restrict__ out, long long* total,
                       long long* nonzero) {
  __shared__ long long part[1024];
  const int T = blockDim.x, t = threadIdx.x;
  const int per = (n + T - 1) / T;
  const int b = t * per, e = min(n, b + per);
  long long s = 0;
  int nz = 0;
  for (int i = b; i < e; ++i) {
    s += in[i];
    nz += in[i] != 0;
  }
  if (nonzero) {  // entries that are not zero
    nz = warp_sum(nz);
    if ((t & 31) == 0 && nz) atomicAdd(reinterpret_cast<unsigned long long*>(nonzero), (unsigned long long)nz);
  }
  part[t] = s;
  __syncthreads();
  for (int off = 1; off < T; off <<= 1) {
    long long v = t >= off ? part[t - off] : 0;
    __syncthreads();
    part[t] += v;
    __syncthreads();
  }
  long long run = part[t] - s;
  for (int i = b; i < e; ++i) {
    out[i] = (int)run;
    run += in[i];
  }
  if (t == T - 1) *total = part[t];
}

// ---- visits -----------------------------------------------------------------
// One warp per tile: the lanes collect the runs of the slices in the tile's
// list (kept in shared memory, in slice order), then walk the tile's visited
// range 32 positions at a time.  A position seen by one slice becomes one
// visit with that slice's info; a position seen by several (all PARTIAL,
// since slices are disjoint) becomes one visit whose info points at a slice
// list [n, s_0 .. s_n-1] in `masks`.  Warp scans of the per-position counts
// place visits and list entries, so the output never depends on scheduling.
// Count mode (kCount) only stores the tile's visit and list-word totals.
// Tiles with more than kMaxLocalSegs runs over at most kSweepPositions
// positions are swept instead: one pass over the slice list counts each
// position's runs in shared memory, a second places the slice lists.  Other
// tiles with more than kMaxLocalSegs runs re-read the slice list for every
// position.
constexpr int kFillWarps = 4;
constexpr int kSweepPositions = 256;

template <bool kFwd, bool kCount>
__global__ void __launch_bounds__(32 * kFillWarps)
    k_visit_warp(const Slice* __restrict__ sl, const int* __restrict__ list,
                 const int* __restrict__ loff, const int* __restrict__ lcnt, int n_tiles,
                 int* __restrict__ vcnt, int* __restrict__ mcnt, const int* __restrict__ voff,
                 const int* __restrict__ moff, int2* __restrict__ visits,
                 int* __restrict__ masks) {
  __shared__ TileRun seg[kFillWarps][kMaxLocalSegs];
  __shared__ int seg_s[kFillWarps][kMaxLocalSegs];
  __shared__ int sweep_cnt[kFillWarps][kSweepPositions];
  __shared__ int sweep_first[kFillWarps][kSweepPositions];
  __shared__ int sweep_ptr[kFillWarps][kSweepPositions];
  const int wib = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x * kFillWarps + wib;
  if (tile >= n_tiles) return;  // whole warp leaves together
  const int* L = list + loff[tile];
  const int S = lcnt[tile];
  int nseg = 0, lo = 0x7fffffff, hi = 0;
  for (int s0 = 0; s0 < S; s0 += 32) {
    const int s = s0 + lane < S ? L[s0 + lane] : -1;
    TileRun r;
    const bool ok = s >= 0 && (kFwd ? fwd_tile_run(sl[s], tile, r) : bwd_tile_run(sl[s], tile, r));
    const unsigned m = __ballot_sync(0xffffffffu, ok);
    if (ok) {
      const int pos = nseg + __popc(m & ((1u << lane) - 1u));
      if (pos < kMaxLocalSegs) {
        seg[wib][pos] = r;
        seg_s[wib][pos] = s;
      }
      lo = min(lo, r.b);
      hi = max(hi, r.e);
    }
    nseg += __popc(m);
  }
  for (int d = 16; d > 0; d >>= 1) {
    lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, d));
    hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, d));
  }
  __syncwarp();
  const bool overflow = nseg > kMaxLocalSegs;
  if (overflow && hi - lo <= kSweepPositions) {
    // Many runs over few positions (fine block-sparse tables): one pass over
    // the list counts, per position, its runs and the first of them.
    int* cnt = sweep_cnt[wib];
    int* first = sweep_first[wib];
    int* ptr = sweep_ptr[wib];
    const int P = hi - lo;
    for (int xi = lane; xi < P; xi += 32) {
      cnt[xi] = 0;
      first[xi] = 0x7fffffff;
    }
    __syncwarp();
    for (int i = lane; i < S; i += 32) {
      TileRun r;
      if (kFwd ? fwd_tile_run(sl[L[i]], tile, r) : bwd_tile_run(sl[L[i]], tile, r)) {
        for (int x = r.b; x < r.e; ++x) {
          atomicAdd(&cnt[x - lo], 1);
          atomicMin(&first[x - lo], i);
        }
      }
    }
    __syncwarp();
    int vbase = kCount ? 0 : voff[tile], mbase = kCount ? 0 : moff[tile];
    for (int x0 = 0; x0 < P; x0 += 32) {
      const int xi = x0 + lane, x = lo + xi;
      int c = 0, first_s = 0;
      bool first_partial = false;
      if (xi < P && (c = cnt[xi]) > 0) {
        first_s = L[first[xi]];
        TileRun r;
        if (kFwd) fwd_tile_run(sl[first_s], tile, r);
        else bwd_tile_run(sl[first_s], tile, r);
        first_partial = !(x >= r.fb && x < r.fe);
      }
      const int vis = c > 0 ? 1 : 0, msz = c >= 2 ? c + 1 : 0;
      int vi = vis, mi = msz;
      for (int d = 1; d < 32; d <<= 1) {
        const int a = __shfl_up_sync(0xffffffffu, vi, d), b = __shfl_up_sync(0xffffffffu, mi, d);
        if (lane >= d) {
          vi += a;
          mi += b;
        }
      }
      if (!kCount && c > 0) {
        int info = visit_info(first_s, first_partial);
        if (c >= 2) {
          const int m = mbase + mi - msz;
          info = visit_list_info(m);
          masks[m] = c;
          ptr[xi] = m + 1;
        }
        visits[vbase + vi - vis] = make_int2(x, info);
      }
      vbase += __shfl_sync(0xffffffffu, vi, 31);
      mbase += __shfl_sync(0xffffffffu, mi, 31);
    }
    if (kCount) {
      if (lane == 0) {
        vcnt[tile] = vbase;
        mcnt[tile] = mbase;
      }
      return;
    }
    __syncwarp();
    // Slice lists of the positions with several runs, in list order: the
    // list is walked 32 entries at a time, and lanes whose runs meet at a
    // position take consecutive places in lane order.
    for (int i0 = 0; i0 < S; i0 += 32) {
      const int i = i0 + lane;
      TileRun r;
      r.b = r.e = 0;
      int s_i = -1;
      if (i < S) {
        s_i = L[i];
        if (!(kFwd ? fwd_tile_run(sl[s_i], tile, r) : bwd_tile_run(sl[s_i], tile, r))) r.b = r.e = 0;
      }
      int len = r.e - r.b, maxlen = len;
      for (int d = 16; d > 0; d >>= 1) maxlen = max(maxlen, __shfl_xor_sync(0xffffffffu, maxlen, d));
      for (int j = 0; j < maxlen; ++j) {
        const bool act = j < len && cnt[r.b + j - lo] >= 2;
        const unsigned m = __match_any_sync(0xffffffffu, act ? r.b + j : -1 - lane);
        const unsigned before = m & ((1u << lane) - 1u);
        int base = 0;
        if (act) base = ptr[r.b + j - lo];
        __syncwarp();
        if (act) {
          masks[base + __popc(before)] = s_i;
          if (before == 0u) ptr[r.b + j - lo] = base + __popc(m);
        }
        __syncwarp();
      }
    }
    return;
  }
  const int n_src = overflow ? S : nseg;
  // run i of this tile (slice index in *s); false when the slice has none
  auto run_of = [&](int i, TileRun& r, int& s) -> bool {
    if (!overflow) {
      r = seg[wib][i];
      s = seg_s[wib][i];
      return true;
    }
    s = L[i];
    return kFwd ? fwd_tile_run(sl[s], tile, r) : bwd_tile_run(sl[s], tile, r);
  };
  int vbase = kCount ? 0 : voff[tile], mbase = kCount ? 0 : moff[tile];
  for (int x0 = lo; x0 < hi; x0 += 32) {
    const int x = x0 + lane;
    int cnt = 0, first_s = 0;
    bool first_partial = false;
    if (x < hi) {
      for (int i = 0; i < n_src; ++i) {
        TileRun r;
        int s;
        if (run_of(i, r, s) && x >= r.b && x < r.e) {
          if (cnt == 0) {
            first_s = s;
            first_partial = !(x >= r.fb && x < r.fe);
          }
          ++cnt;
        }
      }
    }
    const int vis = cnt > 0 ? 1 : 0, msz = cnt >= 2 ? cnt + 1 : 0;
    int vi = vis, mi = msz;
    for (int d = 1; d < 32; d <<= 1) {
      const int a = __shfl_up_sync(0xffffffffu, vi, d), b = __shfl_up_sync(0xffffffffu, mi, d);
      if (lane >= d) {
        vi += a;
        mi += b;
      }
    }
    if (!kCount && cnt > 0) {
      int info = visit_info(first_s, first_partial);
      if (cnt >= 2) {
        int m = mbase + mi - msz;
        info = visit_list_info(m);
        masks[m++] = cnt;
        for (int i = 0; i < n_src; ++i) {
          TileRun r;
          int s;
          if (run_of(i, r, s) && x >= r.b && x < r.e) masks[m++] = s;
        }
      }
      visits[vbase + vi - vis] = make_int2(x, info);
    }
    vbase += __shfl_sync(0xffffffffu, vi, 31);
    mbase += __shfl_sync(0xffffffffu, mi, 31);
  }
  if (kCount && lane == 0) {
    vcnt[tile] = vbase;
    mcnt[tile] = mbase;
  }
}

__device__ __forceinline__ int visit_cost(int info) {
  return (info & 1) ? kPartialCost : kFullCost;
}

// Steps of forward unit u.  pair_mode 0: heads share q-tile u.  1: q-tiles
// 2u and 2u+1 share a head; visits merged on kt.
__global__ void k_fwd_unit_count(const int2* __restrict__ visits, const int* __restrict__ voff,
                                 const int* __restrict__ vcnt, int n_qt, int n_units,
                                 int pair_mode, int* scnt, int* cost_half) {
  const int u = blockIdx.x * blockDim.x + threadIdx.x;
  if (u >= n_units) return;
  if (pair_mode == 0) {
    const int2* a = visits + voff[u];
    int c = 0;
    for (int i = 0; i < vcnt[u]; ++i) c += visit_cost(a[i].y);
    scnt[u] = vcnt[u];
    cost_half[2 * u] = cost_half[2 * u + 1] = c;
    return;
  }
  const int qa = 2 * u, qb = 2 * u + 1;
  const int na = vcnt[qa], nb = qb < n_qt ? vcnt[qb] : 0;
  const int2* a = visits + voff[qa];
  const int2* b = qb < n_qt ? visits + voff[qb] : nullptr;
  int i = 0, j = 0, n = 0, ca = 0, cb = 0;
  while (i < na || j < nb) {
    if (j >= nb || (i < na && a[i].x < b[j].x)) {
      ca += visit_cost(a[i].y);
      ++i;
    } else if (i >= na || b[j].x < a[i].x) {
      cb += visit_cost(b[j].y);
      ++j;
    } else {
      ca += visit_cost(a[i].y);
      cb += visit_cost(b[j].y);
      ++i;
      ++j;
    }
    ++n;
  }
  scnt[u] = n;
  cost_half[2 * u] = ca;
  cost_half[2 * u + 1] = cb;
}

__global__ void k_fwd_unit_fill(const int2* __restrict__ visits, const int* __restrict__ voff,
                                const int* __restrict__ vcnt, int n_qt, int n_units,
                                int pair_mode, const int* __restrict__ soff,
                                const int* __restrict__ gcnt, int4* steps) {
  const int u = blockIdx.x * blockDim.x + threadIdx.x;
  if (u >= n_units || gcnt[u] > 0) return;  // gathered units are filled by k_gather_fill
  int4* o = steps + soff[u];
  if (pair_mode == 0) {
    const int2* a = visits + voff[u];
    for (int i = 0; i < vcnt[u]; ++i) o[i] = make_int4(a[i].x, a[i].y, a[i].y, 0);
    return;
  }
  const int qa = 2 * u, qb = 2 * u + 1;
  const int na = vcnt[qa], nb = qb < n_qt ? vcnt[qb] : 0;
  const int2* a = visits + voff[qa];
  const int2* b = qb < n_qt ? visits + voff[qb] : nullptr;
  int i = 0, j = 0, n = 0;
  while (i < na || j < nb) {
    if (j >= nb || (i < na && a[i].x < b[j].x)) {
      o[n] = make_int4(a[i].x, a[i].y, -1, 0);
      ++i;
    } else if (i >= na || b[j].x < a[i].x) {
      o[n] = make_int4(b[j].x, -1, b[j].y, 0);
      ++j;
    } else {
      o[n] = make_int4(a[i].x, a[i].y, b[j].y, 0);
      ++i;
      ++j;
    }
    ++n;
  }
}

// Warp-parallel forms of k_fwd_unit_count / k_fill (one warp per unit; the
// serial ones above stay for key ranges longer than kUnitWarpTiles tiles).
// A unit of two q-tiles merges their visit lists on kt: the k-tiles either
// list holds are marked in shared-memory bitmaps, and a visit's place in the
// merged list is the count of marked k-tiles below it.
constexpr int kUnitWarpTiles = 8192;
constexpr int kUnitWarpWords = kUnitWarpTiles / 32;
constexpr int kUnitWarps = 2;  // warps per block

// Bitmaps of the k-tiles of lists a and b, their union, and exclusive
// prefix counts of the union's and b's words.
struct UnitBits {
  unsigned a[kUnitWarpWords], b[kUnitWarpWords];
  int pre_u[kUnitWarpWords], pre_b[kUnitWarpWords];
};

__device__ void unit_bits(const int2* a, int na, const int2* b, int nb, int words, UnitBits& m) {
  const int lane = threadIdx.x & 31;
  for (int w = lane; w < words; w += 32) m.a[w] = m.b[w] = 0u;
  __syncwarp();
  for (int i = lane; i < na; i += 32) atomicOr(&m.a[a[i].x >> 5], 1u << (a[i].x & 31));
  for (int i = lane; i < nb; i += 32) atomicOr(&m.b[b[i].x >> 5], 1u << (b[i].x & 31));
  __syncwarp();
  int carry_u = 0, carry_b = 0;
  for (int w0 = 0; w0 < words; w0 += 32) {
    const int w = w0 + lane;
    const int cu = w < words ? __popc(m.a[w] | m.b[w]) : 0, cb = w < words ? __popc(m.b[w]) : 0;
    int iu = cu, ib = cb;  // inclusive warp scans
    for (int d = 1; d < 32; d <<= 1) {
      const int yu = __shfl_up_sync(0xffffffffu, iu, d), yb = __shfl_up_sync(0xffffffffu, ib, d);
      if (lane >= d) {
        iu += yu;
        ib += yb;
      }
    }
    if (w < words) {
      m.pre_u[w] = carry_u + iu - cu;
      m.pre_b[w] = carry_b + ib - cb;
    }
    carry_u += __shfl_sync(0xffffffffu, iu, 31);
    carry_b += __shfl_sync(0xffffffffu, ib, 31);
  }
  __syncwarp();
}

__device__ __forceinline__ int rank_below(const unsigned* bits, const int* pre, int x) {
  return pre[x >> 5] + __popc(bits[x >> 5] & ((1u << (x & 31)) - 1u));
}

__global__ void __launch_bounds__(32 * kUnitWarps)
    k_fwd_unit_count_w(const int2* __restrict__ visits, const int* __restrict__ voff,
                       const int* __restrict__ vcnt, int n_qt, int n_units, int pair_mode,
                       int n_kt, int* scnt, int* cost_half) {
  __shared__ UnitBits sm[kUnitWarps];
  const int u = blockIdx.x * kUnitWarps + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (u >= n_units) return;  // whole warp
  if (pair_mode == 0) {
    const int2* a = visits + voff[u];
    int c = 0;
    for (int i = lane; i < vcnt[u]; i += 32) c += visit_cost(a[i].y);
    c = warp_sum(c);
    if (lane == 0) {
      scnt[u] = vcnt[u];
      cost_half[2 * u] = cost_half[2 * u + 1] = c;
    }
    return;
  }
  const int qa = 2 * u, qb = 2 * u + 1;
  const int na = vcnt[qa], nb = qb < n_qt ? vcnt[qb] : 0;
  const int2* a = visits + voff[qa];
  const int2* b = qb < n_qt ? visits + voff[qb] : visits;
  UnitBits& m = sm[threadIdx.x >> 5];
  const int words = (n_kt + 31) / 32;
  unit_bits(a, na, b, nb, words, m);
  int ca = 0, cb = 0, common = 0;
  for (int i = lane; i < na; i += 32) {
    ca += visit_cost(a[i].y);
    common += (m.b[a[i].x >> 5] >> (a[i].x & 31)) & 1u;
  }
  for (int i = lane; i < nb; i += 32) cb += visit_cost(b[i].y);
  ca = warp_sum(ca);
  cb = warp_sum(cb);
  common = warp_sum(common);
  if (lane == 0) {
    scnt[u] = na + nb - common;
    cost_half[2 * u] = ca;
    cost_half[2 * u + 1] = cb;
  }
}

__global__ void __launch_bounds__(32 * kUnitWarps)
    k_fwd_unit_fill_w(const int2* __restrict__ visits, const int* __restrict__ voff,
                      const int* __restrict__ vcnt, int n_qt, int n_units, int pair_mode,
                      int n_kt, const int* __restrict__ soff, const int* __restrict__ gcnt,
                      int4* steps) {
  __shared__ UnitBits sm[kUnitWarps];
  const int u = blockIdx.x * kUnitWarps + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (u >= n_units || gcnt[u] > 0) return;  // whole warp; gathered units: k_gather_fill
  int4* o = steps + soff[u];
  if (pair_mode == 0) {
    const int2* a = visits + voff[u];
    for (int i = lane; i < vcnt[u]; i += 32) o[i] = make_int4(a[i].x, a[i].y, a[i].y, 0);
    return;
  }
  const int qa = 2 * u, qb = 2 * u + 1;
  const int na = vcnt[qa], nb = qb < n_qt ? vcnt[qb] : 0;
  const int2* a = visits + voff[qa];
  const int2* b = qb < n_qt ? visits + voff[qb] : visits;
  UnitBits& m = sm[threadIdx.x >> 5];
  const int words = (n_kt + 31) / 32;
  unit_bits(a, na, b, nb, words, m);
  for (int i = lane; i < na; i += 32) {
    const int x = a[i].x;
    const bool in_b = (m.b[x >> 5] >> (x & 31)) & 1u;
    const int pos = m.pre_u[x >> 5] + __popc((m.a[x >> 5] | m.b[x >> 5]) & ((1u << (x & 31)) - 1u));
    o[pos] = make_int4(x, a[i].y, in_b ? b[rank_below(m.b, m.pre_b, x)].y : -1, 0);
  }
  for (int j = lane; j < nb; j += 32) {
    const int x = b[j].x;
    if ((m.a[x >> 5] >> (x & 31)) & 1u) continue;  // merged with a's visit above
    const int pos = m.pre_u[x >> 5] + __popc((m.a[x >> 5] | m.b[x >> 5]) & ((1u << (x & 31)) - 1u));
    o[pos] = make_int4(x, -1, b[j].y, 0);
  }
}

__global__ void k_fwd_items(int n_items, int pair_mode, int m, int alternate, int g, int Hkv,
                            int Hq, int pairs,
                            int n_qt, const int* __restrict__ soff, const int* __restrict__ scnt,
                            const int* __restrict__ cost_half, int* items) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= n_items) return;
  int u, qt0, qt1, h0, h1;
  if (pair_mode == 2) {  // `pairs`: groups of 2m heads, m heads per half
    u = idx / (Hkv * pairs);
    const int rem = idx % (Hkv * pairs);
    const int hk = rem / pairs, p = rem % pairs;
    qt0 = qt1 = u;
    h0 = hk * g + 2 * m * p;
    h1 = alternate ? h0 : (2 * m * p + m < g) ? h0 + m : -1;
    if (h1 < 0) qt1 = -1;
  } else if (pair_mode == 0) {
    u = idx / (Hkv * pairs);
    const int rem = idx % (Hkv * pairs);
    const int hk = rem / pairs, p = rem % pairs;
    qt0 = qt1 = u;
    h0 = hk * g + 2 * p;
    h1 = (2 * p + 1 < g) ? h0 + 1 : -1;
    if (h1 < 0) qt1 = -1;
  } else {
    u = idx / Hq;
    h0 = idx % Hq;
    qt0 = 2 * u;
    qt1 = (2 * u + 1 < n_qt) ? 2 * u + 1 : -1;
    h1 = qt1 >= 0 ? h0 : -1;
  }
  int* it = items + (size_t)idx * kFiWords;
  it[kFiQt0] = qt0;
  it[kFiQt1] = qt1;
  it[kFiH0] = h0;
  it[kFiH1] = h1;
  it[kFiStepBeg] = soff[u];
  it[kFiStepEnd] = soff[u] + scnt[u];
  it[kFiSlot] = -1;
  it[kFiCost] = cost_half[2 * u] + (h1 >= 0 ? cost_half[2 * u + 1] : 0);
}

// Split: chunk counts per item, then the chunked item list and merge groups.
__global__ void k_split_count(const int* __restrict__ items, int n_items, int nsplit, int* chunks,
                              int* slots, int* groups) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n_items) return;
  const int* it = items + (size_t)i * kFiWords;
  const int n = it[kFiStepEnd] - it[kFiStepBeg];
  const int c = max(1, min(nsplit, n));
  chunks[i] = c;
  slots[i] = c >= 2 ? c : 0;
  groups[i] = c >= 2 ? 1 : 0;
}

__global__ void k_split_fill(const int* __restrict__ items, int n_items,
                             const int* __restrict__ chunks, const int* __restrict__ coff,
                             const int* __restrict__ soff, const int* __restrict__ goff,
                             int* out_items, int* merges) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n_items) return;
  const int* it = items + (size_t)i * kFiWords;
  const int c = chunks[i];
  const int b = it[kFiStepBeg], n = it[kFiStepEnd] - b;
  for (int k = 0; k < c; ++k) {
    int* o = out_items + (size_t)(coff[i] + k) * kFiWords;
    for (int w = 0; w < kFiWords; ++w) o[w] = it[w];
    if (c >= 2) {
      const int kb = b + (int)((long long)k * n / c), ke = b + (int)((long long)(k + 1) * n / c);
      o[kFiStepBeg] = kb;
      o[kFiStepEnd] = ke;
      o[kFiSlot] = soff[i] + k;
      o[kFiCost] = (int)((long long)it[kFiCost] * (ke - kb) / max(n, 1));
    }
  }
  if (c >= 2) {
    int* m = merges + (size_t)goff[i] * kMgWords;
    m[kMgQt0] = it[kFiQt0];
    m[kMgQt1] = it[kFiQt1];
    m[kMgH0] = it[kFiH0];
    m[kMgH1] = it[kFiH1];
    m[kMgSlotBeg] = soff[i];
    m[kMgSlots] = c;
    m[6] = m[7] = 0;
  }
}

// ---- backward items ---------------------------------------------------------
// One warp per k-tile: its steps (the visits, unless gathered) and the
// items of every kv head.
__global__ void k_bwd_items(int n_kt, int Hkv, int g, const int2* __restrict__ visits,
                            const int* __restrict__ voff, const int* __restrict__ vcnt,
                            const int* __restrict__ soff, const int* __restrict__ gcnt,
                            int4* steps, int* items) {
  const int kt = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (kt >= n_kt) return;  // whole warp
  const int b = soff[kt], ng = gcnt[kt];
  int c = 0, n = ng;
  if (ng > 0) {  // gathered k-tile: its steps are k_bgather_fill's
    c = kPartialCost * ng;
  } else {
    n = vcnt[kt];
    const int2* v = visits + voff[kt];
    for (int i = lane; i < n; i += 32) {
      const int2 x = v[i];
      c += visit_cost(x.y);
      steps[b + i] = make_int4(x.x, x.y, 0, 0);
    }
    c = warp_sum(c);
  }
  for (int hk = lane; hk < Hkv; hk += 32) {
    int* it = items + ((size_t)kt * Hkv + hk) * kBiWords;
    it[kBiKt] = kt;
    it[kBiHkv] = hk;
    it[kBiStepBeg] = b;
    it[kBiStepEnd] = b + n;
    it[kBiCost] = c * g;
    it[5] = it[6] = it[7] = 0;
  }
}

// Visits of each half of the (unsplit) forward items the dQ pass walks: a
// half skips the steps whose info for it is -1.
// alternate: the halves of every item are the same rows, taking the steps in
// turn; the dQ pass walks them as one half over all the steps.
__global__ void k_dq_counts(const int* __restrict__ items, int n_items,
                            const int4* __restrict__ steps, int alternate,
                            int* __restrict__ counts) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n_items) return;
  const int* it = items + (size_t)i * kFiWords;
  int n0 = 0, n1 = 0;
  for (int j = it[kFiStepBeg]; j < it[kFiStepEnd]; ++j) {
    const int4 s = steps[j];
    n0 += (s.y >= 0 || (alternate && s.z >= 0)) ? 1 : 0;
    n1 += (!alternate && s.z >= 0) ? 1 : 0;
  }
  counts[2 * i] = n0;
  counts[2 * i + 1] = n1;
}

// ---- gathered forward units -------------------------------------------------
// One block per forward unit.  A unit gathers when every slice of its q-tiles'
// lists is FULL with ks and ke multiples of kGatherKeys (ke may be Tk), it
// covers 1 .. kGatherMaxBlocks blocks of kGatherKeys keys, and ceil(blocks /
// kGatherSlots) gathered steps are at most 9/10 of its regular steps (a
// gathered step costs about as much as a masked tile step).  The blocks
// are collected in a shared-memory bitmap (order-free, so deterministic).
constexpr int kGatherThreads = 256;
constexpr int kGatherBitmapWords = kGatherMaxTk / kGatherKeys / 32;

struct GatherUnit {
  int qt[2];   // q-tile of each half (-1: none)
  int n_qt;    // distinct q-tiles (1 or 2)
  int p0, p1;  // query rows of the unit: slices outside [p0, p1) are skipped
};

// pair_mode 0: q-tile u (two heads); 1: q-tiles 2u, 2u+1; 2: the slab u of
// `rows` (64 or 32) query rows (head-stacked units).
__device__ __forceinline__ GatherUnit gather_unit(int u, int pair_mode, int n_qt,
                                                  int rows = kSlabRows) {
  GatherUnit g;
  g.p0 = -1;
  g.p1 = 0x7fffffff;
  if (pair_mode == 2) {
    g.qt[0] = g.qt[1] = (rows * u) >> 7;
    g.n_qt = 1;
    g.p0 = rows * u;
    g.p1 = g.p0 + rows;
  } else if (pair_mode == 0) {
    g.qt[0] = g.qt[1] = u;
    g.n_qt = 1;
  } else {
    g.qt[0] = 2 * u;
    g.qt[1] = 2 * u + 1 < n_qt ? 2 * u + 1 : -1;
    g.n_qt = g.qt[1] >= 0 ? 2 : 1;
  }
  return g;
}

// Marks the unit's blocks in `bits` (cleared here); returns false (for the
// whole block) if a slice is not eligible.
// kBwd: the backward's transpose (the unit is a k-tile, the blocks are 8-row
// query blocks of the slices' q ranges, T is Tq).
template <bool kBwd = false>
__device__ bool gather_bitmap(const Slice* __restrict__ sl, const int* __restrict__ list,
                              const int* __restrict__ loff, const int* __restrict__ lcnt,
                              const GatherUnit& gu, int T, unsigned* bits) {
  const int nwords = (((T + kGatherKeys - 1) / kGatherKeys) + 31) / 32;
  for (int w = threadIdx.x; w < nwords; w += blockDim.x) bits[w] = 0u;
  __syncthreads();
  bool bad = false;
  for (int t = 0; t < gu.n_qt; ++t) {
    const int* L = list + loff[gu.qt[t]];
    const int n = lcnt[gu.qt[t]];
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      const Slice x = sl[L[i]];
      if (!kBwd && (x.qe <= gu.p0 || x.qs >= gu.p1)) continue;  // outside the unit's rows
      const int lo = kBwd ? x.qs : x.ks, hi = kBwd ? x.qe : x.ke;
      if (x.t != 0 || lo % kGatherKeys != 0 || (hi % kGatherKeys != 0 && hi != T)) {
        bad = true;
        continue;
      }
      const int b0 = lo / kGatherKeys, b1 = (hi + kGatherKeys - 1) / kGatherKeys;
      for (int w = b0 >> 5; w <= (b1 - 1) >> 5; ++w) {
        const int lo = max(b0 - 32 * w, 0), hi = min(b1 - 32 * w, 32);
        const unsigned m = (hi == 32 ? 0xffffffffu : ((1u << hi) - 1u)) & ~((1u << lo) - 1u);
        atomicOr(&bits[w], m);
      }
    }
  }
  return !__syncthreads_or(bad);
}

// Number of set bits in bits[0, nwords) (block-wide; every thread gets it).
__device__ int block_popc(const unsigned* bits, int nwords, int* red) {
  int c = 0;
  for (int w = threadIdx.x; w < nwords; w += blockDim.x) c += __popc(bits[w]);
  for (int d = 16; d > 0; d >>= 1) c += __shfl_xor_sync(0xffffffffu, c, d);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = c;
  __syncthreads();
  int tot = 0;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) tot += red[i];
  __syncthreads();
  return tot;
}

// gcnt[u] = gathered steps of unit u (0: regular); scnt[u] is replaced by
// it for gathered units.  scnt holds the regular step counts on entry.
__global__ void __launch_bounds__(kGatherThreads)
    k_gather_count(const Slice* __restrict__ sl, const int* __restrict__ list,
                   const int* __restrict__ loff, const int* __restrict__ lcnt, int n_qt,
                   int pair_mode, int Tk, int* __restrict__ scnt, int* __restrict__ gcnt) {
  __shared__ unsigned bits[kGatherBitmapWords];
  __shared__ int red[kGatherThreads / 32];
  const int u = blockIdx.x;
  const GatherUnit gu = gather_unit(u, pair_mode, n_qt);
  const bool ok = gather_bitmap(sl, list, loff, lcnt, gu, Tk, bits);
  const int nwords = (((Tk + kGatherKeys - 1) / kGatherKeys) + 31) / 32;
  const int n = ok ? block_popc(bits, nwords, red) : 0;
  const int steps = (n + kGatherSlots - 1) / kGatherSlots;
  const bool gather = ok && n > 0 && n <= kGatherMaxBlocks && 10 * steps <= 9 * scnt[u];
  if (threadIdx.x == 0) {
    gcnt[u] = gather ? steps : 0;
    if (gather) scnt[u] = steps;
  }
}

// Head-stacked units: slab_steps[u] = gathered steps of the slab u of `rows`
// query rows (0 when one of its slices is not eligible or it has too many
// blocks); tot_steps += the steps, tot_bad += the ineligible slabs, tot_nz
// += the slabs with steps.
__global__ void __launch_bounds__(kGatherThreads)
    k_slab_count(const Slice* __restrict__ sl, const int* __restrict__ list,
                 const int* __restrict__ loff, const int* __restrict__ lcnt, int n_qt, int Tk,
                 int rows, int* __restrict__ slab_steps, long long* tot_steps,
                 long long* tot_bad, long long* tot_nz) {
  __shared__ unsigned bits[kGatherBitmapWords];
  __shared__ int red[kGatherThreads / 32];
  const int u = blockIdx.x;
  const GatherUnit gu = gather_unit(u, 2, n_qt, rows);
  const bool ok = gather_bitmap(sl, list, loff, lcnt, gu, Tk, bits);
  const int nwords = (((Tk + kGatherKeys - 1) / kGatherKeys) + 31) / 32;
  const int n = ok ? block_popc(bits, nwords, red) : 0;
  const int steps = ok && n <= kGatherMaxBlocks ? (n + kGatherSlots - 1) / kGatherSlots : -1;
  if (threadIdx.x == 0) {
    slab_steps[u] = max(steps, 0);
    if (steps >= 0)
      atomicAdd(reinterpret_cast<unsigned long long*>(tot_steps), (unsigned long long)steps);
    else atomicAdd(reinterpret_cast<unsigned long long*>(tot_bad), 1ull);
    if (steps > 0) atomicAdd(reinterpret_cast<unsigned long long*>(tot_nz), 1ull);
  }
}

// Steps, records and half costs of the gathered units.  Dynamic shared
// memory: the bitmap, per-word bit offsets, block starts and per-half row
// masks of up to kGatherMaxBlocks blocks.
constexpr size_t kGatherFillSmem =
    sizeof(unsigned) * kGatherBitmapWords + sizeof(int) * kGatherBitmapWords +
    sizeof(int) * kGatherMaxBlocks + sizeof(unsigned) * 2 * kGatherMaxBlocks * 4;

__global__ void __launch_bounds__(kGatherThreads)
    k_gather_fill(const Slice* __restrict__ sl, const int* __restrict__ list,
                  const int* __restrict__ loff, const int* __restrict__ lcnt, int n_qt,
                  int pair_mode, int rows, int alternate, int Tk,
                  const int* __restrict__ gcnt,
                  const int* __restrict__ goff, const int* __restrict__ soff, int4* steps,
                  int* __restrict__ records, int* __restrict__ cost_half) {
  extern __shared__ unsigned gsm[];
  unsigned* bits = gsm;
  int* woff = reinterpret_cast<int*>(bits + kGatherBitmapWords);
  int* start = woff + kGatherBitmapWords;
  unsigned* rmask = reinterpret_cast<unsigned*>(start + kGatherMaxBlocks);  // [2][blocks][4]
  __shared__ int red[kGatherThreads / 32];
  __shared__ int cost[2];
  const int u = blockIdx.x;
  const int n_steps = gcnt[u];
  if (n_steps == 0) return;  // whole block
  const GatherUnit gu = gather_unit(u, pair_mode, n_qt, rows);
  gather_bitmap(sl, list, loff, lcnt, gu, Tk, bits);
  const int nwords = (((Tk + kGatherKeys - 1) / kGatherKeys) + 31) / 32;
  // exclusive prefix of the words' bit counts (one thread per chunk of words)
  {
    const int per = (nwords + blockDim.x - 1) / blockDim.x;
    const int w0 = threadIdx.x * per, w1 = min(nwords, w0 + per);
    int c = 0;
    for (int w = w0; w < w1; ++w) c += __popc(bits[w]);
    int incl = c;  // inclusive scan over the block's threads, by warps
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += y;
    }
    if (lane == 31) red[wid] = incl;
    __syncthreads();
    int base = 0;
    for (int i = 0; i < wid; ++i) base += red[i];
    int run = base + incl - c;
    for (int w = w0; w < w1; ++w) {
      woff[w] = run;
      run += __popc(bits[w]);
    }
  }
  const int n = n_steps * kGatherSlots;  // slots including unused ones
  for (int i = threadIdx.x; i < n; i += blockDim.x) start[i] = -kGatherKeys;
  for (int i = threadIdx.x; i < 2 * n * 4; i += blockDim.x) rmask[i] = 0u;
  __syncthreads();
  for (int w = threadIdx.x; w < nwords; w += blockDim.x) {
    unsigned m = bits[w];
    int pos = woff[w];
    while (m) {
      const int b = 32 * w + __ffs(m) - 1;
      start[pos++] = b * kGatherKeys;
      m &= m - 1u;
    }
  }
  // row bits: each slice marks its rows of the half's q-tile on its blocks
  for (int h = 0; h < 2; ++h) {
    const int qt = gu.qt[h];
    if (qt < 0 || (h == 1 && pair_mode != 1)) continue;
    const int* L = list + loff[qt];
    const int cnt = lcnt[qt];
    for (int i = threadIdx.x; i < cnt; i += blockDim.x) {
      const Slice x = sl[L[i]];
      uint32_t rb[4] = {0u, 0u, 0u, 0u};
      if (pair_mode == 2) {  // tile rows r, r + rows, ... are all slab row r
        if (x.qe <= gu.p0 || x.qs >= gu.p1) continue;
        const int a = max(x.qs, gu.p0) - gu.p0, b = min(x.qe, gu.p1) - gu.p0;
        for (int o = 0; o < 128; o += rows) add_window(a + o, b + o, rb);
      } else {
        add_window(max(x.qs, 128 * qt) - 128 * qt, min(x.qe, 128 * qt + 128) - 128 * qt, rb);
      }
      const int b0 = x.ks / kGatherKeys, b1 = (x.ke + kGatherKeys - 1) / kGatherKeys;
      for (int b = b0; b < b1; ++b) {
        const int w = b >> 5;
        const int pos = woff[w] + __popc(bits[w] & ((1u << (b & 31)) - 1u));
        for (int k = 0; k < 4; ++k)
          if (rb[k]) atomicOr(&rmask[(h * n + pos) * 4 + k], rb[k]);
      }
    }
  }
  if (threadIdx.x < 2) cost[threadIdx.x] = 0;
  __syncthreads();
  if (pair_mode != 1)  // both halves are the same rows (two heads, or two head pairs)
    for (int i = threadIdx.x; i < n * 4; i += blockDim.x) rmask[n * 4 + i] = rmask[i];
  __syncthreads();
  const int r0 = goff[u], s0 = soff[u];
  for (int i = threadIdx.x; i < n_steps * kGatherWords; i += blockDim.x) {
    const int j = i / kGatherWords, o = i % kGatherWords;
    int v;
    if (o < kGatherSlots) {
      v = start[j * kGatherSlots + o];
    } else {
      const int h = (o - kGatherSlots) / (kGatherSlots * 4);
      const int rem = (o - kGatherSlots) % (kGatherSlots * 4);
      v = (int)rmask[(h * n + j * kGatherSlots + rem / 4) * 4 + rem % 4];
    }
    records[(size_t)(r0 + j) * kGatherWords + o] = v;
  }
  for (int j = threadIdx.x; j < n_steps; j += blockDim.x) {
    int info[2];
    bool slots_used = true;
    for (int k = 0; k < kGatherSlots; ++k) slots_used &= start[j * kGatherSlots + k] >= 0;
    for (int h = 0; h < 2; ++h) {
      unsigned any = 0u, all = ~0u;
      for (int k = 0; k < kGatherSlots * 4; ++k) {
        any |= rmask[(h * n + j * kGatherSlots) * 4 + k];
        all &= rmask[(h * n + j * kGatherSlots) * 4 + k];
      }
      // 0: every slot holds keys and every row sees them all (no mask)
      info[h] = !any ? -1 : (slots_used && all == ~0u ? 0 : 1);
    }
    if (alternate) {  // the halves take the unit's steps in turn
      info[1] = (j & 1) ? info[0] : -1;
      if (j & 1) info[0] = -1;
    }
    for (int h = 0; h < 2; ++h)
      if (info[h] >= 0) atomicAdd(&cost[h], kPartialCost);
    steps[s0 + j] = make_int4(0, info[0], info[1], r0 + j + 1);
  }
  __syncthreads();
  if (threadIdx.x < 2) cost_half[2 * u + threadIdx.x] = cost[threadIdx.x];
}

// Gathered backward units (one block per k-tile): the transpose of the
// forward's.  A k-tile gathers when every slice of its list is FULL with qs
// and qe multiples of kGatherKeys (qe may be Tq), it covers 1 ..
// kGatherMaxBlocks query blocks and ceil(blocks / kGatherSlots) steps are at
// most 9/10 of its visits.  bgcnt[kt] = gathered steps (0: regular);
// bscnt[kt] = the k-tile's step count either way.
__global__ void __launch_bounds__(kGatherThreads)
    k_bgather_count(const Slice* __restrict__ sl, const int* __restrict__ list,
                    const int* __restrict__ loff, const int* __restrict__ lcnt, int Tq,
                    const int* __restrict__ vcnt, int* __restrict__ bgcnt,
                    int* __restrict__ bscnt) {
  __shared__ unsigned bits[kGatherBitmapWords];
  __shared__ int red[kGatherThreads / 32];
  const int kt = blockIdx.x;
  GatherUnit gu;
  gu.qt[0] = kt;
  gu.qt[1] = -1;
  gu.n_qt = 1;
  const bool ok = gather_bitmap<true>(sl, list, loff, lcnt, gu, Tq, bits);
  const int nwords = (((Tq + kGatherKeys - 1) / kGatherKeys) + 31) / 32;
  const int n = ok ? block_popc(bits, nwords, red) : 0;
  const int steps = (n + kGatherSlots - 1) / kGatherSlots;
  const bool gather = ok && n > 0 && n <= kGatherMaxBlocks && 10 * steps <= 9 * vcnt[kt];
  if (threadIdx.x == 0) {
    bgcnt[kt] = gather ? steps : 0;
    bscnt[kt] = gather ? steps : vcnt[kt];
  }
}

// Steps and records of the gathered k-tiles: 16 query-block start rows, then
// 16 x 4 words of key bits (the keys of the k-tile each slot's rows see).
constexpr size_t kBGatherFillSmem =
    sizeof(unsigned) * kGatherBitmapWords + sizeof(int) * kGatherBitmapWords +
    sizeof(int) * kGatherMaxBlocks + sizeof(unsigned) * kGatherMaxBlocks * 4;

__global__ void __launch_bounds__(kGatherThreads)
    k_bgather_fill(const Slice* __restrict__ sl, const int* __restrict__ list,
                   const int* __restrict__ loff, const int* __restrict__ lcnt, int Tq,
                   const int* __restrict__ bgcnt, const int* __restrict__ bgoff,
                   const int* __restrict__ bsoff, int4* steps, int* __restrict__ records) {
  extern __shared__ unsigned gsm[];
  unsigned* bits = gsm;
  int* woff = reinterpret_cast<int*>(bits + kGatherBitmapWords);
  int* start = woff + kGatherBitmapWords;
  unsigned* kmask = reinterpret_cast<unsigned*>(start + kGatherMaxBlocks);  // [blocks][4]
  __shared__ int red[kGatherThreads / 32];
  const int kt = blockIdx.x;
  const int n_steps = bgcnt[kt];
  if (n_steps == 0) return;  // whole block
  GatherUnit gu;
  gu.qt[0] = kt;
  gu.qt[1] = -1;
  gu.n_qt = 1;
  gather_bitmap<true>(sl, list, loff, lcnt, gu, Tq, bits);
  const int nwords = (((Tq + kGatherKeys - 1) / kGatherKeys) + 31) / 32;
  {  // exclusive prefix of the words' bit counts
    const int per = (nwords + blockDim.x - 1) / blockDim.x;
    const int w0 = threadIdx.x * per, w1 = min(nwords, w0 + per);
    int c = 0;
    for (int w = w0; w < w1; ++w) c += __popc(bits[w]);
    int incl = c;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += y;
    }
    if (lane == 31) red[wid] = incl;
    __syncthreads();
    int base = 0;
    for (int i = 0; i < wid; ++i) base += red[i];
    int run = base + incl - c;
    for (int w = w0; w < w1; ++w) {
      woff[w] = run;
      run += __popc(bits[w]);
    }
  }
  const int n = n_steps * kGatherSlots;
  for (int i = threadIdx.x; i < n; i += blockDim.x) start[i] = -kGatherKeys;
  for (int i = threadIdx.x; i < n * 4; i += blockDim.x) kmask[i] = 0u;
  __syncthreads();
  for (int w = threadIdx.x; w < nwords; w += blockDim.x) {
    unsigned m = bits[w];
    int pos = woff[w];
    while (m) {
      start[pos++] = (32 * w + __ffs(m) - 1) * kGatherKeys;
      m &= m - 1u;
    }
  }
  {
    const int* L = list + loff[kt];
    const int cnt = lcnt[kt];
    for (int i = threadIdx.x; i < cnt; i += blockDim.x) {
      const Slice x = sl[L[i]];
      uint32_t kb[4] = {0u, 0u, 0u, 0u};
      add_window(max(x.ks, 128 * kt) - 128 * kt, min(x.ke, 128 * kt + 128) - 128 * kt, kb);
      const int b0 = x.qs / kGatherKeys, b1 = (x.qe + kGatherKeys - 1) / kGatherKeys;
      for (int b = b0; b < b1; ++b) {
        const int w = b >> 5;
        const int pos = woff[w] + __popc(bits[w] & ((1u << (b & 31)) - 1u));
        for (int k = 0; k < 4; ++k)
          if (kb[k]) atomicOr(&kmask[pos * 4 + k], kb[k]);
      }
    }
  }
  __syncthreads();
  const int r0 = bgoff[kt], s0 = bsoff[kt];
  for (int i = threadIdx.x; i < n_steps * kBGatherWords; i += blockDim.x) {
    const int j = i / kBGatherWords, o = i % kBGatherWords;
    const int v = o < kGatherSlots ? start[j * kGatherSlots + o]
                                   : (int)kmask[(j * kGatherSlots) * 4 + (o - kGatherSlots)];
    records[(size_t)(r0 + j) * kBGatherWords + o] = v;
  }
  for (int j = threadIdx.x; j < n_steps; j += blockDim.x)
    steps[s0 + j] = make_int4(0, 1, 0, r0 + j + 1);
}

// ---- ordering ---------------------------------------------------------------
// One block: bitonic sort of keys in `scratch` (n2 = next power of two >= n
// entries), then order[r] = index.  The persistent kernels draw the items in
// this order from a work queue, so the heavy items go first and the light
// ones even out the tail.  The order is by cost octave (descending), then kv
// head, then cost (descending), then index: within an octave the CTAs
// running at one time share few heads, so their K/V (or Q/dO) tiles stay in
// L2.  (Pure kv-head order measured slower: balance comes first.)
// Key bits: [58,64) 63-octave, [50,58) kv head, [24,50) 2^26-1-cost, [0,24) index.
// The keys live in shared memory when they fit (kSortSmemKeys), else in the
// global `scratch`: the network's ~log2(n2)^2/2 passes then cost shared- rather
// than L2-memory latency each.
constexpr int kSortSmemKeys = 16384;

__device__ __forceinline__ unsigned long long sort_key(const int* __restrict__ items, int words,
                                                       int cost_word, int n, int head_word,
                                                       int head_div, int i) {
  if (i >= n) return ~0ull;
  const int* it = items + (size_t)i * words;
  const unsigned long long c = (unsigned int)it[cost_word] & 0x3ffffffu;
  const unsigned long long hk = (unsigned int)(max(it[head_word], 0) / head_div) & 0xffu;
  const unsigned long long oct = 63u - min(63u, (unsigned int)(63 - __clzll((long long)c + 1)));
  return (oct << 58) | (hk << 50) | ((0x3ffffffull - c) << 24) | (unsigned long long)i;
}

__global__ void k_sort_order(const int* __restrict__ items, int words, int cost_word, int n,
                             int n2, unsigned long long* scratch, int* order, int head_word,
                             int head_div) {
  extern __shared__ unsigned long long sort_keys[];
  unsigned long long* keys = n2 <= kSortSmemKeys ? sort_keys : scratch;
  for (int i = threadIdx.x; i < n2; i += blockDim.x) {
    keys[i] = sort_key(items, words, cost_word, n, head_word, head_div, i);
  }
  __syncthreads();
  for (int k = 2; k <= n2; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n2; i += blockDim.x) {
        const int l = i ^ j;
        if (l > i) {
          const unsigned long long a = keys[i], b = keys[l];
          const bool up = (i & k) == 0;
          if ((a > b) == up) {
            keys[i] = b;
            keys[l] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  for (int i = threadIdx.x; i < n; i += blockDim.x) order[i] = (int)(keys[i] & 0xffffffu);
}

// The same network with each thread holding E consecutive keys in registers
// (n2 = 1024 E, 2 <= E <= 16): compare-exchange partners within a thread are
// swapped in registers, partners up to 32 E apart through warp shuffles, and
// only the passes with wider strides go through shared memory with a block
// barrier (15 of the 91 passes for n2 = 8192, instead of all of them).
template <int E>
__device__ __forceinline__ void cmpx(unsigned long long& lo, unsigned long long& hi, bool up) {
  if ((lo > hi) == up) {
    const unsigned long long t = lo;
    lo = hi;
    hi = t;
  }
}

template <int E>
__global__ void __launch_bounds__(1024)
    k_sort_order_blocked(const int* __restrict__ items, int words, int cost_word, int n,
                         int* order, int head_word, int head_div) {
  extern __shared__ unsigned long long sort_keys[];  // n2 = 1024 E keys
  unsigned long long* keys = sort_keys;
  constexpr int n2 = 1024 * E;
  const int t = threadIdx.x, lane = t & 31;
  unsigned long long v[E];
#pragma unroll
  for (int e = 0; e < E; ++e) v[e] = sort_key(items, words, cost_word, n, head_word, head_div, t * E + e);
  bool in_smem = false;
  for (int k = 2; k <= n2; k <<= 1) {
    int j = k >> 1;
    for (; j >= E; j >>= 1) {
      if (j >= 32 * E) {  // partners in other warps: through shared memory
        if (!in_smem) {
#pragma unroll
          for (int e = 0; e < E; ++e) keys[t * E + e] = v[e];
          in_smem = true;
        }
        __syncthreads();
        for (int p = t; p < n2 / 2; p += 1024) {
          const int i = (p / j) * 2 * j + (p % j), l = i + j;
          unsigned long long a = keys[i], b = keys[l];
          cmpx<E>(a, b, (i & k) == 0);
          keys[i] = a;
          keys[l] = b;
        }
        continue;
      }
      if (in_smem) {
        __syncthreads();
#pragma unroll
        for (int e = 0; e < E; ++e) v[e] = keys[t * E + e];
        in_smem = false;
      }
      // partner: lane ^ (j / E), same slot
      const int m = j / E;
      const bool lower = (lane & m) == 0;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const unsigned long long o = __shfl_xor_sync(0xffffffffu, v[e], m);
        const bool up = (((t * E + e) & k) == 0);
        const unsigned long long mn = v[e] < o ? v[e] : o, mx = v[e] < o ? o : v[e];
        v[e] = (lower == up) ? mn : mx;
      }
    }
    if (in_smem) {
      __syncthreads();
#pragma unroll
      for (int e = 0; e < E; ++e) v[e] = keys[t * E + e];
      in_smem = false;
    }
    // strides below E: partners in this thread's registers
#pragma unroll
    for (int jj = E / 2; jj > 0; jj >>= 1) {
      if (jj <= (k >> 1)) {
#pragma unroll
        for (int e = 0; e < E; ++e)
          if ((e & jj) == 0) cmpx<E>(v[e], v[e | jj], (((t * E + e) & k) == 0));
      }
    }
  }
#pragma unroll
  for (int e = 0; e < E; ++e)
    if (t * E + e < n) order[t * E + e] = (int)(v[e] & 0xffffffu);
}

// ---- host helpers -----------------------------------------------------------
// Stream-ordered scratch memory for the planner (freed on the same stream).
struct DevBuf {
  void* p = nullptr;
  cudaStream_t st = nullptr;
  bool own = true;  // false: a view into another buffer (see Arena)
  explicit DevBuf(cudaStream_t s = nullptr) : st(s) {}
  ~DevBuf() {
    if (p && own) cudaFreeAsync(p, st);
  }
  template <class T>
  T* as() {
    return static_cast<T*>(p);
  }
  cudaError_t alloc(size_t bytes) {
    return cudaMallocAsync(&p, bytes > 0 ? bytes : 16, st);
  }
  void* release() {
    void* q = p;
    p = nullptr;
    return q;
  }
};

inline int grid_for(long long n, int block) { return (int)std::max(1LL, (n + block - 1) / block); }

// Dynamic shared-memory limits of the planner's kernels, raised once per
// kernel and device (a bit per device in one word per kernel).
enum AttrSlot : int { kAttrSortGlobal, kAttrSort2, kAttrSort4, kAttrSort8, kAttrSort16,
                      kAttrGatherFill, kAttrBGatherFill, kAttrSlots };
std::atomic<unsigned long long> g_attr_done[kAttrSlots];

cudaError_t smem_limit_once(int slot, const void* func, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (g_attr_done[slot].load(std::memory_order_acquire) & bit) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) g_attr_done[slot].fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// The planner's per-tile and per-unit int arrays, carved from one allocation
// (each a 128-byte aligned run) instead of one allocation apiece: the host
// calls between the planner's reads are what the GPU waits for.
struct Arena {
  DevBuf buf;
  size_t cap = 0, used = 0;  // in ints
  explicit Arena(cudaStream_t s) : buf(s) {}
  static size_t run(long long n) { return (size_t)((std::max(1LL, n) + 31) / 32 * 32); }
  cudaError_t reserve(size_t ints) {
    cap = ints;
    return buf.alloc(sizeof(int) * ints);
  }
  bool take(DevBuf& d, long long n) {  // d views n ints
    const size_t r = run(n);
    if (used + r > cap) return false;
    d.p = buf.as<int>() + used;
    d.own = false;
    used += r;
    return true;
  }
};

#define FFA_CUDA(x)                                      \
  do {                                                   \
    cudaError_t e_ = (x);                                \
    if (e_ != cudaSuccess) {                             \
      return FFA_ERR_CUDA;                               \
    }                                                    \
  } while (0)

// ---- small device -> host reads ----------------------------------------------
// The planner reads a few counts back to size its lists.  A copy-engine read
// (cudaMemcpyAsync) would queue behind any large transfer the caller has in
// flight on another stream (e.g. the previous call's results going to the
// host) and wait for all of it; instead a one-block kernel writes the words
// into mapped pinned host memory, one small buffer per host thread, allocated
// on first use and kept for the thread's life (unified addressing gives it
// the same address on every device).
__global__ void k_to_host(const unsigned int* __restrict__ src, int words,
                          volatile unsigned int* dst) {
  for (int i = threadIdx.x; i < words; i += blockDim.x) dst[i] = src[i];
}

constexpr int kMailboxWords = 64;

unsigned int* host_mailbox(unsigned int** dev_view) {
  thread_local unsigned int* box = nullptr;
  thread_local unsigned int* dbox = nullptr;
  if (!box) {
    unsigned int* b = nullptr;
    // portable: a host thread may plan on several devices
    if (cudaHostAlloc(&b, kMailboxWords * sizeof(unsigned int),
                      cudaHostAllocMapped | cudaHostAllocPortable) != cudaSuccess)
      return nullptr;
    unsigned int* d = nullptr;
    if (cudaHostGetDevicePointer(&d, b, 0) != cudaSuccess) {
      cudaFreeHost(b);
      return nullptr;
    }
    box = b;
    dbox = d;
  }
  *dev_view = dbox;
  return box;
}

// Copies `bytes` (a multiple of 4, at most 256) from device memory to `dst`
// and waits for the stream; falls back to a copy-engine read when no mapped
// buffer could be had.
ffa_status_t read_to_host(void* dst, const void* src, size_t bytes, cudaStream_t st) {
  unsigned int* dview = nullptr;
  unsigned int* box = bytes % 4 == 0 && bytes <= kMailboxWords * 4 ? host_mailbox(&dview) : nullptr;
  if (!box) {
    FFA_CUDA(cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToHost, st));
    FFA_CUDA(cudaStreamSynchronize(st));
    return FFA_OK;
  }
  k_to_host<<<1, 64, 0, st>>>(static_cast<const unsigned int*>(src), (int)(bytes / 4), dview);
  note_launches(1);
  FFA_CUDA(cudaGetLastError());
  FFA_CUDA(cudaStreamSynchronize(st));
  memcpy(dst, box, bytes);
  return FFA_OK;
}

// Exclusive scan of in[0, n) into out, total into *dtot (device), no read back:
// independent scans are launched back to back and their totals read at once.
// nonzero (optional, zeroed by the caller): += the count of nonzero entries.
ffa_status_t scan_launch(const int* in, int n, int* out, long long* dtot, cudaStream_t st,
                         long long* nonzero = nullptr) {
  if (n > 0) {
    k_scan<<<1, 1024, 0, st>>>(in, n, out, dtot, nonzero);
    note_launches(1);
  } else FFA_CUDA(cudaMemsetAsync(dtot, 0, sizeof(long long), st));
  FFA_CUDA(cudaGetLastError());
  return FFA_OK;
}

ffa_status_t scan(const int* in, int n, int* out, long long* dtot, long long* htot,
                  cudaStream_t st) {
  const ffa_status_t rc = scan_launch(in, n, out, dtot, st);
  if (rc != FFA_OK) return rc;
  return read_to_host(htot, dtot, sizeof(long long), st);
}

// head_word: the item word holding a head, head_div: divisor to its kv head.
ffa_status_t sort_items(const int* items, int words, int cost_word, int head_word, int head_div,
                        int n, int* order, cudaStream_t st) {
  if (n <= 0) return FFA_OK;
  if (n >= (1 << 24)) return FFA_ERR_UNSUPPORTED;
  int n2 = 1;
  while (n2 < n) n2 <<= 1;
  if (n2 >= 2048 && n2 <= kSortSmemKeys) {
    const int sm = (int)(sizeof(unsigned long long) * (size_t)n2);
#define FFA_SORT_BLOCKED(E)                                                                    \
  do {                                                                                         \
    FFA_CUDA(smem_limit_once(kAttrSort##E, (const void*)k_sort_order_blocked<E>, sm));          \
    k_sort_order_blocked<E><<<1, 1024, sm, st>>>(items, words, cost_word, n, order, head_word, \
                                                 head_div);                                    \
  } while (0)
    if (n2 == 2048) FFA_SORT_BLOCKED(2);
    else if (n2 == 4096) FFA_SORT_BLOCKED(4);
    else if (n2 == 8192) FFA_SORT_BLOCKED(8);
    else FFA_SORT_BLOCKED(16);
#undef FFA_SORT_BLOCKED
    note_launches(1);
    FFA_CUDA(cudaGetLastError());
    return FFA_OK;
  }
  DevBuf scratch(st);
  if (n2 > kSortSmemKeys) FFA_CUDA(scratch.alloc(sizeof(unsigned long long) * (size_t)n2));
  const size_t smem = n2 <= kSortSmemKeys ? sizeof(unsigned long long) * (size_t)n2 : 0;
  FFA_CUDA(smem_limit_once(kAttrSortGlobal, (const void*)k_sort_order,
                           (int)(sizeof(unsigned long long) * kSortSmemKeys)));
  k_sort_order<<<1, 1024, smem, st>>>(items, words, cost_word, n, n2,
                                      scratch.as<unsigned long long>(), order, head_word, head_div);
  note_launches(1);
  FFA_CUDA(cudaGetLastError());
  return FFA_OK;  // consumed by later work on `st`; the planner synchronizes before returning
}

void free_plan(ffa_plan_s* p) {
  if (!p) return;
  void* bufs[] = {p->slices, p->fwd_steps, p->fwd_items, p->fwd_order, p->merges,
                  p->bwd_steps, p->bwd_items, p->bwd_order, p->err, p->fwd_masks,
                  p->bwd_masks, p->dq_counts, p->tickets, p->gathers, p->bgathers};
  for (void* b : bufs)
    if (b) cudaFree(b);
  if (!p->dq_alias) {
    if (p->dq_items) cudaFree(p->dq_items);
    if (p->dq_order) cudaFree(p->dq_order);
  }
  delete p;
}

// The plan's lists are stream-ordered allocations on the planning stream (a
// plain cudaMalloc may stop work on other streams from overlapping, e.g. a
// caller's copies of the previous call's results); the planner synchronizes
// that stream before it returns, so they are ready for any stream after.
ffa_status_t build_plan(ffa_plan_s* p, const int32_t* qr, const int32_t* kr, const int32_t* ty,
                        int split_below, cudaStream_t st) {
  const int S = p->S;
  FFA_CUDA(cudaMallocAsync(&p->slices, sizeof(Slice) * (size_t)std::max(S, 1), st));
  FFA_CUDA(cudaMallocAsync(&p->err, 2 * sizeof(int), st));
  FFA_CUDA(cudaMallocAsync(&p->tickets, 4 * sizeof(int), st));
  FFA_CUDA(cudaMemsetAsync(p->err, 0, 2 * sizeof(int), st));
  DevBuf flags_area(st);
  FFA_CUDA(flags_area.alloc(192));
  int* flags = flags_area.as<int>();
  unsigned long long* area = reinterpret_cast<unsigned long long*>(flags + 4);
  long long* dtot = reinterpret_cast<long long*>(flags + 8);
  FFA_CUDA(cudaMemsetAsync(flags, 0, 192, st));
  if (S > 0) {
    k_pack_slices<<<grid_for(S, 256), 256, 0, st>>>(qr, kr, ty, S, p->slices);
    note_launches(1);
    k_check_slices<<<grid_for(S, 256), 256, 0, st>>>(p->slices, S, p->Tq, p->Tk, flags, area);
    note_launches(1);
    FFA_CUDA(cudaGetLastError());
  }
  // per-tile slice lists (q-tiles for the forward and the overlap check,
  // k-tiles for the backward)
  const int n_qt = p->n_qt, n_kt = p->n_kt, g = p->Hq / p->Hkv;
  long long tot = 0;
  ffa_status_t rc = FFA_OK;
  // per-tile / per-unit arrays: 12 over q-tiles (lists, visits, units,
  // costs), 10 over k-tiles, 4 over 64-row slabs
  const long long n_slabs_max = ((long long)p->Tq + kSlabRows / 2 - 1) / (kSlabRows / 2);
  Arena arena(st);
  FFA_CUDA(arena.reserve(12 * Arena::run(n_qt) + 10 * Arena::run(n_kt) +
                         3 * Arena::run(n_slabs_max) + Arena::run(2 * n_slabs_max)));
#define FFA_TAKE(d, n) \
  do {                 \
    if (!arena.take(d, n)) return FFA_ERR_CUDA; \
  } while (0)
  DevBuf qlcnt(st), qloff(st), qlist(st), klcnt(st), kloff(st), klist(st);
  FFA_TAKE(qlcnt, n_qt);
  FFA_TAKE(qloff, n_qt);
  FFA_TAKE(klcnt, n_kt);
  FFA_TAKE(kloff, n_kt);
  if (n_qt > 0) {
    k_tile_slices<true><<<n_qt, kListThreads, 0, st>>>(p->slices, S, nullptr, qlcnt.as<int>(),
                                                       nullptr);
    note_launches(1);
    FFA_CUDA(cudaGetLastError());
  }
  if (n_kt > 0) {
    k_tile_slices<false><<<n_kt, kListThreads, 0, st>>>(p->slices, S, nullptr, klcnt.as<int>(),
                                                        nullptr);
    note_launches(1);
    FFA_CUDA(cudaGetLastError());
  }
  long long lt[2];  // list lengths: q-tile lists, k-tile lists
  if ((rc = scan_launch(qlcnt.as<int>(), n_qt, qloff.as<int>(), dtot, st))) return rc;
  if ((rc = scan_launch(klcnt.as<int>(), n_kt, kloff.as<int>(), dtot + 1, st))) return rc;
  if ((rc = read_to_host(lt, dtot, sizeof lt, st))) return rc;
  tot = lt[0];
  if (tot > 0x7fffffffLL || lt[1] > 0x7fffffffLL) return FFA_ERR_UNSUPPORTED;
  FFA_CUDA(qlist.alloc(sizeof(int) * (size_t)tot));
  if (n_qt > 0) {
    k_tile_slices<true><<<n_qt, kListThreads, 0, st>>>(p->slices, S, qloff.as<int>(), nullptr,
                                                       qlist.as<int>());
    note_launches(1);
    k_check_overlap<<<n_qt, kListThreads, 0, st>>>(p->slices, qlist.as<int>(), qloff.as<int>(),
                                                   qlcnt.as<int>(), flags);
    note_launches(1);
    FFA_CUDA(cudaGetLastError());
  }
  tot = lt[1];
  FFA_CUDA(klist.alloc(sizeof(int) * (size_t)tot));
  if (n_kt > 0) {
    k_tile_slices<false><<<n_kt, kListThreads, 0, st>>>(p->slices, S, kloff.as<int>(), nullptr,
                                                        klist.as<int>());
    note_launches(1);
    FFA_CUDA(cudaGetLastError());
  }
  int hfa[6];  // flags[4], then the area (64-bit) right after them
  if ((rc = read_to_host(hfa, flags, sizeof hfa, st))) return rc;
  if (hfa[0]) return FFA_ERR_RANGE;
  if (hfa[1]) return FFA_ERR_OVERLAP;
  unsigned long long harea = 0;
  memcpy(&harea, hfa + 4, sizeof harea);
  p->area = (int64_t)harea;

  // forward visits
  DevBuf vcnt(st), voff(st), visits(st), fmcnt(st), fmoff(st);
  FFA_TAKE(vcnt, n_qt);
  FFA_TAKE(voff, n_qt);
  FFA_TAKE(fmcnt, n_qt);
  FFA_TAKE(fmoff, n_qt);
  k_visit_warp<true, true><<<grid_for(n_qt, kFillWarps), 32 * kFillWarps, 0, st>>>(
      p->slices, qlist.as<int>(), qloff.as<int>(), qlcnt.as<int>(), n_qt, vcnt.as<int>(),
      fmcnt.as<int>(), nullptr, nullptr, nullptr, nullptr);
  note_launches(1);
  FFA_CUDA(cudaGetLastError());
  // backward visits (transposed lists), counted now so that one read returns
  // both directions' totals
  DevBuf bcnt(st), boff(st), bvis(st), bmcnt(st), bmoff(st);
  FFA_TAKE(bcnt, n_kt);
  FFA_TAKE(boff, n_kt);
  FFA_TAKE(bmcnt, n_kt);
  FFA_TAKE(bmoff, n_kt);
  k_visit_warp<false, true><<<grid_for(n_kt, kFillWarps), 32 * kFillWarps, 0, st>>>(
      p->slices, klist.as<int>(), kloff.as<int>(), klcnt.as<int>(), n_kt, bcnt.as<int>(),
      bmcnt.as<int>(), nullptr, nullptr, nullptr, nullptr);
  note_launches(1);
  FFA_CUDA(cudaGetLastError());
  long long vm[4];  // forward visits, slice-list words; backward visits, slice-list words
  if ((rc = scan_launch(vcnt.as<int>(), n_qt, voff.as<int>(), dtot, st))) return rc;
  if ((rc = scan_launch(fmcnt.as<int>(), n_qt, fmoff.as<int>(), dtot + 1, st))) return rc;
  if ((rc = scan_launch(bcnt.as<int>(), n_kt, boff.as<int>(), dtot + 2, st))) return rc;
  if ((rc = scan_launch(bmcnt.as<int>(), n_kt, bmoff.as<int>(), dtot + 3, st))) return rc;
  if ((rc = read_to_host(vm, dtot, sizeof vm, st))) return rc;
  tot = vm[0];
  if (tot > 0x7fffffffLL) return FFA_ERR_UNSUPPORTED;
  FFA_CUDA(visits.alloc(sizeof(int2) * (size_t)tot));
  const long long mtot = vm[1];
  if (mtot > (1LL << 29)) return FFA_ERR_UNSUPPORTED;
  p->n_fwd_masks = mtot;
  FFA_CUDA(cudaMallocAsync(&p->fwd_masks, sizeof(int) * (size_t)std::max(1LL, mtot), st));
  k_visit_warp<true, false><<<grid_for(n_qt, kFillWarps), 32 * kFillWarps, 0, st>>>(
      p->slices, qlist.as<int>(), qloff.as<int>(), qlcnt.as<int>(), n_qt, nullptr, nullptr,
      voff.as<int>(), fmoff.as<int>(), visits.as<int2>(), p->fwd_masks);
  note_launches(1);
  FFA_CUDA(cudaGetLastError());
  if (vm[2] > 0x7fffffffLL) return FFA_ERR_UNSUPPORTED;
  FFA_CUDA(bvis.alloc(sizeof(int2) * (size_t)vm[2]));
  const long long bmtot = vm[3];
  if (bmtot > (1LL << 29)) return FFA_ERR_UNSUPPORTED;
  p->n_bwd_masks = bmtot;
  FFA_CUDA(cudaMallocAsync(&p->bwd_masks, sizeof(int) * (size_t)std::max(1LL, bmtot), st));
  k_visit_warp<false, false><<<grid_for(n_kt, kFillWarps), 32 * kFillWarps, 0, st>>>(
      p->slices, klist.as<int>(), kloff.as<int>(), klcnt.as<int>(), n_kt, nullptr, nullptr,
      boff.as<int>(), bmoff.as<int>(), bvis.as<int2>(), p->bwd_masks);
  note_launches(1);
  FFA_CUDA(cudaGetLastError());
  // gathered k-tiles (full slices, 8-row aligned query ranges): their step
  // counts replace the visit counts; scanned with the forward's below
  DevBuf bgcnt(st), bgoff(st), bscnt(st), bsoff(st);
  FFA_TAKE(bgcnt, n_kt);
  FFA_TAKE(bgoff, n_kt);
  FFA_TAKE(bscnt, n_kt);
  FFA_TAKE(bsoff, n_kt);
  if (p->Tq <= kGatherMaxTk && n_kt > 0) {
    k_bgather_count<<<n_kt, kGatherThreads, 0, st>>>(p->slices, klist.as<int>(), kloff.as<int>(),
                                                     klcnt.as<int>(), p->Tq, bcnt.as<int>(),
                                                     bgcnt.as<int>(), bscnt.as<int>());
    note_launches(1);
    FFA_CUDA(cudaGetLastError());
  } else {
    FFA_CUDA(cudaMemsetAsync(bgcnt.p, 0, sizeof(int) * n_kt, st));
    FFA_CUDA(cudaMemcpyAsync(bscnt.p, bcnt.p, sizeof(int) * n_kt, cudaMemcpyDeviceToDevice, st));
  }
  // forward units -> steps
  int pair_mode = g >= 2 ? 0 : 1;
  int n_units = pair_mode == 0 ? n_qt : (n_qt + 1) / 2;
  DevBuf scnt(st), soff(st), cost_half(st), steps(st);
  FFA_TAKE(scnt, n_units);
  FFA_TAKE(soff, n_units);
  FFA_TAKE(cost_half, 2LL * n_units);
  const bool unit_warps = n_kt <= kUnitWarpTiles;
  if (unit_warps)
    k_fwd_unit_count_w<<<grid_for(n_units, kUnitWarps), 32 * kUnitWarps, 0, st>>>(
        visits.as<int2>(), voff.as<int>(), vcnt.as<int>(), n_qt, n_units, pair_mode, n_kt,
        scnt.as<int>(), cost_half.as<int>());
  else
    k_fwd_unit_count<<<grid_for(n_units, 128), 128, 0, st>>>(visits.as<int2>(), voff.as<int>(),
                                                             vcnt.as<int>(), n_qt, n_units,
                                                             pair_mode, scnt.as<int>(),
                                                             cost_half.as<int>());
  note_launches(1);
  FFA_CUDA(cudaGetLastError());
  // gathered units (full, 8-key aligned slices): their step counts replace
  // the regular ones before the step offsets are scanned
  DevBuf gcnt(st), goff(st);
  FFA_TAKE(gcnt, n_units);
  FFA_TAKE(goff, n_units);
  FFA_CUDA(cudaMemsetAsync(gcnt.p, 0, sizeof(int) * n_units, st));
  if (p->Tk <= kGatherMaxTk && n_units > 0) {
    k_gather_count<<<n_units, kGatherThreads, 0, st>>>(p->slices, qlist.as<int>(), qloff.as<int>(),
                                                       qlcnt.as<int>(), n_qt, pair_mode, p->Tk,
                                                       scnt.as<int>(), gcnt.as<int>());
    note_launches(1);
    FFA_CUDA(cudaGetLastError());
  }
  // head-stacked units (slabs of 64 rows with heads stacked in pairs, or of
  // 32 rows with heads in fours): counted beside the q-tile units and chosen
  // after the read below when every slab gathers and they take at most 9/10
  // of the chosen units' work (the planner specification gives the counts)
  const bool try_stack = pair_mode == 0 && g >= 4 && g % 2 == 0 && p->Tk <= kGatherMaxTk &&
                         n_qt > 0;
  const bool try_stack4 = try_stack && g % 4 == 0;
  const int n_slabs = (p->Tq + kSlabRows - 1) / kSlabRows;
  const int n_slabs4 = (p->Tq + kSlabRows / 2 - 1) / (kSlabRows / 2);
  DevBuf slab_steps(st), slab_steps4(st), slab_off(st), slab_cost(st);
  if (try_stack) FFA_TAKE(slab_steps, n_slabs);
  if (try_stack4) FFA_TAKE(slab_steps4, n_slabs4);
  // one read: forward steps and gathered records, 64-row slab steps and
  // ineligible slabs, backward steps and gathered records, units and 64-row
  // slabs with steps, 32-row slab steps, ineligible and nonzero slabs
  FFA_CUDA(cudaMemsetAsync(dtot + 4, 0, 12 * sizeof(long long), st));
  if (try_stack) {
    k_slab_count<<<n_slabs, kGatherThreads, 0, st>>>(
        p->slices, qlist.as<int>(), qloff.as<int>(), qlcnt.as<int>(), n_qt, p->Tk, kSlabRows,
        slab_steps.as<int>(), dtot + 6, dtot + 7, dtot + 11);
    note_launches(1);
    FFA_CUDA(cudaGetLastError());
  }
  if (try_stack4) {
    k_slab_count<<<n_slabs4, kGatherThreads, 0, st>>>(
        p->slices, qlist.as<int>(), qloff.as<int>(), qlcnt.as<int>(), n_qt, p->Tk,
        kSlabRows / 2, slab_steps4.as<int>(), dtot + 12, dtot + 13, dtot + 14);
    note_launches(1);
    FFA_CUDA(cudaGetLastError());
  }
  long long sg[12];
  if ((rc = scan_launch(scnt.as<int>(), n_units, soff.as<int>(), dtot + 4, st, dtot + 10)))
    return rc;
  if ((rc = scan_launch(gcnt.as<int>(), n_units, goff.as<int>(), dtot + 5, st))) return rc;
  if ((rc = scan_launch(bscnt.as<int>(), n_kt, bsoff.as<int>(), dtot + 8, st))) return rc;
  if ((rc = scan_launch(bgcnt.as<int>(), n_kt, bgoff.as<int>(), dtot + 9, st))) return rc;
  if ((rc = read_to_host(sg, dtot + 4, sizeof sg, st))) return rc;
  const long long bs[2] = {sg[4], sg[5]};  // backward steps, gathered records
  long long nz_units = sg[6];             // forward units with steps
  int stack_rows = 0;
  long long half_steps = (long long)g * sg[0];  // work of the units chosen so far
  if (try_stack && sg[3] == 0 && sg[2] > 0 &&
      10LL * ((g + 3) / 4) * sg[2] <= 9LL * (g / 2) * sg[0]) {
    stack_rows = kSlabRows;
    half_steps = (long long)(g / 2) * sg[2];
  }
  if (try_stack4 && sg[9] == 0 && sg[8] > 0 && 10LL * (g / 4) * sg[8] <= 9LL * half_steps)
    stack_rows = kSlabRows / 2;
  const bool stacked = stack_rows > 0;
  int* u_scnt = scnt.as<int>();
  int* u_soff = soff.as<int>();
  int* u_gcnt = gcnt.as<int>();
  int* u_goff = goff.as<int>();
  int* u_cost = cost_half.as<int>();
  if (stacked) {  // every step gathered: record r is step r, offsets shared
    const bool four = stack_rows != kSlabRows;
    pair_mode = 2;
    n_units = four ? n_slabs4 : n_slabs;
    FFA_TAKE(slab_off, n_units);
    FFA_TAKE(slab_cost, 2LL * n_units);
    FFA_CUDA(cudaMemsetAsync(slab_cost.p, 0, sizeof(int) * 2 * n_units, st));
    int* ss = four ? slab_steps4.as<int>() : slab_steps.as<int>();
    if ((rc = scan_launch(ss, n_units, slab_off.as<int>(), dtot, st))) return rc;
    u_scnt = u_gcnt = ss;
    u_soff = u_goff = slab_off.as<int>();
    u_cost = slab_cost.as<int>();
    sg[0] = sg[1] = four ? sg[8] : sg[2];
    nz_units = four ? sg[10] : sg[7];
    p->stacked = stack_rows;
    // one half of an item holds all four heads: the two halves take the
    // slab's steps in turn instead (merged at the end of the item)
    p->alternate = four && g == 4;
  }
  tot = sg[0];
  if (tot > 0x7fffffffLL || sg[1] > (1LL << 24)) return FFA_ERR_UNSUPPORTED;
  p->n_fwd_steps = tot;
  p->n_gathers = sg[1];
  FFA_CUDA(steps.alloc(sizeof(int4) * (size_t)tot));
  FFA_CUDA(cudaMallocAsync(&p->gathers,
                           sizeof(int) * kGatherWords * (size_t)std::max(1LL, sg[1]), st));
  if (!stacked) {
    if (unit_warps)
      k_fwd_unit_fill_w<<<grid_for(n_units, kUnitWarps), 32 * kUnitWarps, 0, st>>>(
          visits.as<int2>(), voff.as<int>(), vcnt.as<int>(), n_qt, n_units, pair_mode, n_kt,
          soff.as<int>(), gcnt.as<int>(), steps.as<int4>());
    else
      k_fwd_unit_fill<<<grid_for(n_units, 128), 128, 0, st>>>(visits.as<int2>(), voff.as<int>(),
                                                              vcnt.as<int>(), n_qt, n_units,
                                                              pair_mode, soff.as<int>(),
                                                              gcnt.as<int>(), steps.as<int4>());
    note_launches(1);
    FFA_CUDA(cudaGetLastError());
  }
  if (sg[1] > 0) {
    FFA_CUDA(smem_limit_once(kAttrGatherFill, (const void*)k_gather_fill, (int)kGatherFillSmem));
    k_gather_fill<<<n_units, kGatherThreads, kGatherFillSmem, st>>>(
        p->slices, qlist.as<int>(), qloff.as<int>(), qlcnt.as<int>(), n_qt, pair_mode,
        stacked ? stack_rows : kSlabRows, p->alternate, p->Tk, u_gcnt, u_goff, u_soff,
        steps.as<int4>(), p->gathers, u_cost);
    note_launches(1);
    FFA_CUDA(cudaGetLastError());
  }
  // forward items
  // head pairs per kv head (groups of 2m heads for stacked units, m heads a half)
  const int m_heads = stacked ? 128 / stack_rows : 1;
  const int pairs = pair_mode == 2 ? (g + 2 * m_heads - 1) / (2 * m_heads) : (g + 1) / 2;
  const long long n_items = pair_mode != 1 ? (long long)n_units * p->Hkv * pairs
                                           : (long long)n_units * p->Hq;
  if (n_items > 0x7fffffffLL / kFiWords) return FFA_ERR_UNSUPPORTED;
  DevBuf items(st);
  FFA_CUDA(items.alloc(sizeof(int) * kFiWords * (size_t)n_items));
  k_fwd_items<<<grid_for(n_items, 128), 128, 0, st>>>((int)n_items, pair_mode, m_heads,
                                                      p->alternate, g, p->Hkv, p->Hq,
                                                      pairs, n_qt, u_soff, u_scnt, u_cost,
                                                      items.as<int>());
  note_launches(1);
  FFA_CUDA(cudaGetLastError());
  // items with steps: every item of a unit with steps
  const long long hlive = nz_units * (n_units > 0 ? n_items / n_units : 0);
  const int threshold = split_below == 0 ? 2 * p->num_sms : split_below;
  long long final_items = n_items;
  if (split_below >= 0 && hlive > 0 && hlive < threshold && !stacked) {
    const int nsplit = (int)std::min<long long>(16, (threshold + hlive - 1) / hlive);
    DevBuf chunks(st), coff(st), slots(st), sloff(st), groups(st), goff(st), nitems(st),
        merges(st);
    const size_t nb = sizeof(int) * (size_t)n_items;
    FFA_CUDA(chunks.alloc(nb));
    FFA_CUDA(coff.alloc(nb));
    FFA_CUDA(slots.alloc(nb));
    FFA_CUDA(sloff.alloc(nb));
    FFA_CUDA(groups.alloc(nb));
    FFA_CUDA(goff.alloc(nb));
    k_split_count<<<grid_for(n_items, 128), 128, 0, st>>>(items.as<int>(), (int)n_items, nsplit,
                                                          chunks.as<int>(), slots.as<int>(),
                                                          groups.as<int>());
    note_launches(1);
    FFA_CUDA(cudaGetLastError());
    long long n_chunks = 0, n_slots = 0, n_groups = 0;
    if ((rc = scan(chunks.as<int>(), (int)n_items, coff.as<int>(), dtot, &n_chunks, st))) return rc;
    if ((rc = scan(slots.as<int>(), (int)n_items, sloff.as<int>(), dtot, &n_slots, st))) return rc;
    if ((rc = scan(groups.as<int>(), (int)n_items, goff.as<int>(), dtot, &n_groups, st))) return rc;
    FFA_CUDA(nitems.alloc(sizeof(int) * kFiWords * (size_t)n_chunks));
    FFA_CUDA(merges.alloc(sizeof(int) * kMgWords * (size_t)std::max(1LL, n_groups)));
    k_split_fill<<<grid_for(n_items, 128), 128, 0, st>>>(
        items.as<int>(), (int)n_items, chunks.as<int>(), coff.as<int>(), sloff.as<int>(),
        goff.as<int>(), nitems.as<int>(), merges.as<int>());
    note_launches(1);
    FFA_CUDA(cudaGetLastError());
    FFA_CUDA(cudaStreamSynchronize(st));
    std::swap(items.p, nitems.p);
    // the unsplit list stays for the dQ pass of the backward
    p->dq_items = static_cast<int*>(nitems.release());
    p->n_dq_items = n_items;
    p->dq_alias = false;
    final_items = n_chunks;
    p->n_merges = n_groups;
    p->n_slots = (int)n_slots;
    p->merges = static_cast<int*>(merges.release());
  }
  p->n_fwd_items = final_items;
  FFA_CUDA(cudaMallocAsync(&p->fwd_order, sizeof(int) * (size_t)std::max(1LL, final_items), st));
  rc = sort_items(items.as<int>(), kFiWords, kFiCost, kFiH0, p->Hq / p->Hkv, (int)final_items,
                  p->fwd_order, st);
  if (rc != FFA_OK) return rc;
  p->fwd_items = items.as<int>();
  items.release();
  p->fwd_steps = steps.as<int4>();
  steps.release();
  if (p->dq_alias) {
    p->dq_items = p->fwd_items;
    p->dq_order = p->fwd_order;
    p->n_dq_items = p->n_fwd_items;
  } else {
    FFA_CUDA(cudaMallocAsync(&p->dq_order, sizeof(int) * (size_t)std::max<int64_t>(1, p->n_dq_items), st));
    rc = sort_items(p->dq_items, kFiWords, kFiCost, kFiH0, p->Hq / p->Hkv, (int)p->n_dq_items,
                    p->dq_order, st);
    if (rc != FFA_OK) return rc;
  }
  p->grid_dq = (int)std::max<int64_t>(1, std::min<int64_t>(p->num_sms, p->n_dq_items));
  FFA_CUDA(cudaMallocAsync(&p->dq_counts, sizeof(int) * 2 * (size_t)std::max<int64_t>(1, p->n_dq_items), st));
  if (p->n_dq_items > 0) {
    k_dq_counts<<<grid_for(p->n_dq_items, 128), 128, 0, st>>>(p->dq_items, (int)p->n_dq_items,
                                                             p->fwd_steps, p->alternate,
                                                             p->dq_counts);
    note_launches(1);
    FFA_CUDA(cudaGetLastError());
  }

  // backward (visits and step counts were made with the forward's)
  if (bs[0] > 0x7fffffffLL || bs[1] > (1LL << 24)) return FFA_ERR_UNSUPPORTED;
  p->n_bwd_steps = bs[0];
  p->n_bgathers = bs[1];
  FFA_CUDA(cudaMallocAsync(&p->bwd_steps, sizeof(int4) * (size_t)std::max(1LL, bs[0]), st));
  FFA_CUDA(cudaMallocAsync(&p->bgathers,
                           sizeof(int) * kBGatherWords * (size_t)std::max(1LL, bs[1]), st));
  const long long nb_items = (long long)n_kt * p->Hkv;
  p->n_bwd_items = nb_items;
  FFA_CUDA(cudaMallocAsync(&p->bwd_items, sizeof(int) * kBiWords * (size_t)std::max(1LL, nb_items), st));
  FFA_CUDA(cudaMallocAsync(&p->bwd_order, sizeof(int) * (size_t)std::max(1LL, nb_items), st));
  k_bwd_items<<<grid_for(n_kt, 4), 128, 0, st>>>(n_kt, p->Hkv, g, bvis.as<int2>(),
                                                       boff.as<int>(), bcnt.as<int>(),
                                                       bsoff.as<int>(), bgcnt.as<int>(),
                                                       p->bwd_steps, p->bwd_items);
  note_launches(1);
  FFA_CUDA(cudaGetLastError());
  if (bs[1] > 0) {
    FFA_CUDA(smem_limit_once(kAttrBGatherFill, (const void*)k_bgather_fill,
                             (int)kBGatherFillSmem));
    k_bgather_fill<<<n_kt, kGatherThreads, kBGatherFillSmem, st>>>(
        p->slices, klist.as<int>(), kloff.as<int>(), klcnt.as<int>(), p->Tq, bgcnt.as<int>(),
        bgoff.as<int>(), bsoff.as<int>(), p->bwd_steps, p->bgathers);
    note_launches(1);
    FFA_CUDA(cudaGetLastError());
  }
  rc = sort_items(p->bwd_items, kBiWords, kBiCost, kBiHkv, 1, (int)nb_items, p->bwd_order, st);
  if (rc != FFA_OK) return rc;
  p->grid_fwd = (int)std::max(1LL, std::min<long long>(p->num_sms, final_items));
  p->grid_bwd = (int)std::max(1LL, std::min<long long>(p->num_sms, nb_items));
  FFA_CUDA(cudaStreamSynchronize(st));
  return FFA_OK;
}
#undef FFA_TAKE

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Sink arguments: none (num_sink == 0), or fp32 logits in a known layout.
bool sink_args_ok(const float* sink, int32_t n, int32_t layout) {
  if (n < 0 || n > FFA_MAX_SINK) return false;
  if (layout != FFA_SINK_SH && layout != FFA_SINK_SSH) return false;
  if (n > 0 && (!sink || (reinterpret_cast<uintptr_t>(sink) & 3u))) return false;
  return true;
}

std::atomic<uint64_t> g_launches{0};

}  // namespace

// True when the calling thread's current device is the one the plan was
// built on (its lists, tickets and error word live there).
bool on_plan_device(const ffa_plan_s* p) {
  int dev = -1;
  return cudaGetDevice(&dev) == cudaSuccess && dev == p->device;
}

void note_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }
uint64_t g_launches_total() { return g_launches.load(std::memory_order_relaxed); }

// 2-D tensor map over a row-major [rows][cols] bf16 matrix: boxes of
// box_rows rows x 64 columns (128 bytes), 128-byte swizzle, zero fill outside.
// An 8-row box fills exactly one 1024-byte swizzle atom, so boxes written at
// 1024-byte aligned offsets of a tile lay out rows as one 128-row box would.
bool encode_tile_map(void* map128, const void* base, int rows, int cols_elems, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols_elems, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols_elems * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(static_cast<CUtensorMap*>(map128), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                  const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace ffa

using namespace ffa;

extern "C" {

ffa_status_t ffa_plan_create(ffa_plan_t* plan, const int32_t* q_ranges, const int32_t* k_ranges,
                             const int32_t* mask_types, int32_t num_slices, int32_t total_q,
                             int32_t total_k, int32_t num_heads_q, int32_t num_heads_kv,
                             int32_t head_dim, int32_t num_sms, int32_t split_below,
                             ffa_stream_t stream) {
  if (!plan) return FFA_ERR_INVALID_ARG;
  *plan = nullptr;
  if (num_slices < 0 || total_q <= 0 || total_k <= 0 || num_heads_q <= 0 || num_heads_kv <= 0 ||
      split_below < -1 || num_sms < 0)
    return FFA_ERR_INVALID_ARG;
  if (num_slices > 0 && (!q_ranges || !k_ranges || !mask_types)) return FFA_ERR_INVALID_ARG;
  if (num_heads_q % num_heads_kv != 0 || (head_dim != 64 && head_dim != 128))
    return FFA_ERR_UNSUPPORTED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FFA_ERR_CUDA;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return FFA_ERR_CUDA;
  if (prop.major != 10 || prop.minor != 3) return FFA_ERR_UNSUPPORTED;
  ffa_plan_s* p = new ffa_plan_s();
  p->device = dev;
  p->Tq = total_q;
  p->Tk = total_k;
  p->Hq = num_heads_q;
  p->Hkv = num_heads_kv;
  p->D = head_dim;
  p->S = num_slices;
  p->num_sms = num_sms > 0 ? num_sms : prop.multiProcessorCount;
  p->n_qt = (total_q + kTile - 1) / kTile;
  p->n_kt = (total_k + kTile - 1) / kTile;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  ffa_status_t rc = build_plan(p, q_ranges, k_ranges, mask_types, split_below, st);
  if (rc != FFA_OK) {
    cudaStreamSynchronize(st);
    free_plan(p);
    return rc;
  }
  *plan = p;
  return FFA_OK;
}

ffa_status_t ffa_plan_destroy(ffa_plan_t plan) {
  if (!plan) return FFA_ERR_INVALID_ARG;
  // Work using the plan runs on the plan's device: wait for that device, free
  // there, and give the caller back its own current device.
  int cur = -1;
  const bool have_cur = cudaGetDevice(&cur) == cudaSuccess;
  const bool switched = have_cur && cur != plan->device && cudaSetDevice(plan->device) == cudaSuccess;
  cudaDeviceSynchronize();
  free_plan(plan);
  if (switched) cudaSetDevice(cur);
  return FFA_OK;
}

ffa_status_t ffa_plan_info(ffa_plan_t p, ffa_plan_info_t* info) {
  if (!p || !info) return FFA_ERR_INVALID_ARG;
  info->fwd_steps = p->n_fwd_steps;
  info->fwd_items = p->n_fwd_items;
  info->bwd_steps = p->n_bwd_steps;
  info->bwd_items = p->n_bwd_items;
  info->merges = p->n_merges;
  info->grid_fwd = p->grid_fwd;
  info->grid_bwd = p->grid_bwd;
  info->area = p->area;
  info->fwd_masks = p->n_fwd_masks;
  info->bwd_masks = p->n_bwd_masks;
  info->gathers = p->n_gathers;
  info->bgathers = p->n_bgathers;
  info->stacked = p->stacked;
  return FFA_OK;
}

ffa_status_t ffa_plan_export(ffa_plan_t p, int32_t which, int32_t* dst, int64_t capacity,
                             int64_t* written) {
  if (!p || !written || (capacity > 0 && !dst)) return FFA_ERR_INVALID_ARG;
  if (!on_plan_device(p)) return FFA_ERR_INVALID_ARG;
  const void* src = nullptr;
  int64_t words = 0;
  switch (which) {
    case 0: src = p->fwd_steps; words = 4 * p->n_fwd_steps; break;
    case 1: src = p->fwd_items; words = kFiWords * p->n_fwd_items; break;
    case 2: src = p->fwd_order; words = p->n_fwd_items; break;
    case 3: src = p->bwd_steps; words = 4 * p->n_bwd_steps; break;
    case 4: src = p->bwd_items; words = kBiWords * p->n_bwd_items; break;
    case 5: src = p->bwd_order; words = p->n_bwd_items; break;
    case 6: src = p->merges; words = kMgWords * p->n_merges; break;
    case 7: src = p->fwd_masks; words = p->n_fwd_masks; break;
    case 8: src = p->bwd_masks; words = p->n_bwd_masks; break;
    case 9: src = p->gathers; words = kGatherWords * p->n_gathers; break;
    case 10: src = p->bgathers; words = kBGatherWords * p->n_bgathers; break;
    default: return FFA_ERR_INVALID_ARG;
  }
  *written = words;
  if (words > capacity) return FFA_ERR_INVALID_ARG;
  if (words > 0 && cudaMemcpy(dst, src, sizeof(int32_t) * words, cudaMemcpyDeviceToHost) !=
                       cudaSuccess)
    return FFA_ERR_CUDA;
  return FFA_OK;
}

size_t ffa_fwd_workspace_size(ffa_plan_t p) { return p ? fwd_workspace_bytes(p) : 0; }
size_t ffa_bwd_workspace_size(ffa_plan_t p) { return p ? bwd_workspace_bytes(p) : 0; }

ffa_status_t ffa_fwd_ex(ffa_plan_t p, const void* q, const void* k, const void* v,
                        const float* sink, int32_t num_sink, int32_t sink_layout,
                        float softmax_scale, float softcap, void* out, float* lse,
                        void* workspace, size_t workspace_bytes, ffa_stream_t stream) {
  if (!p || !q || !k || !v || !out || !lse) return FFA_ERR_INVALID_ARG;
  if (!on_plan_device(p)) return FFA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse))
    return FFA_ERR_INVALID_ARG;
  if (!sink_args_ok(sink, num_sink, sink_layout)) return FFA_ERR_INVALID_ARG;
  if (!(softcap >= 0.f && softcap <= 3.0e38f)) return FFA_ERR_INVALID_ARG;  // also rejects NaN
  const size_t need = fwd_workspace_bytes(p);
  if (workspace_bytes < need || (need > 0 && (!workspace || !aligned16(workspace))))
    return FFA_ERR_WORKSPACE;
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf((float)p->D);
  SinkArgs sk;
  sk.sink = sink;
  sk.n = num_sink;
  sk.layout = sink_layout;
  return launch_fwd(p, q, k, v, scale, out, lse, workspace, workspace_bytes,
                    reinterpret_cast<cudaStream_t>(stream), sk, softcap);
}

ffa_status_t ffa_fwd(ffa_plan_t p, const void* q, const void* k, const void* v,
                     float softmax_scale, void* out, float* lse, void* workspace,
                     size_t workspace_bytes, ffa_stream_t stream) {
  return ffa_fwd_ex(p, q, k, v, nullptr, 0, FFA_SINK_SH, softmax_scale, 0.f, out, lse, workspace,
                    workspace_bytes, stream);
}

ffa_status_t ffa_bwd_ex(ffa_plan_t p, const void* q, const void* k, const void* v, const void* out,
                        const void* dout, const float* lse, const float* sink, int32_t num_sink,
                        int32_t sink_layout, float softmax_scale, float softcap, void* dq, void* dk,
                        void* dv, float* dsink, void* workspace, size_t workspace_bytes,
                        ffa_stream_t stream) {
  if (!p || !q || !k || !v || !out || !dout || !lse || !dq || !dk || !dv)
    return FFA_ERR_INVALID_ARG;
  if (!on_plan_device(p)) return FFA_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, out, dout, lse, dq, dk, dv};
  for (const void* x : ptrs)
    if (!aligned16(x)) return FFA_ERR_INVALID_ARG;
  if (!sink_args_ok(sink, num_sink, sink_layout)) return FFA_ERR_INVALID_ARG;
  if (dsink && (reinterpret_cast<uintptr_t>(dsink) & 3u)) return FFA_ERR_INVALID_ARG;
  if (!(softcap >= 0.f && softcap <= 3.0e38f)) return FFA_ERR_INVALID_ARG;  // also rejects NaN
  const size_t need = bwd_workspace_bytes(p);
  if (workspace_bytes < need || (need > 0 && (!workspace || !aligned16(workspace))))
    return FFA_ERR_WORKSPACE;
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf((float)p->D);
  SinkArgs sk;
  sk.sink = sink;
  sk.n = num_sink;
  sk.layout = sink_layout;
  return launch_bwd(p, q, k, v, out, dout, lse, scale, dq, dk, dv, workspace, workspace_bytes,
                    reinterpret_cast<cudaStream_t>(stream), sk, dsink, softcap);
}

ffa_status_t ffa_bwd(ffa_plan_t p, const void* q, const void* k, const void* v, const void* out,
                     const void* dout, const float* lse, float softmax_scale, void* dq, void* dk,
                     void* dv, void* workspace, size_t workspace_bytes, ffa_stream_t stream) {
  return ffa_bwd_ex(p, q, k, v, out, dout, lse, nullptr, 0, FFA_SINK_SH, softmax_scale, 0.f, dq,
                    dk, dv, nullptr, workspace, workspace_bytes, stream);
}

ffa_status_t ffa_get_last_device_error(ffa_plan_t p, int32_t* code, int32_t* where,
                                       ffa_stream_t stream) {
  if (!p || !code || !where) return FFA_ERR_INVALID_ARG;
  if (!on_plan_device(p)) return FFA_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int h[2] = {0, 0};
  if (cudaMemcpyAsync(h, p->err, sizeof h, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaMemsetAsync(p->err, 0, sizeof h, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return FFA_ERR_CUDA;
  *code = h[0];
  *where = h[1];
  return FFA_OK;
}

ffa_status_t ffa_plan_set_events(ffa_plan_t p, void* const* events, int32_t n) {
  if (!p || (n != 0 && n != 6) || (n == 6 && !events)) return FFA_ERR_INVALID_ARG;
  p->use_events = n == 6;
  for (int i = 0; i < 6; ++i) p->events[i] = n == 6 ? static_cast<cudaEvent_t>(events[i]) : nullptr;
  return FFA_OK;
}

ffa_status_t ffa_plan_set_wait_limit(ffa_plan_t p, uint64_t ns) {
  if (!p || ns == 0) return FFA_ERR_INVALID_ARG;
  p->wait_ns = ns;
  return FFA_OK;
}

uint64_t ffa_kernel_launch_count(void) { return ffa::g_launches_total(); }

const char* ffa_status_string(ffa_status_t s) {
  switch (s) {
    case FFA_OK: return "ok";
    case FFA_ERR_INVALID_ARG: return "invalid argument";
    case FFA_ERR_RANGE: return "slice range out of bounds or bad mask type";
    case FFA_ERR_OVERLAP: return "slice rectangles overlap";
    case FFA_ERR_UNSUPPORTED: return "unsupported configuration";
    case FFA_ERR_WORKSPACE: return "workspace too small";
    case FFA_ERR_TIMEOUT: return "device wait timed out";
    case FFA_ERR_CUDA: return "CUDA runtime error";
  }
  return "unknown status";
}

}  // extern "C"
