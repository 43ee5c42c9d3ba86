// Internal layout shared by the planner, forward and backward translation
// units of libffa.so.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ffa.h"
#include "ffa_segments.cuh"

namespace ffa {

constexpr int kTile = 128;  // q rows and k columns per tile

// A slice as stored by the plan: [qs, qe) x [ks, ke), mask type t.
using Slice = SliceDesc;

// Visit info of one (q-tile, k-tile) pair (-1 in a step: the half skips it):
//   (s << 2) | partial   one slice s sees the tile (FULL when bit 0 is clear);
//   (m << 2) | 3         several slices see parts of it: masks[m] = n and
//                        masks[m+1 .. m+n] are their indices, ascending.
// Slices are disjoint, so a FULL tile always has exactly one slice.
__host__ __device__ constexpr int visit_info(int slice, bool partial) {
  return (slice << 2) | (partial ? 1 : 0);
}
__host__ __device__ constexpr int visit_list_info(int m) { return (m << 2) | 3; }

// Gathered forward steps (step.w = r + 1 > 0; x unused): for units whose
// slices are all FULL with 8-key aligned key ranges, the 8-key blocks any of
// their rows sees are packed 16 to a K/V tile.  Record r (kGatherWords
// int32): kGatherSlots block start keys (-kGatherKeys for an unused slot,
// loaded as zero-filled rows), then per half kGatherSlots x 4 words of row
// bits (bit i of word w: row 32w + i of the half's q-tile sees the slot).
constexpr int kGatherKeys = 8;
constexpr int kGatherSlots = 16;
constexpr int kGatherWords = kGatherSlots + 2 * kGatherSlots * 4;
// Gathered backward steps (step.w = r + 1 > 0 in the k-tile's list): the
// transpose, for k-tiles whose slices are all FULL with 8-row aligned query
// ranges.  Record r (kBGatherWords int32): kGatherSlots query-block start
// rows (-kGatherKeys: unused), then kGatherSlots x 4 words of key bits (bit i
// of word w: key 32w + i of the k-tile is seen by the slot's rows).
constexpr int kBGatherWords = kGatherSlots + kGatherSlots * 4;
constexpr int kGatherMaxBlocks = 2048;  // 8-key blocks per gathered unit
constexpr int kGatherMaxTk = 1 << 19;   // key count up to which units may gather
// Head-stacked forward units (plan.stacked = R, 64 or 32): a unit is a slab
// of R query rows, and a half of an item is that slab for 128 / R
// consecutive query heads h, h + 1, ... stacked in one 128-row tile (tile row
// r: query row R * slab + r % R of head h + r / R).  Every step of such a plan
// is gathered, with the same row bits for r, r + R, ...
constexpr int kSlabRows = 64;

#ifdef __CUDACC__
// Adds [lo, hi) (tile-local, any range) to a 128-bit mask of tile columns.
__device__ __forceinline__ void add_window(int lo, int hi, uint32_t (&b)[4]) {
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const int a = max(lo - 32 * w, 0), e = min(hi - 32 * w, 32);
    if (e > a) b[w] |= (e == 32 ? 0xffffffffu : ((1u << e) - 1u)) & ~((1u << a) - 1u);
  }
}

// Keys of k-tile kt that query row `row` sees under slice sl, tile-local.
__device__ __forceinline__ void row_window(const Slice& sl, int row, int kt, int& lo, int& hi) {
  lo = hi = 0;
  if (row >= sl.qs && row < sl.qe) {
    lo = sl.ks + ((sl.t & 2) ? row - sl.qs : 0) - kt * kTile;
    hi = sl.ke - ((sl.t & 1) ? sl.qe - 1 - row : 0) - kt * kTile;
  }
}

// Query rows of q-tile qt that key `key` is seen by under slice sl, tile-local.
__device__ __forceinline__ void key_window(const Slice& sl, int key, int qt, int& lo, int& hi) {
  lo = hi = 0;
  if (key < sl.ks || key >= sl.ke) return;
  int a = (sl.t & 1) ? key + sl.qe - sl.ke : sl.qs;
  a = a > sl.qs ? a : sl.qs;
  int b = (sl.t & 2) ? key - sl.ks + sl.qs + 1 : sl.qe;
  b = b < sl.qe ? b : sl.qe;
  lo = a - qt * kTile;
  hi = b - qt * kTile;
}

// Visible columns of one PARTIAL step for one thread's row (kRow: window of
// query row `pos` over the keys of tile t) or key (window of key `pos` over
// the queries of tile t): the union over the step's slice or slice list.
template <bool kRow>
__device__ __forceinline__ void step_mask(int info, const Slice* __restrict__ slices,
                                          const int* __restrict__ masks, int pos, int t,
                                          uint32_t (&b)[4]) {
  b[0] = b[1] = b[2] = b[3] = 0u;
  int lo, hi;
  if ((info & 3) != 3) {
    const Slice sl = slices[info >> 2];
    if (kRow) row_window(sl, pos, t, lo, hi);
    else key_window(sl, pos, t, lo, hi);
    add_window(lo, hi, b);
    return;
  }
  const int* ml = masks + (info >> 2);
  const int n = ml[0];
  for (int i = 0; i < n; ++i) {
    const Slice sl = slices[ml[1 + i]];
    if (kRow) row_window(sl, pos, t, lo, hi);
    else key_window(sl, pos, t, lo, hi);
    add_window(lo, hi, b);
  }
}

// Visible columns of a gathered step for query row `row_in` of half h: slot s
// holds keys [start_s, start_s + 8) in columns [8s, 8s + 8); the columns of a
// slot are set when the row's bit is set, keys at or past Tk never.
// All 32 words are loaded up front and independently (four 16-byte loads
// for the starts), so the record costs one memory round trip.
__device__ __forceinline__ void gather_mask(const int* __restrict__ rec, int h, int row_in,
                                            int Tk, uint32_t (&b)[4]) {
  int y[kGatherSlots];
  uint32_t bits[kGatherSlots];
  const int4* r4 = reinterpret_cast<const int4*>(rec);
#pragma unroll
  for (int q = 0; q < kGatherSlots / 4; ++q) {
    const int4 v = r4[q];
    y[4 * q] = v.x;
    y[4 * q + 1] = v.y;
    y[4 * q + 2] = v.z;
    y[4 * q + 3] = v.w;
  }
  const int* rows = rec + kGatherSlots + h * kGatherSlots * 4 + (row_in >> 5);
#pragma unroll
  for (int s = 0; s < kGatherSlots; ++s) bits[s] = (uint32_t)rows[4 * s];
  b[0] = b[1] = b[2] = b[3] = 0u;
#pragma unroll
  for (int s = 0; s < kGatherSlots; ++s) {
    const int valid = max(0, min(kGatherKeys, Tk - y[s]));  // 0 for unused slots too
    const uint32_t on = (y[s] >= 0) && ((bits[s] >> (row_in & 31)) & 1u) ? 1u : 0u;
    b[s >> 2] |= (((1u << valid) - 1u) & (0u - on)) << (kGatherKeys * (s & 3));
  }
}

// Visible columns of a gathered backward step for key `key_in` of the
// k-tile: slot s holds query rows [start_s, start_s + 8) in columns
// [8s, 8s + 8); set when the key's bit is set, rows at or past Tq never.
__device__ __forceinline__ void gather_key_mask(const int* __restrict__ rec, int key_in, int Tq,
                                                uint32_t (&b)[4]) {
  int y[kGatherSlots];
  uint32_t bits[kGatherSlots];
  const int4* r4 = reinterpret_cast<const int4*>(rec);
#pragma unroll
  for (int q = 0; q < kGatherSlots / 4; ++q) {
    const int4 v = r4[q];
    y[4 * q] = v.x;
    y[4 * q + 1] = v.y;
    y[4 * q + 2] = v.z;
    y[4 * q + 3] = v.w;
  }
  const int* keys = rec + kGatherSlots + (key_in >> 5);
#pragma unroll
  for (int s = 0; s < kGatherSlots; ++s) bits[s] = (uint32_t)keys[4 * s];
  b[0] = b[1] = b[2] = b[3] = 0u;
#pragma unroll
  for (int s = 0; s < kGatherSlots; ++s) {
    const int valid = max(0, min(kGatherKeys, Tq - y[s]));
    const uint32_t on = (y[s] >= 0) && ((bits[s] >> (key_in & 31)) & 1u) ? 1u : 0u;
    b[s >> 2] |= (((1u << valid) - 1u) & (0u - on)) << (kGatherKeys * (s & 3));
  }
}

__device__ __forceinline__ bool mask_bit(const uint32_t (&b)[4], int c) {
  return (b[c >> 5] >> (c & 31)) & 1u;
}
#endif

// Forward step (int4): x = k-tile, y = info for half 0, z = info for half 1.
// Forward item (8 x int32):
enum FwdItem : int {
  kFiQt0 = 0,     // q-tile of half 0
  kFiQt1 = 1,     // q-tile of half 1 (-1: half 1 idle)
  kFiH0 = 2,      // query head of half 0
  kFiH1 = 3,      // query head of half 1 (-1: half 1 idle)
  kFiStepBeg = 4, // first step (index into the step array)
  kFiStepEnd = 5, // one past the last step
  kFiSlot = 6,    // -1: write out/lse; else partial-result slot (split items)
  kFiCost = 7,
  kFiWords = 8
};
// Backward step (int4): x = q-tile, y = info.
// Backward item (8 x int32):
enum BwdItem : int {
  kBiKt = 0, kBiHkv = 1, kBiStepBeg = 2, kBiStepEnd = 3, kBiCost = 4, kBiWords = 8
};
// Merge group (8 x int32): halves of one split forward item.
enum MergeGroup : int {
  kMgQt0 = 0, kMgQt1 = 1, kMgH0 = 2, kMgH1 = 3, kMgSlotBeg = 4, kMgSlots = 5, kMgWords = 8
};

}  // namespace ffa

struct ffa_plan_s {
  int device = 0;
  int Tq = 0, Tk = 0, Hq = 0, Hkv = 0, D = 0, S = 0;
  int num_sms = 0;
  int n_qt = 0, n_kt = 0;
  ffa::Slice* slices = nullptr;  // device [S]
  int4* fwd_steps = nullptr;
  int64_t n_fwd_steps = 0;
  int* fwd_items = nullptr;
  int64_t n_fwd_items = 0;
  int* fwd_order = nullptr;
  int* merges = nullptr;
  int64_t n_merges = 0;
  int n_slots = 0;  // partial-result slots (split forward items)
  int stacked = 0;  // slab rows of head-stacked forward units (64 or 32), 0: q-tile units
  int alternate = 0;  // items' halves are the same rows, taking the steps in turn (merged)
  int* fwd_masks = nullptr;  // slice lists of multi-slice forward visits
  int64_t n_fwd_masks = 0;
  int* gathers = nullptr;  // gathered step records [n_gathers][kGatherWords]
  int64_t n_gathers = 0;
  int* bgathers = nullptr;  // gathered backward records [n_bgathers][kBGatherWords]
  int64_t n_bgathers = 0;
  int4* bwd_steps = nullptr;
  int64_t n_bwd_steps = 0;
  int* bwd_masks = nullptr;  // slice lists of multi-slice backward visits
  int64_t n_bwd_masks = 0;
  int* bwd_items = nullptr;
  int64_t n_bwd_items = 0;
  int* bwd_order = nullptr;
  // Unsplit forward items for the dQ pass of the backward (aliases the
  // forward list when no item was split).
  int* dq_items = nullptr;
  int* dq_order = nullptr;
  int* dq_counts = nullptr;  // [n_dq_items][2]: visits of each half of a dQ item
  int64_t n_dq_items = 0;
  bool dq_alias = true;
  int* err = nullptr;  // device [2]: code, location
  int* tickets = nullptr;  // device [3]: work-queue counters (forward, dK/dV, dQ)
  int grid_fwd = 0, grid_bwd = 0, grid_dq = 0;
  cudaEvent_t events[6] = {};  // optional phase events (ffa_plan_set_events)
  bool use_events = false;
  int64_t area = 0;
  uint64_t wait_ns = 2000000000ull;
};

namespace ffa {
// Optional attention-sink logits (fp32): layout 0 is [n][Hq], layout 1 is
// [Tq][n][Hq]; n == 0 means no sink.
struct SinkArgs {
  const float* sink = nullptr;
  int n = 0;
  int layout = 0;
};
// Implemented in ffa_fwd.cu / ffa_bwd.cu.
ffa_status_t launch_fwd(ffa_plan_s* p, const void* q, const void* k, const void* v, float scale,
                        void* out, float* lse, void* ws, size_t ws_bytes, cudaStream_t st,
                        const SinkArgs& sink = SinkArgs(), float softcap = 0.f);
size_t fwd_workspace_bytes(const ffa_plan_s* p);
// dsink (when non-null and sink.n > 0) receives the sink gradient, in the
// sink's own layout, overwritten.
ffa_status_t launch_bwd(ffa_plan_s* p, const void* q, const void* k, const void* v,
                        const void* out, const void* dout, const float* lse, float scale,
                        void* dq, void* dk, void* dv, void* ws, size_t ws_bytes, cudaStream_t st,
                        const SinkArgs& sink = SinkArgs(), float* dsink = nullptr,
                        float softcap = 0.f);
// Softcap c > 0: every score x = scale * q.k becomes c * tanh(x / c).  In
// base-2 units the kernels use x2 = c log2(e) tanh(raw * scale / c).
//
// tanh(u) ~ u * sum_k kTanhPoly[k] * u^(2k) on |u| <= kTanhPolyRange: the odd
// polynomial of degree 9 with the smallest largest error relative to tanh
// (1.26e-6 in fp64, 1.33e-6 when evaluated by Horner in fp32), so a capped
// score c tanh(x / c) is off by at most 1.4e-6 |x| whatever the cap;
// written by tanh_poly.py in this package.
constexpr int kTanhPolyTerms = 5;
constexpr double kTanhPolyRange = 0.75;
constexpr double kTanhPoly[kTanhPolyTerms] = {
    9.99998743192078265e-01,
    -3.33262889929604456e-01,
    1.32458877985800832e-01,
    -4.97348543713007282e-02,
    1.26672359966334969e-02};
struct CapConsts {
  float a = 0.f;   // scale / c
  float c2 = 0.f;  // c * log2(e)
  // Fast path: for |raw| <= smax (u = raw * a within the polynomial's range)
  // the capped base-2 score is raw * R(raw^2), R(z) = sum_k r[k] z^k with
  // r[k] = log2(e) * scale * kTanhPoly[k] * a^(2k); r2 holds each r[k]
  // twice, the operand form of the packed two-lane FMAs, which then read it
  // from the kernel's parameters instead of holding it in registers.
  float r[kTanhPolyTerms] = {};
  float2 r2[kTanhPolyTerms] = {};
  // tanh itself (the backward also needs 1 - tanh^2): tanh(raw * a) =
  // raw * T(raw^2), T(z) = sum_k t[k] z^k, t[k] = kTanhPoly[k] * a^(2k+1),
  // as pairs.
  float2 t2[kTanhPolyTerms] = {};
  float smax = 0.f;
};
// Fills CapConsts for softmax scale `scale` and cap c > 0 (host side, in
// double so that c log2(e) and the powers of a neither overflow nor flush).
inline CapConsts make_cap_consts(float scale, float c) {
  CapConsts k;
  const double a = (double)scale / (double)c;
  k.a = (float)a;
  k.c2 = (float)((double)c * 1.4426950408889634);
  double apow = 1.0;
  for (int i = 0; i < kTanhPolyTerms; ++i) {
    k.r[i] = (float)(1.4426950408889634 * (double)scale * kTanhPoly[i] * apow);
    k.r2[i] = make_float2(k.r[i], k.r[i]);
    const float t = (float)(kTanhPoly[i] * apow * a);
    k.t2[i] = make_float2(t, t);
    apow *= a * a;
  }
  const double sm = kTanhPolyRange / a;
  k.smax = sm < 3.0e38 ? (float)sm : 3.0e38f;
  return k;
}
size_t bwd_workspace_bytes(const ffa_plan_s* p);
// Implemented in ffa_plan.cu.
bool on_plan_device(const ffa_plan_s* p);  // current device == the plan's device
// box_rows: 128 for whole tiles, kGatherKeys for the slots of gathered steps.
bool encode_tile_map(void* map128, const void* base, int rows, int cols_elems,
                     int box_rows = 128);
void note_launches(int n);  // adds to the count reported by ffa_kernel_launch_count
// Records phase event i of the plan on `st` when the caller asked for them.
inline void record_phase(const ffa_plan_s* p, int i, cudaStream_t st) {
  if (p->use_events) cudaEventRecord(p->events[i], st);
}
}  // namespace ffa
