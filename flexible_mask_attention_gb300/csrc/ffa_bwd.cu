// Backward kernels of flexible-mask attention for sm_103a, in two passes
// without atomics:
//
//   1. preprocess: -lse * log2(e) and -delta = -<dO, O> per (head, row), fp32,
//      stored negated so the kernels add them with FMAs;
//   2. dK/dV pass, one work item per (k-tile, kv head).  K and V stay in
//      shared memory; the item loops over every (q-tile, query head of the
//      group) that sees the k-tile:
//          S^T  = K Q^T                (tcgen05, SS)  -> TMEM
//          dP^T = V dO^T               (tcgen05, SS)  -> TMEM
//          P^T  = 2^(S^T*scale*log2e - lse2), masked on PARTIAL steps
//          dS^T = P^T * (dP^T - delta)
//          dV  += P^T dO               (tcgen05, A = P^T from TMEM)
//          dK  += dS^T Q               (tcgen05, A = dS^T from TMEM)
//      dK, dV accumulate in TMEM and are written once per item;
//   3. dQ pass, one work unit per (q-tile, query head), over the k-tiles the
//      q-tile sees (the forward's visits):
//          S  = Q K^T, dP = dO V^T     (tcgen05, SS)  -> TMEM
//          dS = 2^(S*scale*log2e - lse2) * (dP - delta), masked
//          dQ += dS K                  (tcgen05, A = dS from TMEM)
//      dQ accumulates in TMEM and is written once (bf16) per unit.
// This is the standard softmax-attention gradient; the mask only decides
// which entries of P are zero.  Recomputing S and dP in the dQ pass costs two
// extra MMAs per tile pair but removes the fp32 dQ reductions, which on this
// part cost more than the recomputation, and makes dQ deterministic.
#include <cuda_bf16.h>
#include <math.h>

#include <mutex>

#include "ffa_internal.cuh"
#include "ffa_ptx.cuh"

namespace ffa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ void drain_wait_b(uint32_t bar, uint32_t parity, uint64_t ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_test(bar, parity)) {
    if (globaltimer_ns() - t0 > ns) return;
  }
}

// ============================================================================
// dK / dV pass
// Warp roles (384 threads): warps 0-7 P/dS in two warpgroups (thread = key =
// TMEM lane; warpgroup w owns query columns [64w, 64w+64)) and the dK/dV
// epilogue, warp 8 TMA producer, warp 9 MMA issuer (TMEM owner), warps 10-11
// loaders of dO and of -lse2 / -delta for plans with gathered steps (idle
// otherwise); registers split 200 / 104 between them (ffa_ptx.cuh).
// TMEM columns: dV [0,D), dK [D,2D), S^T [2D,2D+128), dP^T [2D+128,2D+256).
// Warpgroup w owns dP^T columns [64w, 64w+64) of that range and, once it has
// read a 32-column chunk, overwrites the chunk with bf16 pairs: dS^T in its
// first 16 columns, P^T in its last 16.  Both later MMAs take their A operand
// from there, so shared memory carries only the four bf16 tiles.
template <int D>
struct KvCfg {
  static constexpr int kThreads = kSplitThreads;
  static constexpr int kChunks = D / 64;
  static constexpr int kTileBytes = 128 * D * 2;
  // Q is read first (by the S^T MMA), so it gets the deeper ring; -lse2 and
  // -delta (read with dP^T) travel with dO.
  static constexpr int kQStages = D == 128 ? 3 : 4;
  static constexpr int kDOStages = D == 128 ? 2 : 4;
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kTileBytes;
  static constexpr int kQOff = 2 * kTileBytes;
  static constexpr int kDOOff = kQOff + kQStages * kTileBytes;
  static constexpr int kLseOff = kDOOff + kDOStages * kTileBytes;  // per dO stage: -lse2, -delta
  static constexpr int kLseStageBytes = 2 * 128 * 4;
  static constexpr int kBarOff = kLseOff + kDOStages * kLseStageBytes;
  static constexpr int kBKVFull = 0, kBKVEmpty = 1, kBQFull = 2, kBQEmpty = 2 + kQStages,
                       kBDOFull = 2 + 2 * kQStages, kBSdpFull = kBDOFull + kDOStages,
                       kBSFree = kBSdpFull + 1,
                       kBPFull = kBSFree + 1, kBDkvFull = kBPFull + 2,
                       kBDkvEmpty = kBDkvFull + 1, kBDrain = kBDkvEmpty + 1,
                       kBSFull = kBDrain + 1, kBItemFull = kBSFull + 1,
                       kBItemEmpty = kBItemFull + kItemRing, kNumBars = kBItemEmpty + kItemRing;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  // The dynamic shared memory base must be 1024-byte aligned (checked on entry).
  static constexpr int kSlotOff = kMiscOff + 64;  // work-queue slots
  static constexpr int kSmemBytes = kSlotOff + 4 * kItemRing;
  static constexpr int kTdV = 0, kTdK = D, kTS = 2 * D, kTdP = 2 * D + 128;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

struct KvParams {
  const int4* steps;
  const int* items;
  const int* order;
  int* ticket;  // work-queue counter, zero at launch
  int n_items;
  const Slice* slices;
  const int* masks;  // slice lists of multi-slice visits
  const int* bgathers;  // gathered backward step records
  int Tq, Tk, Hkv, g, qpad;
  float scale, scale_log2;
  const float* nlse2;   // [Hq][qpad] -lse * log2(e)
  const float* ndelta;  // [Hq][qpad] -rowsum(dO * O)
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int* err;
  uint64_t wait_ns;
  CapConsts cap;  // used by the softcap instantiation only
};

// P^T and dS^T for one key row (TMEM lane) over the 32 queries
// [q0+32c, q0+32c+32) of the step (chunk c of this warpgroup's 64), from the
// S^T values already in registers (s) and the dP^T values read from TMEM here:
//   p = 2^(s * scale * log2e - lse2), ds = p * (dp - delta).
// They go back, as bf16 pairs, over the dP^T chunk they were read from:
// dS^T in columns [q0+32c, +16), P^T in [q0+32c+16, +16).
// Softcap (kCapMode > 0): scores capped to c tanh(scale s / c); then
// x = c log2e tanh(..) - lse2 and dS also carries the factor 1 - tanh^2.
// tanh comes from the exponential identity (kCapExp) or, when every score of
// the warp is in its range, from the odd polynomial (kCapPoly).
enum CapMode : int { kCapNone = 0, kCapExp = 1, kCapPoly = 2 };

// tanh(s * a) of two raw scores by the polynomial (their |s| <= cap.smax).
__device__ __forceinline__ float2 tanh_poly2(float2 sv, const CapConsts& cap) {
  const float2 w = __fmul2_rn(sv, sv);
  float2 r = cap.t2[kTanhPolyTerms - 1];
#pragma unroll
  for (int k = kTanhPolyTerms - 2; k >= 0; --k) r = __ffma2_rn(r, w, cap.t2[k]);
  return __fmul2_rn(sv, r);
}

// True for every lane when all n raw scores of every lane of the warp lie in
// the tanh polynomial's range (warp-uniform).
template <int n>
__device__ __forceinline__ bool scores_in_poly_range(const uint32_t* s, float smax) {
  float mx0 = -INFINITY, mx1 = -INFINITY, mn0 = INFINITY, mn1 = INFINITY;
#pragma unroll
  for (int c = 0; c + 3 < n; c += 4) {
    mx0 = fmax3(mx0, __uint_as_float(s[c]), __uint_as_float(s[c + 1]));
    mx1 = fmax3(mx1, __uint_as_float(s[c + 2]), __uint_as_float(s[c + 3]));
    mn0 = fmin3(mn0, __uint_as_float(s[c]), __uint_as_float(s[c + 1]));
    mn1 = fmin3(mn1, __uint_as_float(s[c + 2]), __uint_as_float(s[c + 3]));
  }
  const float big = fmaxf(fmaxf(mx0, mx1), -fminf(mn0, mn1));
  return __all_sync(0xffffffffu, big <= smax);
}

template <bool kPartial, int kCapMode, int c>
__device__ __forceinline__ void pds_chunk(const uint32_t (&s)[64], uint32_t tP, int q0,
                                          const float* nl, const float* nd, float scale_log2,
                                          const CapConsts& cap, uint32_t m_lo, uint32_t m_hi) {
  const float2 sc2 = make_float2(scale_log2, scale_log2);
  {
    uint32_t dp[32];
    tmem_ld32(tP + q0 + 32 * c, dp);
    uint32_t pp[16], dd[16];
#pragma unroll
    for (int e = 0; e < 32; e += 4) {
      const float4 l4 = *reinterpret_cast<const float4*>(nl + q0 + 32 * c + e);
      const float4 d4 = *reinterpret_cast<const float4*>(nd + q0 + 32 * c + e);
#pragma unroll
      for (int u = 0; u < 4; u += 2) {
        const int lc = 32 * c + e + u;  // column within this warpgroup's half
        const float2 nlp = u == 0 ? make_float2(l4.x, l4.y) : make_float2(l4.z, l4.w);
        const float2 ndp = u == 0 ? make_float2(d4.x, d4.y) : make_float2(d4.z, d4.w);
        const float2 sv = make_float2(__uint_as_float(s[lc]), __uint_as_float(s[lc + 1]));
        float2 th = make_float2(0.f, 0.f);
        if (kCapMode == kCapExp) th = make_float2(tanh_exp(sv.x * cap.a), tanh_exp(sv.y * cap.a));
        if (kCapMode == kCapPoly) th = tanh_poly2(sv, cap);
        const float2 x = kCapMode != kCapNone
                             ? __ffma2_rn(th, make_float2(cap.c2, cap.c2), nlp)
                             : __ffma2_rn(sv, sc2, nlp);
        float2 p = make_float2(ex2_approx(x.x), ex2_approx(x.y));
        if (kPartial) {  // bits of this warpgroup's 64 columns: m_lo (0-31), m_hi (32-63)
          const uint32_t mw = c == 0 ? m_lo : m_hi;
          p.x = ((mw >> (lc & 31)) & 1u) ? p.x : 0.f;
          p.y = ((mw >> ((lc + 1) & 31)) & 1u) ? p.y : 0.f;
        }
        const float2 dpd = __fadd2_rn(
            make_float2(__uint_as_float(dp[e + u]), __uint_as_float(dp[e + u + 1])), ndp);
        float2 ds = __fmul2_rn(p, dpd);
        if (kCapMode != kCapNone)
          ds = __fmul2_rn(ds, __ffma2_rn(make_float2(-th.x, -th.y), th, make_float2(1.f, 1.f)));
        pp[(e + u) >> 1] = pack_bf16x2(p.x, p.y);
        dd[(e + u) >> 1] = pack_bf16x2(ds.x, ds.y);
      }
    }
    tmem_st16(tP + q0 + 32 * c, dd);
    tmem_st16(tP + q0 + 32 * c + 16, pp);
  }
}

// kGather: the plan has gathered backward steps (instantiated apart).
template <int D, bool kCap, bool kGather>
__global__ void __launch_bounds__(KvCfg<D>::kThreads, 1)
    ffa_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ CUtensorMap tm_do,
                        const __grid_constant__ CUtensorMap tm_q8,
                        const __grid_constant__ CUtensorMap tm_do8, const KvParams P) {
  using C = KvCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  if ((smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) record_error(P.err, kDevBadSmemAlign, 1);
    return;
  }
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sbase + C::kBarOff + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);
  int* abort_flag = reinterpret_cast<int*>(smem + C::kMiscOff + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    mbar_init(bar(C::kBKVFull), 1);
    mbar_init(bar(C::kBKVEmpty), 1);
    for (int s = 0; s < C::kQStages; ++s) {
      mbar_init(bar(C::kBQFull + s), 1);
      mbar_init(bar(C::kBQEmpty + s), 1);
    }
    for (int s = 0; s < C::kDOStages; ++s) mbar_init(bar(C::kBDOFull + s), 1);
    mbar_init(bar(C::kBSdpFull), 1);
    mbar_init(bar(C::kBSFull), 1);
    for (int s = 0; s < kItemRing; ++s) {
      mbar_init(bar(C::kBItemFull + s), 1);
      // MMA thread + elementwise threads (+ lane 0 of the dO and -lse2 / -delta warps)
      mbar_init(bar(C::kBItemEmpty + s), 1 + 256 + (kGather ? 2 : 0));
    }
    mbar_init(bar(C::kBSFree), 256);
    mbar_init(bar(C::kBPFull), 256);
    mbar_init(bar(C::kBPFull + 1), 256);
    mbar_init(bar(C::kBDkvFull), 1);
    mbar_init(bar(C::kBDkvEmpty), 256);
    mbar_init(bar(C::kBDrain), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl ctl{abort_flag, P.err, P.wait_ns};
  const int g = P.g;
  const ItemQueue queue{reinterpret_cast<int*>(smem + C::kSlotOff), bar(C::kBItemFull),
                        bar(C::kBItemEmpty)};

  if (warp >= 8) {
  reg_dealloc<kSplitNarrowRegs>();
  if (warp == 8 || (kGather && warp >= 10)) {
    // ------------------------------------------------------------ producers
    // Warp 8 draws the items and loads K / V and Q; it loads dO, -lse2 and
    // -delta too unless the plan has gathered steps.  Each lane-issued copy
    // costs the issuing warp some 60 cycles, so with gathered steps (16
    // query blocks of 8 rows per tile: 2 x 16 boxes per tile with D = 128)
    // the dO tiles go to warp 10 and their -lse2 / -delta pieces to warp 11,
    // which take the items from the work queue like the consumers and wait
    // on the dO ring themselves.  Lane 0 of the loading warp waits on the
    // rings and sets each barrier's byte count (warp 10 for the dO ring: a
    // barrier may see warp 11's bytes before that, its phase cannot complete
    // without the arrival).  Without gathered steps lane 0 alone runs the
    // loop; with them the whole warp does, and the 16 query blocks of a
    // gathered tile (8 rows each at 1024-byte aligned slots; unused ones read
    // zero rows from row -8) and their 32-byte pieces of -lse2 and -delta
    // (unused ones copy row 0's, finite values that their masked columns
    // never use) are copied by lanes 0-15 after a __syncwarp that orders
    // them behind the waits.
    const int role = warp == 8 ? 0 : warp - 9;  // 0: items, K/V, Q; 1: dO; 2: -lse2, -delta
    const bool load_q = role == 0;
    const bool load_do = kGather ? role == 1 : true;
    const bool load_lse = kGather ? role == 2 : true;
    if (lane == 0) {
      if (role == 0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_q8);
      }
      if (load_do) {
        prefetch_tmap(&tm_do);
        prefetch_tmap(&tm_do8);
      }
    }
    uint32_t kv_cnt = 0, q_cnt = 0, do_cnt = 0;  // tiles issued
    bool ok = true;
    const unsigned pm = kGather ? 0xffffffffu : 1u;  // lanes running the loop
    if (kGather || lane == 0)
    for (int r = 0; ok; ++r) {
      int idx = -1;
      if (lane == 0) {
        if (role == 0) {
          const int pos = atomicAdd(P.ticket, 1);
          idx = pos < P.n_items ? P.order[pos] : -1;
          ok = queue_publish(queue, r, idx, ctl, 409);
        } else {
          ok = queue_take(queue, r, idx, ctl, 409 + role);
        }
      }
      ok = __shfl_sync(pm, ok, 0);
      idx = __shfl_sync(pm, idx, 0);
      if (!ok || idx < 0) break;
      const int* it = P.items + (size_t)idx * kBiWords;
      const int sb = it[kBiStepBeg], se = it[kBiStepEnd];
      if (se <= sb) continue;
      const int kt = it[kBiKt], hk = it[kBiHkv];
      if (role == 0) {
        if (lane == 0) {
          ok = mbar_wait(bar(C::kBKVEmpty), (kv_cnt & 1) ^ 1, ctl, 400);
          if (ok) {
            mbar_arrive_expect_tx(bar(C::kBKVFull), 2 * C::kTileBytes);
            for (int c = 0; c < C::kChunks; ++c) {
              tma_load_2d(sbase + C::kKOff + c * 16384, &tm_k, bar(C::kBKVFull), hk * D + c * 64,
                          kt * 128);
              tma_load_2d(sbase + C::kVOff + c * 16384, &tm_v, bar(C::kBKVFull), hk * D + c * 64,
                          kt * 128);
            }
          }
        }
        if (!(ok = __shfl_sync(pm, ok, 0))) break;
        ++kv_cnt;
      }
      const int n_it = (se - sb) * g;
      for (int i = 0; i < n_it; ++i) {
        const int4 stp = P.steps[sb + i / g];
        const int qt = stp.x;
        const int h = hk * g + i % g;
        const bool gat = kGather && stp.w > 0;
        // this lane's query block (read while the ring slots are awaited)
        const int y = gat && lane < kGatherSlots
                          ? P.bgathers[(size_t)(stp.w - 1) * kBGatherWords + lane] : 0;
        if (load_q) {
          const int qs = q_cnt % C::kQStages;
          if (lane == 0) {
            ok = mbar_wait(bar(C::kBQEmpty + qs), ((q_cnt / C::kQStages) & 1) ^ 1, ctl, 401);
            if (ok) mbar_arrive_expect_tx(bar(C::kBQFull + qs), C::kTileBytes);
          }
          if (!(ok = __shfl_sync(pm, ok, 0))) break;
          __syncwarp(pm);
          if (gat) {
            if (lane < kGatherSlots)
              for (int c = 0; c < C::kChunks; ++c)
                tma_load_2d(sbase + C::kQOff + qs * C::kTileBytes + c * 16384 + lane * 1024,
                            &tm_q8, bar(C::kBQFull + qs), h * D + c * 64, y);
          } else if (lane == 0) {
            for (int c = 0; c < C::kChunks; ++c)
              tma_load_2d(sbase + C::kQOff + qs * C::kTileBytes + c * 16384, &tm_q,
                          bar(C::kBQFull + qs), h * D + c * 64, qt * 128);
          }
          ++q_cnt;
        }
        if (load_do || load_lse) {
          const int ds = do_cnt % C::kDOStages;
          if (lane == 0) {
            // The dO stage (and its -lse2 / -delta) of iteration do_cnt - kDOStages
            // is free once that iteration's dV / dK MMAs are done, the moment
            // its Q stage is handed back: wait on that Q-empty phase, so the
            // MMA thread commits one barrier per iteration instead of two.
            if (do_cnt >= (uint32_t)C::kDOStages) {
              const uint32_t c0 = do_cnt - C::kDOStages;
              ok = mbar_wait(bar(C::kBQEmpty + c0 % C::kQStages), (c0 / C::kQStages) & 1, ctl,
                             402);
            }
            if (ok && load_do)
              mbar_arrive_expect_tx(bar(C::kBDOFull + ds), C::kTileBytes + C::kLseStageBytes);
          }
          if (!(ok = __shfl_sync(pm, ok, 0))) break;
          __syncwarp(pm);
          if (load_do) {
            if (gat) {
              if (lane < kGatherSlots)
                for (int c = 0; c < C::kChunks; ++c)
                  tma_load_2d(sbase + C::kDOOff + ds * C::kTileBytes + c * 16384 + lane * 1024,
                              &tm_do8, bar(C::kBDOFull + ds), h * D + c * 64, y);
            } else if (lane == 0) {
              for (int c = 0; c < C::kChunks; ++c)
                tma_load_2d(sbase + C::kDOOff + ds * C::kTileBytes + c * 16384, &tm_do,
                            bar(C::kBDOFull + ds), h * D + c * 64, qt * 128);
            }
          }
          if (load_lse) {
            const uint32_t ls = sbase + C::kLseOff + ds * C::kLseStageBytes;
            if (gat) {
              if (lane < kGatherSlots) {
                const size_t row = (size_t)h * P.qpad + (y > 0 ? y : 0);
                bulk_load(ls + lane * 32, P.nlse2 + row, 32, bar(C::kBDOFull + ds));
                bulk_load(ls + 512 + lane * 32, P.ndelta + row, 32, bar(C::kBDOFull + ds));
              }
            } else if (lane == 0) {
              bulk_load(ls, P.nlse2 + (size_t)h * P.qpad + qt * 128, 512, bar(C::kBDOFull + ds));
              bulk_load(ls + 512, P.ndelta + (size_t)h * P.qpad + qt * 128, 512,
                        bar(C::kBDOFull + ds));
            }
          }
          ++do_cnt;
        }
      }
    }
    if (!ok && lane == 0) {
      // let this warp's copies in flight land before the CTA exits
      if (kv_cnt > 0) drain_wait_b(bar(C::kBKVFull), (kv_cnt - 1) & 1, kDrainNs);
      for (uint32_t i = q_cnt > (uint32_t)C::kQStages ? q_cnt - C::kQStages : 0; i < q_cnt; ++i)
        drain_wait_b(bar(C::kBQFull + i % C::kQStages), (i / C::kQStages) & 1, kDrainNs);
      for (uint32_t i = do_cnt > (uint32_t)C::kDOStages ? do_cnt - C::kDOStages : 0; i < do_cnt;
           ++i)
        drain_wait_b(bar(C::kBDOFull + i % C::kDOStages), (i / C::kDOStages) & 1, kDrainNs);
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16(128, 128, false, false);
      constexpr uint32_t kIdAcc = idesc_bf16(128, D, false, true);  // A K-major, B MN-major
      constexpr uint32_t kTile16 = C::kTileBytes >> 4;
      // Base descriptors: K-major (k) and MN-major (m) views of each buffer.
      const uint64_t dKk = sdesc_sw128(sbase + C::kKOff, 16, 1024);
      const uint64_t dVk = sdesc_sw128(sbase + C::kVOff, 16, 1024);
      const uint64_t dQk = sdesc_sw128(sbase + C::kQOff, 16, 1024);
      const uint64_t dQm = sdesc_sw128(sbase + C::kQOff, 16384, 1024);
      const uint64_t dDOk = sdesc_sw128(sbase + C::kDOOff, 16, 1024);
      const uint64_t dDOm = sdesc_sw128(sbase + C::kDOOff, 16384, 1024);
      auto issue_st = [&](int qstage) {  // S^T = K Q^T
        const uint64_t qd = dQk + qstage * kTile16;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 1024 + (kk & 3) * 2;  // 16-byte units
          mma_ss_at(tmem + C::kTS, dKk, off, qd, off, kIdS, kk > 0 ? 1u : 0u);
        }
      };
      uint32_t kv_cnt = 0, q_cnt = 0, sf_cnt = 0, p_cnt = 0, dkv_cnt = 0;
      bool ok = true;
      for (int r = 0; ok; ++r) {
        int idx;
        if (!(ok = queue_take(queue, r, idx, ctl, 509)) || idx < 0) break;
        const int* it = P.items + (size_t)idx * kBiWords;
        const int sb = it[kBiStepBeg], se = it[kBiStepEnd];
        if (se <= sb) continue;
        // Waits on TMA barriers need no tcgen05 fence (the copies and the MMAs
        // are async-proxy operations ordered by the barrier); the waits on the
        // elementwise warps' arrivals are followed by one, and every MMA that
        // rewrites TMEM they read is issued after such a fence.
        if (!(ok = mbar_wait(bar(C::kBKVFull), kv_cnt & 1, ctl, 500))) break;
        ++kv_cnt;
        const int n_it = (se - sb) * g;
        {  // S^T of the first iteration
          const int qs = q_cnt % C::kQStages;
          if (!(ok = mbar_wait(bar(C::kBQFull + qs), (q_cnt / C::kQStages) & 1, ctl, 501))) break;
          issue_st(qs);
          mma_commit(bar(C::kBSFull));
        }
        for (int i = 0; i < n_it; ++i) {
          const uint32_t c = q_cnt + (uint32_t)i;
          const int qs = c % C::kQStages, ds = c % C::kDOStages;
          if (!(ok = mbar_wait(bar(C::kBDOFull + ds), (c / C::kDOStages) & 1, ctl, 502))) break;
          // dP^T = V dO^T; its columns were last read by the previous dV / dK MMAs.
          {
            const uint64_t dod = dDOk + ds * kTile16;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk >> 2) * 1024 + (kk & 3) * 2;
              mma_ss_at(tmem + C::kTdP, dVk, off, dod, off, kIdS, kk > 0 ? 1u : 0u);
            }
          }
          mma_commit(bar(C::kBSdpFull));
          if (i + 1 < n_it) {
            // S^T of the next iteration as soon as this S^T is in registers.
            const uint32_t c1 = c + 1;
            const int st1 = c1 % C::kQStages;
            if (!(ok = mbar_wait(bar(C::kBSFree), sf_cnt & 1, ctl, 503))) break;
            ++sf_cnt;
            if (!(ok = mbar_wait(bar(C::kBQFull + st1), (c1 / C::kQStages) & 1, ctl, 504))) break;
            tc_fence_after();
            issue_st(st1);
            mma_commit(bar(C::kBSFull));
          }
          if (!(ok = mbar_wait(bar(C::kBPFull), p_cnt & 1, ctl, 505))) break;
          tc_fence_after();
          if (i == 0) {
            if (!(ok = mbar_wait(bar(C::kBDkvEmpty), (dkv_cnt & 1) ^ 1, ctl, 506))) break;
            ++dkv_cnt;
            tc_fence_after();
          }
          const uint32_t acc0 = i > 0 ? 1u : 0u;
          const uint64_t dom = dDOm + ds * kTile16;
          const uint64_t qm = dQm + qs * kTile16;
          // queries [16kk, 16kk+16) with kk = 4w + 2c + h: warpgroup w, chunk c,
          // half h of the chunk's dS^T (and, 16 columns on, P^T) pairs.  Chunk 0
          // of both warpgroups first (kk = 0 is issued first: it starts the sum).
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            if (c == 1) {
              if (!(ok = mbar_wait(bar(C::kBPFull + 1), p_cnt & 1, ctl, 508))) break;
              tc_fence_after();
            }
#pragma unroll
            for (int w = 0; w < 2; ++w) {
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const int kk = 4 * w + 2 * c + h;
                const uint32_t ta = tmem + C::kTdP + 64 * w + 32 * c + 8 * h;
                const uint32_t acc = (acc0 || kk > 0) ? 1u : 0u;
                mma_ts_at(tmem + C::kTdV, ta + 16, dom, kk * 128, kIdAcc, acc);
                mma_ts_at(tmem + C::kTdK, ta, qm, kk * 128, kIdAcc, acc);
              }
            }
          }
          if (!ok) break;
          ++p_cnt;
          mma_commit(bar(C::kBQEmpty + qs));  // also frees the iteration's dO stage
        }
        if (!ok) break;
        // a pending S-free arrival of the last iteration is consumed here
        if (!(ok = mbar_wait(bar(C::kBSFree), sf_cnt & 1, ctl, 507))) break;
        ++sf_cnt;
        tc_fence_after();  // the next item's first S^T rewrites those columns
        q_cnt += (uint32_t)n_it;
        mma_commit(bar(C::kBDkvFull));
        mma_commit(bar(C::kBKVEmpty));
      }
      mma_commit(bar(C::kBDrain));
      drain_wait_b(bar(C::kBDrain), 0, kDrainNs);
    }
  }
  } else {
    reg_alloc<kSplitWideRegs>();
    // ------------------------------------------------------------ P / dS warps
    const int wg = warp >> 2;             // query columns [64wg, 64wg+64)
    const int j = threadIdx.x & 127;      // key lane
    const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_addr + C::kTS + 64 * wg;
    const uint32_t tP = tmem + lane_addr + C::kTdP;
    uint32_t sdp_cnt = 0, dkv_cnt = 0;
    bool ok = true;
    for (int r = 0; ok; ++r) {
      int idx = -1;
      const bool w = queue_take(queue, r, idx, ctl, 609);
      if (!(ok = __all_sync(0xffffffffu, w)) || idx < 0) break;
      const int* it = P.items + (size_t)idx * kBiWords;
      const int sb = it[kBiStepBeg], se = it[kBiStepEnd];
      const int kt = it[kBiKt], hk = it[kBiHkv];
      const int key = kt * 128 + j;
      const int n_it = (se - sb) * g;
      int4 st_next = n_it > 0 ? P.steps[sb] : make_int4(0, -1, -1, 0);
      for (int i = 0; i < n_it; ++i) {
        const int4 st = st_next;
        if (i + 1 < n_it) st_next = P.steps[sb + (i + 1) / g];  // prefetch the next descriptor
        const int qt = st.x, info = st.y;
        uint32_t vb[4] = {~0u, ~0u, ~0u, ~0u};
        if (info & 1) {
          if (kGather && st.w > 0)
            gather_key_mask(P.bgathers + (size_t)(st.w - 1) * kBGatherWords, j, P.Tq, vb);
          else
            step_mask<false>(info, P.slices, P.masks, key, qt, vb);
        }
        const float* nl = reinterpret_cast<const float*>(
            smem + C::kLseOff + (sdp_cnt % C::kDOStages) * C::kLseStageBytes);
        const float* nd = nl + 128;
        // S^T first: its buffer is released before dP^T is even complete, so
        // the next S^T can follow dP^T on the tensor pipe at once.
        const bool w = mbar_wait(bar(C::kBSFull), sdp_cnt & 1, ctl, 600);
        if (!(ok = __all_sync(0xffffffffu, w))) break;
        tc_fence_after();
        uint32_t s[64];
        tmem_ld64(tS, s);
        tc_fence_before();
        mbar_arrive(bar(C::kBSFree));
        const bool w2 = mbar_wait(bar(C::kBSdpFull), sdp_cnt & 1, ctl, 601);
        if (!(ok = __all_sync(0xffffffffu, w2))) break;
        ++sdp_cnt;
        tc_fence_after();
        const uint32_t m_lo = wg ? vb[2] : vb[0], m_hi = wg ? vb[3] : vb[1];
        const bool poly = kCap && scores_in_poly_range<64>(s, P.cap.smax);
        // Each 32-query chunk is signalled on its own, so the dV / dK MMAs of
        // the first chunk run while the second is computed.
#define FFA_PDS(chunk)                                                                       \
  do {                                                                                       \
    if (!kCap) {                                                                             \
      if (info & 1)                                                                          \
        pds_chunk<true, kCapNone, chunk>(s, tP, 64 * wg, nl, nd, P.scale_log2, P.cap, m_lo,  \
                                         m_hi);                                              \
      else                                                                                   \
        pds_chunk<false, kCapNone, chunk>(s, tP, 64 * wg, nl, nd, P.scale_log2, P.cap, m_lo, \
                                          m_hi);                                             \
    } else if (poly) {                                                                       \
      if (info & 1)                                                                          \
        pds_chunk<true, kCapPoly, chunk>(s, tP, 64 * wg, nl, nd, P.scale_log2, P.cap, m_lo,  \
                                         m_hi);                                              \
      else                                                                                   \
        pds_chunk<false, kCapPoly, chunk>(s, tP, 64 * wg, nl, nd, P.scale_log2, P.cap, m_lo, \
                                          m_hi);                                             \
    } else {                                                                                 \
      if (info & 1)                                                                          \
        pds_chunk<true, kCapExp, chunk>(s, tP, 64 * wg, nl, nd, P.scale_log2, P.cap, m_lo,   \
                                        m_hi);                                               \
      else                                                                                   \
        pds_chunk<false, kCapExp, chunk>(s, tP, 64 * wg, nl, nd, P.scale_log2, P.cap, m_lo,  \
                                         m_hi);                                              \
    }                                                                                        \
  } while (0)
        FFA_PDS(0);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(C::kBPFull));
        FFA_PDS(1);
#undef FFA_PDS
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(C::kBPFull + 1));
      }
      if (!ok) break;
      // ---- dK / dV epilogue: warpgroup wg writes columns [wg*D/2, (wg+1)*D/2)
      constexpr int kHalf = D / 2;
      uint4* pv = reinterpret_cast<uint4*>(P.dv + ((size_t)key * P.Hkv + hk) * D + wg * kHalf);
      uint4* pk = reinterpret_cast<uint4*>(P.dk + ((size_t)key * P.Hkv + hk) * D + wg * kHalf);
      const bool store = key < P.Tk;
      if (n_it > 0) {
        const bool w = mbar_wait(bar(C::kBDkvFull), dkv_cnt & 1, ctl, 610);
        if (!(ok = __all_sync(0xffffffffu, w))) break;
        ++dkv_cnt;
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < 2 * (kHalf / 32); ++c) {
          const bool is_k = c >= kHalf / 32;
          const int cc = is_k ? c - kHalf / 32 : c;
          uint32_t u[32];
          tmem_ld32(tmem + lane_addr + (is_k ? C::kTdK : C::kTdV) + wg * kHalf + 32 * cc, u);
          if (c == 2 * (kHalf / 32) - 1) {
            tc_fence_before();
            mbar_arrive(bar(C::kBDkvEmpty));
          }
          const float sc = is_k ? P.scale : 1.f;
          uint4* dst = (is_k ? pk : pv) + cc * 4;
          if (store) {
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[v] = make_uint4(
                  pack_bf16x2(__uint_as_float(u[8 * v]) * sc, __uint_as_float(u[8 * v + 1]) * sc),
                  pack_bf16x2(__uint_as_float(u[8 * v + 2]) * sc, __uint_as_float(u[8 * v + 3]) * sc),
                  pack_bf16x2(__uint_as_float(u[8 * v + 4]) * sc, __uint_as_float(u[8 * v + 5]) * sc),
                  pack_bf16x2(__uint_as_float(u[8 * v + 6]) * sc, __uint_as_float(u[8 * v + 7]) * sc));
          }
        }
      } else if (store) {
#pragma unroll
        for (int v = 0; v < kHalf / 8; ++v) pv[v] = pk[v] = make_uint4(0, 0, 0, 0);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ============================================================================
// dQ pass
// Work units: the halves of the planner's unsplit forward items, i.e. one
// (q-tile, query head) with its visits in k-tile order (in head-stacked
// plans a 64-row slab of two query heads, tile rows 0-63 and 64-127).
// Warp roles (384 threads): warps 0-7 dS warps in two warpgroups (thread =
// query row = TMEM lane; warpgroup w owns key columns [64w, 64w+64)) and the
// dQ epilogue, warp 8 TMA producer, warp 9 MMA issuer, warp 10 V loader for
// plans with gathered steps, idle otherwise as warp 11 is; registers split
// 200 / 104 as in the dK/dV pass.
// TMEM columns: S of even steps [0,128), of odd steps [128,256), dP
// [256,384), dQ [384,384+D).  Warpgroup w writes its dS pairs over columns
// [64w, 64w+32) of its step's S buffer (read by itself first); the dQ MMA
// reads them from TMEM.
template <int D>
struct DqCfg {
  static constexpr int kThreads = kSplitThreads;
  static constexpr int kChunks = D / 64;
  static constexpr int kTileBytes = 128 * D * 2;
  // K is read by the S MMA of a step and again by its dQ MMA at the end, so
  // it gets the deeper ring; V (read by the dP MMA only) is released as soon
  // as that MMA completes.
  static constexpr int kKStages = D == 128 ? 3 : 4;
  static constexpr int kVStages = D == 128 ? 2 : 4;
  static constexpr int kQOff = 0;
  static constexpr int kDOOff = kTileBytes;
  static constexpr int kKOff = 2 * kTileBytes;
  static constexpr int kVOff = kKOff + kKStages * kTileBytes;
  static constexpr int kBarOff = kVOff + kVStages * kTileBytes;
  // K and V of step c both land on step barrier c % kStepBars (warp 8 sets
  // the byte count of both): one wait per step covers the two tiles that the
  // S and dP MMAs of the step read back to back.  Each ring keeps its own
  // release barriers; kStepBars is the deeper ring's depth, so a tile is
  // only copied once the step barrier's previous phase has completed.
  static constexpr int kStepBars = kKStages > kVStages ? kKStages : kVStages;
  static constexpr int kBQFull = 0, kBQEmpty = 1, kBStepFull = 2,
                       kBKEmpty = kBStepFull + kStepBars, kBVEmpty = kBKEmpty + kKStages,
                       kBDpFree = kBVEmpty + kVStages,
                       kBDsFull = kBDpFree + 1, kBDqFull = kBDsFull + 1,
                       kBDqEmpty = kBDqFull + 1, kBDrain = kBDqEmpty + 1,
                       kBItemFull = kBDrain + 1, kBItemEmpty = kBItemFull + kItemRing,
                       kNumBars = kBItemEmpty + kItemRing;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;  // TMEM base, abort flag, queue slots
  static constexpr int kSmemBytes = kMiscOff + 64;
  static constexpr int kTS0 = 0, kTdP = 256, kTdQ = 384;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

struct DqParams {
  const int4* steps;
  const int* items;
  const int* order;
  int* ticket;  // work-queue counter, zero at launch
  const int* counts;  // visits of each half of an item
  int n_items;
  const Slice* slices;
  const int* masks;  // slice lists of multi-slice visits
  const int* gathers;  // gathered step records
  int Tq, Tk, Hq, g, qpad;
  int stack;  // head-stacked units: slab rows R (a half: R rows of 128 / R heads), or 0
  int alternate;  // an item's halves are the same rows, taking its steps in turn
  float scale, scale_log2;
  const float* nlse2;
  const float* ndelta;
  __nv_bfloat16* dq;
  int* err;
  uint64_t wait_ns;
  CapConsts cap;  // used by the softcap instantiation only
};

// dS = 2^(x - lse2) * (dP - delta) for 32 columns of one query row (x the
// base-2 score, capped by kCapMode as in pds_chunk), masked by the bits mw of
// the chunk when `partial`, as bf16 pairs.  c0: the chunk's first column in dp.
template <int kCapMode>
__device__ __forceinline__ void dq_ds_chunk(const uint32_t (&s)[32], const uint32_t (&dp)[64],
                                            int c0, uint32_t mw, bool partial, float2 nl2,
                                            float nd, float2 sc2, const CapConsts& cap,
                                            uint32_t (&dd)[16]) {
#pragma unroll
  for (int e = 0; e < 32; e += 2) {
    const int lc = c0 + e;
    const float2 sv = make_float2(__uint_as_float(s[e]), __uint_as_float(s[e + 1]));
    float2 th = make_float2(0.f, 0.f);
    if (kCapMode == kCapExp) th = make_float2(tanh_exp(sv.x * cap.a), tanh_exp(sv.y * cap.a));
    if (kCapMode == kCapPoly) th = tanh_poly2(sv, cap);
    const float2 x = kCapMode != kCapNone ? __ffma2_rn(th, make_float2(cap.c2, cap.c2), nl2)
                                          : __ffma2_rn(sv, sc2, nl2);
    float2 p = make_float2(ex2_approx(x.x), ex2_approx(x.y));
    if (partial) {
      p.x = ((mw >> (e & 31)) & 1u) ? p.x : 0.f;
      p.y = ((mw >> ((e + 1) & 31)) & 1u) ? p.y : 0.f;
    }
    float2 ds = __fmul2_rn(
        p, __fadd2_rn(make_float2(__uint_as_float(dp[lc]), __uint_as_float(dp[lc + 1])),
                      make_float2(nd, nd)));
    if (kCapMode != kCapNone)
      ds = __fmul2_rn(ds, __ffma2_rn(make_float2(-th.x, -th.y), th, make_float2(1.f, 1.f)));
    dd[e >> 1] = pack_bf16x2(ds.x, ds.y);
  }
}

__device__ __forceinline__ bool half_active(const int* it, int h) {
  return it[kFiQt0 + h] >= 0 && it[kFiH0 + h] >= 0;
}

__device__ __forceinline__ int half_info(const int4& st, int h) { return h == 0 ? st.y : st.z; }

// The dQ pass's view of a step: items whose two halves are the same rows
// taking the steps in turn (alternate) are walked as half 0 over all steps.
__device__ __forceinline__ int dq_info(const int4& st, int h, bool alternate) {
  return alternate ? (h == 0 ? max(st.y, st.z) : -1) : half_info(st, h);
}

// kGather: the plan has gathered steps (instantiated apart, as in the forward).
template <int D, bool kCap, bool kGather>
__global__ void __launch_bounds__(DqCfg<D>::kThreads, 1)
    ffa_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_do,
                      const __grid_constant__ CUtensorMap tm_k8,
                      const __grid_constant__ CUtensorMap tm_v8,
                      const __grid_constant__ CUtensorMap tm_q64,
                      const __grid_constant__ CUtensorMap tm_do64, const DqParams P) {
  using C = DqCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  if ((smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) record_error(P.err, kDevBadSmemAlign, 2);
    return;
  }
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sbase + C::kBarOff + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);
  int* abort_flag = reinterpret_cast<int*>(smem + C::kMiscOff + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    mbar_init(bar(C::kBQFull), 1);
    mbar_init(bar(C::kBQEmpty), 1);
    for (int s = 0; s < C::kStepBars; ++s) mbar_init(bar(C::kBStepFull + s), 1);
    for (int s = 0; s < C::kKStages; ++s) mbar_init(bar(C::kBKEmpty + s), 1);
    for (int s = 0; s < C::kVStages; ++s) mbar_init(bar(C::kBVEmpty + s), 1);
    mbar_init(bar(C::kBDpFree), 256);
    mbar_init(bar(C::kBDsFull), 256);
    mbar_init(bar(C::kBDqFull), 1);
    mbar_init(bar(C::kBDqEmpty), 256);
    mbar_init(bar(C::kBDrain), 1);
    for (int s = 0; s < kItemRing; ++s) {
      mbar_init(bar(C::kBItemFull + s), 1);
      // MMA thread + dS threads (+ lane 0 of the V warp)
      mbar_init(bar(C::kBItemEmpty + s), 1 + 256 + (kGather ? 1 : 0));
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl ctl{abort_flag, P.err, P.wait_ns};
  const ItemQueue queue{reinterpret_cast<int*>(smem + C::kMiscOff + 16), bar(C::kBItemFull),
                        bar(C::kBItemEmpty)};

  if (warp >= 8) {
  reg_dealloc<kSplitNarrowRegs>();
  if (warp == 8 || (kGather && warp == 10)) {
    // ------------------------------------------------------------ producers
    // Warp 8 draws the items and loads Q / dO and K, and V too unless the
    // plan has gathered steps; then warp 10 loads V (a gathered tile is 16
    // slots x D / 64 boxes per tensor, and each lane-issued copy costs the
    // issuing warp some 60 cycles), taking the items from the work queue like
    // the consumers and waiting on the V ring itself.  Lane 0 of each loading
    // warp waits on its ring's release; warp 8's sets the step barrier's byte
    // count for the step's K and V (warp 10's V copies may land on it first:
    // its phase cannot complete without that arrival).  With gathered steps
    // the whole warp runs the loop and the 16 slots of a gathered K/V tile
    // (8 rows each, 1024-byte aligned, unused ones reading zero rows from row
    // -8) are copied by lanes 0-15 in parallel after a __syncwarp that orders
    // them behind the wait; without them lane 0 runs it alone (measured
    // faster there).
    const bool role0 = warp == 8;
    const bool load_k = role0, load_v = !kGather || !role0;
    if (lane == 0) {
      if (role0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_do);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_k8);
      }
      if (load_v) {
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_v8);
      }
    }
    auto load_kv = [&](uint32_t dst, const CUtensorMap* m, const CUtensorMap* m8, uint32_t b,
                       int hk, const int4& stp, int y) {
      if (kGather && stp.w > 0) {
        if (lane < kGatherSlots)
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_2d(dst + c * 16384 + lane * 1024, m8, b, hk * D + c * 64, y);
      } else if (lane == 0) {
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_2d(dst + c * 16384, m, b, hk * D + c * 64, stp.x * 128);
      }
    };
    uint32_t k_cnt = 0, v_cnt = 0, q_cnt = 0;
    bool ok = true;
    // without gathered steps lane 0 runs the loop alone
    const unsigned pm = kGather ? 0xffffffffu : 1u;
    if (kGather || lane == 0)
    for (int r = 0; ok; ++r) {
      int idx = -1;
      if (lane == 0) {
        if (role0) {
          const int pos = atomicAdd(P.ticket, 1);
          idx = pos < P.n_items ? P.order[pos] : -1;
          ok = queue_publish(queue, r, idx, ctl, 809);
        } else {
          ok = queue_take(queue, r, idx, ctl, 810);
        }
      }
      ok = __shfl_sync(pm, ok, 0);
      idx = __shfl_sync(pm, idx, 0);
      if (!ok || idx < 0) break;
      const int* it = P.items + (size_t)idx * kFiWords;
      const int sb = it[kFiStepBeg], se = it[kFiStepEnd];
      if (se <= sb) continue;
      for (int h = 0; ok && h < 2; ++h) {
        if (!half_active(it, h)) continue;
        const int n = P.counts[2 * idx + h];
        if (n == 0) continue;
        const int qt = it[kFiQt0 + h], head = it[kFiH0 + h], hk = head / P.g;
        if (role0) {
          if (lane == 0) {
            ok = mbar_wait(bar(C::kBQEmpty), (q_cnt & 1) ^ 1, ctl, 800);
            if (ok) {
              mbar_arrive_expect_tx(bar(C::kBQFull), 2 * C::kTileBytes);
              if (kGather && P.stack) {  // heads head, head + 1, ... of the R-row slab qt
                const int R = P.stack;
                for (int j = 0; j < 128 / R; ++j)
                  for (int c = 0; c < C::kChunks; ++c) {
                    const uint32_t o = c * 16384 + j * (R * 128);
                    tma_load_2d(sbase + C::kQOff + o, &tm_q64, bar(C::kBQFull),
                                (head + j) * D + c * 64, qt * R);
                    tma_load_2d(sbase + C::kDOOff + o, &tm_do64, bar(C::kBQFull),
                                (head + j) * D + c * 64, qt * R);
                  }
              } else {
                for (int c = 0; c < C::kChunks; ++c) {
                  tma_load_2d(sbase + C::kQOff + c * 16384, &tm_q, bar(C::kBQFull),
                              head * D + c * 64, qt * 128);
                  tma_load_2d(sbase + C::kDOOff + c * 16384, &tm_do, bar(C::kBQFull),
                              head * D + c * 64, qt * 128);
                }
              }
            }
          }
          if (!(ok = __shfl_sync(pm, ok, 0))) break;
          ++q_cnt;
        }
        for (int j = sb; j < se; ++j) {
          const int4 st = P.steps[j];
          if (dq_info(st, h, kGather && P.alternate) < 0) continue;
          // this lane's slot start (read while the ring slots are awaited)
          const int y = kGather && st.w > 0 && lane < kGatherSlots
                            ? P.gathers[(size_t)(st.w - 1) * kGatherWords + lane] : 0;
          if (load_k) {
            const int ks = k_cnt % C::kKStages;
            if (lane == 0) {
              ok = mbar_wait(bar(C::kBKEmpty + ks), ((k_cnt / C::kKStages) & 1) ^ 1, ctl, 801);
              if (ok)  // the step's K and V (V's copies may land first)
                mbar_arrive_expect_tx(bar(C::kBStepFull + k_cnt % C::kStepBars), 2 * C::kTileBytes);
            }
            if (!(ok = __shfl_sync(pm, ok, 0))) break;
            __syncwarp(pm);
            load_kv(sbase + C::kKOff + ks * C::kTileBytes, &tm_k, &tm_k8,
                    bar(C::kBStepFull + k_cnt % C::kStepBars), hk, st, y);
            ++k_cnt;
          }
          if (load_v) {
            const int vs = v_cnt % C::kVStages;
            if (lane == 0) {
              ok = mbar_wait(bar(C::kBVEmpty + vs), ((v_cnt / C::kVStages) & 1) ^ 1, ctl, 802);
            }
            if (!(ok = __shfl_sync(pm, ok, 0))) break;
            __syncwarp(pm);
            load_kv(sbase + C::kVOff + vs * C::kTileBytes, &tm_v, &tm_v8,
                    bar(C::kBStepFull + v_cnt % C::kStepBars), hk, st, y);
            ++v_cnt;
          }
        }
      }
    }
    if (!ok && lane == 0) {
      // let this warp's copies in flight land before the CTA exits
      if (q_cnt > 0) drain_wait_b(bar(C::kBQFull), (q_cnt - 1) & 1, kDrainNs);
      const uint32_t n_cp = k_cnt > v_cnt ? k_cnt : v_cnt;  // steps this warp copied into
      for (uint32_t i = n_cp > (uint32_t)C::kStepBars ? n_cp - C::kStepBars : 0; i < n_cp; ++i)
        drain_wait_b(bar(C::kBStepFull + i % C::kStepBars), (i / C::kStepBars) & 1, kDrainNs);
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16(128, 128, false, false);
      constexpr uint32_t kIdQ = idesc_bf16(128, D, false, true);  // A from TMEM, B MN-major
      constexpr uint32_t kTile16 = C::kTileBytes >> 4;
      const uint64_t dQk = sdesc_sw128(sbase + C::kQOff, 16, 1024);
      const uint64_t dDOk = sdesc_sw128(sbase + C::kDOOff, 16, 1024);
      const uint64_t dKk = sdesc_sw128(sbase + C::kKOff, 16, 1024);
      const uint64_t dKm = sdesc_sw128(sbase + C::kKOff, 16384, 1024);
      const uint64_t dVk = sdesc_sw128(sbase + C::kVOff, 16, 1024);
      auto issue_s = [&](int buf, int stage) {  // S = Q K^T
        const uint64_t kd = dKk + stage * kTile16;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 1024 + (kk & 3) * 2;  // 16-byte units
          mma_ss_at(tmem + C::kTS0 + 128 * buf, dQk, off, kd, off, kIdS, kk > 0 ? 1u : 0u);
        }
      };
      auto issue_dp = [&](int stage) {  // dP = dO V^T
        const uint64_t vd = dVk + stage * kTile16;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 1024 + (kk & 3) * 2;
          mma_ss_at(tmem + C::kTdP, dDOk, off, vd, off, kIdS, kk > 0 ? 1u : 0u);
        }
      };
      uint32_t kv_cnt = 0, q_cnt = 0, dpf_cnt = 0, ds_cnt = 0, dqe_cnt = 0;
      bool ok = true;
      for (int r = 0; ok; ++r) {
        int idx;
        if (!(ok = queue_take(queue, r, idx, ctl, 909)) || idx < 0) break;
        const int* it = P.items + (size_t)idx * kFiWords;
        const int sb = it[kFiStepBeg], se = it[kFiStepEnd];
        if (se <= sb) continue;
        for (int h = 0; ok && h < 2; ++h) {
          if (!half_active(it, h)) continue;
          const int n = P.counts[2 * idx + h];
          if (n == 0) continue;
          if (!(ok = mbar_wait(bar(C::kBQFull), q_cnt & 1, ctl, 900))) break;
          ++q_cnt;
          tc_fence_after();
          {  // step 0: S and dP
            const int ks = kv_cnt % C::kKStages, vs = kv_cnt % C::kVStages;
            if (!(ok = mbar_wait(bar(C::kBStepFull + kv_cnt % C::kStepBars),
                                 (kv_cnt / C::kStepBars) & 1, ctl, 901)))
              break;  // K and V of the step
            tc_fence_after();
            issue_s(0, ks);
            issue_dp(vs);
            // V is read by the dP MMA only; the same arrival tells the dS
            // warps that this step's S and dP are in TMEM
            mma_commit(bar(C::kBVEmpty + vs));
          }
          for (int v = 0; v < n; ++v) {
            const uint32_t c = kv_cnt + (uint32_t)v;
            const int stage = c % C::kKStages;  // K of this step (read by its dQ MMA)
            if (v + 1 < n) {
              const uint32_t c1 = c + 1;
              const int k1 = c1 % C::kKStages, v1 = c1 % C::kVStages;
              if (!(ok = mbar_wait(bar(C::kBStepFull + c1 % C::kStepBars), (c1 / C::kStepBars) & 1,
                                   ctl, 903)))
                break;  // K and V of step v + 1
              tc_fence_after();
              issue_s((v + 1) & 1, k1);
              if (!(ok = mbar_wait(bar(C::kBDpFree), dpf_cnt & 1, ctl, 904))) break;
              ++dpf_cnt;
              tc_fence_after();
              issue_dp(v1);
              mma_commit(bar(C::kBVEmpty + v1));  // V free; S and dP of step v + 1 ready
            }
            if (!(ok = mbar_wait(bar(C::kBDsFull), ds_cnt & 1, ctl, 906))) break;
            ++ds_cnt;
            tc_fence_after();
            if (v == 0) {
              if (!(ok = mbar_wait(bar(C::kBDqEmpty), (dqe_cnt & 1) ^ 1, ctl, 907))) break;
              ++dqe_cnt;
              tc_fence_after();
            }
            const uint64_t km = dKm + stage * kTile16;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)  // dS pairs of keys [16kk, 16kk+16)
              mma_ts_at(tmem + C::kTdQ, tmem + C::kTS0 + 128 * (v & 1) + 64 * (kk >> 2) + 8 * (kk & 3),
                        km, kk * 128, kIdQ, (v > 0 || kk > 0) ? 1u : 0u);
            mma_commit(bar(C::kBKEmpty + stage));
          }
          if (!ok) break;
          // the dS warps' dP-free arrival of the last step
          if (!(ok = mbar_wait(bar(C::kBDpFree), dpf_cnt & 1, ctl, 908))) break;
          ++dpf_cnt;
          kv_cnt += (uint32_t)n;
          mma_commit(bar(C::kBDqFull));
          mma_commit(bar(C::kBQEmpty));
        }
      }
      mma_commit(bar(C::kBDrain));
      drain_wait_b(bar(C::kBDrain), 0, kDrainNs);
    }
  }
  } else {
    reg_alloc<kSplitWideRegs>();
    // ------------------------------------------------------------ dS warps
    const int wg = warp >> 2;         // key columns [64wg, 64wg+64)
    const int t = threadIdx.x & 127;  // query row within the tile = TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
    uint32_t sd_cnt = 0, dq_cnt = 0;
    bool ok = true;
    const float2 sc2 = make_float2(P.scale_log2, P.scale_log2);
    for (int r = 0; ok; ++r) {
      int idx = -1;
      const bool w = queue_take(queue, r, idx, ctl, 1009);
      if (!(ok = __all_sync(0xffffffffu, w)) || idx < 0) break;
      const int* it = P.items + (size_t)idx * kFiWords;
      const int sb = it[kFiStepBeg], se = it[kFiStepEnd];
      for (int h = 0; ok && h < 2; ++h) {
        if (!half_active(it, h) || (kGather && P.alternate && h == 1)) continue;
        const int qt = it[kFiQt0 + h];
        // tile row -> query row and head (head-stacked: R-row slab of 128 / R heads)
        const bool stk = kGather && P.stack;
        const int row = stk ? qt * P.stack + (t & (P.stack - 1)) : qt * 128 + t;
        const int head = it[kFiH0 + h] + (stk ? t / P.stack : 0);
        const float nl = P.nlse2[(size_t)head * P.qpad + row];
        const float nd = P.ndelta[(size_t)head * P.qpad + row];
        const float2 nl2 = make_float2(nl, nl);
        int v = 0;
        int4 st_next = sb < se ? P.steps[sb] : make_int4(0, -1, -1, 0);
        for (int j = sb; j < se; ++j) {
          const int4 st = st_next;
          if (j + 1 < se) st_next = P.steps[j + 1];  // prefetch the next step descriptor
          const int info = dq_info(st, h, kGather && P.alternate);
          if (info < 0) continue;
          // A gathered step's column mask (every step of such a unit is one;
          // none for a step whose rows all see all its keys) is read while
          // the scores are awaited; a PARTIAL tile's after.
          uint32_t vb[4] = {~0u, ~0u, ~0u, ~0u};
          if (kGather && st.w > 0 && (info & 1))
            gather_mask(P.gathers + (size_t)(st.w - 1) * kGatherWords, h, t, P.Tk, vb);
          // S and dP of the step are in TMEM once its V stage is handed back
          // (one arrival per step on the V ring serves both)
          const bool w = mbar_wait(bar(C::kBVEmpty + sd_cnt % C::kVStages),
                                   (sd_cnt / C::kVStages) & 1, ctl, 1000);
          if (!(ok = __all_sync(0xffffffffu, w))) break;
          ++sd_cnt;
          tc_fence_after();
          uint32_t dp[64];
          tmem_ld64(tmem + lane_addr + C::kTdP + 64 * wg, dp);
          tc_fence_before();
          mbar_arrive(bar(C::kBDpFree));
          if ((info & 1) && !(kGather && st.w > 0))
            step_mask<true>(info, P.slices, P.masks, row, st.x, vb);
          const uint32_t m_lo = wg ? vb[2] : vb[0], m_hi = wg ? vb[3] : vb[1];
          const uint32_t tSb = tmem + lane_addr + C::kTS0 + 128 * (v & 1) + 64 * wg;
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t s[32];
            tmem_ld32(tSb + 32 * c, s);
            const uint32_t mw = c == 0 ? m_lo : m_hi;
            uint32_t dd[16];
            if (!kCap)
              dq_ds_chunk<kCapNone>(s, dp, 32 * c, mw, info & 1, nl2, nd, sc2, P.cap, dd);
            else if (scores_in_poly_range<32>(s, P.cap.smax))
              dq_ds_chunk<kCapPoly>(s, dp, 32 * c, mw, info & 1, nl2, nd, sc2, P.cap, dd);
            else
              dq_ds_chunk<kCapExp>(s, dp, 32 * c, mw, info & 1, nl2, nd, sc2, P.cap, dd);
            // chunk c writes columns [64wg + 16c, 64wg + 16c + 16), read by chunk 0
            tmem_st16(tSb + 16 * c, dd);
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(bar(C::kBDsFull));
          ++v;
        }
        if (!ok) break;
        // ---- epilogue: dQ * scale -> bf16; warpgroup wg writes columns [wg*D/2, (wg+1)*D/2)
        constexpr int kHalf = D / 2;
        uint4* dst = reinterpret_cast<uint4*>(P.dq + ((size_t)row * P.Hq + head) * D + wg * kHalf);
        const bool store = row < P.Tq;
        if (v > 0) {
          const bool w = mbar_wait(bar(C::kBDqFull), dq_cnt & 1, ctl, 1010);
          if (!(ok = __all_sync(0xffffffffu, w))) break;
          ++dq_cnt;
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < kHalf / 32; ++c) {
            uint32_t u[32];
            tmem_ld32(tmem + lane_addr + C::kTdQ + wg * kHalf + 32 * c, u);
            if (c == kHalf / 32 - 1) {
              tc_fence_before();
              mbar_arrive(bar(C::kBDqEmpty));
            }
            if (store) {
#pragma unroll
              for (int q4 = 0; q4 < 4; ++q4)
                dst[4 * c + q4] = make_uint4(
                    pack_bf16x2(__uint_as_float(u[8 * q4]) * P.scale,
                                __uint_as_float(u[8 * q4 + 1]) * P.scale),
                    pack_bf16x2(__uint_as_float(u[8 * q4 + 2]) * P.scale,
                                __uint_as_float(u[8 * q4 + 3]) * P.scale),
                    pack_bf16x2(__uint_as_float(u[8 * q4 + 4]) * P.scale,
                                __uint_as_float(u[8 * q4 + 5]) * P.scale),
                    pack_bf16x2(__uint_as_float(u[8 * q4 + 6]) * P.scale,
                                __uint_as_float(u[8 * q4 + 7]) * P.scale));
            }
          }
        } else if (store) {
#pragma unroll
          for (int c = 0; c < kHalf / 8; ++c) dst[c] = make_uint4(0, 0, 0, 0);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// -delta = -rowsum(dO * O), -lse2 = -lse * log2(e); padded rows get 0.
// HBM-bound (it reads out and dout once).  A block covers 64 consecutive rows
// of one head: each warp takes 8 of them, D / 8 lanes per row reading 16
// bytes each (a warp's load covers 2 or 4 whole rows, 512 contiguous bytes
// when Hq = 1 and full 32-byte sectors always), issues all of its loads
// before using any, and sums each row with a shuffle tree in a fixed order;
// the block's lse reads and scratch writes are contiguous.
constexpr int kPreRows = 64;  // rows per block (8 warps x 8 rows)

template <int D>
__global__ void __launch_bounds__(256)
    ffa_bwd_pre_kernel(const __nv_bfloat16* __restrict__ out,
                       const __nv_bfloat16* __restrict__ dout, const float* __restrict__ lse,
                       int Tq, int Hq, int qpad, float* __restrict__ nlse2,
                       float* __restrict__ ndelta) {
  constexpr int kLanes = D / 8;              // lanes per row, 16 bytes each
  constexpr int kRowsPerLoad = 32 / kLanes;  // rows one warp-wide load covers
  constexpr int kIters = 8 / kRowsPerLoad;   // loads per lane and tensor
  const int h = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = lane / kLanes, li = lane % kLanes;
  const int q_base = blockIdx.x * kPreRows + warp * 8;
  uint4 a[kIters], b[kIters];
#pragma unroll
  for (int it = 0; it < kIters; ++it) {
    const int q = q_base + it * kRowsPerLoad + sub;
    if (q < Tq) {
      const size_t off = ((size_t)q * Hq + h) * D + li * 8;
      a[it] = *reinterpret_cast<const uint4*>(out + off);
      b[it] = *reinterpret_cast<const uint4*>(dout + off);
    } else {
      a[it] = b[it] = make_uint4(0, 0, 0, 0);
    }
  }
#pragma unroll
  for (int it = 0; it < kIters; ++it) {
    const uint32_t aw[4] = {a[it].x, a[it].y, a[it].z, a[it].w};
    const uint32_t bw[4] = {b[it].x, b[it].y, b[it].z, b[it].w};
    float dsum = 0.f;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float2 fa = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&aw[t]));
      const float2 fb = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&bw[t]));
      dsum = fmaf(fa.x, fb.x, dsum);
      dsum = fmaf(fa.y, fb.y, dsum);
    }
#pragma unroll
    for (int o = kLanes / 2; o > 0; o >>= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, o);
    const int q = q_base + it * kRowsPerLoad + sub;
    if (li == 0 && q < qpad) {
      // -inf stays -inf (such rows see no key); padded rows get 0
      const float l2 = q < Tq ? lse[(size_t)h * Tq + q] * kLog2e : 0.f;
      nlse2[(size_t)h * qpad + q] = -l2;
      ndelta[(size_t)h * qpad + q] = -dsum;
    }
  }
}

// Gradient of the attention-sink logits, which enter only the normaliser:
//   dsink_s = -sum_i exp(sink_s - lse_i) delta_i = sum_i 2^(sink_s log2 e + nlse2_i) ndelta_i
// over the rows i of the head (nlse2 = -lse log2 e and ndelta = -delta from
// the preprocess kernel).  Layout 0 ([n][Hq]): one block per (s, head), each
// thread sums a fixed stride of rows and the block adds the partial sums in a
// fixed tree, so the result does not depend on scheduling.  Layout 1
// ([Tq][n][Hq]): one thread per element, no sum.
__global__ void __launch_bounds__(256)
    ffa_dsink_kernel(const float* __restrict__ sink, int n, int layout, int Tq, int Hq, int qpad,
                     const float* __restrict__ nlse2, const float* __restrict__ ndelta,
                     float* __restrict__ dsink) {
  if (layout == 0) {
    __shared__ float red[256];
    const int s = blockIdx.x / Hq, h = blockIdx.x % Hq;
    const float sg = sink[(size_t)s * Hq + h] * kLog2e;
    const float* nl = nlse2 + (size_t)h * qpad;
    const float* nd = ndelta + (size_t)h * qpad;
    float acc = 0.f;
    for (int i = threadIdx.x; i < Tq; i += 256) {
      const float e = sg + nl[i];
      if (e > -INFINITY && e < INFINITY) acc = fmaf(exp2f(e), nd[i], acc);
    }
    red[threadIdx.x] = acc;
    __syncthreads();
    for (int w = 128; w > 0; w >>= 1) {
      if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
      __syncthreads();
    }
    if (threadIdx.x == 0) dsink[(size_t)s * Hq + h] = red[0];
  } else {
    const long long idx = (long long)blockIdx.x * 256 + threadIdx.x;  // (row * n + s) * Hq + h
    if (idx >= (long long)Tq * n * Hq) return;
    const int h = (int)(idx % Hq), i = (int)(idx / Hq / n);
    const float e = sink[idx] * kLog2e + nlse2[(size_t)h * qpad + i];
    dsink[idx] = (e > -INFINITY && e < INFINITY) ? exp2f(e) * ndelta[(size_t)h * qpad + i] : 0.f;
  }
}

template <int D, bool kCap, bool kGather>
ffa_status_t launch_bwd_d(ffa_plan_s* p, const void* q, const void* k, const void* v,
                          const void* out, const void* dout, const float* lse, float scale,
                          void* dq, void* dk, void* dv, void* ws, cudaStream_t st,
                          const SinkArgs& sk, float* dsink, float softcap) {
  CapConsts cap;
  if (kCap) cap = make_cap_consts(scale, softcap);
  const int qpad = p->n_qt * 128;
  float* nlse2 = static_cast<float*>(ws);
  float* ndelta = nlse2 + (size_t)p->Hq * qpad;
  {
    record_phase(p, 2, st);
    const dim3 grid((unsigned)(qpad / kPreRows), (unsigned)p->Hq);
    ffa_bwd_pre_kernel<D><<<grid, 256, 0, st>>>(
        static_cast<const __nv_bfloat16*>(out), static_cast<const __nv_bfloat16*>(dout), lse,
        p->Tq, p->Hq, qpad, nlse2, ndelta);
    note_launches(1);
    if (cudaGetLastError() != cudaSuccess) return FFA_ERR_CUDA;
  }
  if (sk.n > 0 && dsink) {
    const unsigned blocks =
        sk.layout == 0 ? (unsigned)(sk.n * p->Hq)
                       : (unsigned)(((long long)p->Tq * sk.n * p->Hq + 255) / 256);
    if (blocks > 0) {
      ffa_dsink_kernel<<<blocks, 256, 0, st>>>(sk.sink, sk.n, sk.layout, p->Tq, p->Hq, qpad, nlse2,
                                               ndelta, dsink);
      note_launches(1);
      if (cudaGetLastError() != cudaSuccess) return FFA_ERR_CUDA;
    }
  }
  alignas(64) CUtensorMap tq, tk, tv, tdo, tk8, tv8, tq8, tdo8, tq64, tdo64;
  if (!encode_tile_map(&tq, q, p->Tq, p->Hq * D) || !encode_tile_map(&tk, k, p->Tk, p->Hkv * D) ||
      !encode_tile_map(&tv, v, p->Tk, p->Hkv * D) || !encode_tile_map(&tdo, dout, p->Tq, p->Hq * D) ||
      !encode_tile_map(&tk8, k, p->Tk, p->Hkv * D, kGatherKeys) ||
      !encode_tile_map(&tv8, v, p->Tk, p->Hkv * D, kGatherKeys) ||
      !encode_tile_map(&tq8, q, p->Tq, p->Hq * D, kGatherKeys) ||
      !encode_tile_map(&tdo8, dout, p->Tq, p->Hq * D, kGatherKeys) ||
      !encode_tile_map(&tq64, q, p->Tq, p->Hq * D, p->stacked ? p->stacked : kSlabRows) ||
      !encode_tile_map(&tdo64, dout, p->Tq, p->Hq * D, p->stacked ? p->stacked : kSlabRows))
    return FFA_ERR_INVALID_ARG;
  const float scale_log2 = scale * kLog2e;
  {
    using C = KvCfg<D>;
    KvParams P;
    P.steps = p->bwd_steps;
    P.items = p->bwd_items;
    P.order = p->bwd_order;
    P.ticket = p->tickets + 1;
    P.n_items = (int)p->n_bwd_items;
    P.slices = p->slices;
    P.masks = p->bwd_masks;
    P.bgathers = p->bgathers;
    P.Tq = p->Tq;
    P.Tk = p->Tk;
    P.Hkv = p->Hkv;
    P.g = p->Hq / p->Hkv;
    P.qpad = qpad;
    P.scale = scale;
    P.scale_log2 = scale_log2;
    P.nlse2 = nlse2;
    P.ndelta = ndelta;
    P.dk = static_cast<__nv_bfloat16*>(dk);
    P.cap = cap;
    P.dv = static_cast<__nv_bfloat16*>(dv);
    P.err = p->err;
    P.wait_ns = p->wait_ns;
    // the dK/dV pass gathers when the backward lists have gathered steps
    const bool bg = p->n_bgathers > 0;
    auto kern = bg ? ffa_bwd_dkdv_kernel<D, kCap, true> : ffa_bwd_dkdv_kernel<D, kCap, false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) !=
        cudaSuccess)
      return FFA_ERR_CUDA;
    if (!(bg ? split_regs_ok<ffa_bwd_dkdv_kernel<D, kCap, true>>()
             : split_regs_ok<ffa_bwd_dkdv_kernel<D, kCap, false>>()))
      return FFA_ERR_UNSUPPORTED;
    if (cudaMemsetAsync(P.ticket, 0, sizeof(int), st) != cudaSuccess) return FFA_ERR_CUDA;
    record_phase(p, 3, st);
    kern<<<p->grid_bwd, C::kThreads, C::kSmemBytes, st>>>(tq, tk, tv, tdo, tq8, tdo8, P);
    note_launches(1);
    if (cudaGetLastError() != cudaSuccess) return FFA_ERR_CUDA;
  }
  {
    using C = DqCfg<D>;
    DqParams P;
    P.steps = p->fwd_steps;
    P.items = p->dq_items;
    P.order = p->dq_order;
    P.ticket = p->tickets + 2;
    P.counts = p->dq_counts;
    P.n_items = (int)p->n_dq_items;
    P.slices = p->slices;
    P.masks = p->fwd_masks;
    P.gathers = p->gathers;
    P.Tq = p->Tq;
    P.Tk = p->Tk;
    P.Hq = p->Hq;
    P.g = p->Hq / p->Hkv;
    P.qpad = qpad;
    P.stack = p->stacked;
    P.alternate = p->alternate;
    P.scale = scale;
    P.scale_log2 = scale_log2;
    P.nlse2 = nlse2;
    P.ndelta = ndelta;
    P.dq = static_cast<__nv_bfloat16*>(dq);
    P.cap = cap;
    P.err = p->err;
    P.wait_ns = p->wait_ns;
    if (cudaFuncSetAttribute(ffa_bwd_dq_kernel<D, kCap, kGather>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) != cudaSuccess)
      return FFA_ERR_CUDA;
    if (!split_regs_ok<ffa_bwd_dq_kernel<D, kCap, kGather>>()) return FFA_ERR_UNSUPPORTED;
    if (cudaMemsetAsync(P.ticket, 0, sizeof(int), st) != cudaSuccess) return FFA_ERR_CUDA;
    record_phase(p, 4, st);
    ffa_bwd_dq_kernel<D, kCap, kGather><<<p->grid_dq, C::kThreads, C::kSmemBytes, st>>>(
        tq, tk, tv, tdo, tk8, tv8, tq64, tdo64, P);
    note_launches(1);
    if (cudaGetLastError() != cudaSuccess) return FFA_ERR_CUDA;
  }
  record_phase(p, 5, st);
  return FFA_OK;
}

}  // namespace

size_t bwd_workspace_bytes(const ffa_plan_s* p) {
  const size_t qpad = (size_t)p->n_qt * 128;
  return 2 * qpad * p->Hq * sizeof(float);
}

ffa_status_t launch_bwd(ffa_plan_s* p, const void* q, const void* k, const void* v,
                        const void* out, const void* dout, const float* lse, float scale,
                        void* dq, void* dk, void* dv, void* ws, size_t, cudaStream_t st,
                        const SinkArgs& sink, float* dsink, float softcap) {
  const bool c = softcap > 0.f, g = p->n_gathers > 0;
#define FFA_BWD(DD, CC, GG)                                                                   \
  launch_bwd_d<DD, CC, GG>(p, q, k, v, out, dout, lse, scale, dq, dk, dv, ws, st, sink, dsink, \
                           softcap)
  if (p->D == 128)
    return c ? (g ? FFA_BWD(128, true, true) : FFA_BWD(128, true, false))
             : (g ? FFA_BWD(128, false, true) : FFA_BWD(128, false, false));
  if (p->D == 64)
    return c ? (g ? FFA_BWD(64, true, true) : FFA_BWD(64, true, false))
             : (g ? FFA_BWD(64, false, true) : FFA_BWD(64, false, false));
#undef FFA_BWD
  return FFA_ERR_UNSUPPORTED;
}

}  // namespace ffa

// ---------------------------------------------------------------------------
// Allocation-free backward.
//
// Some callers cannot allocate device memory at the point where they run the
// backward: runtimes that forbid allocation once they have started, hosts
// whose own memory manager owns every byte of the GPU, or latency-critical
// loops that must not pay for (or synchronise on) an allocation.
// ffa_bwd_noalloc serves them: its scratch (log2-scaled lse and delta) lives
// in the array below, which every GPU that loads this library holds until the
// process exits.  All calls share it, so calls whose kernels overlap on the
// GPU race.  The first call on a device resolves the array's address for
// that device; make that first call before any stream capture.
namespace ffa {
namespace {

constexpr size_t kNoAllocScratchBytes = 64ull << 20;  // 64 MiB
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array for the current device.  Host code
// cannot use the array's name as a device address; the runtime resolves it
// once per device (with that device current).
ffa_status_t noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FFA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FFA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return FFA_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return FFA_OK;
}

bool aligned16_b(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace ffa

extern "C" size_t ffa_bwd_noalloc_max_workspace(void) { return ffa::kNoAllocScratchBytes; }

extern "C" ffa_status_t ffa_bwd_noalloc(ffa_plan_t p, const void* q, const void* k, const void* v,
                                        const void* out, const void* dout, const float* lse,
                                        float softmax_scale, void* dq, void* dk, void* dv,
                                        ffa_stream_t stream) {
  using namespace ffa;
  if (!p || !q || !k || !v || !out || !dout || !lse || !dq || !dk || !dv)
    return FFA_ERR_INVALID_ARG;
  // The scratch address below is resolved for the current device, and the
  // plan's lists live on the plan's device: both must be the same GPU.
  if (!on_plan_device(p)) return FFA_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, out, dout, lse, dq, dk, dv};
  for (const void* x : ptrs)
    if (!aligned16_b(x)) return FFA_ERR_INVALID_ARG;
  const size_t need = bwd_workspace_bytes(p);
  if (need > kNoAllocScratchBytes) return FFA_ERR_WORKSPACE;
  void* ws = nullptr;
  const ffa_status_t rc = noalloc_scratch(&ws);
  if (rc != FFA_OK) return rc;
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf((float)p->D);
  return launch_bwd(p, q, k, v, out, dout, lse, scale, dq, dk, dv, ws, need,
                    reinterpret_cast<cudaStream_t>(stream));
}
