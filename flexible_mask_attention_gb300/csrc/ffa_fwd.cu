// Forward kernel of flexible-mask attention for sm_103a, and the logsumexp
// merge of split work items.
//
// One persistent CTA per SM walks its share of the planner's work items.  An
// item holds two 128-row halves (two query heads of one kv head, or two
// consecutive q-tiles of one head; in head-stacked plans each half is one
// 64-row slab of two query heads) that share every K/V tile load.
//
// Warp roles (384 threads, three warpgroups):
//   warps 0-3  softmax for half 0 (thread = query row = TMEM lane)
//   warps 4-7  softmax for half 1
//   warp  8    TMA producer: Q tiles, then a ring of K/V stages (stage u
//              of an item: V of step u - 1 with K of step u)
//   warp  9    tcgen05 MMA issuer (and TMEM owner)
//   warp  10   V loader for plans with gathered steps (idle otherwise)
//   warp  11   idle
// Registers: the control warpgroup (warps 8-11) shrinks to 104 per thread
// and the softmax warpgroups grow to 200 (the split in ffa_ptx.cuh).
// TMEM (512 columns): S0 [0,128), S1 [128,256), O0 [256,256+D), O1 [384,384+D).
// P (bf16) is written back over the first 64 columns of S and read from TMEM
// by the P*V MMA.
//
// Per k-tile step j, the MMA order is  PV0(j), S0(j+1), PV1(j), S1(j+1), so
// one half's softmax overlaps the other half's MMAs.  Because tcgen05 MMAs
// complete in issue order, the commit that announces S_h(j+1) also tells the
// softmax warps that PV_h(j) is done, which is when O_h may be rescaled.
//
// Online softmax (fp32, base 2): m is the running row maximum of
// scale*log2(e)*s; it is only raised when a new maximum exceeds it by more
// than 8 (then O and l are rescaled), so p = 2^(x - m) stays below 256.
// Masked entries become -inf (only on PARTIAL steps), a row with no visible
// key keeps l = 0 and is written as out = 0, lse = -inf.
//
// Softcap (optional, a separate instantiation): scores become
// c * tanh(scale * s / c) before the softmax; the tile maximum is capped the
// same way (tanh is increasing) and masked entries stay -inf.  When every
// score of a warp's 32 rows lies in the range of the odd tanh polynomial
// (|scale * s / c| <= 0.75), the capped scores come from that polynomial on the
// FMA pipe (one MUFU operation per score, the exponential); otherwise from
// tanh(u) = 1 - 2 / (e^(2u) + 1), which costs two more.
//
// Attention sink (optional): the sink logits of a row join its normaliser
// only.  The epilogue of an unsplit item (or the merge of a split one) adds
// log2 sum_s 2^(sink_s log2 e) to the keys' log-normaliser and scales out by
// the keys' share of the total, so a row with no visible key gets out = 0
// and lse = logsumexp(sink).
#include <cuda_bf16.h>
#include <math.h>

#include <type_traits>

#include "ffa_internal.cuh"
#include "ffa_ptx.cuh"

namespace ffa {
namespace {

constexpr int kFwdThreads = kSplitThreads;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;

template <int D>
struct FwdCfg {
  static constexpr int kChunks = D / 64;          // 128-byte column chunks per row
  static constexpr int kTileBytes = 128 * D * 2;  // one 128 x D bf16 tile
  static constexpr int kStages = D == 128 ? 2 : 4;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = 2 * kTileBytes;
  static constexpr int kVOff = kKOff + kStages * kTileBytes;
  static constexpr int kBarOff = kVOff + kStages * kTileBytes;
  // barrier indices
  // K/V ring: stage u of an item holds V of step u - 1 and K of step u (the
  // first only K, the last only V; see the producer)
  static constexpr int kBQFull = 0, kBQEmpty = 1, kBStFull = 2, kBStEmpty = 2 + kStages,
                       kBSFull = 2 + 2 * kStages, kBPFull = kBSFull + 2, kBOFull = kBPFull + 2,
                       kBOEmpty = kBOFull + 2, kBDrain = kBOEmpty + 2,
                       kBItemFull = kBDrain + 1, kBItemEmpty = kBItemFull + kItemRing,
                       kBHandFull = kBItemEmpty + kItemRing, kBHandEmpty = kBHandFull + 1,
                       kNumBars = kBHandEmpty + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;  // TMEM base, abort flag, queue slots
  // alternating items: half 1's row state (m, l) handed to half 0
  static constexpr int kHandOff = kMiscOff + 64;
  static constexpr int kSmemBytes = kHandOff + 128 * 8 + 1024;  // + alignment slack
  // Output staging (plans with short items, see launch_fwd): its barriers
  // (per half: chunk written, chunk read by the store) and one 64-column
  // bf16 chunk of a half's output tile per half, past the end of the
  // unstaged layout, which stays as it is.
  static constexpr int kEpiBarOff = kHandOff + 128 * 8;
  static constexpr int kEpiOff = (kEpiBarOff + 4 * 8 + 1023) / 1024 * 1024;
  static constexpr int kEpiHalfBytes = 128 * 64 * 2;
  static constexpr int kSmemBytesStaged = kEpiOff + 2 * kEpiHalfBytes + 1024;
  static_assert(kSmemBytesStaged <= 227 * 1024, "shared memory budget");
};

struct FwdParams {
  const int4* steps;
  const int* items;
  const int* order;
  int* ticket;  // work-queue counter, zero at launch
  int n_items;
  const Slice* slices;
  const int* masks;  // slice lists of multi-slice visits
  const int* gathers;  // gathered step records
  int Tq, Tk, Hq, g;
  int stack;  // head-stacked units: slab rows R (a half: R rows of 128 / R heads), or 0
  int alternate;  // an item's halves are the same rows, taking its steps in turn
  float scale_log2;
  __nv_bfloat16* out;
  float* lse;
  float* part_o;    // [slot][2][128][D]
  float* part_lse;  // [slot][2][128], log2 units
  int* err;
  uint64_t wait_ns;
  const float* sink;  // optional sink logits
  int n_sink, sink_layout;
  CapConsts cap;      // used by the softcap instantiation only
};

// Tensor maps of the output for staged stores (128-row and slab-row boxes);
// an empty parameter for kernels that store from registers.
struct OutMaps {
  CUtensorMap o, o64;
  __device__ const CUtensorMap* map() const { return &o; }
  __device__ const CUtensorMap* map64() const { return &o64; }
};
struct NoOutMaps {
  __device__ const CUtensorMap* map() const { return nullptr; }
  __device__ const CUtensorMap* map64() const { return nullptr; }
};
template <bool kStage>
using OutMapsT = typename std::conditional<kStage, OutMaps, NoOutMaps>::type;

// Capped score in base-2 units for raw score x (-inf stays -inf).
__device__ __forceinline__ float capped2(float x, const CapConsts& c) {
  return x == -INFINITY ? -INFINITY : c.c2 * tanh_exp(x * c.a);
}

// The same on the polynomial's range |x| <= c.smax (-inf stays -inf).
__device__ __forceinline__ float capped2_poly(float x, const CapConsts& c) {
  if (x == -INFINITY) return -INFINITY;
  const float w = x * x;
  float r = c.r[kTanhPolyTerms - 1];
#pragma unroll
  for (int k = kTanhPolyTerms - 2; k >= 0; --k) r = fmaf(r, w, c.r[k]);
  return x * r;
}

// Exponent modes of one softmax tile (see exp_tile).
enum ExpMode : int {
  kExpPlain = 0,    // p = 2^(s * scale * log2e - m)
  kExpCapExp = 1,   // capped score from the exponential identity of tanh
  kExpCapPoly = 2,  // capped score from the tanh polynomial (every score in range)
  kExpCapPolyMask = 3  // the same on a PARTIAL step: masked columns forced to p = 0
};

// p = 2^(x - mu) for the 128 scores of one row (x the base-2 score, capped
// or not), written as bf16 pairs over S columns [0, 64); returns their sum.
// Masked scores arrive as -inf.  The polynomial modes first turn the raw
// scores into x - mu in place (the polynomial of -inf is not -inf, so in
// kExpCapPolyMask the row's column mask puts -inf back), then exponentiate.
template <int kMode>
__device__ __forceinline__ float exp_tile(uint32_t (&u)[128], uint32_t tS, float mu,
                                          float scale_log2, const CapConsts& cap,
                                          const uint32_t (&vb)[4]) {
  const float2 sc2 = make_float2(scale_log2, scale_log2);
  const float2 nm2 = make_float2(-mu, -mu);
  if (kMode >= kExpCapPoly) {
    // capped base-2 scores minus mu, in place
#pragma unroll
    for (int c = 0; c < 128; c += 2) {
      const float2 sv = make_float2(__uint_as_float(u[c]), __uint_as_float(u[c + 1]));
      const float2 w = __fmul2_rn(sv, sv);
      float2 r = cap.r2[kTanhPolyTerms - 1];
#pragma unroll
      for (int k = kTanhPolyTerms - 2; k >= 0; --k) r = __ffma2_rn(r, w, cap.r2[k]);
      float2 t = __ffma2_rn(sv, r, nm2);
      if (kMode == kExpCapPolyMask) {
        t.x = mask_bit(vb, c) ? t.x : -INFINITY;
        t.y = mask_bit(vb, c + 1) ? t.y : -INFINITY;
      }
      u[c] = __float_as_uint(t.x);
      u[c + 1] = __float_as_uint(t.y);
    }
  }
  float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                   make_float2(0.f, 0.f)};
#pragma unroll
  for (int q4 = 0; q4 < 4; ++q4) {
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int c = 32 * q4 + 2 * i;
      const float2 sv = make_float2(__uint_as_float(u[c]), __uint_as_float(u[c + 1]));
      float2 t;
      if (kMode == kExpPlain) t = __ffma2_rn(sv, sc2, nm2);
      else if (kMode == kExpCapExp) t = make_float2(capped2(sv.x, cap) - mu, capped2(sv.y, cap) - mu);
      else t = sv;
      const float2 p = make_float2(ex2_approx(t.x), ex2_approx(t.y));
      acc[i & 3] = __fadd2_rn(acc[i & 3], p);
      pk[i] = pack_bf16x2(p.x, p.y);
    }
    tmem_st16(tS + 16 * q4, pk);
  }
  return (acc[0].x + acc[0].y) + (acc[1].x + acc[1].y) + (acc[2].x + acc[2].y) +
         (acc[3].x + acc[3].y);
}

// log2 of sum_s exp(sink_s) for (row, head) (-inf without sinks); sink logits
// are natural-log values.  layout 0: sink[s][Hq], layout 1: sink[row][s][Hq].
__device__ __forceinline__ float sink_log2(const float* sink, int n, int layout, int row, int head,
                                           int Hq) {
  if (n <= 0) return -INFINITY;
  const float* b = layout == 0 ? sink + head : sink + (size_t)row * n * Hq + head;
  float mx = -INFINITY;
  for (int s = 0; s < n; ++s) mx = fmaxf(mx, b[(size_t)s * Hq] * kLog2e);
  if (mx == -INFINITY) return -INFINITY;
  float sum = 0.f;
  for (int s = 0; s < n; ++s) sum += exp2f(b[(size_t)s * Hq] * kLog2e - mx);
  return mx + log2f(sum);
}

// log2(2^a + 2^b), -inf when both are -inf.
__device__ __forceinline__ float log2_add(float a, float b) {
  const float mx = fmaxf(a, b);
  if (mx == -INFINITY) return -INFINITY;
  return mx + log2f(exp2f(a - mx) + exp2f(b - mx));
}

// Wait that ignores the abort flag (used to drain copies in flight).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_test(bar, parity)) {
    if (globaltimer_ns() - t0 > ns) return;
  }
}

// kGather: the plan has gathered steps (instantiated apart, so that plans
// without them run code with no trace of the gathered paths).  kStage: the
// bf16 output leaves through shared memory and TMA stores (see the epilogue).
template <int D, bool kCap, bool kGather, bool kStage>
__global__ void __launch_bounds__(kFwdThreads, 1)
    ffa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_k8,
                   const __grid_constant__ CUtensorMap tm_v8,
                   const __grid_constant__ CUtensorMap tm_q64, const FwdParams P,
                   const __grid_constant__ OutMapsT<kStage> om) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sbase + C::kBarOff + 8 * i; };
  auto epi_full = [&](int h) -> uint32_t { return sbase + C::kEpiBarOff + 8 * h; };
  auto epi_free = [&](int h) -> uint32_t { return sbase + C::kEpiBarOff + 16 + 8 * h; };
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
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar(C::kBStFull + s), 1);   // warp 8's arrival with the stage's bytes
      mbar_init(bar(C::kBStEmpty + s), 1);  // the MMA thread's commit
    }
    for (int h = 0; h < 2; ++h) {
      mbar_init(bar(C::kBSFull + h), 1);
      mbar_init(bar(C::kBPFull + h), 128);
      mbar_init(bar(C::kBOFull + h), 1);
      mbar_init(bar(C::kBOEmpty + h), 128);
    }
    mbar_init(bar(C::kBDrain), 1);
    mbar_init(bar(C::kBHandFull), 128);   // half 1's threads
    mbar_init(bar(C::kBHandEmpty), 128);  // half 0's threads
    if (kStage)
      for (int h = 0; h < 2; ++h) {
        mbar_init(epi_full(h), 128);  // the half's threads wrote the chunk
        mbar_init(epi_free(h), 1);    // its store has read the chunk
      }
    for (int s = 0; s < kItemRing; ++s) {
      mbar_init(bar(C::kBItemFull + s), 1);
      // MMA thread + softmax threads (+ lane 0 of the V warp)
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
    // Warp 8 draws the items and loads Q and K, and V too unless the plan
    // has gathered steps; then warp 10 loads V (a gathered tile is 16 slots x
    // D / 64 boxes per tensor, and each lane-issued copy costs the issuing
    // warp some 60 cycles), taking the items from the work queue like the
    // consumers and waiting on the ring itself.  The ring's stage u of an
    // item (n steps, stages 0..n) holds V of step u - 1 and K of step u: the
    // two tiles the MMA thread needs next once step u - 1's P is ready, so
    // one wait and one release per step cover both.  Lane 0 of warp 8 waits
    // on the ring and sets each stage's byte count (both tiles'); warp 10's
    // V copies may land on the stage's barrier before that arrival, whose
    // phase cannot complete without it.  With gathered steps the whole warp
    // runs the loop and the 16 slots of a gathered tile (8 rows each,
    // 1024-byte aligned, unused ones reading zero rows from row -8) are
    // copied by lanes 0-15 in parallel after a __syncwarp that orders them
    // behind the wait; without them lane 0 runs it alone.
    const bool role0 = warp == 8;
    const bool load_v = !kGather || !role0;
    if (lane == 0) {
      if (role0) {
        prefetch_tmap(&tm_q);
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
    uint32_t u_cnt = 0, q_cnt = 0;  // ring stages and Q tiles issued
    bool ok = true;
    const unsigned pm = kGather ? 0xffffffffu : 1u;  // lanes running the loop
    if (kGather || lane == 0)
    for (int r = 0; ok; ++r) {
      int idx = -1;
      if (lane == 0) {
        if (role0) {
          const int pos = atomicAdd(P.ticket, 1);
          idx = pos < P.n_items ? P.order[pos] : -1;
          ok = queue_publish(queue, r, idx, ctl, 109);
        } else {
          ok = queue_take(queue, r, idx, ctl, 110);
        }
      }
      ok = __shfl_sync(pm, ok, 0);
      idx = __shfl_sync(pm, idx, 0);
      if (!ok || idx < 0) break;
      const int* it = P.items + (size_t)idx * kFiWords;
      const int sb = it[kFiStepBeg], se = it[kFiStepEnd];
      if (se <= sb) continue;
      const bool act1 = it[kFiQt1] >= 0 && it[kFiH1] >= 0;
      const int hk = it[kFiH0] / P.g;
      if (role0) {
        if (lane == 0) {
          ok = mbar_wait(bar(C::kBQEmpty), (q_cnt & 1) ^ 1, ctl, 100);
          if (ok) {
            mbar_arrive_expect_tx(bar(C::kBQFull), (act1 ? 2 : 1) * C::kTileBytes);
            if (kGather && P.stack) {
              // a half: the slab's R rows of heads h, h + 1, ..., tile rows
              // [R j, R j + R) for head h + j (128 R bytes apart in each
              // 128-byte column chunk); tm_q64's box is R rows
              const int R = P.stack;
              for (int hh = 0; hh < (act1 ? 2 : 1); ++hh)
                for (int j = 0; j < 128 / R; ++j)
                  for (int c = 0; c < C::kChunks; ++c)
                    tma_load_2d(sbase + C::kQOff + hh * C::kTileBytes + c * 16384 + j * (R * 128),
                                &tm_q64, bar(C::kBQFull), (it[kFiH0 + hh] + j) * D + c * 64,
                                it[kFiQt0 + hh] * R);
            } else {
              for (int c = 0; c < C::kChunks; ++c)
                tma_load_2d(sbase + C::kQOff + c * 16384, &tm_q, bar(C::kBQFull),
                            it[kFiH0] * D + c * 64, it[kFiQt0] * 128);
              if (act1)
                for (int c = 0; c < C::kChunks; ++c)
                  tma_load_2d(sbase + C::kQOff + C::kTileBytes + c * 16384, &tm_q,
                              bar(C::kBQFull), it[kFiH1] * D + c * 64, it[kFiQt1] * 128);
            }
          }
        }
        if (!(ok = __shfl_sync(pm, ok, 0))) break;
        ++q_cnt;
      }
      const int n = se - sb;
      for (int u = 0; u <= n; ++u) {
        const bool has_k = u < n, has_v = u > 0;
        const bool mine = role0 ? has_k : has_v;  // this warp copies a tile into the stage
        const int4 stp = mine ? P.steps[sb + (role0 ? u : u - 1)] : make_int4(0, -1, -1, 0);
        // this lane's slot start of that tile (read while the stage is awaited)
        const int y = kGather && mine && stp.w > 0 && lane < kGatherSlots
                          ? P.gathers[(size_t)(stp.w - 1) * kGatherWords + lane] : 0;
        const int stage = u_cnt % C::kStages;
        if (lane == 0) {
          ok = mbar_wait(bar(C::kBStEmpty + stage), ((u_cnt / C::kStages) & 1) ^ 1, ctl,
                         role0 ? 101 : 102);
          if (ok && role0)
            mbar_arrive_expect_tx(bar(C::kBStFull + stage),
                                  ((has_k ? 1 : 0) + (has_v ? 1 : 0)) * C::kTileBytes);
        }
        if (!(ok = __shfl_sync(pm, ok, 0))) break;
        __syncwarp(pm);
        if (role0 && has_k)
          load_kv(sbase + C::kKOff + stage * C::kTileBytes, &tm_k, &tm_k8,
                  bar(C::kBStFull + stage), hk, stp, y);
        if (load_v && has_v) {
          const int4 stv = role0 ? P.steps[sb + u - 1] : stp;  // warp 8 alone: no gathered steps
          load_kv(sbase + C::kVOff + stage * C::kTileBytes, &tm_v, &tm_v8,
                  bar(C::kBStFull + stage), hk, stv, y);
        }
        ++u_cnt;
      }
    }
    if (!ok && lane == 0) {
      // Aborted: let this warp's copies already issued land before the CTA exits.
      if (q_cnt > 0) drain_wait(bar(C::kBQFull), (q_cnt - 1) & 1, kDrainNs);
      for (uint32_t i = u_cnt > (uint32_t)C::kStages ? u_cnt - C::kStages : 0; i < u_cnt; ++i)
        drain_wait(bar(C::kBStFull + i % C::kStages), (i / C::kStages) & 1, kDrainNs);
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16(128, 128, false, false);
      constexpr uint32_t kIdPV = idesc_bf16(128, D, false, true);
      constexpr uint32_t kTile16 = C::kTileBytes >> 4;
      const uint64_t dQ = sdesc_sw128(sbase + C::kQOff, 16, 1024);     // K-major
      const uint64_t dK = sdesc_sw128(sbase + C::kKOff, 16, 1024);     // K-major
      const uint64_t dV = sdesc_sw128(sbase + C::kVOff, 16384, 1024);  // MN-major
      auto issue_s = [&](int h, int stage) {
        const uint64_t qd = dQ + h * kTile16, kd = dK + stage * kTile16;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 1024 + (kk & 3) * 2;  // 16-byte units
          mma_ss_at(tmem + h * 128, qd, off, kd, off, kIdS, kk > 0 ? 1u : 0u);
        }
      };
      auto issue_pv = [&](int h, int stage, bool acc) {
        const uint64_t vd = dV + stage * kTile16;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts_at(tmem + 256 + h * 128, tmem + h * 128 + kk * 8, vd, kk * 128, kIdPV,
                    (acc || kk > 0) ? 1u : 0u);
      };
      uint32_t u_cnt = 0, q_cnt = 0, p_cnt[2] = {0, 0}, oe_cnt[2] = {0, 0};  // u: ring stages
      const bool alt_items = kGather && P.alternate;
      bool ok = true;
      for (int r = 0; ok; ++r) {
        int idx;
        if (!(ok = queue_take(queue, r, idx, ctl, 209)) || idx < 0) break;
        const int* it = P.items + (size_t)idx * kFiWords;
        const int sb = it[kFiStepBeg], se = it[kFiStepEnd];
        if (se <= sb) continue;
        const bool act1 = it[kFiQt1] >= 0 && it[kFiH1] >= 0;
        // Waits on TMA barriers need no tcgen05 fence: the copies and the MMAs
        // that read them are both async-proxy operations ordered by the
        // barrier.  A fence follows the waits on the softmax warps' arrivals
        // (their TMEM reads and writes must come before the MMAs that reuse
        // those columns), and every S MMA is issued after such a fence.
        if (!(ok = mbar_wait(bar(C::kBQFull), q_cnt & 1, ctl, 200))) break;
        ++q_cnt;
        bool first_pv[2] = {true, true};
        int4 cur = P.steps[sb];
        int4 nxt = sb + 1 < se ? P.steps[sb + 1] : make_int4(0, -1, -1, 0);
        {  // the item's first stage: K of its first step
          const int stage = u_cnt % C::kStages;
          if (!(ok = mbar_wait(bar(C::kBStFull + stage), (u_cnt / C::kStages) & 1, ctl, 201)))
            break;
          if (cur.y >= 0) {
            issue_s(0, stage);
            mma_commit(bar(C::kBSFull + 0));
          }
          if (act1 && cur.z >= 0) {
            issue_s(1, stage);
            mma_commit(bar(C::kBSFull + 1));
          }
          mma_commit(bar(C::kBStEmpty + stage));  // every S of this step is issued
          ++u_cnt;
        }
        for (int j = sb; ok && j < se; ++j) {
          // the stage of V(j) and K(j + 1): one wait for both, released once
          // this step's P V and the next step's S are issued
          const int stage = u_cnt % C::kStages;
          const bool has_next = j + 1 < se;
          // step descriptors are read two steps ahead: the load of step j + 2
          // has a whole step to land
          const int4 nxt2 = j + 2 < se ? P.steps[j + 2] : make_int4(0, -1, -1, 0);
          if (!(ok = mbar_wait(bar(C::kBStFull + stage), (u_cnt / C::kStages) & 1, ctl, 214)))
            break;
          if (alt_items && has_next && (nxt.y >= 0 || nxt.z >= 0)) {
            // halves that take the steps in turn: the next step's S (the other
            // half's buffer, whose P went to PV a step ago) goes before this
            // step's PV, so one half's softmax runs while the other's does
            const int hn = nxt.y >= 0 ? 0 : 1;
            issue_s(hn, stage);
            mma_commit(bar(C::kBSFull + hn));
          }
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int info = h == 0 ? cur.y : (act1 ? cur.z : -1);
            if (info >= 0) {
              if (!(ok = mbar_wait(bar(C::kBPFull + h), p_cnt[h] & 1, ctl, 210 + h))) break;
              ++p_cnt[h];
              if (first_pv[h]) {
                if (!(ok = mbar_wait(bar(C::kBOEmpty + h), (oe_cnt[h] & 1) ^ 1, ctl, 212 + h)))
                  break;
                ++oe_cnt[h];
              }
              tc_fence_after();
              issue_pv(h, stage, !first_pv[h]);
              first_pv[h] = false;
            }
            const int ninfo = h == 0 ? nxt.y : (act1 ? nxt.z : -1);
            if (!alt_items && has_next && ninfo >= 0) {
              issue_s(h, stage);
              mma_commit(bar(C::kBSFull + h));
            }
          }
          if (!ok) break;
          mma_commit(bar(C::kBStEmpty + stage));  // V(j) and K(j + 1) read
          ++u_cnt;
          cur = nxt;
          nxt = nxt2;
        }
        if (!ok) break;
#pragma unroll
        for (int h = 0; h < 2; ++h)
          if (!first_pv[h]) mma_commit(bar(C::kBOFull + h));
        mma_commit(bar(C::kBQEmpty));
      }
      // Every MMA issued so far must finish before TMEM is released.
      mma_commit(bar(C::kBDrain));
      drain_wait(bar(C::kBDrain), 0, kDrainNs);
    }
  }
  } else {
    reg_alloc<kSplitWideRegs>();
    // ------------------------------------------------------------ softmax
    const int h = warp >> 2;
    const int row_in = threadIdx.x & 127;
    const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_addr + h * 128;
    const uint32_t tO = tmem + lane_addr + 256 + h * 128;
    const uint32_t tO1 = tmem + lane_addr + 256 + 128;  // half 1's O (alternating items)
    float2* hand = reinterpret_cast<float2*>(smem + C::kHandOff);
    const bool alt = kGather && P.alternate;
    uint32_t s_cnt = 0, o_cnt = 0, o1_cnt = 0, hand_cnt = 0, e_cnt = 0;
    const bool elected = kStage && row_in == 0;  // issues the half's output stores
    bool pending_read = false;
    if (elected) {
      prefetch_tmap(om.map());
      prefetch_tmap(om.map64());
    }
    bool ok = true;
    for (int r = 0; ok; ++r) {
      int idx = -1;
      const bool w = queue_take(queue, r, idx, ctl, 309);
      if (!(ok = __all_sync(0xffffffffu, w)) || idx < 0) break;
      const int* it = P.items + (size_t)idx * kFiWords;
      const int sb = it[kFiStepBeg], se = it[kFiStepEnd];
      const bool act1 = it[kFiQt1] >= 0 && it[kFiH1] >= 0;
      if (h == 1 && !act1) continue;
      const int qt = it[kFiQt0 + h], slot = it[kFiSlot];
      // tile row -> query row and head (head-stacked: R-row slab of 128 / R heads)
      const bool stk = kGather && P.stack;
      const int row = stk ? qt * P.stack + (row_in & (P.stack - 1)) : qt * 128 + row_in;
      const int head = it[kFiH0 + h] + (stk ? row_in / P.stack : 0);
      float m = -INFINITY, l = 0.f;
      bool visited = false, vis1 = false;  // vis1: half 1 had a step (alternating items)
      int4 st_next = sb < se ? P.steps[sb] : make_int4(0, -1, -1, 0);
      for (int j = sb; j < se; ++j) {
        const int4 st = st_next;
        if (j + 1 < se) st_next = P.steps[j + 1];  // prefetch the next step descriptor
        const int info = h == 0 ? st.y : st.z;
        vis1 |= st.z >= 0;
        if (info < 0) continue;
        // The column mask of a PARTIAL (or gathered) step depends on the plan
        // only: its reads overlap the wait for S.
        uint32_t vb[4] = {~0u, ~0u, ~0u, ~0u};
        if (info & 1) {
          if (kGather && st.w > 0)
            gather_mask(P.gathers + (size_t)(st.w - 1) * kGatherWords, h, row_in, P.Tk, vb);
          else
            step_mask<true>(info, P.slices, P.masks, row, st.x, vb);
        }
        const bool w = mbar_wait(bar(C::kBSFull + h), s_cnt & 1, ctl, 300 + h);
        if (!(ok = __all_sync(0xffffffffu, w))) break;
        ++s_cnt;
        tc_fence_after();
        uint32_t u[128];
        tmem_ld128(tS, u);
        float mn = INFINITY;
        if (kCap) {
          // Smallest raw score of the row, masked columns included: with the
          // masked maximum below it bounds every score the row sees.
          float mn0 = INFINITY, mn1 = INFINITY, mn2 = INFINITY, mn3 = INFINITY;
#pragma unroll
          for (int c = 0; c < 128; c += 8) {
            mn0 = fmin3(mn0, __uint_as_float(u[c]), __uint_as_float(u[c + 1]));
            mn1 = fmin3(mn1, __uint_as_float(u[c + 2]), __uint_as_float(u[c + 3]));
            mn2 = fmin3(mn2, __uint_as_float(u[c + 4]), __uint_as_float(u[c + 5]));
            mn3 = fmin3(mn3, __uint_as_float(u[c + 6]), __uint_as_float(u[c + 7]));
          }
          mn = fminf(fminf(mn0, mn1), fminf(mn2, mn3));
        }
        const bool lo_in_range = -mn <= P.cap.smax;
        if (info & 1) {
          // PARTIAL (or gathered) step: keep the keys this row sees.
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (!mask_bit(vb, c)) u[c] = 0xff800000u;  // -inf
        }
        // Row maximum: four independent chains of 3-input max.
        float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
        for (int c = 0; c < 128; c += 8) {
          mx0 = fmax3(mx0, __uint_as_float(u[c]), __uint_as_float(u[c + 1]));
          mx1 = fmax3(mx1, __uint_as_float(u[c + 2]), __uint_as_float(u[c + 3]));
          mx2 = fmax3(mx2, __uint_as_float(u[c + 4]), __uint_as_float(u[c + 5]));
          mx3 = fmax3(mx3, __uint_as_float(u[c + 6]), __uint_as_float(u[c + 7]));
        }
        const float mx = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
        // Softcap: the polynomial serves when every score of the warp's rows
        // lies in its range (a warp-uniform choice), else the exponential form.
        const bool poly = kCap && __all_sync(0xffffffffu, lo_in_range && mx <= P.cap.smax);
        const float m_cand = kCap ? (poly ? capped2_poly(mx, P.cap) : capped2(mx, P.cap))
                                  : mx * P.scale_log2;
        const bool raise = m_cand > m + kRescaleThreshold;
        const bool rescale_o = raise && visited && m > -INFINITY;
        const float alpha = raise ? exp2f(m - m_cand) : 1.f;
        if (__any_sync(0xffffffffu, rescale_o)) {
          const float a = rescale_o ? alpha : 1.f;
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + 32 * c, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * a);
            tmem_st32(tO + 32 * c, o);
          }
          tmem_st_wait();
        }
        if (raise) {
          l *= alpha;
          m = m_cand;
        }
        const float mu = m == -INFINITY ? 0.f : m;
        // p = 2^(x - m) two lanes at a time, four partial row sums; P (bf16
        // pairs) goes over S columns [0, 64): every S value is in registers.
        if (!kCap)
          l += exp_tile<kExpPlain>(u, tS, mu, P.scale_log2, P.cap, vb);
        else if (!poly)
          l += exp_tile<kExpCapExp>(u, tS, mu, P.scale_log2, P.cap, vb);
        else if (info & 1)
          l += exp_tile<kExpCapPolyMask>(u, tS, mu, P.scale_log2, P.cap, vb);
        else
          l += exp_tile<kExpCapPoly>(u, tS, mu, P.scale_log2, P.cap, vb);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(C::kBPFull + h));
        visited = true;
      }
      if (!ok) break;
      // ---- alternating item: half 1 hands its (m, l) to half 0, which merges
      // the two halves' states by logsumexp and writes the rows
      float a0 = 1.f, a1 = 0.f;
      if (alt) {
        if (h == 1) {
          const bool w = mbar_wait(bar(C::kBHandEmpty), (hand_cnt & 1) ^ 1, ctl, 320);
          if (!(ok = __all_sync(0xffffffffu, w))) break;
          ++hand_cnt;
          hand[row_in] = make_float2(m, l);
          mbar_arrive(bar(C::kBHandFull));
          continue;
        }
        const bool w = mbar_wait(bar(C::kBHandFull), hand_cnt & 1, ctl, 321);
        if (!(ok = __all_sync(0xffffffffu, w))) break;
        ++hand_cnt;
        const float2 st1 = hand[row_in];
        mbar_arrive(bar(C::kBHandEmpty));
        const float mm = fmaxf(visited ? m : -INFINITY, vis1 ? st1.x : -INFINITY);
        a0 = visited && mm > -INFINITY ? exp2f(m - mm) : 0.f;
        a1 = vis1 && mm > -INFINITY ? exp2f(st1.x - mm) : 0.f;
        l = a0 * l + a1 * st1.y;
        m = mm;
      }
      // ---- epilogue: O / l -> out (bf16) or a partial slot (fp32).  With
      // kStage the bf16 rows go through the half's staging chunk in shared
      // memory, 64 columns at a time, and leave by TMA stores (rows past Tq
      // are clipped by the tensor map); otherwise each thread stores its row
      // from registers (each warp store then touches 32 rows 4 KB and more
      // apart: slower per item, which only matters where items are short,
      // while the staging area takes 32 KB from the L1 cache).
      const bool nonempty = l > 0.f;
      float inv_l = nonempty ? 1.f / l : 0.f;
      // Row log2-normaliser: the keys', plus the sink's for an unsplit item
      // (split items leave the sink to the merge).
      float lse2 = nonempty ? m + log2f(l) : -INFINITY;
      if (P.n_sink > 0 && slot < 0 && row < P.Tq) {
        const float tot = log2_add(lse2, sink_log2(P.sink, P.n_sink, P.sink_layout, row, head, P.Hq));
        if (nonempty) inv_l *= exp2f(lse2 - tot);
        lse2 = tot;
      }
      if (visited) {
        const bool w = mbar_wait(bar(C::kBOFull + h), o_cnt & 1, ctl, 310 + h);
        if (!(ok = __all_sync(0xffffffffu, w))) break;
        ++o_cnt;
        tc_fence_after();
      }
      const bool read1 = alt && vis1;  // half 0 merges half 1's O
      if (read1) {
        const bool w = mbar_wait(bar(C::kBOFull + 1), o1_cnt & 1, ctl, 312);
        if (!(ok = __all_sync(0xffffffffu, w))) break;
        ++o1_cnt;
        tc_fence_after();
      }
      // O columns [32 cc, 32 cc + 32) of this row, unnormalised; the last
      // chunk's read hands O back to the MMA thread
      auto load_o = [&](int cc, uint32_t (&u)[32]) {
        if (visited) {
          tmem_ld32(tO + 32 * cc, u);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) u[i] = 0u;
        }
        if (read1) {
          uint32_t u1[32];
          tmem_ld32(tO1 + 32 * cc, u1);
#pragma unroll
          for (int i = 0; i < 32; ++i)
            u[i] = __float_as_uint(
                fmaf(a1, __uint_as_float(u1[i]), visited ? a0 * __uint_as_float(u[i]) : 0.f));
        }
        if (cc == D / 32 - 1) {
          tc_fence_before();
          if (visited) mbar_arrive(bar(C::kBOEmpty + h));
          if (read1) mbar_arrive(bar(C::kBOEmpty + 1));
        }
      };
      if constexpr (kStage) {
        if (slot < 0) {
          const uint32_t ebuf = sbase + C::kEpiOff + h * C::kEpiHalfBytes;
#pragma unroll 1
          for (int c = 0; c < D / 64; ++c) {
            if (elected && pending_read) {
              bulk_wait_read_all();
              mbar_arrive(epi_free(h));
              pending_read = false;
            }
            const bool w = mbar_wait(epi_free(h), (e_cnt & 1) ^ 1, ctl, 330 + h);
            if (!(ok = __all_sync(0xffffffffu, w))) break;
            uint32_t pk[32];
#pragma unroll
            for (int sub = 0; sub < 2; ++sub) {
              uint32_t u[32];
              load_o(2 * c + sub, u);
#pragma unroll
              for (int i = 0; i < 16; ++i)
                pk[16 * sub + i] = pack_bf16x2(__uint_as_float(u[2 * i]) * inv_l,
                                               __uint_as_float(u[2 * i + 1]) * inv_l);
            }
            // the 128-byte swizzle of the tensor map: 16-byte piece k of tile
            // row r sits at piece k ^ (r & 7) of the row's 128 bytes
#pragma unroll
            for (int k = 0; k < 8; ++k)
              st_shared_v4(ebuf + row_in * 128 + ((k ^ (row_in & 7)) << 4), pk[4 * k], pk[4 * k + 1],
                           pk[4 * k + 2], pk[4 * k + 3]);
            fence_proxy_async_smem();
            mbar_arrive(epi_full(h));
            if (elected) {
              ok = mbar_wait(epi_full(h), e_cnt & 1, ctl, 332 + h);
              if (ok) {
                const int h0 = it[kFiH0 + h];
                if (stk) {  // tile rows [R j, R j + R): slab qt of head h0 + j
                  const int R = P.stack;
                  for (int j = 0; j < 128 / R; ++j)
                    tma_store_2d(om.map64(), ebuf + j * (R * 128), (h0 + j) * D + 64 * c, qt * R);
                } else {
                  tma_store_2d(om.map(), ebuf, h0 * D + 64 * c, qt * 128);
                }
                bulk_commit_group();
                if (c + 1 < D / 64) {
                  bulk_wait_read_all();
                  mbar_arrive(epi_free(h));
                } else {
                  pending_read = true;  // waited for at the next use of the buffer
                }
              }
            }
            ++e_cnt;
            if (!(ok = __all_sync(0xffffffffu, ok))) break;
          }
          if (!ok) break;
        } else {
          const size_t pbase = ((size_t)slot * 2 + h) * 128 + row_in;
          float4* dst_f = reinterpret_cast<float4*>(P.part_o + pbase * D);
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t u[32];
            load_o(c, u);
#pragma unroll
            for (int v = 0; v < 8; ++v)
              dst_f[8 * c + v] = make_float4(
                  __uint_as_float(u[4 * v]) * inv_l, __uint_as_float(u[4 * v + 1]) * inv_l,
                  __uint_as_float(u[4 * v + 2]) * inv_l, __uint_as_float(u[4 * v + 3]) * inv_l);
          }
        }
      } else {
        const bool store = slot >= 0 || row < P.Tq;
        const size_t pbase = slot >= 0 ? ((size_t)slot * 2 + h) * 128 + row_in : 0;
        uint4* dst_b = reinterpret_cast<uint4*>(P.out + ((size_t)row * P.Hq + head) * D);
        float4* dst_f = slot >= 0 ? reinterpret_cast<float4*>(P.part_o + pbase * D) : nullptr;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t u[32];
          if (visited) {
            tmem_ld32(tO + 32 * c, u);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) u[i] = 0u;
          }
          if (read1) {
            uint32_t u1[32];
            tmem_ld32(tO1 + 32 * c, u1);
#pragma unroll
            for (int i = 0; i < 32; ++i)
              u[i] = __float_as_uint(
                  fmaf(a1, __uint_as_float(u1[i]), visited ? a0 * __uint_as_float(u[i]) : 0.f));
          }
          if (c == D / 32 - 1) {
            tc_fence_before();
            if (visited) mbar_arrive(bar(C::kBOEmpty + h));
            if (read1) mbar_arrive(bar(C::kBOEmpty + 1));
          }
          if (!store) continue;
          if (slot < 0) {
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst_b[4 * c + v] = make_uint4(
                  pack_bf16x2(__uint_as_float(u[8 * v]) * inv_l, __uint_as_float(u[8 * v + 1]) * inv_l),
                  pack_bf16x2(__uint_as_float(u[8 * v + 2]) * inv_l, __uint_as_float(u[8 * v + 3]) * inv_l),
                  pack_bf16x2(__uint_as_float(u[8 * v + 4]) * inv_l, __uint_as_float(u[8 * v + 5]) * inv_l),
                  pack_bf16x2(__uint_as_float(u[8 * v + 6]) * inv_l, __uint_as_float(u[8 * v + 7]) * inv_l));
          } else {
#pragma unroll
            for (int v = 0; v < 8; ++v)
              dst_f[8 * c + v] = make_float4(
                  __uint_as_float(u[4 * v]) * inv_l, __uint_as_float(u[4 * v + 1]) * inv_l,
                  __uint_as_float(u[4 * v + 2]) * inv_l, __uint_as_float(u[4 * v + 3]) * inv_l);
          }
        }
      }
      if (slot < 0) {
        if (row < P.Tq) P.lse[(size_t)head * P.Tq + row] = lse2 * kLn2;
      } else {
        P.part_lse[((size_t)slot * 2 + h) * 128 + row_in] = lse2;
      }
    }
    // the output stores must complete before the CTA's shared memory goes
    if (elected) bulk_wait_all();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Logsumexp merge of split items: one block per (group, half), one thread per row.
template <int D>
__global__ void __launch_bounds__(128)
    ffa_merge_kernel(const int* __restrict__ merges, const float* __restrict__ part_o,
                     const float* __restrict__ part_lse, int Tq, int Hq,
                     __nv_bfloat16* __restrict__ out, float* __restrict__ lse,
                     const float* __restrict__ sink, int n_sink, int sink_layout) {
  const int grp = blockIdx.x >> 1, h = blockIdx.x & 1;
  const int* mg = merges + (size_t)grp * kMgWords;
  const int qt = mg[kMgQt0 + h], head = mg[kMgH0 + h];
  if (qt < 0 || head < 0) return;
  const int row_in = threadIdx.x, row = qt * 128 + row_in;
  if (row >= Tq) return;
  const int s0 = mg[kMgSlotBeg], ns = mg[kMgSlots];
  float mx = -INFINITY;
  for (int s = 0; s < ns; ++s)
    mx = fmaxf(mx, part_lse[((size_t)(s0 + s) * 2 + h) * 128 + row_in]);
  float acc[D];
#pragma unroll
  for (int d = 0; d < D; ++d) acc[d] = 0.f;
  float wsum = 0.f;
  if (mx > -INFINITY) {
    for (int s = 0; s < ns; ++s) {
      const size_t base = ((size_t)(s0 + s) * 2 + h) * 128 + row_in;
      const float w = exp2f(part_lse[base] - mx);
      wsum += w;
      const float4* src = reinterpret_cast<const float4*>(part_o + base * D);
#pragma unroll
      for (int v = 0; v < D / 4; ++v) {
        const float4 x = src[v];
        acc[4 * v] += w * x.x;
        acc[4 * v + 1] += w * x.y;
        acc[4 * v + 2] += w * x.z;
        acc[4 * v + 3] += w * x.w;
      }
    }
  }
  float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  float lse2 = wsum > 0.f ? mx + log2f(wsum) : -INFINITY;
  if (n_sink > 0) {  // the sink joins the merged normaliser once
    const float tot = log2_add(lse2, sink_log2(sink, n_sink, sink_layout, row, head, Hq));
    if (wsum > 0.f) inv *= exp2f(lse2 - tot);
    lse2 = tot;
  }
  uint4* dst = reinterpret_cast<uint4*>(out + ((size_t)row * Hq + head) * D);
#pragma unroll
  for (int v = 0; v < D / 8; ++v) {
    uint4 w;
    w.x = pack_bf16x2(acc[8 * v + 0] * inv, acc[8 * v + 1] * inv);
    w.y = pack_bf16x2(acc[8 * v + 2] * inv, acc[8 * v + 3] * inv);
    w.z = pack_bf16x2(acc[8 * v + 4] * inv, acc[8 * v + 5] * inv);
    w.w = pack_bf16x2(acc[8 * v + 6] * inv, acc[8 * v + 7] * inv);
    dst[v] = w;
  }
  lse[(size_t)head * Tq + row] = lse2 * kLn2;
}

template <int D, bool kCap, bool kGather, bool kStage>
ffa_status_t launch_fwd_d(ffa_plan_s* p, const void* q, const void* k, const void* v, float scale,
                          void* out, float* lse, void* ws, cudaStream_t st, const SinkArgs& sk,
                          float softcap) {
  using C = FwdCfg<D>;
  alignas(64) CUtensorMap tq, tk, tv, tk8, tv8, tq64;
  OutMapsT<kStage> om;
  if (!encode_tile_map(&tq, q, p->Tq, p->Hq * D) || !encode_tile_map(&tk, k, p->Tk, p->Hkv * D) ||
      !encode_tile_map(&tv, v, p->Tk, p->Hkv * D) ||
      !encode_tile_map(&tk8, k, p->Tk, p->Hkv * D, kGatherKeys) ||
      !encode_tile_map(&tv8, v, p->Tk, p->Hkv * D, kGatherKeys) ||
      !encode_tile_map(&tq64, q, p->Tq, p->Hq * D, p->stacked ? p->stacked : kSlabRows))
    return FFA_ERR_INVALID_ARG;
  if constexpr (kStage) {
    if (!encode_tile_map(&om.o, out, p->Tq, p->Hq * D) ||
        !encode_tile_map(&om.o64, out, p->Tq, p->Hq * D, p->stacked ? p->stacked : kSlabRows))
      return FFA_ERR_INVALID_ARG;
  }
  FwdParams P;
  P.steps = p->fwd_steps;
  P.items = p->fwd_items;
  P.order = p->fwd_order;
  P.ticket = p->tickets;
  P.n_items = (int)p->n_fwd_items;
  P.slices = p->slices;
  P.masks = p->fwd_masks;
  P.gathers = p->gathers;
  P.Tq = p->Tq;
  P.Tk = p->Tk;
  P.Hq = p->Hq;
  P.g = p->Hq / p->Hkv;
  P.stack = p->stacked;
  P.alternate = p->alternate;
  const int smem = kStage ? C::kSmemBytesStaged : C::kSmemBytes;
  P.scale_log2 = scale * kLog2e;
  P.out = static_cast<__nv_bfloat16*>(out);
  P.lse = lse;
  P.part_o = static_cast<float*>(ws);
  P.part_lse = P.part_o ? P.part_o + (size_t)p->n_slots * 2 * 128 * D : nullptr;
  P.err = p->err;
  P.wait_ns = p->wait_ns;
  P.sink = sk.sink;
  P.n_sink = sk.n;
  P.sink_layout = sk.layout;
  if (kCap) P.cap = make_cap_consts(scale, softcap);
  if (cudaFuncSetAttribute(ffa_fwd_kernel<D, kCap, kGather, kStage>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return FFA_ERR_CUDA;
  if (!split_regs_ok<ffa_fwd_kernel<D, kCap, kGather, kStage>>()) return FFA_ERR_UNSUPPORTED;
  if (cudaMemsetAsync(P.ticket, 0, sizeof(int), st) != cudaSuccess) return FFA_ERR_CUDA;
  record_phase(p, 0, st);
  ffa_fwd_kernel<D, kCap, kGather, kStage><<<p->grid_fwd, kFwdThreads, smem, st>>>(
      tq, tk, tv, tk8, tv8, tq64, P, om);
  note_launches(1);
  if (cudaGetLastError() != cudaSuccess) return FFA_ERR_CUDA;
  if (p->n_merges > 0) {
    ffa_merge_kernel<D><<<(int)(2 * p->n_merges), 128, 0, st>>>(
        p->merges, P.part_o, P.part_lse, p->Tq, p->Hq, P.out, lse, sk.sink, sk.n, sk.layout);
    note_launches(1);
    if (cudaGetLastError() != cudaSuccess) return FFA_ERR_CUDA;
  }
  record_phase(p, 1, st);
  return FFA_OK;
}

}  // namespace

size_t fwd_workspace_bytes(const ffa_plan_s* p) {
  return (size_t)p->n_slots * 2 * 128 * (p->D + 1) * sizeof(float);
}

ffa_status_t launch_fwd(ffa_plan_s* p, const void* q, const void* k, const void* v, float scale,
                        void* out, float* lse, void* ws, size_t, cudaStream_t st,
                        const SinkArgs& sink, float softcap) {
  const bool cap = softcap > 0.f, g = p->n_gathers > 0;
  // Staged output where the items average at most 16 steps of 128 x 128
  // visible pairs (visible pairs x query heads over items x two halves of
  // 128 x 128; this follows the steps the items run within 5% on long
  // items): the epilogue is then a large share of an item (GB300: forward
  // 2-5% faster on short documents and small blocks), while on longer items
  // the 32 KB of staging taken from the L1 cache costs more than it saves.
  // Capped plans keep the direct stores (no staged instantiation).
  const bool stage = !cap && p->area * p->Hq <= 16LL * 2 * 128 * 128 * p->n_fwd_items;
#define FFA_FWD(DD, CC, GG, SS) \
  launch_fwd_d<DD, CC, GG, SS>(p, q, k, v, scale, out, lse, ws, st, sink, softcap)
  if (p->D == 128) {
    if (cap) return g ? FFA_FWD(128, true, true, false) : FFA_FWD(128, true, false, false);
    if (stage) return g ? FFA_FWD(128, false, true, true) : FFA_FWD(128, false, false, true);
    return g ? FFA_FWD(128, false, true, false) : FFA_FWD(128, false, false, false);
  }
  if (p->D == 64) {
    if (cap) return g ? FFA_FWD(64, true, true, false) : FFA_FWD(64, true, false, false);
    if (stage) return g ? FFA_FWD(64, false, true, true) : FFA_FWD(64, false, false, true);
    return g ? FFA_FWD(64, false, true, false) : FFA_FWD(64, false, false, false);
  }
#undef FFA_FWD
  return FFA_ERR_UNSUPPORTED;
}

}  // namespace ffa
