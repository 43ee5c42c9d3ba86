// Backward kernels of flexible-mask attention for sm_103a.
//
//   1. preprocess: -delta[h][q] = -<dO, O> (fp32), -lse * log2(e), and
//      dQaccum = 0 (stored negated so the main kernel adds them with FMAs);
//   2. main: one work item per (k-tile, kv head).  The 128 x D tiles of K and
//      V stay in shared memory; the item loops over every (q-tile, query head
//      of the group) that sees the k-tile:
//          S^T  = K Q^T           (tcgen05, SS)      -> TMEM
//          dP^T = V dO^T          (tcgen05, SS)      -> TMEM
//          P^T  = 2^(S^T*scale*log2e - lse2), masked on PARTIAL steps
//          dS^T = P^T * (dP^T - delta)
//          dV  += P^T dO          (tcgen05, A = P^T from TMEM)
//          dK  += dS^T Q          (tcgen05, A = dS^T from TMEM)
//          dQ^T = K^T dS^T        (tcgen05, both operands from shared memory;
//                                  dQ = dS K when D = 64)
//      dK and dV accumulate in TMEM and are written once per item (no
//      atomics); each dQ tile is added into the fp32 dQaccum.
//   3. convert: dq = bf16(dQaccum).
// This is the standard softmax-attention gradient; the mask only decides
// which entries of P are zero.
//
// Warp roles of the main kernel (320 threads):
//   warps 0-3  P/dS warps (thread = key = TMEM lane), dK/dV epilogue
//   warps 4-7  dQ warps (thread = query row = TMEM lane): TMEM -> fp32 atomics
//   warp  8    TMA producer (K, V per item; Q, dO two-stage rings)
//   warp  9    MMA issuer, TMEM owner
// TMEM columns: dV [0,D), dK [D,2D), S^T [2D,2D+128), dP^T [2D+128,2D+256);
// the dQ tile reuses the S^T columns once P^T has been consumed.
#include <cuda_bf16.h>
#include <math.h>

#include <mutex>

#include "ffa_internal.cuh"
#include "ffa_ptx.cuh"

namespace ffa {
namespace {

constexpr int kBwdThreads = 320;
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct BwdCfg {
  static constexpr int kChunks = D / 64;
  static constexpr int kTileBytes = 128 * D * 2;
  static constexpr int kStages = 2;
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kTileBytes;
  static constexpr int kQOff = 2 * kTileBytes;
  static constexpr int kDOOff = kQOff + kStages * kTileBytes;
  static constexpr int kDSOff = kDOOff + kStages * kTileBytes;  // 128 x 128 bf16
  static constexpr int kLseOff = kDSOff + 128 * 128 * 2;         // per stage: -lse2[128], -delta[128]
  static constexpr int kLseStageBytes = 2 * 128 * 4;
  static constexpr int kBarOff = kLseOff + kStages * kLseStageBytes;
  static constexpr int kBKVFull = 0, kBKVEmpty = 1, kBQFull = 2, kBQEmpty = 2 + kStages,
                       kBDOFull = 2 + 2 * kStages, kBDOEmpty = 2 + 3 * kStages,
                       kBSdpFull = 2 + 4 * kStages, kBPFull = kBSdpFull + 1,
                       kBDqFull = kBPFull + 1, kBDqFree = kBDqFull + 1, kBDkvFull = kBDqFree + 1,
                       kBDkvEmpty = kBDkvFull + 1, kBDrain = kBDkvEmpty + 1,
                       kNumBars = kBDrain + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  // The dynamic shared memory base must be 1024-byte aligned (checked on entry).
  static constexpr int kSmemBytes = kMiscOff + 64;
  // TMEM columns
  static constexpr int kTdV = 0, kTdK = D, kTS = 2 * D, kTdP = 2 * D + 128;
};

struct BwdParams {
  const int4* steps;
  const int* items;
  const int* order;
  int n_items;
  const Slice* slices;
  int Tq, Tk, Hq, g, qpad;
  float scale, scale_log2;
  const float* nlse2;   // [Hq][qpad] -lse * log2(e)
  const float* ndelta;  // [Hq][qpad] -rowsum(dO * O)
  float* dq_acc;       // [Tq][Hq][D]
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int* err;
  uint64_t wait_ns;
};

__device__ __forceinline__ bool bwd_item_at(const BwdParams& P, int r, const int*& it) {
  const int G = gridDim.x, b = blockIdx.x;
  const int pos = r * G + ((r & 1) ? (G - 1 - b) : b);
  if (pos >= P.n_items) return false;
  it = P.items + (size_t)P.order[pos] * kBiWords;
  return true;
}

__device__ __forceinline__ void drain_wait_b(uint32_t bar, uint32_t parity, uint64_t ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_test(bar, parity)) {
    if (globaltimer_ns() - t0 > ns) return;
  }
}

// Query rows of this step visible to key `key` under a PARTIAL step's slice,
// in local coordinates [lo, hi) of the q-tile.
__device__ __forceinline__ void key_query_window(const Slice& sl, int key, int qt, int& lo,
                                                 int& hi) {
  lo = hi = 0;
  if (key < sl.ks || key >= sl.ke) return;
  int a = (sl.t & 1) ? key + sl.qe - sl.ke : sl.qs;
  a = a > sl.qs ? a : sl.qs;
  int b = (sl.t & 2) ? key - sl.ks + sl.qs + 1 : sl.qe;
  b = b < sl.qe ? b : sl.qe;
  lo = a - qt * 128;
  hi = b - qt * 128;
}

// P^T and dS^T for one key row j over the 128 queries of the step:
//   p = 2^(s * scale * log2e - lse2), ds = p * (dp - delta)
// written as bf16 pairs to TMEM (over the first 64 columns of S^T and dP^T)
// and dS to the 128-byte swizzled shared-memory tile (row j, query chunks).
template <bool kPartial>
__device__ __forceinline__ void pds_tile(uint32_t tS, uint32_t tP, const float* nl,
                                         const float* nd, float scale_log2, int lo, int hi, int j,
                                         uint8_t* ds_row) {
  const float2 sc2 = make_float2(scale_log2, scale_log2);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t r[64];  // r[0..32): S^T, r[32..64): dP^T
    tmem_ld32x2(tS + 32 * c, tP + 32 * c, r);
    uint32_t pp[16], dd[16];
#pragma unroll
    for (int e = 0; e < 32; e += 4) {
      const float4 l4 = *reinterpret_cast<const float4*>(nl + 32 * c + e);
      const float4 d4 = *reinterpret_cast<const float4*>(nd + 32 * c + e);
#pragma unroll
      for (int u = 0; u < 4; u += 2) {
        const int col = 32 * c + e + u;
        const float2 nlp = u == 0 ? make_float2(l4.x, l4.y) : make_float2(l4.z, l4.w);
        const float2 ndp = u == 0 ? make_float2(d4.x, d4.y) : make_float2(d4.z, d4.w);
        const float2 x = __ffma2_rn(
            make_float2(__uint_as_float(r[e + u]), __uint_as_float(r[e + u + 1])), sc2, nlp);
        float2 p = make_float2(ex2_approx(x.x), ex2_approx(x.y));
        if (kPartial) {
          p.x = (col >= lo && col < hi) ? p.x : 0.f;
          p.y = (col + 1 >= lo && col + 1 < hi) ? p.y : 0.f;
        }
        const float2 dpd = __fadd2_rn(
            make_float2(__uint_as_float(r[32 + e + u]), __uint_as_float(r[32 + e + u + 1])), ndp);
        const float2 ds = __fmul2_rn(p, dpd);
        pp[(e + u) >> 1] = pack_bf16x2(p.x, p.y);
        dd[(e + u) >> 1] = pack_bf16x2(ds.x, ds.y);
      }
    }
    tmem_st16(tS + 16 * c, pp);
    tmem_st16(tP + 16 * c, dd);
    // dS row j, queries [32c, 32c+32): four 16-byte units of the swizzled row
    // of query chunk c/2.
    uint8_t* base = ds_row + (c >> 1) * 16384;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int unit = (c & 1) * 4 + u;
      *reinterpret_cast<uint4*>(base + ((unit ^ (j & 7)) << 4)) =
          make_uint4(dd[4 * u], dd[4 * u + 1], dd[4 * u + 2], dd[4 * u + 3]);
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    ffa_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                   const BwdParams P) {
  using C = BwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  if ((smem_u32(smem) & 1023u) != 0) {
    // The swizzled tile layout needs a 1024-byte aligned base; refuse to run.
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
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar(C::kBQFull + s), 1);
      mbar_init(bar(C::kBQEmpty + s), 1);
      mbar_init(bar(C::kBDOFull + s), 1);
      mbar_init(bar(C::kBDOEmpty + s), 1);
    }
    mbar_init(bar(C::kBSdpFull), 1);
    mbar_init(bar(C::kBPFull), 128);
    mbar_init(bar(C::kBDqFull), 1);
    mbar_init(bar(C::kBDqFree), 128);
    mbar_init(bar(C::kBDkvFull), 1);
    mbar_init(bar(C::kBDkvEmpty), 128);
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

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      prefetch_tmap(&tm_do);
      uint32_t kv_cnt = 0, q_cnt = 0;
      bool ok = true, q_only = false;  // q_only: Q of iteration q_cnt issued, its dO not yet
      const int* it;
      for (int r = 0; ok && bwd_item_at(P, r, it); ++r) {
        const int sb = it[kBiStepBeg], se = it[kBiStepEnd];
        if (se <= sb) continue;
        const int kt = it[kBiKt], hk = it[kBiHkv];
        if (!(ok = mbar_wait(bar(C::kBKVEmpty), (kv_cnt & 1) ^ 1, ctl, 400))) break;
        mbar_arrive_expect_tx(bar(C::kBKVFull), 2 * C::kTileBytes);
        for (int c = 0; c < C::kChunks; ++c) {
          tma_load_2d(sbase + C::kKOff + c * 16384, &tm_k, bar(C::kBKVFull), hk * D + c * 64,
                      kt * 128);
          tma_load_2d(sbase + C::kVOff + c * 16384, &tm_v, bar(C::kBKVFull), hk * D + c * 64,
                      kt * 128);
        }
        ++kv_cnt;
        const int n_it = (se - sb) * g;
        for (int i = 0; i < n_it; ++i) {
          const int qt = P.steps[sb + i / g].x;
          const int h = hk * g + i % g;
          const int stage = q_cnt % C::kStages;
          const uint32_t ph = (q_cnt / C::kStages) & 1;
          if (!(ok = mbar_wait(bar(C::kBQEmpty + stage), ph ^ 1, ctl, 401))) break;
          mbar_arrive_expect_tx(bar(C::kBQFull + stage), C::kTileBytes + C::kLseStageBytes);
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_2d(sbase + C::kQOff + stage * C::kTileBytes + c * 16384, &tm_q,
                        bar(C::kBQFull + stage), h * D + c * 64, qt * 128);
          const uint32_t ls = sbase + C::kLseOff + stage * C::kLseStageBytes;
          bulk_load(ls, P.nlse2 + (size_t)h * P.qpad + qt * 128, 512, bar(C::kBQFull + stage));
          bulk_load(ls + 512, P.ndelta + (size_t)h * P.qpad + qt * 128, 512,
                    bar(C::kBQFull + stage));
          q_only = true;
          if (!(ok = mbar_wait(bar(C::kBDOEmpty + stage), ph ^ 1, ctl, 402))) break;
          q_only = false;
          mbar_arrive_expect_tx(bar(C::kBDOFull + stage), C::kTileBytes);
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_2d(sbase + C::kDOOff + stage * C::kTileBytes + c * 16384, &tm_do,
                        bar(C::kBDOFull + stage), h * D + c * 64, qt * 128);
          ++q_cnt;
        }
      }
      if (!ok) {
        if (kv_cnt > 0) drain_wait_b(bar(C::kBKVFull), (kv_cnt - 1) & 1, kDrainNs);
        for (uint32_t i = q_cnt > (uint32_t)C::kStages ? q_cnt - C::kStages : 0; i < q_cnt; ++i) {
          drain_wait_b(bar(C::kBQFull + i % C::kStages), (i / C::kStages) & 1, kDrainNs);
          drain_wait_b(bar(C::kBDOFull + i % C::kStages), (i / C::kStages) & 1, kDrainNs);
        }
        if (q_only)
          drain_wait_b(bar(C::kBQFull + q_cnt % C::kStages), (q_cnt / C::kStages) & 1, kDrainNs);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16(128, 128, false, false);
      constexpr uint32_t kIdAcc = idesc_bf16(128, D, false, true);   // A from TMEM, B MN-major
      constexpr uint32_t kIdDq = idesc_bf16(128, D == 128 ? 128 : D, true, true);  // both MN-major
      const uint32_t kA = sbase + C::kKOff, vA = sbase + C::kVOff, dsA = sbase + C::kDSOff;
      uint32_t kv_cnt = 0, q_cnt = 0, p_cnt = 0, dqf_cnt = 0, dkv_cnt = 0;
      bool ok = true, dq_pending = false;
      const int* it;
      for (int r = 0; ok && bwd_item_at(P, r, it); ++r) {
        const int sb = it[kBiStepBeg], se = it[kBiStepEnd];
        if (se <= sb) continue;
        if (!(ok = mbar_wait(bar(C::kBKVFull), kv_cnt & 1, ctl, 500))) break;
        ++kv_cnt;
        const int n_it = (se - sb) * g;
        for (int i = 0; i < n_it; ++i) {
          const int stage = q_cnt % C::kStages;
          const uint32_t ph = (q_cnt / C::kStages) & 1;
          const uint32_t qA = sbase + C::kQOff + stage * C::kTileBytes;
          const uint32_t doA = sbase + C::kDOOff + stage * C::kTileBytes;
          if (!(ok = mbar_wait(bar(C::kBQFull + stage), ph, ctl, 501))) break;
          if (!(ok = mbar_wait(bar(C::kBDOFull + stage), ph, ctl, 502))) break;
          tc_fence_after();
          // dP^T = V dO^T first: its columns were freed by the previous dK MMA.
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
            mma_ss(tmem + C::kTdP, sdesc_sw128(vA + off, 16, 1024), sdesc_sw128(doA + off, 16, 1024),
                   kIdS, kk > 0 ? 1u : 0u);
          }
          // S^T = K Q^T reuses the previous dQ tile's columns.
          if (dq_pending) {
            if (!(ok = mbar_wait(bar(C::kBDqFree), dqf_cnt & 1, ctl, 503))) break;
            ++dqf_cnt;
            tc_fence_after();
          }
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
            mma_ss(tmem + C::kTS, sdesc_sw128(kA + off, 16, 1024), sdesc_sw128(qA + off, 16, 1024),
                   kIdS, kk > 0 ? 1u : 0u);
          }
          mma_commit(bar(C::kBSdpFull));
          if (!(ok = mbar_wait(bar(C::kBPFull), p_cnt & 1, ctl, 504))) break;
          ++p_cnt;
          tc_fence_after();
          if (i == 0) {
            if (!(ok = mbar_wait(bar(C::kBDkvEmpty), (dkv_cnt & 1) ^ 1, ctl, 505))) break;
            ++dkv_cnt;
            tc_fence_after();
          }
          const uint32_t acc0 = i > 0 ? 1u : 0u;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            mma_ts(tmem + C::kTdV, tmem + C::kTS + kk * 8, sdesc_sw128(doA + kk * 2048, 16384, 1024),
                   kIdAcc, (acc0 || kk > 0) ? 1u : 0u);
            mma_ts(tmem + C::kTdK, tmem + C::kTdP + kk * 8, sdesc_sw128(qA + kk * 2048, 16384, 1024),
                   kIdAcc, (acc0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(bar(C::kBDOEmpty + stage));
          mma_commit(bar(C::kBQEmpty + stage));
          if constexpr (D == 128) {
            // dQ^T = K^T dS^T: lanes = head dim, columns = queries, so the dQ
            // warps reduce whole 128-byte row segments.
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ss(tmem + C::kTS, sdesc_sw128(kA + kk * 2048, 16384, 1024),
                     sdesc_sw128(dsA + kk * 2048, 16384, 1024), kIdDq, kk > 0 ? 1u : 0u);
          } else {
            // dQ = dS K: lanes = queries.
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ss(tmem + C::kTS, sdesc_sw128(dsA + kk * 2048, 16384, 1024),
                     sdesc_sw128(kA + kk * 2048, 16384, 1024), kIdDq, kk > 0 ? 1u : 0u);
          }
          mma_commit(bar(C::kBDqFull));
          dq_pending = true;
          ++q_cnt;
        }
        if (!ok) break;
        mma_commit(bar(C::kBDkvFull));
        mma_commit(bar(C::kBKVEmpty));
      }
      mma_commit(bar(C::kBDrain));
      drain_wait_b(bar(C::kBDrain), 0, kDrainNs);
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ P / dS warps
    const int j = threadIdx.x;  // key lane
    const uint32_t lane_addr = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tS = tmem + lane_addr + C::kTS;
    const uint32_t tP = tmem + lane_addr + C::kTdP;
    uint8_t* ds_row = smem + C::kDSOff + j * 128;
    uint32_t sdp_cnt = 0, dkv_cnt = 0;
    bool ok = true;
    const int* it;
    for (int r = 0; ok && bwd_item_at(P, r, it); ++r) {
      const int sb = it[kBiStepBeg], se = it[kBiStepEnd];
      const int kt = it[kBiKt], hk = it[kBiHkv];
      const int key = kt * 128 + j;
      const int n_it = (se - sb) * g;
      for (int i = 0; i < n_it; ++i) {
        const int4 st = P.steps[sb + i / g];
        const int qt = st.x, info = st.y;
        const int h = hk * g + i % g;
        int lo = 0, hi = 128;
        if (info & 1) key_query_window(P.slices[info >> 1], key, qt, lo, hi);
        const float* nl = reinterpret_cast<const float*>(smem + C::kLseOff +
                                                         (sdp_cnt % C::kStages) * C::kLseStageBytes);
        const float* nd = nl + 128;
        bool w = mbar_wait(bar(C::kBSdpFull), sdp_cnt & 1, ctl, 600);
        if (!(ok = __all_sync(0xffffffffu, w))) break;
        ++sdp_cnt;
        tc_fence_after();
        if (info & 1) pds_tile<true>(tS, tP, nl, nd, P.scale_log2, lo, hi, j, ds_row);
        else pds_tile<false>(tS, tP, nl, nd, P.scale_log2, 0, 128, j, ds_row);
        tmem_st_wait();
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(C::kBPFull));
      }
      if (!ok) break;
      // ---- dK / dV epilogue (written once per item; zeros when no query sees the tile)
      uint4* pv = reinterpret_cast<uint4*>(P.dv + ((size_t)key * (P.Hq / g) + hk) * D);
      uint4* pk = reinterpret_cast<uint4*>(P.dk + ((size_t)key * (P.Hq / g) + hk) * D);
      const bool store = key < P.Tk;
      if (n_it > 0) {
        bool w = mbar_wait(bar(C::kBDkvFull), dkv_cnt & 1, ctl, 610);
        if (!(ok = __all_sync(0xffffffffu, w))) break;
        ++dkv_cnt;
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < 2 * (D / 32); ++c) {
          const bool is_k = c >= D / 32;
          const int cc = is_k ? c - D / 32 : c;
          uint32_t u[32];
          tmem_ld32(tmem + lane_addr + (is_k ? C::kTdK : C::kTdV) + 32 * cc, u);
          if (c == 2 * (D / 32) - 1) {
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
        for (int v = 0; v < D / 8; ++v) pv[v] = pk[v] = make_uint4(0, 0, 0, 0);
      }
    }
  } else {
    // ------------------------------------------------------------ dQ warps
    const int t = threadIdx.x - 128;  // TMEM lane: head-dim index (D = 128) or query row
    const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
    uint32_t dq_cnt = 0;
    bool ok = true;
    const int* it;
    for (int r = 0; ok && bwd_item_at(P, r, it); ++r) {
      const int sb = it[kBiStepBeg], se = it[kBiStepEnd];
      const int hk = it[kBiHkv];
      const int n_it = (se - sb) * g;
      for (int i = 0; i < n_it; ++i) {
        const int4 st = P.steps[sb + i / g];
        const int qt = st.x, info = st.y;
        const int h = hk * g + i % g;
        // rows of this q-tile that can receive a non-zero dQ
        int q_lo = qt * 128, q_hi = min(P.Tq, qt * 128 + 128);
        if (info & 1) {
          const Slice sl = P.slices[info >> 1];
          q_lo = max(q_lo, sl.qs);
          q_hi = min(q_hi, sl.qe);
        }
        bool w = mbar_wait(bar(C::kBDqFull), dq_cnt & 1, ctl, 700);
        if (!(ok = __all_sync(0xffffffffu, w))) break;
        ++dq_cnt;
        tc_fence_after();
        if constexpr (D == 128) {
          // lane t = head-dim index; columns = queries of the tile.  Read the
          // whole tile, hand the columns back to the MMA warp, then reduce.
          uint32_t u[128];
          tmem_ld128(tmem + lane_addr + C::kTS, u);
          tc_fence_before();
          mbar_arrive(bar(C::kBDqFree));
          float* col = P.dq_acc + ((size_t)qt * 128 * P.Hq + h) * D + t;
          const size_t row_stride = (size_t)P.Hq * D;
#pragma unroll
          for (int e = 0; e < 128; ++e) {
            const int q = qt * 128 + e;
            if (q >= q_lo && q < q_hi)
              red_add_f32(col + (size_t)e * row_stride, __uint_as_float(u[e]) * P.scale);
          }
        } else {
          // lane t = query row; columns = head dim
          const int q = qt * 128 + t;
          const bool add = q >= q_lo && q < q_hi;
          float* dst = P.dq_acc + ((size_t)q * P.Hq + h) * D;
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t u[32];
            tmem_ld32(tmem + lane_addr + C::kTS + 32 * c, u);
            if (c == D / 32 - 1) {
              tc_fence_before();
              mbar_arrive(bar(C::kBDqFree));
            }
            if (add) {
#pragma unroll
              for (int v = 0; v < 8; ++v)
                red_add_v4(dst + 32 * c + 4 * v, __uint_as_float(u[4 * v]) * P.scale,
                           __uint_as_float(u[4 * v + 1]) * P.scale,
                           __uint_as_float(u[4 * v + 2]) * P.scale,
                           __uint_as_float(u[4 * v + 3]) * P.scale);
            }
          }
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

// -delta = -rowsum(dO * O), -lse2 = -lse * log2(e) (padded rows: 0), dQaccum = 0.
template <int D>
__global__ void ffa_bwd_pre_kernel(const __nv_bfloat16* __restrict__ out,
                                   const __nv_bfloat16* __restrict__ dout,
                                   const float* __restrict__ lse, int Tq, int Hq, int qpad,
                                   float* __restrict__ lse2, float* __restrict__ delta,
                                   float* __restrict__ dq_acc) {
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;  // (q, h)
  if (idx >= (long long)qpad * Hq) return;
  const int q = (int)(idx / Hq), h = (int)(idx % Hq);
  float dsum = 0.f, l2 = 0.f;
  if (q < Tq) {
    const uint4* o4 = reinterpret_cast<const uint4*>(out + ((size_t)q * Hq + h) * D);
    const uint4* d4 = reinterpret_cast<const uint4*>(dout + ((size_t)q * Hq + h) * D);
    float4* z = reinterpret_cast<float4*>(dq_acc + ((size_t)q * Hq + h) * D);
#pragma unroll
    for (int v = 0; v < D / 8; ++v) {
      const uint4 a = o4[v], b = d4[v];
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const float2 fa = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&aw[t]));
        const float2 fb = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&bw[t]));
        dsum = fmaf(fa.x, fb.x, dsum);
        dsum = fmaf(fa.y, fb.y, dsum);
      }
    }
#pragma unroll
    for (int v = 0; v < D / 4; ++v) z[v] = make_float4(0.f, 0.f, 0.f, 0.f);
    const float lv = lse[(size_t)h * Tq + q];
    l2 = lv * kLog2e;  // -inf stays -inf: such rows have no visible key
  }
  lse2[(size_t)h * qpad + q] = -l2;
  delta[(size_t)h * qpad + q] = -dsum;
}

template <int D>
__global__ void ffa_dq_convert_kernel(const float* __restrict__ acc, __nv_bfloat16* __restrict__ dq,
                                      long long n8) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n8) return;
  const float4 a = reinterpret_cast<const float4*>(acc)[2 * i];
  const float4 b = reinterpret_cast<const float4*>(acc)[2 * i + 1];
  reinterpret_cast<uint4*>(dq)[i] = make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w),
                                               pack_bf16x2(b.x, b.y), pack_bf16x2(b.z, b.w));
}

template <int D>
ffa_status_t launch_bwd_d(ffa_plan_s* p, const void* q, const void* k, const void* v,
                          const void* out, const void* dout, const float* lse, float scale,
                          void* dq, void* dk, void* dv, void* ws, cudaStream_t st) {
  using C = BwdCfg<D>;
  const int qpad = p->n_qt * 128;
  float* lse2 = static_cast<float*>(ws);
  float* delta = lse2 + (size_t)p->Hq * qpad;
  float* dq_acc = delta + (size_t)p->Hq * qpad;
  {
    const long long n = (long long)qpad * p->Hq;
    ffa_bwd_pre_kernel<D><<<(unsigned)((n + 255) / 256), 256, 0, st>>>(
        static_cast<const __nv_bfloat16*>(out), static_cast<const __nv_bfloat16*>(dout), lse,
        p->Tq, p->Hq, qpad, lse2, delta, dq_acc);
    note_launches(1);
    if (cudaGetLastError() != cudaSuccess) return FFA_ERR_CUDA;
  }
  alignas(64) CUtensorMap tq, tk, tv, tdo;
  if (!encode_tile_map(&tq, q, p->Tq, p->Hq * D) || !encode_tile_map(&tk, k, p->Tk, p->Hkv * D) ||
      !encode_tile_map(&tv, v, p->Tk, p->Hkv * D) || !encode_tile_map(&tdo, dout, p->Tq, p->Hq * D))
    return FFA_ERR_INVALID_ARG;
  BwdParams P;
  P.steps = p->bwd_steps;
  P.items = p->bwd_items;
  P.order = p->bwd_order;
  P.n_items = (int)p->n_bwd_items;
  P.slices = p->slices;
  P.Tq = p->Tq;
  P.Tk = p->Tk;
  P.Hq = p->Hq;
  P.g = p->Hq / p->Hkv;
  P.qpad = qpad;
  P.scale = scale;
  P.scale_log2 = scale * kLog2e;
  P.nlse2 = lse2;
  P.ndelta = delta;
  P.dq_acc = dq_acc;
  P.dk = static_cast<__nv_bfloat16*>(dk);
  P.dv = static_cast<__nv_bfloat16*>(dv);
  P.err = p->err;
  P.wait_ns = p->wait_ns;
  if (cudaFuncSetAttribute(ffa_bwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           C::kSmemBytes) != cudaSuccess)
    return FFA_ERR_CUDA;
  ffa_bwd_kernel<D><<<p->grid_bwd, kBwdThreads, C::kSmemBytes, st>>>(tq, tk, tv, tdo, P);
  note_launches(1);
  if (cudaGetLastError() != cudaSuccess) return FFA_ERR_CUDA;
  const long long n8 = (long long)p->Tq * p->Hq * D / 8;
  ffa_dq_convert_kernel<D><<<(unsigned)((n8 + 255) / 256), 256, 0, st>>>(
      dq_acc, static_cast<__nv_bfloat16*>(dq), n8);
  note_launches(1);
  if (cudaGetLastError() != cudaSuccess) return FFA_ERR_CUDA;
  return FFA_OK;
}

}  // namespace

size_t bwd_workspace_bytes(const ffa_plan_s* p) {
  const size_t qpad = (size_t)p->n_qt * 128;
  return (2 * qpad * p->Hq + (size_t)p->Tq * p->Hq * p->D) * sizeof(float);
}

ffa_status_t launch_bwd(ffa_plan_s* p, const void* q, const void* k, const void* v,
                        const void* out, const void* dout, const float* lse, float scale,
                        void* dq, void* dk, void* dv, void* ws, size_t, cudaStream_t st) {
  if (p->D == 128) return launch_bwd_d<128>(p, q, k, v, out, dout, lse, scale, dq, dk, dv, ws, st);
  if (p->D == 64) return launch_bwd_d<64>(p, q, k, v, out, dout, lse, scale, dq, dk, dv, ws, st);
  return FFA_ERR_UNSUPPORTED;
}

}  // namespace ffa

// ---------------------------------------------------------------------------
// Allocation-free backward.
//
// Some callers cannot allocate device memory at the point where they run the
// backward: code running while a stream is being captured into a graph,
// runtimes that forbid allocation after start-up, or hosts whose memory
// manager owns every allocation.  ffa_bwd_noalloc serves them: its scratch
// (log2-scaled lse, delta and the fp32 dQ accumulator) lives in the array
// below, which every GPU that loads this library holds until the process
// exits.  All calls share it, so calls whose kernels overlap on the GPU race.
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
