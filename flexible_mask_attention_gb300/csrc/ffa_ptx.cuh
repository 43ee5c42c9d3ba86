// Inline-PTX building blocks for sm_103a: mbarriers with bounded waits, TMA
// tile loads, and the tcgen05 tensor-core path (TMEM allocation, MMA issue,
// commit, TMEM loads/stores, descriptors).  Written from the public PTX ISA
// (tcgen05, cp.async.bulk.tensor, mbarrier sections).
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace ffa {

// ----------------------------------------------------------------------------
// Error word shared by all kernels: the first failure is kept.
enum DeviceError : int {
  kDevOk = 0,
  kDevTimeout = 1,      // a bounded mbarrier wait ran out
  kDevBadSmemAlign = 2, // dynamic shared memory base not 1024-byte aligned
  kDevBadPlan = 3,      // a work item referenced data out of range
};

__device__ __forceinline__ void record_error(int* err, int code, int where) {
  if (err != nullptr) {
    if (atomicCAS(err, 0, code) == 0) err[1] = where;
  }
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ----------------------------------------------------------------------------
// mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bound for the waits that let a CTA's own copies and MMAs land before it
// exits after a failure; independent of the caller's wait limit.
constexpr uint64_t kDrainNs = 2000000000ull;

// Shared state for bounded waits inside one CTA.
struct WaitCtl {
  int* abort_flag;       // shared memory flag: set once any role gives up
  int* err;              // global error word
  uint64_t timeout_ns;   // wall-clock limit for one wait
};

// Wait until the phase with the given parity has completed.  Gives up after
// ctl.timeout_ns (or as soon as another role of the CTA gave up), records
// kDevTimeout with a location code, and returns false.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const WaitCtl& ctl,
                                          int where) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_test(bar, parity)) return true;
    if (it < 4 || (it & 63u) == 0) {
      if (*(volatile int*)ctl.abort_flag) return false;
      if (globaltimer_ns() - t0 > ctl.timeout_ns) {
        *(volatile int*)ctl.abort_flag = 1;
        record_error(ctl.err, kDevTimeout, where);
        return false;
      }
    }
  }
}

// ----------------------------------------------------------------------------
// Dynamic work queue of a persistent kernel.  One producer thread draws item
// positions from a global ticket counter (zeroed before the launch) and
// publishes the item index through a ring of kItemRing shared-memory slots,
// -1 once the list is exhausted; every consumer thread reads every slot.  The
// slot's "full" barrier counts the producer's arrival, its "empty" barrier
// the consumers' (mbarrier arrive/wait order the slot write before the reads).
// Items are drawn in cost-descending order, so each CTA takes the next
// heaviest item whenever it runs out of work (greedy assignment at run time).
constexpr int kItemRing = 4;

struct ItemQueue {
  int* slot;        // shared [kItemRing]
  uint32_t full0;   // mbarrier of slot 0; slot s's barrier is at + 8 s
  uint32_t empty0;
};

__device__ __forceinline__ bool queue_publish(const ItemQueue& q, int r, int value,
                                              const WaitCtl& ctl, int where) {
  const int s = r % kItemRing;
  if (!mbar_wait(q.empty0 + 8 * s, ((r / kItemRing) & 1) ^ 1, ctl, where)) return false;
  q.slot[s] = value;
  mbar_arrive(q.full0 + 8 * s);
  return true;
}

__device__ __forceinline__ bool queue_take(const ItemQueue& q, int r, int& value,
                                           const WaitCtl& ctl, int where) {
  const int s = r % kItemRing;
  if (!mbar_wait(q.full0 + 8 * s, (r / kItemRing) & 1, ctl, where)) return false;
  value = *reinterpret_cast<volatile int*>(q.slot + s);
  mbar_arrive(q.empty0 + 8 * s);
  return true;
}

// ----------------------------------------------------------------------------
// TMA (tiled, 2-D) and bulk copies, completing on an mbarrier.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
// Tiled 2-D store from shared memory, tracked by the issuing thread's bulk
// async-group; elements outside the tensor's extent are not written.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// This thread's bulk groups have finished reading their shared memory sources.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// This thread's bulk groups have completed (their writes performed).
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ----------------------------------------------------------------------------
// tcgen05: TMEM allocation (one full warp), fences, MMA, commit.
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrive once on the mbarrier when every MMA issued so far by this thread is done.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// Instruction descriptor, kind::f16 with bf16 A/B and fp32 accumulation.
// Bits: [4,6) D format (1 = f32), [7,10) A format (1 = bf16), [10,13) B format,
// 15 A major (1 = MN), 16 B major, [17,23) N >> 3, [24,29) M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) |
         ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Shared-memory matrix descriptor for the 128-byte swizzle layout.
// [0,14) start >> 4, [16,30) leading byte offset >> 4, [32,46) stride byte
// offset >> 4, [46,48) = 1 (tcgen05 descriptor), [61,64) = 2 (128B swizzle).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// MMAs whose shared-memory descriptors are a base descriptor plus an offset in
// 16-byte units (the start field holds address >> 4 in 14 bits; shared-memory
// addresses stay below 256 KB, so the add never carries out of the field),
// with the add inside the same asm block.  Building every descriptor in C++
// per MMA left the single MMA thread issuing slower than the tensor pipe
// drains: measured on GB300, chained 128x128x16 MMAs from one thread ran at
// about 1460 TFLOPS whole-GPU that way and at about 2380 TFLOPS in this form.
__device__ __forceinline__ void mma_ss_at(uint32_t d_tmem, uint64_t a_desc, uint32_t a_off,
                                          uint64_t b_desc, uint32_t b_off, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 da, db;\n\t"
      "add.s64 da, %1, %5;\n\t"
      "add.s64 db, %2, %6;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "l"((uint64_t)a_off),
      "l"((uint64_t)b_off)
      : "memory");
}
__device__ __forceinline__ void mma_ts_at(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                          uint32_t b_off, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 db;\n\t"
      "add.s64 db, %2, %5;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate), "l"((uint64_t)b_off)
      : "memory");
}

// ----------------------------------------------------------------------------
// TMEM <-> registers.  32x32b shape: lane i of the warp reads/writes TMEM lane
// (warp_quarter * 32 + i); .xN covers N consecutive 32-bit columns.
// Each load waits for completion inside the same asm block, so no use of the
// registers can be scheduled before the data has landed.
#define FFA_R8(b) "=r"(r[b + 0]), "=r"(r[b + 1]), "=r"(r[b + 2]), "=r"(r[b + 3]), \
                  "=r"(r[b + 4]), "=r"(r[b + 5]), "=r"(r[b + 6]), "=r"(r[b + 7])
#define FFA_W8(b) "r"(r[b + 0]), "r"(r[b + 1]), "r"(r[b + 2]), "r"(r[b + 3]), \
                  "r"(r[b + 4]), "r"(r[b + 5]), "r"(r[b + 6]), "r"(r[b + 7])

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : FFA_R8(0), FFA_R8(8), FFA_R8(16), FFA_R8(24)
      : "r"(taddr)
      : "memory");
}

// 128 consecutive columns in one instruction, waited inside the same asm block.
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, uint32_t (&r)[128]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x128.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95,%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, [%128];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : FFA_R8(0), FFA_R8(8), FFA_R8(16), FFA_R8(24), FFA_R8(32), FFA_R8(40), FFA_R8(48), FFA_R8(56), FFA_R8(64), FFA_R8(72), FFA_R8(80), FFA_R8(88), FFA_R8(96), FFA_R8(104), FFA_R8(112), FFA_R8(120)
      : "r"(taddr)
      : "memory");
}

// 64 consecutive columns in one instruction, waited inside the same asm block.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : FFA_R8(0), FFA_R8(8), FFA_R8(16), FFA_R8(24), FFA_R8(32), FFA_R8(40), FFA_R8(48), FFA_R8(56)
      : "r"(taddr)
      : "memory");
}

// Two 32-column loads from independent addresses behind a single wait.
__device__ __forceinline__ void tmem_ld32x2(uint32_t ta, uint32_t tb, uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : FFA_R8(0), FFA_R8(8), FFA_R8(16), FFA_R8(24), FFA_R8(32), FFA_R8(40), FFA_R8(48), FFA_R8(56)
      : "r"(ta), "r"(tb)
      : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : FFA_R8(0), FFA_R8(8)
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      FFA_W8(0), FFA_W8(8), FFA_W8(16), FFA_W8(24)
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      FFA_W8(0), FFA_W8(8)
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

#undef FFA_R8
#undef FFA_W8

// Two fp32 -> packed bf16x2 (round to nearest even); `lo` lands in bits [0,16).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// Fire-and-forget fp32 reduction into global memory.
__device__ __forceinline__ void red_add_f32(float* addr, float a) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(addr), "f"(a) : "memory");
}

// Fire-and-forget fp32 vector reduction into global memory (no return value).
__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b),
               "f"(c), "f"(d)
               : "memory");
}

// Maximum of three floats in one instruction.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Minimum of three floats in one instruction.
__device__ __forceinline__ float fmin3(float a, float b, float c) {
  float d;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// tanh from the identity tanh(u) = 1 - 2 / (e^(2u) + 1), with the hardware
// base-2 exponential and reciprocal: absolute error of a few 1e-7, exactly
// +-1 once e^(2u) overflows or underflows.  (Used for the softcap, where
// only absolute errors of the capped score matter.)
__device__ __forceinline__ float tanh_exp(float u) {
  const float e = ex2_approx(u * 2.8853900817779268f);  // 2 log2(e)
  return 1.f - 2.f * rcp_approx(e + 1.f);
}

// Register split of the 384-thread kernels (three warpgroups, one CTA per
// SM).  They compile to 168 registers per thread (65536 / 384, rounded down
// to a multiple of 8); the control warpgroup (producer, MMA issuer, two idle
// warps) shrinks to 104 and the two elementwise warpgroups grow to 200:
// 2 * 128 * 200 + 128 * 104 = 384 * 168, so the exchange always completes.
constexpr int kSplitThreads = 384;
constexpr int kSplitLaunchRegs = 168;
constexpr int kSplitWideRegs = 200;
constexpr int kSplitNarrowRegs = 104;
static_assert(2 * 128 * kSplitWideRegs + 128 * kSplitNarrowRegs == kSplitThreads * kSplitLaunchRegs,
              "register exchange between warpgroups must balance");

// True when the kernel was built with exactly kSplitLaunchRegs registers per
// thread; otherwise the register exchange above could block forever and the
// kernel must not be launched.
template <auto Kernel>
inline bool split_regs_ok() {
  static const int regs = [] {
    cudaFuncAttributes fa;
    return cudaFuncGetAttributes(&fa, Kernel) == cudaSuccess ? fa.numRegs : -1;
  }();
  return regs == kSplitLaunchRegs;
}

// Per-warpgroup register rebalancing; every warp of the warpgroup executes it.
template <int N>
__device__ __forceinline__ void reg_dealloc() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void reg_alloc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

}  // namespace ffa
