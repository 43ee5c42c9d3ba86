/*
 * ffa.h -- C ABI of the flexible-mask flash attention library (libffa.so),
 * built for NVIDIA GB300 (sm_103a).
 *
 * The operation (MagiAttention pages, quickstart card "Single-GPU
 * Flex-Flash-Attention", flex_flash_attn_func): softmax attention over a
 * packed token stream whose mask is a list of slices.  Slice s is
 * (q_range [qs, qe), k_range [ks, ke), mask_type); inside it query row i sees
 * keys [lo, hi) with
 *     lo = ks + (i - qs)        if mask_type has bit 1 set (inverse causal),
 *          ks                   otherwise;
 *     hi = ke - (qe - 1 - i)    if mask_type has bit 0 set (causal),
 *          ke                   otherwise
 * (card "Calculate KV Interval Boundaries for Mask Types"), so causal is
 * bottom-right aligned in the slice's rectangle.  A row sees the union of its
 * intervals over all slices containing it.  out_i = sum_j softmax_j(scale *
 * q_i.k_j) v_j, lse_i = log sum_j exp(scale * q_i.k_j) (natural log), and a
 * row that sees no key gives out = 0, lse = -inf.  Query head h uses key/value
 * head h / (Hq / Hkv).
 *
 * Conventions for every call
 *   - Tensors are caller-owned DEVICE pointers, contiguous, 16-byte aligned:
 *       q, out, dout, dq   [Tq][Hq][D]   bf16
 *       k, v, dk, dv       [Tk][Hkv][D]  bf16
 *       lse                [Hq][Tq]      fp32 (head-major)
 *       q_ranges, k_ranges [S][2] int32 (device), mask_types [S] int32 (device)
 *   - Supported: D in {64, 128}; Hq % Hkv == 0; 0 <= start <= end <= T for
 *     every range.  Slices with an empty range are allowed and do nothing.
 *     The (q x k) rectangles of non-empty slices must be pairwise disjoint.
 *   - Work is queued on `stream` and returns immediately, except
 *     ffa_plan_create, which synchronises `stream` while it sizes the plan.
 *   - ffa_fwd / ffa_bwd never allocate: scratch memory is the caller's
 *     `workspace` of at least the size the *_workspace_size call reports.
 *   - Every call that takes a plan must run with the plan's device current
 *     (the one current at ffa_plan_create); otherwise it returns
 *     FFA_ERR_INVALID_ARG before touching the GPU (ffa_plan_destroy switches
 *     to the plan's device itself).
 *   - Errors come back as an ffa_status_t; nothing aborts the process.
 *     Device-side failures (a bounded wait that ran out) are reported by
 *     ffa_get_last_device_error.
 */
#ifndef FFA_H_
#define FFA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* ffa_stream_t; /* same as cudaStream_t; NULL = legacy default */

typedef enum {
  FFA_FULL = 0,        /* every (q, k) pair of the rectangle */
  FFA_CAUSAL = 1,      /* bottom-right aligned lower triangle */
  FFA_INV_CAUSAL = 2,  /* top-left aligned upper triangle */
  FFA_BI_CAUSAL = 3    /* both clamps: a band */
} ffa_mask_t;

typedef enum {
  FFA_OK = 0,
  FFA_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned pointer */
  FFA_ERR_RANGE = 2,       /* a range outside [0, T] or start > end, bad mask type */
  FFA_ERR_OVERLAP = 3,     /* two non-empty slice rectangles intersect */
  FFA_ERR_UNSUPPORTED = 4, /* head_dim not in {64, 128}, Hq % Hkv != 0, device not sm_103 */
  FFA_ERR_WORKSPACE = 5,   /* workspace smaller than required */
  FFA_ERR_TIMEOUT = 6,     /* a kernel's bounded wait ran out (see ffa_get_last_device_error) */
  FFA_ERR_CUDA = 7         /* a CUDA runtime call failed */
} ffa_status_t;

/* Opaque plan: the tile work lists derived from one slice table and shape.
 * It owns device memory for its metadata only and may be reused by any
 * number of ffa_fwd / ffa_bwd calls on the same device. */
typedef struct ffa_plan_s* ffa_plan_t;

/* Build a plan (the slice planner and tile scheduler).
 *   q_ranges, k_ranges: device int32 [num_slices][2]; mask_types: device
 *   int32 [num_slices] (ffa_mask_t values).  total_q / total_k are Tq / Tk.
 *   num_sms: CTAs the persistent kernels will use (0 = every SM of the
 *   current device).  split_below: split forward work items into key chunks
 *   (merged by logsumexp) while fewer than this many items exist (0 = twice
 *   num_sms, -1 = never split).
 * Runs validation and planning kernels on `stream` and synchronises it.
 * Returns FFA_ERR_RANGE / FFA_ERR_OVERLAP for a bad slice table. */
ffa_status_t ffa_plan_create(ffa_plan_t* plan, const int32_t* q_ranges, const int32_t* k_ranges,
                             const int32_t* mask_types, int32_t num_slices, int32_t total_q,
                             int32_t total_k, int32_t num_heads_q, int32_t num_heads_kv,
                             int32_t head_dim, int32_t num_sms, int32_t split_below,
                             ffa_stream_t stream);

/* Free a plan and its device memory (synchronises the plan's device first;
 * the caller's current device is unchanged afterwards). */
ffa_status_t ffa_plan_destroy(ffa_plan_t plan);

/* Sizes of the plan's work lists, in int32 words; see ffa_plan_export. */
typedef struct {
  int64_t fwd_steps;  /* 4 words per step */
  int64_t fwd_items;  /* 8 words per item */
  int64_t bwd_steps;  /* 4 words per step */
  int64_t bwd_items;  /* 8 words per item */
  int64_t merges;     /* 8 words per merge group */
  int32_t grid_fwd;   /* CTAs of the forward kernel */
  int32_t grid_bwd;   /* CTAs of the backward kernel */
  int64_t area;       /* visible (q, k) pairs per head: sum over rows of |keys seen| */
  int64_t fwd_masks;  /* words of the forward slice lists (multi-slice visits) */
  int64_t bwd_masks;  /* words of the backward slice lists */
  int64_t gathers;    /* gathered forward step records, 144 words each */
  int64_t bgathers;   /* gathered backward step records, 80 words each */
  int64_t stacked;    /* slab rows (64 or 32) of head-stacked forward units, 0: none (below) */
} ffa_plan_info_t;

ffa_status_t ffa_plan_info(ffa_plan_t plan, ffa_plan_info_t* info);

/* Copy one work list to HOST memory (used to check the planner bit for bit).
 *   which: 0 fwd steps, 1 fwd items, 2 fwd order, 3 bwd steps, 4 bwd items,
 *          5 bwd order, 6 merge groups, 7 fwd slice lists, 8 bwd slice lists,
 *          9 gathered forward step records, 10 gathered backward step records.
 *   A step's visit info is (s << 2) | partial when one slice s sees the tile
 *   pair, or (m << 2) | 3 when several do; then list[m] = n and list[m+1 ..
 *   m+n] are their slice indices, ascending (the tile is computed once and
 *   masked by the union of their windows).
 *   Gathered forward steps (a forward unit whose slices are all FULL with key
 *   ranges aligned to 8 keys, when that takes at most 9/10 of its tile steps):
 *   step (0, info0, info1, r + 1) computes 16 blocks of 8 keys packed into
 *   one K/V tile; record r holds the 16 block start keys (-8: unused slot),
 *   then for each half 16 x 4 words of row bits (bit i of word w: row
 *   32 w + i of the half's q-tile sees that block); info_h is 0 when all 16
 *   slots hold keys and every row of half h sees them all (no mask), else 1
 *   when half h has a row bit set, else -1.
 *   Gathered backward steps, the transpose (a k-tile whose slices are all FULL
 *   with query ranges aligned to 8 rows, when that takes at most 9/10 of its
 *   visits): step (0, 1, 0, r + 1) computes 16 blocks of 8 query rows packed
 *   into one Q / dO tile; record r holds the 16 block start rows (-8: unused)
 *   then 16 x 4 words of key bits (bit i of word w: key 32 w + i of the
 *   k-tile is seen by that block's rows).
 *   Head-stacked forward units (info.stacked = R; with Hq / Hkv even and at
 *   least 4, when every R-row slab of the queries meets only FULL slices
 *   with 8-aligned key ranges and slab units take at most 9/10 of the work
 *   otherwise chosen; R = 32 needs Hq / Hkv a multiple of 4): the units are
 *   R-row slabs, every step is gathered, and an item (s, s, h, h + m), with
 *   m = 128 / R, holds in half 0 the slab's rows of heads h .. h + m - 1
 *   stacked as tile rows [R j, R j + R) for head h + j (half 1: heads
 *   h + m ..; idle, slab and head -1, past the group); a record's row bits
 *   r, r + R, ... all stand for slab row r.  With R = 32 and Hq / Hkv = 4
 *   an item is (s, s, h, h): both halves hold the same rows and take the
 *   slab's steps in turn (even steps half 0, odd ones half 1), merged by
 *   logsumexp in the kernel.  Such plans are not split.
 *   dst: host int32 buffer of `capacity` words; *written receives the count.
 * Synchronises the plan's stream. */
ffa_status_t ffa_plan_export(ffa_plan_t plan, int32_t which, int32_t* dst, int64_t capacity,
                             int64_t* written);

/* Workspace bytes ffa_fwd / ffa_bwd need for this plan (0 is possible). */
size_t ffa_fwd_workspace_size(ffa_plan_t plan);
size_t ffa_bwd_workspace_size(ffa_plan_t plan);

/* Forward: out[Tq][Hq][D] (bf16) and lse[Hq][Tq] (fp32, natural log).
 *   softmax_scale <= 0 selects 1/sqrt(D), the default the quickstart
 *   card gives.  workspace: device memory of ffa_fwd_workspace_size
 *   bytes (may be NULL when that size is 0), contents need not be set.
 * Rows that see no key are written as out = 0, lse = -inf. */
ffa_status_t ffa_fwd(ffa_plan_t plan, const void* q, const void* k, const void* v,
                     float softmax_scale, void* out, float* lse, void* workspace,
                     size_t workspace_bytes, ffa_stream_t stream);

/* Attention sink (MagiAttention pages: the `sink` argument of
 * flex_flash_attn_func in the quickstart card, and the FlashAttention
 * "with sink" cards, which give its two layouts).  The pages do not state the
 * formula; this library reads it as: each sink value s is a logit in natural
 * log units, NOT multiplied by softmax_scale, that joins only the row's
 * normaliser,
 *     lse_i = log( sum_j exp(scale * q_i.k_j) + sum_s exp(sink_s) ),
 *     out_i = sum_j exp(scale * q_i.k_j - lse_i) v_j,
 * so a row that sees no key gets out = 0 and lse = log sum_s exp(sink_s), and
 *     dsink_s = - sum_i exp(sink_s - lse_i) <dout_i, out_i>.
 * Layouts of the fp32 DEVICE array (4-byte aligned):
 *     FFA_SINK_SH   [num_sink][Hq]      one set per query head (dsink sums over rows)
 *     FFA_SINK_SSH  [Tq][num_sink][Hq]  one set per (row, query head)
 * A sink value of -inf contributes nothing. */
typedef enum { FFA_SINK_SH = 0, FFA_SINK_SSH = 1 } ffa_sink_layout_t;
#define FFA_MAX_SINK 64 /* largest num_sink accepted */

/* Softcap (MagiAttention quickstart card: the `softcap` argument of
 * flex_flash_attn_func, default 0; the pages give no formula).  This library
 * reads it as the usual smooth cap: for softcap = c > 0 every score
 * x = scale * q_i.k_j becomes c * tanh(x / c) before the softmax (the
 * backward carries the factor 1 - tanh^2 into dS); c = 0 means no cap.
 *
 * ffa_fwd with optional sink logits and softcap (num_sink = 0 and
 * softcap = 0: identical to ffa_fwd; sink may then be NULL).  Returns
 * FFA_ERR_INVALID_ARG for num_sink outside [0, FFA_MAX_SINK], an unknown
 * layout, a NULL / misaligned sink when num_sink > 0, or a negative or
 * non-finite softcap.  lse includes the sink term. */
ffa_status_t ffa_fwd_ex(ffa_plan_t plan, const void* q, const void* k, const void* v,
                        const float* sink, int32_t num_sink, int32_t sink_layout,
                        float softmax_scale, float softcap, void* out, float* lse,
                        void* workspace, size_t workspace_bytes, ffa_stream_t stream);

/* Backward of ffa_fwd for the loss L with dL/dout = dout.
 *   out, lse: the forward's results; dq, dk, dv receive the gradients
 *   (bf16, every element written; keys seen by no query get 0).
 *   workspace: device memory of ffa_bwd_workspace_size bytes. */
ffa_status_t ffa_bwd(ffa_plan_t plan, const void* q, const void* k, const void* v,
                     const void* out, const void* dout, const float* lse, float softmax_scale,
                     void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                     ffa_stream_t stream);

/* Backward of ffa_fwd_ex.  out and lse are ffa_fwd_ex's results for the same
 * sink and softcap (the sink acts on dq, dk, dv only through lse).  dsink: fp32 DEVICE
 * array in the sink's layout, overwritten with the sink gradient, or NULL to
 * skip it; ignored when num_sink = 0.  The per-head sums of the "sh" layout
 * are taken in a fixed order, so repeated calls give identical results. */
ffa_status_t ffa_bwd_ex(ffa_plan_t plan, const void* q, const void* k, const void* v,
                        const void* out, const void* dout, const float* lse, const float* sink,
                        int32_t num_sink, int32_t sink_layout, float softmax_scale, float softcap,
                        void* dq, void* dk, void* dv, float* dsink, void* workspace,
                        size_t workspace_bytes, ffa_stream_t stream);

/* Backward without any allocation: the same computation as ffa_bwd, with its
 * scratch memory taken from a fixed array inside the library instead of a
 * caller workspace.  (No counterpart in the MagiAttention pages.)  For callers
 * that cannot allocate device memory when they run the backward: runtimes
 * that forbid allocation once they have started, hosts whose own memory
 * manager owns every byte of the GPU, or latency-critical loops that must not
 * pay for (or synchronise on) an allocation.
 *   - The array holds ffa_bwd_noalloc_max_workspace() bytes (64 MiB) on every
 *     GPU that loads this library, until the process exits.  A plan whose
 *     ffa_bwd_workspace_size exceeds it gets FFA_ERR_WORKSPACE.
 *   - The first call on a device resolves the array's device address (with
 *     that device current); make that first call before any stream capture.
 *   - Every call shares the array and rewrites all of the scratch it reads;
 *     calls whose kernels overlap on the GPU (other streams) race.
 *   - Arguments as for ffa_bwd; nothing is allocated or freed. */
ffa_status_t ffa_bwd_noalloc(ffa_plan_t plan, const void* q, const void* k, const void* v,
                             const void* out, const void* dout, const float* lse,
                             float softmax_scale, void* dq, void* dk, void* dv,
                             ffa_stream_t stream);

/* Size in bytes of the fixed scratch array ffa_bwd_noalloc uses. */
size_t ffa_bwd_noalloc_max_workspace(void);

/* Read and clear the device error word the plan's kernels write:
 *   *code = 0 none, 1 bounded wait timed out, 2 shared memory misaligned,
 *   3 bad work item; *where = the location tag of the first failure.
 * Synchronises `stream`. */
ffa_status_t ffa_get_last_device_error(ffa_plan_t plan, int32_t* code, int32_t* where,
                                       ffa_stream_t stream);

/* Bounded-wait limit for the plan's kernels, in nanoseconds (default 2e9).
 * A wait that runs out makes the kernel stop and report FFA_ERR_TIMEOUT. */
ffa_status_t ffa_plan_set_wait_limit(ffa_plan_t plan, uint64_t nanoseconds);

/* Instrumentation: CUDA events (cudaEvent_t values, created by the caller)
 * that ffa_fwd / ffa_bwd record on their stream around their kernels:
 *   events[0], events[1]: before / after the forward kernel (and merge);
 *   events[2], events[3], events[4], events[5]: before the backward
 *   preprocess, before the dK/dV pass, before the dQ pass, after the dQ pass.
 * n_events must be 6, or 0 to stop recording.  The plan keeps the handles
 * only; the caller owns and destroys the events. */
ffa_status_t ffa_plan_set_events(ffa_plan_t plan, void* const* events, int32_t n_events);

/* Human-readable name of a status code (static storage). */
const char* ffa_status_string(ffa_status_t status);

/* Number of CUDA kernels this library has launched in the calling process
 * (planner, forward, merge and backward kernels).  For instrumentation. */
uint64_t ffa_kernel_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* FFA_H_ */
