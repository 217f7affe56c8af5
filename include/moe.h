/*
 * moe.h - C ABI of the int4 routed-expert MoE layer for one NVIDIA GB300
 * (sm_103a).  One layer forward: noaux_tc sigmoid router with score
 * correction bias and group-limited top-k, renormalised gate weights times
 * routed_scaling_factor, a bit-exact routing plan, int4 group-32
 * dequant -> fp32 SwiGLU routed experts, the weighted combine and the
 * always-on shared expert.
 *
 * What the operations are (page title, then section):
 *  - "GLM-5.2 on a 32 GB Mac - native MLX port of the Colibri hierarchy",
 *    N1 "GLM-5.2 graph" (MoE bullet): sigmoid scores plus correction bias
 *    select, the un-biased sigmoid weights, true top-8, optional
 *    normalisation / routed scale, shared expert in parallel.
 *  - same page, "G2 implementation status": offset-binary Q4
 *    (bias = -8 * scale), lower expert id wins exact ties, unweighted shared
 *    expert; "G2 - native GLM-5.2 correctness spine": dequant -> f32
 *    multiply-accumulate.
 *  - same page, N4 "Scheduling and prediction" and "G3 implementation
 *    status": route the whole batch first, stable unique expert union, each
 *    expert run once over every row that chose it, rows composed in route
 *    order.
 *  - "colibri-strix/README.md", "What's implemented": DeepSeek-V3-style
 *    sigmoid router (noaux_tc, routed_scaling_factor), shared expert,
 *    batch-union MoE; "Experimental resident CUDA backend": invalid requests
 *    fail instead of silently falling back.
 *  - "Model support - run anything mlx-lm runs", 6.4 "GLM-5.2": RMSNorm with
 *    multiplicative weight and double-accumulated reduction.
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers unless stated otherwise; the
 *    caller owns them.  Weights are borrowed: they must stay valid and
 *    unchanged until moe_destroy.  The library never copies or repacks them.
 *  - Work is enqueued on the given stream (a cudaStream_t passed as void*;
 *    NULL = the legacy default stream) and returns without synchronising.
 *  - Argument, shape and capacity errors are detected on the host before
 *    any launch and return a negative moe_status_t; nothing is launched then.
 *    MOE_ERR_CUDA reports a CUDA error (message in moe_last_error).
 *  - A handle is not re-entrant: do not call it from two host threads at
 *    once, and do not have two of its calls in flight on different streams
 *    (they share the handle's workspace).
 *  - There is no CPU fallback: without a usable GB300 every call fails.
 *
 * Data formats:
 *  - int4 weights: symmetric q in [-8, 7] stored offset-binary u = q + 8,
 *    two per byte, the low nibble holding the even K index.  Rows are
 *    K-contiguous.  One fp16 scale (IEEE binary16 bits) per 32 consecutive K
 *    of a row; dequantised value = (u - 8) * scale.
 *  - Routed expert tensors are stacked over experts: gate/up
 *    [E][I][H/2] bytes + [E][I][H/32] scales, down [E][H][I/2] +
 *    [E][H][I/32].  Shared expert: the same without the E dimension, with
 *    I = shared_inter.
 *  - Router weight fp32 [E][H] row-major, bias fp32 [E].
 *  - Activations x: [T][H] fp32 or bf16, row-major.  Output y: [T][H] fp32.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1, /* NULL pointer, negative size, misaligned pointer */
  MOE_ERR_UNSUPPORTED = -2, /* shape outside what the kernels handle */
  MOE_ERR_CAPACITY = -3,    /* T > max_tokens of the handle */
  MOE_ERR_CUDA = -4,        /* a CUDA call failed; see moe_last_error */
  MOE_ERR_OOM = -5          /* workspace allocation failed at create */
} moe_status_t;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype_t;

/* Expert weight formats ("GLM-5.2 on a 32 GB Mac", N2: symmetric int4/int8
 * with per-row or grouped scales; "G2 implementation status": offset-binary
 * Q4 with bias -8 * scale, Q8 scaling the signed two's-complement byte).
 *   MOE_W_INT4: two elements a byte, element 2j in the low nibble of byte j,
 *               value (u - 8) * scale for the stored code u.
 *   MOE_W_INT8: one signed two's-complement byte an element, value
 *               q * scale. */
typedef enum { MOE_W_INT4 = 0, MOE_W_INT8 = 1 } moe_wformat_t;

/* Layer geometry.  Requirements (else MOE_ERR_UNSUPPORTED):
 *   hidden % 256 == 0 and 256 <= hidden <= 12288;
 *   inter % 32 == 0, shared_inter % 32 == 0 (if n_shared), both <= 8192;
 *   1 <= n_experts <= 1024, n_experts % n_group == 0;
 *   1 <= topk_group <= n_group, 1 <= top_k <= 32,
 *   top_k <= topk_group * (n_experts / n_group);
 *   group_size 32 or 0; weight_format MOE_W_INT4 or MOE_W_INT8;
 *   n_shared in {0, 1}; 1 <= max_tokens <= 65536.
 * int4 in either scale layout runs every path but the single-token
 * tensor-core kernel (grouped int4 only); int8 runs on the SIMT batch path
 * at every T. */
typedef struct {
  int hidden;                  /* H */
  int inter;                   /* I, routed expert intermediate size */
  int n_experts;               /* E */
  int top_k;                   /* k */
  int n_group;                 /* expert groups for the group limit */
  int topk_group;              /* groups kept per token */
  float routed_scaling_factor; /* multiplies the renormalised gate weights */
  int n_shared;                /* 0 or 1 always-on shared expert */
  int shared_inter;            /* shared expert intermediate size */
  int group_size;              /* fp16 scales along K: one per 32 values (32) or one
                                  per row (0, Colibri's whole-row group) */
  int max_tokens;              /* largest T any call on this handle may pass */
  int weight_format;           /* moe_wformat_t of every expert matrix */
} moe_config_t;

/* Device pointers, borrowed for the handle's lifetime.  Every pointer must
 * be 16-byte aligned.  sh_* may be NULL when n_shared == 0.  Shapes for
 * MOE_W_INT4 with group_size 32; a MOE_W_INT8 row holds K bytes instead of
 * K/2, and with group_size 0 a row has one scale instead of K/32. */
typedef struct {
  const float* router_w;    /* [E][H] fp32 */
  const float* router_bias; /* [E] fp32 score-correction bias */
  const uint8_t* gate_q;    /* [E][I][H/2] */
  const uint16_t* gate_s;   /* [E][I][H/32] fp16 bits */
  const uint8_t* up_q;      /* [E][I][H/2] */
  const uint16_t* up_s;     /* [E][I][H/32] */
  const uint8_t* down_q;    /* [E][H][I/2] */
  const uint16_t* down_s;   /* [E][H][I/32] */
  const uint8_t* sh_gate_q; /* [Is][H/2] */
  const uint16_t* sh_gate_s;
  const uint8_t* sh_up_q;   /* [Is][H/2] */
  const uint16_t* sh_up_s;
  const uint8_t* sh_down_q; /* [H][Is/2] */
  const uint16_t* sh_down_s;
} moe_weights_t;

/* Routing outputs (device, caller-owned; any member may be NULL to skip it).
 *   topk_ids [T][k] int32  selected experts, biased score descending, ties
 *                          to the lower id
 *   topk_w   [T][k] fp32   gate weights (un-biased sigmoid, renormalised
 *                          over the k, times routed_scaling_factor)
 *   counts   [E]    int32  entries routed to each expert
 *   offsets  [E+1]  int32  exclusive prefix sum of counts
 *   perm     [T*k]  int32  entry indices i = t*k + j grouped by expert
 *                          ascending, ascending i inside an expert
 *   active   [E]    int32  experts with count > 0, ascending (first
 *                          n_active entries are written)
 *   n_active [1]    int32 */
typedef struct {
  int32_t* topk_ids;
  float* topk_w;
  int32_t* counts;
  int32_t* offsets;
  int32_t* perm;
  int32_t* active;
  int32_t* n_active;
} moe_plan_t;

typedef struct moe_layer moe_layer_t;

/* Validate cfg and w, allocate the handle's device workspace (sized for
 * cfg->max_tokens) on the current CUDA device, and return the handle in
 * *out.  On failure *out is set to NULL and the message is available from
 * moe_last_error(NULL) on this thread.
 * Every weight array must lie in device (or managed) memory of the current
 * device, inside allocations that hold all the bytes its shape implies
 * (checked with cuMemGetAddressRange, following adjacent allocations);
 * otherwise MOE_ERR_INVALID_ARG names the array.  The check cannot see a
 * tensor that is too short inside a larger allocation. */
moe_status_t moe_layer_create(const moe_config_t* cfg, const moe_weights_t* w,
                              moe_layer_t** out);

/* Route T tokens (RMSNorm first when rms_gamma is given, see moe_forward):
 * logits, selection and the routing plan.  x: [T][H] of dtype.  T == 0 is a
 * no-op.  Outputs go to the non-NULL members of *plan_out. */
moe_status_t moe_route(moe_layer_t* h, const void* x, moe_dtype_t dtype, int T,
                       const float* rms_gamma, float rms_eps, moe_plan_t* plan_out,
                       void* stream);

/* Full layer forward on T tokens:
 *   x_hat = rms_gamma ? RMSNorm(x) * rms_gamma : x  (eps = rms_eps; the sum
 *           of squares is reduced in fp64)
 *   y     = (accumulate ? y : 0) + sum_j w_tj * E_{id_tj}(x_hat_t) + S(x_hat_t)
 * where E_e is routed expert e's SwiGLU and S the shared expert.  y: [T][H]
 * fp32.  y may alias x only for the residual-stream form (dtype MOE_F32,
 * accumulate = 1, rms_gamma != NULL, y == x exactly); otherwise they must
 * not overlap.  plan_out may be NULL.  T == 0 is a no-op.
 * x and y (and x of moe_route) are device memory, or pinned host memory that
 * is mapped into the device's address space (cudaHostAlloc,
 * cudaHostRegister): the kernels then read x and write y across the host
 * link themselves, with no staging copy.  Any other pointer is refused with
 * MOE_ERR_INVALID_ARG before a launch (each call asks the driver,
 * cudaPointerGetAttributes). */
moe_status_t moe_forward(moe_layer_t* h, const void* x, moe_dtype_t dtype, int T,
                         float* y, const float* rms_gamma, float rms_eps, int accumulate,
                         moe_plan_t* plan_out, void* stream);

/* Free the workspace and the handle.  Waits for the handle's work to finish
 * (device synchronise).  NULL is ignored. */
void moe_destroy(moe_layer_t* h);

/* Last error message of the handle (or of this thread when h == NULL). */
const char* moe_last_error(const moe_layer_t* h);

/* Bytes of device workspace moe_layer_create allocates for cfg (0 if cfg is
 * invalid). */
size_t moe_workspace_bytes(const moe_config_t* cfg);

/* Phase tracing (CUDA events between the kernels of moe_forward).
 * moe_trace_enable(h, n): when n > 0, the next n moe_forward calls each
 * record one CUDA event before their first kernel and one after every
 * kernel, on the call's stream; later calls are not traced.  A traced call
 * launches its kernels without the programmatic-dependent-launch overlap so
 * that each duration belongs to one kernel.  n == 0 disables and frees the
 * events.  Returns MOE_ERR_INVALID_ARG for n < 0 or n > 65536.
 * moe_trace_read(h, ms, cap, n_calls, n_phases): waits for the traced calls
 * (cudaEventSynchronize), writes the duration in milliseconds of phase p of
 * traced call c to ms[c * n_phases + p] for c < min(cap, traced calls)
 * (0 for phases the call did not run), stores the counts, and restarts the
 * trace for the next n calls.  ms must hold cap * n_phases floats, with
 * n_phases = 12 (the phase ids of moe_trace_phase_name).
 * moe_trace_phase_name(p): static name of phase p (NULL when out of range).
 * Tracing is off by default. */
moe_status_t moe_trace_enable(moe_layer_t* h, int n_calls);
moe_status_t moe_trace_read(moe_layer_t* h, float* ms, int cap, int* n_calls, int* n_phases);
const char* moe_trace_phase_name(int phase);

/* Device-side status: copies the handle's device error word to *flags
 * (synchronous), clears it, and returns MOE_ERR_CUDA when it was non-zero.
 * Bit 0: a bounded wait inside a kernel gave up (about one second) and the
 * kernel returned early; the outputs of that call are not valid.  When the
 * word was non-zero the handle's grid-barrier state is also reset, so that
 * later calls run normally again (a call that gave up leaves it out of step). */
moe_status_t moe_device_status(moe_layer_t* h, int32_t* flags);

/* Self-test of the recovery above: puts the handle in the state a call that
 * gave up leaves (its count of grid-barrier rounds one ahead of the device
 * counter), so that the next single-token or small-batch call gives up after
 * about one to two seconds with bit 0 set.  Host-side only; MOE_ERR_INVALID_ARG
 * for a NULL handle. */
moe_status_t moe_selftest_desync(moe_layer_t* h);

/* Self-test of the bounded waits behind bit 0 of moe_device_status, with no
 * layer: one warp waits on something that never completes and gives up after
 * about one second, the way the layer's kernels do, leaving the device usable.
 *   which = 0: the grid-barrier wait (a counter in device memory that stays
 *              below its target);
 *   which = 1: an mbarrier wait (a phase nobody arrives on).
 * Synchronous: allocates 256 bytes of device memory on the current device,
 * launches one warp on the legacy default stream, waits for it, frees the
 * memory and writes the kernel's error word to *flags (bit 0: the wait gave
 * up).  Returns MOE_ERR_INVALID_ARG for which outside {0, 1} or flags NULL
 * (before touching the device), MOE_ERR_CUDA if a CUDA call fails; messages
 * through moe_last_error(NULL). */
moe_status_t moe_selftest_bounded_wait(int which, int32_t* flags);

/* Routing without any allocation (the pages have no counterpart: it serves
 * this library's callers, not a step of the method).
 *
 * Same result as moe_route on a handle created with cfg: optional RMSNorm,
 * router logits, noaux_tc selection and the routing plan of T tokens, written
 * to the non-NULL members of *plan_out.  It takes the router weight and bias
 * directly instead of a handle, and keeps its intermediate buffers in one
 * fixed 2 MiB block of static device memory per device instead of a
 * workspace.  It is meant for callers that cannot allocate device memory at
 * run time: a serving process that hands all of HBM to its expert cache at
 * start-up and allows no later cudaMalloc, or a router-only prefetcher that
 * decides which experts to fetch next without holding their weights (and so
 * without a layer handle).  It calls no cudaMalloc, cudaFree or allocating
 * library routine.
 *
 *   cfg       geometry; validated like moe_layer_create (MOE_ERR_UNSUPPORTED,
 *             with the reason in moe_last_error(NULL)); max_tokens is not used
 *             and may hold any value
 *   router_w  [E][H] fp32, router_bias [E] fp32, x [T][H] of dtype,
 *             rms_gamma [H] or NULL: device pointers, 16-byte aligned.  Every
 *             call checks that router_w and router_bias lie in device memory
 *             of the current device, inside allocations that hold all E*H*4
 *             and E*4 bytes (MOE_ERR_INVALID_ARG otherwise: a host pointer or
 *             a short buffer would become an out-of-bounds read on the GPU);
 *             x and rms_gamma are not checked this way
 *   plan_out  as for moe_route (NULL members, or a NULL plan_out, are kept in
 *             the scratch)
 * Limit: T * (hidden + n_experts) * 4 + 16 * T * top_k + 12 * n_experts, each
 * buffer rounded up to 256 bytes, must fit in the 2 MiB block (for example
 * T <= 64 at hidden = 6144, n_experts = 256, top_k = 8); larger T returns
 * MOE_ERR_CAPACITY with the sizes in moe_last_error(NULL).  T == 0 is a no-op.
 * The first call on a device looks up that device's block
 * (cudaGetSymbolAddress) with the device current; make that first call before
 * capturing any stream.  A call whose stream is not being captured looks the
 * address up again, so a device reset (after which the array can move) is
 * safe once such a call has run; a call made during a capture uses the address
 * of the last call that was not.  Nothing in the block needs to start at zero.  All
 * calls on one device share the block: two calls in flight at the same time
 * (on different streams or from different threads) race and give wrong
 * results, so serialise them.  Errors are reported through
 * moe_last_error(NULL) of the calling thread. */
moe_status_t moe_route_noalloc(const moe_config_t* cfg, const float* router_w,
                               const float* router_bias, const void* x, moe_dtype_t dtype,
                               int T, const float* rms_gamma, float rms_eps,
                               moe_plan_t* plan_out, void* stream);

/* ---- Expert slot cache (host only) ---------------------------------------
 *
 * The residency policy of the expert tier below, as a plain host object so
 * that its decisions can be driven and checked without a GPU.  "GLM-5.2 on a
 * 32 GB Mac - native MLX port of the Colibri hierarchy", "What Colibri is
 * actually doing": item 4 (per-layer bounded LRU with a monotonic use
 * clock), item 5 (pinned hot store, never evicted), item 6 (live repinning
 * with a 25 % + 4 hysteresis), item 8 (a call admits the union of its
 * experts, each once).
 *
 * n_slots slots hold experts 0..n_experts-1; at most n_pinned of them are
 * pinned; a call's union must fit in the unpinned ones, so
 * n_slots - n_pinned >= call_slots.  Kinds written per expert: 0 = hit in
 * the hot store, 1 = hit in an LRU slot, 2 = loaded (the slot must be
 * filled; a resident expert may have been evicted for it).
 *   admit     one call's distinct experts: hits advance the use clock in the
 *             order given; a load takes the lowest free slot, else the least
 *             recently used unpinned slot holding no expert of the set; every
 *             expert counts one use
 *   prefetch  the same placement, counting no use and leaving resident
 *             experts as they are
 *   pin       makes the experts resident and pins their slots
 *   repin     at a safe point: pins the hottest resident unpinned experts
 *             into free hot-store capacity, then up to max_swaps times
 *             replaces the coldest pin (fewest uses, then the higher id) by
 *             the hottest resident unpinned expert (most uses, then the lower
 *             id) when uses(hot) > 1.25 uses(cold) + 4; returns the changes
 *             (-1 for a NULL cache or max_swaps < 0)
 *   query     counters; slot_of[e] = slot, -(slot + 2) when pinned, -1 when
 *             absent; uses[e] = admissions of e (NULL outputs are skipped)
 * An operation that fails (ids outside [0, n_experts) or repeated, more
 * loads than free or evictable slots, too many pins) changes nothing and
 * returns MOE_ERR_INVALID_ARG with the reason in moe_last_error(NULL).  A
 * cache is used by one thread at a time. */
typedef struct moe_slot_cache moe_slot_cache_t;
typedef struct {
  uint64_t hits_pinned; /* admitted experts found pinned */
  uint64_t hits_lru;    /* admitted experts found in an LRU slot */
  uint64_t misses;      /* admitted experts that were loaded */
  uint64_t loads;       /* slots filled by admit, prefetch and pin */
  uint64_t evictions;   /* resident experts displaced by a load */
  int32_t n_resident;
  int32_t n_pinned;
} moe_slot_cache_stats_t;

moe_status_t moe_slot_cache_create(int n_experts, int n_slots, int n_pinned, int call_slots,
                                   moe_slot_cache_t** out);
moe_status_t moe_slot_cache_admit(moe_slot_cache_t* c, const int32_t* ids, int n,
                                  int32_t* slot, int32_t* kind);
moe_status_t moe_slot_cache_prefetch(moe_slot_cache_t* c, const int32_t* ids, int n,
                                     int32_t* slot, int32_t* kind);
moe_status_t moe_slot_cache_pin(moe_slot_cache_t* c, const int32_t* ids, int n, int32_t* slot,
                                int32_t* kind);
int moe_slot_cache_repin(moe_slot_cache_t* c, int max_swaps);
moe_status_t moe_slot_cache_query(const moe_slot_cache_t* c, moe_slot_cache_stats_t* stats,
                                  int32_t* slot_of, uint64_t* uses);
void moe_slot_cache_destroy(moe_slot_cache_t* c);

/* ---- Expert tier: routed experts in host memory, a bounded set in HBM ----
 *
 * The GPU edition of the pages' expert hierarchy ("GLM-5.2 on a 32 GB Mac",
 * "What Colibri is actually doing", items 4-10): the routed experts of a
 * layer live in pinned host memory (reached over the host link) and
 * tcfg->n_slots of them are held in HBM slots managed by the slot cache
 * above; the router and the shared expert stay resident.
 *
 * moe_tier_create(cfg, w, tcfg, out): cfg as for moe_layer_create.  In w,
 *   router_w, router_bias and sh_* are device pointers (as for
 *   moe_layer_create); gate_q ... down_s are the routed arrays of all
 *   n_experts in host memory that is page-locked (cudaHostAlloc or
 *   cudaHostRegister), in the same layout; they are borrowed for the tier's
 *   lifetime and only read.  The tier allocates the workspace, the HBM slots
 *   (n_slots experts) and one copy stream.  Needs 1 <= n_slots <= n_experts,
 *   0 <= n_pinned and n_slots - n_pinned >= min(n_experts,
 *   max_tokens * top_k), so that one call's union always fits
 *   (MOE_ERR_INVALID_ARG otherwise).
 *
 * moe_tier_forward: the layer of moe_forward (same arguments and result, y
 *   within the same tolerance of the oracle), computed as follows:
 *   1. route the tokens on `stream` and wait for the union of their experts
 *      (a small device-to-host copy; the host blocks until routing is done);
 *   2. admit the union in the slot cache; copy every loaded expert from host
 *      memory into its slot on the copy stream (item 9: bounded async reads);
 *   3. launch the experts that are resident (and the shared expert) first,
 *      then, once the copies have landed, the loaded ones (item 9: resident
 *      experts are submitted before the miss reads finish); then the
 *      weighted combine.
 *   The experts run on the SIMT batch kernels (every weight format).  A slot
 *   is never read before its copy has completed and never overwritten while a
 *   call that reads it may still run (item 10: no partially filled slot is
 *   published).  All calls of one tier use one stream.
 * moe_tier_prefetch(t, ids, n): loads the experts not yet resident (no use
 *   counted) on the copy stream and returns without waiting (item 10).
 * moe_tier_prefetch_routed(t, x, dtype, T, rms_gamma, rms_eps, stream):
 *   routes x with this tier's router and prefetches the union (item 10,
 *   PILOT: the next layer's router applied to the current state).  Waits
 *   for the routing, not for the copies.
 * moe_tier_pin(t, ids, n): loads (if needed) and pins experts (item 5).
 * moe_tier_repin(t, max_swaps, changed): moe_slot_cache_repin at a safe
 *   point; *changed (may be NULL) receives its result.
 * moe_tier_query(t, stats, slot_of, uses, h2d_bytes): the slot cache's
 *   query; *h2d_bytes (may be NULL) = expert bytes copied into HBM so far.
 * moe_tier_last_error(t): the tier's last message (moe_last_error(NULL) for
 *   failures of moe_tier_create).
 * A CUDA failure inside forward, prefetch or pin (MOE_ERR_CUDA) leaves the
 *   tier unusable: the slots may not hold what its cache records, so every
 *   later forward, prefetch and pin returns MOE_ERR_CUDA; destroy it.
 * moe_tier_destroy(t): waits for the tier's work and frees it (NULL is
 *   ignored). */
typedef struct moe_tier moe_tier_t;
typedef struct {
  int n_slots;  /* HBM expert slots */
  int n_pinned; /* of which the hot store may hold this many */
} moe_tier_config_t;

moe_status_t moe_tier_create(const moe_config_t* cfg, const moe_weights_t* w,
                             const moe_tier_config_t* tcfg, moe_tier_t** out);
moe_status_t moe_tier_forward(moe_tier_t* t, const void* x, moe_dtype_t dtype, int T, float* y,
                              const float* rms_gamma, float rms_eps, int accumulate,
                              moe_plan_t* plan_out, void* stream);
moe_status_t moe_tier_prefetch(moe_tier_t* t, const int32_t* ids, int n);
moe_status_t moe_tier_prefetch_routed(moe_tier_t* t, const void* x, moe_dtype_t dtype, int T,
                                      const float* rms_gamma, float rms_eps, void* stream);
moe_status_t moe_tier_pin(moe_tier_t* t, const int32_t* ids, int n);
moe_status_t moe_tier_repin(moe_tier_t* t, int max_swaps, int* changed);
moe_status_t moe_tier_query(moe_tier_t* t, moe_slot_cache_stats_t* stats, int32_t* slot_of,
                            uint64_t* uses, uint64_t* h2d_bytes);
const char* moe_tier_last_error(const moe_tier_t* t);
void moe_tier_destroy(moe_tier_t* t);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H_ */
