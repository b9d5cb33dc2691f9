/*
 * moe_gb300.h -- C ABI of libmoe_gb300.so: one routed Mixture-of-Experts FFN
 * layer with IQ4_NL expert weights and a sigmoid router, for one NVIDIA
 * GB300 GPU (sm_103a).
 *
 * What the layer computes (HelloSun/xing4_0-29b-IQ4_NL_EPQ model card,
 * sections "模型與路由" and "對純 NumPy：整層"; PocketLLM "Xing4.0-29B-A4B: the
 * design record", sections 1, 2 and 4; zhuai.tech "FFN: feature processing
 * inside each layer"), for each token t with input row x[t]:
 *
 *   l[e]  = x[t] . Wr[e]  (+ b[t][e])             router logits, fp32
 *   s[e]  = sigmoid(l[e])
 *   S     = the k experts with the largest s, in descending order
 *   w[j]  = scale * s[S_j] / sum_{i in S} s[i]   (scale = 2.0 for Xing4)
 *   FFN_e(v) = Down_e( silu(Gate_e v) * (Up_e v) ),  silu(g) = g / (1 + e^-g)
 *   out[t] = sum_j w[j] * FFN_{S_j}(x[t]) + FFN_shared(x[t])
 *
 * Each expert matrix is IQ4_NL: rows of 18-byte blocks, each block one fp16
 * scale d followed by 16 bytes holding 32 4-bit indices i; weight = d *
 * table[i] with the 16-entry table {-127,-104,-83,-65,-49,-35,-22,-10,1,13,
 * 25,38,53,69,89,113}.  Within a block, weight j (0..15) is the low nibble
 * of index byte j and weight j+16 its high nibble.
 *
 * Conventions for every entry point:
 *   - Every data pointer is a DEVICE pointer owned by the caller, unless the
 *     argument says otherwise.  Arrays are dense and row-major.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default).
 *     Route and forward calls are asynchronous on it; they never allocate,
 *     never synchronise and never copy data back to the host, so they can be
 *     captured in a CUDA graph.  (PocketLLM design record, section 6 "Where
 *     a decode step's time goes": a route-count read back to the host cost a
 *     copy and a stream drain per layer and was what refused graph capture.)
 *   - Everything a call will need is sized and allocated when the layer is
 *     created, and a shape the kernels cannot run is refused there, not in
 *     the middle of a request (PocketLLM design record, section 5 "The
 *     prefill chunk is a function of the card": a configuration that cannot
 *     fit is a refusal at load rather than an out-of-memory error inside a
 *     request).
 *   - Host-checkable errors (NULL pointer, bad size, T > max_tokens,
 *     misaligned base pointer) return a status and launch nothing.  Base
 *     pointers read with 16-byte vector loads are checked for 16-byte
 *     alignment, not only their row strides (FLASHNEXT-RESEARCH.md, section
 *     4 "Second target: 216 F32 GEMVs on a bare cuBLAS SGEMM": a guard that
 *     checked the stride but not the base pointer of a float4-read operand
 *     let an offset view fault).  Errors only the device can see (an expert
 *     id outside [0, E) handed to moe_forward, a device wait that gave up)
 *     set a sticky word in the layer that moe_layer_check() reports; the
 *     offending route contributes zero.
 *   - No call falls back to another implementation when its own cannot run:
 *     it returns an error status (HelloSun/xing4_0-29b-IQ4_NL_EPQ model card,
 *     "已知陷阱": fail loudly rather than quietly fall back to a different
 *     path).  Where the layer has two GPU paths for a batch size (the
 *     single-launch decode kernel and the tensor-core kernels), which one
 *     runs is fixed at create from the shape and the device.
 *   - A layer is used by one stream at a time; separate layers are
 *     independent.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_GB300_ABI_VERSION 1

typedef struct moe_layer_s *moe_layer_t; /* opaque, owned by the library */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,       /* NULL pointer, negative size, bad enum   */
  MOE_ERR_UNSUPPORTED_SHAPE = 2, /* shape outside the limits below          */
  MOE_ERR_MISALIGNED = 3,        /* a base pointer breaks its alignment rule*/
  MOE_ERR_OUT_OF_MEMORY = 4,     /* cudaMalloc failed in create             */
  MOE_ERR_CUDA = 5,              /* a CUDA call failed; see moe_last_error  */
  MOE_ERR_TIMEOUT = 6,           /* a bounded device wait gave up           */
  MOE_ERR_BAD_EXPERT_ID = 7,     /* an id outside [0, E) reached forward    */
  MOE_ERR_TOO_MANY_TOKENS = 8,   /* T > max_tokens given at create          */
  MOE_ERR_OVERFLOW = 9           /* an activation left fp16 range (batched  *
                                  * tensor-core path); outputs are invalid  */
} moe_status;

typedef enum { MOE_DT_BF16 = 0, MOE_DT_FP32 = 1 } moe_dtype;

/* Layer shape.  Limits: hidden and expert_ffn multiples of 32 in [32, 16384];
 * 1 <= n_experts <= 256; 1 <= top_k <= min(n_experts, 8); n_shared 0 or 1;
 * 1 <= max_tokens <= 65536; routed_scaling > 0; flags a combination of the
 * MOE_FLAG_* bits below (other bits: MOE_ERR_INVALID_ARG). */
typedef struct {
  int32_t hidden;       /* H                                                */
  int32_t n_experts;    /* E routed experts                                 */
  int32_t top_k;        /* k experts per token                              */
  int32_t expert_ffn;   /* F, intermediate width of every expert            */
  int32_t n_shared;     /* 1: one always-on shared expert, weight 1         */
  float routed_scaling; /* scale applied to the renormalised weights        */
  int32_t max_tokens;   /* largest T any later call may pass                */
  uint32_t flags;       /* MOE_FLAG_* bits, 0 for the plain router          */
} moe_shapes;

/* Selection-only score bias (noaux_tc) [EPQ, "模型與路由": sigmoid plus the
 * per-expert probability bias ffn_exp_probs_b].  With this flag the
 * logit_bias argument of moe_route and moe_layer_forward_routed is not added
 * to the logits: expert e is ranked by sigmoid(l_e) + b_e, while the weights
 * are still routed_scaling * s_e / sum(s) of the unbiased s_e = sigmoid(l_e).
 * Without it the bias is added to the logit before the sigmoid and so enters
 * both the ranking and the weights.  moe_route_noalloc has no layer and always
 * takes the logit reading. */
#define MOE_FLAG_SELECTION_BIAS 1u

/* Deterministic combine [PocketLLM, "Xing4.0-29B-A4B: the design record",
 * section 4: float atomics make the top-k sum differ from run to run].
 * Batches on the multi-launch paths (above 16 tokens, or above 8 for shapes
 * the batch kernel does not take) then store each route's weighted down
 * output once (no atomics) and add a token's routes in slot order, the
 * shared expert last, so equal inputs give equal output bits on every call.
 * It costs an extra [routes][H] fp32 buffer (max_tokens * (top_k +
 * n_shared) rows, allocated at create) and one write and one read of it per
 * call.  The single-launch decode kernels (up to 16 tokens) are
 * deterministic with or without the flag. */
#define MOE_FLAG_DETERMINISTIC 2u

/* Host input and output for moe_layer_forward_routed_host: the layer holds
 * a device copy buffer for x and one for out, each max_tokens * hidden * 4
 * bytes, allocated at create. */
#define MOE_FLAG_HOST_IO 4u

/* Cooperative launches for the single-launch decode kernels (up to 16
 * tokens), which hold one CTA on every SM and wait device-wide inside.  At
 * create the layer checks that one CTA fits on every SM; without this flag
 * the kernels are plain launches (a cooperative launch adds about 3 us of
 * launch latency to every call that is not replayed from a CUDA graph), so
 * a caller must not keep SMs busy with other kernels, on other streams or
 * through MPS or green contexts, while a decode call runs: its waits would
 * run out and the call would report MOE_ERR_TIMEOUT.  With the flag the
 * runtime starts each such launch only once its whole grid can be resident
 * at the same time. */
#define MOE_FLAG_COOPERATIVE 8u

/* Expert weights in IQ4_NL blocks (18 bytes each, no alignment needed).
 *   up, gate: [E][F][H/32] blocks     down: [E][H][F/32] blocks
 *   sh_up, sh_gate: [F][H/32]         sh_down: [H][F/32]  (NULL if no shared)
 * The library copies and re-lays them out; see moe_layer_create. */
typedef struct {
  const void *up;
  const void *gate;
  const void *down;
  const void *sh_up;
  const void *sh_gate;
  const void *sh_down;
} moe_weights;

/* Create a layer.  Copies the weights into library-owned device memory in an
 * internal layout (same byte count: 8 blocks' scales and nibbles grouped in
 * 144-byte units, rows padded with zero blocks to a multiple of 256 weights
 * where H or F is not one) and allocates every workspace later calls need for
 * up to max_tokens tokens, so that no later call allocates or can run out of
 * memory (PocketLLM design record, section 5: refuse at load, not inside a
 * request).  The layer belongs to the device current at create; create also
 * raises the kernels' shared-memory limits on that device and checks that the
 * single-launch decode kernels' grids (one CTA per SM, with device-wide waits
 * inside: the one-token kernel for T = 1 on the Xing4 and K2-Horizon hidden
 * sizes, the multi-token kernel for up to 8 tokens) can be resident all at
 * once -- if not, those batches run on the other kernels instead.  Runs on `stream` and synchronises
 * it before returning, so the caller may free its weight buffers afterwards.
 * On success *out holds the layer; on failure *out is NULL and nothing is
 * leaked. */
moe_status moe_layer_create(const moe_shapes *shapes, const moe_weights *weights,
                            void *stream, moe_layer_t *out);

/* Free a layer and its device memory (synchronises the device first).
 * NULL is accepted and ignored. */
moe_status moe_layer_destroy(moe_layer_t layer);

/* Router (steps: logits, sigmoid, top-k, renormalise, scale).
 *   x           [T][H], MOE_DT_BF16 or MOE_DT_FP32, 16-byte aligned
 *   router_w    [E][H] fp32, 16-byte aligned (the layer's ffn_gate_inp)
 *   logit_bias  NULL, or fp32 with row t at logit_bias + t*bias_row_stride
 *               (stride 0: one [E] row for every token), 16-byte aligned;
 *               added to the logit before the sigmoid, or with
 *               MOE_FLAG_SELECTION_BIAS to the sigmoid score for ranking only
 *   ids         [T][k] int32 out, descending score; equal scores -> lower id
 *   weights     [T][k] fp32 out, sum to routed_scaling per token
 * 0 <= T <= max_tokens; T == 0 returns MOE_OK and launches nothing.
 * The ids and weights stay on the device (PocketLLM design record, section
 * 6: no route count is read back), ready for moe_forward on the same
 * stream. */
moe_status moe_route(moe_layer_t layer, const void *x, moe_dtype x_dtype, int32_t T,
                     const float *router_w, const float *logit_bias,
                     int64_t bias_row_stride, int32_t *ids, float *weights,
                     void *stream);

/* Expert part of the layer for given routes (steps: per-expert histogram,
 * prefix sum and permutation; gather; dequantising up/gate projection with
 * SwiGLU; down projection; weighted combine with the shared expert).
 *   x        [T][H] as in moe_route
 *   ids      [T][k] int32, each in [0, E); 4-byte aligned
 *   weights  [T][k] fp32, any values; 4-byte aligned
 *   out      [T][H], MOE_DT_BF16 or MOE_DT_FP32, 16-byte aligned; the sum is
 *            formed in fp32 and rounded once (bf16: nearest-even)
 * The routed sum and the shared expert are accumulated in fp32.  Above 8
 * tokens the order of those additions is whatever order the atomics commit
 * in (up to k+1 terms per element), so outputs may differ in the last bits
 * between runs, unless the layer was created with MOE_FLAG_DETERMINISTIC;
 * up to 8 tokens every addition has a fixed order.
 * The per-expert histogram, prefix sum and permutation run on the device
 * (PocketLLM design record, section 4: a CSR route table consumed by one
 * grouped kernel; section 6: the counts are never read back), so the call
 * is graph-capturable.  The single-launch decode kernels (T <= 8; T = 1 has
 * its own, which splits the routed experts into 32-output units, one per SM)
 * hold every SM of the device for the duration of the call and wait
 * device-wide inside: a layer whose grid of one CTA per SM cannot be
 * resident takes the multi-launch path (checked at create), and with
 * MOE_FLAG_COOPERATIVE the runtime starts each launch only once its whole
 * grid can be resident.  Their waits are bounded; one that gives up is
 * reported by moe_layer_check() as MOE_ERR_TIMEOUT. */
moe_status moe_forward(moe_layer_t layer, const void *x, moe_dtype x_dtype, int32_t T,
                       const int32_t *ids, const float *weights, void *out,
                       moe_dtype out_dtype, void *stream);

/* Dense FFN block: out[t] = W_down (silu(W_gate x[t]) * (W_up x[t])) for
 * every token, no router and no weight [PocketLLM, "Xing4.0-29B-A4B: the
 * design record", section 1: the first two of the forty blocks are dense
 * (first_k_dense_replace = 2); EPQ, "模型與路由": dense FFN width 9,216].
 * The block is a layer created with n_experts = 1, top_k = 1, n_shared = 0
 * (routed_scaling is not used) holding the FFN as expert 0; this call runs
 * it on the same kernels as moe_forward with every token routed to expert 0
 * at weight 1.  Arguments and errors as for moe_forward; a layer of any
 * other shape returns MOE_ERR_INVALID_ARG. */
moe_status moe_dense_forward(moe_layer_t layer, const void *x, moe_dtype x_dtype, int32_t T,
                             void *out, moe_dtype out_dtype, void *stream);

/* moe_route followed by moe_forward on the same stream, with the same
 * arguments; ids and weights are written as by moe_route.  For small T the
 * two run fused in as few launches as the layer allows. */
moe_status moe_layer_forward_routed(moe_layer_t layer, const void *x, moe_dtype x_dtype,
                                    int32_t T, const float *router_w,
                                    const float *logit_bias, int64_t bias_row_stride,
                                    int32_t *ids, float *weights, void *out,
                                    moe_dtype out_dtype, void *stream);

/* moe_layer_forward_routed with x and out in host memory, for a layer
 * created with MOE_FLAG_HOST_IO: one call moves x (T * hidden elements of
 * x_dtype) to the device, runs the layer, and moves out back, all enqueued
 * on `stream`.  When the device can address a host buffer directly
 * (page-locked or registered memory, 16-byte aligned; on GB300 over the
 * NVLink-C2C link to the Grace host) and the call runs on a single-launch
 * decode kernel (up to 16 tokens), the kernel writes out through it, and
 * the one-token and batch kernels also take bf16 x from there (each CTA
 * copies its share into the layer's device buffer, so x crosses the link
 * once; fp32 x is read by every CTA at one token), so no copy is enqueued.
 * An x or out that is not taken that way (fp32 x above one token, other
 * kernels, memory the device cannot address) goes through the layer's
 * device buffers with cudaMemcpyAsync (page-locked buffers keep those
 * copies asynchronous).
 * Either way x_host and out_host must stay valid and
 * untouched until the stream has passed the call.  router_w,
 * logit_bias, ids and weights are device pointers as for
 * moe_layer_forward_routed.  MOE_ERR_INVALID_ARG for a layer without the
 * flag or a NULL host pointer; otherwise errors as for
 * moe_layer_forward_routed. */
moe_status moe_layer_forward_routed_host(moe_layer_t layer, const void *x_host, moe_dtype x_dtype,
                                         int32_t T, const float *router_w, const float *logit_bias,
                                         int64_t bias_row_stride, int32_t *ids, float *weights,
                                         void *out_host, moe_dtype out_dtype, void *stream);

/* Residual update and RMS normalisation between stacked layers (PocketLLM
 * design record, section 2: the residual stream is carried in fp32 and the
 * sublayer gets the narrow type):
 *   resid[t] += delta[t]   (skipped when delta is NULL)
 *   u[t] = bf16( resid[t] / sqrt(mean_c(resid[t][c]^2) + eps) )
 *   resid [T][H] fp32 in/out; delta [T][H] bf16 or fp32; u [T][H] bf16 out.
 * All three 16-byte aligned; H a multiple of 8; T >= 0. */
moe_status moe_residual_rmsnorm(float *resid, const void *delta, moe_dtype delta_dtype,
                                void *u, int32_t T, int32_t H, float eps, void *stream);

/* One step of a stack of layers on the fp32 residual stream: the residual
 * update and RMS normalisation above, then this layer routed and applied to
 * the normalised input (PocketLLM design record, section 2 for the residual
 * stream; the layer as for moe_layer_forward_routed):
 *   resid_out[t] = resid_in[t] + delta[t]   (delta NULL: resid_in[t])
 *   u_out[t]     = bf16( resid_out[t] / sqrt(mean_c(resid_out[t][c]^2) + eps) )
 *   ids, weights, out = the layer on u_out, as moe_layer_forward_routed.
 * resid_in, resid_out [T][H] fp32 (they must not overlap: resid_out is a
 * separate buffer, a caller stacking layers alternates two); delta [T][H]
 * bf16 or fp32 (the previous layer's out) or NULL; u_out [T][H] bf16.  Every
 * pointer is a device pointer, 16-byte aligned.  For one token on a layer
 * whose one-token kernel applies, the whole step is that kernel's single
 * launch (it forms u itself, with the same arithmetic as
 * moe_residual_rmsnorm, bit for bit); otherwise it is moe_residual_rmsnorm's
 * launch followed by moe_layer_forward_routed's.  Errors as for those two
 * calls; MOE_ERR_INVALID_ARG when resid_out overlaps resid_in or delta. */
moe_status moe_layer_forward_routed_resid(moe_layer_t layer, const float *resid_in, const void *delta,
                                          moe_dtype delta_dtype, float *resid_out, void *u_out, float eps,
                                          int32_t T, const float *router_w, const float *logit_bias,
                                          int64_t bias_row_stride, int32_t *ids, float *weights, void *out,
                                          moe_dtype out_dtype, void *stream);

/* Router for callers that cannot allocate device memory.  The paper has no
 * counterpart: this entry point exists for callers that may not call
 * cudaMalloc themselves or let a library do it -- code inside a host
 * framework that owns every device allocation, a stream-ordered pool that
 * must not grow, or a serving step that may not allocate once it is up.
 * It computes what moe_route computes (same arguments and layouts, no layer
 * object) on the CUDA-core router kernels; moe_route takes batches of 256
 * or more bf16 tokens (n_experts <= 128) to a tensor-core router instead.
 * Both select from fp32 logits, so their ids agree wherever a token's top
 * k+1 scores are further apart than the logits' rounding (~1e-6) and their
 * weights agree to about 1e-6.  Its fp32 logits scratch is a fixed
 * file-scope device array of 262,144 floats (1 MiB) that every GPU which
 * loads the library keeps until the process exits.
 *   T * n_experts > 262,144 returns MOE_ERR_UNSUPPORTED_SHAPE; nothing is
 *   allocated or freed.  The first call on a device (and the first after a
 *   cudaDeviceReset, which moves the array) looks up the array's device
 *   address (cudaGetSymbolAddress) and caches it, so make that first call
 *   before any stream capture.  Every call shares the one array: calls
 *   whose kernels overlap on the GPU (for example on two streams) race on
 *   it.  The scratch is fully written before it is read, so nothing needs
 *   clearing between calls. */
moe_status moe_route_noalloc(const void *x, moe_dtype x_dtype, int32_t T, int32_t hidden,
                             int32_t n_experts, int32_t top_k, float routed_scaling,
                             const float *router_w, const float *logit_bias,
                             int64_t bias_row_stride, int32_t *ids, float *weights,
                             void *stream);

/* Synchronise the device and report (then clear) the layer's sticky device
 * error: MOE_OK, MOE_ERR_BAD_EXPERT_ID, MOE_ERR_TIMEOUT or MOE_ERR_OVERFLOW
 * (batches of more than 8 tokens run on fp16 tensor-core operands; an input
 * or SwiGLU value beyond fp16 range is reported, never silently clipped). */
moe_status moe_layer_check(moe_layer_t layer);

/* Bytes of IQ4_NL weights held for the layer (routed + shared). */
int64_t moe_layer_weight_bytes(moe_layer_t layer);

/* Number of kernels this library has launched in the process so far (all
 * layers, all threads).  Diagnostics: lets a caller count launches per call. */
int64_t moe_launch_count(void);

/* Stage timing, a profiling aid (the pages have no counterpart).
 *
 * moe_layer_enable_timing(layer, calls) makes every later call of
 * moe_forward / moe_layer_forward_routed on `layer` record five CUDA events
 * on its stream into the next of `calls` slots (a ring): call start, start
 * of the up/gate grouped GEMM, its end, end of the down-projection grouped
 * GEMM, call end.  The single-launch decode path has no separate stages: it
 * reports its one kernel as the up/gate stage.  The events are recorded with
 * cudaEventRecordExternal, so inside stream capture they become event-record
 * nodes and every replay of the graph refreshes them; such an event stays
 * bound to the graph, so after capturing calls, destroy the graph and call
 * moe_layer_enable_timing again (0, or a new count: fresh events) before
 * calling the layer outside it (a reused slot otherwise fails with
 * MOE_ERR_CUDA).  calls = 0 disables timing and frees the events; calls must
 * be <= 4096.  Not safe while a call on the layer is in flight.
 *
 * moe_layer_stage_times(layer, ms, max_calls, n) synchronises on the events
 * and writes, for the n (<= max_calls) slots recorded since timing was
 * enabled (oldest first), four durations in milliseconds: routing + plan +
 * gather, up/gate, down, combine.  ms holds max_calls * 4 floats (host). */
moe_status moe_layer_enable_timing(moe_layer_t layer, int32_t calls);
moe_status moe_layer_stage_times(moe_layer_t layer, float *ms, int32_t max_calls, int32_t *n);

/* Test hook for the device-wait error path (no counterpart in the pages).
 *
 * moe_test_barrier_slack(layer, 1) makes the single-launch decode kernels
 * (batches of up to 8 tokens) expect one arrival more than their grid can
 * give at a device-wide wait (the multi-token kernel's wait for every CTA's
 * h; the one-token kernel's wait for the first selected expert's h), so that
 * the wait can never be met: every CTA polls up to its bounded limit (2^21 reads of the
 * counter, well under a minute), then finishes the call without the missing
 * arrival; moe_layer_check() returns MOE_ERR_TIMEOUT and the call's output
 * must not be used.  The layer stays usable: slack 0 restores normal calls.
 * Applies to calls enqueued after it returns (a captured graph keeps the
 * value it was captured with); the tensor-core path has no grid-wide wait
 * and ignores it.  MOE_ERR_INVALID_ARG for a NULL layer or a slack other
 * than 0 or 1. */
moe_status moe_test_barrier_slack(moe_layer_t layer, int32_t slack);

/* Static name of a status code. */
const char *moe_status_string(moe_status status);

/* Detail of the last error returned on the calling thread (static storage,
 * overwritten by the next failing call on that thread). */
const char *moe_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
