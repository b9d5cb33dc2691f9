// C ABI of libmoe_gb300 (declared in include/moe_gb300.h).
//
// Failure policy (PocketLLM design record, section 5: refuse at load rather
// than fail inside a request; EPQ model card, EPQ_REQUIRE_PAGER: fail loudly
// instead of falling back): create validates the shape and allocates every
// workspace for max_tokens up front; route and forward only validate their
// arguments (including base-pointer alignment for vector loads) and launch.
#include <algorithm>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <new>

#include "moe_internal.cuh"

using moe::Layer;

namespace moe {
static std::atomic<int64_t> g_launches{0};
void count_launches(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }
}  // namespace moe

namespace {

thread_local char g_err[512] = "";

moe_status fail(moe_status s, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return s;
}

}  // namespace

moe_status moe::report_error(moe_status s, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return s;
}

namespace {

moe_status cuda_fail(cudaError_t e, const char *where) {
  if (e == cudaErrorMemoryAllocation)
    return fail(MOE_ERR_OUT_OF_MEMORY, "%s: %s", where, cudaGetErrorString(e));
  return fail(MOE_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

#define MOE_CUDA(call, where)                  \
  do {                                         \
    cudaError_t e_ = (call);                   \
    if (e_ != cudaSuccess) return cuda_fail(e_, where); \
  } while (0)

int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

bool is_device_ptr(const void *p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

// Device address of a host buffer the device can read and write directly
// (page-locked or registered memory), or nullptr.
void *device_view(const void *host) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, host) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (a.type != cudaMemoryTypeHost) return nullptr;
  return a.devicePointer;
}

void free_layer(Layer *L) {
  if (!L) return;
  void *ptrs[] = {L->gu, L->dn, L->logits, L->offsets, L->active, L->route_token,
                  L->route_weight, L->h32, L->out_acc, L->err, L->sync, L->x16, L->h16,
                  L->tiles_ug, L->tiles_dn, L->tile_counts, L->ybuf, L->route_pos,
                  L->dense_ids, L->dense_w, L->rlog, L->x_stage, L->out_stage, L->hr,
                  L->hsh, L->useq, L->ulog, L->bseq, L->blog, L->bpart, L->bhq};
  for (void *p : ptrs)
    if (p) cudaFree(p);
  if (L->tev) {
    for (int i = 0; i < L->tev_slots * moe::kStageEvents; ++i) cudaEventDestroy(L->tev[i]);
    delete[] L->tev;
  }
  delete L;
}

// The stage-timing events of the call being issued, or nullptr.
cudaEvent_t *timing_slot(Layer *L) {
  return L->tev ? L->tev + (size_t)L->tev_next * moe::kStageEvents : nullptr;
}
void timing_advance(Layer *L) {
  if (!L->tev) return;
  L->tev_next = (L->tev_next + 1) % L->tev_slots;
  L->tev_used = std::min(L->tev_used + 1, L->tev_slots);
}
cudaError_t rec(cudaEvent_t e, cudaStream_t st) {
  return cudaEventRecordWithFlags(e, st, cudaEventRecordExternal);
}

moe_status check_x(const Layer *L, const void *x, moe_dtype xdt, int32_t T) {
  if (!L) return fail(MOE_ERR_INVALID_ARG, "layer is NULL");
  if (T < 0) return fail(MOE_ERR_INVALID_ARG, "T = %d is negative", T);
  if (T > L->max_tokens)
    return fail(MOE_ERR_TOO_MANY_TOKENS, "T = %d exceeds max_tokens = %d", T, L->max_tokens);
  if (xdt != MOE_DT_BF16 && xdt != MOE_DT_FP32)
    return fail(MOE_ERR_INVALID_ARG, "x_dtype %d is not MOE_DT_BF16 or MOE_DT_FP32", (int)xdt);
  if (T > 0 && !x) return fail(MOE_ERR_INVALID_ARG, "x is NULL");
  if (T > 0 && !moe::aligned(x, 16)) return fail(MOE_ERR_MISALIGNED, "x is not 16-byte aligned");
  return MOE_OK;
}

moe_status route_impl(Layer *L, const void *x, moe_dtype xdt, int32_t T, const float *wr,
                      const float *bias, int64_t bstride, int32_t *ids, float *w,
                      cudaStream_t st) {
  moe_status s = check_x(L, x, xdt, T);
  if (s != MOE_OK) return s;
  if (T == 0) return MOE_OK;
  if (!wr || !ids || !w) return fail(MOE_ERR_INVALID_ARG, "router_w, ids and weights must be non-NULL");
  if (!moe::aligned(wr, 16)) return fail(MOE_ERR_MISALIGNED, "router_w is not 16-byte aligned");
  if (!moe::aligned(ids, 4) || !moe::aligned(w, 4))
    return fail(MOE_ERR_MISALIGNED, "ids/weights are not 4-byte aligned");
  if (bias && bstride < 0) return fail(MOE_ERR_INVALID_ARG, "bias_row_stride is negative");
  int parts;
  if (moe::router_tc_supported(*L, xdt, T)) {  // large bf16 batches: tensor cores
    parts = moe::router_tc_parts(*L, T);
    MOE_CUDA(moe::launch_router_tc(*L, x, T, wr, L->logits, parts, st), "router logits");
  } else {
    parts = moe::router_parts(T, L->E, L->H, L->sms, 1 << 30);
    MOE_CUDA(moe::launch_router_logits(*L, x, xdt, T, wr, L->logits, parts, st), "router logits");
  }
  MOE_CUDA(moe::launch_router_topk(*L, L->logits, parts, bias, bstride, T, ids, w, st), "router top-k");
  return MOE_OK;
}

// ev: the call's stage-timing events (nullable); ev[0] was recorded by the
// caller when start_recorded.
moe_status forward_impl(Layer *L, const void *x, moe_dtype xdt, int32_t T, const int32_t *ids,
                        const float *w, void *out, moe_dtype odt, cudaStream_t st,
                        cudaEvent_t *ev = nullptr, bool start_recorded = false) {
  moe_status s = check_x(L, x, xdt, T);
  if (s != MOE_OK) return s;
  if (odt != MOE_DT_BF16 && odt != MOE_DT_FP32)
    return fail(MOE_ERR_INVALID_ARG, "out_dtype %d is not MOE_DT_BF16 or MOE_DT_FP32", (int)odt);
  if (T == 0) return MOE_OK;
  if (!ids || !w || !out) return fail(MOE_ERR_INVALID_ARG, "ids, weights and out must be non-NULL");
  if (!moe::aligned(ids, 4) || !moe::aligned(w, 4))
    return fail(MOE_ERR_MISALIGNED, "ids/weights are not 4-byte aligned");
  if (!moe::aligned(out, 16)) return fail(MOE_ERR_MISALIGNED, "out is not 16-byte aligned");
  if (ev && !start_recorded) MOE_CUDA(rec(ev[0], st), "timing event");
  const bool batch = moe::batch_decode_supported(*L, T);
  if (batch || moe::fused_decode_supported(*L, T)) {
    if (ev) MOE_CUDA(rec(ev[1], st), "timing event");
    if (batch)
      MOE_CUDA(moe::launch_decode_batch(*L, x, xdt, T, nullptr, nullptr, 0, ids, w, nullptr, nullptr, out, odt, st),
               "batch decode");
    else
      MOE_CUDA(moe::launch_decode_fused(*L, x, xdt, T, nullptr, nullptr, 0, ids, w, nullptr, nullptr,
                                        out, odt, st),
               "fused decode");
    if (ev) {
      MOE_CUDA(rec(ev[2], st), "timing event");
      MOE_CUDA(rec(ev[3], st), "timing event");
      MOE_CUDA(rec(ev[4], st), "timing event");
    }
    return MOE_OK;
  }
  // (the gather below also clears the fp32 output accumulator)
  const bool gemv = moe::gemv_mma_supported(*L, T);
  MOE_CUDA(moe::launch_route_plan(*L, ids, w, T, st, !gemv), "route plan");
  if (gemv) {
    MOE_CUDA(moe::launch_gather_x16(*L, x, xdt, T, st), "gather");
    MOE_CUDA(moe::launch_gemv_mma(*L, st, ev ? ev + 1 : nullptr), "batched decode expert GEMVs");
  } else {
    MOE_CUDA(moe::launch_prefill_tc(*L, x, xdt, T, st, ev ? ev + 1 : nullptr), "tensor-core expert GEMMs");
  }
  if (L->deterministic)
    MOE_CUDA(moe::launch_combine_ordered(*L, T, out, odt, st), "ordered combine");
  else
    MOE_CUDA(moe::launch_finalize(*L, T, out, odt, st), "finalize");
  if (ev) MOE_CUDA(rec(ev[4], st), "timing event");
  return MOE_OK;
}

}  // namespace

extern "C" {

const char *moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "MOE_ERR_UNSUPPORTED_SHAPE";
    case MOE_ERR_MISALIGNED: return "MOE_ERR_MISALIGNED";
    case MOE_ERR_OUT_OF_MEMORY: return "MOE_ERR_OUT_OF_MEMORY";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_BAD_EXPERT_ID: return "MOE_ERR_BAD_EXPERT_ID";
    case MOE_ERR_TOO_MANY_TOKENS: return "MOE_ERR_TOO_MANY_TOKENS";
    case MOE_ERR_OVERFLOW: return "MOE_ERR_OVERFLOW";
  }
  return "MOE_ERR_UNKNOWN";
}

const char *moe_last_error(void) { return g_err; }

int64_t moe_launch_count(void) { return moe::g_launches.load(std::memory_order_relaxed); }

moe_status moe_layer_create(const moe_shapes *sh, const moe_weights *wt, void *stream,
                            moe_layer_t *out) {
  if (!out) return fail(MOE_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (!sh || !wt) return fail(MOE_ERR_INVALID_ARG, "shapes and weights must be non-NULL");
  const int H = sh->hidden, E = sh->n_experts, k = sh->top_k, F = sh->expert_ffn, S = sh->n_shared;
  if (H < 32 || H > 16384 || H % 32) return fail(MOE_ERR_UNSUPPORTED_SHAPE, "hidden = %d: need a multiple of 32 in [32, 16384]", H);
  if (F < 32 || F > 16384 || F % 32) return fail(MOE_ERR_UNSUPPORTED_SHAPE, "expert_ffn = %d: need a multiple of 32 in [32, 16384]", F);
  if (E < 1 || E > 256) return fail(MOE_ERR_UNSUPPORTED_SHAPE, "n_experts = %d: need 1..256", E);
  if (k < 1 || k > 8 || k > E) return fail(MOE_ERR_UNSUPPORTED_SHAPE, "top_k = %d: need 1..min(n_experts, 8)", k);
  if (S != 0 && S != 1) return fail(MOE_ERR_UNSUPPORTED_SHAPE, "n_shared = %d: need 0 or 1", S);
  if (!(sh->routed_scaling > 0.f)) return fail(MOE_ERR_INVALID_ARG, "routed_scaling must be > 0");
  if (sh->max_tokens < 1 || sh->max_tokens > 65536) return fail(MOE_ERR_UNSUPPORTED_SHAPE, "max_tokens = %d: need 1..65536", sh->max_tokens);
  if (sh->flags & ~(MOE_FLAG_SELECTION_BIAS | MOE_FLAG_DETERMINISTIC | MOE_FLAG_HOST_IO | MOE_FLAG_COOPERATIVE))
    return fail(MOE_ERR_INVALID_ARG, "flags = 0x%x: unknown bits", sh->flags);
  if (!wt->up || !wt->gate || !wt->down) return fail(MOE_ERR_INVALID_ARG, "up, gate and down must be non-NULL");
  if (S && (!wt->sh_up || !wt->sh_gate || !wt->sh_down)) return fail(MOE_ERR_INVALID_ARG, "shared expert weights must be non-NULL when n_shared = 1");
  const void *wps[] = {wt->up, wt->gate, wt->down, S ? wt->sh_up : wt->up,
                       S ? wt->sh_gate : wt->up, S ? wt->sh_down : wt->up};
  for (const void *p : wps)
    if (!is_device_ptr(p)) return fail(MOE_ERR_INVALID_ARG, "expert weights must be device memory");

  Layer *L = new (std::nothrow) Layer();
  if (!L) return fail(MOE_ERR_OUT_OF_MEMORY, "host allocation failed");
  L->H = H; L->E = E; L->k = k; L->F = F; L->S = S;
  L->scale = sh->routed_scaling;
  L->sel_bias = (sh->flags & MOE_FLAG_SELECTION_BIAS) ? 1 : 0;
  L->deterministic = (sh->flags & MOE_FLAG_DETERMINISTIC) ? 1 : 0;
  L->coop = (sh->flags & MOE_FLAG_COOPERATIVE) ? 1 : 0;
  L->max_tokens = sh->max_tokens;
  L->Hp = (int)round_up(H, moe::kSBW);
  L->Fp = (int)round_up(F, moe::kSBW);
  L->gu_row_bytes = (int64_t)(L->Hp / moe::kSBW) * moe::kSBBytes;
  L->dn_row_bytes = (int64_t)(L->Fp / moe::kSBW) * moe::kSBBytes;
  L->gu_expert_bytes = 2 * (int64_t)L->Fp * L->gu_row_bytes;
  L->dn_expert_bytes = (int64_t)L->Hp * L->dn_row_bytes;
  L->weight_bytes = (int64_t)(E + S) * 3 * F * (H / 32) * 18;
  L->max_routes = sh->max_tokens * k + S * sh->max_tokens;
  cudaStream_t st = (cudaStream_t)stream;
  {
    cudaError_t e0 = cudaGetDevice(&L->device);
    if (e0 == cudaSuccess) e0 = cudaDeviceGetAttribute(&L->sms, cudaDevAttrMultiProcessorCount, L->device);
    // kernel attributes of this device, and whether the single-launch decode
    // grid can be resident at once
    if (e0 == cudaSuccess) e0 = moe::decode_prepare(*L);
    if (e0 == cudaSuccess && sh->max_tokens >= 2) e0 = moe::batch_decode_prepare(*L);
    if (e0 == cudaSuccess) e0 = moe::router_tc_prepare();
    if (e0 != cudaSuccess) {
      free_layer(L);
      return cuda_fail(e0, "moe_layer_create: device set-up");
    }
  }

#define ALLOC(ptr, bytes)                                                          \
  do {                                                                             \
    cudaError_t e_ = cudaMalloc((void **)&(ptr), (size_t)(bytes));                 \
    if (e_ != cudaSuccess) { free_layer(L); return cuda_fail(e_, "cudaMalloc " #ptr); } \
  } while (0)

  const int64_t gu_total = (int64_t)(E + S) * L->gu_expert_bytes;
  const int64_t dn_total = (int64_t)(E + S) * L->dn_expert_bytes;
  ALLOC(L->gu, gu_total);
  ALLOC(L->dn, dn_total);
  ALLOC(L->logits, sizeof(float) * moe::router_logits_floats(sh->max_tokens, E));
  ALLOC(L->offsets, sizeof(int) * (E + S + 1));
  ALLOC(L->active, sizeof(int) * (E + S + 1));
  ALLOC(L->route_token, sizeof(int) * (int64_t)L->max_routes);
  ALLOC(L->route_weight, sizeof(float) * (int64_t)L->max_routes);
  ALLOC(L->h32, sizeof(float) * (int64_t)std::min(sh->max_tokens, moe::kFusedMaxTokens) * (k + S) * L->Fp);
  if (L->unit_resident) {
    ALLOC(L->hr, sizeof(float) * (int64_t)k * L->Fp);
    ALLOC(L->hsh, sizeof(float) * (int64_t)L->Fp);
    ALLOC(L->useq, sizeof(unsigned long long) * moe::unit_decode_seq_words());
    ALLOC(L->ulog, sizeof(unsigned long long) * (int64_t)L->sms * E);
  }
  if (L->batch_smem_limit > 0) {
    ALLOC(L->bseq, sizeof(unsigned long long) * moe::batch_decode_seq_words());
    ALLOC(L->blog, sizeof(unsigned long long) * moe::batch_decode_log_words(*L));
    ALLOC(L->bpart, sizeof(float) * moe::batch_decode_part_floats(*L));
    ALLOC(L->bhq, sizeof(float) * moe::batch_decode_hq_floats());
  }
  ALLOC(L->out_acc, sizeof(float) * (int64_t)sh->max_tokens * H);
  ALLOC(L->err, sizeof(unsigned));
  ALLOC(L->sync, 4 * sizeof(unsigned));
  ALLOC(L->rlog, sizeof(unsigned long long) * moe::kLogitCopies * moe::kFusedMaxTokens * E);
  if (sh->flags & MOE_FLAG_HOST_IO) {
    ALLOC(L->x_stage, sizeof(float) * (int64_t)sh->max_tokens * H);
    ALLOC(L->out_stage, sizeof(float) * (int64_t)sh->max_tokens * H);
  }
  // batched tensor-core path (also taken by small batches whose shape the
  // single-launch decode kernel does not cover)
  ALLOC(L->x16, sizeof(__half) * (int64_t)L->max_routes * L->Hp);
  ALLOC(L->h16, sizeof(__half) * (int64_t)L->max_routes * L->Fp);
  ALLOC(L->tiles_ug, sizeof(moe::TcTile) * (int64_t)moe::tc_max_tiles(*L, true));
  ALLOC(L->tiles_dn, sizeof(moe::TcTile) * (int64_t)moe::tc_max_tiles(*L, false));
  ALLOC(L->tile_counts, 2 * sizeof(int));
  if (E == 1 && k == 1) {
    ALLOC(L->dense_ids, sizeof(int32_t) * (int64_t)sh->max_tokens);
    ALLOC(L->dense_w, sizeof(float) * (int64_t)sh->max_tokens);
  }
  if (L->deterministic) {
    ALLOC(L->ybuf, sizeof(float) * (int64_t)L->max_routes * L->Hp);
    ALLOC(L->route_pos, sizeof(int) * (int64_t)sh->max_tokens * k);
  }
#undef ALLOC

  cudaError_t e = cudaSuccess;
  if (e == cudaSuccess) e = cudaMemsetAsync(L->gu, 0, (size_t)gu_total, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(L->dn, 0, (size_t)dn_total, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(L->err, 0, sizeof(unsigned), st);
  if (e == cudaSuccess && L->dense_ids) {
    e = cudaMemsetAsync(L->dense_ids, 0, sizeof(int32_t) * (size_t)sh->max_tokens, st);
    if (e == cudaSuccess) e = moe::launch_fill(L->dense_w, 1.0f, sh->max_tokens, st);
  }
  if (e == cudaSuccess) e = cudaMemsetAsync(L->sync, 0, 4 * sizeof(unsigned), st);
  if (e == cudaSuccess && L->useq)
    e = cudaMemsetAsync(L->useq, 0, sizeof(unsigned long long) * moe::unit_decode_seq_words(), st);
  if (e == cudaSuccess && L->ulog)
    e = cudaMemsetAsync(L->ulog, 0, sizeof(unsigned long long) * (size_t)L->sms * E, st);
  if (e == cudaSuccess && L->bseq)
    e = cudaMemsetAsync(L->bseq, 0, sizeof(unsigned long long) * moe::batch_decode_seq_words(), st);
  if (e == cudaSuccess && L->blog)
    e = cudaMemsetAsync(L->blog, 0, sizeof(unsigned long long) * (size_t)moe::batch_decode_log_words(*L), st);
  if (e == cudaSuccess)
    e = cudaMemsetAsync(L->rlog, 0,
                        sizeof(unsigned long long) * moe::kLogitCopies * moe::kFusedMaxTokens * E, st);
  const int64_t up_bytes = (int64_t)F * (H / 32) * 18;
  const int64_t dn_bytes = (int64_t)H * (F / 32) * 18;
  for (int x = 0; x < E + S && e == cudaSuccess; ++x) {
    const bool shared = x == E;
    const uint8_t *up = shared ? (const uint8_t *)wt->sh_up : (const uint8_t *)wt->up + x * up_bytes;
    const uint8_t *gate = shared ? (const uint8_t *)wt->sh_gate : (const uint8_t *)wt->gate + x * up_bytes;
    const uint8_t *down = shared ? (const uint8_t *)wt->sh_down : (const uint8_t *)wt->down + x * dn_bytes;
    uint8_t *gu = L->gu + x * L->gu_expert_bytes;
    uint8_t *dn = L->dn + x * L->dn_expert_bytes;
    e = moe::launch_repack(gate, F, H, gu, L->gu_row_bytes, 2 * moe::kGroupRows, 0, st);
    if (e == cudaSuccess)
      e = moe::launch_repack(up, F, H, gu, L->gu_row_bytes, 2 * moe::kGroupRows, moe::kGroupRows, st);
    if (e == cudaSuccess) e = moe::launch_repack(down, H, F, dn, L->dn_row_bytes, 0, 0, st);
  }
  if (e == cudaSuccess) e = moe::tc_prepare(*L);
  if (e == cudaSuccess) e = moe::gemv_prepare(*L);
  if (e == cudaSuccess) e = moe::batch_decode_maps(*L);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) {
    free_layer(L);
    return cuda_fail(e, "moe_layer_create");
  }
  *out = reinterpret_cast<moe_layer_t>(L);
  return MOE_OK;
}

moe_status moe_layer_destroy(moe_layer_t layer) {
  if (!layer) return MOE_OK;
  cudaDeviceSynchronize();
  free_layer(reinterpret_cast<Layer *>(layer));
  return MOE_OK;
}

moe_status moe_route(moe_layer_t layer, const void *x, moe_dtype x_dtype, int32_t T,
                     const float *router_w, const float *logit_bias, int64_t bias_row_stride,
                     int32_t *ids, float *weights, void *stream) {
  return route_impl(reinterpret_cast<Layer *>(layer), x, x_dtype, T, router_w, logit_bias,
                    bias_row_stride, ids, weights, (cudaStream_t)stream);
}

moe_status moe_forward(moe_layer_t layer, const void *x, moe_dtype x_dtype, int32_t T,
                       const int32_t *ids, const float *weights, void *out, moe_dtype out_dtype,
                       void *stream) {
  Layer *L = reinterpret_cast<Layer *>(layer);
  cudaEvent_t *ev = (L && T > 0) ? timing_slot(L) : nullptr;
  moe_status r = forward_impl(L, x, x_dtype, T, ids, weights, out, out_dtype, (cudaStream_t)stream, ev);
  if (r == MOE_OK && ev) timing_advance(L);
  return r;
}

moe_status moe_dense_forward(moe_layer_t layer, const void *x, moe_dtype x_dtype, int32_t T,
                             void *out, moe_dtype out_dtype, void *stream) {
  Layer *L = reinterpret_cast<Layer *>(layer);
  if (!L) return fail(MOE_ERR_INVALID_ARG, "layer is NULL");
  if (!L->dense_ids)
    return fail(MOE_ERR_INVALID_ARG, "moe_dense_forward needs a layer with n_experts = 1 and top_k = 1 (got %d, %d)",
                L->E, L->k);
  cudaEvent_t *ev = T > 0 ? timing_slot(L) : nullptr;
  moe_status r = forward_impl(L, x, x_dtype, T, L->dense_ids, L->dense_w, out, out_dtype,
                              (cudaStream_t)stream, ev);
  if (r == MOE_OK && ev) timing_advance(L);
  return r;
}

// moe_layer_forward_routed; x_import as for launch_decode_fused and
// launch_decode_batch (the host-buffer call passes it, nullptr otherwise)
static moe_status forward_routed_impl(moe_layer_t layer, const void *x, moe_dtype x_dtype, int32_t T,
                                      const float *router_w, const float *logit_bias, int64_t bias_row_stride,
                                      int32_t *ids, float *weights, void *out, moe_dtype out_dtype, void *stream,
                                      void *x_import) {
  Layer *L = reinterpret_cast<Layer *>(layer);
  cudaStream_t st = (cudaStream_t)stream;
  if (out_dtype != MOE_DT_BF16 && out_dtype != MOE_DT_FP32)
    return fail(MOE_ERR_INVALID_ARG, "out_dtype %d is not MOE_DT_BF16 or MOE_DT_FP32", (int)out_dtype);
  if (T > 0 && !out) return fail(MOE_ERR_INVALID_ARG, "out is NULL");
  if (T > 0 && out && !moe::aligned(out, 16)) return fail(MOE_ERR_MISALIGNED, "out is not 16-byte aligned");
  if (L && T > 0 && T <= L->max_tokens && (moe::batch_decode_supported(*L, T) || moe::fused_decode_supported(*L, T))) {
    moe_status s = check_x(L, x, x_dtype, T);
    if (s != MOE_OK) return s;
    if (!router_w || !ids || !weights) return fail(MOE_ERR_INVALID_ARG, "router_w, ids and weights must be non-NULL");
    if (!moe::aligned(router_w, 16)) return fail(MOE_ERR_MISALIGNED, "router_w is not 16-byte aligned");
    if (!moe::aligned(ids, 4) || !moe::aligned(weights, 4))
      return fail(MOE_ERR_MISALIGNED, "ids/weights are not 4-byte aligned");
    if (logit_bias && bias_row_stride < 0) return fail(MOE_ERR_INVALID_ARG, "bias_row_stride is negative");
    cudaEvent_t *ev = timing_slot(L);
    if (ev) {
      MOE_CUDA(rec(ev[0], st), "timing event");
      MOE_CUDA(rec(ev[1], st), "timing event");
    }
    if (moe::batch_decode_supported(*L, T))
      MOE_CUDA(moe::launch_decode_batch(*L, x, x_dtype, T, router_w, logit_bias, bias_row_stride, nullptr, nullptr,
                                        ids, weights, out, out_dtype, st, x_import),
               "batch decode");
    else
      MOE_CUDA(moe::launch_decode_fused(*L, x, x_dtype, T, router_w, logit_bias, bias_row_stride, nullptr,
                                        nullptr, ids, weights, out, out_dtype, st, x_import),
               "fused decode");
    if (ev) {
      MOE_CUDA(rec(ev[2], st), "timing event");
      MOE_CUDA(rec(ev[3], st), "timing event");
      MOE_CUDA(rec(ev[4], st), "timing event");
      timing_advance(L);
    }
    return MOE_OK;
  }
  cudaEvent_t *ev = (L && T > 0) ? timing_slot(L) : nullptr;
  if (ev) MOE_CUDA(rec(ev[0], st), "timing event");
  moe_status s = route_impl(L, x, x_dtype, T, router_w, logit_bias, bias_row_stride, ids, weights, st);
  if (s != MOE_OK) return s;
  s = forward_impl(L, x, x_dtype, T, ids, weights, out, out_dtype, st, ev, true);
  if (s == MOE_OK && ev) timing_advance(L);
  return s;
}

moe_status moe_layer_forward_routed(moe_layer_t layer, const void *x, moe_dtype x_dtype,
                                    int32_t T, const float *router_w, const float *logit_bias,
                                    int64_t bias_row_stride, int32_t *ids, float *weights,
                                    void *out, moe_dtype out_dtype, void *stream) {
  return forward_routed_impl(layer, x, x_dtype, T, router_w, logit_bias, bias_row_stride, ids, weights, out,
                             out_dtype, stream, nullptr);
}

moe_status moe_layer_forward_routed_host(moe_layer_t layer, const void *x_host, moe_dtype x_dtype,
                                         int32_t T, const float *router_w, const float *logit_bias,
                                         int64_t bias_row_stride, int32_t *ids, float *weights,
                                         void *out_host, moe_dtype out_dtype, void *stream) {
  Layer *L = reinterpret_cast<Layer *>(layer);
  if (!L) return fail(MOE_ERR_INVALID_ARG, "layer is NULL");
  if (!L->x_stage || !L->out_stage)
    return fail(MOE_ERR_INVALID_ARG, "the layer was not created with MOE_FLAG_HOST_IO");
  if (x_dtype != MOE_DT_BF16 && x_dtype != MOE_DT_FP32)
    return fail(MOE_ERR_INVALID_ARG, "x_dtype %d is not MOE_DT_BF16 or MOE_DT_FP32", (int)x_dtype);
  if (out_dtype != MOE_DT_BF16 && out_dtype != MOE_DT_FP32)
    return fail(MOE_ERR_INVALID_ARG, "out_dtype %d is not MOE_DT_BF16 or MOE_DT_FP32", (int)out_dtype);
  if (T < 0) return fail(MOE_ERR_INVALID_ARG, "T = %d is negative", T);
  if (T > L->max_tokens)
    return fail(MOE_ERR_TOO_MANY_TOKENS, "T = %d exceeds max_tokens = %d", T, L->max_tokens);
  if (T == 0) return MOE_OK;
  if (!x_host || !out_host) return fail(MOE_ERR_INVALID_ARG, "x_host and out_host must be non-NULL");
  cudaStream_t st = (cudaStream_t)stream;
  const size_t n = (size_t)T * L->H;
  // The single-launch decode kernels (up to 16 tokens) store each output
  // element once, so they write out through the host buffer itself when the
  // device can address it (page-locked memory; on GB300 over the NVLink-C2C
  // link to the Grace host): no copy-engine round trip after the kernel.
  // The one-token and batch kernels also take x from there, so a step is
  // one launch: bf16 x crosses the link once, each CTA bringing its share
  // into the layer's device buffer (every CTA needs all of x; 152 reads of
  // it over the link cost 5 us more per call at one token).  fp32 x is read
  // by every CTA at one token and copied in above it, as is x for the
  // multi-token kernel of other shapes.
  void *od = nullptr;
  if (moe::batch_decode_supported(*L, T) || moe::fused_decode_supported(*L, T)) {
    od = device_view(out_host);
    if (od && !moe::aligned(od, 16)) od = nullptr;
  }
  const bool bf16 = x_dtype == MOE_DT_BF16;
  if (od && ((T == 1 && moe::unit_decode_supported(*L)) || (bf16 && moe::batch_decode_supported(*L, T)))) {
    void *xd = device_view(x_host);
    if (xd && moe::aligned(xd, 16))
      return forward_routed_impl(layer, xd, x_dtype, T, router_w, logit_bias, bias_row_stride, ids, weights, od,
                                 out_dtype, stream, bf16 ? L->x_stage : nullptr);
  }
  MOE_CUDA(cudaMemcpyAsync(L->x_stage, x_host, n * (x_dtype == MOE_DT_BF16 ? 2 : 4), cudaMemcpyHostToDevice, st),
           "copy x to the device");
  const moe_status s = moe_layer_forward_routed(layer, L->x_stage, x_dtype, T, router_w, logit_bias,
                                                bias_row_stride, ids, weights, od ? od : L->out_stage, out_dtype,
                                                stream);
  if (s != MOE_OK || od) return s;
  MOE_CUDA(cudaMemcpyAsync(out_host, L->out_stage, n * (out_dtype == MOE_DT_BF16 ? 2 : 4),
                           cudaMemcpyDeviceToHost, st),
           "copy out to the host");
  return MOE_OK;
}

moe_status moe_residual_rmsnorm(float *resid, const void *delta, moe_dtype delta_dtype, void *u,
                                int32_t T, int32_t H, float eps, void *stream) {
  if (T < 0 || H <= 0 || H % 8) return fail(MOE_ERR_INVALID_ARG, "need T >= 0 and H a positive multiple of 8");
  if (delta_dtype != MOE_DT_BF16 && delta_dtype != MOE_DT_FP32)
    return fail(MOE_ERR_INVALID_ARG, "delta_dtype %d is not MOE_DT_BF16 or MOE_DT_FP32", (int)delta_dtype);
  if (!(eps >= 0.f)) return fail(MOE_ERR_INVALID_ARG, "eps must be >= 0");
  if (T == 0) return MOE_OK;
  if (!resid || !u) return fail(MOE_ERR_INVALID_ARG, "resid and u must be non-NULL");
  if (!moe::aligned(resid, 16) || !moe::aligned(u, 16) || (delta && !moe::aligned(delta, 16)))
    return fail(MOE_ERR_MISALIGNED, "resid, delta and u must be 16-byte aligned");
  MOE_CUDA(moe::launch_residual_rmsnorm(resid, delta, delta_dtype, resid, u, T, H, eps, (cudaStream_t)stream),
           "residual rmsnorm");
  return MOE_OK;
}

moe_status moe_layer_forward_routed_resid(moe_layer_t layer, const float *resid_in, const void *delta,
                                          moe_dtype delta_dtype, float *resid_out, void *u_out, float eps,
                                          int32_t T, const float *router_w, const float *logit_bias,
                                          int64_t bias_row_stride, int32_t *ids, float *weights, void *out,
                                          moe_dtype out_dtype, void *stream) {
  Layer *L = reinterpret_cast<Layer *>(layer);
  if (!L) return fail(MOE_ERR_INVALID_ARG, "layer is NULL");
  if (T < 0) return fail(MOE_ERR_INVALID_ARG, "T = %d is negative", T);
  if (T > L->max_tokens) return fail(MOE_ERR_TOO_MANY_TOKENS, "T = %d exceeds max_tokens = %d", T, L->max_tokens);
  if (delta_dtype != MOE_DT_BF16 && delta_dtype != MOE_DT_FP32)
    return fail(MOE_ERR_INVALID_ARG, "delta_dtype %d is not MOE_DT_BF16 or MOE_DT_FP32", (int)delta_dtype);
  if (!(eps >= 0.f)) return fail(MOE_ERR_INVALID_ARG, "eps must be >= 0");
  if (out_dtype != MOE_DT_BF16 && out_dtype != MOE_DT_FP32)
    return fail(MOE_ERR_INVALID_ARG, "out_dtype %d is not MOE_DT_BF16 or MOE_DT_FP32", (int)out_dtype);
  if (L->H % 8) return fail(MOE_ERR_UNSUPPORTED_SHAPE, "hidden %d is not a multiple of 8", L->H);
  if (T == 0) return MOE_OK;
  if (!resid_in || !resid_out || !u_out || !out || !router_w || !ids || !weights)
    return fail(MOE_ERR_INVALID_ARG, "resid_in, resid_out, u_out, out, router_w, ids and weights must be non-NULL");
  const size_t rb = sizeof(float) * (size_t)T * L->H;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(resid_in), b0 = reinterpret_cast<uintptr_t>(resid_out);
  if (a0 < b0 + rb && b0 < a0 + rb) return fail(MOE_ERR_INVALID_ARG, "resid_in and resid_out overlap");
  if (delta) {
    const size_t db = (delta_dtype == MOE_DT_BF16 ? 2 : 4) * (size_t)T * L->H;
    const uintptr_t d0 = reinterpret_cast<uintptr_t>(delta);
    if (d0 < b0 + rb && b0 < d0 + db) return fail(MOE_ERR_INVALID_ARG, "delta and resid_out overlap");
  }
  if (!moe::aligned(resid_in, 16) || !moe::aligned(resid_out, 16) || !moe::aligned(u_out, 16) ||
      (delta && !moe::aligned(delta, 16)) || !moe::aligned(out, 16) || !moe::aligned(router_w, 16))
    return fail(MOE_ERR_MISALIGNED, "resid_in, delta, resid_out, u_out, out and router_w must be 16-byte aligned");
  if (!moe::aligned(ids, 4) || !moe::aligned(weights, 4))
    return fail(MOE_ERR_MISALIGNED, "ids/weights are not 4-byte aligned");
  if (logit_bias && bias_row_stride < 0) return fail(MOE_ERR_INVALID_ARG, "bias_row_stride is negative");
  cudaStream_t st = (cudaStream_t)stream;
  if (T == 1 && moe::unit_decode_supported(*L)) {
    const moe::ResidStep rs{resid_in, delta, delta_dtype == MOE_DT_BF16 ? 1 : 0, resid_out,
                            reinterpret_cast<__nv_bfloat16 *>(u_out), eps};
    MOE_CUDA(moe::launch_decode_unit(*L, u_out, MOE_DT_BF16, router_w, logit_bias, nullptr, nullptr, ids, weights,
                                     out, out_dtype, st, &rs),
             "one-token decode");
    return MOE_OK;
  }
  MOE_CUDA(moe::launch_residual_rmsnorm(resid_in, delta, delta_dtype, resid_out, u_out, T, L->H, eps, st),
           "residual rmsnorm");
  return moe_layer_forward_routed(layer, u_out, MOE_DT_BF16, T, router_w, logit_bias, bias_row_stride, ids,
                                  weights, out, out_dtype, stream);
}

moe_status moe_layer_enable_timing(moe_layer_t layer, int32_t calls) {
  Layer *L = reinterpret_cast<Layer *>(layer);
  if (!L) return fail(MOE_ERR_INVALID_ARG, "layer is NULL");
  if (calls < 0 || calls > 4096) return fail(MOE_ERR_INVALID_ARG, "calls = %d: need 0..4096", calls);
  if (L->tev) {
    for (int i = 0; i < L->tev_slots * moe::kStageEvents; ++i) cudaEventDestroy(L->tev[i]);
    delete[] L->tev;
    L->tev = nullptr;
  }
  L->tev_slots = L->tev_next = L->tev_used = 0;
  if (calls == 0) return MOE_OK;
  const int n = calls * moe::kStageEvents;
  cudaEvent_t *ev = new cudaEvent_t[n];
  for (int i = 0; i < n; ++i) {
    const cudaError_t e = cudaEventCreate(&ev[i]);
    if (e != cudaSuccess) {
      for (int j = 0; j < i; ++j) cudaEventDestroy(ev[j]);
      delete[] ev;
      return cuda_fail(e, "cudaEventCreate");
    }
  }
  L->tev = ev;
  L->tev_slots = calls;
  return MOE_OK;
}

moe_status moe_layer_stage_times(moe_layer_t layer, float *ms, int32_t max_calls, int32_t *n) {
  Layer *L = reinterpret_cast<Layer *>(layer);
  if (!L || !n || (max_calls > 0 && !ms) || max_calls < 0)
    return fail(MOE_ERR_INVALID_ARG, "layer, n and ms must be non-NULL, max_calls >= 0");
  const int used = std::min(L->tev_used, (int)max_calls);
  const int first = (L->tev_next - L->tev_used + L->tev_slots) % std::max(L->tev_slots, 1);
  for (int i = 0; i < used; ++i) {
    const cudaEvent_t *ev = L->tev + (size_t)((first + i) % L->tev_slots) * moe::kStageEvents;
    MOE_CUDA(cudaEventSynchronize(ev[moe::kStageEvents - 1]), "timing event");
    for (int k = 0; k + 1 < moe::kStageEvents; ++k)
      MOE_CUDA(cudaEventElapsedTime(&ms[(size_t)i * 4 + k], ev[k], ev[k + 1]), "timing event");
  }
  *n = used;
  return MOE_OK;
}

moe_status moe_test_barrier_slack(moe_layer_t layer, int32_t slack) {
  Layer *L = reinterpret_cast<Layer *>(layer);
  if (!L) return fail(MOE_ERR_INVALID_ARG, "layer is NULL");
  if (slack < 0 || slack > 1) return fail(MOE_ERR_INVALID_ARG, "slack = %d: need 0 or 1", slack);
  L->barrier_slack = slack;
  return MOE_OK;
}

moe_status moe_layer_check(moe_layer_t layer) {
  Layer *L = reinterpret_cast<Layer *>(layer);
  if (!L) return fail(MOE_ERR_INVALID_ARG, "layer is NULL");
  MOE_CUDA(cudaDeviceSynchronize(), "moe_layer_check");
  unsigned err = 0;
  MOE_CUDA(cudaMemcpy(&err, L->err, sizeof(unsigned), cudaMemcpyDeviceToHost), "read error word");
  MOE_CUDA(cudaMemset(L->err, 0, sizeof(unsigned)), "clear error word");
  if (err & moe::kErrTimeout) return fail(MOE_ERR_TIMEOUT, "a bounded device wait gave up");
  if (err & moe::kErrOverflow) return fail(MOE_ERR_OVERFLOW, "an activation left fp16 range on the tensor-core path");
  if (err & moe::kErrBadId) return fail(MOE_ERR_BAD_EXPERT_ID, "an expert id outside [0, E) reached moe_forward");
  return MOE_OK;
}

int64_t moe_layer_weight_bytes(moe_layer_t layer) {
  Layer *L = reinterpret_cast<Layer *>(layer);
  return L ? L->weight_bytes : -1;
}

}  // extern "C"
