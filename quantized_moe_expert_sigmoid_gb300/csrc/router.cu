// Sigmoid top-k router (HelloSun/xing4_0-29b-IQ4_NL_EPQ model card, "模型與路由":
// expert_gating_func = sigmoid, expert_weights_norm = yes, expert_weights_scale
// = 2.0, 4 of 64 experts; the router matrix ffn_gate_inp is fp32).
//
// Step 1 (logits): l[t][e] = x[t] . Wr[e] + b[t][e], fp32 accumulation.
//   - small T: one warp per expert streams its Wr row once with 128-bit loads
//     and serves every token (Wr is read from HBM exactly once);
//   - large T: a 32-token x 64-expert register-tiled SIMT product through
//     shared memory (Wr rows are reused by 32 tokens per tile), the next K
//     chunk's global loads overlapping the current chunk's FMAs.
// Step 2 (selection): one warp per token; the k largest logits are taken in
// descending order (sigmoid is monotone, so this is the order of the
// scores), equal logits going to the lower id; s = 1/(1+e^-l) for the k
// selected; w = scale * s / sum(s).
#include <float.h>

#include <algorithm>

#include <cudaTypedefs.h>

#include <mutex>

#include "device_utils.cuh"
#include "moe_internal.cuh"

namespace moe {
namespace {

template <typename XT>
__device__ __forceinline__ float4 load_x4(const XT *p);

template <>
__device__ __forceinline__ float4 load_x4<float>(const float *p) {
  return *reinterpret_cast<const float4 *>(p);
}

template <>
__device__ __forceinline__ float4 load_x4<__nv_bfloat16>(const __nv_bfloat16 *p) {
  const uint2 v = *reinterpret_cast<const uint2 *>(p);
  float4 r;
  r.x = __uint_as_float(v.x << 16);
  r.y = __uint_as_float(v.x & 0xFFFF0000u);
  r.z = __uint_as_float(v.y << 16);
  r.w = __uint_as_float(v.y & 0xFFFF0000u);
  return r;
}

constexpr int kSmallTokens = 4;  // tokens per pass in the small-T kernel

template <typename XT>
__global__ void __launch_bounds__(256) router_logits_small(const XT *__restrict__ x, int T, int H,
                                                           const float *__restrict__ wr, int E,
                                                           const float *__restrict__ bias,
                                                           int64_t bstride,
                                                           float *__restrict__ logits) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * 8 + warp;
  pdl_wait();  // x may come from the previous launch
  pdl_launch_dependents();
  if (e >= E) return;
  const float *w = wr + (int64_t)e * H;
  for (int t0 = 0; t0 < T; t0 += kSmallTokens) {
    float acc[kSmallTokens];
#pragma unroll
    for (int i = 0; i < kSmallTokens; ++i) acc[i] = 0.f;
    for (int c = lane * 4; c < H; c += 128) {
      const float4 wv = *reinterpret_cast<const float4 *>(w + c);
#pragma unroll
      for (int i = 0; i < kSmallTokens; ++i) {
        if (t0 + i < T) {
          const float4 xv = load_x4<XT>(x + (int64_t)(t0 + i) * H + c);
          acc[i] = fmaf(xv.x, wv.x, acc[i]);
          acc[i] = fmaf(xv.y, wv.y, acc[i]);
          acc[i] = fmaf(xv.z, wv.z, acc[i]);
          acc[i] = fmaf(xv.w, wv.w, acc[i]);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < kSmallTokens; ++i) {
      float v = acc[i];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0 && t0 + i < T) {
        if (bias) v += bias[(int64_t)(t0 + i) * bstride + e];
        logits[(int64_t)(t0 + i) * E + e] = v;
      }
    }
  }
}

constexpr int kTM = 32, kTN = 64, kKC = 32;

// 32 tokens x 64 experts per CTA, 256 threads of 2 tokens x 4 experts.  The
// next K chunk's x and Wr values are loaded into registers while the current
// chunk is multiplied out of shared memory, so the global latency is paid
// once, not once per chunk.  x is kept token-major and Wr transposed to
// k-major in shared memory: every inner step is two 16-byte x reads
// (broadcast within the warp) and four 16-byte Wr reads for 32 FMAs.
// blockIdx.z = K part: columns [z*kc, (z+1)*kc) of H; part z's partial sums
// go to logits + z * T * E (a bias, if given, with part 0), summed by the
// top-k kernel in part order.  Splitting K gives several CTAs per SM at
// prefill sizes.
template <typename XT>
__global__ void __launch_bounds__(256) router_logits_tiled(const XT *__restrict__ x, int T, int H,
                                                           const float *__restrict__ wr, int E,
                                                           const float *__restrict__ bias,
                                                           int64_t bstride, int kc,
                                                           float *__restrict__ logits) {
  __shared__ __align__(16) float xs[kTM][kKC + 4];
  __shared__ __align__(16) float ws[kKC][kTN + 4];
  const int tid = threadIdx.x;
  const int ty = tid >> 4, tx = tid & 15;  // tokens 2ty, 2ty+1; experts 4tx .. 4tx+3
  const int t0 = blockIdx.x * kTM, e0 = blockIdx.y * kTN;
  // load mapping: x token lt, k offset lk (4 values); Wr expert le, k offset lw (8 values)
  const int lt = tid >> 3, lk = (tid & 7) * 4;
  const int le = tid & 63, lw = (tid >> 6) * 8;
  const bool xv_ok = t0 + lt < T, wv_ok = e0 + le < E;
  const XT *xp = x + (int64_t)(t0 + lt) * H + lk;
  const float *wp = wr + (int64_t)(e0 + le) * H + lw;
  const int kb = blockIdx.z * kc, ke = min(H, kb + kc);
  pdl_wait();  // x may come from the previous launch
  pdl_launch_dependents();
  logits += (int64_t)blockIdx.z * T * E;
  if (blockIdx.z != 0) bias = nullptr;
  float4 xr = make_float4(0.f, 0.f, 0.f, 0.f), wr0 = xr, wr1 = xr;
  if (kb < ke) {
    if (xv_ok) xr = load_x4<XT>(xp + kb);
    if (wv_ok) {
      wr0 = *reinterpret_cast<const float4 *>(wp + kb);
      wr1 = *reinterpret_cast<const float4 *>(wp + kb + 4);
    }
  }
  float acc[2][4] = {};
  for (int k0 = kb; k0 < ke; k0 += kKC) {
    *reinterpret_cast<float4 *>(&xs[lt][lk]) = xr;
    ws[lw + 0][le] = wr0.x;
    ws[lw + 1][le] = wr0.y;
    ws[lw + 2][le] = wr0.z;
    ws[lw + 3][le] = wr0.w;
    ws[lw + 4][le] = wr1.x;
    ws[lw + 5][le] = wr1.y;
    ws[lw + 6][le] = wr1.z;
    ws[lw + 7][le] = wr1.w;
    __syncthreads();
    if (k0 + kKC < ke) {  // next chunk in flight during this one's FMAs
      if (xv_ok) xr = load_x4<XT>(xp + k0 + kKC);
      if (wv_ok) {
        wr0 = *reinterpret_cast<const float4 *>(wp + k0 + kKC);
        wr1 = *reinterpret_cast<const float4 *>(wp + k0 + kKC + 4);
      }
    }
#pragma unroll
    for (int kk = 0; kk < kKC; kk += 4) {
      const float4 a0 = *reinterpret_cast<const float4 *>(&xs[2 * ty][kk]);
      const float4 a1 = *reinterpret_cast<const float4 *>(&xs[2 * ty + 1][kk]);
      const float av0[4] = {a0.x, a0.y, a0.z, a0.w}, av1[4] = {a1.x, a1.y, a1.z, a1.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float4 b = *reinterpret_cast<const float4 *>(&ws[kk + j][tx * 4]);
        acc[0][0] = fmaf(av0[j], b.x, acc[0][0]);
        acc[0][1] = fmaf(av0[j], b.y, acc[0][1]);
        acc[0][2] = fmaf(av0[j], b.z, acc[0][2]);
        acc[0][3] = fmaf(av0[j], b.w, acc[0][3]);
        acc[1][0] = fmaf(av1[j], b.x, acc[1][0]);
        acc[1][1] = fmaf(av1[j], b.y, acc[1][1]);
        acc[1][2] = fmaf(av1[j], b.z, acc[1][2]);
        acc[1][3] = fmaf(av1[j], b.w, acc[1][3]);
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int t = t0 + ty * 2 + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + tx * 4 + j;
      if (e >= E) continue;
      float v = acc[i][j];
      if (bias) v += bias[(int64_t)t * bstride + e];
      logits[(int64_t)t * E + e] = v;
    }
  }
}

// One warp per token.  E <= 256: lane holds experts lane + 32*i, i < 8.
// The logits are the sum of `parts` K-partial arrays, added in part order,
// plus the optional bias b[t][e] (row stride bstride; 0 = one row for all).
__global__ void __launch_bounds__(256) router_topk_kernel(const float *__restrict__ logits, int parts,
                                                          const float *__restrict__ bias,
                                                          int64_t bstride, int T, int E, int k,
                                                          float scale, int sel,
                                                          int32_t *__restrict__ ids,
                                                          float *__restrict__ weights) {
  const int lane = threadIdx.x & 31;
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  pdl_wait();  // the logits come from the previous launch
  pdl_launch_dependents();
  if (t >= T) return;
  // selection key per expert: the biased logit (logit mode), or the sigmoid
  // score plus the bias (selection mode, whose weights use the plain score)
  float v[8], lraw[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = lane + 32 * i;
    float l = -FLT_MAX, key = -FLT_MAX;
    if (e < E) {
      // the K-split parts, added in part order; unrolled so that their
      // loads are in flight together
      l = 0.f;
      for (int z0 = 0; z0 < parts; z0 += kRouterMaxParts) {
        float pz[kRouterMaxParts];
#pragma unroll
        for (int z = 0; z < kRouterMaxParts; ++z)
          pz[z] = z0 + z < parts ? logits[(int64_t)(z0 + z) * T * E + (int64_t)t * E + e] : 0.f;
#pragma unroll
        for (int z = 0; z < kRouterMaxParts; ++z)
          if (z0 + z < parts) l = (z0 + z == 0) ? pz[z] : l + pz[z];
      }
      const float b = bias ? bias[(int64_t)t * bstride + e] : 0.f;
      if (sel) {
        key = 1.0f / (1.0f + expf(-l)) + b;
      } else {
        l += b;
        key = l;
      }
    }
    lraw[i] = (l == l) ? l : -FLT_MAX;
    v[i] = (key == key) ? key : -FLT_MAX;  // NaN never wins
  }
  unsigned taken = 0;
  int my_id = 0;
  float my_s = 0.f, ssum = 0.f;
  for (int j = 0; j < k; ++j) {
    float best = -INFINITY;
    int bid = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !((taken >> i) & 1u) && (v[i] > best || (v[i] == best && e < bid))) {
        best = v[i];
        bid = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ob = __shfl_xor_sync(0xffffffffu, best, o);
      const int oid = __shfl_xor_sync(0xffffffffu, bid, o);
      if (ob > best || (ob == best && oid < bid)) {
        best = ob;
        bid = oid;
      }
    }
    if ((bid & 31) == lane) taken |= 1u << (bid >> 5);
    // the winner's logit, from the lane that holds it
    float lw = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (i == (bid >> 5)) lw = lraw[i];
    lw = __shfl_sync(0xffffffffu, lw, bid & 31);
    const float s = 1.0f / (1.0f + expf(-lw));
    ssum += s;
    if (lane == j) {
      my_id = bid;
      my_s = s;
    }
  }
  if (lane < k) {
    ids[(int64_t)t * k + lane] = my_id;
    weights[(int64_t)t * k + lane] = scale * my_s / ssum;
  }
}

}  // namespace

int router_parts(int T, int E, int H, int sms, int max_parts) {
  if (T <= 16) return 1;
  const int cap = T <= kRouterSmallT ? kRouterMaxPartsSmall : kRouterMaxParts;
  const int tiles = ((T + kTM - 1) / kTM) * ((E + kTN - 1) / kTN);
  const int nkc = (H + kKC - 1) / kKC;  // 32-wide K chunks
  const int want = std::max(kRouterMaxParts, std::max(1, sms) / tiles);
  return std::max(1, std::min(std::min(want, cap), std::min(max_parts, nkc)));
}

cudaError_t launch_router_logits(const Layer &L, const void *x, moe_dtype xdt, int T,
                                 const float *wr, float *logits, int parts, cudaStream_t stream) {
  const float *bias = nullptr;  // added by the top-k kernel
  const int64_t bias_stride = 0;
  if (T <= 16) {
    dim3 grid((L.E + 7) / 8);
    if (xdt == MOE_DT_BF16)
      return count_and_check(launch_pdl(router_logits_small<__nv_bfloat16>, grid, dim3(256), 0, stream,
                                        (const __nv_bfloat16 *)x, T, L.H, wr, L.E, bias, bias_stride, logits));
    else
      return count_and_check(launch_pdl(router_logits_small<float>, grid, dim3(256), 0, stream, (const float *)x,
                                        T, L.H, wr, L.E, bias, bias_stride, logits));
  } else {
    const int kc = ((L.H + parts - 1) / parts + kKC - 1) / kKC * kKC;
    dim3 grid((T + kTM - 1) / kTM, (L.E + kTN - 1) / kTN, parts);
    if (xdt == MOE_DT_BF16)
      return count_and_check(launch_pdl(router_logits_tiled<__nv_bfloat16>, grid, dim3(256), 0, stream,
                                        (const __nv_bfloat16 *)x, T, L.H, wr, L.E, bias, bias_stride, kc,
                                        logits));
    else
      return count_and_check(launch_pdl(router_logits_tiled<float>, grid, dim3(256), 0, stream, (const float *)x,
                                        T, L.H, wr, L.E, bias, bias_stride, kc, logits));
  }
}

cudaError_t launch_router_topk(const Layer &L, const float *logits, int parts, const float *bias,
                               int64_t bias_stride, int T, int32_t *ids, float *weights,
                               cudaStream_t stream) {
  const int warps_per_block = 8;
  const int blocks = (T + warps_per_block - 1) / warps_per_block;
  return count_and_check(launch_pdl(router_topk_kernel, dim3(blocks), dim3(32 * warps_per_block), 0, stream,
                                    logits, parts, bias, bias_stride, T, L.E, L.k, L.scale, L.sel_bias, ids,
                                    weights));
}

}  // namespace moe

// ---------------------------------------------------------------------------
// Router for callers that cannot allocate device memory.
//
// Some callers may not call cudaMalloc at all: code running where the
// allocator is owned by someone else (a host framework's memory pool, a
// stream-ordered pool that must not grow), or a step that may not allocate
// once a service is up.  moe_route_noalloc runs the same two router kernels
// as moe_route, but the logits scratch lives in the file-scope array below
// instead of a layer's workspace, and no layer is needed.
// ---------------------------------------------------------------------------
namespace moe {
namespace {

constexpr int64_t kNoAllocMaxLogits = int64_t(1) << 18;  // T * n_experts <= 262,144 (1 MiB)
static __device__ __align__(256) float g_noalloc_logits[kNoAllocMaxLogits];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
float *g_noalloc_ptr[kMaxDevices] = {};
unsigned long long g_noalloc_ctx[kMaxDevices] = {};  // context the cached address belongs to

PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;

// Unique id of the calling thread's current context (driver entry points
// resolved once, under g_noalloc_mu).  A cudaDeviceReset ends the context;
// the next one gets a new id, and the module -- with the array -- is loaded
// again at a new address.
cudaError_t current_context_id(unsigned long long *id) {
  if (!g_ctx_current || !g_ctx_id) {
    void *f1 = nullptr, *f2 = nullptr;
    cudaDriverEntryPointQueryResult q1, q2;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 4000, cudaEnableDefault, &q1);
    if (e == cudaSuccess)
      e = cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2);
    if (e != cudaSuccess) return e;
    if (q1 != cudaDriverEntryPointSuccess || q2 != cudaDriverEntryPointSuccess || !f1 || !f2)
      return cudaErrorNotSupported;
    g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f1);
    g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f2);
  }
  CUcontext ctx = nullptr;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS || !ctx) return cudaErrorDeviceUninitialized;
  return g_ctx_id(ctx, id) == CUDA_SUCCESS ? cudaSuccess : cudaErrorDeviceUninitialized;
}

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is asked of
// the runtime (with that device current) and cached per device, together
// with the id of the context it was taken in; a call in a later context of
// the same device (after a cudaDeviceReset) looks the address up again.
cudaError_t noalloc_scratch(float **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  unsigned long long ctx = 0;
  if (g_noalloc_ptr[dev] && current_context_id(&ctx) == cudaSuccess && g_noalloc_ctx[dev] == ctx) {
    *out = g_noalloc_ptr[dev];
    return cudaSuccess;
  }
  // first call on this device, or in a new context of it: the lookup also
  // binds the device's primary context to this thread when none is
  void *ptr = nullptr;
  e = cudaGetSymbolAddress(&ptr, g_noalloc_logits);
  if (e != cudaSuccess) return e;
  e = current_context_id(&ctx);
  if (e != cudaSuccess) return e;
  g_noalloc_ptr[dev] = static_cast<float *>(ptr);
  g_noalloc_ctx[dev] = ctx;
  *out = g_noalloc_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_route_noalloc(const void *x, moe_dtype x_dtype, int32_t T,
                                        int32_t hidden, int32_t n_experts, int32_t top_k,
                                        float routed_scaling, const float *router_w,
                                        const float *logit_bias, int64_t bias_row_stride,
                                        int32_t *ids, float *weights, void *stream) {
  using moe::report_error;
  if (T < 0) return report_error(MOE_ERR_INVALID_ARG, "T = %d is negative", T);
  if (x_dtype != MOE_DT_BF16 && x_dtype != MOE_DT_FP32)
    return report_error(MOE_ERR_INVALID_ARG, "x_dtype %d is not MOE_DT_BF16 or MOE_DT_FP32", (int)x_dtype);
  if (hidden < 32 || hidden > 16384 || hidden % 32)
    return report_error(MOE_ERR_UNSUPPORTED_SHAPE, "hidden = %d: need a multiple of 32 in [32, 16384]", hidden);
  if (n_experts < 1 || n_experts > 256)
    return report_error(MOE_ERR_UNSUPPORTED_SHAPE, "n_experts = %d: need 1..256", n_experts);
  if (top_k < 1 || top_k > 8 || top_k > n_experts)
    return report_error(MOE_ERR_UNSUPPORTED_SHAPE, "top_k = %d: need 1..min(n_experts, 8)", top_k);
  if (!(routed_scaling > 0.f)) return report_error(MOE_ERR_INVALID_ARG, "routed_scaling must be > 0");
  if ((int64_t)T * n_experts > moe::kNoAllocMaxLogits)
    return report_error(MOE_ERR_UNSUPPORTED_SHAPE,
                        "T * n_experts = %lld exceeds the %lld-logit scratch of moe_route_noalloc",
                        (long long)T * n_experts, (long long)moe::kNoAllocMaxLogits);
  if (T == 0) return MOE_OK;
  if (!x || !router_w || !ids || !weights)
    return report_error(MOE_ERR_INVALID_ARG, "x, router_w, ids and weights must be non-NULL");
  if (!moe::aligned(x, 16) || !moe::aligned(router_w, 16) || (logit_bias && !moe::aligned(logit_bias, 16)))
    return report_error(MOE_ERR_MISALIGNED, "x, router_w and logit_bias must be 16-byte aligned");
  if (!moe::aligned(ids, 4) || !moe::aligned(weights, 4))
    return report_error(MOE_ERR_MISALIGNED, "ids/weights are not 4-byte aligned");
  if (logit_bias && bias_row_stride < 0)
    return report_error(MOE_ERR_INVALID_ARG, "bias_row_stride is negative");
  float *logits = nullptr;
  cudaError_t e = moe::noalloc_scratch(&logits);
  if (e != cudaSuccess)
    return report_error(MOE_ERR_CUDA, "moe_route_noalloc scratch address: %s", cudaGetErrorString(e));
  moe::Layer L;  // shape fields only; the router kernels read nothing else
  L.H = hidden;
  L.E = n_experts;
  L.k = top_k;
  L.scale = routed_scaling;
  L.sel_bias = 0;  // logit_bias is added to the logits
  cudaStream_t st = (cudaStream_t)stream;
  int dev = 0, sms = 1;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return report_error(MOE_ERR_CUDA, "moe_route_noalloc: device query failed");
  const int parts = moe::router_parts(T, n_experts, hidden, sms,
                                      (int)(moe::kNoAllocMaxLogits / ((int64_t)T * n_experts)));
  e = moe::launch_router_logits(L, x, x_dtype, T, router_w, logits, parts, st);
  if (e == cudaSuccess)
    e = moe::launch_router_topk(L, logits, parts, logit_bias, bias_row_stride, T, ids, weights, st);
  if (e != cudaSuccess) return report_error(MOE_ERR_CUDA, "moe_route_noalloc: %s", cudaGetErrorString(e));
  return MOE_OK;
}
