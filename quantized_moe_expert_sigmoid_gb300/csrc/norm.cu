// Residual update and unweighted RMS normalisation between stacked layers
// (PocketLLM "Xing4.0-29B-A4B: the design record", section 2: the residual
// streams are carried in fp32 while the sublayer is handed the narrow type).
//   r_out[t] = r_in[t] + delta[t];  u[t] = bf16(r_out[t] / sqrt(mean(r_out[t]^2) + eps))
// (r_out may be r_in: the update in place)
// One CTA per token, 8 elements per thread per step, fp32 throughout, one
// round-to-nearest-even to bf16 at the end.
#include "device_utils.cuh"
#include "moe_internal.cuh"

namespace moe {
namespace {

__device__ __forceinline__ void load8(const float *p, float v[8]) {
  const float4 a = *reinterpret_cast<const float4 *>(p);
  const float4 b = *reinterpret_cast<const float4 *>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

__device__ __forceinline__ void load8(const __nv_bfloat16 *p, float v[8]) {
  const uint4 a = *reinterpret_cast<const uint4 *>(p);
  const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

template <typename DT>
__global__ void __launch_bounds__(256) residual_rmsnorm_kernel(const float *resid_in,
                                                               const DT *__restrict__ delta, float *resid_out,
                                                               int H, float eps,
                                                               __nv_bfloat16 *__restrict__ u) {
  __shared__ float red[8];
  const int t = blockIdx.x;
  pdl_wait();  // the residual and the layer output come from earlier launches
  pdl_launch_dependents();
  const float *ri = resid_in + (int64_t)t * H;
  float *r = resid_out + (int64_t)t * H;
  const bool write = delta != nullptr || resid_in != resid_out;
  float ss = 0.f;
  for (int c = threadIdx.x * 8; c < H; c += blockDim.x * 8) {
    float v[8];
    load8(ri + c, v);
    if (delta) {
      float d[8];
      load8(delta + (int64_t)t * H + c, d);
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] += d[i];
    }
    if (write) {
      reinterpret_cast<float4 *>(r + c)[0] = make_float4(v[0], v[1], v[2], v[3]);
      reinterpret_cast<float4 *>(r + c)[1] = make_float4(v[4], v[5], v[6], v[7]);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) ss = fmaf(v[i], v[i], ss);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) tot += red[i];
  const float inv = 1.0f / sqrtf(tot / (float)H + eps);
  for (int c = threadIdx.x * 8; c < H; c += blockDim.x * 8) {
    float v[8];
    load8(r + c, v);  // this thread's own writes from the first loop
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * i] * inv, v[2 * i + 1] * inv);
      o[i] = *reinterpret_cast<uint32_t *>(&b);
    }
    *reinterpret_cast<uint4 *>(u + (int64_t)t * H + c) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

}  // namespace

cudaError_t launch_residual_rmsnorm(const float *resid_in, const void *delta, moe_dtype ddt, float *resid_out,
                                    void *u, int T, int H, float eps, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  if (ddt == MOE_DT_BF16)
    return count_and_check(launch_pdl(residual_rmsnorm_kernel<__nv_bfloat16>, dim3(T), dim3(256), 0, stream,
                                      resid_in, (const __nv_bfloat16 *)delta, resid_out, H, eps,
                                      (__nv_bfloat16 *)u));
  return count_and_check(launch_pdl(residual_rmsnorm_kernel<float>, dim3(T), dim3(256), 0, stream, resid_in,
                                    (const float *)delta, resid_out, H, eps, (__nv_bfloat16 *)u));
}

}  // namespace moe
