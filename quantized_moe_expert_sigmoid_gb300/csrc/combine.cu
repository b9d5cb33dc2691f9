// Output stage of the batched path (PocketLLM "Xing4.0-29B-A4B: the design
// record", section 4: the weighted routed sum and the shared expert are
// added in fp32 and rounded once; float atomics in whatever order the
// hardware commits them make the top-4 sum differ from run to run).
//
// finalize: the down epilogue has added w * y of every route into an fp32
// accumulator with atomics; out = round(out_acc).
//
// ordered (deterministic combine): the down epilogue has stored w * y of
// route p at ybuf[p] (one writer per element, no atomics), and
//   out[t] = ((ybuf[pos(t,0)] + ybuf[pos(t,1)]) + ... + ybuf[pos(t,k-1)])
//            + ybuf[offsets[E] + t]
// in slot order, the shared expert last, then one rounding.  Dropped routes
// (an invalid id, pos -1) add nothing.  Every step has a fixed order, so
// equal inputs give equal bits.
#include "device_utils.cuh"
#include "moe_internal.cuh"

namespace moe {
namespace {

__device__ __forceinline__ void store4(void *out, int64_t i4, float4 v, int bf16) {
  if (bf16) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 o;
    o.x = *reinterpret_cast<uint32_t *>(&lo);
    o.y = *reinterpret_cast<uint32_t *>(&hi);
    reinterpret_cast<uint2 *>(out)[i4] = o;
  } else {
    reinterpret_cast<float4 *>(out)[i4] = v;
  }
}

__global__ void finalize_kernel(const float *__restrict__ acc, int64_t n, void *out, int bf16) {
  const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  pdl_wait();  // the accumulator comes from the previous launch
  pdl_launch_dependents();
  if (i * 4 >= n) return;
  store4(out, i, *reinterpret_cast<const float4 *>(acc + i * 4), bf16);  // n is a multiple of 32
}

// One thread per (token, 4 consecutive outputs); a warp covers 128 outputs
// of one token, so each ybuf row is read in full 512-byte runs.
__global__ void combine_ordered_kernel(const float *__restrict__ ybuf, const int *__restrict__ route_pos,
                                       const int *__restrict__ offsets, int T, int k, int E, int S,
                                       int H, int Hp, void *out, int bf16) {
  const int h4 = H / 4;
  const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  pdl_wait();  // the per-route rows come from the previous launch
  pdl_launch_dependents();
  if (i >= (int64_t)T * h4) return;
  const int t = (int)(i / h4), c = (int)(i % h4) * 4;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j = 0; j < k; ++j) {
    const int pos = route_pos[(int64_t)t * k + j];
    if (pos < 0) continue;
    const float4 y = __ldcs(reinterpret_cast<const float4 *>(ybuf + (int64_t)pos * Hp + c));
    acc.x += y.x;
    acc.y += y.y;
    acc.z += y.z;
    acc.w += y.w;
  }
  if (S) {
    const float4 y = __ldcs(reinterpret_cast<const float4 *>(ybuf + (int64_t)(offsets[E] + t) * Hp + c));
    acc.x += y.x;
    acc.y += y.y;
    acc.z += y.z;
    acc.w += y.w;
  }
  store4(out, i, acc, bf16);
}

__global__ void fill_kernel(float *__restrict__ dst, float v, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) dst[i] = v;
}

}  // namespace

cudaError_t launch_fill(float *dst, float value, int n, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  fill_kernel<<<(n + 255) / 256, 256, 0, stream>>>(dst, value, n);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_finalize(const Layer &L, int T, void *out, moe_dtype odt, cudaStream_t stream) {
  const int64_t n = (int64_t)T * L.H;
  const int64_t threads = n / 4;
  return count_and_check(launch_pdl(finalize_kernel, dim3((unsigned)((threads + 255) / 256)), dim3(256), 0,
                                    stream, (const float *)L.out_acc, n, out, odt == MOE_DT_BF16 ? 1 : 0));
}

cudaError_t launch_combine_ordered(const Layer &L, int T, void *out, moe_dtype odt,
                                   cudaStream_t stream) {
  if (!L.ybuf || !L.route_pos) return cudaErrorInvalidValue;
  const int64_t threads = (int64_t)T * (L.H / 4);
  return count_and_check(launch_pdl(combine_ordered_kernel, dim3((unsigned)((threads + 255) / 256)), dim3(256),
                                    0, stream, (const float *)L.ybuf, (const int *)L.route_pos,
                                    (const int *)L.offsets, T, L.k, L.E, L.S, L.H, L.Hp, out,
                                    odt == MOE_DT_BF16 ? 1 : 0));
}

}  // namespace moe
