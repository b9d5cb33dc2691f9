// CUDA-core expert path, valid for any number of tokens.
//
// Up/gate + SwiGLU (zhuai.tech "FFN: feature processing inside each layer":
// y = W_down(act(x W_gate) * (x W_up)); PocketLLM design record, section 2:
// silu(gate) * up is handed to the down projection in fp32):
//   h[pos][f] = silu(Gate_e[f] . x[t]) * (Up_e[f] . x[t])   for each route pos
// Down + combine (section 4: routes grouped by expert, one writer per atomic
// target row; the routed and shared sums are fp32):
//   out_acc[t][n] += w_pos * (Down_e[n] . h[pos])
//
// Dequantisation happens in registers: a lane reads one 32-bit word of
// indices (8 consecutive weights of one block) per superblock, looks each
// index up in a 16-entry table in shared memory (entries sit in distinct
// banks) and multiplies by the block's fp16 scale.  A warp covers a
// superblock (32 words) with one 128-byte coalesced load per row.
//
// Grid: blockIdx.x walks the experts that have routes (from the plan's
// active list), so only min(E, T*k) + S expert slots are launched.
#include "moe_internal.cuh"

namespace moe {
namespace {

// IQ4_NL 16-entry table (HelloSun/xing4_0-29b-IQ4_NL_EPQ model card:
// "16-entry nonlinear table + single fp16 scale"; values as given with the
// synthetic workload definition), in the layer's label order: label j < 8
// is table entry 2j, label j + 8 is entry 2j + 1.
__constant__ float c_codebook[16] = {-127.f, -83.f, -49.f, -22.f, 1.f,  25.f, 53.f, 89.f,
                                     -104.f, -65.f, -35.f, -10.f, 13.f, 38.f, 69.f, 113.f};

__device__ __forceinline__ void load_x8(const float *p, float v[8]) {
  const float4 a = *reinterpret_cast<const float4 *>(p);
  const float4 b = *reinterpret_cast<const float4 *>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

__device__ __forceinline__ void load_x8(const __nv_bfloat16 *p, float v[8]) {
  const uint4 a = *reinterpret_cast<const uint4 *>(p);
  const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// sum_m table[q_m] * v[m] over the 8 nibbles of q
__device__ __forceinline__ float dot8(uint32_t q, const float v[8], const float *tab) {
  float s = 0.f;
#pragma unroll
  for (int m = 0; m < 8; ++m) s = fmaf(tab[(q >> (4 * m)) & 15u], v[m], s);
  return s;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

constexpr int kRowsPerCta = 8;  // one output row per warp

template <typename XT>
__global__ void __launch_bounds__(256) upgate_simt_kernel(Layer L, const XT *__restrict__ x) {
  __shared__ float tab[16];
  if (threadIdx.x < 16) tab[threadIdx.x] = c_codebook[threadIdx.x];
  __syncthreads();
  const int a = blockIdx.x;
  if (a >= L.active[L.E + L.S]) return;
  const int e = L.active[a];
  const int seg0 = L.offsets[e], seg1 = L.offsets[e + 1];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int f = blockIdx.y * kRowsPerCta + warp;
  if (f >= L.Fp) return;
  const int64_t grow = (int64_t)(f / kGroupRows) * (2 * kGroupRows) + f % kGroupRows;
  const uint8_t *wg = L.gu + e * L.gu_expert_bytes + grow * L.gu_row_bytes;
  const uint8_t *wu = wg + kGroupRows * L.gu_row_bytes;
  const int nsb = L.Hp / kSBW;
  const int blk = lane >> 2;
  for (int pos = seg0; pos < seg1; ++pos) {
    const int t = L.route_token[pos];
    const XT *xt = x + (int64_t)t * L.H;
    float accg = 0.f, accu = 0.f;
    for (int sb = 0; sb < nsb; ++sb) {
      const int c = sb * kSBW + 8 * lane;
      if (c >= L.H) continue;  // padded tail: zero weights, no x there
      float v[8];
      load_x8(xt + c, v);
      const uint8_t *pg = wg + sb * kSBBytes;
      const uint8_t *pu = wu + sb * kSBBytes;
      const float dg = __half2float(reinterpret_cast<const __half *>(pg)[blk]);
      const float du = __half2float(reinterpret_cast<const __half *>(pu)[blk]);
      const uint32_t qg = reinterpret_cast<const uint32_t *>(pg + 16)[lane];
      const uint32_t qu = reinterpret_cast<const uint32_t *>(pu + 16)[lane];
      accg = fmaf(dg, dot8(qg, v, tab), accg);
      accu = fmaf(du, dot8(qu, v, tab), accu);
    }
    const float g = warp_sum(accg), u = warp_sum(accu);
    if (lane == 0) L.h32[(int64_t)pos * L.Fp + f] = g / (1.0f + expf(-g)) * u;
  }
}

__global__ void __launch_bounds__(256) down_simt_kernel(Layer L) {
  __shared__ float tab[16];
  if (threadIdx.x < 16) tab[threadIdx.x] = c_codebook[threadIdx.x];
  __syncthreads();
  const int a = blockIdx.x;
  if (a >= L.active[L.E + L.S]) return;
  const int e = L.active[a];
  const int seg0 = L.offsets[e], seg1 = L.offsets[e + 1];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.y * kRowsPerCta + warp;
  if (n >= L.H) return;
  const uint8_t *wd = L.dn + e * L.dn_expert_bytes + (int64_t)n * L.dn_row_bytes;
  const int nsb = L.Fp / kSBW;
  const int blk = lane >> 2;
  for (int pos = seg0; pos < seg1; ++pos) {
    const float *hp = L.h32 + (int64_t)pos * L.Fp;
    float acc = 0.f;
    for (int sb = 0; sb < nsb; ++sb) {
      float v[8];
      load_x8(hp + sb * kSBW + 8 * lane, v);
      const uint8_t *p = wd + sb * kSBBytes;
      const float d = __half2float(reinterpret_cast<const __half *>(p)[blk]);
      const uint32_t q = reinterpret_cast<const uint32_t *>(p + 16)[lane];
      acc = fmaf(d, dot8(q, v, tab), acc);
    }
    const float y = warp_sum(acc);
    if (lane == 0) atomicAdd(&L.out_acc[(int64_t)L.route_token[pos] * L.H + n], L.route_weight[pos] * y);
  }
}

__global__ void finalize_kernel(const float *__restrict__ acc, int64_t n, void *out, int bf16) {
  const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  const int64_t i4 = i * 4;
  if (i4 >= n) return;
  const float4 v = *reinterpret_cast<const float4 *>(acc + i4);  // n is a multiple of 32
  if (bf16) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 o;
    o.x = *reinterpret_cast<uint32_t *>(&lo);
    o.y = *reinterpret_cast<uint32_t *>(&hi);
    reinterpret_cast<uint2 *>(out)[i] = o;
  } else {
    reinterpret_cast<float4 *>(out)[i] = v;
  }
}

}  // namespace

static int active_slots(const Layer &L, int T) {
  const int64_t routed = (int64_t)T * L.k;
  return (int)(routed < L.E ? routed : L.E) + L.S;
}

cudaError_t launch_upgate_simt(const Layer &L, const void *x, moe_dtype xdt, int T,
                               cudaStream_t stream) {
  dim3 grid(active_slots(L, T), L.Fp / kRowsPerCta);
  if (xdt == MOE_DT_BF16)
    upgate_simt_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(L, (const __nv_bfloat16 *)x);
  else
    upgate_simt_kernel<float><<<grid, 256, 0, stream>>>(L, (const float *)x);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_down_simt(const Layer &L, int T, cudaStream_t stream) {
  dim3 grid(active_slots(L, T), (L.H + kRowsPerCta - 1) / kRowsPerCta);
  down_simt_kernel<<<grid, 256, 0, stream>>>(L);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_finalize(const Layer &L, int T, void *out, moe_dtype odt, cudaStream_t stream) {
  const int64_t n = (int64_t)T * L.H;
  const int64_t threads = (n + 3) / 4;
  const int bs = 256;
  finalize_kernel<<<(unsigned)((threads + bs - 1) / bs), bs, 0, stream>>>(
      L.out_acc, n, out, odt == MOE_DT_BF16 ? 1 : 0);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace moe
