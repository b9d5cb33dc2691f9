// Router logits of a large bf16 batch on GB300's tensor cores.
//
// l[t][e] = x[t] . Wr[e] in fp32 (HelloSun/xing4_0-29b-IQ4_NL_EPQ model
// card, "模型與路由": the router matrix is fp32; PocketLLM "Xing4.0-29B-A4B:
// the design record", section 4: routing decisions must not depend on the
// arithmetic path).  x is bf16, so it enters a bf16 MMA exactly.  Every fp32
// router weight is the exact sum of three bf16 values: hi = bf16(w), mid =
// bf16(w - hi), lo = bf16(w - hi - mid) -- each residual is exact in fp32
// and the last one has at most 8 significant bits.  The products of bf16
// values are exact in fp32, so
//     l = x.hi + x.mid + x.lo
// accumulated in the fp32 TMEM accumulator has the rounding behaviour of an
// fp32 dot product: the logits match the CUDA-core router to ~1e-6, far
// inside the 1e-4 score gap that fixes every routing decision.
//
// CTA = (256-token tile, K part).  Warp 0 issues the TMA copies of the x tile
// of every 64-wide k-step (bf16, 128-byte swizzle, K-major, straight from
// the caller's x); warps 2-5 read the fp32 router rows of the k-step, split
// them and write the three bf16 A tiles (rows >= E stay zero); one thread of
// warp 1 issues 3 x 4 tcgen05.mma (M 128, N 256, K 16) per k-step into one
// TMEM accumulator.  The epilogue writes the part's partial logits
// logits[part][t][e]; the top-k kernel adds the parts in part order and the
// bias.
#include <cuda.h>

#include <algorithm>

#include "device_utils.cuh"
#include "moe_internal.cuh"
#include "tc_utils.cuh"

namespace moe {
namespace {

constexpr int kRtN = 256;                   // tokens per tile (MMA N)
constexpr int kRtKS = 64;                   // K per k-step (one 128-byte bf16 row)
constexpr int kRtStages = 2;
constexpr int kRtATile = 128 * kRtKS * 2;   // 16 KB: 128 rows (experts, zero-padded)
constexpr int kRtAStage = 3 * kRtATile;     // hi, mid, lo
constexpr int kRtBTile = kRtN * kRtKS * 2;  // 32 KB
constexpr int kRtStage = kRtAStage + kRtBTile;
constexpr int kRtSplitWarps = 4;
constexpr int kRtThreads = 32 * (2 + kRtSplitWarps);
constexpr uint64_t kRtWaitNs = 1000000000ull;

__device__ __forceinline__ void rt_wait(uint64_t *bar, uint32_t parity, volatile int *abort) {
  if (*abort) return;
  if (!mbar_wait_ns(bar, parity, kRtWaitNs)) *abort = 1;
}

// w -> three bf16 bit patterns whose sum is w exactly
__device__ __forceinline__ void split3(float w, uint16_t &hi, uint16_t &mid, uint16_t &lo) {
  const __nv_bfloat16 h = __float2bfloat16_rn(w);
  const float r1 = w - __bfloat162float(h);
  const __nv_bfloat16 m = __float2bfloat16_rn(r1);
  const float r2 = r1 - __bfloat162float(m);
  const __nv_bfloat16 l = __float2bfloat16_rn(r2);
  hi = __bfloat16_as_ushort(h);
  mid = __bfloat16_as_ushort(m);
  lo = __bfloat16_as_ushort(l);
}

__global__ void __launch_bounds__(kRtThreads, 1)
    router_logits_tc(const __grid_constant__ CUtensorMap x_map, const float *__restrict__ wr, int T,
                     int H, int E, int ks_per_part, float *__restrict__ logits, unsigned *err) {
  extern __shared__ uint8_t smem_dyn[];
  __shared__ uint64_t a_full[kRtStages], b_full[kRtStages], empty[kRtStages], acc_full, fin_bar;
  __shared__ uint32_t tmem_holder;
  __shared__ int abort_flag;
  volatile int *abort = &abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile = blockIdx.x, part = blockIdx.y;
  const int nks = (H + kRtKS - 1) / kRtKS;
  const int ks0 = part * ks_per_part, ks1 = min(nks, ks0 + ks_per_part);
  uint8_t *base = smem_dyn + ((1024u - (smem_addr(smem_dyn) & 1023u)) & 1023u);

  if (tid == 0) {
    for (int s = 0; s < kRtStages; ++s) {
      mbar_init(&a_full[s], kRtSplitWarps);
      mbar_init(&b_full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&acc_full, 1);
    mbar_init(&fin_bar, 1);
    fence_mbar_init();
    abort_flag = 0;
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(&tmem_holder)),
                 "r"(kRtN)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // the A rows >= E stay zero for the whole kernel
  if (warp >= 2) {
    for (int i = tid - 64; i < kRtStages * 3 * 128 * 8; i += 32 * kRtSplitWarps) {
      const int row = (i / 8) % 128;
      if (row >= E)
        *reinterpret_cast<uint4 *>(base + (i / (128 * 8 * 3)) * kRtStage + ((i / (128 * 8)) % 3) * kRtATile +
                                   row * 128 + (i % 8) * 16) = make_uint4(0, 0, 0, 0);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_holder;

  if (warp == 0) {
    // ---- x tiles by TMA ----
    if (lane == 0) {
      uint32_t q = 0;
      for (int ks = ks0; ks < ks1 && !*abort; ++ks, ++q) {
        const int s = q % kRtStages;
        if (q >= kRtStages) rt_wait(&empty[s], ((q / kRtStages) - 1) & 1u, abort);
        if (*abort) break;
        mbar_arrive_expect_tx(&b_full[s], kRtBTile);
        tma_load_2d(base + s * kRtStage + kRtAStage, &x_map, ks * kRtKS, tile * kRtN, &b_full[s]);
      }
      for (int s = 0; s < kRtStages; ++s) {  // nothing in flight at exit
        const uint32_t uses = q / kRtStages + ((uint32_t)s < q % kRtStages ? 1u : 0u);
        if (uses > 0) mbar_wait_ns(&b_full[s], (uses - 1) & 1u, kRtWaitNs);
      }
    }
  } else if (warp == 1) {
    // ---- MMA issue: D += A_hi B + A_mid B + A_lo B ----
    if (lane == 0) {
      // D fp32 (bits 4-5 = 1), A and B bf16 (bits 7-9, 10-12 = 1), K-major,
      // N >> 3 at bit 17, M >> 4 at bit 24
      const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kRtN >> 3) << 17) |
                             ((uint32_t)(128 >> 4) << 24);
      uint32_t q = 0;
      for (int ks = ks0; ks < ks1; ++ks, ++q) {
        const int s = q % kRtStages;
        rt_wait(&a_full[s], (q / kRtStages) & 1u, abort);
        rt_wait(&b_full[s], (q / kRtStages) & 1u, abort);
        if (*abort) continue;
        tc_fence_after();
        const uint32_t as = smem_addr(base + s * kRtStage), bs = as + kRtAStage;
#pragma unroll
        for (int pidx = 0; pidx < 3; ++pidx)
#pragma unroll
          for (int k16 = 0; k16 < kRtKS / 16; ++k16)
            umma_f16(tmem, sw128_desc(as + pidx * kRtATile + 32 * k16), sw128_desc(bs + 32 * k16), idesc,
                     (q | pidx | k16) != 0);
        umma_commit(&empty[s]);
      }
      if (!*abort && ks1 > ks0) umma_commit(&acc_full);
      umma_commit(&fin_bar);
      mbar_wait_ns(&fin_bar, 0, kRtWaitNs);
    }
  } else {
    // ---- split the router rows into the three bf16 A tiles ----
    const int st = tid - 64;  // 0..127: rows st/2 (+64), half st%2 of the k-step
    const int half = st & 1;
    uint32_t q = 0;
    for (int ks = ks0; ks < ks1; ++ks, ++q) {
      const int s = q % kRtStages;
      if (q >= kRtStages) rt_wait(&empty[s], ((q / kRtStages) - 1) & 1u, abort);
      uint8_t *stage = base + s * kRtStage;
      for (int row = st >> 1; row < E; row += 64) {
        const int k0 = ks * kRtKS + 32 * half;
        float w[32];
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
          if (k0 + j < H) v = *reinterpret_cast<const float4 *>(wr + (int64_t)row * H + k0 + j);
          w[j] = v.x;
          w[j + 1] = v.y;
          w[j + 2] = v.z;
          w[j + 3] = v.w;
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {  // chunk 4*half + c: 8 values
          uint32_t ph[4], pm[4], pl[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint16_t h0, m0, l0, h1, m1, l1;
            split3(w[8 * c + 2 * u], h0, m0, l0);
            split3(w[8 * c + 2 * u + 1], h1, m1, l1);
            ph[u] = (uint32_t)h0 | ((uint32_t)h1 << 16);
            pm[u] = (uint32_t)m0 | ((uint32_t)m1 << 16);
            pl[u] = (uint32_t)l0 | ((uint32_t)l1 << 16);
          }
          const int off = row * 128 + (((4 * half + c) ^ (row & 7)) << 4);
          *reinterpret_cast<uint4 *>(stage + off) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
          *reinterpret_cast<uint4 *>(stage + kRtATile + off) = make_uint4(pm[0], pm[1], pm[2], pm[3]);
          *reinterpret_cast<uint4 *>(stage + 2 * kRtATile + off) = make_uint4(pl[0], pl[1], pl[2], pl[3]);
        }
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // A tiles -> tensor core
      __syncwarp();
      if (lane == 0) mbar_arrive(&a_full[s]);
    }
    // ---- epilogue: TMEM lanes 0..E-1 are the experts, columns the tokens ----
    if (ks1 > ks0) rt_wait(&acc_full, 0, abort);  // the host never makes an empty part
    tc_fence_after();
    const int quad = warp & 3;  // warps 2..5 -> lane quarters 2, 3, 0, 1
    const bool live = __shfl_sync(0xffffffffu, (*abort == 0 && ks1 > ks0) ? 1 : 0, 0) != 0;
    const int e = 32 * quad + lane;
    float *out = logits + (int64_t)part * T * E;
    if (live && 32 * quad < E) {
      for (int c0 = 0; c0 < kRtN; c0 += 16) {
        uint32_t v[16];
        tmem_ld16_nowait(tmem + ((uint32_t)(32 * quad) << 16) + c0, v);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int t = tile * kRtN + c0 + j;
          if (t < T && e < E) out[(int64_t)t * E + e] = __uint_as_float(v[j]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kRtN)
                 : "memory");
  }
  if (tid == 0 && abort_flag) atomicOr(err, kErrTimeout);
}

size_t rt_smem() { return 1024 + (size_t)kRtStages * kRtStage; }

}  // namespace

bool router_tc_supported(const Layer &L, moe_dtype xdt, int T) {
  return xdt == MOE_DT_BF16 && T >= kRtN && L.E <= 128 && L.H % 8 == 0;
}

// K parts so that tiles x parts fills the SMs once, none of them empty.
int router_tc_parts(const Layer &L, int T) {
  const int sms = std::max(1, L.sms);
  const int tiles = (T + kRtN - 1) / kRtN;
  const int nks = (L.H + kRtKS - 1) / kRtKS;
  const int want = std::max(1, std::min(std::min(kRouterMaxParts, nks), sms / tiles));
  const int per = (nks + want - 1) / want;
  return (nks + per - 1) / per;
}

cudaError_t router_tc_prepare() {
  return cudaFuncSetAttribute(router_logits_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)rt_smem());
}

cudaError_t launch_router_tc(const Layer &L, const void *x, int T, const float *wr, float *logits,
                             int parts, cudaStream_t stream) {
  if (!L.err || parts < 1) return cudaErrorInvalidValue;
  cudaError_t e;
  CUtensorMap x_map;  // the caller's x: [T][H] bf16, K-major
  if ((e = encode_2d(&x_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<void *>(x), (uint64_t)L.H,
                     (uint64_t)T, (uint64_t)L.H * 2, kRtKS, kRtN, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
    return e;
  const int nks = (L.H + kRtKS - 1) / kRtKS;
  const int ks_per_part = (nks + parts - 1) / parts;
  if ((int64_t)(parts - 1) * ks_per_part >= nks) return cudaErrorInvalidValue;  // an empty part
  dim3 grid((T + kRtN - 1) / kRtN, parts);
  router_logits_tc<<<grid, kRtThreads, rt_smem(), stream>>>(x_map, wr, T, L.H, L.E, ks_per_part, logits,
                                                            L.err);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace moe
