// Batched decode path (up to 64 tokens; batches of up to 8 normally take the
// single-launch decode kernel): grouped IQ4_NL GEMV with the
// dequantisation in registers and the multiply-adds on the tensor cores.
//
// At these batch sizes an expert holds a handful of tokens (64 tokens top-4
// over 64 experts: ~4 each), so the layer is a bandwidth problem -- every
// selected expert's 6.2 MB is read once -- and the cost per weight byte is
// the decode from 4-bit label to a multiplicand.  Each weight is decoded once
// into registers, and one warp-wide mma.sync (m16n8k16, f16 operands, fp32
// accumulate) then multiplies a 16-row x 16-weight tile by up to 8 tokens, so
// the per-token work is one instruction per 2,048 multiply-adds instead of
// one dp2a per two (PocketLLM "Xing4.0-29B-A4B: the design record", section
// 4: one grouped kernel over a CSR route table serves both prefill and
// decode; here the group is an expert's routes in the plan's order).
//
// Work unit: (active expert, 128 consecutive weight rows).  Up/gate: rows
// 128g..128g+127 of the interleaved gate/up matrix = the gate and the up
// rows of outputs 64g..64g+63, K = Hp; down: rows 128m..128m+127 of W_down,
// K = Fp.  Persistent CTAs (one per SM) take units round-robin.  Per CTA:
//   warp 8     producer: for each 256-wide K step of a unit, one 2D TMA copy
//              of the 128 rows' superblock (128 x 144 B, scales + labels)
//              and 2D TMA copies of the activation rows of the unit's routes
//              (fp16, route order, 16 rows x 64 columns per box, 128-byte
//              swizzle) into a ring of stages
//   warps 0-15 warp w owns rows 16 (w % 8) .. +15 of the unit and half w / 8
//              of each 256-wide K step (blocks 4 (w / 8) .. +3): per
//              32-weight block it decodes its two rows' labels (PRMT table
//              lookups, then the 0x64XX fp16 trick: exact integer codes in
//              fp16), runs two MMAs per 8 tokens against the activation
//              fragments and adds d * (block sum) into fp32 accumulators.
//              Two warps per tile keep four warps per scheduler in flight:
//              the per-block chain (load, decode, MMA, MMA, scale) is long.
//   epilogue   warps 8-15 hand their K-half sums to warps 0-7 through
//              shared memory; up/gate: warps 4-7 (up rows) then hand theirs
//              to warps 0-3 (gate rows of the same outputs);
//              h = route weight * silu(g) * u -> fp16 h16 [route][Fp].
//              down: y = W_down (w h) of each route is added into the fp32
//              output accumulator with atomics, or stored once per route
//              for the slot-ordered deterministic combine.
//
// Token permutation: MMA column n of an 8-token tile is route slot
// (n >> 1) + 4 (n & 1) of the tile, so the two tokens that one quarter of a
// warp reads in a 16-byte activation load sit in rows whose 128-byte-swizzle
// phases differ by 4 -- eight distinct bank groups per quarter warp, no
// shared-memory bank conflicts.
//
// K permutation: in one m16n8k16 MMA, lane (g, c) (g = lane / 4, c = lane %
// 4) supplies A at logical columns {2c, 2c+1, 2c+8, 2c+9} and B at the same
// rows of B.  A dot product does not care which physical weight sits at
// which logical k, as long as A and B agree: lane c takes the 8 weights of
// label word c of the block (weights 8c..8c+7), the first MMA of the block
// uses 8c..8c+3 and the second 8c+4..8c+7, and the activation fragment is
// read at the same physical columns (one 16-byte load per token and block).
// Every wait is bounded; a timeout sets the layer's sticky error word.
#include <cuda.h>

#include "device_utils.cuh"
#include "moe_internal.cuh"
#include "tc_utils.cuh"

namespace moe {
namespace {

constexpr int kGmTiles = 8;                   // 16-row MMA tiles of a unit
constexpr int kGmWarps = 2 * kGmTiles;        // compute warps: two per tile, one per half of K
constexpr int kGmThreads = (kGmWarps + 1) * 32;
constexpr int kGmRows = 16 * kGmTiles;        // weight rows per unit
constexpr int kGmMaxTok = 32;                 // routes of one expert per pass
constexpr int kGmNt = kGmMaxTok / 8;          // 8-token MMA tiles per pass
constexpr int kGmBoxRows = 16;                // activation rows per TMA box
constexpr int kGmStages = 6;
constexpr int kGmWStage = kGmRows * kSBBytes;                 // 18,432 B
constexpr int kGmBStage = kGmMaxTok * kSBW * 2;               // 16,384 B: 32 routes x 256 fp16
constexpr int kGmStage = kGmBStage + kGmWStage;               // 34,816 B (1 KB multiple)
constexpr int kGmXch = kGmTiles * kGmNt * 32 * 4;             // floats of one exchange of partial sums
constexpr size_t kGmSmem = 1024 + (size_t)kGmStages * kGmStage + (size_t)kGmXch * 4;
constexpr uint64_t kGmWaitNs = 1000000000ull;  // 1 s per wait before the CTA gives up
static_assert(kGmStage % 1024 == 0, "128-byte-swizzled boxes need 1 KB aligned stages");
static_assert(kGmSmem <= 232448, "shared memory");

struct GmParams {
  const int *offsets;        // [E+S+1] route segment starts (route order)
  const int *active;         // [E+S+1] active expert ids, [E+S] = count
  const float *route_weight; // [routes]
  const int *route_token;    // [routes]
  __half *h16;               // up/gate output [routes][Fp], route weight folded in
  float *out_acc;            // down: [T][H] fp32 accumulator (atomics), or
  float *ybuf;               //   [routes][Hp] per-route rows (deterministic), else nullptr
  unsigned *err;
  int E, S, H, Hp, Fp;
  int units_per_expert;      // 128-row units of one expert's matrix
  int ksteps;                // 256-wide K steps (superblock columns)
  int64_t rows_per_expert;   // 2 * Fp (up/gate) or Hp (down)
};

// Bounded wait, suspended in hardware between checks: a waiting warp takes no
// issue slots from the sixteen that decode and multiply.
__device__ __forceinline__ void wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *abort) {
  if (*abort) return;
  if (!mbar_wait_suspend(bar, parity, kGmWaitNs)) *abort = 1;
}

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 8 labels (nibble m = weight m) -> four fp16x2 words of the exact integer
// codes, weights (0,1), (2,3), (4,5), (6,7).  The PRMT lookup gives the
// codes + 128 as bytes; a byte v under the high byte 0x64 is the fp16 value
// 1024 + v, so subtracting 1152 leaves the code exactly.
__device__ __forceinline__ void iq4_decode8_f16(uint32_t q, uint32_t (&h)[4]) {
  const uint32_t qx = q ^ 0x88888888u;
  const uint32_t b0 = prmt(kTL0, kTL1, q) ^ prmt(kTH0, kTH1, qx) ^ 0x80808080u;
  const uint32_t b1 = prmt(kTL0, kTL1, q >> 16) ^ prmt(kTH0, kTH1, qx >> 16) ^ 0x80808080u;
  const __half2 off = __half2half2(__ushort_as_half((unsigned short)0x6480));  // 1152
  uint32_t v[4] = {prmt(b0, 0x64646464u, 0x5140), prmt(b0, 0x64646464u, 0x5342),
                   prmt(b1, 0x64646464u, 0x5140), prmt(b1, 0x64646464u, 0x5342)};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __half2 t = __hsub2(*reinterpret_cast<const __half2 *>(&v[i]), off);
    h[i] = *reinterpret_cast<uint32_t *>(&t);
  }
}

__device__ __forceinline__ float half_lo(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w & 0xFFFF))); }
__device__ __forceinline__ float half_hi(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w >> 16))); }

// One 256-wide K step of a warp's 16 rows (its half: four 32-weight blocks)
// against NT tiles of 8 routes.  st: the stage; w0, w1: the rows row_a and
// row_a + 8 in its weight part.
template <int NT>
__device__ __forceinline__ void kstep(const uint8_t *st, const uint8_t *w0, const uint8_t *w1, int khalf,
                                      int c, int slot_g, float (&acc)[kGmNt][4]) {
  // fp16 scales of this warp's four blocks (bytes 8 khalf .. +7 of the row's header)
  const uint2 sc0 = *reinterpret_cast<const uint2 *>(w0 + 8 * khalf);
  const uint2 sc1 = *reinterpret_cast<const uint2 *>(w1 + 8 * khalf);
  const uint32_t *l0 = reinterpret_cast<const uint32_t *>(w0 + 16 + 64 * khalf + 4 * c);
  const uint32_t *l1 = reinterpret_cast<const uint32_t *>(w1 + 16 + 64 * khalf + 4 * c);
#pragma unroll
  for (int jj = 0; jj < 4; ++jj) {  // blocks 4 khalf + jj of the superblock
    uint32_t h0[4], h1[4];
    iq4_decode8_f16(l0[4 * jj], h0);
    iq4_decode8_f16(l1[4 * jj], h1);
    const uint32_t sw0 = jj < 2 ? sc0.x : sc0.y, sw1 = jj < 2 ? sc1.x : sc1.y;
    const float d0 = (jj & 1) ? half_hi(sw0) : half_lo(sw0);
    const float d1 = (jj & 1) ? half_hi(sw1) : half_lo(sw1);
    // activation chunk (4 (jj & 1) + c) of the 64-column box 2 khalf + jj / 2;
    // 128-byte swizzle: 16-byte chunk index XOR (row & 7), and row & 7 is
    // the route slot's phase slot_g in every tile
    const uint8_t *bbox = st + (size_t)(2 * khalf + (jj >> 1)) * (kGmMaxTok * 128);
    const int cofs = ((4 * (jj & 1) + c) ^ slot_g) << 4;
#pragma unroll
    for (int tn = 0; tn < NT; ++tn) {
      const uint4 b = *reinterpret_cast<const uint4 *>(bbox + (tn * 8 + slot_g) * 128 + cofs);
      float dd[4] = {0.f, 0.f, 0.f, 0.f};
      mma_f16(dd, h0[0], h1[0], h0[1], h1[1], b.x, b.y);
      mma_f16(dd, h0[2], h1[2], h0[3], h1[3], b.z, b.w);
      acc[tn][0] = fmaf(d0, dd[0], acc[tn][0]);
      acc[tn][1] = fmaf(d0, dd[1], acc[tn][1]);
      acc[tn][2] = fmaf(d1, dd[2], acc[tn][2]);
      acc[tn][3] = fmaf(d1, dd[3], acc[tn][3]);
    }
  }
}

template <bool UG>
__global__ void __launch_bounds__(kGmThreads, 1)
    gemv_mma_kernel(const GmParams p, const __grid_constant__ CUtensorMap w_map,
                    const __grid_constant__ CUtensorMap b_map) {
  extern __shared__ uint8_t smem_dyn[];
  __shared__ uint64_t full_bar[kGmStages], empty_bar[kGmStages];
  __shared__ int abort_flag;
  volatile int *abort = &abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint8_t *base = smem_dyn + ((1024u - (smem_addr(smem_dyn) & 1023u)) & 1023u);
  float *xch = reinterpret_cast<float *>(base + (size_t)kGmStages * kGmStage);  // [8 tiles][kGmNt][32][4]

  if (tid == 0) {
    for (int s = 0; s < kGmStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kGmWarps);
    }
    fence_mbar_init();
    abort_flag = 0;
  }
  __syncthreads();
  pdl_wait();  // the route plan, activations and accumulators come from earlier launches

  const int n_act = p.active[p.E + p.S];
  const int n_units = n_act * p.units_per_expert;
  const int ks = p.ksteps;

  if (warp == kGmWarps) {
    // ================================ producer ================================
    if (lane == 0) {
      uint32_t q = 0;
      for (int u = blockIdx.x; u < n_units && !*abort; u += gridDim.x) {
        const int e = p.active[u / p.units_per_expert];
        const int m = u % p.units_per_expert;
        const int r0 = p.offsets[e], nr = p.offsets[e + 1] - r0;
        const int wrow = (int)(e * p.rows_per_expert) + m * kGmRows;
        for (int t0 = 0; t0 < nr; t0 += kGmMaxTok) {
          const int nt = min(kGmMaxTok, nr - t0);
          const int nbox = (nt + kGmBoxRows - 1) / kGmBoxRows;
          for (int k = 0; k < ks; ++k, ++q) {
            const int s = q % kGmStages;
            if (q >= (uint32_t)kGmStages) wait_or_abort(&empty_bar[s], ((q / kGmStages) - 1) & 1u, abort);
            if (*abort) break;
            uint8_t *st = base + (size_t)s * kGmStage;
            mbar_arrive_expect_tx(&full_bar[s], (uint32_t)(kGmWStage + nbox * 4 * kGmBoxRows * 128));
            tma_load_2d(st + kGmBStage, &w_map, k * (kSBBytes / 4), wrow, &full_bar[s]);
            for (int b = 0; b < nbox; ++b)
#pragma unroll
              for (int c = 0; c < 4; ++c)  // four 64-column boxes of the 256-wide step
                tma_load_2d(st + c * (kGmMaxTok * 128) + b * (kGmBoxRows * 128), &b_map,
                            k * kSBW + 64 * c, r0 + t0 + b * kGmBoxRows, &full_bar[s]);
          }
        }
      }
      // no copy may still be landing when the CTA exits
      for (int s = 0; s < kGmStages; ++s) {
        const uint32_t uses = q / kGmStages + ((uint32_t)s < q % kGmStages ? 1u : 0u);
        if (uses > 0) mbar_wait_ns(&full_bar[s], (uses - 1) & 1u, kGmWaitNs);
      }
    }
    return;
  }

  // ============================== compute warps ==============================
  const int g = lane >> 2, c = lane & 3;
  const int tile = warp % kGmTiles, khalf = warp / kGmTiles;
  const int row_a = 16 * tile + g;  // rows row_a and row_a + 8 of the unit
  const int slot_g = (g >> 1) | ((g & 1) << 2);  // route slot of MMA column g
  uint32_t q = 0;
  for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
    const int e = p.active[u / p.units_per_expert];
    const int m = u % p.units_per_expert;
    const int r0 = p.offsets[e], nr = p.offsets[e + 1] - r0;
    for (int t0 = 0; t0 < nr; t0 += kGmMaxTok) {
      const int nt = min(kGmMaxTok, nr - t0);
      const int ntile = (nt + 7) >> 3;
      float acc[kGmNt][4];
#pragma unroll
      for (int j = 0; j < kGmNt; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
      for (int k = 0; k < ks; ++k, ++q) {
        const int s = q % kGmStages;
        wait_or_abort(&full_bar[s], (q / kGmStages) & 1u, abort);
        const uint8_t *st = base + (size_t)s * kGmStage;
        const uint8_t *w0 = st + kGmBStage + (size_t)row_a * kSBBytes;
        const uint8_t *w1 = w0 + 8 * kSBBytes;
        if (!*abort) {
          // the tile count is warp-uniform: one specialised loop per count,
          // so no predicated-off MMA tile takes issue slots
          switch (ntile) {
            case 1: kstep<1>(st, w0, w1, khalf, c, slot_g, acc); break;
            case 2: kstep<2>(st, w0, w1, khalf, c, slot_g, acc); break;
            case 3: kstep<3>(st, w0, w1, khalf, c, slot_g, acc); break;
            default: kstep<4>(st, w0, w1, khalf, c, slot_g, acc); break;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[s]);
      }

      // ------------------------------- epilogue -------------------------------
      // accumulator (tn, i): weight row row_a (+8 for i >= 2), MMA column
      // 2c + (i & 1), which is route slot t0 + 8 tn + c + 4 (i & 1)
      // the second K half's sums join the first's
      named_sync(1, kGmWarps * 32);
      if (khalf == 1) {
        float *dst = xch + (size_t)tile * (kGmNt * 32 * 4);
#pragma unroll
        for (int tn = 0; tn < kGmNt; ++tn)
          if (tn < ntile)
            *reinterpret_cast<float4 *>(dst + (tn * 32 + lane) * 4) =
                make_float4(acc[tn][0], acc[tn][1], acc[tn][2], acc[tn][3]);
      }
      named_sync(1, kGmWarps * 32);
      if (khalf == 0) {
        const float *src = xch + (size_t)tile * (kGmNt * 32 * 4);
#pragma unroll
        for (int tn = 0; tn < kGmNt; ++tn)
          if (tn < ntile) {
            const float4 v = *reinterpret_cast<const float4 *>(src + (tn * 32 + lane) * 4);
            acc[tn][0] += v.x;
            acc[tn][1] += v.y;
            acc[tn][2] += v.z;
            acc[tn][3] += v.w;
          }
      }
      if (UG) {
        // tiles 4..7 hold the up rows of the outputs whose gate rows tiles
        // 0..3 hold: hand them over through shared memory
        named_sync(1, kGmWarps * 32);
        if (khalf == 0 && tile >= 4) {
          float *dst = xch + (size_t)(tile - 4) * (kGmNt * 32 * 4);
#pragma unroll
          for (int tn = 0; tn < kGmNt; ++tn)
            if (tn < ntile)
              *reinterpret_cast<float4 *>(dst + (tn * 32 + lane) * 4) =
                  make_float4(acc[tn][0], acc[tn][1], acc[tn][2], acc[tn][3]);
        }
        named_sync(1, kGmWarps * 32);
        if (khalf == 0 && tile < 4 && !*abort) {
          const float *src = xch + (size_t)tile * (kGmNt * 32 * 4);
          const int f0 = m * 64 + 16 * tile + g;  // outputs f0 and f0 + 8
#pragma unroll
          for (int tn = 0; tn < kGmNt; ++tn) {
            if (tn < ntile) {
              const float4 uv = *reinterpret_cast<const float4 *>(src + (tn * 32 + lane) * 4);
              const float uu[4] = {uv.x, uv.y, uv.z, uv.w};
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int slot = t0 + tn * 8 + c + 4 * (i & 1);
                if (slot < nr) {
                  const float gv = acc[tn][i];
                  const float h = gv / (1.0f + __expf(fminf(-gv, 80.0f))) * uu[i] * p.route_weight[r0 + slot];
                  if (!(fabsf(h) <= 65504.f)) atomicOr(p.err, kErrOverflow);
                  p.h16[(int64_t)(r0 + slot) * p.Fp + f0 + (i >= 2 ? 8 : 0)] = __float2half_rn(h);
                }
              }
            }
          }
        }
      } else if (khalf == 0 && !*abort) {
        const int n_lo = m * kGmRows + row_a;  // output rows n_lo and n_lo + 8
#pragma unroll
        for (int tn = 0; tn < kGmNt; ++tn) {
          if (tn < ntile) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int slot = t0 + tn * 8 + c + 4 * (i & 1);
              const int n = n_lo + (i >= 2 ? 8 : 0);
              if (slot < nr && n < p.H) {
                if (p.ybuf)
                  p.ybuf[(int64_t)(r0 + slot) * p.Hp + n] = acc[tn][i];
                else
                  atomicAdd(p.out_acc + (int64_t)p.route_token[r0 + slot] * p.H + n, acc[tn][i]);
              }
            }
          }
        }
      }
    }
  }
  if (tid == 0) pdl_launch_dependents();
  __syncwarp();
  if (lane == 0 && warp == 0 && *abort) atomicOr(p.err, kErrTimeout);
}

template <bool UG>
cudaError_t launch_one(const Layer &L, const CUtensorMap &w_map, const CUtensorMap &b_map,
                       cudaStream_t stream) {
  GmParams p;
  p.offsets = L.offsets;
  p.active = L.active;
  p.route_weight = L.route_weight;
  p.route_token = L.route_token;
  p.h16 = L.h16;
  p.out_acc = L.out_acc;
  p.ybuf = L.deterministic ? L.ybuf : nullptr;
  p.err = L.err;
  p.E = L.E;
  p.S = L.S;
  p.H = L.H;
  p.Hp = L.Hp;
  p.Fp = L.Fp;
  p.units_per_expert = UG ? 2 * L.Fp / kGmRows : L.Hp / kGmRows;
  p.ksteps = UG ? L.Hp / kSBW : L.Fp / kSBW;
  p.rows_per_expert = UG ? 2 * (int64_t)L.Fp : L.Hp;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L.sms);
  cfg.blockDim = dim3(kGmThreads);
  cfg.dynamicSmemBytes = kGmSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, gemv_mma_kernel<UG>, p, w_map, b_map);
  count_launches(1);
  return e;
}

}  // namespace

bool gemv_mma_supported(const Layer &L, int T) {
  return T >= 1 && T <= kGemvMaxTokens && L.gemv_ready;
}

cudaError_t gemv_prepare(Layer &L) {
  L.gemv_ready = 0;
  cudaError_t e = cudaFuncSetAttribute(gemv_mma_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kGmSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gemv_mma_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGmSmem);
  if (e != cudaSuccess) return e;
  // weight superblock columns of 128 rows: 36 words (144 B) x 128 rows
  e = encode_2d(&L.map_gu_sb, CU_TENSOR_MAP_DATA_TYPE_UINT32, L.gu, (uint64_t)L.gu_row_bytes / 4,
                (uint64_t)(L.E + L.S) * 2 * L.Fp, (uint64_t)L.gu_row_bytes, kSBBytes / 4, kGmRows,
                CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e == cudaSuccess)
    e = encode_2d(&L.map_dn_sb, CU_TENSOR_MAP_DATA_TYPE_UINT32, L.dn, (uint64_t)L.dn_row_bytes / 4,
                  (uint64_t)(L.E + L.S) * L.Hp, (uint64_t)L.dn_row_bytes, kSBBytes / 4, kGmRows,
                  CU_TENSOR_MAP_SWIZZLE_NONE);
  // activation rows in route order, boxes of 16 rows x 64 fp16 (128 B)
  if (e == cudaSuccess)
    e = encode_2d(&L.map_x16_16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, L.x16, (uint64_t)L.Hp,
                  (uint64_t)L.max_routes, (uint64_t)L.Hp * 2, 64, kGmBoxRows, CU_TENSOR_MAP_SWIZZLE_128B);
  if (e == cudaSuccess)
    e = encode_2d(&L.map_h16_16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, L.h16, (uint64_t)L.Fp,
                  (uint64_t)L.max_routes, (uint64_t)L.Fp * 2, 64, kGmBoxRows, CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  L.gemv_ready = (2 * L.Fp) % kGmRows == 0 && L.Hp % kGmRows == 0 ? 1 : 0;
  return cudaSuccess;
}

cudaError_t launch_gemv_mma(const Layer &L, cudaStream_t stream, cudaEvent_t *ev) {
  cudaError_t e;
  if (ev && (e = cudaEventRecordWithFlags(ev[0], stream, cudaEventRecordExternal)) != cudaSuccess) return e;
  if ((e = launch_one<true>(L, L.map_gu_sb, L.map_x16_16, stream)) != cudaSuccess) return e;
  if (ev && (e = cudaEventRecordWithFlags(ev[1], stream, cudaEventRecordExternal)) != cudaSuccess) return e;
  if ((e = launch_one<false>(L, L.map_dn_sb, L.map_h16_16, stream)) != cudaSuccess) return e;
  if (ev) return cudaEventRecordWithFlags(ev[2], stream, cudaEventRecordExternal);
  return cudaSuccess;
}

}  // namespace moe
