// Whole MoE layer for ONE token in one launch.  The routed experts' gate/up
// rows are split into (expert, 32-output block) units, one per CTA, and every
// CTA owns a slice of the output rows, for which it computes the down
// projection of every selected expert and of the shared expert.
//
// The steps and where they run (PocketLLM "Xing4.0-29B-A4B: the design
// record", section 6: the pages' decode step was bound by the time between
// dependent steps, not by bytes; the layer's arithmetic is that of the
// HelloSun model card's whole-layer check: out = sum over the selected
// experts of w * down(silu(gate x) * up x) + the shared expert):
//   1. router logit of expert e on CTA G - E + e, published as a tagged word
//      into every CTA's private copy (copy c of logit e at [e][c]: a router's
//      G stores are coalesced and no line has several writers); every CTA
//      selects the top-k itself;
//   2. the shared expert needs no routing, so its gate/up outputs are
//      computed while the logits travel: CTA c takes outputs
//      [c F / G, (c+1) F / G), four warps per output;
//   3. routed unit r = slot * NB + b (NB = F / 32) on CTA r % G: the 32 gate
//      and 32 up rows of outputs [32 b, 32 b + 32) of the slot's expert, one
//      warp per output;
//   4. every h value goes to global memory, and each expert (and the shared
//      expert) has an arrival counter that its producers advance;
//   5. CTA c owns output rows [c H / G, (c+1) H / G): once an expert's
//      counter is complete it quantises that expert's h and multiplies its
//      W_down rows (copied into shared memory as soon as the top-k was
//      known); the expert sums are added in a fixed order (slot order, then
//      the shared expert), so the output is bit-reproducible.
// The Xing4 layer at one token moves 31.9 MB: 4 routed units of 32 outputs
// x 4 experts = 128 units of 129 KB of gate/up rows, 24 rows x 576 B of each
// W_down per CTA, and the shared expert.
//
// Grid: one CTA per SM, 32 warps; the counter waits need every CTA resident
// (checked at create: one CTA fits on every SM; with MOE_FLAG_COOPERATIVE
// the launch is cooperative).  Counters and logit tags are never reset: each
// counter only grows (a fixed number of arrivals per call), the call's epoch
// is the exit counter / G read at the start (no CTA of this call has exited
// yet), and a logit word is current when its tag is epoch + 1.
//
// Arithmetic (as in the multi-token decode kernel): x and h are 16-bit
// integers with one power-of-two scale per 32-block, the weights exact int8
// codes, dp2a products summed exactly in int32 per 16 or 32 weights, then
// scaled in fp32 by weight scale x activation scale (x route weight).
#include <float.h>

#include <algorithm>

#include "device_utils.cuh"
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kUW = 32;                 // warps per CTA
constexpr int kUT = kUW * 32;           // threads per CTA
constexpr int kUOut = 32;               // outputs (h values) per routed unit
constexpr int kUChunkOut = 4;           // outputs per ring stage
constexpr int kUStages = kUOut / kUChunkOut;
constexpr int kUMaxUnits = 2;           // routed units per CTA
constexpr int kUMaxK = 8;
constexpr int kUShWarps = 4;            // warps per shared-expert output (K split)
constexpr int kUMaxShOut = (kUW - 1) / kUShWarps;  // shared-expert outputs per CTA (not the top-k warp)
constexpr int kUShStage = kUStages - 2;  // the shared gate/up rows wait in ring stages 6 and 7
constexpr int kUMaxRows = 32;           // output rows per CTA (one warp each)
constexpr int kUMaxNB = 32;             // F <= 1024: 32-blocks of h per expert
constexpr int kUTopkWarp = kUW - 1;     // selects the experts while the others compute
constexpr int kUMaxH = 4096;            // a residual-stream step: 256 threads x 8 elements x 2
constexpr uint32_t kUSpin = 1u << 21;   // counter polls before giving up (each an L2 round trip)
constexpr uint64_t kUWaitNs = 500000000ull;

// useq words: [0] exits (G per call), [1] shared-expert h (G per call),
// [2 + j] slot j's h (NB per call), [2 + kUMaxK] x imported (G per call)
constexpr int kUSeqExit = 0, kUSeqShared = 1, kUSeqSlot0 = 2, kUSeqX = kUSeqSlot0 + kUMaxK;

struct UParams {
  Layer L;
  const void *x;
  int x_bf16;
  const float *wr, *bias;
  const int32_t *ids_in;
  const float *w_in;
  int32_t *ids_out;
  float *w_out;
  void *out;
  int out_bf16;
  int wr_smem;  // 1: the router row is bulk-copied into shared memory
  ResidStep rs;  // rs.r_in != nullptr: x is formed from the residual stream here
  uint16_t *x_import;  // non-null: bf16 x is host memory, brought into this device buffer first
  int nr_max;   // largest output-row slice of a CTA (sizes the W_down row region)
};

__device__ __forceinline__ float uwarp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ void red_release_add64(unsigned long long *p, unsigned long long v) {
  asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void red_relaxed_add64(unsigned long long *p, unsigned long long v) {
  asm volatile("red.relaxed.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_acquire64(const unsigned long long *p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ bool spin_until_geq64(const unsigned long long *ctr, unsigned long long target) {
  for (uint32_t i = 0; i < kUSpin; ++i)
    if (ld_acquire64(ctr) >= target) return true;
  return false;
}

// gate row of output f in the interleaved up/gate layout (64-row groups)
__device__ __forceinline__ int gate_row(int f) { return (f / kGroupRows) * (2 * kGroupRows) + f % kGroupRows; }

// 32 activations (fp32, one per lane) -> one int16 block: lane pairs packed
// into hq[0..15] by the even lanes, the block's power-of-two scale returned.
__device__ __forceinline__ float quant_block32(float v, uint32_t *hq, int lane) {
  float m = fabsf(v);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const float sc = act_block_scale(m);
  const float inv = __uint_as_float((uint32_t)(254u << 23) - __float_as_uint(sc));
  const int q = max(-32767, min(32767, __float2int_rn(v * inv)));
  const int qn = __shfl_down_sync(0xffffffffu, q, 1);
  if ((lane & 1) == 0) hq[lane >> 1] = (uint32_t)(q & 0xFFFF) | ((uint32_t)qn << 16);
  return sc;
}

// One IQ4_NL block (16 label bytes) against 32 int16 activations h0..h3.
__device__ __forceinline__ int dot_block32(const uint4 q, const uint4 h0, const uint4 h1, const uint4 h2,
                                           const uint4 h3) {
  uint32_t c0, c1, c2, c3, c4, c5, c6, c7;
  iq4_decode8(q.x, c0, c1);
  iq4_decode8(q.y, c2, c3);
  iq4_decode8(q.z, c4, c5);
  iq4_decode8(q.w, c6, c7);
  // four independent chains of four dp2a (one chain of sixteen is
  // latency-bound when few warps share the SM)
  return (dot8_dp2a(c0, c1, h0, 0) + dot8_dp2a(c2, c3, h1, 0)) + (dot8_dp2a(c4, c5, h2, 0) + dot8_dp2a(c6, c7, h3, 0));
}

// Dynamic shared memory: ring (its start also holds the shared expert's
// gate/up rows until the routed rows arrive), int16 x, x block scales, the
// router row, then W_down rows: (k + 1) slices of nr_max rows.
template <int NSB>
__host__ __device__ constexpr size_t unit_smem_fixed() {
  return (size_t)kUStages * 8 * NSB * kSBBytes + (size_t)NSB * 256 * 2 + (size_t)NSB * 8 * 4 +
         (size_t)NSB * 256 * 4;
}
static_assert(2 * kUMaxShOut <= (kUStages - kUShStage) * 2 * kUChunkOut, "shared rows fit the last two stages");

// One warp's part of gate . x and up . x: superblock pairs [k0, k1).
template <int NSB>
__device__ __forceinline__ void upgate_part(const uint8_t *rowg, const uint8_t *rowu, const int16_t *xq,
                                            const float *sx, int lane, int k0, int k1, float &g, float &u) {
  const int lofs = (lane >> 4) * kSBBytes + 16 + ((lane >> 1) & 7) * 16 + (lane & 1) * 8;
  const int dofs = (lane >> 4) * kSBBytes + ((lane >> 1) & 7) * 2;
  const int16_t *xr = xq + lane * 16;
  const float *sxr = sx + (lane >> 1);
  float accg = 0.f, accu = 0.f;
  for (int k = k0; k < k1; ++k) {
    const uint2 qg = *reinterpret_cast<const uint2 *>(rowg + lofs + 2 * kSBBytes * k);
    const uint2 qu = *reinterpret_cast<const uint2 *>(rowu + lofs + 2 * kSBBytes * k);
    const float dg = __half2float(*reinterpret_cast<const __half *>(rowg + dofs + 2 * kSBBytes * k));
    const float du = __half2float(*reinterpret_cast<const __half *>(rowu + dofs + 2 * kSBBytes * k));
    const uint4 xa = *reinterpret_cast<const uint4 *>(xr + 512 * k);
    const uint4 xb = *reinterpret_cast<const uint4 *>(xr + 512 * k + 8);
    const float sxv = sxr[16 * k];
    uint32_t g0, g1, g2, g3, u0, u1, u2, u3;
    iq4_decode8(qg.x, g0, g1);
    iq4_decode8(qg.y, g2, g3);
    iq4_decode8(qu.x, u0, u1);
    iq4_decode8(qu.y, u2, u3);
    const int sg = dot8_dp2a(g2, g3, xb, dot8_dp2a(g0, g1, xa, 0));
    const int su = dot8_dp2a(u2, u3, xb, dot8_dp2a(u0, u1, xa, 0));
    accg = fmaf((float)sg, dg * sxv, accg);
    accu = fmaf((float)su, du * sxv, accu);
  }
  g = uwarp_sum(accg);
  u = uwarp_sum(accu);
}

// NSB: superblocks per up/gate row (H padded = 256 NSB); an even count, so
// that a warp's lanes cover two superblocks per step.  NL: router logits per
// lane in the top-k (E <= 32 NL); the top-k runs once per call from a cold
// instruction cache, so its length is its cost.
template <int NSB, int NL>
__global__ void __launch_bounds__(kUT, 1) decode_unit_kernel(const UParams p) {
  static_assert(NSB % 2 == 0, "two superblocks per warp step");
  static_assert(NSB * 256 <= kUMaxH, "bf16 x fits the x buffer");
  constexpr int kHp = NSB * 256;
  constexpr int kRB = NSB * kSBBytes;           // bytes of one up/gate row
  constexpr int kChunk = 2 * kUChunkOut * kRB;  // 4 gate rows, then their 4 up rows
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t full_bar[kUStages], wr_bar, sh_bar, dsh_bar, drt_bar;
  __shared__ int n_issued, status;
  __shared__ unsigned long long epoch_s;
  __shared__ int sel_id[kUMaxK];
  __shared__ float sel_w[kUMaxK];
  __shared__ float red[kUW], part_g[kUW], part_u[kUW];
  __shared__ float hs_q[kUMaxK + 1][kUMaxNB];
  __shared__ __align__(16) uint16_t xs_s[kUMaxH];  // x formed from the residual stream (bf16)
  __shared__ float red8[8];

  const Layer &L = p.L;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, c = blockIdx.x;
  const int H = L.H, E = L.E, K = L.k, S = L.S, NB = L.Fp / kUOut;
  const int R = K * NB;
  const int64_t db = L.dn_row_bytes;
  const bool do_route = p.ids_in == nullptr;
  const int my_e = c - (G - E);  // router expert of this CTA when >= 0
  const bool router = do_route && my_e >= 0;
  const unsigned uG = (unsigned)G;
  const int n0 = (int)((unsigned)c * (unsigned)H / uG), n1 = (int)((unsigned)(c + 1) * (unsigned)H / uG);
  const int nr = n1 - n0;
  const int fs0 = S ? (int)((unsigned)c * (unsigned)L.Fp / uG) : 0;
  const int nfs = S ? (int)((unsigned)(c + 1) * (unsigned)L.Fp / uG) - fs0 : 0;
  const int n_mine = c < R ? (R - 1 - c) / G + 1 : 0;  // routed units of this CTA: c, c + G, ...

  uint8_t *ring = smem;
  const uint64_t wpol = l2_evict_first();  // expert weights: read once per call
  // shared gate/up rows [nfs gate][nfs up], in the last two ring stages until
  // the shared slice is computed (a routed unit's first stages go out first)
  uint8_t *sg_rows = smem + (size_t)kUShStage * kChunk;
  int16_t *xq = reinterpret_cast<int16_t *>(smem + (size_t)kUStages * kChunk);
  float *sx = reinterpret_cast<float *>(xq + kHp);
  float *wrs = sx + kHp / 32;
  uint8_t *dn_rows = reinterpret_cast<uint8_t *>(wrs + kHp);  // [k + 1][nr_max][db]: slots, then shared
  const size_t dn_slice = (size_t)p.nr_max * db;

  // one thread: ring stages [s0, s1) of a unit (4 outputs each: 4 gate rows, 4 up rows)
  auto issue_unit = [&](int e, int b, int s0, int s1) {
    if (s0 == 0) ++n_issued;
    const uint8_t *base = L.gu + (int64_t)e * L.gu_expert_bytes + (int64_t)gate_row(kUOut * b) * kRB;
#pragma unroll 1
    for (int s = s0; s < s1; ++s) {
      const uint8_t *g = base + (int64_t)(s * kUChunkOut) * kRB;
      mbar_arrive_expect_tx(&full_bar[s], (uint32_t)kChunk);
      bulk_g2s_hint(ring + (size_t)s * kChunk, g, (uint32_t)(kUChunkOut * kRB), &full_bar[s], wpol);
      bulk_g2s_hint(ring + (size_t)s * kChunk + kUChunkOut * kRB, g + (int64_t)kGroupRows * kRB,
               (uint32_t)(kUChunkOut * kRB), &full_bar[s], wpol);
    }
  };

  // ---- set-up; the router row and the shared gate/up rows go out before
  // the wait for the previous grid (weights are immutable) ----
  if (tid == 0) {
    for (int s = 0; s < kUStages; ++s) mbar_init(&full_bar[s], 1);
    mbar_init(&wr_bar, 1);
    mbar_init(&sh_bar, 1);
    mbar_init(&dsh_bar, 1);
    mbar_init(&drt_bar, 1);
    fence_mbar_init();
    status = 0;
    n_issued = 0;
    if (router && p.wr_smem) {
      mbar_arrive_expect_tx(&wr_bar, (uint32_t)(H * 4));
      bulk_g2s(wrs, p.wr + (int64_t)my_e * H, (uint32_t)(H * 4), &wr_bar);
    }
    if (S) {
      mbar_arrive_expect_tx(&sh_bar, (uint32_t)(2 * nfs * kRB));
      const uint8_t *sgu = L.gu + (int64_t)E * L.gu_expert_bytes;
      int f = fs0, at = 0;  // outputs [fs0, fs0 + nfs), in at most two 64-row groups
      while (f < fs0 + nfs) {
        const int n = min(fs0 + nfs, (f / kGroupRows + 1) * kGroupRows) - f;
        const uint8_t *g = sgu + (int64_t)gate_row(f) * kRB;
        bulk_g2s_hint(sg_rows + (size_t)at * kRB, g, (uint32_t)(n * kRB), &sh_bar, wpol);
        bulk_g2s_hint(sg_rows + (size_t)(nfs + at) * kRB, g + (int64_t)kGroupRows * kRB, (uint32_t)(n * kRB),
                 &sh_bar, wpol);
        f += n;
        at += n;
      }
    }
  }
  __syncthreads();
  // the next grid starts once every CTA of this one has passed this point
  // (so all of them hold their SMs already); it waits for this one to
  // finish before it reads
  pdl_launch_dependents();
  pdl_wait();  // x, the outputs and the counters may belong to the previous grid

  // ---- a trunk step: r_out = r_in + delta and x = u = bf16(rmsnorm(r_out)),
  // computed by every CTA for the whole token (3,584 values) with the
  // arithmetic of the separate residual-RMSNorm kernel (threads 0..255, 8
  // elements each per 2,048, the 8 warp sums added in order), so u is the
  // same bit for bit; CTA 0 also writes r_out and u ----
  const void *xsrc = p.x;
  int xbf = p.x_bf16;
  if (p.rs.r_in) {
    float v[2][8];
    if (warp < 8) {
      float ss = 0.f;
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        const int cc = tid * 8 + 2048 * m;
        if (cc < H) {
          const float4 a = *reinterpret_cast<const float4 *>(p.rs.r_in + cc);
          const float4 b2 = *reinterpret_cast<const float4 *>(p.rs.r_in + cc + 4);
          v[m][0] = a.x; v[m][1] = a.y; v[m][2] = a.z; v[m][3] = a.w;
          v[m][4] = b2.x; v[m][5] = b2.y; v[m][6] = b2.z; v[m][7] = b2.w;
          if (p.rs.delta) {
            if (p.rs.delta_bf16) {
              const uint4 d = *reinterpret_cast<const uint4 *>(reinterpret_cast<const uint16_t *>(p.rs.delta) + cc);
              const uint32_t dw[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                v[m][2 * i] += __uint_as_float(dw[i] << 16);
                v[m][2 * i + 1] += __uint_as_float(dw[i] & 0xFFFF0000u);
              }
            } else {
              const float4 d0 = *reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(p.rs.delta) + cc);
              const float4 d1 = *reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(p.rs.delta) + cc + 4);
              v[m][0] += d0.x; v[m][1] += d0.y; v[m][2] += d0.z; v[m][3] += d0.w;
              v[m][4] += d1.x; v[m][5] += d1.y; v[m][6] += d1.z; v[m][7] += d1.w;
            }
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) ss = fmaf(v[m][i], v[m][i], ss);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      if (lane == 0) red8[warp] = ss;
    }
    __syncthreads();
    if (warp < 8) {
      float tot = 0.f;
      for (int i = 0; i < 8; ++i) tot += red8[i];
      const float inv = 1.0f / sqrtf(tot / (float)H + p.rs.eps);
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        const int cc = tid * 8 + 2048 * m;
        if (cc < H) {
          uint32_t o[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 bb = __floats2bfloat162_rn(v[m][2 * i] * inv, v[m][2 * i + 1] * inv);
            o[i] = *reinterpret_cast<uint32_t *>(&bb);
          }
          const uint4 packed = make_uint4(o[0], o[1], o[2], o[3]);
          *reinterpret_cast<uint4 *>(xs_s + cc) = packed;
          if (c == 0) {
            *reinterpret_cast<float4 *>(p.rs.r_out + cc) = make_float4(v[m][0], v[m][1], v[m][2], v[m][3]);
            *reinterpret_cast<float4 *>(p.rs.r_out + cc + 4) = make_float4(v[m][4], v[m][5], v[m][6], v[m][7]);
            *reinterpret_cast<uint4 *>(p.rs.u_out + cc) = packed;
          }
        }
      }
    }
    __syncthreads();
    xsrc = xs_s;
    xbf = 1;
  }

  if (tid == 0) {
    epoch_s = ld_acquire64(&L.useq[kUSeqExit]) / (unsigned long long)G;
    if (S && nr > 0) {  // the shared expert's W_down rows of this CTA's output rows
      mbar_arrive_expect_tx(&dsh_bar, (uint32_t)(nr * db));
      bulk_g2s_hint(dn_rows + (size_t)K * dn_slice, L.dn + (int64_t)E * L.dn_expert_bytes + (int64_t)n0 * db,
               (uint32_t)(nr * db), &dsh_bar, wpol);
    }
  }

  // ---- x in host memory (the host-buffer call): every CTA copies its share
  // of x's 16-byte chunks into a device buffer and reads x from there once
  // every CTA has, so x crosses the host link once per call instead of once
  // per CTA.  Every launch adds one arrival per CTA, imported or not (a
  // launch without an import adds it on the way out), so the counter's
  // target follows the call epoch ----
  if (p.x_import) {
    const unsigned nch = (unsigned)H / 8u;
    const int q0 = (int)((unsigned)c * nch / uG), q1 = (int)((unsigned)(c + 1) * nch / uG);
    if (tid < q1 - q0)
      reinterpret_cast<uint4 *>(p.x_import)[q0 + tid] = reinterpret_cast<const uint4 *>(p.x)[q0 + tid];
    __syncthreads();
    if (tid == 0) {
      red_release_add64(&L.useq[kUSeqX], 1ull);
      if (!spin_until_geq64(&L.useq[kUSeqX], (epoch_s + 1) * (unsigned long long)G)) {
        atomicOr(&status, 1);
        atomicOr(L.err, kErrTimeout);
      }
    }
    __syncthreads();
  }

  // ---- bf16 x to shared memory, one 16-byte load per thread, all in flight
  // together: one round trip per CTA where the router's strided reads and
  // the quantisation's reads would each wait for their own ----
  if (!p.rs.r_in && xbf) {
    const uint16_t *xg = p.x_import ? p.x_import : static_cast<const uint16_t *>(p.x);
    for (int i = tid; i < H / 8; i += kUT)
      *reinterpret_cast<uint4 *>(xs_s + 8 * i) = __ldcg(reinterpret_cast<const uint4 *>(xg + 8 * i));
    for (int i = H / 8 * 8 + tid; i < H; i += kUT) xs_s[i] = xg[i];
    __syncthreads();
    xsrc = xs_s;
  }

  // ---- router logit of expert my_e: fp32 dot, warp partials added in warp
  // order, one tagged word into every CTA's copy ----
  if (router) {
    if (p.wr_smem && !mbar_wait_ns(&wr_bar, 0, kUWaitNs)) atomicOr(&status, 2);
    const float *w = p.wr_smem ? wrs : p.wr + (int64_t)my_e * H;
    float acc = 0.f;
    for (int i = tid; i < H; i += kUT) {
      const float xv = xbf ? __uint_as_float((uint32_t)reinterpret_cast<const uint16_t *>(xsrc)[i] << 16)
                           : reinterpret_cast<const float *>(xsrc)[i];
      acc = fmaf(xv, w[i], acc);
    }
    acc = uwarp_sum(acc);
    if (lane == 0) red[warp] = acc;
  }
  __syncthreads();  // (also publishes epoch_s)
  const unsigned long long epoch = epoch_s;
  const uint32_t tag = (uint32_t)(epoch + 1);
  if (router && warp * 32 < G) {  // every publishing warp adds the 32 warp partials in the same order
    float v = uwarp_sum(red[lane]);
    if (p.bias && !L.sel_bias) v += p.bias[my_e];
    if (tid < G)
      st_relaxed_u64(&L.ulog[(int64_t)my_e * G + tid], ((unsigned long long)tag << 32) | __float_as_uint(v));
  }

  // ---- while the logits travel: the top-k warp selects the experts and
  // sends out this CTA's routed rows; the other warps quantise x and compute
  // the shared expert's gate/up slice (four warps per output, K split in
  // four) ----
  if (warp == kUTopkWarp) {
    if (do_route) {
      constexpr int kNl = NL;
      float lraw[kNl];
      bool have = false;
      const unsigned long long *cp = L.ulog + c;  // this CTA's copy: logit e at cp[e * G]
      for (uint32_t poll = 0; poll < kUSpin && !have; ++poll) {
        bool mine = true;
#pragma unroll
        for (int i = 0; i < kNl; ++i) {
          const int e = lane + 32 * i;
          lraw[i] = -FLT_MAX;
          if (e < E) {
            const unsigned long long w = ld_relaxed_u64(cp + (int64_t)e * G);
            mine &= (uint32_t)(w >> 32) == tag;
            lraw[i] = __uint_as_float((uint32_t)w);
          }
        }
        have = __all_sync(0xffffffffu, mine);
      }
      if (!have) {
        if (lane < K) sel_id[lane] = -1;
        if (lane == 0) {
          atomicOr(&status, 1);
          atomicOr(L.err, kErrTimeout);
        }
      } else {
        // selection key: the logit (bias already added), or in selection
        // mode the sigmoid score plus the bias; NaN never wins
        uint32_t key[kNl];
#pragma unroll
        for (int i = 0; i < kNl; ++i) {
          const int e = lane + 32 * i;
          float l = lraw[i];
          if (L.sel_bias && e < E) {
            l = 1.0f / (1.0f + expf(-l));
            if (p.bias) l += p.bias[e];
          }
          key[i] = (e < E && l == l) ? float_order_key(l) : 0u;
        }
        // k rounds of a warp arg-max: the largest key, then the lowest
        // expert id holding it (equal keys go to the lower id)
        unsigned taken = 0;
        int my_id = 0;
#pragma unroll 1
        for (int j = 0; j < K; ++j) {
          uint32_t lk = 0;
          int li = 0;
#pragma unroll
          for (int i = 0; i < kNl; ++i)
            if (!((taken >> i) & 1u) && lane + 32 * i < E && key[i] > lk) {
              lk = key[i];
              li = i;
            }
          const uint32_t m = __reduce_max_sync(0xffffffffu, lk);
          const int bid =
              (int)__reduce_min_sync(0xffffffffu, lk == m ? (uint32_t)(lane + 32 * li) : 0xffffffffu);
          if ((bid & 31) == lane) taken |= 1u << (bid >> 5);
          if (lane == j) my_id = bid;
        }
        // the winner's unbiased logit, from the lane that holds it
        float wl = -FLT_MAX;
#pragma unroll
        for (int i = 0; i < kNl; ++i) {
          const float li = __shfl_sync(0xffffffffu, lraw[i], my_id & 31);
          if (i == (my_id >> 5)) wl = li;
        }
        const float my_s = lane < K ? 1.0f / (1.0f + expf(-((wl == wl) ? wl : -FLT_MAX))) : 0.f;
        const float ssum = uwarp_sum(my_s);
        if (lane < K) {
          const float wgt = L.scale * my_s / ssum;
          sel_id[lane] = my_id;
          sel_w[lane] = wgt;
          if (c == 0) {
            p.ids_out[lane] = my_id;
            p.w_out[lane] = wgt;
          }
        }
      }
    } else if (lane < K) {
      const int id = p.ids_in[lane];
      const bool valid = id >= 0 && id < E;
      if (!valid && c == 0) atomicOr(L.err, kErrBadId);
      sel_id[lane] = valid ? id : -1;
      sel_w[lane] = p.w_in[lane];
    }
    __syncwarp();
    if (lane == 0) {
      // this CTA's first routed unit (all but the stages holding the shared
      // rows), then its W_down rows of every selected expert
      if (n_mine > 0 && sel_id[c / NB] >= 0) issue_unit(sel_id[c / NB], c % NB, 0, S ? kUShStage : kUStages);
      uint32_t bytes = 0;
      for (int j = 0; j < K; ++j) bytes += sel_id[j] >= 0 && nr > 0 ? (uint32_t)(nr * db) : 0u;
      mbar_arrive_expect_tx(&drt_bar, bytes);
      for (int j = 0; j < K; ++j)
        if (sel_id[j] >= 0 && nr > 0)
          bulk_g2s_hint(dn_rows + (size_t)j * dn_slice, L.dn + (int64_t)sel_id[j] * L.dn_expert_bytes + (int64_t)n0 * db,
                   (uint32_t)(nr * db), &drt_bar, wpol);
    }
  } else {
    // ---- x to 16-bit integers per 32-block: four threads per block, eight
    // elements each ----
    for (int j = tid; j < kHp / 8 && warp != kUTopkWarp; j += kUT) {
      const int e0 = j * 8;
      float v[8];
      if (xbf && e0 + 8 <= H) {
        const uint4 w = *reinterpret_cast<const uint4 *>(reinterpret_cast<const uint16_t *>(xsrc) + e0);
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
  #pragma unroll
        for (int q = 0; q < 4; ++q) {
          v[2 * q] = __uint_as_float(ww[q] << 16);
          v[2 * q + 1] = __uint_as_float(ww[q] & 0xFFFF0000u);
        }
      } else {
  #pragma unroll
        for (int q = 0; q < 8; ++q)
          v[q] = e0 + q >= H ? 0.f
                 : xbf ? __uint_as_float((uint32_t)reinterpret_cast<const uint16_t *>(xsrc)[e0 + q] << 16)
                       : reinterpret_cast<const float *>(xsrc)[e0 + q];
      }
      float m = 0.f;
  #pragma unroll
      for (int q = 0; q < 8; ++q) m = fmaxf(m, fabsf(v[q]));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
      const float sc = act_block_scale(m);
      const float inv = __uint_as_float((uint32_t)(254u << 23) - __float_as_uint(sc));
      uint32_t pk[4];
  #pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int q0 = max(-32767, min(32767, __float2int_rn(v[2 * q] * inv)));
        const int q1 = max(-32767, min(32767, __float2int_rn(v[2 * q + 1] * inv)));
        pk[q] = (uint32_t)(q0 & 0xFFFF) | ((uint32_t)q1 << 16);
      }
      *reinterpret_cast<uint4 *>(xq + e0) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      if ((j & 3) == 0) sx[j >> 2] = sc;
    }
    named_sync(1, kUT - 32);  // xq and sx complete (the top-k warp does not wait)
    const int o = warp / kUShWarps, q = warp % kUShWarps;
    if (S && o < nfs) {
      if (!mbar_wait_ns(&sh_bar, 0, kUWaitNs)) atomicOr(&status, 2);
      constexpr int kP = NSB / 2, kPer = (kP + kUShWarps - 1) / kUShWarps;
      float g, u;
      upgate_part<NSB>(sg_rows + (size_t)o * kRB, sg_rows + (size_t)(nfs + o) * kRB, xq, sx, lane, q * kPer,
                       min(kP, (q + 1) * kPer), g, u);
      if (lane == 0) {
        part_g[warp] = g;
        part_u[warp] = u;
      }
    }
  }
  __syncthreads();
  if (S) {
    if (tid < nfs) {  // the four K parts of output fs0 + tid, added in order
      float g = 0.f, u = 0.f;
#pragma unroll
      for (int q = 0; q < kUShWarps; ++q) {
        g += part_g[tid * kUShWarps + q];
        u += part_u[tid * kUShWarps + q];
      }
      L.hsh[fs0 + tid] = g / (1.0f + expf(-g)) * u;
    }
    // (this CTA arrives on the shared counter after its routed units: a
    // release waits until the CTA's earlier stores are acknowledged, which
    // takes microseconds while the routed rows stream in, and thread 0
    // computes a routed output)
  }

  // Quantised h of every expert, as the down projection reads it: block b
  // of expert j is 16 words of int16 pairs, stored as four 16-byte chunks at
  // hq4[(j * 4 + k) * NB + b], so that lanes taking consecutive blocks read
  // consecutive 16-byte words (no bank conflicts); hs_q[j][b] its scale
  // with the route weight folded in.  Global copies of the routed experts'
  // quantised h: words [k][NB][16] at L.hr, then scales [k][NB].
  uint4 *hq4 = reinterpret_cast<uint4 *>(ring);
  uint32_t *hr_q = reinterpret_cast<uint32_t *>(L.hr);
  float *hr_s = L.hr + (size_t)K * NB * 16;

  // ---- routed units: warp w computes output 32 b + w (both rows) and
  // SwiGLU; warp 0 quantises the unit's 32 h values (one block) and writes
  // them to global memory ----
  int n_done = 0;  // units whose rows went through the ring before this one (a skipped unit issues none)
  for (int iu = 0; iu < n_mine; ++iu) {
    const int u = c + iu * G;
    const int slot = u / NB, b = u % NB;
    const int e = sel_id[slot];
    if (tid == 0 && e >= 0) {
      if (iu > 0 || !S) issue_unit(e, b, iu > 0 ? 0 : kUStages, kUStages);
      else issue_unit(e, b, kUShStage, kUStages);  // the stages the shared rows held
    }
    float hv = 0.f;
    if (e >= 0) {
      const int s = warp / kUChunkOut;
      if (!mbar_wait_ns(&full_bar[s], (uint32_t)n_done & 1u, kUWaitNs)) atomicOr(&status, 2);
      ++n_done;
      const uint8_t *rowg = ring + (size_t)s * kChunk + (warp % kUChunkOut) * kRB;
      float g, uu;
      upgate_part<NSB>(rowg, rowg + kUChunkOut * kRB, xq, sx, lane, 0, NSB / 2, g, uu);
      hv = g / (1.0f + expf(-g)) * uu;
    }
    if (lane == 0) red[warp] = hv;
    __syncthreads();  // the unit's h in shared memory; every ring stage consumed
    if (warp == 0) {
      const float sc = quant_block32(red[lane], hr_q + (size_t)u * 16, lane);
      if (lane == 0) hr_s[u] = sc * (e >= 0 ? sel_w[slot] : 0.f);
    }
    __syncthreads();
    if (tid == 0) red_release_add64(&L.useq[kUSeqSlot0 + slot], 1ull);
  }
  __syncthreads();  // (the shared h stores above, for CTAs without a routed unit)
  if (S && tid == 0) red_release_add64(&L.useq[kUSeqShared], 1ull);  // this CTA's shared h

  // ---- down projection of output rows [n0, n1), every expert in one pass,
  // once every counter is complete (thread j < k waits for slot j, thread k
  // for the shared expert) ----
  {
    unsigned mask = S ? 1u << K : 0u;  // bit j: slot j, bit K: the shared expert
    for (int j = 0; j < K; ++j) mask |= sel_id[j] >= 0 ? 1u << j : 0u;
    if (tid <= K && ((mask >> tid) & 1u)) {
      const bool sh = tid == K;
      const unsigned long long target =
          sh ? (epoch + 1) * (unsigned long long)G
             : (epoch + 1) * (unsigned long long)NB + (tid == 0 ? (unsigned)L.barrier_slack : 0u);
      if (!spin_until_geq64(&L.useq[sh ? kUSeqShared : kUSeqSlot0 + tid], target)) {
        atomicOr(&status, 1);
        atomicOr(L.err, kErrTimeout);
      }
    }
    if (tid == 32 && (mask & ((1u << K) - 1u)) && !mbar_wait_ns(&drt_bar, 0, kUWaitNs)) atomicOr(&status, 2);
    if (tid == 64 && S && nr > 0 && !mbar_wait_ns(&dsh_bar, 0, kUWaitNs)) atomicOr(&status, 2);
    __syncthreads();
    // routed blocks: thread t copies 16-byte chunk t & 3 of block t >> 2 (and
    // one scale); shared blocks: warp w quantises block w of the shared h
    for (int t = tid; t < R * 4; t += kUT) {
      const int i = t >> 2, k4 = t & 3, j = i / NB, b = i - j * NB;
      if ((mask >> j) & 1u) {
        hq4[(j * 4 + k4) * NB + b] = __ldcg(reinterpret_cast<const uint4 *>(hr_q) + t);
        if (k4 == 0) hs_q[j][b] = __ldcg(hr_s + i);
      }
    }
    if (S) {
      for (int b = warp; b < NB; b += kUW) {
        const float v = __ldcg(L.hsh + b * kUOut + lane);
        float m = fabsf(v);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        const float sc = act_block_scale(m);
        const float inv = __uint_as_float((uint32_t)(254u << 23) - __float_as_uint(sc));
        const int q = max(-32767, min(32767, __float2int_rn(v * inv)));
        const int qn = __shfl_down_sync(0xffffffffu, q, 1);
        if ((lane & 1) == 0) {  // word lane / 2 of the block: chunk (lane / 2) / 4, component (lane / 2) % 4
          uint32_t *dst = reinterpret_cast<uint32_t *>(hq4 + (K * 4 + (lane >> 3)) * NB + b);
          dst[(lane >> 1) & 3] = (uint32_t)(q & 0xFFFF) | ((uint32_t)qn << 16);
        }
        if (lane == 0) hs_q[K][b] = sc;
      }
    }
    __syncthreads();
    // warp w: output row n0 + w.  Lane l takes block l (and l + 32, ...) of
    // every selected expert's W_down row -- independent work the compiler
    // interleaves -- summed in slot order per lane and then across the warp;
    // the shared expert's row sum is added last.
    if (warp < nr) {
      auto block_dot = [&](int j, int b) -> float {
        const uint8_t *sb = dn_rows + (size_t)j * dn_slice + (size_t)warp * db + (b >> 3) * kSBBytes;
        const uint4 q = *reinterpret_cast<const uint4 *>(sb + 16 + (b & 7) * 16);
        const float d = __half2float(*reinterpret_cast<const __half *>(sb + (b & 7) * 2));
        const uint4 *hp = hq4 + (size_t)j * 4 * NB + b;
        return (float)dot_block32(q, hp[0], hp[NB], hp[2 * NB], hp[3 * NB]) * (d * hs_q[j][b]);
      };
      float acc = 0.f;
      for (int b = lane; b < NB; b += 32) {
#pragma unroll
        for (int j = 0; j < kUMaxK; ++j)
          if (j < K && ((mask >> j) & 1u)) acc += block_dot(j, b);
      }
      float out_v = uwarp_sum(acc);
      if (S) {
        float sh = 0.f;
        for (int b = lane; b < NB; b += 32) sh += block_dot(K, b);
        out_v += uwarp_sum(sh);
      }
      if (lane == 0) {
        if (p.out_bf16)
          reinterpret_cast<__nv_bfloat16 *>(p.out)[n0 + warp] = __float2bfloat16_rn(out_v);
        else
          reinterpret_cast<float *>(p.out)[n0 + warp] = out_v;
      }
    }
  }

  // ---- exit: copies still in flight after a timeout land first ----
  if (tid == 0) {
    if (status & 3) {
      for (int s = 0; s < kUStages; ++s)
        if (n_issued > 0) mbar_wait_ns(&full_bar[s], (uint32_t)(n_issued - 1) & 1u, kUWaitNs);
      if (S) {
        mbar_wait_ns(&sh_bar, 0, kUWaitNs);
        if (nr > 0) mbar_wait_ns(&dsh_bar, 0, kUWaitNs);
      }
      mbar_wait_ns(&drt_bar, 0, kUWaitNs);
      if (router && p.wr_smem) mbar_wait_ns(&wr_bar, 0, kUWaitNs);
      if (status & 2) atomicOr(L.err, kErrTimeout);
    }
    if (!p.x_import) red_relaxed_add64(&L.useq[kUSeqX], 1ull);  // (before the exit: read by later calls only)
    red_release_add64(&L.useq[kUSeqExit], 1ull);
  }
}

int unit_nsb(const Layer &L) { return L.Hp / kSBW; }

int unit_nr_max(const Layer &L) { return L.sms > 0 ? (L.H + L.sms - 1) / L.sms : 0; }

template <int NSB>
size_t unit_smem(const Layer &L) {
  return unit_smem_fixed<NSB>() + (size_t)(L.k + 1) * unit_nr_max(L) * (size_t)L.dn_row_bytes;
}

int unit_nl(const Layer &L) { return L.E <= 64 ? 2 : 4; }

// The shared-memory limit of an instance is raised to the largest any
// layer may ask for (the attribute belongs to the function on the current
// device, not to one layer); the occupancy check uses this layer's size.
template <int NSB, int NL>
cudaError_t unit_prepare_one(const Layer &L, int *per_sm) {
  // the dynamic limit is what the device allows a block beyond the
  // kernel's static shared memory
  cudaFuncAttributes fa;
  int optin = 0;
  cudaError_t e = cudaFuncGetAttributes(&fa, decode_unit_kernel<NSB, NL>);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, L.device);
  if (e != cudaSuccess) return e;
  const size_t limit = optin > (int)fa.sharedSizeBytes ? (size_t)optin - fa.sharedSizeBytes : 0;
  if (unit_smem<NSB>(L) > limit) {
    *per_sm = 0;  // does not fit: this layer's one-token calls take the multi-token kernel
    return cudaSuccess;
  }
  e = cudaFuncSetAttribute(decode_unit_kernel<NSB, NL>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)limit);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, decode_unit_kernel<NSB, NL>, kUT, unit_smem<NSB>(L));
}

template <int NSB, int NL>
cudaError_t unit_launch(const UParams &p, int grid, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kUT);
  cfg.dynamicSmemBytes = unit_smem<NSB>(p.L);
  cfg.stream = stream;
  // programmatic serialization: the next call's launch overlaps this call's
  // tail; cooperative (on request): started only once every CTA can be
  // resident at once, which the counter waits need
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeCooperative;
  attr[1].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.L.coop ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, decode_unit_kernel<NSB, NL>, p);
}

// Shapes the kernel takes (every limit below is a static array or a
// shared-memory region of the kernel).
bool unit_shape_ok(const Layer &L) {
  const int nsb = unit_nsb(L);
  if ((nsb != 14 && nsb != 10) || L.sms < 1) return false;
  const int G = L.sms, NB = L.Fp / kUOut, R = L.k * NB;
  if (L.k > kUMaxK || L.E > G || L.E > 128 || NB > kUMaxNB) return false;
  if (unit_nr_max(L) > kUMaxRows) return false;                    // one warp per output row
  if (L.S && (L.Fp + G - 1) / G > kUMaxShOut) return false;         // shared outputs per CTA
  if ((R + G - 1) / G > kUMaxUnits) return false;
  if ((int64_t)NB * 64 > (int64_t)kUStages * 8 * nsb * kSBBytes) return false;  // quantised h fits the ring
  if ((int64_t)std::max(L.H, L.Fp) * G >= ((int64_t)1 << 32)) return false;   // 32-bit splits
  const size_t smem = nsb == 14 ? unit_smem<14>(L) : unit_smem<10>(L);
  return smem <= 232448;  // the exact bound (static + dynamic) is checked when the layer is prepared
}

}  // namespace

cudaError_t unit_decode_prepare(Layer &L) {
  L.unit_resident = 0;
  if (!unit_shape_ok(L)) return cudaSuccess;
  int n = 0;
  const int nsb = unit_nsb(L), nl = unit_nl(L);
  cudaError_t e = nsb == 14 ? (nl == 2 ? unit_prepare_one<14, 2>(L, &n) : unit_prepare_one<14, 4>(L, &n))
                            : (nl == 2 ? unit_prepare_one<10, 2>(L, &n) : unit_prepare_one<10, 4>(L, &n));
  if (e != cudaSuccess) return e;
  L.unit_resident = n >= 1 ? 1 : 0;
  return cudaSuccess;
}

int unit_decode_seq_words() { return kUSeqX + 1; }

bool unit_decode_supported(const Layer &L) {
  return L.unit_resident && L.hr && L.hsh && L.useq && L.ulog && unit_shape_ok(L);
}

cudaError_t launch_decode_unit(const Layer &L, const void *x, moe_dtype xdt, const float *wr, const float *bias,
                               const int32_t *ids_in, const float *w_in, int32_t *ids_out, float *w_out,
                               void *out, moe_dtype odt, cudaStream_t stream, const ResidStep *rs,
                               void *x_import) {
  if (!unit_decode_supported(L)) return cudaErrorInvalidConfiguration;
  if (rs && (L.H > kUMaxH || L.H % 8)) return cudaErrorInvalidConfiguration;
  if (x_import && (rs || xdt != MOE_DT_BF16 || L.H % 8 || !aligned(x_import, 16) || !aligned(x, 16)))
    return cudaErrorInvalidValue;
  UParams p;
  p.L = L;
  p.x = x;
  p.x_bf16 = xdt == MOE_DT_BF16;
  p.x_import = static_cast<uint16_t *>(x_import);
  p.rs = rs ? *rs : ResidStep{nullptr, nullptr, 0, nullptr, nullptr, 0.f};
  p.wr = wr;
  p.bias = bias;
  p.ids_in = ids_in;
  p.w_in = w_in;
  p.ids_out = ids_out;
  p.w_out = w_out;
  p.out = out;
  p.out_bf16 = odt == MOE_DT_BF16;
  p.wr_smem = (wr && aligned(wr, 16) && (L.H % 4) == 0) ? 1 : 0;
  p.nr_max = unit_nr_max(L);
  count_launches(1);
  const int nsb = unit_nsb(L), nl = unit_nl(L);
  cudaError_t e = nsb == 14 ? (nl == 2 ? unit_launch<14, 2>(p, L.sms, stream) : unit_launch<14, 4>(p, L.sms, stream))
                            : (nl == 2 ? unit_launch<10, 2>(p, L.sms, stream) : unit_launch<10, 4>(p, L.sms, stream));
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace moe
