// Whole MoE layer for 2..16 tokens in one launch.  Every expert that some
// token selected (and the shared expert) becomes an entry of a plan; each
// entry's gate/up rows are cut into (entry, 32-output block) units spread
// over the CTAs, and every CTA owns a slice of the output rows, for which it
// computes the down projection of every plan entry.  Weights stream through
// one ring of shared-memory stages per CTA: first the CTA's up/gate stages
// (8 outputs x gate and up rows x one half of the hidden dimension), then one
// stage per plan entry holding that expert's W_down rows of the CTA's output
// slice.  A weight byte is read once per call, whatever the batch.
//
// The steps (PocketLLM "Xing4.0-29B-A4B: the design record", section 4: one
// grouped pass over a per-expert route table, each expert's weights applied
// to all of its tokens; section 6: a decode step is bound by the time between
// dependent steps; the arithmetic is the HelloSun model card's whole-layer
// check, out[t] = sum over t's selected experts of w * down(silu(gate x) *
// up x) + the shared expert):
//   1. router logits of expert e on CTA G - E + e for every token, published
//      as tagged words into every CTA's private copy; warp t of every CTA
//      selects token t's top-k itself;
//   2. every CTA builds the same plan: the shared expert, then the selected
//      experts in increasing id, each with its routes in increasing token;
//   3. unit r = entry * NB + b on CTA r % G: warp items of 8 outputs' gate
//      and up rows against the entry's tokens (4 tokens per register pass);
//      the hidden dimension in two halves, the first half's sums kept in
//      global memory; the unit's 32 h values per route are quantised to one
//      16-bit block and counted on the entry's arrival counter;
//   4. down items (route, group of 8 output rows): W_down rows from the ring,
//      the route's quantised h from L2, a fixed-order cross-lane reduction;
//   5. out[t][n] = the token's routed partial sums in slot order + the
//      shared expert's, written once (no atomics, bit-reproducible).
// Counters are reset by the call after next (two sets, by call parity); the
// call's epoch is the exit counter / G read at its start, as in the
// one-token kernel.  Every wait is bounded and reports MOE_ERR_TIMEOUT.
#include <float.h>

#include <algorithm>

#include "device_utils.cuh"
#include "moe_internal.cuh"
#include "tc_utils.cuh"

namespace moe {
namespace {

constexpr int kBW = 32;                       // warps per CTA
constexpr int kBT = kBW * 32;                 // threads per CTA
constexpr int kBMaxT = kBatchMaxTokens;       // tokens per call
constexpr int kBMaxK = 8;
constexpr int kBChunk = 8;                    // outputs per up/gate stage (one warp each)
constexpr int kBUnit = 32;                    // outputs per unit (one h block)
constexpr int kBTokPass = 4;                  // tokens per register pass of an up/gate item
constexpr int kBRowGroup = 8;                 // output rows per down item
constexpr int kBMaxRoutes = kBMaxT * (kBMaxK + 1);
constexpr int kBMaxPlan = 129;                // E (<= 128) experts + the shared expert
constexpr int kBMaxGroups = 192;              // token groups: <= kBMaxPlan + kBMaxRoutes / 4
constexpr int kBMaxSlots = 16;                // ring stages
constexpr int kBMaxRows = 32;                 // output rows per CTA
constexpr int kBMaxUnits = 64;                // units per CTA
constexpr int kBMaxNB = 32;                   // F <= 1024
constexpr int kBPre = 4;                      // stages issued before the grid-dependency wait
constexpr int kBMinSlots = 4;                 // ring stages at least (the early ones at most kBPre)
constexpr uint64_t kBWaitNs = 500000000ull;   // every wait gives up after 0.5 s

// bseq words: [0] exits (G per call); [1 + parity * kBSet + entry] the
// entry's unit arrivals in calls of that parity (NB per call), and
// [1 + parity * kBSet + kBMaxPlan] the CTAs that have imported their share
// of x (G per call, host-buffer calls only)
constexpr int kBSet = kBMaxPlan + 1;
constexpr int kBSeqWords = 1 + 2 * kBSet;

struct BParams {
  Layer L;
  const void *x;
  int x_bf16;
  uint16_t *x_import;  // non-null: bf16 x is host memory, brought into this device buffer first
  int T;
  const float *wr, *bias;
  int64_t bstride;
  const int32_t *ids_in;
  const float *w_in;
  int32_t *ids_out;
  float *w_out;
  void *out;
  int out_bf16;
  int ns;       // ring stages
  int xw;       // int16 columns of x per token in shared memory (Hp)
  int nr_max;   // largest output-row slice of a CTA
  int wr_smem;  // 1: the router row is bulk-copied into shared memory
};

__device__ __forceinline__ float bwarp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ void b_red_release_add64(unsigned long long *p, unsigned long long v) {
  asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long b_ld_acquire64(const unsigned long long *p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// gate row of output f in the interleaved up/gate layout (64-row groups)
__device__ __forceinline__ int b_gate_row(int f) { return (f / kGroupRows) * (2 * kGroupRows) + f % kGroupRows; }

// Sum of v[0..7] over the warp's 32 lanes, all eight at once: after three
// exchange rounds each lane holds one index, two plain rounds finish the
// sum.  Lane l ends with the total of index (l >> 2) & 7.  The order of the
// additions is fixed, so the result is reproducible.
__device__ __forceinline__ float transpose_sum8(float (&v)[8], int lane) {
  const bool b4 = (lane >> 4) & 1, b3 = (lane >> 3) & 1, b2 = (lane >> 2) & 1;
  float a[4], b[2], s;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float send = b4 ? v[k] : v[k + 4];
    const float keep = b4 ? v[k + 4] : v[k];
    a[k] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
  }
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const float send = b3 ? a[k] : a[k + 2];
    const float keep = b3 ? a[k + 2] : a[k];
    b[k] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
  {
    const float send = b2 ? b[0] : b[1];
    const float keep = b2 ? b[1] : b[0];
    s = keep + __shfl_xor_sync(0xffffffffu, send, 4);
  }
  s += __shfl_xor_sync(0xffffffffu, s, 2);
  s += __shfl_xor_sync(0xffffffffu, s, 1);
  return s;  // index 4 * b4 + 2 * b3 + b2 = (lane >> 2) & 7
}

// One IQ4_NL block (16 label bytes) against 32 int16 activations h0..h3.
__device__ __forceinline__ int b_dot_block32(const uint4 q, const uint4 h0, const uint4 h1, const uint4 h2,
                                             const uint4 h3) {
  uint32_t c0, c1, c2, c3, c4, c5, c6, c7;
  iq4_decode8(q.x, c0, c1);
  iq4_decode8(q.y, c2, c3);
  iq4_decode8(q.z, c4, c5);
  iq4_decode8(q.w, c6, c7);
  return (dot8_dp2a(c0, c1, h0, 0) + dot8_dp2a(c2, c3, h1, 0)) + (dot8_dp2a(c4, c5, h2, 0) + dot8_dp2a(c6, c7, h3, 0));
}

// 32 activations (fp32, one per lane) -> one int16 block: lane pairs packed
// into hq[0..15] by the even lanes, the block's power-of-two scale returned.
__device__ __forceinline__ float b_quant_block32(float v, uint32_t *hq, int lane) {
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

// The hidden dimension in two parts of whole superblock pairs: part 0 the
// first NH0 = 2 ceil(NSB / 4) superblocks, part 1 the other NH1 (8 + 6 for
// H 3,584; 6 + 4 for 2,560).  A ring stage holds NH0 superblocks of 16 rows
// (part 1's box reads past the row end, which the tensor copy fills with
// zeros that are never used).
template <int NSB>
__host__ __device__ constexpr int part0_sbs() {
  return (NSB / 2 + 1) / 2 * 2;
}
template <int NSB>
__host__ __device__ constexpr int part_row_bytes() {
  return part0_sbs<NSB>() * kSBBytes;
}


// x columns [col0, col0 + width) of tokens 0..T-1 -> int16 blocks in shared
// memory (rows of xw columns): four threads per 32-block, eight elements
// each.  Threads [t0, kBT) take part (a multiple of 32 of them).
__device__ __forceinline__ void quantize_x(const void *x, int xbf, int T, int H, int col0, int width, int xw,
                                           int16_t *xq, float *sx, int t0) {
  const int per = width / 8;  // chunks per token (a multiple of 32)
  for (int j = threadIdx.x - t0; j < T * per; j += kBT - t0) {
    const int t = j / per, e0 = col0 + (j - t * per) * 8;
    float v[8];
    const size_t base = (size_t)t * H;
    if (xbf && e0 + 8 <= H) {
      const uint4 w = *reinterpret_cast<const uint4 *>(reinterpret_cast<const uint16_t *>(x) + base + e0);
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
               : xbf ? __uint_as_float((uint32_t)reinterpret_cast<const uint16_t *>(x)[base + e0 + q] << 16)
                     : reinterpret_cast<const float *>(x)[base + e0 + q];
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
    const int c = e0 - col0;
    *reinterpret_cast<uint4 *>(xq + (size_t)t * xw + c) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    if ((j & 3) == 0) sx[t * (xw / 32) + c / 32] = sc;
  }
}

// The same for x already in shared memory as bf16 at xq (rows of xw
// elements, the first H of each valid): each chunk of 8 is read and
// replaced by its int16 codes.
__device__ __forceinline__ void quantize_x_smem(int T, int H, int xw, int16_t *xq, float *sx, int t0) {
  const int per = xw / 8;
  for (int j = threadIdx.x - t0; j < T * per; j += kBT - t0) {
    const int t = j / per, c = (j - t * per) * 8;
    uint16_t *src = reinterpret_cast<uint16_t *>(xq) + (size_t)t * xw + c;
    float v[8];
    if (c + 8 <= H) {
      const uint4 w = *reinterpret_cast<const uint4 *>(src);
      const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        v[2 * q] = __uint_as_float(ww[q] << 16);
        v[2 * q + 1] = __uint_as_float(ww[q] & 0xFFFF0000u);
      }
    } else {
#pragma unroll
      for (int q = 0; q < 8; ++q) v[q] = c + q < H ? __uint_as_float((uint32_t)src[q] << 16) : 0.f;
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
    *reinterpret_cast<uint4 *>(src) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    if ((j & 3) == 0) sx[t * (xw / 32) + c / 32] = sc;
  }
}

// Dynamic shared memory, from its first 128-byte boundary: the down partial
// sums [routes][nr_max] (fp32) and the h values of this CTA's units
// [routes][32] (fp32; a route's h values come from one unit per output
// block); then int16 x [T][xw] and its block scales [T][xw / 32]; then the
// ring of ns stages.  The ring's last stage holds the router row until the
// plan is made; once the up/gate work is done, the span from x to the end
// of the ring holds the down ring.
struct BLayout {
  size_t x, sx, ring;  // byte offsets from the aligned base
};
__host__ __device__ inline size_t round128(size_t v) { return (v + 127) & ~(size_t)127; }
__host__ __device__ inline BLayout batch_layout(int T, int xw, int routes, int nr_max) {
  BLayout l;
  l.x = round128((size_t)routes * nr_max * 4 + (size_t)routes * kBUnit * 4);
  l.sx = l.x + (size_t)T * xw * 2;
  l.ring = round128(l.sx + (size_t)T * (xw / 32) * 4);
  return l;
}
__host__ __device__ inline size_t batch_fixed_bytes(int T, int xw, int routes, int nr_max) {
  return 128 + batch_layout(T, xw, routes, nr_max).ring;  // + room to align the base
}

template <int NSB>
__host__ __device__ inline size_t batch_stage_bytes(int nr_max, int64_t db) {
  const size_t ug = (size_t)2 * kBChunk * part_row_bytes<NSB>();
  const size_t dn = (size_t)nr_max * db;
  return ug > dn ? ug : dn;
}

// A warp's share of one up/gate item, copied out of the ring into
// registers (so that the ring slot is free again long before the item's
// arithmetic is done): NST superblock pairs of a gate row and an up row,
// lane: 16 weights of block (lane >> 1) & 7 of superblock 2k + (lane >> 4)
// (the mapping of the one-token kernel), and the two block scales.
template <int NST>
struct UgRegs {
  uint2 qg[NST], qu[NST];
  __half2 d[NST];  // (gate scale, up scale)
};

template <int NST>
__device__ __forceinline__ void ug_load(const uint8_t *rg, const uint8_t *ru, int nst, int lane, UgRegs<NST> &w) {
  const int lofs = (lane >> 4) * kSBBytes + 16 + ((lane >> 1) & 7) * 16 + (lane & 1) * 8;
  const int dofs = (lane >> 4) * kSBBytes + ((lane >> 1) & 7) * 2;
#pragma unroll
  for (int k = 0; k < NST; ++k)
    if (k < nst) {
      w.qg[k] = *reinterpret_cast<const uint2 *>(rg + lofs + 2 * kSBBytes * k);
      w.qu[k] = *reinterpret_cast<const uint2 *>(ru + lofs + 2 * kSBBytes * k);
      w.d[k] = __halves2half2(*reinterpret_cast<const __half *>(rg + dofs + 2 * kSBBytes * k),
                              *reinterpret_cast<const __half *>(ru + dofs + 2 * kSBBytes * k));
    }
}

// Adds the item's gate and up sums for NTK tokens over the first NS steps
// of w to ag, au; token t's int16 x for this lane starts at xq[xo[t]], and
// its block scale is sx[xo[t] / 32] (x rows and parts start on 32-element
// blocks, and a lane's 16 elements lie in one block).
template <int NS, int NST, int NTK>
__device__ __forceinline__ void ug_compute(const UgRegs<NST> &w, const int16_t *xq, const float *sx,
                                           const int (&xo)[4], float (&ag)[4], float (&au)[4]) {
#pragma unroll
  for (int k = 0; k < NS; ++k) {
    uint32_t g0, g1, g2, g3, u0, u1, u2, u3;
    iq4_decode8(w.qg[k].x, g0, g1);
    iq4_decode8(w.qg[k].y, g2, g3);
    iq4_decode8(w.qu[k].x, u0, u1);
    iq4_decode8(w.qu[k].y, u2, u3);
    const float dg = __low2float(w.d[k]), du = __high2float(w.d[k]);
#pragma unroll
    for (int t = 0; t < NTK; ++t) {
      const uint4 xa = *reinterpret_cast<const uint4 *>(xq + xo[t] + 512 * k);
      const uint4 xb = *reinterpret_cast<const uint4 *>(xq + xo[t] + 512 * k + 8);
      const float sxv = sx[(xo[t] >> 5) + 16 * k];
      const int sg = dot8_dp2a(g2, g3, xb, dot8_dp2a(g0, g1, xa, 0));
      const int su = dot8_dp2a(u2, u3, xb, dot8_dp2a(u0, u1, xa, 0));
      ag[t] = fmaf((float)sg, dg * sxv, ag[t]);
      au[t] = fmaf((float)su, du * sxv, au[t]);
    }
  }
}

template <int NS, int NST>
__device__ __forceinline__ void ug_compute_n(int m, const UgRegs<NST> &w, const int16_t *xq, const float *sx,
                                             const int (&xo)[4], float (&ag)[4], float (&au)[4]) {
  switch (m) {
    case 1: ug_compute<NS, NST, 1>(w, xq, sx, xo, ag, au); break;
    case 2: ug_compute<NS, NST, 2>(w, xq, sx, xo, ag, au); break;
    case 3: ug_compute<NS, NST, 3>(w, xq, sx, xo, ag, au); break;
    default: ug_compute<NS, NST, 4>(w, xq, sx, xo, ag, au); break;
  }
}

// NSB: superblocks per up/gate row (H padded = 256 NSB), even.  NL: router
// logits per lane in the top-k (E <= 32 NL).
// XIMP: bf16 x is host memory and is imported first (a separate instance,
// so that the device-memory kernel carries none of it)
template <int NSB, int NL, bool XIMP>
__global__ void __launch_bounds__(kBT, 1)
    decode_batch_kernel(const BParams p, const __grid_constant__ CUtensorMap gu_map) {
  static_assert(NSB % 2 == 0, "two halves of whole superblocks");
  constexpr int kNH0 = part0_sbs<NSB>(), kNH1 = NSB - kNH0;  // superblocks of the two parts
  constexpr int kPB = part_row_bytes<NSB>();   // bytes of one row of a stage
  constexpr int kBox0 = kNH0 * kSBBytes / 8;   // part 1's column in the tensor map (64-bit words)
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ uint64_t full_bar[kBMaxSlots], wr_bar, x_bar;
  __shared__ uint64_t dbar[kBMaxSlots];  // the down ring's stages
  __shared__ int dslot_stage[kBMaxSlots], dslot_done[kBMaxSlots], dissued_upto;
  __shared__ int slot_done[kBMaxSlots];
  __shared__ int slot_stage[kBMaxSlots];  // the stage last issued into each ring slot
  __shared__ int status, n_plan_s, n_routes_s, issued_upto;
  __shared__ unsigned long long epoch_s;
  __shared__ int sel_id[kBMaxT * kBMaxK];   // [t * K + j]
  __shared__ float sel_w[kBMaxT * kBMaxK];
  __shared__ int cnt_e[128], ent_of[128];
  __shared__ int rank_s[kBMaxT * kBMaxK];
  __shared__ int pe[kBMaxPlan], pstart[kBMaxPlan + 1];
  __shared__ int rtok[kBMaxRoutes], rplan[kBMaxRoutes];
  __shared__ float rw[kBMaxRoutes];
  __shared__ int rof[kBMaxT][kBMaxK + 1];
  __shared__ int ucnt[kBMaxUnits];
  __shared__ int u_grp[kBMaxUnits], u_b[kBMaxUnits];  // token group and block of each of this CTA's units
  __shared__ int grp_ent[kBMaxGroups], grp_c0[kBMaxGroups], pgroups[kBMaxPlan];
  __shared__ int n_groups_s;
  __shared__ float red_r[kBW];

  const Layer &L = p.L;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, c = blockIdx.x;
  const int T = p.T, H = L.H, E = L.E, K = L.k, S = L.S, NB = L.Fp / kBUnit;
  const int64_t db = L.dn_row_bytes;
  const bool do_route = p.ids_in == nullptr;
  const int my_e = c - (G - E);
  const bool router = do_route && my_e >= 0;
  const unsigned uG = (unsigned)G;
  const int n0 = (int)((unsigned)c * (unsigned)H / uG), n1 = (int)((unsigned)(c + 1) * (unsigned)H / uG);
  const int nr = n1 - n0;
  const int ns = p.ns, xw = p.xw, nr_max = p.nr_max;
  const int R_cap = T * (K + S);

  uint8_t *sbase = smem + ((128u - (smem_addr(smem) & 127u)) & 127u);  // 128-byte aligned
  const BLayout lay = batch_layout(T, xw, R_cap, nr_max);
  float *part = reinterpret_cast<float *>(sbase);  // [route][nr_max]
  float *h_s = part + R_cap * nr_max;                // [route][32]
  int16_t *xq = reinterpret_cast<int16_t *>(sbase + lay.x);
  float *sx = reinterpret_cast<float *>(sbase + lay.sx);
  // (the ring starts on a 128-byte boundary, which the tensor copies need)
  uint8_t *ring = sbase + lay.ring;
  const size_t kStage = batch_stage_bytes<NSB>(nr_max, db);
  float *wrs = reinterpret_cast<float *>(ring + (size_t)(ns - 1) * kStage);

  uint32_t *bhq = reinterpret_cast<uint32_t *>(L.bhq);         // [route][32][16] quantised h
  float *bhs = L.bhq + (size_t)kBMaxRoutes * kBMaxNB * 16;     // [route][32] its scales x route weight

  // ---- set-up; the router row and the shared expert's first stages go out
  // before the wait for the previous grid (weights are immutable) ----
  const bool pre = S && c < NB;  // this CTA's first unit is the shared expert's block c
  const uint64_t wpol = l2_evict_first();  // expert weights: read once per call
  if (tid == 0) {
    for (int s = 0; s < kBMaxSlots; ++s) mbar_init(&full_bar[s], 1);
    mbar_init(&wr_bar, 1);
    mbar_init(&x_bar, 1);
    for (int s = 0; s < kBMaxSlots; ++s) mbar_init(&dbar[s], 1);
    dissued_upto = 0;
    fence_mbar_init();
    status = 0;
    issued_upto = 0;
    if (router && p.wr_smem) {
      mbar_arrive_expect_tx(&wr_bar, (uint32_t)(H * 4));
      bulk_g2s(wrs, p.wr + (int64_t)my_e * H, (uint32_t)(H * 4), &wr_bar);
    }
    if (pre) {  // stages 0..3 (both parts of chunks 0 and 1 of unit c, the shared expert's block c)
      const int row0 = E * 2 * L.Fp + b_gate_row(kBUnit * c);
      for (int st = 0; st < kBPre; ++st) {
        const int q = st >> 1, part = st & 1;
        uint8_t *dst = ring + (size_t)st * kStage;
        slot_stage[st] = st;
        mbar_arrive_expect_tx(&full_bar[st], (uint32_t)(2 * kBChunk * kPB));
        tma_load_2d_hint(dst, &gu_map, part * kBox0, row0 + kBChunk * q, &full_bar[st], wpol);
        tma_load_2d_hint(dst + kBChunk * kPB, &gu_map, part * kBox0, row0 + kBChunk * q + kGroupRows, &full_bar[st],
                         wpol);
      }
      issued_upto = kBPre;
    }
  }
  for (int s = tid; s < kBMaxSlots; s += kBT) {
    slot_done[s] = 0;
    if (!(pre && s < kBPre)) slot_stage[s] = -1;
    dslot_done[s] = 0;
    dslot_stage[s] = -1;
  }
  for (int i = tid; i < kBMaxUnits; i += kBT) ucnt[i] = 0;
  __syncthreads();
  pdl_launch_dependents();
  pdl_wait();  // x, the outputs and the counters may belong to the previous grid

  if (tid == 0) epoch_s = b_ld_acquire64(&L.bseq[0]) / (unsigned long long)G;
  __syncthreads();
  const unsigned long long epoch = epoch_s;
  const uint32_t tag = (uint32_t)(epoch + 1);
  const int par = (int)(epoch & 1ull);
  unsigned long long *ctr = L.bseq + 1 + par * kBSet;  // this call's arrival counters
  if (c == 0)  // the next call's counters (nothing of this call touches them)
    for (int i = tid; i < kBSet; i += kBT) L.bseq[1 + (1 - par) * kBSet + i] = 0ull;
  // x in host memory (the host-buffer call): every CTA copies its share of
  // x's 16-byte chunks into a device buffer, which the bulk copy below reads
  // once all G CTAs have (this call's import counter), so x crosses the host
  // link once per call instead of once per CTA
  const uint16_t *xg = XIMP ? p.x_import : static_cast<const uint16_t *>(p.x);
  if constexpr (XIMP) {
    const unsigned nch = (unsigned)(T * H) / 8u;
    const int q0 = (int)((unsigned)c * nch / (unsigned)G), q1 = (int)((unsigned)(c + 1) * nch / (unsigned)G);
    for (int i = tid; i < q1 - q0; i += kBT)
      reinterpret_cast<uint4 *>(p.x_import)[q0 + i] = reinterpret_cast<const uint4 *>(p.x)[q0 + i];
    __syncthreads();
  }
  // bf16 x goes into shared memory in one bulk copy (rows of xw elements),
  // where the router reads it and the quantiser then replaces it in place
  const bool x_smem = p.x_bf16 != 0;
  if (x_smem && tid == 0) {
    if constexpr (XIMP) {
      b_red_release_add64(&ctr[kBMaxPlan], 1ull);
      const uint64_t t0 = global_ns();
      bool have = false;
      for (uint32_t poll = 0; !have; ++poll) {
        have = b_ld_acquire64(&ctr[kBMaxPlan]) >= (unsigned long long)G;
        if (!have && (poll & 15) == 15 && global_ns() - t0 > kBWaitNs) break;
      }
      if (!have) {
        atomicOr(&status, 1);
        atomicOr(L.err, kErrTimeout);
      }
      // the other CTAs' stores (generic proxy) before the bulk copy's reads
      asm volatile("fence.proxy.async.global;" ::: "memory");
    }
    const uint32_t rowb = (uint32_t)H * 2;
    mbar_arrive_expect_tx(&x_bar, rowb * (uint32_t)T);
    if (xw == H)
      bulk_g2s(xq, xg, rowb * (uint32_t)T, &x_bar);
    else
      for (int t = 0; t < T; ++t) bulk_g2s(xq + (size_t)t * xw, xg + (size_t)t * H, rowb, &x_bar);
  }

  // ---- router logits of expert my_e for every token: 32 / T warps per
  // token (a short rolled loop: this code runs once per call, from a cold
  // instruction cache), eight elements per lane and step; the warps' sums
  // of a token are added in warp order ----
  const int wpt = kBW / T;  // warps per token
  if (router) {
    if (p.wr_smem && !mbar_wait_ns(&wr_bar, 0, kBWaitNs)) atomicOr(&status, 2);
    if (x_smem && !mbar_wait_suspend(&x_bar, 0, kBWaitNs)) atomicOr(&status, 2);
    const float *w = p.wr_smem ? wrs : p.wr + (int64_t)my_e * H;
    const int t = warp / wpt;
    float acc = 0.f;
    if (t < T) {
#pragma unroll 1
      for (int i8 = (warp - t * wpt) * 32 + lane; i8 < H / 8; i8 += wpt * 32) {
        const int i = i8 * 8;
        const float4 w0 = *reinterpret_cast<const float4 *>(w + i);
        const float4 w1 = *reinterpret_cast<const float4 *>(w + i + 4);
        float4 a, b;
        if (x_smem) {
          const uint4 q = *reinterpret_cast<const uint4 *>(reinterpret_cast<const uint16_t *>(xq) + (size_t)t * xw + i);
          a = make_float4(__uint_as_float(q.x << 16), __uint_as_float(q.x & 0xFFFF0000u),
                          __uint_as_float(q.y << 16), __uint_as_float(q.y & 0xFFFF0000u));
          b = make_float4(__uint_as_float(q.z << 16), __uint_as_float(q.z & 0xFFFF0000u),
                          __uint_as_float(q.w << 16), __uint_as_float(q.w & 0xFFFF0000u));
        } else {
          a = *reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(p.x) + (size_t)t * H + i);
          b = *reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(p.x) + (size_t)t * H + i + 4);
        }
        acc = fmaf(a.x, w0.x, acc);
        acc = fmaf(a.y, w0.y, acc);
        acc = fmaf(a.z, w0.z, acc);
        acc = fmaf(a.w, w0.w, acc);
        acc = fmaf(b.x, w1.x, acc);
        acc = fmaf(b.y, w1.y, acc);
        acc = fmaf(b.z, w1.z, acc);
        acc = fmaf(b.w, w1.w, acc);
      }
    }
    acc = bwarp_sum(acc);
    if (lane == 0) red_r[warp] = acc;
  }
  __syncthreads();
  if (router && warp * 32 < G) {  // every publishing warp adds a token's warp sums in the same order
#pragma unroll 1
    for (int t = 0; t < T; ++t) {
      float v = 0.f;
      for (int k = 0; k < wpt; ++k) v += red_r[t * wpt + k];
      if (p.bias && !L.sel_bias) v += p.bias[(int64_t)t * p.bstride + my_e];
      if (tid < G)
        st_relaxed_u64(&L.blog[((int64_t)t * E + my_e) * G + tid], ((unsigned long long)tag << 32) | __float_as_uint(v));
    }
  }

  // ---- warp t selects token t's experts; the other warps quantise x (the
  // whole row, or its first half) ----
  if (warp < T) {
    const int t = warp;
    if (do_route) {
      float lraw[NL];
      bool have = false;
      const unsigned long long *cp = L.blog + (int64_t)t * E * G + c;  // logit e at cp[e * G]
      const uint64_t t0 = global_ns();
      for (uint32_t poll = 0; !have; ++poll) {
        bool mine = true;
#pragma unroll
        for (int i = 0; i < NL; ++i) {
          const int e = lane + 32 * i;
          lraw[i] = -FLT_MAX;
          if (e < E) {
            const unsigned long long wv = ld_relaxed_u64(cp + (int64_t)e * G);
            mine &= (uint32_t)(wv >> 32) == tag;
            lraw[i] = __uint_as_float((uint32_t)wv);
          }
        }
        have = __all_sync(0xffffffffu, mine);
        if (!have && (poll & 63) == 63 && __shfl_sync(0xffffffffu, global_ns() - t0 > kBWaitNs, 0)) break;
      }
      if (!have) {
        if (lane < K) sel_id[t * K + lane] = -1;
        if (lane == 0) {
          atomicOr(&status, 1);
          atomicOr(L.err, kErrTimeout);
        }
      } else {
        const float *brow = p.bias ? p.bias + (int64_t)t * p.bstride : nullptr;
        uint32_t key[NL];
#pragma unroll
        for (int i = 0; i < NL; ++i) {
          const int e = lane + 32 * i;
          float l = lraw[i];
          if (L.sel_bias && e < E) {
            l = 1.0f / (1.0f + expf(-l));
            if (brow) l += brow[e];
          }
          key[i] = (e < E && l == l) ? float_order_key(l) : 0u;
        }
        // k rounds of a warp arg-max: the largest key, then the lowest id
        unsigned taken = 0;
        int my_id = 0;
#pragma unroll 1
        for (int j = 0; j < K; ++j) {
          uint32_t lk = 0;
          int li = 0;
#pragma unroll
          for (int i = 0; i < NL; ++i)
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
        float wl = -FLT_MAX;
#pragma unroll
        for (int i = 0; i < NL; ++i) {
          const float li = __shfl_sync(0xffffffffu, lraw[i], my_id & 31);
          if (i == (my_id >> 5)) wl = li;
        }
        const float my_s = lane < K ? 1.0f / (1.0f + expf(-((wl == wl) ? wl : -FLT_MAX))) : 0.f;
        const float ssum = bwarp_sum(my_s);
        if (lane < K) {
          const float wgt = L.scale * my_s / ssum;
          sel_id[t * K + lane] = my_id;
          sel_w[t * K + lane] = wgt;
          if (c == 0) {
            p.ids_out[t * K + lane] = my_id;
            p.w_out[t * K + lane] = wgt;
          }
        }
      }
    } else if (lane < K) {
      const int id = p.ids_in[t * K + lane];
      const bool valid = id >= 0 && id < E;
      if (!valid && c == 0) atomicOr(L.err, kErrBadId);
      sel_id[t * K + lane] = valid ? id : -1;
      sel_w[t * K + lane] = p.w_in[t * K + lane];
    }
  } else {
    if (x_smem) {
      if (!mbar_wait_suspend(&x_bar, 0, kBWaitNs)) atomicOr(&status, 2);
      quantize_x_smem(T, H, xw, xq, sx, T * 32);
    } else {
      quantize_x(p.x, p.x_bf16, T, H, 0, xw, xw, xq, sx, T * 32);
    }
  }
  __syncthreads();

  // ---- the plan, the same on every CTA: entry 0 the shared expert (every
  // token, weight 1), then the selected experts in increasing id, each with
  // its routes ordered by (token, slot) ----
  if (warp == 0) {
    // routes (t, j) in order, 32 at a time: a route's rank among its
    // expert's routes is the count carried from earlier groups plus its
    // matching lanes below it
    for (int e = lane; e < E; e += 32) cnt_e[e] = 0;
    __syncwarp();
    for (int i0 = 0; i0 < T * K; i0 += 32) {
      const int i = i0 + lane;
      const int id = i < T * K ? sel_id[i] : -1;
      const unsigned peers = __match_any_sync(0xffffffffu, id);
      const int below = __popc(peers & ((1u << lane) - 1u));
      const int carried = id >= 0 ? cnt_e[id] : 0;
      __syncwarp();
      if (id >= 0) {
        rank_s[i] = carried + below;
        if (below == 0) cnt_e[id] = carried + __popc(peers);
      }
      __syncwarp();
    }
    // entries and route starts: a scan over the experts
    int base = S ? T : 0, ent = S;
    if (lane == 0) {
      pstart[0] = 0;
      if (S) pe[0] = E;
    }
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int n = e < E ? cnt_e[e] : 0;
      const bool u = n > 0;
      int incl = n;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      const unsigned m = __ballot_sync(0xffffffffu, u);
      const int my_ent = ent + __popc(m & ((1u << lane) - 1u));
      if (u) {
        pe[my_ent] = e;
        pstart[my_ent] = base + incl - n;
        ent_of[e] = my_ent;
      }
      base += __shfl_sync(0xffffffffu, incl, 31);
      ent += __popc(m);
    }
    if (lane == 0) {
      pstart[ent] = base;
      n_plan_s = ent;
      n_routes_s = base;
    }
    __syncwarp();
    // each entry's routes in token groups of at most 4 (one register pass)
    int gbase = 0;
    for (int e0 = 0; e0 < ent; e0 += 32) {
      const int e = e0 + lane;
      const int ng = e < ent ? (pstart[e + 1] - pstart[e] + kBTokPass - 1) / kBTokPass : 0;
      int incl = ng;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (e < ent) {
        pgroups[e] = ng;
        for (int g = 0; g < ng; ++g) {
          grp_ent[gbase + incl - ng + g] = e;
          grp_c0[gbase + incl - ng + g] = g * kBTokPass;
        }
      }
      gbase += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) n_groups_s = gbase;
  }
  __syncthreads();
  if (S && tid < T) {  // the shared expert's routes: token t is route t
    rtok[tid] = tid;
    rw[tid] = 1.0f;
    rplan[tid] = 0;
    rof[tid][K] = tid;
  }
  if (tid < T * K) {
    const int t = tid / K, j = tid - t * K, id = sel_id[tid];
    int r = -1;
    if (id >= 0) {
      const int ent = ent_of[id];
      r = pstart[ent] + rank_s[tid];
      rtok[r] = t;
      rw[r] = sel_w[tid];
      rplan[r] = ent;
    }
    rof[t][j] = r;
  }
  __syncthreads();
  const int n_plan = n_plan_s, n_routes = n_routes_s;
  const int n_units = n_groups_s * NB;  // unit r: token group r / NB, output block r % NB
  const int n_mine = c < n_units ? (n_units - 1 - c) / G + 1 : 0;
  const int s_ug = 8 * n_mine;            // up/gate stages: n_mine units x 4 chunks x 2 parts
  // (the entries' W_down stages go through the down ring afterwards)
  const int rg = (nr + kBRowGroup - 1) / kBRowGroup;  // row groups of a down stage
  for (int iu = tid; iu < n_mine; iu += kBT) {
    const int r = c + iu * G, g = r / NB;
    u_grp[iu] = g;
    u_b[iu] = r - g * NB;
  }
  __syncthreads();

  // one thread: up/gate stage s = 8 iu + 2 q + part into ring slot s % ns:
  // the 8 gate and the 8 up rows of chunk q of unit iu, that part of the
  // hidden dimension, two 2D tensor copies
  auto issue_stage = [&](int s) {
    const int slot = s % ns;
    uint8_t *dst = ring + (size_t)slot * kStage;
    uint64_t *bar = &full_bar[slot];
    *reinterpret_cast<volatile int *>(&slot_stage[slot]) = s;  // before the arrival that opens its phase
    const int iu = s >> 3, q = (s >> 1) & 3, part = s & 1;
    const int row0 = pe[grp_ent[u_grp[iu]]] * 2 * L.Fp + b_gate_row(kBUnit * u_b[iu] + kBChunk * q);
    mbar_arrive_expect_tx(bar, (uint32_t)(2 * kBChunk * kPB));
    tma_load_2d_hint(dst, &gu_map, part * kBox0, row0, bar, wpol);
    tma_load_2d_hint(dst + kBChunk * kPB, &gu_map, part * kBox0, row0 + kGroupRows, bar, wpol);
    atomicMax(&issued_upto, s + 1);
  };
  if (tid == 0)
    for (int s = pre ? kBPre : 0; s < min(ns, s_ug); ++s) issue_stage(s);

  // Wait until stage s (in ring slot `slot`, its lap-th use) has landed.  A
  // warp may reach a stage while its slot still serves the stage one lap
  // earlier, when a parity wait would see that older phase as complete; so
  // first the slot must carry stage s's tag (its issuer writes the tag
  // before the arrival that opens the stage's phase), then the phase's
  // parity identifies it.
  auto wait_tagged = [&](int *tags, uint64_t *bars, int s, int slot, int lap) -> bool {
    if (*reinterpret_cast<volatile int *>(&tags[slot]) != s) {
      const uint64_t t0 = global_ns();
      for (uint32_t poll = 0; *reinterpret_cast<volatile int *>(&tags[slot]) != s; ++poll) {
        __nanosleep(256);
        if ((poll & 15) == 15 && global_ns() - t0 > kBWaitNs) return false;
      }
    }
    // suspended in hardware until the phase completes: a waiting warp takes
    // no issue slots from the warps that compute
    return mbar_wait_suspend(&bars[slot], (uint32_t)lap & 1u, kBWaitNs);
  };
  auto wait_stage = [&](int s, int slot, int lap) -> bool { return wait_tagged(slot_stage, full_bar, s, slot, lap); };
  // lane 0, after the warp is done with stage s: the stage's last user frees
  // its slot for stage s + ns
  auto release_stage = [&](int s, int slot, int need) {
    if (atomicAdd(&slot_done[slot], 1) + 1 == need) {
      slot_done[slot] = 0;
      if (s + ns < s_ug && *reinterpret_cast<volatile int *>(&status) == 0) issue_stage(s + ns);
    }
  };

  // ---- up/gate: warp w computes output 8 q + o (q = w / 8, o = w % 8) of
  // each of the CTA's units, over both parts of the hidden dimension (stages
  // 8 iu + 2 q and 8 iu + 2 q + 1); the rows go from the ring into registers
  // first, so a slot is free as soon as the stage's 8 warps hold them ----
  {
    const int q = warp >> 3, o = warp & 7;
    int s0 = 2 * q, slot0 = s0 % ns, lap0 = s0 / ns;
    for (int iu = 0; iu < n_mine; ++iu) {
      const int gi = u_grp[iu], ent = grp_ent[gi], b = u_b[iu];
      const int f = kBUnit * b + kBChunk * q + o;
      const int r0 = pstart[ent] + grp_c0[gi], nt = min(kBTokPass, pstart[ent + 1] - r0);
      const int slot1 = slot0 + 1 == ns ? 0 : slot0 + 1, lap1 = slot1 == 0 ? lap0 + 1 : lap0;
      {
        const int m = nt;
        int xo[kBTokPass];
        float ag[kBTokPass], au[kBTokPass];
#pragma unroll
        for (int u = 0; u < kBTokPass; ++u) {
          const int tk = u < m ? rtok[r0 + u] : 0;
          xo[u] = tk * xw + 16 * lane;
          ag[u] = au[u] = 0.f;
        }
        UgRegs<kNH0 / 2> wreg;
        // part 0
        bool ok = *reinterpret_cast<volatile int *>(&status) == 0;
        if (ok && !wait_stage(s0, slot0, lap0)) {
          ok = false;
          if (lane == 0) atomicOr(&status, 2);
        }
        if (ok) ug_load<kNH0 / 2>(ring + (size_t)slot0 * kStage + o * kPB,
                                  ring + (size_t)slot0 * kStage + (kBChunk + o) * kPB, kNH0 / 2, lane, wreg);
        __syncwarp();
        if (lane == 0) release_stage(s0, slot0, kBChunk);
        if (ok) ug_compute_n<kNH0 / 2, kNH0 / 2>(m, wreg, xq, sx, xo, ag, au);
        // part 1
        if (ok && !wait_stage(s0 + 1, slot1, lap1)) {
          ok = false;
          if (lane == 0) atomicOr(&status, 2);
        }
        if (ok) ug_load<kNH0 / 2>(ring + (size_t)slot1 * kStage + o * kPB,
                                  ring + (size_t)slot1 * kStage + (kBChunk + o) * kPB, kNH1 / 2, lane, wreg);
        __syncwarp();
        if (lane == 0) release_stage(s0 + 1, slot1, kBChunk);
        if (ok) {
#pragma unroll
          for (int u = 0; u < kBTokPass; ++u) xo[u] += kNH0 * 256;
          ug_compute_n<kNH1 / 2, kNH0 / 2>(m, wreg, xq, sx, xo, ag, au);
          // every token's gate and up sums at once: lane 8t holds token t's
          // gate sum, lane 8t + 4 its up sum
          float v[8];
#pragma unroll
          for (int u = 0; u < kBTokPass; ++u) {
            v[2 * u] = u < m ? ag[u] : 0.f;
            v[2 * u + 1] = u < m ? au[u] : 0.f;
          }
          const float tot = transpose_sum8(v, lane);
          const float tot_u = __shfl_down_sync(0xffffffffu, tot, 4);
          const int tt = lane >> 3;
          if ((lane & 7) == 0 && tt < m)
            h_s[(r0 + tt) * kBUnit + kBChunk * q + o] = tot / (1.0f + expf(-tot)) * tot_u;
        }
      }
      // the unit's 32 outputs: the last of its 32 warps quantises the h blocks
      __syncwarp();
      int last = 0;
      if (lane == 0) {
        __threadfence_block();
        last = atomicAdd(&ucnt[iu], 1) == kBUnit - 1;
      }
      if (__shfl_sync(0xffffffffu, last, 0)) {
        __threadfence_block();
        for (int rr = r0; rr < r0 + nt; ++rr) {
          const float v = h_s[rr * kBUnit + lane];
          const float sc = b_quant_block32(v, bhq + ((size_t)rr * kBMaxNB + b) * 16, lane);
          if (lane == 0) bhs[(size_t)rr * kBMaxNB + b] = sc * rw[rr];
        }
        __syncwarp();
        if (lane == 0) b_red_release_add64(&ctr[ent], 1ull);
      }
      // next unit: stage s0 + 8
      s0 += 8;
      slot0 += 8;
      while (slot0 >= ns) {
        slot0 -= ns;
        ++lap0;
      }
    }
  }

  // ---- down: the entries' W_down rows of this CTA's output slice stream
  // through a ring that takes the span from x to the end of the up/gate
  // ring, free now (entry d in slot d % nsd, one bulk copy each) ----
  __syncthreads();
  uint8_t *dring = sbase + lay.x;
  const size_t dstage = round128((size_t)nr_max * db);
  const int nsd = (int)min((size_t)kBMaxSlots, (size_t)(ring + (size_t)ns * kStage - dring) / dstage);
  auto issue_down = [&](int d) {
    const int slot = d % nsd;
    *reinterpret_cast<volatile int *>(&dslot_stage[slot]) = d;
    if (nr > 0) {
      const uint32_t bytes = (uint32_t)(nr * db);
      mbar_arrive_expect_tx(&dbar[slot], bytes);
      bulk_g2s_hint(dring + (size_t)slot * dstage, L.dn + (int64_t)pe[d] * L.dn_expert_bytes + (int64_t)n0 * db,
                    bytes, &dbar[slot], wpol);
    } else {
      mbar_arrive(&dbar[slot]);
    }
    atomicMax(&dissued_upto, d + 1);
  };
  if (tid == 0 && status == 0)
    for (int d = 0; d < min(nsd, n_plan); ++d) issue_down(d);
  // ---- down items (route r, row group g), items w, w + 32, ... per warp;
  // the entry's stage is freed by the last of its items ----
  for (int j = warp; j < n_routes * rg; j += kBW) {
    const int r = j / rg, g = j - r * rg;
    const int ent = rplan[r];
    const int slot = ent % nsd;
    const int need = (pstart[ent + 1] - pstart[ent]) * rg;
    bool ok = *reinterpret_cast<volatile int *>(&status) == 0;
    if (ok && !wait_tagged(dslot_stage, dbar, ent, slot, ent / nsd)) {
      ok = false;
      if (lane == 0) atomicOr(&status, 2);
    }
    if (ok) {  // every unit of the entry has published its h blocks
      int have = 0;
      if (lane == 0) {
        const uint64_t t0 = global_ns();
        for (uint32_t poll = 0;; ++poll) {
          if (b_ld_acquire64(&ctr[ent]) >=
              (unsigned long long)(NB * pgroups[ent] + (ent == 0 ? L.barrier_slack : 0))) {
            have = 1;
            break;
          }
          if ((poll & 15) == 15 && global_ns() - t0 > kBWaitNs) break;
          __nanosleep(256);
        }
        if (!have) {
          atomicOr(&status, 1);
          atomicOr(L.err, kErrTimeout);
        }
      }
      ok = __shfl_sync(0xffffffffu, have, 0) != 0;
      if (ok) (void)b_ld_acquire64(&ctr[ent]);  // every lane acquires before it reads h
    }
    if (ok) {
      const int rlo = g * kBRowGroup, rhi = min(nr, rlo + kBRowGroup);
      float v[kBRowGroup];
#pragma unroll
      for (int n = 0; n < kBRowGroup; ++n) v[n] = 0.f;
      if (lane < NB) {
        const uint4 *hp = reinterpret_cast<const uint4 *>(bhq + ((size_t)r * kBMaxNB + lane) * 16);
        const uint4 h0 = __ldcg(hp), h1 = __ldcg(hp + 1), h2 = __ldcg(hp + 2), h3 = __ldcg(hp + 3);
        const float hsv = __ldcg(bhs + (size_t)r * kBMaxNB + lane);
        const uint8_t *wb = dring + (size_t)slot * dstage + (lane >> 3) * kSBBytes;
#pragma unroll
        for (int n = 0; n < kBRowGroup; ++n)
          if (rlo + n < rhi) {
            const uint8_t *row = wb + (size_t)(rlo + n) * db;
            const uint4 qv = *reinterpret_cast<const uint4 *>(row + 16 + (lane & 7) * 16);
            const float d = __half2float(*reinterpret_cast<const __half *>(row + (lane & 7) * 2));
            v[n] = (float)b_dot_block32(qv, h0, h1, h2, h3) * (d * hsv);
          }
      }
      const float tot = transpose_sum8(v, lane);
      const int n = (lane >> 2) & 7;
      if ((lane & 3) == 0 && rlo + n < rhi) part[r * nr_max + rlo + n] = tot;
    }
    __syncwarp();
    if (lane == 0 && atomicAdd(&dslot_done[slot], 1) + 1 == need) {
      dslot_done[slot] = 0;
      if (ent + nsd < n_plan && *reinterpret_cast<volatile int *>(&status) == 0) issue_down(ent + nsd);
    }
  }
  __syncthreads();

  // ---- out[t][n0 + n]: the token's routes in slot order, then the shared
  // expert ----
  for (int i = tid; i < T * nr; i += kBT) {
    const int t = i / nr, n = i - t * nr;
    float acc = 0.f;
    for (int j = 0; j < K; ++j) {
      const int rr = rof[t][j];
      if (rr >= 0) acc += part[rr * nr_max + n];
    }
    if (S) acc += part[rof[t][K] * nr_max + n];
    if (p.out_bf16)
      reinterpret_cast<__nv_bfloat16 *>(p.out)[(size_t)t * H + n0 + n] = __float2bfloat16_rn(acc);
    else
      reinterpret_cast<float *>(p.out)[(size_t)t * H + n0 + n] = acc;
  }

  // ---- exit: copies still in flight after a timeout land first ----
  if (tid == 0) {
    if (status & 3) {
      for (int s = max(0, issued_upto - ns); s < issued_upto; ++s)
        mbar_wait_ns(&full_bar[s % ns], (uint32_t)(s / ns) & 1u, kBWaitNs);
      if (nsd > 0)
        for (int d = max(0, dissued_upto - nsd); d < dissued_upto; ++d)
          mbar_wait_ns(&dbar[d % nsd], (uint32_t)(d / nsd) & 1u, kBWaitNs);
      if (router && p.wr_smem) mbar_wait_ns(&wr_bar, 0, kBWaitNs);
      if (x_smem) mbar_wait_ns(&x_bar, 0, kBWaitNs);
      if (status & 2) atomicOr(L.err, kErrTimeout);
    }
    b_red_release_add64(&L.bseq[0], 1ull);
  }
}

int batch_nsb(const Layer &L) { return L.Hp / kSBW; }
int batch_nl(const Layer &L) { return L.E <= 64 ? 2 : 4; }
int batch_nr_max(const Layer &L) { return L.sms > 0 ? (L.H + L.sms - 1) / L.sms : 0; }

size_t batch_stage(const Layer &L) {
  return batch_nsb(L) == 14 ? batch_stage_bytes<14>(batch_nr_max(L), L.dn_row_bytes)
                            : batch_stage_bytes<10>(batch_nr_max(L), L.dn_row_bytes);
}

// Shapes the kernel takes (each limit is a static array, a register tile or
// a box of the tensor map).
bool batch_shape_ok(const Layer &L) {
  const int nsb = batch_nsb(L);
  if ((nsb != 14 && nsb != 10) || L.sms < 1) return false;
  const int G = L.sms, NB = L.Fp / kBUnit;
  if (L.k > kBMaxK || L.E > 128 || L.E > G || NB > kBMaxNB || NB > G) return false;
  if (batch_nr_max(L) > kBMaxRows) return false;
  // token groups: every entry, plus one per 4 routes beyond an entry's first 4
  const int64_t max_groups = std::min(L.E, kBMaxT * L.k) + L.S + (kBMaxT * (L.k + L.S)) / kBTokPass;
  if (max_groups > kBMaxGroups || (max_groups * NB + G - 1) / G > kBMaxUnits) return false;
  if ((size_t)L.H * 4 > batch_stage(L)) return false;  // the router row fits one ring stage
  if (L.H % 8) return false;                              // eight-element router loads
  if ((int64_t)std::max(L.H, L.Fp) * G >= ((int64_t)1 << 32)) return false;
  return true;
}

// Passes over the hidden dimension, ring depth and shared-memory bytes of a
// call with T tokens; false if no configuration fits.
bool batch_plan(const Layer &L, int T, int &ns, int &xw, size_t &smem) {
  if (L.batch_smem_limit <= 0) return false;
  const size_t stage = batch_stage(L);
  const int nr_max = batch_nr_max(L), routes = T * (L.k + L.S);
  xw = L.Hp;  // every token's whole row of x
  const size_t fixed = batch_fixed_bytes(T, xw, routes, nr_max);
  if (fixed >= (size_t)L.batch_smem_limit) return false;
  const size_t n = std::min<size_t>(kBMaxSlots, ((size_t)L.batch_smem_limit - fixed) / stage);
  if (n < (size_t)kBMinSlots) return false;
  ns = (int)n;
  smem = fixed + n * stage;
  return true;
}

template <int NSB, int NL>
cudaError_t batch_prepare_one(Layer &L) {
  cudaFuncAttributes fa;
  int optin = 0;
  cudaFuncAttributes fi;
  cudaError_t e = cudaFuncGetAttributes(&fa, decode_batch_kernel<NSB, NL, false>);
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&fi, decode_batch_kernel<NSB, NL, true>);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, L.device);
  if (e != cudaSuccess) return e;
  const int fixed = (int)std::max(fa.sharedSizeBytes, fi.sharedSizeBytes);
  const int limit = optin > fixed ? optin - fixed : 0;
  e = cudaFuncSetAttribute(decode_batch_kernel<NSB, NL, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, limit);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(decode_batch_kernel<NSB, NL, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, limit);
  if (e != cudaSuccess) return e;
  L.batch_smem_limit = limit;
  int ns, xw;
  size_t smem;
  if (!batch_plan(L, kBMaxT, ns, xw, smem)) {
    L.batch_smem_limit = 0;
    return cudaSuccess;
  }
  int per_sm = 0, per_sm_i = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_batch_kernel<NSB, NL, false>, kBT, smem);
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm_i, decode_batch_kernel<NSB, NL, true>, kBT, smem);
  if (e != cudaSuccess) return e;
  if (std::min(per_sm, per_sm_i) < 1) L.batch_smem_limit = 0;
  return cudaSuccess;
}

template <int NSB, int NL>
cudaError_t batch_launch(const BParams &p, const CUtensorMap &map, size_t smem, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.L.sms);
  cfg.blockDim = dim3(kBT);
  cfg.dynamicSmemBytes = smem;
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
  return p.x_import ? cudaLaunchKernelEx(&cfg, decode_batch_kernel<NSB, NL, true>, p, map)
                    : cudaLaunchKernelEx(&cfg, decode_batch_kernel<NSB, NL, false>, p, map);
}

}  // namespace

cudaError_t batch_decode_prepare(Layer &L) {
  L.batch_smem_limit = 0;
  if (!batch_shape_ok(L)) return cudaSuccess;
  const int nsb = batch_nsb(L), nl = batch_nl(L);
  cudaError_t e = nsb == 14 ? (nl == 2 ? batch_prepare_one<14, 2>(L) : batch_prepare_one<14, 4>(L))
                            : (nl == 2 ? batch_prepare_one<10, 2>(L) : batch_prepare_one<10, 4>(L));
  return e;
}

// the up/gate weight rows as a 2D tensor of 64-bit words: one box is part 0
// of a row (NH0 superblocks) for 8 consecutive rows
cudaError_t batch_decode_maps(Layer &L) {
  if (L.batch_smem_limit <= 0) return cudaSuccess;
  const int nh0 = batch_nsb(L) == 14 ? part0_sbs<14>() : part0_sbs<10>();
  return encode_2d(&L.map_gu_half, CU_TENSOR_MAP_DATA_TYPE_UINT64, L.gu, (uint64_t)L.gu_row_bytes / 8,
                   (uint64_t)(L.E + L.S) * 2 * L.Fp, (uint64_t)L.gu_row_bytes, (uint32_t)(nh0 * kSBBytes / 8),
                   kBChunk, CU_TENSOR_MAP_SWIZZLE_NONE);
}

int batch_decode_seq_words() { return kBSeqWords; }
int64_t batch_decode_hq_floats() { return (int64_t)kBMaxRoutes * kBMaxNB * 17; }
int64_t batch_decode_part_floats(const Layer &L) { return (int64_t)kBMaxRoutes * L.Fp * 2; }
int64_t batch_decode_log_words(const Layer &L) { return (int64_t)kBMaxT * L.E * L.sms; }

bool batch_decode_supported(const Layer &L, int T) {
  if (T < 2 || T > kBMaxT || T > L.max_tokens || L.batch_smem_limit <= 0) return false;
  if (!L.bseq || !L.blog || !L.bpart || !L.bhq || !batch_shape_ok(L)) return false;
  int ns, xw;
  size_t smem;
  return batch_plan(L, T, ns, xw, smem);
}

cudaError_t launch_decode_batch(const Layer &L, const void *x, moe_dtype xdt, int T, const float *wr,
                                const float *bias, int64_t bstride, const int32_t *ids_in, const float *w_in,
                                int32_t *ids_out, float *w_out, void *out, moe_dtype odt, cudaStream_t stream,
                                void *x_import) {
  if (!batch_decode_supported(L, T)) return cudaErrorInvalidConfiguration;
  if (x_import && (xdt != MOE_DT_BF16 || L.H % 8 || !aligned(x_import, 16) || !aligned(x, 16)))
    return cudaErrorInvalidValue;
  BParams p;
  size_t smem;
  if (!batch_plan(L, T, p.ns, p.xw, smem)) return cudaErrorInvalidConfiguration;
  p.L = L;
  p.x = x;
  p.x_bf16 = xdt == MOE_DT_BF16;
  p.x_import = static_cast<uint16_t *>(x_import);
  p.T = T;
  p.wr = wr;
  p.bias = bias;
  p.bstride = bstride;
  p.ids_in = ids_in;
  p.w_in = w_in;
  p.ids_out = ids_out;
  p.w_out = w_out;
  p.out = out;
  p.out_bf16 = odt == MOE_DT_BF16;
  p.nr_max = batch_nr_max(L);
  p.wr_smem = (wr && aligned(wr, 16) && (L.H % 4) == 0) ? 1 : 0;
  count_launches(1);
  const int nsb = batch_nsb(L), nl = batch_nl(L);
  cudaError_t e = nsb == 14 ? (nl == 2 ? batch_launch<14, 2>(p, L.map_gu_half, smem, stream)
                                       : batch_launch<14, 4>(p, L.map_gu_half, smem, stream))
                            : (nl == 2 ? batch_launch<10, 2>(p, L.map_gu_half, smem, stream)
                                       : batch_launch<10, 4>(p, L.map_gu_half, smem, stream));
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace moe
