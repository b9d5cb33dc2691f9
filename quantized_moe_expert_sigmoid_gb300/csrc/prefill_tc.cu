// Batched path (T > 8 tokens) on GB300's 5th-generation tensor cores.
//
// The routes are grouped by expert (route plan), so each expert's work is a
// dense contraction over its tokens -- the grouped kernel over a CSR route
// table of PocketLLM's "Xing4.0-29B-A4B: the design record", section 4,
// re-built for tcgen05:
//   gather     x rows of every route -> fp16 rows in route order (x16)
//   up/gate    per tile (expert, 128 outputs, <= 256 routes): the gate and
//              the up rows of the same outputs are two M = 128 MMAs on one
//              activation tile, G = Wg x16^T and U = Wu x16^T in two TMEM
//              accumulators; h = silu(G) * U -> fp16
//   down       per tile (expert, 256 hidden rows, <= 256 routes): two
//              M = 128 MMAs on one h tile; out_acc[token][row] +=
//              route weight * Y (fp32), or with the deterministic combine
//              ybuf[route][row] = route weight * Y, one writer per element
//   finalize   out = round(out_acc), or the slot-ordered sum of ybuf
// Operands are fp16 (kind::f16, fp32 accumulate): the IQ4_NL codes are
// integers |c| <= 127, exact in fp16, and the per-block scale is applied when
// a tile is dequantised (one rounding of d * code); bf16 weights and h would
// cost ~3e-3 mean relative error on this layer, fp16 ~4e-4.
//
// CTA (persistent, one per SM, 19 warps):
//   warp 0      activation producer: 2D TMA copies of the fp16 activation
//               tile of every 64-wide k-step (128-byte swizzle, K-major)
//   warp 1      owns TMEM; one thread issues the tcgen05.mma of each k-step
//               once its A and B stages are full and commits them to the
//               stages' "empty" mbarriers
//   warp 2      weight producer: 2D TMA copies of the 4-bit labels of every
//               k-step (32 bytes of each of the tile's 256 weight rows)
//   warps 3-18  dequantisers (two threads per weight row, 32 weights of a
//               k-step each; the fp16 block scales come from global memory
//               one superblock ahead): fp16 d * code into the 128-byte-
//               swizzled K-major A stages; after a tile the same warps read
//               TMEM (tcgen05.ld 32x32b) for the epilogue
// Every wait is bounded; a timeout sets the layer's sticky error word.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "device_utils.cuh"
#include "moe_internal.cuh"
#include "tc_utils.cuh"

namespace moe {
namespace {

constexpr int kNT = 256;            // routes per tile (MMA N upper bound)
constexpr int kTM = 128;            // rows per MMA (M)
constexpr int kRowsTile = 2 * kTM;  // weight rows per tile: two MMAs share each B tile
constexpr int kKS = 64;             // K per k-step: one 128-byte swizzle row of fp16
constexpr int kKSteps = kSBW / kKS; // k-steps per superblock
constexpr int kDqWarps = 16;
constexpr int kDq = kDqWarps * 32;  // two dequantising threads per weight row
constexpr int kDqWarp0 = 3;         // warps 0..2: activation producer, MMA, weight producer
constexpr int kThreadsTC = kDq + 32 * kDqWarp0;
constexpr int kAStages = 3;
constexpr int kBStages = 3;
constexpr int kLabStages = 4;       // label stages, tiles of up to 256 routes
constexpr int kLabStagesSmall = 12; // tiles of up to 64 routes: the activation
                                    // stages shrink to 8 KB and the weight
                                    // labels get the room (more bytes in flight)
constexpr int kATile = kTM * kKS * 2;        // 16 KB
constexpr int kAStage = 2 * kATile;          // 32 KB
constexpr int kLabStage = kRowsTile * 32;    // labels of one k-step: 32 bytes per row
constexpr uint64_t kWaitNs = 1000000000ull;  // 1 s per wait before the CTA gives up
static_assert(kDq == 2 * kRowsTile, "two dequantising threads per weight row");

// labels -> biased bytes (code + 128) for the fp16 conversion: the int8
// decode of device_utils.cuh with every code's sign bit flipped afterwards
// (the flip cannot go into the tables: their sign bits drive PRMT's
// sign-replicate mode).  Both XORs fold into one three-input logic op.
__device__ __forceinline__ void iq4_decode8_biased(uint32_t q, uint32_t &c0, uint32_t &c1) {
  const uint32_t qx = q ^ 0x88888888u;
  c0 = prmt(kTL0, kTL1, q) ^ prmt(kTH0, kTH1, qx) ^ 0x80808080u;
  c1 = prmt(kTL0, kTL1, q >> 16) ^ prmt(kTH0, kTH1, qx >> 16) ^ 0x80808080u;
}

// four biased bytes -> two fp16x2 of d * code.  0x64XX as fp16 is 1024 + XX
// exactly, so (v - 1152) is the integer code exactly, and the product with
// the block scale is rounded once.
__device__ __forceinline__ void codes_to_half(uint32_t c, __half2 d2, uint32_t &lo, uint32_t &hi) {
  const __half2 off = __half2half2(__ushort_as_half((unsigned short)0x6480));  // 1152
  const uint32_t a = prmt(c, 0x64646464u, 0x5140);
  const uint32_t b = prmt(c, 0x64646464u, 0x5342);
  __half2 ha = __hmul2(__hsub2(*reinterpret_cast<const __half2 *>(&a), off), d2);
  __half2 hb = __hmul2(__hsub2(*reinterpret_cast<const __half2 *>(&b), off), d2);
  lo = *reinterpret_cast<uint32_t *>(&ha);
  hi = *reinterpret_cast<uint32_t *>(&hb);
}

struct TcParams {
  const TcTile *tiles;
  const int *n_tiles;
  const uint8_t *w;          // superblock rows of this matrix kind, all experts
  int64_t row_bytes;         // bytes per weight row
  int64_t rows_per_expert;   // 2 * Fp (up/gate) or Hp (down)
  const int *route_token;
  const float *route_weight;
  __half *h16;       // up/gate output [routes][Fp]
  float *out_acc;    // down output accumulator [T][H]
  float *ybuf;       // nullptr, or per-route down outputs [routes][Hp] (deterministic combine)
  unsigned *err;
  int H, Hp, Fp;
};

// Bounded wait shared by all roles: once any wait of the CTA has run out
// (`abort` set), every later wait returns at once, so a lost copy costs one
// budget, not one per wait.
__device__ __forceinline__ void wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *abort) {
  if (*abort) return;
  if (!mbar_wait_ns(bar, parity, kWaitNs)) *abort = 1;
}

// Weight row (within its expert) that tile row r (0..255) of m-tile m
// reads.  Up/gate: rows 0..127 are the gate rows, 128..255 the up rows, of
// outputs 128m..128m+127; the matrix interleaves gate and up in groups of
// 64 rows (group g: gate of outputs 64g.., then up of the same outputs).
template <bool UG>
__device__ __forceinline__ int tile_row(int m, int r) {
  if (UG) {
    const int a = r >> 7, rr = r & (kTM - 1);
    return 4 * kGroupRows * m + a * kGroupRows + (rr < kGroupRows ? rr : rr + kGroupRows);
  }
  return kRowsTile * m + r;
}

// Shared memory of a configuration: A stages, activation stages of NT rows,
// label stages.
template <int NT>
__host__ __device__ constexpr int tc_lab_stages() { return NT == kNT ? kLabStages : kLabStagesSmall; }
template <int NT>
__host__ __device__ constexpr size_t tc_smem_of() {
  return 1024 + (size_t)kAStages * kAStage + (size_t)kBStages * NT * kKS * 2 +
         (size_t)tc_lab_stages<NT>() * kLabStage;
}

// UG = true: up/gate + SwiGLU epilogue; UG = false: down + weighted scatter.
// NT: routes per tile at most (256; or 64, for batches whose experts all have
// at most 64 routes).
template <bool UG, int NT>
__global__ void __launch_bounds__(kThreadsTC, 1)
    grouped_gemm_tc(const TcParams p, const __grid_constant__ CUtensorMap b_map,
                    const __grid_constant__ CUtensorMap lab_map) {
  constexpr int kTmemCols = 2 * NT;
  constexpr int kBTileT = NT * kKS * 2;
  constexpr int kLabSt = tc_lab_stages<NT>();
  extern __shared__ uint8_t smem_dyn[];
  __shared__ uint64_t a_full[kAStages], a_empty[kAStages], b_full[kBStages], b_empty[kBStages],
      lab_full[kLabSt], lab_empty[kLabSt], acc_full, acc_empty, fin_bar;
  __shared__ uint32_t tmem_holder;
  __shared__ int abort_flag;
  volatile int *abort = &abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nsb = (UG ? p.Hp : p.Fp) / kSBW;  // superblock columns along K
  const int nks = nsb * kKSteps;
  const int ntiles = *p.n_tiles;
  // 128-byte swizzled tiles need 1024-byte aligned bases (the launch adds
  // 1 KB of slack for this)
  uint8_t *a_base = smem_dyn + ((1024u - (smem_addr(smem_dyn) & 1023u)) & 1023u);
  uint8_t *b_base = a_base + kAStages * kAStage;
  uint8_t *lab_base = b_base + kBStages * kBTileT;

  if (tid == 0) {
    for (int s = 0; s < kAStages; ++s) {
      mbar_init(&a_full[s], kDqWarps);
      mbar_init(&a_empty[s], 1);
    }
    for (int s = 0; s < kBStages; ++s) {
      mbar_init(&b_full[s], 1);
      mbar_init(&b_empty[s], 1);
    }
    for (int s = 0; s < kLabSt; ++s) {
      mbar_init(&lab_full[s], 1);
      mbar_init(&lab_empty[s], kDqWarps);
    }
    mbar_init(&acc_full, 1);
    mbar_init(&acc_empty, kDqWarps);
    mbar_init(&fin_bar, 1);
    fence_mbar_init();
    abort_flag = 0;
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(&tmem_holder)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_holder;

  if (warp == 0 || warp == 2) {
    // ===================== producers (activations / labels) =====================
    if (lane == 0) {
      const bool act = warp == 0;
      const int nst = act ? kBStages : kLabSt;
      uint64_t *full = act ? b_full : lab_full;
      uint64_t *empty = act ? b_empty : lab_empty;
      uint32_t q = 0;
      for (int ti = blockIdx.x; ti < ntiles && !*abort; ti += gridDim.x) {
        const TcTile t = p.tiles[ti];
        const int wrow0 = (int)(t.expert * p.rows_per_expert) + t.mtile * kRowsTile;
        for (int ks = 0; ks < nks; ++ks, ++q) {
          const int s = q % nst;
          if (q >= (uint32_t)nst) wait_or_abort(&empty[s], ((q / nst) - 1) & 1u, abort);
          if (*abort) break;
          if (act) {
            mbar_arrive_expect_tx(&full[s], kBTileT);
            tma_load_2d(b_base + s * kBTileT, &b_map, ks * kKS, t.row0, &full[s]);
          } else {
            uint8_t *dst = lab_base + s * kLabStage;
            const int xo = (ks >> 2) * kSBBytes + 16 + 32 * (ks & 3);  // blocks 2kk, 2kk+1
            mbar_arrive_expect_tx(&full[s], kLabStage);
            if (UG) {  // gate rows of groups 2m, 2m+1, then their up rows (tile_row order)
              tma_load_2d(dst, &lab_map, xo, wrow0, &full[s]);
              tma_load_2d(dst + 64 * 32, &lab_map, xo, wrow0 + 2 * kGroupRows, &full[s]);
              tma_load_2d(dst + 128 * 32, &lab_map, xo, wrow0 + kGroupRows, &full[s]);
              tma_load_2d(dst + 192 * 32, &lab_map, xo, wrow0 + 3 * kGroupRows, &full[s]);
            } else {
              tma_load_2d(dst, &lab_map, xo, wrow0, &full[s]);
            }
          }
        }
      }
      // no copy may still be landing in shared memory when the CTA exits:
      // wait for the last phase issued on every full barrier (the normal
      // path has consumed them all already, so these return at once)
      for (int s = 0; s < nst; ++s) {
        const uint32_t uses = q / nst + ((uint32_t)s < q % nst ? 1u : 0u);
        if (uses > 0) mbar_wait_ns(&full[s], (uses - 1) & 1u, kWaitNs);
      }
    }
  } else if (warp == 1) {
    // ============================ MMA issue ============================
    if (lane == 0) {
      uint32_t q = 0, tcount = 0;
      for (int ti = blockIdx.x; ti < ntiles; ti += gridDim.x, ++tcount) {
        const int count = p.tiles[ti].count;
        const int n_mma = min(NT, (count + 15) & ~15);
        const uint32_t idesc =
            (1u << 4) | ((uint32_t)(n_mma >> 3) << 17) | ((uint32_t)(kTM >> 4) << 24);
        if (tcount > 0) wait_or_abort(&acc_empty, (tcount - 1) & 1u, abort);  // TMEM drained
        tc_fence_after();
        for (int ks = 0; ks < nks; ++ks, ++q) {
          const int sa = q % kAStages, sb = q % kBStages;
          wait_or_abort(&a_full[sa], (q / kAStages) & 1u, abort);
          wait_or_abort(&b_full[sb], (q / kBStages) & 1u, abort);
          if (*abort) continue;
          tc_fence_after();
          const uint32_t as = smem_addr(a_base + sa * kAStage);
          const uint32_t bs = smem_addr(b_base + sb * kBTileT);
#pragma unroll
          for (int a = 0; a < 2; ++a)
#pragma unroll
            for (int k16 = 0; k16 < kKS / 16; ++k16)
              umma_f16(tmem + a * NT, sw128_desc(as + a * kATile + 32 * k16),
                       sw128_desc(bs + 32 * k16), idesc, (ks | k16) != 0);
          umma_commit(&a_empty[sa]);  // the A stage may be rewritten once these finish
          umma_commit(&b_empty[sb]);  // ... and the B stage refilled
        }
        if (!*abort) umma_commit(&acc_full);
      }
      // every MMA issued has finished before TMEM is released
      umma_commit(&fin_bar);
      mbar_wait_ns(&fin_bar, 0, kWaitNs);
    }
  } else {
    // ====================== dequantise + epilogue ======================
    const int dt = tid - 32 * kDqWarp0;
    const int r = dt >> 1, blk = dt & 1;  // tile row, block parity within a k-step
    const int a = r >> 7, rr = r & (kTM - 1);
    const int quad = warp & 3;            // TMEM lanes 32*quad .. 32*quad+31
    const int qc = (warp - kDqWarp0) >> 2;  // column quarter of the epilogue
    // fp16 scales of the row's superblocks: 16 bytes each, one superblock ahead
    auto row_ptr = [&](int ti) -> const uint8_t * {
      if (ti >= ntiles) return nullptr;
      const TcTile tn = p.tiles[ti];
      return p.w + ((int64_t)tn.expert * p.rows_per_expert + tile_row<UG>(tn.mtile, r)) * p.row_bytes;
    };
    const uint8_t *rowp = row_ptr(blockIdx.x);
    uint4 sc_cur = make_uint4(0, 0, 0, 0), sc_nxt = sc_cur;
    if (rowp) sc_cur = __ldg(reinterpret_cast<const uint4 *>(rowp));
    uint32_t q = 0, tcount = 0;
    for (int ti = blockIdx.x; ti < ntiles; ti += gridDim.x, ++tcount) {
      const TcTile t = p.tiles[ti];
      const uint8_t *nrowp = row_ptr(ti + gridDim.x);
      for (int sbc = 0; sbc < nsb; ++sbc) {
        if (sbc + 1 < nsb)
          sc_nxt = __ldg(reinterpret_cast<const uint4 *>(rowp + (sbc + 1) * kSBBytes));
        else if (nrowp)
          sc_nxt = __ldg(reinterpret_cast<const uint4 *>(nrowp));
#pragma unroll
        for (int kk = 0; kk < kKSteps; ++kk, ++q) {
          const int sl = q % kLabSt;
          wait_or_abort(&lab_full[sl], (q / kLabSt) & 1u, abort);
          const uint4 lab = *reinterpret_cast<const uint4 *>(lab_base + sl * kLabStage + r * 32 + blk * 16);
          __syncwarp();
          if (lane == 0) mbar_arrive(&lab_empty[sl]);  // the labels are in registers
          const int sa = q % kAStages;
          if (q >= kAStages) wait_or_abort(&a_empty[sa], ((q / kAStages) - 1) & 1u, abort);
          const uint32_t sw = kk == 0 ? sc_cur.x : kk == 1 ? sc_cur.y : kk == 2 ? sc_cur.z : sc_cur.w;
          const __half2 d2 = __half2half2(__ushort_as_half((unsigned short)(blk ? sw >> 16 : sw & 0xFFFF)));
          const uint32_t ww[4] = {lab.x, lab.y, lab.z, lab.w};
          uint8_t *arow = a_base + sa * kAStage + a * kATile + rr * 128;
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {  // 8 weights: chunk 4*blk + cc of the row's k-step
            const int c = 4 * blk + cc;
            uint32_t b0, b1, h0, h1, h2, h3;
            iq4_decode8_biased(ww[cc], b0, b1);
            codes_to_half(b0, d2, h0, h1);
            codes_to_half(b1, d2, h2, h3);
            *reinterpret_cast<uint4 *>(arow + ((c ^ (rr & 7)) << 4)) = make_uint4(h0, h1, h2, h3);
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // A tile -> tensor core
          __syncwarp();
          if (lane == 0) mbar_arrive(&a_full[sa]);
        }
        sc_cur = sc_nxt;
      }
      rowp = nrowp;

      // ---- epilogue: TMEM -> registers -> global ----
      wait_or_abort(&acc_full, tcount & 1u, abort);
      tc_fence_after();
      // Down: the tile's route tokens and weights, read once into the first
      // A stage -- every MMA of the tile has finished, and no dequantiser
      // writes an A stage again before the barrier closing this epilogue.
      int *ep_tok = reinterpret_cast<int *>(a_base);
      float *ep_w = reinterpret_cast<float *>(a_base + NT * sizeof(int));
      if (!UG) {
        for (int j = dt; j < t.count; j += kDq) {
          ep_tok[j] = p.route_token[t.row0 + j];
          ep_w[j] = p.route_weight[t.row0 + j];
        }
        named_sync(1, kDq);
      }
      const bool live = __shfl_sync(0xffffffffu, *abort == 0 ? 1 : 0, 0) != 0;
      const int trow = 32 * quad + lane;  // accumulator row (TMEM lane) of this thread
      const uint32_t tbase = tmem + ((uint32_t)(32 * quad) << 16);
      if (live) {
        for (int c0 = qc * (NT / 4); c0 < (qc + 1) * (NT / 4) && c0 < t.count; c0 += 16) {
          uint32_t g[16], u[16];
          tmem_ld16_nowait(tbase + c0, g);
          tmem_ld16_nowait(tbase + NT + c0, u);
          tmem_wait_ld();
          if (UG) {
            const int f = t.mtile * kTM + trow;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int col = c0 + j;
              if (col < t.count) {
                const float gv = __uint_as_float(g[j]), uv = __uint_as_float(u[j]);
                // silu(g) = g / (1 + e^-g); e^-g capped at e^80 keeps the
                // fast divide in range (the quotient is ~0 there anyway)
                const float h = __fdividef(gv, 1.0f + __expf(fminf(-gv, 80.0f))) * uv;
                if (!(fabsf(h) <= 65504.f)) atomicOr(p.err, kErrOverflow);
                p.h16[(int64_t)(t.row0 + col) * p.Fp + f] = __float2half_rn(h);
              }
            }
          } else {
            const int n0 = t.mtile * kRowsTile + trow, n1 = n0 + kTM;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int col = c0 + j;
              if (col < t.count) {
                const float wgt = ep_w[col];
                if (p.ybuf) {  // one writer per element; the combine adds in slot order
                  float *yrow = p.ybuf + (int64_t)(t.row0 + col) * p.Hp;
                  if (n0 < p.H) yrow[n0] = wgt * __uint_as_float(g[j]);
                  if (n1 < p.H) yrow[n1] = wgt * __uint_as_float(u[j]);
                } else {
                  float *orow = p.out_acc + (int64_t)ep_tok[col] * p.H;
                  if (n0 < p.H) atomicAdd(orow + n0, wgt * __uint_as_float(g[j]));
                  if (n1 < p.H) atomicAdd(orow + n1, wgt * __uint_as_float(u[j]));
                }
              }
            }
          }
        }
      }
      tc_fence_before();
      if (!UG) named_sync(1, kDq);  // ep_tok / ep_w read by all before A is rewritten
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                 : "memory");
  }
  if (tid == 0 && abort_flag) atomicOr(p.err, kErrTimeout);
}

// x rows in route order as fp16 (zero beyond H); out-of-range magnitudes
// flag an overflow.
template <typename XT>
__global__ void gather_x16_kernel(const XT *__restrict__ x, const int *__restrict__ route_token,
                                  const int *__restrict__ total, int H, int Hp, int max_rows,
                                  __half *__restrict__ x16, unsigned *err, float4 *__restrict__ zero,
                                  unsigned zero_n4) {
  // one 8-element chunk; the launcher keeps max_rows * Hp / 8 below 2^32, so
  // the row split is a 32-bit division (a 64-bit one is a long sequence)
  const unsigned i = blockIdx.x * blockDim.x + threadIdx.x;
  pdl_wait();  // the route plan (and x) come from earlier launches
  pdl_launch_dependents();
  // clear the output accumulator of the batched paths (grid-stride; the
  // grid has a thread per chunk, more than the accumulator's float4s)
  if (zero)
    for (unsigned j = i; j < zero_n4; j += gridDim.x * blockDim.x) zero[j] = make_float4(0.f, 0.f, 0.f, 0.f);
  const unsigned hp8 = (unsigned)Hp / 8u;
  const int row = (int)(i / hp8);
  const int c8 = (int)(i % hp8);
  if (row >= max_rows || row >= *total) return;
  float v[8];
  if (c8 * 8 < H) {
    const XT *src = x + (int64_t)route_token[row] * H + c8 * 8;
    if constexpr (sizeof(XT) == 2) {
      const uint4 a = *reinterpret_cast<const uint4 *>(src);
      const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        v[2 * k] = __uint_as_float(w[k] << 16);
        v[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
      }
    } else {
      const float4 a = *reinterpret_cast<const float4 *>(src);
      const float4 b = *reinterpret_cast<const float4 *>(src + 4);
      v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
      v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
  } else {
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] = 0.f;
  }
  bool big = false;
  uint32_t o[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    big |= !(fabsf(v[2 * k]) <= 65504.f) || !(fabsf(v[2 * k + 1]) <= 65504.f);
    __half2 h = __floats2half2_rn(v[2 * k], v[2 * k + 1]);
    o[k] = *reinterpret_cast<uint32_t *>(&h);
  }
  if (big) atomicOr(err, kErrOverflow);
  *reinterpret_cast<uint4 *>(x16 + row * Hp + c8 * 8) = make_uint4(o[0], o[1], o[2], o[3]);
}

}  // namespace

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::mutex g_encode_mu;
}  // namespace


cudaError_t get_encode() {
  std::lock_guard<std::mutex> lock(g_encode_mu);
  if (g_encode) return cudaSuccess;
  cudaDriverEntryPointQueryResult q;
  void *fn = nullptr;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                    cudaEnableDefault, &q);
  if (e != cudaSuccess) return e;
  if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return cudaSuccess;
}

cudaError_t encode_2d(CUtensorMap *map, CUtensorMapDataType dt, void *base, uint64_t inner,
                      uint64_t rows, uint64_t row_pitch, uint32_t box_inner, uint32_t box_rows,
                      CUtensorMapSwizzle swz) {
  cudaError_t e = get_encode();
  if (e != cudaSuccess) return e;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {row_pitch};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, dt, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swz, CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

static_assert(tc_smem_of<kNT>() <= 232448 && tc_smem_of<64>() <= 232448, "shared memory");


int tc_tile_routes(int T) { return T <= 64 ? 64 : kNT; }

int tc_max_tiles(const Layer &L, bool up_gate) {
  // route tiles of 64 (small batches) or 256 routes, plus one partial tile per expert
  const int64_t route_tiles = (int64_t)L.max_routes / 64 + L.E + L.S;
  return (int)(route_tiles * (up_gate ? L.Fp / kTM : L.Hp / kRowsTile));
}

cudaError_t tc_prepare(Layer &L) {
  cudaError_t e = get_encode();
  if (e != cudaSuccess) return e;
  // labels of one k-step: 32 bytes of each of 64 (up/gate: one gate/up
  // group) or 256 (down) consecutive rows
  e = encode_2d(&L.map_gu_lab, CU_TENSOR_MAP_DATA_TYPE_UINT8, L.gu, (uint64_t)L.gu_row_bytes,
                (uint64_t)(L.E + L.S) * 2 * L.Fp, (uint64_t)L.gu_row_bytes, 32, kGroupRows,
                CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e == cudaSuccess)
    e = encode_2d(&L.map_dn_lab, CU_TENSOR_MAP_DATA_TYPE_UINT8, L.dn, (uint64_t)L.dn_row_bytes,
                  (uint64_t)(L.E + L.S) * L.Hp, (uint64_t)L.dn_row_bytes, 32, kRowsTile,
                  CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e == cudaSuccess)
    e = encode_2d(&L.map_x16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, L.x16, (uint64_t)L.Hp,
                (uint64_t)L.max_routes, (uint64_t)L.Hp * 2, kKS, kNT, CU_TENSOR_MAP_SWIZZLE_128B);
  if (e == cudaSuccess)
    e = encode_2d(&L.map_x16_64, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, L.x16, (uint64_t)L.Hp,
                  (uint64_t)L.max_routes, (uint64_t)L.Hp * 2, kKS, 64, CU_TENSOR_MAP_SWIZZLE_128B);
  if (e == cudaSuccess)
    e = encode_2d(&L.map_h16_64, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, L.h16, (uint64_t)L.Fp,
                  (uint64_t)L.max_routes, (uint64_t)L.Fp * 2, kKS, 64, CU_TENSOR_MAP_SWIZZLE_128B);
  if (e == cudaSuccess)
    e = encode_2d(&L.map_h16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, L.h16, (uint64_t)L.Fp,
                  (uint64_t)L.max_routes, (uint64_t)L.Fp * 2, kKS, kNT, CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(grouped_gemm_tc<true, kNT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)tc_smem_of<kNT>());
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(grouped_gemm_tc<false, kNT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)tc_smem_of<kNT>());
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(grouped_gemm_tc<true, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)tc_smem_of<64>());
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(grouped_gemm_tc<false, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)tc_smem_of<64>());
  return e;
}

cudaError_t launch_gather_x16(const Layer &L, const void *x, moe_dtype xdt, int T, cudaStream_t stream) {
  const int max_rows = T * L.k + L.S * T;
  const int64_t chunks = (int64_t)max_rows * (L.Hp / 8);
  if (chunks + 255 >= ((int64_t)1 << 32)) return cudaErrorInvalidValue;  // 32-bit chunk index
  const int gb = (int)((chunks + 255) / 256);
  float4 *zero = L.deterministic ? nullptr : reinterpret_cast<float4 *>(L.out_acc);
  const unsigned zero_n4 = (unsigned)((int64_t)T * L.H / 4);  // H is a multiple of 32
  if (xdt == MOE_DT_BF16)
    return count_and_check(launch_pdl(gather_x16_kernel<__nv_bfloat16>, dim3(gb), dim3(256), 0, stream,
                                      (const __nv_bfloat16 *)x, (const int *)L.route_token,
                                      (const int *)(L.offsets + L.E + L.S), L.H, L.Hp, max_rows, L.x16, L.err,
                                      zero, zero_n4));
  return count_and_check(launch_pdl(gather_x16_kernel<float>, dim3(gb), dim3(256), 0, stream, (const float *)x,
                                    (const int *)L.route_token, (const int *)(L.offsets + L.E + L.S), L.H,
                                    L.Hp, max_rows, L.x16, L.err, zero, zero_n4));
}

cudaError_t launch_prefill_tc(const Layer &L, const void *x, moe_dtype xdt, int T,
                              cudaStream_t stream, cudaEvent_t *ev) {
  cudaError_t e;
  // gather x in route order as fp16
  if ((e = launch_gather_x16(L, x, xdt, T, stream)) != cudaSuccess) return e;

  TcParams p;
  p.route_token = L.route_token;
  p.route_weight = L.route_weight;
  p.h16 = L.h16;
  p.out_acc = L.out_acc;
  p.ybuf = L.deterministic ? L.ybuf : nullptr;
  p.err = L.err;
  p.H = L.H;
  p.Hp = L.Hp;
  p.Fp = L.Fp;
  // up/gate + SwiGLU
  p.tiles = L.tiles_ug;
  p.n_tiles = L.tile_counts;
  p.w = L.gu;
  p.row_bytes = L.gu_row_bytes;
  p.rows_per_expert = 2 * (int64_t)L.Fp;
  if (ev && (e = cudaEventRecordWithFlags(ev[0], stream, cudaEventRecordExternal)) != cudaSuccess) return e;
  // batches of at most 64 tokens: route tiles of <= 64 (the plan splits
  // there), the small-tile configuration
  const bool small = tc_tile_routes(T) == 64;
  if (small)
    grouped_gemm_tc<true, 64><<<L.sms, kThreadsTC, tc_smem_of<64>(), stream>>>(p, L.map_x16_64, L.map_gu_lab);
  else
    grouped_gemm_tc<true, kNT><<<L.sms, kThreadsTC, tc_smem_of<kNT>(), stream>>>(p, L.map_x16, L.map_gu_lab);
  count_launches(1);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (ev && (e = cudaEventRecordWithFlags(ev[1], stream, cudaEventRecordExternal)) != cudaSuccess) return e;
  // down + weighted scatter
  p.tiles = L.tiles_dn;
  p.n_tiles = L.tile_counts + 1;
  p.w = L.dn;
  p.row_bytes = L.dn_row_bytes;
  p.rows_per_expert = L.Hp;
  if (small)
    grouped_gemm_tc<false, 64><<<L.sms, kThreadsTC, tc_smem_of<64>(), stream>>>(p, L.map_h16_64, L.map_dn_lab);
  else
    grouped_gemm_tc<false, kNT><<<L.sms, kThreadsTC, tc_smem_of<kNT>(), stream>>>(p, L.map_h16, L.map_dn_lab);
  count_launches(1);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (ev) return cudaEventRecordWithFlags(ev[2], stream, cudaEventRecordExternal);
  return cudaSuccess;
}

}  // namespace moe
