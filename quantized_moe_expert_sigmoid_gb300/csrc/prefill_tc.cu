// Batched path (T > 8 tokens) on GB300's 5th-generation tensor cores.
//
// The routes are grouped by expert (route plan), so each expert's work is a
// dense contraction over its tokens -- the grouped kernel over a CSR route
// table of PocketLLM's "Xing4.0-29B-A4B: the design record", section 4,
// re-built for tcgen05:
//   gather     x rows of every route -> fp16 rows in route order (x16)
//   up/gate    per tile (expert, 128 outputs, <= 256 routes):
//              G = Wg x16^T and U = Wu x16^T in two TMEM accumulators
//              (M = 128, N = routes, K = hidden), h = silu(G) * U -> fp16
//   down       per tile (expert, 128 hidden rows, <= 256 routes):
//              Y = Wd h^T; out_acc[token][row] += route weight * Y (fp32)
//   finalize   out = round(out_acc)
// Operands are fp16 (kind::f16, fp32 accumulate): the IQ4_NL codes are
// integers |c| <= 127, exact in fp16, and the per-block scale is applied when
// a tile is dequantised (one rounding of d * code); bf16 weights and h would
// cost ~3e-3 mean relative error on this layer, fp16 ~4e-4.
//
// CTA (persistent, one per SM, 288 threads):
//   warp 0     producer: 2D TMA copies of raw IQ4_NL superblock columns
//              (144-byte units, no swizzle) and of the fp16 activation tile
//              for every 64-wide k-step (128-byte swizzle, K-major)
//   warps 1-8  consumers: dequantise the raw rows into fp16 A tiles in the
//              same 128-byte-swizzled K-major layout; after a named barrier
//              one thread issues the tcgen05.mma of the k-step and commits
//              them to the stage's "empty" mbarrier; after a tile, the same
//              warps read TMEM (tcgen05.ld 32x32b) for the epilogue.
// Every wait is bounded; a timeout sets the layer's sticky error word.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "device_utils.cuh"
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kNT = 256;   // routes per tile (MMA N upper bound)
constexpr int kTM = 128;   // weight rows per MMA (M)
constexpr int kKS = 64;    // K per k-step: one 128-byte swizzle row of fp16
constexpr int kConsWarps = 8;
constexpr int kCons = kConsWarps * 32;
constexpr int kThreadsTC = kCons + 32;
constexpr int kOpStages = 2;
constexpr int kRawStages = 2;
constexpr int kATile = kTM * kKS * 2;  // 16 KB
constexpr int kBTile = kNT * kKS * 2;  // 32 KB
constexpr uint64_t kWaitNs = 1000000000ull;  // 1 s per wait before the CTA gives up

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

__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFF);
  d |= (uint64_t)1 << 16;            // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;  // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;            // descriptor version
  d |= (uint64_t)2 << 61;            // 128-byte swizzle
  return d;
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int c0, int c1,
                                            uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void umma_f16(uint32_t tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15},"
      " [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

struct TcParams {
  const TcTile *tiles;
  const int *n_tiles;
  const int *route_token;
  const float *route_weight;
  __half *h16;       // up/gate output [routes][Fp]
  float *out_acc;    // down output accumulator [T][H]
  unsigned *err;
  int H, Hp, Fp;
  int64_t gu_rows_per_expert;  // 2 * Fp
  int64_t dn_rows_per_expert;  // Hp
};

// Bounded wait shared by all roles: once any wait of the CTA has run out
// (`abort` set), every later wait returns at once, so a lost copy costs one
// budget, not one per wait.
__device__ __forceinline__ void wait_or_abort(uint64_t *bar, uint32_t parity, volatile int *abort) {
  if (*abort) return;
  if (!mbar_wait_ns(bar, parity, kWaitNs)) *abort = 1;
}

// UG = true: up/gate (two A tiles per k-step: gate and up rows of the same
// 128 outputs); UG = false: down (one A tile of 128 hidden rows).
template <bool UG>
__global__ void __launch_bounds__(kThreadsTC, 1)
    grouped_gemm_tc(const TcParams p, const __grid_constant__ CUtensorMap raw_map,
                    const __grid_constant__ CUtensorMap b_map) {
  constexpr int NA = UG ? 2 : 1;
  constexpr int kRawRows = NA * kTM;
  constexpr int kRawBytes = kRawRows * kSBBytes;
  constexpr int kOpBytes = NA * kATile + kBTile;
  constexpr int kTmemCols = UG ? 512 : 256;
  constexpr int kKSteps = kSBW / kKS;
  extern __shared__ uint8_t smem_dyn[];
  __shared__ uint64_t op_full[kOpStages], op_empty[kOpStages], raw_full[kRawStages],
      raw_empty[kRawStages], acc_bar, fin_bar;
  __shared__ uint32_t tmem_holder;
  __shared__ int abort_flag;
  volatile int *abort = &abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nsb = (UG ? p.Hp : p.Fp) / kSBW;  // superblock columns along K
  const int ntiles = *p.n_tiles;
  // 128-byte swizzled tiles need 1024-byte aligned bases (the launch adds
  // 1 KB of slack for this)
  uint8_t *op_base = smem_dyn + ((1024u - (smem_addr(smem_dyn) & 1023u)) & 1023u);
  uint8_t *raw_base = op_base + kOpStages * kOpBytes;

  if (tid == 0) {
    for (int s = 0; s < kOpStages; ++s) {
      mbar_init(&op_full[s], 1);
      mbar_init(&op_empty[s], 1);
    }
    for (int r = 0; r < kRawStages; ++r) {
      mbar_init(&raw_full[r], 1);
      mbar_init(&raw_empty[r], kConsWarps);
    }
    mbar_init(&acc_bar, 1);
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

  if (warp == 0) {
    // ============================ producer ============================
    if (lane == 0) {
      uint32_t q = 0, v = 0;
      for (int ti = blockIdx.x; ti < ntiles && !*abort; ti += gridDim.x) {
        const TcTile t = p.tiles[ti];
        for (int sbc = 0; sbc < nsb && !*abort; ++sbc, ++v) {
          const int r = v % kRawStages;
          if (v >= kRawStages) wait_or_abort(&raw_empty[r], ((v / kRawStages) - 1) & 1u, abort);
          if (*abort) break;
          uint8_t *raw = raw_base + r * kRawBytes;
          mbar_arrive_expect_tx(&raw_full[r], kRawBytes);
          if (UG) {  // gate rows of groups 2m, 2m+1, then their up rows
            const int row0 = (int)(t.expert * p.gu_rows_per_expert) + t.mtile * (4 * kGroupRows);
            tma_load_2d(raw, &raw_map, sbc * kSBBytes, row0, &raw_full[r]);
            tma_load_2d(raw + 64 * kSBBytes, &raw_map, sbc * kSBBytes, row0 + 2 * kGroupRows,
                        &raw_full[r]);
            tma_load_2d(raw + 128 * kSBBytes, &raw_map, sbc * kSBBytes, row0 + kGroupRows,
                        &raw_full[r]);
            tma_load_2d(raw + 192 * kSBBytes, &raw_map, sbc * kSBBytes, row0 + 3 * kGroupRows,
                        &raw_full[r]);
          } else {
            const int row0 = (int)(t.expert * p.dn_rows_per_expert) + t.mtile * kTM;
            tma_load_2d(raw, &raw_map, sbc * kSBBytes, row0, &raw_full[r]);
          }
          for (int kk = 0; kk < kKSteps; ++kk, ++q) {
            const int s = q % kOpStages;
            if (q >= kOpStages) wait_or_abort(&op_empty[s], ((q / kOpStages) - 1) & 1u, abort);
            if (*abort) break;
            uint8_t *bdst = op_base + s * kOpBytes + NA * kATile;
            mbar_arrive_expect_tx(&op_full[s], kBTile);
            tma_load_2d(bdst, &b_map, sbc * kSBW + kk * kKS, t.row0, &op_full[s]);
          }
        }
      }
      // no copy may still be landing in shared memory when the CTA exits:
      // wait for the last phase issued on every full barrier (the normal
      // path has consumed them all already, so these return at once)
      for (int r = 0; r < kRawStages; ++r) {
        const uint32_t uses = v / kRawStages + ((uint32_t)r < v % kRawStages ? 1u : 0u);
        if (uses > 0) mbar_wait_ns(&raw_full[r], (uses - 1) & 1u, kWaitNs);
      }
      for (int s = 0; s < kOpStages; ++s) {
        const uint32_t uses = q / kOpStages + ((uint32_t)s < q % kOpStages ? 1u : 0u);
        if (uses > 0) mbar_wait_ns(&op_full[s], (uses - 1) & 1u, kWaitNs);
      }
    }
  } else {
    // ============================ consumers ============================
    // Every consumer thread runs the same trip counts whatever happens, so
    // the named barrier below always completes; an abort only skips waits
    // and MMA issue.
    const int ct = tid - 32;
    uint32_t q = 0, v = 0, tcount = 0;
    for (int ti = blockIdx.x; ti < ntiles; ti += gridDim.x) {
      const TcTile t = p.tiles[ti];
      const int n_mma = min(kNT, (t.count + 15) & ~15);
      const uint32_t idesc = (1u << 4) | ((uint32_t)(n_mma >> 3) << 17) | ((uint32_t)(kTM >> 4) << 24);
      for (int sbc = 0; sbc < nsb; ++sbc, ++v) {
        const int r = v % kRawStages;
        wait_or_abort(&raw_full[r], (v / kRawStages) & 1u, abort);
        const uint8_t *raw = raw_base + r * kRawBytes;
        for (int kk = 0; kk < kKSteps; ++kk, ++q) {
          const int s = q % kOpStages;
          if (q >= kOpStages) wait_or_abort(&op_empty[s], ((q / kOpStages) - 1) & 1u, abort);
          uint8_t *stage = op_base + s * kOpBytes;
          // ---- dequantise this k-step's A rows into the swizzled fp16 tile(s)
          if (UG) {  // thread = one raw row: 0..127 gate, 128..255 up; 64 weights
            const int rr = ct;
            const uint8_t *row = raw + rr * kSBBytes;
            const int tr = rr & (kTM - 1);
            uint8_t *atile = stage + (rr >> 7) * kATile + tr * 128;
            const uint32_t sc = *reinterpret_cast<const uint32_t *>(row + 4 * kk);  // 2 fp16 scales
            const uint4 w0 = *reinterpret_cast<const uint4 *>(row + 16 + 32 * kk);
            const uint4 w1 = *reinterpret_cast<const uint4 *>(row + 32 + 32 * kk);
            const uint32_t ww[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
            for (int c = 0; c < 8; ++c) {  // chunk c = weights 8c..8c+7 of the k-step
              const unsigned short dbits = (unsigned short)(c < 4 ? (sc & 0xFFFF) : (sc >> 16));
              const __half2 d2 = __half2half2(__ushort_as_half(dbits));
              uint32_t b0, b1, h0, h1, h2, h3;
              iq4_decode8_biased(ww[c], b0, b1);
              codes_to_half(b0, d2, h0, h1);
              codes_to_half(b1, d2, h2, h3);
              *reinterpret_cast<uint4 *>(atile + ((c ^ (tr & 7)) << 4)) = make_uint4(h0, h1, h2, h3);
            }
          } else {  // two threads per row: block 2kk + half, 32 weights each
            const int rr = ct >> 1, half = ct & 1;
            const uint8_t *row = raw + rr * kSBBytes;
            uint8_t *atile = stage + rr * 128;
            const unsigned short dbits = *reinterpret_cast<const unsigned short *>(row + 2 * (2 * kk + half));
            const __half2 d2 = __half2half2(__ushort_as_half(dbits));
            const uint4 w = *reinterpret_cast<const uint4 *>(row + 16 + 16 * (2 * kk + half));
            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
              const int c = 4 * half + cc;
              uint32_t b0, b1, h0, h1, h2, h3;
              iq4_decode8_biased(ww[cc], b0, b1);
              codes_to_half(b0, d2, h0, h1);
              codes_to_half(b1, d2, h2, h3);
              *reinterpret_cast<uint4 *>(atile + ((c ^ (rr & 7)) << 4)) = make_uint4(h0, h1, h2, h3);
            }
          }
          if (kk == kKSteps - 1) {  // this warp is done with the raw stage
            __syncwarp();
            if (lane == 0) mbar_arrive(&raw_empty[r]);
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // A tiles -> tensor core
          named_sync(1, kCons);
          if (ct == 0) {
            wait_or_abort(&op_full[s], (q / kOpStages) & 1u, abort);
            if (!*abort) {
              tc_fence_after();
              const uint32_t bsm = smem_addr(stage + NA * kATile);
#pragma unroll
              for (int a = 0; a < NA; ++a) {
                const uint32_t asm_ = smem_addr(stage + a * kATile);
#pragma unroll
                for (int k16 = 0; k16 < kKS / 16; ++k16)
                  umma_f16(tmem + a * kNT, sw128_desc(asm_ + 32 * k16), sw128_desc(bsm + 32 * k16),
                           idesc, (sbc | kk | k16) != 0);
              }
              umma_commit(&op_empty[s]);  // frees A and B of this stage once the MMAs finish
              if (sbc == nsb - 1 && kk == kKSteps - 1) umma_commit(&acc_bar);
            }
          }
        }
      }
      // ---- epilogue: TMEM -> registers -> global ----
      wait_or_abort(&acc_bar, tcount & 1u, abort);
      tc_fence_after();
      const bool live = !*abort;            // warp-uniform enough: only gates stores
      const int quad = warp & 3;            // TMEM lanes 32*quad .. 32*quad+31
      const int colh = (warp - 1) >> 2;     // which half of the columns
      const int trow = 32 * quad + lane;    // tile row of this thread
      const uint32_t tbase = tmem + ((uint32_t)(32 * quad) << 16);
      for (int c0 = colh * (kNT / 2); c0 < (colh + 1) * (kNT / 2) && c0 < t.count; c0 += 16) {
        uint32_t g[16];
        tmem_ld16(tbase + c0, g);
        if (UG) {
          uint32_t u[16];
          tmem_ld16(tbase + kNT + c0, u);
          const int f = t.mtile * kTM + trow;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int col = c0 + j;
            if (live && col < t.count) {
              const float gv = __uint_as_float(g[j]), uv = __uint_as_float(u[j]);
              const float h = gv / (1.0f + expf(-gv)) * uv;
              if (!(fabsf(h) <= 65504.f)) atomicOr(p.err, kErrOverflow);
              p.h16[(int64_t)(t.row0 + col) * p.Fp + f] = __float2half_rn(h);
            }
          }
        } else {
          const int n = t.mtile * kTM + trow;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int col = c0 + j;
            if (live && col < t.count && n < p.H) {
              const int pos = t.row0 + col;
              atomicAdd(p.out_acc + (int64_t)p.route_token[pos] * p.H + n,
                        p.route_weight[pos] * __uint_as_float(g[j]));
            }
          }
        }
      }
      tc_fence_before();
      ++tcount;
    }
    // all MMAs this thread issued have finished before TMEM is released
    if (ct == 0) {
      umma_commit(&fin_bar);
      mbar_wait_ns(&fin_bar, 0, kWaitNs);
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

// Tile lists from the route plan: for every expert with routes, route tiles
// of <= 256 and, per route tile, every 128-row weight tile.  Lane 0 walks
// the (expert, route tile) pairs; the warp writes their weight tiles.
__global__ void build_tiles_kernel(const int *offsets, const int *active, int n_slots_idx,
                                   int ug_mtiles, int dn_mtiles, TcTile *ug, TcTile *dn,
                                   int *counts, int max_ug, int max_dn) {
  const int lane = threadIdx.x;
  const int n_act = active[n_slots_idx];
  int nu = 0, nd = 0;
  for (int i = 0; i < n_act; ++i) {
    const int e = active[i];
    const int beg = offsets[e], cnt = offsets[e + 1] - beg;
    for (int n0 = 0; n0 < cnt; n0 += kNT) {
      const int c = min(kNT, cnt - n0);
      for (int m = lane; m < ug_mtiles; m += 32)
        if (nu + m < max_ug) ug[nu + m] = TcTile{e, m, beg + n0, c};
      for (int m = lane; m < dn_mtiles; m += 32)
        if (nd + m < max_dn) dn[nd + m] = TcTile{e, m, beg + n0, c};
      nu = min(nu + ug_mtiles, max_ug);
      nd = min(nd + dn_mtiles, max_dn);
    }
  }
  if (lane == 0) {
    counts[0] = nu;
    counts[1] = nd;
  }
}

// x rows in route order as fp16 (zero beyond H); out-of-range magnitudes
// flag an overflow.
template <typename XT>
__global__ void gather_x16_kernel(const XT *__restrict__ x, const int *__restrict__ route_token,
                                  const int *__restrict__ total, int H, int Hp, int max_rows,
                                  __half *__restrict__ x16, unsigned *err) {
  const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;  // one 8-element chunk
  const int hp8 = Hp / 8;
  const int64_t row = i / hp8;
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

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::mutex g_encode_mu;
int g_sms_tc = 0;

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
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {row_pitch};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, dt, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swz, CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <bool UG>
size_t tc_smem() {
  constexpr int NA = UG ? 2 : 1;
  return 1024 + (size_t)kOpStages * (NA * kATile + kBTile) + (size_t)kRawStages * NA * kTM * kSBBytes;
}

}  // namespace

int tc_max_tiles(const Layer &L, bool up_gate) {
  const int64_t n_tiles = (int64_t)L.max_routes / kNT + L.E + L.S;
  return (int)(n_tiles * (up_gate ? L.Fp / kTM : L.Hp / kTM));
}

cudaError_t tc_prepare(Layer &L) {
  cudaError_t e = get_encode();
  if (e != cudaSuccess) return e;
  e = encode_2d(&L.map_gu_raw, CU_TENSOR_MAP_DATA_TYPE_UINT8, L.gu, (uint64_t)L.gu_row_bytes,
                (uint64_t)(L.E + L.S) * 2 * L.Fp, (uint64_t)L.gu_row_bytes, kSBBytes, 64,
                CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e == cudaSuccess)
    e = encode_2d(&L.map_dn_raw, CU_TENSOR_MAP_DATA_TYPE_UINT8, L.dn, (uint64_t)L.dn_row_bytes,
                  (uint64_t)(L.E + L.S) * L.Hp, (uint64_t)L.dn_row_bytes, kSBBytes, kTM,
                  CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e == cudaSuccess)
    e = encode_2d(&L.map_x16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, L.x16, (uint64_t)L.Hp,
                  (uint64_t)L.max_routes, (uint64_t)L.Hp * 2, kKS, kNT, CU_TENSOR_MAP_SWIZZLE_128B);
  if (e == cudaSuccess)
    e = encode_2d(&L.map_h16, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, L.h16, (uint64_t)L.Fp,
                  (uint64_t)L.max_routes, (uint64_t)L.Fp * 2, kKS, kNT, CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(grouped_gemm_tc<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)tc_smem<true>());
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(grouped_gemm_tc<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)tc_smem<false>());
  if (e == cudaSuccess && g_sms_tc == 0) {
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&g_sms_tc, cudaDevAttrMultiProcessorCount, dev);
  }
  return e;
}

cudaError_t launch_prefill_tc(const Layer &L, const void *x, moe_dtype xdt, int T,
                              cudaStream_t stream) {
  const int max_rows = T * L.k + L.S * T;
  // tile lists
  build_tiles_kernel<<<1, 32, 0, stream>>>(L.offsets, L.active, L.E + L.S, L.Fp / kTM, L.Hp / kTM,
                                           L.tiles_ug, L.tiles_dn, L.tile_counts,
                                           tc_max_tiles(L, true), tc_max_tiles(L, false));
  count_launches(1);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // gather x in route order as fp16
  const int64_t chunks = (int64_t)max_rows * (L.Hp / 8);
  const int gb = (int)((chunks + 255) / 256);
  if (xdt == MOE_DT_BF16)
    gather_x16_kernel<__nv_bfloat16><<<gb, 256, 0, stream>>>(
        (const __nv_bfloat16 *)x, L.route_token, L.offsets + L.E + L.S, L.H, L.Hp, max_rows, L.x16, L.err);
  else
    gather_x16_kernel<float><<<gb, 256, 0, stream>>>((const float *)x, L.route_token, L.offsets + L.E + L.S,
                                                     L.H, L.Hp, max_rows, L.x16, L.err);
  count_launches(1);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  TcParams p;
  p.route_token = L.route_token;
  p.route_weight = L.route_weight;
  p.h16 = L.h16;
  p.out_acc = L.out_acc;
  p.err = L.err;
  p.H = L.H;
  p.Hp = L.Hp;
  p.Fp = L.Fp;
  p.gu_rows_per_expert = 2 * (int64_t)L.Fp;
  p.dn_rows_per_expert = L.Hp;
  // up/gate + SwiGLU
  p.tiles = L.tiles_ug;
  p.n_tiles = L.tile_counts;
  grouped_gemm_tc<true><<<g_sms_tc, kThreadsTC, tc_smem<true>(), stream>>>(p, L.map_gu_raw, L.map_x16);
  count_launches(1);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // down + weighted scatter
  p.tiles = L.tiles_dn;
  p.n_tiles = L.tile_counts + 1;
  grouped_gemm_tc<false><<<g_sms_tc, kThreadsTC, tc_smem<false>(), stream>>>(p, L.map_dn_raw, L.map_h16);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace moe
